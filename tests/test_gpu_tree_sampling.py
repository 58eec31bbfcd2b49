"""GPU parity of stochastic tree verification against the fp64 CPU oracle.

Paths and lengths must match the oracle exactly, except on sequences whose
first differing path entry was decided by a draw the oracle flags as within
1e-6 of its decision boundary (acceptance uniform against min(1, P/q), or the
final inverse-CDF draw against a cumulative sum); those are counted and
reported.  Plus the properties the method fixes at any
size: the first emitted token follows the target distribution (chi-square over
replicas), a chain-shaped tree agrees with the chain verify.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_36_gb300 as sv
from speculative_decoding_verification_36_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run(x, seed, stream=None):
    path, length = sv.spec_tree_verify_sampling(
        x["target"].to(DEV), x["draft"].to(DEV),
        None if x["tokens"].numel() == 0 else x["tokens"].to(DEV),
        None if x["parents"].numel() == 0 else x["parents"].to(DEV),
        x["temperature"], seed, stream=stream)
    torch.cuda.synchronize()
    return path.cpu().numpy(), length.cpu().numpy()


def compare(path, length, ref):
    """(mismatching sequences, boundary sequences that differ).  A difference
    is excused only when the first path entry that differs was decided by a
    draw the oracle flags as within 1e-6 of its boundary."""
    mism, bnd = [], []
    for b in range(len(length)):
        if length[b] == ref["length"][b] and np.array_equal(path[b], ref["path"][b]):
            continue
        diff = np.nonzero(path[b] != ref["path"][b])[0]
        j = int(diff[0]) if diff.size else -1
        (bnd if j >= 0 and ref["length"][b] > 0 and ref["boundary_at"][b, j] else mism).append(b)
    return mism, bnd


def check_valid(path, length, x):
    """Structure that holds at any size: the accepted prefix is a root-down
    path of the tree, then one token in [0, V), then -1 padding."""
    tok = x["tokens"].cpu().numpy()
    par = x["parents"].cpu().numpy()
    V = x["target"].shape[-1]
    for b in range(len(length)):
        L = int(length[b])
        assert 1 <= L <= path.shape[1]
        u = -1
        for j in range(L - 1):
            kids = [c for c in range(par.shape[1]) if par[b, c] == u and tok[b, c] == path[b, j]]
            assert kids, (b, j)
            u = kids[0]
        assert 0 <= path[b, L - 1] < V
        assert (path[b, L:] == -1).all()


def random_parents(N, rng):
    par = np.array([int(rng.integers(-1, i)) if i else -1 for i in range(N)], dtype=np.int32)
    return par


CASES = [
    # (label, B, V, dtype, parents, temperature)
    ("binary depth 4, full V", 8, 128256, torch.bfloat16, None, 1.0),
    ("binary depth 4, tau 0.5", 8, 4096, torch.bfloat16, None, 0.5),
    ("scalar path V=1001", 6, 1001, torch.float32, None, 1.0),
    ("wide fan: 40 root children", 6, 1000, torch.float32, [-1] * 40, 1.0),
    ("wide fan bf16, 64 children, tau 2", 4, 2048, torch.bfloat16, [-1] * 64, 2.0),
    ("random 100 nodes", 4, 257, torch.float32, "rand100", 1.0),
    ("random 300 nodes", 3, 512, torch.bfloat16, "rand300", 0.8),
    ("1024 nodes", 2, 64, torch.float32, "rand1024", 1.0),
    ("single node", 8, 9, torch.float32, [-1], 1.0),
    ("tiny vocabulary", 8, 1, torch.float32, [-1, 0, 0], 1.0),
    ("binary depth 2, V=2^20", 2, 1 << 20, torch.bfloat16, [-1, -1, 0, 0, 1, 1], 1.0),
]


@pytest.mark.parametrize("label,B,V,dtype,parents,tau", CASES, ids=[c[0] for c in CASES])
def test_tree_sampling_parity(label, B, V, dtype, parents, tau):
    if isinstance(parents, str):
        parents = random_parents(int(parents[4:]), np.random.default_rng(int(parents[4:])))
    p = wl.TreePreset("t", B, 4, V, dtype, 7)
    x = wl.make_tree_sampling(p, tau, seed=3, parents=parents)
    path, length = run(x, seed=99)
    check_valid(path, length, x)
    ref = oracle.tree_verify_sampling(x["target"], x["draft"], x["tokens"], x["parents"], tau, 99)
    mism, bnd = compare(path, length, ref)
    print(f"{label}: lengths {length.tolist()} boundary-differences {bnd} "
          f"flagged {int(ref['boundary'].sum())}")
    assert not mism, (mism, path[mism], ref["path"][mism])


def test_tree_sampling_c5_shapes_full():
    """B = 32, the complete binary tree of depth 4, V = 128256, bf16."""
    p = wl.preset("c5")
    x = wl.make_tree_sampling(p, 1.0, seed=0)
    path, length = run(x, seed=5)
    check_valid(path, length, x)
    ref = oracle.tree_verify_sampling(x["target"], x["draft"], x["tokens"], x["parents"], 1.0, 5)
    mism, bnd = compare(path, length, ref)
    print(f"c5 stochastic: mean length {length.mean():.3f} boundary-differences {bnd}")
    assert not mism


def test_tree_sampling_without_nodes_draws_from_root():
    g = torch.Generator().manual_seed(4)
    t = torch.randn(5, 1, 700, generator=g)
    d = torch.randn(5, 1, 700, generator=g)
    x = dict(target=t, draft=d, tokens=torch.zeros(5, 0, dtype=torch.int32),
             parents=torch.zeros(5, 0, dtype=torch.int32), temperature=1.0)
    path, length = run(x, seed=8)
    assert (length == 1).all()
    ref = oracle.tree_verify_sampling(t, d, x["tokens"], x["parents"], 1.0, 8)
    mism, _ = compare(path, length, ref)
    assert not mism


def test_tree_sampling_chain_equals_chain_verify():
    """A tree whose node i hangs under node i-1 is the chain of K = N drafts:
    same draws (acceptance counter (b, i, 0), final (b, n, 1)), same tokens."""
    K, B, V = 6, 16, 3000
    c = wl.make_chain(wl.preset("c3", B=B, K=K, V=V), seed=2)
    t = c["target"]
    # draft row i of the chain is draft row i of the tree; the last row is unused
    d = torch.cat([c["draft"], c["draft"][:, -1:]], dim=1).contiguous()
    par = torch.arange(-1, K - 1, dtype=torch.int32).expand(B, K).contiguous()
    x = dict(target=t, draft=d, tokens=c["tokens"], parents=par, temperature=c["temperature"])
    path, length = run(x, seed=31)
    tokens, n = sv.spec_verify(t.to(DEV), c["draft"].to(DEV), c["tokens"].to(DEV),
                               c["temperature"], 31)
    torch.cuda.synchronize()
    ref = oracle.tree_verify_sampling(t, d, c["tokens"], par, c["temperature"], 31)
    ok = ref["boundary"] == 0
    assert np.array_equal(length[ok], n.cpu().numpy()[ok] + 1)
    assert np.array_equal(path[ok], tokens.cpu().numpy()[ok])


def test_tree_sampling_first_token_follows_target():
    """10^5 replicas of one tree (root with 3 children, each with 2): the first
    emitted token follows softmax(root target row / tau)."""
    from scipy import stats
    R, V = 100_000, 12
    g = torch.Generator().manual_seed(23)
    par = [-1, -1, -1, 0, 0, 1, 1, 2, 2]
    N = len(par)
    t = 1.5 * torch.randn(N + 1, V, generator=g)
    d = t + 1.2 * torch.randn(N + 1, V, generator=g)
    tau = 0.9
    Q = torch.softmax(d.double() / tau, -1)
    toks = torch.empty(R, N, dtype=torch.int32)
    for i, pr in enumerate(par):
        toks[:, i] = torch.multinomial(Q[pr + 1], R, replacement=True, generator=g).int()
    x = dict(target=t.expand(R, N + 1, V).contiguous(), draft=d.expand(R, N + 1, V).contiguous(),
             tokens=toks, parents=torch.tensor(par, dtype=torch.int32).expand(R, N).contiguous(),
             temperature=tau)
    path, length = run(x, seed=77)
    P0 = torch.softmax(t[0].double() / tau, -1).numpy()
    counts = np.bincount(path[:, 0], minlength=V)
    assert stats.chisquare(counts, P0 * R).pvalue > 1e-4
    # a sample of the replicas against the oracle
    sel = slice(0, 2000)
    ref = oracle.tree_verify_sampling(x["target"][sel], x["draft"][sel], toks[sel],
                                      x["parents"][sel], tau, 77)
    mism, _ = compare(path[sel], length[sel], ref)
    assert not mism


def test_tree_sampling_bad_data_is_flagged():
    p = wl.TreePreset("t", 4, 2, 300, torch.float32, 1)
    x = wl.make_tree_sampling(p, 1.0, seed=1)
    x["target"][1, 2, 17] = float("nan")
    x["parents"] = x["parents"].clone()
    x["parents"][2, 3] = 5  # a parent after its child
    x["draft"][3, 0, :] = float("-inf")  # no finite draft entry at the root
    sv.spec_get_status()
    path, length = run(x, seed=0)
    assert sv.spec_get_status() & sv.SPEC_FLAG_BAD_DATA
    assert list(length[1:]) == [-1, -1, -1] and (path[1:] == -1).all()
    ref = oracle.tree_verify_sampling(x["target"], x["draft"], x["tokens"], x["parents"], 1.0, 0)
    assert list(ref["length"][1:]) == [-1, -1, -1]
    mism, _ = compare(path, length, ref)
    assert not mism
    assert sv.spec_get_status() == 0


def test_tree_sampling_deterministic_across_streams():
    p = wl.TreePreset("t", 6, 3, 5000, torch.bfloat16, 2)
    x = wl.make_tree_sampling(p, 1.0, seed=4)
    a = run(x, seed=12)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = run(x, seed=12, stream=s)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
