"""GPU parity: the CUDA verify path against the fp64 CPU oracle.

Accepted counts and token ids must match the oracle exactly, except on
sequences whose first difference is a draw within 1e-6 of a decision boundary
(counted and reported, see parity.py).  Probabilities exported by the stats
entry points must agree with the oracle to 1e-5 relative.  The greedy chain,
the tree path and the tree mask must match bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_36_gb300 as sv
from speculative_decoding_verification_36_gb300 import workloads as wl
from parity import chain_report, oracle_chain_threads, oracle_greedy_threads, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _dev(t):
    return None if t is None else t.to(DEV)


def run_chain(x, seed, stream=None):
    tokens, n = sv.spec_verify(_dev(x["target"]), _dev(x["draft"]), _dev(x["tokens"]),
                               x["temperature"], seed, stream=stream)
    torch.cuda.synchronize()
    return tokens.cpu().numpy(), n.cpu().numpy()


def check_chain_outputs(tokens, n, x, K, V):
    """Properties that hold at any size."""
    drafts = x["tokens"].cpu().numpy()
    for b in range(len(n)):
        assert 0 <= n[b] <= K
        assert np.array_equal(tokens[b, :n[b]], drafts[b, :n[b]])
        assert 0 <= tokens[b, n[b]] < V
        assert (tokens[b, n[b] + 1:] == -1).all()


SAMPLING_CASES = [
    ("c1", {}),                           # B=1 K=4 V=32000 fp32, tau 1
    ("c2", dict(B=16)),                   # full V=128256 bf16, tau 1, spike prior
    ("c3", dict(B=12)),                   # full V=152064 bf16, K=8, tau 0.7, Zipf prior
    ("c2", dict(B=8, V=1000)),            # vector path, one ragged chunk
    ("c2", dict(B=8, V=1001)),            # scalar path: rows not 16-byte aligned
    ("c3", dict(B=6, V=4093, K=1)),
    ("c1", dict(B=5, V=7, K=3)),          # tiny vocabulary
    ("c1", dict(B=5, V=1, K=2)),          # a single token
    ("c2", dict(B=4, K=0, V=2048)),       # no drafts: the bonus token only
    ("c1", dict(B=3, K=31, V=600)),       # acceptance scan across a 32-lane boundary
    ("c1", dict(B=2, K=40, V=300)),
    ("c1", dict(B=2, K=255, V=64)),       # the largest K: 511 rows, eight 32-position chunks
    ("c3", dict(B=3, K=2, V=1048576)),    # 342 tail slices per row: the CDF search takes 3 rounds
    ("c1", dict(B=2, K=2, V=999999)),     # fp32 scalar path, 652 tail slices per row
    ("c2", dict(B=2048, K=2, V=512)),     # many short sequences (small-batch scheduling)
    ("c2", dict(B=2100, K=3, V=6400)),    # 2100 queue entries with the full-size scheduling
]


@pytest.mark.parametrize("name,over", SAMPLING_CASES)
def test_sampling_parity(name, over):
    p = wl.preset(name, **over)
    x = wl.make_chain(p, seed=11)
    tokens, n = run_chain(x, seed=11)
    check_chain_outputs(tokens, n, x, p.K, p.V)
    ref = oracle.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 11)
    rep = chain_report(tokens, n, ref)
    print(f"{name} {over}: n={n.tolist()[:16]} boundary={rep['boundary']} "
          f"boundary_draws={rep['boundary_draws']}")
    assert not rep["mismatch"], rep


@pytest.mark.parametrize("name,over", [("c1", dict(B=6, temperature=0.05)),     # c = 28.9: sharp rows
                                       ("c2", dict(B=6, V=4096, temperature=0.05)),
                                       ("c1", dict(B=6, temperature=20.0)),       # c = 0.07: flat rows
                                       ("c3", dict(B=4, V=8192, temperature=20.0)),
                                       ("c2", dict(B=3, K=6, V=1001, temperature=3.0))])
def test_sampling_parity_extreme_temperatures(name, over):
    """The acceptance test (exponent from error-free differences, ex2) and
    log2(sT / sD) (float pairs) across temperatures whose exponent
    differences are very large or very small."""
    p = wl.preset(name, **over)
    x = wl.make_chain(p, seed=17)
    tokens, n = run_chain(x, seed=17)
    check_chain_outputs(tokens, n, x, p.K, p.V)
    ref = oracle.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 17)
    rep = chain_report(tokens, n, ref)
    print(f"{name} {over}: n={n.tolist()} boundary={rep['boundary']}")
    assert not rep["mismatch"], rep
    out = sv.spec_verify_stats(_dev(x["target"]), _dev(x["draft"]), _dev(x["tokens"]), p.temperature, 17)
    torch.cuda.synchronize()
    same = out["n"].cpu().numpy() == ref["n"]
    e_z = rel_err(out["resid_mass"].cpu().numpy()[same], ref["resid_mass"][same]).max()
    assert e_z <= 1e-5, e_z


@pytest.mark.parametrize("name,over", [("c1", {}), ("c3", dict(B=8)), ("c2", dict(B=4, V=1001)),
                                       ("c2", dict(B=6))])
def test_sampling_probabilities(name, over):
    p = wl.preset(name, **over)
    x = wl.make_chain(p, seed=5)
    out = sv.spec_verify_stats(_dev(x["target"]), _dev(x["draft"]), _dev(x["tokens"]),
                               p.temperature, 5)
    torch.cuda.synchronize()
    ref = oracle.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 5)
    rs = out["row_stats"].cpu().numpy()
    assert rel_err(rs[..., 0], ref["row_logmax"]).max() <= 1e-6
    e_sum = rel_err(rs[..., 1], ref["row_sum"]).max()
    pq = out["pq"].cpu().numpy()
    examined = np.isfinite(ref["px"])
    e_p = rel_err(pq[..., 0][examined], ref["px"][examined]).max()
    e_q = rel_err(pq[..., 1][examined], ref["qx"][examined]).max()
    n = out["n"].cpu().numpy()
    same = n == ref["n"]
    e_z = rel_err(out["resid_mass"].cpu().numpy()[same], ref["resid_mass"][same]).max()
    print(f"{name}: rel err sum {e_sum:.2e} p {e_p:.2e} q {e_q:.2e} Z {e_z:.2e}")
    assert e_sum <= 1e-5 and e_p <= 1e-5 and e_q <= 1e-5 and e_z <= 1e-5


@pytest.mark.parametrize("name,over", [("c1", {}), ("c3", dict(B=8)), ("c2", dict(B=4, V=1001)),
                                       ("c2", dict(B=4, K=0, V=2048)), ("c1", dict(B=3, K=40, V=300))])
def test_row_entropy(name, over):
    """Entropy of every row's softmax from the statistics pass, against the
    oracle; asking for it leaves the tokens unchanged."""
    p = wl.preset(name, **over)
    x = wl.make_chain(p, seed=8)
    if name == "c1":  # masked vocabulary entries in the first target row
        x["target"][0, 0, ::7] = -float("inf")
    out = sv.spec_verify_stats(_dev(x["target"]), _dev(x["draft"]), _dev(x["tokens"]),
                               p.temperature, 9, entropy=True)
    plain_t, plain_n = run_chain(x, seed=9)
    h = out["row_entropy"].cpu().numpy()
    rows = torch.cat([x["target"], x["draft"]], dim=1) if p.K > 0 else x["target"]
    ref = oracle.row_entropy(rows, p.temperature)
    err = np.abs(h - ref) / np.maximum(1.0, np.abs(ref))
    print(f"{name}: entropy err {err.max():.2e}")
    assert err.max() <= 1e-5
    assert np.array_equal(out["tokens"].cpu().numpy(), plain_t)
    assert np.array_equal(out["n"].cpu().numpy(), plain_n)


@pytest.mark.parametrize("name", ["c3", "c2"])
def test_full_size_whole_batch(name):
    """The benchmark's launch at its full size (c3: B=256, V=152064, K=8;
    c2: B=64, V=128256), every sequence against the oracle.  The draws within
    1e-6 of a decision boundary are counted and printed."""
    p = wl.preset(name)
    x = wl.make_chain(p, device=DEV, seed=0)
    tokens, n = sv.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 0)
    torch.cuda.synchronize()
    tokens, n = tokens.cpu().numpy(), n.cpu().numpy()
    check_chain_outputs(tokens, n, x, p.K, p.V)
    ref = oracle_chain_threads(x["target"], x["draft"], x["tokens"], p.temperature, 0)
    rep = chain_report(tokens, n, ref)
    print(f"{name} full batch B={p.B}: mean n={n.mean():.3f} boundary_draws={rep['boundary_draws']} "
          f"boundary_only_differences={len(rep['boundary'])}")
    assert not rep["mismatch"], rep
    assert sv.spec_get_status() == 0


def test_identical_draft_accepts_everything():
    p = wl.preset("c2", B=16, V=5000)
    x = wl.make_chain(p, seed=2)
    x["draft"] = x["target"][:, :p.K].clone().contiguous()
    tokens, n = run_chain(x, seed=9)
    assert (n == p.K).all()
    assert np.array_equal(tokens[:, :p.K], x["tokens"].numpy())
    ref = oracle.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 9)
    assert not chain_report(tokens, n, ref)["mismatch"]


def test_deterministic_across_runs_and_streams():
    p = wl.preset("c3", B=32, V=20000)
    x = wl.make_chain(p, seed=4)
    a = run_chain(x, seed=123)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        b = run_chain(x, seed=123)
    c = run_chain(x, seed=124)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert not (np.array_equal(a[0], c[0]) and np.array_equal(a[1], c[1]))


def test_neg_inf_logits_are_masked_tokens():
    p = wl.preset("c2", B=8, V=3000)
    x = wl.make_chain(p, seed=8)
    t = x["target"].clone()
    d = x["draft"].clone()
    t[:, :, 100:2000] = float("-inf")
    d[:, :, 500:900] = float("-inf")
    x["target"], x["draft"] = t, d
    tokens, n = run_chain(x, seed=8)
    ref = oracle.spec_verify(t, d, x["tokens"], p.temperature, 8)
    assert not chain_report(tokens, n, ref)["mismatch"]
    # no emitted token can carry zero target probability
    for b in range(p.B):
        assert not (100 <= tokens[b, n[b]] < 2000)


def test_bad_data_is_flagged_not_trapped():
    p = wl.preset("c1", B=6, V=512)
    x = wl.make_chain(p, seed=3)
    t, d, k = x["target"].clone(), x["draft"].clone(), x["tokens"].clone()
    t[1, 2, 7] = float("nan")
    d[2, 0, :] = float("-inf")
    k[3, 1] = p.V
    t[4, 0, 9] = float("inf")
    sv.spec_get_status()  # clear
    tokens, n = sv.spec_verify(t.to(DEV), d.to(DEV), k.to(DEV), p.temperature, 3)
    torch.cuda.synchronize()
    flags = sv.spec_get_status()
    assert flags & sv.SPEC_FLAG_BAD_DATA
    assert not flags & sv.SPEC_FLAG_TIMEOUT
    tokens, n = tokens.cpu().numpy(), n.cpu().numpy()
    ref = oracle.spec_verify(t, d, k, p.temperature, 3)
    assert list(n[1:5]) == [-1, -1, -1, -1] and (tokens[1:5] == -1).all()
    assert not chain_report(tokens, n, ref)["mismatch"]
    # the flag is sticky until read, then clear
    assert sv.spec_get_status() == 0


def test_gpu_adversarial_draft_is_lossless():
    """A draft that puts almost all of its mass where the target has almost
    none: 10^6 replicas match the oracle and the emitted tokens follow p."""
    from scipy import stats
    K, V, R = 2, 6, 1_000_000
    target = torch.zeros(K + 1, V)
    target[:, 0], target[:, 1], target[:, V - 1] = 3.0, 2.5, -6.0
    draft = torch.zeros(K, V)
    draft[:, V - 1] = 8.0
    P = torch.softmax(target.double(), -1).numpy()
    Q = torch.softmax(draft.double(), -1)
    g = torch.Generator().manual_seed(8)
    x = torch.stack([torch.multinomial(Q[i], R, replacement=True, generator=g) for i in range(K)],
                    dim=1).int()
    tokens, n = sv.spec_verify(target.to(DEV).expand(R, K + 1, V).contiguous(),
                               draft.to(DEV).expand(R, K, V).contiguous(), x.to(DEV), 1.0, 77)
    torch.cuda.synchronize()
    tokens, n = tokens.cpu().numpy(), n.cpu().numpy()
    for j in range(K + 1):
        reached = n >= j
        counts = np.bincount(tokens[reached, j], minlength=V)
        assert stats.chisquare(counts, P[j] * reached.sum()).pvalue > 1e-4
    ref = oracle.spec_verify(target, draft, x, 1.0, 77, broadcast=True, n_seq=R)
    assert not chain_report(tokens, n, ref)["mismatch"]


def test_gpu_chi_square_losslessness():
    """V = 8, K = 3, 10^6 replicas of one sequence with drafts drawn from q:
    the token emitted at each reached position follows p (chi-square), and
    every replica matches the oracle."""
    from scipy import stats
    K, V, R = 3, 8, 1_000_000
    g = torch.Generator().manual_seed(17)
    target = (2 * torch.randn(K + 1, V, generator=g)).float()
    draft = (target[:K] + 1.5 * torch.randn(K, V, generator=g)).float()
    P = torch.softmax(target.double(), -1).numpy()
    Q = torch.softmax(draft.double(), -1)
    x = torch.stack([torch.multinomial(Q[i], R, replacement=True, generator=g) for i in range(K)],
                    dim=1).int()
    tokens, n = sv.spec_verify(target.to(DEV).expand(R, K + 1, V).contiguous(),
                               draft.to(DEV).expand(R, K, V).contiguous(), x.to(DEV), 1.0, 2024)
    torch.cuda.synchronize()
    tokens, n = tokens.cpu().numpy(), n.cpu().numpy()
    for j in range(K + 1):
        reached = n >= j
        counts = np.bincount(tokens[reached, j], minlength=V)
        assert stats.chisquare(counts, P[j] * reached.sum()).pvalue > 1e-4
    ref = oracle.spec_verify(target, draft, x, 1.0, 2024, broadcast=True, n_seq=R)
    rep = chain_report(tokens, n, ref)
    print(f"chi-square replicas: boundary={len(rep['boundary'])} draws={rep['boundary_draws']}")
    assert not rep["mismatch"]


# --------------------------------------------------------------------------
# greedy chain
# --------------------------------------------------------------------------
@pytest.mark.parametrize("over", [dict(B=64), dict(B=16, V=1001), dict(B=8, V=1, K=3),
                                  dict(B=8, K=0, V=512), dict(B=3, K=255, V=96)])
def test_greedy_parity(over):
    p = wl.preset("c4", **over)
    x = wl.make_chain(p, seed=21)
    tokens, n = run_chain(x, seed=0)
    ref = oracle.spec_verify_greedy(x["target"], x["tokens"])
    assert np.array_equal(tokens, ref["tokens"]) and np.array_equal(n, ref["n"])


def test_greedy_full_size_whole_batch_and_row_argmax():
    """c4 at full size (B=1024, K=4, V=128256): every sequence against the
    oracle, every row's argmax against torch.argmax."""
    p = wl.preset("c4")
    x = wl.make_chain(p, device=DEV, seed=0)
    tokens, n, amax = sv.spec_verify_greedy_argmax(x["target"], x["tokens"])
    torch.cuda.synchronize()
    assert torch.equal(amax.long(), torch.argmax(x["target"].float(), dim=-1))
    ref = oracle_greedy_threads(x["target"], x["tokens"])
    assert np.array_equal(tokens.cpu().numpy(), ref["tokens"])
    assert np.array_equal(n.cpu().numpy(), ref["n"])
    # tokens equal the argmax with probability 0.7 per position
    assert abs((n.float().mean().item()) - sum(0.7 ** i for i in range(1, 5))) < 0.1


def test_greedy_ties_lowest_index_wins():
    B, K, V = 6, 2, 4096
    t = torch.zeros(B, K + 1, V, dtype=torch.bfloat16)
    t[:, :, :] = -5.0
    # exact ties of the maximum at two or more places, across chunks and lanes
    spots = [(0, [3, 4000]), (1, [0, 1]), (2, [4095, 2048]), (3, [9, 10, 11]), (4, [1500, 7]),
             (5, [2000, 3000])]
    for b, idx in spots:
        for i in idx:
            t[b, :, i] = 7.0
    t[:, :, 50] = float("-inf")
    x = torch.full((B, K), 0, dtype=torch.int32)
    tokens, n, amax = sv.spec_verify_greedy_argmax(t.to(DEV), x.to(DEV))
    amax = amax.cpu()
    for b, idx in spots:
        assert (amax[b] == min(idx)).all()
    ref = oracle.spec_verify_greedy(t, x)
    assert np.array_equal(tokens.cpu().numpy(), ref["tokens"])


# --------------------------------------------------------------------------
# tree
# --------------------------------------------------------------------------
def run_tree(tr):
    path, length, mask = sv.spec_tree_verify_greedy(_dev(tr["target"]), _dev(tr["tokens"]),
                                                    _dev(tr["parents"]))
    torch.cuda.synchronize()
    return path.cpu().numpy(), length.cpu().numpy(), mask.cpu().numpy().view(np.uint32)


def test_tree_c5_full():
    p = wl.preset("c5")
    tr = wl.make_tree(p, seed=0)
    path, length, mask = run_tree(tr)
    ref = oracle.tree_verify_greedy(tr["target"], tr["tokens"], tr["parents"])
    assert np.array_equal(path, ref["path"])
    assert np.array_equal(length, ref["length"])
    assert np.array_equal(mask, ref["mask"])
    print(f"c5 accepted path lengths: {length.tolist()}")


@pytest.mark.parametrize("N,V,seed", [(100, 257, 1), (300, 512, 2), (1024, 64, 3), (1, 9, 4)])
def test_tree_random_shapes(N, V, seed):
    rng = np.random.default_rng(seed)
    # random BFS-ordered parents: each node hangs under an earlier node or the root
    par = np.array([int(rng.integers(-1, i)) for i in range(N)], dtype=np.int32)
    par[0] = -1
    p = wl.TreePreset("t", 3, 1, V, torch.float32 if seed % 2 else torch.bfloat16, seed)
    tr = wl.make_tree(p, seed=seed, parents=par)
    path, length, mask = run_tree(tr)
    ref = oracle.tree_verify_greedy(tr["target"], tr["tokens"], tr["parents"])
    assert np.array_equal(path, ref["path"])
    assert np.array_equal(length, ref["length"])
    assert np.array_equal(mask, ref["mask"])


def test_tree_without_nodes_emits_root_argmax():
    t = torch.randn(3, 1, 1000)
    path, length, mask = sv.spec_tree_verify_greedy(t.to(DEV), None, None)
    assert (length.cpu() == 1).all()
    assert torch.equal(path.cpu()[:, 0].long(), torch.argmax(t[:, 0], -1))


def test_tree_bad_parent_is_flagged():
    p = wl.preset("c5", B=3, V=512)
    tr = wl.make_tree(p, seed=1)
    par = tr["parents"].clone()
    par[1, 5] = 9  # a parent after its child
    tr["parents"] = par
    sv.spec_get_status()
    path, length, mask = run_tree(tr)
    assert sv.spec_get_status() & sv.SPEC_FLAG_BAD_DATA
    ref = oracle.tree_verify_greedy(tr["target"], tr["tokens"], tr["parents"])
    assert np.array_equal(path, ref["path"]) and np.array_equal(length, ref["length"])
    assert np.array_equal(mask, ref["mask"])
    assert length[1] == -1


def test_bad_data_after_the_first_rejection_still_flags_the_sequence():
    """Decisions are taken as soon as positions 0..n are resolved; the rows
    after n are still checked before the outputs are written."""
    B, K, V = 6, 4, 512
    g = torch.Generator().manual_seed(5)
    t = 2.0 * torch.randn(B, K + 1, V, generator=g)
    d = t[:, :K].clone()
    x = torch.randint(0, V, (B, K), generator=g, dtype=torch.int32)
    # position 0 rejects for certain: q(x_0) near 1, p(x_0) near 0
    for b in range(B):
        d[b, 0, x[b, 0]] = 40.0
        t[b, 0, x[b, 0]] = -40.0
    t[0, 3, 11] = float("nan")         # a target row after n = 0
    d[1, 2, :] = float("-inf")          # a draft row with no mass after n = 0
    x[2, 3] = V                          # a token out of range after n = 0
    t[3, K, 5] = float("inf")           # the bonus row (never drawn from here)
    # sequence 4: clean; sequence 5: every draft accepted (q = p), bad bonus row
    d[5] = t[5, :K]
    x[5] = torch.argmax(t[5, :K], dim=-1).to(torch.int32)
    t[5, K, 0] = float("nan")
    sv.spec_get_status()
    for dt in (torch.float32, torch.bfloat16):
        tt, dd = t.to(dt), d.to(dt)
        tokens, n = sv.spec_verify(tt.to(DEV), dd.to(DEV), x.to(DEV), 1.0, 17)
        torch.cuda.synchronize()
        assert sv.spec_get_status() & sv.SPEC_FLAG_BAD_DATA
        tokens, n = tokens.cpu().numpy(), n.cpu().numpy()
        ref = oracle.spec_verify(tt, dd, x, 1.0, 17)
        assert list(ref["n"][[0, 1, 2, 3, 5]]) == [-1] * 5 and ref["n"][4] == 0
        assert list(n) == list(ref["n"])
        assert np.array_equal(tokens, ref["tokens"]), (tokens, ref["tokens"])
    assert sv.spec_get_status() == 0
