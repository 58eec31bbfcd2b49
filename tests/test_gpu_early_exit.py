"""GPU parity of the early-exit verify (spec_verify_early_exit): tokens and
counts equal the oracle's with the used-rows reading of the bad-data rule
(and spec_verify's on valid inputs); rows after the first rejection never
change the result."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_36_gb300 as sv
from speculative_decoding_verification_36_gb300 import workloads as wl
from parity import chain_report

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def _dev(x):
    return x.to(DEV).contiguous()


@pytest.mark.parametrize("name,over", [
    ("c1", {}), ("c2", dict(B=24)), ("c3", dict(B=32)), ("c3", dict(B=6, V=4093, K=1)),
    ("c2", dict(B=4, K=0, V=2048)), ("c1", dict(B=5, V=7, K=3)), ("c1", dict(B=3, K=31, V=600)),
    ("c1", dict(B=2, K=40, V=300)), ("c3", dict(B=3, K=2, V=1048576)), ("c2", dict(B=2100, K=3, V=6400)),
])
def test_early_exit_parity(name, over):
    p = wl.preset(name, **over)
    x = wl.make_chain(p, seed=11)
    t, d, k = _dev(x["target"]), _dev(x["draft"]), _dev(x["tokens"])
    tok_e, n_e = sv.spec_verify_early_exit(t, d, k, p.temperature, 11)
    tok_f, n_f = sv.spec_verify(t, d, k, p.temperature, 11)
    torch.cuda.synchronize()
    assert sv.spec_get_status() == 0
    # the same tokens as the full-read verify on valid inputs (same uniforms)
    assert torch.equal(tok_e, tok_f) and torch.equal(n_e, n_f)
    ref = oracle.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 11, used_rows_only=True)
    rep = chain_report(tok_e.cpu().numpy(), n_e.cpu().numpy(), ref)
    assert not rep["mismatch"], rep


def test_early_exit_ignores_rows_after_the_first_rejection():
    B, K, V = 8, 4, 512
    g = torch.Generator().manual_seed(8)
    t = 2.0 * torch.randn(B, K + 1, V, generator=g)
    d = t[:, :K].clone()
    x = torch.randint(0, V, (B, K), generator=g, dtype=torch.int32)
    for b in range(B):  # position 0 rejects for certain
        d[b, 0, x[b, 0]] = 40.0
        t[b, 0, x[b, 0]] = -40.0
    t[0, 3, 11] = float("nan")
    d[1, 2, :] = float("-inf")
    x[2, 3] = V
    t[3, K, 5] = float("inf")
    # sequence 4: a bad row that is used (position 0)
    d[4, 0, 7] = float("nan")
    # sequence 5: every draft accepted (q = p) and a bad bonus row: used
    d[5] = t[5, :K]
    x[5] = torch.argmax(t[5, :K], dim=-1).to(torch.int32)
    t[5, K, 0] = float("nan")
    sv.spec_get_status()
    for dt in (torch.float32, torch.bfloat16):
        tt, dd = t.to(dt), d.to(dt)
        tokens, n = sv.spec_verify_early_exit(_dev(tt), _dev(dd), _dev(x), 1.0, 23)
        torch.cuda.synchronize()
        assert sv.spec_get_status() & sv.SPEC_FLAG_BAD_DATA
        ref = oracle.spec_verify(tt, dd, x, 1.0, 23, used_rows_only=True)
        assert ref["n"].tolist() == [0, 0, 0, 0, -1, -1, 0, 0]
        assert n.cpu().tolist() == ref["n"].tolist()
        assert np.array_equal(tokens.cpu().numpy(), ref["tokens"])
    assert sv.spec_get_status() == 0


def test_early_exit_full_size_c3_sampled():
    p = wl.preset("c3")
    x = wl.make_chain(p, device=DEV, seed=4)
    tok_e, n_e = sv.spec_verify_early_exit(x["target"], x["draft"], x["tokens"], p.temperature, 4)
    tok_f, n_f = sv.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 4)
    torch.cuda.synchronize()
    assert sv.spec_get_status() == 0
    assert torch.equal(tok_e, tok_f) and torch.equal(n_e, n_f)
    sel = list(range(0, p.B, 16))
    ref = oracle.spec_verify(x["target"][sel].cpu(), x["draft"][sel].cpu(), x["tokens"][sel].cpu(),
                             p.temperature, 4, seq_ids=sel, used_rows_only=True)
    rep = chain_report(tok_e[sel].cpu().numpy(), n_e[sel].cpu().numpy(), ref)
    assert not rep["mismatch"], rep


# --------------------------------------------------------------------------
# greedy (temperature 0): rows after the first mismatch are not read
# --------------------------------------------------------------------------
@pytest.mark.parametrize("over", [dict(B=64), dict(B=16, V=1001), dict(B=8, K=1, V=512),
                                  dict(B=5, K=31, V=300), dict(B=3, K=40, V=96), dict(B=6, K=0, V=128),
                                  dict(B=700, K=3, V=2048)])
def test_greedy_early_exit_parity(over):
    p = wl.preset("c4", **over)
    x = wl.make_chain(p, seed=12)
    t, k = _dev(x["target"]), _dev(x["tokens"])
    tok_e, n_e = sv.spec_verify_early_exit(t, None, k, 0.0, 0)
    tok_f, n_f = sv.spec_verify(t, None, k, 0.0, 0)
    torch.cuda.synchronize()
    assert sv.spec_get_status() == 0
    assert torch.equal(tok_e, tok_f) and torch.equal(n_e, n_f)
    ref = oracle.spec_verify_greedy(x["target"], x["tokens"], used_rows_only=True)
    assert np.array_equal(tok_e.cpu().numpy(), ref["tokens"]) and np.array_equal(n_e.cpu().numpy(), ref["n"])


def test_greedy_early_exit_ignores_rows_after_the_first_mismatch():
    B, K, V = 10, 4, 640
    g = torch.Generator().manual_seed(9)
    t = 3.0 * torch.randn(B, K + 1, V, generator=g)
    am = torch.argmax(t, dim=-1).to(torch.int32)
    x = am[:, :K].clone()
    x[:, 1] = (am[:, 1] + 1) % V  # every sequence mismatches at position 1
    t[0, 2, 9] = float("nan")      # after n: ignored
    t[1, 3, :] = float("-inf")     # after n: ignored
    x[2, 3] = V + 5                 # after n: ignored
    t[3, K, 4] = float("inf")      # bonus row after n: ignored
    t[4, 1, 2] = float("nan")      # at n: used
    x[5, 1] = -3                    # the mismatching token itself is out of range: used
    t[6, 0, 0] = float("inf")      # before n: used
    x[7] = am[7, :K]                # all match, the bonus row is used ...
    t[7, K, 1] = float("nan")      # ... and bad
    x[8] = am[8, :K]                # all match, clean: n = K
    sv.spec_get_status()
    for dt in (torch.float32, torch.bfloat16):
        tt = t.to(dt)
        ref = oracle.spec_verify_greedy(tt, x, used_rows_only=True)
        assert ref["n"].tolist() == [1, 1, 1, 1, -1, -1, -1, -1, K, 1]
        tokens, n = sv.spec_verify_early_exit(_dev(tt), None, _dev(x), 0.0, 0)
        torch.cuda.synchronize()
        assert sv.spec_get_status() & sv.SPEC_FLAG_BAD_DATA
        assert n.cpu().tolist() == ref["n"].tolist()
        assert np.array_equal(tokens.cpu().numpy(), ref["tokens"])
    assert sv.spec_get_status() == 0


def test_greedy_early_exit_full_size_c4():
    p = wl.preset("c4")
    x = wl.make_chain(p, device=DEV, seed=5)
    tok_e, n_e = sv.spec_verify_early_exit(x["target"], None, x["tokens"], 0.0, 0)
    tok_f, n_f = sv.spec_verify(x["target"], None, x["tokens"], 0.0, 0)
    torch.cuda.synchronize()
    assert sv.spec_get_status() == 0
    assert torch.equal(tok_e, tok_f) and torch.equal(n_e, n_f)
    sel = list(range(0, p.B, 64))
    ref = oracle.spec_verify_greedy(x["target"][sel].cpu(), x["tokens"][sel].cpu(), used_rows_only=True)
    assert np.array_equal(tok_e[sel].cpu().numpy(), ref["tokens"])
    assert np.array_equal(n_e[sel].cpu().numpy(), ref["n"])


# --------------------------------------------------------------------------
# greedy tree: the rows under a rejected node are not read
# --------------------------------------------------------------------------
def _tree_inputs(B, V, par, p_match, seed, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    N = len(par)
    t = (3.0 * torch.randn(B, N + 1, V, generator=g)).to(dtype)
    am = torch.argmax(t.float(), dim=-1)
    tok = torch.empty(B, N, dtype=torch.int32)
    for i, p in enumerate(par):
        keep = torch.rand(B, generator=g) < p_match
        tok[:, i] = torch.where(keep, am[:, p + 1], torch.randint(0, V, (B,), generator=g)).to(torch.int32)
    parents = torch.tensor(par, dtype=torch.int32).unsqueeze(0).expand(B, N).contiguous()
    return t.contiguous(), tok, parents


def _binary(depth):
    return [int(x) for x in wl.complete_binary_parents(depth).tolist()]


@pytest.mark.parametrize("label,B,V,par,dtype", [
    ("binary depth 4 (c5 shape)", 32, 4096, _binary(4), torch.bfloat16),
    ("binary depth 3, fp32 scalar", 16, 1001, _binary(3), torch.float32),
    ("32-node chain", 8, 512, [-1] + list(range(31)), torch.bfloat16),
    ("32 root children", 8, 512, [-1] * 32, torch.bfloat16),
    ("single node", 8, 64, [-1], torch.float32),
    ("random 20 nodes", 12, 300, [-1, 0, 0, 1, -1, 2, 3, 3, 4, 0, 5, 9, 6, 12, 1, 8, 8, 11, 2, 17], torch.bfloat16),
    ("33 nodes: every row is read", 4, 256, _binary(4) + [29, 29, 30], torch.bfloat16),
])
def test_tree_early_exit_parity(label, B, V, par, dtype):
    t, tok, parents = _tree_inputs(B, V, par, 0.7, seed=len(par) + B)
    full = sv.spec_tree_verify_greedy(_dev(t), _dev(tok), _dev(parents))
    early = sv.spec_tree_verify_greedy(_dev(t), _dev(tok), _dev(parents), early_exit=True)
    torch.cuda.synchronize()
    assert sv.spec_get_status() == 0
    for f, e in zip(full, early):
        assert torch.equal(f, e), label
    ref = oracle.tree_verify_greedy(t, tok, parents, used_rows_only=True)
    assert np.array_equal(early[0].cpu().numpy(), ref["path"])
    assert np.array_equal(early[1].cpu().numpy(), ref["length"])
    assert np.array_equal(early[2].cpu().numpy().view(np.uint32), ref["mask"])


def test_tree_early_exit_ignores_rows_under_rejected_nodes():
    par = _binary(3)
    N, B, V = len(par), 24, 700
    t, tok, parents = _tree_inputs(B, V, par, 0.6, seed=3, dtype=torch.float32)
    am = torch.argmax(t, dim=-1)
    t2, tok2 = t.clone(), tok.clone()
    for b in range(B):
        acc = []
        for i, p in enumerate(par):
            acc.append(bool((p < 0 or acc[p]) and int(tok[b, i]) == int(am[b, p + 1])))
        for i, p in enumerate(par):
            if not acc[i]:
                t2[b, i + 1, 5] = float("nan")  # a rejected node's row
            if p >= 0 and not acc[p]:
                tok2[b, i] = V + 9                # a token under a rejected node
    sv.spec_get_status()
    clean = sv.spec_tree_verify_greedy(_dev(t), _dev(tok), _dev(parents), early_exit=True)
    spoiled = sv.spec_tree_verify_greedy(_dev(t2), _dev(tok2), _dev(parents), early_exit=True)
    torch.cuda.synchronize()
    assert sv.spec_get_status() == 0
    for c, s in zip(clean, spoiled):
        assert torch.equal(c, s)
    # used bad data is flagged: the root row, and a parent index anywhere
    t3 = t.clone()
    t3[0, 0, 1] = float("inf")
    par3 = parents.clone()
    par3[1, N - 1] = N + 4
    for tt, pp, b in ((t3, parents, 0), (t, par3, 1)):
        ref = oracle.tree_verify_greedy(tt, tok, pp, used_rows_only=True)
        path, length, mask = sv.spec_tree_verify_greedy(_dev(tt), _dev(tok), _dev(pp), early_exit=True)
        torch.cuda.synchronize()
        assert sv.spec_get_status() & sv.SPEC_FLAG_BAD_DATA
        assert int(length[b]) == -1 and ref["length"][b] == -1
        assert np.array_equal(length.cpu().numpy(), ref["length"])
        assert np.array_equal(path.cpu().numpy(), ref["path"])
    assert sv.spec_get_status() == 0


def test_tree_early_exit_full_size_c5():
    p = wl.preset("c5")
    x = wl.make_tree(p, device=DEV, seed=6)
    full = sv.spec_tree_verify_greedy(x["target"], x["tokens"], x["parents"])
    early = sv.spec_tree_verify_greedy(x["target"], x["tokens"], x["parents"], early_exit=True)
    torch.cuda.synchronize()
    assert sv.spec_get_status() == 0
    for f, e in zip(full, early):
        assert torch.equal(f, e)
    ref = oracle.tree_verify_greedy(x["target"][:8].cpu(), x["tokens"][:8].cpu(), x["parents"][:8].cpu(),
                                    used_rows_only=True)
    assert np.array_equal(early[0][:8].cpu().numpy(), ref["path"])
    assert np.array_equal(early[1][:8].cpu().numpy(), ref["length"])
