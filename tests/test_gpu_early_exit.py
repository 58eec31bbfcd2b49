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
