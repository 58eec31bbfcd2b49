"""GPU parity of the suggested next draft length (spec_verify_khint_*).

The oracle recomputes, from the same seeded inputs, the accepted counts n,
the entropy of every target row and the suggestion (oracle.adaptive_k).  The
kernel's mean entropy comes from fp32 row statistics, so the thresholds are
placed in gaps of the oracle's means, at least 1e-4 (relative) from every one
of them: there the suggestion must match exactly on every sequence whose n
matches (n itself follows the chain parity bar: a difference is excused only
at a draw within 1e-6 of its decision boundary).
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_36_gb300 as sv
from speculative_decoding_verification_36_gb300 import workloads as wl
from parity import chain_report

pytestmark = pytest.mark.gpu
DEV = "cuda"
MARGIN = 1e-4


def _gap_threshold(hbar, q):
    """A value near quantile q of hbar, at least MARGIN (relative) from each."""
    v = np.unique(hbar[np.isfinite(hbar)])
    if v.size == 0:
        return 1.0
    order = np.argsort(np.abs(np.arange(v.size + 1) - q * v.size))
    for j in order:  # candidate gaps, nearest to the quantile first
        lo = v[j - 1] if j > 0 else v[0] - 1.0
        hi = v[j] if j < v.size else v[-1] + 1.0
        t = 0.5 * (lo + hi)
        if np.all(np.abs(v - t) > MARGIN * np.maximum(1.0, np.abs(v))):
            return float(t)
    raise AssertionError("no threshold gap")


def _oracle_khint(x, p, seed):
    ref = oracle.spec_verify(x["target"].cpu(), x["draft"].cpu(), x["tokens"].cpu(),
                             p.temperature, seed)
    h = oracle.row_entropy(x["target"].cpu(), p.temperature)
    base = oracle.adaptive_k(h, ref["n"], p.K, -np.inf, np.inf, 0, 255)
    return ref, h, base["mean_entropy"]


def _check(x, p, seed, k_min, k_max, ref, h, hbar):
    h_lo = _gap_threshold(hbar, 1 / 3)
    h_hi = max(h_lo, _gap_threshold(hbar, 2 / 3))
    want = oracle.adaptive_k(h, ref["n"], p.K, h_lo, h_hi, k_min, k_max)
    tokens, n, k_next, hmean = sv.spec_verify_khint(
        x["target"].to(DEV), x["draft"].to(DEV), x["tokens"].to(DEV), p.temperature, seed,
        h_lo, h_hi, k_min, k_max)
    torch.cuda.synchronize()
    tokens, n, k_next, hmean = (t.cpu().numpy() for t in (tokens, n, k_next, hmean))
    rep = chain_report(tokens, n, ref)
    assert not rep["mismatch"], rep
    same = n == ref["n"]
    assert np.array_equal(k_next[same], want["k_next"][same])
    good = same & (n >= 0)
    err = np.abs(hmean[good] - want["mean_entropy"][good]) / np.maximum(1.0, np.abs(want["mean_entropy"][good]))
    assert err.size == 0 or err.max() <= 1e-5, err.max()
    assert np.isnan(hmean[n < 0]).all() and (k_next[n < 0] == -1).all()
    # every move is one step from K, inside the clamp
    ok = k_next[n >= 0]
    assert ((ok >= k_min) & (ok <= k_max)).all()
    return k_next, n, want


CASES = [
    ("c3", dict(B=16), 1, 16),            # bf16 V=152064, K=8, tau 0.7
    ("c1", dict(B=6), 2, 6),              # fp32 V=32000, K=4
    ("c2", dict(B=12, V=1001), 0, 10),    # scalar path (rows not 16-byte aligned)
    ("c2", dict(B=8, K=0, V=2048), 0, 3),  # the bonus row only
    ("c1", dict(B=4, K=40, V=300), 30, 50),  # means over more than 32 rows
]


@pytest.mark.parametrize("name,over,k_min,k_max", CASES)
def test_khint_matches_the_oracle(name, over, k_min, k_max):
    p = wl.preset(name, **over)
    x = wl.make_chain(p, seed=21)
    ref, h, hbar = _oracle_khint(x, p, 21)
    k_next, n, want = _check(x, p, 21, k_min, k_max, ref, h, hbar)
    print(f"{name} {over}: k_next={k_next.tolist()[:16]} n={n.tolist()[:16]}")
    assert sv.spec_get_status() == 0


def test_khint_closed_form_batch():
    """Rows uniform over M tokens (entropy ln M), drafts forcing n = 3, 0, 1
    and a bad sequence: the suggestions are 3, 2, 4 and -1 at thresholds 1.2
    and 1.9 (means 2.5 ln 2, 3 ln 2, 1.5 ln 2)."""
    K, V = 3, 64
    M = (8, 1, 64, 2)
    target = torch.full((4, K + 1, V), -float("inf"))
    for i, m in enumerate(M):
        target[:, i, :m] = 0.0
    draft = target[:, :K].clone()
    tokens = torch.zeros(4, K, dtype=torch.int32)
    draft[1, 0] = -float("inf")
    draft[1, 0, :32] = 0.0
    tokens[1, 0] = 10
    tokens[2, 0] = 3
    tokens[2, 1] = 5
    draft[2, 1] = 0.0
    target[3, 2, 7] = float("nan")
    for dt in (torch.float32, torch.bfloat16):
        t, n, k, hm = sv.spec_verify_khint(target.to(dt).to(DEV), draft.to(dt).to(DEV), tokens.to(DEV), 0.7, 5,
                                           1.2, 1.9, 1, 8)
        torch.cuda.synchronize()
        assert n.tolist() == [3, 0, 1, -1]
        assert k.tolist() == [3, 2, 4, -1]
        hm = hm.cpu().numpy()
        want = np.log(2.0) * np.array([2.5, 3.0, 1.5])
        assert np.abs(hm[:3] - want).max() < 1e-5
        assert np.isnan(hm[3])
        assert sv.spec_get_status() == sv.SPEC_FLAG_BAD_DATA


def test_khint_full_size_c3():
    """The full c3 batch (B=256): every sequence against the oracle."""
    p = wl.preset("c3")
    x = wl.make_chain(p, device=DEV, seed=3)
    ref, h, hbar = _oracle_khint(x, p, 3)
    k_next, n, want = _check(x, p, 3, 1, 16, ref, h, hbar)
    # the entropy pass sums the rows exactly as the plain verify does: the
    # same tokens and counts bit for bit
    t0, n0 = sv.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 3)
    t1, n1, _, _ = sv.spec_verify_khint(x["target"], x["draft"], x["tokens"], p.temperature, 3, 1.0, 2.0, 1, 16)
    torch.cuda.synchronize()
    assert torch.equal(t0, t1) and torch.equal(n0, n1)
    # the thresholds split the batch: some sequences move each way
    assert (k_next == p.K + 1).any() and (k_next == p.K - 1).any() and (k_next == p.K).any()
    assert sv.spec_get_status() == 0


def test_khint_argument_checks():
    p = wl.preset("c2", B=2, K=2, V=256)
    x = wl.make_chain(p, device=DEV, seed=1)
    args = (x["target"], x["draft"], x["tokens"])
    for bad in ((2.0, 1.0, 0, 4), (0.0, 1.0, 5, 4), (0.0, 1.0, -1, 4), (0.0, 1.0, 0, 256),
                (float("nan"), 1.0, 0, 4)):
        with pytest.raises(sv.SpecError) as e:
            sv.spec_verify_khint(*args, p.temperature, 1, *bad)
        assert e.value.code == -6
    with pytest.raises(sv.SpecError) as e:
        sv.spec_verify_khint(*args, 0.0, 1, 0.0, 1.0, 0, 4)
    assert e.value.code == -3
