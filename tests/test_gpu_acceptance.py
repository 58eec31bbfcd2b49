"""GPU acceptance statistics (spec_acceptance_stats) against the oracle, and
at scale against the page's expected-tokens formula through the verify
kernel itself."""
import math

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_36_gb300 as sv

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def _gpu(n, K):
    r = sv.spec_acceptance_stats(torch.as_tensor(n, dtype=torch.int32, device=DEV), K)
    torch.cuda.synchronize()
    return r["hist"].cpu().numpy().astype(np.uint64), r["alpha"].cpu().numpy(), float(r["mean_tokens"])


@pytest.mark.parametrize("B,K", [(100003, 8), (1, 1), (4096, 255), (20000, 1024), (777, 0)])
def test_matches_oracle(B, K):
    rng = np.random.default_rng(B + K)
    n = rng.integers(-3, K + 3, size=B).astype(np.int32)  # includes bad and out-of-range values
    hist, alpha, mean = _gpu(n, K)
    ref = oracle.acceptance_stats(n, K)
    assert np.array_equal(hist, ref["hist"])
    # both sides divide the same exact integer counts
    assert np.array_equal(np.isnan(alpha), np.isnan(ref["alpha"]))
    assert np.allclose(alpha, ref["alpha"], rtol=1e-15, atol=0, equal_nan=True)
    assert mean == pytest.approx(ref["mean_tokens"], rel=1e-15, abs=0) or (
        math.isnan(mean) and math.isnan(ref["mean_tokens"]))


def test_empty_batch():
    hist, alpha, mean = _gpu(np.zeros(0, dtype=np.int32), 3)
    assert hist.tolist() == [0] * 5 and np.isnan(alpha).all() and math.isnan(mean)


@pytest.mark.parametrize("alpha", [0.7, 0.9])
def test_verify_outputs_follow_the_closed_form(alpha):
    """One million sequences through spec_verify on rows built so that every
    drafted token is accepted with probability alpha (q = (1, 0), p = (alpha,
    1 - alpha)); the statistics kernel then recovers alpha at every position
    and the mean tokens per iteration (1 - alpha^(K+1)) / (1 - alpha)."""
    K, B, V = 4, 1 << 20, 2
    lp = torch.tensor([math.log(alpha), math.log(1 - alpha)], dtype=torch.float32)
    lq = torch.tensor([0.0, -float("inf")], dtype=torch.float32)
    target = lp.expand(B, K + 1, V).contiguous().to(DEV)
    draft = lq.expand(B, K, V).contiguous().to(DEV)
    tokens = torch.zeros((B, K), dtype=torch.int32, device=DEV)
    _, n = sv.spec_verify(target, draft, tokens, 1.0, 77)
    r = sv.spec_acceptance_stats(n, K)
    torch.cuda.synchronize()
    assert sv.spec_get_status() == 0
    hist = r["hist"].cpu().numpy()
    assert hist[K + 1] == 0 and hist.sum() == B
    a = r["alpha"].cpu().numpy()
    for i in range(K):
        reached = int(hist[i:K + 1].sum())
        assert abs(a[i] - alpha) < 5 * math.sqrt(alpha * (1 - alpha) / reached)
    nn = n.cpu().numpy().astype(np.float64) + 1
    expect = (1 - alpha ** (K + 1)) / (1 - alpha)
    assert abs(float(r["mean_tokens"]) - expect) < 5 * nn.std() / math.sqrt(B)
