"""spec_verify_bf16_static_scratch: the same verify kernels on the library's
fixed per-device scratch buffer instead of its memory pool.

Collected last (file name), and also correct when run alone: each test
compares two consecutive static-scratch calls with the pool-backed entry point
on the same inputs and seeds, so leftover state in the buffer from any earlier
call, in this file or another, would show up as a mismatch."""
import pytest
import torch

import speculative_decoding_verification_36_gb300 as sv
from speculative_decoding_verification_36_gb300 import _lib
from speculative_decoding_verification_36_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def _pair(p, seed_a, seed_b):
    xa = wl.make_chain(p, device=DEV, seed=seed_a)
    xb = wl.make_chain(p, device=DEV, seed=seed_b)
    return xa, xb


@pytest.mark.parametrize("name,overrides", [
    ("c2", dict(B=16, V=32000)),            # sampling path, several slices per row
    ("c3", dict(B=8, V=152064)),            # the benchmark's vocabulary, ragged last slice
    ("c2", dict(B=5, V=1000, K=0)),         # bonus draw only
    ("c4", dict(B=32, V=32000)),            # temperature 0: greedy path
])
def test_matches_pool_entry_point_on_consecutive_calls(name, overrides):
    p = wl.preset(name, **overrides)
    xa, xb = _pair(p, 1, 2)
    sv.spec_get_status()
    outs = []
    for x, seed in ((xa, 11), (xb, 12)):  # two calls back to back on one stream
        t, n = sv.spec_verify_static_scratch(x["target"], x["draft"], x["tokens"], p.temperature,
                                             seed)
        outs.append((t.clone(), n.clone()))
    torch.cuda.synchronize()
    for (t, n), (x, seed) in zip(outs, ((xa, 11), (xb, 12))):
        t_ref, n_ref = sv.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, seed)
        torch.cuda.synchronize()
        assert torch.equal(t, t_ref)
        assert torch.equal(n, n_ref)
    assert sv.spec_get_status() == 0


def test_caller_buffers_are_written_in_place():
    p = wl.preset("c2", B=4, V=4096)
    x = wl.make_chain(p, device=DEV, seed=3)
    out_t = torch.full((p.B, p.K + 1), -7, dtype=torch.int32, device=DEV)
    out_n = torch.full((p.B,), -7, dtype=torch.int32, device=DEV)
    t, n = sv.spec_verify_static_scratch(x["target"], x["draft"], x["tokens"], p.temperature, 5,
                                         out_tokens=out_t, out_n_accepted=out_n)
    assert t.data_ptr() == out_t.data_ptr() and n.data_ptr() == out_n.data_ptr()
    t_ref, n_ref = sv.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 5)
    torch.cuda.synchronize()
    assert torch.equal(out_t, t_ref) and torch.equal(out_n, n_ref)


def test_oversized_problem_is_refused_without_launch():
    # Scratch grows with the number of rows and input with their length: 512
    # sequences of K = 255 drafts over V = 16 need about 13 MB of scratch
    # (per-row tickets, partials, row statistics) from 8 MB of logits, more
    # than the 8 MiB buffer.  Only shapes are used before the refusal, but the
    # inputs are real device buffers of the declared shapes all the same.
    B, K, V = 512, 255, 16
    target = torch.zeros((B, K + 1, V), dtype=torch.bfloat16, device=DEV)
    draft = torch.zeros((B, K, V), dtype=torch.bfloat16, device=DEV)
    tokens = torch.zeros((B, K), dtype=torch.int32, device=DEV)
    out_t = torch.full((B, K + 1), -7, dtype=torch.int32, device=DEV)
    out_n = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    with pytest.raises(sv.SpecError) as err:
        sv.spec_verify_static_scratch(target, draft, tokens, 0.7, 1, out_tokens=out_t,
                                      out_n_accepted=out_n)
    assert err.value.code == _lib.SPEC_ERR_SCRATCH
    torch.cuda.synchronize()
    assert bool((out_t == -7).all()) and bool((out_n == -7).all())
