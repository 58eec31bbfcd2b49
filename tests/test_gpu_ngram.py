"""GPU parity of n-gram (prompt-lookup) drafting (spec_ngram_draft) with the
CPU oracle: drafts, draft counts and match lengths must be bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_36_gb300 as sv
from speculative_decoding_verification_36_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def _run(tokens, lengths, n_min, n_max, K):
    t = torch.as_tensor(tokens, dtype=torch.int32).to(DEV).contiguous()
    ln = torch.as_tensor(lengths, dtype=torch.int32).to(DEV).contiguous()
    drafts, nd, ml = sv.spec_ngram_draft(t, ln, n_min, n_max, K)
    torch.cuda.synchronize()
    return drafts.cpu().numpy(), nd.cpu().numpy(), ml.cpu().numpy()


def _check(tokens, lengths, n_min, n_max, K):
    drafts, nd, ml = _run(tokens, lengths, n_min, n_max, K)
    ref = oracle.ngram_draft(np.asarray(tokens, dtype=np.int32), np.asarray(lengths, dtype=np.int32),
                             n_min, n_max, K)
    np.testing.assert_array_equal(nd, ref["n_drafts"])
    np.testing.assert_array_equal(ml, ref["match_len"])
    np.testing.assert_array_equal(drafts, ref["drafts"])
    return ref


def test_ngram_random_small_alphabet():
    rng = np.random.default_rng(3)
    for trial in range(30):
        B = int(rng.integers(1, 40))
        Lmax = int(rng.integers(1, 300))
        toks = rng.integers(0, int(rng.integers(2, 7)), size=(B, Lmax)).astype(np.int32)
        lengths = rng.integers(0, Lmax + 1, size=B).astype(np.int32)
        n_min = int(rng.integers(1, 5))
        n_max = n_min + int(rng.integers(0, 6))
        K = int(rng.integers(0, 12))
        _check(toks, lengths, n_min, n_max, K)
    assert sv.spec_get_status() == 0


def test_ngram_long_histories_span_several_chunks():
    # 4096 candidate ends per CTA: these rows span up to 6 CTAs, and the best
    # match must win across them (longest first, then latest)
    h = wl.make_ngram_histories(24, 23000, V=64, seed=5, copy_prob=0.6)
    for n_min, n_max, K in ((1, 4, 8), (3, 8, 16), (2, 2, 5), (6, 32, 64)):
        ref = _check(h["tokens"].numpy(), h["lengths"].numpy(), n_min, n_max, K)
    assert (ref["n_drafts"] > 0).any()


def test_ngram_edge_cases_and_bad_lengths():
    toks = np.array([[7, 7, 7, 7, 7, 7, 7, 7],
                     [1, 2, 3, 1, 2, 3, 1, 2],
                     [5, 0, 0, 0, 0, 0, 0, 0],
                     [1, 2, 1, 2, 0, 0, 0, 0],
                     [3, 3, 0, 0, 0, 0, 0, 0],
                     [9, 9, 9, 9, 9, 9, 9, 9]], dtype=np.int32)
    lengths = np.array([8, 8, 1, 4, 0, 9], dtype=np.int32)  # the last is past the row: bad
    for n_min, n_max, K in ((1, 1, 3), (1, 3, 0), (2, 3, 5), (4, 8, 2), (1, 32, 4096)):
        drafts, nd, ml = _run(toks, lengths, n_min, n_max, K)
        ref = oracle.ngram_draft(toks, lengths, n_min, n_max, K)
        np.testing.assert_array_equal(nd, ref["n_drafts"])
        np.testing.assert_array_equal(ml, ref["match_len"])
        np.testing.assert_array_equal(drafts, ref["drafts"])
        assert nd[5] == -1 and ml[5] == -1
        assert sv.spec_get_status() & sv.SPEC_FLAG_BAD_DATA
    assert sv.spec_get_status() == 0


def test_ngram_full_size_repetitive_workload():
    # B = 256 histories of up to 16384 tokens over a 128256-token vocabulary
    h = wl.make_ngram_histories(256, 16384, seed=1)
    ref = _check(h["tokens"].numpy(), h["lengths"].numpy(), 1, 4, 8)
    assert (ref["match_len"] == 4).mean() > 0.3  # copies make long matches common
    _check(h["tokens"].numpy(), h["lengths"].numpy(), 2, 16, 32)
    assert sv.spec_get_status() == 0


def test_ngram_rejects_bad_arguments():
    t = torch.zeros((2, 8), dtype=torch.int32, device=DEV)
    ln = torch.full((2,), 8, dtype=torch.int32, device=DEV)
    for n_min, n_max, K in ((0, 2, 4), (3, 2, 4), (1, 33, 4), (1, 2, -1), (1, 2, 4097)):
        with pytest.raises(sv.SpecError):
            sv.spec_ngram_draft(t, ln, n_min, n_max, K)


def test_ngram_timed_workload_whole_batch():
    """The timed workload (256 histories of up to 131072 tokens, 32 chunks per
    sequence, about 13 chunks claimed per scan CTA), every sequence against
    the oracle, twice in a row (fresh scratch and claim counter each call)."""
    h = wl.make_ngram_histories(16, 131072, seed=1)
    tok = h["tokens"].repeat(16, 1)
    ln = h["lengths"].repeat(16)
    ref = oracle.ngram_draft(tok.numpy(), ln.numpy(), 1, 4, 8)
    for _ in range(2):
        drafts, nd, ml = _run(tok, ln, 1, 4, 8)
        np.testing.assert_array_equal(nd, ref["n_drafts"])
        np.testing.assert_array_equal(ml, ref["match_len"])
        np.testing.assert_array_equal(drafts, ref["drafts"])
    assert sv.spec_get_status() == 0


def test_ngram_rows_off_16_byte_boundaries():
    """Rows that cannot take bulk copies are staged with plain loads: a stride
    that is not a multiple of 4 tokens, and a base pointer 4 bytes past a
    16-byte boundary, both over histories of several chunks."""
    h = wl.make_ngram_histories(12, 23001, V=40, seed=8, copy_prob=0.6)
    _check(h["tokens"].numpy(), h["lengths"].numpy(), 2, 6, 9)
    h = wl.make_ngram_histories(12, 23000, V=40, seed=9, copy_prob=0.6)
    B, S = h["tokens"].shape
    flat = torch.zeros(B * S + 1, dtype=torch.int32, device=DEV)
    t = flat[1:].view(B, S)
    t.copy_(h["tokens"].to(DEV))
    assert t.data_ptr() % 16 == 4
    ln = h["lengths"].to(DEV)
    drafts, nd, ml = sv.spec_ngram_draft(t, ln, 1, 5, 7)
    torch.cuda.synchronize()
    ref = oracle.ngram_draft(h["tokens"].numpy(), h["lengths"].numpy(), 1, 5, 7)
    np.testing.assert_array_equal(nd.cpu().numpy(), ref["n_drafts"])
    np.testing.assert_array_equal(ml.cpu().numpy(), ref["match_len"])
    np.testing.assert_array_equal(drafts.cpu().numpy(), ref["drafts"])
    assert sv.spec_get_status() == 0


def test_ngram_match_at_every_chunk_boundary():
    """Histories whose only earlier occurrence of the suffix straddles a
    4096-token chunk boundary (the match's tokens sit in the halo staged
    before the chunk), at each boundary of a 5-chunk row."""
    S, n = 5 * 4096, 6
    for boundary in range(4096, S, 4096):
        for shift in (-3, 0, 1, 4):
            row = np.arange(S, dtype=np.int32) + 1000  # all distinct
            suffix = np.array([7, 8, 9, 10, 11, 12], dtype=np.int32)
            e = boundary + shift  # the occurrence ends at e (exclusive)
            row[e - n:e] = suffix
            L = S - 5
            row[L - n:L] = suffix
            ref = _check(row[None, :], np.array([L], dtype=np.int32), 1, 8, 5)
            assert ref["match_len"][0] == n and ref["drafts"][0, 0] == row[e]


def test_ngram_two_full_grids_side_by_side():
    """Two timed-workload calls on two streams at once: each persistent scan
    grid is sized to the whole device, so each starts with only part of it
    resident beside the other.  No scan CTA waits for another (entries are
    claimed from a counter), so both finish with no expired wait and with
    the results of the same calls made alone."""
    hs = [wl.make_ngram_histories(16, 131072, seed=s) for s in (1, 2)]
    xs = [(h["tokens"].repeat(16, 1).to(DEV), h["lengths"].repeat(16).to(DEV)) for h in hs]
    alone = [sv.spec_ngram_draft(t, ln, 1, 4, 8) for t, ln in xs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(device=DEV) for _ in range(2)]
    for _ in range(3):
        got = []
        for (t, ln), s in zip(xs, streams):
            with torch.cuda.stream(s):
                got.append(sv.spec_ngram_draft(t, ln, 1, 4, 8, stream=s))
        torch.cuda.synchronize()
        assert sv.spec_get_status() == 0
        for g, a in zip(got, alone):
            for x, y in zip(g, a):
                assert torch.equal(x, y)
