"""Output guards and an injected allocation failure on the GPU.

Every output buffer is surrounded by canary words: a call must write its
outputs and nothing next to them.  A scratch allocation that fails (forced
through the library's test hook) must return SPEC_ERR_CUDA without touching
the outputs, and the next call must work."""
import ctypes

import numpy as np
import pytest
import torch

import speculative_decoding_verification_36_gb300 as sv
from speculative_decoding_verification_36_gb300 import _lib
from speculative_decoding_verification_36_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
G = 64  # guard elements on each side
CANARY_I = 0x5A5A1234
CANARY_F = -12345.25


class Guarded:
    """An output tensor with canary words on both sides."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape)) if len(shape) else 1
        self.buf = torch.empty(n + 2 * G, dtype=dtype, device=DEV)
        self.fill = CANARY_I if dtype in (torch.int32, torch.int64) else CANARY_F
        self.buf.fill_(self.fill)
        self.t = self.buf[G:G + n].view(shape)

    def intact(self):
        b = self.buf.cpu()
        return bool((b[:G] == self.fill).all() and (b[-G:] == self.fill).all())


def _chain(name, **over):
    p = wl.preset(name, **over)
    x = wl.make_chain(p, device=DEV, seed=2)
    return p, x


def test_chain_outputs_are_guarded():
    for name, over in (("c2", dict(B=5, K=5, V=1000)), ("c1", dict(B=3, K=2, V=257)), ("c4", dict(B=7, V=999))):
        p, x = _chain(name, **over)
        tok, n = Guarded((p.B, p.K + 1), torch.int32), Guarded((p.B,), torch.int32)
        sv.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 1, out_tokens=tok.t, out_n_accepted=n.t)
        # the early exit (sampled, or greedy at temperature 0)
        tok2, n2 = Guarded((p.B, p.K + 1), torch.int32), Guarded((p.B,), torch.int32)
        sv.spec_verify_early_exit(x["target"], x["draft"], x["tokens"], p.temperature, 1,
                                  out_tokens=tok2.t, out_n_accepted=n2.t)
        torch.cuda.synchronize()
        assert tok2.intact() and n2.intact()
        assert torch.equal(tok.t, tok2.t)
        assert tok.intact() and n.intact(), name
        assert (n.t >= 0).all()
    assert sv.spec_get_status() == 0


def test_stats_outputs_are_guarded():
    p, x = _chain("c2", B=4, K=3, V=2048)
    B, K, R = p.B, p.K, 2 * p.K + 1
    outs = dict(tok=Guarded((B, K + 1), torch.int32), n=Guarded((B,), torch.int32),
                rs=Guarded((B, R, 2), torch.float32), pq=Guarded((B, K, 2), torch.float32),
                res=Guarded((B,), torch.float32), ent=Guarded((B, R), torch.float32))
    lib = _lib.load()
    with torch.cuda.device(DEV):
        _lib.check(lib.spec_verify_stats_bf16(
            x["target"].data_ptr(), x["draft"].data_ptr(), x["tokens"].data_ptr(), B, K, p.V,
            ctypes.c_float(p.temperature), 1, outs["tok"].t.data_ptr(), outs["n"].t.data_ptr(),
            outs["rs"].t.data_ptr(), outs["pq"].t.data_ptr(), outs["res"].t.data_ptr(),
            outs["ent"].t.data_ptr(), torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    for k, g in outs.items():
        assert g.intact(), k


def test_tree_and_ngram_outputs_are_guarded():
    tr = wl.make_tree(wl.preset("c5", B=3, V=777), device=DEV, seed=5)
    B, N = 3, tr["tokens"].shape[1]
    path, ln, mask = Guarded((B, N + 1), torch.int32), Guarded((B,), torch.int32), Guarded((B, N, 1), torch.int32)
    for ee in (False, True):
        sv.spec_tree_verify_greedy(tr["target"], tr["tokens"], tr["parents"], out_path=path.t, out_len=ln.t,
                                   out_mask=mask.t, early_exit=ee)
        torch.cuda.synchronize()
        assert path.intact() and ln.intact() and mask.intact()
    h = wl.make_ngram_histories(6, 5000, V=50, seed=3)
    d, nd, ml = Guarded((6, 7), torch.int32), Guarded((6,), torch.int32), Guarded((6,), torch.int32)
    sv.spec_ngram_draft(h["tokens"].to(DEV), h["lengths"].to(DEV), 1, 5, 7, out_drafts=d.t, out_n_drafts=nd.t,
                        out_match_len=ml.t)
    torch.cuda.synchronize()
    assert d.intact() and nd.intact() and ml.intact()
    assert sv.spec_get_status() == 0


def test_a_failed_scratch_allocation_is_reported_and_harmless():
    lib = _lib.load()
    p, x = _chain("c2", B=6, K=4, V=3000)
    ref_tok, ref_n = sv.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 9)
    torch.cuda.synchronize()
    tok, n = Guarded((p.B, p.K + 1), torch.int32), Guarded((p.B,), torch.int32)
    assert lib.spec_test_fail_allocations(1) == 0
    with pytest.raises(sv.SpecError) as err:
        sv.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 9, out_tokens=tok.t,
                       out_n_accepted=n.t)
    assert "failed on request" in str(err.value)
    torch.cuda.synchronize()
    # nothing was launched: the outputs keep their canary fill
    assert (tok.buf.cpu() == CANARY_I).all() and (n.buf.cpu() == CANARY_I).all()
    # the next call allocates normally and gives the same result as before
    sv.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 9, out_tokens=tok.t, out_n_accepted=n.t)
    torch.cuda.synchronize()
    assert torch.equal(tok.t, ref_tok) and torch.equal(n.t, ref_n) and tok.intact()
    assert lib.spec_test_fail_allocations(0) == 0
    assert sv.spec_get_status() == 0


def test_concurrent_calls_from_two_host_threads():
    """Two host threads, each on its own stream, call the sampled verify, the
    early exit and the tree verify back to back at the same time (the binding
    releases the GIL inside the library).  Every result equals the same call
    made alone: the scratch pool, the shared side stream and the device state
    are safe under concurrent callers, and concurrent persistent launches
    make progress."""
    import threading
    chains = [_chain("c2", B=8, K=4, V=5000 + 100 * k) for k in range(2)]
    tr = wl.make_tree(wl.preset("c5", B=4, depth=3, V=3000), device=DEV, seed=9)
    want = []
    for (p, x) in chains:
        a = sv.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 5)
        e = sv.spec_verify_early_exit(x["target"], x["draft"], x["tokens"], p.temperature, 5)
        want.append((a, e))
    wt = sv.spec_tree_verify_greedy(tr["target"], tr["tokens"], tr["parents"])
    torch.cuda.synchronize()
    errors = []

    def worker(k):
        try:
            p, x = chains[k]
            s = torch.cuda.Stream(device=DEV)
            with torch.cuda.stream(s):
                for _ in range(40):
                    a = sv.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 5)
                    e = sv.spec_verify_early_exit(x["target"], x["draft"], x["tokens"], p.temperature, 5)
                    t = sv.spec_tree_verify_greedy(tr["target"], tr["tokens"], tr["parents"])
                    s.synchronize()
                    for got, ref in ((a, want[k][0]), (e, want[k][1]), (t, wt)):
                        if not all(torch.equal(g, r) for g, r in zip(got, ref)):
                            errors.append(k)
                            return
        except Exception as exc:  # reported below
            errors.append(repr(exc))

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=300)
    assert not errors, errors
    assert sv.spec_get_status() == 0


def test_every_bounded_wait_gives_up_on_a_slot_nothing_writes():
    """Each bounded-wait helper of the kernels, run on a slot that nothing
    writes under a lowered limit, gives up and flags SPEC_FLAG_TIMEOUT (the
    decision read also reports no decision); on a slot already written none
    flags anything.  The device status word is untouched and the next call
    works."""
    try:
        sv.spec_test_spin_limit(2000)
        expired, written = sv.spec_test_wait_probe()
    finally:
        sv.spec_test_spin_limit(0)
    assert expired == 0x7F, hex(expired)
    assert written == 0, hex(written)
    assert sv.spec_get_status() == 0
    p, x = _chain("c2", B=4, K=3, V=3000)
    a = sv.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 2)
    torch.cuda.synchronize()
    assert (a[1] >= 0).all() and sv.spec_get_status() == 0


def test_a_lowered_wait_limit_never_hangs_or_writes_out_of_place():
    """A full-width sampled verify with every wait limited to one poll (most of
    its waits find their slot already written, so whether one runs out depends
    on timing) returns; if a wait ran out the status word says so (and a row
    left without statistics is reported as bad data), and in any
    case nothing is written outside the outputs or out of range, and a call
    that flagged nothing gives the normal result.  With the default limit back
    the next call matches the oracle."""
    import oracle
    from parity import chain_report
    p, x = _chain("c3", B=64)
    want_t, want_n = sv.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 4)
    torch.cuda.synchronize()
    tok, n = Guarded((p.B, p.K + 1), torch.int32), Guarded((p.B,), torch.int32)
    assert sv.spec_get_status() == 0
    try:
        sv.spec_test_spin_limit(1)
        for _ in range(3):
            sv.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 4, out_tokens=tok.t,
                           out_n_accepted=n.t)
            torch.cuda.synchronize()
            status = sv.spec_get_status()
            # an expired wait on a row's partials leaves the row without
            # statistics, which is also reported as bad data
            assert status in (0, sv.SPEC_FLAG_TIMEOUT, sv.SPEC_FLAG_TIMEOUT | sv.SPEC_FLAG_BAD_DATA), status
            assert tok.intact() and n.intact()
            # a sequence whose commit was given up keeps its previous value
            nn, tt = n.t.cpu().numpy(), tok.t.cpu().numpy()
            assert (((nn >= -1) & (nn <= p.K)) | (nn == CANARY_I)).all()
            assert (((tt >= -1) & (tt < p.V)) | (tt == CANARY_I)).all()
            if status == 0:
                assert torch.equal(tok.t, want_t) and torch.equal(n.t, want_n)
    finally:
        sv.spec_test_spin_limit(0)
    tokens, n2 = sv.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 4)
    torch.cuda.synchronize()
    assert sv.spec_get_status() == 0
    assert torch.equal(tokens, want_t) and torch.equal(n2, want_n)
    sel = [0, 17, 40, 63]
    idx = torch.tensor(sel)
    ref = oracle.spec_verify(x["target"][idx].cpu(), x["draft"][idx].cpu(), x["tokens"][idx].cpu(),
                             p.temperature, 4, seq_ids=sel)
    rep = chain_report(tokens.cpu().numpy()[sel], n2.cpu().numpy()[sel], ref)
    assert not rep["mismatch"], rep


def test_ngram_lowered_wait_limit_returns_and_flags_only_timeouts():
    """N-gram drafting with every stage wait limited to one poll: the scan's
    consumers may give up on a stage whose bulk copy is still landing; the
    call still returns (the producer drains its copies with its own limit),
    flags at most a timeout, writes nothing out of place and only values a
    history holds (a chunk left unscanned reads as no match).  With the
    default limit back the next call matches the oracle."""
    import oracle
    h = wl.make_ngram_histories(64, 40000, V=50, seed=12, copy_prob=0.6)
    tok, ln = h["tokens"].to(DEV), h["lengths"].to(DEV)
    B, K = tok.shape[0], 9
    d, nd, ml = Guarded((B, K), torch.int32), Guarded((B,), torch.int32), Guarded((B,), torch.int32)
    assert sv.spec_get_status() == 0
    try:
        sv.spec_test_spin_limit(1)
        for _ in range(3):
            sv.spec_ngram_draft(tok, ln, 1, 6, K, out_drafts=d.t, out_n_drafts=nd.t, out_match_len=ml.t)
            torch.cuda.synchronize()
            status = sv.spec_get_status()
            assert status in (0, sv.SPEC_FLAG_TIMEOUT), status
            assert d.intact() and nd.intact() and ml.intact()
            n_, m_, d_ = nd.t.cpu().numpy(), ml.t.cpu().numpy(), d.t.cpu().numpy()
            assert ((n_ >= 0) & (n_ <= K)).all() and ((m_ == 0) | ((m_ >= 1) & (m_ <= 6))).all()
            assert ((d_ >= -1) & (d_ < 50)).all()
    finally:
        sv.spec_test_spin_limit(0)
    drafts, nd2, ml2 = sv.spec_ngram_draft(tok, ln, 1, 6, K)
    torch.cuda.synchronize()
    assert sv.spec_get_status() == 0
    ref = oracle.ngram_draft(h["tokens"].numpy(), h["lengths"].numpy(), 1, 6, K)
    np.testing.assert_array_equal(nd2.cpu().numpy(), ref["n_drafts"])
    np.testing.assert_array_equal(ml2.cpu().numpy(), ref["match_len"])
    np.testing.assert_array_equal(drafts.cpu().numpy(), ref["drafts"])


def test_two_full_capacity_launches_side_by_side():
    """Two full-size c3 verifies (B=256, grids sized to the whole device) on
    two streams at once: each launch starts with only part of its grid
    resident, beside the other.  Work goes only to CTAs that have started
    (each CTA's first claims follow a per-launch ticket), so both finish
    with no expired wait and with the results of the same calls made alone."""
    p = wl.preset("c3")
    xs = [wl.make_chain(p, device=DEV, seed=40 + k) for k in range(2)]
    want = []
    for k, x in enumerate(xs):
        want.append(sv.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 100 + k))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(device=DEV) for _ in range(2)]
    for rnd in range(5):
        got = []
        for k, (x, s) in enumerate(zip(xs, streams)):
            with torch.cuda.stream(s):
                got.append(sv.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 100 + k))
        torch.cuda.synchronize()
        assert sv.spec_get_status() == 0, rnd
        for k in range(2):
            assert torch.equal(got[k][0], want[k][0]) and torch.equal(got[k][1], want[k][1]), (rnd, k)
