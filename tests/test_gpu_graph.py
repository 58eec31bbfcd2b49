"""Stream capture: the verify calls can be captured into a CUDA graph (the
scratch then comes from graph memory nodes and is filled on the captured
stream) and replayed over new inputs copied into the same buffers."""
import pytest
import torch

import speculative_decoding_verification_36_gb300 as sv
from speculative_decoding_verification_36_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.mark.parametrize("name,over", [("c1", {}), ("c2", dict(B=16, V=20000)), ("c4", dict(B=32, V=20000))])
def test_captured_verify_replays_like_eager_calls(name, over):
    p = wl.preset(name, **over)
    sets = [wl.make_chain(p, device=DEV, seed=s) for s in range(3)]
    x0 = sets[0]
    tgt = x0["target"].clone()
    drf = x0["draft"].clone() if x0["draft"] is not None else None
    tok = x0["tokens"].clone()
    seed = 31
    # an eager call first: it creates the library's per-device state and pool
    sv.spec_verify(tgt, drf, tok, p.temperature, seed)
    sv.spec_verify_early_exit(tgt, drf, tok, p.temperature, seed)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out_t, out_n = sv.spec_verify(tgt, drf, tok, p.temperature, seed)
        ee_t, ee_n = sv.spec_verify_early_exit(tgt, drf, tok, p.temperature, seed)
    for x in sets:
        tgt.copy_(x["target"])
        if drf is not None:
            drf.copy_(x["draft"])
        tok.copy_(x["tokens"])
        g.replay()
        ref_t, ref_n = sv.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, seed)
        torch.cuda.synchronize()
        assert torch.equal(out_t, ref_t) and torch.equal(out_n, ref_n)
        assert torch.equal(ee_t, ref_t) and torch.equal(ee_n, ref_n)
    assert sv.spec_get_status() == 0


def test_captured_tree_verify_replays_like_eager_calls():
    tp = wl.preset("c5", B=8, depth=3, V=10000)
    sets = [wl.make_tree(tp, device=DEV, seed=s) for s in range(3)]
    tgt, tok, par = (sets[0][k].clone() for k in ("target", "tokens", "parents"))
    sv.spec_tree_verify_greedy(tgt, tok, par)
    sv.spec_tree_verify_greedy(tgt, tok, par, early_exit=True)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = sv.spec_tree_verify_greedy(tgt, tok, par)
        out_e = sv.spec_tree_verify_greedy(tgt, tok, par, early_exit=True)
    for x in sets:
        tgt.copy_(x["target"])
        tok.copy_(x["tokens"])
        par.copy_(x["parents"])
        g.replay()
        ref = sv.spec_tree_verify_greedy(x["target"], x["tokens"], x["parents"])
        torch.cuda.synchronize()
        for a, b, c in zip(out, out_e, ref):
            assert torch.equal(a, c) and torch.equal(b, c)
    assert sv.spec_get_status() == 0


def test_captured_ngram_drafting_replays_like_eager_calls():
    """The scan and the finishing launch (programmatic stream serialisation)
    captured together, replayed over new histories."""
    sets = [wl.make_ngram_histories(24, 9000, V=60, seed=s, copy_prob=0.6) for s in range(3)]
    tok = sets[0]["tokens"].to(DEV)
    ln = sets[0]["lengths"].to(DEV)
    sv.spec_ngram_draft(tok, ln, 1, 6, 7)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = sv.spec_ngram_draft(tok, ln, 1, 6, 7)
    for h in sets:
        tok.copy_(h["tokens"].to(DEV))
        ln.copy_(h["lengths"].to(DEV))
        g.replay()
        ref = sv.spec_ngram_draft(h["tokens"].to(DEV), h["lengths"].to(DEV), 1, 6, 7)
        torch.cuda.synchronize()
        for a, b in zip(out, ref):
            assert torch.equal(a, b)
    assert sv.spec_get_status() == 0


def test_captured_stochastic_tree_replays_like_eager_calls():
    """The statistics launch and the walk's cluster launch (programmatically
    dependent on it) captured together, replayed over new trees."""
    tp = wl.preset("c5", B=6, depth=3, V=6000)
    sets = [wl.make_tree_sampling(tp, 1.0, device=DEV, seed=s) for s in range(3)]
    tgt, drf, tok, par = (sets[0][k].clone() for k in ("target", "draft", "tokens", "parents"))
    sv.spec_tree_verify_sampling(tgt, drf, tok, par, 1.0, 7)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = sv.spec_tree_verify_sampling(tgt, drf, tok, par, 1.0, 7)
    for x in sets:
        for buf, k in ((tgt, "target"), (drf, "draft"), (tok, "tokens"), (par, "parents")):
            buf.copy_(x[k])
        g.replay()
        ref = sv.spec_tree_verify_sampling(x["target"], x["draft"], x["tokens"], x["parents"], 1.0, 7)
        torch.cuda.synchronize()
        for a, b in zip(out, ref):
            assert torch.equal(a, b)
    assert sv.spec_get_status() == 0
