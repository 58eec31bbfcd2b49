"""Comparison helpers for the GPU parity tests (no test functions here).

The CUDA path accumulates softmax sums in fp32; the oracle works in fp64.  A
decision (accept / reject, or which token an inverse CDF lands on) may only
differ where the oracle's own draw lies within 1e-6 of the decision boundary:
|u - min(1, p/q)| < 1e-6 for an acceptance draw, or a distance below 1e-6 * Z
from w * Z to the nearest cumulative sum for a resampling draw.  Such
sequences are counted and reported; every other sequence must match exactly.
"""
from __future__ import annotations

import numpy as np

BOUNDARY = 1e-6


def chain_report(tokens, n, ref):
    """Compare GPU chain outputs with the oracle's.

    Returns dict(mismatch=[...] sequences differing outside the boundary
    window, boundary=[...] sequences differing inside it, boundary_draws=count
    of oracle draws inside the window)."""
    tokens = np.asarray(tokens)
    n = np.asarray(n)
    mism, bnd = [], []
    for b in range(len(n)):
        if n[b] == ref["n"][b] and np.array_equal(tokens[b], ref["tokens"][b]):
            continue
        if n[b] != ref["n"][b] and ref["n"][b] >= 0 and n[b] >= 0:
            i = min(int(n[b]), int(ref["n"][b]))
            (bnd if ref["acc_margin"][b, i] < BOUNDARY else mism).append(b)
        elif n[b] == ref["n"][b] and n[b] >= 0 and ref["sample_margin"][b] < BOUNDARY:
            bnd.append(b)
        else:
            mism.append(b)
    am = ref["acc_margin"]
    draws = int(np.sum(am[np.isfinite(am)] < BOUNDARY) +
                np.sum(ref["sample_margin"][np.isfinite(ref["sample_margin"])] < BOUNDARY))
    return dict(mismatch=mism, boundary=bnd, boundary_draws=draws)


def rel_err(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.abs(a - b) / np.maximum(np.abs(b), 1e-300)


def oracle_chain_threads(target, draft, tokens, temperature, seed, threads=None, **kw):
    """oracle.spec_verify over a whole batch, split into chunks that run on
    host threads (the oracle's C code runs without the GIL).  Each chunk
    passes its batch indices as sequence numbers, so the result is that of
    one call over the whole batch.  Inputs may live on any device."""
    import os
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    target, draft, tokens = target.cpu(), draft.cpu(), tokens.cpu()
    B = target.shape[0]
    threads = threads or min(16, os.cpu_count() or 1)
    bounds = np.linspace(0, B, min(B, 4 * threads) + 1).astype(int)
    chunks = [(int(a), int(b)) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]

    def one(c):
        a, b = c
        return oracle.spec_verify(target[a:b], draft[a:b], tokens[a:b], temperature, seed,
                                  seq_ids=np.arange(a, b), **kw)

    with ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(one, chunks))
    return {k: np.concatenate([p[k] for p in parts]) for k in parts[0]}


def oracle_greedy_threads(target, tokens, threads=None, **kw):
    """oracle.spec_verify_greedy over a whole batch on host threads."""
    import os
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    target, tokens = target.cpu(), tokens.cpu()
    B = target.shape[0]
    threads = threads or min(16, os.cpu_count() or 1)
    bounds = np.linspace(0, B, min(B, 4 * threads) + 1).astype(int)
    chunks = [(int(a), int(b)) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]

    def one(c):
        a, b = c
        return oracle.spec_verify_greedy(target[a:b], tokens[a:b], **kw)

    with ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(one, chunks))
    return {k: np.concatenate([p[k] for p in parts]) for k in parts[0]}
