"""fp64 CPU oracle for the speculative-decoding verify step (ctypes binding).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (``speculative_decoding_verification_36_gb300``)
never imports, links or runs it, and the two share no code: the only common
Python module is the seeded input generator, which holds none of the method's
arithmetic.

The arithmetic lives in ``spec_oracle.c`` (plain C, fp64, single-threaded);
this module only compiles it with gcc on first use and marshals arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

DTYPE_F32 = 0
DTYPE_BF16 = 1


def build(force: bool = False) -> str:
    """Compile ``spec_oracle.c`` into ``_build/liboracle.so`` (plain -O2)."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            os.makedirs(_BUILD_DIR, exist_ok=True)
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                                   "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    i32, i64, u64, f64 = ctypes.c_int, ctypes.c_longlong, ctypes.c_uint64, ctypes.c_double
    lib.oracle_philox4x64_10.argtypes = [P, P, P]
    lib.oracle_philox4x64_10.restype = None
    lib.oracle_uniform.argtypes = [u64, u64, u64, u64]
    lib.oracle_uniform.restype = f64
    lib.oracle_spec_verify.argtypes = [P, P, i32, i64, i64, P, i64, i32, i32, i32, f64, u64, P, i32,
                                       P, P, P, P, P, P, P, P, P, P, P, P, P]
    lib.oracle_spec_verify.restype = i32
    lib.oracle_spec_verify_greedy.argtypes = [P, i32, i64, P, i64, i32, i32, i32, i32, P, P, P]
    lib.oracle_spec_verify_greedy.restype = i32
    lib.oracle_tree_verify_greedy.argtypes = [P, i32, P, P, i32, i32, i32, i32, P, P, P]
    lib.oracle_tree_verify_greedy.restype = i32
    lib.oracle_acceptance_stats.argtypes = [P, i32, i32, P, P, P]
    lib.oracle_acceptance_stats.restype = None
    lib.oracle_row_entropy.argtypes = [P, i32, i64, i32, f64, P]
    lib.oracle_row_entropy.restype = None
    lib.oracle_adaptive_k.argtypes = [P, P, i32, i32, f64, f64, i32, i32, P, P]
    lib.oracle_adaptive_k.restype = None
    lib.oracle_tree_verify_sampling.argtypes = [P, P, i32, P, P, i32, i32, i32, f64, u64, P, P, P]
    lib.oracle_tree_verify_sampling.restype = i32
    lib.oracle_ngram_draft.argtypes = [P, i64, P, i32, i32, i32, i32, P, P, P]
    lib.oracle_ngram_draft.restype = i32
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _as_logits(x):
    """Return (contiguous numpy array of raw bits/values, dtype code).

    Accepts numpy float32 arrays, numpy uint16 arrays holding bfloat16 bits, or
    CPU torch tensors of dtype float32 / bfloat16 (copied bit-exactly)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), DTYPE_BF16
            if x.dtype == torch.float32:
                return x.numpy(), DTYPE_F32
            raise TypeError(f"unsupported logits dtype {x.dtype}")
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, DTYPE_F32
    if x.dtype == np.uint16:
        return x, DTYPE_BF16
    raise TypeError(f"unsupported logits dtype {x.dtype}")


def _as_i32(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().to(torch.int32).contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x, dtype=np.int32)


def philox4x64_10(counter, key):
    """Raw Philox-4x64-10 block for a 4-word counter and a 2-word key."""
    lib = _load()
    c = np.ascontiguousarray(counter, dtype=np.uint64)
    k = np.ascontiguousarray(key, dtype=np.uint64)
    out = np.zeros(4, dtype=np.uint64)
    lib.oracle_philox4x64_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, b: int, position: int, stream: int) -> float:
    """The verify step's uniform draw for (seed, sequence, position, stream)."""
    return _load().oracle_uniform(seed, b, position, stream)


def spec_verify(target, draft, draft_tokens, temperature: float, seed: int,
                broadcast: bool = False, n_seq: int | None = None, seq_ids=None,
                used_rows_only: bool = False):
    """Speculative-sampling verification of a batch (temperature > 0).

    target: [B, K+1, V]; draft: [B, K, V]; draft_tokens: [B, K].  With
    ``broadcast=True`` target/draft hold ONE sequence ([K+1, V], [K, V]) that
    is shared by all ``n_seq`` batch entries (each entry still draws its own
    uniforms through its batch index).  ``seq_ids`` (optional, [B]) gives the
    sequence number each batch entry draws its uniforms with, so that a subset
    of a larger batch reproduces that batch's draws.  ``used_rows_only``
    checks for bad data only the rows the result depends on (positions 0..n,
    and target row K when every draft is accepted), as the early-exit verify
    does.  Returns a dict of numpy arrays:
    tokens [B, K+1], n [B] and the per-sequence diagnostics documented in
    spec_oracle.c.
    """
    lib = _load()
    t, dt = _as_logits(target)
    d, dd = _as_logits(draft)
    if dt != dd:
        raise TypeError("target and draft logits must share a dtype")
    x = _as_i32(draft_tokens)
    if broadcast:
        K1, V = t.shape[-2], t.shape[-1]
        K = K1 - 1
        B = int(n_seq if n_seq is not None else x.shape[0])
        t_stride, d_stride = 0, 0
    else:
        B, K1, V = t.shape
        K = K1 - 1
        t_stride, d_stride = K1 * V, K * V
    if x.ndim == 1:
        x = x.reshape(1, -1)
    tok_stride = 0 if x.shape[0] == 1 and B > 1 else K
    R = 2 * K + 1
    out = dict(
        tokens=np.full((B, K + 1), -1, dtype=np.int32),
        n=np.zeros(B, dtype=np.int32),
        row_logmax=np.zeros((B, R)), row_sum=np.zeros((B, R)),
        px=np.zeros((B, K)), qx=np.zeros((B, K)), u=np.zeros((B, K)),
        acc_margin=np.zeros((B, K)),
        resid_mass=np.zeros(B), theta=np.zeros(B), w=np.zeros(B),
        sample_margin=np.zeros(B), degenerate=np.zeros(B, dtype=np.int32),
    )
    # keep a valid pointer even when K == 0 (empty draft array)
    d_buf = d if d.size else np.zeros(1, dtype=d.dtype)
    x_buf = x if x.size else np.zeros(1, dtype=np.int32)
    ids = None
    if seq_ids is not None:
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64).reshape(-1))
        if ids.shape[0] != B:
            raise ValueError("seq_ids must have one entry per sequence")
    rc = lib.oracle_spec_verify(
        _ptr(t), _ptr(d_buf), dt, t_stride, d_stride, _ptr(x_buf), tok_stride,
        B, K, V, float(temperature), int(seed) & (2**64 - 1),
        _ptr(ids) if ids is not None else None, int(bool(used_rows_only)),
        _ptr(out["tokens"]), _ptr(out["n"]), _ptr(out["row_logmax"]), _ptr(out["row_sum"]),
        _ptr(out["px"]), _ptr(out["qx"]), _ptr(out["u"]), _ptr(out["acc_margin"]),
        _ptr(out["resid_mass"]), _ptr(out["theta"]), _ptr(out["w"]),
        _ptr(out["sample_margin"]), _ptr(out["degenerate"]))
    if rc != 0:
        raise MemoryError("oracle_spec_verify failed to allocate")
    return out


def spec_verify_greedy(target, draft_tokens, used_rows_only: bool = False):
    """Greedy verification (temperature 0).  target [B, K+1, V]; tokens [B, K].
    ``used_rows_only`` checks for bad data only what the result depends on,
    in position order (rows 0..n, tokens x_0..x_n, row K when all match), as
    the early-exit verify does."""
    lib = _load()
    t, dt = _as_logits(target)
    x = _as_i32(draft_tokens)
    B, K1, V = t.shape
    K = K1 - 1
    x_buf = x if x.size else np.zeros(1, dtype=np.int32)
    tokens = np.full((B, K1), -1, dtype=np.int32)
    n = np.zeros(B, dtype=np.int32)
    argmax = np.zeros((B, K1), dtype=np.int32)
    lib.oracle_spec_verify_greedy(_ptr(t), dt, K1 * V, _ptr(x_buf), K, B, K, V, int(bool(used_rows_only)),
                                  _ptr(tokens), _ptr(n), _ptr(argmax))
    return dict(tokens=tokens, n=n, row_argmax=argmax)


def tree_verify_greedy(target, tree_tokens, parent_idx, used_rows_only: bool = False):
    """Greedy tree verification.  target [B, N+1, V]; tokens, parents [B, N].
    ``used_rows_only`` checks for bad data only what the result depends on
    (every parent index, the root's row, the tokens of nodes whose parent is
    accepted and the rows of accepted nodes), as the early-exit verify does."""
    lib = _load()
    t, dt = _as_logits(target)
    tok = _as_i32(tree_tokens)
    par = _as_i32(parent_idx)
    B, N1, V = t.shape
    N = N1 - 1
    W = (N + 31) // 32
    path = np.full((B, N1), -1, dtype=np.int32)
    length = np.zeros(B, dtype=np.int32)
    mask = np.zeros((B, N, max(W, 0)), dtype=np.uint32)
    tok_buf = tok if tok.size else np.zeros(1, dtype=np.int32)
    par_buf = par if par.size else np.zeros(1, dtype=np.int32)
    mask_buf = mask if mask.size else np.zeros(1, dtype=np.uint32)
    rc = lib.oracle_tree_verify_greedy(_ptr(t), dt, _ptr(tok_buf), _ptr(par_buf), B, N, V,
                                       int(bool(used_rows_only)), _ptr(path), _ptr(length), _ptr(mask_buf))
    if rc != 0:
        raise MemoryError("oracle_tree_verify_greedy failed to allocate")
    return dict(path=path, length=length, mask=mask)


def acceptance_stats(n_accepted, K: int):
    """Histogram of accepted counts, per-position acceptance rate and mean
    tokens per iteration.  n_accepted [B] int32 (-1 marks a bad sequence)."""
    lib = _load()
    n = np.ascontiguousarray(np.asarray(n_accepted, dtype=np.int32).reshape(-1))
    hist = np.zeros(K + 2, dtype=np.uint64)
    alpha = np.zeros(max(K, 1), dtype=np.float64)
    mean = np.zeros(1, dtype=np.float64)
    n_buf = n if n.size else np.zeros(1, dtype=np.int32)
    lib.oracle_acceptance_stats(_ptr(n_buf), int(n.size), int(K), _ptr(hist), _ptr(alpha), _ptr(mean))
    return dict(hist=hist, alpha=alpha[:K], mean_tokens=float(mean[0]))


def row_entropy(logits, temperature: float):
    """Entropy (nats) of softmax(logits / temperature) along the last axis;
    the leading axes are kept.  NaN for a bad row."""
    lib = _load()
    t, dt = _as_logits(logits)
    shape = t.shape[:-1]
    V = t.shape[-1]
    rows = int(np.prod(shape)) if len(shape) else 1
    out = np.zeros(max(rows, 1), dtype=np.float64)
    t_buf = t if t.size else np.zeros(1, dtype=t.dtype)
    lib.oracle_row_entropy(_ptr(t_buf), dt, rows, V, float(temperature), _ptr(out))
    return out[:rows].reshape(shape)


def adaptive_k(target_entropy, n_accepted, K: int, h_lo: float, h_hi: float, k_min: int, k_max: int):
    """Suggested next draft length per sequence from the mean entropy of the
    target rows 0..n the iteration consulted.  target_entropy [B, K+1] (nats),
    n_accepted [B] (-1: bad).  Returns dict(k_next [B] int32 (-1 for a bad
    sequence), mean_entropy [B] float64)."""
    if not (0 <= k_min <= k_max) or not (h_lo <= h_hi):
        raise ValueError("need 0 <= k_min <= k_max and h_lo <= h_hi")
    lib = _load()
    h = np.ascontiguousarray(np.asarray(target_entropy, dtype=np.float64))
    n = np.ascontiguousarray(np.asarray(n_accepted, dtype=np.int32).reshape(-1))
    B = n.size
    if h.shape != (B, K + 1):
        raise ValueError(f"target_entropy must be [B, K+1] = [{B}, {K + 1}]")
    k_next = np.zeros(max(B, 1), dtype=np.int32)
    hmean = np.zeros(max(B, 1), dtype=np.float64)
    h_buf = h if h.size else np.zeros(1, dtype=np.float64)
    n_buf = n if n.size else np.zeros(1, dtype=np.int32)
    lib.oracle_adaptive_k(_ptr(h_buf), _ptr(n_buf), int(B), int(K), float(h_lo), float(h_hi), int(k_min),
                          int(k_max), _ptr(k_next), _ptr(hmean))
    return dict(k_next=k_next[:B], mean_entropy=hmean[:B])


def tree_verify_sampling(target, draft, tree_tokens, parent_idx, temperature: float, seed: int):
    """Stochastic verification of a token tree.  target, draft [B, N+1, V];
    tokens, parents [B, N].  Returns dict(path [B, N+1], length [B],
    boundary_at [B, N+1] (1 where a draw that decided that path entry lay
    within 1e-6 of its decision boundary), boundary [B] (any of them))."""
    lib = _load()
    t, dt = _as_logits(target)
    d, dd = _as_logits(draft)
    if dd != dt or d.shape != t.shape:
        raise ValueError("target and draft must share dtype and shape")
    tok = _as_i32(tree_tokens)
    par = _as_i32(parent_idx)
    B, N1, V = t.shape
    N = N1 - 1
    path = np.full((B, N1), -1, dtype=np.int32)
    length = np.zeros(B, dtype=np.int32)
    boundary = np.zeros((B, N1), dtype=np.int32)
    tok_buf = tok if tok.size else np.zeros(1, dtype=np.int32)
    par_buf = par if par.size else np.zeros(1, dtype=np.int32)
    rc = lib.oracle_tree_verify_sampling(_ptr(t), _ptr(d), dt, _ptr(tok_buf), _ptr(par_buf), B, N, V,
                                         float(temperature), int(seed) & (2**64 - 1), _ptr(path),
                                         _ptr(length), _ptr(boundary))
    if rc != 0:
        raise MemoryError("oracle_tree_verify_sampling failed to allocate")
    return dict(path=path, length=length, boundary_at=boundary, boundary=boundary.any(axis=1).astype(np.int32))


def ngram_draft(tokens, lengths, n_min: int, n_max: int, K: int):
    """N-gram (prompt-lookup) drafts.  tokens [B, Lmax] int32 histories (row b
    holds lengths[b] valid tokens), lengths [B].  Returns dict(drafts [B, K]
    (-1 padded), n_drafts [B], match_len [B]); a length outside [0, Lmax]
    gives n_drafts = match_len = -1."""
    lib = _load()
    tok = _as_i32(tokens)
    if tok.ndim != 2:
        raise ValueError("tokens must be [B, Lmax]")
    B, Lmax = tok.shape
    ln = np.ascontiguousarray(np.asarray(lengths, dtype=np.int32).reshape(-1))
    if ln.size != B:
        raise ValueError("lengths must have B entries")
    drafts = np.full((B, max(K, 0)), -1, dtype=np.int32)
    n_drafts = np.zeros(B, dtype=np.int32)
    match_len = np.zeros(B, dtype=np.int32)
    tok_buf = tok if tok.size else np.zeros(1, dtype=np.int32)
    ln_buf = ln if ln.size else np.zeros(1, dtype=np.int32)
    d_buf = drafts if drafts.size else np.zeros(1, dtype=np.int32)
    lib.oracle_ngram_draft(_ptr(tok_buf), int(Lmax), _ptr(ln_buf), int(B), int(n_min), int(n_max), int(K),
                           _ptr(d_buf), _ptr(n_drafts), _ptr(match_len))
    return dict(drafts=drafts, n_drafts=n_drafts, match_len=match_len)
