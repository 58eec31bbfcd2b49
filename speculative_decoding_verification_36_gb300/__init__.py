"""GB300-native speculative-decoding verify step.

A thin binding over libspecverify.so (C ABI in include/specverify.h).  Each
function checks and marshals torch CUDA tensors (device, dtype, contiguity,
shapes), allocates outputs that were not given, and calls the C entry point of
the same name on the current stream; every step of the verify path runs in the
library's CUDA kernels.  There is no CPU fallback.

    spec_verify(target_logits, draft_logits, draft_tokens, temperature, seed)
    spec_verify_early_exit(...)       # reads only the rows the result depends on
    spec_verify_static_scratch(...)   # no allocation: a fixed per-device scratch buffer
    spec_verify_stats(...)            # plus row statistics, p(x), q(x), mass
    spec_verify_khint(..., h_lo, h_hi, k_min, k_max)  # plus a suggested next draft length
    spec_verify_greedy_argmax(...)    # greedy chain plus every row's argmax
    spec_tree_verify_greedy(target_logits, tree_tokens, parent_idx)
    spec_tree_verify_sampling(target_logits, draft_logits, tree_tokens, parent_idx, T, seed)
    spec_acceptance_stats(n_accepted, K)  # histogram, alpha, mean tokens
    spec_ngram_draft(tokens, lengths, n_min, n_max, K)  # prompt-lookup drafts
    spec_get_status()                 # device status word (bad data, timeouts)
"""
from __future__ import annotations

import torch

from . import _lib
from ._lib import SPEC_FLAG_BAD_DATA, SPEC_FLAG_TIMEOUT, SpecError

__all__ = [
    "spec_verify", "spec_verify_early_exit", "spec_verify_static_scratch", "spec_verify_stats", "spec_verify_khint",
    "spec_verify_greedy_argmax",
    "spec_tree_verify_greedy", "spec_tree_verify_sampling", "spec_acceptance_stats", "spec_ngram_draft",
    "spec_get_status", "spec_test_spin_limit", "spec_test_wait_probe", "SpecError",
    "SPEC_FLAG_BAD_DATA", "SPEC_FLAG_TIMEOUT",
]


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _is_bf16(t: torch.Tensor, name: str) -> bool:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype == torch.bfloat16:
        return True
    if t.dtype == torch.float32:
        return False
    raise TypeError(f"{name} must be float32 or bfloat16, got {t.dtype}")


def _ptr(t):
    if t is None or t.numel() == 0:
        return None
    return t.data_ptr()


def _same_device(t: torch.Tensor, device, name: str):
    # a pointer into another GPU's memory is not readable by this device's kernels
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device} (all tensors of a call share one GPU)")


def _i32(t: torch.Tensor, shape, name: str, device=None):
    if not isinstance(t, torch.Tensor) or t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if device is not None:
        _same_device(t, device, name)
    return t


def _out(t, shape, dtype, device, name):
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    if t.dtype != dtype or not t.is_contiguous() or tuple(t.shape) != tuple(shape) or t.device != device:
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)} on {device}")
    return t


def _chain_args(target_logits, draft_logits, draft_tokens, temperature):
    bf16 = _is_bf16(target_logits, "target_logits")
    if target_logits.dim() != 3:
        raise ValueError("target_logits must be [B, K+1, V]")
    B, K1, V = target_logits.shape
    K = K1 - 1
    if temperature > 0 and K > 0:
        if draft_logits is None:
            raise ValueError("draft_logits is required when temperature > 0")
        if _is_bf16(draft_logits, "draft_logits") != bf16:
            raise TypeError("target_logits and draft_logits must share a dtype")
        if tuple(draft_logits.shape) != (B, K, V):
            raise ValueError(f"draft_logits has shape {tuple(draft_logits.shape)}, expected {(B, K, V)}")
        _same_device(draft_logits, target_logits.device, "draft_logits")
    if K > 0:
        _i32(draft_tokens, (B, K), "draft_tokens", target_logits.device)
    return bf16, B, K, V


def spec_verify(target_logits, draft_logits, draft_tokens, temperature: float, seed: int,
                out_tokens=None, out_n_accepted=None, stream=None):
    """Verify K drafted tokens per sequence; returns (out_tokens [B,K+1], n [B])."""
    bf16, B, K, V = _chain_args(target_logits, draft_logits, draft_tokens, temperature)
    dev = target_logits.device
    out_tokens = _out(out_tokens, (B, K + 1), torch.int32, dev, "out_tokens")
    out_n_accepted = _out(out_n_accepted, (B,), torch.int32, dev, "out_n_accepted")
    lib = _lib.load()
    fn = lib.spec_verify_bf16 if bf16 else lib.spec_verify_f32
    with torch.cuda.device(dev):
        _lib.check(fn(_ptr(target_logits), _ptr(draft_logits) if temperature > 0 else None,
                      _ptr(draft_tokens) if K > 0 else None, B, K, V, float(temperature),
                      int(seed) & (2**64 - 1), _ptr(out_tokens), _ptr(out_n_accepted),
                      _stream(stream)))
    return out_tokens, out_n_accepted


def spec_verify_early_exit(target_logits, draft_logits, draft_tokens, temperature: float, seed: int,
                           out_tokens=None, out_n_accepted=None, stream=None):
    """spec_verify that reads only the rows its result depends on (positions
    up to the first rejection, and the bonus row when every draft is
    accepted); bad data is checked on those rows only.  Temperature 0 is the
    greedy verify with the same early exit (draft_logits may be None).
    Returns (out_tokens [B,K+1], n [B])."""
    bf16, B, K, V = _chain_args(target_logits, draft_logits, draft_tokens, temperature)
    dev = target_logits.device
    out_tokens = _out(out_tokens, (B, K + 1), torch.int32, dev, "out_tokens")
    out_n_accepted = _out(out_n_accepted, (B,), torch.int32, dev, "out_n_accepted")
    lib = _lib.load()
    fn = lib.spec_verify_early_exit_bf16 if bf16 else lib.spec_verify_early_exit_f32
    with torch.cuda.device(dev):
        _lib.check(fn(_ptr(target_logits), _ptr(draft_logits) if temperature > 0 else None,
                      _ptr(draft_tokens) if K > 0 else None, B, K, V, float(temperature),
                      int(seed) & (2**64 - 1), _ptr(out_tokens), _ptr(out_n_accepted),
                      _stream(stream)))
    return out_tokens, out_n_accepted


def spec_verify_static_scratch(target_logits, draft_logits, draft_tokens, temperature: float,
                               seed: int, out_tokens=None, out_n_accepted=None, stream=None):
    """spec_verify for bf16 logits with the library's fixed per-device scratch
    buffer instead of its memory pool (no device allocation by the library).
    Calls that overlap in time on one device race on that buffer.  Pass
    out_tokens / out_n_accepted to keep this wrapper allocation-free too."""
    bf16, B, K, V = _chain_args(target_logits, draft_logits, draft_tokens, temperature)
    if not bf16:
        raise TypeError("spec_verify_static_scratch takes bf16 logits")
    dev = target_logits.device
    out_tokens = _out(out_tokens, (B, K + 1), torch.int32, dev, "out_tokens")
    out_n_accepted = _out(out_n_accepted, (B,), torch.int32, dev, "out_n_accepted")
    lib = _lib.load()
    with torch.cuda.device(dev):
        _lib.check(lib.spec_verify_bf16_static_scratch(
            _ptr(target_logits), _ptr(draft_logits) if temperature > 0 else None,
            _ptr(draft_tokens) if K > 0 else None, B, K, V, float(temperature),
            int(seed) & (2**64 - 1), _ptr(out_tokens), _ptr(out_n_accepted), _stream(stream)))
    return out_tokens, out_n_accepted


def spec_verify_stats(target_logits, draft_logits, draft_tokens, temperature: float, seed: int,
                      stream=None, entropy: bool = False):
    """spec_verify plus the intermediate probabilities (temperature > 0).

    Returns dict(tokens [B,K+1], n [B], row_stats [B,2K+1,2] (max z/tau, sum
    exp(z/tau - max)), pq [B,K,2] (p_i(x_i), q_i(x_i)), resid_mass [B]) and,
    with entropy=True, row_entropy [B,2K+1] (nats)."""
    if not temperature > 0:
        raise ValueError("spec_verify_stats needs temperature > 0")
    bf16, B, K, V = _chain_args(target_logits, draft_logits, draft_tokens, temperature)
    dev = target_logits.device
    tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    n = torch.empty((B,), dtype=torch.int32, device=dev)
    row_stats = torch.empty((B, 2 * K + 1, 2), dtype=torch.float32, device=dev)
    pq = torch.empty((B, K, 2), dtype=torch.float32, device=dev)
    resid = torch.empty((B,), dtype=torch.float32, device=dev)
    ent = torch.empty((B, 2 * K + 1), dtype=torch.float32, device=dev) if entropy else None
    lib = _lib.load()
    fn = lib.spec_verify_stats_bf16 if bf16 else lib.spec_verify_stats_f32
    with torch.cuda.device(dev):
        _lib.check(fn(_ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens) if K > 0 else None,
                      B, K, V, float(temperature), int(seed) & (2**64 - 1), _ptr(tokens), _ptr(n),
                      _ptr(row_stats), _ptr(pq), _ptr(resid), _ptr(ent) if entropy else None,
                      _stream(stream)))
    out = dict(tokens=tokens, n=n, row_stats=row_stats, pq=pq, resid_mass=resid)
    if entropy:
        out["row_entropy"] = ent
    return out


def spec_verify_khint(target_logits, draft_logits, draft_tokens, temperature: float, seed: int,
                      h_lo: float, h_hi: float, k_min: int, k_max: int, stream=None, out_tokens=None,
                      out_n_accepted=None, out_k_next=None, out_mean_entropy=None):
    """spec_verify plus a suggested next draft length per sequence (temperature > 0).

    The mean entropy (nats) of target rows 0..n moves K one step up when below
    h_lo, one step down when above h_hi; the result is clamped to [k_min,
    k_max], -1 for a bad sequence.  Returns (tokens [B,K+1], n [B], k_next [B]
    int32, mean_entropy [B] float32)."""
    bf16, B, K, V = _chain_args(target_logits, draft_logits, draft_tokens, temperature)
    dev = target_logits.device
    tokens = _out(out_tokens, (B, K + 1), torch.int32, dev, "out_tokens")
    n = _out(out_n_accepted, (B,), torch.int32, dev, "out_n_accepted")
    k_next = _out(out_k_next, (B,), torch.int32, dev, "out_k_next")
    hmean = _out(out_mean_entropy, (B,), torch.float32, dev, "out_mean_entropy")
    lib = _lib.load()
    fn = lib.spec_verify_khint_bf16 if bf16 else lib.spec_verify_khint_f32
    with torch.cuda.device(dev):
        _lib.check(fn(_ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens) if K > 0 else None,
                      B, K, V, float(temperature), int(seed) & (2**64 - 1), float(h_lo), float(h_hi),
                      int(k_min), int(k_max), _ptr(tokens), _ptr(n), _ptr(k_next), _ptr(hmean),
                      _stream(stream)))
    return tokens, n, k_next, hmean


def spec_verify_greedy_argmax(target_logits, draft_tokens, stream=None):
    """Greedy chain verification that also returns every target row's argmax.

    Returns (out_tokens [B,K+1], n [B], row_argmax [B,K+1])."""
    bf16, B, K, V = _chain_args(target_logits, None, draft_tokens, 0.0)
    dev = target_logits.device
    tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    n = torch.empty((B,), dtype=torch.int32, device=dev)
    amax = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    lib = _lib.load()
    fn = lib.spec_verify_greedy_argmax_bf16 if bf16 else lib.spec_verify_greedy_argmax_f32
    with torch.cuda.device(dev):
        _lib.check(fn(_ptr(target_logits), _ptr(draft_tokens) if K > 0 else None, B, K, V,
                      _ptr(tokens), _ptr(n), _ptr(amax), _stream(stream)))
    return tokens, n, amax


def spec_tree_verify_greedy(target_logits, tree_tokens, parent_idx, out_path=None, out_len=None,
                            out_mask=None, stream=None, early_exit: bool = False):
    """Greedy verification of a candidate tree per sequence.

    target_logits [B, N+1, V]; tree_tokens, parent_idx [B, N] int32.
    Returns (out_path [B, N+1], out_len [B], out_mask [B, N, ceil(N/32)] as int32 bits).
    early_exit=True calls spec_tree_verify_greedy_early_exit_*: the rows under
    a rejected node are not read (and bad data there is not reported)."""
    bf16 = _is_bf16(target_logits, "target_logits")
    if target_logits.dim() != 3:
        raise ValueError("target_logits must be [B, N+1, V]")
    B, N1, V = target_logits.shape
    N = N1 - 1
    W = (N + 31) // 32
    dev = target_logits.device
    if N > 0:
        _i32(tree_tokens, (B, N), "tree_tokens", dev)
        _i32(parent_idx, (B, N), "parent_idx", dev)
    out_path = _out(out_path, (B, N + 1), torch.int32, dev, "out_path")
    out_len = _out(out_len, (B,), torch.int32, dev, "out_len")
    # torch has no uint32 arithmetic on every version: the mask words travel as int32 bits
    out_mask = _out(out_mask, (B, N, W), torch.int32, dev, "out_mask")
    lib = _lib.load()
    if early_exit:
        fn = lib.spec_tree_verify_greedy_early_exit_bf16 if bf16 else lib.spec_tree_verify_greedy_early_exit_f32
    else:
        fn = lib.spec_tree_verify_greedy_bf16 if bf16 else lib.spec_tree_verify_greedy_f32
    with torch.cuda.device(dev):
        _lib.check(fn(_ptr(target_logits), _ptr(tree_tokens) if N > 0 else None,
                      _ptr(parent_idx) if N > 0 else None, B, N, V, _ptr(out_path), _ptr(out_len),
                      _ptr(out_mask), _stream(stream)))
    return out_path, out_len, out_mask


def spec_tree_verify_sampling(target_logits, draft_logits, tree_tokens, parent_idx, temperature: float,
                              seed: int, out_path=None, out_len=None, stream=None):
    """Stochastic verification of a candidate tree per sequence (temperature > 0).

    target_logits, draft_logits [B, N+1, V] (draft row u+1: the distribution
    node u's children were drawn from); tree_tokens, parent_idx [B, N] int32.
    Returns (out_path [B, N+1], out_len [B])."""
    if not temperature > 0:
        raise ValueError("spec_tree_verify_sampling needs temperature > 0 (spec_tree_verify_greedy is T = 0)")
    bf16 = _is_bf16(target_logits, "target_logits")
    if target_logits.dim() != 3:
        raise ValueError("target_logits must be [B, N+1, V]")
    if _is_bf16(draft_logits, "draft_logits") != bf16:
        raise TypeError("target_logits and draft_logits must share a dtype")
    if tuple(draft_logits.shape) != tuple(target_logits.shape):
        raise ValueError(f"draft_logits has shape {tuple(draft_logits.shape)}, expected "
                         f"{tuple(target_logits.shape)}")
    B, N1, V = target_logits.shape
    N = N1 - 1
    dev = target_logits.device
    _same_device(draft_logits, dev, "draft_logits")
    if N > 0:
        _i32(tree_tokens, (B, N), "tree_tokens", dev)
        _i32(parent_idx, (B, N), "parent_idx", dev)
    out_path = _out(out_path, (B, N + 1), torch.int32, dev, "out_path")
    out_len = _out(out_len, (B,), torch.int32, dev, "out_len")
    lib = _lib.load()
    fn = lib.spec_tree_verify_sampling_bf16 if bf16 else lib.spec_tree_verify_sampling_f32
    with torch.cuda.device(dev):
        _lib.check(fn(_ptr(target_logits), _ptr(draft_logits), _ptr(tree_tokens) if N > 0 else None,
                      _ptr(parent_idx) if N > 0 else None, B, N, V, float(temperature),
                      int(seed) & (2**64 - 1), _ptr(out_path), _ptr(out_len), _stream(stream)))
    return out_path, out_len


def spec_acceptance_stats(n_accepted, K: int, stream=None):
    """Acceptance statistics of verify outputs on the device.

    n_accepted: int32 [B] (-1 = bad sequence).  Returns dict(hist uint64-valued
    int64 [K+2], alpha float64 [K], mean_tokens float64 scalar tensor)."""
    if (not isinstance(n_accepted, torch.Tensor) or n_accepted.dtype != torch.int32 or n_accepted.dim() != 1
            or not n_accepted.is_contiguous() or not n_accepted.is_cuda):
        raise TypeError("n_accepted must be a contiguous 1-D int32 CUDA tensor")
    dev = n_accepted.device
    B = n_accepted.shape[0]
    hist = torch.empty((K + 2,), dtype=torch.int64, device=dev)
    alpha = torch.empty((max(K, 0),), dtype=torch.float64, device=dev)
    mean = torch.empty((1,), dtype=torch.float64, device=dev)
    lib = _lib.load()
    with torch.cuda.device(dev):
        _lib.check(lib.spec_acceptance_stats(_ptr(n_accepted) if B > 0 else None, B, int(K),
                                             _ptr(hist), _ptr(alpha) if K > 0 else None, _ptr(mean),
                                             _stream(stream)))
    return dict(hist=hist, alpha=alpha, mean_tokens=mean[0])


def spec_ngram_draft(tokens, lengths, n_min: int, n_max: int, K: int, out_drafts=None, out_n_drafts=None,
                     out_match_len=None, stream=None):
    """N-gram (prompt-lookup) drafts from token histories on the device.

    tokens: int32 [B, Lmax] (row b's first lengths[b] entries are its history);
    lengths: int32 [B].  Returns (drafts int32 [B, K] (-1 padded), n_drafts
    int32 [B], match_len int32 [B])."""
    if tokens.dim() != 2:
        raise ValueError("tokens must be [B, Lmax]")
    B, Lmax = tokens.shape
    _i32(tokens, (B, Lmax), "tokens")
    dev = tokens.device
    _i32(lengths, (B,), "lengths", dev)
    drafts = _out(out_drafts, (B, max(int(K), 0)), torch.int32, dev, "out_drafts")  # K < 0: the C layer refuses
    n_drafts = _out(out_n_drafts, (B,), torch.int32, dev, "out_n_drafts")
    match_len = _out(out_match_len, (B,), torch.int32, dev, "out_match_len")
    lib = _lib.load()
    with torch.cuda.device(dev):
        _lib.check(lib.spec_ngram_draft(_ptr(tokens), _ptr(lengths), B, Lmax, int(n_min), int(n_max), int(K),
                                        _ptr(drafts), _ptr(n_drafts), _ptr(match_len), _stream(stream)))
    return drafts, n_drafts, match_len


def spec_get_status(stream=None, device=None) -> int:
    """Synchronise and return (then clear) the device status word: an OR of
    SPEC_FLAG_BAD_DATA / SPEC_FLAG_TIMEOUT set since the last read."""
    import ctypes
    flags = ctypes.c_uint32(0)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _lib.check(_lib.load().spec_get_status(_stream(stream), ctypes.addressof(flags)))
    return int(flags.value)


def spec_test_spin_limit(iterations: int, device=None) -> None:
    """Test hook for failure-detection tests: every bounded wait inside the
    kernels of later calls on the device gives up after `iterations` polls and
    flags SPEC_FLAG_TIMEOUT; 0 restores the default limit.  Synchronises the
    device first."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _lib.check(_lib.load().spec_test_spin_limit(int(iterations)))


def spec_test_wait_probe(device=None) -> tuple:
    """Test hook: runs every bounded-wait helper of the library on a slot that
    nothing writes and on one already written, under the current limit.
    Returns (helpers that gave up on the unwritten slot, helpers that flagged
    the written one) as bit masks; a correct library gives (0x7f, 0)."""
    import ctypes
    flags = (ctypes.c_uint32 * 2)()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _lib.check(_lib.load().spec_test_wait_probe(ctypes.addressof(flags)))
    return int(flags[0]), int(flags[1])
