"""C-ABI checks that need no GPU: the library builds and loads, exports every
symbol include/specverify.h declares, and rejects bad arguments on the host
with the documented codes before any CUDA call."""
import ctypes
import math

import pytest

from speculative_decoding_verification_36_gb300 import _lib, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def test_header_declares_expected_entry_points():
    names = set(_lib.header_symbols())
    assert {"spec_verify_f32", "spec_verify_bf16", "spec_tree_verify_greedy_f32",
            "spec_tree_verify_greedy_bf16", "spec_get_status", "spec_status_string"} <= names
    assert names == set(_lib.SIGNATURES), "binding signatures and header disagree"


def test_library_exports_every_header_symbol(lib):
    for name in _lib.header_symbols():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, 99):
        assert isinstance(lib.spec_status_string(code), bytes)


# fake, never-dereferenced device addresses: the host checks return before any use
FAKE = 0x10000


def _chain(lib, fn="spec_verify_f32", target=FAKE, draft=FAKE, tokens=FAKE, B=2, K=3, V=16,
           temperature=1.0, out_tokens=FAKE, out_n=FAKE):
    return getattr(lib, fn)(target, draft, tokens, B, K, V, temperature, 0, out_tokens, out_n, None)


CHAIN_FNS = ["spec_verify_f32", "spec_verify_bf16", "spec_verify_bf16_static_scratch"]


@pytest.mark.parametrize("fn", CHAIN_FNS)
def test_null_pointers(lib, fn):
    assert _chain(lib, fn, target=None) == _lib.SPEC_ERR_NULL
    assert _chain(lib, fn, out_tokens=None) == _lib.SPEC_ERR_NULL
    assert _chain(lib, fn, out_n=None) == _lib.SPEC_ERR_NULL
    assert _chain(lib, fn, tokens=None) == _lib.SPEC_ERR_NULL
    assert _chain(lib, fn, draft=None) == _lib.SPEC_ERR_NULL


@pytest.mark.parametrize("fn", CHAIN_FNS)
def test_bad_shapes(lib, fn):
    assert _chain(lib, fn, B=-1) == _lib.SPEC_ERR_SHAPE
    assert _chain(lib, fn, K=-1) == _lib.SPEC_ERR_SHAPE
    assert _chain(lib, fn, K=256) == _lib.SPEC_ERR_SHAPE
    assert _chain(lib, fn, V=0) == _lib.SPEC_ERR_SHAPE
    assert _chain(lib, fn, B=2**30, K=255, V=2**30) == _lib.SPEC_ERR_SHAPE


@pytest.mark.parametrize("fn", CHAIN_FNS)
@pytest.mark.parametrize("tau", [math.nan, -1.0, 1e-35])
def test_bad_temperature(lib, fn, tau):
    assert _chain(lib, fn, temperature=tau) == _lib.SPEC_ERR_TEMPERATURE


@pytest.mark.parametrize("fn", CHAIN_FNS)
def test_empty_batch_is_a_noop(lib, fn):
    # B == 0 returns before touching the device
    assert _chain(lib, fn, B=0) == _lib.SPEC_OK
    assert _chain(lib, fn, B=0, temperature=0.0) == _lib.SPEC_OK


def test_greedy_needs_no_draft(lib):
    # temperature 0 does not require draft logits; a bad shape still fails first
    assert _chain(lib, draft=None, temperature=0.0, V=0) == _lib.SPEC_ERR_SHAPE
    assert _chain(lib, draft=None, temperature=0.0, B=0) == _lib.SPEC_OK


def test_tree_checks(lib):
    f = lib.spec_tree_verify_greedy_bf16
    assert f(None, FAKE, FAKE, 1, 3, 8, FAKE, FAKE, FAKE, None) == _lib.SPEC_ERR_NULL
    assert f(FAKE, None, FAKE, 1, 3, 8, FAKE, FAKE, FAKE, None) == _lib.SPEC_ERR_NULL
    assert f(FAKE, FAKE, FAKE, 1, 3, 8, FAKE, FAKE, None, None) == _lib.SPEC_ERR_NULL
    assert f(FAKE, FAKE, FAKE, 1, 1025, 8, FAKE, FAKE, FAKE, None) == _lib.SPEC_ERR_SHAPE
    assert f(FAKE, FAKE, FAKE, 1, -1, 8, FAKE, FAKE, FAKE, None) == _lib.SPEC_ERR_SHAPE
    assert f(FAKE, FAKE, FAKE, 0, 3, 8, FAKE, FAKE, FAKE, None) == _lib.SPEC_OK


@pytest.mark.parametrize("fn", ["spec_tree_verify_sampling_f32", "spec_tree_verify_sampling_bf16"])
def test_tree_sampling_checks(lib, fn):
    f = getattr(lib, fn)

    def call(t=FAKE, d=FAKE, tok=FAKE, par=FAKE, B=1, N=3, V=8, tau=1.0, path=FAKE, ln=FAKE):
        return f(t, d, tok, par, B, N, V, tau, 0, path, ln, None)

    assert call(t=None) == _lib.SPEC_ERR_NULL
    assert call(d=None) == _lib.SPEC_ERR_NULL
    assert call(tok=None) == _lib.SPEC_ERR_NULL
    assert call(par=None) == _lib.SPEC_ERR_NULL
    assert call(path=None) == _lib.SPEC_ERR_NULL
    assert call(ln=None) == _lib.SPEC_ERR_NULL
    assert call(tok=None, par=None, N=0, B=0) == _lib.SPEC_OK  # no nodes: no tree arrays needed
    for tau in (0.0, -1.0, math.nan, 1e-35):
        assert call(tau=tau) == _lib.SPEC_ERR_TEMPERATURE
    assert call(N=1025) == _lib.SPEC_ERR_SHAPE
    assert call(N=-1) == _lib.SPEC_ERR_SHAPE
    assert call(V=0) == _lib.SPEC_ERR_SHAPE
    assert call(B=-1) == _lib.SPEC_ERR_SHAPE
    assert call(B=0) == _lib.SPEC_OK


def test_python_binding_rejects_cpu_tensors():
    import torch
    import speculative_decoding_verification_36_gb300 as sv
    t = torch.zeros(1, 2, 8)
    with pytest.raises(ValueError):
        sv.spec_verify(t, t[:, :1], torch.zeros(1, 1, dtype=torch.int32), 1.0, 0)


def test_python_binding_rejects_host_and_foreign_device_tensors():
    import torch
    import speculative_decoding_verification_36_gb300 as sv
    from speculative_decoding_verification_36_gb300 import _same_device
    with pytest.raises(TypeError):
        sv.spec_acceptance_stats(torch.zeros(4, dtype=torch.int32), 3)
    with pytest.raises(ValueError):
        sv.spec_ngram_draft(torch.zeros(2, 8, dtype=torch.int32), torch.zeros(2, dtype=torch.int32), 1, 2, 3)
    with pytest.raises(ValueError):
        sv.spec_tree_verify_greedy(torch.zeros(1, 3, 8), torch.zeros(1, 2, dtype=torch.int32),
                                   torch.zeros(1, 2, dtype=torch.int32))
    # every tensor of a call must live on the target logits' device
    _same_device(torch.zeros(1), torch.device("cpu"), "x")
    with pytest.raises(ValueError):
        _same_device(torch.zeros(1), torch.device("meta"), "x")


def test_ngram_checks(lib):
    f = lib.spec_ngram_draft

    def call(tok=FAKE, ln=FAKE, B=2, stride=8, n_min=1, n_max=4, K=3, d=FAKE, nd=FAKE, ml=FAKE):
        return f(tok, ln, B, stride, n_min, n_max, K, d, nd, ml, None)

    assert call(tok=None) == _lib.SPEC_ERR_NULL
    assert call(ln=None) == _lib.SPEC_ERR_NULL
    assert call(nd=None) == _lib.SPEC_ERR_NULL
    assert call(d=None) == _lib.SPEC_ERR_NULL
    assert call(d=None, K=0, B=0) == _lib.SPEC_OK
    for bad in (dict(B=-1), dict(stride=0), dict(stride=2**30 + 1), dict(n_min=0), dict(n_min=5, n_max=4),
                dict(n_max=33), dict(K=-1), dict(K=4097)):
        assert call(**bad) == _lib.SPEC_ERR_SHAPE, bad
    # 32-bit (sequence, chunk) entries: B * ceil(stride / 4096) stays below
    # 2^31 - 2^20, refused on the host before any device work
    chunks = -(-2**30 // 4096)
    limit_b = ((2**31 - 2**20) + chunks - 1) // chunks
    assert call(B=limit_b, stride=2**30) == _lib.SPEC_ERR_SHAPE
    assert call(B=0, stride=2**30) == _lib.SPEC_OK
