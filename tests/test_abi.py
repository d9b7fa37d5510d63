"""The C ABI library loads, exports every entry point include/dec.h declares, and rejects bad
arguments on the host before touching a GPU (these tests need no GPU)."""
import ctypes as C
import os
import re

import pytest

from tts_autoregressive_decode_gb300 import _lib as L
from tts_autoregressive_decode_gb300 import native_build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return L.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "dec.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dec_[a-z_]+)\s*\(", src)))


def test_header_declarations_match_binding():
    assert declared_functions() == sorted(L.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_build_targets_sm_103a_only():
    assert B.ARCH == "-gencode=arch=compute_103a,code=sm_103a"


def _cfg(**kw):
    base = dict(kind=0, layers=1, hidden=256, q_heads=4, kv_heads=2, head_dim=64, inter=768,
                norm_eps=1e-6, rope_theta=1e6, weight_dtype=0, max_pos=64, ring=0, window=0,
                max_streams=1, flags=0)
    base.update(kw)
    return L.DecConfig(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(kind=7), L.DEC_E_ARG),
    (dict(head_dim=96), L.DEC_E_UNSUPPORTED),
    (dict(hidden=260), L.DEC_E_UNSUPPORTED),
    (dict(q_heads=3), L.DEC_E_ARG),
    (dict(q_heads=18, kv_heads=1), L.DEC_E_UNSUPPORTED),
    (dict(max_streams=9), L.DEC_E_ARG),
    (dict(max_pos=0), L.DEC_E_ARG),
    (dict(weight_dtype=5), L.DEC_E_ARG),
    (dict(norm_eps=float("nan")), L.DEC_E_ARG),
    (dict(kind=1, q_heads=4, kv_heads=2, ring=10, window=10), L.DEC_E_ARG),
    (dict(kind=1, q_heads=4, kv_heads=4, ring=10, window=11), L.DEC_E_ARG),
    (dict(max_streams=8, inter=8192), L.DEC_E_UNSUPPORTED),
])
def test_create_rejects_bad_configs_on_the_host(lib, kw, status):
    cfg = _cfg(**kw)
    out = C.c_void_p()
    w = L.DecWeights()
    st = lib.dec_create(C.byref(cfg), C.byref(w), None, C.byref(out))
    assert st == status
    assert out.value is None
    assert lib.dec_last_error(None)


def test_null_arguments(lib):
    out = C.c_void_p()
    assert lib.dec_create(None, None, None, C.byref(out)) == L.DEC_E_ARG
    assert lib.dec_step(None, 1, None, None, None) == L.DEC_E_ARG
    assert lib.dec_reset(None, 0) == L.DEC_E_ARG
    assert lib.dec_sync(None) == L.DEC_E_ARG
    assert lib.dec_get_len(None, 0) == -1
    assert lib.dec_set_mrope(None, None, 0) == L.DEC_E_ARG
    assert lib.dec_step_mrope(None, 1, None, None, None, None) == L.DEC_E_ARG
    assert lib.dec_prefill_mrope(None, 0, 1, None, None, None) == L.DEC_E_ARG
    lib.dec_destroy(None)


def test_mrope_axis_maps_from_sections():
    from tts_autoregressive_decode_gb300.decoder import mrope_axes
    a = mrope_axes(128, (24, 20, 20))
    assert [a.count(k) for k in range(3)] == [24, 20, 20]
    assert a[:7] == [0, 1, 2, 0, 1, 2, 0] and a[58:] == [1, 2, 0, 0, 0, 0]
    assert mrope_axes(128, (16, 24, 24), interleaved=False) == [0] * 16 + [1] * 24 + [2] * 24
    assert mrope_axes(64, (32, 0, 0)) == [0] * 32
    for bad in ((20, 20, 20), (10, 27, 27), (-1, 33, 32)):
        with pytest.raises(ValueError):
            mrope_axes(128, bad)


def test_stateless_entries_validate_before_launch(lib):
    buf = C.create_string_buffer(64)
    p = C.addressof(buf)
    p16 = (p + 15) // 16 * 16
    assert lib.dec_gemv(0, p16, 4, 12, p16, 1, p16, None) == L.DEC_E_UNSUPPORTED   # K % 8
    assert lib.dec_gemv(0, p16, 4, 16, p16, 9, p16, None) == L.DEC_E_ARG           # m > 8
    assert lib.dec_gemv(3, p16, 4, 16, p16, 1, p16, None) == L.DEC_E_ARG           # dtype
    assert lib.dec_gemv(0, p16 + 4, 4, 16, p16, 1, p16, None) == L.DEC_E_UNSUPPORTED
    assert lib.dec_attention(1, 4, 2, 96, 8, p16, p16, p16, p16, p16, p16, 1 << 20, None) \
        == L.DEC_E_UNSUPPORTED
    need = lib.dec_attention_workspace_bytes(2, 16, 8, 128, 4160)
    assert need >= 2 * 16 * 65 * 128 * 4
    assert lib.dec_attention(2, 16, 8, 128, 4160, p16, p16, p16, p16, p16, p16, need - 1, None) \
        == L.DEC_E_ARG
    assert lib.dec_attention_workspace_bytes(0, 1, 1, 64, 1) == 0
