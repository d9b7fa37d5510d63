"""dec_attention_noalloc: the attention entry point for callers that cannot allocate device
memory (a real-time audio thread, where cudaMalloc/cudaFree may synchronize the device; a host
application whose allocator owns the device-memory budget).  Its scratch is the library's static
device array, so two calls in a row must each give what dec_attention gives with a freshly
allocated workspace.  Collected last on purpose: a run that stops at the first failure has run
every other test before it."""
import ctypes as C

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tts_autoregressive_decode_gb300 import _lib, native_build
    native_build.build()
    return _lib


def _case(seed, m, H, G, d, lens):
    g = torch.Generator().manual_seed(seed)
    cap = max(lens) + 5
    q = torch.randn(m, H, d, generator=g).cuda()
    k = torch.randn(m, G, cap, d, generator=g).cuda()
    v = torch.randn(m, G, cap, d, generator=g).cuda()
    L = torch.tensor(lens, dtype=torch.int32).cuda()
    return q, k, v, L, cap


def _with_workspace(L, m, H, G, d, cap, q, k, v, lens):
    nbytes = L.load().dec_attention_workspace_bytes(m, H, G, d, cap)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    st = L.load().dec_attention(m, H, G, d, cap, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                lens.data_ptr(), out.data_ptr(), ws.data_ptr(), nbytes,
                                torch.cuda.current_stream().cuda_stream)
    L.check(st)
    return out


def _noalloc(L, m, H, G, d, cap, q, k, v, lens):
    out = torch.empty_like(q)
    st = L.load().dec_attention_noalloc(m, H, G, d, cap, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                        lens.data_ptr(), out.data_ptr(),
                                        torch.cuda.current_stream().cuda_stream)
    L.check(st)
    return out


def test_two_calls_in_a_row_match_the_workspace_entry(lib):
    cases = [(1, 3, 16, 8, 128, [700, 1, 333]),   # GQA group 2, several chunks and a ragged tail
             (2, 2, 4, 2, 64, [65, 129])]          # another shape: the array keeps stale data
    for seed, m, H, G, d, lens in cases:
        q, k, v, Ld, cap = _case(seed, m, H, G, d, lens)
        got = _noalloc(lib, m, H, G, d, cap, q, k, v, Ld)
        want = _with_workspace(lib, m, H, G, d, cap, q, k, v, Ld)
        torch.cuda.synchronize()
        diff = float((got - want).abs().max())
        assert diff <= 2e-5, (seed, diff)
        assert torch.isfinite(got).all()


def test_oversized_request_is_rejected(lib):
    q, k, v, Ld, _ = _case(3, 2, 16, 8, 128, [8, 8])
    out = torch.empty_like(q)
    st = lib.load().dec_attention_noalloc(2, 16, 8, 128, 32768, q.data_ptr(), k.data_ptr(),
                                          v.data_ptr(), Ld.data_ptr(), out.data_ptr(),
                                          torch.cuda.current_stream().cuda_stream)
    assert st == lib.DEC_E_UNSUPPORTED
    assert b"static scratch" in lib.load().dec_last_error(None)


def test_capacity_at_the_exact_limit(lib):
    # m = 1, 16/8 heads, d = 128: 504 chunks of 64 keys fill the 4 MiB array (capacity 32256);
    # one key more needs a 505th chunk and is rejected with the state of the array untouched
    m, H, G, d = 1, 16, 8, 128
    L = lib.load()
    assert L.dec_attention_workspace_bytes(m, H, G, d, 32256) <= 4 << 20
    assert L.dec_attention_workspace_bytes(m, H, G, d, 32257) > 4 << 20
    q, k, v, Ld, cap = _case(4, m, H, G, d, [32256])
    assert cap >= 32256
    k, v = k[:, :, :32256].contiguous(), v[:, :, :32256].contiguous()
    got = _noalloc(lib, m, H, G, d, 32256, q, k, v, Ld)
    want = _with_workspace(lib, m, H, G, d, 32256, q, k, v, Ld)
    torch.cuda.synchronize()
    assert float((got - want).abs().max()) <= 2e-5
    out = torch.empty_like(q)
    st = L.dec_attention_noalloc(m, H, G, d, 32257, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                 Ld.data_ptr(), out.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    assert st == lib.DEC_E_UNSUPPORTED
    assert b"static scratch" in L.dec_last_error(None)
