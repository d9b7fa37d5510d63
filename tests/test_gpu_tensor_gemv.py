"""The tensor-core GEMV (DEC_FLAG_TENSOR_GEMV: tcgen05.mma with TMEM accumulators, TMA weight
tiles, x in three bf16 terms) against the CPU oracle: steps of 3 and 8 streams and prefill
blocks of up to 8 rows.  Its k split, the partial tiles finished by the last CTA, the deferred
RMSNorm scale and the SwiGLU / residual epilogues all run here; the FMA kernels that serve the
same shapes by default agree with it within rounding."""
import os

import numpy as np
import pytest

import oracle
from tts_autoregressive_decode_gb300 import workloads as W

from _parity import Stats, check_rows  # noqa: E402

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def D():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tts_autoregressive_decode_gb300 import decoder, native_build
    native_build.build()
    oracle.set_threads(os.cpu_count() or 1)
    return decoder


def _steps(D, w, n):
    syn = W.generate(w, steps=n)
    orc = oracle.OracleModel(syn)
    tc = D.Decoder.from_synthetic(syn, flags=D.L.DEC_FLAG_TENSOR_GEMV)
    fma = D.Decoder.from_synthetic(syn)
    st = Stats()
    m = w.streams
    for t in range(n):
        pos = tc.lengths(m)
        assert pos == [orc.length(s) for s in range(m)]
        x = torch.from_numpy(np.ascontiguousarray(syn.inputs[t])).cuda()
        a = tc.step(x, pos)
        b = fma.step(x, pos)
        want = orc.step(syn.inputs[t], pos)
        check_rows(a.cpu().numpy(), want, True, st, f"{w.name} step {t} tensor")
        check_rows(b.cpu().numpy(), want, True, None, f"{w.name} step {t} fma")
    tc.sync()
    fma.sync()
    return st


def test_small_talker_bf16_three_streams(D):
    # o-proj (K 512, N 392: a partial last tile) takes the tensor cores
    st = _steps(D, W.SMALL_TALKER_BF16, W.SMALL_TALKER_BF16.steps)
    print(f"small_talker_bf16: {st.line()}")


def test_talker_h2048_l28_bf16_m8_first_steps(D):
    # all four GEMVs of the 28-layer stack, 8 streams: split tiles, RMSNorm deferred, SwiGLU
    st = _steps(D, W.TALKER_H2048_L28_M8, 3)
    print(f"talker_h2048_l28_bf16_m8: {st.line()}")


def test_prefill_28_layer_bf16_blocks(D):
    """A 20-row block (8 + 8 + 4) of the 28-layer bf16 talker after its 2048-position prefill:
    blocks of 8 and of 4 rows through the tensor cores, then a step that reads the rows."""
    w = W.TALKER_H2048_L28
    syn = W.generate(w, steps=2)
    syn.max_pos = 2048 + 24
    orc = oracle.OracleModel(syn)
    dec = D.Decoder.from_synthetic(syn, flags=D.L.DEC_FLAG_TENSOR_GEMV)
    st = Stats()
    x = np.random.default_rng(11).standard_normal((20, w.hidden)).astype(np.float32)
    got = dec.prefill(0, torch.from_numpy(x).cuda()).cpu().numpy()
    check_rows(got, orc.prefill(0, x), True, st, "28-layer prefill, tensor GEMV")
    pos = dec.lengths(1)
    xs = np.ascontiguousarray(syn.inputs[0][:1])
    check_rows(dec.step(torch.from_numpy(xs).cuda(), pos).cpu().numpy(), orc.step(xs, pos), True, st,
               "step after the block")
    dec.sync()
    print(f"28-layer prefill (tensor GEMV): {st.line()}")


def test_repeated_steps_are_bitwise_equal(D):
    """The finishing CTA adds the partial tiles in CTA order, whichever arrives last: two
    decoders on the same inputs give the same bits."""
    w = W.TALKER_H2048_L28_M8
    syn = W.generate(w, steps=2)
    a = D.Decoder.from_synthetic(syn, flags=D.L.DEC_FLAG_TENSOR_GEMV)
    b = D.Decoder.from_synthetic(syn, flags=D.L.DEC_FLAG_TENSOR_GEMV)
    for t in range(2):
        pos = a.lengths(w.streams)
        x = torch.from_numpy(np.ascontiguousarray(syn.inputs[t])).cuda()
        ya, yb = a.step(x, pos), b.step(x, pos)
        torch.cuda.synchronize()
        assert torch.equal(ya, yb), t
    a.sync()
    b.sync()
