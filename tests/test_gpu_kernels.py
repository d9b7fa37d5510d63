"""Per-kernel parity on the GPU through the C ABI: the row-major GEMV and the split-K decode
attention, against the CPU oracle on the same seeded inputs (ragged sizes, several tiles)."""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

U32 = 2.0 ** -24


@pytest.fixture(scope="module")
def dec():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tts_autoregressive_decode_gb300 import decoder
    from tts_autoregressive_decode_gb300 import native_build
    native_build.build()
    return decoder


def _bf16(a):
    from tts_autoregressive_decode_gb300.workloads import f32_to_bf16_bits
    return f32_to_bf16_bits(a)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N,K", [(1, 8), (7, 24), (130, 392), (301, 1000), (4096, 2048),
                                 (2048, 6144), (1536, 512)])
@pytest.mark.parametrize("m", [1, 2, 3, 4, 5, 7, 8])
def test_gemv_matches_oracle(dec, dtype, N, K, m):
    rng = np.random.default_rng(N * 7 + K + m)
    Wf = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    W = _bf16(Wf) if dtype == "bf16" else Wf
    Wexact = (W.astype(np.uint32) << 16).view(np.float32) if dtype == "bf16" else W
    x = rng.standard_normal((m, K)).astype(np.float32)
    Wd = dec.to_device(W, "cuda")
    xd = torch.from_numpy(x).cuda()
    y = dec.gemv(Wd, xd, bf16=(dtype == "bf16"))
    torch.cuda.synchronize()
    y = y.cpu().numpy().astype(np.float64)
    for r in range(m):
        want = oracle.matvec(W, x[r])
        # any summation order of K f32 products is within K * u * sum|w x| of the exact sum;
        # twice that covers both sides
        bound = 2 * K * U32 * (np.abs(Wexact).astype(np.float64) @ np.abs(x[r])) + 1e-30
        assert np.all(np.abs(y[r] - want) <= bound), (r, np.max(np.abs(y[r] - want) / bound))


def _attn_case(rng, m, H, G, d, cap, lens):
    q = rng.standard_normal((m, H, d)).astype(np.float32)
    k = rng.standard_normal((m, G, cap, d)).astype(np.float32)
    v = rng.standard_normal((m, G, cap, d)).astype(np.float32)
    return q, k, v, np.asarray(lens, np.int32)


@pytest.mark.parametrize("H,G,d", [(4, 2, 64), (16, 8, 128), (6, 2, 64), (8, 8, 64),
                                   (16, 2, 128)])
@pytest.mark.parametrize("lens", [[1], [2], [63], [64], [65], [129, 1, 700], [4160]])
def test_attention_matches_oracle(dec, H, G, d, lens):
    rng = np.random.default_rng(H * 100 + G * 10 + d + len(lens) + lens[0])
    m = len(lens)
    cap = max(lens) + 3
    q, k, v, L = _attn_case(rng, m, H, G, d, cap, lens)
    qd, kd, vd = (torch.from_numpy(a).cuda() for a in (q, k, v))
    Ld = torch.from_numpy(L).cuda()
    ws = torch.zeros(dec.attention_workspace_bytes(m, H, G, d, cap), dtype=torch.uint8,
                     device="cuda")
    out = dec.attention(qd, kd, vd, Ld, workspace=ws)
    out2 = dec.attention(qd, kd, vd, Ld, workspace=ws)   # tickets left clean: same again
    torch.cuda.synchronize()
    out = out.cpu().numpy()
    assert np.array_equal(out, out2.cpu().numpy())
    for r in range(m):
        n = lens[r]
        # the oracle's cache is position-major [L][G][d]
        want = oracle.gqa_attention(q[r], k[r, :, :n].transpose(1, 0, 2),
                                    v[r, :, :n].transpose(1, 0, 2))
        assert np.max(np.abs(out[r] - want)) < 2e-5, (r, np.max(np.abs(out[r] - want)))


def test_attention_single_key_is_exactly_its_value(dec):
    rng = np.random.default_rng(5)
    q, k, v, L = _attn_case(rng, 2, 16, 8, 128, 8, [1, 1])
    out = dec.attention(*(torch.from_numpy(a).cuda() for a in (q, k, v, L)))
    torch.cuda.synchronize()
    out = out.cpu().numpy()
    for r in range(2):
        for h in range(16):
            assert np.array_equal(out[r, h], v[r, h // 2, 0])
