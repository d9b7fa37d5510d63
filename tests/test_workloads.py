"""The seeded input generator: the recipe it states, its determinism, and the independence of
its draw categories.  No arithmetic of the decode step lives there, so these tests pin only the
inputs both sides consume."""
import numpy as np
import pytest

from tts_autoregressive_decode_gb300 import workloads as W

torch = pytest.importorskip("torch")


def test_bf16_rounding_matches_torch_round_to_nearest_even():
    rng = np.random.default_rng(0)
    a = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 3,
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 0.0, -0.0,
                                  65504.0, 1e-30], np.float32)])
    want = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(W.f32_to_bf16_bits(a), want)


def test_generation_is_deterministic_and_categories_are_independent():
    w = W.TALKER_H256_L1
    a, b = W.generate(w, steps=3), W.generate(w, steps=7)
    for la, lb in zip(a.layers, b.layers):
        for k in la:
            assert np.array_equal(la[k], lb[k]), k  # the step count does not move the weights
    assert np.array_equal(a.prefill_k[0], b.prefill_k[0])
    assert np.array_equal(a.inputs, b.inputs[:3])   # inputs are one stream, drawn in step order
    c = W.generate(w, steps=3)
    assert np.array_equal(a.inputs, c.inputs) and np.array_equal(a.final_norm, c.final_norm)


def test_value_distributions_follow_the_recipe():
    w = W.TALKER_H256_L1
    s = W.generate(w, steps=64)
    lin = np.concatenate([s.layers[0][k].ravel() for k in ("wq", "wk", "wv", "wo", "wgate",
                                                             "wup", "wdown")])
    assert abs(lin.std() / 0.02 - 1) < 0.02 and abs(lin.mean()) < 5e-4
    norms = np.concatenate([s.layers[0]["in_norm"], s.layers[0]["post_norm"], s.final_norm])
    assert abs(norms.mean() - 1) < 2e-3 and abs(norms.std() / 0.01 - 1) < 0.1
    assert abs(s.inputs.std() - 1) < 0.02
    assert abs(s.prefill_k[0].std() - 1) < 0.02


def test_workload_shapes_and_lengths_are_the_stated_ones():
    c3 = W.TALKER_H2048_L28
    assert (c3.layers, c3.hidden, c3.q_heads, c3.kv_heads, c3.head_dim, c3.inter) == \
        (28, 2048, 16, 8, 128, 6144)
    assert c3.weight_dtype == "bf16" and W.prefill_lengths(c3) == [2048] and c3.steps == 128
    c5 = W.TALKER_H2048_L28_M8
    ls = W.prefill_lengths(c5)
    assert len(ls) == 8 and all(512 <= n <= 4096 for n in ls) and len(set(ls)) > 1
    codec = W.CODEC_D512_L8
    assert (codec.ring, codec.window, codec.layers, codec.steps) == (250, 250, 8, 600)
    assert W.prefill_lengths(codec) == [0]
    fl = W.FLOWLM_D1024_L6
    assert (fl.ring, fl.window, W.max_pos(fl), fl.layers, fl.hidden) == (320, 320, 320, 6, 1024)
    assert W.prefill_lengths(fl) == [256] and not fl.layer_scale and fl.head


def test_bf16_workloads_store_bit_patterns_of_the_rounded_draws():
    s = W.generate(W.SMALL_TALKER_BF16)
    wq = s.layers[0]["wq"]
    assert wq.dtype == np.uint16
    widened = (wq.astype(np.uint32) << 16).view(np.float32)
    assert np.all(np.isfinite(widened)) and abs(widened.std() / 0.02 - 1) < 0.05
    assert s.layers[0]["in_norm"].dtype == np.float32  # vectors stay f32
