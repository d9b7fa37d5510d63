"""The benchmark's algorithmic byte counts, recomputed here from the layer shapes.

The roofline's "achieved" figure is these bytes over a measured time, so a change to the
workloads or to the accounting must show up as a failing number here."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from tts_autoregressive_decode_gb300 import workloads as W  # noqa: E402


def test_gate_up_launch_bytes_of_the_28_layer_talker():
    w = W.TALKER_H2048_L28
    stage, _, nbytes = bench.dominant_kernel(w, 1)
    assert stage == 3
    # 2 x 6144 interleaved bf16 rows of 2048, then x, the norm weight and the 6144 outputs in f32
    assert nbytes == 12288 * 2048 * 2 + 4 * (2048 + 2048 + 6144) == 50_372_608


def test_step_bytes_of_the_28_layer_talker_at_2048():
    w = W.TALKER_H2048_L28
    h, I, d, H, G, L = 2048, 6144, 128, 16, 8, 28
    weights = L * 2 * ((H + 2 * G) * d * h + h * H * d + 2 * I * h + h * I)
    vectors = 4 * (L * (2 * h + 2 * d) + h)          # two RMSNorms and q/k norms a layer, final norm
    kv = L * 2 * (2048 + 1) * G * d * 4              # K and V of 2049 keys
    assert bench.step_bytes(w, [2048]) == weights + vectors + kv
    assert bench.step_bytes(w, [2048]) == 3_289_059_328  # 3.30 GB averaged over 2048..2175


def test_codec_ring_bytes_do_not_depend_on_position():
    w = W.CODEC_D512_L8
    assert bench.kv_bytes(w, [0]) == bench.kv_bytes(w, [1000])
    assert bench.kv_bytes(w, [0]) == w.layers * (2 * w.ring * w.hidden * 4 + 4 * w.ring)


def test_throughput_counts_every_replica():
    assert bench.job_throughput(4, 100, 2.0) == 200.0
