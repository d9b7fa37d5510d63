"""ctypes declarations of the C ABI in include/dec.h (argument marshalling only).

Loading fails loudly when libttsdec.so has not been built: there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libttsdec.so")

DEC_OK, DEC_E_ARG, DEC_E_POS, DEC_E_CAPACITY, DEC_E_UNSUPPORTED, DEC_E_CUDA, \
    DEC_E_DEVICE_CHECK = range(7)
STATUS_NAMES = {0: "DEC_OK", 1: "DEC_E_ARG", 2: "DEC_E_POS", 3: "DEC_E_CAPACITY",
                4: "DEC_E_UNSUPPORTED", 5: "DEC_E_CUDA", 6: "DEC_E_DEVICE_CHECK"}
DEC_QWEN3_TALKER, DEC_CODEC_WINDOWED = 0, 1
DEC_F32, DEC_BF16 = 0, 1
DEC_FLAG_TAPS, DEC_FLAG_NO_GRAPH, DEC_FLAG_PERSISTENT, DEC_FLAG_TENSOR_GEMV = 1, 2, 4, 8

# every symbol include/dec.h declares
EXPORTS = ("dec_create", "dec_destroy", "dec_last_error", "dec_set_stream", "dec_prefill_kv",
           "dec_prefill", "dec_prefill_block_rows", "dec_read_eos", "dec_step", "dec_step_host",
           "dec_set_mrope", "dec_step_mrope", "dec_prefill_mrope", "dec_reset", "dec_sync", "dec_get_len", "dec_read_kv",
           "dec_read_tap", "dec_kernels_per_step", "dec_truncate", "dec_launch_stage",
           "dec_gemv", "dec_attention_workspace_bytes", "dec_attention",
           "dec_attention_noalloc", "dec_flow_create", "dec_flow_step", "dec_flow_destroy",
           "dec_flow_last_error", "dec_flow_kernels_per_step", "dec_inject_stall")


class DecFlowConfig(C.Structure):
    _fields_ = [("dim", C.c_int32), ("latent", C.c_int32), ("cond", C.c_int32),
                ("blocks", C.c_int32), ("ln_eps", C.c_float), ("lsd_steps", C.c_int32)]


FLOW_BLOCK_FIELDS = ("ada_w", "ada_b", "ln_w", "ln_b", "m0_w", "m0_b", "m2_w", "m2_b")


class DecFlowWeights(C.Structure):
    _fields_ = ([(n, C.c_void_p) for n in ("ip_w", "ip_b", "cond_w", "cond_b", "t_const")] +
                [(n, C.POINTER(C.c_void_p)) for n in FLOW_BLOCK_FIELDS] +
                [(n, C.c_void_p) for n in ("fada_w", "fada_b", "f_w", "f_b")])


class DecConfig(C.Structure):
    _fields_ = [("kind", C.c_int32), ("layers", C.c_int32), ("hidden", C.c_int32),
                ("q_heads", C.c_int32), ("kv_heads", C.c_int32), ("head_dim", C.c_int32),
                ("inter", C.c_int32), ("norm_eps", C.c_float), ("rope_theta", C.c_double),
                ("weight_dtype", C.c_int32), ("max_pos", C.c_int32), ("ring", C.c_int32),
                ("window", C.c_int32), ("max_streams", C.c_int32), ("flags", C.c_uint32)]


LAYER_FIELDS = ("q", "k", "v", "o", "gate", "up", "down",
                "in_norm", "q_norm", "k_norm", "post_norm",
                "in_proj", "out_proj", "lin1", "lin2",
                "ln1_w", "ln1_b", "ln2_w", "ln2_b", "ls1", "ls2")


class DecLayerWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in LAYER_FIELDS]


class DecWeights(C.Structure):
    _fields_ = [("layers", C.POINTER(DecLayerWeights)), ("final_norm", C.c_void_p),
                ("final_norm_b", C.c_void_p), ("eos_w", C.c_void_p), ("eos_b", C.c_float)]


class DecError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


_lib = None
_lock = threading.Lock()


def load() -> C.CDLL:
    """Load libttsdec.so (built by tts_autoregressive_decode_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: the CUDA decode library has not been "
                               "built (python -m tts_autoregressive_decode_gb300.native_build)")
        L = C.CDLL(LIB_PATH)
        vp, i32, sz = C.c_void_p, C.c_int, C.c_size_t
        L.dec_create.argtypes = [C.POINTER(DecConfig), C.POINTER(DecWeights), vp, C.POINTER(vp)]
        L.dec_create.restype = i32
        L.dec_destroy.argtypes = [vp]
        L.dec_destroy.restype = None
        L.dec_last_error.argtypes = [vp]
        L.dec_last_error.restype = C.c_char_p
        L.dec_set_stream.argtypes = [vp, vp]
        L.dec_prefill_kv.argtypes = [vp, i32, vp, vp, i32]
        L.dec_prefill.argtypes = [vp, i32, i32, vp, vp]
        L.dec_prefill_block_rows.argtypes = [vp]
        L.dec_read_eos.argtypes = [vp, i32, vp]
        L.dec_flow_create.argtypes = [C.POINTER(DecFlowConfig), C.POINTER(DecFlowWeights), vp,
                                      C.POINTER(vp)]
        L.dec_flow_create.restype = i32
        L.dec_flow_step.argtypes = [vp, vp, vp, vp]
        L.dec_flow_step.restype = i32
        L.dec_flow_destroy.argtypes = [vp]
        L.dec_flow_destroy.restype = None
        L.dec_flow_last_error.argtypes = [vp]
        L.dec_flow_last_error.restype = C.c_char_p
        L.dec_flow_kernels_per_step.argtypes = [vp]
        L.dec_flow_kernels_per_step.restype = i32
        L.dec_prefill_block_rows.restype = i32
        L.dec_step.argtypes = [vp, i32, vp, C.POINTER(C.c_int32), vp]
        L.dec_set_mrope.argtypes = [vp, C.POINTER(C.c_int32), i32]
        L.dec_step_mrope.argtypes = [vp, i32, vp, C.POINTER(C.c_int32), vp, vp]
        L.dec_prefill_mrope.argtypes = [vp, i32, i32, vp, vp, vp]
        L.dec_step_host.argtypes = [vp, i32, vp, C.POINTER(C.c_int32), vp]
        L.dec_reset.argtypes = [vp, i32]
        L.dec_sync.argtypes = [vp]
        L.dec_get_len.argtypes = [vp, i32]
        L.dec_read_kv.argtypes = [vp, i32, i32, i32, vp, vp]
        L.dec_read_tap.argtypes = [vp, i32, i32, vp]
        L.dec_kernels_per_step.argtypes = [vp, i32]
        L.dec_truncate.argtypes = [vp, i32, i32]
        L.dec_inject_stall.argtypes = [vp, i32, i32]
        L.dec_launch_stage.argtypes = [vp, i32, i32, i32, i32]
        L.dec_gemv.argtypes = [i32, vp, i32, i32, vp, i32, vp, vp]
        L.dec_attention_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
        L.dec_attention_workspace_bytes.restype = sz
        L.dec_attention.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp]
        L.dec_attention_noalloc.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        for f in ("dec_set_stream", "dec_prefill_kv", "dec_step", "dec_step_host", "dec_reset",
                  "dec_sync", "dec_read_kv", "dec_read_tap", "dec_gemv", "dec_attention",
                  "dec_attention_noalloc",
                  "dec_truncate", "dec_launch_stage", "dec_prefill", "dec_read_eos",
                  "dec_set_mrope", "dec_step_mrope", "dec_prefill_mrope", "dec_inject_stall"):
            getattr(L, f).restype = i32
        L.dec_get_len.restype = i32
        L.dec_kernels_per_step.restype = i32
        _lib = L
        return L


def check(status: int, ctx=None) -> None:
    if status != DEC_OK:
        msg = load().dec_last_error(ctx).decode(errors="replace")
        raise DecError(status, msg)


def check_flow(status: int, head=None) -> None:
    if status != DEC_OK:
        msg = load().dec_flow_last_error(head).decode(errors="replace")
        raise DecError(status, msg)
