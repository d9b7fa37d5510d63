"""GB300-native (sm_103a) single-token autoregressive decode step of a Qwen3-style TTS talker
layer stack, plus its windowed KV-ring (codec) variant, behind a C ABI (include/dec.h).

    build()                       compile libttsdec.so in-tree (nvcc, sm_103a)
    Decoder                       a decode context over device-resident weights
    gemv, attention               the stateless kernel entry points
    workloads                     the synthetic, seeded workload definitions
"""
import importlib

__all__ = ["Decoder", "gemv", "attention", "attention_workspace_bytes", "build"]


def build(force: bool = False) -> str:
    return importlib.import_module(__name__ + ".native_build").build(force=force)


def __getattr__(name):
    if name in ("Decoder", "gemv", "attention", "attention_workspace_bytes"):
        return getattr(importlib.import_module(__name__ + ".decoder"), name)
    raise AttributeError(name)
