"""GB300-native MoE expert layer: routing, expert sort, permute, grouped GEMMs
(bf16 and fine-grained FP8) with fused SwiGLU, and the weighted combine.

The compute lives in ``libmoe.so`` (hand-written sm_103a CUDA behind a C ABI,
declared in ``include/moe.h``); :mod:`.moe` is its thin Python binding and
:mod:`.synth` draws the seeded synthetic inputs.
"""
__all__ = ["synth", "moe"]
