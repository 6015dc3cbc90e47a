"""GB300-native NVFP4 weight path: quantiser and W4A16 GEMM with fused LoRA.

The compute lives in ``libnvfp4.so`` (hand-written CUDA for sm_103a behind a
C ABI, declared in ``include/nvfp4.h``).  :mod:`.binding` marshals arguments
to it; :mod:`.synth` draws seeded inputs.  Nothing here computes on the CPU.
"""
