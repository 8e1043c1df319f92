"""Exact multi-head attention forward (tiled online softmax) for NVIDIA B300 (sm_103a).

The compute path is ``libattn.so`` (CUDA kernels behind a C ABI, declared in ``include/attn.h``);
``exact_tiled_attention_50_b300.attn`` is its thin Python binding. ``inputs`` draws the seeded
synthetic inputs used by the tests and the benchmark.
"""
