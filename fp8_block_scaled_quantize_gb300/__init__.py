"""GB300-native FP8 quantized actor linear layer.

Fine-grained FP8 E4M3 quantizers (1x128 groups for activations and gradients,
128x128 blocks for weights, fused 128x1 groups for WGrad), block-scaled FP8
GEMMs for FProp / DGrad / WGrad on tcgen05 tensor cores, and the UAQ
invariant-scaling fold, all in hand-written CUDA for sm_103a behind the C ABI
declared in ``include/rlq.h`` (``librlq.so``).

``fp8_block_scaled_quantize_gb300.rlq`` is the thin ctypes binding (it loads
the library on first use and raises if it is missing: there is no fallback);
``fp8_block_scaled_quantize_gb300.inputs`` draws the seeded synthetic inputs.
"""
