"""CPU oracle for fine-grained FP8 quantisation and the block-scaled FP8 GEMM.

TEST INFRASTRUCTURE ONLY.  Nothing in the library calls this package: only
the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it.  It shares no code with the CUDA path.

What it computes follows DeepSeek-V3 "Infrastructure" §3.3 (FP8 training):
  * §3.3.2 "fine-grained quantization": activations are grouped and scaled
    per 1x128 tile (one token, 128 channels), weights per 128x128 block;
  * §3.3.2 "online quantization": the max absolute value of every tile or
    block is taken at use time, the scale follows from it and the values
    are cast to FP8;
  * §3.3.2 "mantissa over exponents": E4M3 for every tensor;
  * §3.3.2 "increasing accumulation precision": each N_C = 128 slice of the
    inner dimension is multiplied on the tensor cores, then dequantised by
    the product of the two group scales and added into an FP32 accumulator.
The explicit formulas are those of "DeepSeek-V3 FP8 动态量化" (Figure 7
explainer, section "Fine-grained quantization"): s_x = absmax / F_max,
FP8(x) = round(x / s_x), out += MMA(FP8(x), FP8(w)) * s_x * s_w.

Readings where the pages are silent (each is listed with its reason in the
design notes of the repository):
  * F_max = 448, the largest finite E4M3 value of the OCP "FN" encoding
    (1 sign, 4 exponent, 3 mantissa bits, bias 7, no infinities);
  * round() is round-to-nearest-even with saturation to +-448;
  * the quotient x / s is an IEEE float32 division, rounded once to float32
    before the rounding to E4M3;
  * the stored scale is s itself (float32), not 1/s;
  * a group whose absmax is 0 gets s = 0 and all-zero codes;
  * power-of-two ("rounded") scales, §3.3.3 (1): the smallest 2^k with
    absmax / 2^k <= 448;
  * the GEMM reference value of each 128-wide K block is its exact sum
    (computed in float64, where it is exact), scaled by s_a * s_b in
    float64 and summed over the blocks in float64.

Parity with DeepSeek's own kernels is unpinned: the pages print no code and
no numeric output of a quantised tile or GEMM.
"""
from .e4m3 import (E4M3_MAX, e4m3_decode, e4m3_encode, e4m3_all_finite_values)
from .quantize import (quantize_groups, quantize_act_1x128, quantize_act_128x1,
                       quantize_weight_128x128, bf16_bits_to_f32, pow2_scale,
                       dequantize_1x128, requant_1x128_to_128x1, swiglu, bf16_round_f64,
                       swiglu_quantize_1x128)
from .gemm import gemm_block_scaled, grouped_gemm_block_scaled, bf16_round
from .moe import moe_combine

__all__ = [
    "E4M3_MAX", "e4m3_decode", "e4m3_encode", "e4m3_all_finite_values",
    "quantize_groups", "quantize_act_1x128", "quantize_act_128x1",
    "quantize_weight_128x128", "bf16_bits_to_f32", "pow2_scale",
    "dequantize_1x128", "requant_1x128_to_128x1", "swiglu", "bf16_round_f64", "swiglu_quantize_1x128",
    "gemm_block_scaled", "grouped_gemm_block_scaled", "bf16_round", "moe_combine",
]
