/*
 * CPU oracle for the memory-bound decoder-layer fusions -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, fp64 C written from the definitions on the source pages. It shares no code with the
 * CUDA library (no common header, helper, table or constant) and is used only by the tests, by the
 * smoke check and by the bench's CPU-baseline leg. Nothing in the product path links or calls it.
 *
 * Sources (cited by page title and section):
 *  [P1] "TensorRT-LLM: Compiling Inference Engines Ahead of Time", section "Fusing operations, measured":
 *       the RMSNorm chain (float cast, square, mean, epsilon, reciprocal square root, scaling, cast back,
 *       weight) with the residual addition fused in front of it; the gated MLP takes gate and up from one
 *       stacked projection and combines them per element as g / (1 + exp(-g)) * up.
 *  [P2] "TensorRT-LLM" architecture walkthrough, "Part V continued: Deep dive: quantization co-designed
 *       with the hardware": activations in FP8 E4M3 with a per-tensor or per-block scale (the format is
 *       the one of Micikevicius et al., "FP8 Formats for Deep Learning"); its NVFP4 paragraph gives the
 *       Blackwell 4-bit format (E2M1 elements, an E4M3 scale per 16 of them, an fp32 scale per tensor).
 *  [P5] "Introduction to torch.compile and How It Works with vLLM", section 3 (custom passes): the SiLU
 *       activation and the FP8 quantisation that follows it are rewritten into a single fused kernel;
 *       section 4 reports AllReduce + RMSNorm (+ FP8 quantisation) fused as well.
 *
 * Conventions: bf16 values are passed as their 16-bit patterns (uint16_t), row-major. Every function
 * processes rows independently, so a caller may pass pointers offset to any row with a smaller T.
 * Return value: 0 on success, -1 on an invalid argument (null pointer with T > 0, T < 0, width <= 0).
 */
#ifndef MBD_ORACLE_H
#define MBD_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* bf16 pattern -> exact double. */
double orc_bf16_to_double(uint16_t b);
/* double -> nearest bf16 pattern, ties to even (8 significant bits, subnormals, overflow to inf). */
uint16_t orc_bf16_round(double v);
/* The exact sum of n finite bf16 values (n <= 8), rounded once to bf16, ties to even; a zero sum is +0. */
uint16_t orc_bf16_sum(const uint16_t* v, int n);

/* OCP E4M3FN: bias 7, 3 mantissa bits, max finite 448 (0x7E), no infinities, NaN 0x7F / 0xFF.
 * encode: nearest code by exhaustive search over the 127 non-negative finite magnitudes, ties to the
 * even code, magnitudes above 448 saturate to 448, the sign bit is set for negative inputs. */
double orc_e4m3_decode(uint8_t code);
uint8_t orc_e4m3_encode(double v);

/* E2M1, the NVFP4 element format [P2, NVFP4 paragraph]: a 4-bit float with a sign bit, 2 exponent bits and
 * 1 mantissa bit whose largest magnitude is 6. With exponent bias 1, codes 0..7 stand for 0, 0.5, 1, 1.5, 2,
 * 3, 4, 6 and bit 3 is the sign. encode: nearest magnitude by exhaustive search, ties to the even code,
 * anything above 6 saturates to 6, and the sign is kept on a zero. */
double orc_e2m1_decode(uint8_t code);
uint8_t orc_e2m1_encode(double v);

/* SiLU [P1]: g / (1 + exp(-g)). */
double orc_silu(double g);

/* Fused residual add + RMSNorm [P1]:
 *   s = bf16(x + r)                     -> residual_out (the updated residual stream)
 *   inv = 1 / sqrt(sum(s^2) / H + eps)
 *   v = w * s * inv                     -> v_out (exact, fp64) and out (bf16 of v)
 * v_out and out may be NULL. */
int orc_add_rmsnorm(const uint16_t* x, const uint16_t* r, const uint16_t* w, int64_t T, int64_t H,
                    float eps, uint16_t* residual_out, double* v_out, uint16_t* out);

/* mode: 0 = static per-tensor scale (scale[0] is read), 1 = dynamic per-token (scale[t] is written).
 * The scale is the dequantisation multiplier: v ~ q * scale. Dynamic: scale_t = fp32(max_j |v_j| / 448);
 * codes are e4m3(v / scale) with the fp32 scale widened to double; a zero scale gives code 0. */
int orc_add_rmsnorm_quant_fp8(const uint16_t* x, const uint16_t* r, const uint16_t* w, int64_t T,
                              int64_t H, float eps, int mode, float* scale, uint16_t* residual_out,
                              uint8_t* q_out, double* v_out);

/* The single-GPU half of the AllReduce + RMSNorm fusion [P5 s.4]: n partial activations (one per
 * tensor-parallel rank) are reduced to x = bf16(sum_k partial_k) -- the exact sum rounded once, what a
 * bf16 all-reduce hands to the next kernel -- and x then goes through the fused residual add + RMSNorm
 * above. The sum is carried in double: exact whenever the partials' exponents span fewer than ~45 bits
 * (every generated input), otherwise within 2^-53 relative. partials is an array of n row-major [T, H]
 * bf16 tensors, 1 <= n <= 8; n == 1 gives exactly orc_add_rmsnorm. */
int orc_allreduce_add_rmsnorm(const uint16_t* const* partials, int n, const uint16_t* r, const uint16_t* w,
                              int64_t T, int64_t H, float eps, uint16_t* residual_out, double* v_out,
                              uint16_t* out);
int orc_allreduce_add_rmsnorm_quant_fp8(const uint16_t* const* partials, int n, const uint16_t* r,
                                        const uint16_t* w, int64_t T, int64_t H, float eps, int mode,
                                        float* scale, uint16_t* residual_out, uint8_t* q_out, double* v_out);

/* NVFP4 quantisation [P2, NVFP4 paragraph: each run of 16 consecutive E2M1 elements carries an E4M3 scale and
 * the tensor as a whole an fp32 scale], applied to the unrounded row values v (the norm's v or SwiGLU's h). With S the per-tensor fp32 scale
 * (read; finite and > 0, else the call fails) and amax_b the largest |v| of 16-element block b:
 *     sf_b = E4M3(amax_b / (6 S))                 (the block scale, so that amax_b maps to about 6)
 *     q_j  = E2M1(v_j / (dec(sf_b) S))             (0 when dec(sf_b) == 0)
 * and v_j ~ dec(q_j) * dec(sf_b) * S. Outputs: q packed two codes per byte, element 2i in the low nibble,
 * [T, W/2]; sf [T, W/16] E4M3 codes, row-major. The width must be a multiple of 16. */
int orc_add_rmsnorm_quant_nvfp4(const uint16_t* x, const uint16_t* r, const uint16_t* w, int64_t T, int64_t H,
                                float eps, float tensor_scale, uint16_t* residual_out, uint8_t* q_out,
                                uint8_t* sf_out, double* v_out);
int orc_swiglu_quant_nvfp4(const uint16_t* gate_up, int64_t T, int64_t I, float tensor_scale, uint8_t* q_out,
                           uint8_t* sf_out, double* h_out);

/* SwiGLU over a stacked gate_up row [P1]: h[t,j] = silu(gu[t,j]) * gu[t,I+j], computed in fp64 with no
 * rounding of silu(g) before the product. h_out (exact) and out (bf16 of h) may be NULL. */
int orc_swiglu(const uint16_t* gate_up, int64_t T, int64_t I, double* h_out, uint16_t* out);

/* Quantize(SiLU(gate) * up) [P5], scale convention as for the norm. */
int orc_swiglu_quant_fp8(const uint16_t* gate_up, int64_t T, int64_t I, int mode, float* scale,
                         uint8_t* q_out, double* h_out);

#ifdef __cplusplus
}
#endif

#endif /* MBD_ORACLE_H */
