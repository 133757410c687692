/*
 * moe_oracle.h -- CPU oracle for the fused MoE expert layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * and its Python binding) may include, link, load or call this code.  Only
 * the test suite, the smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no source with the CUDA path.
 *
 * What it computes (plain, slow, obviously correct):
 *   top-k routing with a softmax over the selected logits, a stable counting
 *   sort of the (token, k) slots into expert-contiguous order, per-expert
 *   W13 GEMM on exactly dequantised operands, SwiGLU with optional gate/up
 *   clamp (or the non-gated ReLU^2), re-quantisation of the GEMM2 input,
 *   per-expert W2 GEMM and the routing-weighted top-k combine; and the same
 *   expert computation on the batched-expert input format.  Sources:
 *     - "PR #40082 report: Integrate flashinfer b12x MoE and FP4 GEMM kernels
 *       for SM120/121" (prhub.com.cn), sec. 实现拆解 item 1: the layer's steps
 *       (routing, the gate/up GEMM, SwiGLU, the down GEMM, the reduction)
 *       in one call that receives bf16 activations and quantises them.
 *     - same page, sec. 关键源码片段 (process_weights_after_loading): the
 *       per-expert fp32 global weight scale is multiplied into the block
 *       scales, the product re-cast to the block-scale type, and the global
 *       scale set to 1; the activation global scale is 1 because the kernel
 *       quantises activations dynamically per block.
 *     - "FlashInfer CuTeDSL MegaMoE kernel-drop update workflow"
 *       (bjdmk.com.cn/news/5453900), sec. 三 (kernel_helpers re-exports):
 *       NVFP4 blocks of 16 (nvfp4_quantize_per_block_16), MXFP8 blocks of 32
 *       (mxfp8_quantize_per_block_32), and sec. 三 (comm.py): an optional
 *       gate/up clamp (resolve_gate_up_clamp).
 *     - same PR #40082 page, sec. 风险与影响 item 4: MoE models without a
 *       gated act-and-mul MLP, such as Nemotron's ReLU^2 experts.
 *     - "PR 38050 analysis report" (prhub.com.cn, vLLM PR 38050), sec.
 *       实现拆解: the batched-experts variant that takes activations already
 *       grouped per expert ([E, max tokens per expert, H] plus per-expert
 *       counts) and returns the expert outputs in the same layout.
 *   The element formats themselves (e2m1, e4m3 "fn", e8m0, bf16) are the
 *   public OCP Microscaling v1.0 / OCP 8-bit float definitions.
 *
 * Arithmetic: every dot product is accumulated in double and rounded once to
 * fp32 (the width of the GPU accumulator).  Quantisation decisions (block
 * amax, scale, element codes) are taken in fp32, the precision the kernels
 * take them in.  GEMM2 output is kept in fp32 (not rounded to bf16).
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_FMT_BF16 = 0, ORC_FMT_MXFP8 = 1, ORC_FMT_NVFP4 = 2 };

/* ---- element codecs --------------------------------------------------- */
float    orc_bf16_to_f32(uint16_t b);
uint16_t orc_f32_to_bf16(float x);            /* round to nearest even */
float    orc_e4m3_to_f32(uint8_t c);          /* OCP e4m3 "fn": 0x7F/0xFF NaN */
uint8_t  orc_f32_to_e4m3(float x);            /* RNE, saturate to +-448 */
float    orc_e2m1_to_f32(uint8_t c);          /* low 4 bits: s e e m */
uint8_t  orc_f32_to_e2m1(float x);            /* RNE, saturate to +-6 */
float    orc_e8m0_to_f32(uint8_t c);          /* 2^(c-127); 0xFF NaN */

/* ---- block quantisers (one block) -------------------------------------
 * NVFP4, 16 elements: sf = e4m3(amax/6), q_i = e2m1(x_i / sf) (both
 * divisions fp32, correctly rounded); sf == 0 gives all-zero codes.
 * codes[] receives one 4-bit code per byte (unpacked).
 * MXFP8, 32 elements: X = floor(log2 amax) - 8 clamped to [-127,127],
 * sf = X + 127 (e8m0), q_i = e4m3(x_i * 2^-X); amax == 0 gives sf = 127 and
 * zero codes.                                                              */
void orc_quant_nvfp4_block16(const float *x, uint8_t *codes, uint8_t *sf);
void orc_quant_mxfp8_block32(const float *x, uint8_t *codes, uint8_t *sf);

/* Quantise a row of n values (n a multiple of the block) into the canonical
 * packed layout: NVFP4 two codes per byte, element 2j in the low nibble;
 * MXFP8 one e4m3 byte per element.  sf gets n/16 (NVFP4) or n/32 (MXFP8)
 * bytes.  Returns 0, or -1 for BF16 / bad n.                              */
int orc_quant_row(int fmt, const float *x, int n, uint8_t *codes, uint8_t *sf);

/* Dequantise a canonical packed row back to fp32 (exact).                 */
int orc_dequant_row(int fmt, const uint8_t *codes, const uint8_t *sf, int n,
                    float *out);

/* NVFP4 global-scale fold: out[i] = e4m3(float(sf[i]) * gs) (fp32 product). */
void orc_fold_scales(const uint8_t *sf, int64_t n, float gs, uint8_t *out);

/* ---- routing and permutation ------------------------------------------ */
/* ids[t*K+k]: k-th best expert (value descending, index ascending on ties);
 * w[t*K+k] = exp(l_k - l_max) / sum_j exp(l_j - l_max) over the K selected. */
void orc_route(const float *logits, int T, int E, int K, int32_t *ids,
               float *w);
/* Stable counting sort of slots s = t*K+k by expert: offsets[E+1],
 * perm[row] = slot, inv[slot] = row.                                      */
void orc_permute(const int32_t *ids, int T, int K, int E, int32_t *offsets,
                 int32_t *perm, int32_t *inv);

/* ---- the layer -------------------------------------------------------- */
enum { ORC_ACT_SWIGLU = 0, ORC_ACT_RELU2 = 1 };

typedef struct {
    int H, I, E, K, fmt;
    float clamp;          /* > 0 and finite: clamp gate and up to [-L, L] */
    int act;              /* ORC_ACT_SWIGLU (gated, W13 has 2I rows) or
                             ORC_ACT_RELU2 (non-gated, W13 has I rows:
                             h = max(G, 0)^2; no clamp)                  */
} orc_cfg;

/* Canonical weights (row-major, reduction dim contiguous):
 *   BF16 : w13 uint16 [E,2I,H], w2 uint16 [E,H,I]; sf, gs unused
 *   MXFP8: w13 e4m3 [E,2I,H], w13_sf e8m0 [E,2I,H/32]; w2 [E,H,I], [E,H,I/32]
 *   NVFP4: w13 u8 [E,2I,H/2], w13_sf e4m3 [E,2I,H/16], w13_gs f32 [E];
 *          w2 u8 [E,H,I/2], w2_sf e4m3 [E,H,I/16], w2_gs f32 [E]
 * Rows 0..I-1 of W13 are the gate projection, rows I..2I-1 the up one.
 * With ORC_ACT_RELU2, W13 is the single up projection [E,I,H] (likewise for
 * its scales).                                                             */
typedef struct {
    const void *w13; const uint8_t *w13_sf; const float *w13_gs;
    const void *w2;  const uint8_t *w2_sf;  const float *w2_gs;
} orc_weights;

/* Whole layer over T tokens.  hidden bf16 [T,H], logits f32 [T,E],
 * out bf16 [T,H].  Optional outputs (NULL to skip): ids/w [T*K],
 * offsets [E+1], perm [T*K], xq_codes/xq_sf (the GEMM1 input quantisation
 * per token, canonical layout; NV/MX only), h [T*K, I] (GEMM2 input after
 * re-quantisation, dequantised, in permuted row order), y [T*K, H] (GEMM2
 * output, fp32, permuted row order).  Returns 0 or a negative error.     */
int orc_forward(const orc_cfg *cfg, const orc_weights *wt,
                const uint16_t *hidden, const float *logits, int T,
                uint16_t *out, int32_t *ids, float *w, int32_t *offsets,
                int32_t *perm, uint8_t *xq_codes, uint8_t *xq_sf, float *h,
                float *y);

/* Brute force for one token, no permutation: out_f32[j] (before bf16
 * rounding) and out[j] = bf16(out_f32[j]).                              */
int orc_token_forward(const orc_cfg *cfg, const orc_weights *wt,
                      const uint16_t *hidden_row, const float *logits_row,
                      float *out_f32, uint16_t *out);

/* Batched-expert format: no routing, permutation or combine.  hidden bf16
 * [E,M,H]: expert e's rows are rows 0..counts[e]-1 of block e (counts[e]
 * <= M).  Each such row goes through GEMM1 input quantisation, GEMM1, the
 * activation with re-quantisation and GEMM2 of expert e; out bf16 [E,M,H]
 * receives bf16(GEMM2 output) in the same rows (other rows are left as
 * they are); y (optional) the fp32 GEMM2 output.  Returns 0 or -1.       */
int orc_forward_batched(const orc_cfg *cfg, const orc_weights *wt,
                        const uint16_t *hidden, const int32_t *counts, int M,
                        uint16_t *out, float *y);

/* Bulk codec helpers (tests): kind 0 bf16 (uint16 codes), 1 e4m3,
 * 2 e2m1 (one code per byte), 3 e8m0.  Encoding e8m0 is not defined.  */
int orc_encode_n(int kind, const float *x, int64_t n, void *codes);
int orc_decode_n(int kind, const void *codes, int64_t n, float *x);

/* Number of threads the OpenMP runtime will use (1 without OpenMP).    */
int orc_num_threads(void);
void orc_set_num_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
