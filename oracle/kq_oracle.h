/*
 * kq_oracle.h -- reference (oracle) for k-quant super-block decoding and the
 * products built on it.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library may include, link
 * or call this code; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no source with the CUDA path.
 *
 * Sources followed (page title, section):
 *   "GGUF in transformers" (Hugging Face blog), section "What is the GGUF file
 *     format?" -- Q4_K_M mixes 4-bit tensors with higher-precision ones;
 *     section "Reusing ggml's Metal kernels" -- the quantization kernel reads
 *     packed weights directly, including only the selected MoE experts.
 *   "ANE Fieldfare" README (Show HN page), section "How it works" -- the router
 *     picks the top 8 of 128 experts, a shared FFN runs for every token.
 *   The byte layouts of Q4_K / Q5_K / Q6_K are not printed on the pages; this
 *   file encodes the public GGUF k-quant layout as read by this library
 *   (readings listed in the design notes), and the dequantization formulas
 *     Q4_K, Q5_K:  w = d * sc_j * q - dmin * m_j   (j = 32-weight sub-block)
 *     Q6_K:        w = d * sc_j * (q - 32)        (j = 16-weight sub-block)
 *   IA4 (group-affine INT4, "ANE Fieldfare" README, "Requirements": an
 *   mlx-community 4-bit checkpoint; MLX's affine form as read by this
 *   library): 144-byte blocks of 256 weights, 4 bf16 scales, 4 bf16 biases,
 *   128 code bytes (byte 32g+l: weight 64g+l low nibble, 64g+32+l high nibble)
 *     IA4:         w = scale_g * q + bias_g      (g = 64-weight group)
 *
 * Everything is computed in fp64; dequantized values are exact in fp64 for all
 * finite inputs whose fp16 exponents differ by less than ~30 binades, and are
 * rounded once to fp32 (round to nearest even) where an fp32 result is asked.
 */
#ifndef KQ_ORACLE_H
#define KQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_Q4_K = 1, ORACLE_Q5_K = 2, ORACLE_Q6_K = 3, ORACLE_IA4 = 4 };
enum { ORACLE_X_F32 = 0, ORACLE_X_BF16 = 1 };

/* bytes of one 256-weight super-block: 144 / 176 / 210, or 0 for a bad type */
int oracle_block_bytes(int type);

/* IEEE 754 binary16 / bfloat16 bit patterns -> double, from the definitions */
double oracle_half_to_double(uint16_t h);
double oracle_bf16_to_double(uint16_t b);

/* Unpacked integer fields of one block.
 *   Q4_K: d, dmin (fp16 bits), sc[0..7], m[0..7] in 0..63, q[0..255] in 0..15
 *   Q5_K: as Q4_K with q in 0..31
 *   Q6_K: d (fp16 bits), sc[0..15] in -128..127, q[0..255] in 0..63 (unbiased) */
typedef struct {
    uint16_t d_bits, dmin_bits;
    int sc[16];
    int m[8];
    int q[256];
} oracle_fields;

int  oracle_unpack(int type, const uint8_t *blk, oracle_fields *f);
int  oracle_pack(int type, const oracle_fields *f, uint8_t *blk);

/* Exact dequantized weights of one block (fp64). */
int  oracle_dequant_block_f64(int type, const uint8_t *blk, double w[256]);

/* n_blocks consecutive blocks -> n_blocks*256 fp32 values, each the fp64 value
 * rounded once to fp32. */
int  oracle_dequant(int type, const uint8_t *blocks, int64_t n_blocks, float *out);

/* y[m][n] = sum_{k<K} w[n][k] * x[m][k] in fp64, with s[m][n] = sum |w*x|.
 * W: N rows, each ceil(K/256) consecutive blocks (weights at k >= K are not
 * part of the matrix).  x: M rows of K values, fp32 or bf16 bit patterns.
 * y and s: M x N doubles (s may be NULL).  n_threads <= 1 runs serially. */
int  oracle_matvec(int type, const uint8_t *W, int64_t N, int64_t K,
                   const void *x, int x_dtype, int64_t M,
                   double *y, double *s, int n_threads);

/* Routed-expert product.  Expert e's matrix starts at W + e*N*ceil(K/256)*bytes.
 * ids[M][top_k]; x is [M][K] (x_per_slot = 0) or [M][top_k][K] (x_per_slot = 1).
 *   gate == NULL: y is [M][top_k][N], y[m][t] = W_{ids[m][t]} x_{m(,t)}
 *   gate != NULL: y is [M][N],        y[m]    = sum_t gate[m][t] * W_{ids[m][t]} x_{m(,t)}
 * s (optional) has y's shape and holds the matching sum of |terms|.
 * Returns -1 for a bad argument, -2 for an expert id outside [0, n_experts). */
int  oracle_moe_matvec(int type, const uint8_t *W_experts, int n_experts,
                       const int32_t *ids, const float *gate,
                       const void *x, int x_dtype, int x_per_slot,
                       int64_t N, int64_t K, int64_t M, int top_k,
                       double *y, double *s, int n_threads);

#ifdef __cplusplus
}
#endif
#endif
