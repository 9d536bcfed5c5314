/*
 * kq.h -- C ABI of libkq: decode-time products against GGUF k-quant weights
 * on one NVIDIA GB300 (sm_103a).
 *
 * What the library computes (sources: page title, section):
 *   "GGUF in transformers" (Hugging Face blog), "What is the GGUF file
 *     format?": Q4_K_M checkpoints keep most tensors in 4-bit k-quants and the
 *     sensitive ones in Q6_K; Q5_K_M and Q6_K are the larger variants.
 *   same page, "Reusing ggml's Metal kernels": the quantization kernel reads
 *     the packed weights directly for matrix operations, including only the
 *     experts an MoE layer selected, instead of expanding the whole matrix
 *     before each decode step.
 *   same page, "Fine-tune from a GGUF checkpoint" / "Load GGUF with
 *     transformers": the fallback that dequantizes weights (kq_dequant).
 *   "ANE Fieldfare" README (Show HN page), "How it works": each token's router
 *     picks 8 of 128 experts and a shared FFN runs for every token;
 *     "Speculative decoding": verify blocks of up to 16 tokens, so products
 *     run for M = 1..16 tokens at once.
 *
 * Block formats (256 weights each; little-endian; the byte layout is the
 * public GGUF layout as this library reads it -- the pages do not print it):
 *   KQ_Q4_K  144 B: d fp16 | dmin fp16 | 12 B: 8 six-bit scales, 8 six-bit
 *            mins | 128 B 4-bit codes.   w = d*sc_j*q - dmin*m_j, j = 32-weight sub-block
 *   KQ_Q5_K  176 B: as Q4_K with 32 B of 5th code bits before the codes (q in 0..31).
 *   KQ_Q6_K  210 B: 128 B low nibbles | 64 B high bit pairs | 16 int8 scales | d fp16.
 *            w = d*sc_j*(q - 32), j = 16-weight sub-block, q in 0..63
 *   KQ_IA4   144 B: 4 bf16 scales | 4 bf16 biases | 128 B 4-bit codes in the
 *            Q4_K code order (byte 32g+l: weight 64g+l low nibble, 64g+32+l
 *            high nibble).  w = scale_g*q + bias_g, g = 64-weight group.
 *            Group-affine INT4 ("ANE Fieldfare" README, "Requirements": the
 *            experts come from an mlx-community 4-bit checkpoint; the pages do
 *            not print its layout -- this library takes MLX's affine form,
 *            groups of 64, bf16 scales and biases), regrouped from MLX's
 *            arrays by kq_ia4_pack.  Not accepted by kq_unpack or chains.
 *
 * Matrices: W has N rows; row n is ceil(K/256) consecutive blocks, rows are
 * consecutive (no padding).  Weights at positions k >= K in a row's last block
 * are not part of the matrix and are never used.  K must be a multiple of 32.
 * x is M rows of K values (row-major, fp32 or bfloat16); y is M rows of N
 * fp32 values (row-major).
 *
 * Memory and ownership: every pointer argument is a device pointer owned by
 * the caller.  The library allocates nothing, keeps no per-call state and does
 * not synchronize; work is enqueued on `stream` (0 = legacy default stream).
 * W must be 16-byte aligned; its allocation must be readable up to the next
 * 16-byte boundary past its last byte (always true for cudaMalloc and the
 * PyTorch caching allocator).  x must be 16-byte aligned; y 4-byte aligned.
 * Outputs must not overlap inputs.
 *
 * Ordering: kernels are launched with programmatic stream serialization.
 * Before waiting for the preceding kernel on the stream they read only W
 * (and the expert weights), so W must not be written by the immediately
 * preceding kernel; x, y, ids and gates are accessed only after that kernel
 * has completed.
 *
 * Errors: argument errors are returned before anything is enqueued.  A failed
 * launch returns KQ_ERR_CUDA (the CUDA error is available from
 * kq_last_cuda_error).  Kernels never trap: a problem found on the device
 * (an expert id out of range, a bounded wait that expired) is recorded in the
 * library's device error word, read with kq_device_error.
 */
#ifndef KQ_H
#define KQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *kq_stream_t; /* same type as cudaStream_t */

typedef enum { KQ_Q4_K = 1, KQ_Q5_K = 2, KQ_Q6_K = 3, KQ_IA4 = 4 } kq_type;
typedef enum { KQ_F32 = 0, KQ_BF16 = 1 } kq_dtype;

typedef int kq_status;
#define KQ_OK 0
#define KQ_ERR_ARG (-1)         /* null pointer, negative size, bad dtype       */
#define KQ_ERR_TYPE (-2)        /* unknown block type                           */
#define KQ_ERR_SHAPE (-3)       /* K not a multiple of 32, n not a multiple of 256 */
#define KQ_ERR_UNSUPPORTED (-4) /* a size outside the path's limits (M, top_k, K) */
#define KQ_ERR_ALIGN (-5)       /* pointer alignment rule broken                 */
#define KQ_ERR_CUDA (-6)        /* a CUDA call failed (see kq_last_cuda_error)   */
#define KQ_ERR_WORKSPACE (-7)   /* workspace missing or too small                */
#define KQ_ERR_DEVICE (-8)      /* the device error word was set (kq_device_error) */

/* Bytes of one 256-weight block: 144, 176, 210, 144; 0 for an unknown type. */
size_t kq_block_bytes(int type);

/*
 * Regroup a group-affine INT4 matrix in MLX's layout into KQ_IA4 blocks.
 *   q       [N][K/8] uint32: code k of a row in bits 4(k%8)..4(k%8)+3 of word k/8
 *   scales  [N][K/64] bf16 bit patterns, biases [N][K/64]: group G covers
 *           weights 64G..64G+63, w = scale*q + bias
 *   blocks  [N][ceil(K/256)] KQ_IA4 blocks (16-byte aligned); groups past K
 *           in a row's last block get zero scale, bias and codes.
 * K a multiple of 64 (else KQ_ERR_SHAPE); q 4-byte, scales and biases 2-byte
 * aligned.  Stream-ordered, one launch; a load-time conversion, not a product.
 */
kq_status kq_ia4_pack(const uint32_t *q, const uint16_t *scales, const uint16_t *biases, int64_t N, int64_t K,
                      void *blocks, kq_stream_t stream);

/*
 * Integer fields of n_blocks consecutive blocks (the super-block unpacker the
 * products use, exposed for inspection).  Any output may be NULL.  k-quant
 * types only (KQ_IA4 blocks have no such fields: KQ_ERR_TYPE).
 *   codes     [n_blocks][256] uint8: q (Q4_K 0..15, Q5_K 0..31, Q6_K 0..63, unbiased)
 *   scales    [n_blocks][16]  int8 : Q4_K/Q5_K sc_0..sc_7 (0..63, entries 8..15
 *                                    untouched); Q6_K sc_0..sc_15 (-128..127)
 *   mins      [n_blocks][8]   uint8: Q4_K/Q5_K m_0..m_7 (untouched for Q6_K)
 *   d_bits    [n_blocks]      fp16 bit pattern of d
 *   dmin_bits [n_blocks]      fp16 bit pattern of dmin (untouched for Q6_K)
 */
kq_status kq_unpack(int type, const void *blocks, int64_t n_blocks, uint8_t *codes, int8_t *scales,
                    uint8_t *mins, uint16_t *d_bits, uint16_t *dmin_bits, kq_stream_t stream);

/*
 * Dequantize n weights (n a multiple of 256) stored as n/256 consecutive
 * blocks into fp32: out[i] = the exact weight rounded once to fp32.
 * blocks: 16-byte aligned.  out: 16-byte aligned, n floats.
 */
kq_status kq_dequant(int type, const void *blocks, float *out, int64_t n, kq_stream_t stream);

/*
 * The same weights as kq_dequant, written as bfloat16 bit patterns: out[i] is
 * kq_dequant's fp32 out[i] rounded to the nearest bf16, ties to even (a NaN
 * stays a NaN).  The expansion "GGUF in transformers" describes for
 * GgufConfig(dequantize=True, dtype=torch.bfloat16) ("Load GGUF with
 * transformers"), at half the bytes written of the fp32 form.
 * blocks: 16-byte aligned.  out: 16-byte aligned, n uint16 values.  n a
 * multiple of 256.  Errors as kq_dequant.
 */
kq_status kq_dequant_bf16(int type, const void *blocks, uint16_t *out, int64_t n, kq_stream_t stream);

/*
 * y[m][n] = sum_{k<K} w[n][k] * x[m][k] for m < M, n < N, dequantizing W on
 * the fly (each weight byte is read from memory once per call).
 *   x_dtype KQ_F32 or KQ_BF16; M in 1..16; K a multiple of 32.
 * Accumulation is fp32 in a fixed order, so repeated calls give identical y;
 * the order (hence the last bits of y) differs between paths: M = 1, and
 * M = 2..4 with bf16 x when M x images fit beside the weight ring in shared
 * memory (exact integer dots per block; each row then equals that token's
 * M = 1 product bit for bit); otherwise M = 2..16 with bf16 x on the tensor
 * cores (weights rounded to bf16); M >= 2 with fp32 x on the CUDA cores.
 * Accuracy, for finite x and weights and partial sums in fp32's normal range:
 * |y - y_exact| <= e * sum_k |w[n][k] x[m][k]|, where
 *   - M = 1, and M = 2..4 with bf16 x: x is held exactly in shared memory (per
 *     256 values a 24-bit integer image with a power-of-two scale; the values
 *     off its grid listed beside it, or, past 32 of them, the whole block kept
 *     as bf16; fp32 x as two bf16 parts hi and lo, dropping <= 2^-18 |x|).
 *     Each lane's 128-weight half-block sum d*Y - dmin*Mi is formed from
 *     exact integers and rounded to fp32 where that is provably within a
 *     bound of the exact value, else exactly (one rounding): within 2^-11 for
 *     bf16 x and for the lo part, within 4.6e-5 for the hi part of fp32 x.
 *     Listed and kept values add fl(w x), w the exactly rounded weight.
 *     bf16 x:  e <= 2^-11 + 2^-24 D;
 *     fp32 x:  e <= 4.6e-5 + 2^-19 + 2^-18 + 2^-24 D (below 1e-4: this path
 *     takes K <= 16384), D = 3 ceil(K/256) + 40 bounding the fp32 additions
 *     from a term to y;
 *   - tensor cores (bf16 x): each weight rounded once to fp32, then to bf16:
 *     e <= 2^-8 + 2^-24 (ceil(K/16) + 8), taking each 16-term MMA step as one
 *     rounding into the fp32 accumulator;
 *   - M >= 2 with fp32 x: each weight rounded once to fp32, fp32 FMAs:
 *     e <= 2^-24 (2 ceil(K/256) + 16).
 */
kq_status kq_matvec(int type, const void *W, const void *x, int x_dtype, float *y, int64_t N, int64_t K,
                    int64_t M, kq_stream_t stream);

/*
 * Chains of one-token products run by one persistent launch.
 *
 * "GGUF in transformers", "Keeping the CPU and GPU working together": a
 * decode step is a sequence of products, and the device should not idle
 * between them.  A chain runs n_ops products y_i = W_i x_i (one token each)
 * in one launch: weights stream continuously across op boundaries, and an op
 * with wait_previous != 0 reads its x only after every earlier op of the
 * chain has finished (a grid-wide barrier), so x_i may be computed from
 * earlier outputs by the caller's own kernels only between runs, or be an
 * earlier op's y.  Ops without wait_previous may run concurrently with the
 * ops before them and must not read their outputs.
 *
 * Usage: size = kq_chain_workspace_size(ops, n); allocate a device workspace
 * of that many bytes (256-byte aligned); kq_chain_prepare once (synchronous:
 * it plans the chain and copies it into the workspace); then kq_chain_run any
 * number of times.  The pointers and shapes of the ops are fixed by prepare;
 * the data behind them may change between runs.  The workspace (owned by the
 * caller) holds the compiled chain, grid-barrier counters and split-K
 * partial sums; two runs must not use one workspace at the same time.
 */
typedef struct kq_op {
  int32_t type;          /* KQ_Q4_K, KQ_Q5_K or KQ_Q6_K (not KQ_IA4)            */
  int32_t x_dtype;       /* KQ_F32 or KQ_BF16                                   */
  int32_t wait_previous; /* nonzero: start after all earlier ops have finished  */
  int32_t reserved;      /* must be 0                                           */
  const void *W;         /* N x ceil(K/256) blocks, 16-byte aligned             */
  const void *x;         /* K values, 16-byte aligned                           */
  float *y;              /* N floats, 4-byte aligned                            */
  int64_t N, K;          /* N >= 1; K a multiple of 32, at most 16384           */
} kq_op;

typedef struct kq_chain_plan {
  int64_t opaque[8];
} kq_chain_plan;

/* Workspace bytes for the chain; 0 if an op's shape is outside this path. */
size_t kq_chain_workspace_size(const kq_op *ops, int n_ops);

/*
 * Plan the chain into workspace and *plan.  Errors: KQ_ERR_ARG (null or
 * overlapping buffers: an op's y may not overlap any W, any x of the same or
 * an earlier op, or an x read before the next wait_previous), KQ_ERR_TYPE,
 * KQ_ERR_SHAPE, KQ_ERR_UNSUPPORTED (K > 16384), KQ_ERR_ALIGN,
 * KQ_ERR_WORKSPACE (workspace NULL, misaligned or smaller than
 * kq_chain_workspace_size).  Enqueues copies on stream and synchronizes it.
 */
kq_status kq_chain_prepare(const kq_op *ops, int n_ops, void *workspace, size_t workspace_bytes,
                           kq_chain_plan *plan, kq_stream_t stream);

/*
 * Run a prepared chain on stream.  A chain with wait_previous ops is a
 * cooperative launch (one CTA per SM must be able to start, else
 * KQ_ERR_CUDA).  A chain without them (independent products sharing one
 * launch, e.g. q|k|v) is an ordinary launch with programmatic stream
 * serialization, like kq_matvec.
 */
kq_status kq_chain_run(const kq_chain_plan *plan, void *workspace, kq_stream_t stream);

/*
 * Routed-expert products (MoE decode and verify blocks).
 *
 * "GGUF in transformers", "Reusing ggml's Metal kernels": only the experts an
 * MoE layer selected are read.  "ANE Fieldfare" README, "How it works": each
 * token's router picks top_k of n_experts (8 of 128).
 *
 *   W_experts   n_experts matrices of N rows x ceil(K/256) blocks, back to
 *               back: expert e starts at W_experts + e*N*ceil(K/256)*block_bytes
 *   expert_ids  [M][top_k] int32
 *   gate_w      [M][top_k] fp32, or NULL
 *   x           [M][K] (x_per_slot = 0) or [M][top_k][K] (x_per_slot = 1)
 *   y           gate_w != NULL: [M][N],  y[m] = sum_j gate_w[m][j] * W_{ids[m][j]} x_{m(,j)}
 *               gate_w == NULL: [M][top_k][N], y[m][j] = W_{ids[m][j]} x_{m(,j)}
 *
 * The (token, slot) pairs are grouped by expert on the device, and every
 * distinct routed expert's rows are read from memory once per call.  Sums
 * are fp32 in a fixed order (the gate-weighted sum adds slots in order).
 * Accuracy: each pair's product takes kq_matvec's M = 1 arithmetic (the same
 * exact x image and per-lane combine), so each y[m][j] (or each gated term
 * g y) is within kq_matvec's M = 1 bound with D increased by 2 + top_k.
 * An id outside [0, n_experts) never faults: its pair is dropped (no
 * contribution; without gate_w its output row is not written) and the
 * workspace's error word is set (kq_moe_check).
 *
 * workspace: kq_moe_workspace_size(N, M, top_k, n_experts) bytes of device
 * memory, 256-byte aligned, zero-filled once before first use (arrival
 * counters return to zero after every call); one call at a time per
 * workspace.  After a call it holds the grouping, for inspection: at byte
 * 256, int32 D (distinct experts), expert[Dmax] (ascending ids),
 * offset[Dmax + 1], pair[M*top_k] (pair index m*top_k + j, grouped by expert,
 * (m, j) order within an expert), Dmax = min(n_experts, M*top_k).
 *
 * Limits: M*top_k <= 512, n_experts <= 4096, K a multiple of 32, 32 rows of
 * one expert at most 100 KB (K <= 5632 for Q4_K, 4608 for Q5_K, 3584 for
 * Q6_K); else KQ_ERR_UNSUPPORTED.
 */
size_t kq_moe_workspace_size(int64_t N, int64_t M, int32_t top_k, int32_t n_experts);

kq_status kq_moe_matvec(int type, const void *W_experts, int32_t n_experts, const int32_t *expert_ids,
                        const float *gate_w, const void *x, int x_dtype, int x_per_slot, float *y, int64_t N,
                        int64_t K, int64_t M, int32_t top_k, void *workspace, size_t workspace_bytes,
                        kq_stream_t stream);

/*
 * kq_moe_matvec without a workspace: the same product, with its scratch in a
 * fixed 2 MiB array inside libkq (one per device).  The pages have no
 * counterpart of this call: it exists for callers that cannot allocate
 * device memory (a C host with no device allocator, or a decode loop that
 * must not allocate), which therefore cannot pass the workspace above.
 *   - Limit: the call returns KQ_ERR_WORKSPACE when the workspace
 *     kq_moe_workspace_size(N, M, top_k, n_experts) would exceed 2 MiB.
 *   - It allocates nothing.  The first call on each device looks up the
 *     array's address once (cudaGetSymbolAddress); make that first call
 *     before any stream capture begins.
 *   - The array keeps what the last call left, laid out for that call's
 *     shape; a call with gate_w first clears its own arrival counters (a
 *     stream-ordered cudaMemsetAsync on the array, which allocates nothing).
 *     A routed id out of range is reported in the library's device error
 *     word (kq_device_error), not in a workspace.
 *   - Calls that overlap in time (on any stream or host thread) share the
 *     array and race: issue them one after another.
 */
kq_status kq_moe_matvec_noalloc(int type, const void *W_experts, int32_t n_experts, const int32_t *expert_ids,
                                const float *gate_w, const void *x, int x_dtype, int x_per_slot, float *y,
                                int64_t N, int64_t K, int64_t M, int32_t top_k, kq_stream_t stream);

/*
 * Self-test of the kernels' bounded waits: launches one small kernel whose
 * wait can never succeed -- kind 0 an mbarrier that no copy completes, kind 1
 * a grid-barrier counter that no CTA increments -- through the same wait
 * functions the products use, with a short poll limit (milliseconds).  The
 * wait gives up, sets a self-test error word (not the library's) and the
 * kernel returns.  Synchronizes stream; *observed_code receives the code the
 * wait recorded: 1 (wait timed out) when the mechanism works.  The context
 * stays usable afterwards.  Errors: KQ_ERR_ARG (kind not 0/1, NULL
 * observed_code), KQ_ERR_CUDA.
 */
kq_status kq_selftest_wait(int kind, int *observed_code, kq_stream_t stream);

/*
 * Synchronize stream and read the workspace's error word: KQ_ERR_DEVICE if a
 * routed id was out of range since the last check (the word is then
 * cleared), else KQ_OK.
 */
kq_status kq_moe_check(void *workspace, kq_stream_t stream);

/*
 * The MoE router: for each of M tokens, the top_k experts of its n_experts
 * router logits and their gate weights, and optionally the grouping of the
 * (token, slot) pairs by expert.
 *
 * "GGUF in transformers", "Reusing ggml's Metal kernels": a top-k kernel
 * combining softmax and top-k routing; "ANE Fieldfare" README, "How it works"
 * (8 of 128 experts per token) and "Speculative decoding" (a GPU planning
 * kernel groups a verify block's tokens by expert).
 *
 *   logits      [M][n_experts] fp32 (device).
 *   expert_ids  [M][top_k] int32: the top_k largest logits of each token in
 *               descending order; equal logits in ascending expert order; a
 *               NaN logit ranks below every number.
 *   gate_w      [M][top_k] fp32: exp(l_j - l_0) / sum_i exp(l_i - l_0) over the
 *               selected logits l_0 >= l_1 >= ... (a softmax over all experts,
 *               renormalized over the selected ones).
 *   workspace   NULL, or a kq_moe_matvec workspace (256-byte aligned): the
 *               grouping is written in the plan layout kq_moe_matvec leaves
 *               there (at byte 256: D, expert[Dmax], offset[Dmax+1], pairs),
 *               Dmax = min(M*top_k, n_experts).
 * Limits: M*top_k <= 512, n_experts <= 4096, 1 <= top_k <= min(32, n_experts)
 * (else KQ_ERR_UNSUPPORTED).  Stream-ordered (programmatic dependent launch).
 */
kq_status kq_moe_route(const float *logits, int64_t M, int32_t n_experts, int32_t top_k, int32_t *expert_ids,
                       float *gate_w, void *workspace, size_t workspace_bytes, kq_stream_t stream);

/*
 * The expert FFN of one MoE layer: routed experts plus an optional shared
 * expert, gate|up -> activation -> down -> gate-weighted combine.
 *
 * "ANE Fieldfare" README, "How it works": each layer runs a shared FFN that
 * every token goes through plus the 8 routed experts it picked, each a small
 * feed-forward block.  The pages give neither the activation nor the order of
 * the final sums; this library takes the gated form
 *   h_j  = act(W_gate[e_j] x) * (W_up[e_j] x)        (e_j = expert_ids[m][j])
 *   hs   = act(Ws_gate x) * (Ws_up x)
 *   y[m] = sum_j gate_w[m][j] * (W_down[e_j] h_j)  +  Ws_down hs
 * with the routed terms added in slot order and the shared term last, all in
 * fp32 (h kept in fp32).  act is a parameter:
 *   KQ_ACT_SILU       g / (1 + exp(-g))
 *   KQ_ACT_GELU_TANH  0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3)))
 *
 * Weights (device, 16-byte aligned, same block layout as kq_matvec):
 *   W_gate, W_up  [n_experts][F][H/256 blocks] of type_gate_up
 *   W_down        [n_experts][H][F/256 blocks] of type_down
 *   Ws_gate, Ws_up [SH][H/256 blocks] (type_gate_up), Ws_down [H][SH/256 blocks]
 *                 (type_down); all NULL and SH = 0 for no shared expert.
 * x [M][H] fp32 or bf16 (16-byte aligned); y [M][H] fp32; expert_ids, gate_w
 * [M][top_k] (an id outside [0, n_experts) drops its pair and sets the
 * workspace error word, read by kq_moe_check).
 * Two launches on stream (programmatic dependent launch); the workspace
 * (kq_moe_ffn_workspace_size bytes, 256-byte aligned, zero-filled once before
 * first use) holds the error word, the grouping plan at byte 256 (as in
 * kq_moe_matvec), arrival counters (back at zero after each call) and the fp32
 * intermediates; h [M*top_k][F] and hs [M][SH] start at the offsets
 * kq_moe_ffn_offsets returns (for inspection).
 * Errors: KQ_ERR_ARG, KQ_ERR_TYPE, KQ_ERR_SHAPE (H, F or SH not a multiple of
 * 32), KQ_ERR_UNSUPPORTED (M*top_k > 512, n_experts > 4096, a K above 16384 or
 * rows too wide for a 100 KB tile), KQ_ERR_ALIGN, KQ_ERR_WORKSPACE.
 */
#define KQ_ACT_SILU 0
#define KQ_ACT_GELU_TANH 1

typedef struct kq_moe_ffn_weights {
  int32_t type_gate_up; /* block type of W_gate, W_up, Ws_gate, Ws_up */
  int32_t type_down;    /* block type of W_down, Ws_down              */
  int32_t n_experts;
  int32_t act;          /* KQ_ACT_SILU or KQ_ACT_GELU_TANH            */
  int64_t F;            /* routed expert width                        */
  int64_t SH;           /* shared expert width, 0 = none              */
  const void *W_gate, *W_up, *W_down;
  const void *Ws_gate, *Ws_up, *Ws_down;
} kq_moe_ffn_weights;

size_t kq_moe_ffn_workspace_size(int64_t H, int64_t F, int64_t SH, int64_t M, int32_t top_k, int32_t n_experts);
kq_status kq_moe_ffn_offsets(int64_t H, int64_t F, int64_t SH, int64_t M, int32_t top_k, int32_t n_experts,
                             size_t *h_offset, size_t *hs_offset);
kq_status kq_moe_ffn(const kq_moe_ffn_weights *w, const int32_t *expert_ids, const float *gate_w, const void *x,
                     int x_dtype, float *y, int64_t H, int64_t M, int32_t top_k, void *workspace,
                     size_t workspace_bytes, kq_stream_t stream);

/*
 * Read the device error word (KQ_OK when clean); with clear != 0 also reset
 * it.  Synchronizes the device.
 */
kq_status kq_device_error(int *code, int clear);

/* Last CUDA error code seen by a failing call on this host thread (0 if none). */
int kq_last_cuda_error(void);

/* Text for a status code. */
const char *kq_status_string(kq_status status);

#ifdef __cplusplus
}
#endif
#endif /* KQ_H */
