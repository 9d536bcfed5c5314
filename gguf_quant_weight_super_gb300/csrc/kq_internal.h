// kq_internal.h -- declarations shared by the translation units of libkq.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "kq_decode.cuh"
#include "kq_ptx.cuh"

namespace kq {

constexpr int kMaxSmemPerBlock = 227 * 1024;  // opt-in shared memory per CTA on sm_103a

int current_device_id();  // current CUDA device (0..63)
int num_sms();            // SM count of the current device (cached per device)
int* device_error_ptr();  // device address of the error word on the current device

struct GemvPlan {
  int nb, R, KB, nranges, KC, slot_row_bytes, stage_bytes, grid, tiles_per_cta;
  int64_t ntiles;
};
GemvPlan plan_gemv_batched(int qtype, int64_t N, int K, int M);

// M >= 1 tokens, x staged in shared memory windows (kq_gemv_batched.cu)
cudaError_t launch_gemv_batched(int qtype, const void* W, const void* x, int x_bf16, float* y, int64_t N, int K,
                                int M, cudaStream_t stream, bool pdl);

// One-token products (kq_gemv.cu): a single product, or a program of
// products run by one persistent launch with grid-wide ordering between
// dependent ones and split-K partial sums in the program's workspace.
// (M tokens: 1, or 2..4 with bf16 x; y is [M][N])
cudaError_t launch_matvec1(int qtype, const void* W, const void* x, int x_bf16, float* y, int64_t N, int K,
                           cudaStream_t stream, bool pdl, int M = 1);
struct ProgOpDesc {
  int type, x_bf16, wait_previous;
  const void* W;
  const void* x;
  float* y;
  int64_t N, K;
};
struct ProgPlan {
  int n_ops, nb_max, nimg, S, slot;  // nimg: x images in shared memory (2 when an op has fp32 x)
  int coop;       // grid barriers: cooperative launch
  int final_fix;  // split-K sums remain after the last op
  int xk;         // x dtypes of the ops: 1 all bf16, 2 all fp32, 0 both
  int64_t smem, ws_bytes;
};
// workspace bytes of a program (0: some op cannot run on this path)
size_t prog_workspace_size(const ProgOpDesc* descs, int n_ops);
// plans the program, writes it into ws (stream-ordered, then synchronizes)
cudaError_t prog_prepare(const ProgOpDesc* descs, int n_ops, void* ws, size_t ws_bytes, ProgPlan* plan,
                         cudaStream_t stream);
cudaError_t prog_run(const ProgPlan* plan, void* ws, cudaStream_t stream);

// M = 2..16 tokens, bf16 x, on the tensor cores (kq_tc.cu)
bool tc_supported(int qtype, int64_t N, int K, int M);
cudaError_t launch_tc(int qtype, const void* W, const void* x, float* y, int64_t N, int K, int M,
                      cudaStream_t stream, bool pdl);

// Routed-expert products (kq_moe.cu).  Workspace: error word (offset 0),
// plan, per-tile arrival counters, per-pair partial results.
struct MoeLayout {
  int Dmax;
  int64_t ntiles;
  size_t plan_off, cnt_off, part_off, bytes;
};
MoeLayout moe_layout(int64_t N, int64_t M, int top_k, int n_experts);
bool moe_supported(int qtype, int64_t K, int64_t M, int top_k, int n_experts);
cudaError_t launch_moe(int qtype, const void* W, int n_experts, const int32_t* ids, const float* gate,
                       const void* x, int x_bf16, int x_per_slot, float* y, int64_t N, int K, int M, int top_k,
                       void* ws, cudaStream_t st);
cudaError_t launch_moe_err(int qtype, const void* W, int n_experts, const int32_t* ids, const float* gate,
                           const void* x, int x_bf16, int x_per_slot, float* y, int64_t N, int K, int M, int top_k,
                           void* ws, int* err, cudaStream_t st);
// the same product with a library-owned static scratch array (no workspace)
size_t moe_static_scratch_bytes();
cudaError_t launch_moe_static(int qtype, const void* W, int n_experts, const int32_t* ids, const float* gate,
                              const void* x, int x_bf16, int x_per_slot, float* y, int64_t N, int K, int M,
                              int top_k, cudaStream_t st);

// Expert FFN of a layer (kq_moe.cu): gate|up + activation, then down + gated combine.
struct FfnWeights {
  int type_gu, type_dn, n_experts, act;
  int64_t F, SH;
  const void *W_gate, *W_up, *W_down, *Ws_gate, *Ws_up, *Ws_down;
};
struct FfnLayout {
  int Dmax;
  size_t plan_off, cnt_off, part_off, h_off, hs_off, sp_off, bytes;
};
FfnLayout ffn_layout(int64_t H, int64_t F, int64_t SH, int64_t M, int top_k, int n_experts);
bool ffn_supported(int type_gu, int type_dn, int64_t H, int64_t F, int64_t SH, int64_t M, int top_k, int n_experts);
cudaError_t launch_moe_ffn(const FfnWeights& fw, const int32_t* ids, const float* gate, const void* x, int x_bf16,
                           float* y, int64_t H, int M, int top_k, void* ws, cudaStream_t st);

// Bounded-wait self-test (kq_selftest.cu): 0 = mbarrier wait, 1 = grid-barrier wait.
cudaError_t run_selftest_wait(int kind, int* observed, cudaStream_t st);

// MoE router (kq_route.cu): top-k + softmax over the selected logits, and the
// grouping plan (written at ws + 256 in kq_moe_matvec's layout when ws is set)
bool route_supported(int64_t M, int E, int top_k);
size_t route_plan_bytes(int64_t M, int top_k, int E);
cudaError_t launch_route(const float* logits, int M, int E, int top_k, int* ids, float* gate, void* ws,
                         cudaStream_t st);

cudaError_t launch_dequant(int qtype, const void* blocks, void* out, int out_bf16, int64_t n_blocks,
                           cudaStream_t stream);
cudaError_t launch_ia4_pack(const uint32_t* q, const uint16_t* scales, const uint16_t* biases, int64_t N, int64_t K,
                            void* blocks, cudaStream_t stream);
cudaError_t launch_unpack(int qtype, const void* blocks, int64_t n_blocks, uint8_t* codes, int8_t* scales,
                          uint8_t* mins, uint16_t* d_bits, uint16_t* dmin_bits, cudaStream_t stream);

}  // namespace kq
