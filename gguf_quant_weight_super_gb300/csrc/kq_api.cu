// kq_api.cu -- the extern "C" entry points of libkq (declared in include/kq.h):
// argument checks, kernel choice, launch, and the device error word.
#include <cstdio>
#include <cstring>

#include "../../include/kq.h"
#include "kq_internal.h"

namespace kq {

// The library's device error word (one per device that loads the library).
__device__ int g_device_error = 0;

namespace {
constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices] = {0};
int* g_err_ptr[kMaxDevices] = {nullptr};
thread_local int t_last_cuda_error = 0;

}  // namespace

int current_device_id() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  return (dev >= 0 && dev < kMaxDevices) ? dev : 0;
}

int num_sms() {
  const int dev = current_device_id();
  if (!g_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

int* device_error_ptr() {
  const int dev = current_device_id();
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  return g_err_ptr[dev];
}

static kq_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return KQ_OK;
  t_last_cuda_error = static_cast<int>(e);
  return KQ_ERR_CUDA;
}

static bool valid_type(int t) { return t == KQ_Q4_K || t == KQ_Q5_K || t == KQ_Q6_K || t == KQ_IA4; }
static bool kquant_type(int t) { return t == KQ_Q4_K || t == KQ_Q5_K || t == KQ_Q6_K; }  // unpack, chains
static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace kq

using namespace kq;

extern "C" {

size_t kq_block_bytes(int type) { return valid_type(type) ? static_cast<size_t>(block_bytes_of(type)) : 0; }

kq_status kq_ia4_pack(const uint32_t* q, const uint16_t* scales, const uint16_t* biases, int64_t N, int64_t K,
                      void* blocks, kq_stream_t stream) {
  if (N < 0 || K < 0) return KQ_ERR_ARG;
  if (K % 64) return KQ_ERR_SHAPE;
  if (N == 0 || K == 0) return KQ_OK;
  if (!q || !scales || !biases || !blocks) return KQ_ERR_ARG;
  if (!aligned(q, 4) || !aligned(scales, 2) || !aligned(biases, 2) || !aligned(blocks, 16)) return KQ_ERR_ALIGN;
  return cuda_status(launch_ia4_pack(q, scales, biases, N, K, blocks, reinterpret_cast<cudaStream_t>(stream)));
}

kq_status kq_unpack(int type, const void* blocks, int64_t n_blocks, uint8_t* codes, int8_t* scales, uint8_t* mins,
                    uint16_t* d_bits, uint16_t* dmin_bits, kq_stream_t stream) {
  if (!kquant_type(type)) return KQ_ERR_TYPE;
  if (n_blocks < 0) return KQ_ERR_ARG;
  if (n_blocks == 0) return KQ_OK;
  if (!blocks) return KQ_ERR_ARG;
  if (!aligned(blocks, 16)) return KQ_ERR_ALIGN;
  return cuda_status(launch_unpack(type, blocks, n_blocks, codes, scales, mins, d_bits, dmin_bits,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

kq_status kq_dequant(int type, const void* blocks, float* out, int64_t n, kq_stream_t stream) {
  if (!valid_type(type)) return KQ_ERR_TYPE;
  if (n < 0) return KQ_ERR_ARG;
  if (n % 256) return KQ_ERR_SHAPE;
  if (n == 0) return KQ_OK;
  if (!blocks || !out) return KQ_ERR_ARG;
  if (!aligned(blocks, 16) || !aligned(out, 16)) return KQ_ERR_ALIGN;
  return cuda_status(launch_dequant(type, blocks, out, 0, n / 256, reinterpret_cast<cudaStream_t>(stream)));
}

kq_status kq_dequant_bf16(int type, const void* blocks, uint16_t* out, int64_t n, kq_stream_t stream) {
  if (!valid_type(type)) return KQ_ERR_TYPE;
  if (n < 0) return KQ_ERR_ARG;
  if (n % 256) return KQ_ERR_SHAPE;
  if (n == 0) return KQ_OK;
  if (!blocks || !out) return KQ_ERR_ARG;
  if (!aligned(blocks, 16) || !aligned(out, 16)) return KQ_ERR_ALIGN;
  return cuda_status(launch_dequant(type, blocks, out, 1, n / 256, reinterpret_cast<cudaStream_t>(stream)));
}

kq_status kq_matvec(int type, const void* W, const void* x, int x_dtype, float* y, int64_t N, int64_t K, int64_t M,
                    kq_stream_t stream) {
  if (!valid_type(type)) return KQ_ERR_TYPE;
  if (x_dtype != KQ_F32 && x_dtype != KQ_BF16) return KQ_ERR_ARG;
  if (N < 0 || K < 0 || M < 0) return KQ_ERR_ARG;
  if (M > 16) return KQ_ERR_UNSUPPORTED;
  if (K % 32 || K > (int64_t(1) << 24)) return KQ_ERR_SHAPE;
  if (N == 0 || M == 0) return KQ_OK;
  if (!y) return KQ_ERR_ARG;
  if (K == 0) return cuda_status(cudaMemsetAsync(y, 0, sizeof(float) * N * M, reinterpret_cast<cudaStream_t>(stream)));
  if (!W || !x) return KQ_ERR_ARG;
  if (!aligned(W, 16) || !aligned(x, 16) || !aligned(y, 4)) return KQ_ERR_ALIGN;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int bf16 = (x_dtype == KQ_BF16);
  cudaError_t e = cudaErrorNotSupported;
  if (M == 1 || (M <= 4 && bf16)) e = launch_matvec1(type, W, x, bf16, y, N, static_cast<int>(K), st, true, M);
  if (e == cudaErrorNotSupported && bf16 && tc_supported(type, N, static_cast<int>(K), static_cast<int>(M)))
    e = launch_tc(type, W, x, y, N, static_cast<int>(K), static_cast<int>(M), st, true);
  if (e == cudaErrorNotSupported)
    e = launch_gemv_batched(type, W, x, bf16, y, N, static_cast<int>(K), static_cast<int>(M), st, true);
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_status(e);
}

static_assert(sizeof(ProgPlan) <= sizeof(kq_chain_plan), "plan storage");

static bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bn && b0 < a0 + an;
}

static kq_status check_chain(const kq_op* ops, int n_ops) {
  if (!ops || n_ops <= 0) return KQ_ERR_ARG;
  int last_wait = 0;
  for (int i = 0; i < n_ops; ++i) {
    const kq_op& o = ops[i];
    if (!kquant_type(o.type)) return KQ_ERR_TYPE;
    if (o.x_dtype != KQ_F32 && o.x_dtype != KQ_BF16) return KQ_ERR_ARG;
    if (o.reserved != 0 || o.N <= 0 || o.K <= 0) return KQ_ERR_ARG;
    if (o.K % 32) return KQ_ERR_SHAPE;
    if (o.K > 16384) return KQ_ERR_UNSUPPORTED;
    if (!o.W || !o.x || !o.y) return KQ_ERR_ARG;
    if (!aligned(o.W, 16) || !aligned(o.x, 16) || !aligned(o.y, 4)) return KQ_ERR_ALIGN;
    if (i > 0 && o.wait_previous) last_wait = i;
    // x may not be an output of an op that can still be running
    for (int j = last_wait; j < i; ++j)
      if (overlaps(o.x, o.K * (o.x_dtype == KQ_BF16 ? 2 : 4), ops[j].y, ops[j].N * 4)) return KQ_ERR_ARG;
  }
  for (int i = 0; i < n_ops; ++i) {
    const size_t yb = ops[i].N * 4;
    for (int j = 0; j < n_ops; ++j) {
      const int64_t nbj = (ops[j].K + 255) / 256;
      if (overlaps(ops[i].y, yb, ops[j].W, nbj * ops[j].N * block_bytes_of(ops[j].type))) return KQ_ERR_ARG;
      if (j != i && overlaps(ops[i].y, yb, ops[j].y, ops[j].N * 4)) return KQ_ERR_ARG;
      if (j <= i && overlaps(ops[i].y, yb, ops[j].x, ops[j].K * (ops[j].x_dtype == KQ_BF16 ? 2 : 4)))
        return KQ_ERR_ARG;
    }
  }
  return KQ_OK;
}

static void to_desc(const kq_op* ops, int n_ops, ProgOpDesc* d) {
  for (int i = 0; i < n_ops; ++i) {
    d[i].type = ops[i].type;
    d[i].x_bf16 = ops[i].x_dtype == KQ_BF16;
    d[i].wait_previous = ops[i].wait_previous != 0;
    d[i].W = ops[i].W;
    d[i].x = ops[i].x;
    d[i].y = ops[i].y;
    d[i].N = ops[i].N;
    d[i].K = ops[i].K;
  }
}

size_t kq_chain_workspace_size(const kq_op* ops, int n_ops) {
  if (check_chain(ops, n_ops) != KQ_OK) return 0;
  ProgOpDesc* d = new ProgOpDesc[n_ops];
  to_desc(ops, n_ops, d);
  const size_t b = prog_workspace_size(d, n_ops);
  delete[] d;
  return b;
}

kq_status kq_chain_prepare(const kq_op* ops, int n_ops, void* workspace, size_t workspace_bytes,
                           kq_chain_plan* plan, kq_stream_t stream) {
  const kq_status st = check_chain(ops, n_ops);
  if (st != KQ_OK) return st;
  if (!plan) return KQ_ERR_ARG;
  if (!workspace || !aligned(workspace, 256)) return KQ_ERR_WORKSPACE;
  ProgOpDesc* d = new ProgOpDesc[n_ops];
  to_desc(ops, n_ops, d);
  const size_t need = prog_workspace_size(d, n_ops);
  if (need == 0) { delete[] d; return KQ_ERR_UNSUPPORTED; }
  if (workspace_bytes < need) { delete[] d; return KQ_ERR_WORKSPACE; }
  ProgPlan p = {};
  const cudaError_t e = prog_prepare(d, n_ops, workspace, workspace_bytes, &p,
                                     reinterpret_cast<cudaStream_t>(stream));
  delete[] d;
  if (e != cudaSuccess) return cuda_status(e);
  memset(plan, 0, sizeof(*plan));
  memcpy(plan, &p, sizeof(p));
  return KQ_OK;
}

kq_status kq_chain_run(const kq_chain_plan* plan, void* workspace, kq_stream_t stream) {
  if (!plan || !workspace) return KQ_ERR_ARG;
  ProgPlan p;
  memcpy(&p, plan, sizeof(p));
  if (p.n_ops <= 0) return KQ_ERR_ARG;
  cudaError_t e = prog_run(&p, workspace, reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_status(e);
}

size_t kq_moe_workspace_size(int64_t N, int64_t M, int32_t top_k, int32_t n_experts) {
  if (N <= 0 || M <= 0 || top_k <= 0 || n_experts <= 0 || M * top_k > 512) return 0;
  return moe_layout(N, M, top_k, n_experts).bytes;
}

kq_status kq_moe_matvec(int type, const void* W_experts, int32_t n_experts, const int32_t* expert_ids,
                        const float* gate_w, const void* x, int x_dtype, int x_per_slot, float* y, int64_t N,
                        int64_t K, int64_t M, int32_t top_k, void* workspace, size_t workspace_bytes,
                        kq_stream_t stream) {
  if (!valid_type(type)) return KQ_ERR_TYPE;
  if (x_dtype != KQ_F32 && x_dtype != KQ_BF16) return KQ_ERR_ARG;
  if (N < 0 || K < 0 || M < 0 || top_k <= 0 || n_experts <= 0) return KQ_ERR_ARG;
  if (K % 32) return KQ_ERR_SHAPE;
  if (N == 0 || M == 0) return KQ_OK;
  if (K == 0 || !moe_supported(type, K, M, top_k, n_experts)) return KQ_ERR_UNSUPPORTED;
  if (!W_experts || !expert_ids || !x || !y) return KQ_ERR_ARG;
  if (!aligned(W_experts, 16) || !aligned(x, 16) || !aligned(y, 4) || !aligned(expert_ids, 4) ||
      (gate_w && !aligned(gate_w, 4)))
    return KQ_ERR_ALIGN;
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < moe_layout(N, M, top_k, n_experts).bytes)
    return KQ_ERR_WORKSPACE;
  cudaError_t e = launch_moe(type, W_experts, n_experts, expert_ids, gate_w, x, x_dtype == KQ_BF16,
                             x_per_slot ? 1 : 0, y, N, static_cast<int>(K), static_cast<int>(M), top_k, workspace,
                             reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return KQ_ERR_UNSUPPORTED;
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_status(e);
}

kq_status kq_moe_matvec_noalloc(int type, const void* W_experts, int32_t n_experts, const int32_t* expert_ids,
                                const float* gate_w, const void* x, int x_dtype, int x_per_slot, float* y, int64_t N,
                                int64_t K, int64_t M, int32_t top_k, kq_stream_t stream) {
  if (!valid_type(type)) return KQ_ERR_TYPE;
  if (x_dtype != KQ_F32 && x_dtype != KQ_BF16) return KQ_ERR_ARG;
  if (N < 0 || K < 0 || M < 0 || top_k <= 0 || n_experts <= 0) return KQ_ERR_ARG;
  if (K % 32) return KQ_ERR_SHAPE;
  if (N == 0 || M == 0) return KQ_OK;
  if (K == 0 || !moe_supported(type, K, M, top_k, n_experts)) return KQ_ERR_UNSUPPORTED;
  if (moe_layout(N, M, top_k, n_experts).bytes > moe_static_scratch_bytes()) return KQ_ERR_WORKSPACE;
  if (!W_experts || !expert_ids || !x || !y) return KQ_ERR_ARG;
  if (!aligned(W_experts, 16) || !aligned(x, 16) || !aligned(y, 4) || !aligned(expert_ids, 4) ||
      (gate_w && !aligned(gate_w, 4)))
    return KQ_ERR_ALIGN;
  cudaError_t e = launch_moe_static(type, W_experts, n_experts, expert_ids, gate_w, x, x_dtype == KQ_BF16,
                                    x_per_slot ? 1 : 0, y, N, static_cast<int>(K), static_cast<int>(M), top_k,
                                    reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return KQ_ERR_UNSUPPORTED;
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_status(e);
}

kq_status kq_moe_route(const float* logits, int64_t M, int32_t n_experts, int32_t top_k, int32_t* expert_ids,
                       float* gate_w, void* workspace, size_t workspace_bytes, kq_stream_t stream) {
  if (M < 0 || n_experts <= 0 || top_k <= 0) return KQ_ERR_ARG;
  if (M == 0) return KQ_OK;
  if (!route_supported(M, n_experts, top_k)) return KQ_ERR_UNSUPPORTED;
  if (!logits || !expert_ids || !gate_w) return KQ_ERR_ARG;
  if (!aligned(logits, 4) || !aligned(expert_ids, 4) || !aligned(gate_w, 4)) return KQ_ERR_ALIGN;
  if (workspace && (!aligned(workspace, 256) || workspace_bytes < route_plan_bytes(M, top_k, n_experts)))
    return KQ_ERR_WORKSPACE;
  cudaError_t e = launch_route(logits, static_cast<int>(M), n_experts, top_k, expert_ids, gate_w, workspace,
                               reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_status(e);
}

size_t kq_moe_ffn_workspace_size(int64_t H, int64_t F, int64_t SH, int64_t M, int32_t top_k, int32_t n_experts) {
  if (H <= 0 || F <= 0 || SH < 0 || M <= 0 || top_k <= 0 || n_experts <= 0 || M * top_k > 512) return 0;
  return ffn_layout(H, F, SH, M, top_k, n_experts).bytes;
}

kq_status kq_moe_ffn_offsets(int64_t H, int64_t F, int64_t SH, int64_t M, int32_t top_k, int32_t n_experts,
                             size_t* h_offset, size_t* hs_offset) {
  if (!kq_moe_ffn_workspace_size(H, F, SH, M, top_k, n_experts) || !h_offset || !hs_offset) return KQ_ERR_ARG;
  const FfnLayout L = ffn_layout(H, F, SH, M, top_k, n_experts);
  *h_offset = L.h_off;
  *hs_offset = L.hs_off;
  return KQ_OK;
}

kq_status kq_moe_ffn(const kq_moe_ffn_weights* w, const int32_t* expert_ids, const float* gate_w, const void* x,
                     int x_dtype, float* y, int64_t H, int64_t M, int32_t top_k, void* workspace,
                     size_t workspace_bytes, kq_stream_t stream) {
  if (!w) return KQ_ERR_ARG;
  if (!valid_type(w->type_gate_up) || !valid_type(w->type_down)) return KQ_ERR_TYPE;
  if (x_dtype != KQ_F32 && x_dtype != KQ_BF16) return KQ_ERR_ARG;
  if (w->act != KQ_ACT_SILU && w->act != KQ_ACT_GELU_TANH) return KQ_ERR_ARG;
  if (H < 0 || w->F <= 0 || w->SH < 0 || M < 0 || top_k <= 0 || w->n_experts <= 0) return KQ_ERR_ARG;
  if (H % 32 || w->F % 32 || w->SH % 32) return KQ_ERR_SHAPE;
  if (H == 0 || M == 0) return KQ_OK;
  if (!ffn_supported(w->type_gate_up, w->type_down, H, w->F, w->SH, M, top_k, w->n_experts))
    return KQ_ERR_UNSUPPORTED;
  if (!w->W_gate || !w->W_up || !w->W_down || !expert_ids || !gate_w || !x || !y) return KQ_ERR_ARG;
  if (w->SH > 0 && (!w->Ws_gate || !w->Ws_up || !w->Ws_down)) return KQ_ERR_ARG;
  if (!aligned(w->W_gate, 16) || !aligned(w->W_up, 16) || !aligned(w->W_down, 16) || !aligned(x, 16) ||
      !aligned(y, 4) || !aligned(expert_ids, 4) || !aligned(gate_w, 4))
    return KQ_ERR_ALIGN;
  if (w->SH > 0 && (!aligned(w->Ws_gate, 16) || !aligned(w->Ws_up, 16) || !aligned(w->Ws_down, 16)))
    return KQ_ERR_ALIGN;
  if (!workspace || !aligned(workspace, 256) ||
      workspace_bytes < ffn_layout(H, w->F, w->SH, M, top_k, w->n_experts).bytes)
    return KQ_ERR_WORKSPACE;
  FfnWeights fw;
  fw.type_gu = w->type_gate_up;
  fw.type_dn = w->type_down;
  fw.n_experts = w->n_experts;
  fw.act = w->act;
  fw.F = w->F;
  fw.SH = w->SH;
  fw.W_gate = w->W_gate;
  fw.W_up = w->W_up;
  fw.W_down = w->W_down;
  fw.Ws_gate = w->Ws_gate;
  fw.Ws_up = w->Ws_up;
  fw.Ws_down = w->Ws_down;
  cudaError_t e = launch_moe_ffn(fw, expert_ids, gate_w, x, x_dtype == KQ_BF16, y, H, static_cast<int>(M), top_k,
                                 workspace, reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return KQ_ERR_UNSUPPORTED;
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_status(e);
}

kq_status kq_selftest_wait(int kind, int* observed_code, kq_stream_t stream) {
  if ((kind != 0 && kind != 1) || !observed_code) return KQ_ERR_ARG;
  return cuda_status(run_selftest_wait(kind, observed_code, reinterpret_cast<cudaStream_t>(stream)));
}

kq_status kq_moe_check(void* workspace, kq_stream_t stream) {
  if (!workspace) return KQ_ERR_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_status(e);
  if (v) {
    e = cudaMemsetAsync(workspace, 0, sizeof(int), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_status(e);
    return KQ_ERR_DEVICE;
  }
  return KQ_OK;
}

kq_status kq_device_error(int* code, int clear) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int));
  if (e != cudaSuccess) return cuda_status(e);
  if (clear && v) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_status(e);
  }
  if (code) *code = v;
  return v ? KQ_ERR_DEVICE : KQ_OK;
}

int kq_last_cuda_error(void) { return t_last_cuda_error; }

const char* kq_status_string(kq_status s) {
  switch (s) {
    case KQ_OK: return "ok";
    case KQ_ERR_ARG: return "invalid argument";
    case KQ_ERR_TYPE: return "unknown block type";
    case KQ_ERR_SHAPE: return "unsupported shape (K must be a multiple of 32; dequant n a multiple of 256)";
    case KQ_ERR_UNSUPPORTED: return "unsupported size (M must be 1..16, top_k 1..32)";
    case KQ_ERR_ALIGN: return "misaligned pointer";
    case KQ_ERR_CUDA: return "CUDA error";
    case KQ_ERR_WORKSPACE: return "workspace missing or too small";
    case KQ_ERR_DEVICE: return "device error word set";
    default: return "unknown status";
  }
}

}  // extern "C"
