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
// one token, x held in registers per quad (kq_gemv1.cu); returns
// cudaErrorNotSupported when the shape is outside its limits
cudaError_t launch_gemv1(int qtype, const void* W, const void* x, int x_bf16, float* y, int64_t N, int K,
                         cudaStream_t stream, bool pdl);

cudaError_t launch_dequant(int qtype, const void* blocks, float* out, int64_t n_blocks, cudaStream_t stream);
cudaError_t launch_unpack(int qtype, const void* blocks, int64_t n_blocks, uint8_t* codes, int8_t* scales,
                          uint8_t* mins, uint16_t* d_bits, uint16_t* dmin_bits, cudaStream_t stream);

}  // namespace kq
