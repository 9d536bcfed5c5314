// kq_dequant.cu -- block -> fp32 weights, and block -> integer fields.
//
// Dequantization without a product is the fallback the loader uses when packed
// kernels are not available ("GGUF in transformers", sections "Load GGUF with
// transformers" and "Fine-tune from a GGUF checkpoint": GgufConfig(dequantize=
// True) expands the weights).  The integer unpack exposes the same in-register
// decode the products use (kq_decode.cuh) so its codes and scales can be
// compared bit for bit.
//
// Exactness: for Q4_K/Q5_K, d*sc (<= 17 significant bits), q and dmin*m are
// exact in fp32, so w = fma(d*sc, q, -(dmin*m)) rounds once -- the correctly
// rounded value of the exact weight.  For Q6_K, d*sc*(q-32) has at most 23
// significant bits and is exact.
#include "kq_internal.h"

namespace kq {
namespace {

constexpr int THREADS = 256;
constexpr int GROUPS = THREADS / 8;  // one 8-lane group per block

// Two fp32 weights as one bf16 pair, each rounded to nearest even (lo in the low half).
__device__ __forceinline__ uint32_t bf16_pair(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// OutT float: fp32 weights; OutT uint16_t: the same weights rounded to bf16.
template <int QT, typename OutT>
__global__ void __launch_bounds__(THREADS) dequant_kernel(const uint8_t* __restrict__ blocks, OutT* __restrict__ out,
                                                          int64_t n_blocks) {
  constexpr int BB = Fmt<QT>::BYTES;
  constexpr int P = Fmt<QT>::P;
  constexpr int L = Fmt<QT>::L;
  const int j = threadIdx.x & 7;
  for (int64_t b = static_cast<int64_t>(blockIdx.x) * GROUPS + (threadIdx.x >> 3); b < n_blocks;
       b += static_cast<int64_t>(gridDim.x) * GROUPS) {
    LaneFields<QT> fl;
    lane_fields<QT>(blocks + b * BB, j, fl);
    const float d = fl.d, dmin = fl.dmin;
    OutT* o = out + b * 256;
#pragma unroll
    for (int p = 0; p < P; ++p) {
      const float dsc = d * static_cast<float>(fl.sc[p]);
      const float mm = dmin * static_cast<float>(fl.m[p]);
      float w[L];
#pragma unroll
      for (int i = 0; i < L; ++i) {
        const float q = static_cast<float>(code_of<QT>(fl, p * L + i));
        if constexpr (QT == T_Q6_K) w[i] = dsc * (q - 32.0f);
        else w[i] = __fmaf_rn(dsc, q, -mm);
      }
      OutT* dst = o + part_pos<QT>(j, p);
      if constexpr (sizeof(OutT) == 4) {
#pragma unroll
        for (int i = 0; i < L; i += 4)
          *reinterpret_cast<float4*>(dst + i) = make_float4(w[i], w[i + 1], w[i + 2], w[i + 3]);
      } else {
#pragma unroll
        for (int i = 0; i < L; i += 8)
          *reinterpret_cast<uint4*>(dst + i) = make_uint4(bf16_pair(w[i], w[i + 1]), bf16_pair(w[i + 2], w[i + 3]),
                                                          bf16_pair(w[i + 4], w[i + 5]), bf16_pair(w[i + 6], w[i + 7]));
      }
    }
  }
}

template <int QT>
__global__ void __launch_bounds__(THREADS) unpack_kernel(const uint8_t* __restrict__ blocks, int64_t n_blocks,
                                                         uint8_t* codes, int8_t* scales, uint8_t* mins,
                                                         uint16_t* d_bits, uint16_t* dmin_bits) {
  constexpr int BB = Fmt<QT>::BYTES;
  constexpr int P = Fmt<QT>::P;
  constexpr int L = Fmt<QT>::L;
  const int j = threadIdx.x & 7;
  for (int64_t b = static_cast<int64_t>(blockIdx.x) * GROUPS + (threadIdx.x >> 3); b < n_blocks;
       b += static_cast<int64_t>(gridDim.x) * GROUPS) {
    LaneFields<QT> fl;
    lane_fields<QT>(blocks + b * BB, j, fl);
#pragma unroll
    for (int p = 0; p < P; ++p) {
      const int pos = part_pos<QT>(j, p);
      if (codes)
        for (int i = 0; i < L; ++i) codes[b * 256 + pos + i] = static_cast<uint8_t>(code_of<QT>(fl, p * L + i));
      // scale index: 32-weight sub-block (Q4_K/Q5_K) or 16-weight (Q6_K)
      const int si = (QT == T_Q6_K) ? pos / 16 : pos / 32;
      if (scales) scales[b * 16 + si] = static_cast<int8_t>(fl.sc[p]);
      if (mins && QT != T_Q6_K) mins[b * 8 + si] = static_cast<uint8_t>(fl.m[p]);
    }
    if (j == 0) {
      if (d_bits) d_bits[b] = static_cast<uint16_t>(fl.d_bits);
      if (dmin_bits) dmin_bits[b] = static_cast<uint16_t>(fl.dmin_bits);
    }
  }
}

int grid_for(int64_t n_blocks) {
  const int64_t need = (n_blocks + GROUPS - 1) / GROUPS;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  return static_cast<int>(need < cap ? need : cap);
}

}  // namespace

cudaError_t launch_dequant(int qtype, const void* blocks, void* out, int out_bf16, int64_t n_blocks,
                           cudaStream_t stream) {
  if (n_blocks == 0) return cudaSuccess;
  const uint8_t* b = static_cast<const uint8_t*>(blocks);
  const int grid = grid_for(n_blocks);
  float* of = static_cast<float*>(out);
  uint16_t* oh = static_cast<uint16_t*>(out);
  switch (qtype * 2 + (out_bf16 ? 1 : 0)) {
    case T_Q4_K * 2: dequant_kernel<T_Q4_K, float><<<grid, THREADS, 0, stream>>>(b, of, n_blocks); break;
    case T_Q5_K * 2: dequant_kernel<T_Q5_K, float><<<grid, THREADS, 0, stream>>>(b, of, n_blocks); break;
    case T_Q6_K * 2: dequant_kernel<T_Q6_K, float><<<grid, THREADS, 0, stream>>>(b, of, n_blocks); break;
    case T_Q4_K * 2 + 1: dequant_kernel<T_Q4_K, uint16_t><<<grid, THREADS, 0, stream>>>(b, oh, n_blocks); break;
    case T_Q5_K * 2 + 1: dequant_kernel<T_Q5_K, uint16_t><<<grid, THREADS, 0, stream>>>(b, oh, n_blocks); break;
    case T_Q6_K * 2 + 1: dequant_kernel<T_Q6_K, uint16_t><<<grid, THREADS, 0, stream>>>(b, oh, n_blocks); break;
    case T_IA4 * 2: dequant_kernel<T_IA4, float><<<grid, THREADS, 0, stream>>>(b, of, n_blocks); break;
    case T_IA4 * 2 + 1: dequant_kernel<T_IA4, uint16_t><<<grid, THREADS, 0, stream>>>(b, oh, n_blocks); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Group-affine INT4 (an MLX 4-bit checkpoint) -> IA4 blocks.  The source is
// row-major: codes q[N][K/8] as 32-bit words, code k of a row in bits
// 4(k%8)..4(k%8)+3 of word k/8; scales and biases [N][K/64] bf16, group
// G = weights 64G..64G+63, w = scale*q + bias.  One thread per (row, group):
// the group's scale and bias go to the block header, its 64 codes to the 32
// code bytes of chunk g = G%4 in the Q4_K order (byte 32g+l: weight 64g+l in
// the low nibble, 64g+32+l in the high one).  Groups past K in a row's last
// block get zero scale, bias and codes.
// ---------------------------------------------------------------------------
__global__ void ia4_pack_kernel(const uint32_t* __restrict__ q, const uint16_t* __restrict__ scales,
                                const uint16_t* __restrict__ biases, int64_t N, int64_t K, uint8_t* __restrict__ blocks) {
  const int64_t ng = K / 64, nb = (K + 255) / 256;
  const int64_t total = N * nb * 4;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t n = t / (nb * 4), r = t - n * nb * 4;
    const int64_t b = r >> 2;
    const int g = static_cast<int>(r & 3);
    const int64_t G = 4 * b + g;
    uint8_t* blk = blocks + (n * nb + b) * 144;
    const bool in = G < ng;
    reinterpret_cast<uint16_t*>(blk)[g] = in ? scales[n * ng + G] : static_cast<uint16_t>(0);
    reinterpret_cast<uint16_t*>(blk + 8)[g] = in ? biases[n * ng + G] : static_cast<uint16_t>(0);
    uint32_t out[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) out[i] = 0u;
    if (in) {
      const uint32_t* src = q + n * (K / 8) + G * 8;  // the group's 8 words: weights 64G + 8i + j
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = src[i];
#pragma unroll
      for (int l = 0; l < 32; ++l) {
        const uint32_t lo = (w[l >> 3] >> (4 * (l & 7))) & 15u;             // weight 64G + l
        const uint32_t hi = (w[4 + (l >> 3)] >> (4 * (l & 7))) & 15u;       // weight 64G + 32 + l
        out[l >> 2] |= (lo | (hi << 4)) << (8 * (l & 3));
      }
    }
    uint4* dst = reinterpret_cast<uint4*>(blk + 16 + 32 * g);
    dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
  }
}

cudaError_t launch_ia4_pack(const uint32_t* q, const uint16_t* scales, const uint16_t* biases, int64_t N, int64_t K,
                            void* blocks, cudaStream_t stream) {
  const int64_t total = N * ((K + 255) / 256) * 4;
  if (total == 0) return cudaSuccess;
  const int64_t want = (total + 255) / 256;
  const int grid = static_cast<int>(want < 152 * 16 ? want : 152 * 16);
  ia4_pack_kernel<<<grid, 256, 0, stream>>>(q, scales, biases, N, K, static_cast<uint8_t*>(blocks));
  return cudaGetLastError();
}

cudaError_t launch_unpack(int qtype, const void* blocks, int64_t n_blocks, uint8_t* codes, int8_t* scales,
                          uint8_t* mins, uint16_t* d_bits, uint16_t* dmin_bits, cudaStream_t stream) {
  if (n_blocks == 0) return cudaSuccess;
  const uint8_t* b = static_cast<const uint8_t*>(blocks);
  const int grid = grid_for(n_blocks);
  switch (qtype) {
    case T_Q4_K: unpack_kernel<T_Q4_K><<<grid, THREADS, 0, stream>>>(b, n_blocks, codes, scales, mins, d_bits, dmin_bits); break;
    case T_Q5_K: unpack_kernel<T_Q5_K><<<grid, THREADS, 0, stream>>>(b, n_blocks, codes, scales, mins, d_bits, dmin_bits); break;
    case T_Q6_K: unpack_kernel<T_Q6_K><<<grid, THREADS, 0, stream>>>(b, n_blocks, codes, scales, mins, d_bits, dmin_bits); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace kq
