// kq_decode.cuh -- in-register decoding of k-quant super-blocks (256 weights).
//
// Formats (GGUF k-quants; byte layouts are this library's reading of the
// public GGUF layout, which the source pages do not print):
//   Q4_K, 144 B: d (fp16) | dmin (fp16) | 12 B of 8 six-bit scales + 8 six-bit
//                mins | 128 B of 4-bit codes.       w = d*sc_j*q - dmin*m_j
//   Q5_K, 176 B: d | dmin | 12 B scales/mins | 32 B of 5th bits | 128 B codes.
//   Q6_K, 210 B: 128 B low nibbles | 64 B high bit pairs | 16 int8 scales | d.
//                                                       w = d*sc_j*(q - 32)
// ("GGUF in transformers", section "What is the GGUF file format?", names the
// Q4_K_M / Q5_K_M / Q6_K variants these blocks make up.)
//   IA4,  144 B: 4 bf16 scales | 4 bf16 biases | 128 B of 4-bit codes in the
//                Q4_K code order; group g = weights 64g..64g+63 (sub-blocks
//                2g, 2g+1).                      w = scale_g*q + bias_g
//                The group-affine INT4 format of an MLX 4-bit checkpoint
//                ("ANE Fieldfare" README, "Requirements": the model is an
//                mlx-community 4-bit checkpoint), regrouped by kq_ia4_pack into
//                blocks of 256 weights.  It decodes as Q4_K with, per group,
//                d*sc := scale_g and dmin*m := -bias_g (sc = m = 1).
//
// Work split: a block is decoded by 8 lanes; lane j owns 32 of its weights,
// as P "parts" of L consecutive weights:
//   Q4_K/Q5_K: P=2, L=16.  g = j/2, h = j%2; part 0 = weights 64g+16h+[0,16)
//              (sub-block 2g, low nibbles), part 1 = weights 64g+32+16h+[0,16)
//              (sub-block 2g+1, high nibbles) of qs bytes 32g+16h+[0,16).
//   Q6_K:      P=4, L=8.   h = j/4, l0 = 8*(j%4); part t = weights
//              128h+32t+l0+[0,8), scale index 8h+2t+l0/16.
//
// Instead of converting each code to float, a code q is placed into the
// mantissa of 1.0: f = 1 + q/2^s (s = 4, 5, 6 for Q4_K, Q5_K, Q6_K) with one
// byte-permute per weight.  A part's contribution is then
//     sum_i w_i x_i = A * sum_i f_i x_i + B * sum_i x_i
// with A = 2^s d sc and B = -(A + dmin m) (Q4_K/Q5_K) or B = -(2^s+32) d sc
// (Q6_K); sum_i x_i is a property of x alone and is precomputed per part.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace kq {

enum : int { T_Q4_K = 1, T_Q5_K = 2, T_Q6_K = 3, T_IA4 = 4 };

// Q4_K and IA4 share the code layout (nibbles of 128 bytes after a 16-byte header).
template <int QT> constexpr bool kQ4Codes = (QT == T_Q4_K || QT == T_IA4);

template <int QT> struct Fmt;
template <> struct Fmt<T_Q4_K> { static constexpr int BYTES = 144, P = 2, L = 16, SHIFT = 4; };
template <> struct Fmt<T_Q5_K> { static constexpr int BYTES = 176, P = 2, L = 16, SHIFT = 5; };
template <> struct Fmt<T_Q6_K> { static constexpr int BYTES = 210, P = 4, L = 8, SHIFT = 6; };
template <> struct Fmt<T_IA4> { static constexpr int BYTES = 144, P = 2, L = 16, SHIFT = 4; };

__host__ __device__ constexpr int block_bytes_of(int qt) {
  return (qt == T_Q4_K || qt == T_IA4) ? 144 : qt == T_Q5_K ? 176 : qt == T_Q6_K ? 210 : 0;
}

// Position (within the block) of the first weight of part p of lane j.
template <int QT>
__device__ __forceinline__ int part_pos(int j, int p) {
  if constexpr (QT == T_Q6_K) return 128 * (j >> 2) + 32 * p + 8 * (j & 3);
  else return 64 * (j >> 1) + 32 * p + 16 * (j & 1);
}

__device__ __forceinline__ float half_bits_to_float(uint32_t bits16) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16)));
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// IA4 group g of a block header (words x, y: scales 0-1, 2-3; z, w: biases):
// d := scale_g, dmin := -bias_g, so that the Q4_K formulas apply with sc = m = 1.
__device__ __forceinline__ float ia4_scale(uint4 hdr, int g) {
  return bf16_bits_to_float(((g < 2 ? hdr.x : hdr.y) >> (16 * (g & 1))) & 0xFFFFu);
}
__device__ __forceinline__ float ia4_neg_bias(uint4 hdr, int g) {
  return -bf16_bits_to_float(((g < 2 ? hdr.z : hdr.w) >> (16 * (g & 1))) & 0xFFFFu);
}

// f = 1 + q / 2^s from a byte holding 0x80 | (q << (7 - s)): the byte becomes
// mantissa bits 16..23 (bit 23 is the exponent's lowest bit) under 0x3F.
__device__ __forceinline__ float byte_to_f(uint32_t pre, int k) {
  return __int_as_float(static_cast<int>(__byte_perm(pre, 0x3F000000u, 0x7044u | (k << 8))));
}

// Load 8 bytes starting at a 2-byte aligned address (shared or global) with
// three aligned 32-bit loads and funnel shifts.  Reads up to 4 bytes past the
// 8 requested, always inside the same 16-byte granule pair.
__device__ __forceinline__ uint2 ld8_a2(const uint8_t* p) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
  const uint32_t sh = static_cast<uint32_t>(a & 3) * 8;
  const uint32_t w0 = w[0], w1 = w[1], w2 = w[2];
  return make_uint2(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh));
}

// Q4_K/Q5_K scales: bytes [sc_{2g}, sc_{2g+1}, m_{2g}, m_{2g+1}] from the
// 12-byte field s[0..11] held in words h1 = s[0..3], h2 = s[4..7], h3 = s[8..11].
//   j < 4 : sc_j = s[j] & 63,                     m_j = s[j+4] & 63
//   j >= 4: sc_j = (s[j+4] & 15) | (s[j-4]>>6)<<4, m_j = (s[j+4]>>4) | (s[j]>>6)<<4
__device__ __forceinline__ uint32_t scale_min_bytes(uint32_t h1, uint32_t h2, uint32_t h3, int g) {
  if (g < 2) {
    const uint32_t j = 2 * g;
    return __byte_perm(h1, h2, j | ((j + 1) << 4) | ((j + 4) << 8) | ((j + 5) << 12)) & 0x3F3F3F3Fu;
  }
  const uint32_t i = 2 * g - 4;
  const uint32_t lowv = __byte_perm(h3, 0u, i | ((i + 1) << 4) | (i << 8) | ((i + 1) << 12));
  const uint32_t lows = (lowv & 0x00000F0Fu) | ((lowv >> 4) & 0x0F0F0000u);
  const uint32_t highv = __byte_perm(h1, h2, i | ((i + 1) << 4) | ((i + 4) << 8) | ((i + 5) << 12));
  return lows | ((highv >> 2) & 0x30303030u);
}

// ---------------------------------------------------------------------------
// Pre-bytes: 4 codes per 32-bit word, each byte = 0x80 | (q << (7 - s)).
// ---------------------------------------------------------------------------

// Q4_K: word of 4 qs bytes -> (low-nibble codes, high-nibble codes).
__device__ __forceinline__ void q4k_pre(uint32_t wq, uint32_t& lo, uint32_t& hi) {
  lo = ((wq << 3) & 0x78787878u) | 0x80808080u;
  hi = ((wq >> 1) & 0x78787878u) | 0x80808080u;
}

// Q5_K: codes of sub-blocks 2g (low nibble, 5th bit = bit 2g of qh) and 2g+1
// (high nibble, bit 2g+1).  Rotations move bit 2g / 2g+1 of each qh byte to bit 6.
__device__ __forceinline__ void q5k_pre(uint32_t wq, uint32_t wh, int g, uint32_t& lo, uint32_t& hi) {
  const uint32_t rlo = __funnelshift_l(wh, wh, (6 - 2 * g) & 31);
  const uint32_t rhi = __funnelshift_l(wh, wh, (5 - 2 * g) & 31);
  lo = ((wq << 2) & 0x3C3C3C3Cu) | (rlo & 0x40404040u) | 0x80808080u;
  hi = ((wq >> 2) & 0x3C3C3C3Cu) | (rhi & 0x40404040u) | 0x80808080u;
}

// Q6_K: a = 4 bytes of ql[64h+l..], b = ql[64h+32+l..], c = qh[32h+l..];
// parts t = 0..3 take (a low, c bits 0-1), (b low, c 2-3), (a high, c 4-5), (b high, c 6-7).
__device__ __forceinline__ void q6k_pre(uint32_t a, uint32_t b, uint32_t c, uint32_t (&pre)[4]) {
  pre[0] = ((a << 1) & 0x1E1E1E1Eu) | ((c << 5) & 0x60606060u) | 0x80808080u;
  pre[1] = ((b << 1) & 0x1E1E1E1Eu) | ((c << 3) & 0x60606060u) | 0x80808080u;
  pre[2] = ((a >> 3) & 0x1E1E1E1Eu) | ((c << 1) & 0x60606060u) | 0x80808080u;
  pre[3] = ((b >> 3) & 0x1E1E1E1Eu) | ((c >> 1) & 0x60606060u) | 0x80808080u;
}

// ---------------------------------------------------------------------------
// One lane's share of one block: raw fields -> 32 f values + per-part (A, B).
// `blk` points at the block (shared or global memory); Q4_K/Q5_K blocks must
// be 16-byte aligned, Q6_K blocks 2-byte aligned.
// ---------------------------------------------------------------------------
template <int QT> struct LaneDecoded {
  float f[32];
  float A[Fmt<QT>::P];
  float B[Fmt<QT>::P];
};

// Integer view of the same lane share, for the unpack / dequant kernels.
template <int QT> struct LaneFields {
  uint32_t pre[8];        // pre-bytes, 4 codes per word, in weight order of the parts
  int sc[Fmt<QT>::P];     // scale of each part
  int m[Fmt<QT>::P];      // min of each part (Q4_K/Q5_K)
  uint32_t d_bits, dmin_bits;
  float d, dmin;          // decoded (IA4: scale and minus bias of the lane's group)
};

template <int QT>
__device__ __forceinline__ void lane_fields(const uint8_t* blk, int j, LaneFields<QT>& o) {
  if constexpr (QT == T_Q6_K) {
    const int h = j >> 2, l0 = 8 * (j & 3);
    const uint2 a = ld8_a2(blk + 64 * h + l0);
    const uint2 b = ld8_a2(blk + 64 * h + 32 + l0);
    const uint2 c = ld8_a2(blk + 128 + 32 * h + l0);
    uint32_t p0[4], p1[4];
    q6k_pre(a.x, b.x, c.x, p0);
    q6k_pre(a.y, b.y, c.y, p1);
#pragma unroll
    for (int t = 0; t < 4; ++t) { o.pre[2 * t] = p0[t]; o.pre[2 * t + 1] = p1[t]; }
    // scales 8h + (l0>>4) + 2t, t = 0..3: bytes at stride 2 from that offset
    const uint2 s = ld8_a2(blk + 192 + 8 * h + (l0 >> 4));
    const uint32_t se = __byte_perm(s.x, s.y, 0x6420);
    o.sc[0] = static_cast<int>(static_cast<int8_t>(se & 0xFF));
    o.sc[1] = static_cast<int>(static_cast<int8_t>((se >> 8) & 0xFF));
    o.sc[2] = static_cast<int>(static_cast<int8_t>((se >> 16) & 0xFF));
    o.sc[3] = static_cast<int>(static_cast<int8_t>(se >> 24));
    o.m[0] = o.m[1] = o.m[2] = o.m[3] = 0;
    o.d_bits = reinterpret_cast<const uint16_t*>(blk + 208)[0];
    o.dmin_bits = 0;
    o.d = half_bits_to_float(o.d_bits);
    o.dmin = 0.0f;
  } else {
    const int g = j >> 1, hh = j & 1;
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
    constexpr int QS = kQ4Codes<QT> ? 16 : 48;
    const uint4 qs = *reinterpret_cast<const uint4*>(blk + QS + 32 * g + 16 * hh);
    const uint32_t wq[4] = {qs.x, qs.y, qs.z, qs.w};
    if constexpr (kQ4Codes<QT>) {
#pragma unroll
      for (int w = 0; w < 4; ++w) q4k_pre(wq[w], o.pre[w], o.pre[4 + w]);
    } else {
      const uint4 qh = *reinterpret_cast<const uint4*>(blk + 16 + 16 * hh);
      const uint32_t wh[4] = {qh.x, qh.y, qh.z, qh.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) q5k_pre(wq[w], wh[w], g, o.pre[w], o.pre[4 + w]);
    }
    if constexpr (QT == T_IA4) {
      o.sc[0] = o.sc[1] = o.m[0] = o.m[1] = 1;
      o.d_bits = o.dmin_bits = 0;
      o.d = ia4_scale(hdr, g);
      o.dmin = ia4_neg_bias(hdr, g);
    } else {
      const uint32_t v = scale_min_bytes(hdr.y, hdr.z, hdr.w, g);
      o.sc[0] = v & 0xFF;
      o.sc[1] = (v >> 8) & 0xFF;
      o.m[0] = (v >> 16) & 0xFF;
      o.m[1] = v >> 24;
      o.d_bits = hdr.x & 0xFFFF;
      o.dmin_bits = hdr.x >> 16;
      o.d = half_bits_to_float(o.d_bits);
      o.dmin = half_bits_to_float(o.dmin_bits);
    }
  }
}

// Code of weight i (0..31 in part order) from the pre-bytes.
template <int QT>
__device__ __forceinline__ int code_of(const LaneFields<QT>& o, int i) {
  const uint32_t byte = (o.pre[i >> 2] >> (8 * (i & 3))) & 0x7F;
  return static_cast<int>(byte >> (7 - Fmt<QT>::SHIFT));
}

// Float decode for the products.  `nvalid` = number of leading parts that lie
// inside the matrix (parts past K get A = B = 0 and contribute exactly 0).
template <int QT>
__device__ __forceinline__ void lane_decode(const uint8_t* blk, int j, int nvalid, LaneDecoded<QT>& o) {
  LaneFields<QT> fl;
  lane_fields<QT>(blk, j, fl);
#pragma unroll
  for (int w = 0; w < 8; ++w) {
#pragma unroll
    for (int k = 0; k < 4; ++k) o.f[4 * w + k] = byte_to_f(fl.pre[w], k);
  }
  constexpr float S = static_cast<float>(1 << Fmt<QT>::SHIFT);
  const float d = fl.d;
  if constexpr (QT == T_Q6_K) {
    const float dS = d * S, dB = -(S + 32.0f) * d;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float sc = static_cast<float>(fl.sc[p]);
      const bool ok = p < nvalid;
      o.A[p] = ok ? dS * sc : 0.0f;
      o.B[p] = ok ? dB * sc : 0.0f;
    }
  } else {
    const float dmin = fl.dmin;
    const float dS = d * S;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const float a = dS * static_cast<float>(fl.sc[p]);
      const float mm = dmin * static_cast<float>(fl.m[p]);
      const bool ok = p < nvalid;
      o.A[p] = ok ? a : 0.0f;
      o.B[p] = ok ? -(a + mm) : 0.0f;
    }
  }
}

// Number of leading parts of lane j inside the first `rem` weights of a block
// (rem = 256 except in the last block of a row whose length is not a multiple
// of 256; rem is a multiple of 32).
template <int QT>
__device__ __forceinline__ int lane_valid_parts(int j, int rem) {
  if (rem >= 256) return Fmt<QT>::P;
  int n = 0;
#pragma unroll
  for (int p = 0; p < Fmt<QT>::P; ++p) n += (part_pos<QT>(j, p) + Fmt<QT>::L <= rem) ? 1 : 0;
  return n;
}

}  // namespace kq
