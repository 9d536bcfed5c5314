// kq_lane.cuh -- the per-lane arithmetic of the CUDA-core products with one
// x vector per pass (one-token products, routed-expert products): the
// shared-memory image of x as block-floating-point integer limbs, and the
// exact integer dot products of one lane's 64 weights of a block.
//
// "GGUF in transformers", section "Reusing ggml's Metal kernels": products
// read the packed super-blocks directly; the dequantization formulas
//   Q4_K/Q5_K: w = d*sc_j*q - dmin*m_j (32-weight sub-blocks),
//   Q6_K:      w = d*sc_j*(q - 32)     (16-weight sub-blocks)
// are applied per sub-block to exact integer sums, never per weight.
//
// x image: for every run of 128 consecutive values a power-of-two scale
// s = 2^(e - 14) (bf16 x, 2 byte limbs) or 2^(e - 22) (fp32 x, 3 limbs), e the
// binary exponent of the run's largest |x|, and m_k = rint(x_k / s),
// |m_k| <= 2^14 (2^22).  Every bf16 value within 2^7 of its run maximum is
// exact; otherwise |x_k - s*m_k| <= s/2.  Exact integer sums of m over every
// 16- and 32-run sit beside the limbs.
//
// Lane c of a quad owns 64 weights of a block (Q4_K/Q5_K: sub-blocks 2c,
// 2c+1; Q6_K: four 16-runs of one 128-half); with bf16 x its contribution is
// an exact int32 (bounds stated at each core), scaled once in fp32.
#pragma once

#include "kq_internal.h"

namespace kq {
namespace lane {

constexpr int XWB = 80;  // padded limb words per 256-block

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ int dp_us(uint32_t a, uint32_t b, int c) {  // unsigned codes x signed limb
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp_uu(uint32_t a, uint32_t b, int c) {  // unsigned codes x unsigned limb
  int d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
// signed byte p of v, sign-extended
__device__ __forceinline__ int sbyte(uint32_t v, int p) {
  uint32_t d;
  const uint32_t sel = static_cast<uint32_t>(p | ((p | 8) << 4) | ((p | 8) << 8) | ((p | 8) << 12));
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(d) : "r"(v), "r"(sel));
  return static_cast<int>(d);
}
// Shared-memory loads by 32-bit shared-window address.
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t w4(const uint4& v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }
// 16 bytes from a 2-byte aligned shared address (five aligned words, funnel shifts)
__device__ __forceinline__ uint4 lds16_a2(uint32_t a) {
  const uint32_t w = a & ~3u, sh = (a & 3u) * 8;
  const uint32_t w0 = lds32(w), w1 = lds32(w + 4), w2 = lds32(w + 8), w3 = lds32(w + 12), w4v = lds32(w + 16);
  return make_uint4(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh), __funnelshift_r(w2, w3, sh),
                    __funnelshift_r(w3, w4v, sh));
}
// 8 bytes from a 2-byte aligned shared address
__device__ __forceinline__ uint2 lds8_a2(uint32_t a) {
  const uint32_t w = a & ~3u, sh = (a & 3u) * 8;
  const uint32_t w0 = lds32(w), w1 = lds32(w + 4), w2 = lds32(w + 8);
  return make_uint2(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh));
}
__device__ __forceinline__ int wpad_i(int i) { return i + 4 * (i >> 4); }


// ------------------------------------------------------------- x image
// Shared-memory layout for nb blocks and NL limbs (16-byte aligned base):
//   limb[NL][nb*80] words   word i of block b at b*80 + wpad(i), byte j = x[256b+4i+j]
//   si16q[nb*16]            16-run sums in Q6_K lane order: [b*16 + 4c + p] = run 8(c>>1) + (c&1) + 2p
//   si32[nb*8]              32-run sums
//   scale[nb*2]             128-run scales
struct XImg {
  uint32_t* limb;
  int* si16q;
  int* si32;
  float* scale;
  int plane;  // words per limb plane
  uint32_t limb_s, si16q_s, si32_s, scale_s;  // the same as shared-window addresses
};
__host__ __device__ inline size_t ximg_bytes(int nb, int nl) {
  return static_cast<size_t>(nb) * (320 * nl + 64 + 32 + 8);
}
__device__ __forceinline__ XImg ximg_at(uint8_t* base, int nb, int nl) {
  XImg xi;
  xi.plane = nb * XWB;
  xi.limb = reinterpret_cast<uint32_t*>(base);
  xi.si16q = reinterpret_cast<int*>(base + static_cast<size_t>(nb) * 320 * nl);
  xi.si32 = xi.si16q + nb * 16;
  xi.scale = reinterpret_cast<float*>(xi.si32 + nb * 8);
  xi.limb_s = smem_u32(xi.limb);
  xi.si16q_s = smem_u32(xi.si16q);
  xi.si32_s = smem_u32(xi.si32);
  xi.scale_s = smem_u32(xi.scale);
  return xi;
}

// Limb word of four integers: byte k of each (k = 0 least significant).
__device__ __forceinline__ uint32_t pack_byte(int m0, int m1, int m2, int m3, int k) {
  const uint32_t sel = static_cast<uint32_t>(k | ((4 + k) << 4));
  const uint32_t a = __byte_perm(static_cast<uint32_t>(m0), static_cast<uint32_t>(m1), sel);
  const uint32_t b = __byte_perm(static_cast<uint32_t>(m2), static_cast<uint32_t>(m3), sel);
  return __byte_perm(a, b, 0x5410);
}

// Writes oct o of the image from its integer values m[8] and the run's scale
// (all lanes of the warp call it: the 16- and 32-run sums are shuffled).
template <int NL>
__device__ __forceinline__ void put_oct(const int (&m)[8], float scale, int o, int noct, const XImg& xi) {
  int isum = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) isum += m[j];
  const int s16 = isum + __shfl_xor_sync(0xFFFFFFFFu, isum, 1);
  const int s32 = s16 + __shfl_xor_sync(0xFFFFFFFFu, s16, 2);
  if (o < noct) {
    const int b = o >> 5, i = o & 31;
#pragma unroll
    for (int l = 0; l < NL; ++l) {
      const int k = NL - 1 - l;  // limb 0 = the most significant byte (signed)
      const uint2 wv = make_uint2(pack_byte(m[0], m[1], m[2], m[3], k), pack_byte(m[4], m[5], m[6], m[7], k));
      *reinterpret_cast<uint2*>(xi.limb + l * xi.plane + b * XWB + wpad_i(2 * i)) = wv;
    }
    if ((o & 15) == 0) xi.scale[o >> 4] = scale;
    if ((o & 3) == 0) xi.si32[o >> 2] = s32;
    if ((o & 1) == 0) {
      const int r = (o >> 1) & 15;  // 16-run within the block
      const int h = r >> 3, rr = r & 7;
      xi.si16q[b * 16 + 4 * (2 * h + (rr & 1)) + (rr >> 1)] = s16;
    }
  }
}

// An oct whose 128-run maximum mx is zero, subnormal or huge (the exponent
// taken with frexpf, the values scaled with ldexpf): out of line, rare.
template <int NL>
__device__ __noinline__ void stage_oct_slow(float v0, float v1, float v2, float v3, float v4, float v5, float v6,
                                            float v7, float mx, int o, int noct, const XImg& xi) {
  int e = 0;
  frexpf(mx, &e);
  const int shift = (NL == 2 ? 14 : 22) - e;
  const float v[8] = {v0, v1, v2, v3, v4, v5, v6, v7};
  int m[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) m[j] = (mx > 0.0f) ? __float2int_rn(ldexpf(v[j], shift)) : 0;
  put_oct<NL>(m, (mx > 0.0f) ? ldexpf(1.0f, -shift) : 0.0f, o, noct, xi);
}

// All consumer threads: quantize x[0..K) (zero past K up to nb*256) into xi.
// Thread t takes "octs" (8 consecutive values) t, t+T, ...; the 32 octs of a
// warp are one 256-block, 16 lanes one 128-run.  All global loads of a pass
// (up to 6 octs a thread) are issued before any is used.
template <int NL, int NTHR>
__device__ void stage_x(const void* xp, int x_bf16, int K, int nb, const XImg& xi, int tid) {
  constexpr int MAXO = 6;
  const int noct = nb * 32;
  const int lane = tid & 31;
  for (int base = 0; base < noct; base += MAXO * NTHR) {
    float v[MAXO][8];
#pragma unroll
    for (int it = 0; it < MAXO; ++it) {
      const int o = base + it * NTHR + tid;
#pragma unroll
      for (int j = 0; j < 8; ++j) v[it][j] = 0.0f;
      if (o < noct && 8 * o < K) {  // K is a multiple of 32: an oct is all in or all out
        if (x_bf16) {
          const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(xp) + 8 * o);
          v[it][0] = __uint_as_float(u.x << 16); v[it][1] = __uint_as_float(u.x & 0xFFFF0000u);
          v[it][2] = __uint_as_float(u.y << 16); v[it][3] = __uint_as_float(u.y & 0xFFFF0000u);
          v[it][4] = __uint_as_float(u.z << 16); v[it][5] = __uint_as_float(u.z & 0xFFFF0000u);
          v[it][6] = __uint_as_float(u.w << 16); v[it][7] = __uint_as_float(u.w & 0xFFFF0000u);
        } else {
          const float4 a = *reinterpret_cast<const float4*>(static_cast<const float*>(xp) + 8 * o);
          const float4 b = *reinterpret_cast<const float4*>(static_cast<const float*>(xp) + 8 * o + 4);
          v[it][0] = a.x; v[it][1] = a.y; v[it][2] = a.z; v[it][3] = a.w;
          v[it][4] = b.x; v[it][5] = b.y; v[it][6] = b.z; v[it][7] = b.w;
        }
      }
    }
#pragma unroll
    for (int it = 0; it < MAXO; ++it) {
      const int o = base + it * NTHR + tid;
      if (o - lane >= noct) continue;  // whole warp past the end (noct is a multiple of 32)
      float mx = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) mx = fmaxf(mx, fabsf(v[it][j]));
#pragma unroll
      for (int w = 1; w < 16; w <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, w));
      // mx = f * 2^e, f in [0.5, 1): from the bits for normal values
      const uint32_t mb = __float_as_uint(mx);
      const int be = static_cast<int>((mb >> 23) & 0xFF);
      if (__any_sync(0xFFFFFFFFu, be < 40 || be > 200)) {  // a run of this warp takes the slow path
        stage_oct_slow<NL>(v[it][0], v[it][1], v[it][2], v[it][3], v[it][4], v[it][5], v[it][6], v[it][7], mx, o,
                           noct, xi);
        continue;
      }
      const int shift = (NL == 2 ? 14 : 22) - (be - 126);
      const float p2 = __uint_as_float(static_cast<uint32_t>(127 + shift) << 23);
      int m[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) m[j] = __float2int_rn(v[it][j] * p2);  // exact: power-of-two scale
      put_oct<NL>(m, __uint_as_float(static_cast<uint32_t>(127 - shift) << 23), o, noct, xi);
    }
  }
}

// ------------------------------------------------------- lane block cores
// Per-lane constants of the Q4_K/Q5_K scale unpacking (lane c owns
// sub-blocks j = 2c, 2c+1 of the 12-byte scale field s[0..11]):
//   j < 4 : sc = s[j] & 63,                      m = s[j+4] & 63
//   j >= 4: sc = (s[j+4] & 15) | (s[j-4]>>6)<<4,  m = (s[j+4]>>4) | (s[j]>>6)<<4
struct ScaleLane {
  uint32_t selP, mA, mB, selQ, mH;
  bool lowsrc;
};
__device__ __forceinline__ ScaleLane scale_lane(int c) {
  ScaleLane s;
  if (c < 2) {
    const uint32_t j = 2 * c;
    s.selP = j | ((j + 1) << 4) | ((j + 4) << 8) | ((j + 5) << 12);
    s.mA = 0x3F3F3F3Fu; s.mB = 0; s.selQ = 0; s.mH = 0; s.lowsrc = true;
  } else {
    const uint32_t i = 2 * c - 4;
    s.selP = i | ((i + 1) << 4) | (i << 8) | ((i + 1) << 12);
    s.mA = 0x00000F0Fu; s.mB = 0x0F0F0000u;
    s.selQ = i | ((i + 1) << 4) | ((i + 4) << 8) | ((i + 5) << 12);
    s.mH = 0x30303030u; s.lowsrc = false;
  }
  return s;
}

// x slice of one block for lane c: NL limb planes x 16 words, in the lane's
// part order (Q4_K/Q5_K: parts 0,1 = words 0..7, 8..15; Q6_K: part p = words 4p..4p+3).
template <int NL>
struct XSlice {
  uint32_t w[NL][16];
};
template <int QT, int NL>
__device__ __forceinline__ void load_slice(uint32_t xl, uint32_t plane, XSlice<NL>& X) {
#pragma unroll
  for (int l = 0; l < NL; ++l)
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      // word offsets (relative, padded layout) of the lane's 4-word groups
      const int off = (QT == T_Q6_K) ? ((p == 0) ? 0 : (p == 1) ? 8 : (p == 2) ? 20 : 28) : 4 * p;
      const uint4 u = lds128(xl + l * plane + 4 * off);
      X.w[l][4 * p] = u.x; X.w[l][4 * p + 1] = u.y; X.w[l][4 * p + 2] = u.z; X.w[l][4 * p + 3] = u.w;
    }
}

// Q4_K / Q5_K: lane c's 64 weights of the block at bp (16-byte aligned);
// si = the lane's two 32-run sums of m, s = the 128-run scale.
template <int QT, int NL>
__device__ __forceinline__ float core_q45(uint32_t bp, const XSlice<NL>& X, int2 si, float s, int c,
                                          const ScaleLane& sl, float acc) {
  const uint4 hdr = lds128(bp);
  constexpr int QS = kQ4Codes<QT> ? 16 : 48;
  const uint4 q0 = lds128(bp + QS + 32 * c);
  const uint4 q1 = lds128(bp + QS + 32 * c + 16);
  uint4 h0 = make_uint4(0, 0, 0, 0), h1 = make_uint4(0, 0, 0, 0);
  if constexpr (QT == T_Q5_K) { h0 = lds128(bp + 16); h1 = lds128(bp + 32); }
  int I[2][NL];
#pragma unroll
  for (int p = 0; p < 2; ++p)
#pragma unroll
    for (int l = 0; l < NL; ++l) I[p][l] = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint32_t q = (w < 4) ? w4(q0, w) : w4(q1, w - 4);
    uint32_t lo, hi;
    if constexpr (kQ4Codes<QT>) {
      lo = q & 0x0F0F0F0Fu;
      hi = q & 0xF0F0F0F0u;  // 16 x the high nibble: the factor leaves T_1 exactly
    } else {
      const uint32_t hb = (w < 4) ? w4(h0, w) : w4(h1, w - 4);
      lo = (q & 0x0F0F0F0Fu) | (__funnelshift_l(hb, hb, (4 - 2 * c) & 31) & 0x10101010u);
      hi = ((q >> 4) & 0x0F0F0F0Fu) | (__funnelshift_l(hb, hb, (3 - 2 * c) & 31) & 0x10101010u);
    }
    I[0][0] = dp_us(lo, X.w[0][w], I[0][0]);
    I[1][0] = dp_us(hi, X.w[0][8 + w], I[1][0]);
#pragma unroll
    for (int l = 1; l < NL; ++l) {
      I[0][l] = dp_uu(lo, X.w[l][w], I[0][l]);
      I[1][l] = dp_uu(hi, X.w[l][8 + w], I[1][l]);
    }
  }
  // scales and mins of sub-blocks 2c, 2c+1
  int sc0 = 1, sc1 = 1, m0 = 1, m1 = 1;
  float d, dmin;
  if constexpr (QT == T_IA4) {  // the lane's two sub-blocks are group c: one scale, one bias
    d = ia4_scale(hdr, c);
    dmin = ia4_neg_bias(hdr, c);
  } else {
    const uint32_t P = __byte_perm(sl.lowsrc ? hdr.y : hdr.w, hdr.z, sl.selP);
    const uint32_t Q = __byte_perm(hdr.y, hdr.z, sl.selQ);
    const uint32_t L = (P & sl.mA) | ((P >> 4) & sl.mB) | ((Q >> 2) & sl.mH);
    sc0 = static_cast<int>(L & 0xFF);
    sc1 = static_cast<int>((L >> 8) & 0xFF);
    m0 = static_cast<int>((L >> 16) & 0xFF);
    m1 = static_cast<int>(L >> 24);
    d = half_bits_to_float(hdr.x & 0xFFFF);
    dmin = half_bits_to_float(hdr.x >> 16);
  }
  if constexpr (NL == 2) {
    const int T0 = I[0][0] * 256 + I[0][1];
    int T1 = I[1][0] * 256 + I[1][1];
    if constexpr (kQ4Codes<QT>) T1 >>= 4;  // exact: every term is a multiple of 16
    const int Y = sc0 * T0 + sc1 * T1;
    const int Mi = m0 * si.x + m1 * si.y;
    return __fmaf_rn(s, __fmaf_rn(d, static_cast<float>(Y), -dmin * static_cast<float>(Mi)), acc);
  } else {
    int Yl[NL];
#pragma unroll
    for (int l = 0; l < NL; ++l) {
      int t1 = I[1][l];
      if constexpr (kQ4Codes<QT>) t1 >>= 4;
      Yl[l] = sc0 * I[0][l] + sc1 * t1;
    }
    const float Yf = __fmaf_rn(static_cast<float>(Yl[0]), 65536.0f,
                               __fmaf_rn(static_cast<float>(Yl[1]), 256.0f, static_cast<float>(Yl[2])));
    const float Mf = __fmaf_rn(static_cast<float>(m0), static_cast<float>(si.x),
                               static_cast<float>(m1) * static_cast<float>(si.y));
    return __fmaf_rn(s, __fmaf_rn(d, Yf, -dmin * Mf), acc);
  }
}

// Q6_K: lane c's four 16-runs (128-half h = c>>1, runs 8h + 2p + (c&1)) of
// the block at bp (2-byte aligned).
template <int NL>
__device__ __forceinline__ float core_q6(uint32_t bp, const XSlice<NL>& X, int4 si, float s, int c,
                                         float acc) {
  const int h = c >> 1, e = c & 1;
  const uint4 qa = lds16_a2(bp + 64 * h + 16 * e);
  const uint4 qb = lds16_a2(bp + 64 * h + 32 + 16 * e);
  const uint4 qh = lds16_a2(bp + 128 + 32 * h + 16 * e);
  const uint2 sv = lds8_a2(bp + 192 + 8 * h);
  const uint32_t se = __byte_perm(sv.x, sv.y, e ? 0x7531 : 0x6420);  // scales 8h + 2p + e, p = 0..3
  const float d = half_bits_to_float(lds16(bp + 208));
  int I[4][NL];
#pragma unroll
  for (int p = 0; p < 4; ++p)
#pragma unroll
    for (int l = 0; l < NL; ++l) I[p][l] = 0;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint32_t a = w4(qa, w), b = w4(qb, w), hv = w4(qh, w);
    uint32_t cd[4];
    cd[0] = (a & 0x0F0F0F0Fu) | ((hv << 4) & 0x30303030u);
    cd[1] = (b & 0x0F0F0F0Fu) | ((hv << 2) & 0x30303030u);
    cd[2] = ((a >> 4) & 0x0F0F0F0Fu) | (hv & 0x30303030u);
    cd[3] = ((b >> 4) & 0x0F0F0F0Fu) | ((hv >> 2) & 0x30303030u);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      I[p][0] = dp_us(cd[p], X.w[0][4 * p + w], I[p][0]);
#pragma unroll
      for (int l = 1; l < NL; ++l) I[p][l] = dp_uu(cd[p], X.w[l][4 * p + w], I[p][l]);
    }
  }
  const int sc0 = sbyte(se, 0), sc1 = sbyte(se, 1), sc2 = sbyte(se, 2), sc3 = sbyte(se, 3);
  const float sd = s * d;
  if constexpr (NL == 2) {
    const int T0 = I[0][0] * 256 + I[0][1] - 32 * si.x;
    const int T1 = I[1][0] * 256 + I[1][1] - 32 * si.y;
    const int T2 = I[2][0] * 256 + I[2][1] - 32 * si.z;
    const int T3 = I[3][0] * 256 + I[3][1] - 32 * si.w;
    const int Ya = sc0 * T0 + sc1 * T1;  // |.| < 2^31 for any int8 scales
    const int Yb = sc2 * T2 + sc3 * T3;
    acc = __fmaf_rn(sd, static_cast<float>(Ya), acc);
    return __fmaf_rn(sd, static_cast<float>(Yb), acc);
  } else {
    int Yl[NL];
#pragma unroll
    for (int l = 0; l < NL; ++l) Yl[l] = sc0 * I[0][l] + sc1 * I[1][l] + sc2 * I[2][l] + sc3 * I[3][l];
    const float Yf = __fmaf_rn(static_cast<float>(Yl[0]), 65536.0f,
                               __fmaf_rn(static_cast<float>(Yl[1]), 256.0f, static_cast<float>(Yl[2])));
    float Z = static_cast<float>(sc0) * static_cast<float>(si.x);
    Z = __fmaf_rn(static_cast<float>(sc1), static_cast<float>(si.y), Z);
    Z = __fmaf_rn(static_cast<float>(sc2), static_cast<float>(si.z), Z);
    Z = __fmaf_rn(static_cast<float>(sc3), static_cast<float>(si.w), Z);
    return __fmaf_rn(sd, __fmaf_rn(-32.0f, Z, Yf), acc);
  }
}


// ----------------------------------------------- several tokens per block
// The same lane arithmetic for MT tokens: the block's bytes are read and its
// codes and scales unpacked once, then dotted with every token's x slice.

// Q4_K / Q5_K (see core_q45): acc[t] += this lane's part of token t's row sum.
template <int QT, int NL, int MT>
__device__ __forceinline__ void core_q45_mt(uint32_t bp, const XSlice<NL> (&X)[MT], const int2 (&si)[MT],
                                            const float (&s)[MT], int c, const ScaleLane& sl, float (&acc)[MT]) {
  const uint4 hdr = lds128(bp);
  constexpr int QS = kQ4Codes<QT> ? 16 : 48;
  const uint4 q0 = lds128(bp + QS + 32 * c);
  const uint4 q1 = lds128(bp + QS + 32 * c + 16);
  uint4 h0 = make_uint4(0, 0, 0, 0), h1 = make_uint4(0, 0, 0, 0);
  if constexpr (QT == T_Q5_K) { h0 = lds128(bp + 16); h1 = lds128(bp + 32); }
  int I[MT][2][NL];
#pragma unroll
  for (int t = 0; t < MT; ++t)
#pragma unroll
    for (int p = 0; p < 2; ++p)
#pragma unroll
      for (int l = 0; l < NL; ++l) I[t][p][l] = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint32_t q = (w < 4) ? w4(q0, w) : w4(q1, w - 4);
    uint32_t lo, hi;
    if constexpr (kQ4Codes<QT>) {
      lo = q & 0x0F0F0F0Fu;
      hi = q & 0xF0F0F0F0u;  // 16 x the high nibble: the factor leaves T_1 exactly
    } else {
      const uint32_t hb = (w < 4) ? w4(h0, w) : w4(h1, w - 4);
      lo = (q & 0x0F0F0F0Fu) | (__funnelshift_l(hb, hb, (4 - 2 * c) & 31) & 0x10101010u);
      hi = ((q >> 4) & 0x0F0F0F0Fu) | (__funnelshift_l(hb, hb, (3 - 2 * c) & 31) & 0x10101010u);
    }
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      I[t][0][0] = dp_us(lo, X[t].w[0][w], I[t][0][0]);
      I[t][1][0] = dp_us(hi, X[t].w[0][8 + w], I[t][1][0]);
#pragma unroll
      for (int l = 1; l < NL; ++l) {
        I[t][0][l] = dp_uu(lo, X[t].w[l][w], I[t][0][l]);
        I[t][1][l] = dp_uu(hi, X[t].w[l][8 + w], I[t][1][l]);
      }
    }
  }
  int sc0 = 1, sc1 = 1, m0 = 1, m1 = 1;
  float d, dmin;
  if constexpr (QT == T_IA4) {  // the lane's two sub-blocks are group c: one scale, one bias
    d = ia4_scale(hdr, c);
    dmin = ia4_neg_bias(hdr, c);
  } else {
    const uint32_t P = __byte_perm(sl.lowsrc ? hdr.y : hdr.w, hdr.z, sl.selP);
    const uint32_t Q = __byte_perm(hdr.y, hdr.z, sl.selQ);
    const uint32_t L = (P & sl.mA) | ((P >> 4) & sl.mB) | ((Q >> 2) & sl.mH);
    sc0 = static_cast<int>(L & 0xFF);
    sc1 = static_cast<int>((L >> 8) & 0xFF);
    m0 = static_cast<int>((L >> 16) & 0xFF);
    m1 = static_cast<int>(L >> 24);
    d = half_bits_to_float(hdr.x & 0xFFFF);
    dmin = half_bits_to_float(hdr.x >> 16);
  }
#pragma unroll
  for (int t = 0; t < MT; ++t) {
    if constexpr (NL == 2) {
      const int T0 = I[t][0][0] * 256 + I[t][0][1];
      int T1 = I[t][1][0] * 256 + I[t][1][1];
      if constexpr (kQ4Codes<QT>) T1 >>= 4;
      const int Y = sc0 * T0 + sc1 * T1;
      const int Mi = m0 * si[t].x + m1 * si[t].y;
      acc[t] = __fmaf_rn(s[t], __fmaf_rn(d, static_cast<float>(Y), -dmin * static_cast<float>(Mi)), acc[t]);
    } else {
      int Yl[NL];
#pragma unroll
      for (int l = 0; l < NL; ++l) {
        int t1 = I[t][1][l];
        if constexpr (kQ4Codes<QT>) t1 >>= 4;
        Yl[l] = sc0 * I[t][0][l] + sc1 * t1;
      }
      const float Yf = __fmaf_rn(static_cast<float>(Yl[0]), 65536.0f,
                                 __fmaf_rn(static_cast<float>(Yl[1]), 256.0f, static_cast<float>(Yl[2])));
      const float Mf = __fmaf_rn(static_cast<float>(m0), static_cast<float>(si[t].x),
                                 static_cast<float>(m1) * static_cast<float>(si[t].y));
      acc[t] = __fmaf_rn(s[t], __fmaf_rn(d, Yf, -dmin * Mf), acc[t]);
    }
  }
}

// Q6_K (see core_q6), MT tokens.
template <int NL, int MT>
__device__ __forceinline__ void core_q6_mt(uint32_t bp, const XSlice<NL> (&X)[MT], const int4 (&si)[MT],
                                           const float (&s)[MT], int c, float (&acc)[MT]) {
  const int h = c >> 1, e = c & 1;
  const uint4 qa = lds16_a2(bp + 64 * h + 16 * e);
  const uint4 qb = lds16_a2(bp + 64 * h + 32 + 16 * e);
  const uint4 qh = lds16_a2(bp + 128 + 32 * h + 16 * e);
  const uint2 sv = lds8_a2(bp + 192 + 8 * h);
  const uint32_t se = __byte_perm(sv.x, sv.y, e ? 0x7531 : 0x6420);  // scales 8h + 2p + e, p = 0..3
  const float d = half_bits_to_float(lds16(bp + 208));
  int I[MT][4][NL];
#pragma unroll
  for (int t = 0; t < MT; ++t)
#pragma unroll
    for (int p = 0; p < 4; ++p)
#pragma unroll
      for (int l = 0; l < NL; ++l) I[t][p][l] = 0;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint32_t a = w4(qa, w), b = w4(qb, w), hv = w4(qh, w);
    uint32_t cd[4];
    cd[0] = (a & 0x0F0F0F0Fu) | ((hv << 4) & 0x30303030u);
    cd[1] = (b & 0x0F0F0F0Fu) | ((hv << 2) & 0x30303030u);
    cd[2] = ((a >> 4) & 0x0F0F0F0Fu) | (hv & 0x30303030u);
    cd[3] = ((b >> 4) & 0x0F0F0F0Fu) | ((hv >> 2) & 0x30303030u);
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        I[t][p][0] = dp_us(cd[p], X[t].w[0][4 * p + w], I[t][p][0]);
#pragma unroll
        for (int l = 1; l < NL; ++l) I[t][p][l] = dp_uu(cd[p], X[t].w[l][4 * p + w], I[t][p][l]);
      }
  }
  const int sc0 = sbyte(se, 0), sc1 = sbyte(se, 1), sc2 = sbyte(se, 2), sc3 = sbyte(se, 3);
#pragma unroll
  for (int t = 0; t < MT; ++t) {
    const float sd = s[t] * d;
    if constexpr (NL == 2) {
      const int T0 = I[t][0][0] * 256 + I[t][0][1] - 32 * si[t].x;
      const int T1 = I[t][1][0] * 256 + I[t][1][1] - 32 * si[t].y;
      const int T2 = I[t][2][0] * 256 + I[t][2][1] - 32 * si[t].z;
      const int T3 = I[t][3][0] * 256 + I[t][3][1] - 32 * si[t].w;
      const int Ya = sc0 * T0 + sc1 * T1;
      const int Yb = sc2 * T2 + sc3 * T3;
      acc[t] = __fmaf_rn(sd, static_cast<float>(Ya), acc[t]);
      acc[t] = __fmaf_rn(sd, static_cast<float>(Yb), acc[t]);
    } else {
      int Yl[NL];
#pragma unroll
      for (int l = 0; l < NL; ++l)
        Yl[l] = sc0 * I[t][0][l] + sc1 * I[t][1][l] + sc2 * I[t][2][l] + sc3 * I[t][3][l];
      const float Yf = __fmaf_rn(static_cast<float>(Yl[0]), 65536.0f,
                                 __fmaf_rn(static_cast<float>(Yl[1]), 256.0f, static_cast<float>(Yl[2])));
      float Z = static_cast<float>(sc0) * static_cast<float>(si[t].x);
      Z = __fmaf_rn(static_cast<float>(sc1), static_cast<float>(si[t].y), Z);
      Z = __fmaf_rn(static_cast<float>(sc2), static_cast<float>(si[t].z), Z);
      Z = __fmaf_rn(static_cast<float>(sc3), static_cast<float>(si[t].w), Z);
      acc[t] = __fmaf_rn(sd, __fmaf_rn(-32.0f, Z, Yf), acc[t]);
    }
  }
}


}  // namespace lane
}  // namespace kq
