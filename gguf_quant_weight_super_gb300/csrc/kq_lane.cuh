// kq_lane.cuh -- the per-lane arithmetic of the CUDA-core products that stage
// x in shared memory (one-token and few-token products, routed-expert
// products): the exact shared-memory image of x, and the exact integer dot
// products of one lane's 64 weights of a block.
//
// "GGUF in transformers", section "Reusing ggml's Metal kernels": products
// read the packed super-blocks directly; the dequantization formulas
//   Q4_K/Q5_K: w = d*sc_j*q - dmin*m_j (32-weight sub-blocks),
//   Q6_K:      w = d*sc_j*(q - 32)     (16-weight sub-blocks)
// are applied per sub-block to exact integer sums, never per weight.
//
// The x image (one per bf16 vector; an fp32 vector is staged as two, its
// bf16 rounding hi = bf16(x) and the rounding of the rest lo = bf16(x - hi),
// which leaves out at most 2^-18 |x| per element):
//  * every block of 256 consecutive values has a power-of-two scale
//    s = 2^(e-22), e the binary exponent of the block's largest |x| (2^-149
//    at the least);
//  * a value that is an integer multiple m of s -- every bf16 value within
//    2^15 of its block's maximum -- is held exactly as m, |m| <= 2^22, split
//    into three byte limbs (the top one signed);
//  * any other value is held as m = 0 and listed with its block (its index
//    and bf16 bits), up to ECAP per block; a block with more listed values
//    keeps all 256 values as bf16 instead ("raw" block);
//  * exact integer sums of m over every 16- and 32-run sit beside the limbs.
// So the image represents x exactly; nothing in a product is rounded before
// the per-lane combine.
//
// Codes times limbs are summed exactly with dp4a over 64-weight chunks; a
// block's (or chunk's) contribution d*Y - dmin*Mi (Q6_K: d*Y) is then formed
// from exact integers Y, Mi and rounded once (see combine45), and a listed
// value adds fl(w_k * x_k) with w_k the exactly rounded fp32 weight.
#pragma once

#include <cuda_bf16.h>

#include "kq_internal.h"

namespace kq {
namespace lane {

constexpr int XWB = 84;               // words per block in each limb plane: 64 limb words + 20 side words
constexpr int NLB = 3;                // limb planes (24-bit integers)
constexpr int ECAP = 32;              // listed values a block holds in its side words
constexpr uint32_t kRaw = 0xFFFFu;    // entry count of a block kept as raw bf16 values

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
__device__ __forceinline__ uint32_t lds8(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(a));
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

// f * 2^e for e in [-190, 191]: two exact power-of-two products (only a
// result outside the normal range rounds).
__device__ __forceinline__ float mul_pow2(float f, int e) {
  const int e1 = e < -126 ? -64 : (e > 127 ? 64 : 0);
  return (f * __uint_as_float(static_cast<uint32_t>(127 + e1) << 23)) *
         __uint_as_float(static_cast<uint32_t>(127 + e - e1) << 23);
}
// v rounded to the nearest fp32 (ties to even), in single-precision and
// integer operations only: |v| below 2^48 is split into two parts of 24 bits,
// each converted exactly, and one fma rounds their sum once; a larger |v|
// first drops its low 16 bits into a sticky bit (the result keeps at least 32
// significant bits, so the one rounding is unchanged) and is scaled back by
// 2^16 exactly.
__device__ __forceinline__ float ll2f_rn(long long v) {
  const unsigned long long a = v < 0 ? 0ull - static_cast<unsigned long long>(v) : static_cast<unsigned long long>(v);
  unsigned long long b = a;
  float scale = 1.0f;
  if (a >= (1ull << 48)) {
    b = (a >> 16) | ((a & 0xFFFFull) != 0 ? 1ull : 0ull);
    scale = 65536.0f;
  }
  const float r = __fmaf_rn(__uint2float_rn(static_cast<uint32_t>(b >> 24)), 16777216.0f,
                            __uint2float_rn(static_cast<uint32_t>(b & 0xFFFFFFull))) * scale;
  return v < 0 ? -r : r;
}
// 2^e as a float for e in [-149, 127] (subnormal below -126)
__device__ __forceinline__ float pow2f(int e) {
  return e >= -126 ? __uint_as_float(static_cast<uint32_t>(127 + e) << 23) : __uint_as_float(1u << (e + 149));
}

// ------------------------------------------------------------- x image
// Shared-memory layout for nb blocks: three limb planes of nb * 84 words;
// word wpad(i) of block b (b * 84 + i + 4 (i >> 4), i < 64) holds byte l of m
// for x[256b + 4i .. 256b + 4i + 3] in plane l (plane 0 = the top, signed
// byte).  The 20 side words of each block and plane -- group g < 4 at
// b * 84 + 16 + 20g, group 4 at b * 84 + 80, four words each -- hold:
//   plane 0, g = 0:     header {scale, scale, entry count (or kRaw), 0}
//   plane 0, g = 1, 2:  32-run sums, sum j at group 1 + j / 4, word j % 4
//   plane 0, g = 3, 4:  entries 0..7
//   plane 1, g = c < 4: 16-run sums in Q6_K lane order: word p = run 8(c>>1) + (c&1) + 2p
//   plane 1, g = 4:     entries 8..11
//   plane 2, g = 0..4:  entries 12..31
// One scale per block: s = 2^(e - 22), e the binary exponent of the block's
// largest |x|.  An entry is (bf16 bits << 16) | index within the block.  A
// raw block keeps value k as the bf16 half (k & 1) of word wpad((k & 127) / 2)
// of plane k / 128.  The side groups put the 16-byte slices of neighbouring
// blocks (84 words apart) and of one block's chunks in different bank groups.
struct XImg {
  uint32_t* limb;
  int plane;        // words per plane
  uint32_t limb_s;  // shared-window address of limb
};
__host__ __device__ inline size_t ximg_bytes(int nb) { return static_cast<size_t>(nb) * NLB * XWB * 4; }
__device__ __forceinline__ XImg ximg_at(uint8_t* base, int nb) {
  XImg xi;
  xi.plane = nb * XWB;
  xi.limb = reinterpret_cast<uint32_t*>(base);
  xi.limb_s = smem_u32(xi.limb);
  return xi;
}
__host__ __device__ constexpr int side_w(int g, int i) { return (g < 4 ? 16 + 20 * g : 80) + i; }
// shared addresses of a block's side data
__device__ __forceinline__ uint32_t hdr_s(const XImg& xi, int b) { return xi.limb_s + 4 * (b * XWB + side_w(0, 0)); }
__device__ __forceinline__ uint32_t si32_s(const XImg& xi, int b, int c) {  // sums 2c, 2c+1
  return xi.limb_s + 4 * (b * XWB + side_w(1 + (c >> 1), 2 * (c & 1)));
}
__device__ __forceinline__ uint32_t si16_s(const XImg& xi, int b, int c) {  // chunk c's four 16-run sums
  return xi.limb_s + 4 * (xi.plane + b * XWB + side_w(c, 0));
}
__device__ __forceinline__ int ent_word(const XImg& xi, int b, int j) {
  return j < 8 ? b * XWB + 76 + j
               : j < 12 ? xi.plane + b * XWB + 80 + (j - 8)
                        : 2 * xi.plane + b * XWB + side_w((j - 12) >> 2, (j - 12) & 3);
}
__device__ __forceinline__ int raw_word(const XImg& xi, int b, int k) {
  return (k >> 7) * xi.plane + b * XWB + wpad_i((k & 127) >> 1);
}

// Limb word of four integers: byte k of each (k = 0 least significant).
__device__ __forceinline__ uint32_t pack_byte(int m0, int m1, int m2, int m3, int k) {
  const uint32_t sel = static_cast<uint32_t>(k | ((4 + k) << 4));
  const uint32_t a = __byte_perm(static_cast<uint32_t>(m0), static_cast<uint32_t>(m1), sel);
  const uint32_t b = __byte_perm(static_cast<uint32_t>(m2), static_cast<uint32_t>(m3), sel);
  return __byte_perm(a, b, 0x5410);
}

// Off-grid values of an oct (odd: bit j set for value j): the block's entry
// list when the warp's total fits, else the oct's raw bf16 values.  Every
// lane of the warp calls it (the positions come from a warp scan).  Rare.
static __device__ __noinline__ void put_odd(float v0, float v1, float v2, float v3, float v4, float v5, float v6,
                                            float v7, uint32_t odd, int b, int i, const XImg xi, int lane) {
  const float v[8] = {v0, v1, v2, v3, v4, v5, v6, v7};
  const int n = __popc(odd);
  int incl = n;
#pragma unroll
  for (int w = 1; w < 32; w <<= 1) {
    const int t = __shfl_up_sync(0xFFFFFFFFu, incl, w);
    if (lane >= w) incl += t;
  }
  const int total = __shfl_sync(0xFFFFFFFFu, incl, 31);
  if (total <= ECAP) {
    int slot = incl - n;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if ((odd >> j) & 1u)
        xi.limb[ent_word(xi, b, slot++)] = (__float_as_uint(v[j]) & 0xFFFF0000u) | static_cast<uint32_t>(8 * i + j);
  } else {  // a raw block: all 256 values as bf16 (written after the limbs, which it replaces)
    __syncwarp();
    uint4 rv;
    rv.x = (__float_as_uint(v[0]) >> 16) | (__float_as_uint(v[1]) & 0xFFFF0000u);
    rv.y = (__float_as_uint(v[2]) >> 16) | (__float_as_uint(v[3]) & 0xFFFF0000u);
    rv.z = (__float_as_uint(v[4]) >> 16) | (__float_as_uint(v[5]) & 0xFFFF0000u);
    rv.w = (__float_as_uint(v[6]) >> 16) | (__float_as_uint(v[7]) & 0xFFFF0000u);
    *reinterpret_cast<uint4*>(xi.limb + raw_word(xi, b, 8 * i)) = rv;
  }
  if (i == 0) xi.limb[b * XWB + side_w(0, 2)] = total <= ECAP ? static_cast<uint32_t>(total) : kRaw;
}

// The scale exponent of a run whose maximum mx is zero, subnormal or huge
// (frexpf; the grid no finer than 2^-149).  Rare.
static __device__ __noinline__ int run_shift_slow(float mx) {
  if (!(mx > 0.0f)) return 0;
  int e = 0;
  frexpf(mx, &e);
  return min(22 - e, 149);
}

// Oct o (values 8o .. 8o+7, exact bf16 values as floats) of the image; every
// lane of the warp calls it together for the 32 octs of one block (lane =
// oct within the block).  The block's scale is set by its largest |v|.
__device__ __forceinline__ void put_oct(const float (&v)[8], int o, const XImg& xi, int lane) {
  float mx = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) mx = fmaxf(mx, fabsf(v[j]));
  // block maximum: non-negative floats order as their bit patterns
  mx = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(mx)));
  // shift = 22 - e, mx = f * 2^e, f in [0.5, 1): from the bits for normal values
  const int be = static_cast<int>((__float_as_uint(mx) >> 23) & 0xFFu);
  const int shift = (be >= 40 && be <= 200) ? 148 - be : run_shift_slow(mx);
  // m = v * 2^shift where that is an integer (exact: a power-of-two product
  // of a value whose run maximum keeps it below 2^22), else 0 and listed
  int m[8];
  uint32_t odd = 0;  // values not on the grid
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float t = mul_pow2(v[j], shift);
    const float r = rintf(t);
    m[j] = (r == t) ? __float2int_rn(r) : 0;
    odd |= (r == t) ? 0u : (1u << j);
  }
  const int b = o >> 5, i = o & 31;
#pragma unroll
  for (int l = 0; l < NLB; ++l) {
    const int k = NLB - 1 - l;  // plane 0 = the most significant byte (signed)
    const uint2 wv = make_uint2(pack_byte(m[0], m[1], m[2], m[3], k), pack_byte(m[4], m[5], m[6], m[7], k));
    *reinterpret_cast<uint2*>(xi.limb + l * xi.plane + b * XWB + wpad_i(2 * i)) = wv;
  }
  int isum = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) isum += m[j];
  const int s16 = isum + __shfl_xor_sync(0xFFFFFFFFu, isum, 1);
  const int s32 = s16 + __shfl_xor_sync(0xFFFFFFFFu, s16, 2);
  if ((i & 3) == 0) {  // 32-run j = i / 4
    const int j = i >> 2;
    xi.limb[b * XWB + side_w(1 + (j >> 2), j & 3)] = static_cast<uint32_t>(s32);
  }
  if ((i & 1) == 0) {  // 16-run r = i / 2, in Q6_K lane order
    const int r = i >> 1, h = r >> 3, rr = r & 7;
    xi.limb[xi.plane + b * XWB + side_w(2 * h + (rr & 1), rr >> 1)] = static_cast<uint32_t>(s16);
  }
  if (i < 2) xi.limb[b * XWB + side_w(0, i)] = __float_as_uint(pow2f(-shift));  // the block's scale (twice)
  if (__any_sync(0xFFFFFFFFu, odd != 0)) put_odd(v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7], odd, b, i, xi, lane);
  else if (i == 0) xi.limb[b * XWB + side_w(0, 2)] = 0u;  // no entries
}

// All NTHR threads: the image of x[0..K) (zero past K up to nb*256); with
// fp32 x two images, hi and lo.  Thread t takes octs t, t+NTHR, ...; the 32
// octs of a warp are one block.  All global loads of a pass (up to 6 octs a
// thread) are issued before any is used.
// Blocks [b0, b1) of the image (b0 = 0, b1 = nb: all of x).
template <int NTHR>
__device__ void stage_x(const void* xp, int x_bf16, int K, int nb, const XImg& xh, const XImg& xl, int tid, int b0 = 0,
                        int b1 = -1) {
  constexpr int MAXO = 6;
  const int noct = (b1 < 0 ? nb : b1) * 32;
  const int lane = tid & 31;
  for (int base = b0 * 32; base < noct; base += MAXO * NTHR) {
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
      if (x_bf16) {
        put_oct(v[it], o, xh, lane);
      } else {
        float hi[8], lo[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          hi[j] = __bfloat162float(__float2bfloat16_rn(v[it][j]));
          lo[j] = isfinite(hi[j]) ? __bfloat162float(__float2bfloat16_rn(v[it][j] - hi[j])) : 0.0f;
        }
        put_oct(hi, o, xh, lane);
        put_oct(lo, o, xl, lane);
      }
    }
  }
}

// ------------------------------------------------------- lane block cores
// A chunk is 64 weights of a block: Q4_K/Q5_K/IA4 chunk c = sub-blocks 2c,
// 2c+1 (code bytes 32c..32c+31: low nibbles, then high nibbles); Q6_K chunk
// c = the four 16-runs 8(c>>1) + (c&1) + 2p of 128-half c>>1.  Two layouts
// use the same pieces: a quad's lane c takes chunk c of one block (routed
// experts), or a lane takes all four chunks of its own block and combines
// once per block (one-token products).
//
// Per-lane constants of the Q4_K/Q5_K scale unpacking for chunk c
// (sub-blocks j = 2c, 2c+1 of the 12-byte scale field s[0..11]):
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

// x slice of one chunk: 3 limb planes x 16 words, in the chunk's part order
// (Q4_K/Q5_K: parts 0,1 = words 0..7, 8..15; Q6_K: part p = words 4p..4p+3).
struct XSlice {
  uint32_t w[NLB][16];
};
template <int QT>
__device__ __forceinline__ void load_slice(uint32_t xl, uint32_t plane, XSlice& X) {
#pragma unroll
  for (int l = 0; l < NLB; ++l)
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      // word offsets (relative, padded layout) of the chunk's 4-word groups
      const int off = (QT == T_Q6_K) ? ((p == 0) ? 0 : (p == 1) ? 8 : (p == 2) ? 20 : 28) : 4 * p;
      const uint4 u = lds128(xl + l * plane + 4 * off);
      X.w[l][4 * p] = u.x; X.w[l][4 * p + 1] = u.y; X.w[l][4 * p + 2] = u.z; X.w[l][4 * p + 3] = u.w;
    }
}
// word offset of chunk c's slice within a block
template <int QT>
__device__ __forceinline__ int slice_off(int c) {
  return (QT == T_Q6_K) ? (40 * (c >> 1) + 4 * (c & 1)) : 20 * c;
}

// Exact integer sums of (part of) a Q4_K/Q5_K/IA4 block:
//   Y = Y0 2^16 + Y1 2^8 + Y2 = sum_j sc_j T_j  (T_j = sum q m over sub-block j),
//   Mi = sum_j m_j X_j                          (X_j = sum m over sub-block j).
// Per block |Y0| < 2^27, |Y1|, |Y2| < 2^28, |Mi| < 2^36.
struct Acc45 {
  int Y0, Y1, Y2;
  long long Mi;
};
// Exact integer sums of (part of) a Q6_K block: Y = sum_p sc_p T_p (limbs as
// above, each < 2^29) and Z = sum_p sc_p X_p over its 16-runs.
struct Acc6 {
  int Y0, Y1, Y2;
  long long Z;
};

// d Y - dmin Mi without the block scale, for d and dmin fp16- or bf16-valued
// (so their fp32 mantissas end in 13 zero bits).
//  * When the binary exponents of d and dmin differ by -12..7 the two terms
//    can cancel (w = d sc q - dmin m near 0): d = a 2^A, dmin = b 2^B with
//    11-bit integers a, b, and the difference is formed exactly in 64-bit
//    integers over the unit 2^min(A,B) (|alpha Y|, |beta Mi| < 2^60) and
//    rounded once.
//  * Otherwise one term is below 1/126 of the other for every weight (d >= 2^7
//    dmin, or dmin m >= 2^12 d > 2 d sc q), so |w| bounds both terms to within
//    a factor of two and three fp32 roundings stay within 5u of sum|w m|.
// (exponents far apart, zero, subnormal or non-finite: out of line, rare)
static __device__ __noinline__ float combine45_far(float d, float dmin, int Y0, int Y1, int Y2, long long Mi) {
  const long long Y = (static_cast<long long>(Y0) << 16) + (static_cast<long long>(Y1) << 8) + Y2;
  return __fmaf_rn(d, ll2f_rn(Y), -dmin * ll2f_rn(Mi));
}
__device__ __forceinline__ float combine45(float d, float dmin, const Acc45& A) {
  const uint32_t ud = __float_as_uint(d), um = __float_as_uint(dmin);
  const int ed = static_cast<int>((ud >> 23) & 0xFFu), em = static_cast<int>((um >> 23) & 0xFFu);
  const int de = ed - em;
  if (ed != 0 && em != 0 && ed != 255 && em != 255 && de >= -12 && de <= 7) {
    int a = static_cast<int>(((ud & 0x7FFFFFu) | 0x800000u) >> 13);
    int b = static_cast<int>(((um & 0x7FFFFFu) | 0x800000u) >> 13);
    if (ud >> 31) a = -a;
    if (um >> 31) b = -b;
    const int alpha = de > 0 ? a * (1 << de) : a;   // |alpha| < 2^18
    const int beta = de < 0 ? b * (1 << -de) : b;   // |beta| < 2^23
    long long P = static_cast<long long>(alpha) * A.Y0;
    P = P * 256 + static_cast<long long>(alpha) * A.Y1;
    P = P * 256 + static_cast<long long>(alpha) * A.Y2;
    P -= static_cast<long long>(beta) * A.Mi;
    return mul_pow2(ll2f_rn(P), min(ed, em) - 137);  // unit 2^(min exponent - 127 - 10)
  }
  return combine45_far(d, dmin, A.Y0, A.Y1, A.Y2, A.Mi);
}

// Q4_K / Q5_K / IA4: adds chunk c of the block at bp (16-byte aligned) to A;
// si = the chunk's two 32-run sums of m; sc0, sc1, m0, m1 its sub-blocks'
// scales and mins (1 for IA4).
template <int QT>
__device__ __forceinline__ void chunk45(uint32_t bp, const XSlice& X, int2 si, int c, int sc0, int sc1, int m0,
                                        int m1, Acc45& A) {
  constexpr int QS = kQ4Codes<QT> ? 16 : 48;
  const uint4 q0 = lds128(bp + QS + 32 * c);
  const uint4 q1 = lds128(bp + QS + 32 * c + 16);
  uint4 h0 = make_uint4(0, 0, 0, 0), h1 = make_uint4(0, 0, 0, 0);
  if constexpr (QT == T_Q5_K) { h0 = lds128(bp + 16); h1 = lds128(bp + 32); }
  int I[2][NLB];
#pragma unroll
  for (int p = 0; p < 2; ++p)
#pragma unroll
    for (int l = 0; l < NLB; ++l) I[p][l] = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint32_t q = (w < 4) ? w4(q0, w) : w4(q1, w - 4);
    uint32_t lo, hi;
    if constexpr (kQ4Codes<QT>) {
      lo = q & 0x0F0F0F0Fu;
      hi = q & 0xF0F0F0F0u;  // 16 x the high nibble: the factor leaves the sums exactly
    } else {
      const uint32_t hb = (w < 4) ? w4(h0, w) : w4(h1, w - 4);
      lo = (q & 0x0F0F0F0Fu) | (__funnelshift_l(hb, hb, (4 - 2 * c) & 31) & 0x10101010u);
      hi = ((q >> 4) & 0x0F0F0F0Fu) | (__funnelshift_l(hb, hb, (3 - 2 * c) & 31) & 0x10101010u);
    }
    I[0][0] = dp_us(lo, X.w[0][w], I[0][0]);
    I[1][0] = dp_us(hi, X.w[0][8 + w], I[1][0]);
#pragma unroll
    for (int l = 1; l < NLB; ++l) {
      I[0][l] = dp_uu(lo, X.w[l][w], I[0][l]);
      I[1][l] = dp_uu(hi, X.w[l][8 + w], I[1][l]);
    }
  }
  if constexpr (kQ4Codes<QT>) {
#pragma unroll
    for (int l = 0; l < NLB; ++l) I[1][l] >>= 4;  // exact: every term is a multiple of 16
  }
  A.Y0 += sc0 * I[0][0] + sc1 * I[1][0];
  A.Y1 += sc0 * I[0][1] + sc1 * I[1][1];
  A.Y2 += sc0 * I[0][2] + sc1 * I[1][2];
  A.Mi += static_cast<long long>(m0) * si.x + static_cast<long long>(m1) * si.y;
}
// Scales and mins of chunk c's sub-blocks (2c, 2c+1) from the block header
// (quad layout: the per-lane constants of scale_lane).
__device__ __forceinline__ void chunk_scales(const uint4& hdr, const ScaleLane& sl, int& sc0, int& sc1, int& m0,
                                             int& m1) {
  const uint32_t P = __byte_perm(sl.lowsrc ? hdr.y : hdr.w, hdr.z, sl.selP);
  const uint32_t Q = __byte_perm(hdr.y, hdr.z, sl.selQ);
  const uint32_t L = (P & sl.mA) | ((P >> 4) & sl.mB) | ((Q >> 2) & sl.mH);
  sc0 = static_cast<int>(L & 0xFF);
  sc1 = static_cast<int>((L >> 8) & 0xFF);
  m0 = static_cast<int>((L >> 16) & 0xFF);
  m1 = static_cast<int>(L >> 24);
}
// Scale bytes (sc of sub-blocks 4h..4h+3) and min bytes of half h of a block.
__device__ __forceinline__ void half_scales(const uint4& hdr, int h, uint32_t& scb, uint32_t& mb) {
  scb = h ? ((hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u)) : (hdr.y & 0x3F3F3F3Fu);
  mb = h ? (((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u)) : (hdr.z & 0x3F3F3F3Fu);
}

// d Y - dmin Mi in fp32 when that is provably within (3 lim + 1) u of the
// result (u = 2^-24), else exactly (combine45).  The fp32 form's error is at
// most 3u bnd + u |v| (the int-to-float conversions and the two-step limb sum
// take at most 3u of bnd = |d| (|Y0| 2^16 + |Y1| 2^8 + |Y2|) + |dmin Mi|); it
// is kept when bnd <= lim |v|:
//   kLimBf16 = 2^11 (bf16 x, and the lo image of fp32 x): < 2^-11 |v|;
//   kLimHi = 2^8 (the hi image of fp32 x): < 769 u |v| < 4.6e-5 |v|.
// |v| is at most the sum of |w m| over the weights summed, so these are
// bounds relative to sum |w x|.
constexpr float kLimBf16 = 2048.0f;
constexpr float kLimHi = 256.0f;
__device__ __forceinline__ float combine45_checked(float d, float dmin, const Acc45& A, float lim) {
  const float y0 = __int2float_rn(A.Y0), y1 = __int2float_rn(A.Y1), y2 = __int2float_rn(A.Y2);
  const float yf = __fmaf_rn(y0, 65536.0f, __fmaf_rn(y1, 256.0f, y2));
  const float yb = __fmaf_rn(fabsf(y0), 65536.0f, __fmaf_rn(fabsf(y1), 256.0f, fabsf(y2)));
  const float mt = dmin * ll2f_rn(A.Mi);
  const float v = __fmaf_rn(d, yf, -mt);
  if (__fmaf_rn(fabsf(d), yb, fabsf(mt)) <= lim * fabsf(v)) return v;
  return combine45(d, dmin, A);
}
// acc + s (d Y - dmin Mi): one block's (Q4_K/Q5_K) or one group's (IA4, group
// c) sums, in fp32 within the bound lim gives (combine45_checked).
template <int QT>
__device__ __forceinline__ float finish45(uint32_t bp, const Acc45& A, float s, int c, float lim, float acc) {
  const uint4 hdr = lds128(bp);
  float d, dmin;
  if constexpr (QT == T_IA4) {
    d = ia4_scale(hdr, c);
    dmin = ia4_neg_bias(hdr, c);
  } else {
    d = half_bits_to_float(hdr.x & 0xFFFF);
    dmin = half_bits_to_float(hdr.x >> 16);
  }
  return __fmaf_rn(s, combine45_checked(d, dmin, A, lim), acc);
}

// Q6_K: adds chunk c of the block at bp (2-byte aligned) to A; si = the
// chunk's four 16-run sums.
__device__ __forceinline__ void chunk6(uint32_t bp, const XSlice& X, int4 si, int c, Acc6& A) {
  const int h = c >> 1, e = c & 1;
  const uint4 qa = lds16_a2(bp + 64 * h + 16 * e);
  const uint4 qb = lds16_a2(bp + 64 * h + 32 + 16 * e);
  const uint4 qh = lds16_a2(bp + 128 + 32 * h + 16 * e);
  const uint2 sv = lds8_a2(bp + 192 + 8 * h);
  const uint32_t se = __byte_perm(sv.x, sv.y, e ? 0x7531 : 0x6420);  // scales 8h + 2p + e, p = 0..3
  int I[4][NLB];
#pragma unroll
  for (int p = 0; p < 4; ++p)
#pragma unroll
    for (int l = 0; l < NLB; ++l) I[p][l] = 0;
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
      for (int l = 1; l < NLB; ++l) I[p][l] = dp_uu(cd[p], X.w[l][4 * p + w], I[p][l]);
    }
  }
  const int sc0 = sbyte(se, 0), sc1 = sbyte(se, 1), sc2 = sbyte(se, 2), sc3 = sbyte(se, 3);
  A.Y0 += sc0 * I[0][0] + sc1 * I[1][0] + sc2 * I[2][0] + sc3 * I[3][0];
  A.Y1 += sc0 * I[0][1] + sc1 * I[1][1] + sc2 * I[2][1] + sc3 * I[3][1];
  A.Y2 += sc0 * I[0][2] + sc1 * I[1][2] + sc2 * I[2][2] + sc3 * I[3][2];
  A.Z += static_cast<long long>(sc0) * si.x + static_cast<long long>(sc1) * si.y +
         static_cast<long long>(sc2) * si.z + static_cast<long long>(sc3) * si.w;
}
// acc + s d Y, Y = sum_p sc_p (T_p - 32 X_p) an exact integer with |Y| <= sum
// |w_k / d| |m_k|: one rounding to fp32, one in the fma.
__device__ __forceinline__ float finish6(uint32_t bp, const Acc6& A, float s, float acc) {
  const float d = half_bits_to_float(lds16(bp + 208));
  const long long Y = (static_cast<long long>(A.Y0) << 16) + (static_cast<long long>(A.Y1) << 8) + A.Y2 - 32 * A.Z;
  return __fmaf_rn(s * d, ll2f_rn(Y), acc);
}

// One chunk c of the block at bp, combined on its own (quad layout).
template <int QT>
__device__ __forceinline__ float core_q45(uint32_t bp, const XSlice& X, int2 si, float s, int c, const ScaleLane& sl,
                                          float lim, float acc) {
  Acc45 A = {0, 0, 0, 0};
  int sc0 = 1, sc1 = 1, m0 = 1, m1 = 1;
  if constexpr (QT != T_IA4) chunk_scales(lds128(bp), sl, sc0, sc1, m0, m1);  // IA4: one group, sc = m = 1
  chunk45<QT>(bp, X, si, c, sc0, sc1, m0, m1, A);
  return finish45<QT>(bp, A, s, c, lim, acc);
}
__device__ __forceinline__ float core_q6(uint32_t bp, const XSlice& X, int4 si, float s, int c, float acc) {
  Acc6 A = {0, 0, 0, 0};
  chunk6(bp, X, si, c, A);
  return finish6(bp, A, s, acc);
}

// Weight k of the block at bp as the exactly rounded fp32 value (the
// definition's d*sc*q - dmin*m, d*sc*(q-32) or scale*q + bias, one rounding);
// hdr = the block's first 16 bytes (Q4_K, Q5_K, IA4; Q6_K reads its own d).
template <int QT>
__device__ __forceinline__ float w_at_h(uint32_t bp, int k, const uint4& hdr) {
  if constexpr (QT == T_Q6_K) {
    const int h = k >> 7, r = k & 127, t = r >> 5, l = r & 31;
    const uint32_t qlb = lds8(bp + 64 * h + 32 * (t & 1) + l);
    const uint32_t qhb = lds8(bp + 128 + 32 * h + l);
    const int q = static_cast<int>(((qlb >> (4 * (t >> 1))) & 15u) | (((qhb >> (2 * t)) & 3u) << 4));
    const int sc = static_cast<int>(static_cast<int8_t>(lds8(bp + 192 + (k >> 4))));
    const float d = half_bits_to_float(lds16(bp + 208));
    return d * static_cast<float>(sc * (q - 32));  // the integer product is exact
  } else {
    constexpr int QS = kQ4Codes<QT> ? 16 : 48;
    const uint32_t cb = lds8(bp + QS + 32 * (k >> 6) + (k & 31));
    int q = static_cast<int>((cb >> (4 * ((k >> 5) & 1))) & 15u);
    if constexpr (QT == T_Q5_K) q |= static_cast<int>((lds8(bp + 16 + (k & 31)) >> (k >> 5)) & 1u) << 4;
    if constexpr (QT == T_IA4) {
      const int g = k >> 6;
      return __fmaf_rn(ia4_scale(hdr, g), static_cast<float>(q), -ia4_neg_bias(hdr, g));
    } else {
      const uint32_t bs = scale_min_bytes(hdr.y, hdr.z, hdr.w, k >> 6);  // [sc_2g, sc_2g+1, m_2g, m_2g+1]
      const int hb = (k >> 5) & 1;
      const int sc = static_cast<int>((bs >> (8 * hb)) & 0xFFu), m = static_cast<int>((bs >> (16 + 8 * hb)) & 0xFFu);
      const float d = half_bits_to_float(hdr.x & 0xFFFF), dmin = half_bits_to_float(hdr.x >> 16);
      return __fmaf_rn(d * static_cast<float>(sc), static_cast<float>(q), -(dmin * static_cast<float>(m)));
    }
  }
}

// The listed values of block b (cnt <= ECAP) for the R rows whose blocks are
// at rp: this lane takes entries first, first + step, ... (at most 16); each
// entry's word is read once for all the rows, each row's header once for all
// entries.  acc[i] += the sum of fl(w_k x_k) over them, w_k the exactly
// rounded weight, summed on its own first (at most 17 fp32 additions from a
// product to acc).
// R row addresses / R row sums passed by value (the rare paths below are out
// of line, so that the integer core keeps its registers).
template <int R>
struct RowAddr {
  uint32_t v[R];
};
template <int R>
struct RowSum {
  float v[R];
};
template <int QT, int R>
__device__ __noinline__ RowSum<R> entries_rows_ol(const XImg xi, int b, int cnt, int first, int step,
                                                  const RowAddr<R> rp_, RowSum<R> acc_) {
  const uint32_t (&rp)[R] = rp_.v;
  float (&acc)[R] = acc_.v;
  uint4 hd[R];
  float t[R];
#pragma unroll
  for (int i = 0; i < R; ++i) {
    hd[i] = QT == T_Q6_K ? make_uint4(0, 0, 0, 0) : lds128(rp[i]);
    t[i] = 0.0f;
  }
#pragma unroll 1
  for (int j = first; j < cnt; j += step) {
    const uint32_t e = lds32(xi.limb_s + 4 * ent_word(xi, b, j));
    const int k = static_cast<int>(e & 0xFFu);
    const float xv = __uint_as_float(e & 0xFFFF0000u);
#pragma unroll
    for (int i = 0; i < R; ++i) t[i] = __fmaf_rn(w_at_h<QT>(rp[i], k, hd[i]), xv, t[i]);
  }
#pragma unroll
  for (int i = 0; i < R; ++i) acc[i] = __fadd_rn(acc[i], t[i]);
  return acc_;
}
template <int QT, int R>
__device__ __forceinline__ void entries_rows(const XImg& xi, int b, int cnt, int first, int step,
                                             const uint32_t (&rp)[R], float (&acc)[R]) {
  RowAddr<R> ra;
  RowSum<R> rs;
#pragma unroll
  for (int i = 0; i < R; ++i) { ra.v[i] = rp[i]; rs.v[i] = acc[i]; }
  rs = entries_rows_ol<QT, R>(xi, b, cnt, first, step, ra, rs);
#pragma unroll
  for (int i = 0; i < R; ++i) acc[i] = rs.v[i];
}

// A raw block (all 256 values kept as bf16): chunk cc of block b for the R
// rows at rp: acc[i] += the sum of fl(w_k x_k) over the chunk's 64 weights,
// w_k the exactly rounded fp32 weight of w_at_h, summed as four running sums
// of 16 products, added pairwise (at most 19 fp32 additions from a product
// to acc).  The chunk's x values are read once for all the rows; each code
// byte is decoded once per row.
__device__ __forceinline__ float nib_f(uint32_t w, int s) {  // (w >> s) & 15 as a float, exactly
  return __uint_as_float(0x4B000000u | ((w >> s) & 15u)) - 8388608.0f;
}
template <int QT, int R>
__device__ __noinline__ RowSum<R> raw_rows_ol(const XImg xi, int b, int cc, const RowAddr<R> rp_, RowSum<R> acc_) {
  const uint32_t (&rp)[R] = rp_.v;
  float (&acc)[R] = acc_.v;
  // x of the chunk's weights, in the order the codes come: Q4_K/Q5_K/IA4 lo
  // nibbles 64cc + i, hi nibbles 64cc + 32 + i (i < 32); Q6_K part p, value i:
  // weight 128 (cc >> 1) + 32 p + 16 (cc & 1) + i (i < 16)
  uint32_t xw[32];  // bf16 pairs (even value low)
#pragma unroll
  for (int q4 = 0; q4 < 16; ++q4) {
    const int k = (QT == T_Q6_K) ? 128 * (cc >> 1) + 32 * (q4 >> 2) + 16 * (cc & 1) + 4 * (q4 & 3)
                                 : 64 * cc + 32 * (q4 >> 3) + 4 * (q4 & 7);
    const uint2 v = lds64(xi.limb_s + 4 * raw_word(xi, b, k));
    xw[2 * q4] = v.x;
    xw[2 * q4 + 1] = v.y;
  }
  auto xv = [&](int idx) {  // x of the idx-th weight of the chunk (in code order)
    const uint32_t w = xw[idx >> 1];
    return __uint_as_float((idx & 1) ? (w & 0xFFFF0000u) : (w << 16));
  };
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const uint32_t bp = rp[i];
    float a[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if constexpr (QT == T_Q6_K) {
      const int h = cc >> 1, e = cc & 1;
      const uint4 qa = lds16_a2(bp + 64 * h + 16 * e);
      const uint4 qb = lds16_a2(bp + 64 * h + 32 + 16 * e);
      const uint4 qh = lds16_a2(bp + 128 + 32 * h + 16 * e);
      const uint2 sv = lds8_a2(bp + 192 + 8 * h);
      const uint32_t se = __byte_perm(sv.x, sv.y, e ? 0x7531 : 0x6420);  // scales 8h + 2p + e
      const float d = half_bits_to_float(lds16(bp + 208));
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int sc = sbyte(se, p);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t av = w4(qa, w), bv = w4(qb, w), hv = w4(qh, w);
          const uint32_t cd = p == 0 ? ((av & 0x0F0F0F0Fu) | ((hv << 4) & 0x30303030u))
                            : p == 1 ? ((bv & 0x0F0F0F0Fu) | ((hv << 2) & 0x30303030u))
                            : p == 2 ? (((av >> 4) & 0x0F0F0F0Fu) | (hv & 0x30303030u))
                                     : (((bv >> 4) & 0x0F0F0F0Fu) | ((hv >> 2) & 0x30303030u));
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int q = static_cast<int>((cd >> (8 * j)) & 0xFFu);
            a[j] = __fmaf_rn(d * static_cast<float>(sc * (q - 32)), xv(16 * p + 4 * w + j), a[j]);
          }
        }
      }
    } else {
      constexpr int QS = kQ4Codes<QT> ? 16 : 48;
      const uint4 q0 = lds128(bp + QS + 32 * cc), q1 = lds128(bp + QS + 32 * cc + 16);
      uint4 h0 = make_uint4(0, 0, 0, 0), h1 = make_uint4(0, 0, 0, 0);
      if constexpr (QT == T_Q5_K) { h0 = lds128(bp + 16); h1 = lds128(bp + 32); }
      const uint4 hdr = lds128(bp);
      float A0, B0, A1, B1;  // lo nibbles: sub-block 2cc (IA4: group cc), hi: 2cc + 1
      if constexpr (QT == T_IA4) {
        A0 = A1 = ia4_scale(hdr, cc);
        B0 = B1 = ia4_neg_bias(hdr, cc);
      } else {
        const uint32_t bs = scale_min_bytes(hdr.y, hdr.z, hdr.w, cc);  // [sc_2g, sc_2g+1, m_2g, m_2g+1]
        const float d = half_bits_to_float(hdr.x & 0xFFFF), dmin = half_bits_to_float(hdr.x >> 16);
        A0 = d * static_cast<float>(bs & 0xFFu);
        A1 = d * static_cast<float>((bs >> 8) & 0xFFu);
        B0 = dmin * static_cast<float>((bs >> 16) & 0xFFu);
        B1 = dmin * static_cast<float>(bs >> 24);
      }
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const uint32_t q = (w < 4) ? w4(q0, w) : w4(q1, w - 4);
        uint32_t hb = 0;
        if constexpr (QT == T_Q5_K) hb = (w < 4) ? w4(h0, w) : w4(h1, w - 4);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float qlo = nib_f(q, 8 * j), qhi = nib_f(q, 8 * j + 4);
          if constexpr (QT == T_Q5_K) {
            qlo += static_cast<float>(((hb >> (8 * j + 2 * cc)) & 1u) << 4);
            qhi += static_cast<float>(((hb >> (8 * j + 2 * cc + 1)) & 1u) << 4);
          }
          a[j] = __fmaf_rn(__fmaf_rn(A0, qlo, -B0), xv(4 * w + j), a[j]);
          a[j] = __fmaf_rn(__fmaf_rn(A1, qhi, -B1), xv(32 + 4 * w + j), a[j]);
        }
      }
    }
    acc[i] = __fadd_rn(acc[i], __fadd_rn(__fadd_rn(a[0], a[1]), __fadd_rn(a[2], a[3])));
  }
  return acc_;
}
template <int QT, int R>
__device__ __forceinline__ void raw_rows(const XImg& xi, int b, int cc, const uint32_t (&rp)[R], float (&acc)[R]) {
  RowAddr<R> ra;
  RowSum<R> rs;
#pragma unroll
  for (int i = 0; i < R; ++i) { ra.v[i] = rp[i]; rs.v[i] = acc[i]; }
  rs = raw_rows_ol<QT, R>(xi, b, cc, ra, rs);
#pragma unroll
  for (int i = 0; i < R; ++i) acc[i] = rs.v[i];
}


// Quad layout: one image's contribution of block b to the rows at rp[0..R)
// (R rows per quad), lane c taking chunk c: the integer image, then the
// values it leaves out (every fourth one).
template <int QT, int R>
__device__ __forceinline__ void block_rows(const XImg& xi, int b, const uint32_t (&rp)[R], int c, const ScaleLane& sl,
                                           float lim, float (&acc)[R]) {
  const uint4 bh = lds128(hdr_s(xi, b));
  const float s = __uint_as_float(bh.x);
  const uint32_t cnt = bh.z;
  if (cnt <= static_cast<uint32_t>(ECAP)) {
    XSlice X;
    load_slice<QT>(xi.limb_s + 4 * (b * XWB + slice_off<QT>(c)), 4 * xi.plane, X);
    if constexpr (QT == T_Q6_K) {
      const uint4 sv = lds128(si16_s(xi, b, c));
      const int4 si = make_int4(static_cast<int>(sv.x), static_cast<int>(sv.y), static_cast<int>(sv.z),
                                static_cast<int>(sv.w));
#pragma unroll
      for (int i = 0; i < R; ++i) acc[i] = core_q6(rp[i], X, si, s, c, acc[i]);
    } else {
      const uint2 sv = lds64(si32_s(xi, b, c));
      const int2 si = make_int2(static_cast<int>(sv.x), static_cast<int>(sv.y));
#pragma unroll
      for (int i = 0; i < R; ++i) acc[i] = core_q45<QT>(rp[i], X, si, s, c, sl, lim, acc[i]);
    }
  }
  if (cnt > static_cast<uint32_t>(ECAP)) {
    raw_rows<QT, R>(xi, b, c, rp, acc);
  } else if (cnt != 0) {
    entries_rows<QT, R>(xi, b, static_cast<int>(cnt), c, 4, rp, acc);
  }
}

// Pair layout: one image's contribution of block b to the rows at rp[0..R),
// this lane taking chunks 2h, 2h+1 (half h of the block): the exact sums of
// the half, combined once per row (IA4: once per group), then every second
// value the image leaves out.
template <int QT, int R>
__device__ __forceinline__ void block_half(const XImg& xi, int b, int h, const uint32_t (&rp)[R], float lim,
                                           float (&acc)[R]) {
  const uint4 bh = lds128(hdr_s(xi, b));
  const float s = __uint_as_float(bh.x);
  const uint32_t cnt = bh.z;
  const uint32_t xl = xi.limb_s + 4 * b * XWB;
  if (cnt <= static_cast<uint32_t>(ECAP)) {
    if constexpr (QT == T_Q6_K) {
      Acc6 A[R];
#pragma unroll
      for (int i = 0; i < R; ++i) A[i] = Acc6{0, 0, 0, 0};
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int c = 2 * h + k;
        XSlice X;
        load_slice<QT>(xl + 4 * slice_off<QT>(c), 4 * xi.plane, X);
        const uint4 sv = lds128(si16_s(xi, b, c));
        const int4 si = make_int4(static_cast<int>(sv.x), static_cast<int>(sv.y), static_cast<int>(sv.z),
                                  static_cast<int>(sv.w));
#pragma unroll
        for (int i = 0; i < R; ++i) chunk6(rp[i], X, si, c, A[i]);
      }
#pragma unroll
      for (int i = 0; i < R; ++i) acc[i] = finish6(rp[i], A[i], s, acc[i]);
    } else {
      Acc45 A[R];
      uint32_t scb[R], mb[R];  // the half's scale and min bytes, per row
#pragma unroll
      for (int i = 0; i < R; ++i) {
        A[i] = Acc45{0, 0, 0, 0};
        if constexpr (QT != T_IA4) half_scales(lds128(rp[i]), h, scb[i], mb[i]);
      }
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int c = 2 * h + k;
        XSlice X;
        load_slice<QT>(xl + 4 * slice_off<QT>(c), 4 * xi.plane, X);
        const uint2 sv = lds64(si32_s(xi, b, c));
        const int2 si = make_int2(static_cast<int>(sv.x), static_cast<int>(sv.y));
#pragma unroll
        for (int i = 0; i < R; ++i) {
          if constexpr (QT == T_IA4) {  // each group has its own scale and bias (sc = m = 1)
            chunk45<QT>(rp[i], X, si, c, 1, 1, 1, 1, A[i]);
            acc[i] = finish45<QT>(rp[i], A[i], s, c, lim, acc[i]);
            A[i] = Acc45{0, 0, 0, 0};
          } else {
            const int sc0 = static_cast<int>((scb[i] >> (16 * k)) & 0xFFu);
            const int sc1 = static_cast<int>((scb[i] >> (16 * k + 8)) & 0xFFu);
            const int m0 = static_cast<int>((mb[i] >> (16 * k)) & 0xFFu);
            const int m1 = static_cast<int>((mb[i] >> (16 * k + 8)) & 0xFFu);
            chunk45<QT>(rp[i], X, si, c, sc0, sc1, m0, m1, A[i]);
          }
        }
      }
      if constexpr (QT != T_IA4) {
#pragma unroll
        for (int i = 0; i < R; ++i) acc[i] = finish45<QT>(rp[i], A[i], s, 0, lim, acc[i]);
      }
    }
  }
  if (cnt > static_cast<uint32_t>(ECAP)) {
    raw_rows<QT, R>(xi, b, 2 * h, rp, acc);
    raw_rows<QT, R>(xi, b, 2 * h + 1, rp, acc);
  } else if (cnt != 0) {
    entries_rows<QT, R>(xi, b, static_cast<int>(cnt), h, 2, rp, acc);
  }
}

}  // namespace lane
}  // namespace kq
