// kq_gemv.cu -- one-token products y = W x (M = 1) against Q4_K / Q5_K / Q6_K
// rows: a single matrix, or a program of matrices run by one persistent launch.
//
// "GGUF in transformers", section "Reusing ggml's Metal kernels": decode-time
// products read the packed super-blocks directly and dequantize on the fly;
// section "Keeping the CPU and GPU working together": the device should not
// idle between the operations of a decode step.
//
// Arithmetic (exact integer products, one rounding per lane and block):
//  * x is staged once per product into shared memory as block-floating-point
//    integers: for every run of 128 consecutive values a power-of-two scale
//    s = 2^(e - 14) (bf16 x) or 2^(e - 22) (fp32 x), e the binary exponent of
//    the run's largest |x|, and m_k = rint(x_k / s), |m_k| <= 2^14 (2^22),
//    split into byte limbs (hi signed, lower ones unsigned).  Every bf16 value
//    within 2^7 of its run maximum is represented exactly; otherwise the error
//    is at most s/2 <= 2^-15 * max|x| (2^-23 for fp32 x).  Exact integer sums
//    of m over every 16- and 32-run are staged beside the limbs.
//  * a lane owns 64 weights of a block (Q4_K/Q5_K: sub-blocks 2c, 2c+1;
//    Q6_K: four 16-runs of one 128-half); codes times limbs are summed
//    exactly by dp4a, and with bf16 x the lane's whole block contribution is
//    an exact int32:
//        Q4_K/Q5_K:  y += s * (d * sum_p sc_p*T_p  -  dmin * sum_p m_p*X_p)
//        Q6_K:       y += s * d * sum_p sc_p*(T_p - 32*X_p)
//    with T_p = sum q*m and X_p = sum m over part p (bounds: |sum| < 2^31 for
//    every 6-bit scale and, for Q6_K, every int8 scale taken in pairs).  With
//    fp32 x the per-limb integer sums are combined in fp32.
//
// Execution (GB300: 152 SMs, 227 KB shared memory per CTA):
//  * one CTA per SM: a producer warp and NC consumer warps;
//  * the producer walks the CTA's units -- (tile of TT rows, K-part) of every
//    op, in op order -- and keeps a CTA-wide ring of S shared-memory slots
//    full with 1-D TMA bulk copies: one copy per stage when a stage holds
//    whole rows, else one copy per row segment of KC blocks.  Weights never
//    depend on earlier ops, so the producer runs ahead across op boundaries;
//  * consumer warp w owns rows w*TT/8 .. of a tile; quad q of the warp takes
//    one of those rows and one block phase (block b0+ph, b0+ph+P, ...), so a
//    stage of TT rows x KC blocks keeps all 64 quads busy whenever KC is a
//    multiple of P = 64/TT; row sums reduce over fixed shuffle trees
//    (deterministic);
//  * a tile whose K is split across CTAs writes its partial row sums to the
//    workspace; the last CTA to finish the tile (arrival counter) adds them in
//    part order and writes y;
//  * an op flagged "wait for previous" starts with a grid barrier (all CTAs
//    resident: cooperative launch) before its x is read; single products
//    instead use programmatic dependent launch, streaming weights before
//    griddepcontrol.wait.
#include "kq_internal.h"

namespace kq {

namespace {

#ifndef KQ_NC
#define KQ_NC 7
#endif
constexpr int NC = KQ_NC;              // consumer warps (+1 producer: 8 warps, all registers usable)
constexpr int TT = 32;                 // rows per tile (4 per quad)
constexpr int NTHC = NC * 32;          // consumer threads
constexpr int NTH = NTHC + 32;         // + one producer warp
constexpr int RING_MAX = 8;                // ring slots at most
constexpr int CONSUMER_BAR = 1;        // named barrier of the consumer warps
constexpr int XWB = 80;                // padded limb words per 256-block
constexpr int MAX_NB = 64;             // K <= 16384
// Largest stage (32 row segments): 48 KB keeps a ring of at least 4 slots.
constexpr int64_t kSlotCap = 48 * 1024;

}  // namespace

// Device op descriptor (geometry computed on the host).
struct KqOp {
  const uint8_t* W;
  const void* x;
  float* y;
  float* part;       // split K: partial row sums [KS][ntiles*TT] (workspace), else null
  int64_t pad0;
  int64_t N;
  int64_t row_bytes;
  int32_t K, nb, type, x_bf16;
  int32_t KS, kpb;   // K-parts per tile, blocks per K-part
  int32_t KC;        // blocks per stage
  int32_t srb;       // row stride inside a stage
  int32_t ntiles, nunits, rot;
  int32_t flags;     // OP_WAIT: grid barrier first; OP_NEWX: stage x
};
enum : int32_t { OP_WAIT = 1, OP_NEWX = 2 };

struct ProgArgs {
  const KqOp* ops;   // program in global memory (PROG) ...
  KqOp op0;          // ... or the single op
  int n_ops;
  int S, slot;       // ring slots, slot bytes
  int nb_max, nl_max;
  int* barrier;      // grid barrier arrivals (programs with OP_WAIT), zero at launch
  int* err;
  int pf;            // L2 prefetch distance in stages
  int final_fix;     // split-K sums remain after the last op: final grid barrier
};

namespace {

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

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(CONSUMER_BAR), "n"(NTHC) : "memory");
}

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

// All consumer threads: quantize x[0..K) (zero past K up to nb*256) into xi.
// Thread t takes "octs" (8 consecutive values) t, t+T, ...; the 32 octs of a
// warp are one 256-block, 16 lanes one 128-run.  All global loads are issued
// before any is used.
template <int NL>
__device__ void stage_x(const void* xp, int x_bf16, int K, int nb, const XImg& xi, int tid) {
  constexpr int MAXO = 8;
  const int noct = nb * 32;
  const int lane = tid & 31;
  for (int base = 0; base < noct; base += MAXO * NTHC) {
    float v[MAXO][8];
#pragma unroll
    for (int it = 0; it < MAXO; ++it) {
      const int o = base + it * NTHC + tid;
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
      const int o = base + it * NTHC + tid;
      if (o - lane >= noct) continue;  // whole warp past the end (noct is a multiple of 32)
      float mx = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) mx = fmaxf(mx, fabsf(v[it][j]));
#pragma unroll
      for (int w = 1; w < 16; w <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, w));
      // mx = f * 2^e, f in [0.5, 1): from the bits for normal values, frexpf otherwise
      const uint32_t mb = __float_as_uint(mx);
      const int be = static_cast<int>((mb >> 23) & 0xFF);
      const bool fast = be >= 40 && be <= 200;
      int e = be - 126;
      if (!fast) frexpf(mx, &e);
      const int shift = (NL == 2 ? 14 : 22) - e;
      int m[8];
      if (fast) {
        const float p2 = __uint_as_float(static_cast<uint32_t>(127 + shift) << 23);
#pragma unroll
        for (int j = 0; j < 8; ++j) m[j] = __float2int_rn(v[it][j] * p2);  // exact: power-of-two scale
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) m[j] = (mx > 0.0f) ? __float2int_rn(ldexpf(v[it][j], shift)) : 0;
      }
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
        if ((o & 15) == 0)
          xi.scale[o >> 4] = (mx > 0.0f) ? (fast ? __uint_as_float(static_cast<uint32_t>(127 - shift) << 23)
                                                 : ldexpf(1.0f, -shift)) : 0.0f;
        if ((o & 3) == 0) xi.si32[o >> 2] = s32;
        if ((o & 1) == 0) {
          const int r = (o >> 1) & 15;  // 16-run within the block
          const int h = r >> 3, rr = r & 7;
          xi.si16q[b * 16 + 4 * (2 * h + (rr & 1)) + (rr >> 1)] = s16;
        }
      }
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
  constexpr int QS = (QT == T_Q4_K) ? 16 : 48;
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
    if constexpr (QT == T_Q4_K) {
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
  const uint32_t P = __byte_perm(sl.lowsrc ? hdr.y : hdr.w, hdr.z, sl.selP);
  const uint32_t Q = __byte_perm(hdr.y, hdr.z, sl.selQ);
  const uint32_t L = (P & sl.mA) | ((P >> 4) & sl.mB) | ((Q >> 2) & sl.mH);
  const int sc0 = static_cast<int>(L & 0xFF), sc1 = static_cast<int>((L >> 8) & 0xFF);
  const int m0 = static_cast<int>((L >> 16) & 0xFF), m1 = static_cast<int>(L >> 24);
  const float d = half_bits_to_float(hdr.x & 0xFFFF);
  const float dmin = half_bits_to_float(hdr.x >> 16);
  if constexpr (NL == 2) {
    const int T0 = I[0][0] * 256 + I[0][1];
    int T1 = I[1][0] * 256 + I[1][1];
    if constexpr (QT == T_Q4_K) T1 >>= 4;  // exact: every term is a multiple of 16
    const int Y = sc0 * T0 + sc1 * T1;
    const int Mi = m0 * si.x + m1 * si.y;
    return __fmaf_rn(s, __fmaf_rn(d, static_cast<float>(Y), -dmin * static_cast<float>(Mi)), acc);
  } else {
    int Yl[NL];
#pragma unroll
    for (int l = 0; l < NL; ++l) {
      int t1 = I[1][l];
      if constexpr (QT == T_Q4_K) t1 >>= 4;
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

// ------------------------------------------------------------ work walk
// Unit k of this CTA in op o: u = ((cta - rot) mod G) + k*G; tile u / KS,
// K-part u % KS; the part's blocks are split into stages of KC blocks.
__device__ __forceinline__ int first_unit(const KqOp& o, int cta, int G) {
  int u = cta - (o.rot % G);
  return u < 0 ? u + G : u;
}

// Producer: lane i copies row i's segment (blocks [b0, b0+n)) of the tile
// into slot + i*srb, as its 16-byte aligned superset; arrive on full.
__device__ __forceinline__ void produce(const KqOp& o, int tile, int b0, int n, uint8_t* slot, uint64_t* full,
                                       int lane, int BB) {
  const int64_t r0 = static_cast<int64_t>(tile) * TT;
  uint32_t len = 0;
  const uint8_t* src = nullptr;
  if (r0 + lane < o.N) {
    const uintptr_t s0 =
        reinterpret_cast<uintptr_t>(o.W + (r0 + lane) * o.row_bytes + static_cast<int64_t>(b0) * BB);
    const uintptr_t e0 = s0 + static_cast<uintptr_t>(n) * BB;
    const uintptr_t as = s0 & ~uintptr_t(15), ae = (e0 + 15) & ~uintptr_t(15);
    src = reinterpret_cast<const uint8_t*>(as);
    len = static_cast<uint32_t>(ae - as);
  }
  const uint32_t total = __reduce_add_sync(0xFFFFFFFFu, len);
  if (lane == 0) mbar_arrive_expect_tx(full, total);
  __syncwarp();
  if (len) bulk_g2s(slot + lane * o.srb, src, len, full);
}

// Bounded wait until the grid-wide arrival counter reaches target.
__device__ __forceinline__ bool grid_wait(const int* counter, int target, int* err) {
  for (uint32_t i = 0; i < (1u << 26); ++i) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
    if (v >= target) return true;
    __nanosleep(64);
  }
  record_error(err, DEV_ERR_MBAR_TIMEOUT);
  return false;
}

struct Ring {
  uint64_t* full;
  uint64_t* empty;
  uint8_t* base;
  uint32_t base_s;  // shared-window address of base
  int S, slot;
};
// Per-unit cross-warp reduction: RS buffers of NC x TT partial row sums and
// an arrival count each; the last warp of a unit adds the warps' partials.
struct Red {
  float* buf;  // [RS][NC][TT]
  int* cnt;    // [RS]
  int RS;
};
// Running position of the consumers (identical in every consumer warp).
struct Walk {
  int64_t q;     // stages consumed
  int64_t us;    // units finished
  int cb;        // blocks seen, mod NC: chunk-to-warp rotation
  bool failed;
};

// Consumers: every unit of op o for this CTA.  Quad q of every warp owns the
// tile rows q, q+8, q+16, q+24; the stage's blocks are dealt to the warps
// round-robin (continuing across stages), so a warp applies one x slice to
// the 4 rows of each of its 8 quads.
template <int QT, int NL>
__device__ void consume_op(const KqOp& o, const XImg& xi, const Ring& rg, const Red& rd, Walk& wk, int* err,
                           int cta, int G) {
  constexpr int BB = Fmt<QT>::BYTES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = lane >> 2, c = lane & 3;
  const ScaleLane sl = scale_lane(c);
  const int xoff = (QT == T_Q6_K) ? (40 * (c >> 1) + 4 * (c & 1)) : 20 * c;
  for (int u = first_unit(o, cta, G); u < o.nunits; u += G) {
    const int tile = u / o.KS, kp = u - tile * o.KS;
    const int kb0 = kp * o.kpb;
    const int kb1 = min(o.nb, kb0 + o.kpb);
    const int64_t row0 = static_cast<int64_t>(tile) * TT;
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int b0 = kb0; b0 < kb1; b0 += o.KC) {
      const int n = min(o.KC, kb1 - b0);
      const int slot = static_cast<int>(wk.q % rg.S);
      if (!wk.failed) {
        const bool ok = mbar_wait(&rg.full[slot], static_cast<uint32_t>((wk.q / rg.S) & 1), err);
        wk.failed = !__all_sync(0xFFFFFFFFu, ok);
      }
      int bi = warp - wk.cb;
      if (bi < 0) bi += NC;
      if (!wk.failed && bi < n) {
        // the lane's rows q, q+8, q+16, q+24 (rows past N are computed on
        // stale shared memory and never written)
        const uint32_t sp = rg.base_s + static_cast<uint32_t>(slot) * rg.slot;
        const uint32_t seg0 = static_cast<uint32_t>(row0 * o.row_bytes) + static_cast<uint32_t>(b0 * BB);
        uint32_t rp[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = quad + 8 * i;
          // W is 16-byte aligned: the segment's offset in its 16-byte granule
          const uint32_t off = (seg0 + static_cast<uint32_t>(r) * static_cast<uint32_t>(o.row_bytes)) & 15u;
          rp[i] = sp + r * o.srb + off + bi * BB;
        }
        for (; bi < n; bi += NC) {
          const int b = b0 + bi;
          XSlice<NL> X;
          load_slice<QT, NL>(xi.limb_s + 4 * (b * XWB + xoff), 4 * xi.plane, X);
          const float s = __uint_as_float(lds32(xi.scale_s + 4 * (2 * b + (c >> 1))));
          if constexpr (QT == T_Q6_K) {
            const uint4 sv = lds128(xi.si16q_s + 4 * (16 * b + 4 * c));
            const int4 si = make_int4(static_cast<int>(sv.x), static_cast<int>(sv.y), static_cast<int>(sv.z),
                                      static_cast<int>(sv.w));
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = core_q6<NL>(rp[i], X, si, s, c, acc[i]);
          } else {
            const uint2 sv = lds64(xi.si32_s + 4 * (8 * b + 2 * c));
            const int2 si = make_int2(static_cast<int>(sv.x), static_cast<int>(sv.y));
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = core_q45<QT, NL>(rp[i], X, si, s, c, sl, acc[i]);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) rp[i] += NC * BB;
        }
      }
      wk.cb = (wk.cb + n) % NC;
      __syncwarp();
      if (lane == 0) mbar_arrive(&rg.empty[slot]);
      ++wk.q;
    }
    // this warp's partial row sums: over the quad's lanes, then to shared memory
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[i] = __fadd_rn(acc[i], __shfl_xor_sync(0xFFFFFFFFu, acc[i], 1));
      acc[i] = __fadd_rn(acc[i], __shfl_xor_sync(0xFFFFFFFFu, acc[i], 2));
    }
    const int rs = static_cast<int>(wk.us % rd.RS);
    ++wk.us;
    float* rb = rd.buf + static_cast<size_t>(rs) * NC * TT;
    if (c == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) rb[warp * TT + quad + 8 * i] = acc[i];
    }
    __syncwarp();
    int last = 0;
    if (lane == 0) {
      __threadfence_block();
      last = (atomicAdd(&rd.cnt[rs], 1) == NC - 1) ? 1 : 0;
    }
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (!last) continue;
    // last warp of the unit: add the warps' partials in warp order
    __threadfence_block();
    float v = rb[lane];
#pragma unroll
    for (int w = 1; w < NC; ++w) v = __fadd_rn(v, rb[w * TT + lane]);
    __syncwarp();
    if (lane == 0) rd.cnt[rs] = 0;
    const int64_t row = row0 + lane;
    if (row < o.N && !wk.failed) {
      if (o.KS == 1) o.y[row] = v;
      else o.part[static_cast<int64_t>(kp) * o.ntiles * TT + row] = v;  // added at the next grid barrier
    }
  }
}

// Split-K epilogue of op o, after a grid barrier: this CTA's slice of rows,
// y = sum of the K-parts' partial sums in part order.
__device__ __forceinline__ void fixup_op(const KqOp& o, int cta, int G, int ctid) {
  const int64_t stride = static_cast<int64_t>(o.ntiles) * TT;
  for (int64_t r = static_cast<int64_t>(cta) * NTHC + ctid; r < o.N; r += static_cast<int64_t>(G) * NTHC) {
    float v = __ldcg(o.part + r);
    for (int k = 1; k < o.KS; ++k) v = __fadd_rn(v, __ldcg(o.part + k * stride + r));
    o.y[r] = v;
  }
}

template <int NL>
__device__ __forceinline__ void consume_any(const KqOp& o, const XImg& xi, const Ring& rg, const Red& rd, Walk& wk,
                                            int* err, int cta, int G) {
  if (o.type == T_Q4_K) consume_op<T_Q4_K, NL>(o, xi, rg, rd, wk, err, cta, G);
  else if (o.type == T_Q5_K) consume_op<T_Q5_K, NL>(o, xi, rg, rd, wk, err, cta, G);
  else consume_op<T_Q6_K, NL>(o, xi, rg, rd, wk, err, cta, G);
}

template <bool PROG>
__device__ __forceinline__ KqOp load_op(const ProgArgs& a, int i) {
  if constexpr (PROG) return a.ops[i];
  else return a.op0;
}

// Producer cursor over this CTA's stages: (op, unit, first block).
struct StageCursor {
  KqOp o;
  int oi, u, tile, kb1, b0;
  bool valid;
};
__device__ __forceinline__ void cur_unit(StageCursor& c) {
  c.tile = c.u / c.o.KS;
  const int kp = c.u - c.tile * c.o.KS;
  c.b0 = kp * c.o.kpb;
  c.kb1 = min(c.o.nb, c.b0 + c.o.kpb);
}
template <bool PROG>
__device__ __forceinline__ void cur_seek(const ProgArgs& a, StageCursor& c, int cta, int G) {
  for (; c.oi < a.n_ops; ++c.oi) {
    c.o = load_op<PROG>(a, c.oi);
    c.u = first_unit(c.o, cta, G);
    if (c.u < c.o.nunits) { cur_unit(c); c.valid = true; return; }
  }
  c.valid = false;
}
template <bool PROG>
__device__ __forceinline__ void cur_start(const ProgArgs& a, StageCursor& c, int cta, int G) {
  c.oi = 0;
  cur_seek<PROG>(a, c, cta, G);
}
template <bool PROG>
__device__ __forceinline__ void cur_next(const ProgArgs& a, StageCursor& c, int cta, int G) {
  c.b0 += c.o.KC;
  if (c.b0 < c.kb1) return;
  c.u += G;
  if (c.u < c.o.nunits) { cur_unit(c); return; }
  ++c.oi;
  cur_seek<PROG>(a, c, cta, G);
}
// L2 prefetch of a stage's row segments (lane i: row i).
__device__ __forceinline__ void prefetch_stage(const StageCursor& c, int lane) {
  const int BB = block_bytes_of(c.o.type);
  const int n = min(c.o.KC, c.kb1 - c.b0);
  const int64_t row = static_cast<int64_t>(c.tile) * TT + lane;
  if (row < c.o.N) {
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(c.o.W + row * c.o.row_bytes + static_cast<int64_t>(c.b0) * BB);
    const uintptr_t e0 = s0 + static_cast<uintptr_t>(n) * BB;
    const uintptr_t as = s0 & ~uintptr_t(15), ae = (e0 + 15) & ~uintptr_t(15);
    bulk_prefetch_l2(reinterpret_cast<const void*>(as), static_cast<uint32_t>(ae - as));
  }
}

// Shared memory: barriers and counters (256 B), the ring, the reduction
// buffers, the x image.
__host__ __device__ inline size_t red_bytes(int S) { return static_cast<size_t>(S + 1) * NC * TT * 4; }

template <bool PROG>
__global__ void __launch_bounds__(NTH, 1) prog_kernel(const __grid_constant__ ProgArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  Ring rg;
  rg.full = reinterpret_cast<uint64_t*>(smem);
  rg.empty = rg.full + RING_MAX;
  rg.base = smem + 256;
  rg.base_s = smem_u32(rg.base);
  rg.S = a.S;
  rg.slot = a.slot;
  Red rd;
  rd.cnt = reinterpret_cast<int*>(rg.empty + RING_MAX);  // RING_MAX + 1 ints
  rd.RS = a.S + 1;
  rd.buf = reinterpret_cast<float*>(rg.base + static_cast<size_t>(a.S) * a.slot);
  uint8_t* xbase = reinterpret_cast<uint8_t*>(rd.buf) + red_bytes(a.S);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.S; ++s) { mbar_init(&rg.full[s], 1); mbar_init(&rg.empty[s], NC); }
    for (int s = 0; s <= a.S; ++s) rd.cnt[s] = 0;
  }
  fence_mbar_init();
  __syncthreads();

  if (warp == NC) {
    // ------------------------------------------------------------ producer
    pdl_launch_dependents();
    int64_t q = 0;
    StageCursor cc, pc;
    cur_start<PROG>(a, cc, cta, G);
    pc = cc;
    for (int k = 0; k < a.pf && pc.valid; ++k) cur_next<PROG>(a, pc, cta, G);
    while (cc.valid) {
      const int slot = static_cast<int>(q % a.S);
      if (q >= a.S) {
        const bool ok = mbar_wait(&rg.empty[slot], static_cast<uint32_t>((q / a.S - 1) & 1), a.err);
        if (!__all_sync(0xFFFFFFFFu, ok)) break;
      }
      if (pc.valid) {  // ask L2 for the stage a.pf stages ahead
        prefetch_stage(pc, lane);
        cur_next<PROG>(a, pc, cta, G);
      }
      produce(cc.o, cc.tile, cc.b0, min(cc.o.KC, cc.kb1 - cc.b0), rg.base + static_cast<size_t>(slot) * a.slot,
              &rg.full[slot], lane, block_bytes_of(cc.o.type));
      cur_next<PROG>(a, cc, cta, G);
      ++q;
    }
    // leave only after the copies in flight have landed (bounded)
    if (lane == 0)
      for (int64_t r = (q > a.S ? q - a.S : 0); r < q; ++r)
        mbar_wait(&rg.full[r % a.S], static_cast<uint32_t>((r / a.S) & 1), nullptr);
    return;
  }

  // --------------------------------------------------------------- consumers
  pdl_wait();
  pdl_launch_dependents();
  const int ctid = threadIdx.x;
  Walk wk = {0, 0, 0, false};
  int barriers = 0;
  int fixed = 0;  // ops before this index have their split-K sums added
  for (int oi = 0; oi < a.n_ops; ++oi) {
    const KqOp o = load_op<PROG>(a, oi);
    const int NL = o.x_bf16 ? 2 : 3;
    if (oi > 0 && (o.flags & OP_WAIT)) {
      // publish this CTA's outputs so far, then wait for the rest of the grid
      consumer_sync();
      ++barriers;
      if (ctid == 0) {
        __threadfence();
        atomicAdd(a.barrier, 1);
        grid_wait(a.barrier, barriers * G, a.err);  // on timeout the error word is set
      }
      consumer_sync();
      __threadfence();
      // split-K sums of the ops finished so far (no later op reads them: the
      // host plans no split for an op whose output feeds a later x)
      if constexpr (PROG) {
        for (; fixed < oi; ++fixed) {
          const KqOp f = load_op<PROG>(a, fixed);
          if (f.KS > 1) fixup_op(f, cta, G, ctid);
        }
      }
    }
    const XImg xi = ximg_at(xbase, a.nb_max, a.nl_max);
    if (oi == 0 || (o.flags & (OP_NEWX | OP_WAIT))) {
      consumer_sync();  // every consumer is done with the previous x image
      if (NL == 2) stage_x<2>(o.x, 1, o.K, o.nb, xi, ctid);
      else stage_x<3>(o.x, 0, o.K, o.nb, xi, ctid);
      consumer_sync();
    }
    if (NL == 2) consume_any<2>(o, xi, rg, rd, wk, a.err, cta, G);
    else consume_any<3>(o, xi, rg, rd, wk, a.err, cta, G);
  }
  if (a.barrier) {
    // final barrier (only when split-K sums remain), then the exit count: the
    // last CTA to leave resets both counters for the next launch
    consumer_sync();
    if (a.final_fix) {
      ++barriers;
      if (ctid == 0) {
        __threadfence();
        atomicAdd(a.barrier, 1);
        grid_wait(a.barrier, barriers * G, a.err);
      }
      consumer_sync();
      __threadfence();
      if constexpr (PROG) {
        for (; fixed < a.n_ops; ++fixed) {
          const KqOp f = load_op<PROG>(a, fixed);
          if (f.KS > 1) fixup_op(f, cta, G, ctid);
        }
      }
      consumer_sync();
    }
    if (ctid == 0) {
      __threadfence();
      const int v = atomicAdd(a.barrier + 1, 1);
      if (v == G - 1) { atomicExch(a.barrier, 0); atomicExch(a.barrier + 1, 0); }
    }
  }
}

// -------------------------------------------------------------------------
// Host side: geometry and launch.
// -------------------------------------------------------------------------

// Row stride of a stage of kc blocks: the row segment's 16-byte aligned
// superset (Q6_K: plus 16 bytes, the unaligned reads' slack), rounded to an
// odd number of 16-byte units so that neighbouring rows start in different banks.
int seg_stride(int type, int kc) {
  const int BB = block_bytes_of(type);
  const int slack = (type == T_Q6_K) ? 16 : 0;
  int srb = (kc * BB + 15 + slack + 15) & ~15;
  if ((srb / 16) % 2 == 0) srb += 16;
  return srb;
}

// Geometry of one op: K-parts KS (only with a workspace) and stage width KC.
// cost = block-chunks of the busiest CTA (a chunk = one block for 32 rows,
// dealt to one warp), plus a fixed cost per stage and per split.
bool plan_op(KqOp& o, int G, bool allow_split, int64_t slot_cap) {
  const int BB = block_bytes_of(o.type);
  if (!BB || o.K <= 0 || o.K % 32 || o.N <= 0) return false;
  o.nb = (o.K + 255) / 256;
  if (o.nb > MAX_NB) return false;
  o.row_bytes = static_cast<int64_t>(o.nb) * BB;
  const int64_t ntiles = (o.N + TT - 1) / TT;
  if (ntiles > (int64_t(1) << 28)) return false;
  int kcmax = o.nb;
  while (kcmax > 1 && static_cast<int64_t>(TT) * seg_stride(o.type, kcmax) > slot_cap) --kcmax;
  if (static_cast<int64_t>(TT) * seg_stride(o.type, kcmax) > slot_cap) return false;
  // K-parts (with a workspace): minimise the busiest CTA's blocks,
  // ceil(tiles*KS / G) * ceil(nb / KS), plus one block per split level
  int KS = 1;
  int64_t best = ((ntiles + G - 1) / G) * o.nb;
  for (int k2 = 2; allow_split && k2 <= 8; k2 *= 2) {
    const int kpb2 = (o.nb + k2 - 1) / k2;
    if (kpb2 < 2 || (k2 - 1) * kpb2 >= o.nb) break;
    const int64_t c = ((ntiles * k2 + G - 1) / G) * kpb2 + (k2 / 2);
    if (c < best) { best = c; KS = k2; }
  }
  o.KS = KS;
  o.kpb = (o.nb + KS - 1) / KS;
  // stages of a part: as few as fit, evened out
  const int nst = (o.kpb + kcmax - 1) / kcmax;
  o.KC = (o.kpb + nst - 1) / nst;
  o.srb = seg_stride(o.type, o.KC);
  o.ntiles = static_cast<int32_t>(ntiles);
  o.nunits = static_cast<int32_t>(ntiles * KS);
  return true;
}

int64_t stage_bytes(const KqOp& o) { return static_cast<int64_t>(TT) * o.srb; }

struct LaunchGeom {
  int S, slot;
  size_t smem;
};

bool ring_geom(int64_t max_stage, int nb_max, int nl_max, LaunchGeom& g) {
  g.slot = static_cast<int>((max_stage + 127) & ~int64_t(127));
  const size_t fixed = 256 + ximg_bytes(nb_max, nl_max);
  int S = RING_MAX;
  while (S >= 2 && fixed + static_cast<size_t>(S) * g.slot + red_bytes(S) > static_cast<size_t>(kMaxSmemPerBlock)) --S;
  if (S < 2) return false;
  g.S = S;
  g.smem = fixed + static_cast<size_t>(S) * g.slot + red_bytes(S);
  return true;
}

template <bool PROG>
cudaError_t launch_prog(ProgArgs& a, const LaunchGeom& g, bool cooperative, cudaStream_t st, bool pdl) {
  a.S = g.S;
  a.slot = g.slot;
  static bool smem_set[64] = {false};
  const int dev = current_device_id();
  if (!smem_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(prog_kernel<PROG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kMaxSmemPerBlock);
    if (e != cudaSuccess) return e;
    smem_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms());
  cfg.blockDim = dim3(NTH);
  cfg.dynamicSmemBytes = g.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (cooperative) {
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na].val.cooperative = 1;
    ++na;
  }
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, prog_kernel<PROG>, a);
}

// Program workspace: header (grid barrier counter), ops, split-K partials and counters.
constexpr size_t kHeaderBytes = 256;

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace

namespace {
int g_prefetch_stages = 8;  // L2 prefetch distance (stages beyond the one being copied)
}  // namespace
void set_prefetch_stages(int pf) { g_prefetch_stages = pf < 0 ? 0 : pf; }

cudaError_t launch_matvec1(int qtype, const void* W, const void* x, int x_bf16, float* y, int64_t N, int K,
                           cudaStream_t stream, bool pdl) {
  if (N == 0) return cudaSuccess;
  ProgArgs a = {};
  KqOp& o = a.op0;
  o.W = static_cast<const uint8_t*>(W);
  o.x = x;
  o.y = y;
  o.N = N;
  o.K = K;
  o.type = qtype;
  o.x_bf16 = x_bf16;
  o.flags = OP_NEWX;
  if (!plan_op(o, num_sms(), false, kSlotCap)) return cudaErrorNotSupported;
  LaunchGeom g;
  if (!ring_geom(stage_bytes(o), o.nb, x_bf16 ? 2 : 3, g)) return cudaErrorNotSupported;
  a.ops = nullptr;
  a.n_ops = 1;
  a.nb_max = o.nb;
  a.nl_max = x_bf16 ? 2 : 3;
  a.barrier = nullptr;
  a.err = device_error_ptr();
  a.pf = g_prefetch_stages;
  return launch_prog<false>(a, g, false, stream, pdl);
}

// Plans the whole program on the host and returns the workspace bytes it
// needs (0 if some op cannot run here).
namespace {
// Whether op i's output may be split across CTAs: no later op reads it as x
// (its sums are only complete after the next grid barrier).
bool split_allowed(const ProgOpDesc* d, int n_ops, int i) {
  const uintptr_t y0 = reinterpret_cast<uintptr_t>(d[i].y);
  const uintptr_t y1 = y0 + static_cast<uintptr_t>(d[i].N) * sizeof(float);
  for (int j = i + 1; j < n_ops; ++j) {
    const uintptr_t x0 = reinterpret_cast<uintptr_t>(d[j].x);
    const uintptr_t x1 = x0 + static_cast<uintptr_t>(d[j].K) * (d[j].x_bf16 ? 2 : 4);
    if (x0 < y1 && y0 < x1) return false;
  }
  return true;
}

// Plan every op of a program; false if some op cannot run on this path.
bool plan_prog(const ProgOpDesc* descs, int n_ops, KqOp* ops, size_t* part_bytes) {
  const int G = num_sms();
  size_t pb = 0;
  for (int i = 0; i < n_ops; ++i) {
    KqOp o = {};
    o.W = static_cast<const uint8_t*>(descs[i].W);
    o.x = descs[i].x;
    o.y = descs[i].y;
    o.N = descs[i].N;
    o.K = static_cast<int32_t>(descs[i].K);
    o.type = descs[i].type;
    o.x_bf16 = descs[i].x_bf16;
    if (!plan_op(o, G, split_allowed(descs, n_ops, i), kSlotCap)) return false;
    if (o.KS > 1) pb += align256(static_cast<size_t>(o.ntiles) * o.KS * TT * sizeof(float));
    ops[i] = o;
  }
  *part_bytes = pb;
  return true;
}
}  // namespace

size_t prog_workspace_size(const ProgOpDesc* descs, int n_ops) {
  if (n_ops <= 0) return 0;
  KqOp* ops = new KqOp[n_ops];
  size_t pb = 0;
  const bool ok = plan_prog(descs, n_ops, ops, &pb);
  delete[] ops;
  return ok ? align256(kHeaderBytes + static_cast<size_t>(n_ops) * sizeof(KqOp)) + pb : 0;
}

cudaError_t prog_prepare(const ProgOpDesc* descs, int n_ops, void* ws, size_t ws_bytes, ProgPlan* plan,
                         cudaStream_t stream) {
  const int G = num_sms();
  if (n_ops <= 0) return cudaErrorInvalidValue;
  KqOp* ops = new KqOp[n_ops];
  size_t pb = 0;
  if (!plan_prog(descs, n_ops, ops, &pb)) { delete[] ops; return cudaErrorNotSupported; }
  const size_t need = align256(kHeaderBytes + static_cast<size_t>(n_ops) * sizeof(KqOp)) + pb;
  if (ws_bytes < need) { delete[] ops; return cudaErrorInvalidValue; }
  uint8_t* w = static_cast<uint8_t*>(ws);
  size_t off = align256(kHeaderBytes + static_cast<size_t>(n_ops) * sizeof(KqOp));
  int nb_max = 1, nl_max = 2, any_wait = 0, last_wait = 0, final_fix = 0;
  int64_t max_stage = 0, rot = 0;
  for (int i = 0; i < n_ops; ++i) {
    KqOp& o = ops[i];
    o.flags = 0;
    if (i > 0 && descs[i].wait_previous) { o.flags |= OP_WAIT; any_wait = 1; last_wait = i; rot = 0; }
    if (i == 0 || descs[i].x != descs[i - 1].x || descs[i].K != descs[i - 1].K ||
        descs[i].x_bf16 != descs[i - 1].x_bf16)
      o.flags |= OP_NEWX;
    o.rot = static_cast<int32_t>(rot % G);
    rot += o.nunits;
    if (o.KS > 1) {
      o.part = reinterpret_cast<float*>(w + off);
      off += align256(static_cast<size_t>(o.ntiles) * o.KS * TT * sizeof(float));
    }
    if (o.nb > nb_max) nb_max = o.nb;
    if (!o.x_bf16) nl_max = 3;
    if (stage_bytes(o) > max_stage) max_stage = stage_bytes(o);
  }
  for (int i = last_wait; i < n_ops; ++i)
    if (ops[i].KS > 1) final_fix = 1;  // not summed at any later grid barrier
  LaunchGeom g;
  if (!ring_geom(max_stage, nb_max, nl_max, g)) { delete[] ops; return cudaErrorNotSupported; }
  plan->n_ops = n_ops;
  plan->nb_max = nb_max;
  plan->nl_max = nl_max;
  plan->S = g.S;
  plan->slot = g.slot;
  plan->coop = (any_wait || final_fix) ? 1 : 0;
  plan->final_fix = final_fix;
  plan->smem = static_cast<int64_t>(g.smem);
  plan->ws_bytes = static_cast<int64_t>(need);
  // the header's barrier counters start at zero; the ops follow the header
  cudaError_t e = cudaMemsetAsync(ws, 0, kHeaderBytes, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(w + kHeaderBytes, ops, sizeof(KqOp) * n_ops, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  delete[] ops;
  return e;
}

cudaError_t prog_run(const ProgPlan* plan, void* ws, cudaStream_t stream) {
  ProgArgs a = {};
  a.ops = reinterpret_cast<const KqOp*>(static_cast<const uint8_t*>(ws) + kHeaderBytes);
  a.n_ops = plan->n_ops;
  a.nb_max = plan->nb_max;
  a.nl_max = plan->nl_max;
  a.barrier = plan->coop ? static_cast<int*>(ws) : nullptr;
  a.final_fix = plan->final_fix;
  a.err = device_error_ptr();
  a.pf = g_prefetch_stages;
  LaunchGeom g;
  g.S = plan->S;
  g.slot = plan->slot;
  g.smem = static_cast<size_t>(plan->smem);
  // grid barriers need every CTA resident: cooperative launch
  return launch_prog<true>(a, g, plan->coop != 0, stream, plan->coop == 0);
}

}  // namespace kq
