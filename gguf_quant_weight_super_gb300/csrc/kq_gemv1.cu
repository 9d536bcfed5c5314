// kq_gemv1.cu -- fused dequantize + matrix x vector for one token (M = 1):
//     y[n] = sum_k w[n][k] * x[k]   for Q4_K / Q5_K / Q6_K weights.
//
// "GGUF in transformers", section "Reusing ggml's Metal kernels": decode-time
// products read the packed weights directly.  At one token the product is
// bound by the weight stream (0.56 to 0.82 bytes per weight), so the kernel is
// built to keep HBM busy while spending as few instructions per weight as the
// SM's integer pipe allows:
//
//  * x is converted once per CTA into block-floating-point integers: for every
//    run of 32 consecutive x values (one Q4_K/Q5_K sub-block, two Q6_K
//    sub-blocks) a power-of-two scale s = 2^(e - 14) (bf16 x) or 2^(e - 22)
//    (fp32 x), e the binary exponent of the run's largest |x|, and integers
//    m_k = rint(x_k / s), stored as 2 (or 3) byte limbs.  For bf16 x every
//    value within 2^7 of the run maximum is represented exactly; otherwise
//    |x_k - s*m_k| <= s/2 <= 2^-15 * max|x| (2^-23 for fp32 x).
//  * The codes of a sub-block are multiplied with the limbs by 4-way integer
//    dot products (dp4a), exactly, in int32; a part's contribution is
//        d*sc * s * (sum q*m)  -  dmin*m * (sum x)      (Q4_K, Q5_K)
//        d*sc * s * (sum q*m)  -  32*d*sc * (sum x)     (Q6_K)
//    accumulated in fp32; the sums of x use the exact x.
//  * persistent grid, one CTA of NW warps per SM; a warp owns a tile of TR
//    rows and a K-range and streams the tile's row segments (up to 8 blocks)
//    into its own ring of shared-memory stages with 1-D TMA bulk copies
//    (cp.async.bulk + mbarrier), requesting the first stages before
//    griddepcontrol.wait so the stream overlaps the previous kernel under
//    programmatic dependent launch;
//  * the warp's 8 quads of 4 lanes form 4 block slots x 2 row slots: a quad
//    loads its block's x limbs into registers once and applies them to RPQ
//    rows; lane c of a quad owns 64 weights of each block;
//  * when rows are too few to occupy every warp, K is split into ranges whose
//    partial sums are added, in range order, by the last warp to finish.
#include "kq_internal.h"

namespace kq {
namespace {

// Geometry (chosen by measurement on GB300; see the design notes).
#ifndef KQ_G1_NW
#define KQ_G1_NW 16
#endif
#ifndef KQ_G1_SMAX
#define KQ_G1_SMAX 2
#endif
#ifndef KQ_G1_KCMAX
#define KQ_G1_KCMAX 8
#endif
#ifndef KQ_G1_RPQ
#define KQ_G1_RPQ 2
#endif
#ifndef KQ_G1_MINB
#define KQ_G1_MINB 1
#endif
#ifndef KQ_G1_SMEM_CAP
#define KQ_G1_SMEM_CAP (227 * 1024)
#endif
#ifndef KQ_G1_ROWCONTIG_MAXNB
#define KQ_G1_ROWCONTIG_MAXNB 16
#endif

constexpr int NW = KQ_G1_NW;        // warps per CTA
constexpr int SMAX = KQ_G1_SMAX;    // ring stages per warp (at most)
constexpr int RPQ = KQ_G1_RPQ;      // rows per quad (2 row slots per warp)
constexpr int TR = 2 * RPQ;         // rows per warp tile
constexpr int KCMAX = KQ_G1_KCMAX;  // blocks per stage
constexpr int MINB = KQ_G1_MINB;    // CTAs per SM the register budget allows (2: room for the next kernel)
constexpr int SMEM_CAP = KQ_G1_SMEM_CAP;
constexpr int BAR_BYTES = (NW * SMAX * 8 + 127) / 128 * 128;

// Limb word i (x positions 4i..4i+3) lives at padded index i + 4*(i/16), so
// the 16-word slices read by the lanes of a quad fall in distinct banks.
__host__ __device__ __forceinline__ int wpad(int i) { return i + 4 * (i >> 4); }

template <int QT> struct Part;
template <> struct Part<T_Q4_K> { static constexpr int P = 2, PL = 32; };
template <> struct Part<T_Q5_K> { static constexpr int P = 2, PL = 32; };
template <> struct Part<T_Q6_K> { static constexpr int P = 4, PL = 16; };

// Position in the block of the first weight of part p of quad lane c.
template <int QT>
__host__ __device__ __forceinline__ int ppos(int c, int p) {
  if constexpr (QT == T_Q6_K) return 128 * (c >> 1) + 32 * p + 16 * (c & 1);
  else return 64 * c + 32 * p;
}

struct G1Args {
  const uint8_t* W;
  int64_t N;
  int K;
  int nb;
  int64_t row_bytes;
  const void* x;
  int x_bf16;
  float* y;
  int* err;
  int KB;             // blocks per K-range (multiple of 4 except a row's last range)
  int nr;             // K-ranges per row
  int S;              // ring stages per warp
  int KC;             // blocks per stage
  int srb;            // bytes per row inside a stage
  int rowcontig;      // a stage holds whole rows: one copy of TR consecutive rows
  int stage_bytes;
  int64_t ntiles;
  int tiles_per_cta;
};

// Shared-memory image of x: NL limb planes of padded words, the scale of each
// 32-run, and the sum of each 16-run of x.
template <int NL>
struct XImage {
  uint32_t* limb[NL];   // limb 0 = most significant (signed bytes), others unsigned bytes
  float* scale;         // [nb*8]
  float* sum16;         // [nb*16]
};

template <int NL>
__device__ void stage_x(const G1Args& a, const XImage<NL>& xi) {
  // thread t handles limb words t, t+T, ... (x positions 4w..4w+3); the 8
  // threads of a 32-run share its maximum through shuffles, the 4 threads of a
  // 16-run its sum.  All global loads are issued before any is used.
  constexpr int MAXIT = 16;  // words per thread; nb*64 <= MAXIT*blockDim.x is checked on the host
  const int nword = a.nb * 64;
  float v[MAXIT][4];
#pragma unroll
  for (int it = 0; it < MAXIT; ++it) {
    const int wq = it * blockDim.x + threadIdx.x;
    const int k0 = wq * 4;
    v[it][0] = v[it][1] = v[it][2] = v[it][3] = 0.0f;
    if (wq < nword && k0 < a.K) {  // K is a multiple of 32: a word is all in or all out
      if (a.x_bf16) {
        const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.x) + k0);
        v[it][0] = __uint_as_float(u.x << 16); v[it][1] = __uint_as_float(u.x & 0xFFFF0000u);
        v[it][2] = __uint_as_float(u.y << 16); v[it][3] = __uint_as_float(u.y & 0xFFFF0000u);
      } else {
        const float4 u = *reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + k0);
        v[it][0] = u.x; v[it][1] = u.y; v[it][2] = u.z; v[it][3] = u.w;
      }
    }
  }
#pragma unroll
  for (int it = 0; it < MAXIT; ++it) {
    const int wq = it * blockDim.x + threadIdx.x;
    if (it * static_cast<int>(blockDim.x) >= nword) break;  // uniform across the block
    float mx = fmaxf(fmaxf(fabsf(v[it][0]), fabsf(v[it][1])), fmaxf(fabsf(v[it][2]), fabsf(v[it][3])));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
    float sm = __fadd_rn(__fadd_rn(v[it][0], v[it][1]), __fadd_rn(v[it][2], v[it][3]));
    sm = __fadd_rn(sm, __shfl_xor_sync(0xFFFFFFFFu, sm, 1));
    sm = __fadd_rn(sm, __shfl_xor_sync(0xFFFFFFFFu, sm, 2));
    if (wq < nword) {
      // e: binary exponent of mx (mx = f * 2^e, f in [0.5, 1)); read from the
      // bits for normal values, from frexpf for the rare subnormal / huge run
      int e;
      const uint32_t mb = __float_as_uint(mx);
      const int be = static_cast<int>((mb >> 23) & 0xFF);
      const bool fast = be >= 40 && be <= 200;
      if (fast) e = be - 126;
      else frexpf(mx, &e);
      const int shift = (NL == 2 ? 14 : 22) - e;   // m = rint(x * 2^shift), |m| < 2^14 (2^22)
      const float p2 = fast ? __uint_as_float(static_cast<uint32_t>(127 + shift) << 23) : 0.0f;
      uint32_t wl[NL];
#pragma unroll
      for (int l = 0; l < NL; ++l) wl[l] = 0;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float xs2 = fast ? v[it][t] * p2 : ldexpf(v[it][t], shift);  // exact: power-of-two scale
        const int m = (mx > 0.0f) ? __float2int_rn(xs2) : 0;
        // m = hi * 256^(NL-1) + ... + lo, lo (and mid) in 0..255, hi signed
        if constexpr (NL == 2) {
          wl[1] |= static_cast<uint32_t>(m & 0xFF) << (8 * t);
          wl[0] |= static_cast<uint32_t>((m >> 8) & 0xFF) << (8 * t);
        } else {
          wl[2] |= static_cast<uint32_t>(m & 0xFF) << (8 * t);
          wl[1] |= static_cast<uint32_t>((m >> 8) & 0xFF) << (8 * t);
          wl[0] |= static_cast<uint32_t>((m >> 16) & 0xFF) << (8 * t);
        }
      }
      const int idx = wpad(wq);
#pragma unroll
      for (int l = 0; l < NL; ++l) xi.limb[l][idx] = wl[l];
      if ((wq & 7) == 0)
        xi.scale[wq >> 3] = (mx > 0.0f) ? (fast ? __uint_as_float(static_cast<uint32_t>(127 - shift) << 23)
                                                : ldexpf(1.0f, -shift)) : 0.0f;
      if ((wq & 3) == 0) xi.sum16[wq >> 2] = sm;
    }
  }
  __syncthreads();
}

__device__ __forceinline__ uint4 lds16_unaligned(const uint8_t* p) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
  const uint32_t sh = static_cast<uint32_t>(a & 3) * 8;
  const uint32_t w0 = w[0], w1 = w[1], w2 = w[2], w3 = w[3], w4 = w[4];
  return make_uint4(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh), __funnelshift_r(w2, w3, sh),
                    __funnelshift_r(w3, w4, sh));
}

__device__ __forceinline__ uint32_t wsel(const uint4& v, int w) {
  return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
}

// signed / unsigned 4-way byte dot products accumulated in int32
__device__ __forceinline__ int dp_s(uint32_t codes, uint32_t limb, int acc) {
  return __dp4a(static_cast<int>(codes), static_cast<int>(limb), acc);  // codes < 128: same as unsigned
}
__device__ __forceinline__ int dp_u(uint32_t codes, uint32_t limb, int acc) {
  return static_cast<int>(__dp4a(codes, limb, static_cast<unsigned>(acc)));
}

// x slice of one block for lane c, held in registers.
template <int QT, int NL>
struct XSlice {
  uint32_t w[NL][16];            // limb words, in the lane's part order
  float s[Part<QT>::P];          // run scale of each part
  float X[Part<QT>::P];          // sum of x over each part
};

template <int QT, int NL>
__device__ __forceinline__ void load_slice(const XImage<NL>& xi, int b, int c, XSlice<QT, NL>& xs) {
  constexpr int P = Part<QT>::P;
#pragma unroll
  for (int p = 0; p < P; ++p) {
    const int pos = b * 256 + ppos<QT>(c, p);     // first x position of the part
    constexpr int NW_P = Part<QT>::PL / 4;         // limb words per part
#pragma unroll
    for (int l = 0; l < NL; ++l)
#pragma unroll
      for (int j = 0; j < NW_P; j += 4) {
        const uint4 u = *reinterpret_cast<const uint4*>(xi.limb[l] + wpad(pos / 4 + j));
        xs.w[l][p * NW_P + j] = u.x; xs.w[l][p * NW_P + j + 1] = u.y;
        xs.w[l][p * NW_P + j + 2] = u.z; xs.w[l][p * NW_P + j + 3] = u.w;
      }
    xs.s[p] = xi.scale[pos / 32];
    if constexpr (QT == T_Q6_K) xs.X[p] = xi.sum16[pos / 16];
    else xs.X[p] = __fadd_rn(xi.sum16[pos / 16], xi.sum16[pos / 16 + 1]);
  }
}

// Integer dot of 4 codes with the 4 matching x values: limb-weighted sum.
template <int NL>
__device__ __forceinline__ void dot4(uint32_t codes, const uint32_t (&w)[NL][16], int j, int (&I)[NL]) {
  I[0] = dp_s(codes, w[0][j], I[0]);
#pragma unroll
  for (int l = 1; l < NL; ++l) I[l] = dp_u(codes, w[l][j], I[l]);
}

template <int NL>
__device__ __forceinline__ float limbs_to_float(const int (&I)[NL]) {
  if constexpr (NL == 2) return static_cast<float>(I[0] * 256 + I[1]);  // |.| < 2^24: exact
  else return __fmaf_rn(static_cast<float>(I[0]), 65536.0f, __fmaf_rn(static_cast<float>(I[1]), 256.0f, static_cast<float>(I[2])));
}

// acc += sum over lane c's parts of block b: A_p * T_p + B_p * X_p.
template <int QT, int NL>
__device__ __forceinline__ float2 rowblock(const uint8_t* b, int c, int rem, const XSlice<QT, NL>& xs, float2 acc) {
  constexpr int P = Part<QT>::P;
  constexpr int PL = Part<QT>::PL;
  int I[P][NL];
#pragma unroll
  for (int p = 0; p < P; ++p)
#pragma unroll
    for (int l = 0; l < NL; ++l) I[p][l] = 0;
  float A[P], B[P];
  if constexpr (QT == T_Q6_K) {
    const int h = c >> 1, l0 = 16 * (c & 1);
    const uint4 qa = lds16_unaligned(b + 64 * h + l0);
    const uint4 qb = lds16_unaligned(b + 64 * h + 32 + l0);
    const uint4 qh = lds16_unaligned(b + 128 + 32 * h + l0);
    const uint2 s = ld8_a2(b + 192 + 8 * h + (c & 1));
    const uint32_t se = __byte_perm(s.x, s.y, 0x6420);  // scales 8h + 2t + (c & 1), t = 0..3
    const float d = half_bits_to_float(reinterpret_cast<const uint16_t*>(b + 208)[0]);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float dsc = d * static_cast<float>(static_cast<int8_t>((se >> (8 * t)) & 0xFF));
      const bool ok = ppos<QT>(c, t) + PL <= rem;
      A[t] = ok ? dsc * xs.s[t] : 0.0f;
      B[t] = ok ? -32.0f * dsc : 0.0f;
    }
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint32_t av = wsel(qa, w), bv = wsel(qb, w), hv = wsel(qh, w);
      // 6-bit codes: low nibble | (2 high bits) << 4
      const uint32_t c0 = (av & 0x0F0F0F0Fu) | ((hv << 4) & 0x30303030u);
      const uint32_t c1 = (bv & 0x0F0F0F0Fu) | ((hv << 2) & 0x30303030u);
      const uint32_t c2 = ((av >> 4) & 0x0F0F0F0Fu) | (hv & 0x30303030u);
      const uint32_t c3 = ((bv >> 4) & 0x0F0F0F0Fu) | ((hv >> 2) & 0x30303030u);
      dot4<NL>(c0, xs.w, 0 * 4 + w, I[0]);  // part t uses limb words 4t..4t+3
      dot4<NL>(c1, xs.w, 1 * 4 + w, I[1]);
      dot4<NL>(c2, xs.w, 2 * 4 + w, I[2]);
      dot4<NL>(c3, xs.w, 3 * 4 + w, I[3]);
    }
  } else {
    const uint4 hdr = *reinterpret_cast<const uint4*>(b);
    constexpr int QS = (QT == T_Q4_K) ? 16 : 48;
    const uint4 q0 = *reinterpret_cast<const uint4*>(b + QS + 32 * c);
    const uint4 q1 = *reinterpret_cast<const uint4*>(b + QS + 32 * c + 16);
    uint4 h0 = make_uint4(0, 0, 0, 0), h1 = make_uint4(0, 0, 0, 0);
    if constexpr (QT == T_Q5_K) {
      h0 = *reinterpret_cast<const uint4*>(b + 16);
      h1 = *reinterpret_cast<const uint4*>(b + 32);
    }
    const uint32_t v = scale_min_bytes(hdr.y, hdr.z, hdr.w, c);
    const float d = half_bits_to_float(hdr.x & 0xFFFF);
    const float dmin = half_bits_to_float(hdr.x >> 16);
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const float dsc = d * static_cast<float>((v >> (8 * p)) & 0xFF);
      const float mm = dmin * static_cast<float>((v >> (16 + 8 * p)) & 0xFF);
      const bool ok = ppos<QT>(c, p) + PL <= rem;
      A[p] = ok ? dsc * xs.s[p] : 0.0f;
      B[p] = ok ? -mm : 0.0f;
    }
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const uint32_t q = (w < 4) ? wsel(q0, w) : wsel(q1, w - 4);
      uint32_t lo, hi;
      if constexpr (QT == T_Q4_K) {
        lo = q & 0x0F0F0F0Fu;
        hi = (q >> 4) & 0x0F0F0F0Fu;
      } else {
        const uint32_t hb = (w < 4) ? wsel(h0, w) : wsel(h1, w - 4);
        lo = (q & 0x0F0F0F0Fu) | (__funnelshift_l(hb, hb, (4 - 2 * c) & 31) & 0x10101010u);
        hi = ((q >> 4) & 0x0F0F0F0Fu) | (__funnelshift_l(hb, hb, (3 - 2 * c) & 31) & 0x10101010u);
      }
      dot4<NL>(lo, xs.w, w, I[0]);
      dot4<NL>(hi, xs.w, 8 + w, I[1]);
    }
  }
  float T[P];
#pragma unroll
  for (int p = 0; p < P; ++p) T[p] = limbs_to_float<NL>(I[p]);
#pragma unroll
  for (int p = 0; p < P; p += 2) {
    acc = ffma2(make_float2(A[p], A[p + 1]), make_float2(T[p], T[p + 1]), acc);
    acc = ffma2(make_float2(B[p], B[p + 1]), make_float2(xs.X[p], xs.X[p + 1]), acc);
  }
  return acc;
}

// Row segment [b0, b0+nblk) of row r0+i as a 16-byte aligned superset.
template <int BB>
__device__ __forceinline__ uint32_t seg_of(const G1Args& a, int64_t row, int b0, int nblk, const uint8_t*& src) {
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(a.W + row * a.row_bytes + static_cast<int64_t>(b0) * BB);
  const uintptr_t e0 = s0 + static_cast<uintptr_t>(nblk) * BB;
  const uintptr_t as = s0 & ~uintptr_t(15), ae = (e0 + 15) & ~uintptr_t(15);
  src = reinterpret_cast<const uint8_t*>(as);
  return static_cast<uint32_t>(ae - as);
}

// Whole warp: copy the TR row segments of one stage into a ring slot (lane i
// issues row i's copy; lane 0 first posts the byte count on the barrier).
template <int BB>
__device__ __forceinline__ void issue_stage(const G1Args& a, int64_t tile, int b0, int nblk, uint8_t* slot,
                                            uint64_t* bar, int lane) {
  if (a.rowcontig) {  // whole rows: the tile's rows are one contiguous byte range
    if (lane == 0) {
      const int64_t r0 = tile * TR;
      const int64_t nrows = min_i64(TR, a.N - r0);
      const uintptr_t s0 = reinterpret_cast<uintptr_t>(a.W + r0 * a.row_bytes);
      const uintptr_t e0 = s0 + static_cast<uintptr_t>(nrows * a.row_bytes);
      const uintptr_t as = s0 & ~uintptr_t(15), ae = (e0 + 15) & ~uintptr_t(15);
      const uint32_t len = static_cast<uint32_t>(ae - as);
      mbar_arrive_expect_tx(bar, len);
      bulk_g2s(slot, reinterpret_cast<const uint8_t*>(as), len, bar);
    }
    __syncwarp();
    return;
  }
  const int64_t row = tile * TR + lane;
  const bool mine = lane < TR && row < a.N;
  const uint8_t* src = nullptr;
  const uint32_t len = mine ? seg_of<BB>(a, row, b0, nblk, src) : 0u;
  const uint32_t total = __reduce_add_sync(0xFFFFFFFFu, len);
  if (lane == 0) mbar_arrive_expect_tx(bar, total);
  __syncwarp();
  if (mine) bulk_g2s(slot + lane * a.srb, src, len, bar);
}

// A stage cursor: (unit u, block offset cb within the unit's K-range).
struct Cursor {
  int64_t u;
  int cb;
};

template <int QT, int NL>
__global__ void __launch_bounds__(NW * 32, MINB) gemv1_kernel(const G1Args a) {
  constexpr int BB = Fmt<QT>::BYTES;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint8_t* ring = smem + BAR_BYTES;
  const int nwords = wpad(a.nb * 64);
  XImage<NL> xi;
  uint32_t* lp = reinterpret_cast<uint32_t*>(ring + static_cast<size_t>(NW) * a.S * a.stage_bytes);
#pragma unroll
  for (int l = 0; l < NL; ++l) xi.limb[l] = lp + l * nwords;
  xi.scale = reinterpret_cast<float*>(lp + NL * nwords);
  xi.sum16 = xi.scale + a.nb * 8;
  float* part = xi.sum16 + a.nb * 16;  // [tiles_per_cta][TR][nr] when nr > 1
  int* cnt = reinterpret_cast<int*>(part + (a.nr > 1 ? a.tiles_per_cta * TR * a.nr : 0));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = lane >> 2, c = lane & 3;
  const int bs = quad & 3, rs = quad >> 2;  // block slot, row slot
  uint64_t* wbar = bars + warp * SMAX;
  uint8_t* wring = ring + static_cast<size_t>(warp) * a.S * a.stage_bytes;

  if (lane == 0)
    for (int s = 0; s < a.S; ++s) mbar_init(&wbar[s], 1);
  if (a.nr > 1)
    for (int t = threadIdx.x; t < a.tiles_per_cta; t += blockDim.x) cnt[t] = 0;
  fence_mbar_init();
  __syncthreads();

  const int64_t my_tiles = (a.ntiles > blockIdx.x) ? (a.ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int64_t my_units = my_tiles * a.nr;
  auto unit_tile = [&](int64_t u) -> int64_t { return blockIdx.x + (u / a.nr) * static_cast<int64_t>(gridDim.x); };
  auto range_len = [&](int r) -> int { return min(a.KB, a.nb - r * a.KB); };

  // stage cursor: next stage (unit, block offset) to copy into the ring
  auto advance = [&](Cursor& k) {
    const int rl = range_len(static_cast<int>(k.u % a.nr));
    k.cb += a.KC;
    if (k.cb >= rl) { k.u += NW; k.cb = 0; }
  };
  auto stage_blocks = [&](const Cursor& k) {
    const int r = static_cast<int>(k.u % a.nr);
    return min(a.KC, range_len(r) - k.cb);
  };
  Cursor tc = {warp, 0};
  int64_t issued = 0;
  auto issue_next = [&]() {
    issue_stage<BB>(a, unit_tile(tc.u), static_cast<int>(tc.u % a.nr) * a.KB + tc.cb, stage_blocks(tc),
                    wring + (issued % a.S) * a.stage_bytes, &wbar[issued % a.S], lane);
    ++issued;
    advance(tc);
  };
  while (issued < a.S && tc.u < my_units) issue_next();

  pdl_wait();
  pdl_launch_dependents();
  stage_x<NL>(a, xi);

  bool failed = false;
  int64_t q = 0, q_fail = 0;
  for (int64_t u = warp; u < my_units; u += NW) {
    const int64_t tile = unit_tile(u);
    const int r = static_cast<int>(u % a.nr);
    const int rb0 = r * a.KB, rl = range_len(r);
    float2 acc[RPQ];
#pragma unroll
    for (int k = 0; k < RPQ; ++k) acc[k] = make_float2(0.f, 0.f);

    for (int cb = 0; cb < rl; cb += a.KC) {
      const int n = min(a.KC, rl - cb);
      const int slot = static_cast<int>(q % a.S);
      const uint8_t* sp = wring + slot * a.stage_bytes;
      if (!failed) {
        const bool ok = mbar_wait(&wbar[slot], static_cast<uint32_t>((q / a.S) & 1), a.err);
        failed = __any_sync(0xFFFFFFFFu, !ok);
        if (failed) q_fail = q;
      }
      if (!failed) {
        // the rows of this quad: rs, rs+2, rs+4, ...
        const uint8_t* rowp[RPQ];
        bool rok[RPQ];
#pragma unroll
        for (int k = 0; k < RPQ; ++k) {
          const int lr = rs + 2 * k;
          const int64_t row = tile * TR + lr;
          rok[k] = row < a.N;
          if (a.rowcontig) {
            const uintptr_t s0 = reinterpret_cast<uintptr_t>(a.W + tile * TR * a.row_bytes);
            rowp[k] = sp + (s0 & 15) + lr * a.row_bytes;
          } else {
            const uintptr_t s0 = reinterpret_cast<uintptr_t>(a.W + row * a.row_bytes +
                                                             static_cast<int64_t>(rb0 + cb) * BB);
            rowp[k] = sp + lr * a.srb + (s0 & 15);
          }
        }
        for (int sb = 0; sb < n; sb += 4) {
          const int bi = sb + bs;           // block of this quad within the stage
          if (bi < n) {
            const int b = rb0 + cb + bi;    // block within the row
            const int rem = min(256, a.K - b * 256);
            XSlice<QT, NL> xsl;
            load_slice<QT, NL>(xi, b, c, xsl);
#pragma unroll
            for (int k = 0; k < RPQ; ++k)
              if (rok[k]) acc[k] = rowblock<QT, NL>(rowp[k] + bi * BB, c, rem, xsl, acc[k]);
          }
        }
      }
      ++q;
      __syncwarp();
      if (!failed && tc.u < my_units) {
        fence_proxy_async_smem();
        issue_next();
      }
    }
    if (failed) continue;
    // row sums over the 16 lanes that share a row slot (4 block slots x 4 lanes)
    float rsum[RPQ];
#pragma unroll
    for (int k = 0; k < RPQ; ++k) {
      float v = __fadd_rn(acc[k].x, acc[k].y);
      v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, 1));
      v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, 2));
      v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, 4));
      v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, 8));
      rsum[k] = v;
    }
    const int64_t il = (tile - blockIdx.x) / gridDim.x;
    const bool writer = (bs == 0 && c == 0);  // lanes 0 and 16
    if (a.nr == 1) {
      if (writer)
#pragma unroll
        for (int k = 0; k < RPQ; ++k) {
          const int64_t row = tile * TR + rs + 2 * k;
          if (row < a.N) a.y[row] = rsum[k];
        }
    } else {
      if (writer)
#pragma unroll
        for (int k = 0; k < RPQ; ++k) part[(il * TR + rs + 2 * k) * a.nr + r] = rsum[k];
      __threadfence_block();
      __syncwarp();
      int last = 0;
      if (lane == 0) last = (atomicAdd(&cnt[il], 1) == a.nr - 1);
      last = __shfl_sync(0xFFFFFFFFu, last, 0);
      if (last) {
        __threadfence_block();
        if (lane < TR) {
          const int64_t row = tile * TR + lane;
          if (row < a.N) {
            const float* pp = part + (il * TR + lane) * a.nr;
            float v = pp[0];
            for (int rr = 1; rr < a.nr; ++rr) v = __fadd_rn(v, pp[rr]);
            a.y[row] = v;
          }
        }
      }
    }
  }
  if (failed && lane == 0)
    for (int64_t rr = q_fail; rr < issued; ++rr)
      mbar_wait(&wbar[rr % a.S], static_cast<uint32_t>((rr / a.S) & 1), nullptr);
}

size_t g1_smem(int nb, int NL, int S, int stage_bytes, int nr, int tiles_per_cta) {
  size_t s = BAR_BYTES + static_cast<size_t>(NW) * S * stage_bytes;
  s += static_cast<size_t>(NL) * wpad(nb * 64) * 4;          // limb planes
  s += static_cast<size_t>(nb) * (8 + 16) * 4;               // run scales, 16-run sums
  if (nr > 1) s += static_cast<size_t>(tiles_per_cta) * TR * nr * 4 + tiles_per_cta * 4;
  return s;
}

template <int QT, int NL>
cudaError_t launch_g1(const G1Args& a, size_t smem, int grid, cudaStream_t st, bool pdl) {
  auto kern = gemv1_kernel<QT, NL>;
  static bool smem_set[64] = {false};
  const int dev = current_device_id();
  if (!smem_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmemPerBlock);
    if (e != cudaSuccess) return e;
    smem_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(NW * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int QT>
cudaError_t launch_g1_t(const G1Args& a, size_t smem, int grid, cudaStream_t st, bool pdl) {
  return a.x_bf16 ? launch_g1<QT, 2>(a, smem, grid, st, pdl) : launch_g1<QT, 3>(a, smem, grid, st, pdl);
}

}  // namespace

cudaError_t launch_gemv1(int qtype, const void* W, const void* x, int x_bf16, float* y, int64_t N, int K,
                         cudaStream_t stream, bool pdl) {
  if (N == 0) return cudaSuccess;
  const int BB = block_bytes_of(qtype);
  G1Args a = {};
  a.W = static_cast<const uint8_t*>(W);
  a.N = N;
  a.K = K;
  a.nb = (K + 255) / 256;
  a.row_bytes = static_cast<int64_t>(a.nb) * BB;
  a.x = x;
  a.x_bf16 = x_bf16;
  a.y = y;
  a.err = device_error_ptr();
  a.ntiles = (N + TR - 1) / TR;
  const int grid = static_cast<int>(min_i64(a.ntiles, num_sms()));
  a.tiles_per_cta = static_cast<int>((a.ntiles + grid - 1) / grid);
  // split K only when tiles are too few to give every warp two units
  const int64_t target = 2LL * num_sms() * NW;
  int64_t nr = (target + a.ntiles - 1) / a.ntiles;
  const int max_nr = (a.nb + 3) / 4;
  if (nr > max_nr) nr = max_nr;
  if (nr < 1) nr = 1;
  int KB = static_cast<int>((a.nb + nr - 1) / nr);
  KB = (KB + 3) / 4 * 4;
  a.KB = KB;
  a.nr = (a.nb + KB - 1) / KB;
  const int NL = x_bf16 ? 2 : 3;
  if (a.nb * 64 > 16 * NW * 32) return cudaErrorNotSupported;  // x words per thread (stage_x)
  // ring: whole-row stages (one copy per stage) when they fit, else row
  // segments of up to KCMAX blocks; deepest ring that fits
  const int slack = (qtype == T_Q6_K) ? 32 : 0;
  size_t smem = 0;
  bool fit = false;
  if (a.nr == 1 && a.nb <= KQ_G1_ROWCONTIG_MAXNB) {
    const int stage = static_cast<int>(((TR * a.row_bytes + 32 + 15) / 16) * 16);
    for (int S = SMAX; S >= 2 && !fit; --S) {
      smem = g1_smem(a.nb, NL, S, stage, 1, a.tiles_per_cta);
      if (smem <= static_cast<size_t>(SMEM_CAP)) {
        a.KC = a.nb;
        a.S = S;
        a.srb = static_cast<int>(a.row_bytes);
        a.stage_bytes = stage;
        a.rowcontig = 1;
        fit = true;
      }
    }
  }
  for (int kc = (KB < KCMAX ? KB : KCMAX); kc >= 4 && !fit; kc -= 4) {
    for (int S = SMAX; S >= 2 && !fit; --S) {
      int srb = (kc * BB + slack + 15) & ~15;
      if ((srb / 16) % 2 == 0) srb += 16;  // odd multiple of 16 bytes: rows start in different banks
      smem = g1_smem(a.nb, NL, S, TR * srb, a.nr, a.tiles_per_cta);
      if (smem <= static_cast<size_t>(SMEM_CAP)) {
        a.KC = kc;
        a.S = S;
        a.srb = srb;
        a.stage_bytes = TR * srb;
        fit = true;
      }
    }
  }
  if (!fit) return cudaErrorNotSupported;
  switch (qtype) {
    case T_Q4_K: return launch_g1_t<T_Q4_K>(a, smem, grid, stream, pdl);
    case T_Q5_K: return launch_g1_t<T_Q5_K>(a, smem, grid, stream, pdl);
    case T_Q6_K: return launch_g1_t<T_Q6_K>(a, smem, grid, stream, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kq
