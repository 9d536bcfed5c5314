// kq_gemv_batched.cu -- fused dequantize + matrix x small batch of vectors on CUDA
// cores, for Q4_K / Q5_K / Q6_K weights:  y[m][n] = sum_k w[n][k] * x[m][k].
//
// "GGUF in transformers", section "Reusing ggml's Metal kernels": the
// quantization kernel reads the packed weights directly and never expands the
// whole matrix before a decode-time product.  This is that operation for
// sm_103a.  Decode is bound by the weight stream, so every weight byte is read
// from HBM exactly once and the arithmetic per weight is kept small enough for
// the CUDA cores to keep pace with HBM:
//
//  * persistent grid, one CTA (NW warps) per SM;
//  * a row is handled by a "quad" of 4 lanes, lane c owning chunk c of every
//    block (64 weights: sub-blocks 2c and 2c+1 for Q4_K/Q5_K; four 16-weight
//    runs for Q6_K), so each lane decodes 2 (or 4) scales per 64 weights;
//  * work units are (tile of TR rows) x (K-range of KB blocks); every warp owns
//    a ring of S shared-memory stages that it fills with 1-D TMA bulk copies
//    of its units' row segments (Q6_K's 210-byte blocks are fetched as the
//    16-byte aligned superset and addressed at their true offset);
//  * x (fp32) lives in shared memory; lanes turn codes into floats
//    f = 1 + q/2^s with one byte-permute each, form every weight exactly
//    rounded, w = (f - 1) 2^s d sc - dmin m (f - 1 is exact), and accumulate
//    w x with packed fp32x2 FMAs;
//  * K-range partial sums of a tile are combined, in range order, by the last
//    warp of the CTA to finish one of that tile's units;
//  * weight tiles are requested before griddepcontrol.wait, so under
//    programmatic dependent launch the weight stream overlaps the previous
//    kernel's tail; x and y are touched only after the wait.
//
// Summation order depends only on the matrix shape: per row, each quad sums
// per lane over SEG-block segments, folds a segment over its 4 lanes in a fixed
// butterfly, adds segments in order into its K-range value, and K-range values
// are added in order.  Results are therefore bit-identical for every M, tile
// shape and x-window split (a launch that continues a row adds onto y, which
// holds exactly the running sum).
#include "kq_internal.h"

namespace kq {

namespace {

constexpr int NW = 16;           // warps per CTA
constexpr int S = 4;             // ring stages per warp
constexpr int SEG = 2;           // blocks per reduction segment
constexpr int STAGE_TARGET = 3072;
constexpr int KB_MAX = 8;        // blocks per K-range at most
constexpr int BAR_BYTES = (NW * S * 8 + 127) / 128 * 128;

// Quad layout per format: P parts of PL consecutive weights per lane.
template <int QT> struct QuadFmt;
template <> struct QuadFmt<T_Q4_K> { static constexpr int P = 2, PL = 32; };
template <> struct QuadFmt<T_Q5_K> { static constexpr int P = 2, PL = 32; };
template <> struct QuadFmt<T_Q6_K> { static constexpr int P = 4, PL = 16; };
template <> struct QuadFmt<T_IA4> { static constexpr int P = 2, PL = 32; };

// position within the block of the first weight of part p of quad lane c
template <int QT>
__device__ __forceinline__ int qpos(int c, int p) {
  if constexpr (QT == T_Q6_K) return 128 * (c >> 1) + 32 * p + 16 * (c & 1);
  else return 64 * c + 32 * p;
}

struct GemvArgs {
  const uint8_t* W;
  int64_t N;
  int K;
  int nb;                // blocks per row
  int64_t row_bytes;
  const void* x;
  int x_bf16;
  int M;
  float* y;
  int* err;
  // geometry (host-computed)
  int KB;                // blocks per K-range (a multiple of SEG)
  int nranges;           // K-ranges per row in total
  int r_begin, r_end;    // K-ranges handled by this launch
  int accumulate;        // add onto y (this launch continues rows started earlier)
  int KC;                // blocks per ring stage
  int slot_row_bytes;
  int stage_bytes;
  int64_t ntiles;        // ceil(N / TR)
  int tiles_per_cta;     // ceil(ntiles / gridDim.x)
  int xblk0, xblks;      // x window: first block, number of blocks
};

// ---------------------------------------------------------------------------
// x staging: fp32 copy of x[:, window] (zero past K) and per-PL-run sums.
// ---------------------------------------------------------------------------
template <int PL>
__device__ void stage_x(const GemvArgs& a, float* xs, float* Xs) {
  const int wlen = a.xblks * 256;
  const int k0 = a.xblk0 * 256;
  const int tid = threadIdx.x, nthr = blockDim.x;
  for (int m = 0; m < a.M; ++m) {
    float* xr = xs + m * wlen;
    if (a.x_bf16) {
      const uint16_t* src = static_cast<const uint16_t*>(a.x) + static_cast<int64_t>(m) * a.K;
      for (int i = tid * 8; i < wlen; i += nthr * 8) {
        const int k = k0 + i;
        float v[8];
        if (k < a.K) {  // K is a multiple of 32: a group of 8 is all in or all out
          const uint4 u = *reinterpret_cast<const uint4*>(src + k);
          const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            v[2 * t] = __uint_as_float(uw[t] << 16);
            v[2 * t + 1] = __uint_as_float(uw[t] & 0xFFFF0000u);
          }
        } else {
#pragma unroll
          for (int t = 0; t < 8; ++t) v[t] = 0.0f;
        }
        *reinterpret_cast<float4*>(xr + i) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4*>(xr + i + 4) = make_float4(v[4], v[5], v[6], v[7]);
      }
    } else {
      const float* src = static_cast<const float*>(a.x) + static_cast<int64_t>(m) * a.K;
      for (int i = tid * 4; i < wlen; i += nthr * 4) {
        const int k = k0 + i;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < a.K) v = *reinterpret_cast<const float4*>(src + k);
        *reinterpret_cast<float4*>(xr + i) = v;
      }
    }
  }
  __syncthreads();
  const int nrun = wlen / PL;
  for (int t = tid; t < a.M * nrun; t += nthr) {
    const int m = t / nrun, r = t % nrun;
    const float* p = xs + m * wlen + r * PL;
    float s = p[0];
#pragma unroll
    for (int i = 1; i < PL; ++i) s = __fadd_rn(s, p[i]);
    Xs[m * nrun + r] = s;
  }
  __syncthreads();
}

__device__ __forceinline__ int range_blocks(const GemvArgs& a, int r) { return min(a.KB, a.nb - r * a.KB); }

// Request TR row segments [b0, b0+nblk) of tile `tile` into one ring stage.
template <int TR, int BB>
__device__ __forceinline__ void issue_job(const GemvArgs& a, int64_t tile, int b0, int nblk, uint8_t* slot,
                                          uint64_t* bar) {
  const int64_t r0 = tile * TR;
  const int nrows = static_cast<int>(min_i64(TR, a.N - r0));
  uint32_t total = 0;
  const uint8_t* src[TR];
  uint32_t len[TR];
#pragma unroll
  for (int i = 0; i < TR; ++i) {
    if (i < nrows) {
      const uintptr_t s0 =
          reinterpret_cast<uintptr_t>(a.W + (r0 + i) * a.row_bytes + static_cast<int64_t>(b0) * BB);
      const uintptr_t e0 = s0 + static_cast<uintptr_t>(nblk) * BB;
      const uintptr_t as = s0 & ~uintptr_t(15), ae = (e0 + 15) & ~uintptr_t(15);
      src[i] = reinterpret_cast<const uint8_t*>(as);
      len[i] = static_cast<uint32_t>(ae - as);
      total += len[i];
    }
  }
  mbar_arrive_expect_tx(bar, total);
#pragma unroll
  for (int i = 0; i < TR; ++i)
    if (i < nrows) bulk_g2s(slot + i * a.slot_row_bytes, src[i], len[i], bar);
}

// Pre-bytes -> 4 weights -> two fp32x2 FMAs against 4 consecutive x values.
// f = 1 + q/2^k, so f - 1 is exact and w = (f - 1) A - Mm (A = 2^k d sc,
// Mm = dmin m, or 32 d sc for Q6_K) is the exact weight rounded once.
__device__ __forceinline__ float2 fma4(uint32_t pre, const float4& xv, float2 a, float2 mm, float2 s) {
  const float2 one = make_float2(-1.0f, -1.0f);
  const float2 w01 = ffma2(fadd2(make_float2(byte_to_f(pre, 0), byte_to_f(pre, 1)), one), a, mm);
  const float2 w23 = ffma2(fadd2(make_float2(byte_to_f(pre, 2), byte_to_f(pre, 3)), one), a, mm);
  s = ffma2(w01, make_float2(xv.x, xv.y), s);
  s = ffma2(w23, make_float2(xv.z, xv.w), s);
  return s;
}

// Q4_K: low nibble -> byte 0x80 | q (f = 1 + q/128); high -> 0x80 | q << 3 (f = 1 + q/16).
__device__ __forceinline__ uint32_t q4_lo(uint32_t w) { return (w & 0x0F0F0F0Fu) | 0x80808080u; }
__device__ __forceinline__ uint32_t q4_hi(uint32_t w) { return ((w >> 1) & 0x78787878u) | 0x80808080u; }
// Q5_K: the 5th bit of the low (high) nibble's code is bit 2c (2c+1) of each qh
// byte, rotated to bit 4; f = 1 + q/128 for both.
__device__ __forceinline__ uint32_t q5_lo(uint32_t w, uint32_t h, int c) {
  return (w & 0x0F0F0F0Fu) | (__funnelshift_l(h, h, (4 - 2 * c) & 31) & 0x10101010u) | 0x80808080u;
}
__device__ __forceinline__ uint32_t q5_hi(uint32_t w, uint32_t h, int c) {
  return ((w >> 4) & 0x0F0F0F0Fu) | (__funnelshift_l(h, h, (3 - 2 * c) & 31) & 0x10101010u) | 0x80808080u;
}
// Q6_K: 6-bit code = low nibble | (2 high bits) << 4; f = 1 + q/128.
__device__ __forceinline__ uint32_t q6_t0(uint32_t a, uint32_t h) { return (a & 0x0F0F0F0Fu) | ((h << 4) & 0x30303030u) | 0x80808080u; }
__device__ __forceinline__ uint32_t q6_t1(uint32_t b, uint32_t h) { return (b & 0x0F0F0F0Fu) | ((h << 2) & 0x30303030u) | 0x80808080u; }
__device__ __forceinline__ uint32_t q6_t2(uint32_t a, uint32_t h) { return ((a >> 4) & 0x0F0F0F0Fu) | (h & 0x30303030u) | 0x80808080u; }
__device__ __forceinline__ uint32_t q6_t3(uint32_t b, uint32_t h) { return ((b >> 4) & 0x0F0F0F0Fu) | ((h >> 2) & 0x30303030u) | 0x80808080u; }

// 16 bytes at a 2-byte aligned shared-memory address (five aligned words).
__device__ __forceinline__ uint4 lds16_a2(const uint8_t* p) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
  const uint32_t sh = static_cast<uint32_t>(a & 3) * 8;
  const uint32_t w0 = w[0], w1 = w[1], w2 = w[2], w3 = w[3], w4 = w[4];
  return make_uint4(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh), __funnelshift_r(w2, w3, sh),
                    __funnelshift_r(w3, w4, sh));
}

__device__ __forceinline__ float2 f2(float v) { return make_float2(v, v); }

__device__ __forceinline__ uint32_t word_of(const uint4& v, int w) {
  return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
}

// One block of R rows for quad lane c; `rem` = weights of the block inside K.
// acc[i][m] += sum_{part p} w*x over the lane's parts, each weight the exactly
// rounded fp32 value (parts past K have zero weights).
template <int QT, int R, int MT>
__device__ __forceinline__ void do_block(const uint8_t* const (&blk)[R], const bool (&rok)[R], int c, int rem,
                                         const float* xb, const float* Xb, int xstride, int Xstride, int M,
                                         float2 (&acc)[R][MT]) {
  constexpr int P = QuadFmt<QT>::P;
  constexpr int PL = QuadFmt<QT>::PL;
  float A[R][P], B[R][P];
  uint4 raw[R][4];
#pragma unroll
  for (int i = 0; i < R; ++i) {
    if (!rok[i]) continue;
    const uint8_t* b = blk[i];
    if constexpr (QT == T_Q6_K) {
      const int h = c >> 1, l0 = 16 * (c & 1);
      raw[i][0] = lds16_a2(b + 64 * h + l0);
      raw[i][1] = lds16_a2(b + 64 * h + 32 + l0);
      raw[i][2] = lds16_a2(b + 128 + 32 * h + l0);
      // scales 8h + 2t + (c&1), t = 0..3
      const uint2 s = ld8_a2(b + 192 + 8 * h + (c & 1));
      const uint32_t se = __byte_perm(s.x, s.y, 0x6420);
      const float d = half_bits_to_float(reinterpret_cast<const uint16_t*>(b + 208)[0]);
      const float dA = 128.0f * d, dB = -32.0f * d;
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const float sc = static_cast<float>(static_cast<int8_t>((se >> (8 * p)) & 0xFF));
        const bool ok = qpos<QT>(c, p) + PL <= rem;
        A[i][p] = ok ? dA * sc : 0.0f;
        B[i][p] = ok ? dB * sc : 0.0f;  // minus the subtracted constant
      }
    } else {
      const uint4 hdr = *reinterpret_cast<const uint4*>(b);
      constexpr int QS = kQ4Codes<QT> ? 16 : 48;
      raw[i][0] = *reinterpret_cast<const uint4*>(b + QS + 32 * c);
      raw[i][1] = *reinterpret_cast<const uint4*>(b + QS + 32 * c + 16);
      if constexpr (QT == T_Q5_K) {
        raw[i][2] = *reinterpret_cast<const uint4*>(b + 16);
        raw[i][3] = *reinterpret_cast<const uint4*>(b + 32);
      }
      // IA4: quad lane c's two parts are group c (sc = m = 1, d = scale, dmin = -bias)
      const uint32_t v = (QT == T_IA4) ? 0x01010101u : scale_min_bytes(hdr.y, hdr.z, hdr.w, c);
      const float d = (QT == T_IA4) ? ia4_scale(hdr, c) : half_bits_to_float(hdr.x & 0xFFFF);
      const float dmin = (QT == T_IA4) ? ia4_neg_bias(hdr, c) : half_bits_to_float(hdr.x >> 16);
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const float sS = (kQ4Codes<QT> && p == 1) ? 16.0f : 128.0f;
        const float av = (sS * d) * static_cast<float>((v >> (8 * p)) & 0xFF);
        const float mm = dmin * static_cast<float>((v >> (16 + 8 * p)) & 0xFF);
        const bool ok = qpos<QT>(c, p) + PL <= rem;
        A[i][p] = ok ? av : 0.0f;
        B[i][p] = ok ? -mm : 0.0f;
      }
    }
  }
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    if (m >= M) break;
    const float* xm = xb + m * xstride;
    float2 Sx[R][P];
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
      for (int p = 0; p < P; ++p) Sx[i][p] = make_float2(0.f, 0.f);
    if constexpr (QT == T_Q6_K) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        float4 xv[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) xv[t] = *reinterpret_cast<const float4*>(xm + qpos<QT>(c, t) + 4 * w);
#pragma unroll
        for (int i = 0; i < R; ++i) {
          if (!rok[i]) continue;
          const uint32_t a = word_of(raw[i][0], w), bq = word_of(raw[i][1], w), h = word_of(raw[i][2], w);
          Sx[i][0] = fma4(q6_t0(a, h), xv[0], f2(A[i][0]), f2(B[i][0]), Sx[i][0]);
          Sx[i][1] = fma4(q6_t1(bq, h), xv[1], f2(A[i][1]), f2(B[i][1]), Sx[i][1]);
          Sx[i][2] = fma4(q6_t2(a, h), xv[2], f2(A[i][2]), f2(B[i][2]), Sx[i][2]);
          Sx[i][3] = fma4(q6_t3(bq, h), xv[3], f2(A[i][3]), f2(B[i][3]), Sx[i][3]);
        }
      }
    } else {
      // the lane's 32 qs bytes = 8 words; word w holds weights l = 4w..4w+3 of both sub-blocks
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float4 xlo = *reinterpret_cast<const float4*>(xm + 64 * c + 4 * w);
        const float4 xhi = *reinterpret_cast<const float4*>(xm + 64 * c + 32 + 4 * w);
#pragma unroll
        for (int i = 0; i < R; ++i) {
          if (!rok[i]) continue;
          const uint32_t q = word_of(raw[i][w >> 2], w & 3);
          if constexpr (kQ4Codes<QT>) {
            Sx[i][0] = fma4(q4_lo(q), xlo, f2(A[i][0]), f2(B[i][0]), Sx[i][0]);
            Sx[i][1] = fma4(q4_hi(q), xhi, f2(A[i][1]), f2(B[i][1]), Sx[i][1]);
          } else {
            const uint32_t hb = word_of(raw[i][2 + (w >> 2)], w & 3);
            Sx[i][0] = fma4(q5_lo(q, hb, c), xlo, f2(A[i][0]), f2(B[i][0]), Sx[i][0]);
            Sx[i][1] = fma4(q5_hi(q, hb, c), xhi, f2(A[i][1]), f2(B[i][1]), Sx[i][1]);
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < R; ++i) {
      if (!rok[i]) continue;
#pragma unroll
      for (int p = 0; p < P; ++p) acc[i][m] = fadd2(acc[i][m], Sx[i][p]);
    }
  }
}

template <int QT, int R, int MT>
__global__ void __launch_bounds__(NW * 32, 1) gemv_kernel(const GemvArgs a) {
  constexpr int TR = 8 * R;
  constexpr int BB = Fmt<QT>::BYTES;
  constexpr int PL = QuadFmt<QT>::PL;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint8_t* ring = smem + BAR_BYTES;
  const int wlen = a.xblks * 256;
  float* xs = reinterpret_cast<float*>(ring + static_cast<size_t>(NW) * S * a.stage_bytes);
  float* Xs = xs + a.M * wlen;
  const int nr = a.r_end - a.r_begin;
  const bool direct = (nr == 1);  // one range per tile in this launch: write (or add onto) y directly
  float* part = Xs + a.M * (wlen / PL);  // [tiles_per_cta][TR][nr][M] when !direct
  int* cnt = reinterpret_cast<int*>(part + (direct ? 0 : a.tiles_per_cta * TR * nr * a.M));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = lane >> 2, c = lane & 3;
  uint64_t* wbar = bars + warp * S;
  uint8_t* wring = ring + static_cast<size_t>(warp) * S * a.stage_bytes;

  if (lane == 0)
    for (int s = 0; s < S; ++s) mbar_init(&wbar[s], 1);
  if (!direct)
    for (int t = threadIdx.x; t < a.tiles_per_cta; t += blockDim.x) cnt[t] = 0;
  fence_mbar_init();
  __syncthreads();

  // this CTA's tiles: blockIdx.x + i*gridDim.x; units u = i*nr + (range - r_begin)
  const int64_t my_tiles = (a.ntiles > blockIdx.x) ? (a.ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int64_t my_units = my_tiles * nr;
  auto unit_tile = [&](int64_t u) -> int64_t { return blockIdx.x + (u / nr) * static_cast<int64_t>(gridDim.x); };
  auto unit_range = [&](int64_t u) -> int { return a.r_begin + static_cast<int>(u % nr); };

  // producer state (lane 0): next job (unit pu, block offset pcb within its range)
  int64_t pu = warp;
  int pcb = 0;
  int64_t issued = 0;
  auto issue_next = [&]() {
    const int r = unit_range(pu);
    const int rlen = range_blocks(a, r);
    const int nblk = min(a.KC, rlen - pcb);
    issue_job<TR, BB>(a, unit_tile(pu), r * a.KB + pcb, nblk, wring + (issued % S) * a.stage_bytes,
                      &wbar[issued % S]);
    ++issued;
    pcb += nblk;
    if (pcb >= rlen) { pu += NW; pcb = 0; }
  };
  if (lane == 0)
    while (issued < S && pu < my_units) issue_next();

  pdl_wait();
  pdl_launch_dependents();
  stage_x<PL>(a, xs, Xs);

  bool failed = false;
  int64_t q = 0;  // jobs consumed
  int64_t q_fail = 0;
  for (int64_t u = warp; u < my_units; u += NW) {
    const int64_t tile = unit_tile(u);
    const int r = unit_range(u);
    const int rb0 = r * a.KB, rlen = range_blocks(a, r);
    float2 acc[R][MT];
    float racc[R][MT];
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
      for (int m = 0; m < MT; ++m) { acc[i][m] = make_float2(0.f, 0.f); racc[i][m] = 0.f; }
    bool rok[R];
#pragma unroll
    for (int i = 0; i < R; ++i) rok[i] = tile * TR + quad * R + i < a.N;

    for (int cb = 0; cb < rlen; cb += a.KC) {
      const int nblk = min(a.KC, rlen - cb);
      const int slot = static_cast<int>(q % S);
      uint8_t* sp = wring + slot * a.stage_bytes;
      if (!failed) {
        const bool ok = mbar_wait(&wbar[slot], static_cast<uint32_t>((q / S) & 1), a.err);
        failed = __any_sync(0xFFFFFFFFu, !ok);
        if (failed) q_fail = q;
      }
      if (!failed) {
        const uint8_t* rbase[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
          const int lr = quad * R + i;
          const uintptr_t s0 = reinterpret_cast<uintptr_t>(a.W + (tile * TR + lr) * a.row_bytes +
                                                           static_cast<int64_t>(rb0 + cb) * BB);
          rbase[i] = sp + lr * a.slot_row_bytes + (s0 & 15);
        }
        for (int bi = 0; bi < nblk; ++bi) {
          const int b = rb0 + cb + bi;
          const int rem = min(256, a.K - b * 256);
          const uint8_t* bp[R];
#pragma unroll
          for (int i = 0; i < R; ++i) bp[i] = rbase[i] + bi * BB;
          const int bw = b - a.xblk0;
          do_block<QT, R, MT>(bp, rok, c, rem, xs + bw * 256, Xs + bw * (256 / PL), wlen, wlen / PL, a.M, acc);
          const bool seg_end = ((b + 1 - rb0) % SEG == 0) || (cb + bi + 1 == rlen);
          if (seg_end) {
#pragma unroll
            for (int i = 0; i < R; ++i)
#pragma unroll
              for (int m = 0; m < MT; ++m) {
                if (m < a.M) {
                  float sg = __fadd_rn(acc[i][m].x, acc[i][m].y);
                  sg = __fadd_rn(sg, __shfl_xor_sync(0xFFFFFFFFu, sg, 2));
                  sg = __fadd_rn(sg, __shfl_xor_sync(0xFFFFFFFFu, sg, 1));
                  racc[i][m] = __fadd_rn(racc[i][m], sg);
                  acc[i][m] = make_float2(0.f, 0.f);
                }
              }
          }
        }
      }
      ++q;
      __syncwarp();
      if (lane == 0 && !failed && pu < my_units) {
        fence_proxy_async_smem();
        issue_next();
      }
    }
    if (failed) continue;
    const int64_t il = (tile - blockIdx.x) / gridDim.x;  // tile index within this CTA
    if (direct) {
      if (c == 0) {
#pragma unroll
        for (int i = 0; i < R; ++i) {
          const int64_t row = tile * TR + quad * R + i;
          if (row < a.N)
#pragma unroll
            for (int m = 0; m < MT; ++m)
              if (m < a.M) {
                float* dst = a.y + static_cast<int64_t>(m) * a.N + row;
                *dst = a.accumulate ? __fadd_rn(*dst, racc[i][m]) : racc[i][m];
              }
        }
      }
    } else {
      // publish this unit's partials; the tile's last finisher combines them in range order
      if (c == 0) {
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
          for (int m = 0; m < MT; ++m)
            if (m < a.M) part[((il * TR + quad * R + i) * nr + (r - a.r_begin)) * a.M + m] = racc[i][m];
      }
      __threadfence_block();
      __syncwarp();
      int last = 0;
      if (lane == 0) last = (atomicAdd(&cnt[il], 1) == nr - 1);
      last = __shfl_sync(0xFFFFFFFFu, last, 0);
      if (last) {
        __threadfence_block();
        for (int o = lane; o < TR * a.M; o += 32) {
          const int lr = o / a.M, m = o % a.M;
          const int64_t row = tile * TR + lr;
          if (row >= a.N) continue;
          const float* pp = part + ((il * TR + lr) * nr) * a.M + m;
          float* dst = a.y + static_cast<int64_t>(m) * a.N + row;
          float v = a.accumulate ? __fadd_rn(*dst, pp[0]) : pp[0];
          for (int rr = 1; rr < nr; ++rr) v = __fadd_rn(v, pp[rr * a.M]);
          *dst = v;
        }
      }
    }
  }
  // never leave while bulk copies into this CTA's shared memory are in flight
  if (failed && lane == 0) {
    for (int64_t rr = q_fail; rr < issued; ++rr)
      mbar_wait(&wbar[rr % S], static_cast<uint32_t>((rr / S) & 1), nullptr);
  }
}

template <int QT, int R, int MT>
cudaError_t launch_t(const GemvArgs& a, size_t smem, int grid, cudaStream_t st, bool pdl) {
  auto kern = gemv_kernel<QT, R, MT>;
  static bool smem_set[64] = {false};
  const int dev = current_device_id();
  if (!smem_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmemPerBlock);
    if (e != cudaSuccess) return e;
    smem_set[dev] = true;
  }
  if (smem > static_cast<size_t>(kMaxSmemPerBlock)) return cudaErrorInvalidConfiguration;
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
cudaError_t launch_q(const GemvArgs& a, int R, size_t smem, int grid, cudaStream_t st, bool pdl) {
  if (R == 2) return launch_t<QT, 2, 1>(a, smem, grid, st, pdl);  // only chosen for M == 1
  if (a.M <= 1) return launch_t<QT, 1, 1>(a, smem, grid, st, pdl);
  if (a.M <= 2) return launch_t<QT, 1, 2>(a, smem, grid, st, pdl);
  if (a.M <= 4) return launch_t<QT, 1, 4>(a, smem, grid, st, pdl);
  if (a.M <= 8) return launch_t<QT, 1, 8>(a, smem, grid, st, pdl);
  return launch_t<QT, 1, 16>(a, smem, grid, st, pdl);
}

// Shared memory of one launch over `nr_win` ranges whose x window has xblks blocks.
size_t gemv_smem(const GemvPlan& p, int qtype, int M, int nr_win, int xblks) {
  const int TR = 8 * p.R;
  const int PL = (qtype == T_Q6_K) ? 16 : 32;
  size_t s = BAR_BYTES + static_cast<size_t>(NW) * S * p.stage_bytes;
  s += static_cast<size_t>(M) * xblks * 256 * 4;         // x
  s += static_cast<size_t>(M) * xblks * (256 / PL) * 4;  // run sums
  if (nr_win > 1) s += static_cast<size_t>(p.tiles_per_cta) * TR * nr_win * M * 4 + p.tiles_per_cta * 4;
  return s;
}

}  // namespace

GemvPlan plan_gemv_batched(int qtype, int64_t N, int K, int M) {
  GemvPlan p = {};
  const int BB = block_bytes_of(qtype);
  p.nb = (K + 255) / 256;
  p.R = 1;  // two rows per quad spill at 128 registers
  const int TR = 8 * p.R;
  // K-ranges: enough units to give every warp of the machine work, and short
  // enough (KB <= KB_MAX) that one range of x fits in shared memory for any M.
  // Depends on (N, K) and the SM count only, so the summation order is the
  // same for every M.
  const int64_t tiles8 = (N + 7) / 8;
  const int64_t target = 2LL * num_sms() * NW;
  int64_t nr = (target + tiles8 - 1) / tiles8;
  const int max_nr = (p.nb + SEG - 1) / SEG;
  if (nr > max_nr) nr = max_nr;
  if (nr < 1) nr = 1;
  int KB = static_cast<int>((p.nb + nr - 1) / nr);
  KB = (KB + SEG - 1) / SEG * SEG;
  if (KB > KB_MAX) KB = KB_MAX;
  p.KB = KB;
  p.nranges = (p.nb + KB - 1) / KB;
  p.ntiles = (N + TR - 1) / TR;
  p.grid = static_cast<int>(min_i64(p.ntiles, num_sms()));
  p.tiles_per_cta = static_cast<int>((p.ntiles + p.grid - 1) / p.grid);
  // ring stage: TR rows x KC blocks (+32 bytes per row for unaligned Q6_K
  // segments); shrink KC until one range of x (M tokens) fits beside the rings
  const int row_slack = (qtype == T_Q6_K) ? 32 : 0;
  int kc = (STAGE_TARGET / TR - row_slack) / BB;
  if (kc < 1) kc = 1;
  if (kc > KB) kc = KB;
  for (;; --kc) {
    p.KC = kc;
    // row stride in the stage: a multiple of 16 bytes with an odd count of
    // 16-byte units, so the 16-byte loads of neighbouring rows fall in
    // different shared-memory banks
    int srb = (kc * BB + row_slack + 15) & ~15;
    if ((srb / 16) % 2 == 0) srb += 16;
    p.slot_row_bytes = srb;
    p.stage_bytes = TR * p.slot_row_bytes;
    if (kc == 1 || gemv_smem(p, qtype, M, 1, KB) <= static_cast<size_t>(kMaxSmemPerBlock)) break;
  }
  return p;
}

cudaError_t launch_gemv_batched(int qtype, const void* W, const void* x, int x_bf16, float* y, int64_t N, int K, int M,
                        cudaStream_t stream, bool pdl) {
  if (N == 0 || M == 0) return cudaSuccess;
  const GemvPlan p = plan_gemv_batched(qtype, N, K, M);
  GemvArgs a = {};
  a.W = static_cast<const uint8_t*>(W);
  a.N = N;
  a.K = K;
  a.nb = p.nb;
  a.row_bytes = static_cast<int64_t>(p.nb) * block_bytes_of(qtype);
  a.x = x;
  a.x_bf16 = x_bf16;
  a.M = M;
  a.y = y;
  a.err = device_error_ptr();
  a.KB = p.KB;
  a.nranges = p.nranges;
  a.KC = p.KC;
  a.slot_row_bytes = p.slot_row_bytes;
  a.stage_bytes = p.stage_bytes;
  a.ntiles = p.ntiles;
  a.tiles_per_cta = p.tiles_per_cta;
  // one launch per x window: as many whole K-ranges as fit in shared memory;
  // a later launch adds onto y, which continues the in-order range sum exactly
  int r0 = 0;
  while (r0 < p.nranges) {
    int r1 = p.nranges;
    for (;;) {
      const int xb0 = r0 * p.KB, xb1 = (r1 * p.KB < p.nb) ? r1 * p.KB : p.nb;
      if (gemv_smem(p, qtype, M, r1 - r0, xb1 - xb0) <= static_cast<size_t>(kMaxSmemPerBlock)) break;
      if (r1 - r0 == 1) return cudaErrorInvalidConfiguration;
      --r1;
    }
    a.r_begin = r0;
    a.r_end = r1;
    a.accumulate = (r0 > 0);
    a.xblk0 = r0 * p.KB;
    a.xblks = ((r1 * p.KB < p.nb) ? r1 * p.KB : p.nb) - a.xblk0;
    const size_t smem = gemv_smem(p, qtype, M, r1 - r0, a.xblks);
    cudaError_t e;
    switch (qtype) {
      case T_Q4_K: e = launch_q<T_Q4_K>(a, p.R, smem, p.grid, stream, pdl); break;
      case T_Q5_K: e = launch_q<T_Q5_K>(a, p.R, smem, p.grid, stream, pdl); break;
      case T_Q6_K: e = launch_q<T_Q6_K>(a, p.R, smem, p.grid, stream, pdl); break;
      case T_IA4: e = launch_q<T_IA4>(a, p.R, smem, p.grid, stream, pdl); break;
      default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    r0 = r1;
  }
  return cudaSuccess;
}

}  // namespace kq
