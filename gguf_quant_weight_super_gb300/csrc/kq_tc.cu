// kq_tc.cu -- products for M = 2..16 tokens (bf16 x) on the 5th-generation
// tensor cores:  y[m][n] = sum_k w[n][k] * x[m][k].
//
// "ANE Fieldfare" README, "Speculative decoding": verify blocks of up to 16
// tokens read every weight once for all of them.  "GGUF in transformers",
// "Reusing ggml's Metal kernels": weights stay packed in memory and are
// dequantized on the fly.
//
// With 16 tokens a CUDA-core product spends about half an instruction per
// weight per token; here the CUDA cores only dequantize (about two
// instructions per weight for any M) and tcgen05.mma does the products:
//  * one CTA per tile of 128 rows (the MMA's M) and K-part; a producer warp
//    streams the tile's raw blocks into a shared-memory ring, KC blocks of all
//    128 rows per stage: one 2-D tensor TMA copy (Q4_K, Q5_K; rows past N
//    are zero-filled) or one 1-D bulk copy per row segment (Q6_K, whose
//    210-byte blocks do not start on 16-byte boundaries);
//  * twelve dequantization warps in three groups of four: warp w owns TMEM
//    lane quarter w & 3 (one row per thread), group w >> 2 takes every third
//    256-weight block of the part; each weight is
//    computed in fp32 as w = d*sc*q - dmin*m (Q4_K, Q5_K) or d*sc*(q - 32)
//    (Q6_K), rounded once to bf16 and written with tcgen05.st straight into
//    tensor memory (A operand, 128 columns per block, ring of SA blocks);
//    the same warps copy the block's slice of x (bf16, rows m >= M zero) into
//    shared memory in the no-swizzle K-major core-matrix layout (B operand);
//  * one thread issues 16 MMAs (K = 16 each, M = 128, N = 16, fp32
//    accumulator in TMEM) per block and commits them to the block's "free"
//    barrier; after the last block the accumulator is read back with
//    tcgen05.ld (one row per thread, one column per token) and written to y.
// Precision: each weight is rounded once to bf16 (relative error <= 2^-9),
// so |y - y_exact| <= 2^-9 * sum_k |w x| plus fp32 accumulation error; bf16 x
// is exact in the MMA.  This path therefore serves bf16 x only (tolerance
// 4e-3 of sum |w x|); fp32 x stays on the CUDA cores.
#include <cuda.h>

#include "kq_lane.cuh"

namespace kq {

using namespace lane;

namespace {

constexpr int TR = 128;                     // rows per tile (MMA M)
constexpr int TN = 16;                      // MMA N: tokens, zero padded
constexpr int NDQ = 12;                     // dequantization warps
constexpr int NGRP = NDQ / 4;               // groups of four (one TMEM lane quarter per warp)
constexpr int NTH_TC = (NDQ + 2) * 32;      // + producer warp + MMA warp
constexpr int SRAW_MAX = 4;                 // raw ring stages at most
constexpr int SA = NGRP;                    // A/B stages (one 256-weight block each): stage g is group g's
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t A_COL0 = 128;            // A stage s: TMEM columns A_COL0 + 128 s
constexpr int B_STAGE_BYTES = 2 * 32 * 128; // 16 rows x 256 bf16 (2 row groups x 32 core matrices)
constexpr int HDR_BYTES = 256;

struct TcArgs {
  CUtensorMap tmap;   // W as [N rows][row_bytes/4] uint32, box [KC*BB/4][128] (when use_tmap)
  int use_tmap;
  const uint8_t* W;
  const uint16_t* x;  // bf16 [M][K]
  float* y;           // [M][N]
  int64_t N, row_bytes;
  int K, nb, M, type;
  int KC;    // blocks per raw stage
  int srb;   // raw row stride in shared memory
  int Sraw;  // raw stages
  int KS;    // K-parts = cluster size (partial accumulators added through DSMEM)
  int kpb;   // blocks per K-part
  int* err;
};

// Shared-memory matrix descriptor: no swizzle, K-major core matrices of
// 8 rows x 16 bytes; lbo = byte step between core matrices along K, sbo =
// along M/N; bits 46-47 = 1 (descriptor version for this architecture).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFF) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32) | (static_cast<uint64_t>(1) << 46);
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N = 16, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(TN >> 3) << 17) |
                            (static_cast<uint32_t>(TR >> 4) << 24);

// fp32 value 0.5 + byte/2^(8+8*pos) from a byte of v (PRMT into a float's mantissa):
// pos 2: 0.5 + b/256; pos 1: 0.5 + b/65536.
__device__ __forceinline__ float byte_float(uint32_t v, int t, int pos) {
  const uint32_t sel = (pos == 2) ? (4u | (4u << 4) | (static_cast<uint32_t>(t) << 8) | (7u << 12))
                                  : (4u | (static_cast<uint32_t>(t) << 4) | (4u << 8) | (7u << 12));
  return __uint_as_float(__byte_perm(v, 0x3F000000u, sel));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Four weights (bytes t = 0..3 of v, placed at byte position pos) as two
// packed bf16 pairs.  With f = 0.5 + q/2^k and A = 2^k d sc the weight is
// w = f A - (A/2 + Mt) (Mt = dmin m; 0 for Q6_K's offset form).  When
// A/2 + Mt is exact in fp32 (exact_c) that is one fma, rounded once;
// otherwise (d and dmin far apart in exponent) w = (f - 0.5) A - Mt, where
// f - 0.5 = q/2^k is exact: rounded once as well.  Then one rounding to bf16.
__device__ __forceinline__ void four_weights(uint32_t v, int pos, float A, float Mt, bool exact_c, uint32_t& p0,
                                             uint32_t& p1) {
  const float2 a = make_float2(A, A);
  float2 f01 = make_float2(byte_float(v, 0, pos), byte_float(v, 1, pos));
  float2 f23 = make_float2(byte_float(v, 2, pos), byte_float(v, 3, pos));
  float2 c;
  if (exact_c) {
    const float C = -(0.5f * A + Mt);
    c = make_float2(C, C);
  } else {
    const float2 h = make_float2(-0.5f, -0.5f);
    f01 = fadd2(f01, h);
    f23 = fadd2(f23, h);
    c = make_float2(-Mt, -Mt);
  }
  const float2 w01 = ffma2(f01, a, c), w23 = ffma2(f23, a, c);
  p0 = pack_bf16(w01.x, w01.y);
  p1 = pack_bf16(w23.x, w23.y);
}
// Whether a + b is exact in fp32 (the TwoSum error term is zero).
__device__ __forceinline__ bool sum_exact(float a, float b) {
  const float s = __fadd_rn(a, b), bb = __fsub_rn(s, a), aa = __fsub_rn(s, bb);
  return __fadd_rn(__fsub_rn(a, aa), __fsub_rn(b, bb)) == 0.0f;
}

// Half g (weights 128g .. 128g+127) of the block at bp (shared address) of
// this thread's row, as bf16 pairs into TMEM columns [taddr, taddr + 64).
template <int QT>
__device__ __forceinline__ void dequant_half(uint32_t bp, int g, uint32_t taddr) {
  uint32_t col[16];
  if constexpr (QT != T_Q6_K) {
    const uint4 hdr = lds128(bp);
    const float d = half_bits_to_float(hdr.x & 0xFFFF), dmin = half_bits_to_float(hdr.x >> 16);
    // scales and mins of sub-blocks 4g .. 4g+3 (bytes)
    uint32_t scb, mb;
    if (g == 0) {
      scb = hdr.y & 0x3F3F3F3Fu;
      mb = hdr.z & 0x3F3F3F3Fu;
    } else {
      scb = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
      mb = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
    }
    constexpr int QS = kQ4Codes<QT> ? 16 : 48;
    uint4 qh0 = make_uint4(0, 0, 0, 0), qh1 = qh0;
    if constexpr (QT == T_Q5_K) { qh0 = lds128(bp + 16); qh1 = lds128(bp + 32); }
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {  // chunk c = 2g + cc: sub-blocks 2c (low nibbles), 2c+1 (high)
      const int c = 2 * g + cc;
      float dsl, dml, dsh, dmh;
      if constexpr (QT == T_IA4) {  // chunk c is group c: one scale and one bias for both sub-blocks
        dsl = dsh = ia4_scale(hdr, c);
        dml = dmh = ia4_neg_bias(hdr, c);
      } else {
        dsl = d * static_cast<float>((scb >> (16 * cc)) & 0xFF);
        dml = dmin * static_cast<float>((mb >> (16 * cc)) & 0xFF);
        dsh = d * static_cast<float>((scb >> (16 * cc + 8)) & 0xFF);
        dmh = dmin * static_cast<float>((mb >> (16 * cc + 8)) & 0xFF);
      }
      const uint4 qa = lds128(bp + QS + 32 * c), qb = lds128(bp + QS + 32 * c + 16);
      // Q4_K high nibbles sit at byte position 1 (f = 0.5 + q/4096): A = 4096 d sc
      const float Al = 256.0f * dsl, Ah = (kQ4Codes<QT> ? 4096.0f : 256.0f) * dsh;
      const bool exl = sum_exact(0.5f * Al, dml), exh = sum_exact(0.5f * Ah, dmh);
#pragma unroll
      for (int part = 0; part < 2; ++part) {  // 0: low nibbles, 1: high nibbles
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          const uint32_t q = (w < 4) ? w4(qa, w) : w4(qb, w - 4);
          if constexpr (kQ4Codes<QT>) {
            if (part == 0) {
              // 0.5 + q/256, q in 0..15:  w = f*(256 d sc) - (128 d sc + dmin m)
              four_weights(q & 0x0F0F0F0Fu, 2, Al, dml, exl, col[2 * w], col[2 * w + 1]);
            } else {
              // 16q in byte position 1: f = 0.5 + 16q/65536 = 0.5 + q/4096
              four_weights(q & 0xF0F0F0F0u, 1, Ah, dmh, exh, col[2 * w], col[2 * w + 1]);
            }
          } else {
            const uint32_t hb = (w < 4) ? w4(qh0, w) : w4(qh1, w - 4);
            uint32_t v;
            if (part == 0) v = (q & 0x0F0F0F0Fu) | (((hb >> (2 * c)) & 0x01010101u) << 4);
            else v = ((q >> 4) & 0x0F0F0F0Fu) | (((hb >> (2 * c + 1)) & 0x01010101u) << 4);
            four_weights(v, 2, part ? Ah : Al, part ? dmh : dml, part ? exh : exl, col[2 * w], col[2 * w + 1]);
          }
        }
        tmem_st16(taddr + 32 * cc + 16 * part, col);
      }
    }
  } else {  // Q6_K: half g is 128-half h = g
    const int h = g;
    const float d = half_bits_to_float(lds16(bp + 208));
    const uint2 sv = lds8_a2(bp + 192 + 8 * h);  // scales 8h .. 8h+7
    float ds[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) ds[i] = d * static_cast<float>(sbyte(i < 4 ? sv.x : sv.y, i & 3));
    uint4 ql[4], qh[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) ql[i] = lds16_a2(bp + 64 * h + 16 * i);
#pragma unroll
    for (int i = 0; i < 2; ++i) qh[i] = lds16_a2(bp + 128 + 32 * h + 16 * i);
#pragma unroll
    for (int p = 0; p < 4; ++p) {  // weights 128h + 32p + l, l = 0..31
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const uint32_t a = w4(ql[w >> 2], w & 3), b = w4(ql[2 + (w >> 2)], w & 3), hv = w4(qh[w >> 2], w & 3);
        uint32_t v;
        if (p == 0) v = (a & 0x0F0F0F0Fu) | ((hv << 4) & 0x30303030u);
        else if (p == 1) v = (b & 0x0F0F0F0Fu) | ((hv << 2) & 0x30303030u);
        else if (p == 2) v = ((a >> 4) & 0x0F0F0F0Fu) | (hv & 0x30303030u);
        else v = ((b >> 4) & 0x0F0F0F0Fu) | ((hv >> 2) & 0x30303030u);
        const float A = ds[2 * p + (w >> 2)];
        // 0.5 + q/256, q in 0..63:  w = f*(256 d sc) - 160 d sc  ( = d sc (q - 32); 160 d sc is exact)
        four_weights(v, 2, 256.0f * A, 32.0f * A, true, col[2 * (w & 7)], col[2 * (w & 7) + 1]);
      }
      tmem_st16(taddr + 16 * p, col);
    }
  }
}

// This block's x: 16 tokens x 256 values = 512 chunks of 16 bytes over the
// 128 threads of a group (rows m >= M are zero).
__device__ __forceinline__ void load_b(const TcArgs& a, int blk, int t128, uint4 (&v)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int u = t128 + 128 * i;
    const int n = u & 15, kc = u >> 4;  // token, 8-value chunk within the block (tokens vary fastest:
                                        // 8 neighbouring threads store 8 consecutive 16-byte rows)
    const int k = 256 * blk + 8 * kc;
    v[i] = make_uint4(0, 0, 0, 0);
    if (n < a.M && k < a.K) v[i] = *reinterpret_cast<const uint4*>(a.x + static_cast<int64_t>(n) * a.K + k);
  }
}
// ... stored in the no-swizzle K-major core-matrix layout of the B stage.
__device__ __forceinline__ void store_b(int t128, const uint4 (&v)[4], uint8_t* bstage) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int u = t128 + 128 * i;
    const int n = u & 15, kc = u >> 4;
    *reinterpret_cast<uint4*>(bstage + kc * 128 + (n >> 3) * 4096 + (n & 7) * 16) = v[i];
  }
}

template <int QT>
__global__ void __launch_bounds__(NTH_TC, 1) tc_kernel(const __grid_constant__ TcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* raw_full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* raw_empty = raw_full + SRAW_MAX;
  uint64_t* a_full = raw_empty + SRAW_MAX;
  uint64_t* a_empty = a_full + SA;
  uint64_t* d_full = a_empty + SA;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(d_full + 1);
  uint8_t* bring = smem + HDR_BYTES;
  uint8_t* raw = bring + SA * B_STAGE_BYTES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kp = static_cast<int>(blockIdx.x) % a.KS;  // = cluster rank
  const int64_t row0 = static_cast<int64_t>(blockIdx.x / a.KS) * TR;
  const int kb0 = kp * a.kpb;
  const int nbk = max(0, min(a.nb, kb0 + a.kpb) - kb0);  // blocks of this K-part
  constexpr int BB = Fmt<QT>::BYTES;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SRAW_MAX; ++s) { mbar_init(&raw_full[s], 1); mbar_init(&raw_empty[s], NDQ); }
    for (int s = 0; s < SA; ++s) { mbar_init(&a_full[s], 4); mbar_init(&a_empty[s], 1); }
    mbar_init(d_full, 1);
    fence_mbar_init();
  }
  if (warp == 0) { tmem_alloc(tmem_slot, TMEM_COLS); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const int nst = (nbk + a.KC - 1) / a.KC;

  if (warp == NDQ) {
    // ------------------------------------------------------------- producer
    pdl_launch_dependents();
    const uint64_t pol = l2_evict_first_policy();  // the weights are read once per launch
    bool failed = false;
    for (int k = 0; k < nst && !failed; ++k) {
      const int slot = k % a.Sraw;
      if (k >= a.Sraw) {
        const bool ok = mbar_wait(&raw_empty[slot], static_cast<uint32_t>((k / a.Sraw - 1) & 1), a.err);
        if (!__all_sync(0xFFFFFFFFu, ok)) { failed = true; break; }
      }
      const int b0 = kb0 + k * a.KC, n = min(a.KC, kb0 + nbk - b0);
      uint8_t* sp = raw + static_cast<size_t>(slot) * TR * a.srb;
      if (a.use_tmap) {
        if (lane == 0) {
          mbar_arrive_expect_tx(&raw_full[slot], static_cast<uint32_t>(TR * a.srb));
          asm volatile(
              "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
              "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(sp)),
              "l"(reinterpret_cast<uint64_t>(&a.tmap)), "r"(b0 * BB / 4), "r"(static_cast<int>(row0)),
              "r"(smem_u32(&raw_full[slot])), "l"(pol)
              : "memory");
        }
        __syncwarp();
        continue;
      }
      uint32_t len[4];
      const uint8_t* src[4];
      uint32_t tot = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = lane + 32 * i;
        len[i] = 0;
        src[i] = nullptr;
        if (row0 + r < a.N) {
          const uintptr_t s0 = reinterpret_cast<uintptr_t>(a.W + (row0 + r) * a.row_bytes + static_cast<int64_t>(b0) * BB);
          const uintptr_t as = s0 & ~uintptr_t(15), ae = (s0 + static_cast<uintptr_t>(n) * BB + 15) & ~uintptr_t(15);
          src[i] = reinterpret_cast<const uint8_t*>(as);
          len[i] = static_cast<uint32_t>(ae - as);
          tot += len[i];
        }
      }
      tot = __reduce_add_sync(0xFFFFFFFFu, tot);
      if (lane == 0) mbar_arrive_expect_tx(&raw_full[slot], tot);
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (len[i]) bulk_g2s_hint(sp + (lane + 32 * i) * a.srb, src[i], len[i], &raw_full[slot], pol);
    }
    if (lane == 0)  // leave only after the copies in flight have landed (bounded)
      for (int k = (nst > a.Sraw ? nst - a.Sraw : 0); k < nst; ++k)
        mbar_wait(&raw_full[k % a.Sraw], static_cast<uint32_t>((k / a.Sraw) & 1), nullptr);
  } else if (warp == NDQ + 1) {
    // ------------------------------------------------------------ MMA issue
    bool failed = false;
    if (lane == 0) {
      for (int j = 0; j < nbk; ++j) {
        const int sa = j % SA;
        if (!failed) failed = !mbar_wait(&a_full[sa], static_cast<uint32_t>((j / SA) & 1), a.err);
        tc_fence_after();
        if (!failed) {
          const uint32_t bs = smem_u32(bring + sa * B_STAGE_BYTES);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            tc_mma_ts(tbase, tbase + A_COL0 + 128 * sa + 8 * i, smem_desc(bs + 256 * i, 128, 4096), kIdesc,
                      (j | i) != 0);
        }
        tc_commit(&a_empty[sa]);  // the block's A and B stage may be refilled once its MMAs complete
      }
      tc_commit(d_full);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------- dequantization warps
    pdl_wait();  // x is written by earlier kernels
    const int q = warp & 3, g = warp >> 2;
    const int r = 32 * q + lane;          // row in tile (= TMEM lane)
    const int t128 = 32 * q + lane;       // thread index within the group
    bool failed = false;
    uint4 xb[4];
    if (g < nbk) load_b(a, kb0 + g, t128, xb);  // x of the group's first block; later ones one block ahead
    for (int k = 0; k < nst; ++k) {
      const int slot = k % a.Sraw;
      if (!failed) {
        const bool ok = mbar_wait(&raw_full[slot], static_cast<uint32_t>((k / a.Sraw) & 1), a.err);
        failed = !__all_sync(0xFFFFFFFFu, ok);
      }
      const int b0 = kb0 + k * a.KC, n = min(a.KC, kb0 + nbk - b0);
      uint32_t rowp = smem_u32(raw + static_cast<size_t>(slot) * TR * a.srb + r * a.srb);
      if (!a.use_tmap)
        rowp += static_cast<uint32_t>(reinterpret_cast<uintptr_t>(a.W + (row0 + r) * a.row_bytes +
                                                                  static_cast<int64_t>(b0) * BB) & 15);
      for (int bi = 0; bi < n; ++bi) {
        const int j = k * a.KC + bi;  // block within the part
        if (j % NGRP != g) continue;
        const int sa = g;
        uint4 xn[4];
        if (j + NGRP < nbk) load_b(a, kb0 + j + NGRP, t128, xn);
        if (j >= NGRP && !failed) {
          const bool ok = mbar_wait(&a_empty[sa], static_cast<uint32_t>((j / NGRP - 1) & 1), a.err);
          failed = !__all_sync(0xFFFFFFFFu, ok);
        }
        tc_fence_after();
        if (!failed) {
          // rows past N dequantize zeros or stale shared memory; their outputs are never written
          const uint32_t ta = tbase + (static_cast<uint32_t>(32 * q) << 16) + A_COL0 + 128 * sa;
          dequant_half<QT>(rowp + bi * BB, 0, ta);
          dequant_half<QT>(rowp + bi * BB, 1, ta + 64);
          store_b(t128, xb, bring + sa * B_STAGE_BYTES);
        }
        tmem_wait_st();
        fence_proxy_async_smem();  // B writes -> visible to the tensor core
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[sa]);
#pragma unroll
        for (int i = 0; i < 4; ++i) xb[i] = xn[i];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&raw_empty[slot]);
    }
    // ------------------------------------------------------------- epilogue
    if (g == 0) {
      const bool ok = !failed && (nbk == 0 || mbar_wait(d_full, 0, a.err));
      tc_fence_after();
      uint32_t v[16];
      tmem_ld16(tbase + (static_cast<uint32_t>(32 * q) << 16), v);
      tmem_wait_ld();
      if (nbk == 0 || !ok)
        for (int m = 0; m < 16; ++m) v[m] = 0;  // an empty K-part adds nothing
      if (a.KS == 1) {
        const int64_t row = row0 + r;
        if (ok && row < a.N)
          for (int m = 0; m < a.M; ++m) a.y[static_cast<int64_t>(m) * a.N + row] = __uint_as_float(v[m]);
      } else {
        // this K-part's 128 x 16 partial sums, in the (now idle) B ring
        float4* red = reinterpret_cast<float4*>(bring) + r * 4;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          red[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                               __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
      }
    }
  }
  if (a.KS > 1) {
    // K-parts of a tile form one cluster: rank 0 adds the partials in rank order
    cluster_sync();
    if (kp == 0 && warp < 4) {
      const int r = 32 * warp + lane;
      const int64_t row = row0 + r;
      const uint32_t mine = smem_u32(bring) + 64 * r;
      float s[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) s[i] = 0.0f;
      for (int rk = 0; rk < a.KS; ++rk) {
        const uint32_t src = cluster_map(mine, rk);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 t = ld_cluster_f4(src + 16 * i);
          s[4 * i] = __fadd_rn(s[4 * i], t.x);
          s[4 * i + 1] = __fadd_rn(s[4 * i + 1], t.y);
          s[4 * i + 2] = __fadd_rn(s[4 * i + 2], t.z);
          s[4 * i + 3] = __fadd_rn(s[4 * i + 3], t.w);
        }
      }
      if (row < a.N)
        for (int m = 0; m < a.M; ++m) a.y[static_cast<int64_t>(m) * a.N + row] = s[m];
    }
    cluster_sync();  // peers keep their shared memory until rank 0 has read it
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, TMEM_COLS);
  }
}

size_t tc_smem(int srb, int Sraw) {
  const size_t b = HDR_BYTES + SA * B_STAGE_BYTES + static_cast<size_t>(Sraw) * TR * srb;
  return b < 120 * 1024 ? 120 * 1024 : b;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no
// link-time dependency on the driver library); encodings cached per weight.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool encode_tmap(CUtensorMap& m, const void* W, int64_t N, int64_t row_bytes, int box_bytes) {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  if (!fn) return false;
  struct Entry { const void* W; int64_t N, row_bytes; int box; CUtensorMap m; };
  static thread_local Entry cache[32];
  static thread_local int next = 0;
  for (auto& e : cache)
    if (e.W == W && e.N == N && e.row_bytes == row_bytes && e.box == box_bytes) { m = e.m; return true; }
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes / 4), static_cast<cuuint64_t>(N)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_bytes / 4), static_cast<cuuint32_t>(TR)};
  const cuuint32_t estr[2] = {1, 1};
  if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(W), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  cache[next] = {W, N, row_bytes, box_bytes, m};
  next = (next + 1) % 32;
  return true;
}

}  // namespace

bool tc_supported(int qtype, int64_t N, int K, int M) {
  return block_bytes_of(qtype) && M >= 2 && M <= TN && N >= 1 && K >= 32 && K % 32 == 0;
}

cudaError_t launch_tc(int qtype, const void* W, const void* x, float* y, int64_t N, int K, int M,
                      cudaStream_t stream, bool pdl) {
  if (!tc_supported(qtype, N, K, M)) return cudaErrorNotSupported;
  TcArgs a = {};
  a.W = static_cast<const uint8_t*>(W);
  a.x = static_cast<const uint16_t*>(x);
  a.y = y;
  a.N = N;
  a.K = K;
  a.nb = (K + 255) / 256;
  a.M = M;
  a.type = qtype;
  const int BB = block_bytes_of(qtype);
  a.row_bytes = static_cast<int64_t>(a.nb) * BB;
  a.err = device_error_ptr();
  // raw stages: KC blocks of all 128 rows.  Q4_K/Q5_K rows are 16-byte
  // multiples: one tensor copy per stage, rows packed at KC*BB (an odd number
  // of 16-byte units for odd KC: conflict-free row-per-thread reads).  Q6_K:
  // one copy per row segment (16-byte aligned superset plus slack), rows at
  // an odd number of 16-byte units.
  a.use_tmap = 0;
  size_t smem = 0;
  bool fit = false;
  for (int pass = 0; pass < 2 && !fit; ++pass) {
    // tensor copies need every stage start (b0*BB bytes) and width (KC*BB) to be
    // 16-byte multiples: only block sizes that are (144, 176; not Q6_K's 210)
    const bool tm = (pass == 0) && (BB % 16 == 0);
    if (pass == 0 && !tm) continue;
    for (int KC = 5; KC >= 1 && !fit; KC -= (tm ? 2 : 1)) {
      if (tm && KC * BB / 4 > 256) continue;
      int srb = KC * BB;
      if (!tm) {
        srb = (KC * BB + 15 + 16 + 15) & ~15;
        if ((srb / 16) % 2 == 0) srb += 16;
      }
      for (int S = SRAW_MAX; S >= 2 && !fit; --S) {
        smem = tc_smem(srb, S);
        if (smem <= static_cast<size_t>(kMaxSmemPerBlock)) {
          if (tm && !encode_tmap(a.tmap, W, N, a.row_bytes, KC * BB)) break;
          a.KC = KC; a.srb = srb; a.Sraw = S; a.use_tmap = tm ? 1 : 0; fit = true;
        }
      }
    }
  }
  if (!fit) return cudaErrorNotSupported;
  // K-parts (clusters of up to 8 CTAs): fewest waves x (blocks per CTA + the
  // per-CTA start-up, worth about 8 blocks: first raw stage, TMEM, epilogue)
  const int G = num_sms();
  const int64_t ntiles = (N + TR - 1) / TR;
  int64_t best = -1;
  for (int ks = 1; ks <= 8; ks *= 2) {
    const int kpb = (a.nb + ks - 1) / ks;
    if (ks > 1 && (ks - 1) * kpb >= a.nb) break;
    const int64_t cost = ((ntiles * ks + G - 1) / G) * (kpb + 8);
    if (best < 0 || cost < best) { best = cost; a.KS = ks; a.kpb = kpb; }
  }
  const void* fn = nullptr;
  switch (qtype) {
    case T_Q4_K: fn = reinterpret_cast<const void*>(tc_kernel<T_Q4_K>); break;
    case T_Q5_K: fn = reinterpret_cast<const void*>(tc_kernel<T_Q5_K>); break;
    case T_Q6_K: fn = reinterpret_cast<const void*>(tc_kernel<T_Q6_K>); break;
    case T_IA4: fn = reinterpret_cast<const void*>(tc_kernel<T_IA4>); break;
    default: return cudaErrorInvalidValue;
  }
  static bool smem_set[64][8] = {};
  const int dev = current_device_id();
  if (!smem_set[dev][qtype]) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmemPerBlock);
    if (e != cudaSuccess) return e;
    smem_set[dev][qtype] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ntiles * a.KS));
  cfg.blockDim = dim3(NTH_TC);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = static_cast<unsigned>(a.KS);
  attr[na].val.clusterDim.y = 1;
  attr[na].val.clusterDim.z = 1;
  ++na;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  void* args[] = {&a};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace kq
