// kq_gemv_kernel.cuh -- one-token products y = W x (M = 1; also M = 2..4 with bf16 x)
// against Q4_K / Q5_K / Q6_K rows: a single matrix, or a program of matrices
// run by one persistent launch.
//
// "GGUF in transformers", section "Reusing ggml's Metal kernels": decode-time
// products read the packed super-blocks directly and dequantize on the fly;
// section "Keeping the CPU and GPU working together": the device should not
// idle between the operations of a decode step.
//
// Arithmetic (exact integer products; see kq_lane.cuh):
//  * x is staged into shared memory as an exact image: for every block of 256
//    values a power-of-two scale s = 2^(e-22), e the binary exponent of the
//    block's largest |x|; values on that grid (every bf16 value within 2^15 of
//    the block maximum) as 24-bit integers m = x/s in three byte limbs, the
//    others listed beside the block (index and bf16 value; past 32 of them the
//    block keeps all 256 values as bf16).  fp32 x is staged as two such
//    images, hi = bf16(x) and lo = bf16(x - hi);
//  * a lane owns a 64-weight chunk or a 128-weight half of a block; codes
//    times limbs are summed exactly by dp4a and the lane's contribution
//        Q4_K/Q5_K:  y += s * (d * sum_p sc_p*T_p  -  dmin * sum_p m_p*X_p)
//        Q6_K:       y += s * d * sum_p sc_p*(T_p - 32*X_p)
//    (T_p = sum q*m, X_p = sum m over part p) is formed from exact integers
//    and rounded to fp32 within a proven bound (combine45_checked); listed and
//    kept values add fl(w*x) with w the exactly rounded fp32 weight.

// Execution (GB300: 152 SMs, 227 KB shared memory per CTA):
//  * one CTA per SM: a producer warp and NC consumer warps;
//  * the producer walks the CTA's units -- (tile of TT rows, K-part) of every
//    op, in op order -- and keeps a CTA-wide ring of S shared-memory slots
//    full with 1-D TMA bulk copies: one copy per stage when a stage holds
//    whole rows, else one copy per row segment of KC blocks, all with an L2
//    evict-first policy (weights are read once; activations stay in L2).
//    Weights never depend on earlier ops, so the producer runs ahead across
//    op boundaries;
//  * a stage's blocks are dealt to the consumer warps round-robin (continuing
//    across stages); quad q of a warp owns the tile rows q, q+8, ... (R of
//    them: a tile is 8R rows), so one x slice, loaded once per block, serves
//    R rows; a unit's row sums are added over the quad's lanes by shuffles and
//    over the warps in warp order by the unit's last warp (deterministic);
//  * in a program with grid barriers a tile's K may be split across CTAs: the
//    parts' row sums go to the workspace and are added in part order, each CTA
//    for its slice of rows, before the barrier that follows the one after
//    which they are complete (or after a final barrier);
//  * an op flagged "wait for previous" starts with a grid barrier (all CTAs
//    resident: cooperative launch) before its x is read; single products
//    instead use programmatic dependent launch, streaming weights before
//    griddepcontrol.wait.
#pragma once

#include <algorithm>
#include <vector>

#include "kq_lane.cuh"

namespace kq {

using namespace lane;

namespace {

#ifndef KQ_NC
#define KQ_NC 11
#endif
// Built with KQ_TIMELINE (the timeline library only; see build.py): thread 0
// of every CTA records the global timer at four points of every program op --
// 0 grid barrier passed, 1 x staged, 3 arriving at the barrier before the op
// (the previous ops' work done) -- for the first kTlCtas CTAs and kTlOps ops.
#ifdef KQ_TIMELINE
constexpr int kTlCtas = 160, kTlOps = 512;
__device__ unsigned long long g_kq_timeline[kTlCtas * kTlOps * 4];
__device__ __forceinline__ void tl_mark(int oi, int k) {
  if (threadIdx.x == 0 && blockIdx.x < kTlCtas && oi < kTlOps) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    g_kq_timeline[(blockIdx.x * kTlOps + oi) * 4 + k] = t;
  }
}
#define KQ_TL(oi, k) tl_mark((oi), (k))
#else
#define KQ_TL(oi, k) ((void)0)
#endif
constexpr int NC = KQ_NC;              // consumer warps (+1 producer: 12 warps, three warpgroups, 170 registers a thread)
constexpr int TT = 32;                 // rows per tile (4 per quad)
constexpr int NTHC = NC * 32;          // consumer threads
constexpr int NTH = NTHC + 32;         // + one producer warp
constexpr int RING_MAX = 8;                // ring slots at most
constexpr int CONSUMER_BAR = 1;        // named barrier of the consumer warps
constexpr int MAX_NB = 64;             // K <= 16384
// Shared memory header: full and empty mbarriers (RING_MAX each) and the
// reduction counters (RING_MAX + 1).
constexpr int kHdrBytes = 512;
static_assert(16 * RING_MAX + 4 * (RING_MAX + 1) <= kHdrBytes, "header");
constexpr int kMaxTokens1 = 4;         // tokens of one single-product launch (bf16 x when more than one)
// Largest stage (32 row segments): 48 KB keeps a ring of at least 4 slots.
constexpr int64_t kSlotCap = 48 * 1024;
// Largest stage of whole rows (one bulk copy), by rows per quad: a taller
// tile (more x reuse) may take a larger stage and a shorter ring.
__host__ __device__ constexpr int64_t whole_cap(int R) { return R >= 4 ? 72 * 1024 : R == 2 ? 56 * 1024 : 48 * 1024; }

}  // namespace

// Device op descriptor (geometry computed on the host).
struct KqOp {
  const uint8_t* W;
  const void* x;
  float* y;
  float* part;       // split K: partial row sums [KS][ntiles*TT] (workspace), else null
  int32_t R;         // rows per quad: a tile is 8R rows (programs: R = 4)
  int32_t contig;    // stages are whole rows, copied as one block (row stride in a stage = row_bytes)
  int64_t N;
  int64_t row_bytes;
  int32_t K, nb, type, x_bf16;
  int32_t KS, kpb;   // K-parts per tile, blocks per K-part
  int32_t KC;        // blocks per stage
  int32_t srb;       // row stride inside a stage
  int32_t ntiles, nunits, rot;
  int32_t flags;     // OP_WAIT: grid barrier first; OP_NEWX: stage x
  // first op of an x (OP_NEWX or OP_WAIT) in a program: per CTA the blocks
  // [lo, hi) of x its units in the ops sharing that x read (lo | hi << 16),
  // or null (all of x)
  const int32_t* xrange;
};
enum : int32_t { OP_WAIT = 1, OP_NEWX = 2 };

struct ProgArgs {
  const KqOp* ops;   // program in global memory (PROG) ...
  KqOp op0;          // ... or the single op
  int n_ops;
  int S, slot;       // ring slots, slot bytes
  int nb_max, nimg;  // blocks per row and x images the shared memory holds
  int* barrier;      // grid barrier arrivals (programs with OP_WAIT), zero at launch
  int* err;
  int final_fix;     // split-K sums remain after the last op: final grid barrier
};

namespace {

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(CONSUMER_BAR), "n"(NTHC) : "memory");
}

// ------------------------------------------------------------ work walk
// Unit k of this CTA in op o: u = ((cta - rot) mod G) + k*G; tile u / KS,
// K-part u % KS; the part's blocks are split into stages of KC blocks.
__host__ __device__ __forceinline__ int first_unit(const KqOp& o, int cta, int G) {
  int u = cta - (o.rot % G);
  return u < 0 ? u + G : u;
}

// Producer: lane i copies row i's segment (blocks [b0, b0+n)) of the tile
// into slot + i*srb, as its 16-byte aligned superset; arrive on full.  A
// stage of whole rows is one contiguous block: lane 0 copies its 16-byte
// aligned superset with one bulk copy (fewer, larger copies stream faster).
__device__ __forceinline__ void produce(const KqOp& o, int tile, int b0, int n, uint8_t* slot, uint64_t* full,
                                       int lane, int BB, uint64_t pol) {
  const int64_t r0 = static_cast<int64_t>(tile) * (8 * o.R);
  if (o.contig) {
    if (lane == 0) {
      const int64_t nrows = min_i64(8 * o.R, o.N - r0);
      const uintptr_t s0 = reinterpret_cast<uintptr_t>(o.W + r0 * o.row_bytes);
      const uintptr_t as = s0 & ~uintptr_t(15), ae = (s0 + nrows * o.row_bytes + 15) & ~uintptr_t(15);
      mbar_arrive_expect_tx(full, static_cast<uint32_t>(ae - as));
      bulk_g2s_hint(slot, reinterpret_cast<const void*>(as), static_cast<uint32_t>(ae - as), full, pol);
    }
    return;
  }
  uint32_t len = 0;
  const uint8_t* src = nullptr;
  if (lane < 8 * o.R && r0 + lane < o.N) {
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
  if (len) bulk_g2s_hint(slot + lane * o.srb, src, len, full, pol);
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
  int slot;        // ring slot of the next stage
  uint32_t phase;  // parity of the ring lap of the next stage
  int rs;          // reduction buffer of the next unit
  int cb;          // pairs of blocks seen, mod NC: pair-to-warp rotation
  bool failed;
};

// Consumers: every unit of op o for this CTA.  Quad q of every warp owns the
// tile rows q, q+8, ... (R of them; a tile is 8R rows).  A stage's blocks are
// dealt to the warps (continuing across stages) in pairs -- lanes c of every
// quad take block 2g + (c >> 1) of pair g, half c & 1 of it (two 64-weight
// chunks, one 128-value run), for the R rows of the quad, and combine once per
// row and half -- or, with BLK, one by one: lane c takes chunk c of the block
// and combines once per row and chunk.  NI x images: with
// SUM they are the hi and lo images of one fp32 x (one output), else NI
// tokens' bf16 x (y is [NI][N]; each token's rows take exactly the one-token
// arithmetic).
// BLK: the items dealt to the warps are single blocks (lane c = chunk c, one
// combine per chunk; programs: twice the items per stage, so a stage's slot
// is released sooner -- dense sweep chain 1.42 -> 1.36 ms) instead of pairs
// (single products: fewer combines -- the long Q4_K product 3.38 -> 3.77 TB/s).
template <int QT, int R, int NI, bool SUM, bool BLK = false>
__device__ void consume_op(const KqOp& o, const XImg (&xs)[NI], const Ring& rg, const Red& rd, Walk& wk, int* err,
                           int cta, int G) {
  constexpr int BB = Fmt<QT>::BYTES;
  constexpr int MT = SUM ? 1 : NI;  // outputs per row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = lane >> 2, c = lane & 3;
  for (int u = first_unit(o, cta, G); u < o.nunits; u += G) {
    const int tile = u / o.KS, kp = u - tile * o.KS;
    const int kb0 = kp * o.kpb;
    const int kb1 = min(o.nb, kb0 + o.kpb);
    const int64_t row0 = static_cast<int64_t>(tile) * (8 * R);
    float acc[MT][R];
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
      for (int i = 0; i < R; ++i) acc[t][i] = 0.0f;
    int items = 0;      // items of the unit (all warps)
    bool mine = false;  // this warp has an item in the unit
    for (int b0 = kb0; b0 < kb1; b0 += o.KC) {
      const int n = min(o.KC, kb1 - b0);
      const int ng = BLK ? n : (n + 1) >> 1;  // items: blocks, or pairs of blocks
      const int slot = wk.slot;
      if (!wk.failed) {
        const bool ok = mbar_wait(&rg.full[slot], wk.phase, err);
        wk.failed = !__all_sync(0xFFFFFFFFu, ok);
      }
      int gi = warp - wk.cb;
      if (gi < 0) gi += NC;
      mine = mine || gi < ng;
      items += ng;
      if (!wk.failed && gi < ng) {
        // the quad's rows q, q+8, q+16, q+24 (rows past N are computed on
        // stale shared memory and never written)
        const uint32_t sp = rg.base_s + static_cast<uint32_t>(slot) * rg.slot;
        const uint32_t seg0 = static_cast<uint32_t>(row0 * o.row_bytes) + static_cast<uint32_t>(b0 * BB);
        uint32_t rp[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
          const int r = quad + 8 * i;
          // W is 16-byte aligned: the segment's offset in its 16-byte granule
          // (one offset for a stage copied as one block)
          const uint32_t off =
              (seg0 + (o.contig ? 0u : static_cast<uint32_t>(r) * static_cast<uint32_t>(o.row_bytes))) & 15u;
          rp[i] = sp + r * o.srb + off + (BLK ? gi : 2 * gi + (c >> 1)) * BB;
        }
        const ScaleLane sl = scale_lane(c);
        for (; gi < ng; gi += NC) {
          const int bl = BLK ? gi : 2 * gi + (c >> 1);  // this lane's block within the stage
          if constexpr (BLK) {
            const int b = b0 + bl;
            if constexpr (SUM) {
#pragma unroll 1
              for (int t = 0; t < NI; ++t)
                block_rows<QT, R>(t ? xs[NI - 1] : xs[0], b, rp, c, sl, t ? kLimBf16 : kLimHi, acc[0]);
            } else {
#pragma unroll
              for (int t = 0; t < NI; ++t) block_rows<QT, R>(xs[t], b, rp, c, sl, kLimBf16, acc[t]);
            }
          } else if (bl < n) {
            const int b = b0 + bl;
            // the hi image of fp32 x takes the tighter fp32 combine check
            // (kLimHi), bf16 images and the lo image (2^-9 of the value) kLimBf16
            if constexpr (SUM) {  // hi and lo images of one x: one copy of the code, two passes
#pragma unroll 1
              for (int t = 0; t < NI; ++t)
                block_half<QT, R>(t ? xs[NI - 1] : xs[0], b, c & 1, rp, t ? kLimBf16 : kLimHi, acc[0]);
            } else {
#pragma unroll
              for (int t = 0; t < NI; ++t) block_half<QT, R>(xs[t], b, c & 1, rp, kLimBf16, acc[t]);
            }
          }
#pragma unroll
          for (int i = 0; i < R; ++i) rp[i] += (BLK ? 1 : 2) * NC * BB;
        }
      }
      wk.cb = (wk.cb + ng) % NC;
      __syncwarp();
      if (lane == 0) mbar_arrive(&rg.empty[slot]);
      if (++wk.slot == rg.S) { wk.slot = 0; wk.phase ^= 1u; }
    }
    // A unit's buffer is used again RS = S + 1 units later: a warp reaches
    // that unit only after every warp has passed a later stage of the ring,
    // which the unit's last warp does only after adding the unit up.
    const int rs = wk.rs;
    if (++wk.rs == rd.RS) wk.rs = 0;
    if (!mine) continue;  // no item in the unit: its buffer row stays zero
    // this warp's partial row sums: over the quad's lanes, then to shared memory
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
      for (int i = 0; i < R; ++i) {
        acc[t][i] = __fadd_rn(acc[t][i], __shfl_xor_sync(0xFFFFFFFFu, acc[t][i], 1));
        acc[t][i] = __fadd_rn(acc[t][i], __shfl_xor_sync(0xFFFFFFFFu, acc[t][i], 2));
      }
    float* rb = rd.buf + static_cast<size_t>(rs) * NC * TT * MT;  // [MT][NC][TT]
    if (c == 0) {
#pragma unroll
      for (int i = 0; i < R; ++i)
#pragma unroll
        for (int t = 0; t < MT; ++t) rb[(t * NC + warp) * TT + quad + 8 * i] = acc[t][i];
    }
    __syncwarp();
    int last = 0;
    if (lane == 0) {
      __threadfence_block();
      last = (atomicAdd(&rd.cnt[rs], 1) == min(items, NC) - 1) ? 1 : 0;  // the warps with an item
    }
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (!last) continue;
    // last warp of the unit: add the NC partials in warp order (zero where a
    // warp had no item), then clear them
    __threadfence_block();
    float v[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      v[t] = rb[t * NC * TT + lane];
#pragma unroll
      for (int w = 1; w < NC; ++w) v[t] = __fadd_rn(v[t], rb[(t * NC + w) * TT + lane]);
#pragma unroll
      for (int w = 0; w < NC; ++w) rb[(t * NC + w) * TT + lane] = 0.0f;
    }
    __syncwarp();
    if (lane == 0) rd.cnt[rs] = 0;
    const int64_t row = row0 + lane;
    if (lane < 8 * R && row < o.N && !wk.failed) {
      if (o.KS == 1) {
#pragma unroll
        for (int t = 0; t < MT; ++t) o.y[t * o.N + row] = v[t];
      } else {
        o.part[static_cast<int64_t>(kp) * o.ntiles * TT + row] = v[0];  // added at the next grid barrier
      }
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

// A program op: bf16 x (one image) or fp32 x (hi and lo images), any format
// (XK0: the program's x dtypes, 1 = bf16 only, 2 = fp32 only, 0 = both).
// Programs take tiles of 32 rows.
template <int QT, int XK0>
__device__ __forceinline__ void consume_bf16(const KqOp& o, const XImg (&x1)[1], const Ring& rg, const Red& rd,
                                             Walk& wk, int* err, int cta, int G) {
  if constexpr (QT == T_Q6_K) {  // Q6_K ops whose 32-row stage would not fit the chain's slots take 16 rows
    if (o.R == 2) { consume_op<QT, 2, 1, false, true>(o, x1, rg, rd, wk, err, cta, G); return; }
  }
  consume_op<QT, 4, 1, false, true>(o, x1, rg, rd, wk, err, cta, G);
}
template <int XK0>
__device__ __forceinline__ void consume_any(const KqOp& o, bool bf16, const XImg (&xs)[2], const Ring& rg,
                                            const Red& rd, Walk& wk, int* err, int cta, int G) {
  const XImg x1[1] = {xs[0]};
  if (XK0 == 1 || (XK0 == 0 && bf16)) {
    if (o.type == T_Q4_K) consume_bf16<T_Q4_K, XK0>(o, x1, rg, rd, wk, err, cta, G);
    else if (o.type == T_Q5_K) consume_bf16<T_Q5_K, XK0>(o, x1, rg, rd, wk, err, cta, G);
    else consume_bf16<T_Q6_K, XK0>(o, x1, rg, rd, wk, err, cta, G);
  } else {
    if (o.type == T_Q4_K) consume_op<T_Q4_K, 4, 2, true, true>(o, xs, rg, rd, wk, err, cta, G);
    else if (o.type == T_Q5_K) consume_op<T_Q5_K, 4, 2, true, true>(o, xs, rg, rd, wk, err, cta, G);
    else consume_op<T_Q6_K, 4, 2, true, true>(o, xs, rg, rd, wk, err, cta, G);
  }
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
// Shared memory: barriers and counters (256 B), the ring, the reduction
// buffers, the x image.
__host__ __device__ inline size_t red_bytes(int S, int mt = 1) { return static_cast<size_t>(S + 1) * NC * TT * 4 * mt; }
// x images of a launch: one per token, 16-byte aligned
__host__ __device__ inline size_t ximg_stride(int nb) { return (ximg_bytes(nb) + 15) & ~size_t(15); }

// PROG: ops in global memory (any types); else the single op a.op0, whose
// type and x dtype are the template's QT0 and XK0 (one instantiation per
// format and x dtype keeps the single-product code small).  XK0: 1 = bf16 x
// (MT0 tokens), 2 = fp32 x (one token, hi and lo images), 0 = either (programs).
template <bool PROG, int QT0, int XK0, int R0, int MT0 = 1>
__global__ void __launch_bounds__(NTH, 1) prog_kernel(const __grid_constant__ ProgArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  Ring rg;
  rg.full = reinterpret_cast<uint64_t*>(smem);
  rg.empty = rg.full + RING_MAX;
  rg.base = smem + kHdrBytes;
  rg.base_s = smem_u32(rg.base);
  rg.S = a.S;
  rg.slot = a.slot;
  Red rd;
  rd.cnt = reinterpret_cast<int*>(rg.empty + RING_MAX);  // RING_MAX + 1 ints
  rd.RS = a.S + 1;
  rd.buf = reinterpret_cast<float*>(rg.base + static_cast<size_t>(a.S) * a.slot);
  uint8_t* xbase = reinterpret_cast<uint8_t*>(rd.buf) + red_bytes(a.S, MT0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.S; ++s) { mbar_init(&rg.full[s], 1); mbar_init(&rg.empty[s], NC); }
    for (int s = 0; s <= a.S; ++s) rd.cnt[s] = 0;
  }
  for (size_t i = threadIdx.x; i < red_bytes(a.S, MT0) / 4; i += NTH) rd.buf[i] = 0.0f;
  fence_mbar_init();
  __syncthreads();

  if (warp == NC) {
    // ------------------------------------------------------------ producer
    pdl_launch_dependents();
    int q = 0, slot = 0;
    uint32_t lap = 0;  // parity of the ring lap
    const uint64_t pol = l2_evict_first_policy();  // weights are read once per launch
    StageCursor cc;
    cur_start<PROG>(a, cc, cta, G);
    while (cc.valid) {
      if (q >= a.S) {  // the slot's previous stage has been consumed
        const bool ok = mbar_wait(&rg.empty[slot], lap ^ 1u, a.err);
        if (!__all_sync(0xFFFFFFFFu, ok)) break;
      }
      produce(cc.o, cc.tile, cc.b0, min(cc.o.KC, cc.kb1 - cc.b0), rg.base + static_cast<size_t>(slot) * a.slot,
              &rg.full[slot], lane, block_bytes_of(cc.o.type), pol);
      cur_next<PROG>(a, cc, cta, G);
      ++q;
      if (++slot == a.S) { slot = 0; lap ^= 1u; }
    }
    // leave only after the copies in flight have landed (bounded)
    if (lane == 0)
      for (int r = (q > a.S ? q - a.S : 0); r < q; ++r)
        mbar_wait(&rg.full[r % a.S], static_cast<uint32_t>((r / a.S) & 1), nullptr);
    return;
  }

  // --------------------------------------------------------------- consumers
  pdl_wait();
  pdl_launch_dependents();
  const int ctid = threadIdx.x;
  Walk wk = {0, 0u, 0, 0, false};
  int barriers = 0;
  // Split-K sums: no later op reads them (the host plans no split for an op
  // whose output feeds a later x), so the sums of the ops before the last
  // barrier passed are added just before the next barrier, off the path from
  // a barrier to the next op's first product (CTAs that finish early do it
  // while the rest of the grid finishes).
  int fixed = 0;     // ops before this index have their split-K sums added
  int complete = 0;  // ops before this index have all their partial sums written
  KqOp nxt = load_op<PROG>(a, 0);  // the next op's descriptor, loaded one op ahead
  for (int oi = 0; oi < a.n_ops; ++oi) {
    const KqOp o = nxt;
    if (PROG && oi + 1 < a.n_ops) nxt = load_op<PROG>(a, oi + 1);
    // the blocks of x this CTA reads until the next x (read before any wait:
    // the table is written at planning time)
    int xr = -1;
    if (PROG && o.xrange && (oi == 0 || (o.flags & (OP_NEWX | OP_WAIT)))) xr = __ldg(o.xrange + cta);
    const bool bf16 = XK0 ? (XK0 == 1) : (o.x_bf16 != 0);  // a program of one x dtype is compiled for it
    if (PROG && oi > 0 && (o.flags & OP_WAIT)) {
      if constexpr (PROG) {
        for (; fixed < complete; ++fixed) {
          const KqOp f = load_op<PROG>(a, fixed);
          if (f.KS > 1) fixup_op(f, cta, G, ctid);
        }
      }
      // publish this CTA's outputs so far, then wait for the rest of the grid
      consumer_sync();
      ++barriers;
      KQ_TL(oi, 3);
      if (ctid == 0) {
        grid_arrive(a.barrier);
        grid_wait(a.barrier, barriers * G, a.err);  // on timeout the error word is set
      }
      KQ_TL(oi, 0);
      consumer_sync();
      complete = oi;
    }
    if constexpr (!PROG) {
      // fp32 x: the hi and lo images of the one token; bf16 x: one image per
      // token (x is [MT0][K])
      constexpr int NI = XK0 == 2 ? 2 : MT0;
      XImg xs[NI];
#pragma unroll
      for (int t = 0; t < NI; ++t) xs[t] = ximg_at(xbase + t * ximg_stride(a.nb_max), a.nb_max);
      consumer_sync();
      if constexpr (XK0 == 2) {
        stage_x<NTHC>(o.x, 0, o.K, o.nb, xs[0], xs[NI - 1], ctid);
      } else {
#pragma unroll
        for (int t = 0; t < NI; ++t)
          stage_x<NTHC>(static_cast<const uint16_t*>(o.x) + static_cast<size_t>(t) * o.K, 1, o.K, o.nb, xs[t], xs[t],
                        ctid);
      }
      consumer_sync();
      consume_op<QT0, R0, NI, XK0 == 2>(o, xs, rg, rd, wk, a.err, cta, G);
      continue;
    }
    const XImg xs2[2] = {ximg_at(xbase, a.nb_max), ximg_at(xbase + (a.nimg > 1 ? ximg_stride(a.nb_max) : 0), a.nb_max)};
    if (oi == 0 || (o.flags & (OP_NEWX | OP_WAIT))) {
      consumer_sync();  // every consumer is done with the previous x image
      if (xr < 0) stage_x<NTHC>(o.x, bf16 ? 1 : 0, o.K, o.nb, xs2[0], xs2[1], ctid);
      else stage_x<NTHC>(o.x, bf16 ? 1 : 0, o.K, o.nb, xs2[0], xs2[1], ctid, xr & 0xFFFF, xr >> 16);
      consumer_sync();
    }
    KQ_TL(oi, 1);
    consume_any<XK0>(o, bf16, xs2, rg, rd, wk, a.err, cta, G);
  }
  if constexpr (PROG) {  // sums complete since the last barrier
    for (; fixed < complete; ++fixed) {
      const KqOp f = load_op<PROG>(a, fixed);
      if (f.KS > 1) fixup_op(f, cta, G, ctid);
    }
  }
  if constexpr (PROG) {
    consumer_sync();
    KQ_TL(a.n_ops, 3);  // all of this CTA's ops done
  }
  if (PROG && a.barrier) {
    // final barrier (only when split-K sums of the last stage remain), then
    // the exit count: the last CTA to leave resets both counters for the next
    // launch
    consumer_sync();
    if (a.final_fix) {
      ++barriers;
      if (ctid == 0) {
        grid_arrive(a.barrier);
        grid_wait(a.barrier, barriers * G, a.err);
      }
      consumer_sync();
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

// Widest stage (blocks) of an op of tile height 8R: whole rows if they fit a
// whole-row stage, else the widest row segments that fit a slot (0: none).
int op_kcmax(const KqOp& o, int64_t slot_cap) {
  const int TTo = 8 * o.R;
  if (static_cast<int64_t>(TTo) * o.row_bytes + 32 <= whole_cap(o.R)) return o.nb;
  int kcmax = o.nb;
  while (kcmax > 1 && static_cast<int64_t>(TTo) * seg_stride(o.type, kcmax) > slot_cap) --kcmax;
  return static_cast<int64_t>(TTo) * seg_stride(o.type, kcmax) > slot_cap ? 0 : kcmax;
}

// Whether nb blocks split into KS parts of ceil(nb/KS) >= 2 blocks, none empty.
bool split_ok(int nb, int KS) {
  const int kpb = (nb + KS - 1) / KS;
  return KS == 1 || (kpb >= 2 && (KS - 1) * kpb < nb);
}

// K-parts KS of an op (planned tiles) and its stages: as few as fit, evened out.
void set_split(KqOp& o, int KS, int kcmax) {
  o.KS = KS;
  o.kpb = (o.nb + KS - 1) / KS;
  const int nst = (o.kpb + kcmax - 1) / kcmax;
  o.KC = (o.kpb + nst - 1) / nst;
  o.srb = seg_stride(o.type, o.KC);
  // whole rows per stage: one copy per stage, rows at their memory stride
  o.contig = (o.KS == 1 && o.KC == o.nb) ? 1 : 0;
  if (o.contig) o.srb = static_cast<int32_t>(o.row_bytes);
  o.nunits = static_cast<int32_t>(static_cast<int64_t>(o.ntiles) * KS);
}

// Geometry of one op: K-parts KS (only with a workspace) and stage width KC.
// cost = block-chunks of the busiest CTA (a chunk = one block for 32 rows,
// dealt to one warp), plus a fixed cost per stage and per split.
bool plan_op(KqOp& o, int G, bool allow_split, int64_t slot_cap, bool allow_short_tiles = false, int force_R = 0) {
  const int BB = block_bytes_of(o.type);
  if (!BB || o.K <= 0 || o.K % 32 || o.N <= 0) return false;
  o.nb = (o.K + 255) / 256;
  if (o.nb > MAX_NB) return false;
  o.row_bytes = static_cast<int64_t>(o.nb) * BB;
  // tile height 8R: the busiest CTA's rows, rounds * 8R, with shorter tiles
  // charged for their lost x reuse (one x slice serves R rows)
  // Heights whose tile of whole rows fits one slot are preferred: such a
  // stage is one bulk copy (per-row copies of short segments stream slower).
  o.R = 4;
  if (allow_short_tiles) {
    bool any_whole = false;
    for (int r : {4, 2, 1}) any_whole = any_whole || 8 * r * o.row_bytes + 32 <= whole_cap(r);
    double best = -1.0;
    for (int r : {4, 2, 1}) {
      if (any_whole && 8 * r * o.row_bytes + 32 > whole_cap(r)) continue;
      const int64_t nt = (o.N + 8 * r - 1) / (8 * r);
      const double cost = static_cast<double>((nt + G - 1) / G) * 8 * r * (1.0 + 0.08 * (4 / r - 1));
      if (best < 0 || cost < best - 1e-9) { best = cost; o.R = r; }
    }
  }
  if (force_R) o.R = force_R;
  const int TTo = 8 * o.R;
  const int64_t ntiles = (o.N + TTo - 1) / TTo;
  if (ntiles > (int64_t(1) << 28)) return false;
  o.ntiles = static_cast<int32_t>(ntiles);
  const int kcmax = op_kcmax(o, slot_cap);
  if (kcmax < 1) return false;
  // K-parts (with a workspace): minimise the busiest CTA's blocks,
  // ceil(tiles*KS / G) * ceil(nb / KS), plus one block per split level
  int KS = 1;
  int64_t best = ((ntiles + G - 1) / G) * o.nb;
  for (int k2 = 2; allow_split && k2 <= 8; k2 *= 2) {
    if (!split_ok(o.nb, k2)) break;
    const int kpb2 = (o.nb + k2 - 1) / k2;
    const int64_t c = ((ntiles * k2 + G - 1) / G) * kpb2 + (k2 / 2);
    if (c < best) { best = c; KS = k2; }
  }
  set_split(o, KS, kcmax);
  return true;
}

int64_t stage_bytes(const KqOp& o) { return static_cast<int64_t>(8 * o.R) * o.srb + (o.contig ? 32 : 0); }

struct LaunchGeom {
  int S, slot;
  size_t smem;
};

// nimg x images of nb_max blocks; mt outputs per row (reduction buffers)
bool ring_geom(int64_t max_stage, int nb_max, int nimg, LaunchGeom& g, int mt = 1) {
  g.slot = static_cast<int>((max_stage + 127) & ~int64_t(127));
  const size_t fixed = kHdrBytes + nimg * ximg_stride(nb_max);
  int S = RING_MAX;
  while (S >= 2 && fixed + static_cast<size_t>(S) * g.slot + red_bytes(S, mt) > static_cast<size_t>(kMaxSmemPerBlock))
    --S;
  if (S < 2) return false;
  g.S = S;
  g.smem = fixed + static_cast<size_t>(S) * g.slot + red_bytes(S, mt);
  return true;
}

template <bool PROG, int QT0, int XK0, int R0, int MT0 = 1>
cudaError_t launch_prog(ProgArgs& a, const LaunchGeom& g, bool cooperative, cudaStream_t st, bool pdl) {
  a.S = g.S;
  a.slot = g.slot;
  static bool smem_set[64] = {false};
  const int dev = current_device_id();
  if (!smem_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(prog_kernel<PROG, QT0, XK0, R0, MT0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
  return cudaLaunchKernelEx(&cfg, prog_kernel<PROG, QT0, XK0, R0, MT0>, a);
}

// Program workspace: header (grid barrier counter), ops, split-K partials and counters.
constexpr size_t kHeaderBytes = 256;

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// One single-product instantiation per (x dtype, tokens, rows per quad) of
// format QT: XK 1 = bf16 x (MT tokens), 2 = fp32 x (one token).
template <int QT, int XK, int MT>
cudaError_t launch_single_r(int R, ProgArgs& a, const LaunchGeom& g, cudaStream_t st, bool pdl) {
  switch (R) {
    case 4: return launch_prog<false, QT, XK, 4, MT>(a, g, false, st, pdl);
    case 2: return launch_prog<false, QT, XK, 2, MT>(a, g, false, st, pdl);
    case 1: return launch_prog<false, QT, XK, 1, MT>(a, g, false, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}
template <int QT>
cudaError_t launch_single_fmt(int XK, int MT, int R, ProgArgs& a, const LaunchGeom& g, cudaStream_t st, bool pdl) {
  if (XK == 2) return MT == 1 ? launch_single_r<QT, 2, 1>(R, a, g, st, pdl) : cudaErrorNotSupported;
  switch (MT) {
    case 1: return launch_single_r<QT, 1, 1>(R, a, g, st, pdl);
    case 2: return launch_single_r<QT, 1, 2>(R, a, g, st, pdl);
    case 3: return launch_single_r<QT, 1, 3>(R, a, g, st, pdl);
    case 4: return launch_single_r<QT, 1, 4>(R, a, g, st, pdl);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace

// Single products of one format (one translation unit each, compiled in
// parallel): kq_gemv_q4k.cu, kq_gemv_q5k.cu, kq_gemv_q6k.cu, kq_gemv_ia4.cu.
cudaError_t launch_single_q4k(int XK, int MT, int R, ProgArgs& a, int S, int slot, size_t smem, cudaStream_t st,
                              bool pdl);
cudaError_t launch_single_q5k(int XK, int MT, int R, ProgArgs& a, int S, int slot, size_t smem, cudaStream_t st,
                              bool pdl);
cudaError_t launch_single_q6k(int XK, int MT, int R, ProgArgs& a, int S, int slot, size_t smem, cudaStream_t st,
                              bool pdl);
cudaError_t launch_single_ia4(int XK, int MT, int R, ProgArgs& a, int S, int slot, size_t smem, cudaStream_t st,
                              bool pdl);

}  // namespace kq
