// kq_moe.cu -- routed-expert products: every selected expert's rows are read
// from memory once and applied to all (token, slot) pairs routed to it.
//
// "GGUF in transformers", section "Reusing ggml's Metal kernels": the kernel
// reads the packed weights directly, including only the experts an MoE layer
// selected.  "ANE Fieldfare" README, "How it works": each token's router
// picks 8 of 128 experts; "Speculative decoding": a planning step groups the
// tokens of a verify block by expert so each expert is read once.
//
// One launch, a one-dimensional grid of up to two segments: a shared
// expert's CTAs (expert FFN only: every token, tiles split by token pairs),
// then one CTA per (distinct-expert rank d, row tile), rank-major:
//  * grouping (every CTA, in shared memory): the routed ids are checked
//    (an id outside [0, n_experts) is recorded in the workspace error word and
//    its pair dropped), the distinct experts are ranked in ascending id order,
//    and CTA (d, tile) takes the d-th one, e, with its pairs (token m, slot j)
//    in (m, j) order.  The CTAs of tile 0 also write this plan to the
//    workspace (expert of each rank, offsets, pairs) for inspection;
//  * the CTA copies its tile of expert e (whole rows, as large as fits in
//    100 KB: 256, 128 or 64 rows, a quad of lanes per 4, 2 or 1 of them; wider
//    rows 32 or 16 rows, 2 or 4 quads per row) with one TMA bulk copy -- in
//    gate|up mode the same rows of both matrices, two copies -- then for each
//    pair stages that pair's x as block-float limbs and applies the rows to it
//    with the lane cores of kq_lane.cuh (gate|up mode: act(gate) * up);
//  * if no routed id is valid at all and there is no shared expert, the
//    gated outputs are zero (empty sums);
//  * without gate weights the result of pair (m, j) is row j of token m's
//    output block (y[m][j][n]); with gate weights it goes to the workspace and
//    the last CTA to finish each group of rows (arrival counters) writes
//    y[m][n] = sum_j g[m][j] * part[m][j][n] in slot order, then adds the
//    shared expert's part (deterministic).
#include "kq_lane.cuh"

namespace kq {

using namespace lane;

namespace {

constexpr int MT_MIN = 16;      // rows per tile at the most quads per row (sizes the tile counters)
constexpr int MW = 8;           // warps
constexpr int MTH = MW * 32;
constexpr int kMaxPairs = 512;  // M * top_k
constexpr int kMaxExperts = 4096;
constexpr int64_t kMaxTileBytes = 100 * 1024;  // 32 rows at most (API limit)
constexpr int kSharedTokens = 2;  // tokens per shared-expert CTA (the tile is re-read from L2 by its siblings)

// One segment of a launch: the routed experts (the grid's first Dmax * ntiles
// CTAs, expert e at W + e * expert_bytes) or the shared expert (one matrix
// applied to every token).
struct MoeSeg {
  const uint8_t* W;
  const uint8_t* W2;     // gate|up mode: the up rows (same shape as W), else null
  int64_t expert_bytes;  // N * row_bytes
  int64_t row_bytes;
  int64_t N;
  int K, nb, nph, rq, rt, ntiles;  // quads per row, rows per quad, rows per tile = 8 * MW * rq / nph
  int x_per_slot;  // routed: x row of pair (m, j) is m * top_k + j (1) or m (0); shared: always m
  const void* x;
  float* out;  // result of pair p (routed) or token m (shared): out[p or m][N]
};

struct MoeArgs {
  MoeSeg seg[2];   // routed, shared
  int nseg;        // 1, or 2 with a shared expert
  int tgroups;     // shared expert: CTAs per tile, each taking kSharedTokens tokens
  int ids_ready;   // the ids were complete before the preceding kernel released this one
  int gu;          // gate|up mode: out = act(W x) * (W2 x)
  int act;         // KQ_ACT_* of the gate|up mode
  int G;           // gated combine: rows per arrival counter (divides both segments' tile heights)
  int type, x_bf16;
  int n_experts, M, top_k;
  const int32_t* ids;
  const float* gate;  // non-null: y[m][n] = sum_j g[m][j] * part[m][j][n] (+ shared[m][n])
  float* y;
  int* err;   // workspace error word
  int* plan;  // workspace plan: D, expert_of[Dmax], offset[Dmax + 1], pairs[M * top_k]
  int* cnt;   // per-group arrival counters (gate case)
  int Dmax;
};

struct MoeSmem {
  int16_t ids[kMaxPairs];    // validated expert ids (-1: dropped)
  uint32_t bits[kMaxExperts / 32];
  int16_t pairs[kMaxPairs];  // this CTA's pairs (routed) or tokens (shared)
  int misc[8];  // 0: e, 1: D, 2: np, 3: offset of e, 4: valid pairs, 5: groups this CTA combines
};

__host__ __device__ inline size_t moe_ximg_offset() { return (sizeof(MoeSmem) + 16 + 127) & ~size_t(127); }

// Row sums of one pair over the tile for the RQ rows of this quad (rows
// rp, rp + rstride, ...; nph quads per row, the quad of phase ph taking blocks
// ph, ph + nph, ...): each block's x slice is loaded once for all RQ rows.
// NI x images (fp32 x: hi and lo) add into the same sums.
// (Out of line, one copy per rows-per-quad: the kernel calls it for up to three
// tile shapes and two matrices, and inlined copies overflowed the instruction
// cache.)
template <int NI>
struct XImgs {
  XImg v[NI];
};
template <int QT, int NI, int RQ>
__device__ __noinline__ float4 pair_rows_ol(uint32_t rp, uint32_t rstride, int nb, const XImgs<NI> xs_, int ph,
                                            int nph, int c, const ScaleLane sl) {
  const XImg (&xs)[NI] = xs_.v;
  constexpr int BB = Fmt<QT>::BYTES;
  float a[RQ];
#pragma unroll
  for (int i = 0; i < RQ; ++i) a[i] = 0.0f;
  for (int b = ph; b < nb; b += nph) {
    uint32_t rb[RQ];
#pragma unroll
    for (int i = 0; i < RQ; ++i) rb[i] = rp + i * rstride + b * BB;
#pragma unroll
    for (int t = 0; t < NI; ++t) block_rows<QT, RQ>(xs[t], b, rb, c, sl, (NI == 1 || t != 0) ? kLimBf16 : kLimHi, a);
  }
#pragma unroll
  for (int i = 0; i < RQ; ++i) {
    float v = a[i];
    v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, 1));
    v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, 2));
    for (int o = 4; o < 4 * nph; o <<= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    a[i] = v;
  }
  return make_float4(a[0], RQ > 1 ? a[RQ > 1 ? 1 : 0] : 0.0f, RQ > 2 ? a[RQ > 2 ? 2 : 0] : 0.0f,
                     RQ > 3 ? a[RQ > 3 ? 3 : 0] : 0.0f);
}
template <int QT, int NI, int RQ>
__device__ __forceinline__ void pair_rows(uint32_t rp, uint32_t rstride, int nb, const XImg (&xs)[NI], int ph,
                                          int nph, int c, const ScaleLane& sl, float (&acc)[4]) {
  XImgs<NI> xv;
#pragma unroll
  for (int t = 0; t < NI; ++t) xv.v[t] = xs[t];
  const float4 r = pair_rows_ol<QT, NI, RQ>(rp, rstride, nb, xv, ph, nph, c, sl);
  acc[0] = r.x; acc[1] = r.y; acc[2] = r.z; acc[3] = r.w;
}

// The activation of the gate|up mode, in fp32 with CUDA's expf / tanhf.
//   KQ_ACT_SILU: g / (1 + exp(-g));  KQ_ACT_GELU_TANH: the tanh form of GELU,
//   0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))).
__device__ __forceinline__ float ffn_act(int act, float g) {
  if (act == 1) return 0.5f * g * (1.0f + tanhf(0.7978845608028654f * (g + 0.044715f * g * g * g)));
  return g / (1.0f + expf(-g));
}

template <int QT, int XK>
__global__ void __launch_bounds__(MTH, 2) moe_kernel(const __grid_constant__ MoeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  MoeSmem& sm = *reinterpret_cast<MoeSmem*>(smem + 16);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // 1-D grid: the shared expert's CTAs (tile, token group) first -- each runs
  // up to kSharedTokens tokens, the siblings of a tile adjacent so that their
  // copies of it meet in L2 -- then the routed CTAs (rank d, tile), d-major
  const int nshared = a.nseg > 1 ? a.seg[1].ntiles * a.tgroups : 0;
  const bool shared_seg = static_cast<int>(blockIdx.x) < nshared;
  const int rb = static_cast<int>(blockIdx.x) - nshared;
  const int d = shared_seg ? 0 : rb / a.seg[0].ntiles;
  const int tile = shared_seg ? static_cast<int>(blockIdx.x) / a.tgroups : rb - d * a.seg[0].ntiles;
  const int tok0 = shared_seg ? (static_cast<int>(blockIdx.x) - tile * a.tgroups) * kSharedTokens : 0;
  const MoeSeg sg = shared_seg ? a.seg[1] : a.seg[0];
  const int MK = a.M * a.top_k;
  int nb_max = a.seg[0].nb;
  if (a.nseg > 1 && a.seg[1].nb > nb_max) nb_max = a.seg[1].nb;
  constexpr int NI = XK == 2 ? 2 : 1;  // fp32 x: hi and lo images
  XImg xs[NI];
#pragma unroll
  for (int t = 0; t < NI; ++t) xs[t] = ximg_at(smem + moe_ximg_offset() + t * ximg_bytes(nb_max), sg.nb);
  uint8_t* tile_buf = smem + moe_ximg_offset() + ((NI * ximg_bytes(nb_max) + 127) & ~size_t(127));

  // ---- grouping: validated ids, presence bits, the d-th distinct expert
  auto group = [&]() {
    const int nwords = (a.n_experts + 31) >> 5;
    for (int i = tid; i < nwords; i += MTH) sm.bits[i] = 0;
    if (tid == 0) sm.misc[5] = 0;
    __syncthreads();
    for (int i = tid; i < MK; i += MTH) {
      int id = a.ids[i];
      if (id < 0 || id >= a.n_experts) {
        record_error(a.err, DEV_ERR_EXPERT_ID);
        id = -1;
      } else {
        atomicOr(&sm.bits[id >> 5], 1u << (id & 31));
      }
      sm.ids[i] = static_cast<int16_t>(id);
    }
    __syncthreads();
    if (warp == 0) {
      // rank d among set bits, scanning the words in order
      int base = 0, e = -1;
      for (int w0 = 0; w0 < nwords; w0 += 32) {
        const int w = w0 + lane;
        const uint32_t bits = w < nwords ? sm.bits[w] : 0u;
        const int cnt = __popc(bits);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += t;
        }
        const int excl = base + incl - cnt;
        if (e < 0 && d >= excl && d < excl + cnt) {
          uint32_t b = bits;
          for (int k = 0; k < d - excl; ++k) b &= b - 1;  // drop the lower set bits
          e = 32 * w + __ffs(b) - 1;
        }
        base += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
      e = __reduce_max_sync(0xFFFFFFFFu, e);
      if (lane == 0) { sm.misc[0] = e; sm.misc[1] = base; }
    }
    __syncthreads();
  };

  // ---- the tile: one bulk copy of whole rows (two in gate|up mode)
  const int64_t r0 = static_cast<int64_t>(tile) * sg.rt;
  const int nrows = static_cast<int>(min_i64(sg.rt, sg.N - r0));
  const uint32_t part_bytes = static_cast<uint32_t>((sg.rt * sg.row_bytes + 32 + 15) & ~int64_t(15));
  uintptr_t s0 = 0, as = 0, s2 = 0, as2 = 0;
  auto issue = [&](int e) {
    const int64_t off = (shared_seg ? 0 : e * sg.expert_bytes) + r0 * sg.row_bytes;
    s0 = reinterpret_cast<uintptr_t>(sg.W + off);
    as = s0 & ~uintptr_t(15);
    const uintptr_t ae = (s0 + nrows * sg.row_bytes + 15) & ~uintptr_t(15);
    s2 = a.gu ? reinterpret_cast<uintptr_t>(sg.W2 + off) : 0;
    as2 = s2 & ~uintptr_t(15);
    const uintptr_t ae2 = (s2 + nrows * sg.row_bytes + 15) & ~uintptr_t(15);
    if (tid == 0) {
      mbar_init(bar, 1);
      fence_mbar_init();
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>((ae - as) + (a.gu ? ae2 - as2 : 0)));
      if (shared_seg && a.tgroups > 1) {  // siblings read the same tile: keep it in L2
        bulk_g2s(tile_buf, reinterpret_cast<const void*>(as), static_cast<uint32_t>(ae - as), bar);
        if (a.gu)
          bulk_g2s(tile_buf + part_bytes, reinterpret_cast<const void*>(as2), static_cast<uint32_t>(ae2 - as2), bar);
      } else {
        const uint64_t pol = l2_evict_first_policy();  // a weight tile is read once per call
        bulk_g2s_hint(tile_buf, reinterpret_cast<const void*>(as), static_cast<uint32_t>(ae - as), bar, pol);
        if (a.gu)
          bulk_g2s_hint(tile_buf + part_bytes, reinterpret_cast<const void*>(as2), static_cast<uint32_t>(ae2 - as2),
                        bar, pol);
      }
    }
  };

  // The weights never depend on the preceding kernel; the routed ids do,
  // unless they were complete before it released this grid (ids_ready).  So
  // what can start before the wait -- the grouping, the tile copy -- does.
  const bool early_ids = a.ids_ready != 0;
  const bool zero_fill = a.gate && a.nseg == 1 && !shared_seg && d == 0;  // the CTAs that zero y if D == 0
  if (early_ids) {
    group();
    if (shared_seg || sm.misc[0] >= 0) issue(sm.misc[0]);
    else if (!(zero_fill && sm.misc[1] == 0)) return;  // fewer distinct experts than this rank
  } else if (shared_seg) {
    issue(0);
  }
  pdl_wait();  // gates and x (and, without ids_ready, the ids) come from earlier kernels
  pdl_launch_dependents();
  if (!early_ids) group();
  const int e = sm.misc[0], D = sm.misc[1];
  if (zero_fill && D == 0) {  // no valid pair, no shared expert: the gated outputs are zero
    for (int i = tid; i < a.M * nrows; i += MTH)
      a.y[static_cast<int64_t>(i / nrows) * sg.N + r0 + i % nrows] = 0.0f;
  }
  if (!shared_seg && e < 0) return;  // fewer distinct experts than this rank
  if (!early_ids && !shared_seg) issue(e);

  // ---- the pairs in (m, slot) order (routed), or this CTA's tokens (shared)
  if (shared_seg) {
    const int nt = static_cast<int>(min_i64(kSharedTokens, a.M - tok0));
    if (tid < nt) sm.pairs[tid] = static_cast<int16_t>(tok0 + tid);
    if (tid == 0) sm.misc[2] = nt;
  } else if (warp == 0) {
    int np = 0, below = 0, valid = 0;
    for (int i0 = 0; i0 < MK; i0 += 32) {
      const int i = i0 + lane;
      const int id = i < MK ? sm.ids[i] : -1;
      const uint32_t mine = __ballot_sync(0xFFFFFFFFu, id == e);
      if (id == e) sm.pairs[np + __popc(mine & ((1u << lane) - 1))] = static_cast<int16_t>(i);
      np += __popc(mine);
      below += __popc(__ballot_sync(0xFFFFFFFFu, id >= 0 && id < e));
      valid += __popc(__ballot_sync(0xFFFFFFFFu, id >= 0));
    }
    if (lane == 0) { sm.misc[2] = np; sm.misc[3] = below; sm.misc[4] = valid; }
  }
  __syncthreads();
  const int np = sm.misc[2];
  if (!shared_seg && tile == 0) {  // the plan, for inspection
    for (int j = tid; j < np; j += MTH) a.plan[1 + 2 * a.Dmax + 1 + sm.misc[3] + j] = sm.pairs[j];
    if (tid == 0) {
      a.plan[1 + d] = e;
      a.plan[1 + a.Dmax + d] = sm.misc[3];
      if (d == 0) { a.plan[0] = D; a.plan[1 + a.Dmax + D] = sm.misc[4]; }
    }
  }

  // ---- apply the rows to every pair: quad rows rq0 + i * (64 / nph), i < rq
  const int quad = lane >> 2, c = lane & 3;
  const int rq0 = warp * (8 / sg.nph) + quad / sg.nph, ph = quad % sg.nph;
  const int rstep = 8 * MW / sg.nph;
  const ScaleLane sl = scale_lane(c);
  const uint32_t rp = smem_u32(tile_buf) + static_cast<uint32_t>(s0 - as) + static_cast<uint32_t>(rq0 * sg.row_bytes);
  const uint32_t rp2 =
      smem_u32(tile_buf) + part_bytes + static_cast<uint32_t>(s2 - as2) + static_cast<uint32_t>(rq0 * sg.row_bytes);
  const uint32_t rstride = static_cast<uint32_t>(rstep * sg.row_bytes);
  bool ok = true;
  for (int j = 0; j < np; ++j) {
    const int pr = sm.pairs[j];
    const int m = shared_seg ? pr : pr / a.top_k;
    const int64_t xrow = (!shared_seg && sg.x_per_slot) ? pr : m;
    const void* xp = XK == 1 ? static_cast<const void*>(static_cast<const uint16_t*>(sg.x) + xrow * sg.K)
                             : static_cast<const void*>(static_cast<const float*>(sg.x) + xrow * sg.K);
    __syncthreads();  // the previous pair is done with the x image
    stage_x<MTH>(xp, XK == 1, sg.K, sg.nb, xs[0], xs[NI - 1], tid);
    __syncthreads();
    if (j == 0) ok = mbar_wait(bar, 0, a.err);
    float v[4], u[4];
    if (sg.rq == 4) pair_rows<QT, NI, 4>(rp, rstride, sg.nb, xs, ph, sg.nph, c, sl, v);
    else if (sg.rq == 2) pair_rows<QT, NI, 2>(rp, rstride, sg.nb, xs, ph, sg.nph, c, sl, v);
    else pair_rows<QT, NI, 1>(rp, rstride, sg.nb, xs, ph, sg.nph, c, sl, v);
    if (a.gu) {
      if (sg.rq == 4) pair_rows<QT, NI, 4>(rp2, rstride, sg.nb, xs, ph, sg.nph, c, sl, u);
      else if (sg.rq == 2) pair_rows<QT, NI, 2>(rp2, rstride, sg.nb, xs, ph, sg.nph, c, sl, u);
      else pair_rows<QT, NI, 1>(rp2, rstride, sg.nb, xs, ph, sg.nph, c, sl, u);
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = ffn_act(a.act, v[i]) * u[i];
    }
    if (ok && c == 0 && ph == 0) {
      float* out = sg.out + static_cast<int64_t>(pr) * sg.N + r0;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (i < sg.rq && rq0 + i * rstep < nrows) out[rq0 + i * rstep] = v[i];
    }
  }
  if (np == 0 && tid == 0) ok = mbar_wait(bar, 0, a.err);  // the copy must land before the CTA exits
  if (!a.gate) return;

  // ---- gate-weighted combine, per group of G rows, by the last CTA to finish it
  const int g0 = static_cast<int>(r0 / a.G), ng = (nrows + a.G - 1) / a.G;
  const int expected = D + (a.nseg > 1 ? a.tgroups : 0);
  __threadfence();
  __syncthreads();
  if (tid < ng && atomicAdd(&a.cnt[g0 + tid], 1) == expected - 1) atomicOr(&sm.misc[5], 1 << tid);
  __syncthreads();
  const int mine = sm.misc[5];
  if (!mine) return;
  __threadfence();
  const float* part = a.seg[0].out;
  const float* spart = a.nseg > 1 ? a.seg[1].out : nullptr;
  for (int i = tid; i < a.M * nrows; i += MTH) {
    const int m = i / nrows, r = i - m * nrows;
    if (!((mine >> (r / a.G)) & 1)) continue;
    const float* pp = part + static_cast<int64_t>(m) * a.top_k * sg.N + r0 + r;
    const int16_t* id = sm.ids + m * a.top_k;
    const float* g = a.gate + m * a.top_k;
    float v = 0.0f;
    int j = 0;
    for (; j + 4 <= a.top_k; j += 4) {  // four loads in flight, applied in slot order; dropped pairs skipped
      float p[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) p[q] = id[j + q] >= 0 ? __ldcg(pp + static_cast<int64_t>(j + q) * sg.N) : 0.0f;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (id[j + q] >= 0) v = __fmaf_rn(g[j + q], p[q], v);
    }
    for (; j < a.top_k; ++j)
      if (id[j] >= 0) v = __fmaf_rn(g[j], __ldcg(pp + static_cast<int64_t>(j) * sg.N), v);
    if (spart) v = __fadd_rn(v, __ldcg(spart + static_cast<int64_t>(m) * sg.N + r0 + r));
    a.y[static_cast<int64_t>(m) * sg.N + r0 + r] = v;
  }
  if (tid < ng && ((mine >> tid) & 1)) a.cnt[g0 + tid] = 0;  // ready for the next call
}

template <int QT, int XK>
cudaError_t launch_moe_t(const MoeArgs& a, size_t smem, cudaStream_t st) {
  static bool smem_set[64] = {false};
  const int dev = current_device_id();
  if (!smem_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(moe_kernel<QT, XK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kMaxSmemPerBlock);
    if (e != cudaSuccess) return e;
    smem_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.Dmax * a.seg[0].ntiles + (a.nseg > 1 ? a.seg[1].ntiles * a.tgroups : 0));
  cfg.blockDim = dim3(MTH);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_kernel<QT, XK>, a);
}

size_t a256(size_t v) { return (v + 255) & ~size_t(255); }

// Tile shape: the largest tile of at most kMaxTileBytes, from 256 rows (a quad per
// 4 rows, each block's x slice serving all 4) down to 16 rows (4 quads per row).
// Fewer, larger tiles mean fewer CTAs paying the fixed costs (grouping, copy
// latency, x staging) per byte of weights.
void moe_tile_shape(int64_t row_bytes, int& nph, int& rq) {
  nph = 4;
  rq = 1;
  for (int r = 4; r >= 1; r >>= 1)
    if (8 * MW * r * row_bytes + 32 <= kMaxTileBytes) { nph = 1; rq = r; break; }
  if (nph == 4 && 8 * MW / 2 * row_bytes + 32 <= kMaxTileBytes) nph = 2;
  if (nph > 1) rq = 1;
}

}  // namespace

MoeLayout moe_layout(int64_t N, int64_t M, int top_k, int n_experts) {
  MoeLayout L;
  const int64_t MK = M * top_k;
  L.Dmax = static_cast<int>(MK < n_experts ? MK : n_experts);
  L.ntiles = (N + MT_MIN - 1) / MT_MIN;  // the most tiles any rows-per-tile choice makes
  L.plan_off = 256;
  L.cnt_off = L.plan_off + a256(sizeof(int) * (1 + 2 * static_cast<size_t>(L.Dmax) + 1 + MK));
  L.part_off = L.cnt_off + a256(sizeof(int) * static_cast<size_t>(L.ntiles));
  L.bytes = L.part_off + a256(sizeof(float) * static_cast<size_t>(MK) * N);
  return L;
}

bool moe_supported(int qtype, int64_t K, int64_t M, int top_k, int n_experts) {
  const int BB = block_bytes_of(qtype);
  const int64_t row_bytes = ((K + 255) / 256) * BB;
  return BB && M * top_k <= kMaxPairs && n_experts <= kMaxExperts && (K + 255) / 256 <= 64 &&
         32 * row_bytes + 32 <= kMaxTileBytes;
}

namespace {

void fill_seg(MoeSeg& s, int qtype, const void* W, const void* W2, int64_t N, int K, const void* x, int x_per_slot,
              float* out) {
  s.nb = (K + 255) / 256;
  s.row_bytes = static_cast<int64_t>(s.nb) * block_bytes_of(qtype);
  s.N = N;
  s.K = K;
  s.expert_bytes = N * s.row_bytes;
  s.W = static_cast<const uint8_t*>(W);
  s.W2 = static_cast<const uint8_t*>(W2);
  s.x = x;
  s.x_per_slot = x_per_slot;
  s.out = out;
  moe_tile_shape(W2 ? 2 * s.row_bytes : s.row_bytes, s.nph, s.rq);  // gate|up: both matrices' rows in the tile
  s.rt = 8 * MW * s.rq / s.nph;
  s.ntiles = static_cast<int>((N + s.rt - 1) / s.rt);
}

size_t seg_tile_bytes(const MoeSeg& s) {
  const size_t one = (static_cast<size_t>(s.rt * s.row_bytes) + 32 + 15) & ~size_t(15);
  return s.W2 ? 2 * one : one;
}

cudaError_t launch_args(MoeArgs& a, int qtype, cudaStream_t st) {
  const int XK = a.x_bf16 ? 1 : 2, NI = a.x_bf16 ? 1 : 2;
  int nb = a.seg[0].nb;
  size_t tb = seg_tile_bytes(a.seg[0]);
  if (a.nseg > 1) {
    nb = nb > a.seg[1].nb ? nb : a.seg[1].nb;
    tb = tb > seg_tile_bytes(a.seg[1]) ? tb : seg_tile_bytes(a.seg[1]);
  }
  const size_t smem = moe_ximg_offset() + ((NI * ximg_bytes(nb) + 127) & ~size_t(127)) + tb;
  if (smem > static_cast<size_t>(kMaxSmemPerBlock)) return cudaErrorNotSupported;
  switch (qtype * 4 + XK) {
    case T_Q4_K * 4 + 1: return launch_moe_t<T_Q4_K, 1>(a, smem, st);
    case T_Q4_K * 4 + 2: return launch_moe_t<T_Q4_K, 2>(a, smem, st);
    case T_Q5_K * 4 + 1: return launch_moe_t<T_Q5_K, 1>(a, smem, st);
    case T_Q5_K * 4 + 2: return launch_moe_t<T_Q5_K, 2>(a, smem, st);
    case T_Q6_K * 4 + 1: return launch_moe_t<T_Q6_K, 1>(a, smem, st);
    case T_Q6_K * 4 + 2: return launch_moe_t<T_Q6_K, 2>(a, smem, st);
    case T_IA4 * 4 + 1: return launch_moe_t<T_IA4, 1>(a, smem, st);
    case T_IA4 * 4 + 2: return launch_moe_t<T_IA4, 2>(a, smem, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_moe_err(int qtype, const void* W, int n_experts, const int32_t* ids, const float* gate,
                           const void* x, int x_bf16, int x_per_slot, float* y, int64_t N, int K, int M, int top_k,
                           void* ws, int* err, cudaStream_t st) {
  const MoeLayout L = moe_layout(N, M, top_k, n_experts);
  uint8_t* w = static_cast<uint8_t*>(ws);
  MoeArgs a = {};
  fill_seg(a.seg[0], qtype, W, nullptr, N, K, x, x_per_slot, gate ? reinterpret_cast<float*>(w + L.part_off) : y);
  a.nseg = 1;
  a.G = a.seg[0].rt;
  a.type = qtype;
  a.x_bf16 = x_bf16;
  a.n_experts = n_experts;
  a.M = M;
  a.top_k = top_k;
  a.ids = ids;
  a.gate = gate;
  a.y = y;
  a.err = err;
  a.plan = reinterpret_cast<int*>(w + L.plan_off);
  a.cnt = reinterpret_cast<int*>(w + L.cnt_off);
  a.Dmax = L.Dmax;
  return launch_args(a, qtype, st);
}

// ---------------------------------------------------------------------------
// The expert FFN of a layer in two launches:
//   1. gate|up: h[p][f] = act((W_gate[e] x_m)[f]) * (W_up[e] x_m)[f] for every
//      routed pair p = (m, j), e = ids[m][j], and hs[m][s] likewise with the
//      shared expert's matrices;
//   2. down: part[p] = W_down[e] h[p], sp[m] = Ws_down hs[m], then
//      y[m] = sum_j g[m][j] part[(m, j)] + sp[m] (slot order, then the shared term).
// h, hs, part and sp live in the workspace; both launches plan the grouping.
// ---------------------------------------------------------------------------
FfnLayout ffn_layout(int64_t H, int64_t F, int64_t SH, int64_t M, int top_k, int n_experts) {
  FfnLayout L;
  const int64_t MK = M * top_k;
  L.Dmax = static_cast<int>(MK < n_experts ? MK : n_experts);
  L.plan_off = 256;
  L.cnt_off = L.plan_off + a256(sizeof(int) * (1 + 2 * static_cast<size_t>(L.Dmax) + 1 + MK));
  L.part_off = L.cnt_off + a256(sizeof(int) * static_cast<size_t>((H + MT_MIN - 1) / MT_MIN));
  L.h_off = L.part_off + a256(sizeof(float) * static_cast<size_t>(MK * H));
  L.hs_off = L.h_off + a256(sizeof(float) * static_cast<size_t>(MK * F));
  L.sp_off = L.hs_off + a256(sizeof(float) * static_cast<size_t>(M * SH));
  L.bytes = L.sp_off + a256(sizeof(float) * static_cast<size_t>(SH > 0 ? M * H : 0));
  return L;
}

bool ffn_supported(int type_gu, int type_dn, int64_t H, int64_t F, int64_t SH, int64_t M, int top_k, int n_experts) {
  auto fits = [](int qt, int64_t K, int mats) {
    const int BB = block_bytes_of(qt);
    const int64_t row_bytes = ((K + 255) / 256) * BB;
    return BB && (K + 255) / 256 <= 64 && mats * (16 * row_bytes + 48) <= kMaxTileBytes;
  };
  return M * top_k <= kMaxPairs && n_experts <= kMaxExperts && fits(type_gu, H, 2) && fits(type_dn, F, 1) &&
         (SH == 0 || fits(type_dn, SH, 1));
}

cudaError_t launch_moe_ffn(const FfnWeights& fw, const int32_t* ids, const float* gate, const void* x, int x_bf16,
                           float* y, int64_t H, int M, int top_k, void* ws, cudaStream_t st) {
  const FfnLayout L = ffn_layout(H, fw.F, fw.SH, M, top_k, fw.n_experts);
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* h = reinterpret_cast<float*>(w + L.h_off);
  float* hs = reinterpret_cast<float*>(w + L.hs_off);
  MoeArgs a = {};
  a.n_experts = fw.n_experts;
  a.M = M;
  a.top_k = top_k;
  a.ids = ids;
  a.err = static_cast<int*>(ws);
  a.plan = reinterpret_cast<int*>(w + L.plan_off);
  a.cnt = reinterpret_cast<int*>(w + L.cnt_off);
  a.Dmax = L.Dmax;
  a.nseg = fw.SH > 0 ? 2 : 1;
  a.tgroups = (M + kSharedTokens - 1) / kSharedTokens;

  // 1. gate|up with the activation
  fill_seg(a.seg[0], fw.type_gu, fw.W_gate, fw.W_up, fw.F, static_cast<int>(H), x, 0, h);
  if (fw.SH > 0) fill_seg(a.seg[1], fw.type_gu, fw.Ws_gate, fw.Ws_up, fw.SH, static_cast<int>(H), x, 0, hs);
  a.gu = 1;
  a.act = fw.act;
  a.type = fw.type_gu;
  a.x_bf16 = x_bf16;
  a.gate = nullptr;
  a.y = nullptr;
  a.G = 0;
  cudaError_t e = launch_args(a, fw.type_gu, st);
  if (e != cudaSuccess) return e;

  // 2. down with the gated combine (and the shared term); the ids were read
  //    by launch 1 after its own wait, so they are complete before launch 1
  //    releases this one
  a.ids_ready = 1;
  fill_seg(a.seg[0], fw.type_dn, fw.W_down, nullptr, H, static_cast<int>(fw.F), h, 1,
           reinterpret_cast<float*>(w + L.part_off));
  if (fw.SH > 0)
    fill_seg(a.seg[1], fw.type_dn, fw.Ws_down, nullptr, H, static_cast<int>(fw.SH), hs, 0,
             reinterpret_cast<float*>(w + L.sp_off));
  a.gu = 0;
  a.type = fw.type_dn;
  a.x_bf16 = 0;  // h is fp32
  a.gate = gate;
  a.y = y;
  a.G = a.seg[0].rt;
  if (fw.SH > 0 && a.seg[1].rt < a.G) a.G = a.seg[1].rt;  // tile heights are powers of two: the smaller divides
  return launch_args(a, fw.type_dn, st);
}

cudaError_t launch_moe(int qtype, const void* W, int n_experts, const int32_t* ids, const float* gate,
                       const void* x, int x_bf16, int x_per_slot, float* y, int64_t N, int K, int M, int top_k,
                       void* ws, cudaStream_t st) {
  return launch_moe_err(qtype, W, n_experts, ids, gate, x, x_bf16, x_per_slot, y, N, K, M, top_k, ws,
                        static_cast<int*>(ws), st);
}

// ---------------------------------------------------------------------------
// Allocation-free variant: the same kernel with its scratch in a file-scope
// device array instead of a caller workspace.  For callers that cannot
// allocate device memory at all -- a plain C host embedding libkq with no
// device allocator of its own, or a decode loop that must not allocate -- and
// so cannot provide the workspace kq_moe_matvec needs.  The array keeps what
// the last call left; its layout depends on the call's shape, so a gated call
// first clears its own arrival counters (one stream-ordered memset, no
// allocation).  Bad ids are reported in the library's device error word
// (kq_device_error).  One array per device: calls that overlap in time (any
// stream, any host thread) race on it and must not be issued.
// ---------------------------------------------------------------------------
namespace {
constexpr size_t kMoeStaticScratch = 2u << 20;  // bytes: M*top_k*N <= ~500K outputs
static __device__ __align__(256) uint8_t g_moe_scratch[kMoeStaticScratch];
uint8_t* g_moe_scratch_ptr[64] = {nullptr};
}  // namespace

size_t moe_static_scratch_bytes() { return kMoeStaticScratch; }

cudaError_t launch_moe_static(int qtype, const void* W, int n_experts, const int32_t* ids, const float* gate,
                              const void* x, int x_bf16, int x_per_slot, float* y, int64_t N, int K, int M,
                              int top_k, cudaStream_t st) {
  const MoeLayout L = moe_layout(N, M, top_k, n_experts);
  if (L.bytes > kMoeStaticScratch) return cudaErrorInvalidValue;
  const int dev = current_device_id();
  if (!g_moe_scratch_ptr[dev]) {  // once per device, with that device current
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_moe_scratch);
    if (e != cudaSuccess) return e;
    g_moe_scratch_ptr[dev] = static_cast<uint8_t*>(p);
  }
  if (gate) {  // the counters of this shape start at zero whatever an earlier call of another shape left there
    const cudaError_t e = cudaMemsetAsync(g_moe_scratch_ptr[dev] + L.cnt_off, 0, sizeof(int) * L.ntiles, st);
    if (e != cudaSuccess) return e;
  }
  return launch_moe_err(qtype, W, n_experts, ids, gate, x, x_bf16, x_per_slot, y, N, K, M, top_k,
                        g_moe_scratch_ptr[dev], device_error_ptr(), st);
}

}  // namespace kq
