// kq_moe.cu -- routed-expert products: every selected expert's rows are read
// from memory once and applied to all (token, slot) pairs routed to it.
//
// "GGUF in transformers", section "Reusing ggml's Metal kernels": the kernel
// reads the packed weights directly, including only the experts an MoE layer
// selected.  "ANE Fieldfare" README, "How it works": each token's router
// picks 8 of 128 experts; "Speculative decoding": a planning step groups the
// tokens of a verify block by expert so each expert is read once.
//
// One launch, grid (row tile, distinct-expert rank d):
//  * grouping (every CTA, in shared memory): the routed ids are checked
//    (an id outside [0, n_experts) is recorded in the workspace error word and
//    its pair dropped), the distinct experts are ranked in ascending id order,
//    and CTA (tile, d) takes the d-th one, e, with its pairs (token m, slot j)
//    in (m, j) order.  The CTAs of tile 0 also write this plan to the
//    workspace (expert of each rank, offsets, pairs) for inspection;
//  * the CTA copies its tile of expert e (whole rows, as large as fits in
//    100 KB: 256, 128 or 64 rows, a quad of lanes per 4, 2 or 1 of them; wider
//    rows 32 or 16 rows, 2 or 4 quads per row) with one TMA bulk copy, then for
//    each pair stages that pair's x as block-float limbs and applies the rows
//    to it with the lane cores of kq_lane.cuh;
//  * if no routed id is valid at all, the gated outputs are zero (empty sums);
//  * without gate weights the result of pair (m, j) is row j of token m's
//    output block (y[m][j][n]); with gate weights it goes to the workspace and
//    the last CTA to finish the tile (arrival counter) writes
//    y[m][n] = sum_j g[m][j] * part[m][j][n] in slot order (deterministic).
#include "kq_lane.cuh"

namespace kq {

using namespace lane;

namespace {

constexpr int MT_MIN = 16;      // rows per tile at the most quads per row (sizes the tile counters)
constexpr int kForcePhases = 0; // 0: quads per row chosen per shape
constexpr int kForceRows = 0;   // 0: rows per quad chosen per shape
constexpr int MW = 8;           // warps
constexpr int MTH = MW * 32;
constexpr int kMaxPairs = 512;  // M * top_k
constexpr int kMaxExperts = 4096;
constexpr int64_t kMaxTileBytes = 100 * 1024;  // 32 rows at most (API limit)

struct MoeArgs {
  const uint8_t* W;
  int64_t expert_bytes;  // N * row_bytes
  int64_t row_bytes;
  int64_t N;
  int K, nb, type, x_bf16, x_per_slot;
  int n_experts, M, top_k, ntiles;
  const int32_t* ids;
  const float* gate;
  const void* x;
  float* y;
  int* err;   // workspace error word
  int* plan;  // workspace plan: D, expert_of[Dmax], offset[Dmax + 1], pairs[M * top_k]
  int* cnt;   // per-tile arrival counters (gate case)
  float* part;
  int Dmax;
  int nph, rq, rt;  // quads per row (block phases), rows per quad, rows per tile = 8 * MW * rq / nph
};

struct MoeSmem {
  int ids[kMaxPairs];
  uint32_t bits[kMaxExperts / 32];
  int pairs[kMaxPairs];
  int misc[8];  // 0: e, 1: D, 2: np, 3: offset of e, 4: valid pairs, 5: last
};

__host__ __device__ inline size_t moe_ximg_offset() { return (sizeof(MoeSmem) + 16 + 127) & ~size_t(127); }

// Row sums of one pair over the tile for the RQ rows of this quad (rows
// rp, rp + rstride, ...; nph quads per row, the quad of phase ph taking blocks
// ph, ph + nph, ...): each block's x slice is loaded once for all RQ rows.
template <int QT, int NL, int RQ>
__device__ __forceinline__ void pair_rows(uint32_t rp, uint32_t rstride, int nb, const XImg& xi, int ph, int nph,
                                          int c, const ScaleLane& sl, float (&acc)[4]) {
  constexpr int BB = Fmt<QT>::BYTES;
  const int xoff = (QT == T_Q6_K) ? (40 * (c >> 1) + 4 * (c & 1)) : 20 * c;
#pragma unroll
  for (int i = 0; i < RQ; ++i) acc[i] = 0.0f;
  for (int b = ph; b < nb; b += nph) {
    XSlice<NL> X;
    load_slice<QT, NL>(xi.limb_s + 4 * (b * XWB + xoff), 4 * xi.plane, X);
    const float s = __uint_as_float(lds32(xi.scale_s + 4 * (2 * b + (c >> 1))));
    if constexpr (QT == T_Q6_K) {
      const uint4 sv = lds128(xi.si16q_s + 4 * (16 * b + 4 * c));
      const int4 si = make_int4(static_cast<int>(sv.x), static_cast<int>(sv.y), static_cast<int>(sv.z),
                                static_cast<int>(sv.w));
#pragma unroll
      for (int i = 0; i < RQ; ++i) acc[i] = core_q6<NL>(rp + i * rstride + b * BB, X, si, s, c, acc[i]);
    } else {
      const uint2 sv = lds64(xi.si32_s + 4 * (8 * b + 2 * c));
      const int2 si = make_int2(static_cast<int>(sv.x), static_cast<int>(sv.y));
#pragma unroll
      for (int i = 0; i < RQ; ++i) acc[i] = core_q45<QT, NL>(rp + i * rstride + b * BB, X, si, s, c, sl, acc[i]);
    }
  }
#pragma unroll
  for (int i = 0; i < RQ; ++i) {
    float v = acc[i];
    v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, 1));
    v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, 2));
    for (int o = 4; o < 4 * nph; o <<= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    acc[i] = v;
  }
}

template <int QT, int NL>
__global__ void __launch_bounds__(MTH) moe_kernel(const __grid_constant__ MoeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  MoeSmem& sm = *reinterpret_cast<MoeSmem*>(smem + 16);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x, d = blockIdx.y;
  const int MK = a.M * a.top_k;
  const XImg xi = ximg_at(smem + moe_ximg_offset(), a.nb, NL);
  uint8_t* tile_buf = smem + moe_ximg_offset() + ((ximg_bytes(a.nb, NL) + 127) & ~size_t(127));

  pdl_wait();  // routed ids, gates and x come from earlier kernels
  pdl_launch_dependents();

  // ---- grouping: validated ids, presence bits, the d-th distinct expert
  const int nwords = (a.n_experts + 31) >> 5;
  for (int i = tid; i < nwords; i += MTH) sm.bits[i] = 0;
  __syncthreads();
  for (int i = tid; i < MK; i += MTH) {
    int id = a.ids[i];
    if (id < 0 || id >= a.n_experts) {
      record_error(a.err, DEV_ERR_EXPERT_ID);
      id = -1;
    } else {
      atomicOr(&sm.bits[id >> 5], 1u << (id & 31));
    }
    sm.ids[i] = id;
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
  const int e = sm.misc[0], D = sm.misc[1];
  if (D == 0 && a.gate && d == 0) {  // no valid pair at all: the gated outputs of this tile are zero
    const int64_t r0 = static_cast<int64_t>(tile) * a.rt;
    const int nrows = static_cast<int>(min_i64(a.rt, a.N - r0));
    for (int i = tid; i < a.M * nrows; i += MTH)
      a.y[static_cast<int64_t>(i / nrows) * a.N + r0 + i % nrows] = 0.0f;
  }
  if (e < 0) return;  // fewer distinct experts than this rank

  // ---- the expert's tile: one bulk copy of whole rows
  const int64_t r0 = static_cast<int64_t>(tile) * a.rt;
  const int nrows = static_cast<int>(min_i64(a.rt, a.N - r0));
  const uint8_t* src = a.W + e * a.expert_bytes + r0 * a.row_bytes;
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(src);
  const uintptr_t as = s0 & ~uintptr_t(15), ae = (s0 + nrows * a.row_bytes + 15) & ~uintptr_t(15);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(ae - as));
    bulk_g2s_hint(tile_buf, reinterpret_cast<const void*>(as), static_cast<uint32_t>(ae - as), bar,
                  l2_evict_first_policy());  // an expert tile is read once per call
  }

  // ---- the expert's pairs in (m, slot) order, and its plan offset
  if (warp == 0) {
    int np = 0, below = 0, valid = 0;
    for (int i0 = 0; i0 < MK; i0 += 32) {
      const int i = i0 + lane;
      const int id = i < MK ? sm.ids[i] : -1;
      const uint32_t mine = __ballot_sync(0xFFFFFFFFu, id == e);
      if (id == e) sm.pairs[np + __popc(mine & ((1u << lane) - 1))] = i;
      np += __popc(mine);
      below += __popc(__ballot_sync(0xFFFFFFFFu, id >= 0 && id < e));
      valid += __popc(__ballot_sync(0xFFFFFFFFu, id >= 0));
    }
    if (lane == 0) { sm.misc[2] = np; sm.misc[3] = below; sm.misc[4] = valid; }
  }
  __syncthreads();
  const int np = sm.misc[2];
  if (tile == 0) {  // the plan, for inspection
    for (int j = tid; j < np; j += MTH) a.plan[1 + 2 * a.Dmax + 1 + sm.misc[3] + j] = sm.pairs[j];
    if (tid == 0) {
      a.plan[1 + d] = e;
      a.plan[1 + a.Dmax + d] = sm.misc[3];
      if (d == 0) { a.plan[0] = D; a.plan[1 + a.Dmax + D] = sm.misc[4]; }
    }
  }

  // ---- apply the rows to every pair: quad rows rq0 + i * (64 / nph), i < rq
  const int quad = lane >> 2, c = lane & 3;
  const int rq0 = warp * (8 / a.nph) + quad / a.nph, ph = quad % a.nph;
  const int rstep = 8 * MW / a.nph;
  const ScaleLane sl = scale_lane(c);
  const uint32_t rp = smem_u32(tile_buf) + static_cast<uint32_t>(s0 - as) + static_cast<uint32_t>(rq0 * a.row_bytes);
  const uint32_t rstride = static_cast<uint32_t>(rstep * a.row_bytes);
  bool ok = true;
  for (int j = 0; j < np; ++j) {
    const int pr = sm.pairs[j];
    const int m = pr / a.top_k;
    const int64_t xrow = a.x_per_slot ? pr : m;
    const void* xp = a.x_bf16 ? static_cast<const void*>(static_cast<const uint16_t*>(a.x) + xrow * a.K)
                              : static_cast<const void*>(static_cast<const float*>(a.x) + xrow * a.K);
    __syncthreads();  // the previous pair is done with the x image
    stage_x<NL, MTH>(xp, NL == 2, a.K, a.nb, xi, tid);
    __syncthreads();
    if (j == 0) ok = mbar_wait(bar, 0, a.err);
    float v[4];
    if (a.rq == 4) pair_rows<QT, NL, 4>(rp, rstride, a.nb, xi, ph, a.nph, c, sl, v);
    else if (a.rq == 2) pair_rows<QT, NL, 2>(rp, rstride, a.nb, xi, ph, a.nph, c, sl, v);
    else pair_rows<QT, NL, 1>(rp, rstride, a.nb, xi, ph, a.nph, c, sl, v);
    if (ok && c == 0 && ph == 0) {
      float* out = (a.gate ? a.part : a.y) + static_cast<int64_t>(pr) * a.N + r0;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (i < a.rq && rq0 + i * rstep < nrows) out[rq0 + i * rstep] = v[i];
    }
  }
  if (np == 0 && tid == 0) ok = mbar_wait(bar, 0, a.err);  // the copy must land before the CTA exits
  if (!a.gate) return;

  // ---- gate-weighted combine by the tile's last CTA
  __threadfence();
  __syncthreads();
  if (tid == 0) sm.misc[5] = (atomicAdd(&a.cnt[tile], 1) == D - 1) ? 1 : 0;
  __syncthreads();
  if (!sm.misc[5]) return;
  __threadfence();
  for (int i = tid; i < a.M * nrows; i += MTH) {
    const int m = i / nrows, r = i - m * nrows;
    const float* pp = a.part + static_cast<int64_t>(m) * a.top_k * a.N + r0 + r;
    const int* id = sm.ids + m * a.top_k;
    const float* g = a.gate + m * a.top_k;
    float v = 0.0f;
    int j = 0;
    for (; j + 4 <= a.top_k; j += 4) {  // four loads in flight, applied in slot order; dropped pairs skipped
      float p[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) p[q] = id[j + q] >= 0 ? __ldcg(pp + static_cast<int64_t>(j + q) * a.N) : 0.0f;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (id[j + q] >= 0) v = __fmaf_rn(g[j + q], p[q], v);
    }
    for (; j < a.top_k; ++j)
      if (id[j] >= 0) v = __fmaf_rn(g[j], __ldcg(pp + static_cast<int64_t>(j) * a.N), v);
    a.y[static_cast<int64_t>(m) * a.N + r0 + r] = v;
  }
  if (tid == 0) a.cnt[tile] = 0;  // ready for the next call
}

template <int QT, int NL>
cudaError_t launch_moe_t(const MoeArgs& a, size_t smem, cudaStream_t st) {
  static bool smem_set[64] = {false};
  const int dev = current_device_id();
  if (!smem_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(moe_kernel<QT, NL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kMaxSmemPerBlock);
    if (e != cudaSuccess) return e;
    smem_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.ntiles, a.Dmax);
  cfg.blockDim = dim3(MTH);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_kernel<QT, NL>, a);
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
  if (kForcePhases) nph = kForcePhases;
  if (kForceRows) rq = kForceRows;
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

cudaError_t launch_moe_err(int qtype, const void* W, int n_experts, const int32_t* ids, const float* gate,
                           const void* x, int x_bf16, int x_per_slot, float* y, int64_t N, int K, int M, int top_k,
                           void* ws, int* err, cudaStream_t st) {
  const MoeLayout L = moe_layout(N, M, top_k, n_experts);
  uint8_t* w = static_cast<uint8_t*>(ws);
  MoeArgs a = {};
  a.nb = (K + 255) / 256;
  a.row_bytes = static_cast<int64_t>(a.nb) * block_bytes_of(qtype);
  a.N = N;
  a.expert_bytes = N * a.row_bytes;
  a.W = static_cast<const uint8_t*>(W);
  a.K = K;
  a.type = qtype;
  a.x_bf16 = x_bf16;
  a.x_per_slot = x_per_slot;
  a.n_experts = n_experts;
  a.M = M;
  a.top_k = top_k;
  a.ids = ids;
  a.gate = gate;
  a.x = x;
  a.y = y;
  a.err = err;
  a.plan = reinterpret_cast<int*>(w + L.plan_off);
  a.cnt = reinterpret_cast<int*>(w + L.cnt_off);
  a.part = reinterpret_cast<float*>(w + L.part_off);
  a.Dmax = L.Dmax;
  const int NL = x_bf16 ? 2 : 3;
  moe_tile_shape(a.row_bytes, a.nph, a.rq);
  a.rt = 8 * MW * a.rq / a.nph;
  a.ntiles = static_cast<int>((N + a.rt - 1) / a.rt);
  const size_t smem = moe_ximg_offset() + ((ximg_bytes(a.nb, NL) + 127) & ~size_t(127)) +
                      static_cast<size_t>(a.rt * a.row_bytes + 32);
  if (smem > static_cast<size_t>(kMaxSmemPerBlock)) return cudaErrorNotSupported;
  switch (qtype * 4 + NL) {
    case T_Q4_K * 4 + 2: return launch_moe_t<T_Q4_K, 2>(a, smem, st);
    case T_Q4_K * 4 + 3: return launch_moe_t<T_Q4_K, 3>(a, smem, st);
    case T_Q5_K * 4 + 2: return launch_moe_t<T_Q5_K, 2>(a, smem, st);
    case T_Q5_K * 4 + 3: return launch_moe_t<T_Q5_K, 3>(a, smem, st);
    case T_Q6_K * 4 + 2: return launch_moe_t<T_Q6_K, 2>(a, smem, st);
    case T_Q6_K * 4 + 3: return launch_moe_t<T_Q6_K, 3>(a, smem, st);
    default: return cudaErrorInvalidValue;
  }
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
// so cannot provide the workspace kq_moe_matvec needs.  The array is zero at
// module load; the arrival counters return to zero after every call; bad ids
// are reported in the library's device error word (kq_device_error).  One
// array per device: calls that overlap in time (any stream, any host thread)
// race on it and must not be issued.
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
  if (moe_layout(N, M, top_k, n_experts).bytes > kMoeStaticScratch) return cudaErrorInvalidValue;
  const int dev = current_device_id();
  if (!g_moe_scratch_ptr[dev]) {  // once per device, with that device current
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_moe_scratch);
    if (e != cudaSuccess) return e;
    g_moe_scratch_ptr[dev] = static_cast<uint8_t*>(p);
  }
  return launch_moe_err(qtype, W, n_experts, ids, gate, x, x_bf16, x_per_slot, y, N, K, M, top_k,
                        g_moe_scratch_ptr[dev], device_error_ptr(), st);
}

}  // namespace kq
