// kq_route.cu -- the MoE router: top-k over each token's expert logits, the
// gate weights as a softmax over the selected logits, and (optionally) the
// grouping of the (token, slot) pairs by expert that kq_moe_matvec plans.
//
// "GGUF in transformers", section "Reusing ggml's Metal kernels": a top-k
// kernel combines the softmax and the top-k selection of the MoE router.
// "ANE Fieldfare" README, "How it works": each token's router picks 8 of 128
// experts; "Speculative decoding": a planning kernel on the GPU groups the
// tokens of a verify block by expert.
//
// Reading (the pages give no formula): the k largest logits of a token in
// descending order, ties to the lower expert index, a NaN below every number;
// gate_j = exp(l_j - l_0) / sum_i exp(l_i - l_0) over the selected logits
// (which equals a softmax over all experts renormalized over the selected ones).
//
// One CTA: warp w routes tokens w, w + 16, ...; each round of a token's
// selection is one warp-wide argmax over the lanes' own best logits not yet
// taken (see select_token), so a round costs one warp reduction.  The
// grouping then runs on the ids in shared memory: presence bits, ranks by a
// warp prefix count, per-rank counts and offsets, and a stable placement of
// the pairs in (token, slot) order.
#include "kq_internal.h"

namespace kq {
namespace {

constexpr int RW = 16;  // warps
constexpr int RTH = RW * 32;
constexpr int kRouteMaxPairs = 512;
constexpr int kRouteMaxExperts = 4096;

struct RouteSmem {
  uint32_t taken[RW][kRouteMaxExperts / 32];  // per warp: experts chosen for its current token
  int ids[kRouteMaxPairs];
  uint32_t bits[kRouteMaxExperts / 32];
  int wordpre[kRouteMaxExperts / 32];
  int expert_of[kRouteMaxPairs];
  int off[kRouteMaxPairs + 1];
  int run[kRouteMaxPairs];
  int pairs[kRouteMaxPairs];
  int misc[4];  // 0: distinct experts
};

// (a, ia) ranks above (b, ib): the larger number, a NaN below every number,
// ties (equal numbers, or two NaNs) to the lower index.
__device__ __forceinline__ bool ranks_above(float a, int ia, float b, int ib) {
  const bool an = isnan(a), bn = isnan(b);
  if (an != bn) return bn;
  if (!an && a != b) return a > b;
  return ia < ib;
}

// The warp-wide winner of (v, i) over the lanes.
__device__ __forceinline__ void warp_best(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    const int oi = __shfl_xor_sync(0xFFFFFFFFu, i, o);
    if (ranks_above(ov, oi, v, i)) { v = ov; i = oi; }
  }
}

// One token's selection.  Lane l owns experts l, l + 32, ...; it keeps the
// best of its own not-yet-taken experts, so a round is one warp reduction of
// the 32 lane bests, after which only the winning lane rescans its own
// experts.  EPL > 0: the lane's EPL logits stay in registers (E <= 32 * EPL);
// EPL == 0: they are re-read from the row, with a taken bitmask in shared
// memory.  Returns the lane's selected logit (lane j < top_k: the j-th).
template <int EPL>
__device__ __forceinline__ float select_token(const float* __restrict__ row, int E, int top_k, int lane,
                                              uint32_t* taken, int* ids_s, int* ids_g) {
  const float kNaN = __int_as_float(0x7FC00000);
  float v[EPL > 0 ? EPL : 1];
  uint32_t tk = 0u;  // EPL > 0: bit i = expert lane + 32 i taken
  if constexpr (EPL > 0) {
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      v[i] = e < E ? row[e] : kNaN;
    }
  } else {
    for (int w = lane; w < ((E + 31) >> 5); w += 32) taken[w] = 0u;
    __syncwarp();
  }
  auto local_best = [&](float& bv, int& bi) {
    bv = kNaN;
    bi = E;  // sentinel: every expert ranks above it
    if constexpr (EPL > 0) {
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((tk >> i) & 1u) && ranks_above(v[i], e, bv, bi)) { bv = v[i]; bi = e; }
      }
    } else {
      for (int e = lane; e < E; e += 32) {
        if ((taken[e >> 5] >> (e & 31)) & 1u) continue;
        const float x = row[e];
        if (ranks_above(x, e, bv, bi)) { bv = x; bi = e; }
      }
    }
  };
  float lbv;
  int lbi;
  local_best(lbv, lbi);
  float sel_v = 0.0f;
  for (int j = 0; j < top_k; ++j) {
    float bv = lbv;
    int bi = lbi;
    warp_best(bv, bi);  // every lane holds the winner; bi < E since top_k <= E
    if (lane == j) sel_v = bv;
    if ((bi & 31) == lane) {  // the owner records it, takes it out and finds its next best
      ids_s[j] = bi;
      ids_g[j] = bi;
      if constexpr (EPL > 0) {
        tk |= 1u << (bi >> 5);
      } else {
        taken[bi >> 5] |= 1u << (bi & 31);
      }
      local_best(lbv, lbi);
    }
  }
  __syncwarp();
  return sel_v;
}

template <int EPL>
__global__ void __launch_bounds__(RTH, 1) route_kernel(const float* __restrict__ logits, int M, int E, int top_k,
                                                       int* __restrict__ ids_out, float* __restrict__ gate_out,
                                                       int* plan, int Dmax) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  RouteSmem& sm = *reinterpret_cast<RouteSmem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nwords = (E + 31) >> 5;
  pdl_wait();  // the logits come from an earlier kernel
  pdl_launch_dependents();

  for (int m = warp; m < M; m += RW) {
    const int64_t base = static_cast<int64_t>(m) * top_k;
    const float sel_v = select_token<EPL>(logits + static_cast<int64_t>(m) * E, E, top_k, lane, sm.taken[warp],
                                          sm.ids + base, ids_out + base);
    // gates: exp(l_j - l_0) / sum, the sum in slot order
    const float l0 = __shfl_sync(0xFFFFFFFFu, sel_v, 0);
    const float ex = lane < top_k ? expf(sel_v - l0) : 0.0f;
    float sum = 0.0f;
    for (int j = 0; j < top_k; ++j) sum += __shfl_sync(0xFFFFFFFFu, ex, j);
    if (lane < top_k) gate_out[base + lane] = ex / sum;
  }
  if (!plan) return;

  // ---- grouping of the pairs by expert (the plan kq_moe_matvec leaves in its workspace)
  __syncthreads();
  const int MK = M * top_k;
  for (int i = tid; i < nwords; i += RTH) sm.bits[i] = 0u;
  __syncthreads();
  for (int i = tid; i < MK; i += RTH) atomicOr(&sm.bits[sm.ids[i] >> 5], 1u << (sm.ids[i] & 31));
  __syncthreads();
  if (warp == 0) {
    int base = 0;
    for (int w0 = 0; w0 < nwords; w0 += 32) {
      const int w = w0 + lane;
      const int cnt = w < nwords ? __popc(sm.bits[w]) : 0;
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
      }
      if (w < nwords) sm.wordpre[w] = base + incl - cnt;
      base += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (lane == 0) sm.misc[0] = base;
  }
  __syncthreads();
  const int D = sm.misc[0];
  auto rank_of = [&](int id) {
    return sm.wordpre[id >> 5] + __popc(sm.bits[id >> 5] & ((1u << (id & 31)) - 1u));
  };
  for (int id = tid; id < E; id += RTH)
    if ((sm.bits[id >> 5] >> (id & 31)) & 1u) sm.expert_of[rank_of(id)] = id;
  for (int r = tid; r < D; r += RTH) sm.run[r] = 0;
  __syncthreads();
  for (int i = tid; i < MK; i += RTH) atomicAdd(&sm.run[rank_of(sm.ids[i])], 1);
  __syncthreads();
  if (warp == 0) {
    int base = 0;
    for (int r0 = 0; r0 < D; r0 += 32) {  // offsets: exclusive prefix of the counts
      const int r = r0 + lane;
      const int cnt = r < D ? sm.run[r] : 0;
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
      }
      if (r < D) { sm.off[r] = base + incl - cnt; sm.run[r] = 0; }
      base += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (lane == 0) sm.off[D] = base;
    __syncwarp();
    // stable placement in (token, slot) order: lanes of a chunk with the same
    // rank take consecutive places; the lowest of them advances the count
    for (int i0 = 0; i0 < MK; i0 += 32) {
      const int i = i0 + lane;
      const int r = i < MK ? rank_of(sm.ids[i]) : -1 - lane;
      const uint32_t same = __match_any_sync(0xFFFFFFFFu, r);
      const uint32_t below = same & ((1u << lane) - 1u);
      if (i < MK) sm.pairs[sm.off[r] + sm.run[r] + __popc(below)] = i;
      __syncwarp();
      if (i < MK && below == 0) sm.run[r] += __popc(same);
      __syncwarp();
    }
  }
  __syncthreads();
  for (int r = tid; r < D; r += RTH) { plan[1 + r] = sm.expert_of[r]; plan[1 + Dmax + r] = sm.off[r]; }
  for (int i = tid; i < MK; i += RTH) plan[2 + 2 * Dmax + i] = sm.pairs[i];
  if (tid == 0) { plan[0] = D; plan[1 + Dmax + D] = MK; }
}

}  // namespace

bool route_supported(int64_t M, int E, int top_k) {
  return M * top_k <= kRouteMaxPairs && E <= kRouteMaxExperts && top_k >= 1 && top_k <= 32 && top_k <= E;
}

size_t route_plan_bytes(int64_t M, int top_k, int E) {
  const int64_t MK = M * top_k;
  const int64_t Dmax = MK < E ? MK : E;
  return 256 + sizeof(int) * static_cast<size_t>(2 + 2 * Dmax + MK);
}

template <int EPL>
cudaError_t launch_route_t(const float* logits, int M, int E, int top_k, int* ids, float* gate, int* plan, int Dmax,
                           cudaStream_t st) {
  static bool smem_set[64] = {false};
  const int dev = current_device_id();
  if (!smem_set[dev]) {
    const cudaError_t e =
        cudaFuncSetAttribute(route_kernel<EPL>, cudaFuncAttributeMaxDynamicSharedMemorySize, sizeof(RouteSmem));
    if (e != cudaSuccess) return e;
    smem_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(RTH);
  cfg.dynamicSmemBytes = sizeof(RouteSmem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, route_kernel<EPL>, logits, M, E, top_k, ids, gate, plan, Dmax);
}

cudaError_t launch_route(const float* logits, int M, int E, int top_k, int* ids, float* gate, void* ws,
                         cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  const int MK = M * top_k;
  const int Dmax = MK < E ? MK : E;
  int* plan = ws ? reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + 256) : nullptr;
  if (E <= 32) return launch_route_t<1>(logits, M, E, top_k, ids, gate, plan, Dmax, st);
  if (E <= 64) return launch_route_t<2>(logits, M, E, top_k, ids, gate, plan, Dmax, st);
  if (E <= 128) return launch_route_t<4>(logits, M, E, top_k, ids, gate, plan, Dmax, st);
  if (E <= 256) return launch_route_t<8>(logits, M, E, top_k, ids, gate, plan, Dmax, st);
  return launch_route_t<0>(logits, M, E, top_k, ids, gate, plan, Dmax, st);
}

}  // namespace kq
