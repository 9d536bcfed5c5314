// kq_gemv.cu -- host side of the one-token products (kq_gemv_kernel.cuh):
// a single product (its kernels instantiated per format in kq_gemv_q4k.cu,
// kq_gemv_q5k.cu, kq_gemv_q6k.cu, kq_gemv_ia4.cu), and programs of products
// run by one persistent launch (planned here, kernels instantiated here).
#include "kq_gemv_kernel.cuh"

namespace kq {

namespace {
// Dispatch of a single product to its format's translation unit.
cudaError_t launch_single(int qtype, int XK, int MT, int R, ProgArgs& a, const LaunchGeom& g, cudaStream_t st,
                          bool pdl) {
  switch (qtype) {
    case T_Q4_K: return launch_single_q4k(XK, MT, R, a, g.S, g.slot, g.smem, st, pdl);
    case T_Q5_K: return launch_single_q5k(XK, MT, R, a, g.S, g.slot, g.smem, st, pdl);
    case T_Q6_K: return launch_single_q6k(XK, MT, R, a, g.S, g.slot, g.smem, st, pdl);
    case T_IA4: return launch_single_ia4(XK, MT, R, a, g.S, g.slot, g.smem, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

cudaError_t launch_matvec1(int qtype, const void* W, const void* x, int x_bf16, float* y, int64_t N, int K,
                           cudaStream_t stream, bool pdl, int M) {
  if (N == 0) return cudaSuccess;
  if (M < 1 || M > kMaxTokens1 || (M > 1 && !x_bf16)) return cudaErrorNotSupported;
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
  if (!plan_op(o, num_sms(), false, kSlotCap, true)) return cudaErrorNotSupported;
  LaunchGeom g;
  const int nimg = x_bf16 ? M : 2;
  if (!ring_geom(stage_bytes(o), o.nb, nimg, g, M)) return cudaErrorNotSupported;
  a.ops = nullptr;
  a.n_ops = 1;
  a.nb_max = o.nb;
  a.nimg = nimg;
  a.barrier = nullptr;
  a.err = device_error_ptr();
  // the instantiation for (format, x dtype, tokens, rows per quad); fp32 x takes one token
  return launch_single(qtype, x_bf16 ? 1 : 2, M, o.R, a, g, stream, pdl);
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

// K-parts of the ops of one stage (ops [i, j) between grid barriers): their
// units are dealt to the CTAs round-robin, continuing from op to op, so the
// parts are chosen together -- every combination of 1, 2, 4 or 8 parts per op
// (where the op may split) is dealt out on the host and the one whose busiest
// CTA has the fewest weight bytes (plus a fixed cost per unit) is kept.
constexpr int64_t kUnitCost = 12288;  // bytes-equivalent of a unit's fixed work (waits, reduction)

void balance_stage(const ProgOpDesc* d, int n_ops, KqOp* ops, int i, int j, int G) {
  int cand[8][4], nc[8];
  const int n = j - i;
  if (n > 8) return;
  int64_t combos = 1;
  for (int k = 0; k < n; ++k) {
    const KqOp& o = ops[i + k];
    nc[k] = 0;
    cand[k][nc[k]++] = 1;
    if (split_allowed(d, n_ops, i + k))
      for (int ks = 2; ks <= 8; ks *= 2)
        if (split_ok(o.nb, ks)) cand[k][nc[k]++] = ks;
    combos *= nc[k];
  }
  if (combos > 4096) return;
  std::vector<int64_t> load(G);
  int64_t best = -1;
  int pick[8] = {0}, cur[8] = {0};
  for (int64_t cmb = 0; cmb < combos; ++cmb) {
    int64_t r = cmb;
    for (int k = 0; k < n; ++k) { cur[k] = cand[k][r % nc[k]]; r /= nc[k]; }
    std::fill(load.begin(), load.end(), 0);
    int64_t rot = 0;
    for (int k = 0; k < n; ++k) {
      const KqOp& o = ops[i + k];
      const int KS = cur[k], kpb = (o.nb + KS - 1) / KS, BB = block_bytes_of(o.type);
      const int64_t units = static_cast<int64_t>(o.ntiles) * KS;
      for (int64_t u = 0; u < units; ++u) {
        const int kp = static_cast<int>(u % KS);
        const int blocks = std::min(o.nb, (kp + 1) * kpb) - kp * kpb;
        load[(u + rot) % G] += static_cast<int64_t>(8 * o.R) * blocks * BB + kUnitCost;
      }
      rot += units;
    }
    const int64_t mx = *std::max_element(load.begin(), load.end());
    if (best < 0 || mx < best) {
      best = mx;
      for (int k = 0; k < n; ++k) pick[k] = cur[k];
    }
  }
  for (int k = 0; k < n; ++k) {
    KqOp& o = ops[i + k];
    if (o.KS != pick[k]) set_split(o, pick[k], op_kcmax(o, kSlotCap));
  }
}

// Plan every op of a program; false if some op cannot run on this path.
// K is split only in programs with grid barriers (a program without them is
// an ordinary launch that overlaps its neighbours and needs no final barrier).
bool plan_prog(const ProgOpDesc* descs, int n_ops, KqOp* ops, size_t* part_bytes) {
  const int G = num_sms();
  bool any_wait = false;
  for (int i = 1; i < n_ops; ++i) any_wait = any_wait || descs[i].wait_previous;
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
    const bool split = any_wait && split_allowed(descs, n_ops, i);
    if (!plan_op(o, G, split, kSlotCap)) return false;
    // a bf16 Q6_K op whose 32-row whole-row stage exceeds the other ops'
    // largest (the 4B sweep's LM head, 67 KB) would set the chain's slot size
    // and leave two slots: 16-row tiles keep it at 34 KB
    if (o.type == T_Q6_K && o.x_bf16 && o.contig && stage_bytes(o) > kSlotCap) {
      KqOp o2 = o;
      if (plan_op(o2, G, split, kSlotCap, false, 2) && o2.contig) o = o2;
    }
    ops[i] = o;
  }
  if (any_wait)
    for (int i = 0; i < n_ops;) {
      int j = i + 1;
      while (j < n_ops && !descs[j].wait_previous) ++j;
      balance_stage(descs, n_ops, ops, i, j, G);
      i = j;
    }
  for (int i = 0; i < n_ops; ++i)
    if (ops[i].KS > 1) pb += align256(static_cast<size_t>(ops[i].ntiles) * ops[i].KS * TT * sizeof(float));
  *part_bytes = pb;
  return true;
}

// Ops that start an x (the first op, or one that waits or reads a new x).
bool starts_x(const ProgOpDesc* descs, int i) {
  return i == 0 || descs[i].wait_previous || descs[i].x != descs[i - 1].x || descs[i].K != descs[i - 1].K ||
         descs[i].x_bf16 != descs[i - 1].x_bf16;
}
size_t xrange_bytes(const ProgOpDesc* descs, int n_ops, int G) {
  size_t n = 0;
  for (int i = 0; i < n_ops; ++i) n += starts_x(descs, i) ? 1 : 0;
  return align256(n * G * sizeof(int32_t));
}
// Blocks of x that CTA cta reads in ops [i, j) (all sharing one x): the
// union of its units' K-parts (one K-part per op when the grid is a multiple
// of the op's K-parts, every unit of a CTA then having the same one).
int32_t cta_xrange(const KqOp* ops, int i, int j, int cta, int G) {
  int lo = 1 << 15, hi = 0;
  for (int k = i; k < j; ++k) {
    const KqOp& o = ops[k];
    const int u = first_unit(o, cta, G);
    if (u >= o.nunits) continue;
    int a = 0, b = o.nb;
    if (o.KS > 1 && G % o.KS == 0) {
      const int kp = u % o.KS;
      a = kp * o.kpb;
      b = std::min(o.nb, a + o.kpb);
    }
    lo = std::min(lo, a);
    hi = std::max(hi, b);
  }
  if (hi <= lo) lo = hi = 0;  // no unit: nothing to stage
  return lo | (hi << 16);
}
}  // namespace

size_t prog_workspace_size(const ProgOpDesc* descs, int n_ops) {
  if (n_ops <= 0) return 0;
  KqOp* ops = new KqOp[n_ops];
  size_t pb = 0;
  const bool ok = plan_prog(descs, n_ops, ops, &pb);
  delete[] ops;
  return ok ? align256(kHeaderBytes + static_cast<size_t>(n_ops) * sizeof(KqOp)) + pb +
                  xrange_bytes(descs, n_ops, num_sms())
            : 0;
}

cudaError_t prog_prepare(const ProgOpDesc* descs, int n_ops, void* ws, size_t ws_bytes, ProgPlan* plan,
                         cudaStream_t stream) {
  const int G = num_sms();
  if (n_ops <= 0) return cudaErrorInvalidValue;
  KqOp* ops = new KqOp[n_ops];
  size_t pb = 0;
  if (!plan_prog(descs, n_ops, ops, &pb)) { delete[] ops; return cudaErrorNotSupported; }
  const size_t need =
      align256(kHeaderBytes + static_cast<size_t>(n_ops) * sizeof(KqOp)) + pb + xrange_bytes(descs, n_ops, G);
  if (ws_bytes < need) { delete[] ops; return cudaErrorInvalidValue; }
  uint8_t* w = static_cast<uint8_t*>(ws);
  size_t off = align256(kHeaderBytes + static_cast<size_t>(n_ops) * sizeof(KqOp));
  int nb_max = 1, any_bf16 = 0, any_f32 = 0, any_wait = 0, last_wait = 0, final_fix = 0;
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
    if (o.x_bf16) any_bf16 = 1;
    else any_f32 = 1;
    if (stage_bytes(o) > max_stage) max_stage = stage_bytes(o);
  }
  for (int i = last_wait; i < n_ops; ++i)
    if (ops[i].KS > 1) final_fix = 1;  // not summed at any later grid barrier
  // per x: the blocks each CTA stages (after the partial sums)
  std::vector<int32_t> xr;
  for (int i = 0; i < n_ops;) {
    int j = i + 1;
    while (j < n_ops && !starts_x(descs, j)) ++j;
    ops[i].xrange = reinterpret_cast<const int32_t*>(w + off) + xr.size();
    for (int c = 0; c < G; ++c) xr.push_back(cta_xrange(ops, i, j, c, G));
    for (int k = i + 1; k < j; ++k) ops[k].xrange = nullptr;
    i = j;
  }
  LaunchGeom g;
  const int nimg = any_f32 ? 2 : 1;  // fp32 x takes two images (hi, lo)
  if (!ring_geom(max_stage, nb_max, nimg, g)) { delete[] ops; return cudaErrorNotSupported; }
  plan->n_ops = n_ops;
  plan->nb_max = nb_max;
  plan->nimg = nimg;
  plan->xk = any_bf16 && any_f32 ? 0 : any_f32 ? 2 : 1;
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
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(w + off, xr.data(), sizeof(int32_t) * xr.size(), cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  delete[] ops;
  return e;
}

cudaError_t prog_run(const ProgPlan* plan, void* ws, cudaStream_t stream) {
  ProgArgs a = {};
  a.ops = reinterpret_cast<const KqOp*>(static_cast<const uint8_t*>(ws) + kHeaderBytes);
  a.n_ops = plan->n_ops;
  a.nb_max = plan->nb_max;
  a.nimg = plan->nimg;
  a.barrier = plan->coop ? static_cast<int*>(ws) : nullptr;
  a.final_fix = plan->final_fix;
  a.err = device_error_ptr();
  LaunchGeom g;
  g.S = plan->S;
  g.slot = plan->slot;
  g.smem = static_cast<size_t>(plan->smem);
  // grid barriers need every CTA resident: cooperative launch
  const bool coop = plan->coop != 0;
  if (plan->xk == 1) return launch_prog<true, 0, 1, 4>(a, g, coop, stream, !coop);  // one x dtype: compiled for it
  if (plan->xk == 2) return launch_prog<true, 0, 2, 4>(a, g, coop, stream, !coop);
  return launch_prog<true, 0, 0, 4>(a, g, coop, stream, !coop);
}

}  // namespace kq

#ifdef KQ_TIMELINE
// The timeline library's stamps ([cta][op][4] global-timer values) for the
// last program launch: copied to host memory dst (bytes at most).
extern "C" int kq_timeline_read(void* dst, size_t bytes) {
  const size_t n = bytes < sizeof(kq::g_kq_timeline) ? bytes : sizeof(kq::g_kq_timeline);
  return static_cast<int>(cudaMemcpyFromSymbol(dst, kq::g_kq_timeline, n));
}
#endif
