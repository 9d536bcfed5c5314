// kq_gemv_q6k.cu -- the one-token kernel's single-product instantiations
// for Q6_K blocks (kq_gemv_kernel.cuh): every (x dtype, tokens, rows per quad).
#include "kq_gemv_kernel.cuh"

namespace kq {

cudaError_t launch_single_q6k(int XK, int MT, int R, ProgArgs& a, int S, int slot, size_t smem, cudaStream_t st,
                              bool pdl) {
  const LaunchGeom g = {S, slot, smem};
  return launch_single_fmt<T_Q6_K>(XK, MT, R, a, g, st, pdl);
}

}  // namespace kq
