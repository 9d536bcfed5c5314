// kq_gemv_q4k.cu -- the one-token kernel's single-product instantiations
// for Q4_K blocks (kq_gemv_kernel.cuh): every (x dtype, tokens, rows per quad).
#include "kq_gemv_kernel.cuh"

namespace kq {

cudaError_t launch_single_q4k(int XK, int MT, int R, ProgArgs& a, int S, int slot, size_t smem, cudaStream_t st,
                              bool pdl) {
  const LaunchGeom g = {S, slot, smem};
  return launch_single_fmt<T_Q4_K>(XK, MT, R, a, g, st, pdl);
}

}  // namespace kq
