// kq_gemv_ia4.cu -- the one-token kernel's single-product instantiations
// for IA4 blocks (kq_gemv_kernel.cuh): every (x dtype, tokens, rows per quad).
#include "kq_gemv_kernel.cuh"

namespace kq {

cudaError_t launch_single_ia4(int XK, int MT, int R, ProgArgs& a, int S, int slot, size_t smem, cudaStream_t st,
                              bool pdl) {
  const LaunchGeom g = {S, slot, smem};
  return launch_single_fmt<T_IA4>(XK, MT, R, a, g, st, pdl);
}

}  // namespace kq
