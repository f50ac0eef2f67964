// tc_small.cu -- instantiations of the tensor-core GEMM for the small tile
// class (128 x 64 outputs per tile), stage counts 2, 3 and 4.
#include "tc_gemm.cuh"

namespace lbg {

template <int S>
static TcKernel pick(bool f8, bool linear) {
  if (linear) return tc_kernel_entry<64, S, false, true>();
  return f8 ? tc_kernel_entry<64, S, true, false>() : tc_kernel_entry<64, S, false, false>();
}

TcKernel tc_kernel_small(int stages, bool f8, bool linear) {
  if (linear && f8) return TcKernel{};
  switch (stages) {
    case 2: return pick<2>(f8, linear);
    case 3: return pick<3>(f8, linear);
    case 4: return pick<4>(f8, linear);
    default: return TcKernel{};
  }
}

}  // namespace lbg
