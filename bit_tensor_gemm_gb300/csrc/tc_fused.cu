// tc_fused.cu -- instantiations of the tensor-core GEMM with in-kernel int8 ->
// fp16 conversion of one operand (8-bit only, 3 fp16 stages behind 8 int8 staging stages, 128 x 64 or 128 x 128
// tiles): fuse 1 converts B (skinny M: B is the large operand), fuse 2
// converts A (skinny N).
#include "tc_gemm.cuh"

namespace lbg {

TcKernel tc_kernel_fused(int fuse, int tile_n, bool linear) {
  if (fuse == 1) {
    if (tile_n == 64)
      return linear ? tc_kernel_entry<64, 3, false, true, 1>() : tc_kernel_entry<64, 3, false, false, 1>();
    if (tile_n == 128)
      return linear ? tc_kernel_entry<128, 3, false, true, 1>()
                    : tc_kernel_entry<128, 3, false, false, 1>();
  } else if (fuse == 2 && !linear) {
    if (tile_n == 64) return tc_kernel_entry<64, 3, false, false, 2>();
    if (tile_n == 128) return tc_kernel_entry<128, 3, false, false, 2>();
  }
  return TcKernel{};
}

}  // namespace lbg
