// tc_ts.cu -- instantiations of the 8-bit tensor-core GEMM that converts one
// operand in the kernel and reads it from tensor memory: 128 x 64 or 128 x 128
// tiles with double-buffered accumulators and K slices of 128 elements (6 or 4
// stages) or 256 (3 or 2 stages) (tc_ts.cuh), 128 x 256
// tiles with 4 stages and one accumulator (tc_ts256.cuh).  TRANS = false
// converts A, TRANS = true converts B.
#include "tc_ts.cuh"
#include "tc_ts256.cuh"

namespace lbg {

template <int BN, int SK>
static TcKernel pick_ts(bool trans, bool linear) {
  // as many A slots (SK / 2 columns each) as tensor memory holds beside the
  // two BN-column accumulators
  constexpr int S = (512 - 2 * BN) / (SK / 2);
  if (trans)
    return linear ? tc_ts_entry<BN, S, SK, true, true>() : tc_ts_entry<BN, S, SK, true, false>();
  return linear ? tc_ts_entry<BN, S, SK, false, true>() : tc_ts_entry<BN, S, SK, false, false>();
}

template <int S, int GS, int SG>
static TcKernel pick_ts256(bool trans, bool linear) {
  if (trans)
    return linear ? tc_ts256_entry<S, GS, SG, true, true>() : tc_ts256_entry<S, GS, SG, true, false>();
  return linear ? tc_ts256_entry<S, GS, SG, false, true>() : tc_ts256_entry<S, GS, SG, false, false>();
}

TcKernel tc_kernel_ts(int tile_n, bool trans, bool linear, int slice) {
  if (tile_n == 256) return pick_ts256<4, 4, 2>(trans, linear);
  if (slice == 256) {
    if (tile_n == 64) return pick_ts<64, 256>(trans, linear);
    if (tile_n == 128) return pick_ts<128, 256>(trans, linear);
    return TcKernel{};
  }
  if (tile_n == 64) return pick_ts<64, 128>(trans, linear);
  if (tile_n == 128) return pick_ts<128, 128>(trans, linear);
  return TcKernel{};
}

}  // namespace lbg
