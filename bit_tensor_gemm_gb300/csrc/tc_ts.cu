// tc_ts.cu -- instantiations of the 8-bit tensor-core GEMM that converts one
// operand in the kernel and reads it from tensor memory: 128 x 64 or 128 x 128
// tiles with 6 or 4 stages and double-buffered accumulators (tc_ts.cuh), 128 x 256
// tiles with 4 stages and one accumulator (tc_ts256.cuh).  TRANS = false
// converts A, TRANS = true converts B.
#include "tc_ts.cuh"
#include "tc_ts256.cuh"

namespace lbg {

template <int BN>
static TcKernel pick_ts(bool trans, bool linear) {
  constexpr int S = BN == 64 ? 6 : 4;  // as many 64-column A slots as tensor memory holds
  if (trans)
    return linear ? tc_ts_entry<BN, S, true, true>() : tc_ts_entry<BN, S, true, false>();
  return linear ? tc_ts_entry<BN, S, false, true>() : tc_ts_entry<BN, S, false, false>();
}

template <int S, int GS, int SG>
static TcKernel pick_ts256(bool trans, bool linear) {
  if (trans)
    return linear ? tc_ts256_entry<S, GS, SG, true, true>() : tc_ts256_entry<S, GS, SG, true, false>();
  return linear ? tc_ts256_entry<S, GS, SG, false, true>() : tc_ts256_entry<S, GS, SG, false, false>();
}

TcKernel tc_kernel_ts(int tile_n, bool trans, bool linear) {
  if (tile_n == 256) return pick_ts256<4, 4, 2>(trans, linear);
  if (tile_n == 64) return pick_ts<64>(trans, linear);
  if (tile_n == 128) return pick_ts<128>(trans, linear);
  return TcKernel{};
}

}  // namespace lbg
