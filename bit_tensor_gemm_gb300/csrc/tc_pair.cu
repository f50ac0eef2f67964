// tc_pair.cu -- instantiations of the CTA-pair tensor-core GEMM for the large
// tile class (256 x 256 outputs per pair of CTAs), stage counts 4, 5 and 6
// (the variants), and 2 and 3 for int32 outputs (measurements of the stage
// dimension through lbgemm_run_tile).
#include "tc_pair.cuh"

namespace lbg {

template <int S, bool F8, bool LINEAR>
static TcKernel pair_entry() {
  using L = PairLayout<S>;
  TcKernel k;
  k.launch = &tc_pair_launch<S, F8, LINEAR>;
  k.func = reinterpret_cast<const void*>(&tc_pair_kernel<S, F8, LINEAR>);
  k.threads = 320;
  k.smem = L::kDynSmem;
  k.tmem_cols = L::kTmemCols;
  k.tile_m = kPairTile;
  k.tile_n = kPairTile;
  k.b_box_rows = 128;  // each CTA of the pair loads half of B's tile rows
  k.cluster = 2;
  k.stages = S;
  return k;
}

template <int S>
static TcKernel pick(bool f8, bool linear) {
  if (linear) return pair_entry<S, false, true>();
  return f8 ? pair_entry<S, true, false>() : pair_entry<S, false, false>();
}

template <int S>
static TcKernel pick_int32(bool f8) {
  return f8 ? pair_entry<S, true, false>() : pair_entry<S, false, false>();
}

TcKernel tc_kernel_pair(int stages, bool f8, bool linear) {
  if (linear && f8) return TcKernel{};
  switch (stages) {
    case 2: return linear ? TcKernel{} : pick_int32<2>(f8);
    case 3: return linear ? TcKernel{} : pick_int32<3>(f8);
    case 4: return pick<4>(f8, linear);
    case 5: return pick<5>(f8, linear);
    case 6: return pick<6>(f8, linear);
    default: return TcKernel{};
  }
}

}  // namespace lbg
