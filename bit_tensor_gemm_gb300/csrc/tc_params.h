// tc_params.h -- launch parameters and the registry of tensor-core kernel
// instantiations (one per tile class x stage count x operand kind x epilogue).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace lbg {

struct TcParams {
  int M, N, K;
  int num_kb;    // 128-byte K slices per tile row
  int chunk_kb;  // slices per exact fp32 accumulation chunk
  int tiles_m, tiles_n, num_tiles, group_m;
  int dp_tiles;   // leading tiles (in tile order) computed whole, one unit each
  int splits;     // K pieces of each remaining tile (> 1: its partial tiles are
                  // added into C, zeroed there beforehand)
  int num_units;  // dp_tiles + (num_tiles - dp_tiles) * splits; grid * stream_k
  int stream_k;   // in-kernel-conversion kernels only: > 0 shares the tile-major
                  // order of all K slices out evenly, CTA b taking the b-th
                  // contiguous run, cut at tile ends into up to stream_k units,
                  // every one added into C (zeroed there beforehand)
  int vec_ok;    // rows of C/Y are 16-byte aligned: C goes out by TMA stores,
                 // Y by 16-byte vector stores
  int32_t* C;
  const float* sx;
  const float* sw;
  __nv_bfloat16* Y;
  int* status;
};

// (A map, B map, C map, params, grid, programmatic dependent launch, stream)
typedef cudaError_t (*TcLaunchFn)(const CUtensorMap*, const CUtensorMap*, const CUtensorMap*,
                                  const TcParams*, int, bool, cudaStream_t);

struct TcKernel {
  TcLaunchFn launch = nullptr;
  const void* func = nullptr;
  int smem = 0;
  int tmem_cols = 0;
  int tile_m = 128;     // output rows per tile (per CTA pair for cluster 2)
  int tile_n = 0;
  int b_box_rows = 0;   // rows of B per TMA box (0: tile_n)
  int cluster = 1;      // CTAs per tile: 2 for the cta_group::2 kernel
  int stages = 0;
  int threads = 320;
  int slice = 0;  // K elements per slice of the in-kernel-conversion kernels (0: others)
};

// Dynamic shared memory to request so that the CTAs that fit on one SM by
// shared memory never need more than the 512 TMEM columns of that SM.
inline constexpr int tc_smem_request(int used, int tmem_cols) {
  constexpr int kSmPerSm = 233472;  // 228 KB shared memory per SM
  const int max_ctas = 512 / tmem_cols;
  const int min_req = kSmPerSm / (max_ctas + 1) + 1;  // one more CTA cannot fit
  return used > min_req ? used : min_req;
}

// tile: 0 small (128 x 64), 1 medium (128 x 128), stages 2..4;
// 2 large (256 x 256 on a pair of CTAs, cta_group::2 MMAs), stages 4..6.
TcKernel tc_kernel_small(int stages, bool f8, bool linear);
TcKernel tc_kernel_medium(int stages, bool f8, bool linear);
TcKernel tc_kernel_pair(int stages, bool f8, bool linear);
// One operand converted from int8 in the kernel and fed to the MMA from tensor
// memory (8-bit only): trans = false converts A, trans = true converts B (C is
// written transposed from the accumulator); tile_n 64, 128 or 256; slice: K
// elements per pipeline slice of the 64- and 128-wide kernels (128 or 256).
TcKernel tc_kernel_ts(int tile_n, bool trans, bool linear, int slice = 128);

}  // namespace lbg
