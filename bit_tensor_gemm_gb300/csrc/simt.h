// simt.h -- launchers of the CUDA-core kernels (simt.cu).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace lbg {

// Exact re-encoding of operand rows (bits 8: int8 -> fp16 rows of Kp halves,
// Kp % 8 == 0; bits 4: packed int4 -> e4m3 rows of Kp bytes, Kp % 16 == 0;
// bits 1: +-1 bits -> e4m3 rows of Kp == K bytes), zero padded, for up to two
// operands in one launch (rows_b may be 0).
// The same launch can also clear a rectangle of an int32 matrix (rows
// [r0, r1), columns [c0, c1), row stride ld elements) that the GEMM launched
// after it adds partial tiles into; C == nullptr clears nothing.
struct ZeroRect {
  int32_t* C = nullptr;
  int64_t ld = 0, r0 = 0, r1 = 0, c0 = 0, c1 = 0;
};
cudaError_t launch_encode_pair(int bits, const void* a, int64_t rows_a, void* enc_a,
                               const void* b, int64_t rows_b, void* enc_b, int64_t K, int64_t Kp,
                               int sm_count, cudaStream_t s, const ZeroRect& zero = ZeroRect{});
// M <= 16, K % 16 == 0, A and B 16-byte aligned.  Y != nullptr selects the
// linear epilogue (bf16 Y with scales sx, sw) instead of int32 C.
cudaError_t launch_skinny_s8(const int8_t* A, const int8_t* B, int M, int N, int K, int32_t* C,
                             const float* sx, const float* sw, void* Y, int sm_count,
                             cudaStream_t s);
// Per-row symmetric int8 quantisation of bf16 rows (Q: M x K int8, S: M fp32).
// 8-bit GEMM with a small side X (MX <= 32 rows, K <= hmma_skinny_max_k(MX))
// against W (NW rows) on the warp-level fp16 MMA; out[x][w] (or out[w][x]
// when trans); K % 16 == 0 and 16-byte-aligned rows.  Linear layer when Y is
// given.  hmma_skinny.cu.
int64_t hmma_skinny_max_k(int MX);
cudaError_t launch_hmma_skinny(const int8_t* X, const int8_t* W, int MX, int NW, int K,
                               bool trans, int32_t* C, const float* sx, const float* sw, void* Y,
                               int chunk_elems, int sm_count, cudaStream_t s);
// 8-bit GEMM with a small side X (1 <= MX <= 16 rows) against W (NW rows),
// K % 16 == 0, K <= stream_mma_max_k(), 16-byte-aligned rows: W streamed once
// through a bulk-copy ring, warp-level fp16 MMAs; out[x][w] (or out[w][x]
// when trans); the linear layer when Y is given (not trans).  early_w: W is
// not written by the grid launched before (its copies may start at once).
// Wait time-outs set *status.  stream_mma.cu.
int64_t stream_mma_max_k();
cudaError_t launch_stream_mma(const int8_t* X, const int8_t* W, int MX, int NW, int K, bool trans,
                              int32_t* C, const float* sx, const float* sw, void* Y, bool early_w,
                              int sm_count, int* status, cudaStream_t s);
cudaError_t launch_quant_rows_bf16(const void* X, int64_t M, int64_t K, int8_t* Q, float* S,
                                   cudaStream_t s);
// Small 8-bit GEMM on dp4a, one launch; K % 16 == 0, A and B 16-byte aligned.
// The linear layer's scaling of int32 sums S (M x N, row-major) into bf16 Y
// with row scales sx (M) and column scales sw (N); launched as a
// programmatic dependent of the grid that computed S.
cudaError_t launch_scale_sums(const int32_t* S, int64_t M, int64_t N, const float* sx,
                              const float* sw, void* Y, int sm_count, cudaStream_t s);
cudaError_t launch_small_s8(const int8_t* A, const int8_t* B, int64_t M, int64_t N, int64_t K,
                            int32_t* C, cudaStream_t s);
// The same for packed signed nibbles (K elements per row, K % 32 == 0).
cudaError_t launch_small_s4(const uint8_t* A, const uint8_t* B, int64_t M, int64_t N, int64_t K,
                            int32_t* C, cudaStream_t s);
// 1-bit GEMM, tile class 0..2 and 2..4 stages; K % 32 == 0.
cudaError_t launch_b1_popc(int tile, int stages, const uint32_t* A, const uint32_t* B, int64_t M,
                           int64_t N, int64_t K, int32_t* C, cudaStream_t s);
void b1_tile_shape(int tile, int* bm, int* bn);
// One-thread kernel whose mbarrier wait runs out after limit_ns.
cudaError_t launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t s);

}  // namespace lbg
