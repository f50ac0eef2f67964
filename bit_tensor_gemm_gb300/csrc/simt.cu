// simt.cu -- the CUDA-core kernels of the library:
//   * exact operand re-encoding for the tensor-core path (int8 -> fp16,
//     packed int4 -> e4m3), HBM-bound streaming passes;
//   * the skinny 8-bit GEMM (M <= 16) on dp4a, which streams B once from HBM
//     instead of re-encoding it;
//   * the 1-bit GEMM on XOR + popcount.
//
// Method: "Leveraging Large-Scale Data for Efficient Low-Bit CUTLASS GEMM
// Optimization via Neural Networks" (press summary page), intro (1-, 4-,
// 8-bit GEMM) and section 1 (tiles of C looping over K with a multi-stage
// load pipeline).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "ptx.cuh"
#include "simt.h"

namespace lbg {

// ---------------------------------------------------------------------------
// Exact re-encoding of up to two operands in one launch.  Rows of K values
// become rows of Kp >= K (zero padded).  The kernel lets a dependent launch
// (the GEMM, which waits for this grid's completion before its first read)
// start its prologue early.

struct CvtJob {
  const void* src;
  int64_t rows;
  void* dst;
  int fast;  // 8-byte aligned source rows
};

__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// A kernel launched as a programmatic dependent may start while the grid
// before it in the stream is still running: it waits for that grid (and its
// memory operations) here before its first access to global memory.
__device__ __forceinline__ void wait_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Launch with programmatic stream serialisation: the kernel may be scheduled
// as soon as the previous grid in the stream has let dependents launch; the
// kernel itself must call wait_prior_grid() before touching global memory.
template <typename... KArgs, typename... Args>
static cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Clears the rectangle z of an int32 matrix, grid-stride over the whole grid;
// 16-byte stores when the rows and columns allow.
__device__ __forceinline__ void zero_rect(const ZeroRect& z) {
  if (z.C == nullptr) return;
  const int64_t w = z.c1 - z.c0, h = z.r1 - z.r0;
  const int64_t nt = (int64_t)gridDim.x * blockDim.x;
  const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const bool vec = w % 4 == 0 && z.c0 % 4 == 0 && z.ld % 4 == 0 &&
                   (reinterpret_cast<uintptr_t>(z.C) & 15) == 0;
  if (vec) {
    const int64_t wq = w / 4;
    for (int64_t i = t0; i < h * wq; i += nt) {
      const int64_t r = i / wq, c = i - r * wq;
      *reinterpret_cast<int4*>(z.C + (z.r0 + r) * z.ld + z.c0 + 4 * c) = make_int4(0, 0, 0, 0);
    }
  } else {
    for (int64_t i = t0; i < h * w; i += nt) {
      const int64_t r = i / w, c = i - r * w;
      z.C[(z.r0 + r) * z.ld + z.c0 + c] = 0;
    }
  }
}

// int8 -> fp16; each thread writes 8 halves (16 bytes).
__global__ void cvt_s8_f16_kernel(CvtJob ja, CvtJob jb, int64_t K, int64_t Kp, ZeroRect z) {
  allow_dependent_launch();
  wait_prior_grid();
  zero_rect(z);
  const int64_t vec_per_row = Kp / 8;
  const int64_t total_a = ja.rows * vec_per_row;
  const int64_t total = total_a + jb.rows * vec_per_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const bool in_a = i < total_a;
    const int64_t ii = in_a ? i : i - total_a;
    const CvtJob& j = in_a ? ja : jb;
    const int64_t r = ii / vec_per_row;
    const int64_t c = (ii - r * vec_per_row) * 8;
    const int8_t* src = static_cast<const int8_t*>(j.src) + r * K + c;
    __align__(16) __half h[8];
    if (j.fast && c + 8 <= K) {
      const uint2 w = __ldg(reinterpret_cast<const uint2*>(src));
      const uint32_t lo = w.x, hi = w.y;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        h[q] = __short2half_rn((short)(int8_t)(lo >> (8 * q)));
        h[4 + q] = __short2half_rn((short)(int8_t)(hi >> (8 * q)));
      }
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q) h[q] = __short2half_rn(c + q < K ? (short)src[q] : (short)0);
    }
    *reinterpret_cast<uint4*>(static_cast<__half*>(j.dst) + r * Kp + c) =
        *reinterpret_cast<const uint4*>(h);
  }
}

// int8 -> fp16 for K % 16 == 0 and 16-byte-aligned rows.  Then Kp == K, so
// both operands are flat arrays and the fp16 of input byte x sits at output
// byte 2x: the kernel streams 8-byte units (a warp loads 256 contiguous bytes
// and stores 512), four units in flight per thread, converting four bytes at
// a time with integer and half2 arithmetic: the fp16 with bits 0x6400 | u is
// 1024 + u, so (v ^ 0x80) as u, minus 1152, is v exactly.
__device__ __forceinline__ void s8x4_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t a = __byte_perm(u, 0x64646464u, 0x5140);
  const uint32_t b = __byte_perm(u, 0x64646464u, 0x7362);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  const __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
  const __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
  lo = *reinterpret_cast<const uint32_t*>(&ha);
  hi = *reinterpret_cast<const uint32_t*>(&hb);
}

__device__ __forceinline__ uint4 s8x8_f16x8(int2 v) {
  uint4 o;
  s8x4_f16x2((uint32_t)v.x, o.x, o.y);
  s8x4_f16x2((uint32_t)v.y, o.z, o.w);
  return o;
}

// units: 8-byte groups; na of operand a, then nb of operand b
__global__ void cvt_s8_f16_flat_kernel(const int2* __restrict__ a, int64_t na, uint4* ea,
                                       const int2* __restrict__ b, int64_t nb, uint4* eb,
                                       ZeroRect z) {
  allow_dependent_launch();
  wait_prior_grid();
  zero_rect(z);
  const int64_t total = na + nb;
  const int64_t nt = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * nt < total; i += 4 * nt) {
    int2 v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int64_t u = i + q * nt;
      v[q] = u < na ? __ldg(a + u) : __ldg(b + (u - na));
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int64_t u = i + q * nt;
      const uint4 o = s8x8_f16x8(v[q]);
      if (u < na)
        ea[u] = o;
      else
        eb[u - na] = o;
    }
  }
  for (; i < total; i += nt) {
    if (i < na)
      ea[i] = s8x8_f16x8(__ldg(a + i));
    else
      eb[i - na] = s8x8_f16x8(__ldg(b + (i - na)));
  }
}

// packed int4 (two per byte, low nibble first) -> e4m3 bytes; K is even.
// Each thread writes 16 output bytes from 8 input bytes through a 256-entry
// table (byte -> two e4m3 codes) built per block with CUDA's fp8 conversion.
__global__ void cvt_s4_e4m3_kernel(CvtJob ja, CvtJob jb, int64_t K, int64_t Kp, ZeroRect z) {
  allow_dependent_launch();
  wait_prior_grid();
  zero_rect(z);
  __shared__ uint16_t table[256];
  for (int b = threadIdx.x; b < 256; b += blockDim.x) {
    const int lo = (b & 15) >= 8 ? (b & 15) - 16 : (b & 15);
    const int hi = (b >> 4) >= 8 ? (b >> 4) - 16 : (b >> 4);
    const uint16_t elo = __nv_cvt_float_to_fp8((float)lo, __NV_SATFINITE, __NV_E4M3);
    const uint16_t ehi = __nv_cvt_float_to_fp8((float)hi, __NV_SATFINITE, __NV_E4M3);
    table[b] = (uint16_t)(elo | (ehi << 8));
  }
  __syncthreads();
  const int64_t in_row = K / 2;
  const int64_t vec_per_row = Kp / 16;
  const int64_t total_a = ja.rows * vec_per_row;
  const int64_t total = total_a + jb.rows * vec_per_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const bool in_a = i < total_a;
    const int64_t ii = in_a ? i : i - total_a;
    const CvtJob& j = in_a ? ja : jb;
    const int64_t r = ii / vec_per_row;
    const int64_t cb = (ii - r * vec_per_row) * 8;  // input byte column
    const uint8_t* src = static_cast<const uint8_t*>(j.src) + r * in_row + cb;
    uint32_t o[4];
    if (j.fast && cb + 8 <= in_row) {
      const uint2 w = __ldg(reinterpret_cast<const uint2*>(src));
      o[0] = table[w.x & 0xFF] | ((uint32_t)table[(w.x >> 8) & 0xFF] << 16);
      o[1] = table[(w.x >> 16) & 0xFF] | ((uint32_t)table[w.x >> 24] << 16);
      o[2] = table[w.y & 0xFF] | ((uint32_t)table[(w.y >> 8) & 0xFF] << 16);
      o[3] = table[(w.y >> 16) & 0xFF] | ((uint32_t)table[w.y >> 24] << 16);
    } else {
      uint16_t t[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) t[q] = cb + q < in_row ? table[src[q]] : (uint16_t)0;
#pragma unroll
      for (int q = 0; q < 4; ++q) o[q] = t[2 * q] | ((uint32_t)t[2 * q + 1] << 16);
    }
    *reinterpret_cast<uint4*>(static_cast<uint8_t*>(j.dst) + r * Kp + 2 * cb) =
        make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// +-1 bits (32 per word, bit 1 = +1) -> e4m3 bytes, one per element: every
// +-1 is an e4m3 value, so the tensor-core route stays exact.  Rows of W
// words become rows of 32 W bytes.  Each thread expands one word through a
// 16-entry table (four bits -> four codes) built per block with CUDA's fp8
// conversion of +1 and -1.
__global__ void cvt_b1_e4m3_kernel(CvtJob ja, CvtJob jb, int64_t W, ZeroRect z) {
  allow_dependent_launch();
  wait_prior_grid();
  zero_rect(z);
  __shared__ uint32_t nib[16];
  if (threadIdx.x < 16) {
    const uint32_t pos = __nv_cvt_float_to_fp8(1.0f, __NV_SATFINITE, __NV_E4M3);
    const uint32_t neg = __nv_cvt_float_to_fp8(-1.0f, __NV_SATFINITE, __NV_E4M3);
    uint32_t v = 0;
    for (int q = 0; q < 4; ++q) v |= (((threadIdx.x >> q) & 1) ? pos : neg) << (8 * q);
    nib[threadIdx.x] = v;
  }
  __syncthreads();
  const int64_t total_a = ja.rows * W;
  const int64_t total = total_a + jb.rows * W;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const bool in_a = i < total_a;
    const int64_t ii = in_a ? i : i - total_a;
    const CvtJob& j = in_a ? ja : jb;
    const uint32_t word = __ldg(static_cast<const uint32_t*>(j.src) + ii);
    uint32_t o[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) o[q] = nib[(word >> (4 * q)) & 15u];
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(j.dst) + ii * 32);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// ---------------------------------------------------------------------------
// Per-row symmetric int8 quantisation of bf16 activations (the step before a
// quantised linear layer): s = max(absmax(row), 1e-12) / 127 and
// q = clamp(round_half_even(x / s), -127, 127), all in fp32 with IEEE
// division.  WPR warps per row (8 rows of one warp, or one row of eight
// warps, per 256-thread block: few rows are spread over more threads); two
// passes over the row (max, then codes).
template <int WPR>
__global__ void __launch_bounds__(256)
    quant_rows_bf16_kernel(const __nv_bfloat16* __restrict__ X, int64_t M, int64_t K,
                           int8_t* __restrict__ Q, float* __restrict__ S, int vec) {
  constexpr int T = 32 * WPR;  // threads per row
  // the GEMM launched after this grid waits for it to finish before reading
  // Q and S, but may launch (and set up) meanwhile
  allow_dependent_launch();
  const int t = threadIdx.x % T;
  const int64_t row = (int64_t)blockIdx.x * (256 / T) + threadIdx.x / T;
  if (WPR == 1 && row >= M) return;  // (WPR > 1: one row per block, grid = M)
  const __nv_bfloat16* x = X + row * K;
  int8_t* q = Q + row * K;
  float amax = 0.0f;
  if (vec) {
    for (int64_t k = (int64_t)t * 8; k < K; k += T * 8) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + k));
      const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&v);
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(__bfloat162float(h[j])));
    }
  } else {
    for (int64_t k = t; k < K; k += T) amax = fmaxf(amax, fabsf(__bfloat162float(x[k])));
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if (WPR > 1) {
    __shared__ float part[WPR];
    if ((t & 31) == 0) part[t >> 5] = amax;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < WPR; ++w) amax = fmaxf(amax, part[w]);
  }
  const float sc = __fdiv_rn(fmaxf(amax, 1e-12f), 127.0f);
  if (t == 0) S[row] = sc;
  auto code = [&](float v) -> int8_t {
    float r = rintf(__fdiv_rn(v, sc));
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    return (int8_t)(int)r;
  };
  if (vec) {
    for (int64_t k = (int64_t)t * 8; k < K; k += T * 8) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + k));
      const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&v);
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        lo |= (uint32_t)(uint8_t)code(__bfloat162float(h[j])) << (8 * j);
        hi |= (uint32_t)(uint8_t)code(__bfloat162float(h[4 + j])) << (8 * j);
      }
      *reinterpret_cast<uint2*>(q + k) = make_uint2(lo, hi);
    }
  } else {
    for (int64_t k = t; k < K; k += T) q[k] = code(__bfloat162float(x[k]));
  }
}

// ---------------------------------------------------------------------------
// Skinny 8-bit GEMM: M <= MT rows of A against all N rows of B, for M <= 16.
// HBM-bound on B, which is streamed exactly once.  Persistent warps each own
// groups of NR consecutive rows of B; a lane covers 16 bytes of K per step
// (512 bytes per warp-step); each batch issues the loads of PF steps for all
// NR rows before consuming any of them.  A rows come through L1.
constexpr int kSkWarps = 8;

template <int NR>
__device__ __forceinline__ void skinny_load_step(int4 (&dst)[NR], const int8_t* __restrict__ B,
                                                 int K, int N, int n0, int k) {
#pragma unroll
  for (int r = 0; r < NR; ++r)
    dst[r] = (k < K && n0 + r < N)
                 ? __ldg(reinterpret_cast<const int4*>(B + (int64_t)(n0 + r) * K + k))
                 : make_int4(0, 0, 0, 0);
}

// Combines a warp's partial sums of one group (halving butterfly: at each
// step a lane keeps half of its values -- the upper half if the step's lane
// bit is set -- plus its partner's copy of that half; once one value is left
// the remaining steps simply add), writes the group's outputs and clears acc.
template <int MT, int NR, bool LINEAR>
__device__ __forceinline__ void skinny_finish(int (&acc)[MT * NR], int lane, int M, int N, int n0,
                                              int32_t* __restrict__ C,
                                              const float* __restrict__ sx,
                                              const float* __restrict__ sw,
                                              __nv_bfloat16* __restrict__ Y) {
  constexpr int NV = MT * NR;
  int n = NV;
  int idx_base = 0;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    if (n > 1) {
      const bool upper = (lane & off) != 0;
      const int h = n / 2;
#pragma unroll
      for (int i = 0; i < (NV > 1 ? NV / 2 : 1); ++i) {
        if (i < h) {
          const int send = upper ? acc[i] : acc[i + h];
          const int keep = upper ? acc[i + h] : acc[i];
          acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
      }
      if (upper) idx_base += h;
      n = h;
    } else {
      acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], off);
    }
  }
  // Lanes that share idx_base hold the same totals; the lowest one writes.
  const int owner_mask = (NV >= 32) ? 0 : (32 / NV) - 1;
  if ((lane & owner_mask) == 0) {
#pragma unroll
    for (int j = 0; j < (NV >= 32 ? NV / 32 : 1); ++j) {
      const int idx = idx_base + j;
      const int m = idx / NR, r = idx % NR;
      if (m < M && n0 + r < N) {
        if (LINEAR)
          Y[(int64_t)m * N + n0 + r] = __float2bfloat16_rn((float)acc[j] * sx[m] * sw[n0 + r]);
        else
          C[(int64_t)m * N + n0 + r] = acc[j];
      }
    }
  }
#pragma unroll
  for (int i = 0; i < NV; ++i) acc[i] = 0;
}

template <int MT, int NR, int PF, int MINB, bool LINEAR>
__global__ void __launch_bounds__(kSkWarps * 32, MINB)
    skinny_s8_kernel(const int8_t* __restrict__ A, const int8_t* __restrict__ B, int M, int N,
                     int K, int32_t* __restrict__ C, const float* __restrict__ sx,
                     const float* __restrict__ sw, __nv_bfloat16* __restrict__ Y) {
  constexpr int NV = MT * NR;
  // launched as a programmatic dependent: A (and its scales) may come from
  // the grid before this one (the activation quantiser), which may still be
  // running; wait for it before the first read
  wait_prior_grid();
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * kSkWarps;
  const int groups = (N + NR - 1) / NR;
  const int steps = (K + 511) / 512;
  int acc[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) acc[i] = 0;
  for (int g = blockIdx.x * kSkWarps + (threadIdx.x >> 5); g < groups; g += nwarps) {
    const int n0 = g * NR;
    for (int s0 = 0; s0 < steps; s0 += PF) {
      // issue every load of this batch of PF steps, then consume them
      int4 v[PF][NR];
#pragma unroll
      for (int q = 0; q < PF; ++q)
        skinny_load_step<NR>(v[q], B, K, N, n0, (s0 + q) * 512 + lane * 16);
#pragma unroll
      for (int q = 0; q < PF; ++q) {
        const int k = (s0 + q) * 512 + lane * 16;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const int4 a = (m < M && k < K)
                             ? __ldg(reinterpret_cast<const int4*>(A + (int64_t)m * K + k))
                             : make_int4(0, 0, 0, 0);
#pragma unroll
          for (int r = 0; r < NR; ++r) {
            int t = acc[m * NR + r];
            t = __dp4a(a.x, v[q][r].x, t);
            t = __dp4a(a.y, v[q][r].y, t);
            t = __dp4a(a.z, v[q][r].z, t);
            t = __dp4a(a.w, v[q][r].w, t);
            acc[m * NR + r] = t;
          }
        }
      }
    }
    skinny_finish<MT, NR, LINEAR>(acc, lane, M, N, n0, C, sx, sw, Y);
  }
}

// ---------------------------------------------------------------------------
// Small 8-bit (and 4-bit) GEMM on CUDA cores (dp4a), for problems too small
// to pay for the re-encoding pass and a second launch: one launch, the
// packed operands read directly (nibbles sign-extended to int8 in
// registers).  CTA tile 64 x 64, 256 threads as a 16 x 16 grid, thread
// (ty, tx) owning rows ty + 16 i and columns tx + 16 j; K staged 64 bytes at
// a time through a two-stage cp.async ring.  Out-of-range rows and K bytes
// load as zero (a zero nibble is the value 0).  Requires rows of a multiple
// of 16 bytes (K % 16 == 0 for int8, K % 32 == 0 for nibbles) and 16-byte
// aligned A and B.
constexpr int kSmKS = 64;           // bytes of K per stage
constexpr int kSmStride = kSmKS + 16;  // padded smem row, 16-byte aligned

__device__ __forceinline__ void small_load_tile(int8_t* dst, const int8_t* src, int64_t rows,
                                                int64_t K, int64_t r0, int64_t k0) {
  // 64 rows x 64 bytes = 256 chunks of 16 bytes: one per thread
  const int r = threadIdx.x >> 2, c = (threadIdx.x & 3) * 16;
  const int64_t gr = r0 + r, gk = k0 + c;
  const bool ok = gr < rows && gk < K;
  const int8_t* g = ok ? src + gr * K + gk : src;
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst + r * kSmStride + c));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(g), "r"(ok ? 16 : 0)
               : "memory");
}

// Signed nibbles (two per byte, element 2j in the low nibble of byte j) of a
// 32-bit word into two words of four signed int8: the low nibbles (elements
// 0, 2, 4, 6) and the high ones (1, 3, 5, 7).  A nibble n is (n ^ 8) - 8.
__device__ __forceinline__ void s4x8_to_s8(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = __vsub4((w & 0x0F0F0F0Fu) ^ 0x08080808u, 0x08080808u);
  hi = __vsub4(((w >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u, 0x08080808u);
}

// S4: the operands are packed signed nibbles; KB is the row length in bytes
// (K for int8, K / 2 for nibbles).  A dot product does not depend on the
// order of K, so the low and the high nibbles of the same bytes of A and B
// are paired as two dp4a terms.
template <bool S4>
__global__ void __launch_bounds__(256)
    small_dp4a_kernel(const int8_t* __restrict__ A, const int8_t* __restrict__ B, int64_t M,
                      int64_t N, int64_t K, int32_t* __restrict__ C) {
  __shared__ __align__(16) int8_t sA[2][64 * kSmStride];
  __shared__ __align__(16) int8_t sB[2][64 * kSmStride];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int64_t m0 = (int64_t)blockIdx.y * 64, n0 = (int64_t)blockIdx.x * 64;
  const int64_t num_kt = (K + kSmKS - 1) / kSmKS;
  int acc[4][4] = {};
  small_load_tile(sA[0], A, M, K, m0, 0);
  small_load_tile(sB[0], B, N, K, n0, 0);
  asm volatile("cp.async.commit_group;" ::: "memory");
  for (int64_t kt = 0; kt < num_kt; ++kt) {
    const int cur = (int)(kt & 1);
    if (kt + 1 < num_kt) {
      small_load_tile(sA[cur ^ 1], A, M, K, m0, (kt + 1) * kSmKS);
      small_load_tile(sB[cur ^ 1], B, N, K, n0, (kt + 1) * kSmKS);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    __syncthreads();
#pragma unroll
    for (int c = 0; c < kSmKS; c += 16) {
      int4 a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        a[i] = *reinterpret_cast<const int4*>(sA[cur] + (ty + 16 * i) * kSmStride + c);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        b[j] = *reinterpret_cast<const int4*>(sB[cur] + (tx + 16 * j) * kSmStride + c);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          int s = acc[i][j];
          if (S4) {
            const uint32_t av[4] = {(uint32_t)a[i].x, (uint32_t)a[i].y, (uint32_t)a[i].z,
                                    (uint32_t)a[i].w};
            const uint32_t bv[4] = {(uint32_t)b[j].x, (uint32_t)b[j].y, (uint32_t)b[j].z,
                                    (uint32_t)b[j].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t al, ah, bl, bh;
              s4x8_to_s8(av[q], al, ah);
              s4x8_to_s8(bv[q], bl, bh);
              s = __dp4a((int)al, (int)bl, s);
              s = __dp4a((int)ah, (int)bh, s);
            }
          } else {
            s = __dp4a(a[i].x, b[j].x, s);
            s = __dp4a(a[i].y, b[j].y, s);
            s = __dp4a(a[i].z, b[j].z, s);
            s = __dp4a(a[i].w, b[j].w, s);
          }
          acc[i][j] = s;
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + ty + 16 * i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = n0 + tx + 16 * j;
      if (n < N) C[m * N + n] = acc[i][j];
    }
  }
}

// ---------------------------------------------------------------------------
// 1-bit GEMM on CUDA cores: C[m][n] = K - 2 * sum_w popc(A[m][w] ^ B[n][w]).
// CTA tile BM x BN, 256 threads as a 16 x 16 grid, thread (ty, tx) owning rows
// ty + 16 i and columns tx + 16 j; K staged 32 words at a time through a
// STAGES-deep cp.async ring.  Out-of-range rows and words are zero in both
// operands, so they add no differing bits.
constexpr int kB1KW = 32;            // words per stage
constexpr int kB1Stride = kB1KW + 4;  // padded smem row (16-byte aligned)

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, int bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int ROWS, bool VEC>
__device__ __forceinline__ void b1_load_tile(uint32_t* dst, const uint32_t* src, int64_t rows,
                                             int64_t W, int64_t r0, int64_t w0) {
  const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  if (VEC) {
    constexpr int kChunks = ROWS * kB1KW / 4;
    for (int i = threadIdx.x; i < kChunks; i += 256) {
      const int r = i / (kB1KW / 4), c = (i % (kB1KW / 4)) * 4;
      const int64_t gr = r0 + r, gw = w0 + c;
      const bool ok = gr < rows && gw < W;
      const uint32_t* g = ok ? src + gr * W + gw : src;
      cp_async_16(base + (r * kB1Stride + c) * 4, g, ok ? 16 : 0);
    }
  } else {
    constexpr int kWords = ROWS * kB1KW;
    for (int i = threadIdx.x; i < kWords; i += 256) {
      const int r = i / kB1KW, c = i % kB1KW;
      const int64_t gr = r0 + r, gw = w0 + c;
      const bool ok = gr < rows && gw < W;
      const uint32_t* g = ok ? src + gr * W + gw : src;
      cp_async_4(base + (r * kB1Stride + c) * 4, g, ok ? 4 : 0);
    }
  }
}

template <int BM, int BN, int STAGES, bool VEC>
__global__ void __launch_bounds__(256)
    b1_popc_kernel(const uint32_t* __restrict__ A, const uint32_t* __restrict__ B, int64_t M,
                   int64_t N, int64_t K, int32_t* __restrict__ C) {
  constexpr int TM = BM / 16, TN = BN / 16;
  extern __shared__ __align__(16) uint32_t b1_smem[];
  uint32_t* sA = b1_smem;
  uint32_t* sB = b1_smem + STAGES * BM * kB1Stride;
  const int64_t W = K / 32;
  const int64_t m0 = (int64_t)blockIdx.y * BM, n0 = (int64_t)blockIdx.x * BN;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int64_t num_kt = (W + kB1KW - 1) / kB1KW;

  int acc[TM][TN];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0;

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < num_kt) {
      b1_load_tile<BM, VEC>(sA + s * BM * kB1Stride, A, M, W, m0, s * kB1KW);
      b1_load_tile<BN, VEC>(sB + s * BN * kB1Stride, B, N, W, n0, s * kB1KW);
    }
    cp_async_commit();
  }
  for (int64_t kt = 0; kt < num_kt; ++kt) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    {  // prefetch the stage STAGES-1 ahead into the slot freed last iteration
      const int64_t nk = kt + STAGES - 1;
      const int slot = (int)(nk % STAGES);
      if (nk < num_kt) {
        b1_load_tile<BM, VEC>(sA + slot * BM * kB1Stride, A, M, W, m0, nk * kB1KW);
        b1_load_tile<BN, VEC>(sB + slot * BN * kB1Stride, B, N, W, n0, nk * kB1KW);
      }
      cp_async_commit();
    }
    const int slot = (int)(kt % STAGES);
    const uint32_t* a_s = sA + slot * BM * kB1Stride;
    const uint32_t* b_s = sB + slot * BN * kB1Stride;
#pragma unroll 2
    for (int w = 0; w < kB1KW; w += 4) {
      uint4 a[TM], b[TN];
#pragma unroll
      for (int i = 0; i < TM; ++i)
        a[i] = *reinterpret_cast<const uint4*>(a_s + (ty + 16 * i) * kB1Stride + w);
#pragma unroll
      for (int j = 0; j < TN; ++j)
        b[j] = *reinterpret_cast<const uint4*>(b_s + (tx + 16 * j) * kB1Stride + w);
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j)
          acc[i][j] += __popc(a[i].x ^ b[j].x) + __popc(a[i].y ^ b[j].y) +
                       __popc(a[i].z ^ b[j].z) + __popc(a[i].w ^ b[j].w);
    }
  }
  cp_async_wait<0>();
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int64_t m = m0 + ty + 16 * i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < TN; ++j) {
      const int64_t n = n0 + tx + 16 * j;
      if (n < N) C[m * N + n] = (int32_t)(K - 2 * (int64_t)acc[i][j]);
    }
  }
}

// ---------------------------------------------------------------------------
// Self-test of the bounded wait: one thread waits on an mbarrier that nothing
// will ever signal, through the same helper the GEMM kernel uses, with a short
// limit.  The wait gives up, raises the status word and the kernel returns.
__global__ void wait_selftest_kernel(int* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    const uint32_t b = smem_addr(&bar);
    mbar_init(b, 1);
    abort_flag = 0;
    fence_barrier_init();
    mbar_wait(b, 0, &abort_flag, status, limit_ns);
  }
}

// ---------------------------------------------------------------------------
// The linear layer's scaling of int32 sums: Y[m][n] = bf16(S[m][n] * sx[m] *
// sw[n]), the products in the order of the GEMM kernels' linear epilogues.
// Four elements per thread when rows are whole 16-byte groups.
__global__ void scale_sums_kernel(const int32_t* S, int64_t M, int64_t N, const float* sx,
                                  const float* sw, __nv_bfloat16* Y, int vec) {
  allow_dependent_launch();
  wait_prior_grid();
  const int64_t nt = (int64_t)gridDim.x * blockDim.x;
  const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (vec) {
    const int64_t nq = N / 4;
    for (int64_t q = t0; q < M * nq; q += nt) {
      const int64_t m = q / nq, n = (q - m * nq) * 4;
      const int4 v = __ldcs(reinterpret_cast<const int4*>(S + m * N + n));
      const float a = sx[m];
      const float4 w = *reinterpret_cast<const float4*>(sw + n);
      __nv_bfloat162 lo = __floats2bfloat162_rn((float)v.x * a * w.x, (float)v.y * a * w.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn((float)v.z * a * w.z, (float)v.w * a * w.w);
      uint2 o;
      o.x = *reinterpret_cast<const uint32_t*>(&lo);
      o.y = *reinterpret_cast<const uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(Y + m * N + n) = o;
    }
  } else {
    for (int64_t e = t0; e < M * N; e += nt) {
      const int64_t m = e / N, n = e - m * N;
      Y[e] = __float2bfloat16_rn((float)S[e] * sx[m] * sw[n]);
    }
  }
}

// ---------------------------------------------------------------------------
// host launchers

cudaError_t launch_scale_sums(const int32_t* S, int64_t M, int64_t N, const float* sx,
                              const float* sw, void* Y, int sm_count, cudaStream_t s) {
  if (M == 0 || N == 0) return cudaSuccess;
  auto al = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; };
  const int vec = N % 4 == 0 && al(S, 16) && al(sw, 16) && al(Y, 8);
  const int64_t work = vec ? M * (N / 4) : M * N;
  int64_t blocks = (work + 255) / 256;
  blocks = std::min<int64_t>(std::max<int64_t>(blocks, 1), (int64_t)sm_count * 8);
  return launch_dependent(scale_sums_kernel, dim3((unsigned)blocks), dim3(256), 0, s, S, M, N, sx,
                          sw, static_cast<__nv_bfloat16*>(Y), vec);
}

cudaError_t launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

static int grid_for(int64_t work, int threads, int sm_count) {
  int64_t blocks = (work + threads - 1) / threads;
  const int64_t cap = (int64_t)sm_count * 16;
  if (blocks > cap) blocks = cap;
  return (int)(blocks < 1 ? 1 : blocks);
}

cudaError_t launch_quant_rows_bf16(const void* X, int64_t M, int64_t K, int8_t* Q, float* S,
                                   cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  const int vec = (K % 8 == 0) && ((reinterpret_cast<uintptr_t>(X) & 15) == 0) &&
                  ((reinterpret_cast<uintptr_t>(Q) & 7) == 0);
  // eight warps per row while that leaves the rows' threads within a few
  // waves of the GPU (a warp per row leaves it mostly idle: 2048 x 4096 took
  // 19 us that way); beyond that one warp per row, eight rows per block
  if (M <= 8192) {
    quant_rows_bf16_kernel<8><<<(unsigned)M, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(X), M,
                                                          K, Q, S, vec);
  } else {
    const unsigned grid = (unsigned)((M + 7) / 8);
    quant_rows_bf16_kernel<1><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(X), M, K, Q,
                                                   S, vec);
  }
  return cudaGetLastError();
}

cudaError_t launch_encode_pair(int bits, const void* a, int64_t rows_a, void* enc_a,
                               const void* b, int64_t rows_b, void* enc_b, int64_t K, int64_t Kp,
                               int sm_count, cudaStream_t s, const ZeroRect& zero) {
  if (rows_a + rows_b == 0 && zero.C == nullptr) return cudaSuccess;
  const int64_t row_bytes = bits == 8 ? K : bits == 4 ? K / 2 : K / 8;
  auto fast = [&](const void* p) {
    return (int)(row_bytes % 8 == 0 && (reinterpret_cast<uintptr_t>(p) & 7) == 0);
  };
  CvtJob ja{a, rows_a, enc_a, a ? fast(a) : 0};
  CvtJob jb{b, rows_b, enc_b, b ? fast(b) : 0};
  // threads enough for the clearing too (about four 16-byte stores each)
  const int64_t zero_threads =
      zero.C ? ((zero.r1 - zero.r0) * (zero.c1 - zero.c0) + 15) / 16 : 0;
  auto with_zero = [&](int grid) {
    const int64_t zb = std::min<int64_t>((zero_threads + 255) / 256, (int64_t)sm_count * 16);
    return (int)std::max<int64_t>(grid, zb);
  };
  if (bits == 1) {  // K % 32 == 0 and Kp == K: rows are contiguous words
    const int64_t W = K / 32;
    return launch_dependent(cvt_b1_e4m3_kernel,
                            dim3(with_zero(grid_for((rows_a + rows_b) * W, 256, sm_count))),
                            dim3(256), 0, s, ja, jb, W, zero);
  }
  auto aligned16 = [&](const void* p) {
    return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15) == 0;
  };
  if (bits == 8 && K % 16 == 0 && aligned16(a) && aligned16(b) && aligned16(enc_a) &&
      aligned16(enc_b)) {
    const int64_t na = a ? rows_a * (K / 8) : 0, nb = b ? rows_b * (K / 8) : 0;
    int64_t blocks = (na + nb + 4 * 256 - 1) / (4 * 256);
    blocks = std::min<int64_t>(std::max<int64_t>(blocks, 1), (int64_t)sm_count * 8);
    return launch_dependent(cvt_s8_f16_flat_kernel, dim3(with_zero((int)blocks)), dim3(256), 0, s,
                            static_cast<const int2*>(a), na, static_cast<uint4*>(enc_a),
                            static_cast<const int2*>(b), nb, static_cast<uint4*>(enc_b), zero);
  }
  const int64_t vec = bits == 8 ? Kp / 8 : Kp / 16;
  const int grid = with_zero(grid_for((rows_a + rows_b) * vec, 256, sm_count));
  if (bits == 8)
    return launch_dependent(cvt_s8_f16_kernel, dim3(grid), dim3(256), 0, s, ja, jb, K, Kp, zero);
  return launch_dependent(cvt_s4_e4m3_kernel, dim3(grid), dim3(256), 0, s, ja, jb, K, Kp, zero);
}

cudaError_t launch_small_s8(const int8_t* A, const int8_t* B, int64_t M, int64_t N, int64_t K,
                            int32_t* C, cudaStream_t s) {
  if (M == 0 || N == 0) return cudaSuccess;
  const dim3 grid((unsigned)((N + 63) / 64), (unsigned)((M + 63) / 64));
  small_dp4a_kernel<false><<<grid, 256, 0, s>>>(A, B, M, N, K, C);
  return cudaGetLastError();
}

cudaError_t launch_small_s4(const uint8_t* A, const uint8_t* B, int64_t M, int64_t N, int64_t K,
                            int32_t* C, cudaStream_t s) {
  if (M == 0 || N == 0) return cudaSuccess;
  const dim3 grid((unsigned)((N + 63) / 64), (unsigned)((M + 63) / 64));
  small_dp4a_kernel<true><<<grid, 256, 0, s>>>(reinterpret_cast<const int8_t*>(A),
                                               reinterpret_cast<const int8_t*>(B), M, N, K / 2, C);
  return cudaGetLastError();
}

template <int MT, int NR, int PF, int MINB, bool LINEAR>
static cudaError_t skinny_go(const int8_t* A, const int8_t* B, int M, int N, int K, int32_t* C,
                             const float* sx, const float* sw, void* Y, int sm_count,
                             cudaStream_t s) {
  const int groups = (N + NR - 1) / NR;
  const int want = (groups + kSkWarps - 1) / kSkWarps;
  const int grid = want < sm_count * MINB ? want : sm_count * MINB;
  return launch_dependent(skinny_s8_kernel<MT, NR, PF, MINB, LINEAR>, dim3(grid),
                          dim3(kSkWarps * 32), 0, s, A, B, M, N, K, C, sx, sw,
                          static_cast<__nv_bfloat16*>(Y));
}

template <bool LINEAR>
static cudaError_t skinny_pick(const int8_t* A, const int8_t* B, int M, int N, int K, int32_t* C,
                               const float* sx, const float* sw, void* Y, int sm, cudaStream_t s) {
  // (rows of A, rows of B per warp, steps per load batch, CTAs per SM), the
  // fastest of a sweep of these on GB300 at N = 11008 and 65536, K = 4096
  if (M <= 1) return skinny_go<1, 2, 4, 3, LINEAR>(A, B, M, N, K, C, sx, sw, Y, sm, s);
  if (M <= 2) return skinny_go<2, 2, 4, 3, LINEAR>(A, B, M, N, K, C, sx, sw, Y, sm, s);
  if (M <= 4) return skinny_go<4, 2, 4, 2, LINEAR>(A, B, M, N, K, C, sx, sw, Y, sm, s);
  if (M <= 8) return skinny_go<8, 4, 2, 2, LINEAR>(A, B, M, N, K, C, sx, sw, Y, sm, s);
  return skinny_go<16, 4, 2, 2, LINEAR>(A, B, M, N, K, C, sx, sw, Y, sm, s);
}

cudaError_t launch_skinny_s8(const int8_t* A, const int8_t* B, int M, int N, int K, int32_t* C,
                             const float* sx, const float* sw, void* Y, int sm_count,
                             cudaStream_t s) {
  return Y != nullptr ? skinny_pick<true>(A, B, M, N, K, C, sx, sw, Y, sm_count, s)
                      : skinny_pick<false>(A, B, M, N, K, C, sx, sw, Y, sm_count, s);
}

template <int BM, int BN, int STAGES>
static cudaError_t b1_go(const uint32_t* A, const uint32_t* B, int64_t M, int64_t N, int64_t K,
                         int32_t* C, cudaStream_t s) {
  const int smem = STAGES * (BM + BN) * kB1Stride * 4;
  const bool vec = ((K / 32) % 4 == 0) && ((reinterpret_cast<uintptr_t>(A) & 15) == 0) &&
                   ((reinterpret_cast<uintptr_t>(B) & 15) == 0);
  const dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + BM - 1) / BM));
  if (vec) {
    auto k = b1_popc_kernel<BM, BN, STAGES, true>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    k<<<grid, 256, smem, s>>>(A, B, M, N, K, C);
  } else {
    auto k = b1_popc_kernel<BM, BN, STAGES, false>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    k<<<grid, 256, smem, s>>>(A, B, M, N, K, C);
  }
  return cudaGetLastError();
}

template <int BM, int BN>
static cudaError_t b1_stages(int stages, const uint32_t* A, const uint32_t* B, int64_t M,
                             int64_t N, int64_t K, int32_t* C, cudaStream_t s) {
  switch (stages) {
    case 2: return b1_go<BM, BN, 2>(A, B, M, N, K, C, s);
    case 3: return b1_go<BM, BN, 3>(A, B, M, N, K, C, s);
    default: return b1_go<BM, BN, 4>(A, B, M, N, K, C, s);
  }
}

cudaError_t launch_b1_popc(int tile, int stages, const uint32_t* A, const uint32_t* B, int64_t M,
                           int64_t N, int64_t K, int32_t* C, cudaStream_t s) {
  if (M == 0 || N == 0) return cudaSuccess;
  switch (tile) {
    case 0: return b1_stages<64, 64>(stages, A, B, M, N, K, C, s);
    case 1: return b1_stages<128, 64>(stages, A, B, M, N, K, C, s);
    default: return b1_stages<128, 128>(stages, A, B, M, N, K, C, s);
  }
}

void b1_tile_shape(int tile, int* bm, int* bn) {
  *bm = tile == 0 ? 64 : 128;
  *bn = tile == 2 ? 128 : 64;
}

}  // namespace lbg
