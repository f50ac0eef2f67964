// hmma_skinny.cu -- the 8-bit GEMM for a small side of at most 32 rows on the
// warp-level fp16 MMA (mma.sync m16n8k16, fp32 accumulators), with the int8
// operands converted to fp16 in registers.
//
// Method: "Leveraging Large-Scale Data for Efficient Low-Bit CUTLASS GEMM
// Optimization via Neural Networks" (press summary page), intro (8-bit GEMM)
// and section 4 (the linear layer, whose token count is small at inference).
//
// GB300 design.  With one side of only a few rows the product streams the
// large operand ("W", whose rows are the MMA's n8 columns) from HBM once and
// the arithmetic is small; but the integer paths are slow on this GPU (dp4a
// and the int8 mma.sync both measure about 150 TOPS), while mma.sync on fp16
// measures about 600 TFLOP/s.  Every int8 value is an fp16 value, products are
// exact, and an fp32 sum of integers is exact while its magnitude stays within
// 2^24; the fp32 fragments are added into int32 registers every 1024 K.  The
// sum over K does not depend on the order of K, so lane (g, t) feeds its 16
// bytes of K positions 16 (t + 4h) of a step (of W's row g and of X's rows g,
// g + 8) to four MMAs as its fragment columns: the k pairs (2t, 2t+1) and
// (2t+8, 2t+9) of MMA i are bytes 4i..4i+3 of the 16.  The conversion: the
// fp16 with bits 0x6400 | u is 1024 + u, so (v ^ 0x80) placed in the low byte,
// minus 1152, is v, exactly.
//
// Streaming W.  HBM delivers full bandwidth to coalesced rows: every load
// instruction of a warp copies 256 contiguous bytes of each of two rows
// (cp.async, 16 bytes a lane) into a PF-stage ring of the warp in shared
// memory, which the lanes then read in fragment order (rows 320 bytes apart,
// so the 16-byte reads of a quarter-warp -- rows g and g + 1 -- fall in
// distinct banks).  The work is spread over every SM with enough warps to
// hide the latency of each warp's instruction chain: a CTA owns U units of
// 16 rows of W (two n8 tiles), and its 16 warps split them into U x KP items,
// KP parts of K each (steps kp, kp + KP, ...); the parts' int32 sums are
// added in shared memory at the end.  The CTA keeps its 16 MT rows of X as
// int8 in shared memory (row stride = 64 mod 128 bytes), converted where used.
// One launch, no scratch.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "simt.h"

namespace lbg {
namespace {

constexpr int kHmWarps = 16;
constexpr int kHmNT = 2;                   // n8 tiles per warp
constexpr int kHmRows = 8 * kHmNT;         // rows of W per warp
constexpr int kHmStep = 256;               // K elements per step
constexpr int kHmPF = 2;                   // steps of W in flight per warp
constexpr int kHmPitch = kHmStep + 64;     // bytes between rows of a stage (= 64 mod 128)
constexpr int kHmSmemMax = 232448;         // shared memory a CTA may use
constexpr int kHmStageBytes = kHmRows * kHmPitch;
constexpr int kHmRingBytes = kHmWarps * kHmPF * kHmStageBytes;


// 4 int8 (one 32-bit word) -> two f16x2 words: bytes (0, 1) and (2, 3).
__device__ __forceinline__ void s8x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t a = __byte_perm(u, 0x64646464u, 0x5140);
  const uint32_t b = __byte_perm(u, 0x64646464u, 0x7362);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
  __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
  lo = *reinterpret_cast<const uint32_t*>(&ha);
  hi = *reinterpret_cast<const uint32_t*>(&hb);
}

__device__ __forceinline__ void cvt16(const int4 v, uint32_t (&o)[8]) {
  s8x4_to_f16x2((uint32_t)v.x, o[0], o[1]);
  s8x4_to_f16x2((uint32_t)v.y, o[2], o[3]);
  s8x4_to_f16x2((uint32_t)v.z, o[4], o[5]);
  s8x4_to_f16x2((uint32_t)v.w, o[6], o[7]);
}

__device__ __forceinline__ void hmma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9},"
      " {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(ok ? 16 : 0)
               : "memory");
}

__device__ __forceinline__ int4 lds16(uint32_t addr) {
  int4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// row stride of int8 X in shared memory: >= K, = 64 mod 128
__host__ __device__ constexpr int hm_xstride(int K) { return (K + 127) / 128 * 128 + 64; }

// X: MX rows (the small side), W: NW rows, both K-major int8 (K % 16 == 0).
// Output element (x, w) goes to out[x * NW + w], or out[w * MX + x] when TRANS.
template <int MT, bool TRANS, bool LINEAR>
__global__ void __launch_bounds__(kHmWarps * 32)
    hmma_skinny_kernel(const int8_t* __restrict__ X, const int8_t* __restrict__ W, int MX, int NW,
                       int K, int32_t* __restrict__ C, const float* __restrict__ sx,
                       const float* __restrict__ sw, __nv_bfloat16* __restrict__ Y,
                       int chunk_steps, int U, int KP) {
  constexpr int NACC = 4 / MT;  // independent accumulators per (m tile, n8 tile)
  // launched as a programmatic dependent: X (and its scales) may come from
  // the grid before this one (the activation quantiser), which may still be
  // running; wait for it before the first read
  asm volatile("griddepcontrol.wait;" ::: "memory");
  extern __shared__ int4 hm_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int m0 = blockIdx.y * (MT * 16);
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(hm_smem);
  const uint32_t ring = sbase + (uint32_t)(warp * kHmPF * kHmStageBytes);
  const uint32_t xs = sbase + kHmRingBytes;
  const int xstride = hm_xstride(K);

  // X rows m0 .. m0 + 16 MT - 1 into shared memory (zero beyond MX), coalesced
  const int chunks = K / 16;
  for (int i = threadIdx.x; i < MT * 16 * chunks; i += kHmWarps * 32) {
    const int r = i / chunks, c = i - r * chunks;
    const int m = m0 + r;
    cp_async16(xs + r * xstride + 16 * c, X + (int64_t)(m < MX ? m : 0) * K + 16 * c, m < MX);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");

  const int steps = (K + kHmStep - 1) / kHmStep;
  const int units = (NW + kHmRows - 1) / kHmRows;
  const int u_local = warp % U, kp = warp / U;  // this warp's item of the CTA
  const bool active = kp < KP;
  // this item's steps of a unit: kp, kp + KP, ... (none for an idle warp or unit)
  auto item_steps = [&](int unit) {
    return active && unit < units && kp < steps ? (steps - kp + KP - 1) / KP : 0;
  };
  // step s of the 16 rows from n0 into stage q: each instruction copies 256
  // contiguous bytes of two rows; always one (possibly empty) group per call
  auto fill = [&](int n0, int q, int s) {
    if (s < steps) {
      const int k = s * kHmStep + 16 * (lane & 15);
#pragma unroll
      for (int r = 0; r < kHmRows; r += 2) {
        const int row = n0 + r + (lane >> 4);
        const bool ok = row < NW && k < K;
        cp_async16(ring + q * kHmStageBytes + (r + (lane >> 4)) * kHmPitch + 16 * (lane & 15),
                   W + (ok ? (int64_t)row * K + k : 0), ok);
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  auto fill_first = [&](int unit) {
    const int my = item_steps(unit);
#pragma unroll
    for (int q = 0; q < kHmPF; ++q) fill(unit * kHmRows, q, q < my ? kp + KP * q : steps);
  };
  // the first unit's W copies are in flight while X lands
  fill_first(blockIdx.x * U + u_local);
  asm volatile("cp.async.wait_group %0;" ::"n"(kHmPF) : "memory");  // X has landed
  __syncthreads();

  // partial sums of every item, added at the end (reuses the rings)
  int32_t* red = reinterpret_cast<int32_t*>(hm_smem);
  for (int ubase = blockIdx.x * U; ubase < units; ubase += gridDim.x * U) {
    const int unit = ubase + u_local;
    const int n0 = unit * kHmRows;
    const int my_steps = item_steps(unit);

    float accf[MT][kHmNT][NACC][4];
    int32_t acci[MT][kHmNT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int j = 0; j < kHmNT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acci[mt][j][e] = 0;
#pragma unroll
          for (int c = 0; c < NACC; ++c) accf[mt][j][c][e] = 0.f;
        }
    int since_drain = 0;
    for (int i0 = 0; i0 < my_steps; i0 += kHmPF) {
#pragma unroll
      for (int q = 0; q < kHmPF; ++q) {
        const int it = i0 + q;
        if (it >= my_steps) break;
        const int s = kp + KP * it;
        // the copies of step s (every lane's) have landed
        asm volatile("cp.async.wait_group %0;" ::"n"(kHmPF - 1) : "memory");
        __syncwarp();
#pragma unroll
        for (int h = 0; h < kHmStep / 64; ++h) {
          const int k = s * kHmStep + 16 * (t + 4 * h);
          uint32_t xa[MT][2][8];  // rows g and g + 8 of each m tile, fp16 pairs
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int r = 0; r < 2; ++r)
              cvt16(k < K ? lds16(xs + (16 * mt + 8 * r + g) * xstride + k)
                          : make_int4(0, 0, 0, 0),
                    xa[mt][r]);
#pragma unroll
          for (int j = 0; j < kHmNT; ++j) {
            uint32_t wb[8];
            cvt16(lds16(ring + q * kHmStageBytes + (8 * j + g) * kHmPitch + 16 * (t + 4 * h)),
                  wb);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
              for (int mt = 0; mt < MT; ++mt)
                hmma16816(accf[mt][j][((h & 1) * 4 + i) % NACC], xa[mt][0][2 * i],
                          xa[mt][1][2 * i], xa[mt][0][2 * i + 1], xa[mt][1][2 * i + 1], wb[2 * i],
                          wb[2 * i + 1]);
          }
        }
        __syncwarp();    // every lane has read stage q
        fill(n0, q, it + kHmPF < my_steps ? s + KP * kHmPF : steps);
        if (++since_drain == chunk_steps) {  // exact fp32 partial sums -> int32
          since_drain = 0;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int j = 0; j < kHmNT; ++j)
#pragma unroll
              for (int e = 0; e < 4; ++e)
#pragma unroll
                for (int c = 0; c < NACC; ++c) {
                  acci[mt][j][e] += __float2int_rn(accf[mt][j][c][e]);
                  accf[mt][j][c][e] = 0.f;
                }
        }
      }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");  // nothing left in flight
    __syncthreads();  // every ring is read: its memory holds the partial sums now
    // item (u_local, kp) at red[((kp * U + u_local) * 16 MT + row) * 16 + col]
    if (active) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int j = 0; j < kHmNT; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            int32_t v = acci[mt][j][e];
#pragma unroll
            for (int c = 0; c < NACC; ++c) v += __float2int_rn(accf[mt][j][c][e]);
            const int row = 16 * mt + g + 8 * (e >> 1), col = 8 * j + 2 * t + (e & 1);
            red[((kp * U + u_local) * 16 * MT + row) * kHmRows + col] = v;
          }
    }
    __syncthreads();
    const int outs = U * 16 * MT * kHmRows;
    for (int i = threadIdx.x; i < outs; i += kHmWarps * 32) {
      // TRANS: consecutive threads take consecutive x (contiguous in the output)
      const int ul = i / (16 * MT * kHmRows), rem = i - ul * (16 * MT * kHmRows);
      const int row = TRANS ? rem % (16 * MT) : rem / kHmRows;
      const int col = TRANS ? rem / (16 * MT) : rem % kHmRows;
      const int x = m0 + row, w = (ubase + ul) * kHmRows + col;
      if (x >= MX || w >= NW) continue;
      int32_t v = 0;
      for (int q = 0; q < KP; ++q) v += red[((q * U + ul) * 16 * MT + row) * kHmRows + col];
      const int64_t off = TRANS ? (int64_t)w * MX + x : (int64_t)x * NW + w;
      if (LINEAR)
        Y[off] = __float2bfloat16_rn((float)v * sx[x] * sw[w]);
      else
        C[off] = v;
    }
    __syncthreads();  // the rings are free again
    fill_first(ubase + gridDim.x * U + u_local);  // the next unit's first steps
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

template <int MT, bool TRANS, bool LINEAR>
cudaError_t hmma_go(const int8_t* X, const int8_t* W, int MX, int NW, int K, int32_t* C,
                    const float* sx, const float* sw, void* Y, int chunk_elems, int sm_count,
                    cudaStream_t s) {
  auto kern = hmma_skinny_kernel<MT, TRANS, LINEAR>;
  const int smem = kHmRingBytes + MT * 16 * hm_xstride(K);
  // raise the shared-memory limit once per device (to the most any K needs);
  // the kernel's shared memory allows one CTA per SM
  static std::atomic<int> ready[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!ready[dev].load()) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kHmSmemMax);
    if (e != cudaSuccess) return e;
    ready[dev].store(1);
  }
  // U units of 16 rows per CTA, so that one wave of CTAs covers W; the 16
  // warps split each unit's K into KP parts
  const int units = (NW + kHmRows - 1) / kHmRows;
  const int m_blocks = (MX + MT * 16 - 1) / (MT * 16);
  const int ctas = sm_count / m_blocks > 0 ? sm_count / m_blocks : 1;
  int U = (units + ctas - 1) / ctas;
  if (U > kHmWarps) U = kHmWarps;
  const int KP = kHmWarps / U;
  const int gx = (units + U - 1) / U < ctas ? (units + U - 1) / U : ctas;
  const int chunk_steps = chunk_elems / kHmStep > 0 ? chunk_elems / kHmStep : 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(gx, m_blocks);
  cfg.blockDim = dim3(kHmWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, X, W, MX, NW, K, C, sx, sw,
                            static_cast<__nv_bfloat16*>(Y), chunk_steps, U, KP);
}

template <bool TRANS, bool LINEAR>
cudaError_t hmma_pick(const int8_t* X, const int8_t* W, int MX, int NW, int K, int32_t* C,
                      const float* sx, const float* sw, void* Y, int chunk, int sm,
                      cudaStream_t s) {
  if (MX <= 16) return hmma_go<1, TRANS, LINEAR>(X, W, MX, NW, K, C, sx, sw, Y, chunk, sm, s);
  return hmma_go<2, TRANS, LINEAR>(X, W, MX, NW, K, C, sx, sw, Y, chunk, sm, s);
}

}  // namespace

int64_t hmma_skinny_max_k(int MX) {
  // the CTA's rows of X (16 or 32, int8) next to the W rings in shared memory
  const int64_t rows = MX <= 16 ? 16 : 32;
  return ((kHmSmemMax - kHmRingBytes) / rows - 64) / 128 * 128;
}

cudaError_t launch_hmma_skinny(const int8_t* X, const int8_t* W, int MX, int NW, int K,
                               bool trans, int32_t* C, const float* sx, const float* sw, void* Y,
                               int chunk_elems, int sm_count, cudaStream_t s) {
  const int c = chunk_elems, sm = sm_count;
  if (Y != nullptr)
    return trans ? hmma_pick<true, true>(X, W, MX, NW, K, C, sx, sw, Y, c, sm, s)
                 : hmma_pick<false, true>(X, W, MX, NW, K, C, sx, sw, Y, c, sm, s);
  return trans ? hmma_pick<true, false>(X, W, MX, NW, K, C, sx, sw, Y, c, sm, s)
               : hmma_pick<false, false>(X, W, MX, NW, K, C, sx, sw, Y, c, sm, s);
}

}  // namespace lbg
