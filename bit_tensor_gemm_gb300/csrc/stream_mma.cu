// stream_mma.cu -- the 8-bit GEMM (and linear layer) with a small side of at
// most 16 rows, streaming the large operand once from HBM through a TMA bulk
// copy ring in shared memory, on warp-level fp16 MMAs.
//
// Method: "Leveraging Large-Scale Data for Efficient Low-Bit CUTLASS GEMM
// Optimization via Neural Networks" (press summary page), intro (8-bit GEMM)
// and section 4 (the linear layer, with few tokens at inference).
//
// GB300 design.  A product with at most 16 rows on one side reads the other
// operand ("W", N rows of K bytes) once and does little arithmetic, so its
// time is that of the W stream.  Each CTA (one per SM) owns a contiguous
// block of W's rows; a producer warp copies them, 8 rows (one n8 tile of the
// MMA) per stage, with one cp.async.bulk of the stage's contiguous rows into
// a ring of up to 8 stages, completing on the stage's mbarrier (measured on
// GB300: row-sized 4 KB copies stream markedly slower than 32 KB ones).  The 16
// consumer warps split K: warp w owns K elements [w KS, (w + 1) KS), KS =
// ceil(K / 16 / 64) * 64 <= 256, and keeps the small operand X's fp16
// fragments for its slice in registers for the whole kernel (converted once;
// zero past K and past the small side's rows).  Per stage a warp reads its
// 8 x KS bytes of W, converts them to fp16 and issues KS / 16 MMAs
// m16n8k16 (X rows on the M side, W rows on the N side) into one fp32
// fragment.  Every int8 is an fp16 value, so products are exact, and a
// slice's sum is at most 256 * 2^14 = 2^22 in magnitude: exact in fp32.  The
// warps store their partial tiles as int32 into the stage's slot of a
// reduction buffer and arrive on its barrier; the producer warp adds the 16
// partials in int32, writes the 16 x 8 outputs (int32 C, or bf16 Y =
// acc * sx * sw for the linear layer), and only then refills the stage, so a
// refill also frees the slot's partials.  K order: lane (g, t) of a warp
// feeds its 16 bytes at K offset 64 j + 16 t of rows g (W) and g, g + 8 (X)
// to four MMAs, bytes 4i..4i+3 as the k pairs (2t, 2t+1), (2t+8, 2t+9) of
// MMA i; the sum over K does not depend on the order.  Int8 to fp16: the fp16
// with bits 0x6400 | u is 1024 + u, so (v ^ 0x80) in the low byte, minus
// 1152, is v exactly.  Every wait is bounded (2 s); a time-out sets the
// device status word and the CTA winds down after its copies in flight land.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "ptx.cuh"
#include "simt.h"

namespace lbg {
namespace {

constexpr int kStWarps = 16;                     // consumer warps (K slices)
constexpr int kStThreads = (kStWarps + 1) * 32;  // + the producer warp
constexpr int kStRows = 8;                       // W rows per stage
constexpr int kStMaxStages = 8;
constexpr int kStMaxK = 4096;
constexpr int kStSmemMax = 232448;
constexpr int kStRedBytes = kStWarps * 32 * 16;  // one stage's partial tiles (int32 x4 per lane)

__host__ __device__ constexpr int st_ks(int K) { return (K / 16 + 63) / 64 * 64; }
// W stage: 8 rows of K bytes, plus the bytes a slice may read past row 7's K
__host__ __device__ constexpr int st_stage_bytes(int K) {
  return (kStRows * K + 16 * st_ks(K) - K + 127) / 128 * 128;
}
// per stage: W and the partial tiles; then barriers full[S], red[S], the
// abort flag, and the linear layer's scales (sx of the small side, sw of this
// CTA's rows)
__host__ __device__ constexpr int st_scale_offset(int K, int S) {
  return S * (st_stage_bytes(K) + kStRedBytes) + 16 * S + 16;
}
__host__ __device__ constexpr int st_smem(int K, int S, int rows) {
  return st_scale_offset(K, S) + 4 * (16 + rows);
}

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

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
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

// X: MX <= 16 rows (the small side), W: NW rows, both K-major int8, K % 16 ==
// 0, K <= 4096.  Output (x, w) goes to out[x * NW + w], or out[w * MX + x]
// when TRANS.  EARLY_W: W does not depend on the grid before this one, so its
// first stages are requested before waiting on that grid.
template <bool TRANS, bool LINEAR, bool EARLY_W>
__global__ void __launch_bounds__(kStThreads, 1)
    stream_mma_kernel(const int8_t* __restrict__ X, const int8_t* __restrict__ W, int MX, int NW,
                      int K, int S, int32_t* __restrict__ C, const float* __restrict__ sx,
                      const float* __restrict__ sw, __nv_bfloat16* __restrict__ Y, int* status) {
  extern __shared__ __align__(128) uint8_t st_smem_buf[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int KS = st_ks(K), pitch = K, stage_bytes = st_stage_bytes(K);
  const uint32_t ring = smem_addr(st_smem_buf);
  const uint32_t red = ring + S * stage_bytes;
  const uint32_t bars = red + S * kStRedBytes;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto red_bar = [&](int s) { return bars + 8u * (S + s); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(st_smem_buf + S * stage_bytes +
                                                             S * kStRedBytes + 16 * S);
  // this CTA's rows of W: [r0, r1), balanced over the grid
  const int r0 = (int)((int64_t)NW * blockIdx.x / gridDim.x);
  const int r1 = (int)((int64_t)NW * (blockIdx.x + 1) / gridDim.x);
  const int stages = (r1 - r0 + kStRows - 1) / kStRows;
  float* s_sx = reinterpret_cast<float*>(st_smem_buf + st_scale_offset(K, S));
  float* s_sw = s_sx + 16;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(red_bar(s), kStWarps * 32);  // every consumer lane arrives
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kStWarps) {
    // ---- producer: W copies, then per stage the reduction and the outputs --------------
    int issued = 0;
    auto issue = [&](int st) {  // lane 0: the copy of stage st (contiguous rows) into its slot
      const int slot = st % S, n0 = r0 + st * kStRows;
      const int rows = min(kStRows, r1 - n0);
      mbar_arrive_expect_tx(full_bar(slot), (uint32_t)(rows * K));
      bulk_load(ring + slot * stage_bytes, W + (int64_t)n0 * K, (uint32_t)(rows * K),
                    full_bar(slot));
    };
    if (!EARLY_W) asm volatile("griddepcontrol.wait;" ::: "memory");
    issued = min(stages, S);
    if (lane == 0)
      for (int st = 0; st < issued; ++st) issue(st);
    // the next grid may start its prologue; it waits for this one's end
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (LINEAR) {  // the scales this CTA's outputs use, into shared memory
      if (EARLY_W) asm volatile("griddepcontrol.wait;" ::: "memory");  // sx may be the quantiser's
      if (lane < 16) s_sx[lane] = lane < MX ? sx[lane] : 0.f;
      for (int i = lane; i < r1 - r0; i += 32) s_sw[i] = sw[r0 + i];
      __syncwarp();
    }
    int done = 0;
    for (; done < stages; ++done) {
      const int slot = done % S;
      if (!mbar_wait(red_bar(slot), (uint32_t)((done / S) & 1), abort_flag, status)) break;
      // 16 partial tiles of int32: lane (g, t) adds its four outputs
      int32_t acc[4] = {0, 0, 0, 0};
#pragma unroll
      for (int w = 0; w < kStWarps; ++w) {
        const int4 v = lds16(red + slot * kStRedBytes + (w * 32 + lane) * 16);
        acc[0] += v.x;
        acc[1] += v.y;
        acc[2] += v.z;
        acc[3] += v.w;
      }
      __syncwarp();  // every lane has read the slot's partials
      if (issued < stages) {  // refill the slot: its W was read, its partials too
        if (lane == 0) issue(issued);
        ++issued;
      }
      const int n0 = r0 + done * kStRows;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int x = g + 8 * (e >> 1), w = n0 + 2 * t + (e & 1);
        if (x >= MX || w >= r1) continue;
        if (LINEAR) {
          Y[(int64_t)x * NW + w] = __float2bfloat16_rn((float)acc[e] * s_sx[x] * s_sw[w - r0]);
        } else {
          const int64_t off = TRANS ? (int64_t)w * MX + x : (int64_t)x * NW + w;
          C[off] = acc[e];
        }
      }
    }
    // after a time-out: let the copies in flight land before the CTA exits
    if (lane == 0)
      for (int st = done; st < issued; ++st) {
        const int slot = st % S;
        mbar_wait(full_bar(slot), (uint32_t)((st / S) & 1), abort_flag, status);
      }
    __syncwarp();
  } else {
    // ---- consumers: warp `warp` owns K slice [warp KS, warp KS + KS) ---------------------
    asm volatile("griddepcontrol.wait;" ::: "memory");  // X may come from the grid before
    const int kb = warp * KS;
    const int blocks = KS / 64;  // 1..4
    uint32_t xa[4][2][8];        // [block j][row g / g + 8][fp16 pairs]
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int x = g + 8 * r, k = kb + 64 * j + 16 * t;
        int4 v = make_int4(0, 0, 0, 0);
        if (j < blocks && x < MX && k < K)
          v = __ldg(reinterpret_cast<const int4*>(X + (int64_t)x * K + k));
        cvt16(v, xa[j][r]);
      }
    }
    for (int st = 0; st < stages; ++st) {
      const int slot = st % S;
      if (!mbar_wait(full_bar(slot), (uint32_t)((st / S) & 1), abort_flag, status)) break;
      float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};  // two MMA chains
      const uint32_t wrow = ring + slot * stage_bytes + g * pitch + kb + 16 * t;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (j < blocks) {
          uint32_t wb[8];
          cvt16(lds16(wrow + 64 * j), wb);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            hmma16816(d[i & 1], xa[j][0][2 * i], xa[j][1][2 * i], xa[j][0][2 * i + 1],
                      xa[j][1][2 * i + 1], wb[2 * i], wb[2 * i + 1]);
        }
      }
      // exact partial sums (|.| <= 2^22 each) as int32 into the slot's buffer
      const uint32_t dst = red + slot * kStRedBytes + (warp * 32 + lane) * 16;
      st_shared_v4(dst, __float2int_rn(d[0][0]) + __float2int_rn(d[1][0]),
                   __float2int_rn(d[0][1]) + __float2int_rn(d[1][1]),
                   __float2int_rn(d[0][2]) + __float2int_rn(d[1][2]),
                   __float2int_rn(d[0][3]) + __float2int_rn(d[1][3]));
      mbar_arrive(red_bar(slot));  // releases this lane's partials and its reads of W
    }
  }
}

template <bool TRANS, bool LINEAR, bool EARLY>
cudaError_t stream_go(const int8_t* X, const int8_t* W, int MX, int NW, int K, int32_t* C,
                      const float* sx, const float* sw, void* Y, int sm_count, int* status,
                      cudaStream_t s) {
  auto kern = stream_mma_kernel<TRANS, LINEAR, EARLY>;
  static std::atomic<int> ready[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!ready[dev].load()) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kStSmemMax);
    if (e != cudaSuccess) return e;
    ready[dev].store(1);
  }
  const int tiles = (NW + kStRows - 1) / kStRows;
  const int grid = tiles < sm_count ? tiles : sm_count;
  const int rows = (NW + grid - 1) / grid;  // most rows a CTA owns
  int S = kStMaxStages;
  while (S > 2 && st_smem(K, S, rows) > kStSmemMax) --S;
  if (st_smem(K, S, rows) > kStSmemMax) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kStThreads);
  cfg.dynamicSmemBytes = st_smem(K, S, rows);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, X, W, MX, NW, K, S, C, sx, sw,
                            static_cast<__nv_bfloat16*>(Y), status);
}

}  // namespace

int64_t stream_mma_max_k() { return kStMaxK; }

cudaError_t launch_stream_mma(const int8_t* X, const int8_t* W, int MX, int NW, int K, bool trans,
                              int32_t* C, const float* sx, const float* sw, void* Y, bool early_w,
                              int sm_count, int* status, cudaStream_t s) {
  if (MX < 1 || MX > 16 || K < 16 || K > kStMaxK || K % 16 || NW < 1) return cudaErrorInvalidValue;
  if (Y != nullptr) {
    if (trans) return cudaErrorInvalidValue;
    return early_w ? stream_go<false, true, true>(X, W, MX, NW, K, C, sx, sw, Y, sm_count, status, s)
                   : stream_go<false, true, false>(X, W, MX, NW, K, C, sx, sw, Y, sm_count, status,
                                                   s);
  }
  return trans ? stream_go<true, false, false>(X, W, MX, NW, K, C, sx, sw, Y, sm_count, status, s)
               : stream_go<false, false, false>(X, W, MX, NW, K, C, sx, sw, Y, sm_count, status, s);
}

}  // namespace lbg
