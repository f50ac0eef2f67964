// tc_gemm.cuh -- the tensor-core kernel of the 8-bit and 4-bit GEMM on sm_103a.
//
// Method: "Leveraging Large-Scale Data for Efficient Low-Bit CUTLASS GEMM
// Optimization via Neural Networks" (press summary page), section 1: C is cut
// into uniform thread-block tiles, each looping over K, with a multi-stage
// pipeline overlapping loads and math; tile shape and stage count are the
// template parameters (BN, STAGES) here.
//
// GB300 design.  sm_103a has no integer tcgen05 MMA, so the integer operands
// arrive already re-encoded by an exact conversion pass: int8 -> fp16 (every
// int8 is an fp16 value) for kind::f16, and int4 -> e4m3 (every value in
// [-8, 7] is an e4m3 value) for kind::f8f6f4.  Products are then exact, and
// fp32 sums of integers are exact while their magnitude stays below 2^24, so
// the K loop is cut into chunks short enough that no fp32 accumulator can
// reach that bound (chunk_kb k-blocks); each chunk's fp32 tile is read out of
// TMEM, converted to int32 and added in registers.  Two TMEM accumulators
// alternate so that the MMA never waits for the read-out of the previous
// chunk or tile.
//
// One persistent CTA per SM slot walks output tiles of 128 x BN.  Warp roles:
//   warp 0      TMA producer: fills a STAGES-deep ring of (A, B) tiles, each a
//               128-byte-wide K slice (64 fp16 or 128 e4m3 elements) stored
//               with the 128-byte swizzle.
//   warp 1      allocates TMEM; one thread issues tcgen05.mma (4 per stage).
//   warps 2..9  epilogue: TMEM -> registers -> exact int32 sums -> global.
//               int32 C goes through a per-warp 32 x 32 staging tile in
//               shared memory (128-byte swizzle, conflict-free writes) and a
//               TMA bulk store, so each store is whole 128-byte rows; bf16 Y
//               of the linear layer is stored from registers.
// Every mbarrier wait is bounded; a wait that runs out raises the device
// status word and winds the CTA down (waiting for its own copies in flight
// and for its MMAs) before TMEM is freed.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"
#include "tc_params.h"

namespace lbg {

constexpr int kTcBM = 128;
constexpr int kTcEpiWarps = 8;
constexpr int kTcThreads = 32 * (2 + kTcEpiWarps);  // 320

template <int BN, int STAGES>
struct TcLayout {
  static constexpr int kABytes = kTcBM * 128;
  static constexpr int kBBytes = BN * 128;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kRingBytes = kStageBytes * STAGES;
  // barriers: full[S], empty[S], acc_full[2], acc_empty[2], mma_done
  static constexpr int kNumBars = 2 * STAGES + 5;
  static constexpr int kTmemCols = 2 * BN;
  // epilogue staging: per epilogue warp, one or two 32-row x 128-byte tiles
  // (two where that keeps as many CTAs per SM: a warp then fills one while
  // the other is stored)
  static constexpr int kOneBuf = kTcEpiWarps * 32 * 128;
  static constexpr int kFixed = kRingBytes + 8 * kNumBars + 8 + 1024;
  static constexpr int ctas_per_sm(int used) {
    return (512 / kTmemCols) < 233472 / (tc_smem_request(used, kTmemCols) + 1024)
               ? 512 / kTmemCols
               : 233472 / (tc_smem_request(used, kTmemCols) + 1024);
  }
  static constexpr int kEpiBufs = kFixed + 2 * kOneBuf <= 232448 &&
                                          ctas_per_sm(kFixed + 2 * kOneBuf) ==
                                              ctas_per_sm(kFixed + kOneBuf)
                                      ? 2
                                      : 1;
  static constexpr int kEpiOffset = kRingBytes;
  static constexpr int kEpiBytes = kEpiBufs * kOneBuf;
  static constexpr int kBarOffset = kEpiOffset + kEpiBytes;
  static constexpr int kTmemSlotOffset = kBarOffset + 8 * kNumBars;
  static constexpr int kAbortOffset = kTmemSlotOffset + 4;
  static constexpr int kUsedBytes = kAbortOffset + 4;
  static constexpr int kDynSmem = kUsedBytes + 1024;  // slack to align the ring to 1024
  static_assert(kDynSmem <= 232448, "shared memory of one CTA");
};

// Unit u -> tile t and its K slices [kb0, kb1); returns whether the unit's
// partial tile is added into C (else stored).  Units below dp_tiles are whole
// tiles; the rest cut each of the remaining tiles into `splits` K pieces, in
// tile-major order.  With a grid of G CTAs stepping through the units, the
// whole tiles fill complete waves when dp_tiles is a multiple of G and the
// pieces share out the last, partial wave.
__device__ __forceinline__ bool unit_range(int u, const TcParams& p, int& t, int& kb0, int& kb1) {
  if (u < p.dp_tiles) {
    t = u;
    kb0 = 0;
    kb1 = p.num_kb;
    return false;
  }
  const int v = u - p.dp_tiles;
  const int q = v / p.splits;
  const int sp = v - q * p.splits;
  t = p.dp_tiles + q;
  kb0 = (int)((int64_t)sp * p.num_kb / p.splits);
  kb1 = (int)((int64_t)(sp + 1) * p.num_kb / p.splits);
  return p.splits > 1;
}

__device__ __forceinline__ void tile_coords(int t, const TcParams& p, int& tm, int& tn) {
  const int per_group = p.group_m * p.tiles_n;
  const int g = t / per_group;
  const int first = g * p.group_m;
  const int gs = min(p.tiles_m - first, p.group_m);
  const int r = t - g * per_group;
  tm = first + r % gs;
  tn = r / gs;
}

// Waits without the abort short-cut: used to drain work already in flight.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
  uint64_t start = global_timer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 63u && global_timer_ns() - start > kWaitLimitNs) return false;
  }
}

template <int BN, bool LINEAR>
__device__ __forceinline__ void store_group(const TcParams& p, int m, int n0,
                                            const int32_t (&acc)[32]) {
  if (!LINEAR) {
    int32_t* crow = p.C + (int64_t)m * p.N;
    if (p.vec_ok && n0 + 32 <= p.N) {
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        int4 v = make_int4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
        *reinterpret_cast<int4*>(crow + n0 + j) = v;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (n0 + j < p.N) crow[n0 + j] = acc[j];
    }
  } else {
    const float s = p.sx[m];
    __nv_bfloat16* yrow = p.Y + (int64_t)m * p.N;
    if (p.vec_ok && n0 + 32 <= p.N) {
      uint32_t packed[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        float y0 = (float)acc[j] * s * __ldg(p.sw + n0 + j);
        float y1 = (float)acc[j + 1] * s * __ldg(p.sw + n0 + j + 1);
        __nv_bfloat162 h = __floats2bfloat162_rn(y0, y1);
        packed[j / 2] = *reinterpret_cast<uint32_t*>(&h);
      }
#pragma unroll
      for (int j = 0; j < 16; j += 4)
        *reinterpret_cast<uint4*>(yrow + n0 + 2 * j) =
            make_uint4(packed[j], packed[j + 1], packed[j + 2], packed[j + 3]);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (n0 + j < p.N) yrow[n0 + j] = __float2bfloat16_rn((float)acc[j] * s * p.sw[n0 + j]);
    }
  }
}

// 16 int8 values (one 16-byte chunk) -> 16 fp16 values (two chunks), exact:
// with u = v + 128 in [0, 255], the fp16 with bits 0x6400 | u is 1024 + u,
// and (1024 + u) - 1152 = v is representable, so the subtraction is exact.
__device__ __forceinline__ void s8x16_to_f16(const int4 in, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {(uint32_t)in.x ^ 0x80808080u, (uint32_t)in.y ^ 0x80808080u,
                         (uint32_t)in.z ^ 0x80808080u, (uint32_t)in.w ^ 0x80808080u};
  uint32_t o[8];
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t a = __byte_perm(w[i], 0x64646464u, 0x5140);  // bytes 0,1 -> low bytes
    const uint32_t b = __byte_perm(w[i], 0x64646464u, 0x7362);  // bytes 2,3
    __half2 ha = *reinterpret_cast<const __half2*>(&a);
    __half2 hb = *reinterpret_cast<const __half2*>(&b);
    ha = __hsub2(ha, bias);
    hb = __hsub2(hb, bias);
    o[2 * i] = *reinterpret_cast<const uint32_t*>(&ha);
    o[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&hb);
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

template <int BN, int STAGES, bool F8, bool LINEAR>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const TcParams p) {
  using L = TcLayout<BN, STAGES>;
  constexpr int kBkElems = F8 ? 128 : 64;  // elements per 128-byte K slice
  constexpr uint32_t kIdesc = instr_desc(kTcBM, BN);
  constexpr int kGroups = BN / 2 / 32;     // 32-column groups per epilogue thread

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar0 = sbase + L::kBarOffset;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t done_bar = bar0 + 8u * (2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlotOffset);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbortOffset);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), kTcEpiWarps);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;


  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      // When launched as a dependent of the re-encoding grid, wait for that
      // grid to finish (and its writes to be visible) before the first load.
      asm volatile("griddepcontrol.wait;" ::: "memory");
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int w = blockIdx.x; ok && w < p.num_units; w += gridDim.x) {
        int t, kbb, kbe, tm, tn;
        unit_range(w, p, t, kbb, kbe);
        tile_coords(t, p, tm, tn);
        for (int kb = kbb; kb < kbe; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const uint32_t sa = sbase + stage * L::kStageBytes;
          mbar_arrive_expect_tx(full_bar(stage), L::kStageBytes);
          tma_load_2d(sa, &tmA, full_bar(stage), kb * kBkElems, tm * kTcBM);
          tma_load_2d(sa + L::kABytes, &tmB, full_bar(stage), kb * kBkElems, tn * BN);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Wind-down: wait for this CTA's own copies still in flight.
        int64_t back = issued < STAGES ? issued : STAGES;
        int s = stage;
        uint32_t ph = phase;
        for (int64_t i = 0; i < back; ++i) {
          if (--s < 0) {
            s = STAGES - 1;
            ph ^= 1u;
          }
          mbar_wait_drain(full_bar(s), ph);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t u = 0;
      bool ok = true;
      for (int w = blockIdx.x; ok && w < p.num_units; w += gridDim.x) {
        int t, kbb, kbe;
        unit_range(w, p, t, kbb, kbe);
        const int num_chunks = (kbe - kbb + p.chunk_kb - 1) / p.chunk_kb;
        for (int c = 0; ok && c < num_chunks; ++c, ++u) {
          const int buf = u & 1;
          if (!mbar_wait(acce_bar(buf), ((u >> 1) & 1u) ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * BN;
          const int kb0 = kbb + c * p.chunk_kb;
          const int kb1 = min(kb0 + p.chunk_kb, kbe);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(full_bar(stage), phase, abort_flag, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = sbase + stage * L::kStageBytes;
            const uint64_t adesc = smem_desc_sw128(sa);
            const uint64_t bdesc = smem_desc_sw128(sa + L::kABytes);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              // each MMA consumes 32 bytes of K: advance the start address by 2 x 16 B
              const uint32_t accumulate = (kb > kb0 || k > 0) ? 1u : 0u;
              if (F8)
                mma_f8(d_tmem, adesc + 2 * k, bdesc + 2 * k, kIdesc, accumulate);
              else
                mma_f16(d_tmem, adesc + 2 * k, bdesc + 2 * k, kIdesc, accumulate);
            }
            mma_commit(empty_bar(stage));
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (ok) mma_commit(accf_bar(buf));
        }
      }
      mma_commit(done_bar);  // arrives once every MMA issued above has completed
    }
  } else {
    // ---------------- epilogue ----------------
    // C may have been cleared by the grid this kernel was launched as a
    // dependent of: wait for that grid before the first store into C.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int e = warp - 2;
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int row = quarter * 32 + lane;
    const int col0 = (e >> 2) * (BN / 2);
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const uint32_t stage_addr = sbase + L::kEpiOffset + e * (L::kEpiBufs * 32 * 128);
    uint32_t stores = 0;  // TMA stores issued by this warp (staging buffer = stores % kEpiBufs)
    uint32_t u = 0;
    int32_t acc[kGroups][32];
    bool ok = true;
    for (int w = blockIdx.x; ok && w < p.num_units; w += gridDim.x) {
      int t, kbb, kbe, tm, tn;
      const bool adds = unit_range(w, p, t, kbb, kbe);
      tile_coords(t, p, tm, tn);
      const int num_chunks = (kbe - kbb + p.chunk_kb - 1) / p.chunk_kb;
      for (int c = 0; c < num_chunks; ++c, ++u) {
        const int buf = u & 1;
        int got = 0;
        if (lane == 0) got = mbar_wait(accf_bar(buf), (u >> 1) & 1u, abort_flag, p.status);
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int g = 0; g < kGroups; ++g) {
          uint32_t v[32];
          tmem_ld32(tmem_base + lane_addr + buf * BN + col0 + g * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int32_t x = __float2int_rn(__uint_as_float(v[j]));
            acc[g][j] = (c == 0) ? x : acc[g][j] + x;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce_bar(buf));
      }
      if (!ok) break;
      if (!LINEAR && p.vec_ok) {
        // Row `lane` of the warp's 32 x 32 staging tile holds this thread's 32
        // columns; 16-byte chunk q sits at chunk q ^ (row % 8), the layout a
        // 128-byte-swizzled TMA box has.  The TMA store clips rows >= M and
        // columns >= N.
#pragma unroll
        for (int g = 0; g < kGroups; ++g, ++stores) {
          // the store that last used this buffer has read it
          if (lane == 0) bulk_wait_read<L::kEpiBufs - 1>();
          __syncwarp();
          const uint32_t buf = stage_addr + (stores % L::kEpiBufs) * (32 * 128);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            st_shared_v4(buf + lane * 128 + ((q ^ (lane & 7)) << 4), acc[g][4 * q],
                         acc[g][4 * q + 1], acc[g][4 * q + 2], acc[g][4 * q + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            // split K: every piece adds its partial sums into C (cleared by
            // the host); integer addition makes the order irrelevant
            if (adds)
              tma_reduce_add_2d(&tmC, buf, tn * BN + col0 + g * 32, tm * kTcBM + quarter * 32);
            else
              tma_store_2d(&tmC, buf, tn * BN + col0 + g * 32, tm * kTcBM + quarter * 32);
            bulk_commit();
          }
        }
      } else {
        const int m = tm * kTcBM + row;
        if (m < p.M) {
#pragma unroll
          for (int g = 0; g < kGroups; ++g)
            store_group<BN, LINEAR>(p, m, tn * BN + col0 + g * 32, acc[g]);
        }
      }
    }
    if (lane == 0) bulk_wait_all();
  }

  __syncthreads();
  if (warp == 1) {
    if (lane == 0) mbar_wait_drain(done_bar, 0);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, L::kTmemCols);
  }
}

template <int BN, int STAGES, bool F8, bool LINEAR>
cudaError_t tc_launch(const CUtensorMap* a, const CUtensorMap* b, const CUtensorMap* c,
                      const TcParams* p, int grid, bool pdl, cudaStream_t stream) {
  using L = TcLayout<BN, STAGES>;
  // The dynamic shared memory limit was raised once per device by the caller.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = tc_smem_request(L::kDynSmem, L::kTmemCols);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<BN, STAGES, F8, LINEAR>, *a, *b, *c, *p);
}

template <int BN, int STAGES, bool F8, bool LINEAR>
TcKernel tc_kernel_entry() {
  using L = TcLayout<BN, STAGES>;
  TcKernel k;
  k.launch = &tc_launch<BN, STAGES, F8, LINEAR>;
  k.func = reinterpret_cast<const void*>(&tc_gemm_kernel<BN, STAGES, F8, LINEAR>);
  k.threads = kTcThreads;
  k.smem = tc_smem_request(L::kDynSmem, L::kTmemCols);
  k.tmem_cols = L::kTmemCols;
  k.tile_n = BN;
  k.stages = STAGES;
  return k;
}

}  // namespace lbg
