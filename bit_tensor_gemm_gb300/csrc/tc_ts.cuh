// tc_ts.cuh -- the tensor-core 8-bit GEMM that converts one operand from int8
// inside the kernel and feeds it to the MMA from tensor memory.
//
// Method: the tiling of "Leveraging Large-Scale Data for Efficient Low-Bit
// CUTLASS GEMM Optimization via Neural Networks" (press summary page), section
// 1: uniform output tiles, a K loop per tile, a multi-stage load pipeline
// (template parameter STAGES).  The integer product is exact as in
// tc_gemm.cuh: int8 values are fp16 values, products are exact, and the K loop
// is cut into chunks in which no fp32 sum can pass 2^24, each chunk's fp32
// tile being added into int32 registers.
//
// GB300 design.  The re-encoding pass that tc_gemm_kernel depends on costs 3
// bytes of HBM traffic per int8 element (read 1, write 2) and one more read of
// 2 bytes by the GEMM: for a problem whose operands are large next to its
// arithmetic that is most of the time.  Here the MMA's A operand (the "L"
// operand, 128 rows per tile) stays int8 in global memory:
//   - TMA copies each K slice of its 128 rows (SK / 128 boxes of 16 KB,
//     128-byte rows with the 128-byte swizzle) into a staging ring in shared
//     memory;
//   - four converter warps, one per 32-lane quarter of tensor memory, read
//     their rows (thread t of quarter q owns row 32q + t; with the swizzle the
//     32 threads' 16-byte reads hit distinct banks), turn each 64 int8 values
//     into 32 words of packed fp16 (exact: the fp16 with bits 0x6400 | (v+128)
//     is 1024 + v + 128, minus 1152 gives v) and store them with tcgen05.st
//     into a ring of 64-column slots of tensor memory;
//   - the MMA thread issues tcgen05.mma with A read from tensor memory and B
//     (the "S" operand, BN rows, re-encoded to fp16 ahead by the library's
//     pass) read from shared memory.
// Compared with converting into shared memory (the operand tile would be
// written as fp16 and read again by the MMA), the tensor-memory route moves
// 16 KB instead of 80 KB of shared memory per 128-row K slice.
//
// Slice size (template parameter SK: 128 or 256 elements).  Every slice
// costs each role a fixed number of barrier operations (a wait for the int8
// data, a wait for the freed slot, arrivals, a commit) of roughly 100 cycles
// each on GB300; instrumented, the roles of a 64-element version spent ~1000
// cycles per slice, of which the MMAs (four of 128 x BN x 16) and the
// conversion were only a third.  Longer slices cut those operations per
// byte, but a slice's A slot takes SK / 2 columns of tensor memory: beside
// two 128-column accumulators only two 256-element slots fit, too shallow a
// pipeline (measured: the 64-wide kernel is up to 10 % faster with 256, the
// 128-wide one up to 14 % slower).
//
// Output.  D's lane i and column j hold the sum for L-row i and S-row j.
// TRANS = false: L is the GEMM's A, S its B, C[i][j] as in tc_gemm_kernel
// (TMA bulk stores of swizzled 32 x 32 blocks, or plain stores).
// TRANS = true: L is the GEMM's B and S its A, so C[j][i] = D[i][j]: the
// warp's 32 lanes hold 32 consecutive columns of C for one row of C, and each
// of its stores writes 128 contiguous bytes (red.add under split K).
//
// Tensor memory: two fp32 accumulators of BN columns (alternating per K chunk,
// as in tc_gemm_kernel), then STAGES slots of SK / 2 columns for A.
//
// Roles (448 threads):
//   warp 0 lane 0   TMA producer of the int8 staging ring (L operand)
//   warp 1          tensor-memory allocation; lane 0 issues MMAs and commits
//   warps 2..9      epilogue (two per tensor-memory quarter, half the columns each)
//   warps 10..13    converters; lane 0 of warp 10 also issues the TMA of the
//                   S operand into the shared-memory slot of the same stage,
//                   once that stage's MMAs have completed
// Every wait is bounded; on a time-out the CTA winds down as tc_gemm_kernel
// does (its own copies in flight and its MMAs are waited for before tensor
// memory is freed).
#pragma once
#include "tc_gemm.cuh"

namespace lbg {

constexpr int kTsConvWarps = 4;
constexpr int kTsThreads = 32 * (2 + kTcEpiWarps + kTsConvWarps);  // 448

__host__ __device__ constexpr int ts_tmem_cols(int need) {
  return need <= 32 ? 32 : need <= 64 ? 64 : need <= 128 ? 128 : need <= 256 ? 256 : 512;
}

// SK: K elements per slice (one staging stage, one A slot), 128 or 256.
template <int BN, int STAGES, int SK>
struct TsLayout {
  static_assert(SK == 128 || SK == 256, "K slices of 128 or 256 elements");
  // one slice of the S operand: SK / 64 fp16 boxes of 64 elements (128-byte
  // rows, 128-byte swizzle) of BN rows each
  static constexpr int kSBoxBytes = BN * 128;
  static constexpr int kSBoxes = SK / 64;
  static constexpr int kSBytes = kSBoxes * kSBoxBytes;
  static constexpr int kRingBytes = kSBytes * STAGES;
  static constexpr int kEpiOffset = kRingBytes;
  static constexpr int kEpiBytes = kTcEpiWarps * 32 * 128;
  static constexpr int kStgOffset = kEpiOffset + kEpiBytes;
  static constexpr int kStgStages = STAGES;
  // SK / 128 TMA boxes of 128 rows x 128 int8 (128-byte swizzle)
  static constexpr int kStgBoxBytes = kTcBM * 128;
  static constexpr int kStgBoxes = SK / 128;
  static constexpr int kStgStageBytes = kStgBoxBytes * kStgBoxes;
  static constexpr int kStgBytes = kStgStageBytes * kStgStages;
  // barriers: full[S], empty[S], conv[S], acc_full[2], acc_empty[2], mma_done,
  // stg_full[SS], stg_empty[SS]
  static constexpr int kNumBars = 3 * STAGES + 5 + 2 * kStgStages;
  static constexpr int kBarOffset = kStgOffset + kStgBytes;
  static constexpr int kTmemSlotOffset = kBarOffset + 8 * kNumBars;
  static constexpr int kAbortOffset = kTmemSlotOffset + 4;
  static constexpr int kUsedBytes = kAbortOffset + 4;
  static constexpr int kDynSmem = kUsedBytes + 1024;  // slack to align the ring to 1024
  static constexpr int kAccCols = 2 * BN;
  static constexpr int kACol0 = kAccCols;  // first column of the A slots
  static constexpr int kASlotCols = SK / 2;  // packed fp16 pairs per row
  static constexpr int kTmemCols = ts_tmem_cols(kAccCols + kASlotCols * STAGES);
  static_assert(kAccCols + kASlotCols * STAGES <= 512, "tensor memory holds 512 columns");
  static_assert(kDynSmem <= 232448, "shared memory per CTA");
};

// Unit w of this CTA (w % gridDim.x == blockIdx.x): a tile t and its K
// slices [kb0, kb1) (kb0 == kb1: nothing to do).  With stream_k the CTA's
// run of the tile-major slice order is cut at tile ends; the i-th piece is
// unit blockIdx.x + i * gridDim.x.
__device__ __forceinline__ void ts_unit(int w, const TcParams& p, int& t, int& kb0, int& kb1) {
  if (!p.stream_k) {
    unit_range(w, p, t, kb0, kb1);
    return;
  }
  const int g = (int)gridDim.x;
  const int b = w % g, i = w / g;
  const int64_t total = (int64_t)p.num_tiles * p.num_kb;
  const int64_t s0 = (int64_t)b * total / g, s1 = (int64_t)(b + 1) * total / g;
  const int64_t a = i == 0 ? s0 : (s0 / p.num_kb + i) * p.num_kb;
  if (a >= s1) {
    t = kb0 = kb1 = 0;
    return;
  }
  const int64_t e = min(s1, (a / p.num_kb + 1) * p.num_kb);
  t = (int)(a / p.num_kb);
  kb0 = (int)(a - (int64_t)t * p.num_kb);
  kb1 = kb0 + (int)(e - a);
}

template <int BN, int STAGES, int SK, bool TRANS, bool LINEAR>
__global__ void __launch_bounds__(kTsThreads, 1)
    tc_ts_kernel(const __grid_constant__ CUtensorMap tmL, const __grid_constant__ CUtensorMap tmS,
                 const __grid_constant__ CUtensorMap tmC, const TcParams p) {
  using L = TsLayout<BN, STAGES, SK>;
  constexpr int kQuarters = SK / 64;  // 64-element pieces a converter handles per slice
  constexpr int SS = L::kStgStages;
  constexpr uint32_t kIdesc = instr_desc(kTcBM, BN);
  constexpr int kGroups = BN / 2 / 32;  // 32-column groups per epilogue thread

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar0 = sbase + L::kBarOffset;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto conv_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (3 * STAGES + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (3 * STAGES + 2 + b); };
  const uint32_t done_bar = bar0 + 8u * (3 * STAGES + 4);
  auto stgf_bar = [&](int s) { return bar0 + 8u * (3 * STAGES + 5 + s); };
  auto stge_bar = [&](int s) { return bar0 + 8u * (3 * STAGES + 5 + SS + s); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlotOffset);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbortOffset);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(conv_bar(s), kTsConvWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), kTcEpiWarps);
    }
    mbar_init(done_bar, 1);
    for (int s = 0; s < SS; ++s) {
      mbar_init(stgf_bar(s), 1);
      mbar_init(stge_bar(s), kTsConvWarps);
    }
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
    // ---------------- TMA producer of the int8 staging ring ----------------
    // The L operand is the caller's int8 array: stream order already put every
    // earlier write to it before the re-encoding grid this kernel may overlap.
    if (lane == 0) {
      tma_prefetch_desc(&tmL);
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int w = blockIdx.x; ok && w < p.num_units; w += gridDim.x) {
        int t, kbb, kbe, tm, tn;
        ts_unit(w, p, t, kbb, kbe);
        tile_coords(t, p, tm, tn);
        for (int kb = kbb; kb < kbe; ++kb) {
          if (!mbar_wait(stge_bar(stage), phase ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const uint32_t st = sbase + L::kStgOffset + stage * L::kStgStageBytes;
          mbar_arrive_expect_tx(stgf_bar(stage), L::kStgStageBytes);
#pragma unroll
          for (int b = 0; b < L::kStgBoxes; ++b)
            tma_load_2d(st + b * L::kStgBoxBytes, &tmL, stgf_bar(stage), kb * SK + 128 * b,
                        tm * kTcBM);
          ++issued;
          if (++stage == SS) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Wind-down: wait for this CTA's own copies still in flight.
        const int64_t back = issued < SS ? issued : SS;
        int s = stage;
        uint32_t ph = phase;
        for (int64_t i = 0; i < back; ++i) {
          if (--s < 0) {
            s = SS - 1;
            ph ^= 1u;
          }
          mbar_wait_drain(stgf_bar(s), ph);
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
        ts_unit(w, p, t, kbb, kbe);
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
            if (!mbar_wait(full_bar(stage), phase, abort_flag, p.status) ||
                !mbar_wait(conv_bar(stage), phase, abort_flag, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t s_addr = sbase + stage * L::kSBytes;
            const uint32_t a_tmem = tmem_base + L::kACol0 + stage * L::kASlotCols;
#pragma unroll
            for (int k = 0; k < SK / 16; ++k) {
              // K = 16 per MMA: 8 columns of A, 32 bytes (2 x 16 B) of each B
              // row, in 64-element box k / 4 of the slice
              const uint64_t bdesc = smem_desc_sw128(s_addr + (k >> 2) * L::kSBoxBytes);
              const uint32_t accumulate = (kb > kb0 || k > 0) ? 1u : 0u;
              mma_f16_ts(d_tmem, a_tmem + 8 * k, bdesc + 2 * (k & 3), kIdesc, accumulate);
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
  } else if (warp >= 2 + kTcEpiWarps) {
    // ---------------- converters ----------------
    const int quarter = warp & 3;  // tensor-memory lanes this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const bool loader = warp == 2 + kTcEpiWarps && lane == 0;
    if (loader) {
      tma_prefetch_desc(&tmS);
      // The S operand comes from the re-encoding grid this kernel may have
      // been launched as a dependent of: wait for it before the first load.
      asm volatile("griddepcontrol.wait;" ::: "memory");
    }
    // 128-byte swizzle: 16-byte chunk q of row r sits at chunk q ^ (r % 8)
    const int swz = row & 7;
    // The slices this CTA converts, in order: (unit w, slice kb), each in
    // pieces of 64 elements.
    int w = (int)blockIdx.x - (int)gridDim.x;  // the unit before this CTA's first
    int kb = 0, kbe = 0, tn = 0;
    auto advance = [&]() -> bool {  // next slice into (kb, tn); false at the end
      if (++kb < kbe) return true;
      for (w += gridDim.x; w < p.num_units; w += gridDim.x) {
        int t, kbb, tm;
        ts_unit(w, p, t, kbb, kbe);
        tile_coords(t, p, tm, tn);
        if (kbb < kbe) {
          kb = kbb;
          return true;
        }
      }
      return false;
    };
    int os = 0, ss = 0;  // stage and staging slot of the slice being prepared
    uint32_t oph = 0, sph = 0;
    int ls = 0;          // loader: next stage to fill, and its phase
    uint32_t lph = 0;
    int64_t issued = 0;
    // wait until slot (os, ss) may be written and its int8 data has landed;
    // the loader also fills the S operand of stage os (two boxes)
    auto acquire = [&]() -> bool {
      int got = 1;
      if (lane == 0) {
        got = mbar_wait(empty_bar(os), oph ^ 1u, abort_flag, p.status);
        if (got && loader) {
          const uint32_t dst = sbase + os * L::kSBytes;
          mbar_arrive_expect_tx(full_bar(os), L::kSBytes);
#pragma unroll
          for (int b = 0; b < L::kSBoxes; ++b)
            tma_load_2d(dst + b * L::kSBoxBytes, &tmS, full_bar(os), kb * SK + 64 * b, tn * BN);
          ++issued;
          if (++ls == STAGES) {
            ls = 0;
            lph ^= 1u;
          }
        }
        got = got && mbar_wait(stgf_bar(ss), sph, abort_flag, p.status);
      }
      return __shfl_sync(0xffffffffu, got, 0) != 0;
    };
    // piece h (64 elements, 32 words) of this thread's row of staging slot ss:
    // box h / 2, 16-byte chunks 4 (h % 2) .. 4 (h % 2) + 3 of the row
    auto convert = [&](int h, uint32_t (&words)[32]) {
      const uint8_t* src = smem + L::kStgOffset + ss * L::kStgStageBytes +
                           (h >> 1) * L::kStgBoxBytes + row * 128;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int4 v = *reinterpret_cast<const int4*>(src + (((4 * (h & 1) + q) ^ swz) << 4));
        uint4 lo, hi;
        s8x16_to_f16(v, lo, hi);
        words[8 * q + 0] = lo.x;
        words[8 * q + 1] = lo.y;
        words[8 * q + 2] = lo.z;
        words[8 * q + 3] = lo.w;
        words[8 * q + 4] = hi.x;
        words[8 * q + 5] = hi.y;
        words[8 * q + 6] = hi.z;
        words[8 * q + 7] = hi.w;
      }
    };
    bool have = advance();
    bool ok = true;
    uint32_t cur[32];
    if (have) {
      ok = acquire();
      if (ok) convert(0, cur);
    }
    while (ok && have) {
      // Store each piece as soon as it is converted: tcgen05.st reads its
      // registers when it issues, so the next piece is converted into the
      // same registers while the stores are in flight, and the slice waits
      // for its stores once.  Its A slot and staging slot are handed on
      // before the next slice's wait (a slot and its int8 data) begins.
      const uint32_t slot = tmem_base + lane_addr + L::kACol0 + os * L::kASlotCols;
#pragma unroll
      for (int h = 0; h < kQuarters; ++h) {
        if (h > 0) convert(h, cur);
        tmem_st32(slot + 32 * h, cur);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(conv_bar(os));
        mbar_arrive(stge_bar(ss));
      }
      if (++os == STAGES) {
        os = 0;
        oph ^= 1u;
      }
      if (++ss == SS) {
        ss = 0;
        sph ^= 1u;
      }
      have = advance();
      if (have) {
        ok = acquire();
        if (ok) convert(0, cur);
      }
    }
    if (!ok && loader) {
      // Wind-down: wait for the S copies this thread still has in flight.
      const int64_t back = issued < STAGES ? issued : STAGES;
      int s2 = ls;
      uint32_t ph = lph;
      for (int64_t i = 0; i < back; ++i) {
        if (--s2 < 0) {
          s2 = STAGES - 1;
          ph ^= 1u;
        }
        mbar_wait_drain(full_bar(s2), ph);
      }
    }
  } else {
    // ---------------- epilogue ----------------
    // C may have been cleared by the grid this kernel was launched as a
    // dependent of: wait for that grid before the first store into C.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int e = warp - 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int col0 = (e >> 2) * (BN / 2);
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const uint32_t stage_addr = sbase + L::kEpiOffset + e * (32 * 128);
    uint32_t u = 0;
    int32_t acc[kGroups][32];
    bool ok = true;
    // partial tiles (split K, stream-K) are added into C, cleared beforehand
    const bool adds = p.splits > 1 || p.stream_k > 0;
    for (int w = blockIdx.x; ok && w < p.num_units; w += gridDim.x) {
      int t, kbb, kbe, tm, tn;
      ts_unit(w, p, t, kbb, kbe);
      tile_coords(t, p, tm, tn);
      const int num_chunks = (kbe - kbb + p.chunk_kb - 1) / p.chunk_kb;
      if (num_chunks == 0) continue;  // an empty stream-K unit
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
      const int i = tm * kTcBM + row;  // L row
      if (TRANS) {
        // C[j][i]: for a fixed j the warp's lanes write 32 consecutive ints
        if (i < p.M) {
#pragma unroll
          for (int g = 0; g < kGroups; ++g) {
            const int j0 = tn * BN + col0 + g * 32;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int jj = j0 + j;
              if (jj < p.N) {
                const int64_t off = (int64_t)jj * p.M + i;
                if (LINEAR) {
                  p.Y[off] = __float2bfloat16_rn((float)acc[g][j] * p.sx[jj] * p.sw[i]);
                } else if (adds) {
                  atomicAdd(p.C + off, acc[g][j]);
                } else {
                  p.C[off] = acc[g][j];
                }
              }
            }
          }
        }
      } else if (!LINEAR && p.vec_ok) {
        // swizzled 32 x 32 staging tile per warp, then a TMA bulk store (as
        // in tc_gemm_kernel); the store clips rows >= M and columns >= N
#pragma unroll
        for (int g = 0; g < kGroups; ++g) {
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
#pragma unroll
          for (int q = 0; q < 8; ++q)
            st_shared_v4(stage_addr + lane * 128 + ((q ^ (lane & 7)) << 4), acc[g][4 * q],
                         acc[g][4 * q + 1], acc[g][4 * q + 2], acc[g][4 * q + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int x = tn * BN + col0 + g * 32, y = tm * kTcBM + quarter * 32;
            if (adds)
              tma_reduce_add_2d(&tmC, stage_addr, x, y);
            else
              tma_store_2d(&tmC, stage_addr, x, y);
            bulk_commit();
          }
        }
      } else if (i < p.M) {
#pragma unroll
        for (int g = 0; g < kGroups; ++g)
          store_group<BN, LINEAR>(p, i, tn * BN + col0 + g * 32, acc[g]);
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

template <int BN, int STAGES, int SK, bool TRANS, bool LINEAR>
cudaError_t tc_ts_launch(const CUtensorMap* l, const CUtensorMap* s, const CUtensorMap* c,
                         const TcParams* p, int grid, bool pdl, cudaStream_t stream) {
  using L = TsLayout<BN, STAGES, SK>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTsThreads);
  cfg.dynamicSmemBytes = tc_smem_request(L::kDynSmem, L::kTmemCols);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, tc_ts_kernel<BN, STAGES, SK, TRANS, LINEAR>, *l, *s, *c, *p);
}

template <int BN, int STAGES, int SK, bool TRANS, bool LINEAR>
TcKernel tc_ts_entry() {
  using L = TsLayout<BN, STAGES, SK>;
  TcKernel k;
  k.launch = &tc_ts_launch<BN, STAGES, SK, TRANS, LINEAR>;
  k.func = reinterpret_cast<const void*>(&tc_ts_kernel<BN, STAGES, SK, TRANS, LINEAR>);
  k.threads = kTsThreads;
  k.smem = tc_smem_request(L::kDynSmem, L::kTmemCols);
  k.tmem_cols = L::kTmemCols;
  k.tile_n = BN;
  k.stages = STAGES;
  k.slice = SK;
  return k;
}

}  // namespace lbg
