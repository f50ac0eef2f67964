// tc_ts256.cuh -- the 8-bit tensor-core GEMM with in-kernel int8 -> fp16
// conversion of one operand (fed to the MMA from tensor memory), 128 x 256
// output tiles.
//
// Method: the tiling of "Leveraging Large-Scale Data for Efficient Low-Bit
// CUTLASS GEMM Optimization via Neural Networks" (press summary page), section
// 1: uniform output tiles, a K loop per tile, a multi-stage load pipeline.
// Exactness as in tc_gemm.cuh: int8 values are fp16 values, products are
// exact, and the K loop is cut into chunks whose fp32 sums cannot pass 2^24;
// each chunk's tile is added into int32 registers.
//
// GB300 design.  An MMA of N = 256 per SM keeps the tensor pipe busy across
// the issuing thread's barrier waits (measured on GB300: M = 128, N = 128 MMAs
// lose about 40 % of the pipe to a wait per 64-element K slice, N = 256 MMAs
// lose nothing).  With 256 accumulator columns, tensor memory (512 columns)
// holds one accumulator and 256 columns of the converted operand, so the
// accumulator is single-buffered: the MMA pauses while a chunk's tile is read
// out (measured alone: 82 % of the pipe with a 16-slice chunk).
//
// K is consumed in 64-element slices (one 128-byte fp16 row segment, 4 MMAs of
// K = 16) in groups of GS slices: a barrier wait costs the waiting warp a few
// hundred cycles on GB300, so the conversion side synchronises once per group.
// The L operand (MMA A, 128 rows per tile) stays int8 in global memory; TMA
// brings a group's 64 * GS K bytes of its 128 rows (boxes of 128 bytes x 128
// rows, 128-byte swizzle) into a staging ring.  The S operand (MMA B, 256 rows
// per tile) is the caller's other operand re-encoded to fp16 ahead; TMA brings
// its slices (32 KB, 128-byte swizzle) into a ring of its own.  Tensor memory:
// the accumulator (columns 0..255) and 256 / (32 GS) A slots of 32 GS columns,
// one group each.
//
// Roles (352 threads):
//   warp 0 lane 0    TMA of the int8 staging ring (one stage per group)
//   warp 1           tensor-memory allocation; lane 0 issues MMAs and commits
//   warps 2..9       workers, two per tensor-memory quarter (quarter = warp % 4,
//                    h = (warp - 2) / 4): convert slices [h GS/2, (h+1) GS/2) of
//                    each group for their quarter's 32 rows into the group's A
//                    slot (tcgen05.st), and read out columns [128h, 128h+128)
//                    of the accumulator at the end of each chunk
//   warp 10 lane 0   TMA of the S ring (one slice per stage)
// A worker first converts every group of the chunk c it must read out next;
// then it reads c out as soon as c's MMAs are done, converting ahead (up to R
// groups, the A slots) while it waits.  No wait can close a cycle: group q
// needs the MMA of group q - R, which needs only conversions and read-outs
// ordered before q.
//
// Output: TRANS = false: C[i][j] for L-row i and S-row j (TMA bulk stores of
// swizzled 32 x 32 blocks, or plain stores); TRANS = true: C[j][i] with
// coalesced 128-byte stores (atomics under split K); LINEAR: bf16 Y with the
// row and column scales.  Every wait is bounded; on a time-out the CTA winds
// down (own copies in flight, own MMAs) before tensor memory is freed.
#pragma once
#include "tc_gemm.cuh"

namespace lbg {

constexpr int kT2Workers = 8;
constexpr int kT2Threads = 32 * (3 + kT2Workers);  // 352
constexpr int kT2BN = 256;

template <int STAGES, int GS, int SG>
struct T2Layout {
  static constexpr int kSlots = kT2BN / (32 * GS);     // A slots in tensor memory
  static constexpr int kSBytes = kT2BN * 128;          // one fp16 K slice of 256 rows
  static constexpr int kEpiOffset = kSBytes * STAGES;
  static constexpr int kEpiBytes = kT2Workers * 32 * 128;
  static constexpr int kStgOffset = kEpiOffset + kEpiBytes;
  static constexpr int kBoxBytes = kTcBM * 128;        // 128 rows x 128 int8 (two slices)
  static constexpr int kStgStageBytes = kBoxBytes * (GS / 2);
  static constexpr int kBarOffset = kStgOffset + kStgStageBytes * SG;
  // barriers: sfull[S], sempty[S], conv[A], aempty[A], stgf[SG], stge[SG], accf, acce, done
  static constexpr int kNumBars = 2 * STAGES + 2 * kSlots + 2 * SG + 3;
  static constexpr int kTmemSlotOffset = kBarOffset + 8 * kNumBars;
  static constexpr int kAbortOffset = kTmemSlotOffset + 4;
  static constexpr int kDynSmem = kAbortOffset + 4 + 1024;
  static constexpr int kACol0 = kT2BN;
  static constexpr int kTmemCols = 512;
  static_assert(GS == 2 || GS == 4, "groups of 2 or 4 slices");
  static_assert(kDynSmem <= 232448, "shared memory per CTA");
};

// Groups of a unit with slices [kbb, kbe): GS slices each, starting at kbb
// (the last may be short); chunks of p.chunk_kb slices (a multiple of GS)
// start at kbb too.
template <int GS>
__device__ __forceinline__ int t2_groups(int kbb, int kbe) {
  return (kbe - kbb + GS - 1) / GS;
}

// All lanes of the warp wait; the result is the same in every lane.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort,
                                               int* status) {
  const bool ok = mbar_wait(bar, parity, abort, status);
  return __all_sync(0xffffffffu, ok);
}

template <int STAGES, int GS, int SG, bool TRANS, bool LINEAR>
__global__ void __launch_bounds__(kT2Threads, 1)
    tc_ts256_kernel(const __grid_constant__ CUtensorMap tmL, const __grid_constant__ CUtensorMap tmS,
                    const __grid_constant__ CUtensorMap tmC, const TcParams p) {
  using L = T2Layout<STAGES, GS, SG>;
  constexpr int R = L::kSlots;
  constexpr int G = SG;
  constexpr uint32_t kIdesc = instr_desc(kTcBM, kT2BN);
  const int chunk_groups = p.chunk_kb / GS;  // the host makes chunk_kb a multiple of GS

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar0 = sbase + L::kBarOffset;
  auto sfull_bar = [&](int s) { return bar0 + 8u * s; };
  auto sempty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto conv_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto aempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + R + a); };
  auto stgf_bar = [&](int g) { return bar0 + 8u * (2 * STAGES + 2 * R + g); };
  auto stge_bar = [&](int g) { return bar0 + 8u * (2 * STAGES + 2 * R + G + g); };
  const uint32_t accf_bar = bar0 + 8u * (2 * STAGES + 2 * R + 2 * G);
  const uint32_t acce_bar = accf_bar + 8;
  const uint32_t done_bar = accf_bar + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlotOffset);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbortOffset);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(sfull_bar(s), 1);
      mbar_init(sempty_bar(s), 1);
    }
    for (int a = 0; a < R; ++a) {
      mbar_init(conv_bar(a), kT2Workers);
      mbar_init(aempty_bar(a), 1);
    }
    for (int g = 0; g < G; ++g) {
      mbar_init(stgf_bar(g), 1);
      mbar_init(stge_bar(g), kT2Workers);
    }
    mbar_init(accf_bar, 1);
    mbar_init(acce_bar, kT2Workers);
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

  if (warp == 0 || warp == 2 + kT2Workers) {
    // ---------------- TMA producers: int8 groups (warp 0), S slices (warp 10) --------
    const bool is_s = warp != 0;
    if (lane == 0) {
      const CUtensorMap* map = is_s ? &tmS : &tmL;
      tma_prefetch_desc(map);
      // The S operand comes from the re-encoding grid this kernel may have
      // been launched as a dependent of; the int8 operand is the caller's,
      // ordered before that grid by the stream.
      if (is_s) asm volatile("griddepcontrol.wait;" ::: "memory");
      const int depth = is_s ? STAGES : G;
      const uint32_t bytes = is_s ? L::kSBytes : L::kStgStageBytes;
      const int step = is_s ? 1 : GS;
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int w = blockIdx.x; ok && w < p.num_units; w += gridDim.x) {
        int t, kbb, kbe, tm, tn;
        unit_range(w, p, t, kbb, kbe);
        tile_coords(t, p, tm, tn);
        for (int kb = kbb; kb < kbe; kb += step) {
          const uint32_t eb = is_s ? sempty_bar(stage) : stge_bar(stage);
          const uint32_t fb = is_s ? sfull_bar(stage) : stgf_bar(stage);
          if (!mbar_wait(eb, phase ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(fb, bytes);
          if (is_s) {
            tma_load_2d(sbase + stage * L::kSBytes, map, fb, kb * 64, tn * kT2BN);
          } else {
#pragma unroll
            for (int b = 0; b < GS / 2; ++b)
              tma_load_2d(sbase + L::kStgOffset + stage * L::kStgStageBytes + b * L::kBoxBytes,
                          map, fb, (kb + 2 * b) * 64, tm * kTcBM);
          }
          ++issued;
          if (++stage == depth) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Wind-down: wait for this thread's copies still in flight.
        const int64_t back = issued < depth ? issued : depth;
        for (int64_t i = 0; i < back; ++i) {
          if (--stage < 0) {
            stage = depth - 1;
            phase ^= 1u;
          }
          mbar_wait_drain(is_s ? sfull_bar(stage) : stgf_bar(stage), phase);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      int s = 0, a = 0;
      uint32_t sph = 0, aph = 0;
      uint32_t chunk = 0;  // chunks issued so far (all units)
      bool ok = true;
      for (int w = blockIdx.x; ok && w < p.num_units; w += gridDim.x) {
        int t, kbb, kbe;
        unit_range(w, p, t, kbb, kbe);
        for (int kb0 = kbb; ok && kb0 < kbe; kb0 += p.chunk_kb, ++chunk) {
          // the previous chunk's tile has been read out of the accumulator
          if (chunk > 0 && !mbar_wait(acce_bar, (chunk - 1) & 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int kb1 = min(kb0 + p.chunk_kb, kbe);
          for (int kp = kb0; kp < kb1; kp += GS) {
            if (!mbar_wait(conv_bar(a), aph, abort_flag, p.status)) {
              ok = false;
              break;
            }
            for (int h = 0; h < GS && kp + h < kb1; ++h) {
              if (!mbar_wait(sfull_bar(s), sph, abort_flag, p.status)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t bdesc = smem_desc_sw128(sbase + s * L::kSBytes);
              const uint32_t a_tmem = tmem_base + L::kACol0 + a * (32 * GS) + h * 32;
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_f16_ts(tmem_base, a_tmem + 8 * k, bdesc + 2 * k, kIdesc,
                           (kp + h > kb0 || k > 0) ? 1u : 0u);
              mma_commit(sempty_bar(s));
              if (++s == STAGES) {
                s = 0;
                sph ^= 1u;
              }
            }
            if (!ok) break;
            mma_commit(aempty_bar(a));
            if (++a == R) {
              a = 0;
              aph ^= 1u;
            }
          }
          if (ok) mma_commit(accf_bar);
        }
      }
      mma_commit(done_bar);  // arrives once every MMA issued above has completed
    }
  } else {
    // ---------------- workers: conversion and read-out ----------------
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const uint32_t stage_addr = sbase + L::kEpiOffset + (warp - 2) * (32 * 128);

    // conversion cursor: unit cw, group cq of cnq; global group index cj
    int cw = (int)blockIdx.x, cq = 0, cnq = 0;
    int64_t cj = 0;
    bool c_have = false;
    for (; cw < p.num_units; cw += gridDim.x) {
      int t, kbb, kbe;
      unit_range(cw, p, t, kbb, kbe);
      cnq = t2_groups<GS>(kbb, kbe);
      if (cnq > 0) {
        c_have = true;
        break;
      }
    }
    // read-out cursor: unit dw, its groups dnq, next chunk's first group dq;
    // global index of that chunk's first group dfirst
    int dw = (int)blockIdx.x, dnq = 0, dq = 0;
    int64_t dfirst = 0;
    bool d_have = false;
    for (; dw < p.num_units; dw += gridDim.x) {
      int t, kbb, kbe;
      unit_range(dw, p, t, kbb, kbe);
      dnq = t2_groups<GS>(kbb, kbe);
      if (dnq > 0) {
        d_have = true;
        break;
      }
    }
    int a = 0, g = 0;
    uint32_t aph = 0, gph = 0;
    uint32_t chunk = 0;
    int32_t acc[4][32];
    bool ok = true;
    while (ok && (c_have || d_have)) {
      const int64_t dlast = d_have ? dfirst + min(chunk_groups, dnq - dq) - 1 : 0;
      bool convert;
      if (!c_have) {
        convert = false;
      } else if (!d_have || cj <= dlast) {
        convert = true;  // the pending chunk still needs this group
      } else if (cj > dlast + R) {
        convert = false;  // every slot is ahead: the read-out comes first
      } else {
        // The pending chunk is fully converted: read it out as soon as its
        // MMAs are done, else convert ahead while a slot and its data are
        // ready.  Neither wait here can block the other side for good.
        int choice = -1;
        if (lane == 0) {
          const uint64_t start = global_timer_ns();
          for (uint32_t i = 0;; ++i) {
            if (mbar_test(accf_bar, chunk & 1u)) {
              choice = 0;
              break;
            }
            if (mbar_test(aempty_bar(a), aph ^ 1u) && mbar_test(stgf_bar(g), gph)) {
              choice = 1;
              break;
            }
            if ((i & 63u) == 63u) {
              if (*abort_flag) break;
              if (global_timer_ns() - start > kWaitLimitNs) {
                *abort_flag = 1;
                atomicOr(p.status, kStatusTimeout);
                break;
              }
            }
          }
        }
        choice = __shfl_sync(0xffffffffu, choice, 0);
        if (choice < 0) {
          ok = false;
          break;
        }
        convert = choice == 1;
      }
      if (convert) {
        // ---- convert this worker's slices of group cj into A slot a ----
        if (!mbar_wait_warp(aempty_bar(a), aph ^ 1u, abort_flag, p.status) ||
            !mbar_wait_warp(stgf_bar(g), gph, abort_flag, p.status)) {
          ok = false;
          break;
        }
        const uint8_t* stg = smem + L::kStgOffset + g * L::kStgStageBytes + row * 128;
#pragma unroll
        for (int jj = 0; jj < GS / 2; ++jj) {
          const int j = half * (GS / 2) + jj;  // slice of the group
          // 128-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ (r % 8)
          const uint8_t* src = stg + (j >> 1) * L::kBoxBytes;
          uint32_t words[32];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int c16 = 4 * (j & 1) + q;
            const int4 v = *reinterpret_cast<const int4*>(src + ((c16 ^ (row & 7)) << 4));
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
          tmem_st32(tmem_base + lane_addr + L::kACol0 + a * (32 * GS) + j * 32, words);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(conv_bar(a));
          mbar_arrive(stge_bar(g));
        }
        if (++a == R) {
          a = 0;
          aph ^= 1u;
        }
        if (++g == G) {
          g = 0;
          gph ^= 1u;
        }
        ++cj;
        if (++cq >= cnq) {
          c_have = false;
          cq = 0;
          for (cw += gridDim.x; cw < p.num_units; cw += gridDim.x) {
            int t, kbb, kbe;
            unit_range(cw, p, t, kbb, kbe);
            cnq = t2_groups<GS>(kbb, kbe);
            if (cnq > 0) {
              c_have = true;
              break;
            }
          }
        }
      } else {
        // ---- read out the chunk starting at group dq of unit dw ----
        if (!mbar_wait_warp(accf_bar, chunk & 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const bool first = dq == 0;
#pragma unroll
        for (int gq = 0; gq < 4; ++gq) {
          uint32_t v[32];
          tmem_ld32(tmem_base + lane_addr + half * 128 + gq * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int32_t x = __float2int_rn(__uint_as_float(v[j]));
            acc[gq][j] = first ? x : acc[gq][j] + x;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce_bar);
        ++chunk;
        const int n_in_chunk = min(chunk_groups, dnq - dq);
        dfirst += n_in_chunk;
        dq += n_in_chunk;
        if (dq >= dnq) {
          // ---- the unit's tile is complete: store it ----
          // (C may have been cleared by the grid this kernel was launched as
          // a dependent of: that grid is complete before the first store)
          asm volatile("griddepcontrol.wait;" ::: "memory");
          int t, kb_a, kb_b, tm, tn;
          unit_range(dw, p, t, kb_a, kb_b);
          tile_coords(t, p, tm, tn);
          const int i = tm * kTcBM + row;  // L row
          const int j0 = tn * kT2BN + half * 128;
          if (TRANS) {
            if (i < p.M) {
#pragma unroll
              for (int gq = 0; gq < 4; ++gq) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                  const int jj = j0 + gq * 32 + j;
                  if (jj < p.N) {
                    const int64_t off = (int64_t)jj * p.M + i;
                    if (LINEAR)
                      p.Y[off] = __float2bfloat16_rn((float)acc[gq][j] * p.sx[jj] * p.sw[i]);
                    else if (p.splits > 1)
                      atomicAdd(p.C + off, acc[gq][j]);
                    else
                      p.C[off] = acc[gq][j];
                  }
                }
              }
            }
          } else if (!LINEAR && p.vec_ok) {
#pragma unroll
            for (int gq = 0; gq < 4; ++gq) {
              if (lane == 0) bulk_wait_read_all();
              __syncwarp();
#pragma unroll
              for (int q = 0; q < 8; ++q)
                st_shared_v4(stage_addr + lane * 128 + ((q ^ (lane & 7)) << 4), acc[gq][4 * q],
                             acc[gq][4 * q + 1], acc[gq][4 * q + 2], acc[gq][4 * q + 3]);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                const int x = j0 + gq * 32, y = tm * kTcBM + quarter * 32;
                if (p.splits > 1)
                  tma_reduce_add_2d(&tmC, stage_addr, x, y);
                else
                  tma_store_2d(&tmC, stage_addr, x, y);
                bulk_commit();
              }
            }
          } else if (i < p.M) {
#pragma unroll
            for (int gq = 0; gq < 4; ++gq) store_group<kT2BN, LINEAR>(p, i, j0 + gq * 32, acc[gq]);
          }
          d_have = false;
          dq = 0;
          for (dw += gridDim.x; dw < p.num_units; dw += gridDim.x) {
            int kbb, kbe;
            unit_range(dw, p, t, kbb, kbe);
            dnq = t2_groups<GS>(kbb, kbe);
            if (dnq > 0) {
              d_have = true;
              break;
            }
          }
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

template <int STAGES, int GS, int SG, bool TRANS, bool LINEAR>
cudaError_t tc_ts256_launch(const CUtensorMap* l, const CUtensorMap* s, const CUtensorMap* c,
                            const TcParams* p, int grid, bool pdl, cudaStream_t stream) {
  using L = T2Layout<STAGES, GS, SG>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kT2Threads);
  cfg.dynamicSmemBytes = tc_smem_request(L::kDynSmem, L::kTmemCols);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, tc_ts256_kernel<STAGES, GS, SG, TRANS, LINEAR>, *l, *s, *c, *p);
}

template <int STAGES, int GS, int SG, bool TRANS, bool LINEAR>
TcKernel tc_ts256_entry() {
  using L = T2Layout<STAGES, GS, SG>;
  TcKernel k;
  k.launch = &tc_ts256_launch<STAGES, GS, SG, TRANS, LINEAR>;
  k.func = reinterpret_cast<const void*>(&tc_ts256_kernel<STAGES, GS, SG, TRANS, LINEAR>);
  k.threads = kT2Threads;
  k.smem = tc_smem_request(L::kDynSmem, L::kTmemCols);
  k.tmem_cols = L::kTmemCols;
  k.tile_n = kT2BN;
  k.stages = STAGES;
  return k;
}

}  // namespace lbg
