// tc_pair.cuh -- the CTA-pair tensor-core kernel of the large tile class:
// 256 x 256 output tiles, each computed by the two CTAs of a cluster with
// tcgen05 MMAs of cta_group::2.
//
// Method: the tiling of "Leveraging Large-Scale Data for Efficient Low-Bit
// CUTLASS GEMM Optimization via Neural Networks" (press summary page), section
// 1: uniform output tiles, a K loop per tile, a multi-stage load pipeline; the
// stage count is the template parameter STAGES.  Operands arrive re-encoded
// (int8 -> fp16, int4 and +-1 -> e4m3) and K is cut into exact fp32 chunks,
// exactly as in the single-CTA kernel (tc_gemm.cuh).
//
// GB300 design.  A cta_group::2 MMA of M = 256 reads A's rows 0..127 and B's
// rows 0..127 from the even CTA's shared memory and A's rows 128..255 and B's
// rows 128..255 from the odd CTA's, at the same offsets, and writes D's rows
// 0..127 (all 256 columns) to the even CTA's TMEM and rows 128..255 to the odd
// CTA's.  Per 128-byte K slice each SM stages 32 KB for its 128 x 256 outputs,
// against 48 KB for the single-CTA 128 x 256 tile: six stages fit, and each
// SM reads a third less shared memory per MMA.
//
// Roles (320 threads in each CTA of the pair):
//   warp 0 lane 0  producer: TMA of this CTA's half of A and of B.  The bytes
//                  of both CTAs are counted on the even CTA's full barrier
//                  (.cta_group::2 lets a load signal the peer's barrier); the
//                  even producer arms it for both halves.  Each producer waits
//                  on its own empty barrier, on which the MMA commits arrive by
//                  multicast.
//   warp 1         TMEM allocation for the pair (cta_group::2, in both CTAs);
//                  in the even CTA, lane 0 issues the MMAs and the commits.
//   warps 2..9     epilogue of this CTA's 128 rows, as in the single-CTA
//                  kernel; the "accumulator read" arrivals of both CTAs go to
//                  the even CTA's barrier (16 arrivals per phase).
// Every wait is bounded.  When a wait runs out, the odd producer reports the
// number of stage fills it issued to the even CTA; after a cluster barrier the
// even producer waits for every fill that may still be in flight (arming, or
// completing, the half that one side never issued) before either CTA leaves.
#pragma once
#include "tc_gemm.cuh"

namespace lbg {

constexpr int kPairTile = 256;  // output rows and columns of one pair tile

template <int STAGES>
struct PairLayout {
  static constexpr int kABytes = 128 * 128;  // this CTA's 128 rows of A, one K slice
  static constexpr int kBBytes = 128 * 128;  // this CTA's 128 rows of B
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kEpiOffset = kStageBytes * STAGES;
  // epilogue staging: per epilogue warp, one or two 32-row x 128-byte tiles
  // (two, where they fit: a warp then fills one while the other is stored)
  static constexpr int kEpiBufs =
      kEpiOffset + 2 * kTcEpiWarps * 32 * 128 + 8 * (2 * STAGES + 5) + 24 + 1024 <= 232448 ? 2
                                                                                          : 1;
  static constexpr int kEpiBytes = kEpiBufs * kTcEpiWarps * 32 * 128;
  // barriers: full[S], empty[S], acc_full[2], acc_empty[2], mma_done
  static constexpr int kNumBars = 2 * STAGES + 5;
  static constexpr int kBarOffset = kEpiOffset + kEpiBytes;
  static constexpr int kPeerIssuedOffset = kBarOffset + 8 * kNumBars;  // int64
  static constexpr int kTmemSlotOffset = kPeerIssuedOffset + 8;
  static constexpr int kAbortOffset = kTmemSlotOffset + 4;
  static constexpr int kUsedBytes = kAbortOffset + 4;
  static constexpr int kDynSmem = kUsedBytes + 1024;  // slack to align the ring to 1024
  static constexpr int kTmemCols = 512;              // two 256-column fp32 accumulators
  static_assert(kDynSmem <= 232448, "shared memory of one CTA");
  // the stage ring holds a whole C tile of this CTA (8 warps x 4 groups of
  // 32 x 128 bytes) from 4 stages on
  static constexpr bool kRingHoldsC = kEpiOffset >= kTcEpiWarps * 4 * 32 * 128;
};

// ---- cluster and cta_group::2 forms ------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// Address of the same shared-memory offset in CTA `cta` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, uint32_t cta) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(cta));
  return r;
}

// All threads of both CTAs; orders earlier shared-memory writes (local and
// remote) before everything after the barrier in either CTA.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void st_cluster_u64(uint32_t addr, uint64_t v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

__device__ __forceinline__ void mbar_complete_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.complete_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// mbar_wait with cluster-scope acquire (the phase is completed by arrivals
// from both CTAs).
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  volatile int* abort, int* status) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t start = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - start > kWaitLimitNs) {
        *abort = 1;
        atomicOr(status, kStatusTimeout);
        return false;
      }
    }
  }
}

// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier of this CTA or of its peer (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void mma_pair_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_pair_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the barrier at offset `bar` in both CTAs of the pair once every
// pair MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  const uint16_t both = 3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(both)
      : "memory");
}

// ---- the kernel ----------------------------------------------------------------------------

template <int STAGES, bool F8, bool LINEAR>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(320, 1)
    tc_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const TcParams p) {
  using L = PairLayout<STAGES>;
  constexpr int kBkElems = F8 ? 128 : 64;
  constexpr uint32_t kIdesc = instr_desc(kPairTile, kPairTile);
  constexpr int kGroups = kPairTile / 2 / 32;  // 32-column groups per epilogue thread

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
  volatile int64_t* peer_issued = reinterpret_cast<volatile int64_t*>(smem + L::kPeerIssuedOffset);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_rank();
  const bool even = rank == 0;
  const int cid = (int)cluster_index();
  const int ncl = (int)cluster_count();

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), 2 * kTcEpiWarps);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    *peer_issued = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(tmem_slot), L::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  int64_t prod_issued = 0;  // stage fills issued by this CTA's producer
  if (warp == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      asm volatile("griddepcontrol.wait;" ::: "memory");
      const int row_off = (int)rank * 128;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int w = cid; ok && w < p.num_units; w += ncl) {
        int t, kbb, kbe, tm, tn;
        unit_range(w, p, t, kbb, kbe);
        tile_coords(t, p, tm, tn);
        for (int kb = kbb; kb < kbe; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const uint32_t sa = sbase + stage * L::kStageBytes;
          const uint32_t fb = cluster_map(full_bar(stage), 0);
          if (even) mbar_arrive_expect_tx(full_bar(stage), 2 * L::kStageBytes);
          tma_load_2d_pair(sa, &tmA, fb, kb * kBkElems, tm * kPairTile + row_off);
          tma_load_2d_pair(sa + L::kABytes, &tmB, fb, kb * kBkElems, tn * kPairTile + row_off);
          ++prod_issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!even) st_cluster_u64(cluster_map(smem_addr((const void*)peer_issued), 0),
                                (uint64_t)prod_issued);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (even CTA) ----------------
    if (even && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t u = 0;
      bool ok = true;
      for (int w = cid; ok && w < p.num_units; w += ncl) {
        int t, kbb, kbe;
        unit_range(w, p, t, kbb, kbe);
        const int num_chunks = (kbe - kbb + p.chunk_kb - 1) / p.chunk_kb;
        for (int c = 0; ok && c < num_chunks; ++c, ++u) {
          const int buf = u & 1;
          if (!mbar_wait_cluster(acce_bar(buf), ((u >> 1) & 1u) ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * kPairTile;
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
              const uint32_t accumulate = (kb > kb0 || k > 0) ? 1u : 0u;
              if (F8)
                mma_pair_f8(d_tmem, adesc + 2 * k, bdesc + 2 * k, kIdesc, accumulate);
              else
                mma_pair_f16(d_tmem, adesc + 2 * k, bdesc + 2 * k, kIdesc, accumulate);
            }
            mma_commit_pair(empty_bar(stage));
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (ok) mma_commit_pair(accf_bar(buf));
        }
      }
      mma_commit_pair(done_bar);  // both CTAs: every MMA issued above has completed
    }
  } else {
    // ---------------- epilogue (both CTAs) ----------------
    // C may have been cleared by the grid this kernel was launched as a
    // dependent of: wait for that grid before the first store into C.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int e = warp - 2;
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int row = quarter * 32 + lane;
    const int col0 = (e >> 2) * (kPairTile / 2);
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const uint32_t stage_addr = sbase + L::kEpiOffset + e * (L::kEpiBufs * 32 * 128);
    const int row_off = (int)rank * 128;
    uint32_t u = 0;
    uint32_t stores = 0;  // TMA stores issued by this warp (staging buffer = stores % kEpiBufs)
    int32_t acc[kGroups][32];
    bool ok = true;
    for (int w = cid; ok && w < p.num_units; w += ncl) {
      int t, kbb, kbe, tm, tn;
      const bool adds = unit_range(w, p, t, kbb, kbe);
      tile_coords(t, p, tm, tn);
      const int num_chunks = (kbe - kbb + p.chunk_kb - 1) / p.chunk_kb;
      // The cluster's last unit: once its final accumulator is complete no
      // copy or MMA touches either CTA's stage ring any more, so each warp
      // stages all its groups of C there (where the ring is large enough) and
      // issues their stores back to back.
      const bool last_unit = L::kRingHoldsC && w + ncl >= p.num_units;
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
        if (c == 0) {
          // the first chunk lands in acc itself: all loads, then one wait
#pragma unroll
          for (int g = 0; g < kGroups; ++g)
            tmem_ld32(tmem_base + lane_addr + buf * kPairTile + col0 + g * 32,
                      reinterpret_cast<uint32_t(&)[32]>(acc[g]));
          tmem_ld_wait();
#pragma unroll
          for (int g = 0; g < kGroups; ++g)
#pragma unroll
            for (int j = 0; j < 32; ++j)
              acc[g][j] = __float2int_rn(__uint_as_float((uint32_t)acc[g][j]));
        } else {
#pragma unroll
          for (int g = 0; g < kGroups; ++g) {
            uint32_t v[32];
            tmem_ld32(tmem_base + lane_addr + buf * kPairTile + col0 + g * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[g][j] += __float2int_rn(__uint_as_float(v[j]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (even)
            mbar_arrive(acce_bar(buf));
          else
            mbar_arrive_cluster(cluster_map(acce_bar(buf), 0));
        }
      }
      if (!ok) break;
      const int m0 = tm * kPairTile + row_off;
      if (!LINEAR && p.vec_ok) {
#pragma unroll
        for (int g = 0; g < kGroups; ++g, ++stores) {
          uint32_t buf;
          if (last_unit) {
            buf = sbase + (e * kGroups + g) * (32 * 128);
          } else {
            // the store that last used this buffer has read it
            if (lane == 0) bulk_wait_read<L::kEpiBufs - 1>();
            __syncwarp();
            buf = stage_addr + (stores % L::kEpiBufs) * (32 * 128);
          }
#pragma unroll
          for (int q = 0; q < 8; ++q)
            st_shared_v4(buf + lane * 128 + ((q ^ (lane & 7)) << 4), acc[g][4 * q],
                         acc[g][4 * q + 1], acc[g][4 * q + 2], acc[g][4 * q + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int x = tn * kPairTile + col0 + g * 32, y = m0 + quarter * 32;
            if (adds)
              tma_reduce_add_2d(&tmC, buf, x, y);
            else
              tma_store_2d(&tmC, buf, x, y);
            bulk_commit();
          }
        }
      } else {
        const int m = m0 + row;
        if (m < p.M) {
#pragma unroll
          for (int g = 0; g < kGroups; ++g)
            store_group<kPairTile, LINEAR>(p, m, tn * kPairTile + col0 + g * 32, acc[g]);
        }
      }
    }
    if (lane == 0) bulk_wait_all();
  }

  __syncthreads();
  cluster_sync_all();  // the odd producer's fill count has reached the even CTA
  if (even && warp == 0 && lane == 0) {
    // Wait for every stage fill that may still be in flight.  Fill j + STAGES
    // is only issued once fill j was consumed, so only the last STAGES fills
    // of the side that issued more can be pending; a fill one side never
    // issued gets its half armed (odd side issued it) or completed (even side
    // issued it) here, so that its phase completes once the issued half lands.
    const int64_t ip = *peer_issued;
    const int64_t hi = prod_issued > ip ? prod_issued : ip;
    for (int64_t j = hi - STAGES > 0 ? hi - STAGES : 0; j < hi; ++j) {
      const int s = (int)(j % STAGES);
      const uint32_t par = (uint32_t)((j / STAGES) & 1);
      if (j >= prod_issued)
        mbar_arrive_expect_tx(full_bar(s), L::kStageBytes);
      else if (j >= ip)
        mbar_complete_tx(full_bar(s), L::kStageBytes);
      mbar_wait_drain(full_bar(s), par);
    }
  }
  if (warp == 1 && lane == 0) mbar_wait_drain(done_bar, 0);
  __syncwarp();
  tc_fence_before();
  cluster_sync_all();  // no copy, MMA or arrival targets either CTA any more
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, L::kTmemCols);
  }
}

template <int STAGES, bool F8, bool LINEAR>
cudaError_t tc_pair_launch(const CUtensorMap* a, const CUtensorMap* b, const CUtensorMap* c,
                           const TcParams* p, int grid, bool pdl, cudaStream_t stream) {
  using L = PairLayout<STAGES>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);  // a multiple of 2 (the cluster size is fixed in the kernel)
  cfg.blockDim = dim3(320);
  cfg.dynamicSmemBytes = L::kDynSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, tc_pair_kernel<STAGES, F8, LINEAR>, *a, *b, *c, *p);
}

}  // namespace lbg
