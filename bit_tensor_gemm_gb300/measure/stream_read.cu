// stream_read.cu -- how fast can this GPU read a buffer of a given size?
//
// A stand-alone measurement program (not part of the library): the floor
// that a kernel streaming its operand once from HBM can reach at the sizes
// the linear layer reads (45 MB of 11008 x 4096 int8 weights), next to larger
// reads.  Three read kernels -- 16-byte loads, grid-strided or one contiguous
// slice per CTA with several loads in flight per thread, and a contiguous
// slice per CTA streamed by cp.async.bulk into a shared-memory ring -- each
// timed with CUDA events (a) alone, after a 512 MB write that evicts L2, and
// (b) back to back over six rotating buffers; and an empty kernel between
// two events.  Every mbarrier wait is bounded.
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 \
//       -o stream_read bit_tensor_gemm_gb300/measure/stream_read.cu && ./stream_read
#include <cuda_runtime.h>
#include <cstdio>
#include <cstdint>
#include <vector>
#include <algorithm>

#define CK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { printf("CUDA %s at %d: %s\n", #x, __LINE__, cudaGetErrorString(e_)); return 1; } } while (0)

__device__ unsigned long long g_sink;
__device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }
__device__ int g_err;

template <int UNROLL>
__global__ void __launch_bounds__(512) read_plain(const int4* __restrict__ p, int64_t n16) {
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  uint32_t acc = 0;
  for (; i + (UNROLL - 1) * stride < n16; i += UNROLL * stride) {
    int4 v[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) v[u] = __ldcs(p + i + u * stride);
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < n16; i += stride) {
    int4 v = __ldcs(p + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  if (acc == 0x12345678u) atomicAdd(&g_sink, 1ull);
}

// contiguous slice per CTA: thread-block-local chunked loads (each warp owns
// consecutive 16B lanes of a chunk), UNROLL chunks in flight
template <int UNROLL>
__global__ void __launch_bounds__(512) read_slice(const int4* __restrict__ p, int64_t n16) {
  const int64_t per = (n16 + gridDim.x - 1) / gridDim.x;
  const int64_t b0 = per * blockIdx.x, b1 = min(n16, b0 + per);
  uint32_t acc = 0;
  int64_t i = b0 + threadIdx.x;
  for (; i + (UNROLL - 1) * 512 < b1; i += UNROLL * 512) {
    int4 v[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) v[u] = __ldcs(p + i + u * 512);
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < b1; i += 512) {
    int4 v = __ldcs(p + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  if (acc == 0x12345678u) atomicAdd(&g_sink, 1ull);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* b, int n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(n));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t phase) {
  uint32_t ok;
  asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
               : "=r"(ok) : "r"(smem_u32(b)), "r"(phase) : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t phase) {
  for (int it = 0; it < (1 << 22); ++it)
    if (mbar_try(b, phase)) return true;
  atomicExch(&g_err, 1);
  return false;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// (b) TMA bulk ring: CHUNK bytes per stage, S stages
template <int CHUNK, int S>
__global__ void __launch_bounds__(256) read_bulk(const uint8_t* __restrict__ p, int64_t nbytes) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ uint64_t full[S], empty[S];
  const int64_t per = ((nbytes + gridDim.x - 1) / gridDim.x + 15) / 16 * 16;
  const int64_t b0 = per * blockIdx.x, b1 = min(nbytes, b0 + per);
  const int64_t nchunks = b1 > b0 ? (b1 - b0 + CHUNK - 1) / CHUNK : 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], blockDim.x / 32); }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int64_t c = 0; c < nchunks && c < S; ++c) {
      const uint32_t bytes = (uint32_t)imin64((int64_t)CHUNK, b1 - (b0 + c * CHUNK));
      mbar_expect_tx(&full[c], bytes);
      bulk_g2s(sm + c * CHUNK, p + b0 + c * CHUNK, bytes, &full[c]);
    }
  }
  uint32_t acc = 0;
  int64_t issued = nchunks < S ? nchunks : S, consumed = 0;
  for (int64_t c = 0; c < nchunks; ++c) {
    const int s = (int)(c % S);
    const uint32_t ph = (uint32_t)((c / S) & 1);
    if (!mbar_wait(&full[s], ph)) break;
    consumed = c + 1;
    const uint32_t bytes = (uint32_t)imin64((int64_t)CHUNK, b1 - (b0 + c * CHUNK));
    const int4* q = reinterpret_cast<const int4*>(sm + s * CHUNK);
    for (uint32_t i = threadIdx.x; i < bytes / 16; i += blockDim.x) {
      int4 v = q[i];
      acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (threadIdx.x == 0 && c + S < nchunks) {
      if (!mbar_wait(&empty[s], ph)) break;
      const int64_t cn = c + S;
      const uint32_t nb = (uint32_t)imin64((int64_t)CHUNK, b1 - (b0 + cn * CHUNK));
      mbar_expect_tx(&full[s], nb);
      bulk_g2s(sm + s * CHUNK, p + b0 + cn * CHUNK, nb, &full[s]);
      issued = cn + 1;
    }
  }
  // after a failed wait: let this CTA's copies in flight land before exiting
  if (threadIdx.x == 0)
    for (int64_t c = consumed; c < issued; ++c) mbar_wait(&full[c % S], (uint32_t)((c / S) & 1));
  __syncthreads();
  if (acc == 0x12345678u) atomicAdd(&g_sink, 1ull);
}

int main() {
  int dev = 0, sms = 0;
  CK(cudaSetDevice(dev));
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int64_t sizes[] = {11008LL * 4096, 22LL << 20, 90LL << 20, 256LL << 20};
  const int NB = 6;
  const int64_t maxb = 256LL << 20;
  std::vector<uint8_t*> bufs(NB);
  for (auto& b : bufs) { CK(cudaMalloc(&b, maxb)); CK(cudaMemset(b, 1, maxb)); }
  uint8_t* flush; CK(cudaMalloc(&flush, 512LL << 20));
  cudaEvent_t e0, e1; CK(cudaEventCreate(&e0)); CK(cudaEventCreate(&e1));
  auto set_smem = [&](auto k, int bytes) { return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes); };
  CK(set_smem(read_bulk<16384, 12>, 16384 * 12));
  CK(set_smem(read_bulk<32768, 6>, 32768 * 6));
  CK(set_smem(read_bulk<8192, 24>, 8192 * 24));
  for (int64_t nbytes : sizes) {
    const int64_t n16 = nbytes / 16;
    struct V { const char* name; int grid; int kind; };
    std::vector<V> vs = {
      {"plain u4 g=152x4", sms * 4, 0}, {"plain u8 g=152x4", sms * 4, 1},
      {"plain u4 g=152x8 (256t)", sms * 8, 2},
      {"slice u4 g=152", sms, 3}, {"slice u8 g=152", sms, 4}, {"slice u8 g=304", 2 * sms, 4},
      {"bulk 16Kx12 g=152", sms, 5}, {"bulk 32Kx6 g=152", sms, 6}, {"bulk 8Kx24 g=152", sms, 7},
      {"bulk 16Kx12 g=148", 148, 5},
    };
    for (auto& v : vs) {
      auto launch = [&](uint8_t* b) {
        switch (v.kind) {
          case 0: read_plain<4><<<v.grid, 512>>>((const int4*)b, n16); break;
          case 1: read_plain<8><<<v.grid, 512>>>((const int4*)b, n16); break;
          case 2: read_plain<4><<<v.grid, 256>>>((const int4*)b, n16); break;
          case 3: read_slice<4><<<v.grid, 512>>>((const int4*)b, n16); break;
          case 4: read_slice<8><<<v.grid, 512>>>((const int4*)b, n16); break;
          case 5: read_bulk<16384, 12><<<v.grid, 256, 16384 * 12>>>(b, nbytes); break;
          case 6: read_bulk<32768, 6><<<v.grid, 256, 32768 * 6>>>(b, nbytes); break;
          case 7: read_bulk<8192, 24><<<v.grid, 256, 8192 * 24>>>(b, nbytes); break;
        }
      };
      // warm
      for (int i = 0; i < 3; ++i) launch(bufs[i % NB]);
      CK(cudaDeviceSynchronize());
      // single launches after flush
      std::vector<float> ts;
      for (int r = 0; r < 15; ++r) {
        CK(cudaMemsetAsync(flush, r, 512LL << 20));
        CK(cudaEventRecord(e0));
        launch(bufs[r % NB]);
        CK(cudaEventRecord(e1));
        CK(cudaEventSynchronize(e1));
        float ms; CK(cudaEventElapsedTime(&ms, e0, e1)); ts.push_back(ms);
      }
      std::sort(ts.begin(), ts.end());
      const float single = ts[ts.size() / 2];
      // back to back over rotating buffers
      CK(cudaMemsetAsync(flush, 7, 512LL << 20));
      const int R = 30;
      CK(cudaEventRecord(e0));
      for (int r = 0; r < R; ++r) launch(bufs[r % NB]);
      CK(cudaEventRecord(e1));
      CK(cudaEventSynchronize(e1));
      float msb; CK(cudaEventElapsedTime(&msb, e0, e1));
      CK(cudaGetLastError());
      int err = 0; CK(cudaMemcpyFromSymbol(&err, g_err, sizeof err));
      printf("%6.1f MB  %-26s single %7.2f us (%6.0f GB/s)   b2b %7.2f us (%6.0f GB/s)  err=%d\n",
             nbytes / 1e6, v.name, single * 1e3, nbytes / (single * 1e-3) / 1e9, msb / R * 1e3,
             nbytes / (msb / R * 1e-3) / 1e9, err);
    }
  }
  // an empty kernel, for the launch + event floor
  {
    std::vector<float> ts;
    for (int r = 0; r < 15; ++r) {
      CK(cudaEventRecord(e0));
      read_plain<4><<<1, 32>>>((const int4*)bufs[0], 0);
      CK(cudaEventRecord(e1));
      CK(cudaEventSynchronize(e1));
      float ms; CK(cudaEventElapsedTime(&ms, e0, e1)); ts.push_back(ms);
    }
    std::sort(ts.begin(), ts.end());
    printf("empty kernel between events: %.2f us\n", ts[7] * 1e3);
  }
  return 0;
}
