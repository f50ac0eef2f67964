// api.cu -- the C ABI (include/lbgemm.h): argument checks, variant
// selection, scratch management, TMA descriptors and kernel dispatch.
//
// Method: "Leveraging Large-Scale Data for Efficient Low-Bit CUTLASS GEMM
// Optimization via Neural Networks" (press summary page).  Intro and section 3:
// the selector maps (M, N, K, SM count) to one of the templates at run time;
// section 2: nine templates (three tile sizes x 2/3/4 stages), each dataset
// sample labelled with its fastest one; section 4: comparison with a default
// template.  Here the selector is a table filled by a timing sweep on the
// device itself, with a nearest-shape fallback.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <dlfcn.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "lbgemm.h"
#include "simt.h"
#include "tc_params.h"

namespace lbg {
int mlp_pick(int bits, int64_t M, int64_t N, int64_t K, int sm_count);
lbgemm_status mlp_load_file(const char* path);
}

// Device status word: kernels OR error bits into it (see lbgemm_device_status).
__device__ int g_lbgemm_status_word;

namespace {

using lbg::TcKernel;
using lbg::TcParams;

constexpr int kNumVariants = 9;
constexpr int kDefaultVariant = 7;  // large tile, middle stage level (5 stages)
constexpr int kMaxDevices = 64;
// M <= 4 runs on the dp4a kernel that streams B once (measured on GB300: at
// one to four rows it beats the warp-MMA kernel, which pays for 16-row MMAs)
constexpr int kSkinnyMaxM = 4;
constexpr int64_t kSkinnyKernelMaxM = 16;  // rows the dp4a streaming kernel takes at most
constexpr int kGroupM = 16;  // M-tiles per group of the tile order (L2 reuse)
// 1-bit problems below this many bit-MACs go to the popcount kernel, with
// its 64 x 64 tile and 3 stages: there the expansion pass and the second
// launch cost more than they save.  Measured on GB300 over the 729-shape
// grid: the popcount kernel takes most shapes up to 2^26 bit-MACs and the
// tensor cores most from 2^27, and 113 of its 177 wins are this variant
// (the 128 x 128 tile leaves most SMs idle on such problems).
constexpr double kPopcMaxWork = 134217728.0;
constexpr int kPopcRuleVariant = 1;
// 4-bit problems with K <= kSmallS4MaxK and at most kSmallS4MaxWork MACs go
// to the one-launch dp4a kernel on the packed nibbles (measured on GB300 over
// the grid: it wins most shapes with K <= 256 up to 2^26 MACs and none with
// K >= 512).
constexpr int64_t kSmallS4MaxK = 256;
constexpr double kSmallS4MaxWork = 67108864.0;
// 8-bit problems with K <= kSmallMaxK and at most kSmallMaxWork MACs go to the
// one-launch dp4a kernel.
constexpr int64_t kSmallMaxK = 512;
// 8-bit problems on the in-kernel-conversion kernel (see fused_route).
constexpr int64_t kFusedMaxSide = 512;
constexpr int64_t kFusedMinOther = 1024;
// The linear layer on that kernel splits K only when the split plan's waves
// of units cost at most this share of the unsplit grid's: the split runs a
// second grid to scale the int32 sums (measured on GB300, 64 tokens x 4096 x
// 4096, 32 tiles on 152 SMs, 26.9 -> 19.5 us; 64 x 4096 x 11008, 50.2 ->
// 25.6 us; 64 x 11008 x 4096, 86 tiles, split plan at 0.79 of the grid: no
// gain).
constexpr double kLinearSplitGain = 0.7;
// ... and takes stream-K instead where that schedule's cost model (each CTA's
// run of K slices plus one partial tile) is at most this share of the plan
// chosen so far: where the tiles make a fractional number of waves
// (measured on GB300: 192 tokens x 11008 x 4096, 172 tiles on 152 SMs, 53.2
// -> 46.1 us; 128 x 28672 x 8192, 92.2 -> 82.5 us; where it predicts less
// it measured no gain or a loss, e.g. 256 x 14336 x 4096, 53.2 -> 55.9 us).
constexpr double kLinearStreamGain = 0.85;
// Small side of the warp-level fp16 MMA kernel (hmma_skinny.cu): any problem
// up to kWarpMmaMaxSide rows; with more rows (up to kWarpMmaMaxSideSmall,
// each 32 rows re-reading the large operand) only small problems with
// 256 < K <= 2048, where the re-encoding route's two launches cost more
// (measured on GB300: 64-256 x 1024-4096 x 1024-2048, 3-7 us faster; with a
// side of 16384, or K of 4096, slower), and where the one-launch dp4a kernel
// does (K of 272-512: 8.8-10.9 us against 12.9 us; at K <= 256 the dp4a
// kernel is as fast or faster).
constexpr int64_t kWarpMmaMaxSide = 32;
// Small side of the streaming warp-MMA kernel (stream_mma.cu).
constexpr int64_t kStreamMaxSide = 16;
constexpr int64_t kWarpMmaMaxSideSmall = 256;
constexpr int64_t kWarpMmaMaxArea = int64_t(1) << 19;  // min(M, N) * max(M, N)
constexpr int64_t kWarpMmaMaxKSmall = 2048;
constexpr double kSmallMaxWork = 268435456.0;
constexpr size_t kFlushBytes = size_t(256) << 20;  // twice the 129 MB L2

thread_local std::string t_last_error;
std::atomic<int64_t> g_launches{0};
std::atomic<int> g_chunk_s8{1024};
std::atomic<int> g_chunk_s4{131072};
std::atomic<int> g_chunk_b1{1 << 23};
std::atomic<int> g_tail_split{1};  // 0 whole-problem splits only, 1 also a last partial wave, 2 forced
// K elements per slice of the 64/128-wide conversion kernels; 0: by tile and
// use (measured on GB300 over the grid shapes the dispatch gives these
// kernels: 256-element slices make the 64-wide kernel up to 10 % faster, e.g.
// 64 x 16384 x 16384 81.9 -> 74.3 us, and the 128-wide one up to 14 % slower
// for the GEMM, its tensor memory then holding only two slots; for the linear
// layer the 128-wide kernel is 8 % faster with them over 35 layers of 96-512
// tokens on 4096-28672 x 4096-11008 weights, up to 16 % at 384 tokens, and
// within 4 % of its 128-element time on each of them)
std::atomic<int> g_fused_slice{0};
// in-kernel-conversion schedule: 0 split K by the cost model, 1 stream-K
// wherever every CTA gets two slices
std::atomic<int> g_stream_k{0};

int fused_slice(int tile_n, bool linear) {
  const int s = g_fused_slice.load();
  return s ? s : (tile_n == 64 || linear) ? 256 : 128;
}

lbgemm_status fail(lbgemm_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

lbgemm_status cuda_fail(cudaError_t e, const char* what) {
  return fail(LBGEMM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ---- per-device state ------------------------------------------------------------

struct Scratch {
  void* ptr = nullptr;
  size_t bytes = 0;
  cudaEvent_t done = nullptr;  // recorded after the last use
  bool used = false;
};

struct DeviceState {
  bool ready = false;
  bool supported = false;
  int sm_count = 0;
  int* status = nullptr;
  Scratch ws;           // operand re-encoding scratch
  Scratch host_stage;   // device staging for lbgemm_run_host
  Scratch flush;        // buffer written between timed runs to evict L2
  Scratch quant;        // quantised activations of lbgemm_linear_quant
  std::map<const void*, int> occupancy;
  // lbgemm_run_host's copy streams (host-to-device, device-to-host) and events
  cudaStream_t copy_in = nullptr, copy_out = nullptr;
  std::vector<cudaEvent_t> host_events;
};

std::mutex g_mu;     // device state
std::mutex g_ws_mu;  // the internal re-encoding scratch
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

lbgemm_status device_state(DeviceState** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(LBGEMM_ERR_UNSUPPORTED, "device %d", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    d.supported = (major == 10 && minor == 3);
    if (d.supported) {
      e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_lbgemm_status_word);
      if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status word)");
      if (!g_encode) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
          return fail(LBGEMM_ERR_CUDA, "cuTensorMapEncodeTiled entry point not found");
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
      }
    }
    d.ready = true;
  }
  if (!d.supported)
    return fail(LBGEMM_ERR_UNSUPPORTED, "device %d is not an sm_103 GPU (this library is built "
                "for sm_103a only)", dev);
  *out = &d;
  return LBGEMM_OK;
}

// Whether `stream` is being captured into a CUDA graph.
bool capturing(cudaStream_t stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  return cudaStreamIsCapturing(stream, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive;
}

// Scratch for one call, in *ptr.  Normally the per-device buffer `s`, grown
// to at least `bytes` (synchronising the device when it must reallocate),
// this use ordered after the previous one on another stream by its event.
// While `stream` is being captured into a CUDA graph, a stream-ordered
// allocation instead (an allocation node of the graph, freed again by
// scratch_release within it): the graph then holds no address of the shared
// buffer, which a later call may reallocate, and no dependency on work
// outside the capture.
lbgemm_status scratch_acquire(Scratch& s, size_t bytes, cudaStream_t stream, void** ptr) {
  *ptr = nullptr;
  if (capturing(stream)) {
    cudaError_t e = cudaMallocAsync(ptr, std::max<size_t>(bytes, 256), stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync (scratch, stream capture)");
    return LBGEMM_OK;
  }
  if (s.bytes < bytes) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize (scratch growth)");
    // grow by at least half again, so that a run of ever larger problems
    // reallocates a logarithmic number of times (exactly `bytes` if that fails)
    size_t want = std::max<size_t>({bytes, size_t(1) << 20, s.bytes + s.bytes / 2});
    if (s.ptr) cudaFree(s.ptr);
    s.ptr = nullptr;
    s.bytes = 0;
    e = cudaMalloc(&s.ptr, want);
    if (e == cudaErrorMemoryAllocation && want > bytes) {
      cudaGetLastError();  // clear the failed attempt
      want = bytes;
      e = cudaMalloc(&s.ptr, want);
    }
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc (scratch)");
    s.bytes = want;
    s.used = false;
  }
  if (!s.done) {
    cudaError_t e = cudaEventCreateWithFlags(&s.done, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
  }
  if (s.used) {
    cudaError_t e = cudaStreamWaitEvent(stream, s.done, 0);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent");
  }
  *ptr = s.ptr;
  return LBGEMM_OK;
}

// Ends a use of the scratch that scratch_acquire handed out as `ptr`.
lbgemm_status scratch_release(Scratch& s, cudaStream_t stream, void* ptr) {
  if (ptr && ptr != s.ptr) {  // the graph's own allocation
    cudaError_t e = cudaFreeAsync(ptr, stream);
    return e == cudaSuccess ? LBGEMM_OK : cuda_fail(e, "cudaFreeAsync (scratch)");
  }
  cudaError_t e = cudaEventRecord(s.done, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  s.used = true;
  return LBGEMM_OK;
}

// ---- shapes, checks, variants ----------------------------------------------------------

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

lbgemm_status check_gemm_args(int bits, int64_t M, int64_t N, int64_t K, const void* A,
                              const void* B, const void* C) {
  if (bits != 8 && bits != 4 && bits != 1)
    return fail(LBGEMM_ERR_INVALID_ARG, "bits must be 8, 4 or 1 (got %d)", bits);
  if (M < 0 || N < 0) return fail(LBGEMM_ERR_INVALID_ARG, "negative M or N");
  if (K < 1) return fail(LBGEMM_ERR_INVALID_ARG, "K must be >= 1");
  if (M > INT32_MAX || N > INT32_MAX)
    return fail(LBGEMM_ERR_INVALID_ARG, "M and N must be below 2^31");
  const int64_t kmax = bits == 8 ? 131071 : bits == 4 ? (int64_t(1) << 25) - 1 : INT32_MAX - 1;
  if (K > kmax)
    return fail(LBGEMM_ERR_INVALID_ARG, "K=%lld can overflow int32 for %d-bit operands (max %lld)",
                (long long)K, bits, (long long)kmax);
  if (bits == 4 && K % 2) return fail(LBGEMM_ERR_ALIGNMENT, "4-bit rows need an even K");
  if (bits == 1 && K % 32) return fail(LBGEMM_ERR_ALIGNMENT, "1-bit rows need K %% 32 == 0");
  if (M == 0 || N == 0) return LBGEMM_OK;
  if (!A || !B || !C) return fail(LBGEMM_ERR_INVALID_ARG, "null operand pointer");
  if (!aligned16(A) || !aligned16(B) || !aligned16(C))
    return fail(LBGEMM_ERR_ALIGNMENT, "operand pointers must be 16-byte aligned");
  return LBGEMM_OK;
}

// Pipeline stages of variant v: levels 0, 1, 2 of the stage dimension are
// 2, 3, 4 stages for the single-CTA tiles and 4, 5, 6 for the CTA-pair large
// tile, whose 256 x 256 tile needs at least 4 stages in flight to cover the
// load latency (and stages cost it half as much shared memory per SM).
int variant_stages(int variant) {
  return variant / 3 == 2 ? variant % 3 + 4 : variant % 3 + 2;
}

// A tensor-core kernel instantiation: tile class (0 small, 1 medium, 2
// large) and stage count, packed as tile * 8 + stages.  The nine variants
// are nine of them; lbgemm_run_tile reaches the others the library compiles.
int spec_of(int variant) { return (variant / 3) * 8 + variant_stages(variant); }

TcKernel tc_kernel(int spec, bool f8, bool linear) {
  const int tile = spec / 8, stages = spec % 8;
  switch (tile) {
    case 0: return lbg::tc_kernel_small(stages, f8, linear);
    case 1: return lbg::tc_kernel_medium(stages, f8, linear);
    default: return lbg::tc_kernel_pair(stages, f8, linear);
  }
}

// Padded K of the re-encoded operands (row strides stay multiples of 16 bytes).
int64_t enc_kp(int bits, int64_t K) { return bits == 8 ? round_up(K, 8) : round_up(K, 16); }

size_t enc_bytes(int bits, int64_t rows, int64_t K) {
  const int64_t kp = enc_kp(bits, K);
  return (size_t)round_up(rows * kp * (bits == 8 ? 2 : 1), 256);
}

// Scratch of the linear layer on the in-kernel-conversion route: the
// re-encoded X, then room for the int32 sums of a split K (64- and 128-wide
// tiles).
size_t fused_linear_scratch(int64_t M, int64_t N, int64_t K, int tile_n) {
  size_t b = enc_bytes(8, M, K);
  if (tile_n != 256) b += (size_t)round_up(M * N * 4, 256);
  return b;
}

bool skinny_ok(int64_t M, int64_t K, const void* A, const void* B) {
  return M <= kSkinnyMaxM && K % 16 == 0 && aligned16(A) && aligned16(B);
}

// Problems this small run faster as one dp4a launch than as re-encoding plus
// a tensor-core launch.  Measured on GB300 over M, N, K in {64..2048}: the
// dp4a kernel wins for K <= 512 up to 2^28 MACs and loses from K = 1024 on
// (its K loop is latency-bound, one 64-byte stage per memory round trip).
bool small_ok(int64_t M, int64_t N, int64_t K, const void* A, const void* B) {
  return K <= kSmallMaxK && (double)M * (double)N * (double)K <= kSmallMaxWork && K % 16 == 0 &&
         aligned16(A) && aligned16(B);
}

// ---- selection table --------------------------------------------------------------------

// One table entry: the tile x stage variant measured fastest on the
// tensor-core kernel (the label of [LBG] section 2, used by lbgemm_select and
// lbgemm_run_encoded), and the kernel the default dispatch runs for the shape
// (route and its parameter: the variant for LBGEMM_ROUTE_TABLE and
// LBGEMM_ROUTE_POPC, the tile width for LBGEMM_ROUTE_FUSED, else 0).
// route < 0: no measured route (the shape rules decide).
struct Choice {
  int variant = kDefaultVariant;
  int route = -1;
  int param = 0;
};

using Key = std::tuple<int, int, int64_t, int64_t, int64_t>;  // sm, bits, M, N, K
std::mutex g_table_mu;
std::map<Key, Choice> g_table;
std::once_flag g_table_once;
std::string g_table_default_path;  // the file loaded at first use ("" if none)

lbgemm_status table_load_file(const char* path);

bool file_exists(const std::string& path) {
  FILE* f = fopen(path.c_str(), "r");
  if (!f) return false;
  fclose(f);
  return true;
}

// The data directory shipped beside the library (data/ next to its lib/).
std::string shipped_data_dir() {
  Dl_info info;
  if (!dladdr(reinterpret_cast<void*>(&shipped_data_dir), &info) || !info.dli_fname) return "";
  std::string so = info.dli_fname;
  const size_t slash = so.rfind('/');
  return (slash == std::string::npos ? std::string(".") : so.substr(0, slash)) + "/../data/";
}

// Loaded once per process, before the first use of the table: the table
// named by LBGEMM_TABLE ("" or "none": no table), else the GB300 table
// shipped beside the library (data/lbgemm_table_gb300.txt); and the selector
// networks shipped there (data/mlp_gb300_s<bits>.txt) unless LBGEMM_MLP is
// "" or "none".  A file that fails to load is reported on stderr and skipped.
void ensure_default_table() {
  std::call_once(g_table_once, [] {
    const std::string saved = t_last_error;
    const std::string dir = shipped_data_dir();
    std::string path;
    const char* env = std::getenv("LBGEMM_TABLE");
    if (env) {
      if (env[0] != '\0' && std::strcmp(env, "none") != 0) path = env;
    } else if (!dir.empty() && file_exists(dir + "lbgemm_table_gb300.txt")) {
      path = dir + "lbgemm_table_gb300.txt";
    }
    if (!path.empty()) {
      if (table_load_file(path.c_str()) == LBGEMM_OK)
        g_table_default_path = path;
      else
        fprintf(stderr, "lbgemm: selection table %s not loaded: %s\n", path.c_str(),
                t_last_error.c_str());
    }
    const char* envm = std::getenv("LBGEMM_MLP");
    const bool nets = !envm || (envm[0] != '\0' && std::strcmp(envm, "none") != 0);
    for (int bits : {8, 4, 1}) {
      const std::string net = dir + "mlp_gb300_s" + std::to_string(bits) + ".txt";
      if (!nets || dir.empty() || !file_exists(net)) continue;
      if (lbg::mlp_load_file(net.c_str()) != LBGEMM_OK)
        fprintf(stderr, "lbgemm: selector network %s not loaded: %s\n", net.c_str(),
                t_last_error.c_str());
    }
    t_last_error = saved;
  });
}

bool table_exact(int sm, int bits, int64_t M, int64_t N, int64_t K, Choice* out) {
  ensure_default_table();
  std::lock_guard<std::mutex> lock(g_table_mu);
  auto it = g_table.find(Key{sm, bits, M, N, K});
  if (it == g_table.end()) return false;
  *out = it->second;
  return true;
}

int table_select(int sm, int bits, int64_t M, int64_t N, int64_t K) {
  Choice c;
  if (table_exact(sm, bits, M, N, K, &c)) return c.variant;
  // not swept: the learned selector when one is loaded for this bit width
  const int v = lbg::mlp_pick(bits, M, N, K, sm);
  if (v >= 0) return v;
  std::lock_guard<std::mutex> lock(g_table_mu);
  int best = kDefaultVariant;
  double best_d = 0;
  bool have = false;
  const double lm = std::log2((double)std::max<int64_t>(M, 1));
  const double ln = std::log2((double)std::max<int64_t>(N, 1));
  const double lk = std::log2((double)std::max<int64_t>(K, 1));
  for (auto lo = g_table.lower_bound(Key{sm, bits, 0, 0, 0}); lo != g_table.end(); ++lo) {
    if (std::get<0>(lo->first) != sm || std::get<1>(lo->first) != bits) break;
    const double d = std::fabs(lm - std::log2((double)std::get<2>(lo->first))) +
                     std::fabs(ln - std::log2((double)std::get<3>(lo->first))) +
                     std::fabs(lk - std::log2((double)std::get<4>(lo->first)));
    if (!have || d < best_d - 1e-12) {
      best = lo->second.variant;
      best_d = d;
      have = true;
    }
  }
  return best;
}

// ---- TMA descriptors -----------------------------------------------------------------------

lbgemm_status encode_kmajor(CUtensorMap* map, const void* base, int64_t rows, int64_t kp,
                            bool f16, int box_rows) {
  const int esize = f16 ? 2 : 1;
  cuuint64_t dims[2] = {(cuuint64_t)kp, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(kp * esize)};
  cuuint32_t box[2] = {(cuuint32_t)(128 / esize), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                        2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(LBGEMM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return LBGEMM_OK;
}

// Work units a kernel can run at once on this device: resident CTAs per SM
// times the SM count, or for a CTA-pair kernel the clusters of two that fit
// at once (pairs must sit in one GPC, so this can be below half the SMs).
int unit_slots(DeviceState& d, const TcKernel& k) {
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = d.occupancy.find(k.func);
  if (it != d.occupancy.end()) return it->second;
  cudaFuncSetAttribute(k.func, cudaFuncAttributeMaxDynamicSharedMemorySize, k.smem);
  int slots = 0;
  if (k.cluster > 1) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(d.sm_count / k.cluster * k.cluster);
    cfg.blockDim = dim3(k.threads);
    cfg.dynamicSmemBytes = k.smem;
    int nc = 0;
    if (cudaOccupancyMaxActiveClusters(&nc, k.func, &cfg) != cudaSuccess || nc < 1) {
      cudaGetLastError();
      nc = 1;
    }
    slots = std::min(nc, d.sm_count / k.cluster);
  } else {
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k.func, k.threads, k.smem) !=
        cudaSuccess) {
      cudaGetLastError();
      occ = 1;
    }
    occ = std::max(1, std::min(occ, 512 / k.tmem_cols));
    slots = d.sm_count * occ;
  }
  d.occupancy[k.func] = slots;
  return slots;
}

// ---- the tensor-core path (bits 8 and 4, and the linear layer) --------------------------------

// Re-encodes operand a (and b, when rows_b > 0) in one launch.
// The same launch clears `zero` (the part of C that the GEMM launched after
// it adds partial tiles into), when given.
lbgemm_status encode_operands(DeviceState& d, int bits, const void* a, int64_t rows_a, void* enc_a,
                              const void* b, int64_t rows_b, void* enc_b, int64_t K,
                              cudaStream_t stream, const lbg::ZeroRect& zero = lbg::ZeroRect{}) {
  cudaError_t e = lbg::launch_encode_pair(bits, a, rows_a, enc_a, b, rows_b, enc_b, K,
                                          enc_kp(bits, K), d.sm_count, stream, zero);
  if (e != cudaSuccess) return cuda_fail(e, "operand re-encoding launch");
  g_launches += (rows_a + rows_b) > 0 || zero.C ? 1 : 0;
  return LBGEMM_OK;
}

// How the K dimension is shared out among CTAs.  Whole output tiles, one
// per unit, fill the complete waves of the device's CTA slots.  The tiles of
// a last, partial wave that would keep at most half of the slots busy are
// cut along K into `splits` pieces (at least 4 K slices each), so that the
// wave's pieces keep more slots busy and end sooner; so is the whole problem
// when it has at most half a wave of tiles.  Pieces add their int32 partial
// tiles into C, cleared beforehand: only for int32 C stored by TMA (the
// linear layer scales the whole sum).
struct KPlan {
  int dp_tiles = 0;  // TcParams::dp_tiles
  int splits = 1;    // TcParams::splits
  bool adds() const { return splits > 1; }
};

KPlan plan_k(DeviceState& d, const TcKernel& k, int bits, int64_t M, int64_t N, int64_t K,
             bool linear, bool vec_ok) {
  KPlan kp;
  if (linear || !vec_ok) return kp;
  const int bk = bits == 8 ? 64 : 128;
  const int64_t num_kb = (enc_kp(bits, K) + bk - 1) / bk;
  const int64_t tiles = ((M + k.tile_m - 1) / k.tile_m) * ((N + k.tile_n - 1) / k.tile_n);
  const int64_t slots = unit_slots(d, k);
  const int mode = g_tail_split.load();
  int64_t full = tiles / slots, rem = tiles - full * slots;
  if (full > 0 && mode == 0) return kp;
  if (mode == 2 && rem == 0) {  // forced: the last full wave is the tail
    --full;
    rem = slots;
  }
  if (rem == 0) return kp;
  const int64_t fit = slots / rem;  // pieces per tail tile that still fit the wave
  int64_t splits = std::min<int64_t>(std::min<int64_t>(fit, num_kb / 4), 64);
  if (mode == 2) splits = std::max<int64_t>(splits, std::min<int64_t>(num_kb, 2));
  if (splits < 2) return kp;
  kp.dp_tiles = (int)(full * slots);
  kp.splits = (int)splits;
  return kp;
}

// The rectangle of C that holds the split tiles (those from dp_tiles on, in
// the kernels' tile order), as rows [r0, r1) and columns [c0, c1), clipped to
// M x N.
void split_tiles_box(const TcKernel& k, int64_t M, int64_t N, int dp_tiles, int64_t* r0,
                     int64_t* r1, int64_t* c0, int64_t* c1) {
  const int64_t tiles_m = (M + k.tile_m - 1) / k.tile_m, tiles_n = (N + k.tile_n - 1) / k.tile_n;
  const int64_t tiles = tiles_m * tiles_n;
  int64_t tm_lo = tiles_m, tm_hi = -1, tn_lo = tiles_n, tn_hi = -1;
  for (int64_t t = dp_tiles; t < tiles; ++t) {
    // the tile order of the kernels: groups of kGroupM tile rows, column-major inside
    const int64_t per_group = (int64_t)kGroupM * tiles_n;
    const int64_t g = t / per_group, first = g * kGroupM;
    const int64_t gs = std::min<int64_t>(tiles_m - first, kGroupM);
    const int64_t r = t - g * per_group;
    const int64_t tm = first + r % gs, tn = r / gs;
    tm_lo = std::min(tm_lo, tm);
    tm_hi = std::max(tm_hi, tm);
    tn_lo = std::min(tn_lo, tn);
    tn_hi = std::max(tn_hi, tn);
  }
  *r0 = tm_lo * k.tile_m;
  *r1 = std::min<int64_t>((tm_hi + 1) * k.tile_m, M);
  *c0 = tn_lo * k.tile_n;
  *c1 = std::min<int64_t>((tn_hi + 1) * k.tile_n, N);
}

// The part of C that split tiles add into, as a rectangle for the encoder
// launch to clear (nothing when no tile is split).
lbg::ZeroRect split_rect(const TcKernel& k, const KPlan& kp, int64_t M, int64_t N, int32_t* C) {
  lbg::ZeroRect z;
  if (!kp.adds()) return z;
  z.C = C;
  z.ld = N;
  if (kp.dp_tiles == 0) {
    z.r1 = M;
    z.c1 = N;
  } else {
    split_tiles_box(k, M, N, kp.dp_tiles, &z.r0, &z.r1, &z.c0, &z.c1);
  }
  return z;
}

// Clears the part of C that split tiles add into (when no encoder launch
// precedes the GEMM).
lbgemm_status clear_split_tiles(const TcKernel& k, const KPlan& kp, int64_t M, int64_t N,
                                int32_t* C, cudaStream_t stream) {
  if (!kp.adds()) return LBGEMM_OK;
  cudaError_t e;
  if (kp.dp_tiles == 0) {
    e = cudaMemsetAsync(C, 0, (size_t)(M * N) * sizeof(int32_t), stream);
  } else {
    int64_t r0, r1, c0, c1;
    split_tiles_box(k, M, N, kp.dp_tiles, &r0, &r1, &c0, &c1);
    e = cudaMemset2DAsync(C + r0 * N + c0, (size_t)N * sizeof(int32_t), 0,
                          (size_t)(c1 - c0) * sizeof(int32_t), (size_t)(r1 - r0), stream);
  }
  return e == cudaSuccess ? LBGEMM_OK : cuda_fail(e, "clearing C for split tiles");
}

lbgemm_status run_tc_encoded(DeviceState& d, int bits, int64_t M, int64_t N, int64_t K,
                             const void* encA, const void* encB, int32_t* C, const float* sx,
                             const float* sw, void* Y, int spec, bool after_encode,
                             const KPlan* planned, cudaStream_t stream) {
  const bool f8 = bits != 8;  // 4-bit and 1-bit operands are e4m3-encoded
  const bool linear = Y != nullptr;
  TcKernel k = tc_kernel(spec, f8, linear);
  if (!k.launch)
    return fail(LBGEMM_ERR_UNSUPPORTED, "no kernel for tile %d with %d stages", spec / 8, spec % 8);
  const int64_t kp = enc_kp(bits, K);
  CUtensorMap ma, mb;
  lbgemm_status st = encode_kmajor(&ma, encA, M, kp, !f8, 128);
  if (st != LBGEMM_OK) return st;
  st = encode_kmajor(&mb, encB, N, kp, !f8, k.b_box_rows ? k.b_box_rows : k.tile_n);
  if (st != LBGEMM_OK) return st;

  TcParams p{};
  p.M = (int)M;
  p.N = (int)N;
  p.K = (int)K;
  const int bk = f8 ? 128 : 64;
  p.num_kb = (int)((kp + bk - 1) / bk);
  const int chunk_elems =
      bits == 8 ? g_chunk_s8.load() : bits == 4 ? g_chunk_s4.load() : g_chunk_b1.load();
  p.chunk_kb = std::max(1, chunk_elems / bk);
  p.tiles_m = (int)((M + k.tile_m - 1) / k.tile_m);
  p.tiles_n = (int)((N + k.tile_n - 1) / k.tile_n);
  p.num_tiles = p.tiles_m * p.tiles_n;
  p.group_m = kGroupM;
  p.C = C;
  p.sx = sx;
  p.sw = sw;
  p.Y = static_cast<__nv_bfloat16*>(Y);
  p.status = d.status;
  if (linear)
    p.vec_ok = (N % 8 == 0) && aligned16(Y);
  else
    p.vec_ok = (N % 4 == 0) && aligned16(C);
  KPlan plan;
  if (planned) {
    plan = *planned;
  } else {  // not planned by the caller: plan here and clear C now
    plan = plan_k(d, k, bits, M, N, K, linear, p.vec_ok);
    st = clear_split_tiles(k, plan, M, N, C, stream);
    if (st != LBGEMM_OK) return st;
  }
  p.dp_tiles = plan.dp_tiles;
  p.splits = plan.splits;
  p.num_units = plan.dp_tiles + (p.num_tiles - plan.dp_tiles) * plan.splits;
  CUtensorMap mc;
  std::memset(&mc, 0, sizeof mc);
  if (!linear && p.vec_ok) {
    cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)(N * 4)};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(&mc, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, C, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
      return fail(LBGEMM_ERR_CUDA, "cuTensorMapEncodeTiled (C) failed (%d)", (int)r);
  }
  // whole waves: dp_tiles is a multiple of the slots, so each CTA (pair) takes
  // the same number of whole tiles before the pieces of the last wave
  const int grid =
      (int)std::min<int64_t>(p.num_units, (int64_t)unit_slots(d, k)) * k.cluster;
  // Right after our own re-encoding launch, the GEMM is a programmatic
  // dependent launch: its prologue (barriers, TMEM, descriptor prefetch)
  // overlaps the encoder's tail and its producer waits for the encoder's
  // completion before the first operand load.
  cudaError_t e = k.launch(&ma, &mb, &mc, &p, grid, after_encode, stream);
  if (e != cudaSuccess) return cuda_fail(e, "tensor-core GEMM launch");
  g_launches += 1;
  return LBGEMM_OK;
}

lbgemm_status run_tc(DeviceState& d, int bits, int64_t M, int64_t N, int64_t K, const void* A,
                     const void* B, int32_t* C, const float* sx, const float* sw, void* Y,
                     int spec, void* ws, cudaStream_t stream) {
  uint8_t* encA = static_cast<uint8_t*>(ws);
  uint8_t* encB = encA + enc_bytes(bits, M, K);
  // Plan K splits first: the encoder launch clears the part of C that split
  // tiles add into, and the GEMM is launched as its dependent.
  KPlan plan;
  const bool linear = Y != nullptr;
  TcKernel k = tc_kernel(spec, bits != 8, linear);
  if (k.launch) {
    plan = plan_k(d, k, bits, M, N, K, linear, (N % 4 == 0) && aligned16(C));
  }
  // the encoder also clears the part of C that split tiles add into
  lbgemm_status st = encode_operands(d, bits, A, M, encA, B, N, encB, K, stream,
                                     split_rect(k, plan, M, N, C));
  if (st != LBGEMM_OK) return st;
  return run_tc_encoded(d, bits, M, N, K, encA, encB, C, sx, sw, Y, spec, true, &plan, stream);
}

// Work schedule of the 64- and 128-wide in-kernel-conversion kernels for
// rows_l rows converted in the kernel (128 per tile), rows_s re-encoded rows
// (tile_n per tile), K slices of `slice` elements, on `slots` CTA slots: K
// pieces per tile (splits), or stream-K (stream_pieces > 0: units per CTA).
// The cost of a plan is counted in whole-tile times: waves of units, a unit
// costing its share of the tile's K plus, when split, its partial tile of C
// (4 tile_n bytes per row against K).  The GEMM takes the cheapest split (up
// to 16 pieces, at least 4 slices of 64 each), stream-K only when forced;
// the linear layer splits only at kLinearSplitGain of the whole grid's cost
// and takes stream-K (each CTA's run plus one partial tile) at
// kLinearStreamGain of the plan chosen so far.
struct FusedSchedule {
  int splits = 1;
  int stream_pieces = 0;
};

FusedSchedule fused_schedule(int64_t rows_l, int64_t rows_s, int64_t K, int tile_n, int slice,
                             bool linear, int64_t slots, bool force_stream) {
  FusedSchedule fs;
  const int64_t tiles = ((rows_l + 127) / 128) * ((rows_s + tile_n - 1) / tile_n);
  const int64_t kp = enc_kp(8, K);
  const int64_t num_kb = (kp + 63) / 64;
  const double c_share = 4.0 * tile_n / (double)K;
  double best = 1e30;
  for (int sp = 1; sp <= 16 && (sp == 1 || num_kb / sp >= 4); ++sp) {
    const int64_t waves = (tiles * sp + slots - 1) / slots;
    const double cost = (double)waves * (1.0 / sp + (sp > 1 ? c_share : 0.0));
    if (cost < best - 1e-9) {
      best = cost;
      fs.splits = sp;
    }
  }
  const double whole = (double)((tiles + slots - 1) / slots);
  const int64_t kslices = (kp + slice - 1) / slice;
  const int64_t total = tiles * kslices;
  // stream-K: each CTA's run of slices plus about one partial tile more than
  // its whole tiles
  const int64_t run = total >= 2 * slots ? (total + slots - 1) / slots : 0;
  const double sk_cost =
      run ? (double)run / kslices + ((double)run / kslices + 1.0) * c_share : 1e30;
  bool stream = force_stream && run > 0;
  if (linear && !stream) {
    double chosen = best;
    if (best > kLinearSplitGain * whole) {
      fs.splits = 1;
      chosen = whole;
    }
    stream = sk_cost <= kLinearStreamGain * chosen;
  }
  if (stream) {
    fs.splits = 1;
    fs.stream_pieces = (int)((run + kslices - 1) / kslices + 1);
  }
  return fs;
}

// 8-bit problems with one operand converted in the kernel: only the other
// operand is re-encoded ahead.  large_b: B is converted (the kernel computes
// C transposed, rows of B on the tensor-memory A side); else A is converted.
// Requires K % 16 == 0 (16-byte int8 row strides for TMA).
lbgemm_status run_tc_fused(DeviceState& d, bool large_b, int tile_n, int64_t M, int64_t N,
                           int64_t K, const void* A, const void* B, int32_t* C, const float* sx,
                           const float* sw, void* Y, void* ws, cudaStream_t stream) {
  const bool linear = Y != nullptr;
  TcKernel k = lbg::tc_kernel_ts(tile_n, large_b, linear, fused_slice(tile_n, linear));
  if (!k.launch) return fail(LBGEMM_ERR_UNSUPPORTED, "no fused kernel (tile %d)", tile_n);
  // rows of the converted (L) and of the re-encoded (S) operand
  const int64_t rows_l = large_b ? N : M, rows_s = large_b ? M : N;
  const void* opl = large_b ? B : A;
  const void* ops = large_b ? A : B;
  const int64_t kp = enc_kp(8, K);  // == K when K % 16 == 0
  // C goes out by TMA stores (untransposed, aligned) or by coalesced atomics
  // (transposed); both can add split-K partial tiles.
  const bool vec_ok = !large_b && (linear ? (N % 8 == 0) && aligned16(Y)
                                          : (N % 4 == 0) && aligned16(C));
  // K pieces per tile.  The 128 x 256 kernel (compute-bound, one
  // accumulator): split only a problem of at most half a wave of tiles.  The
  // 64- and 128-wide kernels stream the int8 operand: as many pieces (up to
  // 16, at least 4 K slices each) as make the waves of units over the CTA
  // slots shortest, a unit costing its share of the tile's int8 rows plus
  // its partial tile of C (4 tile_n bytes per row against K) -- e.g. 128
  // tiles on 152 slots at K = 16384: 7 pieces (896 units in 6 waves, 6/7 of a
  // tile each) instead of one wave with 128 of the 152 slots busy (measured
  // on GB300: 64 x 16384 x 16384, 114 -> 106 us).
  // The linear layer splits K only when converting W (the transposed kernel)
  // with the 64- or 128-wide tile, and only where the split plan's waves cost
  // at most kLinearSplitGain of the unsplit grid's: it then runs as the plain
  // GEMM kernel adding int32 partial sums into a workspace after the
  // re-encoded operand in `ws` (fused_linear_scratch), and a second grid
  // scales the sums into Y.
  // Stream-K (64- and 128-wide kernels; the linear layer by its cost model,
  // the GEMM only when lbgemm_set_fused_stream_k asks): every CTA slot takes
  // an equal run of the tile-major order of all K slices, cut at tile ends
  // into pieces that each add a partial tile.  For the GEMM it measured no
  // faster than the split plan (e.g. 512 x 4096 x 1024: 21.5 against 15.4
  // us): a slice costs the kernel the same ~1200 cycles either way, bound by
  // the SM's shared- and tensor-memory traffic, so a shorter run per CTA buys
  // little against the extra partial tiles; the linear layer gains where its
  // tiles make a fractional number of waves (kLinearStreamGain).
  const bool linear_split = linear && large_b && tile_n != 256;
  int splits = 1, stream_pieces = 0;
  if ((!linear && (vec_ok || large_b)) || linear_split) {
    if (tile_n == 256) {
      KPlan kpl = plan_k(d, k, 8, rows_l, rows_s, K, linear, true);
      splits = kpl.dp_tiles == 0 ? kpl.splits : 1;
    } else {
      const FusedSchedule fs = fused_schedule(rows_l, rows_s, K, tile_n, k.slice, linear,
                                              unit_slots(d, k), g_stream_k.load() != 0);
      splits = fs.splits;
      stream_pieces = fs.stream_pieces;
    }
  }
  const bool partial = splits > 1 || stream_pieces > 0;
  // the linear layer with K shared out (split or stream-K): the plain kernel
  // adds into int32 sums, scaled into Y by a second grid below
  int32_t* sums = nullptr;
  if (linear && partial) {
    sums = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + enc_bytes(8, rows_s, K));
    k = lbg::tc_kernel_ts(tile_n, large_b, false, fused_slice(tile_n, true));
    if (!k.launch) return fail(LBGEMM_ERR_UNSUPPORTED, "no fused kernel (tile %d)", tile_n);
  }
  int32_t* Cout = sums ? sums : C;
  // the encoder also clears C (or the sums) when K is split: partial tiles
  // are added into it
  lbg::ZeroRect zero;
  if (partial) {
    zero.C = Cout;
    zero.ld = N;
    zero.r1 = M;
    zero.c1 = N;
  }
  lbgemm_status st = encode_operands(d, 8, ops, rows_s, ws, nullptr, 0, nullptr, K, stream, zero);
  if (st != LBGEMM_OK) return st;
  CUtensorMap ml, ms;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows_l};
  cuuint64_t strides[1] = {(cuuint64_t)K};
  // the int8 operand is staged in 128-element boxes (128-byte swizzle); the
  // 256-wide kernel steps through K in 64-element slices, the others in
  // 128-element slices
  const bool pairs = tile_n == 256;
  const int slice = pairs ? 64 : k.slice;
  cuuint32_t box[2] = {128u, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(&ml, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(opl), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(LBGEMM_ERR_CUDA, "cuTensorMapEncodeTiled (int8) failed (%d)", (int)r);
  st = encode_kmajor(&ms, ws, rows_s, kp, true, tile_n);
  if (st != LBGEMM_OK) return st;
  TcParams p{};
  p.M = (int)rows_l;
  p.N = (int)rows_s;
  p.K = (int)K;
  p.num_kb = (int)((kp + slice - 1) / slice);
  p.chunk_kb = std::max(1, g_chunk_s8.load() / slice);
  if (pairs) p.chunk_kb = std::max(4, p.chunk_kb & ~3);  // whole groups of 4 slices
  p.tiles_m = (int)((rows_l + 127) / 128);
  p.tiles_n = (int)((rows_s + tile_n - 1) / tile_n);
  p.num_tiles = p.tiles_m * p.tiles_n;
  p.group_m = kGroupM;
  p.splits = splits;
  p.num_units = p.num_tiles * splits;
  if (stream_pieces > 0) {
    p.stream_k = stream_pieces;
    p.num_units = (int)unit_slots(d, k) * stream_pieces;
  }
  p.C = Cout;
  p.sx = sx;
  p.sw = sw;
  p.Y = sums ? nullptr : static_cast<__nv_bfloat16*>(Y);
  p.status = d.status;
  p.vec_ok = vec_ok;
  CUtensorMap mc;
  std::memset(&mc, 0, sizeof mc);
  if (!linear && vec_ok) {
    cuuint64_t cd[2] = {(cuuint64_t)N, (cuuint64_t)M};
    cuuint64_t cs[1] = {(cuuint64_t)(N * 4)};
    cuuint32_t cb[2] = {32, 32};
    r = g_encode(&mc, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, C, cd, cs, cb, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(LBGEMM_ERR_CUDA, "cuTensorMapEncodeTiled (C) failed (%d)", (int)r);
  }
  const int grid = (int)std::min<int64_t>(p.num_units, (int64_t)unit_slots(d, k));
  cudaError_t e = k.launch(&ml, &ms, &mc, &p, grid, true, stream);
  if (e != cudaSuccess) return cuda_fail(e, "fused tensor-core GEMM launch");
  g_launches += 1;
  if (sums) {
    e = lbg::launch_scale_sums(sums, M, N, sx, sw, Y, d.sm_count, stream);
    if (e != cudaSuccess) return cuda_fail(e, "linear-layer scaling launch");
    g_launches += 1;
  }
  return LBGEMM_OK;
}

// The warp-level fp16 MMA kernel for a small side (<= kWarpMmaMaxSide rows):
// X is the small operand, W the large one; C (or Y) is written transposed
// from the kernel's point of view when the small side is B.
lbgemm_status run_warpmma(DeviceState& d, int64_t M, int64_t N, int64_t K, const int8_t* A,
                          const int8_t* B, int32_t* C, const float* sx, const float* sw, void* Y,
                          cudaStream_t stream) {
  const bool small_a = M <= N;
  cudaError_t e =
      small_a ? lbg::launch_hmma_skinny(A, B, (int)M, (int)N, (int)K, false, C, sx, sw, Y,
                                        g_chunk_s8.load(), d.sm_count, stream)
              : lbg::launch_hmma_skinny(B, A, (int)N, (int)M, (int)K, true, C, sw, sx, Y,
                                        g_chunk_s8.load(), d.sm_count, stream);
  if (e != cudaSuccess) return cuda_fail(e, "warp-MMA GEMM launch");
  g_launches += 1;
  return LBGEMM_OK;
}

// The streaming kernel takes a problem with a small side of at most 16 rows
// against at least 1024 (measured on GB300, 5-16 rows x 11008 x 4096, back to
// back over rotating weights: 12.6-13.3 us against 14.2 on the warp-MMA
// kernel; the dp4a kernel stays ahead up to 4 rows), K <= 4096.
bool stream_ok(int64_t M, int64_t N, int64_t K, const void* A, const void* B) {
  return std::min(M, N) <= kStreamMaxSide && std::max(M, N) >= 1024 && K % 16 == 0 &&
         K <= lbg::stream_mma_max_k() && aligned16(A) && aligned16(B);
}

// The warp-MMA kernel takes the problem: small side <= kWarpMmaMaxSide rows,
// X fits its shared memory, K % 16 == 0, aligned operands.
bool warpmma_ok(int64_t M, int64_t N, int64_t K, const void* A, const void* B) {
  const int64_t lo = std::min(M, N);
  return lo <= kWarpMmaMaxSide && K % 16 == 0 && K <= lbg::hmma_skinny_max_k((int)lo) &&
         aligned16(A) && aligned16(B);
}

// The same kernel for a small problem with a side of up to
// kWarpMmaMaxSideSmall rows and 256 < K <= 2048: M*N <= 2^19 (2^18 past
// K = 1024), or the one-launch dp4a kernel's problems (K <= 512,
// M*N*K <= 2^28).
bool warpmma_small_ok(int64_t M, int64_t N, int64_t K, const void* A, const void* B) {
  const int64_t lo = std::min(M, N), hi = std::max(M, N);
  // past 1024 of K, half the area: the in-kernel conversion kernel with
  // 128-element slices is faster there (e.g. 64 x 8192 x 2048: 21.1 -> 17.1 us)
  const int64_t max_area = K <= 1024 ? kWarpMmaMaxArea : kWarpMmaMaxArea / 2;
  const bool area = lo * hi <= max_area ||
                    (K <= kSmallMaxK && (double)M * (double)N * (double)K <= kSmallMaxWork);
  return lo <= kWarpMmaMaxSideSmall && K > 256 && K <= kWarpMmaMaxKSmall && area &&
         K % 16 == 0 && K <= lbg::hmma_skinny_max_k((int)lo) && aligned16(A) && aligned16(B);
}

// Route of the in-kernel-conversion kernel for an 8-bit problem (1: B is
// converted in the kernel, 2: A is; 0: re-encode both) and its tile width
// along the re-encoded operand.  Measured on GB300 over the grid of small
// side 64-512, large side 1024-16384 and K 512-16384 (both orientations),
// against re-encoding and the warp-MMA kernel: skipping the large operand's
// re-encoding pass wins once the large side reaches 4096 rows, at K >= 4096
// from 2048 rows, at K >= 8192 from 1024, and with at most 256 rows on the
// small side from K = 2048 (e.g. 512 x 4096 x 1024: 17.0 -> 15.0 us;
// 256 x 8192 x 2048: 27.3 -> 21.1 us; 256 x 16384 x 16384: 275 -> 146 us).
// The tile: 64 up to 64 rows, else 128, but 256 (CTA pairs) for a small side
// of 129-256 or 385-512 rows with the large side and K both large, where the
// pairs' shared re-encoded tile pays.
int fused_route(int64_t M, int64_t N, int64_t K, const void* A, const void* B, int* tile_n) {
  if (K % 16 || !aligned16(A) || !aligned16(B)) return 0;
  const int64_t lo = std::min(M, N), hi = std::max(M, N);
  if (!(lo <= kFusedMaxSide && hi >= kFusedMinOther) || K < 512) return 0;
  const bool go =
      hi >= 4096 || K >= 8192 || (hi >= 2048 && K >= 4096) || (lo <= 256 && K >= 2048);
  if (!go) return 0;
  bool pairs = false;
  if (lo > 128 && lo <= 256)
    pairs = (hi >= 16384 && K >= 1024) || (hi >= 8192 && K >= 16384);
  else if (lo > 384)
    pairs = (hi >= 8192 && K >= 2048) || (hi >= 16384 && K >= 1024) || K >= 16384;
  *tile_n = lo <= 64 ? 64 : pairs ? 256 : 128;
  return M <= N ? 1 : 2;
}

// The kernel lbgemm_run (linear = false) or lbgemm_linear (linear = true)
// picks for a problem with the default dispatch; *tile_n is the in-kernel
// conversion kernel's tile width (LBGEMM_ROUTE_FUSED) and *fuse which
// operand it converts (1: B, 2: A).  The dispatchers call this, so the
// introspection entry point cannot drift from them.
bool route_runs(int bits, int64_t M, int64_t N, int64_t K, const void* A, const void* B, int route,
                int param);

int route_of(int bits, int64_t M, int64_t N, int64_t K, const void* A, const void* B, bool linear,
             int* tile_n, int* fuse) {
  *tile_n = 0;
  *fuse = 0;
  if (M == 0 || N == 0) return LBGEMM_ROUTE_NONE;
  if (linear) {
    // 5-8 tokens past the streaming kernel's K: the dp4a kernel still wins up
    // to K = 8192 (measured on GB300: 8 x 28672 x 8192, 77.8 -> 71.7 us; 8 x
    // 8192 x 8192, 32.3 -> 31.0; at K = 11008 and beyond it loses to the
    // in-kernel-conversion kernel, 26.9 against 34.8 us for 8 x 4096 x 11008)
    if (skinny_ok(M, K, A, B) ||
        (M <= 2 * kSkinnyMaxM && K > lbg::stream_mma_max_k() && K <= 8192 &&
         skinny_ok(1, K, A, B)))
      return LBGEMM_ROUTE_SKINNY;
    if (M <= kStreamMaxSide && stream_ok(M, N, K, A, B)) return LBGEMM_ROUTE_STREAM;
    if (warpmma_ok(M, N, K, A, B)) return LBGEMM_ROUTE_WARPMMA;
    if (fused_route(M, N, K, A, B, tile_n) == 1) {
      // the linear layer keeps the 128-wide tile where the GEMM would take
      // CTA pairs: with its 256-element K slices and K shared out where the
      // grid is short it is faster on every layer measured on GB300 (400-512
      // tokens: 512 x 28672 x 8192, 230 -> 200 us; 512 x 8192 x 28672, 250 ->
      // 230 us; 512 x 4096 x 16384, 150 -> 78 us; 256 tokens, equal or faster
      // up to 28672 x 8192)
      if (*tile_n == 256) *tile_n = 128;
      *fuse = 1;
      return LBGEMM_ROUTE_FUSED;
    }
    *tile_n = 0;
    return LBGEMM_ROUTE_TABLE;
  }
  if (bits == 1) {
    return (double)M * (double)N * (double)K < kPopcMaxWork ? LBGEMM_ROUTE_POPC
                                                             : LBGEMM_ROUTE_TABLE;
  }
  if (bits == 4) {
    return K <= kSmallS4MaxK && (double)M * (double)N * (double)K <= kSmallS4MaxWork &&
                   route_runs(4, M, N, K, A, B, LBGEMM_ROUTE_SMALL, 0)
               ? LBGEMM_ROUTE_SMALL
               : LBGEMM_ROUTE_TABLE;
  }
  if (bits != 8) return LBGEMM_ROUTE_TABLE;
  if (skinny_ok(M, K, A, B)) return LBGEMM_ROUTE_SKINNY;
  if (stream_ok(M, N, K, A, B)) return LBGEMM_ROUTE_STREAM;
  if (warpmma_ok(M, N, K, A, B) || warpmma_small_ok(M, N, K, A, B)) return LBGEMM_ROUTE_WARPMMA;
  if (small_ok(M, N, K, A, B)) return LBGEMM_ROUTE_SMALL;
  *fuse = fused_route(M, N, K, A, B, tile_n);
  if (*fuse) return LBGEMM_ROUTE_FUSED;
  *tile_n = 0;
  return LBGEMM_ROUTE_TABLE;
}

// Whether the kernel of (route, param) runs this problem: its size limits,
// K alignment and operand alignment.  Every tensor-core variant runs every
// problem (LBGEMM_ROUTE_TABLE, param = variant).
bool route_runs(int bits, int64_t M, int64_t N, int64_t K, const void* A, const void* B, int route,
                int param) {
  const bool a16 = K % 16 == 0 && aligned16(A) && aligned16(B);
  const int64_t lo = std::min(M, N);
  switch (route) {
    case LBGEMM_ROUTE_TABLE: return param >= 0 && param < kNumVariants;
    case LBGEMM_ROUTE_POPC: return bits == 1 && param >= 0 && param < kNumVariants;
    case LBGEMM_ROUTE_SKINNY: return bits == 8 && M <= kSkinnyKernelMaxM && a16;
    case LBGEMM_ROUTE_WARPMMA:
      return bits == 8 && lo <= kWarpMmaMaxSideSmall && a16 &&
             K <= lbg::hmma_skinny_max_k((int)lo);
    case LBGEMM_ROUTE_SMALL:
      return (bits == 8 && a16) ||
             (bits == 4 && K % 32 == 0 && aligned16(A) && aligned16(B));
    case LBGEMM_ROUTE_FUSED: return bits == 8 && (param == 64 || param == 128 || param == 256) && a16;
    case LBGEMM_ROUTE_STREAM:
      return bits == 8 && lo <= kStreamMaxSide && a16 && K <= lbg::stream_mma_max_k();
    default: return false;
  }
}

// The routes of the linear layer (X = A is the token side; Y is M x N bf16):
// the tensor-core variants, the dp4a and streaming kernels for few tokens,
// the warp-MMA kernel, and the in-kernel conversion of W.
bool linear_route_runs(int64_t M, int64_t N, int64_t K, const void* X, const void* W, int route,
                       int param) {
  const bool a16 = K % 16 == 0 && aligned16(X) && aligned16(W);
  switch (route) {
    case LBGEMM_ROUTE_TABLE: return param >= 0 && param < kNumVariants;
    case LBGEMM_ROUTE_SKINNY: return M <= kSkinnyKernelMaxM && a16;
    case LBGEMM_ROUTE_STREAM:
      return M <= kStreamMaxSide && a16 && K <= lbg::stream_mma_max_k();
    case LBGEMM_ROUTE_WARPMMA:
      return std::min(M, N) <= kWarpMmaMaxSide && a16 &&
             K <= lbg::hmma_skinny_max_k((int)std::min(M, N));
    case LBGEMM_ROUTE_FUSED:
      return (param == 64 || param == 128 || param == 256) && M <= N && a16;
    default: return false;
  }
}

// The candidates the timing sweep measures for a shape (16-byte-aligned
// operands): the nine tensor-core variants, and each shape-route kernel that
// runs the problem within the domain where it can plausibly win (kept small
// so the sweep ends in minutes): the 1-bit popcount kernel's nine variants
// below 2^34 bit-MACs; the dp4a kernel streaming B for M <= 16; the warp-MMA
// kernel for a small side of up to 256 rows; the one-launch dp4a kernel up to
// 2^31 MACs and K <= 4096; the in-kernel conversion kernel at tile widths 64
// and 128 (and 256 once the small side exceeds 64 rows) for a small side of
// up to 1024 rows.
int candidate_list(int bits, int64_t M, int64_t N, int64_t K, int* routes, int* params, int max) {
  const void* al = reinterpret_cast<const void*>(uintptr_t(256));
  int n = 0;
  auto add = [&](int r, int p) {
    if (n < max) {
      routes[n] = r;
      params[n] = p;
    }
    ++n;
  };
  for (int v = 0; v < kNumVariants; ++v) add(LBGEMM_ROUTE_TABLE, v);
  const double work = (double)M * (double)N * (double)K;
  const int64_t lo = std::min(M, N);
  if (bits == 1 && work < 17179869184.0)
    for (int v = 0; v < kNumVariants; ++v) add(LBGEMM_ROUTE_POPC, v);
  if (bits == 4 && K % 32 == 0 && work <= 2147483648.0 && K <= 8192) add(LBGEMM_ROUTE_SMALL, 0);
  if (bits != 8 || K % 16) return n;
  if (route_runs(8, M, N, K, al, al, LBGEMM_ROUTE_SKINNY, 0)) add(LBGEMM_ROUTE_SKINNY, 0);
  if (route_runs(8, M, N, K, al, al, LBGEMM_ROUTE_STREAM, 0)) add(LBGEMM_ROUTE_STREAM, 0);
  if (route_runs(8, M, N, K, al, al, LBGEMM_ROUTE_WARPMMA, 0)) add(LBGEMM_ROUTE_WARPMMA, 0);
  if (work <= 2147483648.0 && K <= 4096) add(LBGEMM_ROUTE_SMALL, 0);
  if (lo <= 1024) {
    add(LBGEMM_ROUTE_FUSED, 64);
    add(LBGEMM_ROUTE_FUSED, 128);
    if (lo > 64) add(LBGEMM_ROUTE_FUSED, 256);
  }
  return n;
}

// The kernel the default dispatch runs: the table's measured route for the
// exact shape when it has one that runs these operands, else the shape rules
// (route_of), with the variant from table_select on the tensor-core route.
struct Pick {
  int route = LBGEMM_ROUTE_NONE;
  int param = 0;
  int spec = -1;  // LBGEMM_ROUTE_TABLE: an explicit kernel spec instead of variant `param`
};

int tc_spec(const Pick& p) { return p.spec >= 0 ? p.spec : spec_of(p.param); }

Pick pick_route(int sm, int bits, int64_t M, int64_t N, int64_t K, const void* A, const void* B) {
  Pick p;
  if (M == 0 || N == 0) return p;
  Choice c;
  if (table_exact(sm, bits, M, N, K, &c) && c.route >= 0 &&
      route_runs(bits, M, N, K, A, B, c.route, c.param)) {
    p.route = c.route;
    p.param = c.param;
    return p;
  }
  int tile = 0, fuse = 0;
  p.route = route_of(bits, M, N, K, A, B, false, &tile, &fuse);
  p.param = p.route == LBGEMM_ROUTE_TABLE   ? table_select(sm, bits, M, N, K)
            : p.route == LBGEMM_ROUTE_POPC  ? kPopcRuleVariant
            : p.route == LBGEMM_ROUTE_FUSED ? tile
                                            : 0;
  return p;
}

// Scratch bytes of a route: both re-encoded operands on the tensor-core
// route, the re-encoded smaller operand on the in-kernel conversion route,
// none elsewhere.
size_t route_scratch(int bits, int64_t M, int64_t N, int64_t K, const Pick& p) {
  if (p.route == LBGEMM_ROUTE_TABLE) return enc_bytes(bits, M, K) + enc_bytes(bits, N, K);
  if (p.route == LBGEMM_ROUTE_FUSED) return enc_bytes(8, std::min(M, N), K);
  return 0;
}

// Runs one route on checked arguments.  Scratch: the caller's `ws` when
// internal_ws is false (checked here), else the per-device buffer.
lbgemm_status run_route(DeviceState& d, int bits, int64_t M, int64_t N, int64_t K, const void* A,
                        const void* B, int32_t* C, const Pick& p, void* ws, size_t ws_bytes,
                        bool internal_ws, cudaStream_t stream) {
  cudaError_t e;
  switch (p.route) {
    case LBGEMM_ROUTE_NONE: return LBGEMM_OK;
    case LBGEMM_ROUTE_POPC:
      // XOR + popcount on CUDA cores, no re-encoding
      e = lbg::launch_b1_popc(p.param / 3, p.param % 3 + 2, static_cast<const uint32_t*>(A),
                              static_cast<const uint32_t*>(B), M, N, K, C, stream);
      if (e != cudaSuccess) return cuda_fail(e, "1-bit popcount GEMM launch");
      g_launches += 1;
      return LBGEMM_OK;
    case LBGEMM_ROUTE_SKINNY:
      e = lbg::launch_skinny_s8(static_cast<const int8_t*>(A), static_cast<const int8_t*>(B),
                                (int)M, (int)N, (int)K, C, nullptr, nullptr, nullptr, d.sm_count,
                                stream);
      if (e != cudaSuccess) return cuda_fail(e, "skinny GEMM launch");
      g_launches += 1;
      return LBGEMM_OK;
    case LBGEMM_ROUTE_WARPMMA:
      return run_warpmma(d, M, N, K, static_cast<const int8_t*>(A), static_cast<const int8_t*>(B),
                         C, nullptr, nullptr, nullptr, stream);
    case LBGEMM_ROUTE_SMALL:
      e = bits == 4 ? lbg::launch_small_s4(static_cast<const uint8_t*>(A),
                                           static_cast<const uint8_t*>(B), M, N, K, C, stream)
                    : lbg::launch_small_s8(static_cast<const int8_t*>(A),
                                           static_cast<const int8_t*>(B), M, N, K, C, stream);
      if (e != cudaSuccess) return cuda_fail(e, "small GEMM launch");
      g_launches += 1;
      return LBGEMM_OK;
    case LBGEMM_ROUTE_STREAM:
      // the small side is X; C is written transposed from its point of view
      // when that side is B
      e = M <= N ? lbg::launch_stream_mma(static_cast<const int8_t*>(A),
                                          static_cast<const int8_t*>(B), (int)M, (int)N, (int)K,
                                          false, C, nullptr, nullptr, nullptr, false, d.sm_count,
                                          d.status, stream)
                 : lbg::launch_stream_mma(static_cast<const int8_t*>(B),
                                          static_cast<const int8_t*>(A), (int)N, (int)M, (int)K,
                                          true, C, nullptr, nullptr, nullptr, false, d.sm_count,
                                          d.status, stream);
      if (e != cudaSuccess) return cuda_fail(e, "streaming GEMM launch");
      g_launches += 1;
      return LBGEMM_OK;
    default: break;
  }
  const size_t need = route_scratch(bits, M, N, K, p);
  if (!internal_ws) {
    if (!ws || ws_bytes < need)
      return fail(LBGEMM_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, ws_bytes);
    if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0)
      return fail(LBGEMM_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
    if (p.route == LBGEMM_ROUTE_FUSED)
      return run_tc_fused(d, N >= M, p.param, M, N, K, A, B, C, nullptr, nullptr, nullptr, ws,
                          stream);
    return run_tc(d, bits, M, N, K, A, B, C, nullptr, nullptr, nullptr, tc_spec(p), ws, stream);
  }
  std::lock_guard<std::mutex> lock(g_ws_mu);
  void* scratch = nullptr;
  lbgemm_status st = scratch_acquire(d.ws, need, stream, &scratch);
  if (st != LBGEMM_OK) return st;
  if (p.route == LBGEMM_ROUTE_FUSED)
    st = run_tc_fused(d, N >= M, p.param, M, N, K, A, B, C, nullptr, nullptr, nullptr, scratch,
                      stream);
  else
    st = run_tc(d, bits, M, N, K, A, B, C, nullptr, nullptr, nullptr, tc_spec(p), scratch,
                stream);
  lbgemm_status st2 = scratch_release(d.ws, stream, scratch);
  return st != LBGEMM_OK ? st : st2;
}

lbgemm_status run_any(int bits, int64_t M, int64_t N, int64_t K, const void* A, const void* B,
                      int32_t* C, int variant, void* ws, size_t ws_bytes, bool internal_ws,
                      cudaStream_t stream) {
  lbgemm_status st = check_gemm_args(bits, M, N, K, A, B, C);
  if (st != LBGEMM_OK) return st;
  if (variant < -1 || variant >= kNumVariants)
    return fail(LBGEMM_ERR_INVALID_ARG, "variant %d out of range", variant);
  if (M == 0 || N == 0) return LBGEMM_OK;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != LBGEMM_OK) return st;
  Pick p;
  if (variant < 0) {
    p = pick_route(d->sm_count, bits, M, N, K, A, B);
  } else {
    p.route = LBGEMM_ROUTE_TABLE;
    p.param = variant;
  }
  return run_route(*d, bits, M, N, K, A, B, C, p, ws, ws_bytes, internal_ws, stream);
}

// The linear layer.  route < 0: by the shape rules (variant < 0) or the
// tensor-core variant `variant`; else that route with its parameter (the
// variant of LBGEMM_ROUTE_TABLE, the tile width of LBGEMM_ROUTE_FUSED).
// early_w: W is not written by the grid launched before this call on the
// stream (the caller's own quantiser), so the streaming kernel may start
// reading it before that grid ends.
lbgemm_status run_linear(int64_t M, int64_t N, int64_t K, const int8_t* X, const float* sx,
                         const int8_t* W, const float* sw, void* Y, int variant,
                         cudaStream_t stream, int route = -1, int param = 0,
                         bool early_w = false) {
  lbgemm_status st = check_gemm_args(8, M, N, K, X, W, Y);
  if (st != LBGEMM_OK) return st;
  if (variant < -1 || variant >= kNumVariants)
    return fail(LBGEMM_ERR_INVALID_ARG, "variant %d out of range", variant);
  if (route >= 0 && !linear_route_runs(M, N, K, X, W, route, param))
    return fail(LBGEMM_ERR_INVALID_ARG, "route %d (param %d) cannot run this linear layer", route,
                param);
  if (M == 0 || N == 0) return LBGEMM_OK;
  if (!sx || !sw) return fail(LBGEMM_ERR_INVALID_ARG, "null scale pointer");
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != LBGEMM_OK) return st;
  int fuse_tile = param, fuse = 0;
  if (route < 0) {
    route = variant < 0 ? route_of(8, M, N, K, X, W, true, &fuse_tile, &fuse) : LBGEMM_ROUTE_TABLE;
    if (route == LBGEMM_ROUTE_TABLE)
      variant = variant < 0 ? table_select(d->sm_count, 8, M, N, K) : variant;
  } else if (route == LBGEMM_ROUTE_TABLE) {
    variant = param;
  }
  if (route == LBGEMM_ROUTE_SKINNY) {
    cudaError_t e =
        lbg::launch_skinny_s8(X, W, (int)M, (int)N, (int)K, nullptr, sx, sw, Y, d->sm_count, stream);
    if (e != cudaSuccess) return cuda_fail(e, "skinny linear launch");
    g_launches += 1;
    return LBGEMM_OK;
  }
  if (route == LBGEMM_ROUTE_STREAM) {
    cudaError_t e = lbg::launch_stream_mma(X, W, (int)M, (int)N, (int)K, false, nullptr, sx, sw, Y,
                                           early_w, d->sm_count, d->status, stream);
    if (e != cudaSuccess) return cuda_fail(e, "streaming linear launch");
    g_launches += 1;
    return LBGEMM_OK;
  }
  if (route == LBGEMM_ROUTE_WARPMMA)
    return run_warpmma(*d, M, N, K, X, W, nullptr, sx, sw, Y, stream);
  if (route == LBGEMM_ROUTE_FUSED) {
    // small token counts: only X is re-encoded; the kernel converts W itself
    std::lock_guard<std::mutex> lock(g_ws_mu);
    void* scratch = nullptr;
    st = scratch_acquire(d->ws, fused_linear_scratch(M, N, K, fuse_tile), stream, &scratch);
    if (st != LBGEMM_OK) return st;
    st = run_tc_fused(*d, true, fuse_tile, M, N, K, X, W, nullptr, sx, sw, Y, scratch, stream);
    lbgemm_status st2 = scratch_release(d->ws, stream, scratch);
    return st != LBGEMM_OK ? st : st2;
  }
  std::lock_guard<std::mutex> lock(g_ws_mu);
  const size_t need = enc_bytes(8, M, K) + enc_bytes(8, N, K);
  void* scratch = nullptr;
  st = scratch_acquire(d->ws, need, stream, &scratch);
  if (st != LBGEMM_OK) return st;
  st = run_tc(*d, 8, M, N, K, X, W, nullptr, sx, sw, Y, spec_of(variant), scratch, stream);
  lbgemm_status st2 = scratch_release(d->ws, stream, scratch);
  return st != LBGEMM_OK ? st : st2;
}

// A table entry's route must be one the dispatch can run at the entry's sizes
// (16-byte-aligned operands; the 8-bit routes need K % 16 == 0).
bool entry_route_ok(int bits, int64_t M, int64_t N, int64_t K, int route, int param) {
  const void* al = reinterpret_cast<const void*>(uintptr_t(256));
  return route >= 0 && route != LBGEMM_ROUTE_NONE && route_runs(bits, M, N, K, al, al, route, param);
}

// Reads "sm_count bits M N K variant [route param]" lines ('#' comments) and
// merges them into the table; nothing is merged if any line is malformed.
lbgemm_status table_load_file(const char* path) {
  if (!path) return fail(LBGEMM_ERR_INVALID_ARG, "null path");
  FILE* f = fopen(path, "r");
  if (!f) return fail(LBGEMM_ERR_INVALID_ARG, "cannot open %s", path);
  std::vector<std::pair<Key, Choice>> rows;
  char line[256];
  int lineno = 0;
  while (fgets(line, sizeof line, f)) {
    ++lineno;
    const char* s = line;
    while (*s == ' ' || *s == '\t') ++s;
    if (*s == '#' || *s == '\n' || *s == '\0') continue;
    int sm, bits, v, route = -1, param = 0;
    long long M, N, K;
    char extra[2];
    const int got = sscanf(s, "%d %d %lld %lld %lld %d %d %d %1s", &sm, &bits, &M, &N, &K, &v,
                           &route, &param, extra);
    const bool shape_ok = (got == 6 || got == 8) && sm >= 1 &&
                          (bits == 8 || bits == 4 || bits == 1) && M >= 1 && N >= 1 && K >= 1 &&
                          v >= 0 && v < kNumVariants;
    if (got == 6) route = -1;
    if (!shape_ok || (got == 8 && !entry_route_ok(bits, M, N, K, route, param))) {
      fclose(f);
      return fail(LBGEMM_ERR_INVALID_ARG, "%s:%d: malformed table line", path, lineno);
    }
    Choice c;
    c.variant = v;
    c.route = route;
    c.param = route >= 0 ? param : 0;
    rows.push_back({Key{sm, bits, M, N, K}, c});
  }
  fclose(f);
  std::lock_guard<std::mutex> lock(g_table_mu);
  for (auto& r : rows) g_table[r.first] = r.second;
  return LBGEMM_OK;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

}  // namespace

// =============================================================================================
extern "C" {

int lbgemm_num_variants(void) { return kNumVariants; }
int lbgemm_default_variant(void) { return kDefaultVariant; }

lbgemm_status lbgemm_variant_info(int bits, int variant, int* tile_m, int* tile_n, int* tile_k,
                                  int* stages) {
  if ((bits != 8 && bits != 4 && bits != 1) || variant < 0 || variant >= kNumVariants)
    return fail(LBGEMM_ERR_INVALID_ARG, "unknown bits/variant");
  const int tile = variant / 3;
  const int bm = tile == 2 ? 256 : 128, bn = 64 << tile, bk = bits == 8 ? 64 : 128;
  if (tile_m) *tile_m = bm;
  if (tile_n) *tile_n = bn;
  if (tile_k) *tile_k = bk;
  if (stages) *stages = variant_stages(variant);
  return LBGEMM_OK;
}

lbgemm_status lbgemm_run(int bits, int64_t M, int64_t N, int64_t K, const void* A, const void* B,
                         int32_t* C, void* stream) {
  try {
    return run_any(bits, M, N, K, A, B, C, -1, nullptr, 0, true, as_stream(stream));
  } catch (...) {
    return fail(LBGEMM_ERR_CUDA, "internal error");
  }
}

lbgemm_status lbgemm_run_variant(int bits, int64_t M, int64_t N, int64_t K, const void* A,
                                 const void* B, int32_t* C, int variant, void* stream) {
  try {
    return run_any(bits, M, N, K, A, B, C, variant, nullptr, 0, true, as_stream(stream));
  } catch (...) {
    return fail(LBGEMM_ERR_CUDA, "internal error");
  }
}

lbgemm_status lbgemm_run_fused(int64_t M, int64_t N, int64_t K, const int8_t* A, const int8_t* B,
                               int32_t* C, int tile_n, void* stream) {
  try {
    lbgemm_status st = check_gemm_args(8, M, N, K, A, B, C);
    if (st != LBGEMM_OK) return st;
    if (tile_n != 64 && tile_n != 128 && tile_n != 256)
      return fail(LBGEMM_ERR_INVALID_ARG, "tile_n must be 64, 128 or 256 (got %d)", tile_n);
    if (K % 16) return fail(LBGEMM_ERR_ALIGNMENT, "the fused kernel needs K %% 16 == 0");
    if (M == 0 || N == 0) return LBGEMM_OK;
    DeviceState* d = nullptr;
    st = device_state(&d);
    if (st != LBGEMM_OK) return st;
    const bool large_b = N >= M;
    std::lock_guard<std::mutex> lock(g_ws_mu);
    void* scratch = nullptr;
    st = scratch_acquire(d->ws, enc_bytes(8, large_b ? M : N, K), as_stream(stream), &scratch);
    if (st != LBGEMM_OK) return st;
    st = run_tc_fused(*d, large_b, tile_n, M, N, K, A, B, C, nullptr, nullptr, nullptr, scratch,
                      as_stream(stream));
    lbgemm_status st2 = scratch_release(d->ws, as_stream(stream), scratch);
    return st != LBGEMM_OK ? st : st2;
  } catch (...) {
    return fail(LBGEMM_ERR_CUDA, "internal error");
  }
}

lbgemm_status lbgemm_run_warpmma(int64_t M, int64_t N, int64_t K, const int8_t* A,
                                 const int8_t* B, int32_t* C, void* stream) {
  try {
    lbgemm_status st = check_gemm_args(8, M, N, K, A, B, C);
    if (st != LBGEMM_OK) return st;
    if (std::min(M, N) > kWarpMmaMaxSideSmall)
      return fail(LBGEMM_ERR_INVALID_ARG, "the warp-MMA kernel needs min(M, N) <= %d",
                  (int)kWarpMmaMaxSideSmall);
    if (K % 16) return fail(LBGEMM_ERR_ALIGNMENT, "the warp-MMA kernel needs K %% 16 == 0");
    if (M == 0 || N == 0) return LBGEMM_OK;
    if (K > lbg::hmma_skinny_max_k((int)std::min(M, N)))
      return fail(LBGEMM_ERR_INVALID_ARG, "the warp-MMA kernel takes K <= %lld here",
                  (long long)lbg::hmma_skinny_max_k((int)std::min(M, N)));
    DeviceState* d = nullptr;
    st = device_state(&d);
    if (st != LBGEMM_OK) return st;
    return run_warpmma(*d, M, N, K, A, B, C, nullptr, nullptr, nullptr, as_stream(stream));
  } catch (...) {
    return fail(LBGEMM_ERR_CUDA, "internal error");
  }
}

lbgemm_status lbgemm_run_popc(int64_t M, int64_t N, int64_t K, const uint32_t* A,
                              const uint32_t* B, int32_t* C, int variant, void* stream) {
  try {
    lbgemm_status st = check_gemm_args(1, M, N, K, A, B, C);
    if (st != LBGEMM_OK) return st;
    if (variant < -1 || variant >= kNumVariants)
      return fail(LBGEMM_ERR_INVALID_ARG, "variant %d out of range", variant);
    if (M == 0 || N == 0) return LBGEMM_OK;
    DeviceState* d = nullptr;
    st = device_state(&d);
    if (st != LBGEMM_OK) return st;
    if (variant < 0) variant = kDefaultVariant;
    cudaError_t e = lbg::launch_b1_popc(variant / 3, variant % 3 + 2, A, B, M, N, K, C,
                                        as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, "1-bit popcount GEMM launch");
    g_launches += 1;
    return LBGEMM_OK;
  } catch (...) {
    return fail(LBGEMM_ERR_CUDA, "internal error");
  }
}

size_t lbgemm_workspace_size(int bits, int64_t M, int64_t N, int64_t K) {
  if ((bits != 8 && bits != 4 && bits != 1) || M <= 0 || N <= 0 || K <= 0) return 0;
  if (bits == 1 && K % 32) return 0;
  return enc_bytes(bits, M, K) + enc_bytes(bits, N, K);
}

lbgemm_status lbgemm_run_ws(int bits, int64_t M, int64_t N, int64_t K, const void* A,
                            const void* B, int32_t* C, int variant, void* workspace,
                            size_t workspace_bytes, void* stream) {
  try {
    return run_any(bits, M, N, K, A, B, C, variant, workspace, workspace_bytes, false,
                   as_stream(stream));
  } catch (...) {
    return fail(LBGEMM_ERR_CUDA, "internal error");
  }
}

lbgemm_status lbgemm_quantize_rows(int64_t M, int64_t K, const void* X, int8_t* Q, float* S,
                                   void* stream) {
  try {
    if (M < 0 || K < 1) return fail(LBGEMM_ERR_INVALID_ARG, "quantize: M >= 0 and K >= 1");
    if (M == 0) return LBGEMM_OK;
    if (!X || !Q || !S) return fail(LBGEMM_ERR_INVALID_ARG, "quantize: null pointer");
    DeviceState* d = nullptr;
    lbgemm_status st = device_state(&d);
    if (st != LBGEMM_OK) return st;
    cudaError_t e = lbg::launch_quant_rows_bf16(X, M, K, Q, S, as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
    g_launches += 1;
    return LBGEMM_OK;
  } catch (...) {
    return fail(LBGEMM_ERR_CUDA, "internal error");
  }
}

lbgemm_status lbgemm_linear_quant(int64_t M, int64_t N, int64_t K, const void* X, const int8_t* W,
                                  const float* sw, void* Y, void* stream) {
  try {
    lbgemm_status st = check_gemm_args(8, M, N, K, X, W, Y);
    if (st != LBGEMM_OK) return st;
    if (M == 0 || N == 0) return LBGEMM_OK;
    if (!sw) return fail(LBGEMM_ERR_INVALID_ARG, "null scale pointer");
    DeviceState* d = nullptr;
    st = device_state(&d);
    if (st != LBGEMM_OK) return st;
    cudaStream_t s = as_stream(stream);
    static std::mutex quant_mu;
    std::lock_guard<std::mutex> lock(quant_mu);
    const size_t qbytes = (size_t)round_up(M * K, 256);
    void* scratch = nullptr;
    st = scratch_acquire(d->quant, qbytes + (size_t)M * sizeof(float), s, &scratch);
    if (st != LBGEMM_OK) return st;
    int8_t* Q = static_cast<int8_t*>(scratch);
    float* S = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + qbytes);
    cudaError_t e = lbg::launch_quant_rows_bf16(X, M, K, Q, S, s);
    if (e != cudaSuccess) {
      scratch_release(d->quant, s, scratch);
      return cuda_fail(e, "quantize launch");
    }
    g_launches += 1;
    // W is the caller's, not written by the quantiser launched just before
    st = run_linear(M, N, K, Q, S, W, sw, Y, -1, s, -1, 0, true);
    lbgemm_status st2 = scratch_release(d->quant, s, scratch);
    return st != LBGEMM_OK ? st : st2;
  } catch (...) {
    return fail(LBGEMM_ERR_CUDA, "internal error");
  }
}

size_t lbgemm_encoded_size(int bits, int64_t rows, int64_t K) {
  if ((bits != 8 && bits != 4 && bits != 1) || rows <= 0 || K <= 0) return 0;
  return enc_bytes(bits, rows, K);
}

lbgemm_status lbgemm_encode(int bits, int64_t rows, int64_t K, const void* src, void* dst,
                            void* stream) {
  try {
    if (bits != 8 && bits != 4 && bits != 1)
      return fail(LBGEMM_ERR_INVALID_ARG, "encode: bits must be 8, 4 or 1");
    lbgemm_status st = check_gemm_args(bits, rows, 1, K, src, dst, dst);
    if (st != LBGEMM_OK || rows == 0) return st;
    DeviceState* d = nullptr;
    st = device_state(&d);
    if (st != LBGEMM_OK) return st;
    return encode_operands(*d, bits, src, rows, dst, nullptr, 0, nullptr, K, as_stream(stream));
  } catch (...) {
    return fail(LBGEMM_ERR_CUDA, "internal error");
  }
}

lbgemm_status lbgemm_run_encoded(int bits, int64_t M, int64_t N, int64_t K, const void* A_enc,
                                 const void* B_enc, int32_t* C, int variant, void* stream) {
  try {
    if (bits != 8 && bits != 4 && bits != 1)
      return fail(LBGEMM_ERR_INVALID_ARG, "bits must be 8, 4 or 1");
    lbgemm_status st = check_gemm_args(bits, M, N, K, A_enc, B_enc, C);
    if (st != LBGEMM_OK) return st;
    if (variant < -1 || variant >= kNumVariants)
      return fail(LBGEMM_ERR_INVALID_ARG, "variant %d out of range", variant);
    if (M == 0 || N == 0) return LBGEMM_OK;
    DeviceState* d = nullptr;
    st = device_state(&d);
    if (st != LBGEMM_OK) return st;
    if (variant < 0) variant = table_select(d->sm_count, bits, M, N, K);
    return run_tc_encoded(*d, bits, M, N, K, A_enc, B_enc, C, nullptr, nullptr, nullptr,
                          spec_of(variant),
                          false, nullptr, as_stream(stream));
  } catch (...) {
    return fail(LBGEMM_ERR_CUDA, "internal error");
  }
}

lbgemm_status lbgemm_linear(int64_t M, int64_t N, int64_t K, const int8_t* X, const float* sx,
                            const int8_t* W, const float* sw, void* Y, void* stream) {
  try {
    return run_linear(M, N, K, X, sx, W, sw, Y, -1, as_stream(stream));
  } catch (...) {
    return fail(LBGEMM_ERR_CUDA, "internal error");
  }
}

lbgemm_status lbgemm_linear_variant(int64_t M, int64_t N, int64_t K, const int8_t* X,
                                    const float* sx, const int8_t* W, const float* sw, void* Y,
                                    int variant, void* stream) {
  try {
    return run_linear(M, N, K, X, sx, W, sw, Y, variant, as_stream(stream));
  } catch (...) {
    return fail(LBGEMM_ERR_CUDA, "internal error");
  }
}

lbgemm_status lbgemm_linear_candidate(int64_t M, int64_t N, int64_t K, const int8_t* X,
                                      const float* sx, const int8_t* W, const float* sw, void* Y,
                                      int route, int param, void* stream) {
  try {
    if (route < 0) return fail(LBGEMM_ERR_INVALID_ARG, "route %d out of range", route);
    return run_linear(M, N, K, X, sx, W, sw, Y, -1, as_stream(stream), route, param);
  } catch (...) {
    return fail(LBGEMM_ERR_CUDA, "internal error");
  }
}

int lbgemm_route(int bits, int64_t M, int64_t N, int64_t K, int linear, int* tile_n) {
  if ((bits != 8 && bits != 4 && bits != 1) || (linear && bits != 8) || M < 0 || N < 0 || K < 1)
    return -1;
  // the route of 16-byte-aligned operands: any aligned address will do, the
  // rules read only its alignment
  const void* aligned = reinterpret_cast<const void*>(uintptr_t(256));
  int t = 0, f = 0;
  const int r = route_of(bits, M, N, K, aligned, aligned, linear != 0, &t, &f);
  if (tile_n) *tile_n = t;
  return r;
}

int lbgemm_dispatch_for(int sm_count, int bits, int64_t M, int64_t N, int64_t K, int* param) {
  if ((bits != 8 && bits != 4 && bits != 1) || M < 0 || N < 0 || K < 1 || sm_count < 1) return -1;
  const void* aligned = reinterpret_cast<const void*>(uintptr_t(256));
  const Pick p = pick_route(sm_count, bits, M, N, K, aligned, aligned);
  if (param) *param = p.param;
  return p.route;
}

int lbgemm_candidates(int bits, int64_t M, int64_t N, int64_t K, int* routes, int* params,
                      int max) {
  if ((bits != 8 && bits != 4 && bits != 1) || M < 1 || N < 1 || K < 1 || max < 0) return -1;
  if (max > 0 && (!routes || !params)) return -1;
  return candidate_list(bits, M, N, K, routes, params, max);
}

lbgemm_status lbgemm_run_candidate(int bits, int64_t M, int64_t N, int64_t K, const void* A,
                                   const void* B, int32_t* C, int route, int param,
                                   void* stream) {
  try {
    lbgemm_status st = check_gemm_args(bits, M, N, K, A, B, C);
    if (st != LBGEMM_OK) return st;
    if (!route_runs(bits, std::max<int64_t>(M, 1), std::max<int64_t>(N, 1), K, A, B, route, param))
      return fail(LBGEMM_ERR_INVALID_ARG, "route %d (param %d) cannot run this problem", route,
                  param);
    if (M == 0 || N == 0) return LBGEMM_OK;
    DeviceState* d = nullptr;
    st = device_state(&d);
    if (st != LBGEMM_OK) return st;
    Pick p;
    p.route = route;
    p.param = param;
    return run_route(*d, bits, M, N, K, A, B, C, p, nullptr, 0, true, as_stream(stream));
  } catch (...) {
    return fail(LBGEMM_ERR_CUDA, "internal error");
  }
}

lbgemm_status lbgemm_run_tile(int bits, int64_t M, int64_t N, int64_t K, const void* A,
                              const void* B, int32_t* C, int tile, int stages, void* stream) {
  try {
    lbgemm_status st = check_gemm_args(bits, M, N, K, A, B, C);
    if (st != LBGEMM_OK) return st;
    if (tile < 0 || tile > 2 || stages < 2 || stages > (tile == 2 ? 6 : 4))
      return fail(LBGEMM_ERR_UNSUPPORTED, "no tensor-core kernel for tile %d with %d stages", tile,
                  stages);
    if (M == 0 || N == 0) return LBGEMM_OK;
    DeviceState* d = nullptr;
    st = device_state(&d);
    if (st != LBGEMM_OK) return st;
    Pick p;
    p.route = LBGEMM_ROUTE_TABLE;
    p.spec = tile * 8 + stages;
    return run_route(*d, bits, M, N, K, A, B, C, p, nullptr, 0, true, as_stream(stream));
  } catch (...) {
    return fail(LBGEMM_ERR_CUDA, "internal error");
  }
}

int lbgemm_select_for(int sm_count, int bits, int64_t M, int64_t N, int64_t K) {
  if ((bits != 8 && bits != 4 && bits != 1) || M < 1 || N < 1 || K < 1) return -1;
  return table_select(sm_count, bits, M, N, K);
}

int lbgemm_select(int bits, int64_t M, int64_t N, int64_t K) {
  DeviceState* d = nullptr;
  if (device_state(&d) != LBGEMM_OK) return -1;
  return lbgemm_select_for(d->sm_count, bits, M, N, K);
}

lbgemm_status lbgemm_table_set_for(int sm_count, int bits, int64_t M, int64_t N, int64_t K,
                                   int variant) {
  return lbgemm_table_set_choice_for(sm_count, bits, M, N, K, variant, -1, 0);
}

lbgemm_status lbgemm_table_set_choice_for(int sm_count, int bits, int64_t M, int64_t N, int64_t K,
                                          int variant, int route, int param) {
  if ((bits != 8 && bits != 4 && bits != 1) || M < 1 || N < 1 || K < 1 || sm_count < 1 ||
      variant < 0 || variant >= kNumVariants)
    return fail(LBGEMM_ERR_INVALID_ARG, "bad table entry");
  if (route >= 0 && !entry_route_ok(bits, M, N, K, route, param))
    return fail(LBGEMM_ERR_INVALID_ARG, "route %d (param %d) cannot run %d-bit %lldx%lldx%lld",
                route, param, bits, (long long)M, (long long)N, (long long)K);
  ensure_default_table();
  std::lock_guard<std::mutex> lock(g_table_mu);
  Choice c;
  c.variant = variant;
  c.route = route >= 0 ? route : -1;
  c.param = route >= 0 ? param : 0;
  g_table[Key{sm_count, bits, M, N, K}] = c;
  return LBGEMM_OK;
}

int lbgemm_table_get_for(int sm_count, int bits, int64_t M, int64_t N, int64_t K, int* variant,
                         int* route, int* param) {
  if ((bits != 8 && bits != 4 && bits != 1) || M < 1 || N < 1 || K < 1 || sm_count < 1) return -1;
  Choice c;
  if (!table_exact(sm_count, bits, M, N, K, &c)) return 0;
  if (variant) *variant = c.variant;
  if (route) *route = c.route;
  if (param) *param = c.param;
  return 1;
}

lbgemm_status lbgemm_table_set(int bits, int64_t M, int64_t N, int64_t K, int variant) {
  DeviceState* d = nullptr;
  lbgemm_status st = device_state(&d);
  if (st != LBGEMM_OK) return st;
  return lbgemm_table_set_for(d->sm_count, bits, M, N, K, variant);
}

lbgemm_status lbgemm_table_clear(void) {
  ensure_default_table();
  std::lock_guard<std::mutex> lock(g_table_mu);
  g_table.clear();
  return LBGEMM_OK;
}

int64_t lbgemm_table_size(void) {
  ensure_default_table();
  std::lock_guard<std::mutex> lock(g_table_mu);
  return (int64_t)g_table.size();
}

const char* lbgemm_table_default_path(void) {
  ensure_default_table();
  return g_table_default_path.c_str();
}

lbgemm_status lbgemm_table_load(const char* path) {
  ensure_default_table();
  return table_load_file(path);
}

lbgemm_status lbgemm_table_save(const char* path) {
  if (!path) return fail(LBGEMM_ERR_INVALID_ARG, "null path");
  ensure_default_table();
  FILE* f = fopen(path, "w");
  if (!f) return fail(LBGEMM_ERR_INVALID_ARG, "cannot write %s", path);
  fprintf(f, "# sm_count bits M N K variant [route param]\n");
  {
    std::lock_guard<std::mutex> lock(g_table_mu);
    for (auto& kv : g_table) {
      fprintf(f, "%d %d %lld %lld %lld %d", std::get<0>(kv.first), std::get<1>(kv.first),
              (long long)std::get<2>(kv.first), (long long)std::get<3>(kv.first),
              (long long)std::get<4>(kv.first), kv.second.variant);
      if (kv.second.route >= 0) fprintf(f, " %d %d", kv.second.route, kv.second.param);
      fprintf(f, "\n");
    }
  }
  const bool ok = fclose(f) == 0;
  return ok ? LBGEMM_OK : fail(LBGEMM_ERR_INVALID_ARG, "cannot write %s", path);
}

int lbgemm_choose_candidate(const float* times, int count, int default_index,
                            float keep_within) {
  if (!times || count < 1 || default_index < 0 || default_index >= count || !(keep_within >= 0))
    return -1;
  int best = 0;
  for (int i = 0; i < count; ++i) {
    if (!(times[i] >= 0)) return -1;  // rejects NaN and negatives
    if (times[i] < times[best]) best = i;
  }
  if (times[default_index] <= times[best] * (1.0f + keep_within)) return default_index;
  return best;
}

int lbgemm_choose(const float* times, int default_variant, float keep_within) {
  return lbgemm_choose_candidate(times, kNumVariants, default_variant, keep_within);
}

lbgemm_status lbgemm_time_candidates(int bits, int64_t M, int64_t N, int64_t K, const void* A,
                                     const void* B, int32_t* C, int count, const int* routes,
                                     const int* params, int warmup, int reps, int flush_l2,
                                     float* times, void* stream) {
  try {
    if (!times || !routes || !params || count < 1 || reps < 1 || warmup < 0)
      return fail(LBGEMM_ERR_INVALID_ARG, "bad timing args");
    lbgemm_status st = check_gemm_args(bits, M, N, K, A, B, C);
    if (st != LBGEMM_OK) return st;
    if (M == 0 || N == 0) return fail(LBGEMM_ERR_INVALID_ARG, "nothing to time (M or N is 0)");
    for (int c = 0; c < count; ++c)
      if (!route_runs(bits, M, N, K, A, B, routes[c], params[c]))
        return fail(LBGEMM_ERR_INVALID_ARG, "candidate %d (route %d, param %d) cannot run this "
                    "problem", c, routes[c], params[c]);
    cudaStream_t s = as_stream(stream);
    DeviceState* d = nullptr;
    st = device_state(&d);
    if (st != LBGEMM_OK) return st;
    void* flush_buf = nullptr;
    if (flush_l2) {
      std::lock_guard<std::mutex> lock(g_mu);
      st = scratch_acquire(d->flush, kFlushBytes, s, &flush_buf);
      if (st != LBGEMM_OK) return st;
    }
    auto run = [&](int c) {
      Pick p;
      p.route = routes[c];
      p.param = params[c];
      return run_route(*d, bits, M, N, K, A, B, C, p, nullptr, 0, true, s);
    };
    for (int c = 0; c < count && st == LBGEMM_OK; ++c)
      for (int w = 0; w < warmup && st == LBGEMM_OK; ++w) st = run(c);
    if (st != LBGEMM_OK) return st;
    // one event pair per candidate, reused every round; each round runs every
    // candidate once (interleaved, so a drift of the clocks touches them all
    // alike) and is read back before the next
    std::vector<cudaEvent_t> ev(2 * (size_t)count, nullptr);
    cudaError_t e = cudaSuccess;
    for (auto& x : ev)
      if (e == cudaSuccess) e = cudaEventCreate(&x);
    std::vector<std::vector<float>> samples(count, std::vector<float>(reps));
    for (int r = 0; r < reps && e == cudaSuccess && st == LBGEMM_OK; ++r) {
      for (int c = 0; c < count && e == cudaSuccess && st == LBGEMM_OK; ++c) {
        if (flush_l2) e = cudaMemsetAsync(flush_buf, r & 0xFF, kFlushBytes, s);
        if (e == cudaSuccess) e = cudaEventRecord(ev[2 * c], s);
        if (e == cudaSuccess) st = run(c);
        if (e == cudaSuccess && st == LBGEMM_OK) e = cudaEventRecord(ev[2 * c + 1], s);
      }
      if (e == cudaSuccess && st == LBGEMM_OK) e = cudaEventSynchronize(ev[2 * count - 1]);
      for (int c = 0; c < count && e == cudaSuccess && st == LBGEMM_OK; ++c)
        e = cudaEventElapsedTime(&samples[c][r], ev[2 * c], ev[2 * c + 1]);
    }
    for (auto& x : ev)
      if (x) cudaEventDestroy(x);
    if (e != cudaSuccess) return cuda_fail(e, "timing");
    if (st != LBGEMM_OK) return st;
    if (flush_l2) {
      std::lock_guard<std::mutex> lock(g_mu);
      st = scratch_release(d->flush, s, flush_buf);
      if (st != LBGEMM_OK) return st;
    }
    for (int c = 0; c < count; ++c) {
      std::sort(samples[c].begin(), samples[c].end());
      times[c] = reps % 2 ? samples[c][reps / 2]
                          : 0.5f * (samples[c][reps / 2 - 1] + samples[c][reps / 2]);
    }
    return LBGEMM_OK;
  } catch (...) {
    return fail(LBGEMM_ERR_CUDA, "internal error");
  }
}

lbgemm_status lbgemm_time_variants(int bits, int64_t M, int64_t N, int64_t K, const void* A,
                                   const void* B, int32_t* C, int warmup, int reps, int flush_l2,
                                   float* times, void* stream) {
  int routes[kNumVariants], params[kNumVariants];
  for (int v = 0; v < kNumVariants; ++v) {
    routes[v] = LBGEMM_ROUTE_TABLE;
    params[v] = v;
  }
  return lbgemm_time_candidates(bits, M, N, K, A, B, C, kNumVariants, routes, params, warmup,
                                reps, flush_l2, times, stream);
}

// Blocks of a host-buffer call: the larger of M and N is cut into blocks of
// whole 256-row (or 256-column) pieces; the other operand goes in whole
// first, then each block's slice of the cut operand is copied in, its GEMM
// runs, and its part of C is copied out, the copies in and out on copy
// streams of their own so that they overlap each other and the GEMMs.  A
// block carries about kHostBlockBytes of copies; small problems run as one.
constexpr int64_t kHostBlockBytes = int64_t(8) << 20;
constexpr int kHostMaxBlocks = 16;

lbgemm_status host_streams(DeviceState& d) {
  if (d.copy_in) return LBGEMM_OK;
  cudaError_t e = cudaStreamCreateWithFlags(&d.copy_in, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&d.copy_out, cudaStreamNonBlocking);
  for (int i = 0; e == cudaSuccess && i < 2 * kHostMaxBlocks + 3; ++i) {
    cudaEvent_t ev = nullptr;
    e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e == cudaSuccess) d.host_events.push_back(ev);
  }
  return e == cudaSuccess ? LBGEMM_OK : cuda_fail(e, "copy streams for lbgemm_run_host");
}

lbgemm_status lbgemm_run_host(int bits, int64_t M, int64_t N, int64_t K, const void* A_host,
                              const void* B_host, int32_t* C_host, int variant, void* stream) {
  try {
    lbgemm_status st = check_gemm_args(bits, M, N, K, A_host, B_host, C_host);
    if (st != LBGEMM_OK) return st;
    if (M == 0 || N == 0) return LBGEMM_OK;
    DeviceState* d = nullptr;
    st = device_state(&d);
    if (st != LBGEMM_OK) return st;
    cudaStream_t s = as_stream(stream);
    const int64_t row_bytes = bits == 8 ? K : bits == 4 ? K / 2 : K / 8;
    const size_t a_bytes = (size_t)round_up(M * row_bytes, 256);
    const size_t b_bytes = (size_t)round_up(N * row_bytes, 256);
    const size_t c_bytes = (size_t)(M * N * 4);
    static std::mutex host_mu;
    std::lock_guard<std::mutex> lock(host_mu);
    st = host_streams(*d);
    if (st != LBGEMM_OK) return st;
    void* stage = nullptr;
    st = scratch_acquire(d->host_stage, a_bytes + b_bytes + round_up(c_bytes, 256), s, &stage);
    if (st != LBGEMM_OK) return st;
    uint8_t* dA = static_cast<uint8_t*>(stage);
    uint8_t* dB = dA + a_bytes;
    int32_t* dC = reinterpret_cast<int32_t*>(dB + b_bytes);
    // Cut M (rows of A and C) or N (rows of B, columns of C): the operand
    // copied in whole waits for nothing to overlap it, the copies out overlap
    // the blocks' copies in.  Column blocks of C leave by 2-D copies, which
    // keep near full speed while C spans at most 256 MB of host memory and
    // drop to ~0.6 of it beyond (measured); so columns only where that fits
    // and the estimate of copy time favours them, or ties with N > M (the
    // blocks' GEMMs then overlap the copy of the larger operand).
    const double c_out = 4.0 * (double)M * (double)N;
    const double t_rows = (double)(N * row_bytes) + std::max((double)(M * row_bytes), c_out);
    const double t_cols = (double)(M * row_bytes) + std::max((double)(N * row_bytes), 1.15 * c_out);
    const bool by_rows =
        c_out > double(int64_t(256) << 20) || t_cols > t_rows || (t_cols == t_rows && M >= N);
    const int64_t cut = by_rows ? M : N, other = by_rows ? N : M;
    const int64_t piped = cut * (row_bytes + 4 * other);  // bytes the blocks copy
    int64_t nb = std::min<int64_t>((piped + kHostBlockBytes - 1) / kHostBlockBytes, kHostMaxBlocks);
    const int64_t rows = round_up((cut + nb - 1) / nb, 256);
    nb = (cut + rows - 1) / rows;
    if (nb == 1) {  // small: everything in order on the caller's stream
      cudaError_t e =
          cudaMemcpyAsync(dA, A_host, (size_t)(M * row_bytes), cudaMemcpyHostToDevice, s);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(dB, B_host, (size_t)(N * row_bytes), cudaMemcpyHostToDevice, s);
      if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy");
      st = run_any(bits, M, N, K, dA, dB, dC, variant, nullptr, 0, true, s);
      if (st != LBGEMM_OK) return st;
      e = cudaMemcpyAsync(C_host, dC, c_bytes, cudaMemcpyDeviceToHost, s);
      if (e != cudaSuccess) return cuda_fail(e, "device-to-host copy");
      st = scratch_release(d->host_stage, s, stage);
      if (st != LBGEMM_OK) return st;
      e = cudaStreamSynchronize(s);
      return e == cudaSuccess ? LBGEMM_OK : cuda_fail(e, "cudaStreamSynchronize");
    }
    cudaEvent_t* ev = d->host_events.data();  // [0] start, [1] whole operand in,
    // block i in at [2 + i], its GEMM done at [2 + kHostMaxBlocks + i], [last] all out
    cudaEvent_t ev_start = ev[0], ev_whole = ev[1], ev_out = ev[2 + 2 * kHostMaxBlocks];
    const uint8_t* cut_host = static_cast<const uint8_t*>(by_rows ? A_host : B_host);
    uint8_t* cut_dev = by_rows ? dA : dB;
    // the copies start after the caller's earlier work on `s` (the staging
    // buffer's previous user included)
    cudaError_t e = cudaEventRecord(ev_start, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(d->copy_in, ev_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(d->copy_out, ev_start, 0);
    if (e == cudaSuccess)
      e = by_rows ? cudaMemcpyAsync(dB, B_host, (size_t)(N * row_bytes), cudaMemcpyHostToDevice,
                                    d->copy_in)
                  : cudaMemcpyAsync(dA, A_host, (size_t)(M * row_bytes), cudaMemcpyHostToDevice,
                                    d->copy_in);
    if (e == cudaSuccess) e = cudaEventRecord(ev_whole, d->copy_in);
    for (int64_t i = 0; e == cudaSuccess && i < nb; ++i) {
      const int64_t r0 = i * rows, r = std::min(rows, cut - r0);
      e = cudaMemcpyAsync(cut_dev + r0 * row_bytes, cut_host + r0 * row_bytes,
                          (size_t)(r * row_bytes), cudaMemcpyHostToDevice, d->copy_in);
      if (e == cudaSuccess) e = cudaEventRecord(ev[2 + i], d->copy_in);
    }
    if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy");
    e = cudaStreamWaitEvent(s, ev_whole, 0);
    for (int64_t i = 0; e == cudaSuccess && i < nb; ++i) {
      const int64_t r0 = i * rows, r = std::min(rows, cut - r0);
      e = cudaStreamWaitEvent(s, ev[2 + i], 0);
      if (e != cudaSuccess) break;
      // a column block's C (M x r) is dense on the device at dC + r0 * M
      st = by_rows ? run_any(bits, r, N, K, dA + r0 * row_bytes, dB, dC + r0 * N, variant,
                             nullptr, 0, true, s)
                   : run_any(bits, M, r, K, dA, dB + r0 * row_bytes, dC + r0 * M, variant,
                             nullptr, 0, true, s);
      if (st != LBGEMM_OK) return st;
      e = cudaEventRecord(ev[2 + kHostMaxBlocks + i], s);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(d->copy_out, ev[2 + kHostMaxBlocks + i], 0);
      if (e != cudaSuccess) break;
      e = by_rows ? cudaMemcpyAsync(C_host + r0 * N, dC + r0 * N, (size_t)(r * N * 4),
                                    cudaMemcpyDeviceToHost, d->copy_out)
                  : cudaMemcpy2DAsync(C_host + r0, (size_t)(N * 4), dC + r0 * M, (size_t)(r * 4),
                                      (size_t)(r * 4), (size_t)M, cudaMemcpyDeviceToHost,
                                      d->copy_out);
    }
    if (e == cudaSuccess) e = cudaEventRecord(ev_out, d->copy_out);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ev_out, 0);
    if (e != cudaSuccess) return cuda_fail(e, "pipelined host copies");
    st = scratch_release(d->host_stage, s, stage);
    if (st != LBGEMM_OK) return st;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    return LBGEMM_OK;
  } catch (...) {
    return fail(LBGEMM_ERR_CUDA, "internal error");
  }
}

lbgemm_status lbgemm_set_exact_chunk(int bits, int k_elems) {
  if (bits == 8) {
    if (k_elems < 64 || k_elems > 1024 || k_elems % 64)
      return fail(LBGEMM_ERR_INVALID_ARG, "8-bit chunk must be a multiple of 64 in [64, 1024]");
    g_chunk_s8 = k_elems;
    return LBGEMM_OK;
  }
  if (bits == 4) {
    if (k_elems < 128 || k_elems > 262144 || k_elems % 128)
      return fail(LBGEMM_ERR_INVALID_ARG, "4-bit chunk must be a multiple of 128 in [128, 262144]");
    g_chunk_s4 = k_elems;
    return LBGEMM_OK;
  }
  if (bits == 1) {
    if (k_elems < 128 || k_elems > (1 << 24) || k_elems % 128)
      return fail(LBGEMM_ERR_INVALID_ARG, "1-bit chunk must be a multiple of 128 in [128, 2^24]");
    g_chunk_b1 = k_elems;
    return LBGEMM_OK;
  }
  return fail(LBGEMM_ERR_INVALID_ARG, "bits must be 8, 4 or 1");
}

lbgemm_status lbgemm_set_fused_slice(int k_elems) {
  if (k_elems != 0 && k_elems != 128 && k_elems != 256)
    return fail(LBGEMM_ERR_INVALID_ARG, "the fused slice must be 0, 128 or 256 (got %d)", k_elems);
  g_fused_slice = k_elems;
  return LBGEMM_OK;
}

int lbgemm_get_fused_slice(void) { return g_fused_slice.load(); }

lbgemm_status lbgemm_fused_schedule(int64_t M, int64_t N, int64_t K, int tile_n, int linear,
                                    int sm_count, int* splits, int* stream_pieces) {
  if ((tile_n != 64 && tile_n != 128) || M < 1 || N < 1 || K < 1 || sm_count < 1 ||
      (linear && M > N))
    return fail(LBGEMM_ERR_INVALID_ARG, "bad fused-schedule query");
  const bool large_b = linear || N >= M;
  FusedSchedule fs;
  if (linear || large_b || N % 4 == 0)
    fs = fused_schedule(large_b ? N : M, large_b ? M : N, K, tile_n,
                        fused_slice(tile_n, linear != 0), linear != 0, sm_count,
                        g_stream_k.load() != 0);
  if (splits) *splits = fs.splits;
  if (stream_pieces) *stream_pieces = fs.stream_pieces;
  return LBGEMM_OK;
}

lbgemm_status lbgemm_set_fused_stream_k(int mode) {
  if (mode < 0 || mode > 1)
    return fail(LBGEMM_ERR_INVALID_ARG, "the stream-K mode must be 0 or 1 (got %d)", mode);
  g_stream_k = mode;
  return LBGEMM_OK;
}

int lbgemm_get_fused_stream_k(void) { return g_stream_k.load(); }

lbgemm_status lbgemm_set_tail_split(int mode) {
  if (mode < 0 || mode > 2) return fail(LBGEMM_ERR_INVALID_ARG, "tail split mode must be 0, 1 or 2");
  g_tail_split = mode;
  return LBGEMM_OK;
}

int lbgemm_get_tail_split(void) { return g_tail_split.load(); }

int lbgemm_get_exact_chunk(int bits) {
  return bits == 8 ? g_chunk_s8.load()
         : bits == 4 ? g_chunk_s4.load()
         : bits == 1 ? g_chunk_b1.load()
                     : -1;
}

lbgemm_status lbgemm_device_status(void* stream) {
  DeviceState* d = nullptr;
  lbgemm_status st = device_state(&d);
  if (st != LBGEMM_OK) return st;
  cudaError_t e = cudaStreamSynchronize(as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int word = 0;
  e = cudaMemcpy(&word, d->status, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
  if (word != 0) {
    const int zero = 0;
    cudaMemcpy(d->status, &zero, sizeof zero, cudaMemcpyHostToDevice);
    return fail(LBGEMM_ERR_TIMEOUT, "a device-side wait ran out of time (status %d)", word);
  }
  return LBGEMM_OK;
}

lbgemm_status lbgemm_selftest_timeout(void* stream) {
  DeviceState* d = nullptr;
  lbgemm_status st = device_state(&d);
  if (st != LBGEMM_OK) return st;
  cudaError_t e = lbg::launch_wait_selftest(d->status, 100000000ull, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  g_launches += 1;
  return LBGEMM_OK;
}

const char* lbgemm_last_error(void) { return t_last_error.c_str(); }

}  // extern "C"

// Lets other translation units of the library report a failure through
// lbgemm_last_error().
namespace lbg {
lbgemm_status report_error(lbgemm_status st, const char* message) {
  return fail(st, "%s", message);
}

void ensure_defaults() { ensure_default_table(); }

// Scratch bytes that lbgemm_run_ws(bits, M, N, K, A, B, C, variant, ...)
// needs: the route the dispatch takes (variant < 0) or the tensor-core
// variant's.  Argument errors are reported as that call reports them.
lbgemm_status scratch_for_call(int bits, int64_t M, int64_t N, int64_t K, const void* A,
                               const void* B, const void* C, int variant, size_t* bytes) {
  *bytes = 0;
  lbgemm_status st = check_gemm_args(bits, M, N, K, A, B, C);
  if (st != LBGEMM_OK) return st;
  if (variant < -1 || variant >= kNumVariants)
    return fail(LBGEMM_ERR_INVALID_ARG, "variant %d out of range", variant);
  if (M == 0 || N == 0) return LBGEMM_OK;
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != LBGEMM_OK) return st;
  Pick p;
  if (variant < 0) {
    p = pick_route(d->sm_count, bits, M, N, K, A, B);
  } else {
    p.route = LBGEMM_ROUTE_TABLE;
    p.param = variant;
  }
  *bytes = route_scratch(bits, M, N, K, p);
  return LBGEMM_OK;
}
}  // namespace lbg

extern "C" {

int64_t lbgemm_launch_count(void) { return g_launches.load(); }

}  // extern "C"
