/*
 * lbgemm.h -- C ABI of the low-bit integer GEMM library for GB300 (sm_103a).
 *
 * Method source, cited below as [LBG]: "Leveraging Large-Scale Data for
 * Efficient Low-Bit CUTLASS GEMM Optimization via Neural Networks", IEEE
 * Transactions on Big Data (press summary page).
 *   intro      : GEMM on 1-, 4- and 8-bit operands; a selector picks the
 *                kernel template per (M, N, K, SM count) at run time.
 *   section 1  : C = A x B is split into uniform thread-block tiles, each
 *                looping over K; tile shape and pipeline stage count are the
 *                two tuning parameters.
 *   section 2  : nine templates = {small, medium, large} tile x {2, 3, 4}
 *                stages; each sample is labelled with its fastest template.
 *   section 4  : the selected template is compared with a default template,
 *                for a GEMM and for a linear layer.
 *
 * Conventions shared by every entry point
 *   - Operands: A is M x K, B is N x K, both K-major with dense rows;
 *     C[m][n] = sum_k A[m][k] * B[n][k] (C = A . B^T), C is M x N row-major
 *     int32.  K counts logical elements (bits when bits == 1).
 *   - Element formats by `bits`:
 *       8 : int8, rows of K bytes, full range [-128, 127].
 *       4 : signed nibbles, two per byte, element 2j in the low nibble of
 *           byte j; rows of K/2 bytes; value = (nibble ^ 8) - 8.
 *       1 : +-1 values, 32 per uint32 word, element k = bit k%32 of word
 *           k/32, bit 1 = +1, bit 0 = -1; rows of K/32 words;
 *           C[m][n] = K - 2 * popcount(A[m] XOR B[n]).
 *   - Pointers: A, B, C (and X, W, sx, sw, Y, workspace) are DEVICE pointers
 *     of the current CUDA device, owned by the caller, 16-byte aligned.  The
 *     library keeps no reference to them after the call returns.
 *   - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *     stream.  Every compute call is asynchronous on that stream.
 *   - Errors: argument errors are detected on the host and returned before
 *     anything is launched.  A launch failure returns LBGEMM_ERR_CUDA.  A
 *     device-side wait that exceeds its time limit (about 2 s) makes the
 *     kernel stop and sets a device status word that lbgemm_device_status()
 *     reports.  lbgemm_last_error() gives a message for the last failure on
 *     the calling thread.
 *   - Shape limits: M, N >= 0 (0 is a no-op), K >= 1; the result must fit
 *     int32: K <= 131071 for bits 8, K <= 2^25 - 1 for bits 4, K < 2^31 for
 *     bits 1.  Alignment: K % 2 == 0 for bits 4 and K % 32 == 0 for bits 1
 *     (rows must hold whole bytes / words); any K for bits 8.
 */
#ifndef LBGEMM_H
#define LBGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LBGEMM_OK = 0,
  LBGEMM_ERR_INVALID_ARG = 1, /* null pointer, bad bits, negative size, K out of range  */
  LBGEMM_ERR_ALIGNMENT = 2,   /* K not a whole number of bytes/words, pointer not 16-B aligned */
  LBGEMM_ERR_UNSUPPORTED = 3, /* no sm_103a device current, or variant not available     */
  LBGEMM_ERR_CUDA = 4,        /* a CUDA runtime or driver call failed                      */
  LBGEMM_ERR_TIMEOUT = 5,     /* a device-side wait ran out (reported by lbgemm_device_status) */
  LBGEMM_ERR_WORKSPACE = 6    /* caller-supplied workspace smaller than lbgemm_workspace_size */
} lbgemm_status;

/* Number of tile x stage variants (9) and the index of the default one.
 * Variant v has tile class v / 3 (0 small, 1 medium, 2 large) and stage level
 * v % 3.  [LBG] section 2 names three stage counts (2, 3, 4); here the levels
 * are 2, 3, 4 stages for the small (128 x 64) and medium (128 x 128) tiles and
 * 4, 5, 6 stages for the large tile (256 x 256, computed by a pair of CTAs).
 * The default (large tile, middle level = 7) is this library's reading of
 * the unnamed "default template" of section 4. */
int lbgemm_num_variants(void);
int lbgemm_default_variant(void);

/* Tile shape and stage count of variant v of the tensor-core kernel for
 * operands of `bits` (tile_m x tile_n output tile, tile_k logical elements
 * per pipeline stage: 64 for bits 8, 128 for bits 4 and 1).
 * Returns LBGEMM_ERR_INVALID_ARG for an unknown v or bits. */
lbgemm_status lbgemm_variant_info(int bits, int variant, int* tile_m, int* tile_n, int* tile_k,
                                  int* stages);

/* C = A . B^T with the variant the selection table picks for
 * (bits, M, N, K, SM count).  [LBG] intro, sections 1-2.  Every bit width
 * runs on the tensor cores through an exact re-encoding of its operands
 * (int8 -> fp16, int4 -> e4m3, +-1 -> e4m3), except these shape rules, in
 * order (the 8-bit ones need K % 16 == 0 and 16-byte-aligned operands):
 * 8-bit problems with M <= 4 run on a dp4a kernel that streams B once;
 * 8-bit problems with min(M, N) <= 16, max(M, N) >= 1024 and K <= 4096 on
 * a warp-level fp16 MMA kernel that streams the large operand once through a
 * bulk-copy ring (LBGEMM_ROUTE_STREAM);
 * 8-bit problems with min(M, N) <= 32 (and K within the limit of
 * lbgemm_run_warpmma) on the warp-level fp16 MMA kernel, which streams the
 * large operand once; small 8-bit problems with min(M, N) <= 256,
 * 256 < K <= 2048 and either M*N <= 2^19 (2^18 with K > 1024) or
 * (K <= 512 and M*N*K <= 2^28) on
 * the warp-level fp16 MMA kernel too (each 32 rows of the small side re-read
 * the large one); 8-bit problems with K <= 512 and M*N*K <= 2^28 on a
 * one-launch dp4a kernel; 8-bit problems with min(M, N) <= 512,
 * max(M, N) >= 1024, K >= 512 and one of max(M, N) >= 4096, K >= 8192,
 * (max(M, N) >= 2048 and K >= 4096) or (min(M, N) <= 256 and K >= 2048),
 * on a tensor-core kernel that converts the large operand itself
 * (lbgemm_run_fused), with only the small one re-encoded ahead; 4-bit
 * problems with K <= 256 (K % 32 == 0) and M*N*K <= 2^26 on the one-launch
 * dp4a kernel over the packed nibbles; and 1-bit problems with M*N*K < 2^27
 * on the XOR-popcount kernel of lbgemm_run_popc (variant 1: 64 x 64 tile, 3
 * stages).  These rules apply to shapes the
 * selection table holds no measured route for; a table entry with a route
 * (lbgemm_table_set_choice_for, or a route column in a loaded table file)
 * runs that kernel instead, whenever it can run the given operands.
 * Scratch memory for the re-encoding is
 * taken from a per-device buffer the library grows with cudaMalloc on demand
 * (by at least half again each time);
 * calls from different streams are ordered on it with events; a call that
 * grows the buffer synchronises the device.  While `stream` is being
 * captured into a CUDA graph, a call takes its scratch from stream-ordered
 * allocations instead (cudaMallocAsync / cudaFreeAsync, which become
 * allocation nodes of the graph): the graph needs no warm-up of the buffer,
 * depends on nothing outside the capture and stays valid when a later call
 * reallocates the buffer.  The library's per-device state must exist before
 * the first capture on a device (any one call made outside capture). */
lbgemm_status lbgemm_run(int bits, int64_t M, int64_t N, int64_t K, const void* A, const void* B,
                         int32_t* C, void* stream);

/* As lbgemm_run, forcing variant v (0..8) of the tensor-core kernel (no shape
 * rule and no table route applies); -1 means "as lbgemm_run". */
lbgemm_status lbgemm_run_variant(int bits, int64_t M, int64_t N, int64_t K, const void* A,
                                 const void* B, int32_t* C, int variant, void* stream);

/* 8-bit C = A . B^T forced onto the kernel that converts one operand from
 * int8 itself and feeds it to the tensor cores from tensor memory; only the
 * other operand is re-encoded ahead (scratch: its fp16 copy, from the same
 * per-device buffer as lbgemm_run).  The larger operand is the converted one
 * (B when N >= M; C is then produced transposed from the accumulator).
 * tile_n (64, 128 or 256) is the tile width along the re-encoded operand.
 * Requires K % 16 == 0 and 16-byte-aligned A and B (LBGEMM_ERR_ALIGNMENT
 * otherwise).  lbgemm_run takes this route by itself for the shapes where it
 * is measured faster; this entry exists for tests and timing.  [LBG]
 * section 1 (tiled GEMM with a multi-stage pipeline). */
lbgemm_status lbgemm_run_fused(int64_t M, int64_t N, int64_t K, const int8_t* A, const int8_t* B,
                               int32_t* C, int tile_n, void* stream);

/* 8-bit C = A . B^T forced onto the warp-level fp16 MMA kernel for problems
 * with a small side: min(M, N) <= 256 rows, and K at most 4224 (small side
 * <= 16) or 2048 (> 16) so that 16 or 32 rows of the small operand fit the
 * kernel's shared memory (LBGEMM_ERR_INVALID_ARG otherwise).
 * Both operands stay int8 in memory and are converted to fp16 in registers;
 * the large side is streamed from HBM once per 32 rows of the small side.
 * No scratch, one launch.
 * Requires K % 16 == 0 and 16-byte-aligned A and B (LBGEMM_ERR_ALIGNMENT).
 * lbgemm_run takes this route by itself for the shapes where it is measured
 * faster; this entry exists for tests and timing.  [LBG] intro (8-bit GEMM),
 * section 4 (linear layers with few tokens). */
lbgemm_status lbgemm_run_warpmma(int64_t M, int64_t N, int64_t K, const int8_t* A,
                                 const int8_t* B, int32_t* C, void* stream);

/* C = A . B^T on one tensor-core kernel named by tile class (0 small
 * 128 x 64, 1 medium 128 x 128, 2 large 256 x 256 on a CTA pair) and stage
 * count: 2..4 for the small and medium tiles, 2..6 for the large one (2 and
 * 3 beyond the variant table's levels, for measurements of the stage
 * dimension).  Re-encoding and scratch as lbgemm_run_variant;
 * LBGEMM_ERR_UNSUPPORTED for a pair the library does not compile.  [LBG]
 * sections 1-2 (tile shape and stage count). */
lbgemm_status lbgemm_run_tile(int bits, int64_t M, int64_t N, int64_t K, const void* A,
                              const void* B, int32_t* C, int tile, int stages, void* stream);

/* Bytes of scratch that lbgemm_run_ws needs for this problem on the
 * tensor-core route (0 for bad arguments): the re-encoded A and B. */
size_t lbgemm_workspace_size(int bits, int64_t M, int64_t N, int64_t K);

/* As lbgemm_run_variant, with caller-owned scratch: `workspace` is a device
 * buffer of at least lbgemm_workspace_size() bytes, 256-byte aligned, not
 * used by any other call in flight.  This entry point allocates nothing. */
lbgemm_status lbgemm_run_ws(int bits, int64_t M, int64_t N, int64_t K, const void* A,
                            const void* B, int32_t* C, int variant, void* workspace,
                            size_t workspace_bytes, void* stream);

/* For callers that cannot allocate GPU memory at all -- code running where
 * cudaMalloc is forbidden or unsafe, such as inside a host callback, a custom
 * allocator's own hooks, or a plugin whose host process owns every device
 * allocation -- and that also cannot hand over a workspace of their own.
 * The paper has no counterpart; this is a convenience of this library.
 *
 * Same result as lbgemm_run_variant / lbgemm_run_ws, but the operand
 * re-encoding scratch is a fixed array of LBGEMM_STATIC_SCRATCH_BYTES (32 MiB)
 * compiled into the library: every GPU that loads the library holds it until
 * the process exits, and this call allocates nothing.  The caller still
 * passes A, B and C.  Problems whose scratch (lbgemm_workspace_size) exceeds
 * the array are rejected with LBGEMM_ERR_WORKSPACE before anything runs.
 * The scratch is that of the kernel the call runs: on the tensor-core route
 * both re-encoded operands (lbgemm_workspace_size: for 8-bit operands
 * (M + N) * round_up(K, 8) * 2 bytes, e.g. M = N = 2048 at K = 4096; for
 * 1-bit operands (M + N) * K bytes); on the in-kernel conversion route the
 * smaller operand's fp16 copy only; none on the routes that read int8 (or
 * 1-bit words) directly, so with variant -1 a linear-layer-shaped 16 x 11008
 * x 4096 product runs whatever its size.
 *
 * The first call on each device looks up the array's device address (with
 * that device current); make that first call before any stream capture.
 * The library caches per-device state (this address among it) for the life
 * of the process: cudaDeviceReset while the library is in use is not
 * supported.
 * Every call shares the one array: calls that can overlap on the GPU (other
 * streams, other threads) race on it and must be ordered by the caller.  The
 * array keeps whatever the last call wrote; each call rewrites every byte its
 * GEMM reads (zero padding included), so nothing stale is read. */
#define LBGEMM_STATIC_SCRATCH_BYTES ((size_t)32 << 20)
lbgemm_status lbgemm_run_static(int bits, int64_t M, int64_t N, int64_t K, const void* A,
                                const void* B, int32_t* C, int variant, void* stream);

/* ---- pre-encoded operands ------------------------------------------------------
 * The tensor-core path first re-encodes each operand exactly (int8 -> fp16,
 * int4 -> e4m3, +-1 -> e4m3 one byte per element; rows padded with zeros to
 * a multiple of 8 halves / 16 bytes).  A caller that reuses an operand (the weights of a
 * linear layer) can encode it once and call lbgemm_run_encoded, which runs
 * the GEMM kernel alone.  The encoded layout is private to this library
 * version: only lbgemm_encode may write it. */
size_t lbgemm_encoded_size(int bits, int64_t rows, int64_t K);
/* dst: device buffer of lbgemm_encoded_size(bits, rows, K) bytes, 16-byte
 * aligned.  src: rows x K operand in the format of `bits` (8, 4 or 1). */
lbgemm_status lbgemm_encode(int bits, int64_t rows, int64_t K, const void* src, void* dst,
                            void* stream);
/* C = A . B^T from encoded operands (variant -1 = table). */
lbgemm_status lbgemm_run_encoded(int bits, int64_t M, int64_t N, int64_t K, const void* A_enc,
                                 const void* B_enc, int32_t* C, int variant, void* stream);

/* The 1-bit product on CUDA cores: C[m][n] = K - 2 * sum_w popc(A[m][w] ^
 * B[n][w]) with XOR and __popc, no re-encoding and no scratch.  [LBG]
 * intro (1-bit GEMM).  A, B: uint32 words, K/32 per row; K % 32 == 0.
 * Variant v picks the CTA tile (v / 3: 0 = 64 x 64, 1 = 128 x 64,
 * 2 = 128 x 128 outputs, 256 threads) and v % 3 + 2 cp.async stages of 32
 * words of K; -1 = variant 7.  Asynchronous on `stream`. */
lbgemm_status lbgemm_run_popc(int64_t M, int64_t N, int64_t K, const uint32_t* A,
                              const uint32_t* B, int32_t* C, int variant, void* stream);

/* Quantised linear layer, [LBG] section 4 (a linear layer on the low-bit
 * GEMM): Y[m][n] = bf16_round_nearest_even( (float)acc[m][n] * sx[m] * sw[n] )
 * with acc = X . W^T exact in int32.  X: int8 M x K (per-token scale sx, fp32
 * [M]); W: int8 N x K (per-output-channel scale sw, fp32 [N]); Y: bf16 M x N
 * row-major, passed as void* (2 bytes per element).  The scale product is
 * formed in fp32, left to right.  K <= 131071.  The shape rules of
 * lbgemm_run apply: M <= 4 (M <= 8 when 4096 < K <= 8192) on the dp4a
 * kernel that streams W once, M <= 16 (N >= 1024, K <= 4096) on the
 * streaming warp-MMA kernel, M <= 32 on the warp-level fp16 MMA kernel,
 * M <= 512 (with N >= 1024 and N, K as lbgemm_run says) on the kernel that
 * converts W itself (64-wide tiles up to 64 tokens, else 128-wide, never
 * the CTA-pair tile; where its tiles would leave most SMs idle or make a fractional number of waves, K is shared out
 * over CTAs (split or stream-K) into int32 sums in library scratch and a
 * second grid scales them into Y), larger M on the tensor-core variant
 * table. */
lbgemm_status lbgemm_linear(int64_t M, int64_t N, int64_t K, const int8_t* X, const float* sx,
                            const int8_t* W, const float* sw, void* Y, void* stream);

/* As lbgemm_linear, forcing variant v (-1 = table). */
lbgemm_status lbgemm_linear_variant(int64_t M, int64_t N, int64_t K, const int8_t* X,
                                    const float* sx, const int8_t* W, const float* sw, void* Y,
                                    int variant, void* stream);

/* As lbgemm_linear, forced onto one kernel: route LBGEMM_ROUTE_TABLE (param =
 * variant), LBGEMM_ROUTE_SKINNY (M <= 16), LBGEMM_ROUTE_STREAM (M <= 16,
 * K <= 4096), LBGEMM_ROUTE_WARPMMA (min(M, N) <= 32) or LBGEMM_ROUTE_FUSED
 * (param = tile width 64, 128 or 256); the 8-bit routes need K % 16 == 0 and
 * 16-byte-aligned X and W.  LBGEMM_ERR_INVALID_ARG if that kernel cannot run
 * the layer.  For tests and timing. */
lbgemm_status lbgemm_linear_candidate(int64_t M, int64_t N, int64_t K, const int8_t* X,
                                      const float* sx, const int8_t* W, const float* sw, void* Y,
                                      int route, int param, void* stream);

/* Per-token (per-row) symmetric int8 quantisation of activations, the step in
 * front of a quantised linear layer ([LBG] section 4 and conclusion: low-bit
 * layers of quantised networks; the page gives no quantiser, this is the
 * plainest one): for each row of X (bf16, M x K row-major),
 *   s[m] = max(max_k |X[m][k]|, 1e-12) / 127                (fp32)
 *   Q[m][k] = clamp(round_half_even(X[m][k] / s[m]), -127, 127)
 * with IEEE fp32 division, so the codes are reproducible bit for bit.
 * Q: int8 M x K, S: fp32 [M]; device pointers owned by the caller. */
lbgemm_status lbgemm_quantize_rows(int64_t M, int64_t K, const void* X, int8_t* Q, float* S,
                                   void* stream);

/* The linear layer on unquantised activations: lbgemm_quantize_rows of X
 * (bf16 M x K) into library scratch, then lbgemm_linear with the resulting
 * codes and per-token scales against W (int8 N x K, scales sw).  Y: bf16 M x N.
 * The scratch (M*K + 4*M bytes) comes from a per-device buffer the library
 * grows with cudaMalloc. */
lbgemm_status lbgemm_linear_quant(int64_t M, int64_t N, int64_t K, const void* X, const int8_t* W,
                                  const float* sw, void* Y, void* stream);

/* ---- selection table: [LBG] sections 2-3 ------------------------------------
 * The table maps (bits, M, N, K) on this device's SM count to a variant.  A
 * shape with no entry takes the learned selector's choice when a network is
 * loaded for its bit width (below), else the entry of the nearest one of the
 * same bits and SM count (distance: sum of |log2| differences of M, N, K;
 * ties to the first in (M, N, K) order); an empty table gives the default. */
int lbgemm_select(int bits, int64_t M, int64_t N, int64_t K);
lbgemm_status lbgemm_table_set(int bits, int64_t M, int64_t N, int64_t K, int variant);
/* The same two for an explicit SM count (no device needed). */
int lbgemm_select_for(int sm_count, int bits, int64_t M, int64_t N, int64_t K);

/* The kernels of the default dispatch. */
typedef enum {
  LBGEMM_ROUTE_TABLE = 0,   /* re-encoding + the variant table's tensor-core kernel */
  LBGEMM_ROUTE_POPC = 1,    /* 1-bit XOR-popcount kernel (lbgemm_run_popc)            */
  LBGEMM_ROUTE_SKINNY = 2,  /* dp4a kernel streaming B once (M <= 4)                 */
  LBGEMM_ROUTE_WARPMMA = 3, /* warp-level fp16 MMA kernel (lbgemm_run_warpmma)        */
  LBGEMM_ROUTE_SMALL = 4,   /* one-launch dp4a kernel (8-bit, or 4-bit nibbles)      */
  LBGEMM_ROUTE_FUSED = 5,   /* in-kernel conversion kernel (lbgemm_run_fused)         */
  LBGEMM_ROUTE_NONE = 6,    /* M == 0 or N == 0: nothing runs                        */
  LBGEMM_ROUTE_STREAM = 7   /* small side <= 16, K <= 4096: warp-level fp16 MMAs on the
                               large operand streamed once through a bulk-copy ring    */
} lbgemm_route_id;

/* The shape rules listed at lbgemm_run: the kernel lbgemm_run (linear = 0)
 * runs for a shape with no measured table route, or lbgemm_linear (linear
 * != 0, bits 8) runs, for 16-byte-aligned operands; with LBGEMM_ROUTE_FUSED,
 * *tile_n (if not null) receives the kernel's tile width (64, 128 or 256),
 * else 0.  The dispatchers use the same function.  Host only; -1 on bad bits
 * or sizes (the alignment rules of K are not checked here). */
int lbgemm_route(int bits, int64_t M, int64_t N, int64_t K, int linear, int* tile_n);

/* The kernel lbgemm_run runs for these sizes (16-byte-aligned operands) on a
 * device with sm_count SMs: the table's measured route for the exact shape
 * if it has one, else lbgemm_route's rule.  *param (if not null) receives
 * the route's parameter: the variant for LBGEMM_ROUTE_TABLE (the table's
 * choice) and LBGEMM_ROUTE_POPC, the tile width for LBGEMM_ROUTE_FUSED, else
 * 0.  Host only; -1 on bad arguments. */
int lbgemm_dispatch_for(int sm_count, int bits, int64_t M, int64_t N, int64_t K, int* param);
lbgemm_status lbgemm_table_set_for(int sm_count, int bits, int64_t M, int64_t N, int64_t K,
                                   int variant);
/* An entry with a measured route as well: variant is the tensor-core label
 * (what lbgemm_select returns), (route, param) the kernel lbgemm_run runs for
 * exactly this shape (param as lbgemm_dispatch_for gives it); route -1 stores
 * no route.  LBGEMM_ERR_INVALID_ARG if that kernel cannot run the shape. */
lbgemm_status lbgemm_table_set_choice_for(int sm_count, int bits, int64_t M, int64_t N, int64_t K,
                                          int variant, int route, int param);
/* The entry for exactly this shape: 1 (and its fields; route -1 when it has
 * no route), 0 if there is none, -1 on bad arguments. */
int lbgemm_table_get_for(int sm_count, int bits, int64_t M, int64_t N, int64_t K, int* variant,
                         int* route, int* param);
lbgemm_status lbgemm_table_clear(void);
int64_t lbgemm_table_size(void);
/* Text file, one entry per line: "sm_count bits M N K variant", optionally
 * followed by "route param"; '#' starts a comment line.  Loading merges the
 * file's entries into the table (none if any line is malformed). */
lbgemm_status lbgemm_table_load(const char* path);
lbgemm_status lbgemm_table_save(const char* path);
/* The table is filled once per process, before its first use, from the file
 * named by the environment variable LBGEMM_TABLE (unset: the GB300 table
 * shipped with the library, data/lbgemm_table_gb300.txt beside its lib/
 * directory; "" or "none": nothing); at the same moment the selector
 * networks shipped there (data/mlp_gb300_s<bits>.txt) are loaded unless
 * LBGEMM_MLP is "" or "none".  The table path loaded, or "" if none. */
const char* lbgemm_table_default_path(void);

/* ---- learned selector: [LBG] section 3 ------------------------------------------
 * A feed-forward network -- inputs log2(M), log2(N), log2(K) and the SM count,
 * standardised; three hidden ReLU layers of 128; nine outputs -- trained
 * offline on sweep timings (bit_tensor_gemm_gb300/selector_mlp.py writes the
 * text file).  Once a nine-class network is loaded for a bit width,
 * lbgemm_select answers shapes that have no table entry with the network's
 * top class (before the nearest-entry rule); a network trained on a single
 * SM count (the file's SM standard deviation is 1) answers for that SM count
 * only.  The network runs on the host in float32.  lbgemm_mlp_load replaces
 * the network of the file's bit width; LBGEMM_ERR_INVALID_ARG for a missing
 * or malformed file.  The shipped GB300 networks load by default (see
 * lbgemm_table_default_path). */
lbgemm_status lbgemm_mlp_load(const char* path);
lbgemm_status lbgemm_mlp_clear(void);
/* Top class of the network loaded for `bits` (and the second one in *second
 * when not NULL), or -1 when none is loaded or the arguments are bad. */
int lbgemm_mlp_predict(int bits, int64_t M, int64_t N, int64_t K, int sm_count, int* second);

/* The stored choice from nine measured times: the fastest variant (lowest
 * index on ties), unless times[default_variant] is within keep_within
 * (relative) of it, in which case the default is kept.  -1 on bad input. */
int lbgemm_choose(const float* times, int default_variant, float keep_within);

/* The same rule over `count` measured candidates (lbgemm_candidates order):
 * the fastest (lowest index on ties), unless times[default_index] is within
 * keep_within of it.  -1 on bad input. */
int lbgemm_choose_candidate(const float* times, int count, int default_index, float keep_within);

/* Timing step of the sweep, [LBG] section 2: runs every variant on the given
 * operands `warmup` times, then `reps` rounds in which each variant runs once
 * (interleaved), each run timed with CUDA events on `stream`, and writes the
 * median milliseconds per variant to times[9].
 * With flush_l2 != 0, a 256 MB library-owned buffer (allocated on first use)
 * is overwritten before each timed run, outside the timed interval, so every
 * run starts with operands out of L2.  Uses the internal workspace like
 * lbgemm_run.  Synchronises `stream`; C holds the product afterwards. */
lbgemm_status lbgemm_time_variants(int bits, int64_t M, int64_t N, int64_t K, const void* A,
                                   const void* B, int32_t* C, int warmup, int reps, int flush_l2,
                                   float* times, void* stream);

/* The candidate kernels the timing sweep measures for a shape, as (route,
 * param) pairs: the nine tensor-core variants (LBGEMM_ROUTE_TABLE, param =
 * variant) first, then each shape-route kernel that runs the problem within
 * the domain where it can plausibly win: for 1-bit below 2^34 bit-MACs the
 * popcount kernel's nine variants (LBGEMM_ROUTE_POPC, param = its variant);
 * for 4-bit with K % 32 == 0, M*N*K <= 2^31 and K <= 8192 the one-launch dp4a
 * kernel on the packed nibbles (LBGEMM_ROUTE_SMALL);
 * for 8-bit with K % 16 == 0 the dp4a kernel streaming B (M <= 16), the
 * warp-level fp16 MMA kernel (small side <= 256 within its K limit), the
 * one-launch dp4a kernel (M*N*K <= 2^31, K <= 4096), and, for a small side
 * of at most 1024 rows, the in-kernel conversion kernel at tile widths 64 and
 * 128 (and 256 once the small side exceeds 64 rows).  Writes up to `max`
 * pairs and returns how many there are (-1 on bad arguments).  Host only. */
int lbgemm_candidates(int bits, int64_t M, int64_t N, int64_t K, int* routes, int* params,
                      int max);

/* C = A . B^T on one candidate kernel (route, param) as lbgemm_candidates
 * lists them (any pair whose kernel runs the problem); scratch as
 * lbgemm_run.  LBGEMM_ERR_INVALID_ARG if that kernel cannot run it. */
lbgemm_status lbgemm_run_candidate(int bits, int64_t M, int64_t N, int64_t K, const void* A,
                                   const void* B, int32_t* C, int route, int param, void* stream);

/* As lbgemm_time_variants, for `count` candidates (routes[i], params[i]):
 * the median milliseconds of each goes to times[i].  An even `reps` takes the
 * mean of the two middle samples. */
lbgemm_status lbgemm_time_candidates(int bits, int64_t M, int64_t N, int64_t K, const void* A,
                                     const void* B, int32_t* C, int count, const int* routes,
                                     const int* params, int warmup, int reps, int flush_l2,
                                     float* times, void* stream);

/* Host-buffer convenience, for callers whose operands live in host memory:
 * copies A and B to device staging buffers that the library owns (grown with
 * cudaMalloc on demand), runs lbgemm_run_variant, copies C back to the host
 * buffer and synchronises `stream`.  Problems that copy more than 8 MB run in
 * blocks (up to 16) of the larger of M and N, each of whole 256-row (or
 * 256-column) pieces: the other operand is copied in whole, then each block's
 * rows of A (or B) on one library-owned stream, its GEMM on `stream`, and its
 * rows (or columns, by a 2-D copy) of C out on another library-owned stream,
 * so the two copy directions and the GEMMs overlap.  Pinned host memory gives
 * the fastest copies.  Not for use under stream capture. */
lbgemm_status lbgemm_run_host(int bits, int64_t M, int64_t N, int64_t K, const void* A_host,
                              const void* B_host, int32_t* C_host, int variant, void* stream);

/* ---- exactness tuning ----------------------------------------------------------
 * The tensor-core path sums fp32 products of exact encodings in chunks of
 * k_elems along K and adds the chunks in int32.  A chunk is exact while
 * k_elems * max|a*b| <= 2^24 (every integer of magnitude <= 2^24 is an fp32
 * value): max|a*b| = 2^14 for bits 8 (k_elems <= 1024), 2^6 for bits 4
 * (k_elems <= 262144) and 1 for bits 1 (k_elems <= 2^24).  Defaults: 1024,
 * 131072 and 2^23.  k_elems must be a multiple of 64 (bits 8) or 128 (bits 4
 * and 1).  Process-wide; affects calls launched afterwards. */
lbgemm_status lbgemm_set_exact_chunk(int bits, int k_elems);
int lbgemm_get_exact_chunk(int bits);

/* ---- K splits of a partial last wave -------------------------------------------
 * The tensor-core GEMM kernels run whole output tiles in waves of the
 * device's CTA slots.  When the tiles of the last wave would fill at most half
 * of the slots, each of them is cut along K into pieces (at least 4 K slices
 * each, as many as fit the wave) whose int32 partial tiles are added into C by
 * TMA reduce-add, after the part of C they cover is cleared; a problem with at
 * most half a wave of tiles is split the same way.  A scheduling choice only:
 * C is the same exact int32 result in every mode.
 * mode 0: split only problems of at most half a wave; 1 (default): also the
 * last partial wave; 2: always cut the last wave's tiles (at least 2 pieces,
 * or 1 K slice each) -- for tests.  Splits need int32 C with N % 4 == 0 and a
 * 16-byte-aligned C; never for the linear layer.  Applies to the re-encoding
 * route (lbgemm_run, lbgemm_run_variant, lbgemm_run_encoded); process-wide;
 * affects calls launched afterwards.  Returns LBGEMM_ERR_INVALID_ARG for a
 * mode outside 0..2. */
lbgemm_status lbgemm_set_tail_split(int mode);
int lbgemm_get_tail_split(void);

/* ---- K slices of the in-kernel conversion kernels -------------------------------
 * The 64- and 128-wide in-kernel-conversion kernels (LBGEMM_ROUTE_FUSED with
 * tile 64 or 128, lbgemm_run_fused) step through K in slices of 128 or 256
 * elements: each slice costs the kernel's roles a fixed number of barrier
 * operations, and longer slices leave fewer slots in tensor memory (6 or 4
 * slots of 128, 3 or 2 of 256).  0 (the default): 256 for the 64-wide
 * kernel and for the linear layer on the 128-wide one, 128 for the GEMM on
 * the 128-wide one (measured fastest on GB300); 128 or 256: that size for
 * both, GEMM and linear layer.  A scheduling choice only: C is the same exact int32
 * result.  Process-wide; affects calls launched afterwards;
 * LBGEMM_ERR_INVALID_ARG for another value. */
lbgemm_status lbgemm_set_fused_slice(int k_elems);
int lbgemm_get_fused_slice(void);

/* ---- work schedule of the in-kernel conversion kernels --------------------------
 * How the 64- and 128-wide in-kernel-conversion kernels share K out over the
 * CTAs when the output tiles alone would not keep the GPU busy: split K
 * (every tile cut into the same number of pieces) or stream-K (every CTA
 * takes an equal run of the tile-major order of all K slices, cut at tile
 * ends; the pieces of a tile are added into C, cleared beforehand).
 * 0 (the default): the library's cost model of waves and partial tiles
 * picks split K for the GEMM, and split K or stream-K for the linear layer
 * (stream-K where its tiles make a fractional number of waves: 192 tokens x
 * 11008 x 4096 measured 53 -> 46 us on GB300); 1: stream-K wherever every
 * CTA gets at least two slices (for the GEMM measured no faster than the
 * split plan: the kernel's per-slice cost does not fall with a shorter run).
 * A scheduling choice only: C is the same exact int32 result, Y the same
 * scaled values.  Process-wide; affects calls launched afterwards;
 * LBGEMM_ERR_INVALID_ARG for another value. */
lbgemm_status lbgemm_set_fused_stream_k(int mode);
int lbgemm_get_fused_stream_k(void);

/* The schedule the 64- or 128-wide in-kernel-conversion kernel takes for an
 * 8-bit GEMM (linear = 0) or linear layer (linear != 0, M <= N) on a device
 * with sm_count SMs (one CTA per SM), 16-byte-aligned operands, under the
 * current slice and stream-K settings: *splits K pieces per tile (1: whole
 * tiles), or *stream_pieces > 0 for stream-K (units per CTA; *splits = 1).
 * Host only.  The converted operand is the larger one (B when N >= M; W for
 * the linear layer), R its rows, S the other's; tiles = ceil(R/128) *
 * ceil(S/tile_n); costs are in whole-tile times on `sm_count` slots:
 * split p (1 <= p <= 16, p = 1 or ceil(K/64)/p >= 4) costs
 * ceil(tiles*p/sm_count) * (1/p + (p > 1 ? 4*tile_n/K : 0)), the cheapest p
 * wins (the first on ties); stream-K, possible when tiles*k >= 2*sm_count
 * with k = ceil(ceil8(K)/slice), costs r/k + (r/k + 1) * 4*tile_n/K with
 * r = ceil(tiles*k/sm_count) and takes r/k rounded up plus 1 pieces.  A GEMM
 * converting A (N < M) with N % 4 != 0 runs whole tiles.  The GEMM takes the
 * cheapest split (stream-K only when lbgemm_set_fused_stream_k forces it);
 * the linear layer keeps a split only if its cost is at most 0.7 of
 * ceil(tiles/sm_count), else whole tiles, and then takes stream-K if its
 * cost is at most 0.85 of the plan kept (or when forced).
 * LBGEMM_ERR_INVALID_ARG for another tile_n or bad sizes. */
lbgemm_status lbgemm_fused_schedule(int64_t M, int64_t N, int64_t K, int tile_n, int linear,
                                    int sm_count, int* splits, int* stream_pieces);

/* ---- status ------------------------------------------------------------------ */

/* Synchronises `stream`, then returns LBGEMM_ERR_TIMEOUT if any kernel of this
 * library on the current device stopped on a wait limit since the last call
 * (and clears that record), else LBGEMM_OK. */
lbgemm_status lbgemm_device_status(void* stream);

/* Diagnostic of the failure path: launches a one-thread kernel that waits on
 * an mbarrier nothing will signal, through the same bounded-wait code the
 * GEMM kernels use, with a 0.1 s limit.  The wait gives up, the kernel
 * returns, and the next lbgemm_device_status() on that stream returns
 * LBGEMM_ERR_TIMEOUT (and clears it).  Nothing hangs or faults. */
lbgemm_status lbgemm_selftest_timeout(void* stream);

/* Message for the last failing call on this thread ("" if none). */
const char* lbgemm_last_error(void);

/* Number of kernels this library has launched in this process (all devices). */
int64_t lbgemm_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* LBGEMM_H */
