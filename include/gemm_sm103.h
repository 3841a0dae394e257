/*
 * gemm_sm103.h -- C ABI of the GB300 (sm_103a) fp16 GEMM library
 * (libgemm_sm103.so).
 *
 * The operation (from "03: Matrix multiplication", the phobos-lang.dev tutorial:
 * its kernel and the paragraph under it):
 *
 *     C[M,N] = A[M,K] * B[K,N]
 *
 * A, B and C are IEEE binary16 (fp16), dense, row-major and contiguous:
 * element (i,k) of A is at A + i*K + k, (k,j) of B at B + k*N + j, (i,j) of C
 * at C + i*N + j. Products are summed in fp32 (tcgen05 tensor-core MMAs with
 * an fp32 accumulator in tensor memory) and each output is converted to fp16
 * exactly once, round-to-nearest-even, when it is stored.
 *
 * Output tiles are visited in the grouped order of the Triton matmul
 * tutorial's program-id code, as restated and worked through in the kernl
 * notebook "2 - matmul offsets.ipynb" (its first markdown cell):
 *   num_pid_m = ceil(M / TILE_M), num_pid_n = ceil(N / TILE_N)
 *   num_pid_in_group = group_size_m * num_pid_n
 *   group_id    = pid / num_pid_in_group
 *   first_pid_m = group_id * group_size_m
 *   gsm         = min(num_pid_m - first_pid_m, group_size_m)
 *   pid_m       = first_pid_m + pid % gsm
 *   pid_n       = (pid % num_pid_in_group) / gsm
 * A persistent grid of at most one CTA per SM walks pid = blockIdx.x,
 * blockIdx.x + gridDim.x, ... so the CTAs resident at any moment work on
 * neighbouring pids and share A and B panels in L2.
 *
 * Conventions shared by every entry point:
 *   - Pointers named A, B, C, d_* are DEVICE pointers of the current CUDA
 *     device (cudaGetDevice). The caller owns them; the library keeps no
 *     reference after the call returns.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Work is
 *     enqueued asynchronously; no host synchronisation happens unless an entry
 *     point says so.
 *   - The GEMM kernels are launched with programmatic stream serialisation
 *     (programmatic dependent launch): a GEMM may be scheduled while the
 *     previous kernel in its stream still runs, and reads its operands and
 *     writes C only after that kernel has completed (griddepcontrol.wait), so
 *     stream order holds as usual. They also allow the next kernel in the
 *     stream to be scheduled early (griddepcontrol.launch_dependents on
 *     entry); a following kernel that the caller launches with the same
 *     attribute must wait the same way (griddepcontrol.wait or
 *     cudaGridDependencySynchronize) before it reads C. Kernels launched
 *     without that attribute are unaffected.
 *   - Return value: a gemm_status_t. Argument errors are detected on the host
 *     before anything is enqueued. GEMM_ERR_CUDA means a CUDA runtime call
 *     failed; gemm_last_cuda_error() returns its cudaError_t.
 *   - The library allocates nothing per call. On the first call on a device
 *     it allocates one 4-byte device status word (cudaMalloc) and sets kernel
 *     attributes; make that first call before any CUDA-graph stream capture.
 *     The status word lives until the process exits.
 */
#ifndef GEMM_SM103_H
#define GEMM_SM103_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1, /* negative extent, group_size_m <= 0, NULL with work to do, aliasing */
    GEMM_ERR_UNSUPPORTED = 2, /* a pointer that is not 2-byte aligned (not an fp16 address), an
                                 extent or pitch above 2^30, an unknown tile config; for
                                 gemm_f16_f32acc_noalloc also any operand a tensor map cannot
                                 describe (a base not 16-byte aligned, N or K not a multiple
                                 of 8) */
    GEMM_ERR_CUDA = 3,        /* a CUDA runtime call failed (see gemm_last_cuda_error) */
    GEMM_ERR_TIMEOUT = 4      /* a kernel's bounded wait expired (reported by gemm_query_status) */
} gemm_status_t;

/* Tile configurations (TILE_M x TILE_N x TILE_K). */
typedef enum {
    GEMM_TILE_AUTO = 0,       /* the library picks: the configuration gemm_autotune chose for
                                 this (M, N, K) on the current device; else 128x128x64_SPLITK
                                 when there are at most 38 tiles of 128x128 and K >= 2048
                                 (K >= 1024 when M <= 128), or at most 76 and K >= 4096;
                                 64x64x64 when its tiles fit one wave (at most 152) and
                                 M <= 128 or K <= 512; else 128x64x64 on the same terms;
                                 128x256x64 when M <= 128; with at most 38 tiles of 256x256,
                                 256x256x64_PAIR_STREAMK if K >= 10240 (every tile in two k
                                 halves), 256x256x128_PAIR if K > 512 (every tile in two
                                 column halves), else 128x128x64; 128x256x64 with fewer than
                                 76 (less than one wave of CTA pairs) and K < 2048, or with
                                 K <= 256; 256x256x64_PAIR_STREAMK when K >= 4096, there are
                                 76 to 608 (one to eight waves) and the last wave holds more
                                 than 38; otherwise 256x256x64_PAIR */
    GEMM_TILE_128x256x64 = 1, /* 1 CTA per tile, 4-stage TMA ring, 2 TMEM accumulators */
    GEMM_TILE_128x64x32 = 2,  /* the notebook's worked-example tile (BLOCK_SIZE_M 128,
                                 BLOCK_SIZE_N 64, BLOCK_SIZE_K 32) */
    GEMM_TILE_256x256x64_PAIR = 3, /* a 2-CTA cluster per tile (tcgen05 cta_group::2): each
                                 CTA stages 128 rows of A and 128 columns of B, 6 stages.
                                 The pair configurations (3, 4, 8, 9) alternate the k
                                 direction over each cluster's tiles: its 2nd, 4th, ... tile
                                 sums its k steps from the last down to the first, so a wave
                                 of tiles starts on the panel chunks the previous wave left
                                 in L2. The fp32 sum order of a tile thus depends on its
                                 place in the schedule: fixed for a given device, shape,
                                 group_size_m and configuration (repeated calls give the same
                                 bits); with two group sizes an entry of a tile past the
                                 first wave may round one fp16 ulp apart */
    GEMM_TILE_256x256x128_PAIR = 4, /* as 3 with 128-deep k steps, 3 stages */
    GEMM_TILE_128x128x64 = 5, /* 1 CTA per tile, 6 stages: twice the tiles of 128x256 for
                                 problems with few tiles */
    GEMM_TILE_128x128x64_SPLITK = 6, /* a cluster of S = 2, 4 or 8 CTAs per 128x128 tile, each
                                 running 1/S of the k steps; the fp32 partials are summed
                                 through distributed shared memory (S: the largest of 2, 4
                                 and 8 with S <= ceil(K/64), tiles * S <= SMs, and
                                 tiles * S <= 64 for S = 8; S = 1 runs the 128x128x64
                                 kernel) */
    GEMM_TILE_128x64x64 = 7,  /* 1 CTA per tile, 8 stages of 64-deep k steps: four times the
                                 tiles of 128x256 and A rows of 128 bytes, for problems whose
                                 time is each CTA's operand loads */
    GEMM_TILE_256x256x128_PAIR_ALIGNED = 8, /* the aligned, mask-free form of 4 ("03: Matrix
                                 multiplication", the @ph.aligned decorator and the paragraph
                                 under its listing): the caller promises that M and N are
                                 multiples of 256 and K of 128, and the kernel carries no edge
                                 tests. Any other extents give GEMM_ERR_UNSUPPORTED, as do
                                 operands a tensor map cannot describe when no workspace is
                                 given. Never chosen by GEMM_TILE_AUTO (4 computes the same
                                 bits); gemm_autotune times it only on whole tiles */
    GEMM_TILE_256x256x64_PAIR_STREAMK = 9, /* 3 with a stream-K schedule where the last partial
                                 wave of tiles holds more than half of the resident clusters
                                 (and there is at least one full wave): that wave and one full
                                 wave are split by k iterations, one contiguous range per
                                 cluster; and where at most half of the resident clusters
                                 hold a tile each with K >= 10240 (160 k steps of 64): every
                                 tile split into two k halves on two clusters. A tile shared
                                 by two clusters has its first k steps' fp32 partial sums
                                 passed through a workspace and added before the one fp16
                                 rounding (a fixed order: results are deterministic).
                                 Elsewhere it runs as 3. The workspace (about
                                 40 MB: 2 x resident clusters x 256 KiB, plus flags) is
                                 allocated on the first stream-K launch on each stream of a
                                 device and kept until exit; make that first call outside
                                 stream capture (under capture without one, 3 runs instead).
                                 Launches on one stream share it; do not replay a graph that
                                 holds such a launch concurrently with other stream-K work of
                                 the stream it was captured on */
    GEMM_TILE_64x64x64 = 10,  /* 1 CTA per 64x64 tile (tcgen05 M = 64), 8 stages: twice the
                                 CTAs of 128x64x64 for problems whose time is each SM's
                                 operand loads */
    GEMM_TILE_COUNT = 11      /* number of values above, GEMM_TILE_AUTO included */
} gemm_tile_cfg_t;

/*
 * C = A * B, fp16 in, fp32 accumulate, fp16 out (see the header comment).
 *
 *   A            device, fp16 [M,K] row-major; 2-byte aligned
 *   B            device, fp16 [K,N] row-major; 2-byte aligned
 *   C            device, fp16 [M,N] row-major; 2-byte aligned; must not
 *                overlap A or B. Fully overwritten.
 *   M, N, K      extents, 0 <= M, N, K <= 2^30
 *   Operands whose bases are 16-byte aligned and whose row pitches (here K
 *   for A, N for B and C) are multiples of 8 elements run the TMA kernels;
 *   any other operands run a generic kernel that fills the same shared-memory
 *   stages with plain loads and writes C with direct stores (the same tensor
 *   core path and result; 128x256x64 tiles, whatever tile_cfg asks for).
 *   group_size_m GROUP_SIZE_M of the grouped tile order, >= 1. Values above
 *                num_pid_m give the same order as num_pid_m.
 *   stream       cudaStream_t
 *
 * Edge cases: M == 0 or N == 0 is a no-op returning GEMM_OK. K == 0 writes
 * C = +0 (the empty sum). Extents that are not whole tiles are handled by the
 * kernel: the TMA zero-fills loads past M, N and K, and stores are masked.
 */
int gemm_f16_f32acc(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                    int32_t group_size_m, void* stream);

/*
 * As gemm_f16_f32acc, with an explicit tile configuration (gemm_tile_cfg_t)
 * and an optional tile trace.
 *
 *   tile_trace   NULL, or a device int32 array of 3 * num_tiles entries
 *                (num_tiles = ceil(M/TILE_M) * ceil(N/TILE_N), the tile of
 *                gemm_tile_shape; when the operands take the generic-load
 *                kernel (gemm_f16_f32acc_strided), its 128 x 256 tile: size
 *                the array for the larger count). The library cannot check
 *                the array's size: a shorter one is written past its end. When given,
 *                the kernel's scheduler writes, for every pid it processes,
 *                tile_trace[3*pid + 0] = pid_m, [3*pid + 1] = pid_n,
 *                [3*pid + 2] = the CTA (blockIdx.x) that processed it, or for
 *                the CTA-pair configurations the cluster (blockIdx.x / 2) that
 *                processed it (for a split tail tile: its first column half).
 *                Used to check the kernel's own order against the integer map.
 */
int gemm_f16_f32acc_tiled(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                          int32_t group_size_m, int32_t tile_cfg, int32_t* tile_trace, void* stream);

/*
 * As gemm_f16_f32acc_tiled with explicit row pitches (leading dimensions),
 * for operands that are views into larger row-major arrays. This covers the
 * general strides of the Triton tutorial's pointer arithmetic (the kernl
 * notebook's last code cell: stride_am, stride_bk, stride_cm with unit column
 * strides):
 *
 *   element (i,k) of A at A + i*lda + k,  (k,j) of B at B + k*ldb + j,
 *   element (i,j) of C at C + i*ldc + j.
 *
 *   lda >= K, ldb >= N, ldc >= N, each at most 2^30; A, B, C 2-byte aligned.
 *   Pitches that are multiples of 8 elements with 16-byte aligned bases take
 *   the TMA kernels, any others the generic-load kernel (gemm_f16_f32acc).
 *   M, N, K need no alignment: loads past the extents read zeros and stores
 *   stop at column N, so the padding columns [N, ldc) of C are never written.
 *   Errors as for gemm_f16_f32acc (a pitch below its row length is
 *   GEMM_ERR_INVALID_ARG). Column strides other than 1 are not supported.
 */
int gemm_f16_f32acc_strided(const void* A, int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc, int64_t M,
                            int64_t N, int64_t K, int32_t group_size_m, int32_t tile_cfg, int32_t* tile_trace,
                            void* stream);

/*
 * Times every tile configuration (1 .. GEMM_TILE_COUNT-1) on these operands
 * and remembers the fastest for (M, N, K) on the current device, so that
 * GEMM_TILE_AUTO (and gemm_tile_shape / gemm_launch_plan for it) uses it from
 * then on. The analogue of the tutorial kernel's autotuning over a list of
 * configurations keyed on the problem shape.
 *
 *   A, lda, B, ldb, C, ldc, M, N, K, group_size_m
 *              as for gemm_f16_f32acc_strided; C is overwritten (it holds
 *              A*B afterwards). The operands must suit the TMA kernels
 *              (16-byte aligned bases, pitches multiples of 8), else
 *              GEMM_ERR_UNSUPPORTED; M == 0 or N == 0 -> GEMM_ERR_INVALID_ARG.
 *   reps       timed launches per configuration, 1..10000 (after 2 warm-up
 *              launches), timed with CUDA events on `stream`
 *   best_cfg   host int32, or NULL: the chosen configuration
 *   us_per_cfg host array of GEMM_TILE_COUNT floats, or NULL: [c] = mean
 *              microseconds per launch of configuration c (-1 for the
 *              aligned configuration when the extents are not whole tiles:
 *              not timed), [0] = the best
 *
 * Synchronous (waits for its events): not for use under stream capture.
 * gemm_autotune_clear() forgets every choice.
 */
int gemm_autotune(const void* A, int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc, int64_t M, int64_t N,
                  int64_t K, int32_t group_size_m, int32_t reps, int32_t* best_cfg, float* us_per_cfg, void* stream);
int gemm_autotune_clear(void);

/*
 * Bytes of workspace gemm_f16_f32acc_strided_ws needs to run these operands
 * through the TMA kernels (host-only, no device work): 0 when every operand
 * already suits them; otherwise room for a copy, with 16-byte aligned rows
 * and a pitch rounded up to 8 elements, of each operand that does not (A:
 * M x K, B: K x N, C: M x N), each copy 256-byte aligned. The pointers and
 * pitches are only inspected, never dereferenced. Arguments are validated
 * as for gemm_f16_f32acc_strided (same errors); bytes is a host pointer
 * (NULL -> GEMM_ERR_INVALID_ARG).
 */
int gemm_workspace_bytes(const void* A, int64_t lda, const void* B, int64_t ldb, const void* C, int64_t ldc,
                         int64_t M, int64_t N, int64_t K, uint64_t* bytes);

/*
 * As gemm_f16_f32acc_strided, with a caller-owned device workspace for
 * operands a tensor map cannot describe. When workspace is 256-byte aligned
 * and holds at least gemm_workspace_bytes(...) bytes, each such operand is
 * first copied into it (A and B; an HBM-bound row copy kernel), the TMA
 * kernels run on the copies with tile_cfg, and a C copy is then written back
 * to C (stream-ordered, all on `stream`). Otherwise (workspace NULL, too
 * small or misaligned) the call runs the generic-load kernel exactly as
 * gemm_f16_f32acc_strided does. Operands that already suit the TMA kernels
 * are used in place and need no workspace.
 *
 *   workspace        device pointer or NULL; owned by the caller, must not
 *                    overlap A, B or C (GEMM_ERR_INVALID_ARG), and must not
 *                    be used by anything else until the call's work on
 *                    `stream` has finished
 *   workspace_bytes  its size in bytes
 */
int gemm_f16_f32acc_strided_ws(const void* A, int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc,
                               int64_t M, int64_t N, int64_t K, int32_t group_size_m, int32_t tile_cfg,
                               int32_t* tile_trace, void* workspace, uint64_t workspace_bytes, void* stream);

/*
 * Tile shape a configuration uses for a problem (GEMM_TILE_AUTO depends on M): writes TILE_M, TILE_N,
 * TILE_K (host pointers, each may be NULL) and returns GEMM_OK, or
 * GEMM_ERR_UNSUPPORTED for an unknown tile_cfg. No device work.
 */
int gemm_tile_shape(int32_t tile_cfg, int64_t M, int64_t N, int64_t K, int32_t* tile_m,
                    int32_t* tile_n, int32_t* tile_k);

/*
 * The tile configuration a tile_cfg (GEMM_TILE_AUTO included) resolves to
 * for (M, N, K) on the current device: the configuration gemm_autotune chose
 * for this shape, else the rule of GEMM_TILE_AUTO; other values map to
 * themselves. GEMM_ERR_UNSUPPORTED for an unknown tile_cfg. No device work.
 */
int gemm_tile_config(int32_t tile_cfg, int64_t M, int64_t N, int64_t K, int32_t* resolved);

/*
 * How the current device would schedule a problem (no kernel launch):
 *   grid_ctas    CTAs of the persistent grid (2 per cluster for the CTA-pair
 *                configurations)
 *   num_tiles    output tiles (program ids)
 *   split_tiles  CTA-pair configurations: how many of the last pids are
 *                computed as two 256 x 128 column halves by two clusters. The
 *                persistent schedule runs units u = cluster, cluster + clusters,
 *                ...: unit u < num_tiles - split_tiles is pid u; the remaining
 *                units are the halves of the last split_tiles pids, two per pid
 *                in pid order. A last wave of R tiles is split when 2R fits in
 *                one wave of clusters. For GEMM_TILE_256x256x64_PAIR_STREAMK
 *                when its stream-K schedule applies: the number S of
 *                stream-K tiles (the last S pids); pids below num_tiles - S
 *                are whole tiles taken in turn by the clusters, and the
 *                S x ceil(K/64) iterations of the others are split into one
 *                contiguous range per cluster, cluster c holding iterations
 *                [c*I/C, (c+1)*I/C) (I iterations, C = grid_ctas / 2:
 *                every resident cluster, or 2 S clusters for the k-halves form,
 *                where S = num_tiles).
 * Host pointers, each may be NULL. Sets up the configuration's per-device
 * state on first use (like a launch). GEMM_ERR_CUDA without a device.
 */
int gemm_launch_plan(int32_t tile_cfg, int64_t M, int64_t N, int64_t K, int32_t* grid_ctas, int32_t* num_tiles,
                     int32_t* split_tiles);

/*
 * The grouped pid -> (pid_m, pid_n) map, evaluated on the device by the same
 * device function the GEMM kernel's scheduler calls, for any tile shape.
 *
 *   tile_m, tile_n  tile extents, >= 1
 *   d_pid_m, d_pid_n device int32 arrays of num_tiles entries each (written)
 * Returns GEMM_ERR_INVALID_ARG for bad extents or NULL outputs with tiles.
 */
int gemm_tile_schedule(int64_t M, int64_t N, int32_t tile_m, int32_t tile_n, int32_t group_size_m,
                       int32_t* d_pid_m, int32_t* d_pid_n, void* stream);

/*
 * The same grouped map evaluated on the host by the same function the
 * kernels use (the group and band divisions as multiply-shift divisions by
 * constants fixed for the launch), for pids [pid0, pid0 + count): writes
 * pid_m[i], pid_n[i] for pid pid0 + i to HOST arrays of `count` entries.
 * Needs no GPU; for checking the map against an independent implementation.
 * Source: as gemm_tile_schedule.
 *   M, N, tile_m, tile_n, group_size_m   as for gemm_tile_schedule
 * Returns GEMM_ERR_INVALID_ARG for bad extents, a negative count, NULL
 * outputs with count > 0, or a range outside [0, tiles);
 * GEMM_ERR_UNSUPPORTED if the tile count exceeds INT32_MAX.
 */
int gemm_tile_map_host(int64_t M, int64_t N, int32_t tile_m, int32_t tile_n, int32_t group_size_m, int64_t pid0,
                       int32_t count, int32_t* pid_m, int32_t* pid_n);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word. Returns GEMM_ERR_TIMEOUT if a kernel launched since the last query
 * gave up on a bounded wait (its output is then incomplete), GEMM_OK
 * otherwise, or GEMM_ERR_CUDA if synchronisation failed. After a timeout it
 * also synchronises the device and clears the ready flags of the device's
 * stream-K workspaces (an aborted launch may leave one raised); query the
 * status after a timeout before launching more stream-K work.
 */
int gemm_query_status(void* stream);

/* Static string naming a gemm_status_t value. Never NULL. */
const char* gemm_status_string(int status);

/* The cudaError_t of the most recent failed CUDA call in this library
 * (0 if none). */
int gemm_last_cuda_error(void);

/*
 * Upper bound, in nanoseconds of %globaltimer, on every mbarrier wait inside
 * the kernels. When one expires the kernel records GEMM_ERR_TIMEOUT in the
 * status word, stops issuing work, waits (again bounded) for its copies and
 * MMAs in flight, frees its tensor memory and returns. 0 restores the default
 * (2 s, or the GEMM_WATCHDOG_NS environment variable). Process-wide.
 */
int gemm_set_watchdog_ns(uint64_t ns);

/*
 * Test hook for failure detection. mode 0 = off (default); mode 1 = the TMA
 * producer issues no loads, so the MMA warp's bounded wait on the first stage
 * expires and the kernel reports GEMM_ERR_TIMEOUT without touching C beyond
 * what it had already written. No fault, trap or unbounded wait is involved.
 * Process-wide.
 */
int gemm_set_fault_injection(int32_t mode);

/* Number of kernels the GEMM entry points (the workspace copies included) and
 * gemm_tile_schedule have launched in this process, all devices. The row
 * softmax keeps its own count (softmax_launch_count). */
uint64_t gemm_launch_count(void);

/*
 * gemm_f16_f32acc_noalloc -- the same GEMM as gemm_f16_f32acc, run with the
 * one-CTA 128x256x64 tile, for callers that cannot allocate device memory when they
 * call it. The pages have no counterpart to this entry point: it exists for
 * callers such as inference-runtime plugins whose enqueue step must not
 * allocate, hosts that reserve all device memory up front and own it through
 * their own allocator, and latency-critical loops that cannot take the
 * implicit synchronisation of a cudaMalloc. gemm_f16_f32acc allocates its 4-byte status word with cudaMalloc on its
 * first call on a device; this entry point calls no cudaMalloc, cudaFree or
 * allocating library routine. Its only scratch is a file-scope device array
 * of 256 bytes (64 32-bit words, one word used: the watchdog status word),
 * present on every GPU that loads the library until the process exits.
 *
 *   A, B, C, M, N, K, group_size_m, stream
 *              as for gemm_f16_f32acc, with the same validation and errors,
 *              except that operands a tensor map cannot describe (bases not
 *              16-byte aligned, N or K not a multiple of 8) give
 *              GEMM_ERR_UNSUPPORTED: this entry point has no generic kernel
 *   d_status   NULL, or a device uint32_t that receives, in stream order after
 *              the kernel, this call's raw status word: 0 = complete; bit 0
 *              set = a bounded wait expired (the output is then incomplete),
 *              and bits 8..15 then name the role whose wait expired first
 *              (1 TMA producer, 2 MMA issuer, 3 epilogue, 4 drain after an
 *              abort; several CTAs may OR in different roles). Test bit 0,
 *              not equality with 1. The watchdog limit and the test hook of
 *              gemm_set_watchdog_ns and gemm_set_fault_injection apply here
 *              as to every other entry point.
 *
 * The first call on a device (with that device current) looks up the
 * scratch array's device address (cudaGetSymbolAddress) and sets the
 * kernel's shared-memory attribute; make that first call before any stream
 * capture. A call whose scratch need exceeds the array is rejected with
 * GEMM_ERR_UNSUPPORTED before anything is enqueued (this kernel needs one
 * word for any extents). Every call shares the array, which keeps the last
 * call's contents: each call clears the status word on its stream before the
 * kernel runs, so calls that overlap on the GPU (different streams, no
 * ordering between them) race on it.
 */
int gemm_f16_f32acc_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                            int32_t group_size_m, uint32_t* d_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_SM103_H */
