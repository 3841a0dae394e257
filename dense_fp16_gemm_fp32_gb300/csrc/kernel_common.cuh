// Pieces shared by the GEMM kernels: launch parameters, the device status
// word, bounded mbarrier waits and the fp32 -> fp16 packing of the epilogue.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "ptx.cuh"
#include "tile_map.cuh"

#include <cuda.h>

namespace gemm103 {

// Device status word: bit 0 = a bounded wait expired; bits 8..15 = which role.
enum : uint32_t { kStatusTimeout = 1u };
enum : uint32_t { kWhereProducer = 1u, kWhereMma = 2u, kWhereEpilogue = 3u, kWhereDrain = 4u };

struct GemmParams {
    uint16_t* C;  // fp16 bits, row i at C + i * ldc
    int64_t ldc;  // row pitch of C in elements (a multiple of 8)
    int32_t M, N, K;
    int32_t num_pid_m, num_pid_n, num_tiles, num_k_tiles;
    int32_t group_size_m;  // already clamped to [1, num_pid_m]
    TileMap map;           // the grouped map's divisors for this launch
    uint32_t* status;
    int32_t* trace;  // NULL or 3 * num_tiles entries
    uint64_t watchdog_ns;
    int32_t fault_mode;  // 1: the producer issues nothing (watchdog test)
    // CTA-pair kernel only: pids [num_full_tiles, num_tiles) are computed as two
    // column halves each; work units are the full tiles followed by the halves.
    int32_t num_full_tiles;
    int32_t num_units;
    // Generic-load kernel only (operands TMA cannot describe): A and B through
    // plain loads, row pitches in elements, any value >= the row length.
    const uint16_t* A;
    const uint16_t* B;
    int64_t lda, ldb;
    // Stream-K pair kernel only: pids [0, sk_first_tile) are whole tiles taken
    // in turn by the clusters; the iterations (tile, k step) of pids
    // [sk_first_tile, num_tiles), sk_iters in all, are split into one
    // contiguous range per cluster. sk_ws holds one fp32 partial tile per
    // stream-K pid, sk_flags one ready flag per pid, CTA and epilogue warp.
    int32_t sk_first_tile;
    int32_t sk_iters;
    float* sk_ws;
    uint32_t* sk_flags;
};

struct Watch {
    volatile uint32_t* abort;  // shared: set by the first wait that expires
    uint32_t* status;          // global status word
    uint64_t limit_ns;
};

template <bool kClusterScope>
__device__ __forceinline__ bool try_wait_scoped(uint32_t a, uint32_t parity)
{
    return kClusterScope ? mbar_try_wait_cluster(a, parity) : mbar_try_wait(a, parity);
}

// Wait for the phase of `bar` with the given parity. Returns false if the
// CTA is aborting or the wait exceeded the limit (which starts the abort).
// kClusterScope: acquire at cluster scope, for barriers the peer CTA arrives on.
template <bool kClusterScope = false>
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, const Watch& w, uint32_t where)
{
    const uint32_t a = smem_addr(bar);
    if (try_wait_scoped<kClusterScope>(a, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (try_wait_scoped<kClusterScope>(a, parity)) return true;
        if (*w.abort) return false;
        if (global_timer_ns() - t0 > w.limit_ns) {
            *w.abort = 1u;
            atomicOr(w.status, kStatusTimeout | (where << 8));
            return false;
        }
    }
}

// Bounded wait used while aborting: ignores the abort flag.
template <bool kClusterScope = false>
__device__ __forceinline__ void wait_phase_drain(uint64_t* bar, uint32_t parity, const Watch& w)
{
    const uint32_t a = smem_addr(bar);
    const uint64_t t0 = global_timer_ns();
    while (!try_wait_scoped<kClusterScope>(a, parity)) {
        if (global_timer_ns() - t0 > w.limit_ns) {
            atomicOr(w.status, kStatusTimeout | (kWhereDrain << 8));
            return;
        }
    }
}

// wait_phase for a whole warp: every lane waits, and the result is made
// warp-uniform. Keeping the producer and MMA schedules warp-uniform (all lanes
// run the loops and compute the descriptors, one lane issues) lets the
// compiler keep the tcgen05 operands in uniform registers; a loop whose trip
// depends on one lane's wait results cannot, and the MMA issue rate drops to
// about two thirds of the tensor-core rate.
template <bool kClusterScope = false>
__device__ __forceinline__ bool warp_wait_phase(uint64_t* bar, uint32_t parity, const Watch& w, uint32_t where)
{
    const bool ok = wait_phase<kClusterScope>(bar, parity, w, where);
    return __all_sync(0xffffffffu, ok) != 0;
}

// Wait until the global flag is non-zero (acquire at GPU scope), every lane
// polling. Bounded like wait_phase: false if the CTA is aborting or the wait
// ran out (which starts the abort).
__device__ __forceinline__ bool warp_wait_flag(const uint32_t* flag, const Watch& w, uint32_t where)
{
    bool ok = ld_acquire_gpu(flag) != 0u;
    if (__all_sync(0xffffffffu, ok)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        ok = ld_acquire_gpu(flag) != 0u;
        if (__all_sync(0xffffffffu, ok)) return true;
        if (__any_sync(0xffffffffu, *w.abort != 0u)) return false;
        if (__any_sync(0xffffffffu, global_timer_ns() - t0 > w.limit_ns)) {
            if ((threadIdx.x & 31) == 0) {
                *w.abort = 1u;
                atomicOr(w.status, kStatusTimeout | (where << 8));
            }
            __syncwarp();
            return false;
        }
        __nanosleep(100);
    }
}

// C[row, n0 .. n0 + ncols) = +0 for the columns below N (the K == 0 case).
// No element at or past column N is written.
__device__ __forceinline__ void store_zero_row(uint16_t* crow, int32_t n0, int32_t ncols, int32_t N)
{
    for (int32_t c = 0; c < ncols; c += 8) {
        const int32_t n = n0 + c;
        if (n + 8 <= N && (reinterpret_cast<uintptr_t>(crow + n) & 15u) == 0) {
            *reinterpret_cast<uint4*>(crow + n) = make_uint4(0u, 0u, 0u, 0u);
        } else {
            for (int32_t e = 0; e < 8 && n + e < N; ++e) crow[n + e] = 0;
        }
    }
}

__device__ __forceinline__ uint32_t pack_half2_rn(uint32_t lo_bits, uint32_t hi_bits)
{
    const __half2 h = __floats2half2_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Epilogue staging: each epilogue warp owns two 32-row x COLS-column fp16
// buffers laid out with the TMA swizzle of their row length (COLS = 64: 128-
// byte rows, 16-byte chunk j of row r at chunk j ^ (r & 7); COLS = 32: 64-byte
// rows, chunk j ^ ((r >> 1) & 3)), so the 32 lanes' 16-byte shared stores are
// conflict free and the TMA store reads them unswizzled. Wider blocks mean one
// proxy fence and one TMA store per 64 columns instead of per 32 (the fence and
// the store issue cost about as much per block as the tensor-memory load and
// the conversion together): measured faster where the epilogue is exposed
// (few tiles per CTA), about 0.7 % slower at 8192^3 where it always overlaps
// the main loop; each configuration picks its width.
template <int COLS>
struct EpiStaging {
    static_assert(COLS == 32 || COLS == 64, "64- or 128-byte staging rows");
    static constexpr int BUF_BYTES = 32 * COLS * 2;
    static constexpr int WARP_BYTES = 2 * BUF_BYTES;
    static constexpr int CHUNKS = COLS / 8;  // 16-byte chunks per row
};

// Drains one fp32 accumulator held in tensor memory to C through TMA stores.
//   t_row     tensor-memory address of (this warp's first lane, first column)
//   staging   this warp's 2 staging buffers (EpiStaging<COLS>, 1024-byte aligned)
//   c_row0    first C row of this warp's 32 rows; n0 first C column of the tile
//   M, N, C, ldc  extents, base and row pitch of C
//   release   called by every lane once all tensor-memory reads are done
// The accumulator is narrowed to fp16 once (round to nearest even). Rows past
// M are clipped by the TMA unit; blocks entirely outside C are not stored.
// The TMA unit writes whole 16-byte granules at the right edge of the tensor,
// so a block whose columns end inside a granule past N (N not a multiple of
// 8) is written with masked direct stores instead, leaving C's padding
// columns untouched. Only lane 0 issues TMA stores, so lane 0 alone waits on
// the bulk groups. kDirect: every block is written with direct stores (C's
// base or pitch is not one a TMA store can address). Direct stores are the
// slower form even where nothing overlaps the epilogue (measured: each lane
// owns a row, so a warp's 16-byte stores touch 32 cache lines at once).
// kAligned: the caller guarantees that the tile lies wholly inside C (M and N
// whole multiples of the tile), so the edge tests are compiled out and every
// block is one TMA store.
// add(col, r): called with the lane's fp32 accumulator bits of columns
// [col, col + 32) of its row before they are narrowed (the stream-K finisher
// adds the other k range's partial sums there); NoAddend does nothing.
struct NoAddend {
    __device__ __forceinline__ void operator()(int, uint32_t (&)[32]) const {}
};

// ROWS: accumulator rows per warp, 32 (M = 128 tiles) or 16 (M = 64 tiles,
// whose rows sit in the first 16 lanes of each warp's 32: the other lanes'
// values are read and dropped; C's tensor map then has 16-row boxes).
template <int TN, int COLS, bool kDirect = false, bool kAligned = false, int ROWS = 32, class Release, class Addend>
__device__ __forceinline__ void epilogue_tma_store(uint32_t t_row, uint8_t* staging, const CUtensorMap* tmap_c,
                                                   int32_t c_row0, int32_t n0, int32_t M, int32_t N,
                                                   uint16_t* C, int64_t ldc, int lane, Release release, Addend add)
{
    static_assert(ROWS == 32 || ROWS == 16, "32 or 16 rows per warp");
    const bool live = lane < ROWS;
    using St = EpiStaging<COLS>;
    static_assert(TN % COLS == 0, "whole blocks");
    const uint32_t stage0 = smem_addr(staging);
    const uint32_t row_off = static_cast<uint32_t>(lane) * (COLS * 2);
    const uint32_t swz = COLS == 64 ? static_cast<uint32_t>(lane & 7) : static_cast<uint32_t>((lane >> 1) & 3);
#pragma unroll 1
    for (int c = 0; c < TN / COLS; ++c) {
        uint32_t h[COLS / 2];
        {
            uint32_t r0[32];
            tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * COLS), r0);
            if constexpr (COLS == 64) {
                uint32_t r1[32];
                tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * COLS + 32), r1);
                tmem_ld_wait();
                add(c * COLS + 32, r1);
#pragma unroll
                for (int i = 0; i < 16; ++i) h[16 + i] = pack_half2_rn(r1[2 * i], r1[2 * i + 1]);
            } else {
                tmem_ld_wait();
            }
            if (c == TN / COLS - 1) release();
            add(c * COLS, r0);
#pragma unroll
            for (int i = 0; i < 16; ++i) h[i] = pack_half2_rn(r0[2 * i], r0[2 * i + 1]);
        }
        const int32_t x = n0 + c * COLS;
        static_assert(!(kDirect && kAligned), "the aligned form stores through TMA");
        if (kDirect || (!kAligned && (N & 7) != 0 && x + COLS > N)) {  // or right edge inside a 16-byte granule
            const int32_t row = c_row0 + lane;
            if (live && row < M && x < N) {
                uint16_t* dst = C + static_cast<int64_t>(row) * ldc + x;
                if (x + COLS <= N && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
#pragma unroll
                    for (int j = 0; j < St::CHUNKS; ++j)
                        reinterpret_cast<uint4*>(dst)[j] = make_uint4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
                } else {
#pragma unroll
                    for (int e = 0; e < COLS; ++e) {
                        if (x + e < N) dst[e] = static_cast<uint16_t>(e & 1 ? (h[e >> 1] >> 16) : (h[e >> 1] & 0xFFFFu));
                    }
                }
            }
            if (!kDirect && lane == 0) bulk_commit_group();  // one group per block, as below
            continue;
        }
        const uint32_t buf = stage0 + static_cast<uint32_t>((c & 1) * St::BUF_BYTES);
        // The store that last used this buffer must have read it. Every block
        // commits one bulk group (empty for blocks stored directly or outside
        // C), so with an even number of blocks per tile the group that last
        // used this buffer is the one before the latest (block c-1, or the
        // previous tile's last block, used the other buffer); with an odd
        // number, block 0 follows the previous tile's last block in the same
        // buffer, so it waits for every group.
        if (lane == 0) {
            if ((TN / COLS) % 2 == 1 && c == 0)
                bulk_wait_group_read<0>();
            else
                bulk_wait_group_read<1>();
        }
        __syncwarp();
        if (live) {
#pragma unroll
            for (int j = 0; j < St::CHUNKS; ++j)
                st_shared_v4(buf + row_off + ((static_cast<uint32_t>(j) ^ swz) << 4), h[4 * j], h[4 * j + 1],
                             h[4 * j + 2], h[4 * j + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            if (kAligned || (c_row0 < M && x < N)) tma_store_2d(tmap_c, staging + (c & 1) * St::BUF_BYTES, x, c_row0);
            bulk_commit_group();  // an empty group keeps the per-buffer accounting uniform
        }
    }
}

template <int TN, int COLS, bool kDirect = false, bool kAligned = false, int ROWS = 32, class Release>
__device__ __forceinline__ void epilogue_tma_store(uint32_t t_row, uint8_t* staging, const CUtensorMap* tmap_c,
                                                   int32_t c_row0, int32_t n0, int32_t M, int32_t N,
                                                   uint16_t* C, int64_t ldc, int lane, Release release)
{
    epilogue_tma_store<TN, COLS, kDirect, kAligned, ROWS>(t_row, staging, tmap_c, c_row0, n0, M, N, C, ldc, lane,
                                                          release, NoAddend{});
}

// ---------------------------------------------------------------- generic loads
// For operands a tensor map cannot describe (a base that is not 16-byte
// aligned, a row pitch that is not a multiple of 8 elements), the stages are
// filled with plain loads by kLoaderThreads threads, in exactly the layout the
// TMA unit would write: 16-byte chunks placed by the 128-byte swizzle (chunk
// bits [4,7) of the shared-memory offset XOR bits [7,10)), zeros past M, N, K.
// Each loader thread issues all of its loads of a stage before its first
// shared-memory store (one memory round trip per stage), then makes its
// writes visible to the tensor cores (fence.proxy.async) and arrives on the
// stage's full barrier.
constexpr int kLoaderThreads = 256;

__device__ __forceinline__ uint32_t swizzle128(uint32_t off) { return off ^ ((off >> 3) & 0x70u); }

// Eight consecutive fp16 values from src (2-byte aligned); element e is read
// only if e < avail (zero otherwise, and all zero when !row_ok).
__device__ __forceinline__ uint4 load8_f16(const uint16_t* src, bool row_ok, int32_t avail)
{
    if (!row_ok || avail <= 0) return make_uint4(0u, 0u, 0u, 0u);
    const uintptr_t a = reinterpret_cast<uintptr_t>(src);
    if (avail >= 8 && (a & 15u) == 0) return __ldg(reinterpret_cast<const uint4*>(src));
    uint32_t w[4];
    if (avail >= 8 && (a & 3u) == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = __ldg(reinterpret_cast<const uint32_t*>(src) + i);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = (2 * i < avail) ? __ldg(src + 2 * i) : 0u;
            const uint32_t hi = (2 * i + 1 < avail) ? __ldg(src + 2 * i + 1) : 0u;
            w[i] = lo | (hi << 16);
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// One stage: A rows m0.. (TM x 64, K-major, rows of 128 B) and B rows k0..
// (64 x TN, N-major, 64-column boxes of 64 rows x 128 B), as the TMA loads of
// the same stage would leave them. lt = loader thread index.
template <int TM, int TN>
__device__ __forceinline__ void load_stage_generic(const GemmParams& p, uint32_t a_stage, uint32_t b_stage, int32_t m0,
                                                   int32_t n0, int32_t k0, int lt)
{
    constexpr int TK = 64;
    constexpr int A_ROW_CHUNKS = TK / 8;
    constexpr int B_ROW_CHUNKS = TN / 8;
    constexpr int A_PER = TM * A_ROW_CHUNKS / kLoaderThreads;
    constexpr int B_PER = TK * B_ROW_CHUNKS / kLoaderThreads;
    static_assert(A_PER * kLoaderThreads == TM * A_ROW_CHUNKS && B_PER * kLoaderThreads == TK * B_ROW_CHUNKS,
                  "whole chunks per loader thread");
    constexpr uint32_t B_BOX = TK * 128;
    uint4 va[A_PER], vb[B_PER];
#pragma unroll
    for (int i = 0; i < A_PER; ++i) {
        const int q = lt + kLoaderThreads * i;
        const int r = q / A_ROW_CHUNKS, c = q % A_ROW_CHUNKS;
        const int32_t gm = m0 + r, gk = k0 + 8 * c;
        va[i] = load8_f16(p.A + static_cast<int64_t>(gm) * p.lda + gk, gm < p.M, p.K - gk);
    }
#pragma unroll
    for (int i = 0; i < B_PER; ++i) {
        const int q = lt + kLoaderThreads * i;
        const int k = q / B_ROW_CHUNKS, c = q % B_ROW_CHUNKS;
        const int32_t gk = k0 + k, gn = n0 + 8 * c;
        vb[i] = load8_f16(p.B + static_cast<int64_t>(gk) * p.ldb + gn, gk < p.K, p.N - gn);
    }
#pragma unroll
    for (int i = 0; i < A_PER; ++i) {
        const int q = lt + kLoaderThreads * i;
        const int r = q / A_ROW_CHUNKS, c = q % A_ROW_CHUNKS;
        st_shared_v4(a_stage + swizzle128(static_cast<uint32_t>(r * TK * 2 + c * 16)), va[i].x, va[i].y, va[i].z,
                     va[i].w);
    }
#pragma unroll
    for (int i = 0; i < B_PER; ++i) {
        const int q = lt + kLoaderThreads * i;
        const int k = q / B_ROW_CHUNKS, c = q % B_ROW_CHUNKS;
        const uint32_t off = static_cast<uint32_t>(c >> 3) * B_BOX + static_cast<uint32_t>(k * 128 + (c & 7) * 16);
        st_shared_v4(b_stage + swizzle128(off), vb[i].x, vb[i].y, vb[i].z, vb[i].w);
    }
}

}  // namespace gemm103
