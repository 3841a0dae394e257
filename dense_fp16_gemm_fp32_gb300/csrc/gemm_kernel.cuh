// Persistent, warp-specialised fp16 GEMM with fp32 accumulation for sm_103a.
//
//   C[M,N] (fp16) = A[M,K] (fp16, row-major) * B[K,N] (fp16, row-major)
//
// The computation is the tiled matrix multiply of "03: Matrix multiplication"
// (phobos-lang.dev tutorial): a CTA owns a TILE_M x TILE_N tile of C, each turn
// of the k loop brings a TILE_M x TILE_K panel of A and a TILE_K x TILE_N panel
// of B into shared memory, their product is added to an fp32 accumulator, and
// the accumulator is narrowed to fp16 once, when the tile is stored. Tiles are
// visited in the grouped order of the kernl notebook "2 - matmul offsets.ipynb"
// (tile_map.cuh).
//
// GB300 mapping (one CTA of 192 threads per SM, persistent over tiles; the
// generic-load form adds loader warps 6..12, see TileCfg):
//   warp 0           TMA producer (one elected lane issues): per k step, one A box (TILE_K x TILE_M,
//                    K contiguous) and TILE_N/64 B boxes (64 x TILE_K, N
//                    contiguous) into an S-stage shared-memory ring, tracked by
//                    full/empty mbarriers. Loads past M, N or K are zero-filled
//                    by the TMA unit, so edge tiles need no masking on load and
//                    a partial last k step adds exact zeros.
//   warp 1           allocates tensor memory (two TILE_N-column fp32
//                    accumulators) and runs the MMA schedule; one elected lane issues tcgen05.mma kind::f16
//                    (M=128, N=TILE_N, K=16), A K-major and B N-major straight
//                    from the swizzled shared-memory tiles, and commits each
//                    stage back to its empty barrier and each finished tile to
//                    an accumulator-full barrier.
//   warps 2..5       epilogue: tcgen05.ld of 64 accumulator columns at a time
//                    (warp w reads TMEM lanes 32*(w%4)..+31, i.e. tile rows),
//                    one round-to-nearest-even conversion to fp16, a swizzled
//                    shared-memory staging buffer and a TMA store of each
//                    32-row x 64-column block (the TMA unit clips rows and
//                    columns past C).
//                    The accumulator is double buffered, so tile i's epilogue
//                    runs under tile i+1's main loop.
// Every mbarrier wait is bounded by %globaltimer; on expiry the CTA records a
// timeout in the device status word, stops issuing, waits (bounded) for its
// own copies and MMAs in flight, frees its tensor memory and returns.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "kernel_common.cuh"
#include "ptx.cuh"
#include "tile_map.cuh"

namespace gemm103 {

// kGeneric: the stages are filled by plain loads (load_stage_generic) from
// warps 0 and 6..12 instead of TMA, and C is written with direct stores, for
// operands whose base or row pitch a tensor map cannot describe.
template <int TM_, int TN_, int TK_, int STAGES_, bool kGeneric_ = false>
struct TileCfg {
    static constexpr int TM = TM_, TN = TN_, TK = TK_, STAGES = STAGES_;
    static constexpr bool kGeneric = kGeneric_;
    // M = 128: row i of the accumulator in tensor-memory lane i. M = 64: rows
    // 16q .. 16q + 15 in the first 16 lanes of lane quadrant q (each epilogue
    // warp reads its quadrant and keeps 16 rows).
    static_assert(TM == 128 || TM == 64, "one-CTA tcgen05 tile of 128 or 64 rows");
    static_assert(TN % 64 == 0 && TN >= 64 && TN <= 256, "B is loaded in 64-column boxes; MMA N <= 256");
    static_assert(TK == 64 || TK == 32, "A rows of 128 B (128B swizzle) or 64 B (64B swizzle)");
    static_assert(!kGeneric || TK == 64, "generic loads write the 128-byte swizzle");

    static constexpr int NUM_THREADS = kGeneric ? 192 + kLoaderThreads - 32 : 192;
    static constexpr int FULL_ARRIVALS = kGeneric ? kLoaderThreads : 1;
    static constexpr int EPI_THREADS = 128;

    static constexpr int A_STAGE = TM * TK * 2;      // bytes of one A panel
    static constexpr int B_BOX = TK * 64 * 2;        // one 64-column B box: TK rows of 128 B
    static constexpr int B_STAGE = (TN / 64) * B_BOX;
    static constexpr uint32_t STAGE_TX = A_STAGE + B_STAGE;

    // A: K-major, rows of TK*2 bytes; core-matrix groups of 8 rows.
    static constexpr uint32_t A_SWIZZLE = TK == 64 ? kSwizzle128B : kSwizzle64B;
    static constexpr uint32_t A_SBO = 8 * TK * 2;
    static constexpr uint32_t A_KSTEP = 32;  // bytes of 16 fp16 along K
    // B: N-major, rows (one per k) of 64 fp16 = 128 bytes, 128B swizzle;
    // next 8 k rows at +1024 B, next 64 columns (next box) at +B_BOX.
    static constexpr uint32_t B_LBO = B_BOX;
    static constexpr uint32_t B_SBO = 1024;
    static constexpr uint32_t B_KSTEP = 16 * 128;  // bytes of 16 k rows

    static constexpr uint32_t IDESC = make_idesc_f16_f32acc(TM, TN, /*a_mn_major=*/false, /*b_mn_major=*/true);
    static constexpr uint32_t TMEM_COLS = (2 * TN <= 32) ? 32 : (2 * TN <= 64) ? 64 : (2 * TN <= 128) ? 128
                                        : (2 * TN <= 256) ? 256 : 512;

    static constexpr int EPI_WARPS = EPI_THREADS / 32;
    static constexpr int EPI_ROWS = TM / EPI_WARPS;  // accumulator rows per epilogue warp
    static constexpr int EPI_COLS = TN >= 64 ? 64 : 32;  // columns per epilogue store block
    static constexpr int STAGING_BYTES = EPI_WARPS * EpiStaging<EPI_COLS>::WARP_BYTES;
    static constexpr int BAR_BYTES = (2 * STAGES + 5) * 8 + 8;
    static constexpr int SMEM_BYTES =
        1024 /*alignment slack*/ + STAGES * (A_STAGE + B_STAGE) + STAGING_BYTES + BAR_BYTES;
    static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB per-CTA shared memory limit");
};

template <class Cfg>
__global__ void __launch_bounds__(Cfg::NUM_THREADS, 1)
    gemm_f16_f32acc_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                           const __grid_constant__ CUtensorMap tmap_c, const GemmParams p)
{
    griddep_launch_dependents();  // the next kernel in the stream may start its prologue
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);  // swizzled tiles need 1024 B alignment
    uint8_t* sA = smem;
    uint8_t* sB = sA + Cfg::STAGES * Cfg::A_STAGE;
    uint8_t* sC = sB + Cfg::STAGES * Cfg::B_STAGE;  // epilogue staging, one EpiStaging per epilogue warp
    uint64_t* full = reinterpret_cast<uint64_t*>(sC + Cfg::STAGING_BYTES);
    uint64_t* empty = full + Cfg::STAGES;
    uint64_t* acc_full = empty + Cfg::STAGES;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int lane = static_cast<int>(threadIdx.x & 31);

    // Prologue, shortest path to the first TMA load: thread 64 initialises the
    // barriers while warp 0 maps its first tile; after one __syncthreads the
    // producer starts, and warp 1 allocates tensor memory meanwhile, then
    // meets the epilogue warps on named barrier 1 for its address.
    if (threadIdx.x == 0 && p.num_k_tiles > 0 && !Cfg::kGeneric) {
        tma_prefetch_desc(&tmap_a);
        tma_prefetch_desc(&tmap_b);
        tma_prefetch_desc(&tmap_c);
    }
    TileCoord first_tc{0, 0};
    if (warp == 0) first_tc = grouped_tile(static_cast<int32_t>(blockIdx.x), p.map);
    if (threadIdx.x == 64) {
        for (int s = 0; s < Cfg::STAGES; ++s) {
            mbar_init(&full[s], Cfg::FULL_ARRIVALS);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], Cfg::EPI_WARPS);  // one arrive per epilogue warp
        }
        mbar_init(drain, 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    __syncthreads();
    uint32_t tmem_base = 0;
    if (warp >= 1 && warp < 2 + Cfg::EPI_WARPS) {  // warp 1 and the epilogue warps
        if (warp == 1) {
            tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
            tmem_relinquish_alloc_permit();
        }
        tc_fence_before_sync();
        named_barrier_sync(1, 32 * (1 + Cfg::EPI_WARPS));
        tc_fence_after_sync();
        tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
    }
    // launched with programmatic stream serialisation, this grid may start
    // while the previous kernel in the stream runs: nothing below touches
    // global memory before that kernel has completed
    griddep_wait();
    const Watch w{abort_flag, p.status, p.watchdog_ns};

    if (Cfg::kGeneric && (warp == 0 || warp >= 6)) {
        // ------------------------------------------------------------ generic loaders
        // Eight warps fill each stage with plain loads; every thread arrives on
        // the stage's full barrier after its writes (kLoaderThreads arrivals).
        const int lt = (warp == 0 ? 0 : warp - 5) * 32 + lane;
        if (p.num_k_tiles > 0 && p.fault_mode != 1) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            const uint32_t a_base = smem_addr(sA);
            const uint32_t b_base = smem_addr(sB);
            for (int32_t tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
                const TileCoord tc = grouped_tile(tile, p.map);
                for (int32_t kt = 0; kt < p.num_k_tiles; ++kt) {
                    ok = warp_wait_phase(&empty[stage], phase ^ 1u, w, kWhereProducer);
                    if (!ok) break;
                    load_stage_generic<Cfg::TM, Cfg::TN>(p, a_base + stage * Cfg::A_STAGE, b_base + stage * Cfg::B_STAGE,
                                                         tc.pid_m * Cfg::TM, tc.pid_n * Cfg::TN, kt * Cfg::TK, lt);
                    fence_proxy_async_smem();  // the tensor cores read these writes
                    mbar_arrive(&full[stage]);
                    if (++stage == Cfg::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 0) {
        // ------------------------------------------------------------ producer
        // The whole warp runs the schedule; one lane, elected with elect.sync, issues.
        if (p.num_k_tiles > 0 && p.fault_mode != 1) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, issued_parity = 0;  // per stage: ever issued / parity of the last issue
            bool ok = true;
            for (int32_t tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
                const TileCoord tc = tile == static_cast<int32_t>(blockIdx.x)
                                         ? first_tc
                                         : grouped_tile(tile, p.map);
                const int32_t m0 = tc.pid_m * Cfg::TM;
                const int32_t n0 = tc.pid_n * Cfg::TN;
                for (int32_t kt = 0; kt < p.num_k_tiles; ++kt) {
                    ok = warp_wait_phase(&empty[stage], phase ^ 1u, w, kWhereProducer);
                    if (!ok) break;
                    const int32_t k0 = kt * Cfg::TK;
                    if (elect_one()) {
                        mbar_arrive_expect_tx(&full[stage], Cfg::STAGE_TX);
                        tma_load_2d(sA + stage * Cfg::A_STAGE, &tmap_a, &full[stage], k0, m0);
#pragma unroll
                        for (int j = 0; j < Cfg::TN / 64; ++j)
                            tma_load_2d(sB + stage * Cfg::B_STAGE + j * Cfg::B_BOX, &tmap_b, &full[stage],
                                        n0 + 64 * j, k0);
                    }
                    __syncwarp();
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == Cfg::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok && lane == 0) {  // aborting: every load already issued lands before the CTA exits
                for (int s = 0; s < Cfg::STAGES; ++s)
                    if (issued & (1u << s)) wait_phase_drain(&full[s], (issued_parity >> s) & 1u, w);
            }
            __syncwarp();
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the schedule and computes the descriptors; one
        // lane elected with elect.sync (the same lane every time: the warp is
        // converged) issues the MMAs and the commits, the accumulator's commit
        // in the same block as the last k step's MMAs. Measured against
        // `lane == 0` as the issuing condition: 1-2 % faster on the 128 x 256
        // and 128 x 128 tiles, 6 % on 64-deep CTA-pair stages.
        if (p.num_k_tiles > 0) {
            int stage = 0;
            uint32_t phase = 0;
            int buf = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            const uint32_t a_base = smem_addr(sA);
            const uint32_t b_base = smem_addr(sB);
            for (int32_t tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
                ok = warp_wait_phase(&acc_empty[buf], acc_phase ^ 1u, w, kWhereMma);
                if (!ok) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * Cfg::TN);
                for (int32_t kt = 0; kt < p.num_k_tiles; ++kt) {
                    ok = warp_wait_phase(&full[stage], phase, w, kWhereMma);
                    if (!ok) break;
                    tc_fence_after_sync();
                    const uint32_t a_s = a_base + stage * Cfg::A_STAGE;
                    const uint32_t b_s = b_base + stage * Cfg::B_STAGE;
                    uint64_t ad[Cfg::TK / 16], bd[Cfg::TK / 16];
#pragma unroll
                    for (int kk = 0; kk < Cfg::TK / 16; ++kk) {
                        ad[kk] = make_smem_desc(a_s + kk * Cfg::A_KSTEP, 16u, Cfg::A_SBO, Cfg::A_SWIZZLE);
                        bd[kk] = make_smem_desc(b_s + kk * Cfg::B_KSTEP, Cfg::B_LBO, Cfg::B_SBO, kSwizzle128B);
                    }
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < Cfg::TK / 16; ++kk)
                            tc_mma_f16_ss(d_tmem, ad[kk], bd[kk], Cfg::IDESC, (kt > 0 || kk > 0) ? 1u : 0u);
                        tc_commit(&empty[stage]);  // frees the stage when these MMAs are done
                        if (kt == p.num_k_tiles - 1) tc_commit(&acc_full[buf]);  // accumulator complete
                    }
                    __syncwarp();
                    if (++stage == Cfg::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (++buf == 2) {
                    buf = 0;
                    acc_phase ^= 1u;
                }
            }
            // every MMA issued above has finished before tensor memory is freed
            if (elect_one()) {
                tc_commit(drain);
                wait_phase_drain(drain, 0u, w);
            }
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const int row = q * Cfg::EPI_ROWS + lane;  // valid for lane < EPI_ROWS
        int buf = 0;
        uint32_t acc_phase = 0;
        for (int32_t tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
            const TileCoord tc = grouped_tile(tile, p.map);
            if (p.trace != nullptr && warp == 2 && lane == 0) {
                p.trace[3 * static_cast<int64_t>(tile) + 0] = tc.pid_m;
                p.trace[3 * static_cast<int64_t>(tile) + 1] = tc.pid_n;
                p.trace[3 * static_cast<int64_t>(tile) + 2] = static_cast<int32_t>(blockIdx.x);
            }
            const int32_t gm = tc.pid_m * Cfg::TM + row;
            const int32_t n0 = tc.pid_n * Cfg::TN;
            uint16_t* crow = p.C + static_cast<int64_t>(gm) * p.ldc;
            if (p.num_k_tiles == 0) {  // K == 0: the empty sum
                if (lane < Cfg::EPI_ROWS && gm < p.M) store_zero_row(crow, n0, Cfg::TN, p.N);
                continue;
            }
            bool ok = wait_phase(&acc_full[buf], acc_phase, w, kWhereEpilogue);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after_sync();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * Cfg::TN);
            uint64_t* release_bar = &acc_empty[buf];
            epilogue_tma_store<Cfg::TN, Cfg::EPI_COLS, Cfg::kGeneric, false, Cfg::EPI_ROWS>(t_row, sC + (warp - 2) * EpiStaging<Cfg::EPI_COLS>::WARP_BYTES, &tmap_c,
                                        tc.pid_m * Cfg::TM + q * Cfg::EPI_ROWS, n0, p.M, p.N, p.C, p.ldc, lane, [&]() {
                                            tc_fence_before_sync();
                                            __syncwarp();
                                            if (lane == 0) mbar_arrive(release_bar);
                                        });
            if (++buf == 2) {
                buf = 0;
                acc_phase ^= 1u;
            }
        }
        if (lane == 0) bulk_wait_group_read<0>();  // every store of C has read its staging buffer
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

// Eight consecutive fp16 values to dst (2-byte aligned); element e is
// written only if e < avail. The widest stores dst's alignment allows.
__device__ __forceinline__ void store8_f16(uint16_t* dst, uint4 v, int32_t avail)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(dst);
    if (avail >= 8 && (a & 15u) == 0) {
        *reinterpret_cast<uint4*>(dst) = v;
        return;
    }
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if (avail >= 8 && (a & 3u) == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) reinterpret_cast<uint32_t*>(dst)[i] = w[i];
        return;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e)
        if (e < avail) dst[e] = static_cast<uint16_t>(w[e >> 1] >> (16 * (e & 1)));
}

// Row-by-row copy of an fp16 matrix between two row pitches (either side may
// be any 2-byte aligned address and pitch): dst[r*ldd + c] = src[r*lds + c]
// for r < rows, c < cols. Used to repack operands a tensor map cannot describe
// into a caller-provided workspace, and to copy C back out of it. HBM-bound:
// each thread moves runs of 8 elements with the widest loads and stores the
// two sides' alignment allows; CTAs take rows in a grid stride.
__global__ void __launch_bounds__(256) copy_rows_f16_kernel(const uint16_t* __restrict__ src, int64_t lds,
                                                            uint16_t* __restrict__ dst, int64_t ldd, int32_t rows,
                                                            int32_t cols)
{
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const uint16_t* s = src + r * lds;
        uint16_t* d = dst + r * ldd;
        for (int32_t c = 8 * static_cast<int32_t>(threadIdx.x); c < cols; c += 8 * static_cast<int32_t>(blockDim.x))
            store8_f16(d + c, load8_f16(s + c, true, cols - c), cols - c);
    }
}

// The grouped map alone, one thread per pid (same device function as above).
__global__ void tile_schedule_kernel(int32_t num_tiles, const TileMap map, int32_t* pid_m, int32_t* pid_n)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t pid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; pid < num_tiles; pid += stride) {
        const TileCoord t = grouped_tile(static_cast<int32_t>(pid), map);
        pid_m[pid] = t.pid_m;
        pid_n[pid] = t.pid_n;
    }
}

}  // namespace gemm103
