// CTA-pair variant of the persistent fp16 GEMM (fp32 accumulation) for sm_103a.
//
// Same computation and tile order as gemm_kernel.cuh (the tiled matrix
// multiply of "03: Matrix multiplication", phobos-lang.dev tutorial, with the
// grouped order of the kernl notebook "2 - matmul offsets.ipynb"), but each
// 256 x 256 output tile is computed by a cluster of two CTAs on two SMs with
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16):
//
//   * CTA r of the pair (r = %cluster_ctarank) loads rows [128r, 128r + 128)
//     of the tile's A panel and columns [128r, 128r + 128) of its B panel into
//     its own shared memory; the MMA reads A from each CTA's memory for that
//     CTA's half of the rows and B from both, so each SM stages 32 KiB per
//     64 k-values for the same 128 x 256 x 64 of work that costs 48 KiB alone.
//   * Both CTAs' TMA loads complete on the even CTA's full barrier, which the
//     even CTA arms with the pair's total byte count.
//   * The even CTA's MMA warp runs the schedule; one elected lane issues the MMAs
//     and commits each stage to the empty barriers of both CTAs and each
//     finished accumulator to the accumulator-full barriers of both CTAs (one
//     multicast commit reaching the barrier at the same offset in each CTA).
//   * Each CTA's epilogue reads its 128 rows of the fp32 accumulator from its
//     own tensor memory, narrows them once to fp16 and writes them with TMA
//     stores of 32-row x 32-column blocks (64 columns for the pair's last
//     unit) through swizzled staging buffers;
//     each epilogue warp arrives on the even CTA's accumulator-empty barrier
//     as soon as its reads are done.
//   * Tensor memory (2 x 256 fp32 columns, double buffered) is allocated and
//     freed by one warp of each CTA together (cta_group::2).
// Tail: when the last partial wave of tiles would leave more than half of the
// clusters idle, the host marks those last pids as split; each is computed as
// two 256 x 128 column halves (N = 128 MMAs) by two clusters, so the last wave
// takes about half a tile's time. No partial sums cross CTAs.
// Stream-K (PairCfg STREAMK): when the last partial wave holds more than half
// of the clusters, the last wave plus one full wave of tiles are computed as
// one contiguous range of (tile, k step) iterations per cluster: a cluster
// first takes its whole tiles pid = cluster, cluster + clusters, ... below
// sk_first_tile, then its iteration range, walked from its end: first the
// head (the first k steps) of the tile its range ends in, last the tail of
// the tile its range starts in (each range holds at least a tile's k steps,
// so a tile is shared by at most two clusters, and the head of a shared
// tile lies in the lower-numbered cluster). The head's fp32 partial sums go
// to a workspace slot and a ready flag is raised; the tail, the cluster's
// last unit, waits for the flag, copies the partial into its now idle stage
// ring and adds it to its own sums before the one fp16 narrowing. A cluster
// only ever waits on a lower-numbered one, which the hardware dispatched
// before it and which raises the flag without waiting on anything. The sum
// order is fixed by the launch: results are deterministic. This follows the
// stream-K decomposition (Osama, Merrill, Cecka, Garland and Owens,
// "Stream-K: Work-centric Parallel Decomposition for Dense Matrix-Matrix
// Multiplication on the GPU", PPoPP 2023), in its hybrid form (whole tiles
// first, one stream-K wave and a half at the end). The host also launches a
// k-halves form of it for problems with few tiles and a long K: 2 x tiles
// clusters and every tile's iterations as the stream-K range, so that each
// cluster's range is exactly one half of one tile (a head or a tail).
// Successive whole tiles of a cluster alternate the k direction (UnitWalk).
// Waits are bounded as in gemm_kernel.cuh. Before a CTA may exit, its
// producer waits until every stage has been released (so no commit still
// targets it) and the MMA thread waits until both epilogues have released
// both accumulators; the pair then meets at a cluster barrier.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "kernel_common.cuh"
#include "ptx.cuh"
#include "tile_map.cuh"

namespace gemm103 {

// TK is the depth of one pipeline stage (64 or 128). A stage's A panel is
// stored as TK/64 sub-tiles of 128 rows x 64 k (one 128-byte swizzle span per
// row); its B panel as CTA_N/64 boxes of TK k rows x 64 columns. Deeper stages
// amortise the per-stage wait, fence and commits over more MMAs.
// ALIGNED: the aligned specialisation of "03: Matrix multiplication" (the
// @ph.aligned contract: every extent a whole number of tiles, so no masks).
// The host launches it only when M and N are multiples of 256 and K of TK;
// the epilogue's edge tests are then compiled out (loads need none: a TMA box
// never reaches past the tensor when the extents are whole tiles).
// STREAMK: the stream-K schedule described above (the host launches it only
// when it applies; otherwise the plain form of the same configuration runs).
template <int STAGES_, int TK_ = 64, bool ALIGNED_ = false, bool STREAMK_ = false>
struct PairCfg {
    static constexpr int TM = 256, TN = 256, TK = TK_, STAGES = STAGES_;  // tile of the pair
    static constexpr bool ALIGNED = ALIGNED_;
    static constexpr bool STREAMK = STREAMK_;
    static_assert(!(ALIGNED && STREAMK), "one specialisation at a time");
    static_assert(TK == 64 || TK == 128, "stage depth of 64 or 128");
    static constexpr int CTA_M = 128;                                     // A / D rows per CTA
    static constexpr int CTA_N = 128;                                     // B columns per CTA
    static constexpr int NUM_THREADS = 192;
    static constexpr int EPI_WARPS = 4;

    static constexpr int A_SUB = CTA_M * 64 * 2;          // 16 KiB: 128 rows x 64 k
    static constexpr int A_STAGE = (TK / 64) * A_SUB;
    static constexpr int B_BOX = TK * 64 * 2;             // 64 columns x TK rows
    static constexpr int B_STAGE = (CTA_N / 64) * B_BOX;
    static constexpr uint32_t PAIR_STAGE_TX = 2u * (A_STAGE + B_STAGE);

    static constexpr uint32_t A_SBO = 1024;       // 8 rows x 128 B
    static constexpr uint32_t A_KSTEP = 32;       // 16 fp16 along K inside a sub-tile
    static constexpr uint32_t B_LBO = B_BOX;      // next 64 columns
    static constexpr uint32_t B_SBO = 1024;       // next 8 k rows
    static constexpr uint32_t B_KSTEP = 16 * 128; // 16 k rows

    static constexpr uint32_t IDESC = make_idesc_f16_f32acc(TM, TN, /*a_mn_major=*/false, /*b_mn_major=*/true);
    // a column half of a tile (the split tail): N = 128, one 64-column B box per CTA
    static constexpr uint32_t IDESC_HALF = make_idesc_f16_f32acc(TM, TN / 2, false, true);
    static constexpr uint32_t PAIR_STAGE_TX_HALF = 2u * (A_STAGE + B_STAGE / 2);
    static constexpr uint32_t ACC_COLS = TN;      // one accumulator: 128 lanes x 256 fp32 columns per CTA
    static constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;

    // Columns per epilogue store block: 32 while the next unit's main loop
    // runs alongside (measured least interference with it), 64 for the
    // pair's last unit, whose epilogue nothing overlaps, and for every unit
    // when K <= WIDE_EPI_MAX_K, where a unit's epilogue outlasts its main loop
    // (fewer proxy fences and TMA stores: measured 1-18 % faster on such
    // shapes). Each warp's staging holds two 64-column buffers.
    static constexpr int EPI_COLS = 32;
    static constexpr int EPI_COLS_LAST = 64;
    static constexpr int WIDE_EPI_MAX_K = 1024;
    static constexpr int STAGING_BYTES = EPI_WARPS * EpiStaging<EPI_COLS_LAST>::WARP_BYTES;
    // stream-K: one partial-copy barrier per epilogue warp; each warp's partial
    // (32 rows x 256 fp32) lands in its 32 KiB of the idle stage ring
    static constexpr int SK_BARS = STREAMK ? EPI_WARPS : 0;
    static constexpr uint32_t SK_WARP_BYTES = 32u * TN * 4u;
    static_assert(!STREAMK || EPI_WARPS * SK_WARP_BYTES <= STAGES * (A_STAGE + B_STAGE), "partials fit the ring");
    static constexpr int BAR_BYTES = (2 * STAGES + 5 + SK_BARS) * 8 + 8;
    static constexpr int SMEM_BYTES = 1024 + STAGES * (A_STAGE + B_STAGE) + STAGING_BYTES + BAR_BYTES;
    static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB per-CTA shared memory limit");
    static_assert(TMEM_COLS <= 512, "tensor memory holds 512 columns");
};

// Role of a work unit's k range: the whole tile's, the head (first k steps)
// of a stream-K tile shared with the next cluster (its partial goes to the
// workspace), or the tail of one (which adds the head's partial before
// narrowing).
enum : int32_t { kUnitWhole = 0, kUnitHead = 1, kUnitTail = 2 };

// Work unit u of the persistent schedule: the full tiles in pid order, then
// the two column halves of each pid in [num_full_tiles, num_tiles), pid by pid.
struct PairUnit {
    TileCoord tc;
    int32_t pid;
    int32_t half;    // -1: the whole 256-column tile; 0 / 1: columns [0,128) / [128,256)
    int32_t kb, ke;  // k steps [kb, ke) of the tile
    int32_t role;    // kUnitWhole, kUnitHead or kUnitTail
    bool rev;        // k steps taken from ke - 1 down to kb (every other whole unit of a cluster)
    bool last;       // the cluster's last unit
};

__device__ __forceinline__ PairUnit pair_unit(int32_t u, const GemmParams& p)
{
    PairUnit r;
    if (u < p.num_full_tiles) {
        r.pid = u;
        r.half = -1;
    } else {
        const int32_t v = u - p.num_full_tiles;
        r.pid = p.num_full_tiles + (v >> 1);
        r.half = v & 1;
    }
    r.tc = grouped_tile(r.pid, p.map);
    r.kb = 0;
    r.ke = p.num_k_tiles;
    r.role = kUnitWhole;
    return r;
}

// The units one cluster processes, in order; every warp walks its own copy,
// so the producer, MMA and epilogue warps see the same sequence.
//
// A cluster's whole-tile units alternate their k direction: its 1st, 3rd, ...
// unit sweeps k upwards, its 2nd, 4th, ... downwards. The clusters' j-th units
// run side by side as one wave, and consecutive waves of the grouped order
// share A and B panels; a wave that starts where the previous one ended finds
// the panel chunks that wave touched last still in L2, where an upward sweep
// after an upward sweep needs the chunks it touched first, long evicted once a
// wave's panels outgrow the cache.
template <bool kStreamK>
struct UnitWalk {
    int32_t u, step;     // next whole-tile unit and the stride (the cluster count)
    int32_t it, it_end;  // stream-K: the cluster's remaining iteration range, taken from its end
    bool flip;           // direction of the next whole unit

    __device__ __forceinline__ UnitWalk(int32_t pair, int32_t num_pairs, const GemmParams& p)
        : u(pair), step(num_pairs), it(0), it_end(0), flip(false)
    {
        if constexpr (kStreamK) {
            const int64_t T = p.sk_iters;
            it = static_cast<int32_t>(static_cast<int64_t>(pair) * T / num_pairs);
            it_end = static_cast<int32_t>(static_cast<int64_t>(pair + 1) * T / num_pairs);
        }
    }

    __device__ __forceinline__ bool next(PairUnit& r, const GemmParams& p)
    {
        if constexpr (!kStreamK) {
            if (u >= p.num_units) return false;
            r = pair_unit(u, p);
            r.rev = flip;
            flip = !flip;
            u += step;
            r.last = u >= p.num_units;
            return true;
        } else {
            const int32_t KT = p.num_k_tiles;
            if (u < p.sk_first_tile) {
                r.pid = u;
                r.kb = 0;
                r.ke = KT;
                r.role = kUnitWhole;
                r.rev = flip;
                flip = !flip;
                u += step;
            } else {
                if (it >= it_end) return false;
                const int32_t t = (it_end - 1) / KT;
                r.kb = max(it, t * KT) - t * KT;
                r.ke = it_end - t * KT;
                r.pid = p.sk_first_tile + t;
                // a range holds at least KT iterations, or (the k-halves form)
                // is exactly the first or the second half of one tile, so the
                // piece where it ends begins at k step 0 (a head, unless the
                // whole tile) and the piece where it starts runs to the last
                // k step (a tail)
                r.role = r.kb > 0 ? kUnitTail : (r.ke < KT ? kUnitHead : kUnitWhole);
                r.rev = false;
                it_end = t * KT + r.kb;
            }
            r.half = -1;
            r.tc = grouped_tile(r.pid, p.map);
            r.last = u >= p.sk_first_tile && it >= it_end;
            return true;
        }
    }
};

// The stream-K workspace block of one epilogue warp: 32 rows x TN fp32, the
// 16-byte chunk j (columns 4j .. 4j+3) of lane l's row at index j * 32 + l,
// so that each store or load of a warp covers 512 contiguous bytes.
template <int TN>
__device__ __forceinline__ size_t sk_block(int32_t slot, uint32_t rank, int q)
{
    return ((static_cast<size_t>(slot) * 2 + rank) * 4 + static_cast<size_t>(q)) * (32u * TN);
}

// Stream-K head: this warp's 32 accumulator rows, unrounded, to its workspace
// block (see sk_block). release() runs once every tensor-memory read is done.
template <int TN, class Release>
__device__ __forceinline__ void epilogue_store_partial(uint32_t t_row, uint4* ws, int lane, Release release)
{
#pragma unroll 1
    for (int c = 0; c < TN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), r);
        tmem_ld_wait();
        if (c == TN / 32 - 1) release();
#pragma unroll
        for (int j = 0; j < 8; ++j)
            ws[(c * 8 + j) * 32 + lane] = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
    }
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::NUM_THREADS, 1)
    gemm_f16_f32acc_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                                const __grid_constant__ CUtensorMap tmap_b,
                                const __grid_constant__ CUtensorMap tmap_c,
                                const __grid_constant__ CUtensorMap tmap_c_last, const GemmParams p)
{
    griddep_launch_dependents();  // the next kernel in the stream may start its prologue
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* sA = smem;
    uint8_t* sB = sA + Cfg::STAGES * Cfg::A_STAGE;
    uint8_t* sC = sB + Cfg::STAGES * Cfg::B_STAGE;  // epilogue staging, one EpiStaging per epilogue warp
    uint64_t* full = reinterpret_cast<uint64_t*>(sC + Cfg::STAGING_BYTES);
    uint64_t* empty = full + Cfg::STAGES;
    uint64_t* acc_full = empty + Cfg::STAGES;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint64_t* sk_bar = drain + 1;  // Cfg::SK_BARS of them
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sk_bar + Cfg::SK_BARS);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int lane = static_cast<int>(threadIdx.x & 31);
    const uint32_t rank = cluster_ctarank();  // 0: even CTA (issues the MMAs), 1: odd CTA
    const int32_t pair = static_cast<int32_t>(blockIdx.x >> 1);
    const int32_t num_pairs = static_cast<int32_t>(gridDim.x >> 1);

    // Prologue, shortest path to the first TMA load: thread 64 initialises the
    // barriers and every thread arrives on the cluster barrier at once; warp
    // 0 maps its first unit and warp 1 allocates the pair's tensor memory
    // before waiting on it. The cluster barrier (both CTAs' barriers exist
    // before either CTA signals the other) is all the producer waits for; the
    // MMA and epilogue warps then meet warp 1 on named barrier 1 for the
    // tensor-memory address.
    if (threadIdx.x == 0 && p.num_k_tiles > 0) {
        tma_prefetch_desc(&tmap_a);
        tma_prefetch_desc(&tmap_b);
        tma_prefetch_desc(&tmap_c);
        tma_prefetch_desc(&tmap_c_last);
    }
    if (threadIdx.x == 64) {
        for (int s = 0; s < Cfg::STAGES; ++s) {
            mbar_init(&full[s], 1);   // even CTA: one arrive (with the pair's byte count)
            mbar_init(&empty[s], 1);  // one commit from the MMA thread
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 2 * Cfg::EPI_WARPS);  // even CTA: every epilogue warp of the pair
        }
        mbar_init(drain, 1);
        for (int b = 0; b < Cfg::SK_BARS; ++b) mbar_init(&sk_bar[b], 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    cluster_arrive();
    UnitWalk<Cfg::STREAMK> walk(pair, num_pairs, p);  // the producer's walk: its first unit mapped here
    PairUnit un0{};
    bool have0 = false;
    if (warp == 0) have0 = walk.next(un0, p);
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish_alloc_permit_pair();
    }
    cluster_wait();
    uint32_t tmem_base = 0;
    if (warp >= 1) {  // warp 1 and the epilogue warps
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

    if (warp == 0) {
        // ------------------------------------------------------------ producer (both CTAs)
        // The whole warp runs the schedule; one lane, elected with elect.sync, issues.
        if (p.num_k_tiles > 0 && p.fault_mode != 1) {
            const uint32_t full0_even = map_shared_to_rank(smem_addr(&full[0]), 0);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            PairUnit un = un0;
            for (bool have = have0; ok && have; have = walk.next(un, p)) {
                const int32_t m0 = un.tc.pid_m * Cfg::TM + static_cast<int32_t>(rank) * Cfg::CTA_M;
                // whole tile: this CTA's 128 of 256 columns; half tile: its 64 of the half's 128
                const int32_t n0 = un.half < 0 ? un.tc.pid_n * Cfg::TN + static_cast<int32_t>(rank) * Cfg::CTA_N
                                               : un.tc.pid_n * Cfg::TN + un.half * (Cfg::TN / 2) +
                                                     static_cast<int32_t>(rank) * (Cfg::CTA_N / 2);
                const int nbox = un.half < 0 ? Cfg::CTA_N / 64 : Cfg::CTA_N / 128;
                const uint32_t tx = un.half < 0 ? Cfg::PAIR_STAGE_TX : Cfg::PAIR_STAGE_TX_HALF;
                for (int32_t i = 0; i < un.ke - un.kb; ++i) {
                    ok = warp_wait_phase<true>(&empty[stage], phase ^ 1u, w, kWhereProducer);
                    if (!ok) break;
                    const uint32_t fb = full0_even + 8u * static_cast<uint32_t>(stage);
                    const int32_t k0 = (un.rev ? un.ke - 1 - i : un.kb + i) * Cfg::TK;
                    if (elect_one()) {
                        if (rank == 0) mbar_arrive_expect_tx(&full[stage], tx);
#pragma unroll
                        for (int j = 0; j < Cfg::TK / 64; ++j)
                            tma_load_2d_pair(sA + stage * Cfg::A_STAGE + j * Cfg::A_SUB, &tmap_a, fb, k0 + 64 * j, m0);
                        for (int j = 0; j < nbox; ++j)
                            tma_load_2d_pair(sB + stage * Cfg::B_STAGE + j * Cfg::B_BOX, &tmap_b, fb, n0 + 64 * j, k0);
                    }
                    __syncwarp();
                    if (++stage == Cfg::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // every stage released: no commit from the MMA thread still targets this CTA
            for (int i = 0; ok && i < Cfg::STAGES; ++i) {
                ok = warp_wait_phase<true>(&empty[stage], phase ^ 1u, w, kWhereProducer);
                if (++stage == Cfg::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (even CTA)
        // The whole warp runs the schedule and computes the descriptors; one
        // elected lane (elect.sync: the same lane every time in the converged
        // warp) issues the MMAs and the commits, including the accumulator's
        // commit after the last k step (tcgen05.commit tracks the MMAs of the
        // thread that issues it).
        if (rank == 0 && p.num_k_tiles > 0) {
            int stage = 0;
            uint32_t phase = 0;
            int buf = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            const uint32_t a_base = smem_addr(sA);
            const uint32_t b_base = smem_addr(sB);
            PairUnit un;
            while (ok && walk.next(un, p)) {
                const uint32_t idesc = un.half < 0 ? Cfg::IDESC : Cfg::IDESC_HALF;
                ok = warp_wait_phase<true>(&acc_empty[buf], acc_phase ^ 1u, w, kWhereMma);
                if (!ok) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf) * Cfg::ACC_COLS;
                const int32_t nk = un.ke - un.kb;  // the stages arrive in the producer's k order
                for (int32_t i = 0; i < nk; ++i) {
                    ok = warp_wait_phase(&full[stage], phase, w, kWhereMma);
                    if (!ok) break;
                    tc_fence_after_sync();
                    const uint32_t a_s = a_base + stage * Cfg::A_STAGE;
                    const uint32_t b_s = b_base + stage * Cfg::B_STAGE;
                    uint64_t ad[Cfg::TK / 16], bd[Cfg::TK / 16];
#pragma unroll
                    for (int kk = 0; kk < Cfg::TK / 16; ++kk) {
                        ad[kk] = make_smem_desc(a_s + (kk / 4) * Cfg::A_SUB + (kk % 4) * Cfg::A_KSTEP, 16u, Cfg::A_SBO,
                                                kSwizzle128B);
                        bd[kk] = make_smem_desc(b_s + kk * Cfg::B_KSTEP, Cfg::B_LBO, Cfg::B_SBO, kSwizzle128B);
                    }
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < Cfg::TK / 16; ++kk)
                            tc_mma_f16_ss_pair(d_tmem, ad[kk], bd[kk], idesc, (i > 0 || kk > 0) ? 1u : 0u);
                        tc_commit_pair_multicast(smem_addr(&empty[stage]), 0x3);  // the stage is free in both CTAs
                        if (i == nk - 1)  // accumulator complete, in both CTAs
                            tc_commit_pair_multicast(smem_addr(&acc_full[buf]), 0x3);
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
            // both epilogues have released both accumulators: no arrive still targets this CTA
            for (int i = 0; ok && i < 2; ++i) {
                ok = warp_wait_phase<true>(&acc_empty[buf], acc_phase ^ 1u, w, kWhereMma);
                if (++buf == 2) {
                    buf = 0;
                    acc_phase ^= 1u;
                }
            }
            // every MMA issued above has finished before tensor memory is freed
            if (elect_one()) {
                tc_commit_pair(map_shared_to_rank(smem_addr(drain), 0));
                wait_phase_drain(drain, 0u, w);
            }
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t acc_empty0_even = map_shared_to_rank(smem_addr(&acc_empty[0]), 0);
        int buf = 0;
        uint32_t acc_phase = 0;
        PairUnit un;
        while (walk.next(un, p)) {
            const TileCoord tc = un.tc;
            if (p.trace != nullptr && un.half <= 0 && un.role != kUnitHead && rank == 0 && warp == 2 && lane == 0) {
                p.trace[3 * static_cast<int64_t>(un.pid) + 0] = tc.pid_m;
                p.trace[3 * static_cast<int64_t>(un.pid) + 1] = tc.pid_n;
                p.trace[3 * static_cast<int64_t>(un.pid) + 2] = pair;
            }
            const int32_t gm = tc.pid_m * Cfg::TM + static_cast<int32_t>(rank) * Cfg::CTA_M + row;
            const int32_t n0 = tc.pid_n * Cfg::TN + (un.half > 0 ? Cfg::TN / 2 : 0);
            const int32_t ncols = un.half < 0 ? Cfg::TN : Cfg::TN / 2;
            uint16_t* crow = p.C + static_cast<int64_t>(gm) * p.ldc;
            if (p.num_k_tiles == 0) {  // K == 0: the empty sum
                if (gm < p.M) store_zero_row(crow, n0, ncols, p.N);
                continue;
            }
            bool ok = wait_phase<true>(&acc_full[buf], acc_phase, w, kWhereEpilogue);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after_sync();
            const uint32_t t_row =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf) * Cfg::ACC_COLS;
            const uint32_t release_addr = acc_empty0_even + 8u * static_cast<uint32_t>(buf);
            // The accumulator's tensor-memory reads are complete (tcgen05.wait::ld)
            // before the arrive: a relaxed arrive orders nothing else that the MMA
            // warp depends on, and a release at cluster scope measured 3-14 %
            // slower where the epilogue is exposed (few k steps per tile).
            const auto release = [&]() {
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster_relaxed(release_addr);
            };
            const int32_t c_row0 = tc.pid_m * Cfg::TM + static_cast<int32_t>(rank) * Cfg::CTA_M + q * 32;
            uint8_t* staging = sC + (warp - 2) * EpiStaging<Cfg::EPI_COLS_LAST>::WARP_BYTES;
            constexpr bool kA = Cfg::ALIGNED;
            if constexpr (Cfg::STREAMK) {
                if (un.role != kUnitWhole) {
                    const int32_t slot = un.pid - p.sk_first_tile;
                    uint32_t* flag = p.sk_flags + (static_cast<size_t>(slot) * 2 + rank) * 4 + q;
                    const float* blk = p.sk_ws + sk_block<Cfg::TN>(slot, rank, q);
                    if (un.role == kUnitHead) {
                        // the partial sums, then the flag (release at GPU scope, after every lane's stores)
                        epilogue_store_partial<Cfg::TN>(t_row, reinterpret_cast<uint4*>(const_cast<float*>(blk)), lane,
                                                        release);
                        __threadfence();
                        __syncwarp();
                        if (lane == 0) st_release_gpu(flag, 1u);
                    } else {
                        // tail, the cluster's last unit: its MMAs are complete, so the stage ring is
                        // idle; the head's partial is copied into this warp's 32 KiB of it
                        if (!warp_wait_flag(flag, w, kWhereEpilogue)) break;
                        uint8_t* part = sA + static_cast<uint32_t>(q) * Cfg::SK_WARP_BYTES;
                        if (lane == 0) {
                            fence_proxy_async_global();
                            mbar_arrive_expect_tx(&sk_bar[q], Cfg::SK_WARP_BYTES);
                            bulk_load_1d(part, blk, Cfg::SK_WARP_BYTES, &sk_bar[q]);
                        }
                        if (!warp_wait_phase(&sk_bar[q], 0u, w, kWhereEpilogue)) break;
                        const uint32_t part0 = smem_addr(part) + static_cast<uint32_t>(lane) * 16u;
                        // tail sums + head sums, then the one narrowing
                        const auto add = [&](int col, uint32_t(&r)[32]) {
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const uint4 v = ld_shared_v4(part0 + static_cast<uint32_t>((col / 4 + j) * 32 * 16));
                                r[4 * j] = __float_as_uint(__uint_as_float(r[4 * j]) + __uint_as_float(v.x));
                                r[4 * j + 1] = __float_as_uint(__uint_as_float(r[4 * j + 1]) + __uint_as_float(v.y));
                                r[4 * j + 2] = __float_as_uint(__uint_as_float(r[4 * j + 2]) + __uint_as_float(v.z));
                                r[4 * j + 3] = __float_as_uint(__uint_as_float(r[4 * j + 3]) + __uint_as_float(v.w));
                            }
                        };
                        if (lane == 0) bulk_wait_group_read<0>();
                        __syncwarp();
                        epilogue_tma_store<Cfg::TN, Cfg::EPI_COLS_LAST>(t_row, staging, &tmap_c_last, c_row0, n0, p.M,
                                                                        p.N, p.C, p.ldc, lane, release, add);
                        if (lane == 0) *flag = 0u;  // consumed: the next launch starts from a cleared flag
                    }
                    if (++buf == 2) {
                        buf = 0;
                        acc_phase ^= 1u;
                    }
                    continue;
                }
            }
            if (!un.last && p.K > Cfg::WIDE_EPI_MAX_K) {
                if (un.half < 0)
                    epilogue_tma_store<Cfg::TN, Cfg::EPI_COLS, false, kA>(t_row, staging, &tmap_c, c_row0, n0, p.M,
                                                                          p.N, p.C, p.ldc, lane, release);
                else
                    epilogue_tma_store<Cfg::TN / 2, Cfg::EPI_COLS, false, kA>(t_row, staging, &tmap_c, c_row0, n0,
                                                                              p.M, p.N, p.C, p.ldc, lane, release);
            } else {  // 64-column buffers overlap the 32-column ones: drain earlier stores first
                if (lane == 0) bulk_wait_group_read<0>();
                __syncwarp();
                if (un.half < 0)
                    epilogue_tma_store<Cfg::TN, Cfg::EPI_COLS_LAST, false, kA>(t_row, staging, &tmap_c_last, c_row0,
                                                                               n0, p.M, p.N, p.C, p.ldc, lane, release);
                else
                    epilogue_tma_store<Cfg::TN / 2, Cfg::EPI_COLS_LAST, false, kA>(
                        t_row, staging, &tmap_c_last, c_row0, n0, p.M, p.N, p.C, p.ldc, lane, release);
            }
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
    if (*abort_flag != 0u) {
        // aborting: give copies already issued by either CTA time to land
        for (int i = 0; i < 64; ++i) __nanosleep(1000);
    }
    cluster_arrive();
    cluster_wait();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace gemm103
