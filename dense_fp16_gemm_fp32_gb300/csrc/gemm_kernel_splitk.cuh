// Split-K form of the one-CTA GEMM for problems with few output tiles.
//
// When M x N holds fewer 128 x 128 tiles than there are SMs, the one-tile-
// per-CTA kernels leave most SMs idle and each busy SM must pull a whole
// K panel of A and B by itself. Here a thread-block cluster of S CTAs
// (S = 2, 4 or 8) computes one tile: CTA `rank` runs the k steps
// [rank * ceil(nk/S), ...) of the tile through the same TMA ring, tcgen05
// MMAs and TMEM accumulator as gemm_f16_f32acc_kernel, then
//   1. its epilogue warps copy the fp32 partial tile from tensor memory into
//      its own shared memory (the drained stage ring is reused);
//   2. cluster barrier: every partial is complete and visible;
//   3. CTA `rank` sums rows [rank * 128/S, (rank+1) * 128/S) of all S
//      partials, every thread reading the peers' shared memory through
//      distributed shared memory (mapa + ld.shared::cluster, 4 x S loads in
//      flight) and adding in rank order, narrows each sum to fp16 once (round
//      to nearest even) and stores it to C;
//   4. cluster barrier: no CTA exits while a peer may still read its partial.
// No workspace, no second launch, no atomics: the sum over the S partials is
// in a fixed order, so results are deterministic. The fp32 accumulation is
// the same as in the other kernels; only the order of the k-step sums differs.
#pragma once

#include "gemm_kernel.cuh"

namespace gemm103 {

// fp32 partial tile in shared memory: row r at r * TN * 4 bytes, 16-byte
// chunk c of the row at chunk position c ^ (r & 7), so that the epilogue's
// row-per-lane stores and the reduction's row-contiguous loads are both free
// of bank conflicts.
template <int TN>
__device__ __forceinline__ uint32_t partial_offset(int r, int c)
{
    return static_cast<uint32_t>(r * TN * 4 + ((c ^ (r & 7)) << 4));
}

// Narrows one float4 of sums to fp16 (round to nearest even) and stores the
// columns below N of C[gm, gn .. gn+3].
__device__ __forceinline__ void store4_f16(const GemmParams& p, int32_t gm, int32_t gn, float4 acc)
{
    const uint32_t h0 = pack_half2_rn(__float_as_uint(acc.x), __float_as_uint(acc.y));
    const uint32_t h1 = pack_half2_rn(__float_as_uint(acc.z), __float_as_uint(acc.w));
    uint16_t* dst = p.C + static_cast<int64_t>(gm) * p.ldc + gn;
    if (gn + 4 <= p.N) {
        *reinterpret_cast<uint2*>(dst) = make_uint2(h0, h1);  // 8-byte aligned: 16-byte C rows, gn % 4 == 0
    } else {
        const uint16_t hv[4] = {static_cast<uint16_t>(h0 & 0xFFFFu), static_cast<uint16_t>(h0 >> 16),
                                static_cast<uint16_t>(h1 & 0xFFFFu), static_cast<uint16_t>(h1 >> 16)};
        for (int j = 0; j < 4 && gn + j < p.N; ++j) dst[j] = hv[j];
    }
}

template <class Cfg, int S>
__global__ void __launch_bounds__(Cfg::NUM_THREADS, 1)
    gemm_f16_f32acc_splitk_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                                  const GemmParams p)
{
    static_assert(Cfg::TM == 128 && Cfg::TK == 64 && !Cfg::kGeneric, "one-CTA TMA tile");
    static_assert(Cfg::STAGES * Cfg::A_STAGE >= Cfg::TM * Cfg::TN * 4, "the partial tile fits in the A ring");
    griddep_launch_dependents();  // the next kernel in the stream may start its prologue
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* sA = smem;
    uint8_t* sB = sA + Cfg::STAGES * Cfg::A_STAGE;
    uint8_t* sC = sB + Cfg::STAGES * Cfg::B_STAGE;
    uint64_t* full = reinterpret_cast<uint64_t*>(sC + Cfg::STAGING_BYTES);
    uint64_t* empty = full + Cfg::STAGES;
    uint64_t* acc_full = empty + Cfg::STAGES;
    uint64_t* drain = acc_full + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int lane = static_cast<int>(threadIdx.x & 31);
    static_assert(S == 2 || S == 4 || S == 8, "cluster of 2, 4 or 8 CTAs");
    const int32_t rank = static_cast<int32_t>(cluster_ctarank());
    const int32_t tile = static_cast<int32_t>(blockIdx.x) / S;
    const TileCoord tc = grouped_tile(tile, p.map);
    const int32_t m0 = tc.pid_m * Cfg::TM;
    const int32_t n0 = tc.pid_n * Cfg::TN;
    const int32_t per = (p.num_k_tiles + S - 1) / S;
    const int32_t kt0 = rank * per;
    const int32_t kt1 = min(p.num_k_tiles, kt0 + per);
    const bool has_k = kt1 > kt0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&acc_full[0], 1);
        mbar_init(drain, 1);
        *abort_flag = 0u;
        fence_mbar_init();
        if (has_k) {
            tma_prefetch_desc(&tmap_a);
            tma_prefetch_desc(&tmap_b);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish_alloc_permit();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
    // launched with programmatic stream serialisation, this grid may start
    // while the previous kernel in the stream runs: nothing below touches
    // global memory before that kernel has completed
    griddep_wait();
    const Watch w{abort_flag, p.status, p.watchdog_ns};

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (has_k && p.fault_mode != 1) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, issued_parity = 0;
            bool ok = true;
            for (int32_t kt = kt0; kt < kt1; ++kt) {
                ok = warp_wait_phase(&empty[stage], phase ^ 1u, w, kWhereProducer);
                if (!ok) break;
                const int32_t k0 = kt * Cfg::TK;
                if (elect_one()) {
                    mbar_arrive_expect_tx(&full[stage], Cfg::STAGE_TX);
                    tma_load_2d(sA + stage * Cfg::A_STAGE, &tmap_a, &full[stage], k0, m0);
#pragma unroll
                    for (int j = 0; j < Cfg::TN / 64; ++j)
                        tma_load_2d(sB + stage * Cfg::B_STAGE + j * Cfg::B_BOX, &tmap_b, &full[stage], n0 + 64 * j, k0);
                }
                __syncwarp();
                issued |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == Cfg::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok && lane == 0) {
                for (int s = 0; s < Cfg::STAGES; ++s)
                    if (issued & (1u << s)) wait_phase_drain(&full[s], (issued_parity >> s) & 1u, w);
            }
            __syncwarp();
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (has_k) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            const uint32_t a_base = smem_addr(sA);
            const uint32_t b_base = smem_addr(sB);
            for (int32_t kt = kt0; kt < kt1; ++kt) {
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
                        tc_mma_f16_ss(tmem_base, ad[kk], bd[kk], Cfg::IDESC, (kt > kt0 || kk > 0) ? 1u : 0u);
                    tc_commit(&empty[stage]);
                    if (kt == kt1 - 1) tc_commit(&acc_full[0]);  // the partial accumulator is complete
                }
                __syncwarp();
                if (++stage == Cfg::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (elect_one()) {
                tc_commit(drain);
                wait_phase_drain(drain, 0u, w);
            }
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------ partial tile -> shared memory
        const int q = warp & 3;
        const int row = q * 32 + lane;
        bool ok = false;
        if (has_k) {
            ok = wait_phase(&acc_full[0], 0u, w, kWhereEpilogue);
            ok = __all_sync(0xffffffffu, ok) != 0;
        }
        // the ring's last readers were the MMAs (complete: acc_full or the drain)
        fence_proxy_async_smem();
        const uint32_t part = smem_addr(sA);
        if (ok) {
            tc_fence_after_sync();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < Cfg::TN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    st_shared_v4(part + partial_offset<Cfg::TN>(row, c * 8 + j), r[4 * j], r[4 * j + 1], r[4 * j + 2],
                                 r[4 * j + 3]);
            }
        } else {  // no k steps for this CTA (or an aborted wait): a zero partial
#pragma unroll 4
            for (int c = 0; c < Cfg::TN / 4; ++c) st_shared_v4(part + partial_offset<Cfg::TN>(row, c), 0u, 0u, 0u, 0u);
        }
    }

    // every partial of the cluster is complete and visible
    tc_fence_before_sync();
    cluster_arrive();
    cluster_wait();

    {
        // ------------------------------------------------------------ reduction and store
        // Every warp of the CTA, four granules per thread in flight (measured 1-12 %
        // faster than the four epilogue warps with two).
        if (p.trace != nullptr && rank == 0 && warp == 2 && lane == 0) {
            p.trace[3 * static_cast<int64_t>(tile) + 0] = tc.pid_m;
            p.trace[3 * static_cast<int64_t>(tile) + 1] = tc.pid_n;
            p.trace[3 * static_cast<int64_t>(tile) + 2] = tile;
        }
        constexpr int C4 = Cfg::TN / 4;  // float4 granules per row
        constexpr int ROWS = Cfg::TM / S;
        constexpr int ITEMS = ROWS * C4;
        constexpr int T = Cfg::NUM_THREADS;
        constexpr int GR = 4;
        const int e = static_cast<int>(threadIdx.x);
        const uint32_t part = smem_addr(sA);
        // GR granules per pass: GR * S remote loads in flight per thread
        for (int i0 = e; i0 < ITEMS; i0 += GR * T) {
            float4 v[GR][S];
#pragma unroll
            for (int g = 0; g < GR; ++g) {
                const int i = i0 + g * T;
                if (i < ITEMS) {
                    const uint32_t off = part + partial_offset<Cfg::TN>(rank * ROWS + i / C4, i % C4);
#pragma unroll
                    for (int k = 0; k < S; ++k)
                        v[g][k] = ld_shared_cluster_v4(map_shared_to_rank(off, static_cast<uint32_t>(k)));
                }
            }
#pragma unroll
            for (int g = 0; g < GR; ++g) {
                const int i = i0 + g * T;
                if (i < ITEMS) {
                    float4 acc = v[g][0];
#pragma unroll
                    for (int k = 1; k < S; ++k) {
                        acc.x += v[g][k].x;
                        acc.y += v[g][k].y;
                        acc.z += v[g][k].z;
                        acc.w += v[g][k].w;
                    }
                    const int r = rank * ROWS + i / C4, c4 = i % C4;
                    if (m0 + r < p.M && n0 + 4 * c4 < p.N) store4_f16(p, m0 + r, n0 + 4 * c4, acc);
                }
            }
        }
    }

    // no CTA leaves while a peer may still read its partial
    cluster_arrive();
    cluster_wait();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace gemm103
