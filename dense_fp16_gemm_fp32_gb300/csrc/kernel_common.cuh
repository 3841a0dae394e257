// Pieces shared by the GEMM kernels: launch parameters, the device status
// word, bounded mbarrier waits and the fp32 -> fp16 packing of the epilogue.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace gemm103 {

// Device status word: bit 0 = a bounded wait expired; bits 8..15 = which role.
enum : uint32_t { kStatusTimeout = 1u };
enum : uint32_t { kWhereProducer = 1u, kWhereMma = 2u, kWhereEpilogue = 3u, kWhereDrain = 4u };

struct GemmParams {
    uint16_t* C;  // fp16 bits, [M,N] row-major
    int32_t M, N, K;
    int32_t num_pid_m, num_pid_n, num_tiles, num_k_tiles;
    int32_t group_size_m;  // already clamped to [1, num_pid_m]
    uint32_t* status;
    int32_t* trace;  // NULL or 3 * num_tiles entries
    uint64_t watchdog_ns;
    int32_t fault_mode;  // 1: the producer issues nothing (watchdog test)
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

__device__ __forceinline__ uint32_t pack_half2_rn(uint32_t lo_bits, uint32_t hi_bits)
{
    const __half2 h = __floats2half2_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
    return *reinterpret_cast<const uint32_t*>(&h);
}

}  // namespace gemm103
