// Row softmax kernels for sm_103a: the fused softmax of "02: Fused softmax"
// (phobos-lang.dev tutorial). For each row i of an fp32 array stored `ldx`
// wide, over its first n columns:
//     m = max_j x[i,j],   y[i,j] = exp(x[i,j] - m) / sum_k exp(x[i,k] - m).
// One pass over memory: a row is read once into registers, reduced twice
// (maximum, then sum of the shifted exponentials) and written once.
//
// The work is HBM-bound (8 bytes moved per element, a handful of ALU ops),
// so the design is about keeping loads in flight, not about tensor cores:
//   * rows of up to 1024 columns: one warp per row, the row in registers
//     (V float4 per lane), warp-shuffle reductions, no shared memory;
//   * longer rows: one CTA (T threads) per row, or a thread-block cluster of
//     CL CTAs per row, each CTA holding a slice of 8·4·T columns in registers;
//     per-warp partials meet in shared memory and per-CTA partials are read
//     across the cluster through distributed shared memory.
// All grids are persistent (a multiple of the resident CTAs per SM), rows
// handed out in a grid stride. float4 accesses when every row starts on a
// 16-byte boundary, scalar coalesced accesses otherwise; the one-CTA-per-row
// kernels use the streaming (evict-first) cache hint, the others default
// caching (each the faster of the two as measured). Columns at or past n are
// neither read nor written.
//
// Arithmetic: exp(x - m) is computed as 2^((x - m)·log2e) with the hardware
// ex2.approx (x - m is formed first, so no intermediate overflows for any
// finite row); per-thread sums use four partial accumulators, then a shuffle
// tree; the quotient is a multiply by the IEEE reciprocal of the sum.
// IEEE special values: a NaN or +inf in a row, or a row of all -inf, gives
// NaN for the whole row (through the sum); a -inf entry gives 0.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"

namespace softmax103 {

struct SoftmaxParams {
    const float* X;
    float* Y;
    int64_t ldx;  // row pitches, elements
    int64_t ldy;
    int64_t M;    // rows
    int32_t n;    // columns of each row that belong to it
};

constexpr float kLog2e = 1.44269504088896340736f;
constexpr int kSliceVec = 8;  // float4 per thread in the CTA / cluster kernels

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

__device__ __forceinline__ float ex2_approx(float a)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
    return r;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Loads this thread's share of the columns [col0, col0 + NT·4·V) of one row
// into v; columns at or past n read as -inf. Vector form: float4 number
// t + NT·i holds columns col0 + 4(t + NT·i) + 0..3. Scalar form: column
// col0 + t + NT·i. Both are coalesced across the NT cooperating threads.
template <bool kStream>
__device__ __forceinline__ float4 ld4(const float* p)
{
    if constexpr (kStream) return __ldcs(reinterpret_cast<const float4*>(p));
    return *reinterpret_cast<const float4*>(p);
}

template <bool kStream>
__device__ __forceinline__ float ld1(const float* p)
{
    if constexpr (kStream) return __ldcs(p);
    return *p;
}

template <bool kStream>
__device__ __forceinline__ void st4(float* p, float4 q)
{
    if constexpr (kStream) __stcs(reinterpret_cast<float4*>(p), q);
    else *reinterpret_cast<float4*>(p) = q;
}

template <bool kStream>
__device__ __forceinline__ void st1(float* p, float x)
{
    if constexpr (kStream) __stcs(p, x);
    else *p = x;
}

// kStream: loads and stores with the streaming (evict-first) cache hint,
// else default caching; which is faster depends on the kernel (measured).
template <int NT, int V, bool kVec, bool kStream>
__device__ __forceinline__ void load_slice(const float* row, int col0, int n, int t, float (&v)[4 * V])
{
    if constexpr (kVec) {
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const int e = col0 + 4 * (t + NT * i);
            if (e + 4 <= n) {
                const float4 q = ld4<kStream>(row + e);
                v[4 * i + 0] = q.x;
                v[4 * i + 1] = q.y;
                v[4 * i + 2] = q.z;
                v[4 * i + 3] = q.w;
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) v[4 * i + k] = (e + k < n) ? ld1<kStream>(row + e + k) : neg_inf();
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4 * V; ++i) {
            const int e = col0 + t + NT * i;
            v[i] = (e < n) ? ld1<kStream>(row + e) : neg_inf();
        }
    }
}

// Stores v with the index mapping of load_slice; columns at or past n are
// not written.
template <int NT, int V, bool kVec, bool kStream>
__device__ __forceinline__ void store_slice(float* row, int col0, int n, int t, const float (&v)[4 * V])
{
    if constexpr (kVec) {
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const int e = col0 + 4 * (t + NT * i);
            if (e + 4 <= n) {
                st4<kStream>(row + e, make_float4(v[4 * i + 0], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (e + k < n) st1<kStream>(row + e + k, v[4 * i + k]);
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4 * V; ++i) {
            const int e = col0 + t + NT * i;
            if (e < n) st1<kStream>(row + e, v[i]);
        }
    }
}

template <int N>
__device__ __forceinline__ float thread_max(const float (&v)[N])
{
    float m = v[0];
#pragma unroll
    for (int i = 1; i < N; ++i) m = fmaxf(m, v[i]);
    return m;
}

// v[i] <- exp(v[i] - m) in place; returns the thread's sum of the new values.
template <int N>
__device__ __forceinline__ float exp_shifted_sum(float (&v)[N], float m)
{
    static_assert(N % 4 == 0, "four partial sums");
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < N; ++i) {
        v[i] = ex2_approx((v[i] - m) * kLog2e);
        s[i & 3] += v[i];
    }
    return (s[0] + s[1]) + (s[2] + s[3]);
}

template <int N>
__device__ __forceinline__ void scale(float (&v)[N], float r)
{
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] *= r;
}

// One warp per row (n <= 128·V), persistent grid stride over rows.
// (Measured: keeping two to eight rows in flight per warp was slower.)
template <int V, bool kVec>
__global__ void __launch_bounds__(256) softmax_rows_warp_kernel(SoftmaxParams p)
{
    const int lane = threadIdx.x & 31;
    const int64_t first = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t stride = (int64_t(gridDim.x) * blockDim.x) >> 5;
    for (int64_t r = first; r < p.M; r += stride) {
        float v[4 * V];
        load_slice<32, V, kVec, false>(p.X + r * p.ldx, 0, p.n, lane, v);
        const float m = warp_max(thread_max(v));
        const float s = warp_sum(exp_shifted_sum(v, m));
        scale(v, 1.0f / s);
        store_slice<32, V, kVec, false>(p.Y + r * p.ldy, 0, p.n, lane, v);
    }
}

// Combines partial results (m_q, s_q), s_q = sum over the part of
// exp(x - m_q), into the row's: m = max m_q, s = sum_q s_q·exp(m_q - m).
// A part whose maximum is -inf holds only -inf (or no columns) and adds 0.
__device__ __forceinline__ void combine(float& s, float mq, float sq, float m_row)
{
    if (mq != neg_inf()) s += sq * ex2_approx((mq - m_row) * kLog2e);
}

// One CTA of T threads per row (CL == 1), or a cluster of CL CTAs per row,
// CTA `rank` holding columns [rank·S, (rank+1)·S) with S = 4·kSliceVec·T.
// Every CTA of a cluster walks the same rows, so the cluster barriers match.
//
// One barrier per row (two with a cluster): each warp reduces its columns to
// (m_w, s_w) with s_w = sum exp(x - m_w), keeping exp(x - m_w) in registers;
// the warps' pairs meet in shared memory (and the CTAs' pairs across the
// cluster), every thread combines them into the row's (m, s) in a fixed
// order, and scales its values by exp(m_w - m) / s. The partial slots are
// double buffered by row parity: a slot is rewritten two rows later, after
// a barrier that every reader of it has passed.
template <int T, int CL, bool kVec>
__global__ void __launch_bounds__(T, (CL >= 4 ? 1024 : 768) / T) softmax_rows_cta_kernel(SoftmaxParams p)
{
    constexpr int V = kSliceVec;
    constexpr int S = 4 * V * T;
    constexpr int W = T / 32;
    constexpr bool kStream = CL == 1;  // measured: streaming hints help one CTA per row, hurt clusters
    __shared__ float2 warp_part[2][W];  // [row parity][warp]: (m_w, s_w)
    __shared__ float2 cta_part[2];      // [row parity]: this CTA's (m, s), read by the cluster

    const int t = threadIdx.x;
    const int lane = t & 31;
    const int warp = t >> 5;
    uint32_t rank = 0;
    if constexpr (CL > 1) rank = gemm103::cluster_ctarank();
    const int col0 = int(rank) * S;
    const int64_t first = blockIdx.x / CL;
    const int64_t stride = gridDim.x / CL;

    int b = 0;
    for (int64_t r = first; r < p.M; r += stride, b ^= 1) {
        float v[4 * V];
        load_slice<T, V, kVec, kStream>(p.X + r * p.ldx, col0, p.n, t, v);

        const float mw = warp_max(thread_max(v));
        float sw = 0.f;
        if (mw != neg_inf()) sw = exp_shifted_sum(v, mw);
        else {
#pragma unroll
            for (int i = 0; i < 4 * V; ++i) v[i] = 0.f;
        }
        sw = warp_sum(sw);
        if (lane == 0) warp_part[b][warp] = make_float2(mw, sw);
        __syncthreads();

        float m = warp_part[b][0].x;
#pragma unroll
        for (int w = 1; w < W; ++w) m = fmaxf(m, warp_part[b][w].x);
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) combine(s, warp_part[b][w].x, warp_part[b][w].y, m);
        if constexpr (CL > 1) {
            if (t == 0) cta_part[b] = make_float2(m, s);
            gemm103::cluster_arrive();
            gemm103::cluster_wait();
            const uint32_t a = gemm103::smem_addr(&cta_part[b]);
            float2 q[CL];
#pragma unroll
            for (int k = 0; k < CL; ++k) {
                const uint32_t ra = gemm103::map_shared_to_rank(a, k);
                q[k] = make_float2(gemm103::ld_shared_cluster_f32(ra), gemm103::ld_shared_cluster_f32(ra + 4));
            }
            m = q[0].x;
#pragma unroll
            for (int k = 1; k < CL; ++k) m = fmaxf(m, q[k].x);
            s = 0.f;
            // every CTA combines the partials in rank order: the same s everywhere
#pragma unroll
            for (int k = 0; k < CL; ++k) combine(s, q[k].x, q[k].y, m);
        }

        // values hold exp(x - m_w) (0 where m_w is -inf): y = that · exp(m_w - m) / s
        scale(v, ex2_approx((mw - m) * kLog2e) / s);
        store_slice<T, V, kVec, kStream>(p.Y + r * p.ldy, col0, p.n, t, v);
    }
    if constexpr (CL > 1) {
        // no CTA leaves while a peer may still read its partials
        gemm103::cluster_arrive();
        gemm103::cluster_wait();
    }
}

}  // namespace softmax103
