// C ABI of the sm_103a row softmax (declared in include/softmax_sm103.h):
// argument validation, the choice among the warp-per-row, CTA-per-row and
// cluster-per-row kernels, persistent grid sizing and the launch.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "softmax_kernel.cuh"
#include "softmax_sm103.h"

namespace gemm103 {
int record_cuda_error(cudaError_t e);  // gemm_api.cu: stores the code, returns GEMM_ERR_CUDA
}

namespace {

using softmax103::SoftmaxParams;

constexpr int kMaxDevices = 64;
constexpr int kWarpBlock = 256;           // 8 rows per CTA in the warp-per-row kernel
constexpr int64_t kMaxPitch = int64_t(1) << 31;
constexpr int kCtaSlice = 4 * softmax103::kSliceVec;  // columns per thread in the CTA kernels
constexpr int kKernels = 28;  // 8 warp + 6 CTA/cluster kernels, float4 and scalar forms


// One launch shape: the kernel family and its template arguments.
struct Shape {
    int threads_per_row;  // 32: one warp per row
    int block;            // threads per CTA
    int cluster;          // CTAs per row
    int v;                // float4 per lane (warp kernel)
};

int pow2_at_least(int64_t x)
{
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

// n <= 1024: one warp, V = ceil(n / 128) float4 per lane; n <= 8192: one CTA
// of 64, 128 or 256 threads; longer rows: a cluster of 2, 4 or 8 CTAs of 256.
Shape choose(int64_t n)
{
    Shape s{};
    if (n <= 1024) {
        s.threads_per_row = 32, s.block = kWarpBlock, s.cluster = 1;
        s.v = int((n + 127) / 128);
    } else if (n <= 256 * kCtaSlice) {
        const int t = pow2_at_least((n + kCtaSlice - 1) / kCtaSlice);
        s.threads_per_row = s.block = t < 64 ? 64 : t;
        s.cluster = 1, s.v = softmax103::kSliceVec;
    } else {
        s.threads_per_row = s.block = 256;
        s.cluster = pow2_at_least((n + 256 * kCtaSlice - 1) / (256 * kCtaSlice));
        s.v = softmax103::kSliceVec;
    }
    return s;
}

// A kernel, its index in the per-device cache and its dynamic shared memory.
struct Kernel {
    void* fn;
    int index;
    int smem;
};

// kVec: every row starts on a 16-byte boundary (float4 accesses).
template <bool kVec>
Kernel kernel_for(const Shape& s)
{
    using namespace softmax103;
    const int base = kVec ? 0 : kKernels / 2;
    if (s.threads_per_row == 32) {
        switch (s.v) {
            case 1: return {reinterpret_cast<void*>(softmax_rows_warp_kernel<1, kVec>), base + 0, 0};
            case 2: return {reinterpret_cast<void*>(softmax_rows_warp_kernel<2, kVec>), base + 1, 0};
            case 3: return {reinterpret_cast<void*>(softmax_rows_warp_kernel<3, kVec>), base + 2, 0};
            case 4: return {reinterpret_cast<void*>(softmax_rows_warp_kernel<4, kVec>), base + 3, 0};
            case 5: return {reinterpret_cast<void*>(softmax_rows_warp_kernel<5, kVec>), base + 4, 0};
            case 6: return {reinterpret_cast<void*>(softmax_rows_warp_kernel<6, kVec>), base + 5, 0};
            case 7: return {reinterpret_cast<void*>(softmax_rows_warp_kernel<7, kVec>), base + 6, 0};
            default: return {reinterpret_cast<void*>(softmax_rows_warp_kernel<8, kVec>), base + 7, 0};
        }
    }
    if (s.cluster == 1) {
        switch (s.block) {
            case 64: return {reinterpret_cast<void*>(softmax_rows_cta_kernel<64, 1, kVec>), base + 8, 0};
            case 128: return {reinterpret_cast<void*>(softmax_rows_cta_kernel<128, 1, kVec>), base + 9, 0};
            default: return {reinterpret_cast<void*>(softmax_rows_cta_kernel<256, 1, kVec>), base + 10, 0};
        }
    }
    switch (s.cluster) {
        case 2: return {reinterpret_cast<void*>(softmax_rows_cta_kernel<256, 2, kVec>), base + 11, 0};
        case 4: return {reinterpret_cast<void*>(softmax_rows_cta_kernel<256, 4, kVec>), base + 12, 0};
        default: return {reinterpret_cast<void*>(softmax_rows_cta_kernel<256, 8, kVec>), base + 13, 0};
    }
}

struct DeviceState {
    bool ready = false;
    int sm_count = 0;
    int resident[kKernels] = {};  // CTAs per SM (clusters per device for cluster kernels); 0 = not queried
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::atomic<uint64_t> g_launches{0};

cudaLaunchAttribute cluster_attr(int cl)
{
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeClusterDimension;
    a.val.clusterDim.x = cl;
    a.val.clusterDim.y = 1;
    a.val.clusterDim.z = 1;
    return a;
}

// Grid of the persistent launch: every resident CTA (or cluster), but no
// more CTAs than the rows need.
int grid_for(const Shape& s, const Kernel& k, int64_t M, int* grid)
{
    void* kernel = k.fn;
    const int index = k.index;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return gemm103::record_cuda_error(e);
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& d = g_dev[dev];
    if (!d.ready) {
        e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return gemm103::record_cuda_error(e);
        d.ready = true;
    }
    if (d.resident[index] == 0) {
        if (k.smem > 48 * 1024) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, k.smem);
            if (e != cudaSuccess) return gemm103::record_cuda_error(e);
        }
        int r = 0;
        if (s.cluster == 1) {
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r, kernel, s.block, k.smem);
        } else {
            cudaLaunchConfig_t q = {};
            cudaLaunchAttribute a = cluster_attr(s.cluster);
            q.gridDim = dim3(s.cluster * d.sm_count, 1, 1);
            q.blockDim = dim3(s.block, 1, 1);
            q.dynamicSmemBytes = k.smem;
            q.attrs = &a;
            q.numAttrs = 1;
            e = cudaOccupancyMaxActiveClusters(&r, kernel, &q);
        }
        if (e != cudaSuccess) return gemm103::record_cuda_error(e);
        d.resident[index] = r < 1 ? 1 : r;
    }
    int64_t units;  // CTAs (cluster == 1) or clusters
    int64_t need;   // units the rows can use
    if (s.cluster == 1) {
        units = int64_t(d.resident[index]) * d.sm_count;
        need = s.threads_per_row == 32 ? (M + kWarpBlock / 32 - 1) / (kWarpBlock / 32) : M;
    } else {
        units = d.resident[index];
        need = M;
    }
    if (need < units) units = need;
    *grid = int(units * s.cluster);
    return GEMM_OK;
}

template <bool kVec>
int launch(const SoftmaxParams& p, cudaStream_t stream)
{
    const Shape s = choose(p.n);
    const Kernel k = kernel_for<kVec>(s);
    int grid = 0;
    int rc = grid_for(s, k, p.M, &grid);
    if (rc != GEMM_OK) return rc;
    cudaLaunchConfig_t lc = {};
    cudaLaunchAttribute a = cluster_attr(s.cluster);
    lc.gridDim = dim3(grid, 1, 1);
    lc.blockDim = dim3(s.block, 1, 1);
    lc.dynamicSmemBytes = k.smem;
    lc.stream = stream;
    lc.attrs = s.cluster > 1 ? &a : nullptr;
    lc.numAttrs = s.cluster > 1 ? 1 : 0;
    void* args[] = {const_cast<SoftmaxParams*>(&p)};
    const cudaError_t e = cudaLaunchKernelExC(&lc, k.fn, args);
    if (e != cudaSuccess) return gemm103::record_cuda_error(e);
    g_launches.fetch_add(1);
    return GEMM_OK;
}

}  // namespace

extern "C" {

int softmax_rows_f32(const float* X, int64_t ldx, float* Y, int64_t ldy, int64_t M, int64_t n, void* stream)
{
    if (M < 0 || n < 0) return GEMM_ERR_INVALID_ARG;
    if (M == 0 || n == 0) return GEMM_OK;
    if (X == nullptr || Y == nullptr || ldx < n || ldy < n) return GEMM_ERR_INVALID_ARG;
    if (n > SOFTMAX_MAX_COLS || ldx > kMaxPitch || ldy > kMaxPitch) return GEMM_ERR_UNSUPPORTED;
    const uintptr_t x = reinterpret_cast<uintptr_t>(X), y = reinterpret_cast<uintptr_t>(Y);
    if ((x & 3u) != 0 || (y & 3u) != 0) return GEMM_ERR_UNSUPPORTED;
    using u128 = unsigned __int128;
    const u128 x_end = static_cast<u128>(x) + (static_cast<u128>(M - 1) * ldx + n) * 4;
    const u128 y_end = static_cast<u128>(y) + (static_cast<u128>(M - 1) * ldy + n) * 4;
    const bool in_place = x == y && ldx == ldy;
    if (!in_place && y < x_end && x < y_end) return GEMM_ERR_INVALID_ARG;

    SoftmaxParams p;
    p.X = X, p.Y = Y, p.ldx = ldx, p.ldy = ldy, p.M = M, p.n = static_cast<int32_t>(n);
    const bool vec = (x & 15u) == 0 && (y & 15u) == 0 && (ldx & 3) == 0 && (ldy & 3) == 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return vec ? launch<true>(p, s) : launch<false>(p, s);
}

int softmax_rows_plan(int64_t M, int64_t n, int32_t* threads_per_row, int32_t* cluster_ctas, int32_t* grid_ctas)
{
    if (M < 0 || n < 1) return GEMM_ERR_INVALID_ARG;
    if (n > SOFTMAX_MAX_COLS) return GEMM_ERR_UNSUPPORTED;
    const Shape s = choose(n);
    if (threads_per_row != nullptr) *threads_per_row = s.threads_per_row;
    if (cluster_ctas != nullptr) *cluster_ctas = s.cluster;
    if (grid_ctas != nullptr) {
        int grid = 0;
        const int rc = grid_for(s, kernel_for<true>(s), M, &grid);
        if (rc != GEMM_OK) return rc;
        *grid_ctas = grid;
    }
    return GEMM_OK;
}

uint64_t softmax_launch_count(void) { return g_launches.load(); }

}  // extern "C"
