// Grouped program-id -> output-tile map.
//
// Source: the program-id code of the Triton matmul tutorial as restated and
// worked through in the kernl notebook "2 - matmul offsets.ipynb" (first
// markdown cell, then code cells [4]-[7]): tiles are taken in bands of
// group_size_m tile rows; inside a band the walk is column-major (the tile row
// changes fastest); the last band is clamped to the rows that remain, and the
// row inside the band is the full pid modulo the band's height.
//
// group_size_m must lie in [1, num_pid_m]; the host clamps larger values to
// num_pid_m, which yields the same order (one band holding every row), and
// keeps group_size_m * num_pid_n within the tile count. The host builds the
// launch's TileMap (make_tile_map); the kernels evaluate the map with
// multiply-shift divisions (a few cycles instead of a few hundred for the
// three integer divisions).
#pragma once

#include <stdint.h>

namespace gemm103 {

struct TileCoord {
    int32_t pid_m;
    int32_t pid_n;
};

// Division by a divisor fixed for the launch: one multiply-high, one add and
// one shift (the round-up method of division by invariant integers, Granlund
// and Montgomery, PLDI 1994), exact for every 32-bit dividend. With
// s = ceil(log2 d) and m = floor(2^32 (2^s - d) / d) + 1,
// n / d = (mulhi(m, n) + n) >> s, the sum taken in 64 bits.
struct FastDiv {
    uint32_t d, mul, shift;
};

inline FastDiv make_fast_div(uint32_t d)
{
    uint32_t s = 0;
    while ((uint64_t(1) << s) < d) ++s;
    const uint64_t m = ((uint64_t(1) << 32) * ((uint64_t(1) << s) - d)) / d + 1;
    return FastDiv{d, static_cast<uint32_t>(m), s};
}

__host__ __device__ __forceinline__ uint32_t fast_div(uint32_t n, uint32_t mul, uint32_t shift)
{
#ifdef __CUDA_ARCH__
    const uint32_t hi = __umulhi(n, mul);
#else
    const uint32_t hi = static_cast<uint32_t>((static_cast<uint64_t>(n) * mul) >> 32);
#endif
    return static_cast<uint32_t>((static_cast<uint64_t>(hi) + n) >> shift);
}

// The grouped map's constants for one launch: the divisors are the group's
// tile count (group_size_m * num_pid_n), the band height of a full group
// (group_size_m) and that of the clamped last group.
struct TileMap {
    int32_t num_pid_m, group_size_m;
    uint32_t group_tiles;
    FastDiv by_group, by_band, by_last_band;
};

inline TileMap make_tile_map(int32_t num_pid_m, int32_t num_pid_n, int32_t group_size_m)
{
    TileMap t;
    t.num_pid_m = num_pid_m;
    t.group_size_m = group_size_m;
    t.group_tiles = static_cast<uint32_t>(group_size_m) * static_cast<uint32_t>(num_pid_n);
    const int32_t rem = num_pid_m % group_size_m;
    t.by_group = make_fast_div(t.group_tiles > 0 ? t.group_tiles : 1u);
    t.by_band = make_fast_div(static_cast<uint32_t>(group_size_m));
    t.by_last_band = make_fast_div(static_cast<uint32_t>(rem == 0 ? group_size_m : rem));
    return t;
}

// pid -> (pid_m, pid_n): band = min(num_pid_m - first_pid_m, group_size_m),
// pid_m = first_pid_m + pid mod band, pid_n = (pid mod group_tiles) / band.
__host__ __device__ __forceinline__ TileCoord grouped_tile(int32_t pid, const TileMap& t)
{
    const uint32_t n = static_cast<uint32_t>(pid);
    const uint32_t group_id = fast_div(n, t.by_group.mul, t.by_group.shift);
    const int32_t first_pid_m = static_cast<int32_t>(group_id) * t.group_size_m;
    const bool clamped = t.num_pid_m - first_pid_m < t.group_size_m;
    const uint32_t band = clamped ? t.by_last_band.d : t.by_band.d;
    const uint32_t mul = clamped ? t.by_last_band.mul : t.by_band.mul;
    const uint32_t shift = clamped ? t.by_last_band.shift : t.by_band.shift;
    const uint32_t in_group = n - group_id * t.group_tiles;
    TileCoord c;
    c.pid_m = first_pid_m + static_cast<int32_t>(n - fast_div(n, mul, shift) * band);
    c.pid_n = static_cast<int32_t>(fast_div(in_group, mul, shift));
    return c;
}

}  // namespace gemm103
