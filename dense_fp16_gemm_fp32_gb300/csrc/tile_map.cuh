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
// keeps group_size_m * num_pid_n within the tile count.
#pragma once

#include <stdint.h>

namespace gemm103 {

struct TileCoord {
    int32_t pid_m;
    int32_t pid_n;
};

__host__ __device__ __forceinline__ TileCoord grouped_tile(int32_t pid, int32_t num_pid_m, int32_t num_pid_n,
                                                           int32_t group_size_m)
{
    const int32_t num_pid_in_group = group_size_m * num_pid_n;
    const int32_t group_id = pid / num_pid_in_group;
    const int32_t first_pid_m = group_id * group_size_m;
    const int32_t rows_left = num_pid_m - first_pid_m;
    const int32_t band = rows_left < group_size_m ? rows_left : group_size_m;
    TileCoord t;
    t.pid_m = first_pid_m + pid % band;
    t.pid_n = (pid % num_pid_in_group) / band;
    return t;
}

}  // namespace gemm103
