// Host-side description of one compiled kernel variant (plain data; no device code).
#pragma once

#include <cstddef>
#include <cuda_runtime.h>

#include "bl_types.cuh"

namespace bl {

// `cap` is the largest n + rhs-rows-per-pass the variant holds (0: any order); `rhs_max` the
// right-hand sides one pass solves (0: any; -1: the variant does not solve).
struct KernelEntry {
    int family;          // 0 = tile, 1 = blocked, 2 = warp, 3 = thread (potrf only)
    int p, s, nb;        // tile geometry (p, s), warp geometry (p lanes, s = rows per lane; nb bit 0:
                         // whole-square slabs, bit 1: packed f32x2 update), blocked panel width nb (s = 2: the column-block
                         // tensor-core kernel), or thread capacity nb (p = 2: a pair of lanes per matrix;
                         // s = 1: fully unrolled at n = nb)
    int cap;
    int rhs_max;
    int threads, per_cta;
    size_t smem;
    cudaError_t (*launch)(const BatchArgs &, cudaStream_t);
};

const KernelEntry *entries_f32(int *count);
const KernelEntry *entries_f64(int *count);
const KernelEntry *entries_c64(int *count);
const KernelEntry *entries_c128(int *count);

}  // namespace bl
