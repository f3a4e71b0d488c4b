// Compiled kernel variants for f32 (float): lane-row geometries (P, R), register-tile geometries (P, S)
// and blocked
// panel widths. The dispatcher picks among them; see dispatch.cpp.
#include "launch.cuh"

namespace bl {

static const KernelEntry k_entries_f32[] = {
    warp_entry<float, 4, 2>(),
    warp_entry<float, 8, 1>(),
    warp_entry<float, 4, 4>(),
    warp_entry<float, 4, 4, true>(),
    warp_entry<float, 8, 2>(),
    warp_entry<float, 8, 2, true>(),
    warp_entry<float, 16, 1>(),
    warp_entry<float, 8, 3>(),
    warp_entry<float, 4, 8>(),
    warp_entry<float, 4, 8, true>(),
    warp_entry<float, 8, 4>(),
    warp_entry<float, 8, 4, true>(),
    warp_entry<float, 16, 2>(),
    warp_entry<float, 16, 2, true>(),
    warp_entry<float, 16, 2, true, true>(),
    warp_entry<float, 16, 2, true, true, true, true>(),
    warp_entry<float, 8, 4, true, true>(),
    warp_entry<float, 8, 4, true, true, true, true>(),
    warp_entry<float, 8, 2, true, true>(),
    warp_entry<float, 8, 2, true, true, true, true>(),
    warp_entry<float, 32, 1>(),
    tile_entry<float, 2, 2>(),
    tile_entry<float, 2, 4>(),
    tile_entry<float, 4, 3>(),
    tile_entry<float, 4, 4>(),
    tile_entry<float, 4, 6>(),
    tile_entry<float, 4, 8>(),
    tile_entry<float, 4, 9>(),
    tile_entry<float, 8, 5>(),
    tile_entry<float, 8, 6>(),
    tile_entry<float, 8, 8>(),
    tile_entry<float, 8, 9>(),
    tile_entry<float, 16, 6>(),
    tile_entry<float, 16, 8>(),
    tile_entry<float, 16, 9>(),
    tile_entry<float, 16, 10>(),
    blocked_entry<float, 32>(),
    blocked_entry<float, 64>(),
    colblock_entry<float>(),
};

const KernelEntry *entries_f32(int *count) {
    *count = static_cast<int>(sizeof(k_entries_f32) / sizeof(k_entries_f32[0]));
    return k_entries_f32;
}

}  // namespace bl
