// Compiled kernel variants for f64 (double): lane-row geometries (P, R), register-tile geometries (P, S)
// and blocked
// panel widths. The dispatcher picks among them; see dispatch.cpp.
#include "launch.cuh"

namespace bl {

static const KernelEntry k_entries_f64[] = {
    thread_entry<double, 8>(),
    thread_entry<double, 12>(),
    thread_entry<double, 18>(),
    thread_entry<double, 12, 2>(),
    thread_entry<double, 18, 2>(),
    thread_entry<double, 8, 1, true>(),
    thread_entry<double, 12, 1, true>(),
    thread_entry<double, 16, 1, true>(),
    thread_entry<double, 17, 1, true>(),
    thread_entry<double, 18, 1, true>(),
    warp_entry<double, 4, 2>(),
    warp_entry<double, 8, 1>(),
    warp_entry<double, 4, 4>(),
    warp_entry<double, 4, 4, true>(),
    warp_entry<double, 8, 2>(),
    warp_entry<double, 8, 2, true>(),
    warp_entry<double, 16, 1>(),
    warp_entry<double, 8, 3>(),
    warp_entry<double, 8, 3, true>(),
    warp_entry<double, 8, 4>(),
    warp_entry<double, 8, 4, true>(),
    warp_entry<double, 16, 2>(),
    warp_entry<double, 32, 1>(),
    tile_entry<double, 2, 2>(),
    tile_entry<double, 2, 4>(),
    tile_entry<double, 4, 3>(),
    tile_entry<double, 4, 4>(),
    tile_entry<double, 4, 5>(),
    tile_entry<double, 4, 6>(),
    tile_entry<double, 4, 8>(),
    tile_entry<double, 4, 9>(),
    tile_entry<double, 8, 5>(),
    tile_entry<double, 8, 6>(),
    tile_entry<double, 8, 8>(),
    tile_entry<double, 8, 9>(),
    tile_entry<double, 16, 6>(),
    tile_entry<double, 16, 8>(),
    blocked_entry<double, 16>(),
    blocked_entry<double, 32>(),
};

const KernelEntry *entries_f64(int *count) {
    *count = static_cast<int>(sizeof(k_entries_f64) / sizeof(k_entries_f64[0]));
    return k_entries_f64;
}

}  // namespace bl
