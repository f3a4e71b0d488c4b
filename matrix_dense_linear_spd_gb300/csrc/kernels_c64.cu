// Compiled kernel variants for c64 (cf32): lane-row geometries (P, R), register-tile geometries (P, S)
// and blocked
// panel widths. The dispatcher picks among them; see dispatch.cpp.
#include "launch.cuh"

namespace bl {

static const KernelEntry k_entries_c64[] = {
    warp_entry<cf32, 4, 2>(),
    warp_entry<cf32, 8, 1>(),
    warp_entry<cf32, 4, 4>(),
    warp_entry<cf32, 4, 4, true>(),
    warp_entry<cf32, 8, 2>(),
    warp_entry<cf32, 8, 2, true>(),
    warp_entry<cf32, 16, 1>(),
    warp_entry<cf32, 8, 3>(),
    warp_entry<cf32, 8, 3, true>(),
    warp_entry<cf32, 16, 2>(),
    warp_entry<cf32, 16, 2, true>(),
    warp_entry<cf32, 32, 1>(),
    tile_entry<cf32, 2, 2>(),
    tile_entry<cf32, 2, 4>(),
    tile_entry<cf32, 4, 3>(),
    tile_entry<cf32, 4, 4>(),
    tile_entry<cf32, 4, 6>(),
    tile_entry<cf32, 4, 8>(),
    tile_entry<cf32, 4, 9>(),
    tile_entry<cf32, 8, 5>(),
    tile_entry<cf32, 8, 6>(),
    tile_entry<cf32, 8, 8>(),
    tile_entry<cf32, 8, 9>(),
    tile_entry<cf32, 16, 6>(),
    tile_entry<cf32, 16, 8>(),
    tile_entry<cf32, 16, 9>(),
    blocked_entry<cf32, 32>(),
};

const KernelEntry *entries_c64(int *count) {
    *count = static_cast<int>(sizeof(k_entries_c64) / sizeof(k_entries_c64[0]));
    return k_entries_c64;
}

}  // namespace bl
