// Compiled kernel variants for c128 (cf64): lane-row geometries (P, R), register-tile geometries (P, S)
// and blocked
// panel widths. The dispatcher picks among them; see dispatch.cpp.
#include "launch.cuh"

namespace bl {

static const KernelEntry k_entries_c128[] = {
    thread_entry<cf64, 8>(),
    thread_entry<cf64, 12>(),
    thread_entry<cf64, 18>(),
    thread_entry<cf64, 12, 2>(),
    thread_entry<cf64, 18, 2>(),
    warp_entry<cf64, 4, 2>(),
    warp_entry<cf64, 8, 1>(),
    warp_entry<cf64, 16, 1>(),
    tile_entry<cf64, 2, 2>(),
    tile_entry<cf64, 2, 4>(),
    tile_entry<cf64, 4, 3>(),
    tile_entry<cf64, 4, 4>(),
    tile_entry<cf64, 4, 6>(),
    tile_entry<cf64, 8, 4>(),
    tile_entry<cf64, 8, 5>(),
    tile_entry<cf64, 8, 6>(),
    tile_entry<cf64, 16, 4>(),
    tile_entry<cf64, 16, 5>(),
    blocked_entry<cf64, 16>(),
};

const KernelEntry *entries_c128(int *count) {
    *count = static_cast<int>(sizeof(k_entries_c128) / sizeof(k_entries_c128[0]));
    return k_entries_c128;
}

}  // namespace bl
