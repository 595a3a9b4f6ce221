// mla_layout.cuh -- the shared-memory layout of a gathered KV block (and of the
// query tile), shared by the split kernel and the gather probe.
#pragma once

namespace mla {

// Byte offset of column c (0 <= c < row width) of operand row `row` in a tile
// of `rows` rows laid out as four 128B-swizzled 128-column chunks followed by
// one 64B-swizzled 64-column chunk (the canonical K-major layouts; the same
// bytes read as MN-major give V^T).
__device__ __forceinline__ int tile_offset(int row, int c, int rows)
{
    if (c < 512) {
        const int chunk = c >> 7, kb = c & 127;
        return chunk * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 +
               (((kb >> 4) ^ (row & 7)) << 4) + (kb & 15);
    }
    const int kb = c - 512;
    return 4 * rows * 128 + (row >> 3) * 512 + (row & 7) * 64 +
           (((kb >> 4) ^ ((row & 7) >> 1)) << 4) + (kb & 15);
}

}  // namespace mla
