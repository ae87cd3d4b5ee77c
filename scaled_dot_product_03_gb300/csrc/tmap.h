// tmap.h -- TMA tensor maps built from the caller's strides (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gbattn {

// Returned by the encoders below when the driver refuses a tensor map (the
// reason is kept for tmap_refusal()).  No launch path returns this code.
constexpr cudaError_t kTmapRefused = cudaErrorInvalidPitchValue;
// The calling thread's last refused encoding: dims and byte strides.
const char *tmap_refusal();

// Byte strides of the (rows, heads, batch) dims of a view of 2-byte
// elements, for a tensor map of extents dims (d, rows, heads, batch): a dim
// of extent 1 is never stepped, so it gets the smallest legal stride (16)
// whatever the caller's stride for it is.
inline void tmap_strides(int64_t ss, int64_t sh, int64_t sb, const uint64_t dims[4], uint64_t out[3]) {
    const int64_t el[3] = {ss, sh, sb};
    for (int i = 0; i < 3; ++i) out[i] = dims[i + 1] == 1 ? 16 : (uint64_t)el[i] * 2;
}

// 4-D tiled tensor map over a (d, s, h, b) view of 16-bit elements
// (dtype 0 = fp16, 1 = bf16), 128-byte swizzle, box {64, box_rows, 1, 1}.
// dims are element counts innermost first, strides_bytes are the byte
// strides of dims 1..3 (each a multiple of 16).  Out-of-range rows read as 0.
cudaError_t make_tmap_16bit(CUtensorMap *map, const void *ptr, int dtype, const uint64_t dims[4],
                            const uint64_t strides_bytes[3], uint32_t box_rows);

// 3-D tiled tensor map over a contiguous fp32 array [heads][rows][cols]
// (cols innermost), 128-byte swizzle, box {box_cols, box_rows, 1}; used as
// the target of bulk reduce-adds.  box_cols * 4 must be 128.
cudaError_t make_tmap_f32_acc(CUtensorMap *map, void *ptr, uint64_t cols, uint64_t rows, uint64_t heads,
                              uint32_t box_cols, uint32_t box_rows);

}  // namespace gbattn
