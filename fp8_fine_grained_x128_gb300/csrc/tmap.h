// tmap.h -- host-side helpers shared by the GEMM kernels: construction of 2-D
// TMA tensor maps (128-byte swizzle) and the choice of the tile raster.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace fp8fg {

// Tensor map over a row-major [rows][inner] matrix (row stride in bytes),
// boxes of box_inner x box_rows elements, 128-byte swizzle, zero fill
// outside the matrix.  false if the driver's encoder is unavailable or
// rejects the arguments (base / stride alignment, box size).
bool make_map_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *ptr, uint64_t inner, uint64_t rows,
                 uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapL2promotion l2);

// Raster band of a persistent GEMM over (M / 128) x (N / bn) tiles whose A
// operand holds a_bytes and B b_bytes, for tile_coords_raster: keep the
// smaller operand resident in L2 when one fits comfortably (the whole A:
// GM = all M-tiles, M fastest; else the whole B: GM = 0, N fastest), so each
// operand is read from HBM about once; otherwise bands of 16 M-tiles, where
// the grid's concurrent tiles (about 16 x 9.5 of 128 x 256) read the fewest
// operand bytes per K step.
inline int raster_band(int64_t M, int64_t a_bytes, int64_t b_bytes)
{
    constexpr int64_t kResident = (int64_t)64 << 20;
    const int64_t mtiles = M / 128;
    if (a_bytes <= kResident) return (int)mtiles;
    if (b_bytes <= kResident) return 0;
    return (int)(mtiles < 16 ? mtiles : 16);
}

}  // namespace fp8fg
