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
// operand holds a_bytes (K bytes per row) and B b_bytes, for
// tile_coords_raster: keep the smaller operand resident in L2 when it fits
// well inside it (the whole A: GM = all M-tiles, M fastest; else the whole B:
// GM = 0, N fastest), so each operand is read from HBM about once; otherwise
// bands of M-tiles whose A rows take about 32 MB, at least 8 tiles.
// Measured on one GB300 (dram__bytes_read of the MLP step's GEMMs): B
// resident cut the wgrad 28672x4096x8192 from 774 to 341 MB; a 59 MB B did
// not stay resident (486 -> 462 MB, 3% slower), hence the 40 MB bound.
inline int raster_band(int64_t M, int64_t a_bytes, int64_t b_bytes)
{
    constexpr int64_t kResident = (int64_t)40 << 20;
    const int64_t mtiles = M / 128;
    if (a_bytes <= kResident) return (int)mtiles;
    if (b_bytes <= kResident) return 0;
    int64_t gm = ((int64_t)32 << 20) / (a_bytes / mtiles);
    gm = gm < 8 ? 8 : gm;
    return (int)(gm < mtiles ? gm : mtiles);
}

}  // namespace fp8fg
