// band.h -- parameters and launch of the banded narrow-group tcgen05 kernel
// (csrc/tc_band_sm103.cu), shared by the host planner and the kernel.
#pragma once
#include <stdint.h>
#include <cuda.h>           // CUtensorMap (header-only use)
#include <cuda_runtime.h>

namespace cbd {

// Banded narrow-group tcgen05 kernel parameters (C/G = K/G in {8, 16, 32},
// C % 64 == 0, strides 1 or 2): output classes (a, b) = (hi % sh, wi % sw),
// class index a * sw + b; a work unit is (image, band of 4 output rows,
// segment of segw output columns) of one 64-channel block; a window is a
// (column shift, staged-row offset) position of the 128 GEMM rows in the
// staged band, read by the taps of one or more classes.
constexpr int kBandMaxTaps = 32;
struct BandParams {
    CUtensorMap tmap_dy;  // dy as {K, Wo, Ho, N}, box {64, 32, rows, 1}, 128B swizzle, zero outside dy
    // dx pixels of class (a, b) = a * sw + b as {C, wc[b], hc[a], N} (pixel
    // (sh*i + a, sw*j + b)), box {64, segw, 1, 1}, 128B swizzle: the epilogue's
    // TMA stores; encoded only for classes with pixels (bit c of dx_maps)
    CUtensorMap tmap_dx[4];
    int32_t dx_maps;
    const void *w;        // filter (KYXC), read to build the block-diagonal B
    void *dx;
    int32_t *status;
    int64_t wait_budget;
    int32_t N, C, Hi, Wi;
    int32_t sh, sw;
    int32_t cg;           // channels per group
    int32_t ntaps;        // Y * X
    int32_t ncls;         // sh * sw
    int32_t rows;         // staged dy rows per unit: 4 + (max - min row offset)
    int32_t segw;         // output columns per unit: 32 - (max - min column offset)
    int32_t oy_min, ox_min;
    int32_t stages;       // A stages (2..6)
    int32_t tmem_cols;    // TMEM allocation: two buffers of ncls x 64 columns, rounded up to a power of 2
    int32_t bands, segs;  // per image: ceil(rows of class a = 0 / 4), ceil(columns of class b = 0 / segw)
    int32_t units;        // units of one 64-channel block: N * bands * segs
    int32_t cblocks;      // C / 64
    int32_t hc[2], wc[2]; // output rows i / columns j of each row / column residue
    int32_t nwin;         // dy windows (column shift, staged-row offset) that some class's tap reads
    int32_t win[kBandMaxTaps];         // window: column shift | staged-row offset << 8
    int8_t win_tap[kBandMaxTaps][4];   // per window and class: the filter tap (y*X + x) reading it, or -1
#ifdef CBD_PHASE_TIMES
    unsigned long long *phase_log;
#endif
};

// narrow groups on tcgen05, dy staged once per band and reused by every tap
cudaError_t launch_tc_band(const BandParams &p, int grid, cudaStream_t s);
size_t tc_band_smem_bytes(int cg, int ncls, int nwin, int stage_bytes, int stages);

}  // namespace cbd
