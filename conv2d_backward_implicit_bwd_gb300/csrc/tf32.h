// tf32.h -- launchers of the fp32 tensor-core path (three-term TF32 split)
// and of the 4-byte layout transposes around it.
#pragma once
#include <stdint.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace cbd {

// Tile of the fp32 tensor-core kernel: 128 dx pixels x 128 channels, k step of
// 32 channels (one 128-byte row per operand row).
constexpr int kTf32BN = 128;
constexpr int kTf32BK = 32;
// fp32 problems below this many useful FLOP stay on the CUDA cores, where one
// launch costs less than the filter split plus the tensor-core kernel.
constexpr double kTf32MinFlop = 1e9;

// Split the filter into the two fp32 arrays the fp32 tensor-core kernel reads,
// laid out [G][C/G][Y][X][K/G] (k contiguous, so B is K-major):
//   hi = w rounded to the nearest value with a 10-bit mantissa (ties to even),
//   lo = w - hi (exact in fp32).
// `w` is KYXC ([K][Y][X][C/G]) when gkcyx == 0, GKCYX ([K][C/G][Y][X]) otherwise.
cudaError_t launch_tf32_split_w(const float *w, float *w_hi, float *w_lo, const Geom &g, int gkcyx, int num_sms,
                                cudaStream_t s);

// The fp32 NHWC dgrad kernel.  Uses TcParams with these meanings:
//   tmap_a[ci]   dy (fp32 NHWC) as im2col {K, Wo, Ho, N}, 32 channels x 128 pixels
//   tmap_w       w_hi as 5-D {Kg, X, Y, Cg, G}, box {32, 1, 1, 128, 1}
//   tmap_w_half  w_lo, same view
//   kb_per_tap   ceil(Kg / 32), n_tiles ceil(Cg / 128)
cudaError_t launch_tf32(const TcParams &p, int grid, cudaStream_t s);

// out[b][c][r] = in[b][r][c] for 4-byte elements (r < R, c < Cc).
cudaError_t launch_transpose_b32(const void *in, void *out, int64_t batch, int64_t R, int64_t Cc, int num_sms,
                                 cudaStream_t s);

}  // namespace cbd
