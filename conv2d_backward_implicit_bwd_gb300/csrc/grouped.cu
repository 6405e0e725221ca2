// grouped.cu -- bf16 NHWC/KYXC dgrad for narrow groups (C/G = K/G = 8 or 16,
// G a multiple of 8), e.g. the grouped 3x3 layers of ResNeXt-style networks
// (a workload named on page "[igemm_dynamic] v4r1 bwd dynamic kernel").
//
// With 8 channels per group the arithmetic intensity is ~14 FLOP per byte:
// the kernel is bound by HBM traffic (dy read, dx written), not by math, so it
// runs on CUDA cores and is built around coalescing instead of a padded GEMM.
//   * A warp owns 8 consecutive groups and 8 (16-channel groups: 4) dx pixels
//     of one row that belong to the same column residue class (wi = r, r + sw,
//     ...; the v4r1 split of pages "Backward data" and "[igemm_dynamic] v4r1
//     bwd dynamic kernel" applied per pixel), so all share the class's taps.
//   * Lane = 8 * pixel slot + group: for every pixel the 8 lanes of a slot load
//     and store one full 128-byte line (8 groups x 8 bf16 channels).
//   * w is staged once per CTA in shared memory as fp32 [y][x][k][c/4][g]; the
//     8 groups of a warp read one 128-byte wavefront per chunk, reused for all
//     of the lane's pixels.  Accumulators stay small (8 fp32 per pixel), so
//     occupancy stays high.
//   * A row's residue class, taps and first dy row come from small tables of
//     the planner's class decomposition: no per-pixel divisions.
//   * Pixels that no tap reaches are written as +0 by the same pass (no
//     separate fill).
// Accumulation in fp32 (packed fma.rn.f32x2: two output channels per
// instruction, each an ordinary fp32 fused multiply-add), one RNE rounding to
// bf16 per output.
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>

#include "internal.h"

namespace cbd {

__device__ __forceinline__ void bf16x8_to_float(const uint4 &u, float *f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint4 float_to_bf16x8(const float *f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Warp layout: lane = 8 * slot + gl, slot in [0, 4) picks pixels, gl in [0, 8)
// one of 8 consecutive groups.  A warp item is one dx row segment: image n,
// row hi, column residue r (pixels wi = r, r + sw, ...) and 8 groups; it walks
// the segment 4*PPL pixels at a time, each lane owning PPL of them.
template <int CG, int PPL>
__global__ void __launch_bounds__(256) grouped_dgrad_kernel(const __grid_constant__ GroupedParams p) {
    constexpr int V = CG / 8;   // 16-byte bf16 vectors per group row of dy / dx
    constexpr int F4 = CG / 4;  // float4 chunks per group row of w
    constexpr int PIX = 4 * PPL;
    extern __shared__ float4 wsm[];  // w as fp32 [y][x][k][chunk][g] (float4 per entry)
    const Geom &g = p.g;
    const uint4 *w = static_cast<const uint4 *>(p.w);
    const uint4 *dy = static_cast<const uint4 *>(p.dy);
    uint4 *dx = static_cast<uint4 *>(p.dx);

    // stage w: global bf16 [g*Kg + k][y][x][c] -> shared fp32 [y][x][k][c/4][g]
    const int rows = g.K * g.Y * g.X;  // (k_global, y, x) rows of CG channels
    for (int e = threadIdx.x; e < rows * V; e += blockDim.x) {
        const int v = e % V, rr = e / V;
        const int x = rr % g.X, y = (rr / g.X) % g.Y, kg = rr / (g.X * g.Y);
        const int gi = kg / CG, k = kg % CG;
        float f[8];
        bf16x8_to_float(w[e], f);
        const int base = (((y * g.X + x) * CG + k) * F4 + 2 * v) * g.G + gi;
        wsm[base] = make_float4(f[0], f[1], f[2], f[3]);
        wsm[base + g.G] = make_float4(f[4], f[5], f[6], f[7]);
    }
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int gl = lane & 7, slot = lane >> 3;
    const int warps = gridDim.x * (blockDim.x >> 5);
    const int total = g.N * g.Hi * g.sw * p.gblocks;  // < 2^31 (checked by the planner)
    for (int item = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); item < total; item += warps) {
        const int gb = item % p.gblocks;
        int rest = item / p.gblocks;
        const int r = rest % g.sw;
        rest /= g.sw;
        const int hi = rest % g.Hi, n = rest / g.Hi;
        if (r >= g.Wi) continue;
        const int gi = gb * 8 + gl;
        // residue classes of this row and column: ty/tx, taps, and the class index
        // of the first pixel (ht for the row; wt of pixel wi = r for the column)
        const int rc = p.row_class[hi % g.sh], cc = p.col_class[r];
        const int taps_y = rc >> 16, ty = rc & 0xFFFF;
        const int taps_x = cc >> 16, tx = cc & 0xFFFF;
        const int ht = (hi + g.ph - ty * g.dh) / g.sh;   // exact when taps_y > 0
        const int wt0 = (r + g.pw - tx * g.dw) / g.sw;   // exact when taps_x > 0; +1 per pixel step
        const int cnt = (g.Wi - r + g.sw - 1) / g.sw;    // pixels of this residue in the row
        uint4 *orow = dx + (((int64_t)n * g.Hi + hi) * g.Wi * g.C + (int64_t)gi * CG) / 8;
        const int kv = g.K / 8;  // dy pixel stride in 16-byte vectors
        for (int p0 = 0; p0 < cnt; p0 += PIX) {
            // accumulators as fp32 pairs (channels c, c + 1): one packed f32x2 FMA
            // updates two outputs
            uint64_t acc[PPL][CG / 2];
#pragma unroll
            for (int q = 0; q < PPL; ++q)
#pragma unroll
                for (int c = 0; c < CG / 2; ++c) acc[q][c] = 0ull;
            for (int jj = 0; jj < taps_y; ++jj) {
                const int ho = ht - jj * g.DH;
                if (ho < 0 || ho >= g.Ho) continue;
                const int y = ty + g.YT * jj;
                const int64_t rowv = ((int64_t)n * g.Ho + ho) * g.Wo * kv + gi * V;
                for (int ii = 0; ii < taps_x; ++ii) {
                    const int x = tx + g.XT * ii;
                    uint4 raw[PPL][V];
#pragma unroll
                    for (int q = 0; q < PPL; ++q) {
                        const int pq = p0 + slot + 4 * q;
                        const int wo = wt0 + pq - ii * g.DW;
                        const bool ok = pq < cnt && wo >= 0 && wo < g.Wo;
#pragma unroll
                        for (int v = 0; v < V; ++v)
                            raw[q][v] = ok ? dy[rowv + (int64_t)wo * kv + v] : make_uint4(0u, 0u, 0u, 0u);
                    }
                    const ulonglong2 *wt =
                        reinterpret_cast<const ulonglong2 *>(wsm) + (y * g.X + x) * CG * F4 * g.G + gi;
#pragma unroll
                    for (int k = 0; k < CG; ++k) {
                        uint64_t wp[CG / 2];
#pragma unroll
                        for (int f = 0; f < F4; ++f) {
                            const ulonglong2 a = wt[(k * F4 + f) * g.G];
                            wp[2 * f] = a.x;
                            wp[2 * f + 1] = a.y;
                        }
#pragma unroll
                        for (int q = 0; q < PPL; ++q) {
                            const uint4 u = raw[q][k / 8];
                            const uint32_t word = (k % 8) < 2 ? u.x : (k % 8) < 4 ? u.y : (k % 8) < 6 ? u.z : u.w;
                            const uint32_t bits = (k & 1) ? (word & 0xFFFF0000u) : (word << 16);
                            uint64_t d2;
                            asm("mov.b64 %0, {%1, %1};" : "=l"(d2) : "r"(bits));
#pragma unroll
                            for (int c = 0; c < CG / 2; ++c)
                                asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc[q][c]) : "l"(d2), "l"(wp[c]));
                        }
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < PPL; ++q) {
                const int pq = p0 + slot + 4 * q;
                if (pq >= cnt) continue;
                float f[CG];
#pragma unroll
                for (int c = 0; c < CG / 2; ++c) {
                    f[2 * c] = __uint_as_float((uint32_t)acc[q][c]);
                    f[2 * c + 1] = __uint_as_float((uint32_t)(acc[q][c] >> 32));
                }
                uint4 *o = orow + (int64_t)(r + g.sw * pq) * g.C / 8;
#pragma unroll
                for (int v = 0; v < V; ++v) o[v] = float_to_bf16x8(&f[8 * v]);
            }
        }
    }
}

cudaError_t launch_grouped(const GroupedParams &p, int num_sms, cudaStream_t s) {
    const size_t smem = (size_t)p.g.K * p.g.Y * p.g.X * p.g.Cg * 4;  // fp32 copy of w
    const int per_sm = (int)std::max<size_t>(1, std::min<size_t>(4, (size_t)(220 * 1024) / std::max<size_t>(smem, 1)));
    const int blocks = (num_sms > 0 ? num_sms : 148) * per_sm;
    if (p.g.Cg == 8) {
        cudaError_t e = cudaFuncSetAttribute(grouped_dgrad_kernel<8, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        grouped_dgrad_kernel<8, 2><<<blocks, 256, smem, s>>>(p);
    } else {
        cudaError_t e = cudaFuncSetAttribute(grouped_dgrad_kernel<16, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        grouped_dgrad_kernel<16, 1><<<blocks, 256, smem, s>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace cbd
