// tc_fwd_sm103.cu -- forward convolution (bf16 NHWC x, KYXC w -> NHWC y) on the
// 5th-generation tensor cores, with the geometry of a dgrad plan.  It is the
// adjoint of the backward-data path (the forward kernels that the multi-kernel
// lowering of page "Backward data" is paired with), used to check
// <conv(x, w), dy> = <x, dgrad(dy, w)> on the GPU.
//
// Per group gi the forward pass is one implicit GEMM:
//   D[m, k] = sum over taps (y, x) and c < Cg of A[m, (y, x, c)] * B[(y, x, c), k]
//   A[m, (y, x, c)] = x[n, ho*sh - ph + y*dh, wo*sw - pw + x*dw, gi*Cg + c]  (zero outside x)
//   B[(y, x, c), k] = w[gi*Kg + k, y, x, c]
//   y[n, ho, wo, gi*Kg + k] = bf16_rne(D[m, k]),   m = (n, ho, wo)
// A comes from one TMA im2col map over x whose traversal strides are the
// convolution strides: its bounding box walks exactly the Wo x Ho base pixels
// (wo*sw - pw, ho*sh - ph) and the filter tap is the im2col offset
// (x*dw, y*dh).  w rows are c-contiguous, so B is K-major: one TMA box of
// 64 c x BN k per stage lands as BN 128-byte rows.  Tile 128 x BN, K step 64,
// one CTA per SM, persistent over all tiles.  Roles: warps 0-3 epilogue
// (TMEM -> bf16 -> dense y rows, shared with the dgrad kernels), warp 4 the A
// loads and the stage byte count, warp 5 TMEM allocation and the single-thread
// tcgen05.mma issue, warp 6 the B loads.  Every barrier wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "device_util.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace cbd {

template <int BN>
struct FwdCfg {
    static constexpr int STAGES = BN == 256 ? 4 : 6;
    static constexpr int A_BYTES = 128 * 64 * 2;
    static constexpr int B_BYTES = BN * 64 * 2;
    static constexpr int TMEM_COLS = 2 * BN;  // double-buffered accumulator
    static constexpr int STAGE_OUT_BYTES = 4 * 32 * 128;
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM = 1024 + STAGES * (A_BYTES + B_BYTES) + STAGE_OUT_BYTES + BAR_BYTES;
    static constexpr int MMA_WARP = 5;
    static constexpr int B_WARP = 6;
    static constexpr int THREADS = 32 * 7;
};

// kind::f16 instruction descriptor with both operands K-major
template <int BN>
__device__ __forceinline__ constexpr uint32_t idesc_bf16_kk() {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

struct FwdTile {
    int mb, nb, gi;
};
__device__ __forceinline__ FwdTile fwd_tile(const FwdParams &p, int t) {
    FwdTile r;
    r.mb = t % p.m_tiles;
    const int rest = t / p.m_tiles;
    r.nb = rest % p.n_tiles;
    r.gi = rest / p.n_tiles;
    return r;
}

template <int BN>
__global__ void __launch_bounds__(FwdCfg<BN>::THREADS, 1) tc_fwd_kernel(const __grid_constant__ FwdParams p) {
    using Cfg = FwdCfg<BN>;
    constexpr int S = Cfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + S * Cfg::A_BYTES;
    uint8_t *stage = sB + S * Cfg::B_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(stage + Cfg::STAGE_OUT_BYTES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * S + 4);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(tmem_slot + 1);

    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S);
    const uint32_t tfull0 = smem_u32(bars + 2 * S), tempty0 = smem_u32(bars + 2 * S + 2);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const Geom &g = p.g;
    const int num_kb = g.Y * g.X * p.kb_per_tap;  // k blocks of every tile

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);   // warp 4's arrive.expect_tx
            mbar_init(empty0 + 8 * s, 1);  // the stage's MMA commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull0 + 8 * b, 1);
            mbar_init(tempty0 + 8 * b, 128);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async_smem();
    }
    if (warp == Cfg::MMA_WARP) {
        tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
        tc_fence_before();
    }
    if (warp == 4 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_x)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_w)) : "memory");
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 4 || warp == Cfg::B_WARP) {
        // ------------------------------------------------------------ producers
        const bool do_a = warp == 4;
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true, issued = false;
            const int HoWo = g.Ho * g.Wo;
            for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
                const FwdTile tl = fwd_tile(p, t);
                const int m0 = tl.mb * 128;
                const int n0 = m0 / HoWo, rem = m0 - n0 * HoWo;
                const int bh = (rem / g.Wo) * g.sh - g.ph, bw = (rem % g.Wo) * g.sw - g.pw;  // base pixel of row 0
                for (int kb = 0; kb < num_kb; ++kb, ++it) {
                    const int tap = kb / p.kb_per_tap;
                    const int c0 = (kb - tap * p.kb_per_tap) * 64;
                    const int ty = tap / g.X, tx = tap - ty * g.X;
                    const uint32_t s = it % S, ph = (it / S) & 1;
                    if (!mbar_wait_bounded(empty0 + 8 * s, ph ^ 1, p.wait_budget, abort_flag, p.status,
                                           kDevTimeoutProducer)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full_s = full0 + 8 * s;
                    // (the B box may land before this arrive: the transaction count
                    // dips below zero while the single arrival is pending)
                    if (do_a) {
                        mbar_arrive_expect_tx(full_s, (uint32_t)(Cfg::A_BYTES + Cfg::B_BYTES));
                        tma_load_im2col(smem_u32(sA + s * Cfg::A_BYTES), &p.tmap_x, full_s, tl.gi * g.Cg + c0, bw, bh,
                                        n0, (uint16_t)(tx * g.dw), (uint16_t)(ty * g.dh));
                    } else {
                        tma_load_5d(smem_u32(sB + s * Cfg::B_BYTES), &p.tmap_w, full_s, c0, tx, ty, tl.nb * BN,
                                    tl.gi);
                    }
                    issued = true;
                }
            }
            if (!ok && issued) {
                for (int q = 0; q < 100; ++q) __nanosleep(1000);
            }
        }
        __syncwarp();
    } else if (warp == Cfg::MMA_WARP) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_kk<BN>();
            const uint64_t a_desc0 = smem_desc_sw128(smem_u32(sA), 16, 1024);
            const uint64_t b_desc0 = smem_desc_sw128(smem_u32(sB), 16, 1024);
            uint32_t it = 0, tc = 0;
            bool ok = true, issued = false;
            for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x, ++tc) {
                const uint32_t b = tc & 1, tph = (tc >> 1) & 1;
                if (!mbar_wait_bounded(tempty0 + 8 * b, tph ^ 1, p.wait_budget, abort_flag, p.status,
                                       kDevTimeoutMma)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + b * BN;
                for (int kb = 0; kb < num_kb; ++kb, ++it) {
                    const uint32_t s = it % S, ph = (it / S) & 1;
                    if (!mbar_wait_bounded(full0 + 8 * s, ph, p.wait_budget, abort_flag, p.status, kDevTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // both operands K-major: a 16-deep k step is 32 bytes along the row
                    const uint64_t ad0 = a_desc0 + (uint64_t)((s * Cfg::A_BYTES) >> 4);
                    const uint64_t bd0 = b_desc0 + (uint64_t)((s * Cfg::B_BYTES) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma(d_tmem, ad0 + (uint64_t)(2 * kk), bd0 + (uint64_t)(2 * kk), idesc, (kb | kk) != 0 ? 1u : 0u);
                    issued = true;
                    tc_commit(empty0 + 8 * s);
                }
                if (!ok) break;
                tc_commit(tfull0 + 8 * b);
            }
            if (!ok && issued) {
                for (int q = 0; q < 100; ++q) __nanosleep(1000);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue (warps 0-3)
        const int row = warp * 32 + lane;
        __nv_bfloat16 *y = static_cast<__nv_bfloat16 *>(p.y);
        const int64_t M = (int64_t)g.N * g.Ho * g.Wo;
        uint32_t tc = 0;
        for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++tc) {
            const FwdTile tl = fwd_tile(p, t);
            const uint32_t b = tc & 1, tph = (tc >> 1) & 1;
            bool ok = mbar_wait_bounded(tfull0 + 8 * b, tph, p.wait_budget, abort_flag, p.status, kDevTimeoutEpilogue);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const int64_t m = (int64_t)tl.mb * 128 + row;
            const bool rvalid = m < M;
            const int64_t off = rvalid ? m * g.K + (int64_t)tl.gi * g.Kg + (int64_t)tl.nb * BN : 0;
            const uint32_t tbase = tmem_base + ((uint32_t)(warp * 32) << 16) + b * BN;
            epilogue_rows<BN>(tbase, stage + warp * 4096, lane, rvalid, off, tl.nb * BN, g.Kg, y);
            tc_fence_before();
            mbar_arrive(tempty0 + 8 * b);
        }
    }

    __syncthreads();
    if (warp == Cfg::MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

template <int BN>
static cudaError_t launch_fwd_bn(const FwdParams &p, int grid, cudaStream_t s) {
    using Cfg = FwdCfg<BN>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(tc_fwd_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    tc_fwd_kernel<BN><<<grid, Cfg::THREADS, Cfg::SMEM, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_fwd(const FwdParams &p, int bn, int grid, cudaStream_t s) {
    if (grid <= 0 || p.total_tiles <= 0) return cudaSuccess;
    return bn == 256 ? launch_fwd_bn<256>(p, grid, s) : launch_fwd_bn<128>(p, grid, s);
}

}  // namespace cbd
