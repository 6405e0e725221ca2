// simt.cu -- CUDA-core kernels: the dx fill, the tiled SIMT implicit GEMM
// (fp32 path, and the bf16 fallback for shapes the tensor-core kernel does
// not take), and the bounded-wait self-test.
#include <cuda_bf16.h>
#include <stdint.h>

#include "device_util.cuh"
#include "internal.h"
#include "tf32.h"

namespace cbd {

// ---------------------------------------------------------------------------
// Fill: dx := +0 at every pixel that no sub-GEMM writes.  A pixel is written
// iff its row residue (hi % sh) and column residue (wi % sw) both belong to a
// class with at least one tap; the planner encodes those residues as bit
// masks.  The pages never state the zero-initialisation; it follows from dx
// being fully overwritten (torch-IR `torch.overwrite.tensor.contents` on page
// "Non-unit stride input backward different input and dispatches between BOO
// and Fusilli").  NHWC: one 16-byte store per 8 bf16 / 4 fp32 channels of an
// uncovered pixel (consecutive threads -> consecutive chunks).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) fill_kernel(const FillParams p) {
    if (p.vec16) {
        // one block per dx row (n, hi): a row no class writes is one contiguous
        // run of Wi*C elements; in a written row only the uncovered columns
        // (C elements each) are zeroed
        const uint32_t cpp = (uint32_t)((int64_t)p.C * p.esize / 16);  // 16-byte chunks per pixel
        const uint32_t cpr = cpp * (uint32_t)p.Wi;                     // chunks per row
        uint4 *out = reinterpret_cast<uint4 *>(p.dx);
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        const uint32_t rows = (uint32_t)p.N * (uint32_t)p.Hi;
        for (uint32_t r = blockIdx.x; r < rows; r += gridDim.x) {
            const uint32_t hi = r % (uint32_t)p.Hi;
            uint4 *row = out + (size_t)r * cpr;
            if (!((p.cov_h >> (hi % (uint32_t)p.sh)) & 1ull)) {
                for (uint32_t u = threadIdx.x; u < cpr; u += blockDim.x) row[u] = z;
            } else if (p.cov_w != ~0ull) {
                for (uint32_t u = threadIdx.x; u < cpr; u += blockDim.x) {
                    const uint32_t wi = u / cpp;
                    if (!((p.cov_w >> (wi % (uint32_t)p.sw)) & 1ull)) row[u] = z;
                }
            }
        }
        return;
    }
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t first = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t total = (int64_t)p.N * p.C * p.Hi * p.Wi;
    for (int64_t e = first; e < total; e += stride) {
        int hi, wi;
        if (p.layout == 0) {
            wi = (int)(e % p.Wi);
            hi = (int)((e / p.Wi) % p.Hi);
        } else {
            int64_t pix = e / p.C;
            wi = (int)(pix % p.Wi);
            hi = (int)((pix / p.Wi) % p.Hi);
        }
        bool cov = ((p.cov_h >> (hi % p.sh)) & 1ull) && ((p.cov_w >> (wi % p.sw)) & 1ull);
        if (!cov) {
            if (p.esize == 4)
                reinterpret_cast<float *>(p.dx)[e] = 0.f;
            else
                reinterpret_cast<uint16_t *>(p.dx)[e] = 0;
        }
    }
}

cudaError_t launch_fill(const FillParams &p, int num_sms, cudaStream_t s) {
    int64_t blocks;
    if (p.vec16) {
        blocks = (int64_t)p.N * p.Hi;  // one block per dx row
    } else {
        blocks = ((int64_t)p.N * p.C * p.Hi * p.Wi + 255) / 256;
    }
    int64_t cap = (int64_t)(num_sms > 0 ? num_sms : 148) * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    fill_kernel<<<(unsigned)blocks, 256, 0, s>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// SIMT implicit GEMM over all sub-GEMMs in one launch.  One 64x64 output tile
// per block: rows are the class's (n, ht, wt) positions, columns the input
// channels of one group.  The reduction runs over (tap, k) with
//   A[m, (tap, k)] = dy[n, gi*Kg + k, ht - j*DH, wt - i*DW]   (0 outside dy)
//   B[(tap, k), c] = w[gi*Kg + k, c, ty + YT*j, tx + XT*i]
// and the result goes to dx[n, gi*Cg + c, ht*sh + ty*dh - ph, wt*sw + tx*dw - pw].
// fp32 accumulation; each thread owns a 4x4 micro-tile.
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ float ld_as_float(const T *p, int64_t i);
template <>
__device__ __forceinline__ float ld_as_float<float>(const float *p, int64_t i) {
    return __ldg(p + i);
}
template <>
__device__ __forceinline__ float ld_as_float<__nv_bfloat16>(const __nv_bfloat16 *p, int64_t i) {
    return __bfloat162float(p[i]);
}
template <typename T>
__device__ __forceinline__ void st_from_float(T *p, int64_t i, float v);
template <>
__device__ __forceinline__ void st_from_float<float>(float *p, int64_t i, float v) {
    p[i] = v;
}
template <>
__device__ __forceinline__ void st_from_float<__nv_bfloat16>(__nv_bfloat16 *p, int64_t i, float v) {
    p[i] = __float2bfloat16_rn(v);
}

template <typename T>
__global__ void __launch_bounds__(256) simt_dgrad_kernel(const __grid_constant__ SimtParams p) {
    constexpr int BM = 64, BN = 64, BK = 16;
    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[BK][BN + 4];
    const Geom &g = p.g;
    const Strides &st = p.st;
    const T *dy = static_cast<const T *>(p.dy);
    const T *w = static_cast<const T *>(p.w);
    T *dx = static_cast<T *>(p.dx);

    const int tile = blockIdx.x;
    int ci = 0;
    for (int i = 1; i < p.num_classes; ++i)
        if (tile >= p.cls[i].tile_begin) ci = i;
    const ClassDesc &c = p.cls[ci];
    const int local = tile - c.tile_begin;
    const int nb = local % p.n_tiles;
    const int rest = local / p.n_tiles;
    const int mb = rest % c.m_tiles;
    const int gi = rest / c.m_tiles;

    const int tid = threadIdx.x;
    const int HTWT = c.HT * c.WT;
    const int Kred = c.taps_y * c.taps_x * g.Kg;

    // the A row this thread loads
    const int arow = tid % BM;
    const int am = mb * BM + arow;
    int an = -1, aht = 0, awt = 0;
    if (am < c.M) {
        an = am / HTWT;
        int rem = am - an * HTWT;
        aht = c.ht_lo + rem / c.WT;
        awt = c.wt_lo + rem % c.WT;
    }
    // the B column this thread loads
    const int bcol = tid % BN;
    const int bc = nb * BN + bcol;

    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    const int tr = tid / 16, tc = tid % 16;
    for (int r0 = 0; r0 < Kred; r0 += BK) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int kk = tid / BM + 4 * q;
            const int r = r0 + kk;
            float va = 0.f, vb = 0.f;
            if (r < Kred) {
                const int tap = r / g.Kg, k = r - tap * g.Kg;
                const int j = tap / c.taps_x, i = tap - j * c.taps_x;
                if (an >= 0) {
                    const int ho = aht - j * g.DH, wo = awt - i * g.DW;
                    if (ho >= 0 && ho < g.Ho && wo >= 0 && wo < g.Wo)
                        va = ld_as_float<T>(dy, an * st.dy_n + (int64_t)(gi * g.Kg + k) * st.dy_k + ho * st.dy_h +
                                                    wo * st.dy_w);
                }
                if (bc < g.Cg) {
                    const int y = c.ty + g.YT * j, x = c.tx + g.XT * i;
                    vb = ld_as_float<T>(w, (int64_t)(gi * g.Kg + k) * st.w_k + bc * st.w_c + y * st.w_y + x * st.w_x);
                }
            }
            As[kk][arow] = va;
            Bs[kk][bcol] = vb;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][tr * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tc * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = mb * BM + tr * 4 + i;
        if (m >= c.M) continue;
        const int n = m / HTWT;
        const int rem = m - n * HTWT;
        const int hi = (c.ht_lo + rem / c.WT) * g.sh + c.ty * g.dh - g.ph;
        const int wi = (c.wt_lo + rem % c.WT) * g.sw + c.tx * g.dw - g.pw;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int cc = nb * BN + tc * 4 + j;
            if (cc >= g.Cg) continue;
            st_from_float<T>(dx, n * st.dx_n + (int64_t)(gi * g.Cg + cc) * st.dx_c + hi * st.dx_h + wi * st.dx_w,
                             acc[i][j]);
        }
    }
}

// fp32 variant: 64 x BN tiles (BN = 64, or 32 where C/G <= 32) with a 4-stage
// cp.async pipeline of 16-deep slices -- each thread gathers its A and B
// elements of a slice with 4-byte copies (zero-filled outside dy, past the
// class's reduction or past C/G) while the FMAs run on the slices already in
// shared memory, so the reduction pays one memory latency instead of one per
// slice.  The 16 k of a slice are split over four groups of 64 threads:
// thread (kg, lt) accumulates an 8 x BN/8 micro-tile over k = 4kg .. 4kg+3 of
// every slice (8 + BN/8 shared-memory reads per 8 x BN/8 FMAs), and the four
// partial tiles are summed at the end in a fixed order ((0 + 2) + (1 + 3)).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

template <int BN>
__global__ void __launch_bounds__(256) simt_dgrad_f32_kernel(const __grid_constant__ SimtParams p) {
    constexpr int BM = 64, BK = 16, S = 4, TM = 8, TN = BN / 8;
    constexpr int A_LD = BM + 4, B_LD = BN + 4;  // row pitch (floats): 16-byte aligned rows
    constexpr int AQ = BM * BK / 256, BQ = BN * BK / 256;  // elements per thread and slice
    __shared__ __align__(16) float smem[S * BK * (A_LD + B_LD)];
    static_assert(2 * BM * BN <= S * BK * (A_LD + B_LD), "reduction buffer");
    float(*As)[BK][A_LD] = reinterpret_cast<float(*)[BK][A_LD]>(smem);
    float(*Bs)[BK][B_LD] = reinterpret_cast<float(*)[BK][B_LD]>(smem + S * BK * A_LD);
    const Geom &g = p.g;
    const Strides &st = p.st;
    const float *dy = static_cast<const float *>(p.dy);
    const float *w = static_cast<const float *>(p.w);
    float *dx = static_cast<float *>(p.dx);

    const int tile = blockIdx.x;
    int ci = 0;
    for (int i = 1; i < p.num_classes; ++i)
        if (tile >= p.cls[i].tile_begin) ci = i;
    const ClassDesc &c = p.cls[ci];
    const int local = tile - c.tile_begin;
    const int nb = local % p.n_tiles;
    const int rest = local / p.n_tiles;
    const int mb = rest % c.m_tiles;
    const int gi = rest / c.m_tiles;

    const int tid = threadIdx.x;
    const int HTWT = c.HT * c.WT;
    const int Kred = c.taps_y * c.taps_x * g.Kg;
    const int nslices = (Kred + BK - 1) / BK;

    // the A row and the B column this thread gathers
    const int arow = tid % BM;
    const int am = mb * BM + arow;
    int an = -1, aht = 0, awt = 0;
    if (am < c.M) {
        an = am / HTWT;
        const int rem = am - an * HTWT;
        aht = c.ht_lo + rem / c.WT;
        awt = c.wt_lo + rem % c.WT;
    }
    const int bcol = tid % BN;
    const int bc = nb * BN + bcol;
    const float *dy_n = dy + (an >= 0 ? (int64_t)an * st.dy_n : 0) + (int64_t)gi * g.Kg * st.dy_k;
    const float *w_g = w + (int64_t)gi * g.Kg * st.w_k + (int64_t)(bc < g.Cg ? bc : 0) * st.w_c;

    // reduction index r = tap*Kg + k of each element this thread issues next,
    // kept as (r, k, i, j) counters advanced by BK per slice (no divisions in
    // the loop); A element q sits at slice row tid / BM + (256 / BM) q, B
    // element q at tid / BN + (256 / BN) q
    struct Ctr {
        int r, k, i, j;
    };
    auto start = [&](int r) {
        Ctr q;
        const int tap = r / g.Kg;
        q.r = r;
        q.k = r - tap * g.Kg;
        q.j = tap / c.taps_x;
        q.i = tap - q.j * c.taps_x;
        return q;
    };
    auto advance = [&](Ctr &q) {
        q.r += BK;
        q.k += BK;
        while (q.k >= g.Kg) {
            q.k -= g.Kg;
            if (++q.i == c.taps_x) {
                q.i = 0;
                ++q.j;
            }
        }
    };
    Ctr qa[AQ], qb[BQ];
#pragma unroll
    for (int q = 0; q < AQ; ++q) qa[q] = start(tid / BM + (256 / BM) * q);
#pragma unroll
    for (int q = 0; q < BQ; ++q) qb[q] = start(tid / BN + (256 / BN) * q);
    auto issue = [&](int slice) {
        const int sb = slice % S;
#pragma unroll
        for (int q = 0; q < AQ; ++q) {
            const int kk = tid / BM + (256 / BM) * q;
            const float *src = dy;
            bool v = false;
            if (qa[q].r < Kred && an >= 0) {
                const int ho = aht - qa[q].j * g.DH, wo = awt - qa[q].i * g.DW;
                v = ho >= 0 && ho < g.Ho && wo >= 0 && wo < g.Wo;
                if (v) src = dy_n + (int64_t)qa[q].k * st.dy_k + (int64_t)ho * st.dy_h + (int64_t)wo * st.dy_w;
            }
            cp_async_4(smem_u32(&As[sb][kk][arow]), src, v ? 4u : 0u);
            advance(qa[q]);
        }
#pragma unroll
        for (int q = 0; q < BQ; ++q) {
            const int kk = tid / BN + (256 / BN) * q;
            const float *src = w;
            const bool v = qb[q].r < Kred && bc < g.Cg;
            if (v)
                src = w_g + (int64_t)qb[q].k * st.w_k + (int64_t)(c.ty + g.YT * qb[q].j) * st.w_y +
                      (int64_t)(c.tx + g.XT * qb[q].i) * st.w_x;
            cp_async_4(smem_u32(&Bs[sb][kk][bcol]), src, v ? 4u : 0u);
            advance(qb[q]);
        }
    };

    // Kg a multiple of BK: every slice lies within one tap, so a thread's
    // elements of a slice share the tap's bounds check and base address and
    // step by whole rows of k (counters (k0, i, j) of the next slice to issue)
    const bool tap_slices = g.Kg % BK == 0;
    int fk = 0, fi = 0, fj = 0;
    auto issue_tap = [&](int slice) {
        const int sb = slice % S;
        const int ho = aht - fj * g.DH, wo = awt - fi * g.DW;
        const bool va = an >= 0 && ho >= 0 && ho < g.Ho && wo >= 0 && wo < g.Wo;
        const float *pa = va ? dy_n + (int64_t)(fk + tid / BM) * st.dy_k + (int64_t)ho * st.dy_h + (int64_t)wo * st.dy_w
                             : dy;
        const int64_t da = va ? (int64_t)(256 / BM) * st.dy_k : 0;
#pragma unroll
        for (int q = 0; q < AQ; ++q)
            cp_async_4(smem_u32(&As[sb][tid / BM + (256 / BM) * q][arow]), pa + q * da, va ? 4u : 0u);
        const bool vb = bc < g.Cg;
        const float *pb = vb ? w_g + (int64_t)(fk + tid / BN) * st.w_k + (int64_t)(c.ty + g.YT * fj) * st.w_y +
                                   (int64_t)(c.tx + g.XT * fi) * st.w_x
                             : w;
        const int64_t db = vb ? (int64_t)(256 / BN) * st.w_k : 0;
#pragma unroll
        for (int q = 0; q < BQ; ++q)
            cp_async_4(smem_u32(&Bs[sb][tid / BN + (256 / BN) * q][bcol]), pb + q * db, vb ? 4u : 0u);
        fk += BK;
        if (fk == g.Kg) {
            fk = 0;
            if (++fi == c.taps_x) {
                fi = 0;
                ++fj;
            }
        }
    };

    const int kg = tid >> 6, lt = tid & 63, tr = lt >> 3, tc = lt & 7;
    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

    for (int sl = 0; sl < S - 1; ++sl) {
        if (sl < nslices) {
            if (tap_slices)
                issue_tap(sl);
            else
                issue(sl);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    for (int sl = 0; sl < nslices; ++sl) {
        asm volatile("cp.async.wait_group %0;" ::"n"(S - 2) : "memory");  // slice sl has landed
        __syncthreads();
        if (sl + S - 1 < nslices) {  // refills the buffer read in iteration sl - 1
            if (tap_slices)
                issue_tap(sl + S - 1);
            else
                issue(sl + S - 1);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        const int sb = sl % S;
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
            const int kk = kg * 4 + k4;
            float a[TM], b[TN];
#pragma unroll
            for (int i = 0; i < TM; i += 4) {
                const float4 v = *reinterpret_cast<const float4 *>(&As[sb][kk][tr * TM + i]);
                a[i] = v.x, a[i + 1] = v.y, a[i + 2] = v.z, a[i + 3] = v.w;
            }
#pragma unroll
            for (int j = 0; j < TN; j += 4) {
                const float4 v = *reinterpret_cast<const float4 *>(&Bs[sb][kk][tc * TN + j]);
                b[j] = v.x, b[j + 1] = v.y, b[j + 2] = v.z, b[j + 3] = v.w;
            }
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();

    // sum the four k groups' partial tiles: (0 + 2) + (1 + 3), then the final
    // tile in red[BM*BN ..)
    float *red = smem;
    auto put = [&](float *dst) {
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) dst[(tr * TM + i) * BN + tc * TN + j] = acc[i][j];
    };
    auto add = [&](const float *src) {
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] += src[(tr * TM + i) * BN + tc * TN + j];
    };
    if (kg >= 2) put(red + (kg - 2) * BM * BN);
    __syncthreads();
    if (kg < 2) add(red + kg * BM * BN);
    __syncthreads();
    if (kg == 1) put(red);
    __syncthreads();
    if (kg == 0) {
        add(red);
        put(red + BM * BN);
    }
    __syncthreads();

    // store the tile, consecutive threads on dx's contiguous index (channels
    // for NHWC, pixels for NCHW)
    const float *fin = red + BM * BN;
    const bool chan_inner = st.dx_c == 1;
#pragma unroll 4
    for (int e = tid; e < BM * BN; e += 256) {
        const int row = chan_inner ? e / BN : e % BM;
        const int col = chan_inner ? e % BN : e / BM;
        const int m = mb * BM + row, cc = nb * BN + col;
        if (m >= c.M || cc >= g.Cg) continue;
        const int n = m / HTWT;
        const int rem = m - n * HTWT;
        const int hi = (c.ht_lo + rem / c.WT) * g.sh + c.ty * g.dh - g.ph;
        const int wi = (c.wt_lo + rem % c.WT) * g.sw + c.tx * g.dw - g.pw;
        dx[n * st.dx_n + (int64_t)(gi * g.Cg + cc) * st.dx_c + hi * st.dx_h + wi * st.dx_w] = fin[row * BN + col];
    }
}

cudaError_t launch_simt(const SimtParams &p, int dtype, cudaStream_t s) {
    if (p.total_tiles <= 0) return cudaSuccess;
    if (dtype == 1)
        simt_dgrad_kernel<__nv_bfloat16><<<p.total_tiles, 256, 0, s>>>(p);
    else if (p.bn == 32)
        simt_dgrad_f32_kernel<32><<<p.total_tiles, 256, 0, s>>>(p);
    else
        simt_dgrad_f32_kernel<64><<<p.total_tiles, 256, 0, s>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Self-test of the bounded wait: a barrier that nothing arrives on.
// ---------------------------------------------------------------------------
__global__ void selftest_wait_kernel(int32_t *status, int64_t budget) {
    __shared__ alignas(8) uint64_t bar;
    __shared__ int32_t abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        (void)mbar_wait_bounded(smem_u32(&bar), 0, budget, &abort_flag, status, kDevTimeoutSelftest);
    }
}

cudaError_t launch_selftest_wait(int32_t *status, int64_t budget, cudaStream_t s) {
    selftest_wait_kernel<<<1, 32, 0, s>>>(status, budget);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Layout transposes for NCHW/GKCYX problems on the tensor-core paths (2-byte
// elements for bf16, 4-byte for fp32): out[b][c][r] = in[b][r][c] (r < R,
// c < Cc), 64x64 tiles through shared memory so that both the reads and the
// writes run along contiguous rows.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) transpose_kernel(const T *__restrict__ in, T *__restrict__ out, int64_t batch,
                                                        int64_t R, int64_t Cc) {
    __shared__ T t[64][64 + 4 / sizeof(T)];  // one extra 4-byte word per row: conflict-free columns
    const int64_t tr_n = (R + 63) / 64, tc_n = (Cc + 63) / 64;
    const int64_t tiles = batch * tr_n * tc_n;
    const int x = threadIdx.x & 31, y = threadIdx.x >> 5;  // 32 x 8 threads
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const int64_t tc = tile % tc_n, rest = tile / tc_n;
        const int64_t tr = rest % tr_n, b = rest / tr_n;
        const T *src = in + b * R * Cc;
        T *dst = out + b * R * Cc;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int64_t r = tr * 64 + y + 8 * k;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t c = tc * 64 + x + 32 * h;
                t[y + 8 * k][x + 32 * h] = (r < R && c < Cc) ? src[r * Cc + c] : (T)0;
            }
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int64_t c = tc * 64 + y + 8 * k;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t r = tr * 64 + x + 32 * h;
                if (r < R && c < Cc) dst[c * R + r] = t[x + 32 * h][y + 8 * k];
            }
        }
        __syncthreads();
    }
}

// Narrow inner dimension (Cc < 32, e.g. the Y*X taps of a filter): a block
// takes a slab of up to 64 rows of one batch item, which is contiguous in the
// input (at most 64*31 elements), stages it in shared memory with all of a
// thread's loads in flight at once, and writes its Cc output rows of up to 64
// contiguous elements each.
constexpr int kNarrowRows = 64;
template <typename T>
__global__ void __launch_bounds__(256) transpose_narrow_kernel(const T *__restrict__ in, T *__restrict__ out,
                                                               int64_t batch, int64_t R, int64_t Cc) {
    constexpr int PER = kNarrowRows * 32 / 256;  // elements per thread, upper bound
    __shared__ T slab[kNarrowRows * 32];
    // a tensor holds fewer than 2^31 elements, so slab indices fit 32 bits
    const int slabs_r = (int)((R + kNarrowRows - 1) / kNarrowRows);
    const int slabs = (int)batch * slabs_r;
    const int cc = (int)Cc;
    for (int sl = blockIdx.x; sl < slabs; sl += gridDim.x) {
        const int64_t b = sl / slabs_r;
        const int64_t r0 = (int64_t)(sl - (int)b * slabs_r) * kNarrowRows;
        const int nr = (int)(R - r0 < kNarrowRows ? R - r0 : kNarrowRows);
        const int n = nr * cc;
        const T *src = in + (b * R + r0) * Cc;
        T v[PER];
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            const int e = threadIdx.x + 256 * q;
            if (256 * q < n) v[q] = e < n ? src[e] : (T)0;  // (block-uniform skip of empty passes)
        }
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            const int e = threadIdx.x + 256 * q;
            if (256 * q < n && e < n) slab[e] = v[q];
        }
        __syncthreads();
        T *dst = out + b * Cc * R + r0;
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            if (256 * q >= kNarrowRows * cc) break;
            const int e = threadIdx.x + 256 * q;  // output row c = e / 64, element r = e % 64
            const int c = e / kNarrowRows, r = e % kNarrowRows;
            if (c < cc && r < nr) dst[(int64_t)c * R + r] = slab[r * cc + c];
        }
        __syncthreads();
    }
}

template <typename T>
static cudaError_t launch_transpose(const void *in, void *out, int64_t batch, int64_t R, int64_t Cc, int num_sms,
                                   cudaStream_t s) {
    const int64_t tiles = batch * ((R + 63) / 64) * ((Cc + 63) / 64);
    if (tiles <= 0) return cudaSuccess;
    const int64_t cap = (int64_t)(num_sms > 0 ? num_sms : 148) * 8;
    if (Cc < 32) {
        const int64_t blocks = batch * ((R + kNarrowRows - 1) / kNarrowRows);
        transpose_narrow_kernel<T><<<(unsigned)(blocks < cap ? blocks : cap), 256, 0, s>>>(
            static_cast<const T *>(in), static_cast<T *>(out), batch, R, Cc);
        return cudaGetLastError();
    }
    transpose_kernel<T><<<(unsigned)(tiles < cap ? tiles : cap), 256, 0, s>>>(static_cast<const T *>(in),
                                                                              static_cast<T *>(out), batch, R, Cc);
    return cudaGetLastError();
}

cudaError_t launch_transpose_b16(const void *in, void *out, int64_t batch, int64_t R, int64_t Cc, int num_sms,
                                 cudaStream_t s) {
    return launch_transpose<uint16_t>(in, out, batch, R, Cc, num_sms, s);
}

cudaError_t launch_transpose_b32(const void *in, void *out, int64_t batch, int64_t R, int64_t Cc, int num_sms,
                                 cudaStream_t s) {
    return launch_transpose<uint32_t>(in, out, batch, R, Cc, num_sms, s);
}

}  // namespace cbd
