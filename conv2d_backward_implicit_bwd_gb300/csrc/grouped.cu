// grouped.cu -- bf16 NHWC/KYXC dgrad for narrow groups (C/G = K/G = 8 or 16,
// G a multiple of 8), e.g. the grouped 3x3 layers of ResNeXt-style networks
// (a workload named on page "[igemm_dynamic] v4r1 bwd dynamic kernel").
//
// With 8 channels per group the arithmetic intensity is ~14 FLOP per byte, so
// the kernel is bound by HBM traffic (dy read, dx written).  Per group and
// filter tap the contraction is a dense 8x8 (16x16) block:
//   dx[p, c] += sum over k < Kg of dy[p', k] * w[gi*Kg + k, y, x, c]
// which the warp-level tensor-core instruction mma.sync m16n8k8 (m16n8k16)
// executes exactly, with no padding: 16 dx pixels x 8 channels x 8 k per
// instruction.  That takes the multiply-adds off the CUDA-core issue slots,
// which bounded a direct FMA kernel; the design is then about moving bytes:
//   * A CTA owns one block of 8 groups (128 or 256 contiguous bytes per
//     pixel) and walks items (n, hi, 64-pixel chunk of the row).  Per item it
//     stages the dy rows of the row class's taps (cp.async, 16 bytes per
//     thread, zero-filled outside dy) in shared memory -- the next item's rows
//     load while the current item computes (two buffers).
//   * A warp computes one unit: 16 outputs of one column residue class (the
//     v4r1 split of pages "Backward data" and "[igemm_dynamic] v4r1 bwd dynamic
//     kernel", per pixel) for all 8 groups.  Per tap (j, i) the dy pixels of
//     16 consecutive outputs are consecutive staged pixels, so ldmatrix reads
//     the A fragments directly; B fragments (w) are built once per CTA for all
//     taps.
//   * Pixel lines in shared memory are XOR-swizzled in 16-byte segments so
//     that 8 consecutive pixels' segment of one group hit 8 bank groups.
//   * Accumulators (fp32) leave as bf16 (RNE) straight from the fragments: for
//     8-channel groups the 4 lanes of a fragment row swap words so that each
//     lane holds whole groups and writes 16-byte segments (a pixel's 128-byte
//     line in two store instructions); pixels no tap reaches are written as +0
//     by the same pass (no separate fill).
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>

#include "internal.h"
#include "tc_common.cuh"

namespace cbd {

template <int CG>
struct GCfg {
    // 2 warps per CTA for 8-channel groups: with the units of an item in
    // (residue, m-tile) order, each warp then takes one m-tile of every residue
    // class, and classes with many and few taps share out evenly
    static constexpr int THREADS = CG == 8 ? 64 : 128;
    static constexpr int WARPS = THREADS / 32;
    static constexpr int LINE = 8 * CG * 2;     // bytes per pixel of one 8-group block
    static constexpr int SEGS = LINE / 16;      // 16-byte segments per pixel line
    static constexpr int NR = CG == 8 ? 1 : 4;  // B-fragment registers per (tap, lane)
    static constexpr int NT = CG / 8;           // n-tiles of 8 output channels
    static constexpr int MT = 4;                // m-tiles of 16 pixels per residue and chunk (at most)
};

// shared-memory address of segment s of staged pixel q (segments XOR-swizzled
// by q mod 8 so that 8 consecutive pixels' segment s fall in 8 bank groups)
template <int CG>
__device__ __forceinline__ uint32_t seg_addr(uint32_t base, int q, int s) {
    return base + (uint32_t)q * GCfg<CG>::LINE + ((uint32_t)(s ^ (q & 7)) << 4);
}


struct GItem {
    int n, hi, wc;       // image, dx row, chunk of the row
    int w0, npx;         // first dx column and pixel count of the chunk
    int tyn, ty, ht;     // the row's class: taps, first tap, class row
    int wo_lo;           // first staged dy column
};

// row class and staged window of item (n, hi, wc)
__device__ __forceinline__ void finish_item(const GroupedParams &p, GItem &m) {
    const Geom &g = p.g;
    m.w0 = m.wc * p.wch;
    m.npx = min(p.wch, g.Wi - m.w0);
    const int rc = p.row_class[m.hi % g.sh];
    m.tyn = rc >> 16;
    m.ty = rc & 0xFFFF;
    m.ht = (m.hi + g.ph - m.ty * g.dh) / g.sh;  // exact when tyn > 0
    m.wo_lo = m.wc * (p.wch / g.sw) + p.wo_c;
}

// the item `step` items after m (step = CTAs per group block, pre-split into
// chunk / row / image digits on the host): mixed-radix add with carries
__device__ __forceinline__ GItem next_item(const GroupedParams &p, const GItem &m) {
    const Geom &g = p.g;
    GItem r;
    r.wc = m.wc + p.step_wc;
    int carry = r.wc >= p.nwch;
    r.wc -= carry ? p.nwch : 0;
    r.hi = m.hi + p.step_hi + carry;
    carry = r.hi >= g.Hi;
    r.hi -= carry ? g.Hi : 0;
    r.n = m.n + p.step_n + carry;
    finish_item(p, r);
    return r;
}

// Within each quad of lanes (4*k .. 4*k+3, t = lane % 4): o[j] = w[t] of lane
// 4*k + j, a 4 x 4 transpose of 32-bit words in two butterfly stages (lanes
// t ^ 1 swap two words, then lanes t ^ 2 swap two), all register indices static.
__device__ __forceinline__ void quad_transpose(const uint32_t (&w)[4], uint32_t (&o)[4], int lane) {
    const bool odd = lane & 1, hi2 = lane & 2;
    // stage 1: pair base p = t & ~1 ends with x = {w_p[t&1], w_p+1[t&1], w_p[2+(t&1)], w_p+1[2+(t&1)]}
    const uint32_t r0 = __shfl_xor_sync(0xffffffffu, odd ? w[0] : w[1], 1);
    const uint32_t r1 = __shfl_xor_sync(0xffffffffu, odd ? w[2] : w[3], 1);
    const uint32_t x0 = odd ? r0 : w[0], x1 = odd ? w[1] : r0;
    const uint32_t x2 = odd ? r1 : w[2], x3 = odd ? w[3] : r1;
    // stage 2: lanes t and t ^ 2 swap their other half
    const uint32_t q0 = __shfl_xor_sync(0xffffffffu, hi2 ? x0 : x2, 2);
    const uint32_t q1 = __shfl_xor_sync(0xffffffffu, hi2 ? x1 : x3, 2);
    o[0] = hi2 ? q0 : x0;
    o[1] = hi2 ? q1 : x1;
    o[2] = hi2 ? x2 : q0;
    o[3] = hi2 ? x3 : q1;
}

template <int CG>
__global__ void __launch_bounds__(GCfg<CG>::THREADS, CG == 8 ? 10 : 3) grouped_dgrad_kernel(const __grid_constant__ GroupedParams p) {
    using C = GCfg<CG>;
    constexpr int LOG_SEGS = CG == 8 ? 3 : 4;
    constexpr int NTHREADS = C::THREADS;
    constexpr int PSTEP = NTHREADS / GCfg<CG>::SEGS;  // staged pixels per pass of the CTA
    extern __shared__ __align__(128) uint8_t gsm[];
    const Geom &g = p.g;
    const uint32_t *wfrag = reinterpret_cast<const uint32_t *>(gsm);  // B fragments (layout below)
    const uint32_t buf0 = smem_u32(gsm + p.wfrag_bytes);             // two buffers of [tyn][span] pixel lines
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int gb = blockIdx.x % p.gblocks;
    const int cta = blockIdx.x / p.gblocks;
    const int64_t cofs = (int64_t)gb * 8 * CG;  // first channel of the block (dy and dx)

    // B fragments of the block's 8 groups for every tap.  The groups' w rows
    // (8*CG rows of Y*X*CG contiguous bf16) are first copied to shared memory
    // (16-byte loads), then lane (gid, tig) takes, for group gl,
    // w[gi*Kg + k][y][x][n] with k = 2 tig (+1) (+8 for the second half of a
    // 16-deep step) and n = gid (+8 for the second n-tile)
    {
        const int ntap = g.Y * g.X;
        const int rowh = ntap * CG;          // bf16 per k row
        const int nraw = 8 * CG * rowh / 8;  // 16-byte pieces of the block's rows
        const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.w) + cofs * rowh);
        uint4 *raw = reinterpret_cast<uint4 *>(gsm + p.wfrag_bytes);
        for (int e = threadIdx.x; e < nraw; e += NTHREADS) raw[e] = src[e];
        __syncthreads();
        const uint16_t *rw = reinterpret_cast<const uint16_t *>(raw);
        uint32_t *wf = reinterpret_cast<uint32_t *>(gsm);
        for (int e = threadIdx.x; e < ntap * C::NR * 32 * 8; e += NTHREADS) {
            // CG = 8: [tap][group half][lane][4 groups] (16 contiguous bytes per lane
            // and half: conflict-free 16-byte loads); CG = 16: [tap][NR][lane][8 groups]
            const int gl = CG == 8 ? ((e >> 7) & 1) * 4 + (e & 3) : e & 7;
            const int l = CG == 8 ? (e >> 2) & 31 : (e >> 3) & 31;
            const int r = (e >> 8) % C::NR, tap = e / (256 * C::NR);
            const int nt = r >> 1, kh = r & 1;
            const int n = nt * 8 + (l >> 2), k = 2 * (l & 3) + 8 * kh;
            const int base = (gl * CG + k) * rowh + tap * CG + n;
            wf[e] = (uint32_t)rw[base] | ((uint32_t)rw[base + rowh] << 16);
        }
        __syncthreads();
    }

    const int64_t kbytes = (int64_t)g.K * 2;
    const int mi = lane >> 3;                       // ldmatrix: lane addresses row lane % 8 of matrix mi
    const int trow = (mi & 1) * 8 + (lane & 7);     // this lane's A row within the 16-row tile

    auto stage = [&](const GItem &m, int b) {
        const uint32_t bb = buf0 + (uint32_t)b * p.buf_bytes;
        for (int jj = 0; jj < m.tyn; ++jj) {
            const int ho = m.ht - jj * g.DH;
            const bool hok = ho >= 0 && ho < g.Ho;
            const uint8_t *rowp = static_cast<const uint8_t *>(p.dy) +
                                  ((int64_t)m.n * g.Ho + (hok ? ho : 0)) * g.Wo * kbytes + cofs * 2;
            // thread t copies segment t % SEGS of pixels t / SEGS, + PSTEP, ...: the
            // segment's swizzled slot is the same for all of them (PSTEP % 8 == 0)
            const int s = threadIdx.x & (C::SEGS - 1);
            int q = threadIdx.x >> LOG_SEGS;
            uint32_t dst = seg_addr<CG>(bb + (uint32_t)(jj * p.span * C::LINE), q, s);
            int wo = m.wo_lo + q;
            const uint8_t *src = rowp + (int64_t)wo * kbytes + s * 16;
            for (; q < p.span; q += PSTEP, wo += PSTEP, dst += PSTEP * C::LINE, src += PSTEP * kbytes) {
                const bool ok = hok && wo >= 0 && wo < g.Wo;
                cp_async_16(dst, ok ? src : static_cast<const uint8_t *>(p.dy), ok ? 16u : 0u);
            }
        }
    };

    // first item of this CTA: (n, hi, wc) = cta in mixed radix (N, Hi, nwch)
    GItem m;
    m.wc = cta % p.nwch;
    m.hi = (cta / p.nwch) % g.Hi;
    m.n = cta / (p.nwch * g.Hi);
    finish_item(p, m);
    int b = 0;
    if (m.n < g.N) stage(m, 0);
    cp_async_commit();
    const int nunits = g.sw * p.per_r;
    while (m.n < g.N) {
        const GItem mn = next_item(p, m);
        if (mn.n < g.N) stage(mn, b ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();

        // units (column residue r, 16-pixel m-tile mt) of this item: warp w
        // takes units w, w + WARPS, ...; a unit covers all 8 groups of the block
        const uint32_t bb = buf0 + (uint32_t)b * p.buf_bytes;
        const int64_t cbytes = (int64_t)g.C * 2;
        uint8_t *dxrow = static_cast<uint8_t *>(p.dx) + ((((int64_t)m.n * g.Hi + m.hi) * g.Wi + m.w0) * g.C + cofs) * 2;
        int r = warp / p.per_r, mt = warp - r * p.per_r;
        for (int u = warp; u < nunits; u += C::WARPS) {
            if (r + g.sw * 16 * mt < m.npx) {
                const int cc = p.col_class[r];  // w0 is a multiple of sw
                const int txn = cc >> 16, tx = cc & 0xFFFF;
                float acc[8][4 * C::NT];
#pragma unroll
                for (int gl = 0; gl < 8; ++gl)
#pragma unroll
                    for (int v = 0; v < 4 * C::NT; ++v) acc[gl][v] = 0.f;
                if (m.tyn > 0 && txn > 0) {
                    const int qrow = p.col_q[r] + mt * 16 + trow;  // staged pixel of this lane's row, tap i = 0
                    for (int jj = 0; jj < m.tyn; ++jj) {
                        const int ho = m.ht - jj * g.DH;
                        if (ho < 0 || ho >= g.Ho) continue;  // staged as zeros: nothing to add
                        const int y = m.ty + g.YT * jj;
                        const uint32_t rowb = bb + (uint32_t)(jj * p.span * C::LINE);
                        for (int ii = 0; ii < txn; ++ii) {
                            const int tap = y * g.X + tx + g.XT * ii;
                            const int q = min(qrow - ii * g.DW, p.span - 1);
                            const uint32_t arow = rowb + (uint32_t)q * C::LINE;
                            const int qs = q & 7;
                            if (CG == 8) {
                                // fragments of the 8 groups: two 16-byte loads
                                const uint4 *wl = reinterpret_cast<const uint4 *>(wfrag + tap * 256 + lane * 4);
                                const uint4 f0 = wl[0], f1 = wl[32];
                                const uint32_t bfr[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
                                for (int gp = 0; gp < 4; ++gp) {
                                    // matrices: rows 0-7 | 8-15 of group 2gp, then of group 2gp + 1
                                    const int seg = 2 * gp + (mi >> 1);
                                    uint32_t a0, a1, a2, a3;
                                    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                                                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                                                 : "r"(arow + ((uint32_t)(seg ^ qs) << 4)));
                                    asm volatile(
                                        "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5}, "
                                        "{%6}, {%0, %1, %2, %3};"
                                        : "+f"(acc[2 * gp][0]), "+f"(acc[2 * gp][1]), "+f"(acc[2 * gp][2]),
                                          "+f"(acc[2 * gp][3])
                                        : "r"(a0), "r"(a1), "r"(bfr[2 * gp]));
                                    asm volatile(
                                        "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5}, "
                                        "{%6}, {%0, %1, %2, %3};"
                                        : "+f"(acc[2 * gp + 1][0]), "+f"(acc[2 * gp + 1][1]), "+f"(acc[2 * gp + 1][2]),
                                          "+f"(acc[2 * gp + 1][3])
                                        : "r"(a2), "r"(a3), "r"(bfr[2 * gp + 1]));
                                }
                            } else {
#pragma unroll
                                for (int gl = 0; gl < 8; ++gl) {
                                    // matrices (rows 0-7 | 8-15) x (k 0-7 | 8-15) of group gl
                                    const int seg = 2 * gl + (mi >> 1);
                                    uint32_t a0, a1, a2, a3;
                                    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                                                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                                                 : "r"(arow + ((uint32_t)(seg ^ qs) << 4)));
#pragma unroll
                                    for (int nt = 0; nt < C::NT; ++nt) {
                                        const uint32_t b0 = wfrag[((tap * C::NR + 2 * nt) * 32 + lane) * 8 + gl];
                                        const uint32_t b1 = wfrag[((tap * C::NR + 2 * nt + 1) * 32 + lane) * 8 + gl];
                                        asm volatile(
                                            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
                                            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                                            : "+f"(acc[gl][4 * nt]), "+f"(acc[gl][4 * nt + 1]),
                                              "+f"(acc[gl][4 * nt + 2]), "+f"(acc[gl][4 * nt + 3])
                                            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
                                    }
                                }
                            }
                        }
                    }
                }
                // accumulators -> bf16 -> dx: lane (gid, tig) holds rows gid, gid + 8
                // and channels nt*8 + 2 tig (+1) of every group (16-channel groups:
                // 4-byte stores, the 4 lanes of a row covering 16 contiguous bytes)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int q = r + g.sw * (mt * 16 + gid + 8 * h);
                    if (CG == 8) {
                        // the 4 lanes of a row swap words so that lane tig holds all
                        // 8 channels of groups tig and 4 + tig: two 16-byte stores
                        // per lane, a row's 128-byte line in two instructions
                        uint32_t wlo[4], whi[4], olo[4], ohi[4];
#pragma unroll
                        for (int gl = 0; gl < 4; ++gl) {
                            __nv_bfloat162 a = __floats2bfloat162_rn(acc[gl][2 * h], acc[gl][2 * h + 1]);
                            __nv_bfloat162 b = __floats2bfloat162_rn(acc[gl + 4][2 * h], acc[gl + 4][2 * h + 1]);
                            wlo[gl] = *reinterpret_cast<uint32_t *>(&a);
                            whi[gl] = *reinterpret_cast<uint32_t *>(&b);
                        }
                        quad_transpose(wlo, olo, lane);
                        quad_transpose(whi, ohi, lane);
                        if (q < m.npx) {
                            uint4 *o = reinterpret_cast<uint4 *>(dxrow + q * cbytes);
                            o[tig] = make_uint4(olo[0], olo[1], olo[2], olo[3]);
                            o[4 + tig] = make_uint4(ohi[0], ohi[1], ohi[2], ohi[3]);
                        }
                        continue;
                    }
                    if (q >= m.npx) continue;
                    uint32_t *o = reinterpret_cast<uint32_t *>(dxrow + q * cbytes) + tig;
#pragma unroll
                    for (int gl = 0; gl < 8; ++gl)
#pragma unroll
                        for (int nt = 0; nt < C::NT; ++nt) {
                            __nv_bfloat162 v =
                                __floats2bfloat162_rn(acc[gl][4 * nt + 2 * h], acc[gl][4 * nt + 2 * h + 1]);
                            o[(gl * C::NT + nt) * 4] = *reinterpret_cast<uint32_t *>(&v);
                        }
                }
            }
            mt += C::WARPS;
            while (mt >= p.per_r) {
                mt -= p.per_r;
                ++r;
            }
        }
        __syncthreads();  // every warp is done with buffer b before it is restaged
        m = mn;
        b ^= 1;
    }
    cp_async_wait<0>();
}

// Chunk width, staged span and shared memory of a geometry (the planner
// checks that it fits; the launch uses the same numbers).
GroupedLayout grouped_layout(const Geom &g) {
    GroupedLayout L;
    const int line = 8 * g.Cg * 2;
    const int nr = g.Cg == 8 ? 1 : 4;
    const int tymax = (g.Y + g.YT - 1) / g.YT;
    L.wfrag_bytes = g.Y * g.X * 8 * nr * 32 * 4;
    const int raw_w = 8 * g.Cg * g.Y * g.X * g.Cg * 2;  // the block's w rows, staged once at the start
    for (int wch = 64; wch >= 16; wch /= 2) {
        L.wch = std::max(g.sw, wch - wch % g.sw);
        L.span = (L.wch - 1 + (g.X - 1) * g.dw) / g.sw + 2;
        L.buf_bytes = tymax * L.span * line;
        L.smem = L.wfrag_bytes + std::max(2 * L.buf_bytes, raw_w);
        if (L.smem <= 200 * 1024 && L.wch / g.sw <= 64) break;
    }
    return L;
}

template <int CG>
static cudaError_t launch_grouped_cg(const GroupedParams &p, const GroupedLayout &L, int num_sms, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(grouped_dgrad_kernel<CG>, cudaFuncAttributeMaxDynamicSharedMemorySize, L.smem);
    if (e != cudaSuccess) return e;
    // CTAs that fit on an SM at once (registers and shared memory): the item
    // loop is persistent, so the grid must be exactly one wave
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, grouped_dgrad_kernel<CG>, GCfg<CG>::THREADS, L.smem) !=
            cudaSuccess ||
        per_sm < 1) {
        cudaGetLastError();
        per_sm = 1;
    }
    const int sms = num_sms > 0 ? num_sms : 148;
    int per_gb = std::max(1, (sms * per_sm + p.gblocks - 1) / p.gblocks);
    const int64_t items = (int64_t)p.g.N * p.g.Hi * p.nwch;
    per_gb = (int)std::min<int64_t>(per_gb, items);
    GroupedParams q = p;
    q.step_wc = per_gb % q.nwch;
    q.step_hi = (per_gb / q.nwch) % q.g.Hi;
    q.step_n = per_gb / (q.nwch * q.g.Hi);
    grouped_dgrad_kernel<CG><<<per_gb * p.gblocks, GCfg<CG>::THREADS, L.smem, s>>>(q);
    return cudaGetLastError();
}

cudaError_t launch_grouped(GroupedParams &p, int num_sms, cudaStream_t s) {
    const GroupedLayout L = grouped_layout(p.g);
    const Geom &g = p.g;
    p.wch = L.wch;
    p.span = L.span;
    p.wfrag_bytes = L.wfrag_bytes;
    p.buf_bytes = L.buf_bytes;
    p.nwch = (g.Wi + L.wch - 1) / L.wch;
    p.per_r = (L.wch / g.sw + 15) / 16;
    // first staged dy column of a chunk at w0 (a multiple of sw):
    // floor((w0 + pw - (X-1) dw) / sw) = w0 / sw + floor((pw - (X-1) dw) / sw)
    const int a = g.pw - (g.X - 1) * g.dw;
    p.wo_c = a >= 0 ? a / g.sw : -((-a + g.sw - 1) / g.sw);
    // residue r of a class with first tap tx: its output t = 0 reads dy column
    // (w0 + r + pw - tx dw) / sw for tap i = 0, staged at that minus the first column
    for (int r = 0; r < g.sw && r < 64; ++r) {
        const int tx = p.col_class[r] & 0xFFFF;
        const int num = r + g.pw - tx * g.dw;  // a multiple of sw where the class has taps
        p.col_q[r] = ((p.col_class[r] >> 16) > 0 ? num / g.sw : 0) - p.wo_c;
    }
    return p.g.Cg == 8 ? launch_grouped_cg<8>(p, L, num_sms, s) : launch_grouped_cg<16>(p, L, num_sms, s);
}

}  // namespace cbd
