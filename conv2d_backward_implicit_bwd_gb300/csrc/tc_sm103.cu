// tc_sm103.cu -- bf16 NHWC/KYXC dgrad on the 5th-generation tensor cores
// (tcgen05 + TMEM), all sub-GEMMs of a plan in one persistent launch.
//
// Per residue class (ty, tx) and group gi the sub-GEMM is
//   D[m, c] = sum over taps (j, i) and k < Kg of A[m, (j, i, k)] * B[(j, i, k), c]
//   A[m, (j, i, k)] = dy[n, ht - j*DH, wt - i*DW, gi*Kg + k]     (zero outside dy)
//   B[(j, i, k), c] = w[gi*Kg + k, ty + YT*j, tx + XT*i, c]
//   dx[n, ht*sh + ty*dh - ph, wt*sw + tx*dw - pw, gi*Cg + c] = bf16_rne(D[m, c])
// with m enumerating the class's (n, ht, wt) positions.  This is the v4r1
// backward-data multi-kernel split (pages "Backward data" and "[igemm_dynamic]
// v4r1 bwd dynamic kernel"): stride > 1 needs no zero insertion, and the
// filter flip of the BOO IR (`1 - x` index, page "Non-unit stride input
// backward different input and dispatches between BOO and Fusilli") becomes
// the decreasing dy row ho = ht - j*DH.  Out-of-range dy rows read as zero
// (the "OOB dims in getGemmA" point of the rocMLIR review); the epilogue
// writes only rows of the class that exist in dx (the "OOB write" point).
//
// Tile: 128 (m) x BN (c) with BN in {128, 256}, K step 64 (one 128-byte
// swizzled row per operand row), S pipeline slots.  With C/G <= 128 a
// 256-wide tile may hold a class pair: two classes with the same rows and tap
// counts read the same dy rows for every tap (ho = ht - j*DH), so one A load
// and one N = 256 MMA per k slice serve both; columns 128-255 then belong to
// the second class (residues pty, ptx: its own filter taps and dx pixels).
// Roles (one CTA per SM):
//   warps 0-3      epilogue: tcgen05.ld of the fp32 accumulator (warp q reads
//                  TMEM lanes 32q..32q+31 = tile rows), RNE to bf16, 16-byte
//                  stores to the class's strided dx pixels;
//   warp 4         A producer (im2col mode, the default): one lane issues, per
//                  stage, a single TMA im2col load of the 128 A rows -- each
//                  class has its own rank-4 map over dy whose bounding box is
//                  the class's (ht, wt) range shifted to tap (taps-1), so the
//                  map walks the class rows in (n, ht, wt) order and the tap
//                  (j, i) is the im2col offset; rows outside dy (padding,
//                  borders, the flip's out-of-range taps, the M tail) read as
//                  zero; the BN/64 TMA boxes of B (w is c-contiguous, so B is
//                  MN-major: 64 k x 64 c per box) come from BN/64 more warps
//                  after the MMA warp, one box each;
//   warps 4..4+S-1 producers (cp.async mode, where a 64-channel block may cross
//                  a group boundary or a bounding box exceeds the im2col corner
//                  range): producer warp s loads every stage of slot s,
//                  gathering A rows with 16-byte cp.async (zero-fill outside dy
//                  or past Kg; 4 rows x 128 B per instruction), waits for its
//                  own copies, fences them to the async proxy and arrives;
//                  lane 0 issues the B boxes;
//   last warp      TMEM allocation and the single-thread tcgen05.mma issue
//                  (M=128, N=BN, K=16, bf16 x bf16 -> fp32), committing each
//                  stage back to its slot and each finished tile to the
//                  epilogue.  The accumulator is double-buffered in TMEM (2*BN
//                  columns) so the epilogue of tile t overlaps the MMAs of t+1.
// Every barrier wait is bounded (device_util.cuh); on a timeout the kernel
// records the status word, drains what it started and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "device_util.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace cbd {

template <int BN, bool IM2COL>
struct TcCfg {
    static constexpr int BM = 128;
    static constexpr int BK = 64;
    static constexpr int STAGES = BN == 256 ? 4 : 6;
    static constexpr int PRODUCER_WARPS = IM2COL ? 1 : STAGES;  // cp.async: one warp per slot; im2col: one
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int ROWTAB_BYTES = IM2COL ? 0 : STAGES * BM * 8;  // per producer warp: 128 x {pixel, ht|wt}
    static constexpr int BAR_BYTES = 256;
    static constexpr int STAGE_OUT_BYTES = 4 * 32 * 128;  // epilogue staging: 4 warps x 32 rows x 128 B
    static constexpr int SMEM = 1024 + STAGES * (A_BYTES + B_BYTES) + ROWTAB_BYTES + STAGE_OUT_BYTES + BAR_BYTES;
    static constexpr int MMA_WARP = 4 + PRODUCER_WARPS;
    // im2col mode: TMA issue is serialised per issuing thread, so warp 4 issues
    // only the A load and warps B_WARP.. one 64-column B box each, on other SM
    // sub-partitions
    static constexpr int B_WARP = MMA_WARP + 1;
    static constexpr int B_WARPS = IM2COL ? BN / 64 : 0;
    static constexpr int THREADS = 32 * (MMA_WARP + 1 + B_WARPS);
};

template <int BN, bool IM2COL>
__global__ void __launch_bounds__(TcCfg<BN, IM2COL>::THREADS, 1) tc_dgrad_kernel(const __grid_constant__ TcParams p) {
    using Cfg = TcCfg<BN, IM2COL>;
    constexpr int S = Cfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + S * Cfg::A_BYTES;
    uint8_t *stage = sB + S * Cfg::B_BYTES;  // epilogue staging (1024-aligned)
    int2 *rowtab = reinterpret_cast<int2 *>(stage + Cfg::STAGE_OUT_BYTES);
    uint64_t *bars = reinterpret_cast<uint64_t *>(stage + Cfg::STAGE_OUT_BYTES + Cfg::ROWTAB_BYTES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * S + 4);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(tmem_slot + 1);

    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S);
    const uint32_t tfull0 = smem_u32(bars + 2 * S), tempty0 = smem_u32(bars + 2 * S + 2);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const Geom &g = p.g;
    if (threadIdx.x == 0) CBD_PHASE(p, kPhEntry);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            // im2col: one arrive.expect_tx per stage; cp.async: the 32 lanes of the slot's warp
            mbar_init(full0 + 8 * s, IM2COL ? 1 : 32);
            mbar_init(empty0 + 8 * s, 1);
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
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_w)) : "memory");
        if (IM2COL)
            for (int ci = 0; ci < p.num_classes; ++ci)
                asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_a[ci])) : "memory");
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (threadIdx.x == 0) CBD_PHASE(p, kPhSetup);

    if (IM2COL && (warp == 4 || warp >= Cfg::B_WARP)) {
        // ------------------------------------------------------------ producers (TMA)
        // Lane 0 of warp 4 issues per stage the im2col load of the 128 A rows
        // (the class's map walks its (n, ht, wt) rows in order; the tap is the
        // im2col offset) and the stage's byte count; lane 0 of B warp q issues
        // B box q (64 k x 64 c).
        const bool do_a = warp == 4;
        const int cb_lo = do_a ? 0 : warp - Cfg::B_WARP, cb_hi = do_a ? 0 : cb_lo + 1;
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true, issued = false;
            SnakeTiles tiles(blockIdx.x, gridDim.x, p.total_tiles);
            for (int t; ok && tiles.next(t);) {
                const TileCoord tcd = decode_tile(p, t);
                const ClassDesc &c = p.cls[tcd.ci];
                const int num_kb = c.taps_y * c.taps_x * p.kb_per_tap;
                // first row of the tile -> base pixel of tap (taps_y-1, taps_x-1)
                const int HTWT = c.HT * c.WT;
                const int m0 = tcd.mb * 128;
                const int n0 = m0 / HTWT, rem = m0 - n0 * HTWT;
                const int bh = c.ht_lo + rem / c.WT - (c.taps_y - 1) * g.DH;
                const int bw = c.wt_lo + rem % c.WT - (c.taps_x - 1) * g.DW;
                const CUtensorMap *amap = &p.tmap_a[tcd.ci];
                for (int kb = 0; kb < num_kb; ++kb, ++it) {
                    const int tap = kb / p.kb_per_tap;
                    const int k0 = (kb - tap * p.kb_per_tap) * 64;
                    const int j = tap / c.taps_x, i = tap - j * c.taps_x;
                    const uint32_t s = it % S, ph = (it / S) & 1;
                    if (!mbar_wait_bounded(empty0 + 8 * s, ph ^ 1, p.wait_budget, abort_flag, p.status,
                                           kDevTimeoutProducer)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full_s = full0 + 8 * s;
                    // (a B box may land before this arrive: the transaction count
                    // dips below zero while the single arrival is still pending,
                    // so the phase cannot complete early)
                    if (do_a) {
                        mbar_arrive_expect_tx(full_s, (uint32_t)(Cfg::A_BYTES + Cfg::B_BYTES));
                        tma_load_im2col(smem_u32(sA + s * Cfg::A_BYTES), amap, full_s, tcd.gi * g.Kg + k0, bw, bh,
                                        n0, (uint16_t)((c.taps_x - 1 - i) * g.DW),
                                        (uint16_t)((c.taps_y - 1 - j) * g.DH));
                        if (it == 0) CBD_PHASE(p, kPhFirstIssue);
                    }
                    const uint32_t bdst = smem_u32(sB + s * Cfg::B_BYTES);
                    for (int cb = cb_lo; cb < cb_hi; ++cb) {
                        // a class pair's tile: boxes 2, 3 are the second class's filter tap (its 128 columns)
                        const bool second = BN == 256 && c.pty >= 0 && cb >= 2;
                        const int col = second ? (cb - 2) * 64 : tcd.nb * BN + cb * 64;
                        const int ty = second ? c.pty : c.ty, tx = second ? c.ptx : c.tx;
                        tma_load_5d(bdst + cb * 8192, &p.tmap_w, full_s, col, tx + g.XT * i, ty + g.YT * j, k0,
                                    tcd.gi);
                    }
                    issued = true;
                }
            }
            if (do_a && issued) CBD_PHASE(p, kPhLastIssue);
            if (!ok && issued) {
                for (int q = 0; q < 100; ++q) __nanosleep(1000);
            }
        }
        __syncwarp();
    } else if (!IM2COL && warp >= 4 && warp < Cfg::MMA_WARP) {
        // ------------------------------------------------------------ producers (cp.async)
        const int pw = warp - 4;                 // this warp owns pipeline slot pw
        const int chunk = lane & 7;              // 16-byte chunk of the 128-byte k row
        const int rsub = lane >> 3;              // rows rsub + 4*q, q < 32
        const __nv_bfloat16 *dy = static_cast<const __nv_bfloat16 *>(p.dy);
        int2 *tab = rowtab + pw * 128;
        const uint32_t full_s = full0 + 8 * pw, empty_s = empty0 + 8 * pw;
        const uint32_t a_slot = smem_u32(sA + pw * Cfg::A_BYTES);
        const uint32_t b_slot = smem_u32(sB + pw * Cfg::B_BYTES);
        uint32_t it = 0;   // global stage counter of this CTA (all slots)
        bool ok = true, issued_tma = false;
        SnakeTiles tiles(blockIdx.x, gridDim.x, p.total_tiles);
        for (int t; ok && tiles.next(t);) {
            const TileCoord tcd = decode_tile(p, t);
            const ClassDesc &c = p.cls[tcd.ci];
            const uint32_t num_kb = (uint32_t)(c.taps_y * c.taps_x * p.kb_per_tap);
            // first stage of this tile that lands in my slot
            uint32_t mine = it + (uint32_t)((pw - (int)(it % S) + S) % S);
            if (mine < it + num_kb) {
                // row table of the tile: pixel index of tap (0,0) and (ht, wt) as two
                // signed 16-bit halves (class rows may start at a negative ht); rows
                // past M get ht = -32768, which no tap brings back inside dy
                const int HTWT = c.HT * c.WT;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int r = lane + 32 * q;
                    const int m = tcd.mb * 128 + r;
                    int2 e = make_int2(0, (int)0x80000000u);
                    if (m < c.M) {
                        const int n = m / HTWT;
                        const int rem = m - n * HTWT;
                        const int ht = c.ht_lo + rem / c.WT, wt = c.wt_lo + rem % c.WT;
                        e = make_int2((n * g.Ho + ht) * g.Wo + wt, (int)(((uint32_t)ht << 16) | ((uint32_t)wt & 0xFFFFu)));
                    }
                    tab[r] = e;
                }
                __syncwarp();
            }
            int2 rinfo[32];
#pragma unroll
            for (int q = 0; q < 32; ++q) rinfo[q] = tab[rsub + 4 * q];
            __syncwarp();
            for (; mine < it + num_kb; mine += S) {
                const int kb = (int)(mine - it);
                const int tap = kb / p.kb_per_tap;
                const int k0 = (kb - tap * p.kb_per_tap) * 64;
                const int j = tap / c.taps_x, i = tap - j * c.taps_x;
                const uint32_t use = mine / S;
                if (!mbar_wait_bounded(empty_s, (use & 1) ^ 1, p.wait_budget, abort_flag, p.status,
                                       kDevTimeoutProducer)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_expect_tx(full_s, (uint32_t)Cfg::B_BYTES);
#pragma unroll
                    for (int cb = 0; cb < BN / 64; ++cb)
                        tma_load_5d(b_slot + cb * 8192, &p.tmap_w, full_s, tcd.nb * BN + cb * 64, c.tx + g.XT * i,
                                    c.ty + g.YT * j, k0, tcd.gi);
                    issued_tma = true;
                }
                const int dh = j * g.DH, dw = i * g.DW;
                const int dpix = dh * g.Wo + dw;
                const int kch = k0 + chunk * 8;
                const bool kval = kch < g.Kg;
                const int64_t kofs = (int64_t)tcd.gi * g.Kg + kch;
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    const int ht = rinfo[q].y >> 16, wt = (int)(short)(rinfo[q].y & 0xFFFF);
                    const int ho = ht - dh, wo = wt - dw;
                    const bool v = kval && ho >= 0 && ho < g.Ho && wo >= 0 && wo < g.Wo;
                    const __nv_bfloat16 *src = v ? dy + ((int64_t)(rinfo[q].x - dpix) * g.K + kofs) : dy;
                    // row r = rsub + 4q: (r & 7) == (rsub & 7) ^ (4 * (q & 1)) since rsub < 4
                    const uint32_t sw = (uint32_t)((chunk ^ ((rsub + 4 * q) & 7)) << 4);
                    cp_async_16(a_slot + (uint32_t)(rsub + 4 * q) * 128u + sw, src, v ? 16u : 0u);
                }
                cp_async_commit();
                cp_async_wait<0>();
                fence_proxy_async_smem();
                mbar_arrive(full_s);
            }
            it += num_kb;
        }
        cp_async_wait<0>();
        if (!ok && issued_tma) {
            // let TMA loads already in flight land before the block exits
            for (int q = 0; q < 100; ++q) __nanosleep(1000);
        }
    } else if (warp == Cfg::MMA_WARP) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16<BN>();
            uint32_t it = 0, tc = 0;
            bool ok = true, issued = false;
            SnakeTiles tiles(blockIdx.x, gridDim.x, p.total_tiles);
            for (int t; ok && tiles.next(t); ++tc) {
                const TileCoord tcd = decode_tile(p, t);
                const ClassDesc &c = p.cls[tcd.ci];
                const int num_kb = c.taps_y * c.taps_x * p.kb_per_tap;
                const uint32_t b = tc & 1, tph = (tc >> 1) & 1;
                if (!mbar_wait_bounded(tempty0 + 8 * b, tph ^ 1, p.wait_budget, abort_flag, p.status,
                                       kDevTimeoutMma)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (tc == 1) CBD_PHASE(p, kPhMma1Start);
                const uint32_t d_tmem = tmem_base + b * BN;
                for (int kb = 0; kb < num_kb; ++kb, ++it) {
                    const uint32_t s = it % S, ph = (it / S) & 1;
                    if (!mbar_wait_bounded(full0 + 8 * s, ph, p.wait_budget, abort_flag, p.status, kDevTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    if (it == 0) CBD_PHASE(p, kPhFirstFull);
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sA + s * Cfg::A_BYTES);
                    const uint32_t b_addr = smem_u32(sB + s * Cfg::B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = smem_desc_sw128(a_addr + kk * 32, 16, 1024);
                        const uint64_t bd = smem_desc_sw128(b_addr + kk * 2048, 8192, 1024);
                        tc_mma(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    issued = true;
                    tc_commit(empty0 + 8 * s);
                }
                if (!ok) break;
                tc_commit(tfull0 + 8 * b);
                if (tc == 0) CBD_PHASE(p, kPhMma0Done);
                CBD_PHASE(p, kPhMmaLast);
            }
            if (!ok && issued) {
                for (int q = 0; q < 100; ++q) __nanosleep(1000);
            }
        }
        __syncwarp();
    } else if (warp < 4) {
        // ------------------------------------------------------------ epilogue
        const int row = warp * 32 + lane;  // TMEM lane = tile row
        __nv_bfloat16 *dx = static_cast<__nv_bfloat16 *>(p.dx);
        uint32_t tc = 0;
        if (p.fill) fill_uncovered(p, threadIdx.x, 128);  // threads 0..127 are the epilogue warps
        if (threadIdx.x == 0) CBD_PHASE(p, kPhFillDone);
        SnakeTiles tiles(blockIdx.x, gridDim.x, p.total_tiles);
        for (int t; tiles.next(t); ++tc) {
            const TileCoord tcd = decode_tile(p, t);
            const ClassDesc &c = p.cls[tcd.ci];
            const uint32_t b = tc & 1, tph = (tc >> 1) & 1;
            bool ok = mbar_wait_bounded(tfull0 + 8 * b, tph, p.wait_budget, abort_flag, p.status, kDevTimeoutEpilogue);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            if (threadIdx.x == 0 && tc < 2) CBD_PHASE(p, tc == 0 ? kPhEpi0Start : kPhEpi1Start);
            const int m = tcd.mb * 128 + row;
            const bool rvalid = m < c.M;
            int64_t off = 0;
            if (rvalid) {
                const int HTWT = c.HT * c.WT;
                const int n = m / HTWT;
                const int rem = m - n * HTWT;
                const int hi = (c.ht_lo + rem / c.WT) * g.sh + c.ty * g.dh - g.ph;
                const int wi = (c.wt_lo + rem % c.WT) * g.sw + c.tx * g.dw - g.pw;
                off = (((int64_t)n * g.Hi + hi) * g.Wi + wi) * g.C + (int64_t)tcd.gi * g.Cg + (int64_t)tcd.nb * BN;
            }
            const uint32_t tbase = tmem_base + ((uint32_t)(warp * 32) << 16) + b * BN;
            if (BN == 256 && c.pty >= 0) {
                // class pair: columns 0-127 are this class's dx pixel, 128-255 the second class's
                int64_t off2 = 0;
                if (rvalid) {
                    const int HTWT = c.HT * c.WT;
                    const int n = m / HTWT;
                    const int rem = m - n * HTWT;
                    const int hi = (c.ht_lo + rem / c.WT) * g.sh + c.pty * g.dh - g.ph;
                    const int wi = (c.wt_lo + rem % c.WT) * g.sw + c.ptx * g.dw - g.pw;
                    off2 = (((int64_t)n * g.Hi + hi) * g.Wi + wi) * g.C + (int64_t)tcd.gi * g.Cg;
                }
                epilogue_chunks(tbase, 2, stage + warp * 4096, lane, rvalid, off, 0, g.Cg, dx);
                epilogue_chunks(tbase + 128, 2, stage + warp * 4096, lane, rvalid, off2, 0, g.Cg, dx);
            } else {
                epilogue_rows<BN>(tbase, stage + warp * 4096, lane, rvalid, off, tcd.nb * BN, g.Cg, dx);
            }
            tc_fence_before();
            mbar_arrive(tempty0 + 8 * b);
            if (threadIdx.x == 0) {
                if (tc < 2) CBD_PHASE(p, tc == 0 ? kPhEpi0Done : kPhEpi1Done);
                CBD_PHASE(p, kPhEpiLast);
            }
        }
    }

    __syncthreads();
    if (threadIdx.x == 0) CBD_PHASE(p, kPhExit);
    if (warp == Cfg::MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

size_t tc_smem_bytes(int bn, bool im2col) {
    if (bn == 256) return im2col ? TcCfg<256, true>::SMEM : TcCfg<256, false>::SMEM;
    return im2col ? TcCfg<128, true>::SMEM : TcCfg<128, false>::SMEM;
}

template <int BN, bool IM2COL>
static cudaError_t launch_tc_cfg(const TcParams &p, int grid, cudaStream_t s) {
    using Cfg = TcCfg<BN, IM2COL>;
    // the dynamic shared-memory opt-in is per device: set it for the current one
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(tc_dgrad_kernel<BN, IM2COL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Cfg::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    tc_dgrad_kernel<BN, IM2COL><<<grid, Cfg::THREADS, Cfg::SMEM, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_tc(const TcParams &p, int bn, int grid, cudaStream_t s) {
    if (grid <= 0 || p.total_tiles <= 0) return cudaSuccess;
    if (bn == 256) return p.im2col ? launch_tc_cfg<256, true>(p, grid, s) : launch_tc_cfg<256, false>(p, grid, s);
    return p.im2col ? launch_tc_cfg<128, true>(p, grid, s) : launch_tc_cfg<128, false>(p, grid, s);
}

}  // namespace cbd
