// tc_band_sm103.cu -- bf16 NHWC/KYXC dgrad for narrow groups (C/G = K/G in
// {8, 16, 32}, strides 1 or 2) on the tcgen05 tensor cores, with each band of
// dy staged in shared memory once and read by every filter tap from there.
//
// The residue classes of the v4r1 backward-data split (pages "Backward data"
// and "[igemm_dynamic] v4r1 bwd dynamic kernel") are taken here per output
// pixel: with strides sh, sw <= 2, dx pixel (hi, wi) = (sh*i + a, sw*j + b)
// belongs to class (a, b), and a filter tap (y, x) reaches it iff
// a + ph - y*dh and b + pw - x*dw are multiples of sh and sw; it then reads
//   dy[n, i + oy, j + ox, k],  oy = (a + ph - y*dh) / sh,  ox = (b + pw - x*dw) / sw
// (zero outside dy).  So every tap of every class reads the same dy window,
// shifted by a few rows (oy) and columns (ox).  A work unit is one image n,
// one band of four output rows i, one segment of segw = 32 - (max ox - min ox)
// output columns j and one 64-channel block.  Its A operand is a band of dy:
// rows i0 + min oy .. i0 + 3 + max oy, 32 pixels from column j0 + min ox, 64
// channels (128 bytes) per pixel, loaded by one TMA box with 128-byte swizzle,
// pixels outside dy zero-filled.  The 128 GEMM rows m = 32 * (i - i0) +
// (j - j0) of a class then read, for a tap, 128 consecutive staged pixels
// starting at staged row oy - min oy, pixel ox - min ox: the tap's A is the
// staged band at a (4 KB * row + 128 B * pixel) offset.  The tensor core's
// 128-byte swizzle follows the absolute shared-memory address bits (the
// same property that lets a K-major descriptor advance 32 bytes per k
// slice), so a window may start at any pixel: measured on this kernel's
// parity tests, which fail at every shifted window when the descriptor's
// base-offset field is set to the shift instead of 0.  Rows j - j0 >= segw
// read past their staged row (into the next row, or past the stage) and are
// never stored.
//
// The groups of a 64-channel block are folded into one GEMM with a
// block-diagonal B, but the MMAs skip the all-zero blocks: the 16-deep k
// slice s of the block (channels 16s .. 16s+15) meets only the output
// channels of its own groups (NB = max(16, Cg) of them).  And one MMA serves
// every class whose tap reads the same window: per window and k slice, one
// M = 128, N = classes x NB, K = 16 MMA whose B stacks, class by class, the
// NB x 16 block of that class's tap (zero for a class with no tap on the
// window).  A tcgen05.mma of M = 128 and N <= 64 costs ~50 SM clocks however
// small N is, so the MMA count is what matters: a 3x3 stride-2 layer has 9
// taps but 4 windows, 16 MMAs per unit instead of 36.  The first window's
// MMAs overwrite every accumulator column (zero B blocks included), the rest
// accumulate; classes without taps thus come out as zero.  B of every window
// is built from w by the CTA's threads at start (8 x 8 transposes of w's
// (k, c) blocks) and stays resident: one K-major 128-byte-swizzled tile per
// window, row n = class * NB + channel offset, 128 bytes = the block's 64 k.
//
// Per unit the accumulators of all classes (classes x 64 fp32 columns,
// column = (c / NB) * classes * NB + class * NB + c % NB for channel c) sit
// in one TMEM buffer; two buffers let the epilogue of one unit overlap the
// MMAs of the next.  Roles (320 threads):
//   warps 0-7   epilogue: warp w drains TMEM lanes 32*(w % 4) .. (output row
//               i0 + w % 4) of the classes c with c % 2 == w / 4, rounding to
//               bf16 into swizzled shared memory, from where one TMA tensor
//               store per class writes the row's segw pixels (the class's dx
//               map clips rows and columns past its last);
//   warp 8      producer: one lane issues each unit's band load;
//   warp 9      TMEM allocation and the single-thread tcgen05.mma issue.
// Every dx pixel belongs to exactly one (unit, class, row, column), so the
// kernel writes all of dx and needs no separate fill.  Each CTA keeps one
// 64-channel block (its B) for the whole launch and walks that block's units
// with a stride of the CTAs sharing it, so neighbouring bands are loaded at
// about the same time and their shared halo rows come from L2.  Every barrier
// wait is bounded; on a timeout the kernel records the status word, lets its
// loads land and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "device_util.cuh"
#include "internal.h"
#include "band.h"
#include "tc_common.cuh"

namespace cbd {

struct BandCfg {
    static constexpr int ROW_BYTES = 32 * 128;  // one staged dy row: 32 pixels x 64 channels
    static constexpr int STAGE_OUT_BYTES = 8 * 32 * 128;  // epilogue staging: 8 warps x 32 rows x 128 B
    static constexpr int BAR_BYTES = 256;
    static constexpr int EPI_WARPS = 8;
    static constexpr int PROD_WARP = 8;
    static constexpr int MMA_WARP = 9;
    static constexpr int THREADS = 32 * 10;
    // requested at least this much shared memory so that one CTA holds an SM
    // (its TMEM allocation then never waits for another CTA's)
    static constexpr int MIN_SMEM = 120 * 1024;
};

__host__ __device__ __forceinline__ int band_nb(int cg) { return cg < 16 ? 16 : cg; }

// [A stages | B tiles | staging | barriers]: a window's last rows read up to
// (32 - segw) * 128 <= 2 KB past its stage, which stays inside the next stage
// or the B tiles (one window's tile is at least 16 rows x 128 B).
size_t tc_band_smem_bytes(int cg, int ncls, int nwin, int stage_bytes, int stages) {
    const size_t btile = (size_t)ncls * band_nb(cg) * 128;  // one window's B: classes x NB rows of 128 B
    size_t s = 1024 + (size_t)stages * stage_bytes + (size_t)nwin * btile + BandCfg::STAGE_OUT_BYTES +
               BandCfg::BAR_BYTES;
    return s < (size_t)BandCfg::MIN_SMEM ? (size_t)BandCfg::MIN_SMEM : s;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, M = 128, N = nb.
__device__ __forceinline__ uint32_t idesc_bf16_kk(int nb) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(nb >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c0, int c1,
                                            int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// 16 TMEM columns of this warp's 32 lanes into v[o .. o+16) (no wait)
template <int O>
__device__ __forceinline__ void tmem_ld16_issue(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(v[O + 0]), "=r"(v[O + 1]), "=r"(v[O + 2]), "=r"(v[O + 3]), "=r"(v[O + 4]), "=r"(v[O + 5]),
          "=r"(v[O + 6]), "=r"(v[O + 7]), "=r"(v[O + 8]), "=r"(v[O + 9]), "=r"(v[O + 10]), "=r"(v[O + 11]),
          "=r"(v[O + 12]), "=r"(v[O + 13]), "=r"(v[O + 14]), "=r"(v[O + 15])
        : "r"(taddr)
        : "memory");
}

// TMA tensor store of one staged box (4-D map) from shared memory, in this
// thread's bulk async-group
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, uint32_t src, int c0, int c1, int c2, int c3) {
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// the bulk stores of this thread have finished reading shared memory
__device__ __forceinline__ void tma_store_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// the bulk stores of this thread are complete (written to global memory)
__device__ __forceinline__ void tma_store_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Drain one class of one warp's 32 accumulator rows (TMEM lane = GEMM row =
// output column j0 + lane of output row i0 + warp % 4): its 64 channels sit in
// 64 / NB blocks of NB columns, `stride` columns apart.  Rounded to bf16
// (RNE) and staged by rows (pixel = lane) with 16-byte chunks XOR-swizzled by
// row: the 128-byte swizzle of the class's dx store map, whose box (64
// channels x segw pixels of this output row) lane 0 then stores with one TMA
// tensor store when `store` is set.  The map clips rows and columns past the
// class's last; lanes >= segw lie outside the box.  Lane 0 first waits until
// its previous store has read the staging buffer.
__device__ __forceinline__ void band_epilogue(uint32_t taddr, int nb, uint32_t stride, uint8_t *stage, int lane,
                                              bool store, const CUtensorMap *map, int c0, int j0, int i, int n) {
    const uint32_t sbase = smem_u32(stage);
    uint32_t va[32], vb[32];
    // channel 16q .. 16q+15 at column (16q / nb) * stride + 16q % nb
    tmem_ld16_issue<0>(taddr + (uint32_t)(0 / nb) * stride + (0 % nb), va);
    tmem_ld16_issue<16>(taddr + (uint32_t)(16 / nb) * stride + (16 % nb), va);
    tmem_ld16_issue<0>(taddr + (uint32_t)(32 / nb) * stride + (32 % nb), vb);
    tmem_ld16_issue<16>(taddr + (uint32_t)(48 / nb) * stride + (48 % nb), vb);
    if (lane == 0) tma_store_wait_read();
    __syncwarp();
    tmem_wait_ld(va);
    tmem_wait_ld(vb);
    stage_half(va, sbase, lane, 0);
    stage_half(vb, sbase, lane, 1);
    fence_proxy_async_smem();  // the staged rows, visible to the store's async proxy
    __syncwarp();
    if (lane == 0 && store) tma_store_4d(map, sbase, c0, j0, i, n);
}

struct BandUnit {
    int n, i0, j0;
};
__device__ __forceinline__ BandUnit band_unit(const BandParams &p, int u) {
    BandUnit r;
    const int seg = u % p.segs;
    const int t = u / p.segs;
    const int band = t % p.bands;
    r.n = t / p.bands;
    r.i0 = band * 4;
    r.j0 = seg * p.segw;
    return r;
}

__global__ void __launch_bounds__(BandCfg::THREADS, 1) tc_band_dgrad_kernel(const __grid_constant__ BandParams p) {
    using Cfg = BandCfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = p.stages;
    const int nb = band_nb(p.cg);
    const uint32_t ncol = (uint32_t)(p.ncls * nb);            // MMA N: every class's NB channels
    const uint32_t btile = ncol * 128;                         // one window's B tile
    const uint32_t stage_bytes = (uint32_t)p.rows * Cfg::ROW_BYTES;
    // [A stages | B tiles | epilogue staging | barriers], all 1024-aligned
    uint8_t *sA = smem;
    uint8_t *sB = sA + (size_t)S * stage_bytes;
    uint8_t *stage = sB + (size_t)p.nwin * btile;
    uint64_t *bars = reinterpret_cast<uint64_t *>(stage + Cfg::STAGE_OUT_BYTES);
    // bars: full[0..S) | empty[0..S) | tfull[2] | tempty[2]   (S <= 6)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * 6 + 4);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(tmem_slot + 1);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S);
    const uint32_t tfull0 = smem_u32(bars + 2 * S), tempty0 = smem_u32(bars + 2 * S + 2);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int cb = blockIdx.x % p.cblocks;  // this CTA's 64-channel block
    const int local = blockIdx.x / p.cblocks, nlocal = gridDim.x / p.cblocks;
    const uint32_t tcols = (uint32_t)p.ncls * 64;  // one accumulator buffer
    if (threadIdx.x == 0) CBD_PHASE(p, kPhEntry);

    // B tiles, one per window: row n = class * NB + c % NB of window w's tile
    // (128 bytes, 16-byte chunk q stored at chunk q ^ (n % 8)) holds the
    // block's 64 k: B_w[n][k] = w[cb*64 + k, tap(w, class), c mod Cg] where k
    // and channel c share a group, else 0 (the MMA of k slice s reads bytes
    // 32s .. 32s+31, where c = (16s / NB) * NB + n % NB).  Written as 8 x 8
    // blocks (k chunk kq, c chunk cq of one group) transposed in registers;
    // each thread's first block is read from w before anything else, so the
    // read's latency overlaps the barrier set-up, the TMEM allocation and the
    // zero fill.
    const int cg = p.cg, mch = cg / 8;             // 8-channel chunks per group
    const int64_t rowlen = (int64_t)p.ntaps * cg;  // bf16 per filter row k (KYXC)
    const uint16_t *wp = static_cast<const uint16_t *>(p.w);
    const int nblk = p.nwin * p.ncls * cg;         // per (window, class): 64/cg groups x mch*mch blocks
    struct Blk {
        const uint16_t *src;
        int wi, cls, kq, cq;
    };
    auto block_of = [&](int idx) {
        Blk b;
        const int wc = idx / cg, r = idx - wc * cg;
        b.wi = wc / p.ncls;
        b.cls = wc - b.wi * p.ncls;
        const int t = p.win_tap[b.wi][b.cls];
        const int grp = r / (mch * mch), rem = r - grp * mch * mch;
        b.kq = grp * mch + rem / mch;
        b.cq = grp * mch + rem % mch;
        b.src = t < 0 ? nullptr
                      : wp + ((int64_t)cb * 64 + 8 * b.kq) * rowlen + (int64_t)t * cg + (8 * b.cq - grp * cg);
        return b;
    };
    auto load_block = [&](const Blk &b, uint32_t (&in)[8][4]) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint4 v = *reinterpret_cast<const uint4 *>(b.src + kk * rowlen);
            in[kk][0] = v.x; in[kk][1] = v.y; in[kk][2] = v.z; in[kk][3] = v.w;
        }
    };
    auto write_block = [&](const Blk &b, const uint32_t (&in)[8][4]) {
        uint8_t *tile = sB + (size_t)b.wi * btile;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
            uint32_t o[4];
#pragma unroll
            for (int mm = 0; mm < 4; ++mm)
                o[mm] = __byte_perm(in[2 * mm][cc >> 1], in[2 * mm + 1][cc >> 1], (cc & 1) ? 0x7632 : 0x5410);
            const int n = b.cls * nb + (8 * b.cq + cc) % nb;
            *reinterpret_cast<uint4 *>(tile + n * 128 + ((b.kq ^ (n & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    };
    Blk first;
    first.src = nullptr;
    uint32_t in0[8][4];
    if ((int)threadIdx.x < nblk) {
        first = block_of(threadIdx.x);
        if (first.src) load_block(first, in0);
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull0 + 8 * b, 1);
            mbar_init(tempty0 + 8 * b, 32 * Cfg::EPI_WARPS);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == Cfg::MMA_WARP) {
        tmem_alloc(smem_u32(tmem_slot), (uint32_t)p.tmem_cols);
        tc_fence_before();
    }
    {
        uint4 *b4 = reinterpret_cast<uint4 *>(sB);
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        for (int i = threadIdx.x; i < (int)(p.nwin * btile / 16); i += Cfg::THREADS) b4[i] = z;
    }
    // Producer (one lane of warp PROD_WARP): the A loads of this CTA's units,
    // issued up to `limit` loads from where the previous call stopped.  The
    // first unit's loads go out before B is written, so that band is in
    // flight meanwhile (issuing all S stages there delayed the B build's reads
    // of w behind them: first MMA 4.5 instead of 3.6 us).
    int pu = local;
    uint32_t pit = 0;
    bool pok = true;
    auto produce = [&](uint32_t limit) {
        for (; pu < p.units && pit < limit; pu += nlocal, ++pit) {
            const uint32_t s = pit % (uint32_t)S, ph = (pit / (uint32_t)S) & 1;
            if (!mbar_wait_bounded(empty0 + 8 * s, ph ^ 1, p.wait_budget, abort_flag, p.status,
                                   kDevTimeoutProducer)) {
                pok = false;
                return;
            }
            const BandUnit un = band_unit(p, pu);
            const uint32_t dst = smem_u32(sA) + s * stage_bytes;
            mbar_arrive_expect_tx(full0 + 8 * s, stage_bytes);
            tma_load_4d(dst, &p.tmap_dy, full0 + 8 * s, cb * 64, un.j0 + p.ox_min, un.i0 + p.oy_min, un.n);
            if (pit == 0) CBD_PHASE(p, kPhFirstIssue);
        }
    };
    __syncthreads();  // barriers initialised, B zeroed
    if (warp == Cfg::PROD_WARP && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_dy)) : "memory");
        produce(1u);
    }
    if (first.src) write_block(first, in0);
    for (int idx = threadIdx.x + Cfg::THREADS; idx < nblk; idx += Cfg::THREADS) {
        const Blk b = block_of(idx);
        if (!b.src) continue;
        uint32_t in[8][4];
        load_block(b, in);
        write_block(b, in);
    }
    fence_proxy_async_smem();  // generic-proxy writes, read by the tensor cores
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (threadIdx.x == 0) CBD_PHASE(p, kPhSetup);

    if (warp == Cfg::PROD_WARP) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            if (pok) produce(0xffffffffu);
            if (pit > 0) CBD_PHASE(p, kPhLastIssue);
            if (!pok && pit > 0) {
                for (int q = 0; q < 100; ++q) __nanosleep(1000);
            }
        }
        __syncwarp();
    } else if (warp == Cfg::MMA_WARP) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_kk((int)ncol);
            const uint64_t adesc0 = smem_desc_sw128(smem_u32(sA), 16, 1024);
            const uint64_t bdesc0 = smem_desc_sw128(smem_u32(sB), 16, 1024);
            bool ok = true, issued = false;
            uint32_t it = 0;
            for (int u = local; u < p.units; u += nlocal, ++it) {
                const uint32_t b = it & 1, tph = (it >> 1) & 1;
                if (!mbar_wait_bounded(tempty0 + 8 * b, tph ^ 1, p.wait_budget, abort_flag, p.status,
                                       kDevTimeoutMma)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t s = it % (uint32_t)S, ph = (it / (uint32_t)S) & 1;
                if (!mbar_wait_bounded(full0 + 8 * s, ph, p.wait_budget, abort_flag, p.status, kDevTimeoutMma)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (it == 0) CBD_PHASE(p, kPhFirstFull);
                if (it == 1) CBD_PHASE(p, kPhMma1Start);
                // descriptors advance by address / 16 in their low 14 bits (all
                // shared-memory addresses < 256 KB, so no carry leaves the field)
                const uint64_t a_stage = adesc0 + ((s * stage_bytes) >> 4);
                const uint32_t d_buf = tmem_base + b * tcols;
                // (unrolled over the table's capacity: the window entries are
                // then fixed parameter offsets, read ahead of the MMAs; 8 % less
                // issue time per MMA on a stride-1 layer)
#pragma unroll
                for (int wi = 0; wi < kBandMaxTaps; ++wi) {
                    if (wi >= p.nwin) break;
                    const int win = p.win[wi];
                    const uint64_t ad = a_stage + ((((uint32_t)(win & 0xff)) * 128u +
                                                    ((uint32_t)(win >> 8)) * Cfg::ROW_BYTES) >> 4);
                    const uint64_t bd = bdesc0 + ((wi * btile) >> 4);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const int gi = (ks * 16) / nb, sl = ks - gi * (nb / 16);
                        tc_mma(d_buf + (uint32_t)gi * ncol, ad + 2 * ks, bd + 2 * ks, idesc,
                               (wi > 0 || sl > 0) ? 1u : 0u);
                    }
                }
                issued = true;
                tc_commit(empty0 + 8 * s);
                tc_commit(tfull0 + 8 * b);
                if (it == 0) CBD_PHASE(p, kPhMma0Done);
                CBD_PHASE(p, kPhMmaLast);
            }
            if (!ok && issued) {
                for (int q = 0; q < 100; ++q) __nanosleep(1000);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int qr = warp & 3, half = warp >> 2;
        uint32_t it = 0;
        for (int u = local; u < p.units; u += nlocal, ++it) {
            const uint32_t b = it & 1, tph = (it >> 1) & 1;
            bool ok = mbar_wait_bounded(tfull0 + 8 * b, tph, p.wait_budget, abort_flag, p.status, kDevTimeoutEpilogue);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            if (threadIdx.x == 0 && it == 0) CBD_PHASE(p, kPhEpi0Start);
            if (threadIdx.x == 0 && it == 1) CBD_PHASE(p, kPhEpi1Start);
            const BandUnit un = band_unit(p, u);
            const int i = un.i0 + qr;
            for (int c = half; c < p.ncls; c += 2) {
                const int a = c / p.sw, bb = c - a * p.sw;
                const bool store = i < p.hc[a] && un.j0 < p.wc[bb] && ((p.dx_maps >> c) & 1);
                const uint32_t tb = tmem_base + ((uint32_t)(qr * 32) << 16) + b * tcols + (uint32_t)(c * nb);
                band_epilogue(tb, nb, ncol, stage + warp * 4096, lane, store, &p.tmap_dx[c], cb * 64, un.j0, i, un.n);
            }
            tc_fence_before();
            mbar_arrive(tempty0 + 8 * b);
            if (threadIdx.x == 0 && it == 0) CBD_PHASE(p, kPhEpi0Done);
            if (threadIdx.x == 0 && it == 1) CBD_PHASE(p, kPhEpi1Done);
            if (lane == 0 && qr == 0) CBD_PHASE(p, kPhEpiLast);
        }
        if (lane == 0) tma_store_wait_all();
    }

    __syncthreads();
    if (threadIdx.x == 0) CBD_PHASE(p, kPhExit);
    if (warp == Cfg::MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem_base, (uint32_t)p.tmem_cols);
    }
}

cudaError_t launch_tc_band(const BandParams &p, int grid, cudaStream_t s) {
    if (grid <= 0 || p.units <= 0) return cudaSuccess;
    const size_t smem = tc_band_smem_bytes(p.cg, p.ncls, p.nwin, p.rows * BandCfg::ROW_BYTES, p.stages);
    cudaError_t e = cudaFuncSetAttribute(tc_band_dgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    tc_band_dgrad_kernel<<<grid, BandCfg::THREADS, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace cbd
