// tf32_sm103.cu -- fp32 NHWC dgrad on the 5th-generation tensor cores with a
// three-term TF32 split, all sub-GEMMs of a plan in one persistent launch.
//
// The sub-GEMMs are those of the bf16 kernels (one per filter-tap residue
// class and group: the v4r1 backward-data split of pages "Backward data" and
// "[igemm_dynamic] v4r1 bwd dynamic kernel"), on fp32 data:
//   D[m, c] = sum over taps (j, i) and k < Kg of A[m, (j, i, k)] * B[(j, i, k), c]
//   A = dy rows of the class (zero outside dy), B = the filter slice of the tap.
// A TF32 tensor-core product keeps 10 mantissa bits of each operand, too few
// for fp32 results (|err| <= 1e-5 * sum |dy*w| per element).  Each operand is
// therefore split as x = hi + lo with hi = x rounded to 10 mantissa bits and
// lo = x - hi (exact in fp32), and every k step issues three MMAs into one
// fp32 accumulator:
//   hi_A * hi_B + hi_A * lo_B + lo_A * hi_B
// leaving out lo_A * lo_B (about 2^-22 of |a*b|) and the 10-bit truncation of
// the lo terms (about 2^-21): products about as exact as fp32 FFMA, on the
// tensor pipe.  The hi parts carry exactly 10 mantissa bits, so the result is
// the same whether the MMA truncates or rounds its fp32 inputs.
//
// Tile 128 (m) x 128 (c), k step 32 channels (one 128-byte swizzled row per
// operand row), 4 pipeline slots of A, B_hi, B_lo (48 KB each) in shared
// memory; the split A of each slot lives in tensor memory (A operand of the
// MMA), so shared memory carries only the TMA writes, one read of A and the
// MMA's reads of B.  Roles (one CTA per SM, persistent over the tiles):
//   warps 0-3   epilogue: tcgen05.ld of the fp32 accumulator (warp q reads
//               TMEM lanes 32q..32q+31 = tile rows), staged through shared
//               memory and written as 16-byte stores, 8 lanes per 128 bytes of
//               a dx pixel; before the first tile they zero the dx pixels no
//               class writes;
//   warp 4      A producer: one TMA im2col load of the 128 A rows per stage
//               (the class's map walks its (n, ht, wt) rows, the tap is the
//               im2col offset, rows outside dy read as zero) and the stage's
//               byte count;
//   warp 5      TMEM allocation and the single-thread tcgen05.mma issue
//               (kind::tf32, M=128, N=128, K=8, A from TMEM, B from shared
//               memory), committing each stage back to its slot and each
//               finished tile to the epilogue (accumulator double-buffered in
//               TMEM);
//   warp 6      B producer: the hi and lo boxes of the pre-split filter
//               (k contiguous, so B is K-major like A);
//   warps 7-10  split A: each thread reads one landed A row (its TMEM lane),
//               writes hi and lo to the slot's 64 TMEM columns (tcgen05.st),
//               waits for the stores and arrives.
// Every barrier wait is bounded; on a timeout the kernel records the status
// word, drains what it started and returns.
#include <cuda.h>
#include <stdint.h>

#include <algorithm>

#include "device_util.cuh"
#include "internal.h"
#include "tc_common.cuh"
#include "tf32.h"

namespace cbd {

constexpr int32_t kDevTimeoutConvert = 0x105;

struct Tf32Cfg {
    static constexpr int BN = kTf32BN;
    static constexpr int STAGES = 4;
    static constexpr int A_BYTES = 128 * 128;  // 128 rows x 32 fp32
    static constexpr int B_BYTES = BN * 128;   // BN rows x 32 fp32
    static constexpr int SLOT_BYTES = A_BYTES + 2 * B_BYTES;  // A (fp32, as loaded), B hi, B lo
    // TMEM: the double-buffered accumulator in columns [0, 2*BN), then per slot
    // the split A (32 columns of hi, 32 of lo; lane = tile row)
    static constexpr int A_COL = 2 * BN;
    static constexpr int TMEM_COLS = 512;
    static constexpr int STAGE_OUT_BYTES = 4 * 32 * 128;  // epilogue staging: 4 warps x 32 rows x 128 B
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM = 1024 + STAGES * SLOT_BYTES + STAGE_OUT_BYTES + BAR_BYTES;
    static constexpr int A_WARP = 4, MMA_WARP = 5, B_WARP = 6, SPLIT_WARP = 7, SPLIT_WARPS = 4;
    static constexpr int SPLIT_THREADS = 32 * SPLIT_WARPS;
    static constexpr int THREADS = 32 * (SPLIT_WARP + SPLIT_WARPS);
};
static_assert(Tf32Cfg::SMEM <= 227 * 1024, "shared memory of the fp32 tensor-core kernel");
static_assert(Tf32Cfg::A_COL + Tf32Cfg::STAGES * 64 <= Tf32Cfg::TMEM_COLS, "tensor memory of the fp32 kernel");

// Instruction descriptor, kind::tf32: fp32 accumulator, tf32 A and B, both
// K-major, M = 128, N = BN.
template <int BN>
__device__ __forceinline__ constexpr uint32_t idesc_tf32() {
    return (1u << 4)                  // D format: f32
           | (2u << 7)                // A format: tf32
           | (2u << 10)               // B format: tf32
           | ((uint32_t)(BN >> 3) << 17)
           | ((uint32_t)(128 >> 4) << 24);
}

// A from tensor memory (lane = row, one 32-bit column per k), B from shared memory.
__device__ __forceinline__ void tc_mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 columns of this warp's 32 TMEM lanes from registers.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

// x rounded to 10 explicit mantissa bits, ties to even (add half an ulp of the
// kept part plus the kept lsb, then clear the 13 dropped bits).  Inf and NaN
// pass unchanged; a value that would round past the largest finite one is
// truncated instead.
__device__ __forceinline__ float tf32_round(float x) {
    const uint32_t u = __float_as_uint(x);
    if ((u & 0x7F800000u) == 0x7F800000u) return x;
    uint32_t r = (u + 0xFFFu + ((u >> 13) & 1u)) & 0xFFFFE000u;
    if ((r & 0x7F800000u) == 0x7F800000u) r = u & 0xFFFFE000u;
    return __uint_as_float(r);
}

// Zero the dx pixels no class writes (fp32 NHWC, 16-byte stores); dx rows are
// spread over the CTAs of the launch as in the bf16 kernels.
__device__ __forceinline__ void fill_uncovered_f32(const TcParams &p, int tid, int nthreads) {
    const Geom &g = p.g;
    const uint32_t cpp = (uint32_t)g.C / 4;     // 16-byte chunks per pixel
    const uint32_t cpr = cpp * (uint32_t)g.Wi;  // per row
    float4 *out = static_cast<float4 *>(p.dx);
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    const uint32_t rows = (uint32_t)g.N * (uint32_t)g.Hi;
    const bool all_cols = p.cov_w == ~0ull;
    for (uint32_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const uint32_t hi = r % (uint32_t)g.Hi;
        float4 *row = out + (size_t)r * cpr;
        if (!((p.cov_h >> (hi % (uint32_t)g.sh)) & 1ull)) {
            for (uint32_t u = tid; u < cpr; u += nthreads) row[u] = z;
        } else if (!all_cols) {
            for (uint32_t u = tid; u < cpr; u += nthreads) {
                const uint32_t wi = u / cpp;
                if (!((p.cov_w >> (wi % (uint32_t)g.sw)) & 1ull)) row[u] = z;
            }
        }
    }
}

// One 32-column chunk of this warp's 32 rows -> dx: each thread writes its
// row's 128 bytes into the warp's 4 KB staging slice (16-byte pieces XOR-
// swizzled by row), then 8 lanes per row store 4 rows per instruction.
__device__ __forceinline__ void store_chunk_f32(const uint32_t (&v)[32], uint32_t sbase, int lane,
                                                const int64_t (&roff)[8], const bool (&rok)[8], int col, int Cg,
                                                float *dx, bool atomic) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const uint32_t a = sbase + (uint32_t)lane * 128u + ((uint32_t)(q ^ (lane & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v[4 * q]), "r"(v[4 * q + 1]),
                     "r"(v[4 * q + 2]), "r"(v[4 * q + 3])
                     : "memory");
    }
    __syncwarp();
    const int ch = lane & 7;
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int row = it * 4 + (lane >> 3);
        const uint32_t a = sbase + (uint32_t)row * 128u + ((uint32_t)(ch ^ (row & 7)) << 4);
        float4 val;
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(val.x), "=f"(val.y), "=f"(val.z), "=f"(val.w)
                     : "r"(a)
                     : "memory");
        if (rok[it] && col + ch * 4 < Cg) {
            float4 *dst = reinterpret_cast<float4 *>(dx + roff[it] + ch * 4);
            if (atomic)
                atomicAdd(dst, val);
            else
                *dst = val;
        }
    }
    __syncwarp();
}

// Drain one warp's 32 accumulator rows (TMEM columns [taddr, taddr + BN)) to
// dx.  `off` is the dx element offset of this thread's row at the tile's
// first channel, `col0` that channel's index within the group; channels >= Cg
// are not written.  The next 32 columns load while the current ones store.
template <int BN>
__device__ __forceinline__ void epilogue_rows_f32(uint32_t taddr, uint8_t *stage, int lane, bool rvalid, int64_t off,
                                                  int col0, int Cg, float *dx, bool atomic) {
    constexpr int NC = BN / 32;
    static_assert(NC % 2 == 0, "chunks are drained in pairs");
    const uint32_t sbase = smem_u32(stage);
    int64_t roff[8];
    bool rok[8];
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int row = it * 4 + (lane >> 3);
        const uint32_t lo = __shfl_sync(0xffffffffu, (uint32_t)(uint64_t)off, row);
        const uint32_t hi = __shfl_sync(0xffffffffu, (uint32_t)((uint64_t)off >> 32), row);
        roff[it] = (int64_t)(((uint64_t)hi << 32) | lo);
        rok[it] = __shfl_sync(0xffffffffu, rvalid ? 1 : 0, row) != 0;
    }
    uint32_t va[32], vb[32];
    tmem_ld32_issue(taddr, va);
    tmem_wait_ld(va);
#pragma unroll 1
    for (int cc = 0; cc < NC; cc += 2) {
        tmem_ld32_issue(taddr + (cc + 1) * 32, vb);
        store_chunk_f32(va, sbase, lane, roff, rok, col0 + cc * 32, Cg, dx + cc * 32, atomic);
        tmem_wait_ld(vb);
        if (cc + 2 < NC) tmem_ld32_issue(taddr + (cc + 2) * 32, va);
        store_chunk_f32(vb, sbase, lane, roff, rok, col0 + (cc + 1) * 32, Cg, dx + (cc + 1) * 32, atomic);
        if (cc + 2 < NC) tmem_wait_ld(va);
    }
}

// Work of CTA w of nw.  Whole tiles w, w + nw, ... below t_dp (every full
// round of tiles); with p.streamk the remaining tiles (fewer than nw) are cut
// into equal ranges of their k blocks, one range per CTA, so that the last
// round occupies every SM.  A range that does not cover its whole tile ends in
// an atomic epilogue (fp32 adds into dx, which the launch before zeroed);
// every tail segment is added atomically, whole or not.
struct Tf32Seg {
    int t, kb0, kb1;
    bool atomic;
};
struct Tf32Iter {
    int nw, T, t_dp, next_t;
    int64_t u, u_end;
    __device__ __forceinline__ Tf32Iter(const TcParams &p, int w, int nw_) : nw(nw_), T(p.total_tiles), next_t(w) {
        t_dp = p.streamk ? (T / nw) * nw : T;
        u = (int64_t)w * p.units_total / nw;
        u_end = (int64_t)(w + 1) * p.units_total / nw;
    }
    __device__ __forceinline__ static int nkb(const TcParams &p, int ci) {
        return p.cls[ci].taps_y * p.cls[ci].taps_x * p.kb_per_tap;
    }
    __device__ __forceinline__ bool next(const TcParams &p, Tf32Seg &sg) {
        if (next_t < t_dp) {
            sg.t = next_t;
            sg.kb0 = 0;
            sg.kb1 = nkb(p, class_of_tile(p, next_t));
            sg.atomic = false;
            next_t += nw;
            return true;
        }
        if (!p.streamk || u >= u_end) return false;
        // tail tiles class by class (each class's tiles are contiguous) to the
        // one that holds unit u
        int64_t base = 0;
        for (int ci = 0; ci < p.num_classes; ++ci) {
            const int tb = p.cls[ci].tile_begin;
            const int te = ci + 1 < p.num_classes ? p.cls[ci + 1].tile_begin : T;
            const int lo = tb > t_dp ? tb : t_dp;
            if (lo >= te) continue;
            const int n = nkb(p, ci);
            const int64_t cu = (int64_t)(te - lo) * n;
            if (u < base + cu) {
                const int tl = (int)((u - base) / n);
                const int64_t ts = base + (int64_t)tl * n;  // unit of this tile's k block 0
                sg.t = lo + tl;
                sg.kb0 = (int)(u - ts);
                sg.kb1 = (int)(u_end - ts < n ? u_end - ts : n);
                sg.atomic = true;
                u = ts + sg.kb1;
                return true;
            }
            base += cu;
        }
        return false;
    }
};

// Zero the dx region of every tail tile (t >= t_dp) before the kernel adds
// its k-block ranges into it: one block per tile, 128 rows x 128 channels.
__global__ void __launch_bounds__(256) tf32_zero_tiles_kernel(const __grid_constant__ TcParams p, int t_dp) {
    const Geom &g = p.g;
    float *dx = static_cast<float *>(p.dx);
    for (int t = t_dp + blockIdx.x; t < p.total_tiles; t += gridDim.x) {
        const TileCoord tcd = decode_tile(p, t);
        const ClassDesc &c = p.cls[tcd.ci];
        const int HTWT = c.HT * c.WT;
        for (int e = threadIdx.x; e < 128 * (kTf32BN / 4); e += blockDim.x) {
            const int r = e / (kTf32BN / 4), q = e % (kTf32BN / 4);
            const int m = tcd.mb * 128 + r;
            const int col = tcd.nb * kTf32BN + 4 * q;
            if (m >= c.M || col >= g.Cg) continue;
            const int n = m / HTWT, rem = m - n * HTWT;
            const int hi = (c.ht_lo + rem / c.WT) * g.sh + c.ty * g.dh - g.ph;
            const int wi = (c.wt_lo + rem % c.WT) * g.sw + c.tx * g.dw - g.pw;
            const int64_t off = (((int64_t)n * g.Hi + hi) * g.Wi + wi) * g.C + (int64_t)tcd.gi * g.Cg + col;
            *reinterpret_cast<float4 *>(dx + off) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
}

__global__ void __launch_bounds__(Tf32Cfg::THREADS, 1) tf32_dgrad_kernel(const __grid_constant__ TcParams p) {
    using Cfg = Tf32Cfg;
    constexpr int S = Cfg::STAGES;
    constexpr int BN = Cfg::BN;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *stage = smem + S * Cfg::SLOT_BYTES;  // epilogue staging (1024-aligned)
    uint64_t *bars = reinterpret_cast<uint64_t *>(stage + Cfg::STAGE_OUT_BYTES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3 * S + 4);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(tmem_slot + 1);

    // slot s: [A (fp32, as loaded) | B_hi | B_lo]; its split A sits in TMEM columns A_COL + 64 s
    auto slot_a = [&](uint32_t s) { return smem_u32(smem + s * Cfg::SLOT_BYTES); };
    const uint32_t full0 = smem_u32(bars), split0 = smem_u32(bars + S), empty0 = smem_u32(bars + 2 * S);
    const uint32_t tfull0 = smem_u32(bars + 3 * S), tempty0 = smem_u32(bars + 3 * S + 2);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const Geom &g = p.g;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);                       // the A producer's arrive.expect_tx
            mbar_init(split0 + 8 * s, Cfg::SPLIT_THREADS);     // every splitting thread
            mbar_init(empty0 + 8 * s, 1);                      // the stage's MMA commit
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
    if (warp == Cfg::A_WARP && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_w)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_w_half)) : "memory");
        for (int ci = 0; ci < p.num_classes; ++ci)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_a[ci])) : "memory");
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == Cfg::A_WARP || warp == Cfg::B_WARP) {
        // ------------------------------------------------------------ producers (TMA)
        const bool do_a = warp == Cfg::A_WARP;
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true, issued = false;
            Tf32Iter segs(p, blockIdx.x, gridDim.x);
            Tf32Seg sg;
            while (ok && segs.next(p, sg)) {
                const TileCoord tcd = decode_tile(p, sg.t);
                const ClassDesc &c = p.cls[tcd.ci];
                // first row of the tile -> base pixel of tap (taps_y-1, taps_x-1)
                const int HTWT = c.HT * c.WT;
                const int m0 = tcd.mb * 128;
                const int n0 = m0 / HTWT, rem = m0 - n0 * HTWT;
                const int bh = c.ht_lo + rem / c.WT - (c.taps_y - 1) * g.DH;
                const int bw = c.wt_lo + rem % c.WT - (c.taps_x - 1) * g.DW;
                const CUtensorMap *amap = &p.tmap_a[tcd.ci];
                for (int kb = sg.kb0; kb < sg.kb1; ++kb, ++it) {
                    const int tap = kb / p.kb_per_tap;
                    const int k0 = (kb - tap * p.kb_per_tap) * kTf32BK;
                    const int j = tap / c.taps_x, i = tap - j * c.taps_x;
                    const uint32_t s = it % S, ph = (it / S) & 1;
                    if (!mbar_wait_bounded(empty0 + 8 * s, ph ^ 1, p.wait_budget, abort_flag, p.status,
                                           kDevTimeoutProducer)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full_s = full0 + 8 * s;
                    const uint32_t a_dst = slot_a(s);
                    // (the B boxes may land before this arrive: the transaction
                    // count dips below zero while the single arrival is pending)
                    if (do_a) {
                        mbar_arrive_expect_tx(full_s, (uint32_t)(Cfg::A_BYTES + 2 * Cfg::B_BYTES));
                        tma_load_im2col(a_dst, amap, full_s, tcd.gi * g.Kg + k0, bw, bh, n0,
                                        (uint16_t)((c.taps_x - 1 - i) * g.DW), (uint16_t)((c.taps_y - 1 - j) * g.DH));
                    } else {
                        const int y = c.ty + g.YT * j, x = c.tx + g.XT * i;
                        tma_load_5d(a_dst + Cfg::A_BYTES, &p.tmap_w, full_s, k0, x, y, tcd.nb * BN, tcd.gi);
                        tma_load_5d(a_dst + Cfg::A_BYTES + Cfg::B_BYTES, &p.tmap_w_half, full_s, k0, x, y,
                                    tcd.nb * BN, tcd.gi);
                    }
                    issued = true;
                }
            }
            if (!ok && issued) {
                for (int q = 0; q < 100; ++q) __nanosleep(1000);
            }
        }
        __syncwarp();
    } else if (warp >= Cfg::SPLIT_WARP) {
        // ------------------------------------------------------------ A split (4 warps)
        // a warp may address only its quarter of the TMEM lanes: warp q % 4
        // takes tile rows 32*(q % 4) .. +31, one row (32 fp32 = 128 swizzled
        // bytes) per thread, and writes hi and lo as 32 TMEM columns each
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16) + Cfg::A_COL;
        uint32_t it = 0;
        bool ok = true;
        Tf32Iter segs(p, blockIdx.x, gridDim.x);
        Tf32Seg sg;
        while (ok && segs.next(p, sg)) {
            for (int kb = sg.kb0; kb < sg.kb1; ++kb, ++it) {
                const uint32_t s = it % S, ph = (it / S) & 1;
                if (!mbar_wait_bounded(full0 + 8 * s, ph, p.wait_budget, abort_flag, p.status, kDevTimeoutConvert)) {
                    ok = false;
                    break;
                }
                const uint32_t a = slot_a(s) + (uint32_t)row * 128u;
                uint32_t hi[32], lo[32];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    // k = 4j .. 4j+3 sit in 16-byte chunk j, stored at chunk j ^ (row % 8)
                    float4 v;
                    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                                 : "r"(a + ((uint32_t)(j ^ (row & 7)) << 4))
                                 : "memory");
                    const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float h = tf32_round(e[q]);
                        hi[4 * j + q] = __float_as_uint(h);
                        lo[4 * j + q] = __float_as_uint(e[q] - h);
                    }
                }
                tmem_st32(lane_base + s * 64, hi);
                tmem_st32(lane_base + s * 64 + 32, lo);
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                mbar_arrive(split0 + 8 * s);
            }
        }
    } else if (warp == Cfg::MMA_WARP) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_tf32<BN>();
            const uint64_t desc0 = smem_desc_sw128(smem_u32(smem), 16, 1024);
            constexpr uint64_t B_HI = Cfg::A_BYTES >> 4, B_LO = (Cfg::A_BYTES + Cfg::B_BYTES) >> 4;
            uint32_t it = 0, tc = 0;
            bool ok = true, issued = false;
            Tf32Iter segs(p, blockIdx.x, gridDim.x);
            Tf32Seg sg;
            for (; ok && segs.next(p, sg); ++tc) {
                const uint32_t b = tc & 1, tph = (tc >> 1) & 1;
                if (!mbar_wait_bounded(tempty0 + 8 * b, tph ^ 1, p.wait_budget, abort_flag, p.status,
                                       kDevTimeoutMma)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + b * BN;
                for (int kb = sg.kb0; kb < sg.kb1; ++kb, ++it) {
                    const uint32_t s = it % S, ph = (it / S) & 1;
                    // the split barrier follows the TMA barrier (the splitting
                    // threads waited on it), so B has landed and A sits in TMEM
                    if (!mbar_wait_bounded(split0 + 8 * s, ph, p.wait_budget, abort_flag, p.status, kDevTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t d0 = desc0 + (uint64_t)((s * Cfg::SLOT_BYTES) >> 4);
                    const uint32_t a_t = tmem_base + Cfg::A_COL + s * 64;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        // 8-deep k step: 8 TMEM columns of A, 32 bytes along B's 128-byte rows
                        const uint32_t a_hi = a_t + 8 * kk, a_lo = a_t + 32 + 8 * kk;
                        const uint64_t b_hi = d0 + B_HI + 2 * kk, b_lo = d0 + B_LO + 2 * kk;
                        tc_mma_tf32_ts(d_tmem, a_hi, b_hi, idesc, (kb != sg.kb0 || kk != 0) ? 1u : 0u);
                        tc_mma_tf32_ts(d_tmem, a_hi, b_lo, idesc, 1u);
                        tc_mma_tf32_ts(d_tmem, a_lo, b_hi, idesc, 1u);
                    }
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
        const int row = warp * 32 + lane;  // TMEM lane = tile row
        float *dx = static_cast<float *>(p.dx);
        uint32_t tc = 0;
        if (p.fill) fill_uncovered_f32(p, threadIdx.x, 128);
        Tf32Iter segs(p, blockIdx.x, gridDim.x);
        Tf32Seg sg;
        for (; segs.next(p, sg); ++tc) {
            const TileCoord tcd = decode_tile(p, sg.t);
            const ClassDesc &c = p.cls[tcd.ci];
            const uint32_t b = tc & 1, tph = (tc >> 1) & 1;
            bool ok = mbar_wait_bounded(tfull0 + 8 * b, tph, p.wait_budget, abort_flag, p.status, kDevTimeoutEpilogue);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
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
            epilogue_rows_f32<BN>(tbase, stage + warp * 4096, lane, rvalid, off, tcd.nb * BN, g.Cg, dx, sg.atomic);
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

cudaError_t launch_tf32(const TcParams &p, int grid, cudaStream_t s) {
    if (grid <= 0 || p.total_tiles <= 0) return cudaSuccess;
    if (p.streamk) {
        const int t_dp = (p.total_tiles / grid) * grid;
        const int tail = p.total_tiles - t_dp;
        if (tail > 0) {
            tf32_zero_tiles_kernel<<<tail, 256, 0, s>>>(p, t_dp);
            cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return e;
        }
    }
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        cudaError_t e =
            cudaFuncSetAttribute(tf32_dgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Tf32Cfg::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    tf32_dgrad_kernel<<<grid, Tf32Cfg::THREADS, Tf32Cfg::SMEM, s>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Filter split: per group and tap, the [Kg][Cg] plane of w (KYXC: c
// contiguous; GKCYX: c at a stride of the tap count) becomes the [Cg][Kg]
// plane of w_hi / w_lo (k contiguous, planes of one c row a tap apart), in
// 32 x 32 tiles through shared memory so that reads run along c and writes
// along k.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) tf32_split_w_kernel(const float *__restrict__ w, float *__restrict__ w_hi,
                                                           float *__restrict__ w_lo, int G, int Kg, int Cg, int taps,
                                                           int gkcyx) {
    __shared__ float tile[32][33];
    const int kt = (Kg + 31) / 32, ct = (Cg + 31) / 32;
    const int64_t tiles = (int64_t)G * taps * kt * ct;
    const int x = threadIdx.x & 31, y = threadIdx.x >> 5;  // 32 x 8 threads
    // source element strides of (k, c, tap) and destination strides of (c, tap)
    const int64_t s_k = (int64_t)Cg * taps, s_c = gkcyx ? taps : 1, s_t = gkcyx ? 1 : Cg;
    const int64_t d_c = (int64_t)taps * Kg, d_t = Kg;
    for (int64_t tl = blockIdx.x; tl < tiles; tl += gridDim.x) {
        int64_t r = tl;
        const int cb = (int)(r % ct); r /= ct;
        const int kb = (int)(r % kt); r /= kt;
        const int t = (int)(r % taps);
        const int64_t gi = r / taps;
        const float *src = w + gi * Kg * s_k + (int64_t)t * s_t;
        const int64_t dst0 = gi * Cg * d_c + (int64_t)t * d_t;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int k = kb * 32 + y + 8 * q, c = cb * 32 + x;
            tile[y + 8 * q][x] = (k < Kg && c < Cg) ? src[k * s_k + c * s_c] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int c = cb * 32 + y + 8 * q, k = kb * 32 + x;
            if (k < Kg && c < Cg) {
                const float v = tile[x][y + 8 * q];
                const float h = tf32_round(v);
                const int64_t o = dst0 + c * d_c + k;
                w_hi[o] = h;
                w_lo[o] = v - h;
            }
        }
        __syncthreads();
    }
}

cudaError_t launch_tf32_split_w(const float *w, float *w_hi, float *w_lo, const Geom &g, int gkcyx, int num_sms,
                                cudaStream_t s) {
    const int taps = g.Y * g.X;
    const int64_t tiles = (int64_t)g.G * taps * ((g.Kg + 31) / 32) * ((g.Cg + 31) / 32);
    if (tiles <= 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>(tiles, (int64_t)(num_sms > 0 ? num_sms : 148) * 8);
    tf32_split_w_kernel<<<(unsigned)blocks, 256, 0, s>>>(w, w_hi, w_lo, g.G, g.Kg, g.Cg, taps, gkcyx);
    return cudaGetLastError();
}

}  // namespace cbd
