// tc2_sm103.cu -- bf16 NHWC/KYXC dgrad on pairs of SMs (tcgen05 cta_group::2).
//
// Same sub-GEMMs as tc_sm103.cu (one per filter-tap residue class and group,
// the v4r1 backward-data split of pages "Backward data" and "[igemm_dynamic]
// v4r1 bwd dynamic kernel"), but each output tile is 256 (m) x BN (c), BN in
// {128, 256, 512}, and is computed by a cluster of two CTAs on two SMs:
//   * CTA rank r of the pair loads the tile's A rows [128r, 128r+128) (TMA
//     im2col, one map per class, exactly as in the 1-SM kernel) and its half
//     of the B columns of every MMA of the tile (TMA boxes of 64 k x 64 c)
//     into its own shared memory.  Both CTAs' loads complete on the leader's
//     (rank 0) stage barrier (`.cta_group::2` TMA), which expects the bytes of
//     both.
//   * The leader's single MMA thread issues M=256, N=min(BN, 256), K=16
//     `tcgen05.mma.cta_group::2` instructions (two per k slice for BN=512)
//     that read A and B from both CTAs' shared memory and accumulate rows
//     [128r, 128r+128) in CTA r's TMEM; each stage is committed back to both
//     CTAs' empty barriers and each finished tile to both CTAs'
//     accumulator-full barriers (one commit that arrives on the barrier of
//     both CTAs of the pair).
//   * Each CTA's four epilogue warps drain their own TMEM rows (RNE to bf16,
//     16-byte stores to the class's strided dx pixels) and release the
//     leader's accumulator-empty barrier (remote arrive from the peer).
// Per SM and per 128x256x64 step this moves 32 KB of operands into shared
// memory instead of 48 KB (each SM loads only half of B); a 512-wide tile
// moves 24 KB per 128x256x64 of work.  Every CTA fetches its own operands
// from L2 (no multicast); the pairs are bound by that operand delivery
// (~40 bytes per SM clock measured), which is why the widest tile runs
// closest to the MMA rate.
// Schedules: whole tiles in LPT class order over the persistent pairs; or
// (SegmentIter) split-K, where S pairs share each 256 x 512 tile over 1/S of
// its k-blocks and exchange fp32 partials through a workspace so that each
// pair adds and stores 1/S of the columns (the epilogue's reduce-scatter); or
// the opt-in stream-K.  PLAIN instantiations read A as a plain matrix.
// Every barrier wait is bounded; both CTAs meet in a cluster barrier before
// deallocating TMEM and exiting.
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "device_util.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace cbd {

// First column of split s's slice of a BN-wide tile cut into S slices
// (multiples of 64 columns; slice S - 1 ends at BN).
__device__ __forceinline__ int split_col(int s, int S, int BN) { return (s * BN / S) / 64 * 64; }

// one non-blocking test of an mbarrier phase
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

template <int BN_>
struct Tc2Cfg {
    static constexpr int BN = BN_;          // tile width of the pair: 128, 256 or 512
    static constexpr int BNH = BN / 2;      // columns of B held by each CTA
    // one MMA instruction is at most 256 wide: a 512-wide tile issues two per
    // 16-deep k slice (columns [0, 256) and [256, 512) of the tile), which
    // halves the A bytes per output column; its accumulator takes all 512
    // TMEM columns, so it is single-buffered
    static constexpr int MMA_N = BN < 256 ? BN : 256;
    static constexpr int NMMA = BN / MMA_N;
    static constexpr int QPM = MMA_N / 128;  // 64-column B boxes per MMA per CTA
    static constexpr int STAGES = BN == 512 ? 4 : BN == 256 ? 6 : 8;
    static constexpr int ACC_BUFS = BN == 512 ? 1 : 2;
    static constexpr int A_BYTES = 128 * 64 * 2;
    static constexpr int B_BYTES = BNH * 64 * 2;
    static constexpr int TMEM_COLS = ACC_BUFS * BN;
    static constexpr int STAGE_OUT_BYTES = 4 * 32 * 128;  // epilogue staging: 4 warps x 32 rows x 128 B
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM = 1024 + STAGES * (A_BYTES + B_BYTES) + STAGE_OUT_BYTES + BAR_BYTES;
    static constexpr int MMA_WARP = 5;
    // TMA issue is serialised per issuing thread, so the loads of a stage are
    // spread over warps on different SM sub-partitions: warps 6.. issue the
    // 64-column B boxes (one or two each), warp 4 the A loads -- on tiles
    // narrower than 512 (a stage every 256 or 512 MMA clocks) alternating with
    // warp A2_WARP (odd stages), which took the 1x1 stride-2 layer's main loop
    // from 13.3 to 11.7 us.
    static constexpr int B_WARP = 6;
    static constexpr int BOXES = BNH / 64;
    static constexpr int B_WARPS = BOXES < 2 ? BOXES : 2;
    static constexpr int BOXES_PER_WARP = BOXES / B_WARPS;
    static constexpr int A2_WARP = BN < 512 ? B_WARP + B_WARPS : -1;
    static constexpr int THREADS = 32 * (B_WARP + B_WARPS + (BN < 512 ? 1 : 0));
};

// PLAIN: the specialisation for plans whose every class reads dy as a plain
// matrix (one tap per class, the class rows covering all of dy's pixels in
// order, e.g. 1x1 filters and the 1x2 stride-(1,2) layer): A rows come from a
// 2-D tiled map {K, N*Ho*Wo} at row m, with no im2col offsets.  The dynamic
// kernel (PLAIN = false) serves every shape with the same tiles.
template <int BN_, bool PLAIN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Tc2Cfg<BN_>::THREADS, 1)
    tc2_dgrad_kernel(const __grid_constant__ TcParams p) {
    using Cfg = Tc2Cfg<BN_>;
    constexpr int S = Cfg::STAGES;
    constexpr int BN = Cfg::BN;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + S * Cfg::A_BYTES;
    uint8_t *stage = sB + S * Cfg::B_BYTES;  // epilogue staging (1024-aligned)
    uint64_t *bars = reinterpret_cast<uint64_t *>(stage + Cfg::STAGE_OUT_BYTES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * S + 4);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(tmem_slot + 1);
    const uint32_t gather_bar = smem_u32(bars + 2 * S + 5);  // split-K: partials landed in shared memory

    const uint32_t rank = cluster_ctarank();  // CTA within the pair: 0 = leader
    const uint32_t pl = 0;                    // cluster rank of the pair's leader
    const bool leader = rank == 0;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S);
    const uint32_t tfull0 = smem_u32(bars + 2 * S), tempty0 = smem_u32(bars + 2 * S + 2);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const Geom &g = p.g;
    // scheduling unit: the pair (cluster of two CTAs)
    const int pair = blockIdx.x / 2, npairs = gridDim.x / 2;
    // 512-wide whole tiles: the epilogue releases the accumulator by 256-column
    // halves (tempty[0], tempty[1]), so the next tile's MMAs into the first half
    // start while the second is drained
    const bool half_release = BN == 512 && p.splitk <= 1 && !p.streamk;
    if (threadIdx.x == 0) CBD_PHASE(p, kPhEntry);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);   // leader: one arrive.expect_tx for both CTAs' bytes
            mbar_init(empty0 + 8 * s, 1);   // one commit per stage from the leader's MMA thread
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull0 + 8 * b, 1);   // one commit per tile
            mbar_init(tempty0 + 8 * b, 8);  // leader: 4 epilogue warps of each CTA
        }
        mbar_init(gather_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async_smem();
    }
    if (warp == Cfg::MMA_WARP) {
        tmem_alloc2(smem_u32(tmem_slot), Cfg::TMEM_COLS);
        tc_fence_before();
    }
    if (warp == 4 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_w)) : "memory");
        for (int ci = 0; ci < p.num_classes; ++ci)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_a[ci])) : "memory");
    }
    // barriers of both CTAs initialised and TMEM allocated before any remote operation
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (threadIdx.x == 0) CBD_PHASE(p, kPhSetup);
    if (threadIdx.x == 0 && !leader) {
        // the pair's MMAs write this CTA's rows at the leader's TMEM address
        if (ld_shared_cluster_u32(mapa_shared(smem_u32(tmem_slot), pl)) != tmem_base)
            record_status(p.status, kDevFaultIndex);
    }

    if (warp == 4 || warp >= Cfg::B_WARP) {
        // ------------------------------------------------------------ producers
        const bool do_a = warp == 4 || warp == Cfg::A2_WARP;  // A loads + the stage's byte count
        const uint32_t a_par = warp == Cfg::A2_WARP ? 1u : 0u;  // the A issuers split the stages by parity
        // B boxes of this warp
        const int cb_lo = do_a ? 0 : (warp - Cfg::B_WARP) * Cfg::BOXES_PER_WARP;
        const int cb_hi = do_a ? 0 : cb_lo + Cfg::BOXES_PER_WARP;
        if (lane == 0) {
            const uint32_t full_leader0 = mapa_shared(full0, pl);
            uint32_t it = 0;
            bool ok = true, issued = false;
            if (do_a) CBD_PHASE(p, kPhProdStart);
            SegmentIter segs(p, pair, npairs);
            Segment sg;
            while (ok && segs.next(p, sg)) {
                if (do_a && it == 0) CBD_PHASE(p, kPhProdSeg);
                const TileCoord tcd = decode_tile(p, sg.t);
                const ClassDesc &c = p.cls[tcd.ci];
                const int HTWT = c.HT * c.WT;
                const int m0 = tcd.mb * 256 + (int)rank * 128;
                const int n0 = m0 / HTWT, rem = m0 - n0 * HTWT;
                const int bh = c.ht_lo + rem / c.WT - (c.taps_y - 1) * g.DH;
                const int bw = c.wt_lo + rem % c.WT - (c.taps_x - 1) * g.DW;
                const CUtensorMap *amap = &p.tmap_a[tcd.ci];
                if (do_a && it == 0) CBD_PHASE(p, kPhProdTile);
                for (int kb = sg.kb0; kb < sg.kb1; ++kb, ++it) {
                    if (Cfg::A2_WARP >= 0 && do_a && (it & 1u) != a_par) continue;  // the other A issuer's stage
                    const int tap = kb / p.kb_per_tap;
                    const int k0 = (kb - tap * p.kb_per_tap) * 64;
                    const int j = tap / c.taps_x, i = tap - j * c.taps_x;
                    const uint32_t s = it % S, ph = (it / S) & 1;
                    if (do_a && it == 0) CBD_PHASE(p, kPhProdPreWait);
                    if (!mbar_wait_bounded(empty0 + 8 * s, ph ^ 1, p.wait_budget, abort_flag, p.status,
                                           kDevTimeoutProducer)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bar = full_leader0 + 8 * s;
                    if (do_a && it == 0) CBD_PHASE(p, kPhProdWaited);
                    // (B loads of a split producer may complete before this arrive:
                    // the transaction count dips below zero while the arrival is
                    // still pending, so the phase cannot complete early)
                    if (do_a) {
                        if (leader)
                            mbar_arrive_expect_tx(full0 + 8 * s, (uint32_t)(2 * (Cfg::A_BYTES + Cfg::B_BYTES)));
                        if constexpr (PLAIN)
                            tma_load_2d_pair(smem_u32(sA + s * Cfg::A_BYTES), amap, bar, tcd.gi * g.Kg + k0, m0);
                        else
                            tma_load_im2col_pair(smem_u32(sA + s * Cfg::A_BYTES), amap, bar, tcd.gi * g.Kg + k0, bw,
                                                 bh, n0, (uint16_t)((c.taps_x - 1 - i) * g.DW),
                                                 (uint16_t)((c.taps_y - 1 - j) * g.DH));
                        if (it == 0) CBD_PHASE(p, kPhFirstIssue);
                    }
                    const uint32_t bdst = smem_u32(sB + s * Cfg::B_BYTES);
                    // box q feeds MMA q / QPM: this CTA's half of that MMA's columns
                    for (int cb = cb_lo; cb < cb_hi; ++cb) {
                        const int col = tcd.nb * BN + (cb / Cfg::QPM) * Cfg::MMA_N + (int)rank * (Cfg::MMA_N / 2) +
                                        (cb % Cfg::QPM) * 64;
                        tma_load_5d_pair(bdst + cb * 8192, &p.tmap_w, bar, col, c.tx + g.XT * i, c.ty + g.YT * j, k0,
                                         tcd.gi);
                    }
                    if (warp == Cfg::B_WARP && it == 0) CBD_PHASE(p, kPhBFirst);
                    issued = true;
                }
            }
            if (do_a && issued) CBD_PHASE(p, kPhLastIssue);
            if (!ok && issued) {
                for (int q = 0; q < 100; ++q) __nanosleep(1000);
            }
        }
        __syncwarp();
    } else if (warp == Cfg::MMA_WARP) {
        // ------------------------------------------------------------ MMA (leader only)
        if (leader && lane == 0) {
            constexpr uint32_t idesc = idesc_bf16<Cfg::MMA_N, 256>();
            const uint64_t a_desc0 = smem_desc_sw128(smem_u32(sA), 16, 1024);
            const uint64_t b_desc0 = smem_desc_sw128(smem_u32(sB), 8192, 1024);
            uint32_t it = 0, tc = 0;
            bool ok = true, issued = false;
            SegmentIter segs(p, pair, npairs);
            Segment sg;
            for (; ok && segs.next(p, sg); ++tc) {
                const uint32_t b = tc % Cfg::ACC_BUFS, tph = (tc / Cfg::ACC_BUFS) & 1;
                if (!mbar_wait_bounded(tempty0 + 8 * b, tph ^ 1, p.wait_budget, abort_flag, p.status,
                                       kDevTimeoutMma)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (tc == 1) CBD_PHASE(p, kPhMma1Start);
                const uint32_t d_tmem = tmem_base + b * BN;
                if (half_release) {
                    // 512-wide whole tiles: columns [0, 256) are free (tempty[0]);
                    // the N = 256 MMAs into [256, 512) wait for tempty[1], so the
                    // stages they need are held (at most S) until the epilogue has
                    // drained that half.  Each column's k order is unchanged.
                    bool h1 = mbar_test_wait(tempty0 + 8, tph ^ 1);
                    if (h1) tc_fence_after();
                    int pend = sg.kb0;            // first k-block whose upper-half MMAs are pending
                    const uint32_t it0 = it;      // stage counter at k-block kb0
                    auto upper = [&](int q) {
                        const uint32_t sq = (it0 + (uint32_t)(q - sg.kb0)) % S;
                        const uint64_t ad0 = a_desc0 + (uint64_t)((sq * Cfg::A_BYTES) >> 4);
                        const uint64_t bd0 = b_desc0 + (uint64_t)((sq * Cfg::B_BYTES) >> 4);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_mma2(d_tmem + Cfg::MMA_N, ad0 + (uint64_t)(2 * kk),
                                    bd0 + (uint64_t)(128 * kk + ((Cfg::QPM * 8192) >> 4)), idesc,
                                    (q != sg.kb0 || kk != 0) ? 1u : 0u);
                        tc_commit2_mc(empty0 + 8 * sq, (uint16_t)0x3);
                    };
                    for (int kb = sg.kb0; kb < sg.kb1; ++kb, ++it) {
                        const uint32_t s = it % S, ph = (it / S) & 1;
                        if (!mbar_wait_bounded(full0 + 8 * s, ph, p.wait_budget, abort_flag, p.status,
                                               kDevTimeoutMma)) {
                            ok = false;
                            break;
                        }
                        if (it == 0) CBD_PHASE(p, kPhFirstFull);
                        const uint64_t ad0 = a_desc0 + (uint64_t)((s * Cfg::A_BYTES) >> 4);
                        const uint64_t bd0 = b_desc0 + (uint64_t)((s * Cfg::B_BYTES) >> 4);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_mma2(d_tmem, ad0 + (uint64_t)(2 * kk), bd0 + (uint64_t)(128 * kk), idesc,
                                    (kb != sg.kb0 || kk != 0) ? 1u : 0u);
                        issued = true;
                        if (!h1) {
                            h1 = mbar_test_wait(tempty0 + 8, tph ^ 1);
                            if (!h1 && kb + 1 - pend >= S) {  // every stage held: wait for the upper half
                                if (!mbar_wait_bounded(tempty0 + 8, tph ^ 1, p.wait_budget, abort_flag, p.status,
                                                       kDevTimeoutMma)) {
                                    ok = false;
                                    break;
                                }
                                h1 = true;
                            }
                            if (h1) tc_fence_after();
                        }
                        if (h1) {
                            for (; pend <= kb; ++pend) upper(pend);
                        }
                    }
                    if (ok && pend < sg.kb1) {
                        if (!mbar_wait_bounded(tempty0 + 8, tph ^ 1, p.wait_budget, abort_flag, p.status,
                                               kDevTimeoutMma)) {
                            ok = false;
                        } else {
                            tc_fence_after();
                            for (; pend < sg.kb1; ++pend) upper(pend);
                        }
                    }
                    if (!ok) break;
                    tc_commit2_mc(tfull0 + 8 * b, (uint16_t)0x3);
                    if (tc == 0) CBD_PHASE(p, kPhMma0Done);
                    CBD_PHASE(p, kPhMmaLast);
                    continue;
                }
                for (int kb = sg.kb0; kb < sg.kb1; ++kb, ++it) {
                    const uint32_t s = it % S, ph = (it / S) & 1;
                    // the stage barrier orders the TMA writes of both CTAs before the MMA
                    // reads them; no tcgen05 fence is needed per stage
                    if (!mbar_wait_bounded(full0 + 8 * s, ph, p.wait_budget, abort_flag, p.status, kDevTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    if (it == 0) CBD_PHASE(p, kPhFirstFull);
                    // descriptors: start address in 16-byte units in the low bits; k step of
                    // 16 elements = 32 bytes in A (K-major), 16 rows = 2048 bytes in B (MN-major)
                    const uint64_t ad0 = a_desc0 + (uint64_t)((s * Cfg::A_BYTES) >> 4);
                    const uint64_t bd0 = b_desc0 + (uint64_t)((s * Cfg::B_BYTES) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                        for (int h = 0; h < Cfg::NMMA; ++h)
                            tc_mma2(d_tmem + h * Cfg::MMA_N, ad0 + (uint64_t)(2 * kk),
                                    bd0 + (uint64_t)(128 * kk + h * ((Cfg::QPM * 8192) >> 4)), idesc,
                                    (kb != sg.kb0 || kk != 0) ? 1u : 0u);
                    issued = true;
                    // the slot of both CTAs is free once these MMAs have read it
                    tc_commit2_mc(empty0 + 8 * s, (uint16_t)0x3);
                }
                if (!ok) break;
                tc_commit2_mc(tfull0 + 8 * b, (uint16_t)0x3);
                if (tc == 0) CBD_PHASE(p, kPhMma0Done);
                CBD_PHASE(p, kPhMmaLast);
            }
            if (!ok && issued) {
                for (int q = 0; q < 100; ++q) __nanosleep(1000);
            }
        }
        __syncwarp();
    } else if (warp < 4) {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int row = warp * 32 + lane;  // TMEM lane = this CTA's tile row
        __nv_bfloat16 *dx = static_cast<__nv_bfloat16 *>(p.dx);
        const uint32_t tempty_leader0 = mapa_shared(tempty0, pl);
        uint32_t tc = 0;
        if (p.fill) fill_uncovered(p, threadIdx.x, 128);  // threads 0..127 are the epilogue warps
        if (threadIdx.x == 0) CBD_PHASE(p, kPhFillDone);
        SegmentIter segs(p, pair, npairs);
        Segment sg;
        const size_t slot_f4 = (size_t)(BN / 4) * 128;  // one CTA's 128 x BN fp32 partial, in float4
        for (; segs.next(p, sg); ++tc) {
            const TileCoord tcd = decode_tile(p, sg.t);
            const ClassDesc &c = p.cls[tcd.ci];
            const uint32_t b = tc % Cfg::ACC_BUFS, tph = (tc / Cfg::ACC_BUFS) & 1;
            bool ok = mbar_wait_bounded(tfull0 + 8 * b, tph, p.wait_budget, abort_flag, p.status, kDevTimeoutEpilogue);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            if (threadIdx.x == 0 && tc < 2) CBD_PHASE(p, tc == 0 ? kPhEpi0Start : kPhEpi1Start);
            const uint32_t tbase = tmem_base + ((uint32_t)(warp * 32) << 16) + b * BN;
            const int m = tcd.mb * 256 + (int)rank * 128 + row;
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
            if (p.splitk > 1) {
                // split-K reduce-scatter: column slice s of the tile is stored by
                // the tile's split s.  Every split parks its fp32 partial of the
                // other slices in the workspace (per tile: [CTA rank][contributor]
                // blocks of BN/4 x 128 float4, the contributor index skipping the
                // slice's own split), raises its flag, then adds the other splits'
                // partials of its own slice while draining it to dx.
                const int S = p.splitk, q = sg.split;
                const size_t blk = (size_t)(BN / 4) * 128;
                float4 *tile_ws = p.partials + (size_t)sg.t * 2 * (S - 1) * blk;
                for (int s2 = 0; s2 < S; ++s2) {
                    if (s2 == q) continue;
                    const int lo = split_col(s2, S, BN), hi = split_col(s2 + 1, S, BN);
                    const int r = q < s2 ? q : q - 1;
                    store_partial_chunks(tbase + lo, (hi - lo) / 64, row,
                                         tile_ws + ((size_t)rank * (S - 1) + r) * blk + (size_t)(lo / 4) * 128);
                }
                __threadfence();
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (threadIdx.x == 0) CBD_PHASE(p, kPhEpi1Start);  // partials of the other slices written
                const int lo = split_col(q, S, BN), hi = split_col(q + 1, S, BN);
                // The other splits' partials of this slice: (S - 1) contiguous
                // blocks of (hi - lo) x 512 bytes.  They land in the pipeline's
                // shared memory (free: the tile's MMAs are done and this pair
                // has no other segment) with one bulk copy each, so the sum below
                // reads shared memory instead of waiting on L2 per 32 columns.
                const uint32_t part_bytes = (uint32_t)(hi - lo) * 512u;
                const bool land =
                    (uint64_t)(S - 1) * part_bytes <= (uint64_t)Cfg::STAGES * (Cfg::A_BYTES + Cfg::B_BYTES);
                const float4 *parts_g = tile_ws + (size_t)rank * (S - 1) * blk + (size_t)(lo / 4) * 128;
                if (threadIdx.x == 0) {
                    st_release_gpu(p.flags + ((size_t)sg.t * S + q) * 2 + rank, p.epoch);
                    // the other splits of this tile (same CTA rank), bounded wait each
                    for (int s2 = 0; s2 < S; ++s2) {
                        if (s2 == q) continue;
                        const int32_t *f = p.flags + ((size_t)sg.t * S + s2) * 2 + rank;
                        const long long t0 = clock64();
                        while (ld_acquire_gpu(f) != p.epoch) {
                            if (clock64() - t0 > p.wait_budget) {
                                record_status(p.status, kDevTimeoutPartial);
                                break;
                            }
                        }
                    }
                    CBD_PHASE(p, kPhMma1Start);  // (split-K: the other splits' flags acquired)
                    if (land && part_bytes > 0) {
                        fence_proxy_async_global();  // generic-proxy writes of the other SMs, read by the copy engine
                        mbar_arrive_expect_tx(gather_bar, (uint32_t)(S - 1) * part_bytes);
                        for (int r = 0; r < S - 1; ++r)
                            bulk_load_g2s(smem_u32(sA) + (uint32_t)r * part_bytes, parts_g + (size_t)r * blk,
                                          part_bytes, gather_bar);
                    }
                }
                asm volatile("bar.sync 1, 128;" ::: "memory");
                for (int s2 = 0; s2 < S; ++s2)  // each thread's own acquire of the partials it reads
                    if (s2 != q) (void)ld_acquire_gpu(p.flags + ((size_t)sg.t * S + s2) * 2 + rank);
                const float4 *parts = parts_g;
                size_t pstride = blk;
                if (land && part_bytes > 0) {
                    // on a timeout the status word is set and the sum reads whatever landed
                    (void)mbar_wait_bounded(gather_bar, 0, p.wait_budget, abort_flag, p.status, kDevTimeoutPartial);
                    parts = reinterpret_cast<const float4 *>(sA);
                    pstride = part_bytes / 16;
                }
                if (threadIdx.x == 0) CBD_PHASE(p, kPhEpi1Done);  // partials landed
                epilogue_chunks(tbase + lo, (hi - lo) / 64, stage + warp * 4096, lane, rvalid, off + lo,
                                tcd.nb * BN + lo, g.Cg, dx, parts, S - 1, pstride, row);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(tempty_leader0 + 8 * b);
                continue;
            }
            if (!sg.owner) {
                // stream-K contributor: park the fp32 partial, then raise this CTA's flag
                store_partial_rows<BN>(tbase, row, p.partials + (size_t)(pair * 2 + rank) * slot_f4);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(tempty_leader0 + 8 * b);
                __threadfence();
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (threadIdx.x == 0) st_release_gpu(p.flags + pair * 2 + rank, p.epoch);
                continue;
            }
            const int nparts = pair - sg.q_first;
            if (nparts > 0) {
                // partials of the earlier stretches of this tile (bounded wait per worker)
                for (int q = sg.q_first; q < pair; ++q) {
                    const int32_t *f = p.flags + q * 2 + rank;
                    const long long t0 = clock64();
                    while (ld_acquire_gpu(f) != p.epoch) {
                        if (clock64() - t0 > p.wait_budget) {
                            record_status(p.status, kDevTimeoutPartial);
                            break;
                        }
                    }
                }
            }
            const float4 *parts = nparts > 0 ? p.partials + (size_t)(sg.q_first * 2 + rank) * slot_f4 : nullptr;
            if (half_release) {
                // columns [0, 256), then release that half; then [256, 512)
                epilogue_chunks(tbase, 4, stage + warp * 4096, lane, rvalid, off, tcd.nb * BN, g.Cg, dx);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(tempty_leader0);
                epilogue_chunks(tbase + 256, 4, stage + warp * 4096, lane, rvalid, off + 256, tcd.nb * BN + 256, g.Cg,
                                dx);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(tempty_leader0 + 8);
            } else {
                epilogue_rows<BN>(tbase, stage + warp * 4096, lane, rvalid, off, tcd.nb * BN, g.Cg, dx, parts, nparts,
                                  2 * slot_f4, row);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(tempty_leader0 + 8 * b);
            }
            if (threadIdx.x == 0) {
                if (tc < 2) CBD_PHASE(p, tc == 0 ? kPhEpi0Done : kPhEpi1Done);
                CBD_PHASE(p, kPhEpiLast);
            }
        }
    }

    // no remote arrive or MMA may target a CTA that has left
    cluster_sync_all();
    if (threadIdx.x == 0) CBD_PHASE(p, kPhExit);
    if (warp == Cfg::MMA_WARP) {
        tc_fence_after();
        tmem_dealloc2(tmem_base, Cfg::TMEM_COLS);
    }
}

template <int BN, bool PLAIN>
static cudaError_t launch_tc2_bn(const TcParams &p, int grid, cudaStream_t s) {
    using Cfg = Tc2Cfg<BN>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(tc2_dgrad_kernel<BN, PLAIN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Cfg::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    tc2_dgrad_kernel<BN, PLAIN><<<grid, Cfg::THREADS, Cfg::SMEM, s>>>(p);
    return cudaGetLastError();
}

template <bool PLAIN>
static cudaError_t launch_tc2_a(const TcParams &p, int bn, int grid, cudaStream_t s) {
    if (bn == 512) return launch_tc2_bn<512, PLAIN>(p, grid, s);
    return bn == 256 ? launch_tc2_bn<256, PLAIN>(p, grid, s) : launch_tc2_bn<128, PLAIN>(p, grid, s);
}

cudaError_t launch_tc2(const TcParams &p, int bn, int grid, cudaStream_t s) {
    if (grid <= 0 || p.total_tiles <= 0) return cudaSuccess;
    return p.a_plain ? launch_tc2_a<true>(p, bn, grid, s) : launch_tc2_a<false>(p, bn, grid, s);
}

// SM pairs (clusters of two CTAs, one CTA per SM) that can be resident at once.
int tc2_max_pairs(int num_sms) {
    static int cached[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev];
    using Cfg = Tc2Cfg<256>;
    cudaFuncSetAttribute(tc2_dgrad_kernel<256, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(num_sms & ~1), 1, 1);
    cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, tc2_dgrad_kernel<256, false>, &cfg) != cudaSuccess ||
        clusters <= 0) {
        cudaGetLastError();
        clusters = num_sms / 2;
    }
    if (dev >= 0 && dev < 64) cached[dev] = clusters;
    return clusters;
}

}  // namespace cbd
