// tc_common.cuh -- PTX wrappers and tile bookkeeping shared by the 1-SM and
// 2-SM tcgen05 dgrad kernels: TMA (tile, im2col), mbarriers, TMEM
// allocation, tcgen05.mma / commit / ld, shared-memory matrix descriptors and
// the instruction descriptor for bf16 x bf16 -> fp32.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "device_util.cuh"
#include "internal.h"

namespace cbd {

// --- PTX wrappers ----------------------------------------------------------
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c0, int c1,
                                            int c2, int c3, int c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
        : "memory");
}

// im2col-mode load of a rank-4 map {C, W, H, N}: 128 consecutive pixels of
// the map's bounding box (raster order W, H, N) starting at base pixel
// (w, h, n), each shifted by (ow, oh), 64 channels from c; pixels outside the
// tensor read as zero.  Lands as 128 rows of 128 bytes, 128-byte swizzled.
__device__ __forceinline__ void tma_load_im2col(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c, int w,
                                                int h, int n, uint16_t ow, uint16_t oh) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.im2col.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], {%7, %8};" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c), "r"(w), "r"(h), "r"(n), "r"(bar), "h"(ow), "h"(oh)
        : "memory");
}

// Bulk copy (no tensor map) of `bytes` contiguous bytes from global memory to
// this CTA's shared memory, completing on the barrier at `bar`; both addresses
// 16-byte aligned, `bytes` a multiple of 16.
__device__ __forceinline__ void bulk_load_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Split TMEM load: issue 32 columns without waiting, and wait for every
// outstanding load of this warp.  The wait names the destination registers
// as read-write operands, so no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&v)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]),
                   "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]),
                   "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]),
                   "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]),
                   "+r"(v[29]), "+r"(v[30]), "+r"(v[31])
                 :
                 : "memory");
}

// Shared-memory matrix descriptor (tcgen05): start address, leading and
// stride byte offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;  // descriptor version for tcgen05
    d |= 2ull << 61;  // SWIZZLE_128B
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A K-major,
// B MN-major (c contiguous), M = 128, N = BN.
template <int BN, int BM = 128>
__device__ __forceinline__ constexpr uint32_t idesc_bf16() {
    return (1u << 4)                  // D format: f32
           | (1u << 7)                // A format: bf16
           | (1u << 10)               // B format: bf16
           | (0u << 15)               // A major: K
           | (1u << 16)               // B major: MN
           | ((uint32_t)(BN >> 3) << 17)
           | ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&v)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[32]), "=r"(v[33]), "=r"(v[34]), "=r"(v[35]), "=r"(v[36]), "=r"(v[37]), "=r"(v[38]), "=r"(v[39]),
          "=r"(v[40]), "=r"(v[41]), "=r"(v[42]), "=r"(v[43]), "=r"(v[44]), "=r"(v[45]), "=r"(v[46]), "=r"(v[47]),
          "=r"(v[48]), "=r"(v[49]), "=r"(v[50]), "=r"(v[51]), "=r"(v[52]), "=r"(v[53]), "=r"(v[54]), "=r"(v[55]),
          "=r"(v[56]), "=r"(v[57]), "=r"(v[58]), "=r"(v[59]), "=r"(v[60]), "=r"(v[61]), "=r"(v[62]), "=r"(v[63])
        : "r"(taddr + 32)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Drain one warp's 32 accumulator rows (TMEM lanes = tile rows, columns
// [taddr, taddr + BN)) to dx.  Each 64-column chunk is rounded to bf16 (RNE),
// written by each thread (its row) into the warp's 4 KB shared-memory slice
// with XOR-swizzled 16-byte chunks, then read back so that 8 lanes cover one
// row's 128 contiguous bytes: every store instruction writes four full
// 128-byte row segments instead of 32 scattered 16-byte pieces.  TMEM is read
// 32 columns at a time, the next load in flight while the current columns are
// converted and stored.  `off` is the dx element offset of this thread's row
// at the tile's first channel, `col0` that channel's index within the group;
// channels >= Cg are not written.  With `parts` set, the fp32 partial tiles of
// `nparts` stream-K workers (slots `pstride` float4 apart, layout [64 column
// chunks of 4][128 rows], this thread's row `prow`) are added before rounding.
__device__ __forceinline__ void add_partials32(uint32_t (&v)[32], const float4 *parts, int nparts, size_t pstride,
                                               int prow, int cc, int half) {
    for (int w = 0; w < nparts; ++w) {
        const float4 *pp = parts + (size_t)w * pstride + (size_t)(cc * 16 + half * 8) * 128 + prow;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 a = pp[(size_t)i * 128];
            v[4 * i] = __float_as_uint(__uint_as_float(v[4 * i]) + a.x);
            v[4 * i + 1] = __float_as_uint(__uint_as_float(v[4 * i + 1]) + a.y);
            v[4 * i + 2] = __float_as_uint(__uint_as_float(v[4 * i + 2]) + a.z);
            v[4 * i + 3] = __float_as_uint(__uint_as_float(v[4 * i + 3]) + a.w);
        }
    }
}

// 32 fp32 columns of this thread's row -> bf16 -> 16-byte chunks 4*half .. 4*half+3
// of the row's 128 staged bytes (chunk index XOR row % 8)
__device__ __forceinline__ void stage_half(const uint32_t (&v)[32], uint32_t sbase, int lane, int half) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            __nv_bfloat162 h2 =
                __floats2bfloat162_rn(__uint_as_float(v[8 * q + 2 * e]), __uint_as_float(v[8 * q + 2 * e + 1]));
            pk[e] = *reinterpret_cast<uint32_t *>(&h2);
        }
        const uint32_t a = sbase + (uint32_t)lane * 128u + ((uint32_t)((4 * half + q) ^ (lane & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(pk[0]), "r"(pk[1]), "r"(pk[2]),
                     "r"(pk[3])
                     : "memory");
    }
}

// (NC 64-column chunks from taddr; epilogue_rows<BN> drains BN columns)
__device__ __forceinline__ void epilogue_chunks(uint32_t taddr, int NC, uint8_t *stage, int lane, bool rvalid,
                                                int64_t off, int col0, int Cg, __nv_bfloat16 *dx,
                                                const float4 *parts = nullptr, int nparts = 0, size_t pstride = 0,
                                                int prow = 0) {
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
    const int ch = lane & 7;
    uint32_t va[32], vb[32];
    tmem_ld32_issue(taddr, va);
    tmem_wait_ld(va);
#pragma unroll 1
    for (int cc = 0; cc < NC; ++cc) {
        tmem_ld32_issue(taddr + cc * 64 + 32, vb);
        add_partials32(va, parts, nparts, pstride, prow, cc, 0);
        stage_half(va, sbase, lane, 0);
        tmem_wait_ld(vb);
        if (cc + 1 < NC) tmem_ld32_issue(taddr + (cc + 1) * 64, va);
        add_partials32(vb, parts, nparts, pstride, prow, cc, 1);
        stage_half(vb, sbase, lane, 1);
        __syncwarp();
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int row = it * 4 + (lane >> 3);
            const uint32_t a = sbase + (uint32_t)row * 128u + ((uint32_t)(ch ^ (row & 7)) << 4);
            uint4 val;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(val.x), "=r"(val.y), "=r"(val.z), "=r"(val.w)
                         : "r"(a)
                         : "memory");
            const int col = col0 + cc * 64 + ch * 8;
            if (rok[it] && col < Cg) *reinterpret_cast<uint4 *>(dx + roff[it] + cc * 64 + ch * 8) = val;
        }
        __syncwarp();
        if (cc + 1 < NC) tmem_wait_ld(va);
    }
}

template <int BN>
__device__ __forceinline__ void epilogue_rows(uint32_t taddr, uint8_t *stage, int lane, bool rvalid, int64_t off,
                                              int col0, int Cg, __nv_bfloat16 *dx, const float4 *parts = nullptr,
                                              int nparts = 0, size_t pstride = 0, int prow = 0) {
    epilogue_chunks(taddr, BN / 64, stage, lane, rvalid, off, col0, Cg, dx, parts, nparts, pstride, prow);
}

// Park one warp's 32 accumulator rows (NC 64-column chunks from taddr) as an
// fp32 partial tile (stream-K contributor, split-K scatter): column chunk c
// of 4 floats of row r at slot[c * 128 + r].
__device__ __forceinline__ void store_partial_chunks(uint32_t taddr, int NC, int prow, float4 *slot) {
#pragma unroll 1
    for (int cc = 0; cc < NC; ++cc) {
        uint32_t v[64];
        tmem_ld64(taddr + cc * 64, v);
#pragma unroll
        for (int i = 0; i < 16; ++i)
            slot[(size_t)(cc * 16 + i) * 128 + prow] =
                make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]), __uint_as_float(v[4 * i + 2]),
                            __uint_as_float(v[4 * i + 3]));
    }
}
template <int BN>
__device__ __forceinline__ void store_partial_rows(uint32_t taddr, int prow, float4 *slot) {
    store_partial_chunks(taddr, BN / 64, prow, slot);
}

__device__ __forceinline__ int ld_acquire_gpu(const int32_t *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(int32_t *p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---- clusters and SM pairs (tcgen05 cta_group::2) -------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ uint32_t ld_shared_cluster_u32(uint32_t cluster_addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
    return v;
}
__device__ __forceinline__ void tmem_alloc2(uint32_t slot, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}
__device__ __forceinline__ void tc_mma2(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive (once) on the barrier at this shared-memory offset in every CTA of
// `mask` when all prior tcgen05 operations of this thread have completed.
__device__ __forceinline__ void tc_commit2_mc(uint32_t bar, uint16_t mask) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
                 "h"(mask)
                 : "memory");
}
__device__ __forceinline__ void tma_load_5d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c0, int c1,
                                                 int c2, int c3, int c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
        : "memory");
}
__device__ __forceinline__ void tma_load_im2col_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c, int w,
                                                     int h, int n, uint16_t ow, uint16_t oh) {
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.im2col.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], {%7, %8};" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c), "r"(w), "r"(h), "r"(n), "r"(bar), "h"(ow), "h"(oh)
        : "memory");
}

// Pair-mode 2-D tile load (rows of a plain matrix): box at (c0 = column,
// c1 = row), bytes completing on the pair leader's barrier.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

// Zero the dx pixels that no residue class writes (bf16 NHWC, 16-byte
// stores), spread over the CTAs of the launch: CTA b takes dx rows b,
// b + gridDim.x, ...; a row no class writes is one contiguous run, a written
// row is zeroed only at its uncovered columns.  Run by a CTA's epilogue warps
// while the first tile's main loop is still in flight.
__device__ __forceinline__ void fill_uncovered(const TcParams &p, int tid, int nthreads) {
    const Geom &g = p.g;
    const uint32_t cpp = (uint32_t)g.C / 8;     // 16-byte chunks per pixel
    const uint32_t cpr = cpp * (uint32_t)g.Wi;  // per row
    uint4 *out = static_cast<uint4 *>(p.dx);
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    const uint32_t rows = (uint32_t)g.N * (uint32_t)g.Hi;
    const bool all_cols = p.cov_w == ~0ull;
    for (uint32_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const uint32_t hi = r % (uint32_t)g.Hi;
        uint4 *row = out + (size_t)r * cpr;
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

// Tiles of worker b of G in snake order: round k takes tile k*G + b for even k
// and k*G + G-1-b for odd k, so that the descending-cost (LPT) tile order of a
// launch spreads evenly over the workers (on the 5x5 stride-3 layer the
// busiest CTA's k-blocks drop from 34 to 32 against a mean of 29.9).
struct SnakeTiles {
    int b, G, total, k;
    __device__ __forceinline__ SnakeTiles(int b_, int G_, int total_) : b(b_), G(G_), total(total_), k(0) {}
    __device__ __forceinline__ bool next(int &t) {
        while ((int64_t)k * G < total) {
            t = k * G + ((k & 1) ? G - 1 - b : b);
            ++k;
            if (t < total) return true;
        }
        return false;
    }
};

// A stretch [kb0, kb1) of the k-blocks of tile t handled by one worker (CTA or
// SM pair).  `owner`: the stretch ends the tile, so this worker stores the
// tile, first adding the partial tiles of workers q_first .. self-1 (stream-K).
struct Segment {
    int t, kb0, kb1;
    bool owner;
    int q_first;
    int split;  // split-K: this worker's index among the tile's splits
};

__device__ __forceinline__ int class_of_tile(const TcParams &p, int t) {
    int ci = 0;
    for (int i = 1; i < p.num_classes; ++i)
        if (t >= p.cls[i].tile_begin) ci = i;
    return ci;
}

// Work of worker w of nw.  Static schedule: whole tiles w, w + nw, ...
// Stream-K: the units [w*U/nw, (w+1)*U/nw) of the (tile, k-block) sequence,
// visited from the last stretch to the first, so a worker's only partial
// stretch (the one that does not reach its tile's end) comes first and the
// stretch it owns after earlier workers' partials comes last.
struct SegmentIter {
    int w, nw, next_t, u, u_lo;
    SnakeTiles whole;  // whole-tile schedule
    __device__ __forceinline__ SegmentIter(const TcParams &p, int w_, int nw_)
        : w(w_), nw(nw_), next_t(w_), whole(w_, nw_, p.total_tiles) {
        u_lo = (int)((int64_t)w * p.units_total / nw);
        u = (int)((int64_t)(w + 1) * p.units_total / nw);
    }
    __device__ __forceinline__ int nkb(const TcParams &p, int ci) const {
        return p.cls[ci].taps_y * p.cls[ci].taps_x * p.kb_per_tap;
    }
    __device__ __forceinline__ bool next(const TcParams &p, Segment &sg) {
        if (p.splitk > 1) {
            // split-K: worker w takes split w % S of tile w / S (one unit per
            // worker, all units in one wave)
            if (next_t < 0 || w >= p.total_tiles * p.splitk) return false;
            const int S = p.splitk;
            sg.t = w / S;
            sg.split = w - sg.t * S;
            const int n = nkb(p, class_of_tile(p, sg.t));
            sg.kb0 = (int)((int64_t)sg.split * n / S);
            sg.kb1 = (int)((int64_t)(sg.split + 1) * n / S);
            sg.owner = true;
            sg.q_first = w;
            next_t = -1;
            return true;
        }
        sg.split = 0;
        if (!p.streamk) {
            if (!whole.next(sg.t)) return false;
            sg.kb0 = 0;
            sg.kb1 = nkb(p, class_of_tile(p, sg.t));
            sg.owner = true;
            sg.q_first = w;
            return true;
        }
        if (u <= u_lo) return false;
        const int last = u - 1;
        int ci = 0;
        for (int i = 1; i < p.num_classes; ++i)
            if (last >= p.cls[i].unit_begin) ci = i;
        const ClassDesc &c = p.cls[ci];
        const int n = nkb(p, ci);
        const int tl = (last - c.unit_begin) / n;
        const int ts = c.unit_begin + tl * n, te = ts + n;
        const int s0 = u_lo > ts ? u_lo : ts;
        sg.t = c.tile_begin + tl;
        sg.kb0 = s0 - ts;
        sg.kb1 = u - ts;
        sg.owner = u == te;
        int q = w;
        if (sg.owner && s0 > ts)
            while (q > 0 && (int)((int64_t)q * p.units_total / nw) > ts) --q;  // u_hi(q-1) > ts
        sg.q_first = q;
        u = s0;
        return true;
    }
};

struct TileCoord {
    int ci, mb, nb, gi;
};

__device__ __forceinline__ TileCoord decode_tile(const TcParams &p, int t) {
    int ci = 0;
    for (int i = 1; i < p.num_classes; ++i)
        if (t >= p.cls[i].tile_begin) ci = i;
    const ClassDesc &c = p.cls[ci];
    int local = t - c.tile_begin;
    TileCoord r;
    r.ci = ci;
    if (p.raster_m) {
        r.mb = local % c.m_tiles;
        int rest = local / c.m_tiles;
        r.nb = rest % p.n_tiles;
        r.gi = rest / p.n_tiles;
    } else {
        r.nb = local % p.n_tiles;
        int rest = local / p.n_tiles;
        r.mb = rest % c.m_tiles;
        r.gi = rest / c.m_tiles;
    }
    return r;
}

}  // namespace cbd
