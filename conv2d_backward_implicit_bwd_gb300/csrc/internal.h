// internal.h -- types shared by the host planner, the C ABI and the kernels.
//
// The decomposition (pages "Backward data" / "[igemm_dynamic] v4r1 bwd
// dynamic kernel", the v4r1 backward-data gridwise-GEMM strategy): per
// spatial dim with stride s, dilation d, pad p and filter length F,
//   g = gcd(s, d), T = s / g (YTilde / XTilde), D = d / g;
//   class t in [0, T) owns taps y = t + T*j, j < ceil((F - t) / T);
//   it writes dx rows hi = ht*s + t*d - p for ht in [ht_lo, ht_lo + HT) (all
//   such rows inside [0, Hi)), and tap j of row ht reads dy row ho = ht - j*D
//   (zero when ho is outside [0, Ho)).
// One sub-GEMM per pair of non-empty row/column classes:
//   M = N * HT * WT rows (n, ht, wt), N_gemm = C/G, K_gemm = K/G * taps.
#pragma once
#include <stdint.h>
#include <cuda.h>           // CUtensorMap (header-only use)
#include <cuda_runtime.h>

namespace cbd {

constexpr int kMaxClasses = 64;   // non-empty sub-GEMMs per plan
constexpr int kMaxTcClasses = 16; // sub-GEMMs per tensor-core launch (more classes -> several launches)

struct ClassDesc {
    int32_t ty, tx;          // row / column residue class
    int32_t taps_y, taps_x;  // taps of each class (>= 1 for a non-empty sub-GEMM)
    int32_t ht_lo, HT;       // first class row index and count
    int32_t wt_lo, WT;       // first class column index and count
    int32_t M;               // N * HT * WT
    int32_t m_tiles;         // ceil(M / BM) for the kernel that runs this class
    int32_t tile_begin;      // first tile of this class in the launch's schedule
    int32_t gemm_id;         // consecutive id of the sub-GEMM
    int32_t unit_begin;      // first (tile, k-block) unit of this class in the launch (stream-K)
    int32_t pty, ptx;        // 1-SM kernel, 256-wide tiles of C/G <= 128: residues of a second class with the
                             // same rows and tap counts, computed in the tile's upper 128 columns (else -1)
};

struct Geom {
    int32_t N, C, K, Hi, Wi, Ho, Wo, Y, X;
    int32_t ph, pw, sh, sw, dh, dw, G, Cg, Kg;
    int32_t YT, XT, DH, DW;
};

// Element strides of the logical index orders dy[n][k][ho][wo],
// w[k][c][y][x] (c within the group) and dx[n][c][hi][wi] for either layout.
struct Strides {
    int64_t dy_n, dy_k, dy_h, dy_w;
    int64_t w_k, w_c, w_y, w_x;
    int64_t dx_n, dx_c, dx_h, dx_w;
};

struct SimtParams {
    Geom g;
    Strides st;
    const void *dy;
    const void *w;
    void *dx;
    int32_t num_classes;
    int32_t bn;           // tile width: 64, or 32 (fp32 kernel, C/G <= 32)
    int32_t n_tiles;      // ceil(Cg / bn)
    int32_t total_tiles;  // sum over classes of G * m_tiles * n_tiles
    ClassDesc cls[kMaxClasses];
};

struct FillParams {
    void *dx;
    int32_t esize;        // bytes per element
    int32_t layout;       // 0 NCHW, 1 NHWC
    int32_t vec16;        // 1: NHWC, C*esize % 16 == 0 and dx 16-byte aligned -> 16-byte stores
    int32_t N, C, Hi, Wi;
    int32_t sh, sw;
    uint64_t cov_h, cov_w; // bit r set: rows/cols with index % s == r are written by a sub-GEMM
};

// Tensor-core (tcgen05) kernel parameters.
struct TcParams {  // 128-byte aligned through CUtensorMap
    CUtensorMap tmap_w;   // w viewed as 5-D {Cg, X, Y, Kg, G}, box {64, 1, 1, 64, 1}, 128B swizzle
    CUtensorMap tmap_w_half;  // fp32 tensor-core path only: the low part of the split filter (same view as tmap_w)
    CUtensorMap tmap_a[kMaxTcClasses];  // per class: dy as im2col {K, Wo, Ho, N}, 64 ch x 128 px, 128B swizzle
    const void *dy;
    void *dx;
    int32_t *status;      // device status word (0 = ok)
    int64_t wait_budget;  // SM clock cycles a blocking wait may spin before giving up
    Geom g;
    int32_t num_classes;
    int32_t n_tiles;      // ceil(Cg / BN)
    int32_t kb_per_tap;   // ceil(Kg / 64)
    int32_t total_tiles;
    int32_t im2col;       // 1: A rows by TMA im2col loads (tmap_a), 0: cp.async gather
    int32_t a_plain;      // 1 (SM-pair kernel): every class reads dy as a plain matrix {K, N*Ho*Wo} (tmap_a 2-D)
    int32_t fill;         // 1: the epilogue warps also zero the dx pixels no class writes
    int32_t raster_m;     // 1: consecutive tiles walk m-blocks first (else n-blocks first)
    int32_t streamk;      // 1: workers take equal ranges of (tile, k-block) units (2-SM kernel)
    int32_t splitk;       // S > 1 (2-SM kernel): S SM pairs per tile, each a 1/S range of its k-blocks; the
                          // pairs exchange fp32 partials (workspace `partials`) and each stores 1/S of the columns
    int32_t units_total;  // sum over tiles of their k-blocks
    int32_t epoch;        // tag of this launch's partial-tile flags (never 0)
    float4 *partials;     // stream-K: per worker and CTA rank, one 128 x 256 fp32 partial tile
    int32_t *flags;       // stream-K: per worker and CTA rank, == epoch once its partial is written
    uint64_t cov_h, cov_w;  // residues of rows / columns some class writes (as in FillParams)
    const void *w;        // narrow-group kernel: the filter (KYXC), read to build its block-diagonal B
    int32_t bd_cg;        // narrow-group kernel: channels per real group (g holds the folded 64-channel blocks)
    int32_t interleave;   // narrow-group kernel: classes of equal m-blocks interleaved tile by tile
#ifdef CBD_PHASE_TIMES
    unsigned long long *phase_log;  // instrumented build: per CTA, kPhaseSlots globaltimer stamps (ns)
#endif
    ClassDesc cls[kMaxTcClasses];
};

#ifdef CBD_PHASE_TIMES
// Instrumented build only (compiled with -DCBD_PHASE_TIMES): timeline slots of
// the tensor-core kernels, one globaltimer stamp each per CTA.
constexpr int kPhaseSlots = 24;
constexpr int kPhaseLogCtas = 1024;  // CTAs a timeline buffer holds (grids are at most one CTA per SM)
enum : int {
    kPhEntry = 0,       // kernel entry (thread 0)
    kPhSetup = 1,       // barriers initialised, TMEM allocated, CTAs synchronised
    kPhFillDone = 2,    // epilogue warps finished zeroing uncovered pixels
    kPhFirstIssue = 3,  // A producer issued its first load
    kPhFirstFull = 4,   // MMA thread saw the first stage land
    kPhMma0Done = 5,    // MMA thread committed the first tile
    kPhEpi0Start = 6,   // epilogue saw the first accumulator
    kPhEpi0Done = 7,    // epilogue stored the first tile (warp 0)
    kPhMma1Start = 8,   // MMA thread started the second tile
    kPhEpi1Start = 9,
    kPhEpi1Done = 10,
    kPhMmaLast = 11,    // MMA thread committed its last tile
    kPhEpiLast = 12,    // epilogue stored its last tile
    kPhExit = 13,       // after the final CTA barrier (thread 0)
    kPhLastIssue = 14,  // A producer issued its last load
    kPhProdStart = 15,  // A producer about to decode its first tile
    kPhProdWaited = 16, // A producer passed its first empty-slot wait
    kPhBFirst = 17,     // first B producer issued its first load
    kPhProdSeg = 18,    // A producer: first segment of its schedule known
    kPhProdTile = 19,   // A producer: first tile decoded
    kPhProdPreWait = 20,// A producer: about to wait for its first free stage
};
#endif

// Forward-convolution kernel parameters (x has dx's shape, y has dy's shape).
struct FwdParams {
    CUtensorMap tmap_x;   // x as im2col {C, Wi, Hi, N}, traversal strides (sw, sh), 64 ch x 128 px, 128B swizzle
    CUtensorMap tmap_w;   // w as {Cg, X, Y, Kg, G}, box {64, 1, 1, BN, 1}: B rows of 64 c (K-major)
    void *y;
    int32_t *status;
    int64_t wait_budget;
    Geom g;
    int32_t m_tiles;      // ceil(N*Ho*Wo / 128)
    int32_t n_tiles;      // ceil(Kg / BN)
    int32_t total_tiles;  // m_tiles * n_tiles * G
    int32_t kb_per_tap;   // ceil(Cg / 64)
};

// Narrow-group kernel parameters (C/G = K/G in {8, 16}, G % 8 == 0).
struct GroupedParams {
    const void *dy;
    const void *w;
    void *dx;
    Geom g;
    int32_t gblocks;         // G / 8
    int32_t row_class[64];   // per row residue hi % sh: (taps_y << 16) | ty (taps 0: no class writes it)
    int32_t col_class[64];   // per column residue wi % sw: (taps_x << 16) | tx
    int32_t col_q[64];       // per column residue r: staged pixel of output t = 0, tap i = 0
    int32_t wch;             // dx pixels per item (a multiple of sw)
    int32_t span;            // staged dy pixels per tap row (covers every tap of an item)
    int32_t wfrag_bytes;     // shared memory of the w fragments
    int32_t buf_bytes;       // shared memory of one staged-dy buffer
    int32_t nwch;            // items per dx row
    int32_t per_r;           // 16-pixel m-tiles per column residue and item
    int32_t wo_c;            // first staged dy column of an item = w0 / sw + wo_c
    int32_t step_wc, step_hi, step_n;  // the item stride (CTAs per group block) as (chunk, row, image)
};

struct GroupedLayout {
    int32_t wch, span, wfrag_bytes, buf_bytes, smem;
};
GroupedLayout grouped_layout(const Geom &g);

// Status codes written by kernels (first writer wins).
enum : int32_t {
    kDevOk = 0,
    kDevTimeoutProducer = 0x101,
    kDevTimeoutMma = 0x102,
    kDevTimeoutEpilogue = 0x103,
    kDevTimeoutSelftest = 0x1FF,
    kDevTimeoutPartial = 0x104,
    kDevFaultIndex = 0x201,
};

cudaError_t launch_fill(const FillParams &p, int num_sms, cudaStream_t s);
cudaError_t launch_simt(const SimtParams &p, int dtype, cudaStream_t s);
cudaError_t launch_grouped(GroupedParams &p, int num_sms, cudaStream_t s);
cudaError_t launch_tc(const TcParams &p, int bn, int grid, cudaStream_t s);
cudaError_t launch_tc2(const TcParams &p, int bn, int grid, cudaStream_t s);  // grid: 2 CTAs per SM pair
cudaError_t launch_fwd(const FwdParams &p, int bn, int grid, cudaStream_t s);
// narrow groups on tcgen05: 64-channel group blocks, block-diagonal B resident per CTA
cudaError_t launch_tc_grouped(const TcParams &p, int grid, cudaStream_t s);
size_t tc_grouped_smem_bytes(int taps);
// out[b][c][r] = in[b][r][c] for bf16 elements (layout changes of NCHW/GKCYX problems)
cudaError_t launch_transpose_b16(const void *in, void *out, int64_t batch, int64_t R, int64_t Cc, int num_sms,
                                 cudaStream_t s);
int tc2_max_pairs(int num_sms);
cudaError_t launch_selftest_wait(int32_t *status, int64_t budget, cudaStream_t s);
size_t tc_smem_bytes(int bn, bool im2col);

}  // namespace cbd
