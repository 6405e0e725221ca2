// capi.cpp -- host planner and C ABI (include/conv_bwd_data.h).
//
// Planner: the v4r1 backward-data multi-kernel decomposition (pages
// "Backward data", rocMLIR pull request 246, and "[igemm_dynamic] v4r1 bwd
// dynamic kernel", MIOpen pull request 272).  Problem -> plan -> run mirrors
// the library workflow described in "Re: MIOpen package LFS files" (Problem,
// Find solution, Load kernel, Run on GPU), with a single solution per
// problem and ahead-of-time compiled kernels: one compiled kernel serves every
// shape, which receives the shape at run time (the "dynamic kernel" idea of
// MIOpen pull request 272).
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <numeric>
#include <string>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "../../include/conv_bwd_data.h"
#include "internal.h"
#include "band.h"
#include "tf32.h"

using namespace cbd;

struct conv_bwd_plan_s {
    conv_bwd_desc desc;
    Geom g;
    Strides st;
    int32_t path = CONV_BWD_PATH_SIMT;
    int32_t bn = 64;                      // tensor-core tile width (N_gemm)
    std::vector<ClassDesc> classes;       // gemm_id order
    std::vector<int> sched;               // launch order (indices into classes)
    std::vector<uint8_t> row_cov, col_cov;
    uint64_t cov_h = 0, cov_w = 0;
    bool any_uncovered = false;
    double useful_flop = 0, algo_bytes = 0;
    // device side
    bool has_device = false;
    int device = -1;
    int num_sms = 0;
    int32_t *d_status = nullptr;
    bool owns_status = true;              // false: the status word is borrowed (no-allocation entry point)
    int64_t wait_budget = 0;
    bool timing = false;
    bool fill_ran = false;
    cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};
    // TMA descriptor cache (keyed by the filter pointer)
    const void *tmap_w_ptr = nullptr;
    CUtensorMap tmap_w, tmap_w_half;
    const void *tmap_a_ptr = nullptr;     // dy pointer the per-class im2col maps were encoded for
    const void *tmap_dx_ptr = nullptr;    // dx pointer the banded kernel's store maps were encoded for
    std::vector<CUtensorMap> tmap_a;      // per class (gemm_id order)
    bool im2col = false;                  // A rows by TMA im2col loads (else cp.async gather)
    bool two_sm = false;                  // 256x256 tiles on SM pairs (cta_group::2)
    bool a_plain = false;                 // SM-pair kernel specialised for dy read as a plain matrix
    bool grouped_tc = false;              // narrow groups on tcgen05 (block-diagonal B), else warp-level MMA
    bool fuse = false;                    // 1-SM tiles of 256 columns computing two classes (C/G <= 128) at once
    bool grouped_band = false;            // narrow groups on tcgen05 with dy staged once per band (band params)
    BandParams band;                      // its geometry (pointers and the dy map filled by run)
    int max_pairs = 0;                    // co-resident SM pairs of the 2-SM kernel
    float4 *d_partials = nullptr;         // stream-K workspace: per pair and CTA, one 128x256 fp32 tile
    int32_t *d_flags = nullptr;           // stream-K flags, tagged with the launch epoch
    int32_t splitk = 1;                   // SM pairs per tile (split-K reduce-scatter), 1 = whole tiles
    float4 *d_ws = nullptr;               // split-K workspace: fp32 partials of the other splits' column slices
    int32_t *d_ws_flags = nullptr;        // split-K flags, one per (tile, split, CTA rank), tagged with the epoch
    int32_t epoch = 0;
    // forward convolution with the same geometry (the adjoint of run): maps
    // keyed by the x and w pointers
    const void *fwd_x_ptr = nullptr, *fwd_w_ptr = nullptr;
    CUtensorMap fwd_tmap_x, fwd_tmap_w;
    // pipelined run_host: batch chunks run on plans of their own (sharing this
    // plan's status word) so that the copies of one chunk overlap the compute
    // of another; [0] has chunk_n images, [1] the last chunk's count if smaller
    conv_bwd_plan_s *chunk_plan[2] = {nullptr, nullptr};
    int32_t chunk_n = 0, chunks = 0;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    std::vector<cudaEvent_t> hev;  // start, done, then per chunk: inputs copied, output computed
    // bf16 NCHW/GKCYX problems on the tensor-core (or narrow-group) path: layout
    // transposes into plan-owned NHWC/KYXC scratch around a plan of the same
    // geometry in NHWC/KYXC (sharing this plan's status word)
    conv_bwd_plan_s *nhwc_plan = nullptr;
    void *t_dy = nullptr, *t_w = nullptr, *t_dx = nullptr;
    // fp32 tensor-core path: the filter split into hi and lo parts, laid out
    // [G][C/G][Y][X][K/G] (re-split by every run, w being an input).  Owned by
    // the plan that allocated them; an NCHW parent lends its own to its NHWC
    // twin, a pipelined run_host to its chunk plans.
    float *w_hi = nullptr, *w_lo = nullptr;
    bool owns_wsplit = false;
#ifdef CBD_PHASE_TIMES
    unsigned long long *d_phase = nullptr;  // instrumented build: per-CTA timeline of the tensor-core kernel
#endif
    int32_t w_gkcyx = 0;  // 1: run() receives the filter as GKCYX (the NCHW parent's w)
    int32_t tf32_split = -1;  // tail split of the fp32 tensor-core schedule: -1 by cost, 0 never, 1 always
    std::mutex mu;
};

namespace {

int64_t floor_div(int64_t a, int64_t b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }
int64_t ceil_div_s(int64_t a, int64_t b) { return -floor_div(-a, b); }

struct DimClass {
    int t, taps, lo, cnt;
};

// Residue classes of one spatial dim.  Returns T (tilde factor) and D (dy
// step per tap index); fills the per-class taps and row ranges, the coverage
// residue mask (bit r: indices i with i % s == r are written), the per-index
// coverage, and the count of (o, f) pairs whose tap lands inside [0, In).
void plan_dim(int64_t In, int64_t Out, int64_t F, int64_t s, int64_t d, int64_t p, int &T, int &D,
              std::vector<DimClass> &cls, uint64_t &mask, std::vector<uint8_t> &cov, int64_t &useful) {
    int64_t g = std::gcd(s, d);
    T = (int)(s / g);
    D = (int)(d / g);
    cls.clear();
    mask = 0;
    cov.assign((size_t)In, 0);
    for (int t = 0; t < T; ++t) {
        int taps = t < F ? (int)((F - t + T - 1) / T) : 0;
        int64_t lo = ceil_div_s(p - (int64_t)t * d, s);
        int64_t hi = floor_div(In - 1 + p - (int64_t)t * d, s);
        int64_t cnt = std::max<int64_t>(0, hi - lo + 1);
        cls.push_back({t, taps, (int)lo, (int)cnt});
        if (taps > 0 && cnt > 0) {
            int64_t r = ((int64_t)t * d - p) % s;
            if (r < 0) r += s;
            mask |= 1ull << r;
            for (int64_t q = lo; q < lo + cnt; ++q) cov[(size_t)(q * s + (int64_t)t * d - p)] = 1;
        }
    }
    useful = 0;
    for (int64_t o = 0; o < Out; ++o)
        for (int64_t f = 0; f < F; ++f) {
            int64_t i = o * s - p + f * d;
            if (i >= 0 && i < In) ++useful;
        }
}

bool ranges_overlap(const void *a, size_t na, const void *b, size_t nb) {
    uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + nb && y < x + na;
}

size_t elem_size(int32_t dt) { return dt == CONV_BWD_BF16 ? 2 : 4; }

const char *env(const char *k);

// NVTX range (domain "conv_bwd_data") around each entry point that enqueues
// work, so that a profiler timeline shows which kernels and copies belong to
// which call.  Header-only NVTX: without an attached tool the calls return
// at once.
nvtxDomainHandle_t nvtx_domain() {
    static nvtxDomainHandle_t d = nvtxDomainCreateA("conv_bwd_data");
    return d;
}
struct NvtxRange {
    explicit NvtxRange(const char *name) {
        nvtxEventAttributes_t a = {};
        a.version = NVTX_VERSION;
        a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
        a.messageType = NVTX_MESSAGE_TYPE_ASCII;
        a.message.ascii = name;
        nvtxDomainRangePushEx(nvtx_domain(), &a);
    }
    ~NvtxRange() { nvtxDomainRangePop(nvtx_domain()); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

// L2 sector promotion of the TMA maps (256 B by default).
CUtensorMapL2promotion l2_promotion() {
    if (const char *f = env("CONVBWD_DEBUG_L2PROMO")) {
        if (f[0] == '0') return CU_TENSOR_MAP_L2_PROMOTION_NONE;
        if (f[0] == '1') return CU_TENSOR_MAP_L2_PROMOTION_L2_128B;
    }
    return CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
}

typedef CUresult (*PFN_encodeTiled)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                     const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                     CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                     CUtensorMapFloatOOBfill);

PFN_encodeTiled get_encode_tiled() {
    static PFN_encodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_encodeTiled)p;
    });
    return fn;
}

// w (KYXC, bf16) as a 5-D tensor {Cg, X, Y, Kg, G}: a box {64, 1, 1, 64, 1}
// is a 64(k) x 64(c) slice of one filter tap, c contiguous (128 bytes per k
// row, 128-byte swizzle).  Coordinates past Cg or past Kg (the next group's
// rows) read as zero.
bool encode_w_map(conv_bwd_plan_s *p, const void *w) {
    PFN_encodeTiled enc = get_encode_tiled();
    if (!enc) return false;
    const Geom &g = p->g;
    cuuint64_t dims[5] = {(cuuint64_t)g.Cg, (cuuint64_t)g.X, (cuuint64_t)g.Y, (cuuint64_t)g.Kg, (cuuint64_t)g.G};
    cuuint64_t strides[4] = {(cuuint64_t)g.Cg * 2, (cuuint64_t)g.X * g.Cg * 2, (cuuint64_t)g.Y * g.X * g.Cg * 2,
                             (cuuint64_t)g.Kg * g.Y * g.X * g.Cg * 2};
    cuuint32_t box[5] = {64, 1, 1, 64, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(&p->tmap_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(w), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     l2_promotion(), CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

typedef CUresult (*PFN_encodeIm2col)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                      const cuuint64_t *, const int *, const int *, cuuint32_t, cuuint32_t,
                                      const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                      CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

PFN_encodeIm2col get_encode_im2col() {
    static PFN_encodeIm2col fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_encodeIm2col)p;
    });
    return fn;
}

// Bounding-box corners of class c's im2col map over dy {K, Wo, Ho, N}: the
// base pixel of tap (taps-1) walks ht - (taps_y-1)*DH over the class rows, so
// the box spans [lo, dim - 1 + hi] with lo/hi below (index 0 = W, 1 = H).
void im2col_corners(const Geom &g, const ClassDesc &c, int lo[2], int hi[2]) {
    lo[0] = c.wt_lo - (c.taps_x - 1) * g.DW;
    lo[1] = c.ht_lo - (c.taps_y - 1) * g.DH;
    hi[0] = lo[0] + c.WT - g.Wo;
    hi[1] = lo[1] + c.HT - g.Ho;
}

// One im2col map per class: 64 channels x 128 pixels per load, 128-byte
// swizzle, pixels outside dy read as zero.  Plans specialised for a plain A
// matrix get a 2-D tiled map of dy as {K, N*Ho*Wo} instead (box 64 x 128,
// rows past the last pixel read as zero), one copy per class.
bool encode_a_maps(conv_bwd_plan_s *p, const void *dy) {
    const Geom &g = p->g;
    if (p->a_plain) {
        PFN_encodeTiled enc = get_encode_tiled();
        if (!enc) return false;
        p->tmap_a.resize(p->classes.size());
        cuuint64_t dims[2] = {(cuuint64_t)g.K, (cuuint64_t)g.N * g.Ho * g.Wo};
        cuuint64_t strides[1] = {(cuuint64_t)g.K * 2};
        cuuint32_t box[2] = {64, 128};
        cuuint32_t estr[2] = {1, 1};
        for (size_t i = 0; i < p->classes.size(); ++i)
            if (enc(&p->tmap_a[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(dy), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, l2_promotion(),
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return false;
        return true;
    }
    PFN_encodeIm2col enc = get_encode_im2col();
    if (!enc) return false;
    // 128-byte pixel rows: 64 bf16 channels, or 32 fp32 ones (fp32 tensor-core path)
    const bool f32 = p->desc.dtype == CONV_BWD_F32;
    const cuuint64_t es = f32 ? 4 : 2;
    p->tmap_a.resize(p->classes.size());
    cuuint64_t dims[4] = {(cuuint64_t)g.K, (cuuint64_t)g.Wo, (cuuint64_t)g.Ho, (cuuint64_t)g.N};
    cuuint64_t strides[3] = {(cuuint64_t)g.K * es, (cuuint64_t)g.Wo * g.K * es, (cuuint64_t)g.Ho * g.Wo * g.K * es};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    for (size_t i = 0; i < p->classes.size(); ++i) {
        int lo[2], hi[2];
        im2col_corners(g, p->classes[i], lo, hi);
        CUresult r = enc(&p->tmap_a[i], f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                         const_cast<void *>(dy), dims, strides, lo, hi, f32 ? 32 : 64, 128, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, l2_promotion(),
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return false;
    }
    return true;
}

// Banded narrow-group kernel: dy as {K, Wo, Ho, N}, box {64 channels, 32
// pixels, rows, 1 image}, 128-byte swizzle; coordinates outside dy (negative
// ones included) read as zero.
// Banded kernel's dx stores: the pixels (sh*i + a, sw*j + b) of class (a, b)
// as {C, wc[b], hc[a], N}, one box = 64 channels of segw consecutive j of one
// output row; rows and columns past the class's last are clipped by the map.
bool encode_band_dx_maps(conv_bwd_plan_s *p, void *dx) {
    PFN_encodeTiled enc = get_encode_tiled();
    if (!enc) return false;
    const Geom &g = p->g;
    BandParams &b = p->band;
    b.dx_maps = 0;
    for (int a = 0; a < b.sh; ++a)
        for (int c = 0; c < b.sw; ++c) {
            if (b.hc[a] <= 0 || b.wc[c] <= 0) continue;
            const int ci = a * b.sw + c;
            uint16_t *base = static_cast<uint16_t *>(dx) + ((int64_t)a * g.Wi + c) * g.C;  // bf16 elements
            cuuint64_t dims[4] = {(cuuint64_t)g.C, (cuuint64_t)b.wc[c], (cuuint64_t)b.hc[a], (cuuint64_t)g.N};
            cuuint64_t strides[3] = {(cuuint64_t)b.sw * g.C * 2, (cuuint64_t)b.sh * g.Wi * g.C * 2,
                                     (cuuint64_t)g.Hi * g.Wi * g.C * 2};
            cuuint32_t box[4] = {64, (cuuint32_t)b.segw, 1, 1};
            cuuint32_t estr[4] = {1, 1, 1, 1};
            if (enc(&b.tmap_dx[ci], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return false;
            b.dx_maps |= 1 << ci;
        }
    return true;
}

bool encode_band_map(conv_bwd_plan_s *p, const void *dy) {
    PFN_encodeTiled enc = get_encode_tiled();
    if (!enc) return false;
    const Geom &g = p->g;
    cuuint64_t dims[4] = {(cuuint64_t)g.K, (cuuint64_t)g.Wo, (cuuint64_t)g.Ho, (cuuint64_t)g.N};
    cuuint64_t strides[3] = {(cuuint64_t)g.K * 2, (cuuint64_t)g.Wo * g.K * 2, (cuuint64_t)g.Ho * g.Wo * g.K * 2};
    cuuint32_t box[4] = {64, 32, (cuuint32_t)p->band.rows, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(&p->band.tmap_dy, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(dy), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, l2_promotion(),
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 tensor-core path: the split filter (w_hi, w_lo, [G][Cg][Y][X][Kg]) as
// 5-D {Kg, X, Y, Cg, G}; a box {32, 1, 1, 128, 1} is 128 c rows of 32 k
// (128 bytes, 128-byte swizzle: B K-major).  k past Kg and c past Cg read as
// zero.
bool encode_tf32_w_maps(conv_bwd_plan_s *p) {
    PFN_encodeTiled enc = get_encode_tiled();
    if (!enc) return false;
    const Geom &g = p->g;
    cuuint64_t dims[5] = {(cuuint64_t)g.Kg, (cuuint64_t)g.X, (cuuint64_t)g.Y, (cuuint64_t)g.Cg, (cuuint64_t)g.G};
    cuuint64_t strides[4] = {(cuuint64_t)g.Kg * 4, (cuuint64_t)g.X * g.Kg * 4, (cuuint64_t)g.Y * g.X * g.Kg * 4,
                             (cuuint64_t)g.Cg * g.Y * g.X * g.Kg * 4};
    cuuint32_t box[5] = {(cuuint32_t)kTf32BK, 1, 1, (cuuint32_t)kTf32BN, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    float *parts[2] = {p->w_hi, p->w_lo};
    CUtensorMap *maps[2] = {&p->tmap_w, &p->tmap_w_half};
    for (int i = 0; i < 2; ++i)
        if (enc(maps[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, parts[i], dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, l2_promotion(),
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    return true;
}

// Forward convolution: the im2col walk over x visits the Wo x Ho base pixels
// (wo*sw - pw, ho*sh - ph) with traversal strides (sw, sh), so the bounding box
// runs from (-pw, -ph) to the last base pixel.
void fwd_corners(const Geom &g, int lo[2], int hi[2]) {
    lo[0] = -g.pw;
    lo[1] = -g.ph;
    hi[0] = -g.pw + (g.Wo - 1) * g.sw - (g.Wi - 1);
    hi[1] = -g.ph + (g.Ho - 1) * g.sh - (g.Hi - 1);
}

bool fwd_supported(const conv_bwd_plan_s *p) {
    const conv_bwd_desc &d = p->desc;
    const Geom &g = p->g;
    if (d.dtype != CONV_BWD_BF16 || d.layout != CONV_BWD_NHWC_KYXC) return false;
    if (g.Cg % 8 || g.Kg % 8 || (g.G > 1 && g.Cg % 64)) return false;
    if (g.sh > 8 || g.sw > 8 || (g.X - 1) * g.dw > 127 || (g.Y - 1) * g.dh > 127) return false;
    if ((int64_t)d.N * g.Ho * g.Wo >= (1LL << 31) - 128) return false;
    int lo[2], hi[2];
    fwd_corners(g, lo, hi);
    for (int q = 0; q < 2; ++q)
        if (lo[q] < -128 || lo[q] > 127 || hi[q] < -128 || hi[q] > 127) return false;
    return true;
}

int fwd_bn(const Geom &g) { return g.Kg >= 256 ? 256 : 128; }

bool encode_fwd_maps(conv_bwd_plan_s *p, const void *x, const void *w) {
    PFN_encodeIm2col enc_i = get_encode_im2col();
    PFN_encodeTiled enc_t = get_encode_tiled();
    if (!enc_i || !enc_t) return false;
    const Geom &g = p->g;
    cuuint64_t xdims[4] = {(cuuint64_t)g.C, (cuuint64_t)g.Wi, (cuuint64_t)g.Hi, (cuuint64_t)g.N};
    cuuint64_t xstr[3] = {(cuuint64_t)g.C * 2, (cuuint64_t)g.Wi * g.C * 2, (cuuint64_t)g.Hi * g.Wi * g.C * 2};
    cuuint32_t trav[4] = {1, (cuuint32_t)g.sw, (cuuint32_t)g.sh, 1};
    int lo[2], hi[2];
    fwd_corners(g, lo, hi);
    if (enc_i(&p->fwd_tmap_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(x), xdims, xstr, lo, hi, 64, 128,
              trav, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, l2_promotion(),
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    cuuint64_t wdims[5] = {(cuuint64_t)g.Cg, (cuuint64_t)g.X, (cuuint64_t)g.Y, (cuuint64_t)g.Kg, (cuuint64_t)g.G};
    cuuint64_t wstr[4] = {(cuuint64_t)g.Cg * 2, (cuuint64_t)g.X * g.Cg * 2, (cuuint64_t)g.Y * g.X * g.Cg * 2,
                          (cuuint64_t)g.Kg * g.Y * g.X * g.Cg * 2};
    cuuint32_t box[5] = {64, 1, 1, (cuuint32_t)fwd_bn(g), 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return enc_t(&p->fwd_tmap_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(w), wdims, wstr, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, l2_promotion(),
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

const char *env(const char *k) {
    const char *v = std::getenv(k);
    return (v && *v) ? v : nullptr;
}

conv_bwd_status validate(const conv_bwd_desc *d) {
    if (!d) return CONV_BWD_ERR_INVALID_ARG;
    if (d->N < 1 || d->C < 1 || d->K < 1 || d->Hi < 1 || d->Wi < 1 || d->Y < 1 || d->X < 1)
        return CONV_BWD_ERR_INVALID_ARG;
    if (d->pad_h < 0 || d->pad_w < 0 || d->stride_h < 1 || d->stride_w < 1 || d->dil_h < 1 || d->dil_w < 1 ||
        d->groups < 1)
        return CONV_BWD_ERR_INVALID_ARG;
    if (d->C % d->groups || d->K % d->groups) return CONV_BWD_ERR_INVALID_ARG;
    if (d->layout != CONV_BWD_NCHW_GKCYX && d->layout != CONV_BWD_NHWC_KYXC) return CONV_BWD_ERR_INVALID_ARG;
    if (d->dtype != CONV_BWD_F32 && d->dtype != CONV_BWD_BF16) return CONV_BWD_ERR_INVALID_ARG;
    int64_t eh = d->Hi + 2LL * d->pad_h - (int64_t)d->dil_h * (d->Y - 1) - 1;
    int64_t ew = d->Wi + 2LL * d->pad_w - (int64_t)d->dil_w * (d->X - 1) - 1;
    if (eh < 0 || ew < 0) return CONV_BWD_ERR_INVALID_ARG;
    if (d->stride_h > 64 || d->stride_w > 64) return CONV_BWD_ERR_UNSUPPORTED;
    return CONV_BWD_OK;
}

// Two classes can share a 1-SM tile: same rows and tap counts.
bool fusable_classes(const ClassDesc &a, const ClassDesc &b) {
    return a.taps_y == b.taps_y && a.taps_x == b.taps_x && a.ht_lo == b.ht_lo && a.HT == b.HT && a.wt_lo == b.wt_lo &&
           a.WT == b.WT;
}

// The classes of the tensor-core launches, in schedule order: with class
// pairing on, each class takes the first later class it can share tiles with
// (its residues become the entry's pty, ptx).  `map` gets each entry's class
// index (its im2col map).
void launch_classes(const conv_bwd_plan_s *p, std::vector<ClassDesc> &out, std::vector<int> &map) {
    out.clear();
    map.clear();
    std::vector<char> used(p->classes.size(), 0);
    for (size_t a = 0; a < p->sched.size(); ++a) {
        const int idx = p->sched[a];
        if (used[(size_t)idx]) continue;
        used[(size_t)idx] = 1;
        ClassDesc c = p->classes[(size_t)idx];
        if (p->fuse)
            for (size_t b = a + 1; b < p->sched.size(); ++b) {
                const int j = p->sched[b];
                if (used[(size_t)j] || !fusable_classes(c, p->classes[(size_t)j])) continue;
                c.pty = p->classes[(size_t)j].ty;
                c.ptx = p->classes[(size_t)j].tx;
                used[(size_t)j] = 1;
                break;
            }
        out.push_back(c);
        map.push_back(idx);
    }
}

// Banded narrow-group kernel: output classes (a, b) = (hi % sh, wi % sw) with
// strides <= 2; tap (y, x) reaches class (a, b) iff a + ph - y*dh and
// b + pw - x*dw are multiples of the strides, and reads dy at row offset
// oy = (a + ph - y*dh) / sh and column offset ox = (b + pw - x*dw) / sw from
// the class's output index (i, j).  Fills the geometry of `bp` and returns
// whether the kernel applies (shared memory for at least two A stages, at
// least 16 output columns per 32-pixel staged row).
bool plan_band(const conv_bwd_desc &d, const Geom &g, BandParams &bp) {
    if (d.dtype != CONV_BWD_BF16 || d.layout != CONV_BWD_NHWC_KYXC || g.Cg != g.Kg) return false;
    if (!(g.Cg == 8 || g.Cg == 16 || g.Cg == 32) || g.C % 64 != 0) return false;
    if (g.sh > 2 || g.sw > 2 || g.Y * g.X > kBandMaxTaps) return false;
    if (g.Hi >= (1 << 20) || g.Wi >= (1 << 20)) return false;
    std::memset(&bp, 0, sizeof(bp));
    bp.N = g.N; bp.C = g.C; bp.Hi = g.Hi; bp.Wi = g.Wi; bp.sh = g.sh; bp.sw = g.sw;
    bp.cg = g.Cg; bp.ntaps = g.Y * g.X; bp.ncls = g.sh * g.sw; bp.cblocks = g.C / 64;
    // per residue: taps and their offsets
    std::vector<std::pair<int, int>> rt[2], ct[2];  // (filter index, offset)
    int oy_min = 1 << 30, oy_max = -(1 << 30), ox_min = 1 << 30, ox_max = -(1 << 30);
    for (int a = 0; a < g.sh; ++a)
        for (int y = 0; y < g.Y; ++y) {
            const int64_t num = (int64_t)a + g.ph - (int64_t)y * g.dh;
            if (((num % g.sh) + g.sh) % g.sh) continue;
            const int o = (int)(num / g.sh);
            rt[a].push_back({y, o});
            oy_min = std::min(oy_min, o); oy_max = std::max(oy_max, o);
        }
    for (int b = 0; b < g.sw; ++b)
        for (int x = 0; x < g.X; ++x) {
            const int64_t num = (int64_t)b + g.pw - (int64_t)x * g.dw;
            if (((num % g.sw) + g.sw) % g.sw) continue;
            const int o = (int)(num / g.sw);
            ct[b].push_back({x, o});
            ox_min = std::min(ox_min, o); ox_max = std::max(ox_max, o);
        }
    if (oy_min > oy_max || ox_min > ox_max) return false;
    bp.oy_min = oy_min; bp.ox_min = ox_min;
    bp.rows = 4 + oy_max - oy_min;
    bp.segw = 32 - (ox_max - ox_min);
    if (bp.rows > 64 || bp.segw < 16) return false;
    // windows: one per distinct (column shift, row offset); each class reads a
    // window with at most one tap (its row offset fixes y, its column offset x)
    std::memset(bp.win_tap, -1, sizeof(bp.win_tap));
    for (int a = 0; a < g.sh; ++a)
        for (int b = 0; b < g.sw; ++b) {
            const int c = a * g.sw + b;
            for (const auto &ry : rt[a])
                for (const auto &cx : ct[b]) {
                    const int cs = cx.second - ox_min, dr = ry.second - oy_min;
                    const int key = cs | (dr << 8);
                    int wi = 0;
                    while (wi < bp.nwin && bp.win[wi] != key) ++wi;
                    if (wi == bp.nwin) bp.win[bp.nwin++] = key;
                    bp.win_tap[wi][c] = (int8_t)(ry.first * g.X + cx.first);
                }
        }
    for (int a = 0; a < g.sh; ++a) bp.hc[a] = g.Hi > a ? (g.Hi - a + g.sh - 1) / g.sh : 0;
    for (int b = 0; b < g.sw; ++b) bp.wc[b] = g.Wi > b ? (g.Wi - b + g.sw - 1) / g.sw : 0;
    bp.bands = (bp.hc[0] + 3) / 4;
    bp.segs = (bp.wc[0] + bp.segw - 1) / bp.segw;
    const int64_t units = (int64_t)g.N * bp.bands * bp.segs;
    if (units <= 0 || units * bp.cblocks >= (1LL << 31)) return false;
    bp.units = (int)units;
    const int stage_bytes = bp.rows * 32 * 128;
    bp.stages = 0;
    for (int st = 6; st >= 2 && !bp.stages; --st)
        if (tc_band_smem_bytes(g.Cg, bp.ncls, bp.nwin, stage_bytes, st) <= 227 * 1024) bp.stages = st;
    if (!bp.stages) return false;
    bp.tmem_cols = 2 * bp.ncls * 64 <= 128 ? 128 : (2 * bp.ncls * 64 <= 256 ? 256 : 512);
    return true;
}

}  // namespace

namespace cbd {
conv_bwd_status plan_create_borrowed_status(const conv_bwd_desc *desc, int32_t *status, conv_bwd_plan *out);
}

namespace {

// fp32 tensor-core schedule of one launch (classes cls[0..nc) holding `total`
// tiles): tiles that do not fill a last round of the SMs are cut into equal
// k-block ranges over every SM (added into dx after a zeroing launch) when that
// round would leave at least a fifth of the SMs idle and each range keeps a few
// k blocks.  Returns whether to cut, and the k blocks of those tiles.
bool tf32_tail_split(const conv_bwd_plan_s *p, const ClassDesc *cls, size_t nc, int64_t total, int kb_per_tap,
                     int64_t *tail_units) {
    const int nsm = std::max(1, p->num_sms);
    const int64_t t_dp = (total / nsm) * nsm, tail = total - t_dp;
    int64_t units = 0;
    for (size_t i = 0; i < nc; ++i) {
        const int64_t te = i + 1 < nc ? cls[i + 1].tile_begin : total;
        const int64_t lo = std::max<int64_t>(cls[i].tile_begin, t_dp);
        if (te > lo) units += (te - lo) * cls[i].taps_y * cls[i].taps_x * kb_per_tap;
    }
    *tail_units = units;
    if (p->tf32_split >= 0) return tail > 0 && p->tf32_split == 1;
    return tail > 0 && tail * 5 <= (int64_t)nsm * 4 && units >= 4LL * nsm;
}

// K splits of the SM-pair kernel's split-K schedule for this plan (1 = whole
// tiles).  CONVBWD_DEBUG_SPLITK=S forces S (where the S * tiles units fit one
// wave).  By default: a layer whose 256 x 512 tiles number at most a third of
// the SM pairs (so S >= 3 splits fill the GPU) and whose reduction is deep
// enough for every split to keep >= 16 k-blocks: the 512-wide tiles need the
// fewest operand bytes per multiply-add (the pair kernels are bound by operand
// delivery) and the split gives them the whole GPU.  Measured on the dilated
// 3x3 stride-2 layer (C = K = 512, 72 k-blocks, 25 tiles): 35.5-36.9 us with 3
// splits against 37.3-37.6 us for 256-wide whole tiles on 50 pairs; 2 splits
// (39 us) and the 1x1 layer's 32 k-blocks (27-30 us against 21-23 us) lose.
int split_choice(const conv_bwd_plan_s *p, int max_pairs) {
    if (const char *f = env("CONVBWD_DEBUG_SPLITK")) {
        const int S = std::atoi(f);
        return S >= 2 && S <= 8 ? S : 1;
    }
    const Geom &g = p->g;
    if (g.Cg < 512 || max_pairs <= 0) return 1;
    int64_t tiles = 0;
    int min_kb = 1 << 30;
    const int kbt = (g.Kg + 63) / 64;
    for (const ClassDesc &c : p->classes) {
        tiles += (int64_t)g.G * ((c.M + 255) / 256) * ((g.Cg + 511) / 512);
        min_kb = std::min(min_kb, c.taps_y * c.taps_x * kbt);
    }
    if (tiles <= 0) return 1;
    for (int S = (int)std::min<int64_t>(4, max_pairs / tiles); S >= 3; --S)
        if (min_kb / S >= 16) return S;
    return 1;
}

int kHostChunks = 4;  // batch chunks of the pipelined host path (CONVBWD_DEBUG_HOST_CHUNKS overrides)

// Batch chunks for the pipelined host path: 4 chunks of ceil(N/4) images when
// the copies are large enough to be worth overlapping, else 1 (plain path).
// Sets up the chunk plans, copy streams and events on first use.
int host_chunks(conv_bwd_plan_s *p, size_t ndy, size_t ndx) {
    const conv_bwd_desc &d = p->desc;
    if (d.N < 2 || ndy + ndx < (16u << 20) || p->nhwc_plan) return 1;
    if (p->chunks) return p->chunks;
    p->chunks = 1;  // stays 1 (plain path) if any of the setup below fails
    if (const char *f = env("CONVBWD_DEBUG_HOST_CHUNKS")) kHostChunks = std::max(1, std::min(64, std::atoi(f)));
    if (kHostChunks < 2) return 1;
    const int64_t nc = (d.N + kHostChunks - 1) / kHostChunks;
    const int chunks = (int)((d.N + nc - 1) / nc);
    const int64_t tail = d.N - (int64_t)(chunks - 1) * nc;
    conv_bwd_desc cd = d;
    cd.N = nc;
    if (plan_create_borrowed_status(&cd, p->d_status, &p->chunk_plan[0]) != CONV_BWD_OK) return 1;
    if (tail != nc) {
        cd.N = tail;
        if (plan_create_borrowed_status(&cd, p->d_status, &p->chunk_plan[1]) != CONV_BWD_OK) return 1;
    }
    for (auto *c : p->chunk_plan)
        if (c) {  // fp32 tensor-core chunks split the filter into this plan's buffers (same stream, in turn)
            c->w_hi = p->w_hi;
            c->w_lo = p->w_lo;
            c->w_gkcyx = p->w_gkcyx;
        }
    if (cudaStreamCreateWithFlags(&p->h2d, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p->d2h, cudaStreamNonBlocking) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    p->hev.assign(2 + 2 * chunks, nullptr);
    for (auto &e : p->hev)
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            return 1;
        }
    p->chunk_n = (int32_t)nc;
    p->chunks = chunks;
    return chunks;
}

}  // namespace

extern "C" {

int32_t conv_bwd_data_version(void) { return 100; }

const char *conv_bwd_status_string(conv_bwd_status s) {
    switch (s) {
    case CONV_BWD_OK: return "CONV_BWD_OK";
    case CONV_BWD_ERR_INVALID_ARG: return "CONV_BWD_ERR_INVALID_ARG";
    case CONV_BWD_ERR_UNSUPPORTED: return "CONV_BWD_ERR_UNSUPPORTED";
    case CONV_BWD_ERR_MISALIGNED: return "CONV_BWD_ERR_MISALIGNED";
    case CONV_BWD_ERR_CUDA: return "CONV_BWD_ERR_CUDA";
    case CONV_BWD_ERR_DEVICE_TIMEOUT: return "CONV_BWD_ERR_DEVICE_TIMEOUT";
    case CONV_BWD_ERR_DEVICE_FAULT: return "CONV_BWD_ERR_DEVICE_FAULT";
    }
    return "CONV_BWD_UNKNOWN_STATUS";
}

static conv_bwd_status create_impl(const conv_bwd_desc *desc, conv_bwd_plan *out, bool alloc_status) {
    if (!out) return CONV_BWD_ERR_INVALID_ARG;
    *out = nullptr;
    conv_bwd_status st = validate(desc);
    if (st != CONV_BWD_OK) return st;
    const conv_bwd_desc &d = *desc;
    int64_t Ho = (d.Hi + 2LL * d.pad_h - (int64_t)d.dil_h * (d.Y - 1) - 1) / d.stride_h + 1;
    int64_t Wo = (d.Wi + 2LL * d.pad_w - (int64_t)d.dil_w * (d.X - 1) - 1) / d.stride_w + 1;
    const int64_t lim = 0x7fffffffLL;
    if (d.N * d.C * d.Hi * d.Wi > lim || d.N * d.K * Ho * Wo > lim || d.K * (d.C / d.groups) * d.Y * d.X > lim)
        return CONV_BWD_ERR_UNSUPPORTED;

    conv_bwd_plan_s *p = new (std::nothrow) conv_bwd_plan_s();
    if (!p) return CONV_BWD_ERR_CUDA;
    p->desc = d;
    Geom &g = p->g;
    g.N = (int)d.N; g.C = (int)d.C; g.K = (int)d.K; g.Hi = (int)d.Hi; g.Wi = (int)d.Wi;
    g.Ho = (int)Ho; g.Wo = (int)Wo; g.Y = (int)d.Y; g.X = (int)d.X;
    g.ph = d.pad_h; g.pw = d.pad_w; g.sh = d.stride_h; g.sw = d.stride_w; g.dh = d.dil_h; g.dw = d.dil_w;
    g.G = d.groups; g.Cg = (int)(d.C / d.groups); g.Kg = (int)(d.K / d.groups);

    std::vector<DimClass> ch, cw;
    int64_t uh, uw;
    plan_dim(d.Hi, Ho, d.Y, d.stride_h, d.dil_h, d.pad_h, g.YT, g.DH, ch, p->cov_h, p->row_cov, uh);
    plan_dim(d.Wi, Wo, d.X, d.stride_w, d.dil_w, d.pad_w, g.XT, g.DW, cw, p->cov_w, p->col_cov, uw);
    p->useful_flop = 2.0 * (double)d.N * (double)d.K * (double)g.Cg * (double)uh * (double)uw;
    size_t es = elem_size(d.dtype);
    p->algo_bytes = (double)es * ((double)d.N * d.K * Ho * Wo + (double)d.K * g.Cg * d.Y * d.X +
                                  (double)d.N * d.C * d.Hi * d.Wi);
    for (uint8_t v : p->row_cov) p->any_uncovered |= (v == 0);
    for (uint8_t v : p->col_cov) p->any_uncovered |= (v == 0);

    // Non-empty sub-GEMMs, consecutive gemmIds (row class major).
    for (const DimClass &a : ch)
        for (const DimClass &b : cw) {
            if (a.taps == 0 || b.taps == 0 || a.cnt == 0 || b.cnt == 0) continue;
            ClassDesc c{};
            c.ty = a.t; c.tx = b.t; c.taps_y = a.taps; c.taps_x = b.taps;
            c.ht_lo = a.lo; c.HT = a.cnt; c.wt_lo = b.lo; c.WT = b.cnt;
            int64_t M = d.N * (int64_t)a.cnt * b.cnt;
            c.M = (int)M;
            c.gemm_id = (int)p->classes.size();
            c.pty = c.ptx = -1;
            p->classes.push_back(c);
        }
    if ((int)p->classes.size() > kMaxClasses) {
        delete p;
        return CONV_BWD_ERR_UNSUPPORTED;
    }

    // Strides of the logical orders dy[n][k][h][w], w[k][c][y][x], dx[n][c][h][w].
    Strides &s = p->st;
    if (d.layout == CONV_BWD_NCHW_GKCYX) {
        s.dy_w = 1; s.dy_h = Wo; s.dy_k = Ho * Wo; s.dy_n = d.K * Ho * Wo;
        s.w_x = 1; s.w_y = d.X; s.w_c = d.Y * d.X; s.w_k = g.Cg * d.Y * d.X;
        s.dx_w = 1; s.dx_h = d.Wi; s.dx_c = d.Hi * d.Wi; s.dx_n = d.C * d.Hi * d.Wi;
    } else {
        s.dy_k = 1; s.dy_w = d.K; s.dy_h = Wo * d.K; s.dy_n = Ho * Wo * d.K;
        s.w_c = 1; s.w_x = g.Cg; s.w_y = d.X * g.Cg; s.w_k = d.Y * d.X * g.Cg;
        s.dx_c = 1; s.dx_w = d.C; s.dx_h = d.Wi * d.C; s.dx_n = d.Hi * d.Wi * d.C;
    }

    // Kernel path.
    bool tc_ok = d.dtype == CONV_BWD_BF16 && d.layout == CONV_BWD_NHWC_KYXC && g.Cg % 8 == 0 && g.Kg % 8 == 0 &&
                 d.K % 8 == 0 && d.C % 8 == 0 && g.Cg >= 64 && d.Hi < 16384 && d.Wi < 16384;
    // narrow groups: memory-bound kernel on warp-level MMAs (dy rows and w
    // fragments staged in shared memory)
    bool grouped_ok = d.dtype == CONV_BWD_BF16 && d.layout == CONV_BWD_NHWC_KYXC && g.Cg == g.Kg &&
                      (g.Cg == 8 || g.Cg == 16) && g.G % 8 == 0 && d.Y * d.X <= 64 &&
                      d.Hi < (1 << 20) && d.Wi < (1 << 20) && d.stride_w <= 64 &&
                      d.N * d.Hi * ((d.Wi + 15) / 16) < (1LL << 31);  // item count (chunks of >= 16 pixels)
    if (grouped_ok) grouped_ok = grouped_layout(g).smem <= 200 * 1024;
    // narrow groups on tcgen05: the groups of each 64-channel block folded into
    // one GEMM with a block-diagonal B (resident in shared memory, one 8 KB tile
    // per filter tap), A by TMA im2col as on the wide path
    bool grouped_tc = d.dtype == CONV_BWD_BF16 && d.layout == CONV_BWD_NHWC_KYXC && g.Cg == g.Kg &&
                      (g.Cg == 8 || g.Cg == 16 || g.Cg == 32) && d.C % 64 == 0 && d.Y * d.X <= 12 &&
                      d.Hi < 16384 && d.Wi < 16384;
    for (const ClassDesc &c : p->classes) {
        int lo[2], hi[2];
        im2col_corners(g, c, lo, hi);
        for (int q = 0; q < 2; ++q)
            if (lo[q] < -128 || lo[q] > 127 || hi[q] < -128 || hi[q] > 127) grouped_tc = false;
        if ((c.taps_x - 1) * g.DW > 127 || (c.taps_y - 1) * g.DH > 127) grouped_tc = false;
    }
    // narrow groups on tcgen05 with each band of dy staged once and read by
    // every tap (strides <= 2, C % 64 == 0)
    BandParams band;
    const bool band_ok = plan_band(d, g, band);
    // Default order: the banded kernel; then the warp-level MMA kernel, which
    // stages each dy row once per item and reuses it for every tap; then the
    // per-tap tcgen05 kernel, which re-reads dy per tap from L2 (78 vs 51 us
    // for the warp-level kernel on the ResNeXt layer).  CONVBWD_DEBUG_GROUPED
    // = band | mma | tc selects one where it applies.
    int gkind = band_ok ? 3 : (grouped_ok ? 1 : (grouped_tc ? 2 : 0));
    if (const char *gk = env("CONVBWD_DEBUG_GROUPED")) {
        if (!std::strcmp(gk, "tc") && grouped_tc) gkind = 2;
        if (!std::strcmp(gk, "mma") && grouped_ok) gkind = 1;
        if (!std::strcmp(gk, "band") && band_ok) gkind = 3;
    }
    grouped_ok = gkind != 0;
    // fp32 on the tensor cores (three-term TF32 split) for problems large
    // enough to pay for the filter split launch; NHWC/KYXC, 32-channel TMA
    // im2col blocks that stay inside a group, 16-byte pixel strides
    bool tf32_ok = d.dtype == CONV_BWD_F32 && d.layout == CONV_BWD_NHWC_KYXC && d.K % 4 == 0 && d.C % 4 == 0 &&
                   g.Cg % 4 == 0 && g.Kg % 4 == 0 && (g.G == 1 || g.Kg % kTf32BK == 0) && d.Hi < 16384 &&
                   d.Wi < 16384;
    for (const ClassDesc &c : p->classes) {
        int lo[2], hi[2];
        im2col_corners(g, c, lo, hi);
        for (int q = 0; q < 2; ++q)
            if (lo[q] < -128 || lo[q] > 127 || hi[q] < -128 || hi[q] > 127) tf32_ok = false;
        if ((c.taps_x - 1) * g.DW > 127 || (c.taps_y - 1) * g.DH > 127) tf32_ok = false;
    }
    const char *force = env("CONVBWD_DEBUG_PATH");
    const bool tf32_big = p->useful_flop >= kTf32MinFlop || (force && !std::strcmp(force, "tf32"));
    p->path = tc_ok ? CONV_BWD_PATH_TCGEN05
                    : (grouped_ok ? CONV_BWD_PATH_GROUPED
                                  : (tf32_ok && tf32_big ? CONV_BWD_PATH_TF32 : CONV_BWD_PATH_SIMT));
    if (force && !std::strcmp(force, "simt")) p->path = CONV_BWD_PATH_SIMT;
    p->grouped_tc = p->path == CONV_BWD_PATH_GROUPED && gkind == 2;
    p->grouped_band = p->path == CONV_BWD_PATH_GROUPED && gkind == 3;
    if (p->grouped_band) p->band = band;
    // CUDA-core tiles: 64 x 64, or 64 x 32 for fp32 with C/G <= 32 (no idle columns)
    const int simt_bn = d.dtype == CONV_BWD_F32 && g.Cg <= 32 ? 32 : 64;
    p->bn = (p->path == CONV_BWD_PATH_TCGEN05) ? (g.Cg >= 256 ? 256 : 128)
                                               : (p->path == CONV_BWD_PATH_TF32 ? kTf32BN : simt_bn);
    if (const char *f = env("CONVBWD_DEBUG_BN"))
        if (p->path == CONV_BWD_PATH_TCGEN05 && (!std::strcmp(f, "128") || !std::strcmp(f, "256"))) p->bn = std::atoi(f);
    // im2col loads read 64 channels past k0 of dy's flat K axis, exact only
    // when no 64-block crosses a group boundary; rank-4 im2col corners must
    // lie in [-128, 127].  Otherwise the cp.async gather producer runs.
    p->im2col = p->path == CONV_BWD_PATH_TCGEN05 && (g.G == 1 || g.Kg % 64 == 0);
    for (const ClassDesc &c : p->classes) {
        int lo[2], hi[2];
        im2col_corners(g, c, lo, hi);
        for (int q = 0; q < 2; ++q)
            if (lo[q] < -128 || lo[q] > 127 || hi[q] < -128 || hi[q] > 127) p->im2col = false;
        // the tap is the im2col offset: keep it within 7 bits
        if ((c.taps_x - 1) * g.DW > 127 || (c.taps_y - 1) * g.DH > 127) p->im2col = false;
    }
    if (const char *f = env("CONVBWD_DEBUG_NOIM2COL")) p->im2col = p->im2col && f[0] == '0';
    // 256-row tiles on SM pairs (tcgen05 cta_group::2): each SM then loads only
    // half of B.  The tile width comes from a wave-count cost model:
    //   time ~ ceil(tiles(bn) / pairs) * cost(bn)
    // with the measured cost of one tile relative to a 256-wide one (same K):
    // 128 wide 0.85 (more operand bytes per output), 512 wide 1.785 (two N=256
    // MMAs per k slice, fewer A bytes per output, single-buffered accumulator).
    p->two_sm = p->path == CONV_BWD_PATH_TCGEN05 && p->im2col && g.Cg >= 256;  // (C/G < 256: 1-SM tiles measured faster)
    if (const char *f = env("CONVBWD_DEBUG_NO2SM")) p->two_sm = p->two_sm && f[0] == '0';
    if (const char *f = env("CONVBWD_DEBUG_2SM"))
        if (f[0] == '1') p->two_sm = p->path == CONV_BWD_PATH_TCGEN05 && p->im2col && g.Cg >= 128;
    if (p->two_sm) {
        int sms = 0, dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaGetLastError();
        const int64_t pairs = sms > 0 ? sms / 2 : 74;
        auto tiles_of = [&](int bn) {
            int64_t t = 0;
            for (const ClassDesc &c : p->classes) t += (int64_t)g.G * ((c.M + 255) / 256) * ((g.Cg + bn - 1) / bn);
            return t;
        };
        const int widths[3] = {128, 256, 512};
        const double cost[3] = {0.85, 1.0, 1.785};
        double best = 1e300;
        for (int i = 0; i < 3; ++i) {
            if (widths[i] > 128 && g.Cg <= widths[i] / 2) continue;  // at least half the tile is real columns
            const double t = (double)((tiles_of(widths[i]) + pairs - 1) / pairs) * cost[i];
            if (t < best) {
                best = t;
                p->bn = widths[i];
            }
        }
        // SM pairs or 1-SM 128 x 128 tiles: a makespan estimate of both in SM
        // clocks.  Tiles are dealt to workers (pairs, or SMs) in the kernels'
        // snake order, classes with the most taps first; a tile costs its
        // k-blocks times the measured main-loop clocks per k-block of its kind
        // (1-SM 128 wide 710; pairs 128 wide 845, 256 wide 808, 512 wide 1100)
        // and its epilogue, from the per-tile rate of layers whose epilogues set
        // the pace (1-SM 128 x 128: 2400 clocks; pairs: 7100 per 256 columns):
        // added after every 512-wide tile (single-buffered accumulator);
        // otherwise overlapped with the next tile's MMAs (a tile costs the
        // larger of the two) and added once after the last tile.  The 1-SM tiles win on
        // layers with few tiles (one round, or a second round of cheap classes)
        // and on shallow ones whose epilogues set the pace.  Measured on 22
        // layers (1x1 and 3x3, C/G 256..2048, 1..72 k-blocks): 1-SM tiles 0-30 %
        // faster where chosen; where pairs are kept they are faster, or the
        // 1-SM tiles at most 4 % faster.  Tiles deeper than 64 k-blocks keep the
        // pairs, whose split-K reaches ~90 % of the MMA rate.  Any SM-pair
        // override (CONVBWD_DEBUG_2SM=1, tile width, split-K, stream-K, A
        // operand) keeps the pairs.
        const bool pinned = env("CONVBWD_DEBUG_2SM") || env("CONVBWD_DEBUG_BN") || env("CONVBWD_DEBUG_SPLITK") ||
                            env("CONVBWD_DEBUG_STREAMK") || env("CONVBWD_DEBUG_A");
        const int64_t kbt = (g.Kg + 63) / 64;
        int64_t t1 = 0, kb_max = 0;
        for (const ClassDesc &c : p->classes) {
            t1 += (int64_t)g.G * ((c.M + 127) / 128) * ((g.Cg + 127) / 128);
            kb_max = std::max(kb_max, (int64_t)c.taps_y * c.taps_x * kbt);
        }
        if (!pinned && kb_max <= 64 && t1 <= 64 * 2 * pairs) {
            std::vector<const ClassDesc *> order;
            for (const ClassDesc &c : p->classes) order.push_back(&c);
            std::stable_sort(order.begin(), order.end(), [](const ClassDesc *a, const ClassDesc *b) {
                return a->taps_y * a->taps_x > b->taps_y * b->taps_x;
            });
            // snake makespan of `workers` over tiles of `rows` x `bn` whose
            // epilogues take `epi` clocks
            auto makespan = [&](int64_t workers, int rows, int bn, double per_kb, double epi, bool epi_each) {
                int64_t n = 0;
                for (const ClassDesc *c : order) n += (int64_t)g.G * ((c->M + rows - 1) / rows) * ((g.Cg + bn - 1) / bn);
                const int64_t W = std::max<int64_t>(1, std::min(workers, n));
                std::vector<double> load((size_t)W, 0.0);
                int64_t t = 0;
                for (const ClassDesc *c : order) {
                    const int64_t nt = (int64_t)g.G * ((c->M + rows - 1) / rows) * ((g.Cg + bn - 1) / bn);
                    const double mma = (double)(c->taps_y * c->taps_x * kbt) * per_kb;
                    const double cost = epi_each ? mma + epi : std::max(mma, epi);
                    for (int64_t q = 0; q < nt; ++q, ++t) {
                        const int64_t k = t / W, r = t - k * W;
                        load[(size_t)((k & 1) ? W - 1 - r : r)] += cost;
                    }
                }
                return *std::max_element(load.begin(), load.end()) + (epi_each ? 0.0 : epi);
            };
            const double pair_kb = p->bn == 512 ? 1100.0 : (p->bn == 256 ? 808.0 : 845.0);
            const double t_pair = makespan(pairs, 256, p->bn, pair_kb, 7100.0 * p->bn / 256, p->bn == 512);
            const double t_one = makespan(2 * pairs, 128, 128, 710.0, 2400.0, false);
            if (t_one < t_pair) {
                p->two_sm = false;
                p->bn = 128;
            }
        }
    }
    if (const char *f = env("CONVBWD_DEBUG_BN")) {
        if (p->path == CONV_BWD_PATH_TCGEN05 && (!std::strcmp(f, "128") || !std::strcmp(f, "256"))) p->bn = std::atoi(f);
        if (p->two_sm && !std::strcmp(f, "512")) p->bn = 512;
    }
    if (const char *f = env("CONVBWD_DEBUG_STREAMK")) p->tf32_split = f[0] == '1' ? 1 : 0;
    // Plain-matrix specialisation (SM-pair kernel): every class has one tap and
    // its rows are all of dy's pixels in order, so A is dy viewed as the matrix
    // {N*Ho*Wo, K} and loads as 2-D tiles (no im2col offsets).  Off by
    // default (one dynamic kernel for every shape, as in the dynamic-kernel
    // pull request); CONVBWD_DEBUG_A=plain selects it where it applies, and
    // the benchmark reports both on the shapes that qualify.
    if (p->two_sm) {
        bool plain = true;
        for (const ClassDesc &c : p->classes)
            plain = plain && c.taps_y == 1 && c.taps_x == 1 && c.ht_lo == 0 && c.HT == g.Ho && c.wt_lo == 0 &&
                    c.WT == g.Wo;
        const char *f = env("CONVBWD_DEBUG_A");
        p->a_plain = plain && f && !std::strcmp(f, "plain");
    }
    // Class pairs on the 1-SM kernel (C/G <= 128): two classes with the same
    // rows (ht, wt ranges) and tap counts read the same dy rows for every tap
    // (tap (j, i) reads ho = ht - j*DH, wo = wt - i*DW in any class), so one
    // 128 x 256 tile computes both -- one A load and one N = 256 MMA per k
    // slice where two N = 128 tiles would load A twice and issue twice as many
    // MMAs (an N = 256 MMA measured ~200 SM clocks in this kernel against ~175
    // for N = 128).  CONVBWD_DEBUG_FUSE=0 keeps one class per tile.
    if (p->path == CONV_BWD_PATH_TCGEN05 && !p->two_sm && p->im2col && !p->a_plain && g.Cg <= 128) {
        for (size_t a = 0; a < p->classes.size() && !p->fuse; ++a)
            for (size_t b = a + 1; b < p->classes.size() && !p->fuse; ++b)
                p->fuse = fusable_classes(p->classes[a], p->classes[b]);
        if (const char *f = env("CONVBWD_DEBUG_FUSE"))
            if (f[0] == '0') p->fuse = false;
        if (p->fuse) p->bn = 256;
    }

    // Schedule: classes with the longest reduction first (LPT), tiles of one
    // class contiguous; BM = 256 rows on SM pairs, 128 for the 1-SM
    // tensor-core kernel, 64 for SIMT.
    const int bm = p->path == CONV_BWD_PATH_TCGEN05 ? (p->two_sm ? 256 : 128)
                                                    : (p->path == CONV_BWD_PATH_TF32 ? 128 : 64);
    p->sched.resize(p->classes.size());
    std::iota(p->sched.begin(), p->sched.end(), 0);
    std::stable_sort(p->sched.begin(), p->sched.end(), [&](int a, int b) {
        return p->classes[a].taps_y * p->classes[a].taps_x > p->classes[b].taps_y * p->classes[b].taps_x;
    });
    // per-class m tiles and tile offsets for row tiles of `rows` and the plan's tile width
    auto schedule = [p, &g](int rows) {
        const int n_tiles = (g.Cg + p->bn - 1) / p->bn;
        int64_t total = 0;
        for (int idx : p->sched) {
            ClassDesc &c = p->classes[(size_t)idx];
            c.m_tiles = (c.M + rows - 1) / rows;
            c.tile_begin = (int)total;
            total += (int64_t)g.G * c.m_tiles * n_tiles;
        }
        return total;
    };
    if (schedule(bm) > lim) {
        delete p;
        return CONV_BWD_ERR_UNSUPPORTED;
    }

    // Device resources (optional: planning works without a GPU).
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) == cudaSuccess && ndev > 0) {
        cudaGetDevice(&p->device);
        cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
        int clk_khz = 0;
        cudaDeviceGetAttribute(&clk_khz, cudaDevAttrClockRate, p->device);
        if (clk_khz <= 0) clk_khz = 2000000;
        double secs = 2.0;
        if (const char *b = env("CONVBWD_DEBUG_WAIT_SECONDS")) secs = std::atof(b);
        p->wait_budget = (int64_t)(secs * clk_khz * 1000.0);
        if (alloc_status) {
            if (cudaMalloc(&p->d_status, 16) != cudaSuccess || cudaMemset(p->d_status, 0, 16) != cudaSuccess) {
                cudaGetLastError();
                delete p;
                return CONV_BWD_ERR_CUDA;
            }
            p->has_device = true;
#ifdef CBD_PHASE_TIMES
            if (cudaMalloc(&p->d_phase, kPhaseLogCtas * kPhaseSlots * sizeof(unsigned long long)) != cudaSuccess) {
                cudaGetLastError();
                p->d_phase = nullptr;
            }
#endif
            const char *sk = env("CONVBWD_DEBUG_STREAMK");
            if (p->two_sm && sk && sk[0] == '1') {
                // stream-K workspace: only for plans created with the opt-in stream-K
                // schedule (the default whole-tile schedule never touches it)
                p->max_pairs = tc2_max_pairs(p->num_sms);
                const size_t slots = (size_t)p->max_pairs * 2;
                if (cudaMalloc(&p->d_partials, slots * 128 * 64 * sizeof(float4)) != cudaSuccess ||
                    cudaMalloc(&p->d_flags, slots * sizeof(int32_t)) != cudaSuccess ||
                    cudaMemset(p->d_flags, 0, slots * sizeof(int32_t)) != cudaSuccess) {
                    cudaGetLastError();
                    cudaFree(p->d_partials);
                    cudaFree(p->d_flags);
                    p->d_partials = nullptr;
                    p->d_flags = nullptr;
                }
            }
            if (p->two_sm && !(sk && sk[0] == '1') && p->classes.size() <= (size_t)kMaxTcClasses) {
                // Split-K with a reduce-scatter of the fp32 partials: S SM pairs per
                // 256 x 512 tile, each over 1/S of the k-blocks, all tiles in one wave.
                // The widest tile needs the fewest operand bytes per multiply-add (the
                // SM pairs are bound by operand delivery), and the split gives a deep,
                // short layer enough such tiles to fill the GPU.
                int S = split_choice(p, tc2_max_pairs(p->num_sms));
                const int kbt = (g.Kg + 63) / 64;
                for (const ClassDesc &c : p->classes)  // every split keeps at least two k-blocks
                    if (c.taps_y * c.taps_x * kbt < 2 * S) S = 1;
                if (S > 1) {
                    const int bn_s = g.Cg > 256 ? 512 : 256;
                    int64_t tiles = 0;
                    for (const ClassDesc &c : p->classes)
                        tiles += (int64_t)g.G * ((c.M + 255) / 256) * ((g.Cg + bn_s - 1) / bn_s);
                    const size_t blk = (size_t)(bn_s / 4) * 128;
                    const size_t ws = (size_t)tiles * 2 * (S - 1) * blk * sizeof(float4);
                    const size_t nfl = (size_t)tiles * S * 2;
                    if (tiles * S <= tc2_max_pairs(p->num_sms) && cudaMalloc(&p->d_ws, ws) == cudaSuccess &&
                        cudaMalloc(&p->d_ws_flags, nfl * sizeof(int32_t)) == cudaSuccess &&
                        cudaMemset(p->d_ws_flags, 0, nfl * sizeof(int32_t)) == cudaSuccess) {
                        p->splitk = S;
                        p->bn = bn_s;
                        schedule(256);
                    } else {
                        cudaGetLastError();
                        cudaFree(p->d_ws);
                        cudaFree(p->d_ws_flags);
                        p->d_ws = nullptr;
                        p->d_ws_flags = nullptr;
                    }
                }
            }
            const size_t nsplit = (size_t)d.K * g.Cg * d.Y * d.X * sizeof(float);
            if (p->path == CONV_BWD_PATH_TF32) {
                // (CONVBWD_DEBUG_NO_WSPLIT: take the fallback below as if the allocation had failed)
                if (!env("CONVBWD_DEBUG_NO_WSPLIT") && cudaMalloc(&p->w_hi, nsplit) == cudaSuccess &&
                    cudaMalloc(&p->w_lo, nsplit) == cudaSuccess) {
                    p->owns_wsplit = true;
                } else {
                    // no room for the split filter: CUDA-core path, rescheduled for its 64-row tiles
                    cudaGetLastError();
                    cudaFree(p->w_hi);
                    cudaFree(p->w_lo);
                    p->w_hi = p->w_lo = nullptr;
                    p->path = CONV_BWD_PATH_SIMT;
                    p->bn = simt_bn;
                    if (schedule(64) > lim) {
                        conv_bwd_data_destroy(p);
                        return CONV_BWD_ERR_CUDA;
                    }
                }
            }
            // NCHW/GKCYX: run the NHWC/KYXC plan of the same geometry between
            // layout transposes when that plan is on a tensor-core path (bf16:
            // dy, w and dx transposed; fp32: dy and dx, the filter split reads
            // GKCYX directly)
            if (d.layout == CONV_BWD_NCHW_GKCYX && !env("CONVBWD_DEBUG_NO_TRANSPOSE")) {
                conv_bwd_desc nd = d;
                nd.layout = CONV_BWD_NHWC_KYXC;
                conv_bwd_plan child = nullptr;
                if (plan_create_borrowed_status(&nd, p->d_status, &child) == CONV_BWD_OK &&
                    child->path != CONV_BWD_PATH_SIMT) {
                    const bool f32 = d.dtype == CONV_BWD_F32;
                    const size_t ndy = (size_t)d.N * d.K * g.Ho * g.Wo * es, nw = (size_t)d.K * g.Cg * d.Y * d.X * es,
                                 ndx = (size_t)d.N * d.C * d.Hi * d.Wi * es;
                    bool ok = cudaMalloc(&p->t_dy, ndy) == cudaSuccess && cudaMalloc(&p->t_dx, ndx) == cudaSuccess;
                    if (ok && f32)
                        ok = cudaMalloc(&p->w_hi, nsplit) == cudaSuccess && cudaMalloc(&p->w_lo, nsplit) == cudaSuccess;
                    else if (ok)
                        ok = cudaMalloc(&p->t_w, nw) == cudaSuccess;
                    if (ok) {
                        if (f32) {
                            p->owns_wsplit = true;
                            child->w_hi = p->w_hi;
                            child->w_lo = p->w_lo;
                            child->w_gkcyx = 1;
                        }
                        p->nhwc_plan = child;
                        child = nullptr;
                    } else {
                        cudaGetLastError();
                        cudaFree(p->t_dy);
                        cudaFree(p->t_w);
                        cudaFree(p->t_dx);
                        cudaFree(p->w_hi);
                        cudaFree(p->w_lo);
                        p->t_dy = p->t_w = p->t_dx = nullptr;
                        p->w_hi = p->w_lo = nullptr;
                    }
                }
                conv_bwd_data_destroy(child);
            }
        } else {
            p->owns_status = false;  // run() becomes possible once a status word is attached
        }
    } else {
        cudaGetLastError();  // clear "no device"
    }
    *out = p;
    return CONV_BWD_OK;
}

conv_bwd_status conv_bwd_data_create(const conv_bwd_desc *desc, conv_bwd_plan *out) {
    return create_impl(desc, out, true);
}

conv_bwd_status conv_bwd_data_destroy(conv_bwd_plan p) {
    if (!p) return CONV_BWD_OK;
    if (p->has_device) {
        int cur = -1;
        cudaGetDevice(&cur);
        if (cur != p->device) cudaSetDevice(p->device);
        if (p->owns_status) cudaFree(p->d_status);
#ifdef CBD_PHASE_TIMES
        cudaFree(p->d_phase);
#endif
        cudaFree(p->d_partials);
        cudaFree(p->d_flags);
        cudaFree(p->d_ws);
        cudaFree(p->d_ws_flags);
        for (auto &e : p->ev)
            if (e) cudaEventDestroy(e);
        for (auto &e : p->hev)
            if (e) cudaEventDestroy(e);
        cudaFree(p->t_dy);
        cudaFree(p->t_w);
        cudaFree(p->t_dx);
        if (p->owns_wsplit) {
            cudaFree(p->w_hi);
            cudaFree(p->w_lo);
        }
        if (p->h2d) cudaStreamDestroy(p->h2d);
        if (p->d2h) cudaStreamDestroy(p->d2h);
        if (cur != p->device && cur >= 0) cudaSetDevice(cur);
    }
    for (auto *c : p->chunk_plan) conv_bwd_data_destroy(c);  // borrowed status: frees only their own state
    conv_bwd_data_destroy(p->nhwc_plan);
    delete p;
    return CONV_BWD_OK;
}

conv_bwd_status conv_bwd_data_out_dims(const conv_bwd_plan p, int64_t *Ho, int64_t *Wo) {
    if (!p) return CONV_BWD_ERR_INVALID_ARG;
    if (Ho) *Ho = p->g.Ho;
    if (Wo) *Wo = p->g.Wo;
    return CONV_BWD_OK;
}

conv_bwd_status conv_bwd_data_num_subgemms(const conv_bwd_plan p, int32_t *n) {
    if (!p || !n) return CONV_BWD_ERR_INVALID_ARG;
    *n = (int32_t)p->classes.size();
    return CONV_BWD_OK;
}

conv_bwd_status conv_bwd_data_subgemm_info(const conv_bwd_plan p, int32_t id, int32_t *ty, int32_t *tx, int64_t *M,
                                           int64_t *N, int64_t *K, int32_t *taps_y, int32_t *taps_x) {
    if (!p || id < 0 || id >= (int32_t)p->classes.size()) return CONV_BWD_ERR_INVALID_ARG;
    const ClassDesc &c = p->classes[(size_t)id];
    if (ty) *ty = c.ty;
    if (tx) *tx = c.tx;
    if (M) *M = c.M;
    if (N) *N = p->g.Cg;
    if (K) *K = (int64_t)p->g.Kg * c.taps_y * c.taps_x;
    if (taps_y) *taps_y = c.taps_y;
    if (taps_x) *taps_x = c.taps_x;
    return CONV_BWD_OK;
}

conv_bwd_status conv_bwd_data_coverage(const conv_bwd_plan p, uint8_t *row_mask, uint8_t *col_mask) {
    if (!p) return CONV_BWD_ERR_INVALID_ARG;
    if (row_mask) std::memcpy(row_mask, p->row_cov.data(), p->row_cov.size());
    if (col_mask) std::memcpy(col_mask, p->col_cov.data(), p->col_cov.size());
    return CONV_BWD_OK;
}

conv_bwd_status conv_bwd_data_path(const conv_bwd_plan p, int32_t *path, int32_t *launches) {
    if (!p) return CONV_BWD_ERR_INVALID_ARG;
    if (p->nhwc_plan) {  // dy (and bf16 w) transposed in, dx transposed out, around the NHWC plan's kernels
        conv_bwd_status st = conv_bwd_data_path(p->nhwc_plan, path, launches);
        if (launches) *launches += p->t_w ? 3 : 2;
        return st;
    }
    if (path) *path = p->path;
    int gemm_launches = p->classes.empty() ? 0 : 1;
    if (p->path == CONV_BWD_PATH_TCGEN05) {
        std::vector<ClassDesc> lcls;
        std::vector<int> lmap;
        launch_classes(p, lcls, lmap);
        gemm_launches = (int)((lcls.size() + kMaxTcClasses - 1) / kMaxTcClasses);
    }
    // the warp-MMA narrow-group kernel writes every pixel; the tensor-core
    // kernels zero uncovered pixels themselves; without any class the fill
    // kernel alone runs
    const bool mma_grouped = p->path == CONV_BWD_PATH_GROUPED && !p->grouped_tc;
    const bool fill = p->any_uncovered && (p->path == CONV_BWD_PATH_SIMT || (p->classes.empty() && !mma_grouped));
    if (p->path == CONV_BWD_PATH_GROUPED)
        gemm_launches = p->grouped_tc ? (int)((p->classes.size() + kMaxTcClasses - 1) / kMaxTcClasses) : 1;
    if (p->path == CONV_BWD_PATH_TF32) {
        // the filter split, then per launch of up to kMaxTcClasses classes the
        // tensor-core kernel (which fills), preceded by the tile zeroing when its
        // last round of tiles is cut into k-block ranges (the same decision as run)
        gemm_launches = 1;
        const int n_tiles = (p->g.Cg + kTf32BN - 1) / kTf32BN, kbt = (p->g.Kg + kTf32BK - 1) / kTf32BK;
        for (size_t c0 = 0; c0 < p->sched.size(); c0 += kMaxTcClasses) {
            const size_t nc = std::min<size_t>(kMaxTcClasses, p->sched.size() - c0);
            ClassDesc cls[kMaxTcClasses];
            int64_t total = 0, units = 0;
            for (size_t i = 0; i < nc; ++i) {
                cls[i] = p->classes[(size_t)p->sched[c0 + i]];
                cls[i].tile_begin = (int)total;
                total += (int64_t)p->g.G * cls[i].m_tiles * n_tiles;
            }
            gemm_launches += 1 + (p->num_sms > 0 && tf32_tail_split(p, cls, nc, total, kbt, &units) ? 1 : 0);
        }
    }
    if (launches) *launches = (fill ? 1 : 0) + gemm_launches;
    return CONV_BWD_OK;
}

conv_bwd_status conv_bwd_data_tile(const conv_bwd_plan p, int32_t *tile_m, int32_t *tile_n, int32_t *sms) {
    if (!p) return CONV_BWD_ERR_INVALID_ARG;
    if (p->nhwc_plan) return conv_bwd_data_tile(p->nhwc_plan, tile_m, tile_n, sms);
    const bool tc = p->path == CONV_BWD_PATH_TCGEN05, grouped = p->path == CONV_BWD_PATH_GROUPED;
    const bool gtc = p->grouped_tc || p->grouped_band;
    if (tile_m) *tile_m = grouped ? (gtc ? 128 : 0) : tc ? (p->two_sm ? 256 : 128)
                                                                   : p->path == CONV_BWD_PATH_TF32 ? 128 : 64;
    if (tile_n) *tile_n = grouped ? (gtc ? 64 : 0) : p->bn;
    if (sms) *sms = tc && p->two_sm ? 2 : 1;
    return CONV_BWD_OK;
}

conv_bwd_status conv_bwd_data_k_splits(const conv_bwd_plan p, int32_t *k_splits) {
    if (!p || !k_splits) return CONV_BWD_ERR_INVALID_ARG;
    if (p->nhwc_plan) return conv_bwd_data_k_splits(p->nhwc_plan, k_splits);
    *k_splits = p->path == CONV_BWD_PATH_TCGEN05 ? p->splitk : 1;
    return CONV_BWD_OK;
}

conv_bwd_status conv_bwd_data_a_operand(const conv_bwd_plan p, int32_t *a_mode) {
    if (!p || !a_mode) return CONV_BWD_ERR_INVALID_ARG;
    if (p->nhwc_plan) return conv_bwd_data_a_operand(p->nhwc_plan, a_mode);
    const bool tc = p->path == CONV_BWD_PATH_TCGEN05 || p->path == CONV_BWD_PATH_TF32 || p->grouped_tc;
    *a_mode = p->grouped_band ? CONV_BWD_A_BAND
            : !tc ? CONV_BWD_A_GATHER
                  : (p->a_plain ? CONV_BWD_A_PLAIN
                                : (p->im2col || p->path != CONV_BWD_PATH_TCGEN05 ? CONV_BWD_A_IM2COL : CONV_BWD_A_GATHER));
    return CONV_BWD_OK;
}

conv_bwd_status conv_bwd_data_grouped_kernel(const conv_bwd_plan p, int32_t *kind) {
    if (!p || !kind) return CONV_BWD_ERR_INVALID_ARG;
    if (p->nhwc_plan) return conv_bwd_data_grouped_kernel(p->nhwc_plan, kind);
    *kind = p->path != CONV_BWD_PATH_GROUPED ? CONV_BWD_GROUPED_NONE
          : p->grouped_band                  ? CONV_BWD_GROUPED_TC_BAND
          : p->grouped_tc                    ? CONV_BWD_GROUPED_TC_TAPS
                                             : CONV_BWD_GROUPED_WARP_MMA;
    return CONV_BWD_OK;
}

conv_bwd_status conv_bwd_data_work(const conv_bwd_plan p, double *flop, double *bytes) {
    if (!p) return CONV_BWD_ERR_INVALID_ARG;
    if (flop) *flop = p->useful_flop;
    if (bytes) *bytes = p->algo_bytes;
    return CONV_BWD_OK;
}

conv_bwd_status conv_bwd_data_run(conv_bwd_plan p, const void *dy, const void *w, void *dx, void *stream) {
    NvtxRange range("conv_bwd_data_run");
    if (!p || !dy || !w || !dx) return CONV_BWD_ERR_INVALID_ARG;
    if (!p->has_device) return CONV_BWD_ERR_CUDA;
    const conv_bwd_desc &d = p->desc;
    const Geom &g = p->g;
    size_t es = elem_size(d.dtype);
    size_t ndy = (size_t)d.N * d.K * g.Ho * g.Wo * es, nw = (size_t)d.K * g.Cg * d.Y * d.X * es,
           ndx = (size_t)d.N * d.C * d.Hi * d.Wi * es;
    if (ranges_overlap(dy, ndy, dx, ndx) || ranges_overlap(w, nw, dx, ndx)) return CONV_BWD_ERR_INVALID_ARG;
    if (((uintptr_t)dy | (uintptr_t)w | (uintptr_t)dx) % es) return CONV_BWD_ERR_MISALIGNED;
    // Every alignment rule is checked before anything is launched.
    if ((p->path == CONV_BWD_PATH_TCGEN05 || p->path == CONV_BWD_PATH_GROUPED) &&
        ((uintptr_t)dy | (uintptr_t)w | (uintptr_t)dx) % 16)
        return CONV_BWD_ERR_MISALIGNED;
    if (p->path == CONV_BWD_PATH_TF32 && ((uintptr_t)dy | (uintptr_t)dx) % 16) return CONV_BWD_ERR_MISALIGNED;
    if (p->path == CONV_BWD_PATH_TF32 && !p->w_hi) return CONV_BWD_ERR_UNSUPPORTED;  // a plan without its scratch
    cudaStream_t s = (cudaStream_t)stream;
    std::lock_guard<std::mutex> lock(p->mu);

    if (p->nhwc_plan) {
        // dy [N][K][Ho*Wo] -> [N][Ho*Wo][K], (bf16) w [K][Cg][Y*X] -> [K][Y*X][Cg],
        // the NHWC/KYXC plan's kernels, dx [N][Hi*Wi][C] -> [N][C][Hi*Wi]; the
        // fp32 twin's filter split reads GKCYX itself
        auto transpose = d.dtype == CONV_BWD_F32 ? launch_transpose_b32 : launch_transpose_b16;
        if (transpose(dy, p->t_dy, d.N, d.K, (int64_t)g.Ho * g.Wo, p->num_sms, s) != cudaSuccess)
            return CONV_BWD_ERR_CUDA;
        if (p->t_w && transpose(w, p->t_w, d.K, g.Cg, (int64_t)d.Y * d.X, p->num_sms, s) != cudaSuccess)
            return CONV_BWD_ERR_CUDA;
        conv_bwd_status st = conv_bwd_data_run(p->nhwc_plan, p->t_dy, p->t_w ? p->t_w : w, p->t_dx, stream);
        if (st != CONV_BWD_OK) return st;
        if (transpose(p->t_dx, dx, d.N, (int64_t)d.Hi * d.Wi, d.C, p->num_sms, s) != cudaSuccess)
            return CONV_BWD_ERR_CUDA;
        return CONV_BWD_OK;
    }

    if (p->timing) {
        for (auto &e : p->ev)
            if (!e && cudaEventCreate(&e) != cudaSuccess) return CONV_BWD_ERR_CUDA;
    }
    p->fill_ran = false;
    const uint64_t all_w = g.sw >= 64 ? ~0ull : ((1ull << g.sw) - 1);
    if (p->path == CONV_BWD_PATH_GROUPED && p->grouped_band) {
        // every dx pixel is written by the kernel (classes without taps as zero)
        if (p->tmap_a_ptr != dy) {
            if (!encode_band_map(p, dy)) return CONV_BWD_ERR_CUDA;
            p->tmap_a_ptr = dy;
        }
        if (p->tmap_dx_ptr != dx) {
            if (!encode_band_dx_maps(p, dx)) return CONV_BWD_ERR_CUDA;
            p->tmap_dx_ptr = dx;
        }
        BandParams bp = p->band;
        bp.w = w; bp.dx = dx;
        bp.status = p->d_status; bp.wait_budget = p->wait_budget;
#ifdef CBD_PHASE_TIMES
        bp.phase_log = nullptr;
        if (p->d_phase &&
            cudaMemsetAsync(p->d_phase, 0, kPhaseLogCtas * kPhaseSlots * sizeof(unsigned long long), s) == cudaSuccess)
            bp.phase_log = p->d_phase;
#endif
        // each CTA keeps one 64-channel block; as many CTAs per block as fill the SMs
        const int nsm = std::max(1, p->num_sms);
        const int64_t per_cb = std::max<int64_t>(1, std::min<int64_t>(bp.units, nsm / bp.cblocks));
        if (p->timing) cudaEventRecord(p->ev[2], s);
        if (launch_tc_band(bp, (int)(per_cb * bp.cblocks), s) != cudaSuccess) return CONV_BWD_ERR_CUDA;
        if (p->timing) cudaEventRecord(p->ev[3], s);
        return CONV_BWD_OK;
    }
    if (p->path == CONV_BWD_PATH_GROUPED && p->grouped_tc && !p->classes.empty()) {
        // 64-channel group blocks: the kernel sees G' = C / 64 groups of 64
        // channels and builds each block's block-diagonal B from w itself
        if (p->tmap_a_ptr != dy) {
            if (!encode_a_maps(p, dy)) return CONV_BWD_ERR_CUDA;
            p->tmap_a_ptr = dy;
        }
        Geom fg = g;
        fg.G = g.C / 64;
        fg.Cg = fg.Kg = 64;
        if (p->timing) cudaEventRecord(p->ev[2], s);
        for (size_t c0 = 0; c0 < p->sched.size(); c0 += kMaxTcClasses) {
            TcParams tp;
            std::memset(&tp, 0, sizeof(tp));
            tp.dy = dy; tp.dx = dx; tp.w = w; tp.bd_cg = g.Cg;
            tp.status = p->d_status; tp.wait_budget = p->wait_budget;
            tp.g = fg;
#ifdef CBD_PHASE_TIMES
            if (p->d_phase && c0 == 0 &&
                cudaMemsetAsync(p->d_phase, 0, kPhaseLogCtas * kPhaseSlots * sizeof(unsigned long long), s) ==
                    cudaSuccess)
                tp.phase_log = p->d_phase;
#endif
            tp.n_tiles = 1;
            tp.kb_per_tap = 1;
            tp.im2col = 1;
            tp.fill = (c0 == 0 && p->any_uncovered) ? 1 : 0;
            tp.cov_h = p->cov_h;
            tp.cov_w = p->cov_w == all_w ? ~0ull : p->cov_w;
            const size_t nc = std::min<size_t>(kMaxTcClasses, p->sched.size() - c0);
            tp.num_classes = (int)nc;
            int64_t units = 0;  // tiles of one group block
            for (size_t i = 0; i < nc; ++i) {
                const int idx = p->sched[c0 + i];
                tp.cls[i] = p->classes[(size_t)idx];
                tp.cls[i].m_tiles = (tp.cls[i].M + 127) / 128;
                tp.cls[i].tile_begin = (int)units;
                units += tp.cls[i].m_tiles;
                tp.tmap_a[i] = p->tmap_a[(size_t)idx];
            }
            if (units * fg.G > 0x7fffffffLL) return CONV_BWD_ERR_UNSUPPORTED;
            tp.interleave = 1;
            for (size_t i = 1; i < nc; ++i) tp.interleave &= tp.cls[i].m_tiles == tp.cls[0].m_tiles;
            tp.total_tiles = (int)(units * fg.G);
            // each CTA keeps one group block; as many CTAs per block as fill the SMs
            const int nsm = std::max(1, p->num_sms);
            const int64_t per_gb = std::max<int64_t>(1, std::min<int64_t>(units, nsm / fg.G));
            if (launch_tc_grouped(tp, (int)(per_gb * fg.G), s) != cudaSuccess) return CONV_BWD_ERR_CUDA;
        }
        if (p->timing) cudaEventRecord(p->ev[3], s);
        return CONV_BWD_OK;
    }
    if (p->path == CONV_BWD_PATH_GROUPED && !p->grouped_tc) {
        GroupedParams gp;
        std::memset(&gp, 0, sizeof(gp));
        gp.dy = dy; gp.w = w; gp.dx = dx; gp.g = g;
        gp.gblocks = g.G / 8;
        // class of each row / column residue: the class t with t*d == (i + p) mod s
        for (int q = 0; q < g.sh; ++q) gp.row_class[q] = 0;
        for (int q = 0; q < g.sw; ++q) gp.col_class[q] = 0;
        for (int t = 0; t < g.YT; ++t) {
            const int taps = t < g.Y ? (g.Y - t + g.YT - 1) / g.YT : 0;
            const int res = (int)((((int64_t)t * g.dh - g.ph) % g.sh + g.sh) % g.sh);
            gp.row_class[res] = (taps << 16) | t;
        }
        for (int t = 0; t < g.XT; ++t) {
            const int taps = t < g.X ? (g.X - t + g.XT - 1) / g.XT : 0;
            const int res = (int)((((int64_t)t * g.dw - g.pw) % g.sw + g.sw) % g.sw);
            gp.col_class[res] = (taps << 16) | t;
        }
        if (p->timing) cudaEventRecord(p->ev[2], s);
        if (launch_grouped(gp, p->num_sms, s) != cudaSuccess) return CONV_BWD_ERR_CUDA;
        if (p->timing) cudaEventRecord(p->ev[3], s);
        return CONV_BWD_OK;
    }
    // the tensor-core kernels zero uncovered pixels themselves (epilogue warps,
    // during the first tile's main loop); other paths use the fill kernel
    if (p->any_uncovered &&
        ((p->path != CONV_BWD_PATH_TCGEN05 && p->path != CONV_BWD_PATH_TF32) || p->classes.empty())) {
        FillParams fp{};
        fp.dx = dx; fp.esize = (int)es; fp.layout = d.layout;
        fp.N = g.N; fp.C = g.C; fp.Hi = g.Hi; fp.Wi = g.Wi; fp.sh = g.sh; fp.sw = g.sw;
        fp.cov_h = p->cov_h; fp.cov_w = p->cov_w;
        if (fp.cov_w == (g.sw >= 64 ? ~0ull : ((1ull << g.sw) - 1))) fp.cov_w = ~0ull;  // every column written
        fp.vec16 = (d.layout == CONV_BWD_NHWC_KYXC && ((int64_t)d.C * (int64_t)es) % 16 == 0 &&
                    (uintptr_t)dx % 16 == 0) ? 1 : 0;
        if (p->timing) cudaEventRecord(p->ev[0], s);
        if (launch_fill(fp, p->num_sms, s) != cudaSuccess) return CONV_BWD_ERR_CUDA;
        if (p->timing) cudaEventRecord(p->ev[1], s);
        p->fill_ran = true;
    }
    if (p->classes.empty()) return CONV_BWD_OK;

    if (p->path == CONV_BWD_PATH_TF32) {
        if (p->tmap_w_ptr != p->w_hi) {
            if (!encode_tf32_w_maps(p)) return CONV_BWD_ERR_CUDA;
            p->tmap_w_ptr = p->w_hi;
        }
        if (p->tmap_a_ptr != dy) {
            if (!encode_a_maps(p, dy)) return CONV_BWD_ERR_CUDA;
            p->tmap_a_ptr = dy;
        }
        if (launch_tf32_split_w(static_cast<const float *>(w), p->w_hi, p->w_lo, g, p->w_gkcyx, p->num_sms, s) !=
            cudaSuccess)
            return CONV_BWD_ERR_CUDA;
        if (p->timing) cudaEventRecord(p->ev[2], s);  // the sub-GEMM kernel's time excludes the filter split
        for (size_t c0 = 0; c0 < p->sched.size(); c0 += kMaxTcClasses) {
            TcParams tp;
            std::memset(&tp, 0, sizeof(tp));
            tp.tmap_w = p->tmap_w;            // w_hi
            tp.tmap_w_half = p->tmap_w_half;  // w_lo
            tp.dy = dy; tp.dx = dx; tp.status = p->d_status; tp.wait_budget = p->wait_budget;
            tp.g = g;
            tp.n_tiles = (g.Cg + kTf32BN - 1) / kTf32BN;
            tp.kb_per_tap = (g.Kg + kTf32BK - 1) / kTf32BK;
            tp.im2col = 1;
            tp.fill = (c0 == 0 && p->any_uncovered) ? 1 : 0;
            tp.cov_h = p->cov_h;
            tp.cov_w = p->cov_w == all_w ? ~0ull : p->cov_w;
            const size_t nc = std::min<size_t>(kMaxTcClasses, p->sched.size() - c0);
            tp.num_classes = (int)nc;
            int64_t total = 0;
            for (size_t i = 0; i < nc; ++i) {
                const int idx = p->sched[c0 + i];
                tp.cls[i] = p->classes[(size_t)idx];
                tp.cls[i].tile_begin = (int)total;
                total += (int64_t)g.G * tp.cls[i].m_tiles * tp.n_tiles;
                tp.tmap_a[i] = p->tmap_a[(size_t)idx];
            }
            tp.total_tiles = (int)total;
            const int nsm = std::max(1, p->num_sms);
            int grid = (int)std::min<int64_t>(total, nsm);
            int64_t tail_units = 0;
            const bool split = tf32_tail_split(p, tp.cls, nc, total, tp.kb_per_tap, &tail_units);
            if (split) {
                tp.streamk = 1;
                tp.units_total = (int)std::min<int64_t>(tail_units, 0x7fffffff);
                grid = nsm;
            }
            if (launch_tf32(tp, grid, s) != cudaSuccess) return CONV_BWD_ERR_CUDA;
        }
        if (p->timing) cudaEventRecord(p->ev[3], s);
        return CONV_BWD_OK;
    }

    if (p->path == CONV_BWD_PATH_TCGEN05) {
        if (p->tmap_w_ptr != w) {
            if (!encode_w_map(p, w)) return CONV_BWD_ERR_CUDA;
            p->tmap_w_ptr = w;
        }
        if (p->im2col && p->tmap_a_ptr != dy) {
            if (!encode_a_maps(p, dy)) return CONV_BWD_ERR_CUDA;
            p->tmap_a_ptr = dy;
        }
        if (p->timing) cudaEventRecord(p->ev[2], s);
        std::vector<ClassDesc> lcls;
        std::vector<int> lmap;
        launch_classes(p, lcls, lmap);
        // at most kMaxTcClasses sub-GEMMs per launch (their maps travel as kernel parameters)
        for (size_t c0 = 0; c0 < lcls.size(); c0 += kMaxTcClasses) {
            TcParams tp;
            std::memset(&tp, 0, sizeof(tp));
            tp.tmap_w = p->tmap_w;
            tp.dy = dy; tp.dx = dx; tp.status = p->d_status; tp.wait_budget = p->wait_budget;
            tp.g = g;
            tp.n_tiles = (g.Cg + p->bn - 1) / p->bn;
            tp.kb_per_tap = (g.Kg + 63) / 64;
            tp.im2col = p->im2col ? 1 : 0;
            tp.a_plain = p->a_plain ? 1 : 0;
#ifdef CBD_PHASE_TIMES
            if (p->d_phase && c0 == 0 &&
                cudaMemsetAsync(p->d_phase, 0, kPhaseLogCtas * kPhaseSlots * sizeof(unsigned long long), s) ==
                    cudaSuccess)
                tp.phase_log = p->d_phase;
#endif
            tp.fill = (c0 == 0 && p->any_uncovered) ? 1 : 0;  // first launch zeroes the uncovered pixels
            if (const char *f = env("CONVBWD_DEBUG_RASTER_M")) tp.raster_m = f[0] == '1' ? 1 : 0;
            tp.cov_h = p->cov_h;
            tp.cov_w = p->cov_w == all_w ? ~0ull : p->cov_w;
            const size_t nc = std::min<size_t>(kMaxTcClasses, lcls.size() - c0);
            tp.num_classes = (int)nc;
            int64_t total = 0;
            int64_t units = 0;
            for (size_t i = 0; i < nc; ++i) {
                const int idx = lmap[c0 + i];
                tp.cls[i] = lcls[c0 + i];
                tp.cls[i].tile_begin = (int)total;
                tp.cls[i].unit_begin = (int)units;
                const int64_t tiles_c = (int64_t)g.G * tp.cls[i].m_tiles * tp.n_tiles;
                total += tiles_c;
                units += tiles_c * tp.cls[i].taps_y * tp.cls[i].taps_x * tp.kb_per_tap;
                if (p->im2col) tp.tmap_a[i] = p->tmap_a[(size_t)idx];
            }
            tp.total_tiles = (int)total;
            tp.units_total = (int)std::min<int64_t>(units, 0x7fffffff);
            if (p->two_sm && p->splitk > 1) {
                // one unit per SM pair: split q of tile t on pair t * S + q
                tp.splitk = p->splitk;
                tp.partials = p->d_ws;
                tp.flags = p->d_ws_flags;
                p->epoch = p->epoch >= 0x7ffffffe ? 1 : p->epoch + 1;
                tp.epoch = p->epoch;
                if (launch_tc2(tp, p->bn, (int)(2 * total * p->splitk), s) != cudaSuccess) return CONV_BWD_ERR_CUDA;
                continue;
            }
            if (p->two_sm) {
                const int maxp = tc2_max_pairs(p->num_sms);
                int pairs = (int)std::min<int64_t>(total, maxp);
                // Stream-K (equal unit ranges per pair, partial tiles through the
                // workspace) is opt-in: on GB300 the partial-tile traffic costs about
                // what the better balance saves on the shapes measured here.
                bool sk = false;
                if (const char *f = env("CONVBWD_DEBUG_STREAMK"))
                    sk = p->d_partials && f[0] == '1' && units < 0x7fffffff && maxp <= p->max_pairs && p->bn <= 256;
                if (sk) {
                    // every worker gets at least one unit: a worker without units would
                    // never raise the flag its tile's owner waits for
                    pairs = (int)std::min<int64_t>(maxp, units);
                    tp.streamk = 1;
                    tp.partials = p->d_partials;
                    tp.flags = p->d_flags;
                    p->epoch = p->epoch >= 0x7ffffffe ? 1 : p->epoch + 1;
                    tp.epoch = p->epoch;
                }
                if (launch_tc2(tp, p->bn, 2 * pairs, s) != cudaSuccess) return CONV_BWD_ERR_CUDA;
                continue;
            }
            int grid = (int)std::min<int64_t>(total, p->num_sms);
            if (const char *f = env("CONVBWD_DEBUG_GRID")) grid = std::max(1, std::min(grid, std::atoi(f)));
            if (launch_tc(tp, p->bn, grid, s) != cudaSuccess) return CONV_BWD_ERR_CUDA;
        }
        if (p->timing) cudaEventRecord(p->ev[3], s);
        return CONV_BWD_OK;
    }

    SimtParams sp;
    std::memset(&sp, 0, sizeof(sp));
    sp.g = g; sp.st = p->st; sp.dy = dy; sp.w = w; sp.dx = dx;
    sp.num_classes = (int)p->sched.size();
    sp.bn = p->bn;
    sp.n_tiles = (g.Cg + sp.bn - 1) / sp.bn;
    int64_t total = 0;
    for (size_t i = 0; i < p->sched.size(); ++i) {
        sp.cls[i] = p->classes[(size_t)p->sched[i]];
        total += (int64_t)g.G * sp.cls[i].m_tiles * sp.n_tiles;
    }
    sp.total_tiles = (int)total;
    if (p->timing) cudaEventRecord(p->ev[2], s);
    if (launch_simt(sp, d.dtype, s) != cudaSuccess) return CONV_BWD_ERR_CUDA;
    if (p->timing) cudaEventRecord(p->ev[3], s);
    return CONV_BWD_OK;
}

conv_bwd_status conv_bwd_data_run_host(conv_bwd_plan p, const void *dy_h, const void *w_h, void *dx_h, void *dy_d,
                                       void *w_d, void *dx_d, void *stream) {
    NvtxRange range("conv_bwd_data_run_host");
    if (!p || !dy_h || !w_h || !dx_h || !dy_d || !w_d || !dx_d) return CONV_BWD_ERR_INVALID_ARG;
    if (!p->has_device) return CONV_BWD_ERR_CUDA;
    const conv_bwd_desc &d = p->desc;
    size_t es = elem_size(d.dtype);
    size_t ndy = (size_t)d.N * d.K * p->g.Ho * p->g.Wo * es, nw = (size_t)d.K * p->g.Cg * d.Y * d.X * es,
           ndx = (size_t)d.N * d.C * d.Hi * d.Wi * es;
    cudaStream_t s = (cudaStream_t)stream;
    int chunks;
    {
        std::lock_guard<std::mutex> lock(p->mu);
        chunks = host_chunks(p, ndy, ndx);
    }
    if (chunks <= 1) {
        if (cudaMemcpyAsync(dy_d, dy_h, ndy, cudaMemcpyHostToDevice, s) != cudaSuccess) return CONV_BWD_ERR_CUDA;
        if (cudaMemcpyAsync(w_d, w_h, nw, cudaMemcpyHostToDevice, s) != cudaSuccess) return CONV_BWD_ERR_CUDA;
        conv_bwd_status st = conv_bwd_data_run(p, dy_d, w_d, dx_d, stream);
        if (st != CONV_BWD_OK) return st;
        if (cudaMemcpyAsync(dx_h, dx_d, ndx, cudaMemcpyDeviceToHost, s) != cudaSuccess) return CONV_BWD_ERR_CUDA;
        return CONV_BWD_OK;
    }
    // Pipelined over batch chunks (N is the outermost dimension of dy and dx in
    // both layouts): the copy stream brings w and then dy chunk by chunk, the
    // caller's stream runs chunk i once its dy is in, the second copy stream
    // returns dx chunk i once it is computed; the caller's stream finally waits
    // for the last copy, so everything stays ordered on `stream`.
    std::lock_guard<std::mutex> lock(p->mu);
    cudaEvent_t *ev = p->hev.data();
    const size_t dy_img = ndy / d.N, dx_img = ndx / d.N;
    auto n_of = [&](int i) { return i + 1 < chunks ? (int64_t)p->chunk_n : d.N - (int64_t)(chunks - 1) * p->chunk_n; };
    bool ok = cudaEventRecord(ev[0], s) == cudaSuccess && cudaStreamWaitEvent(p->h2d, ev[0], 0) == cudaSuccess &&
              cudaStreamWaitEvent(p->d2h, ev[0], 0) == cudaSuccess &&
              cudaMemcpyAsync(w_d, w_h, nw, cudaMemcpyHostToDevice, p->h2d) == cudaSuccess;
    for (int i = 0; ok && i < chunks; ++i) {
        const size_t off = (size_t)i * p->chunk_n * dy_img;
        ok = cudaMemcpyAsync(static_cast<char *>(dy_d) + off, static_cast<const char *>(dy_h) + off,
                             (size_t)n_of(i) * dy_img, cudaMemcpyHostToDevice, p->h2d) == cudaSuccess &&
             cudaEventRecord(ev[2 + 2 * i], p->h2d) == cudaSuccess;
    }
    for (int i = 0; ok && i < chunks; ++i) {
        conv_bwd_plan_s *cp = (i + 1 < chunks || !p->chunk_plan[1]) ? p->chunk_plan[0] : p->chunk_plan[1];
        ok = cudaStreamWaitEvent(s, ev[2 + 2 * i], 0) == cudaSuccess;
        if (!ok) break;
        conv_bwd_status st = conv_bwd_data_run(cp, static_cast<char *>(dy_d) + (size_t)i * p->chunk_n * dy_img, w_d,
                                               static_cast<char *>(dx_d) + (size_t)i * p->chunk_n * dx_img, stream);
        if (st != CONV_BWD_OK) return st;
        ok = cudaEventRecord(ev[3 + 2 * i], s) == cudaSuccess;
    }
    for (int i = 0; ok && i < chunks; ++i) {
        const size_t off = (size_t)i * p->chunk_n * dx_img;
        ok = cudaStreamWaitEvent(p->d2h, ev[3 + 2 * i], 0) == cudaSuccess &&
             cudaMemcpyAsync(static_cast<char *>(dx_h) + off, static_cast<const char *>(dx_d) + off,
                             (size_t)n_of(i) * dx_img, cudaMemcpyDeviceToHost, p->d2h) == cudaSuccess;
    }
    ok = ok && cudaEventRecord(ev[1], p->d2h) == cudaSuccess && cudaStreamWaitEvent(s, ev[1], 0) == cudaSuccess;
    return ok ? CONV_BWD_OK : CONV_BWD_ERR_CUDA;
}

conv_bwd_status conv_bwd_data_run_forward(conv_bwd_plan p, const void *x, const void *w, void *y, void *stream) {
    NvtxRange range("conv_bwd_data_run_forward");
    if (!p || !x || !w || !y) return CONV_BWD_ERR_INVALID_ARG;
    if (!fwd_supported(p)) return CONV_BWD_ERR_UNSUPPORTED;
    if (!p->has_device || !p->d_status) return CONV_BWD_ERR_CUDA;
    const conv_bwd_desc &d = p->desc;
    const Geom &g = p->g;
    const size_t nx = (size_t)d.N * d.C * d.Hi * d.Wi * 2, nw = (size_t)d.K * g.Cg * d.Y * d.X * 2,
                 ny = (size_t)d.N * d.K * g.Ho * g.Wo * 2;
    if (ranges_overlap(x, nx, y, ny) || ranges_overlap(w, nw, y, ny)) return CONV_BWD_ERR_INVALID_ARG;
    if (((uintptr_t)x | (uintptr_t)w | (uintptr_t)y) % 16) return CONV_BWD_ERR_MISALIGNED;
    std::lock_guard<std::mutex> lock(p->mu);
    if (p->fwd_x_ptr != x || p->fwd_w_ptr != w) {
        if (!encode_fwd_maps(p, x, w)) return CONV_BWD_ERR_CUDA;
        p->fwd_x_ptr = x;
        p->fwd_w_ptr = w;
    }
    FwdParams fp;
    std::memset(&fp, 0, sizeof(fp));
    fp.tmap_x = p->fwd_tmap_x;
    fp.tmap_w = p->fwd_tmap_w;
    fp.y = y;
    fp.status = p->d_status;
    fp.wait_budget = p->wait_budget;
    fp.g = g;
    const int bn = fwd_bn(g);
    const int64_t M = (int64_t)d.N * g.Ho * g.Wo;
    fp.m_tiles = (int)((M + 127) / 128);
    fp.n_tiles = (g.Kg + bn - 1) / bn;
    fp.kb_per_tap = (g.Cg + 63) / 64;
    const int64_t total = (int64_t)fp.m_tiles * fp.n_tiles * g.G;
    if (total >= (1LL << 31)) return CONV_BWD_ERR_UNSUPPORTED;
    fp.total_tiles = (int)total;
    const int grid = (int)std::min<int64_t>(total, p->num_sms);
    if (launch_fwd(fp, bn, grid, (cudaStream_t)stream) != cudaSuccess) return CONV_BWD_ERR_CUDA;
    return CONV_BWD_OK;
}

conv_bwd_status conv_bwd_data_get_status(conv_bwd_plan p, void *stream, int32_t *detail) {
    if (!p) return CONV_BWD_ERR_INVALID_ARG;
    if (detail) *detail = 0;
    if (!p->has_device) return CONV_BWD_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    int32_t h = 0;
    if (cudaMemcpyAsync(&h, p->d_status, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess) return CONV_BWD_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return CONV_BWD_ERR_CUDA;
    if (h == 0) return CONV_BWD_OK;
    if (detail) *detail = h;
    cudaMemsetAsync(p->d_status, 0, 16, s);
    cudaStreamSynchronize(s);
    return (h & 0xF00) == 0x200 ? CONV_BWD_ERR_DEVICE_FAULT : CONV_BWD_ERR_DEVICE_TIMEOUT;
}

conv_bwd_status conv_bwd_data_set_timing(conv_bwd_plan p, int32_t enable) {
    if (!p) return CONV_BWD_ERR_INVALID_ARG;
    p->timing = enable != 0;
    if (p->nhwc_plan) conv_bwd_data_set_timing(p->nhwc_plan, enable);
    return CONV_BWD_OK;
}

conv_bwd_status conv_bwd_data_last_timing(conv_bwd_plan p, float *fill_ms, float *gemm_ms) {
    if (p && p->nhwc_plan) return conv_bwd_data_last_timing(p->nhwc_plan, fill_ms, gemm_ms);  // its kernels
    if (!p || !p->timing || !p->ev[3]) return CONV_BWD_ERR_INVALID_ARG;
    float f = 0.f, m = 0.f;
    if (p->fill_ran) {
        if (cudaEventSynchronize(p->ev[1]) != cudaSuccess) return CONV_BWD_ERR_CUDA;
        cudaEventElapsedTime(&f, p->ev[0], p->ev[1]);
    }
    if (!p->classes.empty()) {
        if (cudaEventSynchronize(p->ev[3]) != cudaSuccess) return CONV_BWD_ERR_CUDA;
        cudaEventElapsedTime(&m, p->ev[2], p->ev[3]);
    }
    if (fill_ms) *fill_ms = f;
    if (gemm_ms) *gemm_ms = m;
    return CONV_BWD_OK;
}

conv_bwd_status conv_bwd_data_selftest_wait_timeout(void *stream, int64_t budget_cycles, int32_t *observed) {
    if (!observed || budget_cycles <= 0) return CONV_BWD_ERR_INVALID_ARG;
    int32_t *d = nullptr;
    if (cudaMalloc(&d, 16) != cudaSuccess) return CONV_BWD_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    conv_bwd_status st = CONV_BWD_OK;
    int32_t h = -1;
    if (cudaMemsetAsync(d, 0, 16, s) != cudaSuccess || launch_selftest_wait(d, budget_cycles, s) != cudaSuccess ||
        cudaMemcpyAsync(&h, d, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
        st = CONV_BWD_ERR_CUDA;
    cudaFree(d);
    if (st != CONV_BWD_OK) return st;
    *observed = (h == kDevTimeoutSelftest) ? CONV_BWD_ERR_DEVICE_TIMEOUT : (h == 0 ? CONV_BWD_OK : CONV_BWD_ERR_DEVICE_FAULT);
    return CONV_BWD_OK;
}

}  // extern "C"

#ifdef CBD_PHASE_TIMES
// Instrumented build only: copy the last tensor-core launch's per-CTA timeline
// (kPhaseSlots globaltimer stamps per CTA, 0 where a slot was not reached) into
// `out` (n_ctas rows); synchronises the device.
extern "C" conv_bwd_status conv_bwd_data_debug_phase_log(conv_bwd_plan p, unsigned long long *out, int32_t n_ctas) {
    if (!p || !out || n_ctas <= 0 || n_ctas > kPhaseLogCtas || !p->d_phase) return CONV_BWD_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return CONV_BWD_ERR_CUDA;
    if (cudaMemcpy(out, p->d_phase, (size_t)n_ctas * kPhaseSlots * sizeof(unsigned long long),
                   cudaMemcpyDeviceToHost) != cudaSuccess)
        return CONV_BWD_ERR_CUDA;
    return CONV_BWD_OK;
}
#endif

namespace cbd {

// Host-only plan (no device allocation) whose kernels will record their
// status in `status`, device memory the caller keeps alive.  Used by the
// no-allocation entry point; the plan is freed with conv_bwd_data_destroy,
// which then leaves `status` alone.
conv_bwd_status plan_create_borrowed_status(const conv_bwd_desc *desc, int32_t *status, conv_bwd_plan *out) {
    conv_bwd_status st = create_impl(desc, out, false);
    if (st != CONV_BWD_OK) return st;
    conv_bwd_plan p = *out;
    if (p->device < 0) {
        conv_bwd_data_destroy(p);
        *out = nullptr;
        return CONV_BWD_ERR_CUDA;
    }
    p->d_status = status;
    p->owns_status = false;
    p->has_device = true;
    return CONV_BWD_OK;
}

int32_t plan_path_of(conv_bwd_plan p) { return p ? p->path : -1; }

}  // namespace cbd
