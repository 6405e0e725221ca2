/*
 * conv_bwd_data.h -- C ABI of the GB300 (sm_103a) convolution backward-data
 * library: dx = dgrad(dy, w) as a stride-decomposed implicit GEMM.
 *
 * What the library computes.  The gradient of a forward 2-D
 * cross-correlation with respect to its input: the grad_input result of
 * `torch.aten.convolution_backward` with output_mask [true, false, false]
 * (page "Non-unit stride input backward different input and dispatches
 * between BOO and Fusilli", torch-IR input):
 *
 *   dx[n, c, hi, wi] = sum over k in group(c), y < Y, x < X, ho, wo with
 *                      ho*sh - ph + y*dh == hi and wo*sw - pw + x*dw == wi
 *                      of dy[n, k, ho, wo] * w[k, c mod (C/G), y, x]
 *
 * dx is fully overwritten; pixels that no filter tap reaches become +0
 * (the same torch-IR overwrites the destination tensor's contents).
 *
 * How.  For stride > 1 the problem is split into one sub-GEMM per filter-tap
 * residue class instead of zero-inserting dy into a dilated tensor: the
 * "v4r1 backward_data" multi-kernel strategy (pages "Backward data", rocMLIR
 * pull request 246, and "[igemm_dynamic] v4r1 bwd dynamic kernel", MIOpen
 * pull request 272).  Per spatial dim with stride s, dilation d, pad p:
 * g = gcd(s, d), YTilde = s / g, and class t in [0, YTilde) owns taps
 * y = t + YTilde*j.  Non-empty classes get consecutive gemmIds 0..n-1 (the
 * review of pull request 246 asks for consecutive gemmId).  The caller never
 * passes kernel ids: the library rebuilds every per-class argument itself
 * (same review), and one run() launches all classes.
 *
 * Memory ownership.  The caller owns dy, w, dx and the stream (any
 * allocator; PyTorch in the bundled binding).  The library owns the plan
 * (host memory) and one 16-byte device status word per plan; fp32 plans on
 * the tensor-core path also own two fp32 copies of the filter (its hi and lo
 * parts), all allocated by conv_bwd_data_create when a CUDA device is present
 * (plans created with the opt-in stream-K override below also own its
 * scratch, 256 KB per SM pair).  conv_bwd_data_run
 * allocates nothing, never synchronises and is ordered on the given stream.
 *
 * Layouts (all tensors dense, row-major in the order written):
 *   CONV_BWD_NCHW_GKCYX: dy [N][K][Ho][Wo], w [K][C/G][Y][X] (= [G][K/G][C/G][Y][X]),
 *                        dx [N][C][Hi][Wi]
 *   CONV_BWD_NHWC_KYXC:  dy [N][Ho][Wo][K], w [K][Y][X][C/G], dx [N][Hi][Wi][C]
 * Group gi owns input channels [gi*C/G, (gi+1)*C/G) and output channels
 * [gi*K/G, (gi+1)*K/G).  Ho = (Hi + 2*ph - dh*(Y-1) - 1)/sh + 1, likewise Wo.
 * Padding is symmetric per dimension.
 *
 * Numerics.  fp32 tensors: fp32 FFMA on CUDA cores; large problems (path
 * CONV_BWD_PATH_TF32) run on the tensor cores with each operand split as
 * x = hi + lo (hi = x rounded to a 10-bit mantissa, lo = x - hi exactly) and
 * three TF32 products hi*hi + hi*lo + lo*hi accumulated in fp32 per term,
 * which keeps each product within about 2^-20 of the exact one (plain TF32
 * would be 2^-10 and miss the fp32 tolerance).  bf16 tensors:
 * bf16 x bf16 products accumulated in fp32 (tensor cores for the NHWC path),
 * one round-to-nearest-even conversion to bf16 at the end (the `arith.extf`,
 * `arith.mulf`/`arith.addf` in f32 and `arith.truncf` ops of the BOO IR on
 * the page above).  The summation order is unspecified.
 *
 * Errors.  Every call returns a conv_bwd_status; nothing throws across the
 * ABI.  Device-side problems (a bounded wait that ran out, an index check
 * that failed) are recorded in the plan's status word and reported by
 * conv_bwd_data_get_status; kernels never trap.
 */
#ifndef CONV_BWD_DATA_H
#define CONV_BWD_DATA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CONV_BWD_OK = 0,
    CONV_BWD_ERR_INVALID_ARG = 1,   /* bad descriptor value, null or overlapping pointer */
    CONV_BWD_ERR_UNSUPPORTED = 2,   /* valid problem outside what this library implements */
    CONV_BWD_ERR_MISALIGNED = 3,    /* pointer or channel stride breaks a 16-byte rule of the path */
    CONV_BWD_ERR_CUDA = 4,          /* a CUDA runtime call failed (or no device) */
    CONV_BWD_ERR_DEVICE_TIMEOUT = 5,/* a bounded device-side wait ran out */
    CONV_BWD_ERR_DEVICE_FAULT = 6   /* a device-side index/consistency check failed */
} conv_bwd_status;

typedef enum { CONV_BWD_F32 = 0, CONV_BWD_BF16 = 1 } conv_bwd_dtype;
typedef enum { CONV_BWD_NCHW_GKCYX = 0, CONV_BWD_NHWC_KYXC = 1 } conv_bwd_layout;

/* Problem descriptor; the fields mirror the driver flags of the tested
 * command lines in "Backward data" (-batchsize -in_channels -out_channels
 * -in_h -in_w -fil_h -fil_w --padding_* --conv_stride_* --dilation_*
 * --groupsize and the layouts).  C and K are totals over all groups. */
typedef struct {
    int64_t N, C, K, Hi, Wi, Y, X;
    int32_t pad_h, pad_w, stride_h, stride_w, dil_h, dil_w, groups;
    int32_t layout; /* conv_bwd_layout */
    int32_t dtype;  /* conv_bwd_dtype */
} conv_bwd_desc;

typedef struct conv_bwd_plan_s *conv_bwd_plan;

/* Which kernel family runs the sub-GEMMs of a plan. */
typedef enum {
    CONV_BWD_PATH_TCGEN05 = 0, /* bf16: persistent tcgen05/TMEM implicit GEMM */
    CONV_BWD_PATH_SIMT = 1,    /* fp32 (or bf16 fallback): CUDA-core tiled implicit GEMM */
    CONV_BWD_PATH_GROUPED = 2, /* bf16 narrow groups, C/G = K/G in {8, 16, 32}: one of three memory-bound
                                  kernels, see conv_bwd_data_grouped_kernel */
    CONV_BWD_PATH_TF32 = 3     /* fp32 NHWC/KYXC with >= 1e9 useful FLOP, K, C, C/G, K/G multiples of 4
                                  (K/G of 32 when G > 1): tcgen05 kind::tf32 with a three-term split */
} conv_bwd_path;
/* The tensor-core and narrow-group kernels read NHWC/KYXC.  An NCHW/GKCYX
 * plan whose NHWC/KYXC twin takes one of them gets plan-owned scratch (dy and
 * dx in NHWC, plus w in KYXC for bf16, allocated by create) and each run
 * transposes dy (and the bf16 w) into it, runs the twin's kernels and
 * transposes dx back (path() reports the twin's path with 3 more launches for
 * bf16, 2 for fp32, whose filter split reads GKCYX directly). */

/* Planner overrides, read at create (for tests and measurements; unset in
 * normal use):
 *   CONVBWD_DEBUG_PATH=simt          CUDA-core path for every plan
 *   CONVBWD_DEBUG_PATH=tf32          fp32 tensor-core path whatever the problem size
 *   CONVBWD_DEBUG_NOIM2COL=1         cp.async A producer instead of TMA im2col
 *   CONVBWD_DEBUG_2SM=1 / _NO2SM=1   SM-pair kernel for C/G >= 128, also where the planner's
 *                                    estimate would pick 1-SM 128 x 128 tiles / never
 *   CONVBWD_DEBUG_BN=128|256|512     tile width
 *   CONVBWD_DEBUG_STREAMK=1|0        stream-K schedule on the SM-pair kernel (its scratch is
 *                                    allocated only then); on the fp32 tensor-core path, the
 *                                    tail split always / never
 *   CONVBWD_DEBUG_NO_WSPLIT=1        fp32 tensor-core plans behave as if the split filter could
 *                                    not be allocated (CUDA-core fallback)
 *   CONVBWD_DEBUG_A=plain            plain-matrix A specialisation where it applies (see below)
 *   CONVBWD_DEBUG_SPLITK=S           split-K over S SM pairs per tile where all units fit one wave
 *   CONVBWD_DEBUG_GROUPED=band|mma|tc  narrow-group kernel (see conv_bwd_data_grouped_kernel) where
 *                                    it applies
 *   CONVBWD_DEBUG_RASTER_M=1         tiles walk m-blocks first
 *   CONVBWD_DEBUG_GRID=n             cap the 1-SM kernel's grid
 *   CONVBWD_DEBUG_L2PROMO=0|1       TMA L2 promotion none / 128 B (default 256 B)
 *   CONVBWD_DEBUG_WAIT_SECONDS=s     budget of every bounded device wait (default 2)
 *   CONVBWD_DEBUG_HOST_CHUNKS=n      batch chunks of the pipelined run_host (default 4)
 *   CONVBWD_DEBUG_NO_TRANSPOSE=1     NCHW plans stay on the CUDA-core path */

/* Validate the descriptor and plan on the host: forward output size, tilde
 * factors, non-empty sub-GEMM list (consecutive gemmIds), coverage of dx,
 * kernel path and tile schedule.  If a CUDA device is visible, also
 * allocates the plan's device status word on the current device (run() must
 * then be called with that device current).  Without a device the plan is
 * still created (so the planner can be queried) and run() returns
 * CONV_BWD_ERR_CUDA.  bf16 NCHW/GKCYX plans on a tensor-core path also
 * allocate the NHWC/KYXC scratch (if that fails they keep the CUDA-core
 * path).  *out is set to NULL on failure.
 * Errors: INVALID_ARG (non-positive sizes, pad < 0, stride/dilation < 1,
 * C or K not divisible by groups, empty forward output, unknown enum),
 * UNSUPPORTED (stride > 64, more than 2^31-1 elements in a tensor, bf16 in a
 * layout/shape no kernel covers), CUDA (device allocation failed). */
conv_bwd_status conv_bwd_data_create(const conv_bwd_desc *desc, conv_bwd_plan *out);

/* Free the plan and its device status word.  NULL is accepted. */
conv_bwd_status conv_bwd_data_destroy(conv_bwd_plan plan);

/* Forward output size (the spatial extent of dy). */
conv_bwd_status conv_bwd_data_out_dims(const conv_bwd_plan plan, int64_t *Ho, int64_t *Wo);

/* Number of non-empty sub-GEMMs; their gemmIds are 0..n-1. */
conv_bwd_status conv_bwd_data_num_subgemms(const conv_bwd_plan plan, int32_t *n);

/* Sub-GEMM `id`: its residue classes (ty, tx), its GEMM sizes per group
 * (M = N * rows of the class, N = C/G, K = K/G * taps) and its tap counts.
 * Any output pointer may be NULL.  INVALID_ARG for an id out of range. */
conv_bwd_status conv_bwd_data_subgemm_info(const conv_bwd_plan plan, int32_t id, int32_t *ty, int32_t *tx,
                                           int64_t *M, int64_t *N, int64_t *K, int32_t *taps_y,
                                           int32_t *taps_x);

/* Coverage of dx: row_mask[hi] (Hi bytes) and col_mask[wi] (Wi bytes) are
 * set to 1 where some sub-GEMM writes that row/column, else 0.  A pixel is
 * written by a sub-GEMM iff both its row and its column are covered; every
 * other pixel is zeroed by the fill kernel.  Either pointer may be NULL. */
conv_bwd_status conv_bwd_data_coverage(const conv_bwd_plan plan, uint8_t *row_mask, uint8_t *col_mask);

/* Kernel path chosen by the planner (conv_bwd_path) and the number of
 * kernel launches one run() makes (fill + sub-GEMM kernel; the fp32
 * tensor-core path counts its filter split and kernel, not the optional tile
 * zeroing; NCHW plans add their transposes). */
conv_bwd_status conv_bwd_data_path(const conv_bwd_plan plan, int32_t *path, int32_t *launches_per_run);

/* Forward convolution with the plan's geometry, y = conv(x, w): the operator
 * whose adjoint run() computes (pages "Backward data" -- the forward kernels the
 * backward-data lowering is paired with -- and "Non-unit stride input backward
 * different input and dispatches between BOO and Fusilli", whose torch-IR input
 * is the backward of aten.convolution):
 *   y[n, ho, wo, k] = sum over c in group(k), y', x' of
 *                     x[n, ho*sh - ph + y'*dh, wo*sw - pw + x'*dw, c] * w[k, y', x', c mod Cg]
 * x has dx's shape ([N][Hi][Wi][C]), y has dy's shape ([N][Ho][Wo][K]), w is
 * run()'s filter; all bf16, caller-owned device pointers, 16-byte aligned; y
 * is fully overwritten (fp32 accumulation, one RNE rounding per element).
 * Supported: bf16 NHWC/KYXC plans with C/G and K/G multiples of 8, C/G a
 * multiple of 64 when G > 1, strides <= 8, (X-1)*dw and (Y-1)*dh <= 127 and
 * the im2col bounding box of x within [-128, 127] per dimension; other plans
 * return CONV_BWD_ERR_UNSUPPORTED before anything is launched.  Stream-ordered
 * like run(), sharing its status word (read it with get_status).  Errors:
 * INVALID_ARG (NULL or overlapping y), MISALIGNED, CUDA. */
conv_bwd_status conv_bwd_data_run_forward(conv_bwd_plan plan, const void *x, const void *w, void *y, void *stream);

/* Output tile of the plan's GEMM kernel: rows (M) and columns (C/G) per tile,
 * and the number of SMs that share one tile (2 for the SM-pair tensor-core
 * kernel, else 1).  The narrow-group tcgen05 kernels report 128 x 64 (one
 * 64-channel block), the warp-MMA one 0 x 0 (it has no tiles).  Any output
 * pointer may be NULL. */
conv_bwd_status conv_bwd_data_tile(const conv_bwd_plan plan, int32_t *tile_m, int32_t *tile_n, int32_t *sms_per_tile);

/* K splits of the plan's SM-pair tensor-core schedule: 1 = every 256-row tile
 * computed whole by one SM pair; S > 1 = split-K with a reduce-scatter: each
 * 256 x 512 (or x 256) tile is shared by S SM pairs, each accumulating 1/S of
 * its k-blocks, which then exchange fp32 partials through a plan-owned
 * workspace (allocated by create) so that each pair adds and stores 1/S of
 * the tile's columns.  Used where the tiles alone cannot fill the GPU; all
 * tiles then run in one wave.  Other paths report 1.  INVALID_ARG for NULL. */
conv_bwd_status conv_bwd_data_k_splits(const conv_bwd_plan plan, int32_t *k_splits);

/* How the plan's GEMM kernel loads its A operand (dy rows):
 *   CONV_BWD_A_IM2COL  TMA im2col loads, one map per residue class (the dynamic
 *                      kernel: any shape, the tap as the im2col offset);
 *   CONV_BWD_A_PLAIN   2-D tiled TMA loads of dy as the matrix {N*Ho*Wo, K}: the
 *                      SM-pair kernel's compile-time specialisation for plans whose
 *                      every class has one tap and covers all of dy's pixels in
 *                      order (1x1 filters, the 1x2 stride-(1,2) layer); selected
 *                      by CONVBWD_DEBUG_A=plain at create.  It plays the "static"
 *                      kernel against the dynamic one of "[igemm_dynamic] v4r1 bwd
 *                      dynamic kernel" (dynamic within 10% of static);
 *   CONV_BWD_A_GATHER  per-thread gathers (cp.async producers, CUDA cores, the
 *                      warp-MMA narrow-group kernel);
 *   CONV_BWD_A_BAND    tiled TMA loads of a band of dy rows (4 output rows plus
 *                      the filter's row reach, 32 pixels, 64 channels), one per
 *                      distinct column offset of the taps, read by every tap
 *                      (the banded narrow-group kernel).
 * INVALID_ARG for a NULL argument. */
typedef enum { CONV_BWD_A_IM2COL = 0, CONV_BWD_A_PLAIN = 1, CONV_BWD_A_GATHER = 2, CONV_BWD_A_BAND = 3 } conv_bwd_a_mode;
conv_bwd_status conv_bwd_data_a_operand(const conv_bwd_plan plan, int32_t *a_mode);

/* Which narrow-group kernel a CONV_BWD_PATH_GROUPED plan runs (bf16 NHWC/KYXC,
 * C/G = K/G; each writes every dx pixel itself, one launch):
 *   CONV_BWD_GROUPED_TC_BAND   (default where it applies: C/G in {8, 16, 32},
 *                              C % 64 == 0, strides 1 or 2, at most 32 filter
 *                              taps, the staged band within shared memory)
 *                              tcgen05 with the groups of each 64-channel block
 *                              folded into a block-diagonal B whose all-zero
 *                              16 x 16 blocks are skipped; each band of dy (4
 *                              output rows x 32 columns of every residue
 *                              class) is staged once and read by every tap;
 *   CONV_BWD_GROUPED_WARP_MMA  (C/G in {8, 16}, G % 8 == 0) warp-level MMA on
 *                              CUDA-core-staged dy rows;
 *   CONV_BWD_GROUPED_TC_TAPS   (C/G in {8, 16, 32}, C % 64 == 0, <= 12 taps)
 *                              tcgen05 with one TMA im2col load of dy per tap;
 *   CONV_BWD_GROUPED_NONE      the plan is not on the narrow-group path.
 * INVALID_ARG for a NULL argument. */
typedef enum {
    CONV_BWD_GROUPED_NONE = 0,
    CONV_BWD_GROUPED_WARP_MMA = 1,
    CONV_BWD_GROUPED_TC_TAPS = 2,
    CONV_BWD_GROUPED_TC_BAND = 3
} conv_bwd_grouped_kernel_kind;
conv_bwd_status conv_bwd_data_grouped_kernel(const conv_bwd_plan plan, int32_t *kind);

/* Useful work: 2 * N * K * (C/G) * Th * Tw floating-point operations, where
 * Th = #{(ho, y): 0 <= ho*sh - ph + y*dh < Hi} counts only taps that land
 * inside dx (likewise Tw).  Also the algorithmic bytes: dy, w and dx each
 * moved once. */
conv_bwd_status conv_bwd_data_work(const conv_bwd_plan plan, double *useful_flop, double *algo_bytes);

/* Compute dx from dy and w on `stream` (a cudaStream_t; NULL = legacy
 * default stream).  dy, w, dx are device pointers in the plan's layout and
 * dtype; they must not overlap.  Asynchronous: returns after enqueueing one
 * kernel (the CUDA-core path adds a fill kernel where some pixel is
 * uncovered; the fp32 tensor-core path first splits the filter and, when it
 * cuts its last round of tiles into k-block ranges, zeroes those tiles' dx
 * region; NCHW plans on a tensor-core path add their layout transposes).
 * Runs of one plan must not overlap on the GPU: the plan's status word (and
 * for fp32 tensor-core plans the split filter, for plans created with the
 * stream-K override its scratch) are shared by its runs.  Each call is an
 * NVTX range "conv_bwd_data_run" in the domain "conv_bwd_data" (as are
 * run_host and run_forward under their own names).
 * Errors: INVALID_ARG (null or overlapping pointers), MISALIGNED (bf16 NHWC
 * tensor-core path needs 16-byte aligned dy, w, dx; the fp32 tensor-core path
 * 16-byte aligned dy and dx), CUDA (launch failure or plan created without a
 * device). */
conv_bwd_status conv_bwd_data_run(conv_bwd_plan plan, const void *dy, const void *w, void *dx, void *stream);

/* End-to-end variant with host buffers: copies dy_host/w_host into the
 * caller's device buffers dy_dev/w_dev, runs, and copies dx_dev back into
 * dx_host, all ordered on `stream` (use pinned host memory for async
 * copies).  When the copies are large (dy + dx >= 16 MiB, N >= 2) the work is
 * pipelined over up to 4 batch chunks: two copy streams owned by the plan
 * bring dy chunk by chunk and return dx chunk by chunk while `stream` computes
 * the chunk in between; they start after the work already queued on `stream`,
 * and `stream` waits for the last copy, so the ordering seen by the caller is
 * unchanged.  Calls on one plan must not overlap (as for run).  Returns after
 * enqueueing; synchronise the stream before reading dx_host.  Same errors as
 * conv_bwd_data_run. */
conv_bwd_status conv_bwd_data_run_host(conv_bwd_plan plan, const void *dy_host, const void *w_host, void *dx_host,
                                       void *dy_dev, void *w_dev, void *dx_dev, void *stream);

/* Synchronise `stream`, read and clear the plan's device status word.
 * Returns OK, DEVICE_TIMEOUT or DEVICE_FAULT (with *detail, if not NULL, set
 * to the device-side location code), or CUDA if the stream reported an
 * error. */
conv_bwd_status conv_bwd_data_get_status(conv_bwd_plan plan, void *stream, int32_t *detail);

/* Per-kernel timing.  When enabled, run() records CUDA events around each
 * kernel it launches on the stream; conv_bwd_data_last_timing synchronises
 * on those events and returns the device time of the last run's fill kernel
 * (0 if it was skipped) and sub-GEMM kernel in milliseconds. */
conv_bwd_status conv_bwd_data_set_timing(conv_bwd_plan plan, int32_t enable);
conv_bwd_status conv_bwd_data_last_timing(conv_bwd_plan plan, float *fill_ms, float *gemm_ms);

/* Device self-test of the bounded-wait mechanism every pipelined kernel
 * uses: a one-thread kernel waits on a shared-memory barrier that nothing
 * ever arrives on, with a budget of `budget_cycles` SM clocks, and must give
 * up and record a timeout.  *observed receives the recorded status code
 * (CONV_BWD_ERR_DEVICE_TIMEOUT when the mechanism works).  Faults nothing,
 * hangs nothing; synchronises the stream. */
conv_bwd_status conv_bwd_data_selftest_wait_timeout(void *stream, int64_t budget_cycles, int32_t *observed);

/* No-allocation variant of conv_bwd_data_run for the bf16 NHWC/KYXC
 * tensor-core path (C/G >= 64, C/G and K/G multiples of 8).  The pages have
 * no counterpart to this call; it exists for callers that cannot allocate
 * device memory (a host framework that owns all device memory through its own
 * pool, or a loop that must not call cudaMalloc because it can synchronise
 * the device or fail mid-run).  It plans on the host from `desc` on every
 * call and allocates no device memory: the kernel's only scratch, its 4-byte
 * status word, lives in a 256-byte file-scope __device__ array that every GPU
 * loading the library holds until the process exits.  The first call on a
 * device looks up that array's device address (once per device, with the
 * device current); make that first call before any stream capture.  Every
 * call shares the array and clears its status word on `stream` before
 * launching; calls whose kernels overlap on the GPU race on it.
 * Arguments: as conv_bwd_data_run, plus `device_status`: NULL for a fully
 * asynchronous call, or a host int that receives the device status code
 * after the call synchronises `stream`.
 * Errors: INVALID_ARG, MISALIGNED and CUDA as conv_bwd_data_run;
 * UNSUPPORTED if the descriptor is not on the tensor-core path or its scratch
 * would exceed the 256-byte maximum; DEVICE_TIMEOUT / DEVICE_FAULT (only
 * with device_status != NULL) as conv_bwd_data_get_status. */
conv_bwd_status conv_bwd_data_run_noalloc(const conv_bwd_desc *desc, const void *dy, const void *w, void *dx,
                                          void *stream, int32_t *device_status);

/* Human-readable status name (static storage). */
const char *conv_bwd_status_string(conv_bwd_status s);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int32_t conv_bwd_data_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CONV_BWD_DATA_H */
