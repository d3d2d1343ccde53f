/*
 * conv3d_fp8.h -- C ABI of the FP8 (e4m3) implicit-GEMM 3D convolution for one NVIDIA GB300
 * (sm_103a).
 *
 * The operation ("[Fix] conv3d fp8: guard padded M rows in the epilogue store", ROCm/FlyDSL pull
 * request 969, sections "Problem" and "Root cause"):
 *
 *   y[n,k,do,ho,wo] = bf16_rn( sx * sw * sum_{c,t,r,s} x[n, c, do*sd+t-pd, ho*sh+r-ph, wo*sw+s-pw]
 *                                                     * w[k, c, t, r, s] )
 *
 * x holds e4m3 ("float8_e4m3fn") bytes in NCDHW order, w holds e4m3 bytes in KCTRS order, taps
 * that fall outside the input read zero, and y is bfloat16 in NCDHW order. sx and sw are the
 * per-tensor fp32 dequantisation scales of x and w. The convolution is evaluated as an implicit
 * GEMM with M = N*Do*Ho*Wo output positions ("npq"), N_gemm = K output channels and
 * K_gemm = C*T*R*S, accumulated in fp32 by the tensor cores. M and N are cut into tiles; the rows
 * and columns that pad the last tiles are never stored: every store is masked on row < npq and on
 * col < K, which is the guard the page adds so that padded rows can no longer overwrite live
 * outputs of another column.
 *
 * Conventions for every entry point:
 *   - Returns a conv3d_status. Argument errors are reported before anything is launched.
 *   - Device pointers are plain CUDA device addresses on the plan's device; the caller owns them.
 *     Only the *_run_host calls take host pointers (x_host, w_host, scales, y_host).
 *   - "stream" is a cudaStream_t passed as void*; NULL means the legacy default stream.
 *   - Nothing here synchronises the device except conv3d_fp8_check and conv3d_fp8_destroy (and
 *     the allocation of a plan's device buffers by its first *_run_host call).
 */
#ifndef CONV3D_FP8_H
#define CONV3D_FP8_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct conv3d_fp8_plan_s *conv3d_fp8_plan_t; /* opaque, owned by the library */

typedef enum {
    CONV3D_OK = 0,
    CONV3D_EINVAL = 1,       /* bad argument: NULL or misaligned pointer, non-positive or empty
                                shape, stride/pad that differ from the plan, wrong current device */
    CONV3D_EUNSUPPORTED = 2, /* a valid convolution this library does not handle: C % 16 != 0,
                                a device that is not sm_103, sizes beyond 32-bit index ranges */
    CONV3D_ENOMEM = 3,       /* the plan's device workspace could not be allocated */
    CONV3D_ECUDA = 4,        /* a CUDA runtime or driver call failed (e.g. a launch error) */
    CONV3D_EDEVICE = 5       /* a kernel reported an error through the plan's status word: one of
                                its bounded waits ran out of time and the kernel stopped early */
} conv3d_status;

/* Optional planning knobs. Zero-initialise and set only what you need. */
typedef struct {
    int splits;          /* 0: the library chooses; >= 1: split K_gemm into this many slices
                            (clamped to the number of 128-wide K blocks) */
    int block_n;         /* 0: the library chooses; else the N tile, a multiple of 32 in [32,256] */
    int max_ctas;        /* 0: one persistent CTA per SM; else an upper bound on the grid */
    int wait_timeout_ms; /* 0: 2000 ms; a bounded wait inside a kernel gives up after this long,
                            records CONV3D_EDEVICE in the status word and the kernel exits */
    int debug_flags;     /* test-only: bit 0 makes the weight-tile loader skip its first arrival,
                            so the MMA warp's bounded wait must run out (exercises the error
                            path without faulting anything) */
    int route;           /* 0: the library chooses; 1: A by cp.async gathers from a zero-padded
                            channels-last copy of x; 2: A by TMA im2col loads (EUNSUPPORTED
                            unless C % 32 == 0, strides <= 8 and -16 <= -pad, pad - (filter-1)
                            <= 15 on every axis); 3: padded-grid route, stride 1 and CTA pairs
                            only: M runs over the zero-padded grid of the input and one TMA
                            im2col load of 128 + S - 1 grid positions feeds the S taps along W
                            (EUNSUPPORTED unless every stride is 1, C % 32 == 0, S <= 129 and
                            every pad <= 15); 4: direct route, one CTA: K_gemm in the KCTRS
                            order of the caller's w, which is read as it is by TMA tiles (no
                            weight re-layout), while a pre-pass writes A = im2col(x) explicitly
                            ([npq][C*T*R*S] bytes in the plan's workspace) for TMA tiles too; the
                            default for GEMMs of at most four 128-row tiles with npq <= K
                            (EUNSUPPORTED with a channels-last x, on CTA pairs, or when x holds
                            2^31 bytes or more) */
    int cta_pair;        /* 0: the library chooses; 1: one CTA per 128-row tile; 2: CTA pairs on
                            256-row tiles (tcgen05 cta_group::2; not on the gather route) */
    int input_layout;    /* 0: x is NCDHW (the library transposes it to channels-last every
                            run); 1: x is NDHWC, channels-last, the layout the TMA im2col unit
                            reads: the im2col and padded-grid routes then read the caller's x
                            directly and the run packs only the weights (the gather route still
                            copies x into a zero-padded buffer). With 1 the padded-grid route
                            also needs every pad <= 15. y stays NCDHW either way. */
    int epilogue;        /* 0: the library chooses (explicit stores); 1: explicit stores masked
                            on row < npq and col < K; 2: TMA stores through a tensor map of y
                            as [N][K][dhw], whose extents drop what lies past the end of an image
                            or past K in hardware (rows spilling into a later image still take
                            guarded stores). 2 needs an output-position route (not the padded
                            grid) and dhw % 8 == 0 (EUNSUPPORTED otherwise); the map of y is
                            re-encoded on the host whenever y differs from the previous run's */
    int overlap;         /* 0: the library chooses; -1: never; P > 0: pack the first P input
                            planes, run the GEMM on the whole waves of tiles that read only
                            those, and meanwhile pack the other planes beside it (one block an
                            SM, next to the GEMM's CTAs), then run the remaining tiles as a second
                            GEMM launch; all on the run's stream, chained by programmatic
                            dependent launches (padded-grid route, one image, an NCDHW x that the
                            tiled transpose takes, a GEMM tile that leaves room for a pack block;
                            EUNSUPPORTED otherwise, or when P leaves no whole wave or no plane to
                            pack beside the GEMM). By default it is taken for layers of at least
                            four waves that meet those conditions when a model of the measured
                            rates finds a plane count whose first GEMM launch hides the rest of
                            the pack and saves more than the overlap costs */
} conv3d_fp8_options;

/* What a plan (or a would-be plan) decided. */
typedef struct {
    int Do, Ho, Wo;           /* output extents: floor((in + 2*pad - filter) / stride) + 1 */
    long long npq;            /* M = N*Do*Ho*Wo */
    int k_gemm;               /* C*T*R*S */
    int block_m, block_n;     /* tile of the GEMM view (block_m: 128, or 256 for CTA pairs) */
    int m_tiles, n_tiles;     /* ceil(npq / block_m) (padded-grid route: N * ceil(Do*Hp*Wp /
                                 block_m) over the padded grid), ceil(K / block_n) */
    int k_blocks;             /* ceil(k_gemm / 128); on the padded-grid route the number of
                                 (t, r, channel block) groups, each S taps wide */
    int splits;               /* K slices of each split tile (fp32 partials + a reduction) */
    int k_blocks_per_split;
    int stages;               /* shared-memory pipeline depth */
    int row_chk;              /* 1 when npq % block_m != 0: the row guard is compiled in */
    int grid;                 /* persistent CTAs launched by the main kernel (2 per pair) */
    int sm_count;
    size_t workspace_bytes;   /* device workspace the plan owns */
    int route;                /* 1: gather, 2: TMA im2col, 3: padded grid, 4: direct (as in
                                 options) */
    int cta_pair;             /* 1: one CTA per tile, 2: CTA pairs (as in options) */
    int full_tiles;           /* tiles computed whole; the other m_tiles*n_tiles - full_tiles
                                 are split `splits` ways. With splits == 1 every tile is whole;
                                 a split count in the options splits every tile; by default
                                 only the tiles of a mostly idle last wave are split */
    int epilogue;             /* 1: explicit guarded stores, 2: TMA stores (as in options) */
    int overlap_planes;       /* input planes packed before the GEMM starts; 0: the pack runs
                                 whole before a single GEMM launch (no overlap) */
    int overlap_units;        /* units of the first GEMM launch (whole waves), with overlap */
} conv3d_fp8_plan_info;

/*
 * Plan a convolution for one shape on `device` (a CUDA ordinal).
 *   N,C,D,H,W: input extents (NCDHW); K: output channels; T,R,S: filter extents.
 *   stride[3], pad[3]: per axis (d, h, w); zero padding, dilation 1, one group.
 * Allocates the plan and its device workspace (packed operands, split-K partials, the status
 * word). Errors: EINVAL (bad shape, empty output), EUNSUPPORTED (C % 16 != 0, not sm_103, index
 * ranges beyond 32 bits), ENOMEM, ECUDA. On error *plan is set to NULL.
 * Defined by: "Root cause" (the GEMM view M = npq, N = K, K_gemm = C*T*R*S and grid_m =
 * ceil(npq / TILE_M), the tiling whose padded rows the store guard must drop). The page prints
 * no host interface: the argument list is this library's.
 */
conv3d_status conv3d_fp8_plan(conv3d_fp8_plan_t *plan, int N, int C, int D, int H, int W, int K,
                              int T, int R, int S, const int stride[3], const int pad[3],
                              int device);

/* As conv3d_fp8_plan, with planning knobs (opts may be NULL). Defined by: as conv3d_fp8_plan;
 * the knobs are this library's (none of them changes what is computed). */
conv3d_status conv3d_fp8_plan_ex(conv3d_fp8_plan_t *plan, int N, int C, int D, int H, int W,
                                 int K, int T, int R, int S, const int stride[3],
                                 const int pad[3], int device, const conv3d_fp8_options *opts);

/*
 * Run the planned convolution, asynchronously on `stream`.
 *   x_ncdhw: N*C*D*H*W e4m3 bytes, contiguous, 16-byte aligned; NDHWC (channels-last) instead
 *            when the plan was made with input_layout = 1 (the A tensor map then points at x:
 *            it is re-encoded on the host whenever x differs from the previous run's).
 *   w_kctrs: K*C*T*R*S e4m3 bytes, contiguous, 16-byte aligned.
 *   scale_x, scale_w: device pointers to one fp32 each (read on the device, so a run can be
 *                     captured in a CUDA graph and the scales may change between replays).
 *   y_ncdhw: N*K*Do*Ho*Wo bfloat16, contiguous, 16-byte aligned; every element is written
 *            exactly once and its prior contents never leak into the result.
 *   stride, pad: must equal the plan's (EINVAL otherwise).
 * The plan's workspace is shared by its runs: at most one run of a plan may be in flight at a
 * time (use one plan per concurrent stream). Errors: EINVAL, ECUDA (launch failure).
 * Kernel-side errors are reported later, by conv3d_fp8_check.
 * Defined by: "Problem" (e4m3 x and w with per-tensor scales from the fp8 cast, BF16 output),
 * "Root cause" (NCDHW store offset, padding taps read zero, padded rows carry a zero
 * accumulator) and "Fix" (stores masked on row < npq as well as col < K; the split-K path guards
 * its reduction the same way).
 */
conv3d_status conv3d_fp8_run(conv3d_fp8_plan_t plan, const void *x_ncdhw, const void *w_kctrs,
                             const float *scale_x, const float *scale_w, void *y_ncdhw,
                             const int stride[3], const int pad[3], void *stream);

/*
 * conv3d_fp8_run with the tensors in host memory (defined by: none -- library plumbing around
 * conv3d_fp8_run, for callers whose data lives on the host). Enqueued on `stream`, in this order:
 * copies of x_host (N*C*D*H*W e4m3 bytes, in the plan's input layout), w_host (K*C*T*R*S bytes)
 * and scales[0] = scale_x, scales[1] = scale_w (two fp32) into device buffers the plan owns; the
 * run of conv3d_fp8_run on those buffers; a copy of y (N*K*Do*Ho*Wo bfloat16, NCDHW) into y_host.
 * One cudaMemcpyAsync per copy. The call returns once all of it is enqueued: y_host holds the
 * result after the stream has passed that point (e.g. cudaStreamSynchronize). The device buffers
 * (x, w, y, each rounded up to 256 bytes, plus 256) are allocated by the plan's first such call
 * and freed by conv3d_fp8_destroy; conv3d_fp8_workspace_size does not count them. The host
 * buffers stay caller-owned; page-locked ones (cudaHostAlloc / cudaHostRegister) let the copies
 * run asynchronously and overlap work on other streams, pageable ones work too (the copies are
 * then staged by the driver). As for conv3d_fp8_run, at most one run of a plan is in flight at a
 * time: to overlap one step's copies with another's compute, use one plan per stream.
 * Errors: EINVAL (NULL pointer, a bfloat16 plan, stride / pad / device mismatch), ENOMEM (the
 * device buffers), ECUDA; then as conv3d_fp8_run.
 */
conv3d_status conv3d_fp8_run_host(conv3d_fp8_plan_t plan, const void *x_host, const void *w_host,
                                  const float scales[2], void *y_host, const int stride[3],
                                  const int pad[3], void *stream);

/*
 * Measurement hook: while ev_begin / ev_end (cudaEvent_t values passed as void*; either may be
 * NULL) are set, every run of this plan records ev_begin on its stream immediately before the
 * main implicit-GEMM kernel and ev_end immediately after it, or after the reduction of its
 * split tiles when it has some, so a caller can time the GEMM apart from the operand packing.
 * The caller owns the events. Pass NULL, NULL to stop. Errors: EINVAL for a NULL plan.
 * Defined by: none (library plumbing, for measurement).
 */
conv3d_status conv3d_fp8_set_timing_events(conv3d_fp8_plan_t plan, void *ev_begin, void *ev_end);

/*
 * Measurement hook of the operand re-layout (defined by: none, library plumbing). While ev_pack
 * (a cudaEvent_t passed as void*) is set, every run of this plan records it on its stream
 * immediately before the pack kernel; with ev_begin of conv3d_fp8_set_timing_events also set, the
 * interval ev_pack -> ev_begin is the pack alone. The caller owns the event; NULL stops.
 * Errors: EINVAL for a NULL plan.
 */
conv3d_status conv3d_fp8_set_pack_timing_event(conv3d_fp8_plan_t plan, void *ev_pack);

/*
 * Write-count hook for tests (defined by: the page's "Verification" -- every output element
 * written exactly once -- checked directly rather than through a NaN pre-fill). Only a library
 * built with C3D_COUNT_WRITES counts: there every store of output element i by a later run of
 * this plan (main kernel, TMA-store box, split-K reduction) also adds one to counts[i], a device
 * array of N*K*Do*Ho*Wo uint32 (NCDHW order, 4-byte aligned, caller-owned, zeroed by the caller);
 * NULL stops. The product build returns EUNSUPPORTED and never counts.
 * Errors: EINVAL (NULL plan, misaligned counts), EUNSUPPORTED (product build).
 */
conv3d_status conv3d_fp8_set_write_counter(conv3d_fp8_plan_t plan, void *counts);

/*
 * Allocation-free run (no counterpart on the subject page; it exists for callers of this library).
 * Some callers cannot call cudaMalloc: a host framework whose caching allocator owns the device's
 * memory pool, a plugin interface that passes tensors in but offers no way to ask for memory, or a
 * latency-critical loop that cannot take the device synchronisation of cudaFree. This entry point
 * needs no plan and allocates nothing: it runs the same kernels as conv3d_fp8_run, with their
 * scratch (packed operands, split-K partials, status word) in a fixed device array of
 * CONV3D_FP8_NOALLOC_SCRATCH_BYTES that the library's device code reserves on every GPU that
 * loads it, until the process exits.
 *   Shape, stride and pad are as for conv3d_fp8_plan (default planning, current device); x, w,
 *   the scales and y are as for conv3d_fp8_run. The call is asynchronous on `stream`.
 *   The first call on each device takes the array's device address and sets a kernel attribute;
 *   make that first call before any stream capture on that device. The address is kept for the
 *   life of the process: after cudaDeviceReset the entry point must not be called again.
 *   Each call rewrites everything of the array it reads: the packed operands (the zero halo of
 *   the padded copy included) and the status word; partials are written before they are read.
 *   All calls share the one array and it keeps the last call's contents: calls whose work overlaps
 *   on the GPU race on it, so serialise them. Kernel-side bounded-wait errors are not returned
 *   here: conv3d_fp8_noalloc_check reads them after the call.
 * Errors: EINVAL, EUNSUPPORTED (as for planning, and when the problem needs more scratch than the
 * array holds: packed x and w plus split-K partials), ECUDA.
 */
#define CONV3D_FP8_NOALLOC_SCRATCH_BYTES (32u << 20)

conv3d_status conv3d_fp8_run_noalloc(int N, int C, int D, int H, int W, int K, int T, int R,
                                     int S, const int stride[3], const int pad[3],
                                     const void *x_ncdhw, const void *w_kctrs,
                                     const float *scale_x, const float *scale_w, void *y_ncdhw,
                                     void *stream);

/*
 * Status of the latest conv3d_fp8_run_noalloc call on the current device (defined by: none,
 * library plumbing: the status word of the kernels' bounded waits, in the shared scratch).
 * Synchronises the device, then reports and clears that call's status word: OK, or EDEVICE when a
 * bounded wait of its kernels ran out. OK when no such call has been made on the device. A later
 * allocation-free call clears the word itself, so check before the next one.
 * Errors: EUNSUPPORTED (device ordinal beyond the entry point's table), ECUDA.
 */
conv3d_status conv3d_fp8_noalloc_check(void);

/* Synchronise the plan's device, then report (and clear) its status word: OK or EDEVICE.
 * Defined by: none (library plumbing: the status word of the kernels' bounded waits). */
conv3d_status conv3d_fp8_check(conv3d_fp8_plan_t plan);

/* Fill *info for an existing plan. Defined by: none (library plumbing); its tile counts are the
 * grid_m = ceil(npq / TILE_M) of "Root cause" for this library's tiles. */
conv3d_status conv3d_fp8_get_info(conv3d_fp8_plan_t plan, conv3d_fp8_plan_info *info);

/*
 * Host-only: what conv3d_fp8_plan_ex would decide for this shape on a GPU with `sm_count` SMs.
 * Touches no device. Same validation and error codes as planning (except ENOMEM / ECUDA).
 * Defined by: none (library plumbing).
 */
conv3d_status conv3d_fp8_describe(int N, int C, int D, int H, int W, int K, int T, int R, int S,
                                  const int stride[3], const int pad[3], int sm_count,
                                  const conv3d_fp8_options *opts, conv3d_fp8_plan_info *info);

/* Bytes of device workspace the plan owns (0 for a NULL plan). Defined by: none (plumbing). */
size_t conv3d_fp8_workspace_size(conv3d_fp8_plan_t plan);

/* Output extents of the plan: floor((in + 2*pad - filter) / stride) + 1 per axis. Defined by:
 * none (plumbing; the plain convolution's output size, which the page assumes). */
conv3d_status conv3d_fp8_out_dims(conv3d_fp8_plan_t plan, int *Do, int *Ho, int *Wo);

/* Synchronise the plan's device, free its workspace and the plan. NULL is a no-op.
 * Defined by: none (library plumbing). */
void conv3d_fp8_destroy(conv3d_fp8_plan_t plan);

/* Static description of a status code. Defined by: none (library plumbing). */
const char *conv3d_fp8_strerror(conv3d_status status);

/*
 * Per-tensor e4m3 quantiser on the GPU: the producer of the e4m3 bytes and scale that
 * conv3d_fp8_run consumes (the "fp8cast" of the subject page's section "Problem"), with no host
 * synchronisation:
 *   amax = max |v|,  s = fp32(amax / 448) (1 when amax == 0),
 *   q = e4m3 round-to-nearest-even of clamp(fp32(v / s), -448, 448) (IEEE fp32 division).
 * NaN inputs are not supported (their codes and the scale are then unspecified).
 */
typedef enum { CONV3D_SRC_F32 = 1, CONV3D_SRC_BF16 = 2 } conv3d_src_type;

/*
 * Quantise n values of src (fp32 or bfloat16, 16-byte aligned device pointer) into n e4m3 bytes
 * at dst_e4m3 (16-byte aligned) and their scale into *scale_out (a device float, which also holds
 * the running amax while the call's kernels execute). Asynchronous on `stream`. Errors: EINVAL
 * (NULL or misaligned pointers, n <= 0, unknown src_type), ECUDA.
 */
conv3d_status conv3d_fp8_quantize(const void *src, int src_type, long long n, void *dst_e4m3,
                                  float *scale_out, void *stream);

/*
 * A run of an e4m3 plan (made with input_layout = 0) from an fp32 or bfloat16 NCDHW x: the amax
 * and the scale of x are computed on the device, the pack quantises x to e4m3 while it transposes
 * it (no separate quantised copy), and the implicit GEMM reads the scale from the device.
 *   x_src: N*C*D*H*W values of src_type, contiguous NCDHW, 16-byte aligned.
 *   w_kctrs, scale_w, y_ncdhw, stride, pad: as for conv3d_fp8_run.
 *   scale_x_out: if not NULL, a device float that receives the scale of x.
 * Errors: EINVAL (as conv3d_fp8_run, a bfloat16 or channels-last plan, unknown src_type), ECUDA.
 */
conv3d_status conv3d_fp8_run_quantize_x(conv3d_fp8_plan_t plan, const void *x_src, int src_type,
                                        const void *w_kctrs, const float *scale_w, void *y_ncdhw,
                                        const int stride[3], const int pad[3], float *scale_x_out,
                                        void *stream);

/*
 * BF16-input twin ("Notes" of the subject page: the BF16 implicit-GEMM conv3d kernel, which guards
 * its padded rows the same way). The same convolution with bfloat16 x and w and no scales:
 *   y = bf16(sum over c, t, r, s of x * w), fp32 accumulation on the tensor cores
 *   (tcgen05.mma kind::f16), BF16 NCDHW output with the same row and column guards, the same
 *   routes, tiles (in bytes), split-K path and scheduler as the e4m3 path.
 * Plans are conv3d_fp8_plan_t values: conv3d_fp8_destroy, _check, _get_info, _out_dims,
 * _workspace_size and _set_timing_events apply to them too; conv3d_fp8_run rejects a bfloat16
 * plan and conv3d_bf16_run an e4m3 one (EINVAL). C must be a multiple of 8 (16 bytes); the im2col
 * and padded-grid routes need C % 16 == 0. k_gemm in the plan info counts elements.
 *   x_ncdhw: N*C*D*H*W bfloat16, contiguous, 16-byte aligned (NDHWC with input_layout = 1).
 *   w_kctrs: K*C*T*R*S bfloat16, contiguous, 16-byte aligned.
 *   y_ncdhw: N*K*Do*Ho*Wo bfloat16, as for conv3d_fp8_run.
 * Errors as for the e4m3 calls.
 */
conv3d_status conv3d_bf16_plan(conv3d_fp8_plan_t *plan, int N, int C, int D, int H, int W, int K,
                               int T, int R, int S, const int stride[3], const int pad[3],
                               int device);
conv3d_status conv3d_bf16_plan_ex(conv3d_fp8_plan_t *plan, int N, int C, int D, int H, int W,
                                  int K, int T, int R, int S, const int stride[3],
                                  const int pad[3], int device, const conv3d_fp8_options *opts);
conv3d_status conv3d_bf16_run(conv3d_fp8_plan_t plan, const void *x_ncdhw, const void *w_kctrs,
                              void *y_ncdhw, const int stride[3], const int pad[3], void *stream);
/* The twin of conv3d_fp8_run_host: bfloat16 x_host and w_host (2 bytes an element), no scales. */
conv3d_status conv3d_bf16_run_host(conv3d_fp8_plan_t plan, const void *x_host, const void *w_host,
                                   void *y_host, const int stride[3], const int pad[3],
                                   void *stream);
/* Host-only planning of the BF16 twin, as conv3d_fp8_describe. */
conv3d_status conv3d_bf16_describe(int N, int C, int D, int H, int W, int K, int T, int R, int S,
                                   const int stride[3], const int pad[3], int sm_count,
                                   const conv3d_fp8_options *opts, conv3d_fp8_plan_info *info);

#ifdef __cplusplus
}
#endif

#endif /* CONV3D_FP8_H */
