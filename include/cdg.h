/*
 * cdg.h -- Conv2d backward-data (dgrad) on one NVIDIA GB300 (sm_103a).
 *
 * The operation (apache/tvm PR #10110, "[CUTLASS] Conv2d dgrad", opening
 * description: "Conv2d dgrad"; the stride-2 case is the "strided dgrad" of the
 * benchmark comment on the same page):
 *
 *     dX[n,h,w,c] = sum over k, r, s and every (p, q) with
 *                   h = p*stride - pad + r*dil,  w = q*stride - pad + s*dil,
 *                   0 <= p < P, 0 <= q < Q,   of  dY[n,p,q,k] * W[k,r,s,c]
 *
 * the gradient of a cross-correlation Conv2d with respect to its input.
 * P = floor((H + 2*pad - dil*(R-1) - 1)/stride) + 1, Q likewise with W and S.
 * Inputs are fp16 or bf16; every product is accumulated in fp32 (the page's
 * closing remark that training needs fp32 accumulation).  Optionally the
 * result is gated by a saved activation x, out = (x > 0) ? dX : +0.0 (the
 * dgrad "activation fusion" of the page's last comments).
 *
 * Layouts: dY  NHWC  [N][P][Q][K]
 *          W   KRSC  [K][R][S][C]      (the forward filter, as stored)
 *          dX  NHWC  [N][H][W][C]      (fp16/bf16 like dY, or fp32)
 *          x   NHWC  [N][H][W][C]      (same type as dY)
 * All tensors are dense and contiguous.  Every pointer passed to prepack or
 * dgrad is a DEVICE pointer, 16-byte aligned.
 *
 * Ownership: the caller owns all tensors and streams; the library never
 * allocates, frees or retains caller memory.  A handle owns its host plan
 * and a 4-byte device status word.  Calls are asynchronous on the given stream.
 *
 * Errors: every function returns a cdg_status_t; nothing aborts or throws
 * across this interface.  On any error other than CDG_ERR_CUDA nothing has
 * been launched.
 *
 * Thread safety: a handle may be used from one thread at a time; calls on one
 * handle from different streams must not overlap on the GPU (they share the
 * handle's status word and its cached descriptors).
 */
#ifndef CDG_H
#define CDG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct cdg_plan_st *cdg_handle_t;
/* A cudaStream_t, passed as an opaque pointer (NULL = the legacy default stream). */
typedef void *cdg_stream_t;

typedef enum {
    CDG_OK = 0,
    CDG_ERR_INVALID_ARG = 1,  /* bad size, NULL pointer, unknown flag            */
    CDG_ERR_UNSUPPORTED = 2,  /* valid but outside what the kernels handle:       */
                              /* C or K not a multiple of 8, stride > 4,          */
                              /* R*S > 128, tensor dims beyond TMA limits         */
    CDG_ERR_ALIGNMENT = 3,    /* a tensor pointer is not 16-byte aligned          */
    CDG_ERR_ALIAS = 4,        /* dX overlaps dY, the packed weights or x          */
    CDG_ERR_CUDA = 5,         /* a CUDA runtime/driver call or launch failed      */
    CDG_ERR_TIMEOUT = 6,      /* a kernel gave up a bounded pipeline wait         */
    CDG_ERR_NO_DEVICE = 7,    /* the handle was planned without a device          */
    CDG_ERR_SCRATCH_TOO_SMALL = 8 /* cdg_dgrad_noalloc: packed weights exceed     */
                                  /* CDG_NOALLOC_MAX_WEIGHT_BYTES                 */
} cdg_status_t;

typedef enum { CDG_F16 = 0, CDG_BF16 = 1 } cdg_dtype_t;

/* Epilogue flags (bit set). */
enum {
    CDG_EPI_RELU_BWD = 1,     /* gate by the saved activation: out = (x > 0) ? v : +0.0 */
    CDG_EPI_OUT_F32 = 2,      /* write dX as fp32 instead of the input type             */
    CDG_EPI_RELU_BWD_BITS = 4, /* the same gate from a packed bit mask (one bit per     */
                              /* element, see cdg_pack_relu_mask): out = bit ? v : +0.0 */
                              /* (not together with CDG_EPI_RELU_BWD)                   */
    CDG_EPI_SUM = 8,          /* also the per-channel sums of the output (cdg_dgrad_sums) */
    CDG_EPI_SUM_X = 16,       /* CDG_EPI_SUM plus the per-channel sums of out * x where   */
                              /* the gate passes; needs CDG_EPI_RELU_BWD                 */
    CDG_EPI_GELU_BWD = 32,    /* GELU backward: out = v * f'(x), x the GELU's saved      */
                              /* input (same layout and type as for CDG_EPI_RELU_BWD),   */
                              /* f(x) = x (1 + erf(x / sqrt 2)) / 2                      */
    CDG_EPI_SILU_BWD = 64     /* SiLU backward: out = v * f'(x), f(x) = x / (1 + e^-x)   */
                              /* (at most one of RELU_BWD, RELU_BWD_BITS, GELU_BWD,      */
                              /* SILU_BWD)                                               */
};

/*
 * Plan one dgrad shape on the current CUDA device.
 *   N, H, W    batch and dX spatial size (the forward input size)
 *   C, K       dX channels and dY channels (forward in / out channels)
 *   R, S       filter size; stride, pad, dil apply to both axes, pad symmetric
 *   dtype      CDG_F16 or CDG_BF16 for dY, W and x
 *   epilogue   CDG_EPI_* bit set
 * On success *out receives a handle (free it with cdg_destroy).  Validation:
 * all sizes >= 1 (pad >= 0), P and Q >= 1, C % 8 == 0, K % 8 == 0, stride <= 4,
 * R*S <= 128.  The plan derives P and Q, splits a strided problem into its
 * stride^2 phase sub-convolutions (each dX pixel residue class (h mod stride,
 * w mod stride) receives a fixed subset of the filter taps), chooses tiles and
 * allocates the 4-byte device status word.
 */
int cdg_plan(int N, int H, int W, int C, int K, int R, int S,
             int stride, int pad, int dil, int dtype, int epilogue, cdg_handle_t *out);

/*
 * The same planning without touching any GPU: num_sms stands in for the
 * device's SM count.  The handle answers the query functions below; prepack
 * and dgrad on it return CDG_ERR_NO_DEVICE.  For inspecting the planner.
 */
int cdg_plan_host(int N, int H, int W, int C, int K, int R, int S,
                  int stride, int pad, int dil, int dtype, int epilogue,
                  int num_sms, cdg_handle_t *out);

/* Release a handle (NULL is ignored).  Synchronises nothing. */
void cdg_destroy(cdg_handle_t h);

/* dY's spatial extents P and Q. */
int cdg_get_output_dims(cdg_handle_t h, int *P, int *Q);

/* Bytes the packed-weight buffer must have (R*S*C*K elements of dtype). */
size_t cdg_packed_weight_bytes(cdg_handle_t h);

/*
 * Planner description, for logs and tests.
 */
typedef struct {
    int P, Q;
    int num_phases;       /* stride^2                                            */
    int phase_taps[16];   /* taps of phase (ph, pw) at index ph*stride + pw       */
    int tile_m;           /* dX pixels per tile (GEMM M tile)                      */
    int tile_n;           /* channels per tile (GEMM N tile)                       */
    int tile_k;           /* dY channels per pipeline stage (GEMM K block)         */
    int a_mode;           /* 0: 4-D boxes over dY per tap, 1: dY rows as a matrix, */
                          /* 2: one halo box per K block for all taps, weights     */
                          /*    streamed per tap (opt-in),                         */
                          /* 3: halo boxes with every weight tile resident in      */
                          /*    shared memory (chosen when the filter fits)        */
    int box_w, box_h, box_n; /* output tile box (a_mode 0 and 2)                   */
    int stages;           /* shared-memory pipeline depth                          */
    int work_items;       /* (phase, m-tile, n-tile) items in one launch           */
    int grid;             /* persistent CTAs                                       */
    int smem_bytes;       /* dynamic shared memory per CTA                         */
    int tmem_cols;        /* tensor-memory columns per CTA                         */
    int cta_pair;         /* 1: CTA pairs share 256-row tiles (2-SM MMA)            */
    int mma_warps;        /* MMA-issuing warps per CTA: 2 splits the work items and */
                          /* the pipeline stages between two issuers (N tile <= 128) */
    int tuned;            /* 1 once cdg_autotune has chosen this plan              */
} cdg_plan_info_t;

int cdg_plan_get_info(cdg_handle_t h, cdg_plan_info_t *info);

/*
 * Re-lay the forward filter W (KRSC, dtype, device) into the packed operand
 * the dgrad kernel reads: Wpacked[r*S + s][c][k] = W[k][r][s][c], i.e. for
 * every tap a C x K matrix with K contiguous.  Wpacked must hold
 * cdg_packed_weight_bytes(h) bytes and not overlap W.  Asynchronous on stream.
 */
int cdg_prepack_weights(cdg_handle_t h, const void *W_krsc, void *Wpacked, cdg_stream_t stream);

/*
 * dX = dgrad(dY, W) for the planned shape, one kernel launch, asynchronous
 * on stream.  relu_mask is the saved activation x for a plan with
 * CDG_EPI_RELU_BWD (NHWC like dX, input dtype), the packed mask for
 * CDG_EPI_RELU_BWD_BITS (cdg_pack_relu_mask's layout), the activation's saved
 * input for CDG_EPI_GELU_BWD or CDG_EPI_SILU_BWD (NHWC like dX, input
 * dtype), else NULL; it must not overlap dX.  Every element of dX is written, including pixels no
 * filter tap reaches (+0.0); dX is never read, so its prior contents do not
 * matter.  dY, Wpacked and x are only read.  No workspace, no allocation.
 * A device-side pipeline timeout (which a correct launch never hits) is
 * reported by cdg_device_status, not here.
 */
int cdg_dgrad(cdg_handle_t h, const void *dY, const void *Wpacked, void *dX,
              const void *relu_mask, cdg_stream_t stream);

/*
 * dgrad with the per-channel sums of its output fused into the epilogue (the
 * epilogue fusion of the Bolt reading notes: a reduction over the output is
 * taken where the output is made, instead of by a second pass that re-reads
 * it).  For a plan made with CDG_EPI_SUM, after dX = dgrad(dY, W) (gated as
 * the plan says):
 *
 *     sums[c]     = sum over n, h, w of out[n,h,w,c]
 *     sums[C + c] = sum over n, h, w with x[n,h,w,c] > 0 of out[n,h,w,c] * x[n,h,w,c]
 *                   (CDG_EPI_SUM_X only)
 *
 * taken from the fp32 values before they are rounded to dX's type.  sums[c]
 * is the bias gradient of a bias added before the ReLU, and BatchNorm's beta
 * gradient; with x the BatchNorm output y = gamma*xhat + beta (the ReLU's
 * input, or relu(y), which gives the same terms), BatchNorm's gamma gradient
 * is (sums[C + c] - beta[c]*sums[c]) / gamma[c].  Positions the gate masks add
 * nothing, whatever x holds there.
 *
 *   sums       device, fp32, C (CDG_EPI_SUM) or 2*C (CDG_EPI_SUM_X) values,
 *              overwritten
 *   workspace  device, cdg_sums_workspace_bytes(h) bytes, overwritten: each
 *              CTA of the launch adds its tiles' column sums into a row of its
 *              own, and a second kernel adds the rows in order
 *
 * Two kernel launches on stream.  The result does not depend on scheduling:
 * every partial sum is taken in a fixed order, so repeated calls give the
 * same bits.  Other arguments and errors as for cdg_dgrad; sums and workspace
 * must be 16-byte aligned and overlap no other tensor (CDG_ERR_ALIAS).
 * cdg_dgrad, cdg_dgrad_noalloc and cdg_autotune refuse plans made with the
 * sum flags (CDG_ERR_INVALID_ARG, CDG_ERR_INVALID_ARG, CDG_ERR_UNSUPPORTED).
 */
int cdg_dgrad_sums(cdg_handle_t h, const void *dY, const void *Wpacked, void *dX, const void *relu_mask, float *sums,
                   void *workspace, cdg_stream_t stream);

/* Bytes of the workspace cdg_dgrad_sums needs: (SM count) x (1 or 2) x C x 4;
 * 0 for a plan without the sum flags. */
size_t cdg_sums_workspace_bytes(cdg_handle_t h);

/*
 * Synchronise stream, then read and clear the handle's device status word:
 * CDG_OK, or CDG_ERR_TIMEOUT if a launch since the last call gave up a
 * bounded wait (its dX is then incomplete).
 */
int cdg_device_status(cdg_handle_t h, cdg_stream_t stream);

/*
 * How long any single pipeline wait of this plan's kernel may take before the
 * launch gives up: it then records CDG_ERR_TIMEOUT (read by
 * cdg_device_status), leaves every loop, waits (again bounded) for its own
 * copies and tensor-core work in flight, releases its tensor memory and
 * returns, leaving dX incomplete.  A correct launch never comes near the
 * default of 4 s; a caller with a watchdog of its own may lower it.
 * ns in [1e5, 6e10] (0.1 ms .. 60 s), else CDG_ERR_INVALID_ARG.  Host only;
 * applies to launches made after the call.
 */
int cdg_plan_set_wait_limit(cdg_handle_t h, unsigned long long ns);

/*
 * TEST ONLY.  stage >= 0: every launch of this plan withholds one operand
 * load -- in each CTA, the pipeline stage with that sequence number gets
 * neither its tensor copies nor their byte count -- so the MMA warp's bounded
 * wait for it runs out and the launch takes the timeout path above (status
 * CDG_ERR_TIMEOUT, dX incomplete).  This exercises the failure path without
 * any fault: every wait in the kernel is bounded.  stage = -1 restores normal
 * launches.  Plans in the halo operand mode or with CTA pairs return
 * CDG_ERR_UNSUPPORTED (their loaders do not take the option).  Host only.
 */
int cdg_plan_withhold_load_for_test(cdg_handle_t h, int stage);

/*
 * Plan-time autotuning, in the manner of cuDNN's Find (the pages' comparison of
 * cuDNN's Get and Find algorithm selection): run the dgrad of this plan's shape
 * under each configuration the planner can produce for it (the planner's own
 * choice; without or with CTA pairs; one MMA warp; with or without halo
 * operand boxes; halo boxes with CTA pairs; phases in order; 128- and
 * 192-channel N tiles), reps timed launches
 * each after one untimed launch, and keep the fastest in the handle
 * (cdg_plan_get_info then reports it, with tuned = 1).  Configurations that
 * come out identical are timed once.  Each timed launch follows a write of a
 * scratch buffer twice the L2 size, so candidates are compared with cold
 * caches, as layers run inside a network step.  The planner's own choice is
 * kept unless another configuration is at least 2 % faster.
 *
 *   dY, Wpacked, dX, relu_mask   as for cdg_dgrad; dX is overwritten (with the
 *                                correct result) many times
 *   reps                         timed launches per configuration, 1..1000
 *   best_ms                      if not NULL, receives the best mean launch time
 *
 * Synchronises stream.  Allocates a 4-byte status word per candidate plan and
 * the flush buffer (all freed before returning).  On CDG_ERR_CUDA or
 * CDG_ERR_TIMEOUT the handle keeps its previous plan.
 */
int cdg_autotune(cdg_handle_t h, const void *dY, const void *Wpacked, void *dX, const void *relu_mask,
                 cdg_stream_t stream, int reps, float *best_ms);

/*
 * Pack the ReLU-backward mask of a saved activation x (NHWC, pixels = N*H*W
 * rows of C channels, dtype CDG_F16 or CDG_BF16) for a plan with
 * CDG_EPI_RELU_BWD_BITS.  Layout: each pixel's C channels as bits, the row
 * padded to whole 16-byte units (cdg_relu_mask_bytes(1, C) bytes a pixel);
 * channel c of pixel p is bit c % 8 of byte p*row + c/8, set when x > 0
 * (x <= 0, -0.0 and NaN give 0); padding bits are 0.  For C a multiple of 128
 * this is exactly one bit per element; the padding lets the dgrad fetch a
 * tile's mask with the same tensor copies as its output, and for C < 128 it
 * still cuts the gate's reads 8x against x.  This variant of the pages'
 * ReLU-backward epilogue fusion is an addition of this library (the pages gate
 * with the activation itself).  C % 8 == 0; x and bits 16-byte aligned, not
 * overlapping; bits holds cdg_relu_mask_bytes(pixels, C) bytes, all of which
 * are written.  Asynchronous on stream.
 */
int cdg_pack_relu_mask(const void *x, void *bits, long long pixels, int C, int dtype, cdg_stream_t stream);

/* Bytes of a packed ReLU mask of `pixels` pixels of C channels (see
 * cdg_pack_relu_mask), or -1 for pixels < 0, C <= 0 or C % 8 != 0.  Host only. */
long long cdg_relu_mask_bytes(long long pixels, int C);

/* Static text for a status code. */
const char *cdg_status_string(int status);

/*
 * dgrad for callers that cannot allocate device memory -- code that runs
 * where cudaMalloc is off limits (inside a memory pool that must not grow,
 * a real-time loop that may not block on the allocator, an embedding runtime
 * that owns all device memory).  This entry point has no counterpart in the
 * pages the method is described on; it is an addition of this library.
 *
 * It computes exactly what cdg_prepack_weights followed by cdg_dgrad
 * computes, but takes the forward filter W in its stored KRSC layout and
 * needs neither a packed-weight buffer nor a device status word from the
 * caller: both live in one scratch array compiled into the library
 * (a file-scope __device__ array that every GPU which loads the library keeps
 * until the process exits).  It calls no cudaMalloc, no cudaFree and no
 * allocating library routine.
 *
 *   h          a plan from cdg_plan, or from cdg_plan_host (which touches no
 *              device; pass the device's SM count as num_sms)
 *   dY, dX, relu_mask   as for cdg_dgrad (device pointers, 16-byte aligned)
 *   W_krsc     the forward filter [K][R][S][C], device pointer
 *
 * Limit: the packed weights (R*S*C*K elements of 2 bytes) must fit in
 * CDG_NOALLOC_MAX_WEIGHT_BYTES (8 MiB: 4,194,304 weights, enough for every
 * ResNet-50 convolution); larger filters return CDG_ERR_SCRATCH_TOO_SMALL
 * before anything is launched.
 *
 * The first call on a device finds the scratch array's device address
 * (cudaGetSymbolAddress, with that device current) and raises the kernels'
 * shared-memory limit; make that first call before any stream capture.
 *
 * Every call on a device shares the one scratch array, which keeps the last
 * call's packed weights; each call clears the status word and re-packs W on
 * its stream first.  Calls whose work overlaps on the GPU (different streams,
 * or different host threads) race on the scratch array and give wrong
 * results: serialise them.  A device-side pipeline timeout is recorded in the
 * scratch status word, not returned here: read it with
 * cdg_dgrad_noalloc_status.
 *
 * A plan from cdg_plan_host that chose CTA pairs has its persistent grid
 * checked against the device (how many pairs fit at once) on its first
 * cdg_dgrad_noalloc call, and reduced if needed.
 */
#define CDG_NOALLOC_MAX_WEIGHT_BYTES (8u << 20)
int cdg_dgrad_noalloc(cdg_handle_t h, const void *dY, const void *W_krsc, void *dX, const void *relu_mask,
                      cdg_stream_t stream);

/*
 * The status word cdg_dgrad_noalloc launches report into, on the current
 * device: synchronise stream, read the word and clear it.  Returns CDG_OK, or
 * CDG_ERR_TIMEOUT if a cdg_dgrad_noalloc launch since the last read gave up a
 * bounded wait (its dX is then incomplete), or CDG_ERR_CUDA.  Allocates
 * nothing (the word is in the library's scratch array).  Because every
 * cdg_dgrad_noalloc call on a device shares the word, read it after each call
 * (or each batch of serialised calls) whose result matters.
 */
int cdg_dgrad_noalloc_status(cdg_stream_t stream);

/*
 * Back-to-back dgrads in one persistent kernel: the backward of a
 * bottleneck's 1x1 -> 3x3 forward pair (conv1 1x1 C1 -> C2, then the
 * activation, then conv2 R2 x S2 C2 -> K2), which runs as
 *
 *     g   = act_bwd(dgrad(dY2, W2), x2)     (conv2's dgrad, gated)
 *     dX1 = dgrad_1x1(g, W1)                 (conv1's dgrad)
 *
 * This is the persistent kernel fusion of the Bolt reading notes (page 5 of
 * the pages, "Persistent kernel (GEMM/Conv) fusion"), with threadblock
 * residence: each CTA computes a tile of g over all C2 channels (ThreadBlock_N
 * = the first dgrad's output channels) and keeps it on chip -- in tensor
 * memory, where it is the A operand of the second GEMM -- so g is never
 * read back from HBM.  The second dgrad is 1x1, stride 1, so a tile of dX1
 * needs exactly the same pixels of g.  g itself is written only if asked
 * (conv1's weight gradient needs it).
 *
 *   conv2: stride 1, pad2, dil2, R2 x S2, C2 = 64 input channels (this kernel),
 *          K2 output channels (dY2's), dY2 NHWC [N][P][Q][K2] with
 *          P = H + 2*pad2 - dil2*(R2-1), W2 KRSC [K2][R2][S2][C2];
 *          its weights and a halo tile of dY2 must fit in shared memory
 *          together with W1 (CDG_ERR_UNSUPPORTED otherwise)
 *   conv1: 1x1, stride 1, pad 0, C1 <= 256 input channels (C1 % 8 == 0),
 *          W1 KRSC [C2][1][1][C1]
 *   x2     the saved tensor of the activation between them, NHWC [N][H][W][C2]:
 *          flags CDG_EPI_RELU_BWD (its output or input; g = (x2 > 0) ? v : +0.0),
 *          CDG_EPI_GELU_BWD or CDG_EPI_SILU_BWD (its input; g = v * f'(x2)),
 *          or none of them (no activation: x2 = NULL)
 *   g      NHWC [N][H][W][C2], written only with CDG_FUSED_WRITE_G (else NULL)
 *   dX1    NHWC [N][H][W][C1]
 * All in dtype (dX1 and g in dtype too); fp32 accumulation in both GEMMs; g
 * is rounded to dtype before the second GEMM, exactly as if it went through
 * memory.  Weights are packed once with cdg_fused_prepack_weights.
 */
typedef struct cdg_fused_st *cdg_fused_t;
#define CDG_FUSED_WRITE_G 256

int cdg_fused_plan(int N, int H, int W, int C1, int C2, int K2, int R2, int S2, int pad2, int dil2, int dtype,
                   int flags, cdg_fused_t *out);
/* The same planning without a device (num_sms stands in for the SM count). */
int cdg_fused_plan_host(int N, int H, int W, int C1, int C2, int K2, int R2, int S2, int pad2, int dil2, int dtype,
                        int flags, int num_sms, cdg_fused_t *out);
void cdg_fused_destroy(cdg_fused_t f);
/* Bytes of the two packed weight buffers (W2: R2*S2*C2*K2, W1: C1*C2 elements). */
int cdg_fused_packed_weight_bytes(cdg_fused_t f, size_t *w2_bytes, size_t *w1_bytes);
/* Pack W2 and W1 (device, KRSC) into W2p and W1p; asynchronous on stream. */
int cdg_fused_prepack_weights(cdg_fused_t f, const void *W2_krsc, const void *W1_krsc, void *W2p, void *W1p,
                              cdg_stream_t stream);
/* One launch on stream.  Errors as for cdg_dgrad (CDG_ERR_ALIAS when an
 * output overlaps an input or the other output).  No allocation. */
int cdg_dgrad_fused(cdg_fused_t f, const void *dY2, const void *W2p, const void *x2, const void *W1p, void *g,
                    void *dX1, cdg_stream_t stream);
/* The first dgrad's planner description (halo tiles, grid, stages), with the
 * fused kernel's shared memory and tensor-memory columns. */
int cdg_fused_get_info(cdg_fused_t f, cdg_plan_info_t *info);
/* Synchronise stream, read and clear the fused plan's device status word. */
int cdg_fused_device_status(cdg_fused_t f, cdg_stream_t stream);

/*
 * Weight gradient (wgrad) of the same cross-correlation Conv2d, the
 * follow-up the apache/tvm PR #10110 page ("[CUTLASS] Conv2d dgrad") names
 * for dgrad, "wgrad + parallel split-k" (merge comment).  The page gives no
 * formula; this library computes the definition
 *
 *   dW[k,r,s,c] = sum over n, p, q of
 *                 dY[n,p,q,k] * x[n, p*stride - pad + r*dil, q*stride - pad + s*dil, c]
 *
 * with x read as zero outside the image.  dY NHWC [N][P][Q][K] and the
 * forward input x NHWC [N][H][W][C] in dtype; dW KRSC [K][R][S][C] in dtype,
 * or fp32 with out_f32 = 1.  fp32 accumulation.  The reduction over the
 * N*P*Q positions is split into `splits` parts that run in parallel; their
 * fp32 partials go to a caller-provided workspace and are added in a fixed
 * order, so results are deterministic.
 */
typedef struct cdg_wgrad_st *cdg_wgrad_t;

typedef struct {
    int P, Q;
    int tile_m;           /* dY channels per tile (GEMM M tile, 128)             */
    int tile_n;           /* x channels per tile and tap                          */
    int taps_per_item;    /* taps whose tiles share one MMA along N (narrow C)    */
    int splits;           /* reduction splits                                     */
    int pos_box[3];       /* positions per block along q, p, n (product 64)      */
    int blocks;           /* position blocks of 64 in the reduction              */
    int stages;           /* shared-memory pipeline depth                         */
    int work_items;       /* (split, tap group, m-tile, n-tile) items in one launch */
    int grid;             /* persistent CTAs                                      */
    int smem_bytes;       /* dynamic shared memory per CTA                        */
    int tmem_cols;        /* tensor-memory columns per CTA                        */
    int x_major;          /* 1 (1x1 filters, K <= 64, C > 64): M tiles pair two   */
                          /* 64-channel slices of x and N runs over the dY        */
                          /* channels, so that no M row is idle; tile_m/tile_n    */
                          /* then count x channels / dY channels                  */
} cdg_wgrad_info_t;

/*
 * Plan one wgrad shape on the current device.  Arguments as for cdg_plan
 * (H, W are x's sizes); out_f32 0 or 1; splits = 0 lets the planner choose
 * (enough work items to fill the SMs), k >= 1 asks for k (capped at the
 * number of position blocks).  Errors: CDG_ERR_INVALID_ARG for bad sizes or
 * flags, CDG_ERR_UNSUPPORTED when C or K is not a multiple of 8, stride > 4,
 * R*S > 128, or H or W is smaller than the stride.  Free with
 * cdg_wgrad_destroy.
 */
int cdg_wgrad_plan(int N, int H, int W, int C, int K, int R, int S, int stride, int pad, int dil, int dtype,
                   int out_f32, int splits, cdg_wgrad_t *out);

/* The same planning without a device (num_sms stands in for the SM count);
 * cdg_wgrad on such a handle returns CDG_ERR_NO_DEVICE. */
int cdg_wgrad_plan_host(int N, int H, int W, int C, int K, int R, int S, int stride, int pad, int dil, int dtype,
                        int out_f32, int splits, int num_sms, cdg_wgrad_t *out);

void cdg_wgrad_destroy(cdg_wgrad_t h);

/* Bytes of the fp32 workspace cdg_wgrad needs: splits * K * R * S * C * 4. */
size_t cdg_wgrad_workspace_bytes(cdg_wgrad_t h);

int cdg_wgrad_get_info(cdg_wgrad_t h, cdg_wgrad_info_t *info);

/*
 * dW = wgrad(dY, x): two kernel launches on stream (the split GEMM, then the
 * ordered reduction), asynchronous.  All pointers are device pointers,
 * 16-byte aligned; workspace holds cdg_wgrad_workspace_bytes(h) bytes and is
 * overwritten; dW may not overlap dY, x or the workspace, nor the workspace
 * dY or x (CDG_ERR_ALIAS).  dY and x are only read.  No allocation.  A
 * device-side pipeline timeout is reported by cdg_wgrad_device_status.
 */
int cdg_wgrad(cdg_wgrad_t h, const void *dY, const void *x, void *dW, void *workspace, cdg_stream_t stream);

/* Synchronise stream, then read and clear the plan's device status word. */
int cdg_wgrad_device_status(cdg_wgrad_t h, cdg_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CDG_H */
