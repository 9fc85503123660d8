/*
 * gbconv: convolution forward, input gradient (dgrad) and weight gradient (wgrad) on one NVIDIA
 * GB300 (sm_103a), exposed as a plain C ABI.
 *
 * Operations (definitions as the source pages state them):
 *
 *   forward   y[n, co, o] = bias[co] + sum_{cl < C_in/G, k} x[n, g*C_in/G + cl, o*stride + k*dil - pad] * w[co, cl, k]
 *             with g = co / (C_out/G), x taken as zero outside the input (cross-correlation, no kernel flip).
 *             Sources: burn-cubecl `src/kernel/conv/im2col.rs`, doc of `im2col` (read position
 *             out*stride + k*dilation - padding, zero outside); teeny-kernels `src/nn/conv/conv2d.rs`,
 *             `conv2d_forward` (group window, weight [C_OUT, C_IN/G, KH, KW]) and `conv2d_bias_forward`
 *             (bias added once after the reduction); oarust `src/rs/ml/matrix/conv.rs`, `conv_1d` and
 *             `conv_2d` (NCL / NCHW inputs, OIK / OIHW weights).
 *
 *   dgrad     dx = the gradient of sum(y * dy) with respect to x for the bias-free forward above:
 *             dx[n, ci, i] = sum over co in ci's group, k, and output positions o with o*stride + k*dil - pad == i
 *             of dy[n, co, o] * w[co, ci - g*C_in/G, k].
 *             Sources: teeny-kernels `conv2d_backward_dx` (the scatter form), oarust `conv_2d_backward`
 *             (an input-gradient pass over input elements, i.e. the gather form).  The library computes the
 *             gather form: every dx element is written once, with no atomics, so results are deterministic.
 *
 *   wgrad     dw = the gradient of sum(y * dy) with respect to w:
 *             dw[co, cl, k] = sum over n and output positions o of dy[n, co, o] * x[n, g*C_in/G + cl, o*stride + k*dil - pad]
 *             (x zero outside the input), and the bias gradient db[co] = sum over n, o of dy[n, co, o].
 *             Sources: burn-cubecl `wgrad_im2col` / `wgrad_im2col_1x1` (the contraction of the output gradient
 *             with the input's columns over every batch position, cut into pieces whose partial sums are added
 *             afterwards: `wgrad_im2col_1x1_split`), teeny-kernels `conv2d_backward_dw` (one sum per weight
 *             element, there accumulated with atomics), oarust `conv_2d_backward` (returns the bias gradient
 *             beside the weight gradient).  The library adds its partial sums in a fixed order, with no atomics.
 *
 *   out size  out = (in + pad + pad_end - dil*(k - 1) - 1) / stride + 1 (floor), rejected when
 *             in + pad + pad_end < dil*(k-1) + 1 (pad_end = pad unless the descriptor asks for (begin, end)
 *             padding).  Source: oarust `Conv1dGeometry::resolve` (symmetric padding); burn-cubecl's
 *             (begin, end) padding pairs.
 *
 * Conventions shared by every entry point:
 *  - All tensors are dense and contiguous in the layouts named by the descriptor.  Activation layouts:
 *    GBCONV_NCHW (NCL for 1-D) or GBCONV_NHWC (NLC for 1-D).  Weight layouts: GBCONV_W_OIHW
 *    [C_out, C_in/G, KH, KW] (OIK for 1-D; the pages' canonical order) or GBCONV_W_OHWI
 *    [C_out, KH, KW, C_in/G] (the channels-last weight order burn-cubecl's im2col column axis uses).
 *  - Data pointers are DEVICE pointers owned by the caller; the library never allocates, frees or
 *    retains them.  `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *    Calls only enqueue work: they return after the launch, not after the kernel finishes.
 *  - Element types: GBCONV_F32 (x, w, y all float) or GBCONV_BF16 (x, w, y all bf16, accumulation in
 *    fp32, one round-to-nearest-even at the store).  bias, when given, is always float [C_out].
 *  - Errors: shape errors return GBCONV_EINVAL before anything is launched; shapes whose 32-bit device
 *    indexing would overflow return GBCONV_EUNSUPPORTED; launch failures return GBCONV_ECUDA.  A kernel
 *    whose internal wait gave up (it never should) records it on the device; gbconv_device_status reads it.
 *  - Every valid shape is served on the GPU.  Which kernel family serves it is reported by gbconv_select.
 */
#ifndef GBCONV_H
#define GBCONV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GBCONV_OK = 0,
  GBCONV_EINVAL = 1,          /* invalid shape or argument (degenerate extent, kernel larger than padded input ...) */
  GBCONV_EUNSUPPORTED = 2,    /* valid, but beyond this library's limits (32-bit element indexing) */
  GBCONV_ECUDA = 3,           /* a CUDA runtime call failed; cudaGetLastError has the detail */
  GBCONV_ETIMEOUT = 4         /* a kernel's bounded internal wait expired (reported by gbconv_device_status) */
} gbconv_status;

typedef enum { GBCONV_NCHW = 0, GBCONV_NHWC = 1 } gbconv_layout;
typedef enum { GBCONV_W_OIHW = 0, GBCONV_W_OHWI = 1 } gbconv_wlayout;
typedef enum { GBCONV_F32 = 0, GBCONV_BF16 = 1 } gbconv_dtype;

/* Kernel families, as reported by gbconv_select. */
typedef enum {
  GBCONV_K_DIRECT = 0,        /* generic direct kernel on CUDA cores (any layout, dtype, groups, stride, dilation) */
  GBCONV_K_DEPTHWISE = 1,     /* NHWC bf16 depthwise direct kernel, bandwidth bound */
  GBCONV_K_POINTWISE = 2,     /* NHWC bf16 1x1: TMA-fed tcgen05 GEMM */
  GBCONV_K_IMPLICIT = 3,      /* NHWC bf16 dense and grouped (C_in/G > 8): implicit GEMM on tcgen05, halo tile in
                                 shared memory (wide images in column strips) */
  GBCONV_K_DGRAD = 4,         /* NHWC bf16 dgrad: stride-phase gather implicit GEMM on tcgen05 (3-D: depth phases at a depth stride) */
  GBCONV_K_DIRECT_DGRAD = 5,  /* generic gather dgrad on CUDA cores */
  GBCONV_K_DEPTHWISE_DGRAD = 6, /* NHWC bf16 depthwise dgrad: gather on CUDA cores, bandwidth bound (3x3 stride 2:
                                    TMA-fed dy tiles, each dy 2x2 block giving a dx 2x2 block) */
  GBCONV_K_DIRECT_WGRAD = 7,   /* generic wgrad on CUDA cores: per-chunk partial sums, then an ordered reduction */
  GBCONV_K_WGRAD = 8,          /* NHWC bf16 wgrad on tcgen05: taps packed into M and N, then an ordered reduction
                                  (H/W strides: one stride phase per work unit; 3-D: one kernel-depth tap per unit) */
  GBCONV_K_SMALLGROUP = 9,     /* NHWC bf16 small groups (1 < G < C, C_in/G = C_out/G in {2, 4, 8}): TMA-fed halo
                                  tiles on CUDA cores */
  GBCONV_K_SMALLGROUP_DGRAD = 10 /* their dgrad: the same tiled kernel at stride 1, a vectorised gather otherwise */
} gbconv_kernel;

typedef enum { GBCONV_OP_FWD = 0, GBCONV_OP_BWD_DATA = 1, GBCONV_OP_BWD_FILTER = 2 } gbconv_op;

typedef enum { GBCONV_PAD_SYMMETRIC = 0, GBCONV_PAD_BEGIN_END = 1 } gbconv_pad_mode;

/* One convolution.  For spatial_dims == 1 only index 0 of in/k/stride/pad/pad_end/dil is read (the
 * length axis).  For spatial_dims == 2 index 0 is height and index 1 is width.  For spatial_dims == 3
 * index 0 is depth, 1 height and 2 width (burn-cubecl `ConvOptions<N>`: one stride, padding and
 * dilation per spatial axis, the same index map on each); the activations are then NCDHW or NDHWC
 * and the weight [C_out, C_in/G, KD, KH, KW] (GBCONV_W_OIHW) or [C_out, KD, KH, KW, C_in/G]
 * (GBCONV_W_OHWI).  Unread entries are ignored.
 * Padding: with pad_mode GBCONV_PAD_SYMMETRIC (0, what a zero-initialised descriptor holds) axis i has
 * pad[i] zeros on both sides and pad_end is not read; with GBCONV_PAD_BEGIN_END it has pad[i] zeros
 * before and pad_end[i] zeros after (burn-cubecl's padding is such a (begin, end) pair per axis).
 * Output extent per axis: (in + pad + pad_end - dil*(k-1) - 1) / stride + 1, floor. */
typedef struct {
  int32_t spatial_dims;       /* 1, 2 or 3 */
  int32_t layout;             /* gbconv_layout of x, y, dy, dx */
  int32_t wlayout;            /* gbconv_wlayout of w */
  int32_t dtype;              /* gbconv_dtype of x, w, y, dy, dx */
  int64_t n, c_in, c_out, groups;
  int64_t in[3], k[3], stride[3], pad[3], dil[3];
  int64_t pad_end[3];         /* end-side padding, read when pad_mode == GBCONV_PAD_BEGIN_END */
  int32_t pad_mode;           /* gbconv_pad_mode */
} gbconv_desc;

/* Output spatial extent of the forward convolution (oarust Conv1dGeometry::resolve applied per axis).
 * out[0] = OH (or L_out for 1-D), out[1] = OW (1 for 1-D); for 3-D out[0] = OD, out[1] = OH,
 * out[2] = OW.  The caller's array holds 3 entries; entries past the rank are set to 1.  Launches nothing.
 * Returns GBCONV_EINVAL for a NULL argument or any shape the forward would reject. */
gbconv_status gbconv_out_shape(const gbconv_desc *desc, int64_t out[3]);

/* Which kernel family would serve `op` for this descriptor (pointers assumed 16-byte aligned).
 * Launches nothing. */
gbconv_status gbconv_select(const gbconv_desc *desc, int32_t op, int32_t *kernel);

/* A one-line description of the plan that would serve `op` for this descriptor (pointers assumed
 * 16-byte aligned): the kernel family, and for the tensor-core implicit GEMM its tile width, work
 * items, stride phases, activation sources, taps, weight residency, pipeline depth and shared memory;
 * for the tensor-core weight gradient its block pairs, chunks, work units, box rows, pitch, MMA groups
 * and width, kernel-depth taps, stride phases and shared memory.
 * Writes at most `len` bytes including the terminating NUL into the caller's host buffer `buf`
 * (truncating if needed).  Launches nothing and needs no GPU.
 * Returns GBCONV_EINVAL for a NULL argument, len < 1, an unknown op, or a shape the call would reject. */
gbconv_status gbconv_describe(const gbconv_desc *desc, int32_t op, char *buf, int64_t len);

/* Forward convolution, y = conv(x, w) (+ bias).
 *   x    : device, [N, C_in, in...] or [N, in..., C_in] per desc->layout, desc->dtype
 *   w    : device, per desc->wlayout, desc->dtype
 *   bias : device float [C_out], or NULL for no bias
 *   y    : device, [N, C_out, out...] or [N, out..., C_out], desc->dtype; fully overwritten
 * Enqueues exactly one kernel on `stream`.  y must not overlap x, w or bias. */
gbconv_status gbconv_fwd(const gbconv_desc *desc, const void *x, const void *w, const float *bias,
                         void *y, void *stream);

/* Input gradient of the forward convolution described by desc (desc is the FORWARD descriptor: its
 * input extent fixes dx's shape, which the output extent alone does not, see burn-cubecl
 * `dgrad_im2col_1x1`, which takes the input shape for the same reason).
 *   dy : device, forward-output shape, desc->dtype
 *   w  : device, forward weight, per desc->wlayout
 *   dx : device, forward-input shape, desc->dtype; fully overwritten (no need to zero it first)
 * Enqueues exactly one kernel on `stream`.  Deterministic: the same inputs give bitwise-equal dx. */
gbconv_status gbconv_bwd_data(const gbconv_desc *desc, const void *dy, const void *w, void *dx, void *stream);

/* Bytes of device staging buffer that gbconv_fwd_host (op GBCONV_OP_FWD; with_bias nonzero when a bias
 * is passed), gbconv_bwd_data_host or gbconv_conv_transpose_host (op GBCONV_OP_BWD_DATA) needs for this descriptor: the weight,
 * the bias, the whole source batch and the whole result batch, each rounded up to 256 bytes.
 * Launches nothing.  Returns GBCONV_EINVAL for a NULL argument, another op, or a shape the call would
 * reject. */
gbconv_status gbconv_host_staging_bytes(const gbconv_desc *desc, int32_t op, int32_t with_bias, int64_t *bytes);

/* gbconv_fwd on HOST buffers: synchronous (done_event NULL), or enqueued with a completion event.
 *   x, w, bias, y : host memory in the layouts gbconv_fwd takes (bias float [C_out] or NULL).
 *                   Page-locked (pinned) memory lets the copies overlap the kernels; pageable memory
 *                   works too, without the overlap.
 *   staging       : device, at least gbconv_host_staging_bytes(desc, GBCONV_OP_FWD, bias != NULL) bytes,
 *                   256-byte aligned, owned by the caller; its contents are undefined afterwards.
 *   slices        : batch slices to pipeline (clamped to [1, min(N, 16)]), or 0 for the library's
 *                   choice, about sqrt(result bytes / 512 KiB) slices.  One slice runs every step on
 *                   `stream` itself.
 *   stream        : the call's copies and kernels start after the work already enqueued there.  A
 *                   call of one slice without a completion event runs on `stream` itself; otherwise
 *                   the copies in, the kernels and the copies out run on three streams the library
 *                   creates per device on first use.
 *   done_event    : NULL: the call returns once y holds the result, and `stream` also waits for every
 *                   copy of the call.  Else a cudaEvent_t (as void*) of the current device that the
 *                   call records when y holds the result, returning as soon as everything is
 *                   enqueued: x, w, bias, y and the staging buffer must then stay valid and untouched
 *                   until the event completes (also after an error return, when it is recorded after
 *                   whatever was enqueued).  Independent calls made this way overlap one call's last
 *                   copy out with the next call's copies in.
 * The batch is cut into slices of consecutive images.  The copy in of slice i+1 (host to device), the
 * kernel of slice i and the copy out of slice i-1 (device to host) run at the same time.  Each slice
 * is one gbconv_fwd call on the staging buffer, so the results are those of gbconv_fwd on the same
 * batch slices (and equal to one call on the whole batch: images are independent).  The enqueueing of host calls on one device is
 * serialised; their copies run in call order.
 * Returns the first failing slice's status, GBCONV_EINVAL for NULL buffers or a staging buffer that is
 * too small or misaligned (nothing enqueued then), GBCONV_ECUDA for a failed copy, and, synchronous
 * only, GBCONV_ETIMEOUT (clearing the record) when a kernel of the library on this device recorded an
 * expired internal wait by the end of the call; with a completion event gbconv_device_status reports
 * that, as for the device-pointer calls. */
gbconv_status gbconv_fwd_host(const gbconv_desc *desc, const void *x, const void *w, const float *bias, void *y,
                              void *staging, int64_t staging_bytes, int32_t slices, void *stream, void *done_event);

/* gbconv_bwd_data on HOST buffers (dy, w and dx in host memory), pipelined, synchronous or with a
 * completion event, as gbconv_fwd_host; staging of at least
 * gbconv_host_staging_bytes(desc, GBCONV_OP_BWD_DATA, 0) bytes. */
gbconv_status gbconv_bwd_data_host(const gbconv_desc *desc, const void *dy, const void *w, void *dx, void *staging,
                                   int64_t staging_bytes, int32_t slices, void *stream, void *done_event);

/* gbconv_conv_transpose on HOST buffers (x, w, bias float [C_in] or NULL, y in host memory), pipelined,
 * synchronous or with a completion event, as gbconv_fwd_host; staging of at least
 * gbconv_host_staging_bytes(desc, GBCONV_OP_BWD_DATA, bias != NULL) bytes. */
gbconv_status gbconv_conv_transpose_host(const gbconv_desc *desc, const void *x, const void *w, const float *bias,
                                         void *y, void *staging, int64_t staging_bytes, int32_t slices, void *stream,
                                         void *done_event);

/* Transposed convolution forward, y = conv_transpose(x, w) (+ bias): by definition the input gradient
 * above applied to x, plus a per-channel bias (oarust `conv_transpose_1d` / `conv_transpose_2d`
 * compute the same scatter with an IOK weight).  desc describes the convolution being transposed:
 * its input extent is y's extent, which fixes what a framework's output_padding selects.
 *   x    : device, forward-output shape [N, C_out, out...] / [N, out..., C_out], desc->dtype
 *   w    : device, the forward weight per desc->wlayout; with GBCONV_W_OIHW this is the transposed
 *          convolution's own [C_in_t = C_out, C_out_t / G = C_in / G, KH, KW] weight
 *   bias : device float [C_in] (the transposed convolution's output channels), or NULL
 *   y    : device, forward-input shape, desc->dtype; fully overwritten
 * Enqueues exactly one kernel on `stream`.  Deterministic, as gbconv_bwd_data. */
gbconv_status gbconv_conv_transpose(const gbconv_desc *desc, const void *x, const void *w, const float *bias,
                                    void *y, void *stream);

/* Bytes of device workspace gbconv_bwd_filter needs for this descriptor (a multiple of 256; may be 0).
 * Launches nothing.  Returns GBCONV_EINVAL for a NULL argument or a shape the forward would reject. */
gbconv_status gbconv_bwd_filter_workspace(const gbconv_desc *desc, int64_t *bytes);

/* Weight gradient of the forward convolution described by desc, and its bias gradient when db != NULL.
 *   x         : device, forward input, desc->layout, desc->dtype
 *   dy        : device, forward-output shape, desc->dtype
 *   dw        : device, the forward weight's shape per desc->wlayout, desc->dtype; fully overwritten
 *               (no need to zero it).  Sums are kept in fp32 and rounded once to desc->dtype.
 *   db        : device float [C_out], fully overwritten, or NULL for no bias gradient
 *   workspace : device scratch of at least gbconv_bwd_filter_workspace(desc) bytes, 16-byte aligned, owned
 *               by the caller; its contents are undefined afterwards.  NULL is allowed when 0 bytes are needed.
 * The sum over batch and positions is cut into fixed chunks; each chunk's partial sums are taken in a
 * fixed order and the chunk sums are added in a fixed order (sixteen runs of consecutive chunks, each in
 * chunk order, then the runs in order), so the same inputs give bitwise-equal dw and db.
 * Enqueues two kernels on `stream` (partial sums, ordered reduction), three when the tensor-core path also
 * computes db.  Returns GBCONV_EINVAL for NULL tensors or a workspace smaller than required. */
gbconv_status gbconv_bwd_filter(const gbconv_desc *desc, const void *x, const void *dy, void *dw, float *db,
                                void *workspace, int64_t workspace_bytes, void *stream);

/* Size of the scratch array gbconv_bwd_filter_noalloc uses: 32 MiB. */
#define GBCONV_NOALLOC_WORKSPACE_BYTES (32u << 20)

/* Weight gradient without any device allocation, for callers that cannot allocate device memory
 * (for example code that runs inside an allocator's own callbacks, a plugin that is handed only its
 * tensors, or an application that reserves all device memory up front and forbids further
 * allocations), and so cannot supply the workspace gbconv_bwd_filter asks for.  The source pages have
 * no counterpart: their weight gradients either accumulate with atomics or allocate their own buffers.
 *
 * Same arguments, results and determinism as gbconv_bwd_filter, minus the workspace: the partial sums
 * go to a fixed array of GBCONV_NOALLOC_WORKSPACE_BYTES in device global memory that the library
 * declares statically.  Every GPU that loads the library holds that array until the process exits.
 *  - Calls no cudaMalloc, cudaFree or other allocating routine.
 *  - Returns GBCONV_EUNSUPPORTED when gbconv_bwd_filter_workspace(desc) exceeds
 *    GBCONV_NOALLOC_WORKSPACE_BYTES (use gbconv_bwd_filter with your own workspace then), and
 *    GBCONV_EINVAL for NULL tensors or a shape the forward would reject.
 *  - The first call on each device looks up the array's device address (cudaGetSymbolAddress, with
 *    that device current) and caches it; make that first call before any stream capture.
 *  - Every call on a device shares the one array, which keeps the last call's contents (nothing has
 *    to start at zero: each call writes every partial sum before reading it).  Calls whose kernels
 *    overlap on the GPU (other streams, other host threads) race on the array and give wrong results:
 *    order them on one stream or synchronise between them.
 * Enqueues the same kernels as gbconv_bwd_filter on `stream`. */
gbconv_status gbconv_bwd_filter_noalloc(const gbconv_desc *desc, const void *x, const void *dy, void *dw, float *db,
                                        void *stream);

/* Re-lays a weight from [C_out, C_in/G, KH, KW] (OIHW) into [C_out, KH, KW, C_in/G] (OHWI), the order the
 * NHWC tensor-core kernels read.  desc->dtype gives the element type; desc->wlayout is ignored.
 * w_oihw and w_ohwi are device pointers that must not overlap.  Enqueues one kernel. */
gbconv_status gbconv_pack_weight(const gbconv_desc *desc, const void *w_oihw, void *w_ohwi, void *stream);

/* Synchronises `stream`, then returns GBCONV_ETIMEOUT if any kernel of this library on the current
 * device recorded an expired internal wait since the last call (and clears the record), else GBCONV_OK
 * (or GBCONV_ECUDA if the synchronisation itself failed). */
gbconv_status gbconv_device_status(void *stream);

/* Sets how long any internal barrier wait of the library's kernels may take before the kernel gives
 * up (records GBCONV_ETIMEOUT for gbconv_device_status, drains its copies and tensor-core work in
 * flight, frees its tensor memory and returns), for kernels enqueued from now on, in this process.
 * ns <= 0 restores the default, 2 s.  No correct launch comes near the default; a short limit is
 * for exercising the failure path.  Returns the previous limit.  The source pages have no
 * counterpart (their kernels have no bounded waits).  Launches nothing. */
int64_t gbconv_set_wait_limit_ns(int64_t ns);

/* Number of kernels this library has enqueued in this process (all devices, all streams). */
uint64_t gbconv_kernels_launched(void);

/* Static, human-readable name of a status code. */
const char *gbconv_status_string(gbconv_status status);

#ifdef __cplusplus
}
#endif

#endif /* GBCONV_H */
