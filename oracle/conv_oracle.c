/*
 * Convolution oracle: the plain, slow, FP64 definition of N-D (1-D, 2-D and
 * 3-D) convolution forward, of its input gradient (dgrad), and of its weight and
 * bias gradients (wgrad).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * Inputs arrive as float32 arrays (bf16 and f32 values are both exactly
 * representable in float32), every product and sum is taken in double, and
 * results are returned as double.  Loops are plain nested loops in the order
 * the definitions below state them; there is no blocking, no reordering and
 * no fusion.
 *
 * Definitions followed (cited by page title and item):
 *  - Output size: oarust 0.8.6 `src/rs/ml/matrix/conv.rs`,
 *    `Conv1dGeometry::resolve` (effective kernel = (k-1)*dil + 1, reject a
 *    padded input shorter than it, out = (in + 2*pad - eff) / stride + 1 with
 *    integer floor division).  The 2-D rule is the same per spatial axis.
 *    With burn-cubecl's (begin, end) padding pairs the padded length is
 *    in + pad_begin + pad_end, and reads use the begin side.
 *  - Spatial rank: burn-cubecl's convolutions take `ConvOptions<N>` with one
 *    stride / padding / dilation per spatial axis and the same index map on
 *    every axis; 3-D is the same sums with a depth axis added.  1-D and 2-D
 *    shapes are carried here as 3-D ones with depth 1.
 *  - Index map: burn-cubecl `src/kernel/conv/im2col.rs`, doc of `im2col`
 *    (input position = out*stride + k*dilation - padding, zero outside the
 *    image; no kernel flip: cross-correlation).
 *  - Groups: teeny-kernels `src/nn/conv/conv2d.rs`, `conv2d_forward`
 *    (c_in_per_group = C_IN/G, group = c_out / (C_OUT/G), weight
 *    [C_OUT, C_IN/G, KH, KW]).
 *  - Bias: teeny-kernels `conv2d_bias_forward` (bias[c_out] added once, after
 *    the reduction).
 *  - Data gradient, scatter form: teeny-kernels `conv2d_backward_dx`
 *    (dx[b, c_in, oh*S + kh - P, ow*S + kw - P] += dy[b, c_out, oh, ow] *
 *    w[c_out, c_in_local, kh, kw], out-of-image positions skipped).
 *  - Data gradient, gather form: oarust `conv_2d_backward` dispatches its
 *    input-gradient pass over input elements; the gather form here is the
 *    exact transpose of the scatter form above.
 *  - Weight gradient: burn-cubecl `wgrad_im2col` (the weight gradient is the
 *    contraction of the output gradient with the input's columns over every
 *    (batch, output position), columns read at out*stride + k*dilation -
 *    padding and zero outside the image) and teeny-kernels
 *    `conv2d_backward_dw` (one sum per (c_out, c_in_local, kh, kw) of dy
 *    times the x element the forward multiplied by that weight).
 *  - Bias gradient: oarust `conv_2d_backward` returns, beside the input and
 *    weight gradients, the gradient of the bias: the sum of the output
 *    gradient over batch and positions, per output channel.
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL 1

typedef struct {
  int64_t n, c_in, c_out, groups;
  int64_t in_h, in_w;    /* 1-D convolution: in_h = 1, k_h = 1, s_h = 1, p_h = 0, d_h = 1 */
  int64_t k_h, k_w;
  int64_t s_h, s_w;
  int64_t p_h, p_w;
  int64_t d_h, d_w;
  int64_t p_h_end, p_w_end;  /* padding after each axis (p_h, p_w are before it) */
  int64_t in_d, k_d, s_d, p_d, p_d_end, d_d;  /* depth axis; 1, 1, 1, 0, 0, 1 for 1-D and 2-D */
  int32_t nhwc;          /* 0: NC(D)HW / NCL activations, 1: N(D)HWC / NLC activations */
  int32_t w_ohwi;        /* 0: OI(D)HW / OIK weight [C_out, C_in/G, (KD,) KH, KW], 1: O(D)HWI [C_out, (KD,) KH, KW, C_in/G] */
} oracle_conv;

/* Output length along one axis, or ORACLE_EINVAL when the effective kernel
 * does not fit the padded input (oarust Conv1dGeometry::resolve). */
int oracle_out_size(int64_t in, int64_t k, int64_t s, int64_t p, int64_t d, int64_t *out) {
  if (in <= 0 || k <= 0 || s <= 0 || d <= 0 || p < 0) return ORACLE_EINVAL;
  int64_t eff = (k - 1) * d + 1;
  int64_t padded = in + 2 * p;
  if (padded < eff) return ORACLE_EINVAL;
  *out = (padded - eff) / s + 1;
  return ORACLE_OK;
}

/* As oracle_out_size, with p_begin zeros before the axis and p_end after it. */
int oracle_out_size2(int64_t in, int64_t k, int64_t s, int64_t p_begin, int64_t p_end, int64_t d, int64_t *out) {
  if (in <= 0 || k <= 0 || s <= 0 || d <= 0 || p_begin < 0 || p_end < 0) return ORACLE_EINVAL;
  int64_t eff = (k - 1) * d + 1;
  int64_t padded = in + p_begin + p_end;
  if (padded < eff) return ORACLE_EINVAL;
  *out = (padded - eff) / s + 1;
  return ORACLE_OK;
}

/* Shape checks of oarust Conv1dGeometry / Conv2dGeometry::resolve: nonzero
 * extents, nonzero stride, dilation and groups, channels divisible by groups. */
int oracle_check(const oracle_conv *c, int64_t *oh, int64_t *ow) {
  if (c->n <= 0 || c->c_in <= 0 || c->c_out <= 0 || c->groups <= 0) return ORACLE_EINVAL;
  if (c->c_in % c->groups != 0 || c->c_out % c->groups != 0) return ORACLE_EINVAL;
  if (oracle_out_size2(c->in_h, c->k_h, c->s_h, c->p_h, c->p_h_end, c->d_h, oh) != ORACLE_OK) return ORACLE_EINVAL;
  if (oracle_out_size2(c->in_w, c->k_w, c->s_w, c->p_w, c->p_w_end, c->d_w, ow) != ORACLE_OK) return ORACLE_EINVAL;
  int64_t od;
  if (oracle_out_size2(c->in_d, c->k_d, c->s_d, c->p_d, c->p_d_end, c->d_d, &od) != ORACLE_OK) return ORACLE_EINVAL;
  return ORACLE_OK;
}

/* Output depth (1 for 1-D and 2-D shapes). */
static int64_t out_depth(const oracle_conv *c) {
  return (c->in_d + c->p_d + c->p_d_end - ((c->k_d - 1) * c->d_d + 1)) / c->s_d + 1;
}

/* Offset of activation element (n, c, d, h, w) in a tensor of C channels and D x H x W spatial
 * extent, in the layout the descriptor names (D = 1 for 1-D and 2-D shapes). */
static int64_t act_index(const oracle_conv *c, int64_t C, int64_t D, int64_t H, int64_t W,
                         int64_t n, int64_t ch, int64_t d, int64_t h, int64_t w) {
  if (c->nhwc) return (((n * D + d) * H + h) * W + w) * C + ch;
  return (((n * C + ch) * D + d) * H + h) * W + w;
}

/* Offset of weight element (co, c_local, kd, kh, kw). */
static int64_t w_index(const oracle_conv *c, int64_t co, int64_t cl, int64_t kd, int64_t kh, int64_t kw) {
  int64_t cpg = c->c_in / c->groups;
  if (c->w_ohwi) return (((co * c->k_d + kd) * c->k_h + kh) * c->k_w + kw) * cpg + cl;
  return (((co * cpg + cl) * c->k_d + kd) * c->k_h + kh) * c->k_w + kw;
}

/* One forward output y[n, co, od, oh, ow]:
 *   bias[co] + sum over c_local < C_in/G, kd, kh, kw of
 *   x[n, g*C_in/G + c_local, od*s_d + kd*d_d - p_d, oh*s_h + kh*d_h - p_h, ow*s_w + kw*d_w - p_w]
 *     * w[co, c_local, kd, kh, kw]
 * with g = co / (C_out/G) and out-of-image x taken as zero. */
double oracle_conv_fwd_at3(const oracle_conv *c, const float *x, const float *w, const float *bias,
                           int64_t n, int64_t co, int64_t od, int64_t oh, int64_t ow) {
  int64_t cpg = c->c_in / c->groups;
  int64_t g = co / (c->c_out / c->groups);
  double acc = 0.0;
  for (int64_t cl = 0; cl < cpg; ++cl) {
    int64_t ci = g * cpg + cl;
    for (int64_t kd = 0; kd < c->k_d; ++kd) {
      int64_t id = od * c->s_d + kd * c->d_d - c->p_d;
      if (id < 0 || id >= c->in_d) continue;
      for (int64_t kh = 0; kh < c->k_h; ++kh) {
        int64_t ih = oh * c->s_h + kh * c->d_h - c->p_h;
        if (ih < 0 || ih >= c->in_h) continue;
        for (int64_t kw = 0; kw < c->k_w; ++kw) {
          int64_t iw = ow * c->s_w + kw * c->d_w - c->p_w;
          if (iw < 0 || iw >= c->in_w) continue;
          double xv = (double)x[act_index(c, c->c_in, c->in_d, c->in_h, c->in_w, n, ci, id, ih, iw)];
          double wv = (double)w[w_index(c, co, cl, kd, kh, kw)];
          acc += xv * wv;
        }
      }
    }
  }
  if (bias) acc += (double)bias[co];
  return acc;
}

double oracle_conv_fwd_at(const oracle_conv *c, const float *x, const float *w, const float *bias,
                          int64_t n, int64_t co, int64_t oh, int64_t ow) {
  return oracle_conv_fwd_at3(c, x, w, bias, n, co, 0, oh, ow);
}

/* Whole forward output, written in the descriptor's activation layout. */
int oracle_conv_fwd(const oracle_conv *c, const float *x, const float *w, const float *bias, double *y) {
  int64_t OH, OW;
  if (oracle_check(c, &OH, &OW) != ORACLE_OK) return ORACLE_EINVAL;
  int64_t OD = out_depth(c);
  for (int64_t n = 0; n < c->n; ++n)
    for (int64_t co = 0; co < c->c_out; ++co)
      for (int64_t od = 0; od < OD; ++od)
        for (int64_t oh = 0; oh < OH; ++oh)
          for (int64_t ow = 0; ow < OW; ++ow)
            y[act_index(c, c->c_out, OD, OH, OW, n, co, od, oh, ow)] =
                oracle_conv_fwd_at3(c, x, w, bias, n, co, od, oh, ow);
  return ORACLE_OK;
}

/* The output position a tap of the forward reads input position i from, along one axis: o with
 * o*s + k*d - p == i, or -1 when there is none inside [0, O). */
static int64_t tap_source(int64_t i, int64_t k, int64_t s, int64_t p, int64_t d, int64_t O) {
  int64_t t = i + p - k * d;
  if (t < 0 || t % s != 0) return -1;
  return t / s < O ? t / s : -1;
}

/* One input-gradient element dx[n, ci, id, ih, iw], gather form:
 *   sum over co in ci's group, kd, kh, kw of dy[n, co, od, oh, ow] * w[co, ci - g*C_in/G, kd, kh, kw]
 * over the taps where od = (id + p_d - kd*d_d) / s_d is an exact integer in [0, OD) (and likewise
 * oh, ow).  These are exactly the (od, oh, ow, kd, kh, kw) whose forward read lands on (id, ih, iw). */
double oracle_conv_dgrad_at3(const oracle_conv *c, const float *dy, const float *w,
                             int64_t n, int64_t ci, int64_t id, int64_t ih, int64_t iw) {
  int64_t OH, OW;
  if (oracle_check(c, &OH, &OW) != ORACLE_OK) return 0.0;
  int64_t OD = out_depth(c);
  int64_t cpg = c->c_in / c->groups;
  int64_t opg = c->c_out / c->groups;
  int64_t g = ci / cpg;
  int64_t cl = ci - g * cpg;
  double acc = 0.0;
  for (int64_t co = g * opg; co < (g + 1) * opg; ++co)
    for (int64_t kd = 0; kd < c->k_d; ++kd) {
      int64_t od = tap_source(id, kd, c->s_d, c->p_d, c->d_d, OD);
      if (od < 0) continue;
      for (int64_t kh = 0; kh < c->k_h; ++kh) {
        int64_t oh = tap_source(ih, kh, c->s_h, c->p_h, c->d_h, OH);
        if (oh < 0) continue;
        for (int64_t kw = 0; kw < c->k_w; ++kw) {
          int64_t ow = tap_source(iw, kw, c->s_w, c->p_w, c->d_w, OW);
          if (ow < 0) continue;
          double gv = (double)dy[act_index(c, c->c_out, OD, OH, OW, n, co, od, oh, ow)];
          double wv = (double)w[w_index(c, co, cl, kd, kh, kw)];
          acc += gv * wv;
        }
      }
    }
  return acc;
}

double oracle_conv_dgrad_at(const oracle_conv *c, const float *dy, const float *w,
                            int64_t n, int64_t ci, int64_t ih, int64_t iw) {
  return oracle_conv_dgrad_at3(c, dy, w, n, ci, 0, ih, iw);
}

/* Whole input gradient, gather form, in the descriptor's activation layout. */
int oracle_conv_dgrad(const oracle_conv *c, const float *dy, const float *w, double *dx) {
  int64_t OH, OW;
  if (oracle_check(c, &OH, &OW) != ORACLE_OK) return ORACLE_EINVAL;
  for (int64_t n = 0; n < c->n; ++n)
    for (int64_t ci = 0; ci < c->c_in; ++ci)
      for (int64_t id = 0; id < c->in_d; ++id)
        for (int64_t ih = 0; ih < c->in_h; ++ih)
          for (int64_t iw = 0; iw < c->in_w; ++iw)
            dx[act_index(c, c->c_in, c->in_d, c->in_h, c->in_w, n, ci, id, ih, iw)] =
                oracle_conv_dgrad_at3(c, dy, w, n, ci, id, ih, iw);
  return ORACLE_OK;
}

/* Whole input gradient, scatter form: the loop structure of teeny-kernels
 * `conv2d_backward_dx`, run serially in double.  Walks the output gradient
 * and adds dy * w into every in-image input position the forward read from. */
int oracle_conv_dgrad_scatter(const oracle_conv *c, const float *dy, const float *w, double *dx) {
  int64_t OH, OW;
  if (oracle_check(c, &OH, &OW) != ORACLE_OK) return ORACLE_EINVAL;
  int64_t OD = out_depth(c);
  int64_t cpg = c->c_in / c->groups;
  int64_t opg = c->c_out / c->groups;
  int64_t total = c->n * c->c_in * c->in_d * c->in_h * c->in_w;
  for (int64_t i = 0; i < total; ++i) dx[i] = 0.0;
  for (int64_t n = 0; n < c->n; ++n)
    for (int64_t co = 0; co < c->c_out; ++co) {
      int64_t g = co / opg;
      for (int64_t od = 0; od < OD; ++od)
        for (int64_t oh = 0; oh < OH; ++oh)
          for (int64_t ow = 0; ow < OW; ++ow) {
            double gv = (double)dy[act_index(c, c->c_out, OD, OH, OW, n, co, od, oh, ow)];
            for (int64_t cl = 0; cl < cpg; ++cl)
              for (int64_t kd = 0; kd < c->k_d; ++kd) {
                int64_t id = od * c->s_d + kd * c->d_d - c->p_d;
                if (id < 0 || id >= c->in_d) continue;
                for (int64_t kh = 0; kh < c->k_h; ++kh) {
                  int64_t ih = oh * c->s_h + kh * c->d_h - c->p_h;
                  if (ih < 0 || ih >= c->in_h) continue;
                  for (int64_t kw = 0; kw < c->k_w; ++kw) {
                    int64_t iw = ow * c->s_w + kw * c->d_w - c->p_w;
                    if (iw < 0 || iw >= c->in_w) continue;
                    dx[act_index(c, c->c_in, c->in_d, c->in_h, c->in_w, n, g * cpg + cl, id, ih, iw)] +=
                        gv * (double)w[w_index(c, co, cl, kd, kh, kw)];
                  }
                }
              }
          }
    }
  return ORACLE_OK;
}

/* One weight-gradient element dw[co, c_local, kd, kh, kw]:
 *   sum over n < N, od < OD, oh < OH, ow < OW of
 *   dy[n, co, od, oh, ow] * x[n, g*C_in/G + c_local, od*s_d + kd*d_d - p_d, oh*s_h + kh*d_h - p_h,
 *                             ow*s_w + kw*d_w - p_w]
 * with g = co / (C_out/G) and out-of-image x taken as zero (those terms are skipped). */
double oracle_conv_wgrad_at3(const oracle_conv *c, const float *x, const float *dy,
                             int64_t co, int64_t cl, int64_t kd, int64_t kh, int64_t kw) {
  int64_t OH, OW;
  if (oracle_check(c, &OH, &OW) != ORACLE_OK) return 0.0;
  int64_t OD = out_depth(c);
  int64_t cpg = c->c_in / c->groups;
  int64_t g = co / (c->c_out / c->groups);
  int64_t ci = g * cpg + cl;
  double acc = 0.0;
  for (int64_t n = 0; n < c->n; ++n)
    for (int64_t od = 0; od < OD; ++od) {
      int64_t id = od * c->s_d + kd * c->d_d - c->p_d;
      if (id < 0 || id >= c->in_d) continue;
      for (int64_t oh = 0; oh < OH; ++oh) {
        int64_t ih = oh * c->s_h + kh * c->d_h - c->p_h;
        if (ih < 0 || ih >= c->in_h) continue;
        for (int64_t ow = 0; ow < OW; ++ow) {
          int64_t iw = ow * c->s_w + kw * c->d_w - c->p_w;
          if (iw < 0 || iw >= c->in_w) continue;
          double gv = (double)dy[act_index(c, c->c_out, OD, OH, OW, n, co, od, oh, ow)];
          double xv = (double)x[act_index(c, c->c_in, c->in_d, c->in_h, c->in_w, n, ci, id, ih, iw)];
          acc += gv * xv;
        }
      }
    }
  return acc;
}

double oracle_conv_wgrad_at(const oracle_conv *c, const float *x, const float *dy,
                            int64_t co, int64_t cl, int64_t kh, int64_t kw) {
  return oracle_conv_wgrad_at3(c, x, dy, co, cl, 0, kh, kw);
}

/* Whole weight gradient, in the descriptor's weight layout. */
int oracle_conv_wgrad(const oracle_conv *c, const float *x, const float *dy, double *dw) {
  int64_t OH, OW;
  if (oracle_check(c, &OH, &OW) != ORACLE_OK) return ORACLE_EINVAL;
  int64_t cpg = c->c_in / c->groups;
  for (int64_t co = 0; co < c->c_out; ++co)
    for (int64_t cl = 0; cl < cpg; ++cl)
      for (int64_t kd = 0; kd < c->k_d; ++kd)
        for (int64_t kh = 0; kh < c->k_h; ++kh)
          for (int64_t kw = 0; kw < c->k_w; ++kw)
            dw[w_index(c, co, cl, kd, kh, kw)] = oracle_conv_wgrad_at3(c, x, dy, co, cl, kd, kh, kw);
  return ORACLE_OK;
}

/* Bias gradient db[co] = sum over n, od, oh, ow of dy[n, co, od, oh, ow]. */
int oracle_conv_bgrad(const oracle_conv *c, const float *dy, double *db) {
  int64_t OH, OW;
  if (oracle_check(c, &OH, &OW) != ORACLE_OK) return ORACLE_EINVAL;
  int64_t OD = out_depth(c);
  for (int64_t co = 0; co < c->c_out; ++co) {
    double acc = 0.0;
    for (int64_t n = 0; n < c->n; ++n)
      for (int64_t od = 0; od < OD; ++od)
        for (int64_t oh = 0; oh < OH; ++oh)
          for (int64_t ow = 0; ow < OW; ++ow)
            acc += (double)dy[act_index(c, c->c_out, OD, OH, OW, n, co, od, oh, ow)];
    db[co] = acc;
  }
  return ORACLE_OK;
}

/* Batched point queries: out[i] = fwd (or dgrad) at the i-th (n, c, h, w)
 * quadruple of idx (depth 0), or the i-th (n, c, d, h, w) quintuple for the
 * *_points3 forms.  Used for sampled checks at sizes where a whole pass
 * would take too long. */
void oracle_conv_fwd_points(const oracle_conv *c, const float *x, const float *w, const float *bias,
                            const int64_t *idx, int64_t count, double *out) {
  for (int64_t i = 0; i < count; ++i)
    out[i] = oracle_conv_fwd_at(c, x, w, bias, idx[4 * i], idx[4 * i + 1], idx[4 * i + 2], idx[4 * i + 3]);
}

void oracle_conv_dgrad_points(const oracle_conv *c, const float *dy, const float *w,
                              const int64_t *idx, int64_t count, double *out) {
  for (int64_t i = 0; i < count; ++i)
    out[i] = oracle_conv_dgrad_at(c, dy, w, idx[4 * i], idx[4 * i + 1], idx[4 * i + 2], idx[4 * i + 3]);
}

/* Batched point queries of the weight gradient: out[i] = dw at the i-th
 * (co, c_local, kh, kw) quadruple of idx (kd = 0). */
void oracle_conv_wgrad_points(const oracle_conv *c, const float *x, const float *dy,
                              const int64_t *idx, int64_t count, double *out) {
  for (int64_t i = 0; i < count; ++i)
    out[i] = oracle_conv_wgrad_at(c, x, dy, idx[4 * i], idx[4 * i + 1], idx[4 * i + 2], idx[4 * i + 3]);
}

/* 3-D point queries: out[i] = fwd at the i-th (n, c, d, h, w) quintuple of idx. */
void oracle_conv_fwd_points3(const oracle_conv *c, const float *x, const float *w, const float *bias,
                             const int64_t *idx, int64_t count, double *out) {
  for (int64_t i = 0; i < count; ++i)
    out[i] = oracle_conv_fwd_at3(c, x, w, bias, idx[5 * i], idx[5 * i + 1], idx[5 * i + 2], idx[5 * i + 3],
                                 idx[5 * i + 4]);
}

/* 3-D point queries of the weight gradient: out[i] = dw at the i-th (co, c_local, kd, kh, kw)
 * quintuple of idx. */
void oracle_conv_wgrad_points3(const oracle_conv *c, const float *x, const float *dy,
                               const int64_t *idx, int64_t count, double *out) {
  for (int64_t i = 0; i < count; ++i)
    out[i] = oracle_conv_wgrad_at3(c, x, dy, idx[5 * i], idx[5 * i + 1], idx[5 * i + 2], idx[5 * i + 3],
                                   idx[5 * i + 4]);
}

/* 3-D point queries of the input gradient: out[i] = dx at the i-th (n, c, d, h, w) quintuple of idx. */
void oracle_conv_dgrad_points3(const oracle_conv *c, const float *dy, const float *w,
                               const int64_t *idx, int64_t count, double *out) {
  for (int64_t i = 0; i < count; ++i)
    out[i] = oracle_conv_dgrad_at3(c, dy, w, idx[5 * i], idx[5 * i + 1], idx[5 * i + 2], idx[5 * i + 3],
                                   idx[5 * i + 4]);
}
