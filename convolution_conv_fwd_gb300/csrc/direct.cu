// Generic direct convolution on CUDA cores: any layout, element type, group
// count, stride, padding and dilation.  One thread per output element, fp32
// accumulation.  This family serves the conv1d fp32 NCL workload and every
// shape the specialised families do not take.
//
// Forward follows teeny-kernels `src/nn/conv/conv2d.rs`, `conv2d_forward`
// (group window, per-tap read position oh*stride + kh*dil - pad, zero
// outside, bias after the reduction as in `conv2d_bias_forward`), with
// dilation per oarust `Conv1dGeometry`.  The input gradient is the gather
// form: each thread owns one dx element and sums the (dy, w) products whose
// forward read lands on it, so nothing is accumulated atomically.  Shapes are
// 3-D (burn-cubecl `ConvOptions<N>`: the same index map on every spatial
// axis); 1-D and 2-D ones have depth 1.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "problem.h"
#include "ptx.cuh"

namespace gbconv {
namespace {

struct DirectArgs {
  int N, Cin, Cout, G, H, W, KH, KW, SH, SW, PH, PW, DH, DW, OH, OW;
  int D, KD, SD, PD, DD, OD;  // depth axis (1, 1, 1, 0, 1, 1 for 1-D and 2-D shapes)
  int nhwc, ohwi;
};

template <typename T> __device__ __forceinline__ float ld(const T* p, int i);
template <> __device__ __forceinline__ float ld<float>(const float* p, int i) { return __ldg(p + i); }
template <> __device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16* p, int i) {
  return __bfloat162float(p[i]);
}
template <typename T> __device__ __forceinline__ T cvt(float v);
template <> __device__ __forceinline__ float cvt<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 cvt<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

__device__ __forceinline__ int act_off(const DirectArgs& a, int C, int D, int H, int W, int n, int c, int d, int h,
                                       int w) {
  return a.nhwc ? (((n * D + d) * H + h) * W + w) * C + c : (((n * C + c) * D + d) * H + h) * W + w;
}

__device__ __forceinline__ int w_off(const DirectArgs& a, int co, int cl, int kd, int kh, int kw) {
  const int cpg = a.Cin / a.G;
  return a.ohwi ? (((co * a.KD + kd) * a.KH + kh) * a.KW + kw) * cpg + cl
                : (((co * cpg + cl) * a.KD + kd) * a.KH + kh) * a.KW + kw;
}

template <typename T>
__global__ void direct_fwd_kernel(DirectArgs a, const T* __restrict__ x, const T* __restrict__ w,
                                  const float* __restrict__ bias, T* __restrict__ y) {
  ptx::grid_dep_wait();  // inputs may come from the previous kernel on the stream
  ptx::grid_dep_launch();
  const int total = a.N * a.Cout * a.OD * a.OH * a.OW;
  const int cpg = a.Cin / a.G, opg = a.Cout / a.G;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    int n, co, od, oh, ow;
    if (a.nhwc) {  // channel fastest, so a warp writes contiguous channels
      co = i % a.Cout;
      int r = i / a.Cout;
      ow = r % a.OW; r /= a.OW;
      oh = r % a.OH; r /= a.OH;
      od = r % a.OD; n = r / a.OD;
    } else {
      ow = i % a.OW;
      int r = i / a.OW;
      oh = r % a.OH; r /= a.OH;
      od = r % a.OD; r /= a.OD;
      co = r % a.Cout; n = r / a.Cout;
    }
    const int g = co / opg;
    float acc = 0.f;
    for (int cl = 0; cl < cpg; ++cl) {
      const int ci = g * cpg + cl;
      for (int kd = 0; kd < a.KD; ++kd) {
        const int id = od * a.SD + kd * a.DD - a.PD;
        if (id < 0 || id >= a.D) continue;
        for (int kh = 0; kh < a.KH; ++kh) {
          const int ih = oh * a.SH + kh * a.DH - a.PH;
          if (ih < 0 || ih >= a.H) continue;
          for (int kw = 0; kw < a.KW; ++kw) {
            const int iw = ow * a.SW + kw * a.DW - a.PW;
            if (iw < 0 || iw >= a.W) continue;
            acc = fmaf(ld(x, act_off(a, a.Cin, a.D, a.H, a.W, n, ci, id, ih, iw)), ld(w, w_off(a, co, cl, kd, kh, kw)),
                       acc);
          }
        }
      }
    }
    if (bias) acc += __ldg(bias + co);
    y[act_off(a, a.Cout, a.OD, a.OH, a.OW, n, co, od, oh, ow)] = cvt<T>(acc);
  }
}

// Small problems: when the whole input and weight fit in shared memory and every output fits one
// block, the block first stages both as fp32, all its threads loading at once, and then each output's
// taps read shared memory.  A launch-latency-bound shape (the fp32 conv1d workload: 12 kFLOP) then
// pays one round trip to memory instead of one dependent global load per tap.
constexpr int kSmallFloats = 8192;   // staged x + w, 32 KB
constexpr int kSmallThreads = 1024;  // one block; each thread takes up to kSmallOutPerThread outputs
constexpr int kSmallOutPerThread = 4;

template <typename T>
__global__ void __launch_bounds__(kSmallThreads) direct_fwd_small_kernel(DirectArgs a, const T* __restrict__ x,
                                                                         const T* __restrict__ w,
                                                                         const float* __restrict__ bias,
                                                                         T* __restrict__ y, int nx, int nw) {
  extern __shared__ float stage[];
  float* xs = stage;
  float* ws = stage + nx;
  ptx::grid_dep_wait();  // inputs may come from the previous kernel on the stream
  ptx::grid_dep_launch();
  for (int i = threadIdx.x; i < nx; i += blockDim.x) xs[i] = ld(x, i);
  for (int i = threadIdx.x; i < nw; i += blockDim.x) ws[i] = ld(w, i);
  __syncthreads();
  const int total = a.N * a.Cout * a.OD * a.OH * a.OW;
  const int cpg = a.Cin / a.G, opg = a.Cout / a.G;
  for (int i = threadIdx.x; i < total; i += blockDim.x) {
    int n, co, od, oh, ow;
    if (a.nhwc) {
      co = i % a.Cout;
      int r = i / a.Cout;
      ow = r % a.OW; r /= a.OW;
      oh = r % a.OH; r /= a.OH;
      od = r % a.OD; n = r / a.OD;
    } else {
      ow = i % a.OW;
      int r = i / a.OW;
      oh = r % a.OH; r /= a.OH;
      od = r % a.OD; r /= a.OD;
      co = r % a.Cout; n = r / a.Cout;
    }
    const int g = co / opg;
    float acc = 0.f;  // the same terms in the same order as direct_fwd_kernel
    for (int cl = 0; cl < cpg; ++cl) {
      const int ci = g * cpg + cl;
      for (int kd = 0; kd < a.KD; ++kd) {
        const int id = od * a.SD + kd * a.DD - a.PD;
        if (id < 0 || id >= a.D) continue;
        for (int kh = 0; kh < a.KH; ++kh) {
          const int ih = oh * a.SH + kh * a.DH - a.PH;
          if (ih < 0 || ih >= a.H) continue;
          for (int kw = 0; kw < a.KW; ++kw) {
            const int iw = ow * a.SW + kw * a.DW - a.PW;
            if (iw < 0 || iw >= a.W) continue;
            acc = fmaf(xs[act_off(a, a.Cin, a.D, a.H, a.W, n, ci, id, ih, iw)], ws[w_off(a, co, cl, kd, kh, kw)], acc);
          }
        }
      }
    }
    if (bias) acc += __ldg(bias + co);
    y[act_off(a, a.Cout, a.OD, a.OH, a.OW, n, co, od, oh, ow)] = cvt<T>(acc);
  }
}

template <typename T>
__global__ void direct_dgrad_kernel(DirectArgs a, const T* __restrict__ dy, const T* __restrict__ w,
                                    const float* __restrict__ bias, T* __restrict__ dx) {
  ptx::grid_dep_wait();  // inputs may come from the previous kernel on the stream
  ptx::grid_dep_launch();
  const int total = a.N * a.Cin * a.D * a.H * a.W;
  const int cpg = a.Cin / a.G, opg = a.Cout / a.G;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    int n, ci, id, ih, iw;
    if (a.nhwc) {
      ci = i % a.Cin;
      int r = i / a.Cin;
      iw = r % a.W; r /= a.W;
      ih = r % a.H; r /= a.H;
      id = r % a.D; n = r / a.D;
    } else {
      iw = i % a.W;
      int r = i / a.W;
      ih = r % a.H; r /= a.H;
      id = r % a.D; r /= a.D;
      ci = r % a.Cin; n = r / a.Cin;
    }
    const int g = ci / cpg, cl = ci - g * cpg;
    float acc = 0.f;
    for (int co = g * opg; co < (g + 1) * opg; ++co) {
      for (int kd = 0; kd < a.KD; ++kd) {
        const int td = id + a.PD - kd * a.DD;
        if (td < 0 || td % a.SD != 0) continue;
        const int od = td / a.SD;
        if (od >= a.OD) continue;
        for (int kh = 0; kh < a.KH; ++kh) {
          const int th = ih + a.PH - kh * a.DH;
          if (th < 0 || th % a.SH != 0) continue;
          const int oh = th / a.SH;
          if (oh >= a.OH) continue;
          for (int kw = 0; kw < a.KW; ++kw) {
            const int tw = iw + a.PW - kw * a.DW;
            if (tw < 0 || tw % a.SW != 0) continue;
            const int ow = tw / a.SW;
            if (ow >= a.OW) continue;
            acc = fmaf(ld(dy, act_off(a, a.Cout, a.OD, a.OH, a.OW, n, co, od, oh, ow)),
                       ld(w, w_off(a, co, cl, kd, kh, kw)), acc);
          }
        }
      }
    }
    if (bias) acc += __ldg(bias + ci);
    dx[act_off(a, a.Cin, a.D, a.H, a.W, n, ci, id, ih, iw)] = cvt<T>(acc);
  }
}

// [C_out, C_in/G, KH, KW] -> [C_out, KH, KW, C_in/G]; one thread per destination element.  A 3-D
// weight is the same re-layout with the kernel's depth and height taken as one axis of KD*KH.
template <typename T>
__global__ void pack_ohwi_kernel(int Cout, int cpg, int KH, int KW, const T* __restrict__ src, T* __restrict__ dst) {
  ptx::grid_dep_wait();  // inputs may come from the previous kernel on the stream
  ptx::grid_dep_launch();
  const int total = Cout * cpg * KH * KW;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int cl = i % cpg;
    int r = i / cpg;
    const int kw = r % KW; r /= KW;
    const int kh = r % KH;
    const int co = r / KH;
    dst[i] = src[((co * cpg + cl) * KH + kh) * KW + kw];
  }
}

DirectArgs make_args(const Problem& p) {
  DirectArgs a;
  a.N = int(p.N); a.Cin = int(p.Cin); a.Cout = int(p.Cout); a.G = int(p.G);
  a.H = int(p.H); a.W = int(p.W); a.KH = int(p.KH); a.KW = int(p.KW);
  a.SH = int(p.SH); a.SW = int(p.SW); a.PH = int(p.PH); a.PW = int(p.PW);
  a.DH = int(p.DH); a.DW = int(p.DW); a.OH = int(p.OH); a.OW = int(p.OW);
  a.D = int(p.D); a.KD = int(p.KD); a.SD = int(p.SD); a.PD = int(p.PD); a.DD = int(p.DD); a.OD = int(p.OD);
  a.nhwc = p.nhwc; a.ohwi = p.ohwi;
  return a;
}

int grid_for(int64_t total, int threads, int num_sms) {
  const int64_t want = (total + threads - 1) / threads;
  return int(std::max<int64_t>(1, std::min<int64_t>(want, int64_t(num_sms) * 32)));
}

}  // namespace

gbconv_status launch_direct_fwd(const Problem& p, const void* x, const void* w, const float* bias, void* y,
                                const Launch& l) {
  const DirectArgs a = make_args(p);
  if (p.x_elems() + p.w_elems() <= kSmallFloats && p.y_elems() <= int64_t(kSmallThreads) * kSmallOutPerThread) {
    const int nx = int(p.x_elems()), nw = int(p.w_elems());
    const int threads = int(std::min<int64_t>(kSmallThreads, (p.y_elems() + 31) / 32 * 32));
    const size_t smem = size_t(nx + nw) * sizeof(float);
    const cudaError_t e =
        p.bf16 ? launch_kernel(direct_fwd_small_kernel<__nv_bfloat16>, dim3(1), dim3(threads), smem, l.stream, a,
                               static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(w), bias,
                               static_cast<__nv_bfloat16*>(y), nx, nw)
               : launch_kernel(direct_fwd_small_kernel<float>, dim3(1), dim3(threads), smem, l.stream, a,
                               static_cast<const float*>(x), static_cast<const float*>(w), bias,
                               static_cast<float*>(y), nx, nw);
    return e == cudaSuccess ? GBCONV_OK : GBCONV_ECUDA;
  }
  const int threads = 256, blocks = grid_for(p.y_elems(), threads, l.num_sms);
  const cudaError_t e =
      p.bf16 ? launch_kernel(direct_fwd_kernel<__nv_bfloat16>, dim3(blocks), dim3(threads), 0, l.stream, a,
                             static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(w), bias,
                             static_cast<__nv_bfloat16*>(y))
             : launch_kernel(direct_fwd_kernel<float>, dim3(blocks), dim3(threads), 0, l.stream, a,
                             static_cast<const float*>(x), static_cast<const float*>(w), bias, static_cast<float*>(y));
  return e == cudaSuccess ? GBCONV_OK : GBCONV_ECUDA;
}

gbconv_status launch_direct_dgrad(const Problem& p, const void* dy, const void* w, const float* bias, void* dx,
                                  const Launch& l) {
  const DirectArgs a = make_args(p);
  const int threads = 256, blocks = grid_for(p.x_elems(), threads, l.num_sms);
  const cudaError_t e =
      p.bf16 ? launch_kernel(direct_dgrad_kernel<__nv_bfloat16>, dim3(blocks), dim3(threads), 0, l.stream, a,
                             static_cast<const __nv_bfloat16*>(dy), static_cast<const __nv_bfloat16*>(w), bias,
                             static_cast<__nv_bfloat16*>(dx))
             : launch_kernel(direct_dgrad_kernel<float>, dim3(blocks), dim3(threads), 0, l.stream, a,
                             static_cast<const float*>(dy), static_cast<const float*>(w), bias,
                             static_cast<float*>(dx));
  return e == cudaSuccess ? GBCONV_OK : GBCONV_ECUDA;
}

gbconv_status launch_pack_weight(const Problem& p, const void* w_oihw, void* w_ohwi, const Launch& l) {
  const int threads = 256, blocks = grid_for(p.w_elems(), threads, l.num_sms);
  const int Cout = int(p.Cout), cpg = int(p.cpg()), KH = int(p.KD * p.KH), KW = int(p.KW);
  const cudaError_t e =
      p.bf16 ? launch_kernel(pack_ohwi_kernel<__nv_bfloat16>, dim3(blocks), dim3(threads), 0, l.stream, Cout, cpg, KH,
                             KW, static_cast<const __nv_bfloat16*>(w_oihw), static_cast<__nv_bfloat16*>(w_ohwi))
             : launch_kernel(pack_ohwi_kernel<float>, dim3(blocks), dim3(threads), 0, l.stream, Cout, cpg, KH, KW,
                             static_cast<const float*>(w_oihw), static_cast<float*>(w_ohwi));
  return e == cudaSuccess ? GBCONV_OK : GBCONV_ECUDA;
}

}  // namespace gbconv
