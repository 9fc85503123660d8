// Depthwise convolution forward (G = C_in = C_out, channel multiplier 1),
// NHWC bf16, on CUDA cores.  The regime is bandwidth bound (about two flops
// per byte), so the kernel is organised around the memory system, not the
// arithmetic: each thread owns 8 consecutive channels (one 16-byte vector)
// of one output column and walks a strip of output rows; a warp covers 32
// channel vectors of one pixel, so every load and store of a warp is one
// contiguous 512-byte run.  Rows shared by vertically adjacent outputs are
// re-read through L1, columns shared by horizontally adjacent outputs are
// read by neighbouring warps of the same block at the same time.
//
// Definition: teeny-kernels `src/nn/conv/conv2d.rs`, `conv2d_forward` with
// G = C_IN = C_OUT (the depthwise case its doc names): output channel c reads
// only input channel c through weight [C, 1, KH, KW].
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "problem.h"
#include "ptx.cuh"

namespace gbconv {
namespace {

struct DwArgs {
  int N, C, H, W, OH, OW, KH, KW, SH, SW, PH, PW, DH, DW;
  int rows_per_thread;  // output rows walked by one thread
  int cv_per_block;     // channel vectors (of 8) per block along x
  int cv_chunks;        // C/8 / cv_per_block
};

constexpr int kThreads = 256;
constexpr int kMaxTaps = 25;  // up to 5x5 kernels: taps x 256 channels x 4 bytes of shared memory

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int KH_, int KW_>
__global__ void __launch_bounds__(kThreads) depthwise_fwd_kernel(DwArgs a, const __nv_bfloat16* __restrict__ x,
                                                                 const __nv_bfloat16* __restrict__ w,
                                                                 const float* __restrict__ bias,
                                                                 __nv_bfloat16* __restrict__ y) {
  ptx::grid_dep_wait();  // inputs may come from the previous kernel on the stream
  ptx::grid_dep_launch();
  const int KH = KH_ > 0 ? KH_ : a.KH;
  const int KW = KW_ > 0 ? KW_ : a.KW;
  const int taps = KH * KW;
  // Weights of this block's channels as fp32, laid out [tap][channel].
  extern __shared__ __align__(16) float ws[];
  const int cpb = a.cv_per_block * 8;
  const int chunk = blockIdx.x % a.cv_chunks;
  const int c0 = chunk * cpb;
  for (int i = threadIdx.y * blockDim.x + threadIdx.x; i < taps * cpb; i += kThreads) {
    const int t = i / cpb, c = i % cpb;
    ws[t * cpb + c] = __bfloat162float(w[(c0 + c) * taps + t]);
  }
  __syncthreads();

  const int ow = (blockIdx.x / a.cv_chunks) * blockDim.y + threadIdx.y;
  const int cv = threadIdx.x;
  const int n = blockIdx.z;
  if (ow >= a.OW) return;
  const int oh0 = blockIdx.y * a.rows_per_thread;
  const int oh1 = min(a.OH, oh0 + a.rows_per_thread);
  const int c = c0 + cv * 8;
  float b[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) b[j] = bias ? __ldg(bias + c + j) : 0.f;

  const uint4* xv = reinterpret_cast<const uint4*>(x);
  uint4* yv = reinterpret_cast<uint4*>(y);
  const int cvec = a.C / 8;
  for (int oh = oh0; oh < oh1; ++oh) {
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = b[j];
#pragma unroll
    for (int kh = 0; kh < KH; ++kh) {
      const int ih = oh * a.SH + kh * a.DH - a.PH;
      if (ih < 0 || ih >= a.H) continue;
      const int row = (n * a.H + ih) * a.W;
#pragma unroll
      for (int kw = 0; kw < KW; ++kw) {
        const int iw = ow * a.SW + kw * a.DW - a.PW;
        if (iw < 0 || iw >= a.W) continue;
        float xf[8];
        unpack8(__ldg(xv + (size_t)(row + iw) * cvec + (c >> 3)), xf);
        const float* wt = ws + (kh * KW + kw) * cpb + cv * 8;
        const float4 w0 = *reinterpret_cast<const float4*>(wt);
        const float4 w1 = *reinterpret_cast<const float4*>(wt + 4);
        acc[0] = fmaf(xf[0], w0.x, acc[0]);
        acc[1] = fmaf(xf[1], w0.y, acc[1]);
        acc[2] = fmaf(xf[2], w0.z, acc[2]);
        acc[3] = fmaf(xf[3], w0.w, acc[3]);
        acc[4] = fmaf(xf[4], w1.x, acc[4]);
        acc[5] = fmaf(xf[5], w1.y, acc[5]);
        acc[6] = fmaf(xf[6], w1.z, acc[6]);
        acc[7] = fmaf(xf[7], w1.w, acc[7]);
      }
    }
    uint4 o;
    o.x = pack2(acc[0], acc[1]);
    o.y = pack2(acc[2], acc[3]);
    o.z = pack2(acc[4], acc[5]);
    o.w = pack2(acc[6], acc[7]);
    yv[(size_t)((n * a.OH + oh) * a.OW + ow) * cvec + (c >> 3)] = o;
  }
}


// Depthwise input gradient (gather form, no atomics: every dx element is written once, in a
// fixed summation order).  The transpose of the forward above, with the same thread layout:
// each thread owns 8 channels of one dx column and walks a strip of dx rows; for dx (ih, iw) a
// tap (kh, kw) contributes dy[(ih + PH - kh*DH) / SH, (iw + PW - kw*DW) / SW] * w[c, kh, kw] when
// both divisions are exact and land inside dy.  teeny-kernels `src/nn/conv/conv2d.rs`,
// `conv2d_backward` scatters the same products into dx with atomics (G = C case).
// S_ > 0: compile-time stride S_ in both dims; 0: runtime strides.
template <int S_>
__global__ void __launch_bounds__(kThreads) depthwise_dgrad_kernel(DwArgs a, const __nv_bfloat16* __restrict__ dy,
                                                                   const __nv_bfloat16* __restrict__ w,
                                                                   const float* __restrict__ bias,
                                                                   __nv_bfloat16* __restrict__ dx) {
  ptx::grid_dep_wait();  // inputs may come from the previous kernel on the stream
  ptx::grid_dep_launch();
  const int KH = a.KH, KW = a.KW, taps = KH * KW;
  const int SH = S_ > 0 ? S_ : a.SH, SW = S_ > 0 ? S_ : a.SW;
  extern __shared__ __align__(16) float ws[];  // [tap][channel] of this block's channels, fp32
  const int cpb = a.cv_per_block * 8;
  const int chunk = blockIdx.x % a.cv_chunks;
  const int c0 = chunk * cpb;
  for (int i = threadIdx.y * blockDim.x + threadIdx.x; i < taps * cpb; i += kThreads) {
    const int t = i / cpb, c = i % cpb;
    ws[t * cpb + c] = __bfloat162float(w[(c0 + c) * taps + t]);
  }
  __syncthreads();

  const int iw = (blockIdx.x / a.cv_chunks) * blockDim.y + threadIdx.y;  // dx column
  const int cv = threadIdx.x;
  const int n = blockIdx.z;
  if (iw >= a.W) return;
  const int ih0 = blockIdx.y * a.rows_per_thread;
  const int ih1 = min(a.H, ih0 + a.rows_per_thread);
  const int c = c0 + cv * 8;
  const uint4* dyv = reinterpret_cast<const uint4*>(dy);
  uint4* dxv = reinterpret_cast<uint4*>(dx);
  const int cvec = a.C / 8;
  float b[8];  // transposed-convolution bias, added after the gather sum
#pragma unroll
  for (int j = 0; j < 8; ++j) b[j] = bias ? __ldg(bias + c + j) : 0.f;
  for (int ih = ih0; ih < ih1; ++ih) {
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    for (int kh = 0; kh < KH; ++kh) {
      const int nh = ih + a.PH - kh * a.DH;
      if (nh < 0 || nh % SH != 0) continue;
      const int oh = nh / SH;
      if (oh >= a.OH) continue;
      const int row = (n * a.OH + oh) * a.OW;
      for (int kw = 0; kw < KW; ++kw) {
        const int nw = iw + a.PW - kw * a.DW;
        if (nw < 0 || nw % SW != 0) continue;
        const int ow = nw / SW;
        if (ow >= a.OW) continue;
        float g[8];
        unpack8(__ldg(dyv + (size_t)(row + ow) * cvec + (c >> 3)), g);
        const float* wt = ws + (kh * KW + kw) * cpb + cv * 8;
        const float4 w0 = *reinterpret_cast<const float4*>(wt);
        const float4 w1 = *reinterpret_cast<const float4*>(wt + 4);
        acc[0] = fmaf(g[0], w0.x, acc[0]);
        acc[1] = fmaf(g[1], w0.y, acc[1]);
        acc[2] = fmaf(g[2], w0.z, acc[2]);
        acc[3] = fmaf(g[3], w0.w, acc[3]);
        acc[4] = fmaf(g[4], w1.x, acc[4]);
        acc[5] = fmaf(g[5], w1.y, acc[5]);
        acc[6] = fmaf(g[6], w1.z, acc[6]);
        acc[7] = fmaf(g[7], w1.w, acc[7]);
      }
    }
    uint4 o;
    o.x = pack2(acc[0] + b[0], acc[1] + b[1]);
    o.y = pack2(acc[2] + b[2], acc[3] + b[3]);
    o.z = pack2(acc[4] + b[4], acc[5] + b[5]);
    o.w = pack2(acc[6] + b[6], acc[7] + b[7]);
    dxv[(size_t)((n * a.H + ih) * a.W + iw) * cvec + (c >> 3)] = o;
  }
}

// Depthwise dgrad for 3x3, stride 2, pad 1, dilation 1 (the common downsampling layer).  A dx
// 2x2 block at (2r, 2c) reads exactly the dy 2x2 block at (r, c):
//   dx[2r  ][2c  ] = dy[r][c] w11
//   dx[2r  ][2c+1] = dy[r][c] w12 + dy[r][c+1] w10
//   dx[2r+1][2c  ] = dy[r][c] w21 + dy[r+1][c] w01
//   dx[2r+1][2c+1] = dy[r][c] w22 + dy[r][c+1] w20 + dy[r+1][c] w02 + dy[r+1][c+1] w00
// (w[kh][kw]; dy outside [0,OH) x [0,OW) is zero).  Each thread owns 8 channels of one dy column
// c and walks a strip of dy rows r, keeping row r+1's two vectors for the next step: two 16-byte
// loads and four 16-byte stores per step, the nine weights of its channels in registers.
template <bool BIAS>
__global__ void __launch_bounds__(kThreads) depthwise3x3s2_dgrad_kernel(DwArgs a, const __nv_bfloat16* __restrict__ dy,
                                                                        const __nv_bfloat16* __restrict__ w,
                                                                        const float* __restrict__ bias,
                                                                        __nv_bfloat16* __restrict__ dx) {
  ptx::grid_dep_wait();  // inputs may come from the previous kernel on the stream
  ptx::grid_dep_launch();
  const int cpb = a.cv_per_block * 8;
  const int chunk = blockIdx.x % a.cv_chunks;
  const int oc = (blockIdx.x / a.cv_chunks) * blockDim.y + threadIdx.y;  // dy column c
  const int ch = chunk * cpb + threadIdx.x * 8;
  const int n = blockIdx.z;
  if (oc >= a.OW) return;
  float wr[9][8];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int t = 0; t < 9; ++t) wr[t][j] = __bfloat162float(w[(ch + j) * 9 + t]);
  float bs[8];  // transposed-convolution bias, added after the gather sum (BIAS only: registers)
#pragma unroll
  for (int j = 0; j < 8; ++j) bs[j] = BIAS ? __ldg(bias + ch + j) : 0.f;
  const uint4* dyv = reinterpret_cast<const uint4*>(dy);
  uint4* dxv = reinterpret_cast<uint4*>(dx);
  const int cvec = a.C / 8, cv = ch >> 3;
  const bool right = oc + 1 < a.OW;       // dy column c+1 exists
  const bool col1 = 2 * oc + 1 < a.W;     // dx column 2c+1 exists
  const int r0 = blockIdx.y * a.rows_per_thread;
  const int r1 = min(a.OH, r0 + a.rows_per_thread);
  const uint4 zero = make_uint4(0, 0, 0, 0);
  auto load = [&](int r, int c) -> uint4 { return __ldg(dyv + (size_t)((n * a.OH + r) * a.OW + c) * cvec + cv); };
  // Rows r and r+1 are in registers when step r starts; the loads of row r+2 are issued first,
  // so a step's stores overlap the next step's loads.
  uint4 cur0 = load(r0, oc), cur1 = right ? load(r0, oc + 1) : zero;
  uint4 nxt0 = r0 + 1 < a.OH ? load(r0 + 1, oc) : zero;
  uint4 nxt1 = (r0 + 1 < a.OH && right) ? load(r0 + 1, oc + 1) : zero;
  for (int r = r0; r < r1; ++r) {
    const bool far = r + 2 < a.OH && r + 1 < r1;
    const uint4 far0 = far ? load(r + 2, oc) : zero;
    const uint4 far1 = (far && right) ? load(r + 2, oc + 1) : zero;
    float a0[8], a1[8], b0[8], b1[8];  // dy[r][c], dy[r][c+1], dy[r+1][c], dy[r+1][c+1]
    unpack8(cur0, a0);
    unpack8(cur1, a1);
    unpack8(nxt0, b0);
    unpack8(nxt1, b1);
    float o00[8], o01[8], o10[8], o11[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      o00[j] = a0[j] * wr[4][j] + bs[j];
      o01[j] = fmaf(a1[j], wr[3][j], a0[j] * wr[5][j]) + bs[j];
      o10[j] = fmaf(b0[j], wr[1][j], a0[j] * wr[7][j]) + bs[j];
      o11[j] = fmaf(b1[j], wr[0][j], fmaf(b0[j], wr[2][j], fmaf(a1[j], wr[6][j], a0[j] * wr[8][j]))) + bs[j];
    }
    auto pack = [](const float (&f)[8]) {
      uint4 o;
      o.x = pack2(f[0], f[1]);
      o.y = pack2(f[2], f[3]);
      o.z = pack2(f[4], f[5]);
      o.w = pack2(f[6], f[7]);
      return o;
    };
    const size_t row0 = (size_t)(n * a.H + 2 * r) * a.W;
    dxv[(row0 + 2 * oc) * cvec + cv] = pack(o00);
    if (col1) dxv[(row0 + 2 * oc + 1) * cvec + cv] = pack(o01);
    if (2 * r + 1 < a.H) {
      const size_t row1 = row0 + a.W;
      dxv[(row1 + 2 * oc) * cvec + cv] = pack(o10);
      if (col1) dxv[(row1 + 2 * oc + 1) * cvec + cv] = pack(o11);
    }
    cur0 = nxt0;
    cur1 = nxt1;
    nxt0 = far0;
    nxt1 = far1;
  }
}

// 3x3, dilation 1, stride S in {1, 2}: the nine weights of the thread's 8
// channels live in registers, and each input row a thread loads is kept in
// registers for every output row of its strip that reads it (rows overlap by
// 3 - S), so a strip of R output rows loads (R*S + 3 - S) input rows instead
// of 3R.  No shared memory is touched in the loop.
template <int S>
__global__ void __launch_bounds__(kThreads, 2) depthwise3x3_kernel(DwArgs a, const __nv_bfloat16* __restrict__ x,
                                                                  const __nv_bfloat16* __restrict__ w,
                                                                  const float* __restrict__ bias,
                                                                  __nv_bfloat16* __restrict__ y) {
  ptx::grid_dep_wait();  // inputs may come from the previous kernel on the stream
  ptx::grid_dep_launch();
  constexpr int kKeep = 3 - S;  // input rows shared by consecutive output rows
  const int cpb = a.cv_per_block * 8;
  const int chunk = blockIdx.x % a.cv_chunks;
  const int ow = (blockIdx.x / a.cv_chunks) * blockDim.y + threadIdx.y;
  const int c = chunk * cpb + threadIdx.x * 8;
  const int n = blockIdx.z;
  if (ow >= a.OW) return;
  float wr[9][8];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int t = 0; t < 9; ++t) wr[t][j] = __bfloat162float(w[(c + j) * 9 + t]);
  float b[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) b[j] = bias ? __ldg(bias + c + j) : 0.f;

  const uint4* xv = reinterpret_cast<const uint4*>(x);
  uint4* yv = reinterpret_cast<uint4*>(y);
  const int cvec = a.C / 8, cv = c >> 3;
  int iw[3];
  bool okw[3];
#pragma unroll
  for (int kw = 0; kw < 3; ++kw) {
    iw[kw] = ow * S + kw - a.PW;
    okw[kw] = iw[kw] >= 0 && iw[kw] < a.W;
  }
  auto load_row = [&](int ih, uint4 (&r)[3]) {
    const bool okh = ih >= 0 && ih < a.H;
#pragma unroll
    for (int kw = 0; kw < 3; ++kw)
      r[kw] = (okh && okw[kw]) ? __ldg(xv + (size_t(n * a.H + ih) * a.W + iw[kw]) * cvec + cv) : make_uint4(0, 0, 0, 0);
  };
  const int oh0 = blockIdx.y * a.rows_per_thread;
  const int oh1 = min(a.OH, oh0 + a.rows_per_thread);
  uint4 keep[kKeep][3];
#pragma unroll
  for (int k = 0; k < kKeep; ++k) load_row(oh0 * S - a.PH + k, keep[k]);
  for (int oh = oh0; oh < oh1; ++oh) {
    uint4 rows[3][3];
#pragma unroll
    for (int k = 0; k < kKeep; ++k)
#pragma unroll
      for (int kw = 0; kw < 3; ++kw) rows[k][kw] = keep[k][kw];
#pragma unroll
    for (int k = kKeep; k < 3; ++k) load_row(oh * S - a.PH + k, rows[k]);
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = b[j];
#pragma unroll
    for (int kh = 0; kh < 3; ++kh)
#pragma unroll
      for (int kw = 0; kw < 3; ++kw) {
        float xf[8];
        unpack8(rows[kh][kw], xf);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = fmaf(xf[j], wr[kh * 3 + kw][j], acc[j]);
      }
    uint4 o;
    o.x = pack2(acc[0], acc[1]);
    o.y = pack2(acc[2], acc[3]);
    o.z = pack2(acc[4], acc[5]);
    o.w = pack2(acc[6], acc[7]);
    yv[(size_t(n * a.OH + oh) * a.OW + ow) * cvec + cv] = o;
#pragma unroll
    for (int k = 0; k < kKeep; ++k)
#pragma unroll
      for (int kw = 0; kw < 3; ++kw) keep[k][kw] = rows[3 - kKeep + k][kw];
  }
}


// ---------------------------------------------------------------- TMA-fed 3x3
// Persistent kernel for the 3x3 / stride 1 or 2 / dilation 1 case with 64-channel
// chunks.  A producer lane streams halo tiles (TR x TC outputs need
// ((TR-1)S+3) x ((TC-1)S+3) input pixels x 64 channels, zero fill supplying the
// padding) through a ring of shared-memory stages with TMA; 256 compute threads
// each own 8 channels of two output pixels per tile, keep their 72 weights in
// registers, and read the taps from shared memory.  DRAM sees each input byte
// once per tile (halo overlap between tiles comes from L2).
// Output tiles are TR x TC = 64 pixels: 4 x 16, or 8 x 8 where that cuts fewer partial tiles (a
// 56-wide output is 3.5 tiles of 16 columns but 7 of 8; a partial tile costs a whole tile's time).
constexpr int kTilePix = 64;
constexpr int kDwStages = 4;
constexpr int kDwCompute = 256;             // compute threads (8 warps)
constexpr int kDwThreads = kDwCompute + 32; // + one producer warp

struct DwTmaArgs {
  const float* bias;
  __nv_bfloat16* y;
  unsigned int* status;
  uint64_t wait_ns;   // bound of every barrier wait (the host sets it; 2 s by default)
  int N, C, H, W, OH, OW, PH, PW;
  int nchunk, tiles_h, tiles_w, tiles_per_chunk;
  int ir, ic, stage_bytes;
};

template <int S, int TR>
__global__ void __launch_bounds__(kDwThreads, 1)
    depthwise3x3_tma_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ DwTmaArgs a,
                            const __nv_bfloat16* __restrict__ w) {
  constexpr int kTC = kTilePix / TR;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kDwStages * a.stage_bytes);
  uint64_t* empty = full + kDwStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kDwStages);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kDwStages; ++i) { ptx::mbar_init(full + i, 1); ptx::mbar_init(empty + i, kDwCompute); }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  ptx::grid_dep_wait();  // inputs may come from the previous kernel on the stream
  ptx::grid_dep_launch();
  // CTAs are split evenly over the channel chunks, so each keeps one chunk's weights.
  const int chunk = blockIdx.x % a.nchunk;
  const int ctas_per_chunk = gridDim.x / a.nchunk;
  const int first = blockIdx.x / a.nchunk;
  if (warp == kDwCompute / 32) {
    if ((threadIdx.x & 31) == 0) {
      ptx::prefetch_tmap(&xmap);
      int st = 0, issued = 0;
      uint32_t ph = 0;
      for (int t = first; t < a.tiles_per_chunk; t += ctas_per_chunk) {
        const int tw = t % a.tiles_w, th = (t / a.tiles_w) % a.tiles_h, n = t / (a.tiles_w * a.tiles_h);
        if (!ptx::mbar_wait(empty + st, ph ^ 1, abort_flag, a.status, 16u, a.wait_ns)) break;
        ++issued;
        ptx::mbar_arrive_expect_tx(full + st, uint32_t(a.stage_bytes));
        asm volatile(
            "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, "
            "%6}], [%2];" ::"r"(ptx::smem_addr(smem + st * a.stage_bytes)),
            "l"(&xmap), "r"(ptx::smem_addr(full + st)), "r"(chunk * 64), "r"(tw * kTC * S - a.PW),
            "r"(th * TR * S - a.PH), "r"(n)
            : "memory");
        if (++st == kDwStages) { st = 0; ph ^= 1; }
      }
      // Drain: copies still in flight write this CTA's shared memory and must land before it leaves
      // (after an abort the compute threads no longer consume them).
      for (int k = max(0, issued - kDwStages); k < issued; ++k)
        ptx::mbar_wait_drain(full + k % kDwStages, uint32_t((k / kDwStages) & 1));
    }
    __syncwarp();
    return;
  }
  // ------------------------------------------------------------ compute threads
  const int cv = threadIdx.x & 7;     // 8-channel vector inside the 64-channel chunk
  const int pix = threadIdx.x >> 3;   // 0..31: output pixels pix and pix + 32 of the tile
  const int c = chunk * 64 + cv * 8;
  float wr[9][8];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int t = 0; t < 9; ++t) wr[t][j] = __bfloat162float(w[(c + j) * 9 + t]);
  float b[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) b[j] = a.bias ? __ldg(a.bias + c + j) : 0.f;
  uint4* yv = reinterpret_cast<uint4*>(a.y);
  const int cvec = a.C / 8;
  int st = 0;
  uint32_t ph = 0;
  for (int t = first; t < a.tiles_per_chunk; t += ctas_per_chunk) {
    const int tw = t % a.tiles_w, th = (t / a.tiles_w) % a.tiles_h, n = t / (a.tiles_w * a.tiles_h);
    if (!ptx::mbar_wait(full + st, ph, abort_flag, a.status, 16u, a.wait_ns)) break;
    const uint32_t base = ptx::smem_addr(smem + st * a.stage_bytes) + cv * 16;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int p = pix + half * 32;
      const int r = p / kTC, col = p % kTC;
      float acc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = b[j];
#pragma unroll
      for (int kh = 0; kh < 3; ++kh)
#pragma unroll
        for (int kw = 0; kw < 3; ++kw) {
          uint4 v;
          asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                       : "r"(base + uint32_t(((r * S + kh) * a.ic + col * S + kw) * 128)));
          float xf[8];
          unpack8(v, xf);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[j] = fmaf(xf[j], wr[kh * 3 + kw][j], acc[j]);
        }
      const int oh = th * TR + r, ow = tw * kTC + col;
      if (oh < a.OH && ow < a.OW) {
        uint4 o;
        o.x = pack2(acc[0], acc[1]);
        o.y = pack2(acc[2], acc[3]);
        o.z = pack2(acc[4], acc[5]);
        o.w = pack2(acc[6], acc[7]);
        yv[(size_t(n * a.OH + oh) * a.OW + ow) * cvec + (c >> 3)] = o;
      }
    }
    ptx::mbar_arrive(empty + st);
    if (++st == kDwStages) { st = 0; ph ^= 1; }
  }
}

// The same persistent TMA design for the input gradient of the 3x3 / stride 2 / pad 1 / dilation 1
// layer, whose dx 2x2 block at (2R, 2C) reads exactly the dy 2x2 block at (R, C) (the gather
// written out above depthwise3x3s2_dgrad_kernel).  A tile is TR x TC dy positions, which need
// (TR+1) x (TC+1) dy pixels (zero fill past the last row and column) and produce 2TR x 2TC dx
// pixels.  Every SM takes an equal share of the tiles; the register-streaming kernel above ran one
// block per (image, column group), which left some SMs two blocks' work and others one.
template <bool BIAS, int TR>
__global__ void __launch_bounds__(kDwThreads, 1)
    depthwise3x3s2_dgrad_tma_kernel(const __grid_constant__ CUtensorMap dymap, const __grid_constant__ DwTmaArgs a,
                                    const __nv_bfloat16* __restrict__ w) {
  constexpr int kTC = kTilePix / TR;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kDwStages * a.stage_bytes);
  uint64_t* empty = full + kDwStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kDwStages);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kDwStages; ++i) { ptx::mbar_init(full + i, 1); ptx::mbar_init(empty + i, kDwCompute); }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  ptx::grid_dep_wait();  // inputs may come from the previous kernel on the stream
  ptx::grid_dep_launch();
  const int chunk = blockIdx.x % a.nchunk;
  const int ctas_per_chunk = gridDim.x / a.nchunk;
  const int first = blockIdx.x / a.nchunk;
  if (warp == kDwCompute / 32) {
    if ((threadIdx.x & 31) == 0) {
      ptx::prefetch_tmap(&dymap);
      int st = 0, issued = 0;
      uint32_t ph = 0;
      for (int t = first; t < a.tiles_per_chunk; t += ctas_per_chunk) {
        const int tw = t % a.tiles_w, th = (t / a.tiles_w) % a.tiles_h, n = t / (a.tiles_w * a.tiles_h);
        if (!ptx::mbar_wait(empty + st, ph ^ 1, abort_flag, a.status, 16u, a.wait_ns)) break;
        ++issued;
        ptx::mbar_arrive_expect_tx(full + st, uint32_t(a.stage_bytes));
        asm volatile(
            "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, "
            "%6}], [%2];" ::"r"(ptx::smem_addr(smem + st * a.stage_bytes)),
            "l"(&dymap), "r"(ptx::smem_addr(full + st)), "r"(chunk * 64), "r"(tw * kTC), "r"(th * TR), "r"(n)
            : "memory");
        if (++st == kDwStages) { st = 0; ph ^= 1; }
      }
      for (int k = max(0, issued - kDwStages); k < issued; ++k)
        ptx::mbar_wait_drain(full + k % kDwStages, uint32_t((k / kDwStages) & 1));
    }
    __syncwarp();
    return;
  }
  // ------------------------------------------------------------ compute threads
  // A warp covers 4 consecutive dy positions x 8 channel vectors: its shared-memory reads are 512
  // contiguous bytes, and each of its stores writes four whole 128-byte lines.
  const int cv = threadIdx.x & 7;
  const int pos = threadIdx.x >> 3;  // dy positions pos and pos + 32 of the tile
  const int c = chunk * 64 + cv * 8;
  float wr[9][8];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int t = 0; t < 9; ++t) wr[t][j] = __bfloat162float(w[(c + j) * 9 + t]);
  float bs[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) bs[j] = BIAS ? __ldg(a.bias + c + j) : 0.f;
  uint4* dxv = reinterpret_cast<uint4*>(a.y);
  const int cvec = a.C / 8;
  int st = 0;
  uint32_t ph = 0;
  for (int t = first; t < a.tiles_per_chunk; t += ctas_per_chunk) {
    const int tw = t % a.tiles_w, th = (t / a.tiles_w) % a.tiles_h, n = t / (a.tiles_w * a.tiles_h);
    if (!ptx::mbar_wait(full + st, ph, abort_flag, a.status, 16u, a.wait_ns)) break;
    const uint32_t base = ptx::smem_addr(smem + st * a.stage_bytes) + cv * 16;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int p = pos + half * 32;
      const int r = p / kTC, col = p % kTC;
      const int R = th * TR + r, C = tw * kTC + col;  // dy position
      if (R < a.OH && C < a.OW) {
        uint4 v00, v01, v10, v11;  // dy[R][C], dy[R][C+1], dy[R+1][C], dy[R+1][C+1]
        const uint32_t q = base + uint32_t((r * a.ic + col) * 128);
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v00.x), "=r"(v00.y), "=r"(v00.z), "=r"(v00.w) : "r"(q));
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v01.x), "=r"(v01.y), "=r"(v01.z), "=r"(v01.w) : "r"(q + 128));
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v10.x), "=r"(v10.y), "=r"(v10.z), "=r"(v10.w) : "r"(q + uint32_t(a.ic * 128)));
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v11.x), "=r"(v11.y), "=r"(v11.z), "=r"(v11.w) : "r"(q + uint32_t(a.ic * 128 + 128)));
        float a0[8], a1[8], b0[8], b1[8];
        unpack8(v00, a0);
        unpack8(v01, a1);
        unpack8(v10, b0);
        unpack8(v11, b1);
        float o00[8], o01[8], o10[8], o11[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          o00[j] = a0[j] * wr[4][j] + bs[j];
          o01[j] = fmaf(a1[j], wr[3][j], a0[j] * wr[5][j]) + bs[j];
          o10[j] = fmaf(b0[j], wr[1][j], a0[j] * wr[7][j]) + bs[j];
          o11[j] = fmaf(b1[j], wr[0][j], fmaf(b0[j], wr[2][j], fmaf(a1[j], wr[6][j], a0[j] * wr[8][j]))) + bs[j];
        }
        auto pack = [](const float (&f)[8]) {
          uint4 o;
          o.x = pack2(f[0], f[1]);
          o.y = pack2(f[2], f[3]);
          o.z = pack2(f[4], f[5]);
          o.w = pack2(f[6], f[7]);
          return o;
        };
        const bool col1 = 2 * C + 1 < a.W;
        const size_t row0 = size_t(n * a.H + 2 * R) * a.W;
        dxv[(row0 + 2 * C) * cvec + (c >> 3)] = pack(o00);
        if (col1) dxv[(row0 + 2 * C + 1) * cvec + (c >> 3)] = pack(o01);
        if (2 * R + 1 < a.H) {
          const size_t row1 = row0 + a.W;
          dxv[(row1 + 2 * C) * cvec + (c >> 3)] = pack(o10);
          if (col1) dxv[(row1 + 2 * C + 1) * cvec + (c >> 3)] = pack(o11);
        }
      }
    }
    ptx::mbar_arrive(empty + st);
    if (++st == kDwStages) { st = 0; ph ^= 1; }
  }
}

// Output tile rows of the TMA-fed kernels: 8 (8 x 8 tiles) when that gives fewer tiles than 4 x 16.
int tile_rows(int oh, int ow) {
  const int64_t t4 = int64_t((oh + 3) / 4) * ((ow + 15) / 16), t8 = int64_t((oh + 7) / 8) * ((ow + 7) / 8);
  return t8 < t4 ? 8 : 4;
}

PFN_cuTensorMapEncodeTiled_v12000 dw_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool dw_tma_supported(const Problem& p) {
  // tiles are laid out for symmetric padding; (begin, end) padding takes the generic kernel
  return p.sym_pad() && p.KH == 3 && p.KW == 3 && p.DH == 1 && p.DW == 1 && p.SH == p.SW && (p.SH == 1 || p.SH == 2) &&
         p.Cin % 64 == 0;
}

template <int S>
gbconv_status launch_dw_tma(const Problem& p, const void* x, const void* w, const float* bias, void* y,
                            const Launch& l) {
  auto fn = dw_encode_fn();
  if (!fn) return GBCONV_ECUDA;
  DwTmaArgs a{};
  a.bias = bias;
  a.y = static_cast<__nv_bfloat16*>(y);
  a.status = l.status;
  a.wait_ns = l.wait_ns;
  a.N = int(p.N); a.C = int(p.Cin); a.H = int(p.H); a.W = int(p.W); a.OH = int(p.OH); a.OW = int(p.OW);
  a.PH = int(p.PH); a.PW = int(p.PW);
  a.nchunk = a.C / 64;
  const int TR = tile_rows(a.OH, a.OW), TC = kTilePix / TR;
  a.tiles_h = (a.OH + TR - 1) / TR;
  a.tiles_w = (a.OW + TC - 1) / TC;
  a.tiles_per_chunk = a.N * a.tiles_h * a.tiles_w;
  a.ir = (TR - 1) * S + 3;
  a.ic = (TC - 1) * S + 3;
  a.stage_bytes = a.ir * a.ic * 128;
  CUtensorMap map;
  cuuint64_t dims[4] = {cuuint64_t(a.C), cuuint64_t(a.W), cuuint64_t(a.H), cuuint64_t(a.N)};
  cuuint64_t strides[3] = {cuuint64_t(a.C) * 2, cuuint64_t(a.W) * a.C * 2, cuuint64_t(a.H) * a.W * a.C * 2};
  cuuint32_t box[4] = {64, cuuint32_t(a.ic), cuuint32_t(a.ir), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return GBCONV_ECUDA;
  const size_t smem = size_t(kDwStages) * a.stage_bytes + 8 * 2 * kDwStages + 16;
  auto kern = TR == 8 ? depthwise3x3_tma_kernel<S, 8> : depthwise3x3_tma_kernel<S, 4>;
  static std::atomic<uint64_t> done[64];  // bit per tile shape
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GBCONV_ECUDA;
  const uint64_t bit = TR == 8 ? 2u : 1u;
  if ((done[dev].load(std::memory_order_acquire) & bit) == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess)
      return GBCONV_ECUDA;
    done[dev].fetch_or(bit, std::memory_order_acq_rel);
  }
  // A multiple of the chunk count, at most one CTA per SM and per tile column of work.
  int grid = std::max(a.nchunk, (l.num_sms / a.nchunk) * a.nchunk);
  grid = std::min<int64_t>(grid, int64_t(a.nchunk) * a.tiles_per_chunk);
  return launch_kernel(kern, dim3(grid), dim3(kDwThreads), smem, l.stream, map, a,
                       static_cast<const __nv_bfloat16*>(w)) == cudaSuccess
             ? GBCONV_OK
             : GBCONV_ECUDA;
}

gbconv_status launch_dw_dgrad_tma(const Problem& p, const void* dy, const void* w, const float* bias, void* dx,
                                  const Launch& l) {
  auto fn = dw_encode_fn();
  if (!fn) return GBCONV_ECUDA;
  DwTmaArgs a{};
  a.bias = bias;
  a.y = static_cast<__nv_bfloat16*>(dx);
  a.status = l.status;
  a.wait_ns = l.wait_ns;
  a.N = int(p.N); a.C = int(p.Cin); a.H = int(p.H); a.W = int(p.W); a.OH = int(p.OH); a.OW = int(p.OW);
  a.nchunk = a.C / 64;
  const int TR = tile_rows(a.OH, a.OW), TC = kTilePix / TR;
  a.tiles_h = (a.OH + TR - 1) / TR;
  a.tiles_w = (a.OW + TC - 1) / TC;
  a.tiles_per_chunk = a.N * a.tiles_h * a.tiles_w;
  a.ir = TR + 1;
  a.ic = TC + 1;
  a.stage_bytes = a.ir * a.ic * 128;
  CUtensorMap map;
  cuuint64_t dims[4] = {cuuint64_t(a.C), cuuint64_t(a.OW), cuuint64_t(a.OH), cuuint64_t(a.N)};
  cuuint64_t strides[3] = {cuuint64_t(a.C) * 2, cuuint64_t(a.OW) * a.C * 2, cuuint64_t(a.OH) * a.OW * a.C * 2};
  cuuint32_t box[4] = {64, cuuint32_t(a.ic), cuuint32_t(a.ir), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(dy), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return GBCONV_ECUDA;
  const size_t smem = size_t(kDwStages) * a.stage_bytes + 8 * 2 * kDwStages + 16;
  auto kern = TR == 8 ? (bias ? depthwise3x3s2_dgrad_tma_kernel<true, 8> : depthwise3x3s2_dgrad_tma_kernel<false, 8>)
                      : (bias ? depthwise3x3s2_dgrad_tma_kernel<true, 4> : depthwise3x3s2_dgrad_tma_kernel<false, 4>);
  static std::atomic<uint64_t> done[64];  // bit per (bias, tile shape)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GBCONV_ECUDA;
  const uint64_t bit = uint64_t(1) << ((bias ? 2 : 0) + (TR == 8 ? 1 : 0));
  if ((done[dev].load(std::memory_order_acquire) & bit) == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
      return GBCONV_ECUDA;
    done[dev].fetch_or(bit, std::memory_order_acq_rel);
  }
  // A multiple of the chunk count, at most one CTA per SM and per tile of work.
  int grid = std::max(a.nchunk, (l.num_sms / a.nchunk) * a.nchunk);
  grid = std::min<int64_t>(grid, int64_t(a.nchunk) * a.tiles_per_chunk);
  return launch_kernel(kern, dim3(grid), dim3(kDwThreads), smem, l.stream, map, a,
                       static_cast<const __nv_bfloat16*>(w)) == cudaSuccess
             ? GBCONV_OK
             : GBCONV_ECUDA;
}

}  // namespace

bool depthwise_supported(const Problem& p) {
  return p.bf16 && p.nhwc && p.G == p.Cin && p.Cin == p.Cout && p.Cin % 8 == 0 && p.KH * p.KW <= kMaxTaps;
}

gbconv_status launch_depthwise_fwd(const Problem& p, const void* x, const void* w, const float* bias, void* y,
                                   const Launch& l) {
  DwArgs a;
  a.N = int(p.N); a.C = int(p.Cin); a.H = int(p.H); a.W = int(p.W); a.OH = int(p.OH); a.OW = int(p.OW);
  a.KH = int(p.KH); a.KW = int(p.KW); a.SH = int(p.SH); a.SW = int(p.SW); a.PH = int(p.PH); a.PW = int(p.PW);
  a.DH = int(p.DH); a.DW = int(p.DW);
  const int cvec = a.C / 8;
  // Largest power-of-two divisor of C/8 up to 32 channel vectors per block row.
  int cvb = 1;
  while (cvb < 32 && cvec % (cvb * 2) == 0) cvb *= 2;
  a.cv_per_block = cvb;
  a.cv_chunks = cvec / cvb;
  const int ty = kThreads / cvb;
  a.rows_per_thread = 4;
  dim3 block(cvb, ty);
  const int64_t gx = ((p.OW + ty - 1) / ty) * a.cv_chunks;
  const int64_t gy = (p.OH + a.rows_per_thread - 1) / a.rows_per_thread;
  if (gx > 0x7FFFFFFF || gy > 65535 || p.N > 65535) return GBCONV_EUNSUPPORTED;
  dim3 grid(unsigned(gx), unsigned(gy), unsigned(p.N));
  const size_t smem = size_t(p.KH * p.KW) * cvb * 8 * sizeof(float);
  auto xb = static_cast<const __nv_bfloat16*>(x);
  auto wb = static_cast<const __nv_bfloat16*>(w);
  auto yb = static_cast<__nv_bfloat16*>(y);
  if (dw_tma_supported(p)) return p.SH == 1 ? launch_dw_tma<1>(p, x, w, bias, y, l) : launch_dw_tma<2>(p, x, w, bias, y, l);
  const bool reg3x3 =
      p.sym_pad() && p.KH == 3 && p.KW == 3 && p.DH == 1 && p.DW == 1 && p.SH == p.SW && (p.SH == 1 || p.SH == 2);
  if (reg3x3) {
    a.rows_per_thread = 8;
    grid.y = unsigned((p.OH + a.rows_per_thread - 1) / a.rows_per_thread);
  }
  cudaError_t e;
  if (reg3x3)
    e = p.SH == 1 ? launch_kernel(depthwise3x3_kernel<1>, grid, block, 0, l.stream, a, xb, wb, bias, yb)
                  : launch_kernel(depthwise3x3_kernel<2>, grid, block, 0, l.stream, a, xb, wb, bias, yb);
  else if (p.KH == 3 && p.KW == 3)
    e = launch_kernel(depthwise_fwd_kernel<3, 3>, grid, block, smem, l.stream, a, xb, wb, bias, yb);
  else
    e = launch_kernel(depthwise_fwd_kernel<0, 0>, grid, block, smem, l.stream, a, xb, wb, bias, yb);
  return e == cudaSuccess ? GBCONV_OK : GBCONV_ECUDA;
}

bool depthwise_dgrad_supported(const Problem& p) { return depthwise_supported(p); }

gbconv_status launch_depthwise_dgrad(const Problem& p, const void* dy, const void* w, const float* bias, void* dx,
                                     const Launch& l) {
  if (!depthwise_dgrad_supported(p)) return GBCONV_EUNSUPPORTED;
  DwArgs a;
  a.N = int(p.N); a.C = int(p.Cin); a.H = int(p.H); a.W = int(p.W); a.OH = int(p.OH); a.OW = int(p.OW);
  a.KH = int(p.KH); a.KW = int(p.KW); a.SH = int(p.SH); a.SW = int(p.SW); a.PH = int(p.PH); a.PW = int(p.PW);
  a.DH = int(p.DH); a.DW = int(p.DW);
  const int cvec = a.C / 8;
  int cvb = 1;  // largest power-of-two divisor of C/8 up to 32 channel vectors per block row
  while (cvb < 32 && cvec % (cvb * 2) == 0) cvb *= 2;
  a.cv_per_block = cvb;
  a.cv_chunks = cvec / cvb;
  a.rows_per_thread = 4;
  const int ty = kThreads / cvb;
  const int64_t gx = ((p.W + ty - 1) / ty) * a.cv_chunks;
  const int64_t gy = (p.H + a.rows_per_thread - 1) / a.rows_per_thread;
  if (gx > 0x7FFFFFFF || gy > 65535 || p.N > 65535) return GBCONV_EUNSUPPORTED;
  const dim3 grid(unsigned(gx), unsigned(gy), unsigned(p.N)), block(cvb, ty);
  const size_t smem = size_t(p.KH * p.KW) * cvb * 8 * sizeof(float);
  auto dyb = static_cast<const __nv_bfloat16*>(dy);
  auto wb = static_cast<const __nv_bfloat16*>(w);
  auto dxb = static_cast<__nv_bfloat16*>(dx);
  if (p.KH == 3 && p.KW == 3 && p.SH == 2 && p.SW == 2 && p.PH == 1 && p.PW == 1 && p.PHe == 1 && p.PWe == 1 &&
      p.DH == 1 && p.DW == 1 &&
      p.OH == (p.H + 1) / 2 && p.OW == (p.W + 1) / 2) {
    if (p.Cin % 64 == 0) return launch_dw_dgrad_tma(p, dy, w, bias, dx, l);
    // One thread per dy column and 8 channels, walking a strip of dy rows: strips as long as
    // possible (each strip start re-reads a dy row) while the grid still fills two blocks per SM.
    // Whole columns measured best for 32x112x112x256 (60.7 us; 8-row strips 68 us, 4-row 83.5 us).
    const int64_t gx3 = ((p.OW + ty - 1) / ty) * a.cv_chunks;
    const int64_t strips = std::max<int64_t>(1, (2 * int64_t(l.num_sms)) / std::max<int64_t>(1, gx3 * p.N));
    a.rows_per_thread = int(std::max<int64_t>(4, (p.OH + strips - 1) / strips));
    const int64_t gy3 = (p.OH + a.rows_per_thread - 1) / a.rows_per_thread;
    if (gx3 > 0x7FFFFFFF || gy3 > 65535) return GBCONV_EUNSUPPORTED;
    auto kern = bias ? depthwise3x3s2_dgrad_kernel<true> : depthwise3x3s2_dgrad_kernel<false>;
    return launch_kernel(kern, dim3(unsigned(gx3), unsigned(gy3), unsigned(p.N)), block, 0, l.stream, a, dyb, wb, bias,
                         dxb) == cudaSuccess
               ? GBCONV_OK
               : GBCONV_ECUDA;
  }
  cudaError_t e;
  if (p.SH == 2 && p.SW == 2)
    e = launch_kernel(depthwise_dgrad_kernel<2>, grid, block, smem, l.stream, a, dyb, wb, bias, dxb);
  else if (p.SH == 1 && p.SW == 1)
    e = launch_kernel(depthwise_dgrad_kernel<1>, grid, block, smem, l.stream, a, dyb, wb, bias, dxb);
  else
    e = launch_kernel(depthwise_dgrad_kernel<0>, grid, block, smem, l.stream, a, dyb, wb, bias, dxb);
  return e == cudaSuccess ? GBCONV_OK : GBCONV_ECUDA;
}

}  // namespace gbconv
