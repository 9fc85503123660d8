// Weight gradient (and bias gradient) of the convolution, deterministic.
//
//   dw[co, cl, kh, kw] = sum over n, oh, ow of dy[n, co, oh, ow] * x[n, g*C_in/G + cl, oh*s_h + kh*d_h - p_h,
//                                                                    ow*s_w + kw*d_w - p_w]
//   db[co]             = sum over n, oh, ow of dy[n, co, oh, ow]
//
// burn-cubecl `wgrad_im2col` computes dw as one contraction of the output gradient with the input's
// columns over every (batch, position), and `wgrad_im2col_1x1_split` cuts that contraction into pieces
// whose partial results are summed afterwards, because the contraction is long and the output small.
// teeny-kernels `conv2d_backward_dw` instead accumulates every CTA's partial sum into dw with atomics,
// whose order (and so whose rounding) changes from run to run.  Here the positions are cut into fixed
// chunks; every partial sum over a chunk is taken in position order by one thread (generic kernel) or
// by one CTA's tensor-core accumulator (tensor-core kernel) and stored in the caller's workspace; a
// second kernel adds the chunks in a fixed order and rounds once.  The same inputs give the same bits.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "problem.h"
#include "ptx.cuh"

namespace gbconv {
namespace {

using bf16 = __nv_bfloat16;

struct WgArgs {
  int N, Cin, Cout, H, W, KH, KW, SH, SW, PH, PW, DH, DW, OH, OW;
  int D, KD, SD, PD, DD, OD;  // depth axis (1, 1, 1, 0, 1, 1 for 1-D and 2-D shapes)
  int cpg, opg;
  int nhwc, ohwi;
  int E;     // weight-gradient elements, in O(D)HWI order (((co*KD + kd)*KH + kh)*KW + kw)*cpg + cl
  int Etot;  // E plus C_out bias-gradient elements when the bias gradient is wanted
  int e0;    // first element this launch computes (E: the bias gradient only)
  int P;     // positions N*OH*OW (the contraction length)
  int S, L;  // chunks and positions per chunk
};

__device__ __forceinline__ float ld_elem(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld_elem(const bf16* p, int64_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void st_elem(float* p, int64_t i, float v) { p[i] = v; }
__device__ __forceinline__ void st_elem(bf16* p, int64_t i, float v) { p[i] = __float2bfloat16_rn(v); }

__device__ __forceinline__ int64_t act_at(const WgArgs& a, int C, int Dd, int Hh, int Ww, int n, int c, int d, int h,
                                          int w) {
  return a.nhwc ? (((int64_t(n) * Dd + d) * Hh + h) * Ww + w) * C + c
                : (((int64_t(n) * C + c) * Dd + d) * Hh + h) * Ww + w;
}

// One thread per (weight-gradient element, chunk): the partial sum over the chunk's positions, in
// position order, with fp32 fused multiply-adds.  Threads of a warp take consecutive c_local, so NHWC
// x reads are coalesced and the dy read is a broadcast.
template <typename T>
__global__ void direct_wgrad_partial_kernel(WgArgs a, const T* __restrict__ x, const T* __restrict__ dy,
                                            float* __restrict__ ws) {
  ptx::grid_dep_wait();
  const int e = a.e0 + int(blockIdx.x) * int(blockDim.x) + int(threadIdx.x);
  const int s = int(blockIdx.y);
  if (e >= a.Etot) return;
  const int p0 = s * a.L, p1 = min(p0 + a.L, a.P);
  float acc = 0.f;
  if (p0 < p1) {
    // position p = ((n*OD + od)*OH + oh)*OW + ow, walked in order
    int ow = p0 % a.OW, q = p0 / a.OW, oh = q % a.OH;
    q /= a.OH;
    int od = q % a.OD, n = q / a.OD;
    if (e < a.E) {
      int t = e;
      const int cl = t % a.cpg;
      t /= a.cpg;
      const int kw = t % a.KW;
      t /= a.KW;
      const int kh = t % a.KH;
      t /= a.KH;
      const int kd = t % a.KD, co = t / a.KD;
      const int ci = (co / a.opg) * a.cpg + cl;
      for (int p = p0; p < p1; ++p) {
        const int id = od * a.SD + kd * a.DD - a.PD;
        const int ih = oh * a.SH + kh * a.DH - a.PH, iw = ow * a.SW + kw * a.DW - a.PW;
        if (id >= 0 && id < a.D && ih >= 0 && ih < a.H && iw >= 0 && iw < a.W)
          acc = fmaf(ld_elem(dy, act_at(a, a.Cout, a.OD, a.OH, a.OW, n, co, od, oh, ow)),
                     ld_elem(x, act_at(a, a.Cin, a.D, a.H, a.W, n, ci, id, ih, iw)), acc);
        if (++ow == a.OW) { ow = 0; if (++oh == a.OH) { oh = 0; if (++od == a.OD) { od = 0; ++n; } } }
      }
    } else {
      const int co = e - a.E;
      for (int p = p0; p < p1; ++p) {
        acc += ld_elem(dy, act_at(a, a.Cout, a.OD, a.OH, a.OW, n, co, od, oh, ow));
        if (++ow == a.OW) { ow = 0; if (++oh == a.OH) { oh = 0; if (++od == a.OD) { od = 0; ++n; } } }
      }
    }
  }
  ws[int64_t(s) * a.Etot + e] = acc;
}

__device__ __forceinline__ void kahan_add(float& acc, float& comp, float v) {
  const float y = v - comp;
  const float t = acc + y;
  comp = (t - acc) - y;
  acc = t;
}

template <typename T>
__device__ __forceinline__ void store_grad(int e, float v, int E, int KH, int KW, int cpg, int ohwi, T* dw, float* db) {
  if (e < E) {
    int t = e;
    const int cl = t % cpg;
    t /= cpg;
    const int kw = t % KW;
    t /= KW;
    const int kh = t % KH, co = t / KH;
    const int64_t o = ohwi ? int64_t(e) : ((int64_t(co) * cpg + cl) * KH + kh) * KW + kw;
    st_elem(dw, o, v);
  } else {
    db[e - E] = v;
  }
}

// Adds the S chunk partials of every element in a fixed order, rounds once, and writes dw in the
// caller's weight layout and db.  A block takes 32*V consecutive elements (V per lane, read as one
// vector when V = 4); warp j sums chunks [j*S/16, (j+1)*S/16) in chunk order, then one thread per
// element adds the sixteen run sums in run order.  Every sum is compensated (Kahan): the order fixes
// the bits, and the compensation keeps the fp32 sum of up to a few hundred partials close to the
// exact one.  The partials were just written and are read once: each warp issues up to six chunk
// loads before it adds any of them, so the reads overlap instead of waiting one round trip each.
// With `discard`, the L2 lines of the partials are dropped once read, so the dead scratch is never
// written back to HBM (the workspace's contents are undefined after the call).  It needs chunk rows
// on 128-byte lines (a 128-byte aligned workspace, Etot a multiple of 32), so that every line a
// block drops holds only elements that block has read.  A block drops lines only when all of its
// 128 columns are in range.
constexpr int kReduceRuns = 16;
constexpr int kReduceBatch = 6;

template <typename T, int V>
__global__ void __launch_bounds__(kReduceRuns * 32, 2) wgrad_reduce_kernel(int E, int Etot, int S, int KH, int KW,
                                                                        int cpg, int ohwi, int discard,
                                                                        const float* __restrict__ ws,
                                                                        T* __restrict__ dw, float* __restrict__ db) {
  ptx::grid_dep_wait();
  __shared__ float part[kReduceRuns][32 * V];
  const int lane = int(threadIdx.x) & 31, j = int(threadIdx.x) >> 5;
  const int e0 = (int(blockIdx.x) * 32 + lane) * V;
  float acc[V], comp[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = comp[v] = 0.f;
  const int s0 = (j * S) / kReduceRuns, s1 = ((j + 1) * S) / kReduceRuns;
  if (V == 4 && e0 + 3 < Etot) {
    // only blocks whose 128 columns are all in range drop lines (then every lane takes this branch)
    const bool drop = discard && (int(blockIdx.x) + 1) * 128 <= Etot;
    for (int s = s0; s < s1; s += kReduceBatch) {
      float4 x[kReduceBatch];
#pragma unroll
      for (int u = 0; u < kReduceBatch; ++u)
        if (s + u < s1) x[u] = __ldcs(reinterpret_cast<const float4*>(ws + int64_t(s + u) * Etot + e0));
#pragma unroll
      for (int u = 0; u < kReduceBatch; ++u)
        if (s + u < s1) {
          kahan_add(acc[0], comp[0], x[u].x);
          kahan_add(acc[1], comp[1], x[u].y);
          kahan_add(acc[2], comp[2], x[u].z);
          kahan_add(acc[3], comp[3], x[u].w);
        }
      if (drop) {
        // the batch's 4 x kReduceBatch lines of this block's 128 columns, one per lane, once every
        // lane's adds have consumed them
        __syncwarp();
        const int u = lane >> 2;
        if (u < kReduceBatch && s + u < s1)
          ptx::discard_l2(ws + int64_t(s + u) * Etot + int(blockIdx.x) * 128 + (lane & 3) * 32);
      }
    }
  } else {
    for (int s = s0; s < s1; ++s)
#pragma unroll
      for (int v = 0; v < V; ++v)
        if (e0 + v < Etot) kahan_add(acc[v], comp[v], ws[int64_t(s) * Etot + e0 + v]);
  }
#pragma unroll
  for (int v = 0; v < V; ++v) part[j][lane * V + v] = acc[v] - comp[v];
  __syncthreads();
  // one thread per element of the block adds the run sums
  const int t = int(threadIdx.x);
  if (t >= 32 * V) return;
  const int e = int(blockIdx.x) * 32 * V + t;
  if (e >= Etot) return;
  float a2 = 0.f, c2 = 0.f;
#pragma unroll
  for (int jj = 0; jj < kReduceRuns; ++jj) kahan_add(a2, c2, part[jj][t]);
  store_grad(e, a2, E, KH, KW, cpg, ohwi, dw, db);
}

constexpr int kChunkPositions = 256;  // target positions per chunk
constexpr int kMaxChunks = 64;

WgArgs direct_args(const Problem& p, bool want_db) {
  WgArgs a{};
  a.N = int(p.N); a.Cin = int(p.Cin); a.Cout = int(p.Cout);
  a.H = int(p.H); a.W = int(p.W); a.KH = int(p.KH); a.KW = int(p.KW);
  a.SH = int(p.SH); a.SW = int(p.SW); a.PH = int(p.PH); a.PW = int(p.PW); a.DH = int(p.DH); a.DW = int(p.DW);
  a.OH = int(p.OH); a.OW = int(p.OW);
  a.D = int(p.D); a.KD = int(p.KD); a.SD = int(p.SD); a.PD = int(p.PD); a.DD = int(p.DD); a.OD = int(p.OD);
  a.cpg = int(p.cpg()); a.opg = int(p.opg());
  a.nhwc = p.nhwc; a.ohwi = p.ohwi;
  a.E = int(p.w_elems());
  a.Etot = a.E + (want_db ? a.Cout : 0);
  a.e0 = 0;
  a.P = int(p.N * p.OD * p.OH * p.OW);
  a.S = int(std::min<int64_t>(kMaxChunks, std::max<int64_t>(1, (int64_t(a.P) + kChunkPositions - 1) / kChunkPositions)));
  a.L = (a.P + a.S - 1) / a.S;
  return a;
}

}  // namespace

int64_t direct_wgrad_workspace(const Problem& p) {
  const WgArgs a = direct_args(p, true);
  return ((int64_t(a.S) * a.Etot * 4 + 255) / 256) * 256;
}

gbconv_status launch_wgrad_reduce(const Problem& p, int S, const float* ws, void* dw, float* db, bool want_db,
                                  const Launch& l) {
  const int E = int(p.w_elems()), Etot = E + (want_db ? int(p.Cout) : 0);
  // float4 reads need every chunk row to start on 16 bytes (the workspace itself is 16-byte aligned)
  const bool vec = Etot % 4 == 0;
  // both weight layouts order (kd, kh, kw) alike, so the kernel's depth and height are one axis here
  const int KDH = int(p.KD * p.KH);
  const int discard = vec && Etot % 32 == 0 && reinterpret_cast<uintptr_t>(ws) % 128 == 0;
  const dim3 grid(vec ? (Etot + 127) / 128 : (Etot + 31) / 32), block(kReduceRuns * 32);
  cudaError_t e;
  if (p.bf16)
    e = vec ? launch_kernel(wgrad_reduce_kernel<bf16, 4>, grid, block, 0, l.stream, E, Etot, S, KDH, int(p.KW),
                            int(p.cpg()), int(p.ohwi), discard, ws, static_cast<bf16*>(dw), db)
            : launch_kernel(wgrad_reduce_kernel<bf16, 1>, grid, block, 0, l.stream, E, Etot, S, KDH, int(p.KW),
                            int(p.cpg()), int(p.ohwi), discard, ws, static_cast<bf16*>(dw), db);
  else
    e = vec ? launch_kernel(wgrad_reduce_kernel<float, 4>, grid, block, 0, l.stream, E, Etot, S, KDH, int(p.KW),
                            int(p.cpg()), int(p.ohwi), discard, ws, static_cast<float*>(dw), db)
            : launch_kernel(wgrad_reduce_kernel<float, 1>, grid, block, 0, l.stream, E, Etot, S, KDH, int(p.KW),
                            int(p.cpg()), int(p.ohwi), discard, ws, static_cast<float*>(dw), db);
  return e == cudaSuccess ? GBCONV_OK : GBCONV_ECUDA;
}

namespace {

gbconv_status launch_partials(const WgArgs& a, const Problem& p, const void* x, const void* dy, float* wsf,
                              const Launch& l) {
  const dim3 grid((a.Etot - a.e0 + 255) / 256, a.S), block(256);
  cudaError_t e;
  if (p.bf16)
    e = launch_kernel(direct_wgrad_partial_kernel<bf16>, grid, block, 0, l.stream, a, static_cast<const bf16*>(x),
                      static_cast<const bf16*>(dy), wsf);
  else
    e = launch_kernel(direct_wgrad_partial_kernel<float>, grid, block, 0, l.stream, a, static_cast<const float*>(x),
                      static_cast<const float*>(dy), wsf);
  return e == cudaSuccess ? GBCONV_OK : GBCONV_ECUDA;
}

}  // namespace

gbconv_status launch_direct_wgrad(const Problem& p, const void* x, const void* dy, void* dw, float* db, void* ws,
                                  const Launch& l) {
  const WgArgs a = direct_args(p, db != nullptr);
  float* wsf = static_cast<float*>(ws);
  const gbconv_status st = launch_partials(a, p, x, dy, wsf, l);
  if (st != GBCONV_OK) return st;
  return launch_wgrad_reduce(p, a.S, wsf, dw, db, db != nullptr, l);
}

gbconv_status launch_bgrad_partials(const Problem& p, const void* dy, int S, float* ws, const Launch& l) {
  WgArgs a = direct_args(p, true);
  a.e0 = a.E;
  a.S = S;
  a.L = (a.P + S - 1) / S;
  return launch_partials(a, p, nullptr, dy, ws, l);
}

}  // namespace gbconv
