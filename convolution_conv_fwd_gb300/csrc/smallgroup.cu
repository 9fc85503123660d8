// Small-group convolution: 1 < G < C with C_in/G = C_out/G = CPG in {2, 4, 8} (grouped 3x3 layers
// of the ResNeXt / RegNet kind), NHWC bf16, on CUDA cores.  Each output channel reads only the CPG
// input channels of its group, so a contraction has CPG * KH * KW terms: far too few for the tensor
// cores' K, and the layer moves about one byte per eight to twenty flops.  The kernels here are
// direct convolutions organised around the memory system.
//
// Definition: teeny-kernels `src/nn/conv/conv2d.rs`, `conv2d_forward` (group window: output channel
// co reads input channels g*C_IN/G .. (g+1)*C_IN/G - 1 with g = co / (C_OUT/G), weight
// [C_OUT, C_IN/G, KH, KW]); oarust `src/rs/ml/matrix/conv.rs`, `conv_2d` (groups).
//
// Forward (and the stride-1 input gradient): a persistent kernel.  A producer lane streams halo
// tiles of the input (the rows and columns a TR x 32 output tile reads, 64 channels, zero fill for
// the padding) into a ring of shared-memory stages with TMA, 128-byte swizzled.  Each of 16 compute
// warps owns four output channels of the 64-channel chunk, each lane one output column, and each
// thread walks the tile's TR rows (8 at unit stride): a warp's weights are the same for all its lanes
// (shared-memory broadcasts, each loaded once per tile), each lane reads its pixels as 8-byte pieces
// that the swizzle spreads over all banks, and at unit stride a 3x3 kernel's input pixel is loaded
// once per kernel column and feeds every output row it reaches.  The tile's outputs go through a
// double-buffered, swizzled shared-memory tile to one TMA tensor store per tile.
// The stride-1 input gradient is the same correlation read the other way round: dx = dy correlated
// with the kernel flipped in both axes, begin padding (K-1)*dil - pad, and the weight transposed
// inside each group (the dgrad's output channel ci takes dy channel g*CPG + o through w[g*CPG + o,
// ci - g*CPG]); the kernel stages its weights that way.
//
// Strided input gradient: the gather form on CUDA cores, one thread per 8 dx channels of one column
// walking a strip of rows, each tap's dy read where (i + pad - k*dil) / stride is exact (teeny-kernels
// `conv2d_backward_dx` scatters the same products with atomics; here every dx element is written
// once, in a fixed order).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "problem.h"
#include "ptx.cuh"

namespace gbconv {
namespace {

constexpr int kTC = 32;                     // output columns per tile (one per lane)
constexpr int kWarps = 16;                  // compute warps, four output channels of the chunk each
constexpr int kCompute = kWarps * 32;
constexpr int kThreads = kCompute;          // thread 0 also issues the loads (no producer warp: at 512
                                            // threads a thread may hold 128 registers)
constexpr int kMaxStages = 4;
constexpr int kSmemLimit = 227 * 1024;
constexpr int kMaxTapTerms = 200;           // taps * CPG: the chunk's weights as fp32 in shared memory

struct SgArgs {
  const float* bias;      // [C] fp32 or null (added once after the sum)
  unsigned int* status;
  uint64_t wait_ns;       // bound of every barrier wait (the host sets it; 2 s by default)
  int N, C;               // batch, channels (C_in == C_out)
  int Hi, Wi, Ho, Wo;     // extents read (x or dy) and written (y or dx)
  int KH, KW, SH, SW, DH, DW, PH, PW;  // the read map: in = out*S + k*D - P (begin-side P)
  int tr;                 // output rows per tile
  int nchunk, tiles_h, tiles_w, tiles_per_chunk;
  int ir, ic;             // halo rows and columns of a tile
  int box_bytes, stage_bytes, stages;
  int out_bytes;          // one output staging tile (tr x 32 pixels x 64 channels, bf16)
  int wbytes;             // the chunk's fp32 weights
};

// Input channels a warp reads per pixel: its four output channels' groups (the same four channels
// for CPG <= 4, the group's eight for CPG = 8).
template <int CPG>
struct In {
  static constexpr int n = CPG <= 4 ? 4 : 8;
};

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

// Weight element for output channel `co` of the read map (a chunk channel), its k-th input channel of
// the group, and tap (kh, kw) of the read map.  Forward: w[co, k, kh, kw].  Transposed (stride-1
// input gradient): the read map's output channel is the dx channel ci, its k-th input the dy channel
// g*CPG + k, and the tap is flipped: w[g*CPG + k, ci - g*CPG, KH-1-kh, KW-1-kw].
template <int CPG>
__device__ __forceinline__ float weight_at(const __nv_bfloat16* __restrict__ w, bool ohwi, bool transposed, int KH,
                                           int KW, int co, int k, int kh, int kw) {
  int o = co, i = k;
  if (transposed) {
    const int g = co / CPG;
    o = g * CPG + k;
    i = co - g * CPG;
    kh = KH - 1 - kh;
    kw = KW - 1 - kw;
  }
  const size_t idx = ohwi ? ((size_t(o) * KH + kh) * KW + kw) * CPG + i : ((size_t(o) * CPG + i) * KH + kh) * KW + kw;
  return __bfloat162float(w[idx]);
}

// Two fp32 lanes in one 64-bit register, and the paired FMA: fma.rn.f32x2 is two independent
// round-to-nearest fp32 FMAs, the same results as two fmaf, in one instruction.
__device__ __forceinline__ uint64_t pack2f(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2f(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// The tap's weights of one warp's 4 channels, laid out [k][channel] in shared memory: for input k, the
// channel pairs (0, 1) and (2, 3) as two packed registers (the same address in every lane: a
// shared-memory broadcast).
template <int CPG>
__device__ __forceinline__ void load_tap_weights(uint32_t wp, uint64_t (&wt)[CPG][2]) {
#pragma unroll
  for (int k = 0; k < CPG; ++k)
    asm volatile("ld.shared.v2.u64 {%0, %1}, [%2];" : "=l"(wt[k][0]), "=l"(wt[k][1]) : "r"(wp + uint32_t(k * 16)));
}

// The warp's input piece of halo pixel `line` (128 bytes per pixel; 128-byte swizzle: the 16-byte
// piece c of line l sits at piece c ^ (l & 7)), as fp32.
template <int CPG>
__device__ __forceinline__ void load_pixel(uint32_t base, int line, int piece, int half, float (&xf)[In<CPG>::n]) {
  const uint32_t addr = base + uint32_t(line * 128 + ((piece ^ (line & 7)) << 4));
  if constexpr (In<CPG>::n == 4) {
    uint32_t u0, u1;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(u0), "=r"(u1) : "r"(addr + uint32_t(half * 8)));
    xf[0] = __uint_as_float(u0 << 16);
    xf[1] = __uint_as_float(u0 & 0xFFFF0000u);
    xf[2] = __uint_as_float(u1 << 16);
    xf[3] = __uint_as_float(u1 & 0xFFFF0000u);
  } else {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    unpack8(v, xf);
  }
}

// The warp's input values as duplicated pairs {x, x}, one per input of the groups it reads.
template <int CPG>
__device__ __forceinline__ void dup_pairs(const float (&xf)[In<CPG>::n], uint64_t (&xd)[In<CPG>::n]) {
#pragma unroll
  for (int i = 0; i < In<CPG>::n; ++i) xd[i] = pack2f(xf[i], xf[i]);
}

// acc pair p (channels 2p, 2p+1, one group) += sum over the group's CPG inputs of x * w, input k
// outermost (each accumulator takes its terms in the order k = 0, 1, ...).
template <int CPG>
__device__ __forceinline__ void group_fma(uint64_t (&acc)[2], const uint64_t (&xd)[In<CPG>::n],
                                          const uint64_t (&wt)[CPG][2]) {
#pragma unroll
  for (int k = 0; k < CPG; ++k)
#pragma unroll
    for (int pp = 0; pp < 2; ++pp) acc[pp] = fma2(xd[(CPG <= 4 ? ((2 * pp) / CPG) * CPG : 0) + k], wt[k][pp], acc[pp]);
}

__device__ __forceinline__ void tma_store_4d(const void* map, uint32_t src, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(map),
               "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// waits until at most N committed bulk groups of this thread still read shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// TR: output rows per tile.  K3: 3x3 kernel at unit stride and dilation, the halo geometry known at
// compile time (CPG <= 4); otherwise any kernel, stride and dilation from the arguments.
template <int CPG, int TR, int K3>
__global__ void __launch_bounds__(kThreads, 1)
    smallgroup_tma_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap ymap,
                          const __grid_constant__ SgArgs a, const __nv_bfloat16* __restrict__ w, int ohwi,
                          int transposed) {
  constexpr int IN = In<CPG>::n;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* out_s = smem + a.stages * a.stage_bytes;                     // 2 output staging tiles
  float* wsm = reinterpret_cast<float*>(out_s + 2 * a.out_bytes);       // [tap][64][CPG]
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(wsm) + a.wbytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + kMaxStages);
  const int KH = K3 ? 3 : a.KH, KW = K3 ? 3 : a.KW;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < a.stages; ++i) ptx::mbar_init(full + i, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  ptx::grid_dep_wait();  // x / dy and w may come from the previous kernel on the stream
  ptx::grid_dep_launch();
  // CTAs are split evenly over the channel chunks, so each stages one chunk's weights once.
  const int chunk = blockIdx.x % a.nchunk;
  const int ctas_per_chunk = gridDim.x / a.nchunk;
  const int first = blockIdx.x / a.nchunk;
  const int taps = KH * KW;
  // Thread 0 issues the halo loads: the k-th tile of this CTA goes to stage k % stages and completes
  // phase k / stages of that stage's barrier.  Stage s is reloaded only after the block-wide barrier
  // that follows the reads of the tile it held.
  int issued = 0;
  auto issue = [&](int k) {
    const int t = first + k * ctas_per_chunk;
    if (t >= a.tiles_per_chunk) return;
    const int tw = t % a.tiles_w, th = (t / a.tiles_w) % a.tiles_h, n = t / (a.tiles_w * a.tiles_h);
    const int s = k % a.stages;
    ptx::mbar_arrive_expect_tx(full + s, uint32_t(a.box_bytes));
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, "
        "%6}], [%2];" ::"r"(ptx::smem_addr(smem + s * a.stage_bytes)),
        "l"(&xmap), "r"(ptx::smem_addr(full + s)), "r"(chunk * 64), "r"(tw * kTC * a.SW - a.PW),
        "r"(th * TR * a.SH - a.PH), "r"(n)
        : "memory");
    issued = k + 1;
  };
  if (threadIdx.x == 0) {
    ptx::prefetch_tmap(&xmap);
    for (int k = 0; k < a.stages; ++k) issue(k);  // the first halos first: they come from HBM
  }
  // weights [tap][warp][k][4 channels] (a warp's channels for one input are one 16-byte piece)
  for (int e = threadIdx.x; e < taps * 64 * CPG; e += kThreads) {
    const int j = e & 3, k = (e >> 2) % CPG, wq = (e / (4 * CPG)) % 16, t = e / (64 * CPG);
    wsm[e] = weight_at<CPG>(w, ohwi != 0, transposed != 0, KH, KW, chunk * 64 + wq * 4 + j, k, t / KW, t % KW);
  }
  __syncthreads();

  const int c = chunk * 64 + warp * 4;  // this warp's 4 output channels
  const int piece = warp >> 1;          // its 16-byte piece of a pixel's 64 channels
  const int half = warp & 1;            // and the 8-byte half of it (CPG <= 4)
  float b[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) b[j] = a.bias ? __ldg(a.bias + c + j) : 0.f;
  const uint32_t wv = ptx::smem_addr(wsm) + uint32_t(warp * CPG * 16);  // tap 0, this warp's weights
  for (int k = 0;; ++k) {
    const int t = first + k * ctas_per_chunk;
    if (t >= a.tiles_per_chunk) break;
    const int tw = t % a.tiles_w, th = (t / a.tiles_w) % a.tiles_h, n = t / (a.tiles_w * a.tiles_h);
    const int st = k % a.stages;
    const bool got = ptx::mbar_wait(full + st, uint32_t((k / a.stages) & 1), abort_flag, a.status, 64u, a.wait_ns);
    const uint32_t base = ptx::smem_addr(smem + st * a.stage_bytes);
    uint64_t acc[TR][2];  // channel pairs (0, 1) and (2, 3) of each row
#pragma unroll
    for (int r = 0; r < TR; ++r) {
      acc[r][0] = pack2f(b[0], b[1]);
      acc[r][1] = pack2f(b[2], b[3]);
    }
    if (got) {
      if constexpr (K3 && CPG <= 4) {
        // Each of the (TR + 2) x 3 halo pixels a thread reads is loaded and converted once and feeds
        // every output row that reads it through its kernel row; the weights of one kernel column
        // (three taps) stay in registers meanwhile.
        constexpr int IC = kTC + 2;
#pragma unroll 1
        for (int kw = 0; kw < 3; ++kw) {
          uint64_t wt[3][CPG][2];
#pragma unroll
          for (int kh = 0; kh < 3; ++kh) load_tap_weights<CPG>(wv + uint32_t((kh * 3 + kw) * 64 * CPG * 4), wt[kh]);
#pragma unroll
          for (int rho = 0; rho < TR + 2; ++rho) {
            float xf[IN];
            uint64_t xd[IN];
            load_pixel<CPG>(base, rho * IC + lane + kw, piece, half, xf);
            dup_pairs<CPG>(xf, xd);
#pragma unroll
            for (int kh = 0; kh < 3; ++kh)
              if (rho - kh >= 0 && rho - kh < TR) group_fma<CPG>(acc[rho - kh], xd, wt[kh]);
          }
        }
      } else {
        const int SH = K3 ? 1 : a.SH, SW = K3 ? 1 : a.SW, DH = K3 ? 1 : a.DH, DW = K3 ? 1 : a.DW;
        const int IC = K3 ? kTC + 2 : a.ic;
#pragma unroll 1
        for (int kh = 0; kh < KH; ++kh) {
#pragma unroll 1
          for (int kw = 0; kw < KW; ++kw) {
            uint64_t wt[CPG][2];
            load_tap_weights<CPG>(wv + uint32_t((kh * KW + kw) * 64 * CPG * 4), wt);
            const int col = lane * SW + kw * DW;
#pragma unroll
            for (int r = 0; r < TR; ++r) {
              float xf[IN];
              uint64_t xd[IN];
              load_pixel<CPG>(base, (r * SH + kh * DH) * IC + col, piece, half, xf);
              dup_pairs<CPG>(xf, xd);
              group_fma<CPG>(acc[r], xd, wt);
            }
          }
        }
      }
    }
    // The output tile: the store that last used this staging buffer must have read it, and all
    // threads must agree to go on (leave together if any of them gave up: the barriers below count
    // every thread).  Past this barrier every thread has finished reading input stage st.
    const int ob = k & 1;
    if (threadIdx.x == 0) bulk_wait_read<1>();
    uint32_t stop;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.eq.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(stop)
        : "r"(uint32_t(got)), "n"(kThreads)
        : "memory");
    if (stop) break;
    if (threadIdx.x == 0) issue(k + a.stages);  // refill the stage just read
    const uint32_t ob_s = ptx::smem_addr(out_s + ob * a.out_bytes);
#pragma unroll
    for (int r = 0; r < TR; ++r) {
      const int line = r * kTC + lane;  // the staging tile is (row, column, 64 channels), swizzled
      float y0, y1, y2, y3;
      unpack2f(acc[r][0], y0, y1);
      unpack2f(acc[r][1], y2, y3);
      asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(ob_s + uint32_t(line * 128 + ((piece ^ (line & 7)) << 4) +
                                                                            half * 8)),
                   "r"(ptx::pack_bf16x2(y0, y1)), "r"(ptx::pack_bf16x2(y2, y3))
                   : "memory");
    }
    ptx::fence_proxy_async_smem();  // the tile's writes before the tensor store reads it
    asm volatile("bar.sync 2, %0;" ::"n"(kThreads) : "memory");
    if (threadIdx.x == 0) {  // rows and columns past the output are clipped by the store
      tma_store_4d(&ymap, ob_s, chunk * 64, tw * kTC, th * TR, n);
      bulk_commit();
    }
  }
  if (threadIdx.x == 0) {
    // Drain: loads still in flight (after an abort) write this CTA's shared memory; the last `stages`
    // issued are the only ones that can be.
    for (int k = max(0, issued - a.stages); k < issued; ++k)
      ptx::mbar_wait_drain(full + (k % a.stages), uint32_t((k / a.stages) & 1));
    bulk_wait_all();  // every tensor store has completed before the CTA leaves
  }
}

// ---------------------------------------------------------------- strided input gradient (gather)
struct SgDgArgs {
  int N, C, H, W, OH, OW, KH, KW, SH, SW, PH, PW, DH, DW;
  int rows_per_thread, cv_per_block, cv_chunks;
  int ohwi;
};

template <int CPG>
__global__ void __launch_bounds__(256) smallgroup_dgrad_kernel(SgDgArgs a, const __nv_bfloat16* __restrict__ dy,
                                                               const __nv_bfloat16* __restrict__ w,
                                                               const float* __restrict__ bias,
                                                               __nv_bfloat16* __restrict__ dx) {
  ptx::grid_dep_wait();  // inputs may come from the previous kernel on the stream
  ptx::grid_dep_launch();
  const int KH = a.KH, KW = a.KW, taps = KH * KW;
  extern __shared__ __align__(16) float wsg[];  // [tap][block channel][CPG]: dx channel's weight per dy channel
  const int cpb = a.cv_per_block * 8;
  const int chunk = blockIdx.x % a.cv_chunks;
  const int c0 = chunk * cpb;
  const int nthreads = blockDim.x * blockDim.y;
  for (int e = threadIdx.y * blockDim.x + threadIdx.x; e < taps * cpb * CPG; e += nthreads) {
    const int o = e % CPG, jj = (e / CPG) % cpb, t = e / (CPG * cpb);
    const int ci = c0 + jj, g = ci / CPG, il = ci - g * CPG, co = g * CPG + o, kh = t / KW, kw = t % KW;
    const size_t idx = a.ohwi ? ((size_t(co) * KH + kh) * KW + kw) * CPG + il : ((size_t(co) * CPG + il) * KH + kh) * KW + kw;
    wsg[e] = __bfloat162float(w[idx]);
  }
  __syncthreads();
  const int iw = (blockIdx.x / a.cv_chunks) * blockDim.y + threadIdx.y;  // dx column
  const int cv = threadIdx.x;
  const int n = blockIdx.z;
  if (iw >= a.W) return;
  const int ih0 = blockIdx.y * a.rows_per_thread;
  const int ih1 = min(a.H, ih0 + a.rows_per_thread);
  const int c = c0 + cv * 8;  // this thread's dx channels; with CPG | 8 they read dy channels c .. c+7
  const uint4* dyv = reinterpret_cast<const uint4*>(dy);
  uint4* dxv = reinterpret_cast<uint4*>(dx);
  const int cvec = a.C / 8;
  float bs[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) bs[j] = bias ? __ldg(bias + c + j) : 0.f;
  for (int ih = ih0; ih < ih1; ++ih) {
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    for (int kh = 0; kh < KH; ++kh) {
      const int nh = ih + a.PH - kh * a.DH;
      if (nh < 0 || nh % a.SH != 0) continue;
      const int oh = nh / a.SH;
      if (oh >= a.OH) continue;
      for (int kw = 0; kw < KW; ++kw) {
        const int nw = iw + a.PW - kw * a.DW;
        if (nw < 0 || nw % a.SW != 0) continue;
        const int ow = nw / a.SW;
        if (ow >= a.OW) continue;
        float g[8];
        unpack8(__ldg(dyv + (size_t(n * a.OH + oh) * a.OW + ow) * cvec + (c >> 3)), g);
        const float* wt = wsg + ((kh * KW + kw) * cpb + cv * 8) * CPG;
#pragma unroll
        for (int o = 0; o < CPG; ++o)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[j] = fmaf(g[(j / CPG) * CPG + o], wt[j * CPG + o], acc[j]);
      }
    }
    uint4 o;
    o.x = ptx::pack_bf16x2(acc[0] + bs[0], acc[1] + bs[1]);
    o.y = ptx::pack_bf16x2(acc[2] + bs[2], acc[3] + bs[3]);
    o.z = ptx::pack_bf16x2(acc[4] + bs[4], acc[5] + bs[5]);
    o.w = ptx::pack_bf16x2(acc[6] + bs[6], acc[7] + bs[7]);
    dxv[(size_t(n * a.H + ih) * a.W + iw) * cvec + (c >> 3)] = o;
  }
}

PFN_cuTensorMapEncodeTiled_v12000 sg_encode_fn() {
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

// The shapes of the regime: bf16 NHWC, 1 < G < C, C_in = C_out, C_in/G in {2, 4, 8}, whole
// 64-channel chunks (a chunk then holds whole groups).
bool regime(const Problem& p) {
  const int64_t cpg = p.G > 0 ? p.Cin / p.G : 0;
  return p.bf16 && p.nhwc && p.G > 1 && p.G < p.Cin && p.Cin == p.Cout && (cpg == 2 || cpg == 4 || cpg == 8) &&
         p.Cin % 64 == 0 && p.KH * p.KW * cpg <= kMaxTapTerms;
}

// The tiled kernel's read map for the forward or the stride-1 input gradient; false when a tile's
// halo does not fit a TMA box or the shared memory.
bool plan(const Problem& p, bool dgrad, SgArgs& a, size_t& smem) {
  if (!regime(p)) return false;
  if (dgrad && (p.SH != 1 || p.SW != 1)) return false;
  a = SgArgs{};
  a.N = int(p.N);
  a.C = int(p.Cin);
  a.KH = int(p.KH); a.KW = int(p.KW); a.DH = int(p.DH); a.DW = int(p.DW);
  if (!dgrad) {
    a.Hi = int(p.H); a.Wi = int(p.W); a.Ho = int(p.OH); a.Wo = int(p.OW);
    a.SH = int(p.SH); a.SW = int(p.SW); a.PH = int(p.PH); a.PW = int(p.PW);
  } else {
    // dx[i] = sum_k dy[i + P - k*D] w[k] = sum_k' dy[i + k'*D - ((K-1)*D - P)] w[K-1-k']
    a.Hi = int(p.OH); a.Wi = int(p.OW); a.Ho = int(p.H); a.Wo = int(p.W);
    a.SH = 1; a.SW = 1;
    a.PH = int((p.KH - 1) * p.DH - p.PH);
    a.PW = int((p.KW - 1) * p.DW - p.PW);
  }
  if (a.SH > 2 || a.SW > 2) return false;
  // 8 output rows per tile at unit row stride, else (or when the halo leaves room for fewer than two
  // stages) 4
  a.wbytes = int(p.KH * p.KW) * 64 * int(p.Cin / p.G) * 4;
  int fixed = 0;
  a.stages = 0;
  for (int tr = (a.SH == 1 ? 8 : 4); tr >= 4 && a.stages < 2; tr -= 4) {
    a.tr = tr;
    const int64_t ir = int64_t(a.tr - 1) * a.SH + int64_t(a.KH - 1) * a.DH + 1;
    const int64_t ic = int64_t(kTC - 1) * a.SW + int64_t(a.KW - 1) * a.DW + 1;
    if (ir > 256 || ic > 256) return false;  // TMA box extents
    a.ir = int(ir);
    a.ic = int(ic);
    a.box_bytes = a.ir * a.ic * 128;
    a.stage_bytes = (a.box_bytes + 1023) & ~1023;
    a.out_bytes = a.tr * kTC * 128;
    fixed = 1024 + 2 * a.out_bytes + a.wbytes + kMaxStages * 8 + 16;
    a.stages = std::max(0, std::min(kMaxStages, (kSmemLimit - fixed) / a.stage_bytes));
  }
  if (a.stages < 2) return false;
  a.nchunk = a.C / 64;
  a.tiles_h = (a.Ho + a.tr - 1) / a.tr;
  a.tiles_w = (a.Wo + kTC - 1) / kTC;
  const int64_t tpc = int64_t(a.N) * a.tiles_h * a.tiles_w;
  if (tpc >= (int64_t(1) << 30)) return false;
  a.tiles_per_chunk = int(tpc);
  smem = size_t(fixed) + size_t(a.stages) * a.stage_bytes;
  return true;
}

// (C, W, H, N) map of an NHWC bf16 tensor with boxes of 64 channels x bw columns x bh rows, 128-byte
// swizzle (zero fill on loads past the edges; stores past them are clipped).
bool encode_act(CUtensorMap* map, const void* base, int C, int W, int H, int N, int bw, int bh) {
  auto fn = sg_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {cuuint64_t(C), cuuint64_t(W), cuuint64_t(H), cuuint64_t(N)};
  cuuint64_t strides[3] = {cuuint64_t(C) * 2, cuuint64_t(W) * C * 2, cuuint64_t(H) * W * C * 2};
  cuuint32_t box[4] = {64, cuuint32_t(bw), cuuint32_t(bh), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int CPG, int TR, int K3>
gbconv_status run_tiled(const CUtensorMap& xmap, const CUtensorMap& ymap, const SgArgs& a, size_t smem,
                        const void* w, int ohwi, int dgrad, const Launch& l) {
  auto kern = smallgroup_tma_kernel<CPG, TR, K3>;
  static std::atomic<int> raised[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GBCONV_ECUDA;
  if (!raised[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit) != cudaSuccess)
      return GBCONV_ECUDA;
    raised[dev].store(1, std::memory_order_release);
  }
  // a multiple of the chunk count, at most one CTA per SM and per tile
  int64_t grid = std::max<int64_t>(a.nchunk, (int64_t(l.num_sms) / a.nchunk) * a.nchunk);
  grid = std::min<int64_t>(grid, int64_t(a.nchunk) * a.tiles_per_chunk);
  return launch_kernel(kern, dim3(unsigned(grid)), dim3(kThreads), smem, l.stream, xmap, ymap, a,
                       static_cast<const __nv_bfloat16*>(w), ohwi, dgrad) == cudaSuccess
             ? GBCONV_OK
             : GBCONV_ECUDA;
}

template <int CPG>
gbconv_status launch_tiled(const Problem& p, bool dgrad, const void* src, const void* w, const float* bias, void* dst,
                           const Launch& l) {
  SgArgs a;
  size_t smem = 0;
  if (!plan(p, dgrad, a, smem)) return GBCONV_EUNSUPPORTED;
  a.bias = bias;
  a.status = l.status;
  a.wait_ns = l.wait_ns;
  CUtensorMap xmap, ymap;
  if (!encode_act(&xmap, src, a.C, a.Wi, a.Hi, a.N, a.ic, a.ir)) return GBCONV_ECUDA;
  if (!encode_act(&ymap, dst, a.C, a.Wo, a.Ho, a.N, kTC, a.tr)) return GBCONV_ECUDA;
  const int ohwi = p.ohwi ? 1 : 0;
  // the compile-time 3x3 variant up to 4 channels per group (at 8 its weights no longer fit the
  // registers next to the accumulators); the read map's stride and dilation decide (the stride-1
  // input gradient reads at unit stride)
  const bool k3 = CPG <= 4 && a.KH == 3 && a.KW == 3 && a.SH == 1 && a.SW == 1 && a.DH == 1 && a.DW == 1;
  if constexpr (CPG <= 4) {
    if (k3) return run_tiled<CPG, 8, 1>(xmap, ymap, a, smem, w, ohwi, int(dgrad), l);
  }
  if (a.tr == 8) return run_tiled<CPG, 8, 0>(xmap, ymap, a, smem, w, ohwi, int(dgrad), l);
  return run_tiled<CPG, 4, 0>(xmap, ymap, a, smem, w, ohwi, int(dgrad), l);
}

template <int CPG>
gbconv_status launch_gather(const Problem& p, const void* dy, const void* w, const float* bias, void* dx,
                            const Launch& l) {
  SgDgArgs a{};
  a.N = int(p.N); a.C = int(p.Cin); a.H = int(p.H); a.W = int(p.W); a.OH = int(p.OH); a.OW = int(p.OW);
  a.KH = int(p.KH); a.KW = int(p.KW); a.SH = int(p.SH); a.SW = int(p.SW); a.PH = int(p.PH); a.PW = int(p.PW);
  a.DH = int(p.DH); a.DW = int(p.DW);
  a.ohwi = p.ohwi ? 1 : 0;
  const int cvec = a.C / 8, taps = a.KH * a.KW;
  // channel vectors per block: a power of two dividing C/8, with the block's weights within 48 KB
  int cvb = 1;
  while (cvb < 32 && cvec % (cvb * 2) == 0 && size_t(taps) * (cvb * 2) * 8 * CPG * 4 <= 48 * 1024) cvb *= 2;
  a.cv_per_block = cvb;
  a.cv_chunks = cvec / cvb;
  a.rows_per_thread = 4;
  const int ty = 256 / cvb;
  const int64_t gx = ((p.W + ty - 1) / ty) * a.cv_chunks;
  const int64_t gy = (p.H + a.rows_per_thread - 1) / a.rows_per_thread;
  if (gx > 0x7FFFFFFF || gy > 65535 || p.N > 65535) return GBCONV_EUNSUPPORTED;
  const size_t smem = size_t(taps) * cvb * 8 * CPG * 4;
  return launch_kernel(smallgroup_dgrad_kernel<CPG>, dim3(unsigned(gx), unsigned(gy), unsigned(p.N)), dim3(cvb, ty),
                       smem, l.stream, a, static_cast<const __nv_bfloat16*>(dy), static_cast<const __nv_bfloat16*>(w),
                       bias, static_cast<__nv_bfloat16*>(dx)) == cudaSuccess
             ? GBCONV_OK
             : GBCONV_ECUDA;
}

}  // namespace

bool smallgroup_supported(const Problem& p) {
  SgArgs a;
  size_t smem;
  return plan(p, false, a, smem);
}

bool smallgroup_dgrad_supported(const Problem& p) {
  if (!regime(p)) return false;
  SgArgs a;
  size_t smem;
  if (p.SH == 1 && p.SW == 1) return plan(p, true, a, smem);
  return int64_t(p.KH) * p.KW * 8 * (p.Cin / p.G) * 4 <= 48 * 1024;  // the gather kernel's weights
}

gbconv_status launch_smallgroup_fwd(const Problem& p, const void* x, const void* w, const float* bias, void* y,
                                    const Launch& l) {
  switch (p.Cin / p.G) {
    case 2: return launch_tiled<2>(p, false, x, w, bias, y, l);
    case 4: return launch_tiled<4>(p, false, x, w, bias, y, l);
    case 8: return launch_tiled<8>(p, false, x, w, bias, y, l);
  }
  return GBCONV_EUNSUPPORTED;
}

gbconv_status launch_smallgroup_dgrad(const Problem& p, const void* dy, const void* w, const float* bias, void* dx,
                                      const Launch& l) {
  if (!smallgroup_dgrad_supported(p)) return GBCONV_EUNSUPPORTED;
  const bool tiled = p.SH == 1 && p.SW == 1;
  switch (p.Cin / p.G) {
    case 2: return tiled ? launch_tiled<2>(p, true, dy, w, bias, dx, l) : launch_gather<2>(p, dy, w, bias, dx, l);
    case 4: return tiled ? launch_tiled<4>(p, true, dy, w, bias, dx, l) : launch_gather<4>(p, dy, w, bias, dx, l);
    case 8: return tiled ? launch_tiled<8>(p, true, dy, w, bias, dx, l) : launch_gather<8>(p, dy, w, bias, dx, l);
  }
  return GBCONV_EUNSUPPORTED;
}

bool smallgroup_describe(const Problem& p, bool dgrad, char* buf, size_t len) {
  SgArgs a;
  size_t smem = 0;
  if (!plan(p, dgrad, a, smem)) return false;
  std::snprintf(buf, len, "smallgroup%s cpg=%d tile=%dx%d halo=%dx%d stages=%d chunks=%d tiles=%d smem=%zu",
                dgrad ? "_dgrad" : "", int(p.Cin / p.G), a.tr, kTC, a.ir, a.ic, a.stages, a.nchunk,
                a.nchunk * a.tiles_per_chunk, smem);
  return true;
}

}  // namespace gbconv
