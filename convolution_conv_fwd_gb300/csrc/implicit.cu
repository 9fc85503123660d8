// Implicit-GEMM convolution on the 5th-generation tensor cores (tcgen05,
// accumulators in TMEM), NHWC bf16, fp32 accumulation.  One kernel template
// serves two regimes:
//
//  * dense forward at unit stride (the 3x3 workload): y = sum over taps of a
//    shifted window of x times the tap's [C_out, C_in] weight slice;
//  * the input gradient at any stride up to 2x2, in gather form: dx is split
//    into stride phases (ih % s_h, iw % s_w); inside one phase every tap that
//    reaches it does so at a fixed integer shift of dy, so each phase is again
//    a sum of shifted windows, now of dy, times transposed weight slices.
//    Each dx element is produced by exactly one accumulator and written once;
//    there are no atomics and the result is deterministic.
//
// No im2col matrix is materialised (burn-cubecl `im2col.rs` notes that the
// column matrix holds every pixel once per tap that reads it, nine times for
// a 3x3).  Instead, a tile of 128 * NSUB consecutive positions of a "virtual
// grid" (the output rows, each widened by the kernel's horizontal reach) is
// computed from one halo tile in shared memory: position q of the tile reads
// tap t at halo row q + off(t), so every tap's A operand is the same halo
// tile with a different start address.  The halo is stored in the no-swizzle
// K-major core-matrix layout ([8-channel chunk][halo row][16 bytes]) whose
// rows are 16 bytes apart, so a shift by any number of rows is a plain
// descriptor offset.
//
// Roles (warp specialised, one CTA per SM, persistent over work items):
//   warps 0-3  epilogue: TMEM -> registers, + bias, -> bf16, NHWC stores
//   warp  4    TMEM allocation; lane 0 issues every tcgen05.mma and commit
//   warps 5-8  producers: cp.async halo fill (zero fill covers the padding)
//              and weight tiles (transposed in registers for the gradient)
//
// Definitions followed: forward as teeny-kernels `conv2d_forward` (read
// position oh*stride + kh*dil - pad, zero outside) with bias added once after
// the reduction as in `conv2d_bias_forward`; gradient as the exact transpose
// of teeny-kernels `conv2d_backward_dx` (scatter), evaluated per input
// element as oarust `conv_2d_backward` dispatches it.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>

#include "problem.h"
#include "ptx.cuh"

namespace gbconv {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kMaxPhases = 4;
constexpr int kMaxTapsPerPhase = 32;
constexpr int kEpiWarps = 4;
constexpr int kMmaWarp = 4;
constexpr int kProdWarps = 4;
constexpr int kProdThreads = kProdWarps * 32;
constexpr int kThreads = (kEpiWarps + 1 + kProdWarps) * 32;
constexpr int kSmemLimit = 227 * 1024;

struct Phase {
  int ntaps;
  int R;       // output rows of the virtual grid per image
  int RS;      // virtual rows per image (R plus the vertical reach of the taps)
  int P;       // virtual grid pitch: valid columns plus the horizontal reach
  int OWv;     // valid columns
  int rmin, cmin;             // input coordinate of virtual (0, 0)
  int out_sh, out_sw, out_ph, out_pw;  // output pixel = (r*out_sh + out_ph, c*out_sw + out_pw)
  int tiles;   // m-tiles of this phase
  int item0;   // first work item of this phase
  int tap_off[kMaxTapsPerPhase];  // halo row offset of tap t
  int tap_w[kMaxTapsPerPhase];    // weight tap index kh*KW + kw
};

struct Args {
  const bf16* in;     // gathered tensor, NHWC [N, Hi, Wi, Ck]: x (forward) or dy (gradient)
  const bf16* w;      // weight, OHWI [C_out, KH, KW, C_in]
  const float* bias;  // [Cn] or null
  bf16* out;          // NHWC [N, Ho, Wo, Cn]: y or dx
  unsigned int* status;
  int N, Hi, Wi, Ck;  // gathered side; Ck is the reduction channel count
  int Cn;             // output channels (the GEMM N extent)
  int Ho, Wo;
  int T;              // KH*KW
  int Cw;             // innermost extent of the weight (the convolution's C_in)
  int kbc, kb_count;  // channels per k-block and k-blocks per tap
  int n_tiles;
  int halo, hp;       // halo rows of a tile, rows per halo slab (hp % 8 == 1)
  int a_stage_bytes, b_tile_bytes, sa, sb;  // stage sizes and ring depths
  int nphase, total_items;
  Phase ph[kMaxPhases];
};

// B tile layout: [k chunk of 8][row group of 8][row % 8][16 bytes].
template <bool DGRAD>
struct BLayout {
  static constexpr uint32_t sbo = DGRAD ? 144 : 128;  // padded for the transposed stores
  __host__ __device__ static constexpr uint32_t lbo(int bn) { return uint32_t(bn / 8) * sbo + 16; }
};

__device__ __forceinline__ void decode_item(const Args& a, int item, int& phase, int& mtile, int& ntile) {
  int p = 0;
  while (p + 1 < a.nphase && item >= a.ph[p + 1].item0) ++p;
  phase = p;
  const int local = item - a.ph[p].item0;
  mtile = local / a.n_tiles;
  ntile = local - mtile * a.n_tiles;
}

// 8x8 transpose of bf16: r[j] holds row j (8 values), out[i] receives column i.
__device__ __forceinline__ void transpose8x8(const uint4 (&r)[8], uint4 (&o)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t sel = (i & 1) ? 0x7632u : 0x5410u;
    uint32_t c[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t v = (i >> 1) == 0 ? r[j].x : (i >> 1) == 1 ? r[j].y : (i >> 1) == 2 ? r[j].z : r[j].w;
      c[j] = v;
    }
    o[i].x = __byte_perm(c[0], c[1], sel);
    o[i].y = __byte_perm(c[2], c[3], sel);
    o[i].z = __byte_perm(c[4], c[5], sel);
    o[i].w = __byte_perm(c[6], c[7], sel);
  }
}

template <int BN, int NSUB, bool DGRAD, bool BRES>
__global__ void __launch_bounds__(kThreads, 1) implicit_gemm_kernel(const __grid_constant__ Args a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  using BL = BLayout<DGRAD>;
  constexpr uint32_t kTmemCols = (2 * NSUB * BN) <= 32 ? 32 : (2 * NSUB * BN);
  constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(128, BN);
  const uint32_t lbo_b = BL::lbo(BN);
  const int KC = a.kbc / 8;

  uint8_t* a_base = smem;
  uint8_t* b_base = a_base + size_t(a.sa) * a.a_stage_bytes;
  const int b_tiles = BRES ? a.T * a.kb_count : a.sb;
  uint64_t* bars = reinterpret_cast<uint64_t*>(b_base + size_t(b_tiles) * a.b_tile_bytes);
  uint64_t* fullA = bars;
  uint64_t* emptyA = fullA + a.sa;
  uint64_t* fullB = emptyA + a.sa;
  uint64_t* emptyB = fullB + a.sb;
  uint64_t* tfull = emptyB + a.sb;
  uint64_t* tempty = tfull + 2;
  uint64_t* bres = tempty + 2;
  uint64_t* fin = bres + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fin + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.sa; ++i) { ptx::mbar_init(fullA + i, kProdThreads); ptx::mbar_init(emptyA + i, 1); }
    for (int i = 0; i < a.sb; ++i) { ptx::mbar_init(fullB + i, kProdThreads); ptx::mbar_init(emptyB + i, 1); }
    for (int i = 0; i < 2; ++i) { ptx::mbar_init(tfull + i, 1); ptx::mbar_init(tempty + i, kEpiWarps * 32); }
    ptx::mbar_init(bres, kProdThreads);
    ptx::mbar_init(fin, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(tmem_slot, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= kEpiWarps + 1) {
    // ------------------------------------------------------------ producers
    const int pt = threadIdx.x - (kEpiWarps + 1) * 32;
    uint64_t* pending = nullptr;  // full barrier of the last committed, not yet signalled cp.async group
    auto flush = [&]() {
      if (pending) {
        ptx::cp_async_wait_all();
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(pending);
        pending = nullptr;
      }
    };
    auto push = [&](uint64_t* bar) {
      ptx::cp_async_commit();
      if (pending) {
        ptx::cp_async_wait_group<1>();
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(pending);
      }
      pending = bar;
    };
    auto wait_empty = [&](uint64_t* bar, uint32_t parity) -> bool {
      if (ptx::mbar_try_wait(bar, parity)) return true;
      flush();
      return ptx::mbar_wait(bar, parity, abort_flag, a.status, 1u);
    };
    // Forward weight tile: rows = output channels n0.., K = input channels of k-block kb, tap wt.
    auto fill_b_fwd = [&](uint8_t* tile, int wt, int kb, int n0) {
      const uint32_t dst0 = ptx::smem_addr(tile);
      for (int c = pt; c < BN * KC; c += kProdThreads) {
        const int kc = c % KC, row = c / KC;
        const bf16* src = a.w + (size_t(n0 + row) * a.T + wt) * a.Cw + kb * a.kbc + kc * 8;
        ptx::cp_async_16(dst0 + kc * lbo_b + (row >> 3) * BL::sbo + (row & 7) * 16, src, 16);
      }
    };
    // Gradient weight tile: rows = input channels n0.., K = output channels of k-block kb, tap wt.
    auto fill_b_dgrad = [&](uint8_t* tile, int wt, int kb, int n0) {
      const uint32_t dst0 = ptx::smem_addr(tile);
      const int rbs = BN / 8;
      for (int u = pt; u < rbs * KC; u += kProdThreads) {
        const int rb = u % rbs, kc = u / rbs;
        uint4 r[8], o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int co = kb * a.kbc + kc * 8 + j;
          r[j] = __ldg(reinterpret_cast<const uint4*>(a.w + (size_t(co) * a.T + wt) * a.Cw + n0 + rb * 8));
        }
        transpose8x8(r, o);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t d = dst0 + kc * lbo_b + rb * BL::sbo + i * 16;
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(d), "r"(o[i].x), "r"(o[i].y), "r"(o[i].z),
                       "r"(o[i].w)
                       : "memory");
        }
      }
    };

    bool ok = true;
    if (BRES) {  // the whole weight stays resident; only one n-tile exists in this mode
      for (int wt = 0; wt < a.T; ++wt)
        for (int kb = 0; kb < a.kb_count; ++kb) fill_b_fwd(b_base + size_t(wt * a.kb_count + kb) * a.b_tile_bytes, wt, kb, 0);
      ptx::cp_async_commit();
      ptx::cp_async_wait_all();
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(bres);
    }
    int sa = 0, sb = 0;
    uint32_t pa = 0, pb = 0;
    const int hs = kProdThreads / KC;  // halo rows advanced per pass of the producer threads
    for (int item = blockIdx.x; ok && item < a.total_items; item += gridDim.x) {
      int phase, mtile, ntile;
      decode_item(a, item, phase, mtile, ntile);
      const Phase& ph = a.ph[phase];
      if (ph.ntaps == 0) continue;
      const int q0 = mtile * 128 * NSUB;
      const int n0 = ntile * BN;
      const int img = ph.RS * ph.P;
      for (int kb = 0; ok && kb < a.kb_count; ++kb) {
        if (!(ok = wait_empty(emptyA + sa, pa ^ 1))) break;
        {
          const uint32_t dst0 = ptx::smem_addr(a_base + size_t(sa) * a.a_stage_bytes);
          const int kc = pt % KC;
          int h = pt / KC;
          int q = q0 + h;
          int n = q / img, rem = q - n * img;
          int r = rem / ph.P, col = rem - r * ph.P;
          const bf16* chan = a.in + kb * a.kbc + kc * 8;
          for (; h < a.halo; h += hs) {
            const int ih = r + ph.rmin, iw = col + ph.cmin;
            const bool valid = n < a.N && ih >= 0 && ih < a.Hi && iw >= 0 && iw < a.Wi;
            const bf16* src = valid ? chan + (size_t(n * a.Hi + ih) * a.Wi + iw) * a.Ck : a.in;
            ptx::cp_async_16(dst0 + kc * (a.hp * 16) + h * 16, src, valid ? 16u : 0u);
            col += hs;
            while (col >= ph.P) {
              col -= ph.P;
              if (++r == ph.RS) { r = 0; ++n; }
            }
          }
        }
        push(fullA + sa);
        if (++sa == a.sa) { sa = 0; pa ^= 1; }
        if (!BRES) {
          for (int t = 0; ok && t < ph.ntaps; ++t) {
            if (!(ok = wait_empty(emptyB + sb, pb ^ 1))) break;
            uint8_t* tile = b_base + size_t(sb) * a.b_tile_bytes;
            if (DGRAD) {
              fill_b_dgrad(tile, ph.tap_w[t], kb, n0);
              ptx::fence_proxy_async_smem();
              ptx::mbar_arrive(fullB + sb);
            } else {
              fill_b_fwd(tile, ph.tap_w[t], kb, n0);
              push(fullB + sb);
            }
            if (++sb == a.sb) { sb = 0; pb ^= 1; }
          }
        }
      }
    }
    flush();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      if (BRES) ok = ptx::mbar_wait(bres, 0, abort_flag, a.status, 2u);
      int sa = 0, sb = 0, it = 0;
      uint32_t pa = 0, pb = 0;
      const uint32_t a_lbo = uint32_t(a.hp) * 16;
      for (int item = blockIdx.x; ok && item < a.total_items; item += gridDim.x, ++it) {
        int phase, mtile, ntile;
        decode_item(a, item, phase, mtile, ntile);
        const Phase& ph = a.ph[phase];
        const int buf = it & 1;
        if (!(ok = ptx::mbar_wait(tempty + buf, ((it >> 1) & 1) ^ 1, abort_flag, a.status, 2u))) break;
        ptx::tc_fence_after();
        const uint32_t acc = tmem + uint32_t(buf * NSUB * BN);
        if (ph.ntaps > 0) {
          for (int kb = 0; ok && kb < a.kb_count; ++kb) {
            if (!(ok = ptx::mbar_wait(fullA + sa, pa, abort_flag, a.status, 2u))) break;
            ptx::tc_fence_after();
            const uint32_t a_addr = ptx::smem_addr(a_base + size_t(sa) * a.a_stage_bytes);
            for (int t = 0; t < ph.ntaps; ++t) {
              uint32_t b_addr;
              if (BRES) {
                b_addr = ptx::smem_addr(b_base + size_t(ph.tap_w[t] * a.kb_count + kb) * a.b_tile_bytes);
              } else {
                if (!(ok = ptx::mbar_wait(fullB + sb, pb, abort_flag, a.status, 2u))) break;
                ptx::tc_fence_after();
                b_addr = ptx::smem_addr(b_base + size_t(sb) * a.b_tile_bytes);
              }
              for (int j = 0; j < a.kbc / 16; ++j) {
                const uint64_t bdesc = ptx::desc_kmajor_noswizzle(b_addr + 2 * j * lbo_b, lbo_b, BL::sbo);
#pragma unroll
                for (int s = 0; s < NSUB; ++s) {
                  const uint32_t arow = uint32_t(s * 128 + ph.tap_off[t]);
                  const uint64_t adesc =
                      ptx::desc_kmajor_noswizzle(a_addr + 2 * j * a_lbo + arow * 16, a_lbo, 128);
                  ptx::mma_bf16(acc + s * BN, adesc, bdesc, kIdesc, (kb | t | j) != 0);
                }
              }
              if (!BRES) {
                ptx::mma_commit(emptyB + sb);
                if (++sb == a.sb) { sb = 0; pb ^= 1; }
              }
            }
            ptx::mma_commit(emptyA + sa);
            if (++sa == a.sa) { sa = 0; pa ^= 1; }
          }
        }
        ptx::mma_commit(tfull + buf);
      }
      ptx::mma_commit(fin);
      ptx::mbar_wait(fin, 0, abort_flag, a.status, 2u);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    int it = 0;
    const uint32_t lane_base = uint32_t(warp * 32) << 16;
    for (int item = blockIdx.x; item < a.total_items; item += gridDim.x, ++it) {
      int phase, mtile, ntile;
      decode_item(a, item, phase, mtile, ntile);
      const Phase& ph = a.ph[phase];
      const int buf = it & 1;
      if (!ptx::mbar_wait(tfull + buf, (it >> 1) & 1, abort_flag, a.status, 4u)) break;
      ptx::tc_fence_after();
      const int n0 = ntile * BN;
      const int img = ph.RS * ph.P;
#pragma unroll 1
      for (int s = 0; s < NSUB; ++s) {
        const int q = mtile * 128 * NSUB + s * 128 + warp * 32 + lane;
        const int n = q / img, rem = q - n * img;
        const int r = rem / ph.P, col = rem - r * ph.P;
        const bool valid = n < a.N && r < ph.R && col < ph.OWv;
        bf16* dst = a.out + (size_t(n * a.Ho + r * ph.out_sh + ph.out_ph) * a.Wo + col * ph.out_sw + ph.out_pw) *
                                a.Cn + n0;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          if (ph.ntaps > 0) {
            ptx::tmem_ld_32(tmem + lane_base + uint32_t(buf * NSUB * BN + s * BN + c * 32), v);
            ptx::tmem_ld_wait();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0u;
          }
          if (valid) {
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              float lo = __uint_as_float(v[2 * j]), hi = __uint_as_float(v[2 * j + 1]);
              if (a.bias) {
                lo += __ldg(a.bias + n0 + c * 32 + 2 * j);
                hi += __ldg(a.bias + n0 + c * 32 + 2 * j + 1);
              }
              pk[j] = ptx::pack_bf16x2(lo, hi);
            }
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) d4[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(tempty + buf);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- host side

struct Plan {
  Args a;
  int bn, nsub;
  bool bres;
  size_t smem;
  int grid;
};

int pick_bn(int64_t cn) {
  for (int bn : {256, 128, 64, 32})
    if (cn % bn == 0) return bn;
  return 0;
}

int pick_kbc(int64_t ck) {
  for (int k : {64, 32, 16})
    if (ck % k == 0) return k;
  return 0;
}

int floordiv(int a, int b) { return (a >= 0) ? a / b : -((-a + b - 1) / b); }

// Fills the stage sizes and checks the shared-memory budget.
bool size_plan(Plan& pl, bool dgrad, int maxoff) {
  Args& a = pl.a;
  const int KC = a.kbc / 8;
  a.halo = 128 * pl.nsub + maxoff;
  a.hp = a.halo + ((1 - a.halo % 8) + 8) % 8;  // hp % 8 == 1 keeps the 8 chunk slabs on distinct banks
  a.a_stage_bytes = KC * a.hp * 16;
  const uint32_t sbo = dgrad ? 144 : 128;
  a.b_tile_bytes = KC * int((pl.bn / 8) * sbo + 16);
  const int bars = 8 * (2 * 8 + 2 * 8 + 4 + 2) + 16;
  for (int sa = 4; sa >= 2; --sa) {
    for (int sb = pl.bres ? 1 : 8; sb >= (pl.bres ? 1 : 2); --sb) {
      const size_t b_bytes = size_t(pl.bres ? a.T * a.kb_count : sb) * a.b_tile_bytes;
      const size_t total = size_t(sa) * a.a_stage_bytes + b_bytes + bars;
      if (total <= size_t(kSmemLimit)) {
        a.sa = sa;
        a.sb = pl.bres ? 1 : sb;
        pl.smem = total;
        return true;
      }
    }
  }
  return false;
}

// Forward at unit stride: one phase, taps at (kh*dh - ph, kw*dw - pw).
bool plan_fwd(const Problem& p, Plan& pl) {
  if (!(p.bf16 && p.nhwc && p.ohwi && p.G == 1 && p.SH == 1 && p.SW == 1)) return false;
  if (p.Cin % 16 != 0 || p.KH * p.KW > kMaxTapsPerPhase) return false;
  const int bn = pick_bn(p.Cout), kbc = pick_kbc(p.Cin);
  if (!bn || !kbc) return false;
  Args& a = pl.a;
  a = Args{};
  a.N = int(p.N); a.Hi = int(p.H); a.Wi = int(p.W); a.Ck = int(p.Cin);
  a.Cn = int(p.Cout); a.Ho = int(p.OH); a.Wo = int(p.OW);
  a.T = int(p.KH * p.KW); a.Cw = int(p.Cin);
  a.kbc = kbc; a.kb_count = int(p.Cin / kbc);
  a.n_tiles = int(p.Cout / bn);
  pl.bn = bn;
  pl.nsub = bn == 256 ? 1 : 2;
  Phase& ph = a.ph[0];
  ph = Phase{};
  const int rmin = -int(p.PH), rmax = int((p.KH - 1) * p.DH - p.PH);
  const int cmin = -int(p.PW), cmax = int((p.KW - 1) * p.DW - p.PW);
  ph.ntaps = a.T;
  ph.R = int(p.OH); ph.OWv = int(p.OW);
  ph.P = int(p.OW) + (cmax - cmin);
  ph.RS = int(p.OH) + (rmax - rmin);
  ph.rmin = rmin; ph.cmin = cmin;
  ph.out_sh = 1; ph.out_sw = 1; ph.out_ph = 0; ph.out_pw = 0;
  for (int kh = 0; kh < p.KH; ++kh)
    for (int kw = 0; kw < p.KW; ++kw) {
      const int t = int(kh * p.KW + kw);
      ph.tap_off[t] = (int(kh * p.DH) - int(p.PH) - rmin) * ph.P + (int(kw * p.DW) - int(p.PW) - cmin);
      ph.tap_w[t] = t;
    }
  const int maxoff = (rmax - rmin) * ph.P + (cmax - cmin);
  const int64_t positions = int64_t(p.N) * ph.RS * ph.P;
  if (positions + maxoff + 256 > 0x7FFFFFFF) return false;
  ph.tiles = int((positions + 128 * pl.nsub - 1) / (128 * pl.nsub));
  ph.item0 = 0;
  a.nphase = 1;
  a.total_items = ph.tiles * a.n_tiles;
  pl.bres = a.n_tiles == 1 && size_t(a.T) * a.kb_count * (size_t(a.kbc / 8) * (bn / 8 * 128 + 16)) <= 110 * 1024;
  if (!size_plan(pl, false, maxoff)) {
    pl.bres = false;
    if (!size_plan(pl, false, maxoff)) return false;
  }
  return true;
}

// Gradient: one phase per (ih % s_h, iw % s_w); each tap that reaches the
// phase does so at row shift (a + p_h - kh*d_h) / s_h of dy (exact division).
bool plan_dgrad(const Problem& p, Plan& pl) {
  if (!(p.bf16 && p.nhwc && p.ohwi && p.G == 1)) return false;
  if (p.SH * p.SW > kMaxPhases || p.Cout % 16 != 0) return false;
  const int bn = pick_bn(p.Cin), kbc = pick_kbc(p.Cout);
  if (!bn || !kbc) return false;
  Args& a = pl.a;
  a = Args{};
  a.N = int(p.N); a.Hi = int(p.OH); a.Wi = int(p.OW); a.Ck = int(p.Cout);
  a.Cn = int(p.Cin); a.Ho = int(p.H); a.Wo = int(p.W);
  a.T = int(p.KH * p.KW); a.Cw = int(p.Cin);
  a.kbc = kbc; a.kb_count = int(p.Cout / kbc);
  a.n_tiles = int(p.Cin / bn);
  pl.bn = bn;
  pl.nsub = bn == 256 ? 1 : 2;
  pl.bres = false;
  Phase phs[kMaxPhases];
  int nph = 0, maxoff = 0;
  for (int ah = 0; ah < p.SH; ++ah)
    for (int aw = 0; aw < p.SW; ++aw) {
      Phase ph{};
      const int R = int((p.H - ah + p.SH - 1) / p.SH), OWv = int((p.W - aw + p.SW - 1) / p.SW);
      if (R <= 0 || OWv <= 0) continue;
      int khs[64], drs[64], nkh = 0, kws[64], dcs[64], nkw = 0;
      for (int kh = 0; kh < p.KH; ++kh) {
        const int num = int(ah + p.PH - kh * p.DH);
        if (((num % p.SH) + p.SH) % p.SH == 0 && nkh < 64) { khs[nkh] = kh; drs[nkh] = floordiv(num, int(p.SH)); ++nkh; }
      }
      for (int kw = 0; kw < p.KW; ++kw) {
        const int num = int(aw + p.PW - kw * p.DW);
        if (((num % p.SW) + p.SW) % p.SW == 0 && nkw < 64) { kws[nkw] = kw; dcs[nkw] = floordiv(num, int(p.SW)); ++nkw; }
      }
      if (nkh * nkw > kMaxTapsPerPhase) return false;
      int rmin = 0, rmax = 0, cmin = 0, cmax = 0;
      for (int i = 0; i < nkh; ++i) { rmin = i ? std::min(rmin, drs[i]) : drs[i]; rmax = i ? std::max(rmax, drs[i]) : drs[i]; }
      for (int i = 0; i < nkw; ++i) { cmin = i ? std::min(cmin, dcs[i]) : dcs[i]; cmax = i ? std::max(cmax, dcs[i]) : dcs[i]; }
      ph.ntaps = nkh * nkw;
      ph.R = R; ph.OWv = OWv;
      ph.P = OWv + (cmax - cmin);
      ph.RS = R + (rmax - rmin);
      ph.rmin = rmin; ph.cmin = cmin;
      ph.out_sh = int(p.SH); ph.out_sw = int(p.SW); ph.out_ph = ah; ph.out_pw = aw;
      for (int i = 0; i < nkh; ++i)
        for (int j = 0; j < nkw; ++j) {
          const int t = i * nkw + j;
          ph.tap_off[t] = (drs[i] - rmin) * ph.P + (dcs[j] - cmin);
          ph.tap_w[t] = int(khs[i] * p.KW + kws[j]);
        }
      const int off = (rmax - rmin) * ph.P + (cmax - cmin);
      maxoff = std::max(maxoff, off);
      const int64_t positions = int64_t(p.N) * ph.RS * ph.P;
      if (positions + off + 256 > 0x7FFFFFFF) return false;
      ph.tiles = int((positions + 128 * pl.nsub - 1) / (128 * pl.nsub));
      phs[nph++] = ph;
    }
  // Longest phases first, so the persistent CTAs finish together.
  std::stable_sort(phs, phs + nph, [](const Phase& x, const Phase& y) { return x.ntaps > y.ntaps; });
  int item = 0;
  for (int i = 0; i < nph; ++i) {
    phs[i].item0 = item;
    item += phs[i].tiles * a.n_tiles;
    a.ph[i] = phs[i];
  }
  a.nphase = nph;
  a.total_items = item;
  return nph > 0 && size_plan(pl, true, maxoff);
}

template <int BN, int NSUB, bool DGRAD, bool BRES>
gbconv_status run(const Plan& pl, const Launch& l) {
  auto kern = implicit_gemm_kernel<BN, NSUB, DGRAD, BRES>;
  // The shared-memory opt-in is a per-device function attribute: set it once per device and size.
  static std::atomic<uint64_t> done[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GBCONV_ECUDA;
  if (done[dev].load(std::memory_order_acquire) < uint64_t(pl.smem)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(pl.smem)) != cudaSuccess)
      return GBCONV_ECUDA;
    done[dev].store(uint64_t(pl.smem), std::memory_order_release);
  }
  kern<<<pl.grid, kThreads, pl.smem, static_cast<cudaStream_t>(l.stream)>>>(pl.a);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? GBCONV_OK : GBCONV_ECUDA;
}

template <bool DGRAD>
gbconv_status dispatch(const Plan& pl, const Launch& l) {
  if (pl.bres) {
    if constexpr (!DGRAD) {
      switch (pl.bn) {
        case 256: return run<256, 1, false, true>(pl, l);
        case 128: return run<128, 2, false, true>(pl, l);
        case 64: return run<64, 2, false, true>(pl, l);
        default: return run<32, 2, false, true>(pl, l);
      }
    }
    return GBCONV_EUNSUPPORTED;
  }
  switch (pl.bn) {
    case 256: return run<256, 1, DGRAD, false>(pl, l);
    case 128: return run<128, 2, DGRAD, false>(pl, l);
    case 64: return run<64, 2, DGRAD, false>(pl, l);
    default: return run<32, 2, DGRAD, false>(pl, l);
  }
}

void finish_plan(Plan& pl, const void* in, const void* w, const float* bias, void* out, const Launch& l) {
  pl.a.in = static_cast<const bf16*>(in);
  pl.a.w = static_cast<const bf16*>(w);
  pl.a.bias = bias;
  pl.a.out = static_cast<bf16*>(out);
  pl.a.status = l.status;
  pl.grid = std::max(1, std::min(pl.a.total_items, l.num_sms));
}

}  // namespace

bool implicit_fwd_supported(const Problem& p) {
  Plan pl;
  return plan_fwd(p, pl);
}

bool implicit_dgrad_supported(const Problem& p) {
  Plan pl;
  return plan_dgrad(p, pl);
}

gbconv_status launch_implicit_fwd(const Problem& p, const void* x, const void* w, const float* bias, void* y,
                                  const Launch& l) {
  Plan pl;
  if (!plan_fwd(p, pl)) return GBCONV_EUNSUPPORTED;
  finish_plan(pl, x, w, bias, y, l);
  return dispatch<false>(pl, l);
}

gbconv_status launch_implicit_dgrad(const Problem& p, const void* dy, const void* w, void* dx, const Launch& l) {
  Plan pl;
  if (!plan_dgrad(p, pl)) return GBCONV_EUNSUPPORTED;
  finish_plan(pl, dy, w, nullptr, dx, l);
  return dispatch<true>(pl, l);
}

}  // namespace gbconv
