// Implicit-GEMM convolution on the 5th-generation tensor cores (tcgen05,
// accumulators in TMEM), NHWC bf16, fp32 accumulation.  One kernel template
// serves two regimes:
//
//  * dense forward at unit stride (the 3x3 workload): y = sum over taps of a
//    shifted window of x times the tap's [C_out, C_in] weight slice;
//  * the input gradient at strides up to 2x2, in gather form: dx is split into
//    stride phases (ih % s_h, iw % s_w); inside one phase every tap that reaches
//    it does so at a fixed integer shift of dy, so each phase is again a sum of
//    shifted windows, now of dy, times the tap's weight slice read transposed.
//    Each dx element is produced by exactly one accumulator and written once;
//    there are no atomics and the result is deterministic.
//
// A 3-D shape adds a depth axis to both: every kernel-depth tap is one more
// activation source (a 5-D box at a fixed depth offset from the item's
// output slice, zero filled outside), and work items run over (batch, depth)
// output slices.
//
// No im2col matrix is materialised (burn-cubecl `im2col.rs` notes that the
// column matrix holds every pixel once per tap that reads it, nine times for
// a 3x3).  Positions are laid out on a per-image "virtual grid": R rows of P
// columns, P being the valid output width plus the kernel's horizontal reach.
// A tile of 128*NSUB consecutive positions reads, for every tap t, the window
// that starts off(t) rows later in one halo block held in shared memory; the
// halo block is a single 4-D TMA box of whole virtual rows (zero fill supplies
// the padding), stored as 128-byte swizzled K-major rows, and because the
// swizzle follows absolute shared-memory addresses a tap is only a different
// descriptor start address.
//
// Weights are TMA boxes of the caller's OHWI tensor: K-major [C_out, C_in]
// slices for the forward, and for the gradient the same bytes read as an
// MN-major operand (C_in is the GEMM N dimension and is contiguous), so no
// transposed copy of the weight is ever made.
//
// Roles (warp specialised, one CTA per SM, persistent over work items):
//   warps 0-7  epilogue: TMEM -> registers, + bias, -> bf16, NHWC stores
//   warp  8    TMEM allocation; lane 0 issues every tcgen05.mma and commit
//   warp  9    lane 0 issues every TMA load
//
// Definitions followed: forward as teeny-kernels `conv2d_forward` (read
// position oh*stride + kh*dil - pad, zero outside) with bias added once after
// the reduction as in `conv2d_bias_forward`; gradient as the exact transpose
// of teeny-kernels `conv2d_backward_dx` (scatter), evaluated per input
// element as oarust `conv_2d_backward` dispatches it.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
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

using bf16 = __nv_bfloat16;

constexpr int kMaxPhases = 8;  // stride phases of a gradient: (depth,) row and column phase
constexpr int kMaxTapsPerPhase = 32;
constexpr int kEpiWarps = 8;
constexpr int kMmaWarp = 8;
constexpr int kTmaWarp = 9;
constexpr int kThreads = 10 * 32;
constexpr int kSmemLimit = 227 * 1024;
constexpr int kKB = 64;  // channels per k-block: one 128-byte swizzled row
constexpr int kMaxSrc = 9;  // activation sources of one phase: stride phases of a strided forward
// Transposed-form staging: per epilogue half, two blocks of 32 positions x 128 channels, rows
// padded to 320 bytes (80 words: rows r and r+1 fall 16 banks apart).
constexpr int kTposPitch = 320;
constexpr int kTposStage = 2 * 2 * 32 * kTposPitch;

struct PhaseHdr {
  int ntaps;
  int R;        // output rows of the virtual grid (per image)
  int P;        // virtual grid pitch: valid columns plus the horizontal reach
  int OWv;      // valid columns
  int rmin, cmin;                      // input coordinate of virtual (0, 0)
  int out_sh, out_sw, out_ph, out_pw;  // output pixel = (r*out_sh + out_ph, c*out_sw + out_pw)
  int bh;       // rows in one halo box
  int a_bytes;  // bytes of one halo box (64 channels x P x bh)
  int tiles;    // m-tiles per image
  int item0;    // first work item of this phase
  // Activation sources.  A strided forward reads its input as s_h x s_w stride phases: through a
  // strided view (TMA element strides = the conv strides) each phase is a dense grid, and every
  // tap reads one of them at a fixed shift.  Source k starts at input offset (src_ah, src_aw)
  // and owns taps [src_t0[k], src_t0[k+1]).  Unit stride: one source at (0, 0) with every tap.
  int row_step, col_step;  // input rows / columns per virtual-grid step (the strides; else 1)
  int nsrc;
  int8_t src_ah[kMaxSrc], src_aw[kMaxSrc];  // < 8 (TMA element strides are at most 8)
  int8_t src_t0[kMaxSrc + 1];                // <= kMaxTapsPerPhase
  // 3-D: source k also reads activation depth j*depth_sd + src_ad[k], j the item's depth slice of
  // this phase: kd*DD - PD for the forward, (ad + PD - kd*DD) / SD for the gradient (dx slice
  // id = ad + j*SD meets dy slice (id + PD - kd*DD) / SD when that divides exactly)
  int src_ad[kMaxSrc];
  int jd;      // 3-D: depth slices of this phase per batch element
  int out_pd;  // 3-D: output depth of the phase's slice j = 0 (the depth phase ad)
  // Column strips: an image wider than one halo box allows is cut into nstrips vertical strips of
  // strip_w valid columns (the last one may be narrower), each with its own virtual grid of pitch
  // P = strip_w + the horizontal reach.  Work items run over (image, strip) pairs.
  int strip_w, nstrips;
};

struct Phase : PhaseHdr {
  int tap_off[kMaxTapsPerPhase];  // halo row offset of tap t
  int tap_w[kMaxTapsPerPhase];    // weight tap index kh*KW + kw
};

struct Args {
  const float* bias;  // [Cn] or null
  bf16* out;          // NHWC [N, Ho, Wo, Cn]: y or dx
  unsigned int* status;
  int N, Cn, Ho, Wo;
  int T;              // KH*KW
  int kb_count;       // 64-channel k-blocks of the reduction (of one group)
  int n_tiles;        // BN-wide output tiles of one group
  // Groups: every group is its own GEMM.  G groups of cg_k reduction channels and cg_n output
  // channels; the activations are read through a view with the group as a dimension of its own, so
  // each group's k-blocks end at the group's last channel (TMA zero fill past it).
  int G, cg_k, cg_n;
  int bias_n;         // bias entries staged in shared memory
  uint64_t wait_ns;   // bound of every barrier wait (the host sets it; 2 s by default)
  int a_stage_bytes, b_tile_bytes, sa, sb;
  int stage_bufs;     // epilogue staging blocks (2: copies of one overlap the next sub-tile)
  int b4d;            // gradient weight tiles come as one 4-D box (C_in a multiple of 64), else 64-wide boxes
  int nphase, total_items;
  int depth_od, depth_sd;  // 3-D: nonzero, and the activation depth step per slice; else 0
  int out_d, out_sd;       // 3-D: output depth, and output depth step between a phase's slices
  Phase ph[kMaxPhases];
};

struct Maps {
  CUtensorMap a[kMaxPhases];  // gathered activations, one box shape per phase
  CUtensorMap b;              // weight viewed as [C_out][KH*KW][C_in]
};

struct Item {
  int phase, n, m, ntile, g;
};

// Item of round r for this CTA.  Items are numbered heaviest phase first; even rounds hand them
// out in CTA order and odd rounds in reverse, so the CTAs that took the heaviest items in one
// round take the lightest in the next (-1 once the items run out).
__device__ __forceinline__ int round_item(int r, int total) {
  const int g = int(gridDim.x), c = int(blockIdx.x);
  const int item = r * g + ((r & 1) ? g - 1 - c : c);
  return item < total ? item : -1;
}

__device__ __forceinline__ Item decode_item(const PhaseHdr* ph, int nphase, int n_tiles, int G, int item) {
  int p = 0;
  while (p + 1 < nphase && item >= ph[p + 1].item0) ++p;
  Item it;
  it.phase = p;
  int local = item - ph[p].item0;
  const int t2 = local % (n_tiles * G);  // (group, output tile) of the item
  it.g = t2 / n_tiles;
  it.ntile = t2 - it.g * n_tiles;
  local /= n_tiles * G;
  it.n = local / ph[p].tiles;
  it.m = local - it.n * ph[p].tiles;
  return it;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];" ::"r"(dst),
      "l"(map), "r"(ptx::smem_addr(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z,
                                            int v, int w) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, "
      "%6, %7}], [%2];" ::"r"(dst),
      "l"(map), "r"(ptx::smem_addr(bar)), "r"(x), "r"(y), "r"(z), "r"(v), "r"(w)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z,
                                            int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, "
      "%6}], [%2];" ::"r"(dst),
      "l"(map), "r"(ptx::smem_addr(bar)), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}

// K-major operand, 128-byte swizzle, 8-row atoms of 1024 bytes.
__device__ __forceinline__ uint64_t desc_sw128_kmajor(uint32_t saddr) { return ptx::desc_kmajor_sw128(saddr); }

// MN-major operand, 128-byte swizzle: `mn_stride` bytes between 64-element
// atoms along N, 1024 bytes between 8-row atoms along K.
__device__ __forceinline__ uint64_t desc_sw128_mnmajor(uint32_t saddr, uint32_t mn_stride) {
  uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((mn_stride >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// MSRC: phases may have several activation sources (a strided forward); otherwise every phase
// has exactly one and the source loops fold away at compile time.
//
// TPOS (BN = 128, NSUB = 2): the product is formed transposed, D^T = W * X^T, with the tile's 128
// output channels on the MMA's M side and its 256 positions on N.  One 128x256x16 MMA then does the
// work of the two 128x128x16 ones and reads 12 KB of operands from shared memory instead of 16 KB
// (the weight slice once, not once per sub-tile): shared-memory bandwidth, not the tensor pipe, is
// what limits the 128x128 form once the TMA writes are added.  The accumulator then holds one
// channel per TMEM lane, so the epilogue writes channel pairs straight from registers.
template <int BN, int NSUB, bool DGRAD, bool BRES, bool MSRC, bool TPOS = false>
__global__ void __launch_bounds__(kThreads, 1)
    implicit_gemm_kernel(const __grid_constant__ Maps maps, const __grid_constant__ Args a) {
  static_assert(!TPOS || (BN == 128 && NSUB == 2), "the transposed form is a 128-channel x 256-position tile");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // Swizzled TMA destinations and operands sit on 1024-byte boundaries.
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr uint32_t kCols = 2 * NSUB * BN;
  constexpr uint32_t kTmemCols = kCols <= 32 ? 32 : kCols <= 64 ? 64 : kCols <= 128 ? 128 : kCols <= 256 ? 256 : 512;
  // The weight operand is MN-major in the gradient (C_in, the GEMM's output dimension, is
  // contiguous): the transpose bit of B, or of A in the transposed form.
  constexpr uint32_t kIdesc = TPOS ? ptx::idesc_bf16_f32(128, 128 * NSUB) | (DGRAD ? (1u << 15) : 0u)
                                   : ptx::idesc_bf16_f32(128, BN) | (DGRAD ? (1u << 16) : 0u);
  constexpr int kBTile = BN * kKB * 2;

  uint8_t* a_base = smem;
  uint8_t* b_base = a_base + size_t(a.sa) * a.a_stage_bytes;
  const int b_tiles = BRES ? a.T * a.kb_count : a.sb;  // resident: every (k-block, tap) tile
  // two staging blocks of 128 rows x (staging group * 2 + 16) bytes
  uint8_t* stage_base = b_base + size_t(b_tiles) * kBTile;
  constexpr int kStageBlock = 128 * ((BN % 128 == 0 ? 128 : 64) * 2 + 16);
  float* bias_s = reinterpret_cast<float*>(stage_base + (TPOS ? kTposStage : a.stage_bufs * kStageBlock));
  // Per-phase tap tables, copied from the kernel parameters: runtime-indexed
  // parameter reads are slow next to shared-memory reads in the MMA loop.
  int* taps_s = reinterpret_cast<int*>(bias_s + a.bias_n);  // [phase][off, w][kMaxTapsPerPhase]
  PhaseHdr* phase_s = reinterpret_cast<PhaseHdr*>(taps_s + kMaxPhases * 2 * kMaxTapsPerPhase);
  uint64_t* bars = reinterpret_cast<uint64_t*>(phase_s + kMaxPhases);
  uint64_t* fullA = bars;
  uint64_t* emptyA = fullA + a.sa;
  uint64_t* fullB = emptyA + a.sa;
  uint64_t* emptyB = fullB + a.sb;
  // One k-block, resident weights and one source: an item's halo stage and every weight tile stay in
  // shared memory for all of its MMAs, so its sub-tiles can be issued one after the other, each
  // committed to its own barrier, and the epilogue starts on sub-tile 0 while sub-tile 1's MMAs run
  // (for a CTA's last item nothing else overlaps its epilogue).
  constexpr bool kSubMajor = !TPOS && !DGRAD && BRES && !MSRC && NSUB > 1;
  // Accumulator-full barriers: one per TMEM buffer, or one per buffer and sub-tile where the
  // sub-tiles may be issued one after the other.
  constexpr int kTf = kSubMajor ? NSUB : 1;
  uint64_t* tfull = emptyB + a.sb;
  uint64_t* tempty = tfull + 2 * kTf;
  uint64_t* bres = tempty + 2;
  uint64_t* fin = bres + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fin + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < a.sa; ++i) { ptx::mbar_init(fullA + i, 1); ptx::mbar_init(emptyA + i, 1); }
    for (int i = 0; i < a.sb; ++i) { ptx::mbar_init(fullB + i, 1); ptx::mbar_init(emptyB + i, 1); }
    for (int i = 0; i < 2 * kTf; ++i) ptx::mbar_init(tfull + i, 1);
    for (int i = 0; i < 2; ++i) ptx::mbar_init(tempty + i, kEpiWarps * 32);
    ptx::mbar_init(bres, 1);
    ptx::mbar_init(fin, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp < kEpiWarps) {
    if (threadIdx.x < a.nphase) phase_s[threadIdx.x] = a.ph[threadIdx.x];
    for (int i = threadIdx.x; i < a.nphase * kMaxTapsPerPhase; i += kEpiWarps * 32) {
      const int p = i / kMaxTapsPerPhase, t = i % kMaxTapsPerPhase;
      taps_s[(p * 2 + 0) * kMaxTapsPerPhase + t] = a.ph[p].tap_off[t];
      taps_s[(p * 2 + 1) * kMaxTapsPerPhase + t] = a.ph[p].tap_w[t];
    }
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(tmem_slot, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Global memory is touched only after the previous kernel on the stream has finished; the next
  // kernel may start its prologue now (this CTA already holds its TMEM).
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      for (int p = 0; p < a.nphase; ++p) ptx::prefetch_tmap(&maps.a[p]);
      ptx::prefetch_tmap(&maps.b);
      // n0: first output channel of the tile inside group g (the weight's C_out rows of group g
      // start at g*cg_n in the forward; the gradient's reduction runs over them, from g*cg_k)
      auto load_b = [&](uint8_t* dst, uint64_t* bar, int wt, int kb, int n0, int g) {
        const uint32_t d = ptx::smem_addr(dst);
        if (DGRAD) {  // MN-major: BN/64 atoms of [64 output channels][64 input channels]
          const int co = g * a.cg_k + kb * kKB;
          if (a.b4d) {
            tma_load_4d(d, &maps.b, bar, 0, co, n0 / 64, wt);
          } else {
#pragma unroll
            for (int h = 0; h < BN / 64; ++h) tma_load_3d(d + h * 8192, &maps.b, bar, n0 + h * 64, wt, co);
          }
        } else {      // K-major: BN output channels x 64 input channels
          tma_load_3d(d, &maps.b, bar, kb * kKB, wt, g * a.cg_n + n0);
        }
      };
      bool ok = true;
      // Resident weights, tile (kb, tap) at index kb * T + tap.  Issued right after the first
      // activation halo: that box comes from HBM and takes longest, the weights are shared by every
      // CTA and mostly come from L2.
      bool b_pending = BRES;
      int issued_a = 0, issued_b = 0;  // loads issued into the A and B rings (for the drain below)
      auto load_resident_b = [&]() {
        ptx::mbar_arrive_expect_tx(bres, uint32_t(a.T * a.kb_count) * kBTile);
        for (int kb = 0; kb < a.kb_count; ++kb)
          for (int wt = 0; wt < a.T; ++wt) load_b(b_base + size_t(kb * a.T + wt) * kBTile, bres, wt, kb, 0, 0);
        b_pending = false;
      };
      int sa = 0, sb = 0;
      uint32_t pa = 0, pb = 0;
      for (int r = 0, item = round_item(0, a.total_items); ok && item >= 0; item = round_item(++r, a.total_items)) {
        const Item it = decode_item(phase_s, a.nphase, a.n_tiles, a.G, item);
        const PhaseHdr& ph = phase_s[it.phase];
        if (ph.ntaps == 0) continue;
        const int ra = (it.m * 128 * NSUB) / ph.P;
        const int kb_rot = item % a.kb_count;
        const int* tw = taps_s + (it.phase * 2 + 1) * kMaxTapsPerPhase;
        for (int kbi = 0; ok && kbi < a.kb_count; ++kbi) {
          const int kb = kbi + kb_rot < a.kb_count ? kbi + kb_rot : kbi + kb_rot - a.kb_count;
          for (int src = 0; ok && src < (MSRC ? ph.nsrc : 1); ++src) {
            if (!(ok = ptx::mbar_wait(emptyA + sa, pa ^ 1, abort_flag, a.status, 1u, a.wait_ns))) break;
            ptx::mbar_arrive_expect_tx(fullA + sa, uint32_t(ph.a_bytes));
            // the item's (image, column strip): the strip's virtual column 0 is phase-grid column
            // strip * strip_w
            const int img = it.n / ph.nstrips, col = (ph.cmin + (it.n - img * ph.nstrips) * ph.strip_w) * ph.col_step;
            if (MSRC && a.depth_od > 0) {  // 3-D: image img is a (batch, depth slice) pair
              const int nn = img / ph.jd, od = img - nn * ph.jd;
              tma_load_5d(ptx::smem_addr(a_base + size_t(sa) * a.a_stage_bytes), &maps.a[it.phase], fullA + sa,
                          kb * kKB, col + ph.src_aw[src], (ra + ph.rmin) * ph.row_step + ph.src_ah[src],
                          od * a.depth_sd + ph.src_ad[src], nn);
            } else if (a.G > 1) {  // (channel in group, group, column, row, image)
              tma_load_5d(ptx::smem_addr(a_base + size_t(sa) * a.a_stage_bytes), &maps.a[it.phase], fullA + sa,
                          kb * kKB, it.g, col + ph.src_aw[src], (ra + ph.rmin) * ph.row_step + ph.src_ah[src], img);
            } else {
              tma_load_4d(ptx::smem_addr(a_base + size_t(sa) * a.a_stage_bytes), &maps.a[it.phase], fullA + sa,
                          kb * kKB, col + ph.src_aw[src], (ra + ph.rmin) * ph.row_step + ph.src_ah[src], img);
            }
            ++issued_a;
            if (++sa == a.sa) { sa = 0; pa ^= 1; }
            if (BRES && b_pending) load_resident_b();
            if (!BRES) {
              const int t0 = ph.src_t0[src], nt = ph.src_t0[src + 1] - t0;
              for (int ti = 0, t = item % nt; ok && ti < nt; ++ti, t = (t + 1 == nt ? 0 : t + 1)) {
                if (!(ok = ptx::mbar_wait(emptyB + sb, pb ^ 1, abort_flag, a.status, 1u, a.wait_ns))) break;
                ptx::mbar_arrive_expect_tx(fullB + sb, uint32_t(kBTile));
                load_b(b_base + size_t(sb) * kBTile, fullB + sb, tw[t0 + t], kb, it.ntile * BN, it.g);
                ++issued_b;
                if (++sb == a.sb) { sb = 0; pb ^= 1; }
              }
            }
          }
        }
      }
      if (BRES && b_pending && ok) load_resident_b();  // a CTA that loaded no halo still owes them
      // Drain: after an abort the MMA thread no longer consumes the stages, but copies still in
      // flight write this CTA's shared memory, so they must land before the CTA leaves.  The k-th
      // load into a ring completes phase k / stages of barrier k % stages.
      for (int k = max(0, issued_a - a.sa); k < issued_a; ++k)
        ptx::mbar_wait_drain(fullA + k % a.sa, uint32_t((k / a.sa) & 1));
      for (int k = max(0, issued_b - a.sb); k < issued_b; ++k)
        ptx::mbar_wait_drain(fullB + k % a.sb, uint32_t((k / a.sb) & 1));
      if (BRES && !b_pending) ptx::mbar_wait_drain(bres, 0);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // Kernel parameters the loop uses, in registers: parameters live in memory, and every MMA's
      // asm statement clobbers memory, so a field read inside the loop is reloaded after each MMA.
      unsigned int* const status = a.status;
      const uint64_t wait_ns = a.wait_ns;
      const int n_sa = a.sa, n_sb = a.sb, a_stage = a.a_stage_bytes, T = a.T;
      bool ok = true;
      if (BRES) ok = ptx::mbar_wait(bres, 0, abort_flag, status, 2u, wait_ns);
      int sa = 0, sb = 0, iter = 0;
      uint32_t pa = 0, pb = 0;
      for (int r = 0, item = round_item(0, a.total_items); ok && item >= 0;
           item = round_item(++r, a.total_items), ++iter) {
        const Item it = decode_item(phase_s, a.nphase, a.n_tiles, a.G, item);
        const PhaseHdr& ph = phase_s[it.phase];
        const int buf = iter & 1;
        if (!(ok = ptx::mbar_wait(tempty + buf, ((iter >> 1) & 1) ^ 1, abort_flag, status, 2u, wait_ns))) break;
        ptx::tc_fence_after();
        const uint32_t acc = tmem + uint32_t(buf * NSUB * BN);
        bool sub_committed = false;  // the sub-tile-major path commits each sub-tile itself
        if (ph.ntaps > 0) {
          const int q0 = it.m * 128 * NSUB;
          const int row0 = q0 - (q0 / ph.P) * ph.P;  // tile start inside the halo block
          const int kbn = a.kb_count;
          const int* toff = taps_s + (it.phase * 2 + 0) * kMaxTapsPerPhase;
          const int* tw = taps_s + (it.phase * 2 + 1) * kMaxTapsPerPhase;
          // k-blocks and taps are walked in an order rotated by the item index (the producer
          // walks the same order): CTAs working at the same time then read different weight
          // tiles, which spreads the L2 traffic of the streamed weights.
          const int kb_rot = item % kbn;
          // Source 0's tap range and rotation, worked out once per item: scalar work between MMA
          // bursts delays the issue (one source is the common case: unit stride, every dgrad).
          const int nsrc = MSRC ? ph.nsrc : 1, nt0 = ph.src_t0[1], tc0 = item % nt0;
          if (kSubMajor && kbn == 1) {
            if ((ok = ptx::mbar_wait(fullA + sa, pa, abort_flag, status, 2u, wait_ns))) {
              const uint32_t a_addr = ptx::smem_addr(a_base + size_t(sa) * a_stage);
#pragma unroll 1
              for (int s = 0; s < NSUB; ++s) {
                int tc = tc0, off_c = toff[tc], w_c = tw[tc];
                for (int ti = 0; ti < nt0; ++ti) {
                  const int tn = tc + 1 == nt0 ? 0 : tc + 1;
                  const int off_n = toff[tn], w_n = tw[tn];
                  const uint64_t ad0 = desc_sw128_kmajor(a_addr + uint32_t(row0 + off_c) * 128);
                  const uint64_t bd0 = desc_sw128_kmajor(ptx::smem_addr(b_base + size_t(w_c) * kBTile));
                  const uint32_t a_lo = uint32_t(ad0) + uint32_t((s * 128 * 128) >> 4), a_hi = uint32_t(ad0 >> 32);
                  const uint32_t b_lo = uint32_t(bd0), b_hi = uint32_t(bd0 >> 32);
#pragma unroll
                  for (int j = 0; j < kKB / 16; ++j)
                    ptx::mma_bf16_lohi(acc + s * BN, a_lo + uint32_t((j * 32) >> 4), a_hi, b_lo + uint32_t((j * 32) >> 4),
                                       b_hi, kIdesc, (ti | j) == 0 ? 0u : 1u);
                  tc = tn;
                  off_c = off_n;
                  w_c = w_n;
                }
                ptx::mma_commit(tfull + buf * kTf + s);
              }
              ptx::mma_commit(emptyA + sa);
              if (++sa == n_sa) { sa = 0; pa ^= 1; }
              sub_committed = true;
            }
          } else
          for (int kbi = 0; ok && kbi < kbn; ++kbi) {
            const int kb = kbi + kb_rot < kbn ? kbi + kb_rot : kbi + kb_rot - kbn;  // the producer's order
            for (int src = 0; ok && src < nsrc; ++src) {
              // TMA-filled stages need no tcgen05 fence: the barrier's transaction count already
              // orders the async-proxy writes before the async-proxy MMA reads.
              if (!(ok = ptx::mbar_wait(fullA + sa, pa, abort_flag, status, 2u, wait_ns))) break;
              const uint32_t a_addr = ptx::smem_addr(a_base + size_t(sa) * a_stage);
              // this source's taps, in the producer's rotated order
              const int t0 = src == 0 ? 0 : ph.src_t0[src];
              const int nt = src == 0 ? nt0 : ph.src_t0[src + 1] - t0;
              int tc = src == 0 ? tc0 : item % nt;
              int off_c = toff[t0 + tc], w_c = tw[t0 + tc];
              for (int ti = 0; ti < nt; ++ti) {
                // fetch the next tap's table entries before this tap's MMAs are issued
                const int tn = tc + 1 == nt ? 0 : tc + 1;
                const int off_n = toff[t0 + tn], w_n = tw[t0 + tn];
                uint32_t b_addr;
                if (BRES) {
                  b_addr = ptx::smem_addr(b_base + size_t(kb * T + w_c) * kBTile);
                } else {
                  if (!(ok = ptx::mbar_wait(fullB + sb, pb, abort_flag, status, 2u, wait_ns))) break;
                  b_addr = ptx::smem_addr(b_base + size_t(sb) * kBTile);
                }
                // Descriptor halves: the low word is (address >> 4) plus the leading-offset field, so
                // per-MMA operand offsets (K step j, sub-tile s) are compile-time adds on it.
                const uint64_t ad0 = desc_sw128_kmajor(a_addr + uint32_t(row0 + off_c) * 128);
                const uint64_t bd0 = DGRAD ? desc_sw128_mnmajor(b_addr, 8192) : desc_sw128_kmajor(b_addr);
                const uint32_t a_lo = uint32_t(ad0), a_hi = uint32_t(ad0 >> 32);
                const uint32_t b_lo = uint32_t(bd0), b_hi = uint32_t(bd0 >> 32);
                const uint32_t first = uint32_t(kbi | src | ti);  // 0 only for the item's first MMA
#pragma unroll
                for (int j = 0; j < kKB / 16; ++j) {
                  const uint32_t b_off = DGRAD ? uint32_t(j * 2048 >> 4) : uint32_t(j * 32 >> 4);
                  if (TPOS) {  // weights as A (128 channels), the 256 halo rows as B
                    ptx::mma_bf16_lohi(acc, b_lo + b_off, b_hi, a_lo + uint32_t((j * 32) >> 4), a_hi, kIdesc,
                                       j == 0 ? first : 1u);
                  } else {
#pragma unroll
                    for (int s = 0; s < NSUB; ++s)
                      ptx::mma_bf16_lohi(acc + s * BN, a_lo + uint32_t((s * 128 * 128 + j * 32) >> 4), a_hi,
                                         b_lo + b_off, b_hi, kIdesc, j == 0 ? first : 1u);
                  }
                }
                if (!BRES) {
                  ptx::mma_commit(emptyB + sb);
                  if (++sb == n_sb) { sb = 0; pb ^= 1; }
                }
                tc = tn;
                off_c = off_n;
                w_c = w_n;
              }
              ptx::mma_commit(emptyA + sa);
              if (++sa == n_sa) { sa = 0; pa ^= 1; }
            }
          }
        }
        if (!sub_committed)
          for (int s = 0; s < kTf; ++s) ptx::mma_commit(tfull + buf * kTf + s);
      }
      ptx::mma_commit(fin);
      // Even after an abort, every MMA issued so far must complete before TMEM is freed and the CTA
      // leaves: this wait ignores the abort flag.
      ptx::mbar_wait_drain(fin, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // Warps w and w+4 share TMEM lanes 32*(w%4).. (32 positions) and split the
    // columns of each 128-column group.  Each converts its accumulators to
    // bf16 into a padded shared-memory staging block; then the pair stores the
    // 32 rows so that consecutive threads write consecutive 16-byte pieces of
    // the same output pixel (whole pixels per warp instruction).
    constexpr int kG = BN % 128 == 0 ? 128 : 64;  // columns per staging group
    constexpr int kPitch = kG * 2 + 16;         // padded row pitch of the staging block, bytes
    const int quad = warp & 3, half = warp >> 2;
    const uint32_t lane_base = uint32_t(quad * 32) << 16;
    // The bias comes from global memory: copied here, after the block-wide barrier, so the
    // producer and MMA warps start without waiting for it.
    for (int i = threadIdx.x; i < a.bias_n; i += kEpiWarps * 32) bias_s[i] = (a.bias && i < a.Cn) ? a.bias[i] : 0.f;
    asm volatile("bar.sync 5, %0;" ::"n"(kEpiWarps * 32) : "memory");
    const uint32_t stage0 = ptx::smem_addr(stage_base + quad * 32 * kPitch);
    int sbuf = 0;  // staging block used next
    int iter = 0;
    for (int r = 0, item = round_item(0, a.total_items); item >= 0; item = round_item(++r, a.total_items), ++iter) {
      const Item it = decode_item(phase_s, a.nphase, a.n_tiles, a.G, item);
      const PhaseHdr& ph = phase_s[it.phase];
      const int buf = iter & 1;
      const bool got = ptx::mbar_wait(tfull + buf * kTf, (iter >> 1) & 1, abort_flag, a.status, 4u, a.wait_ns);
      // Every thread times its own wait, so after an expired wait the 64 threads of a warp pair could
      // disagree, and a thread that carried on would block at the pair barrier below for good: the
      // pair takes one decision (leave if any of its threads gave up).
      // (In the transposed form the four warps of a half work together: the half decides.)
      uint32_t stop;
      asm volatile(
          "{\n\t.reg .pred p, q;\n\tsetp.eq.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\t"
          "selp.u32 %0, 1, 0, q;\n\t}"
          : "=r"(stop)
          : "r"(uint32_t(got)), "r"(TPOS ? 6 + half : 1 + quad), "r"(TPOS ? 128 : 64)
          : "memory");
      if (stop) break;
      ptx::tc_fence_after();
      const int n0 = it.g * a.cg_n + it.ntile * BN;  // first output channel of the tile
      const int n_end = (it.g + 1) * a.cg_n;         // the group's last output channel + 1
      const bool has_bias = a.bias != nullptr;
      // The phase geometry in registers: read from shared memory inside the store loop, every
      // field would be re-read after each staging load (those are asm with memory clobbers).
      const int ph_R = ph.R, ph_P = ph.P, ph_ntaps = ph.ntaps;
      // the item's (image, column strip); the strip's valid columns
      const int nimg = it.n / ph.nstrips, col0 = (it.n - nimg * ph.nstrips) * ph.strip_w;
      const int ph_OWv = min(ph.strip_w, ph.OWv - col0);
      // 3-D: the item's image is batch element nimg / jd at output depth out_pd + (nimg % jd) * out_sd
      const int img = a.depth_od > 0 ? (nimg / ph.jd) * a.out_d + ph.out_pd + (nimg % ph.jd) * a.out_sd : nimg;
      const int row_base = img * a.Ho + ph.out_ph, ph_sh = ph.out_sh, ph_sw = ph.out_sw, ph_pw = ph.out_pw;
      const int Wo = a.Wo, Cn = a.Cn;
      bf16* const out = a.out;
      if constexpr (TPOS) {
        // TMEM lane = output channel, column = tile position; warps w and w+4 take 128 positions
        // each, in chunks of 32.  Lanes 2i and 2i+1 (channels c, c+1) swap one value per pair of
        // positions, so that each lane holds both channels of one position as a 4-byte word; the
        // four warps of a half write their words into a staged [32 positions][128 channels] block
        // (each warp instruction fills two rows, 16 banks each), then store it as whole pixels:
        // consecutive threads write consecutive 16-byte pieces, 256 bytes per pixel.
        const int odd = lane & 1;
        const float bv = has_bias ? bias_s[n0 + quad * 32 + lane] : 0.f;
        const uint32_t stage_h = ptx::smem_addr(stage_base) + uint32_t(half * 2 * 32 * kTposPitch);
        const uint32_t word_off = uint32_t(odd * kTposPitch + (quad * 16 + (lane >> 1)) * 4);
        const int tp = quad * 32 + lane, part = tp & 15, row0 = tp >> 4;  // store role: piece, first row
        const int co = n0 + part * 8;
        const bool live = co < n_end;
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          const int col = half * 128 + ch * 32;
          const uint32_t blk = stage_h + uint32_t(sbuf * 32 * kTposPitch);
          sbuf ^= 1;
          uint32_t v[32];
          if (ph_ntaps > 0) {
            ptx::tmem_ld_32(tmem + lane_base + uint32_t(buf * 256 + col), v);
            ptx::tmem_ld_wait();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0u;
          }
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float f0 = __uint_as_float(v[2 * k]) + bv, f1 = __uint_as_float(v[2 * k + 1]) + bv;
            const float other = __shfl_xor_sync(0xffffffffu, odd ? f0 : f1, 1);
            const uint32_t wd = odd ? ptx::pack_bf16x2(other, f1) : ptx::pack_bf16x2(f0, other);
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(blk + uint32_t(2 * k * kTposPitch) + word_off), "r"(wd)
                         : "memory");
          }
          // With two blocks per half this barrier also proves that the half finished reading the
          // block it is about to overwrite (two chunks ago).
          asm volatile("bar.sync %0, 128;" ::"r"(6 + half) : "memory");
          if (live) {
            uint4 val[4];
            int pix[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int row = row0 + 8 * i;
              asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(val[i].x), "=r"(val[i].y), "=r"(val[i].z), "=r"(val[i].w)
                           : "r"(blk + uint32_t(row * kTposPitch + part * 16)));
              const int q = it.m * 256 + col + row;
              const int r = q / ph_P, colv = q - r * ph_P;
              pix[i] = (r < ph_R && colv < ph_OWv) ? (row_base + r * ph_sh) * Wo + (col0 + colv) * ph_sw + ph_pw : -1;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (pix[i] >= 0) *reinterpret_cast<uint4*>(out + size_t(pix[i]) * Cn + co) = val[i];
          }
        }
      } else {
      bool stopped = false;
#pragma unroll 1
      for (int s = 0; s < NSUB; ++s) {
        if (kTf > 1 && s > 0) {
          // Sub-tile s's accumulators have their own barrier (the MMAs may run sub-tile by sub-tile);
          // the warp pair again takes one decision.
          const bool got_s = ptx::mbar_wait(tfull + buf * kTf + s, (iter >> 1) & 1, abort_flag, a.status, 4u, a.wait_ns);
          uint32_t stop_s;
          asm volatile(
              "{\n\t.reg .pred p, q;\n\tsetp.eq.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, 64, p;\n\t"
              "selp.u32 %0, 1, 0, q;\n\t}"
              : "=r"(stop_s)
              : "r"(uint32_t(got_s)), "r"(1 + quad)
              : "memory");
          if (stop_s) { stopped = true; break; }
          ptx::tc_fence_after();
        }
        const int qbase = it.m * 128 * NSUB + s * 128 + quad * 32;
#pragma unroll 1
        for (int g = 0; g < BN / kG; ++g) {
          // With two staging blocks the barrier after the writes also proves that both warps
          // finished reading the block they are about to overwrite (two sub-tiles ago).
          const uint32_t stage_s = stage0 + uint32_t(sbuf * kStageBlock);
          if (a.stage_bufs == 2) sbuf ^= 1;
          // 1. this warp's half of the group: TMEM -> (+ bias) -> bf16 -> staging row `lane`
          constexpr int kChunks = kG / 64;  // 32-column TMEM loads per warp per group
          uint32_t v[kChunks][32];
          const int c0 = g * kG + half * (kG / 2);
          if (ph_ntaps > 0) {
#pragma unroll
            for (int ch = 0; ch < kChunks; ++ch)
              ptx::tmem_ld_32(tmem + lane_base + uint32_t(buf * NSUB * BN + s * BN + c0 + ch * 32), v[ch]);
            ptx::tmem_ld_wait();
          } else {
#pragma unroll
            for (int ch = 0; ch < kChunks; ++ch)
#pragma unroll
              for (int j = 0; j < 32; ++j) v[ch][j] = 0u;
          }
#pragma unroll
          for (int ch = 0; ch < kChunks; ++ch) {
            float f[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[ch][j]);
            if (has_bias) {
              const float4* b4 = reinterpret_cast<const float4*>(bias_s + n0 + c0 + ch * 32);
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const float4 bb = b4[q];
                f[4 * q] += bb.x; f[4 * q + 1] += bb.y; f[4 * q + 2] += bb.z; f[4 * q + 3] += bb.w;
              }
            }
            const uint32_t d = stage_s + uint32_t(lane * kPitch + (half * (kG / 2) + ch * 32) * 2);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(d + q * 16),
                           "r"(ptx::pack_bf16x2(f[8 * q], f[8 * q + 1])), "r"(ptx::pack_bf16x2(f[8 * q + 2], f[8 * q + 3])),
                           "r"(ptx::pack_bf16x2(f[8 * q + 4], f[8 * q + 5])), "r"(ptx::pack_bf16x2(f[8 * q + 6], f[8 * q + 7]))
                           : "memory");
          }
          asm volatile("bar.sync %0, 64;" ::"r"(1 + quad) : "memory");
          // 2. the pair stores the 32 staged rows: consecutive threads write consecutive 16-byte
          //    pieces of the same output pixel, so each warp store covers whole pixels.
          {
            constexpr int kParts = kG / 8;        // 16-byte pieces per staged row
            constexpr int kRowStep = 64 / kParts; // rows advanced per pass of the pair
            const int tp = half * 32 + lane;
            const int part = tp % kParts;
            const int co = n0 + g * kG + part * 8;
            if (co < n_end) {
              int row = tp / kParts;
              const int q = qbase + row;
              int r = q / ph_P, colv = q - r * ph_P;
              // All staged pieces are read first, then stored: one shared-memory round trip per
              // thread instead of one per store.  (The loads need no memory clobber: the pair
              // barrier above already orders them after the staging writes.)
              constexpr int kIters = 32 / kRowStep;
              uint4 val[kIters];
              int pix[kIters];
#pragma unroll
              for (int i = 0; i < kIters; ++i) {
                asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(val[i].x), "=r"(val[i].y), "=r"(val[i].z), "=r"(val[i].w)
                             : "r"(stage_s + uint32_t(row * kPitch + part * 16)));
                pix[i] = (r < ph_R && colv < ph_OWv) ? (row_base + r * ph_sh) * Wo + (col0 + colv) * ph_sw + ph_pw : -1;
                row += kRowStep;
                colv += kRowStep;
                while (colv >= ph_P) { colv -= ph_P; ++r; }
              }
#pragma unroll
              for (int i = 0; i < kIters; ++i)
                if (pix[i] >= 0) *reinterpret_cast<uint4*>(out + size_t(pix[i]) * Cn + co) = val[i];
            }
          }
          if (a.stage_bufs == 1) asm volatile("bar.sync %0, 64;" ::"r"(1 + quad) : "memory");
        }
      }
      if (stopped) break;
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
  Maps maps;
  int bn, nsub;
  bool bres, dgrad;
  bool tpos;  // channels on M, positions on N (the 128-channel tile)
  int row_step = 1, col_step = 1;  // strided view of the activations (strided 1x1 forward)
  size_t smem;
  int grid;
  // geometry kept for the tensor maps (Di: depth of the activation read, x or dy, when 3-D; else 0)
  int N, Hi, Wi, Ck, Cw, Di;
  int G, Ctot;  // groups, and the activation's channel count (Ck is one group's)
};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

int floordiv(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

int pick_bn(int64_t cn) {
  int best = 0, best_cols = 0;
  for (int bn : {256, 192, 128, 64}) {
    const int64_t cols = ((cn + bn - 1) / bn) * bn;
    if (!best || cols < best_cols) { best = bn; best_cols = int(cols); }
  }
  return best;
}

struct PhaseSpec {
  Phase ph;
  int maxoff;
  // tap t reads the halo at (tdr[t], tdc[t]) rows / columns past virtual (0, 0); the offsets span
  // rspan rows and cspan columns (the horizontal reach)
  int tdr[kMaxTapsPerPhase], tdc[kMaxTapsPerPhase];
  int rspan, cspan;
};

// Lays a phase out on strips of strip_w valid columns: pitch, tap offsets and the largest offset.
void layout_strips(PhaseSpec& s, int strip_w) {
  Phase& ph = s.ph;
  ph.strip_w = strip_w;
  ph.nstrips = (ph.OWv + strip_w - 1) / strip_w;
  ph.P = strip_w + s.cspan;
  for (int t = 0; t < ph.ntaps; ++t) ph.tap_off[t] = s.tdr[t] * ph.P + s.tdc[t];
  s.maxoff = s.rspan * ph.P + s.cspan;
}

// Fills the per-phase box geometry and counts for a tile of 128*nsub positions.
bool finish_phase(PhaseSpec& s, int nsub, int N) {
  Phase& ph = s.ph;
  if (ph.row_step == 0) ph.row_step = 1;
  if (ph.col_step == 0) ph.col_step = 1;
  const int mt = 128 * nsub;
  ph.bh = (ph.P - 1 + mt + s.maxoff + ph.P - 1) / ph.P;
  // TMA box extent limit (a strided view spans stride x the loaded extent)
  if (ph.P * ph.col_step > 256 || ph.bh * ph.row_step > 256) return false;
  ph.a_bytes = 128 * ph.P * ph.bh;
  const int64_t per_img = int64_t(ph.R) * ph.P;
  ph.tiles = int((per_img + mt - 1) / mt);
  return int64_t(N) * ph.nstrips * ph.tiles < (int64_t(1) << 30);
}

bool plan_geometry(const Problem& p, bool dgrad, Plan& pl) {
  if (!(p.bf16 && p.nhwc && p.ohwi)) return false;
  // A real depth axis: kernel-depth taps are more activation sources (5-D TMA boxes).  The gradient
  // also splits dx into depth phases at a depth stride: phase ad holds the slices id = ad + j*SD,
  // each met by the kernel-depth taps with (ad + PD - kd*DD) divisible by SD.
  const bool deep = p.D > 1 || p.KD > 1 || p.OD > 1;
  // Groups: one GEMM per group, the group a dimension of the activation view (5-D boxes, so not
  // with a depth axis as well).
  if (p.G > 1 && deep) return false;
  // At C_in/G <= 8 a group's reduction fills at most an eighth of a 64-channel k-block: the direct
  // (CUDA-core) families take those shapes.
  if (p.G > 1 && p.cpg() <= 8) return false;
  if (p.cpg() % 8 != 0 || p.opg() % 8 != 0) return false;  // 16-byte TMA strides of the group views
  if (deep && dgrad && p.KD > kMaxSrc) return false;
  // A strided forward reads its activations through strided views (TMA element strides <= 8).
  if (!dgrad && (p.SH > 8 || p.SW > 8)) return false;
  if (dgrad && (deep ? p.SD : 1) * p.SH * p.SW > kMaxPhases) return false;
  if (p.Cin % 8 != 0 || p.Cout % 8 != 0) return false;  // 16-byte TMA strides and vector stores
  if (p.KD * p.KH * p.KW > kMaxTapsPerPhase) return false;
  pl = Plan{};
  pl.dgrad = dgrad;
  Args& a = pl.a;
  const int64_t Ck = dgrad ? p.opg() : p.cpg(), Cn = dgrad ? p.Cin : p.Cout;  // Ck: one group's reduction
  const int64_t Cg = dgrad ? p.cpg() : p.opg();                                 // one group's output channels
  pl.bn = pick_bn(Cg);
  pl.nsub = pl.bn <= 128 ? 2 : 1;
  pl.tpos = pl.bn == 128;
  // 3-D: items run over (batch, depth slice) pairs of each phase (its jd slices of y, or of dx)
  a.N = int(p.N);
  a.depth_od = deep ? 1 : 0;
  a.depth_sd = deep ? (dgrad ? 1 : int(p.SD)) : 0;
  a.out_d = deep ? int(dgrad ? p.D : p.OD) : 0;
  a.out_sd = deep && dgrad ? int(p.SD) : 1;
  a.Cn = int(Cn);
  a.G = int(p.G);
  a.cg_k = int(Ck);
  a.cg_n = int(Cg);
  a.Ho = int(p.H);
  a.Wo = int(p.W);
  if (!dgrad) { a.Ho = int(p.OH); a.Wo = int(p.OW); }
  a.T = int(p.KD * p.KH * p.KW);
  a.kb_count = int((Ck + kKB - 1) / kKB);
  a.n_tiles = int((Cg + pl.bn - 1) / pl.bn);
  a.bias_n = int((p.G - 1) * Cg + int64_t(a.n_tiles) * pl.bn);  // covers the last group's last tile
  pl.N = int(p.N);
  pl.G = int(p.G);
  pl.Ctot = int(dgrad ? p.Cout : p.Cin);
  pl.Di = deep ? int(dgrad ? p.OD : p.D) : 0;  // depth of the activation the boxes read (x, or dy)
  pl.Hi = int(dgrad ? p.OH : p.H);
  pl.Wi = int(dgrad ? p.OW : p.W);
  pl.Ck = int(Ck);
  pl.Cw = int(p.cpg());  // the weight's innermost extent [C_out][T][C_in/G]

  PhaseSpec specs[kMaxPhases];
  int nph = 0;
  if (!dgrad) {
    // Tap (kh, kw) reads input (oh*SH + rr, ow*SW + cc), rr = kh*DH - PH, cc = kw*DW - PW.  With
    // rr = SH*dr + ah (0 <= ah < SH) that is row oh + dr of stride phase ah of the input: the
    // taps of one (ah, aw) phase are shifted windows of that phase's dense grid (its strided view),
    // so the forward is the shifted-window GEMM once per phase, all into one accumulator.
    PhaseSpec s{};
    Phase& ph = s.ph;
    int drs[kMaxTapsPerPhase], dcs[kMaxTapsPerPhase], ahs[kMaxTapsPerPhase], aws[kMaxTapsPerPhase];
    int kds[kMaxTapsPerPhase];
    int rmin = 0, rmax = 0, cmin = 0, cmax = 0;
    for (int kd = 0; kd < p.KD; ++kd)
    for (int kh = 0; kh < p.KH; ++kh)
      for (int kw = 0; kw < p.KW; ++kw) {
        const int t = int((kd * p.KH + kh) * p.KW + kw);  // the weight's [KD][KH][KW] tap
        kds[t] = kd;
        const int rr = int(kh * p.DH - p.PH), cc = int(kw * p.DW - p.PW);
        ahs[t] = ((rr % int(p.SH)) + int(p.SH)) % int(p.SH);
        aws[t] = ((cc % int(p.SW)) + int(p.SW)) % int(p.SW);
        drs[t] = (rr - ahs[t]) / int(p.SH);
        dcs[t] = (cc - aws[t]) / int(p.SW);
        rmin = t ? std::min(rmin, drs[t]) : drs[t];
        rmax = t ? std::max(rmax, drs[t]) : drs[t];
        cmin = t ? std::min(cmin, dcs[t]) : dcs[t];
        cmax = t ? std::max(cmax, dcs[t]) : dcs[t];
      }
    ph.ntaps = a.T;
    ph.R = int(p.OH); ph.OWv = int(p.OW);
    ph.P = int(p.OW) + (cmax - cmin);
    ph.rmin = rmin; ph.cmin = cmin;
    ph.out_sh = 1; ph.out_sw = 1;
    ph.row_step = int(p.SH);
    ph.col_step = int(p.SW);
    pl.row_step = int(p.SH);
    pl.col_step = int(p.SW);
    // taps grouped by source, sources in (kernel depth, ah, aw) order
    int k = 0;
    ph.nsrc = 0;
    for (int kd = 0; kd < p.KD; ++kd)
    for (int ah = 0; ah < p.SH; ++ah)
      for (int aw = 0; aw < p.SW; ++aw) {
        const int start = k;
        for (int t = 0; t < a.T; ++t) {
          if (kds[t] != kd || ahs[t] != ah || aws[t] != aw) continue;
          s.tdr[k] = drs[t] - rmin;
          s.tdc[k] = dcs[t] - cmin;
          ph.tap_w[k] = t;
          ++k;
        }
        if (k == start) continue;
        if (ph.nsrc == kMaxSrc) return false;
        ph.src_ah[ph.nsrc] = int8_t(ah);
        ph.src_aw[ph.nsrc] = int8_t(aw);
        ph.src_ad[ph.nsrc] = int(kd * p.DD - p.PD);
        ph.src_t0[ph.nsrc] = int8_t(start);
        ++ph.nsrc;
      }
    ph.src_t0[ph.nsrc] = int8_t(k);
    s.rspan = rmax - rmin;
    s.cspan = cmax - cmin;
    ph.jd = deep ? int(p.OD) : 1;
    ph.out_pd = 0;
    specs[nph++] = s;
  } else {
    const int SD = deep ? int(p.SD) : 1;
    for (int ad = 0; ad < SD; ++ad)
    for (int ah = 0; ah < p.SH; ++ah)
      for (int aw = 0; aw < p.SW; ++aw) {
        PhaseSpec s{};
        Phase& ph = s.ph;
        ph.jd = deep ? int((p.D - ad + SD - 1) / SD) : 1;
        ph.out_pd = ad;
        if (ph.jd <= 0) continue;
        // the kernel-depth taps that reach depth phase ad, and their dy slice offsets
        int kds[kMaxSrc], nkd = 0;
        for (int kd = 0; kd < (deep ? p.KD : 1); ++kd) {
          const int num = deep ? int(ad + p.PD - kd * p.DD) : 0;
          if (((num % SD) + SD) % SD == 0) { ph.src_ad[nkd] = num / SD; kds[nkd++] = kd; }
        }
        ph.R = int((p.H - ah + p.SH - 1) / p.SH);
        ph.OWv = int((p.W - aw + p.SW - 1) / p.SW);
        if (ph.R <= 0 || ph.OWv <= 0) continue;
        int khs[kMaxTapsPerPhase], drs[kMaxTapsPerPhase], nkh = 0;
        int kws[kMaxTapsPerPhase], dcs[kMaxTapsPerPhase], nkw = 0;
        for (int kh = 0; kh < p.KH; ++kh) {
          const int num = int(ah + p.PH - kh * p.DH);
          if (((num % p.SH) + p.SH) % p.SH == 0) { khs[nkh] = kh; drs[nkh] = floordiv(num, int(p.SH)); ++nkh; }
        }
        for (int kw = 0; kw < p.KW; ++kw) {
          const int num = int(aw + p.PW - kw * p.DW);
          if (((num % p.SW) + p.SW) % p.SW == 0) { kws[nkw] = kw; dcs[nkw] = floordiv(num, int(p.SW)); ++nkw; }
        }
        int rmin = 0, rmax = 0, cmin = 0, cmax = 0;
        for (int i = 0; i < nkh; ++i) { rmin = i ? std::min(rmin, drs[i]) : drs[i]; rmax = i ? std::max(rmax, drs[i]) : drs[i]; }
        for (int i = 0; i < nkw; ++i) { cmin = i ? std::min(cmin, dcs[i]) : dcs[i]; cmax = i ? std::max(cmax, dcs[i]) : dcs[i]; }
        ph.ntaps = nkh * nkw * nkd;
        ph.P = ph.OWv + (cmax - cmin);
        ph.rmin = rmin; ph.cmin = cmin;
        ph.out_sh = int(p.SH); ph.out_sw = int(p.SW); ph.out_ph = ah; ph.out_pw = aw;
        // dy is read as it is, one source per kernel-depth tap kd that reaches the phase (zero
        // filled outside dy).  2-D: one source.
        ph.row_step = ph.col_step = 1;
        ph.nsrc = nkd;
        for (int k = 0; k < nkd; ++k) {
          ph.src_ah[k] = ph.src_aw[k] = 0;
          ph.src_t0[k] = int8_t(k * nkh * nkw);
          for (int i = 0; i < nkh; ++i)
            for (int j = 0; j < nkw; ++j) {
              const int t = (k * nkh + i) * nkw + j;
              s.tdr[t] = drs[i] - rmin;
              s.tdc[t] = dcs[j] - cmin;
              ph.tap_w[t] = int((kds[k] * p.KH + khs[i]) * p.KW + kws[j]);
            }
        }
        ph.src_t0[nkd] = int8_t(ph.ntaps);
        s.rspan = rmax - rmin;
        s.cspan = cmax - cmin;
        specs[nph++] = s;
      }
    // Longest phases first, so the persistent CTAs finish together.
    std::stable_sort(specs, specs + nph, [](const PhaseSpec& x, const PhaseSpec& y) { return x.ph.ntaps > y.ph.ntaps; });
  }
  if (nph == 0) return false;
  a.nphase = nph;
  a.b_tile_bytes = pl.bn * kKB * 2;
  pl.bres = !dgrad && a.G == 1 && a.n_tiles == 1 && a.T * a.kb_count * a.b_tile_bytes <= 110 * 1024;
  const size_t block = size_t(128) * ((pl.bn % 128 == 0 ? 128 : 64) * 2 + 16);
  // The fewest column strips per image whose halo boxes fit a box and the shared memory (one strip:
  // whole image rows).
  int max_w = 1;
  for (int i = 0; i < nph; ++i) max_w = std::max(max_w, specs[i].ph.OWv);
  for (int k = 1; k <= max_w; ++k) {
    int item = 0, a_max = 0;
    bool fits = true;
    for (int i = 0; fits && i < nph; ++i) {
      const int imgs = a.N * specs[i].ph.jd;  // (batch, depth slice) pairs; 2-D: the batch
      layout_strips(specs[i], (specs[i].ph.OWv + k - 1) / k);
      if (!finish_phase(specs[i], pl.nsub, imgs)) { fits = false; break; }
      specs[i].ph.item0 = item;
      const int64_t n_all = int64_t(a.n_tiles) * a.G;  // (group, output tile) pairs
      const int64_t n_items = int64_t(imgs) * specs[i].ph.nstrips * specs[i].ph.tiles * n_all;
      if (int64_t(item) + n_items >= (int64_t(1) << 30)) return false;
      item += int(n_items);
      a.ph[i] = specs[i].ph;
      a_max = std::max(a_max, specs[i].ph.a_bytes);
    }
    if (!fits) continue;
    a.total_items = item;
    a.a_stage_bytes = (a_max + 1023) & ~1023;
    // (the transposed form has its own staging layout, of fixed size)
    for (int bufs = pl.tpos ? 1 : 2; bufs >= 1; --bufs) {
      const size_t fixed = 1024 + (pl.tpos ? size_t(kTposStage) : bufs * block) + size_t(a.bias_n) * 4 +
                           size_t(kMaxPhases) * 2 * kMaxTapsPerPhase * 4 + kMaxPhases * sizeof(PhaseHdr) +
                           8 * (2 * 4 + 2 * 8 + 8) + 16;
      // streamed weights: at least four weight stages before a third activation stage
      for (int min_sb = pl.bres ? 1 : 4; min_sb >= (pl.bres ? 1 : 3); --min_sb)
      for (int sa = 3; sa >= 2; --sa) {
        for (int sb = pl.bres ? 1 : 8; sb >= min_sb; --sb) {
          const size_t total =
              fixed + size_t(sa) * a.a_stage_bytes + size_t(pl.bres ? a.T * a.kb_count : sb) * a.b_tile_bytes;
          if (total <= size_t(kSmemLimit)) {
            a.sa = sa;
            a.sb = pl.bres ? 1 : sb;
            a.stage_bufs = bufs;
            pl.smem = total;
            return true;
          }
        }
      }
    }
  }
  return false;
}

bool encode_maps(Plan& pl, const void* in, const void* w) {
  pl.a.b4d = 0;
  auto fn = encode_fn();
  if (!fn) return false;
  const Args& a = pl.a;
  for (int i = 0; i < a.nphase; ++i) {
    const Phase& ph = a.ph[i];
    // A strided view spans stride x the loaded extent and loads every stride-th element (the
    // forward of a strided 1x1); otherwise row_step = col_step = 1.  A 3-D problem adds the
    // activation's depth as a fifth dimension, one slice per box.
    const int rank = (pl.Di > 0 || pl.G > 1) ? 5 : 4;
    const cuuint64_t plane = cuuint64_t(pl.Hi) * pl.Wi * pl.Ctot * 2;
    cuuint64_t dims[5] = {cuuint64_t(pl.Ck), cuuint64_t(pl.Wi), cuuint64_t(pl.Hi), cuuint64_t(pl.N), 1};
    cuuint64_t strides[4] = {cuuint64_t(pl.Ctot) * 2, cuuint64_t(pl.Wi) * pl.Ctot * 2, plane, 0};
    cuuint32_t box[5] = {cuuint32_t(kKB), cuuint32_t(ph.P * pl.col_step), cuuint32_t(ph.bh * pl.row_step), 1, 1};
    cuuint32_t estr[5] = {1, cuuint32_t(pl.col_step), cuuint32_t(pl.row_step), 1, 1};
    if (pl.Di > 0) {
      dims[3] = cuuint64_t(pl.Di);
      dims[4] = cuuint64_t(pl.N);
      strides[3] = plane * cuuint64_t(pl.Di);
    } else if (pl.G > 1) {
      // (channel in group, group, column, row, image): each box stays inside one group's channels
      const cuuint64_t d5[5] = {cuuint64_t(pl.Ck), cuuint64_t(pl.G), cuuint64_t(pl.Wi), cuuint64_t(pl.Hi),
                                cuuint64_t(pl.N)};
      const cuuint64_t s4[4] = {cuuint64_t(pl.Ck) * 2, cuuint64_t(pl.Ctot) * 2, cuuint64_t(pl.Wi) * pl.Ctot * 2, plane};
      const cuuint32_t b5[5] = {cuuint32_t(kKB), 1, cuuint32_t(ph.P * pl.col_step), cuuint32_t(ph.bh * pl.row_step), 1};
      const cuuint32_t e5[5] = {1, 1, cuuint32_t(pl.col_step), cuuint32_t(pl.row_step), 1};
      for (int k = 0; k < 5; ++k) { dims[k] = d5[k]; box[k] = b5[k]; estr[k] = e5[k]; }
      for (int k = 0; k < 4; ++k) strides[k] = s4[k];
    }
    if (fn(&pl.maps.a[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cuuint32_t(rank), const_cast<void*>(in), dims, strides, box,
           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  const int Cout = pl.dgrad ? pl.Ctot : a.Cn;  // the weight's C_out extent (all groups)
  if (pl.dgrad) {
    // The OHWI weight [C_out][T][C_in] viewed as (C_in % 64, C_out, C_in / 64, tap): a box of
    // (64, 64, BN/64, 1) lands as BN/64 contiguous [64 C_out][64 C_in] atoms, the MN-major operand.
    cuuint64_t dims[4] = {64, cuuint64_t(Cout), cuuint64_t((pl.Cw + 63) / 64), cuuint64_t(a.T)};
    cuuint64_t strides[3] = {cuuint64_t(a.T) * pl.Cw * 2, 128, cuuint64_t(pl.Cw) * 2};
    cuuint32_t box[4] = {64, 64, cuuint32_t(pl.bn / 64), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    // The C_in / 64 split needs whole 64-channel blocks; otherwise 64-wide 3-D boxes below.
    pl.a.b4d = pl.Cw % 64 == 0 &&
               fn(&pl.maps.b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(w), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    if (pl.a.b4d) return true;
  }
  cuuint64_t dims[3] = {cuuint64_t(pl.Cw), cuuint64_t(a.T), cuuint64_t(Cout)};
  cuuint64_t strides[2] = {cuuint64_t(pl.Cw) * 2, cuuint64_t(a.T) * pl.Cw * 2};
  cuuint32_t box[3] = {cuuint32_t(kKB), 1, cuuint32_t(pl.dgrad ? kKB : pl.bn)};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(&pl.maps.b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int NSUB, bool DGRAD, bool BRES, bool MSRC = false, bool TPOS = false>
gbconv_status run(const Plan& pl, const Launch& l) {
  auto kern = implicit_gemm_kernel<BN, NSUB, DGRAD, BRES, MSRC, TPOS>;
  // The shared-memory opt-in is a per-device function attribute: raise it once per device.
  static std::atomic<uint64_t> done[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GBCONV_ECUDA;
  if (done[dev].load(std::memory_order_acquire) < uint64_t(pl.smem)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemLimit)) != cudaSuccess)
      return GBCONV_ECUDA;
    done[dev].store(uint64_t(kSmemLimit), std::memory_order_release);
  }
  return launch_kernel(kern, dim3(pl.grid), dim3(kThreads), pl.smem, l.stream, pl.maps, pl.a) == cudaSuccess
             ? GBCONV_OK
             : GBCONV_ECUDA;
}

template <bool DGRAD, bool MSRC>
gbconv_status dispatch_src(const Plan& pl, const Launch& l) {
  if (!DGRAD && pl.bres) {
    switch (pl.bn) {
      case 256: return run<256, 1, false, true, MSRC>(pl, l);
      case 192: return run<192, 1, false, true, MSRC>(pl, l);
      case 128: return run<128, 2, false, true, MSRC, true>(pl, l);
      default: return run<64, 2, false, true, MSRC>(pl, l);
    }
  }
  switch (pl.bn) {
    case 256: return run<256, 1, DGRAD, false, MSRC>(pl, l);
    case 192: return run<192, 1, DGRAD, false, MSRC>(pl, l);
    case 128: return run<128, 2, DGRAD, false, MSRC, true>(pl, l);
    default: return run<64, 2, DGRAD, false, MSRC>(pl, l);
  }
}

template <bool DGRAD>
gbconv_status dispatch(const Plan& pl, const Launch& l) {
  // Several activation sources: a strided forward's stride phases, or a 3-D kernel's depth taps.
  if (pl.a.depth_od > 0 || pl.a.ph[0].nsrc > 1) return dispatch_src<DGRAD, true>(pl, l);
  return dispatch_src<DGRAD, false>(pl, l);
}

gbconv_status launch(const Problem& p, bool dgrad, const void* in, const void* w, const float* bias, void* out,
                     const Launch& l) {
  Plan pl;
  if (!plan_geometry(p, dgrad, pl)) return GBCONV_EUNSUPPORTED;
  pl.a.bias = bias;
  pl.a.out = static_cast<bf16*>(out);
  pl.a.status = l.status;
  pl.a.wait_ns = l.wait_ns;
  pl.grid = std::max(1, std::min(pl.a.total_items, l.num_sms));
  if (!encode_maps(pl, in, w)) return GBCONV_ECUDA;
  return dgrad ? dispatch<true>(pl, l) : dispatch<false>(pl, l);
}

}  // namespace

bool implicit_fwd_supported(const Problem& p) {
  Plan pl;
  return plan_geometry(p, false, pl);
}

bool implicit_dgrad_supported(const Problem& p) {
  Plan pl;
  return plan_geometry(p, true, pl);
}

bool implicit_describe(const Problem& p, bool dgrad, char* buf, size_t len) {
  Plan pl;
  if (!plan_geometry(p, dgrad, pl)) return false;
  const Args& a = pl.a;
  int taps = 0;
  for (int i = 0; i < a.nphase; ++i) taps = std::max(taps, a.ph[i].ntaps);
  std::snprintf(buf, len,
                "implicit_gemm %s m_side=%s bn=%d nsub=%d phases=%d sources=%d taps=%d items=%d kb=%d weights=%s "
                "a_stages=%d b_stages=%d stage_bufs=%d strips=%d smem=%zu",
                dgrad ? "dgrad" : "fwd", pl.tpos ? "channels" : "positions", pl.bn, pl.nsub, a.nphase, a.ph[0].nsrc, taps, a.total_items, a.kb_count,
                pl.bres ? "resident" : "streamed", a.sa, pl.bres ? 0 : a.sb, a.stage_bufs, a.ph[0].nstrips, pl.smem);
  return true;
}

gbconv_status launch_implicit_fwd(const Problem& p, const void* x, const void* w, const float* bias, void* y,
                                  const Launch& l) {
  return launch(p, false, x, w, bias, y, l);
}

gbconv_status launch_implicit_dgrad(const Problem& p, const void* dy, const void* w, const float* bias, void* dx,
                                    const Launch& l) {
  return launch(p, true, dy, w, bias, dx, l);
}

}  // namespace gbconv
