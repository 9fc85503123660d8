// Weight gradient on the 5th-generation tensor cores (tcgen05, accumulators in TMEM), NHWC bf16,
// one group, H/W strides up to 4 (described below at unit stride first).
//
// The contraction (burn-cubecl `wgrad_im2col`: [C_out, positions] x [positions, taps * C_in]) runs
// over positions of the same virtual grid the forward uses: R output rows of P = OW + (KW-1)*DW
// columns per image.  x is read through the virtual grid (x_v row r = input row r - PH, column
// c = input column c - PW, zero outside the image) and dy through the same grid (columns past OW
// are zero), so tap (kh, kw) pairs dy position q with x_v position q + kh*DH*P + kw*DW: every tap is a
// shifted window, and since every tap's product is a separate output no shifted sums are needed.
//
// One MMA covers many taps at once.  Both operands are position-major in shared memory (MN-major,
// 128-byte swizzle, one 128-byte row of 64 channels per position), and an MN-major operand wider than
// 64 is a row of 64-wide atoms at a stride the descriptor states (its leading-byte offset):
//   A (M = 128) = two x atoms DH*P positions apart: kernel rows kh and kh+1 of 64 input channels;
//   B (N = 64*KW) = KW dy atoms DW positions apart: kernel columns KW-1 .. 0 of 64 output channels.
// D[(kh, ci), (kw, co)] accumulates the product of x at q + kh*DH*P and dy at q - (KW-1-j)*DW
// (j = the atom), which is tap (kh, kw = KW-1-j) of the weight gradient.  ceil(KH/2) such MMAs per
// 16 positions cover every tap (a 3x3: two MMAs of M=128, N=192, the second one half used).
//
// Work: one CTA per (64-channel input block, group of nco 64-channel output blocks, chunk of output
// rows); nco = 2 where the accumulators fit TMEM twice, so that x is loaded once for two output blocks
// (each output block has its own dy region and its own MMAs, into its own TMEM columns).  A chunk
// is a run of row blocks (RB rows, with RB*P a multiple of 8 so every TMA box lands on a 1024-byte
// boundary); it is loaded whole into shared memory as boxes of RB virtual rows (x and dy, one
// barrier each) and swept by the MMAs as the boxes land.  At the end the accumulators go to the
// caller's workspace as fp32 partial sums [chunk][co][kh][kw][ci]; launch_wgrad_reduce then adds the
// chunks in chunk order.  No atomics anywhere: the result is deterministic.
//
// An H/W stride (SH, SW) splits x into stride phases: phase (ah, aw) is x at rows ah (mod SH) and
// columns aw (mod SW), read as a dense grid through a strided TMA view.  Tap (kh, kw) reads phase
// ((kh*DH - PH) mod SH, (kw*DW - PW) mod SW), and the taps of one phase sit DH / gcd(DH, SH) phase
// rows (and DW / gcd(DW, SW) phase columns) apart, so each phase is the unit-stride sum above over
// its own taps, with its own N.  A work unit takes one phase and writes only that phase's taps.
//
// A 3-D shape runs the same sums over (batch, output depth) slices, one kernel-depth tap kd per
// unit: the unit pairs dy slice od with x slice od*SD + kd*DD - PD (5-D boxes, zero filled outside
// x) and writes only its kd's taps of the chunk's partial sums.
//
// Roles: warps 0-7 epilogue (TMEM -> workspace), warp 8 TMEM allocation and MMA issue (lane 0),
// warp 9 zero fill and TMA loads (lane 0 issues).
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

constexpr int kEpiWarps = 8;
constexpr int kMmaWarp = 8;
constexpr int kTmaWarp = 9;
constexpr int kThreads = 10 * 32;
constexpr int kFront = 8;       // zero positions ahead of the dy rows: the dy atoms reach back (KW-1)*DW <= 8
constexpr int kMaxBoxes = 24;   // per segment, for x and for dy
constexpr int kSmemLimit = 227 * 1024;
constexpr int kStepBlock = 4;   // 16-position MMA steps issued back to back
constexpr int kMaxWgPhases = 16;  // H/W stride phases (strides up to 4 x 4)

struct TcArgs {
  float* ws;              // [chunk][ws_stride] fp32 partial sums, elements in OHWI order
  unsigned int* status;
  uint64_t wait_ns;       // bound of every barrier wait (the host sets it; 2 s by default)
  int Cin, Cout, KH, KW, DH, DW, PH, PW;
  int SH, SW;             // H/W strides: x is read through a strided view (TMA element strides)
  int ddr, ddc;           // phase-grid rows / columns between a stride phase's consecutive kernel rows / columns
  int KD, SD, DD, PD, OD;  // depth: kernel taps, stride, dilation, begin padding, output depth (2-D: 1, 1, 1, 0, 0)
  int nph;                // stride phases that hold taps (1 at unit stride)
  int KWP;                // most kernel columns in one phase: a group's TMEM columns are KWP * 64
  int P;                  // virtual grid pitch OW + (KWP-1)*ddc
  int RB;                 // virtual rows per TMA box
  int box_bytes;          // RB * P * 128
  int cb_in, pairs, chunks, units;  // pairs: (input block, output block group); units: pairs x chunks x KD x nph
  int nco;                // output blocks per unit (1 or 2)
  int y_bytes;            // one output block's dy region: front pad, a segment's boxes, tail
  int bpi, total_blocks;  // row blocks per image (a (batch, depth) slice when 3-D), row blocks in the batch
  int seg_blocks;         // row blocks one shared-memory load holds
  int xe;                 // x boxes a segment needs beyond its dy boxes
  int gm;                 // MMA groups per 16 positions: ceil(kernel rows of a phase / 2), at most
  int x_bytes;            // x region bytes (the dy region follows)
  int tail;               // zero positions needed after a segment's dy rows
  int ws_stride;          // floats per chunk in the workspace
  // Stride phase q: its kernel rows (A atom 2g+i is row ph_kh[q][2g+i]) and kernel columns (B atom j is
  // column ph_kw[q][nkw-1-j]), the x row and column of its virtual (0, 0) (x row = r * SH + ph_r0), and
  // its MMA instruction descriptor (N = 64 * nkw).
  int8_t ph_kh[kMaxWgPhases][4], ph_kw[kMaxWgPhases][4], ph_nkh[kMaxWgPhases], ph_nkw[kMaxWgPhases];
  int ph_r0[kMaxWgPhases], ph_c0[kMaxWgPhases];
  uint32_t ph_idesc[kMaxWgPhases];
};

struct TcMaps {
  CUtensorMap x;   // (C_in, W, H, N), box (64, P, RB, 1); 3-D: (C_in, W, H, D, N), box (64, P, RB, 1, 1)
  CUtensorMap dy;  // (C_out, OW, OH, N), box (64, P, RB, 1); 3-D: (C_out, OW, OH, OD, N)
};

// A unit's kernel-depth tap, stride phase, chunk and (input block, output block) pair.
struct Unit {
  int kd, ph, chunk, pair;
  __device__ Unit(const TcArgs& a, int u) {
    const int classes = a.KD * a.nph;
    const int cls = u % classes;
    kd = cls / a.nph;
    ph = cls - kd * a.nph;
    const int v = u / classes;
    chunk = v / a.pairs;
    pair = v - chunk * a.pairs;
  }
};

struct Segment {
  int n, rb, nb;  // image, first row block, row blocks
};

// The segments of a chunk, in order: runs of its row blocks inside one image, at most seg_blocks long.
struct SegWalk {
  int b, b1, bpi, cap;
  __device__ SegWalk(const TcArgs& a, int chunk) {
    b = int((int64_t(chunk) * a.total_blocks) / a.chunks);
    b1 = int((int64_t(chunk + 1) * a.total_blocks) / a.chunks);
    bpi = a.bpi;
    cap = a.seg_blocks;
  }
  __device__ bool next(Segment& s) {
    if (b >= b1) return false;
    s.n = b / bpi;
    s.rb = b - s.n * bpi;
    s.nb = min(min(b1 - b, bpi - s.rb), cap);
    b += s.nb;
    return true;
  }
};

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

// MN-major operand, 128-byte swizzle: `atom_stride` bytes between 64-element atoms along M (or N),
// 1024 bytes between 8-position groups along K.
__device__ __forceinline__ uint64_t desc_mn_sw128(uint32_t saddr, uint32_t atom_stride) {
  uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((atom_stride >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// One block of tn 16-position steps (kStepBlock when full), G MMA groups per step, issued back to back.
template <int G>
__device__ __forceinline__ void issue_steps(int tn, uint32_t tmem, uint32_t ncols, uint32_t a_lo, uint32_t a_hi,
                                            uint32_t g_step, uint32_t b_lo, uint32_t b_hi, uint32_t idesc,
                                            uint32_t acc0) {
  if (tn == kStepBlock) {
#pragma unroll
    for (int i = 0; i < kStepBlock; ++i)
#pragma unroll
      for (int g = 0; g < G; ++g)
        ptx::mma_bf16_lohi(tmem + uint32_t(g) * ncols, a_lo + uint32_t(i) * 128u + uint32_t(g) * g_step, a_hi,
                           b_lo + uint32_t(i) * 128u, b_hi, idesc, i == 0 ? acc0 : 1u);
  } else {
    for (int i = 0; i < tn; ++i)
#pragma unroll
      for (int g = 0; g < G; ++g)
        ptx::mma_bf16_lohi(tmem + uint32_t(g) * ncols, a_lo + uint32_t(i) * 128u + uint32_t(g) * g_step, a_hi,
                           b_lo + uint32_t(i) * 128u, b_hi, idesc, i == 0 ? acc0 : 1u);
  }
}

// GM: MMA groups per 16 positions (ceil(KH/2)), and NCO: output blocks per unit (a.nco), template
// parameters so a block of steps issues its MMAs back to back: scalar work between MMAs in the issuing
// thread adds directly to their time.
template <int GM, int NCO>
__global__ void __launch_bounds__(kThreads, 1)
    wgrad_tc_kernel(const __grid_constant__ TcMaps maps, const __grid_constant__ TcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* xs = smem;
  uint8_t* ys = smem + a.x_bytes;  // position 0 of output block 0's dy region; the dy rows start at kFront
  const int y_bytes = a.y_bytes;   // output block c's region starts c * y_bytes later
  uint64_t* xbar = reinterpret_cast<uint64_t*>(ys + NCO * y_bytes);
  uint64_t* ybar = xbar + kMaxBoxes;
  uint64_t* seg_done = ybar + kMaxBoxes;
  uint64_t* acc_full = seg_done + 1;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* fin = acc_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fin + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t acc_cols = uint32_t(GM * a.KWP * 64);  // TMEM columns of one output block's accumulators
  const uint32_t tmem_cols = NCO * acc_cols <= 256 ? 256u : 512u;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kMaxBoxes; ++i) { ptx::mbar_init(xbar + i, 1); ptx::mbar_init(ybar + i, 1); }
    ptx::mbar_init(seg_done, 1);
    ptx::mbar_init(acc_full, 1);
    ptx::mbar_init(acc_empty, kEpiWarps * 32);
    ptx::mbar_init(fin, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(tmem_slot, tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ zero fill and TMA producer
#pragma unroll
    for (int c = 0; c < NCO; ++c)  // the front pads, never written by TMA
      for (int i = lane; i < kFront * 8; i += 32)
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(ptx::smem_addr(ys) + uint32_t(c * y_bytes + i * 16)),
                     "r"(0u)
                     : "memory");
    if (lane == 0) {
      ptx::prefetch_tmap(&maps.x);
      ptx::prefetch_tmap(&maps.dy);
    }
    bool ok = true;
    int seg = 0;            // segments this CTA has loaded
    uint32_t xph = 0, yph = 0;  // bit b: the phase parity box barrier b completes next
    for (int u = int(blockIdx.x); ok && u < a.units; u += int(gridDim.x)) {
      const Unit un(a, u);
      const int cib = un.pair % a.cb_in, cob = (un.pair / a.cb_in) * NCO;  // the group's first output block
      SegWalk walk(a, un.chunk);
      Segment sg;
      while (ok && walk.next(sg)) {
        if (seg > 0) {  // the previous segment's MMAs have finished reading shared memory
          if (lane == 0) ok = ptx::mbar_wait(seg_done, uint32_t(seg - 1) & 1u, abort_flag, a.status, 1u, a.wait_ns);
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) break;
        }
        // The last MMAs of a segment read up to tail positions past its dy rows: zero them (a
        // longer earlier segment may have left dy rows there), then order the writes before the
        // tensor core's reads.
        const uint32_t tail0 = ptx::smem_addr(ys) + uint32_t(kFront * 128 + sg.nb * a.box_bytes);
#pragma unroll
        for (int c = 0; c < NCO; ++c)
          for (int i = lane; i < a.tail * 8; i += 32)
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(tail0 + uint32_t(c * y_bytes + i * 16)), "r"(0u)
                         : "memory");
        ptx::fence_proxy_async_smem();
        __syncwarp();
        const int nxb = sg.nb + a.xe;
        if (lane == 0) {
          const int row0 = sg.rb * a.RB;  // first virtual row of the segment
          // 3-D: segment image sg.n is the (batch, output depth) slice (n, od); x is read at depth
          // od*SD + kd*DD - PD (zero filled outside the input)
          const int nn = a.OD > 0 ? sg.n / a.OD : sg.n, od = a.OD > 0 ? sg.n - nn * a.OD : 0;
          const int xd = od * a.SD + un.kd * a.DD - a.PD;
          // the unit's stride phase: virtual row r, column c read x row r*SH + r0, column c*SW + c0
          const int xr0 = a.ph_r0[un.ph], xc0 = a.ph_c0[un.ph];
          for (int b = 0; b < nxb; ++b) {
            ptx::mbar_arrive_expect_tx(xbar + b, uint32_t(a.box_bytes));
            const int xrow = (row0 + b * a.RB) * a.SH + xr0;
            if (a.OD > 0)
              tma_load_5d(ptx::smem_addr(xs) + uint32_t(b * a.box_bytes), &maps.x, xbar + b, cib * 64, xc0, xrow, xd,
                          nn);
            else
              tma_load_4d(ptx::smem_addr(xs) + uint32_t(b * a.box_bytes), &maps.x, xbar + b, cib * 64, xc0, xrow,
                          sg.n);
            if (b < sg.nb) {  // box b of every output block of the group, on one barrier
              ptx::mbar_arrive_expect_tx(ybar + b, uint32_t(NCO * a.box_bytes));
              for (int c = 0; c < NCO; ++c) {
                const uint32_t dst = ptx::smem_addr(ys) + uint32_t(c * y_bytes + kFront * 128 + b * a.box_bytes);
                if (a.OD > 0)
                  tma_load_5d(dst, &maps.dy, ybar + b, (cob + c) * 64, 0, row0 + b * a.RB, od, nn);
                else
                  tma_load_4d(dst, &maps.dy, ybar + b, (cob + c) * 64, 0, row0 + b * a.RB, sg.n);
              }
            }
          }
        }
        __syncwarp();
        // A segment uses boxes [0, nxb) and [0, nb): each of those barriers completes one phase.
        xph ^= (1u << nxb) - 1u;
        yph ^= (1u << sg.nb) - 1u;
        ++seg;
      }
    }
    // Leave no copy in flight: wait (bounded, whatever the abort state) until every box barrier has
    // completed the phases armed so far (the parity bits hold the next phase of each).
    if (lane == 0 && seg > 0) {
      const uint64_t t0 = ptx::globaltimer();
      for (int b = 0; b < 2 * kMaxBoxes; ++b) {
        uint64_t* bar = b < kMaxBoxes ? xbar + b : ybar + (b - kMaxBoxes);
        const uint32_t next = b < kMaxBoxes ? (xph >> b) & 1u : (yph >> (b - kMaxBoxes)) & 1u;
        while (!ptx::mbar_try_wait(bar, next ^ 1u) && ptx::globaltimer() - t0 < 200000000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      int seg = 0, it = 0;
      // Everything the loop needs, in registers: kernel parameters live in memory, and every MMA's
      // asm statement clobbers memory, so fields read inside the loop would be reloaded per MMA.
      const int P = a.P, xe = a.xe, units = a.units, ddr = a.ddr, ddc = a.ddc;
      const int box_pos = a.RB * a.P;                      // positions per box
      const uint32_t ncols = uint32_t(a.KWP * 64);         // TMEM columns between groups
      // A descriptor words at k = 0.  A step of 16 positions is 2048 bytes, +128 in the start field;
      // group g's A starts 2g*ddr*P positions on.
      const uint64_t ad0 = desc_mn_sw128(ptx::smem_addr(xs), uint32_t(ddr * P) * 128u);
      const uint32_t a_lo0 = uint32_t(ad0), a_hi = uint32_t(ad0 >> 32);
      const uint32_t g_step = uint32_t(2 * ddr * P) * 8u;  // (2*ddr*P*128) >> 4
      uint32_t xph = 0, yph = 0;  // bit b: the phase parity box barrier b completes next
      for (int u = int(blockIdx.x); ok && u < units; u += int(gridDim.x), ++it) {
        if (it > 0) {  // the epilogue has taken the previous unit's accumulators
          if (!(ok = ptx::mbar_wait(acc_empty, uint32_t(it - 1) & 1u, abort_flag, a.status, 2u, a.wait_ns))) break;
          ptx::tc_fence_after();
        }
        // the unit's stride phase: its groups, its N (its kernel columns) and its B atoms
        const Unit un(a, u);
        const int nkw = a.ph_nkw[un.ph], gmu = (a.ph_nkh[un.ph] + 1) / 2;
        const uint32_t idesc = a.ph_idesc[un.ph];
        const int xreach = (2 * gmu - 1) * ddr * P;  // farthest x position an MMA reads past k
        const uint64_t bd0 = desc_mn_sw128(ptx::smem_addr(ys) + uint32_t(kFront - (nkw - 1) * ddc) * 128u,
                                           uint32_t(ddc) * 128u);
        const uint32_t b_lo0 = uint32_t(bd0), b_hi = uint32_t(bd0 >> 32);
        const uint32_t b_next = uint32_t(y_bytes) >> 4;  // the next output block's dy region, in the start field
        SegWalk walk(a, un.chunk);
        Segment sg;
        bool first = true;
        while (ok && walk.next(sg)) {
          const int nb = sg.nb, nxb = sg.nb + xe;
          const int nk = (nb * box_pos + (nkw - 1) * ddc + 15) / 16;
          int xw = 0, yw = 0;  // boxes already waited for
          // Blocks of kStepBlock steps: the boxes the whole block reads are waited for first, then its
          // MMAs go out back to back.
          for (int t0 = 0; ok && t0 < nk; t0 += kStepBlock) {
            const int tn = min(kStepBlock, nk - t0);
            const int kend = 16 * (t0 + tn - 1) + 15;  // last position the block reads (before the shifts)
            for (; ok && yw < nb && kend >= yw * box_pos; ++yw)
              ok = ptx::mbar_wait(ybar + yw, (yph >> yw) & 1u, abort_flag, a.status, 2u, a.wait_ns);
            for (; ok && xw < nxb && kend + xreach >= xw * box_pos; ++xw)
              ok = ptx::mbar_wait(xbar + xw, (xph >> xw) & 1u, abort_flag, a.status, 2u, a.wait_ns);
            if (!ok) break;
            const uint32_t a_lo = a_lo0 + uint32_t(t0) * 128u, b_lo = b_lo0 + uint32_t(t0) * 128u;
            const uint32_t acc0 = (first && t0 == 0) ? 0u : 1u;
            // every group of the kernel (the unit-stride case), or a stride phase's fewer ones; each
            // output block of the unit into its own accumulators
#pragma unroll
            for (int c = 0; c < NCO; ++c) {
              if (gmu == GM)
                issue_steps<GM>(tn, tmem + uint32_t(c) * acc_cols, ncols, a_lo, a_hi, g_step, b_lo + uint32_t(c) * b_next,
                                b_hi, idesc, acc0);
              else
                issue_steps<1>(tn, tmem + uint32_t(c) * acc_cols, ncols, a_lo, a_hi, g_step, b_lo + uint32_t(c) * b_next,
                               b_hi, idesc, acc0);
            }
          }
          ptx::mma_commit(seg_done);
          xph ^= (1u << nxb) - 1u;
          yph ^= (1u << nb) - 1u;
          first = false;
          ++seg;
        }
        if (ok) ptx::mma_commit(acc_full);
      }
      ptx::mma_commit(fin);
      // every MMA issued so far completes before TMEM is freed, abort or not
      ptx::mbar_wait_drain(fin, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue: TMEM -> workspace
    // Warps w and w+4 share TMEM lanes 32*(w%4).. and split the 16-column chunks.  Lane m holds the
    // phase's kernel row 2g + m/64 and input channel m%64 of the block; column n of a group holds the
    // phase's kernel column nkw-1 - n/64 and output channel n%64.  Consecutive lanes store consecutive
    // input channels.
    const int q = warp & 3, h = warp >> 2;
    const uint32_t lane_base = uint32_t(q * 32) << 16;
    const int m = q * 32 + lane;
    const int i_atom = m >> 6, cil = m & 63;
    const size_t co_stride = size_t(a.KD) * a.KH * a.KW * a.Cin;
    int it = 0;
    for (int u = int(blockIdx.x); u < a.units; u += int(gridDim.x), ++it) {
      // One thread waits for the accumulators, polling at most every microsecond; the others block
      // on a hardware barrier.  256 threads polling the mbarrier through the whole MMA phase would
      // take shared-memory bandwidth from the tensor core's operand reads.
      if (threadIdx.x == 0) {
        const uint64_t t0 = ptx::globaltimer();
        while (!ptx::mbar_try_wait(acc_full, uint32_t(it) & 1u)) {
          if (*abort_flag) break;
          if (ptx::globaltimer() - t0 > a.wait_ns) {
            *abort_flag = 1;
            atomicOr(a.status, 4u);
            break;
          }
          __nanosleep(1000);
        }
      }
      // The barrier also makes the give-up decision common to all epilogue threads (the TMEM loads
      // below are warp-collective).
      uint32_t stop;
      asm volatile(
          "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, %2, p;\n\t"
          "selp.u32 %0, 1, 0, q;\n\t}"
          : "=r"(stop)
          : "r"(uint32_t(*abort_flag)), "n"(kEpiWarps * 32)
          : "memory");
      if (stop) break;
      ptx::tc_fence_after();
      const Unit un(a, u);
      const int cib = un.pair % a.cb_in, cob0 = (un.pair / a.cb_in) * NCO;
      const int ci = cib * 64 + cil;
      float* const wsc = a.ws + size_t(un.chunk) * a.ws_stride;
      const int nkh = a.ph_nkh[un.ph], nkw = a.ph_nkw[un.ph];
      for (int ob = 0; ob < NCO; ++ob)  // the unit's output blocks, each with its own accumulators
      for (int g = 0; g < (nkh + 1) / 2; ++g) {
        const int ri = 2 * g + i_atom;
        const int kh = ri < nkh ? a.ph_kh[un.ph][ri] : -1;
        for (int cc = h; cc < 4 * nkw; cc += 2) {  // 16-column chunks
          uint32_t v[16];
          ptx::tmem_ld_16(tmem + lane_base + uint32_t(ob) * acc_cols + uint32_t(g * a.KWP * 64 + cc * 16), v);
          ptx::tmem_ld_wait();
          const int kw = a.ph_kw[un.ph][nkw - 1 - (cc >> 2)];
          const int co0 = (cob0 + ob) * 64 + (cc & 3) * 16;
          if (kh >= 0 && ci < a.Cin) {
            float* dst = wsc + (((size_t(co0) * a.KD + un.kd) * a.KH + kh) * a.KW + kw) * a.Cin + ci;
            const int nco = min(16, a.Cout - co0);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              if (c < nco) *dst = __uint_as_float(v[c]);
              dst += co_stride;
            }
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(acc_empty);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, tmem_cols);
}

// ---------------------------------------------------------------- host side

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

// SMs of the current device (the chunk count, and so the workspace size, follow it); 152 when no
// device can be queried.
int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
      sms > 0)
    return sms;
  cudaGetLastError();
  return 152;
}

int gcd(int a, int b) { return b == 0 ? a : gcd(b, a % b); }

struct TcPlan {
  TcArgs a;
  size_t smem;
  int grid;
  int N, H, W, OH, OW;
  int D, OD;  // depth of x and dy when 3-D, else 0 (4-D tensor maps)
};

bool plan(const Problem& p, int sms, TcPlan& pl) {
  if (!(p.bf16 && p.nhwc && p.G == 1)) return false;
  // An H/W stride splits x into stride phases: phase (ah, aw) is the strided view of x rows
  // ah (mod SH), columns aw (mod SW), and the kernel rows kh with kh*DH - PH = ah (mod SH) (columns
  // alike) reach it, DH / gcd(DH, SH) phase rows apart.  Each phase is a unit-stride weight gradient
  // over its own taps; strides up to 4 (the x view's element strides).
  if (p.SH > 4 || p.SW > 4) return false;
  // a real depth axis: any depth stride (a unit's x slice is a fixed function of the dy slice)
  const bool deep = p.D > 1 || p.KD > 1 || p.OD > 1;
  if (p.Cin % 8 != 0 || p.Cout % 8 != 0) return false;  // 16-byte TMA strides
  const int SH = int(p.SH), SW = int(p.SW);
  const int ddr = int(p.DH) / gcd(int(p.DH), SH), ddc = int(p.DW) / gcd(int(p.DW), SW);
  pl = TcPlan{};
  TcArgs& a = pl.a;
  int nph = 0, kwp = 0, gm = 0;
  for (int ah = 0; ah < SH; ++ah)
    for (int aw = 0; aw < SW; ++aw) {
      int khs[4], kws[4], nkh = 0, nkw = 0;
      for (int kh = 0; kh < p.KH; ++kh)
        if (((int(kh * p.DH - p.PH) - ah) % SH + SH) % SH == 0) {
          if (nkh == 4) return false;  // at most two MMA groups of two kernel rows
          khs[nkh++] = kh;
        }
      for (int kw = 0; kw < p.KW; ++kw)
        if (((int(kw * p.DW - p.PW) - aw) % SW + SW) % SW == 0) {
          if (nkw == 4) return false;  // at most four 64-wide kernel-column atoms in N
          kws[nkw++] = kw;
        }
      if (nkh == 0 || nkw == 0) continue;  // no tap reads this phase
      for (int i = 0; i < 4; ++i) {
        a.ph_kh[nph][i] = int8_t(i < nkh ? khs[i] : -1);
        a.ph_kw[nph][i] = int8_t(i < nkw ? kws[i] : -1);
      }
      a.ph_nkh[nph] = int8_t(nkh);
      a.ph_nkw[nph] = int8_t(nkw);
      // virtual (0, 0) of the phase grid: the x position its first kernel row and column read
      a.ph_r0[nph] = int(khs[0] * p.DH - p.PH);
      a.ph_c0[nph] = int(kws[0] * p.DW - p.PW);
      // A and B both MN-major (transpose bits 15 and 16), M = 128, N = 64 per kernel column
      a.ph_idesc[nph] = ptx::idesc_bf16_f32(128, 64 * nkw) | (1u << 15) | (1u << 16);
      kwp = std::max(kwp, nkw);
      gm = std::max(gm, (nkh + 1) / 2);
      ++nph;
    }
  if (nph == 0) return false;
  if ((kwp - 1) * ddc > kFront) return false;        // the dy atoms reach back at most kFront positions
  if (gm * kwp * 64 > 512) return false;             // the accumulators must fit TMEM
  const int64_t P = p.OW + (kwp - 1) * ddc;
  if (P * SW > 256) return false;                    // TMA box extent (a strided view spans SW x P columns)
  if (int64_t(ddr) * P * 128 >= (int64_t(1) << 18)) return false;  // the A atom stride must fit its field
  a.Cin = int(p.Cin); a.Cout = int(p.Cout); a.KH = int(p.KH); a.KW = int(p.KW);
  a.DH = int(p.DH); a.DW = int(p.DW); a.PH = int(p.PH); a.PW = int(p.PW);
  a.SH = SH; a.SW = SW; a.ddr = ddr; a.ddc = ddc;
  a.nph = nph;
  a.KWP = kwp;
  a.KD = deep ? int(p.KD) : 1;
  a.SD = deep ? int(p.SD) : 1;
  a.DD = deep ? int(p.DD) : 1;
  a.PD = deep ? int(p.PD) : 0;
  a.OD = deep ? int(p.OD) : 0;
  a.P = int(P);
  a.RB = 8 / gcd(int(P), 8);
  if (a.RB * SH > 256) return false;  // TMA box extent of the strided x rows
  a.box_bytes = a.RB * a.P * 128;
  a.gm = gm;
  // x rows past a segment's dy rows that its last MMAs read: the second atom of the last group
  // reaches (2*gm - 1)*ddr rows down, the dy atoms (KWP-1)*ddc positions and a 16-position step on.
  const int64_t reach = int64_t(2 * gm - 1) * ddr * P + (kwp - 1) * ddc + 16;
  a.xe = int((reach + a.RB * P - 1) / (a.RB * P));
  a.tail = int((kwp - 1) * ddc + 16);
  // Two output blocks per unit where the output has an even number of them, both accumulator sets fit
  // TMEM, and a segment of at least two row blocks still fits the shared memory (x is then loaded
  // once for both); else one.
  const int cb_out = int((p.Cout + 63) / 64);
  a.seg_blocks = 0;
  for (int nco = (cb_out % 2 == 0 && 2 * gm * kwp * 64 <= 512) ? 2 : 1; nco >= 1 && a.seg_blocks == 0; --nco)
    for (int sb = kMaxBoxes - a.xe; sb >= (nco == 2 ? 2 : 1); --sb) {
      const int64_t xb = int64_t(sb + a.xe) * a.box_bytes;
      const int64_t yb = ((int64_t(kFront + a.tail) * 128 + int64_t(sb) * a.box_bytes) + 1023) & ~int64_t(1023);
      const int64_t total = 1024 + xb + nco * yb + (2 * kMaxBoxes + 4) * 8 + 16;
      if (total <= kSmemLimit) {
        a.seg_blocks = sb;
        a.nco = nco;
        a.x_bytes = int(xb);
        a.y_bytes = int(yb);
        // at least half the SM's shared memory: one CTA per SM, so no second CTA waits for TMEM
        pl.smem = size_t(std::max<int64_t>(total, kSmemLimit / 2 + 1024));
        break;
      }
    }
  if (a.seg_blocks == 0) return false;
  a.bpi = int((p.OH + a.RB - 1) / a.RB);
  const int64_t tb = p.N * (deep ? p.OD : 1) * a.bpi;  // row blocks over every (batch, depth) slice
  if (tb >= (int64_t(1) << 30)) return false;
  a.total_blocks = int(tb);
  a.cb_in = int((p.Cin + 63) / 64);
  a.pairs = a.cb_in * (cb_out / a.nco);
  // one unit per SM: chunks x pairs x kernel-depth taps x stride phases (a chunk is swept once per
  // depth tap and phase)
  a.chunks = int(std::max<int64_t>(1, std::min<int64_t>(tb, sms / (a.pairs * a.KD * nph))));
  const int64_t units = int64_t(a.pairs) * a.chunks * a.KD * nph;
  if (units >= (int64_t(1) << 30)) return false;
  a.units = int(units);
  pl.grid = std::max(1, std::min(a.units, sms));
  pl.N = int(p.N); pl.H = int(p.H); pl.W = int(p.W); pl.OH = int(p.OH); pl.OW = int(p.OW);
  pl.D = deep ? int(p.D) : 0;
  pl.OD = deep ? int(p.OD) : 0;
  return true;
}

// One activation map: (C, W, H, N), or (C, W, H, D, N) when depth > 0; boxes of 64 channels x P x RB
// rows, read every sw-th column and sh-th row (element strides: the box spans sw*P columns, sh*RB rows).
bool encode_one(CUtensorMap* map, const void* base, int C, int W, int H, int depth, int N, int sw, int sh,
                const TcArgs& a) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t rank = depth > 0 ? 5 : 4;
  const cuuint64_t plane = cuuint64_t(H) * W * C * 2;
  cuuint64_t dims[5] = {cuuint64_t(C), cuuint64_t(W), cuuint64_t(H), cuuint64_t(N), 1};
  cuuint64_t strides[4] = {cuuint64_t(C) * 2, cuuint64_t(W) * C * 2, plane, 0};
  if (depth > 0) {
    dims[3] = cuuint64_t(depth);
    dims[4] = cuuint64_t(N);
    strides[3] = plane * cuuint64_t(depth);
  }
  const cuuint32_t box[5] = {64, cuuint32_t(a.P * sw), cuuint32_t(a.RB * sh), 1, 1};
  const cuuint32_t estr[5] = {1, cuuint32_t(sw), cuuint32_t(sh), 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode(const TcPlan& pl, const void* x, const void* dy, TcMaps& maps) {
  const TcArgs& a = pl.a;
  return encode_one(&maps.x, x, a.Cin, pl.W, pl.H, pl.D, pl.N, a.SW, a.SH, a) &&
         encode_one(&maps.dy, dy, a.Cout, pl.OW, pl.OH, pl.OD, pl.N, 1, 1, a);
}

}  // namespace

bool wgrad_tc_supported(const Problem& p) {
  TcPlan pl;
  return plan(p, device_sms(), pl);
}

int64_t wgrad_tc_workspace(const Problem& p) {
  TcPlan pl;
  if (!plan(p, device_sms(), pl)) return 0;
  return ((int64_t(pl.a.chunks) * (p.w_elems() + p.Cout) * 4 + 255) / 256) * 256;
}

bool wgrad_tc_describe(const Problem& p, char* buf, size_t len) {
  TcPlan pl;
  if (!plan(p, device_sms(), pl)) return false;
  const TcArgs& a = pl.a;
  std::snprintf(buf, len,
                "wgrad_tc pairs=%d chunks=%d units=%d grid=%d rows_per_box=%d pitch=%d seg_blocks=%d x_extra=%d "
                "groups=%d n=%d depth_taps=%d phases=%d out_blocks=%d smem=%zu",
                a.pairs, a.chunks, a.units, pl.grid, a.RB, a.P, a.seg_blocks, a.xe, a.gm, 64 * a.KWP, a.KD, a.nph,
                a.nco, pl.smem);
  return true;
}

gbconv_status launch_wgrad_tc(const Problem& p, const void* x, const void* dy, void* dw, float* db, void* ws,
                              const Launch& l) {
  TcPlan pl;
  if (!plan(p, l.num_sms, pl)) return GBCONV_EUNSUPPORTED;
  TcArgs& a = pl.a;
  a.ws = static_cast<float*>(ws);
  a.status = l.status;
  a.wait_ns = l.wait_ns;
  a.ws_stride = int(p.w_elems() + (db ? p.Cout : 0));
  TcMaps maps;
  if (!encode(pl, x, dy, maps)) return GBCONV_ECUDA;
  auto kern = a.gm == 1 ? (a.nco == 2 ? wgrad_tc_kernel<1, 2> : wgrad_tc_kernel<1, 1>)
                        : (a.nco == 2 ? wgrad_tc_kernel<2, 2> : wgrad_tc_kernel<2, 1>);
  static std::atomic<int> raised[4][64];
  const int variant = (a.gm - 1) * 2 + (a.nco - 1);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GBCONV_ECUDA;
  if (!raised[variant][dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit) != cudaSuccess)
      return GBCONV_ECUDA;
    raised[variant][dev].store(1, std::memory_order_release);
  }
  if (launch_kernel(kern, dim3(pl.grid), dim3(kThreads), pl.smem, l.stream, maps, a) != cudaSuccess)
    return GBCONV_ECUDA;
  float* wsf = static_cast<float*>(ws);
  if (db) {
    const gbconv_status s = launch_bgrad_partials(p, dy, a.chunks, wsf, l);
    if (s != GBCONV_OK) return s;
  }
  return launch_wgrad_reduce(p, a.chunks, wsf, dw, db, db != nullptr, l);
}

}  // namespace gbconv
