// Pointwise (1x1, unit stride, no padding, no dilation, one group) forward as
// a plain TMA-fed GEMM on tcgen05.  burn-cubecl `src/kernel/conv/im2col.rs`
// (doc of `check_pointwise`) states the identity used: every output pixel
// reads only the input pixel under it, so im2col is the identity and the
// convolution is the per-pixel matmul y[(n,h,w), co] = sum_ci x[(n,h,w), ci] *
// w[co, ci].  NHWC x is already the K-major [M = N*H*W, K = C_in] matrix and
// the [C_out, C_in] weight is already the K-major B operand, so both are read
// by TMA straight from the caller's tensors (burn-cubecl's `reshape_input` /
// `reshape_weight` reach the same views by metadata alone).
//
// Roles: warps 0-3 epilogue (TMEM -> bias -> bf16 -> NHWC stores), warp 4
// TMEM allocation + MMA issue (lane 0), warp 5 TMA producer (lane 0).  Tiles
// are 128 rows of M; the weight stays resident in shared memory; A tiles
// stream through a ring of 128-byte-swizzled stages; two TMEM accumulators
// let the epilogue of one tile overlap the MMAs of the next.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <mutex>

#include "problem.h"
#include "ptx.cuh"

namespace gbconv {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kThreads = 6 * 32;
constexpr int kBM = 128, kBK = 64;
constexpr int kATileBytes = kBM * kBK * 2;  // 16 KB
constexpr int kSmemLimit = 227 * 1024;
constexpr int kMaxStages = 8;

struct PwArgs {
  const float* bias;
  bf16* out;
  unsigned int* status;
  uint64_t wait_ns;   // bound of every barrier wait (the host sets it; 2 s by default)
  int M, Cout, K;
  int kb_count, m_tiles, stages;
};

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    pointwise_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                          const __grid_constant__ PwArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 128-byte swizzled tiles must start on 1024-byte boundaries.
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kBTileBytes = BN * kBK * 2;
  constexpr uint32_t kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;
  constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(128, BN);

  uint8_t* b_base = smem;                                      // kb_count tiles of [BN][64] bf16
  uint8_t* a_base = b_base + size_t(a.kb_count) * kBTileBytes;  // stages x [128][64] bf16
  // epilogue staging: 4 warps x 32 rows x (BN*2 + 16) bytes (padded rows: conflict-free 16-byte stores)
  constexpr int kPitch = BN * 2 + 16;
  uint8_t* stage_base = a_base + size_t(a.stages) * kATileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(stage_base + 128 * kPitch);
  uint64_t* full = bars;
  uint64_t* empty = full + a.stages;
  uint64_t* tfull = empty + a.stages;
  uint64_t* tempty = tfull + 2;
  uint64_t* bfull = tempty + 2;
  uint64_t* fin = bfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fin + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < a.stages; ++i) { ptx::mbar_init(full + i, 1); ptx::mbar_init(empty + i, 1); }
    for (int i = 0; i < 2; ++i) { ptx::mbar_init(tfull + i, 1); ptx::mbar_init(tempty + i, 128); }
    ptx::mbar_init(bfull, 1);
    ptx::mbar_init(fin, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 4) {
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

  if (warp == 5) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tmap_a);
      ptx::prefetch_tmap(&tmap_b);
      // The resident weights are issued right after the first activation tile: that tile comes from
      // HBM and takes longest, the weights are shared by every CTA and mostly come from L2.
      auto load_weights = [&]() {
        ptx::mbar_arrive_expect_tx(bfull, uint32_t(a.kb_count) * kBTileBytes);
        for (int kb = 0; kb < a.kb_count; ++kb)
          ptx::tma_load_2d(ptx::smem_addr(b_base + size_t(kb) * kBTileBytes), &tmap_b, bfull, kb * kBK, 0);
      };
      int st = 0, issued = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < a.m_tiles; tile += gridDim.x) {
        for (int kb = 0; kb < a.kb_count; ++kb) {
          if (!(ok = ptx::mbar_wait(empty + st, ph ^ 1, abort_flag, a.status, 8u, a.wait_ns))) break;
          ptx::mbar_arrive_expect_tx(full + st, kATileBytes);
          ptx::tma_load_2d(ptx::smem_addr(a_base + size_t(st) * kATileBytes), &tmap_a, full + st, kb * kBK,
                           tile * kBM);
          if (issued++ == 0) load_weights();
          if (++st == a.stages) { st = 0; ph ^= 1; }
        }
      }
      if (issued == 0) load_weights();  // a CTA without tiles still completes the weight barrier
      // Drain: copies still in flight write this CTA's shared memory and must land before it leaves
      // (after an abort the MMA thread no longer consumes them).  Load k completes phase
      // k / stages of barrier k % stages; the resident weights complete bfull's first phase.
      for (int k = max(0, issued - a.stages); k < issued; ++k)
        ptx::mbar_wait_drain(full + k % a.stages, uint32_t((k / a.stages) & 1));
      ptx::mbar_wait_drain(bfull, 0);
    }
    __syncwarp();
  } else if (warp == 4) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = ptx::mbar_wait(bfull, 0, abort_flag, a.status, 8u, a.wait_ns);
      int st = 0, it = 0;
      uint32_t ph = 0;
      for (int tile = blockIdx.x; ok && tile < a.m_tiles; tile += gridDim.x, ++it) {
        const int buf = it & 1;
        if (!(ok = ptx::mbar_wait(tempty + buf, ((it >> 1) & 1) ^ 1, abort_flag, a.status, 8u, a.wait_ns))) break;
        ptx::tc_fence_after();
        const uint32_t acc = tmem + uint32_t(buf * BN);
        for (int kb = 0; kb < a.kb_count; ++kb) {
          if (!(ok = ptx::mbar_wait(full + st, ph, abort_flag, a.status, 8u, a.wait_ns))) break;
          ptx::tc_fence_after();
          const uint32_t a_addr = ptx::smem_addr(a_base + size_t(st) * kATileBytes);
          const uint32_t b_addr = ptx::smem_addr(b_base + size_t(kb) * kBTileBytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            ptx::mma_bf16(acc, ptx::desc_kmajor_sw128(a_addr + k * 32), ptx::desc_kmajor_sw128(b_addr + k * 32),
                          kIdesc, (kb | k) != 0);
          ptx::mma_commit(empty + st);
          if (++st == a.stages) { st = 0; ph ^= 1; }
        }
        ptx::mma_commit(tfull + buf);
      }
      ptx::mma_commit(fin);
      // every MMA issued so far completes before TMEM is freed, abort or not
      ptx::mbar_wait_drain(fin, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    int it = 0;
    const uint32_t lane_base = uint32_t(warp * 32) << 16;
    for (int tile = blockIdx.x; tile < a.m_tiles; tile += gridDim.x, ++it) {
      const int buf = it & 1;
      const bool got = ptx::mbar_wait(tfull + buf, (it >> 1) & 1, abort_flag, a.status, 8u, a.wait_ns);
      // the TMEM loads below are warp-collective: the warp leaves together if any lane gave up
      if (__any_sync(0xffffffffu, !got)) break;
      ptx::tc_fence_after();
      // TMEM -> (+ bias) -> bf16 -> this warp's staging rows, then whole-row coalesced stores:
      // consecutive lanes write consecutive 16-byte pieces of the same output pixel.
      const uint32_t stage_s = ptx::smem_addr(stage_base + warp * 32 * kPitch);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        ptx::tmem_ld_32(tmem + lane_base + uint32_t(buf * BN + c * 32), v);
        ptx::tmem_ld_wait();
        float f[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
        if (a.bias) {
#pragma unroll
          for (int j = 0; j < 32; ++j) f[j] += __ldg(a.bias + c * 32 + j);
        }
        const uint32_t d = stage_s + uint32_t(lane * kPitch + c * 64);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(d + q * 16),
                       "r"(ptx::pack_bf16x2(f[8 * q], f[8 * q + 1])), "r"(ptx::pack_bf16x2(f[8 * q + 2], f[8 * q + 3])),
                       "r"(ptx::pack_bf16x2(f[8 * q + 4], f[8 * q + 5])), "r"(ptx::pack_bf16x2(f[8 * q + 6], f[8 * q + 7]))
                       : "memory");
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(tempty + buf);  // TMEM is free once read; the stores below use the staging copy
      __syncwarp();
      constexpr int kParts = BN / 8;         // 16-byte pieces per row
      constexpr int kRowStep = 32 / kParts;  // rows per warp pass
      const int part = lane % kParts;
      const int row0 = tile * kBM + warp * 32;
      // All staged pieces are read first, then stored (the __syncwarp above orders the loads
      // after this warp's staging writes).
      constexpr int kIters = 32 / kRowStep;
      uint4 val[kIters];
      asm volatile("" ::: "memory");  // keeps the loads below after the __syncwarp
#pragma unroll
      for (int i = 0; i < kIters; ++i)
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(val[i].x), "=r"(val[i].y), "=r"(val[i].z), "=r"(val[i].w)
                     : "r"(stage_s + uint32_t((lane / kParts + i * kRowStep) * kPitch + part * 16)));
#pragma unroll
      for (int i = 0; i < kIters; ++i) {
        const int r = lane / kParts + i * kRowStep;
        if (row0 + r < a.M) *reinterpret_cast<uint4*>(a.out + size_t(row0 + r) * a.Cout + part * 8) = val[i];
      }
      __syncwarp();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 4) ptx::tmem_dealloc(tmem, kTmemCols);
}

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

// Row-major [rows, cols] bf16 matrix, box [box_rows, 64 columns], 128-byte swizzle, zero fill out of bounds.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {uint32_t(kBK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int pick_bn(int64_t cout) {
  for (int bn : {256, 128, 64, 32})
    if (cout == bn) return bn;
  return 0;
}

size_t smem_for(int bn, int kb_count, int stages) {
  return size_t(kb_count) * bn * kBK * 2 + size_t(stages) * kATileBytes + 1024 + 8 * (2 * kMaxStages + 8) +
         128 * size_t(bn * 2 + 16);
}

int stages_for(int bn, int kb_count) {
  const size_t fixed = smem_for(bn, kb_count, 0);
  if (fixed >= size_t(kSmemLimit)) return 0;
  const int s = int((size_t(kSmemLimit) - fixed) / kATileBytes);
  return std::min(s, kMaxStages);
}

// Two CTAs per SM, each with a 3-stage ring, when both fit one SM's shared memory: two CTAs streaming
// side by side move more bytes per SM than one with a deeper ring (the 1x1 workload: 12.86 us against
// 13.70 with 8 stages on one CTA per SM).
constexpr int kPairStages = 3;
bool two_per_sm(int bn, int kb_count) { return 2 * smem_for(bn, kb_count, kPairStages) <= size_t(kSmemLimit); }

template <int BN>
gbconv_status run(const CUtensorMap& ta, const CUtensorMap& tb, const PwArgs& a, int grid, const Launch& l) {
  const size_t smem = smem_for(BN, a.kb_count, a.stages);
  auto kern = pointwise_gemm_kernel<BN>;
  // The shared-memory opt-in is a per-device function attribute: set it once per device and size.
  static std::atomic<uint64_t> done[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GBCONV_ECUDA;
  if (done[dev].load(std::memory_order_acquire) < uint64_t(smem)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
      return GBCONV_ECUDA;
    done[dev].store(uint64_t(smem), std::memory_order_release);
  }
  return launch_kernel(kern, dim3(grid), dim3(kThreads), smem, l.stream, ta, tb, a) == cudaSuccess ? GBCONV_OK
                                                                                                   : GBCONV_ECUDA;
}

}  // namespace

bool pointwise_supported(const Problem& p) {
  if (!(p.bf16 && p.nhwc && p.G == 1 && p.KH == 1 && p.KW == 1 && p.SH == 1 && p.SW == 1 && p.PH == 0 && p.PW == 0 &&
        p.PHe == 0 && p.PWe == 0))
    return false;
  if (p.Cin % 8 != 0) return false;  // TMA row pitch must be a multiple of 16 bytes
  const int bn = pick_bn(p.Cout);
  if (!bn) return false;
  const int kb_count = int((p.Cin + kBK - 1) / kBK);
  return stages_for(bn, kb_count) >= 3;
}

gbconv_status launch_pointwise_fwd(const Problem& p, const void* x, const void* w, const float* bias, void* y,
                                   const Launch& l) {
  if (!pointwise_supported(p)) return GBCONV_EUNSUPPORTED;
  PwArgs a;
  a.bias = bias;
  a.out = static_cast<bf16*>(y);
  a.status = l.status;
  a.wait_ns = l.wait_ns;
  a.M = int(p.N * p.H * p.W);
  a.Cout = int(p.Cout);
  a.K = int(p.Cin);
  a.kb_count = int((p.Cin + kBK - 1) / kBK);
  a.m_tiles = (a.M + kBM - 1) / kBM;
  const int bn = pick_bn(p.Cout);
  const int per_sm = two_per_sm(bn, a.kb_count) ? 2 : 1;
  a.stages = per_sm == 2 ? kPairStages : stages_for(bn, a.kb_count);
  CUtensorMap ta, tb;
  if (!make_map(&ta, x, uint64_t(a.M), uint64_t(a.K), kBM)) return GBCONV_ECUDA;
  if (!make_map(&tb, w, uint64_t(p.Cout), uint64_t(a.K), uint32_t(bn))) return GBCONV_ECUDA;
  // The fewest rounds the CTA slots allow, over as many CTAs as that many rounds needs: every CTA then
  // takes the same number of tiles (give or take one in the last round) instead of a last round in
  // which a few CTAs work while the rest are done (784 tiles on 2 x 152 slots: 262 CTAs of 3 tiles;
  // with one CTA per SM it was 131 CTAs of 6, not 152 of which 24 take a 6th).
  const int slots = std::max(1, per_sm * l.num_sms);
  const int rounds = (a.m_tiles + slots - 1) / slots;
  const int grid = std::max(1, std::min(a.m_tiles, (a.m_tiles + rounds - 1) / std::max(1, rounds)));
  switch (bn) {
    case 256: return run<256>(ta, tb, a, grid, l);
    case 128: return run<128>(ta, tb, a, grid, l);
    case 64: return run<64>(ta, tb, a, grid, l);
    default: return run<32>(ta, tb, a, grid, l);
  }
}

}  // namespace gbconv
