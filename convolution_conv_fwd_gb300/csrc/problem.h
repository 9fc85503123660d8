// Resolved convolution geometry shared by the host dispatcher and the kernel
// launchers.  A 1-D convolution is carried as a 2-D one with H = KH = 1, and
// 1-D and 2-D ones as 3-D ones with depth 1 (D = KD = SD = DD = OD = 1, PD = 0).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <utility>

#include "../../include/gbconv.h"

namespace gbconv {

struct Problem {
  int64_t N, Cin, Cout, G;
  int64_t H, W, KH, KW, SH, SW, PH, PW, DH, DW;
  int64_t PHe, PWe;  // end-side padding (PH, PW are the begin side); equal to PH, PW when symmetric
  int64_t D, KD, SD, PD, PDe, DD;  // depth axis
  int64_t OH, OW, OD;
  bool nhwc;   // activations channels-last
  bool ohwi;   // weight [C_out, KH, KW, C_in/G]
  bool bf16;   // element type bf16 (else f32)
  int64_t cpg() const { return Cin / G; }   // input channels per group
  int64_t opg() const { return Cout / G; }  // output channels per group
  int64_t x_elems() const { return N * Cin * D * H * W; }
  int64_t y_elems() const { return N * Cout * OD * OH * OW; }
  int64_t w_elems() const { return Cout * cpg() * KD * KH * KW; }
  int elem_bytes() const { return bf16 ? 2 : 4; }
  bool sym_pad() const { return PHe == PH && PWe == PW; }
  // The depth axis does nothing but repeat a 2-D convolution per depth slice (kernel depth 1, unit
  // stride, no depth padding): channels-last, the 3-D tensors are then 2-D ones with N*D images.
  bool depth_trivial() const { return KD == 1 && SD == 1 && PD == 0 && PDe == 0; }
  Problem fold_depth() const {
    Problem q = *this;
    q.N = N * D;
    q.D = q.OD = 1;
    q.DD = 1;
    return q;
  }
};

// Fills `p` from `d` and checks it the way oarust's geometry resolvers do:
// nonzero extents, stride, dilation and groups, channels divisible by groups,
// the effective kernel fitting the padded input.  Element counts must fit the
// kernels' 32-bit indexing.  Returns GBCONV_OK, GBCONV_EINVAL or GBCONV_EUNSUPPORTED.
gbconv_status resolve(const gbconv_desc* d, Problem* p);

// ---- launchers (each enqueues exactly one kernel) ----
struct Launch {
  void* stream;
  unsigned int* status;  // device status word for bounded-wait failures
  int num_sms;
  uint64_t wait_ns;      // bound of the kernels' barrier waits (gbconv_set_wait_limit_ns)
};

// The launch context of the current device for `stream` (false if a CUDA query failed).
bool launch_context(Launch* l, void* stream);

gbconv_status launch_direct_fwd(const Problem& p, const void* x, const void* w, const float* bias, void* y,
                                const Launch& l);
// The dgrad launchers add an optional fp32 bias [C_in] after the gather sum (transposed convolution).
gbconv_status launch_direct_dgrad(const Problem& p, const void* dy, const void* w, const float* bias, void* dx,
                                  const Launch& l);
gbconv_status launch_pack_weight(const Problem& p, const void* w_oihw, void* w_ohwi, const Launch& l);

bool depthwise_supported(const Problem& p);
gbconv_status launch_depthwise_fwd(const Problem& p, const void* x, const void* w, const float* bias, void* y,
                                   const Launch& l);
bool depthwise_dgrad_supported(const Problem& p);
gbconv_status launch_depthwise_dgrad(const Problem& p, const void* dy, const void* w, const float* bias, void* dx,
                                     const Launch& l);

// Small groups (1 < G < C, C_in/G = C_out/G in {2, 4, 8}): tiled forward and stride-1 input
// gradient on CUDA cores, gather input gradient at other strides.
bool smallgroup_supported(const Problem& p);
bool smallgroup_dgrad_supported(const Problem& p);
bool smallgroup_describe(const Problem& p, bool dgrad, char* buf, size_t len);
gbconv_status launch_smallgroup_fwd(const Problem& p, const void* x, const void* w, const float* bias, void* y,
                                    const Launch& l);
gbconv_status launch_smallgroup_dgrad(const Problem& p, const void* dy, const void* w, const float* bias, void* dx,
                                      const Launch& l);

bool pointwise_supported(const Problem& p);
gbconv_status launch_pointwise_fwd(const Problem& p, const void* x, const void* w, const float* bias, void* y,
                                   const Launch& l);

bool implicit_fwd_supported(const Problem& p);
bool implicit_dgrad_supported(const Problem& p);
// Writes the implicit-GEMM plan for p (forward or dgrad) into buf; false if p has none.
bool implicit_describe(const Problem& p, bool dgrad, char* buf, size_t len);
gbconv_status launch_implicit_fwd(const Problem& p, const void* x, const void* w, const float* bias, void* y,
                                  const Launch& l);
gbconv_status launch_implicit_dgrad(const Problem& p, const void* dy, const void* w, const float* bias, void* dx,
                                    const Launch& l);

// Weight gradient.  Every path stores fp32 partial sums per position chunk in the caller's workspace,
// [chunk][element] with elements in OHWI order and then C_out bias-gradient entries, and ends with
// launch_wgrad_reduce, which adds the chunks in a fixed order and writes dw (desc layout and dtype) and db.
int64_t direct_wgrad_workspace(const Problem& p);
gbconv_status launch_direct_wgrad(const Problem& p, const void* x, const void* dy, void* dw, float* db, void* ws,
                                  const Launch& l);
gbconv_status launch_wgrad_reduce(const Problem& p, int S, const float* ws, void* dw, float* db, bool want_db,
                                  const Launch& l);
// Bias-gradient partial sums only, over S equal position chunks, into ws [S][E + C_out] entries E..
gbconv_status launch_bgrad_partials(const Problem& p, const void* dy, int S, float* ws, const Launch& l);
bool wgrad_tc_supported(const Problem& p);
int64_t wgrad_tc_workspace(const Problem& p);
gbconv_status launch_wgrad_tc(const Problem& p, const void* x, const void* dy, void* dw, float* db, void* ws,
                              const Launch& l);
bool wgrad_tc_describe(const Problem& p, char* buf, size_t len);

// Counts one enqueued kernel.
void note_launch();

// Enqueues `kern` with programmatic stream serialization: the launch may begin
// (prologue: barrier init, TMEM allocation, table staging) while the previous
// kernel on the stream drains.  Every kernel of this library calls
// ptx::grid_dep_wait() before its first global-memory access, so results are
// the same as with plain stream order.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, void* stream,
                          Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
  note_launch();
  return e;
}

}  // namespace gbconv
