// The C ABI: argument checks, shape resolution, choice of kernel family and
// the device status word.  Nothing here allocates device memory.
#include <cstdio>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <mutex>

#include "problem.h"

namespace gbconv {

namespace {

// Bounded-wait failures of any kernel of this library on this device set bits here.
__device__ unsigned int g_status_word;

std::atomic<uint64_t> g_launches{0};

constexpr int64_t kDefaultWaitNs = 2000000000;  // 2 s
std::atomic<int64_t> g_wait_ns{kDefaultWaitNs};

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
unsigned int* g_status_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

bool device_context(Launch* l, void* stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return false;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    g_status_ptr[dev] = static_cast<unsigned int*>(p);
    g_num_sms[dev] = sms;
  }
  l->stream = stream;
  l->status = g_status_ptr[dev];
  l->num_sms = g_num_sms[dev];
  l->wait_ns = uint64_t(g_wait_ns.load(std::memory_order_relaxed));
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int64_t kMax32 = 2147483647;

}  // namespace

bool launch_context(Launch* l, void* stream) { return device_context(l, stream); }

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

gbconv_status resolve(const gbconv_desc* d, Problem* p) {
  if (!d || !p) return GBCONV_EINVAL;
  if (d->spatial_dims < 1 || d->spatial_dims > 3) return GBCONV_EINVAL;
  if (d->layout != GBCONV_NCHW && d->layout != GBCONV_NHWC) return GBCONV_EINVAL;
  if (d->wlayout != GBCONV_W_OIHW && d->wlayout != GBCONV_W_OHWI) return GBCONV_EINVAL;
  if (d->dtype != GBCONV_F32 && d->dtype != GBCONV_BF16) return GBCONV_EINVAL;
  if (d->pad_mode != GBCONV_PAD_SYMMETRIC && d->pad_mode != GBCONV_PAD_BEGIN_END) return GBCONV_EINVAL;
  const bool be = d->pad_mode == GBCONV_PAD_BEGIN_END;
  Problem q{};
  q.N = d->n;
  q.Cin = d->c_in;
  q.Cout = d->c_out;
  q.G = d->groups;
  // axis i of the descriptor -> (extent, kernel, stride, pad, pad_end, dilation)
  auto axis = [&](int i, int64_t& in, int64_t& k, int64_t& s, int64_t& p, int64_t& pe, int64_t& dl) {
    in = d->in[i]; k = d->k[i]; s = d->stride[i]; p = d->pad[i]; dl = d->dil[i];
    pe = be ? d->pad_end[i] : p;
  };
  q.D = 1; q.KD = 1; q.SD = 1; q.PD = 0; q.PDe = 0; q.DD = 1;
  if (d->spatial_dims == 1) {  // the length axis is carried as the width
    q.H = 1; q.KH = 1; q.SH = 1; q.PH = 0; q.PHe = 0; q.DH = 1;
    axis(0, q.W, q.KW, q.SW, q.PW, q.PWe, q.DW);
  } else if (d->spatial_dims == 2) {
    axis(0, q.H, q.KH, q.SH, q.PH, q.PHe, q.DH);
    axis(1, q.W, q.KW, q.SW, q.PW, q.PWe, q.DW);
  } else {
    axis(0, q.D, q.KD, q.SD, q.PD, q.PDe, q.DD);
    axis(1, q.H, q.KH, q.SH, q.PH, q.PHe, q.DH);
    axis(2, q.W, q.KW, q.SW, q.PW, q.PWe, q.DW);
  }
  if (q.N <= 0 || q.Cin <= 0 || q.Cout <= 0 || q.G <= 0) return GBCONV_EINVAL;
  if (q.H <= 0 || q.W <= 0 || q.KH <= 0 || q.KW <= 0 || q.D <= 0 || q.KD <= 0) return GBCONV_EINVAL;
  if (q.SH <= 0 || q.SW <= 0 || q.DH <= 0 || q.DW <= 0 || q.PH < 0 || q.PW < 0 || q.PHe < 0 || q.PWe < 0)
    return GBCONV_EINVAL;
  if (q.SD <= 0 || q.DD <= 0 || q.PD < 0 || q.PDe < 0) return GBCONV_EINVAL;
  if (q.Cin % q.G != 0 || q.Cout % q.G != 0) return GBCONV_EINVAL;
  // Keep every intermediate well inside int64 before multiplying.
  const int64_t lim = int64_t(1) << 31;
  if (q.N >= lim || q.Cin >= lim || q.Cout >= lim || q.H >= lim || q.W >= lim || q.KH >= lim || q.KW >= lim ||
      q.SH >= lim || q.SW >= lim || q.PH >= lim || q.PW >= lim || q.PHe >= lim || q.PWe >= lim || q.DH >= lim ||
      q.DW >= lim || q.D >= lim || q.KD >= lim || q.SD >= lim || q.PD >= lim || q.PDe >= lim || q.DD >= lim)
    return GBCONV_EUNSUPPORTED;
  const int64_t effh = (q.KH - 1) * q.DH + 1, effw = (q.KW - 1) * q.DW + 1;
  const int64_t effd = (q.KD - 1) * q.DD + 1;
  if (q.H + q.PH + q.PHe < effh || q.W + q.PW + q.PWe < effw || q.D + q.PD + q.PDe < effd) return GBCONV_EINVAL;
  q.OH = (q.H + q.PH + q.PHe - effh) / q.SH + 1;
  q.OW = (q.W + q.PW + q.PWe - effw) / q.SW + 1;
  q.OD = (q.D + q.PD + q.PDe - effd) / q.SD + 1;
  q.nhwc = d->layout == GBCONV_NHWC;
  q.ohwi = d->wlayout == GBCONV_W_OHWI;
  q.bf16 = d->dtype == GBCONV_BF16;
  // 32-bit device indexing: element counts and the farthest coordinate read.
  auto fits = [](int64_t a, int64_t b, int64_t c, int64_t e, int64_t f) -> bool {
    __int128 v = static_cast<__int128>(a) * b * c * e * f;
    return v <= kMax32;
  };
  if (!fits(q.N, q.Cin, q.D, q.H, q.W) || !fits(q.N, q.Cout, q.OD, q.OH, q.OW) ||
      !fits(q.Cout, q.cpg(), q.KD, q.KH, q.KW))
    return GBCONV_EUNSUPPORTED;
  if ((q.OH - 1) * q.SH + (q.KH - 1) * q.DH > kMax32 || (q.OW - 1) * q.SW + (q.KW - 1) * q.DW > kMax32 ||
      (q.OD - 1) * q.SD + (q.KD - 1) * q.DD > kMax32)
    return GBCONV_EUNSUPPORTED;
  *p = q;
  return GBCONV_OK;
}

namespace {

// The 2-D view the tensor-core and depthwise families work on: 1-D and 2-D shapes as they are, and
// channels-last 3-D shapes whose depth axis only repeats the 2-D convolution (kernel depth 1, unit
// stride, no depth padding) with the depth folded into the batch.  false for every other 3-D shape,
// which the generic kernels serve.
bool planar(const Problem& p, Problem* q) {
  if (!p.depth_trivial()) return false;
  if (p.D == 1) {
    *q = p;
    return true;
  }
  if (!p.nhwc) return false;
  *q = p.fold_depth();
  return true;
}

int32_t select_fwd(const Problem& p, bool aligned) {
  Problem q;
  if (!aligned) return GBCONV_K_DIRECT;
  // a 3-D forward with a real depth axis: the implicit GEMM reads its kernel-depth taps as sources
  if (!planar(p, &q)) return implicit_fwd_supported(p) ? GBCONV_K_IMPLICIT : GBCONV_K_DIRECT;
  if (depthwise_supported(q)) return GBCONV_K_DEPTHWISE;
  if (smallgroup_supported(q)) return GBCONV_K_SMALLGROUP;
  if (pointwise_supported(q)) return GBCONV_K_POINTWISE;
  if (implicit_fwd_supported(q)) return GBCONV_K_IMPLICIT;
  return GBCONV_K_DIRECT;
}

int32_t select_dgrad(const Problem& p, bool aligned) {
  Problem q;
  if (!aligned) return GBCONV_K_DIRECT_DGRAD;
  // a 3-D gradient with a real depth axis: depth phases, whose kernel-depth taps are dy sources
  if (!planar(p, &q)) return implicit_dgrad_supported(p) ? GBCONV_K_DGRAD : GBCONV_K_DIRECT_DGRAD;
  if (depthwise_dgrad_supported(q)) return GBCONV_K_DEPTHWISE_DGRAD;
  if (smallgroup_dgrad_supported(q)) return GBCONV_K_SMALLGROUP_DGRAD;
  if (implicit_dgrad_supported(q)) return GBCONV_K_DGRAD;
  return GBCONV_K_DIRECT_DGRAD;
}

int32_t select_wgrad(const Problem& p, bool aligned) {
  Problem q;
  if (!aligned) return GBCONV_K_DIRECT_WGRAD;
  // a 3-D weight gradient with a real depth axis: one kernel-depth tap per unit
  if (!planar(p, &q)) return wgrad_tc_supported(p) ? GBCONV_K_WGRAD : GBCONV_K_DIRECT_WGRAD;
  return wgrad_tc_supported(q) ? GBCONV_K_WGRAD : GBCONV_K_DIRECT_WGRAD;
}

// The problem a family's launcher takes: the planar view for the 2-D families, the full shape for
// the generic kernels.
Problem launch_view(const Problem& p, int32_t family) {
  Problem q;
  if (family == GBCONV_K_DIRECT || family == GBCONV_K_DIRECT_DGRAD || family == GBCONV_K_DIRECT_WGRAD ||
      !planar(p, &q))
    return p;
  return q;
}

int32_t select_op(const Problem& p, int32_t op, bool aligned) {
  if (op == GBCONV_OP_FWD) return select_fwd(p, aligned);
  if (op == GBCONV_OP_BWD_DATA) return select_dgrad(p, aligned);
  return select_wgrad(p, aligned);
}

bool valid_op(int32_t op) { return op == GBCONV_OP_FWD || op == GBCONV_OP_BWD_DATA || op == GBCONV_OP_BWD_FILTER; }

// The gather dgrad, plus the transposed convolution's bias when one is given.
gbconv_status bwd_data(const gbconv_desc* desc, const void* dy, const void* w, const float* bias, void* dx,
                       void* stream) {
  Problem p;
  gbconv_status s = resolve(desc, &p);
  if (s != GBCONV_OK) return s;
  if (!dy || !w || !dx) return GBCONV_EINVAL;
  Launch l;
  if (!device_context(&l, stream)) return GBCONV_ECUDA;
  const bool aligned = aligned16(dy) && aligned16(w) && aligned16(dx);
  const int32_t k = select_dgrad(p, aligned);
  const Problem q = launch_view(p, k);
  switch (k) {
    case GBCONV_K_DGRAD: return launch_implicit_dgrad(q, dy, w, bias, dx, l);
    case GBCONV_K_DEPTHWISE_DGRAD: return launch_depthwise_dgrad(q, dy, w, bias, dx, l);
    case GBCONV_K_SMALLGROUP_DGRAD: return launch_smallgroup_dgrad(q, dy, w, bias, dx, l);
    default: return launch_direct_dgrad(p, dy, w, bias, dx, l);
  }
}

}  // namespace
}  // namespace gbconv

using namespace gbconv;

extern "C" {

gbconv_status gbconv_out_shape(const gbconv_desc* desc, int64_t out[3]) {
  if (!out) return GBCONV_EINVAL;
  Problem p;
  gbconv_status s = resolve(desc, &p);
  if (s != GBCONV_OK) return s;
  if (desc->spatial_dims == 1) {
    out[0] = p.OW;
    out[1] = 1;
    out[2] = 1;
  } else if (desc->spatial_dims == 2) {
    out[0] = p.OH;
    out[1] = p.OW;
    out[2] = 1;
  } else {
    out[0] = p.OD;
    out[1] = p.OH;
    out[2] = p.OW;
  }
  return GBCONV_OK;
}

gbconv_status gbconv_select(const gbconv_desc* desc, int32_t op, int32_t* kernel) {
  if (!kernel || !valid_op(op)) return GBCONV_EINVAL;
  Problem p;
  gbconv_status s = resolve(desc, &p);
  if (s != GBCONV_OK) return s;
  *kernel = select_op(p, op, true);
  return GBCONV_OK;
}

gbconv_status gbconv_describe(const gbconv_desc* desc, int32_t op, char* buf, int64_t len) {
  if (!buf || len < 1 || !valid_op(op)) return GBCONV_EINVAL;
  Problem p;
  gbconv_status s = resolve(desc, &p);
  if (s != GBCONV_OK) return s;
  const int32_t k = select_op(p, op, true);
  static const char* const names[] = {"direct",       "depthwise",    "pointwise",  "implicit",
                                      "dgrad",        "direct_dgrad", "depthwise_dgrad", "direct_wgrad",
                                      "wgrad",        "smallgroup",   "smallgroup_dgrad"};
  const Problem q = launch_view(p, k);
  if ((k == GBCONV_K_IMPLICIT || k == GBCONV_K_DGRAD) &&
      implicit_describe(q, k == GBCONV_K_DGRAD, buf, size_t(len)))
    return GBCONV_OK;
  if (k == GBCONV_K_WGRAD && wgrad_tc_describe(q, buf, size_t(len))) return GBCONV_OK;
  if ((k == GBCONV_K_SMALLGROUP || k == GBCONV_K_SMALLGROUP_DGRAD) &&
      smallgroup_describe(q, k == GBCONV_K_SMALLGROUP_DGRAD, buf, size_t(len)))
    return GBCONV_OK;
  std::snprintf(buf, size_t(len), "%s", (k >= 0 && k <= GBCONV_K_SMALLGROUP_DGRAD) ? names[k] : "unknown");
  return GBCONV_OK;
}

gbconv_status gbconv_fwd(const gbconv_desc* desc, const void* x, const void* w, const float* bias, void* y,
                         void* stream) {
  Problem p;
  gbconv_status s = resolve(desc, &p);
  if (s != GBCONV_OK) return s;
  if (!x || !w || !y) return GBCONV_EINVAL;
  Launch l;
  if (!device_context(&l, stream)) return GBCONV_ECUDA;
  const bool aligned = aligned16(x) && aligned16(w) && aligned16(y);
  const int32_t k = select_fwd(p, aligned);
  const Problem q = launch_view(p, k);
  switch (k) {
    case GBCONV_K_DEPTHWISE: return launch_depthwise_fwd(q, x, w, bias, y, l);
    case GBCONV_K_SMALLGROUP: return launch_smallgroup_fwd(q, x, w, bias, y, l);
    case GBCONV_K_POINTWISE: return launch_pointwise_fwd(q, x, w, bias, y, l);
    case GBCONV_K_IMPLICIT: return launch_implicit_fwd(q, x, w, bias, y, l);
    default: return launch_direct_fwd(p, x, w, bias, y, l);
  }
}

gbconv_status gbconv_bwd_filter_workspace(const gbconv_desc* desc, int64_t* bytes) {
  if (!bytes) return GBCONV_EINVAL;
  Problem p;
  gbconv_status s = resolve(desc, &p);
  if (s != GBCONV_OK) return s;
  // Enough for whichever path a call takes (the tensor-core path needs aligned pointers).
  int64_t b = direct_wgrad_workspace(p);
  Problem q;
  const Problem& v = planar(p, &q) ? q : p;  // the view the tensor-core path would take
  if (wgrad_tc_supported(v)) b = std::max(b, wgrad_tc_workspace(v));
  *bytes = b;
  return GBCONV_OK;
}

gbconv_status gbconv_bwd_filter(const gbconv_desc* desc, const void* x, const void* dy, void* dw, float* db,
                                void* workspace, int64_t workspace_bytes, void* stream) {
  Problem p;
  gbconv_status s = resolve(desc, &p);
  if (s != GBCONV_OK) return s;
  if (!x || !dy || !dw) return GBCONV_EINVAL;
  const bool aligned = aligned16(x) && aligned16(dy) && aligned16(dw) && aligned16(workspace);
  const int32_t k = select_wgrad(p, aligned);
  const Problem q = launch_view(p, k);
  const int64_t need = k == GBCONV_K_WGRAD ? wgrad_tc_workspace(q) : direct_wgrad_workspace(p);
  if (workspace_bytes < need || (need > 0 && !workspace) || !aligned16(workspace)) return GBCONV_EINVAL;
  Launch l;
  if (!device_context(&l, stream)) return GBCONV_ECUDA;
  if (k == GBCONV_K_WGRAD) return launch_wgrad_tc(q, x, dy, dw, db, workspace, l);
  return launch_direct_wgrad(p, x, dy, dw, db, workspace, l);
}

gbconv_status gbconv_bwd_data(const gbconv_desc* desc, const void* dy, const void* w, void* dx, void* stream) {
  return bwd_data(desc, dy, w, nullptr, dx, stream);
}

gbconv_status gbconv_conv_transpose(const gbconv_desc* desc, const void* x, const void* w, const float* bias, void* y,
                                    void* stream) {
  return bwd_data(desc, x, w, bias, y, stream);
}

gbconv_status gbconv_pack_weight(const gbconv_desc* desc, const void* w_oihw, void* w_ohwi, void* stream) {
  Problem p;
  gbconv_status s = resolve(desc, &p);
  if (s != GBCONV_OK) return s;
  if (!w_oihw || !w_ohwi) return GBCONV_EINVAL;
  Launch l;
  if (!device_context(&l, stream)) return GBCONV_ECUDA;
  return launch_pack_weight(p, w_oihw, w_ohwi, l);
}

gbconv_status gbconv_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GBCONV_ECUDA;
  Launch l;
  if (!device_context(&l, stream)) return GBCONV_ECUDA;
  unsigned int word = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&word, g_status_word, sizeof(word)) != cudaSuccess) return GBCONV_ECUDA;
  if (word != 0 && cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess) return GBCONV_ECUDA;
  return word ? GBCONV_ETIMEOUT : GBCONV_OK;
}

uint64_t gbconv_kernels_launched(void) { return g_launches.load(std::memory_order_relaxed); }

int64_t gbconv_set_wait_limit_ns(int64_t ns) {
  return g_wait_ns.exchange(ns > 0 ? ns : kDefaultWaitNs, std::memory_order_relaxed);
}

const char* gbconv_status_string(gbconv_status status) {
  switch (status) {
    case GBCONV_OK: return "ok";
    case GBCONV_EINVAL: return "invalid argument or shape";
    case GBCONV_EUNSUPPORTED: return "shape beyond the library's 32-bit indexing";
    case GBCONV_ECUDA: return "CUDA runtime error";
    case GBCONV_ETIMEOUT: return "a kernel's bounded internal wait expired";
  }
  return "unknown status";
}

}  // extern "C"
