// Calls on HOST buffers: the batch is moved through a caller-owned device staging buffer in slices,
// so that the copy in of slice i+1, the kernel of slice i and the copy out of slice i-1 run at the
// same time (host-to-device and device-to-host copies on their own copy engines).  Images are
// independent in the forward and in the input gradient, so a slice is the same call on a smaller
// batch.  A call starts after the work already enqueued on the caller's stream; its copies and
// kernels run on three streams of the library (copies in, kernels, copies out), so that the caller's
// stream holds nothing of a call in flight and the next call's copies queue right behind this one's.
//
// Without a completion event the call returns once the result is in the host buffer.  With one, it
// returns after enqueueing and records the event when the result is there: independent calls then
// keep the host link busy back to back, one call's last copy out overlapping the next call's copies
// in.
//
// Per device the library keeps its three streams and a pool of events, made on first use.  Enqueueing
// is serialised per device (a mutex); the copies and kernels of calls in flight run in call order.
// An event of the pool may be recorded again by a later call while an earlier call's stream waits on
// it: a wait applies to the record that precedes it, so that is safe.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "problem.h"

namespace gbconv {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxSlices = 16;
constexpr int kEvents = 2 * kMaxSlices + 1;  // copy-in and kernel events per slice, and the end

struct HostPath {
  std::mutex mu;  // enqueueing, one host call at a time per device
  bool ready = false;
  cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
  cudaEvent_t ev[kEvents] = {};
  cudaEvent_t start = nullptr, joined = nullptr, computed = nullptr;
  unsigned int* word = nullptr;  // pinned host copy of the device status word (synchronous calls)
};

HostPath g_host[kMaxDevices];
std::mutex g_host_init;

int64_t align256(int64_t b) { return (b + 255) & ~int64_t(255); }

// The byte sizes a host call moves: per image of the source (x, or dy) and of the result, the weight,
// the bias.
struct HostSizes {
  int64_t n, src_img, out_img, w, bias;
  int64_t staging() const { return align256(w) + align256(bias) + align256(n * src_img) + align256(n * out_img); }
};

HostSizes host_sizes(const Problem& p, bool dgrad, bool bias) {
  HostSizes s;
  const int64_t eb = p.elem_bytes();
  const int64_t x_img = p.Cin * p.D * p.H * p.W * eb, y_img = p.Cout * p.OD * p.OH * p.OW * eb;
  s.n = p.N;
  s.src_img = dgrad ? y_img : x_img;
  s.out_img = dgrad ? x_img : y_img;
  s.w = p.w_elems() * eb;
  s.bias = bias ? (dgrad ? p.Cin : p.Cout) * int64_t(sizeof(float)) : 0;
  return s;
}

HostPath* host_path(int dev) {
  HostPath& h = g_host[dev];
  std::lock_guard<std::mutex> lk(g_host_init);
  if (!h.ready) {
    if (cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    if (cudaStreamCreateWithFlags(&h.comp, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    if (cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    for (int i = 0; i < kEvents; ++i)
      if (cudaEventCreateWithFlags(&h.ev[i], cudaEventDisableTiming) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&h.start, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&h.joined, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&h.computed, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    if (cudaHostAlloc(reinterpret_cast<void**>(&h.word), sizeof(unsigned int), cudaHostAllocDefault) != cudaSuccess)
      return nullptr;
    h.ready = true;
  }
  return &h;
}

// One device call on a batch slice: the forward, the input gradient, or the transposed convolution.
gbconv_status slice_call(const gbconv_desc& d, bool dgrad, const void* src, const void* w, const float* bias,
                         void* out, cudaStream_t stream) {
  if (!dgrad) return gbconv_fwd(&d, src, w, bias, out, stream);
  return bias ? gbconv_conv_transpose(&d, src, w, bias, out, stream) : gbconv_bwd_data(&d, src, w, out, stream);
}

// Status at the end of a synchronous host call: the pinned copy of the device status word (filled by
// the call's last copy), cleared on the device when set.
gbconv_status end_status(HostPath* h, const Launch& l, cudaStream_t s) {
  if (*h->word == 0) return GBCONV_OK;
  if (cudaMemsetAsync(l.status, 0, sizeof(unsigned int), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
    return GBCONV_ECUDA;
  return GBCONV_ETIMEOUT;  // reported once, as gbconv_device_status does
}

struct Staged {
  uint8_t *w, *src, *out;
  float* bias;
};

// A synchronous call that is not worth slicing: copies, kernel and copy back in order on the
// caller's stream, with no events between streams.
gbconv_status one_slice(HostPath* h, const gbconv_desc& d, bool dgrad, const void* src_h, const void* w_h,
                        const float* bias_h, void* out_h, const Staged& st, const HostSizes& z, const Launch& l) {
  const auto stream = static_cast<cudaStream_t>(l.stream);
  *h->word = 0;
  bool ok = cudaMemcpyAsync(st.w, w_h, size_t(z.w), cudaMemcpyHostToDevice, stream) == cudaSuccess &&
            (!bias_h || cudaMemcpyAsync(st.bias, bias_h, size_t(z.bias), cudaMemcpyHostToDevice, stream) == cudaSuccess) &&
            cudaMemcpyAsync(st.src, src_h, size_t(z.n * z.src_img), cudaMemcpyHostToDevice, stream) == cudaSuccess;
  const gbconv_status call = ok ? slice_call(d, dgrad, st.src, st.w, st.bias, st.out, stream) : GBCONV_OK;
  if (ok && call == GBCONV_OK)
    ok = cudaMemcpyAsync(out_h, st.out, size_t(z.n * z.out_img), cudaMemcpyDeviceToHost, stream) == cudaSuccess &&
         cudaMemcpyAsync(h->word, l.status, sizeof(unsigned int), cudaMemcpyDeviceToHost, stream) == cudaSuccess;
  // the copies enqueued so far use the caller's buffers: the call returns after them
  const bool drained = cudaStreamSynchronize(stream) == cudaSuccess;
  if (call != GBCONV_OK) return call;
  if (!ok || !drained) return GBCONV_ECUDA;
  return end_status(h, l, stream);
}

gbconv_status host_call(const gbconv_desc* desc, bool dgrad, const void* src_h, const void* w_h, const float* bias_h,
                        void* out_h, void* staging, int64_t staging_bytes, int32_t slices, void* stream_v,
                        void* done_v) {
  Problem p;
  gbconv_status s = resolve(desc, &p);
  if (s != GBCONV_OK) return s;
  if (!src_h || !w_h || !out_h || !staging) return GBCONV_EINVAL;
  if ((reinterpret_cast<uintptr_t>(staging) & 255u) != 0) return GBCONV_EINVAL;
  const HostSizes z = host_sizes(p, dgrad, bias_h != nullptr);
  if (staging_bytes < z.staging()) return GBCONV_EINVAL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GBCONV_ECUDA;
  HostPath* h = host_path(dev);
  Launch l;
  if (!h || !launch_context(&l, stream_v)) return GBCONV_ECUDA;
  std::lock_guard<std::mutex> lk(h->mu);
  const auto stream = static_cast<cudaStream_t>(stream_v);
  const auto done = static_cast<cudaEvent_t>(done_v);

  // staging: [w][bias][source, whole batch][result, whole batch]
  Staged st;
  uint8_t* base = static_cast<uint8_t*>(staging);
  st.w = base;
  st.bias = bias_h ? reinterpret_cast<float*>(base + align256(z.w)) : nullptr;
  st.src = base + align256(z.w) + align256(z.bias);
  st.out = st.src + align256(z.n * z.src_img);

  // The call ends with the last slice's copy out, which nothing overlaps, and every slice adds a
  // few microseconds between consecutive copies: about sqrt(result bytes / 512 KB) slices balance
  // the two (measured on the host link: 4-6 slices for 13-17 MB results, 8-16 for 51 MB).
  int64_t ns = slices;
  if (ns <= 0) ns = std::llround(std::sqrt(double(z.n * z.out_img) / double(512 << 10)));
  ns = std::max<int64_t>(1, std::min<int64_t>({ns, z.n, kMaxSlices}));
  if (ns == 1 && !done) return one_slice(h, *desc, dgrad, src_h, w_h, bias_h, out_h, st, z, l);

  // The staging buffer may have been in use on `stream` (a stream-ordered allocator hands it out
  // there): the library's streams start after the work already enqueued on it.
  bool ok = cudaEventRecord(h->start, stream) == cudaSuccess && cudaStreamWaitEvent(h->in, h->start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(h->comp, h->start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(h->out, h->start, 0) == cudaSuccess;
  ok = ok && cudaMemcpyAsync(st.w, w_h, size_t(z.w), cudaMemcpyHostToDevice, h->in) == cudaSuccess;
  if (ok && bias_h) ok = cudaMemcpyAsync(st.bias, bias_h, size_t(z.bias), cudaMemcpyHostToDevice, h->in) == cudaSuccess;
  gbconv_status call = GBCONV_OK;
  for (int64_t i = 0; ok && call == GBCONV_OK && i < ns; ++i) {
    const int64_t lo = z.n * i / ns, hi = z.n * (i + 1) / ns;
    if (hi == lo) continue;
    cudaEvent_t in_done = h->ev[2 * i], k_done = h->ev[2 * i + 1];
    ok = cudaMemcpyAsync(st.src + lo * z.src_img, static_cast<const uint8_t*>(src_h) + lo * z.src_img,
                         size_t((hi - lo) * z.src_img), cudaMemcpyHostToDevice, h->in) == cudaSuccess &&
         cudaEventRecord(in_done, h->in) == cudaSuccess && cudaStreamWaitEvent(h->comp, in_done, 0) == cudaSuccess;
    if (!ok) break;
    gbconv_desc sub = *desc;
    sub.n = hi - lo;
    call = slice_call(sub, dgrad, st.src + lo * z.src_img, st.w, st.bias, st.out + lo * z.out_img, h->comp);
    if (call != GBCONV_OK) break;
    ok = cudaEventRecord(k_done, h->comp) == cudaSuccess && cudaStreamWaitEvent(h->out, k_done, 0) == cudaSuccess &&
         cudaMemcpyAsync(static_cast<uint8_t*>(out_h) + lo * z.out_img, st.out + lo * z.out_img,
                         size_t((hi - lo) * z.out_img), cudaMemcpyDeviceToHost, h->out) == cudaSuccess;
  }
  // Synchronous: the device status word (bounded-wait failures), read after the last kernel (the
  // copy-out stream already waits for it).
  if (!done) {
    *h->word = 0;
    if (ok && call == GBCONV_OK)
      ok = cudaMemcpyAsync(h->word, l.status, sizeof(unsigned int), cudaMemcpyDeviceToHost, h->out) == cudaSuccess;
  }
  // Every copy enqueued so far reads or writes the caller's buffers.  The copy-in and kernel streams
  // join the copy-out stream, and the end of all three is the completion event, or (synchronous) an
  // event the call waits for and `stream` waits on (later work there may reuse the staging buffer).
  cudaEvent_t end = done ? done : h->ev[kEvents - 1];
  bool drained = cudaEventRecord(h->joined, h->in) == cudaSuccess &&
                 cudaStreamWaitEvent(h->out, h->joined, 0) == cudaSuccess &&
                 cudaEventRecord(h->computed, h->comp) == cudaSuccess &&
                 cudaStreamWaitEvent(h->out, h->computed, 0) == cudaSuccess && cudaEventRecord(end, h->out) == cudaSuccess;
  if (!done) drained = drained && cudaStreamWaitEvent(stream, end, 0) == cudaSuccess && cudaEventSynchronize(end) == cudaSuccess;
  if (call != GBCONV_OK) return call;
  if (!ok || !drained) return GBCONV_ECUDA;
  return done ? GBCONV_OK : end_status(h, l, h->out);
}

}  // namespace
}  // namespace gbconv

using namespace gbconv;

extern "C" {

gbconv_status gbconv_host_staging_bytes(const gbconv_desc* desc, int32_t op, int32_t with_bias, int64_t* bytes) {
  if (!bytes || (op != GBCONV_OP_FWD && op != GBCONV_OP_BWD_DATA)) return GBCONV_EINVAL;
  Problem p;
  gbconv_status s = resolve(desc, &p);
  if (s != GBCONV_OK) return s;
  *bytes = host_sizes(p, op == GBCONV_OP_BWD_DATA, with_bias != 0).staging();
  return GBCONV_OK;
}

gbconv_status gbconv_fwd_host(const gbconv_desc* desc, const void* x, const void* w, const float* bias, void* y,
                              void* staging, int64_t staging_bytes, int32_t slices, void* stream, void* done_event) {
  return host_call(desc, false, x, w, bias, y, staging, staging_bytes, slices, stream, done_event);
}

gbconv_status gbconv_bwd_data_host(const gbconv_desc* desc, const void* dy, const void* w, void* dx, void* staging,
                                   int64_t staging_bytes, int32_t slices, void* stream, void* done_event) {
  return host_call(desc, true, dy, w, nullptr, dx, staging, staging_bytes, slices, stream, done_event);
}

gbconv_status gbconv_conv_transpose_host(const gbconv_desc* desc, const void* x, const void* w, const float* bias,
                                         void* y, void* staging, int64_t staging_bytes, int32_t slices, void* stream,
                                         void* done_event) {
  return host_call(desc, true, x, w, bias, y, staging, staging_bytes, slices, stream, done_event);
}

}  // extern "C"
