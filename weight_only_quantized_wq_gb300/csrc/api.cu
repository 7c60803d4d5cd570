// api.cu -- the C ABI declared in include/wq.h: host-side validation, the
// per-device cache, and dispatch to the kernels.  No entry point allocates
// device memory or synchronises (wq_check_device excepted).
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "api.h"
#include "kernels.h"
#include "wq.h"

namespace {

// Device status word: kernels OR bits into it when a barrier wait gives up.
__device__ uint32_t g_status_word;

struct DeviceInfo {
  bool ready = false;
  bool arch_ok = false;
  int sms = 0;
  uint32_t *status = nullptr;  // device address of g_status_word on this device
};

constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::mutex g_mutex;

// Query (once per device) the SM count, the architecture, and the device
// address of the status word.  Must run with that device current.
wq_status device_info(DeviceInfo **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return WQ_ERR_CUDA;
  DeviceInfo &d = g_devices[dev];
  if (!d.ready) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!d.ready) {
      int major = 0, minor = 0, sms = 0;
      if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return WQ_ERR_CUDA;
      d.arch_ok = (major == 10 && minor == 3);
      d.sms = sms;
      if (d.arch_ok) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return WQ_ERR_CUDA;
        d.status = static_cast<uint32_t *>(p);
      }
      d.ready = true;
    }
  }
  if (!d.arch_ok) return WQ_ERR_ARCH;
  *out = &d;
  return WQ_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool valid_wbit(int w) { return w == 2 || w == 4 || w == 8; }

// Shape rules shared by pack, unpack and matmul.
wq_status check_kn(int K, int N, int w_bit) {
  if (!valid_wbit(w_bit)) return WQ_ERR_WBIT;
  if (K <= 0 || N <= 0) return WQ_ERR_SHAPE;
  if (N % 16 != 0 || K % (256 / w_bit) != 0 || N > wq::kMaxN) return WQ_ERR_SHAPE;
  return WQ_OK;
}

// Workspace of a call: the largest over its 64-row slices of the few-token
// kernel (full slices and the remainder).
size_t slice_workspace(int M, int N, int K, int w_bit, int group_size, bool zero, int sms) {
  size_t ws = wq::plan_decode(M < 64 ? M : 64, N, K, w_bit, group_size, zero, sms).workspace;
  if (M > 64 && M % 64 != 0) {
    const size_t r = wq::plan_decode(M % 64, N, K, w_bit, group_size, zero, sms).workspace;
    ws = r > ws ? r : ws;
  }
  return ws;
}

}  // namespace

namespace wq {

wq_status prepare_call(const void *x, wq_dtype x_dtype, const void *packed_w, const void *scales, wq_dtype s_dtype,
                       const int32_t *zeros, int M, int N, int K, int w_bit, int group_size, void *out,
                       wq_dtype out_dtype, Call *c) {
  *c = Call{};
  if (!x || !packed_w || !scales || !out) return WQ_ERR_NULL;
  if (!valid_wbit(w_bit)) return WQ_ERR_WBIT;
  if (M < 0 || N < 0 || K <= 0) return WQ_ERR_SHAPE;
  if (M == 0 || N == 0) {
    c->noop = true;
    return WQ_OK;
  }
  wq_status st = check_kn(K, N, w_bit);
  if (st != WQ_OK) return st;
  if (x_dtype != WQ_F16 && x_dtype != WQ_BF16) return WQ_ERR_DTYPE;
  if (out_dtype != WQ_F32 && out_dtype != WQ_F16 && out_dtype != WQ_BF16) return WQ_ERR_DTYPE;
  if (w_bit == 8) {
    if (s_dtype != WQ_F32 || zeros != nullptr) return WQ_ERR_DTYPE;
    group_size = K;
  } else {
    if (s_dtype != WQ_F16 && s_dtype != WQ_BF16) return WQ_ERR_DTYPE;
    if (group_size == -1) group_size = K;
    if (group_size <= 0 || K % group_size != 0 || group_size % 16 != 0) return WQ_ERR_GROUP;
  }
  if (!aligned(x, 16) || !aligned(packed_w, 16) || !aligned(out, 16) || !aligned(scales, 16) || !aligned(zeros, 16))
    return WQ_ERR_ALIGN;
  DeviceInfo *d = nullptr;
  if ((st = device_info(&d)) != WQ_OK) return st;
  MatmulArgs &a = c->a;
  a.x = x;
  a.packed = packed_w;
  a.scales = scales;
  a.zeros = reinterpret_cast<const uint32_t *>(zeros);
  a.out = out;
  a.out_type = out_dtype == WQ_F32 ? kOutF32 : out_dtype == WQ_F16 ? kOutF16 : kOutBF16;
  a.M = M;
  a.N = N;
  a.K = K;
  a.w_bit = w_bit;
  a.group_size = group_size;
  a.x_bf16 = (x_dtype == WQ_BF16);
  a.s_bf16 = (s_dtype == WQ_BF16);
  a.unit_scale = false;
  a.sym_zero = w_bit == 8 ? 0 : 1 << (w_bit - 1);
  a.wait_limit = 0;  // the default limit
  a.withhold = -1;
  a.err = d->status;
  c->sms = d->sms;
  c->route = route_of(a);
  c->need = c->route == Route::kDecode ? slice_workspace(M, N, K, w_bit, group_size, zeros != nullptr, d->sms) : 0;
  return WQ_OK;
}

Route route_of(const MatmulArgs &a) {
  if (a.w_bit != 4 || !midm_supported(a) || a.M <= kDecodeMaxM) return Route::kDecode;
  if (a.M >= kPrefillMinM && prefill_supported(a)) {
    if (prefill_within_tolerance(a)) return Route::kPrefill;
    const long long tiles = (long long)((a.M + 255) / 256) * ((a.N + 127) / 128);  // of the two-term kernel
    if (a.M >= kSplitMinM && tiles >= kSplitMinTiles) return Route::kPrefillSplit;
  }
  return Route::kMidm;
}

wq_status run_call(const Call &c, void *workspace, size_t workspace_bytes, void *stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (c.route == Route::kPrefill || c.route == Route::kPrefillSplit)
    return launch_prefill(c.a, c.sms, workspace, workspace_bytes, c.route == Route::kPrefillSplit, s) == cudaSuccess
               ? WQ_OK
               : WQ_ERR_CUDA;
  if (c.route == Route::kMidm) {
    const MidmPlan pl = plan_midm(c.a.M, c.a.N, c.a.K, c.sms);
    return launch_midm(c.a, pl, s) == cudaSuccess ? WQ_OK : WQ_ERR_CUDA;
  }
  // Rows are processed 64 at a time (the few-token kernel's largest token tile).
  MatmulArgs a = c.a;
  const int M = c.a.M, N = a.N, K = a.K;
  const bool zero = a.zeros != nullptr;
  const DecodePlan full = plan_decode(M < 64 ? M : 64, N, K, a.w_bit, a.group_size, zero, c.sms, a.unit_scale);
  for (int m0 = 0; m0 < M; m0 += 64) {
    a.M = (M - m0) < 64 ? (M - m0) : 64;
    a.x = static_cast<const uint16_t *>(c.a.x) + (size_t)m0 * K;
    a.out = static_cast<char *>(c.a.out) + (size_t)m0 * N * (a.out_type == kOutF32 || a.out_type == kOutS32 ? 4 : 2);
    const DecodePlan p =
        (a.M == (M < 64 ? M : 64)) ? full : plan_decode(a.M, N, K, a.w_bit, a.group_size, zero, c.sms, a.unit_scale);
    if (launch_decode(a, p, workspace, s) != cudaSuccess) return WQ_ERR_CUDA;
  }
  return WQ_OK;
}

}  // namespace wq

extern "C" {

const char *wq_status_string(wq_status s) {
  switch (s) {
    case WQ_OK: return "ok";
    case WQ_ERR_NULL: return "a required pointer is NULL";
    case WQ_ERR_SHAPE: return "invalid or unsupported shape (need N % 16 == 0, N <= 262144, K % (256 / w_bit) == 0)";
    case WQ_ERR_WBIT: return "w_bit must be 2, 4 or 8";
    case WQ_ERR_GROUP: return "group_size must divide K and be a multiple of 16 (or -1 / K)";
    case WQ_ERR_DTYPE: return "unsupported dtype combination";
    case WQ_ERR_ALIGN: return "pointer not 16-byte aligned";
    case WQ_ERR_WORKSPACE: return "workspace missing or smaller than wq_workspace_bytes()";
    case WQ_ERR_ARCH: return "current device is not compute capability 10.3 (sm_103a)";
    case WQ_ERR_CUDA: return "CUDA runtime error";
    case WQ_ERR_TIMEOUT: return "a kernel gave up waiting on one of its barriers";
  }
  return "unknown status";
}

int wq_chunk_k(int w_bit) { return valid_wbit(w_bit) ? 256 / w_bit : 0; }

size_t wq_packed_bytes(int K, int N, int w_bit) {
  if (check_kn(K, N, w_bit) != WQ_OK) return 0;
  return (size_t)K * N * w_bit / 8;
}

wq_status wq_pack(const void *q_in, int K, int N, int w_bit, void *packed_out, void *stream) {
  if (!q_in || !packed_out) return WQ_ERR_NULL;
  wq_status st = check_kn(K, N, w_bit);
  if (st != WQ_OK) return st;
  if (!aligned(q_in, 16) || !aligned(packed_out, 16)) return WQ_ERR_ALIGN;
  DeviceInfo *d = nullptr;
  if ((st = device_info(&d)) != WQ_OK) return st;
  return wq::launch_pack(q_in, packed_out, K, N, w_bit, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? WQ_OK
             : WQ_ERR_CUDA;
}

wq_status wq_unpack(const void *packed, int K, int N, int w_bit, uint8_t *codes_out, void *stream) {
  if (!packed || !codes_out) return WQ_ERR_NULL;
  wq_status st = check_kn(K, N, w_bit);
  if (st != WQ_OK) return st;
  if (!aligned(packed, 16)) return WQ_ERR_ALIGN;
  DeviceInfo *d = nullptr;
  if ((st = device_info(&d)) != WQ_OK) return st;
  return wq::launch_unpack(packed, codes_out, K, N, w_bit, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? WQ_OK
             : WQ_ERR_CUDA;
}

size_t wq_workspace_bytes(int M, int N, int K, int w_bit, int group_size) {
  if (M <= 0 || check_kn(K, N, w_bit) != WQ_OK) return 0;
  DeviceInfo *d = nullptr;
  if (device_info(&d) != WQ_OK) return 0;
  if (w_bit == 8 || group_size == -1) group_size = K;
  if (group_size <= 0 || K % group_size != 0) return 0;
  // The tensor-core paths need no workspace, whatever the dtypes.
  wq::MatmulArgs a{};
  a.M = M;
  a.N = N;
  a.K = K;
  a.w_bit = w_bit;
  a.group_size = group_size;
  // The tensor-core paths need no workspace; with this much the many-token
  // kernel (int4, same x and scale dtype) runs persistent.  Which of them a
  // call takes depends on its dtypes, so this covers either.
  if (wq::route_of(a) != wq::Route::kDecode)
    return (w_bit == 4 && wq::kPrefillMinM <= M) ? wq::prefill_workspace_bytes(M, N, K, d->sms) : 0;
  // Enough with zeros or without (the zero rows' shared memory can change the split).
  const size_t with_z = slice_workspace(M, N, K, w_bit, group_size, true, d->sms);
  const size_t without = w_bit == 8 ? with_z : slice_workspace(M, N, K, w_bit, group_size, false, d->sms);
  return with_z > without ? with_z : without;
}

wq_status wq_matmul_ex(const void *x, wq_dtype x_dtype, const void *packed_w, const void *scales, wq_dtype s_dtype,
                       const int32_t *zeros, int M, int N, int K, int w_bit, int group_size, void *out,
                       wq_dtype out_dtype, void *workspace, size_t workspace_bytes, void *stream) {
  wq::Call c;
  wq_status st = wq::prepare_call(x, x_dtype, packed_w, scales, s_dtype, zeros, M, N, K, w_bit, group_size, out,
                                  out_dtype, &c);
  if (st != WQ_OK || c.noop) return st;
  if (c.need > 0 && (!workspace || workspace_bytes < c.need)) return WQ_ERR_WORKSPACE;
  if (workspace && !aligned(workspace, 16)) return WQ_ERR_ALIGN;
  return wq::run_call(c, workspace, workspace ? workspace_bytes : 0, stream);
}

wq_status wq_matmul(const void *x, wq_dtype x_dtype, const void *packed_w, const void *scales, wq_dtype s_dtype,
                    const int32_t *zeros, int M, int N, int K, int w_bit, int group_size, float *out,
                    void *workspace, size_t workspace_bytes, void *stream) {
  return wq_matmul_ex(x, x_dtype, packed_w, scales, s_dtype, zeros, M, N, K, w_bit, group_size, out, WQ_F32,
                      workspace, workspace_bytes, stream);
}

// ------------------------------------------------------------------ ternary int2
static wq_status check_t2(int K, int N) {
  if (K <= 0 || N <= 0 || N % 16 != 0 || K % 128 != 0 || N > wq::kMaxN) return WQ_ERR_SHAPE;
  if (K > 65536) return WQ_ERR_SHAPE;  // beyond, an fp32 partial sum could exceed 2^24
  return WQ_OK;
}

static size_t t2_x_bytes(int M, int K) { return ((size_t)M * K * 2 + 255) / 256 * 256; }

// Decode-kernel workspace of a ternary call (64-row slices, unit scale, zero 1).
static size_t t2_decode_workspace(int M, int N, int K, int sms) {
  size_t ws = wq::plan_decode(M < 64 ? M : 64, N, K, 2, K, false, sms, true).workspace;
  if (M > 64 && M % 64 != 0) {
    const size_t r = wq::plan_decode(M % 64, N, K, 2, K, false, sms, true).workspace;
    ws = r > ws ? r : ws;
  }
  return ws;
}

wq_status wq_t2_pack(const void *q_in, int K, int N, void *packed_out, void *stream) {
  if (!q_in || !packed_out) return WQ_ERR_NULL;
  wq_status st = check_t2(K, N);
  if (st != WQ_OK) return st;
  if (!aligned(q_in, 16) || !aligned(packed_out, 16)) return WQ_ERR_ALIGN;
  DeviceInfo *d = nullptr;
  if ((st = device_info(&d)) != WQ_OK) return st;
  return wq::launch_t2_pack(q_in, packed_out, K, N, static_cast<cudaStream_t>(stream)) == cudaSuccess ? WQ_OK
                                                                                                       : WQ_ERR_CUDA;
}

// Offset of the converted activations in a ternary call's workspace: after
// the few-token kernel's counters and partial sums, and never over the
// counters even when this call needs none (another call sharing the
// workspace may, and relies on them staying zero).
static size_t t2_x_offset(size_t dec) {
  const size_t lo = dec > wq::decode_counter_bytes() ? dec : wq::decode_counter_bytes();
  return (lo + 255) / 256 * 256;
}

size_t wq_t2_workspace_bytes(int M, int N, int K) {
  if (M <= 0 || check_t2(K, N) != WQ_OK) return 0;
  DeviceInfo *d = nullptr;
  if (device_info(&d) != WQ_OK) return 0;
  return t2_x_offset(t2_decode_workspace(M, N, K, d->sms)) + t2_x_bytes(M, K);
}

wq_status wq_t2_matmul(const int8_t *x, const void *packed_w, int M, int N, int K, int32_t *out, void *workspace,
                       size_t workspace_bytes, void *stream) {
  if (!x || !packed_w || !out) return WQ_ERR_NULL;
  if (M < 0 || N < 0 || K <= 0) return WQ_ERR_SHAPE;
  if (M == 0 || N == 0) return WQ_OK;
  wq_status st = check_t2(K, N);
  if (st != WQ_OK) return st;
  if (!aligned(x, 16) || !aligned(packed_w, 16) || !aligned(out, 16)) return WQ_ERR_ALIGN;
  DeviceInfo *d = nullptr;
  if ((st = device_info(&d)) != WQ_OK) return st;
  const size_t dec = t2_decode_workspace(M, N, K, d->sms);
  const size_t xoff = t2_x_offset(dec);
  if (!workspace || workspace_bytes < xoff + t2_x_bytes(M, K)) return WQ_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return WQ_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void *xb = static_cast<char *>(workspace) + xoff;
  if (wq::launch_int8_to_bf16(x, xb, (size_t)M * K, s) != cudaSuccess) return WQ_ERR_CUDA;
  wq::Call c;
  wq::MatmulArgs &a = c.a;
  a.x = xb;
  a.packed = packed_w;
  a.scales = nullptr;
  a.zeros = nullptr;
  a.out = out;
  a.out_type = wq::kOutS32;
  a.M = M;
  a.N = N;
  a.K = K;
  a.w_bit = 2;
  a.group_size = K;
  a.x_bf16 = true;
  a.s_bf16 = true;
  a.unit_scale = true;
  a.sym_zero = 1;  // codes are the weights plus one
  a.wait_limit = 0;
  a.withhold = -1;
  a.err = d->status;
  c.sms = d->sms;
  c.route = wq::Route::kDecode;
  c.need = dec;
  return wq::run_call(c, workspace, xoff, stream);
}

int wq_matmul_path(int M, int N, int K, int w_bit, int group_size, wq_dtype x_dtype, wq_dtype s_dtype) {
  if (!valid_wbit(w_bit) || M < 0 || N <= 0 || N % 16 != 0 || K <= 0 || K % (256 / w_bit) != 0) return -1;
  if (x_dtype != WQ_F16 && x_dtype != WQ_BF16) return -1;
  wq::MatmulArgs a{};
  a.M = M;
  a.N = N;
  a.K = K;
  a.w_bit = w_bit;
  a.x_bf16 = x_dtype == WQ_BF16;
  if (w_bit == 8) {
    if (s_dtype != WQ_F32) return -1;
    a.group_size = K;
  } else {
    if (s_dtype != WQ_F16 && s_dtype != WQ_BF16) return -1;
    a.group_size = group_size == -1 ? K : group_size;
    if (a.group_size <= 0 || K % a.group_size != 0 || a.group_size % 16 != 0) return -1;
  }
  a.s_bf16 = s_dtype == WQ_BF16;
  switch (wq::route_of(a)) {
    case wq::Route::kDecode: return 0;
    case wq::Route::kMidm: return 1;
    case wq::Route::kPrefill: return 2;
    case wq::Route::kPrefillSplit: return 3;
  }
  return -1;
}

wq_status wq_check_device(void *stream) {
  DeviceInfo *d = nullptr;
  wq_status st = device_info(&d);
  if (st != WQ_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return WQ_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(v)) != cudaSuccess) return WQ_ERR_CUDA;
  if (v == 0) return WQ_OK;
  const uint32_t zero = 0;
  if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess) return WQ_ERR_CUDA;
  return WQ_ERR_TIMEOUT;
}

}  // extern "C"
