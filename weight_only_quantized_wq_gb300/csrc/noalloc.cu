// noalloc.cu -- wq_matmul_noalloc: wq_matmul with library-owned scratch.
//
// Some callers cannot hand the library a workspace: a plugin inside a host
// framework that owns every device allocation and forbids libraries from
// allocating behind its back, or a latency-critical path that must not pay
// for cudaMalloc (which can synchronise the device).  For them this entry
// point uses a fixed scratch array that lives in the library image itself, so
// no call allocates anything.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds its kNoAllocScratchBytes until the process exits.  In host
// code its name is only a host-side stand-in, so the device address is
// looked up once per device with cudaGetSymbolAddress (with that device
// current) and that address is what the kernels receive.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "api.h"
#include "kernels.h"
#include "wq.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 8u << 20;  // 8 MiB per device

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device (set up on the
// first call made with that device current).
wq_status scratch_for_current_device(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return WQ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return WQ_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return WQ_OK;
}

// Scratch bytes a call may use: the whole array when it needs scratch (the
// many-token kernel never gets it: its persistent mode needs more partial
// tiles than the array holds, and one tile per CTA needs none).
size_t need_scratch_bytes(const wq::Call &c) {
  return c.need > 0 ? kNoAllocScratchBytes : 0;
}

}  // namespace

extern "C" {

wq_status wq_matmul_noalloc(const void *x, wq_dtype x_dtype, const void *packed_w, const void *scales,
                            wq_dtype s_dtype, const int32_t *zeros, int M, int N, int K, int w_bit, int group_size,
                            float *out, void *stream) {
  // Every argument check runs first: an invalid call enqueues nothing.
  wq::Call c;
  wq_status st =
      wq::prepare_call(x, x_dtype, packed_w, scales, s_dtype, zeros, M, N, K, w_bit, group_size, out, WQ_F32, &c);
  if (st != WQ_OK || c.noop) return st;
  if (c.need > kNoAllocScratchBytes) return WQ_ERR_WORKSPACE;
  void *scratch = nullptr;
  if (c.need > 0) {
    if ((st = scratch_for_current_device(&scratch)) != WQ_OK) return st;
    // The arrival counters at the front of the scratch must start at zero;
    // the array keeps whatever the previous call left, so clear them here.
    if (cudaMemsetAsync(scratch, 0, wq::decode_counter_bytes(), static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return WQ_ERR_CUDA;
  }
  return wq::run_call(c, scratch, need_scratch_bytes(c), stream);
}

}  // extern "C"
