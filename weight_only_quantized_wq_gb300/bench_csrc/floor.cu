// floor.cu -- read-only streaming kernel: the practical floor of the time to
// read a buffer once from HBM on this GPU.  Built into its own library
// (libwqfloor.so), used only by the benchmark to put the matmul kernels'
// times next to what a plain read of the same bytes costs.
//
// Each thread reads 16-byte words with non-allocating loads in a grid-stride
// loop (four loads in flight per thread per iteration) and folds them into a
// 32-bit XOR, one value per block written out so the loads cannot be removed.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__global__ void read_kernel(const uint4 *__restrict__ src, size_t n16, uint32_t *__restrict__ sink) {
  uint32_t acc = 0;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = ld_stream(src + i), b = ld_stream(src + i + stride), c = ld_stream(src + i + 2 * stride),
                d = ld_stream(src + i + 3 * stride);
    acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^ d.z ^ d.w;
  }
  for (; i < n16; i += stride) {
    const uint4 a = ld_stream(src + i);
    acc ^= a.x ^ a.y ^ a.z ^ a.w;
  }
  acc ^= __shfl_xor_sync(0xffffffffu, acc, 16);
  acc ^= __shfl_xor_sync(0xffffffffu, acc, 8);
  acc ^= __shfl_xor_sync(0xffffffffu, acc, 4);
  acc ^= __shfl_xor_sync(0xffffffffu, acc, 2);
  acc ^= __shfl_xor_sync(0xffffffffu, acc, 1);
  if ((threadIdx.x & 31) == 0) atomicXor(sink + blockIdx.x, acc);
}

}  // namespace

extern "C" {

// Read `bytes` (a multiple of 16, src 16-byte aligned) once; sink holds at
// least `blocks` uint32.  blocks x threads is the launch shape.  Returns the
// launch's cudaError_t.
__attribute__((visibility("default"))) int wq_floor_read(const void *src, size_t bytes, uint32_t *sink, int blocks,
                                                          int threads, void *stream) {
  read_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<const uint4 *>(src), bytes / 16,
                                                                         sink);
  return (int)cudaGetLastError();
}

}  // extern "C"
