// repack.cu -- wq_pack / wq_unpack kernels: bit-exact permutation between the
// page layout (BitDistiller quant_matmul_kernel; tiny-llm int8_matmul for
// int8) and the tiled layout described in layout.cuh.
#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.h"
#include "layout.cuh"

namespace wq {

// One thread per output word.
template <int W>
__global__ void pack_kernel(const void *__restrict__ qin, uint32_t *__restrict__ out, int K, int N) {
  using G = Geo<W>;
  const int NT = N / 16;
  const size_t total = (size_t)K / G::V * N;
  for (size_t o = (size_t)blockIdx.x * blockDim.x + threadIdx.x; o < total; o += (size_t)gridDim.x * blockDim.x) {
    const int wi = (int)(o & 3), lane = (int)((o >> 2) & 31);
    const size_t tile = o >> 7;
    const int nt = (int)(tile % NT);
    const int kc = (int)(tile / NT);
    uint32_t word = 0;
    if (W == 8) {
      int kk, nn;
      field_coords<W>(lane, wi, 0, kk, nn);
      const int8_t *q = static_cast<const int8_t *>(qin);
      word = *reinterpret_cast<const uint32_t *>(q + (size_t)(nt * 16 + nn) * K + (size_t)kc * G::KC + kk);
    } else {
      const uint32_t *qw = static_cast<const uint32_t *>(qin);
#pragma unroll
      for (int f = 0; f < G::V; ++f) {
        int kk, nn;
        field_coords<W>(lane, wi, f, kk, nn);
        const int k = kc * G::KC + kk, n = nt * 16 + nn;
        const uint32_t code = (qw[(size_t)(k / G::V) * N + n] >> ((k % G::V) * W)) & ((1u << W) - 1u);
        word |= code << (f * W);
      }
    }
    out[o] = word;
  }
}

// One thread per (k, n): codes (K, N) row-major.
template <int W>
__global__ void unpack_kernel(const uint32_t *__restrict__ packed, uint8_t *__restrict__ codes, int K, int N) {
  using G = Geo<W>;
  const int NT = N / 16;
  const size_t total = (size_t)K * N;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int k = (int)(i / N), n = (int)(i % N);
    const int kc = k / G::KC, kk = k % G::KC;
    const int ks = kk >> 4, rem = kk & 15, t = rem >> 2, c = rem & 3;
    const int h = ks / G::WK, j = ks % G::WK;
    const int nt = n >> 4, nn = n & 15, g = nn & 7, r = nn >> 3;
    const int lane = 4 * g + t, wi = 2 * h + r;
    int f;
    if (W == 8)
      f = c;
    else
      f = (c & 1) ? G::H + 2 * j + (c >> 1) : 2 * j + (c >> 1);
    const uint32_t word = packed[(((size_t)kc * NT + nt) * 32 + lane) * 4 + wi];
    codes[i] = (uint8_t)((word >> (f * W)) & ((1u << W) - 1u));
  }
}

// Liger planar ternary bytes (K/4, N) -> the tiled 2-bit layout, one thread
// per output word: the code of (k, n) is field k div R of byte [k mod R][n],
// R = K / 4 (ops/experimental/mm_int8int2.py, pack_weights).  The codes are
// the stored values (weight + 1), so the matmul subtracts 1 as its zero.
__global__ void t2_pack_kernel(const uint8_t *__restrict__ qin, uint32_t *__restrict__ out, int K, int N) {
  using G = Geo<2>;
  const int NT = N / 16, R = K / 4;
  const size_t total = (size_t)K / G::V * N;
  for (size_t o = (size_t)blockIdx.x * blockDim.x + threadIdx.x; o < total; o += (size_t)gridDim.x * blockDim.x) {
    const int wi = (int)(o & 3), lane = (int)((o >> 2) & 31);
    const size_t tile = o >> 7;
    const int nt = (int)(tile % NT);
    const int kc = (int)(tile / NT);
    uint32_t word = 0;
#pragma unroll
    for (int f = 0; f < G::V; ++f) {
      int kk, nn;
      field_coords<2>(lane, wi, f, kk, nn);
      const int k = kc * G::KC + kk, n = nt * 16 + nn;
      const uint32_t code = (qin[(size_t)(k % R) * N + n] >> (2 * (k / R))) & 3u;
      word |= code << (f * 2);
    }
    out[o] = word;
  }
}

// int8 activations -> bf16 (exact: |x| <= 128 needs 8 significant bits),
// four per thread.
__global__ void int8_to_bf16_kernel(const char4 *__restrict__ x, uint2 *__restrict__ y, size_t n4) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
    const char4 v = x[i];
    const uint32_t a = (uint32_t)__float_as_uint((float)v.x) >> 16 | ((uint32_t)__float_as_uint((float)v.y) & 0xFFFF0000u);
    const uint32_t b = (uint32_t)__float_as_uint((float)v.z) >> 16 | ((uint32_t)__float_as_uint((float)v.w) & 0xFFFF0000u);
    y[i] = make_uint2(a, b);
  }
}

static int grid_for(size_t n) {
  size_t b = (n + 255) / 256;
  return (int)(b > 65535 * 4 ? 65535 * 4 : (b ? b : 1));
}

cudaError_t launch_pack(const void *qin, void *out, int K, int N, int w_bit, cudaStream_t s) {
  const size_t words = (size_t)K * N * w_bit / 32;
  const int grid = grid_for(words);
  switch (w_bit) {
    case 2: pack_kernel<2><<<grid, 256, 0, s>>>(qin, (uint32_t *)out, K, N); break;
    case 4: pack_kernel<4><<<grid, 256, 0, s>>>(qin, (uint32_t *)out, K, N); break;
    case 8: pack_kernel<8><<<grid, 256, 0, s>>>(qin, (uint32_t *)out, K, N); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_t2_pack(const void *qin, void *out, int K, int N, cudaStream_t s) {
  const size_t words = (size_t)K * N / 16;
  t2_pack_kernel<<<grid_for(words), 256, 0, s>>>(static_cast<const uint8_t *>(qin), (uint32_t *)out, K, N);
  return cudaGetLastError();
}

cudaError_t launch_int8_to_bf16(const void *x, void *y, size_t n, cudaStream_t s) {
  const size_t n4 = n / 4;
  int8_to_bf16_kernel<<<grid_for(n4), 256, 0, s>>>(static_cast<const char4 *>(x), static_cast<uint2 *>(y), n4);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const void *packed, uint8_t *codes, int K, int N, int w_bit, cudaStream_t s) {
  const int grid = grid_for((size_t)K * N);
  switch (w_bit) {
    case 2: unpack_kernel<2><<<grid, 256, 0, s>>>((const uint32_t *)packed, codes, K, N); break;
    case 4: unpack_kernel<4><<<grid, 256, 0, s>>>((const uint32_t *)packed, codes, K, N); break;
    case 8: unpack_kernel<8><<<grid, 256, 0, s>>>((const uint32_t *)packed, codes, K, N); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace wq
