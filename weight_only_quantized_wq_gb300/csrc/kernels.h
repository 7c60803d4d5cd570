// kernels.h -- internal launchers shared between the kernel files and the C ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace wq {

// Row-major 2-D tensor map of rows x cols elements of elem_bytes (1, 2 or 4)
// with a box of box_cols x box_rows, swizzle 0 (none), 32, 64 or 128 bytes,
// zero fill outside the tensor.  A map holds only these values, so one
// encoded for the same values is reused (cached, thread-safe).
bool encode_2d(CUtensorMap *m, const void *base, int elem_bytes, uint64_t cols, uint64_t rows, uint32_t box_cols,
               uint32_t box_rows, int swizzle = 0);

cudaError_t launch_pack(const void *qin, void *out, int K, int N, int w_bit, cudaStream_t s);
cudaError_t launch_unpack(const void *packed, uint8_t *codes, int K, int N, int w_bit, cudaStream_t s);

// Problem handed to the matmul kernels after host validation.
struct MatmulArgs {
  const void *x;          // (M, K) f16/bf16
  const void *packed;     // wq_pack layout
  const void *scales;     // (G, N) f16/bf16, or (N,) f32 for int8
  const uint32_t *zeros;  // (ceil(G/V), N) or nullptr
  float *out;             // (M, N)
  int M, N, K, w_bit, group_size;
  bool x_bf16, s_bf16;
  uint32_t *err;          // device status word
};

// Split of a few-token kernel over the GPU, chosen on the host.
struct DecodePlan {
  int srows;     // scale rows (groups) one CTA stages in shared memory
  int zrows;     // (MAGIC + zero) rows one CTA builds (srows for asymmetric codes, else 0)
  int zwrows;    // packed zero-word rows one CTA copies in (0 for symmetric codes)
  int smem;      // dynamic shared memory bytes
  int mt;        // 8-row token tiles (1, 2, 4, 8)
  int tn;        // 16-row weight tiles per warp
  int nblocks;   // CTAs along N
  int splits;    // CTAs along K
  int cps;       // chunk rows per split
  bool cluster;  // the splits of a column block form a cluster (reduction in shared memory)
  int fold;      // group schedule: k-steps per group when it divides the chunk, 0 when groups
                 // end on chunk boundaries, -1 otherwise
  size_t workspace;  // bytes: counters, then splits * M * N fp32 partials (0 if splits == 1)
};

// Most K splits whose partial tiles are reduced inside one thread-block cluster.
constexpr int kMaxClusterSplits = 16;

// Arrival counters at the start of every workspace (one per column block).
constexpr int kMaxColumnBlocks = 4096;
constexpr int kMaxN = 16 * 4 * kMaxColumnBlocks;  // 262144 output channels
size_t decode_counter_bytes();

DecodePlan plan_decode(int M, int N, int K, int w_bit, int group_size, bool zero, int sms);
cudaError_t launch_decode(const MatmulArgs &a, const DecodePlan &p, void *workspace, cudaStream_t s);

// Tensor-core path for many tokens (int4 codes, group size a multiple of 64,
// scales in the x dtype).
bool prefill_supported(const MatmulArgs &a);
cudaError_t launch_prefill(const MatmulArgs &a, cudaStream_t s);

// Token count from which wq_matmul takes the tensor-core path.
constexpr int kPrefillMinM = 65;

}  // namespace wq
