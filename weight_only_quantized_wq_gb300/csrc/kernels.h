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
// Liger planar ternary bytes (K/4, N) -> the 2-bit tiled layout (codes = weight + 1).
cudaError_t launch_t2_pack(const void *qin, void *out, int K, int N, cudaStream_t s);
// n int8 values (n % 4 == 0) -> bf16, exactly.
cudaError_t launch_int8_to_bf16(const void *x, void *y, size_t n, cudaStream_t s);

// Output element types of the matmul epilogues: the fp32 result is stored as
// is or rounded once (to nearest even) to fp16 or bf16.
enum OutType : int { kOutF32 = 0, kOutF16 = 1, kOutBF16 = 2, kOutS32 = 3 };  // S32: integer-valued results

// Problem handed to the matmul kernels after host validation.
struct MatmulArgs {
  const void *x;          // (M, K) f16/bf16
  const void *packed;     // wq_pack layout
  const void *scales;     // (G, N) f16/bf16, or (N,) f32 for int8
  const uint32_t *zeros;  // (ceil(G/V), N) or nullptr
  void *out;              // (M, N), element type out_type
  int out_type;           // OutType: fp32, fp16 or bf16
  int M, N, K, w_bit, group_size;
  bool x_bf16, s_bf16;
  bool unit_scale;        // no scales: every group scale is 1 (scales unused)
  int sym_zero;           // zero of every group when zeros == nullptr
  long long wait_limit;   // few-token kernel: SM cycles after which a barrier wait gives up
  int withhold;           // few-token kernel test hook: ring stage never filled (-1: none)
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

DecodePlan plan_decode(int M, int N, int K, int w_bit, int group_size, bool zero, int sms, bool unit_scale = false);
cudaError_t launch_decode(const MatmulArgs &a, const DecodePlan &p, void *workspace, cudaStream_t s);

// Tensor-core path for many tokens (int4 codes, group size a multiple of 64,
// scales in the x dtype).
bool prefill_supported(const MatmulArgs &a);
// Workspace with which the many-token kernel runs persistent with stream-K
// shares (flags, then one fp32 partial tile per CTA), for problems with at
// most a quarter as many tiles as SMs (0 otherwise); with less it runs one
// tile per CTA.
// The flags share the workspace's zero-filled counter region.
size_t prefill_workspace_bytes(int M, int N, int K, int sms);
// split_w: each weight as two terms in the x dtype (w rounded, and the
// rounding residue rounded; within 2^-16 of w), 128 channels per tile, one
// tile per CTA.  For calls where one rounding would exceed the accepted error.
cudaError_t launch_prefill(const MatmulArgs &a, int sms, void *workspace, size_t workspace_bytes, bool split_w,
                           cudaStream_t s);

// Tensor-core path for a moderate number of tokens (int4 codes, group size
// a multiple of 64): exact weights, group scales applied in fp32.
struct MidmPlan {
  int nt;       // tokens per CTA (UMMA N): 16, 32, 64 or 128
  int mtiles;   // token tiles
  int nblocks;  // 128-channel blocks
  int splits;   // K splits (one cluster per channel block and token tile when > 1)
  int cps;      // 64-wide K stages per split
};
bool midm_supported(const MatmulArgs &a);
MidmPlan plan_midm(int M, int N, int K, int sms);
cudaError_t launch_midm(const MatmulArgs &a, const MidmPlan &p, cudaStream_t s);

// Most tokens the few-token kernel takes when a tensor-core path can (int4
// codes, group size a multiple of 64).  Measured on the 8192 x 28672 int4
// weights: the few-token kernel is the fastest up to 64 tokens, the
// many-token kernel from 65 on (the exact tensor-core kernel trails both).
constexpr int kDecodeMaxM = 64;
// Token count from which the many-token kernel (weight rounded once to the x
// dtype) takes over; calls it cannot take within the accepted error, or with
// a scale dtype other than the x dtype, run on the exact tensor-core kernel.
constexpr int kPrefillMinM = 65;
// Where one rounding of the weight would exceed the accepted error (bf16
// below K = 4096), the many-token kernel with each weight as two terms
// (rounded weight and rounded residue, 128 channels per tile) against the
// exact tensor-core kernel, measured with bf16 int4 g128: on the K = 2048,
// N = 28672 weights 57 / 86 / 170 us against 69 / 136 / 270 us at M = 256 /
// 512 / 1024 and equal at 128; with fewer tiles it loses (M = 256, N = 4096:
// 32 tiles, 28 against 17 us; M = 128, N = 8192: 64 tiles, 25 against 17 us)
// and wins from 128 tiles (M = 1024 or 2048 on N = 4096 or 2048: 29 against
// 46 us; M = 256, K = 1024, N = 16384: 19 against 28 us).
constexpr int kSplitMinM = 129;
constexpr int kSplitMinTiles = 128;  // ceil(M / 256) x ceil(N / 128)
// The many-token kernel rounds each dequantized weight once to the x dtype
// (relative error up to 2^-11 for fp16, 2^-9 for bf16).  Over random signs
// the result's error stays near that bound / sqrt(3) of the output's RMS, a
// few times that at the maximum over a large output: within the accepted
// 1e-2 sqrt(K / 4096) of the RMS for fp16 at any K >= 512, but for bf16 only
// from K = 4096 on.  Shorter bf16 problems take the exact path.
inline bool prefill_within_tolerance(const MatmulArgs &a) { return !a.x_bf16 || a.K >= 4096; }

}  // namespace wq
