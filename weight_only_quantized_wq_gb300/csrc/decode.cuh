// decode.cuh -- weight-only quantized matmul for few tokens (M <= 64).
//
// The step is bound by reading the packed weights (the tiny-llm int8_gemv
// docstring makes the same point for small M), so each weight byte is read
// from HBM once, through a shared-memory ring, and turned into tensor-core
// operands in registers.
//
// Swap-AB: the weight tile (16 output channels x 16 k) is the A operand of
// mma.m16n8k16 and the tokens are its N = 8 columns, so the output channels
// fill the MMA's M dimension however few tokens there are.
//
// Ring stage = one chunk row (KC values of K) for the CTA's 16*NW*TN output
// channels: the packed weights (one 1-D bulk copy), the activation slice,
// and the scale / zero rows of the groups the chunk touches (three 2-D tensor
// copies through tensor maps).  One lane of the producer warp issues all four
// copies of a stage.
// A prep warp turns each stage's scale / zero rows into per-column pairs
// (s, -s * (MAGIC + zero)) so that the consumer warps fold a finished group
// into their accumulators with two FMAs per value.
//
// Grouped codes (W = 2, 4) enter the MMA as MAGIC + q, exact in fp16/bf16.
// Per group g and output column n the kernel accumulates in fp32
//   P = sum_k x[m,k] (MAGIC + q[k,n])   (tensor cores)
//   X = sum_k x[m,k]                    (tensor cores, A operand all ones)
// and adds scale[g,n] * (P - (MAGIC + zero[g,n]) * X) = scale * sum_k x (q - zero)
// to the output accumulator: scale and zero cost once per group, not per weight.
// int8 codes (W = 8) are converted exactly and the per-channel scale is
// applied at the end (tiny-llm int8_matmul docstring).
//
// Split-K: when the column blocks alone leave SMs idle, the K range is split;
// each CTA writes its fp32 partial to the workspace and the last CTA to
// arrive for a column block (atomic counter, no waiting) adds the partials in
// split order, so the result does not depend on arrival order.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "dev.cuh"
#include "kernels.h"
#include "layout.cuh"

namespace wq {

constexpr int kDecodeWarps = 4;   // consumer warps per CTA (plus a producer and a prep warp)
constexpr int kDecodeThreads = (kDecodeWarps + 2) * 32;
// Ring depth: about 40 KB of weights in flight per CTA.
__host__ __device__ constexpr int decode_stages(int tn) { return tn >= 4 ? 5 : 8; }
constexpr int kDecodeHeader = 256;  // mbarriers in front of the ring
// Resident CTAs per SM the register budget is sized for: wide accumulator
// sets (token tiles x weight tiles >= 8) get two CTAs per SM and no spills.
__host__ __device__ constexpr int decode_min_blocks(int mt, int tn) { return mt * tn >= 8 ? 2 : 3; }

// Row pitch of the activation slice in shared memory: the 32-bit word count
// is 8 mod 32, which makes the 8-byte B-fragment loads of a warp conflict-free.
template <int W>
__host__ __device__ constexpr int x_pitch() {
  return 4 * (Geo<W>::KC / 2 + ((8 - (Geo<W>::KC / 2) % 32) + 32) % 32);
}

struct DecodeParams {
  CUtensorMap tm_x;  // x (M, K) 16-bit; box (x_pitch/2, 8*MT): the row pitch padding is real data or zeros
  CUtensorMap tm_s;  // scales (G, N) 16-bit; box (cols, gcap)
  CUtensorMap tm_z;  // zeros (ceil(G/V), N) 32-bit; box (cols, 2)
  const uint16_t *x;
  const uint8_t *packed;
  const void *scales;
  const uint32_t *zeros;
  float *out;
  float *partial;
  int *counters;
  uint32_t *err;
  int M, N, K, gs, kspg, nt_total, kch, splits, cps, gcap, stage_bytes;
  bool s_bf16;
};

template <int W, int MT, int TN>
struct DecodeLayout {
  static constexpr int kCols = kDecodeWarps * TN * 16;  // output channels per CTA
  static constexpr int kWBytes = kCols * Geo<W>::KC * W / 8;
  static constexpr int kXBytes = MT * 8 * x_pitch<W>();
  static constexpr int kXOff = kWBytes;
  static constexpr int kSOff = (kXOff + kXBytes + 127) / 128 * 128;
  // Stage = weights | x | scale rows (gcap) | two zero rows | per group row:
  // (s, -s*(MAGIC+z)) for each column.
  static constexpr int kPRow = kCols * 8;
  static __host__ __device__ constexpr int z_off(int gcap) { return (kSOff + gcap * kCols * 2 + 127) / 128 * 128; }
  static __host__ __device__ constexpr int p_off(int gcap, bool zero) {
    return (z_off(gcap) + (zero ? 2 * kCols * 4 : 0) + 127) / 128 * 128;
  }
  static __host__ __device__ constexpr int stage_bytes(int gcap, bool grouped, bool zero) {
    return grouped ? (p_off(gcap, zero) + gcap * kPRow + 127) / 128 * 128 : kSOff;
  }
  // Bytes the tensor copies of one stage deliver (besides the weights).
  static __host__ __device__ constexpr int tma_bytes(int gcap, bool grouped, bool zero) {
    return kXBytes + (grouped ? gcap * kCols * 2 + (zero ? 2 * kCols * 4 : 0) : 0);
  }
};

__device__ __forceinline__ void sts64(uint32_t a, float x, float y) {
  asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(x), "f"(y) : "memory");
}
__device__ __forceinline__ float2 lds64f(uint32_t a) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
  return v;
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kDecodeWarps * 32) : "memory");
}

template <int W, bool BF16, int MT, int TN, bool ZERO>
__global__ void __launch_bounds__(kDecodeThreads, decode_min_blocks(MT, TN))
    decode_kernel(const __grid_constant__ DecodeParams p) {
  using G = Geo<W>;
  using L = DecodeLayout<W, MT, TN>;
  constexpr int NW = kDecodeWarps, STAGES = decode_stages(TN);
  constexpr int XP = x_pitch<W>();
  constexpr bool GROUPED = (W != 8);
  constexpr int COLS = L::kCols;

  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_last;
  __shared__ volatile int s_abort;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);
  uint64_t *empty = full + STAGES;
  uint64_t *ready = empty + STAGES;
  uint8_t *ring = smem + kDecodeHeader;
  static_assert(3 * STAGES * 8 <= kDecodeHeader, "barriers do not fit the header");
  const int SB = p.stage_bytes;
  const int zoff = L::z_off(p.gcap);
  const int poff = L::p_off(p.gcap, ZERO);
  (void)zoff;
  (void)poff;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = blockIdx.x, split = blockIdx.y;
  const int nt0 = nb * NW * TN;
  const int ntiles = min(NW * TN, p.nt_total - nt0);
  const int n0 = nt0 * 16;
  const int c0 = split * p.cps;
  const int nch = min(p.kch, c0 + p.cps) - c0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_addr(&full[i]), 1);
      // a stage is free again once the consumers and (grouped codes) the prep warp are done with it
      mbar_init(smem_addr(&empty[i]), GROUPED ? NW + 1 : NW);
      mbar_init(smem_addr(&ready[i]), 1);
    }
    s_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == NW) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_w = policy_evict_first();
    const uint32_t wbytes = (uint32_t)ntiles * 512u;
    const uint32_t tbytes = (uint32_t)L::tma_bytes(p.gcap, GROUPED, ZERO);
    int issued = 0;
    if (lane == 0) {
      for (int i = 0; i < nch; ++i) {
        const int st = i % STAGES;
        if (i >= STAGES && !mbar_wait(smem_addr(&empty[st]), ((i / STAGES) - 1) & 1, p.err, &s_abort)) break;
        const uint32_t fb = smem_addr(&full[st]);
        const uint32_t base = smem_addr(ring + st * SB);
        const int kc = c0 + i;
        mbar_arrive_expect_tx(fb, wbytes + tbytes);
        bulk_g2s(base, p.packed + ((size_t)kc * p.nt_total + nt0) * 512, wbytes, fb, pol_w);
        tma_load_2d(base + L::kXOff, &p.tm_x, kc * G::KC, 0, fb);
        if (GROUPED) {
          const int g0 = kc * G::KC / p.gs;
          tma_load_2d(base + L::kSOff, &p.tm_s, n0, g0, fb);
          if (ZERO) tma_load_2d(base + zoff, &p.tm_z, n0, g0 / G::V, fb);
        }
        issued = i + 1;
      }
    }
    // No copy may still be writing this CTA's shared memory when it exits.
    if (lane == 0)
      for (int i = max(0, issued - STAGES); i < issued; ++i)
        mbar_wait(smem_addr(&full[i % STAGES]), (i / STAGES) & 1, p.err, nullptr);
    return;
  }

  if (warp == NW + 1) {
    // ------------------------------------------------------------ prep
    // (s, -s * (MAGIC + zero)) for every column of each group that ends in
    // this stage (or is cut off by the end of this CTA's K range).
    if (GROUPED) {
      const int cols = ntiles * 16;
      for (int i = 0; i < nch; ++i) {
        const int st = i % STAGES;
        bool ok = true;
        if (lane == 0) ok = mbar_wait(smem_addr(&full[st]), (i / STAGES) & 1, p.err, &s_abort);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        const uint32_t base = smem_addr(ring + st * SB);
        const int kc = c0 + i;
        const int g0 = kc * G::KC / p.gs;
        const int kend = (kc + 1) * G::KC;  // first k past this stage
        const int glast = (kend - 1) / p.gs;
        for (int g = g0; g <= glast; ++g) {
          if ((g + 1) * p.gs > kend && i != nch - 1) continue;  // group continues in the next stage
          const int r = g - g0;
          const uint32_t srow = base + L::kSOff + r * COLS * 2;
          const uint32_t zrow = base + zoff + (g / G::V - g0 / G::V) * COLS * 4;
          const uint32_t prow = base + poff + r * L::kPRow;
          const int zshift = (g % G::V) * W;
          for (int c = lane; c < cols; c += 32) {
            const float sv = half_bits_to_float(lds16(srow + c * 2), p.s_bf16);
            uint32_t z = 1u << (W - 1);
            if (ZERO) z = (lds32(zrow + c * 4) >> zshift) & ((1u << W) - 1u);
            sts64(prow + c * 8, sv, -sv * (Magic<BF16>::kValue + (float)z));
          }
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_addr(&ready[st]));
          mbar_arrive(smem_addr(&empty[st]));  // done reading this stage's scale / zero rows
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, t = lane & 3;
  float acc[TN][MT][4];
  float accg[TN][MT][4];
  float xs[MT][4];
#pragma unroll
  for (int j = 0; j < MT; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) xs[j][e] = 0.f;
#pragma unroll
  for (int i = 0; i < TN; ++i)
#pragma unroll
    for (int j = 0; j < MT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][j][e] = accg[i][j][e] = 0.f;

  const int kstep0 = c0 * G::KS;
  const int ksteps = nch * G::KS;
  int gi = GROUPED ? kstep0 / p.kspg : 0;               // current group
  int kleft = GROUPED ? p.kspg - kstep0 % p.kspg : 0;  // k-steps left in it

  // A barrier test returns after a long latency even when the phase is
  // complete, so a non-blocking test of each stage's barrier is issued one
  // stage early and its answer is only read when that stage starts.
  bool next_ready = nch > 0 && mbar_test_wait(smem_addr(&full[0]), 0);
  for (int i = 0; i < nch; ++i) {
    const int st = i % STAGES;
    // The weights and x are ready when the copies land; the prep warp's (s, z)
    // pairs are only needed at a group's end, so that wait comes later.
    if (!next_ready && !mbar_wait(smem_addr(&full[st]), (i / STAGES) & 1, p.err, &s_abort)) break;
    if (i + 1 < nch) next_ready = mbar_test_wait(smem_addr(&full[(i + 1) % STAGES]), ((i + 1) / STAGES) & 1);
    const int gi_stage = gi;  // group of this stage's first k: the stage's group row 0
    const uint32_t base = smem_addr(ring + st * SB);
    uint4 wv[TN];
#pragma unroll
    for (int ti = 0; ti < TN; ++ti)
      wv[ti] = (warp * TN + ti) < ntiles ? lds128(base + (warp * TN + ti) * 512 + lane * 16) : make_uint4(0, 0, 0, 0);

#pragma unroll
    for (int ks = 0; ks < G::KS; ++ks) {
      uint32_t b[MT][2];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const uint2 v = lds64(base + L::kXOff + (mt * 8 + g) * XP + ks * 32 + t * 8);
        b[mt][0] = v.x;
        b[mt][1] = v.y;
        if (GROUPED) {
          constexpr uint32_t one = Magic<BF16>::kOnePair;
          mma16816<BF16>(xs[mt], one, one, one, one, v.x, v.y);
        }
      }
      const int h = ks / G::WK, j = ks % G::WK;
#pragma unroll
      for (int ti = 0; ti < TN; ++ti) {
        const uint32_t wg = h ? wv[ti].z : wv[ti].x;
        const uint32_t wg8 = h ? wv[ti].w : wv[ti].y;
        uint32_t a0, a1, a2, a3;
        if constexpr (W == 8) {
          a0 = int8_pair<BF16>(wg, 0);
          a1 = int8_pair<BF16>(wg8, 0);
          a2 = int8_pair<BF16>(wg, 1);
          a3 = int8_pair<BF16>(wg8, 1);
        } else {
          a0 = code_pair<W, BF16>(wg, 2 * j);
          a1 = code_pair<W, BF16>(wg8, 2 * j);
          a2 = code_pair<W, BF16>(wg, 2 * j + 1);
          a3 = code_pair<W, BF16>(wg8, 2 * j + 1);
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          if (GROUPED)
            mma16816<BF16>(accg[ti][mt], a0, a1, a2, a3, b[mt][0], b[mt][1]);
          else
            mma16816<BF16>(acc[ti][mt], a0, a1, a2, a3, b[mt][0], b[mt][1]);
        }
      }
      if (GROUPED && (--kleft == 0 || i * G::KS + ks + 1 == ksteps)) {
        // Group done: fold P and X of this group into the output accumulators.
        mbar_wait(smem_addr(&ready[st]), (i / STAGES) & 1, p.err, &s_abort);
        const int r = gi - gi_stage;  // group row inside this stage
        const uint32_t prow = base + poff + r * L::kPRow;
#pragma unroll
        for (int ti = 0; ti < TN; ++ti)
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const float2 sz = lds64f(prow + ((warp * TN + ti) * 16 + g + 8 * rr) * 8);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              float *a = &acc[ti][mt][2 * rr];
              float *pg = &accg[ti][mt][2 * rr];
              a[0] = fmaf(sz.y, xs[mt][0], fmaf(sz.x, pg[0], a[0]));
              a[1] = fmaf(sz.y, xs[mt][1], fmaf(sz.x, pg[1], a[1]));
              pg[0] = 0.f;
              pg[1] = 0.f;
            }
          }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) xs[mt][e] = 0.f;
        ++gi;
        kleft = p.kspg;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty[st]));
  }

  // -------------------------------------------------------------- epilogue
  const float *sc32 = static_cast<const float *>(p.scales);
  float *dst = p.splits == 1 ? p.out : p.partial + (size_t)split * p.M * p.N;
#pragma unroll
  for (int ti = 0; ti < TN; ++ti) {
    if (warp * TN + ti >= ntiles) continue;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int n = n0 + (warp * TN + ti) * 16 + g + 8 * rr;
      const float s8 = (W == 8 && p.splits == 1) ? __ldg(sc32 + n) : 1.f;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int m = mt * 8 + 2 * t + c;
          if (m < p.M) dst[(size_t)m * p.N + n] = acc[ti][mt][2 * rr + c] * s8;
        }
    }
  }
  if (p.splits == 1) return;

  // Last CTA of this column block adds the partials in split order.
  __threadfence();
  consumer_sync();
  if (threadIdx.x == 0) s_last = (atomicAdd(&p.counters[nb], 1) == p.splits - 1);
  consumer_sync();
  if (!s_last) return;
  __threadfence();
  // Four consecutive columns per thread, every split's partial loaded before any add.
  const int quads = ntiles * 4;  // rows of 16 columns -> 4 float4 each
  for (int idx = threadIdx.x; idx < p.M * quads; idx += NW * 32) {
    const int m = idx / quads, n = n0 + (idx % quads) * 4;
    float4 part[8];
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sp0 = 0; sp0 < p.splits; sp0 += 8) {
      const int cnt = min(8, p.splits - sp0);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (u < cnt) part[u] = __ldcg(reinterpret_cast<const float4 *>(p.partial + ((size_t)(sp0 + u) * p.M + m) * p.N + n));
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (u < cnt) {
          v.x += part[u].x;
          v.y += part[u].y;
          v.z += part[u].z;
          v.w += part[u].w;
        }
    }
    if (W == 8) {
      const float4 s4 = __ldg(reinterpret_cast<const float4 *>(sc32 + n));
      v.x *= s4.x;
      v.y *= s4.y;
      v.z *= s4.z;
      v.w *= s4.w;
    }
    *reinterpret_cast<float4 *>(p.out + (size_t)m * p.N + n) = v;
  }
  if (threadIdx.x == 0) p.counters[nb] = 0;
}

template <int W, bool BF16, int MT, int TN, bool ZERO>
cudaError_t launch_decode_t(const DecodeParams &dp, const DecodePlan &p, cudaStream_t s) {
  auto kern = decode_kernel<W, BF16, MT, TN, ZERO>;
  const int smem = kDecodeHeader + decode_stages(TN) * dp.stage_bytes;
  static int attr_bytes[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && attr_bytes[dev] < smem) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_bytes[dev] = smem;
  }
  dim3 grid(p.nblocks, p.splits);
  kern<<<grid, kDecodeThreads, smem, s>>>(dp);
  return cudaGetLastError();
}

// Per-W launcher (one translation unit per W keeps the build parallel).
template <int W>
cudaError_t launch_decode_w(const DecodeParams &dp, const DecodePlan &p, bool bf16, bool zero, cudaStream_t s);

#define WQ_DECODE_CASE(W, BF, MT, TN, Z) \
  if (bf16 == BF && zero == Z && p.mt == MT && p.tn == TN) return launch_decode_t<W, BF, MT, TN, Z>(dp, p, s);

}  // namespace wq
