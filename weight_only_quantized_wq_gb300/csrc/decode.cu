// decode.cu -- weight-only quantized matmul for few tokens (M <= 64).
//
// The step is bound by reading the packed weights (the tiny-llm int8_gemv
// docstring makes the same point for small M), so each weight byte is read
// from HBM once, through a shared-memory ring filled by 1-D bulk copies, and
// turned into tensor-core operands in registers.
//
// Swap-AB: the weight tile (16 output channels x 16 k) is the A operand of
// mma.m16n8k16 and the tokens are its N = 8 columns, so the output channels
// fill the MMA's M dimension however few tokens there are.
//
// Grouped codes (W = 2, 4) enter the MMA as MAGIC + q, exact in fp16/bf16.
// Per group g and output column n the kernel accumulates, in fp32,
//   P = sum_k x[m,k] (MAGIC + q[k,n]) and X = sum_k x[m,k]
// (X with an extra MMA whose A operand is all ones), then adds
//   scale[g,n] * (P - (MAGIC + zero[g,n]) * X) = scale * sum_k x (q - zero)
// to the output accumulator.  The scale and zero are thus applied once per
// group on fp32 sums instead of once per weight.
// int8 codes (W = 8) are converted exactly and the per-channel scale is
// applied at the end (tiny-llm int8_matmul docstring).
//
// Split-K: when N alone gives too few CTAs, the K range is split; each CTA
// writes its fp32 partial to the workspace and the last CTA to arrive for a
// column block (atomic counter, no waiting) adds the partials in split order,
// so the result does not depend on arrival order.
#include <cstdint>
#include <cuda_runtime.h>

#include "dev.cuh"
#include "kernels.h"
#include "layout.cuh"

namespace wq {

constexpr int kDecodeWarps = 4;   // consumer warps per CTA (plus one producer warp)
constexpr int kDecodeStages = 4;  // ring depth

// Row pitch of the activation slice in shared memory: the 32-bit word count
// is 8 mod 32, which makes the 8-byte B-fragment loads of a warp conflict-free.
template <int W>
constexpr int x_pitch() {
  constexpr int words = Geo<W>::KC / 2;
  return 4 * (words + ((8 - words % 32) + 32) % 32);
}

template <int W, int MT, int TN>
struct DecodeSmem {
  static constexpr int kWBytes = kDecodeWarps * TN * 512;
  static constexpr int kXBytes = MT * 8 * x_pitch<W>();
  static constexpr int kStage = (kWBytes + kXBytes + 127) / 128 * 128;
  static constexpr int kTotal = 128 + kDecodeStages * kStage;
};

struct DecodeParams {
  const uint16_t *x;
  const uint8_t *packed;
  const void *scales;
  const uint32_t *zeros;
  float *out;
  float *partial;
  int *counters;
  uint32_t *err;
  int M, N, K, kspg, nt_total, kch, splits, cps;
  bool s_bf16;
};

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kDecodeWarps * 32) : "memory");
}

template <int W, bool BF16, int MT, int TN, bool ZERO>
__global__ void __launch_bounds__((kDecodeWarps + 1) * 32)
    decode_kernel(const DecodeParams p) {
  using G = Geo<W>;
  using S = DecodeSmem<W, MT, TN>;
  constexpr int NW = kDecodeWarps, STAGES = kDecodeStages;
  constexpr int XP = x_pitch<W>();
  constexpr bool GROUPED = (W != 8);

  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_last;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);
  uint64_t *empty = full + STAGES;
  uint8_t *ring = smem + 128;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = blockIdx.x, split = blockIdx.y;
  const int nt0 = nb * NW * TN;
  const int ntiles = min(NW * TN, p.nt_total - nt0);
  const int c0 = split * p.cps;
  const int nch = min(p.kch, c0 + p.cps) - c0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_addr(&full[i]), 1);
      mbar_init(smem_addr(&empty[i]), NW);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == NW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      const uint32_t wbytes = (uint32_t)ntiles * 512u;
      const uint32_t xrow = G::KC * 2;
      int issued = 0;
      for (int i = 0; i < nch; ++i) {
        const int st = i % STAGES;
        if (i >= STAGES && !mbar_wait(smem_addr(&empty[st]), ((i / STAGES) - 1) & 1, p.err)) break;
        const uint32_t fb = smem_addr(&full[st]);
        const uint32_t base = smem_addr(ring + st * S::kStage);
        mbar_arrive_expect_tx(fb, wbytes + (uint32_t)p.M * xrow);
        bulk_g2s(base, p.packed + ((size_t)(c0 + i) * p.nt_total + nt0) * 512, wbytes, fb, pol_w);
        const uint16_t *xs = p.x + (size_t)(c0 + i) * G::KC;
        for (int m = 0; m < p.M; ++m) bulk_g2s(base + S::kWBytes + m * XP, xs + (size_t)m * p.K, xrow, fb, pol_x);
        issued = i + 1;
      }
      // No copy may still be writing this CTA's shared memory when it exits.
      for (int i = max(0, issued - STAGES); i < issued; ++i)
        mbar_wait(smem_addr(&full[i % STAGES]), (i / STAGES) & 1, p.err);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, t = lane & 3;
  float acc[TN][MT][4];
  float accg[TN][MT][4];
  float xsum[MT][4];
  float sc[TN][2], zc[TN][2];
#pragma unroll
  for (int i = 0; i < TN; ++i)
#pragma unroll
    for (int j = 0; j < MT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][j][e] = accg[i][j][e] = 0.f;
#pragma unroll
  for (int j = 0; j < MT; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) xsum[j][e] = 0.f;

  int nrow[TN];  // row g of each of this warp's tiles (row g + 8 is nrow + 8); -1 if past N
#pragma unroll
  for (int i = 0; i < TN; ++i) {
    const int tl = warp * TN + i;
    nrow[i] = tl < ntiles ? (nt0 + tl) * 16 + g : -1;
  }

  const int kstep0 = c0 * G::KS;
  const int ksteps = nch * G::KS;
  int gi = GROUPED ? kstep0 / p.kspg : 0;           // current group
  int kleft = GROUPED ? p.kspg - kstep0 % p.kspg : 0;  // k-steps left in it
  bool need_sz = GROUPED;
  const uint16_t *sc16 = static_cast<const uint16_t *>(p.scales);
  bool ok = true;

  for (int i = 0; i < nch && ok; ++i) {
    const int st = i % STAGES;
    if (!mbar_wait(smem_addr(&full[st]), (i / STAGES) & 1, p.err)) {
      ok = false;
      break;
    }
    const uint32_t base = smem_addr(ring + st * S::kStage);
    uint4 wv[TN];
#pragma unroll
    for (int ti = 0; ti < TN; ++ti)
      wv[ti] = nrow[ti] >= 0 ? lds128(base + (warp * TN + ti) * 512 + lane * 16) : make_uint4(0, 0, 0, 0);

#pragma unroll
    for (int ks = 0; ks < G::KS; ++ks) {
      if (GROUPED && need_sz) {
        // scale and (MAGIC + zero) of group gi for rows g and g + 8 of each tile
#pragma unroll
        for (int ti = 0; ti < TN; ++ti)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int n = nrow[ti] < 0 ? 0 : nrow[ti] + 8 * r;
            sc[ti][r] = half_bits_to_float(__ldg(sc16 + (size_t)gi * p.N + n), p.s_bf16);
            uint32_t z = 1u << (W - 1);
            if (ZERO) z = (__ldg(p.zeros + (size_t)(gi / G::V) * p.N + n) >> ((gi % G::V) * W)) & ((1u << W) - 1u);
            zc[ti][r] = Magic<BF16>::kValue + (float)z;
          }
        need_sz = false;
      }
      uint32_t b[MT][2];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const uint2 v = lds64(base + S::kWBytes + (mt * 8 + g) * XP + ks * 32 + t * 8);
        b[mt][0] = v.x;
        b[mt][1] = v.y;
      }
      if (GROUPED) {
        constexpr uint32_t one = Magic<BF16>::kOnePair;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) mma16816<BF16>(xsum[mt], one, one, one, one, b[mt][0], b[mt][1]);
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
      if (GROUPED) {
        const int kdone = i * G::KS + ks + 1;
        if (--kleft == 0 || kdone == ksteps) {
#pragma unroll
          for (int ti = 0; ti < TN; ++ti)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int r = e >> 1;
                acc[ti][mt][e] += sc[ti][r] * (accg[ti][mt][e] - zc[ti][r] * xsum[mt][e & 1]);
                accg[ti][mt][e] = 0.f;
              }
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) xsum[mt][e] = 0.f;
          ++gi;
          kleft = p.kspg;
          need_sz = true;
        }
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
    if (nrow[ti] < 0) continue;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int n = nrow[ti] + 8 * r;
      const float s8 = (W == 8 && p.splits == 1) ? __ldg(sc32 + n) : 1.f;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int m = mt * 8 + 2 * t + c;
          if (m < p.M) dst[(size_t)m * p.N + n] = acc[ti][mt][2 * r + c] * s8;
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
  const int rows = ntiles * 16, n0 = nt0 * 16;
  for (int idx = threadIdx.x; idx < p.M * rows; idx += NW * 32) {
    const int m = idx / rows, n = n0 + idx % rows;
    float v = 0.f;
    for (int sp = 0; sp < p.splits; ++sp) v += __ldcg(p.partial + ((size_t)sp * p.M + m) * p.N + n);
    if (W == 8) v *= __ldg(sc32 + n);
    p.out[(size_t)m * p.N + n] = v;
  }
  if (threadIdx.x == 0) p.counters[nb] = 0;
}

// ------------------------------------------------------------------ host side
// The workspace starts with one arrival counter per column block, sized for
// the largest block count any M can use (4 tiles per CTA), so that counters
// never share bytes with the fp32 partials that follow, whatever M a call has.
size_t decode_counter_bytes(int N) {
  const size_t nb_max = (size_t)(N / 16 + kDecodeWarps - 1) / kDecodeWarps;
  return (nb_max * sizeof(int) + 255) / 256 * 256;
}

static int tn_for(int mt) { return mt >= 8 ? 1 : (mt >= 4 ? 2 : 4); }

DecodePlan plan_decode(int M, int N, int K, int w_bit, int sms) {
  DecodePlan p{};
  const int rows = M < 64 ? M : 64;
  p.mt = rows <= 8 ? 1 : rows <= 16 ? 2 : rows <= 32 ? 4 : 8;
  p.tn = tn_for(p.mt);
  const int kc = 256 / w_bit;
  const int nt = N / 16;
  const int kch = K / kc;
  const int tiles_per_cta = kDecodeWarps * p.tn;
  p.nblocks = (nt + tiles_per_cta - 1) / tiles_per_cta;
  // Pick the split that minimises (busiest SM's chunk-tiles) + a small cost per partial.
  double best = 1e300;
  int best_s = 1;
  const int smax = kch < 32 ? kch : 32;
  for (int s = 1; s <= smax; ++s) {
    const int cps = (kch + s - 1) / s;
    const int sreal = (kch + cps - 1) / cps;
    const long ctas = (long)p.nblocks * sreal;
    const long per_sm = (ctas + sms - 1) / sms;
    double cost = (double)per_sm * cps * tiles_per_cta;
    cost += sreal > 1 ? 0.02 * sreal * tiles_per_cta : 0.0;
    if (cost < best * 0.999) {
      best = cost;
      best_s = sreal;
    }
  }
  p.cps = (kch + best_s - 1) / best_s;
  p.splits = (kch + p.cps - 1) / p.cps;
  p.workspace = p.splits > 1 ? decode_counter_bytes(N) + (size_t)p.splits * rows * N * sizeof(float) : 0;
  return p;
}

template <int W, bool BF16, int MT, bool ZERO>
static cudaError_t launch_t(const DecodeParams &dp, const DecodePlan &p, cudaStream_t s) {
  constexpr int TN = (MT >= 8) ? 1 : (MT >= 4 ? 2 : 4);
  using S = DecodeSmem<W, MT, TN>;
  auto kern = decode_kernel<W, BF16, MT, TN, ZERO>;
  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kTotal);
    if (e != cudaSuccess) return e;
    attr_set[dev] = 1;
  }
  dim3 grid(p.nblocks, p.splits);
  kern<<<grid, (kDecodeWarps + 1) * 32, S::kTotal, s>>>(dp);
  return cudaGetLastError();
}

template <int W, bool BF16, bool ZERO>
static cudaError_t launch_mt(const DecodeParams &dp, const DecodePlan &p, cudaStream_t s) {
  switch (p.mt) {
    case 1: return launch_t<W, BF16, 1, ZERO>(dp, p, s);
    case 2: return launch_t<W, BF16, 2, ZERO>(dp, p, s);
    case 4: return launch_t<W, BF16, 4, ZERO>(dp, p, s);
    case 8: return launch_t<W, BF16, 8, ZERO>(dp, p, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode(const MatmulArgs &a, const DecodePlan &p, void *workspace, cudaStream_t s) {
  DecodeParams dp{};
  dp.x = static_cast<const uint16_t *>(a.x);
  dp.packed = static_cast<const uint8_t *>(a.packed);
  dp.scales = a.scales;
  dp.zeros = a.zeros;
  dp.out = a.out;
  dp.err = a.err;
  dp.M = a.M;
  dp.N = a.N;
  dp.K = a.K;
  dp.kspg = a.group_size / 16;
  dp.nt_total = a.N / 16;
  dp.kch = a.K / (256 / a.w_bit);
  dp.splits = p.splits;
  dp.cps = p.cps;
  dp.s_bf16 = a.s_bf16;
  if (p.splits > 1) {
    dp.counters = static_cast<int *>(workspace);
    dp.partial = reinterpret_cast<float *>(static_cast<char *>(workspace) + decode_counter_bytes(a.N));
  }
  const bool z = a.zeros != nullptr;
  if (a.w_bit == 8) return a.x_bf16 ? launch_mt<8, true, false>(dp, p, s) : launch_mt<8, false, false>(dp, p, s);
  if (a.w_bit == 4) {
    if (a.x_bf16) return z ? launch_mt<4, true, true>(dp, p, s) : launch_mt<4, true, false>(dp, p, s);
    return z ? launch_mt<4, false, true>(dp, p, s) : launch_mt<4, false, false>(dp, p, s);
  }
  if (a.w_bit == 2) {
    if (a.x_bf16) return z ? launch_mt<2, true, true>(dp, p, s) : launch_mt<2, true, false>(dp, p, s);
    return z ? launch_mt<2, false, true>(dp, p, s) : launch_mt<2, false, false>(dp, p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace wq
