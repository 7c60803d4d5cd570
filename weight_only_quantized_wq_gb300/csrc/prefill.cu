// prefill.cu -- weight-only quantized matmul for many tokens (tensor cores, tcgen05).
//
// At large M the step is bound by the multiply-adds, so the weights are
// dequantized once per 256-token tile into shared memory in the operand
// layout of the 5th-generation tensor cores, and tcgen05.mma accumulates
// y^T-free:  D[m, n] (TMEM, fp32) += x[m, k] * w[k, n]  over 64-wide K steps.
//
// CTA tile: 256 tokens x 256 output channels, K step 64: two 128 x 256
// accumulators (the whole 512-column TMEM) share each dequantized weight
// tile, so every weight is dequantized once per 256 tokens.
// Roles (10 warps):
//   warp 0      producer: per stage one TMA copy of the x tile (256 x 64,
//               128-byte swizzle), one 1-D bulk copy of the packed weights
//               (256 channels x 64 k), and TMA copies of the scale and zero
//               rows of the stage's group;
//   warp 1      TMEM allocation and the single thread that issues tcgen05.mma;
//   warps 2..9  dequant: w = (q - zero) * scale rounded once to the x dtype,
//               written K-major with the 128-byte swizzle the MMA reads;
//   warps 4..7  (after the main loop) epilogue: tcgen05.ld of the fp32
//               accumulator, one token row per thread, stored to y.
// The scale and zero are applied to the weight (one rounding to bf16/fp16),
// since a per-group rescale of a 128 x 256 TMEM accumulator would cost more
// than the tensor cores gain.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "dev.cuh"
#include "kernels.h"
#include "layout.cuh"
#include "tc.cuh"

namespace wq {

namespace pf {

constexpr int UM = 128;   // UMMA M (tokens per accumulator)
constexpr int BN = 256;   // output channels per CTA (UMMA N)
constexpr int BK = 64;    // K per stage: one 128-byte swizzle atom of bf16
constexpr int STAGES = 3;
constexpr int BSTAGES = 2;            // dequantized B buffers
constexpr int DQ_WARPS = 8;
constexpr int THREADS = (2 + DQ_WARPS) * 32;
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr int W_BYTES = BN * BK / 2;  // 8 KB of packed int4
constexpr int S_BYTES = BN * 2;       // one scale row
constexpr int Z_BYTES = BN * 4;       // one zero-word row
constexpr int HEADER = 1024;          // mbarriers + TMEM address

// Geometry for MS accumulators of 128 tokens each (token tile BM = 128 MS).
template <int MS>
struct Cfg {
  static constexpr int MSUB = MS;
  static constexpr int BM = UM * MS;                  // tokens per CTA
  static constexpr int A_BYTES = BM * BK * 2;         // x tile: 16 or 32 KB
  // stage = A | W | S | Z, 1024-byte aligned (the swizzle atom of A)
  static constexpr int ST_A = 0, ST_W = A_BYTES, ST_S = ST_W + W_BYTES, ST_Z = ST_S + S_BYTES;
  static constexpr int STAGE_BYTES = (ST_Z + Z_BYTES + 1023) / 1024 * 1024;
  static constexpr int SMEM = HEADER + STAGES * STAGE_BYTES + BSTAGES * B_BYTES;
  static constexpr int TMEM_COLS = BN * MS;           // 256 or 512
};

struct Params {
  CUtensorMap tm_x;  // x (M, K) 16-bit, box (64, 256), 128-byte swizzle
  CUtensorMap tm_s;  // scales (G, N) 16-bit, box (256, 1)
  CUtensorMap tm_z;  // zeros (ceil(G/8), N) 32-bit, box (256, 1)
  const uint8_t *packed;
  void *out;
  int out_type;  // OutType
  uint32_t *err;
  int M, N, K, gs, nt_total;
};

template <bool BF16>
__device__ __forceinline__ uint32_t mul2(uint32_t a, uint32_t b) {
  uint32_t d;
  if constexpr (BF16)
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// 32 consecutive fp32 columns of this warp's TMEM lane quarter.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  tc::ld32(taddr, r);
  tc::wait_ld();
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

template <bool BF16, bool ZERO, int MS>
__global__ void __launch_bounds__(THREADS, 1) prefill_kernel(const __grid_constant__ Params p) {
  using C = Cfg<MS>;
  constexpr int MSUB = C::MSUB, BM = C::BM, A_BYTES = C::A_BYTES, STAGE_BYTES = C::STAGE_BYTES;
  constexpr int ST_A = C::ST_A, ST_W = C::ST_W, ST_S = C::ST_S, ST_Z = C::ST_Z, TMEM_COLS = C::TMEM_COLS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment (of the shared-window address) for the swizzled tiles
  uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);          // TMA data of a stage landed
  uint64_t *empty = full + STAGES;                                // MMA done with a stage
  uint64_t *bfull = empty + STAGES;                               // dequantized B written
  uint64_t *bempty = bfull + BSTAGES;                             // MMA done with a B buffer
  uint64_t *accfull = bempty + BSTAGES;                           // accumulator complete
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accfull + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  uint8_t *ring = smem + HEADER;
  uint8_t *bbuf = ring + STAGES * STAGE_BYTES;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Token tiles vary fastest across the grid, so the CTAs that read the same
  // 256-channel weight block run at about the same time and share it in L2.
  const int mb = blockIdx.x, nb = blockIdx.y;
  const int n0 = nb * BN, m0 = mb * BM;
  const int nt0 = n0 / 16;
  const int ntiles = min(BN / 16, p.nt_total - nt0);
  const int nk = p.K / BK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_addr(&full[i]), 1);
      mbar_init(smem_addr(&empty[i]), 1);
    }
    for (int i = 0; i < BSTAGES; ++i) {
      mbar_init(smem_addr(&bfull[i]), DQ_WARPS);
      mbar_init(smem_addr(&bempty[i]), 1);
    }
    mbar_init(smem_addr(accfull), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tc::alloc(smem_addr(tmem_slot), TMEM_COLS);
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int st = i % STAGES;
        if (i >= STAGES && !mbar_wait(smem_addr(&empty[st]), ((i / STAGES) - 1) & 1, p.err, abort_flag)) break;
        const uint32_t fb = smem_addr(&full[st]);
        const uint32_t base = smem_addr(ring + st * STAGE_BYTES);
        const int g = i * BK / p.gs;
        mbar_arrive_expect_tx(fb, A_BYTES + ntiles * 512 + S_BYTES + (ZERO ? Z_BYTES : 0));
        tma_load_2d(base + ST_A, &p.tm_x, i * BK, m0, fb);
        bulk_g2s(base + ST_W, p.packed + ((size_t)i * p.nt_total + nt0) * 512, ntiles * 512, fb, pol);
        tma_load_2d(base + ST_S, &p.tm_s, n0, g, fb);
        if (ZERO) tma_load_2d(base + ST_Z, &p.tm_z, n0, g / 8, fb);
        issued = i + 1;
      }
      for (int i = max(0, issued - STAGES); i < issued; ++i)
        mbar_wait(smem_addr(&full[i % STAGES]), (i / STAGES) & 1, p.err, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id = tc::idesc<BF16>(UM, BN);
      for (int i = 0; i < nk; ++i) {
        const int st = i % STAGES, sb = i % BSTAGES;
        if (!mbar_wait(smem_addr(&full[st]), (i / STAGES) & 1, p.err, abort_flag)) break;
        if (!mbar_wait(smem_addr(&bfull[sb]), (i / BSTAGES) & 1, p.err, abort_flag)) break;
        tc::fence_after();
        const uint32_t a0 = smem_addr(ring + st * STAGE_BYTES + ST_A);
        const uint32_t b0 = smem_addr(bbuf + sb * B_BYTES);
#pragma unroll
        for (int h = 0; h < MSUB; ++h)
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc::mma(tmem + h * BN, tc::sw128_desc(a0 + h * (UM * 128) + kk * 32), tc::sw128_desc(b0 + kk * 32), id,
                 (i | kk) != 0);
        tc::commit(smem_addr(&empty[st]));
        tc::commit(smem_addr(&bempty[sb]));
      }
      tc::commit(smem_addr(accfull));  // every MMA issued above has completed when this fires
    }
  } else {
    // ------------------------------------------------------------ dequant (warps 2..9)
    const int dq = threadIdx.x - 64;  // 0 .. 255
    constexpr uint32_t MAGIC = Magic<BF16>::kPair;
    for (int i = 0; i < nk; ++i) {
      const int st = i % STAGES, sb = i % BSTAGES;
      if (!mbar_wait(smem_addr(&full[st]), (i / STAGES) & 1, p.err, abort_flag)) break;
      if (i >= BSTAGES && !mbar_wait(smem_addr(&bempty[sb]), ((i / BSTAGES) - 1) & 1, p.err, abort_flag)) break;
      const uint32_t base = smem_addr(ring + st * STAGE_BYTES);
      const uint32_t bdst = smem_addr(bbuf + sb * B_BYTES);
      const int g = i * BK / p.gs;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int pr = dq + half * 256;  // (tile, lane) pair 0..511
        const int tile = pr >> 5, ln = pr & 31;
        if (tile < ntiles) {
          const uint4 wv = lds128(base + ST_W + tile * 512 + ln * 16);
          const int gq = ln >> 2, tq = ln & 3;
          const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int col = tile * 16 + gq + 8 * r;  // row of B (output channel within the tile)
            const uint16_t sbits = lds16(base + ST_S + col * 2);
            uint32_t z = 8;
            if (ZERO) z = (lds32(base + ST_Z + col * 4) >> ((g % 8) * 4)) & 15u;
            const uint32_t zz = ((MAGIC & 0xFFFFu) + z) * 0x00010001u;  // (MAGIC + z) in both halves
            const uint32_t ss = (uint32_t)sbits * 0x00010001u;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const uint32_t w = w4[2 * u + r];
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const uint32_t lo = mul2<BF16>(sub_pair<BF16>(code_pair<4, BF16>(w, 2 * j), zz), ss);
                const uint32_t hi = mul2<BF16>(sub_pair<BF16>(code_pair<4, BF16>(w, 2 * j + 1), zz), ss);
                const int k = 32 * u + 16 * j + 4 * tq;
                sts64(bdst + tc::sw128_off(col, k), lo, hi);
              }
            }
          }
        }
      }
      fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&bfull[sb]));
    }
    // ---------------------------------------------------------- epilogue (warps 4..7)
    if (warp >= 4 && warp < 8) {
      const int q = warp & 3;  // TMEM lane quarter this warp may access
      mbar_wait(smem_addr(accfull), 0, p.err, nullptr);
      tc::fence_after();
      for (int h = 0; h < MSUB; ++h) {
        const int m = m0 + h * UM + q * 32 + lane;
        for (int c = 0; c < BN; c += 32) {
          float v[32];
          tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + h * BN + c, v);
          if (m < p.M) {
            const size_t row = (size_t)m * p.N + n0 + c;
            if (n0 + c + 32 <= p.N) {
#pragma unroll
              for (int j = 0; j < 32; j += 4)
                store_out4(p.out, row + j, make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]), p.out_type);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (n0 + c + j < p.N) store_out1(p.out, row + j, v[j], p.out_type);
            }
          }
        }
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace pf

// ------------------------------------------------------------------ host side
bool prefill_supported(const MatmulArgs &a) {
  return a.w_bit == 4 && a.group_size % pf::BK == 0 && a.K % pf::BK == 0 && a.x_bf16 == a.s_bf16;
}

template <bool BF16, bool ZERO, int MS>
static cudaError_t launch_t(const pf::Params &pp, dim3 grid, cudaStream_t s) {
  auto kern = pf::prefill_kernel<BF16, ZERO, MS>;
  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  const int smem = pf::Cfg<MS>::SMEM + 1024;  // + slack for the 1024-byte alignment of the ring
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = 1;
  }
  kern<<<grid, pf::THREADS, smem, s>>>(pp);
  return cudaGetLastError();
}

template <int MS>
static cudaError_t launch_ms(const pf::Params &pp, dim3 grid, bool bf16, bool z, cudaStream_t s) {
  if (bf16) return z ? launch_t<true, true, MS>(pp, grid, s) : launch_t<true, false, MS>(pp, grid, s);
  return z ? launch_t<false, true, MS>(pp, grid, s) : launch_t<false, false, MS>(pp, grid, s);
}

cudaError_t launch_prefill(const MatmulArgs &a, cudaStream_t s) {
  pf::Params pp{};
  const int G = a.K / a.group_size;
  // One 128-token accumulator per CTA up to 128 tokens, two (256 tokens) beyond.
  const int ms = a.M <= pf::UM ? 1 : 2;
  const int bm = pf::UM * ms;
  if (!encode_2d(&pp.tm_x, a.x, 2, (uint64_t)a.K, (uint64_t)a.M, pf::BK, (uint32_t)bm, 128))
    return cudaErrorInvalidValue;
  if (!encode_2d(&pp.tm_s, a.scales, 2, (uint64_t)a.N, (uint64_t)G, pf::BN, 1, 0))
    return cudaErrorInvalidValue;
  if (a.zeros &&
      !encode_2d(&pp.tm_z, a.zeros, 4, (uint64_t)a.N, (uint64_t)((G + 7) / 8), pf::BN, 1, 0))
    return cudaErrorInvalidValue;
  pp.packed = static_cast<const uint8_t *>(a.packed);
  pp.out = a.out;
  pp.out_type = a.out_type;
  pp.err = a.err;
  pp.M = a.M;
  pp.N = a.N;
  pp.K = a.K;
  pp.gs = a.group_size;
  pp.nt_total = a.N / 16;
  dim3 grid((a.M + bm - 1) / bm, (a.N + pf::BN - 1) / pf::BN);
  const bool z = a.zeros != nullptr;
  return ms == 1 ? launch_ms<1>(pp, grid, a.x_bf16, z, s) : launch_ms<2>(pp, grid, a.x_bf16, z, s);
}

}  // namespace wq
