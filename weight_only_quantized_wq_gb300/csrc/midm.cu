// midm.cu -- weight-only quantized matmul for a moderate number of tokens
// (int4 codes), on the 5th-generation tensor cores, with exact weights.
//
// Swap-AB: the dequantized weights are the A operand (128 output channels =
// UMMA M) and a tile of NT tokens of x the B operand (UMMA N = NT, 16..128),
// so D[channel, token] accumulates in TMEM however few tokens there are.
// Per stage (64 values of K, one packed chunk row):
//   warp 0      producers: lane 0 streams a ring of weight slots (1-D bulk
//               copy of the packed weights of the CTA's 128 channels, TMA
//               copies of the stage's scale row and packed zero-word row),
//               lane 1 a ring of x tiles (NT x 64, 128-byte swizzle, rows
//               past M zero-filled);
//   warp 1      TMEM allocation and the single thread issuing tcgen05.mma;
//   warps 2..9  dequantize q - zero (a small integer, exact in fp16 / bf16)
//               into the 128-byte-swizzled A buffer, and fold finished groups.
// Exactness: the MMA sums x (q - zero) over one group into one of two TMEM
// accumulators (double-buffered by group); when a group is complete the
// dequant warps load it (tcgen05.ld: one channel per thread, half of the
// tokens per warp) and add scale * sum to fp32 registers, while the tensor
// core already fills the other accumulator with the next group.  No weight is
// ever rounded; the scale is applied in fp32 (BitDistiller
// quant_matmul_kernel semantics, w = (q - zero) * scale).
// Split-K: the K splits of a channel block form one thread-block cluster and
// their partial tiles are summed in split order through distributed shared
// memory (no workspace), as in the few-token kernel.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <tuple>

#include "dev.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace wq {

namespace mm {

constexpr int CH = 128;        // output channels per CTA (UMMA M)
constexpr int BK = 64;         // K per stage: one int4 chunk row, one swizzle atom of 16-bit values
constexpr int PB = 4;          // group accumulators in TMEM
constexpr int LAG = 2;         // a group is folded when the group LAG later starts
constexpr int DQ_WARPS = 8;
constexpr int THREADS = (2 + DQ_WARPS) * 32;
constexpr int A_BYTES = CH * BK * 2;  // one dequantized A buffer (16 KB)
constexpr int W_BYTES = CH * BK / 2;  // packed int4 of one stage (4 KB)
constexpr int S_BYTES = CH * 2;       // one scale row
constexpr int Z_BYTES = CH * 4;       // one zero-word row
constexpr int W_SLOT = W_BYTES + S_BYTES + Z_BYTES;  // one weight-ring slot (multiple of 128)
constexpr int HEADER = 1024;          // mbarriers, TMEM address, abort flag

// Shared memory of one CTA: header | x ring (XS tiles of NT tokens x 64 K,
// 128-byte swizzle) | ABUF dequantized A buffers | weight ring (WS slots of
// packed weights, scale row, zero-word row).  The weight ring is released by
// the dequant warps as soon as they have read a slot, the x ring by the MMA,
// so the weight stream keeps WS slots in flight whatever the MMA does.
template <int NT>
struct Cfg {
  static constexpr int XS = NT <= 16 ? 8 : NT <= 32 ? 6 : NT <= 64 ? 8 : 5;
  static constexpr int ABUF = NT == 64 ? 4 : 3;
  static constexpr int WS = NT <= 32 ? 8 : 16;
  static constexpr int X_BYTES = NT * 128;  // NT tokens x 64 values of K, 16-bit
  static constexpr int X_OFF = HEADER;
  static constexpr int A_OFF = X_OFF + XS * X_BYTES;
  static constexpr int W_OFF = A_OFF + ABUF * A_BYTES;
  static constexpr int SMEM = W_OFF + WS * W_SLOT;
  static constexpr int TMEM_COLS = PB * NT < 32 ? 32 : PB * NT;  // PB group accumulators
  static constexpr int RP = CH + 4;                            // staging row pitch (floats)
  static_assert(NT * RP * 4 <= W_OFF - X_OFF, "the partial tile must fit the x ring and A buffers");
  static_assert(SMEM + 1024 <= 227 * 1024, "shared memory");
};

struct Params {
  CUtensorMap tm_x;  // x (M, K) 16-bit, box (64, NT), 128-byte swizzle
  CUtensorMap tm_s;  // scales (G, N) 16-bit, box (128, 1)
  CUtensorMap tm_z;  // zero words (ceil(G/8), N) 32-bit, box (128, 1)
  const uint8_t *packed;
  void *out;
  int out_type;  // OutType
  uint32_t *err;
  int M, N, K, gs, nt_total, kch, cps, splits;
  bool s_bf16;
  bool cluster;
};

// Resident CTAs per SM the register budget is sized for (shared memory
// allows two up to 32 tokens, one beyond).
__host__ __device__ constexpr int midm_min_blocks(int nt) { return nt <= 32 ? 2 : 1; }

template <bool BF16, bool ZERO, int NT>
__global__ void __launch_bounds__(THREADS, midm_min_blocks(NT)) midm_kernel(const __grid_constant__ Params p) {
  using C = Cfg<NT>;
  constexpr int XS = C::XS, ABUF = C::ABUF, WS = C::WS;
  constexpr int HALF = NT / 2;  // token columns per dequant warp
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t *xfull = reinterpret_cast<uint64_t *>(smem);  // an x tile landed
  uint64_t *xempty = xfull + XS;                         // MMA done with an x tile
  uint64_t *wfull = xempty + XS;                         // a weight slot landed
  uint64_t *wempty = wfull + WS;                         // dequant done with a weight slot
  uint64_t *afull = wempty + WS;                         // an A buffer is written
  uint64_t *aempty = afull + ABUF;                       // MMA done with an A buffer
  uint64_t *pfull = aempty + ABUF;                       // a group accumulator is complete
  uint64_t *pempty = pfull + PB;                         // a group accumulator was read
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(pempty + PB);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  static_assert((2 * (XS + WS + ABUF + PB)) * 8 + 8 <= HEADER, "barriers do not fit the header");
  uint8_t *xring = smem + C::X_OFF;
  uint8_t *abuf = smem + C::A_OFF;
  uint8_t *wring = smem + C::W_OFF;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = blockIdx.x, split = blockIdx.y, mtile = blockIdx.z;
  const int n0 = nb * CH, nt0 = n0 / 16;
  const int ntiles = min(CH / 16, p.nt_total - nt0);
  const int m0 = mtile * NT;
  const int c0 = split * p.cps;
  const int nk = min(p.kch, c0 + p.cps) - c0;  // stages of this CTA
  const int kbeg = c0 * BK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < XS; ++i) {
      mbar_init(smem_addr(&xfull[i]), 1);
      mbar_init(smem_addr(&xempty[i]), 1);
    }
    for (int i = 0; i < WS; ++i) {
      mbar_init(smem_addr(&wfull[i]), 1);
      mbar_init(smem_addr(&wempty[i]), DQ_WARPS);
    }
    for (int i = 0; i < ABUF; ++i) {
      mbar_init(smem_addr(&afull[i]), DQ_WARPS);
      mbar_init(smem_addr(&aempty[i]), 1);
    }
    for (int i = 0; i < PB; ++i) {
      mbar_init(smem_addr(&pfull[i]), 1);
      mbar_init(smem_addr(&pempty[i]), DQ_WARPS);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tc::alloc(smem_addr(tmem_slot), C::TMEM_COLS);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;

  // Groups are whole stages (gs % 64 == 0): sg stages per group.  Each role
  // walks the groups with counters (no division per stage): group g of the
  // current stage and its position pos inside the group.
  const int sg = p.gs / BK;
  const int gi0 = c0 / sg, pos0 = c0 % sg;

  if (warp == 0) {
    // ------------------------------------------------------------ producers
    // Lane 0 streams the weight ring, lane 1 the x ring: neither waits for
    // the other's slots, so WS weight slots stay in flight while the MMA
    // lags behind the dequant.
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const uint32_t wbytes = (uint32_t)ntiles * 512u;
      int issued = 0, g = gi0, pos = pos0;
      for (int i = 0; i < nk; ++i) {
        const int ws = i % WS;
        if (i >= WS && !mbar_wait(smem_addr(&wempty[ws]), ((i / WS) - 1) & 1, p.err, abort_flag)) break;
        const uint32_t wb = smem_addr(&wfull[ws]);
        const uint32_t wdst = smem_addr(wring + ws * W_SLOT);
        mbar_arrive_expect_tx(wb, wbytes + S_BYTES + (ZERO ? Z_BYTES : 0));
        bulk_g2s(wdst, p.packed + ((size_t)(c0 + i) * p.nt_total + nt0) * 512, wbytes, wb, pol);
        tma_load_2d(wdst + W_BYTES, &p.tm_s, n0, g, wb);
        if (ZERO) tma_load_2d(wdst + W_BYTES + S_BYTES, &p.tm_z, n0, g / 8, wb);
        issued = i + 1;
        if (++pos == sg) {
          pos = 0;
          ++g;
        }
      }
      // No copy may still be writing this CTA's shared memory when it moves on.
      for (int i = max(0, issued - WS); i < issued; ++i)
        mbar_wait(smem_addr(&wfull[i % WS]), (i / WS) & 1, p.err, nullptr);
    } else if (lane == 1) {
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int xs = i % XS;
        if (i >= XS && !mbar_wait(smem_addr(&xempty[xs]), ((i / XS) - 1) & 1, p.err, abort_flag)) break;
        const uint32_t xb = smem_addr(&xfull[xs]);
        mbar_arrive_expect_tx(xb, C::X_BYTES);
        tma_load_2d(smem_addr(xring + xs * C::X_BYTES), &p.tm_x, kbeg + i * BK, m0, xb);
        issued = i + 1;
      }
      for (int i = max(0, issued - XS); i < issued; ++i)
        mbar_wait(smem_addr(&xfull[i % XS]), (i / XS) & 1, p.err, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id = tc::idesc<BF16>(CH, NT);
      int gl = -1, pos = pos0;
      for (int i = 0; i < nk; ++i) {
        const int xs = i % XS, ab = i % ABUF;
        if (!mbar_wait(smem_addr(&xfull[xs]), (i / XS) & 1, p.err, abort_flag)) break;
        if (!mbar_wait(smem_addr(&afull[ab]), (i / ABUF) & 1, p.err, abort_flag)) break;
        const bool first = i == 0 || pos == 0;
        const bool last = i == nk - 1 || pos == sg - 1;
        if (++pos == sg) pos = 0;
        if (first) {
          ++gl;
          if (gl >= PB && !mbar_wait(smem_addr(&pempty[gl % PB]), ((gl / PB) - 1) & 1, p.err, abort_flag)) break;
        }
        tc::fence_after();
        const uint32_t a0 = smem_addr(abuf + ab * A_BYTES);
        const uint32_t b0 = smem_addr(xring + xs * C::X_BYTES);
        const uint32_t d = tmem + (uint32_t)((gl % PB) * NT);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc::mma(d, tc::sw128_desc(a0 + kk * 32), tc::sw128_desc(b0 + kk * 32), id, (first && kk == 0) ? 0u : 1u);
        tc::commit(smem_addr(&xempty[xs]));
        tc::commit(smem_addr(&aempty[ab]));
        if (last) tc::commit(smem_addr(&pfull[gl % PB]));
      }
    }
  } else {
    // ------------------------------------------------------------ dequant + group fold (warps 2..9)
    const int wi = warp - 2;
    const int q = (wi + 2) & 3;  // TMEM lane quarter this warp may read (warp index mod 4)
    const int hf = wi >> 2;      // which half of the token columns it folds
    const int tile = wi;         // 16-channel tile it dequantizes
    const int slot = tc::dq_slot(lane);  // this lane's 16-byte slot of a tile chunk
    const int gq = slot >> 2, tq = slot & 3;
    constexpr uint32_t MAGIC_LO = Magic<BF16>::kPair & 0xFFFFu;
    float acc[HALF];
#pragma unroll
    for (int j = 0; j < HALF; ++j) acc[j] = 0.f;
    // scale of this thread's fold channel for the groups in flight, by group % PB
    static_assert(PB == 4, "one register per group accumulator");
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    auto scale_of = [&](int G) {
      const int j = G % PB;
      return j == 0 ? s0 : j == 1 ? s1 : j == 2 ? s2 : s3;
    };

    // acc += scale * (complete group accumulator G); frees the accumulator.
    auto fold = [&](int G) -> bool {
      if (!mbar_wait(smem_addr(&pfull[G % PB]), (G / PB) & 1, p.err, abort_flag)) return false;
      tc::fence_after();
      const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)((G % PB) * NT + hf * HALF);
      const float s = scale_of(G);
      if constexpr (HALF >= 32) {
#pragma unroll
        for (int c = 0; c < HALF; c += 32) {
          uint32_t r[32];
          tc::ld32(ta + c, r);
          tc::wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) acc[c + j] = fmaf(s, __uint_as_float(r[j]), acc[c + j]);
        }
      } else if constexpr (HALF == 16) {
        uint32_t r[16];
        tc::ld16(ta, r);
        tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[j] = fmaf(s, __uint_as_float(r[j]), acc[j]);
      } else {
        uint32_t r[8];
        tc::ld8(ta, r);
        tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = fmaf(s, __uint_as_float(r[j]), acc[j]);
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&pempty[G % PB]));
      return true;
    };

    // shared-memory offsets of this thread's eight 4-value runs of A
    uint32_t aoff[2][2][2];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int j = 0; j < 2; ++j) aoff[r][u][j] = tc::sw128_off(tile * 16 + gq + 8 * r, 32 * u + 16 * j + 4 * tq);
    uint32_t zz[2] = {(MAGIC_LO + 8u) * 0x00010001u, (MAGIC_LO + 8u) * 0x00010001u};  // (MAGIC + zero) pairs

    int gl = -1, folded = 0;  // groups started, groups folded
    int g = gi0, pos = pos0;
    bool ok = true;
    for (int i = 0; i < nk && ok; ++i) {
      const int ws = i % WS, ab = i % ABUF;
      if (!mbar_wait(smem_addr(&wfull[ws]), (i / WS) & 1, p.err, abort_flag)) break;
      if (i >= ABUF && !mbar_wait(smem_addr(&aempty[ab]), ((i / ABUF) - 1) & 1, p.err, abort_flag)) break;
      const uint32_t base = smem_addr(wring + ws * W_SLOT);
      const bool first = i == 0 || pos == 0;
      if (first) {
        ++gl;
        if (ZERO) {
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const uint32_t z = (lds32(base + W_BYTES + S_BYTES + (tile * 16 + gq + 8 * r) * 4) >> ((g % 8) * 4)) & 15u;
            zz[r] = (MAGIC_LO + z) * 0x00010001u;
          }
        }
        const float sv = half_bits_to_float(lds16(base + W_BYTES + (q * 32 + lane) * 2), p.s_bf16);
        switch (gl % PB) {
          case 0: s0 = sv; break;
          case 1: s1 = sv; break;
          case 2: s2 = sv; break;
          default: s3 = sv; break;
        }
      }
      if (++pos == sg) {
        pos = 0;
        ++g;
      }
      uint4 wv = make_uint4(0u, 0u, 0u, 0u);
      if (tile < ntiles) wv = lds128(base + tile * 512 + slot * 16);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&wempty[ws]));  // the weight slot may be refilled
      if (tile < ntiles) {
        const uint32_t adst = smem_addr(abuf + ab * A_BYTES);
        const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const uint32_t w = w4[2 * u + r];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const uint32_t lo = sub_pair<BF16>(code_pair<4, BF16>(w, 2 * j), zz[r]);
              const uint32_t hi = sub_pair<BF16>(code_pair<4, BF16>(w, 2 * j + 1), zz[r]);
              sts64(adst + aoff[r][u][j], lo, hi);
            }
          }
      }
      fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&afull[ab]));
      if (first && gl >= LAG) ok = fold(folded++);
    }
    while (ok && folded <= gl) ok = fold(folded++);

    // Partial tile -> shared memory as [token][channel], over the x ring and
    // the A buffers: the last group's commit followed every MMA, and every
    // dequant warp wrote its last A tile before that MMA could start.
    float *red = reinterpret_cast<float *>(xring);
#pragma unroll
    for (int j = 0; j < HALF; ++j) red[(hf * HALF + j) * C::RP + q * 32 + lane] = acc[j];
  }

  tc::fence_before();
  __syncthreads();
  // ------------------------------------------------------------ reduction over the K splits, store
  const int rows = min(NT, p.M - m0);
  const int qpr = ntiles * 4;  // float4 quads per token row
  const uint32_t red = smem_addr(xring);
  if (p.cluster) {
    cluster_sync();
    const uint32_t rank = cluster_ctarank();
    for (int qd = threadIdx.x * p.splits + (int)rank; qd < rows * qpr; qd += THREADS * p.splits) {
      const int m = qd / qpr, c4 = (qd % qpr) * 4;
      const uint32_t la = red + (uint32_t)(m * C::RP + c4) * 4u;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int r0 = 0; r0 < p.splits; r0 += 8) {
        float4 u[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (r0 + j < p.splits) u[j] = ld_dsmem_f4(dsmem_addr(la, (uint32_t)(r0 + j)));
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (r0 + j < p.splits) {
            v.x += u[j].x;
            v.y += u[j].y;
            v.z += u[j].z;
            v.w += u[j].w;
          }
      }
      store_out4(p.out, (size_t)(m0 + m) * p.N + n0 + c4, v, p.out_type);
    }
    __syncwarp();
    cluster_sync_relaxed();  // no CTA leaves while another still reads its shared memory
  } else {
    const float *redp = reinterpret_cast<const float *>(xring);
    for (int qd = threadIdx.x; qd < rows * qpr; qd += THREADS) {
      const int m = qd / qpr, c4 = (qd % qpr) * 4;
      store_out4(p.out, (size_t)(m0 + m) * p.N + n0 + c4, *reinterpret_cast<const float4 *>(redp + m * C::RP + c4),
                 p.out_type);
    }
  }
  if (warp == 1) {
    tc::fence_after();
    tc::dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace mm

// ------------------------------------------------------------------ host side
bool midm_supported(const MatmulArgs &a) {
  return a.w_bit == 4 && a.group_size % mm::BK == 0 && a.K % mm::BK == 0;
}

static int midm_nt(int M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128; }

template <bool BF16, bool ZERO, int NT>
static cudaError_t midm_prepare_t(bool big_cluster) {
  auto kern = mm::midm_kernel<BF16, ZERO, NT>;
  static int attr_set[64] = {0};
  static int nonportable[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, mm::Cfg<NT>::SMEM + 1024);
    if (e != cudaSuccess) return e;
    attr_set[dev] = 1;
  }
  if (big_cluster && !nonportable[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    nonportable[dev] = 1;
  }
  return cudaSuccess;
}

static void cluster_cfg(cudaLaunchConfig_t &cfg, cudaLaunchAttribute *attr, int splits) {
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = splits;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
}

// CTAs of one launch shape that can be resident at once (runtime occupancy
// calculator; for clusters also the clusters the GPCs hold).  -1 on error.
template <bool BF16, bool ZERO, int NT>
static long midm_capacity_t(int splits, int sms) {
  auto kern = mm::midm_kernel<BF16, ZERO, NT>;
  if (midm_prepare_t<BF16, ZERO, NT>(splits > 8) != cudaSuccess) return -1;
  const int smem = mm::Cfg<NT>::SMEM + 1024;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, mm::THREADS, smem) != cudaSuccess) return -1;
  // TMEM: every resident CTA holds TMEM_COLS of the SM's 512 columns.
  const int by_tmem = 512 / mm::Cfg<NT>::TMEM_COLS;
  if (per_sm > by_tmem) per_sm = by_tmem;
  long cap = (long)per_sm * sms;
  if (splits > 1) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(1, splits, 1);
    cfg.blockDim = dim3(mm::THREADS);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    cluster_cfg(cfg, attr, splits);
    int nc = 0;
    if (cudaOccupancyMaxActiveClusters(&nc, kern, &cfg) != cudaSuccess) return -1;
    cap = cap < (long)nc * splits ? cap : (long)nc * splits;
  }
  return cap;
}

template <bool BF16, bool ZERO, int NT>
static cudaError_t midm_launch_t(const mm::Params &pp, dim3 grid, cudaStream_t s) {
  auto kern = mm::midm_kernel<BF16, ZERO, NT>;
  cudaError_t e = midm_prepare_t<BF16, ZERO, NT>(pp.splits > 8);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(mm::THREADS);
  cfg.dynamicSmemBytes = mm::Cfg<NT>::SMEM + 1024;  // + slack for the 1024-byte alignment
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (pp.cluster) cluster_cfg(cfg, attr, pp.splits);
  e = cudaLaunchKernelEx(&cfg, kern, pp);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// The capacity of the bf16, asymmetric instantiation stands for all four
// (same shared memory and TMEM; registers do not limit these launches).
static long midm_capacity(int nt, int splits, int sms) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  using Key = std::tuple<int, int, int, int>;
  static std::map<Key, long> cache;
  static std::mutex mu;
  const Key key{dev, nt, splits, sms};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  long c = -1;
  switch (nt) {
    case 16: c = midm_capacity_t<true, true, 16>(splits, sms); break;
    case 32: c = midm_capacity_t<true, true, 32>(splits, sms); break;
    case 64: c = midm_capacity_t<true, true, 64>(splits, sms); break;
    case 128: c = midm_capacity_t<true, true, 128>(splits, sms); break;
  }
  cudaGetLastError();
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = c;
  return c;
}

MidmPlan plan_midm(int M, int N, int K, int sms) {
  MidmPlan best{};
  const int nt = midm_nt(M);
  const int mtiles = (M + nt - 1) / nt;
  const int nblocks = (N + mm::CH - 1) / mm::CH;
  const int kch = K / mm::BK;
  double best_cost = 1e300;
  for (int s = 1; s <= kMaxClusterSplits && s <= kch; ++s) {
    const int cps = (kch + s - 1) / s;
    if ((kch + cps - 1) / cps != s) continue;
    long cap = midm_capacity(nt, s, sms);
    if (cap < 1) cap = sms;  // no answer from the runtime: one CTA per SM
    // Busiest SM's stages, at a rate that grows with the CTAs it runs at
    // once (r / (r + 1)), plus the cluster reduction per wave.
    const long units = (long)nblocks * mtiles * s;
    const long waves = (units + cap - 1) / cap;
    const long per_sm_max = (cap + sms - 1) / sms;
    const long per_sm = units <= cap ? (units + sms - 1) / sms : waves * per_sm_max;
    const double r = (double)(per_sm < per_sm_max ? per_sm : per_sm_max);
    double cost = (double)per_sm * cps / (r / (r + 1.0));
    if (s > 1) cost += (2.0 + 0.5 * s) * waves;
    if (cost < best_cost * 0.999) {
      best_cost = cost;
      best.nt = nt;
      best.splits = s;
      best.cps = cps;
      best.nblocks = nblocks;
      best.mtiles = mtiles;
    }
  }
  return best;
}

template <int NT>
static cudaError_t midm_dispatch(const mm::Params &pp, dim3 grid, bool bf16, bool z, cudaStream_t s) {
  if (bf16) return z ? midm_launch_t<true, true, NT>(pp, grid, s) : midm_launch_t<true, false, NT>(pp, grid, s);
  return z ? midm_launch_t<false, true, NT>(pp, grid, s) : midm_launch_t<false, false, NT>(pp, grid, s);
}

cudaError_t launch_midm(const MatmulArgs &a, const MidmPlan &pl, cudaStream_t s) {
  mm::Params pp{};
  const int G = a.K / a.group_size;
  if (!encode_2d(&pp.tm_x, a.x, 2, (uint64_t)a.K, (uint64_t)a.M, mm::BK, (uint32_t)pl.nt, 128))
    return cudaErrorInvalidValue;
  if (!encode_2d(&pp.tm_s, a.scales, 2, (uint64_t)a.N, (uint64_t)G, mm::CH, 1, 0)) return cudaErrorInvalidValue;
  if (a.zeros && !encode_2d(&pp.tm_z, a.zeros, 4, (uint64_t)a.N, (uint64_t)((G + 7) / 8), mm::CH, 1, 0))
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
  pp.kch = a.K / mm::BK;
  pp.cps = pl.cps;
  pp.splits = pl.splits;
  pp.s_bf16 = a.s_bf16;
  pp.cluster = pl.splits > 1;
  const dim3 grid(pl.nblocks, pl.splits, pl.mtiles);
  const bool z = a.zeros != nullptr;
  switch (pl.nt) {
    case 16: return midm_dispatch<16>(pp, grid, a.x_bf16, z, s);
    case 32: return midm_dispatch<32>(pp, grid, a.x_bf16, z, s);
    case 64: return midm_dispatch<64>(pp, grid, a.x_bf16, z, s);
    case 128: return midm_dispatch<128>(pp, grid, a.x_bf16, z, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace wq
