// prefill.cu -- weight-only quantized matmul for many tokens (tensor cores, tcgen05).
//
// At large M the step is bound by the multiply-adds, so the weights are
// dequantized once per 256-token tile into shared memory in the operand
// layout of the 5th-generation tensor cores, and tcgen05.mma accumulates
// D[m, n] (TMEM, fp32) += x[m, k] * w[k, n] over 64-wide K stages.
//
// Tile: 256 tokens x 256 output channels; two 128 x 256 accumulators (the
// whole 512-column TMEM) share each dequantized weight tile, so every weight
// is dequantized once per 256 tokens.
//
// Scheduling.  Problems with more tiles than a quarter of the SMs run one tile
// per CTA (prefill_kernel: warps 4..7 read the accumulator out after their
// share of the dequant; token tiles vary fastest over the grid, so the CTAs
// that read the same 256-channel weight block run together and share it in
// L2).  Smaller ones (few channel blocks and tokens: most SMs would sit idle)
// run persistent with stream-K shares (prefill_sk_kernel), two CTAs per tile:
// the work is the list of (tile, K stage) units, tile by tile; each CTA takes
// one contiguous share of it, so every SM gets the same number of stages
// whatever the tile count, and a share may start or end inside a tile.  A
// tile cut between CTAs is finished by the CTA holding its first stages (it
// reaches that part last, at the end of its share): every other CTA writes
// its fp32 partial tile to the workspace and raises a flag; the finishing CTA
// waits for those flags (bounded), adds the partials in stage order (a fixed
// order: the result does not depend on timing) and stores the tile.  This is
// Marlin's striped partition of the K loop over the SMs (aphrodite-engine
// marlin_cuda_kernel.cu) with its serial global-lock reduction replaced by
// one fix-up per cut tile.  The launch is cooperative (all CTAs resident),
// so the waits cannot deadlock.  Without a workspace that holds the partial
// tiles, one tile per CTA runs.
// Roles of the persistent kernel (14 warps):
//   warp 0       producer: per stage one TMA copy of the x tile (256 x 64,
//                128-byte swizzle), one 1-D bulk copy of the packed weights
//                (256 channels x 64 k), TMA copies of the scale and zero rows
//                of the stage's group;
//   warp 1       TMEM allocation and the single thread that issues tcgen05.mma;
//   warps 2..9   dequant: w = (q - zero) * scale rounded once to the x dtype,
//                written K-major with the 128-byte swizzle the MMA reads;
//   warps 10..13 epilogue: tcgen05.ld of the fp32 accumulator (one token row
//                per thread), then partial, fix-up or store; the next run of
//                stages starts as soon as the accumulator is read out.
// Roles of the one-tile kernel (11 warps): warp 0 x producer (its own ring
// of x tiles), warp 1 TMEM and the MMA issuer, warp 2 weight producer (a
// short ring of packed weights, scale and zero rows), warps 3..10 dequant,
// of which 4..7 read the accumulator out at the end.
// The scale and zero are applied to the weight (one rounding to bf16/fp16),
// since a per-group rescale of a 128 x 256 TMEM accumulator would cost more
// than the tensor cores gain.  Calls where that rounding could exceed the
// accepted error run the one-tile kernel with two-term weights (the rounded
// weight and its rounded residue, 128 channels per tile) when they have
// enough tiles, else the exact tensor-core kernel.
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
constexpr int BN = 256;   // output channels per tile (UMMA N)
constexpr int BK = 64;    // K per stage: one 128-byte swizzle atom of bf16
constexpr int STAGES = 3;
constexpr int BSTAGES = 2;            // dequantized B buffers
constexpr int DQ_WARPS = 8;
constexpr int EPI_WARPS = 4;
constexpr int THREADS = (3 + DQ_WARPS) * 32;                 // one tile per CTA
constexpr int SK_THREADS = (2 + DQ_WARPS + EPI_WARPS) * 32;  // persistent, stream-K
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr int W_BYTES = BN * BK / 2;  // 8 KB of packed int4
constexpr int S_BYTES = BN * 2;       // one scale row
constexpr int Z_BYTES = BN * 4;       // one zero-word row
constexpr int HEADER = 1024;          // mbarriers + TMEM address
constexpr int kFlagBytes = 16384;     // stream-K flags at the front of the workspace (one int per CTA)

// Geometry for MS accumulators of 128 tokens each (token tile BM = 128 MS).
template <int MS>
struct Cfg {
  static constexpr int MSUB = MS;
  static constexpr int BM = UM * MS;                  // tokens per tile
  static constexpr int A_BYTES = BM * BK * 2;         // x tile: 16 or 32 KB
  // stage = A | W | S | Z, 1024-byte aligned (the swizzle atom of A)
  static constexpr int ST_A = 0, ST_W = A_BYTES, ST_S = ST_W + W_BYTES, ST_Z = ST_S + S_BYTES;
  static constexpr int STAGE_BYTES = (ST_Z + Z_BYTES + 1023) / 1024 * 1024;
  static constexpr int SMEM = HEADER + STAGES * STAGE_BYTES + BSTAGES * B_BYTES;
  static constexpr int TMEM_COLS = BN * MS;           // 256 or 512
};

// Geometry of the one-tile kernel, whose x tiles and weight rows travel in
// separate rings.  An x tile must stay until the MMAs of its stage have read
// it; a weight slot only until the dequant warps hold its words in
// registers.  So the weights run ahead on a short ring of their own and the
// x ring's depth is spent on the x tiles' own latency alone (in one shared
// ring every slot was held for that latency plus the dequant plus the MMAs).
template <int MS>
struct DCfg {
  static constexpr int MSUB = MS;
  static constexpr int BM = UM * MS;                           // tokens per tile
  static constexpr int A_BYTES = BM * BK * 2;                  // x tile: 16 or 32 KB
  static constexpr int XS = MS == 2 ? 4 : 7;                   // x tiles in the ring
  static constexpr int WS = 3;                                 // weight slots
  static constexpr int W_SLOT = W_BYTES + S_BYTES + Z_BYTES;   // packed weights | scale row | zero row
  static constexpr int OFF_X = HEADER;                         // 1024-byte aligned (swizzle atoms)
  static constexpr int OFF_B = OFF_X + XS * A_BYTES;
  static constexpr int OFF_W = OFF_B + BSTAGES * B_BYTES;
  static constexpr int SMEM = OFF_W + WS * W_SLOT;
  static constexpr int TMEM_COLS = BN * MS;                    // 256 or 512
  static_assert(W_SLOT % 128 == 0, "weight slots keep 128-byte alignment");
  static_assert((2 * (XS + WS + BSTAGES) + 1) * 8 + 8 <= HEADER, "barriers do not fit the header");
};

struct Params {
  CUtensorMap tm_x;  // x (M, K) 16-bit, box (64, BM), 128-byte swizzle
  CUtensorMap tm_s;  // scales (G, N) 16-bit, box (256, 1)
  CUtensorMap tm_z;  // zeros (ceil(G/8), N) 32-bit, box (256, 1)
  const uint8_t *packed;
  void *out;
  int out_type;  // OutType
  uint32_t *err;
  int M, N, K, gs, nt_total;
  int tiles_m;       // token tiles
  int nk;            // K stages per tile
  long long units;   // tiles * nk
  int *flags;        // stream-K: one flag per CTA (zero between calls); nullptr: one tile per CTA
  float *partial;    // stream-K: one BM x BN fp32 partial tile per CTA
};

// Stage range [u0, u1) of the unit list that CTA c of `ctas` takes.
__device__ __forceinline__ void share_of(const Params &p, int c, int ctas, long long &u0, long long &u1) {
  u0 = p.units * c / ctas;
  u1 = p.units * (c + 1) / ctas;
}

// One contiguous run of a CTA's share inside one tile.
struct Seg {
  int t, s0, s1;
};
__device__ __forceinline__ Seg seg_at(const Params &p, long long u, long long u1) {
  Seg g;
  g.t = (int)(u / p.nk);
  g.s0 = (int)(u - (long long)g.t * p.nk);
  const long long left = u1 - u;
  g.s1 = (int)(left < (long long)(p.nk - g.s0) ? g.s0 + left : p.nk);
  return g;
}

template <bool BF16>
__device__ __forceinline__ uint32_t mul2(uint32_t a, uint32_t b) {
  uint32_t d;
  if constexpr (BF16)
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

template <bool BF16>
__device__ __forceinline__ uint32_t fma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  if constexpr (BF16)
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  else
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
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

// Bounded wait until the flag at f is non-zero (acquire, device scope).
__device__ __forceinline__ bool wait_flag(const int *f, uint32_t *err, volatile int *abort) {
  const long long t0 = clock64();
  for (uint32_t it = 0;; ++it) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    if (v != 0) return true;
    if ((it & 63u) == 63u) {
      if (*abort) return false;
      if (clock64() - t0 > kWaitLimitCycles) {
        atomicOr(err, kDevErrTimeout);
        *abort = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ void epilogue_sync() {
  asm volatile("bar.sync 2, %0;" ::"n"(EPI_WARPS * 32) : "memory");
}

template <bool BF16, bool ZERO, int MS>
__global__ void __launch_bounds__(SK_THREADS, 1) prefill_sk_kernel(const __grid_constant__ Params p) {
  using C = Cfg<MS>;
  constexpr int MSUB = C::MSUB, BM = C::BM, A_BYTES = C::A_BYTES, STAGE_BYTES = C::STAGE_BYTES;
  constexpr int ST_A = C::ST_A, ST_W = C::ST_W, ST_S = C::ST_S, ST_Z = C::ST_Z, TMEM_COLS = C::TMEM_COLS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment (of the shared-window address) for the swizzled tiles
  uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);  // TMA data of a stage landed
  uint64_t *empty = full + STAGES;                      // MMA done with a stage
  uint64_t *bfull = empty + STAGES;                     // dequantized B written
  uint64_t *bempty = bfull + BSTAGES;                   // MMA done with a B buffer
  uint64_t *accfull = bempty + BSTAGES;                 // the accumulator of a run is complete
  uint64_t *accempty = accfull + 1;                     // the epilogue has read the accumulator out
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accempty + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  uint8_t *ring = smem + HEADER;
  uint8_t *bbuf = ring + STAGES * STAGE_BYTES;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x, ctas = gridDim.x;
  long long u0, u1;
  share_of(p, cta, ctas, u0, u1);
  auto tile_n0 = [&](int t) { return (t / p.tiles_m) * BN; };
  auto tile_m0 = [&](int t) { return (t % p.tiles_m) * BM; };

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
    mbar_init(smem_addr(accempty), EPI_WARPS);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tc::alloc(smem_addr(tmem_slot), TMEM_COLS);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int i = 0, issued = 0;
      bool ok = true;
      for (long long u = u0; u < u1 && ok;) {
        const Seg g = seg_at(p, u, u1);
        u += g.s1 - g.s0;
        const int n0 = tile_n0(g.t), m0 = tile_m0(g.t), nt0 = n0 / 16;
        const int ntiles = min(BN / 16, p.nt_total - nt0);
        for (int s = g.s0; s < g.s1; ++s, ++i) {
          const int st = i % STAGES;
          if (i >= STAGES && !mbar_wait(smem_addr(&empty[st]), ((i / STAGES) - 1) & 1, p.err, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_addr(&full[st]);
          const uint32_t base = smem_addr(ring + st * STAGE_BYTES);
          const int gi = s * BK / p.gs;
          mbar_arrive_expect_tx(fb, A_BYTES + ntiles * 512 + S_BYTES + (ZERO ? Z_BYTES : 0));
          tma_load_2d(base + ST_A, &p.tm_x, s * BK, m0, fb);
          bulk_g2s(base + ST_W, p.packed + ((size_t)s * p.nt_total + nt0) * 512, ntiles * 512, fb, pol);
          tma_load_2d(base + ST_S, &p.tm_s, n0, gi, fb);
          if (ZERO) tma_load_2d(base + ST_Z, &p.tm_z, n0, gi / 8, fb);
          issued = i + 1;
        }
      }
      for (int i2 = max(0, issued - STAGES); i2 < issued; ++i2)
        mbar_wait(smem_addr(&full[i2 % STAGES]), (i2 / STAGES) & 1, p.err, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id = tc::idesc<BF16>(UM, BN);
      int i = 0, j = 0;
      bool ok = true;
      for (long long u = u0; u < u1 && ok; ++j) {
        const Seg g = seg_at(p, u, u1);
        u += g.s1 - g.s0;
        // the epilogue must have read the previous run's accumulator out
        if (j >= 1 && !mbar_wait(smem_addr(accempty), (j - 1) & 1, p.err, abort_flag)) break;
        for (int s = g.s0; s < g.s1; ++s, ++i) {
          const int st = i % STAGES, sb = i % BSTAGES;
          if (!mbar_wait(smem_addr(&full[st]), (i / STAGES) & 1, p.err, abort_flag) ||
              !mbar_wait(smem_addr(&bfull[sb]), (i / BSTAGES) & 1, p.err, abort_flag)) {
            ok = false;
            break;
          }
          tc::fence_after();
          const uint32_t a0 = smem_addr(ring + st * STAGE_BYTES + ST_A);
          const uint32_t b0 = smem_addr(bbuf + sb * B_BYTES);
#pragma unroll
          for (int h = 0; h < MSUB; ++h)
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              tc::mma(tmem + h * BN, tc::sw128_desc(a0 + h * (UM * 128) + kk * 32), tc::sw128_desc(b0 + kk * 32), id,
                      (s != g.s0 || kk != 0) ? 1u : 0u);
          tc::commit(smem_addr(&empty[st]));
          tc::commit(smem_addr(&bempty[sb]));
        }
        if (ok) tc::commit(smem_addr(accfull));  // every MMA of the run has completed when this fires
      }
    }
  } else if (warp < 2 + DQ_WARPS) {
    // ------------------------------------------------------------ dequant (warps 2..9)
    const int dq = threadIdx.x - 64;  // 0 .. 255
    constexpr uint32_t MAGIC = Magic<BF16>::kPair;
    int i = 0;
    bool ok = true;
    for (long long u = u0; u < u1 && ok;) {
      const Seg g = seg_at(p, u, u1);
      u += g.s1 - g.s0;
      const int nt0 = tile_n0(g.t) / 16;
      const int ntiles = min(BN / 16, p.nt_total - nt0);
      for (int s = g.s0; s < g.s1; ++s, ++i) {
        const int st = i % STAGES, sb = i % BSTAGES;
        if (!mbar_wait(smem_addr(&full[st]), (i / STAGES) & 1, p.err, abort_flag) ||
            (i >= BSTAGES && !mbar_wait(smem_addr(&bempty[sb]), ((i / BSTAGES) - 1) & 1, p.err, abort_flag))) {
          ok = false;
          break;
        }
        const uint32_t base = smem_addr(ring + st * STAGE_BYTES);
        const uint32_t bdst = smem_addr(bbuf + sb * B_BYTES);
        const int gi = s * BK / p.gs;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int pr = dq + half * 256;  // (tile, lane) pair 0..511
          const int tile = pr >> 5, ln = tc::dq_slot(pr & 31);
          if (tile < ntiles) {
            const uint4 wv = lds128(base + ST_W + tile * 512 + ln * 16);
            const int gq = ln >> 2, tq = ln & 3;
            const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const int col = tile * 16 + gq + 8 * r;  // row of B (output channel within the tile)
              const uint16_t sbits = lds16(base + ST_S + col * 2);
              uint32_t z = 8;
              if (ZERO) z = (lds32(base + ST_Z + col * 4) >> ((gi % 8) * 4)) & 15u;
              const uint32_t zz = ((MAGIC & 0xFFFFu) + z) * 0x00010001u;  // (MAGIC + z) in both halves
              const uint32_t ss = (uint32_t)sbits * 0x00010001u;
#pragma unroll
              for (int uu = 0; uu < 2; ++uu) {
                const uint32_t w = w4[2 * uu + r];
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                  const uint32_t lo = mul2<BF16>(sub_pair<BF16>(code_pair<4, BF16>(w, 2 * jj), zz), ss);
                  const uint32_t hi = mul2<BF16>(sub_pair<BF16>(code_pair<4, BF16>(w, 2 * jj + 1), zz), ss);
                  const int k = 32 * uu + 16 * jj + 4 * tq;
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
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 10..13)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int j = 0;
    for (long long u = u0; u < u1; ++j) {
      const Seg g = seg_at(p, u, u1);
      u += g.s1 - g.s0;
      const int n0 = tile_n0(g.t), m0 = tile_m0(g.t);
      if (!mbar_wait_idle(smem_addr(accfull), j & 1, p.err, abort_flag)) break;
      tc::fence_after();
      const bool tail = g.s0 > 0;                  // another CTA finishes this tile
      const bool head = g.s0 == 0 && g.s1 < p.nk;  // this CTA finishes it, adding later CTAs' partials
      // The CTAs whose shares start inside this tile after this run: cta + 1 .. last.
      int last = cta;
      if (head) {
        const long long tile_end = (long long)(g.t + 1) * p.nk;
        for (int cc = cta + 1; cc < ctas; ++cc) {
          long long v0, v1;
          share_of(p, cc, ctas, v0, v1);
          if (v0 >= tile_end) break;
          last = cc;
          if (!wait_flag(p.flags + cc, p.err, abort_flag)) break;
        }
      }
      // The first contributor's partial is loaded one 32-column chunk ahead,
      // so its round trips overlap the accumulator reads and the stores.
      float4 nxt[8];
      auto load_first = [&](int h, int c) {
        const float *src = p.partial + ((size_t)(cta + 1) * BM + h * UM + q * 32 + lane) * BN + c;
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) nxt[jj] = __ldcg(reinterpret_cast<const float4 *>(src + 4 * jj));
      };
      if (last > cta) load_first(0, 0);
      for (int h = 0; h < MSUB; ++h) {
        const int row = h * UM + q * 32 + lane;  // token row of the tile
        const int m = m0 + row;
        for (int c = 0; c < BN; c += 32) {
          float v[32];
          tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + h * BN + c, v);
          if (tail) {
            float *dst = p.partial + ((size_t)cta * BM + row) * BN + c;
#pragma unroll
            for (int jj = 0; jj < 32; jj += 4)
              *reinterpret_cast<float4 *>(dst + jj) = make_float4(v[jj], v[jj + 1], v[jj + 2], v[jj + 3]);
            continue;
          }
          if (last > cta) {  // in stage order: the first contributor, then the others
            float4 cur[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) cur[jj] = nxt[jj];
            const int hn = c + 32 < BN ? h : h + 1, cn = c + 32 < BN ? c + 32 : 0;
            if (hn < MSUB) load_first(hn, cn);
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              v[4 * jj] += cur[jj].x;
              v[4 * jj + 1] += cur[jj].y;
              v[4 * jj + 2] += cur[jj].z;
              v[4 * jj + 3] += cur[jj].w;
            }
          }
          for (int cc = cta + 2; cc <= last; ++cc) {
            const float *src = p.partial + ((size_t)cc * BM + row) * BN + c;
            float4 w[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) w[jj] = __ldcg(reinterpret_cast<const float4 *>(src + 4 * jj));
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              v[4 * jj] += w[jj].x;
              v[4 * jj + 1] += w[jj].y;
              v[4 * jj + 2] += w[jj].z;
              v[4 * jj + 3] += w[jj].w;
            }
          }
          if (m < p.M) {
            const size_t o = (size_t)m * p.N + n0 + c;
            if (n0 + c + 32 <= p.N) {
#pragma unroll
              for (int jj = 0; jj < 32; jj += 4)
                store_out4(p.out, o + jj, make_float4(v[jj], v[jj + 1], v[jj + 2], v[jj + 3]), p.out_type);
            } else {
#pragma unroll
              for (int jj = 0; jj < 32; ++jj)
                if (n0 + c + jj < p.N) store_out1(p.out, o + jj, v[jj], p.out_type);
            }
          }
        }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(accempty));  // the MMA may overwrite the accumulator
      if (tail) {
        // publish this CTA's partial: every epilogue thread's stores, then the flag
        __threadfence();
        epilogue_sync();
        if (warp == 2 + DQ_WARPS && lane == 0)
          asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p.flags + cta), "r"(1) : "memory");
      } else if (head) {
        // every thread has read the partials: the flags are zero again for the next call
        epilogue_sync();
        if (warp == 2 + DQ_WARPS && lane == 0)
          for (int cc = cta + 1; cc <= last; ++cc) p.flags[cc] = 0;
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

// One tile per CTA (blockIdx.x: token tile, blockIdx.y: channel block); warps
// 4..7 read the accumulator out after their share of the dequant.
// SPLIT: each weight enters the MMA as two terms, w1 = w rounded to the x
// dtype and w2 = (w - w1) rounded (w2 from one fma: (q - z) s - w1 exactly,
// then one rounding), so w1 + w2 is w within 2^-16 of it instead of 2^-8;
// the tile is then 128 channels, w1 in the B rows 0..127 and w2 in 128..255
// of the same 256-row operand, and the epilogue adds the two halves of the
// accumulator.  Twice the MMA work per weight, for calls where one rounding
// would exceed the accepted error (bf16 below K = 4096).
template <bool BF16, bool ZERO, int MS, bool SPLIT>
__global__ void __launch_bounds__(THREADS, 1) prefill_kernel(const __grid_constant__ Params p) {
  using C = DCfg<MS>;
  constexpr int CB = SPLIT ? BN / 2 : BN;  // output channels per tile
  constexpr int MSUB = C::MSUB, BM = C::BM, A_BYTES = C::A_BYTES, XS = C::XS, WS = C::WS;
  constexpr int W_SLOT = C::W_SLOT, TMEM_COLS = C::TMEM_COLS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment (of the shared-window address) for the swizzled tiles
  uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t *xfull = reinterpret_cast<uint64_t *>(smem);  // x tile of a stage landed
  uint64_t *xempty = xfull + XS;                          // MMAs done with an x tile
  uint64_t *wfull = xempty + XS;                          // weight rows of a stage landed
  uint64_t *wempty = wfull + WS;                          // every dequant warp holds them in registers
  uint64_t *bfull = wempty + WS;                          // dequantized B written
  uint64_t *bempty = bfull + BSTAGES;                     // MMA done with a B buffer
  uint64_t *accfull = bempty + BSTAGES;                   // accumulator complete
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accfull + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  uint8_t *xring = smem + C::OFF_X;
  uint8_t *bbuf = smem + C::OFF_B;
  uint8_t *wring = smem + C::OFF_W;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Token tiles vary fastest across the grid, so the CTAs that read the same
  // 256-channel weight block run at about the same time and share it in L2.
  const int mb = blockIdx.x, nb = blockIdx.y;
  const int n0 = nb * CB, m0 = mb * BM;
  const int nt0 = n0 / 16;
  const int ntiles = min(CB / 16, p.nt_total - nt0);
  const int nk = p.K / BK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < XS; ++i) {
      mbar_init(smem_addr(&xfull[i]), 1);
      mbar_init(smem_addr(&xempty[i]), 1);
    }
    for (int i = 0; i < WS; ++i) {
      mbar_init(smem_addr(&wfull[i]), 1);
      mbar_init(smem_addr(&wempty[i]), DQ_WARPS);
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
    // ------------------------------------------------------------ x producer
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int s = i % XS;
        if (i >= XS && !mbar_wait(smem_addr(&xempty[s]), ((i / XS) - 1) & 1, p.err, abort_flag)) break;
        const uint32_t fb = smem_addr(&xfull[s]);
        mbar_arrive_expect_tx(fb, A_BYTES);
        tma_load_2d(smem_addr(xring + s * A_BYTES), &p.tm_x, i * BK, m0, fb);
        issued = i + 1;
      }
      // No copy may still be writing this CTA's shared memory when it exits.
      for (int i = max(0, issued - XS); i < issued; ++i)
        mbar_wait(smem_addr(&xfull[i % XS]), (i / XS) & 1, p.err, nullptr);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ weight producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int s = i % WS;
        if (i >= WS && !mbar_wait(smem_addr(&wempty[s]), ((i / WS) - 1) & 1, p.err, abort_flag)) break;
        const uint32_t fb = smem_addr(&wfull[s]);
        const uint32_t base = smem_addr(wring + s * W_SLOT);
        const int g = i * BK / p.gs;
        mbar_arrive_expect_tx(fb, ntiles * 512 + CB * 2 + (ZERO ? CB * 4 : 0));  // scale and zero boxes of CB
        bulk_g2s(base, p.packed + ((size_t)i * p.nt_total + nt0) * 512, ntiles * 512, fb, pol);
        tma_load_2d(base + W_BYTES, &p.tm_s, n0, g, fb);
        if (ZERO) tma_load_2d(base + W_BYTES + S_BYTES, &p.tm_z, n0, g / 8, fb);
        issued = i + 1;
      }
      for (int i = max(0, issued - WS); i < issued; ++i)
        mbar_wait(smem_addr(&wfull[i % WS]), (i / WS) & 1, p.err, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id = tc::idesc<BF16>(UM, BN);
      for (int i = 0; i < nk; ++i) {
        const int s = i % XS, sb = i % BSTAGES;
        if (!mbar_wait(smem_addr(&bfull[sb]), (i / BSTAGES) & 1, p.err, abort_flag)) break;
        if (!mbar_wait(smem_addr(&xfull[s]), (i / XS) & 1, p.err, abort_flag)) break;
        tc::fence_after();
        const uint32_t a0 = smem_addr(xring + s * A_BYTES);
        const uint32_t b0 = smem_addr(bbuf + sb * B_BYTES);
#pragma unroll
        for (int h = 0; h < MSUB; ++h)
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc::mma(tmem + h * BN, tc::sw128_desc(a0 + h * (UM * 128) + kk * 32), tc::sw128_desc(b0 + kk * 32), id,
                    (i | kk) != 0 ? 1u : 0u);
        tc::commit(smem_addr(&xempty[s]));
        tc::commit(smem_addr(&bempty[sb]));
      }
      tc::commit(smem_addr(accfull));  // every MMA issued above has completed when this fires
    }
  } else {
    // ------------------------------------------------------------ dequant (warps 3..10)
    const int dq = threadIdx.x - 96;  // 0 .. 255
    constexpr uint32_t MAGIC = Magic<BF16>::kPair;
    for (int i = 0; i < nk; ++i) {
      const int s = i % WS, sb = i % BSTAGES;
      if (!mbar_wait(smem_addr(&wfull[s]), (i / WS) & 1, p.err, abort_flag)) break;
      const uint32_t base = smem_addr(wring + s * W_SLOT);
      const int g = i * BK / p.gs;
      // This thread's words, scales and zeros of the stage into registers;
      // then the weight slot goes back to the producer.
      constexpr int HALVES = CB * 2 / 256;  // (tile, lane) pairs per thread
      uint4 wv[2];
      uint32_t zz[2][2], ss[2][2];
#pragma unroll
      for (int half = 0; half < HALVES; ++half) {
        const int pr = dq + half * 256;  // (tile, lane) pair 0..511
        const int tile = pr >> 5, ln = tc::dq_slot(pr & 31);
        wv[half] = make_uint4(0u, 0u, 0u, 0u);
        if (tile < ntiles) {
          wv[half] = lds128(base + tile * 512 + ln * 16);
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int col = tile * 16 + (ln >> 2) + 8 * r;  // row of B (output channel within the tile)
            const uint16_t sbits = lds16(base + W_BYTES + col * 2);
            uint32_t z = 8;
            if (ZERO) z = (lds32(base + W_BYTES + S_BYTES + col * 4) >> ((g % 8) * 4)) & 15u;
            zz[half][r] = ((MAGIC & 0xFFFFu) + z) * 0x00010001u;  // (MAGIC + z) in both halves
            ss[half][r] = (uint32_t)sbits * 0x00010001u;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&wempty[s]));
      if (i >= BSTAGES && !mbar_wait(smem_addr(&bempty[sb]), ((i / BSTAGES) - 1) & 1, p.err, abort_flag)) break;
      const uint32_t bdst = smem_addr(bbuf + sb * B_BYTES);
#pragma unroll
      for (int half = 0; half < HALVES; ++half) {
        const int pr = dq + half * 256;
        const int tile = pr >> 5, ln = tc::dq_slot(pr & 31);
        if (tile < ntiles) {
          const int gq = ln >> 2, tq = ln & 3;
          const uint32_t w4[4] = {wv[half].x, wv[half].y, wv[half].z, wv[half].w};
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int col = tile * 16 + gq + 8 * r;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const uint32_t w = w4[2 * u + r];
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const uint32_t d0 = sub_pair<BF16>(code_pair<4, BF16>(w, 2 * j), zz[half][r]);      // q - z, exact
                const uint32_t d1 = sub_pair<BF16>(code_pair<4, BF16>(w, 2 * j + 1), zz[half][r]);
                const uint32_t lo = mul2<BF16>(d0, ss[half][r]);
                const uint32_t hi = mul2<BF16>(d1, ss[half][r]);
                const int k = 32 * u + 16 * j + 4 * tq;
                sts64(bdst + tc::sw128_off(col, k), lo, hi);
                if constexpr (SPLIT) {  // the rounding residues, in B rows 128..255
                  const uint32_t lo2 = fma2<BF16>(d0, ss[half][r], lo ^ 0x80008000u);
                  const uint32_t hi2 = fma2<BF16>(d1, ss[half][r], hi ^ 0x80008000u);
                  sts64(bdst + tc::sw128_off(col + BN / 2, k), lo2, hi2);
                }
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
        for (int c = 0; c < CB; c += 32) {
          float v[32];
          tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + h * BN + c, v);
          if constexpr (SPLIT) {  // + the residue terms' columns
            float v2[32];
            tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + h * BN + BN / 2 + c, v2);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] += v2[j];
          }
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

template <bool BF16, bool ZERO, int MS, bool SPLIT>
static cudaError_t launch_t(const pf::Params &pp, dim3 grid, bool persistent, cudaStream_t s) {
  auto kern = persistent ? pf::prefill_sk_kernel<BF16, ZERO, MS> : pf::prefill_kernel<BF16, ZERO, MS, SPLIT>;
  static int attr_set[64][2] = {{0}};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  // + slack for the 1024-byte alignment of the rings
  const int smem = (persistent ? pf::Cfg<MS>::SMEM : pf::DCfg<MS>::SMEM) + 1024;
  if (!attr_set[dev][persistent]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set[dev][persistent] = 1;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(persistent ? pf::SK_THREADS : pf::THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (persistent) {  // every CTA resident at once: the fix-up waits cannot deadlock
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, pp);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int MS, bool SPLIT>
static cudaError_t launch_ms_s(const pf::Params &pp, dim3 grid, bool sk, bool bf16, bool z, cudaStream_t s) {
  if (bf16)
    return z ? launch_t<true, true, MS, SPLIT>(pp, grid, sk, s) : launch_t<true, false, MS, SPLIT>(pp, grid, sk, s);
  return z ? launch_t<false, true, MS, SPLIT>(pp, grid, sk, s) : launch_t<false, false, MS, SPLIT>(pp, grid, sk, s);
}

template <int MS>
static cudaError_t launch_ms(const pf::Params &pp, dim3 grid, bool sk, bool bf16, bool z, bool split,
                             cudaStream_t s) {
  return split ? launch_ms_s<MS, true>(pp, grid, false, bf16, z, s) : launch_ms_s<MS, false>(pp, grid, sk, bf16, z, s);
}

// CTAs of the persistent launch: one per SM (the kernel's shared memory and
// TMEM allow one), at most two per tile (each cut tile then has about one
// partial to add), at most one per stage of work.
static long long prefill_ctas(long long tiles, long long units, int sms) {
  long long c = sms < 2 * tiles ? sms : 2 * tiles;
  return units < c ? units : c;
}

size_t prefill_workspace_bytes(int M, int N, int K, int sms) {
  const int bm = M <= pf::UM ? pf::UM : 2 * pf::UM;
  const long long tiles = (long long)((M + bm - 1) / bm) * ((N + pf::BN - 1) / pf::BN);
  if (4 * tiles > sms) return 0;  // one tile per CTA
  const long long units = tiles * (K / pf::BK);
  return (size_t)pf::kFlagBytes + (size_t)prefill_ctas(tiles, units, sms) * bm * pf::BN * sizeof(float);
}

cudaError_t launch_prefill(const MatmulArgs &a, int sms, void *workspace, size_t workspace_bytes, bool split_w,
                           cudaStream_t s) {
  pf::Params pp{};
  const int G = a.K / a.group_size;
  // One 128-token accumulator per tile up to 128 tokens, two (256 tokens) beyond.
  const int ms = a.M <= pf::UM ? 1 : 2;
  const int bm = pf::UM * ms;
  const int cb = split_w ? pf::BN / 2 : pf::BN;  // output channels per tile
  if (!encode_2d(&pp.tm_x, a.x, 2, (uint64_t)a.K, (uint64_t)a.M, pf::BK, (uint32_t)bm, 128))
    return cudaErrorInvalidValue;
  if (!encode_2d(&pp.tm_s, a.scales, 2, (uint64_t)a.N, (uint64_t)G, (uint32_t)cb, 1, 0))
    return cudaErrorInvalidValue;
  if (a.zeros &&
      !encode_2d(&pp.tm_z, a.zeros, 4, (uint64_t)a.N, (uint64_t)((G + 7) / 8), (uint32_t)cb, 1, 0))
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
  pp.tiles_m = (a.M + bm - 1) / bm;
  pp.nk = a.K / pf::BK;
  const long long tiles = (long long)pp.tiles_m * ((a.N + pf::BN - 1) / pf::BN);
  pp.units = tiles * pp.nk;
  // One tile per CTA, unless that leaves most SMs idle (fewer tiles than half
  // the SMs) and the workspace holds the partial tiles: then persistent CTAs
  // with stream-K shares.  With at least half the SMs busy, one tile per CTA
  // measured faster on the 8192 x 28672 weights (no fix-ups, and neighbouring
  // CTAs share each weight block in L2).
  dim3 grid((unsigned)pp.tiles_m, (unsigned)((a.N + cb - 1) / cb));
  bool sk = false;
  const size_t want = split_w ? 0 : prefill_workspace_bytes(a.M, a.N, a.K, sms);
  if (want > 0 && workspace && workspace_bytes >= want) {
    grid = dim3((unsigned)prefill_ctas(tiles, pp.units, sms));
    sk = true;
    pp.flags = static_cast<int *>(workspace);
    pp.partial = reinterpret_cast<float *>(static_cast<char *>(workspace) + pf::kFlagBytes);
  }
  const bool z = a.zeros != nullptr;
  return ms == 1 ? launch_ms<1>(pp, grid, sk, a.x_bf16, z, split_w, s)
                 : launch_ms<2>(pp, grid, sk, a.x_bf16, z, split_w, s);
}

}  // namespace wq
