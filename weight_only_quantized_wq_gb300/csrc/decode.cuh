// decode.cuh -- weight-only quantized matmul for few tokens (M <= 64).
//
// The step is bound by reading the packed weights (the tiny-llm int8_gemv
// docstring makes the same point for small M), so each weight byte is read
// from HBM once, through a deep shared-memory ring, and turned into
// tensor-core operands in registers.
//
// Roles (5 warps): one producer lane first copies the scale rows and the
// packed zero-word rows of all of the CTA's groups (two 2-D tensor copies),
// then, per slot of a ring stage (one chunk row of KC values of K; two slots
// per stage), a 1-D bulk copy of the packed weights of the CTA's 16*4*TN
// output channels and a 2-D tensor copy of the activation slice.  Four
// consumer warps (TN tiles of 16 channels each) build the (MAGIC + zero)
// pairs once, then wait for a stage, compute its slots and release it.
// Nothing else couples the warps, so a finished group is folded without
// waiting for anyone.
//
// Swap-AB: the weight tile (16 output channels x 16 k) is the A operand of
// mma.m16n8k16 and the tokens are its N = 8 columns, so the output channels
// fill the MMA's M dimension however few tokens there are.
//
// Exact group arithmetic (W = 2, 4): one shift and one LOP3 per pair turn two
// codes into MAGIC + q (exact in fp16 / bf16) and one subtraction of
// MAGIC + zero gives q - zero, a small integer, exactly (2-bit codes: six of
// a word's eight pairs are masked in place or after one shared shift and
// fixed by one exact fma; fp16 4-bit codes: the odd fields likewise).  The MMA sums
// x (q - zero) over one group in fp32 and the group's scale is applied to that
// sum (one FMA per value): no weight is ever rounded.  int8 codes (W = 8) are
// converted exactly and the per-channel scale is applied at the end (tiny-llm
// int8_matmul docstring).
//
// Group schedule (template FOLD): FOLD > 0 when the group size 16*FOLD divides
// the chunk (a group can end only after every FOLD-th k-step); FOLD == 0 when
// the chunk divides the group size (groups end on chunk boundaries); FOLD < 0
// for any other multiple of 16.  A CTA's K range may end inside a group
// (split-K); that partial group is folded at the range's end.
//
// Split-K: when the column blocks alone leave SMs idle, the K range is split.
// Up to 16 splits of a column block form one thread-block cluster: every CTA
// leaves its fp32 partial tile in its own shared memory, and after a cluster
// barrier each CTA sums one slice of the tile over the cluster's CTAs
// (distributed shared memory, split order) and writes it -- no global
// round trip, no workspace.  Beyond 16 splits each CTA writes its partial to
// the workspace and the last CTA to arrive for a column block (atomic
// counter, no waiting) adds the partials in split order.  Either way the
// result does not depend on arrival order.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "dev.cuh"
#include "kernels.h"
#include "layout.cuh"

namespace wq {

constexpr int kDecodeWarps = 4;  // consumer warps per CTA (plus one producer warp)
constexpr int kDecodeThreads = (kDecodeWarps + 1) * 32;
constexpr int kDecodeHeader = 256;  // mbarriers in front of the staged rows
// Ring depth in chunk rows (slots): 12 to 24 KB of weights in flight per CTA;
// 7- and 8-octet token tiles (56 or 64 rows of x per slot) keep 4, so that
// three CTAs fit an SM's shared memory (measured 86.6 against 96.5 us at c5
// M=64 with 8 octets).
__host__ __device__ constexpr int decode_stages(int mt) { return mt >= 7 ? 4 : 6; }
// A ring stage holds this many chunk rows (slots): one barrier wait and one
// release per pair of chunk rows.
constexpr int kSlotsPerStage = 2;
// Resident CTAs per SM the register budget is sized for.
// (every shape compiles to at most ~122 registers under this bound, no spills)
__host__ __device__ constexpr int decode_min_blocks(int, int) { return 3; }

__host__ __device__ constexpr int align128(int v) { return (v + 127) / 128 * 128; }

// Row pitch of the activation slice in shared memory: the 32-bit word count
// is 8 mod 32, which makes the 8-byte B-fragment loads of a warp conflict-free.
__host__ __device__ constexpr int x_pitch(int w) { return 4 * ((128 / w) + ((8 - (128 / w) % 32) + 32) % 32); }

// Shared-memory layout of one CTA: barriers | scales as stored (16-bit, one
// row per group) | (MAGIC + zero) pairs (one row per group, asymmetric codes
// only: zrows = srows, else 0) | packed zero words as stored (zwrows rows) |
// ring of stages, each of kSlotsPerStage slots (packed weights of one chunk
// row, then its activation slice).  The scale and
// zero-word rows arrive by TMA, one box each, so srows and zwrows are at most
// 256.
struct DecodeSmem {
  int w, mt, tn, srows, zrows, zwrows;
  __host__ __device__ constexpr int cols() const { return kDecodeWarps * tn * 16; }
  __host__ __device__ constexpr int s_off() const { return kDecodeHeader; }
  __host__ __device__ constexpr int z_off() const { return align128(s_off() + srows * cols() * 2); }
  __host__ __device__ constexpr int zw_off() const { return align128(z_off() + zrows * cols() * 4); }
  __host__ __device__ constexpr int ring_off() const { return align128(zw_off() + zwrows * cols() * 4); }
  __host__ __device__ constexpr int w_bytes() const { return cols() * 32; }  // one chunk row of weights
  __host__ __device__ constexpr int x_off() const { return w_bytes(); }
  __host__ __device__ constexpr int x_bytes() const { return mt * 8 * x_pitch(w); }
  __host__ __device__ constexpr int slot_bytes() const { return align128(x_off() + x_bytes()); }
  __host__ __device__ constexpr int stage_bytes() const { return kSlotsPerStage * slot_bytes(); }
  __host__ __device__ constexpr int bytes() const { return ring_off() + decode_stages(mt) * slot_bytes(); }
};

struct DecodeParams {
  CUtensorMap tm_x;  // x (M, K) 16-bit; box (x_pitch/2, 8*MT): the row pitch padding is real data or zeros
  CUtensorMap tm_s;  // scales (G, N) 16-bit; box (CTA columns, srows)       [grouped codes]
  CUtensorMap tm_z;  // zero words (ceil(G/V), N) 32-bit; box (CTA columns, zwrows) [asymmetric]
  const uint8_t *packed;
  const void *scales;     // (G, N) 16-bit, or (N,) fp32 for int8
  const uint32_t *zeros;  // (ceil(G / V), N) or nullptr
  void *out;
  int out_type;  // OutType
  float *partial;
  int *counters;
  uint32_t *err;
  int M, N, K, gs, nt_total, kch, splits, cps, srows, zrows, zwrows;
  long long wait_limit;  // SM cycles after which a barrier wait gives up
  int withhold;          // test hook: ring stage the producer never arms or fills (-1: none)
  int sym_zero;     // zero of every group without zero words
  bool unit_scale;  // every group scale is 1 (no scale rows)
  bool s_bf16;
  bool cluster;  // the splits of a column block form a cluster (reduction in shared memory)
};

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kDecodeWarps * 32) : "memory");
}


template <int W, bool BF16, int MT, int TN, bool ZERO, int FOLD>
__global__ void __launch_bounds__(kDecodeThreads, decode_min_blocks(MT, TN))
    decode_kernel(const __grid_constant__ DecodeParams p) {
  using G = Geo<W>;
  constexpr int NW = kDecodeWarps, STAGES = decode_stages(MT) / kSlotsPerStage;
  constexpr int SLOT = DecodeSmem{W, MT, TN, 0, 0, 0}.slot_bytes();
  constexpr int KS = G::KS, KC = G::KC, WK = G::WK, V = G::V;
  constexpr int XP = x_pitch(W);
  constexpr bool GROUPED = (W != 8);
  constexpr int CC = NW * TN * 16;  // output channels per CTA

  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_last;
  __shared__ volatile int s_abort;
  const DecodeSmem L{W, MT, TN, p.srows, p.zrows, p.zwrows};
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);
  uint64_t *empty = full + STAGES;
  uint64_t *meta = empty + STAGES;  // the scale and zero-word rows have landed
  static_assert((2 * STAGES + 1) * 8 <= kDecodeHeader, "barriers do not fit the header");
  const uint16_t *s_sm = reinterpret_cast<const uint16_t *>(smem + L.s_off());  // [srows][CC] scales
  const uint32_t *z_sm = reinterpret_cast<const uint32_t *>(smem + L.z_off());  // [zrows][CC] MAGIC + zero pairs
  uint8_t *ring = smem + L.ring_off();
  const int SB = L.stage_bytes();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = blockIdx.x, split = blockIdx.y;
  const int nt0 = nb * NW * TN;
  const int ntiles = min(NW * TN, p.nt_total - nt0);
  const int n0 = nt0 * 16;
  const int c0 = split * p.cps;
  const int nch = min(p.kch, c0 + p.cps) - c0;
  const int kbeg = c0 * KC, kend = kbeg + nch * KC;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_addr(&full[i]), 1);
      mbar_init(smem_addr(&empty[i]), NW * 32);  // every consumer lane arrives
    }
    mbar_init(smem_addr(meta), 1);
    s_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == NW) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_w = policy_evict_first();
    const uint32_t wbytes = (uint32_t)ntiles * 512u;
    const uint32_t xbytes = (uint32_t)L.x_bytes();
    int issued = 0;
    const int g0 = GROUPED ? kbeg / p.gs : 0;
    if (GROUPED && lane == 0) {  // this CTA's scale rows (and zero-word rows) ahead of the ring
      const uint32_t mb = smem_addr(meta);
      mbar_arrive_expect_tx(mb, (uint32_t)(L.srows * CC * 2 + L.zwrows * CC * 4));
      if (!p.unit_scale) tma_load_2d(smem_addr(smem + L.s_off()), &p.tm_s, n0, g0, mb);
      if (ZERO) tma_load_2d(smem_addr(smem + L.zw_off()), &p.tm_z, n0, g0 / V, mb);
    }
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0;  // phase parity of the ring's current lap
      const int nst = (nch + kSlotsPerStage - 1) / kSlotsPerStage;
      for (int i = 0; i < nst; ++i) {
        if (i >= STAGES && !mbar_wait(smem_addr(&empty[st]), ph ^ 1u, p.err, &s_abort, p.wait_limit)) break;
        if (i == p.withhold) {  // test hook: the consumers' wait for this stage must run out
          issued = i + 1;
          if (++st == STAGES) {
            st = 0;
            ph ^= 1u;
          }
          continue;
        }
        const uint32_t fb = smem_addr(&full[st]);
        const uint32_t base = smem_addr(ring + st * SB);
        const int ns = min(kSlotsPerStage, nch - i * kSlotsPerStage);
        mbar_arrive_expect_tx(fb, (uint32_t)ns * (wbytes + xbytes));
        for (int j = 0; j < ns; ++j) {
          const int kc = c0 + i * kSlotsPerStage + j;
          bulk_g2s(base + j * SLOT, p.packed + ((size_t)kc * p.nt_total + nt0) * 512, wbytes, fb, pol_w);
          tma_load_2d(base + j * SLOT + L.x_off(), &p.tm_x, kc * KC, 0, fb);
        }
        issued = i + 1;
        if (++st == STAGES) {
          st = 0;
          ph ^= 1u;
        }
      }
      // No copy may still be writing this CTA's shared memory when it exits.
      for (int i = max(0, issued - STAGES); i < issued; ++i)
        if (i != p.withhold) mbar_wait(smem_addr(&full[i % STAGES]), (i / STAGES) & 1, p.err, nullptr, p.wait_limit);
      if (GROUPED) mbar_wait(smem_addr(meta), 0, p.err, nullptr, p.wait_limit);
    }
    __syncwarp();
    if (p.cluster) {  // the consumers' two cluster barriers
      cluster_sync();
      cluster_sync_relaxed();
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, t = lane & 3;
  const int wt0 = warp * TN;  // first tile of this warp within the CTA

  // The scale rows stay as stored (16-bit, converted when a group is
  // folded); the packed zero words become one (MAGIC + zero) pair per group
  // and column, built once per CTA.
  const int g0 = GROUPED ? kbeg / p.gs : 0;
  if constexpr (GROUPED) {
    const bool ok = mbar_wait(smem_addr(meta), 0, p.err, &s_abort, p.wait_limit);
    if (ZERO && ok) {
      const int ng = (kend - 1) / p.gs - g0 + 1;
      const int wr0 = g0 / V;
      const uint32_t *zw = reinterpret_cast<const uint32_t *>(smem + L.zw_off());
      uint32_t *zz_out = reinterpret_cast<uint32_t *>(smem + L.z_off());
      for (int idx = threadIdx.x; idx < ng * (CC / 4); idx += NW * 32) {
        const int row = idx / (CC / 4), c = (idx % (CC / 4)) * 4;
        const int gi = g0 + row, sh = (gi % V) * W;
        const uint4 w4 = *reinterpret_cast<const uint4 *>(zw + (gi / V - wr0) * CC + c);
        const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
        uint32_t zp[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          zp[e] = ((Magic<BF16>::kPair & 0xFFFFu) + ((ww[e] >> sh) & ((1u << W) - 1u))) * 0x00010001u;
        *reinterpret_cast<uint4 *>(zz_out + row * CC + c) = make_uint4(zp[0], zp[1], zp[2], zp[3]);
      }
    }
    consumer_sync();
  }

  float acc[TN][MT][4];
  float accg[TN][MT][4];
#pragma unroll
  for (int i = 0; i < TN; ++i)
#pragma unroll
    for (int j = 0; j < MT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][j][e] = accg[i][j][e] = 0.f;

  // (MAGIC + zero) of the current group for rows g and g + 8 of every tile
  uint32_t zz[TN][2];
  // fp16 int4 only: 960 - (1024 + zero), the fma addend of the odd fields
  constexpr bool kOddFma = W == 4 && !BF16;
  uint32_t zz16[TN][2];
  // 2-bit codes: the fma addends -(MAGIC/4 + zero) and -(MAGIC/16 + zero)
  uint32_t n2[TN][2], n4[TN][2];
  auto set_zeros = [&](int gi) {
#pragma unroll
    for (int ti = 0; ti < TN; ++ti)
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        if constexpr (ZERO)
          zz[ti][rr] = z_sm[(gi - g0) * CC + (wt0 + ti) * 16 + g + 8 * rr];
        else
          zz[ti][rr] = ((Magic<BF16>::kPair & 0xFFFFu) + (uint32_t)p.sym_zero) * 0x00010001u;
        if constexpr (kOddFma) zz16[ti][rr] = sub_pair<false>(kF16NineSixty, zz[ti][rr]);
        if constexpr (W == 2) {
          n2[ti][rr] = sub_pair<BF16>(Int2InPlace<BF16>::kMagic3of4, zz[ti][rr]);
          n4[ti][rr] = sub_pair<BF16>(Int2InPlace<BF16>::kMagic15of16, zz[ti][rr]);
        }
      }
  };
  // acc += scale[gi] * (sum over group gi); the group sum restarts.
  auto fold = [&](int gi) {
#pragma unroll
    for (int ti = 0; ti < TN; ++ti)
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const float s =
            p.unit_scale ? 1.f : half_bits_to_float(s_sm[(gi - g0) * CC + (wt0 + ti) * 16 + g + 8 * rr], p.s_bf16);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            acc[ti][mt][2 * rr + c] = fmaf(s, accg[ti][mt][2 * rr + c], acc[ti][mt][2 * rr + c]);
            accg[ti][mt][2 * rr + c] = 0.f;
          }
      }
  };

  int cur_g = g0;
  int next_fold = GROUPED ? min((g0 + 1) * p.gs, kend) : kend;
  if constexpr (GROUPED) set_zeros(g0);

  // A barrier test returns after some latency even when the phase is
  // complete, so a non-blocking test of each stage's barrier is issued one
  // stage early and its answer is only read when that stage starts.
  const int nst = (nch + kSlotsPerStage - 1) / kSlotsPerStage;
  bool next_ready = nst > 0 && mbar_test_wait(smem_addr(&full[0]), 0);
  int st = 0, st1 = 1 % STAGES;  // this stage and the next (ring positions)
  uint32_t ph = 0, ph1 = STAGES == 1 ? 1u : 0u;  // their phase parities
  for (int i = 0; i < nst; ++i) {
    if (!next_ready && !mbar_wait(smem_addr(&full[st]), ph, p.err, &s_abort, p.wait_limit)) break;
    if (i + 1 < nst) next_ready = mbar_test_wait(smem_addr(&full[st1]), ph1);
#pragma unroll
    for (int sl = 0; sl < kSlotsPerStage; ++sl) {
      if (sl > 0 && i * kSlotsPerStage + sl >= nch) break;
      const uint32_t base = smem_addr(ring + st * SB) + sl * SLOT;
      const int kc0 = kbeg + (i * kSlotsPerStage + sl) * KC;
      uint4 wv[TN];
#pragma unroll
      for (int ti = 0; ti < TN; ++ti)
        wv[ti] = (wt0 + ti) < ntiles ? lds128(base + (wt0 + ti) * 512 + lane * 16) : make_uint4(0, 0, 0, 0);

#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        if constexpr (GROUPED) {
          const bool maybe = FOLD == 0 ? (ks == 0) : FOLD > 0 ? (ks % (FOLD > 0 ? FOLD : 1) == 0) : true;
          if (maybe && kc0 + ks * 16 == next_fold) {  // a group ended before this k-step
            fold(cur_g);
            ++cur_g;
            next_fold = min(next_fold + p.gs, kend);
            set_zeros(cur_g);
          }
        }
        uint32_t b[MT][2];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const uint2 v = lds64(base + L.x_off() + (mt * 8 + g) * XP + ks * 32 + t * 8);
          b[mt][0] = v.x;
          b[mt][1] = v.y;
        }
        const int h = ks / WK, j = ks % WK;
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
          } else if constexpr (kOddFma) {
            // fields 2j and 2j + 1 from one shift by 8 j
            const uint32_t v = wg >> (8 * j), v8 = wg8 >> (8 * j);
            a0 = sub_pair<false>(and_or(v, 0x000F000Fu, Magic<false>::kPair), zz[ti][0]);
            a1 = sub_pair<false>(and_or(v8, 0x000F000Fu, Magic<false>::kPair), zz[ti][1]);
            a2 = fma_h2(and_or(v, 0x00F000F0u, Magic<false>::kPair), kF16Sixteenth, zz16[ti][0]);
            a3 = fma_h2(and_or(v8, 0x00F000F0u, Magic<false>::kPair), kF16Sixteenth, zz16[ti][1]);
          } else if constexpr (W == 2) {
            a0 = int2_pair<BF16>(wg, 2 * j, zz[ti][0], n2[ti][0], n4[ti][0]);
            a1 = int2_pair<BF16>(wg8, 2 * j, zz[ti][1], n2[ti][1], n4[ti][1]);
            a2 = int2_pair<BF16>(wg, 2 * j + 1, zz[ti][0], n2[ti][0], n4[ti][0]);
            a3 = int2_pair<BF16>(wg8, 2 * j + 1, zz[ti][1], n2[ti][1], n4[ti][1]);
          } else {
            a0 = sub_pair<BF16>(code_pair<W, BF16>(wg, 2 * j), zz[ti][0]);
            a1 = sub_pair<BF16>(code_pair<W, BF16>(wg8, 2 * j), zz[ti][1]);
            a2 = sub_pair<BF16>(code_pair<W, BF16>(wg, 2 * j + 1), zz[ti][0]);
            a3 = sub_pair<BF16>(code_pair<W, BF16>(wg8, 2 * j + 1), zz[ti][1]);
          }
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            if (GROUPED)
              mma16816<BF16>(accg[ti][mt], a0, a1, a2, a3, b[mt][0], b[mt][1]);
            else
              mma16816<BF16>(acc[ti][mt], a0, a1, a2, a3, b[mt][0], b[mt][1]);
          }
        }
      }
    }  // slots of the stage
    mbar_arrive(smem_addr(&empty[st]));  // this lane is done with the stage
    st = st1;
    ph = ph1;
    if (++st1 == STAGES) {
      st1 = 0;
      ph1 ^= 1u;
    }
  }
  if constexpr (GROUPED) fold(cur_g);

  // -------------------------------------------------------------- epilogue
  const float *sc32 = static_cast<const float *>(p.scales);
  if (p.cluster) {
    // Partial tile -> own shared memory (the ring is free: every stage was consumed).
    constexpr int RP = CC + 4;  // row pitch (floats): fragment stores are conflict-free
    const uint32_t red = smem_addr(ring);
    consumer_sync();
#pragma unroll
    for (int ti = 0; ti < TN; ++ti)
#pragma unroll
      for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int m = mt * 8 + 2 * t + c;
            if (m < p.M) sts_f32(red + (m * RP + (wt0 + ti) * 16 + g + 8 * rr) * 4, acc[ti][mt][2 * rr + c]);
          }
    cluster_sync();
    // This CTA's slice of the tile, summed over the cluster in split order.
    const uint32_t rank = cluster_ctarank();
    const int qpr = ntiles * 4;  // float4 quads per row
    const int nq = p.M * qpr;
    for (int q = threadIdx.x * p.splits + (int)rank; q < nq; q += NW * 32 * p.splits) {
      const int m = q / qpr, col = (q % qpr) * 4;
      const uint32_t la = red + (m * RP + col) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      // up to eight remote loads in flight before the adds (still in split order)
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
      if (W == 8) {
        const float4 s4 = __ldg(reinterpret_cast<const float4 *>(sc32 + n0 + col));
        v.x *= s4.x;
        v.y *= s4.y;
        v.z *= s4.z;
        v.w *= s4.w;
      }
      store_out4(p.out, (size_t)m * p.N + n0 + col, v, p.out_type);
    }
    __syncwarp();
    cluster_sync_relaxed();  // no CTA leaves while another still reads its shared memory
    return;
  }
  // One split: the result itself (in the output type); more: this split's
  // fp32 partial in the workspace.
  void *dst = p.splits == 1 ? p.out : static_cast<void *>(p.partial + (size_t)split * p.M * p.N);
  const int dst_type = p.splits == 1 ? p.out_type : kOutF32;
#pragma unroll
  for (int ti = 0; ti < TN; ++ti) {
    if (wt0 + ti >= ntiles) continue;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int n = n0 + (wt0 + ti) * 16 + g + 8 * rr;
      const float s8 = (W == 8 && p.splits == 1) ? __ldg(sc32 + n) : 1.f;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int m = mt * 8 + 2 * t + c;
          if (m < p.M) store_out1(dst, (size_t)m * p.N + n, acc[ti][mt][2 * rr + c] * s8, dst_type);
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
      for (int q = 0; q < 8; ++q)
        if (q < cnt) part[q] = __ldcg(reinterpret_cast<const float4 *>(p.partial + ((size_t)(sp0 + q) * p.M + m) * p.N + n));
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q < cnt) {
          v.x += part[q].x;
          v.y += part[q].y;
          v.z += part[q].z;
          v.w += part[q].w;
        }
    }
    if (W == 8) {
      const float4 s4 = __ldg(reinterpret_cast<const float4 *>(sc32 + n));
      v.x *= s4.x;
      v.y *= s4.y;
      v.z *= s4.z;
      v.w *= s4.w;
    }
    store_out4(p.out, (size_t)m * p.N + n, v, p.out_type);
  }
  if (threadIdx.x == 0) p.counters[nb] = 0;
}

// Kernel attributes a launch (or an occupancy query) of `smem` dynamic
// shared memory and clusters of more than eight CTAs needs, set once per
// device and size.
template <int W, bool BF16, int MT, int TN, bool ZERO, int FOLD>
cudaError_t prepare_decode_t(int smem, bool big_cluster) {
  auto kern = decode_kernel<W, BF16, MT, TN, ZERO, FOLD>;
  static int attr_bytes[64] = {0};
  static bool nonportable[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (attr_bytes[dev] < smem) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_bytes[dev] = smem;
  }
  if (big_cluster && !nonportable[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    nonportable[dev] = true;
  }
  return cudaSuccess;
}

template <int W, bool BF16, int MT, int TN, bool ZERO, int FOLD>
cudaError_t launch_decode_t(const DecodeParams &dp, const DecodePlan &p, cudaStream_t s) {
  auto kern = decode_kernel<W, BF16, MT, TN, ZERO, FOLD>;
  const int smem = p.smem;
  cudaError_t e = prepare_decode_t<W, BF16, MT, TN, ZERO, FOLD>(smem, dp.cluster && p.splits > 8);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(p.nblocks, p.splits);
  cfg.blockDim = dim3(kDecodeThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (dp.cluster) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = p.splits;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  e = cudaLaunchKernelEx(&cfg, kern, dp);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// CTAs of one launch that can be resident at once, from the runtime's
// occupancy calculator: CTAs per SM x SMs, and for a cluster launch of
// `splits` CTAs the clusters the GPCs can hold x splits.  -1 on error.
template <int W, bool BF16, int MT, int TN, bool ZERO, int FOLD>
long decode_capacity_t(int smem, int splits, int sms) {
  auto kern = decode_kernel<W, BF16, MT, TN, ZERO, FOLD>;
  const bool cluster = splits > 1 && splits <= kMaxClusterSplits;
  if (prepare_decode_t<W, BF16, MT, TN, ZERO, FOLD>(smem, cluster && splits > 8) != cudaSuccess) return -1;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDecodeThreads, smem) != cudaSuccess) return -1;
  long cap = (long)per_sm * sms;
  if (cluster) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(1, splits);
    cfg.blockDim = dim3(kDecodeThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = splits;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int nc = 0;
    if (cudaOccupancyMaxActiveClusters(&nc, kern, &cfg) != cudaSuccess) return -1;
    cap = cap < (long)nc * splits ? cap : (long)nc * splits;
  }
  return cap;
}

// Launcher for one code width and group schedule (decode_inst.cu, compiled
// once per pair the build lists).
template <int W, int FOLD>
cudaError_t launch_decode_wf(const DecodeParams &dp, const DecodePlan &p, bool bf16, bool zero, cudaStream_t s);

template <int W, int FOLD>
long decode_capacity_wf(int mt, int tn, bool zero, int smem, int splits, int sms);

#define WQ_DECODE_CASE(W, BF, MT, TN, Z, F)                               \
  if (bf16 == BF && zero == Z && p.mt == MT && p.tn == TN && p.fold == F) \
    return launch_decode_t<W, BF, MT, TN, Z, F>(dp, p, s);

// The capacity of the bf16 instantiation stands for both activation types
// (the plan, and so the workspace size, must not depend on the x dtype).
#define WQ_DECODE_CAPACITY(W, MT, TN, Z, F) \
  if (zero == Z && mt == MT && tn == TN) return decode_capacity_t<W, true, MT, TN, Z, F>(smem, splits, sms);

}  // namespace wq
