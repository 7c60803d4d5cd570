// decode.cu -- host side of the few-token kernel: work split and dispatch.
#include <cuda.h>
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <tuple>

#include "decode.cuh"

namespace wq {

// The workspace starts with a fixed region of kMaxColumnBlocks arrival
// counters (enough for N up to 16 * 4 * kMaxColumnBlocks), so that counters
// never share bytes with the fp32 partials that follow, whatever M and N a
// call has: a workspace left zeroed by one call is ready for any other.
size_t decode_counter_bytes() { return (size_t)kMaxColumnBlocks * sizeof(int); }

// Group schedule of the kernel instantiations (decode_inst.cu is compiled for
// these values): int4 chunks span 64 k, int2 chunks 128 k, int8 chunks 32 k.
static int fold_for(int w_bit, int gs) {
  const int kc = 256 / w_bit;
  if (w_bit == 8 || gs % kc == 0) return 0;
  if (kc % gs == 0) {
    const int f = gs / 16;
    if (w_bit == 4 && f == 2) return 2;
    if (w_bit == 2 && (f == 2 || f == 4)) return f;
  }
  return -1;
}

// Scale rows and zero-word rows one CTA's K range touches, for splits of cps chunk rows.
static void rows_for(int K, int kc, int gs, int cps, int V, int *srows, int *zrows) {
  int sr = 1, zr = 1;
  const int kch = K / kc;
  for (int c0 = 0; c0 < kch; c0 += cps) {
    const int kb = c0 * kc, ke = (c0 + cps < kch ? c0 + cps : kch) * kc;
    const int ga = kb / gs, gb = (ke - 1) / gs;
    sr = gb - ga + 1 > sr ? gb - ga + 1 : sr;
    zr = gb / V - ga / V + 1 > zr ? gb / V - ga / V + 1 : zr;
  }
  *srows = sr;
  *zrows = zr;
}

// Resident-CTA capacity of one launch shape (decode_capacity_t), asked once
// per device and shape.  Clusters of up to kMaxClusterSplits CTAs carry the
// K splits; more splits run as independent CTAs.
static long capacity(int w_bit, int fold, int mt, int tn, bool zero, int smem, int splits, int sms) {
  const int cs = (splits > 1 && splits <= kMaxClusterSplits) ? splits : 1;
  const bool z = zero && w_bit != 8;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  using Key = std::tuple<int, int, int, int, int, bool, int, int>;
  static std::map<Key, long> cache;
  static std::mutex mu;
  const Key key{dev, w_bit, fold, mt, tn, z, smem, cs};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  long c = -1;
  switch (w_bit * 16 + fold) {
    case 2 * 16 + 0: c = decode_capacity_wf<2, 0>(mt, tn, z, smem, cs, sms); break;
    case 2 * 16 + 2: c = decode_capacity_wf<2, 2>(mt, tn, z, smem, cs, sms); break;
    case 2 * 16 + 4: c = decode_capacity_wf<2, 4>(mt, tn, z, smem, cs, sms); break;
    case 2 * 16 - 1: c = decode_capacity_wf<2, -1>(mt, tn, z, smem, cs, sms); break;
    case 4 * 16 + 0: c = decode_capacity_wf<4, 0>(mt, tn, z, smem, cs, sms); break;
    case 4 * 16 + 2: c = decode_capacity_wf<4, 2>(mt, tn, z, smem, cs, sms); break;
    case 4 * 16 - 1: c = decode_capacity_wf<4, -1>(mt, tn, z, smem, cs, sms); break;
    case 8 * 16 + 0: c = decode_capacity_wf<8, 0>(mt, tn, z, smem, cs, sms); break;
  }
  cudaGetLastError();  // a failed query leaves no error behind for the next launch
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = c;
  return c;
}

static DecodePlan plan_decode_search(int M, int N, int K, int w_bit, int group_size, bool zero, int sms,
                                     bool unit_scale) {
  DecodePlan best{};
  const int rows = M < 64 ? M : 64;
  // token octets per MMA column block: the MMAs per weight fragment grow with
  // it, so it follows M closely (every octet is one more mma.sync per fragment)
  const int mt = rows <= 32 ? (rows + 7) / 8 : rows <= 40 ? 5 : rows <= 48 ? 6 : rows <= 56 ? 7 : 8;
  const int kc = 256 / w_bit;
  const int nt = N / 16;
  const int kch = K / kc;
  const int gs = (w_bit == 8 || group_size <= 0) ? K : group_size;
  const bool grouped = w_bit != 8;
  const int V = 32 / w_bit;
  // Two 16-channel tiles per warp (the CTA covers 128 channels) keep three
  // CTAs of four consumer warps on an SM; 48- and 64-row slices take one.
  const int tn = mt >= 4 ? 1 : 2;
  const int nblocks = (nt + kDecodeWarps * tn - 1) / (kDecodeWarps * tn);
  const double unit_bytes = (double)tn * kDecodeWarps * 512.0;  // one chunk row of a CTA
  const int fold = fold_for(w_bit, gs);
  double best_cost = 1e300;
  const int smax = kch < 256 ? kch : 256;
  for (int s = 1; s <= smax; ++s) {
    const int cps = (kch + s - 1) / s;
    const int sreal = (kch + cps - 1) / cps;
    if (s != sreal) continue;
    int srows = 0, zwrows = 0;
    if (grouped) rows_for(K, kc, gs, cps, V, &srows, &zwrows);
    if (unit_scale) srows = 0;  // no scale rows are staged
    if (!zero) zwrows = 0;
    const int zrows = zero ? srows : 0;  // one (MAGIC + zero) row per group
    if (srows > 256 || zwrows > 256) continue;  // one TMA box each
    const int smem = DecodeSmem{w_bit, mt, tn, srows, zrows, zwrows}.bytes();
    if (smem > 200 * 1024) continue;
    long cap = capacity(w_bit, fold, mt, tn, zero, smem, sreal, sms);
    if (cap < 0) {  // no answer from the runtime: the register budget the kernel is compiled for
      int occ = decode_min_blocks(mt, tn);
      const int by_smem = (228 * 1024) / (smem + 1024);
      cap = (long)sms * (occ < by_smem ? occ : by_smem);
    }
    if (cap < 1) continue;
    // Estimated time in microseconds.  The busiest SM streams per_sm CTAs'
    // chunk rows; an SM's rate grows with the CTAs it runs at once (r), as
    // their warps hide each other's latency (rate r / (r + 3) of about
    // 60 KB/us, fitted to measured decode launches).  Each wave then pays the
    // K-split reduction: a cluster's barriers and remote loads cost about
    // 0.3 us + 0.5 us per split, plus a round trip per eight splits beyond
    // the first eight; through the workspace the last CTA of a column block
    // adds the partials, its threads taking a round trip of about 1 us per
    // eight splits for every 128 quads of outputs.
    const long units = (long)nblocks * sreal;
    const long waves = (units + cap - 1) / cap;
    const long per_sm_max = (cap + sms - 1) / sms;
    const long per_sm = units <= cap ? (units + sms - 1) / sms : waves * per_sm_max;
    const double r = (double)(per_sm < per_sm_max ? per_sm : per_sm_max);
    double cost = (double)per_sm * cps * unit_bytes / (60e3 * r / (r + 3.0));
    if (sreal == 1) cost += 0.3 * waves;
    else if (sreal <= kMaxClusterSplits) cost += (0.3 + 0.5 * sreal + 1.0 * ((sreal + 7) / 8 - 1)) * waves;
    else cost += (2.0 + 1.0 * ((rows * kDecodeWarps * tn * 4 + 127) / 128) * ((sreal + 7) / 8)) * waves;
    if (cost < best_cost * 0.999) {
      best_cost = cost;
      best.mt = mt;
      best.tn = tn;
      best.nblocks = nblocks;
      best.splits = sreal;
      best.cps = cps;
      best.srows = srows;
      best.zrows = zrows;
      best.zwrows = zwrows;
      best.smem = smem;
    }
  }
  best.fold = fold;
  best.cluster = best.splits > 1 && best.splits <= kMaxClusterSplits;
  best.workspace = best.splits > kMaxClusterSplits
                       ? decode_counter_bytes() + (size_t)best.splits * rows * N * sizeof(float)
                       : 0;
  return best;
}

// The plan of a shape, searched once per device and shape (a call then costs
// one lookup instead of a search over every split count).
DecodePlan plan_decode(int M, int N, int K, int w_bit, int group_size, bool zero, int sms, bool unit_scale) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  using Key = std::tuple<int, int, int, int, int, int, bool, int, bool>;
  static std::map<Key, DecodePlan> cache;
  static std::mutex mu;
  const Key key{dev, M, N, K, w_bit, group_size, zero, sms, unit_scale};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  const DecodePlan p = plan_decode_search(M, N, K, w_bit, group_size, zero, sms, unit_scale);
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() > 4096) cache.clear();  // bounded: a process with many shapes searches again
  cache.emplace(key, p);
  return p;
}

cudaError_t launch_decode(const MatmulArgs &a, const DecodePlan &p, void *workspace, cudaStream_t s) {
  DecodeParams dp{};
  dp.packed = static_cast<const uint8_t *>(a.packed);
  dp.err = a.err;
  dp.scales = a.scales;
  dp.zeros = a.zeros;
  dp.out = a.out;
  dp.out_type = a.out_type;
  dp.M = a.M;
  dp.N = a.N;
  dp.K = a.K;
  dp.gs = a.group_size;
  dp.nt_total = a.N / 16;
  dp.kch = a.K / (256 / a.w_bit);
  dp.splits = p.splits;
  dp.cps = p.cps;
  dp.srows = p.srows;
  dp.zrows = p.zrows;
  dp.zwrows = p.zwrows;
  dp.s_bf16 = a.s_bf16;
  dp.unit_scale = a.unit_scale;
  dp.wait_limit = a.wait_limit > 0 ? a.wait_limit : kWaitLimitCycles;
  dp.withhold = a.withhold;
  dp.sym_zero = a.sym_zero;
  dp.cluster = p.cluster;
  if (p.splits > 1 && !p.cluster) {
    dp.counters = static_cast<int *>(workspace);
    dp.partial = reinterpret_cast<float *>(static_cast<char *>(workspace) + decode_counter_bytes());
  }
  // Tensor map of the activation slice of a slot (rows past M read as zeros).
  if (!encode_2d(&dp.tm_x, a.x, 2, (uint64_t)a.K, (uint64_t)a.M, (uint32_t)(x_pitch(a.w_bit) / 2), (uint32_t)(p.mt * 8)))
    return cudaErrorInvalidValue;
  // Scale rows and zero-word rows of a CTA: one box of (CTA columns x rows) each.
  const uint32_t cols = (uint32_t)(kDecodeWarps * p.tn * 16);
  if (a.w_bit != 8) {
    const int G = a.K / a.group_size, V = 32 / a.w_bit;
    if (!a.unit_scale && !encode_2d(&dp.tm_s, a.scales, 2, (uint64_t)a.N, (uint64_t)G, cols, (uint32_t)p.srows))
      return cudaErrorInvalidValue;
    if (a.zeros && !encode_2d(&dp.tm_z, a.zeros, 4, (uint64_t)a.N, (uint64_t)((G + V - 1) / V), cols, (uint32_t)p.zwrows))
      return cudaErrorInvalidValue;
  }
  const bool z = a.zeros != nullptr;
  const bool bf = a.x_bf16;
  switch (a.w_bit * 16 + p.fold) {
    case 2 * 16 + 0: return launch_decode_wf<2, 0>(dp, p, bf, z, s);
    case 2 * 16 + 2: return launch_decode_wf<2, 2>(dp, p, bf, z, s);
    case 2 * 16 + 4: return launch_decode_wf<2, 4>(dp, p, bf, z, s);
    case 2 * 16 - 1: return launch_decode_wf<2, -1>(dp, p, bf, z, s);
    case 4 * 16 + 0: return launch_decode_wf<4, 0>(dp, p, bf, z, s);
    case 4 * 16 + 2: return launch_decode_wf<4, 2>(dp, p, bf, z, s);
    case 4 * 16 - 1: return launch_decode_wf<4, -1>(dp, p, bf, z, s);
    case 8 * 16 + 0: return launch_decode_wf<8, 0>(dp, p, bf, false, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace wq
