// decode.cu -- host side of the few-token kernel: work split and dispatch.
#include <cuda.h>
#include <cuda_runtime.h>

#include "decode.cuh"

namespace wq {

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
    tried = true;
  }
  return fn;
}

// Row-major 2-D tensor (rows x cols, `esize`-byte elements) and a box of
// (box_cols x box_rows), no swizzle, zero fill outside the tensor.
static bool encode_2d(CUtensorMap *m, const void *base, int esize, uint64_t cols, uint64_t rows, uint32_t box_cols,
                      uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * (uint64_t)esize};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(base),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The workspace starts with a fixed region of kMaxColumnBlocks arrival
// counters (enough for N up to 16 * 4 * kMaxColumnBlocks), so that counters
// never share bytes with the fp32 partials that follow, whatever M and N a
// call has: a workspace left zeroed by one call is ready for any other.
size_t decode_counter_bytes() { return (size_t)kMaxColumnBlocks * sizeof(int); }

// Largest number of groups any chunk row of KC values touches.
static int groups_per_chunk(int K, int kc, int gs) {
  int best = 1;
  for (int c = 0; c < K / kc; ++c) {
    const int r = ((c + 1) * kc - 1) / gs - (c * kc) / gs + 1;
    best = r > best ? r : best;
  }
  return best;
}

static int align128(int v) { return (v + 127) / 128 * 128; }

static int x_pitch_for(int w_bit) {
  const int words = (256 / w_bit) / 2;
  return 4 * (words + ((8 - words % 32) + 32) % 32);
}

// Mirrors DecodeLayout<W, MT, TN>::stage_bytes.
static int stage_bytes_for(int w_bit, int mt, int tn, int gcap, bool zero) {
  const int kc = 256 / w_bit;
  const int cols = kDecodeWarps * tn * 16;
  const int soff = align128(cols * kc * w_bit / 8 + mt * 8 * x_pitch_for(w_bit));
  if (w_bit == 8) return soff;
  const int zoff = align128(soff + gcap * cols * 2);
  const int poff = align128(zoff + (zero ? 2 * cols * 4 : 0));
  return align128(poff + gcap * cols * 8);
}

DecodePlan plan_decode(int M, int N, int K, int w_bit, int group_size, bool zero, int sms) {
  DecodePlan best{};
  const int rows = M < 64 ? M : 64;
  const int mt = rows <= 8 ? 1 : rows <= 16 ? 2 : rows <= 32 ? 4 : 8;
  const int kc = 256 / w_bit;
  const int nt = N / 16;
  const int kch = K / kc;
  const int gs = (w_bit == 8 || group_size <= 0) ? K : group_size;
  const int gcap = w_bit == 8 ? 0 : groups_per_chunk(K, kc, gs);
  int tns[2] = {4, 2};
  int ntn = 2;
  if (mt == 4) { tns[0] = 2; ntn = 1; }
  if (mt == 8) { tns[0] = 1; ntn = 1; }
  double best_cost = 1e300;
  for (int a = 0; a < ntn; ++a) {
    const int tn = tns[a];
    const int nblocks = (nt + kDecodeWarps * tn - 1) / (kDecodeWarps * tn);
    const int smem = kDecodeHeader + decode_stages(tn) * stage_bytes_for(w_bit, mt, tn, gcap, zero);
    int occ = decode_min_blocks(mt, tn);  // the register budget the kernel is compiled for
    const int by_smem = (228 * 1024) / (smem + 1024);
    occ = occ < by_smem ? occ : by_smem;
    if (occ < 1) occ = 1;
    const long slots = (long)sms * occ;
    const int smax = kch < 64 ? kch : 64;
    for (int s = 1; s <= smax; ++s) {
      const int cps = (kch + s - 1) / s;
      const int sreal = (kch + cps - 1) / cps;
      if (s != sreal) continue;
      const long units = (long)nblocks * sreal;
      // weight bytes the busiest SM streams (one wave if the units fit the slots)
      const long per_sm = units <= slots ? (units + sms - 1) / sms : ((units + slots - 1) / slots) * occ;
      double cost = (double)per_sm * cps * tn * kDecodeWarps * 512.0;
      // the partial sums' round trip, spread over the SMs
      if (sreal > 1) cost += 8.0 * rows * (double)N * sreal / sms;
      if (tn < 4) cost *= 1.05;  // narrower CTAs spend more instructions per weight on the activations
      if (cost < best_cost * 0.999) {
        best_cost = cost;
        best.mt = mt;
        best.tn = tn;
        best.nblocks = nblocks;
        best.splits = sreal;
        best.cps = cps;
      }
    }
  }
  best.gcap = gcap;
  best.stage_bytes = stage_bytes_for(w_bit, best.mt, best.tn, gcap, zero);
  best.workspace = best.splits > 1 ? decode_counter_bytes() + (size_t)best.splits * rows * N * sizeof(float) : 0;
  return best;
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
  dp.gs = a.group_size;
  dp.kspg = a.group_size / 16;
  dp.nt_total = a.N / 16;
  dp.kch = a.K / (256 / a.w_bit);
  dp.splits = p.splits;
  dp.cps = p.cps;
  dp.gcap = p.gcap;
  dp.stage_bytes = p.stage_bytes;
  dp.s_bf16 = a.s_bf16;
  if (p.splits > 1) {
    dp.counters = static_cast<int *>(workspace);
    dp.partial = reinterpret_cast<float *>(static_cast<char *>(workspace) + decode_counter_bytes());
  }
  // Tensor maps for the activation slice and the scale / zero rows of a stage.
  const int kc = 256 / a.w_bit;
  const int cols = kDecodeWarps * p.tn * 16;
  if (!encode_2d(&dp.tm_x, a.x, 2, (uint64_t)a.K, (uint64_t)a.M, (uint32_t)(x_pitch_for(a.w_bit) / 2),
                 (uint32_t)(p.mt * 8)))
    return cudaErrorInvalidValue;
  if (a.w_bit != 8) {
    const int G = a.K / a.group_size;
    if (!encode_2d(&dp.tm_s, a.scales, 2, (uint64_t)a.N, (uint64_t)G, (uint32_t)cols, (uint32_t)p.gcap))
      return cudaErrorInvalidValue;
    if (a.zeros) {
      const int V = 32 / a.w_bit;
      if (!encode_2d(&dp.tm_z, a.zeros, 4, (uint64_t)a.N, (uint64_t)((G + V - 1) / V), (uint32_t)cols, 2u))
        return cudaErrorInvalidValue;
    }
  }
  (void)kc;
  const bool z = a.zeros != nullptr;
  switch (a.w_bit) {
    case 2: return launch_decode_w<2>(dp, p, a.x_bf16, z, s);
    case 4: return launch_decode_w<4>(dp, p, a.x_bf16, z, s);
    case 8: return launch_decode_w<8>(dp, p, a.x_bf16, false, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace wq
