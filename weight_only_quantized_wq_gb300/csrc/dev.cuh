// dev.cuh -- device primitives shared by the libwq kernels (sm_103a).
//
// Hand-written PTX wrappers: mbarriers with time-bounded waits, 1-D bulk
// copies (cp.async.bulk, no multicast), warp-level tensor-core MMA, and the
// bit tricks that turn packed integer codes into fp16/bf16 operands.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kernels.h"

namespace wq {

// Bits recorded in the library's device status word.
constexpr uint32_t kDevErrTimeout = 1u;

// A barrier wait gives up after this many SM clock cycles (about 4 s at the
// 2.07 GHz maximum clock; longer at lower clocks).  The SM cycle counter is
// read instead of %globaltimer: a %globaltimer read can stall for a large
// part of a microsecond, which would be paid on every wait that misses.
constexpr long long kWaitLimitCycles = 8000000000ll;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}


// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (bulk copies, tensor core).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the same condition (try_wait may suspend the thread).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `bar` with the given parity to complete.  Gives up
// after `limit` SM cycles (kWaitLimitCycles unless a caller lowers it),
// records kDevErrTimeout in *err, raises the CTA's abort flag and returns
// false.  When `abort` is given, a raised flag (another thread of the CTA gave
// up) also ends the wait at once; waits that must see their copies land
// before the CTA exits pass nullptr.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t *err, volatile int *abort,
                                          long long limit = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0u) {
      if (abort && *abort) return false;
      if (clock64() - t0 > limit) {
        atomicOr(err, kDevErrTimeout);
        if (abort) *abort = 1;
        return false;
      }
    }
  }
}

// mbar_wait for threads with nothing else to do for a long time (an epilogue
// waiting for a whole K range): between tests the thread sleeps, so it takes
// no issue slots from the warps doing the work.  Same limit and abort rules.
__device__ __forceinline__ bool mbar_wait_idle(uint32_t bar, uint32_t parity, uint32_t *err, volatile int *abort,
                                               unsigned sleep_ns = 256) {
  if (mbar_test_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    __nanosleep(sleep_ns);
    if (mbar_test_wait(bar, parity)) return true;
    if (abort && *abort) return false;
    if (clock64() - t0 > kWaitLimitCycles) {
      atomicOr(err, kDevErrTimeout);
      if (abort) *abort = 1;
      return false;
    }
  }
}

// ---------------------------------------------------------------- bulk copy
// L2 policy: weights are read exactly once per call; let them go first.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 1-D bulk copy global -> this CTA's shared memory, completing `bytes` of
// transaction count on `bar`.  dst, src 16-byte aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// 2-D tensor copy global -> this CTA's shared memory through a tensor map
// (TMA), completing the box's bytes on `bar`.  c0 is the innermost coordinate;
// c0 * element size must be a multiple of 16 bytes.  Parts of the box outside
// the tensor are filled with zeros.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(tmap), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}


// ---------------------------------------------------------------- clusters
// Barrier over every thread of every CTA of the cluster (release / acquire).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Cluster barrier that orders no memory operation: for "every CTA is done
// reading the others' shared memory", where each read has already returned
// its value (so nothing waits for this thread's global stores to drain).
__device__ __forceinline__ void cluster_sync_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory location in the cluster's CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a)
               : "memory");
  return v;
}
__device__ __forceinline__ void sts64(uint32_t a, uint32_t x, uint32_t y) {
  asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(a), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ void sts_f32(uint32_t a, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}

// ---------------------------------------------------------------- loads
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint16_t lds16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}

// ---------------------------------------------------------------- MMA
// D += A * B, m16n8k16, fp32 accumulate.  A row-major 16x16 (4 regs), B
// column-major 16x8 (2 regs), C/D 16x8 fp32 (4 regs).
template <bool BF16>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  if constexpr (BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// ---------------------------------------------------------------- dequant
// (a & b) | c as one LOP3.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Magic-exponent conversion.  A float whose exponent makes the unit in the
// last place exactly 1 turns an integer u written into its low mantissa bits
// into the value MAGIC + u, exactly: 1024 + u for fp16 (10 fraction bits),
// 128 + u for bf16 (7 fraction bits).  Two values per 32-bit register.
template <bool BF16>
struct Magic {
  static constexpr uint32_t kPair = BF16 ? 0x43004300u : 0x64006400u;  // (128, 128) or (1024, 1024)
  static constexpr float kValue = BF16 ? 128.0f : 1024.0f;
  static constexpr uint32_t kOnePair = BF16 ? 0x3F803F80u : 0x3C003C00u;  // (1.0, 1.0)
};

// Pair i of a packed word: fields i and i + 32/(2*W_BIT) land in the low and
// high 16-bit halves as (MAGIC + code).  W_BIT 2 or 4.
template <int W_BIT, bool BF16>
__device__ __forceinline__ uint32_t code_pair(uint32_t w, int i) {
  constexpr uint32_t mask = W_BIT == 4 ? 0x000F000Fu : 0x00030003u;
  return and_or(w >> (W_BIT * i), mask, Magic<BF16>::kPair);
}

// Both 16-bit halves a - b (fp16 or bf16 pairs, round to nearest even).
template <bool BF16>
__device__ __forceinline__ uint32_t sub_pair(uint32_t a, uint32_t b) {
  uint32_t d;
  if constexpr (BF16)
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Both fp16 halves a * b + c, one rounding.
__device__ __forceinline__ uint32_t fma_h2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// fp16 int4 without the shift for odd fields: masking field 2i + 1 in place
// gives the fp16 value 1024 + 16 q (16 q stays inside the 10 fraction bits).
// (1024 + 16 q) * (1/16) - (64 + z) = q - z exactly, in one fma with
// c = 960 - (1024 + z), built once per group from the (1024 + z) pair.
constexpr uint32_t kF16Sixteenth = 0x2C002C00u;  // (1/16, 1/16)
constexpr uint32_t kF16NineSixty = 0x63806380u;  // (960, 960)

// Both 16-bit halves a * b + c (fp16 or bf16 pairs), one rounding.
template <bool BF16>
__device__ __forceinline__ uint32_t fma_pair(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  if constexpr (BF16)
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  else
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// 2-bit fields taken in place.  Masking the field at bits p..p+1 of each
// 16-bit half (p = 0, 2, 4: inside the 7 fraction bits of a bf16, and of an
// fp16) gives MAGIC + 2^p q exactly; (MAGIC + 2^p q) * 2^-p - (MAGIC 2^-p + z)
// = q - z exactly, in one fma whose addend is built once per group from the
// (MAGIC + z) pair as (1 - 2^-p) MAGIC - (MAGIC + z).  Three of a word's
// eight pairs need no shift and three more share one shift by 8.
template <bool BF16>
struct Int2InPlace {
  static constexpr uint32_t kQuarter = BF16 ? 0x3E803E80u : 0x34003400u;    // (1/4, 1/4)
  static constexpr uint32_t kSixteenth = BF16 ? 0x3D803D80u : 0x2C002C00u;  // (1/16, 1/16)
  static constexpr uint32_t kMagic3of4 = BF16 ? 0x42C042C0u : 0x62006200u;  // 3/4 MAGIC: 96 or 768
  static constexpr uint32_t kMagic15of16 = BF16 ? 0x42F042F0u : 0x63806380u;  // 15/16 MAGIC: 120 or 960
};

// Pair i (0..7) of a word of 2-bit codes (fields i and i + 8 in the low and
// high halves, as code_pair<2> takes them) as the exact q - zero pair.
// zz = (MAGIC + z), n2 = -(MAGIC/4 + z), n4 = -(MAGIC/16 + z).
template <bool BF16>
__device__ __forceinline__ uint32_t int2_pair(uint32_t w, int i, uint32_t zz, uint32_t n2, uint32_t n4) {
  using P = Int2InPlace<BF16>;
  const int s = i == 3 ? 6 : i == 7 ? 14 : i >= 4 ? 8 : 0;  // shift that brings the field into bits 0..5
  const int pos = (i == 1 || i == 5) ? 2 : (i == 2 || i == 6) ? 4 : 0;
  const uint32_t v = and_or(s ? w >> s : w, 0x00030003u << pos, Magic<BF16>::kPair);
  if (pos == 0) return sub_pair<BF16>(v, zz);
  return fma_pair<BF16>(v, pos == 2 ? P::kQuarter : P::kSixteenth, pos == 2 ? n2 : n4);
}

// Signed int8 bytes (lo, hi) of a word -> exact fp16/bf16 pair.
template <bool BF16>
__device__ __forceinline__ uint32_t int8_pair(uint32_t w, int hi_half) {
  if constexpr (BF16) {
    // q = q7 - 128 s (q7 = low seven bits, s = sign bit).  With the bytes in
    // the low byte of each 16-bit half: (0x4300 | q7) is the bf16 value 128 + q7
    // and (0x4300 | s << 7) is 128 or 256; their difference is q, exactly.
    const uint32_t t = __byte_perm(w, 0u, hi_half ? 0x4342u : 0x4140u);
    const uint32_t a = and_or(t, 0x007F007Fu, Magic<true>::kPair);
    const uint32_t b = and_or(t, 0x00800080u, Magic<true>::kPair);
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
  } else {
    // 0x64uu is the fp16 value 1024 + u (u = q + 128); subtract 1152 from both halves.
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t h = __byte_perm(u, 0x64646464u, hi_half ? 0x7362u : 0x5140u);
    uint32_t r;
    asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64806480u));
    return r;
  }
}

// ---------------------------------------------------------------- output
// out[idx .. idx + 3] = v (idx a multiple of 4; out 16-byte aligned).
__device__ __forceinline__ void store_out4(void *out, size_t idx, float4 v, int ot) {
  if (ot == kOutF32) {
    *reinterpret_cast<float4 *>(static_cast<float *>(out) + idx) = v;
  } else if (ot == kOutS32) {
    *reinterpret_cast<int4 *>(static_cast<int *>(out) + idx) =
        make_int4(__float2int_rn(v.x), __float2int_rn(v.y), __float2int_rn(v.z), __float2int_rn(v.w));
  } else if (ot == kOutF16) {
    __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    *reinterpret_cast<uint2 *>(static_cast<__half *>(out) + idx) =
        make_uint2(*reinterpret_cast<uint32_t *>(&a), *reinterpret_cast<uint32_t *>(&b));
  } else {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(out) + idx) =
        make_uint2(*reinterpret_cast<uint32_t *>(&a), *reinterpret_cast<uint32_t *>(&b));
  }
}
// out[idx] = v.
__device__ __forceinline__ void store_out1(void *out, size_t idx, float v, int ot) {
  if (ot == kOutF32)
    static_cast<float *>(out)[idx] = v;
  else if (ot == kOutS32)
    static_cast<int *>(out)[idx] = __float2int_rn(v);
  else if (ot == kOutF16)
    static_cast<__half *>(out)[idx] = __float2half_rn(v);
  else
    static_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ float half_bits_to_float(uint16_t h, bool bf16) {
  if (bf16) return __uint_as_float(static_cast<uint32_t>(h) << 16);
  float f;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
  return f;
}

}  // namespace wq
