// decode_inst.cu -- instantiations of the few-token kernel for one code width
// and one group schedule.  The build compiles this file once per (WQ_W,
// WQ_FOLD) pair it lists, so the instantiations compile in parallel.
#include "decode.cuh"

#if !defined(WQ_W) || !defined(WQ_FOLD)
#error "compile with -DWQ_W=<2|4|8> -DWQ_FOLD=<fold>"
#endif

namespace wq {

template <>
cudaError_t launch_decode_wf<WQ_W, WQ_FOLD>(const DecodeParams &dp, const DecodePlan &p, bool bf16, bool zero,
                                            cudaStream_t s) {
#define SHAPES(BF, Z)                       \
  WQ_DECODE_CASE(WQ_W, BF, 1, 2, Z, WQ_FOLD) \
  WQ_DECODE_CASE(WQ_W, BF, 2, 2, Z, WQ_FOLD) \
  WQ_DECODE_CASE(WQ_W, BF, 3, 2, Z, WQ_FOLD) \
  WQ_DECODE_CASE(WQ_W, BF, 4, 1, Z, WQ_FOLD) \
  WQ_DECODE_CASE(WQ_W, BF, 5, 1, Z, WQ_FOLD) \
  WQ_DECODE_CASE(WQ_W, BF, 6, 1, Z, WQ_FOLD) \
  WQ_DECODE_CASE(WQ_W, BF, 7, 1, Z, WQ_FOLD) \
  WQ_DECODE_CASE(WQ_W, BF, 8, 1, Z, WQ_FOLD)
#if WQ_W == 8
  SHAPES(true, false)
  SHAPES(false, false)
#else
  SHAPES(true, true)
  SHAPES(true, false)
  SHAPES(false, true)
  SHAPES(false, false)
#endif
#undef SHAPES
  return cudaErrorInvalidValue;
}

template <>
long decode_capacity_wf<WQ_W, WQ_FOLD>(int mt, int tn, bool zero, int smem, int splits, int sms) {
#define SHAPES(Z)                            \
  WQ_DECODE_CAPACITY(WQ_W, 1, 2, Z, WQ_FOLD) \
  WQ_DECODE_CAPACITY(WQ_W, 2, 2, Z, WQ_FOLD) \
  WQ_DECODE_CAPACITY(WQ_W, 3, 2, Z, WQ_FOLD) \
  WQ_DECODE_CAPACITY(WQ_W, 4, 1, Z, WQ_FOLD) \
  WQ_DECODE_CAPACITY(WQ_W, 5, 1, Z, WQ_FOLD) \
  WQ_DECODE_CAPACITY(WQ_W, 6, 1, Z, WQ_FOLD) \
  WQ_DECODE_CAPACITY(WQ_W, 7, 1, Z, WQ_FOLD) \
  WQ_DECODE_CAPACITY(WQ_W, 8, 1, Z, WQ_FOLD)
#if WQ_W == 8
  SHAPES(false)
#else
  SHAPES(true)
  SHAPES(false)
#endif
#undef SHAPES
  return -1;
}

}  // namespace wq
