// decode_w4.cu -- instantiations of the few-token kernel for 4-bit grouped codes.
#include "decode.cuh"

namespace wq {

template <>
cudaError_t launch_decode_w<4>(const DecodeParams &dp, const DecodePlan &p, bool bf16, bool zero, cudaStream_t s) {
#define CASES(BF, Z)                    \
  WQ_DECODE_CASE(4, BF, 1, 4, Z)        \
  WQ_DECODE_CASE(4, BF, 1, 2, Z)        \
  WQ_DECODE_CASE(4, BF, 2, 4, Z)        \
  WQ_DECODE_CASE(4, BF, 2, 2, Z)        \
  WQ_DECODE_CASE(4, BF, 4, 2, Z)        \
  WQ_DECODE_CASE(4, BF, 8, 1, Z)
  CASES(true, true)
  CASES(true, false)
  CASES(false, true)
  CASES(false, false)
#undef CASES
  return cudaErrorInvalidValue;
}

}  // namespace wq
