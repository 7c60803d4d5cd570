// decode_w8.cu -- instantiations of the few-token kernel for int8 per-channel codes.
#include "decode.cuh"

namespace wq {

template <>
cudaError_t launch_decode_w<8>(const DecodeParams &dp, const DecodePlan &p, bool bf16, bool zero, cudaStream_t s) {
#define CASES(BF)                        \
  WQ_DECODE_CASE(8, BF, 1, 4, false)     \
  WQ_DECODE_CASE(8, BF, 1, 2, false)     \
  WQ_DECODE_CASE(8, BF, 2, 4, false)     \
  WQ_DECODE_CASE(8, BF, 2, 2, false)     \
  WQ_DECODE_CASE(8, BF, 4, 2, false)     \
  WQ_DECODE_CASE(8, BF, 8, 1, false)
  CASES(true)
  CASES(false)
#undef CASES
  return cudaErrorInvalidValue;
}

}  // namespace wq
