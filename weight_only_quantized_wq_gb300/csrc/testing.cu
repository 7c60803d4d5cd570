// testing.cu -- wq_testing_decode_timeout (include/wq_testing.h): the
// few-token kernel with a short barrier-wait limit and one ring stage the
// producer withholds, for the failure-path tests.
#include <cuda_runtime.h>

#include "api.h"
#include "kernels.h"
#include "wq_testing.h"

extern "C" {

wq_status wq_testing_decode_timeout(const void *x, wq_dtype x_dtype, const void *packed_w, const void *scales,
                                    wq_dtype s_dtype, const int32_t *zeros, int M, int N, int K, int w_bit,
                                    int group_size, float *out, void *workspace, size_t workspace_bytes,
                                    long long wait_limit_cycles, int withhold_stage, void *stream) {
  if (wait_limit_cycles < 10000 || wait_limit_cycles > 8000000000ll || withhold_stage < 0) return WQ_ERR_SHAPE;
  if (M > 64) return WQ_ERR_SHAPE;
  wq::Call c;
  wq_status st = wq::prepare_call(x, x_dtype, packed_w, scales, s_dtype, zeros, M, N, K, w_bit, group_size, out,
                                  WQ_F32, &c);
  if (st != WQ_OK || c.noop) return st;
  if (c.route != wq::Route::kDecode) return WQ_ERR_SHAPE;
  if (c.need > 0 && (!workspace || workspace_bytes < c.need)) return WQ_ERR_WORKSPACE;
  c.a.wait_limit = wait_limit_cycles;
  c.a.withhold = withhold_stage;
  return wq::run_call(c, workspace, workspace_bytes, stream);
}

}  // extern "C"
