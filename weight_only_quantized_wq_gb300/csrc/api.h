// api.h -- host-side validation and dispatch shared by the C entry points.
#pragma once

#include <cstddef>
#include <cstdint>

#include "kernels.h"
#include "wq.h"

namespace wq {

// Which kernel a call runs on.
enum class Route {
  kDecode,   // few tokens, or codes / groups the tensor-core paths do not take (64-token slices)
  kMidm,     // tensor cores, exact weights, group scale in fp32
  kPrefill,  // tensor cores, weight rounded once to the x dtype (many tokens)
  kPrefillSplit,  // the same kernel, each weight as two terms (rounded, residue): bf16 below K = 4096
};

// Route of a validated call (x and scale dtypes only matter for kPrefill).
Route route_of(const MatmulArgs &a);

// One validated matmul call: the arguments the kernels take, the route, and
// the workspace bytes it needs.
struct Call {
  MatmulArgs a;        // M is the whole call's token count
  int sms = 0;
  bool noop = false;   // M == 0 or N == 0: nothing to do
  Route route = Route::kDecode;
  size_t need = 0;     // workspace bytes (0: none)
};

// Every host check of wq_matmul, in order, before anything touches a device
// (the device query comes last).  Fills *c on WQ_OK.
wq_status prepare_call(const void *x, wq_dtype x_dtype, const void *packed_w, const void *scales, wq_dtype s_dtype,
                       const int32_t *zeros, int M, int N, int K, int w_bit, int group_size, void *out,
                       wq_dtype out_dtype, Call *c);

// Enqueue the kernels of a prepared call on `stream`; workspace holds at
// least c.need bytes (zero-filled counters) when c.need > 0, and
// workspace_bytes in all (more lets the many-token kernel run persistent).
wq_status run_call(const Call &c, void *workspace, size_t workspace_bytes, void *stream);

}  // namespace wq
