// verify_w20.cu -- the verify kernel built a second time with 20 consumer warps
// in five groups of four (in its own namespace).  Sampled rows are bound by
// instruction issue, and the extra warps hide more of their latency; greedy
// rows stream better with 16.  spec_verify.cu launches this build for rounds
// with drafter logits when the four-groups-of-five build (verify_w20p5.cu)
// would not double-buffer, and the 16-warp build for rounds without them.
// Its slices stream in several chunks, so its draw segments are long: it
// stages them through shared memory (SPEC_VERIFY_DRAW_STAGE).
#define SPEC_VERIFY_CONSUMER_WARPS 20
#define SPEC_VERIFY_DRAW_STAGE 1
#define specv specv_w20
#include "verify_kernel.cuh"
#undef specv

#include "verify_variants.h"

namespace verify_variants {

KernelVariant w20_variant() {
  KernelVariant v;
  v.threads = specv_w20::kThreads;
  v.groups = specv_w20::kGroups;
  v.head_bytes_raw = static_cast<int>(sizeof(specv_w20::SmemHead));
  v.consumer_warps = specv_w20::kConsumerWarps;
  v.kernel[0] = reinterpret_cast<void*>(&specv_w20::verify_accept_kernel<float, false, false>);
  v.kernel[1] = reinterpret_cast<void*>(&specv_w20::verify_accept_kernel<float, true, false>);
  v.kernel[2] = reinterpret_cast<void*>(&specv_w20::verify_accept_kernel<specv_w20::bf16_tag, false, false>);
  v.kernel[3] = reinterpret_cast<void*>(&specv_w20::verify_accept_kernel<specv_w20::bf16_tag, true, false>);
  v.kernel_exact[0] = reinterpret_cast<void*>(&specv_w20::verify_accept_kernel<float, false, true>);
  v.kernel_exact[1] = reinterpret_cast<void*>(&specv_w20::verify_accept_kernel<float, true, true>);
  v.kernel_exact[2] = reinterpret_cast<void*>(&specv_w20::verify_accept_kernel<specv_w20::bf16_tag, false, true>);
  v.kernel_exact[3] = reinterpret_cast<void*>(&specv_w20::verify_accept_kernel<specv_w20::bf16_tag, true, true>);
  return v;
}

}  // namespace verify_variants
