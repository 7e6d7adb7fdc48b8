// verify_w20p5.cu -- the verify kernel built a third time: 20 consumer warps in
// four groups of five (in its own namespace).  Each chunk is split five ways,
// so four groups cover the consumers and the ring needs only a multiple of
// four slots: when a CTA's whole row slice fits one slot, every group then
// owns two slots and double-buffers, where the five-group build owns one.
// spec_verify.cu launches it for rounds whose slices fit that way: with
// drafter logits always (the 8-lane sampled round: 17.6 -> 17.1 us), greedy
// rounds only with slots above 8 KB (the 8-lane greedy round: 6.36 -> 6.3 us).
#define SPEC_VERIFY_CONSUMER_WARPS 20
#define SPEC_VERIFY_PIECES 5
#define SPEC_VERIFY_LAZY_VEC_TAIL 1
#define specv specv_w20p5
#include "verify_kernel.cuh"
#undef specv

#include "verify_variants.h"

namespace verify_variants {

KernelVariant w20p5_variant() {
  KernelVariant v;
  v.threads = specv_w20p5::kThreads;
  v.groups = specv_w20p5::kGroups;
  v.head_bytes_raw = static_cast<int>(sizeof(specv_w20p5::SmemHead));
  v.consumer_warps = specv_w20p5::kConsumerWarps;
  v.kernel[0] = reinterpret_cast<void*>(&specv_w20p5::verify_accept_kernel<float, false, false>);
  v.kernel[1] = reinterpret_cast<void*>(&specv_w20p5::verify_accept_kernel<float, true, false>);
  v.kernel[2] = reinterpret_cast<void*>(&specv_w20p5::verify_accept_kernel<specv_w20p5::bf16_tag, false, false>);
  v.kernel[3] = reinterpret_cast<void*>(&specv_w20p5::verify_accept_kernel<specv_w20p5::bf16_tag, true, false>);
  v.kernel_exact[0] = reinterpret_cast<void*>(&specv_w20p5::verify_accept_kernel<float, false, true>);
  v.kernel_exact[1] = reinterpret_cast<void*>(&specv_w20p5::verify_accept_kernel<float, true, true>);
  v.kernel_exact[2] = reinterpret_cast<void*>(&specv_w20p5::verify_accept_kernel<specv_w20p5::bf16_tag, false, true>);
  v.kernel_exact[3] = reinterpret_cast<void*>(&specv_w20p5::verify_accept_kernel<specv_w20p5::bf16_tag, true, true>);
  return v;
}

}  // namespace verify_variants
