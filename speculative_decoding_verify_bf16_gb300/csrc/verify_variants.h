// verify_variants.h -- what the host needs to know about one build of the verify
// kernel (consumer-warp count, threads, shared-memory header, kernel entry
// points).  Host code only; shared by spec_verify.cu and the verify_w20*.cu builds.
#pragma once

namespace verify_variants {

struct KernelVariant {
  int threads = 0;         // threads per CTA
  int groups = 0;          // consumer-warp groups (ring slots come in multiples)
  int head_bytes_raw = 0;  // sizeof the shared-memory header
  int consumer_warps = 0;
  void* kernel[4] = {nullptr, nullptr, nullptr, nullptr};        // [dtype * 2 + aligned], lazy sweep
  void* kernel_exact[4] = {nullptr, nullptr, nullptr, nullptr};  // the same with row statistics
};

// The 20-consumer-warp builds: five groups of four (verify_w20.cu) and four
// groups of five (verify_w20p5.cu).
KernelVariant w20_variant();
KernelVariant w20p5_variant();

}  // namespace verify_variants
