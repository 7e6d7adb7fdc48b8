// spec_verify.cu -- host side of the C ABI declared in include/spec_verify.h:
// argument checks, launch-shape selection and kernel launches.  The library
// allocates no device memory; it caches per-device kernel attributes only.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "commit_kernel.cuh"
#include "spec_verify.h"
#include "verify_kernel.cuh"
#include "verify_variants.h"

namespace {

using specv::bf16_tag;
using verify_variants::KernelVariant;
using verify_variants::w20_variant;
using verify_variants::w20p5_variant;

constexpr int kMaxDevices = 64;

struct DeviceCache {
  bool ready = false;
  int sms = 0;
  int smem_optin = 0;
  bool verify_attr[12] = {};  // per kernel build and instantiation
  bool commit_attr = false;
};

std::mutex g_mutex;
DeviceCache g_cache[kMaxDevices];

int env_int(const char* name, int fallback) {
  const char* v = std::getenv(name);
  if (v == nullptr || *v == '\0') return fallback;
  return std::atoi(v);
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

int device_cache(DeviceCache** out, int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPEC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceCache& c = g_cache[dev];
  if (!c.ready) {
    if (cudaDeviceGetAttribute(&c.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&c.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
      return SPEC_ERR_CUDA;
    c.ready = true;
  }
  *out = &c;
  if (dev_out) *dev_out = dev;
  return SPEC_OK;
}

struct VerifyShape {
  int cluster;
  int slice;
  int slot_bytes;
  int nslots;
  int head_bytes;
  int smem;
  int active;  // clusters of this shape resident at once (0 if unknown)
};

// One cluster of `cluster` CTAs per lane; each CTA reduces `slice` elements of
// every row of its lane.  The cluster is the larger of (a) the smallest power
// of two that gives about 1.5 CTAs per SM and (b) the smallest that keeps a
// CTA's share of an average lane (rows / lanes rows, counted 1.5 times for
// drafter rows of sampled lanes) at or below 1 MB; never fewer than 2048
// elements per CTA.  The caller then shrinks it until clusters fit (see
// spec_verify_accept).  The ring holds whole slices when they fit a 40 KB slot.
VerifyShape choose_shape(const KernelVariant& kv, int lanes, int rows, int V, int esize, bool aligned, int sms,
                         int smem_optin, int force_cluster) {
  VerifyShape s{};
  const int vec = 16 / esize;
  int C = force_cluster > 0 ? force_cluster : env_int("SPEC_VERIFY_CLUSTER", 0);
  if (C <= 0) {
    int c_fill = 1;
    while (c_fill < specv::kMaxCluster && static_cast<int64_t>(lanes) * c_fill * 2 < 3LL * sms) c_fill *= 2;
    const double lane_bytes = 1.5 * rows / lanes * static_cast<double>(V) * esize;
    int c_size = 1;
    while (c_size < specv::kMaxCluster && lane_bytes / c_size > 1024.0 * 1024) c_size *= 2;
    C = c_fill > c_size ? c_fill : c_size;
    while (C > 1 && (V + C - 1) / C < 2048) C /= 2;
  }
  if (C > specv::kMaxCluster) C = specv::kMaxCluster;
  s.cluster = C;
  s.slice = static_cast<int>(round_up((V + C - 1) / C, vec));
  s.head_bytes = static_cast<int>(round_up(kv.head_bytes_raw, 128));
  if (!aligned) {
    s.slot_bytes = 16;
    s.nslots = 0;
    s.smem = s.head_bytes;
    return s;
  }
  const int64_t slice_bytes = static_cast<int64_t>(s.slice) * esize;
  // Slots of up to 40 KB: a 152 KB slice then streams in four 38 KB pieces,
  // one per consumer-warp group (measured faster than five of 30 KB).
  const int64_t slot_max = static_cast<int64_t>(env_int("SPEC_VERIFY_SLOT_KB", 40)) * 1024;
  const int64_t chunks = (slice_bytes + slot_max - 1) / slot_max;
  s.slot_bytes = static_cast<int>(round_up((slice_bytes + chunks - 1) / chunks, 16));
  // With 8 consumer warps 88 KB keeps two CTAs per SM possible; with more the
  // CTA fills an SM and the ring takes all the shared memory left.
  const int64_t ring_kb = env_int("SPEC_VERIFY_RING_KB", 0);
  const int64_t ring = ring_kb > 0 ? ring_kb * 1024
                                   : (kv.consumer_warps <= 8 ? 88 * 1024 : smem_optin - s.head_bytes);
  // A multiple of the kernel's consumer-warp groups (each group owns its slots).
  int nslots = static_cast<int>(ring / s.slot_bytes);
  nslots -= nslots % kv.groups;
  if (nslots < kv.groups) nslots = kv.groups;
  if (nslots > specv::kMaxSlots) nslots = specv::kMaxSlots - specv::kMaxSlots % kv.groups;
  s.nslots = nslots;
  s.smem = s.head_bytes + nslots * s.slot_bytes;
  return s;
}

// The 16-consumer-warp build of the kernel (this translation unit).
KernelVariant w16_variant() {
  KernelVariant v;
  v.threads = specv::kThreads;
  v.groups = specv::kGroups;
  v.head_bytes_raw = static_cast<int>(sizeof(specv::SmemHead));
  v.consumer_warps = specv::kConsumerWarps;
  v.kernel[0] = reinterpret_cast<void*>(&specv::verify_accept_kernel<float, false, false>);
  v.kernel[1] = reinterpret_cast<void*>(&specv::verify_accept_kernel<float, true, false>);
  v.kernel[2] = reinterpret_cast<void*>(&specv::verify_accept_kernel<bf16_tag, false, false>);
  v.kernel[3] = reinterpret_cast<void*>(&specv::verify_accept_kernel<bf16_tag, true, false>);
  v.kernel_exact[0] = reinterpret_cast<void*>(&specv::verify_accept_kernel<float, false, true>);
  v.kernel_exact[1] = reinterpret_cast<void*>(&specv::verify_accept_kernel<float, true, true>);
  v.kernel_exact[2] = reinterpret_cast<void*>(&specv::verify_accept_kernel<bf16_tag, false, true>);
  v.kernel_exact[3] = reinterpret_cast<void*>(&specv::verify_accept_kernel<bf16_tag, true, true>);
  return v;
}

// Kernel builds: 0 = 16 consumer warps (4 groups of 4), 1 = 20 warps (5 groups
// of 4), 2 = 20 warps (4 groups of 5).
constexpr int kBuildW16 = 0, kBuildW20 = 1, kBuildW20P5 = 2, kBuilds = 3;

// Rounds with drafter logits may hold sampled lanes, whose sweep is bound by
// instruction issue: 20 consumer warps hide more of its latency.  Greedy-only
// rounds stream better with 16.  SPEC_VERIFY_BUILD=0|1|2 (or the older
// SPEC_VERIFY_WARPS=16|20) forces a build; -1 means "choose by shape".
int forced_build() {
  const int b = env_int("SPEC_VERIFY_BUILD", -1);
  if (b >= 0 && b < kBuilds) return b;
  const int w = env_int("SPEC_VERIFY_WARPS", 0);
  if (w == 16) return kBuildW16;
  if (w == 20) return kBuildW20;
  return -1;
}

const KernelVariant& variant(int which) {
  static const KernelVariant kVariants[kBuilds] = {w16_variant(), w20_variant(), w20p5_variant()};
  return kVariants[which];
}

int kernel_index(int dtype, bool aligned) { return dtype * 2 + (aligned ? 1 : 0); }

// Rounds without drafter logits whose rows are at most this many bytes run on
// the small-round kernel (one CTA per lane, plain loads): the 1-lane round of
// four 4 KB rows takes 2.45 us on the cluster kernel, which sets up a cluster,
// a ring and its barriers for 16 KB.  A forced build or cluster size, or
// SPEC_VERIFY_SMALL=0, keeps the cluster kernel.
constexpr int kSmallRowBytes = 16 * 1024;

bool use_small(bool with_draft, int V, int esize) {
  if (with_draft || static_cast<int64_t>(V) * esize > kSmallRowBytes) return false;
  if (env_int("SPEC_VERIFY_SMALL", 1) == 0) return false;
  return forced_build() < 0 && env_int("SPEC_VERIFY_CLUSTER", 0) <= 0;
}

void* small_kernel(int dtype, bool aligned) {
  static void* const k[4] = {reinterpret_cast<void*>(&specv::verify_small_kernel<float, false>),
                             reinterpret_cast<void*>(&specv::verify_small_kernel<float, true>),
                             reinterpret_cast<void*>(&specv::verify_small_kernel<bf16_tag, false>),
                             reinterpret_cast<void*>(&specv::verify_small_kernel<bf16_tag, true>)};
  return k[kernel_index(dtype, aligned)];
}

bool is_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Clusters that can be resident at once, per device / kernel / cluster size /
// shared memory (cached; cudaOccupancyMaxActiveClusters).
struct ClusterFit {
  int dev;
  void* kernel;
  int smem;
  int cluster;
  int active;
};
constexpr int kFitCache = 128;
ClusterFit g_fit[kFitCache];
int g_fit_n = 0;

int max_active_clusters(int dev, void* kernel, int threads, int cluster, int smem) {
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    for (int i = 0; i < g_fit_n; ++i)
      if (g_fit[i].dev == dev && g_fit[i].kernel == kernel && g_fit[i].smem == smem &&
          g_fit[i].cluster == cluster)
        return g_fit[i].active;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cluster), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = static_cast<unsigned>(cluster);
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_fit_n < kFitCache) g_fit[g_fit_n++] = ClusterFit{dev, kernel, smem, cluster, n};
  return n;
}

// The next smaller cluster size tried when one does not fit.
int smaller_cluster(int c) {
  static const int kSizes[] = {16, 12, 8, 6, 4, 2, 1};
  for (int s : kSizes)
    if (s < c) return s;
  return 1;
}

__global__ void round_uniforms_kernel(uint64_t seed, uint32_t lane_base, int32_t lanes, int32_t positions,
                                      float* out) {
  const int64_t total = static_cast<int64_t>(lanes) * positions;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int b = static_cast<int>(i / positions), j = static_cast<int>(i % positions);
    const float2 u = specv::round_uniforms(seed, lane_base + static_cast<uint32_t>(b), j);
    out[2 * i] = u.x;
    out[2 * i + 1] = u.y;
  }
}

// The shape spec_verify_accept launches: choose_shape, then, since a cluster
// must fit into one GPU processing cluster, smaller clusters until one fits.
// When every lane could run at once (few lanes) the cluster also shrinks until
// all of them fit together, so that no lane waits for a second wave.
int resolve_shape(DeviceCache* dc, int dev, int which, int lanes, int rows, int V, int dtype, bool aligned,
                  VerifyShape* out, void** kernel_out) {
  const KernelVariant& kv = variant(which);
  const int esize = (dtype == SPEC_BF16) ? 2 : 4;
  VerifyShape s = choose_shape(kv, lanes, rows, V, esize, aligned, dc->sms, dc->smem_optin, 0);
  if (s.smem > dc->smem_optin) return SPEC_ERR_UNSUPPORTED;
  void* kernel = kv.kernel[kernel_index(dtype, aligned)];
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    bool& done = dc->verify_attr[which * 4 + kernel_index(dtype, aligned)];
    if (!done) {
      // Both instantiations (lazy sweep and row statistics) share the shape.
      for (void* k : {kernel, kv.kernel_exact[kernel_index(dtype, aligned)]}) {
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, dc->smem_optin) != cudaSuccess ||
            cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
          return SPEC_ERR_CUDA;
      }
      done = true;
    }
  }
  const bool forced = env_int("SPEC_VERIFY_CLUSTER", 0) > 0;
  for (;;) {
    const int active = max_active_clusters(dev, kernel, kv.threads, s.cluster, s.smem);
    s.active = active;
    const bool few = static_cast<int64_t>(lanes) * s.cluster <= 2LL * dc->sms;
    if (s.cluster == 1 || (active > 0 && (forced || !few || active >= lanes))) break;
    s = choose_shape(kv, lanes, rows, V, esize, aligned, dc->sms, dc->smem_optin, smaller_cluster(s.cluster));
  }
  *out = s;
  if (kernel_out) *kernel_out = kernel;
  return SPEC_OK;
}

// The build and shape a launch uses.  The four-groups-of-five build runs when
// one slot holds a CTA's whole row slice and the ring holds two slots per group
// (each group double-buffers): for rounds with drafter logits always then (the
// 8-lane sampled round 17.6 -> 17.1 us), for greedy rounds only with slots
// above the parallel-issue size (the 8-lane greedy round 6.33 -> 6.23 us; the
// 1-lane round of 4 KB rows is faster with 16 warps).  Otherwise rounds with
// drafter logits take the five-groups-of-four build and greedy rounds the
// 16-warp one.
int resolve_launch(DeviceCache* dc, int dev, bool with_draft, int lanes, int rows, int V, int dtype, bool aligned,
                   VerifyShape* out, void** kernel_out, int* which_out) {
  const int forced = forced_build();
  int which = forced >= 0 ? forced : kBuildW20P5;
  int rc = resolve_shape(dc, dev, which, lanes, rows, V, dtype, aligned, out, kernel_out);
  if (forced < 0) {
    const int esize = (dtype == SPEC_BF16) ? 2 : 4;
    const bool fits = rc == SPEC_OK && aligned &&
                      static_cast<int64_t>(out->slice) * esize <= out->slot_bytes &&
                      out->nslots >= 2 * variant(kBuildW20P5).groups &&
                      (with_draft || out->slot_bytes > specv::kParallelIssueSlotBytes);
    if (!fits) {
      which = with_draft ? kBuildW20 : kBuildW16;
      rc = resolve_shape(dc, dev, which, lanes, rows, V, dtype, aligned, out, kernel_out);
    }
  }
  *which_out = which;
  return rc;
}

// The small-round launch: one CTA per lane, programmatic dependent launch as
// for the cluster kernel.
int launch_small(const spec_verify_args* a, int esize, bool aligned, void* stream) {
  specv::VerifyParams p{};
  p.target = static_cast<const uint8_t*>(a->target_logits);
  p.draft = nullptr;
  p.ld_bytes = a->ld * esize;
  p.V = a->V;
  p.lanes = a->lanes;
  p.rows = a->rows;
  p.draft_tokens = a->draft_tokens;
  p.draft_lens = a->draft_lens;
  p.row_offsets = a->row_offsets;
  p.temps = a->temperatures;
  p.seed = a->seed;
  p.committed = a->committed;
  p.out_tokens = a->out_tokens;
  p.lane_status = a->lane_status;
  p.row_stats = a->row_stats;
  p.lane_base = a->lane_base;
  p.flags = a->flags;
  p.cluster = 1;
  p.slice = a->V;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a->lanes), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(specv::kSmallThreads), 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  void* kargs[] = {&p};
  if (cudaLaunchKernelExC(&cfg, small_kernel(a->dtype, aligned), kargs) != cudaSuccess) {
    cudaGetLastError();
    return SPEC_ERR_CUDA;
  }
  return SPEC_OK;
}

}  // namespace

extern "C" {

int spec_round_uniforms(uint64_t seed, uint32_t lane_base, int32_t lanes, int32_t positions, float* out,
                        void* stream) {
  if (lanes < 0 || positions < 0) return SPEC_ERR_INVALID_ARG;
  const int64_t total = static_cast<int64_t>(lanes) * positions;
  if (total == 0) return SPEC_OK;
  if (out == nullptr) return SPEC_ERR_INVALID_ARG;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  round_uniforms_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      seed, lane_base, lanes, positions, out);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}


int32_t spec_row_budget(int32_t draft_tokens, int32_t row_budget, int32_t lanes) {
  if (lanes <= 0 || draft_tokens < 0 || row_budget < 0) return -SPEC_ERR_INVALID_ARG;
  const int32_t rows = (row_budget == 0) ? 8 : row_budget;
  int32_t per_lane = rows / lanes - 1;
  if (per_lane > draft_tokens) per_lane = draft_tokens;
  return per_lane < 0 ? 0 : per_lane;
}

const char* spec_status_string(int status) {
  switch (status) {
    case SPEC_OK: return "SPEC_OK";
    case SPEC_ERR_INVALID_ARG: return "SPEC_ERR_INVALID_ARG";
    case SPEC_ERR_UNSUPPORTED: return "SPEC_ERR_UNSUPPORTED";
    case SPEC_ERR_CUDA: return "SPEC_ERR_CUDA";
    case SPEC_ERR_NONFINITE: return "SPEC_ERR_NONFINITE";
    case SPEC_ERR_TOKEN_RANGE: return "SPEC_ERR_TOKEN_RANGE";
    case SPEC_ERR_LAYOUT: return "SPEC_ERR_LAYOUT";
    case SPEC_ERR_TIMEOUT: return "SPEC_ERR_TIMEOUT";
    default: return "SPEC_ERR_UNKNOWN";
  }
}

int spec_verify_launch_shape(int32_t lanes, int32_t rows, int32_t V, spec_dtype dtype, int32_t with_draft,
                             int32_t* cluster_ctas, int32_t* threads, int32_t* slice, int32_t* smem_bytes) {
  if (lanes <= 0 || rows < lanes || V <= 0 || (dtype != SPEC_F32 && dtype != SPEC_BF16))
    return SPEC_ERR_INVALID_ARG;
  DeviceCache* dc = nullptr;
  int dev = 0;
  if (device_cache(&dc, &dev) != SPEC_OK) return SPEC_ERR_CUDA;
  if (use_small(with_draft != 0, V, dtype == SPEC_BF16 ? 2 : 4)) {
    if (cluster_ctas) *cluster_ctas = 1;
    if (threads) *threads = specv::kSmallThreads;
    if (slice) *slice = V;
    if (smem_bytes) *smem_bytes = 0;
    return SPEC_OK;
  }
  VerifyShape s{};
  int which = 0;
  const int rc = resolve_launch(dc, dev, with_draft != 0, lanes, rows, V, dtype, true, &s, nullptr, &which);
  if (rc != SPEC_OK) return rc;
  if (cluster_ctas) *cluster_ctas = s.cluster;
  if (threads) *threads = variant(which).threads;
  if (slice) *slice = s.slice;
  if (smem_bytes) *smem_bytes = s.smem;
  return SPEC_OK;
}

int spec_verify_accept(const spec_verify_args* a, void* stream) {
  if (a == nullptr) return SPEC_ERR_INVALID_ARG;
  if (a->target_logits == nullptr || a->draft_tokens == nullptr || a->draft_lens == nullptr ||
      a->row_offsets == nullptr || a->temperatures == nullptr || a->committed == nullptr ||
      a->out_tokens == nullptr)
    return SPEC_ERR_INVALID_ARG;
  if (a->V <= 0 || a->lanes <= 0 || a->rows < a->lanes || a->ld < a->V) return SPEC_ERR_INVALID_ARG;
  if (a->dtype != SPEC_F32 && a->dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (static_cast<int64_t>(a->lanes) * specv::kMaxCluster > INT32_MAX) return SPEC_ERR_INVALID_ARG;

  DeviceCache* dc = nullptr;
  int dev = 0;
  if (device_cache(&dc, &dev) != SPEC_OK) return SPEC_ERR_CUDA;

  const int esize = (a->dtype == SPEC_BF16) ? 2 : 4;
  const bool aligned = is_aligned16(a->target_logits) &&
                       (a->draft_logits == nullptr || is_aligned16(a->draft_logits)) &&
                       ((a->ld * esize) % 16 == 0);
  if (use_small(a->draft_logits != nullptr, a->V, esize)) return launch_small(a, esize, aligned, stream);
  VerifyShape s{};
  void* kernel = nullptr;
  int which = 0;
  const int rc = resolve_launch(dc, dev, a->draft_logits != nullptr, a->lanes, a->rows, a->V, a->dtype, aligned, &s,
                                &kernel, &which);
  if (rc != SPEC_OK) return rc;
  // Row statistics need the exact sweep's instantiation (same shape).
  if (a->row_stats) kernel = variant(which).kernel_exact[kernel_index(a->dtype, aligned)];

  specv::VerifyParams p{};
  p.target = static_cast<const uint8_t*>(a->target_logits);
  p.draft = static_cast<const uint8_t*>(a->draft_logits);
  p.ld_bytes = a->ld * esize;
  p.V = a->V;
  p.lanes = a->lanes;
  p.rows = a->rows;
  p.draft_tokens = a->draft_tokens;
  p.draft_lens = a->draft_lens;
  p.row_offsets = a->row_offsets;
  p.temps = a->temperatures;
  p.seed = a->seed;
  p.committed = a->committed;
  p.out_tokens = a->out_tokens;
  p.lane_status = a->lane_status;
  p.row_stats = a->row_stats;
  p.lane_base = a->lane_base;
  p.flags = a->flags;
  p.cluster = s.cluster;
  p.slice = s.slice;
  p.slot_bytes = s.slot_bytes;
  p.nslots = s.nslots;
  p.head_bytes = s.head_bytes;
  // More lanes than resident clusters: take them longest first.
  const int order_env = env_int("SPEC_VERIFY_ORDER", -1);
  p.order_by_cost = order_env >= 0 ? (order_env != 0) : (s.active > 0 && a->lanes > s.active);

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(s.cluster * a->lanes), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(variant(which).threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(s.smem);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = static_cast<unsigned>(s.cluster);
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  void* kargs[] = {&p};
  if (cudaLaunchKernelExC(&cfg, kernel, kargs) != cudaSuccess) {
    cudaGetLastError();
    return SPEC_ERR_CUDA;
  }
  return SPEC_OK;
}

int spec_commit_state(const void* staged, void* live, const int32_t* committed, int32_t lanes,
                      int32_t cols, uint64_t bytes_per_col, uint64_t staged_lane_stride,
                      uint64_t staged_col_stride, uint64_t live_lane_stride, int32_t* lane_status,
                      void* stream) {
  if (lanes < 0 || cols <= 0) return SPEC_ERR_INVALID_ARG;
  if (lanes == 0 || bytes_per_col == 0) return SPEC_OK;
  if (staged == nullptr || live == nullptr || committed == nullptr) return SPEC_ERR_INVALID_ARG;
  if (bytes_per_col > staged_col_stride && cols > 1) return SPEC_ERR_INVALID_ARG;
  if (lanes > 1 && (bytes_per_col > live_lane_stride ||
                    static_cast<uint64_t>(cols - 1) * staged_col_stride + bytes_per_col > staged_lane_stride))
    return SPEC_ERR_INVALID_ARG;

  DeviceCache* dc = nullptr;
  if (device_cache(&dc, nullptr) != SPEC_OK) return SPEC_ERR_CUDA;

  specv::CommitParams p{};
  p.staged = static_cast<const uint8_t*>(staged);
  p.live = static_cast<uint8_t*>(live);
  p.committed = committed;
  p.lane_status = lane_status;
  p.lanes = lanes;
  p.cols = cols;
  p.bytes_per_col = bytes_per_col;
  p.staged_lane_stride = staged_lane_stride;
  p.staged_col_stride = staged_col_stride;
  p.live_lane_stride = live_lane_stride;
  p.test_withhold = env_int("SPEC_COMMIT_TEST_WITHHOLD_COPY", 0) != 0;

  const bool aligned = is_aligned16(staged) && is_aligned16(live) && bytes_per_col % 16 == 0 &&
                       staged_lane_stride % 16 == 0 && staged_col_stride % 16 == 0 &&
                       live_lane_stride % 16 == 0;

  cudaLaunchConfig_t cfg = {};
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  void* kargs[] = {&p};
  void* kernel = nullptr;

  if (aligned) {
    // Three CTAs per SM, each one thread driving two 32 KB buffers: more
    // independent issuers beat deeper queues (one CTA with six buffers ran
    // at 93 % of the measured copy bandwidth, this shape at 98 %).
    int chunk = env_int("SPEC_COMMIT_CHUNK_KB", 32) * 1024;
    int nbuf = env_int("SPEC_COMMIT_NBUF", 2);
    int per_sm = env_int("SPEC_COMMIT_CTAS_PER_SM", 3);
    if (nbuf < 2) nbuf = 2;
    if (nbuf > specv::kCommitMaxBufs) nbuf = specv::kCommitMaxBufs;
    if (per_sm < 1) per_sm = 1;
    if (static_cast<uint64_t>(chunk) > bytes_per_col) chunk = static_cast<int>(bytes_per_col);
    while (specv::kCommitHead + static_cast<int64_t>(nbuf) * chunk > dc->smem_optin && nbuf > 2) --nbuf;
    while (specv::kCommitHead + static_cast<int64_t>(nbuf) * chunk > dc->smem_optin) chunk /= 2;
    chunk = static_cast<int>(chunk / 16 * 16);
    if (chunk < 16) chunk = 16;
    p.chunk_bytes = static_cast<uint32_t>(chunk);
    p.chunks_per_lane = (bytes_per_col + chunk - 1) / chunk;
    p.total_items = p.chunks_per_lane * static_cast<uint64_t>(lanes);
    p.nbuf = nbuf;
    uint64_t grid = static_cast<uint64_t>(dc->sms) * per_sm;
    if (grid > p.total_items) grid = p.total_items;
    kernel = reinterpret_cast<void*>(&specv::commit_bulk_kernel);
    const int smem = specv::kCommitHead + nbuf * chunk;
    {
      std::lock_guard<std::mutex> lock(g_mutex);
      if (!dc->commit_attr) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dc->smem_optin) !=
            cudaSuccess)
          return SPEC_ERR_CUDA;
        dc->commit_attr = true;
      }
    }
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(specv::kCommitThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  } else {
    kernel = reinterpret_cast<void*>(&specv::commit_bytes_kernel);
    const uint64_t total = static_cast<uint64_t>(lanes) * bytes_per_col;
    uint64_t grid = (total + 255) / 256;
    const uint64_t cap = static_cast<uint64_t>(dc->sms) * 8;
    if (grid > cap) grid = cap;
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = 0;
  }
  if (cudaLaunchKernelExC(&cfg, kernel, kargs) != cudaSuccess) {
    cudaGetLastError();
    return SPEC_ERR_CUDA;
  }
  return SPEC_OK;
}

}  // extern "C"
