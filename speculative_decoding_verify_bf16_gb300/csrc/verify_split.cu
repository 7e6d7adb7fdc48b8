// verify_split.cu -- the work-list verify kernel (verify_split.cuh) and its
// host side: launch shape, workspace layout and the launch itself.  The
// element-level helpers (the row sweep, merges, the compensated acceptance
// test, the draw weights) are those of verify_kernel.cuh, built here in a
// namespace of their own.
#define SPEC_VERIFY_CONSUMER_WARPS 20
#define SPEC_VERIFY_PIECES 5
#define specv specv_split
#include "verify_kernel.cuh"
#undef specv

#include <cuda_runtime.h>

#include <cstdlib>
#include <mutex>

#include "verify_split.cuh"
#include "verify_split_host.h"

namespace split_host {

using specv_split_impl::kDrawChunkS;
using specv_split_impl::kGroupsS;
using specv_split_impl::kMaxLanesS;
using specv_split_impl::kMaxSlotsS;
using specv_split_impl::kThreadsS;

namespace {

int env_int(const char* name, int fallback) {
  const char* v = std::getenv(name);
  if (v == nullptr || *v == '\0') return fallback;
  return std::atoi(v);
}

constexpr int kMinChunkBytes = 8192;
constexpr int kMaxChunkBytes = 24576;  // two slots per consumer group fit the ring

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Pass-1 chunks per row with the smallest chunk any launch uses: the bound
// the workspace is sized for.
int max_chunks_per_row(int V, int esize) {
  return static_cast<int>(ceil_div(static_cast<int64_t>(V) * esize, kMinChunkBytes));
}

int head_bytes() { return static_cast<int>((sizeof(specv_split_impl::SplitSmem) + 127) / 128 * 128); }

std::mutex g_attr_mutex;
bool g_attr_done[64][2] = {};

}  // namespace

uint64_t workspace_bytes(int lanes, int rows, int V, int esize) {
  const int nchunk = max_chunks_per_row(V, esize);
  const int nchunk2 = static_cast<int>(ceil_div(V, kDrawChunkS));
  const int64_t n1max = specv_split_impl::max_pass1_items(lanes, rows, nchunk);
  return specv_split_impl::ws_layout(lanes, n1max, nchunk2).total;
}

bool eligible(int lanes, bool aligned) { return aligned && lanes <= kMaxLanesS; }

int choose(const SplitShapeIn& in, SplitShape* out) {
  const int vec = 16 / in.esize;
  // Pass-1 chunk: about eight items per CTA on an estimate of the round's
  // bytes (the target rows; drafter rows only add items), 8-24 KB.
  const int64_t row_bytes = static_cast<int64_t>(in.V) * in.esize;
  const int64_t est_bytes = row_bytes * in.rows;
  int64_t chunk_bytes = est_bytes / (static_cast<int64_t>(in.sms) * 8);
  const int forced_kb = env_int("SPEC_SPLIT_CHUNK_KB", 0);
  if (forced_kb > 0) chunk_bytes = static_cast<int64_t>(forced_kb) * 1024;
  if (chunk_bytes < kMinChunkBytes) chunk_bytes = kMinChunkBytes;
  if (chunk_bytes > kMaxChunkBytes) chunk_bytes = kMaxChunkBytes;
  int64_t chunk = chunk_bytes / in.esize / vec * vec;
  const int64_t v_round = ceil_div(in.V, vec) * vec;
  if (chunk > v_round) chunk = v_round;
  out->chunk = static_cast<int>(chunk);
  out->nchunk = static_cast<int>(ceil_div(in.V, chunk));
  out->nchunk2 = static_cast<int>(ceil_div(in.V, kDrawChunkS));
  out->slot_bytes = static_cast<int>(ceil_div(chunk * in.esize, 16) * 16);
  out->head_bytes = head_bytes();
  int nslots = (in.smem_optin - out->head_bytes) / out->slot_bytes;
  if (nslots > kMaxSlotsS) nslots = kMaxSlotsS;
  nslots -= nslots % kGroupsS;
  if (nslots < kGroupsS) return SPEC_ERR_UNSUPPORTED;
  out->nslots = nslots;
  out->smem = out->head_bytes + nslots * out->slot_bytes;
  // One CTA per SM, fewer when the round has few items.
  const int64_t est_items = static_cast<int64_t>(in.rows) * out->nchunk;
  int64_t grid = ceil_div(est_items, 2);
  const int forced_grid = env_int("SPEC_SPLIT_GRID", 0);
  if (forced_grid > 0) grid = forced_grid;
  if (grid > in.sms) grid = in.sms;
  if (grid < 1) grid = 1;
  out->grid = static_cast<int>(grid);
  out->threads = kThreadsS;
  return SPEC_OK;
}

int launch(const spec_verify_args* a, int dev, int sms, int smem_optin, void* stream) {
  const int esize = (a->dtype == SPEC_BF16) ? 2 : 4;
  SplitShapeIn in{a->lanes, a->rows, a->V, esize, sms, smem_optin};
  SplitShape s{};
  const int rc = choose(in, &s);
  if (rc != SPEC_OK) return rc;
  const int nchunk_max = max_chunks_per_row(a->V, esize);
  const int64_t n1max = specv_split_impl::max_pass1_items(a->lanes, a->rows, nchunk_max);
  const specv_split_impl::WsLayout L = specv_split_impl::ws_layout(a->lanes, n1max, s.nchunk2);
  if (a->workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0)
    return SPEC_ERR_INVALID_ARG;

  void* kernel = (a->dtype == SPEC_BF16)
                     ? reinterpret_cast<void*>(&specv_split_impl::verify_split_kernel<specv_split::bf16_tag>)
                     : reinterpret_cast<void*>(&specv_split_impl::verify_split_kernel<float>);
  {
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    bool& done = g_attr_done[dev & 63][a->dtype == SPEC_BF16 ? 1 : 0];
    if (!done) {
      if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin) != cudaSuccess)
        return SPEC_ERR_CUDA;
      done = true;
    }
  }

  specv_split_impl::SplitParams p{};
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
  p.ws = static_cast<uint8_t*>(a->workspace);
  p.layout = L;
  p.chunk = s.chunk;
  p.nchunk = s.nchunk;
  p.nchunk2 = s.nchunk2;
  p.slot_bytes = s.slot_bytes;
  p.nslots = s.nslots;
  p.head_bytes = s.head_bytes;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(s.grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(s.threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(s.smem);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  void* kargs[] = {&p};
  if (cudaLaunchKernelExC(&cfg, kernel, kargs) != cudaSuccess) {
    cudaGetLastError();
    return SPEC_ERR_CUDA;
  }
  return SPEC_OK;
}

}  // namespace split_host
