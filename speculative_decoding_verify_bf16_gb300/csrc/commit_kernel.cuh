// commit_kernel.cuh -- roll per-lane recurrent state to the committed count.
//
// ignis docs, "Speculative decoding" -- "One round, step by step", step 5, and
// FreeToken issue #828, "Design" (per-request state): the verify forward stages
// one snapshot per column; the commit keeps only the snapshot of the last
// committed column, so a rejected draft leaves no trace in the live state.
//
// The copy is a pure HBM stream (one read and one write of bytes_per_col per
// lane).  Aligned layouts go through the TMA unit: one thread per CTA keeps a
// ring of shared-memory buffers busy with bulk global->shared loads and bulk
// shared->global stores, both with an evict-first L2 policy since every byte is
// touched once.  Other layouts use a plain byte loop.
#pragma once

#include <cstdint>

#include "device_ptx.cuh"
#include "spec_verify.h"

namespace specv {

constexpr int kCommitThreads = 32;
constexpr int kCommitMaxBufs = 8;
constexpr int kCommitHead = 128;  // mbarriers, ahead of the buffers

struct CommitParams {
  const uint8_t* staged;
  uint8_t* live;
  const int32_t* committed;
  int32_t* lane_status;
  int32_t lanes;
  int32_t cols;
  uint64_t bytes_per_col;
  uint64_t staged_lane_stride;
  uint64_t staged_col_stride;
  uint64_t live_lane_stride;
  uint32_t chunk_bytes;    // bytes per work item (multiple of 16)
  uint64_t chunks_per_lane;
  uint64_t total_items;    // lanes * chunks_per_lane
  int32_t nbuf;
  int32_t test_withhold;   // tests only: CTA 0 announces its first load but never issues it
};

// Committed column of lane b, or -1 if the lane must keep its live state.
__device__ __forceinline__ int commit_column(const CommitParams& p, int b) {
  if (p.lane_status != nullptr && p.lane_status[b] != SPEC_OK) return -1;
  const int c = __ldg(p.committed + b);
  return (c >= 1 && c <= p.cols) ? c - 1 : -1;
}

// Lanes whose count is out of range get SPEC_ERR_LAYOUT (CTA 0 only).
__device__ __forceinline__ void commit_mark_layout(const CommitParams& p) {
  if (blockIdx.x != 0 || p.lane_status == nullptr) return;
  for (int b = threadIdx.x; b < p.lanes; b += blockDim.x) {
    const int c = __ldg(p.committed + b);
    if (p.lane_status[b] == SPEC_OK && (c < 1 || c > p.cols)) p.lane_status[b] = SPEC_ERR_LAYOUT;
  }
}

__global__ void __launch_bounds__(kCommitThreads) commit_bulk_kernel(const CommitParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint8_t* bufs = smem + kCommitHead;

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.nbuf; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncthreads();
  griddep_wait();  // committed[] is written by the verify kernel

  if (threadIdx.x == 0) {
    const uint64_t pol = policy_evict_first();
    uint64_t next = blockIdx.x;
    uint8_t* pend_dst[kCommitMaxBufs];
    uint32_t pend_size[kCommitMaxBufs];
    int pend_lane[kCommitMaxBufs];
    uint32_t parity = 0;  // bit i: parity of the next phase of bars[i]

    // Issue the next valid work item of this CTA into buffer `slot`.
    auto issue = [&](int slot) -> bool {
      while (next < p.total_items) {
        const uint64_t item = next;
        next += gridDim.x;
        const int b = static_cast<int>(item / p.chunks_per_lane);
        const int col = commit_column(p, b);
        if (col < 0) continue;
        const uint64_t off = (item % p.chunks_per_lane) * p.chunk_bytes;
        const uint64_t rem = p.bytes_per_col - off;
        const uint32_t size = rem < p.chunk_bytes ? static_cast<uint32_t>(rem) : p.chunk_bytes;
        const uint8_t* src = p.staged + b * p.staged_lane_stride + col * p.staged_col_stride + off;
        pend_dst[slot] = p.live + b * p.live_lane_stride + off;
        pend_size[slot] = size;
        pend_lane[slot] = b;
        mbar_arrive_expect_tx(&bars[slot], size);
        if (p.test_withhold && blockIdx.x == 0 && item == 0) return true;  // tests only: never copied
        bulk_g2s_hint(bufs + static_cast<size_t>(slot) * p.chunk_bytes, src, size, &bars[slot], pol);
        return true;
      }
      return false;
    };

    int inflight = 0;
    for (int s = 0; s < p.nbuf; ++s) {
      if (!issue(s)) break;
      ++inflight;
    }
    int slot = 0;
    bool timed_out = false;
    while (inflight > 0) {
      if (!mbar_wait_bounded(&bars[slot], (parity >> slot) & 1u)) {
        timed_out = true;
        break;
      }
      parity ^= 1u << slot;
      bulk_s2g_hint(pend_dst[slot], bufs + static_cast<size_t>(slot) * p.chunk_bytes, pend_size[slot], pol);
      bulk_commit_group();
      bulk_wait_group_read<0>();  // buffer free again
      --inflight;
      if (issue(slot)) ++inflight;
      slot = (slot + 1 == p.nbuf) ? 0 : slot + 1;
    }
    if (timed_out) {
      // A load never landed: every lane this CTA still had work for -- the
      // lanes of the loads in flight and of every item it has not issued --
      // reports SPEC_ERR_TIMEOUT (its live state may be partly written); the
      // loads in flight land before the CTA exits.
      for (int i = 0; i < inflight; ++i) {
        if (p.lane_status) p.lane_status[pend_lane[slot]] = SPEC_ERR_TIMEOUT;
        mbar_wait_bounded(&bars[slot], (parity >> slot) & 1u);
        slot = (slot + 1 == p.nbuf) ? 0 : slot + 1;
      }
      for (; next < p.total_items; next += gridDim.x) {
        const int b = static_cast<int>(next / p.chunks_per_lane);
        if (p.lane_status && commit_column(p, b) >= 0) p.lane_status[b] = SPEC_ERR_TIMEOUT;
      }
    }
    bulk_wait_group<0>();
  }
  __syncthreads();
  commit_mark_layout(p);
}

// Layouts without 16-byte alignment: one byte per thread and step.
__global__ void commit_bytes_kernel(const CommitParams p) {
  griddep_wait();
  const uint64_t total = static_cast<uint64_t>(p.lanes) * p.bytes_per_col;
  for (uint64_t i = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
    const int b = static_cast<int>(i / p.bytes_per_col);
    const uint64_t off = i % p.bytes_per_col;
    const int col = commit_column(p, b);
    if (col < 0) continue;
    p.live[b * p.live_lane_stride + off] =
        p.staged[b * p.staged_lane_stride + col * p.staged_col_stride + off];
  }
  __syncthreads();
  commit_mark_layout(p);
}

}  // namespace specv
