// verify_split.cuh -- the verify round as a persistent work list over the whole GPU.
//
// The same round as verify_kernel.cuh (ignis docs, "Speculative decoding" --
// "One round, step by step"; strata2signal, "Guess, then check"), split finer:
// where that kernel gives each lane one thread-block cluster (at most one GPC,
// so a round of few lanes leaves most SMs idle), this one runs one CTA per SM
// and hands out the round as items:
//
//   pass-1 item   one vocabulary chunk of one row (target row j, or drafter row
//                 j of a sampled lane) of one lane: the producer warp claims it
//                 from a global counter, streams it into a shared-memory ring
//                 with a bulk copy, and a group of consumer warps reduces it to
//                 a partial (max, lowest index of the max, and for sampled rows
//                 the exp2 sum against a reference), written to the workspace.
//   lane finish   the group that completes a lane's last pass-1 item (a counter
//                 per lane) merges the lane's partials in chunk order, runs the
//                 acceptance scan and writes the outputs; for a sampled lane it
//                 publishes the draw's row pair as pass-2 items.
//   pass-2 item   one chunk of the draw's weights max(0, p_n - q_n) (or p_k),
//                 summed from the row pair re-read from L2; claimed before any
//                 pass-1 item, so draws overlap the streaming of other lanes.
//   draw finish   the group completing a lane's last pass-2 item finds the chunk
//                 that holds u' * W from the chunk sums and walks it to the token.
//
// Every sum the draw compares is recomputed by the same code in the same order
// where it is walked, so the walk agrees with the sums bit for bit.  Partials
// are merged in chunk order, so results do not depend on which CTA took which
// item.
//
// The workspace is caller-owned device memory that must be zero before the
// first launch; every launch leaves its counters at zero again (each finisher
// resets its lane's counters, the last CTA to exit resets the shared ones and
// the queue's ready flags); the partials and draw descriptors are scratch that
// the next launch overwrites before reading.  Every wait is bounded (2 s
// without progress): a launch in which any wait gives up reports
// SPEC_ERR_TIMEOUT for every lane, commits nothing, and still leaves the
// counters at zero.
#pragma once

#include <cstdint>

namespace specv_split_impl {

using namespace specv_split;

constexpr int kGroupsS = 4;                     // consumer-warp groups
constexpr int kGroupWarpsS = 5;                 // warps per group
constexpr int kConsumerWarpsS = kGroupsS * kGroupWarpsS;
constexpr int kProducerWarpS = kConsumerWarpsS;
constexpr int kThreadsS = (kConsumerWarpsS + 1) * 32;
constexpr int kGroupThreads = kGroupWarpsS * 32;
constexpr int kMaxLanesS = 2048;                // item prefix kept in shared memory
constexpr int kMaxSlotsS = 32;
constexpr int kDrawSeg = 1024;                  // pass-2 elements per warp of a group
constexpr int kDrawChunkS = kGroupWarpsS * kDrawSeg;  // pass-2 elements per item

enum ItemKind : int32_t { kItemP1 = 0, kItemP2 = 1, kItemStatus = 2, kItemStop = 3 };
enum DrawModeS : int32_t { kModeResidual = 1, kModeBonus = 2, kModeFromP = 3 };

// Shared counters at the start of the workspace, each in its own 32-byte sector.
struct __align__(256) WsHeader {
  uint32_t p1_claim;     uint32_t pad0[7];  // pass-1 items claimed
  uint32_t p2_claim;     uint32_t pad1[7];  // pass-2 items claimed
  uint32_t p2_reserved;  uint32_t pad2[7];  // lanes whose draw has been queued
  uint32_t lanes_done;   uint32_t pad3[7];  // lanes whose outputs are complete
  uint32_t exited;       uint32_t pad4[7];  // CTAs that have finished
  uint32_t error;        uint32_t pad5[7];  // a wait gave up somewhere in this launch
  uint32_t pad6[16];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

// What pass 2 of a sampled lane needs (written by its lane finisher).
struct __align__(32) DrawDesc {
  int32_t n;     // position of the draw (the first rejected row, or k)
  int32_t mode;  // DrawModeS
  float mp, l2sp;  // target row: scaled reference and log2 of its sum
  float mq, l2sq;  // drafter row n (residual mode)
  float c;         // log2(e) / T
  float u;         // the draw's uniform u'
};

struct DrawPartS {
  float w;     // sum of the chunk's weights (in the fixed order of the group)
  int32_t last;  // largest index of positive weight in the chunk (-1 if none)
};

// Byte offsets of the workspace arrays.
struct WsLayout {
  uint64_t cnt1, cnt2, queue, ready, desc, part1, part2, total;
};

__host__ __device__ inline uint64_t ws_align(uint64_t x) { return (x + 255) / 256 * 256; }

// n1max bounds the pass-1 items of a launch; nchunk2 is the pass-2 chunks per row.
__host__ __device__ inline WsLayout ws_layout(int lanes, int64_t n1max, int nchunk2) {
  WsLayout L;
  uint64_t o = sizeof(WsHeader);
  L.cnt1 = o;  o = ws_align(o + 4ull * lanes);
  L.cnt2 = o;  o = ws_align(o + 4ull * lanes);
  L.queue = o; o = ws_align(o + 8ull * lanes);  // a lane may queue its draw twice
  L.ready = o; o = ws_align(o + 8ull * lanes);
  L.desc = o;  o = ws_align(o + sizeof(DrawDesc) * static_cast<uint64_t>(lanes));
  L.part1 = o; o = ws_align(o + sizeof(Partial) * static_cast<uint64_t>(n1max));
  L.part2 = o; o = ws_align(o + sizeof(DrawPartS) * static_cast<uint64_t>(lanes) * nchunk2);
  L.total = o;
  return L;
}

// Items a lane can need at most: every row of the lane streamed in `nchunk`
// chunks (a sampled lane reads 2 k + 1 rows for k + 1 row slots), or one
// status item; summed over lanes this is at most 2 * rows * nchunk + lanes.
__host__ __device__ inline int64_t max_pass1_items(int lanes, int rows, int nchunk) {
  return 2ll * rows * nchunk + lanes;
}

struct SplitParams {
  const uint8_t* target;
  const uint8_t* draft;
  int64_t ld_bytes;
  int32_t V;
  int32_t lanes;
  int32_t rows;
  const int32_t* draft_tokens;
  const int32_t* draft_lens;
  const int32_t* row_offsets;
  const float* temps;
  uint64_t seed;
  int32_t* committed;
  int32_t* out_tokens;
  int32_t* lane_status;
  spec_row_stats* row_stats;
  uint32_t lane_base;
  uint32_t flags;
  uint8_t* ws;
  WsLayout layout;
  int32_t chunk;      // pass-1 elements per item (multiple of the vector width)
  int32_t nchunk;     // pass-1 chunks per row
  int32_t nchunk2;    // pass-2 chunks per row
  int32_t slot_bytes; // ring slot (>= chunk * element size)
  int32_t nslots;     // multiple of kGroupsS
  int32_t head_bytes; // offset of the ring in dynamic shared memory
};

struct SlotItem {
  int32_t kind;
  int32_t lane;
  int32_t s;       // pass 1: stream (sampled: 2j target, 2j+1 drafter; greedy: j); pass 2: queue entry
  int32_t chunk;
  int32_t elems;   // pass 1: elements of the chunk
  int32_t bulk;    // pass 1: elements copied into the slot (multiple of the vector width)
  float c;         // pass 1: log2(e) / T (sampled lanes)
  int32_t sampled;
};

// Per-group scratch of the finishers.
struct GroupScratch {
  Partial wpart[kGroupWarpsS];
  Partial fin[kMaxStreams];
  int32_t drafts[kMaxDrafts + 1];
  float xd_t[kMaxDrafts + 1];
  float xd_q[kMaxDrafts + 1];
  float u_acc[kMaxDrafts + 1];
  float u_smp[kMaxDrafts + 1];
  float segw[kGroupWarpsS];
  int32_t segl[kGroupWarpsS];
  int32_t bcast[4];
  float fbcast[4];
};

struct __align__(16) SplitSmem {
  uint64_t full[kMaxSlotsS];
  uint64_t empty[kMaxSlotsS];
  SlotItem item[kMaxSlotsS];
  GroupScratch grp[kGroupsS];
  int32_t lane_item[kMaxLanesS + 1];  // first pass-1 item of each lane (exclusive prefix)
  int32_t scan_tmp[32];
  uint32_t broken;                     // a wait in this CTA gave up
  uint32_t exit_last;                  // this CTA is the last to exit
  uint32_t group_fail[kGroupsS];       // a warp of the group gave up waiting for a slot
};

// ---------------------------------------------------------------------------
// Memory-model helpers (GPU scope)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// atomic add with acquire-release semantics at GPU scope; returns the old value.
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void group_sync(int group) {
  asm volatile("bar.sync %0, %1;" ::"r"(group + 1), "n"(kGroupThreads) : "memory");
}

// A 16-byte partial read from another SM's writes (L2, not L1).
__device__ __forceinline__ Partial load_partial(const Partial* p) {
  const uint4 v = __ldcg(reinterpret_cast<const uint4*>(p));
  return Partial{__uint_as_float(v.x), __uint_as_float(v.y), static_cast<int>(v.z), v.w};
}

__device__ __forceinline__ void store_partial(Partial* p, const Partial& q) {
  __stcg(reinterpret_cast<uint4*>(p), make_uint4(__float_as_uint(q.m), __float_as_uint(q.s),
                                                  static_cast<uint32_t>(q.idx), q.flags));
}

template <typename T>
struct SplitKernel {
  static constexpr int kVec = ElemTraits<T>::kVec;
  static constexpr int kEsize = 16 / kVec;

  const SplitParams& p;
  SplitSmem& sh;
  uint8_t* ring;
  WsHeader* hdr;
  uint32_t* cnt1;
  uint32_t* cnt2;
  uint32_t* queue;
  uint32_t* ready;
  DrawDesc* desc;
  Partial* part1;
  DrawPartS* part2;
  int32_t n1;  // pass-1 items of this launch

  __device__ SplitKernel(const SplitParams& pp, SplitSmem& s, uint8_t* r) : p(pp), sh(s), ring(r) {
    hdr = reinterpret_cast<WsHeader*>(p.ws);
    cnt1 = reinterpret_cast<uint32_t*>(p.ws + p.layout.cnt1);
    cnt2 = reinterpret_cast<uint32_t*>(p.ws + p.layout.cnt2);
    queue = reinterpret_cast<uint32_t*>(p.ws + p.layout.queue);
    ready = reinterpret_cast<uint32_t*>(p.ws + p.layout.ready);
    desc = reinterpret_cast<DrawDesc*>(p.ws + p.layout.desc);
    part1 = reinterpret_cast<Partial*>(p.ws + p.layout.part1);
    part2 = reinterpret_cast<DrawPartS*>(p.ws + p.layout.part2);
    n1 = 0;
  }

  // Status of a lane from its metadata alone (the checks that need no logits).
  __device__ int meta_status(int b, int& k, int& off, bool& sampled) const {
    k = __ldg(p.draft_lens + b);
    off = __ldg(p.row_offsets + b);
    const int end = __ldg(p.row_offsets + b + 1);
    sampled = __ldg(p.temps + b) > 0.f;
    if (k < 0 || off < 0 || end > p.rows || end - off != k + 1) return SPEC_ERR_LAYOUT;
    if (k > kMaxDrafts) return SPEC_ERR_UNSUPPORTED;
    if (sampled && p.draft == nullptr) return SPEC_ERR_INVALID_ARG;
    return SPEC_OK;
  }

  __device__ int lane_items(int b) const {
    int k, off;
    bool sampled;
    if (meta_status(b, k, off, sampled) != SPEC_OK) return 1;  // one status item
    return (sampled ? 2 * k + 1 : k + 1) * p.nchunk;
  }

  // Exclusive prefix of the lanes' item counts, in shared memory (all threads).
  __device__ void build_item_prefix() {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (p.lanes + kThreadsS - 1) / kThreadsS;
    const int b0 = min(p.lanes, tid * per), b1 = min(p.lanes, b0 + per);
    int local = 0;
    for (int b = b0; b < b1; ++b) local += lane_items(b);
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int up = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += up;
    }
    if (lane == 31) sh.scan_tmp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int v = (lane < kThreadsS / 32) ? sh.scan_tmp[lane] : 0;
      int wi = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int up = __shfl_up_sync(0xFFFFFFFFu, wi, o);
        if (lane >= o) wi += up;
      }
      if (lane < kThreadsS / 32) sh.scan_tmp[lane] = wi - v;  // exclusive per warp
      if (lane == kThreadsS / 32 - 1) sh.lane_item[p.lanes] = wi;
    }
    __syncthreads();
    int run = sh.scan_tmp[warp] + incl - local;
    for (int b = b0; b < b1; ++b) {
      sh.lane_item[b] = run;
      run += lane_items(b);
    }
    __syncthreads();
    n1 = sh.lane_item[p.lanes];
  }

  // Lane owning pass-1 item g (binary search over the prefix).
  __device__ int lane_of_item(int g) const {
    int lo = 0, hi = p.lanes - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (sh.lane_item[mid] <= g) lo = mid;
      else hi = mid - 1;
    }
    return lo;
  }

  __device__ const uint8_t* stream_row(int off, bool sampled, int s) const {
    const bool is_draft = sampled && (s & 1);
    const int j = sampled ? (s >> 1) : s;
    return (is_draft ? p.draft : p.target) + static_cast<int64_t>(off + j) * p.ld_bytes;
  }

  // ---------------------------------------------------------------------
  // Producer: lane g of the producer warp fills the slots of group g.
  // ---------------------------------------------------------------------
  __device__ bool claim_p2(uint32_t& item) const {
    uint32_t cur = ld_relaxed(&hdr->p2_claim);
    for (;;) {
      const uint32_t avail = ld_relaxed(&hdr->p2_reserved) * static_cast<uint32_t>(p.nchunk2);
      if (cur >= avail) return false;
      const uint32_t prev = atomicCAS(&hdr->p2_claim, cur, cur + 1);
      if (prev == cur) {
        item = cur;
        return true;
      }
      cur = prev;
    }
  }

  __device__ __noinline__ void producer(int g) {
    const uint32_t ns = static_cast<uint32_t>(p.nslots);
    uint32_t slot = static_cast<uint32_t>(g), par = 0;
    uint32_t fills = 0;
    bool p1_left = true, ok = true;
    const bool withhold = (p.flags & SPEC_VERIFY_TEST_WITHHOLD_COPY) != 0u;
    uint64_t idle_since = 0;
    uint32_t seen_done = 0xFFFFFFFFu, seen_res = 0xFFFFFFFFu;
    for (;;) {
      SlotItem it{};
      it.kind = -1;
      uint32_t q;
      if (claim_p2(q)) {
        it.kind = kItemP2;
        it.s = static_cast<int>(q / static_cast<uint32_t>(p.nchunk2));
        it.chunk = static_cast<int>(q % static_cast<uint32_t>(p.nchunk2));
      } else if (p1_left) {
        const int gi = static_cast<int>(atomicAdd(&hdr->p1_claim, 1u));
        if (gi >= n1) {
          p1_left = false;
        } else {
          const int b = lane_of_item(gi);
          const int r = gi - sh.lane_item[b];
          it.lane = b;
          int k, off;
          bool sampled;
          if (meta_status(b, k, off, sampled) != SPEC_OK) {
            it.kind = kItemStatus;
          } else {
            it.kind = kItemP1;
            it.s = r / p.nchunk;
            it.chunk = r % p.nchunk;
            const int e0 = it.chunk * p.chunk;
            it.elems = min(p.chunk, p.V - e0);
            it.bulk = (it.elems / kVec) * kVec;
            it.sampled = sampled ? 1 : 0;
            it.c = sampled ? __fdiv_rn(kLog2e, __ldg(p.temps + b)) : 0.f;
            if (withhold && gi == n1 - 1 && it.bulk > 0) it.bulk = -it.bulk - 1;  // test only: never copied
          }
        }
      }
      if (it.kind < 0) {
        // Nothing to claim now: stop when every lane is complete, else wait.
        const uint32_t done = ld_relaxed(&hdr->lanes_done);
        const uint32_t res = ld_relaxed(&hdr->p2_reserved);
        if (done >= static_cast<uint32_t>(p.lanes) || ld_relaxed(&hdr->error) != 0u || sh.broken) {
          it.kind = kItemStop;
        } else {
          const uint64_t now = global_ns();
          if (done != seen_done || res != seen_res || idle_since == 0) {
            seen_done = done;
            seen_res = res;
            idle_since = now;
          } else if (now - idle_since > kWaitLimitNs) {
            atomicOr(&hdr->error, 1u);
            it.kind = kItemStop;
          }
          if (it.kind < 0) {
            __nanosleep(128);
            continue;
          }
        }
      }
      if (!mbar_wait_bounded(&sh.empty[slot], par ^ 1u)) {
        ok = false;
        break;
      }
      sh.item[slot] = it;
      if (it.kind == kItemP1 && it.bulk > 0) {
        int k, off;
        bool sampled;
        meta_status(it.lane, k, off, sampled);
        const uint8_t* src = stream_row(off, sampled, it.s) + static_cast<int64_t>(it.chunk) * p.chunk * kEsize;
        mbar_arrive_expect_tx(&sh.full[slot], static_cast<uint32_t>(it.bulk * kEsize));
        bulk_g2s(ring + static_cast<size_t>(slot) * p.slot_bytes, src, static_cast<uint32_t>(it.bulk * kEsize),
                 &sh.full[slot]);
      } else if (it.kind == kItemP1 && it.bulk < -1) {
        // Test only (SPEC_VERIFY_TEST_WITHHOLD_COPY): announce the bytes, copy nothing.
        mbar_arrive_expect_tx(&sh.full[slot], static_cast<uint32_t>((-it.bulk - 1) * kEsize));
      } else {
        mbar_arrive(&sh.full[slot]);
      }
      ++fills;
      if (it.kind == kItemStop) break;
      slot += kGroupsS;
      if (slot >= ns) {
        slot -= ns;
        par ^= 1u;
      }
    }
    if (!ok) {
      sh.broken = 1u;
      atomicOr(&hdr->error, 1u);
    }
    // Drain: the last fill of each of this lane's slots has landed (or gives
    // up) before the CTA's shared memory is released.
    const uint32_t mine = ns / kGroupsS;
    for (uint32_t m = 0; m < mine && m < fills; ++m) {
      // Slot of the m-th most recent fill, and the parity of that fill.
      int64_t idx = static_cast<int64_t>(fills) - 1 - m;  // fill number
      const uint32_t s = static_cast<uint32_t>(g) + static_cast<uint32_t>(idx % mine) * kGroupsS;
      const uint32_t ph = static_cast<uint32_t>((idx / mine) & 1);
      mbar_wait_bounded(&sh.full[s], ph);
    }
  }

  // ---------------------------------------------------------------------
  // Consumers
  // ---------------------------------------------------------------------
  // One pass-1 chunk reduced by the group's warps; the group's partial goes to
  // the workspace.  Returns true if this item completed its lane.
  __device__ void reduce_chunk(const SlotItem& it, const uint4* sv, int gw, int lane, int group, bool timed_out) {
    GroupScratch& gs = sh.grp[group];
    const bool sampled = it.sampled != 0;
    const int e0 = it.chunk * p.chunk;
    Acc a;
    acc_init(a);
    if (!timed_out) {
      const int nvec = it.bulk / kVec;
      const int per = (nvec + kGroupWarpsS - 1) / kGroupWarpsS;
      const int vb = min(nvec, gw * per), ve = min(nvec, vb + per);
      if (sampled && p.row_stats != nullptr) acc_range<T, true, false>(a, sv, vb, ve, e0, it.c, lane);
      else if (sampled) acc_range<T, true, true>(a, sv, vb, ve, e0, it.c, lane);
      else acc_range<T, false>(a, sv, vb, ve, e0, it.c, lane);
      // The chunk's last elements past the copied vectors (the row's ragged end).
      if (gw == kGroupWarpsS - 1 && it.elems > it.bulk) {
        int k, off;
        bool sm;
        meta_status(it.lane, k, off, sm);
        const uint8_t* row = stream_row(off, sampled, it.s);
        for (int e = it.bulk + lane; e < it.elems; e += 32) {
          const float x = ElemTraits<T>::load(row, e0 + e);
          if (sampled) acc_scalar<true>(a, x, e0 + e, it.c);
          else acc_scalar<false>(a, x, e0 + e, it.c);
        }
      }
    }
    const uint32_t fl = acc_bad(a) | (timed_out ? kTimedOut : 0u);
    const Partial wp = sampled ? warp_merge<true>(a.m, a.s, a.idx, fl, it.c)
                               : warp_merge<false>(a.m, a.s, a.idx, fl, it.c);
    if (lane == 0) gs.wpart[gw] = wp;
  }

  // Merge of the group's warp partials (warp 0 of the group, lanes < kGroupWarpsS).
  __device__ Partial group_partial(const SlotItem& it, int group, int lane) {
    GroupScratch& gs = sh.grp[group];
    const Partial q = (lane < kGroupWarpsS) ? gs.wpart[lane] : identity_partial();
    return it.sampled ? warp_merge<true>(q.m, q.s, q.idx, q.flags, it.c)
                      : warp_merge<false>(q.m, q.s, q.idx, q.flags, it.c);
  }

  // ---------------------------------------------------------------------
  // Lane finisher (pass 1 complete): merge, scan, outputs, draw publication.
  // ---------------------------------------------------------------------
  __device__ __noinline__ void finish_lane(int b, int group, int gw, int lane) {
    GroupScratch& gs = sh.grp[group];
    int k, off;
    bool sampled;
    int status = meta_status(b, k, off, sampled);
    const float temp = __ldg(p.temps + b);
    const float c = sampled ? __fdiv_rn(kLog2e, temp) : 0.f;
    const int nstreams = (status != SPEC_OK) ? 0 : (sampled ? 2 * k + 1 : k + 1);
    const int base = sh.lane_item[b];
    // Draft tokens, the logits at them and the uniforms (warp 0), while the
    // other warps merge the partials.
    if (gw == 0 && status == SPEC_OK && lane <= k) {
      const int j = lane;
      if (j < k) {
        const int d = __ldg(p.draft_tokens + off + j);
        gs.drafts[j] = d;
        if (sampled && d >= 0 && d < p.V) {
          gs.xd_t[j] = ElemTraits<T>::load(p.target + static_cast<int64_t>(off + j) * p.ld_bytes, d);
          gs.xd_q[j] = ElemTraits<T>::load(p.draft + static_cast<int64_t>(off + j) * p.ld_bytes, d);
        }
      }
      if (sampled) {
        const float2 u = round_uniforms(p.seed, p.lane_base + static_cast<uint32_t>(b), static_cast<uint32_t>(j));
        gs.u_acc[j] = u.x;
        gs.u_smp[j] = u.y;
      }
    }
    // Stream s of the lane: its chunks' partials merged in chunk order.
    for (int s = gw; s < nstreams; s += kGroupWarpsS) {
      const Partial* src = part1 + base + static_cast<int64_t>(s) * p.nchunk;
      float m = -INFINITY, sum = 0.f;
      int idx = INT_MAX;
      uint32_t fl = 0;
      if (sampled) {
        for (int ch = lane; ch < p.nchunk; ch += 32) {
          const Partial q = load_partial(src + ch);
          merge_part<true>(m, sum, idx, q.m, q.s, q.idx, c);
          fl |= q.flags;
        }
        const Partial r = warp_merge<true>(m, sum, idx, fl, c);
        if (lane == 0) gs.fin[s] = r;
      } else {
        unsigned long long key = 0ull;
        for (int ch = lane; ch < p.nchunk; ch += 32) {
          const Partial q = load_partial(src + ch);
          const unsigned long long kq = argmax_key(q.m, q.idx);
          key = kq > key ? kq : key;
          fl |= q.flags;
        }
        // Warp max of the 64-bit keys: the high word first, then the low word among the winners.
        const uint32_t hi = __reduce_max_sync(0xFFFFFFFFu, static_cast<uint32_t>(key >> 32));
        const uint32_t lo = __reduce_max_sync(0xFFFFFFFFu, (static_cast<uint32_t>(key >> 32) == hi)
                                                               ? static_cast<uint32_t>(key) : 0u);
        fl = __reduce_or_sync(0xFFFFFFFFu, fl);
        if (lane == 0) {
          float mm;
          int ii;
          argmax_key_decode((static_cast<unsigned long long>(hi) << 32) | lo, mm, ii);
          gs.fin[s] = Partial{mm, 0.f, ii, fl};
        }
      }
    }
    group_sync(group);

    if (gw == 0) {
      int st = status;
      bool range_bad = false;
      if (st == SPEC_OK && lane < k) {
        const int d = gs.drafts[lane];
        range_bad = (d < 0 || d >= p.V);
      }
      if (__any_sync(0xFFFFFFFFu, range_bad)) st = SPEC_ERR_TOKEN_RANGE;
      if (st == SPEC_OK) {
        uint32_t fl = 0;
        bool empty_row = false;
        for (int s = lane; s < nstreams; s += 32) {
          fl |= gs.fin[s].flags;
          empty_row |= (gs.fin[s].idx == INT_MAX);
        }
        const uint32_t all = __reduce_or_sync(0xFFFFFFFFu, fl);
        if (all & kTimedOut) st = SPEC_ERR_TIMEOUT;
        else if ((all & kBadValue) || __any_sync(0xFFFFFFFFu, empty_row)) st = SPEC_ERR_NONFINITE;
      }
      int n = 0, mode = 0;
      float lp = NAN, lq = NAN;
      if (st == SPEC_OK && !sampled) {
        const bool stop = lane < k && gs.drafts[lane] != gs.fin[lane].idx;
        const uint32_t mask = __ballot_sync(0xFFFFFFFFu, stop);
        n = mask ? (__ffs(mask) - 1) : k;
      } else if (st == SPEC_OK) {
        // log2(u) < log2 p(d) - log2 q(d) as one compensated fp32 sum of exact terms.
        const bool active = lane < k;
        bool accept = true;
        if (active) {
          const float xt = gs.xd_t[lane], xq = gs.xd_q[lane];
          CompSum dp = log2_prob_terms(xt, gs.fin[2 * lane], c);
          const CompSum dq = log2_prob_terms(xq, gs.fin[2 * lane + 1], c);
          lp = (xt == -INFINITY) ? -INFINITY : dp.value();
          lq = (xq == -INFINITY) ? -INFINITY : dq.value();
          const float u = gs.u_acc[lane];
          if (xt == -INFINITY) {
            accept = false;
          } else if (xq == -INFINITY || u == 0.f) {
            accept = true;
          } else {
            float iu, fu;
            log2_parts(u, iu, fu);
            dp.add(-dq.s);
            dp.add(-dq.c);
            dp.add(-iu);
            dp.add(-fu);
            accept = dp.value() > 0.f;
          }
        }
        const uint32_t mask = __ballot_sync(0xFFFFFFFFu, active && !accept);
        n = mask ? (__ffs(mask) - 1) : k;
        mode = (n < k) ? kModeResidual : kModeBonus;
      }
      // Outputs.
      const bool layout_ok = (status != SPEC_ERR_LAYOUT);
      if (lane == 0) {
        p.committed[b] = (st == SPEC_OK) ? n + 1 : 0;
        if (p.lane_status) p.lane_status[b] = st;
      }
      for (int j = lane; layout_ok && j <= k; j += 32) {
        int tok = -1;
        if (st == SPEC_OK && j <= n) tok = sampled ? (j < n ? gs.drafts[j] : -1) : gs.fin[j].idx;
        const bool drawn_here = sampled && st == SPEC_OK && j == n;
        if (!drawn_here) p.out_tokens[off + j] = tok;
        if (p.row_stats && st == SPEC_OK) {
          spec_row_stats* rs = p.row_stats + off + j;
          const Partial pt = sampled ? gs.fin[2 * j] : gs.fin[j];
          rs->argmax = pt.idx;
          rs->max_logit = pt.m;
          if (sampled) {
            float ip, fp;
            log2_parts(pt.s, ip, fp);
            CompSum l;
            l.add(scaled_ref(pt.m, c));
            l.add(ip);
            l.add(fp);
            rs->lse = __fmul_rn(l.value(), kLn2);
            // k <= 15, so lane j computed position j's log p and log q itself
            rs->logp_d = (j < k) ? __fmul_rn(lp, kLn2) : NAN;
            rs->logq_d = (j < k) ? __fmul_rn(lq, kLn2) : NAN;
          } else {
            rs->lse = NAN;
            rs->logp_d = NAN;
            rs->logq_d = NAN;
          }
          rs->resid_mass = NAN;
          rs->drawn = -1;
          rs->flags = 1 | (drawn_here ? (mode == kModeResidual ? 2 : 4) : 0);
        }
      }
      __syncwarp();  // every lane's outputs are ordered before the publication below
      if (lane == 0) {
        st_relaxed(cnt1 + b, 0u);
        if (sampled && st == SPEC_OK) {
          // The draw's row pair: bring it back into L2, describe it, queue it.
          const int drow = (mode == kModeResidual) ? n : k;
          const Partial pt = gs.fin[2 * drow];
          DrawDesc d;
          d.n = n;
          d.mode = mode;
          d.mp = scaled_ref(pt.m, c);
          d.l2sp = log2f(pt.s);
          d.mq = 0.f;
          d.l2sq = 0.f;
          if (mode == kModeResidual) {
            const Partial pq = gs.fin[2 * n + 1];
            d.mq = scaled_ref(pq.m, c);
            d.l2sq = log2f(pq.s);
          }
          d.c = c;
          d.u = gs.u_smp[n];
          desc[b] = d;
          const int64_t rb = static_cast<int64_t>(p.V) * kEsize / 16 * 16;
          for (int64_t o = 0; o < rb; o += 32768) {
            const uint32_t sz = static_cast<uint32_t>(min(static_cast<int64_t>(32768), rb - o));
            bulk_prefetch_l2(p.target + static_cast<int64_t>(off + drow) * p.ld_bytes + o, sz);
            if (mode == kModeResidual) bulk_prefetch_l2(p.draft + static_cast<int64_t>(off + n) * p.ld_bytes + o, sz);
          }
          publish_draw(b);
        } else {
          __threadfence();
          atomicAdd(&hdr->lanes_done, 1u);
        }
      }
    }
    group_sync(group);
  }

  __device__ void publish_draw(int b) {
    __threadfence();
    const uint32_t i = atomicAdd(&hdr->p2_reserved, 1u);
    queue[i] = static_cast<uint32_t>(b);
    st_release(ready + i, 1u);
  }

  // ---------------------------------------------------------------------
  // Pass 2
  // ---------------------------------------------------------------------
  __device__ DrawCoef coef_of(const DrawDesc& d) const {
    DrawCoef kc;
    kc.mp = d.mp;
    kc.l2sp = d.l2sp;
    kc.mq = d.mq;
    kc.l2sq = d.l2sq;
    kc.c = d.c;
    kc.residual = (d.mode == kModeResidual);
    return kc;
  }

  // Weight sum of warp gw's segment of pass-2 chunk ch, in rounds of 256
  // elements (all loads of the segment in flight together); optionally the
  // sum of each round.  The same code computes the sums the draw compares and
  // re-walks, so both see identical bits.
  __device__ float seg_sum(const DrawCoef& kc, const uint8_t* trow, const uint8_t* qrow, int ch, int gw, int lane,
                           int& last, float (&rsum)[kDrawSeg / kDrawRound]) const {
    constexpr int kR = kDrawSeg / kDrawRound;
    const int s0 = ch * kDrawChunkS + gw * kDrawSeg;
    const int s1 = min(p.V, s0 + kDrawSeg);
    Raw8<T> rt[kR], rq[kR];
#pragma unroll
    for (int u = 0; u < kR; ++u) {
      const int e = s0 + u * kDrawRound + lane * 8;
      if (s0 + u * kDrawRound < s1) {
        load_raw8<T, true>(trow, e, s1, rt[u]);
        if (kc.residual) load_raw8<T, true>(qrow, e, s1, rq[u]);
      }
    }
    float segw = 0.f;
#pragma unroll
    for (int u = 0; u < kR; ++u) {
      rsum[u] = 0.f;
      if (s0 + u * kDrawRound >= s1) continue;
      float w[8], cum[8];
      const int e = s0 + u * kDrawRound + lane * 8;
      draw_piece<T>(kc, rt[u], rq[u], e, s1, w, cum);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (w[i] > 0.f) last = e + i;
      const float R = warp_sum_xor(cum[7]);
      rsum[u] = R;
      segw = __fadd_rn(segw, R);
    }
    return segw;
  }

  __device__ void row_pair(int b, const DrawDesc& d, const uint8_t*& trow, const uint8_t*& qrow) const {
    const int off = __ldg(p.row_offsets + b);
    const int k = __ldg(p.draft_lens + b);
    const int drow = (d.mode == kModeBonus) ? k : d.n;
    trow = p.target + static_cast<int64_t>(off + drow) * p.ld_bytes;
    qrow = (d.mode == kModeResidual) ? p.draft + static_cast<int64_t>(off + d.n) * p.ld_bytes : nullptr;
  }

  // Lane of queue entry e, once its publication is visible (bounded wait).
  __device__ int queued_lane(int e) {
    if (ld_acquire(ready + e) == 0u) {
      const uint64_t t0 = global_ns();
      while (ld_acquire(ready + e) == 0u) {
        if (global_ns() - t0 > kWaitLimitNs) {
          atomicOr(&hdr->error, 1u);
          return -1;
        }
      }
    }
    return static_cast<int>(__ldcg(queue + e));
  }

  __device__ __noinline__ void pass2_item(const SlotItem& it, int group, int gw, int lane) {
    GroupScratch& gs = sh.grp[group];
    if (gw == 0 && lane == 0) gs.bcast[0] = queued_lane(it.s);
    group_sync(group);
    const int b = gs.bcast[0];
    if (b < 0) {
      group_sync(group);
      return;
    }
    DrawDesc d;
    {
      const uint4* dp = reinterpret_cast<const uint4*>(desc + b);
      const uint4 a0 = __ldcg(dp), a1 = __ldcg(dp + 1);
      d.n = static_cast<int>(a0.x);
      d.mode = static_cast<int>(a0.y);
      d.mp = __uint_as_float(a0.z);
      d.l2sp = __uint_as_float(a0.w);
      d.mq = __uint_as_float(a1.x);
      d.l2sq = __uint_as_float(a1.y);
      d.c = __uint_as_float(a1.z);
      d.u = __uint_as_float(a1.w);
    }
    const DrawCoef kc = coef_of(d);
    const uint8_t *trow, *qrow;
    row_pair(b, d, trow, qrow);
    int last = -1;
    float rs[kDrawSeg / kDrawRound];
    const float w = seg_sum(kc, trow, qrow, it.chunk, gw, lane, last, rs);
    last = warp_max_int(last);
    if (lane == 0) {
      gs.segw[gw] = w;
      gs.segl[gw] = last;
    }
    group_sync(group);
    if (gw == 0) {
      int is_last = 0;
      if (lane == 0) {
        float W = 0.f;
        int L = -1;
        for (int x = 0; x < kGroupWarpsS; ++x) {
          W = __fadd_rn(W, gs.segw[x]);
          L = max(L, gs.segl[x]);
        }
        DrawPartS* dst = part2 + static_cast<int64_t>(b) * p.nchunk2 + it.chunk;
        __stcg(reinterpret_cast<float2*>(dst), make_float2(W, __int_as_float(L)));
        __threadfence();
        const uint32_t old = atom_add_acq_rel(cnt2 + b, 1u);
        is_last = (old + 1 == static_cast<uint32_t>(p.nchunk2)) ? 1 : 0;
        gs.bcast[1] = is_last;
      }
    }
    group_sync(group);
    if (gs.bcast[1]) finish_draw(b, d, kc, trow, qrow, group, gw, lane);
    group_sync(group);
  }

  // All of a lane's pass-2 chunks are summed: find the token.
  __device__ __noinline__ void finish_draw(int b, DrawDesc d, const DrawCoef& kc, const uint8_t* trow, const uint8_t* qrow,
                              int group, int gw, int lane) {
    GroupScratch& gs = sh.grp[group];
    const int off = __ldg(p.row_offsets + b);
    const int nc = p.nchunk2;
    const DrawPartS* src = part2 + static_cast<int64_t>(b) * nc;
    // Warp 0: per-lane sums over runs of chunks, then an inclusive scan in lane
    // order; the crossing chunk and the remainder inside it.
    if (gw == 0) {
      const int per = (nc + 31) / 32;
      const int c0 = min(nc, lane * per), c1 = min(nc, c0 + per);
      float run = 0.f;
      int lastpos = -1;
      for (int ch = c0; ch < c1; ++ch) {
        const float2 v = __ldcg(reinterpret_cast<const float2*>(src + ch));
        run = __fadd_rn(run, v.x);
        if (v.x > 0.f) lastpos = max(lastpos, __float_as_int(v.y));
      }
      float incl = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float up = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl = __fadd_rn(up, incl);
      }
      const float W = __shfl_sync(0xFFFFFFFFu, incl, 31);
      const int lastall = warp_max_int(lastpos);
      int chunk = -1;
      float tau = 0.f;
      if (W > 0.f) {
        const float target = __fmul_rn(d.u, W);
        const uint32_t hit = __ballot_sync(0xFFFFFFFFu, incl > target);
        if (hit) {
          const int l = __ffs(hit) - 1;
          float excl = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
          if (lane == 0) excl = 0.f;
          excl = __shfl_sync(0xFFFFFFFFu, excl, l);
          if (lane == l) {
            // The lane's own running sum, offset by the lanes before it exactly
            // as the scan did: its last value gives incl, which is > target,
            // and fl(excl + r) never decreases, so a chunk is always found.
            float r = 0.f;
            for (int ch = c0; ch < c1; ++ch) {
              const float2 v = __ldcg(reinterpret_cast<const float2*>(src + ch));
              const float rn = __fadd_rn(r, v.x);
              if (__fadd_rn(excl, rn) > target) {
                chunk = ch;
                tau = __fsub_rn(target, __fadd_rn(excl, r));
                break;
              }
              r = rn;
            }
          }
          chunk = __shfl_sync(0xFFFFFFFFu, chunk, l);
          tau = __shfl_sync(0xFFFFFFFFu, tau, l);
        }
      }
      if (lane == 0) {
        gs.bcast[2] = chunk;
        gs.bcast[3] = lastall;
        gs.fbcast[0] = tau;
        gs.fbcast[1] = W;
      }
    }
    group_sync(group);
    const int chunk = gs.bcast[2];
    const float W = gs.fbcast[1];
    if (W == 0.f && d.mode == kModeResidual) {
      // The residual has no mass: draw from p_n instead (a second pass 2).
      if (gw == 0 && lane == 0) {
        if (p.row_stats) p.row_stats[off + d.n].resid_mass = 0.f;
        desc[b].mode = kModeFromP;
        st_relaxed(cnt2 + b, 0u);
        publish_draw(b);
      }
      return;
    }
    int token = -1;
    int writer = 0;  // the warp of the group that writes the token
    if (chunk < 0) {
      token = gs.bcast[3];  // rounding left no crossing: the largest index of positive weight
    } else {
      // Re-walk the crossing chunk with the sums of the item that summed it.
      const float tau = gs.fbcast[0];
      int last = -1;
      float rs[kDrawSeg / kDrawRound];
      const float w = seg_sum(kc, trow, qrow, chunk, gw, lane, last, rs);
      last = warp_max_int(last);
      if (lane == 0) {
        gs.segw[gw] = w;
        gs.segl[gw] = last;
      }
      group_sync(group);
      int wsel = -1;
      float q = 0.f;
      for (int x = 0; x < kGroupWarpsS; ++x) {
        const float nx = __fadd_rn(q, gs.segw[x]);
        if (nx > tau) {
          wsel = x;
          break;
        }
        q = nx;
      }
      if (wsel < 0) {
        int lc = -1;
        for (int x = 0; x < kGroupWarpsS; ++x) lc = max(lc, gs.segl[x]);
        token = lc;
      } else {
        writer = wsel;
        if (gw == wsel) {
          const float tau1 = __fsub_rn(tau, q);
          const int s0 = chunk * kDrawChunkS + gw * kDrawSeg;
          const int s1 = min(p.V, s0 + kDrawSeg);
          float run = 0.f;
          int found = -1;
          for (int u = 0; u < kDrawSeg / kDrawRound && found < 0; ++u) {
            const int base = s0 + u * kDrawRound;
            if (base >= s1) break;
            const float nx = __fadd_rn(run, rs[u]);
            if (nx > tau1) {
              Raw8<T> rt, rq;
              const int e = base + lane * 8;
              load_raw8<T, true>(trow, e, s1, rt);
              if (kc.residual) load_raw8<T, true>(qrow, e, s1, rq);
              float wv[8], cum[8];
              draw_piece<T>(kc, rt, rq, e, s1, wv, cum);
              const float tau2 = __fsub_rn(tau1, run);
              float incl = cum[7];
#pragma unroll
              for (int o = 1; o < 32; o <<= 1) {
                const float up = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl = __fadd_rn(up, incl);
              }
              float excl = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
              if (lane == 0) excl = 0.f;
              const uint32_t hit = __ballot_sync(0xFFFFFFFFu, incl > tau2);
              int tok = -1;
              if (hit) {
                const int l = __ffs(hit) - 1;
                if (lane == l) {
                  const float tau3 = __fsub_rn(tau2, excl);
                  int t = -1, lp = -1;
#pragma unroll
                  for (int i = 0; i < 8; ++i) {
                    if (wv[i] > 0.f) lp = e + i;
                    if (t < 0 && cum[i] > tau3) t = e + i;
                  }
                  tok = (t >= 0) ? t : lp;
                }
                tok = __shfl_sync(0xFFFFFFFFu, tok, l);
              } else {
                int lp = -1;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  if (wv[i] > 0.f) lp = e + i;
                tok = warp_max_int(lp);
              }
              found = tok;
            }
            run = nx;
          }
          if (found < 0) found = gs.segl[gw];
          token = found;
        }
      }
    }
    if (gw == writer && lane == 0) {
      p.out_tokens[off + d.n] = token;
      if (p.row_stats) {
        p.row_stats[off + d.n].drawn = token;
        if (d.mode == kModeResidual) p.row_stats[off + d.n].resid_mass = W;
      }
      st_relaxed(cnt2 + b, 0u);
      __threadfence();
      atomicAdd(&hdr->lanes_done, 1u);
    }
  }

  // ---------------------------------------------------------------------
  // Consumer group loop
  // ---------------------------------------------------------------------
  __device__ void consumer(int group, int gw, int lane) {
    GroupScratch& gs = sh.grp[group];
    const uint32_t ns = static_cast<uint32_t>(p.nslots);
    uint32_t slot = static_cast<uint32_t>(group), par = 0;
    if (gw == 0 && lane == 0) sh.group_fail[group] = 0u;
    group_sync(group);
    for (;;) {
      // Every warp of the group agrees on whether the slot arrived: a wait
      // that gives up (a copy that never lands) ends the group's work.
      const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&sh.full[slot], par));
      if (!ok && lane == 0) {
        sh.group_fail[group] = 1u;
        sh.broken = 1u;
        atomicOr(&hdr->error, 1u);
      }
      group_sync(group);
      if (sh.group_fail[group]) return;
      const SlotItem it = sh.item[slot];
      if (it.kind == kItemStop) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.empty[slot]);
        return;
      }
      if (it.kind == kItemP1) {
        const bool timed_out = it.bulk < -1;
        reduce_chunk(it, reinterpret_cast<const uint4*>(ring + static_cast<size_t>(slot) * p.slot_bytes), gw, lane,
                     group, timed_out);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.empty[slot]);
        group_sync(group);
        if (gw == 0) {
          const Partial q = group_partial(it, group, lane);
          int fin = 0;
          if (lane == 0) {
            store_partial(part1 + sh.lane_item[it.lane] + static_cast<int64_t>(it.s) * p.nchunk + it.chunk, q);
            __threadfence();
            const uint32_t need = static_cast<uint32_t>(sh.lane_item[it.lane + 1] - sh.lane_item[it.lane]);
            const uint32_t old = atom_add_acq_rel(cnt1 + it.lane, 1u);
            fin = (old + 1 == need) ? 1 : 0;
            gs.bcast[0] = fin;
          }
        }
        group_sync(group);
        if (gs.bcast[0]) finish_lane(it.lane, group, gw, lane);
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.empty[slot]);
        if (it.kind == kItemStatus) {
          finish_lane(it.lane, group, gw, lane);
        } else {
          pass2_item(it, group, gw, lane);
        }
      }
      slot += kGroupsS;
      if (slot >= ns) {
        slot -= ns;
        par ^= 1u;
      }
    }
  }

  // The last CTA out resets the shared counters (and after an error marks
  // every lane as timed out and clears every lane's counters).
  __device__ void exit_protocol() {
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const uint32_t old = atom_add_acq_rel(&hdr->exited, 1u);
      sh.exit_last = (old + 1 == gridDim.x) ? 1u : 0u;
    }
    __syncthreads();
    if (!sh.exit_last) return;
    const bool err = ld_acquire(&hdr->error) != 0u || ld_relaxed(&hdr->lanes_done) != static_cast<uint32_t>(p.lanes);
    const uint32_t res = ld_relaxed(&hdr->p2_reserved);
    for (uint32_t i = threadIdx.x; i < res && i < 2u * static_cast<uint32_t>(p.lanes); i += blockDim.x) ready[i] = 0u;
    if (err) {
      for (int b = threadIdx.x; b < p.lanes; b += blockDim.x) {
        cnt1[b] = 0u;
        cnt2[b] = 0u;
        p.committed[b] = 0;
        if (p.lane_status) p.lane_status[b] = SPEC_ERR_TIMEOUT;
        const int k = __ldg(p.draft_lens + b), off = __ldg(p.row_offsets + b), end = __ldg(p.row_offsets + b + 1);
        if (k >= 0 && off >= 0 && end <= p.rows && end - off == k + 1)
          for (int j = 0; j <= k; ++j) p.out_tokens[off + j] = -1;
      }
    }
    if (threadIdx.x == 0) {
      hdr->p1_claim = 0u;
      hdr->p2_claim = 0u;
      hdr->p2_reserved = 0u;
      hdr->lanes_done = 0u;
      hdr->error = 0u;
      hdr->exited = 0u;
    }
  }
};

template <typename T>
__global__ void __launch_bounds__(kThreadsS, 1) verify_split_kernel(const SplitParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SplitSmem& sh = *reinterpret_cast<SplitSmem*>(smem_raw);
  SplitKernel<T> K(p, sh, smem_raw + p.head_bytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid < p.nslots) {
    mbar_init(&sh.full[tid], 1);
    mbar_init(&sh.empty[tid], kGroupWarpsS);
    fence_mbar_init();
  }
  if (tid == 0) sh.broken = 0u;
  const bool meta_early = (p.flags & SPEC_VERIFY_META_BEFORE_WAIT) != 0u;
  if (!meta_early) griddep_wait();
  K.build_item_prefix();  // ends with a CTA barrier (barrier initialisation visible too)
  if (meta_early) griddep_wait();  // the workspace and the logits only after the previous kernel
  if (tid == 0) griddep_launch_dependents();

  if (warp == kProducerWarpS) {
    if (lane < kGroupsS) K.producer(lane);
  } else {
    K.consumer(warp / kGroupWarpsS, warp % kGroupWarpsS, lane);
  }
  K.exit_protocol();
}

}  // namespace specv_split_impl
