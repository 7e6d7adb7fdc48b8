// verify_kernel.cuh -- the fused verify-accept kernel.
//
// One thread-block cluster per lane.  Each CTA of the cluster owns a contiguous
// slice of the vocabulary and reduces that slice of every row the lane needs:
// the k_b + 1 target rows and, on a sampled lane, the k_b drafter rows
// (ignis docs, "Speculative decoding" -- "One round, step by step", steps 3-4).
//
//   pass 1   a producer thread streams the slices through a shared-memory ring
//            with bulk (TMA) copies; eight consumer warps keep, per thread, the
//            running argmax (lowest index on ties) and, for sampled lanes, the
//            online max / sum of 2^((x - max) * log2(e) / T)
//   reduce   warp shuffles -> per-CTA partial per row -> pushed into every CTA
//            of the cluster through distributed shared memory
//   scan     every CTA finishes the per-row reductions and runs the lane's
//            acceptance scan (<= 15 drafts, one lane of warp 0 per position)
//   pass 2   sampled lanes only: the cluster re-reads one target row (and one
//            drafter row) from L2, sums the draw weights per slice, exchanges the
//            sums, and the CTA whose slice holds u' * W walks it to the token
//
// Greedy lanes compare raw logits only, so their results are exact.  Sampled
// lanes use fp32 with the hardware exp2; the acceptance test is done in the
// log2 domain: accept iff log2(u) < log2 p(d) - log2 q(d).
#pragma once

#include <cfloat>
#include <cstdint>

#include "device_ptx.cuh"
#include "philox.cuh"
#include "spec_verify.h"

namespace specv {

constexpr int kMaxDrafts = SPEC_MAX_DRAFTS;      // 15
constexpr int kMaxStreams = 2 * kMaxDrafts + 1;  // target rows + drafter rows of one lane
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kMaxCluster = 16;
constexpr int kMaxSlots = 16;
constexpr int kDrawRound = 256;  // elements per warp per pass-2 round (32 lanes x 8)

constexpr float kLog2e = 1.4426950408889634f;
constexpr double kLn2d = 0.6931471805599453;

// Partial reduction of one row over some elements (16 bytes, pushed over DSMEM).
struct __align__(16) Partial {
  float m;         // largest logit seen (-inf if none)
  float s;         // sum of 2^((x - m) * c) over the elements (sampled rows)
  int idx;         // lowest index holding m (INT_MAX if none)
  uint32_t flags;  // kBadValue | kTimedOut
};

constexpr uint32_t kBadValue = 1u;  // NaN or +inf in the row
constexpr uint32_t kTimedOut = 2u;  // a bounded wait gave up

struct __align__(16) DrawPartial {
  float w;     // sum of draw weights over one CTA's slice
  int last;    // largest index of positive weight in the slice (-1 if none)
  int pad0, pad1;
};

enum DrawMode : int { kNoDraw = 0, kResidual = 1, kBonus = 2 };

struct __align__(16) SmemHead {
  uint64_t full[kMaxSlots];
  uint64_t empty[kMaxSlots];
  Partial wpart[kMaxStreams][kConsumerWarps];  // per consumer warp
  Partial cpart[kMaxCluster][kMaxStreams];     // per CTA of the cluster (pushed by peers)
  Partial fin[kMaxStreams];                    // this CTA's partial, then the lane's total
  DrawPartial dpart[2][kMaxCluster];           // pass-2 slice sums (pushed by peers)
  float segsum[kConsumerWarps];
  int seglast[kConsumerWarps];
  int drafts[kMaxDrafts + 1];
  float xd_t[kMaxDrafts + 1];  // target logit at d_{j+1} in row j
  float xd_q[kMaxDrafts + 1];  // drafter logit at d_{j+1} in row j
  int scan_n;
  int scan_mode;
  float scan_u;
  uint32_t cta_flags;
};

struct VerifyParams {
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
  int32_t cluster;     // CTAs per lane
  int32_t slice;       // vocabulary elements per CTA (multiple of the vector width)
  int32_t slot_bytes;  // bytes per ring slot (multiple of 16)
  int32_t nslots;
  int32_t head_bytes;  // offset of the ring in dynamic shared memory
};

// ---------------------------------------------------------------------------
// Element access
// ---------------------------------------------------------------------------
template <typename T>
struct ElemTraits;

template <>
struct ElemTraits<float> {
  static constexpr int kVec = 4;  // elements per 16 bytes
  static __device__ __forceinline__ float load(const uint8_t* row, int e) {
    return __ldg(reinterpret_cast<const float*>(row) + e);
  }
};

struct bf16_tag {};

template <>
struct ElemTraits<bf16_tag> {
  static constexpr int kVec = 8;
  static __device__ __forceinline__ float load(const uint8_t* row, int e) {
    const uint32_t bits = __ldg(reinterpret_cast<const unsigned short*>(row) + e);
    return __uint_as_float(bits << 16);
  }
};

// ---------------------------------------------------------------------------
// Running reduction state of one thread for one row
// ---------------------------------------------------------------------------
struct Acc {
  float m;
  float s;
  int idx;
  uint32_t bad;   // fp32 rows: NaN / +inf seen
  uint32_t nan2;  // bf16 rows: packed max with NaN propagation over everything seen
};

__device__ __forceinline__ void acc_init(Acc& a) {
  a.m = -INFINITY;
  a.s = 0.f;
  a.idx = INT_MAX;
  a.bad = 0;
  a.nan2 = 0xFF80FF80u;  // (-inf, -inf)
}

// Merge (m2, s2, i2) into (m, s, idx): max, rescaled sum, lowest index of the max.
template <bool SAMPLED>
__device__ __forceinline__ void merge_part(float& m, float& s, int& idx, float m2, float s2, int i2,
                                           float c) {
  const float nm = fmaxf(m, m2);
  if (SAMPLED) {
    if (nm == -INFINITY) {
      s = s + s2;
    } else {
      s = s * ex2_approx((m - nm) * c) + s2 * ex2_approx((m2 - nm) * c);
    }
  }
  if (m2 > m || (m2 == m && i2 < idx)) idx = i2;
  m = nm;
}

// A new running max `vm` first seen at element `e`: rescale the sum.
template <bool SAMPLED>
__device__ __forceinline__ void acc_raise(Acc& a, float vm, int e, float c) {
  if (SAMPLED) a.s *= ex2_approx((a.m - vm) * c);
  a.m = vm;
  a.idx = e;
}

__device__ __forceinline__ float exp_term(float x, float mm, float c) {
  return ex2_approx((x - mm) * c);
}

// 8 bf16 logits starting at element e0.
template <bool SAMPLED>
__device__ __forceinline__ void acc_bf16x8(Acc& a, const uint4 v, int e0, float c) {
  const uint32_t h = bf16x2_max_nan(bf16x2_max_nan(v.x, v.y), bf16x2_max_nan(v.z, v.w));
  a.nan2 = bf16x2_max_nan(a.nan2, h);
  const float vm = fmaxf(bf16_lo(h), bf16_hi(h));
  if (vm > a.m) {
    const float x[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                        bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
    int i = 0;
#pragma unroll
    for (int t = 7; t >= 0; --t)
      if (x[t] == vm) i = t;
    acc_raise<SAMPLED>(a, vm, e0 + i, c);
  }
  if (SAMPLED) {
    const float mm = (a.m == -INFINITY) ? 0.f : a.m;
    const float e01 = exp_term(bf16_lo(v.x), mm, c) + exp_term(bf16_hi(v.x), mm, c);
    const float e23 = exp_term(bf16_lo(v.y), mm, c) + exp_term(bf16_hi(v.y), mm, c);
    const float e45 = exp_term(bf16_lo(v.z), mm, c) + exp_term(bf16_hi(v.z), mm, c);
    const float e67 = exp_term(bf16_lo(v.w), mm, c) + exp_term(bf16_hi(v.w), mm, c);
    a.s += (e01 + e23) + (e45 + e67);
  }
}

// 4 fp32 logits starting at element e0.
template <bool SAMPLED>
__device__ __forceinline__ void acc_f32x4(Acc& a, const uint4 v, int e0, float c) {
  const float x[4] = {__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                      __uint_as_float(v.w)};
#pragma unroll
  for (int t = 0; t < 4; ++t) a.bad |= !(x[t] <= FLT_MAX);
  const float vm = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
  if (vm > a.m) {
    int i = 0;
#pragma unroll
    for (int t = 3; t >= 0; --t)
      if (x[t] == vm) i = t;
    acc_raise<SAMPLED>(a, vm, e0 + i, c);
  }
  if (SAMPLED) {
    const float mm = (a.m == -INFINITY) ? 0.f : a.m;
    a.s += (exp_term(x[0], mm, c) + exp_term(x[1], mm, c)) +
           (exp_term(x[2], mm, c) + exp_term(x[3], mm, c));
  }
}

// One logit (row tails and unaligned rows).
template <bool SAMPLED>
__device__ __forceinline__ void acc_scalar(Acc& a, float x, int e, float c) {
  a.bad |= !(x <= FLT_MAX);
  if (x > a.m) acc_raise<SAMPLED>(a, x, e, c);
  if (SAMPLED) {
    const float mm = (a.m == -INFINITY) ? 0.f : a.m;
    a.s += exp_term(x, mm, c);
  }
}

template <typename T, bool SAMPLED>
__device__ __forceinline__ void acc_vec(Acc& a, const uint4 v, int e0, float c) {
  if constexpr (ElemTraits<T>::kVec == 8) {
    acc_bf16x8<SAMPLED>(a, v, e0, c);
  } else {
    acc_f32x4<SAMPLED>(a, v, e0, c);
  }
}

__device__ __forceinline__ uint32_t acc_bad(const Acc& a) {
  const float lo = bf16_lo(a.nan2), hi = bf16_hi(a.nan2);
  const bool packed_bad = (lo != lo) || (hi != hi) || lo == INFINITY || hi == INFINITY;
  return (a.bad || packed_bad) ? kBadValue : 0u;
}

// Warp-wide merge; every lane ends with the warp's partial.
template <bool SAMPLED>
__device__ __forceinline__ Partial warp_merge(float m, float s, int idx, uint32_t flags, float c) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
    const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o);
    const int i2 = __shfl_xor_sync(0xFFFFFFFFu, idx, o);
    flags |= __shfl_xor_sync(0xFFFFFFFFu, flags, o);
    merge_part<SAMPLED>(m, s, idx, m2, s2, i2, c);
  }
  return Partial{m, s, idx, flags};
}

__device__ __forceinline__ Partial identity_partial() { return Partial{-INFINITY, 0.f, INT_MAX, 0u}; }

// ---------------------------------------------------------------------------
// Pass-2 draw weights
// ---------------------------------------------------------------------------
struct DrawCoef {
  float mp, l2sp;  // target row: max and log2 of its sum
  float mq, l2sq;  // drafter row (residual only)
  float c;         // log2(e) / T
  bool residual;
};

// Normalised probability 2^((x - m) * c - log2 S), evaluated with explicit
// roundings so that both call sites produce identical bits.
__device__ __forceinline__ float prob_at(float x, float m, float l2s, float c) {
  return ex2_approx(__fmaf_rn(__fsub_rn(x, m), c, -l2s));
}

__device__ __forceinline__ float draw_weight(const DrawCoef& k, float xt, float xq) {
  const float p = prob_at(xt, k.mp, k.l2sp, k.c);
  if (!k.residual) return p;
  const float q = prob_at(xq, k.mq, k.l2sq, k.c);
  return fmaxf(0.f, __fsub_rn(p, q));
}

// Eight consecutive logits of a row from element e (values past `end` read as -inf).
template <typename T, bool ALIGNED>
__device__ __forceinline__ void load8(const uint8_t* row, int e, int end, float (&x)[8]) {
  if (ALIGNED && e + 8 <= end) {
    if constexpr (ElemTraits<T>::kVec == 8) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(row + static_cast<int64_t>(e) * 2));
      x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
      x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z); x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
    } else {
      const uint4* p = reinterpret_cast<const uint4*>(row + static_cast<int64_t>(e) * 4);
      const uint4 v0 = __ldg(p), v1 = __ldg(p + 1);
      x[0] = __uint_as_float(v0.x); x[1] = __uint_as_float(v0.y);
      x[2] = __uint_as_float(v0.z); x[3] = __uint_as_float(v0.w);
      x[4] = __uint_as_float(v1.x); x[5] = __uint_as_float(v1.y);
      x[6] = __uint_as_float(v1.z); x[7] = __uint_as_float(v1.w);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = (e + i < end) ? ElemTraits<T>::load(row, e + i) : -INFINITY;
  }
}

// The eight draw weights of one lane's piece of a pass-2 round, and their
// running sums in element order (cum[7] is the piece's total).
template <typename T, bool ALIGNED>
__device__ __forceinline__ void draw_piece(const DrawCoef& k, const uint8_t* trow,
                                           const uint8_t* qrow, int e, int end, float (&w)[8],
                                           float (&cum)[8]) {
  float xt[8], xq[8];
  load8<T, ALIGNED>(trow, e, end, xt);
  if (k.residual) {
    load8<T, ALIGNED>(qrow, e, end, xq);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) xq[i] = -INFINITY;
  }
  float run = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    w[i] = (e + i < end) ? draw_weight(k, xt[i], xq[i]) : 0.f;
    run = __fadd_rn(run, w[i]);
    cum[i] = run;
  }
}

__device__ __forceinline__ float warp_sum_xor(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

__device__ __forceinline__ int warp_max_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <typename T, bool ALIGNED>
__global__ void __launch_bounds__(kThreads, 2) verify_accept_kernel(const VerifyParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SmemHead& sh = *reinterpret_cast<SmemHead*>(smem_raw);
  uint8_t* ring = smem_raw + p.head_bytes;

  constexpr int kVec = ElemTraits<T>::kVec;
  constexpr int kEsize = 16 / kVec;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int C = p.cluster;
  const uint32_t rank = cluster_ctarank();
  const int b = blockIdx.x / C;

  // ---- set-up that touches only shared memory (overlaps the previous kernel) ----
  if (tid == 0) {
    for (int s = 0; s < p.nslots; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], kConsumerWarps);
    }
    sh.cta_flags = 0;
    fence_mbar_init();
  }
  // Phase A of the cluster barrier: every CTA of the cluster has started.  It is
  // waited on just before the first write into a peer's shared memory.
  cluster_arrive_relaxed();
  griddep_wait();

  // ---- lane metadata (read by every thread; one transaction per warp) ----
  const int k = __ldg(p.draft_lens + b);
  const int off = __ldg(p.row_offsets + b);
  const int off_end = __ldg(p.row_offsets + b + 1);
  const float temp = __ldg(p.temps + b);
  const bool sampled = temp > 0.f;
  int status = SPEC_OK;
  if (k < 0 || off < 0 || off_end > p.rows || off_end - off != k + 1) {
    status = SPEC_ERR_LAYOUT;
  } else if (k > kMaxDrafts) {
    status = SPEC_ERR_UNSUPPORTED;
  } else if (sampled && p.draft == nullptr) {
    status = SPEC_ERR_INVALID_ARG;
  }
  const int nstreams = (status != SPEC_OK) ? 0 : (sampled ? 2 * k + 1 : k + 1);
  const float c = sampled ? __fdiv_rn(kLog2e, temp) : 0.f;

  const int v0 = min(p.V, static_cast<int>(rank) * p.slice);
  const int v1 = min(p.V, v0 + p.slice);
  const int span = v1 - v0;
  const int body = ALIGNED ? (span / kVec) * kVec : 0;
  const int slot_elems = p.slot_bytes / kEsize;

  __syncthreads();  // barrier initialisation visible to every thread

  // Row of stream s: sampled lanes interleave target row j (even s) and drafter
  // row j (odd s); greedy lanes read target rows only.
  auto stream_row = [&](int s) -> const uint8_t* {
    const bool is_draft = sampled && (s & 1);
    const int j = sampled ? (s >> 1) : s;
    return (is_draft ? p.draft : p.target) + static_cast<int64_t>(off + j) * p.ld_bytes;
  };

  // ---- pass 1 ----
  if (warp == kConsumerWarps) {
    // Producer warp.  Lane 0 streams the slices; lanes 1.. fetch the draft tokens
    // and, for sampled lanes, the logits at the draft tokens.
    if (lane == 0) {
      if (ALIGNED) {
        uint32_t it = 0;
        bool ok = true;
        for (int s = 0; s < nstreams && ok; ++s) {
          const uint8_t* row = stream_row(s) + static_cast<int64_t>(v0) * kEsize;
          for (int c0 = 0; c0 < body; c0 += slot_elems) {
            const int L = min(slot_elems, body - c0);
            const uint32_t slot = it % p.nslots;
            const uint32_t par = (it / p.nslots) & 1u;
            if (!mbar_wait_bounded(&sh.empty[slot], par ^ 1u)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&sh.full[slot], static_cast<uint32_t>(L * kEsize));
            bulk_g2s(ring + static_cast<size_t>(slot) * p.slot_bytes, row + static_cast<int64_t>(c0) * kEsize,
                     static_cast<uint32_t>(L * kEsize), &sh.full[slot]);
            ++it;
          }
        }
        // Drain: every copy issued has landed before shared memory is reused.
        const uint32_t first = it > static_cast<uint32_t>(p.nslots) ? it - p.nslots : 0u;
        for (uint32_t i = first; i < it; ++i)
          if (!mbar_wait_bounded(&sh.full[i % p.nslots], (i / p.nslots) & 1u)) ok = false;
        if (!ok) atomicOr(&sh.cta_flags, kTimedOut);
      }
    } else if (lane - 1 < k && status == SPEC_OK) {
      const int j = lane - 1;
      const int d = __ldg(p.draft_tokens + off + j);
      sh.drafts[j] = d;
      if (sampled && d >= 0 && d < p.V) {
        sh.xd_t[j] = ElemTraits<T>::load(p.target + static_cast<int64_t>(off + j) * p.ld_bytes, d);
        sh.xd_q[j] = ElemTraits<T>::load(p.draft + static_cast<int64_t>(off + j) * p.ld_bytes, d);
      }
    }
  } else {
    // Consumer warps.
    uint32_t it = 0;
    bool ok = true;
    for (int s = 0; s < nstreams; ++s) {
      Acc a;
      acc_init(a);
      const uint8_t* row = stream_row(s);
      if (ALIGNED) {
        for (int c0 = 0; c0 < body && ok; c0 += slot_elems) {
          const int L = min(slot_elems, body - c0);
          const uint32_t slot = it % p.nslots;
          const uint32_t par = (it / p.nslots) & 1u;
          if (!mbar_wait_bounded(&sh.full[slot], par)) {
            ok = false;
            break;
          }
          const uint4* sv = reinterpret_cast<const uint4*>(ring + static_cast<size_t>(slot) * p.slot_bytes);
          const int nvec = L / kVec;
          const int ebase = v0 + c0;
          if (sampled) {
#pragma unroll 4
            for (int v = tid; v < nvec; v += kConsumers) acc_vec<T, true>(a, sv[v], ebase + v * kVec, c);
          } else {
#pragma unroll 4
            for (int v = tid; v < nvec; v += kConsumers) acc_vec<T, false>(a, sv[v], ebase + v * kVec, c);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.empty[slot]);
          ++it;
        }
      }
      // Elements outside the bulk-copied body: the row tail, or the whole slice
      // when rows are not 16-byte aligned.
      for (int e = body + tid; e < span && ok; e += kConsumers) {
        const float x = ElemTraits<T>::load(row, v0 + e);
        if (sampled) acc_scalar<true>(a, x, v0 + e, c);
        else acc_scalar<false>(a, x, v0 + e, c);
      }
      const uint32_t fl = acc_bad(a) | (ok ? 0u : kTimedOut);
      const Partial wp = sampled ? warp_merge<true>(a.m, a.s, a.idx, fl, c)
                                 : warp_merge<false>(a.m, a.s, a.idx, fl, c);
      if (lane == 0) sh.wpart[s][warp] = wp;
    }
    if (!ok && lane == 0) atomicOr(&sh.cta_flags, kTimedOut);
  }
  __syncthreads();
  griddep_launch_dependents();

  // ---- CTA partial of every row -> pushed to every CTA of the cluster ----
  if (warp < kConsumerWarps) {
    for (int s = warp; s < nstreams; s += kConsumerWarps) {
      const Partial q = (lane < kConsumerWarps) ? sh.wpart[s][lane] : identity_partial();
      const Partial r = sampled ? warp_merge<true>(q.m, q.s, q.idx, q.flags, c)
                                : warp_merge<false>(q.m, q.s, q.idx, q.flags, c);
      if (lane == 0) sh.fin[s] = r;
    }
  }
  __syncthreads();
  cluster_wait_acquire();  // phase A: all peers are running
  {
    const uint32_t extra = sh.cta_flags;
    for (int t = tid; t < nstreams * C; t += kThreads) {
      const int s = t / C, dst = t % C;
      const Partial q = sh.fin[s];
      st_cluster_v4(cluster_map(&sh.cpart[rank][s], dst), __float_as_uint(q.m), __float_as_uint(q.s),
                    static_cast<uint32_t>(q.idx), q.flags | extra);
    }
  }
  cluster_arrive_release();
  cluster_wait_acquire();  // phase B: every partial has arrived

  const bool leader = (rank == 0);
  if (!sampled && !leader) return;  // greedy lanes: only the leader finishes

  // ---- the lane's totals ----
  if (warp < kConsumerWarps) {
    for (int s = warp; s < nstreams; s += kConsumerWarps) {
      const Partial q = (lane < C) ? sh.cpart[lane][s] : identity_partial();
      const Partial r = sampled ? warp_merge<true>(q.m, q.s, q.idx, q.flags, c)
                                : warp_merge<false>(q.m, q.s, q.idx, q.flags, c);
      if (lane == 0) sh.fin[s] = r;
    }
  }
  __syncthreads();

  // ---- acceptance scan (warp 0; lane j handles position j) ----
  if (warp == 0) {
    int st = status;
    if (st == SPEC_OK) {
      bool range_bad = false;
      if (lane < k) {
        const int d = sh.drafts[lane];
        range_bad = (d < 0 || d >= p.V);
      }
      if (__any_sync(0xFFFFFFFFu, range_bad)) st = SPEC_ERR_TOKEN_RANGE;
    }
    if (st == SPEC_OK) {
      uint32_t fl = 0;
      bool empty_row = false;
      for (int s = lane; s < nstreams; s += 32) {
        fl |= sh.fin[s].flags;
        empty_row |= (sh.fin[s].idx == INT_MAX);
      }
      fl |= sh.cta_flags;
      const uint32_t all = __reduce_or_sync(0xFFFFFFFFu, fl);
      const bool any_empty = __any_sync(0xFFFFFFFFu, empty_row);
      if (all & kTimedOut) st = SPEC_ERR_TIMEOUT;
      else if ((all & kBadValue) || any_empty) st = SPEC_ERR_NONFINITE;
    }

    int n = 0, mode = kNoDraw;
    float uprime = 0.f;
    // log2 p_j(d), log2 q_j(d) at this lane's position.  The scan touches at most
    // 15 positions, so it runs in fp64: the only fp32 inputs are the row maxima,
    // the sums S and the logits themselves.
    double lp = NAN, lq = NAN;
    const double c64 = sampled ? 1.4426950408889634 / static_cast<double>(temp) : 0.0;
    if (st == SPEC_OK) {
      const bool active = lane < k;
      bool stop;
      if (!sampled) {
        const int a = (lane <= k) ? sh.fin[lane].idx : 0;
        stop = active && (sh.drafts[lane] != a);
      } else {
        bool accept = true;
        if (active) {
          const Partial pt = sh.fin[2 * lane], pq = sh.fin[2 * lane + 1];
          lp = (static_cast<double>(sh.xd_t[lane]) - pt.m) * c64 - log2(static_cast<double>(pt.s));
          lq = (static_cast<double>(sh.xd_q[lane]) - pq.m) * c64 - log2(static_cast<double>(pq.s));
          const float u = round_uniforms(p.seed, b, lane).x;
          if (lp == -INFINITY) accept = false;
          else if (lq == -INFINITY) accept = true;
          else accept = log2(static_cast<double>(u)) < lp - lq;
        }
        stop = active && !accept;
      }
      const uint32_t mask = __ballot_sync(0xFFFFFFFFu, stop);
      n = mask ? (__ffs(mask) - 1) : k;
      if (sampled) {
        mode = (n < k) ? kResidual : kBonus;
        float u2 = 0.f;
        if (lane <= k) u2 = round_uniforms(p.seed, b, lane).y;
        uprime = __shfl_sync(0xFFFFFFFFu, u2, n);
      }
    }
    if (lane == 0) {
      sh.scan_n = n;
      sh.scan_mode = (st == SPEC_OK) ? mode : kNoDraw;
      sh.scan_u = uprime;
    }

    // ---- outputs (leader) ----
    if (leader) {
      const bool layout_ok = (status != SPEC_ERR_LAYOUT);
      if (lane == 0) {
        p.committed[b] = (st == SPEC_OK) ? n + 1 : 0;
        if (p.lane_status) p.lane_status[b] = st;
      }
      for (int j = lane; layout_ok && j <= k; j += 32) {
        int tok = -1;
        if (st == SPEC_OK) {
          if (!sampled) tok = (j <= n) ? sh.fin[j].idx : -1;
          else tok = (j < n) ? sh.drafts[j] : -1;
        }
        const bool drawn_here = (st == SPEC_OK) && sampled && j == n;
        if (!drawn_here) p.out_tokens[off + j] = tok;
        if (p.row_stats && st == SPEC_OK) {
          spec_row_stats* rs = p.row_stats + off + j;
          const Partial pt = sh.fin[sampled ? 2 * j : j];
          rs->argmax = pt.idx;
          rs->max_logit = pt.m;
          if (sampled) {
            rs->lse = static_cast<float>(static_cast<double>(pt.m) / temp + log(static_cast<double>(pt.s)));
            rs->logp_d = (j < k) ? static_cast<float>(lp * kLn2d) : NAN;
            rs->logq_d = (j < k) ? static_cast<float>(lq * kLn2d) : NAN;
          } else {
            rs->lse = NAN;
            rs->logp_d = NAN;
            rs->logq_d = NAN;
          }
          if (!(drawn_here && mode == kResidual)) rs->resid_mass = NAN;
          if (!drawn_here) rs->drawn = -1;
          rs->flags = 1 | (drawn_here ? (mode == kResidual ? 2 : 4) : 0);
        }
      }
    }
  }
  __syncthreads();

  if (!sampled || sh.scan_mode == kNoDraw) return;

  // ---- pass 2: draw the model's token (sampled lanes, whole cluster) ----
  const int n = sh.scan_n;
  bool residual = (sh.scan_mode == kResidual);
  int draw_row = residual ? n : k;  // target row whose p enters the weights
  const uint8_t* qrow = p.draft + static_cast<int64_t>(off + n) * p.ld_bytes;
  const float uprime = sh.scan_u;
  const int seg = ((span + kConsumerWarps - 1) / kConsumerWarps + kDrawRound - 1) / kDrawRound * kDrawRound;
  auto make_coef = [&]() {
    DrawCoef kc;
    const Partial pt = sh.fin[2 * draw_row];
    kc.mp = pt.m;
    kc.l2sp = log2f(pt.s);
    kc.c = c;
    kc.residual = residual;
    kc.mq = 0.f;
    kc.l2sq = 0.f;
    if (residual) {
      const Partial pq = sh.fin[2 * n + 1];
      kc.mq = pq.m;
      kc.l2sq = log2f(pq.s);
    }
    return kc;
  };

  float W = 0.f;
  float resid_mass = NAN;
  int buf = 0;
  for (int attempt = 0; attempt < 2; ++attempt) {
    buf = attempt;
    const DrawCoef kc = make_coef();
    const uint8_t* trow = p.target + static_cast<int64_t>(off + draw_row) * p.ld_bytes;
    if (warp < kConsumerWarps) {
      const int s0 = v0 + warp * seg;
      const int s1 = min(v1, s0 + seg);
      float segw = 0.f;
      int last = -1;
      for (int base = s0; base < s1; base += kDrawRound) {
        float w[8], cum[8];
        const int e = base + lane * 8;
        draw_piece<T, ALIGNED>(kc, trow, qrow, e, s1, w, cum);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (w[i] > 0.f) last = e + i;
        segw = __fadd_rn(segw, warp_sum_xor(cum[7]));
      }
      last = warp_max_int(last);
      if (lane == 0) {
        sh.segsum[warp] = segw;
        sh.seglast[warp] = last;
      }
    }
    __syncthreads();
    if (tid < C) {
      float wc = 0.f;
      int lc = -1;
      for (int w = 0; w < kConsumerWarps; ++w) {
        wc = __fadd_rn(wc, sh.segsum[w]);
        lc = max(lc, sh.seglast[w]);
      }
      st_cluster_v2(cluster_map(&sh.dpart[buf][rank], tid), __float_as_uint(wc), static_cast<uint32_t>(lc));
    }
    cluster_arrive_release();
    cluster_wait_acquire();

    W = 0.f;
    for (int r = 0; r < C; ++r) W = __fadd_rn(W, sh.dpart[buf][r].w);
    if (residual) resid_mass = W;
    if (W > 0.f || !residual) break;
    // The residual max(0, p_n - q_n) has no mass: draw from p_n instead.
    residual = false;
    draw_row = n;
    __syncthreads();
  }

  // CTA holding the crossing of u' * W (cumulative sums in CTA order).
  const float target = __fmul_rn(uprime, W);
  int owner = -1;
  float prefix = 0.f;
  for (int r = 0; r < C; ++r) {
    const float next = __fadd_rn(prefix, sh.dpart[buf][r].w);
    if (next > target) {
      owner = r;
      break;
    }
    prefix = next;
  }
  int token = -1;
  bool write = false;
  if (owner < 0) {
    // Rounding left no crossing: the largest index of positive weight.
    int last_r = -1;
    for (int r = 0; r < C; ++r)
      if (sh.dpart[buf][r].w > 0.f) last_r = r;
    if (last_r == static_cast<int>(rank) && tid == 0) {
      token = sh.dpart[buf][rank].last;
      write = true;
    }
  } else if (owner == static_cast<int>(rank)) {
    const float tau = __fsub_rn(target, prefix);
    int wsel = -1;
    float q = 0.f;
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float next = __fadd_rn(q, sh.segsum[w]);
      if (next > tau) {
        wsel = w;
        break;
      }
      q = next;
    }
    if (wsel < 0) {
      if (tid == 0) {
        int lc = -1;
        for (int w = 0; w < kConsumerWarps; ++w) lc = max(lc, sh.seglast[w]);
        token = lc;
        write = true;
      }
    } else if (warp == wsel) {
      const DrawCoef kc = make_coef();
      const uint8_t* trow = p.target + static_cast<int64_t>(off + draw_row) * p.ld_bytes;
      const float tau1 = __fsub_rn(tau, q);
      const int s0 = v0 + warp * seg;
      const int s1 = min(v1, s0 + seg);
      float run = 0.f;
      int found = -1;
      for (int base = s0; base < s1 && found < 0; base += kDrawRound) {
        float w[8], cum[8];
        const int e = base + lane * 8;
        draw_piece<T, ALIGNED>(kc, trow, qrow, e, s1, w, cum);
        const float R = warp_sum_xor(cum[7]);
        const float next = __fadd_rn(run, R);
        if (next > tau1) {
          // The crossing is in this round: inclusive scan over the lanes.
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
              int t = -1, lastpos = -1;
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                if (w[i] > 0.f) lastpos = e + i;
                if (t < 0 && cum[i] > tau3) t = e + i;
              }
              tok = (t >= 0) ? t : lastpos;
            }
            tok = __shfl_sync(0xFFFFFFFFu, tok, l);
          } else {
            int lastpos = -1;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (w[i] > 0.f) lastpos = e + i;
            tok = warp_max_int(lastpos);
          }
          found = tok;
        }
        run = next;
      }
      if (found < 0) found = sh.seglast[warp];
      if (lane == 0) {
        token = found;
        write = true;
      }
    }
  }
  if (write) {
    p.out_tokens[off + n] = token;
    if (p.row_stats) {
      spec_row_stats* rs = p.row_stats + off + n;
      rs->drawn = token;
      if (sh.scan_mode == kResidual) rs->resid_mass = resid_mass;
    }
  }
}

}  // namespace specv
