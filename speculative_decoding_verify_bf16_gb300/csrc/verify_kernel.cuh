// verify_kernel.cuh -- the fused verify-accept kernel.
//
// One thread-block cluster per lane.  Each CTA of the cluster owns a contiguous
// slice of the vocabulary and reduces that slice of every row the lane needs:
// the k_b + 1 target rows and, on a sampled lane, the k_b drafter rows
// (ignis docs, "Speculative decoding" -- "One round, step by step", steps 3-4).
//
//   pass 1   the producer warp streams the slices through a shared-memory
//            ring with bulk (TMA) copies; 16 or 20 consumer warps (per build)
//            take (chunk, piece) items and keep, per lane, the running max and
//            the first vector holding it, and for sampled lanes the sum of
//            2^(x * log2(e) / T - fl(M * log2(e) / T)) against a reference M
//            (the running max, or without row_stats any element at or below it)
//   reduce   greedy rows: one 64-bit key (ordered max, complemented index) per
//            row, combined with shared-memory atomics and sent to the leader
//            CTA; sampled rows: per-warp partials merged per CTA and pushed
//            into every CTA of the cluster through distributed shared memory
//   scan     the leader (greedy) or every CTA (sampled) runs the lane's
//            acceptance scan (<= 15 drafts, one lane of warp 0 per position)
//   pass 2   sampled lanes only: the cluster re-reads one target row (and one
//            drafter row) from L2, sums the draw weights per round and slice,
//            exchanges the sums, and the warp whose segment holds u' * W
//            re-reads the one round that crosses it and walks it to the token
//
// Greedy lanes compare raw logits only, so their results are exact.  Sampled
// lanes use fp32 with the hardware exp2; the acceptance test is done in the
// log2 domain, accept iff log2(u) < log2 p(d) - log2 q(d), as a compensated
// fp32 sum of exactly represented terms.
#pragma once

#include <cfloat>
#include <cstdint>

#include "device_ptx.cuh"
#include "philox.cuh"
#include "spec_verify.h"

namespace specv {

constexpr int kMaxDrafts = SPEC_MAX_DRAFTS;      // 15
constexpr int kMaxStreams = 2 * kMaxDrafts + 1;  // target rows + drafter rows of one lane
// Consumer warps per CTA (16 by default; the 20-warp builds define it before
// including this file).  The CTA occupies a whole SM (one per SM).
#ifndef SPEC_VERIFY_CONSUMER_WARPS
#define SPEC_VERIFY_CONSUMER_WARPS 16
#endif
constexpr int kConsumerWarps = SPEC_VERIFY_CONSUMER_WARPS;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kProducerWarp = kConsumerWarps;    // streams the slices (lane 0)
constexpr int kHelperWarp = kConsumerWarps + 1;  // draft tokens, logits at them, uniforms
constexpr int kThreads = kConsumers + 64;
constexpr int kWarps = kThreads / 32;
constexpr int kCostBuckets = 64;  // lane cost classes for the longest-first lane order
constexpr int kMaxCluster = 16;
constexpr int kMaxSlots = 32;
constexpr int kDrawRound = 256;  // elements per warp per pass-2 round (32 lanes x 8)
#ifndef SPEC_VERIFY_PIECES
#define SPEC_VERIFY_PIECES 4
#endif
constexpr int kPieces = SPEC_VERIFY_PIECES;  // warps sharing one chunk of the ring
#ifndef SPEC_VERIFY_UNROLL
#define SPEC_VERIFY_UNROLL 1
#endif
constexpr int kGroupUnroll = SPEC_VERIFY_UNROLL;  // groups per iteration of the sweep loop
// Consumer warps form kGroups groups of kPieces; group g takes the chunks
// ch = g (mod kGroups).  The ring must have a multiple of kGroups slots so
// that every slot belongs to one group: a warp then only ever waits on a slot
// whose previous phase it consumed itself, which keeps the phase parity of
// mbarrier.try_wait unambiguous.
constexpr int kGroups = kConsumerWarps / kPieces;
static_assert(kConsumerWarps % kPieces == 0, "consumer warps must form whole groups");

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Partial reduction of one row over some elements (16 bytes, pushed over DSMEM).
struct __align__(16) Partial {
  float m;         // largest logit seen (-inf if none)
  float s;         // sum of 2^((x - m) * c) over the elements (sampled rows)
  int idx;         // lowest index holding m (INT_MAX if none)
  uint32_t flags;  // kBadValue | kTimedOut
};

constexpr uint32_t kBadValue = 1u;  // NaN or +inf in the row
constexpr uint32_t kTimedOut = 2u;  // a bounded wait gave up
constexpr uint32_t kEmptyRow = 4u;  // a row with no finite logit (scan flags only)

struct __align__(16) DrawPartial {
  float w;  // sum of draw weights over one CTA's slice
  int pad0, pad1, pad2;
};

enum DrawMode : int { kNoDraw = 0, kResidual = 1, kBonus = 2 };

struct __align__(16) SmemHead {
  uint64_t full[kMaxSlots];
  uint64_t empty[kMaxSlots];
  uint64_t xbar;     // completes when every peer's row partials (or keys) have landed
  uint64_t dbar[2];  // the same for the pass-2 slice sums
  unsigned long long gkey[kMaxDrafts + 1];     // greedy lanes: this CTA's argmax key of every row
  Partial wpart[kMaxStreams][kConsumerWarps];  // per consumer warp
  Partial cpart[kMaxCluster][kMaxStreams];     // per CTA of the cluster (pushed by peers)
  Partial fin[kMaxStreams];                    // this CTA's partial, then the lane's total
  DrawPartial dpart[2][kMaxCluster];           // pass-2 slice sums (pushed by peers)
  float segsum[kConsumerWarps];
  float dcoef[5];  // pass-2 weight coefficients (DrawCoef) of the current attempt
  int drafts[kMaxDrafts + 1];
  float xd_t[kMaxDrafts + 1];  // target logit at d_{j+1} in row j
  float xd_q[kMaxDrafts + 1];  // drafter logit at d_{j+1} in row j
  float u_acc[kMaxDrafts + 1];  // acceptance uniform of position j
  float u_smp[kMaxDrafts + 1];  // draw uniform of position j
  float u_l2i[kMaxDrafts + 1];  // log2 of u_acc[j], split as log2_parts does
  float u_l2f[kMaxDrafts + 1];
  float scan_lp[kMaxDrafts + 1];  // sampled scan: log2 p_j(d), log2 q_j(d) (row statistics)
  float scan_lq[kMaxDrafts + 1];
  int scan_n;
  int scan_mode;
  int scan_st;            // sampled scan: the lane's status
  int draft_range_bad;    // some draft token is outside [0, V)
  uint32_t scan_flags;    // sampled lanes: OR of the merged rows' flags and kEmptyRow
  uint32_t cta_flags;
  int order_hist[kCostBuckets];  // lanes per cost class (longest-first lane order)
  int order_cnt[kWarps];
  int order_bucket, order_j, order_w, order_j2, order_lane;
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
  uint32_t lane_base;  // global index of lane 0 in the Philox counter
  int32_t cluster;     // CTAs per lane
  int32_t slice;       // vocabulary elements per CTA (multiple of the vector width)
  int32_t slot_bytes;  // bytes per ring slot (multiple of 16)
  int32_t nslots;
  int32_t head_bytes;  // offset of the ring in dynamic shared memory
  int32_t order_by_cost;  // clusters take lanes in order of decreasing cost (more lanes than fit at once)
  uint32_t flags;         // SPEC_VERIFY_* flags of spec_verify_args
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

// Sums of sampled rows are kept relative to the scaled reference fl(m * c)
// of the running max m (c = log2(e) / T): s = sum 2^(x * c - fl(m * c)).
// Each term is then one FMA and one exp2, and the reference can always be
// recomputed from m, so merges rescale by 2^(fl(m_i * c) - fl(M * c)).
__device__ __forceinline__ float scaled_ref(float m, float c) { return __fmul_rn(m, c); }

// Merge (m2, s2, i2) into (m, s, idx): max, rescaled sum, lowest index of the max.
template <bool SAMPLED>
__device__ __forceinline__ void merge_part(float& m, float& s, int& idx, float m2, float s2, int i2,
                                           float c) {
  const float nm = fmaxf(m, m2);
  if (SAMPLED) {
    if (nm == -INFINITY) {
      s = s + s2;
    } else {
      const float rn = scaled_ref(nm, c);
      s = s * ex2_approx(scaled_ref(m, c) - rn) + s2 * ex2_approx(scaled_ref(m2, c) - rn);
    }
  }
  if (m2 > m || (m2 == m && i2 < idx)) idx = i2;
  m = nm;
}

// A new running max `vm` first seen at element `e`: rescale the sum.
template <bool SAMPLED>
__device__ __forceinline__ void acc_raise(Acc& a, float vm, int e, float c) {
  if (SAMPLED) a.s *= ex2_approx(scaled_ref(a.m, c) - scaled_ref(vm, c));
  a.m = vm;
  a.idx = e;
}

// 2^(x * c - mr): one FMA and one exp2 (mr = the scaled reference).
__device__ __forceinline__ float exp_term(float x, float mr, float c) {
  return ex2_approx(fmaf(x, c, -mr));
}

// One logit (row tails and unaligned rows).
template <bool SAMPLED>
__device__ __forceinline__ void acc_scalar(Acc& a, float x, int e, float c) {
  a.bad |= !(x <= FLT_MAX);
  if (x > a.m) acc_raise<SAMPLED>(a, x, e, c);
  if (SAMPLED) {
    const float mr = (a.m == -INFINITY) ? 0.f : scaled_ref(a.m, c);
    a.s += exp_term(x, mr, c);
  }
}

// Element e of a 16-byte vector as fp32.
template <typename T>
__device__ __forceinline__ float vec_elem(const uint4 v, int e) {
  if constexpr (ElemTraits<T>::kVec == 8) {
    const uint32_t w = (e < 2) ? v.x : (e < 4) ? v.y : (e < 6) ? v.z : v.w;
    return (e & 1) ? bf16_hi(w) : bf16_lo(w);
  } else {
    const uint32_t w = (e == 0) ? v.x : (e == 1) ? v.y : (e == 2) ? v.z : v.w;
    return __uint_as_float(w);
  }
}

// Packed pairs of fp32 (the f32x2 forms of FMA and add issue both halves as
// one instruction).
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void f2_unpack(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// 2^z of both halves.
__device__ __forceinline__ unsigned long long f2_ex2(unsigned long long z) {
  float lo, hi;
  f2_unpack(z, lo, hi);
  return f2_pack(ex2_approx(lo), ex2_approx(hi));
}

// The two elements of one 32-bit word of a vector as a packed fp32 pair
// (bf16: the low and high halves widened; fp32 vectors give pairs of words).
__device__ __forceinline__ unsigned long long bf16_pair(uint32_t w) {
  return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// acc + sum over the vector's elements of 2^(x * c - mr), as packed pairs;
// c2 = (c, c), nmr2 = (-mr, -mr).
template <typename T>
__device__ __forceinline__ unsigned long long vec_exp_acc(const uint4 v, unsigned long long c2,
                                                          unsigned long long nmr2, unsigned long long acc) {
  if constexpr (ElemTraits<T>::kVec == 8) {
    acc = f2_add(acc, f2_ex2(f2_fma(bf16_pair(v.x), c2, nmr2)));
    acc = f2_add(acc, f2_ex2(f2_fma(bf16_pair(v.y), c2, nmr2)));
    acc = f2_add(acc, f2_ex2(f2_fma(bf16_pair(v.z), c2, nmr2)));
    acc = f2_add(acc, f2_ex2(f2_fma(bf16_pair(v.w), c2, nmr2)));
  } else {
    acc = f2_add(acc, f2_ex2(f2_fma(f2_pack(__uint_as_float(v.x), __uint_as_float(v.y)), c2, nmr2)));
    acc = f2_add(acc, f2_ex2(f2_fma(f2_pack(__uint_as_float(v.z), __uint_as_float(v.w)), c2, nmr2)));
  }
  return acc;
}

template <typename T>
__device__ __forceinline__ uint4 neg_inf_vec() {
  if constexpr (ElemTraits<T>::kVec == 8) return make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
  else return make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
}

// The four vectors v, v + 32, v + 64, v + 96 of one lane's group; with PRED,
// those at or past ve read as -inf (no exponential weight, never a maximum).
template <typename T, bool PRED>
__device__ __forceinline__ void load_group(const uint4* sv, int v, int ve, uint4 (&x)[4]) {
#pragma unroll
  for (int u = 0; u < 4; ++u) x[u] = (!PRED || v + 32 * u < ve) ? sv[v + 32 * u] : neg_inf_vec<T>();
}

// Per-vector maxima of a group, still packed (bf16: a bf16 pair per vector;
// fp32: the vector's max), NaN-propagating.
template <typename T>
__device__ __forceinline__ void group_vec_max(const uint4 (&x)[4], uint32_t (&h)[4]) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    if constexpr (ElemTraits<T>::kVec == 8) {
      h[u] = bf16x2_max_nan(bf16x2_max_nan(x[u].x, x[u].y), bf16x2_max_nan(x[u].z, x[u].w));
    } else {
      h[u] = __float_as_uint(f32_max_nan(f32_max_nan(__uint_as_float(x[u].x), __uint_as_float(x[u].y)),
                                         f32_max_nan(__uint_as_float(x[u].z), __uint_as_float(x[u].w))));
    }
  }
}

// Widen one packed per-vector max to fp32.
template <typename T>
__device__ __forceinline__ float unpack_max(uint32_t h) {
  if constexpr (ElemTraits<T>::kVec == 8) return f32_max_nan(bf16_lo(h), bf16_hi(h));
  else return __uint_as_float(h);
}

// Largest element of the group from its per-vector maxima.
template <typename T>
__device__ __forceinline__ float group_max_nan(const uint32_t (&h)[4]) {
  if constexpr (ElemTraits<T>::kVec == 8) {
    return unpack_max<T>(bf16x2_max_nan(bf16x2_max_nan(h[0], h[1]), bf16x2_max_nan(h[2], h[3])));
  } else {
    return f32_max_nan(f32_max_nan(__uint_as_float(h[0]), __uint_as_float(h[1])),
                       f32_max_nan(__uint_as_float(h[2]), __uint_as_float(h[3])));
  }
}

// Lowest element index of vector vv holding m (the vector is known to hold it).
template <typename T>
__device__ __forceinline__ int vec_find(const uint4* sv, int vv, float m) {
  constexpr int kVec = ElemTraits<T>::kVec;
  const uint4 xv = sv[vv];
  int e = 0;
#pragma unroll
  for (int t = kVec - 1; t >= 0; --t)
    if (vec_elem<T>(xv, t) == m) e = t;
  return vv * kVec + e;
}

// One piece of a chunk in shared memory, processed by one warp: this lane's
// vectors are vb + lane, vb + lane + 32, ... below ve, taken four at a time
// as groups (only the last group of the piece is predicated).  Each group's
// max (NaN-propagating, so that NaN and +inf are flagged) is computed once;
// a lane keeps its running max and the first group that reached it, and the
// element index is looked up in that group after the piece.  Sampled rows
// also sum each group's exponentials relative to the group's own max
// (fl(max * c) as reference, packed fp32 pairs), and fold the group sum into
// the lane's running sum with one rescaling exp2.
//
// LAZY (sampled rows whose max and argmax are not reported): once the lane
// has a finite reference M (the max of the row's groups taken so far, carried
// from piece to piece), a group's exponentials are summed against M
// directly, with no group max.  The sum of 32 terms is at most 32 while no
// element exceeds M; a sum above 2^64, +inf
// or NaN sends the group through the exact path above instead, which raises
// M, rescales, and flags NaN and +inf.  M then stays an element value at or
// below the row max, and every later use of the partial (merges, the
// acceptance test, the draw) needs only that the sum is relative to
// fl(M * c).
constexpr float kLazySumLimit = 18446744073709551616.f;  // 2^64

// Builds whose pieces end in part of a group (a row slice per chunk, split
// five ways) sum a lazy piece's last vectors one at a time and take a row's
// first piece without a merge (SPEC_VERIFY_LAZY_VEC_TAIL): the 8-lane sampled
// round 15.82 -> 15.53 us.  In the build whose pieces are whole groups the
// same code cost the ragged round 0.5 us, so it is left out there.
#ifndef SPEC_VERIFY_LAZY_VEC_TAIL
#define SPEC_VERIFY_LAZY_VEC_TAIL 0
#endif
constexpr bool kLazyVecTail = SPEC_VERIFY_LAZY_VEC_TAIL != 0;

// Ring slots up to this size are filled by one issuing lane per consumer group.
constexpr int kParallelIssueSlotBytes = 8192;

template <typename T, bool SAMPLED, bool LAZY = false>
__device__ __forceinline__ void acc_range(Acc& a, const uint4* sv, int vb, int ve, int ebase, float c,
                                          int lane) {
  float M = -INFINITY, nanacc = -INFINITY;
  float S = 0.f;  // sampled: sum relative to scaled_ref(M)
  float rM = 0.f; // LAZY: scaled_ref(M) while M is finite
  int gv = -1;    // first vector holding M
  if constexpr (LAZY) {
    // A piece continues the row's reference from the pieces before it, so
    // that only a row's first group needs the exact path.
    if (a.m != -INFINITY) {
      M = a.m;
      rM = scaled_ref(M, c);
    }
  }
  const unsigned long long c2 = f2_pack(c, c);
  // LAZY: the group's exponentials against the lane's reference.
  auto lazy_sum = [&](const uint4 (&x)[4]) -> float {
    const unsigned long long nmr2 = f2_pack(-rM, -rM);
    unsigned long long acc = 0ull;  // (+0, +0)
#pragma unroll
    for (int u = 0; u < 4; ++u) acc = vec_exp_acc<T>(x[u], c2, nmr2, acc);
    float lo, hi;
    f2_unpack(acc, lo, hi);
    return lo + hi;
  };
  auto exact = [&](const uint4 (&x)[4], int v) {
    uint32_t h[4];
    group_vec_max<T>(x, h);
    const float gm = group_max_nan<T>(h);
    nanacc = f32_max_nan(nanacc, gm);
    if (SAMPLED && gm != -INFINITY) {
      const float rg = scaled_ref(gm, c);
      const unsigned long long nmr2 = f2_pack(-rg, -rg);
      unsigned long long acc = 0ull;  // (+0, +0)
#pragma unroll
      for (int u = 0; u < 4; ++u) acc = vec_exp_acc<T>(x[u], c2, nmr2, acc);
      float lo, hi;
      f2_unpack(acc, lo, hi);
      const float sg = lo + hi;
      if (gm > M) S = (M == -INFINITY) ? sg : fmaf(S, ex2_approx(scaled_ref(M, c) - rg), sg);
      else S = fmaf(sg, ex2_approx(rg - scaled_ref(M, c)), S);
    }
    if (gm > M) {
      // A new running max (rare after the first groups): the first vector of
      // the group that holds it.
      M = gm;
      if (LAZY) rM = scaled_ref(M, c);
      gv = v + 96;
#pragma unroll
      for (int u = 2; u >= 0; --u)
        if (unpack_max<T>(h[u]) == gm) gv = v + 32 * u;
    }
  };
  auto group = [&](const uint4 (&x)[4], int v) {
    if (LAZY && M != -INFINITY) {
      const float sg = lazy_sum(x);
      if (sg <= kLazySumLimit) {
        S += sg;
        return;
      }
    }
    exact(x, v);
  };
  int v = vb + lane;
  if constexpr (LAZY) {
    // A row's first piece takes its reference from the lane's first element:
    // any finite element value at or below the row max will do.
    if (M == -INFINITY && v < ve) {
      const float x0 = vec_elem<T>(sv[v], 0);
      if (x0 > -INFINITY && x0 <= FLT_MAX) {
        M = x0;
        rM = scaled_ref(M, c);
      }
    }
    // A tight loop of lazily summed groups; a group it cannot take (no
    // reference yet, or a sum out of range) leaves it for the exact path,
    // which is kept out of the loop body.
    for (;;) {
      if (M != -INFINITY) {
#pragma unroll kGroupUnroll
        for (; v + 96 < ve; v += 128) {
          uint4 x[4];
          load_group<T, false>(sv, v, ve, x);
          const float sg = lazy_sum(x);
          if (!(sg <= kLazySumLimit)) break;
          S += sg;
        }
      }
      if (v + 96 >= ve) break;
      uint4 x[4];
      load_group<T, false>(sv, v, ve, x);
      exact(x, v);
      v += 128;
    }
  } else {
#pragma unroll kGroupUnroll
    for (; v + 96 < ve; v += 128) {
      uint4 x[4];
      load_group<T, false>(sv, v, ve, x);
      group(x, v);
    }
  }
  if constexpr (LAZY && kLazyVecTail) {
    // Fewer than four vectors a lane are left: summed one at a time, with
    // no -inf padding; a sum out of range leaves the rest to the exact path.
    if (M != -INFINITY) {
      const unsigned long long nmr2 = f2_pack(-rM, -rM);
      for (; v < ve; v += 32) {
        float lo, hi;
        f2_unpack(vec_exp_acc<T>(sv[v], c2, nmr2, 0ull), lo, hi);
        const float sg = lo + hi;
        if (!(sg <= kLazySumLimit)) break;
        S += sg;
      }
    }
  }
  if (v < ve) {
    uint4 x[4];
    load_group<T, true>(sv, v, ve, x);
    group(x, v);
  }
  if (nanacc != nanacc || nanacc == INFINITY) a.bad = 1;
  if (M == -INFINITY) return;
  if (SAMPLED) {
    if (LAZY && M == a.m) {
      a.s += S;  // the same reference: nothing to rescale
    } else if (LAZY && kLazyVecTail && a.m == -INFINITY) {
      a.m = M;  // the lane's first piece of the row
      a.s = S;
      a.idx = ebase;
    } else {
      // LAZY: any element index marks the partial as holding elements
      const int e = LAZY ? ebase : (M >= a.m) ? ebase + vec_find<T>(sv, gv, M) : INT_MAX;
      merge_part<true>(a.m, a.s, a.idx, M, S, e, c);
    }
  } else if (M > a.m) {
    acc_raise<false>(a, M, ebase + vec_find<T>(sv, gv, M), c);
  }
}

__device__ __forceinline__ uint32_t acc_bad(const Acc& a) {
  const float lo = bf16_lo(a.nan2), hi = bf16_hi(a.nan2);
  const bool packed_bad = (lo != lo) || (hi != hi) || lo == INFINITY || hi == INFINITY;
  return (a.bad || packed_bad) ? kBadValue : 0u;
}

// Warp-wide merge; every lane ends with the warp's max, lowest index of the
// max and flags, lane 0 with the sum.  The max and the index are single warp
// reductions; each lane then rescales its own sum to the warp max once and
// the sums are added by a butterfly.
template <bool SAMPLED>
__device__ __forceinline__ Partial warp_merge(float m, float s, int idx, uint32_t flags, float c) {
  flags = __reduce_or_sync(0xFFFFFFFFu, flags);
  const float M = warp_max_f32(m);
  const int I = __reduce_min_sync(0xFFFFFFFFu, (m == M) ? idx : INT_MAX);
  if (SAMPLED) {
    float t = (M == -INFINITY) ? s : s * ex2_approx(scaled_ref(m, c) - scaled_ref(M, c));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
    s = t;
  }
  return Partial{M, s, I, flags};
}

__device__ __forceinline__ Partial identity_partial() { return Partial{-INFINITY, 0.f, INT_MAX, 0u}; }

// Greedy rows reduce to one 64-bit key per row: the order-preserving bits of
// the max on top and the complemented index below, so that the largest key is
// the largest logit at its lowest index and partial results combine with a
// single atomic max.  -0 is folded into +0 first (the two compare equal, so
// the lower index must win between them).  0 means "no element".
__device__ __forceinline__ unsigned long long argmax_key(float m, int idx) {
  if (idx == INT_MAX) return 0ull;
  uint32_t u = __float_as_uint(__fadd_rn(m, 0.f));
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<unsigned long long>(u) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(idx));
}

__device__ __forceinline__ void argmax_key_decode(unsigned long long key, float& m, int& idx) {
  if (key == 0ull) {
    m = -INFINITY;
    idx = INT_MAX;
    return;
  }
  const uint32_t u = static_cast<uint32_t>(key >> 32);
  m = __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
  idx = static_cast<int>(~static_cast<uint32_t>(key));
}

// A consumer warp's contribution to greedy row s: the warp's max and lowest
// index of it, folded into the CTA's key of the row; flags go straight into
// the CTA's flag word.
__device__ __forceinline__ void fold_greedy_row(SmemHead& sh, int s, float m, int idx, uint32_t flags, int lane) {
  const float M = warp_max_f32(m);
  const int I = __reduce_min_sync(0xFFFFFFFFu, (m == M) ? idx : INT_MAX);
  if (flags) atomicOr(&sh.cta_flags, flags);
  if (lane == 0 && I != INT_MAX) atomicMax(&sh.gkey[s], argmax_key(M, I));
}

// ---------------------------------------------------------------------------
// Compensated fp32 sums for the acceptance test
// ---------------------------------------------------------------------------
// a + b = s + e exactly (Knuth's TwoSum).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float z = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, z)), __fsub_rn(b, z));
}

// Running sum with the rounding errors of every addition carried alongside
// (Ogita, Rump and Oishi, "Accurate sum and dot product", Algorithm Sum2):
// the result is as accurate as a sum in twice the working precision, then
// rounded once.
struct CompSum {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float x) {
    float t, e;
    two_sum(s, x, t, e);
    s = t;
    c = __fadd_rn(c, e);
  }
  __device__ __forceinline__ float value() const { return __fadd_rn(s, c); }
};

// log2 p(d) of a row in the terms its sum was taken in,
//   x_d * c - fl(max * c) - log2(S),
// as a compensated sum: x_d * c split exactly into fl(x_d * c) and the FMA
// remainder, log2(S) into its exact exponent and its fraction.
__device__ __forceinline__ CompSum log2_prob_terms(float xd, const Partial& row, float c) {
  float ip, fp;
  log2_parts(row.s, ip, fp);
  const float t = __fmul_rn(xd, c);
  CompSum r;
  r.add(t);
  r.add(-scaled_ref(row.m, c));
  r.add(-ip);
  r.add(-fp);
  r.add(__fmaf_rn(xd, c, -t));
  return r;
}

// ---------------------------------------------------------------------------
// Pass-2 draw weights
// ---------------------------------------------------------------------------
// A draw needs its weights only up to a common factor, so they are taken
// times S_p, the target row's sum: the weight of element x is
// p'(x) = 2^(fl(x * c - fl(m_p * c))) for a bonus draw and max(0, p'(x) -
// q'(x)) for a residual draw, q'(x) = 2^(fl(fl(x * c - fl(m_q * c)) + e)) over
// the drafter row with e = fl(log2 S_p - log2 S_q) (q(x) * S_p).  A bonus
// weight is one FMA and one exp2.  The residual mass is the weights' total
// times 2^(-log2 S_p).  The sums take the weights as packed pairs and the walk
// as scalars; both round every step identically, so each weight has the same
// bits wherever it is formed, and a lane's eight weights are always added in
// the same order (tree8).
struct DrawCoef {
  float mp;  // target row: scaled reference fl(max * c)
  float mq;  // drafter row (residual only): its scaled reference
  float e;   // fl(log2 S_p - log2 S_q) (residual only)
  float c;   // log2(e) / T
};

// Coefficients of the weights of a draw from target row `rt` (and drafter row
// `rq` for a residual draw, -1 for a bonus draw) given the rows' totals.
__device__ __forceinline__ void draw_coef_store(float* out, const Partial* fin, int rt, int rq, float c) {
  const Partial pt = fin[2 * rt];
  out[0] = scaled_ref(pt.m, c);
  out[1] = log2f(pt.s);
  out[2] = 0.f;
  out[3] = 0.f;
  out[4] = c;
  if (rq >= 0) {
    const Partial pq = fin[2 * rq + 1];
    out[2] = scaled_ref(pq.m, c);
    out[3] = log2f(pq.s);
  }
}

__device__ __forceinline__ DrawCoef draw_coef_load(const float* in) {
  DrawCoef k;
  k.mp = in[0];
  k.mq = in[2];
  k.e = __fsub_rn(in[1], in[3]);
  k.c = in[4];
  return k;
}

template <bool RESID>
__device__ __forceinline__ float draw_weight(const DrawCoef& k, float xt, float xq) {
  const float p = ex2_approx(__fmaf_rn(xt, k.c, -k.mp));
  if (!RESID) return p;
  const float q = ex2_approx(__fadd_rn(__fmaf_rn(xq, k.c, -k.mq), k.e));
  return fmaxf(0.f, __fsub_rn(p, q));
}

// The coefficients duplicated into packed pairs.
struct DrawCoef2 {
  unsigned long long c, nmp, nmq, e, neg1;
};

__device__ __forceinline__ DrawCoef2 pack_coef(const DrawCoef& k) {
  DrawCoef2 r;
  r.c = f2_pack(k.c, k.c);
  r.nmp = f2_pack(-k.mp, -k.mp);
  r.nmq = f2_pack(-k.mq, -k.mq);
  r.e = f2_pack(k.e, k.e);
  r.neg1 = f2_pack(-1.f, -1.f);
  return r;
}

// draw_weight of two elements at once: p' - q' is formed as fma(q', -1, p'),
// rounded once, as the scalar form is.
template <bool RESID>
__device__ __forceinline__ unsigned long long draw_weight2(const DrawCoef2& k, unsigned long long xt,
                                                           unsigned long long xq) {
  const unsigned long long p = f2_ex2(f2_fma(xt, k.c, k.nmp));
  if (!RESID) return p;
  const unsigned long long q = f2_ex2(f2_add(f2_fma(xq, k.c, k.nmq), k.e));
  float lo, hi;
  f2_unpack(f2_fma(q, k.neg1, p), lo, hi);
  return f2_pack(fmaxf(0.f, lo), fmaxf(0.f, hi));
}

// Total of a lane's eight weights: ((w0 + w2) + (w4 + w6)) + ((w1 + w3) + (w5 + w7)),
// the order in which the packed pairs add them.
__device__ __forceinline__ float tree8(const float (&w)[8]) {
  return __fadd_rn(__fadd_rn(__fadd_rn(w[0], w[2]), __fadd_rn(w[4], w[6])),
                   __fadd_rn(__fadd_rn(w[1], w[3]), __fadd_rn(w[5], w[7])));
}

// Eight consecutive logits of a row, kept as raw bits (one 16-byte vector of
// bf16, two of fp32) so that several rounds can be in flight at once.
template <typename T>
struct Raw8 {
  uint4 v[ElemTraits<T>::kVec == 8 ? 1 : 2];
};

template <typename T>
__device__ __forceinline__ float raw_elem(const Raw8<T>& r, int i) {
  if constexpr (ElemTraits<T>::kVec == 8) return vec_elem<T>(r.v[0], i);
  else return vec_elem<T>(r.v[i >> 2], i & 3);
}

// Elements 2j and 2j + 1 as a packed pair.
template <typename T>
__device__ __forceinline__ unsigned long long raw_pair(const Raw8<T>& r, int j) {
  if constexpr (ElemTraits<T>::kVec == 8) {
    return bf16_pair((j == 0) ? r.v[0].x : (j == 1) ? r.v[0].y : (j == 2) ? r.v[0].z : r.v[0].w);
  } else {
    const uint4 v = r.v[j >> 1];
    return (j & 1) ? f2_pack(__uint_as_float(v.z), __uint_as_float(v.w))
                   : f2_pack(__uint_as_float(v.x), __uint_as_float(v.y));
  }
}

// Elements e .. e+7 of a row; those at or past `end` read as -inf.
template <typename T, bool ALIGNED>
__device__ __forceinline__ void load_raw8(const uint8_t* row, int e, int end, Raw8<T>& r) {
  constexpr bool kBf16 = ElemTraits<T>::kVec == 8;
  if (ALIGNED && e + 8 <= end) {
    const uint4* p = reinterpret_cast<const uint4*>(row + static_cast<int64_t>(e) * (kBf16 ? 2 : 4));
    r.v[0] = __ldg(p);
    if constexpr (!kBf16) r.v[1] = __ldg(p + 1);
  } else {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if constexpr (kBf16) {
        w[i] = (e + i < end) ? static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(row) + e + i))
                             : 0xFF80u;
      } else {
        w[i] = (e + i < end) ? __float_as_uint(__ldg(reinterpret_cast<const float*>(row) + e + i))
                             : 0xFF800000u;
      }
    }
    if constexpr (kBf16) {
      r.v[0] = make_uint4(w[0] | (w[1] << 16), w[2] | (w[3] << 16), w[4] | (w[5] << 16), w[6] | (w[7] << 16));
    } else {
      r.v[0] = make_uint4(w[0], w[1], w[2], w[3]);
      r.v[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
  }
}

// Total of the weights of one lane's eight elements, all in range, as packed pairs.
template <typename T, bool RESID>
__device__ __forceinline__ float piece_total(const DrawCoef2& k, const Raw8<T>& rt, const Raw8<T>& rq) {
  unsigned long long w2[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if constexpr (RESID) w2[j] = draw_weight2<true>(k, raw_pair<T>(rt, j), raw_pair<T>(rq, j));
    else w2[j] = draw_weight2<false>(k, raw_pair<T>(rt, j), 0ull);
  }
  float lo, hi;
  f2_unpack(f2_add(f2_add(w2[0], w2[1]), f2_add(w2[2], w2[3])), lo, hi);
  return __fadd_rn(lo, hi);
}

// The eight weights of elements e .. e+7 (0 at or past `end`) as scalars.
template <typename T, bool RESID>
__device__ __forceinline__ void piece_weights(const DrawCoef& k, const Raw8<T>& rt, const Raw8<T>& rq, int e, int end,
                                              float (&w)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if constexpr (RESID) w[i] = (e + i < end) ? draw_weight<true>(k, raw_elem<T>(rt, i), raw_elem<T>(rq, i)) : 0.f;
    else w[i] = (e + i < end) ? draw_weight<false>(k, raw_elem<T>(rt, i), 0.f) : 0.f;
  }
}

// Pass-2 rounds whose loads are issued together: one round's loads are in
// flight while the previous round is summed.  (Four rounds, two in flight,
// pushed the 20-warp builds past their 80 registers into spills, which cost
// more than the extra latency hidden: the ragged 128-lane round 92.7 against
// 84.7 us.)
template <typename T>
__host__ __device__ constexpr int draw_batch() {
  return 2;
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

// One warp's pass-2 segment [s0, s1) is taken in rounds of kDrawRound
// elements; lane l holds elements 8l .. 8l+7 of each round.  `lsum`, when
// given, keeps every lane's total of every round (lsum[r * 32 + lane]).

// Builds that define SPEC_VERIFY_DRAW_STAGE stage the pass-2 rounds of long
// segments (at least kDrawStageMinRounds full rounds) kDrawStage rounds ahead
// in shared memory (cp.async, no registers held): the ragged 128-lane round,
// 13 rounds a warp, 84.6 -> 83.9 us.  Compiled into the build that serves
// the 8-lane sampled round (3 rounds a warp, never staged) the same code
// cost that round 0.5 us, so only the build for streamed slices has it.
#ifndef SPEC_VERIFY_DRAW_STAGE
#define SPEC_VERIFY_DRAW_STAGE 0
#endif
constexpr bool kDrawStaged = SPEC_VERIFY_DRAW_STAGE != 0;
constexpr int kDrawStage = 4;
constexpr int kDrawStageMinRounds = 6;

template <typename T>
__host__ __device__ constexpr int draw_stage_bytes() {  // one warp's staging buffer
  return kDrawStage * 64 * (ElemTraits<T>::kVec == 8 ? 16 : 32);
}

// Sum of the draw weights of the segment (every lane gets it).  Full rounds
// run as packed pairs, either staged through `stage` (a warp's
// draw_stage_bytes of shared memory, or nullptr) or with the next
// half-batch's loads in flight in registers; the last, partial round is
// masked.
template <typename T, bool ALIGNED, bool RESID>
__device__ __forceinline__ float draw_segment_sum(const DrawCoef& kc, const uint8_t* trow, const uint8_t* qrow,
                                                  int s0, int s1, float* lsum, int lane, uint8_t* stage) {
  constexpr int kHalf = draw_batch<T>() / 2;
  const DrawCoef2 k2 = pack_coef(kc);
  const int nfull = (s1 > s0) ? (s1 - s0) / kDrawRound : 0;
  float acc = 0.f;
  bool staged = false;
  if constexpr (kDrawStaged) staged = ALIGNED && stage != nullptr && nfull >= kDrawStageMinRounds;
  if (staged) {
    // Round r of this lane sits at stage + (r mod kDrawStage) * 64 * LB + lane * LB
    // (target) and 32 * LB further (drafter), LB = the bytes of eight elements.
    constexpr int kLB = ElemTraits<T>::kVec == 8 ? 16 : 32;
    constexpr int kEs = ElemTraits<T>::kVec == 8 ? 2 : 4;
    uint8_t* mine = stage + lane * kLB;
    auto issue = [&](int r) {
      const int64_t src = static_cast<int64_t>(s0 + r * kDrawRound + lane * 8) * kEs;
      uint8_t* dst = mine + (r % kDrawStage) * (64 * kLB);
      cp_async16(dst, trow + src);
      if constexpr (kLB == 32) cp_async16(dst + 16, trow + src + 16);
      if constexpr (RESID) {
        cp_async16(dst + 32 * kLB, qrow + src);
        if constexpr (kLB == 32) cp_async16(dst + 32 * kLB + 16, qrow + src + 16);
      }
    };
    // One commit group per round (empty past the end), so that waiting until
    // at most kDrawStage - 1 groups are pending completes round r.
#pragma unroll
    for (int d = 0; d < kDrawStage - 1; ++d) {
      issue(d);  // nfull >= kDrawStageMinRounds > kDrawStage - 1
      cp_async_commit();
    }
    for (int r = 0; r < nfull; ++r) {
      if (r + kDrawStage - 1 < nfull) issue(r + kDrawStage - 1);
      cp_async_commit();
      cp_async_wait<kDrawStage - 1>();
      const uint8_t* src = mine + (r % kDrawStage) * (64 * kLB);
      Raw8<T> rt, rq;
      rt.v[0] = *reinterpret_cast<const uint4*>(src);
      if constexpr (kLB == 32) rt.v[1] = *reinterpret_cast<const uint4*>(src + 16);
      if constexpr (RESID) {
        rq.v[0] = *reinterpret_cast<const uint4*>(src + 32 * kLB);
        if constexpr (kLB == 32) rq.v[1] = *reinterpret_cast<const uint4*>(src + 32 * kLB + 16);
      }
      const float t = piece_total<T, RESID>(k2, rt, rq);
      if (lsum) lsum[r * 32 + lane] = t;
      acc = __fadd_rn(acc, t);
    }
    cp_async_wait<0>();
  } else {
  Raw8<T> rtA[kHalf], rqA[kHalf], rtB[kHalf], rqB[kHalf];
  auto load_half = [&](Raw8<T> (&rt)[kHalf], Raw8<T> (&rq)[kHalf], int r0) {
#pragma unroll
    for (int u = 0; u < kHalf; ++u) {
      if (r0 + u < nfull) {
        const int e = s0 + (r0 + u) * kDrawRound + lane * 8;
        load_raw8<T, ALIGNED>(trow, e, s1, rt[u]);
        if constexpr (RESID) load_raw8<T, ALIGNED>(qrow, e, s1, rq[u]);
      }
    }
  };
  auto sum_half = [&](const Raw8<T> (&rt)[kHalf], const Raw8<T> (&rq)[kHalf], int r0) {
#pragma unroll
    for (int u = 0; u < kHalf; ++u) {
      if (r0 + u < nfull) {
        const float t = piece_total<T, RESID>(k2, rt[u], rq[u]);
        if (lsum) lsum[(r0 + u) * 32 + lane] = t;
        acc = __fadd_rn(acc, t);
      }
    }
  };
  if (nfull > 0) load_half(rtA, rqA, 0);
  for (int r = 0; r < nfull; r += 2 * kHalf) {
    if (r + kHalf < nfull) load_half(rtB, rqB, r + kHalf);
    sum_half(rtA, rqA, r);
    if (r + kHalf >= nfull) break;
    if (r + 2 * kHalf < nfull) load_half(rtA, rqA, r + 2 * kHalf);
    sum_half(rtB, rqB, r + kHalf);
  }
  }
  const int tb = s0 + nfull * kDrawRound;
  if (tb < s1) {
    const int e = tb + lane * 8;
    Raw8<T> rt, rq;
    load_raw8<T, ALIGNED>(trow, e, s1, rt);
    if constexpr (RESID) load_raw8<T, ALIGNED>(qrow, e, s1, rq);
    float w[8];
    piece_weights<T, RESID>(kc, rt, rq, e, s1, w);
    const float t = tree8(w);
    if (lsum) lsum[nfull * 32 + lane] = t;
    acc = __fadd_rn(acc, t);
  }
  return warp_sum_xor(acc);
}

// This lane's eight weights of the round at `base`, and their total (equal,
// bit for bit, to what draw_segment_sum took for it).
template <typename T, bool ALIGNED, bool RESID>
__device__ __forceinline__ float draw_round_weights(const DrawCoef& kc, const uint8_t* trow, const uint8_t* qrow,
                                                    int base, int s1, int lane, float (&w)[8]) {
  const int e = base + lane * 8;
  Raw8<T> rt, rq;
  load_raw8<T, ALIGNED>(trow, e, s1, rt);
  if constexpr (RESID) load_raw8<T, ALIGNED>(qrow, e, s1, rq);
  piece_weights<T, RESID>(kc, rt, rq, e, s1, w);
  return tree8(w);
}

// Largest index of positive weight in the segment (-1 if none): the last
// round, then the last lane, holding weight.  Whole warp.
template <typename T, bool ALIGNED, bool RESID>
__device__ __noinline__ int draw_last_positive(const DrawCoef kc, const uint8_t* trow, const uint8_t* qrow, int s0,
                                               int s1, const float* lsum, int lane) {
  const int nr = (s1 > s0) ? (s1 - s0 + kDrawRound - 1) / kDrawRound : 0;
  float w[8];
  for (int r = nr - 1; r >= 0; --r) {
    const int base = s0 + r * kDrawRound;
    const float lt = lsum ? lsum[r * 32 + lane] : draw_round_weights<T, ALIGNED, RESID>(kc, trow, qrow, base, s1, lane, w);
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, lt > 0.f);
    if (m) {
      if (lsum) draw_round_weights<T, ALIGNED, RESID>(kc, trow, qrow, base, s1, lane, w);
      const int l = 31 - __clz(m);
      int pos = -1;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (w[i] > 0.f) pos = base + lane * 8 + i;
      return __shfl_sync(0xFFFFFFFFu, pos, l);
    }
  }
  return -1;
}

// Segments of at least this many rounds find their crossing round 32 rounds
// at a time (see draw_walk); shorter ones round by round.
#ifndef SPEC_VERIFY_WALK_SKIP_MIN
#define SPEC_VERIFY_WALK_SKIP_MIN 2
#endif
constexpr int kWalkSkipRounds = SPEC_VERIFY_WALK_SKIP_MIN;

// Index of the element at which the running weight sum of the segment first
// exceeds tau: the round from the round totals, the lane from a scan of the
// lane totals, the element from the lane's own running sum; -2 if no round
// crosses.  Where rounding leaves a round (or a lane) with no crossing
// element, the last element of positive weight in it.  Whole warp.

template <typename T, bool ALIGNED, bool RESID>
__device__ __noinline__ int draw_walk(const DrawCoef kc, const uint8_t* trow, const uint8_t* qrow, int s0, int s1,
                                      const float* lsum, float tau, int lane) {
  const int nr = (s1 > s0) ? (s1 - s0 + kDrawRound - 1) / kDrawRound : 0;
  float run = 0.f;
  float w[8];
  int r0 = 0;  // first round to walk one by one
  float skip_next = -1.f;  // the running total through round r0, when the skip found it
  if (lsum && nr >= kWalkSkipRounds) {
    // With the lane totals kept, long segments skip rounds 32 at a time (a
    // few rounds are faster one by one): lane i sums the 32 lane totals of
    // round rb + i, a prefix over the lanes gives the running totals, and a
    // ballot finds the first round past tau.
    for (int rb = 0; rb < nr; rb += 32) {
      const int r = rb + lane;
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
      if (r < nr) {
        // Eight 16-byte loads a lane, rotated so that each quarter-warp's
        // eight lanes read eight different bank groups.
        const float4* lt = reinterpret_cast<const float4*>(lsum + r * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 q4 = lt[(i + lane) & 7];
          a0 = __fadd_rn(a0, q4.x);
          a1 = __fadd_rn(a1, q4.y);
          a2 = __fadd_rn(a2, q4.z);
          a3 = __fadd_rn(a3, q4.w);
        }
      }
      float incl = __fadd_rn(__fadd_rn(a0, a1), __fadd_rn(a2, a3));
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float up = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl = __fadd_rn(up, incl);
      }
      const uint32_t past = __ballot_sync(0xFFFFFFFFu, r < nr && __fadd_rn(run, incl) > tau);
      if (past) {
        const int l = __ffs(past) - 1;
        const float before = __shfl_sync(0xFFFFFFFFu, incl, (l > 0) ? l - 1 : 0);
        const float through = __shfl_sync(0xFFFFFFFFu, incl, l);
        skip_next = __fadd_rn(run, through);  // past tau: round r0 crosses
        if (l > 0) run = __fadd_rn(run, before);
        r0 = rb + l;
        break;
      }
      run = __fadd_rn(run, __shfl_sync(0xFFFFFFFFu, incl, 31));
      r0 = min(nr, rb + 32);
    }
  }
  for (int r = r0; r < nr; ++r) {
    const int base = s0 + r * kDrawRound;
    const float lt = lsum ? lsum[r * 32 + lane] : draw_round_weights<T, ALIGNED, RESID>(kc, trow, qrow, base, s1, lane, w);
    // Round r0, when the skip found it, crosses by construction; its lanes'
    // own scan below may then fall short by a rounding, which takes the
    // last positive weight of the round.
    const float next = (r == r0 && skip_next >= 0.f) ? skip_next : __fadd_rn(run, warp_sum_xor(lt));
    if (next > tau) {
      // With kept totals the round's elements are read again here: the
      // loads go out first, and the lane is found from the kept totals while
      // they are in flight.
      Raw8<T> rt, rq;
      if (lsum) {
        load_raw8<T, ALIGNED>(trow, base + lane * 8, s1, rt);
        if constexpr (RESID) load_raw8<T, ALIGNED>(qrow, base + lane * 8, s1, rq);
      }
      const float tau2 = __fsub_rn(tau, run);
      float incl = lt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float up = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl = __fadd_rn(up, incl);
      }
      float excl = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
      if (lane == 0) excl = 0.f;
      const uint32_t hit = __ballot_sync(0xFFFFFFFFu, incl > tau2);
      const uint32_t pos_lanes = __ballot_sync(0xFFFFFFFFu, lt > 0.f);
      const int l = hit ? (__ffs(hit) - 1) : (pos_lanes ? 31 - __clz(pos_lanes) : 0);
      const float tau3 = __fsub_rn(tau2, excl);
      if (lsum) piece_weights<T, RESID>(kc, rt, rq, base + lane * 8, s1, w);
      int t = -1, lastpos = -1;
      float cum = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        cum = __fadd_rn(cum, w[i]);
        if (w[i] > 0.f) lastpos = base + lane * 8 + i;
        if (hit && t < 0 && cum > tau3) t = base + lane * 8 + i;
      }
      return __shfl_sync(0xFFFFFFFFu, (t >= 0) ? t : lastpos, l);
    }
    run = next;
  }
  return -2;
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------

// Push this CTA's partial of every row of a sampled lane into every CTA of
// the cluster.  A peer's copy goes by st.async and completes the receiver's
// xbar; the CTA's own copy is a plain shared-memory store.
__device__ __forceinline__ void push_partials(SmemHead& sh, int nstreams, int C, uint32_t rank,
                                              uint32_t extra_flags) {
  const int dests = C;
  for (int t = threadIdx.x; t < nstreams * dests; t += kThreads) {
    const int s = t / dests, dst = t % dests;
    const Partial q = sh.fin[s];
    const uint32_t fl = q.flags | extra_flags;
    if (dst == static_cast<int>(rank)) {
      sh.cpart[rank][s] = Partial{q.m, q.s, q.idx, fl};
    } else {
      st_async_v4(cluster_map(&sh.cpart[rank][s], dst), __float_as_uint(q.m), __float_as_uint(q.s),
                  static_cast<uint32_t>(q.idx), fl, cluster_map(&sh.xbar, dst));
    }
  }
}

// Acceptance scan and outputs of a greedy lane, run by one warp that holds
// the lane's combined keys: lane j has the key of row j and `flags` is the
// OR of every CTA's flags.  Draft d_{j+1} is accepted while it equals the
// argmax of row j; the committed tokens are the argmaxes of rows 0..n.
__device__ __forceinline__ void greedy_finish(const VerifyParams& p, const int* drafts, int b, int k, int off,
                                              int status, unsigned long long key, uint32_t flags, int lane) {
  float m;
  int a;
  argmax_key_decode(key, m, a);
  int st = status;
  const bool range_bad = (st == SPEC_OK) && lane < k && (drafts[lane] < 0 || drafts[lane] >= p.V);
  const bool empty_row = (st == SPEC_OK) && lane <= k && key == 0ull;
  const bool any_range_bad = __any_sync(0xFFFFFFFFu, range_bad);
  const bool any_empty = __any_sync(0xFFFFFFFFu, empty_row);
  if (st == SPEC_OK) {
    if (any_range_bad) st = SPEC_ERR_TOKEN_RANGE;
    else if (flags & kTimedOut) st = SPEC_ERR_TIMEOUT;
    else if ((flags & kBadValue) || any_empty) st = SPEC_ERR_NONFINITE;
  }
  const bool stop = (st == SPEC_OK) && lane < k && drafts[lane] != a;
  const uint32_t mask = __ballot_sync(0xFFFFFFFFu, stop);
  const int n = mask ? (__ffs(mask) - 1) : k;
  if (lane == 0) {
    p.committed[b] = (st == SPEC_OK) ? n + 1 : 0;
    if (p.lane_status) p.lane_status[b] = st;
  }
  if (status == SPEC_ERR_LAYOUT) return;
  for (int j = lane; j <= k; j += 32) {
    p.out_tokens[off + j] = (st == SPEC_OK && j <= n) ? a : -1;
    if (p.row_stats && st == SPEC_OK) {
      spec_row_stats* rs = p.row_stats + off + j;
      rs->argmax = a;
      rs->max_logit = m;
      rs->lse = NAN;
      rs->logp_d = NAN;
      rs->logq_d = NAN;
      rs->resid_mass = NAN;
      rs->drawn = -1;
      rs->flags = 1;
    }
  }
}

// Estimated cost class of lane b: the rows it streams, a sampled row pair
// (target and drafter, with exponentials) counting twice a greedy row, plus
// one for the draw.  Lanes that will fail their checks cost 0.
__device__ __forceinline__ int lane_cost(const VerifyParams& p, int b) {
  const int k = __ldg(p.draft_lens + b);
  const float t = __ldg(p.temps + b);
  if (k < 0 || k > kMaxDrafts) return 0;
  return (t > 0.f) ? 4 * k + 3 : k + 1;  // < kCostBuckets
}

// The lane of rank `rank` when lanes are sorted by decreasing cost class
// (ties by index).  Clusters start roughly in index order, so when there are
// more lanes than resident clusters, mapping cluster i to the lane of rank i
// starts the costliest lanes first and lets cheap ones fill the last waves
// (longest-processing-time-first list scheduling).  Every CTA computes the
// same permutation from the lane metadata: a histogram of the cost classes,
// the class holding the rank, then that class's members counted in index
// order.  Called by all threads; returns the same lane in every thread.
__device__ int lane_of_rank(const VerifyParams& p, SmemHead& sh, int rank) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid < kCostBuckets) sh.order_hist[tid] = 0;
  __syncthreads();
  for (int b = tid; b < p.lanes; b += kThreads) atomicAdd(&sh.order_hist[lane_cost(p, b)], 1);
  __syncthreads();
  if (warp == 0) {
    // Lane l holds classes 63 - 2l and 62 - 2l; higher classes rank first.
    const int c0 = kCostBuckets - 1 - 2 * lane, c1 = c0 - 1;
    const int h0 = sh.order_hist[c0], h1 = sh.order_hist[c1];
    int incl = h0 + h1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int up = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += up;
    }
    const int excl = incl - h0 - h1;
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, incl > rank);
    if (lane == __ffs(m) - 1) {
      const bool first = rank < excl + h0;
      sh.order_bucket = first ? c0 : c1;
      sh.order_j = first ? rank - excl : rank - excl - h0;
    }
  }
  __syncthreads();
  const int c = sh.order_bucket, j = sh.order_j;
  const int per = (p.lanes + kWarps - 1) / kWarps;
  const int lo = min(p.lanes, warp * per), hi = min(p.lanes, lo + per);
  int cnt = 0;
  for (int b = lo + lane; b < hi; b += 32) cnt += (lane_cost(p, b) == c) ? 1 : 0;
  cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
  if (lane == 0) sh.order_cnt[warp] = cnt;
  __syncthreads();
  if (warp == 0) {
    const int v = (lane < kWarps) ? sh.order_cnt[lane] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int up = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += up;
    }
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, incl > j);
    if (lane == __ffs(m) - 1) {
      sh.order_w = lane;
      sh.order_j2 = j - (incl - v);
    }
  }
  __syncthreads();
  if (warp == sh.order_w) {
    int need = sh.order_j2;
    for (int base = lo; base < hi; base += 32) {
      const int b = base + lane;
      const uint32_t m = __ballot_sync(0xFFFFFFFFu, b < hi && lane_cost(p, b) == c);
      const int n = __popc(m);
      if (need < n) {
        if (lane == 0) {
          uint32_t mm = m;
          for (int t = 0; t < need; ++t) mm &= mm - 1;  // drop the `need` lowest set bits
          sh.order_lane = base + __ffs(mm) - 1;
        }
        break;
      }
      need -= n;
    }
  }
  __syncthreads();
  return sh.order_lane;
}

// EXACT: the launch reports row statistics (row_stats is set), so sampled
// rows take the exact sweep; otherwise the lazy one.  One instantiation per
// mode keeps each kernel's code to the sweep it runs.
template <typename T, bool ALIGNED, bool EXACT>
__global__ void __launch_bounds__(kThreads, kConsumerWarps <= 8 ? 2 : 1) verify_accept_kernel(const VerifyParams p) {
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
  const bool leader = (rank == 0);
  int b = blockIdx.x / C;

  // ---- set-up that touches only shared memory (overlaps the previous kernel) ----
  // One thread per ring slot initialises its pair of barriers (another thread
  // the exchange barriers); each makes its initialisations visible to the
  // cluster's async proxy before the barrier that follows.
  if (tid < p.nslots - p.nslots % kGroups) {
    mbar_init(&sh.full[tid], 1);
    mbar_init(&sh.empty[tid], kPieces);
    fence_mbar_init();
  } else if (tid == 32 + kMaxSlots) {
    mbar_init(&sh.xbar, 1);
    mbar_init(&sh.dbar[0], 1);
    mbar_init(&sh.dbar[1], 1);
    sh.cta_flags = 0;
    sh.scan_flags = 0;
    fence_mbar_init();
  }
  if (tid <= kMaxDrafts) sh.gkey[tid] = 0ull;
  // The lane metadata may be read before the wait for the previous kernel on
  // the stream only when the caller says that kernel did not write it.
  const bool meta_early = (p.flags & SPEC_VERIFY_META_BEFORE_WAIT) != 0u;
  // Tests only: the producer never issues its last copy, so the waits for it
  // run out and the lane reports SPEC_ERR_TIMEOUT.
  const bool withhold_last = (p.flags & SPEC_VERIFY_TEST_WITHHOLD_COPY) != 0u;
  if (!meta_early) griddep_wait();
  if (p.order_by_cost) b = lane_of_rank(p, sh, b);

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
  if (meta_early) griddep_wait();  // logits and outputs only after the previous kernel
  // Let the next kernel on the stream start its set-up now.  It cannot begin
  // before every CTA of this grid has started and issued this, and it reads
  // nothing of ours before its own griddepcontrol.wait, which waits for this
  // whole grid to finish; issuing it late costs ~0.7 us at the end instead.
  if (tid == 0) griddep_launch_dependents();

  const int v0 = min(p.V, static_cast<int>(rank) * p.slice);
  const int v1 = min(p.V, v0 + p.slice);
  const int span = v1 - v0;
  const int body = ALIGNED ? (span / kVec) * kVec : 0;
  const int slot_elems = p.slot_bytes / kEsize;
  const int nslots = p.nslots - p.nslots % kGroups;  // a multiple of kGroups (host ensures >= kGroups)

  // Bytes this CTA will receive from its peers: their partial of every row
  // (leader of a greedy lane, or every CTA of a sampled lane), then for
  // sampled lanes their pass-2 slice sums.  Announced before this CTA arrives
  // on the cluster barrier, so before any peer can push.
  // (A greedy lane's peers send 16 bytes per row to the leader only.)
  // The thread that initialised these barriers arms them: no other thread is
  // ordered after their initialisation before the barrier below.
  if (tid == 32 + kMaxSlots) {
    const bool receives = sampled || leader;
    mbar_arrive_expect_tx(&sh.xbar, receives ? static_cast<uint32_t>((C - 1) * nstreams * 16) : 0u);
    if (sampled) {
      mbar_arrive_expect_tx(&sh.dbar[0], static_cast<uint32_t>((C - 1) * 16));
      mbar_arrive_expect_tx(&sh.dbar[1], static_cast<uint32_t>((C - 1) * 16));
    }
  }
  __syncthreads();  // barrier initialisation visible to every thread
  // Every CTA of the cluster has started once this phase completes; it is
  // waited on just before the first store into a peer's shared memory.
  cluster_arrive_relaxed();

  // Row of stream s: sampled lanes interleave target row j (even s) and drafter
  // row j (odd s); greedy lanes read target rows only.
  auto stream_row = [&](int s) -> const uint8_t* {
    const bool is_draft = sampled && (s & 1);
    const int j = sampled ? (s >> 1) : s;
    return (is_draft ? p.draft : p.target) + static_cast<int64_t>(off + j) * p.ld_bytes;
  };
  // Pass 1 streams the rows last to first: the row pair most likely to be
  // drawn from is the first rejected one, most often row 0, and streamed
  // last it is the most likely still to be in L2 when the draw re-reads it.
  // Position q of the pass-1 sequence is stream seq_stream(q).
  auto seq_stream = [&](int q) { return nstreams - 1 - q; };

  // ---- pass 1 ----
  if (warp == kProducerWarp && p.slot_bytes <= kParallelIssueSlotBytes) {
    // Small slots (short rows): lane g issues the chunks of consumer group g
    // (chunk i goes to slot i mod nslots, a multiple of kGroups, so each slot
    // is refilled by one lane only).  Issuing a copy costs about as much as
    // moving a few KB, so for small copies independent issuers win (a 1-lane
    // round of 4 KB rows: 2.95 -> 2.40 us); for large ones one lane issuing in
    // order lands the first chunks first and is faster.
    constexpr int nprod = kGroups;
    if (lane < nprod && ALIGNED && body > 0) {
      const int nch = (body + slot_elems - 1) / slot_elems;  // chunks per row
      const uint32_t ns = static_cast<uint32_t>(nslots);
      int s = lane / nch, ci = lane % nch;  // this lane's first chunk is chunk `lane`
      uint32_t slot = static_cast<uint32_t>(lane), par = 0;  // lane < nprod <= nslots
      uint32_t issued = 0;
      bool ok = true;
      while (s < nstreams) {
        if (withhold_last && s == nstreams - 1 && ci == nch - 1) break;
        const int c0 = ci * slot_elems;
        const int L = min(slot_elems, body - c0);
        if (!mbar_wait_bounded(&sh.empty[slot], par ^ 1u)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&sh.full[slot], static_cast<uint32_t>(L * kEsize));
        bulk_g2s(ring + static_cast<size_t>(slot) * p.slot_bytes,
                 stream_row(seq_stream(s)) + static_cast<int64_t>(v0 + c0) * kEsize, static_cast<uint32_t>(L * kEsize),
                 &sh.full[slot]);
        ++issued;
        ci += nprod;
        while (ci >= nch) {
          ci -= nch;
          ++s;
        }
        slot += nprod;
        if (slot >= ns) {
          slot -= ns;
          par ^= 1u;
        }
      }
      // Drain: this lane's last copies (one per slot it owns, newest first)
      // have landed before shared memory is reused; older ones were waited
      // on before their slot was refilled.
      const uint32_t window = ns / static_cast<uint32_t>(nprod);
      for (uint32_t m = 0; m < issued && m < window; ++m) {
        if (slot < static_cast<uint32_t>(nprod)) {
          slot += ns;
          par ^= 1u;
        }
        slot -= nprod;
        if (!mbar_wait_bounded(&sh.full[slot], par)) ok = false;
      }
      if (!ok) atomicOr(&sh.cta_flags, kTimedOut);
    }
  } else if (warp == kProducerWarp) {
    if (lane == 0 && ALIGNED) {
      uint32_t it = 0;
      bool ok = true;
      for (int s = 0; s < nstreams && ok; ++s) {
        const uint8_t* row = stream_row(seq_stream(s)) + static_cast<int64_t>(v0) * kEsize;
        for (int c0 = 0; c0 < body; c0 += slot_elems) {
          if (withhold_last && s == nstreams - 1 && c0 + slot_elems >= body) break;
          const int L = min(slot_elems, body - c0);
          const uint32_t slot = it % nslots;
          const uint32_t par = (it / nslots) & 1u;
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
      const uint32_t first = it > static_cast<uint32_t>(nslots) ? it - nslots : 0u;
      for (uint32_t i = first; i < it; ++i)
        if (!mbar_wait_bounded(&sh.full[i % nslots], (i / nslots) & 1u)) ok = false;
      if (!ok) atomicOr(&sh.cta_flags, kTimedOut);
    }
  } else if (warp == kHelperWarp) {
    // Draft tokens, the logits at them and the lane's uniforms, while the
    // slices stream in.  Lane j handles position j.
    if (status == SPEC_OK && lane <= k) {
      const int j = lane;
      if (j < k) {
        const int d = __ldg(p.draft_tokens + off + j);
        sh.drafts[j] = d;
        if (sampled && d >= 0 && d < p.V) {
          sh.xd_t[j] = ElemTraits<T>::load(p.target + static_cast<int64_t>(off + j) * p.ld_bytes, d);
          sh.xd_q[j] = ElemTraits<T>::load(p.draft + static_cast<int64_t>(off + j) * p.ld_bytes, d);
        }
      }
      if (sampled) {
        const float2 u = round_uniforms(p.seed, p.lane_base + static_cast<uint32_t>(b), static_cast<uint32_t>(j));
        sh.u_acc[j] = u.x;
        sh.u_smp[j] = u.y;
        // The scan's log2(u), split ahead of time.
        float iu = 0.f, fu = 0.f;
        if (u.x != 0.f) log2_parts(u.x, iu, fu);
        sh.u_l2i[j] = iu;
        sh.u_l2f[j] = fu;
      }
    }
    __syncwarp();
    const bool range_bad = status == SPEC_OK && lane < k && (sh.drafts[lane] < 0 || sh.drafts[lane] >= p.V);
    const bool any_bad = __any_sync(0xFFFFFFFFu, range_bad);
    if (lane == 0) sh.draft_range_bad = any_bad ? 1 : 0;
  } else {
    // Consumer warps.  The work items are (chunk, piece): chunk ch of the ring
    // sequence is split into kPieces ranges of vectors, and warp w takes items
    // w, w + kConsumerWarps, ...  Warps therefore work on different chunks at
    // once and only meet at the end.  A warp merges its lanes only when its
    // row changes.
    if (sampled)
      for (int s = 0; s < nstreams; ++s)
        if (lane == 0) sh.wpart[s][warp] = identity_partial();
    bool ok = true;
    // Sampled rows report their exact max and argmax only into row_stats.
    constexpr bool exact_stats = EXACT;
    if (ALIGNED && body > 0) {
      const int nch = (body + slot_elems - 1) / slot_elems;  // chunks per row
      int cur = -1;
      Acc a;
      acc_init(a);
      // Item (chunk ch, piece q) of warp w: q = w mod kPieces, ch = w / kPieces,
      // then every kGroups-th chunk; row s and chunk-in-row ci, ring slot and
      // phase parity advance with it.
      const int q = warp % kPieces;
      int s = (warp / kPieces) / nch, ci = (warp / kPieces) % nch;
      uint32_t slot = static_cast<uint32_t>(warp / kPieces), par = 0;  // first chunk < kGroups <= nslots
      for (; s < nstreams && ok;) {
        if (s != cur) {
          if (cur >= 0) {
            if (sampled) {
              const Partial wp = warp_merge<true>(a.m, a.s, a.idx, acc_bad(a), c);
              if (lane == 0) sh.wpart[seq_stream(cur)][warp] = wp;
            } else {
              fold_greedy_row(sh, seq_stream(cur), a.m, a.idx, acc_bad(a), lane);
            }
          }
          acc_init(a);
          cur = s;
        }
        if (!mbar_wait_bounded(&sh.full[slot], par)) {
          ok = false;
          break;
        }
        const uint4* sv = reinterpret_cast<const uint4*>(ring + static_cast<size_t>(slot) * p.slot_bytes);
        const int c0 = ci * slot_elems;
        const int nvec = min(slot_elems, body - c0) / kVec;
        const int per = (nvec + kPieces - 1) / kPieces;
        const int vb = min(nvec, q * per), ve = min(nvec, vb + per);
        if (sampled && exact_stats) acc_range<T, true, false>(a, sv, vb, ve, v0 + c0, c, lane);
        else if (sampled) acc_range<T, true, true>(a, sv, vb, ve, v0 + c0, c, lane);
        else acc_range<T, false>(a, sv, vb, ve, v0 + c0, c, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.empty[slot]);
        ci += kGroups;
        while (ci >= nch) {
          ci -= nch;
          ++s;
        }
        slot += kGroups;
        if (slot >= static_cast<uint32_t>(nslots)) {
          slot -= nslots;
          par ^= 1u;
        }
      }
      if (cur >= 0) {
        const uint32_t fl = acc_bad(a) | (ok ? 0u : kTimedOut);
        if (sampled) {
          const Partial wp = warp_merge<true>(a.m, a.s, a.idx, fl, c);
          if (lane == 0) sh.wpart[seq_stream(cur)][warp] = wp;
        } else {
          fold_greedy_row(sh, seq_stream(cur), a.m, a.idx, fl, lane);
        }
      }
    }
    // Elements outside the bulk-copied body: the row tail, or the whole slice
    // when rows are not 16-byte aligned.  Each warp folds them into its own
    // entry of every row.
    if (span > body && ok) {
      for (int s = 0; s < nstreams; ++s) {
        const uint8_t* row = stream_row(s);
        Acc a;
        acc_init(a);
        for (int e = body + tid; e < span; e += kConsumers) {
          const float x = ElemTraits<T>::load(row, v0 + e);
          if (sampled) acc_scalar<true>(a, x, v0 + e, c);
          else acc_scalar<false>(a, x, v0 + e, c);
        }
        if (sampled) {
          const Partial wp = warp_merge<true>(a.m, a.s, a.idx, acc_bad(a), c);
          if (lane == 0) {
            Partial o = sh.wpart[s][warp];
            merge_part<true>(o.m, o.s, o.idx, wp.m, wp.s, wp.idx, c);
            o.flags |= wp.flags;
            sh.wpart[s][warp] = o;
          }
        } else {
          fold_greedy_row(sh, s, a.m, a.idx, acc_bad(a), lane);
        }
      }
    }
    if (!ok && lane == 0) atomicOr(&sh.cta_flags, kTimedOut);
  }
  __syncthreads();

  // ---- greedy lanes: the leader gathers every CTA's row keys and finishes ----
  if (!sampled) {
    cluster_wait_acquire();  // every peer is running: its shared memory may be written
    if (warp != 0) return;
    const uint32_t fl = sh.cta_flags;
    if (!leader) {
      // Lane s sends this CTA's key of row s, with the CTA's flags, into
      // the leader's slot of this CTA.
      if (lane < nstreams) {
        const unsigned long long key = sh.gkey[lane];
        st_async_v4(cluster_map(&sh.cpart[rank][lane], 0), static_cast<uint32_t>(key),
                    static_cast<uint32_t>(key >> 32), fl, 0u, cluster_map(&sh.xbar, 0));
      }
      return;
    }
    const bool waited = mbar_wait_bounded(&sh.xbar, 0, kExchangeWaitLimitNs);
    unsigned long long key = 0ull;
    uint32_t flags = fl | (waited ? 0u : kTimedOut);
    if (lane < nstreams) {
      key = sh.gkey[lane];
      for (int r = 1; r < C; ++r) {
        const uint4 e = *reinterpret_cast<const uint4*>(&sh.cpart[r][lane]);
        const unsigned long long kr = (static_cast<unsigned long long>(e.y) << 32) | e.x;
        key = kr > key ? kr : key;
        flags |= e.z;
      }
    }
    greedy_finish(p, sh.drafts, b, k, off, status, key, __reduce_or_sync(0xFFFFFFFFu, flags), lane);
    return;
  }

  // ---- sampled lanes: this CTA's partial of every row ----
  if (warp < kConsumerWarps) {
    for (int s = warp; s < nstreams; s += kConsumerWarps) {
      const Partial q = (lane < kConsumerWarps) ? sh.wpart[s][lane] : identity_partial();
      const Partial r = warp_merge<true>(q.m, q.s, q.idx, q.flags, c);
      if (lane == 0) sh.fin[s] = r;
    }
  }
  __syncthreads();
  cluster_wait_acquire();  // every peer is running: its shared memory may be written
  push_partials(sh, nstreams, C, rank, sh.cta_flags);

  // ---- the lane's totals ----
  if (tid == 0 && !mbar_wait_bounded(&sh.xbar, 0, kExchangeWaitLimitNs)) atomicOr(&sh.cta_flags, kTimedOut);
  __syncthreads();
  if (warp < kConsumerWarps) {
    for (int s = warp; s < nstreams; s += kConsumerWarps) {
      const Partial q = (lane < C) ? sh.cpart[lane][s] : identity_partial();
      const Partial r = warp_merge<true>(q.m, q.s, q.idx, q.flags, c);
      if (lane == 0) {
        sh.fin[s] = r;
        const uint32_t f = r.flags | ((r.idx == INT_MAX) ? kEmptyRow : 0u);
        if (f) atomicOr(&sh.scan_flags, f);
      }
    }
  }
  __syncthreads();

  // ---- acceptance scan (warp 0; lane j handles position j) ----
  // The draft range check, the split log2 of each uniform and the rows'
  // flags are ready before it starts; each lane also forms the draw
  // coefficients of its own rows, so that the chosen row's only need a
  // shuffle once the scan knows it.
  if (warp == 0) {
    int st = status;
    if (st == SPEC_OK && sh.draft_range_bad) st = SPEC_ERR_TOKEN_RANGE;
    if (st == SPEC_OK) {
      const uint32_t all = sh.scan_flags | sh.cta_flags;
      if (all & kTimedOut) st = SPEC_ERR_TIMEOUT;
      else if (all & (kBadValue | kEmptyRow)) st = SPEC_ERR_NONFINITE;
    }

    int n = 0, mode = kNoDraw;
    // log2 p_j(d) and log2 q_j(d) at this lane's position, and the test
    // log2(u) < log2 p - log2 q, as one compensated fp32 sum of exact terms:
    // its rounding error is far below the ~1e-6 relative error of the sums S.
    float lp = NAN, lq = NAN;
    float cmp = 0.f, clp = 0.f, cmq = 0.f, clq = 0.f;  // this lane's rows' draw coefficients
    if (st == SPEC_OK) {
      const bool active = lane < k;
      bool accept = true;
      if (lane <= k) {
        const Partial pt = sh.fin[2 * lane];
        cmp = scaled_ref(pt.m, c);
        clp = log2f(pt.s);
      }
      if (active) {
        const Partial pq = sh.fin[2 * lane + 1];
        cmq = scaled_ref(pq.m, c);
        clq = log2f(pq.s);
        const float xt = sh.xd_t[lane], xq = sh.xd_q[lane];
        CompSum dp = log2_prob_terms(xt, sh.fin[2 * lane], c);
        const CompSum dq = log2_prob_terms(xq, pq, c);
        lp = (xt == -INFINITY) ? -INFINITY : dp.value();
        lq = (xq == -INFINITY) ? -INFINITY : dq.value();
        const float u = sh.u_acc[lane];
        if (xt == -INFINITY) {
          accept = false;  // p(d) = 0
        } else if (xq == -INFINITY || u == 0.f) {
          accept = true;   // q(d) = 0, or log2(u) = -inf
        } else {
          dp.add(-dq.s);
          dp.add(-dq.c);
          dp.add(-sh.u_l2i[lane]);
          dp.add(-sh.u_l2f[lane]);
          accept = dp.value() > 0.f;
        }
      }
      const uint32_t mask = __ballot_sync(0xFFFFFFFFu, active && !accept);
      n = mask ? (__ffs(mask) - 1) : k;
      mode = (n < k) ? kResidual : kBonus;
    }
    // The draw re-reads this CTA's slice of one row pair; on rounds larger
    // than L2 part of it may have left L2 since pass 1: fetch it back now.
    if (lane == 0 && ALIGNED && st == SPEC_OK && body > 0) {
      const int drow = (mode == kResidual) ? n : k;
      const int64_t col = static_cast<int64_t>(v0) * kEsize;
      bulk_prefetch_l2(p.target + static_cast<int64_t>(off + drow) * p.ld_bytes + col,
                       static_cast<uint32_t>(body * kEsize));
      if (mode == kResidual)
        bulk_prefetch_l2(p.draft + static_cast<int64_t>(off + n) * p.ld_bytes + col,
                         static_cast<uint32_t>(body * kEsize));
    }
    const int src = (mode == kResidual) ? n : k;
    const float mp = __shfl_sync(0xFFFFFFFFu, cmp, src & 31), l2sp = __shfl_sync(0xFFFFFFFFu, clp, src & 31);
    const float mq = __shfl_sync(0xFFFFFFFFu, cmq, src & 31), l2sq = __shfl_sync(0xFFFFFFFFu, clq, src & 31);
    if (lane == 0) {
      sh.scan_n = n;
      sh.scan_mode = (st == SPEC_OK) ? mode : kNoDraw;
      sh.scan_st = st;
      if (st == SPEC_OK) {
        // As draw_coef_store writes them for target row src (and drafter
        // row n for a residual draw).
        sh.dcoef[0] = mp;
        sh.dcoef[1] = l2sp;
        sh.dcoef[2] = (mode == kResidual) ? mq : 0.f;
        sh.dcoef[3] = (mode == kResidual) ? l2sq : 0.f;
        sh.dcoef[4] = c;
      }
    }
    if (lane <= kMaxDrafts) {
      sh.scan_lp[lane] = lp;
      sh.scan_lq[lane] = lq;
    }
  }
  __syncthreads();

  // ---- outputs (leader, by the helper warp, which has no part in the draw sums) ----
  if (warp == kHelperWarp && leader) {
    const int st = sh.scan_st, n = sh.scan_n, mode = sh.scan_mode;
    const bool layout_ok = (status != SPEC_ERR_LAYOUT);
    if (lane == 0) {
      p.committed[b] = (st == SPEC_OK) ? n + 1 : 0;
      if (p.lane_status) p.lane_status[b] = st;
    }
    for (int j = lane; layout_ok && j <= k; j += 32) {
      const int tok = (st == SPEC_OK && j < n) ? sh.drafts[j] : -1;
      const bool drawn_here = (st == SPEC_OK) && j == n;
      if (!drawn_here) p.out_tokens[off + j] = tok;
      if (p.row_stats && st == SPEC_OK) {
        spec_row_stats* rs = p.row_stats + off + j;
        const Partial pt = sh.fin[2 * j];
        rs->argmax = pt.idx;
        rs->max_logit = pt.m;
        float ip, fp;
        log2_parts(pt.s, ip, fp);
        CompSum l;
        l.add(scaled_ref(pt.m, c));
        l.add(ip);
        l.add(fp);
        rs->lse = __fmul_rn(l.value(), kLn2);
        rs->logp_d = (j < k) ? __fmul_rn(sh.scan_lp[j], kLn2) : NAN;
        rs->logq_d = (j < k) ? __fmul_rn(sh.scan_lq[j], kLn2) : NAN;
        if (!(drawn_here && mode == kResidual)) rs->resid_mass = NAN;
        if (!drawn_here) rs->drawn = -1;
        rs->flags = 1 | (drawn_here ? (mode == kResidual ? 2 : 4) : 0);
      }
    }
  }

  if (sh.scan_mode == kNoDraw) return;

  // ---- pass 2: draw the model's token (sampled lanes, whole cluster) ----
  const int n = sh.scan_n;
  bool residual = (sh.scan_mode == kResidual);
  int draw_row = residual ? n : k;  // target row whose p enters the weights
  const uint8_t* qrow = p.draft + static_cast<int64_t>(off + n) * p.ld_bytes;
  const float uprime = sh.u_smp[n];
  // Each consumer warp takes one segment of the slice (a multiple of 8
  // elements, so rounds start 16-byte aligned; the last round may be partial).
#ifndef SPEC_VERIFY_SEG_ROUND
#define SPEC_VERIFY_SEG_ROUND 256
#endif
  const int seg = ((span + kConsumerWarps - 1) / kConsumerWarps + SPEC_VERIFY_SEG_ROUND - 1) /
                  SPEC_VERIFY_SEG_ROUND * SPEC_VERIFY_SEG_ROUND;
  // Every lane's total of every round of its warp's segment is kept in the
  // ring (free after pass 1), so that the walk re-reads one lane's eight
  // elements only.  Unaligned launches have no ring; they, and segments with
  // more rounds than fit, recompute the round totals they walk over.
  const int seg_rounds = (seg + kDrawRound - 1) / kDrawRound;
  float* lane_sums = reinterpret_cast<float*>(ring);
  const bool keep_rounds = ALIGNED && static_cast<int64_t>(seg_rounds) * kConsumerWarps * 32 * 4 <=
                                          static_cast<int64_t>(nslots) * p.slot_bytes;
  auto seg_lsum = [&](int w) -> float* {
    return keep_rounds ? lane_sums + static_cast<int64_t>(w) * seg_rounds * 32 : nullptr;
  };
  // Each consumer warp's staging buffer follows the kept lane totals.
  const int64_t lsum_bytes =
      keep_rounds ? (static_cast<int64_t>(seg_rounds) * kConsumerWarps * 32 * 4 + 127) / 128 * 128 : 0;
  const bool stage_fits = kDrawStaged && ALIGNED &&
                          lsum_bytes + static_cast<int64_t>(draw_stage_bytes<T>()) * kConsumerWarps <=
                              static_cast<int64_t>(nslots) * p.slot_bytes;
  uint8_t* const stage =
      (stage_fits && warp < kConsumerWarps) ? ring + lsum_bytes + static_cast<int64_t>(draw_stage_bytes<T>()) * warp
                                            : nullptr;

  float W = 0.f;
  float resid_mass = NAN;
  float dsum = 0.f, dincl = 0.f;  // lane r: CTA r's draw sum, and the running total through CTA r
  int buf = 0;
  for (int attempt = 0; attempt < 2; ++attempt) {
    buf = attempt;
    const DrawCoef kc = draw_coef_load(sh.dcoef);
    const uint8_t* trow = p.target + static_cast<int64_t>(off + draw_row) * p.ld_bytes;
    if (warp < kConsumerWarps) {
      const int s0 = v0 + warp * seg;
      const int s1 = min(v1, s0 + seg);
      const float segw = residual
                             ? draw_segment_sum<T, ALIGNED, true>(kc, trow, qrow, s0, s1, seg_lsum(warp), lane, stage)
                             : draw_segment_sum<T, ALIGNED, false>(kc, trow, qrow, s0, s1, seg_lsum(warp), lane, stage);
      if (lane == 0) sh.segsum[warp] = segw;
    }
    __syncthreads();
    if (warp == 0) {
      // The CTA's sum by the same scan across the lanes (lane w: warp w's
      // segment) that later picks the walking warp, so the two agree.
      float wc = (lane < kConsumerWarps) ? sh.segsum[lane] : 0.f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float up = __shfl_up_sync(0xFFFFFFFFu, wc, o);
        if (lane >= o) wc = __fadd_rn(up, wc);
      }
      wc = __shfl_sync(0xFFFFFFFFu, wc, kConsumerWarps - 1);
      if (tid == static_cast<int>(rank)) {
        sh.dpart[buf][rank] = DrawPartial{wc, 0, 0, 0};
      } else if (tid < C) {
        st_async_v4(cluster_map(&sh.dpart[buf][rank], tid), __float_as_uint(wc), 0u, 0u, 0u,
                    cluster_map(&sh.dbar[buf], tid));
      }
    }
    if (tid == 0 && !mbar_wait_bounded(&sh.dbar[buf], 0, kExchangeWaitLimitNs)) {
      // A peer's draw sum never came: the lane's outputs (already written as
      // OK by the leader) cannot be trusted.
      atomicOr(&sh.cta_flags, kTimedOut);
      if (leader) {
        p.committed[b] = 0;
        if (p.lane_status) p.lane_status[b] = SPEC_ERR_TIMEOUT;
      }
    }
    __syncthreads();

    dsum = (lane < C) ? sh.dpart[buf][lane].w : 0.f;
    dincl = dsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float up = __shfl_up_sync(0xFFFFFFFFu, dincl, o);
      if (lane >= o) dincl = __fadd_rn(up, dincl);
    }
    W = __shfl_sync(0xFFFFFFFFu, dincl, C - 1);
    if (residual) resid_mass = __fmul_rn(W, ex2_approx(-sh.dcoef[1]));  // W / S_p
    if (W > 0.f || !residual) break;
    // The residual max(0, p_n - q_n) has no mass: draw from p_n instead.
    residual = false;
    draw_row = n;
    if (tid == 0) draw_coef_store(sh.dcoef, sh.fin, n, -1, c);
    __syncthreads();
  }

  // The CTA holding the crossing of u' * W (cumulative sums in CTA order, by
  // the scan across the lanes above), and in it the warp whose segment holds
  // it; where rounding leaves no crossing, the last element of positive
  // weight (in the last CTA, and then the last warp, holding weight).
  const float target = __fmul_rn(uprime, W);
  const uint32_t cta_past = __ballot_sync(0xFFFFFFFFu, lane < C && dincl > target);
  const int owner = cta_past ? (__ffs(cta_past) - 1) : -1;
  const float prefix_l = __shfl_sync(0xFFFFFFFFu, dincl, (owner > 0) ? owner - 1 : 0);
  const float prefix = (owner > 0) ? prefix_l : 0.f;
  auto last_warp_with_weight = [&]() {
    int lw = -1;
    for (int w = 0; w < kConsumerWarps; ++w)
      if (sh.segsum[w] > 0.f) lw = w;
    return lw;
  };
  int fw = -1;         // the warp that finds the token in this CTA
  float tau_w = -1.f;  // its threshold within its segment (< 0: the last positive weight)
  if (owner < 0) {
    const uint32_t pos = __ballot_sync(0xFFFFFFFFu, lane < C && dsum > 0.f);
    const int last_r = pos ? (31 - __clz(pos)) : -1;
    if (last_r == static_cast<int>(rank)) fw = last_warp_with_weight();
  } else if (owner == static_cast<int>(rank)) {
    // The warp segments' running totals by one scan across the lanes (lane w
    // holds warp w's sum), the first past tau by a ballot.
    const float tau = __fsub_rn(target, prefix);
    const float sw = (lane < kConsumerWarps) ? sh.segsum[lane] : 0.f;
    float incl = sw;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float up = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl = __fadd_rn(up, incl);
    }
    const uint32_t hit = __ballot_sync(0xFFFFFFFFu, lane < kConsumerWarps && incl > tau);
    const float before = __shfl_sync(0xFFFFFFFFu, incl, hit ? max(__ffs(hit) - 2, 0) : 0);
    if (hit) {
      fw = __ffs(hit) - 1;
      tau_w = (fw > 0) ? __fsub_rn(tau, before) : tau;
    } else {
      fw = last_warp_with_weight();
    }
  }
  if (fw >= 0 && warp == fw) {
    const DrawCoef kc = draw_coef_load(sh.dcoef);
    const uint8_t* trow = p.target + static_cast<int64_t>(off + draw_row) * p.ld_bytes;
    const int s0 = v0 + warp * seg;
    const int s1 = min(v1, s0 + seg);
    int token = -2;
    if (tau_w >= 0.f)
      token = residual ? draw_walk<T, ALIGNED, true>(kc, trow, qrow, s0, s1, seg_lsum(warp), tau_w, lane)
                       : draw_walk<T, ALIGNED, false>(kc, trow, qrow, s0, s1, seg_lsum(warp), tau_w, lane);
    if (token == -2)
      token = residual ? draw_last_positive<T, ALIGNED, true>(kc, trow, qrow, s0, s1, seg_lsum(warp), lane)
                       : draw_last_positive<T, ALIGNED, false>(kc, trow, qrow, s0, s1, seg_lsum(warp), lane);
    if (lane == 0) {
      p.out_tokens[off + n] = token;
      if (p.row_stats) {
        spec_row_stats* rs = p.row_stats + off + n;
        rs->drawn = token;
        if (sh.scan_mode == kResidual) rs->resid_mass = resid_mass;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Small rounds
// ---------------------------------------------------------------------------
// Rounds without drafter logits whose rows are a few KB (every lane greedy;
// a sampled lane reports SPEC_ERR_INVALID_ARG, as in the cluster kernel): one
// CTA per lane, in which warp j reads row j with plain 16-byte loads, eight
// in flight per lane, and reduces each batch of eight as a tree in registers,
// then the warp by shuffles -- no cluster,
// ring or mbarrier, and every row of the lane in flight at once.  The row
// keys (order-preserving max bits over the complemented index), the statuses
// and the outputs are the cluster kernel's (argmax_key, greedy_finish), so
// both give the same bits.
constexpr int kSmallThreads = 32 * (kMaxDrafts + 1);
constexpr int kSmallBatch = 8;  // vectors a lane loads before reducing them

template <typename T, bool ALIGNED>
__global__ void __launch_bounds__(kSmallThreads) verify_small_kernel(const VerifyParams p) {
  constexpr int kVec = ElemTraits<T>::kVec;
  __shared__ unsigned long long keys[kMaxDrafts + 1];
  __shared__ uint32_t rflags[kMaxDrafts + 1];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x;

  // The lane metadata may be read before the wait for the previous kernel on
  // the stream only when the caller says that kernel did not write it.
  const bool meta_early = (p.flags & SPEC_VERIFY_META_BEFORE_WAIT) != 0u;
  if (!meta_early) griddep_wait();
  const int k = __ldg(p.draft_lens + b);
  const int off = __ldg(p.row_offsets + b);
  const int off_end = __ldg(p.row_offsets + b + 1);
  const bool sampled = __ldg(p.temps + b) > 0.f;
  int status = SPEC_OK;
  if (k < 0 || off < 0 || off_end > p.rows || off_end - off != k + 1) {
    status = SPEC_ERR_LAYOUT;
  } else if (k > kMaxDrafts) {
    status = SPEC_ERR_UNSUPPORTED;
  } else if (sampled && p.draft == nullptr) {
    status = SPEC_ERR_INVALID_ARG;
  }
  const bool ok = (status == SPEC_OK) && !sampled;
  // Lane j of warp 0 holds draft j (lane metadata too) and checks its range.
  const int draft = (ok && tid < k) ? __ldg(p.draft_tokens + off + tid) : 0;
  const bool any_range_bad = __any_sync(0xFFFFFFFFu, ok && tid < k && (draft < 0 || draft >= p.V));
  if (meta_early) griddep_wait();  // logits and outputs only after the previous kernel
  if (tid == 0) griddep_launch_dependents();

  if (ok && warp <= k) {
    const uint8_t* row = p.target + static_cast<int64_t>(off + warp) * p.ld_bytes;
    float m = -INFINITY;
    int idx = INT_MAX;
    uint32_t bad = 0;
    // Elements in increasing index order per lane; a strictly larger value
    // takes over, so each lane keeps its lowest index of its max.
    auto take = [&](float x, int e) {
      bad |= !(x <= FLT_MAX) ? 1u : 0u;
      if (x > m) {
        m = x;
        idx = e;
      }
    };
    int e0 = 0;
    if (ALIGNED) {
      const int nvec = p.V / kVec;
      const uint4* rv = reinterpret_cast<const uint4*>(row);
      // A batch is reduced as a tree, not element by element: its max with
      // NaN propagated (a NaN or +inf flags the row), then the lowest index
      // holding that max; a batch takes over only with a strictly larger max,
      // since earlier batches hold lower indices.  Vectors past the row read
      // as -inf, which is never taken.
      const uint32_t ninf = (kVec == 8) ? 0xFF80FF80u : 0xFF800000u;
      for (int v0 = lane; v0 < nvec; v0 += 32 * kSmallBatch) {
        uint4 x[kSmallBatch];
#pragma unroll
        for (int u = 0; u < kSmallBatch; ++u)
          x[u] = (v0 + 32 * u < nvec) ? __ldg(rv + v0 + 32 * u) : make_uint4(ninf, ninf, ninf, ninf);
        float vm[kSmallBatch];
#pragma unroll
        for (int u = 0; u < kSmallBatch; ++u) {
          vm[u] = vec_elem<T>(x[u], 0);
#pragma unroll
          for (int t = 1; t < kVec; ++t) vm[u] = f32_max_nan(vm[u], vec_elem<T>(x[u], t));
        }
#pragma unroll
        for (int w = kSmallBatch / 2; w > 0; w /= 2)
#pragma unroll
          for (int u = 0; u < w; ++u) vm[u] = f32_max_nan(vm[u], vm[u + w]);
        const float mb = vm[0];
        bad |= !(mb <= FLT_MAX) ? 1u : 0u;
        if (mb > m) {
          int vi[kSmallBatch];
#pragma unroll
          for (int u = 0; u < kSmallBatch; ++u) {
            vi[u] = INT_MAX;
#pragma unroll
            for (int t = kVec - 1; t >= 0; --t)
              if (vec_elem<T>(x[u], t) == mb) vi[u] = (v0 + 32 * u) * kVec + t;
          }
#pragma unroll
          for (int w = kSmallBatch / 2; w > 0; w /= 2)
#pragma unroll
            for (int u = 0; u < w; ++u) vi[u] = min(vi[u], vi[u + w]);
          m = mb;
          idx = vi[0];
        }
      }
      e0 = nvec * kVec;
    }
    for (int e = e0 + lane; e < p.V; e += 32) take(ElemTraits<T>::load(row, e), e);
    // The warp's largest key: the high words first, then the low words among them.
    const unsigned long long key = argmax_key(m, idx);
    const uint32_t hi = __reduce_max_sync(0xFFFFFFFFu, static_cast<uint32_t>(key >> 32));
    const uint32_t lo = __reduce_max_sync(0xFFFFFFFFu, (static_cast<uint32_t>(key >> 32) == hi)
                                                           ? static_cast<uint32_t>(key) : 0u);
    bad = __reduce_or_sync(0xFFFFFFFFu, bad);
    if (lane == 0) {
      keys[warp] = (static_cast<unsigned long long>(hi) << 32) | lo;
      rflags[warp] = bad ? kBadValue : 0u;
    }
  }
  __syncthreads();
  if (warp != 0) return;
  // The acceptance scan and outputs, as greedy_finish writes them for the
  // cluster kernel (no waits here, so no time-out), with the draft tokens
  // already in registers.
  const bool has_row = ok && lane <= k;
  const unsigned long long key = has_row ? keys[lane] : 0ull;
  const bool nonfinite = __any_sync(0xFFFFFFFFu, has_row && (rflags[lane] != 0u || key == 0ull));
  float m;
  int a;
  argmax_key_decode(key, m, a);
  int st = status;
  if (st == SPEC_OK) {
    if (any_range_bad) st = SPEC_ERR_TOKEN_RANGE;
    else if (nonfinite) st = SPEC_ERR_NONFINITE;
  }
  const uint32_t stops = __ballot_sync(0xFFFFFFFFu, ok && lane < k && draft != a);
  const int n = (st != SPEC_OK) ? 0 : stops ? (__ffs(stops) - 1) : k;
  if (lane == 0) {
    p.committed[b] = (st == SPEC_OK) ? n + 1 : 0;
    if (p.lane_status) p.lane_status[b] = st;
  }
  if (status == SPEC_ERR_LAYOUT) return;
  for (int j = lane; j <= k; j += 32) {
    p.out_tokens[off + j] = (st == SPEC_OK && j <= n) ? a : -1;
    if (p.row_stats && st == SPEC_OK) {
      spec_row_stats* rs = p.row_stats + off + j;
      rs->argmax = a;
      rs->max_logit = m;
      rs->lse = NAN;
      rs->logp_d = NAN;
      rs->logq_d = NAN;
      rs->resid_mass = NAN;
      rs->drawn = -1;
      rs->flags = 1;
    }
  }
}

}  // namespace specv
