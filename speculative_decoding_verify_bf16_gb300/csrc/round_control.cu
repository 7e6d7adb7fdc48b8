// round_control.cu -- acceptance counts, the per-lane miss back-off, the
// copy-from-the-conversation drafter and per-row logit penalties: the C ABI of
// include/spec_round_control.h.
// All run on the device next to the verify kernel; none allocates memory.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "spec_round_control.h"

namespace {

constexpr int kSlots = SPEC_MAX_DRAFTS;
constexpr int kCountWords = 3 + 2 * kSlots;  // spec_accept_counts as 64-bit words
static_assert(sizeof(spec_accept_counts) == kCountWords * 8, "spec_accept_counts layout");

constexpr int kMissesToWait = 4;   // passes in a row with nothing kept before a wait
constexpr int kFirstWait = 16;     // passes of the first wait
constexpr int kLongestWait = 256;  // the wait doubles up to this

// Whether lane b's round is counted, and its guesses proposed (k) and kept (n).
__device__ __forceinline__ bool lane_round(const int32_t* committed, const int32_t* draft_lens,
                                           const int32_t* lane_status, int b, int& k, int& n) {
  if (lane_status != nullptr && lane_status[b] != SPEC_OK) return false;
  k = draft_lens[b];
  const int c = committed[b];
  if (k < 0 || k > kSlots || c < 1 || c > k + 1) return false;
  n = c - 1;
  return true;
}

// The whole batch into one struct: per-thread partial counts, then warp sums,
// shared-memory sums per CTA and one 64-bit atomic per word and CTA.
__global__ void __launch_bounds__(256) accept_counts_batch_kernel(const int32_t* committed,
                                                                  const int32_t* draft_lens,
                                                                  const int32_t* lane_status, int32_t lanes,
                                                                  unsigned long long* out) {
  __shared__ unsigned long long tot[kCountWords];
  for (int i = threadIdx.x; i < kCountWords; i += blockDim.x) tot[i] = 0ull;
  __syncthreads();
  unsigned int part[kCountWords];
#pragma unroll
  for (int i = 0; i < kCountWords; ++i) part[i] = 0u;
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < lanes; b += gridDim.x * blockDim.x) {
    int k, n;
    if (!lane_round(committed, draft_lens, lane_status, b, k, n)) continue;
    part[0] += 1u;
    part[1] += static_cast<unsigned int>(k);
    part[2] += static_cast<unsigned int>(n);
#pragma unroll
    for (int j = 0; j < kSlots; ++j) {
      part[3 + j] += (k > j) ? 1u : 0u;
      part[3 + kSlots + j] += (n > j) ? 1u : 0u;
    }
  }
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < kCountWords; ++i) {
    const unsigned int w = __reduce_add_sync(0xFFFFFFFFu, part[i]);
    if (lane == 0 && w != 0u) atomicAdd(&tot[i], static_cast<unsigned long long>(w));
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kCountWords; i += blockDim.x)
    if (tot[i] != 0ull) atomicAdd(&out[i], tot[i]);
}

// Lane b into counts[b] (one thread per lane owns its struct).
__global__ void accept_counts_lane_kernel(const int32_t* committed, const int32_t* draft_lens,
                                          const int32_t* lane_status, int32_t lanes, unsigned long long* out) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= lanes) return;
  int k, n;
  if (!lane_round(committed, draft_lens, lane_status, b, k, n)) return;
  unsigned long long* c = out + static_cast<int64_t>(b) * kCountWords;
  c[0] += 1ull;
  c[1] += static_cast<unsigned long long>(k);
  c[2] += static_cast<unsigned long long>(n);
  for (int j = 0; j < k; ++j) c[3 + j] += 1ull;
  for (int j = 0; j < n; ++j) c[3 + kSlots + j] += 1ull;
}

__global__ void backoff_init_kernel(spec_backoff_state* states, int32_t lanes) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < lanes) states[b] = spec_backoff_state{0, kFirstWait, 0, 0};
}

// One pass for every lane (mashbox docs, "Speculative decoding" -- "What it
// does for you"), read with one pass per device call.  A single CTA: first
// whether any lane of the batch guessed (a round that does not speculate
// counts toward no miss run), then each lane's state.
__global__ void __launch_bounds__(1024) backoff_step_kernel(spec_backoff_state* states, const int32_t* proposed,
                                                            const int32_t* committed, const int32_t* lane_status,
                                                            int32_t lanes, int32_t draft_tokens,
                                                            int32_t* next_draft_lens) {
  int guessed = 0;
  for (int b = threadIdx.x; b < lanes; b += blockDim.x) guessed |= (proposed[b] > 0) ? 1 : 0;
  const bool speculates = __syncthreads_or(guessed) != 0;
  for (int b = threadIdx.x; b < lanes; b += blockDim.x) {
    spec_backoff_state s = states[b];
    if (s.wait > 0) {
      s.wait -= 1;  // every pass of a waiting lane counts toward its wait
    } else if (speculates) {
      const bool ok = (lane_status == nullptr || lane_status[b] == SPEC_OK);
      const bool kept = ok && proposed[b] > 0 && committed[b] > 1;
      if (kept) {
        s.misses = 0;
        s.backoff = kFirstWait;
      } else if (++s.misses == kMissesToWait) {
        s.wait = s.backoff;
        s.backoff = min(2 * s.backoff, kLongestWait);
        s.misses = 0;
      }
    }
    states[b] = s;
    next_draft_lens[b] = (s.wait > 0) ? 0 : draft_tokens;
  }
}

constexpr int kNgramThreads = 256;

// Copy from the conversation (mashbox docs, "Speculative decoding" --
// "Options", --speculation ngram), one CTA per lane.  Every end position i of
// the history gets the length of its backward match against the suffix (up to
// mm tokens); the best is the longest match of at least match_min tokens,
// latest position on ties, found as the max of (length << 40 | i).
__global__ void __launch_bounds__(kNgramThreads) ngram_draft_kernel(const int32_t* tokens,
                                                                   const int64_t* hist_offsets, int32_t k,
                                                                   int32_t match_min, int32_t match_max,
                                                                   int32_t* drafts, int32_t draft_stride,
                                                                   int32_t* draft_lens) {
  __shared__ int32_t suffix[SPEC_NGRAM_MAX_MATCH];
  __shared__ unsigned long long best;
  const int b = blockIdx.x;
  const int64_t o0 = hist_offsets[b], o1 = hist_offsets[b + 1];
  const int64_t L = (o1 > o0) ? o1 - o0 : 0;
  const int32_t* h = tokens + o0;
  const int mm = static_cast<int>(L - 1 < match_max ? L - 1 : match_max);  // longest usable match
  if (k == 0 || mm < match_min) {  // nothing can match (includes L < 2)
    if (threadIdx.x == 0) draft_lens[b] = 0;
    return;
  }
  if (threadIdx.x < mm) suffix[threadIdx.x] = h[L - mm + threadIdx.x];
  if (threadIdx.x == 0) best = 0ull;
  __syncthreads();
  unsigned long long mine = 0ull;
  // End positions i in [match_min, L - 1]; the match at i compares h[i - 1 - j]
  // with the suffix's token L - 1 - j.
  for (int64_t i = match_min + threadIdx.x; i < L; i += kNgramThreads) {
    const int lim = static_cast<int>(i < mm ? i : mm);
    int m = 0;
    while (m < lim && h[i - 1 - m] == suffix[mm - 1 - m]) ++m;
    if (m >= match_min) {
      const unsigned long long key = (static_cast<unsigned long long>(m) << 40) | static_cast<unsigned long long>(i);
      mine = key > mine ? key : mine;
    }
  }
  if (mine != 0ull) atomicMax(&best, mine);
  __syncthreads();
  const unsigned long long key = best;
  if (key == 0ull) {
    if (threadIdx.x == 0) draft_lens[b] = 0;
    return;
  }
  const int64_t i = static_cast<int64_t>(key & ((1ull << 40) - 1));
  const int n = static_cast<int>((L - i) < k ? (L - i) : k);
  if (threadIdx.x < n) drafts[static_cast<int64_t>(b) * draft_stride + threadIdx.x] = h[i + threadIdx.x];
  if (threadIdx.x == 0) draft_lens[b] = n;
}

// Per-row presence / frequency penalties (FreeToken #828, PR #836), one CTA
// per lane.  Row j's count of a token is its history count plus its count
// among d_1..d_j.  Threads take (row, history entry) pairs of all the lane's
// rows at once, and (row, draft) pairs for the first occurrence of each draft
// d_1..d_j that is not in the (sorted) history list, so every logit is read and
// written by one thread, once.  The history list is checked first (strictly
// ascending ids, counts >= 1): a lane that breaks it is left untouched and
// reported, since two entries of one id would have two threads update one
// logit and an unsorted list would defeat the search for drafts.
template <bool BF16>
__global__ void __launch_bounds__(256) apply_penalties_kernel(uint8_t* target, int64_t ld_bytes, int32_t V,
                                                              const int32_t* row_offsets,
                                                              const int32_t* draft_tokens,
                                                              const int32_t* draft_lens, const int32_t* pen_tokens,
                                                              const int32_t* pen_counts,
                                                              const int64_t* pen_offsets, const float* presence,
                                                              const float* frequency, int32_t* lane_status) {
  const int b = blockIdx.x;
  const int k = draft_lens[b];
  const int off = row_offsets[b];
  const int64_t h0 = pen_offsets[b], h1 = pen_offsets[b + 1];
  int status = SPEC_OK;
  if (k < 0 || off < 0 || row_offsets[b + 1] - off != k + 1) status = SPEC_ERR_LAYOUT;
  else if (k > SPEC_MAX_DRAFTS) status = SPEC_ERR_UNSUPPORTED;
  bool bad = h1 < h0;
  for (int64_t e = h0 + threadIdx.x; !bad && e < h1; e += blockDim.x)
    bad = pen_counts[e] < 1 || (e > h0 && pen_tokens[e] <= pen_tokens[e - 1]);
  if (__syncthreads_or(bad) && status == SPEC_OK) status = SPEC_ERR_INVALID_ARG;
  if (threadIdx.x == 0 && lane_status != nullptr) lane_status[b] = status;
  if (status != SPEC_OK) return;
  const float pres = presence ? presence[b] : 0.f;
  const float freq = frequency ? frequency[b] : 0.f;
  int d[SPEC_MAX_DRAFTS];
#pragma unroll
  for (int i = 0; i < SPEC_MAX_DRAFTS; ++i) d[i] = (i < k) ? draft_tokens[off + i] : -1;

  auto penalise = [&](int row, int t, int c) {
    uint8_t* r = target + static_cast<int64_t>(off + row) * ld_bytes;
    const float m = __fmul_rn(freq, static_cast<float>(c));
    const float delta = __fadd_rn(m, pres);
    if constexpr (BF16) {
      __nv_bfloat16* p = reinterpret_cast<__nv_bfloat16*>(r) + t;
      *p = __float2bfloat16_rn(__fsub_rn(__bfloat162float(*p), delta));
    } else {
      float* p = reinterpret_cast<float*>(r) + t;
      *p = __fsub_rn(*p, delta);
    }
  };
  auto in_history = [&](int t) {  // binary search of the sorted list
    int64_t lo = h0, hi = h1;
    while (lo < hi) {
      const int64_t mid = (lo + hi) >> 1;
      const int v = pen_tokens[mid];
      if (v == t) return true;
      if (v < t) lo = mid + 1;
      else hi = mid;
    }
    return false;
  };

  const int64_t nh = h1 > h0 ? h1 - h0 : 0;
  // (row, history entry) pairs, all rows at once
  for (int64_t idx = threadIdx.x; idx < (k + 1) * nh; idx += blockDim.x) {
    const int j = static_cast<int>(idx / nh);
    const int64_t e = idx - j * nh;
    const int t = pen_tokens[h0 + e];
    if (t < 0 || t >= V) continue;
    int c = pen_counts[h0 + e];
#pragma unroll
    for (int i = 0; i < SPEC_MAX_DRAFTS; ++i) c += (i < j && d[i] == t) ? 1 : 0;
    if (c > 0) penalise(j, t, c);
  }
  // (row j, draft i < j) pairs for drafts the history does not list, first
  // occurrence of each token in d_1..d_j only
  static_assert((SPEC_MAX_DRAFTS + 1) * (SPEC_MAX_DRAFTS + 1) <= 256, "one thread per (row, draft) pair");
  {
    const int j = threadIdx.x / (SPEC_MAX_DRAFTS + 1), i = threadIdx.x % (SPEC_MAX_DRAFTS + 1);
    if (j <= k && i < j) {
      const int t = d[i];
      bool first = (t >= 0 && t < V);
      int c = 0;
      for (int q = 0; q < j; ++q) {
        if (d[q] == t) {
          ++c;
          if (q < i) first = false;
        }
      }
      if (first && !in_history(t)) penalise(j, t, c);
    }
  }
}

int launch_status() { return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA; }

// (1 - alpha^(g + 1)) / (1 - alpha): expected tokens a round of independent
// guesses that each survive with probability alpha, at depth g.
double tokens_of_alpha(double alpha, int depth) {
  if (alpha >= 1.0) return depth + 1.0;
  return (1.0 - std::pow(alpha, depth + 1)) / (1.0 - alpha);
}

}  // namespace

extern "C" {

int spec_accept_counts_update(const int32_t* committed, const int32_t* draft_lens, const int32_t* lane_status,
                              int32_t lanes, spec_accept_counts* counts, int32_t per_lane, void* stream) {
  if (lanes < 0 || (per_lane != 0 && per_lane != 1)) return SPEC_ERR_INVALID_ARG;
  if (lanes == 0) return SPEC_OK;
  if (committed == nullptr || draft_lens == nullptr || counts == nullptr) return SPEC_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned long long* out = reinterpret_cast<unsigned long long*>(counts);
  const int blocks = (lanes + 255) / 256;
  if (per_lane) {
    accept_counts_lane_kernel<<<blocks, 256, 0, st>>>(committed, draft_lens, lane_status, lanes, out);
  } else {
    accept_counts_batch_kernel<<<blocks < 148 ? blocks : 148, 256, 0, st>>>(committed, draft_lens, lane_status,
                                                                             lanes, out);
  }
  return launch_status();
}

int spec_accept_rates_from_counts(const spec_accept_counts* c, spec_accept_rates* r) {
  if (c == nullptr || r == nullptr) return SPEC_ERR_INVALID_ARG;
  const double rounds = static_cast<double>(c->rounds);
  r->accepted_per_proposed = c->proposed ? static_cast<double>(c->accepted) / c->proposed : NAN;
  r->tokens_per_round = c->rounds ? 1.0 + static_cast<double>(c->accepted) / rounds : NAN;
  double prev = rounds;
  for (int j = 0; j < kSlots; ++j) {
    r->by_slot[j] = c->rounds ? static_cast<double>(c->slot_kept[j]) / rounds : NAN;
    r->given_previous[j] = prev > 0 ? static_cast<double>(c->slot_kept[j]) / prev : NAN;
    prev = static_cast<double>(c->slot_kept[j]);
  }
  r->depth = c->rounds ? static_cast<int32_t>(static_cast<double>(c->proposed) / rounds + 0.5) : 0;
  r->reserved = 0;
  // Bisection on [0, 1]: the expected tokens a round grow with alpha.
  if (!c->rounds || r->depth <= 0) {
    r->implied_alpha = NAN;
  } else if (r->tokens_per_round <= 1.0) {
    r->implied_alpha = 0.0;
  } else if (r->tokens_per_round >= r->depth + 1.0) {
    r->implied_alpha = 1.0;
  } else {
    double lo = 0.0, hi = 1.0;
    for (int it = 0; it < 200; ++it) {
      const double mid = 0.5 * (lo + hi);
      if (tokens_of_alpha(mid, r->depth) < r->tokens_per_round) lo = mid;
      else hi = mid;
    }
    r->implied_alpha = 0.5 * (lo + hi);
  }
  return SPEC_OK;
}

int spec_backoff_init(spec_backoff_state* states, int32_t lanes, void* stream) {
  if (lanes < 0) return SPEC_ERR_INVALID_ARG;
  if (lanes == 0) return SPEC_OK;
  if (states == nullptr) return SPEC_ERR_INVALID_ARG;
  backoff_init_kernel<<<(lanes + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(states, lanes);
  return launch_status();
}

int spec_backoff_step(spec_backoff_state* states, const int32_t* proposed, const int32_t* committed,
                      const int32_t* lane_status, int32_t lanes, int32_t draft_tokens, int32_t* next_draft_lens,
                      void* stream) {
  if (lanes < 0 || draft_tokens < 0 || draft_tokens > SPEC_MAX_DRAFTS) return SPEC_ERR_INVALID_ARG;
  if (lanes == 0) return SPEC_OK;
  if (states == nullptr || proposed == nullptr || committed == nullptr || next_draft_lens == nullptr)
    return SPEC_ERR_INVALID_ARG;
  backoff_step_kernel<<<1, 1024, 0, static_cast<cudaStream_t>(stream)>>>(states, proposed, committed, lane_status,
                                                                        lanes, draft_tokens, next_draft_lens);
  return launch_status();
}

int spec_ngram_draft(const int32_t* tokens, const int64_t* hist_offsets, int32_t lanes, int32_t k,
                     int32_t match_min, int32_t match_max, int32_t* drafts, int32_t draft_stride,
                     int32_t* draft_lens, void* stream) {
  if (lanes < 0 || k < 0 || k > SPEC_MAX_DRAFTS || draft_stride < k || match_min < 1 || match_max < match_min ||
      match_max > SPEC_NGRAM_MAX_MATCH)
    return SPEC_ERR_INVALID_ARG;
  if (lanes == 0) return SPEC_OK;
  if (tokens == nullptr || hist_offsets == nullptr || drafts == nullptr || draft_lens == nullptr)
    return SPEC_ERR_INVALID_ARG;
  ngram_draft_kernel<<<lanes, kNgramThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      tokens, hist_offsets, k, match_min, match_max, drafts, draft_stride, draft_lens);
  return launch_status();
}

int spec_apply_penalties(void* target_logits, spec_dtype dtype, int64_t ld, int32_t V, int32_t lanes,
                         const int32_t* row_offsets, const int32_t* draft_tokens, const int32_t* draft_lens,
                         const int32_t* pen_tokens, const int32_t* pen_counts, const int64_t* pen_offsets,
                         const float* presence, const float* frequency, int32_t* lane_status, void* stream) {
  if (lanes < 0 || V <= 0 || ld < V || (dtype != SPEC_F32 && dtype != SPEC_BF16)) return SPEC_ERR_INVALID_ARG;
  if (lanes == 0) return SPEC_OK;
  if (target_logits == nullptr || row_offsets == nullptr || draft_tokens == nullptr || draft_lens == nullptr ||
      pen_tokens == nullptr || pen_counts == nullptr || pen_offsets == nullptr)
    return SPEC_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* t = static_cast<uint8_t*>(target_logits);
  if (dtype == SPEC_BF16) {
    apply_penalties_kernel<true><<<lanes, 256, 0, st>>>(t, ld * 2, V, row_offsets, draft_tokens, draft_lens,
                                                        pen_tokens, pen_counts, pen_offsets, presence, frequency,
                                                        lane_status);
  } else {
    apply_penalties_kernel<false><<<lanes, 256, 0, st>>>(t, ld * 4, V, row_offsets, draft_tokens, draft_lens,
                                                         pen_tokens, pen_counts, pen_offsets, presence, frequency,
                                                         lane_status);
  }
  return launch_status();
}

}  // extern "C"
