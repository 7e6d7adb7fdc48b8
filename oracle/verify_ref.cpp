// verify_ref.cpp -- plain C++ CPU oracle of the speculative-decoding verify round.
//
// TEST INFRASTRUCTURE ONLY.  A slow, obviously correct float64 statement of
// what the verify round computes, used to check the CUDA library and timed as
// its CPU baseline.  Only tests/, __graft_entry__.smoke() and bench.py's CPU
// legs may load it.  It shares no code, header, constant table or helper with
// the CUDA library and never calls it; it includes only the C++ standard
// library.  Every step is written from the pages' description of the round:
//
//   ignis docs, "Speculative decoding" -- "One round, step by step": a lane
//     holds an anchor and up to k drafts, the model scores the k + 1 columns,
//     the longest run of drafts the model agrees with is kept plus the model's
//     own token (1 .. k + 1 tokens), and the state advances by exactly that run.
//   ignis docs, "Speculative decoding" -- "The row budget": drafts per lane are
//     min(draft tokens, rows / lanes - 1); a budget of 0 means 8.
//   strata2signal, "Draft heads and speculative decoding, in plain words" --
//     "Guess, then check": row j scores the position after guess j; at
//     temperature zero the model takes its single most likely token; with the
//     acceptance rule of Leviathan et al. (2022) / Chen et al. (2023) the
//     output keeps the target's distribution: accept d with probability
//     min(1, p(d) / q(d)), at the first rejection draw from max(0, p - q)
//     normalised, and after k acceptances draw a bonus token from p.
//   FreeToken issue #828 -- "Design" (per-request state): the verify pass stages
//     one snapshot per column and the commit keeps the accepted prefix only.
//
// Readings where the pages are silent (the same ones the library documents):
// argmax ties go to the lowest id and -0 equals +0; -inf logits are allowed,
// NaN or +inf in a row that is read (or a row that is -inf everywhere) fails
// the lane; row j is checked against draft d_{j+1}; drafter rows use the target
// rows' numbering and a lane's last drafter row is not read; T <= 0 is a greedy
// lane and q uses the same T as p; p(d) = 0 rejects, q(d) = 0 < p(d) accepts;
// the inverse-CDF draw walks ids upwards and takes the first cumulative weight
// strictly above u' * W, else the largest id of positive weight, and a residual
// of mass 0 falls back to p; staged column c is the state after consuming
// column c (column 0 = the anchor), so the commit copies column committed - 1.
//
// Uniforms: Philox4x64-10 (Salmon, Moraes, Dror and Shaw, "Parallel Random
// Numbers: As Easy as 1, 2, 3", SC'11) with key (seed, 0) and counter
// (position, lane, 0, 0); word 0 gives the acceptance uniform u_j, word 1 the
// draw's u'; u = (word >> 40) * 2^-24.
//
// Arithmetic is plain IEEE float64 (built with -ffp-contract=off, so no fused
// multiply-adds); sums run sequentially in index order.  Lanes are independent
// and are handed out to std::thread workers one at a time.
//
// Test-only: OREF_MUTATE=<n> at compile time plants one plausible mistake, so
// that tests can show a pin catches it (see the cases marked OREF_MUTATE).
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

#ifndef OREF_MUTATE
#define OREF_MUTATE 0
#endif

namespace {

// Per-lane status codes: the numbers of the library's public contract,
// restated here (not included).
enum : int32_t {
  kOk = 0,
  kInvalidArg = 1,
  kNonFinite = 4,
  kTokenRange = 5,
  kLayout = 6,
};

enum : int32_t { kF32 = 0, kBF16 = 1, kF64 = 2 };

constexpr double kInf = std::numeric_limits<double>::infinity();
constexpr double kNaN = std::numeric_limits<double>::quiet_NaN();

// ---------------------------------------------------------------------------
// Philox4x64-10 (SC'11): per round two 64x64 -> 128-bit products; the high
// halves are xored with the other counter words and the round key; the key
// advances by the Weyl increments (golden ratio, sqrt(3) - 1) between rounds.
// ---------------------------------------------------------------------------
constexpr uint64_t kPhiloxM0 = 0xD2E7470EE14C6C93ull;
constexpr uint64_t kPhiloxM1 = 0xCA5A826395121157ull;
constexpr uint64_t kWeyl0 = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kWeyl1 = 0xBB67AE8584CAA73Bull;
#if OREF_MUTATE == 8
constexpr int kPhiloxRounds = 9;
#else
constexpr int kPhiloxRounds = 10;
#endif

void philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]) {
  uint64_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint64_t k0 = key[0], k1 = key[1];
  for (int r = 0; r < kPhiloxRounds; ++r) {
    const unsigned __int128 p0 = static_cast<unsigned __int128>(kPhiloxM0) * c0;
    const unsigned __int128 p1 = static_cast<unsigned __int128>(kPhiloxM1) * c2;
    const uint64_t hi0 = static_cast<uint64_t>(p0 >> 64), lo0 = static_cast<uint64_t>(p0);
    const uint64_t hi1 = static_cast<uint64_t>(p1 >> 64), lo1 = static_cast<uint64_t>(p1);
    const uint64_t n0 = hi1 ^ c1 ^ k0, n1 = lo1, n2 = hi0 ^ c3 ^ k1, n3 = lo0;
    c0 = n0;
    c1 = n1;
    c2 = n2;
    c3 = n3;
    k0 += kWeyl0;
    k1 += kWeyl1;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

// Top 24 bits of a word, scaled into [0, 1): exact in float32 and float64.
double word_uniform(uint64_t w) { return static_cast<double>(w >> 40) * (1.0 / 16777216.0); }

void round_uniforms(uint64_t seed, uint64_t lane, uint64_t position, double* u_acc, double* u_smp) {
  const uint64_t ctr[4] = {position, lane, 0, 0};
  const uint64_t key[2] = {seed, 0};
  uint64_t w[4];
  philox4x64_10(ctr, key, w);
  *u_acc = word_uniform(w[0]);
  *u_smp = word_uniform(w[1]);
}

// ---------------------------------------------------------------------------
// Logit access: exact widening of the stored element to float64.
// ---------------------------------------------------------------------------
struct Rows {
  const uint8_t* base;
  int32_t dtype;
  int64_t ld;  // elements
  int64_t V;

  double at(int64_t row, int64_t x) const {
    const int64_t i = row * ld + x;
    if (dtype == kBF16) {
      uint16_t h;
      std::memcpy(&h, base + 2 * i, 2);
      const uint32_t bits = static_cast<uint32_t>(h) << 16;  // bf16 = the top half of a float32
      float f;
      std::memcpy(&f, &bits, 4);
      return static_cast<double>(f);
    }
    if (dtype == kF32) {
      float f;
      std::memcpy(&f, base + 4 * i, 4);
      return static_cast<double>(f);
    }
    double d;
    std::memcpy(&d, base + 8 * i, 8);
    return d;
  }
};

// A row can be reduced: no NaN, no +inf, and not -inf everywhere.
bool row_is_valid(const Rows& r, int64_t row) {
  bool finite = false;
  for (int64_t x = 0; x < r.V; ++x) {
    const double v = r.at(row, x);
    if (std::isnan(v) || v == kInf) return false;
    if (std::isfinite(v)) finite = true;
  }
  return finite;
}

// Lowest index of the largest logit, and that logit.
int64_t argmax_lowest(const Rows& r, int64_t row, double* max_out) {
  int64_t best = 0;
  double m = r.at(row, 0);
  for (int64_t x = 1; x < r.V; ++x) {
    const double v = r.at(row, x);
#if OREF_MUTATE == 3
    if (v >= m) {  // planted: ties go to the highest index
#else
    if (v > m) {
#endif
      m = v;
      best = x;
    }
  }
  *max_out = m;
  return best;
}

// softmax(row / T) in float64: zmax = max z, S = sum exp(z - zmax) in index
// order, p(x) = exp(z_x - zmax) / S, lse = zmax + log S.
struct Softmax {
  double zmax, sum, lse, temp;
  double prob(const Rows& r, int64_t row, int64_t x) const {
    return std::exp(r.at(row, x) / temp - zmax) / sum;
  }
};

Softmax softmax_at(const Rows& r, int64_t row, double temp) {
#if OREF_MUTATE == 4
  temp = 1.0;  // planted: the temperature is dropped
#endif
  Softmax s;
  s.temp = temp;
  s.zmax = -kInf;
  for (int64_t x = 0; x < r.V; ++x) s.zmax = std::fmax(s.zmax, r.at(row, x) / temp);
  s.sum = 0.0;
  for (int64_t x = 0; x < r.V; ++x) s.sum += std::exp(r.at(row, x) / temp - s.zmax);
  s.lse = s.zmax + std::log(s.sum);
  return s;
}

// p(d) / q(d) with the edge cases fixed: p(d) = 0 -> 0, q(d) = 0 -> inf.
double acceptance_ratio(double p_d, double q_d) {
  if (p_d == 0.0) return 0.0;
  if (q_d == 0.0) return kInf;
  return p_d / q_d;
}

struct Inputs {
  Rows target, draft;
  bool has_draft;
  int64_t rows;
  const int32_t* draft_tokens;
  const int32_t* draft_lens;
  const int32_t* row_offsets;
  const float* temperatures;
  int32_t lanes;
  uint64_t seed;
  uint64_t lane_base;
  const double* u_acc;  // optional [lanes][u_stride] overrides of the uniforms
  const double* u_smp;
  int32_t u_stride;
};

struct Outputs {
  int32_t* committed;
  int32_t* out_tokens;
  int32_t* lane_status;
  int64_t* argmax;
  double* max_logit;
  double* lse;
  double* logp_d;
  double* logq_d;
  double* resid_mass;
  double* accept_margin;  // [rows]: |u_j - p/q| of each decision made, at off + j
  double* draw_margin;    // [lanes]: distance of u' * W to the nearest CDF boundary, / W
  int32_t* draw_pos;      // [lanes]: position n of the draw (-1 if none)
};

// Inverse-CDF draw from weights w[0..V): the first x whose cumulative weight
// (summed in index order) is strictly above u * W; if rounding leaves none, the
// largest x of positive weight.  Also the distance of u * W to the nearest
// cumulative boundary (0 included), divided by W.
int64_t inverse_cdf(const std::vector<double>& w, double u, double* margin) {
  double W = 0.0;
  for (double v : w) W += v;
  const double target = u * W;
  double cum = 0.0, best = std::fabs(target);
  int64_t token = -1, last_pos = -1;
  for (size_t x = 0; x < w.size(); ++x) {
    cum += w[x];
    best = std::fmin(best, std::fabs(cum - target));
    if (w[x] > 0.0) last_pos = static_cast<int64_t>(x);
#if OREF_MUTATE == 5
    if (token < 0 && cum >= target) token = static_cast<int64_t>(x);  // planted: non-strict
#else
    if (token < 0 && cum > target) token = static_cast<int64_t>(x);
#endif
  }
  *margin = best / W;
  return token >= 0 ? token : last_pos;
}

void verify_lane(const Inputs& in, const Outputs& out, int32_t b, std::vector<double>& wbuf) {
  const int32_t k = in.draft_lens[b];
  const int64_t off = in.row_offsets[b], end = in.row_offsets[b + 1];
  out.committed[b] = 0;
  out.draw_margin[b] = kNaN;
  out.draw_pos[b] = -1;
  // Layout: the lane's k + 1 rows lie inside [0, rows).
  if (k < 0 || off < 0 || end > in.rows || end - off != static_cast<int64_t>(k) + 1) {
    out.lane_status[b] = kLayout;
    return;
  }
  const int64_t V = in.target.V;
  for (int32_t j = 0; j < k; ++j) {
    const int32_t d = in.draft_tokens[off + j];
    if (d < 0 || d >= V) {
      out.lane_status[b] = kTokenRange;
      return;
    }
  }
  const bool sampled = static_cast<double>(in.temperatures[b]) > 0.0;
  if (sampled && !in.has_draft) {
    out.lane_status[b] = kInvalidArg;
    return;
  }
  for (int32_t j = 0; j <= k; ++j)
    if (!row_is_valid(in.target, off + j)) {
      out.lane_status[b] = kNonFinite;
      return;
    }
  if (sampled)
    for (int32_t j = 0; j < k; ++j)
      if (!row_is_valid(in.draft, off + j)) {
        out.lane_status[b] = kNonFinite;
        return;
      }
  out.lane_status[b] = kOk;

  std::vector<int64_t> a(k + 1);
  for (int32_t j = 0; j <= k; ++j) {
    double m;
    a[j] = argmax_lowest(in.target, off + j, &m);
    out.argmax[off + j] = a[j];
    out.max_logit[off + j] = m;
  }

  if (!sampled) {
    // Greedy: keep d_{j+1} while it equals the argmax of row j; the model's
    // token after the run is the argmax of the first row that disagrees.
    int32_t n = 0;
#if OREF_MUTATE == 2
    while (n < k && n + 1 <= k && in.draft_tokens[off + n] == a[n + 1]) ++n;  // planted: row j + 1
#else
    while (n < k && in.draft_tokens[off + n] == a[n]) ++n;
#endif
    for (int32_t i = 0; i <= n; ++i) out.out_tokens[off + i] = static_cast<int32_t>(a[i]);
    out.committed[b] = n + 1;
    return;
  }

  // Sampled: the textbook rule.
  const double T = static_cast<double>(in.temperatures[b]);
  std::vector<Softmax> p(k + 1), q(k);
  for (int32_t j = 0; j <= k; ++j) {
    p[j] = softmax_at(in.target, off + j, T);
    out.lse[off + j] = p[j].lse;
  }
  for (int32_t j = 0; j < k; ++j) q[j] = softmax_at(in.draft, off + j, T);

  auto uniforms = [&](int32_t j, double* ua, double* us) {
    round_uniforms(in.seed, in.lane_base + static_cast<uint64_t>(b), static_cast<uint64_t>(j), ua, us);
    if (in.u_acc) *ua = in.u_acc[static_cast<int64_t>(b) * in.u_stride + j];
    if (in.u_smp) *us = in.u_smp[static_cast<int64_t>(b) * in.u_stride + j];
  };

  int32_t n = k;
  for (int32_t j = 0; j < k; ++j) {
    const int64_t d = in.draft_tokens[off + j];
    const double p_d = p[j].prob(in.target, off + j, d);
    const double q_d = q[j].prob(in.draft, off + j, d);
    out.logp_d[off + j] = p_d > 0.0 ? std::log(p_d) : -kInf;
    out.logq_d[off + j] = q_d > 0.0 ? std::log(q_d) : -kInf;
    if (n == k) {
      double ua, us;
      uniforms(j, &ua, &us);
#if OREF_MUTATE == 1
      const double ratio = acceptance_ratio(q_d, p_d);  // planted: the ratio transposed
#else
      const double ratio = acceptance_ratio(p_d, q_d);
#endif
      out.accept_margin[off + j] = std::fabs(ua - ratio);
      if (!(ua < std::fmin(1.0, ratio))) n = j;
    }
  }

  // The model's token: residual max(0, p_n - q_n) at the first rejection n,
  // else a bonus draw from p_k.
  wbuf.assign(static_cast<size_t>(V), 0.0);
  if (n < k) {
    double mass = 0.0;
    bool any = false;
    for (int64_t x = 0; x < V; ++x) {
      const double px = p[n].prob(in.target, off + n, x);
      const double qx = q[n].prob(in.draft, off + n, x);
#if OREF_MUTATE == 6
      const double w = std::fmax(0.0, qx - px);  // planted: residual transposed
#else
      const double w = std::fmax(0.0, px - qx);
#endif
      wbuf[x] = w;
      mass += w;
      any = any || w > 0.0;
    }
    out.resid_mass[off + n] = mass;
    if (!any)
      for (int64_t x = 0; x < V; ++x) wbuf[x] = p[n].prob(in.target, off + n, x);
  } else {
    for (int64_t x = 0; x < V; ++x) wbuf[x] = p[k].prob(in.target, off + k, x);
  }
  double ua, us;
  uniforms(n, &ua, &us);
  double margin;
  const int64_t token = inverse_cdf(wbuf, us, &margin);
  for (int32_t i = 0; i < n; ++i) out.out_tokens[off + i] = in.draft_tokens[off + i];
  out.out_tokens[off + n] = static_cast<int32_t>(token);
  out.committed[b] = n + 1;
  out.draw_margin[b] = margin;
  out.draw_pos[b] = n;
}

}  // namespace

extern "C" {

// Drafts per lane under a row budget (ignis, "The row budget"):
// max(0, min(draft_tokens, rows / lanes - 1)) with floor division; rows == 0
// means 8.  Returns -1 for lanes <= 0 or a negative argument.
int32_t oref_row_budget(int32_t draft_tokens, int32_t rows, int32_t lanes) {
  if (lanes <= 0 || draft_tokens < 0 || rows < 0) return -1;
  if (rows == 0) rows = 8;
#if OREF_MUTATE == 7
  const int32_t per_lane = (rows + lanes - 1) / lanes - 1;  // planted: ceiling division
#else
  const int32_t per_lane = rows / lanes - 1;
#endif
  const int32_t d = per_lane < draft_tokens ? per_lane : draft_tokens;
  return d < 0 ? 0 : d;
}

void oref_philox4x64_10(const uint64_t* ctr, const uint64_t* key, uint64_t* out) { philox4x64_10(ctr, key, out); }

void oref_round_uniforms(uint64_t seed, uint64_t lane, uint64_t position, double* out2) {
  round_uniforms(seed, lane, position, out2, out2 + 1);
}

// One verify round over every lane.  Logits are [rows][ld] of dtype 0 (float32),
// 1 (bfloat16 bit patterns) or 2 (float64); draft may be NULL when no lane
// samples.  Per-row outputs are written only for rows of lanes that reach them
// and must be pre-filled by the caller (argmax -1, floats NaN, tokens -1).
// u_acc / u_smp (optional, [lanes][u_stride]) replace the Philox uniforms.
// `threads` workers (<= 0: one per hardware thread) take lanes one at a time.
// Returns the number of worker threads used.
int32_t oref_verify_round(const void* target, const void* draft, int32_t dtype, int64_t ld, int64_t rows, int64_t V,
                          const int32_t* draft_tokens, const int32_t* draft_lens, const int32_t* row_offsets,
                          const float* temperatures, int32_t lanes, uint64_t seed, uint64_t lane_base,
                          const double* u_acc, const double* u_smp, int32_t u_stride, int32_t threads,
                          int32_t* committed, int32_t* out_tokens, int32_t* lane_status, int64_t* argmax,
                          double* max_logit, double* lse, double* logp_d, double* logq_d, double* resid_mass,
                          double* accept_margin, double* draw_margin, int32_t* draw_pos) {
  Inputs in;
  in.target = Rows{static_cast<const uint8_t*>(target), dtype, ld, V};
  in.draft = Rows{static_cast<const uint8_t*>(draft), dtype, ld, V};
  in.has_draft = draft != nullptr;
  in.rows = rows;
  in.draft_tokens = draft_tokens;
  in.draft_lens = draft_lens;
  in.row_offsets = row_offsets;
  in.temperatures = temperatures;
  in.lanes = lanes;
  in.seed = seed;
  in.lane_base = lane_base;
  in.u_acc = u_acc;
  in.u_smp = u_smp;
  in.u_stride = u_stride;
  const Outputs out{committed, out_tokens, lane_status, argmax, max_logit, lse, logp_d, logq_d,
                    resid_mass, accept_margin, draw_margin, draw_pos};
  int32_t n = threads;
  if (n <= 0) n = static_cast<int32_t>(std::thread::hardware_concurrency());
  if (n <= 0) n = 1;
  if (n > lanes) n = lanes > 0 ? lanes : 1;
  std::atomic<int32_t> next{0};
  auto worker = [&]() {
    std::vector<double> wbuf;
    for (;;) {
      const int32_t b = next.fetch_add(1);
      if (b >= lanes) return;
      verify_lane(in, out, b, wbuf);
    }
  };
  if (n == 1) {
    worker();
  } else {
    std::vector<std::thread> pool;
    pool.reserve(static_cast<size_t>(n));
    for (int32_t t = 0; t < n; ++t) pool.emplace_back(worker);
    for (auto& t : pool) t.join();
  }
  return n;
}

// The state commit (ignis step 5; FreeToken #828 "Design"): live[b] <-
// staged[b][committed[b] - 1] for every lane whose status is OK (lane_status may
// be NULL) and whose count lies in 1..cols; other lanes keep their live state.
void oref_commit_state(const uint8_t* staged, uint8_t* live, const int32_t* committed, const int32_t* lane_status,
                       int32_t lanes, int32_t cols, uint64_t bytes_per_col) {
  for (int32_t b = 0; b < lanes; ++b) {
    if (lane_status != nullptr && lane_status[b] != kOk) continue;
    const int32_t c = committed[b];
    if (c < 1 || c > cols) continue;
#if OREF_MUTATE == 9
    const int32_t col = c < cols ? c : cols - 1;  // planted: column c instead of c - 1
#else
    const int32_t col = c - 1;
#endif
    std::memcpy(live + static_cast<uint64_t>(b) * bytes_per_col,
                staged + (static_cast<uint64_t>(b) * cols + col) * bytes_per_col, bytes_per_col);
  }
}

}  // extern "C"
