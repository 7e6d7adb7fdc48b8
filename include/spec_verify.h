/*
 * spec_verify.h -- C ABI of the speculative-decoding verify round on GB300 (sm_103a).
 *
 * One verify round (ignis docs, "Speculative decoding" -- "One round, step by
 * step"): each of B lanes holds an anchor and k_b >= 0 drafts d_1..d_{k_b}; the
 * target model has scored the k_b + 1 columns, giving k_b + 1 logit rows per lane.
 * This library does the data-parallel rest of the round on the GPU:
 *
 *   spec_row_budget     how many drafts a lane may carry (ignis, "The row budget")
 *   spec_verify_accept  reduce every row over the vocabulary, find each lane's
 *                       committed run, draw the model's own token (one fused kernel)
 *   spec_commit_state   roll each lane's recurrent state to its committed count
 *
 * Conventions shared by every entry point
 *   - All array pointers are DEVICE pointers unless stated otherwise.  The caller
 *     owns every buffer; the library allocates no memory and keeps no state
 *     between calls except a per-device cache of kernel attributes.  Entry points
 *     are thread-safe.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Calls only enqueue work and return at once; they never
 *     synchronise the device.
 *   - The return value reports errors the host can see (bad arguments, launch
 *     failures).  Errors found on the device (bad offsets, out-of-range tokens,
 *     NaN / +inf logits) are reported per lane in `lane_status`; such a lane
 *     commits nothing.  No kernel traps: waits inside the kernels are bounded and
 *     report SPEC_ERR_TIMEOUT instead.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes: return values of the entry points and per-lane lane_status. */
typedef enum {
  SPEC_OK = 0,
  SPEC_ERR_INVALID_ARG = 1, /* a NULL pointer, size or dtype the call cannot take;
                               per lane: a sampled lane but draft_logits == NULL    */
  SPEC_ERR_UNSUPPORTED = 2, /* per lane: k_b > SPEC_MAX_DRAFTS                     */
  SPEC_ERR_CUDA = 3,        /* a CUDA call failed (launch error, no device, ...)   */
  SPEC_ERR_NONFINITE = 4,   /* per lane: NaN or +inf in a row that is read, or a
                               row that is -inf everywhere                          */
  SPEC_ERR_TOKEN_RANGE = 5, /* per lane: a draft token outside [0, V)              */
  SPEC_ERR_LAYOUT = 6,      /* per lane: row_offsets disagree with draft_lens or
                               leave [0, rows); commit: committed[b] outside 1..cols */
  SPEC_ERR_TIMEOUT = 7      /* per lane: a bounded wait inside a kernel gave up     */
} spec_status;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

/* Most drafts one lane may carry in spec_verify_accept (k_b <= 15).  The pages'
 * drafters propose 1..8 tokens per pass. */
#define SPEC_MAX_DRAFTS 15

/*
 * Flags of spec_verify_args.flags.
 *
 * SPEC_VERIFY_META_BEFORE_WAIT: draft_tokens, draft_lens, row_offsets and
 * temperatures were written before the kernel that precedes this launch on
 * the stream began (by an earlier kernel, a copy or the host).  The kernel then
 * reads them while it waits for that kernel to finish (programmatic dependent
 * launch), which takes one global-memory round trip off each launch.  Without
 * the flag it reads them after the wait, as it must when the preceding kernel
 * produces them.  The logits are always read after the wait.
 */
#define SPEC_VERIFY_META_BEFORE_WAIT 1u

/*
 * SPEC_VERIFY_TEST_WITHHOLD_COPY: for tests of the failure path only.  Each
 * CTA's producer skips its last bulk copy, so the waits for it run out after
 * the kernel's time limit (2 s) and every lane with rows to stream reports
 * SPEC_ERR_TIMEOUT (committed 0).  The launch then returns normally and the
 * context stays usable.  Never set in normal use.
 */
#define SPEC_VERIFY_TEST_WITHHOLD_COPY 2u

/*
 * spec_row_budget -- drafts per lane under a row budget.
 *
 * ignis docs, "Speculative decoding" -- "The row budget": a round carries
 * lanes x (drafts + 1) rows; with a cap of `row_budget` rows each lane drafts
 * min(draft_tokens, row_budget / lanes - 1), and a budget of 0 means 8.
 * Division is floor division and the result is clamped at 0 (8 rows, 3 draft
 * tokens: 3 drafts at 1-2 lanes, 1 at 3-4, none from 5 lanes on).
 *
 * Host-only; touches no GPU.  Returns the drafts per lane (>= 0), or
 * -SPEC_ERR_INVALID_ARG if lanes <= 0, draft_tokens < 0 or row_budget < 0.
 */
int32_t spec_row_budget(int32_t draft_tokens, int32_t row_budget, int32_t lanes);

/* Optional per-row diagnostics written by spec_verify_accept (32 bytes). */
typedef struct {
  int32_t argmax;     /* lowest index of the row's largest logit                   */
  float max_logit;    /* that logit                                                */
  float lse;          /* log sum_x exp(x / T) (sampled lanes; NaN on greedy lanes)  */
  float logp_d;       /* log p_j(d_{j+1}), p_j = softmax(row j / T)  (sampled, j<k_b) */
  float logq_d;       /* log q_j(d_{j+1}), q_j = softmax(draft row j / T)          */
  float resid_mass;   /* sum_x max(0, p_n - q_n) at the first rejected row n        */
  int32_t drawn;      /* token drawn at this row (residual or bonus draw), else -1  */
  int32_t flags;      /* bit 0: row was read; bit 1: residual draw; bit 2: bonus draw */
} spec_row_stats;

typedef struct {
  /* Target logits, row-major [rows][ld] of `dtype`.  Lane b owns rows
   * off[b] .. off[b] + k_b; row off[b] + j scores the position after the anchor
   * and d_1..d_j (strata2signal, "Draft heads and speculative decoding, in plain
   * words" -- "Guess, then check").  Rows whose address is 16-byte aligned
   * (base and ld * element size) are streamed with bulk copies; other layouts
   * take a slower element-wise path with the same results. */
  const void* target_logits;
  /* Drafter logits with the same row numbering and ld: row off[b] + j is q_j,
   * the distribution d_{j+1} was drawn from; rows off[b] .. off[b] + k_b - 1 are
   * read, the lane's last row is not.  May be NULL when no lane samples. */
  const void* draft_logits;
  spec_dtype dtype;           /* element type of both logits arrays              */
  int64_t ld;                 /* row stride in elements, >= V                     */
  int32_t V;                  /* vocabulary size, > 0                              */
  int32_t lanes;              /* B > 0                                            */
  int32_t rows;               /* off[lanes]; rows of every per-row array          */
  const int32_t* draft_tokens;  /* [rows]: draft_tokens[off[b] + j] = d_{j+1}, j < k_b;
                                   the slot off[b] + k_b is not read             */
  const int32_t* draft_lens;    /* [lanes]: k_b, 0 <= k_b <= SPEC_MAX_DRAFTS      */
  const int32_t* row_offsets;   /* [lanes + 1]: off[b + 1] - off[b] == k_b + 1    */
  const float* temperatures;    /* [lanes]: T_b <= 0 greedy lane, > 0 sampled lane */
  uint64_t seed;                /* Philox4x64-10 key of the round's uniforms; the
                                   caller varies it from round to round           */
  int32_t* committed;           /* out [lanes]: c_b in 1..k_b + 1 (0 if the lane failed) */
  int32_t* out_tokens;          /* out [rows]: slot off[b] + i holds committed token i
                                   for i < c_b, -1 for c_b <= i <= k_b            */
  int32_t* lane_status;         /* out [lanes]: spec_status per lane (may be NULL) */
  spec_row_stats* row_stats;    /* out [rows] (may be NULL)                        */
  uint32_t lane_base;           /* global index of lane 0 in the Philox counter: a batch
                                   split into parts (GPUs, streams) with lane_base = the
                                   part's first global lane draws exactly the uniforms
                                   of the unsplit batch; 0 otherwise                */
  uint32_t flags;               /* SPEC_VERIFY_* flags above; 0 for none          */
} spec_verify_args;

/*
 * spec_verify_accept -- the fused verify kernel.
 *
 * Greedy lane (T_b <= 0): a_j = argmax of row j (lowest index on ties); the
 * committed run is d_1..d_n followed by a_n, where n is the number of leading
 * drafts with d_{j+1} == a_j (ignis "One round, step by step", step 4;
 * strata2signal "Guess, then check" and its table).  Since d_{j+1} == a_j for
 * j < n the tokens written are a_0..a_n.
 *
 * Sampled lane (T_b > 0): p_j = softmax(row j / T_b), q_j = softmax(draft row
 * j / T_b).  Draft d_{j+1} is accepted iff u_j < min(1, p_j(d) / q_j(d)); at the
 * first rejection n the model's token is drawn from max(0, p_n - q_n)
 * normalised, or from p_{k_b} if every draft was accepted -- the acceptance rule
 * the strata2signal page cites from Leviathan et al. (2022) as the one that keeps
 * the target's distribution.  The uniforms come from Philox4x64-10 (Salmon et
 * al., SC'11) with key (seed, 0) and counter (j, lane_base + b, 0, 0): word 0 gives u_j,
 * word 1 gives the draw's u'; u = (word >> 40) * 2^-24.  The draw walks token ids
 * upwards and takes the first whose cumulative weight exceeds u' * W.
 *
 * Launch: one thread-block cluster per lane.  When one ring slot holds a
 * CTA's whole row slice and two slots per group fit, the round runs a build
 * with 20 consumer warps in four groups of five (each group double-buffers);
 * a greedy round does so only with slots above 8 KB.  Otherwise a round with
 * draft_logits runs 20 consumer warps in five groups of four (its sampled
 * lanes are bound by instruction issue) and a round without them 16 warps.
 * All compute the same results (sampled lanes within the stated tolerance of
 * the definition).
 * SPEC_VERIFY_BUILD=0|1|2 (16 warps; 20 in groups of four; 20 in groups of
 * five) forces one build.
 *
 * Errors: returns SPEC_ERR_INVALID_ARG for NULL required pointers, V <= 0,
 * lanes <= 0, rows < lanes, ld < V or an unknown dtype; SPEC_ERR_CUDA if the
 * launch fails.  Per-lane errors go to lane_status (see spec_status).
 */
int spec_verify_accept(const spec_verify_args* args, void* stream);

/*
 * spec_commit_state -- roll per-lane recurrent state to the committed count.
 *
 * ignis "One round, step by step", step 5, and FreeToken issue #828, "Design"
 * (per-request state): the verify pass stages one state snapshot per column
 * without touching the live state; the commit keeps exactly the committed
 * prefix, so a rejected draft leaves no trace.  Column c of lane b holds the
 * state after consuming column c (column 0 is the anchor), so
 *
 *   live + b * live_lane_stride  <-  staged + b * staged_lane_stride
 *                                      + (committed[b] - 1) * staged_col_stride
 *
 * copies bytes_per_col bytes for every lane b.  A lane whose committed[b] lies
 * outside 1..cols, or whose lane_status is already non-zero, keeps its live
 * state; the former gets SPEC_ERR_LAYOUT in lane_status.  staged and live must
 * not overlap.  16-byte aligned pointers, strides and sizes use bulk copies;
 * other layouts take a byte-wise path.  If a copy does not complete within the
 * kernel's wait limit (2 s), every lane whose snapshot was not fully copied
 * gets SPEC_ERR_TIMEOUT; such a lane's live state may be partly written.
 *
 * `lane_status` (may be NULL) is read and updated in place, so passing the
 * verify's lane_status skips lanes that failed there.  Launched after
 * spec_verify_accept on the same stream it overlaps that kernel's tail
 * (programmatic dependent launch) and reads committed[] only once the verify
 * kernel has finished.
 *
 * Errors: SPEC_ERR_INVALID_ARG for NULL pointers with lanes > 0, lanes < 0,
 * cols <= 0 or bytes_per_col larger than a stride; SPEC_ERR_CUDA if the launch
 * fails.
 */
int spec_commit_state(const void* staged, void* live, const int32_t* committed,
                      int32_t lanes, int32_t cols, uint64_t bytes_per_col,
                      uint64_t staged_lane_stride, uint64_t staged_col_stride,
                      uint64_t live_lane_stride, int32_t* lane_status, void* stream);

/*
 * spec_round_uniforms -- the uniforms spec_verify_accept draws, for replay and audit.
 *
 * Writes out[(b * positions + j) * 2 + 0] = u_j (the acceptance uniform of the
 * draft at position j of lane b) and out[... + 1] = u'_j (the uniform of an
 * inverse-CDF draw made at position j), for b < lanes and j < positions, from
 * the same device Philox4x64-10 stream the verify kernel uses (key (seed, 0),
 * counter (j, lane_base + b, 0, 0), u = (word >> 40) * 2^-24).  `out` is a
 * device float array of lanes * positions * 2 entries.  Returns
 * SPEC_ERR_INVALID_ARG for a NULL `out` or negative sizes, SPEC_ERR_CUDA if the
 * launch fails.
 */
int spec_round_uniforms(uint64_t seed, uint32_t lane_base, int32_t lanes, int32_t positions, float* out,
                        void* stream);

/* Human-readable name of a spec_status value (static storage, never NULL). */
const char* spec_status_string(int status);

/*
 * Launch-shape overrides.  Environment variables read on every call, for
 * experiments and tests; normal use needs none of them:
 *   SPEC_VERIFY_CLUSTER=C    CTAs per lane (1..16); shrunk only if it cannot be scheduled
 *   SPEC_VERIFY_SLOT_KB=K    largest ring slot in KB (default 40)
 *   SPEC_VERIFY_RING_KB=K    ring size in KB (default: all shared memory left)
 *   SPEC_VERIFY_ORDER=0|1    clusters take lanes longest first (default: only when
 *                            the launch has more lanes than resident clusters)
 *   SPEC_VERIFY_BUILD=0|1|2  which build of the verify kernel runs (see spec_verify_accept);
 *                            SPEC_VERIFY_WARPS=16|20 is the same as 0|1
 *   SPEC_COMMIT_CHUNK_KB, SPEC_COMMIT_NBUF, SPEC_COMMIT_CTAS_PER_SM
 *                            copy shape of spec_commit_state (defaults 32, 2, 3)
 *   SPEC_COMMIT_TEST_WITHHOLD_COPY=1  tests of the failure path only: the
 *                            commit's first CTA never issues its first load, so
 *                            its wait gives up after 2 s (see spec_commit_state)
 * Greedy lanes and the commit give the same results under every override;
 * sampled lanes stay within the stated tolerance of the definition (their
 * fp32 sums are added in an order that follows the shape).
 */

/*
 * spec_verify_launch_shape -- the launch spec_verify_accept would use.
 *
 * Host-only.  Reports the CTAs per lane (one thread-block cluster per lane),
 * threads per CTA, the vocabulary slice each CTA reduces, and the dynamic shared
 * memory per CTA, for a verify over `lanes` lanes and `rows` rows of vocabulary
 * V in `dtype` with 16-byte aligned rows on the current device, after the
 * cluster has been shrunk to what the device can schedule (the same rule the
 * launch applies).  `with_draft` != 0 asks for the launch of a round that
 * passes drafter logits, which can select a different build of the kernel (see
 * spec_verify_accept; `threads` tells the builds apart).  Any output pointer
 * may be NULL.  Returns SPEC_OK, SPEC_ERR_INVALID_ARG, SPEC_ERR_UNSUPPORTED or
 * SPEC_ERR_CUDA.
 */
int spec_verify_launch_shape(int32_t lanes, int32_t rows, int32_t V, spec_dtype dtype, int32_t with_draft,
                             int32_t* cluster_ctas, int32_t* threads, int32_t* slice, int32_t* smem_bytes);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
