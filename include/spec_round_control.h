/*
 * spec_round_control.h -- the rest of a speculative round around the verify:
 * acceptance metrics, the per-lane miss back-off of a drafter, the
 * copy-from-the-conversation (n-gram) drafter and per-row logit penalties.
 *
 * The first two consume the per-lane outputs of spec_verify_accept (committed
 * counts, the draft lengths the round used, lane_status), the drafter writes
 * the next round's drafts; all run on the GPU next to the verify, so a serving
 * loop never copies a round's results to the host to keep its books.  The
 * conventions of spec_verify.h hold: device pointers unless stated otherwise,
 * caller-owned buffers, calls enqueue on `stream` and return at once.
 */
#ifndef SPEC_ROUND_CONTROL_H
#define SPEC_ROUND_CONTROL_H

#include <stdint.h>

#include "spec_verify.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Acceptance counts (strata->signal, "Draft heads and speculative decoding, in
 * plain words" -- "Acceptance: three numbers with one name").  A round of one
 * lane proposes k guesses and keeps the first n = committed - 1 of them.
 */
typedef struct {
  uint64_t rounds;                         /* rounds counted                               */
  uint64_t proposed;                       /* sum of k: guesses proposed                   */
  uint64_t accepted;                       /* sum of n: guesses kept                       */
  uint64_t slot_reached[SPEC_MAX_DRAFTS];  /* [j]: rounds that proposed guess j + 1 (k > j) */
  uint64_t slot_kept[SPEC_MAX_DRAFTS];     /* [j]: rounds in which guess j + 1 survived (n > j) */
} spec_accept_counts;                      /* 264 bytes */

/*
 * spec_accept_counts_update -- add one verify round to the counts.
 *
 * Lane b proposed draft_lens[b] guesses and committed committed[b] tokens.
 * Lanes whose lane_status is not SPEC_OK (lane_status may be NULL: all lanes
 * OK), whose draft length is outside 0..SPEC_MAX_DRAFTS or whose committed
 * count is outside 1..draft_lens[b] + 1 are left out.  per_lane = 0 adds every
 * lane into counts[0] (one struct for the batch); per_lane = 1 adds lane b into
 * counts[b] (counts has `lanes` entries).  counts is device memory the caller
 * zero-fills before the first round.  Reads nothing written by the host in the
 * same call, so it may follow spec_verify_accept on the same stream directly.
 *
 * Errors: SPEC_ERR_INVALID_ARG for NULL committed / draft_lens / counts with
 * lanes > 0, lanes < 0 or per_lane not 0 or 1; SPEC_ERR_CUDA if the launch
 * fails.
 */
int spec_accept_counts_update(const int32_t* committed, const int32_t* draft_lens, const int32_t* lane_status,
                              int32_t lanes, spec_accept_counts* counts, int32_t per_lane, void* stream);

/* The page's quantities, from a set of counts. */
typedef struct {
  double accepted_per_proposed;            /* accepted / proposed                          */
  double tokens_per_round;                 /* 1 + accepted / rounds                        */
  double by_slot[SPEC_MAX_DRAFTS];         /* slot_kept[j] / rounds                        */
  double given_previous[SPEC_MAX_DRAFTS];  /* slot_kept[j] / slot_kept[j - 1] (j = 0: / rounds) */
  int32_t depth;                           /* proposed / rounds, rounded: the alpha's depth g */
  int32_t reserved;
  double implied_alpha;                    /* alpha in [0, 1] with
                                              (1 - alpha^(g + 1)) / (1 - alpha) = tokens_per_round */
} spec_accept_rates;

/*
 * spec_accept_rates_from_counts -- derive the rates (host-only, both pointers
 * host memory).  A ratio with a zero denominator is NaN.  Returns
 * SPEC_ERR_INVALID_ARG for a NULL pointer, SPEC_OK otherwise.
 */
int spec_accept_rates_from_counts(const spec_accept_counts* counts, spec_accept_rates* rates);

/*
 * Miss back-off (mashbox docs, "Speculative decoding" -- "What it does for
 * you"): after 4 counted passes in a row in which the model kept none of a
 * lane's guesses the lane makes no guesses for 16 passes; each further 4 such
 * passes in a row double the wait, up to 256; a pass that keeps a guess sets
 * the wait back to 16.  One verify round is one pass of one device call: a
 * round in which no lane of the batch proposed a guess counts toward no lane's
 * misses, only toward the wait of a lane already waiting, and in a round that
 * speculates every lane that may guess counts, with or without a guess.
 */
typedef struct {
  int32_t misses;   /* counted passes in a row in which no guess was kept */
  int32_t backoff;  /* length of the next wait, 16 .. 256                 */
  int32_t wait;     /* passes left in the current wait; 0: the lane may guess */
  int32_t reserved;
} spec_backoff_state;

/*
 * spec_backoff_init -- state of `lanes` lanes that have not missed yet
 * (misses 0, backoff 16, wait 0).  Errors: SPEC_ERR_INVALID_ARG for a NULL
 * `states` with lanes > 0 or lanes < 0; SPEC_ERR_CUDA if the launch fails.
 */
int spec_backoff_init(spec_backoff_state* states, int32_t lanes, void* stream);

/*
 * spec_backoff_step -- advance every lane by one verify round and write the
 * draft length each lane may use in the next round.
 *
 * proposed[b] is the draft length lane b used in the round (0 while it was
 * waiting); the round kept committed[b] - 1 of its guesses.  A lane whose
 * lane_status is not SPEC_OK (lane_status may be NULL) kept none.  The lane's
 * next draft length is draft_tokens (0 <= draft_tokens <= SPEC_MAX_DRAFTS)
 * unless it is waiting, then 0; next_draft_lens may be the array the next
 * round reads as draft_lens.  One CTA walks all lanes (the round-level
 * "did any lane guess" needs the whole batch).
 *
 * Errors: SPEC_ERR_INVALID_ARG for NULL pointers (other than lane_status) with
 * lanes > 0, lanes < 0 or draft_tokens outside 0..SPEC_MAX_DRAFTS;
 * SPEC_ERR_CUDA if the launch fails.
 */
int spec_backoff_step(spec_backoff_state* states, const int32_t* proposed, const int32_t* committed,
                      const int32_t* lane_status, int32_t lanes, int32_t draft_tokens, int32_t* next_draft_lens,
                      void* stream);

/* Longest suffix spec_ngram_draft matches. */
#define SPEC_NGRAM_MAX_MATCH 16

/*
 * spec_ngram_draft -- copy from the conversation (mashbox docs, "Speculative
 * decoding" -- "Options", --speculation ngram): look up the last few tokens of
 * each lane's history earlier in it and propose the tokens that followed them
 * there.
 *
 * Lane b's history is tokens[hist_offsets[b] .. hist_offsets[b + 1]), L tokens
 * ending with the anchor.  For a match length m the suffix is the last m
 * tokens; an earlier occurrence of it ends at a position i < L.  The drafter
 * takes the longest m in [match_min, match_max] (and m < L) that has an earlier
 * occurrence, the most recent such occurrence (largest i), and proposes the
 * tokens history[i .. min(i + k, L)).  It writes draft_lens[b] (0 when no
 * suffix of an allowed length occurs earlier) and drafts[b * draft_stride + j]
 * for j < draft_lens[b]; the other slots are left as they are.  One CTA per
 * lane reads the lane's history once (plus up to match_max - 1 repeats of each
 * token, from L1).
 *
 * Errors: SPEC_ERR_INVALID_ARG for NULL pointers with lanes > 0, lanes < 0,
 * k outside 0..SPEC_MAX_DRAFTS, draft_stride < k, or match lengths outside
 * 1 <= match_min <= match_max <= SPEC_NGRAM_MAX_MATCH; SPEC_ERR_CUDA if the
 * launch fails.  Offsets must be non-decreasing (a lane with
 * hist_offsets[b + 1] < hist_offsets[b] is treated as empty).
 */
int spec_ngram_draft(const int32_t* tokens, const int64_t* hist_offsets, int32_t lanes, int32_t k,
                     int32_t match_min, int32_t match_max, int32_t* drafts, int32_t draft_stride,
                     int32_t* draft_lens, void* stream);

/*
 * spec_apply_penalties -- per-row presence and frequency penalties on the
 * target logits of a round (FreeToken tracking issue #828, "PRs": #836 verifies
 * on the target side with per-row presence and frequency penalties), applied
 * on the same stream right before spec_verify_accept.
 *
 * THE CALLER'S TARGET LOGITS ARE OVERWRITTEN: the penalised values replace
 * the stored ones in place (keep a copy if the raw logits are needed again).
 *
 * Row j of lane b scores the position after the anchor and d_1..d_j, so token
 * t's count in that row is c = (its count in the lane's history) + (its count
 * among d_1..d_j).  Every token with c > 0 gets
 *     z = x - (frequency[b] * c + presence[b])
 * in fp32 with the roundings in that order (product, sum, difference); a bf16
 * logit is then rounded to the nearest bf16 (ties to even) and stored back.
 * Other tokens and the drafter's logits are not touched.
 *
 * target_logits, dtype, ld, V, lanes, row_offsets, draft_tokens and
 * draft_lens are those of the round's spec_verify_args.  Lane b's history
 * counts are pen_tokens / pen_counts [pen_offsets[b] .. pen_offsets[b + 1]):
 * distinct token ids in ascending order with counts >= 1; ids outside [0, V)
 * are ignored.  presence and frequency are per lane (may be NULL: 0).  One CTA
 * per lane; touches (history + drafts) x (k_b + 1) logits of the lane.
 *
 * lane_status (out [lanes], may be NULL) gets, per lane: SPEC_OK (penalties
 * applied); SPEC_ERR_INVALID_ARG if the lane's history list is not strictly
 * ascending (a repeated or out-of-order id) or holds a count < 1;
 * SPEC_ERR_LAYOUT if row_offsets disagree with draft_lens; SPEC_ERR_UNSUPPORTED
 * if k_b > SPEC_MAX_DRAFTS.  A lane with any of these keeps its logits
 * unchanged.  The list is checked on the device before any logit of the lane
 * is written.  Use a buffer other than the verify's lane_status (the verify
 * writes every lane's status), or read it before the verify runs.
 *
 * Errors: SPEC_ERR_INVALID_ARG for NULL target_logits / row_offsets /
 * draft_tokens / draft_lens / pen_* with lanes > 0, lanes < 0, V <= 0, ld < V
 * or an unknown dtype; SPEC_ERR_CUDA if the launch fails.
 */
int spec_apply_penalties(void* target_logits, spec_dtype dtype, int64_t ld, int32_t V, int32_t lanes,
                         const int32_t* row_offsets, const int32_t* draft_tokens, const int32_t* draft_lens,
                         const int32_t* pen_tokens, const int32_t* pen_counts, const int64_t* pen_offsets,
                         const float* presence, const float* frequency, int32_t* lane_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_ROUND_CONTROL_H */
