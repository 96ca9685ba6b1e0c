/*
 * sdv_draft.h -- n-gram (prompt-lookup) drafting on the host.
 *
 * Source: the splicedso primer on speculative decoding, section "When it
 * works": a variant needs no draft model at all -- n-gram drafting guesses by
 * copying text already in the prompt, and was the best method measured for
 * edits.  Copy-style drafts are deterministic, so they pair with greedy
 * verification (sdv_set_sampling(SDV_SAMPLING_GREEDY) in sdv.h); for rejection
 * sampling their draft distribution is a point mass on the copied token.
 *
 * Rule: take the longest suffix of the history, n tokens long with
 * max_n >= n >= min_n, that also occurs earlier in the history; at its most
 * recent earlier occurrence, copy the tokens that followed it, up to gamma of
 * them and never past the end of the history.  No match: no drafts.
 *
 * Host-only, synchronous, thread-safe (no state).
 */
#ifndef SDV_DRAFT_H
#define SDV_DRAFT_H

#include "sdv.h"

#ifdef __cplusplus
extern "C" {
#endif

/* One sequence.  history [len] (host), 1 <= min_n <= max_n, gamma >= 0;
 * drafts (host, >= gamma entries).  Returns the number of drafts written
 * (0 .. gamma), or -1 on a bad argument. */
int sdv_ngram_draft(const int *history, int len, int min_n, int max_n, int gamma, int *drafts);

/* A batch: sequence b's history is tokens[offsets[b] .. offsets[b + 1]) (host;
 * offsets [B + 1], non-decreasing).  Writes draft_lens [B] and drafts
 * [B, gamma_max] (row b holds draft_lens[b] tokens; the rest are -1).
 * SDV_ERR_INVALID_ARG on a bad argument. */
sdv_status sdv_ngram_draft_batch(const int *tokens, const long long *offsets, int B, int min_n, int max_n,
                                 int gamma_max, int *draft_lens, int *drafts);

#ifdef __cplusplus
}
#endif
#endif /* SDV_DRAFT_H */
