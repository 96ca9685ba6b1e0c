/*
 * sdv_sched.h -- host-side continuous-batching scheduler with an adaptive
 * draft length, driving the verify step of sdv.h.
 *
 * Sources:
 *  - "Speculative Decoding and Batching Compete for the Same Compute Slack on
 *    RDNA4", sections "The budget is fixed, and the batch is inside it" and
 *    "What the budget says to build": one verify pass hides a fixed budget of
 *    token rows under the weight stream; B live sequences commit B of them, so
 *    each may draft about (budget - B) / B tokens, recomputed every step from
 *    the live batch size.
 *  - "Why Static Batching Wastes an RX 9070 XT Agent Swarm and Continuous
 *    Batching Wins It Back", sections "What a draining batch actually costs"
 *    and "Continuous batching refills the slot instead of freezing it": batch
 *    membership is decided every step; a finished sequence leaves and a queued
 *    one takes its slot on the next step.  The two static policies of that
 *    page (frozen width, shrinking width) are kept as comparison policies.
 *
 * The scheduler owns no device memory.  It mirrors what the device-side
 * realignment of sdv_verify_step does to the slot table (length L + a + 1,
 * finishing at the output length, stable compaction of the survivors, each
 * live sequence holding ceil((L + gamma_max + 1) / page_size) pages), so that
 * from the accepted counts alone it knows the next step's live slots, free
 * slots and free pages.  Newly admitted sequences are appended to the device
 * slot table by sdv_admit (sdv.h).
 *
 * Every call is host-only, synchronous and not thread-safe per scheduler.
 */
#ifndef SDV_SCHED_H
#define SDV_SCHED_H

#include "sdv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct sdv_sched sdv_sched;

enum {
  SDV_SCHED_CONTINUOUS = 0,    /* refill free slots from the queue every step */
  SDV_SCHED_STATIC = 1,        /* admit a full group only when every slot is empty; the paid width stays
                                  frozen at the group's size until its last sequence finishes */
  SDV_SCHED_STATIC_SHRINK = 2  /* admit a group only when empty; the paid width shrinks as sequences finish */
};

typedef struct {
  int max_slots;         /* slots of the verify batch (B_max), >= 1 */
  int gamma_max;         /* cap on every draft length; the verify context's gamma_max */
  int budget_rows;       /* verify rows one step may carry: live * (gamma + 1) <= budget_rows when gamma > 0 */
  int page_size;         /* KV positions per page (16) */
  int pool_pages;        /* pages of the KV pool, all free at creation */
  int max_pages_per_seq; /* page-table width: a sequence may never need more */
  int policy;            /* SDV_SCHED_* */
} sdv_sched_config;

/* One planned step. */
typedef struct {
  int live;     /* slots holding an unfinished sequence: the verify batch's B */
  int width;    /* slots the step is paid for (live, or the frozen group width under SDV_SCHED_STATIC) */
  int gamma;    /* draft length of every live slot */
  int rows;     /* R = live * (gamma + 1) */
  int drafts;   /* G = live * gamma */
  int admitted; /* sequences appended at slots [live - admitted, live) by this plan */
} sdv_sched_step;

typedef struct {
  long long steps;          /* completed steps */
  long long emitted;        /* tokens emitted (sum of accepted + 1) */
  long long slot_steps_paid;  /* sum over steps of width */
  long long slot_steps_live;  /* sum over steps of live */
  long long finished;       /* sequences retired */
  long long admitted;       /* sequences admitted */
  int queued;               /* sequences waiting */
  int free_pages;           /* pages the device free stack holds after the last step */
  int live;                 /* sequences holding a slot now */
} sdv_sched_stats;

/* The draft-length rule alone: gamma = clamp(floor((budget_rows - live) / live), 0, gamma_max);
 * 0 when live <= 0.  E.g. budget 24: 23, 11, 5, 2, 0 drafts each at 1, 2, 4, 8, 16 live sequences. */
int sdv_sched_gamma(int budget_rows, int live, int gamma_max);

/* Create a scheduler (host memory only).  SDV_ERR_INVALID_ARG on a bad config. */
sdv_status sdv_sched_create(const sdv_sched_config *cfg, sdv_sched **out);
void sdv_sched_destroy(sdv_sched *s);

/* Queue a sequence in arrival order.  ctx_len: tokens already in its KV cache
 * (prefill is outside the verify step); out_len >= 1: it finishes once it has
 * emitted that many tokens; id: the caller's handle.  SDV_ERR_CAPACITY if the
 * sequence could outgrow max_pages_per_seq or the whole pool. */
sdv_status sdv_sched_submit(sdv_sched *s, long long id, int ctx_len, int out_len);

/* Plan the next step: admit queued sequences in arrival order as the policy
 * allows, while a free slot exists and the free pages cover the newcomer plus
 * one step of growth of every live sequence; then pick gamma from the live
 * count.  admit_ctx / admit_out (host, >= max_slots entries each, may be NULL
 * when nothing is queued) receive the ctx_len and out_len of the admitted
 * sequences; slot_ids (host, >= max_slots, may be NULL) the id of every live
 * slot in slot order.  Calling plan twice without complete in between is
 * SDV_ERR_INVALID_ARG. */
sdv_status sdv_sched_plan(sdv_sched *s, sdv_sched_step *step, int *admit_ctx, int *admit_out,
                          long long *slot_ids);

/* Account the planned step from its accepted counts (host, [live], each in
 * [0, gamma]): every live sequence advances by accepted + 1 tokens; those that
 * reach their output length are retired and the survivors keep their order.
 * finished_ids (host, >= live entries, may be NULL) receives the retired ids in
 * slot order and *n_finished (may be NULL) their count. */
sdv_status sdv_sched_complete(sdv_sched *s, const int *accepted, long long *finished_ids, int *n_finished);

/* Counters since creation. */
sdv_status sdv_sched_get_stats(const sdv_sched *s, sdv_sched_stats *st);

/* Per-slot mirror of the live sequences (host arrays, >= live entries each, any
 * may be NULL): KV length, tokens generated, output length, pages held. */
sdv_status sdv_sched_slots(const sdv_sched *s, int *seq_lens, int *gen_counts, int *out_lens, int *num_pages);

#ifdef __cplusplus
}
#endif
#endif /* SDV_SCHED_H */
