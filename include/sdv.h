/*
 * sdv.h -- C ABI of the ragged batched speculative-verify step on GB300 (sm_103a).
 *
 * The step verifies B live sequences in one pass.  Sequence b brings gamma_b
 * draft tokens, so the batch is ragged: R = sum_b (gamma_b + 1) verify rows and
 * G = sum_b gamma_b draft rows.  One pass
 *   (a) streams one decoder layer's weights (fused QKV, O, SwiGLU gate/up/down;
 *       bf16 or int4 group-32 with fp16 scales) once against all R rows,
 *   (b) runs GQA attention of every row over its own sequence's paged KV cache,
 *       causal inside the draft block,
 *   (c) computes LM-head logits and a softmax for every row,
 *   (d) accepts a prefix of each sequence's drafts by rejection sampling and
 *       draws one more token (residual resample, or a bonus token when every
 *       draft is accepted),
 *   (e) realigns each sequence's KV length, next position, page list and slot
 *       from its own accepted count, never padding to the longest run.
 * Sources: "Speculative Decoding at High Batch Size: Where the 3x Speedup Turns
 * Into a Tax" (section "Why do the headline speedups all come from batch 1?":
 * all drafts verified in one forward pass; FAQ "Does speculative decoding
 * change the output of the model?": rejection sampling keeps the output
 * distribution); the splicedso primer on speculative decoding (section "The
 * idea": keep the agreed guesses up to the first disagreement, add one token of
 * the model's own); "Speculative Decoding and Batching Compete for the Same
 * Compute Slack on RDNA4" (section "The batch also goes ragged": per-sequence
 * accept counts desynchronise positions, masks and KV lengths); "Why Static
 * Batching Wastes an RX 9070 XT Agent Swarm and Continuous Batching Wins It
 * Back" (section "Continuous batching refills the slot instead of freezing it").
 *
 * Conventions for every entry point:
 *  - Pointers marked "device" are CUDA device pointers owned by the caller; the
 *    library never allocates, frees or retains them beyond the call (the
 *    context keeps the weight and workspace pointers given to sdv_create).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Every call only enqueues work on that stream and returns; nothing is
 *    synchronised unless the entry point says so.
 *  - bf16 data are raw 16-bit patterns; "[a, b]" is row-major with b fastest.
 *  - Errors the host can see (null pointer, bad size, missing capacity, CUDA
 *    launch failure) are returned at once and nothing is enqueued.  Errors
 *    only the device can see (a token, page id or draft length out of range,
 *    row counts that do not add up, a distribution with no mass) are written
 *    to the device status word `result->status` (SDV_OK when clean); every
 *    later kernel of the same call reads it and returns without touching its
 *    outputs.  No kernel traps.  Read the word with sdv_read_status.
 */
#ifndef SDV_H
#define SDV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SDV_OK = 0,
  SDV_ERR_INVALID_ARG = 1, /* host: null pointer, non-positive or inconsistent size */
  SDV_ERR_CAPACITY = 2,    /* too few free pages / pages beyond max_pages_per_seq / workspace too small */
  SDV_ERR_PAGE_RANGE = 3,  /* device: page id outside the pool, or pages not covering a row */
  SDV_ERR_CUDA = 4,        /* a CUDA runtime call failed (the CUDA error is in sdv_last_cuda_error) */
  SDV_ERR_TIMEOUT = 5,     /* device: a bounded wait inside a kernel gave up */
  SDV_ERR_BAD_INPUT = 6,   /* device: token >= vocab, gamma_b > gamma_max, row sums mismatch, zero mass */
  SDV_ERR_UNSUPPORTED = 7, /* host: a shape this build has no kernel for (e.g. head_dim not 64/128) */
  SDV_ERR_INTERNAL = 8     /* host: the context itself could not be allocated */
} sdv_status;

enum { SDV_WEIGHTS_BF16 = 0, SDV_WEIGHTS_INT4_G32 = 1 };

/* Model and step dimensions.  head_dim in {64, 128}; n_q a multiple of n_kv;
 * hidden, n_q*head_dim and ffn multiples of 64 (of 256 for int4); page_size 16.
 * gamma_max bounds every gamma_b and sets how many pages realignment keeps;
 * (gamma_max + 1) * n_q / n_kv is at most 64 with head_dim 128, 48 with 64. */
typedef struct {
  int hidden, n_q, n_kv, head_dim, ffn, vocab, page_size, gamma_max;
  int weight_format; /* SDV_WEIGHTS_BF16 or SDV_WEIGHTS_INT4_G32 */
  float rms_eps;     /* RMSNorm epsilon (1e-6) */
  float rope_theta;  /* rotary base (1e6) */
} sdv_config;

/* Weights (device, read-only, must stay valid for the context's life).
 * bf16 projections are [N, K] (row n = output feature n):
 *   w_qkv [(n_q + 2 n_kv) * head_dim, hidden]: query heads, then key heads, then value heads
 *   w_o [hidden, n_q*head_dim], w_gate / w_up [ffn, hidden], w_down [hidden, ffn].
 * int4 group-32 projections: w_* uint8 [N, K/2] (low nibble = even k, two's
 * complement code in [-8, 7]) and s_* fp16 [N, K/32], weight = scale * code.
 * emb and w_lm are bf16 [vocab, hidden]; gains bf16 [hidden]. */
typedef struct {
  const void *emb, *w_qkv, *w_o, *w_gate, *w_up, *w_down, *w_lm;
  const void *s_qkv, *s_o, *s_gate, *s_up, *s_down; /* int4 scales; NULL for bf16 */
  const void *g_attn, *g_ffn, *g_final;
} sdv_weights;

/* One verify step's inputs (device pointers unless noted).
 *  B, R, G (host ints): slots, verify rows sum(gamma_b+1), draft rows sum(gamma_b).
 *  seq_lens [B]    L_b, tokens already in slot b's cache.
 *  draft_lens [B]  gamma_b in [0, gamma_max].
 *  tokens [R]      rows of slot b start at sum_{j<b}(gamma_j+1): row 0 = last
 *                  committed token (position L_b, not yet cached), row i = draft i.
 *  draft_probs [G, V] fp32: row sum_{j<b}gamma_j + i = q_i, the draft
 *                  distribution draft token i+1 was proposed from.
 *  uniforms [R] fp32 in [0,1): row i < gamma_b = acceptance draw of draft i+1,
 *                  row gamma_b = draw of the final token.
 *  kv_pool         bf16 [num_pool_pages, n_kv, 2 (K then V), page_size, head_dim].
 *  page_table [B, max_pages_per_seq]: pool page of each 16-position block; the
 *                  first num_pages[b] entries are valid and must cover
 *                  L_b + gamma_b + 1 positions.  Updated in place by realignment.
 *  num_pages [B]   updated in place by realignment.
 *  free_pages [num_pool_pages]: free stack, top at index *num_free_in - 1;
 *                  updated in place (entries at and above the old top).
 *  num_free_in / num_free_out: device scalars (may be the same pointer).
 *  gen_counts / gen_limits [B] or NULL: tokens generated so far and the output
 *                  length at which a sequence finishes (both NULL = none finish).
 *  tree_parents [R] or NULL: token trees ("Speculative Decoding and Batching
 *                  Compete for the Same Compute Slack on RDNA4", table in "What
 *                  the budget says to build": a small tree at low batch).  Row i
 *                  of slot b is a tree node whose parent is row tree_parents[...]
 *                  of the same slot (-1 for row 0, the root; otherwise < i;
 *                  up to 64 rows per slot).  Node i sits at position L_b +
 *                  depth(i), writes its K/V at slot L_b + i, and attends to the
 *                  cache and its own ancestors.  Trees are verified greedily
 *                  (sdv_set_sampling(SDV_SAMPLING_GREEDY); SDV_ERR_UNSUPPORTED
 *                  otherwise): from the root, descend into the child carrying
 *                  the argmax of the current row (the smallest such index); the
 *                  accepted count is the depth reached, the emitted tokens are
 *                  the path's tokens and the argmax at its end, and realignment
 *                  moves the path's K/V rows to slots L_b + 1 .. L_b + a_b.
 *                  NULL: every slot is a chain (row i's parent is row i - 1). */
typedef struct {
  int B, R, G;
  const int *seq_lens, *draft_lens, *tokens;
  const float *draft_probs, *uniforms;
  void *kv_pool;
  int num_pool_pages;
  int *page_table;
  int max_pages_per_seq;
  int *num_pages;
  int *free_pages;
  const int *num_free_in;
  int *num_free_out;
  const int *gen_counts, *gen_limits;
  const int *tree_parents;
} sdv_batch;

/* One verify step's outputs (device pointers; NULL = not wanted, except status).
 *  accepted [B]          a_b, accepted drafts of slot b.
 *  final_tokens [B]      the token drawn after the accepted prefix.
 *  emitted_tokens [R]    slot b's accepted drafts then its final token, packed
 *                        at emitted_offsets[b]; emitted_offsets [B+1].
 *  new_seq_lens [B]      L_b + a_b + 1 (also the next step's row-0 position).
 *  finished [B]          1 when gen_counts + a_b + 1 >= gen_limits.
 *  new_gen_counts [B]    gen_counts + a_b + 1.
 *  next_src [B], num_live (scalar): surviving slots in order; next slot j comes
 *                        from old slot next_src[j], j < *num_live.
 *  next_seq_lens [B], next_num_pages [B], next_page_table [B, max_pages_per_seq],
 *  next_gen_counts [B]:  the per-slot state gathered through next_src.
 *  accept_tested / accept_accepted [gamma_max]: per draft position, sequences
 *                        that tested it / accepted it (added to, never cleared).
 *  logits [R, V], probs [R, V] fp32: the target's logits and softmax (debug).
 *  status (scalar, required): device status word, see the conventions above. */
typedef struct {
  int *accepted, *final_tokens, *emitted_tokens, *emitted_offsets, *new_seq_lens;
  int *finished, *new_gen_counts;
  int *next_src, *num_live, *next_seq_lens, *next_num_pages, *next_page_table, *next_gen_counts;
  int *accept_tested, *accept_accepted;
  float *logits, *probs;
  int *status;
} sdv_result;

typedef struct sdv_ctx sdv_ctx;

/* Bytes of device workspace a context needs for up to max_rows verify rows
 * and max_slots slots.  0 on invalid config. */
size_t sdv_workspace_size(const sdv_config *cfg, int max_rows, int max_slots);

/* Create a context on the current device.  `workspace` (device, caller-owned,
 * >= sdv_workspace_size bytes, 256-byte aligned) is used by every call on
 * this context, so calls on one context must not overlap in time.  Builds
 * TMA descriptors for the weights and the workspace; enqueues nothing. */
sdv_status sdv_create(const sdv_config *cfg, const sdv_weights *w, void *workspace,
                      size_t workspace_bytes, int max_rows, int max_slots, sdv_ctx **out);
void sdv_destroy(sdv_ctx *ctx);

/* The whole step (a)-(e) for one batch.  See sdv_batch / sdv_result. */
sdv_status sdv_verify_step(sdv_ctx *ctx, const sdv_batch *batch, sdv_result *result, void *stream);

/* Steps (d) and the packing of (e) on given target probabilities: probs [R, V]
 * fp32 (device) replaces the forward.  Uses batch->tokens, draft_lens,
 * draft_probs, uniforms, seq_lens and the realignment fields exactly as
 * sdv_verify_step does, and writes the same result fields except logits/probs.
 * With the same probs, q and u the result is bit-identical to the step's rule. */
sdv_status sdv_accept(sdv_ctx *ctx, const float *probs, const sdv_batch *batch,
                      sdv_result *result, void *stream);

/* sdv_accept without a context, a workspace or any allocation.  The pages
 * describe no such call: it is here for callers that cannot allocate device
 * memory when they verify (memory carved up once at start-up, work recorded
 * inside a CUDA-graph capture where cudaMalloc is not allowed, a plugin whose
 * host owns every allocation).  Same inputs, rule and outputs as sdv_accept;
 * cfg supplies vocab, page_size, gamma_max (<= 63), n_kv and head_dim.
 * Scratch lives in one static device array of about 2.1 MB that every GPU
 * loading the library holds until exit.  Limits: B <= 256, R <= 2048,
 * vocab <= 262144; beyond them SDV_ERR_CAPACITY and nothing is enqueued.
 * The first call on a device looks the array up (cudaGetSymbolAddress) with
 * that device current; make it before any stream capture.  The address is
 * looked up again when a later call finds another CUDA context current (after
 * a cudaDeviceReset), so the first call after a reset is a set-up call too.
 * All calls on a device share the array and it keeps the last call's contents
 * (its counters are cleared by every call); calls that overlap on the GPU race. */
sdv_status sdv_accept_static(const sdv_config *cfg, const float *probs, const sdv_batch *batch,
                             sdv_result *result, void *stream);

/* Step (e) alone from given accepted counts and final tokens (device [B] each,
 * read from result->accepted / result->final_tokens).  Writes emitted
 * tokens/offsets, lengths, pages, free stack and the next-slot view. */
sdv_status sdv_realign(sdv_ctx *ctx, const sdv_batch *batch, sdv_result *result, void *stream);

/* Admission of new sequences into a slot table, the device half of continuous
 * batching ("Why Static Batching Wastes an RX 9070 XT Agent Swarm and
 * Continuous Batching Wins It Back", section "Continuous batching refills the
 * slot instead of freezing it": a finished sequence's slot takes a waiting
 * one on the very next step).  The table is the realignment's next-slot view
 * (result->next_seq_lens, next_num_pages, next_page_table, next_gen_counts)
 * holding `live` survivors; newcomer j goes to slot live + j with length
 * ctx_lens[j] (positions already cached: prefill is not part of the step),
 * generated count 0, output length out_lens[j], and
 * ceil((ctx_lens[j] + gamma_max + 1) / page_size) pages popped from the top of
 * the free stack in admission order (newcomer j's k-th page is the k-th popped
 * for it); the rest of its page-table row is -1.  When gen_limits_prev and
 * next_src are given, the survivors' output lengths are first gathered into
 * gen_limits[0, live) (gen_limits_prev must not alias gen_limits).
 * Host errors: live + n > slots, aliasing, null table pointers.  Device
 * errors in *status: *num_live != live or a negative length (SDV_ERR_BAD_INPUT),
 * too few free pages or a row wider than max_pages_per_seq (SDV_ERR_CAPACITY);
 * nothing is written then.  A nonzero *status on entry makes it a no-op. */
typedef struct {
  int live;                   /* host: survivors already at slots [0, live) */
  int n;                      /* host: sequences appended at slots [live, live + n), n <= 1024 */
  int slots;                  /* host: rows of the slot table */
  const int *num_live;        /* device scalar or NULL: the realignment's survivor count */
  const int *next_src;        /* device [live] or NULL: old slot of each survivor */
  const int *gen_limits_prev; /* device [old B] or NULL: output lengths before the compaction */
  const int *ctx_lens;        /* device [n] */
  const int *out_lens;        /* device [n] */
  int *seq_lens, *num_pages, *gen_counts, *gen_limits; /* device [slots] */
  int *page_table;            /* device [slots, max_pages_per_seq] */
  int max_pages_per_seq;
  int *free_pages;            /* device free stack, top at *num_free - 1 */
  int *num_free;              /* device scalar, lowered by the pages popped */
} sdv_admission;
sdv_status sdv_admit(sdv_ctx *ctx, const sdv_admission *a, int *status, void *stream);

/* y = x W^T for one of the context's projections, fp32 output without
 * rounding (parity tests of the weight-streaming GEMM).  which: 0 qkv, 1 o,
 * 2 gate, 3 up, 4 down, 5 lm_head.  x [rows, K] (device): x_format 0 = bf16,
 * 1 = fp32 (each value enters the MMAs as a bf16 hi + lo pair, the path the
 * step's layer GEMMs take).  y fp32 [rows, N] (device).  rows <= max_rows.
 * The GEMM's own status word is internal: a device-side timeout cannot be
 * read back from this entry point (the step's entry points report it). */
sdv_status sdv_linear(sdv_ctx *ctx, int which, const void *x, int x_format, float *y, int rows, void *stream);

/* Step (b) alone: q fp32 [R, n_q, head_dim] already rotated, the cache
 * already holding every row's K/V at L_b + i.  out fp32 [R, n_q*head_dim].
 * Uses batch->seq_lens, draft_lens, page_table, kv_pool, B, R. */
sdv_status sdv_attention(sdv_ctx *ctx, const void *q, const sdv_batch *batch, void *out,
                         int *status, void *stream);

/* Phases of sdv_verify_step, in launch order, for live timing with CUDA events. */
enum {
  SDV_PHASE_PROLOGUE = 0, /* validation, row tables, embedding + RMSNorm */
  SDV_PHASE_QKV = 1,      /* fused QKV GEMM + RoPE + KV append */
  SDV_PHASE_ATTN = 2,     /* paged attention (+ merge of split sequences) */
  SDV_PHASE_O = 3,        /* O projection + residual */
  SDV_PHASE_FFN = 4,      /* RMSNorm, gate/up + SwiGLU, down + residual, final RMSNorm */
  SDV_PHASE_LMHEAD = 5,   /* LM-head GEMM with per-tile softmax statistics (one kernel) */
  SDV_PHASE_ACCEPT = 6,   /* acceptance + final-token sampling (+ debug probs) */
  SDV_PHASE_REALIGN = 7,  /* realignment */
  SDV_PHASES = 8
};

/* Optional phase timing.  events: n = SDV_PHASES + 1 cudaEvent_t handles
 * (passed as void*, created by the caller); each later sdv_verify_step on
 * this context records events[k] on its stream when phase k starts and
 * events[SDV_PHASES] after the last phase.  A NULL entry skips that
 * boundary: an event recorded between two kernels stops the second from
 * starting while the first finishes, so record only the boundaries you read.
 * events = NULL (n = 0) turns timing off.  The context keeps the handles,
 * not ownership.  A call recorded into a CUDA graph (stream capture) records
 * the events as external event nodes, so they time the graph's runs. */
sdv_status sdv_set_phase_events(sdv_ctx *ctx, void *const *events, int n);

/* Which kernel runs the context's GEMMs: SDV_GEMM_AUTO (by row count),
 * SDV_GEMM_MMA_SYNC (bf16 mma.sync, built for a handful of rows) or
 * SDV_GEMM_TCGEN05 (5th-generation tensor cores with TMEM accumulators, for
 * row counts where the contraction is dense).  Results agree up to fp32
 * summation order.  Host-side setting; takes effect on the next call. */
enum { SDV_GEMM_AUTO = 0, SDV_GEMM_MMA_SYNC = 1, SDV_GEMM_TCGEN05 = 2 };
sdv_status sdv_set_gemm_path(sdv_ctx *ctx, int path);

/* How the step verifies drafts and draws the final token.
 * SDV_SAMPLING_STOCHASTIC (default): rejection sampling against the draft
 *   distributions -- keep draft i+1 iff u < min(1, p/q), then draw from the
 *   residual max(0, p - q) or, with every draft kept, from p ("Speculative
 *   Decoding at High Batch Size", FAQ "Does speculative decoding change the
 *   output of the model?"; splicedso primer, section "The idea").
 * SDV_SAMPLING_GREEDY: the temperature -> 0 case, the usual pairing with
 *   copy-style (n-gram) drafts (splicedso primer, section "When it works"):
 *   keep draft i+1 iff it is the argmax of p at row i (smallest index among
 *   equal maxima), then emit the argmax of the first row not kept.  The output
 *   is then exactly what greedy decoding of the target produces.  draft_probs
 *   and uniforms are not read (may be NULL).
 * Applies to sdv_verify_step and sdv_accept on this context. */
enum { SDV_SAMPLING_STOCHASTIC = 0, SDV_SAMPLING_GREEDY = 1 };
sdv_status sdv_set_sampling(sdv_ctx *ctx, int mode);

/* Which kernel runs the step's attention: SDV_GEMM_AUTO (tcgen05 when
 * head_dim is 128 and the batch has at least 4 sequences, or whenever
 * (gamma_max + 1) * n_q / n_kv exceeds 48; else mma.sync), SDV_GEMM_MMA_SYNC
 * (up to 48 query vectors per sequence and kv head), or SDV_GEMM_TCGEN05
 * (head_dim 128, up to 64 query vectors: up to 48 in one work item, past
 * 48 taken 32 per work item).  A shape
 * the chosen kernel does not take is SDV_ERR_UNSUPPORTED from the step and
 * sdv_attention, before anything is enqueued.  Results agree up to fp32
 * summation order.  Host-side setting; takes effect on the next call. */
sdv_status sdv_set_attention_path(sdv_ctx *ctx, int path);

/* Test hook for the device-side failure path; 0 (the default) turns it off.
 * The pages describe no such call.  With stall_ns > 0, every later call on
 * this context that runs the step's first kernel (sdv_verify_step,
 * sdv_accept, sdv_realign, sdv_attention) has that kernel wait on a barrier
 * that nothing completes, through the same time-bounded wait every pipelined
 * kernel uses, for stall_ns nanoseconds; the wait gives up, records
 * SDV_ERR_TIMEOUT in the status word, and every later kernel of the call
 * returns without touching its outputs.  The context stays usable: set 0 and
 * the next call runs normally.  Host-side setting; takes effect on the next
 * call. */
sdv_status sdv_set_stall_test(sdv_ctx *ctx, unsigned long long stall_ns);

/* Synchronise `stream` and copy the device status word to *host_status. */
sdv_status sdv_read_status(const int *status, int *host_status, void *stream);

/* Last CUDA error code seen by the library on this thread (0 if none). */
int sdv_last_cuda_error(void);

/* Number of kernels the library has launched since load (all contexts). */
unsigned long long sdv_kernel_launches(void);

/* Step timeline (a library built with -DSDV_TRACE; SDV_ERR_UNSUPPORTED from
 * any other build).  table: device memory of 32 x 3 unsigned 64-bit words,
 * owned by the caller, or NULL to stop.  Every kernel the library launches
 * afterwards stamps the GPU global timer (ns) into its row: word 0 the
 * earliest CTA entry (atomic min), word 1 the earliest warp past its wait for
 * the kernel ahead (atomic min), word 2 the latest warp exit (atomic max).
 * The caller fills words 0-1 with a large value and word 2 with 0 before the
 * calls it wants to see.  Rows: 0 prologue, 1 QKV, 2 attention, 3 attention
 * merge, 4 O projection, 5 gate/up, 6 down, 7 final RMSNorm, 8 LM head,
 * 9 acceptance, 10 sampling, 11 realignment, 12 probabilities, 13 admission,
 * 14 plane join/split, 15 other GEMMs (sdv_linear), 16 + r the deferred
 * fixup of the GEMM in row r.  The library must not be in use on another
 * stream while the table is switched (the address is a device constant). */
sdv_status sdv_trace_enable(void *table);

#ifdef __cplusplus
}
#endif
#endif /* SDV_H */
