// Internal host-side interfaces between the C-ABI glue and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/sdv.h"

namespace sdv {

// ---------------------------------------------------------------------------
// weight-streaming GEMM  y[r, n] = sum_k x[r, k] * W[n, k]
// ---------------------------------------------------------------------------

enum Epi : int {
  EPI_F32 = 0,     // y fp32, no rounding
  EPI_RESID = 1,   // out bf16 = round(acc + resid)
  EPI_SWIGLU = 2,  // tile = 64 gate rows + 64 up rows of the same features: out = round(silu(g) * u)
  EPI_QKV = 3,     // RoPE on q/k heads, q -> q buffer, k/v -> KV pages at (seq, pos)
  EPI_LMHEAD = 4   // logits fp32 + per (vocab tile, row) max and sum of exp
};

struct EpiParams {
  float* out_f32 = nullptr;  // output [R, ld_f32] (QKV: q [R, n_q * head_dim])
  long long ld_f32 = 0;
  __nv_bfloat16* out_bf16 = nullptr;  // SWIGLU: hi plane [R, ld_bf16]; lo plane out_lo_off further
  long long out_lo_off = 0;
  int ld_bf16 = 0;
  const float* resid_f32 = nullptr;  // RESID: residual [R, ld_f32]
  // RESID feeding an RMSNorm: also the next GEMM's input x * gain as bf16 hi + lo
  // planes and per-32-column partial sums of x^2, [N / 32, sq_ld]
  const __nv_bfloat16* norm_gain = nullptr;
  __nv_bfloat16* norm_out = nullptr;
  long long norm_lo_off = 0;
  float* sq_out = nullptr;
  int sq_ld = 0;
  // SWIGLU after such a norm: each row scaled by 1 / sqrt(sum(partials) * sq_inv_n + sq_eps)
  const float* sq_in = nullptr;
  int sq_parts = 0;
  float sq_inv_n = 0.f, sq_eps = 0.f;
  // tcgen05 bf16 GEMM: each row's 1 / rms as the main kernel reduced it, [R],
  // written there and read by its fixup kernel (null: the fixup reduces them)
  float* rscale = nullptr;
  // QKV
  __nv_bfloat16* kv_pool = nullptr;
  const int* page_table = nullptr;
  int max_pages = 0;
  const int* row_seq = nullptr;
  const int* row_pos = nullptr;
  const float* rope_cs = nullptr;  // [R, head_dim/2, 2] (cos, sin)
  const long long* kv_row_off = nullptr;  // [R] element offset of (page, slot) of each row's K/V
  int n_q = 0, n_kv = 0, head_dim = 0, page = 0;
  // LMHEAD
  float2* stats = nullptr;  // [m_tiles, stats_ld]
  int* argmax = nullptr;    // [m_tiles, stats_ld] or null: smallest column of each tile's row maximum
  int stats_ld = 0;
};

struct GemmParams {
  int N = 0;        // output features (SWIGLU: ffn features)
  int K = 0;
  int R = 0;        // activation rows
  int m_tiles = 0;  // weight tiles (128 rows; SWIGLU: 64 features)
  int n_tiles = 0;  // activation-row tiles
  int kb = 0;       // k-blocks of 64 per tile
  int x_lo_row = 0; // two-plane activations: row of the lo plane in the activation map
  int int4 = 0;     // weights are int4 group-32
  float* partials = nullptr;  // stream-K partial tiles [2 * grid, 128 * NT]
  int* counters = nullptr;    // per-tile arrival counters, zero between launches
  // tcgen05 kernels: leave tiles cut between CTAs as stored parts for the
  // fixup kernel (one block per cut tile and 16-row chunk) instead of having
  // the last CTA to arrive sum them
  int defer_fixup = 0;
  // tcgen05 kernels: activation rows per tile, group size (the cs CTAs of a
  // group share each weight tile, CTA r of the group taking activation tile
  // tg * cs + r of tile group tg), tile groups (n_tiles = n_groups * cs when
  // cs > 1), the activation map's box height and the pipeline depth
  int nt = 0, cs = 1, n_groups = 0, x_box = 0, stages = 0;
  int multicast = 0;  // the cluster's CTAs share weight tiles by TMA multicast (else a group reads them via L2)
  // tcgen05 kernels: CTA pairs (cta_group::2) -- a unit is 256 weight rows,
  // 128 in each CTA, against the pair's nt activation rows, half loaded by each
  int pair = 0;
  int* status = nullptr;
  EpiParams epi;
};

// Choose the activation tile for R rows (16, 32 or 64).
int gemm_tile_rows(int R);
// Launch the weight-streaming GEMM. a0/a1: weight maps for the two 64-row
// halves of a 128-row tile (same map for plain GEMMs); x: bf16 activation map
// with box (64, nt); xp = 1 (one plane) or 2 (hi plane at row 0, lo plane at
// row p.x_lo_row).
cudaError_t launch_gemm(int epi, int nt, int xp, const CUtensorMap* a0, const CUtensorMap* a1,
                        const CUtensorMap* x, const GemmParams& p, int grid, cudaStream_t stream);
// out[i] = hi[i] + hi[i + lo_off] for i < n (fp32 view of a two-plane activation).
cudaError_t launch_join_planes(const __nv_bfloat16* hi, long long lo_off, float* out, long long n,
                               cudaStream_t stream);
// The same GEMM over int4 group-32 weights (code maps q0, q1; scale maps s0,
// s1; kb counts 256-k blocks; nt in {8, 16, 32}).
int gemm_q4_tile_rows(int R);
cudaError_t launch_gemm_q4(int epi, int nt, int xp, const CUtensorMap* q0, const CUtensorMap* q1,
                           const CUtensorMap* s0, const CUtensorMap* s1, const CUtensorMap* x, const GemmParams& p,
                           int grid, cudaStream_t stream);
// The same GEMM on tcgen05 / TMEM (nt in {16, 32, 64, 128, 256}).
int gemm_tc_q4_tile_rows(int R);
// int4 group-32 weights on tcgen05 (activations always as bf16 hi + lo planes)
cudaError_t launch_gemm_tc_q4(int epi, int nt, const CUtensorMap* q0, const CUtensorMap* q1, const CUtensorMap* s0,
                              const CUtensorMap* s1, const CUtensorMap* x, const GemmParams& p, int grid,
                              cudaStream_t stream);
int gemm_tc_tile_rows(int R);
// The deferred fixup of a tcgen05 GEMM launched with p.defer_fixup over
// `grid` CTAs: every tile cut between CTAs, summed in CTA order, then the
// GEMM's fused epilogue, in parallel over (cut tile, 16-row chunk).
cudaError_t launch_gemm_tc_fixup(int epi, int nt, const GemmParams& p, int grid, cudaStream_t stream);

#ifdef SDV_TRACE
// Set the timeline table of each translation unit's kernels (SDV_TRACE_UNIT).
cudaError_t trace_set_attention(unsigned long long* table);
cudaError_t trace_set_attention_tc(unsigned long long* table);
cudaError_t trace_set_gemm(unsigned long long* table);
cudaError_t trace_set_gemm_q4(unsigned long long* table);
cudaError_t trace_set_gemm_tc(unsigned long long* table);
cudaError_t trace_set_gemm_tc_q4(unsigned long long* table);
cudaError_t trace_set_step_kernels(unsigned long long* table);
#endif
// Activation tensor maps, one per TMA box height: the powers of two 8..256
// (indices 0..5, the mma.sync and int4 kernels' tile heights) and the other
// multiples of 16 up to 256, so that a tcgen05 CTA loads its activation rows
// of a stage with one copy per plane.
constexpr int kXMaps = 17;
constexpr int kXBoxes[kXMaps] = {8, 16, 32, 64, 128, 256, 48, 80, 96, 112, 144, 160, 176, 192, 208, 224, 240};
inline int x_map_index(int box) {
  for (int i = 0; i < kXMaps; ++i)
    if (kXBoxes[i] == box) return i;
  return -1;
}
// bf16 weights on tcgen05: picks the activation tile height and the size of
// the CTA groups that share each weight tile for p.R rows (measured choices,
// see gemm_tc.cu), then launches the GEMM over the SMs and, for tiles cut
// between CTAs, the fixup.  xmaps: kXMaps activation maps (box heights kXBoxes).
cudaError_t launch_gemm_tc(int epi, int xp, const CUtensorMap* a0, const CUtensorMap* a1, const CUtensorMap* xmaps,
                           GemmParams p, int sms, cudaStream_t stream);
// Split fp32 x [n] into bf16 hi (at out) and lo (at out + lo_off) planes.
cudaError_t launch_split_planes(const float* x, __nv_bfloat16* out, long long lo_off, long long n,
                                cudaStream_t stream);

// ---------------------------------------------------------------------------
// attention over the paged cache
// ---------------------------------------------------------------------------

struct AttnParams {
  const float* q = nullptr;           // [R, n_q, D], rotated
  __nv_bfloat16* out = nullptr;       // hi plane [R, n_q * D]
  long long out_lo_off = 0;           // lo plane offset (elements)
  const int* seq_lens = nullptr;
  const int* draft_lens = nullptr;
  const int* row_off = nullptr;   // [B+1]
  const int* page_table = nullptr;
  int max_pages = 0;
  const int* item_off = nullptr;  // [B+1] first work item of each slot
  const int* chunks = nullptr;    // [B] key chunks per (slot, kv head)
  const int* sched = nullptr;     // [0] chunk pages, [1] total items, [2] 1 if any slot's keys are split
  const int4* items = nullptr;    // [items, 2]: (slot, kv head, first page, end page), (L, gamma, row 0, chunks)
  float* part_o = nullptr;        // [items, QMAX, D]
  float2* part_ml = nullptr;      // [items, QMAX]
  const unsigned long long* row_anc = nullptr;  // [R] token trees: ancestor sets (null: block-causal chains)
  int* status = nullptr;
  int B = 0, n_q = 0, n_kv = 0, page = 0;
  // query vectors per work item (0: all of a (slot, kv head) in one item);
  // the items of a (slot, kv head, chunk) then take vectors [h * qsplit, ...)
  int qsplit = 0;
};
constexpr int kAttnQMax = 48;   // query vectors per work item of the mma.sync kernel (and partial slot)
constexpr int kAttnQVecs = 64;  // query vectors per (slot, kv head), (gamma+1) * group, with items split

// The tcgen05 attention kernel (head_dim 128, nq = 16 or 32 query vectors per
// item); split sequences still need launch_attention_merge afterwards.
cudaError_t launch_attention_tc(int nq, const CUtensorMap* kv_map, const AttnParams& p, int grid, cudaStream_t stream);
cudaError_t launch_attention_merge(int head_dim, const AttnParams& p, int R, cudaStream_t stream, const int* row_seq);
// Attention kernel plus the merge of split sequences (row_seq [R] maps rows to slots).
cudaError_t launch_attention_impl(int head_dim, const CUtensorMap* kv_map, const AttnParams& p, int grid, int R,
                                  cudaStream_t stream, const int* row_seq);
size_t attention_smem_bytes(int head_dim);

// ---------------------------------------------------------------------------
// small kernels of the step
// ---------------------------------------------------------------------------

struct StepTables {
  int* row_off = nullptr;    // [B+1]
  int* draft_off = nullptr;  // [B+1]
  int* row_seq = nullptr;    // [R]
  int* row_pos = nullptr;    // [R]
  int* chunks = nullptr;     // [B]
  int* item_off = nullptr;   // [B+1]
  int* sched = nullptr;      // [4]
  int4* items = nullptr;     // [items, 2] attention work items (null: not built)
  float* rope_cs = nullptr;  // [R, D/2, 2]
  long long* kv_row_off = nullptr;  // [R]
  unsigned long long* row_anc = nullptr;  // [R] token trees: bit j = node j is the row's ancestor or itself
};

struct PrologueParams {
  StepTables t;
  const int* seq_lens = nullptr;
  const int* draft_lens = nullptr;
  const int* tokens = nullptr;
  const int* page_table = nullptr;
  const int* num_pages = nullptr;
  const int* tree_parents = nullptr;  // [R] token trees (null: chains)
  int* status = nullptr;
  int B = 0, R = 0, G = 0, gamma_max = 0, vocab = 0, page = 0, max_pages = 0, pool_pages = 0;
  int n_kv = 0, head_dim = 0, target_items = 0;
  float rope_theta = 0.f;
  int check_tokens = 1;
  // attention work items: query vectors per item (0: no split) and query heads;
  // the smallest chunk of pages an item takes (a multiple of 8)
  int qsplit = 0, n_q = 0, min_chunk = 8;
  // test hook (0 = off): block 0 waits this long on a barrier nothing arrives
  // at, through the bounded wait the pipelined kernels use, and records
  // SDV_ERR_TIMEOUT when it gives up
  unsigned long long stall_ns = 0;
  // embedding + attention pre-norm of every row (verify step only; emb = nullptr skips)
  const __nv_bfloat16* emb = nullptr;
  const __nv_bfloat16* gain = nullptr;
  float* x0 = nullptr;
  __nv_bfloat16* h = nullptr;  // hi plane [R, H]
  long long h_lo_off = 0;      // lo plane offset (elements)
  const double* inv_freq = nullptr;  // [head_dim/2] theta^(-2j/head_dim)
  int H = 0;
  float eps = 0.f;
};
// Validation, row tables and attention schedule (block 0), and with emb set the
// embedding + RMSNorm + rotary table + KV destination of each row (one block per row).
cudaError_t launch_prologue(const PrologueParams& p, cudaStream_t stream);

// h = RMSNorm(x) * gain as bf16 hi + lo planes (lo_off elements apart), or
// rounded to one bf16 plane (lo_off == 0).
cudaError_t launch_rmsnorm(const float* x, const __nv_bfloat16* gain, __nv_bfloat16* h, long long lo_off, int R,
                           int H, float eps, const int* status, cudaStream_t stream);

struct AcceptParams {
  const float* z = nullptr;        // logits [R, V] (from_logits)
  const float* probs = nullptr;    // [R, V] (given probabilities)
  const float* draft_probs = nullptr;
  const float* uniforms = nullptr;
  const int* tokens = nullptr;
  const int* draft_lens = nullptr;
  const int* row_off = nullptr;
  const int* draft_off = nullptr;
  const float2* tile_stats = nullptr;  // [m_tiles, stats_ld] LM head's per-tile (max, sum) (from_logits)
  int m_tiles = 0, stats_ld = 0;
  float2* row_stats = nullptr;         // [R] (max, sum) of each row's logits (from_logits)
  const int* tile_argmax = nullptr;    // [m_tiles, stats_ld] per-tile argmax (from_logits, greedy)
  int greedy = 0;                      // greedy verification: argmax tests, argmax final token
  const int* tree_parents = nullptr;   // [R] token trees (greedy only; null: chains)
  int* tree_path = nullptr;            // [G] accepted path of each slot, from its draft offset
  int* chunk_count = nullptr;      // [B] sampling chunks finished per slot (zero between calls)
  unsigned long long* chunk_sums = nullptr;  // [B, 2, chunk_ld]
  int chunk_ld = 0;
  int* accepted = nullptr;
  int* final_tokens = nullptr;
  int* status = nullptr;
  int B = 0, V = 0, R = 0;
};
// Acceptance (one block per slot: its rows' softmax normalisers, then the
// draft tests) and final-token sampling (one warp per vocab chunk and slot).
constexpr int kSampleChunk = 512;         // vocab entries per sampling chunk
constexpr int kMaxSampleChunks = 2048;    // vocab up to 1M
cudaError_t launch_accept(const AcceptParams& p, bool from_logits, cudaStream_t stream);
int accept_chunks(int V);
cudaError_t launch_probs(const float* z, const float2* row_stats, float* probs, int R, int V, const int* status,
                         cudaStream_t stream);

struct RealignParams {
  const int* seq_lens = nullptr;
  const int* draft_lens = nullptr;
  const int* tokens = nullptr;
  const int* row_off = nullptr;
  const int* accepted = nullptr;
  const int* final_tokens = nullptr;
  int* page_table = nullptr;
  int* num_pages = nullptr;
  int* free_pages = nullptr;
  const int* num_free_in = nullptr;
  int* num_free_out = nullptr;
  const int* gen_counts = nullptr;
  const int* gen_limits = nullptr;
  // token trees: the accepted path of each slot (from its draft offset) and the
  // cache its K/V rows move in (null: chains, nothing moves)
  const int* tree_path = nullptr;
  __nv_bfloat16* kv_pool = nullptr;
  int n_kv = 0, head_dim = 0;
  sdv_result res;
  int B = 0, page = 0, gamma_max = 0, max_pages = 0, pool_pages = 0, vocab = 0;
};
cudaError_t launch_realign(const RealignParams& p, cudaStream_t stream);

struct AdmitParams {
  sdv_admission a;
  int gamma_max = 0, page = 0;
  int* status = nullptr;
};
// Append admitted sequences to a slot table (one block).
cudaError_t launch_admit(const AdmitParams& p, cudaStream_t stream);

// count of kernels launched by this library
void note_launch(int n = 1);

// Launch with programmatic stream serialisation: the kernel may start while
// the previous kernel in the stream finishes; it orders itself with
// griddepcontrol.wait where it reads that kernel's results.
// SDV_NO_PDL=1 in the environment launches without the attribute (A/B timing).
bool pdl_enabled();

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  note_launch();
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

}  // namespace sdv
