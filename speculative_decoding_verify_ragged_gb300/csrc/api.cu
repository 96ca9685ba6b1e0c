// C ABI of the verify step: argument checks, workspace layout, TMA
// descriptors and the order of kernel launches on the caller's stream.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>

#include "internal.h"

namespace sdv {

static std::atomic<unsigned long long> g_launches{0};
static thread_local int g_last_cuda_error = 0;

void note_launch(int n) { g_launches.fetch_add(static_cast<unsigned long long>(n), std::memory_order_relaxed); }

bool pdl_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("SDV_NO_PDL");
    return !(v && v[0] == '1');
  }();
  return on;
}

static sdv_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return SDV_ERR_CUDA;
}

#define SDV_CUDA(x)                              \
  do {                                           \
    cudaError_t e__ = (x);                       \
    if (e__ != cudaSuccess) return cuda_fail(e__); \
  } while (0)

static size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// ---------------------------------------------------------------------------
// workspace layout
// ---------------------------------------------------------------------------

struct Layout {
  size_t row_off, draft_off, row_seq, row_pos, row_anc, tree_path, chunks, item_off, sched, items, rope, kv_row_off,
      inv_freq;
  size_t x0, h, h3, q, attn, x1, x1sq, rscale, act, x2, z, lmstats, lmargmax, rowstats, partials, counters;
  size_t part_o, part_ml, accepted, final_tokens, chunk_count, chunk_sums, total;
  int chunk_ld;
  int lm_tiles, max_tiles, target_items, items_max, grid_gemm;
};

static int num_sms_current() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

static bool config_ok(const sdv_config* c) {
  if (!c) return false;
  if (c->hidden <= 0 || c->n_q <= 0 || c->n_kv <= 0 || c->ffn <= 0 || c->vocab <= 0) return false;
  if (c->head_dim != 64 && c->head_dim != 128) return false;
  if (c->n_q % c->n_kv) return false;
  if (c->page_size != 16) return false;
  // query vectors per (slot, kv head): 48 on the mma.sync attention kernel, 64
  // with head_dim 128 (the tcgen05 kernel splits them over two items)
  if (c->gamma_max < 0 || (c->gamma_max + 1) * (c->n_q / c->n_kv) > (c->head_dim == 128 ? kAttnQVecs : kAttnQMax))
    return false;
  const int kmul = c->weight_format == SDV_WEIGHTS_INT4_G32 ? 256 : 64;
  if (c->weight_format != SDV_WEIGHTS_BF16 && c->weight_format != SDV_WEIGHTS_INT4_G32) return false;
  if (c->hidden % kmul || (c->n_q * c->head_dim) % kmul || c->ffn % kmul) return false;
  if (c->ffn % 64) return false;
  if (c->vocab > kMaxSampleChunks * kSampleChunk) return false;  // sampling chunk table
  if (c->hidden > 8 * 1024) return false;   // embedding row held in registers
  return true;
}

static Layout make_layout(const sdv_config& c, int max_rows, int max_slots, int sms) {
  Layout L{};
  const size_t R = static_cast<size_t>(max_rows), B = static_cast<size_t>(max_slots);
  const size_t H = c.hidden, QD = static_cast<size_t>(c.n_q) * c.head_dim, F = c.ffn, V = c.vocab;
  const size_t NQKV = static_cast<size_t>(c.n_q + 2 * c.n_kv) * c.head_dim;
  L.lm_tiles = static_cast<int>((V + 127) / 128);
  const int rt = static_cast<int>((R + 7) / 8);
  const int tiles_qkv = static_cast<int>((NQKV + 127) / 128);
  const int tiles_o = static_cast<int>((H + 127) / 128);
  const int tiles_gu = static_cast<int>((F + 63) / 64);
  int mt = L.lm_tiles;
  if (tiles_qkv > mt) mt = tiles_qkv;
  if (tiles_o > mt) mt = tiles_o;
  if (tiles_gu > mt) mt = tiles_gu;
  L.max_tiles = mt * rt;
  L.grid_gemm = sms;
  // attention items: about two per SM where the keys allow (measured against
  // one and four per SM, 9B-class layer, ctx 2048: B = 32 attention 81 -> 74 us,
  // B = 16 56 -> 50 us, B = 64 and B <= 8 within 2 us)
  L.target_items = 2 * sms;
  // items split by query vectors (more than 32 per slot and kv head) double
  const int parts = (c.gamma_max + 1) * (c.n_q / c.n_kv) > 32 ? 2 : 1;
  L.items_max = parts * (L.target_items + static_cast<int>(B) * c.n_kv) + 8;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += up256(bytes);
    return at;
  };
  L.row_off = take((B + 1) * 4);
  L.draft_off = take((B + 1) * 4);
  L.row_seq = take(R * 4);
  L.row_pos = take(R * 4);
  L.row_anc = take(R * 8);
  L.tree_path = take(R * 4);
  L.chunks = take(B * 4);
  L.item_off = take((B + 1) * 4);
  L.sched = take(64);
  L.items = take(static_cast<size_t>(L.items_max) * 32);
  L.rope = take(R * (c.head_dim / 2) * 2 * 4);
  L.kv_row_off = take(R * 8);
  L.inv_freq = take(static_cast<size_t>(c.head_dim / 2) * 8);
  // the residual stream is fp32; GEMM inputs are bf16 hi + lo planes [2, R, K];
  // the LM head reads one bf16 plane of the final norm
  L.x0 = take(R * H * 4);
  L.h = take(2 * R * H * 2);
  L.h3 = take(R * H * 2);
  L.q = take(R * QD * 4);
  L.attn = take(2 * R * QD * 2);
  L.x1 = take(R * H * 4);
  L.x1sq = take(static_cast<size_t>(H / 32) * R * 4);  // per-32-column partial sums of x1^2
  L.rscale = take(R * 4);                                // the FFN pre-norm's 1 / rms per row
  L.act = take(2 * R * (F > QD ? (F > H ? F : H) : (QD > H ? QD : H)) * 2);
  L.x2 = take(R * H * 4);
  L.z = take(R * V * 4);
  L.lmstats = take(static_cast<size_t>(L.lm_tiles) * R * 8);
  L.lmargmax = take(static_cast<size_t>(L.lm_tiles) * R * 4);
  L.rowstats = take(R * 8);
  L.partials = take(static_cast<size_t>(2) * sms * 128 * 256 * 4);  // two pieces per CTA, tiles up to 256 rows
  L.counters = take(static_cast<size_t>(L.max_tiles) * 4);
  L.part_o = take(static_cast<size_t>(L.items_max) * kAttnQMax * c.head_dim * 4);
  L.part_ml = take(static_cast<size_t>(L.items_max) * kAttnQMax * 8);
  L.accepted = take(B * 4);
  L.final_tokens = take(B * 4);
  L.chunk_ld = accept_chunks(c.vocab);
  L.chunk_count = take(B * 4);
  L.chunk_sums = take(B * 2 * static_cast<size_t>(L.chunk_ld) * 8);
  L.total = o;
  return L;
}

// ---------------------------------------------------------------------------
// TMA descriptors
// ---------------------------------------------------------------------------

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D bf16 matrix [rows, cols] (cols contiguous), box = (64 cols, box_rows), 128-byte swizzle.
static bool encode_bf16_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D byte matrix [rows, cols] (int4 codes, two per byte), box = (128 bytes, 64 rows), 128-byte swizzle.
static bool encode_u8_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {128, 64};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D fp16 matrix [rows, cols] (int4 group scales), box = (8 cols, 64 rows), no swizzle.
static bool encode_f16_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {8, 64};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// KV pool [pages, n_kv, 2, page, D] as a 5-D tensor; box = 64 of D x 16 slots.
static bool encode_kv(CUtensorMap* m, const void* base, const sdv_config& c, int pool_pages) {
  auto fn = encode_fn();
  if (!fn) return false;
  const uint64_t D = c.head_dim, P = c.page_size;
  cuuint64_t dims[5] = {D, P, 2, static_cast<cuuint64_t>(c.n_kv), static_cast<cuuint64_t>(pool_pages)};
  cuuint64_t strides[4] = {D * 2, P * D * 2, 2 * P * D * 2, static_cast<cuuint64_t>(c.n_kv) * 2 * P * D * 2};
  cuuint32_t box[5] = {64, 16, 1, 1, 1};
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int nt_index(int nt) {
  switch (nt) {
    case 8: return 0;
    case 16: return 1;
    case 32: return 2;
    case 64: return 3;
    case 128: return 4;
    default: return 5;
  }
}

}  // namespace sdv

using namespace sdv;

struct sdv_ctx {
  sdv_config cfg;
  sdv_weights w;
  int max_rows, max_slots, sms;
  uint8_t* ws;
  Layout L;
  // layer weights: bf16 maps, or for int4 the code maps (tm_*) and the scale maps (ts_*)
  CUtensorMap tm_qkv, tm_o, tm_gate, tm_up, tm_down, tm_lm;
  CUtensorMap ts_qkv, ts_o, ts_gate, ts_up, ts_down;
  bool int4;
  CUtensorMap tm_h[kXMaps], tm_attn[kXMaps], tm_act[kXMaps], tm_h3[kXMaps];  // activation boxes kXBoxes
  int gemm_path;
  int attn_path;
  int sampling;
  unsigned long long stall_ns;  // test hook, 0 = off
  cudaEvent_t phase_ev[SDV_PHASES + 1];
  bool timing;
};

template <typename T>
static T* ws_ptr(sdv_ctx* c, size_t off) {
  return reinterpret_cast<T*>(c->ws + off);
}

extern "C" {

size_t sdv_workspace_size(const sdv_config* cfg, int max_rows, int max_slots) {
  if (!config_ok(cfg) || max_rows <= 0 || max_slots <= 0 || max_slots > 1024) return 0;
  const int sms = num_sms_current();
  if (sms <= 0) return 0;
  return make_layout(*cfg, max_rows, max_slots, sms).total;
}

sdv_status sdv_create(const sdv_config* cfg, const sdv_weights* w, void* workspace, size_t workspace_bytes,
                      int max_rows, int max_slots, sdv_ctx** out) {
  if (!out || !w || !workspace) return SDV_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg) return SDV_ERR_INVALID_ARG;
  if (cfg->head_dim != 64 && cfg->head_dim != 128) return SDV_ERR_UNSUPPORTED;
  if (!config_ok(cfg) || max_rows <= 0 || max_slots <= 0 || max_slots > 1024) return SDV_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return SDV_ERR_INVALID_ARG;
  if (!w->emb || !w->w_qkv || !w->w_o || !w->w_gate || !w->w_up || !w->w_down || !w->w_lm || !w->g_attn ||
      !w->g_ffn || !w->g_final)
    return SDV_ERR_INVALID_ARG;
  const bool int4 = cfg->weight_format == SDV_WEIGHTS_INT4_G32;
  if (int4 && (!w->s_qkv || !w->s_o || !w->s_gate || !w->s_up || !w->s_down)) return SDV_ERR_INVALID_ARG;
  const int sms = num_sms_current();
  if (sms <= 0) return SDV_ERR_CUDA;
  Layout L = make_layout(*cfg, max_rows, max_slots, sms);
  if (workspace_bytes < L.total) return SDV_ERR_CAPACITY;
  sdv_ctx* c = new (std::nothrow) sdv_ctx();
  if (!c) return SDV_ERR_INTERNAL;
  c->cfg = *cfg;
  c->w = *w;
  c->max_rows = max_rows;
  c->max_slots = max_slots;
  c->sms = sms;
  c->ws = static_cast<uint8_t*>(workspace);
  c->L = L;
  c->timing = false;
  c->gemm_path = SDV_GEMM_AUTO;
  c->attn_path = SDV_GEMM_AUTO;
  c->sampling = SDV_SAMPLING_STOCHASTIC;
  c->stall_ns = 0;
  const uint64_t H = cfg->hidden, QD = static_cast<uint64_t>(cfg->n_q) * cfg->head_dim, F = cfg->ffn,
                 V = cfg->vocab;
  const uint64_t NQKV = static_cast<uint64_t>(cfg->n_q + 2 * cfg->n_kv) * cfg->head_dim;
  c->int4 = int4;
  bool ok = encode_bf16_2d(&c->tm_lm, w->w_lm, V, H, 64);
  if (int4) {
    ok = ok && encode_u8_2d(&c->tm_qkv, w->w_qkv, NQKV, H / 2) && encode_f16_2d(&c->ts_qkv, w->s_qkv, NQKV, H / 32) &&
         encode_u8_2d(&c->tm_o, w->w_o, H, QD / 2) && encode_f16_2d(&c->ts_o, w->s_o, H, QD / 32) &&
         encode_u8_2d(&c->tm_gate, w->w_gate, F, H / 2) && encode_f16_2d(&c->ts_gate, w->s_gate, F, H / 32) &&
         encode_u8_2d(&c->tm_up, w->w_up, F, H / 2) && encode_f16_2d(&c->ts_up, w->s_up, F, H / 32) &&
         encode_u8_2d(&c->tm_down, w->w_down, H, F / 2) && encode_f16_2d(&c->ts_down, w->s_down, H, F / 32);
  } else {
    ok = ok && encode_bf16_2d(&c->tm_qkv, w->w_qkv, NQKV, H, 64) && encode_bf16_2d(&c->tm_o, w->w_o, H, QD, 64) &&
         encode_bf16_2d(&c->tm_gate, w->w_gate, F, H, 64) && encode_bf16_2d(&c->tm_up, w->w_up, F, H, 64) &&
         encode_bf16_2d(&c->tm_down, w->w_down, H, F, 64);
  }
  for (int i = 0; i < kXMaps && ok; ++i) {
    ok = encode_bf16_2d(&c->tm_h[i], c->ws + L.h, 2ull * max_rows, H, kXBoxes[i]) &&
         encode_bf16_2d(&c->tm_attn[i], c->ws + L.attn, 2ull * max_rows, QD, kXBoxes[i]) &&
         encode_bf16_2d(&c->tm_act[i], c->ws + L.act, 2ull * max_rows, F, kXBoxes[i]) &&
         encode_bf16_2d(&c->tm_h3[i], c->ws + L.h3, max_rows, H, kXBoxes[i]);
  }
  if (!ok) {
    delete c;
    return SDV_ERR_CUDA;
  }
  // arrival counters start at zero; every kernel that uses one resets it
  cudaError_t e = cudaMemset(c->ws + L.counters, 0, static_cast<size_t>(L.max_tiles) * 4);
  if (e == cudaSuccess) e = cudaMemset(c->ws + L.chunk_count, 0, static_cast<size_t>(max_slots) * 4);
  if (e == cudaSuccess) {
    // rotary inverse frequencies theta^(-2j/d), in double, computed once
    double inv[128];
    const int half = cfg->head_dim / 2;
    for (int j = 0; j < half; ++j) inv[j] = std::pow(static_cast<double>(cfg->rope_theta), -2.0 * j / cfg->head_dim);
    e = cudaMemcpy(c->ws + L.inv_freq, inv, sizeof(double) * half, cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    delete c;
    return cuda_fail(e);
  }
  *out = c;
  return SDV_OK;
}

void sdv_destroy(sdv_ctx* ctx) { delete ctx; }

sdv_status sdv_set_gemm_path(sdv_ctx* ctx, int path) {
  if (!ctx || path < SDV_GEMM_AUTO || path > SDV_GEMM_TCGEN05) return SDV_ERR_INVALID_ARG;
  ctx->gemm_path = path;
  return SDV_OK;
}

sdv_status sdv_set_sampling(sdv_ctx* ctx, int mode) {
  if (!ctx || (mode != SDV_SAMPLING_STOCHASTIC && mode != SDV_SAMPLING_GREEDY)) return SDV_ERR_INVALID_ARG;
  ctx->sampling = mode;
  return SDV_OK;
}

sdv_status sdv_set_stall_test(sdv_ctx* ctx, unsigned long long stall_ns) {
  if (!ctx) return SDV_ERR_INVALID_ARG;
  ctx->stall_ns = stall_ns;
  return SDV_OK;
}

sdv_status sdv_set_attention_path(sdv_ctx* ctx, int path) {
  if (!ctx || path < SDV_GEMM_AUTO || path > SDV_GEMM_TCGEN05) return SDV_ERR_INVALID_ARG;
  ctx->attn_path = path;
  return SDV_OK;
}

sdv_status sdv_set_phase_events(sdv_ctx* ctx, void* const* events, int n) {
  if (!ctx) return SDV_ERR_INVALID_ARG;
  if (!events || n == 0) {
    ctx->timing = false;
    return SDV_OK;
  }
  if (n != SDV_PHASES + 1) return SDV_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) ctx->phase_ev[i] = static_cast<cudaEvent_t>(events[i]);
  ctx->timing = true;
  return SDV_OK;
}

int sdv_last_cuda_error(void) { return g_last_cuda_error; }

unsigned long long sdv_kernel_launches(void) { return g_launches.load(); }

sdv_status sdv_trace_enable(void* table) {
#ifdef SDV_TRACE
  auto* t = static_cast<unsigned long long*>(table);
  cudaError_t (*const set[])(unsigned long long*) = {trace_set_attention, trace_set_attention_tc, trace_set_gemm,
                                                     trace_set_gemm_q4,   trace_set_gemm_tc,      trace_set_gemm_tc_q4,
                                                     trace_set_step_kernels};
  for (auto f : set) SDV_CUDA(f(t));
  return SDV_OK;
#else
  (void)table;
  return SDV_ERR_UNSUPPORTED;
#endif
}

sdv_status sdv_read_status(const int* status, int* host_status, void* stream) {
  if (!status || !host_status) return SDV_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  SDV_CUDA(cudaMemcpyAsync(host_status, status, sizeof(int), cudaMemcpyDeviceToHost, s));
  SDV_CUDA(cudaStreamSynchronize(s));
  return SDV_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// launch helpers
// ---------------------------------------------------------------------------

static bool batch_ok(const sdv_ctx* c, const sdv_batch* b, bool need_forward) {
  if (!b) return false;
  if (b->B <= 0 || b->B > c->max_slots || b->R < b->B || b->R > c->max_rows || b->G != b->R - b->B) return false;
  if (!b->seq_lens || !b->draft_lens || !b->page_table || !b->num_pages) return false;
  if (b->max_pages_per_seq <= 0 || b->num_pool_pages <= 0) return false;
  if (need_forward && (!b->tokens || !b->kv_pool)) return false;
  return true;
}

static PrologueParams prologue_params(sdv_ctx* c, const sdv_batch* b, int* status, bool check_tokens) {
  PrologueParams p;
  p.t.row_off = ws_ptr<int>(c, c->L.row_off);
  p.t.draft_off = ws_ptr<int>(c, c->L.draft_off);
  p.t.row_seq = ws_ptr<int>(c, c->L.row_seq);
  p.t.row_pos = ws_ptr<int>(c, c->L.row_pos);
  p.t.chunks = ws_ptr<int>(c, c->L.chunks);
  p.t.item_off = ws_ptr<int>(c, c->L.item_off);
  p.t.sched = ws_ptr<int>(c, c->L.sched);
  p.t.items = ws_ptr<int4>(c, c->L.items);
  p.t.rope_cs = ws_ptr<float>(c, c->L.rope);
  p.t.kv_row_off = ws_ptr<long long>(c, c->L.kv_row_off);
  p.t.row_anc = ws_ptr<unsigned long long>(c, c->L.row_anc);
  p.tree_parents = b->tree_parents;
  p.seq_lens = b->seq_lens;
  p.draft_lens = b->draft_lens;
  p.tokens = b->tokens;
  p.page_table = b->page_table;
  p.num_pages = b->num_pages;
  p.status = status;
  p.B = b->B;
  p.R = b->R;
  p.G = b->G;
  p.gamma_max = c->cfg.gamma_max;
  p.vocab = c->cfg.vocab;
  p.page = c->cfg.page_size;
  p.max_pages = b->max_pages_per_seq;
  p.pool_pages = b->num_pool_pages;
  p.n_kv = c->cfg.n_kv;
  p.head_dim = c->cfg.head_dim;
  p.target_items = c->L.target_items;
  p.rope_theta = c->cfg.rope_theta;
  p.check_tokens = check_tokens && b->tokens ? 1 : 0;
  p.stall_ns = c->stall_ns;
  p.n_q = c->cfg.n_q;
  p.qsplit = 0;
  return p;
}

static GemmParams gemm_params(sdv_ctx* c, int N, int K, int R, int m_tiles, int* status) {
  GemmParams g;
  g.N = N;
  g.K = K;
  g.R = R;
  g.m_tiles = m_tiles;
  g.kb = K / 64;
  g.partials = ws_ptr<float>(c, c->L.partials);
  g.counters = ws_ptr<int>(c, c->L.counters);
  g.status = status;
  return g;
}

// The scale map of an int4 projection, or null for bf16 weights.
static const CUtensorMap* q4(const sdv_ctx* c, const CUtensorMap& scales) { return c->int4 ? &scales : nullptr; }

// Rows at and above which the tcgen05 kernel takes the context's GEMMs in
// SDV_GEMM_AUTO mode (below it the mma.sync kernel's 8-row tiles waste less).
constexpr int kTcRows = 17;

// Activation tile heights at and above which the tcgen05 GEMMs leave their
// cut tiles to the parallel fixup kernel (one 16-row chunk per block) rather
// than to the last CTA to arrive, which would walk every chunk of the tile.
constexpr int kDeferFixupRows = 32;

// Slots at and above which auto mode runs attention on tcgen05.
constexpr int kTcAttnSlots = 4;

static bool use_tc(const sdv_ctx* c, int R) {
  return c->gemm_path == SDV_GEMM_TCGEN05 || (c->gemm_path == SDV_GEMM_AUTO && R >= kTcRows);
}

// Run one GEMM: pick the kernel and the activation tile height, then launch
// over min(SMs, units) CTAs (tcgen05 bf16: clusters of CTAs, see gemm_tc.cu).  xmaps: the activation map for each tile height;
// s0, s1: the scale maps of int4 weights (a0, a1 are then code maps).
static cudaError_t run_gemm(sdv_ctx* c, int epi, int xp, const CUtensorMap* a0, const CUtensorMap* a1,
                            const CUtensorMap* xmaps, GemmParams g, cudaStream_t s,
                            const CUtensorMap* s0 = nullptr, const CUtensorMap* s1 = nullptr) {
  if (s0) {
    const bool tcq = use_tc(c, g.R) && xp == 2;
    const int nt = tcq ? gemm_tc_q4_tile_rows(g.R) : gemm_q4_tile_rows(g.R);
    g.kb = g.K / 256;
    g.int4 = 1;
    g.n_tiles = (g.R + nt - 1) / nt;
    const long long units = (long long)g.m_tiles * g.n_tiles * g.kb;
    const int grid = static_cast<int>(units < c->L.grid_gemm ? units : c->L.grid_gemm);
    if (!tcq) return launch_gemm_q4(epi, nt, xp, a0, a1, s0, s1, &xmaps[nt_index(nt)], g, grid, s);
    g.defer_fixup = nt >= kDeferFixupRows ? 1 : 0;
    cudaError_t e = launch_gemm_tc_q4(epi, nt, a0, a1, s0, s1, &xmaps[nt_index(nt)], g, grid, s);
    if (e == cudaSuccess && g.defer_fixup) e = launch_gemm_tc_fixup(epi, nt, g, grid, s);
    return e;
  }
  // bf16 weights on tcgen05: the kernel's own launcher picks the tile height
  // and the cluster size that shares each weight tile
  if (use_tc(c, g.R)) return launch_gemm_tc(epi, xp, a0, a1, xmaps, g, c->L.grid_gemm, s);
  const int nt = gemm_tile_rows(g.R);
  g.n_tiles = (g.R + nt - 1) / nt;
  const long long units = (long long)g.m_tiles * g.n_tiles * g.kb;
  const int grid = static_cast<int>(units < c->L.grid_gemm ? units : c->L.grid_gemm);
  return launch_gemm(epi, nt, xp, a0, a1, &xmaps[nt_index(nt)], g, grid, s);
}

// Which attention kernel a batch takes and how its work items split the query
// vectors.  The tcgen05 kernel takes head_dim 128 with up to 64 query vectors
// per (sequence, kv head) -- up to 48 in one item, past 48 in items of 32, two
// items per chunk of pages, adjacent so that the second reads the pages from
// L2 -- and in auto mode from kTcAttnSlots sequences up, or whenever the
// mma.sync kernel's 48 vectors would not hold them.
struct AttnPlan {
  sdv_status st = SDV_OK;
  bool tc = false;
  int qsplit = 0, nq = 0;
};

static AttnPlan attn_plan(const sdv_ctx* c, int B) {
  AttnPlan a;
  const int nqv_max = (c->cfg.gamma_max + 1) * (c->cfg.n_q / c->cfg.n_kv);
  const bool fits = c->cfg.head_dim == 128 && nqv_max <= kAttnQVecs;
  if (c->attn_path == SDV_GEMM_TCGEN05 && !fits) a.st = SDV_ERR_UNSUPPORTED;
  a.tc = fits && (c->attn_path == SDV_GEMM_TCGEN05 ||
                  (c->attn_path == SDV_GEMM_AUTO && (B >= kTcAttnSlots || nqv_max > kAttnQMax)));
  if (!a.tc && nqv_max > kAttnQMax) a.st = SDV_ERR_UNSUPPORTED;
  if (a.tc) {
    a.qsplit = nqv_max > 48 ? 32 : 0;
    a.nq = a.qsplit ? 32 : (nqv_max > 32 ? 48 : (nqv_max > 16 ? 32 : 16));
  }
  return a;
}

// The smallest chunk of pages per attention item.  Items cover about four per
// SM where the batch has the keys for it; below that, the tcgen05 kernel pays
// a whole pipeline fill, epilogue and merge share per item, so its items take
// at least 32 pages (four 128-key blocks), while the mma.sync kernel's small
// batches keep 8-page items (measured, 9B-class layer, ctx 2048: B = 4,
// gamma 7 attention 47 -> 27 us, B = 8 gamma 3 40 -> 35 us on tcgen05; B = 1 on
// mma.sync 20 -> 22 us with 16 pages, 29 with 32).
static int attn_min_chunk(const AttnPlan& plan) { return plan.tc ? 32 : 8; }

static sdv_status run_attention(sdv_ctx* c, const sdv_batch* b, const float* q, __nv_bfloat16* out,
                                long long out_lo_off, int* status, cudaStream_t s) {
  CUtensorMap kv;
  if (!encode_kv(&kv, b->kv_pool, c->cfg, b->num_pool_pages)) return SDV_ERR_CUDA;
  AttnParams a;
  a.q = q;
  a.out = out;
  a.out_lo_off = out_lo_off;
  a.seq_lens = b->seq_lens;
  a.draft_lens = b->draft_lens;
  a.row_off = ws_ptr<int>(c, c->L.row_off);
  a.page_table = b->page_table;
  a.max_pages = b->max_pages_per_seq;
  a.item_off = ws_ptr<int>(c, c->L.item_off);
  a.chunks = ws_ptr<int>(c, c->L.chunks);
  a.sched = ws_ptr<int>(c, c->L.sched);
  a.items = ws_ptr<int4>(c, c->L.items);
  a.part_o = ws_ptr<float>(c, c->L.part_o);
  a.part_ml = ws_ptr<float2>(c, c->L.part_ml);
  a.row_anc = b->tree_parents ? ws_ptr<unsigned long long>(c, c->L.row_anc) : nullptr;
  a.status = status;
  a.B = b->B;
  a.n_q = c->cfg.n_q;
  a.n_kv = c->cfg.n_kv;
  a.page = c->cfg.page_size;
  const int grid = c->sms;  // one CTA per SM (the ring and the combine buffer take most of shared memory)
  // in auto mode a batch of fewer than kTcAttnSlots sequences keeps the
  // mma.sync kernel (too little KV per CTA to hide the tcgen05 pipeline's
  // fill) unless its vectors do not fit it
  const AttnPlan plan = attn_plan(c, b->B);
  if (plan.st != SDV_OK) return plan.st;
  a.qsplit = plan.qsplit;
  if (plan.tc) {
    SDV_CUDA(launch_attention_tc(plan.nq, &kv, a, grid, s));
    SDV_CUDA(launch_attention_merge(c->cfg.head_dim, a, b->R, s, ws_ptr<int>(c, c->L.row_seq)));
    return SDV_OK;
  }
  SDV_CUDA(launch_attention_impl(c->cfg.head_dim, &kv, a, grid, b->R, s, ws_ptr<int>(c, c->L.row_seq)));
  return SDV_OK;
}

static void fill_accept_scratch(sdv_ctx* c, AcceptParams& a) {
  a.chunk_count = ws_ptr<int>(c, c->L.chunk_count);
  a.chunk_sums = ws_ptr<unsigned long long>(c, c->L.chunk_sums);
  a.chunk_ld = c->L.chunk_ld;
}

static RealignParams realign_params(sdv_ctx* c, const sdv_batch* b, const sdv_result* r, const int* accepted,
                                    const int* final_tokens) {
  RealignParams p;
  p.seq_lens = b->seq_lens;
  p.draft_lens = b->draft_lens;
  p.tokens = b->tokens;
  p.row_off = ws_ptr<int>(c, c->L.row_off);
  p.accepted = accepted;
  p.final_tokens = final_tokens;
  p.page_table = b->page_table;
  p.num_pages = b->num_pages;
  p.free_pages = b->free_pages;
  p.num_free_in = b->num_free_in;
  p.num_free_out = b->num_free_out;
  p.gen_counts = b->gen_counts;
  p.gen_limits = b->gen_limits;
  if (b->tree_parents) {
    p.tree_path = ws_ptr<int>(c, c->L.tree_path);
    p.kv_pool = static_cast<__nv_bfloat16*>(b->kv_pool);
    p.n_kv = c->cfg.n_kv;
    p.head_dim = c->cfg.head_dim;
  }
  p.res = *r;
  p.B = b->B;
  p.page = c->cfg.page_size;
  p.gamma_max = c->cfg.gamma_max;
  p.max_pages = b->max_pages_per_seq;
  p.pool_pages = b->num_pool_pages;
  p.vocab = c->cfg.vocab;
  return p;
}

// Token trees are verified greedily and need the cache their path moves in.
static sdv_status tree_check(const sdv_ctx* c, const sdv_batch* b) {
  if (!b->tree_parents) return SDV_OK;
  if (c->sampling != SDV_SAMPLING_GREEDY) return SDV_ERR_UNSUPPORTED;
  if (!b->kv_pool || !b->tokens) return SDV_ERR_INVALID_ARG;
  return SDV_OK;
}

// The accept kernel's tree fields.
static void tree_accept(sdv_ctx* c, const sdv_batch* b, AcceptParams& a) {
  a.tree_parents = b->tree_parents;
  a.tree_path = b->tree_parents ? ws_ptr<int>(c, c->L.tree_path) : nullptr;
}

static bool result_ok(const sdv_batch* b, const sdv_result* r) {
  if (!r || !r->status) return false;
  if (!b->free_pages || !b->num_free_in || !b->num_free_out) return false;
  if ((r->accept_tested == nullptr) != (r->accept_accepted == nullptr)) return false;
  return true;
}

extern "C" {

sdv_status sdv_verify_step(sdv_ctx* c, const sdv_batch* b, sdv_result* r, void* stream) {
  if (!c || !batch_ok(c, b, true) || !result_ok(b, r)) return SDV_ERR_INVALID_ARG;
  const bool greedy = c->sampling == SDV_SAMPLING_GREEDY;
  if (!greedy && (!b->uniforms || (b->G > 0 && !b->draft_probs))) return SDV_ERR_INVALID_ARG;
  if (const sdv_status ts = tree_check(c, b); ts != SDV_OK) return ts;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const sdv_config& cf = c->cfg;
  const int R = b->R, H = cf.hidden, D = cf.head_dim, QD = cf.n_q * D, F = cf.ffn, V = cf.vocab;
  const int NQKV = (cf.n_q + 2 * cf.n_kv) * D;
  int* status = r->status;
  auto f32 = [&](size_t off) { return ws_ptr<float>(c, off); };
  // inside a stream capture the marks become graph nodes that record their
  // timestamps when the graph runs (external event records)
  cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
  if (c->timing && cudaStreamIsCapturing(s, &capture) != cudaSuccess) capture = cudaStreamCaptureStatusNone;
  auto mark = [&](int k) -> cudaError_t {
    if (!c->timing || !c->phase_ev[k]) return cudaSuccess;
    return capture == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(c->phase_ev[k], s, cudaEventRecordExternal)
                                                    : cudaEventRecord(c->phase_ev[k], s);
  };

  const AttnPlan plan = attn_plan(c, b->B);
  if (plan.st != SDV_OK) return plan.st;
  SDV_CUDA(mark(SDV_PHASE_PROLOGUE));
  PrologueParams pp = prologue_params(c, b, status, true);
  pp.qsplit = plan.qsplit;
  pp.min_chunk = attn_min_chunk(plan);
  pp.emb = static_cast<const __nv_bfloat16*>(c->w.emb);
  pp.gain = static_cast<const __nv_bfloat16*>(c->w.g_attn);
  pp.x0 = f32(c->L.x0);
  pp.h = ws_ptr<__nv_bfloat16>(c, c->L.h);
  pp.h_lo_off = (long long)c->max_rows * H;
  pp.H = H;
  pp.eps = cf.rms_eps;
  pp.inv_freq = ws_ptr<double>(c, c->L.inv_freq);
  SDV_CUDA(launch_prologue(pp, s));
  SDV_CUDA(mark(SDV_PHASE_QKV));
  {  // fused QKV + RoPE + KV append
    GemmParams g = gemm_params(c, NQKV, H, R, (NQKV + 127) / 128, status);
    g.epi.out_f32 = f32(c->L.q);
    g.epi.kv_pool = static_cast<__nv_bfloat16*>(b->kv_pool);
    g.epi.page_table = b->page_table;
    g.epi.max_pages = b->max_pages_per_seq;
    g.epi.row_seq = pp.t.row_seq;
    g.epi.row_pos = pp.t.row_pos;
    g.epi.rope_cs = pp.t.rope_cs;
    g.epi.kv_row_off = pp.t.kv_row_off;
    g.epi.n_q = cf.n_q;
    g.epi.n_kv = cf.n_kv;
    g.epi.head_dim = D;
    g.epi.page = cf.page_size;
    g.x_lo_row = c->max_rows;
    SDV_CUDA(run_gemm(c, EPI_QKV, 2, &c->tm_qkv, &c->tm_qkv, c->tm_h, g, s, q4(c, c->ts_qkv), q4(c, c->ts_qkv)));
  }
  SDV_CUDA(mark(SDV_PHASE_ATTN));
  {
    sdv_status st = run_attention(c, b, f32(c->L.q), ws_ptr<__nv_bfloat16>(c, c->L.attn),
                                  (long long)c->max_rows * QD, status, s);
    if (st != SDV_OK) return st;
  }
  SDV_CUDA(mark(SDV_PHASE_O));
  {  // O projection + residual
    GemmParams g = gemm_params(c, H, QD, R, (H + 127) / 128, status);
    g.epi.out_f32 = f32(c->L.x1);
    g.epi.resid_f32 = f32(c->L.x0);
    g.epi.ld_f32 = H;
    // the FFN pre-norm: x1 * g_ffn as the gate/up input, sums of x1^2 for the row scale
    g.epi.norm_gain = static_cast<const __nv_bfloat16*>(c->w.g_ffn);
    g.epi.norm_out = ws_ptr<__nv_bfloat16>(c, c->L.h);
    g.epi.norm_lo_off = (long long)c->max_rows * H;
    g.epi.sq_out = f32(c->L.x1sq);
    g.epi.sq_ld = c->max_rows;
    g.x_lo_row = c->max_rows;
    SDV_CUDA(run_gemm(c, EPI_RESID, 2, &c->tm_o, &c->tm_o, c->tm_attn, g, s, q4(c, c->ts_o), q4(c, c->ts_o)));
  }
  SDV_CUDA(mark(SDV_PHASE_FFN));
  {  // gate/up + RMSNorm row scale + SwiGLU
    GemmParams g = gemm_params(c, F, H, R, (F + 63) / 64, status);
    g.epi.sq_in = f32(c->L.x1sq);
    g.epi.sq_parts = H / 32;
    g.epi.sq_ld = c->max_rows;
    g.epi.sq_inv_n = 1.0f / static_cast<float>(H);
    g.epi.sq_eps = cf.rms_eps;
    g.epi.rscale = cf.weight_format == SDV_WEIGHTS_BF16 ? f32(c->L.rscale) : nullptr;
    g.epi.out_bf16 = ws_ptr<__nv_bfloat16>(c, c->L.act);
    g.epi.out_lo_off = (long long)c->max_rows * F;
    g.epi.ld_bf16 = F;
    g.x_lo_row = c->max_rows;
    SDV_CUDA(run_gemm(c, EPI_SWIGLU, 2, &c->tm_gate, &c->tm_up, c->tm_h, g, s, q4(c, c->ts_gate), q4(c, c->ts_up)));
  }
  {  // down projection + residual
    GemmParams g = gemm_params(c, H, F, R, (H + 127) / 128, status);
    g.epi.out_f32 = f32(c->L.x2);
    g.epi.resid_f32 = f32(c->L.x1);
    g.epi.ld_f32 = H;
    g.x_lo_row = c->max_rows;
    SDV_CUDA(run_gemm(c, EPI_RESID, 2, &c->tm_down, &c->tm_down, c->tm_act, g, s, q4(c, c->ts_down), q4(c, c->ts_down)));
  }
  SDV_CUDA(launch_rmsnorm(f32(c->L.x2), static_cast<const __nv_bfloat16*>(c->w.g_final),
                          ws_ptr<__nv_bfloat16>(c, c->L.h3), 0, R, H, cf.rms_eps, status, s));
  float* z = r->logits ? r->logits : ws_ptr<float>(c, c->L.z);
  SDV_CUDA(mark(SDV_PHASE_LMHEAD));
  {  // LM head + per-tile softmax statistics
    GemmParams g = gemm_params(c, V, H, R, c->L.lm_tiles, status);
    g.epi.out_f32 = z;
    g.epi.ld_f32 = V;
    g.epi.stats = ws_ptr<float2>(c, c->L.lmstats);
    if (c->sampling == SDV_SAMPLING_GREEDY) g.epi.argmax = ws_ptr<int>(c, c->L.lmargmax);
    g.epi.stats_ld = c->max_rows;
    SDV_CUDA(run_gemm(c, EPI_LMHEAD, 1, &c->tm_lm, &c->tm_lm, c->tm_h3, g, s));
  }
  int* accepted = r->accepted ? r->accepted : ws_ptr<int>(c, c->L.accepted);
  int* final_tokens = r->final_tokens ? r->final_tokens : ws_ptr<int>(c, c->L.final_tokens);
  SDV_CUDA(mark(SDV_PHASE_ACCEPT));
  {
    AcceptParams a;
    a.z = z;
    a.tile_stats = ws_ptr<float2>(c, c->L.lmstats);
    a.tile_argmax = ws_ptr<int>(c, c->L.lmargmax);
    a.greedy = c->sampling == SDV_SAMPLING_GREEDY ? 1 : 0;
    a.m_tiles = c->L.lm_tiles;
    a.stats_ld = c->max_rows;
    a.draft_probs = b->draft_probs;
    a.uniforms = b->uniforms;
    a.tokens = b->tokens;
    a.draft_lens = b->draft_lens;
    a.row_off = pp.t.row_off;
    a.draft_off = pp.t.draft_off;
    a.row_stats = ws_ptr<float2>(c, c->L.rowstats);
    tree_accept(c, b, a);
    fill_accept_scratch(c, a);
    a.accepted = accepted;
    a.final_tokens = final_tokens;
    a.status = status;
    a.B = b->B;
    a.V = V;
    a.R = b->R;
    SDV_CUDA(launch_accept(a, true, s));
  }
  if (r->probs) SDV_CUDA(launch_probs(z, ws_ptr<float2>(c, c->L.rowstats), r->probs, R, V, status, s));
  SDV_CUDA(mark(SDV_PHASE_REALIGN));
  RealignParams rp = realign_params(c, b, r, accepted, final_tokens);
  SDV_CUDA(launch_realign(rp, s));
  SDV_CUDA(mark(SDV_PHASES));
  return SDV_OK;
}

sdv_status sdv_accept(sdv_ctx* c, const float* probs, const sdv_batch* b, sdv_result* r, void* stream) {
  if (!c || !probs || !batch_ok(c, b, false) || !result_ok(b, r)) return SDV_ERR_INVALID_ARG;
  if (!b->tokens) return SDV_ERR_INVALID_ARG;
  if (c->sampling != SDV_SAMPLING_GREEDY && (!b->uniforms || (b->G > 0 && !b->draft_probs))) return SDV_ERR_INVALID_ARG;
  if (const sdv_status ts = tree_check(c, b); ts != SDV_OK) return ts;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PrologueParams pp = prologue_params(c, b, r->status, true);
  SDV_CUDA(launch_prologue(pp, s));
  int* accepted = r->accepted ? r->accepted : ws_ptr<int>(c, c->L.accepted);
  int* final_tokens = r->final_tokens ? r->final_tokens : ws_ptr<int>(c, c->L.final_tokens);
  AcceptParams a;
  a.probs = probs;
  a.greedy = c->sampling == SDV_SAMPLING_GREEDY ? 1 : 0;
  a.draft_probs = b->draft_probs;
  a.uniforms = b->uniforms;
  a.tokens = b->tokens;
  a.draft_lens = b->draft_lens;
  a.row_off = pp.t.row_off;
  a.draft_off = pp.t.draft_off;
  tree_accept(c, b, a);
  fill_accept_scratch(c, a);
  a.accepted = accepted;
  a.final_tokens = final_tokens;
  a.status = r->status;
  a.B = b->B;
  a.V = c->cfg.vocab;
  a.R = b->R;
  SDV_CUDA(launch_accept(a, false, s));
  RealignParams rp = realign_params(c, b, r, accepted, final_tokens);
  SDV_CUDA(launch_realign(rp, s));
  return SDV_OK;
}

sdv_status sdv_realign(sdv_ctx* c, const sdv_batch* b, sdv_result* r, void* stream) {
  if (!c || !batch_ok(c, b, false) || !result_ok(b, r)) return SDV_ERR_INVALID_ARG;
  if (!r->accepted || !r->final_tokens || !b->tokens) return SDV_ERR_INVALID_ARG;
  if (b->tree_parents) return SDV_ERR_UNSUPPORTED;  // the accepted path is not an input
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PrologueParams pp = prologue_params(c, b, r->status, false);
  SDV_CUDA(launch_prologue(pp, s));
  RealignParams rp = realign_params(c, b, r, r->accepted, r->final_tokens);
  SDV_CUDA(launch_realign(rp, s));
  return SDV_OK;
}

sdv_status sdv_admit(sdv_ctx* c, const sdv_admission* a, int* status, void* stream) {
  if (!c || !a || !status) return SDV_ERR_INVALID_ARG;
  if (a->live < 0 || a->n < 0 || a->n > 1024 || a->slots < 0 || a->live + a->n > a->slots) return SDV_ERR_INVALID_ARG;
  if (a->n > 0 && (!a->ctx_lens || !a->out_lens || !a->seq_lens || !a->num_pages || !a->gen_counts ||
                   !a->page_table || !a->free_pages))
    return SDV_ERR_INVALID_ARG;
  if (!a->num_free || !a->gen_limits || a->max_pages_per_seq < 1) return SDV_ERR_INVALID_ARG;
  if ((a->gen_limits_prev == nullptr) != (a->next_src == nullptr)) return SDV_ERR_INVALID_ARG;
  if (a->gen_limits_prev && a->gen_limits_prev == a->gen_limits) return SDV_ERR_INVALID_ARG;
  AdmitParams p;
  p.a = *a;
  p.gamma_max = c->cfg.gamma_max;
  p.page = c->cfg.page_size;
  p.status = status;
  SDV_CUDA(launch_admit(p, static_cast<cudaStream_t>(stream)));
  return SDV_OK;
}

sdv_status sdv_linear(sdv_ctx* c, int which, const void* x, int x_format, float* y, int rows, void* stream) {
  if (!c || !x || !y || rows <= 0 || rows > c->max_rows || which < 0 || which > 5) return SDV_ERR_INVALID_ARG;
  if (x_format != 0 && x_format != 1) return SDV_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const sdv_config& cf = c->cfg;
  const int H = cf.hidden, QD = cf.n_q * cf.head_dim, F = cf.ffn;
  const int NQKV = (cf.n_q + 2 * cf.n_kv) * cf.head_dim;
  const CUtensorMap *wm = nullptr, *sm = nullptr;
  int N = 0, K = 0;
  switch (which) {
    case 0: wm = &c->tm_qkv; sm = q4(c, c->ts_qkv); N = NQKV; K = H; break;
    case 1: wm = &c->tm_o; sm = q4(c, c->ts_o); N = H; K = QD; break;
    case 2: wm = &c->tm_gate; sm = q4(c, c->ts_gate); N = F; K = H; break;
    case 3: wm = &c->tm_up; sm = q4(c, c->ts_up); N = F; K = H; break;
    case 4: wm = &c->tm_down; sm = q4(c, c->ts_down); N = H; K = F; break;
    default: wm = &c->tm_lm; N = cf.vocab; K = H; break;
  }
  const bool xf32 = x_format == 1;
  // a private status word: the sentinel region after the attention schedule
  int* status = ws_ptr<int>(c, c->L.sched) + 8;
  SDV_CUDA(cudaMemsetAsync(status, 0, sizeof(int), s));
  GemmParams g = gemm_params(c, N, K, rows, (N + 127) / 128, status);
  const void* xsrc = x;
  if (xf32) {
    // fp32 input: split into bf16 hi + lo planes [2, rows, K] in the workspace
    __nv_bfloat16* planes = ws_ptr<__nv_bfloat16>(c, c->L.act);
    SDV_CUDA(launch_split_planes(static_cast<const float*>(x), planes, (long long)rows * K, (long long)rows * K, s));
    xsrc = planes;
    g.x_lo_row = rows;
  }
  CUtensorMap xm[kXMaps];
  for (int i = 0; i < kXMaps; ++i)
    if (!encode_bf16_2d(&xm[i], xsrc, (xf32 ? 2ull : 1ull) * rows, K, kXBoxes[i])) return SDV_ERR_CUDA;
  g.epi.out_f32 = y;
  g.epi.ld_f32 = N;
  SDV_CUDA(run_gemm(c, EPI_F32, xf32 ? 2 : 1, wm, wm, xm, g, s, sm, sm));
  return SDV_OK;
}

sdv_status sdv_attention(sdv_ctx* c, const void* q, const sdv_batch* b, void* out, int* status, void* stream) {
  if (!c || !q || !out || !status || !batch_ok(c, b, false) || !b->kv_pool) return SDV_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const AttnPlan plan = attn_plan(c, b->B);
  if (plan.st != SDV_OK) return plan.st;
  PrologueParams pp = prologue_params(c, b, status, false);
  pp.qsplit = plan.qsplit;
  pp.min_chunk = attn_min_chunk(plan);
  SDV_CUDA(launch_prologue(pp, s));
  // the kernel writes bf16 hi + lo planes; a plain fp32 result is their sum,
  // so stage the planes in the workspace and add them into `out`
  __nv_bfloat16* planes = ws_ptr<__nv_bfloat16>(c, c->L.attn);
  const long long n = (long long)b->R * c->cfg.n_q * c->cfg.head_dim;
  sdv_status st = run_attention(c, b, static_cast<const float*>(q), planes, n, status, s);
  if (st != SDV_OK) return st;
  SDV_CUDA(launch_join_planes(planes, n, static_cast<float*>(out), n, s));
  return SDV_OK;
}

}  // extern "C"
