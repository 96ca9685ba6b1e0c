// sdv_accept_static: acceptance, final-token sampling and realignment on given
// probabilities, with no context, no workspace and no allocation.
//
// Some callers cannot allocate device memory at the point where they verify
// drafts: an engine whose memory is carved up once at start-up and must never
// grow, code running inside a CUDA-graph capture (where cudaMalloc is not
// allowed), or a plugin living under a host framework that owns every
// allocation.  For them this entry point keeps its scratch in one fixed array
// of device memory that the library holds for its whole lifetime.
//
// The scratch is a file-scope __device__ array: every GPU that loads the
// library holds kScratchBytes of it until the process exits.  Host code only
// sees a host-side stand-in under the array's name, so the device address is
// fetched with cudaGetSymbolAddress, once per device, with that device
// current, on the first call made on it (make that first call before any
// stream capture).  The address belongs to the device's current CUDA context:
// it is looked up again when a call finds another context current (after a
// cudaDeviceReset, say), which makes that call a set-up call too.  All calls
// on a device share the array and it keeps what the last call left: the
// counters that must start at zero are cleared by each call, and calls whose
// work overlaps on the GPU (different streams without ordering between them)
// race on it.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace sdv {
namespace {

// Limits of the static scratch (each call is checked against them).
constexpr int kMaxSlots = 256;
constexpr int kMaxRows = 2048;
constexpr int kMaxVocab = 262144;
constexpr int kChunkLd = (kMaxVocab + kSampleChunk - 1) / kSampleChunk;  // sampling chunks

// Layout (bytes, 256-aligned regions).
constexpr size_t kAlign = 256;
constexpr size_t al(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }
constexpr size_t kRowOff = 0;
constexpr size_t kDraftOff = kRowOff + al((kMaxSlots + 1) * 4);
constexpr size_t kRowSeq = kDraftOff + al((kMaxSlots + 1) * 4);
constexpr size_t kRowPos = kRowSeq + al(kMaxRows * 4);
constexpr size_t kChunks = kRowPos + al(kMaxRows * 4);
constexpr size_t kItemOff = kChunks + al(kMaxSlots * 4);
constexpr size_t kSched = kItemOff + al((kMaxSlots + 1) * 4);
constexpr size_t kAccepted = kSched + al(64);
constexpr size_t kFinal = kAccepted + al(kMaxSlots * 4);
constexpr size_t kCounters = kFinal + al(kMaxSlots * 4);  // sampling chunks finished per slot
constexpr size_t kChunkSums = kCounters + al(kMaxSlots * 4);
constexpr size_t kScratchBytes = kChunkSums + al((size_t)kMaxSlots * 2 * kChunkLd * 8);

// What every GPU that loads the library holds (about 2.1 MB, nearly all of it
// the sampling chunk sums: 256 slots x 2 kinds x 512 chunks x 8 bytes).
static_assert(kScratchBytes <= 2200000, "the documented size of the static scratch");

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
// device address of g_scratch per device ordinal, and the context it was
// looked up in
void* g_scratch_dev[64] = {};
CUcontext g_scratch_ctx[64] = {};

// The driver's cuCtxGetCurrent, through the runtime's entry-point query (the
// library does not link the driver library directly).
PFN_cuCtxGetCurrent_v4000 ctx_get_current_fn() {
  static PFN_cuCtxGetCurrent_v4000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
  }();
  return fn;
}

CUcontext current_context() {
  CUcontext c = nullptr;
  const auto fn = ctx_get_current_fn();
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

cudaError_t scratch_for_current_device(unsigned char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  const CUcontext now = current_context();
  if (!g_scratch_dev[dev] || !now || now != g_scratch_ctx[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_scratch);  // makes the device's primary context current if none is
    if (e != cudaSuccess) return e;
    g_scratch_dev[dev] = ptr;
    g_scratch_ctx[dev] = current_context();
  }
  *out = static_cast<unsigned char*>(g_scratch_dev[dev]);
  return cudaSuccess;
}

}  // namespace
}  // namespace sdv

using namespace sdv;

extern "C" sdv_status sdv_accept_static(const sdv_config* cfg, const float* probs, const sdv_batch* b,
                                        sdv_result* r, void* stream) {
  if (!cfg || !probs || !b || !r || !r->status) return SDV_ERR_INVALID_ARG;
  if (b->B <= 0 || b->R < b->B || b->G != b->R - b->B) return SDV_ERR_INVALID_ARG;
  if (!b->seq_lens || !b->draft_lens || !b->tokens || !b->uniforms || !b->page_table || !b->num_pages ||
      !b->free_pages || !b->num_free_in || !b->num_free_out || (b->G > 0 && !b->draft_probs))
    return SDV_ERR_INVALID_ARG;
  if ((r->accept_tested == nullptr) != (r->accept_accepted == nullptr)) return SDV_ERR_INVALID_ARG;
  if (b->tree_parents) return SDV_ERR_UNSUPPORTED;  // token trees are verified greedily, with a context
  if (cfg->vocab <= 0 || cfg->page_size <= 0 || cfg->gamma_max < 0 || cfg->gamma_max > 63 ||
      b->max_pages_per_seq <= 0 || b->num_pool_pages <= 0)
    return SDV_ERR_INVALID_ARG;
  if (b->B > kMaxSlots || b->R > kMaxRows || cfg->vocab > kMaxVocab) return SDV_ERR_CAPACITY;
  if (accept_chunks(cfg->vocab) > kChunkLd) return SDV_ERR_INTERNAL;

  unsigned char* s = nullptr;
  cudaError_t e = scratch_for_current_device(&s);
  if (e != cudaSuccess) return SDV_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the arrival counters must start at zero whatever the last call left
  if (cudaMemsetAsync(s + kCounters, 0, kMaxSlots * 4, st) != cudaSuccess) return SDV_ERR_CUDA;

  PrologueParams pp;
  pp.t.row_off = reinterpret_cast<int*>(s + kRowOff);
  pp.t.draft_off = reinterpret_cast<int*>(s + kDraftOff);
  pp.t.row_seq = reinterpret_cast<int*>(s + kRowSeq);
  pp.t.row_pos = reinterpret_cast<int*>(s + kRowPos);
  pp.t.chunks = reinterpret_cast<int*>(s + kChunks);
  pp.t.item_off = reinterpret_cast<int*>(s + kItemOff);
  pp.t.sched = reinterpret_cast<int*>(s + kSched);
  pp.seq_lens = b->seq_lens;
  pp.draft_lens = b->draft_lens;
  pp.tokens = b->tokens;
  pp.page_table = b->page_table;
  pp.num_pages = b->num_pages;
  pp.status = r->status;
  pp.B = b->B;
  pp.R = b->R;
  pp.G = b->G;
  pp.gamma_max = cfg->gamma_max;
  pp.vocab = cfg->vocab;
  pp.page = cfg->page_size;
  pp.max_pages = b->max_pages_per_seq;
  pp.pool_pages = b->num_pool_pages;
  pp.n_kv = cfg->n_kv > 0 ? cfg->n_kv : 1;
  pp.head_dim = cfg->head_dim;
  pp.target_items = 1024;
  pp.check_tokens = 1;
  if (launch_prologue(pp, st) != cudaSuccess) return SDV_ERR_CUDA;

  int* accepted = r->accepted ? r->accepted : reinterpret_cast<int*>(s + kAccepted);
  int* final_tokens = r->final_tokens ? r->final_tokens : reinterpret_cast<int*>(s + kFinal);
  AcceptParams a;
  a.probs = probs;
  a.draft_probs = b->draft_probs;
  a.uniforms = b->uniforms;
  a.tokens = b->tokens;
  a.draft_lens = b->draft_lens;
  a.row_off = pp.t.row_off;
  a.draft_off = pp.t.draft_off;
  a.chunk_count = reinterpret_cast<int*>(s + kCounters);
  a.chunk_sums = reinterpret_cast<unsigned long long*>(s + kChunkSums);
  a.chunk_ld = kChunkLd;
  a.accepted = accepted;
  a.final_tokens = final_tokens;
  a.status = r->status;
  a.B = b->B;
  a.V = cfg->vocab;
  a.R = b->R;
  if (launch_accept(a, false, st) != cudaSuccess) return SDV_ERR_CUDA;

  RealignParams rp;
  rp.seq_lens = b->seq_lens;
  rp.draft_lens = b->draft_lens;
  rp.tokens = b->tokens;
  rp.row_off = pp.t.row_off;
  rp.accepted = accepted;
  rp.final_tokens = final_tokens;
  rp.page_table = b->page_table;
  rp.num_pages = b->num_pages;
  rp.free_pages = b->free_pages;
  rp.num_free_in = b->num_free_in;
  rp.num_free_out = b->num_free_out;
  rp.gen_counts = b->gen_counts;
  rp.gen_limits = b->gen_limits;
  rp.res = *r;
  rp.B = b->B;
  rp.page = cfg->page_size;
  rp.gamma_max = cfg->gamma_max;
  rp.max_pages = b->max_pages_per_seq;
  rp.pool_pages = b->num_pool_pages;
  rp.vocab = cfg->vocab;
  if (launch_realign(rp, st) != cudaSuccess) return SDV_ERR_CUDA;
  return SDV_OK;
}
