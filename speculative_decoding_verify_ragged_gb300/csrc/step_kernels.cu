// The step's small kernels: input validation and ragged row tables, the
// embedding + RMSNorm, the acceptance / final-token sampling, the debug
// softmax, and the realignment of lengths, pages and slots.
//
// Acceptance follows the rejection rule the pages cite for lossless
// speculation ("Speculative Decoding at High Batch Size", FAQ "Does
// speculative decoding change the output of the model?", after Leviathan,
// Kalman and Matias): draft x at row i is kept iff u < min(1, p_i(x)/q_i(x)),
// evaluated as (p >= q and p > 0) or u*q < p in float32; the first rejection
// ends the accepted prefix ("keeps the guesses it agrees with, up to the first
// one it would not have written, and adds one token of its own", splicedso
// primer, section "The idea").  The final token is drawn by inverse CDF from
// max(0, p - q) after a rejection and from p when all drafts are accepted; the
// draw runs on integer weights floor(w * 2^32), so the pick does not depend
// on the order in which a GPU block adds them up.
//
// Realignment gives every sequence its own new length L + a + 1 ("Speculative
// Decoding and Batching Compete for the Same Compute Slack on RDNA4", section
// "The batch also goes ragged": no padding to the longest accepted run),
// trims or extends its page list to cover the next step, and compacts the
// surviving slots in order so finished ones can be refilled ("Why Static
// Batching Wastes an RX 9070 XT Agent Swarm", section "Continuous batching
// refills the slot instead of freezing it").
#include "common.cuh"
#include "internal.h"

namespace sdv {

namespace {

constexpr int kScanThreads = 1024;

// Exclusive scan of one int per thread over a 1024-thread block; returns the
// thread's exclusive prefix and writes the block total to *total.
__device__ int block_exscan(int v, int* total, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
    int ws = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, ws, o);
      if (lane >= o) ws += y;
    }
    s_warp[32 + lane] = ws - w;  // exclusive warp offsets
    if (lane == 31) s_warp[64] = ws;
  }
  __syncthreads();
  const int res = s_warp[32 + warp] + x - v;
  *total = s_warp[64];
  __syncthreads();
  return res;
}

// ---------------------------------------------------------------------------
// prologue: validation + tables + attention schedule (one block)
// ---------------------------------------------------------------------------

// Block 0: validation, row tables, attention schedule.
__device__ void validate_and_tables(const PrologueParams& p, int* s_warp, int* s_poff) {
  __shared__ int s_err;
  const int b = threadIdx.x;
  if (b == 0) {
    *p.status = 0;
    s_err = 0;
  }
  __syncthreads();
  if (p.stall_ns) {
    // the test hook: a wait that nothing ends, given up after stall_ns
    __shared__ __align__(8) uint64_t s_never;
    if (b == 0) {
      mbar_init(&s_never, 1);
      fence_barrier_init();
      if (!mbar_wait(&s_never, 0, p.stall_ns)) set_status(p.status, SDV_ERR_TIMEOUT);
    }
    __syncthreads();
  }
  const bool slot = b < p.B;
  const int gam = slot ? p.draft_lens[b] : 0;
  const int L = slot ? p.seq_lens[b] : 0;
  const int npg = slot ? p.num_pages[b] : 0;
  int err = 0;
  if (slot) {
    if (gam < 0 || gam > p.gamma_max || L < 0) err = SDV_ERR_BAD_INPUT;
    else if (npg < 0 || npg > p.max_pages) err = SDV_ERR_PAGE_RANGE;
    else if ((long long)npg * p.page < (long long)L + gam + 1) err = SDV_ERR_PAGE_RANGE;
  }
  if (err) atomicCAS(&s_err, 0, err);
  const int used = (slot && !err) ? (L + gam + 1 + p.page - 1) / p.page : 0;
  int tot_r, tot_g, tot_pages;
  const int roff = block_exscan(slot ? gam + 1 : 0, &tot_r, s_warp);
  const int goff = block_exscan(slot ? gam : 0, &tot_g, s_warp);
  const int poff = block_exscan(used, &tot_pages, s_warp);
  if (b == 0 && (tot_r != p.R || tot_g != p.G)) atomicCAS(&s_err, 0, SDV_ERR_BAD_INPUT);
  if (slot && !err && p.tree_parents) {
    // a token tree: at most 64 nodes, node 0 the root, every other node's
    // parent an earlier node of the same slot
    bool ok = gam < 64 && roff + gam < p.R;
    for (int i = 0; ok && i <= gam; ++i) {
      const int par = p.tree_parents[roff + i];
      ok = i == 0 ? par == -1 : (par >= 0 && par < i);
    }
    if (!ok) atomicCAS(&s_err, 0, SDV_ERR_BAD_INPUT);
  }
  if (b < p.B) s_poff[b] = poff;
  if (b == 0) s_poff[p.B] = tot_pages;
  __syncthreads();
  if (s_err) {
    if (b == 0) set_status(p.status, s_err);
    return;
  }
  if (slot) {
    p.t.row_off[b] = roff;
    p.t.draft_off[b] = goff;
    if (p.tree_parents) {
      // depth and ancestor set (the node itself included) of every node, in
      // index order: a parent's entries are written before its children read them
      for (int i = 0; i <= gam; ++i) {
        int pos = L;
        unsigned long long anc = 1ull;
        if (i > 0) {
          const int par = p.tree_parents[roff + i];
          pos = p.t.row_pos[roff + par] + 1;
          anc = p.t.row_anc[roff + par] | (1ull << i);
        }
        p.t.row_seq[roff + i] = b;
        p.t.row_pos[roff + i] = pos;
        p.t.row_anc[roff + i] = anc;
      }
    } else {
      for (int i = 0; i <= gam; ++i) {
        p.t.row_seq[roff + i] = b;
        p.t.row_pos[roff + i] = L + i;
      }
    }
  }
  if (b == 0) {
    p.t.row_off[p.B] = tot_r;
    p.t.draft_off[p.B] = tot_g;
  }
  // every page a row reads or writes must be a pool page: one flat loop over
  // all (slot, page) pairs, the slot found by binary search over s_poff; eight
  // loads per thread in flight at a time
  constexpr int kUnroll = 8;
  for (int base = threadIdx.x; base < tot_pages; base += blockDim.x * kUnroll) {
    int pg[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int idx = base + u * blockDim.x;
      pg[u] = 0;
      if (idx < tot_pages) {
        int lo = 0, hi = p.B - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (s_poff[mid] <= idx) lo = mid; else hi = mid - 1;
        }
        pg[u] = p.page_table[(long long)lo * p.max_pages + (idx - s_poff[lo])];
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (pg[u] < 0 || pg[u] >= p.pool_pages) atomicCAS(&s_err, 0, SDV_ERR_PAGE_RANGE);
  }
  if (p.check_tokens) {
    for (int r = threadIdx.x; r < p.R; r += blockDim.x) {
      const int tk = p.tokens[r];
      if (tk < 0 || tk >= p.vocab) atomicCAS(&s_err, 0, SDV_ERR_BAD_INPUT);
    }
  }
  // attention schedule: chunks of pages sized so that items cover the GPU
  const long long units = (long long)tot_pages * p.n_kv;
  int chunk = static_cast<int>((units + p.target_items - 1) / p.target_items);
  chunk = (max(chunk, p.min_chunk) + 7) & ~7;  // whole 128-key blocks
  // a sequence's pages in chunks of `chunk`; a remainder of at most a quarter
  // chunk joins the last whole chunk (an item of a few leftover pages would pay
  // a whole item's pipeline fill)
  int chunks_b = slot ? (used + chunk - 1) / chunk : 0;
  if (chunks_b > 1 && used - (chunks_b - 1) * chunk <= chunk / 4) --chunks_b;
  // whether any slot's keys are split (else the merge kernel has nothing to do)
  const int any_split = __syncthreads_or(chunks_b > 1);
  // the slot's query vectors of one kv head, in items of at most qsplit
  const int nqv = (gam + 1) * (p.n_q / p.n_kv);
  const int halves = (slot && p.qsplit > 0) ? (nqv + p.qsplit - 1) / p.qsplit : 1;
  int tot_items;
  const int ioff = block_exscan(chunks_b * p.n_kv * halves, &tot_items, s_warp);
  // the slot of an item is found by binary search over the item offsets, so
  // that consecutive threads write consecutive records (one thread per slot
  // would write a lone sequence's hundreds of records serially)
  __shared__ int s_ioff[kScanThreads];
  __shared__ int4 s_rec[kScanThreads];
  if (slot) {
    p.t.chunks[b] = chunks_b;
    p.t.item_off[b] = ioff;
    s_ioff[b] = ioff;
    s_rec[b] = make_int4(L, gam, roff, chunks_b);
  }
  __syncthreads();
  if (p.t.items) {
    // item = ioff + (kv head * parts + part) * chunks + chunk; the part's first
    // query vector rides in the upper half of the kv head field
    for (int it = threadIdx.x; it < tot_items; it += blockDim.x) {
      int lo = 0, hi = p.B - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_ioff[mid] <= it) lo = mid; else hi = mid - 1;
      }
      const int4 rec = s_rec[lo];
      const int nb = rec.w;
      const int parts = p.qsplit > 0 ? ((rec.y + 1) * (p.n_q / p.n_kv) + p.qsplit - 1) / p.qsplit : 1;
      const int local = it - s_ioff[lo];
      const int c = local % nb, gh = local / nb;
      const int g = gh / parts, h = gh - g * parts;
      const int p0 = c * chunk;
      const int p1 = c == nb - 1 ? (rec.x + rec.y + 1 + p.page - 1) / p.page : p0 + chunk;
      p.t.items[2 * it] = make_int4(lo, g | ((h * p.qsplit) << 16), p0, p1);
      p.t.items[2 * it + 1] = rec;
    }
  }
  if (b == 0) {
    p.t.item_off[p.B] = tot_items;
    p.t.sched[0] = chunk;
    p.t.sched[1] = tot_items;
    p.t.sched[2] = any_split;
  }
  __syncthreads();
  if (b == 0 && s_err) set_status(p.status, s_err);
}

// ---------------------------------------------------------------------------
// embedding gather + RMSNorm (+ this row's rotary table); RMSNorm alone
// ---------------------------------------------------------------------------

__device__ float block_sum_256(float v, float* s) {
  v = warp_sum(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) s[warp] = v;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += s[w];
  __syncthreads();
  return t;
}

// Rows of the embedding blocks: four per 1024-thread block, a 256-thread
// group each.
constexpr int kRowsPerBlock = 4;
constexpr int kRowThreads = kScanThreads / kRowsPerBlock;

// Sum over the 256 threads of group g (named barrier 1 + g); s: 8 floats of
// the group's own.
__device__ float group_sum_256(float v, float* s, int g) {
  v = warp_sum(v);
  const int lane = threadIdx.x & 31, w = (threadIdx.x % kRowThreads) >> 5;
  if (lane == 0) s[w] = v;
  named_sync(1 + g, kRowThreads);
  float t = 0.f;
  for (int i = 0; i < kRowThreads / 32; ++i) t += s[i];
  named_sync(1 + g, kRowThreads);
  return t;
}

// Every embedding block: rows r_first .. r_first + 3, one 256-thread group
// each: the row's slot and position (one scan of the draft lengths for the
// block), the embedding row into the fp32 residual stream, the attention
// pre-norm, the rotary (cos, sin) table and the element offset of the row's
// K/V in the cache.  Row i of a slot writes its K/V at cache slot L + i; its
// rotary position is L + i in a chain and L + depth(i) in a token tree.
// Inputs that would make an access leave its buffer skip the access; block 0
// reports them in the status word.
__device__ void embed_rows(const PrologueParams& p, int r_first, int* s_warp) {
  __shared__ int s_b[kRowsPerBlock], s_i[kRowsPerBlock], s_depth[kRowsPerBlock];
  __shared__ float s_red[kRowsPerBlock][kRowThreads / 32];
  const int t = threadIdx.x;
  const int gam = t < p.B ? p.draft_lens[t] : 0;
  int tot;
  const int roff = block_exscan(t < p.B ? max(gam, 0) + 1 : 0, &tot, s_warp);
  if (t < kRowsPerBlock) s_b[t] = -1;
  __syncthreads();
  if (t < p.B) {
    for (int q = 0; q < kRowsPerBlock; ++q) {
      const int rq = r_first + q;
      if (rq >= roff && rq < roff + max(gam, 0) + 1) {
        s_b[q] = t;
        s_i[q] = rq - roff;
      }
    }
  }
  __syncthreads();
  // from here on each group works alone (named barrier 1 + g)
  const int g = t / kRowThreads, u = t % kRowThreads;
  const int r = r_first + g;
  const int b = s_b[g];
  if (b < 0 || r >= p.R) return;
  const int si = s_i[g];
  const int slot_pos = p.seq_lens[b] + si;  // cache slot of the row's K/V
  int depth = si;
  if (p.tree_parents) {
    if (u == 0) {
      // parents up to the root; a malformed table ends the walk (block 0 reports it)
      const int r0 = r - si;
      int v = si, d = 0;
      while (v > 0 && d < 64) {
        const int par = p.tree_parents[r0 + v];
        if (par < 0 || par >= v) break;
        v = par;
        ++d;
      }
      s_depth[g] = d;
    }
    named_sync(1 + g, kRowThreads);
    depth = s_depth[g];
  }
  const int pos = p.seq_lens[b] + depth;  // rotary position
  const int tok = p.tokens[r];
  if (u == 0) {
    const int pi = slot_pos / p.page;
    long long off = 0;
    if (slot_pos >= 0 && pi < p.num_pages[b] && pi < p.max_pages) {
      const int pg = p.page_table[(long long)b * p.max_pages + pi];
      if (pg >= 0 && pg < p.pool_pages)
        off = (long long)pg * p.n_kv * 2 * p.page * p.head_dim + (long long)(slot_pos - pi * p.page) * p.head_dim;
    }
    p.t.kv_row_off[r] = off;
  }
  // rotary table: angle = pos * inv_freq_j (double), reduced mod 2 pi, then fp32 sincos
  const int half = p.head_dim >> 1;
  for (int j = u; j < half; j += kRowThreads) {
    const double two_pi = 6.283185307179586476925286766559;
    const double ang = static_cast<double>(pos) * p.inv_freq[j];
    const double red = fma(-rint(ang * (1.0 / two_pi)), two_pi, ang);
    float sn, cs;
    sincosf(static_cast<float>(red), &sn, &cs);
    p.t.rope_cs[((long long)r * half + j) * 2] = cs;
    p.t.rope_cs[((long long)r * half + j) * 2 + 1] = sn;
  }
  if (tok < 0 || tok >= p.vocab) return;
  // embedding row (bf16, eight per 16-byte load) -> fp32 residual stream;
  // RMSNorm from registers; the normalised row as bf16 hi + lo planes
  constexpr int PER8 = 4;  // 8-element vectors per thread: hidden <= 8 * 4 * 256
  const uint4* e8 = reinterpret_cast<const uint4*>(p.emb + (long long)tok * p.H);
  const uint4* g8 = reinterpret_cast<const uint4*>(p.gain);
  const int n8 = p.H >> 3;
  uint4 raw[PER8], gr[PER8];
#pragma unroll
  for (int q = 0; q < PER8; ++q) {
    const int k = u + q * kRowThreads;
    raw[q] = k < n8 ? e8[k] : make_uint4(0u, 0u, 0u, 0u);
    gr[q] = k < n8 ? g8[k] : make_uint4(0u, 0u, 0u, 0u);
  }
  auto lo16 = [](uint32_t w) { return __uint_as_float(w << 16); };
  auto hi16 = [](uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); };
  float ss = 0.f;
  float4* x0 = reinterpret_cast<float4*>(p.x0 + (long long)r * p.H);
#pragma unroll
  for (int q = 0; q < PER8; ++q) {
    const int k = u + q * kRowThreads;
    const uint32_t w[4] = {raw[q].x, raw[q].y, raw[q].z, raw[q].w};
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = lo16(w[i]);
      v[2 * i + 1] = hi16(w[i]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) ss += v[i] * v[i];
    if (k < n8) {
      x0[2 * k] = make_float4(v[0], v[1], v[2], v[3]);
      x0[2 * k + 1] = make_float4(v[4], v[5], v[6], v[7]);
    }
  }
  ss = group_sum_256(ss, s_red[g], g);
  const float inv = 1.0f / sqrtf(ss / static_cast<float>(p.H) + p.eps);
  __nv_bfloat16* h = p.h + (long long)r * p.H;
#pragma unroll
  for (int q = 0; q < PER8; ++q) {
    const int k = u + q * kRowThreads;
    if (k >= n8) continue;
    const uint32_t w[4] = {raw[q].x, raw[q].y, raw[q].z, raw[q].w};
    const uint32_t gw[4] = {gr[q].x, gr[q].y, gr[q].z, gr[q].w};
    uint32_t hv[4], lv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      split_bf16x2(lo16(w[i]) * inv * lo16(gw[i]), hi16(w[i]) * inv * hi16(gw[i]), hv[i], lv[i]);
    *reinterpret_cast<uint4*>(h + 8 * k) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
    *reinterpret_cast<uint4*>(h + p.h_lo_off + 8 * k) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
  }
}

__global__ void __launch_bounds__(kScanThreads) prologue_kernel(const PrologueParams p) {
  SDV_TRACE_SCOPE(kTrPrologue);
  __shared__ int s_warp[80];
  __shared__ int s_poff[kScanThreads + 1];
  griddep_launch_dependents();
  SDV_GRIDDEP_WAIT();  // the previous step's realignment rewrites page tables and counters
  // block 0 validates and builds the tables; block r + 1 prepares row r
  if (blockIdx.x == 0) validate_and_tables(p, s_warp, s_poff);
  else embed_rows(p, (blockIdx.x - 1) * kRowsPerBlock, s_warp);
}

__global__ void __launch_bounds__(256) rmsnorm_kernel(const float* x, const __nv_bfloat16* gain, __nv_bfloat16* h,
                                                      long long lo_off, int H, float eps, const int* status) {
  SDV_TRACE_SCOPE(kTrFinalNorm);
  __shared__ float s_red[32];
  griddep_launch_dependents();
  SDV_GRIDDEP_WAIT();
  // the row is loaded alongside the status word (it lies inside the buffer
  // whatever the verdict); h = x / sqrt(mean(x^2) + eps) * gain as bf16 hi + lo
  // planes lo_off elements apart (lo_off == 0: one rounded plane)
  constexpr int PER4 = 8;  // float4s per thread: hidden <= 8 * 4 * 256
  const int r = blockIdx.x;
  const float4* xr = reinterpret_cast<const float4*>(x + (long long)r * H);
  const int n4 = H >> 2;
  const int st = read_status(status);
  float4 v[PER4];
#pragma unroll
  for (int q = 0; q < PER4; ++q) {
    const int k = threadIdx.x + q * 256;
    v[q] = k < n4 ? xr[k] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (st != 0) return;
  float ss = 0.f;
#pragma unroll
  for (int q = 0; q < PER4; ++q) ss += v[q].x * v[q].x + v[q].y * v[q].y + v[q].z * v[q].z + v[q].w * v[q].w;
  ss = block_sum_256(ss, s_red);
  const float inv = 1.0f / sqrtf(ss / static_cast<float>(H) + eps);
  __nv_bfloat16* hr = h + (long long)r * H;
#pragma unroll
  for (int q = 0; q < PER4; ++q) {
    const int k = threadIdx.x + q * 256;
    if (k < n4) {
      store_planes(hr, lo_off, 4 * k, v[q].x * inv * bf2f(gain[4 * k]));
      store_planes(hr, lo_off, 4 * k + 1, v[q].y * inv * bf2f(gain[4 * k + 1]));
      store_planes(hr, lo_off, 4 * k + 2, v[q].z * inv * bf2f(gain[4 * k + 2]));
      store_planes(hr, lo_off, 4 * k + 3, v[q].w * inv * bf2f(gain[4 * k + 3]));
    }
  }
}

__global__ void join_planes_kernel(const __nv_bfloat16* hi, long long lo_off, float* out, long long n) {
  SDV_TRACE_SCOPE(kTrPlanes);
  griddep_launch_dependents();
  SDV_GRIDDEP_WAIT();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    out[i] = __bfloat162float(hi[i]) + __bfloat162float(hi[i + lo_off]);
}

__global__ void split_planes_kernel(const float* x, __nv_bfloat16* out, long long lo_off, long long n) {
  SDV_TRACE_SCOPE(kTrPlanes);
  griddep_launch_dependents();
  SDV_GRIDDEP_WAIT();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    store_planes(out, lo_off, i, x[i]);
}

// ---------------------------------------------------------------------------
// acceptance + final-token sampling
//
// Kernel A (one block per sequence): the softmax normalisers of the
// sequence's rows from the LM head's per-tile statistics, then every draft's
// test in parallel; the first failing u < min(1, p/q) ends the accepted prefix.
// Kernel B (a few blocks per sequence, one warp per 512-entry vocab chunk):
// integer weight sums of the final row over each chunk (residual and plain);
// the sequence's last block to finish draws the token.  Integer sums make the
// draw independent of block order.
// Stochastic verification from logits runs kernel A's work inside each block
// of kernel B (one launch, one kernel boundary fewer); greedy verification,
// token trees and given probabilities keep kernel A.
// Both read the caller's draft inputs before waiting for the kernel ahead.
// ---------------------------------------------------------------------------

// Timeline rows of points inside the sampling kernel (rows no GEMM fixup
// uses): status read, row statistics merged, draft tests done, chunk sums
// stored, the slot's last block starts, the draw's chunk found.  Columns 0
// and 1: the earliest block to reach the point; column 2: the latest.
enum SamplePhase {
  kTrSmpStatus = 25, kTrSmpMerged = 26, kTrSmpTested = 27, kTrSmpChunks = 28, kTrSmpLast = 29, kTrSmpChunk = 30
};
#ifdef SDV_TRACE
#define SDV_TRACE_PHASE(slot)                            \
  do {                                                   \
    if (c_trace && threadIdx.x == 0) {                   \
      const unsigned long long t_ = trace_clock();       \
      atomicMin(&c_trace[3 * (slot)], t_);               \
      atomicMin(&c_trace[3 * (slot) + 1], t_);           \
      atomicMax(&c_trace[3 * (slot) + 2], t_);           \
    }                                                    \
  } while (0)
#else
#define SDV_TRACE_PHASE(slot) \
  do {                        \
  } while (0)
#endif

constexpr int kAccThreads = 256;
constexpr int kAccWarps = kAccThreads / 32;
constexpr int kVChunk = kSampleChunk;  // vocab entries per sampling warp
constexpr int kPerThread = kVChunk / kAccThreads;
constexpr int kChunksPerThread = kMaxSampleChunks / kAccThreads;  // last block's scan

// The sampling weights are floor(w * 2^32) (fixed point, summed exactly).
// Kernels carry x = w * 2^32, an exact scaling of w, and take the floor in two
// 16-bit halves: x = h * 2^16 + r with h = floor(x / 2^16), r < 2^16 exact, and
// floor(x) = h * 2^16 + floor(r).  A round-down add of 2^23 to a value v in
// [0, 2^23) gives 2^23 + floor(v) exactly, whose bits are kFixBias + floor(v):
// two adds per floor on the FMA pipe instead of a float -> integer conversion
// or 64-bit shifts.  Valid for x in [0, 2^33), i.e. w in [0, 2).
constexpr uint32_t kFixBias = 0x4B000000u;  // the bits of 2^23
constexpr float kFixScale = 4294967296.0f;   // 2^32

__device__ __forceinline__ void fixed_split(float x, uint32_t& hb, uint32_t& lb) {
  const float h = __fadd_rd(__fmul_rn(x, 1.0f / 65536.0f), 8388608.0f);
  hb = __float_as_uint(h);
  lb = __float_as_uint(__fadd_rd(__fmaf_rn(__fsub_rn(h, 8388608.0f), -65536.0f, x), 8388608.0f));
}

// floor(x) of one x in [0, 2^33)
__device__ __forceinline__ unsigned long long fixed_of(float x) {
  uint32_t hb, lb;
  fixed_split(x, hb, lb);
  return (static_cast<unsigned long long>(hb - kFixBias) << 16) + (lb - kFixBias);
}

// Running sums of the biased halves of a lane's terms; the bias comes out once
// (n terms: n * kFixBias, wrapping) and the true halves, below n * 2^17, stay
// exact in 32 bits for n * 32 lanes <= 2^15 terms.
struct FixedAcc {
  uint32_t h = 0, l = 0;
  __device__ __forceinline__ void add(float x) {
    uint32_t hb, lb;
    fixed_split(x, hb, lb);
    h += hb;
    l += lb;
  }
};

// The sampled distribution's x = w * 2^32 for the raw value v of a row: from
// logits 2^((v - M) log2 e) * 2^32 / sum, with nml = -M log2 e and s32 = 2^32 /
// sum; given probabilities times 2^32, clamped to [0, 2) (the weights' range;
// NaN reads as 0).
template <bool FROM_LOGITS>
struct PSource {
  const float* base;  // logits or probabilities
  int V;
  __device__ __forceinline__ float x_of(float v, float nml, float s32) const {
    if constexpr (FROM_LOGITS) {
      return __fmul_rn(exp2f(__fmaf_rn(v, kLog2e, nml)), s32);
    } else {
      return __fmul_rn(fminf(fmaxf(v, 0.f), 1.99999988f), kFixScale);
    }
  }
  __device__ __forceinline__ float x(int row, int j, float nml, float s32) const {
    return x_of(base[(long long)row * V + j], nml, s32);
  }
};

// x of the residual max(0, p - q): (p - q) * 2^32 rounded once, as p - q is
__device__ __forceinline__ float residual_x(float x, float q) {
  return fmaxf(0.f, __fmaf_rn(q, -kFixScale, x));
}

// First row of slot b: the sum of (gamma + 1) over the earlier slots, from the
// caller's draft lengths (so it can be read before the kernel ahead finishes).
__device__ int slot_row0(const int* draft_lens, int b, int* s_tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int part = 0;
  for (int j = threadIdx.x; j < b; j += kAccThreads) part += draft_lens[j] + 1;
  part = warp_sum(part);
  if (lane == 0) s_tmp[warp] = part;
  __syncthreads();
  int t = 0;
  for (int w = 0; w < kAccWarps; ++w) t += s_tmp[w];
  __syncthreads();
  return t;
}

// Argmax merge: the larger value wins, equal values keep the smaller index.
__device__ __forceinline__ void merge_arg(float& m, int& a, float om, int oa) {
  if (om > m || (om == m && oa < a)) {
    m = om;
    a = oa;
  }
}

// Softmax normalisers (max, sum of exp) of rows r0 .. r0 + gam from the LM
// head's per-tile statistics, into s_st, and (greedy) each row's argmax into
// s_arg; write_rows: also into p.row_stats.  The whole block calls it.
// Rows go 8 (or fewer: rounded up to a power of two, rp) at a time; thread t
// takes row t % rp over tiles t / rp, t / rp + 256 / rp, ...: kMergeBatch
// tiles' loads in flight, their maximum first, then each tile's sum scaled by
// one exponential.  Lanes of one row meet by shuffles, warps through shared
// memory (maximum first again).  The order is fixed: every block of a slot
// that calls it gets the same values.
constexpr int kMergeBatch = 20;  // 1187 tiles (a 151936-entry vocabulary) in two rounds at 8 rows

__device__ void merge_slot_stats(const AcceptParams& p, int r0, int gam, float2* s_st, int* s_arg, bool write_rows) {
  __shared__ float s_m[kAccWarps][8], s_s[kAccWarps][8];
  __shared__ int s_g[kAccWarps][8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int n0 = 0; n0 <= gam; n0 += 8) {
    const int nr = min(8, gam + 1 - n0);
    const int lg = nr > 4 ? 3 : (nr > 2 ? 2 : (nr > 1 ? 1 : 0));
    const int rp = 1 << lg;
    const int q = threadIdx.x & (rp - 1);
    const int tstep = kAccThreads >> lg;
    const bool live = q < nr;
    const long long col = r0 + n0 + q;
    float M = -INFINITY, S = 0.f, GM = -INFINITY;
    int GA = 0x7FFFFFFF;
    for (int t0 = threadIdx.x >> lg; t0 < p.m_tiles; t0 += kMergeBatch * tstep) {
      float2 st[kMergeBatch];
#pragma unroll
      for (int i = 0; i < kMergeBatch; ++i) {
        const int tt = t0 + i * tstep;
        st[i] = live && tt < p.m_tiles ? p.tile_stats[(long long)tt * p.stats_ld + col] : make_float2(-INFINITY, 0.f);
      }
      if (p.greedy) {
#pragma unroll
        for (int i = 0; i < kMergeBatch; ++i) {
          const int tt = t0 + i * tstep;
          if (live && tt < p.m_tiles) merge_arg(GM, GA, st[i].x, p.tile_argmax[(long long)tt * p.stats_ld + col]);
        }
      }
      float cm = M;
#pragma unroll
      for (int i = 0; i < kMergeBatch; ++i) cm = fmaxf(cm, st[i].x);
      if (cm > -INFINITY) {
        // exp2(-inf) = 0 takes out the empty terms (and the old sum while M = -inf)
        float acc = S * exp2f((M - cm) * kLog2e);
#pragma unroll
        for (int i = 0; i < kMergeBatch; ++i) acc += st[i].y * exp2f((st[i].x - cm) * kLog2e);
        S = acc;
        M = cm;
      }
    }
    for (int o = rp; o < 32; o <<= 1) {
      const float oM = __shfl_xor_sync(0xffffffffu, M, o);
      const float oS = __shfl_xor_sync(0xffffffffu, S, o);
      merge_ms(M, S, oM, oS);
      if (p.greedy) {
        const float gM = __shfl_xor_sync(0xffffffffu, GM, o);
        const int gA = __shfl_xor_sync(0xffffffffu, GA, o);
        merge_arg(GM, GA, gM, gA);
      }
    }
    if (lane < rp) {
      s_m[warp][lane] = M;
      s_s[warp][lane] = S;
      s_g[warp][lane] = GA;
    }
    __syncthreads();
    if (threadIdx.x < nr) {
      float Mr = -INFINITY, Gm = -INFINITY;
      int Ga = 0x7FFFFFFF;
      for (int w = 0; w < kAccWarps; ++w) {
        Mr = fmaxf(Mr, s_m[w][threadIdx.x]);
        merge_arg(Gm, Ga, s_m[w][threadIdx.x], s_g[w][threadIdx.x]);
      }
      float Sr = 0.f;
      if (Mr > -INFINITY)
        for (int w = 0; w < kAccWarps; ++w) Sr += s_s[w][threadIdx.x] * exp2f((s_m[w][threadIdx.x] - Mr) * kLog2e);
      s_st[n0 + threadIdx.x] = make_float2(Mr, Sr);
      if (write_rows) p.row_stats[r0 + n0 + threadIdx.x] = make_float2(Mr, Sr);
      s_arg[n0 + threadIdx.x] = Ga;
    }
    __syncthreads();
  }
}

template <bool FROM_LOGITS>
__global__ void __launch_bounds__(kAccThreads) accept_kernel(const AcceptParams p) {
  SDV_TRACE_SCOPE(kTrAccept);
  __shared__ int s_tmp[kAccWarps];
  __shared__ float s_m[kAccWarps];  // given probabilities, greedy: per-warp row maxima
  __shared__ int s_g[kAccWarps];
  __shared__ float2 s_st[64];
  __shared__ int s_arg[64];
  __shared__ int s_par[64], s_tok[64];  // token trees: parent and token of each node
  __shared__ int s_a;
  griddep_launch_dependents();
  const int b = blockIdx.x;
  const int V = p.V;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gam = p.draft_lens[b];
  const int r0 = slot_row0(p.draft_lens, b, s_tmp);
  const int g0 = r0 - b;  // draft rows of the earlier slots
  // inputs are validated by the prologue; until its verdict is read every read is bounds-checked
  const bool in_range = gam >= 0 && gam < 64 && r0 >= 0 && r0 + gam < p.R;
  int x = 0;
  float qk = 0.f, uk = 0.f;
  if (in_range && threadIdx.x < gam) {
    x = p.tokens[r0 + threadIdx.x + 1];
    if (x >= 0 && x < V && !p.greedy) {
      qk = p.draft_probs[(long long)(g0 + threadIdx.x) * V + x];
      uk = p.uniforms[r0 + threadIdx.x];
    }
    if (p.tree_parents) {
      s_par[threadIdx.x + 1] = p.tree_parents[r0 + threadIdx.x + 1];
      s_tok[threadIdx.x + 1] = x;
    }
  }
  if (threadIdx.x == 0) s_a = gam;
  SDV_GRIDDEP_WAIT();
  // the status word and the drafts' logits are loaded together (the logit
  // loads stay inside the buffer whatever the verdict)
  const int st = read_status(p.status);
  float zx = 0.f;
  if constexpr (FROM_LOGITS) {
    if (in_range && threadIdx.x < gam && x >= 0 && x < V) zx = p.z[(long long)(r0 + threadIdx.x) * V + x];
  }
  if (st != 0) return;
  __syncthreads();  // s_a is set before any test lowers it
  if constexpr (FROM_LOGITS) {
    merge_slot_stats(p, r0, gam, s_st, s_arg, true);
  }
  if (p.greedy) {
    // greedy verification (temperature -> 0): draft i + 1 is kept iff it is the
    // argmax of row i (the smallest index among equal maxima); the token after
    // the kept prefix is the argmax of its row
    if constexpr (!FROM_LOGITS) {
      // given probabilities: a block-wide argmax of each row
      for (int n = 0; n <= gam; ++n) {
        const float* row = p.probs + (long long)(r0 + n) * V;
        float m = -INFINITY;
        int a = 0x7FFFFFFF;
        for (int j = threadIdx.x; j < V; j += kAccThreads) merge_arg(m, a, row[j], j);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float om = __shfl_xor_sync(0xffffffffu, m, o);
          const int oa = __shfl_xor_sync(0xffffffffu, a, o);
          merge_arg(m, a, om, oa);
        }
        if (lane == 0) {
          s_m[warp] = m;
          s_g[warp] = a;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
          float bm = -INFINITY;
          int ba = 0x7FFFFFFF;
          for (int w = 0; w < kAccWarps; ++w) merge_arg(bm, ba, s_m[w], s_g[w]);
          s_arg[n] = ba;
        }
        __syncthreads();
      }
    }
    if (p.tree_parents) {
      // token tree: from the root, step into the child (smallest index first)
      // whose token is the current node's argmax; the accepted count is the
      // depth reached and the final token the argmax where the walk stops.
      // Every step moves to a larger node index, so the walk ends within gam
      // steps (parents were validated by the prologue).
      if (warp == 0) {
        int node = 0, depth = 0;
        for (int step = 0; step < 64; ++step) {
          const int want = s_arg[node];
          const int c0 = lane, c1 = lane + 32;
          const bool m0 = c0 >= 1 && c0 <= gam && s_par[c0] == node && s_tok[c0] == want;
          const bool m1 = c1 <= gam && s_par[c1] == node && s_tok[c1] == want;
          const unsigned b0 = __ballot_sync(0xffffffffu, m0), b1 = __ballot_sync(0xffffffffu, m1);
          if (b0 == 0u && b1 == 0u) break;
          const int child = b0 ? __ffs(b0) - 1 : 32 + __ffs(b1) - 1;
          if (lane == 0) p.tree_path[g0 + depth] = child;
          ++depth;
          node = child;
        }
        if (lane == 0) {
          p.accepted[b] = depth;
          p.final_tokens[b] = s_arg[node];
        }
      }
      return;
    }
    if (threadIdx.x < gam && x != s_arg[threadIdx.x]) atomicMin(&s_a, static_cast<int>(threadIdx.x));
    __syncthreads();
    if (threadIdx.x == 0) {
      p.accepted[b] = s_a;
      p.final_tokens[b] = s_arg[s_a];
    }
    return;
  }
  if (threadIdx.x < gam) {
    const int k = threadIdx.x;
    float pk;
    if constexpr (FROM_LOGITS) pk = expf(zx - s_st[k].x) / s_st[k].y;
    else pk = p.probs[(long long)(r0 + k) * V + x];
    if (!((pk >= qk && pk > 0.f) || (__fmul_rn(uk, qk) < pk))) atomicMin(&s_a, k);
  }
  __syncthreads();
  if (threadIdx.x == 0) p.accepted[b] = s_a;
}

// FUSED (from logits, stochastic): every block of a slot also merges the
// slot's row statistics and runs the draft tests itself (the same arithmetic
// in the same order as the acceptance kernel, so all blocks agree on the
// accepted count); block 0 stores the count and the row statistics.
template <bool FROM_LOGITS, bool FUSED>
__global__ void __launch_bounds__(kAccThreads, 4) sample_kernel(const AcceptParams p) {
  static_assert(FROM_LOGITS || !FUSED, "the fused tests read logits");
  SDV_TRACE_SCOPE(kTrSample);
  __shared__ unsigned long long s_red[2][kAccWarps];
  __shared__ unsigned long long s_scan[kAccWarps];
  __shared__ int s_last, s_mode, s_chunk, s_tok;
  __shared__ int s_tmp[kAccWarps];
  __shared__ unsigned long long s_T, s_base;
  __shared__ unsigned long long s_cs[2][kMaxSampleChunks];
  griddep_launch_dependents();
  const int b = blockIdx.y;
  const int V = p.V;
  const int nch = (V + kVChunk - 1) / kVChunk;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gam = p.draft_lens[b];
  const int r0 = slot_row0(p.draft_lens, b, s_tmp);
  const int g0 = r0 - b;
  // the final draw's uniform (the caller's, at row r0 + gamma) for the thread
  // that draws, read before the wait (bounds-checked until the verdict)
  float u_fin = 0.f;
  if (threadIdx.x == 0 && gam >= 0 && r0 >= 0 && r0 + gam < p.R) u_fin = p.uniforms[r0 + gam];
  __shared__ float2 s_rst[64];
  // A block that finds the status word set skips the work but still counts
  // itself on the slot's arrival counter below, so the counter returns to
  // zero whatever the status: another slot's last block may set the word
  // while this launch runs, and a counter left short would make a later
  // call's blocks draw from chunk sums not yet written.  The verdict is made
  // block-uniform by the barrier that reduces it.
  bool dead;
  int a = 0;
  if constexpr (FUSED) {
    __shared__ int s_arg[64], s_a;
    // the drafts' tokens, q values and uniforms are the caller's: read before
    // the wait, bounds-checked until the prologue's verdict is known
    const bool in_range = gam >= 0 && gam < 64 && r0 >= 0 && r0 + gam < p.R;
    int x = 0;
    float qk = 0.f, uk = 0.f;
    if (in_range && threadIdx.x < gam) {
      x = p.tokens[r0 + threadIdx.x + 1];
      if (x >= 0 && x < V) {
        qk = p.draft_probs[(long long)(g0 + threadIdx.x) * V + x];
        uk = p.uniforms[r0 + threadIdx.x];
      }
    }
    if (threadIdx.x == 0) s_a = gam;
    SDV_GRIDDEP_WAIT();
    const int st = read_status(p.status);
    float zx = 0.f;
    if (in_range && threadIdx.x < gam && x >= 0 && x < V) zx = p.z[(long long)(r0 + threadIdx.x) * V + x];
    dead = __syncthreads_or(st != 0) != 0;  // also: s_a is set before any test lowers it
    if (!dead) {
      SDV_TRACE_PHASE(kTrSmpStatus);
      merge_slot_stats(p, r0, gam, s_rst, s_arg, blockIdx.x == 0);
      SDV_TRACE_PHASE(kTrSmpMerged);
      if (threadIdx.x < gam) {
        const int k = threadIdx.x;
        const float pk = expf(zx - s_rst[k].x) / s_rst[k].y;
        if (!((pk >= qk && pk > 0.f) || (__fmul_rn(uk, qk) < pk))) atomicMin(&s_a, k);
      }
      __syncthreads();
      a = s_a;
      SDV_TRACE_PHASE(kTrSmpTested);
      if (blockIdx.x == 0 && threadIdx.x == 0) p.accepted[b] = a;
    }
  } else {
    SDV_GRIDDEP_WAIT();
    // the status word, the accepted count and the statistics of every row the
    // final token may come from are loaded together
    const int st = read_status(p.status);
    a = p.accepted[b];
    if constexpr (FROM_LOGITS) {
      if (threadIdx.x <= gam && threadIdx.x < 64 && r0 + (int)threadIdx.x < p.R)
        s_rst[threadIdx.x] = p.row_stats[r0 + threadIdx.x];
    }
    dead = __syncthreads_or(st != 0) != 0;
  }
  const int rf = r0 + a;
  const float* qrow = !dead && a < gam ? p.draft_probs + (long long)(g0 + a) * V : nullptr;
  // x = w * 2^32 of the row: from logits 2^((z - M) log2 e) * 2^32 / sum
  float nml = 0.f, s32 = kFixScale;
  if constexpr (FROM_LOGITS) {
    if (!dead) {
      const float2 rs = s_rst[a];
      nml = -rs.x * kLog2e;
      s32 = __fmul_rn(1.f / rs.y, kFixScale);
    }
  }
  PSource<FROM_LOGITS> src{FROM_LOGITS ? p.z : p.probs, V};

  // chunk sums of the residual weights max(0, p - q) and of the plain weights
  // p: warp w of block x takes chunks x * warps + w, stepping over the slot's
  // blocks; each lane issues all its loads of a chunk before using them and
  // adds 16 terms to each sum (entries past the vocabulary as zeros)
  unsigned long long* cs = p.chunk_sums + (long long)b * p.chunk_ld * 2;
  const float* prow = (FROM_LOGITS ? p.z : p.probs) + (long long)rf * V;
  const bool vec = (V & 3) == 0;  // rows are 16-byte aligned: float4 loads
  constexpr int kVecPerLane = kVChunk / (4 * kWarp);
  constexpr uint32_t kLaneTerms = kVChunk / kWarp;
  static_assert(kLaneTerms * kWarp <= (1u << 15), "the halves' sums stay exact in 32 bits");
  const bool has_q = qrow != nullptr;
  for (int c = blockIdx.x * kAccWarps + warp; !dead && c < nch; c += gridDim.x * kAccWarps) {
    FixedAcc ap, ar;
    const int j0 = c * kVChunk;
    if (vec) {
      float4 zv[kVecPerLane], qv[kVecPerLane];
#pragma unroll
      for (int e = 0; e < kVecPerLane; ++e) {
        const int j = j0 + (e * kWarp + lane) * 4;
        zv[e] = make_float4(0.f, 0.f, 0.f, 0.f);
        qv[e] = zv[e];
        if (j < V) {
          zv[e] = __ldcs(reinterpret_cast<const float4*>(prow + j));
          if (has_q) qv[e] = __ldcs(reinterpret_cast<const float4*>(qrow + j));
        }
      }
#pragma unroll
      for (int e = 0; e < kVecPerLane; ++e) {
        const bool in = j0 + (e * kWarp + lane) * 4 < V;
        const float zz[4] = {zv[e].x, zv[e].y, zv[e].z, zv[e].w};
        const float qq[4] = {qv[e].x, qv[e].y, qv[e].z, qv[e].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float x = in ? src.x_of(zz[k], nml, s32) : 0.f;
          ap.add(x);
          if (has_q) ar.add(residual_x(x, qq[k]));
        }
      }
    } else {
      for (int e = lane; e < kVChunk; e += kWarp) {
        const int j = j0 + e;
        const float x = j < V ? src.x(rf, j, nml, s32) : 0.f;
        ap.add(x);
        if (has_q) ar.add(j < V ? residual_x(x, qrow[j]) : 0.f);
      }
    }
    uint32_t ph = ap.h - kLaneTerms * kFixBias, pl = ap.l - kLaneTerms * kFixBias;
    uint32_t rh = has_q ? ar.h - kLaneTerms * kFixBias : 0u, rl = has_q ? ar.l - kLaneTerms * kFixBias : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ph += __shfl_xor_sync(0xffffffffu, ph, o);
      pl += __shfl_xor_sync(0xffffffffu, pl, o);
      if (has_q) {
        rh += __shfl_xor_sync(0xffffffffu, rh, o);
        rl += __shfl_xor_sync(0xffffffffu, rl, o);
      }
    }
    if (lane == 0) {
      cs[c] = (static_cast<unsigned long long>(rh) << 16) + rl;
      cs[p.chunk_ld + c] = (static_cast<unsigned long long>(ph) << 16) + pl;
    }
  }
  __syncthreads();
  SDV_TRACE_PHASE(kTrSmpChunks);
  if (threadIdx.x == 0) {
    __threadfence();
    const int old = atomicAdd(&p.chunk_count[b], 1);
    s_last = old == (int)gridDim.x - 1 ? 1 : 0;
    // the last block of a call that failed anywhere only resets the counter
    if (s_last && (dead || read_status(p.status) != 0)) {
      p.chunk_count[b] = 0;
      s_last = 0;
    }
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  SDV_TRACE_PHASE(kTrSmpLast);

  // last block of this sequence: pick the mode, the target and the chunk
  {
    for (int k = threadIdx.x; k < nch; k += kAccThreads) {
      s_cs[0][k] = __ldcg(&cs[k]);
      s_cs[1][k] = __ldcg(&cs[p.chunk_ld + k]);
    }
  }
  __syncthreads();
  // totals of both weight kinds (each thread owns kChunksPerThread consecutive chunks)
  unsigned long long own[kChunksPerThread];
  {
    unsigned long long r4 = 0, p4 = 0;
#pragma unroll
    for (int q = 0; q < kChunksPerThread; ++q) {
      const int k = threadIdx.x * kChunksPerThread + q;
      r4 += k < nch ? s_cs[0][k] : 0ull;
      p4 += k < nch ? s_cs[1][k] : 0ull;
    }
    r4 = warp_sum_u64(r4);
    p4 = warp_sum_u64(p4);
    if (lane == 0) {
      s_red[0][warp] = r4;
      s_red[1][warp] = p4;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long tr = 0, tp = 0;
    for (int w = 0; w < kAccWarps; ++w) {
      tr += s_red[0][w];
      tp += s_red[1][w];
    }
    // residual after a rejection; plain p for the bonus, or when the residual has no mass
    const int mode = (qrow && tr > 0) ? 0 : 1;
    const unsigned long long tot = mode == 0 ? tr : tp;
    s_mode = mode;
    s_chunk = tot == 0 ? -1 : 0;
    if (tot != 0) {
      const unsigned long long U = static_cast<unsigned long long>(u_fin * 16777216.0f);
      const unsigned long long hi = __umul64hi(tot, U), lo = tot * U;
      s_T = (hi << 40) | (lo >> 24);
    }
    s_tok = -1;
    p.chunk_count[b] = 0;  // ready for the next call
  }
  __syncthreads();
  if (s_chunk >= 0) {
    // block-wide exclusive scan of the chosen chunk sums; the thread whose
    // range holds T names the chunk
    const unsigned long long* arr = s_cs[s_mode];
    unsigned long long local = 0;
#pragma unroll
    for (int q = 0; q < kChunksPerThread; ++q) {
      const int k = threadIdx.x * kChunksPerThread + q;
      own[q] = k < nch ? arr[k] : 0ull;
      local += own[q];
    }
    unsigned long long incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_scan[warp] = incl;
    __syncthreads();
    unsigned long long run = incl - local;
    for (int w = 0; w < warp; ++w) run += s_scan[w];
    const unsigned long long T = s_T;
#pragma unroll
    for (int q = 0; q < kChunksPerThread; ++q) {
      const int k = threadIdx.x * kChunksPerThread + q;
      if (k < nch && run <= T && T < run + own[q]) {
        s_chunk = k;
        s_base = run;
      }
      run += own[q];
    }
  }
  __syncthreads();
  SDV_TRACE_PHASE(kTrSmpChunk);
  if (s_chunk < 0) {
    if (threadIdx.x == 0) {
      set_status(p.status, SDV_ERR_BAD_INPUT);
      p.final_tokens[b] = -1;
    }
    return;
  }
  // within the chunk: each thread owns kPerThread consecutive entries
  const int mode = s_mode;
  const int j0 = s_chunk * kVChunk + threadIdx.x * kPerThread;
  unsigned long long mine = 0;
  for (int e = 0; e < kPerThread; ++e) {
    const int j = j0 + e;
    if (j < V) {
      const float x = src.x(rf, j, nml, s32);
      mine += fixed_of(mode == 0 ? residual_x(x, qrow[j]) : x);
    }
  }
  unsigned long long incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_scan[warp] = incl;
  __syncthreads();
  unsigned long long woff = 0;
  for (int w = 0; w < warp; ++w) woff += s_scan[w];
  const unsigned long long lo_b = s_base + woff + incl - mine, hi_b = s_base + woff + incl;
  const unsigned long long T = s_T;
  if (lo_b <= T && T < hi_b) {
    unsigned long long run = lo_b;
    for (int e = 0; e < kPerThread; ++e) {
      const int j = j0 + e;
      if (j >= V) break;
      const float x = src.x(rf, j, nml, s32);
      run += fixed_of(mode == 0 ? residual_x(x, qrow[j]) : x);
      if (run > T) {
        s_tok = j;
        break;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) p.final_tokens[b] = s_tok;
}

__global__ void probs_kernel(const float* z, const float2* row_stats, float* probs, int R, int V,
                             const int* status) {
  SDV_TRACE_SCOPE(kTrProbs);
  griddep_launch_dependents();
  SDV_GRIDDEP_WAIT();
  if (read_status(status) != 0) return;
  const long long n = (long long)R * V;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int r = static_cast<int>(i / V);
    const float2 st = row_stats[r];
    probs[i] = expf(z[i] - st.x) / st.y;
  }
}

// ---------------------------------------------------------------------------
// realignment (one block, one thread per slot)
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(kScanThreads) realign_kernel(const RealignParams p) {
  SDV_TRACE_SCOPE(kTrRealign);
  __shared__ int s_warp[80];
  __shared__ int s_err;
  __shared__ int s_need[kScanThreads], s_src[kScanThreads];
  __shared__ int s_amax;
  griddep_launch_dependents();
  SDV_GRIDDEP_WAIT();
  const int b = threadIdx.x;
  const bool slot = b < p.B;
  // the status word and the slot's inputs are loaded together (all inside
  // their buffers whatever the verdict); nothing is written before the check
  const int st = read_status(p.res.status);
  const int top = *p.num_free_in;
  int a = 0, L = 0, gam = 0, npg = 0, gc = 0, gl = 0;
  if (slot) {
    a = p.accepted[b];
    L = p.seq_lens[b];
    gam = p.draft_lens[b];
    npg = p.num_pages[b];
    if (p.gen_counts) gc = p.gen_counts[b];
    if (p.gen_limits) gl = p.gen_limits[b];
  }
  if (st != 0) return;
  if (b == 0) s_err = 0;
  __syncthreads();
  int newlen = 0, need = 0, fin = 0, gen = 0;
  if (slot) {
    // the accepted count and the final token may come from the caller
    // (sdv_realign): both are checked before anything is written
    int ft = 0;
    if (p.final_tokens) ft = p.final_tokens[b];
    if (a < 0 || a > gam || ft < 0 || ft >= p.vocab) {
      atomicCAS(&s_err, 0, SDV_ERR_BAD_INPUT);
      a = 0;  // keeps the scans below in range; nothing is written on an error
    }
    newlen = L + a + 1;
    if (p.gen_counts) gen = gc + a + 1;
    if (p.gen_counts && p.gen_limits) fin = gen >= gl ? 1 : 0;
    need = fin ? 0 : (newlen + p.gamma_max + 1 + p.page - 1) / p.page;
    if (need > p.max_pages) atomicCAS(&s_err, 0, SDV_ERR_CAPACITY);
  }
  const int surplus = slot ? max(0, npg - need) : 0;
  const int deficit = slot ? max(0, need - npg) : 0;
  int tot_emit, tot_s, tot_d, tot_live;
  const int eoff = block_exscan(slot ? a + 1 : 0, &tot_emit, s_warp);
  const int soff = block_exscan(surplus, &tot_s, s_warp);
  const int doff = block_exscan(deficit, &tot_d, s_warp);
  const int loff = block_exscan(slot && !fin ? 1 : 0, &tot_live, s_warp);
  if (b == 0 && tot_d > top + tot_s) atomicCAS(&s_err, 0, SDV_ERR_CAPACITY);
  // a free stack that would outgrow the pool means the caller's state is inconsistent
  if (b == 0 && (top < 0 || (long long)top + tot_s > p.pool_pages)) atomicCAS(&s_err, 0, SDV_ERR_BAD_INPUT);
  __syncthreads();
  const int err = s_err;
  const sdv_result& res = p.res;
  if (err) {
    // no output is touched; the free-stack count passes through unchanged
    if (b == 0) {
      set_status(res.status, err);
      *p.num_free_out = top;
    }
    return;
  }

  // per-slot outputs that do not depend on the page moves
  if (slot) {
    const int r0 = p.row_off[b];
    if (res.emitted_tokens) {
      if (p.tree_path) {
        const int* path = p.tree_path + (r0 - b);  // from the slot's draft offset
        for (int i = 0; i < a; ++i) res.emitted_tokens[eoff + i] = p.tokens[r0 + path[i]];
      } else {
        for (int i = 0; i < a; ++i) res.emitted_tokens[eoff + i] = p.tokens[r0 + 1 + i];
      }
      res.emitted_tokens[eoff + a] = p.final_tokens[b];
    }
    if (res.emitted_offsets) res.emitted_offsets[b] = eoff;
    if (res.new_seq_lens) res.new_seq_lens[b] = newlen;
    if (res.finished) res.finished[b] = fin;
    if (res.new_gen_counts && p.gen_counts) res.new_gen_counts[b] = gen;
    if (res.accepted && res.accepted != p.accepted) res.accepted[b] = a;
    if (res.accept_tested) {
      for (int k = 0; k < gam; ++k) {
        if (a >= k) atomicAdd(&res.accept_tested[k], 1);
        if (a > k) atomicAdd(&res.accept_accepted[k], 1);
      }
    }
  }
  if (b == 0 && res.emitted_offsets) res.emitted_offsets[p.B] = tot_emit;

  // token trees: the K/V of the accepted path's node at depth k moves from
  // cache slot L + node to slot L + k, one depth at a time.  A node's index is
  // at least its depth, so a move never reads a slot that a shallower move
  // wrote; all slots read lie below L + gamma + 1, inside pages the trim keeps.
  if (p.tree_path && p.kv_pool) {
    if (b == 0) s_amax = 0;
    __syncthreads();
    if (slot && a > 0) atomicMax(&s_amax, a);
    if (slot) s_need[b] = -1;
    __syncthreads();
    const int vec = p.head_dim / 8;       // 16-byte vectors of one head row
    const int per_row = p.n_kv * 2 * vec;  // vectors of one position's K and V
    const long long head_stride = (long long)p.page * p.head_dim;
    for (int k = 1; k <= s_amax; ++k) {
      // s_need[b]: this depth's source slot of sequence b, or -1
      if (slot) s_need[b] = k <= a ? L + p.tree_path[p.row_off[b] - b + k - 1] : -1;
      __syncthreads();
      for (int idx = threadIdx.x; idx < p.B * per_row; idx += blockDim.x) {
        const int sb = idx / per_row, e = idx - sb * per_row;
        const int src = s_need[sb];
        if (src < 0) continue;
        const int dst = p.seq_lens[sb] + k;
        if (src == dst) continue;
        const int hk = e / vec, v = e - hk * vec;  // (head, K or V), vector
        const int* pt = p.page_table + (long long)sb * p.max_pages;
        const long long so = ((long long)pt[src / p.page] * p.n_kv * 2 + hk) * head_stride +
                             (long long)(src % p.page) * p.head_dim + v * 8;
        const long long dof = ((long long)pt[dst / p.page] * p.n_kv * 2 + hk) * head_stride +
                              (long long)(dst % p.page) * p.head_dim + v * 8;
        *reinterpret_cast<uint4*>(p.kv_pool + dof) = *reinterpret_cast<const uint4*>(p.kv_pool + so);
      }
      __syncthreads();
    }
  }

  // push every slot's surplus tail pages above the old top, in slot order
  if (slot) {
    for (int j = 0; j < surplus; ++j) {
      const long long e = (long long)b * p.max_pages + need + j;
      p.free_pages[top + soff + j] = p.page_table[e];
      p.page_table[e] = -1;
    }
  }
  __syncthreads();
  // pop the missing pages from the top, in slot order
  if (slot) {
    for (int j = 0; j < deficit; ++j) {
      const int k = doff + j;
      p.page_table[(long long)b * p.max_pages + npg + j] = p.free_pages[top + tot_s - 1 - k];
    }
    p.num_pages[b] = need;
  }
  __syncthreads();
  if (b == 0) *p.num_free_out = top + tot_s - tot_d;

  // stable compaction of the surviving slots
  if (slot) s_need[b] = need;
  if (slot && !fin) {
    s_src[loff] = b;
    if (res.next_src) res.next_src[loff] = b;
    if (res.next_seq_lens) res.next_seq_lens[loff] = newlen;
    if (res.next_num_pages) res.next_num_pages[loff] = need;
    if (res.next_gen_counts && p.gen_counts) res.next_gen_counts[loff] = gen;
  }
  if (b == 0 && res.num_live) *res.num_live = tot_live;
  __syncthreads();
  if (res.next_page_table) {
    // a survivor's row holds its `need` pages, then -1 (the trim above cleared
    // the rest), so only the first `need` entries are read; eight in flight
    constexpr int kUnroll = 8;
    const long long n = (long long)tot_live * p.max_pages;
    for (long long base = threadIdx.x; base < n; base += (long long)blockDim.x * kUnroll) {
      int v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const long long idx = base + (long long)u * blockDim.x;
        v[u] = -1;
        if (idx < n) {
          const int dst = static_cast<int>(idx / p.max_pages);
          const int col = static_cast<int>(idx - (long long)dst * p.max_pages);
          const int src = s_src[dst];
          if (col < s_need[src]) v[u] = p.page_table[(long long)src * p.max_pages + col];
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const long long idx = base + (long long)u * blockDim.x;
        if (idx < n) res.next_page_table[idx] = v[u];
      }
    }
  }
}

}  // namespace

cudaError_t launch_prologue(const PrologueParams& p, cudaStream_t stream) {
  const int grid = p.emb ? (p.R + kRowsPerBlock - 1) / kRowsPerBlock + 1 : 1;
  return launch_pdl(prologue_kernel, dim3(grid), dim3(kScanThreads), 0, stream, p);
}

cudaError_t launch_rmsnorm(const float* x, const __nv_bfloat16* gain, __nv_bfloat16* h, long long lo_off, int R,
                           int H, float eps, const int* status, cudaStream_t stream) {
  return launch_pdl(rmsnorm_kernel, dim3(R), dim3(256), 0, stream, x, gain, h, lo_off, H, eps, status);
}

cudaError_t launch_join_planes(const __nv_bfloat16* hi, long long lo_off, float* out, long long n,
                               cudaStream_t stream) {
  const long long blocks = (n + 255) / 256;
  const int grid = static_cast<int>(blocks < 2048 ? blocks : 2048);
  return launch_pdl(join_planes_kernel, dim3(grid), dim3(256), 0, stream, hi, lo_off, out, n);
}

cudaError_t launch_split_planes(const float* x, __nv_bfloat16* out, long long lo_off, long long n,
                                cudaStream_t stream) {
  const long long blocks = (n + 255) / 256;
  const int grid = static_cast<int>(blocks < 2048 ? blocks : 2048);
  return launch_pdl(split_planes_kernel, dim3(grid), dim3(256), 0, stream, x, out, lo_off, n);
}

// Streaming multiprocessors of the current device (looked up once per device).
static int sms_of_current_device() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

cudaError_t launch_accept(const AcceptParams& p, bool from_logits, cudaStream_t stream) {
  // sampling: about four blocks per SM over the whole batch (what the
  // kernel's registers let an SM hold: one wave; eight and sixteen measured
  // slower, each block merging its slot's row statistics again), never more
  // blocks per slot than its vocabulary has chunks for (one warp per chunk)
  const int nch = (p.V + kVChunk - 1) / kVChunk;
  const int max_per_slot = (nch + kAccWarps - 1) / kAccWarps;
  const int want = 4 * sms_of_current_device() / p.B;  // rounded down: a second wave costs a block's time
  const dim3 grid(want < 1 ? 1 : (want > max_per_slot ? max_per_slot : want), p.B);
  cudaError_t e;
  if (from_logits) {
    // stochastic from logits: the tests run inside the sampling blocks
    if (!p.greedy && !p.tree_parents)
      return launch_pdl(sample_kernel<true, true>, grid, dim3(kAccThreads), 0, stream, p);
    if ((e = launch_pdl(accept_kernel<true>, dim3(p.B), dim3(kAccThreads), 0, stream, p)) != cudaSuccess) return e;
    return p.greedy ? cudaSuccess : launch_pdl(sample_kernel<true, false>, grid, dim3(kAccThreads), 0, stream, p);
  }
  if ((e = launch_pdl(accept_kernel<false>, dim3(p.B), dim3(kAccThreads), 0, stream, p)) != cudaSuccess) return e;
  return p.greedy ? cudaSuccess : launch_pdl(sample_kernel<false, false>, grid, dim3(kAccThreads), 0, stream, p);
}

int accept_chunks(int V) { return (V + kVChunk - 1) / kVChunk; }

cudaError_t launch_probs(const float* z, const float2* row_stats, float* probs, int R, int V, const int* status,
                         cudaStream_t stream) {
  const long long n = (long long)R * V;
  const long long blocks = (n + 255) / 256;
  const int grid = static_cast<int>(blocks < 4096 ? blocks : 4096);
  return launch_pdl(probs_kernel, dim3(grid), dim3(256), 0, stream, z, row_stats, probs, R, V, status);
}

// ---------------------------------------------------------------------------
// admission (one block, one thread per newcomer)
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(kScanThreads) admit_kernel(const AdmitParams p) {
  SDV_TRACE_SCOPE(kTrAdmit);
  __shared__ int s_warp[80];
  __shared__ int s_err;
  __shared__ int s_need[kScanThreads], s_off[kScanThreads];
  griddep_launch_dependents();
  SDV_GRIDDEP_WAIT();
  if (read_status(p.status) != 0) return;
  const sdv_admission& a = p.a;
  const int t = threadIdx.x;
  if (t == 0) s_err = 0;
  __syncthreads();
  if (t == 0 && a.num_live && *a.num_live != a.live) atomicCAS(&s_err, 0, SDV_ERR_BAD_INPUT);
  const bool mine = t < a.n;
  int ctx = 0, need = 0;
  if (mine) {
    ctx = a.ctx_lens[t];
    if (ctx < 0) atomicCAS(&s_err, 0, SDV_ERR_BAD_INPUT);
    need = (ctx + p.gamma_max + 1 + p.page - 1) / p.page;
    if (need > a.max_pages_per_seq) atomicCAS(&s_err, 0, SDV_ERR_CAPACITY);
  }
  int total;
  const int off = block_exscan(mine ? need : 0, &total, s_warp);
  const int top = *a.num_free;
  if (t == 0 && (total > top || top < 0)) atomicCAS(&s_err, 0, SDV_ERR_CAPACITY);
  if (mine) {
    s_need[t] = need;
    s_off[t] = off;
  }
  __syncthreads();
  if (s_err) {
    if (t == 0) set_status(p.status, s_err);
    return;
  }
  if (a.gen_limits_prev && a.next_src)
    for (int j = t; j < a.live; j += blockDim.x) a.gen_limits[j] = a.gen_limits_prev[a.next_src[j]];
  if (mine) {
    const int slot = a.live + t;
    a.seq_lens[slot] = ctx;
    a.num_pages[slot] = need;
    a.gen_counts[slot] = 0;
    a.gen_limits[slot] = a.out_lens[t];
  }
  // page-table rows of the newcomers, all threads over all entries
  const long long n = (long long)a.n * a.max_pages_per_seq;
  for (long long idx = t; idx < n; idx += blockDim.x) {
    const int j = static_cast<int>(idx / a.max_pages_per_seq);
    const int k = static_cast<int>(idx - (long long)j * a.max_pages_per_seq);
    a.page_table[(long long)(a.live + j) * a.max_pages_per_seq + k] =
        k < s_need[j] ? a.free_pages[top - 1 - (s_off[j] + k)] : -1;
  }
  __syncthreads();  // every pop read the old top before the height moves
  if (t == 0) *a.num_free = top - total;
}

cudaError_t launch_admit(const AdmitParams& p, cudaStream_t stream) {
  return launch_pdl(admit_kernel, dim3(1), dim3(kScanThreads), 0, stream, p);
}

cudaError_t launch_realign(const RealignParams& p, cudaStream_t stream) {
  return launch_pdl(realign_kernel, dim3(1), dim3(kScanThreads), 0, stream, p);
}

SDV_TRACE_UNIT(step_kernels)

}  // namespace sdv
