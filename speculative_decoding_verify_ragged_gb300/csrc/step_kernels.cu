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

__global__ void __launch_bounds__(kScanThreads) prologue_kernel(const PrologueParams p) {
  __shared__ int s_warp[80];
  __shared__ int s_err;
  const int b = threadIdx.x;
  if (b == 0) {
    *p.status = 0;
    s_err = 0;
  }
  __syncthreads();
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
  int tot_r, tot_g;
  const int roff = block_exscan(slot ? gam + 1 : 0, &tot_r, s_warp);
  const int goff = block_exscan(slot ? gam : 0, &tot_g, s_warp);
  if (b == 0 && (tot_r != p.R || tot_g != p.G)) atomicCAS(&s_err, 0, SDV_ERR_BAD_INPUT);
  __syncthreads();
  if (s_err) {
    if (b == 0) set_status(p.status, s_err);
    return;
  }
  if (slot) {
    p.t.row_off[b] = roff;
    p.t.draft_off[b] = goff;
    for (int i = 0; i <= gam; ++i) {
      p.t.row_seq[roff + i] = b;
      p.t.row_pos[roff + i] = L + i;
    }
    const int used = (L + gam + 1 + p.page - 1) / p.page;
    for (int j = 0; j < used; ++j) {
      const int pg = p.page_table[(long long)b * p.max_pages + j];
      if (pg < 0 || pg >= p.pool_pages) {
        atomicCAS(&s_err, 0, SDV_ERR_PAGE_RANGE);
        break;
      }
    }
  }
  if (b == 0) {
    p.t.row_off[p.B] = tot_r;
    p.t.draft_off[p.B] = tot_g;
  }
  if (p.check_tokens) {
    for (int r = threadIdx.x; r < p.R; r += blockDim.x) {
      const int tk = p.tokens[r];
      if (tk < 0 || tk >= p.vocab) atomicCAS(&s_err, 0, SDV_ERR_BAD_INPUT);
    }
  }
  // attention schedule: chunks of pages sized so that items cover the GPU
  const int pages_b = slot ? (L + gam + 1 + p.page - 1) / p.page : 0;
  int tot_pages;
  block_exscan(pages_b, &tot_pages, s_warp);
  const long long units = (long long)tot_pages * p.n_kv;
  int chunk = static_cast<int>((units + p.target_items - 1) / p.target_items);
  chunk = max(chunk, 4);
  const int chunks_b = slot ? (pages_b + chunk - 1) / chunk : 0;
  int tot_items;
  const int ioff = block_exscan(chunks_b * p.n_kv, &tot_items, s_warp);
  if (slot) {
    p.t.chunks[b] = chunks_b;
    p.t.item_off[b] = ioff;
  }
  if (b == 0) {
    p.t.item_off[p.B] = tot_items;
    p.t.sched[0] = chunk;
    p.t.sched[1] = tot_items;
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

// h = x / sqrt(mean(x^2) + eps) * gain for one row; x fp32, h fp32 or bf16.
template <typename Out>
__device__ void norm_row(const float* x, const __nv_bfloat16* gain, Out* h, int H, float eps, float* s_red) {
  float ss = 0.f;
  for (int k = threadIdx.x * 4; k < H; k += blockDim.x * 4) {
    const float4 v = *reinterpret_cast<const float4*>(x + k);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = block_sum_256(ss, s_red);
  const float inv = 1.0f / sqrtf(ss / static_cast<float>(H) + eps);
  for (int k = threadIdx.x * 4; k < H; k += blockDim.x * 4) {
    const float4 v = *reinterpret_cast<const float4*>(x + k);
    const float y0 = v.x * inv * bf2f(gain[k]), y1 = v.y * inv * bf2f(gain[k + 1]);
    const float y2 = v.z * inv * bf2f(gain[k + 2]), y3 = v.w * inv * bf2f(gain[k + 3]);
    if constexpr (sizeof(Out) == 4) {
      *reinterpret_cast<float4*>(h + k) = make_float4(y0, y1, y2, y3);
    } else {
      uint2 w;
      w.x = pack_bf16x2(y0, y1);
      w.y = pack_bf16x2(y2, y3);
      *reinterpret_cast<uint2*>(h + k) = w;
    }
  }
}

struct EmbedParams {
  const int* tokens;
  const __nv_bfloat16* emb;
  const __nv_bfloat16* gain;
  float* x0;
  float* h;
  const int* row_pos;
  float* rope_cs;
  int H, head_dim;
  float eps;
  double log2_theta;
  const int* status;
};

__global__ void __launch_bounds__(256) embed_norm_kernel(const EmbedParams p) {
  __shared__ float s_red[32];
  if (read_status(p.status) != 0) return;
  const int r = blockIdx.x;
  const int tok = p.tokens[r];
  // the embedding row enters the fp32 residual stream
  const __nv_bfloat16* e = p.emb + (long long)tok * p.H;
  float* x0 = p.x0 + (long long)r * p.H;
  for (int k = threadIdx.x * 8; k < p.H; k += blockDim.x * 8) {
    const uint4 raw = *reinterpret_cast<const uint4*>(e + k);
    const __nv_bfloat16* v = reinterpret_cast<const __nv_bfloat16*>(&raw);
    *reinterpret_cast<float4*>(x0 + k) = make_float4(bf2f(v[0]), bf2f(v[1]), bf2f(v[2]), bf2f(v[3]));
    *reinterpret_cast<float4*>(x0 + k + 4) = make_float4(bf2f(v[4]), bf2f(v[5]), bf2f(v[6]), bf2f(v[7]));
  }
  __syncthreads();
  norm_row<float>(x0, p.gain, p.h + (long long)r * p.H, p.H, p.eps, s_red);
  // rotary table of this row: angle = pos * theta^(-2j/d), reduced mod 2 pi in double
  const int half = p.head_dim >> 1;
  const int pos = p.row_pos[r];
  for (int j = threadIdx.x; j < half; j += blockDim.x) {
    const double inv = exp2(-(2.0 * j / p.head_dim) * p.log2_theta);
    const double ang = static_cast<double>(pos) * inv;
    const double two_pi = 6.283185307179586476925286766559;
    const double red = ang - two_pi * rint(ang / two_pi);
    float sn, cs;
    sincosf(static_cast<float>(red), &sn, &cs);
    p.rope_cs[((long long)r * half + j) * 2] = cs;
    p.rope_cs[((long long)r * half + j) * 2 + 1] = sn;
  }
}

template <typename Out>
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float* x, const __nv_bfloat16* gain, Out* h, int H,
                                                      float eps, const int* status) {
  __shared__ float s_red[32];
  if (read_status(status) != 0) return;
  const int r = blockIdx.x;
  norm_row<Out>(x + (long long)r * H, gain, h + (long long)r * H, H, eps, s_red);
}

// ---------------------------------------------------------------------------
// acceptance + final-token sampling: one block per slot
// ---------------------------------------------------------------------------

constexpr int kAccThreads = 512;
constexpr int kAccWarps = kAccThreads / 32;
constexpr int kChunk = 1024;        // elements per chunk sum
constexpr int kMaxChunks = 512;     // vocab up to 524288
constexpr int kMaxRowsPerSlot = 64; // gamma_max + 1

template <bool FROM_LOGITS>
struct PSource {
  const float* base;  // logits or probabilities
  int V;
  __device__ __forceinline__ float p(int row, int j, float M, float S) const {
    if constexpr (FROM_LOGITS) {
      return expf(base[(long long)row * V + j] - M) / S;
    } else {
      return base[(long long)row * V + j];
    }
  }
};

template <bool FROM_LOGITS>
__device__ __forceinline__ unsigned long long weight_at(const PSource<FROM_LOGITS>& src, int row, float M, float S,
                                                        const float* qrow, int j) {
  float w = src.p(row, j, M, S);
  if (qrow) w = fmaxf(0.f, w - qrow[j]);
  return static_cast<unsigned long long>(w * 4294967296.0f);
}

template <bool FROM_LOGITS>
__global__ void __launch_bounds__(kAccThreads) accept_kernel(const AcceptParams p) {
  __shared__ unsigned long long s_csum[kMaxChunks];
  __shared__ float s_M[kMaxRowsPerSlot], s_S[kMaxRowsPerSlot];
  __shared__ float s_redm[kAccWarps], s_reds[kAccWarps];
  __shared__ int s_a, s_chunk, s_tok, s_resid;
  __shared__ unsigned long long s_T, s_base;
  if (read_status(p.status) != 0) return;
  if (threadIdx.x == 0) s_tok = -1;
  const int b = blockIdx.x;
  const int gam = p.draft_lens[b];
  const int r0 = p.row_off[b];
  const int g0 = p.draft_off[b];
  const int V = p.V;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  PSource<FROM_LOGITS> src{FROM_LOGITS ? p.z : p.probs, V};

  // softmax normaliser of every row of this slot from the LM head's tile statistics
  if constexpr (FROM_LOGITS) {
    for (int i = 0; i <= gam; ++i) {
      const int r = r0 + i;
      float M = -INFINITY, S = 0.f;
      for (int tt = threadIdx.x; tt < p.m_tiles; tt += kAccThreads) {
        const float2 st = p.tile_stats[(long long)tt * p.stats_ld + r];
        const float nm = fmaxf(M, st.x);
        S = S * exp2f((M - nm) * kLog2e) + st.y * exp2f((st.x - nm) * kLog2e);
        M = nm;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float oM = __shfl_xor_sync(0xffffffffu, M, o);
        const float oS = __shfl_xor_sync(0xffffffffu, S, o);
        const float nm = fmaxf(M, oM);
        S = (M == -INFINITY ? 0.f : S * exp2f((M - nm) * kLog2e)) +
            (oM == -INFINITY ? 0.f : oS * exp2f((oM - nm) * kLog2e));
        M = nm;
      }
      if (lane == 0) {
        s_redm[warp] = M;
        s_reds[warp] = S;
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        float MM = -INFINITY, SS = 0.f;
        for (int w = 0; w < kAccWarps; ++w) {
          const float nm = fmaxf(MM, s_redm[w]);
          SS = (MM == -INFINITY ? 0.f : SS * exp2f((MM - nm) * kLog2e)) +
               (s_redm[w] == -INFINITY ? 0.f : s_reds[w] * exp2f((s_redm[w] - nm) * kLog2e));
          MM = nm;
        }
        s_M[i] = MM;
        s_S[i] = SS;
        p.row_stats[r] = make_float2(MM, SS);
      }
      __syncthreads();
    }
  }

  // acceptance: first draft that fails u < min(1, p/q) ends the prefix
  if (threadIdx.x == 0) {
    int a = gam;
    for (int i = 0; i < gam; ++i) {
      const int x = p.tokens[r0 + i + 1];
      const float pi = src.p(r0 + i, x, FROM_LOGITS ? s_M[i] : 0.f, FROM_LOGITS ? s_S[i] : 1.f);
      const float qi = p.draft_probs[(long long)(g0 + i) * V + x];
      const float ui = p.uniforms[r0 + i];
      const bool ok = (pi >= qi && pi > 0.f) || (__fmul_rn(ui, qi) < pi);
      if (!ok) {
        a = i;
        break;
      }
    }
    s_a = a;
    s_resid = a < gam ? 1 : 0;
  }
  __syncthreads();
  const int a = s_a;
  const int rf = r0 + a;
  const float M = FROM_LOGITS ? s_M[a] : 0.f;
  const float S = FROM_LOGITS ? s_S[a] : 1.f;
  const int nch = (V + kChunk - 1) / kChunk;

  for (int attempt = 0; attempt < 2; ++attempt) {
    const float* qrow = s_resid ? p.draft_probs + (long long)(g0 + a) * V : nullptr;
    for (int c = warp; c < nch; c += kAccWarps) {
      unsigned long long acc = 0;
      for (int e = lane; e < kChunk; e += 32) {
        const int j = c * kChunk + e;
        if (j < V) acc += weight_at(src, rf, M, S, qrow, j);
      }
      acc = warp_sum_u64(acc);
      if (lane == 0) s_csum[c] = acc;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned long long tot = 0;
      for (int c = 0; c < nch; ++c) tot += s_csum[c];
      if (tot == 0 && s_resid) {
        s_resid = 0;  // max(0, p - q) has no mass: fall back to p
        s_chunk = -2;
      } else if (tot == 0) {
        s_chunk = -1;
      } else {
        const unsigned long long U = static_cast<unsigned long long>(p.uniforms[r0 + gam] * 16777216.0f);
        const unsigned long long hi = __umul64hi(tot, U), lo = tot * U;
        const unsigned long long T = (hi << 40) | (lo >> 24);
        unsigned long long cum = 0;
        int c = 0;
        while (c < nch - 1 && cum + s_csum[c] <= T) cum += s_csum[c++];
        s_chunk = c;
        s_T = T;
        s_base = cum;
      }
    }
    __syncthreads();
    if (s_chunk != -2) break;
  }

  if (s_chunk == -1) {
    if (threadIdx.x == 0) {
      set_status(p.status, SDV_ERR_BAD_INPUT);
      p.accepted[b] = a;
      p.final_tokens[b] = -1;
    }
    return;
  }
  if (warp == 0) {
    const float* qrow = s_resid ? p.draft_probs + (long long)(g0 + a) * V : nullptr;
    const int c = s_chunk;
    const unsigned long long T = s_T;
    const int j0 = c * kChunk + lane * 32;
    unsigned long long mine = 0;
    for (int e = 0; e < 32; ++e) {
      const int j = j0 + e;
      if (j < V) mine += weight_at(src, rf, M, S, qrow, j);
    }
    unsigned long long incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const unsigned long long excl = incl - mine;
    const unsigned long long lo_b = s_base + excl, hi_b = s_base + incl;
    if (lo_b <= T && T < hi_b) {
      unsigned long long run = lo_b;
      int pick = -1;
      for (int e = 0; e < 32; ++e) {
        const int j = j0 + e;
        if (j >= V) break;
        run += weight_at(src, rf, M, S, qrow, j);
        if (run > T) {
          pick = j;
          break;
        }
      }
      s_tok = pick;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    p.accepted[b] = a;
    p.final_tokens[b] = s_tok;
  }
}

__global__ void probs_kernel(const float* z, const float2* row_stats, float* probs, int R, int V,
                             const int* status) {
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
  __shared__ int s_warp[80];
  __shared__ int s_err;
  if (read_status(p.res.status) != 0) return;
  const int b = threadIdx.x;
  const bool slot = b < p.B;
  const int top = *p.num_free_in;
  if (b == 0) s_err = 0;
  __syncthreads();
  int a = 0, L = 0, gam = 0, npg = 0, newlen = 0, need = 0, fin = 0, gen = 0;
  if (slot) {
    a = p.accepted[b];
    L = p.seq_lens[b];
    gam = p.draft_lens[b];
    npg = p.num_pages[b];
    newlen = L + a + 1;
    if (p.gen_counts) gen = p.gen_counts[b] + a + 1;
    if (p.gen_counts && p.gen_limits) fin = gen >= p.gen_limits[b] ? 1 : 0;
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

  // per-slot outputs that do not depend on the page moves
  if (slot) {
    const int r0 = p.row_off[b];
    if (res.emitted_tokens) {
      for (int i = 0; i < a; ++i) res.emitted_tokens[eoff + i] = p.tokens[r0 + 1 + i];
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
  if (err) {
    if (b == 0) {
      set_status(res.status, err);
      *p.num_free_out = top;
    }
    return;
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
  if (slot && !fin) {
    if (res.next_src) res.next_src[loff] = b;
    if (res.next_seq_lens) res.next_seq_lens[loff] = newlen;
    if (res.next_num_pages) res.next_num_pages[loff] = need;
    if (res.next_gen_counts && p.gen_counts) res.next_gen_counts[loff] = gen;
  }
  if (b == 0 && res.num_live) *res.num_live = tot_live;
  __syncthreads();
  if (res.next_page_table && res.next_src) {
    const long long n = (long long)tot_live * p.max_pages;
    for (long long idx = threadIdx.x; idx < n; idx += blockDim.x) {
      const int dst = static_cast<int>(idx / p.max_pages);
      const int col = static_cast<int>(idx - (long long)dst * p.max_pages);
      res.next_page_table[idx] = p.page_table[(long long)res.next_src[dst] * p.max_pages + col];
    }
  }
}

}  // namespace

cudaError_t launch_prologue(const PrologueParams& p, cudaStream_t stream) {
  prologue_kernel<<<1, kScanThreads, 0, stream>>>(p);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_embed_norm_rope(const int* tokens, const __nv_bfloat16* emb, const __nv_bfloat16* gain,
                                   float* x0, float* h, const int* row_pos, float* rope_cs, int R, int H,
                                   int head_dim, float eps, float theta, const int* status, cudaStream_t stream) {
  EmbedParams e{tokens, emb, gain, x0, h, row_pos, rope_cs, H, head_dim, eps, log2(static_cast<double>(theta)), status};
  embed_norm_kernel<<<R, 256, 0, stream>>>(e);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const float* x, const __nv_bfloat16* gain, float* h_f32, __nv_bfloat16* h_bf16, int R,
                           int H, float eps, const int* status, cudaStream_t stream) {
  if (h_f32) rmsnorm_kernel<float><<<R, 256, 0, stream>>>(x, gain, h_f32, H, eps, status);
  else rmsnorm_kernel<__nv_bfloat16><<<R, 256, 0, stream>>>(x, gain, h_bf16, H, eps, status);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_accept(const AcceptParams& p, bool from_logits, cudaStream_t stream) {
  if (from_logits) accept_kernel<true><<<p.B, kAccThreads, 0, stream>>>(p);
  else accept_kernel<false><<<p.B, kAccThreads, 0, stream>>>(p);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_probs(const float* z, const float2* row_stats, float* probs, int R, int V, const int* status,
                         cudaStream_t stream) {
  const long long n = (long long)R * V;
  const long long blocks = (n + 255) / 256;
  const int grid = static_cast<int>(blocks < 4096 ? blocks : 4096);
  probs_kernel<<<grid, 256, 0, stream>>>(z, row_stats, probs, R, V, status);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_realign(const RealignParams& p, cudaStream_t stream) {
  realign_kernel<<<1, kScanThreads, 0, stream>>>(p);
  note_launch();
  return cudaGetLastError();
}

}  // namespace sdv
