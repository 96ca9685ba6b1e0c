// Block-causal GQA attention of the verify rows over each sequence's paged KV cache.
//
// Row i of sequence b sits at position L_b + i and attends to positions
// 0 .. L_b + i of its own sequence: the whole cached context plus the draft
// rows before it ("Speculative Decoding and Batching Compete for the Same
// Compute Slack on RDNA4", section "What is the ragged tensor problem...":
// every sequence keeps its own positions, masks and KV length).  Each
// sequence's cache is read once for all of its rows and all query heads that
// share a KV head, and that read does not amortise across the batch ("Why
// Static Batching Wastes an RX 9070 XT Agent Swarm", section "The catch is
// prefill, and it points back at admission"), so the kernel is bound by KV
// bytes:
//
//  * work item = (sequence, KV head, chunk of pages); a device-side schedule
//    sizes the chunks so that the items cover all SMs, whatever the mix of
//    context lengths (a batch of one long sequence and a swarm of 128 alike);
//  * a producer warp streams each (page, KV head) block -- 16 keys and 16
//    values of head_dim -- with 128-byte-swizzled TMA loads into a 16-stage
//    ring; seven consumer warps run QK^T and PV on bf16 mma.sync with an
//    online softmax in fp32.  The item's query vectors (draft rows x query
//    heads of the group, at most 48) form 1-3 tiles of 16; the warps split
//    as (query tile) x (key phase), each key phase taking every KS-th page,
//    so a 16-vector item still keeps seven warps busy, and the phases'
//    (max, sum, output) states are combined in shared memory at the end of
//    the item.  A warp waits only for the pages it reads and releases them
//    itself (the query-tile-0 warp of a page arrives for the warps that skip
//    it), so up to seven pages are in work while the rest of the ring fills;  q (fp32) and the softmax weights enter the MMAs as bf16 hi +
//    lo pairs, so the output keeps ~17 significant bits against the bf16
//    cache; the hi and lo products and even and odd k steps accumulate
//    separately, so no MMA waits on more than three others;
//  * items that cover a whole sequence write the output directly (as bf16 hi +
//    lo planes, the O projection's input); split sequences write (max, sum,
//    unnormalised output) partials that a merge kernel combines (log-sum-exp
//    in base 2).
#include "common.cuh"
#include "internal.h"

namespace sdv {

namespace {

constexpr int kConsumers = 7;
constexpr float kLazy = 8.f;   // log2 headroom of the lazily moved softmax reference  // + the producer: 256 threads, so up to 255 registers a thread
constexpr int kThreads = (kConsumers + 1) * kWarp;

template <int D>
struct ACfg {
  // pages in work (one per consumer warp) plus ~8 in flight from HBM
  static constexpr int STAGES = 16;
  static constexpr int BOX = 64 * 16 * 2;             // one 64-wide half of 16 rows: 2 KB
  static constexpr int HALVES = D / 64;
  static constexpr int PAGE_BYTES = 2 * HALVES * BOX;  // K and V of one (page, kv head)
  static constexpr int QLD = D + 8;                   // padded Q row (bf16 elements)
  static constexpr int Q_BYTES = 2 * kAttnQMax * QLD * 2;  // hi and lo tiles
  static constexpr int OREG = D / 2;                  // output accumulators per thread
  // per-warp softmax states for the key-phase combine: [warp][register][lane]
  static constexpr int COMB_BYTES = kConsumers * (OREG + 4) * kWarp * 4;
  static constexpr int SMEM = 1024 + STAGES * PAGE_BYTES + Q_BYTES + COMB_BYTES + 2 * STAGES * 8 + 64;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

struct Item {
  int b, g, p0, p1, L, gamma, r0, chunks;
};

// The prologue wrote one record per work item: no search, one round trip.
__device__ __forceinline__ Item load_item(const AttnParams& p, int item) {
  const int4 a = p.items[2 * item], c = p.items[2 * item + 1];
  Item it;
  it.b = a.x;
  it.g = a.y & 0xFFFF;  // the mma.sync kernel's items hold every vector (no part offset)
  it.p0 = a.z;
  it.p1 = a.w;
  it.L = c.x;
  it.gamma = c.y;
  it.r0 = c.z;
  it.chunks = c.w;
  return it;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_kernel(const __grid_constant__ CUtensorMap tmKV, const AttnParams p) {
  SDV_TRACE_SCOPE(kTrAttention);
  using C = ACfg<D>;
  constexpr int KK = D / 16;  // k16 steps over the head dimension
  constexpr int QT = kAttnQMax * ACfg<D>::QLD;  // elements of one Q tile
  constexpr int NF = D / 8;   // n8 fragments of the output
  extern __shared__ uint8_t smem_raw[];
  griddep_launch_dependents();
  SDV_GRIDDEP_WAIT();
  if (read_status(p.status) != 0) return;

  uint8_t* smem = align1024(smem_raw);
  __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(smem + C::STAGES * C::PAGE_BYTES);
  float* comb = reinterpret_cast<float*>(smem + C::STAGES * C::PAGE_BYTES + C::Q_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::PAGE_BYTES + C::Q_BYTES + C::COMB_BYTES);
  uint64_t* empty = full + C::STAGES;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers);
    }
    fence_barrier_init();
  }
  __syncthreads();

  const int total_items = p.sched[1];
  const int group = p.n_q / p.n_kv;

  if (warp == kConsumers) {
    // producer warp: the lanes fetch up to 32 page indices of the item at once,
    // lane 0 issues the TMA loads of those pages in order
    int stage = 0;
    uint32_t phase = 0;
    bool dead = false;
    for (int item = blockIdx.x; item < total_items && !dead; item += gridDim.x) {
      const Item it = load_item(p, item);
      for (int base = it.p0; base < it.p1 && !dead; base += kWarp) {
        const int n = min(kWarp, it.p1 - base);
        const int my_pg = lane < n ? p.page_table[(long long)it.b * p.max_pages + base + lane] : 0;
        for (int j = 0; j < n; ++j) {
          const int pg = __shfl_sync(0xffffffffu, my_pg, j);
          int ok = 1;
          if (lane == 0) {
            if (!mbar_wait(&empty[stage], phase ^ 1)) {
              set_status(p.status, SDV_ERR_TIMEOUT);
              ok = 0;
            } else {
              uint8_t* dst = smem + stage * C::PAGE_BYTES;
              mbar_arrive_expect_tx(&full[stage], C::PAGE_BYTES);
#pragma unroll
              for (int kv = 0; kv < 2; ++kv)
#pragma unroll
                for (int h = 0; h < C::HALVES; ++h)
                  tma_load_5d(dst + (kv * C::HALVES + h) * C::BOX, &tmKV, &full[stage], h * 64, 0, kv, it.g, pg);
            }
          }
          if (!__shfl_sync(0xffffffffu, ok, 0)) {
            dead = true;
            break;
          }
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
    // tail: wait until the consumers have released every stage
    if (lane == 0) {
      for (int i = 0; i < C::STAGES && !dead; ++i) {
        if (!mbar_wait(&empty[stage], phase ^ 1)) {
          set_status(p.status, SDV_ERR_TIMEOUT);
          break;
        }
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    return;
  }

  // ---------------- consumers ----------------
  // a timed-out wait marks the CTA dead (see the GEMM kernel): no early return
  bool dead = false;
  const int g8 = lane >> 2, t = lane & 3;
  const int mat = lane >> 3, rr = lane & 7;
  const float scale = kLog2e / sqrtf(static_cast<float>(D));
  int stage = 0;
  uint32_t phase = 0;

  for (int item = blockIdx.x; item < total_items; item += gridDim.x) {
    const Item it = load_item(p, item);
    const int nqv = (it.gamma + 1) * group;
    const int qtiles = (nqv + 15) >> 4;
    const int ks_n = kConsumers / qtiles;  // key phases
    const int qt = warp % qtiles, ks = warp / qtiles;
    const bool active = ks < ks_n;

    // Q tiles (hi, lo): query vector v = row i * group + head-in-group
    constexpr int CPR = D / 4;  // float4 per row
    for (int idx = threadIdx.x; idx < qtiles * 16 * CPR; idx += kConsumers * kWarp) {
      const int v = idx / CPR, ch = idx - v * CPR;
      float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
      if (v < nqv) {
        const int i = v / group, h = it.g * group + (v - (v / group) * group);
        val = *reinterpret_cast<const float4*>(p.q + ((long long)(it.r0 + i) * p.n_q + h) * D + ch * 4);
      }
      uint2 hi, lo;
      split_bf16x2(val.x, val.y, hi.x, lo.x);
      split_bf16x2(val.z, val.w, hi.y, lo.y);
      *reinterpret_cast<uint2*>(qs + v * C::QLD + ch * 4) = hi;
      *reinterpret_cast<uint2*>(qs + QT + v * C::QLD + ch * 4) = lo;
    }
    named_sync(1, kConsumers * kWarp);

    uint32_t qa[KK][4], ql[KK][4];
    if (active) {
#pragma unroll
      for (int kk = 0; kk < KK; ++kk) {
        const int row = qt * 16 + (mat & 1) * 8 + rr;
        const int col = kk * 16 + (mat >> 1) * 8;
        ldsm_x4(smem_u32(qs + row * C::QLD + col), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
        ldsm_x4(smem_u32(qs + QT + row * C::QLD + col), ql[kk][0], ql[kk][1], ql[kk][2], ql[kk][3]);
      }
    }
    // query positions of this thread's two rows
    const int v0 = qt * 16 + g8, v1 = v0 + 8;
    const int qpos0 = it.L + v0 / group, qpos1 = it.L + v1 / group;

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[NF][4];
#pragma unroll
    for (int nf = 0; nf < NF; ++nf) o[nf][0] = o[nf][1] = o[nf][2] = o[nf][3] = 0.f;

    for (int pi = it.p0; pi < it.p1; ++pi) {
      const bool mine = active && (pi - it.p0) % ks_n == ks;
      if (mine && !dead && !mbar_wait(&full[stage], phase)) {
        set_status(p.status, SDV_ERR_TIMEOUT);
        dead = true;
      }
      if (mine && !dead) {
        const uint32_t kbase = smem_u32(smem + stage * C::PAGE_BYTES);
        const uint32_t vbase = kbase + C::HALVES * C::BOX;
        // four independent accumulator sets: (hi, lo) x (even, odd k step)
        float sa[4][2][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int nf = 0; nf < 2; ++nf) sa[a][nf][0] = sa[a][nf][1] = sa[a][nf][2] = sa[a][nf][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KK; ++kk) {
          const int key = (mat >> 1) * 8 + rr;
          const int chunk = kk * 2 + (mat & 1);
          const uint32_t addr = kbase + (chunk >> 3) * C::BOX + key * 128 + (((chunk & 7) ^ rr) << 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(addr, b0, b1, b2, b3);
          const int par = kk & 1;
          mma_bf16(sa[par][0], qa[kk], b0, b1);
          mma_bf16(sa[par][1], qa[kk], b2, b3);
          mma_bf16(sa[2 + par][0], ql[kk], b0, b1);
          mma_bf16(sa[2 + par][1], ql[kk], b2, b3);
        }
        float s[2][4];
#pragma unroll
        for (int nf = 0; nf < 2; ++nf)
#pragma unroll
          for (int e = 0; e < 4; ++e) s[nf][e] = (sa[0][nf][e] + sa[1][nf][e]) + (sa[2][nf][e] + sa[3][nf][e]);
        // scale to base-2 logits and apply the block-causal mask; in a token
        // tree a key at L + d (d >= 0) counts for a row iff node d is the row's
        // node or one of its ancestors
        const int kp0 = pi * p.page;
        const bool tree_tail = p.row_anc != nullptr && kp0 + p.page > it.L;
        unsigned long long anc0 = 0ull, anc1 = 0ull;
        if (tree_tail) {
          if (v0 < nqv) anc0 = p.row_anc[it.r0 + v0 / group];
          if (v1 < nqv) anc1 = p.row_anc[it.r0 + v1 / group];
        }
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nf = 0; nf < 2; ++nf)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int kp = kp0 + nf * 8 + 2 * t + e;
            bool in0 = kp <= qpos0, in1 = kp <= qpos1;
            if (tree_tail) {
              // (padding rows keep the chain's mask: their lanes still vote on rescaling)
              const int d = kp - it.L;
              if (v0 < nqv) in0 = d < 0 || (d < 64 && ((anc0 >> d) & 1ull));
              if (v1 < nqv) in1 = d < 0 || (d < 64 && ((anc1 >> d) & 1ull));
            }
            s[nf][e] = in0 ? s[nf][e] * scale : -INFINITY;
            s[nf][2 + e] = in1 ? s[nf][2 + e] * scale : -INFINITY;
            mx0 = fmaxf(mx0, s[nf][e]);
            mx1 = fmaxf(mx1, s[nf][2 + e]);
          }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        // lazy rescaling: the reference maximum moves only when a logit
        // exceeds it by more than kLazy (so every weight stays <= 2^kLazy);
        // o and l always share the reference, so the result is unchanged
        if (__any_sync(0xffffffffu, mx0 > m0 + kLazy || mx1 > m1 + kLazy)) {
          const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
          const float a0 = exp2f(m0 - (n0 == -INFINITY ? 0.f : n0));
          const float a1 = exp2f(m1 - (n1 == -INFINITY ? 0.f : n1));
          m0 = n0;
          m1 = n1;
          l0 *= a0;
          l1 *= a1;
#pragma unroll
          for (int nf = 0; nf < NF; ++nf) {
            o[nf][0] *= a0;
            o[nf][1] *= a0;
            o[nf][2] *= a1;
            o[nf][3] *= a1;
          }
        }
        const float base0 = m0 == -INFINITY ? 0.f : m0;
        const float base1 = m1 == -INFINITY ? 0.f : m1;
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int nf = 0; nf < 2; ++nf)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            s[nf][e] = exp2f(s[nf][e] - base0);
            s[nf][2 + e] = exp2f(s[nf][2 + e] - base1);
            ps0 += s[nf][e];
            ps1 += s[nf][2 + e];
          }
        l0 += ps0;
        l1 += ps1;
        // P enters the PV product as a bf16 pair hi + lo (about 16 significant
        // bits): a single bf16 P would add ~0.1 % noise to every output
        uint32_t pa[4], pl[4];
        split_bf16x2(s[0][0], s[0][1], pa[0], pl[0]);
        split_bf16x2(s[0][2], s[0][3], pa[1], pl[1]);
        split_bf16x2(s[1][0], s[1][1], pa[2], pl[2]);
        split_bf16x2(s[1][2], s[1][3], pa[3], pl[3]);
#pragma unroll
        for (int nf = 0; nf < NF; nf += 2) {
          const int key = (mat & 1) * 8 + rr;
          const int chunk = nf + (mat >> 1);
          const uint32_t addr = vbase + (chunk >> 3) * C::BOX + key * 128 + (((chunk & 7) ^ rr) << 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(addr, b0, b1, b2, b3);
          mma_bf16(o[nf], pa, b0, b1);
          mma_bf16(o[nf + 1], pa, b2, b3);
          mma_bf16(o[nf], pl, b0, b1);
          mma_bf16(o[nf + 1], pl, b2, b3);
        }
      }
      // the page's readers release it: kConsumers arrivals in all, the
      // query-tile-0 reader standing in for the warps that do not read it
      __syncwarp();
      if (mine && lane == 0) mbar_arrive_count(&empty[stage], qt == 0 ? kConsumers - qtiles + 1 : 1);
      if (++stage == C::STAGES) {
        stage = 0;
        phase ^= 1;
      }
    }

    if (active) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
      l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    }
    // combine the key phases of each query tile: phase 0's warp sums the others'
    // states (in phase order) scaled to the common maximum
    if (ks_n > 1) {
      if (active && ks > 0) {
        float* dst = comb + (size_t)warp * (C::OREG + 4) * kWarp;
        dst[0 * kWarp + lane] = m0;
        dst[1 * kWarp + lane] = m1;
        dst[2 * kWarp + lane] = l0;
        dst[3 * kWarp + lane] = l1;
#pragma unroll
        for (int nf = 0; nf < NF; ++nf)
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[(4 + nf * 4 + e) * kWarp + lane] = o[nf][e];
      }
      named_sync(1, kConsumers * kWarp);
      if (active && ks == 0) {
        float M0 = m0, M1 = m1;
        for (int k = 1; k < ks_n; ++k) {
          const float* src = comb + (size_t)(k * qtiles + qt) * (C::OREG + 4) * kWarp;
          M0 = fmaxf(M0, src[0 * kWarp + lane]);
          M1 = fmaxf(M1, src[1 * kWarp + lane]);
        }
        const float B0 = M0 == -INFINITY ? 0.f : M0, B1 = M1 == -INFINITY ? 0.f : M1;
        const float w0 = exp2f(m0 - B0), w1 = exp2f(m1 - B1);
        l0 *= w0;
        l1 *= w1;
#pragma unroll
        for (int nf = 0; nf < NF; ++nf) {
          o[nf][0] *= w0;
          o[nf][1] *= w0;
          o[nf][2] *= w1;
          o[nf][3] *= w1;
        }
        for (int k = 1; k < ks_n; ++k) {
          const float* src = comb + (size_t)(k * qtiles + qt) * (C::OREG + 4) * kWarp;
          const float u0 = exp2f(src[0 * kWarp + lane] - B0), u1 = exp2f(src[1 * kWarp + lane] - B1);
          l0 += u0 * src[2 * kWarp + lane];
          l1 += u1 * src[3 * kWarp + lane];
#pragma unroll
          for (int nf = 0; nf < NF; ++nf) {
            o[nf][0] += u0 * src[(4 + nf * 4 + 0) * kWarp + lane];
            o[nf][1] += u0 * src[(4 + nf * 4 + 1) * kWarp + lane];
            o[nf][2] += u1 * src[(4 + nf * 4 + 2) * kWarp + lane];
            o[nf][3] += u1 * src[(4 + nf * 4 + 3) * kWarp + lane];
          }
        }
        m0 = M0;
        m1 = M1;
      }
    }

    if (active && ks == 0) {
      if (it.chunks == 1) {
        const float i0 = 1.f / l0, i1 = 1.f / l1;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int v = half ? v1 : v0;
          if (v < nqv) {
            const float inv = half ? i1 : i0;
            const int i = v / group, h = it.g * group + (v - (v / group) * group);
            const long long base = ((long long)(it.r0 + i) * p.n_q + h) * D;
#pragma unroll
            for (int nf = 0; nf < NF; ++nf) {
              const int d = nf * 8 + 2 * t;
              uint32_t hi, lo;
              split_bf16x2(o[nf][half * 2] * inv, o[nf][half * 2 + 1] * inv, hi, lo);
              *reinterpret_cast<uint32_t*>(p.out + base + d) = hi;
              *reinterpret_cast<uint32_t*>(p.out + p.out_lo_off + base + d) = lo;
            }
          }
        }
      } else {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int v = half ? v1 : v0;
          if (v < nqv) {
            float* dst = p.part_o + ((long long)item * kAttnQMax + v) * D;
#pragma unroll
            for (int nf = 0; nf < NF; ++nf) {
              const int d = nf * 8 + 2 * t;
              *reinterpret_cast<float2*>(dst + d) = make_float2(o[nf][half * 2], o[nf][half * 2 + 1]);
            }
            if (t == 0)
              p.part_ml[(long long)item * kAttnQMax + v] = make_float2(half ? m1 : m0, half ? l1 : l0);
          }
        }
      }
    }
    named_sync(1, kConsumers * kWarp);  // Q tile and combine buffer are rewritten by the next item
  }
}

// Merge of a split sequence's chunk partials, four consecutive head-dim
// elements of one (row, query head) per thread: one pass over the chunks in
// chunk order with a running maximum (the unnormalised output and the sum of
// weights are rescaled whenever the maximum moves), loads of eight chunks in
// flight at a time.
template <int D>
__global__ void __launch_bounds__(256) attn_merge_kernel(const AttnParams p, const int* row_seq, int R) {
  SDV_TRACE_SCOPE(kTrMerge);
  constexpr int DV = D / 4;
  griddep_launch_dependents();
  SDV_GRIDDEP_WAIT();
  // the status word and the prologue's split flag first: a step whose slots
  // all fit one item per (slot, kv head) leaves nothing to merge
  const int st = read_status(p.status);
  const int split = p.sched[2];
  if (st != 0 || split == 0) return;
  const int group = p.n_q / p.n_kv;
  const long long n = (long long)R * p.n_q * DV;
  for (long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x; gid < n;
       gid += (long long)gridDim.x * blockDim.x) {
    const int d4 = static_cast<int>(gid % DV);
    const int rh = static_cast<int>(gid / DV);
    const int r = rh / p.n_q, h = rh - (rh / p.n_q) * p.n_q;
    const int b = row_seq[r];
    const int chunks = p.chunks[b];
    if (chunks == 1) continue;
    const int i = r - p.row_off[b];
    const int g = h / group;
    int v = i * group + (h - g * group);
    // items split by query vectors: the part holding v, and v within it
    int parts = 1, part = 0;
    if (p.qsplit > 0) {
      parts = ((p.draft_lens[b] + 1) * group + p.qsplit - 1) / p.qsplit;
      part = v / p.qsplit;
      v -= part * p.qsplit;
    }
    const long long item0 = p.item_off[b] + ((long long)g * parts + part) * chunks;
    const float2* ml = p.part_ml + item0 * kAttnQMax + v;
    const float4* po = reinterpret_cast<const float4*>(p.part_o + (item0 * kAttnQMax + v) * D) + d4;
    constexpr long long kO4 = (long long)kAttnQMax * D / 4;  // float4 stride between chunks
    float M = -INFINITY, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < chunks; c0 += 8) {
      float2 m[8];
      float4 o[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (c0 + q < chunks) {
          m[q] = ml[(long long)(c0 + q) * kAttnQMax];
          o[q] = po[(long long)(c0 + q) * kO4];
        }
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (c0 + q < chunks && m[q].x != -INFINITY) {
          const float nm = fmaxf(M, m[q].x);
          const float a = M == -INFINITY ? 0.f : exp2f(M - nm);
          const float w = exp2f(m[q].x - nm);
          L = L * a + w * m[q].y;
          acc.x = acc.x * a + w * o[q].x;
          acc.y = acc.y * a + w * o[q].y;
          acc.z = acc.z * a + w * o[q].z;
          acc.w = acc.w * a + w * o[q].w;
          M = nm;
        }
      }
    }
    const float inv = 1.f / L;
    const long long base = ((long long)r * p.n_q + h) * D + d4 * 4;
    store_planes(p.out, p.out_lo_off, base, acc.x * inv);
    store_planes(p.out, p.out_lo_off, base + 1, acc.y * inv);
    store_planes(p.out, p.out_lo_off, base + 2, acc.z * inv);
    store_planes(p.out, p.out_lo_off, base + 3, acc.w * inv);
  }
}

// The merge's grid: one thread per (row, query head, 4 dims), at most four
// 256-thread blocks per SM (the rest by grid stride).
dim3 merge_grid(int head_dim, int R, int n_q) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 0;
  const long long n = (long long)R * n_q * (head_dim / 4);
  long long blocks = (n + 255) / 256;
  const long long cap = 4LL * sms;
  if (cap > 0 && blocks > cap) blocks = cap;
  return dim3(static_cast<unsigned>(blocks < 1 ? 1 : blocks));
}

template <int D>
cudaError_t launch_d(const CUtensorMap* kv_map, const AttnParams& p, int grid, int R, cudaStream_t stream,
                     const int* row_seq) {
  auto kern = attn_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, ACfg<D>::SMEM);
  if (e != cudaSuccess) return e;
  if ((e = launch_pdl(kern, dim3(grid), dim3(kThreads), ACfg<D>::SMEM, stream, *kv_map, p)) != cudaSuccess)
    return e;
  return launch_pdl(attn_merge_kernel<D>, merge_grid(D, R, p.n_q), dim3(256), 0, stream, p, row_seq, R);
}

}  // namespace

size_t attention_smem_bytes(int head_dim) { return head_dim == 64 ? ACfg<64>::SMEM : ACfg<128>::SMEM; }

cudaError_t launch_attention_merge(int head_dim, const AttnParams& p, int R, cudaStream_t stream, const int* row_seq) {
  const dim3 grid = merge_grid(head_dim, R, p.n_q);
  if (head_dim == 128) return launch_pdl(attn_merge_kernel<128>, grid, dim3(256), 0, stream, p, row_seq, R);
  if (head_dim == 64) return launch_pdl(attn_merge_kernel<64>, grid, dim3(256), 0, stream, p, row_seq, R);
  return cudaErrorInvalidValue;
}

cudaError_t launch_attention_impl(int head_dim, const CUtensorMap* kv_map, const AttnParams& p, int grid, int R,
                                  cudaStream_t stream, const int* row_seq) {
  if (head_dim == 128) return launch_d<128>(kv_map, p, grid, R, stream, row_seq);
  if (head_dim == 64) return launch_d<64>(kv_map, p, grid, R, stream, row_seq);
  return cudaErrorInvalidValue;
}

SDV_TRACE_UNIT(attention)

}  // namespace sdv
