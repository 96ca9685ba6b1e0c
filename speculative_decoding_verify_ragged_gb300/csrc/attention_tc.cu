// Block-causal GQA attention on the 5th-generation tensor cores (head_dim 128,
// up to 48 query vectors per work item; a (sequence, KV head) with more --
// up to 64 -- comes as adjacent items of 32 from its first vector v0).
//
// Same work items, masking and outputs as the mma.sync kernel (attention.cu):
// row i of sequence b sees positions 0 .. L_b + i of its own paged cache
// ("Speculative Decoding and Batching Compete for the Same Compute Slack on
// RDNA4", section "What is the ragged tensor problem..."), and every byte of
// the cache is read once per step.  The cache read does not amortise over the
// batch, so the kernel must stream it at HBM speed; with the legacy MMA pipe
// the 16-32 query vectors of an item cannot keep up, so here:
//
//  * a KV block is 8 pages = 128 keys; two TMA producer warps land its K and
//    its V (key rows, 128-byte swizzle) in separate rings, three blocks each
//    with 16 query vectors per item (two K and three V with 32, two each with
//    48, where the Q and P buffers take the rest of shared memory);
//  * one thread issues S^T = K Q^T as tcgen05.mma with M = 128 keys and
//    N = twice the item's query vectors (16, 32 or 48): q's bf16 hi rows and lo
//    rows side by side, so each K tile is read once; the softmax adds the two
//    column halves (S double-buffered across blocks);
//  * eight softmax warps own the 128 key lanes, in two groups of four that each
//    take half of the query columns (two warps per SM sub-partition): they mask
//    (q comes pre-scaled to base-2 logits) and keep a per-query bound m, 8
//    above the largest logit seen when it last moved, that moves only when a
//    logit exceeds it (then O is rescaled in TMEM), so the weights
//    p = 2^(s - m) stay <= 1 and need no per-block reduction; they
//    write p as bf16 hi + lo planes (K-major, key columns; two buffers, so the
//    softmax of a block overlaps the PV of the one before) and keep per-lane
//    partial sums of p;
//  * the same thread issues O^T += V^T P^T per page (M = 128 head dims read
//    MN-major straight from the V rows, K = 16 keys, N = the hi and lo rows of
//    p side by side; the epilogue adds the two halves of O);
//  * at the end of an item the softmax warps read O (lane = head dim), sum
//    their partial row sums across lanes and write the normalised output as
//    bf16 hi + lo planes, or (max, sum, unnormalised output) partials that the
//    merge kernel of attention.cu combines for split sequences.
#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace sdv {

namespace {

using namespace tc;

constexpr int D = 128;
constexpr int TC_THREADS = 11 * kWarp;      // K producer, MMA, 2 x 4 softmax / epilogue warps, V producer
constexpr int SM_WARPS = 8;                  // softmax warps: two groups of four, one per half of the columns
constexpr int KEYS = 128;                    // keys per block (8 pages of 16)
constexpr int PAGES = KEYS / 16;
constexpr int HALF = KEYS * 128;             // one 64-dim half of K or V for 128 keys: 16 KB
constexpr int STAGE_BYTES = 2 * HALF;       // K or V of one block (2 halves): 32 KB
constexpr float kLazy = 8.f;                 // log2 headroom of the lazily moved bound over the logits
// the bound before a column's first visible key: finite, so that 2^(s - m)
// and 2^(m - m') need no special case (the first visible logit always moves
// it; a column with no visible key keeps l = 0 and weights 0)
constexpr float kNoMax = -1e30f;

template <int NQ>
struct TaCfg {
  // K and V rings, in blocks: a K slot is free once its QK^T is done, a V slot
  // only after the block's softmax and PV.  Per-role cycle counters showed
  // the softmax warps waiting on QK^T 43 % of the time and the MMA thread on
  // K data: with 16 query vectors three blocks each (R = 512 attention
  // 225 -> 213 us; two K and four V, or four K and two V, were slower)
  static constexpr int KS = NQ == 16 ? 3 : 2;
  static constexpr int VS = NQ == 48 ? 2 : 3;
  static constexpr int OFF_V = KS * STAGE_BYTES;
  // Q and P are B operands of 2 NQ rows: the NQ hi rows, then the NQ lo rows
  static constexpr int Q_HALF = 2 * NQ * 128;    // one 64-dim half of the 2 NQ Q rows
  static constexpr int P_HALF = 2 * NQ * 128;    // one 64-key half of the 2 NQ P rows
  static constexpr int P_BUF = 2 * P_HALF;
  static constexpr int OFF_Q = OFF_V + VS * STAGE_BYTES;
  static constexpr int Q_BUF = 2 * Q_HALF;      // one item's Q; two buffers (the next item's is written early)
  static constexpr int OFF_P = OFF_Q + 2 * Q_BUF;
  static constexpr int OFF_RED = OFF_P + 2 * P_BUF;             // two P buffers
  // per group and block parity: [4 quarters][NQ / 2] maxima or sums, 4 flags
  static constexpr int RED_BYTES = 2 * 2 * (4 * (NQ / 2) * 4 + 16) + 64;
  static constexpr int OFF_BAR = OFF_RED + RED_BYTES;
  static constexpr int NBAR = 2 * KS + 2 * VS + 2 * 2 + 2 * 2 + 2 * 2 + 2;  // k, v, s(2), p(2), q(2), o (full + empty)
  static constexpr int SMEM = 1024 + OFF_BAR + NBAR * 8 + 16;
  // S0, S1 and O, each 2 NQ columns (hi part, lo part)
  static constexpr int TMEM_COLS =
      6 * NQ <= 32 ? 32 : (6 * NQ <= 64 ? 64 : (6 * NQ <= 128 ? 128 : (6 * NQ <= 256 ? 256 : 512)));
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(NQ == 16 || NQ == 32 || NQ == 48, "query vectors per item");
};

// Shared-memory descriptor of a 128-byte-swizzled operand given its two
// strides: lbo between swizzle atoms along the contiguous (MN) dimension of an
// MN-major operand, sbo between 8-row groups.
__device__ __forceinline__ uint64_t desc_sw128_mn(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
               "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
               "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
               : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 8 consecutive 32-bit columns, one lane per thread of the warp.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// 2^x on the special-function unit, subnormal results flushed to zero: a
// softmax weight below 2^-126 of the bound changes no sum.
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Order-preserving float <-> int map, so that an integer warp max is a float max.
__device__ __forceinline__ int f2ord(float x) {
  const int i = __float_as_int(x);
  return i >= 0 ? i : i ^ 0x7FFFFFFF;
}
__device__ __forceinline__ float ord2f(int i) { return __int_as_float(i >= 0 ? i : i ^ 0x7FFFFFFF); }

// v0: the item's first query vector (items of one (slot, kv head) split by
// vectors when there are more than one item holds)
struct Item {
  int b, g, p0, p1, L, gamma, r0, chunks, v0;
};

__device__ __forceinline__ Item load_item(const AttnParams& p, int item) {
  const int4 a = p.items[2 * item], c = p.items[2 * item + 1];
  return Item{a.x, a.y & 0xFFFF, a.z, a.w, c.x, c.y, c.z, c.w, a.y >> 16};
}

template <int NQ>
__global__ void __launch_bounds__(TC_THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmKV, const AttnParams p) {
  SDV_TRACE_SCOPE(kTrAttention);
  using C = TaCfg<NQ>;
  extern __shared__ uint8_t smem_raw[];
  griddep_launch_dependents();

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* k_full = bar;
  uint64_t* k_empty = k_full + C::KS;
  uint64_t* v_full = k_empty + C::KS;
  uint64_t* v_empty = v_full + C::VS;
  uint64_t* s_full = v_empty + C::VS;  // [2]
  uint64_t* s_empty = s_full + 2;     // [2]
  uint64_t* p_full = s_empty + 2;    // [2]
  uint64_t* p_empty = p_full + 2;    // [2]
  uint64_t* q_full = p_empty + 2;   // [2]
  uint64_t* q_empty = q_full + 2;   // [2]
  uint64_t* o_full = q_empty + 2;
  uint64_t* o_empty = o_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + C::NBAR);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // stale ring contents must be finite: keys of partial blocks meet weight 0
  for (int i = threadIdx.x; i < C::OFF_Q / 16; i += TC_THREADS)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::KS; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < C::VS; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], SM_WARPS);  // one arrival per softmax warp
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&p_full[s], SM_WARPS);
      mbar_init(&p_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&q_full[s], SM_WARPS);
      mbar_init(&q_empty[s], 1);
    }
    mbar_init(o_full, 1);
    mbar_init(o_empty, SM_WARPS);
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_s0 = tmem, t_o = tmem + 4 * NQ;  // S buffers at columns [0, 4 NQ), O after them

  SDV_GRIDDEP_WAIT();
  const bool ok = read_status(p.status) == 0;
  const int total_items = ok ? p.sched[1] : 0;

  if (warp == 0 || warp == 10) {
    // ---------------- producers: warp 0 the K rows, warp 10 the V rows, 8 pages per slot ----------------
    const int kv = warp == 0 ? 0 : 1;
    const int NS = kv == 0 ? C::KS : C::VS;
    uint64_t* full = kv == 0 ? k_full : v_full;
    uint64_t* empty = kv == 0 ? k_empty : v_empty;
    uint8_t* ring = smem + (kv == 0 ? 0 : C::OFF_V);
    int stage = 0;
    uint32_t phase = 0;
    bool dead = false;
    for (int item = blockIdx.x; item < total_items && !dead; item += gridDim.x) {
      const Item it = load_item(p, item);
      // the lanes fetch the page indices of up to four blocks (32 pages) per round trip
      for (int base32 = it.p0; base32 < it.p1 && !dead; base32 += kWarp) {
        const int n32 = min(kWarp, it.p1 - base32);
        const int my_pg = lane < n32 ? p.page_table[(long long)it.b * p.max_pages + base32 + lane] : 0;
        for (int o = 0; o < n32 && !dead; o += PAGES) {
          const int n = min(PAGES, n32 - o);
          int okw = 1;
          if (lane == 0) {
            if (!mbar_wait(&empty[stage], phase ^ 1)) {
              set_status(p.status, SDV_ERR_TIMEOUT);
              okw = 0;
            } else {
              mbar_arrive_expect_tx(&full[stage], n * 2 * (16 * 128));
            }
          }
          okw = __shfl_sync(0xffffffffu, okw, 0);
          if (!okw) {
            dead = true;
            break;
          }
          uint8_t* dst = ring + stage * STAGE_BYTES;
          for (int j = 0; j < n; ++j) {
            const int pg = __shfl_sync(0xffffffffu, my_pg, o + j);
            if (lane == 0) {
#pragma unroll
              for (int h = 0; h < 2; ++h)
                tma_load_5d(dst + h * HALF + j * (16 * 128), &tmKV, &full[stage], h * 64, 0, kv, it.g, pg);
            }
          }
          if (++stage == NS) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
    // stay until every block has been consumed (no copy in flight at exit)
    if (lane == 0)
      for (int i = 0; i < NS && !dead; ++i) {
        if (!mbar_wait(&empty[stage], phase ^ 1)) {
          set_status(p.status, SDV_ERR_TIMEOUT);
          break;
        }
        if (++stage == NS) {
          stage = 0;
          phase ^= 1;
        }
      }
    return;
  }

  if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && total_items > 0) {
      // S^T[key, v] += K[key, :] . Q[v, :]: A = K rows (K-major), B = Q rows (K-major)
      constexpr uint32_t idesc_s = idesc_bf16(128, 2 * NQ);
      // O^T[d, v] += V^T[d, key] P^T[key, v]: A = V rows read MN-major, B = P rows (K-major over keys)
      constexpr uint32_t idesc_o = idesc_bf16(128, 2 * NQ) | (1u << 15);
      const uint32_t sm = smem_u32(smem);
      bool dead = false;
      auto wait = [&](uint64_t* b, uint32_t par) {
        if (!dead && !mbar_wait(b, par)) {
          set_status(p.status, SDV_ERR_TIMEOUT);
          dead = true;
        }
        tc_fence_after();
      };
      int ks = 0, vs = 0;
      uint32_t kph = 0, vph = 0;
      uint32_t sph[2] = {0, 0};
      int blk_total = 0;  // S and P buffers = running block count & 1
      int kitem = 0;      // items this CTA has started
      // PV of one block: 8 pages x (P hi, P lo)
      auto pv = [&](int n, bool first_block) {
        wait(&v_full[vs], vph);
        const uint32_t vbase = sm + C::OFF_V + vs * STAGE_BYTES;
        const uint32_t pbase = sm + C::OFF_P + (n & 1) * C::P_BUF;
#pragma unroll
        for (int j = 0; j < PAGES; ++j) {
          const uint64_t a = desc_sw128_mn(vbase + j * 2048, HALF, 1024);
          const uint64_t b = desc_sw128(pbase + (j >> 2) * C::P_HALF + (j & 3) * 32);
          umma_bf16(t_o, a, b, idesc_o, (first_block && j == 0) ? 0u : 1u);
        }
        umma_commit(&v_empty[vs]);
        if (++vs == C::VS) {
          vs = 0;
          vph ^= 1;
        }
      };
      for (int item = blockIdx.x; item < total_items && !dead; item += gridDim.x) {
        const Item it = load_item(p, item);
        const int nblk = (it.p1 - it.p0 + PAGES - 1) / PAGES;
        const int qb = kitem & 1;  // this item's Q buffer
        wait(&q_full[qb], (kitem >> 1) & 1);
        int prev_n = -1;
        for (int b = 0; b < nblk; ++b) {
          const int sb = blk_total & 1;
          wait(&k_full[ks], kph);
          wait(&s_empty[sb], sph[sb] ^ 1);
          const uint32_t kbase = sm + ks * STAGE_BYTES;
          const uint32_t qbase = sm + C::OFF_Q + qb * C::Q_BUF;
          const uint32_t d = t_s0 + sb * 2 * NQ;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t a = desc_sw128(kbase + (kk >> 2) * HALF + (kk & 3) * 32);
            const uint64_t bq = desc_sw128(qbase + (kk >> 2) * C::Q_HALF + (kk & 3) * 32);
            umma_bf16(d, a, bq, idesc_s, kk == 0 ? 0u : 1u);
          }
          umma_commit(&s_full[sb]);
          umma_commit(&k_empty[ks]);
          if (++ks == C::KS) {
            ks = 0;
            kph ^= 1;
          }
          if (b == nblk - 1) umma_commit(&q_empty[qb]);  // the item's last read of Q
          sph[sb] ^= 1;
          ++blk_total;
          if (b > 0) {
            wait(&p_full[prev_n & 1], (prev_n >> 1) & 1);
            if (b == 1 && kitem > 0) wait(o_empty, (kitem - 1) & 1);  // the previous item's O was read
            pv(prev_n, b == 1);
            umma_commit(&p_empty[prev_n & 1]);
          }
          prev_n = blk_total - 1;
        }
        // the last block's PV, then the item's O is complete
        wait(&p_full[prev_n & 1], (prev_n >> 1) & 1);
        if (nblk == 1 && kitem > 0) wait(o_empty, (kitem - 1) & 1);
        pv(prev_n, nblk == 1);
        umma_commit(&p_empty[prev_n & 1]);
        umma_commit(o_full);
        ++kitem;
      }
    }
    __syncwarp();
    named_sync(2, (1 + SM_WARPS) * kWarp);  // every tensor-memory read done
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS) : "memory");
    return;
  }

  // ---------------- softmax + epilogue: warps 2..9, two groups of four ----------------
  {
    constexpr int NH = NQ / 2;                   // query columns per group
    static_assert(NH % 8 == 0, "a group's first column is a multiple of 8 (the P rows' swizzle)");
    const int grp = (warp - 2) >> 2;             // columns [grp * NH, grp * NH + NH)
    const int quarter = warp & 3;                // TMEM lanes 32 * quarter .. + 31
    const int t = quarter * 32 + lane;           // key lane of S, head dim of O
    const int col0 = grp * NH;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    // [2 block parities][4][NH] maxima or sums, then 4 flags: consecutive blocks
    // use alternate halves, so no barrier is needed before the next block writes
    float* red2 = reinterpret_cast<float*>(smem + C::OFF_RED + grp * 2 * (4 * NH * 4 + 16));
    const int bar_id = 3 + grp;
    const int group = p.n_q / p.n_kv;
    const float scale = kLog2e / sqrtf(static_cast<float>(D));
    bool dead = false;
    auto wait = [&](uint64_t* b, uint32_t par) {
      if (!dead && !mbar_wait(b, par)) {
        set_status(p.status, SDV_ERR_TIMEOUT);
        dead = true;
      }
      tc_fence_after();
    };
    auto ld_cols = [&](uint32_t taddr, float (&v)[NH]) {
      if constexpr (NH == 24) {
        float a[16], c[8];
        tmem_ld16(taddr, a);
        tmem_ld8(taddr + 16, c);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = a[j];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[16 + j] = c[j];
      } else if constexpr (NH == 16) {
        tmem_ld16(taddr, v);
      } else {
        tmem_ld8(taddr, v);
      }
    };

    int nb = 0;     // blocks this CTA has processed
    int kitem = 0;  // items this CTA has processed
    // Q buffers alternate by item: item k + 1's Q rows are written at item
    // k's start (from registers loaded at the end of item k - 1, with item
    // records read two items ahead), so the MMA can start item k + 1's QK^T
    // while this group still finishes item k
    constexpr int QPT = NH * (D / 4) / 128;  // float4s of Q per thread
    static_assert(NH * (D / 4) % 128 == 0, "Q rows split evenly over the group");
    auto fetch_q = [&](const Item& iq, float4 (&dst)[QPT]) {
      const int nq = (iq.gamma + 1) * group - iq.v0;  // this item's vectors (NQ at most)
#pragma unroll
      for (int q = 0; q < QPT; ++q) {
        const int idx = t + q * 128;
        const int v = col0 + idx / (D / 4), ch = idx % (D / 4);
        dst[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (v < nq) {
          const int va = iq.v0 + v;
          const int i = va / group, h = iq.g * group + (va - i * group);
          dst[q] = *reinterpret_cast<const float4*>(p.q + ((long long)(iq.r0 + i) * p.n_q + h) * D + ch * 4);
        }
      }
    };
    auto store_q = [&](const float4 (&src)[QPT], int buf) {
      uint8_t* qdst = smem + C::OFF_Q + buf * C::Q_BUF;
#pragma unroll
      for (int q = 0; q < QPT; ++q) {
        const int idx = t + q * 128;
        const int v = col0 + idx / (D / 4), ch = idx % (D / 4);
        // q scaled by log2(e) / sqrt(D): the MMA yields base-2 logits
        uint2 hi, lo;
        split_bf16x2(src[q].x * scale, src[q].y * scale, hi.x, lo.x);
        split_bf16x2(src[q].z * scale, src[q].w * scale, hi.y, lo.y);
        const int off = (ch >> 4) * C::Q_HALF + v * 128 + ((((ch & 15) >> 1) ^ (v & 7)) << 4) + (ch & 1) * 8;
        *reinterpret_cast<uint2*>(qdst + off) = hi;
        *reinterpret_cast<uint2*>(qdst + NQ * 128 + off) = lo;  // lo rows follow the hi rows
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_full[buf]);
    };
    float4 qpre[QPT];
    Item it_cur{}, it_nxt{};
    if (blockIdx.x < total_items) {
      it_cur = load_item(p, blockIdx.x);
      fetch_q(it_cur, qpre);
      store_q(qpre, 0);
    }
    if (blockIdx.x + gridDim.x < total_items) {
      it_nxt = load_item(p, blockIdx.x + gridDim.x);
      fetch_q(it_nxt, qpre);
    }
    for (int item = blockIdx.x; item < total_items; item += gridDim.x, ++kitem) {
      const Item it = it_cur;
      const int nqv = (it.gamma + 1) * group - it.v0;  // this item's vectors, from v0
      const int nblk = (it.p1 - it.p0 + PAGES - 1) / PAGES;
      // vector va (row va / group of the draft block) sees the keys up to
      // L + va / group, i.e. key k when (k - L) * group <= va; columns from
      // nq_g on hold no vector.  In a token tree the ancestor sets decide the
      // keys L .. L + 63
      const bool tree = p.row_anc != nullptr;
      const int nq_g = nqv - col0, va0 = it.v0 + col0;

      // the next item's Q rows into the other buffer, once item k - 1's last
      // QK^T has read it; then the Q rows and the record of the item after it
      const int n1 = item + gridDim.x, n2 = n1 + gridDim.x;
      Item it_n2{};
      if (n2 < total_items) it_n2 = load_item(p, n2);
      if (n1 < total_items) {
        const int buf = (kitem + 1) & 1;
        if (kitem >= 1) wait(&q_empty[buf], ((kitem - 1) >> 1) & 1);
        store_q(qpre, buf);
      }

      float m[NH], l[NH];
#pragma unroll
      for (int j = 0; j < NH; ++j) {
        m[j] = kNoMax;
        l[j] = 0.f;
      }
      // this thread's P column: half of the key range, 16-byte chunk, byte within it
      const int p_half = t >> 6, p_chunk = (t & 63) >> 3, p_byte = (t & 7) * 2;
      for (int b = 0; b < nblk; ++b, ++nb) {
        const int sb = nb & 1;
        float* redb = red2 + sb * (4 * NH + 4);               // this block's half of the scratch
        int* flags = reinterpret_cast<int*>(redb + 4 * NH);  // [4]
        wait(&s_full[sb], (nb >> 1) & 1);
        float s[NH];
        {
          float s_lo[NH];
          ld_cols(t_s0 + lane_off + sb * 2 * NQ + col0, s);
          ld_cols(t_s0 + lane_off + sb * 2 * NQ + NQ + col0, s_lo);
#pragma unroll
          for (int j = 0; j < NH; ++j) s[j] += s_lo[j];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[sb]);
        // mask (block-causal; keys of pages past the item never count); s is in base 2 already
        const int page = it.p0 + b * PAGES + (t >> 4);
        const int key = page < it.p1 ? page * 16 + (t & 15) : 0x7FFFFFFF;
        // column j sees this key when j >= dk (and j < nq_g); keys past the item see no column
        constexpr int kNone = 0x7FFFFFFF, kAll = -0x7FFFFFFF;
        const int dk = page >= it.p1 ? kNone
                       : tree        ? (key <= it.L + 63 ? kAll : kNone)
                                     : (key - it.L) * group - va0;
        bool up = false;
        if (tree && key >= it.L && key <= it.L + 63) {
          // token tree, key L + d: visible to the columns whose node has node d
          // among its ancestors (or is node d)
          const int d = key - it.L;
#pragma unroll
          for (int j = 0; j < NH; ++j) {
            const bool in = col0 + j < nqv && ((p.row_anc[it.r0 + (it.v0 + col0 + j) / group] >> d) & 1ull);
            s[j] = in ? s[j] : -INFINITY;
            up |= s[j] > m[j];
          }
        } else if (dk <= 0) {
          // a key every column sees (the columns past the item's vectors have
          // zero q rows and nothing reads them: they are left unmasked)
#pragma unroll
          for (int j = 0; j < NH; ++j) up |= s[j] > m[j];
        } else {
#pragma unroll
          for (int j = 0; j < NH; ++j) {
            s[j] = j < nq_g && j >= dk ? s[j] : -INFINITY;
            up |= s[j] > m[j];
          }
        }
        // does any logit of the block exceed its bound m?
        const unsigned any_w = __ballot_sync(0xffffffffu, up);
        if (lane == 0) flags[quarter] = any_w != 0u;
        named_sync(bar_id, 128);
        const bool need = (flags[0] | flags[1] | flags[2] | flags[3]) != 0;
        bool rescale = false;
        float sc[NH];  // each column's rescale factor of O (every thread holds them all)
        if (need) {
#pragma unroll
          for (int j = 0; j < NH; ++j) {
            const int wm = __reduce_max_sync(0xffffffffu, f2ord(s[j]));
            if (lane == 0) redb[quarter * NH + j] = ord2f(wm);
          }
          named_sync(bar_id, 128);
#pragma unroll
          for (int j = 0; j < NH; ++j) {
            const float bm = fmaxf(fmaxf(redb[j], redb[NH + j]), fmaxf(redb[2 * NH + j], redb[3 * NH + j]));
            const float mn = fmaxf(m[j], bm + kLazy);
            const float av = exp2f(m[j] - mn);
            rescale |= av != 1.f;
            m[j] = mn;
            l[j] *= av;
            sc[j] = av;
          }
        }
#pragma unroll
        for (int j = 0; j < NH; ++j) {
          s[j] = ex2_ftz(s[j] - m[j]);  // the weight p <= 1, in place (0 for masked keys)
          l[j] += s[j];
        }
        // O is rescaled only once the previous block's PV has finished
        if (rescale && b > 0) {
          wait(&p_empty[(nb - 1) & 1], ((nb - 1) >> 1) & 1);
#pragma unroll
          for (int part = 0; part < 2; ++part) {  // the hi and the lo accumulator, 8 columns at a time
#pragma unroll
            for (int j0 = 0; j0 < NH; j0 += 8) {
              const uint32_t ta = t_o + lane_off + part * NQ + col0 + j0;
              float o[8];
              tmem_ld8(ta, o);
#pragma unroll
              for (int j = 0; j < 8; ++j) o[j] *= sc[j0 + j];
              tmem_st8(ta, o);
            }
          }
        }
        // this P buffer was last read by the PV of block nb - 2
        if (nb >= 2) wait(&p_empty[nb & 1], ((nb - 2) >> 1) & 1);
        {
          // P^T as bf16 hi + lo: row v, key column t (K-major over keys, 128-byte swizzle)
          // (col0 is a multiple of 8, so row col0 + j swizzles like row j)
          uint8_t* pbuf = smem + C::OFF_P + (nb & 1) * C::P_BUF + p_half * C::P_HALF + p_byte + col0 * 128;
          const int pc16 = p_chunk << 4;
#pragma unroll
          for (int j = 0; j < NH; j += 2) {  // two columns per packed conversion
            uint32_t h, lo;
            split_bf16x2(s[j], s[j + 1], h, lo);
            const int off0 = j * 128 + (pc16 ^ ((j & 7) << 4));
            const int off1 = (j + 1) * 128 + (pc16 ^ (((j + 1) & 7) << 4));
            *reinterpret_cast<uint16_t*>(pbuf + off0) = static_cast<uint16_t>(h);
            *reinterpret_cast<uint16_t*>(pbuf + off1) = static_cast<uint16_t>(h >> 16);
            *reinterpret_cast<uint16_t*>(pbuf + NQ * 128 + off0) = static_cast<uint16_t>(lo);  // lo rows follow
            *reinterpret_cast<uint16_t*>(pbuf + NQ * 128 + off1) = static_cast<uint16_t>(lo >> 16);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[nb & 1]);
      }

      // item k + 2's Q rows, in flight during this item's epilogue, written at the next item's start
      if (n2 < total_items) fetch_q(it_n2, qpre);
      it_cur = it_nxt;
      it_nxt = it_n2;

      // the item's O: lane = head dim t, this group's columns
      wait(o_full, kitem & 1);
      float o[NH];
      {
        float o_lo[NH];
        ld_cols(t_o + lane_off + col0, o);
        ld_cols(t_o + lane_off + NQ + col0, o_lo);
#pragma unroll
        for (int j = 0; j < NH; ++j) o[j] += o_lo[j];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_empty);
      // row sums: per-lane partial sums over the keys, summed over the 128 lanes
      // (in the half of the scratch the next block will use: its last readers,
      // two blocks back, have all passed the last block's barrier)
      float* redr = red2 + (nb & 1) * (4 * NH + 4);
#pragma unroll
      for (int j = 0; j < NH; ++j) {
        const float ws = warp_sum(l[j]);
        if (lane == 0) redr[quarter * NH + j] = ws;
      }
      named_sync(bar_id, 128);
#pragma unroll
      for (int j = 0; j < NH; ++j) l[j] = (redr[j] + redr[NH + j]) + (redr[2 * NH + j] + redr[3 * NH + j]);
      named_sync(bar_id, 128);
      if (!dead) {
        if (it.chunks == 1) {
#pragma unroll
          for (int j = 0; j < NH; ++j) {
            const int v = col0 + j;
            if (v < nqv) {
              const int va = it.v0 + v;
              const int i = va / group, h = it.g * group + (va - i * group);
              store_planes(p.out, p.out_lo_off, ((long long)(it.r0 + i) * p.n_q + h) * D + t, o[j] / l[j]);
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < NH; ++j) {
            const int v = col0 + j;
            if (v < nqv) {
              p.part_o[((long long)item * kAttnQMax + v) * D + t] = o[j];
              if (t == 0) p.part_ml[(long long)item * kAttnQMax + v] = make_float2(m[j], l[j]);
            }
          }
        }
      }
    }
    tc_fence_before();
    named_sync(2, (1 + SM_WARPS) * kWarp);  // let warp 1 free the tensor memory
  }
}

template <int NQ>
cudaError_t launch_nq(const CUtensorMap* kv_map, const AttnParams& p, int grid, cudaStream_t stream) {
  auto kern = attn_tc_kernel<NQ>;
  constexpr int smem = TaCfg<NQ>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(TC_THREADS), smem, stream, *kv_map, p);
}

}  // namespace

cudaError_t launch_attention_tc(int nq, const CUtensorMap* kv_map, const AttnParams& p, int grid, cudaStream_t stream) {
  if (nq == 16) return launch_nq<16>(kv_map, p, grid, stream);
  if (nq == 32) return launch_nq<32>(kv_map, p, grid, stream);
  if (nq == 48) return launch_nq<48>(kv_map, p, grid, stream);
  return cudaErrorInvalidValue;
}

SDV_TRACE_UNIT(attention_tc)

}  // namespace sdv
