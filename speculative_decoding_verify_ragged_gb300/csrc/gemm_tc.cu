// Weight-streaming GEMM on the 5th-generation tensor cores (tcgen05, TMEM
// accumulators): y[r, n] = sum_k x[r, k] W[n, k].
//
// Same work split and fused epilogues as the mma.sync kernel (gemm.cu), but
// the MMAs are single-thread tcgen05.mma instructions of M = 128 weight rows x
// N = NT activation rows x K = 16, reading both operands from shared memory
// (K-major, 128-byte swizzle, exactly the TMA tile layout) and accumulating in
// tensor memory.  Once the verify rows grow past a few dozen, the legacy
// mma.sync path (about 300 TFLOP/s on this GPU) cannot keep up with the weight
// stream; these instructions run at the full dense bf16 rate.
//
// Arithmetic intensity: a weight tile streamed against NT activation rows
// carries 2 * NT flops per weight byte pair, so at NT = 256 the weights alone
// ask 7.5 TB/s of the HBM at the tensor peak, and a second 256-row activation
// tile would stream the same weights again.  Past one tile, a group of cs
// CTAs therefore shares each weight tile, CTA r of the group multiplying it
// with its own activation tile tg * cs + r of about R / cs rows, so the
// weights cross HBM once.  The group's CTAs walk the same units at the same
// pace, and the first to ask for a weight line brings it into L2 for the
// others.  (A thread-block cluster sharing the tile by TMA multicast -- two
// CTAs each load one 64-row half into every CTA of the cluster, and a stage
// is refilled only once every CTA has released it -- measured the same; it
// stays selectable for A/B timing.)
//
// From 128 activation rows the CTAs work in pairs (a cluster of two, tcgen05
// cta_group::2): one MMA of M = 256 weight rows (128 in each CTA's shared
// memory) x N = NT activation rows (each CTA holding NT / 2 of them) writes
// each CTA's 128 rows of the product into its own tensor memory.  Per SM a
// k-block then moves 16 KB of weights and NT / 2 activation rows instead of NT
// -- at NT = 256 two thirds of the bytes for the same flops -- and the ring
// holds half again as many stages.  The first CTA of the pair issues the MMAs
// and owns the stage barriers: both CTAs' copies complete on its barriers,
// its commits free the stage and signal the accumulator in both CTAs, and the
// epilogue warps of both CTAs release an accumulator on its barrier.  Each
// CTA loads its activation rows of a stage with one copy per plane (a map of
// that box height exists for every multiple of 16 up to 256): copies of 16 or
// 32 rows measured as much as a third slower than the MMAs they feed.
//
// Warp roles (320 threads):
//  * warp 0: TMA producer (one lane) -- weight half-tiles and activation planes
//    into a multi-stage ring; weights are streamed before waiting for the
//    kernel that writes the activations;
//  * warp 1: allocates 2 x NT columns of tensor memory (two accumulators) and
//    one lane issues the MMAs; tcgen05.commit frees each stage when its MMAs
//    complete and signals each finished accumulator;
//  * warps 2-9: epilogue, two groups of four taking alternate 16-column
//    chunks -- tcgen05.ld the accumulator (lane = weight row), then the
//    stream-K partial/fixup and the fused epilogue shared with the mma.sync
//    kernel, while the MMAs fill the other accumulator.  (With one group the
//    LM head's epilogue took about as long per tile as the tile's MMAs.)
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "gemm_common.cuh"
#include "tcgen05.cuh"

namespace sdv {

namespace {

using namespace gemm;
using namespace tc;
constexpr int TC_THREADS = 10 * kWarp;
constexpr int EC = 16;           // accumulator columns per tcgen05.ld / epilogue chunk
constexpr int kMaxStages = 10;
constexpr int kMaxCluster = 8;   // portable cluster size
// staging row stride: eight lanes of a row reading columns sub + 8 i of four
// consecutive rows hit 32 different banks
constexpr int EPI_LD = BM + 8;
constexpr int EPI_BYTES = EC * EPI_LD * 4;
constexpr int kScaleRows = 256;  // rows of the per-CTA RMSNorm row-scale cache (gate/up)
// alignment slack + epilogue staging (one buffer per epilogue group) + barriers (full, empty, 2 x 2
// accumulator) + TMEM slot and flag + the row-scale cache
constexpr int FIXED_BYTES = 1024 + 2 * EPI_BYTES + (2 * kMaxStages + 4) * 8 + 16 + kScaleRows * 4;

// Bytes of one ring stage in one CTA: the CTA's 128 weight rows and its
// activation rows (all nt of them, or half in a CTA pair) per plane.
__host__ __device__ constexpr int tc_stage_bytes(int nt, int xp, bool pair = false) {
  return A_BYTES + xp * (pair ? nt / 2 : nt) * BK * 2;
}
__host__ __device__ constexpr int tc_stages(int nt, int xp, bool pair = false) {
  return (kSmemBudget - FIXED_BYTES) / tc_stage_bytes(nt, xp, pair) > kMaxStages
             ? kMaxStages
             : (kSmemBudget - FIXED_BYTES) / tc_stage_bytes(nt, xp, pair);
}
static_assert(tc_stages(256, 2) >= 2, "pipeline too shallow");

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// TMA tile load into the same shared-memory offset of every CTA in `mask`,
// each CTA's barrier at `bar`'s offset receiving the bytes.
__device__ __forceinline__ void tma_load_2d_mc(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                               uint16_t mask, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5, %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "h"(mask), "l"(policy)
      : "memory");
}

// Arrive on the barrier at `bar`'s offset in every CTA of `mask` once every
// tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void umma_commit_mc(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}

// ---- CTA pairs (tcgen05 cta_group::2) ----
// The address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
  return a;
}

// TMA tile load into this CTA's shared memory whose completion counts on the
// barrier at cluster address `bar` -- in either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d_pair_hint(void* dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                                      uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
      "[%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// Arrive on the barrier at cluster address `bar` (this CTA's or the peer's).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One MMA of the pair: M = 256 weight rows (128 from each CTA's shared
// memory, at the same offsets), N activation rows (the first half from this
// CTA, the second from the peer), accumulating into the same tensor-memory
// columns of both CTAs (each its own 128 rows).
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                               uint32_t acc) {
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

// Arrive on the barrier at `bar`'s offset in both CTAs of the pair once the
// pair's tcgen05 operations issued so far by this thread complete.
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}

__device__ __forceinline__ uint32_t tmem_columns(int nt) {
  uint32_t c = 32;
  while (c < static_cast<uint32_t>(2 * nt)) c <<= 1;
  return c;
}

// Unit u of the GEMM (weight tile, activation-tile group, k-block) and the
// cluster that owns it: cluster q of Q owns [q * T / Q, (q + 1) * T / Q).
__device__ __forceinline__ int cluster_of_unit(long long u, long long total, int Q) {
  return static_cast<int>(((u + 1) * Q - 1) / total);
}

template <int EPI, int XP, bool PAIR>
__global__ void __launch_bounds__(TC_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                   const __grid_constant__ CUtensorMap tmX, const GemmParams p) {
  SDV_TRACE_SCOPE(SDV_GEMM_SLOT(EPI, p));
  extern __shared__ uint8_t smem_raw[];
  griddep_launch_dependents();

  const int NT = p.nt, S = p.stages, cs = p.cs;
  const bool mc = !PAIR && p.multicast != 0;  // a cluster shares weight tiles by multicast (else through L2)
  const int STAGE = tc_stage_bytes(NT, XP, PAIR);
  const int NTC = PAIR ? NT / 2 : NT;  // activation rows this CTA loads per stage
  uint8_t* smem = align1024(smem_raw);
  float* epi = reinterpret_cast<float*>(smem + S * STAGE);  // [2 groups][EPI_BYTES]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * STAGE + 2 * EPI_BYTES);
  uint64_t* empty = full + kMaxStages;
  uint64_t* tfull = empty + kMaxStages;  // [2] accumulator ready
  uint64_t* tempty = tfull + 2;          // [2] accumulator drained
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* row_scale = reinterpret_cast<float*>(tmem_slot + 4);  // [kScaleRows]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA pairs: half 0 issues the pair's MMAs; the pairs form the groups
  const int half = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
  const int team = PAIR ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int rank = mc ? static_cast<int>(cluster_ctarank()) : team % cs;
  const int q = mc ? static_cast<int>(cluster_id_x()) : team / cs;
  const int Q = static_cast<int>(gridDim.x) / (PAIR ? 2 * cs : cs);
  const uint16_t everyone = static_cast<uint16_t>((1u << cs) - 1u);
  const uint32_t ncols = tmem_columns(NT);
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], mc ? cs : 1);  // one release per CTA of a multicast cluster
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      // one arrival per epilogue warp (of both CTAs of a pair: the issuer's
      // barrier is the one that counts)
      mbar_init(&tempty[b], PAIR ? 16 : 8);
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    // a pair allocates the same columns in both CTAs, one warp of each
    if constexpr (PAIR) {
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                   "r"(ncols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                   "r"(ncols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // every CTA's barriers exist before a peer's multicast, copy or arrival can land on them
  if (mc || PAIR) cluster_sync_all();
  const uint32_t tmem = *tmem_slot;
  // a pair's stage fills and accumulator releases count on the issuing CTA's barriers
  const uint32_t lead_full = PAIR ? cluster_addr(full, 0) : 0u;
  const uint32_t lead_tempty = PAIR ? cluster_addr(tempty, 0) : 0u;

  // units: (weight tile -- of a pair: 256 rows --, activation group, k-block)
  const int m_units = PAIR ? (p.m_tiles + 1) / 2 : p.m_tiles;
  const long long total = (long long)m_units * p.n_groups * p.kb;
  const long long u_begin = (long long)q * total / Q;
  const long long u_end = (long long)(q + 1) * total / Q;
  const int first_tg = static_cast<int>(u_begin / p.kb);  // first (weight tile, group) of this cluster

  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const int my_units = static_cast<int>(u_end - u_begin);
      const int pre = my_units < S ? my_units : S;
      struct Cursor {
        int tg, k, tm, grp;
      };
      auto start_at = [&](long long u) {
        Cursor cu;
        cu.tg = static_cast<int>(u / p.kb);
        cu.k = static_cast<int>(u - (long long)cu.tg * p.kb);
        cu.tm = cu.tg / p.n_groups;
        cu.grp = cu.tg - cu.tm * p.n_groups;
        return cu;
      };
      auto advance = [&](Cursor& cu) {
        if (++cu.k == p.kb) {
          cu.k = 0;
          ++cu.tg;
          if (++cu.grp == p.n_groups) {
            cu.grp = 0;
            ++cu.tm;
          }
        }
      };
      auto weights = [&](const Cursor& cu, int stage) {
        const int tmc = PAIR ? 2 * cu.tm + half : cu.tm;  // this CTA's 128-row weight tile
        const int rowA0 = EPI == EPI_SWIGLU ? tmc * 64 : tmc * BM;
        const int rowA1 = EPI == EPI_SWIGLU ? tmc * 64 : tmc * BM + 64;
        uint8_t* sa = smem + stage * STAGE;
        if constexpr (PAIR) {
          const uint32_t bar = lead_full + 8u * stage;
          if (cs == 1) {
            tma_load_2d_pair_hint(sa, &tmA0, bar, cu.k * BK, rowA0, pol);
            tma_load_2d_pair_hint(sa + A_BYTES / 2, &tmA1, bar, cu.k * BK, rowA1, pol);
          } else {
            tma_load_2d_pair(sa, &tmA0, bar, cu.k * BK, rowA0);
            tma_load_2d_pair(sa + A_BYTES / 2, &tmA1, bar, cu.k * BK, rowA1);
          }
        } else if (cs == 1) {
          tma_load_2d_hint(sa, &tmA0, &full[stage], cu.k * BK, rowA0, pol);
          tma_load_2d_hint(sa + A_BYTES / 2, &tmA1, &full[stage], cu.k * BK, rowA1, pol);
        } else if (!mc) {
          // the group's CTAs read the same weight tile at about the same time:
          // the first brings it into L2 (normal priority), the others hit there
          tma_load_2d(sa, &tmA0, &full[stage], cu.k * BK, rowA0);
          tma_load_2d(sa + A_BYTES / 2, &tmA1, &full[stage], cu.k * BK, rowA1);
        } else if (rank == 0) {
          tma_load_2d_mc(sa, &tmA0, &full[stage], cu.k * BK, rowA0, everyone, pol);
        } else if (rank == 1) {
          tma_load_2d_mc(sa + A_BYTES / 2, &tmA1, &full[stage], cu.k * BK, rowA1, everyone, pol);
        }
      };
      auto acts = [&](const Cursor& cu, int stage) {
        uint8_t* sb = smem + stage * STAGE + A_BYTES;
        // a pair's first CTA loads the first half of the activation tile
        const int row0 = (cu.grp * cs + rank) * NT + half * NTC;
        for (int b = 0; b < NTC; b += p.x_box) {
          if constexpr (PAIR) {
            const uint32_t bar = lead_full + 8u * stage;
            tma_load_2d_pair(sb + b * 128, &tmX, bar, cu.k * BK, row0 + b);
            if constexpr (XP == 2) tma_load_2d_pair(sb + (NTC + b) * 128, &tmX, bar, cu.k * BK, p.x_lo_row + row0 + b);
          } else {
            tma_load_2d(sb + b * 128, &tmX, &full[stage], cu.k * BK, row0 + b);
            if constexpr (XP == 2)
              tma_load_2d(sb + (NTC + b) * 128, &tmX, &full[stage], cu.k * BK, p.x_lo_row + row0 + b);
          }
        }
      };
      // the issuing CTA's barrier expects the bytes of both CTAs of a pair (a
      // peer's copy may land before the expectation: the barrier's pending
      // arrival keeps the phase open until then)
      const bool lead = !PAIR || half == 0;
      const uint32_t mult = PAIR ? 2u : 1u;
      Cursor cw = start_at(u_begin);
      for (int j = 0; j < pre; ++j) {
        if (lead) mbar_expect_tx(&full[j], mult * A_BYTES);
        weights(cw, j);
        advance(cw);
      }
      SDV_GRIDDEP_WAIT();
      if (read_status(p.status) != 0) {
        // the weight copies land before anyone leaves (a peer's are counted
        // on the issuer's barriers; the final cluster barrier holds it)
        if (lead) {
          for (int j = 0; j < pre; ++j) mbar_arrive(&full[j]);
          for (int j = 0; j < pre; ++j) mbar_wait(&full[j], 0);
        }
      } else {
        Cursor ca = start_at(u_begin);
        for (int j = 0; j < pre; ++j) {
          if (lead) mbar_arrive_expect_tx(&full[j], mult * (STAGE - A_BYTES));
          acts(ca, j);
          advance(ca);
        }
        int stage = pre % S;
        uint32_t phase = pre == S ? 1u : 0u;
        bool dead = false;
        for (int j = pre; j < my_units; ++j) {
          // every CTA of the cluster has released this stage
          if (!mbar_wait(&empty[stage], phase ^ 1)) {
            set_status(p.status, SDV_ERR_TIMEOUT);
            dead = true;
            break;
          }
          if (lead) mbar_arrive_expect_tx(&full[stage], mult * STAGE);
          weights(cw, stage);
          acts(cw, stage);
          advance(cw);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
        // stay until the MMAs of the whole cluster have released every stage
        // (no copy in flight and no release still to arrive at exit)
        for (int i = 0; i < S && !dead; ++i) {
          if (!mbar_wait(&empty[stage], phase ^ 1)) {
            set_status(p.status, SDV_ERR_TIMEOUT);
            break;
          }
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (a pair's first CTA) ----------------
    if (lane == 0 && half == 0) {
      SDV_GRIDDEP_WAIT();
      if (read_status(p.status) == 0) {
        const uint32_t idesc = idesc_bf16(PAIR ? 2 * BM : BM, NT);
        bool dead = false;
        int stage = 0;
        uint32_t phase = 0;
        int pc = 0;  // piece index
        for (long long u = u_begin; u < u_end; ++pc) {
          const int tg = static_cast<int>(u / p.kb);
          const int k0 = static_cast<int>(u - (long long)tg * p.kb);
          const int k1 = static_cast<int>(min((long long)p.kb, k0 + (u_end - u)));
          const int buf = pc & 1;
          if (!dead && !mbar_wait(&tempty[buf], ((pc >> 1) & 1) ^ 1)) {
            set_status(p.status, SDV_ERR_TIMEOUT);
            dead = true;
          }
          tc_fence_after();
          const uint32_t d = tmem + buf * NT;
          for (int k = k0; k < k1; ++k) {
            if (!dead && !mbar_wait(&full[stage], phase)) {
              set_status(p.status, SDV_ERR_TIMEOUT);
              dead = true;
            }
            tc_fence_after();
            const uint32_t a_base = smem_u32(smem + stage * STAGE);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t a = desc_sw128(a_base + kk * 32);
#pragma unroll
              for (int pl = 0; pl < XP; ++pl) {
                const uint64_t b = desc_sw128(a_base + A_BYTES + pl * (NTC * 128) + kk * 32);
                if constexpr (PAIR) umma_bf16_pair(d, a, b, idesc, (k > k0 || kk > 0 || pl > 0) ? 1u : 0u);
                else umma_bf16(d, a, b, idesc, (k > k0 || kk > 0 || pl > 0) ? 1u : 0u);
              }
            }
            // frees the stage, in every CTA of the cluster, once these MMAs have read it
            if constexpr (PAIR) umma_commit_pair(&empty[stage]);
            else if (mc) umma_commit_mc(&empty[stage], everyone);
            else umma_commit(&empty[stage]);
            if (++stage == S) {
              stage = 0;
              phase ^= 1;
            }
          }
          // accumulator complete (in both CTAs of a pair)
          if constexpr (PAIR) umma_commit_pair(&tfull[buf]);
          else umma_commit(&tfull[buf]);
          u += k1 - k0;
        }
      }
    }
  } else {
    // ---------------- epilogue warps 2..9 ----------------
    // two groups of four (warps 2-5 and 6-9), each covering the 128 TMEM lanes
    // (a warp reaches lanes 32 * (warp % 4) .. +31) and taking alternate
    // 16-column chunks of every accumulator, with its own staging buffer and
    // named barrier, so that one group's loads and stores overlap the other's
    const int eg = (warp - 2) >> 2;
    const int ebar = 1 + eg;
    float* epi_g = epi + eg * (EPI_BYTES / 4);
    const int quarter = warp & 3;          // TMEM lanes 32*quarter .. +31
    const int m = quarter * 32 + lane;     // weight row within the tile
    SDV_GRIDDEP_WAIT();
    // gate/up after the FFN pre-norm: every row's 1 / rms, reduced once from
    // the O projection's partial sums of x^2 (lanes over rows, so each load
    // is one coalesced line; the first group's four warps take every fourth
    // partial and meet in a fixed order) while the first tile's MMAs run; the
    // rows are this CTA's activation tile (or all rows, when one CTA walks
    // several tiles of at most kScaleRows rows in total)
    int rs_base = 0;
    bool have_scale = false;
    if constexpr (EPI == EPI_SWIGLU) {
      int nrs = 0;
      if (p.epi.sq_in && read_status(p.status) == 0) {
        if (p.n_groups == 1) {
          rs_base = rank * NT;
          nrs = min(NT, p.R - rs_base);
        } else if (p.R <= kScaleRows) {
          nrs = p.R;
        }
      }
      have_scale = nrs > 0;
      const EpiParams& e = p.epi;
      for (int rb = 0; eg == 0 && rb < nrs; rb += kWarp) {
        const int r = rb + lane;
        float acc = 0.f;
        if (r < nrs) {
          constexpr int U = 8;
          for (int q0 = quarter; q0 < e.sq_parts; q0 += 4 * U) {
            float w[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
              const int qq = q0 + 4 * u;
              w[u] = qq < e.sq_parts ? e.sq_in[(long long)qq * e.sq_ld + rs_base + r] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) acc += w[u];
          }
        }
        epi[quarter * kWarp + lane] = acc;
        named_sync(1, 4 * kWarp);
        if (quarter == 0 && r < nrs) {
          const float ss = ((epi[lane] + epi[kWarp + lane]) + epi[2 * kWarp + lane]) + epi[3 * kWarp + lane];
          const float sc = 1.0f / sqrtf(ss * e.sq_inv_n + e.sq_eps);
          row_scale[r] = sc;
          // the fixup kernel reads them back (every CTA of a group writes the same values)
          if (e.rscale) e.rscale[rs_base + r] = sc;
        }
        named_sync(1, 4 * kWarp);
      }
      named_sync(3, 8 * kWarp);  // the scales are ready for both groups
    }
    const float* rs = have_scale ? row_scale : nullptr;
    if (read_status(p.status) == 0) {
      constexpr int LD = EPI_LD;
      bool dead = false;
      int pc = 0;
      for (long long u = u_begin; u < u_end; ++pc) {
        const int tg = static_cast<int>(u / p.kb);
        const int k0 = static_cast<int>(u - (long long)tg * p.kb);
        const int k1 = static_cast<int>(min((long long)p.kb, k0 + (u_end - u)));
        const int tmu = tg / p.n_groups;
        const int tn = (tg - tmu * p.n_groups) * cs + rank;
        const int tm = PAIR ? 2 * tmu + half : tmu;  // this CTA's 128-row weight tile
        const int tile = tm * p.n_tiles + tn;
        const int buf = pc & 1;
        if (!dead && !mbar_wait(&tfull[buf], (pc >> 1) & 1)) {
          set_status(p.status, SDV_ERR_TIMEOUT);
          dead = true;
        }
        tc_fence_after();
        const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + buf * NT;
        const int rows = min(NT, p.R - tn * NT);

        // accumulator columns past the last activation row are never read
        const int cols = (rows + EC - 1) / EC * EC;
        // releases the accumulator (a pair's on the issuing CTA's barrier)
        auto release = [&]() {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if constexpr (PAIR) mbar_arrive_cluster(lead_tempty + 8u * buf);
            else mbar_arrive(&tempty[buf]);
          }
        };
        if (PAIR && tm >= p.m_tiles) {
          // the second half of a pair past the last weight tile: nothing to store
          release();
        } else if (k0 == 0 && k1 == p.kb) {
          // whole tile in this CTA: epilogue straight from tensor memory, this
          // group's chunks eg, eg + 2, ...; a warp releases the accumulator
          // after its last read of it
          bool released = false;
          for (int c0 = eg * EC; c0 < cols; c0 += 2 * EC) {
            float v[16];
            tmem_ld16(t_row + c0, v);
            if (c0 + 2 * EC >= cols) {
              release();
              released = true;
            }
#pragma unroll
            for (int n = 0; n < EC; ++n) epi_g[n * LD + m] = v[n];
            named_sync(ebar, 4 * kWarp);
            epilogue_rows<EPI, LD>(p, epi_g, tm, tn * NT + c0, min(EC, rows - c0), m, rs, rs_base, ebar);
            named_sync(ebar, 4 * kWarp);
          }
          if (!released) release();
        } else {
          // tile cut between clusters: store this piece, the fixup sums them in cluster order
          const int my_slot = 2 * ((q * cs + rank) * (PAIR ? 2 : 1) + half) + (tg == first_tg ? 0 : 1);
          float* mine = p.partials + (size_t)my_slot * BM * NT;
          for (int c0 = eg * EC; c0 < cols; c0 += 2 * EC) {
            float v[16];
            tmem_ld16(t_row + c0, v);
            tc_store_part16(mine, c0, m, v);
          }
          release();
          if (!PAIR && !p.defer_fixup) {
            // one CTA per cluster (cs == 1): the last CTA to arrive sums the
            // parts in CTA order (the first group, once both have stored)
            __threadfence();
            named_sync(3, 8 * kWarp);
          }
          if (!PAIR && !p.defer_fixup && eg == 0) {
            const long long tu = (long long)tg * p.kb;
            const int c_first = cta_of_unit(tu, total, Q);
            const int c_last = cta_of_unit(tu + p.kb - 1, total, Q);
            if (m == 0) {
              const int old = atomicAdd(&p.counters[tile], 1);
              *flag = (old == c_last - c_first) ? 1 : 0;
            }
            named_sync(1, 4 * kWarp);
            if (*flag != 0) {
              __threadfence();
              static_assert(EC == 16, "16-column epilogue chunks");
              tc_fixup_tile<EPI, LD>(p, tile, c_first, c_last, total, epi, m, rows, NT);
              if (m == 0) p.counters[tile] = 0;  // ready for the next launch
            }
          }
        }
        u += k1 - k0;
      }
    }
  }
  // every role is done: the producer saw every stage released by the whole
  // cluster, every accumulator has been read; then no peer touches this CTA's
  // shared memory or barriers any more
  tc_fence_before();
  __syncthreads();
  if (mc || PAIR) cluster_sync_all();
  tc_fence_after();
  if (warp == 1) {
    if constexpr (PAIR)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
  }
}

// Deferred stream-K fixup: block (b, y) handles the boundary between groups
// b and b + 1 of the GEMM's grid when it cuts a (weight tile, group) and is
// that unit range's first such boundary (the others exit), for the
// activation tile of group rank y / (H chunks), the 128-row weight tile
// (y / chunks) % H of the unit (H = 2 with CTA pairs) and the 16-row chunk
// y % chunks; 128 threads, thread m = weight row m.  The parts are summed in
// group order, the same order the last-arriving CTA of a one-CTA group uses,
// so the result does not depend on the mode.
template <int EPI>
__global__ void __launch_bounds__(128, 8) gemm_tc_fixup_kernel(const GemmParams p, int Q) {
  SDV_TRACE_SCOPE(kTrFixup + SDV_GEMM_SLOT(EPI, p));
  constexpr int LD = EPI_LD;
  __shared__ float epi[16 * LD];
  griddep_launch_dependents();
  // which chunk of which cut tile, from the launch's parameters alone: blocks
  // with nothing to do leave before the wait for the GEMM
  const int NT = p.nt, cs = p.cs;
  const int H = p.pair ? 2 : 1;  // 128-row weight tiles per unit
  const long long total = (long long)((p.m_tiles + H - 1) / H) * p.n_groups * p.kb;
  const int qb = blockIdx.x + 1;
  const long long ub = (long long)qb * total / Q;
  const int tg = static_cast<int>(ub / p.kb);
  const long long t0 = (long long)tg * p.kb;
  if (ub == t0) return;                                      // the boundary falls on a tile edge
  if (qb > 1 && (long long)(qb - 1) * total / Q > t0) return;  // an earlier boundary cuts the same tile
  const int chunks = (NT + 15) / 16;
  const int rank = blockIdx.y / (H * chunks);
  const int hc = blockIdx.y - rank * H * chunks;
  const int half = hc / chunks;
  const int tmu = tg / p.n_groups;
  const int tm = tmu * H + half;
  const int tn = (tg - tmu * p.n_groups) * cs + rank;
  if (tn >= p.n_tiles || tm >= p.m_tiles) return;
  const int rows = min(NT, p.R - tn * NT);
  const int c0 = (hc - half * chunks) * 16;
  if (c0 >= rows) return;
  const int m = threadIdx.x;
  const int q_first = cluster_of_unit(t0, total, Q);
  const int q_last = cluster_of_unit(t0 + p.kb - 1, total, Q);
  SDV_GRIDDEP_WAIT();
  // the parts (inside the partials buffer whatever the verdict) and the
  // status word in the same round trip
  const int st = read_status(p.status);
  float v[16];
#pragma unroll
  for (int n = 0; n < 16; ++n) v[n] = 0.f;
  for (int qq0 = q_first; qq0 <= q_last; qq0 += 2) {
    float w[2][16];
#pragma unroll
    for (int i = 0; i < 2; ++i)
      if (qq0 + i <= q_last) {
        const int qq = qq0 + i;
        const int first_tg_qq = static_cast<int>(((long long)qq * total / Q) / p.kb);
        const int slot = 2 * ((qq * cs + rank) * H + half) + (tg == first_tg_qq ? 0 : 1);
        const float* src = p.partials + (size_t)slot * BM * NT + (size_t)c0 * BM + m;
#pragma unroll
        for (int n = 0; n < 16; ++n) w[i][n] = __ldcg(src + (size_t)n * BM);
      }
#pragma unroll
    for (int i = 0; i < 2; ++i)
      if (qq0 + i <= q_last) {
#pragma unroll
        for (int n = 0; n < 16; ++n) v[n] += w[i][n];
      }
  }
  if (st != 0) return;
#pragma unroll
  for (int n = 0; n < 16; ++n) epi[n * LD + m] = v[n];
  __syncthreads();
  // SWIGLU: the rows' 1 / rms as the main kernel reduced them, when it published them
  const float* rs = EPI == EPI_SWIGLU && p.epi.rscale ? p.epi.rscale : nullptr;
  epilogue_rows<EPI, LD>(p, epi, tm, tn * NT + c0, min(16, rows - c0), m, rs, 0);
}

template <int EPI>
cudaError_t launch_fixup_e(const GemmParams& p, int Q, cudaStream_t stream) {
  if (Q < 2) return cudaSuccess;  // one cluster cuts no tile
  const dim3 g(Q - 1, p.cs * (p.pair ? 2 : 1) * ((p.nt + 15) / 16));
  return launch_pdl(gemm_tc_fixup_kernel<EPI>, g, dim3(128), 0, stream, p, Q);
}

cudaError_t launch_fixup(int epi, const GemmParams& p, int Q, cudaStream_t stream) {
  switch (epi) {
    case EPI_F32: return launch_fixup_e<EPI_F32>(p, Q, stream);
    case EPI_RESID: return launch_fixup_e<EPI_RESID>(p, Q, stream);
    case EPI_SWIGLU: return launch_fixup_e<EPI_SWIGLU>(p, Q, stream);
    case EPI_QKV: return launch_fixup_e<EPI_QKV>(p, Q, stream);
    case EPI_LMHEAD: return launch_fixup_e<EPI_LMHEAD>(p, Q, stream);
    default: return cudaErrorInvalidValue;
  }
}

// ---------------------------------------------------------------------------
// host: the launch configuration
// ---------------------------------------------------------------------------

// Activation tile heights at and above which cut tiles go to the parallel
// fixup kernel (one 16-row chunk per block) rather than to the last CTA to
// arrive, which would walk every chunk of the tile.
constexpr int kDeferFixupRows = 32;

using Kern = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, GemmParams);

template <int EPI, int XP>
Kern kernel_of(bool pair) {
  return pair ? reinterpret_cast<Kern>(gemm_tc_kernel<EPI, XP, true>)
              : reinterpret_cast<Kern>(gemm_tc_kernel<EPI, XP, false>);
}

Kern pick_kernel(int epi, int xp, bool pair) {
  switch (epi) {
    case EPI_F32: return xp == 2 ? kernel_of<EPI_F32, 2>(pair) : kernel_of<EPI_F32, 1>(pair);
    case EPI_RESID: return xp == 2 ? kernel_of<EPI_RESID, 2>(pair) : kernel_of<EPI_RESID, 1>(pair);
    case EPI_SWIGLU: return xp == 2 ? kernel_of<EPI_SWIGLU, 2>(pair) : kernel_of<EPI_SWIGLU, 1>(pair);
    case EPI_QKV: return xp == 2 ? kernel_of<EPI_QKV, 2>(pair) : kernel_of<EPI_QKV, 1>(pair);
    case EPI_LMHEAD: return kernel_of<EPI_LMHEAD, 1>(pair);
    default: return nullptr;
  }
}

// CTA pairs from kPairRows activation rows up: measured in the step of the
// 9B-class layer, pairs against single CTAs at 320 rows took QKV 53.6 -> 44.0
// us, gate/up 240.8 -> 184.4, the LM head 497.9 -> 362.9; at 1152 rows 120.6
// -> 92.4, 535.6 -> 426.2 and 1239 -> 1072; below 128 rows, where both are
// bound by the weight stream, they were within 2 % either way.
// SDV_GEMM_PAIR=0|1 in the environment forces them off or on (A/B timing).
constexpr int kPairRows = 128;
int pair_mode() {
  static const int mode = [] {
    const char* v = std::getenv("SDV_GEMM_PAIR");
    if (v && std::strcmp(v, "0") == 0) return 0;
    if (v && std::strcmp(v, "1") == 0) return 1;
    return 2;
  }();
  return mode;
}

// How the single CTAs that take different activation tiles of the same weight
// tile share its read: multicast within a thread-block cluster, or a group of
// consecutive CTAs reading it at about the same time through L2.
// SDV_GEMM_SHARE=mc|l2|off in the environment picks one (A/B timing); the
// default is l2.
int share_mode() {
  static const int mode = [] {
    const char* v = std::getenv("SDV_GEMM_SHARE");
    if (v && std::strcmp(v, "mc") == 0) return 1;
    if (v && std::strcmp(v, "off") == 0) return 0;
    return 2;
  }();
  return mode;
}

int smem_for(int nt, int xp, bool pair = false) {
  return FIXED_BYTES + tc_stages(nt, xp, pair) * tc_stage_bytes(nt, xp, pair);
}

// How many clusters of `cs` CTAs of this kernel fit on the GPU at once (cached).
int active_clusters(Kern k, int cs, int smem, int sms, bool hw_cluster) {
  static std::mutex mu;
  struct Entry {
    Kern k;
    int dev, cs, smem, n;
  };
  static Entry cache[64];
  static int used = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
      if (cache[i].k == k && cache[i].dev == dev && cache[i].cs == cs && cache[i].smem == smem) return cache[i].n;
  }
  int n = 0;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess) {
    if (cs == 1 || !hw_cluster) {
      n = sms / cs;
    } else {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(sms / cs * cs));
      cfg.blockDim = dim3(TC_THREADS);
      cfg.dynamicSmemBytes = static_cast<size_t>(smem);
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
      }
      if (n * cs > sms) n = sms / cs;
    }
  }
  std::lock_guard<std::mutex> lock(mu);
  if (used < 64) cache[used++] = Entry{k, dev, cs, smem, n};
  return n;
}

struct TcChoice {
  int nt = 0, cs = 1, n_tiles = 0, n_groups = 0, grid = 0;
  bool pair = false;
};

int round_up(int x, int m) { return (x + m - 1) / m * m; }

// The tile height and group size for R rows.  One CTA per activation tile of
// at most 256 rows (a power of two) streams each weight tile once per tile;
// a group of cs CTAs shares each weight tile, each with an activation tile of
// about R / cs rows.  Which pays was measured on the crossover sweep's shapes
// (GEMM times in the step, 9B-class layer): for the LM head (one activation
// plane) groups of two at 384 and 512 rows (512: 535 -> 469 us) and nothing
// else (320 rows with 160-row tiles: 501 -> 581 us; 640 and 1152 rows lost
// with every group size); for the layer GEMMs (two planes) groups of two
// from 257 to 512 rows (gate/up at 320: 313 -> 240 us, at 512: 343 -> 296),
// three at 640 (441 -> 417) and six at 1152 (715 -> 537).  Group sizes that
// were not measured to pay are not used.
// CTA pairs: a pair takes 256 weight rows against up to 256 activation rows,
// each CTA loading half the activation tile, so that per SM a k-block moves
// two thirds of the bytes of a one-CTA 128 x 256 tile and the ring holds half
// again as many stages.  Tiles of about R / n rows (n = ceil(R / 256)), and
// pairs in groups of n sharing each weight tile through L2, or one pair per
// group walking the activation tiles of a weight tile back to back.
TcChoice choose_pair(int epi, int xp, const GemmParams& g, int sms, int forced_cs) {
  TcChoice c;
  c.pair = true;
  const int R = g.R;
  const int pairs = active_clusters(pick_kernel(epi, xp, true), 2, smem_for(256, xp, true), sms, true);
  if (pairs < 1) return TcChoice{};
  // tile height: a multiple of 32 (each CTA's half in TMA boxes of at least
  // 16 rows -- narrow boxes cost the producer more copies than the stage's
  // MMAs take), the tile count n that keeps the busiest group's work, NT /
  // (groups of n pairs), smallest
  const int n0 = (R + 255) / 256;
  double best = 0.0;
  // one activation plane (the LM head): the fewest tiles, 256 rows where they
  // fill (1152 rows: 5 tiles of 256 in groups of 5 pairs, 1065 -> 955 us
  // against 6 tiles of 192); two planes: the estimate below
  const int n_last = xp == 1 ? n0 : n0 + 2;
  for (int n = n0; n <= n_last; ++n) {
    const int nt = round_up((R + n - 1) / n, 32);
    if (nt > 256) continue;
    const int tiles = (R + nt - 1) / nt;
    const int groups = pairs / tiles;
    if (groups < 1) continue;
    const double cost = static_cast<double>(nt) / groups;
    if (c.nt == 0 || cost < best * 0.999) {
      best = cost;
      c.nt = nt;
      c.n_tiles = tiles;
    }
  }
  if (c.nt == 0) {
    c.nt = 256;
    c.n_tiles = (R + 255) / 256;
  }
  const long long m_units = (g.m_tiles + 1) / 2;
  const int cs = forced_cs > 0 ? forced_cs : c.n_tiles;
  if (cs > 1 && cs == c.n_tiles && cs <= pairs) {
    c.cs = cs;
    c.n_groups = 1;
    const long long units = m_units * g.kb;
    const int groups = pairs / cs;
    c.grid = static_cast<int>(units < groups ? units : groups) * cs * 2;
    return c;
  }
  c.cs = 1;
  c.n_groups = c.n_tiles;
  const long long units = m_units * c.n_tiles * g.kb;
  c.grid = static_cast<int>(units < pairs ? units : pairs) * 2;
  return c;
}

TcChoice choose(int epi, int xp, const GemmParams& g, int sms) {
  static const int forced = [] {
    // SDV_GEMM_CS=n in the environment: groups of n wherever n tiles cover
    // the rows (A/B timing of the choice)
    const char* v = std::getenv("SDV_GEMM_CS");
    return v ? std::atoi(v) : 0;
  }();
  const int R = g.R;
  if (pair_mode() == 1 || (pair_mode() == 2 && R >= kPairRows)) {
    const TcChoice c = choose_pair(epi, xp, g, sms, forced);
    if (c.grid > 0) return c;
  }
  int cs = 1;
  if (forced > 0) {
    cs = forced;
  } else if (share_mode() != 0) {
    if (xp == 1) cs = (R > 320 && R <= 512) ? 2 : 1;
    else if (R > 256 && R <= 512) cs = 2;
    else if (R > 512 && R <= 768) cs = 3;
    else if (R > 1024 && R <= 1536) cs = 6;
  }
  TcChoice c;
  if (cs > 1 && cs <= kMaxCluster) {
    c.nt = round_up((R + cs - 1) / cs, 16);
    c.n_tiles = (R + c.nt - 1) / c.nt;
    if (c.nt <= 256 && c.n_tiles == cs) {
      const int groups =
          active_clusters(pick_kernel(epi, xp, false), cs, smem_for(c.nt, xp), sms, share_mode() == 1);
      if (groups > 0) {
        const long long units = (long long)g.m_tiles * g.kb;
        c.cs = cs;
        c.n_groups = 1;
        c.grid = static_cast<int>(units < groups ? units : groups) * cs;
        return c;
      }
    }
  }
  c.cs = 1;
  c.nt = gemm_tc_tile_rows(R);
  c.n_tiles = (R + c.nt - 1) / c.nt;
  c.n_groups = c.n_tiles;
  const long long units = (long long)g.m_tiles * c.n_tiles * g.kb;
  c.grid = static_cast<int>(units < sms ? units : sms);
  return c;
}

// The TMA box height for a CTA's nt activation rows: all of them in one copy
// when a map of that height exists, else the largest power of two dividing nt.
int box_for(int nt) {
  if (x_map_index(nt) >= 0) return nt;
  for (int b = 256; b >= 8; b >>= 1)
    if (nt % b == 0) return b;
  return 8;
}

}  // namespace

int gemm_tc_tile_rows(int R) {
  if (R <= 16) return 16;
  if (R <= 32) return 32;
  if (R <= 64) return 64;
  if (R <= 128) return 128;
  return 256;
}

cudaError_t launch_gemm_tc_fixup(int epi, int nt, const GemmParams& p, int grid, cudaStream_t stream) {
  // one CTA per cluster (the int4 kernel): units over (weight tile, activation tile, k-block)
  GemmParams g = p;
  g.nt = nt;
  g.cs = 1;
  g.pair = 0;
  g.n_groups = g.n_tiles;
  return launch_fixup(epi, g, grid, stream);
}

cudaError_t launch_gemm_tc(int epi, int xp, const CUtensorMap* a0, const CUtensorMap* a1, const CUtensorMap* xmaps,
                           GemmParams p, int sms, cudaStream_t stream) {
  if (epi == EPI_LMHEAD) xp = 1;
  const TcChoice c = choose(epi, xp, p, sms);
  if (c.grid < 1) return cudaErrorInvalidConfiguration;
  const Kern k = pick_kernel(epi, xp, c.pair);
  if (!k) return cudaErrorInvalidValue;
  p.nt = c.nt;
  p.cs = c.cs;
  p.n_tiles = c.n_tiles;
  p.n_groups = c.n_groups;
  p.pair = c.pair ? 1 : 0;
  // the kernel reduces the rows' RMSNorm scales once (and publishes them for
  // its fixup) only for rows it can hold; otherwise each chunk reduces them
  if (!(c.n_groups == 1 || p.R <= kScaleRows)) p.epi.rscale = nullptr;
  // a pair's CTA loads half the activation tile
  p.x_box = box_for(c.pair ? c.nt / 2 : c.nt);
  p.stages = tc_stages(c.nt, xp, c.pair);
  p.defer_fixup = (c.pair || c.cs > 1 || c.nt >= kDeferFixupRows) ? 1 : 0;
  p.multicast = !c.pair && c.cs > 1 && share_mode() == 1 ? 1 : 0;
  const int smem = smem_for(c.nt, xp, c.pair);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(c.grid));
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl_enabled()) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (p.multicast || c.pair) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = static_cast<unsigned>(c.pair ? 2 : c.cs);
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  note_launch();
  const CUtensorMap* x = &xmaps[x_map_index(p.x_box)];
  e = cudaLaunchKernelEx(&cfg, k, *a0, *a1, *x, p);
  if (e != cudaSuccess || !p.defer_fixup) return e;
  return launch_fixup(epi, p, c.grid / (c.cs * (c.pair ? 2 : 1)), stream);
}

SDV_TRACE_UNIT(gemm_tc)

}  // namespace sdv
