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
// Warp roles (192 threads):
//  * warp 0: TMA producer (one lane) -- weight half-tiles and activation planes
//    into a multi-stage ring; weights are streamed before waiting for the
//    kernel that writes the activations;
//  * warp 1: allocates 2 x NT columns of tensor memory (two accumulators) and
//    one lane issues the MMAs; tcgen05.commit frees each stage when its MMAs
//    complete and signals each finished accumulator;
//  * warps 2-5: epilogue -- tcgen05.ld the accumulator (lane = weight row),
//    then the stream-K partial/fixup and the fused epilogue shared with the
//    mma.sync kernel, while the MMAs fill the other accumulator.
#include "gemm_common.cuh"
#include "tcgen05.cuh"

namespace sdv {

namespace {

using namespace gemm;
using namespace tc;
constexpr int TC_THREADS = 6 * kWarp;
constexpr int EC = 16;  // accumulator columns per tcgen05.ld / epilogue chunk

template <int NT, int XP>
struct TcCfg {
  static constexpr int B_BYTES = XP * NT * BK * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int EPI_LD = BM + 4;
  static constexpr int EPI_BYTES = EC * EPI_LD * 4;
  static constexpr int FIXED = 1024 + EPI_BYTES + 512;
  static constexpr int FIT = (kSmemBudget - FIXED) / STAGE;
  static constexpr int STAGES = FIT > 10 ? 10 : FIT;
  static constexpr int SMEM = 1024 + STAGES * STAGE + EPI_BYTES + (2 * STAGES + 4) * 8 + 16;
  static constexpr int TMEM_COLS = 2 * NT < 32 ? 32 : 2 * NT;  // power of two for NT in {16..256}
  static_assert(STAGES >= 2, "pipeline too shallow");
  static_assert(SMEM <= kSmemBudget, "shared memory");
  static_assert(NT % 16 == 0 && NT >= 16 && NT <= 256, "tcgen05 N for M = 128");
};

template <int EPI, int NT, int XP>
__global__ void __launch_bounds__(TC_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                   const __grid_constant__ CUtensorMap tmX, const GemmParams p) {
  SDV_TRACE_SCOPE(SDV_GEMM_SLOT(EPI, p));
  using C = TcCfg<NT, XP>;
  extern __shared__ uint8_t smem_raw[];
  griddep_launch_dependents();

  uint8_t* smem = align1024(smem_raw);
  float* epi = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE + C::EPI_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;  // [2] accumulator ready
  uint64_t* tempty = tfull + 2;         // [2] accumulator drained
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);  // one arrival per epilogue warp
    }
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

  const long long total = (long long)p.m_tiles * p.n_tiles * p.kb;
  const int P = gridDim.x;
  const int c = blockIdx.x;
  const long long u_begin = (long long)c * total / P;
  const long long u_end = (long long)(c + 1) * total / P;

  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const int my_units = static_cast<int>(u_end - u_begin);
      const int pre = my_units < C::STAGES ? my_units : C::STAGES;
      struct Cursor {
        int tile, k, tm, tn;
      };
      auto start_at = [&](long long u) {
        Cursor cu;
        cu.tile = static_cast<int>(u / p.kb);
        cu.k = static_cast<int>(u - (long long)cu.tile * p.kb);
        cu.tm = cu.tile / p.n_tiles;
        cu.tn = cu.tile - cu.tm * p.n_tiles;
        return cu;
      };
      auto advance = [&](Cursor& cu) {
        if (++cu.k == p.kb) {
          cu.k = 0;
          ++cu.tile;
          if (++cu.tn == p.n_tiles) {
            cu.tn = 0;
            ++cu.tm;
          }
        }
      };
      auto weights = [&](const Cursor& cu, int stage) {
        const int rowA0 = EPI == EPI_SWIGLU ? cu.tm * 64 : cu.tm * BM;
        const int rowA1 = EPI == EPI_SWIGLU ? cu.tm * 64 : cu.tm * BM + 64;
        uint8_t* sa = smem + stage * C::STAGE;
        tma_load_2d_hint(sa, &tmA0, &full[stage], cu.k * BK, rowA0, pol);
        tma_load_2d_hint(sa + A_BYTES / 2, &tmA1, &full[stage], cu.k * BK, rowA1, pol);
      };
      auto acts = [&](const Cursor& cu, int stage) {
        uint8_t* sb = smem + stage * C::STAGE + A_BYTES;
        tma_load_2d(sb, &tmX, &full[stage], cu.k * BK, cu.tn * NT);
        if constexpr (XP == 2) tma_load_2d(sb + NT * 128, &tmX, &full[stage], cu.k * BK, p.x_lo_row + cu.tn * NT);
      };
      Cursor cw = start_at(u_begin);
      for (int j = 0; j < pre; ++j) {
        mbar_expect_tx(&full[j], A_BYTES);
        weights(cw, j);
        advance(cw);
      }
      SDV_GRIDDEP_WAIT();
      if (read_status(p.status) != 0) {
        for (int j = 0; j < pre; ++j) mbar_arrive(&full[j]);
        for (int j = 0; j < pre; ++j) mbar_wait(&full[j], 0);
      } else {
        Cursor ca = start_at(u_begin);
        for (int j = 0; j < pre; ++j) {
          mbar_arrive_expect_tx(&full[j], C::STAGE - A_BYTES);
          acts(ca, j);
          advance(ca);
        }
        int stage = pre % C::STAGES;
        uint32_t phase = pre == C::STAGES ? 1u : 0u;
        bool dead = false;
        for (int j = pre; j < my_units; ++j) {
          if (!mbar_wait(&empty[stage], phase ^ 1)) {
            set_status(p.status, SDV_ERR_TIMEOUT);
            dead = true;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], C::STAGE);
          weights(cw, stage);
          acts(cw, stage);
          advance(cw);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        // stay until the MMAs have released every stage (no copy in flight at exit)
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
    }
    return;
  }

  if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      SDV_GRIDDEP_WAIT();
      if (read_status(p.status) == 0) {
        constexpr uint32_t idesc = idesc_bf16(BM, NT);
        bool dead = false;
        int stage = 0;
        uint32_t phase = 0;
        int q = 0;  // piece index
        for (long long u = u_begin; u < u_end; ++q) {
          const int tile = static_cast<int>(u / p.kb);
          const int k0 = static_cast<int>(u - (long long)tile * p.kb);
          const int k1 = static_cast<int>(min((long long)p.kb, k0 + (u_end - u)));
          const int buf = q & 1;
          if (!dead && !mbar_wait(&tempty[buf], ((q >> 1) & 1) ^ 1)) {
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
            const uint32_t a_base = smem_u32(smem + stage * C::STAGE);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t a = desc_sw128(a_base + kk * 32);
#pragma unroll
              for (int pl = 0; pl < XP; ++pl) {
                const uint64_t b = desc_sw128(a_base + A_BYTES + pl * (NT * 128) + kk * 32);
                umma_bf16(d, a, b, idesc, (k > k0 || kk > 0 || pl > 0) ? 1u : 0u);
              }
            }
            umma_commit(&empty[stage]);  // frees the stage once these MMAs have read it
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
          umma_commit(&tfull[buf]);  // accumulator complete
          u += k1 - k0;
        }
      }
    }
    __syncwarp();
    named_sync(2, 5 * kWarp);  // every accumulator read
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS) : "memory");
    return;
  }

  // ---------------- epilogue warps 2..5 ----------------
  const int quarter = warp & 3;          // TMEM lanes 32*quarter .. +31
  const int m = quarter * 32 + lane;     // weight row within the tile
  const int tid = m;
  SDV_GRIDDEP_WAIT();
  if (read_status(p.status) == 0) {
    constexpr int LD = C::EPI_LD;
    bool dead = false;
    int q = 0;
    for (long long u = u_begin; u < u_end; ++q) {
      const int tile = static_cast<int>(u / p.kb);
      const int k0 = static_cast<int>(u - (long long)tile * p.kb);
      const int k1 = static_cast<int>(min((long long)p.kb, k0 + (u_end - u)));
      const int tm = tile / p.n_tiles, tn = tile - tm * p.n_tiles;
      const int buf = q & 1;
      if (!dead && !mbar_wait(&tfull[buf], (q >> 1) & 1)) {
        set_status(p.status, SDV_ERR_TIMEOUT);
        dead = true;
      }
      tc_fence_after();
      const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + buf * NT;
      const int rows = min(NT, p.R - tn * NT);

      // accumulator columns past the last activation row are never read
      const int cols = (rows + EC - 1) / EC * EC;
      if (k0 == 0 && k1 == p.kb) {
        // whole tile in this CTA: epilogue straight from tensor memory
        for (int c0 = 0; c0 < cols; c0 += EC) {
          float v[16];
          tmem_ld16(t_row + c0, v);
          if (c0 + EC == cols) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[buf]);
          }
#pragma unroll
          for (int n = 0; n < EC; ++n) epi[n * LD + m] = v[n];
          named_sync(1, 4 * kWarp);
          epilogue_rows<EPI, LD>(p, epi, tm, tn * NT + c0, min(EC, rows - c0), tid);
          named_sync(1, 4 * kWarp);
        }
      } else {
        // tile cut between CTAs: store this piece, the last arrival sums them in CTA order
        const long long tu = (long long)tile * p.kb;
        const int c_first = cta_of_unit(tu, total, P);
        const int c_last = cta_of_unit(tu + p.kb - 1, total, P);
        const int my_slot = 2 * c + (tile == static_cast<int>(u_begin / p.kb) ? 0 : 1);
        float* mine = p.partials + (size_t)my_slot * BM * NT;
        for (int c0 = 0; c0 < cols; c0 += EC) {
          float v[16];
          tmem_ld16(t_row + c0, v);
          tc_store_part16(mine, c0, m, v);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
        if (p.defer_fixup) {  // the fixup kernel sums the parts once this grid is done
          u += k1 - k0;
          continue;
        }
        __threadfence();
        named_sync(1, 4 * kWarp);
        if (m == 0) {
          const int old = atomicAdd(&p.counters[tile], 1);
          *flag = (old == c_last - c_first) ? 1 : 0;
        }
        named_sync(1, 4 * kWarp);
        const bool last = *flag != 0;
        if (last) {
          __threadfence();
          static_assert(EC == 16, "16-column epilogue chunks");
          tc_fixup_tile<EPI, NT, LD>(p, tile, c_first, c_last, total, epi, m, rows);
          if (m == 0) p.counters[tile] = 0;  // ready for the next launch
        }
      }
      u += k1 - k0;
    }
  }
  tc_fence_before();
  named_sync(2, 5 * kWarp);  // let warp 1 free the tensor memory
}

template <int EPI, int NT, int XP>
cudaError_t launch_tc_t(const CUtensorMap* a0, const CUtensorMap* a1, const CUtensorMap* x, const GemmParams& p,
                        int grid, cudaStream_t stream) {
  auto kern = gemm_tc_kernel<EPI, NT, XP>;
  constexpr int smem = TcCfg<NT, XP>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(TC_THREADS), smem, stream, *a0, *a1, *x, p);
}

template <int EPI, int XP>
cudaError_t launch_tc_nt(int nt, const CUtensorMap* a0, const CUtensorMap* a1, const CUtensorMap* x,
                         const GemmParams& p, int grid, cudaStream_t stream) {
  switch (nt) {
    case 16: return launch_tc_t<EPI, 16, XP>(a0, a1, x, p, grid, stream);
    case 32: return launch_tc_t<EPI, 32, XP>(a0, a1, x, p, grid, stream);
    case 64: return launch_tc_t<EPI, 64, XP>(a0, a1, x, p, grid, stream);
    case 128: return launch_tc_t<EPI, 128, XP>(a0, a1, x, p, grid, stream);
    case 256: return launch_tc_t<EPI, 256, XP>(a0, a1, x, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int EPI>
cudaError_t launch_tc_x(int nt, int xp, const CUtensorMap* a0, const CUtensorMap* a1, const CUtensorMap* x,
                        const GemmParams& p, int grid, cudaStream_t stream) {
  return xp == 2 ? launch_tc_nt<EPI, 2>(nt, a0, a1, x, p, grid, stream)
                 : launch_tc_nt<EPI, 1>(nt, a0, a1, x, p, grid, stream);
}

// Deferred stream-K fixup: block (b, chunk) handles the tile holding the
// first unit of CTA b + 1 of the GEMM's grid, when that CTA boundary cuts the
// tile and is the tile's first such boundary (the tile's other boundaries
// exit), for 16-row chunk `chunk` of the tile; 128 threads, thread m = weight
// row m.  The parts are summed in CTA order, exactly as the last-arriving CTA
// would, so the result does not depend on the mode.
template <int EPI, int NT>
__global__ void __launch_bounds__(128) gemm_tc_fixup_kernel(const GemmParams p, int P) {
  SDV_TRACE_SCOPE(kTrFixup + SDV_GEMM_SLOT(EPI, p));
  constexpr int LD = BM + 4;
  __shared__ float epi[16 * LD];
  griddep_launch_dependents();
  SDV_GRIDDEP_WAIT();
  if (read_status(p.status) != 0) return;
  const long long total = (long long)p.m_tiles * p.n_tiles * p.kb;
  const int c = blockIdx.x + 1;
  const long long ub = (long long)c * total / P;
  const int tile = static_cast<int>(ub / p.kb);
  const long long t0 = (long long)tile * p.kb;
  if (ub == t0) return;                                 // the boundary falls on a tile edge
  if (c > 1 && (long long)(c - 1) * total / P > t0) return;  // an earlier boundary cuts the same tile
  const int tn = tile % p.n_tiles;
  const int rows = min(NT, p.R - tn * NT);
  const int c0 = blockIdx.y * 16;
  if (c0 >= rows) return;
  const int m = threadIdx.x;
  const int c_first = cta_of_unit(t0, total, P);
  const int c_last = cta_of_unit(t0 + p.kb - 1, total, P);
  float v[16];
#pragma unroll
  for (int n = 0; n < 16; ++n) v[n] = 0.f;
  for (int cc0 = c_first; cc0 <= c_last; cc0 += 4) {
    float w[4][16];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (cc0 + q <= c_last) {
        const int cc = cc0 + q;
        const int first_tile_cc = static_cast<int>(((long long)cc * total / P) / p.kb);
        const int slot = 2 * cc + (tile == first_tile_cc ? 0 : 1);
        const float* src = p.partials + (size_t)slot * BM * NT + (size_t)c0 * BM + m;
#pragma unroll
        for (int n = 0; n < 16; ++n) w[q][n] = __ldcg(src + (size_t)n * BM);
      }
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (cc0 + q <= c_last) {
#pragma unroll
        for (int n = 0; n < 16; ++n) v[n] += w[q][n];
      }
  }
#pragma unroll
  for (int n = 0; n < 16; ++n) epi[n * LD + m] = v[n];
  __syncthreads();
  epilogue_rows<EPI, LD>(p, epi, tile / p.n_tiles, tn * NT + c0, min(16, rows - c0), m);
}

template <int EPI>
cudaError_t launch_fixup_e(int nt, const GemmParams& p, int grid, cudaStream_t stream) {
  if (grid < 2) return cudaSuccess;  // one CTA cuts no tile
  const dim3 g(grid - 1, (nt + 15) / 16);
  switch (nt) {
    case 16: return launch_pdl(gemm_tc_fixup_kernel<EPI, 16>, g, dim3(128), 0, stream, p, grid);
    case 32: return launch_pdl(gemm_tc_fixup_kernel<EPI, 32>, g, dim3(128), 0, stream, p, grid);
    case 64: return launch_pdl(gemm_tc_fixup_kernel<EPI, 64>, g, dim3(128), 0, stream, p, grid);
    case 128: return launch_pdl(gemm_tc_fixup_kernel<EPI, 128>, g, dim3(128), 0, stream, p, grid);
    case 256: return launch_pdl(gemm_tc_fixup_kernel<EPI, 256>, g, dim3(128), 0, stream, p, grid);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_gemm_tc_fixup(int epi, int nt, const GemmParams& p, int grid, cudaStream_t stream) {
  switch (epi) {
    case EPI_F32: return launch_fixup_e<EPI_F32>(nt, p, grid, stream);
    case EPI_RESID: return launch_fixup_e<EPI_RESID>(nt, p, grid, stream);
    case EPI_SWIGLU: return launch_fixup_e<EPI_SWIGLU>(nt, p, grid, stream);
    case EPI_QKV: return launch_fixup_e<EPI_QKV>(nt, p, grid, stream);
    case EPI_LMHEAD: return launch_fixup_e<EPI_LMHEAD>(nt, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

int gemm_tc_tile_rows(int R) {
  if (R <= 16) return 16;
  if (R <= 32) return 32;
  if (R <= 64) return 64;
  if (R <= 128) return 128;
  return 256;
}

cudaError_t launch_gemm_tc(int epi, int nt, int xp, const CUtensorMap* a0, const CUtensorMap* a1,
                           const CUtensorMap* x, const GemmParams& p, int grid, cudaStream_t stream) {
  switch (epi) {
    case EPI_F32: return launch_tc_x<EPI_F32>(nt, xp, a0, a1, x, p, grid, stream);
    case EPI_RESID: return launch_tc_x<EPI_RESID>(nt, xp, a0, a1, x, p, grid, stream);
    case EPI_SWIGLU: return launch_tc_x<EPI_SWIGLU>(nt, xp, a0, a1, x, p, grid, stream);
    case EPI_QKV: return launch_tc_x<EPI_QKV>(nt, xp, a0, a1, x, p, grid, stream);
    case EPI_LMHEAD: return launch_tc_nt<EPI_LMHEAD, 1>(nt, a0, a1, x, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

SDV_TRACE_UNIT(gemm_tc)

}  // namespace sdv
