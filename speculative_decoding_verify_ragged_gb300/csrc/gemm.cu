// Weight-streaming GEMM for the verify step: y[r, n] = sum_k x[r, k] W[n, k].
//
// The verify pass multiplies a few hundred rows at most (sum over sequences of
// gamma_b + 1) by every weight matrix of the layer and by the LM head, so it
// is bound by reading the weights once from HBM ("Speculative Decoding at
// High Batch Size", section "What does one speculative iteration actually
// cost?": at small batch the step is bound by weight and KV reads that do not
// depend on how many tokens are verified).  The kernel is built for that:
//
//  * one TMA producer warp streams 128-row x 64-k weight tiles (two 64-row
//    boxes, 128-byte swizzle) and the matching activation tile into a deep
//    shared-memory ring (7-10 stages, ~180 KB in flight per SM);
//  * four consumer warps run bf16 mma.sync (m16n8k16, fp32 accumulate) with
//    the weights as the 16-row A operand and the activations as the 8-column
//    B operand, so a handful of rows costs no padding of the weight side.
//    Activations arrive as one bf16 plane (the LM head's input) or as two
//    bf16 planes hi + lo of an fp32 value (about 17 significant bits), each
//    multiplied by the weights: the layer's activations are carried at that
//    precision, so no rounding of them compounds from one GEMM to the next;
//  * work is split stream-K: the (tile, k-block) units of the whole matrix are
//    cut into one contiguous range per CTA (one CTA per SM), so every SM
//    streams the same number of bytes whatever the matrix shape.  A tile cut
//    between CTAs is finished by the last CTA to arrive, which sums the
//    partial tiles in a fixed order (deterministic, no spin-waits);
//  * epilogues are fused: RoPE + K/V page scatter after QKV, residual add after
//    O and down, silu(gate) * up after the gate/up pair, and logits plus
//    per-tile softmax statistics after the LM head.
#include "gemm_common.cuh"

namespace sdv {

namespace {

using namespace gemm;
constexpr int CONSUMERS = 4;
constexpr int THREADS = (CONSUMERS + 1) * kWarp;

template <int NT, int XP>
struct Cfg {
  static constexpr int B_BYTES = XP * NT * BK * 2;  // XP activation planes of NT rows x 64 k
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int EPI_LD = BM + 4;  // padded row of the staged accumulator tile
  static constexpr int EPI_BYTES = NT * EPI_LD * 4;
  static constexpr int FIXED = 1024 + EPI_BYTES + 512;
  static constexpr int FIT = (kSmemBudget - FIXED) / STAGE;
  static constexpr int STAGES = FIT > 10 ? 10 : FIT;
  static constexpr int SMEM = 1024 + STAGES * STAGE + EPI_BYTES + 2 * STAGES * 8 + 16;
  static_assert(STAGES >= 3, "pipeline too shallow");
  static_assert(SMEM <= kSmemBudget, "shared memory");
};

template <int EPI, int NT, int XP>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_ws_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                   const __grid_constant__ CUtensorMap tmX, const GemmParams p) {
  SDV_TRACE_SCOPE(SDV_GEMM_SLOT(EPI, p));
  using C = Cfg<NT, XP>;
  constexpr int NF = NT / 8;  // n8 fragments
  extern __shared__ uint8_t smem_raw[];
  griddep_launch_dependents();

  uint8_t* smem = align1024(smem_raw);
  float* epi = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE + C::EPI_BYTES);
  uint64_t* empty = full + C::STAGES;
  volatile int* flag = reinterpret_cast<volatile int*>(empty + C::STAGES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], CONSUMERS);
    }
    fence_barrier_init();
  }
  __syncthreads();

  const long long total = (long long)p.m_tiles * p.n_tiles * p.kb;
  const int P = gridDim.x;
  const int c = blockIdx.x;
  const long long u_begin = (long long)c * total / P;
  const long long u_end = (long long)(c + 1) * total / P;

  if (warp == CONSUMERS) {
    // ---------------- producer: one elected lane issues all TMA loads ----------------
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const int my_units = static_cast<int>(u_end - u_begin);
      const int pre = my_units < C::STAGES ? my_units : C::STAGES;
      // unit cursors advance by one k-block at a time: no division per stage
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
      // the weights do not depend on earlier kernels: start streaming them
      // before waiting for the kernel that writes the activations
      Cursor cw = start_at(u_begin);
      for (int j = 0; j < pre; ++j) {
        mbar_expect_tx(&full[j], A_BYTES);
        weights(cw, j);
        advance(cw);
      }
      SDV_GRIDDEP_WAIT();
      if (read_status(p.status) != 0) {
        // an earlier kernel failed: let the weight copies land, then leave
        for (int j = 0; j < pre; ++j) mbar_arrive(&full[j]);
        for (int j = 0; j < pre; ++j) mbar_wait(&full[j], 0);
        return;
      }
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
      // tail: stay until the consumers have released every stage, so no copy
      // into this CTA's shared memory is still in flight when it exits
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
  SDV_GRIDDEP_WAIT();
  if (read_status(p.status) != 0) return;  // the producer drains its copies
  // A timed-out wait marks the CTA dead: no more waiting, no early return (the
  // other consumer warps still meet at the named barriers); outputs are then
  // garbage but every access stays in bounds and the status word says why.
  bool dead = false;
  const int mat = lane >> 3, rr = lane & 7;
  float acc[2][NF][4];
  int stage = 0;
  uint32_t phase = 0;

  for (long long u = u_begin; u < u_end;) {
    const int tile = static_cast<int>(u / p.kb);
    const int k0 = static_cast<int>(u - (long long)tile * p.kb);
    const int k1 = static_cast<int>(min((long long)p.kb, k0 + (u_end - u)));
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int nj = 0; nj < NF; ++nj)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[mi][nj][q] = 0.f;

    for (int k = k0; k < k1; ++k) {
      if (!dead && !mbar_wait(&full[stage], phase)) {
        set_status(p.status, SDV_ERR_TIMEOUT);
        dead = true;
      }
      const uint32_t a_base = smem_u32(smem + stage * C::STAGE);
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk) {
        uint32_t a[2][4];
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
          const int row = warp * 32 + mi * 16 + (mat & 1) * 8 + rr;
          const int chunk = kk * 2 + (mat >> 1);
          ldsm_x4(a_base + row * 128 + ((chunk ^ rr) << 4), a[mi][0], a[mi][1], a[mi][2], a[mi][3]);
        }
#pragma unroll
        for (int pl = 0; pl < XP; ++pl) {
          const uint32_t b_base = a_base + A_BYTES + pl * (NT * 128);
          if constexpr (NF == 1) {
            // a single n8 fragment: ldmatrix of the two k-halves of rows 0..7
            const int chunk = kk * 2 + ((lane >> 3) & 1);
            uint32_t b0, b1;
            ldsm_x2(b_base + rr * 128 + ((chunk ^ rr) << 4), b0, b1);
#pragma unroll
            for (int mi = 0; mi < 2; ++mi) mma_bf16(acc[mi][0], a[mi], b0, b1);
          } else {
#pragma unroll
            for (int nj = 0; nj < NF; nj += 2) {
              const int nrow = (nj + (mat >> 1)) * 8 + rr;
              const int chunk = kk * 2 + (mat & 1);
              uint32_t b0, b1, b2, b3;
              ldsm_x4(b_base + nrow * 128 + ((chunk ^ rr) << 4), b0, b1, b2, b3);
#pragma unroll
              for (int mi = 0; mi < 2; ++mi) {
                mma_bf16(acc[mi][nj], a[mi], b0, b1);
                mma_bf16(acc[mi][nj + 1], a[mi], b2, b3);
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == C::STAGES) {
        stage = 0;
        phase ^= 1;
      }
    }

    // stream-K fixup of tiles cut between CTAs, then the fused epilogue
    finish_tile_mma<EPI, NT, C::EPI_LD>(p, acc, tile, k0, k1, total, u_begin, epi, flag);
    u += k1 - k0;
  }
}

template <int EPI, int NT, int XP>
cudaError_t launch_t(const CUtensorMap* a0, const CUtensorMap* a1, const CUtensorMap* x, const GemmParams& p,
                     int grid, cudaStream_t stream) {
  auto kern = gemm_ws_kernel<EPI, NT, XP>;
  constexpr int smem = Cfg<NT, XP>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(THREADS), smem, stream, *a0, *a1, *x, p);
}

template <int EPI, int XP>
cudaError_t launch_nt(int nt, const CUtensorMap* a0, const CUtensorMap* a1, const CUtensorMap* x,
                      const GemmParams& p, int grid, cudaStream_t stream) {
  switch (nt) {
    case 8: return launch_t<EPI, 8, XP>(a0, a1, x, p, grid, stream);
    case 16: return launch_t<EPI, 16, XP>(a0, a1, x, p, grid, stream);
    case 32: return launch_t<EPI, 32, XP>(a0, a1, x, p, grid, stream);
    case 64: return launch_t<EPI, 64, XP>(a0, a1, x, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int EPI>
cudaError_t launch_x(int nt, int xp, const CUtensorMap* a0, const CUtensorMap* a1, const CUtensorMap* x,
                     const GemmParams& p, int grid, cudaStream_t stream) {
  return xp == 2 ? launch_nt<EPI, 2>(nt, a0, a1, x, p, grid, stream)
                 : launch_nt<EPI, 1>(nt, a0, a1, x, p, grid, stream);
}

}  // namespace

int gemm_tile_rows(int R) { return R <= 8 ? 8 : (R <= 16 ? 16 : (R <= 32 ? 32 : 64)); }

cudaError_t launch_gemm(int epi, int nt, int xp, const CUtensorMap* a0, const CUtensorMap* a1,
                        const CUtensorMap* x, const GemmParams& p, int grid, cudaStream_t stream) {
  switch (epi) {
    case EPI_F32: return launch_x<EPI_F32>(nt, xp, a0, a1, x, p, grid, stream);
    case EPI_RESID: return launch_x<EPI_RESID>(nt, xp, a0, a1, x, p, grid, stream);
    case EPI_SWIGLU: return launch_x<EPI_SWIGLU>(nt, xp, a0, a1, x, p, grid, stream);
    case EPI_QKV: return launch_x<EPI_QKV>(nt, xp, a0, a1, x, p, grid, stream);
    case EPI_LMHEAD: return launch_nt<EPI_LMHEAD, 1>(nt, a0, a1, x, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

SDV_TRACE_UNIT(gemm)

}  // namespace sdv
