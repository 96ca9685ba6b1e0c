// Weight-streaming GEMM over int4 group-32 weights: y[r, n] = sum_k x[r, k] W[n, k]
// with W[n, k] = s[n, k / 32] * q[n, k], q a signed 4-bit code and s an fp16
// scale per 32 consecutive k.
//
// The int4 layer moves a quarter of the bf16 bytes, so in the memory-bound
// regime the layer's part of the step shrinks by that much; the weights are
// still read exactly once per step.  The kernel keeps the structure of the
// bf16 mma.sync kernel (TMA producer warp, deep mbarrier ring, four consumer
// warps, stream-K split, fused epilogues) and changes the weight side:
//
//  * a stage holds 256 k: 128 rows x 128 bytes of packed codes (128-byte
//    swizzle) and 128 rows x 8 fp16 scales, plus the activation tile as four
//    64-k sub-tiles per plane;
//  * the MMA's A operand is the codes themselves: -8..7 are exact in bf16, so
//    a code byte becomes a bf16 pair with two integer operations and one
//    exact bf16 subtraction (the nibble is placed in the mantissa of 128,
//    offset by 8 so its sign is folded in, and 136 is subtracted);
//  * each group of 32 k is accumulated in fp32 on its own and then added to
//    the running sum times its scale, so the result is the exact products
//    summed in fp32: no rounding of the dequantised weight, the same
//    precision as the bf16 path.
#include "gemm_common.cuh"

namespace sdv {

namespace {

using namespace gemm;
constexpr int CONSUMERS = 4;
constexpr int THREADS = (CONSUMERS + 1) * kWarp;

template <int NT, int XP>
struct QCfg {
  static constexpr int SUB = NT * 128;             // one 64-k activation sub-tile
  static constexpr int B_BYTES = XP * 4 * SUB;
  static constexpr int STAGE = Q_A_BYTES + B_BYTES;
  static constexpr int EPI_LD = BM + 4;
  static constexpr int EPI_BYTES = NT * EPI_LD * 4;
  static constexpr int FIXED = 1024 + EPI_BYTES + 512;
  static constexpr int FIT = (kSmemBudget - FIXED) / STAGE;
  static constexpr int STAGES = FIT > 8 ? 8 : FIT;
  static constexpr int SMEM = 1024 + STAGES * STAGE + EPI_BYTES + 2 * STAGES * 8 + 16;
  static_assert(STAGE % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");
  static_assert(STAGES >= 2, "pipeline too shallow");
  static_assert(SMEM <= kSmemBudget, "shared memory");
};

template <int EPI, int NT, int XP>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_q4_kernel(const __grid_constant__ CUtensorMap tmQ0, const __grid_constant__ CUtensorMap tmQ1,
                   const __grid_constant__ CUtensorMap tmS0, const __grid_constant__ CUtensorMap tmS1,
                   const __grid_constant__ CUtensorMap tmX, const GemmParams p) {
  SDV_TRACE_SCOPE(SDV_GEMM_SLOT(EPI, p));
  using C = QCfg<NT, XP>;
  constexpr int NF = NT / 8;
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
        const int row0 = EPI == EPI_SWIGLU ? cu.tm * 64 : cu.tm * BM;
        const int row1 = EPI == EPI_SWIGLU ? cu.tm * 64 : cu.tm * BM + 64;
        uint8_t* sa = smem + stage * C::STAGE;
        tma_load_2d_hint(sa, &tmQ0, &full[stage], cu.k * (QK / 2), row0, pol);
        tma_load_2d_hint(sa + Q_CODE_BYTES / 2, &tmQ1, &full[stage], cu.k * (QK / 2), row1, pol);
        tma_load_2d_hint(sa + Q_CODE_BYTES, &tmS0, &full[stage], cu.k * (QK / 32), row0, pol);
        tma_load_2d_hint(sa + Q_CODE_BYTES + Q_SCALE_BYTES / 2, &tmS1, &full[stage], cu.k * (QK / 32), row1, pol);
      };
      auto acts = [&](const Cursor& cu, int stage) {
        uint8_t* sb = smem + stage * C::STAGE + Q_A_BYTES;
#pragma unroll
        for (int pl = 0; pl < XP; ++pl)
#pragma unroll
          for (int kq = 0; kq < 4; ++kq)
            tma_load_2d(sb + (pl * 4 + kq) * C::SUB, &tmX, &full[stage], cu.k * QK + kq * 64,
                        (pl ? p.x_lo_row : 0) + cu.tn * NT);
      };
      // weights first: they do not depend on the kernel that writes the activations
      Cursor cw = start_at(u_begin);
      for (int j = 0; j < pre; ++j) {
        mbar_expect_tx(&full[j], Q_A_BYTES);
        weights(cw, j);
        advance(cw);
      }
      SDV_GRIDDEP_WAIT();
      if (read_status(p.status) != 0) {
        for (int j = 0; j < pre; ++j) mbar_arrive(&full[j]);
        for (int j = 0; j < pre; ++j) mbar_wait(&full[j], 0);
        return;
      }
      Cursor ca = start_at(u_begin);
      for (int j = 0; j < pre; ++j) {
        mbar_arrive_expect_tx(&full[j], C::B_BYTES);
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
  if (read_status(p.status) != 0) return;
  bool dead = false;
  const int g = lane >> 2, t = lane & 3;
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
      const uint8_t* sp = smem + stage * C::STAGE;
      const uint32_t b_stage = smem_u32(sp + Q_A_BYTES);
      // this thread's rows are m = warp*32 + mi*16 + g (+8); row m's 8 group scales sit at scales + m*8
      const __half* scales = reinterpret_cast<const __half*>(sp + Q_CODE_BYTES);
#pragma unroll 2
      for (int gi = 0; gi < QK / 32; ++gi) {
        // codes of group gi: one 16-byte chunk per row (swizzled by row & 7 = g);
        // byte t of each of its four words holds this thread's k pairs
        // (2t, 2t+1), (2t+8, 2t+9) of the first k16 step and the same of the second
        uint32_t a[2][2][4];  // [mi][k16 step][fragment register]
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
          uint32_t r[2][4];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int row = warp * 32 + mi * 16 + h * 8 + g;
            const uint4 w = *reinterpret_cast<const uint4*>(sp + row * 128 + ((gi ^ g) << 4));
            const uint32_t sel = t | ((4 + t) << 4);
            const uint32_t x = __byte_perm(__byte_perm(w.x, w.y, sel), __byte_perm(w.z, w.w, sel), 0x5410);
            codes_to_bf16(x, r[h]);
          }
#pragma unroll
          for (int s2 = 0; s2 < 2; ++s2) {
            a[mi][s2][0] = r[0][2 * s2];
            a[mi][s2][1] = r[1][2 * s2];
            a[mi][s2][2] = r[0][2 * s2 + 1];
            a[mi][s2][3] = r[1][2 * s2 + 1];
          }
        }
        float part[2][NF][4];
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
          for (int nj = 0; nj < NF; ++nj)
#pragma unroll
            for (int q = 0; q < 4; ++q) part[mi][nj][q] = 0.f;
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {
          const int kidx = gi * 2 + s2;  // k16 step within the stage
          const int kq = kidx >> 2, kk = kidx & 3;
#pragma unroll
          for (int pl = 0; pl < XP; ++pl) {
            const uint32_t b_base = b_stage + (pl * 4 + kq) * C::SUB;
            if constexpr (NF == 1) {
              const int chunk = kk * 2 + ((lane >> 3) & 1);
              uint32_t b0, b1;
              ldsm_x2(b_base + rr * 128 + ((chunk ^ rr) << 4), b0, b1);
#pragma unroll
              for (int mi = 0; mi < 2; ++mi) mma_bf16(part[mi][0], a[mi][s2], b0, b1);
            } else {
#pragma unroll
              for (int nj = 0; nj < NF; nj += 2) {
                const int nrow = (nj + (mat >> 1)) * 8 + rr;
                const int chunk = kk * 2 + (mat & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(b_base + nrow * 128 + ((chunk ^ rr) << 4), b0, b1, b2, b3);
#pragma unroll
                for (int mi = 0; mi < 2; ++mi) {
                  mma_bf16(part[mi][nj], a[mi][s2], b0, b1);
                  mma_bf16(part[mi][nj + 1], a[mi][s2], b2, b3);
                }
              }
            }
          }
        }
        // scale the group's exact partial sums into the running sums
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
          const int m0 = warp * 32 + mi * 16 + g;
          const float s0 = __half2float(scales[m0 * 8 + gi]);
          const float s1 = __half2float(scales[(m0 + 8) * 8 + gi]);
#pragma unroll
          for (int nj = 0; nj < NF; ++nj) {
            acc[mi][nj][0] = fmaf(s0, part[mi][nj][0], acc[mi][nj][0]);
            acc[mi][nj][1] = fmaf(s0, part[mi][nj][1], acc[mi][nj][1]);
            acc[mi][nj][2] = fmaf(s1, part[mi][nj][2], acc[mi][nj][2]);
            acc[mi][nj][3] = fmaf(s1, part[mi][nj][3], acc[mi][nj][3]);
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
    finish_tile_mma<EPI, NT, C::EPI_LD>(p, acc, tile, k0, k1, total, u_begin, epi, flag);
    u += k1 - k0;
  }
}

template <int EPI, int NT, int XP>
cudaError_t launch_q_t(const CUtensorMap* q0, const CUtensorMap* q1, const CUtensorMap* s0, const CUtensorMap* s1,
                       const CUtensorMap* x, const GemmParams& p, int grid, cudaStream_t stream) {
  auto kern = gemm_q4_kernel<EPI, NT, XP>;
  constexpr int smem = QCfg<NT, XP>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(THREADS), smem, stream, *q0, *q1, *s0, *s1, *x, p);
}

template <int EPI, int XP>
cudaError_t launch_q_nt(int nt, const CUtensorMap* q0, const CUtensorMap* q1, const CUtensorMap* s0,
                        const CUtensorMap* s1, const CUtensorMap* x, const GemmParams& p, int grid,
                        cudaStream_t stream) {
  switch (nt) {
    case 8: return launch_q_t<EPI, 8, XP>(q0, q1, s0, s1, x, p, grid, stream);
    case 16: return launch_q_t<EPI, 16, XP>(q0, q1, s0, s1, x, p, grid, stream);
    case 32: return launch_q_t<EPI, 32, XP>(q0, q1, s0, s1, x, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int EPI>
cudaError_t launch_q_x(int nt, int xp, const CUtensorMap* q0, const CUtensorMap* q1, const CUtensorMap* s0,
                       const CUtensorMap* s1, const CUtensorMap* x, const GemmParams& p, int grid,
                       cudaStream_t stream) {
  return xp == 2 ? launch_q_nt<EPI, 2>(nt, q0, q1, s0, s1, x, p, grid, stream)
                 : launch_q_nt<EPI, 1>(nt, q0, q1, s0, s1, x, p, grid, stream);
}

}  // namespace

int gemm_q4_tile_rows(int R) { return R <= 8 ? 8 : (R <= 16 ? 16 : 32); }

cudaError_t launch_gemm_q4(int epi, int nt, int xp, const CUtensorMap* q0, const CUtensorMap* q1,
                           const CUtensorMap* s0, const CUtensorMap* s1, const CUtensorMap* x, const GemmParams& p,
                           int grid, cudaStream_t stream) {
  switch (epi) {
    case EPI_F32: return launch_q_x<EPI_F32>(nt, xp, q0, q1, s0, s1, x, p, grid, stream);
    case EPI_RESID: return launch_q_x<EPI_RESID>(nt, xp, q0, q1, s0, s1, x, p, grid, stream);
    case EPI_SWIGLU: return launch_q_x<EPI_SWIGLU>(nt, xp, q0, q1, s0, s1, x, p, grid, stream);
    case EPI_QKV: return launch_q_x<EPI_QKV>(nt, xp, q0, q1, s0, s1, x, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

SDV_TRACE_UNIT(gemm_q4)

}  // namespace sdv
