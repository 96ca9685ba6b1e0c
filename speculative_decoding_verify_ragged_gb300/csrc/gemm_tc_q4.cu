// int4 group-32 weight GEMM on the 5th-generation tensor cores:
// y[r, n] = sum_k x[r, k] W[n, k], W[n, k] = s[n, k / 32] * q[n, k].
//
// Once the verify rows are in the hundreds the int4 layer is no longer bound
// by its (small) weight stream but by the contraction, and the legacy
// mma.sync path of gemm_q4.cu runs at a fraction of the tensor cores' rate.
// This kernel keeps the int4 stream (codes and scales staged by TMA, 256 k per
// stage) and the fused epilogues and stream-K split of the other GEMMs, and
// dequantises in shared memory for tcgen05.mma:
//
//  * w = s * q is exact in fp32 (an fp16 scale times a code in [-8, 7] has at
//    most 14 significant bits), and so is its split into bf16 hi = rn(w) and
//    lo = w - hi (at most 7 more bits), so hi + lo is the weight exactly;
//  * a converter warpgroup writes hi and lo of each 128 x 64 block in the
//    K-major 128-byte-swizzle layout the MMA reads;
//  * the MMA thread issues hi*x_hi into one TMEM accumulator and the small
//    cross terms hi*x_lo + lo*x_hi into a second one, added in the epilogue, so
//    the large accumulator takes a third of the additions (the tensor cores'
//    fp32 accumulation error grows with them); the dropped lo*x_lo term is
//    below 2^-16 of each product.
//
// Warp roles (320 threads): 0 TMA producer; 1 TMEM allocation and MMA issue;
// 2-5 epilogue (tcgen05.ld, stream-K partials, fused epilogue); 6-9 converters.
#include "gemm_common.cuh"
#include "tcgen05.cuh"

namespace sdv {

namespace {

using namespace gemm;
using namespace tc;
constexpr int Q4_THREADS = 10 * kWarp;
constexpr int EC = 16;                     // accumulator columns per tcgen05.ld / epilogue chunk
constexpr int C_STAGE = 2 * A_BYTES;       // one converted 64-k block: hi then lo (32 KB)

template <int NT>
struct TqCfg {
  static constexpr int X_STAGE = 2 * NT * 128;  // activations of 64 k: hi plane then lo plane
  static constexpr int QS = 2, CS = 2;
  static constexpr int EPI_LD = BM + 4;
  static constexpr int EPI_BYTES = EC * EPI_LD * 4;
  static constexpr int FIXED = 1024 + QS * Q_A_BYTES + CS * C_STAGE + EPI_BYTES + 1024;
  static constexpr int FIT = (kSmemBudget - FIXED) / X_STAGE;
  static constexpr int XS = FIT > 6 ? 6 : FIT;
  static constexpr int OFF_C = QS * Q_A_BYTES;
  static constexpr int OFF_X = OFF_C + CS * C_STAGE;
  static constexpr int OFF_EPI = OFF_X + XS * X_STAGE;
  static constexpr int OFF_BAR = OFF_EPI + EPI_BYTES;
  static constexpr int SMEM = 1024 + OFF_BAR + (2 * (QS + CS + XS) + 4) * 8 + 16;
  // two buffers x (main, correction) accumulators of NT columns
  static constexpr int TMEM_COLS = 4 * NT < 32 ? 32 : 4 * NT;
  static_assert(Q_A_BYTES % 1024 == 0 && X_STAGE % 1024 == 0, "1024-byte swizzle alignment");
  static_assert(XS >= 2, "pipeline too shallow");
  static_assert(SMEM <= kSmemBudget, "shared memory");
  static_assert(NT % 16 == 0 && NT >= 16 && NT <= 128, "tcgen05 N for M = 128");
};

// Converter thread `row` (0..127) turns 64 k of its weight row into bf16 hi and
// lo, k-quarter `kq` of a 256-k code stage: codes of groups 2kq and 2kq + 1
// (16 bytes each, 128-byte swizzle by row & 7) times their fp16 scales, written
// as eight 16-byte chunks per plane at chunk c ^ (row & 7) of the row.
__device__ __forceinline__ void convert_row(const uint8_t* qstage, uint8_t* cstage, int row, int kq) {
  const __half* sc = reinterpret_cast<const __half*>(qstage + Q_CODE_BYTES) + row * 8;
  const int sw = row & 7;
  uint8_t* hi_row = cstage + row * 128;
  uint8_t* lo_row = cstage + A_BYTES + row * 128;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int grp = 2 * kq + h;
    const float s = __half2float(sc[grp]);
    const uint4 w = *reinterpret_cast<const uint4*>(qstage + row * 128 + ((grp ^ sw) << 4));
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t r[4];
      codes_to_bf16(words[q], r);  // 8 codes of k = 32*grp + 8*q .. +7, exact in bf16
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r[e]));
        split_bf16x2(f.x * s, f.y * s, hi[e], lo[e]);
      }
      const int chunk = h * 4 + q;  // 8-k chunk within the 64-k block
      const int off = ((chunk ^ sw) << 4);
      *reinterpret_cast<uint4*>(hi_row + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(lo_row + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
  }
}

// 16 columns of the main accumulator plus the same columns of the correction
// accumulator `off` columns further on.
__device__ __forceinline__ void tmem_ld_sum(uint32_t taddr, int off, float (&v)[16]) {
  float w[16];
  tmem_ld16(taddr, v);
  tmem_ld16(taddr + off, w);
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] += w[i];
}

template <int EPI, int NT>
__global__ void __launch_bounds__(Q4_THREADS, 1)
    gemm_tc_q4_kernel(const __grid_constant__ CUtensorMap tmQ0, const __grid_constant__ CUtensorMap tmQ1,
                      const __grid_constant__ CUtensorMap tmS0, const __grid_constant__ CUtensorMap tmS1,
                      const __grid_constant__ CUtensorMap tmX, const GemmParams p) {
  SDV_TRACE_SCOPE(SDV_GEMM_SLOT(EPI, p));
  using C = TqCfg<NT>;
  extern __shared__ uint8_t smem_raw[];
  griddep_launch_dependents();

  uint8_t* smem = align1024(smem_raw);
  float* epi = reinterpret_cast<float*>(smem + C::OFF_EPI);
  uint64_t* qfull = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* qempty = qfull + C::QS;
  uint64_t* cfull = qempty + C::QS;
  uint64_t* cempty = cfull + C::CS;
  uint64_t* xfull = cempty + C::CS;
  uint64_t* xempty = xfull + C::XS;
  uint64_t* tfull = xempty + C::XS;  // [2] accumulator ready
  uint64_t* tempty = tfull + 2;      // [2] accumulator drained
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::QS; ++s) {
      mbar_init(&qfull[s], 1);
      mbar_init(&qempty[s], 4);  // one arrival per converter warp
    }
    for (int s = 0; s < C::CS; ++s) {
      mbar_init(&cfull[s], 4);
      mbar_init(&cempty[s], 1);
    }
    for (int s = 0; s < C::XS; ++s) {
      mbar_init(&xfull[s], 1);
      mbar_init(&xempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
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

  const long long total = (long long)p.m_tiles * p.n_tiles * p.kb;  // units of 256 k
  const int P = gridDim.x;
  const int c = blockIdx.x;
  const long long u_begin = (long long)c * total / P;
  const long long u_end = (long long)(c + 1) * total / P;
  const int my_units = static_cast<int>(u_end - u_begin);

  if (warp == 0) {
    // ---------------- producer: codes + scales per 256 k, activations per 64 k ----------------
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      auto tile_of = [&](long long u, int& tm, int& tn, int& kq) {
        const int tile = static_cast<int>(u / p.kb);
        kq = static_cast<int>(u - (long long)tile * p.kb);
        tm = tile / p.n_tiles;
        tn = tile - tm * p.n_tiles;
      };
      auto codes = [&](long long u, int s) {
        int tm, tn, kq;
        tile_of(u, tm, tn, kq);
        const int row0 = EPI == EPI_SWIGLU ? tm * 64 : tm * BM;
        const int row1 = EPI == EPI_SWIGLU ? tm * 64 : tm * BM + 64;
        uint8_t* sq = smem + s * Q_A_BYTES;
        mbar_arrive_expect_tx(&qfull[s], Q_A_BYTES);
        tma_load_2d_hint(sq, &tmQ0, &qfull[s], kq * (QK / 2), row0, pol);
        tma_load_2d_hint(sq + Q_CODE_BYTES / 2, &tmQ1, &qfull[s], kq * (QK / 2), row1, pol);
        tma_load_2d_hint(sq + Q_CODE_BYTES, &tmS0, &qfull[s], kq * (QK / 32), row0, pol);
        tma_load_2d_hint(sq + Q_CODE_BYTES + Q_SCALE_BYTES / 2, &tmS1, &qfull[s], kq * (QK / 32), row1, pol);
      };
      // code stages first: they do not depend on the kernel that writes the activations
      const int pre = my_units < C::QS ? my_units : C::QS;
      for (int j = 0; j < pre; ++j) codes(u_begin + j, j);
      SDV_GRIDDEP_WAIT();
      bool dead = false;
      int qs = pre % C::QS;
      uint32_t qph = pre == C::QS ? 1u : 0u;
      int xs = 0;
      uint32_t xph = 0;
      const bool ok = read_status(p.status) == 0;
      for (int j = 0; j < my_units && ok && !dead; ++j) {
        if (j >= pre) {
          if (!mbar_wait(&qempty[qs], qph ^ 1)) {
            set_status(p.status, SDV_ERR_TIMEOUT);
            dead = true;
            break;
          }
          codes(u_begin + j, qs);
          if (++qs == C::QS) {
            qs = 0;
            qph ^= 1;
          }
        }
        int tm, tn, kq;
        tile_of(u_begin + j, tm, tn, kq);
        for (int s = 0; s < QK / BK; ++s) {
          if (!mbar_wait(&xempty[xs], xph ^ 1)) {
            set_status(p.status, SDV_ERR_TIMEOUT);
            dead = true;
            break;
          }
          uint8_t* sx = smem + C::OFF_X + xs * C::X_STAGE;
          mbar_arrive_expect_tx(&xfull[xs], C::X_STAGE);
          tma_load_2d(sx, &tmX, &xfull[xs], kq * QK + s * BK, tn * NT);
          tma_load_2d(sx + NT * 128, &tmX, &xfull[xs], kq * QK + s * BK, p.x_lo_row + tn * NT);
          if (++xs == C::XS) {
            xs = 0;
            xph ^= 1;
          }
        }
      }
      // the pre-issued code stages must land before exit even when the step failed
      if (!ok)
        for (int j = 0; j < pre; ++j) mbar_wait(&qfull[j], 0);
      // stay until the consumers have released every stage (no copy in flight at exit)
      for (int i = 0; i < C::XS && ok && !dead; ++i) {
        if (!mbar_wait(&xempty[xs], xph ^ 1)) {
          set_status(p.status, SDV_ERR_TIMEOUT);
          break;
        }
        if (++xs == C::XS) {
          xs = 0;
          xph ^= 1;
        }
      }
      for (int i = 0; i < C::QS && ok && !dead; ++i) {
        if (!mbar_wait(&qempty[qs], qph ^ 1)) {
          set_status(p.status, SDV_ERR_TIMEOUT);
          break;
        }
        if (++qs == C::QS) {
          qs = 0;
          qph ^= 1;
        }
      }
    }
    return;
  }

  if (warp >= 6) {
    // ---------------- converters: codes x scales -> bf16 hi + lo, one row per thread ----------------
    const int row = (warp - 6) * kWarp + lane;
    SDV_GRIDDEP_WAIT();
    if (read_status(p.status) != 0) return;
    bool dead = false;
    int qs = 0, cs = 0;
    uint32_t qph = 0, cph = 0;
    for (int j = 0; j < my_units && !dead; ++j) {
      if (!mbar_wait(&qfull[qs], qph)) {
        set_status(p.status, SDV_ERR_TIMEOUT);
        dead = true;
        break;
      }
      const uint8_t* sq = smem + qs * Q_A_BYTES;
      for (int kq = 0; kq < QK / BK; ++kq) {
        if (!mbar_wait(&cempty[cs], cph ^ 1)) {
          set_status(p.status, SDV_ERR_TIMEOUT);
          dead = true;
          break;
        }
        convert_row(sq, smem + C::OFF_C + cs * C_STAGE, row, kq);
        fence_proxy_async_smem();  // visible to the MMAs that read it
        __syncwarp();
        if (lane == 0) mbar_arrive(&cfull[cs]);
        if (++cs == C::CS) {
          cs = 0;
          cph ^= 1;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&qempty[qs]);
      if (++qs == C::QS) {
        qs = 0;
        qph ^= 1;
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
        int cs = 0, xs = 0;
        uint32_t cph = 0, xph = 0;
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
          const uint32_t d = tmem + buf * 2 * NT, dc = d + NT;
          for (int k = k0; k < k1; ++k) {
            for (int s = 0; s < QK / BK; ++s) {
              if (!dead && !mbar_wait(&cfull[cs], cph)) {
                set_status(p.status, SDV_ERR_TIMEOUT);
                dead = true;
              }
              if (!dead && !mbar_wait(&xfull[xs], xph)) {
                set_status(p.status, SDV_ERR_TIMEOUT);
                dead = true;
              }
              tc_fence_after();
              const uint32_t a_hi = smem_u32(smem + C::OFF_C + cs * C_STAGE);
              const uint32_t b_hi = smem_u32(smem + C::OFF_X + xs * C::X_STAGE);
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk) {
                const uint64_t ah = desc_sw128(a_hi + kk * 32), al = desc_sw128(a_hi + A_BYTES + kk * 32);
                const uint64_t bh = desc_sw128(b_hi + kk * 32), bl = desc_sw128(b_hi + NT * 128 + kk * 32);
                const uint32_t acc = (k > k0 || s > 0 || kk > 0) ? 1u : 0u;
                umma_bf16(d, ah, bh, idesc, acc);
                umma_bf16(dc, ah, bl, idesc, acc);
                umma_bf16(dc, al, bh, idesc, 1u);
              }
              umma_commit(&cempty[cs]);  // frees the converted block and the activations
              umma_commit(&xempty[xs]);  // once these MMAs have read them
              if (++cs == C::CS) {
                cs = 0;
                cph ^= 1;
              }
              if (++xs == C::XS) {
                xs = 0;
                xph ^= 1;
              }
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
      const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + buf * 2 * NT;
      const int rows = min(NT, p.R - tn * NT);

      // accumulator columns past the last activation row are never read
      const int cols = (rows + EC - 1) / EC * EC;
      if (k0 == 0 && k1 == p.kb) {
        // whole tile in this CTA: epilogue straight from tensor memory
        for (int c0 = 0; c0 < cols; c0 += EC) {
          float v[16];
          tmem_ld_sum(t_row + c0, NT, v);
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
          tmem_ld_sum(t_row + c0, NT, v);
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
          tc_fixup_tile<EPI, LD>(p, tile, c_first, c_last, total, epi, m, rows, NT);
          if (m == 0) p.counters[tile] = 0;  // ready for the next launch
        }
      }
      u += k1 - k0;
    }
  }
  tc_fence_before();
  named_sync(2, 5 * kWarp);  // let warp 1 free the tensor memory
}

template <int EPI, int NT>
cudaError_t launch_q4_t(const CUtensorMap* q0, const CUtensorMap* q1, const CUtensorMap* s0, const CUtensorMap* s1,
                        const CUtensorMap* x, const GemmParams& p, int grid, cudaStream_t stream) {
  auto kern = gemm_tc_q4_kernel<EPI, NT>;
  constexpr int smem = TqCfg<NT>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(Q4_THREADS), smem, stream, *q0, *q1, *s0, *s1, *x, p);
}

template <int EPI>
cudaError_t launch_q4_nt(int nt, const CUtensorMap* q0, const CUtensorMap* q1, const CUtensorMap* s0,
                         const CUtensorMap* s1, const CUtensorMap* x, const GemmParams& p, int grid,
                         cudaStream_t stream) {
  switch (nt) {
    case 16: return launch_q4_t<EPI, 16>(q0, q1, s0, s1, x, p, grid, stream);
    case 32: return launch_q4_t<EPI, 32>(q0, q1, s0, s1, x, p, grid, stream);
    case 64: return launch_q4_t<EPI, 64>(q0, q1, s0, s1, x, p, grid, stream);
    case 128: return launch_q4_t<EPI, 128>(q0, q1, s0, s1, x, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int gemm_tc_q4_tile_rows(int R) {
  if (R <= 16) return 16;
  if (R <= 32) return 32;
  if (R <= 64) return 64;
  return 128;
}

cudaError_t launch_gemm_tc_q4(int epi, int nt, const CUtensorMap* q0, const CUtensorMap* q1, const CUtensorMap* s0,
                              const CUtensorMap* s1, const CUtensorMap* x, const GemmParams& p, int grid,
                              cudaStream_t stream) {
  switch (epi) {
    case EPI_F32: return launch_q4_nt<EPI_F32>(nt, q0, q1, s0, s1, x, p, grid, stream);
    case EPI_RESID: return launch_q4_nt<EPI_RESID>(nt, q0, q1, s0, s1, x, p, grid, stream);
    case EPI_SWIGLU: return launch_q4_nt<EPI_SWIGLU>(nt, q0, q1, s0, s1, x, p, grid, stream);
    case EPI_QKV: return launch_q4_nt<EPI_QKV>(nt, q0, q1, s0, s1, x, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

SDV_TRACE_UNIT(gemm_tc_q4)

}  // namespace sdv
