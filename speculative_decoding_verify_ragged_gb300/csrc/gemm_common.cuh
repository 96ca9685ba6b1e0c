// Pieces shared by the two weight-streaming GEMM kernels (bf16 mma.sync in
// gemm.cu, tcgen05 with TMEM accumulators in gemm_tc.cu): tile constants, the
// stream-K split, and the fused epilogues.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace sdv {
namespace gemm {

constexpr int BM = 128;               // weight rows per tile
constexpr int BK = 64;                // k per stage: 128 bytes of bf16 per row
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int kSmemBudget = 227 * 1024;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// int4 group-32 weights: a stage holds 256 k of 128 weight rows
constexpr int QK = 256;                             // k per code stage
constexpr int Q_CODE_BYTES = BM * QK / 2;           // 16 KB of packed codes (128-byte swizzle)
constexpr int Q_SCALE_BYTES = BM * (QK / 32) * 2;   // 2 KB of fp16 scales, 8 per row
constexpr int Q_A_BYTES = Q_CODE_BYTES + Q_SCALE_BYTES;

// Four code bytes (eight int4 codes, low nibble first) -> four bf16 pairs.
__device__ __forceinline__ void codes_to_bf16(uint32_t x, uint32_t (&r)[4]) {
  const uint32_t v = x ^ 0x88888888u;  // code + 8 in each nibble: 0..15
  const uint32_t lo = v & 0x0F0F0F0Fu;
  const uint32_t hi = (v >> 4) & 0x0F0F0F0Fu;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    // byte 0: low nibble of byte j; byte 2: its high nibble; 0x43 above each
    const uint32_t sel = j | (j << 4) | ((4 + j) << 8) | ((4 + j) << 12);
    const uint32_t m = (__byte_perm(lo, hi, sel) & 0x00FF00FFu) | 0x43004300u;  // bf16 (128 + code + 8)
    __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&m);
    const uint32_t k136 = 0x43084308u;  // bf16 136 in both halves
    b = __hsub2(b, *reinterpret_cast<const __nv_bfloat162*>(&k136));  // exact: code in [-8, 7]
    r[j] = *reinterpret_cast<uint32_t*>(&b);
  }
}

// CTA c of P owns units [c*T/P, (c+1)*T/P); the CTA owning unit u:
__device__ __forceinline__ int cta_of_unit(long long u, long long total, int P) {
  return static_cast<int>(((u + 1) * P - 1) / total);
}

// Fused epilogue over rows [row0, row0 + nrows) of one output tile, staged in
// shared memory as epi[n * LD + m] (n = activation row within the run, m =
// weight row within the tile); 128 threads, tid = m for the column-wise kinds.
// Every per-row global load of a batch of rows is issued before any is used,
// so a batch costs one memory latency instead of one per row.
//
// SWIGLU with an RMSNorm row scale: `row_scale`, when given, holds each row's
// 1 / rms already reduced from the partial sums (row_scale[r - rs_base] for
// row r); otherwise each chunk reduces them itself.  `bar`: the named barrier
// of the 128 calling threads.
template <int EPI, int LD>
__device__ __forceinline__ void epilogue_rows(const GemmParams& p, float* epi, int tm, int row0, int nrows,
                                              int tid, const float* row_scale = nullptr, int rs_base = 0,
                                              int bar = 1) {
  const EpiParams& e = p.epi;
  constexpr int RB = 16;  // rows per batch
  if constexpr (EPI == EPI_RESID) {
    if (e.norm_gain) {
      // residual output that an RMSNorm reads next: x, the planes of x * gain,
      // and each warp's 32-column sum of x^2 per row
      const int col = tm * BM + tid;
      const bool ok = col < p.N;
      const int lane = tid & 31;
      const float gn = ok ? bf2f(e.norm_gain[col]) : 0.f;
      for (int n0 = 0; n0 < nrows; n0 += RB) {
        float res[RB];
#pragma unroll
        for (int q = 0; q < RB; ++q) {
          const int n = n0 + q;
          res[q] = (ok && n < nrows) ? e.resid_f32[(long long)(row0 + n) * e.ld_f32 + col] : 0.f;
        }
#pragma unroll
        for (int q = 0; q < RB; ++q) {
          const int n = n0 + q;
          if (n < nrows) {
            const float x = ok ? epi[n * LD + tid] + res[q] : 0.f;
            if (ok) {
              const long long idx = (long long)(row0 + n) * e.ld_f32 + col;
              e.out_f32[idx] = x;
              store_planes(e.norm_out, e.norm_lo_off, idx, x * gn);
            }
            const float ss = warp_sum(x * x);
            if (lane == 0) e.sq_out[(long long)(col >> 5) * e.sq_ld + row0 + n] = ss;
          }
        }
      }
      return;
    }
  }
  if constexpr (EPI == EPI_F32 || EPI == EPI_RESID) {
    const int col = tm * BM + tid;
    if (col < p.N) {
      for (int n0 = 0; n0 < nrows; n0 += RB) {
        float res[RB];
        if constexpr (EPI == EPI_RESID) {
#pragma unroll
          for (int q = 0; q < RB; ++q) {
            const int n = n0 + q;
            res[q] = n < nrows ? e.resid_f32[(long long)(row0 + n) * e.ld_f32 + col] : 0.f;
          }
        }
#pragma unroll
        for (int q = 0; q < RB; ++q) {
          const int n = n0 + q;
          if (n < nrows) {
            const float v = epi[n * LD + tid];
            e.out_f32[(long long)(row0 + n) * e.ld_f32 + col] = EPI == EPI_RESID ? v + res[q] : v;
          }
        }
      }
    }
  } else if constexpr (EPI == EPI_SWIGLU) {
    // tile = 64 gate rows + the 64 up rows of the same features; the product
    // is the next GEMM's input, written as bf16 hi + lo planes
    const int j = tid & 63;
    const int f = tm * 64 + j;
    if (e.sq_in && row_scale) {
      for (int n = tid; n < nrows; n += 4 * kWarp) epi[n * LD + BM] = row_scale[row0 + n - rs_base];
      named_sync(bar, 4 * kWarp);
    } else if (e.sq_in) {
      // the input was x * gain: each row's 1 / rms(x) from the partial sums of x^2
      const int warp = tid >> 5, lane = tid & 31;
      for (int n = warp; n < nrows; n += 4) {
        float ss = 0.f;
        for (int q = lane; q < e.sq_parts; q += 32) ss += e.sq_in[(long long)q * e.sq_ld + row0 + n];
        ss = warp_sum(ss);
        if (lane == 0) epi[n * LD + BM] = 1.0f / sqrtf(ss * e.sq_inv_n + e.sq_eps);
      }
      named_sync(bar, 4 * kWarp);
    }
    if (f < p.N) {
      for (int n = tid >> 6; n < nrows; n += 2) {
        const float sc = e.sq_in ? epi[n * LD + BM] : 1.f;
        const float gt = epi[n * LD + j] * sc;
        const float up = epi[n * LD + 64 + j] * sc;
        const float s = gt / (1.0f + expf(-gt));
        store_planes(e.out_bf16, e.out_lo_off, (long long)(row0 + n) * e.ld_bf16 + f, s * up);
      }
    }
  } else if constexpr (EPI == EPI_QKV) {
    const int D = e.head_dim;
    const int half = D >> 1;
    const int f = tm * BM + tid;
    if (f < p.N) {
      const int hq = f / D;
      const int j = f - hq * D;
      const bool rot = hq < e.n_q + e.n_kv;
      const int jj = j < half ? j : j - half;
      const int kv = hq < e.n_q + e.n_kv ? 0 : 1;
      const long long head_off =
          hq < e.n_q ? 0 : ((long long)(hq - e.n_q - kv * e.n_kv) * 2 + kv) * e.page * D + j;
      for (int n0 = 0; n0 < nrows; n0 += RB) {
        float2 cs[RB];
        long long dst[RB];
#pragma unroll
        for (int q = 0; q < RB; ++q) {
          const int n = n0 + q;
          const int r = row0 + (n < nrows ? n : 0);
          cs[q] = rot ? *reinterpret_cast<const float2*>(e.rope_cs + ((long long)r * half + jj) * 2)
                      : make_float2(1.f, 0.f);
          dst[q] = hq < e.n_q ? 0 : e.kv_row_off[r];
        }
#pragma unroll
        for (int q = 0; q < RB; ++q) {
          const int n = n0 + q;
          if (n < nrows) {
            const int r = row0 + n;
            float x = epi[n * LD + tid];
            if (rot) {
              const float y = j < half ? -epi[n * LD + tid + half] : epi[n * LD + tid - half];
              x = x * cs[q].x + y * cs[q].y;
            }
            if (hq < e.n_q) e.out_f32[(long long)r * (e.n_q * D) + f] = x;  // q stays fp32
            else e.kv_pool[dst[q] + head_off] = f2bf(x);                   // K, V enter the bf16 cache
          }
        }
      }
    }
  } else if constexpr (EPI == EPI_LMHEAD) {
    // eight lanes per activation row, four rows per warp, sixteen rows per
    // pass: a lane holds 16 of the tile's 128 logits of its row (columns
    // sub + 8 i), so the row's maximum and sum of exp take three shuffle
    // levels, and the four rows of a warp run side by side
    const int warp = tid >> 5, lane = tid & 31;
    const int sub = lane & 7;
    for (int n0 = 0; n0 < nrows; n0 += 16) {
      const int n = n0 + warp * 4 + (lane >> 3);
      const bool live = n < nrows;
      const int r = row0 + n;
      float v[16];
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = live ? epi[n * LD + sub + 8 * i] : 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int col = tm * BM + sub + 8 * i;
        if (live && col < p.N) {
          e.out_f32[(long long)r * e.ld_f32 + col] = v[i];
          mx = fmaxf(mx, v[i]);
        }
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      float s = 0.f;
      int arg = 0x7FFFFFFF;  // smallest column holding the tile's maximum (greedy verification)
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int col = tm * BM + sub + 8 * i;
        if (live && col < p.N) {
          s += exp2f((v[i] - mx) * kLog2e);
          if (v[i] == mx) arg = min(arg, col);
        }
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (e.argmax) {
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) arg = min(arg, __shfl_xor_sync(0xffffffffu, arg, o));
      }
      if (live && sub == 0) {
        e.stats[(long long)tm * e.stats_ld + r] = make_float2(mx, s);
        if (e.argmax) e.argmax[(long long)tm * e.stats_ld + r] = arg;
      }
    }
  }
}

// End of one output tile in the mma.sync kernels (4 consumer warps, each
// holding rows warp*32 .. +31 of the tile as two m16 fragments by NT/8 n8
// fragments).  A tile cut between CTAs is stored as a partial; the last CTA
// to arrive sums the pieces in CTA order and runs the epilogue, the others
// return.  A whole tile goes straight to the epilogue.
template <int EPI, int NT, int LD>
__device__ __forceinline__ void finish_tile_mma(const GemmParams& p, float (&acc)[2][NT / 8][4], int tile, int k0,
                                                int k1, long long total, long long u_begin, float* epi,
                                                volatile int* flag) {
  constexpr int NF = NT / 8;
  constexpr int NTHREADS = 4 * kWarp;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int P = gridDim.x, c = blockIdx.x;
  const int tm = tile / p.n_tiles, tn = tile - tm * p.n_tiles;
  if (!(k0 == 0 && k1 == p.kb)) {
    const long long tu = (long long)tile * p.kb;
    const int c_first = cta_of_unit(tu, total, P);
    const int c_last = cta_of_unit(tu + p.kb - 1, total, P);
    const int my_slot = 2 * c + (tile == static_cast<int>(u_begin / p.kb) ? 0 : 1);
    float4* dst = reinterpret_cast<float4*>(p.partials + (size_t)my_slot * BM * NT);
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int nj = 0; nj < NF; ++nj)
        __stcg(&dst[((warp * 2 + mi) * NF + nj) * 32 + lane],
               make_float4(acc[mi][nj][0], acc[mi][nj][1], acc[mi][nj][2], acc[mi][nj][3]));
    __threadfence();
    named_sync(1, NTHREADS);
    if (threadIdx.x == 0) {
      const int old = atomicAdd(&p.counters[tile], 1);
      *flag = (old == c_last - c_first) ? 1 : 0;
    }
    named_sync(1, NTHREADS);
    if (*flag == 0) return;
    __threadfence();
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int nj = 0; nj < NF; ++nj)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[mi][nj][q] = 0.f;
    // pieces are summed in CTA order; the loads of up to four pieces are issued together
    for (int c0 = c_first; c0 <= c_last; c0 += 4) {
      float4 v[4][2][NF];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int cc = c0 + q;
        if (cc <= c_last) {
          const int first_tile_cc = static_cast<int>(((long long)cc * total / P) / p.kb);
          const int slot = 2 * cc + (tile == first_tile_cc ? 0 : 1);
          const float4* src = reinterpret_cast<const float4*>(p.partials + (size_t)slot * BM * NT);
#pragma unroll
          for (int mi = 0; mi < 2; ++mi)
#pragma unroll
            for (int nj = 0; nj < NF; ++nj) v[q][mi][nj] = __ldcg(&src[((warp * 2 + mi) * NF + nj) * 32 + lane]);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (c0 + q <= c_last) {
#pragma unroll
          for (int mi = 0; mi < 2; ++mi)
#pragma unroll
            for (int nj = 0; nj < NF; ++nj) {
              acc[mi][nj][0] += v[q][mi][nj].x;
              acc[mi][nj][1] += v[q][mi][nj].y;
              acc[mi][nj][2] += v[q][mi][nj].z;
              acc[mi][nj][3] += v[q][mi][nj].w;
            }
        }
      }
    }
    if (threadIdx.x == 0) p.counters[tile] = 0;  // ready for the next launch
  }
  // fused epilogue from the tile staged in shared memory
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int nj = 0; nj < NF; ++nj) {
      const int m = warp * 32 + mi * 16 + g;
      const int n = nj * 8 + 2 * t;
      epi[n * LD + m] = acc[mi][nj][0];
      epi[(n + 1) * LD + m] = acc[mi][nj][1];
      epi[n * LD + m + 8] = acc[mi][nj][2];
      epi[(n + 1) * LD + m + 8] = acc[mi][nj][3];
    }
  named_sync(1, NTHREADS);
  epilogue_rows<EPI, LD>(p, epi, tm, tn * NT, min(NT, p.R - tn * NT), threadIdx.x);
  named_sync(1, NTHREADS);
}

// A CTA's part of a tile cut between CTAs in the tcgen05 kernels: four
// epilogue warps, thread m = weight row m; the part is stored column-major in
// the CTA's partial slot, [column][128 weight rows], so that each warp's 32
// rows of one column are 128 contiguous bytes.
__device__ __forceinline__ void tc_store_part16(float* slot_base, int c0, int m, const float (&v)[16]) {
#pragma unroll
  for (int n = 0; n < 16; ++n) __stcg(slot_base + (size_t)(c0 + n) * BM + m, v[n]);
}

// Fixup of a tile cut between CTAs in the tcgen05 kernels, run by the CTA
// that arrives last: the parts of CTAs c_first .. c_last are summed in CTA
// order, 16 columns at a time, and each 16-column chunk goes through the fused
// epilogue.  The loads of up to four parts are issued together, and the next
// chunk's first loads are in flight while the current chunk's epilogue runs.
template <int EPI, int LD>
__device__ __forceinline__ void tc_fixup_tile(const GemmParams& p, int tile, int c_first, int c_last,
                                              long long total, float* epi, int m, int rows, int nt) {
  const int P = gridDim.x;
  const int tm = tile / p.n_tiles, tn = tile - tm * p.n_tiles;
  auto src_of = [&](int cc, int c0) {
    const int first_tile_cc = static_cast<int>(((long long)cc * total / P) / p.kb);
    const int slot = 2 * cc + (tile == first_tile_cc ? 0 : 1);
    return p.partials + (size_t)slot * BM * nt + (size_t)c0 * BM + m;
  };
  auto issue = [&](float (&w)[4][16], int cc0, int c0) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (cc0 + q <= c_last) {
        const float* s = src_of(cc0 + q, c0);
#pragma unroll
        for (int n = 0; n < 16; ++n) w[q][n] = __ldcg(s + (size_t)n * BM);
      }
  };
  auto add = [&](float (&v)[16], const float (&w)[4][16], int cc0) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (cc0 + q <= c_last) {
#pragma unroll
        for (int n = 0; n < 16; ++n) v[n] += w[q][n];
      }
  };
  float w[4][16];
  issue(w, c_first, 0);
  for (int c0 = 0; c0 < rows; c0 += 16) {
    float v[16];
#pragma unroll
    for (int n = 0; n < 16; ++n) v[n] = 0.f;
    add(v, w, c_first);
    for (int cc0 = c_first + 4; cc0 <= c_last; cc0 += 4) {
      issue(w, cc0, c0);
      add(v, w, cc0);
    }
    if (c0 + 16 < rows) issue(w, c_first, c0 + 16);
#pragma unroll
    for (int n = 0; n < 16; ++n) epi[n * LD + m] = v[n];
    named_sync(1, 4 * kWarp);
    epilogue_rows<EPI, LD>(p, epi, tm, tn * nt + c0, min(16, rows - c0), m);
    named_sync(1, 4 * kWarp);
  }
}

}  // namespace gemm
}  // namespace sdv
