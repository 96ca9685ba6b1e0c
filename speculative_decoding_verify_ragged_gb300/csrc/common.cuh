// Device helpers shared by the verify-step kernels (sm_103a).
//
// Inline PTX wrappers for shared-memory mbarriers, TMA tensor loads
// (cp.async.bulk.tensor, no multicast), ldmatrix and the bf16 mma.sync
// tensor-core instruction, plus small numeric helpers.  Every wait on an
// mbarrier is bounded in time: on expiry it reports failure to the caller,
// which records SDV_ERR_TIMEOUT in the status word and returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sdv.h"

namespace sdv {

constexpr int kWarp = 32;

// ---------------------------------------------------------------------------
// status word
// ---------------------------------------------------------------------------

// First error wins; later errors of the same call are dropped.
__device__ __forceinline__ void set_status(int* status, int code) {
  atomicCAS(status, 0, code);
}

__device__ __forceinline__ int read_status(const int* status) {
  return *reinterpret_cast<const volatile int*>(status);
}

// ---------------------------------------------------------------------------
// addresses and timers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Arrive `count` times at once (one thread standing in for several expected arrivals).
__device__ __forceinline__ void mbar_arrive_count(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up after
// `limit_ns` nanoseconds (default 2 s, far beyond any legal wait here).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint64_t limit_ns = 2000000000ull) {
  const uint32_t addr = smem_u32(bar);
  if (mbar_try_wait(addr, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(addr, parity)) return true;
    if ((i & 255u) == 255u && global_timer_ns() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------------------------
// TMA (tensor) loads into shared memory, completion on an mbarrier
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, "
      "%4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_5d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2,
                                            int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6, "
      "%7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------
// ldmatrix / mma.sync (bf16 in, fp32 accumulate)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------
// programmatic dependent launch: every kernel of the step lets the next one
// start as soon as SM resources free up, and waits for the previous one only
// where it reads what that one wrote
// ---------------------------------------------------------------------------

__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// step timeline (builds with -DSDV_TRACE only; other builds compile the
// stamps away).  Each kernel launch stamps the global timer into its slot of
// a device table of kTraceSlots x 3 64-bit words: the earliest CTA's entry,
// the earliest warp past its wait for the kernel ahead, and the latest warp's
// exit.  The table's address is a per-translation-unit constant set through
// the unit's trace_set_<unit>() (SDV_TRACE_UNIT); null disables the stamps.
// ---------------------------------------------------------------------------

constexpr int kTraceSlots = 32;
enum TraceSlot {
  kTrPrologue = 0, kTrQkv = 1, kTrAttention = 2, kTrMerge = 3, kTrO = 4, kTrGateUp = 5, kTrDown = 6,
  kTrFinalNorm = 7, kTrLmHead = 8, kTrAccept = 9, kTrSample = 10, kTrRealign = 11, kTrProbs = 12,
  kTrAdmit = 13, kTrPlanes = 14, kTrLinear = 15, kTrFixup = 16  // kTrFixup + the GEMM's own slot
};

#ifdef SDV_TRACE
static __constant__ unsigned long long* c_trace;

__device__ __forceinline__ unsigned long long trace_clock() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

struct TraceScope {
  int slot;
  __device__ explicit TraceScope(int s) : slot(s) {
    if (c_trace && threadIdx.x == 0) atomicMin(&c_trace[3 * slot], trace_clock());
  }
  __device__ ~TraceScope() {
    if (c_trace && (threadIdx.x & 31) == 0) atomicMax(&c_trace[3 * slot + 2], trace_clock());
  }
};

__device__ __forceinline__ void trace_wait(int slot) {
  if (c_trace && (threadIdx.x & 31) == 0) atomicMin(&c_trace[3 * slot + 1], trace_clock());
}

#define SDV_TRACE_SCOPE(slot_expr)          \
  const int sdv_trace_slot_ = (slot_expr); \
  ::sdv::TraceScope sdv_trace_scope_(sdv_trace_slot_)
#define SDV_GRIDDEP_WAIT()                   \
  do {                                       \
    ::sdv::griddep_wait();                   \
    ::sdv::trace_wait(sdv_trace_slot_);      \
  } while (0)
#define SDV_TRACE_UNIT(unit)                                          \
  cudaError_t trace_set_##unit(unsigned long long* table) {           \
    return cudaMemcpyToSymbol(c_trace, &table, sizeof(table));        \
  }
#else
#define SDV_TRACE_SCOPE(slot_expr) \
  do {                             \
  } while (0)
#define SDV_GRIDDEP_WAIT() ::sdv::griddep_wait()
#define SDV_TRACE_UNIT(unit)
#endif

// The timeline slot of a GEMM launch, from its epilogue (the two residual
// GEMMs told apart by the RMSNorm that only the O projection feeds).
#define SDV_GEMM_SLOT(kind, params)                                                          \
  ((kind) == EPI_QKV      ? ::sdv::kTrQkv                                                    \
   : (kind) == EPI_SWIGLU ? ::sdv::kTrGateUp                                                 \
   : (kind) == EPI_LMHEAD ? ::sdv::kTrLmHead                                                 \
   : (kind) == EPI_RESID  ? ((params).epi.norm_gain ? ::sdv::kTrO : ::sdv::kTrDown)          \
                          : ::sdv::kTrLinear)

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// Consumer-only named barrier (id 1..15) over `n` threads.
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// ---------------------------------------------------------------------------
// numerics
// ---------------------------------------------------------------------------

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ __nv_bfloat16 f2bf(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// x ~= hi + lo with hi = bf16(x) and lo = bf16(x - hi), packed in pairs.
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
  const __nv_bfloat16 l0 = __float2bfloat16_rn(x0 - __bfloat162float(h0));
  const __nv_bfloat16 l1 = __float2bfloat16_rn(x1 - __bfloat162float(h1));
  __nv_bfloat162 hv(h0, h1), lv(l0, l1);
  hi = *reinterpret_cast<uint32_t*>(&hv);
  lo = *reinterpret_cast<uint32_t*>(&lv);
}

// x ~ hi + lo stored in two bf16 planes lo_off elements apart (lo_off == 0: hi only)
__device__ __forceinline__ void store_planes(__nv_bfloat16* hi, long long lo_off, long long idx, float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  hi[idx] = h;
  if (lo_off) hi[idx + lo_off] = __float2bfloat16_rn(x - __bfloat162float(h));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

constexpr float kLog2e = 1.4426950408889634f;

// Merge two softmax partial states (max M, sum of exp(z - M)) into one.
__device__ __forceinline__ void merge_ms(float& M, float& S, float oM, float oS) {
  const float nm = fmaxf(M, oM);
  S = (M == -INFINITY ? 0.f : S * exp2f((M - nm) * kLog2e)) + (oM == -INFINITY ? 0.f : oS * exp2f((oM - nm) * kLog2e));
  M = nm;
}

}  // namespace sdv
