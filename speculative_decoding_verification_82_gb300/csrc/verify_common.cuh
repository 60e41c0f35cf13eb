// verify_common.cuh -- element formats, PTX wrappers (mbarrier, bulk TMA copies), warp
// reductions, row staging, and the finishing group's barriers, reductions and inverse-CDF search
// used by the verification kernel (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_verify.h"

namespace specv {

// ------------------------------------------------------------------ kernel geometry ----
// One CTA per SM, warp-specialised: two groups of eight consumer warps reduce staged chunks (the
// groups take alternate stages; four consumer warps per SM sub-partition hide the latency of the
// special-function unit), one producer warp per group claims work and drives the bulk copies,
// one bookkeeping warp publishes per-chunk results and counts them per request, and a group of
// four finishing warps (one per sub-partition) completes the requests assigned to this CTA.
constexpr int kConsWarps = 16;
constexpr int kGroups = 2;
constexpr int kGroupWarps = kConsWarps / kGroups;
constexpr int kProducerWarp = 16;  // and 17
constexpr int kBookWarp = 18;
constexpr int kFinWarp = 19;   // first of the finishing group's warps
constexpr int kFinWarps = 4;
constexpr int kFinThreads = kFinWarps * 32;
constexpr int kFinBarrier = 1;  // named barrier of the finishing group (0 is __syncthreads)
constexpr int kTagBarrier = 2;  // named barrier of every role but the producers, once the tag is set
constexpr int kThreads = (kFinWarp + kFinWarps) * 32;
constexpr int kStages = 6;                         // staged-chunk ring depth (a multiple of kGroups)
constexpr int kSlots = 16;                         // ring of per-chunk results (partials, merged)
constexpr int kClaim = 4;                          // work items claimed per atomic
constexpr int kChunkVec = 2048;                    // 16-byte vectors per chunk of a row (32 KB)
constexpr int kSubVec = kChunkVec / kGroupWarps;   // vectors per consumer warp (a sub-chunk)
constexpr int kVecPerLane = kSubVec / 32;
constexpr int kResVec = 1024;                      // target vectors per residual work item
constexpr int kResSub = kResVec / kGroupWarps;     // target vectors per consumer warp
constexpr int kDraftSlot = kResVec + 1;            // first slot of the draft range in a stage
constexpr int kStageVec = 2056;                    // >= kChunkVec and >= kDraftSlot + kResVec + 1
constexpr int kStageBytes = kStageVec * 16;
constexpr int kFinDraftSlot = kResSub + 1;         // finishing buffer: draft slot of a residual pair
constexpr int kFinVec = 264;                       // >= kSubVec and >= kFinDraftSlot + kResSub + 1
constexpr int kFinBytes = kFinVec * 16;
constexpr unsigned kFull = 0xffffffffu;
constexpr long long kWaitLimitCycles = 4000000000LL;  // ~2 s at GB300 clocks
static_assert(kVecPerLane * 32 == kSubVec && kResSub % 32 == 0, "warp split");
static_assert(kStageVec >= kChunkVec && kStageVec >= kDraftSlot + kResVec + 1, "stage size");
static_assert(kFinVec >= kSubVec && kFinVec >= kFinDraftSlot + kResSub + 1, "finishing buffer size");
static_assert(kSubVec <= 2 * kFinThreads && kResSub <= 2 * kFinThreads, "a staged sub-chunk is two vectors per finishing thread");
static_assert(kStageBytes % 128 == 0 && kFinBytes % 128 == 0, "alignment");
static_assert(kStages % kGroups == 0 && kSlots % kGroups == 0, "a stage and a slot always serve the same group");

// ------------------------------------------------------------------- element formats ----
// Each logits element type knows how to unpack a 16-byte vector into floats, how to take a
// NaN-propagating maximum over a packed word, and its -inf bit pattern (used as padding).
template <typename T>
struct Elem;

template <>
struct Elem<float> {
  static constexpr int kSize = 4, kPerVec = 4;
  static constexpr uint32_t kNegInf = 0xFF800000u;
  static constexpr uint32_t kNegInfWord = 0xFF800000u;
  __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ __forceinline__ static uint32_t load_raw(const char* p) {
    return __ldg(reinterpret_cast<const unsigned int*>(p));
  }
  __device__ __forceinline__ static void store_raw(unsigned char* p, uint32_t v) {
    *reinterpret_cast<uint32_t*>(p) = v;
  }
  __device__ __forceinline__ static float to_float(uint32_t raw) { return __uint_as_float(raw); }
  __device__ __forceinline__ static float smem_elem(const unsigned char* p) {
    return *reinterpret_cast<const float*>(p);
  }
  // NaN-propagating max of two packed words (one fp32 each)
  __device__ __forceinline__ static uint32_t max_word(uint32_t a, uint32_t b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(__uint_as_float(a)), "f"(__uint_as_float(b)));
    return __float_as_uint(r);
  }
  __device__ __forceinline__ static float word_max(uint32_t w) { return __uint_as_float(w); }
};

template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kSize = 2, kPerVec = 8;
  static constexpr uint32_t kNegInf = 0xFF80u;
  static constexpr uint32_t kNegInfWord = 0xFF80FF80u;
  __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  __device__ __forceinline__ static uint32_t load_raw(const char* p) {
    return __ldg(reinterpret_cast<const unsigned short*>(p));
  }
  __device__ __forceinline__ static void store_raw(unsigned char* p, uint32_t v) {
    *reinterpret_cast<uint16_t*>(p) = (uint16_t)v;
  }
  __device__ __forceinline__ static float to_float(uint32_t raw) { return __uint_as_float(raw << 16); }
  __device__ __forceinline__ static float smem_elem(const unsigned char* p) {
    return __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t*>(p)) << 16);
  }
  __device__ __forceinline__ static uint32_t max_word(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
  }
  __device__ __forceinline__ static float word_max(uint32_t w) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(__uint_as_float(w << 16)), "f"(__uint_as_float(w & 0xFFFF0000u)));
    return r;
  }
};

template <>
struct Elem<__half> {
  static constexpr int kSize = 2, kPerVec = 8;
  static constexpr uint32_t kNegInf = 0xFC00u;
  static constexpr uint32_t kNegInfWord = 0xFC00FC00u;
  __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  __device__ __forceinline__ static uint32_t load_raw(const char* p) {
    return __ldg(reinterpret_cast<const unsigned short*>(p));
  }
  __device__ __forceinline__ static void store_raw(unsigned char* p, uint32_t v) {
    *reinterpret_cast<uint16_t*>(p) = (uint16_t)v;
  }
  __device__ __forceinline__ static float to_float(uint32_t raw) {
    return __half2float(__ushort_as_half((unsigned short)raw));
  }
  __device__ __forceinline__ static float smem_elem(const unsigned char* p) {
    return __half2float(*reinterpret_cast<const __half*>(p));
  }
  __device__ __forceinline__ static uint32_t max_word(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.NaN.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
  }
  __device__ __forceinline__ static float word_max(uint32_t w) {
    const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w));
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(t.x), "f"(t.y));
    return r;
  }
};

// ---------------------------------------------------------------------- PTX wrappers ----
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// 2^x on the special-function unit (subnormal results flush to zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ uint4 lds128(const unsigned char* p) { return *reinterpret_cast<const uint4*>(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n\tfence.proxy.async.shared::cta;" ::: "memory");
}
// Raises the transaction count of the current phase (no arrival).
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test of the phase of `bar` with parity `parity`.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase of `bar` with parity `parity`.  Gives up (returns false) after
// kWaitLimitCycles, or early once *abort is set.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort || clock64() - t0 > kWaitLimitCycles) return false;
  }
}
// mbar_wait by every lane of a warp, with one outcome for the whole warp (false if any lane gave
// up), so that the warp leaves together.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, const volatile int* abort) {
  return __all_sync(kFull, mbar_wait(bar, parity, abort));
}
// Bulk (non-tensor) TMA copy global -> this CTA's shared memory, completing on `bar`.
// Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void tma_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// The same copy with an L2 eviction priority for the lines it reads (a policy from l2_policy).
__device__ __forceinline__ void tma_load_1d_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}
// L2 eviction priorities of bulk copies: none (the default), evict-first (read once), or
// evict-last (read again soon).
enum L2Hint : int { kL2Normal = 0, kL2First = 1, kL2Last = 2 };
__device__ __forceinline__ uint64_t l2_policy(int hint) {
  uint64_t p;
  if (hint == kL2Last)
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  else
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ int ld_volatile(const int* p) { return *reinterpret_cast<const volatile int*>(p); }
// Load with acquire semantics at GPU scope: later reads see what the writer published before it
// released the value (no fence, so earlier stores of this thread need not drain first).
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Orders this thread's earlier generic-proxy accesses of global memory before its later
// async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
// The same for shared memory: earlier reads of a buffer before a bulk copy overwrites it.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// -------------------------------------------------------------------- reductions ----
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(kFull, v, o));
  return v;
}
__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmax_nan(v, __shfl_xor_sync(kFull, v, o));
  return v;
}
__device__ __forceinline__ int warp_min_i(int v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(kFull, v, o));
  return v;
}
__device__ __forceinline__ int warp_or(int v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v |= __shfl_xor_sync(kFull, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}
__device__ __forceinline__ double warp_incl_scan_d(double v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double t = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += t;
  }
  return v;
}
// Inclusive prefix sum across the warp (Kogge-Stone), fixed association.
__device__ __forceinline__ float warp_incl_scan(float v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v = __fadd_rn(v, t);
  }
  return v;
}
// ------------------------------------------------------------- exponent arithmetic ----
// An exponent as an unevaluated fp32 pair hi + lo, |lo| far below one unit of hi's last place
// plus a few such units: fp32 arithmetic that keeps the digits a double would (GB300's FP64
// operations take tens of cycles each).
struct Exp2 {
  float hi, lo;
};
// a + b = s + err exactly (Knuth's two-sum).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& err) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}
// l c - mc with the product l c carried exactly (an fp32 pair from one FMA) and the difference as
// a two-sum: the exponent of 2^(l c - mc) must not lose the digits that a large |l c| would round
// away in plain fp32.
__device__ __forceinline__ Exp2 scaled_logit(float l, float c, float mc) {
  const float p = __fmul_rn(l, c);
  const float e = __fmaf_rn(l, c, -p);  // l c = p + e exactly
  Exp2 x;
  float r;
  two_sum(p, -mc, x.hi, r);
  x.lo = __fadd_rn(r, e);
  return x;
}
__device__ __forceinline__ Exp2 exp2_sub(const Exp2& a, const Exp2& b) {
  Exp2 x;
  float r;
  two_sum(a.hi, -b.hi, x.hi, r);
  x.lo = __fadd_rn(r, __fsub_rn(a.lo, b.lo));
  return x;
}
// 2^x * f for x = hi + lo and fp32 f > 0, in fp32: the integer part of hi as an exact power of
// two, the rest (hi minus its floor, exact, plus lo) through the special-function unit.
// Saturates to +inf / 0.
__device__ __forceinline__ float exp2_times(const Exp2& x, float f) {
  if (!(x.hi > -300.f)) return 0.f;
  if (x.hi > 300.f) return INFINITY;
  const float n = floorf(x.hi);
  const float r = __fmul_rn(ex2(__fadd_rn(__fsub_rn(x.hi, n), x.lo)), f);  // in (0, 2) * f
  return ldexpf(r, (int)n);
}

// ------------------------------------------------------------------------ row staging ----
// A logits row is read as a grid of 16-byte vectors starting at the row's address rounded down to
// 16 bytes: grid vector v holds elements v * VE - phase .. v * VE - phase + VE - 1, where phase is
// the number of elements of the first vector that precede the row.  Vectors lying wholly inside
// the row go by one bulk TMA copy; the (at most two) vectors that straddle the row's start or end
// are read element by element, with -inf in the positions outside the row.
template <typename T>
struct RowGrid {
  const char* grid;  // 16-byte aligned address of grid vector 0
  int phase;         // elements of vector 0 before the row start
  int nvec;          // vectors covering the row
};
template <typename T>
__device__ __forceinline__ RowGrid<T> row_grid(const char* row, int V) {
  constexpr int S = Elem<T>::kSize, VE = Elem<T>::kPerVec;
  RowGrid<T> g;
  const uintptr_t a = (uintptr_t)row;
  g.grid = row - (a & 15u);
  g.phase = (int)((a & 15u) / S);
  g.nvec = (g.phase + V + VE - 1) / VE;
  return g;
}

// Stages grid vectors [v0, v1) of a row (V elements) at `dst`, one warp.  Lane 0 raises the
// transaction count of `bar` and issues the bulk copy (with L2 eviction priority `hint`); the
// lanes fill the straddling vectors with plain loads.  The caller arrives on `bar` after a
// __syncwarp().
template <typename T>
__device__ __forceinline__ void warp_stage(unsigned char* dst, const RowGrid<T>& g, int V, int v0, int v1,
                                           uint64_t* bar, int lane, int hint = kL2Normal) {
  constexpr int S = Elem<T>::kSize, VE = Elem<T>::kPerVec;
  if (v1 <= v0) return;
  const int fa = g.phase > 0 ? 1 : 0;
  const int fb = (g.phase + V) / VE;  // vectors [fa, fb) lie wholly inside the row
  const int a = max(v0, fa), e = min(v1, fb);
  if (a < e && lane == 0) {
    const uint32_t bytes = (uint32_t)(e - a) * 16u;
    mbar_expect_tx(bar, bytes);
    if (hint == kL2Normal)
      tma_load_1d(dst + (size_t)(a - v0) * 16, g.grid + (size_t)a * 16, bytes, bar);
    else
      tma_load_1d_hint(dst + (size_t)(a - v0) * 16, g.grid + (size_t)a * 16, bytes, bar, l2_policy(hint));
  }
  // straddling vectors: grid vector 0 when the row starts mid-vector, grid vector fb when it
  // ends mid-vector
  const int first = (fa == 1 && v0 == 0) ? 0 : -1;
  int last = (fb < g.nvec && fb >= v0 && fb < v1) ? fb : -1;
  if (last == first) last = -1;  // a row inside one vector: the first pass fills it
  if (lane < 2 * VE) {
    const int rv = lane < VE ? first : last;
    const int j = lane % VE;
    if (rv >= 0) {
      const int el = rv * VE + j - g.phase;
      const uint32_t raw =
          (el >= 0 && el < V) ? Elem<T>::load_raw(g.grid + (size_t)g.phase * S + (size_t)el * S) : Elem<T>::kNegInf;
      Elem<T>::store_raw(dst + (size_t)(rv - v0) * 16 + (size_t)j * S, raw);
    }
  }
}

// ------------------------------------------------------------------ finishing group ----
// The kFinWarps finishing warps synchronise on named barrier kFinBarrier.
__device__ __forceinline__ int fin_thread() { return (int)threadIdx.x - kFinWarp * 32; }
__device__ __forceinline__ void fin_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(kFinBarrier), "n"(kFinThreads) : "memory");
}
// The group's barrier, returning the AND of every thread's predicate (a uniform decision).
__device__ __forceinline__ bool fin_all(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred a, b;\n\t"
      "setp.ne.u32 a, %1, 0;\n\t"
      "bar.red.and.pred b, %2, %3, a;\n\t"
      "selp.u32 %0, 1, 0, b;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)p), "n"(kFinBarrier), "n"(kFinThreads)
      : "memory");
  return r != 0;
}
// True in every thread once the leader has waited longer than the limit since t0: a retry loop
// of the group must be left by all its threads together (threads that took different ways would
// meet different barrier instructions), so the leader's clock decides for all.
__device__ __forceinline__ bool fin_timed_out(long long t0) {
  return !fin_all(!(fin_thread() == 0 && clock64() - t0 > kWaitLimitCycles));
}
// Shared-memory scratch of the group's reductions and broadcasts.
struct GroupScratch {
  float wsum[kFinWarps];
  unsigned hit[kFinWarps], pos[kFinWarps];
  int out[4];
  float fout[4];
};
// Sum over the group's threads in a fixed association (each warp's butterfly sum, then the warps
// in order); every thread gets it.
__device__ __forceinline__ float group_sum(GroupScratch& gs, float v) {
  const int ft = fin_thread(), lane = ft & 31, fw = ft >> 5;
  v = warp_sum(v);
  if (lane == 0) gs.wsum[fw] = v;
  fin_sync();
  float s = gs.wsum[0];
#pragma unroll
  for (int w = 1; w < kFinWarps; ++w) s = __fadd_rn(s, gs.wsum[w]);
  fin_sync();
  return s;
}

// ---------------------------------------------------------------- inverse-CDF search ----
// The finishing group finds, in a staged range of `nvec` vectors (nvec <= 2 * kFinThreads), the
// element where the running weight taken in index order first exceeds t; wf(v, w) fills the VE
// weights of vector v.  Thread i sums q = ceil(nvec / kFinThreads) consecutive vectors; a scan of
// the thread sums (each warp, then the warps in order) picks the crossing thread, which walks its
// vectors, then the elements of the chosen vector.  At every level the first part with positive
// weight whose running total exceeds t is taken, otherwise the last part with positive weight
// (rounding), so a zero-weight element is never returned.  Returns the position (vector * VE +
// element) in every thread, or -1 when the range holds no positive weight.
template <int VE, typename WF>
__device__ int group_crossing(GroupScratch& gs, int nvec, float t, WF wf) {
  const int ft = fin_thread(), lane = ft & 31, fw = ft >> 5;
  if (nvec <= 0) return -1;
  const int q = (nvec + kFinThreads - 1) / kFinThreads;
  const int v0 = ft * q;
  float s = 0.f;
  for (int i = 0; i < q; ++i) {
    const int v = v0 + i;
    if (v < nvec) {
      float w[VE];
      wf(v, w);
      float vs = 0.f;
#pragma unroll
      for (int j = 0; j < VE; ++j) vs = __fadd_rn(vs, w[j]);
      s = __fadd_rn(s, vs);
    }
  }
  const float incl = warp_incl_scan(s, lane);
  float excl = __shfl_up_sync(kFull, incl, 1);
  if (lane == 0) excl = 0.f;
  if (lane == 31) gs.wsum[fw] = incl;
  fin_sync();
  float base = 0.f;
  for (int w = 0; w < fw; ++w) base = __fadd_rn(base, gs.wsum[w]);
  const unsigned hit = __ballot_sync(kFull, s > 0.f && __fadd_rn(base, incl) > t);
  const unsigned pos = __ballot_sync(kFull, s > 0.f);
  if (lane == 0) {
    gs.hit[fw] = hit;
    gs.pos[fw] = pos;
  }
  fin_sync();
  int L = -1;
#pragma unroll
  for (int w = 0; w < kFinWarps; ++w)
    if (L < 0 && gs.hit[w]) L = w * 32 + __ffs(gs.hit[w]) - 1;
#pragma unroll
  for (int w = kFinWarps - 1; w >= 0; --w)
    if (L < 0 && gs.pos[w]) L = w * 32 + 31 - __clz(gs.pos[w]);
  if (ft == L) {
    // the thread's vectors in order, then the elements of the chosen vector
    float acc = __fadd_rn(base, excl);
    int pv = -1, lv = -1;
    float pacc = 0.f, lacc = 0.f;
    for (int i = 0; i < q; ++i) {
      const int v = v0 + i;
      if (v >= nvec) break;
      float w[VE];
      wf(v, w);
      float vs = 0.f;
#pragma unroll
      for (int j = 0; j < VE; ++j) vs = __fadd_rn(vs, w[j]);
      if (vs > 0.f) {
        if (pv < 0 && __fadd_rn(acc, vs) > t) {
          pv = v;
          pacc = acc;
        }
        lv = v;
        lacc = acc;
      }
      acc = __fadd_rn(acc, vs);
    }
    if (pv < 0) {
      pv = lv;
      pacc = lacc;
    }
    float w[VE];
    wf(pv, w);
    float r2 = 0.f;
    int pj = -1, lj = -1;
#pragma unroll
    for (int j = 0; j < VE; ++j) {
      r2 = __fadd_rn(r2, w[j]);
      if (w[j] > 0.f) {
        if (pj < 0 && __fadd_rn(pacc, r2) > t) pj = j;
        lj = j;
      }
    }
    gs.out[3] = pv * VE + (pj >= 0 ? pj : lj);
  }
  fin_sync();
  const int found = L < 0 ? -1 : gs.out[3];
  fin_sync();
  return found;
}

}  // namespace specv
