// verify_common.cuh -- element formats, PTX wrappers, reductions, chunk staging and the
// inverse-CDF search shared by the verification kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_verify.h"

namespace specv {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxTiles = 32;  // tiles of 256 16-byte vectors: chunks up to 128 KB
constexpr unsigned kFull = 0xffffffffu;
constexpr long long kWaitLimitCycles = 4000000000LL;  // ~2 s at GB300 clocks

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
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n\tfence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
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
// Waits for phase `parity` of `bar`; gives up after kWaitLimitCycles and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
  return true;
}
// Bulk (non-tensor) TMA copy global -> this CTA's shared memory, completing on `bar`.
// Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void tma_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
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
// 2^x in double with fp32 relative accuracy (~3e-7): the integer part of x scales exactly, the
// fractional part goes through the special-function unit.  Avoids double-precision
// transcendentals, which are slow on this part.
__device__ __forceinline__ double exp2_split(double x) {
  if (!(x > -1070.0)) return x != x ? x : 0.0;
  if (x > 1020.0) return __longlong_as_double(0x7ff0000000000000LL);
  const double n = floor(x);
  return ldexp((double)ex2((float)(x - n)), (int)n);
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
// Block-wide reductions; every thread gets the same value.  `scratch` holds kWarps entries
// (2 * kWarps for block_sum2).
__device__ __forceinline__ float block_max_nan(float v, float* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max_nan(v);
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  float r = scratch[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) r = fmax_nan(r, scratch[w]);
  __syncthreads();
  return r;
}
__device__ __forceinline__ void block_sum2(float& a, float& b, float* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  a = warp_sum(a);
  b = warp_sum(b);
  if (lane == 0) {
    scratch[warp] = a;
    scratch[kWarps + warp] = b;
  }
  __syncthreads();
  float ra = scratch[0], rb = scratch[kWarps];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) {
    ra = __fadd_rn(ra, scratch[w]);
    rb = __fadd_rn(rb, scratch[kWarps + w]);
  }
  __syncthreads();
  a = ra;
  b = rb;
}
__device__ __forceinline__ int block_min_i(int v, int* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_min_i(v);
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  int r = scratch[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) r = min(r, scratch[w]);
  __syncthreads();
  return r;
}

// ------------------------------------------------------------------- chunk staging ----
// A chunk is the element range [e0, e0 + n) of one logits row, staged in shared memory as whole
// 16-byte vectors.  Element e0 sits at slot `slot0`, chosen so that a slot's shared-memory address
// has the same 16-byte phase as the element's global address (then the whole vectors inside the
// chunk can come by one bulk TMA copy).  Slots outside [e0, e0 + n) hold -inf.
struct Geo {
  int e0, n, slot0, nvec;
};

template <typename T>
__device__ __forceinline__ Geo make_geo(const char* row, int e0, int n) {
  constexpr int S = Elem<T>::kSize, VE = Elem<T>::kPerVec;
  Geo g;
  g.e0 = e0;
  g.n = n;
  g.slot0 = (int)((((uintptr_t)row + (size_t)e0 * S) & 15u) / S);
  g.nvec = n > 0 ? (g.slot0 + n + VE - 1) / VE : 0;
  return g;
}

// Issues the loads of chunk `g` of `row` into `buf` (laid out with g.slot0).  The whole vectors
// go by one TMA copy when the row's phase matches the layout, the rest by plain loads of all
// threads.  Thread 0 always arrives once on `bar` (expecting 0 bytes when nothing goes by TMA),
// so every issue completes exactly one phase of `bar`.
template <typename T>
__device__ __forceinline__ void issue_chunk(unsigned char* buf, const char* row, const Geo& g, uint64_t* bar,
                                            uint64_t pol) {
  constexpr int S = Elem<T>::kSize, VE = Elem<T>::kPerVec;
  const char* p = row + (size_t)g.e0 * S;
  const bool phase_ok = (int)(((uintptr_t)p & 15u) / S) == g.slot0;
  int vA = g.slot0 > 0 ? 1 : 0, vB = (g.slot0 + g.n) / VE;
  if (g.n <= 0 || vB <= vA || !phase_ok) vA = vB = 0;
  const uint32_t bytes = (uint32_t)(vB - vA) * 16u;
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(bar, bytes);
    if (bytes) tma_load_1d(buf + vA * 16, p + (ptrdiff_t)(vA * VE - g.slot0) * S, bytes, bar, pol);
  }
  // plain loads: everything when no TMA copy, else only the (at most two) ragged end vectors
  const int total = g.nvec * VE;
  const int head = bytes ? vA * VE : total;
  const int tail0 = bytes ? vB * VE : total;
  const int nplain = head + (total - tail0);
  for (int i = (int)threadIdx.x; i < nplain; i += kThreads) {
    const int s = i < head ? i : tail0 + (i - head);
    const int e = s - g.slot0;
    const uint32_t raw = (e >= 0 && e < g.n) ? Elem<T>::load_raw(p + (ptrdiff_t)e * S) : Elem<T>::kNegInf;
    Elem<T>::store_raw(buf + (size_t)s * S, raw);
  }
}

// NaN-propagating maximum of this thread's vectors of a staged chunk (padding is -inf).
template <typename T>
__device__ __forceinline__ float thread_max(const unsigned char* buf, int nvec) {
  using E = Elem<T>;
  uint32_t m0 = E::kNegInfWord, m1 = E::kNegInfWord;
  for (int v = (int)threadIdx.x; v < nvec; v += kThreads) {
    const uint4 w = *reinterpret_cast<const uint4*>(buf + (size_t)v * 16);
    m0 = E::max_word(m0, E::max_word(w.x, w.y));
    m1 = E::max_word(m1, E::max_word(w.z, w.w));
  }
  return E::word_max(E::max_word(m0, m1));
}

// ---------------------------------------------------------------- inverse-CDF search ----
// Finds in a staged chunk the element where the running weight, taken in index order, first
// exceeds `t`; `wf(v, w)` fills the weights of vector v.  The search is hierarchical: tiles of
// 256 vectors -> warps of 32 vectors -> the lane's vector -> its elements.  At each level it
// takes the first part with positive weight whose running total exceeds t, otherwise the last
// part with positive weight (rounding), so a zero-weight element is never returned.  Returns the
// element's vocabulary index in every thread, or -1 when the chunk holds no positive weight.
template <int VE, typename WF>
__device__ int chunk_crossing(const Geo& g, float t, WF wf, float (*tileW)[kWarps], int* s_int, float* s_flt) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ntiles = (g.nvec + kThreads - 1) / kThreads;
  for (int j = 0; j < ntiles; ++j) {
    const int v = j * kThreads + (int)threadIdx.x;
    float vs = 0.f;
    if (v < g.nvec) {
      float w[VE];
      wf(v, w);
      vs = w[0];
#pragma unroll
      for (int q = 1; q < VE; ++q) vs = __fadd_rn(vs, w[q]);
    }
    const float incl = warp_incl_scan(vs, lane);
    if (lane == 31) tileW[j][warp] = incl;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float run = 0.f, pickR = 0.f, lastR = 0.f;
    int pick = -1, last = -1;
    for (int q = 0; q < ntiles * kWarps; ++q) {
      const float W = tileW[q / kWarps][q % kWarps];
      if (W > 0.f) {
        const float nxt = __fadd_rn(run, W);
        if (nxt > t) {
          pick = q;
          pickR = run;
          break;
        }
        last = q;
        lastR = run;
        run = nxt;
      }
    }
    if (pick < 0) {
      pick = last;
      pickR = lastR;
    }
    s_int[0] = pick;
    s_int[1] = -1;
    s_flt[0] = pickR;
  }
  __syncthreads();
  const int pick = s_int[0];
  const float pickR = s_flt[0];
  if (pick >= 0 && warp == pick % kWarps) {
    const int v = (pick / kWarps) * kThreads + warp * 32 + lane;
    float w[VE];
    float vs = 0.f;
    if (v < g.nvec) {
      wf(v, w);
      vs = w[0];
#pragma unroll
      for (int q = 1; q < VE; ++q) vs = __fadd_rn(vs, w[q]);
    } else {
#pragma unroll
      for (int q = 0; q < VE; ++q) w[q] = 0.f;
    }
    const float incl = warp_incl_scan(vs, lane);
    float excl = __shfl_up_sync(kFull, incl, 1);
    if (lane == 0) excl = 0.f;
    const float end = __fadd_rn(pickR, incl);
    const unsigned hit = __ballot_sync(kFull, vs > 0.f && end > t);
    const unsigned pos = __ballot_sync(kFull, vs > 0.f);
    const int L = hit ? (__ffs(hit) - 1) : (pos ? 31 - __clz(pos) : -1);
    if (lane == L) {
      const float acc = __fadd_rn(pickR, excl);
      float run = 0.f;
      int pj = -1, lj = -1;
#pragma unroll
      for (int q = 0; q < VE; ++q) {
        run = __fadd_rn(run, w[q]);
        if (w[q] > 0.f) {
          if (pj < 0 && __fadd_rn(acc, run) > t) pj = q;
          lj = q;
        }
      }
      if (pj < 0) pj = lj;
      s_int[1] = g.e0 - g.slot0 + v * VE + pj;
    }
  }
  __syncthreads();
  const int tok = s_int[1];
  __syncthreads();
  return tok;
}

}  // namespace specv
