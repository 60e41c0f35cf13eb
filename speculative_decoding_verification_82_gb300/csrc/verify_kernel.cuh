// verify_kernel.cuh -- the verification kernels (sm_103a).
//
// stats_kernel (every call).  A persistent grid streams every logits row once, in chunks of
// ~32 KB staged in shared memory by bulk TMA copies through a two-stage ring per CTA (the next
// chunk is in flight while the current one is reduced).  Per chunk it records either the chunk
// maximum m_c and s_c = sum 2^(l c - m_c c) (temperature softmax, c = log2(e)/T, in the
// online-softmax form so chunks combine exactly), or the chunk's (max, first index) for greedy
// modes.  Work items are ordered request-major; the CTA that completes a request's last chunk
// (an atomic ticket, never a spin) finishes that request: it combines the chunk statistics into
// (m, Z) per row, computes alpha_k = min(1, p_k(x_k)/q_k(x_k)) in double, runs the acceptance
// scan, and draws the emitted token by inverse CDF for the bonus row and the n-gram residual (it
// knows the per-chunk weights, so it re-reads only the one chunk holding the crossing), or takes
// the argmax (greedy chain), or walks the draft tree.
//
// residual_kernel (draft-model chain with T > 0 only).  For a request rejected at position n the
// weights max(0, p_n - q_n) need both rows' global statistics, so this second launch reads the
// pair at n once more, chunk by chunk, and sums the residual per chunk; the last chunk's CTA
// re-reads the crossing chunk and draws the token.
//
// probs_kernel (testing only) writes the normalised p / q rows.
//
// Formulas: "Speculative Decoding in Production: From Draft Models to EAGLE-3 Dynamic Trees for
// 3x-5x Lossless Acceleration", section I.1 (acceptance ratio, uniform test, first-rejection
// stop, normalised positive residual); section III.2 (tree path acceptance).
#pragma once

#include <climits>

#include "verify_common.cuh"

namespace specv {

enum Mode : int { kChain = 0, kNgram = 1, kGreedy = 2, kTree = 3 };
enum Kind : int { kFullP = 0, kExcl = 1, kResid = 2 };

// Per chunk of a logits row, written by stats_kernel.
struct __align__(16) ChunkStat {
  float a;   // chunk maximum
  float s;   // softmax: sum over the chunk of 2^(l c - a c)
  float sx;  // softmax, n-gram target rows: the same sum without the draft token; else = s
  int i;     // softmax: SPEC_ERRF_* bits; argmax modes: first index of the maximum (-1: NaN)
};
// Per logits row, written by the request's finishing CTA.
struct __align__(16) RowStat {
  double Z;  // sum over the row of 2^(l c - mc)
  float mc;  // fp32 product (row maximum) * c
  int err;   // SPEC_ERRF_* bits of the row
  int amax;  // argmax modes: row argmax
  int pad[3];
};
struct __align__(16) ReqState {
  int n;    // accepted prefix length
  int err;  // SPEC_ERRF_* bits
  int pad[2];
};
static_assert(sizeof(ChunkStat) == 16 && sizeof(RowStat) == 32 && sizeof(ReqState) == 16, "layout");

struct Params {
  const void* target;
  const void* draft;
  int B, K, V, R;     // R: target rows per request (K + 1, or N + 1 for trees)
  int rows;           // logits rows per request read by stats_kernel (draft-model chain: 2K + 1)
  int chunk, nchunk;  // elements per chunk (multiple of 8), chunks per row
  int buf_bytes;      // shared-memory bytes of one staged chunk
  int diag;           // 1: draw at every position (per-position outputs requested)
  float c;            // log2(e) / T
  const int32_t* draft_tokens;
  const float* r;
  const float* u;
  const int32_t* parents;
  const int32_t* node_tokens;
  int32_t* num_accepted;
  int32_t* out_tokens;
  float* residual_mass;
  int32_t* err_flags;
  float* accept_prob;
  int32_t* cand_tokens;
  float* pos_mass;
  float* target_probs;
  float* draft_probs;
  int32_t* accept_len;
  int32_t* path_nodes;
  int32_t* node_argmax;
  ChunkStat* cstat;  // [B][rows][nchunk]
  RowStat* rstat;    // [B][rows]
  ReqState* req;     // [B]
  float* wsum;       // [B][K][nchunk] (per-position outputs) or [B][nchunk]
  unsigned* work;    // work-item counter of stats_kernel (zeroed by the host before each call)
  unsigned* tick_a;  // [B] request tickets of stats_kernel (zeroed likewise)
  unsigned* tick_b;  // [B][K] or [B] tickets of residual_kernel (zeroed likewise)
  size_t tick_bytes; // bytes of the two ticket arrays (one contiguous region)
};

template <typename T>
__device__ __forceinline__ const char* row_ptr(const Params& P, int b, int r) {
  constexpr int S = Elem<T>::kSize;
  if (r < P.R) return static_cast<const char*>(P.target) + ((size_t)b * P.R + r) * (size_t)P.V * S;
  return static_cast<const char*>(P.draft) + ((size_t)b * P.K + (r - P.R)) * (size_t)P.V * S;
}
__device__ __forceinline__ int chunk_len(const Params& P, int ch) { return min(P.chunk, P.V - ch * P.chunk); }

// Weight of a chunk in units of the row normaliser: s (or sx) * 2^(RN(a c) - mc).
__device__ __forceinline__ double chunk_weight(float a, float s, float c, float mc) {
  if (a == -INFINITY) return 0.0;
  return (double)s * (double)ex2(__fsub_rn(__fmul_rn(a, c), mc));
}

// ------------------------------------------------------------------ chunk reductions ----
// Online-softmax partial: s (and sx) are sums of 2^(l c - RN(m c)) over the elements seen.
struct Soft {
  float m, s, sx;
};
// 2^(RN(m c) - RN(M c)): rescales a partial taken at maximum m to maximum M (0 when empty).
__device__ __forceinline__ float rescale(float m, float M, float c) {
  return m == -INFINITY ? 0.f : ex2(__fsub_rn(__fmul_rn(m, c), __fmul_rn(M, c)));
}
__device__ __forceinline__ Soft soft_merge(const Soft& a, const Soft& b, float c) {
  const float M = fmax_nan(a.m, b.m);
  if (M == -INFINITY) return a;  // both partials empty
  const float fa = rescale(a.m, M, c), fb = rescale(b.m, M, c);
  Soft r;
  r.m = M;
  r.s = __fmaf_rn(a.s, fa, __fmul_rn(b.s, fb));
  r.sx = __fmaf_rn(a.sx, fa, __fmul_rn(b.sx, fb));
  return r;
}

// This thread's softmax partial over its vectors of a staged chunk; sx leaves out slot (vx, jx).
template <typename T>
__device__ __forceinline__ Soft thread_softmax(const unsigned char* buf, int nvec, float c, int vx, int jx) {
  constexpr int VE = Elem<T>::kPerVec;
  Soft t;
  t.m = thread_max<T>(buf, nvec);
  t.s = t.sx = 0.f;
  if (!(t.m > -INFINITY && t.m < INFINITY)) return t;  // empty, +inf or NaN: the max tells
  const float mc = __fmul_rn(t.m, c);
  for (int v = (int)threadIdx.x; v < nvec; v += kThreads) {
    float f[VE];
    Elem<T>::unpack(*reinterpret_cast<const uint4*>(buf + (size_t)v * 16), f);
    float e[VE];
#pragma unroll
    for (int j = 0; j < VE; ++j) e[j] = ex2(__fmaf_rn(f[j], c, -mc));
    float vs = 0.f;
#pragma unroll
    for (int j = 0; j < VE; ++j) vs = __fadd_rn(vs, e[j]);
    t.s = __fadd_rn(t.s, vs);
    if (v == vx) {
      float vsx = 0.f;
#pragma unroll
      for (int j = 0; j < VE; ++j) vsx = __fadd_rn(vsx, j == jx ? 0.f : e[j]);
      t.sx = __fadd_rn(t.sx, vsx);
    } else {
      t.sx = __fadd_rn(t.sx, vs);
    }
  }
  return t;
}

// Softmax statistics of a staged chunk, merged thread -> warp (shuffles) -> block (thread 0).
// One block barrier.  The result is valid in thread 0 only.
template <typename T>
__device__ __forceinline__ ChunkStat chunk_softmax_stats(const unsigned char* buf, const Geo& g, float c, int vx,
                                                         int jx, float* red /*3*kWarps*/) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  Soft t = thread_softmax<T>(buf, g.nvec, c, vx, jx);
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    Soft u;
    u.m = __shfl_xor_sync(kFull, t.m, o);
    u.s = __shfl_xor_sync(kFull, t.s, o);
    u.sx = __shfl_xor_sync(kFull, t.sx, o);
    t = soft_merge(t, u, c);
  }
  if (lane == 0) {
    red[warp] = t.m;
    red[kWarps + warp] = t.s;
    red[2 * kWarps + warp] = t.sx;
  }
  __syncthreads();
  ChunkStat q;
  q.a = red[0];
  q.s = red[kWarps];
  q.sx = red[2 * kWarps];
  q.i = 0;
  if (threadIdx.x == 0) {
    Soft acc{red[0], red[kWarps], red[2 * kWarps]};
    for (int w = 1; w < kWarps; ++w) acc = soft_merge(acc, Soft{red[w], red[kWarps + w], red[2 * kWarps + w]}, c);
    q.a = acc.m;
    q.s = acc.s;
    q.sx = acc.sx;
    q.i = (isnan(acc.m) || acc.m == INFINITY) ? SPEC_ERRF_NONFINITE : 0;
    if (q.i) q.s = q.sx = 0.f;
  }
  return q;
}

// (max, first index) partials: index -1 marks a NaN, INT_MAX an empty partial.
__device__ __forceinline__ void argmax_merge(float& v, int& i, float v2, int i2) {
  if (i < 0 || i2 == INT_MAX) return;
  if (i2 < 0 || i == INT_MAX || v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

// (max, first index) of a staged chunk; index -1 when it holds a NaN.  One block barrier; the
// result is valid in thread 0 only.
template <typename T>
__device__ __forceinline__ ChunkStat chunk_argmax(const unsigned char* buf, const Geo& g, float* red, int* redi) {
  constexpr int VE = Elem<T>::kPerVec;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float v = thread_max<T>(buf, g.nvec);
  int idx = INT_MAX;
  if (isnan(v)) {
    idx = -1;
  } else {  // this thread's first element equal to its maximum (its vectors are in index order)
    for (int vv = (int)threadIdx.x; vv < g.nvec && idx == INT_MAX; vv += kThreads) {
      float f[VE];
      Elem<T>::unpack(*reinterpret_cast<const uint4*>(buf + (size_t)vv * 16), f);
#pragma unroll
      for (int j = 0; j < VE; ++j) {
        const int e = g.e0 - g.slot0 + vv * VE + j;
        if (idx == INT_MAX && e >= g.e0 && e < g.e0 + g.n && f[j] == v) idx = e;
      }
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float v2 = __shfl_xor_sync(kFull, v, o);
    const int i2 = __shfl_xor_sync(kFull, idx, o);
    argmax_merge(v, idx, v2, i2);
  }
  if (lane == 0) {
    red[warp] = v;
    redi[warp] = idx;
  }
  __syncthreads();
  ChunkStat q;
  q.a = red[0];
  q.i = redi[0];
  q.s = q.sx = 0.f;
  if (threadIdx.x == 0) {
    for (int w = 1; w < kWarps; ++w) argmax_merge(q.a, q.i, red[w], redi[w]);
    if (q.i == INT_MAX) q.i = -1;  // a chunk always holds at least one element
  }
  return q;
}

// ------------------------------------------------------------------ request finishing ----
struct FinishSmem {
  float (*tileW)[kWarps];
  int* s_int;
  float* s_flt;
  double* s_dbl;
  double* s_alpha;
  int* s_misc;
  uint64_t* bar_x;
  unsigned* xphase;
};

// Warp-wide inverse CDF over per-chunk weights W(c) (double), in chunk order: the first chunk
// with positive weight whose running total exceeds u * S, else the last positive one.  Every
// lane gets the chunk, the total weight before it and S.
template <typename WF>
__device__ __forceinline__ void chunk_select(int nchunk, double u, WF W, int& cstar, double& bstar, double& S) {
  const int lane = threadIdx.x & 31;
  double part = 0.0;
  for (int c = lane; c < nchunk; c += 32) part += W(c);
  S = warp_sum_d(part);
  const double tgt = u * S;
  double base = 0.0, blast = 0.0;
  int clast = -1;
  cstar = -1;
  bstar = 0.0;
  for (int c0 = 0; c0 < nchunk; c0 += 32) {
    const int cc = c0 + lane;
    const double w = cc < nchunk ? W(cc) : 0.0;
    const double incl = warp_incl_scan_d(w, lane);
    double ex = __shfl_up_sync(kFull, incl, 1);
    if (lane == 0) ex = 0.0;
    const unsigned hit = __ballot_sync(kFull, w > 0.0 && base + incl > tgt);
    const unsigned pos = __ballot_sync(kFull, w > 0.0);
    if (cstar < 0 && hit) {
      const int L = __ffs(hit) - 1;
      cstar = c0 + L;
      bstar = base + __shfl_sync(kFull, ex, L);
    }
    if (pos) {
      const int L = 31 - __clz(pos);
      clast = c0 + L;
      blast = base + __shfl_sync(kFull, ex, L);
    }
    base += __shfl_sync(kFull, incl, 31);
  }
  if (cstar < 0) {
    cstar = clast;
    bstar = blast;
  }
}

// Inverse-CDF draw for target row `row` of request b from its chunk statistics: weights p
// (kFullP) or p without token x (kExcl).  Finds the crossing chunk from the chunk weights, then
// stages that one chunk (into `buf`) and searches it.  Block-wide; every thread gets the token
// and the residual mass S / Z (taken before any zero-residual fallback).
template <typename T>
__device__ int draw_from_chunks(const Params& P, int b, int row, int kind, int x, unsigned char* buf,
                                const FinishSmem& F, float* mass_out) {
  constexpr int VE = Elem<T>::kPerVec;
  const RowStat rs = P.rstat[(size_t)b * P.rows + row];
  const ChunkStat* cs = P.cstat + ((size_t)b * P.rows + row) * P.nchunk;
  if (threadIdx.x < 32) {
    const double u = (double)__ldg(P.u + b);
    int cstar, k2 = kind;
    double bstar, S;
    auto weight = [&](int c) {
      return chunk_weight(__ldcg(&cs[c].a), k2 == kExcl ? __ldcg(&cs[c].sx) : __ldcg(&cs[c].s), P.c, rs.mc);
    };
    chunk_select(P.nchunk, u, weight, cstar, bstar, S);
    const double S0 = S;
    if (!(S > 0.0)) {  // no residual mass: draw from p
      k2 = kFullP;
      chunk_select(P.nchunk, u, weight, cstar, bstar, S);
    }
    if (threadIdx.x == 0) {
      F.s_misc[0] = cstar;
      F.s_misc[1] = k2;
      F.s_dbl[0] = u * S - bstar;
      F.s_dbl[1] = S0 / rs.Z;
    }
  }
  __syncthreads();
  const int cstar = F.s_misc[0], k2 = F.s_misc[1];
  const float t = (float)F.s_dbl[0];
  *mass_out = (float)F.s_dbl[1];
  if (cstar < 0) return -1;
  const char* rp = row_ptr<T>(P, b, row);
  const Geo g = make_geo<T>(rp, cstar * P.chunk, chunk_len(P, cstar));
  issue_chunk<T>(buf, rp, g, F.bar_x, l2_policy_evict_first());
  bool ok = mbar_wait_bounded(F.bar_x, *F.xphase & 1u);
  if (!ok) ok = mbar_wait_bounded(F.bar_x, *F.xphase & 1u);
  __syncthreads();
  if (threadIdx.x == 0) ++*F.xphase;
  const float c = P.c, mc = rs.mc;
  const int xe = (k2 == kExcl) ? x : -1;
  auto wf = [&](int v, float (&w)[VE]) {
    float f[VE];
    Elem<T>::unpack(*reinterpret_cast<const uint4*>(buf + (size_t)v * 16), f);
#pragma unroll
    for (int j = 0; j < VE; ++j) {
      w[j] = ex2(__fmaf_rn(f[j], c, -mc));
      if (g.e0 - g.slot0 + v * VE + j == xe) w[j] = 0.f;
    }
  };
  const int tok = chunk_crossing<VE>(g, t, wf, F.tileW, F.s_int, F.s_flt);
  return ok ? tok : -1;
}

// Combines the chunk statistics of every row of request b into RowStat (one warp per row).
template <int MODE>
__device__ void combine_rows(const Params& P, int b) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr bool kSoftmax = (MODE == kChain || MODE == kNgram);
  for (int r = warp; r < P.rows; r += kWarps) {
    const ChunkStat* cs = P.cstat + ((size_t)b * P.rows + r) * P.nchunk;
    float m = -INFINITY;
    int fl = 0;
    for (int c = lane; c < P.nchunk; c += 32) {
      const float a = __ldcg(&cs[c].a);
      const int i = __ldcg(&cs[c].i);
      m = fmax_nan(m, a);
      if (kSoftmax)
        fl |= i;
      else if (i < 0)
        fl |= SPEC_ERRF_NONFINITE;
    }
    m = warp_max_nan(m);
    fl = warp_or(fl);
    RowStat rs;
    rs.pad[0] = rs.pad[1] = rs.pad[2] = 0;
    if (kSoftmax) {
      const float mc = __fmul_rn(m, P.c);
      const bool finite_m = !isnan(m) && m != INFINITY && m != -INFINITY;
      double z = 0.0;
      if (!fl && finite_m)
        for (int c = lane; c < P.nchunk; c += 32) z += chunk_weight(__ldcg(&cs[c].a), __ldcg(&cs[c].s), P.c, mc);
      const double Z = warp_sum_d(z);
      rs.Z = Z;
      rs.mc = mc;
      rs.amax = -1;
      rs.err = (fl || !finite_m || !(Z > 0.0) || isinf(Z)) ? (fl | SPEC_ERRF_NONFINITE) : 0;
    } else {
      // lowest index among the chunks whose maximum equals the row maximum
      int idx = INT_MAX;
      for (int c = lane; c < P.nchunk; c += 32) {
        const float a = __ldcg(&cs[c].a);
        const int i = __ldcg(&cs[c].i);
        if (a == m && i >= 0) idx = min(idx, i);
      }
      idx = warp_min_i(idx);
      rs.Z = 0.0;
      rs.mc = m;
      rs.amax = (fl || idx == INT_MAX) ? -1 : idx;
      rs.err = fl ? SPEC_ERRF_NONFINITE : 0;
    }
    if (lane == 0) P.rstat[(size_t)b * P.rows + r] = rs;
  }
  __syncthreads();
}

// Chain / n-gram finishing: alpha, acceptance scan (section I.1 step 2), outputs, and the draws
// this CTA makes (bonus row; n-gram residual).  Block-wide.
template <int MODE, typename T>
__device__ void finish_chain(const Params& P, int b, unsigned char* buf, const FinishSmem& F) {
  constexpr int S = Elem<T>::kSize;
  constexpr bool kSoftmax = (MODE == kChain || MODE == kNgram);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int K = P.K;
  combine_rows<MODE>(P, b);
  if (threadIdx.x == 0) F.s_misc[3] = 0;
  __syncthreads();
  // acceptance probability of every draft position
  for (int k = (int)threadIdx.x; k < K; k += kThreads) {
    const int x = __ldg(P.draft_tokens + (size_t)b * K + k);
    double alpha = 0.0;
    int e = 0;
    if (x < 0 || x >= P.V) {
      e = SPEC_ERRF_BAD_TOKEN;
    } else {
      const RowStat t = P.rstat[(size_t)b * P.rows + k];
      if (kSoftmax) {
        const float lx = Elem<T>::to_float(Elem<T>::load_raw(row_ptr<T>(P, b, k) + (size_t)x * S));
        const double ext = (double)lx * (double)P.c - (double)t.mc;
        if (MODE == kChain) {
          const RowStat d = P.rstat[(size_t)b * P.rows + P.R + k];
          const float dx = Elem<T>::to_float(Elem<T>::load_raw(row_ptr<T>(P, b, P.R + k) + (size_t)x * S));
          if (dx == -INFINITY) {
            alpha = 1.0;  // q(x) = 0
          } else if (lx == -INFINITY) {
            alpha = 0.0;  // p(x) = 0
          } else {
            const double exd = (double)dx * (double)P.c - (double)d.mc;
            const double ratio = exp2_split(ext - exd) * (d.Z / t.Z);
            alpha = ratio >= 1.0 ? 1.0 : ratio;
          }
        } else {
          const double px = lx == -INFINITY ? 0.0 : exp2_split(ext) / t.Z;
          alpha = px >= 1.0 ? 1.0 : px;
        }
      } else {
        alpha = (x == t.amax) ? 1.0 : 0.0;
      }
    }
    F.s_alpha[k] = alpha;
    if (e) atomicOr(&F.s_misc[3], e);
  }
  __syncthreads();
  if (warp == 0) {
    int err = F.s_misc[3];
    for (int r = lane; r < P.rows; r += 32) err |= P.rstat[(size_t)b * P.rows + r].err;
    err = warp_or(err);
    int n = 0;
    if (!err) {
      n = K;
      for (int k0 = 0; k0 < K; k0 += 32) {
        const int k = k0 + lane;
        bool rej = false;
        if (k < K) {
          const double a = F.s_alpha[k];
          rej = kSoftmax ? !((double)__ldg(P.r + (size_t)b * K + k) <= a) : (a != 1.0);
        }
        const unsigned m = __ballot_sync(kFull, rej);
        if (m) {
          n = k0 + __ffs(m) - 1;
          break;
        }
      }
    }
    for (int i = lane; i <= K; i += 32) {
      const size_t o_i = (size_t)b * (K + 1) + i;
      int o = -1;
      if (!err && i < n) o = __ldg(P.draft_tokens + (size_t)b * K + i);
      if (!err && i == n && !kSoftmax) o = P.rstat[(size_t)b * P.rows + n].amax;
      P.out_tokens[o_i] = o;
      if (P.accept_prob && i < K) P.accept_prob[(size_t)b * K + i] = err ? 0.f : (float)F.s_alpha[i];
      if (P.cand_tokens && (err || !kSoftmax)) P.cand_tokens[o_i] = err ? -1 : P.rstat[(size_t)b * P.rows + i].amax;
      if (P.pos_mass && (err || !kSoftmax)) P.pos_mass[o_i] = err ? 0.f : 1.f;
    }
    if (lane == 0) {
      P.num_accepted[b] = n;
      if (P.err_flags) P.err_flags[b] = err;
      if (P.residual_mass && (err || !kSoftmax)) P.residual_mass[b] = err ? 0.f : 1.f;
      ReqState rq;
      rq.n = n;
      rq.err = err;
      rq.pad[0] = rq.pad[1] = 0;
      P.req[b] = rq;
      F.s_misc[4] = n;
      F.s_misc[5] = err;
    }
  }
  __syncthreads();
  if constexpr (kSoftmax) {
    const int n = F.s_misc[4], err = F.s_misc[5];
    if (err) return;
    // draws made here: the bonus row (both modes) and the n-gram residual; with per-position
    // outputs requested every such position, otherwise only the emitted one
    const int kfirst = P.diag ? (MODE == kChain ? K : 0) : n;
    const int klast = P.diag ? K : n;
    for (int k = kfirst; k <= klast; ++k) {
      if (MODE == kChain && k < K) continue;  // residual_kernel draws from max(0, p - q)
      const int kind = (MODE == kNgram && k < K) ? kExcl : kFullP;
      const int x = k < K ? __ldg(P.draft_tokens + (size_t)b * K + k) : -1;
      float mass;
      const int tok = draw_from_chunks<T>(P, b, k, kind, x, buf, F, &mass);
      if (threadIdx.x == 0) {
        const size_t o_k = (size_t)b * (K + 1) + k;
        if (k == n) {
          P.out_tokens[o_k] = tok;
          if (P.residual_mass) P.residual_mass[b] = mass;
        }
        if (P.cand_tokens) P.cand_tokens[o_k] = tok;
        if (P.pos_mass) P.pos_mass[o_k] = mass;
      }
    }
  }
}

// Greedy tree walk (section III.2): from the root, move to the child whose token equals the
// argmax of the current node's row (lowest node index first) until none does.  Warp 0.
__device__ inline void walk_tree(const Params& P, int b) {
  const int lane = threadIdx.x & 31;
  const int N1 = P.R, V = P.V;
  const RowStat* rs = P.rstat + (size_t)b * N1;
  const int32_t* par = P.parents + (size_t)b * N1;
  const int32_t* tok = P.node_tokens + (size_t)b * N1;
  int32_t* path = P.path_nodes + (size_t)b * N1;
  int32_t* out = P.out_tokens + (size_t)b * N1;
  int err = 0;
  for (int i = lane; i < N1; i += 32) {
    err |= rs[i].err;
    const int p = __ldg(par + i);
    if (i == 0 ? (p != -1) : (p < 0 || p >= i)) err |= SPEC_ERRF_BAD_TREE;
    if (i > 0) {
      const int t = __ldg(tok + i);
      if (t < 0 || t >= V) err |= SPEC_ERRF_BAD_TOKEN;
    }
    if (P.node_argmax) P.node_argmax[(size_t)b * N1 + i] = rs[i].amax;
  }
  err = warp_or(err);
  int len = 0;
  if (!err) {
    int cur = 0;
    if (lane == 0) path[0] = 0;
    for (int step = 0; step < N1; ++step) {  // cur strictly increases: at most N1 - 1 moves
      const int a = rs[cur].amax;
      int next = -1;
      for (int c0 = cur + 1; c0 < N1 && next < 0; c0 += 32) {
        const int cc = c0 + lane;
        const bool m = cc < N1 && __ldg(par + cc) == cur && __ldg(tok + cc) == a;
        const unsigned bal = __ballot_sync(kFull, m);
        if (bal) next = c0 + __ffs(bal) - 1;
      }
      if (next < 0) {
        if (lane == 0) out[len] = a;
        break;
      }
      if (lane == 0) {
        out[len] = __ldg(tok + next);
        path[len + 1] = next;
      }
      ++len;
      cur = next;
    }
  }
  for (int i = lane; i < N1; i += 32) {
    if (err || i > len) {
      path[i] = -1;
      out[i] = -1;
    }
  }
  if (lane == 0) {
    P.accept_len[b] = err ? 0 : len;
    if (P.err_flags) P.err_flags[b] = err;
  }
}

// ---------------------------------------------------------------------- stats kernel ----
// Persistent: each CTA claims work items (one chunk of one row; request-major order) from an
// atomic counter, one item ahead of use, and keeps two of them in flight in its two stages.  The
// ticket of an item is taken after its statistics are written; its result is examined one item
// later (so the atomic's latency overlaps the next item), and the CTA whose ticket completed a
// request finishes that request before going on.
template <int MODE, typename T>
__global__ void __launch_bounds__(kThreads, 3) stats_kernel(const Params P) {
  constexpr int VE = Elem<T>::kPerVec;
  constexpr bool kSoftmax = (MODE == kChain || MODE == kNgram);
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint64_t bar[2];
  __shared__ uint64_t bar_x;
  __shared__ unsigned xphase;
  __shared__ float red[3 * kWarps];
  __shared__ int redi[kWarps];
  __shared__ float tileW[kMaxTiles][kWarps];
  __shared__ int s_int[4];
  __shared__ float s_flt[4];
  __shared__ double s_dbl[4];
  __shared__ int s_misc[8];
  __shared__ int s_fin;
  __shared__ unsigned s_item[2];
  __shared__ double s_alpha[MODE == kTree ? 1 : SPEC_MAX_K];

  const int tid = threadIdx.x;
  const int per_req = P.rows * P.nchunk;
  const unsigned total = (unsigned)((long long)P.B * per_req);
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    mbar_init(&bar_x, 1);
    xphase = 0;
    fence_mbar_init();
    s_item[0] = atomicAdd(P.work, 1u);
    s_item[1] = atomicAdd(P.work, 1u);
  }
  __syncthreads();
  const uint64_t pol = l2_policy_evict_first();
  const FinishSmem F{tileW, s_int, s_flt, s_dbl, s_alpha, s_misc, &bar_x, &xphase};

  auto locate = [&](unsigned w, int& b, int& r, int& ch, const char*& rp) {
    b = (int)(w / (unsigned)per_req);
    const int rem = (int)(w - (unsigned)b * (unsigned)per_req);
    r = rem / P.nchunk;
    ch = rem - r * P.nchunk;
    rp = row_ptr<T>(P, b, r);
    return make_geo<T>(rp, ch * P.chunk, chunk_len(P, ch));
  };
  auto finish = [&](int b, unsigned char* buf) {
    __threadfence();
    if constexpr (MODE == kTree) {
      combine_rows<MODE>(P, b);
      if (tid < 32) walk_tree(P, b);
    } else {
      finish_chain<MODE, T>(P, b, buf, F);
    }
  };
  for (int s = 0; s < 2; ++s) {
    if (s_item[s] < total) {
      int b, r, ch;
      const char* rp;
      const Geo g = locate(s_item[s], b, r, ch, rp);
      issue_chunk<T>(smem + s * P.buf_bytes, rp, g, &bar[s], pol);
    }
  }
  int pend_b = -1;      // thread 0: request of the previous item's ticket
  unsigned pend_old = 0;  // thread 0: that ticket's value before the increment
  for (int it = 0;; ++it) {
    const int st = it & 1;
    const unsigned w = s_item[st];
    if (w >= total) break;  // claims increase, so the other stage is empty too
    unsigned claim = 0;
    if (tid == 0) claim = atomicAdd(P.work, 1u);  // the item this stage takes next
    unsigned char* buf = smem + st * P.buf_bytes;
    int b, r, ch;
    const char* rp;
    const Geo g = locate(w, b, r, ch, rp);
    bool ok = mbar_wait_bounded(&bar[st], (uint32_t)(it >> 1) & 1u);
    if (!ok) ok = mbar_wait_bounded(&bar[st], (uint32_t)(it >> 1) & 1u);  // never go on with a copy in flight
    __syncthreads();  // plain-loaded slots of this stage are visible

    ChunkStat q;
    if constexpr (kSoftmax) {
      int vx = -1, jx = -1;
      if (MODE == kNgram && r < P.K) {
        const int x = __ldg(P.draft_tokens + (size_t)b * P.K + r);
        if (x >= g.e0 && x < g.e0 + g.n) {
          const int sl = x - g.e0 + g.slot0;
          vx = sl / VE;
          jx = sl - vx * VE;
        }
      }
      q = chunk_softmax_stats<T>(buf, g, P.c, vx, jx, red);
      if (!ok) q.i |= SPEC_ERRF_TIMEOUT;
    } else {
      q = chunk_argmax<T>(buf, g, red, redi);
      if (!ok) q.i = -1;
    }
    if (tid == 0) {
      s_fin = (pend_b >= 0 && pend_old == (unsigned)(per_req - 1)) ? pend_b : -1;
      P.cstat[((size_t)b * P.rows + r) * P.nchunk + ch] = q;
      __threadfence();
      pend_old = atomicAdd(P.tick_a + b, 1u);
      pend_b = b;
    }
    __syncthreads();
    if (s_fin >= 0) finish(s_fin, buf);  // the previous item's ticket completed its request
    if (tid == 0) s_item[st] = claim;
    __syncthreads();  // every thread is done with this stage and sees the claim
    if (claim < total) {
      const Geo g2 = locate(claim, b, r, ch, rp);
      issue_chunk<T>(buf, rp, g2, &bar[st], pol);
    }
  }
  if (tid == 0) s_fin = (pend_b >= 0 && pend_old == (unsigned)(per_req - 1)) ? pend_b : -1;
  __syncthreads();
  if (s_fin >= 0) finish(s_fin, smem);  // no copy is in flight once the loop has ended
}

// ------------------------------------------------------------------- residual kernel ----
// Draft-model chain, T > 0: the draw from max(0, p_k - q_k) at the rejected position (with
// per-position outputs requested: at every draft position).  One CTA per (request, position,
// chunk); the last chunk of a (request, position) finds the crossing chunk and searches it.
template <typename T>
__global__ void __launch_bounds__(kThreads, 3) residual_kernel(const Params P) {
  constexpr int VE = Elem<T>::kPerVec;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint64_t bar;
  __shared__ float red[2 * kWarps];
  __shared__ float tileW[kMaxTiles][kWarps];
  __shared__ int s_int[4];
  __shared__ float s_flt[4];
  __shared__ double s_dbl[4];
  __shared__ int s_misc[4];
  __shared__ int s_last;

  const int tid = threadIdx.x;
  const int npos = P.diag ? P.K : 1;
  const int b = (int)(blockIdx.x / (unsigned)(npos * P.nchunk));
  const int pk = (int)(blockIdx.x / (unsigned)P.nchunk) % npos;
  const int ch = (int)(blockIdx.x % (unsigned)P.nchunk);
  const ReqState rq = P.req[b];
  const int k = P.diag ? pk : rq.n;
  if (rq.err || k >= P.K) return;  // accepted everything, or failed: nothing to draw here

  unsigned char* bufT = smem;
  unsigned char* bufD = smem + P.buf_bytes;
  const RowStat ts = P.rstat[(size_t)b * P.rows + k];
  const RowStat ds = P.rstat[(size_t)b * P.rows + P.R + k];
  const float c = P.c, mct = ts.mc, mcd = ds.mc;
  const float rho = __fdiv_rn((float)ts.Z, (float)ds.Z);  // max(0, p - q) Z_t = max(0, e - f Z_t / Z_d)
  const char* rT = row_ptr<T>(P, b, k);
  const char* rD = row_ptr<T>(P, b, P.R + k);
  if (tid == 0) {
    mbar_init(&bar, 2);
    fence_mbar_init();
  }
  __syncthreads();
  const uint64_t pol = l2_policy_evict_last();  // the crossing chunk is read again right away
  Geo g = make_geo<T>(rT, ch * P.chunk, chunk_len(P, ch));
  issue_chunk<T>(bufT, rT, g, &bar, pol);
  issue_chunk<T>(bufD, rD, g, &bar, pol);  // laid out like the target row (plain loads if phases differ)
  bool ok = mbar_wait_bounded(&bar, 0);
  if (!ok) ok = mbar_wait_bounded(&bar, 0);
  __syncthreads();

  auto resid = [&](int v, float (&w)[VE]) {
    float f[VE], d[VE];
    Elem<T>::unpack(*reinterpret_cast<const uint4*>(bufT + (size_t)v * 16), f);
    Elem<T>::unpack(*reinterpret_cast<const uint4*>(bufD + (size_t)v * 16), d);
#pragma unroll
    for (int j = 0; j < VE; ++j) {
      const float e = ex2(__fmaf_rn(f[j], c, -mct));
      const float q = ex2(__fmaf_rn(d[j], c, -mcd));
      w[j] = fmaxf(0.f, __fmaf_rn(-q, rho, e));
    }
  };
  float sw = 0.f, unused = 0.f;
  for (int v = tid; v < g.nvec; v += kThreads) {
    float w[VE];
    resid(v, w);
    float vs = 0.f;
#pragma unroll
    for (int j = 0; j < VE; ++j) vs = __fadd_rn(vs, w[j]);
    sw = __fadd_rn(sw, vs);
  }
  block_sum2(sw, unused, red);
  const size_t bk = P.diag ? (size_t)b * P.K + k : (size_t)b;
  if (tid == 0) {
    P.wsum[bk * P.nchunk + ch] = ok ? sw : 0.f;
    __threadfence();
    s_last = (atomicAdd(P.tick_b + bk, 1u) == (unsigned)(P.nchunk - 1));
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // last chunk of (b, k): total residual weight, crossing chunk, search
  if (tid < 32) {
    const ChunkStat* cs = P.cstat + ((size_t)b * P.rows + k) * P.nchunk;
    const double u = (double)__ldg(P.u + b);
    int kind = kResid, cstar;
    double bstar, S;
    auto weight = [&](int q) {
      return kind == kResid ? (double)__ldcg(P.wsum + bk * P.nchunk + q)
                            : chunk_weight(__ldcg(&cs[q].a), __ldcg(&cs[q].s), c, mct);
    };
    chunk_select(P.nchunk, u, weight, cstar, bstar, S);
    const double mass = S / ts.Z;
    if (!(S > 0.0)) {  // no residual mass: draw from p
      kind = kFullP;
      chunk_select(P.nchunk, u, weight, cstar, bstar, S);
    }
    if (tid == 0) {
      s_misc[0] = cstar;
      s_misc[1] = kind;
      s_dbl[0] = u * S - bstar;
      s_dbl[1] = mass;
    }
  }
  __syncthreads();
  const int cstar = s_misc[0], kind = s_misc[1];
  const float t = (float)s_dbl[0];
  const float mass = (float)s_dbl[1];
  int tok = -1;
  if (cstar >= 0) {
    g = make_geo<T>(rT, cstar * P.chunk, chunk_len(P, cstar));
    issue_chunk<T>(bufT, rT, g, &bar, l2_policy_evict_first());
    issue_chunk<T>(bufD, rD, g, &bar, l2_policy_evict_first());
    bool ok2 = mbar_wait_bounded(&bar, 1);
    if (!ok2) ok2 = mbar_wait_bounded(&bar, 1);
    __syncthreads();
    if (kind == kResid) {
      tok = chunk_crossing<VE>(g, t, resid, tileW, s_int, s_flt);
    } else {
      auto full = [&](int v, float (&w)[VE]) {
        float f[VE];
        Elem<T>::unpack(*reinterpret_cast<const uint4*>(bufT + (size_t)v * 16), f);
#pragma unroll
        for (int j = 0; j < VE; ++j) w[j] = ex2(__fmaf_rn(f[j], c, -mct));
      };
      tok = chunk_crossing<VE>(g, t, full, tileW, s_int, s_flt);
    }
    if (!ok2) tok = -1;
  }
  if (tid == 0) {
    const size_t o_k = (size_t)b * (P.K + 1) + k;
    if (k == rq.n) {
      P.out_tokens[o_k] = tok;
      if (P.residual_mass) P.residual_mass[b] = mass;
    }
    if (P.cand_tokens) P.cand_tokens[o_k] = tok;
    if (P.pos_mass) P.pos_mass[o_k] = mass;
  }
}

// ---------------------------------------------------------------------- probs kernel ----
// Testing aid: p_i = 2^(l_i c - mc) / Z for every target row, q likewise for draft rows.
template <typename T>
__global__ void __launch_bounds__(kThreads) probs_kernel(const Params P) {
  const int rowid = blockIdx.x;  // b * rows + r
  const int b = rowid / P.rows, r = rowid - b * P.rows;
  if (P.req[b].err) return;
  float* out = r < P.R ? (P.target_probs ? P.target_probs + ((size_t)b * P.R + r) * P.V : nullptr)
                       : (P.draft_probs ? P.draft_probs + ((size_t)b * P.K + (r - P.R)) * P.V : nullptr);
  if (!out) return;
  const RowStat rs = P.rstat[rowid];
  const char* rp = row_ptr<T>(P, b, r);
  const float invZ = (float)(1.0 / rs.Z);
  for (int i = (int)threadIdx.x; i < P.V; i += kThreads) {
    const float l = Elem<T>::to_float(Elem<T>::load_raw(rp + (size_t)i * Elem<T>::kSize));
    out[i] = __fmul_rn(ex2(__fmaf_rn(l, P.c, -rs.mc)), invZ);
  }
}

// -------------------------------------------------------------------------- launchers ----
struct LaunchPlan {
  size_t smem_stats;  // dynamic shared memory of stats_kernel (two stages)
  size_t smem_resid;  // dynamic shared memory of residual_kernel (target + draft chunk)
  int launch_resid;   // launch residual_kernel
  int launch_probs;   // launch probs_kernel
  int sm_count;       // multiprocessors of the current device
};

template <int MODE, typename T>
cudaError_t launch_mode(const Params& P, const LaunchPlan& L, cudaStream_t stream) {
  auto ks = stats_kernel<MODE, T>;
  cudaError_t e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.smem_stats);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ks, kThreads, L.smem_stats);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const long long items = (long long)P.B * P.rows * P.nchunk;
  const long long cap = (long long)per_sm * L.sm_count;
  const long long grid = items < cap ? items : cap;
  ks<<<(unsigned)grid, kThreads, L.smem_stats, stream>>>(P);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (L.launch_resid) {
    auto kr = residual_kernel<T>;
    e = cudaFuncSetAttribute(kr, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.smem_resid);
    if (e != cudaSuccess) return e;
    const long long nb = (long long)P.B * (P.diag ? P.K : 1) * P.nchunk;
    kr<<<(unsigned)nb, kThreads, L.smem_resid, stream>>>(P);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (L.launch_probs) {
    probs_kernel<T><<<(unsigned)((long long)P.B * P.rows), kThreads, 0, stream>>>(P);
    e = cudaGetLastError();
  }
  return e;
}

template <typename T>
cudaError_t launch_verify(int mode, const Params& P, const LaunchPlan& L, cudaStream_t stream) {
  switch (mode) {
    case kChain: return launch_mode<kChain, T>(P, L, stream);
    case kNgram: return launch_mode<kNgram, T>(P, L, stream);
    case kGreedy: return launch_mode<kGreedy, T>(P, L, stream);
    case kTree: return launch_mode<kTree, T>(P, L, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace specv
