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
  unsigned* tick_a;  // [B] request tickets of stats_kernel (zeroed by the host before each call)
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

// Weight of a chunk in units of the row normaliser: s (or sx) * 2^(a c - mc).
__device__ __forceinline__ double chunk_weight(float a, float s, float c, float mc) {
  if (a == -INFINITY) return 0.0;
  return (double)s * exp2((double)__fmul_rn(a, c) - (double)mc);
}

// ------------------------------------------------------------------ chunk reductions ----
// Softmax statistics of a staged chunk: block max m, s = sum 2^(l c - m c), and the same sum
// with slot (vx, jx) left out (vx < 0: nothing left out).
template <typename T>
__device__ __forceinline__ ChunkStat chunk_softmax_stats(const unsigned char* buf, const Geo& g, float c, int vx,
                                                         int jx, float* red) {
  constexpr int VE = Elem<T>::kPerVec;
  ChunkStat q;
  const float m = block_max_nan(thread_max<T>(buf, g.nvec), red);
  float s = 0.f, sx = 0.f;
  int fl = 0;
  if (isnan(m) || m == INFINITY) {
    fl = SPEC_ERRF_NONFINITE;
  } else if (m != -INFINITY) {
    const float mc = __fmul_rn(m, c);
    for (int v = (int)threadIdx.x; v < g.nvec; v += kThreads) {
      float f[VE];
      Elem<T>::unpack(*reinterpret_cast<const uint4*>(buf + (size_t)v * 16), f);
      float e[VE];
#pragma unroll
      for (int j = 0; j < VE; ++j) e[j] = ex2(__fmaf_rn(f[j], c, -mc));
      float vs = 0.f;
#pragma unroll
      for (int j = 0; j < VE; ++j) vs = __fadd_rn(vs, e[j]);
      s = __fadd_rn(s, vs);
      if (v == vx) {
        float vsx = 0.f;
#pragma unroll
        for (int j = 0; j < VE; ++j) vsx = __fadd_rn(vsx, j == jx ? 0.f : e[j]);
        sx = __fadd_rn(sx, vsx);
      } else {
        sx = __fadd_rn(sx, vs);
      }
    }
    block_sum2(s, sx, red);
  }
  q.a = m;
  q.s = s;
  q.sx = sx;
  q.i = fl;
  return q;
}

// (max, first index) of a staged chunk; index -1 when the chunk holds a NaN.
template <typename T>
__device__ __forceinline__ ChunkStat chunk_argmax(const unsigned char* buf, const Geo& g, float* red, int* redi) {
  constexpr int VE = Elem<T>::kPerVec;
  const float tm = thread_max<T>(buf, g.nvec);
  const float M = block_max_nan(tm, red);
  ChunkStat q;
  q.a = M;
  q.s = q.sx = 0.f;
  if (isnan(M)) {
    q.i = -1;
    return q;
  }
  int idx = INT_MAX;
  if (tm == M) {  // only threads holding a maximal element look for its first position
    for (int v = (int)threadIdx.x; v < g.nvec && idx == INT_MAX; v += kThreads) {
      float f[VE];
      Elem<T>::unpack(*reinterpret_cast<const uint4*>(buf + (size_t)v * 16), f);
#pragma unroll
      for (int j = 0; j < VE; ++j) {
        const int e = g.e0 - g.slot0 + v * VE + j;
        if (idx == INT_MAX && e >= g.e0 && e < g.e0 + g.n && f[j] == M) idx = e;
      }
    }
  }
  q.i = block_min_i(idx, redi);
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
  if (threadIdx.x == 0) {
    auto weight = [&](int c, int kd) {
      return chunk_weight(__ldcg(&cs[c].a), kd == kExcl ? __ldcg(&cs[c].sx) : __ldcg(&cs[c].s), P.c, rs.mc);
    };
    double S = 0.0;
    for (int c = 0; c < P.nchunk; ++c) S += weight(c, kind);
    const double S0 = S;
    int k2 = kind;
    if (!(S > 0.0)) {  // no residual mass: draw from p
      k2 = kFullP;
      S = 0.0;
      for (int c = 0; c < P.nchunk; ++c) S += weight(c, k2);
    }
    const double tgt = (double)__ldg(P.u + b) * S;
    double base = 0.0, bstar = 0.0, blast = 0.0;
    int cstar = -1, clast = -1;
    for (int c = 0; c < P.nchunk; ++c) {
      const double W = weight(c, k2);
      if (W > 0.0) {
        if (cstar < 0 && base + W > tgt) {
          cstar = c;
          bstar = base;
        }
        clast = c;
        blast = base;
        base += W;
      }
    }
    if (cstar < 0) {
      cstar = clast;
      bstar = blast;
    }
    F.s_misc[0] = cstar;
    F.s_misc[1] = k2;
    F.s_dbl[0] = tgt - bstar;
    F.s_dbl[1] = S0 / rs.Z;
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
      double Z = 0.0;
      if (lane == 0 && !fl && finite_m) {
        for (int c = 0; c < P.nchunk; ++c) Z += chunk_weight(__ldcg(&cs[c].a), __ldcg(&cs[c].s), P.c, mc);
      }
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
            const double ratio = exp2(ext - exd) * (d.Z / t.Z);
            alpha = ratio >= 1.0 ? 1.0 : ratio;
          }
        } else {
          const double px = lx == -INFINITY ? 0.0 : exp2(ext) / t.Z;
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
template <int MODE, typename T>
__global__ void __launch_bounds__(kThreads, 3) stats_kernel(const Params P) {
  constexpr int VE = Elem<T>::kPerVec;
  constexpr bool kSoftmax = (MODE == kChain || MODE == kNgram);
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint64_t bar[2];
  __shared__ uint64_t bar_x;
  __shared__ unsigned xphase;
  __shared__ float red[2 * kWarps];
  __shared__ int redi[kWarps];
  __shared__ float tileW[kMaxTiles][kWarps];
  __shared__ int s_int[4];
  __shared__ float s_flt[4];
  __shared__ double s_dbl[4];
  __shared__ int s_misc[8];
  __shared__ int s_last;
  __shared__ double s_alpha[MODE == kTree ? 1 : SPEC_MAX_K];

  const int tid = threadIdx.x;
  const int per_req = P.rows * P.nchunk;
  const long long total = (long long)P.B * per_req;
  const long long G = gridDim.x;
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    mbar_init(&bar_x, 1);
    xphase = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const uint64_t pol = l2_policy_evict_first();
  const FinishSmem F{tileW, s_int, s_flt, s_dbl, s_alpha, s_misc, &bar_x, &xphase};

  auto locate = [&](long long w, int& b, int& r, int& ch, const char*& rp) {
    b = (int)(w / per_req);
    const int rem = (int)(w - (long long)b * per_req);
    r = rem / P.nchunk;
    ch = rem - r * P.nchunk;
    rp = row_ptr<T>(P, b, r);
    return make_geo<T>(rp, ch * P.chunk, chunk_len(P, ch));
  };
  // prologue: fill both stages
  for (int s = 0; s < 2; ++s) {
    const long long w = blockIdx.x + s * G;
    if (w < total) {
      int b, r, ch;
      const char* rp;
      const Geo g = locate(w, b, r, ch, rp);
      issue_chunk<T>(smem + s * P.buf_bytes, rp, g, &bar[s], pol);
    }
  }
  int it = 0;
  for (long long w = blockIdx.x; w < total; w += G, ++it) {
    const int st = it & 1;
    const uint32_t par = (uint32_t)(it >> 1) & 1u;
    unsigned char* buf = smem + st * P.buf_bytes;
    int b, r, ch;
    const char* rp;
    const Geo g = locate(w, b, r, ch, rp);
    bool ok = mbar_wait_bounded(&bar[st], par);
    if (!ok) ok = mbar_wait_bounded(&bar[st], par);  // never proceed with a copy in flight
    __syncthreads();  // plain-loaded slots of this stage are visible

    ChunkStat q;
    if constexpr (kSoftmax) {
      int vx = -1, jx = -1;
      if (MODE == kNgram && r < P.K) {
        const int x = __ldg(P.draft_tokens + (size_t)b * P.K + r);
        if (x >= g.e0 && x < g.e0 + g.n) {
          const int s = x - g.e0 + g.slot0;
          vx = s / VE;
          jx = s - vx * VE;
        }
      }
      q = chunk_softmax_stats<T>(buf, g, P.c, vx, jx, red);
      if (!ok) q.i |= SPEC_ERRF_TIMEOUT;
    } else {
      q = chunk_argmax<T>(buf, g, red, redi);
      if (!ok) q.i = -1;
    }
    if (tid == 0) {
      P.cstat[((size_t)b * P.rows + r) * P.nchunk + ch] = q;
      __threadfence();
      s_last = (atomicAdd(P.tick_a + b, 1u) == (unsigned)(per_req - 1));
    }
    __syncthreads();
    if (s_last) {  // this CTA completed request b
      __threadfence();
      if constexpr (MODE == kTree) {
        combine_rows<MODE>(P, b);
        if (tid < 32) walk_tree(P, b);
      } else {
        finish_chain<MODE, T>(P, b, buf, F);
      }
    }
    __syncthreads();  // every thread is done with this stage
    const long long nxt = w + 2 * G;
    if (nxt < total) {
      const Geo g2 = locate(nxt, b, r, ch, rp);
      issue_chunk<T>(buf, rp, g2, &bar[st], pol);
    }
  }
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
  const float rho = (float)(ts.Z / ds.Z);  // max(0, p - q) * Z_t = max(0, e - f * Z_t / Z_d)
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
  if (tid == 0) {
    const ChunkStat* cs = P.cstat + ((size_t)b * P.rows + k) * P.nchunk;
    double S = 0.0;
    for (int q = 0; q < P.nchunk; ++q) S += (double)__ldcg(P.wsum + bk * P.nchunk + q);
    const double mass = S / ts.Z;
    int kind = kResid;
    if (!(S > 0.0)) {  // no residual mass: draw from p
      kind = kFullP;
      S = 0.0;
      for (int q = 0; q < P.nchunk; ++q) S += chunk_weight(__ldcg(&cs[q].a), __ldcg(&cs[q].s), c, mct);
    }
    const double tgt = (double)__ldg(P.u + b) * S;
    double base = 0.0, bstar = 0.0, blast = 0.0;
    int cstar = -1, clast = -1;
    for (int q = 0; q < P.nchunk; ++q) {
      const double W = kind == kResid ? (double)__ldcg(P.wsum + bk * P.nchunk + q)
                                      : chunk_weight(__ldcg(&cs[q].a), __ldcg(&cs[q].s), c, mct);
      if (W > 0.0) {
        if (cstar < 0 && base + W > tgt) {
          cstar = q;
          bstar = base;
        }
        clast = q;
        blast = base;
        base += W;
      }
    }
    if (cstar < 0) {
      cstar = clast;
      bstar = blast;
    }
    s_misc[0] = cstar;
    s_misc[1] = kind;
    s_dbl[0] = tgt - bstar;
    s_dbl[1] = mass;
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
