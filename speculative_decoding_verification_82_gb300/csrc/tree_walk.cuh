// tree_walk.cuh -- verification of a draft tree by walking it from the root (sm_103a).
//
// Method: "Speculative Decoding in Production: From Draft Models to EAGLE-3 Dynamic Trees for
// 3x-5x Lossless Acceleration" (blog.llmgo.top), section I.1 "Verification via Modified
// Rejection Sampling" (alpha = min(1, p/q), accept iff r <= alpha, residual max(0, p - q)
// normalised), applied to the children of each visited node in turn: a rejected child replaces
// the node's target by its residual and the next sibling is tested against it with the same
// draft distribution q; section III.2 "The Tree Attention Verification Mechanism" for the walk
// (an accepted branch is descended, a rejected one skipped).  T == 0 is the greedy walk: the
// child whose token equals the argmax of the node's row.
//
// One thread-block cluster verifies one request at a time.  CTA `rank` of the cluster owns the
// vocabulary slice [rank * 512 E, (rank + 1) * 512 E) and each of its 512 threads E consecutive
// tokens of it, so the probabilities p and q of the node being visited stay on the SM for the
// whole visit (in registers; q in shared memory where both do not fit).  Row statistics, residual
// masses and the draw's prefix sums are reduced in a fixed order (warp, block, then the cluster's
// CTAs in rank order through distributed shared memory), so every CTA computes bit-identical
// values and takes identical decisions; the cluster barrier is the only synchronisation, and no
// thread ever spins on memory.
//
// Residual algebra: after rejecting siblings with masses R_1 = 1, R_2, ..., the target is
// max(0, p - c q) / R with c = R_1 + ... + R_j (max(0, max(0, p - c q) - R q) equals
// max(0, p - (c + R) q) for q >= 0), so a sibling's test is alpha = min(1, max(0, rho - c) / R)
// with rho = p(x) / q(x) taken from the logits (no cancellation of rounded probabilities), and
// each rejection costs one pass over the registers and one cluster-wide sum.
#pragma once

#include <climits>

#include "verify_common.cuh"

namespace specv {
namespace walk {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxNodes = SPEC_MAX_WALK_NODES;
constexpr int kMaxCluster = 16;
constexpr int kXWords = 6;  // words one CTA contributes to a cluster exchange

struct Params {
  const void* target;  // [B][N1][V]
  const void* draft;   // [B][N1][V] or null (greedy)
  int B, N1, V;
  float c;    // log2(e) / T; 0 selects the greedy walk
  int vec;    // every row starts on a 16-byte boundary
  int cl;     // CTAs per cluster
  const int32_t* node_tokens;  // [B][N1]
  const int32_t* parents;      // [B][N1]
  const float* r;              // [B][N1]
  const float* u;              // [B]
  const float* temps;          // [B] or null: each request's own temperature (0 = greedy)
  int32_t* accept_len;         // [B]
  int32_t* path_nodes;         // [B][N1]
  int32_t* out_tokens;         // [B][N1]
  float* residual_mass;        // [B] or null
  int32_t* err_flags;          // [B] or null
  float* accept_prob;          // [B][N1] or null
};

struct Shared {
  int par[kMaxNodes];
  int tok[kMaxNodes];
  int path[kMaxNodes];
  int kid[kMaxNodes];  // children of the visited node, ascending
  float klx[kMaxNodes], kdx[kMaxNodes], kr[kMaxNodes];  // per child: logits at its token, its r
  float wa[kWarps], wb[kWarps], wc[kWarps], wd[kWarps];
  int wi[kWarps], wj[kWarps];
  uint32_t xbuf[2][kMaxCluster][8];
};

// ---------------------------------------------------------------- cluster primitives ----
__device__ __forceinline__ uint32_t cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// All threads of all CTAs of the cluster; orders the shared-memory writes (local and remote)
// made before it for every thread after it.
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void st_peer_u32(const void* local, uint32_t peer, uint32_t v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(peer));
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}
// Every CTA contributes kXWords words `w` (valid in its threads < cl, which send them); on return
// sm.xbuf[slot][r] holds CTA r's words in every CTA.  The two buffers alternate: a CTA writing
// round k + 1 has passed round k's barrier, so every thread of the cluster has read round k - 1.
__device__ __forceinline__ int exchange(Shared& sm, int& round, const uint32_t (&w)[kXWords], int cl,
                                        uint32_t rank) {
  const int slot = round & 1;
  ++round;
  if ((int)threadIdx.x < cl) {
#pragma unroll
    for (int i = 0; i < kXWords; ++i) st_peer_u32(&sm.xbuf[slot][rank][i], threadIdx.x, w[i]);
  }
  cluster_barrier();
  return slot;
}

// ------------------------------------------------------------------- reductions ----
// (m, Z) pairs of partial softmax normalisers, Z relative to 2^(round(m c)); -inf m means empty.
// The pair with the smaller maximum is rescaled; the combination is commutative (equal maxima
// add the two sums), so both lanes of a butterfly pair get the same result.
__device__ __forceinline__ void mz_combine(float& m, float& z, float m2, float z2, float c) {
  const bool first = m >= m2;
  const float hi = first ? m : m2, lo = first ? m2 : m;
  const float zhi = first ? z : z2, zlo = first ? z2 : z;
  if (hi == -INFINITY || hi != hi) return;
  z = lo == -INFINITY ? zhi : __fadd_rn(zhi, __fmul_rn(zlo, ex2(__fsub_rn(__fmul_rn(lo, c), __fmul_rn(hi, c)))));
  m = hi;
}
__device__ __forceinline__ void warp_mz(float& m, float& z, float c, int width = 32) {
  for (int o = width >> 1; o; o >>= 1) {
    const float m2 = __shfl_xor_sync(kFull, m, o), z2 = __shfl_xor_sync(kFull, z, o);
    mz_combine(m, z, m2, z2, c);
  }
  if (width < 32) {  // lanes [0, width) hold the result: give it to every lane
    m = __shfl_sync(kFull, m, 0);
    z = __shfl_sync(kFull, z, 0);
  }
}
// Smallest power of two >= n (n <= 32).
__device__ __forceinline__ int pow2_width(int n) { return n <= 1 ? 1 : 1 << (32 - __clz(n - 1)); }

// (value, index) maxima, ties to the lower index; INT_MAX marks no element.
__device__ __forceinline__ void vi_combine(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}
__device__ __forceinline__ void warp_vi(float& v, int& i) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float v2 = __shfl_xor_sync(kFull, v, o);
    const int i2 = __shfl_xor_sync(kFull, i, o);
    vi_combine(v, i, v2, i2);
  }
}
// Cluster-wide sum of one float per thread: warp butterfly, warps in order, CTAs in rank order.
__device__ __forceinline__ float cluster_sum(Shared& sm, int& round, float s, int cl, uint32_t rank) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  s = warp_sum(s);
  if (lane == 0) sm.wa[warp] = s;
  __syncthreads();
  uint32_t w[kXWords] = {};
  if (warp == 0) w[0] = __float_as_uint(warp_sum(lane < kWarps ? sm.wa[lane] : 0.f));
  const int slot = exchange(sm, round, w, cl, rank);
  return warp_sum(lane < cl ? __uint_as_float(sm.xbuf[slot][lane][0]) : 0.f);
}
// Block minimum of one int per thread (every thread gets it).
__device__ __forceinline__ int block_min(Shared& sm, int v) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_min_i(v);
  __syncthreads();  // earlier readers of sm.wj are done
  if (lane == 0) sm.wj[warp] = v;
  __syncthreads();
  int m = INT_MAX;
  for (int i = 0; i < kWarps; ++i) m = min(m, sm.wj[i]);
  return m;
}

// ------------------------------------------------------------------- row access ----
template <typename T>
__device__ __forceinline__ const char* row_of(const void* base, const Params& P, int b, int node) {
  return static_cast<const char*>(base) + ((size_t)b * P.N1 + node) * (size_t)P.V * Elem<T>::kSize;
}
// A thread's E values of the visited node's p or q: in registers, or (SM) in shared memory at
// stride kThreads, for the q of geometries whose p and q together do not fit the register file.
template <int E, bool SM>
struct PQ {
  float v[E];
  __device__ __forceinline__ explicit PQ(float*) {}
  __device__ __forceinline__ float& operator[](int k) { return v[k]; }
};
template <int E>
struct PQ<E, true> {
  float* base;  // this thread's first value
  __device__ __forceinline__ explicit PQ(float* b) : base(b) {}
  __device__ __forceinline__ float& operator[](int k) { return base[k * kThreads]; }
};

// This thread's E consecutive elements of a row from element `first` on, as floats; elements
// past the row's end read as -inf.
template <typename T, int E, typename A>
__device__ __forceinline__ void load_seg(const char* row, long long first, int V, bool vec, A& v) {
  constexpr int S = Elem<T>::kSize, VE = Elem<T>::kPerVec;
  static_assert(E % VE == 0, "a segment is whole 16-byte vectors");
  if (vec && first + E <= V) {
    uint4 raw[E / VE];
#pragma unroll
    for (int j = 0; j < E / VE; ++j) raw[j] = __ldg(reinterpret_cast<const uint4*>(row + (first + j * VE) * S));
#pragma unroll
    for (int j = 0; j < E / VE; ++j) {
      float f[VE];
      Elem<T>::unpack(raw[j], f);
#pragma unroll
      for (int i = 0; i < VE; ++i) v[j * VE + i] = f[i];
    }
  } else {
#pragma unroll
    for (int k = 0; k < E; ++k)
      v[k] = (first + k < V) ? Elem<T>::to_float(Elem<T>::load_raw(row + (first + k) * S)) : -INFINITY;
  }
}
template <typename T>
__device__ __forceinline__ float load_elem(const char* row, int x) {
  return Elem<T>::to_float(Elem<T>::load_raw(row + (size_t)x * Elem<T>::kSize));
}

// Children of `cur` in ascending index into sm.kid; returns their number (in every thread).
__device__ __forceinline__ int gather_kids(Shared& sm, int cur, int N1) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();  // earlier readers of sm.kid are done
  int count = 0;
  for (int c0 = cur + 1; c0 < N1; c0 += kThreads) {
    const int c = c0 + (int)threadIdx.x;
    const bool is = c < N1 && sm.par[c] == cur;
    const unsigned bal = __ballot_sync(kFull, is);
    if (lane == 0) sm.wi[warp] = __popc(bal);
    __syncthreads();
    int off = count, tot = 0;
    for (int w = 0; w < kWarps; ++w) {
      if (w < warp) off += sm.wi[w];
      tot += sm.wi[w];
    }
    if (is) sm.kid[off + __popc(bal & ((1u << lane) - 1u))] = c;
    count += tot;
    __syncthreads();
  }
  return count;
}

// Writes the outputs of a request that failed (rank 0 only).
__device__ __forceinline__ void write_failure(const Params& P, int b, int err) {
  const size_t o = (size_t)b * P.N1;
  for (int i = threadIdx.x; i < P.N1; i += kThreads) {
    P.path_nodes[o + i] = -1;
    P.out_tokens[o + i] = -1;
    if (P.accept_prob) P.accept_prob[o + i] = -1.f;
  }
  if (threadIdx.x == 0) {
    P.accept_len[b] = 0;
    if (P.residual_mass) P.residual_mass[b] = 0.f;
    if (P.err_flags) P.err_flags[b] = err;
  }
}

// ------------------------------------------------------------------ one request ----
// G: an instantiation for greedy calls only, whose threads hold no q (so 48 tokens a thread fit
// in registers).
template <typename T, int E, bool SM, bool G>
__device__ void walk_request(const Params& P, Shared& sm, float* dyn, int b, long long first, uint32_t rank,
                             int& round) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int N1 = P.N1, V = P.V, cl = P.cl;
  // the request's temperature: log2(e) / T, formed in double as the host forms the call's own
  float c = P.c;
  bool bad_temp = false;
  if (P.temps) {
    const float Tb = __ldg(P.temps + b);
    bad_temp = !(Tb >= 0.f) || isinf(Tb);
    c = (bad_temp || Tb == 0.f) ? 0.f : (float)(1.4426950408889634 / (double)Tb);
  }
  const bool greedy = G || c == 0.f, vec = P.vec != 0;

  // Stage the tree; the first malformed node decides the error (its parent checked first).
  __syncthreads();  // the previous request's readers of the tree are done
  int key = INT_MAX;
  for (int i = t; i < N1; i += kThreads) {
    const int pa = __ldg(P.parents + (size_t)b * N1 + i), x = __ldg(P.node_tokens + (size_t)b * N1 + i);
    sm.par[i] = pa;
    sm.tok[i] = x;
    int code = 0;
    if (i == 0 ? pa != -1 : (pa < 0 || pa >= i)) code = SPEC_ERRF_BAD_TREE;
    else if (i > 0 && (x < 0 || x >= V)) code = SPEC_ERRF_BAD_TOKEN;
    if (code) key = min(key, (i << 4) | code);
  }
  key = block_min(sm, key);  // its barriers also publish sm.par / sm.tok
  if (bad_temp || key != INT_MAX) {
    if (rank == 0) write_failure(P, b, bad_temp ? SPEC_ERRF_BAD_TEMPERATURE : key & 15);
    return;
  }
  if (rank == 0 && P.accept_prob)
    for (int i = t; i < N1; i += kThreads) P.accept_prob[(size_t)b * N1 + i] = -1.f;
  if (t == 0) sm.path[0] = 0;

  int cur = 0, len = 0, err = 0, final_tok = -1;
  float mass = 1.f;
  for (int depth = 0; depth < N1; ++depth) {
    const int nk = gather_kids(sm, cur, N1);
    const bool need_q = !greedy && nk > 0;
    const char* trow = row_of<T>(P.target, P, b, cur);
    const char* drow = need_q ? row_of<T>(P.draft, P, b, cur) : nullptr;
    PQ<E, false> p(dyn + threadIdx.x);
    PQ<E, SM> q(dyn + threadIdx.x);
    load_seg<T, E>(trow, first, V, vec, p);
    if (need_q) {
      load_seg<T, E>(drow, first, V, vec, q);
    } else {
#pragma unroll
      for (int k = 0; k < E; ++k) q[k] = 0.f;
    }
    // the children's logits at their tokens and their uniforms (after the row loads are issued)
    for (int i = t; i < nk; i += kThreads) {
      const int node = sm.kid[i], x = sm.tok[node];
      sm.klx[i] = load_elem<T>(trow, x);
      if (need_q) {
        sm.kdx[i] = load_elem<T>(drow, x);
        sm.kr[i] = __ldg(P.r + (size_t)b * N1 + node);
      }
    }

    if (greedy) {
      // (max, lowest index) over the raw logits; NaN anywhere fails the request
      float bv = -INFINITY;
      int bi = INT_MAX, nan = 0;
#pragma unroll
      for (int k = 0; k < E; ++k) {
        const long long idx = first + k;
        if (idx < V) {
          nan |= p[k] != p[k];
          if (bi == INT_MAX || p[k] > bv) {
            bv = p[k];
            bi = (int)idx;
          }
        }
      }
      warp_vi(bv, bi);
      nan = warp_or(nan);
      if (lane == 0) {
        sm.wa[warp] = bv;
        sm.wi[warp] = bi;
        sm.wj[warp] = nan;
      }
      __syncthreads();
      uint32_t w[kXWords] = {};
      if (warp == 0) {
        const bool in = lane < kWarps;
        float v = in ? sm.wa[lane] : -INFINITY;
        int i = in ? sm.wi[lane] : INT_MAX;
        warp_vi(v, i);
        w[0] = __float_as_uint(v);
        w[1] = (uint32_t)i;
        w[2] = (uint32_t)warp_or(in ? sm.wj[lane] : 0);
      }
      const int slot = exchange(sm, round, w, cl, rank);
      const bool in = lane < cl;
      float v = in ? __uint_as_float(sm.xbuf[slot][lane][0]) : -INFINITY;
      int a = in ? (int)sm.xbuf[slot][lane][1] : INT_MAX;
      warp_vi(v, a);
      const int f = warp_or(in ? (int)sm.xbuf[slot][lane][2] : 0);
      if (f) {
        err = SPEC_ERRF_NONFINITE;
        break;
      }
      int j = 0;
      while (j < nk && sm.tok[sm.kid[j]] != a) ++j;
      if (rank == 0 && P.accept_prob)
        for (int i = t; i < nk && i <= j; i += kThreads)
          P.accept_prob[(size_t)b * N1 + sm.kid[i]] = i < j ? 0.f : 1.f;
      if (j == nk) {
        final_tok = a;
        break;
      }
      cur = sm.kid[j];
      ++len;
      if (t == 0) sm.path[len] = cur;
      continue;
    }

    // ---- softmax statistics of the target row (and the draft row when there are children) ----
    float mt = -INFINITY, zt = 0.f, md = -INFINITY, zd = 0.f;
    int fl = 0;
#pragma unroll
    for (int k = 0; k < E; ++k) {
      fl |= (p[k] != p[k] || p[k] == INFINITY) ? 1 : 0;
      mt = fmaxf(mt, p[k]);
      if (need_q) {
        fl |= (q[k] != q[k] || q[k] == INFINITY) ? 2 : 0;
        md = fmaxf(md, q[k]);
      }
    }
    // e_k = 2^(l_k c - round(m c)) for the thread's own maximum m replaces the logit in place;
    // p_k = e_k 2^(round(m c) - round(M c)) / Z once the row's M and Z are known
    const float mtl = mt, mdl = md;
    const float mcl_t = __fmul_rn(mtl, c), mcl_d = __fmul_rn(mdl, c);
#pragma unroll
    for (int k = 0; k < E; ++k) {
      p[k] = mtl == -INFINITY ? 0.f : ex2(__fmaf_rn(p[k], c, -mcl_t));
      zt = __fadd_rn(zt, p[k]);
    }
    if (need_q) {
#pragma unroll
      for (int k = 0; k < E; ++k) {
        q[k] = mdl == -INFINITY ? 0.f : ex2(__fmaf_rn(q[k], c, -mcl_d));
        zd = __fadd_rn(zd, q[k]);
      }
    }
    warp_mz(mt, zt, c);
    warp_mz(md, zd, c);
    fl = warp_or(fl);
    if (lane == 0) {
      sm.wa[warp] = mt;
      sm.wb[warp] = zt;
      sm.wc[warp] = md;
      sm.wd[warp] = zd;
      sm.wi[warp] = fl;
    }
    __syncthreads();
    {
      // warp 0 combines the warp partials, then every warp the CTAs' (butterflies: identical
      // values and order in every CTA)
      uint32_t w[kXWords] = {};
      if (warp == 0) {
        const bool in = lane < kWarps;
        float a = in ? sm.wa[lane] : -INFINITY, za = in ? sm.wb[lane] : 0.f;
        float d = in ? sm.wc[lane] : -INFINITY, zd2 = in ? sm.wd[lane] : 0.f;
        warp_mz(a, za, c, kWarps);
        warp_mz(d, zd2, c, kWarps);
        w[0] = __float_as_uint(a);
        w[1] = __float_as_uint(za);
        w[2] = __float_as_uint(d);
        w[3] = __float_as_uint(zd2);
        w[4] = (uint32_t)warp_or(in ? sm.wi[lane] : 0);
      }
      const int slot = exchange(sm, round, w, cl, rank);
      const bool in = lane < cl;
      mt = in ? __uint_as_float(sm.xbuf[slot][lane][0]) : -INFINITY;
      zt = in ? __uint_as_float(sm.xbuf[slot][lane][1]) : 0.f;
      md = in ? __uint_as_float(sm.xbuf[slot][lane][2]) : -INFINITY;
      zd = in ? __uint_as_float(sm.xbuf[slot][lane][3]) : 0.f;
      const int wdt = pow2_width(cl);
      warp_mz(mt, zt, c, wdt);
      warp_mz(md, zd, c, wdt);
      fl = warp_or(in ? (int)sm.xbuf[slot][lane][4] : 0);
    }
    if (fl || mt == -INFINITY || (need_q && md == -INFINITY)) {
      err = SPEC_ERRF_NONFINITE;
      break;
    }
    const float mct = __fmul_rn(mt, c), mcd = __fmul_rn(md, c);
    // p and q themselves are formed only when a rejection or the draw needs them (a first child
    // accepted on its test needs only the statistics): the thread's scale
    // 2^(round(m c) - round(M c)) / Z, its exponent as an exact pair
    bool formed = false;
    auto form_pq = [&]() {
      if (formed) return;
      formed = true;
      Exp2 xt;
      two_sum(mcl_t, -mct, xt.hi, xt.lo);
      const float st = mtl == -INFINITY ? 0.f : exp2_times(xt, __frcp_rn(zt));
#pragma unroll
      for (int k = 0; k < E; ++k) p[k] = __fmul_rn(p[k], st);
      if (need_q) {
        Exp2 xd;
        two_sum(mcl_d, -mcd, xd.hi, xd.lo);
        const float sd = mdl == -INFINITY ? 0.f : exp2_times(xd, __frcp_rn(zd));
#pragma unroll
        for (int k = 0; k < E; ++k) q[k] = __fmul_rn(q[k], sd);
      }
    };

    // ---- the children in order: accept test against the current residual target ----
    float cc = 0.f, R = 1.f;
    int next = -1;
    bool empty = false;
    for (int j = 0; j < nk; ++j) {
      const float lx = sm.klx[j], dx = sm.kdx[j];
      float rho;  // p(x) / q(x)
      if (dx == -INFINITY)
        rho = INFINITY;  // q(x) = 0
      else if (lx == -INFINITY)
        rho = 0.f;  // p(x) = 0
      else
        rho = exp2_times(exp2_sub(scaled_logit(lx, c, mct), scaled_logit(dx, c, mcd)), __fdiv_rn(zd, zt));
      const float alpha = rho == INFINITY ? 1.f : fminf(1.f, __fdiv_rn(fmaxf(__fsub_rn(rho, cc), 0.f), R));
      if (rank == 0 && t == 0 && P.accept_prob) P.accept_prob[(size_t)b * N1 + sm.kid[j]] = alpha;
      if (sm.kr[j] <= alpha) {
        next = sm.kid[j];
        break;
      }
      form_pq();
      cc = __fadd_rn(cc, R);
      float s = 0.f;
#pragma unroll
      for (int k = 0; k < E; ++k) s = __fadd_rn(s, fmaxf(__fsub_rn(p[k], __fmul_rn(cc, q[k])), 0.f));
      R = cluster_sum(sm, round, s, cl, rank);
      if (!(R > 0.f)) {
        empty = true;  // nothing left of the residual: the draw falls back to p
        break;
      }
    }
    if (next >= 0) {
      cur = next;
      ++len;
      if (t == 0) sm.path[len] = cur;
      continue;
    }

    // ---- the draw: smallest token whose cumulative weight exceeds u * S ----
    form_pq();
    const bool resid = need_q && !empty && cc > 0.f;
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < E; ++k) s = __fadd_rn(s, resid ? fmaxf(__fsub_rn(p[k], __fmul_rn(cc, q[k])), 0.f) : p[k]);
    const float incl = warp_incl_scan(s, lane);
    const float up = __shfl_up_sync(kFull, incl, 1);
    const float excl = lane ? up : 0.f;
    if (lane == 31) sm.wa[warp] = incl;
    __syncthreads();
    float wpre = 0.f, W = 0.f;
    for (int k = 0; k < kWarps; ++k) {
      if (k == warp) wpre = W;
      W = __fadd_rn(W, sm.wa[k]);
    }
    uint32_t w[kXWords] = {};
    if (t < cl) w[0] = __float_as_uint(W);
    const int slot = exchange(sm, round, w, cl, rank);
    float S = 0.f, pre = 0.f;
    int rstar = -1, rlast = -1;
    const float u = __ldg(P.u + b);
    float target = 0.f;
    {
      for (int r = 0; r < cl; ++r) S = __fadd_rn(S, __uint_as_float(sm.xbuf[slot][r][0]));
      target = __fmul_rn(u, S);
      float acc = 0.f;
      for (int r = 0; r < cl; ++r) {
        const float Wr = __uint_as_float(sm.xbuf[slot][r][0]);
        const float nxt = __fadd_rn(acc, Wr);
        if (rstar < 0 && nxt > target) {
          rstar = r;
          pre = acc;
        }
        if (Wr > 0.f) rlast = r;
        acc = nxt;
      }
    }
    mass = resid ? S : (empty ? 0.f : 1.f);
    if (rstar >= 0 && (int)rank == rstar) {
      // the first thread holding weight whose cumulative end exceeds the target walks its own
      // tokens; its start is the previous thread's end (at most the target).  Rounding can leave
      // no such thread: then the last thread holding weight takes its last positive token.
      const float endv = __fadd_rn(pre, __fadd_rn(wpre, incl));
      const unsigned hit = __ballot_sync(kFull, endv > target && s > 0.f);
      const unsigned pos = __ballot_sync(kFull, s > 0.f);
      if (lane == 0) {
        sm.wi[warp] = hit ? warp * 32 + __ffs(hit) - 1 : INT_MAX;
        sm.wj[warp] = pos ? warp * 32 + 31 - __clz(pos) : -1;
      }
      __syncthreads();
      int win = INT_MAX, lastt = -1;
      for (int k = 0; k < kWarps; ++k) {
        win = min(win, sm.wi[k]);
        lastt = max(lastt, sm.wj[k]);
      }
      if (t == (win != INT_MAX ? win : lastt)) {
        float run = __fadd_rn(pre, __fadd_rn(wpre, excl));
        int pick = -1, lastpos = -1;
#pragma unroll
        for (int k = 0; k < E; ++k) {
          const float wk = resid ? fmaxf(__fsub_rn(p[k], __fmul_rn(cc, q[k])), 0.f) : p[k];
          run = __fadd_rn(run, wk);
          if (wk > 0.f) {
            lastpos = k;
            if (pick < 0 && run > target) pick = k;
          }
        }
        if (pick < 0 || win == INT_MAX) pick = lastpos;
        P.out_tokens[(size_t)b * N1 + len] = (int)(first + pick);
      }
    } else if (rstar < 0 && rlast >= 0 && (int)rank == rlast) {
      // rounding left u * S at or above the total: the last token with positive weight
      const unsigned pos = __ballot_sync(kFull, s > 0.f);
      if (lane == 0) sm.wi[warp] = pos ? warp * 32 + 31 - __clz(pos) : -1;
      __syncthreads();
      int lastt = -1;
      for (int k = 0; k < kWarps; ++k) lastt = max(lastt, sm.wi[k]);
      if (t == lastt) {
        int lastpos = -1;
#pragma unroll
        for (int k = 0; k < E; ++k) {
          const float wk = resid ? fmaxf(__fsub_rn(p[k], __fmul_rn(cc, q[k])), 0.f) : p[k];
          if (wk > 0.f) lastpos = k;
        }
        P.out_tokens[(size_t)b * N1 + len] = (int)(first + lastpos);
      }
    }
    final_tok = S > 0.f ? -2 : -1;  // -2: written by the CTA that holds the token
    break;
  }

  if (err) {
    __syncthreads();  // rank 0's earlier accept_prob writes come first
    if (rank == 0) write_failure(P, b, err);
    return;
  }
  if (rank == 0) {
    __syncthreads();  // sm.path complete
    const size_t o = (size_t)b * N1;
    for (int i = t; i < N1; i += kThreads) {
      P.path_nodes[o + i] = i <= len ? sm.path[i] : -1;
      if (i != len || final_tok != -2) P.out_tokens[o + i] = i < len ? sm.tok[sm.path[i + 1]] : (i == len ? final_tok : -1);
    }
    if (t == 0) {
      P.accept_len[b] = len;
      if (P.residual_mass) P.residual_mass[b] = mass;
      if (P.err_flags) P.err_flags[b] = 0;
    }
  }
}

// SM: q in dynamic shared memory (E kThreads floats), else in registers; p is always in
// registers.  G: greedy calls only.
template <typename T, int E, bool SM, bool G>
__global__ void __launch_bounds__(kThreads, 1) walk_kernel(const Params P) {
  __shared__ Shared sm;
  extern __shared__ float walk_dyn[];
  const uint32_t rank = cta_rank();
  const long long first = ((long long)rank * kThreads + threadIdx.x) * E;
  int round = 0;
  cluster_barrier();  // every CTA of the cluster runs before any peer writes to it
  for (int b = (int)cluster_index(); b < P.B; b += (int)cluster_count())
    walk_request<T, E, SM, G>(P, sm, walk_dyn, b, first, rank, round);
  cluster_barrier();  // none leaves while a peer may still write to it
}

}  // namespace walk
}  // namespace specv
