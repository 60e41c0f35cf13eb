// verify_kernel.cuh -- the verification kernel (sm_103a).
//
// verify_kernel is persistent (one CTA per SM) and warp-specialised:
//  - two groups of eight consumer warps take alternate stages of a six-stage shared-memory ring;
//    each group has a producer warp that claims work items from an atomic counter (a batch of
//    items per claim, the next batch claimed ahead) and stages each item's logits into its
//    group's stages with bulk TMA copies (an mbarrier per stage for "full" and one for "empty");
//    each consumer warp reduces one contiguous sub-chunk of the staged chunk
//    (temperature-softmax statistics, argmax, or the residual sum) and leaves its partial in a
//    ring of slots; the group's last warp to do so merges the partials and writes the chunk's
//    statistics and its sub-chunk partials;
//  - the bookkeeping warp counts each written chunk on its request (one memory fence per batch
//    of ready chunks, then fire-and-forget reductions);
//  - the finishing group (four warps) owns requests b = blockIdx.x, blockIdx.x + gridDim.x, ...:
//    once a request's count says every chunk is in, it combines the chunk statistics into per-row
//    normalisers, computes alpha_k = min(1, p_k(x_k)/q_k(x_k)), runs the acceptance scan, and
//    draws the emitted token by inverse CDF from the chunk and sub-chunk weights (re-reading only
//    the sub-chunk that holds the crossing), or walks the draft tree.
// Stats work items are ordered request-major.  For chains with draft logits and T > 0 the draw
// after a rejection at position n needs max(0, p_n - q_n), which needs both rows' normalisers
// first; the pair at n is then read a second time by residual work items.  Those are handed out
// from a cursor over the requests in order, and only for requests whose acceptance result is
// already published: a producer takes them ahead of its next stats batch whenever there are some,
// so the second read follows the first closely (often from L2) and no producer ever waits.
//
// Formulas: "Speculative Decoding in Production: From Draft Models to EAGLE-3 Dynamic Trees for
// 3x-5x Lossless Acceleration", section I.1 (acceptance ratio, uniform test, first-rejection
// stop, normalised positive residual); section III.2 (tree path acceptance).
#pragma once

#include <climits>

#include "fastdiv.h"
#include "verify_common.cuh"

namespace specv {

enum Mode : int { kChain = 0, kNgram = 1, kGreedy = 2, kTree = 3 };
// Host-side launch modes of the per-request-temperature chain and n-gram calls (the kernel runs
// MODE kChain / kNgram with PT = true).
enum LaunchMode : int { kChainPT = 4, kNgramPT = 5 };
// The high half of a request's first result word: n | kNoResid for a request verified greedily in a
// per-request-temperature call (no residual pass follows), | err << 16.
constexpr unsigned kNoResid = 0x8000u;
// A residual queue entry: the request's four result words (as in ReqState), then its index in the
// high half of a fifth word; every word tagged with the call's tag in its low half.
constexpr int kQWords = 5;
constexpr unsigned kExitAbort = 1u << 16;  // added to the exit count by a CTA that gave up (grids < 2^16)
enum Kind : int { kFullP = 0, kExcl = 1 };
enum ItemKind : int { kItemStats = 0, kItemResid = 1, kItemSkip = 2, kItemEnd = 3 };

// Per chunk of a logits row (and, with the same layout, per sub-chunk): two 8-byte halves, each a
// value and the call's tag, written together by one 16-byte store.  A reader takes the entry once
// both tags equal the call's (an aligned 8-byte half is read whole), so no memory fence has to
// order these stores before the count that announces them: the count only says when to look.
struct __align__(16) ChunkStat {
  float a;      // maximum (NaN: the range holds a NaN; softmax: +inf makes the row non-finite)
  unsigned ta;  // the call's tag
  float s;      // softmax: sum over the range of 2^(l c - RN(a c)); argmax modes: the bits of the
                // first index of the maximum (INT_MAX: the range is empty)
  unsigned ts;  // the call's tag
};
__device__ __forceinline__ bool cs_ok(const ChunkStat& q, unsigned tag) { return q.ta == tag && q.ts == tag; }
// A residual sum with the call's tag (one 8-byte store), read like a ChunkStat half.
struct __align__(8) TagSum {
  float v;
  unsigned t;
};
// Per logits row, written by the request's finishing group.
struct __align__(16) RowStat {
  double Z;  // sum over the row of 2^(l c - mc)
  float mc;  // fp32 product (row maximum) * c
  int err;   // SPEC_ERRF_* bits of the row
  int amax;  // argmax modes: row argmax
  int pad[3];
};
// Per request: the acceptance result as four self-validating 64-bit words (each a single-copy
// atomic store whose low half is the call's tag), so that readers need no fence and no other
// read, and words an earlier call left never pass: w[0] = n | err << 16 in the high half;
// w[1..3] = the fp32 bits of RN(m_t c), RN(m_d c) and Z_t / Z_d at row n (draft-model chains that
// rejected, without per-position outputs).
struct __align__(16) ReqState {
  unsigned long long w[4];
};
static_assert(sizeof(ChunkStat) == 16 && sizeof(RowStat) == 32 && sizeof(ReqState) == 32, "layout");
__device__ __forceinline__ unsigned long long ld_volatile_u64(const unsigned long long* p) {
  return *reinterpret_cast<const volatile unsigned long long*>(p);
}
__device__ __forceinline__ void st_volatile_u64(unsigned long long* p, unsigned long long v) {
  *reinterpret_cast<volatile unsigned long long*>(p) = v;
}
__device__ __forceinline__ bool req_word_ok(unsigned long long v, unsigned tag) { return (unsigned)v == tag; }
__device__ __forceinline__ unsigned req_word_hi(unsigned long long v) { return (unsigned)(v >> 32); }

struct Params {
  const void* target;
  const void* draft;
  int B, K, V, R;  // R: target rows per request (K + 1, or N + 1 for trees)
  int rows;        // logits rows per request read by the stats items (draft-model chain: 2K + 1)
  int nchunk;      // stats chunks per row (kChunkVec vectors each)
  int nchunk_r;    // residual items per row (kResVec target vectors each)
  int npos;          // residual positions per request (K with per-position outputs, else 1); 0: none
  int diag;          // 1: draw at every position (per-position outputs requested)
  int bonus_first;   // chain modes: the bonus rows stream first (else last)
  int claim;         // stats items a producer claims per atomic (fewer near the end)
  int tail_first;    // 1: near the end of the stats stream, stats items go before residual items
  float c;           // log2(e) / T (calls with one temperature)
  const float* temps;  // [B] per-request temperatures (calls with PT = true), else nullptr
  unsigned total;    // stats items (A per request)
  unsigned total_r;  // residual items (R per request)
  // the divisors of the item decoding: A = rows * nchunk stats items per request, R = npos *
  // nchunk_r residual items per request, nchunk, nchunk_r
  FastDiv fd_A, fd_R, fd_nchunk, fd_nchunk_r;
  // chain modes, stage-major stats items: the items of one non-bonus stage (B * rs * nchunk, rs the
  // rows a request reads per position) and of one request within it (rs * nchunk)
  FastDiv fd_S1, fd_pair;
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
  ChunkStat* cstat;     // [B][rows][nchunk]
  ChunkStat* sstat;     // [B][rows][nchunk][kGroupWarps] sub-chunk partials (softmax modes)
  RowStat* rstat;       // [B][rows]
  ReqState* req;        // [B]
  TagSum* wsub;         // [B][npos][nchunk_r][kGroupWarps] residual weight per sub-range
  unsigned* epoch;      // the tag of the workspace's last call (0 after the workspace is cleared)
  // host only: the workspace, its bytes in this call's layout, and the shape of that layout
  void* ws_base;
  size_t ws_bytes;
  int ws_shape[4];
  // counters, zero between calls: every call leaves them as it found them (see the kernel's end);
  // `epoch` (below) is the one word that a call advances
  unsigned* work;            // stats-item counter
  unsigned* gerr;            // timeout flag
  unsigned* exit_tick;       // exiting CTAs
  unsigned* rc;              // next residual item
  unsigned* rq_tail;         // entries published in the residual queue
  unsigned* tick_a;     // chunks in (zeroed by the finishing group once complete): per request and
                        // position [B][K+1] in the chain modes, per request [B] for trees
  unsigned long long* rq;  // [B][kQWords] the residual queue, in the order the results were
                           // published: each entry the result words, then the request's index
  unsigned* tick_b;     // [B][npos] residual items in (likewise)
};

template <typename T>
__device__ __forceinline__ const char* row_ptr(const Params& P, int b, int r) {
  constexpr int S = Elem<T>::kSize;
  if (r < P.R) return static_cast<const char*>(P.target) + ((size_t)b * P.R + r) * (size_t)P.V * S;
  return static_cast<const char*>(P.draft) + ((size_t)b * P.K + (r - P.R)) * (size_t)P.V * S;
}

// A request's temperature as the kernel uses it: c = log2(e) / T, and whether the request is
// verified greedily (T == 0, or a temperature that fails it, which is read like a greedy one).
// With one temperature per call (PT = false) every request takes the call's.
struct ReqTemp {
  float c;
  int greedy;  // argmax statistics; no draft rows, no draws
  int bad;     // a NaN, negative or infinite temperature: the request fails
};
template <int MODE, bool PT>
__device__ __forceinline__ ReqTemp req_temp(const Params& P, int b) {
  ReqTemp t;
  if constexpr (!PT) {
    t.c = P.c;
    t.greedy = (MODE == kGreedy || MODE == kTree) ? 1 : 0;
    t.bad = 0;
  } else {
    const float T = __ldg(P.temps + b);
    t.bad = (!(T >= 0.f) || isinf(T)) ? 1 : 0;
    t.greedy = (t.bad || T == 0.f) ? 1 : 0;
    // formed in double exactly as the host forms a call's own c
    t.c = t.greedy ? 0.f : (float)(1.4426950408889634 / (double)T);
  }
  return t;
}

// Weight of a chunk (or sub-chunk) relative to the row maximum: s * 2^(RN(a c) - mc), in fp32 (the
// factor 2^(...) already carries the special-function unit's ~2 ulp).
__device__ __forceinline__ float chunk_weight(float a, float s, float c, float mc) {
  if (a == -INFINITY) return 0.f;
  return __fmul_rn(s, ex2(__fsub_rn(__fmul_rn(a, c), mc)));
}
__device__ __forceinline__ ChunkStat ld_chunkstat(const ChunkStat* p) {
  const uint4 v = __ldcg(reinterpret_cast<const uint4*>(p));
  ChunkStat q;
  q.a = __uint_as_float(v.x);
  q.ta = v.y;
  q.s = __uint_as_float(v.z);
  q.ts = v.w;
  return q;
}
__device__ __forceinline__ TagSum ld_tagsum(const TagSum* p) {
  const uint2 v = __ldcg(reinterpret_cast<const uint2*>(p));
  TagSum t;
  t.v = __uint_as_float(v.x);
  t.t = v.y;
  return t;
}
__device__ __forceinline__ RowStat ld_rowstat(const RowStat* p) {
  RowStat r;
  r.Z = __ldcg(&p->Z);
  r.mc = __ldcg(&p->mc);
  r.err = __ldcg(&p->err);
  r.amax = __ldcg(&p->amax);
  r.pad[0] = r.pad[1] = r.pad[2] = 0;
  return r;
}

// ------------------------------------------------------------------- online softmax ----
// Softmax partial: s is the sum of 2^(l c - RN(m c)) over the elements seen.
struct Soft {
  float m, s;
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
  return r;
}
// (max, first index) partials: index -1 marks a NaN, INT_MAX an empty partial.
__device__ __forceinline__ void argmax_merge(float& v, int& i, float v2, int i2) {
  if (i < 0 || i2 == INT_MAX) return;
  if (i2 < 0 || i == INT_MAX || v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

// ---------------------------------------------------------------- shared-memory state ----
struct StageMeta {
  int kind;        // ItemKind
  int b, row, ch;  // request; stats: row and chunk; residual: position row k and residual chunk
  int kk;          // residual: position slot of the counts (k with per-position outputs, else 0)
  int nvec;        // vectors to reduce (stats: the chunk; residual: the target range)
  int e_base;      // element index of the first element of slot 0 (target range)
  int e_lo, e_hi;  // residual: elements [e_lo, e_hi)
  int dshift;      // residual: draft position = kDraftSlot * VE + (e - e_base) + dshift
  float mct, mcd, rho;
  float c;     // log2(e) / T of the item's request
  int greedy;  // the item's request is verified greedily (argmax statistics)
};
struct SlotMeta {
  int kind;        // ItemKind
  unsigned* tick;  // the count this chunk adds to (stats and residual items)
};
// A request of the chain modes while its finishing group takes its positions in turn.
constexpr int kOwnMax = 4;  // requests one finishing group interleaves, position by position
struct FinReq {
  int b;       // the request
  int n;       // its accepted length once decided, -1 before
  int err;     // error bits seen so far
  int tok;     // the emitted token once drawn
  int resid;   // a residual pass was published for position n (draft-model chains)
  int drawn;   // the emitted token is known
  int written; // the outputs were written (no error seen then; rewritten if one turns up later)
  int btok;    // the bonus token, made from the first stage (-1 until then)
  float bmass;
  int greedy, bad;
  float c, u, mass;
  RowStat rt, rd;  // target and draft row statistics at position n
};
constexpr int kFinCs = 512;   // chunk statistics of one request staged for its finishing
constexpr int kFinSs = 512;   // sub-chunk statistics of the rows a draw may read
constexpr int kFinRows = 64;  // row statistics kept in shared memory for finishing
struct Shared {
  uint64_t full[kStages], empty[kStages], pfull[kSlots], pempty[kSlots], fin_bar, cs_bar, ss_bar;
  StageMeta meta[kStages];
  float4 part[kSlots][kGroupWarps];  // warp partials
  SlotMeta pmeta[kSlots];
  int pcnt[kSlots];  // warps of the group that have left their partial
  int abort, last, timed_out;
  int tag_ready;  // sm.tag is set (the producers start before it is)
  float alpha[SPEC_MAX_K];
  ChunkStat fin_cs[kFinCs];
  ChunkStat fin_ss[kFinSs];
  RowStat fin_rs[kFinRows];
  int fin_par[kFinRows], fin_tok[kFinRows];  // a small tree's parents and tokens
  GroupScratch gs;                            // the finishing group's reductions and broadcasts
  FinReq fr[kOwnMax];                         // chain modes: the requests being finished
  RowStat srs[2];                             // chain modes: a position's row statistics
  unsigned tag;  // this call's tag: the workspace's epoch + 1 (never 0, the value of cleared memory)
};

__device__ __forceinline__ void raise_abort(const Params& P, Shared& sm) {
  *reinterpret_cast<volatile int*>(&sm.abort) = 1;
  atomicOr(P.gerr, 1u);
}
__device__ __forceinline__ bool aborted(const Shared& sm) {
  return *reinterpret_cast<const volatile int*>(&sm.abort) != 0;
}

// -------------------------------------------------------------------- item decoding ----
// Stats items of trees are request-major, then row, then chunk: item w < P.total is chunk item
// w mod A of request w / A.  Stats items of the chain modes are position-major ("stages"): stage
// s < K holds the rows of position s of every request (target row s, and draft row s when the
// call reads draft logits), request by request, then row, then chunk; the bonus stage holds every
// request's bonus row (target row K), last, or first when P.bonus_first (calls with residual
// passes: the bonus draw is then made before the acceptance tests end, and the stream ends on the
// last position, which few requests reach).  So the acceptance test at position s of every request
// can be made once stage s is in, and the residual pass of a request rejected there overlaps the
// later stages.  Residual items come in the order of the residual queue (requests in the order
// their results were published), then position slot, then residual chunk: residual item
// w < P.total_r is item w mod R of queue entry w / R.  The stats items are handed out by the
// counter `work`, the residual items by the cursor `rc`; a producer stages a residual item only
// once its queue entry and its request's result are published, and never waits for one while it
// still has stats items.
template <int MODE>
__device__ __forceinline__ void decode_stats(const Params& P, unsigned w, int& b, int& row, int& ch) {
  if constexpr (MODE == kTree) {
    b = (int)fdiv(w, P.fd_A);
    const int off = (int)(w - (unsigned)b * P.fd_A.d);
    row = (int)fdiv((unsigned)off, P.fd_nchunk);
    ch = off - row * P.nchunk;
  } else {
    const unsigned nb = (unsigned)P.B * P.fd_nchunk.d;          // the bonus stage's items
    const unsigned w0 = P.bonus_first ? nb : 0u;                  // the positions' first item
    const unsigned wb = P.bonus_first ? 0u : (unsigned)P.K * P.fd_S1.d;  // the bonus stage's first
    if (w - wb < nb) {  // the bonus stage: one row per request
      const unsigned off = w - wb;
      b = (int)fdiv(off, P.fd_nchunk);
      ch = (int)(off - (unsigned)b * P.fd_nchunk.d);
      row = P.K;
    } else {
      const unsigned st = fdiv(w - w0, P.fd_S1);
      const unsigned off = w - w0 - st * P.fd_S1.d;
      b = (int)fdiv(off, P.fd_pair);
      const int r2off = (int)(off - (unsigned)b * P.fd_pair.d);
      const int r2 = r2off >= P.nchunk ? 1 : 0;  // 0: target row, 1: draft row
      ch = r2off - r2 * P.nchunk;
      row = r2 ? P.R + (int)st : (int)st;
    }
  }
}
// The count a stats chunk of (request b, row) adds to.
template <int MODE>
__device__ __forceinline__ unsigned* stats_tick(const Params& P, int b, int row) {
  if constexpr (MODE == kTree) return P.tick_a + b;
  return P.tick_a + (size_t)b * P.R + (row < P.R ? row : row - P.R);
}
// Lane 0 of a producer that found queue entry e without a residual draw: moves the cursor past the
// entry's items (when it still points into them).
__device__ __forceinline__ void skip_residual(const Params& P, unsigned e) {
  const unsigned lo = e * P.fd_R.d, end = lo + P.fd_R.d;
  unsigned c = *reinterpret_cast<const volatile unsigned*>(P.rc);
  for (int tries = 0; tries < 8 && c >= lo && c < end; ++tries) {
    const unsigned old = atomicCAS(P.rc, c, end);
    if (old == c) return;
    c = old;
  }
}
// A request's acceptance result as its four words read it: every word valid, or only the first
// when that one says no residual parameters follow (an error, per-position outputs, or n = K).
__device__ __forceinline__ bool result_complete(const Params& P, unsigned tag, unsigned long long q0,
                                                unsigned long long q1, unsigned long long q2, unsigned long long q3) {
  if (!req_word_ok(q0, tag)) return false;
  const unsigned hi = req_word_hi(q0);
  if ((hi >> 16) != 0u || P.diag || (int)(hi & 0xFFFFu) >= P.K) return true;
  return req_word_ok(q1, tag) && req_word_ok(q2, tag) && req_word_ok(q3, tag);
}

// Geometry of the target grid vectors [vt0, vt0 + span) of the pair at position k (a residual
// item, or one sub-range of it), with the draft vectors covering the same elements.
template <typename T>
struct ResGeo {
  RowGrid<T> gt, gd;
  int vt0, vt1, vd0, vd1;
  int e_base, e_lo, e_hi, dshift;
};
template <typename T>
__device__ __forceinline__ ResGeo<T> res_geo(const Params& P, int b, int k, int vt0, int span) {
  constexpr int VE = Elem<T>::kPerVec;
  ResGeo<T> q;
  q.gt = row_grid<T>(row_ptr<T>(P, b, k), P.V);
  q.gd = row_grid<T>(row_ptr<T>(P, b, P.R + k), P.V);
  q.vt0 = vt0;
  q.vt1 = min(vt0 + span, q.gt.nvec);
  q.e_base = q.vt0 * VE - q.gt.phase;
  q.e_lo = max(0, q.e_base);
  q.e_hi = min(P.V, q.e_base + span * VE);
  if (q.vt1 > q.vt0) {
    q.vd0 = (q.e_lo + q.gd.phase) / VE;
    q.vd1 = (q.e_hi - 1 + q.gd.phase) / VE + 1;
  } else {
    q.vd0 = q.vd1 = 0;
  }
  q.dshift = q.e_base - (q.vd0 * VE - q.gd.phase);
  return q;
}

// Residual weights max(0, e - q rho) of target vector v of a staged residual range (draft copy
// from slot dslot), where e = 2^(l_t c - mct) and q = 2^(l_d c - mcd): max(0, p - q) in units of
// 1 / Z_t.  Elements outside [e_lo, e_hi) weigh 0.
template <typename T>
__device__ __forceinline__ void resid_weights(const unsigned char* buf, int dslot, int v, int e_base, int e_lo,
                                              int e_hi, int dshift, float c, float mct, float mcd, float rho,
                                              float (&w)[Elem<T>::kPerVec]) {
  constexpr int VE = Elem<T>::kPerVec, S = Elem<T>::kSize;
  float f[VE], d[VE];
  Elem<T>::unpack(lds128(buf + (size_t)v * 16), f);
  if (dshift % VE == 0) {
    Elem<T>::unpack(lds128(buf + (size_t)(dslot + v + dshift / VE) * 16), d);
  } else {
#pragma unroll
    for (int j = 0; j < VE; ++j) d[j] = Elem<T>::smem_elem(buf + (size_t)(dslot * VE + v * VE + j + dshift) * S);
  }
#pragma unroll
  for (int j = 0; j < VE; ++j) {
    const int e = e_base + v * VE + j;
    const float et = ex2(__fmaf_rn(f[j], c, -mct));
    const float qd = ex2(__fmaf_rn(d[j], c, -mcd));
    const bool in = (unsigned)(e - e_lo) < (unsigned)(e_hi - e_lo);
    w[j] = in ? fmaxf(0.f, __fmaf_rn(-qd, rho, et)) : 0.f;
  }
}

// ------------------------------------------------------------------------ producer ----
// Producer of group grp: items it = grp, grp + kGroups, ... of this CTA's sequence (stage
// it % kStages).  The producer holds one batch of up to kClaim residual items from the cursor at a
// time (claimed at the start of a batch of stats items, or at any item once those are out) and
// stages its items, ahead of stats items, once their queue entry is published and complete; it
// reads the entry (which carries the request's result words) at the start of a stats batch and
// looks at it at the next, so that the read does not hold it up.  Only once its stats items are
// out does it wait (bounded) for an entry.  Once both kinds are exhausted it publishes one end
// marker.
template <int MODE, typename T, bool PT>
__device__ void producer_loop(const Params& P, Shared& sm, unsigned char* stages, int grp) {
  const int lane = threadIdx.x & 31;
  // stats claims: batches of consecutive items, the next batch claimed one batch ahead.  Each
  // producer's first batch is fixed (P.claim items from P.claim * (blockIdx.x * kGroups + grp)), so
  // that its first copies start without waiting for an atomic; the counter hands out the rest, in
  // batches of P.claim until fewer than two batches per producer remain, then smaller ones, so that
  // the producers run out of items at about the same time.
  const unsigned claim = (unsigned)max(1, P.claim);
  const unsigned fixed = claim * gridDim.x * (unsigned)kGroups;
  const unsigned nprod = gridDim.x * (unsigned)kGroups;
  unsigned cur = 0, nxt = 0, ccnt = claim, ncnt = claim;
  int pos = 0;
  if (lane == 0) {
    cur = claim * (blockIdx.x * (unsigned)kGroups + (unsigned)grp);
    nxt = fixed + atomicAdd(P.work, claim);
  }
  // residual claims (lane 0): the held items rfirst .. rfirst + rcnt - 1; qreq, the request of queue
  // entry qe once that entry is published; q0..q3 and qb, the entry's words as last read
  unsigned rfirst = 0, qe = 0xffffffffu, rseen = 0;  // rseen: the cursor as this producer last saw it
  int rcnt = 0, qreq = -1;
  // qok: request qreq's result is complete (only draft-model chains have residual items)
  bool rdone = MODE != kChain || P.npos == 0, qok = false;
  bool tag_known = false;  // the call's tag is set (residual words are compared with it)
  unsigned long long q0 = 0, q1 = 0, q2 = 0, q3 = 0, qb = 0;
  bool qload = false;  // q0..q3 and qb were loaded for entry qe and are not looked at yet
  int it = grp;
  // residual parameters of the last request seen (consecutive residual items share them)
  int rb = -1, rk = 0, rerr = 1;
  float rmct = 0.f, rmcd = 0.f, rrho = 0.f, rcc = P.c;
  // per-request temperatures: the temperature of the last request whose stats item was seen
  int tb = -1;
  ReqTemp trt{P.c, 0, 0};
  for (;; it += kGroups) {
    const int s = it % kStages;
    if (!mbar_wait_warp(&sm.empty[s], ((uint32_t)(it / kStages) & 1u) ^ 1u, &sm.abort)) {
      if (lane == 0) raise_abort(P, sm);
      break;
    }
    unsigned char* buf = stages + (size_t)s * kStageBytes;
    StageMeta m;
    m.b = m.row = m.ch = m.kk = 0;
    m.nvec = 0;
    m.e_base = 0;
    m.e_lo = m.e_hi = m.dshift = 0;
    m.mct = m.mcd = m.rho = 0.f;
    m.c = P.c;
    m.greedy = 0;
    m.kind = kItemEnd;
    long long t_poll = 0;
    for (;;) {  // until this stage has an item (a residual batch of a request without a draw is dropped)
      int kind = kItemEnd;
      unsigned w = 0;
      if (lane == 0) {
        const bool sdone = cur + (unsigned)pos >= P.total;
        const bool boundary = pos == 0 || sdone;
        if (!tag_known && !rdone && ld_volatile(&sm.tag_ready)) {
          __threadfence_block();  // sm.tag was written before the flag
          tag_known = true;
        }
        if (boundary && rcnt == 0 && !rdone && tag_known) {
          // batches shrink as the cursor nears the end, so that the last requests' residual items
          // spread over as many producers as possible; once the stats items are out, batches of
          // up to two halve the claims and entry reads each item waits for (measured: 68.6 ->
          // 67.8 us on the headline chain; up to 4: 68.1, up to 8: 69.5)
          const unsigned rrem = P.total_r > rseen ? P.total_r - rseen : 0u;
          const unsigned rk = max(1u, min(sdone ? 2u : (unsigned)kClaim, rrem / ((sdone ? 1u : 2u) * nprod)));
          const unsigned c = atomicAdd(P.rc, rk);
          rseen = c + rk;
          if (c >= P.total_r) {
            rdone = true;
          } else {
            rfirst = c;
            rcnt = (int)min(rk, P.total_r - c);
          }
        }
        const unsigned ne = rcnt > 0 ? fdiv(rfirst, P.fd_R) : 0xffffffffu;  // the held items' entry
        bool rready = rcnt > 0 && ne == qe && qok;
        if (rcnt > 0 && !rready && boundary && tag_known) {
          // the entry's five words (its request and the request's result) in one read: issued at
          // one batch start and looked at the next, when they are in, or at once when the stats
          // items are out
          if (ne == qe && qload) {
            qload = false;
            qreq = req_word_ok(qb, sm.tag) ? (int)req_word_hi(qb) : -1;
            qok = rready = qreq >= 0 && result_complete(P, sm.tag, q0, q1, q2, q3);
          }
          if (!rready) {
            qe = ne;
            qok = false;  // (until these words are looked at)
            const unsigned long long* qw = P.rq + (size_t)ne * kQWords;
            q0 = ld_volatile_u64(qw);
            q1 = ld_volatile_u64(qw + 1);
            q2 = ld_volatile_u64(qw + 2);
            q3 = ld_volatile_u64(qw + 3);
            qb = ld_volatile_u64(qw + 4);
            qload = true;
            if (sdone) {
              qload = false;
              qreq = req_word_ok(qb, sm.tag) ? (int)req_word_hi(qb) : -1;
              qok = rready = qreq >= 0 && result_complete(P, sm.tag, q0, q1, q2, q3);
            }
          }
        }
        // ready residual items go ahead of stats items, except, when P.tail_first is set, near the
        // end of the stats stream (less than one item per producer left to claim), where the stats
        // items go first so that the producers run out of them together
        const bool hold = MODE == kChain && P.tail_first && !sdone &&
                          (P.total > nxt + ncnt ? P.total - nxt - ncnt : 0u) < nprod;
        if (rready && !hold) {
          kind = kItemResid;
          w = rfirst++;
          --rcnt;
        } else if (!sdone) {
          kind = kItemStats;
          w = cur + (unsigned)pos;
          if (++pos == (int)ccnt) {
            pos = 0;
            cur = nxt;
            ccnt = ncnt;
            if (cur < P.total) {
              const unsigned front = nxt + ncnt, rem = P.total > front ? P.total - front : 0u;
              ncnt = max(1u, min(claim, rem / (2u * nprod)));
              nxt = fixed + atomicAdd(P.work, ncnt);
            }
          }
        } else if (rcnt > 0 || !rdone) {
          kind = kItemSkip;  // the held residual items' result is not published yet: poll (bounded)
          if (t_poll == 0) t_poll = clock64();
          if (aborted(sm) || clock64() - t_poll > kWaitLimitCycles) {
            raise_abort(P, sm);
            kind = kItemEnd;
          } else {
            __nanosleep(128);
          }
        }
      }
      kind = __shfl_sync(kFull, kind, 0);
      w = __shfl_sync(kFull, w, 0);
      if (kind == kItemSkip) continue;
      m.kind = kind;
      if (kind == kItemStats) {
        decode_stats<MODE>(P, w, m.b, m.row, m.ch);
        if constexpr (PT) {
          if (m.b != tb) {
            tb = m.b;
            trt = req_temp<MODE, PT>(P, m.b);
          }
          if (trt.greedy && m.row >= P.R) continue;  // a greedy request's draft rows are not read
          m.c = trt.c;
          m.greedy = trt.greedy;
        }
        const RowGrid<T> g = row_grid<T>(row_ptr<T>(P, m.b, m.row), P.V);
        const int v0 = m.ch * kChunkVec, v1 = min(v0 + kChunkVec, g.nvec);
        m.nvec = max(0, v1 - v0);
        constexpr int VE = Elem<T>::kPerVec;
        m.e_base = v0 * VE - g.phase;
        // Rows stream once: evict-first keeps them from crowding out other lines.  (Keeping the
        // first position's pairs of a draft-model chain in L2 with evict-last, for the residual
        // re-read, cut DRAM reads by 35 MB on the headline chain but measured slower: the re-read
        // passes through the SMs' bulk copies either way.)
        const int hint = P.npos > 0 ? kL2First : kL2Normal;
        warp_stage<T>(buf, g, P.V, v0, v1, &sm.full[s], lane, hint);
      } else if (MODE == kChain && kind == kItemResid) {
        const int e = (int)fdiv(w, P.fd_R);  // the queue entry (published: the item was taken only then)
        const int off = (int)(w - (unsigned)e * P.fd_R.d);
        m.b = __shfl_sync(kFull, qreq, 0);
        m.kk = (int)fdiv((unsigned)off, P.fd_nchunk_r);
        m.ch = off - m.kk * P.nchunk_r;
        if (m.b != rb || P.diag) {
          // the request's result, as lane 0 read it (complete: the item was taken only then)
          const unsigned h0 = __shfl_sync(kFull, req_word_hi(q0), 0);
          const unsigned h1 = __shfl_sync(kFull, req_word_hi(q1), 0);
          const unsigned h2 = __shfl_sync(kFull, req_word_hi(q2), 0);
          const unsigned h3 = __shfl_sync(kFull, req_word_hi(q3), 0);
          rb = m.b;
          const int n = (int)(h0 & 0xFFFFu);
          rerr = (int)(h0 >> 16) | (int)(h0 & kNoResid);  // (a greedy request has no residual pass)
          rk = P.diag ? m.kk : n;
          if constexpr (PT) rcc = req_temp<MODE, PT>(P, m.b).c;
          if (!rerr && rk < P.K) {
            if (P.diag) {
              // per-position parameters come from the row statistics, written before the result
              if (lane == 0) __threadfence();
              __syncwarp();
              const RowStat ts = ld_rowstat(P.rstat + (size_t)m.b * P.rows + rk);
              const RowStat ds = ld_rowstat(P.rstat + (size_t)m.b * P.rows + P.R + rk);
              rmct = ts.mc;
              rmcd = ds.mc;
              rrho = __fdiv_rn((float)ts.Z, (float)ds.Z);  // max(0, p - q) Z_t = max(0, e - f Z_t / Z_d)
            } else {
              rmct = __uint_as_float(h1);
              rmcd = __uint_as_float(h2);
              rrho = __uint_as_float(h3);
            }
          }
        }
        if (rerr || rk >= P.K) {  // no residual draw for this request: drop the item
          if (lane == 0) skip_residual(P, (unsigned)e);
          continue;
        }
        m.row = rk;
        m.mct = rmct;
        m.mcd = rmcd;
        m.rho = rrho;
        m.c = rcc;
        const ResGeo<T> q = res_geo<T>(P, m.b, rk, m.ch * kResVec, kResVec);
        m.nvec = max(0, q.vt1 - q.vt0);
        m.e_base = q.e_base;
        m.e_lo = q.e_lo;
        m.e_hi = q.e_hi;
        m.dshift = q.dshift;
        if (m.nvec > 0) {  // (the draw reads one sub-range of these again, soon)
          warp_stage<T>(buf, q.gt, P.V, q.vt0, q.vt1, &sm.full[s], lane);
          warp_stage<T>(buf + (size_t)kDraftSlot * 16, q.gd, P.V, q.vd0, q.vd1, &sm.full[s], lane);
        }
      }
      break;
    }
    if (lane == 0) sm.meta[s] = m;
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.full[s]);
    if (m.kind == kItemEnd) {
      it += kGroups;
      break;
    }
  }
  // Never leave with a copy in flight: wait (bounded, ignoring the abort flag) for the stages
  // this producer filled last.
  const int zero = 0;
  for (int j = it - kStages; j < it; j += kGroups)
    if (j >= 0) mbar_wait(&sm.full[j % kStages], (uint32_t)(j / kStages) & 1u, &zero);
}

// ------------------------------------------------------------------------ consumers ----
// Warp gw of a group reduces vectors [gw * kSubVec, (gw + 1) * kSubVec) of a staged chunk; lane l
// takes vectors gw * kSubVec + l + 32 i.
template <int MODE, typename T>
__device__ __forceinline__ float4 consume_stats(const unsigned char* buf, const StageMeta& m, float c, int gw) {
  using E = Elem<T>;
  constexpr int VE = E::kPerVec;
  constexpr bool kSoftmax = (MODE == kChain || MODE == kNgram);
  const int lane = threadIdx.x & 31;
  const int vbase = gw * kSubVec + lane;
  uint4 vv[kVecPerLane];
#pragma unroll
  for (int i = 0; i < kVecPerLane; ++i) {
    const int v = vbase + 32 * i;
    vv[i] = v < m.nvec ? lds128(buf + (size_t)v * 16) : make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
  }
  if constexpr (kSoftmax) {
    uint32_t m0 = E::kNegInfWord, m1 = E::kNegInfWord;
#pragma unroll
    for (int i = 0; i < kVecPerLane; ++i) {
      m0 = E::max_word(m0, E::max_word(vv[i].x, vv[i].y));
      m1 = E::max_word(m1, E::max_word(vv[i].z, vv[i].w));
    }
    const float M = warp_max_nan(E::word_max(E::max_word(m0, m1)));
    if (!(M > -INFINITY && M < INFINITY)) return make_float4(M, 0.f, 0.f, 0.f);  // empty, NaN or +inf
    const float mc = __fmul_rn(M, c);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kVecPerLane; ++i) {
      float f[VE];
      E::unpack(vv[i], f);
      float vs = 0.f;
#pragma unroll
      for (int j = 0; j < VE; ++j) vs = __fadd_rn(vs, ex2(__fmaf_rn(f[j], c, -mc)));
      s = __fadd_rn(s, vs);
    }
    return make_float4(M, warp_sum(s), 0.f, 0.f);
  } else {
    // per-vector maxima; a lane holding the warp maximum finds its first vector holding it, then
    // the first element of that vector (its vectors are in index order)
    float vmax[kVecPerLane];
#pragma unroll
    for (int i = 0; i < kVecPerLane; ++i)
      vmax[i] = E::word_max(E::max_word(E::max_word(vv[i].x, vv[i].y), E::max_word(vv[i].z, vv[i].w)));
    float mt = vmax[0];
#pragma unroll
    for (int i = 1; i < kVecPerLane; ++i) mt = fmax_nan(mt, vmax[i]);
    const float M = warp_max_nan(mt);
    int idx = INT_MAX;
    if (isnan(M)) {
      idx = -1;
    } else if (M == -INFINITY) {
      // nothing but -inf: the first row element this lane holds (every staged vector holds one)
      if (vbase < m.nvec) idx = max(m.e_base + vbase * VE, 0);
    } else if (mt == M) {
      uint4 sel = vv[0];
      int vi = 0;
#pragma unroll
      for (int i = kVecPerLane - 1; i >= 0; --i) {
        if (vmax[i] == M) {
          sel = vv[i];
          vi = i;
        }
      }
      float f[VE];
      E::unpack(sel, f);
      int jj = VE - 1;
#pragma unroll
      for (int j = VE - 1; j >= 0; --j)
        if (f[j] == M) jj = j;
      idx = m.e_base + (vbase + 32 * vi) * VE + jj;
    }
    idx = warp_min_i(idx);
    return make_float4(M, __int_as_float(idx), 0.f, 0.f);
  }
}

// Residual item: warp gw sums the weights of target vectors [gw * kResSub, (gw + 1) * kResSub).
template <typename T>
__device__ __forceinline__ float4 consume_resid(const unsigned char* buf, const StageMeta& m, float c, int gw) {
  constexpr int VE = Elem<T>::kPerVec;
  const int lane = threadIdx.x & 31;
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kResSub / 32; ++i) {
    const int v = gw * kResSub + lane + 32 * i;
    if (v < m.nvec) {
      float w[VE];
      resid_weights<T>(buf, kDraftSlot, v, m.e_base, m.e_lo, m.e_hi, m.dshift, c, m.mct, m.mcd, m.rho, w);
      float vs = 0.f;
#pragma unroll
      for (int j = 0; j < VE; ++j) vs = __fadd_rn(vs, w[j]);
      s = __fadd_rn(s, vs);
    }
  }
  return make_float4(warp_sum(s), 0.f, 0.f, 0.f);
}

// The group's last warp to leave its partial in slot j merges the partials, writes the chunk's
// statistics (stats items: the chunk and its sub-chunks; residual items: the sum and the sub-range
// sums) and hands the slot to the bookkeeping warp.
template <int MODE, bool PT>
__device__ __forceinline__ void publish_chunk(const Params& P, Shared& sm, const StageMeta& m, int j) {
  constexpr bool kSoftmax = (MODE == kChain || MODE == kNgram);
  const bool soft = PT ? !m.greedy : kSoftmax;  // (per request with per-request temperatures)
  const int lane = threadIdx.x & 31;
  const bool mine = lane < kGroupWarps;
  const float4 pw = sm.part[j][lane % kGroupWarps];
  const float c = PT ? m.c : P.c;
  SlotMeta pm;
  pm.kind = m.kind;
  pm.tick = nullptr;
  if (m.kind == kItemStats) {
    const size_t ci = ((size_t)m.b * P.rows + m.row) * P.nchunk + m.ch;
    uint4 q;
    // lanes 0..kGroupWarps-1 hold the warp partials; xor-shuffles within those lanes merge them
    if (soft) {
      float M = mine ? pw.x : -INFINITY;
#pragma unroll
      for (int o = 1; o < kGroupWarps; o <<= 1) M = fmax_nan(M, __shfl_xor_sync(kFull, M, o));
      const int fl = (isnan(M) || M == INFINITY) ? SPEC_ERRF_NONFINITE : 0;
      float sv = (mine && !fl && M != -INFINITY) ? __fmul_rn(pw.y, rescale(pw.x, M, c)) : 0.f;
#pragma unroll
      for (int o = 1; o < kGroupWarps; o <<= 1) sv = __fadd_rn(sv, __shfl_xor_sync(kFull, sv, o));
      // (a NaN or +inf maximum carries the chunk's non-finite flag)
      q = make_uint4(__float_as_uint(M), sm.tag, __float_as_uint(sv), sm.tag);
      if (mine)  // the sub-chunk partials, for the draws
        *reinterpret_cast<uint4*>(P.sstat + ci * kGroupWarps + lane) =
            make_uint4(__float_as_uint(pw.x), sm.tag, __float_as_uint(pw.y), sm.tag);
    } else {
      float v = mine ? pw.x : -INFINITY;
      int i = mine ? __float_as_int(pw.y) : INT_MAX;
#pragma unroll
      for (int o = 1; o < kGroupWarps; o <<= 1)
        argmax_merge(v, i, __shfl_xor_sync(kFull, v, o), __shfl_xor_sync(kFull, i, o));
      q = make_uint4(__float_as_uint(v), sm.tag, (unsigned)i, sm.tag);
    }
    if (lane == 0) *reinterpret_cast<uint4*>(P.cstat + ci) = q;
    pm.tick = stats_tick<MODE>(P, m.b, m.row);
  } else if (MODE == kChain && m.kind == kItemResid) {
    const size_t bk = (size_t)m.b * P.npos + m.kk;
    const size_t ri = bk * P.nchunk_r + m.ch;
    if (mine) *reinterpret_cast<uint2*>(P.wsub + ri * kGroupWarps + lane) = make_uint2(__float_as_uint(pw.x), sm.tag);
    pm.tick = P.tick_b + bk;
  }
  __syncwarp();
  if (lane == 0) {
    sm.pmeta[j] = pm;
    sm.pcnt[j] = 0;
    mbar_arrive(&sm.pfull[j]);
  }
}

// Group g takes items g, g + 2, g + 4, ... (stage it % kStages, slot it % kSlots).
template <int MODE, typename T, bool PT>
__device__ void consumer_loop(const Params& P, Shared& sm, const unsigned char* stages) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int grp = warp / kGroupWarps, gw = warp % kGroupWarps;
  for (int it = grp;; it += kGroups) {
    const int s = it % kStages;
    if (!mbar_wait_warp(&sm.full[s], (uint32_t)(it / kStages) & 1u, &sm.abort)) {
      if (lane == 0) raise_abort(P, sm);
      return;
    }
    const StageMeta m = sm.meta[s];
    const unsigned char* buf = stages + (size_t)s * kStageBytes;
    float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
    if (m.kind == kItemStats) {
      if constexpr (PT)  // the item's request decides between softmax and argmax statistics
        part = m.greedy ? consume_stats<kGreedy, T>(buf, m, 0.f, gw) : consume_stats<MODE, T>(buf, m, m.c, gw);
      else
        part = consume_stats<MODE, T>(buf, m, P.c, gw);
    } else if (MODE == kChain && m.kind == kItemResid) {
      part = consume_resid<T>(buf, m, PT ? m.c : P.c, gw);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[s]);
    const int j = it % kSlots;
    if (!mbar_wait_warp(&sm.pempty[j], ((uint32_t)(it / kSlots) & 1u) ^ 1u, &sm.abort)) {
      if (lane == 0) raise_abort(P, sm);
      return;
    }
    int last = 0;
    if (lane == 0) {
      sm.part[j][gw] = part;
      __threadfence_block();
      last = atomicAdd(&sm.pcnt[j], 1) == kGroupWarps - 1;
      __threadfence_block();
    }
    if (__shfl_sync(kFull, last, 0)) publish_chunk<MODE, PT>(P, sm, m, j);
    if (m.kind == kItemEnd) return;
  }
}

// ----------------------------------------------------------------------- bookkeeper ----
template <int MODE>
__device__ void book_loop(const Params& P, Shared& sm) {
  const int lane = threadIdx.x & 31;
  // The two groups' item sequences (it = g, g + 2, ...) are each taken in order; the warp takes
  // whichever group's next chunk is ready (never blocking on one group: a group's producer may be
  // waiting for a result that depends on a chunk of the other group).  A group that has published
  // its end marker is passed over.
  static_assert(kGroups == 2, "two consumer groups");
  int nxt0 = 0, nxt1 = 1, g = 0;
  bool ended0 = false, ended1 = false;
  long long t_idle = clock64();
  while (!(ended0 && ended1)) {
    int nb = 0;
    unsigned* tick = nullptr;  // lane i: the count of the i-th chunk of this batch
    while (nb < kSlots && !(ended0 && ended1)) {  // the chunks ready now
      int pick = -1;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int gg = g ^ t;
        if (gg == 0 ? ended0 : ended1) continue;
        const int itg = gg == 0 ? nxt0 : nxt1;
        if (mbar_test_wait(&sm.pfull[itg % kSlots], (uint32_t)(itg / kSlots) & 1u)) {
          pick = gg;
          break;
        }
      }
      pick = __shfl_sync(kFull, pick, 0);
      if (pick < 0) {
        if (nb > 0) break;  // publish what this batch holds
        // (lane 0's clock decides for the warp, which leaves together)
        if (__shfl_sync(kFull, (aborted(sm) || clock64() - t_idle > kWaitLimitCycles) ? 1 : 0, 0)) {
          if (lane == 0) raise_abort(P, sm);
          ended0 = ended1 = true;
          break;
        }
        __nanosleep(32);
        continue;
      }
      t_idle = clock64();
      g = pick;
      const int it = g == 0 ? nxt0 : nxt1;
      const int j = it % kSlots;
      const SlotMeta pm = sm.pmeta[j];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.pempty[j]);
      if (g == 0)
        nxt0 += kGroups;
      else
        nxt1 += kGroups;
      const int gdone = g;
      g ^= 1;
      if (pm.kind == kItemEnd) {
        if (gdone == 0)
          ended0 = true;
        else
          ended1 = true;
        continue;
      }
      if (pm.kind == kItemSkip) continue;
      unsigned* tk = pm.tick;
      if (lane == nb) tick = tk;
      ++nb;
    }
    // no fence: the statistics carry the call's tag, and their readers wait for it
    if (nb > 0 && lane < nb) atomicAdd(tick, 1u);  // result unused: a fire-and-forget reduction
  }
}

// ------------------------------------------------------------------------ finishing ----
// The finishing group (kFinWarps warps, named barrier kFinBarrier) completes the requests
// b = blockIdx.x, blockIdx.x + gridDim.x, ...  Its first warp, the leader, waits for the counts,
// issues the copies and runs the sequential steps (alpha and the acceptance scan, the part
// selections of a draw, the tree walk); the data-parallel steps (combining chunk statistics,
// the sum and the search over a staged sub-chunk) take every thread.  Each function below is
// entered by the whole group with the same arguments unless it says otherwise, and every
// decision that ends or skips work is agreed by the group (fin_all), so that the group reaches
// its barriers together.

// Warp-wide inverse CDF over part weights W(c) (fp32), in order: the first part with positive
// weight whose running total exceeds tgt, else the last positive one.  Every lane gets the part
// and the total weight before it.  (One warp.)
template <typename WF>
__device__ __forceinline__ void select_part(int nparts, float tgt, WF W, int& cstar, float& bstar) {
  const int lane = threadIdx.x & 31;
  float base = 0.f, blast = 0.f;
  int clast = -1;
  cstar = -1;
  bstar = 0.f;
  for (int c0 = 0; c0 < nparts; c0 += 32) {
    const int cc = c0 + lane;
    const float w = cc < nparts ? W(cc) : 0.f;
    const float incl = warp_incl_scan(w, lane);
    float ex = __shfl_up_sync(kFull, incl, 1);
    if (lane == 0) ex = 0.f;
    const unsigned hit = __ballot_sync(kFull, w > 0.f && __fadd_rn(base, incl) > tgt);
    const unsigned pos = __ballot_sync(kFull, w > 0.f);
    if (hit) {
      const int L = __ffs(hit) - 1;
      cstar = c0 + L;
      bstar = __fadd_rn(base, __shfl_sync(kFull, ex, L));
      return;
    }
    if (pos) {
      const int L = 31 - __clz(pos);
      clast = c0 + L;
      blast = __fadd_rn(base, __shfl_sync(kFull, ex, L));
    }
    base = __fadd_rn(base, __shfl_sync(kFull, incl, 31));
  }
  cstar = clast;
  bstar = blast;
}
// (One warp.)
template <typename WF>
__device__ __forceinline__ float total_weight(int nparts, WF W) {
  const int lane = threadIdx.x & 31;
  float part = 0.f;
  for (int c = lane; c < nparts; c += 32) part = __fadd_rn(part, W(c));
  return warp_sum(part);
}

// Waits (bounded, ignoring the abort flag so that no copy is left in flight) for phase ph of a
// finishing barrier whose copies have been issued and whose arrival is made; every thread of the
// group waits.  Returns the group's agreement that the phase completed.
__device__ __forceinline__ bool fin_wait_only(const Params& P, Shared& sm, uint64_t* bar, uint32_t& ph) {
  const int zero = 0;
  bool ok = mbar_wait(bar, ph & 1u, &zero);
  if (!ok) {
    raise_abort(P, sm);
    mbar_wait(bar, ph & 1u, &zero);
  }
  ++ph;
  return fin_all(ok);
}

// Chunk statistics of request b as the finishing group reads them: from the shared-memory copy
// when the request's block fits there, else from global memory.
struct CsReader {
  const ChunkStat* g;
  const ChunkStat* s;
  int nchunk;
  __device__ __forceinline__ ChunkStat operator()(int r, int c) const {
    if (s) return s[r * nchunk + c];
    return ld_chunkstat(g + (size_t)r * nchunk + c);
  }
};
// Rows whose sub-chunk statistics sit in fin_ss (row r0 + i at fin_ss[i * nchunk * kGroupWarps]).
struct SsRows {
  int r0, n;
};
// Waits (bounded) until the n chunk statistics at p in global memory all carry the call's tag;
// the group splits the checks.  False after a timeout.
__device__ __forceinline__ bool await_tagged(const Params& P, Shared& sm, const ChunkStat* p, int n) {
  const long long t0 = clock64();
  for (;;) {
    bool good = true;
    for (int i = fin_thread(); i < n; i += kFinThreads) good = good && cs_ok(ld_chunkstat(p + i), sm.tag);
    if (fin_all(good)) return true;
    if (fin_timed_out(t0)) {
      if (fin_thread() == 0) raise_abort(P, sm);
      return false;
    }
    __nanosleep(128);
  }
}
// Copies request b's chunk statistics into shared memory when they fit, together with the sub-
// chunk statistics of rows ss (when those fit too; otherwise ss.n becomes 0): bulk copies (each
// block contiguous, 16-byte aligned, a multiple of 16 bytes) issued by the leader, completing on
// cs_bar, and issued again (bounded) until every entry carries the call's tag.  The leader
// acquired the request's count before the group barrier that precedes this call; its proxy fence
// orders that acquisition, and the group's earlier reads of the buffers, before the copies.  When
// the statistics do not fit, the group waits for their tags in global memory instead.
__device__ __forceinline__ CsReader stage_request_stats(const Params& P, Shared& sm, int b, SsRows& ss,
                                                        uint32_t& csph, int rows) {
  const int n = rows * P.nchunk;  // the request's first `rows` rows (a greedy request: no draft rows)
  const int nss = P.nchunk * kGroupWarps;
  CsReader rd;
  rd.g = P.cstat + (size_t)b * P.rows * P.nchunk;  // (the request's block holds P.rows rows)
  rd.nchunk = P.nchunk;
  rd.s = nullptr;
  if (n > kFinCs) {
    ss.n = 0;
    await_tagged(P, sm, rd.g, n);
    return rd;
  }
  if (ss.n * nss > kFinSs) ss.n = 0;
  const int nsx = ss.n * nss;
  const ChunkStat* sg = P.sstat + ((size_t)b * P.rows + ss.r0) * nss;
  const long long t0 = clock64();
  for (;;) {
    if (fin_thread() == 0) {
      fence_proxy_async_global();
      fence_proxy_async_shared();
      const uint32_t bytes = (uint32_t)n * (uint32_t)sizeof(ChunkStat);
      const uint32_t sbytes = (uint32_t)nsx * (uint32_t)sizeof(ChunkStat);
      mbar_expect_tx(&sm.cs_bar, bytes + sbytes);
      tma_load_1d(sm.fin_cs, rd.g, bytes, &sm.cs_bar);
      if (sbytes) tma_load_1d(sm.fin_ss, sg, sbytes, &sm.cs_bar);
      mbar_arrive(&sm.cs_bar);
    }
    if (!fin_wait_only(P, sm, &sm.cs_bar, csph)) {  // after a timeout, read global memory instead
      ss.n = 0;
      return rd;
    }
    bool good = true;
    for (int i = fin_thread(); i < n + nsx; i += kFinThreads)
      good = good && cs_ok(i < n ? sm.fin_cs[i] : sm.fin_ss[i - n], sm.tag);
    if (fin_all(good)) break;  // (the barrier also ends the group's reads before a new copy)
    if (fin_timed_out(t0)) {
      if (fin_thread() == 0) raise_abort(P, sm);
      ss.n = 0;
      return rd;
    }
    __nanosleep(128);
  }
  rd.s = sm.fin_cs;
  return rd;
}

// Row statistics of request b (shared-memory copy for the first kFinRows rows).
__device__ __forceinline__ RowStat read_rowstat(const Params& P, const Shared& sm, int b, int r) {
  if (r < kFinRows) return sm.fin_rs[r];
  return ld_rowstat(P.rstat + (size_t)b * P.rows + r);
}

// A draw from target row `row` of request b by inverse CDF: weights p (kFullP) or p without
// token x (kExcl).  draw_begin issues the bulk copies the draw needs (the row's sub-chunk
// statistics unless they are staged already; for kExcl the sub-chunk holding x) so that they
// overlap other work; draw_end picks the crossing chunk from the chunk weights, the crossing
// sub-chunk from the sub-chunk weights, stages that sub-chunk (unless it is the one already
// staged) and searches it.  For kExcl the sub-chunk holding x is summed without x, so no weight
// is ever obtained by subtraction.
struct DrawPlan {
  int row, kind, x;
  int cx, ix;    // kExcl: chunk and sub-chunk holding x
  int sv0, sv1;  // grid vectors staged in the finishing buffer (sv1 <= sv0: none)
  int ss;        // sub-chunk statistics: 0 global memory, 1 being staged at fin_ss, 2 staged already
  int ss_off;    // their offset in fin_ss
};
template <typename T>
__device__ DrawPlan draw_begin(const Params& P, Shared& sm, unsigned char* fbuf, int b, int row, int kind, int x,
                               SsRows& st) {
  constexpr int VE = Elem<T>::kPerVec;
  const int ft = fin_thread(), lane = ft & 31;
  DrawPlan d;
  d.row = row;
  d.kind = kFullP;
  d.x = -1;
  d.cx = d.ix = -1;
  d.sv0 = d.sv1 = 0;
  const int nss = P.nchunk * kGroupWarps;
  if (row >= st.r0 && row < st.r0 + st.n) {
    d.ss = 2;
    d.ss_off = (row - st.r0) * nss;
  } else {
    d.ss = nss <= kFinSs ? 1 : 0;
    d.ss_off = 0;
    if (d.ss) st.n = 0;  // the staged rows are overwritten
  }
  const RowGrid<T> g = row_grid<T>(row_ptr<T>(P, b, row), P.V);
  if (kind == kExcl && x >= 0 && x < P.V) {
    const int pv = (x + g.phase) / VE;
    d.kind = kExcl;
    d.x = x;
    d.cx = pv / kChunkVec;
    d.ix = (pv - d.cx * kChunkVec) / kSubVec;
    d.sv0 = d.cx * kChunkVec + d.ix * kSubVec;
    d.sv1 = min(d.sv0 + kSubVec, g.nvec);
  }
  fin_sync();  // the group's earlier reads of fin_ss and the finishing buffer come first
  if (ft < 32) {
    if (lane == 0) {
      fence_proxy_async_global();  // the statistics were acquired with the request's count
      fence_proxy_async_shared();
      if (d.ss == 1) {
        const uint32_t bytes = (uint32_t)nss * (uint32_t)sizeof(ChunkStat);
        mbar_expect_tx(&sm.ss_bar, bytes);
        tma_load_1d(sm.fin_ss, P.sstat + ((size_t)b * P.rows + row) * nss, bytes, &sm.ss_bar);
        mbar_arrive(&sm.ss_bar);
      }
    }
    if (d.kind == kExcl) {
      warp_stage<T>(fbuf, g, P.V, d.sv0, d.sv1, &sm.fin_bar, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.fin_bar);
    }
  }
  return d;
}

template <typename T>
__device__ int draw_end(const Params& P, Shared& sm, unsigned char* fbuf, uint32_t& fph, uint32_t& ssph, int b,
                        const DrawPlan& d, const CsReader& rd, const RowStat& rs, float u, float c,
                        float* mass_out) {
  constexpr int VE = Elem<T>::kPerVec;
  const int ft = fin_thread(), lane = ft & 31;
  const float mc = rs.mc;
  const int row = d.row;
  const RowGrid<T> g = row_grid<T>(row_ptr<T>(P, b, row), P.V);
  const ChunkStat* srow = P.sstat + ((size_t)b * P.rows + row) * P.nchunk * kGroupWarps;
  const ChunkStat* sss = d.ss ? sm.fin_ss + d.ss_off : nullptr;  // (prestaged rows are checked)
  bool ok = true;
  if (d.ss == 1) {
    ok = fin_wait_only(P, sm, &sm.ss_bar, ssph);
    // a staged entry without the call's tag is not in yet: take the row from global memory then
    bool good = true;
    for (int i = ft; i < P.nchunk * kGroupWarps; i += kFinThreads) good = good && cs_ok(sm.fin_ss[i], sm.tag);
    if (!fin_all(good)) sss = nullptr;
  }
  if (d.kind == kExcl) ok = fin_wait_only(P, sm, &sm.fin_bar, fph) && ok;
  if (!sss) ok = await_tagged(P, sm, srow, P.nchunk * kGroupWarps) && ok;
  const int cx = d.cx, ix = d.ix;
  // kExcl: the staged sub-chunk's weight without x, summed by the group
  float wx = 0.f;
  if (d.kind == kExcl) {
    const int e_base = d.sv0 * VE - g.phase;
    float part = 0.f;
    for (int v = ft; v < d.sv1 - d.sv0; v += kFinThreads) {
      float f[VE];
      Elem<T>::unpack(lds128(fbuf + (size_t)v * 16), f);
      float vs = 0.f;
#pragma unroll
      for (int j = 0; j < VE; ++j) vs = __fadd_rn(vs, e_base + v * VE + j == d.x ? 0.f : ex2(__fmaf_rn(f[j], c, -mc)));
      part = __fadd_rn(part, vs);
    }
    wx = group_sum(sm.gs, part);
  }
  // the leader picks the chunk and the sub-chunk and stages the crossing sub-chunk
  if (ft < 32) {
    auto sub_weight = [&](int ch, int i) {
      const ChunkStat q = sss ? sss[ch * kGroupWarps + i] : ld_chunkstat(srow + (size_t)ch * kGroupWarps + i);
      return chunk_weight(q.a, q.s, c, mc);
    };
    // kExcl: lane i < kGroupWarps keeps sub-chunk i's weight in chunk cx, with x left out of
    // sub-chunk ix
    float wsub_x = 0.f, wcx = 0.f;
    if (d.kind == kExcl) {
      const float wl = (lane < kGroupWarps && lane != ix) ? sub_weight(cx, lane) : 0.f;
      wsub_x = lane == ix ? wx : wl;
      float t = lane < kGroupWarps ? wsub_x : 0.f;
#pragma unroll
      for (int o = 1; o < kGroupWarps; o <<= 1) t = __fadd_rn(t, __shfl_xor_sync(kFull, t, o));
      wcx = __shfl_sync(kFull, t, 0);
    }
    int k2 = d.kind;
    auto weight = [&](int ch) {
      if (k2 == kExcl && ch == cx) return wcx;
      const ChunkStat q = rd(row, ch);
      return chunk_weight(q.a, q.s, c, mc);
    };
    float S = total_weight(P.nchunk, weight);
    const float S0 = S;
    if (!(S > 0.f)) {  // no residual mass: draw from p
      k2 = kFullP;
      S = total_weight(P.nchunk, weight);
    }
    int cstar, sstar = -1;
    float bstar, sbase = 0.f;
    const float tgt = __fmul_rn(u, S);
    select_part(P.nchunk, tgt, weight, cstar, bstar);
    if (cstar >= 0) {
      const bool subx = k2 == kExcl && cstar == cx;
      auto sweight = [&](int i) {  // select_part evaluates part i in lane i
        if (subx) return wsub_x;
        return sub_weight(cstar, i);
      };
      select_part(kGroupWarps, __fsub_rn(tgt, bstar), sweight, sstar, sbase);
    }
    const int restage = (cstar >= 0 && sstar >= 0 && (cstar != d.cx || sstar != d.ix)) ? 1 : 0;
    if (restage) {
      const int sv0 = cstar * kChunkVec + sstar * kSubVec;
      // the group's reads of fbuf ended at the barrier of the sum above (or it was never read)
      if (lane == 0) fence_proxy_async_shared();
      warp_stage<T>(fbuf, g, P.V, sv0, min(sv0 + kSubVec, g.nvec), &sm.fin_bar, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.fin_bar);
    }
    if (lane == 0) {
      sm.gs.out[0] = cstar;
      sm.gs.out[1] = sstar;
      sm.gs.out[2] = k2 | (restage << 4);
      sm.gs.fout[0] = __fsub_rn(__fsub_rn(tgt, bstar), sbase);
      sm.gs.fout[1] = (float)((double)S0 / rs.Z);
    }
  }
  fin_sync();
  const int cstar = sm.gs.out[0], sstar = sm.gs.out[1], k2 = sm.gs.out[2] & 15, restage = sm.gs.out[2] >> 4;
  const float t = sm.gs.fout[0];
  *mass_out = sm.gs.fout[1];
  if (cstar < 0 || sstar < 0) {
    fin_sync();
    return -1;  // the second cannot happen: the chunk holds positive weight
  }
  int sv0 = d.sv0, sv1 = d.sv1;
  if (restage) {
    sv0 = cstar * kChunkVec + sstar * kSubVec;
    sv1 = min(sv0 + kSubVec, g.nvec);
    ok = fin_wait_only(P, sm, &sm.fin_bar, fph) && ok;
  }
  const int e_base = sv0 * VE - g.phase;
  const int xe = (k2 == kExcl) ? d.x : -1;
  auto wf = [&](int v, float (&w)[VE]) {
    float f[VE];
    Elem<T>::unpack(lds128(fbuf + (size_t)v * 16), f);
#pragma unroll
    for (int j = 0; j < VE; ++j) {
      w[j] = ex2(__fmaf_rn(f[j], c, -mc));
      if (e_base + v * VE + j == xe) w[j] = 0.f;
    }
  };
  const int pos = group_crossing<VE>(sm.gs, sv1 - sv0, t, wf);
  return (ok && pos >= 0) ? e_base + pos : -1;
}

// Combines the chunk statistics of every row of request b into RowStat.  G threads share a row
// (G a power of two: each takes chunks g, g + G, ... and a butterfly over the G threads merges
// them); G grows while the group still covers every row in one pass.
// With per-request temperatures (PT) `soft` (softmax or argmax statistics), `cr` (log2(e) / T) and
// `rows` (the rows the request read) are the request's; otherwise the call's.
template <int MODE, bool PT>
__device__ void combine_rows(const Params& P, Shared& sm, int b, const CsReader& rd, bool soft_r, float cr,
                             int rows_r) {
  constexpr bool kSoftmaxMode = (MODE == kChain || MODE == kNgram);
  const bool kSoftmax = PT ? soft_r : kSoftmaxMode;
  const float c = PT ? cr : P.c;
  const int rows = PT ? rows_r : P.rows;
  const int ft = fin_thread();
  const int nch = P.nchunk;
  int G = 1;
  while (G < 32 && G < nch && rows * 2 * G <= kFinThreads) G <<= 1;
  const int g = ft & (G - 1);
  const int rpp = kFinThreads / G;
  for (int r0 = 0; r0 < rows; r0 += rpp) {
    const int r = r0 + ft / G;
    const bool act = r < rows;
    float m = -INFINITY;
    int fl = 0;
    if (act) {
      for (int ch = g; ch < nch; ch += G) {
        const ChunkStat q = rd(r, ch);
        m = fmax_nan(m, q.a);
        if (isnan(q.a) || (kSoftmax && q.a == INFINITY)) fl |= SPEC_ERRF_NONFINITE;
      }
    }
    for (int o = G >> 1; o > 0; o >>= 1) {
      m = fmax_nan(m, __shfl_xor_sync(kFull, m, o));
      fl |= __shfl_xor_sync(kFull, fl, o);
    }
    RowStat rs;
    rs.pad[0] = rs.pad[1] = rs.pad[2] = 0;
    if (kSoftmax) {
      const float mc = __fmul_rn(m, c);
      const bool finite_m = !isnan(m) && m != INFINITY && m != -INFINITY;
      float z = 0.f;
      if (act && !fl && finite_m) {
        for (int ch = g; ch < nch; ch += G) {
          const ChunkStat q = rd(r, ch);
          z = __fadd_rn(z, chunk_weight(q.a, q.s, c, mc));
        }
      }
      for (int o = G >> 1; o > 0; o >>= 1) z = __fadd_rn(z, __shfl_xor_sync(kFull, z, o));
      const double Z = (!fl && finite_m) ? (double)z : 0.0;
      rs.Z = Z;
      rs.mc = mc;
      rs.amax = -1;
      rs.err = (fl || !finite_m || !(Z > 0.0) || isinf(Z)) ? (fl | SPEC_ERRF_NONFINITE) : 0;
    } else {
      // lowest index among the chunks whose maximum equals the row maximum
      int idx = INT_MAX;
      if (act) {
        for (int ch = g; ch < nch; ch += G) {
          const ChunkStat q = rd(r, ch);
          if (q.a == m) idx = min(idx, __float_as_int(q.s));
        }
      }
      for (int o = G >> 1; o > 0; o >>= 1) idx = min(idx, __shfl_xor_sync(kFull, idx, o));
      rs.Z = 0.0;
      rs.mc = m;
      rs.amax = (fl || idx == INT_MAX) ? -1 : idx;
      rs.err = fl ? SPEC_ERRF_NONFINITE : 0;
    }
    if (act && g == 0) {
      P.rstat[(size_t)b * P.rows + r] = rs;
      if (r < kFinRows) sm.fin_rs[r] = rs;
    }
  }
  fin_sync();
}

// Waits (bounded) until *count reaches `want`: the leader polls (with acquire semantics, so the
// statistics counted before it are visible afterwards), then the group agrees.  False on a
// timeout or abort.
__device__ __forceinline__ bool wait_count(const Params& P, Shared& sm, const unsigned* count, unsigned want) {
  int ok = 1;
  if (fin_thread() == 0) {
    ok = 0;
    const long long t0 = clock64();
    for (;;) {
      if (ld_acquire_u32(count) >= want) {
        ok = 1;
        break;
      }
      if (aborted(sm)) break;
      if (clock64() - t0 > kWaitLimitCycles) {
        raise_abort(P, sm);
        break;
      }
      __nanosleep(64);
    }
  }
  return fin_all(ok != 0);
}

// ------------------------------------------------------------------ chain-mode finishing ----
// The finishing group of a CTA finishes the requests b = blockIdx.x + j gridDim.x (j = 0, 1, ...),
// kOwnMax at a time, taking their positions in turn as the stages of the stream come in: at stage
// s it combines the chunk statistics of row s (and draft row s) into row normalisers, computes
// alpha_s and makes the acceptance test (section I.1, steps 1-2).  At a request's first rejection,
// or after its last accepted position, its accepted length n is decided: the n-gram residual and
// the bonus draw are made at once from the row's statistics; a draft-model chain that rejected
// publishes its residual parameters and queues the request for the residual pass (section I.1,
// step 3), which the producers run while later stages stream in, and draws at the end.  A
// request's error bits (a NaN row, a bad token) are known only once all its rows are in, so its
// outputs are final only then: a request that fails is written as failed whatever was decided.

// Combines the chunk statistics of rows r0 and r1 (r1 < 0: none) of request b into RowStat
// (P.rstat, and sm.srs[0] / sm.srs[1]): softmax statistics (soft, c = log2(e) / T) or argmax.  The
// group waits (bounded) until every chunk statistic carries the call's tag (the count only says
// when to look).  G threads share a row, as in combine_rows.
constexpr int kStagePer = 4;  // chunk statistics a thread keeps in registers while combining a stage
__device__ inline void combine_stage(const Params& P, Shared& sm, int b, int r0, int r1, bool soft, float c) {
  const int nr = r1 >= 0 ? 2 : 1;
  const ChunkStat* g0 = P.cstat + ((size_t)b * P.rows + r0) * P.nchunk;
  const ChunkStat* g1 = r1 >= 0 ? P.cstat + ((size_t)b * P.rows + r1) * P.nchunk : g0;
  const int ft = fin_thread(), nch = P.nchunk;
  int G = 1;
  while (G < 32 && G < nch && nr * 2 * G <= kFinThreads) G <<= 1;
  const int g = ft & (G - 1), i = ft / G;
  const bool act = i < nr;
  const ChunkStat* gp = i == 1 ? g1 : g0;
  // Stages of two rows (a target and a draft row): every chunk statistic is read once (one round
  // trip), the copies in registers are checked for the call's tag and read again (bounded) until
  // every tag matches.  Single rows, and rows of more than kStagePer * G chunks, take the passes
  // over global memory below instead (measured faster for the single rows of the n-gram chain).
  const bool held = nr == 2 && nch <= kStagePer * G;
  ChunkStat hq[kStagePer];
  if (held) {
    const long long t0 = clock64();
    for (;;) {
      bool good = true;
#pragma unroll
      for (int k = 0; k < kStagePer; ++k) {
        const int ch = g + k * G;
        if (act && ch < nch) {
          hq[k] = ld_chunkstat(gp + ch);
          good = good && cs_ok(hq[k], sm.tag);
        }
      }
      if (fin_all(good)) break;
      if (fin_timed_out(t0)) {
        if (ft == 0) raise_abort(P, sm);
        break;
      }
      __nanosleep(64);
    }
  } else {
    await_tagged(P, sm, g0, P.nchunk);
    if (r1 >= 0) await_tagged(P, sm, g1, P.nchunk);
  }
  // f(q) over this thread's chunks of its row (from the registers when held)
  auto each = [&](auto&& f) {
    if (!act) return;
    if (held) {
#pragma unroll
      for (int k = 0; k < kStagePer; ++k)
        if (g + k * G < nch) f(hq[k]);
    } else {
      for (int ch = g; ch < nch; ch += G) f(ld_chunkstat(gp + ch));
    }
  };
  float m = -INFINITY;
  int fl = 0;
  each([&](const ChunkStat& q) {
    m = fmax_nan(m, q.a);
    if (isnan(q.a) || (soft && q.a == INFINITY)) fl |= SPEC_ERRF_NONFINITE;
  });
  for (int o = G >> 1; o > 0; o >>= 1) {
    m = fmax_nan(m, __shfl_xor_sync(kFull, m, o));
    fl |= __shfl_xor_sync(kFull, fl, o);
  }
  RowStat rs;
  rs.pad[0] = rs.pad[1] = rs.pad[2] = 0;
  if (soft) {
    const float mc = __fmul_rn(m, c);
    const bool finite_m = !isnan(m) && m != INFINITY && m != -INFINITY;
    float z = 0.f;
    if (!fl && finite_m) each([&](const ChunkStat& q) { z = __fadd_rn(z, chunk_weight(q.a, q.s, c, mc)); });
    for (int o = G >> 1; o > 0; o >>= 1) z = __fadd_rn(z, __shfl_xor_sync(kFull, z, o));
    const double Z = (!fl && finite_m) ? (double)z : 0.0;
    rs.Z = Z;
    rs.mc = mc;
    rs.amax = -1;
    rs.err = (fl || !finite_m || !(Z > 0.0) || isinf(Z)) ? (fl | SPEC_ERRF_NONFINITE) : 0;
  } else {
    int idx = INT_MAX;
    each([&](const ChunkStat& q) {
      if (q.a == m) idx = min(idx, __float_as_int(q.s));
    });
    for (int o = G >> 1; o > 0; o >>= 1) idx = min(idx, __shfl_xor_sync(kFull, idx, o));
    rs.Z = 0.0;
    rs.mc = m;
    rs.amax = (fl || idx == INT_MAX) ? -1 : idx;
    rs.err = fl ? SPEC_ERRF_NONFINITE : 0;
  }
  if (act && g == 0) {
    P.rstat[(size_t)b * P.rows + (i == 1 ? r1 : r0)] = rs;
    sm.srs[i] = rs;
  }
  fin_sync();
}

// The crossing inside one sub-range of a residual item: the element of target vectors
// [vt0, vt0 + kResSub) of the pair at position k where the running residual weight, taken in
// index order, first exceeds t (else the last element with positive weight; -1 when none has).
// Thread i of the finishing group reads the elements of vector vt0 + i of both rows straight from
// global memory (elements outside the row weigh 0) and keeps their weights in registers; one scan
// over the group finds the crossing thread, which finds the element.  Every thread gets the
// position relative to the range's first element.
template <typename T>
__device__ int resid_crossing(const Params& P, Shared& sm, const ResGeo<T>& q, int b, int k, float t, float c,
                              float mct, float mcd, float rho) {
  constexpr int VE = Elem<T>::kPerVec, S = Elem<T>::kSize;
  static_assert(kResSub == kFinThreads, "one vector of the sub-range per finishing thread");
  const int ft = fin_thread(), lane = ft & 31, fw = ft >> 5;
  const char* trow = row_ptr<T>(P, b, k);
  const char* drow = row_ptr<T>(P, b, P.R + k);
  float w[VE];
  float s = 0.f;
  {
    uint32_t lt[VE], ld[VE];
#pragma unroll
    for (int j = 0; j < VE; ++j) {  // every load first, then the arithmetic
      const int e = q.e_base + ft * VE + j;
      const bool in = ft < q.vt1 - q.vt0 && (unsigned)(e - q.e_lo) < (unsigned)(q.e_hi - q.e_lo);
      lt[j] = in ? Elem<T>::load_raw(trow + (size_t)e * S) : Elem<T>::kNegInf;
      ld[j] = in ? Elem<T>::load_raw(drow + (size_t)e * S) : Elem<T>::kNegInf;
    }
#pragma unroll
    for (int j = 0; j < VE; ++j) {
      const int e = q.e_base + ft * VE + j;
      const bool in = ft < q.vt1 - q.vt0 && (unsigned)(e - q.e_lo) < (unsigned)(q.e_hi - q.e_lo);
      const float et = ex2(__fmaf_rn(Elem<T>::to_float(lt[j]), c, -mct));
      const float qd = ex2(__fmaf_rn(Elem<T>::to_float(ld[j]), c, -mcd));
      w[j] = in ? fmaxf(0.f, __fmaf_rn(-qd, rho, et)) : 0.f;
      s = __fadd_rn(s, w[j]);
    }
  }
  const float incl = warp_incl_scan(s, lane);
  float excl = __shfl_up_sync(kFull, incl, 1);
  if (lane == 0) excl = 0.f;
  if (lane == 31) sm.gs.wsum[fw] = incl;
  fin_sync();
  float base = 0.f;
  for (int i = 0; i < fw; ++i) base = __fadd_rn(base, sm.gs.wsum[i]);
  const unsigned hmask = __ballot_sync(kFull, s > 0.f && __fadd_rn(base, incl) > t);
  const unsigned pmask = __ballot_sync(kFull, s > 0.f);
  if (lane == 0) {
    sm.gs.hit[fw] = hmask;
    sm.gs.pos[fw] = pmask;
  }
  fin_sync();
  int L = -1;
#pragma unroll
  for (int i = 0; i < kFinWarps; ++i)
    if (L < 0 && sm.gs.hit[i]) L = i * 32 + __ffs(sm.gs.hit[i]) - 1;
#pragma unroll
  for (int i = kFinWarps - 1; i >= 0; --i)
    if (L < 0 && sm.gs.pos[i]) L = i * 32 + 31 - __clz(sm.gs.pos[i]);
  if (L < 0) return -1;  // (uniform: no element with positive weight)
  if (ft == L) {
    float acc = __fadd_rn(base, excl);
    int pj = -1, lj = -1;
#pragma unroll
    for (int j = 0; j < VE; ++j) {
      if (w[j] > 0.f) {
        if (pj < 0 && __fadd_rn(acc, w[j]) > t) pj = j;
        lj = j;
      }
      acc = __fadd_rn(acc, w[j]);
    }
    sm.gs.out[3] = ft * VE + (pj >= 0 ? pj : lj);
  }
  fin_sync();
  const int pos = sm.gs.out[3];
  fin_sync();  // gs is free again
  return pos;
}

// Draft-model chain: the draw from max(0, p_k - q_k) at position k once every residual item of
// (b, position slot kk) is in (ts, ds: the statistics of target and draft row k).  Every thread
// gets the token (-1 after a timeout) and the residual mass.
template <typename T>
__device__ void residual_draw(const Params& P, Shared& sm, unsigned char* fbuf, uint32_t& fph, uint32_t& ssph,
                              int b, int kk, int k, float c, float u, const RowStat& ts, const RowStat& ds,
                              int* tok_out, float* mass_out) {
  constexpr int VE = Elem<T>::kPerVec;
  const int ft = fin_thread(), lane = ft & 31, fw = ft >> 5;
  const size_t bk = (size_t)b * P.npos + kk;
  // The position's sub-range sums in index order (kGroupWarps per residual item).  Thread ft takes
  // nper consecutive ones, reading them until every one carries the call's tag, and keeps them in
  // shared memory when they all fit (the sub-chunk statistics' buffer is free here).
  const TagSum* wsb0 = P.wsub + bk * P.nchunk_r * kGroupWarps;
  const int nsub = P.nchunk_r * kGroupWarps;
  const int nper = (nsub + kFinThreads - 1) / kFinThreads;
  const int j0 = ft * nper;
  float* cache = reinterpret_cast<float*>(sm.fin_ss);
  const bool cached = nsub <= kFinSs * 4;
  bool sums_ok = true;
  float s = 0.f;
  {
    const long long t0 = clock64();
    for (;;) {
      bool good = true;
      s = 0.f;
      for (int i = 0; i < nper; ++i) {
        const int j = j0 + i;
        if (j < nsub) {
          const TagSum e = ld_tagsum(wsb0 + j);
          good = good && e.t == sm.tag;
          if (cached) cache[j] = e.v;
          s = __fadd_rn(s, e.v);
        }
      }
      if (fin_all(good)) break;
      if (fin_timed_out(t0)) {
        if (ft == 0) raise_abort(P, sm);
        sums_ok = false;
        break;
      }
      __nanosleep(128);
    }
  }
  // One scan of the thread sums over the group (each warp, then the warps in order) gives the
  // total S and the thread whose running total first exceeds u S (else the last one with
  // positive weight); that thread picks the sub-range the same way among its own, and the group
  // searches it (resid_crossing).  No draw after a timeout.
  const float incl = warp_incl_scan(s, lane);
  float excl = __shfl_up_sync(kFull, incl, 1);
  if (lane == 0) excl = 0.f;
  if (lane == 31) sm.gs.wsum[fw] = incl;
  fin_sync();
  float base = 0.f, S = 0.f;
#pragma unroll
  for (int w = 0; w < kFinWarps; ++w) {
    const float ws = sm.gs.wsum[w];
    if (w < fw) base = __fadd_rn(base, ws);
    S = __fadd_rn(S, ws);
  }
  const bool any = sums_ok && S > 0.f;
  const float tgt = __fmul_rn(u, S);
  const unsigned hmask = __ballot_sync(kFull, any && s > 0.f && __fadd_rn(base, incl) > tgt);
  const unsigned pmask = __ballot_sync(kFull, any && s > 0.f);
  if (lane == 0) {
    sm.gs.hit[fw] = hmask;
    sm.gs.pos[fw] = pmask;
  }
  fin_sync();
  int L = -1;
#pragma unroll
  for (int w = 0; w < kFinWarps; ++w)
    if (L < 0 && sm.gs.hit[w]) L = w * 32 + __ffs(sm.gs.hit[w]) - 1;
#pragma unroll
  for (int w = kFinWarps - 1; w >= 0; --w)
    if (L < 0 && sm.gs.pos[w]) L = w * 32 + 31 - __clz(sm.gs.pos[w]);
  const int state = !sums_ok ? 2 : (L < 0 ? 0 : 1);  // 0: no residual mass, 1: a crossing to find
  if (state == 1 && ft == L) {  // the sub-range among the thread's own
    float acc = __fadd_rn(base, excl);
    int pj = -1, lj = -1;
    float pacc = 0.f, lacc = 0.f;
    for (int i = 0; i < nper; ++i) {
      const int j = j0 + i;
      if (j >= nsub) break;
      const float w = cached ? cache[j] : ld_tagsum(wsb0 + j).v;
      if (w > 0.f) {
        if (pj < 0 && __fadd_rn(acc, w) > tgt) {
          pj = j;
          pacc = acc;
        }
        lj = j;
        lacc = acc;
      }
      acc = __fadd_rn(acc, w);
    }
    if (pj < 0) {
      pj = lj;
      pacc = lacc;
    }
    sm.gs.out[1] = pj / kGroupWarps;
    sm.gs.out[2] = pj % kGroupWarps;
    sm.gs.fout[0] = __fsub_rn(tgt, pacc);
  }
  fin_sync();
  const int cstar = sm.gs.out[1], sstar = sm.gs.out[2];
  const float t = sm.gs.fout[0];
  const float rmass = sums_ok ? __fdiv_rn(S, (float)ts.Z) : 0.f;  // S in units of 1 / Z_t
  fin_sync();
  int tok = -1;
  if (state == 1) {
    const ResGeo<T> q = res_geo<T>(P, b, k, cstar * kResVec + sstar * kResSub, kResSub);
    const float rho = __fdiv_rn((float)ts.Z, (float)ds.Z);
    const int pos = resid_crossing<T>(P, sm, q, b, k, t, c, ts.mc, ds.mc, rho);
    tok = pos >= 0 ? q.e_base + pos : -1;
  } else if (state == 0) {  // no residual mass: draw from p
    float unused;
    SsRows none{0, 0};
    CsReader rd;
    rd.g = P.cstat + (size_t)b * P.rows * P.nchunk;
    rd.s = nullptr;
    rd.nchunk = P.nchunk;
    const DrawPlan d = draw_begin<T>(P, sm, fbuf, b, k, kFullP, -1, none);
    tok = draw_end<T>(P, sm, fbuf, fph, ssph, b, d, rd, ts, u, c, &unused);
  }
  *tok_out = tok;
  *mass_out = rmass;
}

// A draw by inverse CDF from target row `row` of request b (p, or p without token x for kExcl),
// from the row's chunk and sub-chunk statistics.  Every thread gets the token and the mass.
template <typename T>
__device__ int row_draw(const Params& P, Shared& sm, unsigned char* fbuf, uint32_t& fph, uint32_t& ssph, int b,
                        int row, int kind, int x, const RowStat& rs, float u, float c, float* mass) {
  SsRows none{0, 0};
  const DrawPlan d = draw_begin<T>(P, sm, fbuf, b, row, kind, x, none);
  CsReader rd;
  rd.g = P.cstat + (size_t)b * P.rows * P.nchunk;
  rd.s = nullptr;
  rd.nchunk = P.nchunk;
  return draw_end<T>(P, sm, fbuf, fph, ssph, b, d, rd, rs, u, c, mass);
}

// The outputs of a request (the leader warp): n, the token and the mass, or a failed request when
// err is set.  The accepted prefix was written as it was accepted.
__device__ __forceinline__ void write_outputs(const Params& P, int b, int n, int tok, float mass, int err) {
  const int lane = fin_thread() & 31, K = P.K;
  for (int i = lane; i <= K; i += 32) {
    const size_t o_i = (size_t)b * (K + 1) + i;
    if (err) {
      P.out_tokens[o_i] = -1;
      if (P.accept_prob && i < K) P.accept_prob[(size_t)b * K + i] = 0.f;
      if (P.cand_tokens) P.cand_tokens[o_i] = -1;
      if (P.pos_mass) P.pos_mass[o_i] = 0.f;
    } else if (i >= n) {
      P.out_tokens[o_i] = i == n ? tok : -1;
    }
  }
  if (lane == 0) {
    P.num_accepted[b] = err ? 0 : n;
    if (P.err_flags) P.err_flags[b] = err;
    if (P.residual_mass) P.residual_mass[b] = err ? 0.f : mass;
  }
}

// The error bits of rows r0 and r1 (r1 < 0: none) of request b from their chunk maxima alone (a
// NaN; where a softmax is taken, +inf or only -inf): all a decided request still needs of a
// later position (the group waits for the tags; the leader warp decides).
__device__ inline int stage_errors(const Params& P, Shared& sm, int b, int r0, int r1, bool soft) {
  const ChunkStat* g0 = P.cstat + ((size_t)b * P.rows + r0) * P.nchunk;
  const ChunkStat* g1 = r1 >= 0 ? P.cstat + ((size_t)b * P.rows + r1) * P.nchunk : g0;
  await_tagged(P, sm, g0, P.nchunk);
  if (r1 >= 0) await_tagged(P, sm, g1, P.nchunk);
  int e = 0;
  if (fin_thread() < 32) {
    const int lane = fin_thread() & 31;
    float m0 = -INFINITY, m1 = -INFINITY;
    int f = 0;
    for (int i = lane; i < P.nchunk; i += 32) {
      const float a = ld_chunkstat(g0 + i).a, d = r1 >= 0 ? ld_chunkstat(g1 + i).a : -INFINITY;
      m0 = fmax_nan(m0, a);
      m1 = fmax_nan(m1, d);
      f |= (isnan(a) || isnan(d) || (soft && (a == INFINITY || d == INFINITY))) ? 1 : 0;
    }
    m0 = warp_max_nan(m0);
    m1 = warp_max_nan(m1);
    f = warp_or(f);
    if (f || (soft && (m0 == -INFINITY || (r1 >= 0 && m1 == -INFINITY)))) e = SPEC_ERRF_NONFINITE;
  }
  return e;
}

// The bonus token of request j from its bonus row's statistics (q.rt): the row's argmax for a
// greedy request, else the draw from p_K (section I.1's bonus read as R6).  With the bonus stage
// streamed first it is made then, ahead of the acceptance tests, so that a request that accepts
// every draft has its token at once.  Per-position outputs of the draft-model and n-gram chains
// make their draws at the end instead.
template <int MODE, typename T, bool PT>
__device__ void bonus_token(const Params& P, Shared& sm, unsigned char* fbuf, uint32_t& fph, uint32_t& ssph,
                            int j) {
  constexpr bool kSoftmax = (MODE == kChain || MODE == kNgram);
  const int ft = fin_thread();
  FinReq& q = sm.fr[j];
  const bool soft = PT ? !q.greedy : kSoftmax;
  const bool late = P.diag && (MODE == kNgram || (MODE == kChain && P.npos > 0));
  if (!soft) {
    if (ft == 0) {
      q.btok = q.rt.amax;
      q.bmass = 1.f;
    }
  } else if (!q.err && !late) {
    float mass;
    const int tok = row_draw<T>(P, sm, fbuf, fph, ssph, q.b, P.K, kFullP, -1, q.rt, q.u, PT ? q.c : P.c, &mass);
    if (ft == 0) {
      q.btok = tok;
      q.bmass = mass;
    }
  }
  fin_sync();
}

// The result of request j is decided at its position n (x: the draft token there).
template <int MODE, typename T, bool PT>
__device__ void decide(const Params& P, Shared& sm, unsigned char* fbuf, uint32_t& fph, uint32_t& ssph, int j,
                       int x) {
  constexpr bool kSoftmax = (MODE == kChain || MODE == kNgram);
  const int ft = fin_thread(), lane = ft & 31;
  FinReq& q = sm.fr[j];
  const int b = q.b, n = q.n, K = P.K, err = q.err;
  const bool soft = PT ? !q.greedy : kSoftmax;
  const float c = PT ? q.c : P.c;
  const bool resid_calls = MODE == kChain && P.npos > 0;           // the call runs residual passes
  const bool late = P.diag && (MODE == kNgram || resid_calls);     // per-position draws, all at the end
  if (resid_calls && !P.diag) {
    // publish the result (with the error bits seen so far), then queue the request: its residual
    // items are handed out in queue order, once the producers see the words complete
    if (ft < 32) {
      const bool resid = soft && !err && n < K;
      const bool wl = lane == 0 || (resid && lane < 4);  // the lanes that write a result word
      unsigned long long word = 0ull;
      if (wl) {
        unsigned hi = (unsigned)n | ((unsigned)err << 16) | (soft ? 0u : kNoResid);
        if (lane > 0)
          hi = __float_as_uint(lane == 1 ? q.rt.mc : lane == 2 ? q.rd.mc : __fdiv_rn((float)q.rt.Z, (float)q.rd.Z));
        word = ((unsigned long long)hi << 32) | sm.tag;
        st_volatile_u64(P.req[b].w + lane, word);
      }
      // the queue entry: its slot, then the same words and the request's index
      unsigned slot = 0u;
      if (lane == 0) slot = atomicAdd(P.rq_tail, 1u);
      slot = __shfl_sync(kFull, slot, 0);
      unsigned long long* qw = P.rq + (size_t)slot * kQWords;
      if (wl) st_volatile_u64(qw + lane, word);
      if (lane == 0) {
        st_volatile_u64(qw + 4, ((unsigned long long)(unsigned)b << 32) | sm.tag);
        q.resid = resid ? 1 : 0;
      }
    }
  } else if (!(resid_calls && P.diag) && ft == 0) {
    // the result word (read by the probability rows' kernel)
    const unsigned hi = (unsigned)n | ((unsigned)err << 16);
    st_volatile_u64(P.req[b].w, ((unsigned long long)hi << 32) | sm.tag);
  }
  if (!soft || err) {  // greedy: the argmax of row n; a failed request draws nothing
    if (ft == 0) {
      q.tok = err ? -1 : (n == K ? q.btok : q.rt.amax);
      q.mass = err ? 0.f : 1.f;
      q.drawn = 1;
    }
  } else if (n == K && !late) {  // the bonus token, made from the first stage
    if (ft == 0) {
      q.tok = q.btok;
      q.mass = q.bmass;
      q.drawn = 1;
      // (per-position outputs of a chain without residual passes: its one position, the bonus row)
      if (P.cand_tokens) P.cand_tokens[(size_t)b * (K + 1) + n] = q.btok;
      if (P.pos_mass) P.pos_mass[(size_t)b * (K + 1) + n] = q.bmass;
    }
  } else if (MODE == kNgram && !late) {  // the n-gram residual, now
    float mass;
    const int tok = row_draw<T>(P, sm, fbuf, fph, ssph, b, n, (MODE == kNgram && n < K) ? kExcl : kFullP,
                                n < K ? x : -1, q.rt, q.u, c, &mass);
    if (ft == 0) {
      q.tok = tok;
      q.mass = mass;
      q.drawn = 1;
      // (per-position outputs of a chain without residual passes: its one position, the bonus row)
      if (P.cand_tokens) P.cand_tokens[(size_t)b * (K + 1) + n] = tok;
      if (P.pos_mass) P.pos_mass[(size_t)b * (K + 1) + n] = mass;
    }
  }
  fin_sync();
  // the outputs as far as known now (a later error rewrites them)
  if (q.drawn && !err && !late) {
    if (ft < 32) write_outputs(P, b, n, q.tok, q.mass, 0);
    if (ft == 0) q.written = 1;
  }
  fin_sync();
}

// The residual draw of request j, whose residual items are all in; its outputs follow when no
// error has turned up so far (draft-model chains without per-position outputs).
template <typename T, bool PT>
__device__ void early_residual_draw(const Params& P, Shared& sm, unsigned char* fbuf, uint32_t& fph,
                                    uint32_t& ssph, int j) {
  const int ft = fin_thread();
  FinReq& q = sm.fr[j];
  if (ft == 0) P.tick_b[(size_t)q.b * P.npos] = 0;  // complete: left as the next call expects it
  int tok;
  float mass;
  residual_draw<T>(P, sm, fbuf, fph, ssph, q.b, 0, q.n, PT ? q.c : P.c, q.u, q.rt, q.rd, &tok, &mass);
  if (ft == 0) {
    q.tok = tok;
    q.mass = mass;
    q.drawn = 1;
  }
  fin_sync();
  if (!q.err) {
    if (ft < 32) write_outputs(P, q.b, q.n, tok, mass, 0);
    if (ft == 0) q.written = 1;
  }
  fin_sync();
}

// Waits (bounded) until *count reaches `want`, making meanwhile the residual draws of the requests
// j < own whose residual items come in (draft-model chains without per-position outputs), so that
// a late rejection's draw does not wait for the end of the stream.  False after a timeout.
template <int MODE, typename T, bool PT>
__device__ bool wait_stage(const Params& P, Shared& sm, unsigned char* fbuf, uint32_t& fph, uint32_t& ssph,
                           int own, const unsigned* count, unsigned want) {
  if (!(MODE == kChain && P.npos > 0 && !P.diag)) return wait_count(P, sm, count, want);
  const int ft = fin_thread();
  long long t0 = clock64();
  for (;;) {
    if (ft == 0) {
      int act = 0;  // 1: the count is in; 2 + j: request j's residual items are in; -1: gave up
      if (ld_acquire_u32(count) >= want) {
        act = 1;
      } else {
        for (int j = 0; j < own && !act; ++j) {
          const FinReq& q = sm.fr[j];
          if (q.resid && !q.drawn && ld_acquire_u32(P.tick_b + (size_t)q.b * P.npos) >= (unsigned)P.nchunk_r)
            act = 2 + j;
        }
        if (!act && (aborted(sm) || clock64() - t0 > kWaitLimitCycles)) {
          raise_abort(P, sm);
          act = -1;
        }
      }
      sm.gs.out[3] = act;
    }
    fin_sync();
    const int act = sm.gs.out[3];
    fin_sync();
    if (act == 1) return true;
    if (act < 0) return false;
    if (act >= 2) {
      early_residual_draw<T, PT>(P, sm, fbuf, fph, ssph, act - 2);
      t0 = clock64();
      continue;
    }
    __nanosleep(64);
  }
}

// Stage s of request j: waits for the stage's rows, combines them, makes the acceptance test.
// False after a timeout.
template <int MODE, typename T, bool PT>
__device__ bool finish_stage(const Params& P, Shared& sm, unsigned char* fbuf, uint32_t& fph, uint32_t& ssph,
                             int j, int s, int own) {
  constexpr int S = Elem<T>::kSize;
  constexpr bool kSoftmax = (MODE == kChain || MODE == kNgram);
  const int ft = fin_thread();
  FinReq& q = sm.fr[j];
  const int b = q.b, K = P.K, R = P.R;
  const bool soft = PT ? !q.greedy : kSoftmax;
  const float c = PT ? q.c : P.c;
  const bool pair = MODE == kChain && soft && s < K;  // the stage holds the draft row too
  // the position's inputs, loaded by the leader while the stage's rows stream in
  int x = 0;
  float rr = 0.f, lx = 0.f, dx = 0.f;
  if (ft == 0 && s < K) {
    x = __ldg(P.draft_tokens + (size_t)b * K + s);
    if (soft) {
      rr = __ldg(P.r + (size_t)b * K + s);
      if (x >= 0 && x < P.V) {
        lx = Elem<T>::to_float(Elem<T>::load_raw(row_ptr<T>(P, b, s) + (size_t)x * S));
        if (MODE == kChain) dx = Elem<T>::to_float(Elem<T>::load_raw(row_ptr<T>(P, b, R + s) + (size_t)x * S));
      }
    }
  }
  unsigned* tick = P.tick_a + (size_t)b * R + s;
  if (!wait_stage<MODE, T, PT>(P, sm, fbuf, fph, ssph, own, tick, (unsigned)P.nchunk * (pair ? 2u : 1u)))
    return false;
  if (ft == 0) *tick = 0;  // complete: the count is left as the next call expects it
  // a request already decided needs only the error bits of its later rows, unless the call asks
  // for outputs at every position (or the rows' statistics)
  if (q.n >= 0 && !P.diag && !P.accept_prob && !P.target_probs && !P.draft_probs) {
    const int e = stage_errors(P, sm, b, s, pair ? R + s : -1, soft);
    if (ft == 0) q.err |= e | ((s < K && (x < 0 || x >= P.V)) ? SPEC_ERRF_BAD_TOKEN : 0);
    fin_sync();
    return true;
  }
  combine_stage(P, sm, b, s, pair ? R + s : -1, soft, c);
  if (ft == 0) {
    const RowStat t = sm.srs[0], d = sm.srs[1];
    int e = t.err | (pair ? d.err : 0);
    float alpha = 0.f;
    bool acc = false;
    const size_t o_s = (size_t)b * (K + 1) + s;
    if (s < K) {
      if (x < 0 || x >= P.V) {
        e |= SPEC_ERRF_BAD_TOKEN;
      } else if (soft) {
        // alpha = p(x) / q(x) = 2^((l_x c - mc_t) - (d_x c - mc_d)) Z_d / Z_t (draft model), or
        // p(x) = 2^(l_x c - mc_t) / Z_t (one-hot draft); capped at 1
        const Exp2 ext = scaled_logit(lx, c, t.mc);
        if (MODE == kChain) {
          if (dx == -INFINITY)
            alpha = 1.f;  // q(x) = 0
          else if (lx == -INFINITY)
            alpha = 0.f;  // p(x) = 0
          else
            alpha = fminf(exp2_times(exp2_sub(ext, scaled_logit(dx, c, d.mc)), __fdiv_rn((float)d.Z, (float)t.Z)),
                          1.f);
        } else {
          alpha = fminf(lx == -INFINITY ? 0.f : exp2_times(ext, __frcp_rn((float)t.Z)), 1.f);
        }
        acc = rr <= alpha;
      } else {
        alpha = (x == t.amax) ? 1.f : 0.f;
        acc = alpha == 1.f;
      }
      if (P.accept_prob) P.accept_prob[(size_t)b * K + s] = alpha;
    }
    if (!soft) {  // greedy per-position outputs: the row's argmax
      if (P.cand_tokens) P.cand_tokens[o_s] = t.amax;
      if (P.pos_mass) P.pos_mass[o_s] = 1.f;
    }
    q.err |= e;
    int decided = 0;
    if (s == K) {  // the bonus row: its statistics are kept for the bonus draw
      if (q.n < 0) {
        q.rt = t;
        q.rd = d;
        if (!P.bonus_first || K == 0) {  // (streamed last: every draft was accepted)
          q.n = K;
          decided = 1;
        }
      }
    } else if (q.n < 0) {
      if (acc) {
        P.out_tokens[o_s] = x;
        if (P.bonus_first && s == K - 1) {  // every draft accepted: the bonus token, made already
          q.n = K;
          decided = 1;
        }
      } else {
        q.n = s;
        q.rt = t;
        q.rd = d;
        decided = 1;
      }
    }
    sm.gs.out[0] = decided;
    sm.gs.out[1] = x;
  }
  fin_sync();
  const int decided = sm.gs.out[0], xs = sm.gs.out[1];
  fin_sync();
  if (s == K && (P.bonus_first || decided)) bonus_token<MODE, T, PT>(P, sm, fbuf, fph, ssph, j);
  if (decided) decide<MODE, T, PT>(P, sm, fbuf, fph, ssph, j, xs);
  return true;
}

// Request j once every stage is in: the remaining draws, then the outputs.  False after a timeout.
template <int MODE, typename T, bool PT>
__device__ bool finalize_request(const Params& P, Shared& sm, unsigned char* fbuf, uint32_t& fph, uint32_t& ssph,
                                 int j) {
  constexpr bool kSoftmax = (MODE == kChain || MODE == kNgram);
  const int ft = fin_thread(), lane = ft & 31;
  FinReq& q = sm.fr[j];
  const int b = q.b, n = q.n, K = P.K, R = P.R;
  const bool soft = PT ? !q.greedy : kSoftmax;
  const float c = PT ? q.c : P.c;
  const int err = (PT && q.bad) ? SPEC_ERRF_BAD_TEMPERATURE : q.err;
  const bool draws = soft && !err;
  auto put_cand = [&](int k, int tok, float mass) {
    if (ft == 0) {
      if (P.cand_tokens) P.cand_tokens[(size_t)b * (K + 1) + k] = tok;
      if (P.pos_mass) P.pos_mass[(size_t)b * (K + 1) + k] = mass;
    }
  };
  if (MODE == kChain && P.npos > 0) {
    if (P.diag) {
      // per-position outputs: now that every row's statistics are in, publish the result and queue
      // the request; the producers read each position's parameters from the row statistics
      if (ft == 0) {
        __threadfence();
        const unsigned hi = (unsigned)n | ((unsigned)err << 16) | (soft ? 0u : kNoResid);
        const unsigned long long word = ((unsigned long long)hi << 32) | sm.tag;
        st_volatile_u64(P.req[b].w, word);
        const unsigned slot = atomicAdd(P.rq_tail, 1u);
        unsigned long long* qw = P.rq + (size_t)slot * kQWords;
        st_volatile_u64(qw, word);
        st_volatile_u64(qw + 4, ((unsigned long long)(unsigned)b << 32) | sm.tag);
      }
      if (draws) {
        for (int kk = 0; kk < K; ++kk) {
          if (!wait_count(P, sm, P.tick_b + (size_t)b * P.npos + kk, (unsigned)P.nchunk_r)) return false;
          if (ft == 0) P.tick_b[(size_t)b * P.npos + kk] = 0;
          const RowStat ts = ld_rowstat(P.rstat + (size_t)b * P.rows + kk);
          const RowStat ds = ld_rowstat(P.rstat + (size_t)b * P.rows + R + kk);
          int tok;
          float mass;
          residual_draw<T>(P, sm, fbuf, fph, ssph, b, kk, kk, c, q.u, ts, ds, &tok, &mass);
          put_cand(kk, tok, mass);
          if (ft == 0 && kk == n) {
            q.tok = tok;
            q.mass = mass;
          }
        }
        float mass;
        const RowStat tb = ld_rowstat(P.rstat + (size_t)b * P.rows + K);
        const int tok = row_draw<T>(P, sm, fbuf, fph, ssph, b, K, kFullP, -1, tb, q.u, c, &mass);
        put_cand(K, tok, mass);
        if (ft == 0 && n == K) {
          q.tok = tok;
          q.mass = mass;
        }
      }
    } else if (q.resid && !q.drawn) {  // the residual pass published at the decision (its result is
                                       // used only when no error turned up since)
      // The draw waits for the residual sums themselves (their tags), not for their count, which
      // saves a round trip; the count returns to zero once its last increments land, as the next
      // call expects it.
      if (ft == 0) atomicAdd(P.tick_b + (size_t)b * P.npos, 0u - (unsigned)P.nchunk_r);
      int tok;
      float mass;
      residual_draw<T>(P, sm, fbuf, fph, ssph, b, 0, n, c, q.u, q.rt, q.rd, &tok, &mass);
      if (ft == 0) {
        q.tok = tok;
        q.mass = mass;
      }
    }
  }
  if (MODE == kNgram && P.diag && draws) {  // per-position outputs: a draw at every position
    for (int k = 0; k <= K; ++k) {
      const RowStat rs = ld_rowstat(P.rstat + (size_t)b * P.rows + k);
      const int x = k < K ? __ldg(P.draft_tokens + (size_t)b * K + k) : -1;
      float mass;
      const int tok = row_draw<T>(P, sm, fbuf, fph, ssph, b, k, k < K ? kExcl : kFullP, x, rs, q.u, c, &mass);
      put_cand(k, tok, mass);
      if (ft == 0 && k == n) {
        q.tok = tok;
        q.mass = mass;
      }
    }
  }
  fin_sync();
  // the outputs, unless they were written already and no error turned up since
  if ((err || !q.written) && ft < 32) write_outputs(P, b, n, q.tok, q.mass, err);
  fin_sync();
  return true;
}

// The finishing group of a chain mode: its requests, kOwnMax at a time, position by position.
template <int MODE, typename T, bool PT>
__device__ void fin_loop_chain(const Params& P, Shared& sm, unsigned char* fbuf) {
  constexpr bool kSoftmax = (MODE == kChain || MODE == kNgram);
  const int ft = fin_thread();
  uint32_t fph = 0, ssph = 0;
  const int G = (int)gridDim.x;
  for (int b0 = blockIdx.x; b0 < P.B; b0 += kOwnMax * G) {
    const int own = min(kOwnMax, (P.B - b0 + G - 1) / G);
    if (ft < own) {
      FinReq& q = sm.fr[ft];
      q.b = b0 + ft * G;
      q.n = -1;
      q.err = 0;
      q.tok = -1;
      q.resid = 0;
      q.drawn = 0;
      q.written = 0;
      q.btok = -1;
      q.bmass = 0.f;
      q.mass = 0.f;
      const ReqTemp rt = req_temp<MODE, PT>(P, q.b);
      q.c = rt.c;
      q.greedy = rt.greedy;
      q.bad = rt.bad;
      q.u = kSoftmax ? __ldg(P.u + q.b) : 0.f;
    }
    fin_sync();
    for (int it = 0; it <= P.K; ++it) {  // the stages in stream order
      const int s = P.bonus_first ? (it == 0 ? P.K : it - 1) : it;
      for (int j = 0; j < own; ++j)
        if (!finish_stage<MODE, T, PT>(P, sm, fbuf, fph, ssph, j, s, own)) return;
    }
    for (int j = 0; j < own; ++j)
      if (!finalize_request<MODE, T, PT>(P, sm, fbuf, fph, ssph, j)) return;
  }
}

// Greedy tree walk (section III.2): from the root, move to the child whose token equals the
// argmax of the current node's row (lowest node index first) until none does.  The group checks
// the tree, writes the per-node argmax and clears the outputs; the leader then walks and writes
// the path.
__device__ inline void walk_tree(const Params& P, Shared& sm, int b) {
  const int ft = fin_thread(), lane = ft & 31;
  const int N1 = P.R, V = P.V;
  const RowStat* rs = P.rstat + (size_t)b * N1;
  const int32_t* par = P.parents + (size_t)b * N1;
  const int32_t* tok = P.node_tokens + (size_t)b * N1;
  if (N1 <= kFinRows) {  // a small tree's parents and tokens were staged in shared memory
    par = sm.fin_par;
    tok = sm.fin_tok;
  }
  int32_t* path = P.path_nodes + (size_t)b * N1;
  int32_t* out = P.out_tokens + (size_t)b * N1;
  int e = 0;
  for (int i = ft; i < N1; i += kFinThreads) {
    e |= i < kFinRows ? sm.fin_rs[i].err : __ldcg(&rs[i].err);
    const int p = par[i];
    if (i == 0 ? (p != -1) : (p < 0 || p >= i)) e |= SPEC_ERRF_BAD_TREE;
    if (i > 0) {
      const int t = tok[i];
      if (t < 0 || t >= V) e |= SPEC_ERRF_BAD_TOKEN;
    }
    if (P.node_argmax) P.node_argmax[(size_t)b * N1 + i] = i < kFinRows ? sm.fin_rs[i].amax : __ldcg(&rs[i].amax);
    path[i] = -1;
    out[i] = -1;
  }
  // the error bits, agreed by the group (one barrier per bit)
  int err = 0;
  if (!fin_all(!(e & SPEC_ERRF_NONFINITE))) err |= SPEC_ERRF_NONFINITE;
  if (!fin_all(!(e & SPEC_ERRF_BAD_TREE))) err |= SPEC_ERRF_BAD_TREE;
  if (!fin_all(!(e & SPEC_ERRF_BAD_TOKEN))) err |= SPEC_ERRF_BAD_TOKEN;
  if (ft >= 32) return;
  int len = 0;
  if (!err) {
    int cur = 0;
    if (lane == 0) path[0] = 0;
    for (int step = 0; step < N1; ++step) {  // cur strictly increases: at most N1 - 1 moves
      const int a = cur < kFinRows ? sm.fin_rs[cur].amax : __ldcg(&rs[cur].amax);
      int next = -1;
      for (int c0 = cur + 1; c0 < N1 && next < 0; c0 += 32) {
        const int cc = c0 + lane;
        const bool m = cc < N1 && par[cc] == cur && tok[cc] == a;
        const unsigned bal = __ballot_sync(kFull, m);
        if (bal) next = c0 + __ffs(bal) - 1;
      }
      if (next < 0) {
        if (lane == 0) out[len] = a;
        break;
      }
      if (lane == 0) {
        out[len] = tok[next];
        path[len + 1] = next;
      }
      ++len;
      cur = next;
    }
  }
  if (lane == 0) {
    P.accept_len[b] = err ? 0 : len;
    if (P.err_flags) P.err_flags[b] = err;
  }
}

// The finishing group's loop over its requests (trees; the chain modes take fin_loop_chain).
template <int MODE, typename T, bool PT>
__device__ void fin_loop(const Params& P, Shared& sm, unsigned char* fbuf) {
  if constexpr (MODE != kTree) {
    fin_loop_chain<MODE, T, PT>(P, sm, fbuf);
  } else {
    const int ft = fin_thread();
    uint32_t csph = 0;
    const unsigned per_req = (unsigned)(P.rows * P.nchunk);
    for (int b = blockIdx.x; b < P.B; b += gridDim.x) {
      const int N1 = P.R;
      if (N1 <= kFinRows) {
        for (int i = ft; i < N1; i += kFinThreads) {
          sm.fin_par[i] = __ldg(P.parents + (size_t)b * N1 + i);
          sm.fin_tok[i] = __ldg(P.node_tokens + (size_t)b * N1 + i);
        }
      }
      if (!wait_count(P, sm, P.tick_a + b, per_req)) return;
      if (ft == 0) P.tick_a[b] = 0;  // complete: the count is left as the next call expects it
      SsRows none{0, 0};
      const CsReader rd = stage_request_stats(P, sm, b, none, csph, P.rows);
      combine_rows<MODE, false>(P, sm, b, rd, false, 0.f, P.rows);
      walk_tree(P, sm, b);
      fin_sync();  // the walk's reads of the shared copies come before the next request's writes
    }
  }
}

// --------------------------------------------------------------------------- kernel ----
template <int MODE, typename T, bool PT>
__global__ void __launch_bounds__(kThreads, 1) verify_kernel(const Params P) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ Shared sm;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kGroupWarps);
    }
    for (int j = 0; j < kSlots; ++j) {
      mbar_init(&sm.pfull[j], 1);
      mbar_init(&sm.pempty[j], 1);
      sm.pcnt[j] = 0;
    }
    mbar_init(&sm.fin_bar, 1);
    mbar_init(&sm.cs_bar, 1);
    mbar_init(&sm.ss_bar, 1);
    sm.abort = 0;
    sm.tag_ready = 0;
    fence_mbar_init();
  }
  __syncthreads();
  unsigned char* fbuf = smem + (size_t)kStages * kStageBytes;
  if (warp >= kProducerWarp && warp < kProducerWarp + kGroups) {
    // the producers start the stream at once: a stats copy needs no tag
    producer_loop<MODE, T, PT>(P, sm, smem, warp - kProducerWarp);
  } else {
    // this call's tag: one past the workspace's last (its epoch, left by the last CTA of the
    // previous call), so that calls replayed from a captured graph get fresh tags too; every
    // other role waits for it (named barrier kTagBarrier), while the first copies are in flight
    if (tid == 0) {
      const unsigned e = __ldg(P.epoch);
      sm.tag = (e + 1u) != 0u ? e + 1u : 1u;
      __threadfence_block();
      *reinterpret_cast<volatile int*>(&sm.tag_ready) = 1;
    }
    asm volatile("bar.sync %0, %1;" ::"n"(kTagBarrier), "n"(kThreads - kGroups * 32) : "memory");
    if (warp < kConsWarps)
      consumer_loop<MODE, T, PT>(P, sm, smem);
    else if (warp == kBookWarp)
      book_loop<MODE>(P, sm);
    else
      fin_loop<MODE, T, PT>(P, sm, fbuf);  // warps kFinWarp .. kFinWarp + kFinWarps - 1
  }
  __syncthreads();
  // The last CTA out reports a timed-out call (never expected) on every request, and leaves the
  // counters zero for the next call (after a timeout the counts too: finishing groups that gave
  // up did not zero theirs).
  if (tid == 0) {
    // count this CTA out, with release and acquire semantics in one atomic; a CTA that gave up
    // (the only way the timeout flag gets set) adds kExitAbort as well, so that the last one out
    // learns of a timeout from the count alone
    const unsigned add = 1u + (aborted(sm) ? kExitAbort : 0u);
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(P.exit_tick), "r"(add) : "memory");
    sm.last = ((old + add) & (kExitAbort - 1u)) == gridDim.x;
    sm.timed_out = (old + add) >= kExitAbort;
  }
  __syncthreads();
  if (sm.last) {
    const bool timed_out = sm.timed_out;
    if (tid == 0) {
      *P.work = 0u;
      *P.rc = 0u;
      if (P.rq_tail) *P.rq_tail = 0u;
      *P.gerr = 0u;
      *P.exit_tick = 0u;
      *P.epoch = sm.tag;
    }
    if (timed_out) {
      const int na = (MODE == kTree) ? P.B : P.B * P.R;  // counts per request, or per request and position
      for (int i = tid; i < na; i += kThreads) P.tick_a[i] = 0u;
      for (int i = tid; i < P.B * P.npos; i += kThreads) P.tick_b[i] = 0u;
      const int width = (MODE == kTree) ? P.R : P.K + 1;
      for (int b = tid; b < P.B; b += kThreads) {
        if (P.err_flags) P.err_flags[b] = SPEC_ERRF_TIMEOUT;
        if (MODE == kTree) {
          P.accept_len[b] = 0;
          for (int i = 0; i < width; ++i) P.path_nodes[(size_t)b * width + i] = -1;
        } else {
          P.num_accepted[b] = 0;
          if (P.residual_mass) P.residual_mass[b] = 0.f;
        }
        for (int i = 0; i < width; ++i) P.out_tokens[(size_t)b * width + i] = -1;
      }
    }
  }
}

// ---------------------------------------------------------------------- probs kernel ----
// Testing aid: p_i = 2^(l_i c - mc) / Z for every target row, q likewise for draft rows.
template <typename T>
__global__ void __launch_bounds__(256) probs_kernel(const Params P) {
  const int rowid = blockIdx.x;  // b * rows + r
  const int b = rowid / P.rows, r = rowid - b * P.rows;
  const unsigned long long w0 = P.req[b].w[0];
  // (the verification kernel before this one left its tag as the epoch; a row with an error, or of
  // a request that failed, has no distribution to write)
  if (!req_word_ok(w0, *P.epoch) || (req_word_hi(w0) >> 16) != 0u) return;
  float* out = r < P.R ? (P.target_probs ? P.target_probs + ((size_t)b * P.R + r) * P.V : nullptr)
                       : (P.draft_probs ? P.draft_probs + ((size_t)b * P.K + (r - P.R)) * P.V : nullptr);
  if (!out) return;
  float c = P.c;
  if (P.temps) {  // per-request temperatures: rows of greedy requests have no softmax to write
    const float Tb = P.temps[b];
    if (!(Tb > 0.f) || isinf(Tb)) return;
    c = (float)(1.4426950408889634 / (double)Tb);
  }
  const RowStat rs = P.rstat[rowid];
  if (rs.err || !(rs.Z > 0.0)) return;
  const char* rp = row_ptr<T>(P, b, r);
  const float invZ = (float)(1.0 / rs.Z);
  for (int i = (int)threadIdx.x; i < P.V; i += 256) {
    const float l = Elem<T>::to_float(Elem<T>::load_raw(rp + (size_t)i * Elem<T>::kSize));
    out[i] = __fmul_rn(ex2(__fmaf_rn(l, c, -rs.mc)), invZ);
  }
}

// -------------------------------------------------------------------------- launchers ----
struct LaunchPlan {
  size_t smem;       // dynamic shared memory of verify_kernel
  int launch_probs;  // launch probs_kernel
  int sm_count;      // multiprocessors of the current device
  int device;        // the current device
};

template <int MODE, typename T, bool PT>
cudaError_t launch_mode(const Params& P, const LaunchPlan& L, cudaStream_t stream) {
  auto ks = verify_kernel<MODE, T, PT>;
  // the shared-memory opt-in and the occupancy, once per device (the same values every call)
  constexpr int kMaxDev = 64;
  static int resident[kMaxDev] = {0};
  int per_sm = (L.device >= 0 && L.device < kMaxDev) ? resident[L.device] : 0;
  cudaError_t e = cudaSuccess;
  if (per_sm < 1) {
    e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.smem);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ks, kThreads, L.smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    if (L.device >= 0 && L.device < kMaxDev) resident[L.device] = per_sm;
  }
  const long long cap = (long long)per_sm * L.sm_count;
  const long long grid = (long long)P.total < cap ? (long long)P.total : cap;
  if (grid >= (long long)kExitAbort) return cudaErrorInvalidConfiguration;  // (the exit count's range)
  ks<<<(unsigned)grid, kThreads, L.smem, stream>>>(P);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (L.launch_probs) {
    probs_kernel<T><<<(unsigned)((long long)P.B * P.rows), 256, 0, stream>>>(P);
    e = cudaGetLastError();
  }
  return e;
}

template <typename T>
cudaError_t launch_verify(int mode, const Params& P, const LaunchPlan& L, cudaStream_t stream) {
  switch (mode) {
    case kChain: return launch_mode<kChain, T, false>(P, L, stream);
    case kNgram: return launch_mode<kNgram, T, false>(P, L, stream);
    case kGreedy: return launch_mode<kGreedy, T, false>(P, L, stream);
    case kTree: return launch_mode<kTree, T, false>(P, L, stream);
    case kChainPT: return launch_mode<kChain, T, true>(P, L, stream);
    case kNgramPT: return launch_mode<kNgram, T, true>(P, L, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace specv
