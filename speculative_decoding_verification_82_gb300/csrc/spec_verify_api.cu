// spec_verify_api.cu -- the C ABI: argument checks, chunk planning, workspace layout, launch.
//
// Host side only; the kernels live in verify_kernel.cuh (instantiated per element type in
// spec_verify_{f32,bf16,f16}.cu).  No call allocates memory or synchronises the host.
#include <math.h>
#include <stdlib.h>

#include <climits>

#include "spec_verify.h"
#include "verify_kernel.cuh"

namespace specv {
extern template cudaError_t launch_verify<float>(int, const Params&, const LaunchPlan&, cudaStream_t);
extern template cudaError_t launch_verify<__nv_bfloat16>(int, const Params&, const LaunchPlan&, cudaStream_t);
extern template cudaError_t launch_verify<__half>(int, const Params&, const LaunchPlan&, cudaStream_t);
}  // namespace specv

namespace {

using specv::ChunkStat;
using specv::Params;
using specv::ReqState;
using specv::RowStat;

constexpr size_t kDefaultChunkBytes = 32 * 1024;

int elem_size(spec_dtype_t dt) { return dt == SPEC_DTYPE_F32 ? 4 : 2; }
bool dtype_ok(int dt) { return dt == SPEC_DTYPE_F32 || dt == SPEC_DTYPE_BF16 || dt == SPEC_DTYPE_F16; }
size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Bytes of logits staged per chunk.  ~32 KB: two stages per CTA and three CTAs per SM keep
// about six chunks in flight per SM.  SPEC_VERIFY_CHUNK_BYTES overrides it (tuning; 4 KB..64 KB).
size_t chunk_target() {
  static const size_t v = [] {
    const char* s = getenv("SPEC_VERIFY_CHUNK_BYTES");
    const long x = s ? atol(s) : 0;
    return (x >= 4096 && x <= 65536) ? (size_t)x : kDefaultChunkBytes;
  }();
  return v;
}

struct Chunking {
  int chunk, nchunk, buf_bytes;
};

// Splits a row of V elements into nchunk near-equal chunks of `chunk` elements (a multiple of 8).
Chunking plan_chunks(int V, int S) {
  Chunking c;
  const size_t row = (size_t)V * S;
  size_t n0 = (row + chunk_target() - 1) / chunk_target();
  if (n0 < 1) n0 = 1;
  long long chunk = ((long long)V + (long long)n0 - 1) / (long long)n0;
  chunk = (chunk + 7) / 8 * 8;
  c.chunk = (int)chunk;
  c.nchunk = (int)(((long long)V + chunk - 1) / chunk);
  c.buf_bytes = c.chunk * S + 32;
  return c;
}

// Workspace layout:
//   work    u32                  work-item counter  } one region, cleared by one
//   tick_a  [B] u32              request tickets    } cudaMemsetAsync per call
//   tick_b  [B][Kc] u32          residual tickets   } (Kc = rows >= K)
//   cstat   [B][rows][nchunk]    ChunkStat          (256-byte aligned regions from here on)
//   rstat   [B][rows]            RowStat
//   req     [B]                  ReqState
//   wsum    [B][Kc][nchunk]      float
struct Layout {
  size_t work, tick_a, tick_b, cstat, rstat, req, wsum, total;
};

Layout layout(int B, int rows, int nchunk) {
  Layout L;
  const size_t b = (size_t)B, r = (size_t)rows, n = (size_t)nchunk;
  size_t off = 0;
  L.work = off;
  off += 4;
  L.tick_a = off;
  off += b * 4;
  L.tick_b = off;
  off = align_up(off + b * r * 4, 256);
  L.cstat = off;
  off = align_up(off + b * r * n * sizeof(ChunkStat), 256);
  L.rstat = off;
  off = align_up(off + b * r * sizeof(RowStat), 256);
  L.req = off;
  off = align_up(off + b * sizeof(ReqState), 256);
  L.wsum = off;
  off = align_up(off + b * r * n * sizeof(float), 256);
  L.total = off;
  return L;
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
  static int cache[64] = {0};
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (dev < 64) cache[dev] = n;
  return n;
}

bool aligned_to(const void* p, int a) { return ((uintptr_t)p % (uintptr_t)a) == 0; }

spec_status_t attach_workspace(Params& P, void* ws, size_t bytes, int B, int rows) {
  const Layout L = layout(B, rows, P.nchunk);
  if (ws == nullptr || bytes < L.total) return SPEC_ERR_WORKSPACE;
  if (((uintptr_t)ws & 255u) != 0) return SPEC_ERR_WORKSPACE;
  char* w = static_cast<char*>(ws);
  P.work = reinterpret_cast<unsigned*>(w + L.work);
  P.tick_a = reinterpret_cast<unsigned*>(w + L.tick_a);
  P.tick_b = reinterpret_cast<unsigned*>(w + L.tick_b);
  P.tick_bytes = L.cstat - L.work;
  P.cstat = reinterpret_cast<ChunkStat*>(w + L.cstat);
  P.rstat = reinterpret_cast<RowStat*>(w + L.rstat);
  P.req = reinterpret_cast<ReqState*>(w + L.req);
  P.wsum = reinterpret_cast<float*>(w + L.wsum);
  return SPEC_OK;
}

spec_status_t launch(spec_dtype_t dtype, int mode, Params& P, specv::LaunchPlan& L, cudaStream_t stream) {
  L.sm_count = sm_count();
  if (L.sm_count <= 0) return SPEC_ERR_CUDA;
  L.smem_stats = 2 * (size_t)P.buf_bytes;
  L.smem_resid = 2 * (size_t)P.buf_bytes;
  // the ticket counters start every call at zero, whatever the workspace held before
  cudaError_t e = cudaMemsetAsync(P.work, 0, P.tick_bytes, stream);
  if (e != cudaSuccess) return SPEC_ERR_CUDA;
  switch (dtype) {
    case SPEC_DTYPE_F32: e = specv::launch_verify<float>(mode, P, L, stream); break;
    case SPEC_DTYPE_BF16: e = specv::launch_verify<__nv_bfloat16>(mode, P, L, stream); break;
    default: e = specv::launch_verify<__half>(mode, P, L, stream); break;
  }
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// Shared body of spec_verify_chain / spec_verify_ngram.
spec_status_t verify_chain_common(bool ngram, const void* target, const void* draft, spec_dtype_t dtype, int B,
                                  int K, int V, float T, const int32_t* x, const float* r, const float* u,
                                  int32_t* num_accepted, int32_t* out_tokens, float* residual_mass,
                                  int32_t* err_flags, float* accept_prob, int32_t* cand_tokens, float* pos_mass,
                                  float* target_probs, float* draft_probs, void* ws, size_t ws_bytes,
                                  spec_stream_t stream) {
  if (!dtype_ok(dtype) || B < 0 || K < 0 || V < 1) return SPEC_ERR_INVALID_ARG;
  if (!(T >= 0.f) || isinf(T)) return SPEC_ERR_INVALID_ARG;
  if (K > SPEC_MAX_K) return SPEC_ERR_UNSUPPORTED;
  if (B == 0) return SPEC_OK;
  const bool greedy = (T == 0.f);
  const bool two_rows = !ngram && !greedy && K > 0;
  if (!target || !num_accepted || !out_tokens) return SPEC_ERR_INVALID_ARG;
  if (K > 0 && !x) return SPEC_ERR_INVALID_ARG;
  if (!greedy && ((K > 0 && !r) || !u)) return SPEC_ERR_INVALID_ARG;
  if (two_rows && !draft) return SPEC_ERR_INVALID_ARG;
  const int S = elem_size(dtype);
  if (!aligned_to(target, S) || (two_rows && !aligned_to(draft, S))) return SPEC_ERR_INVALID_ARG;
  const int rows = two_rows ? 2 * K + 1 : K + 1;
  if ((long long)B * rows > INT_MAX) return SPEC_ERR_UNSUPPORTED;

  Params P = {};
  const Chunking ck = plan_chunks(V, S);
  P.chunk = ck.chunk;
  P.nchunk = ck.nchunk;
  P.buf_bytes = ck.buf_bytes;
  const int diag = (cand_tokens || pos_mass) ? 1 : 0;
  if ((long long)B * rows * P.nchunk > INT_MAX || (long long)B * (diag ? K : 1) * P.nchunk > INT_MAX)
    return SPEC_ERR_UNSUPPORTED;
  spec_status_t st = attach_workspace(P, ws, ws_bytes, B, rows);
  if (st != SPEC_OK) return st;
  P.target = target;
  P.draft = two_rows ? draft : nullptr;
  P.B = B;
  P.K = K;
  P.V = V;
  P.R = K + 1;
  P.rows = rows;
  P.diag = diag;
  P.c = greedy ? 0.f : (float)(1.4426950408889634 / (double)T);  // log2(e) / T
  P.draft_tokens = x;
  P.r = r;
  P.u = u;
  P.num_accepted = num_accepted;
  P.out_tokens = out_tokens;
  P.residual_mass = residual_mass;
  P.err_flags = err_flags;
  P.accept_prob = accept_prob;
  P.cand_tokens = cand_tokens;
  P.pos_mass = pos_mass;
  P.target_probs = greedy ? nullptr : target_probs;
  P.draft_probs = two_rows ? draft_probs : nullptr;
  specv::LaunchPlan L = {};
  L.launch_resid = two_rows ? 1 : 0;
  L.launch_probs = (P.target_probs || P.draft_probs) ? 1 : 0;
  const int mode = greedy ? specv::kGreedy : (ngram ? specv::kNgram : specv::kChain);
  return launch(dtype, mode, P, L, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

size_t spec_verify_workspace_bytes(int B, int rows_per_request, int V, spec_dtype_t dtype) {
  if (B < 0 || rows_per_request < 1 || V < 1 || !dtype_ok(dtype)) return 0;
  const Chunking ck = plan_chunks(V, elem_size(dtype));
  return layout(B, rows_per_request, ck.nchunk).total;
}

spec_status_t spec_verify_chain(const void* target_logits, const void* draft_logits, spec_dtype_t dtype, int B,
                                int K, int V, float temperature, const int32_t* draft_tokens, const float* r,
                                const float* u, int32_t* num_accepted, int32_t* out_tokens, float* residual_mass,
                                int32_t* err_flags, float* accept_prob, int32_t* cand_tokens, float* pos_mass,
                                float* target_probs, float* draft_probs, void* workspace, size_t workspace_bytes,
                                spec_stream_t stream) {
  return verify_chain_common(false, target_logits, draft_logits, dtype, B, K, V, temperature, draft_tokens, r, u,
                             num_accepted, out_tokens, residual_mass, err_flags, accept_prob, cand_tokens, pos_mass,
                             target_probs, draft_probs, workspace, workspace_bytes, stream);
}

spec_status_t spec_verify_ngram(const void* target_logits, spec_dtype_t dtype, int B, int K, int V,
                                float temperature, const int32_t* draft_tokens, const float* r, const float* u,
                                int32_t* num_accepted, int32_t* out_tokens, float* residual_mass, int32_t* err_flags,
                                float* accept_prob, int32_t* cand_tokens, float* pos_mass, float* target_probs,
                                void* workspace, size_t workspace_bytes, spec_stream_t stream) {
  return verify_chain_common(true, target_logits, nullptr, dtype, B, K, V, temperature, draft_tokens, r, u,
                             num_accepted, out_tokens, residual_mass, err_flags, accept_prob, cand_tokens, pos_mass,
                             target_probs, nullptr, workspace, workspace_bytes, stream);
}

spec_status_t spec_verify_tree_greedy(const void* target_logits, spec_dtype_t dtype, int B, int N, int V,
                                      const int32_t* node_tokens, const int32_t* parents, int32_t* accept_len,
                                      int32_t* path_nodes, int32_t* out_tokens, int32_t* err_flags,
                                      int32_t* node_argmax, void* workspace, size_t workspace_bytes,
                                      spec_stream_t stream) {
  if (!dtype_ok(dtype) || B < 0 || N < 0 || V < 1) return SPEC_ERR_INVALID_ARG;
  if (N + 1 > SPEC_MAX_TREE_NODES) return SPEC_ERR_UNSUPPORTED;
  if (B == 0) return SPEC_OK;
  if (!target_logits || !node_tokens || !parents || !accept_len || !path_nodes || !out_tokens)
    return SPEC_ERR_INVALID_ARG;
  const int S = elem_size(dtype);
  if (!aligned_to(target_logits, S)) return SPEC_ERR_INVALID_ARG;
  const int rows = N + 1;
  Params P = {};
  const Chunking ck = plan_chunks(V, S);
  P.chunk = ck.chunk;
  P.nchunk = ck.nchunk;
  P.buf_bytes = ck.buf_bytes;
  if ((long long)B * rows * P.nchunk > INT_MAX) return SPEC_ERR_UNSUPPORTED;
  spec_status_t st = attach_workspace(P, workspace, workspace_bytes, B, rows);
  if (st != SPEC_OK) return st;
  P.target = target_logits;
  P.B = B;
  P.K = 0;
  P.V = V;
  P.R = rows;
  P.rows = rows;
  P.parents = parents;
  P.node_tokens = node_tokens;
  P.accept_len = accept_len;
  P.path_nodes = path_nodes;
  P.out_tokens = out_tokens;
  P.err_flags = err_flags;
  P.node_argmax = node_argmax;
  specv::LaunchPlan L = {};
  return launch(dtype, specv::kTree, P, L, reinterpret_cast<cudaStream_t>(stream));
}

const char* spec_status_string(spec_status_t s) {
  switch (s) {
    case SPEC_OK: return "SPEC_OK";
    case SPEC_ERR_INVALID_ARG: return "SPEC_ERR_INVALID_ARG";
    case SPEC_ERR_CUDA: return "SPEC_ERR_CUDA";
    case SPEC_ERR_WORKSPACE: return "SPEC_ERR_WORKSPACE";
    case SPEC_ERR_UNSUPPORTED: return "SPEC_ERR_UNSUPPORTED";
  }
  return "SPEC_ERR_UNKNOWN";
}

}  // extern "C"
