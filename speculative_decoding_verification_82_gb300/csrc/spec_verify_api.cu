// spec_verify_api.cu -- the C ABI: argument checks, chunk planning, workspace layout, launch.
//
// Host side only; the kernels live in verify_kernel.cuh (instantiated per element type in
// spec_verify_{f32,bf16,f16}.cu).  No call allocates memory or synchronises the host.
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <climits>
#include <cstring>
#include <mutex>

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

int elem_size(spec_dtype_t dt) { return dt == SPEC_DTYPE_F32 ? 4 : 2; }
bool dtype_ok(int dt) { return dt == SPEC_DTYPE_F32 || dt == SPEC_DTYPE_BF16 || dt == SPEC_DTYPE_F16; }
size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// A row of V elements spans at most ceil((V + VE - 1) / VE) 16-byte vectors (VE elements per
// vector; the row may start anywhere inside its first vector).  Stats chunks take kChunkVec of
// them, residual items kResVec.
struct Chunking {
  int nchunk, nchunk_r;
};
Chunking plan_chunks(int V, int S) {
  const long long VE = 16 / S;
  const long long nvec = ((long long)V + VE - 1 + VE - 1) / VE;
  Chunking c;
  c.nchunk = (int)((nvec + specv::kChunkVec - 1) / specv::kChunkVec);
  c.nchunk_r = (int)((nvec + specv::kResVec - 1) / specv::kResVec);
  return c;
}

// Workspace layout:
//   work, gerr, exit_tick, epoch, rq_tail u32 (128 B line) } counters: zero between calls of one
//   rc                           u32 (128 B line)   } shape (each call leaves them zero; the
//   tick_a  [B][rows] u32        chunk counts       } first call of a shape clears them)
//   tick_b  [B][rows] u32        residual counts    }
//   req     [B]                  ReqState           (16-byte aligned; tagged per call)
//   rq      [B][5] u64           residual queue     (result words and request index, tagged per call)
//   cstat   [B][rows][nchunk]    ChunkStat          (256-byte aligned regions from here on)
//   sstat   [B][rows][nchunk][G] ChunkStat          sub-chunk partials (G consumer warps a group)
//   rstat   [B][rows]            RowStat
//   wsub    [B][rows][nchunk_r][G] TagSum (float and tag): residual sums per sub-range
struct Layout {
  size_t work, tick_a, tick_b, req, rq, hdr_end, cstat, sstat, rstat, wsub, total;
};

Layout layout(int B, int rows, const Chunking& ck) {
  Layout L;
  const size_t b = (size_t)B, r = (size_t)rows;
  size_t off = 0;
  L.work = off;
  off += 2 * 128;
  L.tick_a = off;
  off += b * r * 4;
  L.tick_b = off;
  off = align_up(off + b * r * 4, 16);
  L.req = off;
  off += b * sizeof(ReqState);
  L.rq = off;
  off += b * 8 * (size_t)specv::kQWords;
  L.hdr_end = off;
  off = align_up(off, 256);
  const size_t G = specv::kGroupWarps;
  L.cstat = off;
  off = align_up(off + b * r * (size_t)ck.nchunk * sizeof(ChunkStat), 256);
  L.sstat = off;
  off = align_up(off + b * r * (size_t)ck.nchunk * G * sizeof(ChunkStat), 256);
  L.rstat = off;
  off = align_up(off + b * r * sizeof(RowStat), 256);
  L.wsub = off;
  off = align_up(off + b * r * (size_t)ck.nchunk_r * G * sizeof(specv::TagSum), 256);
  L.total = off;
  return L;
}

// Multiprocessors of the current device (cached per device); *device receives the device.
int sm_count(int* device) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
  *device = dev;
  static int cache[64] = {0};
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (dev < 64) cache[dev] = n;
  return n;
}

bool aligned_to(const void* p, int a) { return ((uintptr_t)p % (uintptr_t)a) == 0; }

spec_status_t attach_workspace(Params& P, void* ws, size_t bytes, int B, int rows, const Chunking& ck) {
  const Layout L = layout(B, rows, ck);
  if (ws == nullptr || bytes < L.total) return SPEC_ERR_WORKSPACE;
  if (((uintptr_t)ws & 255u) != 0) return SPEC_ERR_WORKSPACE;
  char* w = static_cast<char*>(ws);
  P.work = reinterpret_cast<unsigned*>(w + L.work);
  P.gerr = P.work + 1;
  P.exit_tick = P.work + 2;
  P.epoch = P.work + 3;
  P.rq_tail = P.work + 4;
  P.rc = reinterpret_cast<unsigned*>(w + L.work + 128);  // residual cursor (a line of its own)
  P.tick_a = reinterpret_cast<unsigned*>(w + L.tick_a);
  P.tick_b = reinterpret_cast<unsigned*>(w + L.tick_b);
  P.req = reinterpret_cast<ReqState*>(w + L.req);
  P.rq = reinterpret_cast<unsigned long long*>(w + L.rq);
  P.cstat = reinterpret_cast<ChunkStat*>(w + L.cstat);
  P.sstat = reinterpret_cast<ChunkStat*>(w + L.sstat);
  P.rstat = reinterpret_cast<RowStat*>(w + L.rstat);
  P.wsub = reinterpret_cast<specv::TagSum*>(w + L.wsub);
  P.ws_base = ws;
  P.ws_bytes = L.total;
  P.ws_shape[0] = B;
  P.ws_shape[1] = rows;
  P.ws_shape[2] = ck.nchunk;
  P.ws_shape[3] = ck.nchunk_r;
  return SPEC_OK;
}

// A workspace's counters are zero between calls (each call leaves them so) and its epoch names the
// last call's tag, but only for calls of one layout: a call of another shape may keep counters
// where the last one left other data, and the statistics there may carry any tag.  So the whole
// workspace (of this call's layout) is cleared on the first call of a shape on it (a workspace not
// seen before included): counters and epoch zero, every tag zero, which no call's tag matches.
// While the shape stays it is not cleared again.  The shapes of the last kWsSeen workspaces are
// kept; one that falls out of the table is simply cleared again.
constexpr int kWsSeen = 64;
struct WsSeen {
  const void* ws;
  int shape[4];
};
std::mutex g_ws_mu;
WsSeen g_ws_seen[kWsSeen];
int g_ws_next = 0;
// True when the call must clear the header first; `forget` drops the entry (a failed launch).
bool workspace_needs_clear(const Params& P, bool forget) {
  std::lock_guard<std::mutex> g(g_ws_mu);
  for (int i = 0; i < kWsSeen; ++i) {
    WsSeen& e = g_ws_seen[i];
    if (e.ws != P.ws_base) continue;
    if (forget) {
      e.ws = nullptr;
      return false;
    }
    if (std::memcmp(e.shape, P.ws_shape, sizeof(e.shape)) == 0) return false;
    std::memcpy(e.shape, P.ws_shape, sizeof(e.shape));
    return true;
  }
  if (forget) return false;
  WsSeen& e = g_ws_seen[g_ws_next];
  g_ws_next = (g_ws_next + 1) % kWsSeen;
  e.ws = P.ws_base;
  std::memcpy(e.shape, P.ws_shape, sizeof(e.shape));
  return true;
}

// Constants of the item decoding's divisions (see fastdiv.h).  pair_rows: the rows a request reads
// per position in the chain modes (2 with draft logits, else 1).
void set_divisors(Params& P, int B, int rows, int pair_rows) {
  const unsigned A = (unsigned)rows * (unsigned)P.nchunk;
  const unsigned R = (unsigned)P.npos * (unsigned)P.nchunk_r;
  const unsigned pair = (unsigned)pair_rows * (unsigned)P.nchunk;
  P.fd_A = specv::make_fastdiv(A);
  P.fd_R = specv::make_fastdiv(R > 0 ? R : 1u);
  P.fd_nchunk = specv::make_fastdiv((unsigned)P.nchunk);
  P.fd_nchunk_r = specv::make_fastdiv((unsigned)P.nchunk_r);
  P.fd_pair = specv::make_fastdiv(pair);
  P.fd_S1 = specv::make_fastdiv((unsigned)B * pair);
}

spec_status_t launch(spec_dtype_t dtype, int mode, Params& P, specv::LaunchPlan& L, cudaStream_t stream) {
  if (workspace_needs_clear(P, false) && cudaMemsetAsync(P.ws_base, 0, P.ws_bytes, stream) != cudaSuccess) {
    workspace_needs_clear(P, true);
    return SPEC_ERR_CUDA;
  }
  L.smem = (size_t)specv::kStages * specv::kStageBytes + specv::kFinBytes;
  cudaError_t e = cudaSuccess;
  switch (dtype) {
    case SPEC_DTYPE_F32: e = specv::launch_verify<float>(mode, P, L, stream); break;
    case SPEC_DTYPE_BF16: e = specv::launch_verify<__nv_bfloat16>(mode, P, L, stream); break;
    default: e = specv::launch_verify<__half>(mode, P, L, stream); break;
  }
  if (e != cudaSuccess) {
    workspace_needs_clear(P, true);  // the next call clears again
    return SPEC_ERR_CUDA;
  }
  return SPEC_OK;
}

// Shared body of spec_verify_chain / spec_verify_ngram.
spec_status_t verify_chain_common(bool ngram, const void* target, const void* draft, spec_dtype_t dtype, int B,
                                  int K, int V, float T, const float* temps, const int32_t* x, const float* r,
                                  const float* u,
                                  int32_t* num_accepted, int32_t* out_tokens, float* residual_mass,
                                  int32_t* err_flags, float* accept_prob, int32_t* cand_tokens, float* pos_mass,
                                  float* target_probs, float* draft_probs, void* ws, size_t ws_bytes,
                                  spec_stream_t stream) {
  if (!dtype_ok(dtype) || B < 0 || K < 0 || V < 1) return SPEC_ERR_INVALID_ARG;
  if (!(T >= 0.f) || isinf(T)) return SPEC_ERR_INVALID_ARG;
  if (K > SPEC_MAX_K) return SPEC_ERR_UNSUPPORTED;
  if (B == 0) return SPEC_OK;
  // with per-request temperatures any request may sample: draft logits (chain), r and u are needed
  const bool greedy = (T == 0.f) && !temps;
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
  P.nchunk = ck.nchunk;
  P.nchunk_r = ck.nchunk_r;
  const int diag = (cand_tokens || pos_mass) ? 1 : 0;
  P.npos = two_rows ? (diag ? K : 1) : 0;
  const long long per_req = (long long)rows * ck.nchunk + (long long)P.npos * ck.nchunk_r;
  if ((long long)B * per_req > INT_MAX) return SPEC_ERR_UNSUPPORTED;
  spec_status_t st = attach_workspace(P, ws, ws_bytes, B, rows, ck);
  if (st != SPEC_OK) return st;
  int device = -1;
  const int sms = sm_count(&device);
  if (sms <= 0) return SPEC_ERR_CUDA;
  P.total = (unsigned)((long long)B * rows * ck.nchunk);
  P.total_r = (unsigned)((long long)B * P.npos * ck.nchunk_r);
  set_divisors(P, B, rows, two_rows ? 2 : 1);
  P.target = target;
  P.draft = two_rows ? draft : nullptr;
  P.B = B;
  P.K = K;
  P.V = V;
  P.R = K + 1;
  P.rows = rows;
  P.diag = diag;
  // the bonus rows stream first when the call runs residual passes (the stream then ends on the
  // last position, which few requests reach); measured slower for calls without residual passes
  P.bonus_first = P.npos > 0 ? 1 : 0;
  // Calls with residual passes: larger stats batches, so that a producer looks for residual items
  // less often and the stats stream, which every later position waits for, runs ahead; and near
  // the end of the stats stream the stats items go first (measured: 72.3 against 77.6 us with
  // per-request temperatures, no change at one temperature).  The n-gram chain streams best in
  // batches of 2 (the headline n-gram workload: 80.7 against 81.3 us with 4).
  P.claim = P.npos > 0 ? 6 : (ngram ? 2 : specv::kClaim);
  P.tail_first = P.npos > 0 ? 1 : 0;
  P.c = (greedy || temps) ? 0.f : (float)(1.4426950408889634 / (double)T);  // log2(e) / T
  P.temps = temps;
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
  L.sm_count = sms;
  L.device = device;
  L.launch_probs = (P.target_probs || P.draft_probs) ? 1 : 0;
  const int mode = temps ? (int)(ngram ? specv::kNgramPT : specv::kChainPT)
                         : (int)(greedy ? specv::kGreedy : (ngram ? specv::kNgram : specv::kChain));
  return launch(dtype, mode, P, L, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

size_t spec_verify_workspace_bytes(int B, int rows_per_request, int V, spec_dtype_t dtype) {
  if (B < 0 || rows_per_request < 1 || V < 1 || !dtype_ok(dtype)) return 0;
  const Chunking ck = plan_chunks(V, elem_size(dtype));
  return layout(B, rows_per_request, ck).total;
}

void spec_verify_workspace_reset(const void* workspace) {
  Params P = {};
  P.ws_base = const_cast<void*>(workspace);
  workspace_needs_clear(P, true);
}

spec_status_t spec_verify_chain(const void* target_logits, const void* draft_logits, spec_dtype_t dtype, int B,
                                int K, int V, float temperature, const float* temperatures,
                                const int32_t* draft_tokens, const float* r, const float* u, int32_t* num_accepted,
                                int32_t* out_tokens, float* residual_mass, int32_t* err_flags, float* accept_prob,
                                int32_t* cand_tokens, float* pos_mass, float* target_probs, float* draft_probs,
                                void* workspace, size_t workspace_bytes, spec_stream_t stream) {
  return verify_chain_common(false, target_logits, draft_logits, dtype, B, K, V, temperature, temperatures,
                             draft_tokens, r, u,
                             num_accepted, out_tokens, residual_mass, err_flags, accept_prob, cand_tokens, pos_mass,
                             target_probs, draft_probs, workspace, workspace_bytes, stream);
}

spec_status_t spec_verify_ngram(const void* target_logits, spec_dtype_t dtype, int B, int K, int V,
                                float temperature, const float* temperatures, const int32_t* draft_tokens,
                                const float* r, const float* u, int32_t* num_accepted, int32_t* out_tokens,
                                float* residual_mass, int32_t* err_flags, float* accept_prob, int32_t* cand_tokens,
                                float* pos_mass, float* target_probs, void* workspace, size_t workspace_bytes,
                                spec_stream_t stream) {
  return verify_chain_common(true, target_logits, nullptr, dtype, B, K, V, temperature, temperatures,
                             draft_tokens, r, u,
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
  P.nchunk = ck.nchunk;
  P.nchunk_r = ck.nchunk_r;
  if ((long long)B * rows * P.nchunk > INT_MAX) return SPEC_ERR_UNSUPPORTED;
  spec_status_t st = attach_workspace(P, workspace, workspace_bytes, B, rows, ck);
  if (st != SPEC_OK) return st;
  int device = -1;
  const int sms = sm_count(&device);
  if (sms <= 0) return SPEC_ERR_CUDA;
  P.total = (unsigned)((long long)B * rows * P.nchunk);
  P.npos = 0;
  P.claim = 2;  // (measured: 42.9 us against 43.7 with 4 on the 61-node greedy tree workload)
  set_divisors(P, B, rows, 1);
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
  L.sm_count = sms;
  L.device = device;
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
