// kv_compact.cu -- spec_kv_compact: accepted-path KV-cache compaction after tree verification
// (sm_103a).
//
// "Speculative Decoding with Medusa, EAGLE and vLLM" (vikram-blog.pages.dev), "System Topology &
// Data Flow" diagram: once the tree is verified, the accepted branch's tokens are committed to the
// KV cache.  The target's forward pass over the flattened tree wrote the KV row of node n into
// slot slots[b][n]; with the accepted path p_0 = 0, p_1, ..., p_L, the row of p_j moves to the
// slot of position j, slots[b][j], so the accepted tokens end up in order in the request's first
// L + 1 slots; every other slot is left alone.
//
// One CTA moves one request's rows in a group of consecutive caches (layers' K or V tensors).  It
// checks the path in two dependent rounds of loads: first the length, the path and every slot at
// once, which give the moves' sources and the move list; then the parent links of the path's
// nodes, loaded together with the first rows to move, so that the check costs no extra round trip
// (nothing is stored unless it holds).  The grid is sized to about kCtasPerSm CTAs per SM, so that
// every CTA is resident from the start and their checks overlap.  A unit of work is one 16-byte
// column of the moved rows of one cache: the thread loads the column of up to kBatch moved rows,
// then stores them, in increasing position.  Along an accepted path
// p_j >= j (a node's index exceeds its parent's) and slots are distinct, so no store lands on a
// row that a later move still reads, and moving in place is safe.  Moves with p_j == j are
// skipped.  The kernel is a gather bound by HBM bandwidth: each moved row is read once and written
// once.  Both go through the streaming cache policy (evict first): the call touches each moved
// byte once, and its dirty rows leave L2 ahead of data that is still in use.
//
// The kernel is launched with programmatic stream serialisation: its CTAs may be placed on the
// SMs while the previous kernel in the stream drains, and each one waits for that kernel's
// completion (griddepcontrol.wait) before its first memory access, so stream order holds for
// every byte it reads or writes.  Each CTA at once lets the next such launch do the same.
#include <stdint.h>

#include "spec_verify.h"

namespace {

constexpr int kMaxCaches = SPEC_MAX_KV_CACHES;
constexpr int kMaxNodes = SPEC_MAX_WALK_NODES;
constexpr int kThreads = 256;
constexpr int kBatch = 5;      // moved rows of one column loaded before they are stored
constexpr int kCtasPerSm = 6;  // grid target: every CTA resident at once

struct KvParams {
  unsigned char* caches[kMaxCaches];  // each [num_slots][row_bytes]
  int C, row_bytes, B, N1;
  int group;                  // caches per CTA
  long long num_slots;
  const int32_t* slots;       // [B][N1]
  const int32_t* parents;     // [B][N1]
  const int32_t* accept_len;  // [B]
  const int32_t* path;        // [B][N1]
  int32_t* err_flags;         // [B] or null
};

__global__ void __launch_bounds__(kThreads, kCtasPerSm) kv_compact_kernel(const KvParams P) {
  __shared__ int32_t node[kMaxNodes];                 // path[j]
  __shared__ int32_t slot[kMaxNodes];                 // slots[n]
  __shared__ int32_t from[kMaxNodes];                 // slots[path[j]]: the source of position j
  __shared__ int32_t src[kMaxNodes], dst[kMaxNodes];  // the move list, in increasing position
  __shared__ int nmove;
  const int grp = blockIdx.x, b = blockIdx.y, t = threadIdx.x;
  const int N1 = P.N1;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (t == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int32_t* pa = P.parents + (size_t)b * N1;
  // first pass: the length, the path and every slot, all at once
  const int L = __ldg(P.accept_len + b);
  bool ok = true;
  for (int j = t; j < N1; j += kThreads) {
    node[j] = __ldg(P.path + (size_t)b * N1 + j);
    const int s = __ldg(P.slots + (size_t)b * N1 + j);
    slot[j] = s;
    ok = ok && s >= 0 && s < P.num_slots;
  }
  __syncthreads();
  ok = ok && L >= 0 && L < N1 && node[0] == 0;
  // the sources (every accepted node must be a valid index; its parent link is checked below)
  for (int j = 1 + t; j <= L && j < N1; j += kThreads) {
    const int n = node[j];
    const bool in = n > 0 && n < N1;
    ok = ok && in;
    from[j] = in ? slot[n] : -1;
  }
  ok = __syncthreads_and(ok);
  if (!ok) {
    if (grp == 0 && t == 0 && P.err_flags) P.err_flags[b] = SPEC_ERRF_BAD_TREE;
    return;
  }
  // the move list in increasing position (a warp ballot keeps the order); moves in place skipped
  if (t < 32) {
    int base = 0;
    for (int j0 = 1; j0 <= L; j0 += 32) {
      const int j = j0 + t;
      const bool mv = j <= L && from[j] != slot[j];
      const unsigned bal = __ballot_sync(0xffffffffu, mv);
      if (mv) {
        const int k = base + __popc(bal & ((1u << t) - 1u));
        src[k] = from[j];
        dst[k] = slot[j];
      }
      base += __popc(bal);
    }
    if (t == 0) nmove = base;
  }
  __syncthreads();
  const int M = nmove;
  const int c0 = grp * P.group, c1 = min(P.C, c0 + P.group);
  const size_t W = (size_t)P.row_bytes;
  const int nvec = P.row_bytes / 16;
  const int units = (c1 - c0) * nvec;  // (cache, 16-byte column) pairs of this CTA
  // the first unit's first batch loads while the parent links are checked
  uint4 tmp[kBatch];
  if (t < units) {
    const int cl = t / nvec, v = t - cl * nvec;
    const unsigned char* base = P.caches[c0 + cl] + (size_t)v * 16;
#pragma unroll
    for (int k = 0; k < kBatch; ++k)
      if (k < M) tmp[k] = __ldcs(reinterpret_cast<const uint4*>(base + (size_t)src[k] * W));
  }
  for (int j = 1 + t; j <= L; j += kThreads) ok = ok && __ldg(pa + node[j]) == node[j - 1];
  ok = __syncthreads_and(ok);
  if (grp == 0 && t == 0 && P.err_flags) P.err_flags[b] = ok ? 0 : SPEC_ERRF_BAD_TREE;
  if (!ok || M == 0) return;
  for (int i = t; i < units; i += kThreads) {
    const int cl = i / nvec, v = i - cl * nvec;
    unsigned char* base = P.caches[c0 + cl] + (size_t)v * 16;
    for (int k0 = 0; k0 < M; k0 += kBatch) {
      if (i != t || k0 != 0) {
#pragma unroll
        for (int k = 0; k < kBatch; ++k)
          if (k0 + k < M) tmp[k] = __ldcs(reinterpret_cast<const uint4*>(base + (size_t)src[k0 + k] * W));
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        if (k0 + k < M) __stcs(reinterpret_cast<uint4*>(base + (size_t)dst[k0 + k] * W), tmp[k]);
    }
  }
}

int sm_count_cached() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
  static int cache[64] = {0};
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (dev < 64) cache[dev] = n;
  return n;
}

}  // namespace

extern "C" spec_status_t spec_kv_compact(void* const* caches, int num_caches, long long num_slots, int row_bytes,
                                         int B, int N, const int32_t* slots, const int32_t* parents,
                                         const int32_t* accept_len, const int32_t* path_nodes, int32_t* err_flags,
                                         spec_stream_t stream) {
  if (num_caches < 0 || num_slots < 0 || row_bytes < 0 || B < 0 || N < 0) return SPEC_ERR_INVALID_ARG;
  if (row_bytes % 16 != 0) return SPEC_ERR_INVALID_ARG;
  if (num_caches > kMaxCaches || N + 1 > kMaxNodes || B > 65535) return SPEC_ERR_UNSUPPORTED;
  if (B == 0 || num_caches == 0) return SPEC_OK;
  if (!caches || !slots || !parents || !accept_len || !path_nodes) return SPEC_ERR_INVALID_ARG;
  KvParams P = {};
  for (int i = 0; i < num_caches; ++i) {
    if (!caches[i] || ((uintptr_t)caches[i] & 15u)) return SPEC_ERR_INVALID_ARG;
    P.caches[i] = static_cast<unsigned char*>(caches[i]);
  }
  const int sms = sm_count_cached();
  if (sms <= 0) return SPEC_ERR_CUDA;
  // caches per CTA: about kCtasPerSm CTAs per SM over the (request, cache group) grid
  const long long target = (long long)kCtasPerSm * sms;
  long long groups = target / B;
  if (groups < 1) groups = 1;
  if (groups > num_caches) groups = num_caches;
  P.group = (int)((num_caches + groups - 1) / groups);
  const int ngroups = (num_caches + P.group - 1) / P.group;
  P.C = num_caches;
  P.row_bytes = row_bytes;
  P.B = B;
  P.N1 = N + 1;
  P.num_slots = num_slots;
  P.slots = slots;
  P.parents = parents;
  P.accept_len = accept_len;
  P.path = path_nodes;
  P.err_flags = err_flags;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ngroups, (unsigned)B);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kv_compact_kernel, P) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
