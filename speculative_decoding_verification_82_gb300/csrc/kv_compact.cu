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
// One CTA moves one request's rows in one cache (a layer's K or V tensor), each thread 16 bytes of
// every row.  Along an accepted path p_j >= j (a node's index exceeds its parent's), so no move
// writes a slot that a later move reads: a thread loads up to kBatch source vectors, then stores
// them, batch after batch in increasing position, in place.  Moves with p_j == j are skipped.
// The kernel is a gather bound by HBM bandwidth: each moved row is read once and written once.
// (Staging whole rows through shared memory with bulk copies, one to three CTAs per SM, measured
// 10 to 15% slower on the benchmark's 2048-byte rows: each CTA's reads and writes then serialise.)
#include <stdint.h>

#include "spec_verify.h"

namespace {

constexpr int kMaxCaches = SPEC_MAX_KV_CACHES;
constexpr int kMaxNodes = SPEC_MAX_WALK_NODES;
constexpr int kBatch = 8;

struct KvParams {
  unsigned char* caches[kMaxCaches];  // each [num_slots][row_bytes]
  int C, row_bytes, B, N1;
  long long num_slots;
  const int32_t* slots;       // [B][N1]
  const int32_t* parents;     // [B][N1]
  const int32_t* accept_len;  // [B]
  const int32_t* path;        // [B][N1]
  int32_t* err_flags;         // [B] or null
};

__global__ void __launch_bounds__(256) kv_compact_kernel(const KvParams P) {
  __shared__ int32_t src[kMaxNodes], dst[kMaxNodes];
  const int c = blockIdx.x, b = blockIdx.y, t = threadIdx.x;
  const int N1 = P.N1;
  const int32_t* sl = P.slots + (size_t)b * N1;
  const int32_t* pa = P.parents + (size_t)b * N1;
  const int32_t* pt = P.path + (size_t)b * N1;
  const int L = __ldg(P.accept_len + b);
  // the path must be an accepted path of the tree and every slot inside the cache
  bool ok = L >= 0 && L < N1 && __ldg(pt) == 0;
  if (ok) {
    for (int j = 1 + t; j <= L; j += blockDim.x) {
      const int n = __ldg(pt + j), prev = __ldg(pt + j - 1);
      ok = ok && n > 0 && n < N1 && __ldg(pa + n) == prev;
    }
    for (int n = t; n < N1; n += blockDim.x) {
      const int s = __ldg(sl + n);
      ok = ok && s >= 0 && s < P.num_slots;
    }
  }
  ok = __syncthreads_and(ok);
  if (c == 0 && t == 0 && P.err_flags) P.err_flags[b] = ok ? 0 : SPEC_ERRF_BAD_TREE;
  if (!ok) return;
  for (int j = 1 + t; j <= L; j += blockDim.x) {
    src[j] = __ldg(sl + __ldg(pt + j));
    dst[j] = __ldg(sl + j);
  }
  __syncthreads();
  unsigned char* base = P.caches[c];
  const size_t W = (size_t)P.row_bytes;
  const int nvec = P.row_bytes / 16;
  for (int v = t; v < nvec; v += blockDim.x) {
    for (int j0 = 1; j0 <= L; j0 += kBatch) {
      uint4 tmp[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int j = j0 + i;
        if (j <= L && src[j] != dst[j]) tmp[i] = *reinterpret_cast<const uint4*>(base + src[j] * W + v * 16);
      }
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int j = j0 + i;
        if (j <= L && src[j] != dst[j]) *reinterpret_cast<uint4*>(base + dst[j] * W + v * 16) = tmp[i];
      }
    }
  }
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
  const int nvec = row_bytes / 16;
  const int threads = nvec >= 256 ? 256 : (nvec >= 32 ? (nvec + 31) / 32 * 32 : 32);
  kv_compact_kernel<<<dim3((unsigned)num_caches, (unsigned)B), threads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(P);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
