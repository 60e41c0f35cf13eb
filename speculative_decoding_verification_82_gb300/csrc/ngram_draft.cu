// ngram_draft.cu -- spec_ngram_draft: prompt n-gram lookup drafting on the GPU (sm_103a).
//
// The draft mechanism of "Accelerating Autoregressive LLM Inference 3x with Lossless
// Speculative Decoding and EAGLE Heads" (x078.com), opening section: a zero-VRAM prompt n-gram
// lookup proposes K candidate tokens (its serving example: --num-speculative-tokens 5
// --ngram-prompt-lookup-max 4).  For n = n_max down to n_min, the context's last n tokens are
// looked up; their most recent earlier occurrence wins, and the draft is the up to K tokens after
// it.
//
// Equivalently, every end position e in [1, L) of the context has a match length m(e): the
// number of tokens before e that equal the context's last tokens, read backwards, capped at
// n_max.  The draft follows the e that maximises (m(e), e) among those with m(e) >= n_min.  One
// CTA takes a context: each thread scores end positions strided by the block size (reads of
// neighbouring positions coalesce), and a 64-bit (m << 32 | e) maximum over the block picks
// the winner.  The context is read once; the work is a few integer compares per token.
#include <stdint.h>

#include "spec_verify.h"
#include "verify_common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kBatch = 8;  // end positions per thread whose first loads are issued together

struct DraftParams {
  const int32_t* ctx;      // [B][Lmax]
  const int32_t* ctx_len;  // [B]
  int B, Lmax, n_max, n_min, K;
  int32_t* draft;          // [B][K]
  int32_t* draft_len;      // [B]
  int32_t* match_n;        // [B] or null
  int32_t* match_end;      // [B] or null
  int32_t* err_flags;      // [B] or null
};

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

__global__ void __launch_bounds__(kThreads) ngram_draft_kernel(const DraftParams P) {
  __shared__ unsigned long long wbest[kThreads / 32];
  __shared__ int32_t suffix[SPEC_MAX_NGRAM];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  for (int b = blockIdx.x; b < P.B; b += gridDim.x) {
    const int32_t* c = P.ctx + (size_t)b * P.Lmax;
    int L = __ldg(P.ctx_len + b);
    const bool bad = L < 0 || L > P.Lmax;
    if (bad) L = 0;
    __syncthreads();  // the previous context's readers of suffix / wbest are done
    if (t < P.n_max) suffix[t] = t < L ? __ldg(c + L - 1 - t) : 0;
    __syncthreads();
    unsigned long long best = 0;
    // kBatch end positions per thread at a time: their first compares load together (one memory
    // round trip per batch); the rare partial matches continue one token at a time
    for (int e0 = t + 1; e0 < L; e0 += kThreads * kBatch) {
      int32_t last[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int e = e0 + i * kThreads;
        last[i] = e < L ? __ldg(c + e - 1) : 0;
      }
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int e = e0 + i * kThreads;
        if (e >= L || last[i] != suffix[0]) continue;
        int m = 1;
        while (m < P.n_max && m < e && __ldg(c + e - 1 - m) == suffix[m]) ++m;
        if (m >= P.n_min) {
          const unsigned long long key = ((unsigned long long)m << 32) | (unsigned)e;
          best = key > best ? key : best;
        }
      }
    }
    best = warp_max_u64(best);
    if (lane == 0) wbest[warp] = best;
    __syncthreads();
    if (warp == 0) {
      best = warp_max_u64(lane < kThreads / 32 ? wbest[lane] : 0ull);
      const int e = best ? (int)(best & 0xffffffffu) : -1;
      const int n = (int)(best >> 32);
      for (int k = lane; k < P.K; k += 32)
        P.draft[(size_t)b * P.K + k] = (e >= 0 && e + k < L) ? __ldg(c + e + k) : -1;
      if (lane == 0) {
        P.draft_len[b] = e >= 0 ? min(P.K, L - e) : 0;
        if (P.match_n) P.match_n[b] = n;
        if (P.match_end) P.match_end[b] = e;
        if (P.err_flags) P.err_flags[b] = bad ? SPEC_ERRF_BAD_TOKEN : 0;
      }
    }
  }
}

}  // namespace

extern "C" spec_status_t spec_ngram_draft(const int32_t* context, const int32_t* context_len, int B, int Lmax,
                                          int n_max, int n_min, int K, int32_t* draft_tokens, int32_t* draft_len,
                                          int32_t* match_n, int32_t* match_end, int32_t* err_flags,
                                          spec_stream_t stream) {
  if (B < 0 || Lmax < 0 || K < 1 || n_min < 1 || n_max < n_min) return SPEC_ERR_INVALID_ARG;
  if (K > SPEC_MAX_K || n_max > SPEC_MAX_NGRAM) return SPEC_ERR_UNSUPPORTED;
  if (B == 0) return SPEC_OK;
  if ((Lmax > 0 && !context) || !context_len || !draft_tokens || !draft_len) return SPEC_ERR_INVALID_ARG;
  DraftParams P;
  P.ctx = context;
  P.ctx_len = context_len;
  P.B = B;
  P.Lmax = Lmax;
  P.n_max = n_max;
  P.n_min = n_min;
  P.K = K;
  P.draft = draft_tokens;
  P.draft_len = draft_len;
  P.match_n = match_n;
  P.match_end = match_end;
  P.err_flags = err_flags;
  const int grid = B < 65536 ? B : 65536;
  ngram_draft_kernel<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(P);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
