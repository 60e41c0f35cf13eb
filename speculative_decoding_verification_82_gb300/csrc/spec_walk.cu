// spec_walk.cu -- spec_verify_tree_walk: argument checks, cluster geometry, launch.
//
// Host side of the tree walk (tree_walk.cuh).  A request goes to one thread-block cluster of
// `cl` CTAs of 512 threads; each thread holds E consecutive tokens of the visited rows (in
// registers; q in shared memory for the 6-CTA geometry of the stochastic walk), so a cluster
// covers V <= cl * 512 * E.
// The grid is as many clusters as fit on the device at once (at most B), each taking requests
// b, b + grid, ...
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "spec_verify.h"
#include "tree_walk.cuh"

namespace {

using specv::walk::Params;

constexpr int kSmallE = 8;   // V <= 4096: one CTA
constexpr int kLargeE = 32;  // otherwise clusters of 1..16 CTAs
constexpr int kShE = 48;     // clusters of kShCl CTAs: p in registers and q in shared memory (96 KB
constexpr int kShCl = 6;     // a CTA), or for greedy calls p alone

struct Geometry {
  int E, cl;
};
// The smallest cluster that covers V (larger vocabularies first grow the cluster, which
// shortens every pass; 16 CTAs is the largest cluster the hardware schedules).
bool plan(int V, Geometry* g) {
  if (V <= specv::walk::kThreads * kSmallE) {
    g->E = kSmallE;
    g->cl = 1;
    return true;
  }
  const long long per_cta = (long long)specv::walk::kThreads * kLargeE;
  for (int cl = 1; cl <= specv::walk::kMaxCluster; cl *= 2) {
    if ((long long)cl * per_cta >= V) {
      g->E = kLargeE;
      g->cl = cl;
      return true;
    }
  }
  return false;
}

// Clusters of `cl` CTAs of instantiation (T, E, SM) resident at once, with `dyn` bytes of dynamic
// shared memory a CTA; found once per device, instantiation and cluster size.
template <typename T, int E, bool SM, bool G = false>
int clusters_that_fit(int cl, size_t dyn) {
  auto kern = specv::walk::walk_kernel<T, E, SM, G>;
  static std::mutex mu;
  static int cache[64][specv::walk::kMaxCluster + 1] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  {
    std::lock_guard<std::mutex> g(mu);
    if (cache[dev][cl] > 0) return cache[dev][cl];
  }
  if (cl > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return -1;
  if (dyn > 0 && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn) != cudaSuccess)
    return -1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)cl);
  cfg.blockDim = dim3(specv::walk::kThreads);
  cfg.dynamicSmemBytes = dyn;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int fit = 0;
  if (cudaOccupancyMaxActiveClusters(&fit, kern, &cfg) != cudaSuccess || fit <= 0) return -1;
  std::lock_guard<std::mutex> g(mu);
  cache[dev][cl] = fit;
  return fit;
}

template <typename T, int E, bool SM, bool G = false>
cudaError_t launch_one(const Params& P, cudaStream_t stream) {
  const size_t dyn = SM ? (size_t)E * specv::walk::kThreads * sizeof(float) : 0;
  const int fit = clusters_that_fit<T, E, SM, G>(P.cl, dyn);
  if (fit <= 0) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)P.cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  const int clusters = P.B < fit ? P.B : fit;
  cfg.gridDim = dim3((unsigned)(clusters * P.cl));
  cfg.blockDim = dim3(specv::walk::kThreads);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, specv::walk::walk_kernel<T, E, SM, G>, P);
}

// The geometry of the call: the smallest cluster with p and q in registers, unless clusters of
// kShCl CTAs cover V and take the batch in fewer waves (their threads hold 1.5 times the tokens,
// but more of them fit at once: 23 against 15 of 8 CTAs on a 152-SM GB300).  A greedy call then
// runs an instantiation without q, whose 48 tokens a thread stay in registers; a walk that samples
// at one temperature keeps p in registers and q in shared memory.  Measured on 16 requests of 61
// nodes at V = 128256: greedy 8.66 against 10.33 us, T = 1 41.9 against 51.6 us; with per-request
// temperatures 43.3 against 39.2 us, whose requests' times differ more, so those keep the
// register geometry.
template <typename T>
cudaError_t launch_typed(const Geometry& g, Params& P, cudaStream_t stream) {
  if (g.E == kSmallE) {
    P.cl = g.cl;
    return launch_one<T, kSmallE, false>(P, stream);
  }
  if (P.c == 0.f && !P.temps && g.cl > kShCl && (long long)kShCl * specv::walk::kThreads * kShE >= P.V) {
    const int f1 = clusters_that_fit<T, kLargeE, false>(g.cl, 0);
    const int f2 = clusters_that_fit<T, kShE, false, true>(kShCl, 0);
    if (f1 > 0 && f2 > 0 && (P.B + f2 - 1) / f2 < (P.B + f1 - 1) / f1) {
      P.cl = kShCl;
      return launch_one<T, kShE, false, true>(P, stream);
    }
  }
  if (P.c > 0.f && !P.temps && g.cl > kShCl && (long long)kShCl * specv::walk::kThreads * kShE >= P.V) {
    const int f1 = clusters_that_fit<T, kLargeE, false>(g.cl, 0);
    const int f2 = clusters_that_fit<T, kShE, true>(kShCl, (size_t)kShE * specv::walk::kThreads * sizeof(float));
    if (f1 > 0 && f2 > 0 && (P.B + f2 - 1) / f2 < (P.B + f1 - 1) / f1) {
      P.cl = kShCl;
      return launch_one<T, kShE, true>(P, stream);
    }
  }
  P.cl = g.cl;
  return launch_one<T, kLargeE, false>(P, stream);
}

bool aligned(const void* p, unsigned a) { return ((uintptr_t)p % a) == 0; }

}  // namespace

extern "C" spec_status_t spec_verify_tree_walk(const void* target_logits, const void* draft_logits,
                                               spec_dtype_t dtype, int B, int N, int V, float temperature,
                                               const float* temperatures, const int32_t* node_tokens, const int32_t* parents, const float* r,
                                               const float* u, int32_t* accept_len, int32_t* path_nodes,
                                               int32_t* out_tokens, float* residual_mass, int32_t* err_flags,
                                               float* accept_prob, spec_stream_t stream) {
  if (!(dtype == SPEC_DTYPE_F32 || dtype == SPEC_DTYPE_BF16 || dtype == SPEC_DTYPE_F16)) return SPEC_ERR_INVALID_ARG;
  if (B < 0 || N < 0 || V < 1) return SPEC_ERR_INVALID_ARG;
  if (!(temperature >= 0.f) || isinf(temperature)) return SPEC_ERR_INVALID_ARG;
  if (N + 1 > SPEC_MAX_WALK_NODES) return SPEC_ERR_UNSUPPORTED;
  Geometry g;
  if (!plan(V, &g)) return SPEC_ERR_UNSUPPORTED;
  if (B == 0) return SPEC_OK;
  // with per-request temperatures any request may sample: draft logits, r and u are needed
  const bool greedy = temperature == 0.f && !temperatures;
  if (!target_logits || !node_tokens || !parents || !accept_len || !path_nodes || !out_tokens)
    return SPEC_ERR_INVALID_ARG;
  if (!greedy && (!draft_logits || !r || !u)) return SPEC_ERR_INVALID_ARG;
  const unsigned S = dtype == SPEC_DTYPE_F32 ? 4u : 2u;
  if (!aligned(target_logits, S) || (!greedy && !aligned(draft_logits, S))) return SPEC_ERR_INVALID_ARG;
  Params P = {};
  P.target = target_logits;
  P.draft = greedy ? nullptr : draft_logits;
  P.B = B;
  P.N1 = N + 1;
  P.V = V;
  P.c = greedy ? 0.f : (float)(1.4426950408889634 / (double)temperature);  // log2(e) / T
  P.vec = ((size_t)V * S) % 16 == 0 && aligned(target_logits, 16) && (greedy || aligned(draft_logits, 16));
  P.cl = g.cl;
  P.node_tokens = node_tokens;
  P.parents = parents;
  P.r = r;
  P.u = u;
  P.temps = temperatures;
  P.accept_len = accept_len;
  P.path_nodes = path_nodes;
  P.out_tokens = out_tokens;
  P.residual_mass = residual_mass;
  P.err_flags = err_flags;
  P.accept_prob = accept_prob;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (dtype) {
    case SPEC_DTYPE_F32: e = launch_typed<float>(g, P, st); break;
    case SPEC_DTYPE_BF16: e = launch_typed<__nv_bfloat16>(g, P, st); break;
    default: e = launch_typed<__half>(g, P, st); break;
  }
  if (e == cudaErrorInvalidConfiguration) return SPEC_ERR_UNSUPPORTED;
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
