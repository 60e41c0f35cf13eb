// spec_verify_static.cu -- spec_verify_chain for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device scratch: a plugin inside an engine that reserved all
// of the GPU's memory for its own pool at start-up, a runtime hook that must not call cudaMalloc
// because cudaMalloc may synchronise the device in the middle of a latency-critical step, or a
// binding from a language with no CUDA allocator at hand.  This entry point serves them: its
// scratch is one file-scope device array, which the driver places in memory when the library's
// device code is loaded on a GPU and which stays there until the process exits.
//
// In host code `g_static_scratch` is only a host-side stand-in for the array, never a device
// address: a kernel handed it would fault, or on a system where the GPU can reach host memory
// silently work on the wrong bytes.  The device address comes from cudaGetSymbolAddress, taken
// once per device with that device current, and is what the kernels receive.
#include <mutex>

#include "spec_verify.h"
#include "verify_kernel.cuh"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[SPEC_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of this GPU's copy of the array (set up on the first call on each device).
spec_status_t scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPEC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return SPEC_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SPEC_OK;
}

}  // namespace

extern "C" spec_status_t spec_verify_chain_static(const void* target_logits, const void* draft_logits,
                                                  spec_dtype_t dtype, int B, int K, int V, float temperature,
                                                  const int32_t* draft_tokens, const float* r, const float* u,
                                                  int32_t* num_accepted, int32_t* out_tokens,
                                                  float* residual_mass, int32_t* err_flags,
                                                  spec_stream_t stream) {
  if (B < 0 || K < 0 || V < 1) return SPEC_ERR_INVALID_ARG;
  if (K > SPEC_MAX_K) return SPEC_ERR_UNSUPPORTED;  // as spec_verify_chain reports it (and 2K + 1 stays small)
  if (B == 0) return SPEC_OK;
  // Scratch this call needs (rows read per request: 2K + 1 with draft logits, K + 1 greedy).
  const int rows = (temperature > 0.f && K > 0) ? 2 * K + 1 : K + 1;
  const size_t need = spec_verify_workspace_bytes(B, rows, V, dtype);
  if (need == 0) return SPEC_ERR_INVALID_ARG;
  if (need > (size_t)SPEC_STATIC_WORKSPACE_BYTES) return SPEC_ERR_UNSUPPORTED;  // batch too large
  void* scratch = nullptr;
  const spec_status_t st = scratch_for_current_device(&scratch);
  if (st != SPEC_OK) return st;
  // spec_verify_chain clears the array (one memset of this call's layout) on the first call of a
  // shape at this address; every later call of that shape relies on the previous call having left
  // the counters at zero, which each call does before it ends, a call whose device wait timed out
  // included (its last CTA zeroes them).  Statistics left behind carry an older call's tag and are
  // never taken.
  return spec_verify_chain(target_logits, draft_logits, dtype, B, K, V, temperature, nullptr, draft_tokens, r, u,
                           num_accepted, out_tokens, residual_mass, err_flags, nullptr, nullptr, nullptr,
                           nullptr, nullptr, scratch, (size_t)SPEC_STATIC_WORKSPACE_BYTES, stream);
}
