// noalloc.cu -- gmlp_forward_noalloc: the fused grouped-MLP forward for callers
// that cannot allocate device memory.  Its scratch lives in a file-scope
// static device array of fixed size instead of a caller-provided workspace;
// the computation is gmlp_forward's, unchanged.
#include <cstdio>
#include <mutex>

#include "internal.h"

namespace gmlp {
namespace {

// Upper bound of the scratch one call may use.  Every GPU that loads this
// library keeps this much device memory reserved until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch per device (the name is only a host-side
// stand-in in host code; the address comes from cudaGetSymbolAddress).
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};

gmlp_status scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_last_error(GMLP_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return set_last_error(GMLP_ERR_UNSUPPORTED_DEVICE, "device index above 63");
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      char msg[256];
      snprintf(msg, sizeof(msg), "cudaGetSymbolAddress of the static scratch failed: %s", cudaGetErrorString(e));
      return set_last_error(GMLP_ERR_CUDA, msg);
    }
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return GMLP_OK;
}

}  // namespace
}  // namespace gmlp

extern "C" gmlp_status gmlp_forward_noalloc(const uint16_t* x, int64_t M, int64_t K, int64_t N,
                                            const int64_t* split_sizes, int32_t G, const gmlp_qweight* W1,
                                            const gmlp_qweight* W2, const float* probs, int32_t act,
                                            const gmlp_recipe* recipe, uint16_t* y, const gmlp_fwd_aux* aux,
                                            gmlp_stream stream) {
  using namespace gmlp;
  if (!recipe) return set_last_error(GMLP_ERR_INVALID_ARG, "recipe is NULL");
  const size_t need = gmlp_forward_workspace_size(M, K, N, G, act, recipe);
  if (need > kNoAllocScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "these sizes need %zu bytes of scratch; gmlp_forward_noalloc has a fixed %zu-byte scratch "
             "(use gmlp_forward with a workspace)",
             need, kNoAllocScratchBytes);
    return set_last_error(GMLP_ERR_WORKSPACE, msg);
  }
  void* scratch = nullptr;
  gmlp_status st = scratch_for_current_device(&scratch);
  if (st != GMLP_OK) return st;
  return gmlp_forward(x, M, K, N, split_sizes, G, W1, W2, probs, act, recipe, y, aux, scratch,
                      kNoAllocScratchBytes, stream);
}
