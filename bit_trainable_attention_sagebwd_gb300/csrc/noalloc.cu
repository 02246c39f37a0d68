// Backward whose scratch lives in a fixed array inside the library, for callers
// that cannot allocate device memory themselves (see sage_attn_bwd_noalloc in
// include/sage_attn.h).  The array is a file-scope __device__ variable: every
// GPU that loads the library holds SAGE_ATTN_NOALLOC_SCRATCH_BYTES of it until
// the process exits.  In host code its name is only a host-side stand-in, so
// the device address is looked up with cudaGetSymbolAddress, once per device.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/sage_attn.h"
#include "args.h"
#include "kernels.h"
#include "layout.h"

namespace {

static __device__ __align__(256) unsigned char g_bwd_scratch[SAGE_ATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices];

// Device address of g_bwd_scratch on the current device (first call per device
// performs the lookup with that device current).
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SAGE_ERR_CUDA;
  std::lock_guard<std::mutex> g(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr) return SAGE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SAGE_OK;
}

bool aligned16(const void* p) { return p != nullptr && ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" int sage_attn_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                                     const float* LSE, const void* dO, void* dQ, void* dK, void* dV,
                                     const void* ws, int B, int H, int N, int D, int causal, int qk_norm,
                                     int k_smooth, float sm_scale, void* stream) {
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(dO) || !aligned16(dQ) ||
      !aligned16(dK) || !aligned16(dV) || !aligned16(ws) || LSE == nullptr || ((uintptr_t)LSE & 3u))
    return SAGE_ERR_INVALID_ARG;
  if (!sage::scale_ok(sm_scale)) return SAGE_ERR_INVALID_ARG;
  const size_t need = sage_attn_bwd_ws_bytes(B, H, N, D);
  if (need == 0) return SAGE_ERR_UNSUPPORTED;
  if (need > (size_t)SAGE_ATTN_NOALLOC_SCRATCH_BYTES) return SAGE_ERR_UNSUPPORTED;  // too large for the array
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != SAGE_OK) return rc;
  const float scale = sage::resolve_scale(sm_scale, D);
  // the launcher zeroes the dQ accumulator and writes every other scratch section
  // before reading it, so nothing left from an earlier call leaks into this one
  return sage::launch_bwd(Q, K, V, O, LSE, dO, dQ, dK, dV, ws, scratch, B, H, N, D, causal != 0, qk_norm != 0,
                          k_smooth != 0, scale, static_cast<cudaStream_t>(stream));
}
