// pfa_attn_bwd_noalloc: the backward pass for callers that must not allocate
// device memory. The dQ accumulation buffer that pfa_attn_bwd takes from the
// caller lives here in a fixed-size array that the library owns for the life of
// the process on every GPU that loads it.
//
// Who needs this: code running where device allocation is off limits, such as a
// host runtime that reserved all device memory up front in its own pool and
// forbids further cudaMalloc calls, a real-time loop where cudaMalloc's implicit
// synchronisation and latency are not acceptable, or a plugin inside another
// framework that only hands it input and output buffers.
#include <cstddef>
#include <mutex>

#include "pfa_internal.h"

namespace {

// Capacity of the shared dQ accumulation buffer: B * H_q * N * d FP32 values.
constexpr size_t kNoallocMaxElems = size_t(1) << 23;  // 8,388,608 values = 32 MiB

// One array per device, created when the library's device code is loaded. In
// host code this name only stands in for the symbol: its device address must be
// looked up with cudaGetSymbolAddress, with the device current.
static __device__ __align__(256) float g_bwd_dq_scratch[kNoallocMaxElems];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
// The array's address per device, and the id of the CUDA context it was taken in:
// a symbol has one address per context, so a call from another context (a
// caller's own driver context, or a primary context created anew after
// cudaDeviceReset) looks it up again.
struct ScratchAddr {
  unsigned long long ctx = 0;
  float* ptr = nullptr;
};
ScratchAddr g_scratch[kMaxDevices];

int scratch_on_current_device(float** out) {
  int dev = 0;
  const cudaError_t ge = cudaGetDevice(&dev);
  if (ge != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    pfa::note_cuda_error(ge);
    return PFA_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  unsigned long long id = 0;
  int rc = pfa::context_id(&id);
  if (rc != PFA_OK) return rc;
  ScratchAddr& s = g_scratch[dev];
  if (id == 0 || id != s.ctx || s.ptr == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_bwd_dq_scratch);
    if (e != cudaSuccess || p == nullptr) {
      pfa::note_cuda_error(e);
      return PFA_ERR_LAUNCH;
    }
    // The lookup created the primary context if none was current.
    if ((rc = pfa::context_id(&id)) != PFA_OK) return rc;
    s.ptr = static_cast<float*>(p);
    s.ctx = id;
  }
  *out = s.ptr;
  return PFA_OK;
}

}  // namespace

extern "C" int pfa_attn_bwd_noalloc(const pfa_bf16* q, const pfa_bf16* k, const pfa_bf16* v,
                                    const pfa_bf16* dO, const float* lse, const float* delta,
                                    pfa_bf16* dq, pfa_bf16* dk, pfa_bf16* dv, int B, int H_q,
                                    int H_kv, int N, int d, int causal, float scale,
                                    pfa_stream_t stream) {
  const size_t need = pfa_bwd_workspace_bytes(B, H_q, N, d);
  if (need == 0) return PFA_ERR_INVALID_ARG;
  if (need > kNoallocMaxElems * sizeof(float)) return PFA_ERR_TOO_LARGE;
  // An unsupported device is reported as such before the symbol lookup.
  int rc = pfa::check_device();
  if (rc != PFA_OK) return rc;
  float* scratch = nullptr;
  if ((rc = scratch_on_current_device(&scratch)) != PFA_OK) return rc;
  // pfa_attn_bwd zeroes the buffer on `stream` before its kernels accumulate into it.
  return pfa_attn_bwd(q, k, v, dO, lse, delta, dq, dk, dv, scratch, B, H_q, H_kv, N, d, causal,
                      scale, stream);
}
