// Internal declarations shared by the host-side launchers of libpfa.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pfa.h"  // status codes and the PFA_DEVERR_* bits kernels OR into the error word

namespace pfa {

// Launches `kern` on `stream` as a programmatic dependent of the kernel before
// it: the two may overlap, and `kern` orders its global memory accesses after
// the previous kernel with grid_dependency_wait() (pfa_device.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Identity (cuCtxGetId) of the CUDA context current on the calling thread; 0 when
// none is current yet. Module symbols have one device address per context.
int context_id(unsigned long long* id);
// PFA_OK if the current device is an sm_103 part and the driver entry points the
// library needs are present; PFA_ERR_UNSUPPORTED (or PFA_ERR_LAUNCH) otherwise.
int check_device();
// Records a CUDA error for pfa_last_error() on this thread and clears it from
// the runtime, so that it is not reported again by a later call.
void note_cuda_error(cudaError_t e);

constexpr int kTile = 128;  // rows of a Q tile and of a K/V tile

// Arguments common to the tiled kernels (all sizes in elements).
struct AttnShape {
  int B, Hq, Hkv, N, d;
  int causal;
  float scale;        // alpha
  float scale_log2;   // alpha * log2(e)
};

struct FwdArgs {
  AttnShape s;
  void* o;                 // bf16 [B, Hq, N, d]
  float* lse;              // [B, Hq, N]
  long long* counters;     // 3 x int64 or null
  long long* monitor;      // 1 + 8 x int64 (operational ones, tie histogram) or null
  int* err;                // device error word
  unsigned long long* err_site;  // where the first bounded wait gave up
  int fix_mode;
  float beta;
  float eps_raw;           // tie tolerance in units of the unscaled score Q.K
  float tau_raw;           // BF16 round-to-one window in units of Q.K
  int profile;             // the unfused BF16 Pbar V study profile (d = 64)
  int pbar;                // the Pbar operand's format: 0 BF16, 1 FP8 E4M3, 2 MXFP4 (d = 64)
};

struct DeltaAltArgs {
  AttnShape s;
  const float* lse;
  float* delta;
  int* err;
  unsigned long long* err_site;
};

struct BwdArgs {
  AttnShape s;
  const float* lse;
  const float* delta;
  float* dq_accum;         // fp32 [B, Hq, N, d], zeroed before the launch; null: no dQ (the
                           // query-outer pass computes it)
  void* dk;                // bf16 [B, Hkv, N, d]
  void* dv;                // bf16 [B, Hkv, N, d]
  int* err;
  unsigned long long* err_site;
};

struct DqArgs {
  AttnShape s;
  const float* lse;
  const float* delta;
  void* dq;                // bf16 [B, Hq, N, d]
  int* err;
  unsigned long long* err_site;
  int split;               // dS enters the dQ product as BF16 hi + lo
};

cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdArgs& a, cudaStream_t stream);
// The forward kernel's study variants: the monitor (a.monitor) and the unfused
// BF16 profile (a.profile, d = 64); counters as in launch_fwd.
cudaError_t launch_fwd_study(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const FwdArgs& a, cudaStream_t stream);
// The fused path at d = 128 with two CTAs per product (cta_group::2); tk maps K
// with 64-row boxes (tile_map rows = 64).
cudaError_t launch_fwd_pair(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdArgs& a, cudaStream_t stream);
// The narrow Pbar formats (a.pbar 1 or 2; d = 64, monitor counted, profile or fused).
cudaError_t launch_fwd_lowp(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdArgs& a, cudaStream_t stream);
// delta = rowsum(dO o O) over `rows` rows of d values; zero_ws non-null: the matching
// rows x d FP32 values of the dQ workspace are zeroed in the same pass.
cudaError_t launch_delta(const void* o, const void* dO, float* delta, long long rows, int d,
                         cudaStream_t stream, float* zero_ws = nullptr);
cudaError_t launch_delta_alt(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const CUtensorMap& tdo, const DeltaAltArgs& a, cudaStream_t stream);
// tdq: FP32 [B*Hq, N, d] map of the dQ workspace with 32-column x 32-row boxes and
// 128-byte swizzle (the reduce-add target of the d = 64 kernel); tdk, tdv: BF16
// [B*Hkv, N, d] maps of dK, dV with 64-column x 32-row boxes and 128-byte swizzle
// (the store targets of the d = 64 kernel's drain warps).
cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& tdk,
                       const CUtensorMap& tdv, const BwdArgs& a, cudaStream_t stream);
// dQ = alpha (P o (dP - delta)) K by the query-outer pass (deterministic; hi/lo dS when a.split).
cudaError_t launch_dq(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      const CUtensorMap& tdo, const DqArgs& a, cudaStream_t stream);
cudaError_t launch_convert_dq(const float* dq_accum, void* dq, long long n, cudaStream_t stream);
// Zeroes n4 float4 values of the dQ workspace on `stream` (a kernel, so that it
// overlaps its neighbours by programmatic dependent launch).
cudaError_t launch_zero_workspace(float* ws, long long n4, cudaStream_t stream);
// One warp whose bounded wait on an mbarrier that nothing completes gives up
// (PFA_DEVERR_TIMEOUT, error site kernel id 4).
cudaError_t launch_wait_probe(int* err, unsigned long long* site, cudaStream_t stream);

}  // namespace pfa
