// C ABI of libpfa (declared in include/pfa.h): argument checks, TMA tensor-map
// encoding, the device error word, and the launch sequence of each entry point.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "pfa_internal.h"

namespace {

// Device error word: kernels OR PFA_DEVERR_* bits into it instead of trapping.
__device__ int g_pfa_device_error;
// Where the first bounded wait gave up since the last clear (0 if none).
__device__ unsigned long long g_pfa_device_error_site;

constexpr int kMaxDevices = 64;
constexpr float kLog2e = 1.4426950408889634f;
// BF16(exp(x)) == 1.0 exactly when x >= -ln(1 - 2^-9): the round-to-one window.
constexpr double kRoundToOneWindow = 1.9550348e-3;

struct DeviceState {
  bool checked = false;
  bool supported = false;
  unsigned long long ctx = 0;  // id of the context the addresses below belong to (0: none yet)
  int* err = nullptr;  // device address of g_pfa_device_error in that context
  unsigned long long* site = nullptr;  // device address of g_pfa_device_error_site
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_get_id = nullptr;
bool g_entry_points_tried = false;

// The most recent CUDA error seen by this thread's calls into the library.
thread_local cudaError_t g_last_cuda_error = cudaSuccess;

// Driver entry points, looked up once (the caller holds g_mu).
void load_entry_points() {
  if (g_entry_points_tried) return;
  g_entry_points_tried = true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess && q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_ctx_get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
  cudaGetLastError();  // a failed lookup leaves nothing pending
}

// Whether the current device is an sm_103 part (looked up once per device; the
// caller holds g_mu).
int check_device_locked(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return PFA_ERR_UNSUPPORTED;
  }
  DeviceState& st = g_dev[dev];
  if (!st.checked) {
    int major = 0, minor = 0;
    const cudaError_t e1 = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    const cudaError_t e2 = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e1 != cudaSuccess || e2 != cudaSuccess) {
      g_last_cuda_error = e1 != cudaSuccess ? e1 : e2;
      cudaGetLastError();
      return PFA_ERR_LAUNCH;
    }
    st.supported = (major == 10 && minor == 3);
    st.checked = true;
  }
  load_entry_points();
  if (!st.supported || g_encode == nullptr || g_ctx_current == nullptr || g_ctx_get_id == nullptr)
    return PFA_ERR_UNSUPPORTED;
  *dev_out = dev;
  return PFA_OK;
}

// Looks up, with the device current, whether it is an sm_103 part and where the
// error words live. Module symbols have one address per CUDA context, so the
// addresses are looked up again whenever the thread's current context is not
// the one they were taken in (a caller's own driver context, or a primary
// context created anew after cudaDeviceReset).
int current_device(DeviceState** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  int rc = check_device_locked(&dev);
  if (rc != PFA_OK) return rc;
  DeviceState& st = g_dev[dev];
  unsigned long long id = 0;
  if ((rc = pfa::context_id(&id)) != PFA_OK) return rc;
  if (id == 0 || id != st.ctx) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_pfa_device_error);
    void* p2 = nullptr;
    if (e == cudaSuccess) e = cudaGetSymbolAddress(&p2, g_pfa_device_error_site);
    if (e != cudaSuccess) {
      g_last_cuda_error = e;
      cudaGetLastError();
      return PFA_ERR_LAUNCH;
    }
    // The lookup created the primary context if none was current.
    if ((rc = pfa::context_id(&id)) != PFA_OK) return rc;
    st.err = static_cast<int*>(p);
    st.site = static_cast<unsigned long long*>(p2);
    st.ctx = id;
  }
  *out = &st;
  return PFA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_sizes(int B, int Hq, int Hkv, int N, int d) {
  if (B < 1 || Hq < 1 || Hkv < 1 || N < 1) return PFA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return PFA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return PFA_ERR_INVALID_ARG;
  const long long elems = static_cast<long long>(B) * Hq * N * d;
  if (elems >= (1ll << 31)) return PFA_ERR_INVALID_ARG;
  return PFA_OK;
}

bool good_scale(float s) { return std::isfinite(s) && s > 0.f; }

// [B*H, N, d] BF16 tensor, boxes of 64 columns (128 bytes, 128B swizzle) x 128 rows.
int tile_map(CUtensorMap* m, const void* base, int BH, int N, int d, int rows = pfa::kTile) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(N) * d * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PFA_OK : PFA_ERR_INVALID_ARG;
}

// [B*H, N, d] FP32 tensor (the dQ workspace), boxes of 32 columns (128 bytes,
// 128B swizzle) x 32 rows: half of one backward drain warp's share of a dQ tile.
int f32_box_map(CUtensorMap* m, const void* base, int BH, int N, int d) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4,
                                 static_cast<cuuint64_t>(N) * d * 4};
  const cuuint32_t box[3] = {32, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PFA_OK : PFA_ERR_INVALID_ARG;
}

pfa::AttnShape shape(int B, int Hq, int Hkv, int N, int d, int causal, float scale) {
  pfa::AttnShape s;
  s.B = B;
  s.Hq = Hq;
  s.Hkv = Hkv;
  s.N = N;
  s.d = d;
  s.causal = causal ? 1 : 0;
  s.scale = scale;
  s.scale_log2 = scale * kLog2e;
  return s;
}

int launched(cudaError_t e) {
  if (e == cudaSuccess) return PFA_OK;
  g_last_cuda_error = e;
  return PFA_ERR_LAUNCH;
}

}  // namespace

namespace pfa {

int context_id(unsigned long long* id) {
  *id = 0;
  if (g_ctx_current == nullptr || g_ctx_get_id == nullptr) return PFA_ERR_UNSUPPORTED;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS) return PFA_ERR_LAUNCH;
  if (ctx == nullptr) return PFA_OK;  // no context current yet
  return g_ctx_get_id(ctx, id) == CUDA_SUCCESS ? PFA_OK : PFA_ERR_LAUNCH;
}

int check_device() {
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  return check_device_locked(&dev);
}

void note_cuda_error(cudaError_t e) {
  if (e == cudaSuccess) return;
  g_last_cuda_error = e;
  cudaGetLastError();
}

}  // namespace pfa

extern "C" {

int pfa_attn_fwd(const pfa_bf16* q, const pfa_bf16* k, const pfa_bf16* v, pfa_bf16* o, float* lse,
                 int B, int H_q, int H_kv, int N, int d, int causal, float scale, int fix_mode,
                 float beta, float eps, pfa_counters* counters, pfa_stream_t stream) {
  return pfa_attn_fwd_ex(q, k, v, o, lse, B, H_q, H_kv, N, d, causal, scale, fix_mode, beta, eps,
                         counters, nullptr, 0u, stream);
}

int pfa_attn_fwd_ex(const pfa_bf16* q, const pfa_bf16* k, const pfa_bf16* v, pfa_bf16* o, float* lse,
                    int B, int H_q, int H_kv, int N, int d, int causal, float scale, int fix_mode,
                    float beta, float eps, pfa_counters* counters, pfa_monitor* monitor,
                    unsigned flags, pfa_stream_t stream) {
  if (!q || !k || !v || !o || !lse) return PFA_ERR_INVALID_ARG;
  int rc = check_sizes(B, H_q, H_kv, N, d);
  if (rc != PFA_OK) return rc;
  if (flags & ~static_cast<unsigned>(PFA_FWD_UNFUSED_BF16_PV | PFA_FWD_PBAR_E4M3 | PFA_FWD_PBAR_MXFP4 |
                                     PFA_FWD_PAIR_CTA))
    return PFA_ERR_INVALID_ARG;
  if ((flags & PFA_FWD_PBAR_E4M3) && (flags & PFA_FWD_PBAR_MXFP4)) return PFA_ERR_INVALID_ARG;
  const bool profile = (flags & PFA_FWD_UNFUSED_BF16_PV) != 0;
  const int pbar = (flags & PFA_FWD_PBAR_E4M3) ? 1 : (flags & PFA_FWD_PBAR_MXFP4) ? 2 : 0;
  const bool pair = (flags & PFA_FWD_PAIR_CTA) != 0;
  if ((profile || pbar) && d != 64) return PFA_ERR_UNSUPPORTED;
  if (pair && (d != 128 || profile || pbar || monitor)) return PFA_ERR_UNSUPPORTED;
  if (!good_scale(scale) || fix_mode < 0 || fix_mode > 2) return PFA_ERR_INVALID_ARG;
  if (fix_mode == 1 && !(std::isfinite(beta) && beta > 1.f)) return PFA_ERR_INVALID_ARG;
  const bool ties = fix_mode != 0 || counters != nullptr || monitor != nullptr;
  if (ties && !(std::isfinite(eps) && eps >= 0.f)) return PFA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      (counters && (reinterpret_cast<uintptr_t>(counters) & 7u)) ||
      (monitor && (reinterpret_cast<uintptr_t>(monitor) & 7u)))
    return PFA_ERR_MISALIGNED;
  DeviceState* dev = nullptr;
  if ((rc = current_device(&dev)) != PFA_OK) return rc;
  CUtensorMap tq, tk, tv;
  if ((rc = tile_map(&tq, q, B * H_q, N, d)) != PFA_OK) return rc;
  if ((rc = tile_map(&tk, k, B * H_kv, N, d)) != PFA_OK) return rc;
  if ((rc = tile_map(&tv, v, B * H_kv, N, d)) != PFA_OK) return rc;
  pfa::FwdArgs a;
  a.s = shape(B, H_q, H_kv, N, d, causal, scale);
  a.o = o;
  a.lse = lse;
  a.counters = reinterpret_cast<long long*>(counters);
  a.monitor = reinterpret_cast<long long*>(monitor);
  a.err = dev->err;
  a.err_site = dev->site;
  a.fix_mode = fix_mode;
  a.beta = fix_mode == 1 ? beta : 2.f;
  a.eps_raw = ties ? eps / scale : 0.f;
  a.tau_raw = static_cast<float>(kRoundToOneWindow / scale);
  a.profile = profile ? 1 : 0;
  a.pbar = pbar;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (pair) {
    // Each CTA of a pair loads half of a K tile: 64-row boxes.
    CUtensorMap tk64;
    if ((rc = tile_map(&tk64, k, B * H_kv, N, d, 64)) != PFA_OK) return rc;
    return launched(pfa::launch_fwd_pair(tq, tk64, tv, a, st));
  }
  if (pbar) return launched(pfa::launch_fwd_lowp(tq, tk, tv, a, st));
  if (profile || monitor) return launched(pfa::launch_fwd_study(tq, tk, tv, a, st));
  return launched(pfa::launch_fwd(tq, tk, tv, a, st));
}

int pfa_attn_delta(const pfa_bf16* o, const pfa_bf16* dO, float* delta, int B, int H_q, int N,
                   int d, pfa_stream_t stream) {
  if (!o || !dO || !delta) return PFA_ERR_INVALID_ARG;
  int rc = check_sizes(B, H_q, H_q, N, d);
  if (rc != PFA_OK) return rc;
  if (!aligned16(o) || !aligned16(dO) || !aligned16(delta)) return PFA_ERR_MISALIGNED;
  DeviceState* dev = nullptr;
  if ((rc = current_device(&dev)) != PFA_OK) return rc;
  return launched(pfa::launch_delta(o, dO, delta, static_cast<long long>(B) * H_q * N, d,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

int pfa_attn_delta_zero(const pfa_bf16* o, const pfa_bf16* dO, float* delta, float* dq_accum, int B,
                        int H_q, int N, int d, pfa_stream_t stream) {
  if (!o || !dO || !delta || !dq_accum) return PFA_ERR_INVALID_ARG;
  int rc = check_sizes(B, H_q, H_q, N, d);
  if (rc != PFA_OK) return rc;
  if (!aligned16(o) || !aligned16(dO) || !aligned16(delta) || !aligned16(dq_accum))
    return PFA_ERR_MISALIGNED;
  DeviceState* dev = nullptr;
  if ((rc = current_device(&dev)) != PFA_OK) return rc;
  return launched(pfa::launch_delta(o, dO, delta, static_cast<long long>(B) * H_q * N, d,
                                    reinterpret_cast<cudaStream_t>(stream), dq_accum));
}

int pfa_attn_delta_alt(const pfa_bf16* q, const pfa_bf16* k, const pfa_bf16* v, const pfa_bf16* dO,
                       const float* lse, float* delta, int B, int H_q, int H_kv, int N, int d,
                       int causal, float scale, pfa_stream_t stream) {
  if (!q || !k || !v || !dO || !lse || !delta) return PFA_ERR_INVALID_ARG;
  int rc = check_sizes(B, H_q, H_kv, N, d);
  if (rc != PFA_OK) return rc;
  if (!good_scale(scale)) return PFA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(lse) ||
      !aligned16(delta))
    return PFA_ERR_MISALIGNED;
  DeviceState* dev = nullptr;
  if ((rc = current_device(&dev)) != PFA_OK) return rc;
  CUtensorMap tq, tk, tv, tdo;
  if ((rc = tile_map(&tq, q, B * H_q, N, d)) != PFA_OK) return rc;
  if ((rc = tile_map(&tk, k, B * H_kv, N, d)) != PFA_OK) return rc;
  if ((rc = tile_map(&tv, v, B * H_kv, N, d)) != PFA_OK) return rc;
  if ((rc = tile_map(&tdo, dO, B * H_q, N, d)) != PFA_OK) return rc;
  pfa::DeltaAltArgs a;
  a.s = shape(B, H_q, H_kv, N, d, causal, scale);
  a.lse = lse;
  a.delta = delta;
  a.err = dev->err;
  a.err_site = dev->site;
  return launched(pfa::launch_delta_alt(tq, tk, tv, tdo, a, reinterpret_cast<cudaStream_t>(stream)));
}

size_t pfa_bwd_workspace_bytes(int B, int H_q, int N, int d) {
  if (check_sizes(B, H_q, H_q, N, d) != PFA_OK) return 0;
  return static_cast<size_t>(B) * H_q * N * d * sizeof(float);
}

}  // extern "C"

namespace {

// Everything the backward kernel's launch needs, checked and encoded before any
// launch, so that an argument error leaves the stream untouched.
struct BwdLaunch {
  CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv;
  pfa::BwdArgs a;
};

// The argument checks shared by pfa_attn_bwd and pfa_attn_bwd_accum, and the
// tensor maps and arguments of the kernel (dq_accum += alpha (P o (dP - delta)) K; dk, dv written).
// dq_accum may be null only when the query-outer pass computes dQ (need_accum false).
int bwd_check(const pfa_bf16* q, const pfa_bf16* k, const pfa_bf16* v, const pfa_bf16* dO,
              const float* lse, const float* delta, const float* dq_accum, const pfa_bf16* dk,
              const pfa_bf16* dv, int B, int H_q, int H_kv, int N, int d, float scale,
              bool need_accum = true) {
  if (!q || !k || !v || !dO || !lse || !delta || !dk || !dv) return PFA_ERR_INVALID_ARG;
  if (need_accum && !dq_accum) return PFA_ERR_INVALID_ARG;
  const int rc = check_sizes(B, H_q, H_kv, N, d);
  if (rc != PFA_OK) return rc;
  if (!good_scale(scale)) return PFA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(lse) ||
      !aligned16(delta) || !aligned16(dk) || !aligned16(dv) || (dq_accum && !aligned16(dq_accum)))
    return PFA_ERR_MISALIGNED;
  return PFA_OK;
}

// dq_accum null: the backward kernel skips dQ (the query-outer pass computes it).
int bwd_prepare(const pfa_bf16* q, const pfa_bf16* k, const pfa_bf16* v, const pfa_bf16* dO,
                const float* lse, const float* delta, float* dq_accum, pfa_bf16* dk, pfa_bf16* dv,
                int B, int H_q, int H_kv, int N, int d, int causal, float scale, BwdLaunch* L) {
  int rc = bwd_check(q, k, v, dO, lse, delta, dq_accum, dk, dv, B, H_q, H_kv, N, d, scale,
                     dq_accum != nullptr);
  if (rc != PFA_OK) return rc;
  DeviceState* dev = nullptr;
  if ((rc = current_device(&dev)) != PFA_OK) return rc;
  if ((rc = tile_map(&L->tq, q, B * H_q, N, d)) != PFA_OK) return rc;
  if ((rc = tile_map(&L->tk, k, B * H_kv, N, d)) != PFA_OK) return rc;
  if ((rc = tile_map(&L->tv, v, B * H_kv, N, d)) != PFA_OK) return rc;
  if ((rc = tile_map(&L->tdo, dO, B * H_q, N, d)) != PFA_OK) return rc;
  if (dq_accum != nullptr) {
    if ((rc = f32_box_map(&L->tdq, dq_accum, B * H_q, N, d)) != PFA_OK) return rc;
  } else {
    L->tdq = CUtensorMap{};   // not used by the kernel that skips dQ
  }
  // dK, dV leave through 64-column x 32-row boxes (d = 64: one drain warp's rows).
  if ((rc = tile_map(&L->tdk, dk, B * H_kv, N, d, 32)) != PFA_OK) return rc;
  if ((rc = tile_map(&L->tdv, dv, B * H_kv, N, d, 32)) != PFA_OK) return rc;
  pfa::BwdArgs& a = L->a;
  a.s = shape(B, H_q, H_kv, N, d, causal, scale);
  a.lse = lse;
  a.delta = delta;
  a.dq_accum = dq_accum;
  a.dk = dk;
  a.dv = dv;
  a.err = dev->err;
  a.err_site = dev->site;
  return PFA_OK;
}

int bwd_launch(const BwdLaunch& L, cudaStream_t st) {
  return launched(pfa::launch_bwd(L.tq, L.tk, L.tv, L.tdo, L.tdq, L.tdk, L.tdv, L.a, st));
}

// dK, dV from the key-outer kernel without its dQ product (L prepared with no dQ
// workspace), then dQ = alpha (P o (dP - delta)) K from the query-outer pass (split: dS as BF16 hi + lo).
int bwd_query_outer(const BwdLaunch& L, pfa_bf16* dq, const float* lse, const float* delta, bool split,
                    cudaStream_t st) {
  pfa::DqArgs da;
  da.s = L.a.s;
  da.lse = lse;
  da.delta = delta;
  da.dq = dq;
  da.err = L.a.err;
  da.err_site = L.a.err_site;
  da.split = split ? 1 : 0;
  const int rc = bwd_launch(L, st);
  if (rc != PFA_OK) return rc;
  return launched(pfa::launch_dq(L.tq, L.tk, L.tv, L.tdo, da, st));
}

}  // namespace

extern "C" {

}  // extern "C"

namespace {

// pfa_attn_bwd; zeroed: the caller vouches that the workspace holds zeros (as
// pfa_attn_delta_zero leaves it), and the zeroing pass is skipped.
int bwd_key_outer(const pfa_bf16* q, const pfa_bf16* k, const pfa_bf16* v, const pfa_bf16* dO,
                  const float* lse, const float* delta, pfa_bf16* dq, pfa_bf16* dk, pfa_bf16* dv,
                  float* dq_accum, int B, int H_q, int H_kv, int N, int d, int causal, float scale,
                  bool zeroed, pfa_stream_t stream) {
  if (!dq) return PFA_ERR_INVALID_ARG;
  int rc = bwd_check(q, k, v, dO, lse, delta, dq_accum, dk, dv, B, H_q, H_kv, N, d, scale);
  if (rc != PFA_OK) return rc;
  if (!aligned16(dq)) return PFA_ERR_MISALIGNED;
  BwdLaunch L;
  if ((rc = bwd_prepare(q, k, v, dO, lse, delta, d == 128 ? nullptr : dq_accum, dk, dv, B, H_q, H_kv,
                        N, d, causal, scale, &L)) != PFA_OK)
    return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // At d = 128 the key-outer kernel has no shared memory left to stage dQ for a tensor
  // reduce and would add it with vector atomics; the query-outer pass is faster there
  // (and deterministic), so it computes dQ and the workspace is not used.
  if (d == 128) return bwd_query_outer(L, dq, lse, delta, /*split=*/false, st);
  const size_t ws = pfa_bwd_workspace_bytes(B, H_q, N, d);
  if (!zeroed &&
      (rc = launched(pfa::launch_zero_workspace(dq_accum, static_cast<long long>(ws / 16), st))) != PFA_OK)
    return rc;
  if ((rc = bwd_launch(L, st)) != PFA_OK) return rc;
  return launched(pfa::launch_convert_dq(dq_accum, dq, static_cast<long long>(ws / sizeof(float)), st));
}

}  // namespace

extern "C" {

int pfa_attn_bwd(const pfa_bf16* q, const pfa_bf16* k, const pfa_bf16* v, const pfa_bf16* dO,
                 const float* lse, const float* delta, pfa_bf16* dq, pfa_bf16* dk, pfa_bf16* dv,
                 float* dq_accum, int B, int H_q, int H_kv, int N, int d, int causal, float scale,
                 pfa_stream_t stream) {
  return bwd_key_outer(q, k, v, dO, lse, delta, dq, dk, dv, dq_accum, B, H_q, H_kv, N, d, causal,
                       scale, false, stream);
}

int pfa_attn_bwd_accum(const pfa_bf16* q, const pfa_bf16* k, const pfa_bf16* v, const pfa_bf16* dO,
                       const float* lse, const float* delta, float* dq_accum, pfa_bf16* dk, pfa_bf16* dv,
                       int B, int H_q, int H_kv, int N, int d, int causal, float scale,
                       pfa_stream_t stream) {
  if (!dq_accum) return PFA_ERR_INVALID_ARG;
  BwdLaunch L;
  const int rc =
      bwd_prepare(q, k, v, dO, lse, delta, dq_accum, dk, dv, B, H_q, H_kv, N, d, causal, scale, &L);
  if (rc != PFA_OK) return rc;
  return bwd_launch(L, reinterpret_cast<cudaStream_t>(stream));
}

int pfa_attn_bwd_ex(const pfa_bf16* q, const pfa_bf16* k, const pfa_bf16* v, const pfa_bf16* dO,
                    const float* lse, const float* delta, pfa_bf16* dq, pfa_bf16* dk, pfa_bf16* dv,
                    float* dq_accum, int B, int H_q, int H_kv, int N, int d, int causal, float scale,
                    unsigned flags, pfa_stream_t stream) {
  if (flags & ~static_cast<unsigned>(PFA_BWD_DQ_DETERMINISTIC | PFA_BWD_DQ_SPLIT | PFA_BWD_WORKSPACE_ZEROED))
    return PFA_ERR_INVALID_ARG;
  if ((flags & (PFA_BWD_DQ_DETERMINISTIC | PFA_BWD_DQ_SPLIT)) == 0)
    return bwd_key_outer(q, k, v, dO, lse, delta, dq, dk, dv, dq_accum, B, H_q, H_kv, N, d, causal,
                         scale, (flags & PFA_BWD_WORKSPACE_ZEROED) != 0, stream);
  // The query-outer pass computes dQ; the key-outer kernel only dK and dV.
  if (!dq) return PFA_ERR_INVALID_ARG;
  int rc = bwd_check(q, k, v, dO, lse, delta, nullptr, dk, dv, B, H_q, H_kv, N, d, scale, false);
  if (rc != PFA_OK) return rc;
  if (!aligned16(dq)) return PFA_ERR_MISALIGNED;
  BwdLaunch L;
  if ((rc = bwd_prepare(q, k, v, dO, lse, delta, nullptr, dk, dv, B, H_q, H_kv, N, d, causal, scale,
                        &L)) != PFA_OK)
    return rc;
  return bwd_query_outer(L, dq, lse, delta, (flags & PFA_BWD_DQ_SPLIT) != 0,
                         reinterpret_cast<cudaStream_t>(stream));
}

const char* pfa_status_string(int status) {
  switch (status) {
    case PFA_OK: return "PFA_OK";
    case PFA_ERR_INVALID_ARG: return "PFA_ERR_INVALID_ARG: invalid pointer, size, mode, beta, eps or scale";
    case PFA_ERR_MISALIGNED: return "PFA_ERR_MISALIGNED: a pointer is not 16-byte aligned";
    case PFA_ERR_UNSUPPORTED: return "PFA_ERR_UNSUPPORTED: current device is not sm_103 or TMA encoding is unavailable";
    case PFA_ERR_LAUNCH: return "PFA_ERR_LAUNCH: a CUDA launch or runtime call failed";
    case PFA_ERR_DEVICE: return "PFA_ERR_DEVICE: a kernel reported a failure in the device error word";
    case PFA_ERR_TOO_LARGE: return "PFA_ERR_TOO_LARGE: B*H_q*N*d exceeds the 8,388,608-value buffer of pfa_attn_bwd_noalloc";
    default: return "PFA_ERR_UNKNOWN";
  }
}

const char* pfa_last_error(void) {
  return g_last_cuda_error == cudaSuccess ? "no CUDA error" : cudaGetErrorString(g_last_cuda_error);
}

int pfa_device_error(int clear) {
  DeviceState* dev = nullptr;
  int rc = current_device(&dev);
  if (rc != PFA_OK) return rc;
  if (cudaDeviceSynchronize() != cudaSuccess) return PFA_ERR_LAUNCH;
  int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_pfa_device_error, sizeof(int)) != cudaSuccess) return PFA_ERR_LAUNCH;
  if (clear) {
    const int zero = 0;
    const unsigned long long zero64 = 0;
    if (cudaMemcpyToSymbol(g_pfa_device_error, &zero, sizeof(int)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_pfa_device_error_site, &zero64, sizeof(zero64)) != cudaSuccess)
      return PFA_ERR_LAUNCH;
  }
  return word;
}

int pfa_wait_probe(pfa_stream_t stream) {
  DeviceState* dev = nullptr;
  const int rc = current_device(&dev);
  if (rc != PFA_OK) return rc;
  return launched(pfa::launch_wait_probe(dev->err, dev->site, reinterpret_cast<cudaStream_t>(stream)));
}

long long pfa_device_error_site(void) {
  DeviceState* dev = nullptr;
  int rc = current_device(&dev);
  if (rc != PFA_OK) return rc;
  if (cudaDeviceSynchronize() != cudaSuccess) return PFA_ERR_LAUNCH;
  unsigned long long site = 0;
  if (cudaMemcpyFromSymbol(&site, g_pfa_device_error_site, sizeof(site)) != cudaSuccess)
    return PFA_ERR_LAUNCH;
  return static_cast<long long>(site & 0x7FFFFFFFFFFFFFFFull);
}

}  // extern "C"
