// The backward preprocessing term delta, two ways:
//  * delta = rowsum(dO o O): a bandwidth-bound pass over two BF16 tensors with
//    16-byte loads and FP32 accumulation (priors.kr post "BF16 플래시 어텐션은 왜
//    수천 스텝 뒤에 무너질까", three-line summary and method, paper §3.2 -- the
//    term through which the rounding error enters);
//  * delta = rowsum(dP o P) with P = exp(alpha Q K^T - lse) and dP = dO V^T
//    recomputed on tcgen05: the mathematically equal alternative that the paper
//    found stable (same sources; bud-325 note, Key claims).
#include "pfa_device.cuh"

namespace pfa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// TPR threads per row, each loading 8 BF16 values (16 bytes) of O and of dO.
// zero_ws non-null: the row's d FP32 values of the dQ workspace are zeroed in the
// same pass (each thread writes the 32 bytes that match its 16 of O and dO), so
// that the backward call can skip its own zeroing pass.
template <int TPR>
__global__ void __launch_bounds__(256) delta_kernel(const uint4* __restrict__ o,
                                                    const uint4* __restrict__ dO,
                                                    float* __restrict__ delta, long long rows,
                                                    float4* __restrict__ zero_ws) {
  constexpr int kRowsPerBlock = 256 / TPR;
  const int sub = threadIdx.x % TPR;
  grid_launch_dependents();
  grid_dependency_wait();   // O is the previous kernel's output
  // The loop condition depends only on the block's base row, so whole warps stay
  // together for the shuffles; rows past the end contribute nothing.
  for (long long base = blockIdx.x * static_cast<long long>(kRowsPerBlock); base < rows;
       base += static_cast<long long>(gridDim.x) * kRowsPerBlock) {
    const long long row = base + threadIdx.x / TPR;
    float acc = 0.f;
    if (row < rows) {
      const uint4 a = __ldg(o + row * TPR + sub);
      const uint4 g = __ldg(dO + row * TPR + sub);
      const uint32_t av[4] = {a.x, a.y, a.z, a.w};
      const uint32_t gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        acc = fmaf(bf16lo_to_f32(av[u]), bf16lo_to_f32(gv[u]), acc);
        acc = fmaf(bf16hi_to_f32(av[u]), bf16hi_to_f32(gv[u]), acc);
      }
      if (zero_ws != nullptr) {
        float4* w = zero_ws + row * (2 * TPR) + 2 * sub;
        w[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        w[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
    if (sub == 0 && row < rows) delta[row] = acc;
  }
}

// ---------------------------------------------------------------------------
// delta via rowsum(dP o P). CTA = one 128-row query tile of one (batch, head).
// warp 0 TMA, warp 1 MMA (S = Q K_j^T into TMEM [0,128), dP = dO V_j^T into
// [128,256)), warps 2..5 one query row per thread.
// ---------------------------------------------------------------------------
constexpr int kThreads = 192;

template <int D>
struct AltLayout {
  static constexpr int kStages = 2;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kPanelBytes = kTile * 128;
  static constexpr int kQ = 0;
  static constexpr int kDO = kQ + kTileBytes;
  static constexpr int kK = kDO + kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kBars = kV + kStages * kTileBytes;
  static constexpr int bQFull = 0;
  static constexpr int bKVFull = 1;
  static constexpr int bKVEmpty = bKVFull + kStages;
  static constexpr int bSFull = bKVEmpty + kStages;
  static constexpr int bSFree = bSFull + 1;
  static constexpr int bDrain = bSFree + 1;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kTmemSlot = kBars + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kBytes = kAbort + 4;
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    delta_alt_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                     const DeltaAltArgs args) {
  using L = AltLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const AttnShape& sh = args.s;
  const int N = sh.N;
  const int n_t = (N + kTile - 1) / kTile;
  const int BHq = sh.B * sh.Hq;
  const int bh = blockIdx.x % BHq;
  const int qt = n_t - 1 - static_cast<int>(blockIdx.x / BHq);
  const int q0 = qt * kTile;
  const int b = bh / sh.Hq;
  const int h = bh % sh.Hq;
  const int bh_kv = b * sh.Hkv + h / (sh.Hq / sh.Hkv);
  const int n_kt = CAUSAL ? min(qt + 1, n_t) : n_t;

  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  auto bar = [&](int i) { return sbase + L::kBars + 8u * static_cast<uint32_t>(i); };
  const WaitCtl ctl{abort_flag, args.err, args.err_site, sbase, 3u};

  if (threadIdx.x == 0) {
    *abort_flag = (sbase & 1023u) ? 1 : 0;
    if (sbase & 1023u) atomicOr(args.err, PFA_DEVERR_SMEM_ALIGN);
    mbar_init(bar(L::bQFull), 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::bKVFull + s), 1);
      mbar_init(bar(L::bKVEmpty + s), 1);
    }
    mbar_init(bar(L::bSFull), 1);
    mbar_init(bar(L::bSFree), 4);
    mbar_init(bar(L::bDrain), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Setup done: let the next kernel on the stream be scheduled as CTAs leave, and
  // order every global access after the kernel before this one.
  grid_launch_dependents();
  grid_dependency_wait();

  if (*abort_flag == 0) {
    if (warp == 0) {
      // TMA producer (whole warp, one elected lane issues).
      mbar_arrive_expect_tx_warp(bar(L::bQFull), 2 * L::kTileBytes);
      for (int p = 0; p < D / 64; ++p) {
        tma_load_3d_warp(sbase + L::kQ + p * L::kPanelBytes, &tmQ, bar(L::bQFull), p * 64, q0, bh);
        tma_load_3d_warp(sbase + L::kDO + p * L::kPanelBytes, &tmdO, bar(L::bQFull), p * 64, q0, bh);
      }
      int issued = 0;
      for (int j = 0; j < n_kt; ++j) {
        const int s = j % L::kStages;
        const uint32_t ph = (j / L::kStages) & 1;
        if (!wait_warp(bar(L::bKVEmpty + s), ph ^ 1, ctl)) break;
        issued = j + 1;
        mbar_arrive_expect_tx_warp(bar(L::bKVFull + s), 2 * L::kTileBytes);
        for (int p = 0; p < D / 64; ++p) {
          tma_load_3d_warp(sbase + L::kK + s * L::kTileBytes + p * L::kPanelBytes, &tmK,
                           bar(L::bKVFull + s), p * 64, j * kTile, bh_kv);
          tma_load_3d_warp(sbase + L::kV + s * L::kTileBytes + p * L::kPanelBytes, &tmV,
                           bar(L::bKVFull + s), p * 64, j * kTile, bh_kv);
        }
      }
      wait_drain(bar(L::bQFull), 0, ctl);
      for (int j = issued > L::kStages ? issued - L::kStages : 0; j < issued; ++j)
        wait_drain(bar(L::bKVFull + j % L::kStages), (j / L::kStages) & 1, ctl);
    } else if (warp == 1) {
      // MMA issuer (whole warp, one elected lane issues).
      constexpr uint32_t id = idesc_bf16(128, 128, false, false);
      bool ok = wait_warp(bar(L::bQFull), 0, ctl);
      for (int j = 0; ok && j < n_kt; ++j) {
        const int s = j % L::kStages;
        const uint32_t ph = (j / L::kStages) & 1;
        if (!(ok = wait_warp(bar(L::bKVFull + s), ph, ctl))) break;
        if (j > 0 && !(ok = wait_warp(bar(L::bSFree), (j - 1) & 1, ctl))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
          umma_bf16_warp(tmem, sdesc_sw128(sbase + L::kQ + koff, 16, 1024),
                         sdesc_sw128(sbase + L::kK + s * L::kTileBytes + koff, 16, 1024), id, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
          umma_bf16_warp(tmem + 128, sdesc_sw128(sbase + L::kDO + koff, 16, 1024),
                         sdesc_sw128(sbase + L::kV + s * L::kTileBytes + koff, 16, 1024), id, kk > 0);
        }
        umma_commit_warp(bar(L::bSFull));
        umma_commit_warp(bar(L::bKVEmpty + s));
      }
      umma_commit_warp(bar(L::bDrain));
      wait_drain(bar(L::bDrain), 0, ctl);
    } else {
      const uint32_t quarter = warp & 3;
      const int r = quarter * 32 + lane;
      const int qrow = q0 + r;
      const uint32_t lane_off = (quarter * 32u) << 16;
      const float lse2 =
          qrow < N ? args.lse[static_cast<size_t>(bh) * N + qrow] * kLog2e : INFINITY;
      float acc[2] = {0.f, 0.f};
      bool ok = true;
      for (int j = 0; j < n_kt; ++j) {
        const int k0 = j * kTile;
        const bool need_mask = (CAUSAL && k0 + kTile > q0) || (k0 + kTile > N);
        if (!(ok = wait_warp(bar(L::bSFull), j & 1, ctl))) break;
        tc_fence_after();
#pragma unroll 1
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t sv[32], pv[32];
          tmem_ld32(tmem + lane_off + c4 * 32, sv);
          tmem_ld_wait32(sv);
          tmem_ld32(tmem + 128 + lane_off + c4 * 32, pv);
          tmem_ld_wait32(pv);
#pragma unroll
          for (int t = 0; t < 32; ++t) {
            float pr = ex2_approx(fmaf(__uint_as_float(sv[t]), sh.scale_log2, -lse2));
            if (need_mask) {
              const int key = k0 + c4 * 32 + t;
              pr = (key < N && (!CAUSAL || key <= qrow)) ? pr : 0.f;
            }
            acc[t & 1] = fmaf(pr, __uint_as_float(pv[t]), acc[t & 1]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::bSFree));
      }
      if (ok && qrow < N) args.delta[static_cast<size_t>(bh) * N + qrow] = acc[0] + acc[1];
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

template <int D, bool CAUSAL>
cudaError_t launch_alt_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const DeltaAltArgs& a, cudaStream_t stream) {
  using L = AltLayout<D>;
  auto kern = delta_alt_kernel<D, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  if (e != cudaSuccess) return e;
  const int n_t = (a.s.N + kTile - 1) / kTile;
  const dim3 grid(static_cast<unsigned>(n_t) * a.s.B * a.s.Hq);
  return launch_pdl(kern, grid, dim3(kThreads), L::kBytes, stream, tq, tk, tv, tdo, a);
}

}  // namespace

cudaError_t launch_delta(const void* o, const void* dO, float* delta, long long rows, int d,
                         cudaStream_t stream, float* zero_ws) {
  const int threads = 256;
  const int tpr = d / 8;
  const long long rows_per_block = threads / tpr;
  long long blocks = (rows + rows_per_block - 1) / rows_per_block;
  if (blocks > 152 * 8) blocks = 152 * 8;
  if (blocks < 1) blocks = 1;
  const dim3 grid(static_cast<unsigned>(blocks));
  if (d == 64)
    return launch_pdl(delta_kernel<8>, grid, dim3(threads), 0, stream, static_cast<const uint4*>(o),
                      static_cast<const uint4*>(dO), delta, rows, reinterpret_cast<float4*>(zero_ws));
  return launch_pdl(delta_kernel<16>, grid, dim3(threads), 0, stream, static_cast<const uint4*>(o),
                    static_cast<const uint4*>(dO), delta, rows, reinterpret_cast<float4*>(zero_ws));
}

cudaError_t launch_delta_alt(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const CUtensorMap& tdo, const DeltaAltArgs& a, cudaStream_t stream) {
  if (a.s.d == 64)
    return a.s.causal ? launch_alt_t<64, true>(tq, tk, tv, tdo, a, stream)
                      : launch_alt_t<64, false>(tq, tk, tv, tdo, a, stream);
  return a.s.causal ? launch_alt_t<128, true>(tq, tk, tv, tdo, a, stream)
                    : launch_alt_t<128, false>(tq, tk, tv, tdo, a, stream);
}

}  // namespace pfa
