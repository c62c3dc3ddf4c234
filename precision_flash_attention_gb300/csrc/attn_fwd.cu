// Forward kernel: S = alpha Q K^T on tcgen05 (FP32 in TMEM), the online safe
// softmax with the repeated-maximum tracker and the per-call shift rule,
// Pbar = exp(S - m) in BF16, Obar += Pbar V on tcgen05 (FP32 in TMEM), then
// O = Obar / l (BF16) and lse = m + ln l (FP32), plus the diagnostic counters.
//
// The method is the one analysed in Qiu & Yao, "Why Low-Precision Transformer
// Training Fails: An Analysis on Flash Attention" (ICLR 2026), as summarised by
// the priors.kr post "BF16 플래시 어텐션은 왜 수천 스텝 뒤에 무너질까" (core idea,
// equations, and the fix of paper §4) and the bud-325 note of the same title
// (Key claims, Method / Algorithm 1).
//
// CTA = one 128-row Q tile of one (batch, query head). 192 threads:
//   warp 0      TMA producer (Q once, then K_j / V_j into a 2-stage ring)
//   warp 1      TMEM owner and single-thread tcgen05.mma issuer
//   warps 2..5  softmax / correction / epilogue, one query row per thread
//               (TMEM lane quarter = warp % 4)
// TMEM: columns [0,128) hold S_j, columns [128, 128+d) hold Obar.
#include "pfa_device.cuh"

namespace pfa {
namespace {

constexpr int kThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kEpsShift = 0.03125f;  // 2^-5

template <int D>
struct FwdLayout {
  static constexpr int kStages = 2;
  static constexpr int kTileBytes = kTile * D * 2;   // 128 rows x D bf16
  static constexpr int kPanelBytes = kTile * 128;    // 128 rows x 64 bf16
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kP = kV + kStages * kTileBytes;
  static constexpr int kBars = kP + kTile * kTile * 2;
  // barrier indices
  static constexpr int bQFull = 0;
  static constexpr int bKFull = 1;                  // + stage
  static constexpr int bVFull = bKFull + kStages;   // + stage
  static constexpr int bKVEmpty = bVFull + kStages; // + stage
  static constexpr int bSFull = bKVEmpty + kStages;
  static constexpr int bSFree = bSFull + 1;
  static constexpr int bPFull = bSFree + 1;
  static constexpr int bODone = bPFull + 1;
  static constexpr int bDrain = bODone + 1;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kTmemSlot = kBars + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kBytes = kAbort + 4;
};

template <int D, int MODE, bool CAUSAL, bool COUNT>
__global__ void __launch_bounds__(kThreads, (D == 64 ? 2 : 1))
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdArgs args) {
  using L = FwdLayout<D>;
  // The tie tracker (running top-2) is needed by the fix modes and by the
  // repeated-row counter, which is reported in every mode.
  constexpr bool kTies = MODE > 0 || COUNT;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const AttnShape& sh = args.s;
  const int N = sh.N;
  const int n_qt = (N + kTile - 1) / kTile;
  const int BHq = sh.B * sh.Hq;
  const int bh = blockIdx.x % BHq;
  const int qt = n_qt - 1 - static_cast<int>(blockIdx.x / BHq);  // heaviest causal tiles first
  const int q0 = qt * kTile;
  const int b = bh / sh.Hq;
  const int h = bh % sh.Hq;
  const int bh_kv = b * sh.Hkv + h / (sh.Hq / sh.Hkv);
  const int n_kt_all = (N + kTile - 1) / kTile;
  const int n_kt = CAUSAL ? min(qt + 1, n_kt_all) : n_kt_all;

  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  auto bar = [&](int i) { return sbase + L::kBars + 8u * static_cast<uint32_t>(i); };
  const WaitCtl ctl{abort_flag, args.err};

  if (threadIdx.x == 0) {
    *abort_flag = (sbase & 1023u) ? 1 : 0;
    if (sbase & 1023u) atomicOr(args.err, PFA_DEVERR_SMEM_ALIGN);
    mbar_init(bar(L::bQFull), 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::bKFull + s), 1);
      mbar_init(bar(L::bVFull + s), 1);
      mbar_init(bar(L::bKVEmpty + s), 1);
    }
    mbar_init(bar(L::bSFull), 1);
    mbar_init(bar(L::bSFree), 4);
    mbar_init(bar(L::bPFull), 4);
    mbar_init(bar(L::bODone), 1);
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
  const uint32_t tS = tmem;
  const uint32_t tO = tmem + 128;

  if (*abort_flag == 0) {
    if (warp == 0) {
      // ---------------- TMA producer ----------------
      if (lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        mbar_arrive_expect_tx(bar(L::bQFull), L::kTileBytes);
        for (int p = 0; p < D / 64; ++p)
          tma_load_3d(sbase + L::kQ + p * L::kPanelBytes, &tmQ, bar(L::bQFull), p * 64, q0, bh);
        int issued = 0;
        for (int j = 0; j < n_kt; ++j) {
          const int s = j % L::kStages;
          const uint32_t ph = (j / L::kStages) & 1;
          if (!wait_thread(bar(L::bKVEmpty + s), ph ^ 1, ctl)) break;
          issued = j + 1;
          mbar_arrive_expect_tx(bar(L::bKFull + s), L::kTileBytes);
          for (int p = 0; p < D / 64; ++p)
            tma_load_3d(sbase + L::kK + s * L::kTileBytes + p * L::kPanelBytes, &tmK,
                        bar(L::bKFull + s), p * 64, j * kTile, bh_kv);
          mbar_arrive_expect_tx(bar(L::bVFull + s), L::kTileBytes);
          for (int p = 0; p < D / 64; ++p)
            tma_load_3d(sbase + L::kV + s * L::kTileBytes + p * L::kPanelBytes, &tmV,
                        bar(L::bVFull + s), p * 64, j * kTile, bh_kv);
        }
        // Drain: every issued copy has landed before shared memory is released.
        wait_drain(bar(L::bQFull), 0, args.err);
        for (int j = issued > L::kStages ? issued - L::kStages : 0; j < issued; ++j) {
          const int s = j % L::kStages;
          const uint32_t ph = (j / L::kStages) & 1;
          wait_drain(bar(L::bKFull + s), ph, args.err);
          wait_drain(bar(L::bVFull + s), ph, args.err);
        }
      }
    } else if (warp == 1) {
      // ---------------- MMA issuer ----------------
      if (lane == 0) {
        constexpr uint32_t idS = idesc_bf16(128, 128, false, false);
        constexpr uint32_t idPV = idesc_bf16(128, D, false, true);
        bool ok = wait_thread(bar(L::bQFull), 0, ctl);
        auto issue_s = [&](int j) {
          const int s = j % L::kStages;
          tc_fence_after();
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
            const uint64_t da = sdesc_sw128(sbase + L::kQ + koff, 16, 1024);
            const uint64_t db = sdesc_sw128(sbase + L::kK + s * L::kTileBytes + koff, 16, 1024);
            umma_bf16(tS, da, db, idS, kk > 0);
          }
          umma_commit(bar(L::bSFull));
        };
        if (ok) ok = wait_thread(bar(L::bKFull + 0), 0, ctl);
        if (ok) issue_s(0);
        for (int j = 0; ok && j < n_kt; ++j) {
          const int s = j % L::kStages;
          const uint32_t ph = (j / L::kStages) & 1;
          if (j + 1 < n_kt) {
            const int s1 = (j + 1) % L::kStages;
            const uint32_t ph1 = ((j + 1) / L::kStages) & 1;
            if (!(ok = wait_thread(bar(L::bKFull + s1), ph1, ctl))) break;
            if (!(ok = wait_thread(bar(L::bSFree), j & 1, ctl))) break;
            issue_s(j + 1);
          }
          if (!(ok = wait_thread(bar(L::bPFull), j & 1, ctl))) break;
          if (!(ok = wait_thread(bar(L::bVFull + s), ph, ctl))) break;
          tc_fence_after();
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint64_t da =
                sdesc_sw128(sbase + L::kP + (kk >> 2) * L::kPanelBytes + (kk & 3) * 32, 16, 1024);
            const uint64_t db =
                sdesc_sw128(sbase + L::kV + s * L::kTileBytes + kk * 2048, L::kPanelBytes, 1024);
            umma_bf16(tO, da, db, idPV, (j > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(bar(L::bKVEmpty + s));
          umma_commit(bar(L::bODone));
        }
        // Drain: no MMA may still read shared memory or write TMEM at teardown.
        umma_commit(bar(L::bDrain));
        wait_drain(bar(L::bDrain), 0, args.err);
      }
    } else {
      // ---------------- softmax warps ----------------
      const uint32_t quarter = warp & 3;
      const int r = quarter * 32 + lane;  // row within the tile == TMEM lane
      const int qrow = q0 + r;
      const uint32_t lane_off = (quarter * 32u) << 16;
      const float sl2 = sh.scale_log2;
      const float alpha = sh.scale;

      float m1 = -INFINITY, m2 = -INFINITY;  // running top-2 of raw scores
      float m_sh = -INFINITY;                // current shift, natural units
      float l = 0.f;
      int cnt = 0;                           // entries within tau of m1 (raw)
      bool ok = true;

      for (int j = 0; j < n_kt; ++j) {
        const int k0 = j * kTile;
        const bool need_mask = (CAUSAL && k0 + kTile > q0) || (k0 + kTile > N);
        if (!(ok = wait_warp(bar(L::bSFull), j & 1, ctl))) break;
        tc_fence_after();

        // Pass 1: tile maximum (and second maximum) over visible keys.
        float a1[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        float a2[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t v[32];
          tmem_ld32(tS + lane_off + c4 * 32, v);
          tmem_ld_wait32(v);
#pragma unroll
          for (int t = 0; t < 32; ++t) {
            float x = __uint_as_float(v[t]);
            if (need_mask) {
              const int key = k0 + c4 * 32 + t;
              const bool vis = key < N && (!CAUSAL || key <= qrow);
              x = vis ? x : -INFINITY;
            }
            if (kTies) a2[t & 3] = fmaxf(a2[t & 3], fminf(a1[t & 3], x));
            a1[t & 3] = fmaxf(a1[t & 3], x);
          }
        }
        float t1 = a1[0], t2 = a2[0];
#pragma unroll
        for (int i = 1; i < 4; ++i) {
          if (kTies) t2 = fmaxf(fmaxf(t2, a2[i]), fminf(t1, a1[i]));
          t1 = fmaxf(t1, a1[i]);
        }
        const float m1_old = m1;
        if (kTies) m2 = fmaxf(fmaxf(m2, t2), fminf(m1, t1));
        m1 = fmaxf(m1, t1);

        // Shift rule (paper §4 equation; Algorithm 1): only rows whose maximum
        // repeats within eps change their shift.
        const float r_m = m1 * alpha;
        float m_new = r_m;
        if (MODE > 0 && (m1 - m2) <= args.eps_raw) {
          if (MODE == 1)
            m_new = r_m > 0.f ? args.beta * r_m : (r_m < 0.f ? 0.f : kEpsShift);
          else
            m_new = r_m + kEpsShift;
        }
        const bool changed = (j > 0) && (m_new != m_sh);
        const float corr = changed ? ex2_approx((m_sh - m_new) * kLog2e) : 1.f;
        l *= corr;
        m_sh = m_new;

        // The previous P.V must be complete before Obar is rescaled or the P
        // buffer is overwritten.
        if (j > 0) {
          if (!(ok = wait_warp(bar(L::bODone), (j - 1) & 1, ctl))) break;
          tc_fence_after();
        }
        if (__any_sync(0xFFFFFFFFu, changed)) {
#pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            uint32_t v[32];
            tmem_ld32(tO + lane_off + c, v);
            tmem_ld_wait32(v);
#pragma unroll
            for (int t = 0; t < 32; ++t) v[t] = __float_as_uint(__uint_as_float(v[t]) * corr);
            tmem_st32(tO + lane_off + c, v);
          }
          tmem_st_wait();
        }

        // Pass 2: Pbar = exp(S - m) in FP32 -> BF16 into the P buffer. l sums the
        // FP32 Pbar, so lse = m + ln l stays exact to FP32 and the backward pass's
        // P = exp(S - lse) is normalised.
        const float mlog2 = m_sh * kLog2e;
        const float thr = m1 - args.tau_raw;
        int cnt_tile = 0;
        float ls[2] = {0.f, 0.f};
#pragma unroll 1
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t v[32];
          tmem_ld32(tS + lane_off + c4 * 32, v);
          tmem_ld_wait32(v);
          if (c4 == 3) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::bSFree));
          }
          uint32_t pk[16];
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            float x0 = __uint_as_float(v[2 * t]);
            float x1 = __uint_as_float(v[2 * t + 1]);
            if (need_mask) {
              const int key = k0 + c4 * 32 + 2 * t;
              const bool vis0 = key < N && (!CAUSAL || key <= qrow);
              const bool vis1 = key + 1 < N && (!CAUSAL || key + 1 <= qrow);
              x0 = vis0 ? x0 : -INFINITY;
              x1 = vis1 ? x1 : -INFINITY;
            }
            if (COUNT) cnt_tile += (x0 >= thr) + (x1 >= thr);
            const float p0 = ex2_approx(fmaf(x0, sl2, -mlog2));
            const float p1 = ex2_approx(fmaf(x1, sl2, -mlog2));
            pk[t] = pack_bf16x2(p0, p1);
            ls[t & 1] += p0 + p1;
          }
          const uint32_t prow = sbase + L::kP + (c4 >> 1) * L::kPanelBytes;
#pragma unroll
          for (int qd = 0; qd < 4; ++qd)
            st_shared_v4(prow + sw128_offset(r, (c4 & 1) * 4 + qd), pk[4 * qd], pk[4 * qd + 1],
                         pk[4 * qd + 2], pk[4 * qd + 3]);
        }
        l += ls[0] + ls[1];
        if (COUNT) cnt = (m1 - m1_old > args.tau_raw) ? cnt_tile : cnt + cnt_tile;
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::bPFull));
      }

      // ---------------- epilogue ----------------
      if (ok && n_kt > 0) ok = wait_warp(bar(L::bODone), (n_kt - 1) & 1, ctl);
      if (ok) {
        tc_fence_after();
        const bool row_ok = qrow < N;
        const float inv_l = 1.f / l;
        __nv_bfloat16* orow =
            reinterpret_cast<__nv_bfloat16*>(args.o) + (static_cast<size_t>(bh) * N + qrow) * D;
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          uint32_t v[32];
          tmem_ld32(tO + lane_off + c, v);
          tmem_ld_wait32(v);
          uint32_t pk[16];
#pragma unroll
          for (int t = 0; t < 16; ++t)
            pk[t] = pack_bf16x2(__uint_as_float(v[2 * t]) * inv_l,
                                __uint_as_float(v[2 * t + 1]) * inv_l);
          if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
            for (int qd = 0; qd < 4; ++qd)
              dst[qd] = make_uint4(pk[4 * qd], pk[4 * qd + 1], pk[4 * qd + 2], pk[4 * qd + 3]);
          }
        }
        if (row_ok) args.lse[static_cast<size_t>(bh) * N + qrow] = m_sh + lg2_approx(l) * kLn2;
        if (COUNT) {
          const bool rep = (m1 - m2) <= args.eps_raw;
          // BF16(Pbar) == 1 under the final shift: entries within tau of m1,
          // unless the shift moved the maximum more than tau below zero.
          const float moved = m_sh - m1 * alpha;
          long long c_rep = row_ok && rep ? 1 : 0;
          long long c_one = row_ok && moved <= args.tau_raw * alpha ? cnt : 0;
          long long c_nf = row_ok && !(l > 0.f && l < INFINITY) ? 1 : 0;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            c_rep += __shfl_xor_sync(0xFFFFFFFFu, c_rep, o);
            c_one += __shfl_xor_sync(0xFFFFFFFFu, c_one, o);
            c_nf += __shfl_xor_sync(0xFFFFFFFFu, c_nf, o);
          }
          if (lane == 0 && args.counters) {
            if (c_rep) atomicAdd(reinterpret_cast<unsigned long long*>(args.counters + 0),
                                 static_cast<unsigned long long>(c_rep));
            if (c_one) atomicAdd(reinterpret_cast<unsigned long long*>(args.counters + 1),
                                 static_cast<unsigned long long>(c_one));
            if (c_nf) atomicAdd(reinterpret_cast<unsigned long long*>(args.counters + 2),
                                static_cast<unsigned long long>(c_nf));
          }
        }
      }
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

template <int D, int MODE, bool CAUSAL, bool COUNT>
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const FwdArgs& a, cudaStream_t stream) {
  using L = FwdLayout<D>;
  auto kern = attn_fwd_kernel<D, MODE, CAUSAL, COUNT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  if (e != cudaSuccess) return e;
  const int n_qt = (a.s.N + kTile - 1) / kTile;
  const dim3 grid(static_cast<unsigned>(n_qt) * a.s.B * a.s.Hq);
  kern<<<grid, kThreads, L::kBytes, stream>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

template <int D, int MODE>
cudaError_t dispatch_causal(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdArgs& a, cudaStream_t st) {
  const bool count = a.counters != nullptr;
  if (a.s.causal)
    return count ? launch_fwd_t<D, MODE, true, true>(tq, tk, tv, a, st)
                 : launch_fwd_t<D, MODE, true, false>(tq, tk, tv, a, st);
  return count ? launch_fwd_t<D, MODE, false, true>(tq, tk, tv, a, st)
               : launch_fwd_t<D, MODE, false, false>(tq, tk, tv, a, st);
}

template <int D>
cudaError_t dispatch_mode(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const FwdArgs& a, cudaStream_t st) {
  switch (a.fix_mode) {
    case 0: return dispatch_causal<D, 0>(tq, tk, tv, a, st);
    case 1: return dispatch_causal<D, 1>(tq, tk, tv, a, st);
    default: return dispatch_causal<D, 2>(tq, tk, tv, a, st);
  }
}

}  // namespace

cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdArgs& a, cudaStream_t stream) {
  if (a.s.d == 64) return dispatch_mode<64>(tq, tk, tv, a, stream);
  return dispatch_mode<128>(tq, tk, tv, a, stream);
}

}  // namespace pfa
