// Backward kernel. Per (key tile, batch, key/value head) one CTA loops over the
// query heads that share the key/value head and over the query tiles, with all
// five products on tcgen05 (FP32 accumulators in TMEM):
//   S^T  = K Q^T              P^T  = exp(alpha S^T - lse)      (recomputed)
//   dP^T = V dO^T             dS^T = alpha P^T o (dP^T - delta)
//   dV  += P^T dO             dK  += dS^T Q                    (stay in TMEM: no atomics)
//   dQ   = dS K               -> FP32 reduce-add into the dQ workspace
// which is the backward pass of the priors.kr post "BF16 플래시 어텐션은 왜 수천
// 스텝 뒤에 무너질까" (equations: dS = alpha P o (dP - delta), dQ = dS K) with the
// standard dK / dV products. The fix of paper §4 does not change the backward
// pass (priors.kr, the fix paragraph; bud-325 note, Results): P is recomputed
// from the saved lse whatever shift the forward pass used.
//
// 192 threads: warp 0 TMA producer, warp 1 TMEM owner + MMA issuer, warps 2..5
// one key row per thread for S^T / dP^T and one query row per thread for dQ.
// TMEM columns: S^T [0,128), dP^T [128,256), dV [256,256+d), dK [256+d,256+2d),
// dQ [384,448) for d = 64 and aliased onto S^T for d = 128.
#include "pfa_device.cuh"

namespace pfa {
namespace {

constexpr int kThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdLayout {
  static constexpr int kStages = (D == 64) ? 2 : 1;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kPanelBytes = kTile * 128;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQ = kV + kTileBytes;                // + stage * tile
  static constexpr int kDO = kQ + kStages * kTileBytes;     // + stage * tile
  static constexpr int kP = kDO + kStages * kTileBytes;     // P^T  [keys][queries] bf16
  static constexpr int kDS = kP + kTile * kTile * 2;        // dS^T [keys][queries] bf16
  static constexpr int kLse = kDS + kTile * kTile * 2;      // 2 slots x 128 floats (scaled by log2 e)
  static constexpr int kDelta = kLse + 2 * kTile * 4;       // 2 slots x 128 floats
  static constexpr int kBars = kDelta + 2 * kTile * 4;
  static constexpr int bKVFull = 0;
  static constexpr int bQFull = 1;                  // + stage
  static constexpr int bQEmpty = bQFull + kStages;  // + stage
  static constexpr int bSFull = bQEmpty + kStages;
  static constexpr int bDPFull = bSFull + 1;
  static constexpr int bSTFree = bDPFull + 1;
  static constexpr int bDPFree = bSTFree + 1;
  static constexpr int bPReady = bDPFree + 1;
  static constexpr int bDSReady = bPReady + 1;
  static constexpr int bPDSFree = bDSReady + 1;
  static constexpr int bDQFull = bPDSFree + 1;
  static constexpr int bDQFree = bDQFull + 1;
  static constexpr int bLse = bDQFree + 1;          // + slot (2): lse/delta staged
  static constexpr int bMMADone = bLse + 2;
  static constexpr int bDrain = bMMADone + 1;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kTmemSlot = kBars + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kBytes = kAbort + 4;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
  static constexpr uint32_t kColDQ = (D == 64) ? 384 : 0;
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const BwdArgs args) {
  using L = BwdLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const AttnShape& sh = args.s;
  const int N = sh.N;
  const int n_t = (N + kTile - 1) / kTile;
  const int BHkv = sh.B * sh.Hkv;
  const int kt = static_cast<int>(blockIdx.x / BHkv);  // kt = 0 has the most causal work
  const int bhk = blockIdx.x % BHkv;
  const int b = bhk / sh.Hkv;
  const int hk = bhk % sh.Hkv;
  const int group = sh.Hq / sh.Hkv;
  const int k0 = kt * kTile;
  const int qt_first = CAUSAL ? kt : 0;
  const int per_head = n_t - qt_first;
  const int n_iter = group * per_head;

  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  auto bar = [&](int i) { return sbase + L::kBars + 8u * static_cast<uint32_t>(i); };
  const WaitCtl ctl{abort_flag, args.err};
  // iteration -> (query head, query tile)
  auto iter_head = [&](int i) { return b * sh.Hq + hk * group + i / per_head; };
  auto iter_q0 = [&](int i) { return (qt_first + i % per_head) * kTile; };

  if (threadIdx.x == 0) {
    *abort_flag = (sbase & 1023u) ? 1 : 0;
    if (sbase & 1023u) atomicOr(args.err, PFA_DEVERR_SMEM_ALIGN);
    mbar_init(bar(L::bKVFull), 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::bQFull + s), 1);
      mbar_init(bar(L::bQEmpty + s), 1);
    }
    mbar_init(bar(L::bSFull), 1);
    mbar_init(bar(L::bDPFull), 1);
    mbar_init(bar(L::bSTFree), 4);
    mbar_init(bar(L::bDPFree), 4);
    mbar_init(bar(L::bPReady), 4);
    mbar_init(bar(L::bDSReady), 4);
    mbar_init(bar(L::bPDSFree), 1);
    mbar_init(bar(L::bDQFull), 1);
    mbar_init(bar(L::bDQFree), 4);
    mbar_init(bar(L::bLse + 0), 128);
    mbar_init(bar(L::bLse + 1), 128);
    mbar_init(bar(L::bMMADone), 1);
    mbar_init(bar(L::bDrain), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (*abort_flag == 0) {
    if (warp == 0) {
      // ---------------- TMA producer ----------------
      if (lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmdO);
        mbar_arrive_expect_tx(bar(L::bKVFull), 2 * L::kTileBytes);
        for (int p = 0; p < D / 64; ++p) {
          tma_load_3d(sbase + L::kK + p * L::kPanelBytes, &tmK, bar(L::bKVFull), p * 64, k0, bhk);
          tma_load_3d(sbase + L::kV + p * L::kPanelBytes, &tmV, bar(L::bKVFull), p * 64, k0, bhk);
        }
        int issued = 0;
        for (int i = 0; i < n_iter; ++i) {
          const int s = i % L::kStages;
          const uint32_t ph = (i / L::kStages) & 1;
          if (!wait_thread(bar(L::bQEmpty + s), ph ^ 1, ctl)) break;
          issued = i + 1;
          const int bhq = iter_head(i);
          const int q0 = iter_q0(i);
          mbar_arrive_expect_tx(bar(L::bQFull + s), 2 * L::kTileBytes);
          for (int p = 0; p < D / 64; ++p) {
            tma_load_3d(sbase + L::kQ + s * L::kTileBytes + p * L::kPanelBytes, &tmQ,
                        bar(L::bQFull + s), p * 64, q0, bhq);
            tma_load_3d(sbase + L::kDO + s * L::kTileBytes + p * L::kPanelBytes, &tmdO,
                        bar(L::bQFull + s), p * 64, q0, bhq);
          }
        }
        wait_drain(bar(L::bKVFull), 0, args.err);
        for (int i = issued > L::kStages ? issued - L::kStages : 0; i < issued; ++i)
          wait_drain(bar(L::bQFull + i % L::kStages), (i / L::kStages) & 1, args.err);
      }
    } else if (warp == 1) {
      // ---------------- MMA issuer ----------------
      if (lane == 0) {
        constexpr uint32_t idKK = idesc_bf16(128, 128, false, false);  // S^T, dP^T
        constexpr uint32_t idKM = idesc_bf16(128, D, false, true);     // dV, dK: B MN-major
        constexpr uint32_t idMM = idesc_bf16(128, D, true, true);      // dQ: A and B MN-major
        const uint32_t tS = tmem + L::kColS, tDP = tmem + L::kColDP, tDV = tmem + L::kColDV,
                       tDK = tmem + L::kColDK, tDQ = tmem + L::kColDQ;
        bool ok = wait_thread(bar(L::bKVFull), 0, ctl);
        for (int i = 0; ok && i < n_iter; ++i) {
          const int s = i % L::kStages;
          const uint32_t ph = (i / L::kStages) & 1;
          const uint32_t sQ = sbase + L::kQ + s * L::kTileBytes;
          const uint32_t sDO = sbase + L::kDO + s * L::kTileBytes;
          if (!(ok = wait_thread(bar(L::bQFull + s), ph, ctl))) break;
          if (i > 0) {
            if (!(ok = wait_thread(bar(L::bSTFree), (i - 1) & 1, ctl))) break;
            if (D == 128 && !(ok = wait_thread(bar(L::bDQFree), (i - 1) & 1, ctl))) break;
          }
          tc_fence_after();
          // S^T = K Q^T : A = K [keys x d] K-major, B = Q [queries x d] K-major.
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
            umma_bf16(tS, sdesc_sw128(sbase + L::kK + koff, 16, 1024), sdesc_sw128(sQ + koff, 16, 1024),
                      idKK, kk > 0);
          }
          umma_commit(bar(L::bSFull));
          if (i > 0 && !(ok = wait_thread(bar(L::bDPFree), (i - 1) & 1, ctl))) break;
          tc_fence_after();
          // dP^T = V dO^T
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
            umma_bf16(tDP, sdesc_sw128(sbase + L::kV + koff, 16, 1024),
                      sdesc_sw128(sDO + koff, 16, 1024), idKK, kk > 0);
          }
          umma_commit(bar(L::bDPFull));
          // dV += P^T dO : A = P^T [keys x queries] K-major, B = dO viewed [d x queries] MN-major.
          if (!(ok = wait_thread(bar(L::bPReady), i & 1, ctl))) break;
          tc_fence_after();
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint32_t aoff = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
            umma_bf16(tDV, sdesc_sw128(sbase + L::kP + aoff, 16, 1024),
                      sdesc_sw128(sDO + kk * 2048, L::kPanelBytes, 1024), idKM,
                      (i > 0 || kk > 0) ? 1u : 0u);
          }
          // dK += dS^T Q ; dQ = dS K (A = dS^T buffer read MN-major, B = K MN-major).
          if (!(ok = wait_thread(bar(L::bDSReady), i & 1, ctl))) break;
          tc_fence_after();
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint32_t aoff = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
            umma_bf16(tDK, sdesc_sw128(sbase + L::kDS + aoff, 16, 1024),
                      sdesc_sw128(sQ + kk * 2048, L::kPanelBytes, 1024), idKM,
                      (i > 0 || kk > 0) ? 1u : 0u);
          }
          if (D == 64 && i > 0 && !(ok = wait_thread(bar(L::bDQFree), (i - 1) & 1, ctl))) break;
          tc_fence_after();
          for (int kk = 0; kk < kTile / 16; ++kk) {
            umma_bf16(tDQ, sdesc_sw128(sbase + L::kDS + kk * 2048, L::kPanelBytes, 1024),
                      sdesc_sw128(sbase + L::kK + kk * 2048, L::kPanelBytes, 1024), idMM, kk > 0);
          }
          umma_commit(bar(L::bDQFull));
          umma_commit(bar(L::bQEmpty + s));
          umma_commit(bar(L::bPDSFree));
        }
        umma_commit(bar(L::bMMADone));
        umma_commit(bar(L::bDrain));
        wait_drain(bar(L::bDrain), 0, args.err);
      }
    } else {
      // ---------------- compute warps ----------------
      const uint32_t quarter = warp & 3;
      const int r = quarter * 32 + lane;  // TMEM lane: key row for S^T/dP^T, query row for dQ
      const int ct = threadIdx.x - 64;    // 0..127
      const uint32_t lane_off = (quarter * 32u) << 16;
      const int key = k0 + r;
      const float sl2 = sh.scale_log2;
      const float alpha = sh.scale;
      const float* lse_s = reinterpret_cast<const float*>(smem + L::kLse);
      const float* dl_s = reinterpret_cast<const float*>(smem + L::kDelta);
      bool ok = true;

      for (int i = 0; ok && i < n_iter; ++i) {
        const int bhq = iter_head(i);
        const int q0 = iter_q0(i);
        const int slot = i & 1;
        {
          const int q = q0 + ct;
          float* lw = reinterpret_cast<float*>(smem + L::kLse) + slot * kTile;
          float* dw = reinterpret_cast<float*>(smem + L::kDelta) + slot * kTile;
          lw[ct] = (q < N) ? args.lse[static_cast<size_t>(bhq) * N + q] * kLog2e : INFINITY;
          dw[ct] = (q < N) ? args.delta[static_cast<size_t>(bhq) * N + q] : 0.f;
        }
        // All 128 compute threads have staged their value (and, by the previous
        // iteration's wait, finished reading this slot two iterations ago).
        mbar_arrive(bar(L::bLse + slot));
        if (!(ok = wait_warp(bar(L::bLse + slot), (i >> 1) & 1, ctl))) break;
        const float* lrow = lse_s + slot * kTile;
        const float* drow = dl_s + slot * kTile;
        const bool need_mask = (CAUSAL && q0 == k0) || (k0 + kTile > N);

        // P^T row: p[c] = exp(alpha s - lse_c), query c visible to this key.
        if (!(ok = wait_warp(bar(L::bSFull), i & 1, ctl))) break;
        tc_fence_after();
        float p[kTile];
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t v[32];
          tmem_ld32(tmem + L::kColS + lane_off + c4 * 32, v);
          tmem_ld_wait32(v);
#pragma unroll
          for (int t = 0; t < 32; ++t) {
            const int c = c4 * 32 + t;
            float pv = ex2_approx(fmaf(__uint_as_float(v[t]), sl2, -lrow[c]));
            if (need_mask) {
              const bool vis = key < N && (!CAUSAL || q0 + c >= key);
              pv = vis ? pv : 0.f;
            }
            p[c] = pv;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::bSTFree));

        if (i > 0 && !(ok = wait_warp(bar(L::bPDSFree), (i - 1) & 1, ctl))) break;
        // P^T (BF16) into the swizzled [keys][queries] buffer.
#pragma unroll
        for (int c8 = 0; c8 < kTile / 8; ++c8) {
          const uint32_t addr = sbase + L::kP + (c8 >> 3) * L::kPanelBytes + sw128_offset(r, c8 & 7);
          st_shared_v4(addr, pack_bf16x2(p[8 * c8 + 0], p[8 * c8 + 1]),
                       pack_bf16x2(p[8 * c8 + 2], p[8 * c8 + 3]),
                       pack_bf16x2(p[8 * c8 + 4], p[8 * c8 + 5]),
                       pack_bf16x2(p[8 * c8 + 6], p[8 * c8 + 7]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::bPReady));

        // dS^T = alpha P^T o (dP^T - delta)
        if (!(ok = wait_warp(bar(L::bDPFull), i & 1, ctl))) break;
        tc_fence_after();
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t v[32];
          tmem_ld32(tmem + L::kColDP + lane_off + c4 * 32, v);
          tmem_ld_wait32(v);
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {
            uint32_t w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int c = c4 * 32 + c8 * 8 + 2 * u;
              const float d0 = alpha * p[c] * (__uint_as_float(v[c8 * 8 + 2 * u]) - drow[c]);
              const float d1 =
                  alpha * p[c + 1] * (__uint_as_float(v[c8 * 8 + 2 * u + 1]) - drow[c + 1]);
              w[u] = pack_bf16x2(d0, d1);
            }
            const int chunk = c4 * 4 + c8;  // 16-byte chunk index over 128 queries
            const uint32_t addr =
                sbase + L::kDS + (chunk >> 3) * L::kPanelBytes + sw128_offset(r, chunk & 7);
            st_shared_v4(addr, w[0], w[1], w[2], w[3]);
          }
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(L::bDPFree));
          mbar_arrive(bar(L::bDSReady));
        }

        // dQ tile -> FP32 reduce-add into the workspace (this thread = query row q0 + r).
        if (!(ok = wait_warp(bar(L::bDQFull), i & 1, ctl))) break;
        tc_fence_after();
        const int q = q0 + r;
        float* dq_row = args.dq_accum + (static_cast<size_t>(bhq) * N + q) * D;
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          uint32_t v[32];
          tmem_ld32(tmem + L::kColDQ + lane_off + c, v);
          tmem_ld_wait32(v);
          if (q < N) {
#pragma unroll
            for (int u = 0; u < 8; ++u)
              atomicAdd(reinterpret_cast<float4*>(dq_row + c) + u,
                        make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]),
                                    __uint_as_float(v[4 * u + 2]), __uint_as_float(v[4 * u + 3])));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::bDQFree));
      }

      // ---------------- epilogue: dK, dV rows of this key tile ----------------
      if (ok) ok = wait_warp(bar(L::bMMADone), 0, ctl);
      if (ok) {
        tc_fence_after();
        const size_t row = static_cast<size_t>(bhk) * N + key;
#pragma unroll 1
        for (int which = 0; which < 2; ++which) {
          const uint32_t col = which == 0 ? L::kColDK : L::kColDV;
          __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(which == 0 ? args.dk : args.dv) + row * D;
#pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + col + lane_off + c, v);
            tmem_ld_wait32(v);
            if (key < N) {
              uint4* dst = reinterpret_cast<uint4*>(out + c);
#pragma unroll
              for (int u = 0; u < 4; ++u)
                dst[u] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * u + 0]), __uint_as_float(v[8 * u + 1])),
                                    pack_bf16x2(__uint_as_float(v[8 * u + 2]), __uint_as_float(v[8 * u + 3])),
                                    pack_bf16x2(__uint_as_float(v[8 * u + 4]), __uint_as_float(v[8 * u + 5])),
                                    pack_bf16x2(__uint_as_float(v[8 * u + 6]), __uint_as_float(v[8 * u + 7])));
            }
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
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL>
cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t stream) {
  using L = BwdLayout<D>;
  auto kern = attn_bwd_kernel<D, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  if (e != cudaSuccess) return e;
  const int n_t = (a.s.N + kTile - 1) / kTile;
  const dim3 grid(static_cast<unsigned>(n_t) * a.s.B * a.s.Hkv);
  kern<<<grid, kThreads, L::kBytes, stream>>>(tq, tk, tv, tdo, a);
  return cudaGetLastError();
}

__global__ void convert_dq_kernel(const float4* __restrict__ src, uint2* __restrict__ dst, long long n4) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 x = src[i];
    dst[i] = make_uint2(pack_bf16x2(x.x, x.y), pack_bf16x2(x.z, x.w));
  }
}

}  // namespace

cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t stream) {
  if (a.s.d == 64)
    return a.s.causal ? launch_bwd_t<64, true>(tq, tk, tv, tdo, a, stream)
                      : launch_bwd_t<64, false>(tq, tk, tv, tdo, a, stream);
  return a.s.causal ? launch_bwd_t<128, true>(tq, tk, tv, tdo, a, stream)
                    : launch_bwd_t<128, false>(tq, tk, tv, tdo, a, stream);
}

// dQ = BF16(dQ workspace); n is a multiple of 4 (d is 64 or 128).
cudaError_t launch_convert_dq(const float* dq_accum, void* dq, long long n, cudaStream_t stream) {
  const long long n4 = n / 4;
  const int threads = 256;
  long long blocks = (n4 + threads - 1) / threads;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  convert_dq_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      reinterpret_cast<const float4*>(dq_accum), reinterpret_cast<uint2*>(dq), n4);
  return cudaGetLastError();
}

}  // namespace pfa
