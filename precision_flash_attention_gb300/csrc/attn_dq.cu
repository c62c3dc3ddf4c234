// dQ by a query-outer pass: dQ = dS K with dS = alpha P o (dP - delta), the dQ
// equation of the priors.kr post "BF16 플래시 어텐션은 왜 수천 스텝 뒤에 무너질까"
// (equations, paper §3.3.1), computed one 128-row query tile at a time over the
// key tiles in order. Each dQ row is summed by one CTA, in one fixed order, into
// an FP32 accumulator in TMEM, so repeated calls give identical bits (the
// key-outer backward kernel adds per-key-tile partial sums into a shared FP32
// buffer in arrival order instead).
//
// SPLIT feeds the dQ product a two-term BF16 expansion of dS: hi = bf16(dS) and
// lo = bf16(dS - hi), two products into the same accumulator, about 16
// significant bits of dS instead of 8. Where several keys share a large feature
// and their dS nearly cancel along it (a sink key copied into other positions),
// the rounding of a single BF16 dS is what separates dQ from its exact value.
//
// CTA = one (batch, query head, 128-row query tile), heaviest causal tiles first.
// 320 threads: warp 0 TMA producer, warp 1 TMEM owner and MMA issuer, warps 2..9
// compute. Each 128-key tile is processed as two 64-key halves u = 2 j, 2 j + 1,
// in two TMEM buffers b = u % 2 at [128 b, 128 b + 128): S_u = Q K_u^T in the
// first 64 columns, dP_u = dO V_u^T in the next 64; dQ sits in [256, 256 + d).
// Compute warp w handles TMEM lane quarter w % 4 (32 query rows) and the 32 keys
// [32 c, 32 c + 32) of each half, c = (w - 2) / 4, so each SM sub-partition runs
// two compute warps. dS (BF16, two keys per 32-bit column) is written over the S
// columns the warp has read: its 32 keys occupy [32 c, 32 c + 32) of the half's
// S, hi in the first 16 columns and lo in the next 16, so key step kk (16 keys) of
// the dQ product reads hi at 32 (kk / 2) + 8 (kk % 2).
// Tensor-core order: S_0, dP_0, S_1, dP_1, then per half u: dQ_u, S_(u+2), dP_(u+2).
// The compute warps form dS_(u+1) while the tensor core runs dQ_u and S_(u+2),
// and in-order execution keeps S_(u+2) (same buffer) from overwriting dS_u before
// dQ_u has read it.
#include "pfa_device.cuh"

namespace pfa {
namespace {

constexpr int kThreads = 320;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kHalf = kTile / 2;   // keys of one half-tile

template <int D>
struct DqLayout {
  static constexpr int kStages = 2;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kPanelBytes = kTile * 128;
  static constexpr int kQ = 0;
  static constexpr int kDO = kQ + kTileBytes;
  static constexpr int kK = kDO + kTileBytes;           // + stage * tile
  static constexpr int kV = kK + kStages * kTileBytes;  // + stage * tile
  static constexpr int kBars = kV + kStages * kTileBytes;
  static constexpr int bQFull = 0;
  static constexpr int bKVFull = 1;                     // + stage
  static constexpr int bKVEmpty = bKVFull + kStages;    // + stage
  static constexpr int bSFull = bKVEmpty + kStages;     // + buffer: S_u and dP_u are in TMEM
  static constexpr int bDSReady = bSFull + 2;           // + buffer: the compute warps wrote dS_u
  static constexpr int bDQDone = bDSReady + 2;          // the last dQ product completed
  static constexpr int bDrain = bDQDone + 1;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kTmemSlot = kBars + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kBytes = kAbort + 4;
  static constexpr uint32_t kColDQ = 256;
  static_assert(kColDQ + D <= 512, "TMEM columns");
  static_assert(kBytes <= 232448, "shared memory budget");
};

// Column of the BF16 dS hi values of key step kk (16 keys) within a half's S
// columns; lo sits 16 columns on.
__device__ __forceinline__ uint32_t ds_col(int kk) {
  return 32u * static_cast<uint32_t>(kk >> 1) + 8u * static_cast<uint32_t>(kk & 1);
}

template <int D, bool CAUSAL, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    attn_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                   const DqArgs args) {
  using L = DqLayout<D>;
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
  const int n_u = 2 * n_kt;   // half-tiles

  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  auto bar = [&](int i) { return sbase + L::kBars + 8u * static_cast<uint32_t>(i); };
  const WaitCtl ctl{abort_flag, args.err, args.err_site, sbase, 5u};

  if (threadIdx.x == 0) {
    *abort_flag = (sbase & 1023u) ? 1 : 0;
    if (sbase & 1023u) atomicOr(args.err, PFA_DEVERR_SMEM_ALIGN);
    mbar_init(bar(L::bQFull), 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::bKVFull + s), 1);
      mbar_init(bar(L::bKVEmpty + s), 1);
    }
    for (int u = 0; u < 2; ++u) {
      mbar_init(bar(L::bSFull + u), 1);
      mbar_init(bar(L::bDSReady + u), 8);
    }
    mbar_init(bar(L::bDQDone), 1);
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
  // Setup done: let the next kernel on the stream be scheduled as CTAs leave, and
  // order every global access after the kernel before this one.
  grid_launch_dependents();
  grid_dependency_wait();

  if (*abort_flag == 0) {
    if (warp == 0) {
      // ---------------- TMA producer (whole warp, one elected lane issues) ----------------
      mbar_arrive_expect_tx_warp(bar(L::bQFull), 2 * L::kTileBytes);
      for (int p = 0; p < D / 64; ++p) {
        tma_load_3d_warp(sbase + L::kQ + p * L::kPanelBytes, &tmQ, bar(L::bQFull), p * 64, q0, bh);
        tma_load_3d_warp(sbase + L::kDO + p * L::kPanelBytes, &tmdO, bar(L::bQFull), p * 64, q0, bh);
      }
      int issued = 0;
      for (int j = 0; j < n_kt; ++j) {
        const int s = j % L::kStages;
        if (!wait_warp(bar(L::bKVEmpty + s), ((j / L::kStages) & 1) ^ 1, ctl)) break;
        issued = j + 1;
        mbar_arrive_expect_tx_warp(bar(L::bKVFull + s), 2 * L::kTileBytes);
        for (int p = 0; p < D / 64; ++p) {
          tma_load_3d_warp(sbase + L::kK + s * L::kTileBytes + p * L::kPanelBytes, &tmK,
                           bar(L::bKVFull + s), p * 64, j * kTile, bh_kv);
          tma_load_3d_warp(sbase + L::kV + s * L::kTileBytes + p * L::kPanelBytes, &tmV,
                           bar(L::bKVFull + s), p * 64, j * kTile, bh_kv);
        }
      }
      // Every issued copy has landed before shared memory is released.
      wait_drain(bar(L::bQFull), 0, ctl);
      for (int j = issued > L::kStages ? issued - L::kStages : 0; j < issued; ++j)
        wait_drain(bar(L::bKVFull + j % L::kStages), (j / L::kStages) & 1, ctl);
    } else if (warp == 1) {
      // ---------------- MMA issuer (whole warp, one elected lane issues) ----------------
      constexpr uint32_t idS = idesc_bf16(128, kHalf, false, false);  // S_u, dP_u: N = 64 keys
      constexpr uint32_t idDQ = idesc_bf16(128, D, false, true);      // dQ: A = dS in TMEM, B = K MN-major
      // S_u = Q K_u^T and dP_u = dO V_u^T into buffer u % 2; K_u, V_u are rows
      // [64 (u % 2), 64 (u % 2) + 64) of the key tile in stage (u / 2) % 2.
      auto issue_sdp = [&](int u) {
        const uint32_t tb = tmem + 128u * static_cast<uint32_t>(u & 1);
        const int s = (u >> 1) % L::kStages;
        const uint32_t hoff = static_cast<uint32_t>(u & 1) * kHalf * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
          umma_bf16_warp(tb, sdesc_sw128(sbase + L::kQ + koff, 16, 1024),
                         sdesc_sw128(sbase + L::kK + s * L::kTileBytes + hoff + koff, 16, 1024), idS, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
          umma_bf16_warp(tb + kHalf, sdesc_sw128(sbase + L::kDO + koff, 16, 1024),
                         sdesc_sw128(sbase + L::kV + s * L::kTileBytes + hoff + koff, 16, 1024), idS, kk > 0);
        }
        umma_commit_warp(bar(L::bSFull + (u & 1)));
      };
      // dQ += dS_u K_u: hi, then lo into the same accumulator.
      auto issue_dq = [&](int u) {
        const uint32_t tb = tmem + 128u * static_cast<uint32_t>(u & 1);
        const int s = (u >> 1) % L::kStages;
        const uint32_t sK = sbase + L::kK + s * L::kTileBytes;
        const int h4 = 4 * (u & 1);   // the half's first key step within the tile
#pragma unroll
        for (int kk = 0; kk < kHalf / 16; ++kk)
          umma_bf16_tmem_a_warp(tmem + L::kColDQ, tb + ds_col(kk),
                                sdesc_sw128(sK + (h4 + kk) * 2048, L::kPanelBytes, 1024), idDQ,
                                (u > 0 || kk > 0) ? 1u : 0u);
        if constexpr (SPLIT) {
#pragma unroll
          for (int kk = 0; kk < kHalf / 16; ++kk)
            umma_bf16_tmem_a_warp(tmem + L::kColDQ, tb + ds_col(kk) + 16u,
                                  sdesc_sw128(sK + (h4 + kk) * 2048, L::kPanelBytes, 1024), idDQ, 1u);
        }
        // The second half's product is the last reader of the tile's K and V.
        if (u & 1) umma_commit_warp(bar(L::bKVEmpty + s));
      };
      // Half u needs its key tile (u / 2) in shared memory; the first half waits.
      auto tile_ready = [&](int u) {
        if (u & 1) return true;
        const int j = u >> 1;
        return wait_warp(bar(L::bKVFull + j % L::kStages), (j / L::kStages) & 1, ctl);
      };
      bool ok = wait_warp(bar(L::bQFull), 0, ctl);
      for (int u = 0; ok && u < 2; ++u) {
        if (!(ok = tile_ready(u))) break;
        tc_fence_after();
        issue_sdp(u);
      }
      for (int u = 0; ok && u < n_u; ++u) {
        if (!(ok = wait_warp(bar(L::bDSReady + (u & 1)), (u >> 1) & 1, ctl))) break;
        tc_fence_after();
        issue_dq(u);
        if (u + 2 < n_u) {
          if (!(ok = tile_ready(u + 2))) break;
          tc_fence_after();
          issue_sdp(u + 2);
        }
      }
      if (ok) umma_commit_warp(bar(L::bDQDone));
      // No MMA may still read shared memory or write TMEM at teardown.
      umma_commit_warp(bar(L::bDrain));
      wait_drain(bar(L::bDrain), 0, ctl);
    } else {
      // ---------------- compute warps ----------------
      const uint32_t quarter = warp & 3;
      const int c = (warp - 2) >> 2;             // keys [32 c, 32 c + 32) of each half
      const int r = quarter * 32 + lane;         // query row within the tile == TMEM lane
      const int qrow = q0 + r;
      const uint32_t lane_off = (quarter * 32u) << 16;
      const bool row_ok = qrow < N;
      const size_t rowi = static_cast<size_t>(bh) * N + qrow;
      // -lse (log2 units) and -delta of this row; rows past N take no part.
      const float nlse2 = row_ok ? -args.lse[rowi] * kLog2e : -INFINITY;
      const float ndelta = row_ok ? -args.delta[rowi] : 0.f;
      const float sl2 = sh.scale_log2;
      bool ok = true;
      for (int u = 0; u < n_u; ++u) {
        const int k0 = (u >> 1) * kTile + (u & 1) * kHalf + 32 * c;   // this warp's first key
        const bool need_mask = (CAUSAL && k0 + 32 > q0) || (k0 + 32 > N);
        const uint32_t tb = tmem + 128u * static_cast<uint32_t>(u & 1) + lane_off + 32u * c;
        if (!(ok = wait_warp(bar(L::bSFull + (u & 1)), (u >> 1) & 1, ctl))) break;
        tc_fence_after();
        uint32_t sv[32], pv[32];
        tmem_ld32(tb, sv);
        tmem_ld32(tb + kHalf, pv);
        tmem_ld_wait32(sv);
        tmem_ld_wait32(pv);
        float ds[32];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float y0, y1;
          fma2(y0, y1, __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]), sl2, nlse2);
          float p0 = ex2_approx(y0), p1 = ex2_approx(y1);
          if (need_mask) {
            const int key = k0 + e;
            if (!(key < N && (!CAUSAL || key <= qrow))) p0 = 0.f;
            if (!(key + 1 < N && (!CAUSAL || key + 1 <= qrow))) p1 = 0.f;
          }
          float t0 = __uint_as_float(pv[e]), t1 = __uint_as_float(pv[e + 1]);
          add2(t0, t1, ndelta, ndelta);
          mul2v(ds[e], ds[e + 1], t0, t1, p0, p1);
        }
        uint32_t hi[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) hi[e] = pack_bf16x2(ds[2 * e], ds[2 * e + 1]);
        tmem_st16(tb, hi);
        if constexpr (SPLIT) {
          uint32_t lo[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            lo[e] = pack_bf16x2(ds[2 * e] - bf16lo_to_f32(hi[e]), ds[2 * e + 1] - bf16hi_to_f32(hi[e]));
          tmem_st16(tb + 16, lo);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::bDSReady + (u & 1)));
      }
      // ---------------- epilogue: dQ = alpha (sum of dS K) -> BF16 ----------------
      if (ok) ok = wait_warp(bar(L::bDQDone), 0, ctl);
      if (ok) {
        tc_fence_after();
        constexpr int kCols = D / 2;   // this warp's dQ columns [kCols c, kCols c + kCols)
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(args.dq) + rowi * D + kCols * c;
#pragma unroll 1
        for (int cc = 0; cc < kCols; cc += 32) {
          uint32_t v[32];
          tmem_ld32(tmem + L::kColDQ + lane_off + kCols * c + cc, v);
          tmem_ld_wait32(v);
          if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(out + cc);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              auto f = [&](int e) { return sh.scale * __uint_as_float(v[8 * q + e]); };
              dst[q] = make_uint4(pack_bf16x2(f(0), f(1)), pack_bf16x2(f(2), f(3)), pack_bf16x2(f(4), f(5)),
                                  pack_bf16x2(f(6), f(7)));
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

template <int D, bool CAUSAL, bool SPLIT>
cudaError_t launch_dq_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const CUtensorMap& tdo, const DqArgs& a, cudaStream_t stream) {
  using L = DqLayout<D>;
  auto kern = attn_dq_kernel<D, CAUSAL, SPLIT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  if (e != cudaSuccess) return e;
  const int n_t = (a.s.N + kTile - 1) / kTile;
  const dim3 grid(static_cast<unsigned>(n_t) * a.s.B * a.s.Hq);
  return launch_pdl(kern, grid, dim3(kThreads), L::kBytes, stream, tq, tk, tv, tdo, a);
}

template <int D, bool CAUSAL>
cudaError_t dispatch_split(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tdo, const DqArgs& a, cudaStream_t stream) {
  return a.split ? launch_dq_t<D, CAUSAL, true>(tq, tk, tv, tdo, a, stream)
                 : launch_dq_t<D, CAUSAL, false>(tq, tk, tv, tdo, a, stream);
}

}  // namespace

cudaError_t launch_dq(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      const CUtensorMap& tdo, const DqArgs& a, cudaStream_t stream) {
  if (a.s.d == 64)
    return a.s.causal ? dispatch_split<64, true>(tq, tk, tv, tdo, a, stream)
                      : dispatch_split<64, false>(tq, tk, tv, tdo, a, stream);
  return a.s.causal ? dispatch_split<128, true>(tq, tk, tv, tdo, a, stream)
                    : dispatch_split<128, false>(tq, tk, tv, tdo, a, stream);
}

}  // namespace pfa
