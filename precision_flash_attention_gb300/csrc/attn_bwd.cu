// Backward kernel. Per (key tile, batch, key/value head) one CTA loops over the
// query heads that share the key/value head and over the query tiles, with all
// five products on tcgen05 (FP32 accumulators in TMEM):
//   S^T  = K Q^T              P^T  = exp(alpha S^T - lse)      (recomputed)
//   dP^T = V dO^T             dS^T = P^T o (dP^T - delta)      (alpha applied at the end)
//   dV  += P^T dO             dK  += dS^T Q                    (stay in TMEM: no atomics)
//   dQ   = dS K               -> alpha dQ reduce-added into the FP32 workspace
// which is the backward pass of the priors.kr post "BF16 플래시 어텐션은 왜 수천
// 스텝 뒤에 무너질까" (equations: dS = alpha P o (dP - delta), dQ = dS K) with the
// standard dK / dV products. The fix of paper §4 does not change the backward
// pass (priors.kr, the fix paragraph; bud-325 note, Results): P is recomputed
// from the saved lse whatever shift the forward pass used.
//
// 384 threads in three warpgroups: warp 0 TMA producer, warp 1 TMEM owner and
// tcgen05.mma issuer, warps 2-3 idle; warps 4-11 compute. Compute warp w owns
// TMEM lane quarter w % 4 (32 keys) and query half (w - 4) / 4 (64 queries).
// P^T and dS^T are cast to BF16 and written back into TMEM over S^T and dP^T
// (each query half over its own input columns), where they are the A operands of
// dV and dK; dS^T also goes to a 128B-swizzled
// shared buffer that the dQ product reads as its (M = queries) A operand.
// TMEM columns: S^T [0,128), dP^T [128,256), dV [256,256+d), dK [256+d,256+2d),
// dQ [384,448) for d = 64 and over dP^T [128,256) for d = 128.
// Tensor-core order per query tile: S^T, dP^T, dV, dK, dQ; the P phase of the
// compute warps overlaps dP^T and the dS phase overlaps dV.
#include "pfa_device.cuh"
#include "pfa_trace.cuh"

PFA_TRACE_BUFFER(g_pfa_bwd_trace);
#define PFA_BWD_TRACE(slot, ev, j) PFA_TRACE_EVENT(g_pfa_bwd_trace, slot, ev, j)

namespace pfa {
namespace {

constexpr int kThreads = 384;
constexpr float kLog2e = 1.4426950408889634f;

// P^T and dS^T (BF16, two per 32-bit column) are written by each query half into
// the first 32 columns of that half's own 64 FP32 input columns, so one half never
// overwrites values the other half has yet to load. Query step kk (16 queries,
// 8 columns) therefore sits at column 8 kk for kk < 4 and 32 + 8 kk after.
__host__ __device__ constexpr uint32_t packed_col(int kk) {
  return 8u * static_cast<uint32_t>(kk) + (kk >= 4 ? 32u : 0u);
}

template <int D>
struct BwdLayout {
  // Query-side stages: the next tile's Q / dO must land within about one
  // iteration, so d = 64 keeps three in flight; d = 128 fits two.
  static constexpr int kStages = (D == 64) ? 3 : 2;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kPanelBytes = kTile * 128;
  // dQ leaves through a TMA reduce-add from a per-warp staging box (d = 64:
  // 32 rows x 32 FP32 columns, 4 KB per compute warp); d = 128 has no room left
  // for the staging and reduce-adds with vector atomics.
  static constexpr bool kTmaDQ = (D == 64);
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQ = kV + kTileBytes;                // + stage * tile
  static constexpr int kDO = kQ + kStages * kTileBytes;     // + stage * tile
  static constexpr int kDS = kDO + kStages * kTileBytes;    // dS^T [keys][queries] bf16, 2 panels
  static constexpr int kDQStage = kDS + kTile * kTile * 2;  // 8 warps x 4 KB (d = 64 only)
  static constexpr int kLse = kDQStage + (kTmaDQ ? 8 * 4096 : 0);  // [slot 2][half 2][lse 64 | delta 64]
  static constexpr int kBars = kLse + 2 * 2 * 128 * 4;
  static constexpr int bKVFull = 0;
  static constexpr int bQFull = 1;                  // + stage
  static constexpr int bQEmpty = bQFull + kStages;  // + stage
  static constexpr int bSFull = bQEmpty + kStages;
  static constexpr int bDPFull = bSFull + 1;
  static constexpr int bPReady = bDPFull + 1;
  static constexpr int bDSReady = bPReady + 1;
  static constexpr int bDQFull = bDSReady + 1;
  static constexpr int bDQFree = bDQFull + 1;
  static constexpr int bLse = bDQFree + 1;          // + 2 * half + slot
  static constexpr int bMMADone = bLse + 4;
  static constexpr int bDrain = bMMADone + 1;
  static constexpr int bRegs = bDrain + 1;          // the compute warps hold their registers
  static constexpr int kNumBars = bRegs + 1;
  static constexpr int kTmemSlot = kBars + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kBytes = kAbort + 4;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
  static constexpr uint32_t kColDQ = (D == 64) ? 384 : 128;
  static constexpr bool kDQAliasesDP = (D != 64);
  static_assert(kDQStage % 1024 == 0, "swizzled staging boxes need 1024-byte alignment");
  static_assert(kBytes <= 232448, "shared memory budget");
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const __grid_constant__ CUtensorMap tmdQ, const BwdArgs args) {
  using L = BwdLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  PFA_TRACE_DECL();

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
  const WaitCtl ctl{abort_flag, args.err, args.err_site, sbase, 2u};
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
    mbar_init(bar(L::bPReady), 8);
    mbar_init(bar(L::bDSReady), 8);
    mbar_init(bar(L::bDQFull), 1);
    mbar_init(bar(L::bDQFree), 8);
    for (int x = 0; x < 4; ++x) mbar_init(bar(L::bLse + x), 4);
    mbar_init(bar(L::bMMADone), 1);
    mbar_init(bar(L::bDrain), 1);
    mbar_init(bar(L::bRegs), 8);
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
  // Register split per warpgroup: launched with 168 per thread (384 x 168 =
  // 64512); warpgroup 0 drops to 72 and the compute warpgroups rise to 216
  // (128 x 72 + 256 x 216 = 64512); all return to 168 before the teardown.
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 72;" ::: "memory");
    if (*abort_flag == 0) {
      if (warp == 0) {
        // ---------------- TMA producer (whole warp, one elected lane issues) ----------------
        tma_prefetch_desc_warp(&tmQ);
        tma_prefetch_desc_warp(&tmK);
        tma_prefetch_desc_warp(&tmV);
        tma_prefetch_desc_warp(&tmdO);
        if (L::kTmaDQ) tma_prefetch_desc_warp(&tmdQ);
        mbar_arrive_expect_tx_warp(bar(L::bKVFull), 2 * L::kTileBytes);
        for (int p = 0; p < D / 64; ++p) {
          tma_load_3d_warp(sbase + L::kK + p * L::kPanelBytes, &tmK, bar(L::bKVFull), p * 64, k0, bhk);
          tma_load_3d_warp(sbase + L::kV + p * L::kPanelBytes, &tmV, bar(L::bKVFull), p * 64, k0, bhk);
        }
        int issued = 0;
        for (int i = 0; i < n_iter; ++i) {
          const int s = i % L::kStages;
          const uint32_t ph = (i / L::kStages) & 1;
          if (!wait_warp(bar(L::bQEmpty + s), ph ^ 1, ctl)) break;
          issued = i + 1;
          const int bhq = iter_head(i);
          const int q0 = iter_q0(i);
          mbar_arrive_expect_tx_warp(bar(L::bQFull + s), 2 * L::kTileBytes);
          for (int p = 0; p < D / 64; ++p) {
            tma_load_3d_warp(sbase + L::kQ + s * L::kTileBytes + p * L::kPanelBytes, &tmQ,
                             bar(L::bQFull + s), p * 64, q0, bhq);
            tma_load_3d_warp(sbase + L::kDO + s * L::kTileBytes + p * L::kPanelBytes, &tmdO,
                             bar(L::bQFull + s), p * 64, q0, bhq);
          }
        }
        wait_drain(bar(L::bKVFull), 0, ctl);
        for (int i = issued > L::kStages ? issued - L::kStages : 0; i < issued; ++i)
          wait_drain(bar(L::bQFull + i % L::kStages), (i / L::kStages) & 1, ctl);
      } else if (warp == 1) {
        // ---------------- MMA issuer (whole warp, one elected lane issues) ----------------
        // Order per query tile i: dV(i), S^T(i+1), dK(i), dQ(i), dP^T(i+1). S^T(i+1)
        // overwrites P^T(i) after dV(i) has read it and runs while the compute warps
        // form dS(i); dP^T(i+1) overwrites dS^T(i) after dK(i) has read it.
        constexpr uint32_t idKK = idesc_bf16(128, 128, false, false);  // S^T, dP^T
        constexpr uint32_t idKM = idesc_bf16(128, D, false, true);     // dV, dK: B MN-major
        constexpr uint32_t idMM = idesc_bf16(128, D, true, true);      // dQ: A and B MN-major
        const uint32_t tS = tmem + L::kColS, tDP = tmem + L::kColDP, tDV = tmem + L::kColDV,
                       tDK = tmem + L::kColDK, tDQ = tmem + L::kColDQ;
        // S^T = K Q^T and dP^T = V dO^T of query tile i.
        auto issue_s = [&](int i) {
          const uint32_t sQ = sbase + L::kQ + (i % L::kStages) * L::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
            umma_bf16_warp(tS, sdesc_sw128(sbase + L::kK + koff, 16, 1024),
                           sdesc_sw128(sQ + koff, 16, 1024), idKK, kk > 0);
          }
          umma_commit_warp(bar(L::bSFull));
        };
        auto issue_dp = [&](int i) {
          const uint32_t sDO = sbase + L::kDO + (i % L::kStages) * L::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
            umma_bf16_warp(tDP, sdesc_sw128(sbase + L::kV + koff, 16, 1024),
                           sdesc_sw128(sDO + koff, 16, 1024), idKK, kk > 0);
          }
          umma_commit_warp(bar(L::bDPFull));
        };
        bool ok = wait_warp(bar(L::bKVFull), 0, ctl);
        if (ok && n_iter > 0 && (ok = wait_warp(bar(L::bQFull), 0, ctl))) {
          tc_fence_after();
          issue_s(0);
          issue_dp(0);
        }
        for (int i = 0; ok && i < n_iter; ++i) {
          const int s = i % L::kStages;
          const uint32_t sQ = sbase + L::kQ + s * L::kTileBytes;
          const uint32_t sDO = sbase + L::kDO + s * L::kTileBytes;
          const bool more = i + 1 < n_iter;
          // dV += P^T dO : A = P^T in TMEM (keys x queries), B = dO as [d x queries].
          if (!(ok = wait_warp(bar(L::bPReady), i & 1, ctl))) break;
          if (lane == 0) PFA_BWD_TRACE(0, 2, i);
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            umma_bf16_tmem_a_warp(tDV, tS + packed_col(kk), sdesc_sw128(sDO + kk * 2048, L::kPanelBytes, 1024),
                                  idKM, (i > 0 || kk > 0) ? 1u : 0u);
          if (more) {
            const int s1 = (i + 1) % L::kStages;
            if (!(ok = wait_warp(bar(L::bQFull + s1), ((i + 1) / L::kStages) & 1, ctl))) break;
            if (lane == 0) PFA_BWD_TRACE(0, 1, i + 1);
            tc_fence_after();
            issue_s(i + 1);
          }
          // dK += dS^T Q : A = dS^T in TMEM; dQ = dS K : A = dS^T smem read MN-major.
          if (!(ok = wait_warp(bar(L::bDSReady), i & 1, ctl))) break;
          if (lane == 0) PFA_BWD_TRACE(0, 3, i);
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            umma_bf16_tmem_a_warp(tDK, tDP + packed_col(kk), sdesc_sw128(sQ + kk * 2048, L::kPanelBytes, 1024),
                                  idKM, (i > 0 || kk > 0) ? 1u : 0u);
          if (!L::kDQAliasesDP && i > 0 && !(ok = wait_warp(bar(L::bDQFree), (i - 1) & 1, ctl))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            umma_bf16_warp(tDQ, sdesc_sw128(sbase + L::kDS + kk * 2048, L::kPanelBytes, 1024),
                           sdesc_sw128(sbase + L::kK + kk * 2048, L::kPanelBytes, 1024), idMM, kk > 0);
          // dQ done also means the dS^T buffer and this Q / dO stage are free.
          umma_commit_warp(bar(L::bDQFull));
          umma_commit_warp(bar(L::bQEmpty + s));
          if (more) {
            // With dQ over the dP^T columns, dP^T(i+1) waits until dQ(i) is drained.
            if (L::kDQAliasesDP && !(ok = wait_warp(bar(L::bDQFree), i & 1, ctl))) break;
            tc_fence_after();
            issue_dp(i + 1);
          }
        }
        umma_commit_warp(bar(L::bMMADone));
        umma_commit_warp(bar(L::bDrain));
        wait_drain(bar(L::bDrain), 0, ctl);
      }
    }
    __syncwarp();
    // Reclaim registers only after both compute warpgroups have taken theirs:
    // otherwise an early exit of this group could take the registers they are
    // waiting for. Their arrival follows their first instruction, so this wait is
    // short; it is bounded like every other wait.
    wait_drain(bar(L::bRegs), 0, ctl);
    asm volatile("setmaxnreg.inc.sync.aligned.u32 168;" ::: "memory");
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 216;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(L::bRegs));
    if (*abort_flag == 0) {
      // ---------------- compute warps ----------------
      const uint32_t quarter = warp & 3;
      const int half = (warp - 4) >> 2;          // query columns [64 half, 64 half + 64)
      const int r = quarter * 32 + lane;         // TMEM lane: key row (S^T, dP^T) / query row (dQ)
      const uint32_t lane_off = (quarter * 32u) << 16;
      const int key = k0 + r;
      const float sl2 = sh.scale_log2;
      const float alpha = sh.scale;
      constexpr int kDH = D / 2;                 // dQ / dK / dV columns per warp
      const uint32_t dq_stage = sbase + L::kDQStage + static_cast<uint32_t>(warp - 4) * 4096u;
      bool ok = true;

      // Per-half staging of lse (x log2 e) and delta: slot [slot][half] holds the
      // half's 64 lse values then its 64 deltas. Thread r of the half stages entry
      // r; the value is loaded one iteration ahead so the load latency overlaps
      // the previous tile.
      auto stage_src = [&](int it) -> const float* {
        const int q = iter_q0(it) + 64 * half + (r & 63);
        if (q >= N) return nullptr;
        const size_t off = static_cast<size_t>(iter_head(it)) * N + q;
        return r < 64 ? args.lse + off : args.delta + off;
      };
      float pre = 0.f;
      bool pre_in = false;
      if (n_iter > 0) {
        const float* src = stage_src(0);
        pre_in = src != nullptr;
        if (pre_in) pre = __ldg(src);
      }

      // dQ of iteration `it` from TMEM (this thread: query row q0 + r, columns
      // [kDH half, kDH half + kDH)) -> alpha dQ reduce-added into the workspace.
      auto drain_dq = [&](int it) -> bool {
        if (!wait_warp(bar(L::bDQFull), it & 1, ctl)) return false;
        tc_fence_after();
        if constexpr (L::kTmaDQ) {
          uint32_t v[32];
          tmem_ld32(tmem + L::kColDQ + lane_off + kDH * half, v);
          tmem_ld_wait32(v);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(L::bDQFree));
          // This warp's previous box has been read out of the staging buffer.
          bulk_wait_read_warp();
#pragma unroll
          for (int c = 0; c < 8; ++c)
            st_shared_v4(dq_stage + sw128_offset(lane, c),
                         __float_as_uint(alpha * __uint_as_float(v[4 * c + 0])),
                         __float_as_uint(alpha * __uint_as_float(v[4 * c + 1])),
                         __float_as_uint(alpha * __uint_as_float(v[4 * c + 2])),
                         __float_as_uint(alpha * __uint_as_float(v[4 * c + 3])));
          fence_proxy_async_smem();
          __syncwarp();
          tma_reduce_add_3d_warp(&tmdQ, dq_stage, kDH * half, iter_q0(it) + 32 * static_cast<int>(quarter),
                                 iter_head(it));
        } else {
          const int q = iter_q0(it) + r;
          float* dq_row = args.dq_accum + (static_cast<size_t>(iter_head(it)) * N + q) * D + kDH * half;
#pragma unroll
          for (int c = 0; c < kDH; c += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + L::kColDQ + lane_off + kDH * half + c, v);
            tmem_ld_wait32(v);
            if (q < N) {
#pragma unroll
              for (int u = 0; u < 8; ++u)
                atomicAdd(reinterpret_cast<float4*>(dq_row + c) + u,
                          make_float4(alpha * __uint_as_float(v[4 * u]), alpha * __uint_as_float(v[4 * u + 1]),
                                      alpha * __uint_as_float(v[4 * u + 2]), alpha * __uint_as_float(v[4 * u + 3])));
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(L::bDQFree));
        }
        return true;
      };

      for (int i = 0; ok && i < n_iter; ++i) {
        const int q0 = iter_q0(i);
        const int slot = i & 1;
        float* stage = reinterpret_cast<float*>(smem + L::kLse) + (slot * 2 + half) * 128;
        // Entry r of this slot was last read two tiles ago; every warp of the half
        // has passed the previous tile's wait since, so no one still reads it.
        stage[r] = r < 64 ? (pre_in ? pre * kLog2e : INFINITY) : (pre_in ? pre : 0.f);
        if (i + 1 < n_iter) {
          const float* src = stage_src(i + 1);
          pre_in = src != nullptr;
          if (pre_in) pre = __ldg(src);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::bLse + 2 * half + slot));
        if (!(ok = wait_warp(bar(L::bLse + 2 * half + slot), (i >> 1) & 1, ctl))) break;
        if (lane == 0 && quarter == 0) PFA_BWD_TRACE(1 + half, 4, i);
        const float* lse_s = stage;
        const float* dl_s = stage + 64;

        // P^T = exp(alpha S^T - lse) for this thread's 64 queries.
        const bool diag = CAUSAL && q0 == k0;
        if (!(ok = wait_warp(bar(L::bSFull), i & 1, ctl))) break;
        if (lane == 0 && quarter == 0) PFA_BWD_TRACE(1 + half, 6, i);
        tc_fence_after();
        uint32_t sv[64];
        tmem_ld64(tmem + L::kColS + lane_off + 64 * half, sv);
        tmem_ld_wait64(sv);
        float p[64];
        const float4* l4 = reinterpret_cast<const float4*>(lse_s);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const float4 lq = l4[u];
          fma2v(p[4 * u], p[4 * u + 1], __uint_as_float(sv[4 * u]), __uint_as_float(sv[4 * u + 1]),
                sl2, sl2, -lq.x, -lq.y);
          fma2v(p[4 * u + 2], p[4 * u + 3], __uint_as_float(sv[4 * u + 2]),
                __uint_as_float(sv[4 * u + 3]), sl2, sl2, -lq.z, -lq.w);
        }
#pragma unroll
        for (int c = 0; c < 64; ++c) p[c] = ex2_approx(p[c]);
        if (diag) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (q0 + 64 * half + c < key) p[c] = 0.f;
        }
        {
          uint32_t pk[32];
#pragma unroll
          for (int u = 0; u < 32; ++u) pk[u] = pack_bf16x2(p[2 * u], p[2 * u + 1]);
          tmem_st32(tmem + L::kColS + lane_off + 64 * half, pk);
        }
        tmem_st_wait();
        if (lane == 0 && quarter == 0) PFA_BWD_TRACE(1 + half, 7, i);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::bPReady));

        // The previous tile's dQ; once drained, its product no longer reads the
        // dS^T buffer that this tile's dS phase writes.
        if (i > 0 && !(ok = drain_dq(i - 1))) break;
        if (lane == 0 && quarter == 0) PFA_BWD_TRACE(1 + half, 5, i);

        // dS^T = P^T o (dP^T - delta) (alpha is applied to dK and dQ at the end).
        if (!(ok = wait_warp(bar(L::bDPFull), i & 1, ctl))) break;
        if (lane == 0 && quarter == 0) PFA_BWD_TRACE(1 + half, 9, i);
        tc_fence_after();
        tmem_ld64(tmem + L::kColDP + lane_off + 64 * half, sv);
        tmem_ld_wait64(sv);
        const float4* d4 = reinterpret_cast<const float4*>(dl_s);
        uint32_t pk[32];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const float4 dq = d4[u];
          float t0, t1, t2, t3;
          fma2v(t0, t1, __uint_as_float(sv[4 * u]), __uint_as_float(sv[4 * u + 1]), 1.f, 1.f, -dq.x, -dq.y);
          fma2v(t2, t3, __uint_as_float(sv[4 * u + 2]), __uint_as_float(sv[4 * u + 3]), 1.f, 1.f, -dq.z, -dq.w);
          mul2v(t0, t1, t0, t1, p[4 * u], p[4 * u + 1]);
          mul2v(t2, t3, t2, t3, p[4 * u + 2], p[4 * u + 3]);
          pk[2 * u] = pack_bf16x2(t0, t1);
          pk[2 * u + 1] = pack_bf16x2(t2, t3);
        }
        tmem_st32(tmem + L::kColDP + lane_off + 64 * half, pk);
        // dS^T row into the swizzled [keys][queries] buffer, panel `half`.
        {
          const uint32_t rowb = sbase + L::kDS + half * L::kPanelBytes;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            st_shared_v4(rowb + sw128_offset(r, c), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
        fence_proxy_async_smem();
        tmem_st_wait();
        if (lane == 0 && quarter == 0) PFA_BWD_TRACE(1 + half, 10, i);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::bDSReady));
      }
      if (ok && n_iter > 0) ok = drain_dq(n_iter - 1);

      // ---------------- epilogue: dK (x alpha), dV rows of this key tile ----------------
      if (ok) ok = wait_warp(bar(L::bMMADone), 0, ctl);
      if (ok) {
        tc_fence_after();
        const size_t row = static_cast<size_t>(bhk) * N + key;
#pragma unroll 1
        for (int which = 0; which < 2; ++which) {
          const uint32_t col = (which == 0 ? L::kColDK : L::kColDV) + kDH * half;
          const float sc = which == 0 ? alpha : 1.f;
          __nv_bfloat16* out =
              reinterpret_cast<__nv_bfloat16*>(which == 0 ? args.dk : args.dv) + row * D + kDH * half;
#pragma unroll 1
          for (int c = 0; c < kDH; c += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + col + lane_off + c, v);
            tmem_ld_wait32(v);
            if (key < N) {
              uint4* dst = reinterpret_cast<uint4*>(out + c);
#pragma unroll
              for (int u = 0; u < 4; ++u)
                dst[u] = make_uint4(pack_bf16x2(sc * __uint_as_float(v[8 * u + 0]), sc * __uint_as_float(v[8 * u + 1])),
                                    pack_bf16x2(sc * __uint_as_float(v[8 * u + 2]), sc * __uint_as_float(v[8 * u + 3])),
                                    pack_bf16x2(sc * __uint_as_float(v[8 * u + 4]), sc * __uint_as_float(v[8 * u + 5])),
                                    pack_bf16x2(sc * __uint_as_float(v[8 * u + 6]), sc * __uint_as_float(v[8 * u + 7])));
            }
          }
        }
      }
    }
    // Every dQ box this warp handed to the TMA unit has completed before the
    // CTA's shared memory is released.
    if (L::kTmaDQ) bulk_wait_all_warp();
    asm volatile("setmaxnreg.dec.sync.aligned.u32 168;" ::: "memory");
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
                         const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a,
                         cudaStream_t stream) {
  using L = BwdLayout<D>;
  auto kern = attn_bwd_kernel<D, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  if (e != cudaSuccess) return e;
  const int n_t = (a.s.N + kTile - 1) / kTile;
  const dim3 grid(static_cast<unsigned>(n_t) * a.s.B * a.s.Hkv);
  kern<<<grid, kThreads, L::kBytes, stream>>>(tq, tk, tv, tdo, tdq, a);
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
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a,
                       cudaStream_t stream) {
  if (a.s.d == 64)
    return a.s.causal ? launch_bwd_t<64, true>(tq, tk, tv, tdo, tdq, a, stream)
                      : launch_bwd_t<64, false>(tq, tk, tv, tdo, tdq, a, stream);
  return a.s.causal ? launch_bwd_t<128, true>(tq, tk, tv, tdo, tdq, a, stream)
                    : launch_bwd_t<128, false>(tq, tk, tv, tdo, tdq, a, stream);
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
