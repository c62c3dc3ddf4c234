// Backward kernel. A work item is one (key tile, batch, key/value head); it loops
// over the query heads that share the key/value head and over the query tiles,
// with all five products on tcgen05 (FP32 accumulators in TMEM):
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
// Persistent: one CTA per SM takes items in heavy-first order (key tile 0 has
// the most causal work), dealt in serpentine rounds of gridDim.x. Barrier phases
// count the CTA's query tiles across items, so an item's first products start
// while the previous item's last dQ is drained and its dK / dV are stored, and
// setup and teardown happen once per SM.
//
// 768 threads in six warpgroups: warp 0 Q / dO producer (TMA), warp 1 TMEM
// owner and tcgen05.mma issuer, warp 2 K / V producer, warp 3 idle; warps 4-19
// compute (P^T, dS^T); warps 20-23 drain dQ out of TMEM and, at d = 64, store
// each item's dK and dV through TMA. Compute warp w owns TMEM lane quarter w % 4
// (32 keys) and query group (w - 4) / 4 (32 queries), so each SM sub-partition
// runs four compute warps whose latencies overlap; drain warp w owns the rows of
// lane quarter w % 4 and all d columns of dQ (and of dK, dV).
// P^T and dS^T are cast to BF16 and written back into TMEM over S^T and dP^T
// (each query group over its own input columns), where they are the A operands
// of dV and dK; dS^T also goes to a 128B-swizzled shared buffer that the dQ
// product reads as its (M = queries) A operand.
// TMEM columns: S^T [0,128), dP^T [128,256), dV [256,256+d), dK [256+d,256+2d),
// dQ [384,448) for d = 64 and over dP^T [128,256) for d = 128.
// Tensor-core order per query tile i: dV(i), S^T(i+1), dK(i), then at d = 64
// dP^T(i+1) and dQ(i), at d = 128 (dQ over dP^T) dQ(i) and dP^T(i+1), so the next
// tile's scores are ready when the compute warps finish dS(i).
#include "pfa_device.cuh"
#include "pfa_trace.cuh"

PFA_TRACE_BUFFER(g_pfa_bwd_trace);
#define PFA_BWD_TRACE(slot, ev, j) PFA_TRACE_EVENT(g_pfa_bwd_trace, slot, ev, j)

namespace pfa {
namespace {

constexpr int kThreads = 768;
constexpr float kLog2e = 1.4426950408889634f;

// P^T and dS^T (BF16, two per 32-bit column) are written by each query group
// into the first 16 columns of that group's own 32 FP32 input columns, so no
// group overwrites values another group has yet to load. Query step kk (16
// queries, 8 columns) therefore sits at column 32 (kk / 2) + 8 (kk % 2).
__host__ __device__ constexpr uint32_t packed_col(int kk) {
  return 32u * static_cast<uint32_t>(kk >> 1) + 8u * static_cast<uint32_t>(kk & 1);
}

template <int D>
struct BwdLayout {
  // Query-side stages: the next tile's Q / dO must land within about one
  // iteration, so d = 64 keeps three in flight; d = 128 fits two.
  static constexpr int kStages = (D == 64) ? 3 : 2;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kPanelBytes = kTile * 128;
  // dQ leaves through a TMA reduce-add from a per-warp staging box (d = 64:
  // 32 rows x 16 FP32 columns with 64-byte swizzle, 2 KB per compute warp);
  // d = 128 has no room left for the staging and reduce-adds with vector atomics.
  static constexpr bool kTmaDQ = (D == 64);
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQ = kV + kTileBytes;                // + stage * tile
  static constexpr int kDO = kQ + kStages * kTileBytes;     // + stage * tile
  // d = 64 double-buffers dS^T so that dS(i) need not wait until dQ(i-1) has read
  // dS(i-1); that takes the dQ drain off the compute warps' critical path.
  static constexpr bool kDSDouble = (D == 64);
  static constexpr int kDSBytes = kTile * kTile * 2;
  static constexpr int kDS = kDO + kStages * kTileBytes;    // dS^T [keys][queries] bf16, 2 panels (x 2)
  static constexpr int kDQStage = kDS + (kDSDouble ? 2 : 1) * kDSBytes;  // 4 drain warps x 8 KB (d = 64 only)
  static constexpr int kLse = kDQStage + (kTmaDQ ? 16 * 2048 : 0);  // [slot 2][group 4][-lse 32 | -delta 32]
  static constexpr int kBars = kLse + 2 * 4 * 64 * 4;
  static constexpr int bKVFull = 0;                 // the item's K, V landed
  static constexpr int bKVEmpty = bKVFull + 1;      // the item's last product read K, V
  static constexpr int bQFull = bKVEmpty + 1;       // + stage
  static constexpr int bQEmpty = bQFull + kStages;  // + stage
  static constexpr int bSFull = bQEmpty + kStages;
  static constexpr int bDPFull = bSFull + 1;
  static constexpr int bPReady = bDPFull + 1;
  static constexpr int bDSReady = bPReady + 1;
  static constexpr int bDQFull = bDSReady + 1;
  static constexpr int bDQFree = bDQFull + 1;
  static constexpr int bLse = bDQFree + 1;          // + 2 * group + slot
  static constexpr int bMMADone = bLse + 8;        // the item's products are done (dK, dV final)
  static constexpr int bDrain = bMMADone + 1;
  static constexpr int bRegs = bDrain + 1;          // the compute warps hold their registers
  static constexpr int bEpiDone = bRegs + 1;        // the drain warps have read the item's dK, dV
  static constexpr int kNumBars = bEpiDone + 1;
  static constexpr int kTmemSlot = kBars + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kBytes = kAbort + 4;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
  static constexpr uint32_t kColDQ = (D == 64) ? 384 : 128;
  // Without the second dS buffer (d = 128) dQ also shares the dP^T columns.
  static_assert(kDSDouble ? (kColDQ >= kColDK + D) : (kColDQ == kColDP), "dQ columns");
  static_assert(kDQStage % 1024 == 0, "swizzled staging boxes need 1024-byte alignment");
  static_assert(kBytes <= 232448, "shared memory budget");
};

// DQ = false leaves dQ to the query-outer pass (attn_dq.cu): no dQ product, no dS
// staging in shared memory and no dQ drain; dK and dV are computed as always.
template <int D, bool CAUSAL, bool DQ>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const __grid_constant__ CUtensorMap tmdQ, const __grid_constant__ CUtensorMap tmdK,
                    const __grid_constant__ CUtensorMap tmdV, const BwdArgs args) {
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
  const int group = sh.Hq / sh.Hkv;
  const int n_items = n_t * BHkv;

  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  auto bar = [&](int i) { return sbase + L::kBars + 8u * static_cast<uint32_t>(i); };
  const WaitCtl ctl{abort_flag, args.err, args.err_site, sbase, 2u};

  // Work item -> key tile kt (item / BHkv: key tile 0, the heaviest, first) and
  // (batch, key/value head). Its iterations cover query head bh0 + i / per_head
  // and query tile qt_first + i % per_head; the roles step through them with a
  // cursor.
  struct Item {
    int bhk, k0, qt_first, n_iter, bh0;
  };
  auto decode = [&](int item) {
    Item it;
    const int kt = item / BHkv;
    it.bhk = item % BHkv;
    it.k0 = kt * kTile;
    it.qt_first = CAUSAL ? kt : 0;
    it.n_iter = group * (n_t - it.qt_first);
    it.bh0 = (it.bhk / sh.Hkv) * sh.Hq + (it.bhk % sh.Hkv) * group;
    return it;
  };
  struct QCursor {
    int bh, q0;
  };
  auto first_of = [&](const Item& it) { return QCursor{it.bh0, it.qt_first * kTile}; };
  auto advance = [&](QCursor c, const Item& it) {
    c.q0 += kTile;
    if (c.q0 >= n_t * kTile) {
      c.q0 = it.qt_first * kTile;
      ++c.bh;
    }
    return c;
  };
  const int item0 = static_cast<int>(blockIdx.x);
  const int stride = static_cast<int>(gridDim.x);
  // The k-th item of this CTA: rounds of gridDim.x items, taken left to right in
  // even rounds and right to left in odd ones, so that a CTA given a heavy item
  // early gets a light one in the next round.
  auto item_at = [&](int k) { return k * stride + ((k & 1) ? stride - 1 - item0 : item0); };

  if (threadIdx.x == 0) {
    *abort_flag = (sbase & 1023u) ? 1 : 0;
    if (sbase & 1023u) atomicOr(args.err, PFA_DEVERR_SMEM_ALIGN);
    mbar_init(bar(L::bKVFull), 1);
    mbar_init(bar(L::bKVEmpty), 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::bQFull + s), 1);
      mbar_init(bar(L::bQEmpty + s), 1);
    }
    mbar_init(bar(L::bSFull), 1);
    mbar_init(bar(L::bDPFull), 1);
    mbar_init(bar(L::bPReady), 16);
    mbar_init(bar(L::bDSReady), 16);
    mbar_init(bar(L::bDQFull), 1);
    mbar_init(bar(L::bDQFree), 4);
    for (int x = 0; x < 8; ++x) mbar_init(bar(L::bLse + x), 4);
    mbar_init(bar(L::bMMADone), 1);
    mbar_init(bar(L::bDrain), 1);
    mbar_init(bar(L::bRegs), 20);
    mbar_init(bar(L::bEpiDone), 4);
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
  if (threadIdx.x == 32) PFA_BWD_TRACE(0, 30, 0);
  // Register split per warpgroup: launched with 80 per thread (768 x 80 =
  // 61440); warpgroup 0 and the drain warpgroup drop to 56 and the compute
  // warpgroups rise to 88 (2 x 128 x 56 + 512 x 88 = 59392); all return to 80
  // before the teardown.
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 56;" ::: "memory");
    if (*abort_flag == 0) {
      if (warp == 0) {
        // ---------------- Q / dO producer (whole warp, one elected lane issues) ----------------
        // One stream of query tiles across all items of this CTA.
        tma_prefetch_desc_warp(&tmQ);
        tma_prefetch_desc_warp(&tmdO);
        if (L::kTmaDQ) {
          if (DQ) tma_prefetch_desc_warp(&tmdQ);
          tma_prefetch_desc_warp(&tmdK);
          tma_prefetch_desc_warp(&tmdV);
        }
        int g = 0;        // query tiles issued by this CTA (all items)
        bool ok = true;
        for (int k = 0, item = item0; ok && item < n_items; ++k, item = item_at(k)) {
          const Item it = decode(item);
          QCursor pc = first_of(it);
          for (int i = 0; i < it.n_iter; ++i, ++g, pc = advance(pc, it)) {
            const int s = g % L::kStages;
            if (!(ok = wait_warp(bar(L::bQEmpty + s), ((g / L::kStages) & 1) ^ 1, ctl))) break;
            if (lane == 0) PFA_BWD_TRACE(4, 40, g);
            mbar_arrive_expect_tx_warp(bar(L::bQFull + s), 2 * L::kTileBytes);
            for (int p = 0; p < D / 64; ++p) {
              tma_load_3d_warp(sbase + L::kQ + s * L::kTileBytes + p * L::kPanelBytes, &tmQ,
                               bar(L::bQFull + s), p * 64, pc.q0, pc.bh);
              tma_load_3d_warp(sbase + L::kDO + s * L::kTileBytes + p * L::kPanelBytes, &tmdO,
                               bar(L::bQFull + s), p * 64, pc.q0, pc.bh);
            }
          }
        }
        // Every issued copy has landed before shared memory is released (earlier
        // ones were consumed before later ones could reuse their stage).
        for (int i = g > L::kStages ? g - L::kStages : 0; i < g; ++i)
          wait_drain(bar(L::bQFull + i % L::kStages), (i / L::kStages) & 1, ctl);
      } else if (warp == 2) {
        // ---------------- K / V producer: one pair per item ----------------
        // The item's K and V once the previous item's last product has read
        // theirs; the next item's pair is prefetched into L2 meanwhile.
        tma_prefetch_desc_warp(&tmK);
        tma_prefetch_desc_warp(&tmV);
        int kv = 0;
        bool ok = true;
        for (int k = 0, item = item0; item < n_items; ++k, item = item_at(k)) {
          const Item it = decode(item);
          if (kv > 0 && !(ok = wait_warp(bar(L::bKVEmpty), (kv - 1) & 1, ctl))) break;
          mbar_arrive_expect_tx_warp(bar(L::bKVFull), 2 * L::kTileBytes);
          for (int p = 0; p < D / 64; ++p) {
            tma_load_3d_warp(sbase + L::kK + p * L::kPanelBytes, &tmK, bar(L::bKVFull), p * 64, it.k0, it.bhk);
            tma_load_3d_warp(sbase + L::kV + p * L::kPanelBytes, &tmV, bar(L::bKVFull), p * 64, it.k0, it.bhk);
          }
          ++kv;
          if (item_at(k + 1) < n_items) {
            const Item nx = decode(item_at(k + 1));
            for (int p = 0; p < D / 64; ++p) {
              tma_prefetch_l2_3d_warp(&tmK, p * 64, nx.k0, nx.bhk);
              tma_prefetch_l2_3d_warp(&tmV, p * 64, nx.k0, nx.bhk);
            }
          }
        }
        if (kv > 0) wait_drain(bar(L::bKVFull), (kv - 1) & 1, ctl);
        (void)ok;
#if defined(PFA_TRACE) && defined(PFA_TRACE_QOBS)
      } else if (warp == 3) {
        // Trace builds only: time at which each query stage of the first item lands.
        const Item it0 = decode(item0);
        for (int g = 0; g < it0.n_iter && g < 1000; ++g) {
          if (!wait_drain(bar(L::bQFull + g % L::kStages), (g / L::kStages) & 1, ctl)) break;
          if (lane == 0) PFA_BWD_TRACE(6, 42, g);
        }
#endif
      } else if (warp == 1) {
        // ---------------- MMA issuer (whole warp, one elected lane issues) ----------------
        // Order per query tile i: dV(i), S^T(i+1), dK(i), then dP^T(i+1) and dQ(i)
        // (d = 64: dP^T first; d = 128, where dQ sits over dP^T: dQ first). S^T(i+1)
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
        // The stage of query tile g (counted across items) is g % kStages.
        int g = 0;
        int kv = 0;
        bool ok = true;
        for (int k = 0, item = item0; ok && item < n_items; ++k, item = item_at(k), ++kv) {
          const Item it = decode(item);
          if (!(ok = wait_warp(bar(L::bKVFull), kv & 1, ctl))) break;
          if (lane == 0) PFA_BWD_TRACE(0, 37, kv);
          if (!(ok = wait_warp(bar(L::bQFull + g % L::kStages), (g / L::kStages) & 1, ctl))) break;
          // With dQ over the dP^T columns (d = 128), dP^T(0) waits until the
          // previous item's last dQ has been drained.
          if (DQ && !L::kDSDouble && g > 0 && !(ok = wait_warp(bar(L::bDQFree), (g - 1) & 1, ctl))) break;
          tc_fence_after();
          issue_s(g);
          issue_dp(g);
          for (int i = 0; ok && i < it.n_iter; ++i) {
            const int gg = g + i;
            const int s = gg % L::kStages;
            const uint32_t sQ = sbase + L::kQ + s * L::kTileBytes;
            const uint32_t sDO = sbase + L::kDO + s * L::kTileBytes;
            const bool more = i + 1 < it.n_iter;
            // dV += P^T dO : A = P^T in TMEM (keys x queries), B = dO as [d x queries].
            if (!(ok = wait_warp(bar(L::bPReady), gg & 1, ctl))) break;
            if (lane == 0) PFA_BWD_TRACE(0, 2, gg);
            // dV(0) and dK(0) overwrite the accumulators: with the drain warps
            // storing dK / dV (d = 64) they wait until the previous item's are read.
            if (L::kTmaDQ && i == 0 && kv > 0 && !(ok = wait_warp(bar(L::bEpiDone), (kv - 1) & 1, ctl)))
              break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              umma_bf16_tmem_a_warp(tDV, tS + packed_col(kk), sdesc_sw128(sDO + kk * 2048, L::kPanelBytes, 1024),
                                    idKM, (i > 0 || kk > 0) ? 1u : 0u);
            if (lane == 0) PFA_BWD_TRACE(0, 43, gg);
            if (more) {
              const int s1 = (gg + 1) % L::kStages;
              if (!(ok = wait_warp(bar(L::bQFull + s1), ((gg + 1) / L::kStages) & 1, ctl))) break;
              if (lane == 0) PFA_BWD_TRACE(0, 1, gg + 1);
              tc_fence_after();
              issue_s(gg + 1);
            }
            // dK += dS^T Q : A = dS^T in TMEM; dQ = dS K : A = dS^T smem read MN-major.
            if (!(ok = wait_warp(bar(L::bDSReady), gg & 1, ctl))) break;
            if (lane == 0) PFA_BWD_TRACE(0, 3, gg);
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              umma_bf16_tmem_a_warp(tDK, tDP + packed_col(kk), sdesc_sw128(sQ + kk * 2048, L::kPanelBytes, 1024),
                                    idKM, (i > 0 || kk > 0) ? 1u : 0u);
            if (lane == 0) PFA_BWD_TRACE(0, 44, gg);
            // dK(i) is the last reader of this Q / dO stage (dQ reads dS and K).
            umma_commit_warp(bar(L::bQEmpty + s));
            if constexpr (!DQ) {
              // dP^T(i+1) overwrites dS^T(i) after dK(i) has read it (issue order).
              if (more) issue_dp(gg + 1);
              continue;
            }
            if constexpr (L::kDSDouble) {
              // dP^T(i+1) overwrites dS^T(i) after dK(i) has read it; dQ(i) reads its
              // own dS buffer and waits only until dQ(i-1) has left TMEM.
              if (more) issue_dp(gg + 1);
              if (lane == 0) PFA_BWD_TRACE(0, 45, gg);
              if (gg > 0 && !(ok = wait_warp(bar(L::bDQFree), (gg - 1) & 1, ctl))) break;
              if (lane == 0) PFA_BWD_TRACE(0, 46, gg);
            }
            tc_fence_after();
            const uint32_t sDS = sbase + L::kDS + (L::kDSDouble ? (gg & 1) * L::kDSBytes : 0);
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              umma_bf16_warp(tDQ, sdesc_sw128(sDS + kk * 2048, L::kPanelBytes, 1024),
                             sdesc_sw128(sbase + L::kK + kk * 2048, L::kPanelBytes, 1024), idMM, kk > 0);
            if (lane == 0) PFA_BWD_TRACE(0, 47, gg);
            umma_commit_warp(bar(L::bDQFull));
            if constexpr (!L::kDSDouble) {
              if (more) {
                // dQ sits over the dP^T columns: dP^T(i+1) waits until dQ(i) is drained.
                if (!(ok = wait_warp(bar(L::bDQFree), gg & 1, ctl))) break;
                tc_fence_after();
                issue_dp(gg + 1);
              }
            }
          }
          g += it.n_iter;
          // The item's products are done once these commits arrive: dK / dV are
          // final and K / V may be replaced.
          if (lane == 0) PFA_BWD_TRACE(0, 31, kv);
          umma_commit_warp(bar(L::bMMADone));
          umma_commit_warp(bar(L::bKVEmpty));
        }
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
    asm volatile("setmaxnreg.inc.sync.aligned.u32 80;" ::: "memory");
  } else if (warp >= 20) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 56;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(L::bRegs));
    if (*abort_flag == 0) {
      // ---------------- drain warps: dQ(i) out of TMEM, alpha dQ into the workspace ----------------
      const uint32_t quarter = warp & 3;
      const uint32_t lane_off = (quarter * 32u) << 16;
      const float alpha = sh.scale;
      const uint32_t dq_stage = sbase + L::kDQStage + static_cast<uint32_t>(warp - 20) * 8192u;
      bool ok = true;
      int g = 0;
      int kv = 0;   // items drained (the MMADone phases)
      for (int k = 0, item = item0; ok && item < n_items; ++k, item = item_at(k)) {
        const Item itm = decode(item);
        QCursor qc = first_of(itm);
        for (int i = 0; DQ && ok && i < itm.n_iter; ++i, ++g, qc = advance(qc, itm)) {
        const int it = g;
        if (!(ok = wait_warp(bar(L::bDQFull), it & 1, ctl))) break;
        if (lane == 0 && quarter == 0) PFA_BWD_TRACE(5, 13, it);
        tc_fence_after();
        if constexpr (L::kTmaDQ) {
          // Two 32 x 32 FP32 boxes (128-byte swizzle) per warp; the previous
          // tile's boxes have been read out before they are rewritten.
          bulk_wait_read_warp();
          if (lane == 0 && quarter == 0) PFA_BWD_TRACE(5, 35, it);
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            uint32_t v[32];
            tmem_ld32(tmem + L::kColDQ + lane_off + 32 * c, v);
            tmem_ld_wait32(v);
            if (c == 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(bar(L::bDQFree));
              if (lane == 0 && quarter == 0) PFA_BWD_TRACE(5, 36, it);
            }
            const uint32_t box = dq_stage + 4096u * c;
#pragma unroll
            for (int u = 0; u < 8; ++u)
              st_shared_v4(box + sw128_offset(lane, u), __float_as_uint(alpha * __uint_as_float(v[4 * u + 0])),
                           __float_as_uint(alpha * __uint_as_float(v[4 * u + 1])),
                           __float_as_uint(alpha * __uint_as_float(v[4 * u + 2])),
                           __float_as_uint(alpha * __uint_as_float(v[4 * u + 3])));
          }
          fence_proxy_async_smem();
          __syncwarp();
          const int y = qc.q0 + 32 * static_cast<int>(quarter);
          tma_reduce_add_3d_warp(&tmdQ, dq_stage, 0, y, qc.bh);
          tma_reduce_add_3d_warp(&tmdQ, dq_stage + 4096u, 32, y, qc.bh);
          if (lane == 0 && quarter == 0) PFA_BWD_TRACE(5, 41, it);
        } else {
          const int q = qc.q0 + static_cast<int>(quarter) * 32 + lane;
          float* dq_row = args.dq_accum + (static_cast<size_t>(qc.bh) * N + q) * D;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(tmem + L::kColDQ + lane_off + 32 * c, v);
            tmem_ld_wait32(v);
            if (c == D / 32 - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(bar(L::bDQFree));
            }
            if (q < N) {
#pragma unroll
              for (int u = 0; u < 8; ++u)
                atomicAdd(reinterpret_cast<float4*>(dq_row + 32 * c) + u,
                          make_float4(alpha * __uint_as_float(v[4 * u]), alpha * __uint_as_float(v[4 * u + 1]),
                                      alpha * __uint_as_float(v[4 * u + 2]), alpha * __uint_as_float(v[4 * u + 3])));
            }
          }
        }
        if (lane == 0 && quarter == 0) PFA_BWD_TRACE(5, 5, it);
        }
        if constexpr (L::kTmaDQ) {
          // ---------------- item epilogue: alpha dK and dV of this key tile ----------------
          // This warp's 32 key rows of dK then dV become two BF16 64-column boxes
          // in its staging area, stored by TMA: the compute warps go straight on
          // to the next item, and the stores leave asynchronously.
          if (ok) ok = wait_warp(bar(L::bMMADone), kv & 1, ctl);
          if (ok) {
            tc_fence_after();
            bulk_wait_read_warp();   // the staging area's last dQ boxes have been read
#pragma unroll 1
            for (int which = 0; which < 2; ++which) {
              const uint32_t col = which == 0 ? L::kColDK : L::kColDV;
              const float sc = which == 0 ? alpha : 1.f;
              const uint32_t box = dq_stage + 4096u * static_cast<uint32_t>(which);
#pragma unroll 1
              for (int c = 0; c < 2; ++c) {   // columns 32 c .. 32 c + 31
                uint32_t v[32];
                tmem_ld32(tmem + col + lane_off + 32 * c, v);
                tmem_ld_wait32(v);
                if (which == 1 && c == 1) {
                  // dK and dV are out of TMEM: the next item may overwrite them.
                  tc_fence_before();
                  __syncwarp();
                  if (lane == 0) mbar_arrive(bar(L::bEpiDone));
                }
                auto f = [&](int e) { return sc * __uint_as_float(v[e]); };
                // 32 BF16 values = 16-byte chunks 4 c .. 4 c + 3 of the 128-byte row.
#pragma unroll
                for (int u = 0; u < 4; ++u)
                  st_shared_v4(box + sw128_offset(lane, 4 * c + u), pack_bf16x2(f(8 * u), f(8 * u + 1)),
                               pack_bf16x2(f(8 * u + 2), f(8 * u + 3)), pack_bf16x2(f(8 * u + 4), f(8 * u + 5)),
                               pack_bf16x2(f(8 * u + 6), f(8 * u + 7)));
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
            const int y = itm.k0 + 32 * static_cast<int>(quarter);
            tma_store_3d_warp(&tmdK, dq_stage, 0, y, itm.bhk);
            tma_store_3d_warp(&tmdV, dq_stage + 4096u, 0, y, itm.bhk);
          }
          ++kv;
        }
      }
    }
    // Every dQ box handed to the TMA unit has completed before the CTA's shared
    // memory is released; registers are reclaimed as warpgroup 0 does.
    if (L::kTmaDQ) bulk_wait_all_warp();
    wait_drain(bar(L::bRegs), 0, ctl);
    asm volatile("setmaxnreg.inc.sync.aligned.u32 80;" ::: "memory");
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 88;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(L::bRegs));
    if (*abort_flag == 0) {
      // ---------------- compute warps ----------------
      const uint32_t quarter = warp & 3;
      const int grp = (warp - 4) >> 2;           // query columns [32 grp, 32 grp + 32)
      const int r = quarter * 32 + lane;         // TMEM lane: key row (S^T, dP^T) / query row (dQ)
      const int rg = r;                          // thread index within the group's 128
      const uint32_t lane_off = (quarter * 32u) << 16;
      const float sl2 = sh.scale_log2;
      const float alpha = sh.scale;
      constexpr int kDG = D / 4;                 // dQ / dK / dV columns per warp
      bool ok = true;

      // Per-group staging of -lse (x log2 e) and -delta: slot [slot][grp] holds
      // the group's 32 values of -lse then its 32 values of -delta. Thread rg < 64
      // of the group stages entry rg; the value is loaded one iteration ahead so
      // the load latency overlaps the previous tile.
      auto stage_src = [&](QCursor c) -> const float* {
        if (rg >= 64) return nullptr;
        const int q = c.q0 + 32 * grp + (rg & 31);
        if (q >= N) return nullptr;
        const size_t off = static_cast<size_t>(c.bh) * N + q;
        return rg < 32 ? args.lse + off : args.delta + off;
      };
      float pre = 0.f;
      bool pre_in = false;
      if (item0 < n_items) {
        const float* src = stage_src(first_of(decode(item0)));
        pre_in = src != nullptr;
        if (pre_in) pre = ld_global_early(src);
      }

      int g = 0;   // query tiles of this CTA so far (all items): the barrier phases
      for (int k = 0, item = item0, kv = 0; ok && item < n_items; ++k, item = item_at(k), ++kv) {
      const Item itm = decode(item);
      const int k0 = itm.k0;
      const int key = k0 + r;
      QCursor cur = first_of(itm);
      for (int i = 0; ok && i < itm.n_iter; ++i, ++g) {
        const int gi = g;
        const int q0 = cur.q0;
        // The next query tile: this item's next one or the next item's first.
        const bool has_nxt = i + 1 < itm.n_iter || item_at(k + 1) < n_items;
        const QCursor nxt = i + 1 < itm.n_iter ? advance(cur, itm) : first_of(decode(item_at(k + 1)));
        const int slot = gi & 1;
        float* stage = reinterpret_cast<float*>(smem + L::kLse) + (slot * 4 + grp) * 64;
        // Entry rg of this slot was last read two tiles ago; every warp of the
        // group has passed the previous tile's wait since, so no one still reads it.
        if (lane == 0 && quarter == 0 && grp < 3) PFA_BWD_TRACE(1 + grp, 26, i);
        if (rg < 64) stage[rg] = rg < 32 ? (pre_in ? -pre * kLog2e : -INFINITY) : (pre_in ? -pre : 0.f);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::bLse + 2 * grp + slot));
        if (lane == 0 && quarter == 0 && grp < 3) PFA_BWD_TRACE(1 + grp, 27, i);
        if (!(ok = wait_warp(bar(L::bLse + 2 * grp + slot), (gi >> 1) & 1, ctl))) break;
        if (lane == 0 && quarter == 0 && grp < 3) PFA_BWD_TRACE(1 + grp, 4, i);

        // P^T = exp(alpha S^T - lse) for this thread's 32 queries.
        const bool diag = CAUSAL && q0 == k0;
        if (!(ok = wait_warp(bar(L::bSFull), gi & 1, ctl))) break;
        if (lane == 0 && quarter == 0 && grp < 3) PFA_BWD_TRACE(1 + grp, 6, i);
        tc_fence_after();
        uint32_t sv[32];
        tmem_ld32(tmem + L::kColS + lane_off + 32 * grp, sv);
        tmem_ld_wait32(sv);
        if (lane == 0 && quarter == 0 && grp < 3) PFA_BWD_TRACE(1 + grp, 11, i);
        float p[32];
        const float4* l4 = reinterpret_cast<const float4*>(stage);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 lq = l4[u];
          fma2v(p[4 * u], p[4 * u + 1], __uint_as_float(sv[4 * u]), __uint_as_float(sv[4 * u + 1]),
                sl2, sl2, lq.x, lq.y);
          fma2v(p[4 * u + 2], p[4 * u + 3], __uint_as_float(sv[4 * u + 2]),
                __uint_as_float(sv[4 * u + 3]), sl2, sl2, lq.z, lq.w);
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) p[c] = ex2_approx(p[c]);
        if (diag) {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (q0 + 32 * grp + c < key) p[c] = 0.f;
        }
        {
          uint32_t pk[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) pk[u] = pack_bf16x2(p[2 * u], p[2 * u + 1]);
          if (lane == 0 && quarter == 0 && grp < 3) PFA_BWD_TRACE(1 + grp, 12, i);
          tmem_st16(tmem + L::kColS + lane_off + 32 * grp, pk);
        }
        tmem_st_wait();
        if (lane == 0 && quarter == 0 && grp < 3) PFA_BWD_TRACE(1 + grp, 7, i);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::bPReady));
        // Prefetch the next tile's entry here: an mbarrier arrive (a release)
        // waits for the arriving lane's loads in flight, and the next arrive of
        // this warp comes after the whole dS phase.
        if (has_nxt) {
          const float* src = stage_src(nxt);
          pre_in = src != nullptr;
          if (pre_in) pre = ld_global_early(src);
        }


        // dS^T = P^T o (dP^T - delta) (alpha is applied to dK and dQ at the end).
        if (!(ok = wait_warp(bar(L::bDPFull), gi & 1, ctl))) break;
        if (lane == 0 && quarter == 0 && grp < 3) PFA_BWD_TRACE(1 + grp, 9, i);
        tc_fence_after();
        uint32_t dv[32];
        tmem_ld32(tmem + L::kColDP + lane_off + 32 * grp, dv);
        tmem_ld_wait32(dv);
        if (lane == 0 && quarter == 0 && grp < 3) PFA_BWD_TRACE(1 + grp, 17, i);
        const float4* d4 = reinterpret_cast<const float4*>(stage + 32);
        uint32_t pk[16];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 nd = d4[u];
          float t0 = __uint_as_float(dv[4 * u]), t1 = __uint_as_float(dv[4 * u + 1]);
          float t2 = __uint_as_float(dv[4 * u + 2]), t3 = __uint_as_float(dv[4 * u + 3]);
          add2(t0, t1, nd.x, nd.y);
          add2(t2, t3, nd.z, nd.w);
          mul2v(t0, t1, t0, t1, p[4 * u], p[4 * u + 1]);
          mul2v(t2, t3, t2, t3, p[4 * u + 2], p[4 * u + 3]);
          pk[2 * u] = pack_bf16x2(t0, t1);
          pk[2 * u + 1] = pack_bf16x2(t2, t3);
        }
        tmem_st16(tmem + L::kColDP + lane_off + 32 * grp, pk);
        // dS^T row into the swizzled [keys][queries] buffer: panel grp / 2, 16-byte
        // chunks 4 (grp % 2) .. 4 (grp % 2) + 3 of the 128-byte row.
        if constexpr (DQ) {
          // The last reader of this buffer, dQ(i-2) (one buffer: dQ(i-1)), was
          // issued before dP^T(i); that product's commit, which this warp waited
          // for, arrives only after every earlier product has completed.
          const uint32_t rowb =
              sbase + L::kDS + (L::kDSDouble ? (gi & 1) * L::kDSBytes : 0) + (grp >> 1) * L::kPanelBytes;
#pragma unroll
          for (int c = 0; c < 4; ++c)
            st_shared_v4(rowb + sw128_offset(r, 4 * (grp & 1) + c), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                         pk[4 * c + 3]);
          if (lane == 0 && quarter == 0 && grp < 3) PFA_BWD_TRACE(1 + grp, 18, i);
          fence_proxy_async_smem();
        }
        tmem_st_wait();
        if (lane == 0 && quarter == 0 && grp < 3) PFA_BWD_TRACE(1 + grp, 10, i);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::bDSReady));
        cur = nxt;
      }

      // ---------------- item epilogue (d = 128): dK (x alpha), dV rows of this key tile ----------------
      // The next item's dV(0) / dK(0), which overwrite these accumulators, wait for
      // its P^T(0) / dS^T(0), which this warp produces only after this epilogue.
      // At d = 64 the drain warps store dK and dV instead.
      if constexpr (!L::kTmaDQ) {
      if (ok) ok = wait_warp(bar(L::bMMADone), kv & 1, ctl);
      if (lane == 0 && quarter == 0 && grp < 3) PFA_BWD_TRACE(1 + grp, 25, kv);
      if (ok) {
        tc_fence_after();
        const size_t row = static_cast<size_t>(itm.bhk) * N + key;
#pragma unroll 1
        for (int which = 0; which < 2; ++which) {
          const uint32_t col = (which == 0 ? L::kColDK : L::kColDV) + kDG * grp;
          const float sc = which == 0 ? alpha : 1.f;
          __nv_bfloat16* out =
              reinterpret_cast<__nv_bfloat16*>(which == 0 ? args.dk : args.dv) + row * D + kDG * grp;
#pragma unroll 1
          for (int c = 0; c < kDG; c += 16) {
            uint32_t v[16];
            tmem_ld16(tmem + col + lane_off + c, v);
            tmem_ld_wait16(v);
            if (lane == 0 && quarter == 0 && grp < 3) PFA_BWD_TRACE(1 + grp, 33 + which, kv);
            if (key < N) {
              uint4* dst = reinterpret_cast<uint4*>(out + c);
#pragma unroll
              for (int u = 0; u < 2; ++u)
                dst[u] = make_uint4(pack_bf16x2(sc * __uint_as_float(v[8 * u + 0]), sc * __uint_as_float(v[8 * u + 1])),
                                    pack_bf16x2(sc * __uint_as_float(v[8 * u + 2]), sc * __uint_as_float(v[8 * u + 3])),
                                    pack_bf16x2(sc * __uint_as_float(v[8 * u + 4]), sc * __uint_as_float(v[8 * u + 5])),
                                    pack_bf16x2(sc * __uint_as_float(v[8 * u + 6]), sc * __uint_as_float(v[8 * u + 7])));
            }
          }
        }
      }
      }
      }
    }
    asm volatile("setmaxnreg.dec.sync.aligned.u32 80;" ::: "memory");
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 32) PFA_BWD_TRACE(0, 32, 0);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL, bool DQ>
cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& tdk,
                         const CUtensorMap& tdv, const BwdArgs& a, cudaStream_t stream) {
  using L = BwdLayout<D>;
  auto kern = attn_bwd_kernel<D, CAUSAL, DQ>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  if (e != cudaSuccess) return e;
  // Persistent: one CTA per SM (at most one per work item).
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const long long n_items = static_cast<long long>((a.s.N + kTile - 1) / kTile) * a.s.B * a.s.Hkv;
  const dim3 grid(static_cast<unsigned>(n_items < sms ? n_items : sms));
  return launch_pdl(kern, grid, dim3(kThreads), L::kBytes, stream, tq, tk, tv, tdo, tdq, tdk, tdv, a);
}

__global__ void zero_kernel(float4* __restrict__ dst, long long n4) {
  grid_launch_dependents();
  grid_dependency_wait();   // the previous kernel may still read the buffer
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

__global__ void convert_dq_kernel(const float4* __restrict__ src, uint2* __restrict__ dst, long long n4) {
  grid_launch_dependents();
  grid_dependency_wait();   // the workspace is the previous kernel's output
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 x = src[i];
    dst[i] = make_uint2(pack_bf16x2(x.x, x.y), pack_bf16x2(x.z, x.w));
  }
}

template <bool DQ>
cudaError_t dispatch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& tdk,
                         const CUtensorMap& tdv, const BwdArgs& a, cudaStream_t stream) {
  if (a.s.d == 64)
    return a.s.causal ? launch_bwd_t<64, true, DQ>(tq, tk, tv, tdo, tdq, tdk, tdv, a, stream)
                      : launch_bwd_t<64, false, DQ>(tq, tk, tv, tdo, tdq, tdk, tdv, a, stream);
  return a.s.causal ? launch_bwd_t<128, true, DQ>(tq, tk, tv, tdo, tdq, tdk, tdv, a, stream)
                    : launch_bwd_t<128, false, DQ>(tq, tk, tv, tdo, tdq, tdk, tdv, a, stream);
}

}  // namespace

cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& tdk,
                       const CUtensorMap& tdv, const BwdArgs& a, cudaStream_t stream) {
  return a.dq_accum != nullptr ? dispatch_bwd<true>(tq, tk, tv, tdo, tdq, tdk, tdv, a, stream)
                               : dispatch_bwd<false>(tq, tk, tv, tdo, tdq, tdk, tdv, a, stream);
}

// Zero the FP32 dQ workspace (n4 float4 values) as a kernel, so that it chains
// with the kernels around it by programmatic dependent launch.
cudaError_t launch_zero_workspace(float* ws, long long n4, cudaStream_t stream) {
  const int threads = 256;
  long long blocks = (n4 + threads - 1) / threads;
  if (blocks > 152 * 8) blocks = 152 * 8;
  if (blocks < 1) blocks = 1;
  return launch_pdl(zero_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream,
                    reinterpret_cast<float4*>(ws), n4);
}

// dQ = BF16(dQ workspace); n is a multiple of 4 (d is 64 or 128).
cudaError_t launch_convert_dq(const float* dq_accum, void* dq, long long n, cudaStream_t stream) {
  const long long n4 = n / 4;
  const int threads = 256;
  long long blocks = (n4 + threads - 1) / threads;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  return launch_pdl(convert_dq_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream,
                    reinterpret_cast<const float4*>(dq_accum), reinterpret_cast<uint2*>(dq), n4);
}

}  // namespace pfa
