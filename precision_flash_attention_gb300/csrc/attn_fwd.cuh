// Forward kernel: S = alpha Q K^T on tcgen05 (FP32 in TMEM), the online safe
// softmax with the repeated-maximum tracker and the per-call shift rule,
// Pbar = exp(S - m) in FP32 cast to BF16, Obar += Pbar V on tcgen05 (FP32 in
// TMEM), then O = Obar / l (BF16) and lse = m + ln l (FP32), plus the
// diagnostic counters.
//
// The method is the one analysed in Qiu & Yao, "Why Low-Precision Transformer
// Training Fails: An Analysis on Flash Attention" (ICLR 2026), as summarised by
// the priors.kr post "BF16 플래시 어텐션은 왜 수천 스텝 뒤에 무너질까" (core idea,
// equations, and the fix of paper §4) and the bud-325 note of the same title
// (Key claims, Method / Algorithm 1).
//
// A work item is two adjacent 128-row Q tiles (t = 0, 1) of one (batch, query
// head). Persistent: one CTA per SM takes items heaviest causal pairs first,
// dealt in serpentine rounds of gridDim.x; barrier phases count across items, so setup and
// teardown happen once per SM and the next item's Q (double buffered for
// d = 64) and K / V stream in while the current item finishes. 384 threads,
// one warpgroup per role group (registers are granted per warpgroup):
//   warp 0      K / V producer (one ring of stages across items)
//   warp 1      TMEM owner and tcgen05.mma issuer
//   warp 2      Q producer (one pair per item)
//   warp 3      idle
//   warps 4..7  softmax of tile 0, warps 8..11 softmax of tile 1; one query row
//               per thread (TMEM lane quarter = warp % 4)
// TMEM (512 columns): S_t in [128 t, 128 t + 128), O_t in [256 + d t, 256 + d t + d).
// Pbar_t (BF16) is the TMEM A operand of Obar_t += Pbar_t V. At d = 64 it has
// its own columns [384 + 64 t, 448 + 64 t): once the softmax has read S_t(j)
// into registers the tensor core computes S_t(j+1), so each softmax warpgroup
// finds its next scores ready when it finishes a tile; the tensor core runs
// S0_j, S1_j, PV0_{j-1}, PV1_{j-1}, ... At d = 128 (no columns left) Pbar_t is
// written over the first 64 columns of S_t and the tensor core runs S0_j,
// PV1_{j-1}, S1_j, PV0_j, ... so that each tile's softmax overlaps the other
// tile's two products.
//
// Template parameters: D (64 or 128), MODE (the shift rule, 0/1/2), CAUSAL, MON
// (0 nothing counted, 1 the diagnostic counters, 2 the counters and the monitor:
// the operational count of BF16 Pbar == 1 handed to the product and the
// histogram of tie multiplicities), PROFILE (d = 64 only: each key tile's product
// Pbar V is rounded to BF16 and accumulated across tiles in BF16, as an
// implementation that stores the unnormalised product in BF16 does; a study
// variant, not the fused path), PBAR (the format of the Pbar operand: BF16, or,
// for the study of narrower formats, FP8 E4M3 or MXFP4 = E2M1 with one
// power-of-two scale per 32 keys; the rounded values are exact in BF16, so the
// BF16 product with FP32 accumulation computes what a product in that format
// with FP32 accumulation does, and l sums the rounded values). The instantiations
// live in attn_fwd.cu (the fused path), attn_fwd_study.cu (monitor and profile)
// and attn_fwd_lowp.cu (the narrow Pbar formats).
#pragma once

#include "pfa_device.cuh"
#include "pfa_trace.cuh"

// Trace builds (-DPFA_TRACE) time the fused path only; the study translation unit
// defines PFA_FWD_NO_TRACE.
#ifndef PFA_FWD_NO_TRACE
PFA_TRACE_BUFFER(g_pfa_fwd_trace);
#define PFA_FWD_TRACE(slot, ev, j) PFA_TRACE_EVENT(g_pfa_fwd_trace, slot, ev, j)
#else
#define PFA_FWD_TRACE(slot, ev, j) \
  do {                             \
  } while (0)
#endif

namespace pfa {
namespace fwd {

constexpr int kThreads = 384;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kEpsShift = 0.03125f;  // 2^-5
// Smallest FP32 value that rounds to BF16 1.0 (the midpoint 1 - 2^-9 ties to 1.0).
constexpr float kBf16OneThreshold = 0.998046875f;
constexpr int kTieBins = 8;            // tie multiplicity 1..7 and >= 8
// Formats of the Pbar operand of the Pbar V product.
constexpr int kPbarBf16 = 0, kPbarE4m3 = 1, kPbarMxfp4 = 2;

// PAIR: the two CTAs of a cluster share each product (cta_group::2, M = 256):
// each CTA holds its own two query tiles, half of each K tile (64 keys, all d
// columns) and half of each V tile (all keys, 64 of the d columns).
template <int D, bool PROFILE, bool PAIR = false>
struct FwdLayout {
  static_assert(!PROFILE || D == 64, "the unfused profile is built for d = 64");
  static_assert(!PAIR || (D == 128 && !PROFILE), "the CTA pairing is built for the fused d = 128 path");
  static constexpr int kStages = (D == 64 || PAIR) ? 3 : 2;
  static constexpr int kQBufs = (D == 64 || PAIR) ? 2 : 1;   // Q pairs in flight
  // d = 64: Pbar_t gets its own TMEM columns [384 + 64 t, 448 + 64 t), so the
  // next S_t can be computed as soon as the softmax holds the current one in
  // registers. d = 128 has no columns left and writes Pbar_t over S_t, and so
  // does the profile, whose tile product U_t = Pbar_t V takes [384 + 64 t, 448 + 64 t).
  static constexpr bool kSplitP = (D == 64) && !PROFILE;
  static constexpr uint32_t kColP = 384;
  static constexpr uint32_t kColU = 384;
  static constexpr int kTileBytes = kTile * D * 2;   // 128 rows x D bf16
  static constexpr int kPanelBytes = kTile * 128;    // 128 rows x 64 bf16
  static constexpr int kKRows = PAIR ? kTile / 2 : kTile;          // keys of a K stage
  static constexpr int kKPanelBytes = kKRows * 128;                 // kKRows x 64 bf16
  static constexpr int kKBytes = kKRows * D * 2;                    // one K stage
  static constexpr int kVBytes = PAIR ? kPanelBytes : kTileBytes;   // one V stage
  static constexpr int kQ = 0;                       // + (buffer * 2 + t) * tile
  static constexpr int kK = kQBufs * 2 * kTileBytes; // + stage * kKBytes
  static constexpr int kV = kK + kStages * kKBytes;  // + stage * kVBytes
  static constexpr int kBars = kV + kStages * kVBytes;
  static constexpr int bQFull = 0;                    // + Q buffer
  static constexpr int bQEmpty = bQFull + kQBufs;     // + Q buffer: the item's products are done
  static constexpr int bKVFull = bQEmpty + kQBufs;    // + stage
  static constexpr int bKVEmpty = bKVFull + kStages;  // + stage
  static constexpr int bSFull = bKVEmpty + kStages;   // + tile
  static constexpr int bPFull = bSFull + 2;           // + tile
  static constexpr int bODone = bPFull + 2;           // + tile
  static constexpr int bSFree = bODone + 2;           // + tile: the softmax holds S_t (split Pbar)
  static constexpr int bPVDone = bSFree + 2;          // + tile: Obar_t += Pbar_t V done (split Pbar)
  static constexpr int bDrain = bPVDone + 2;
  static constexpr int bRegs = bDrain + 1;          // the softmax warps hold their registers
  static constexpr int kNumBars = bRegs + 1;
  static constexpr int kTmemSlot = kBars + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kBytes = kAbort + 4;
  static_assert(kBytes <= 232448, "shared memory budget");
};

template <int D, int MODE, bool CAUSAL, int MON, bool PROFILE, int PBAR = kPbarBf16, bool PAIR = false>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdArgs args) {
  using L = FwdLayout<D, PROFILE, PAIR>;
  static_assert(!PAIR || (MON <= 1 && PBAR == kPbarBf16), "the CTA pairing is built for the fused path");
  constexpr bool kCount = MON >= 1;
  constexpr bool kMonitor = MON >= 2;
  // The repetition flag is needed by the fix modes and by the repeated-row
  // counter, which is reported in every mode.
  constexpr bool kTies = MODE > 0 || kCount;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  PFA_TRACE_DECL();
  // PAIR: the cluster's two CTAs work on one item; the even one (the leader)
  // issues every product of the pair.
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;

  const AttnShape& sh = args.s;
  const int N = sh.N;
  const int n_kt = (N + kTile - 1) / kTile;   // key tiles == query tiles
  // An item is two query tiles of one CTA, or, paired, four: the even CTA's
  // tiles 4g, 4g + 2 and the odd CTA's 4g + 1, 4g + 3 (t = 0 pairs 4g with 4g + 1).
  constexpr int kGroup = PAIR ? 4 : 2;
  const int n_groups = (n_kt + kGroup - 1) / kGroup;
  const int BHq = sh.B * sh.Hq;
  const int n_items = n_groups * BHq;
  const int item0 = static_cast<int>(PAIR ? blockIdx.x >> 1 : blockIdx.x);
  const int stride = static_cast<int>(PAIR ? gridDim.x >> 1 : gridDim.x);
  // The k-th item of this CTA (cluster): rounds of `stride` items, taken left to
  // right in even rounds and right to left in odd ones, so that a CTA given a
  // heavy item early gets a light one in the next round.
  auto item_at = [&](int k) { return k * stride + ((k & 1) ? stride - 1 - item0 : item0); };
  // Work item -> (query tiles, batch and query head); heaviest groups first.
  struct Item {
    int bh, bh_kv, qt0, qt1, last0, last1, n_iter;
    bool has1;
  };
  auto decode = [&](int item) {
    Item it;
    it.bh = item % BHq;
    const int grp = n_groups - 1 - item / BHq;
    const int b = it.bh / sh.Hq, h = it.bh % sh.Hq;
    it.bh_kv = b * sh.Hkv + h / (sh.Hq / sh.Hkv);
    if constexpr (PAIR) {
      // Both CTAs visit the key tiles of the later tile of each product; the
      // earlier tile's rows see the extra diagonal tile fully masked. A tile past
      // the end is loaded as zeros and stores nothing.
      const int base = 4 * grp;
      it.qt0 = base + static_cast<int>(rank);
      it.qt1 = base + 2 + static_cast<int>(rank);
      it.has1 = base + 2 < n_kt;
      it.last0 = CAUSAL ? min(base + 1, n_kt - 1) : n_kt - 1;
      it.last1 = it.has1 ? (CAUSAL ? min(base + 3, n_kt - 1) : n_kt - 1) : -1;
    } else {
      it.qt0 = 2 * grp;
      it.qt1 = it.qt0 + 1;
      it.has1 = it.qt1 < n_kt;
      // Last key tile each query tile visits (-1: the tile does not exist).
      it.last0 = CAUSAL ? it.qt0 : n_kt - 1;
      it.last1 = it.has1 ? (CAUSAL ? it.qt1 : n_kt - 1) : -1;
    }
    it.n_iter = max(it.last0, it.last1) + 1;
    return it;
  };

  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  auto bar = [&](int i) { return sbase + L::kBars + 8u * static_cast<uint32_t>(i); };
  const WaitCtl ctl{abort_flag, args.err, args.err_site, sbase, 1u};

  // PAIR: the leader's Q and K / V barriers complete on its own copies and on one
  // arrival from the odd CTA's warp 1, which forwards the completion of the odd
  // CTA's copies; the leader's PFull_t counts the softmax warps of both CTAs.
  const uint32_t n_full = PAIR && leader ? 2u : 1u;
  if (threadIdx.x == 0) {
    *abort_flag = (sbase & 1023u) ? 1 : 0;
    if (sbase & 1023u) atomicOr(args.err, PFA_DEVERR_SMEM_ALIGN);
    for (int qb = 0; qb < L::kQBufs; ++qb) {
      mbar_init(bar(L::bQFull + qb), n_full);
      mbar_init(bar(L::bQEmpty + qb), 1);
    }
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::bKVFull + s), n_full);
      mbar_init(bar(L::bKVEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(L::bSFull + t), 1);
      mbar_init(bar(L::bPFull + t), PAIR ? 8 : 4);
      mbar_init(bar(L::bODone + t), 1);
      mbar_init(bar(L::bSFree + t), 4);
      mbar_init(bar(L::bPVDone + t), 1);
    }
    mbar_init(bar(L::bDrain), 1);
    mbar_init(bar(L::bRegs), 8);
    fence_mbar_init();
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), 512);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  // PAIR: neither CTA's barriers are signalled by the other before both are set up.
  if constexpr (PAIR) cluster_sync_all();
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Setup done: let the next kernel on the stream be scheduled as CTAs leave, and
  // order every global access after the kernel before this one.
  grid_launch_dependents();
  grid_dependency_wait();
  // Register split per warpgroup. The block is launched with 168 registers per
  // thread (384 x 168 = 64512). Warpgroup 0 (producers, MMA, one idle warp)
  // drops to 64 and the two softmax warpgroups rise to 216: 128 x 64 + 256 x 216
  // = 63488. Each group returns to 168 before the common teardown.
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 64;" ::: "memory");
    if (*abort_flag == 0) {
    if (warp == 0) {
      // ---------------- K / V producer (whole warp, one elected lane issues) ----------------
      // One ring of stages for the key tiles of all items of this CTA.
      tma_prefetch_desc_warp(&tmK);
      tma_prefetch_desc_warp(&tmV);
      int gk = 0;   // key tiles issued
      bool ok = true;
      for (int k = 0, item = item0; ok && item < n_items; ++k, item = item_at(k)) {
        const Item it = decode(item);
        for (int j = 0; j < it.n_iter; ++j, ++gk) {
          const int s = gk % L::kStages;
          if (!(ok = wait_warp(bar(L::bKVEmpty + s), ((gk / L::kStages) & 1) ^ 1, ctl))) break;
          mbar_arrive_expect_tx_warp(bar(L::bKVFull + s), L::kKBytes + L::kVBytes);
          if constexpr (PAIR) {
            // This CTA's half: keys 64 rank .. 64 rank + 63 of K (a map with
            // 64-row boxes), columns 64 rank .. 64 rank + 63 of V.
            for (int p = 0; p < D / 64; ++p)
              tma_load_3d_warp(sbase + L::kK + s * L::kKBytes + p * L::kKPanelBytes, &tmK,
                               bar(L::bKVFull + s), p * 64, j * kTile + 64 * static_cast<int>(rank), it.bh_kv);
            tma_load_3d_warp(sbase + L::kV + s * L::kVBytes, &tmV, bar(L::bKVFull + s),
                             64 * static_cast<int>(rank), j * kTile, it.bh_kv);
          } else {
            for (int p = 0; p < D / 64; ++p) {
              tma_load_3d_warp(sbase + L::kK + s * L::kKBytes + p * L::kKPanelBytes, &tmK,
                               bar(L::bKVFull + s), p * 64, j * kTile, it.bh_kv);
              tma_load_3d_warp(sbase + L::kV + s * L::kVBytes + p * L::kPanelBytes, &tmV,
                               bar(L::bKVFull + s), p * 64, j * kTile, it.bh_kv);
            }
          }
        }
      }
      // Drain: every issued copy has landed before shared memory is released.
      for (int j = gk > L::kStages ? gk - L::kStages : 0; j < gk; ++j)
        wait_drain(bar(L::bKVFull + j % L::kStages), (j / L::kStages) & 1, ctl);
    } else if (warp == 2) {
      // ---------------- Q producer: the pair of query tiles of each item ----------------
      tma_prefetch_desc_warp(&tmQ);
      int ti = 0;   // items issued
      bool ok = true;
      for (int k = 0, item = item0; item < n_items; ++k, item = item_at(k), ++ti) {
        const Item it = decode(item);
        const int qb = ti % L::kQBufs;
        if (!(ok = wait_warp(bar(L::bQEmpty + qb), ((ti / L::kQBufs) & 1) ^ 1, ctl))) break;
        // PAIR: a product reads the tile of both CTAs, so both are always loaded
        // (zeros past the end).
        const int n_t = (PAIR || it.has1) ? 2 : 1;
        mbar_arrive_expect_tx_warp(bar(L::bQFull + qb), n_t * L::kTileBytes);
        for (int t = 0; t < n_t; ++t)
          for (int p = 0; p < D / 64; ++p)
            tma_load_3d_warp(sbase + L::kQ + (qb * 2 + t) * L::kTileBytes + p * L::kPanelBytes, &tmQ,
                             bar(L::bQFull + qb), p * 64, (t ? it.qt1 : it.qt0) * kTile, it.bh);
        // With one Q buffer the next pair waits for this item: start it into L2.
        if (L::kQBufs == 1 && item_at(k + 1) < n_items) {
          const Item nx = decode(item_at(k + 1));
          for (int t = 0; t < (nx.has1 ? 2 : 1); ++t)
            for (int p = 0; p < D / 64; ++p)
              tma_prefetch_l2_3d_warp(&tmQ, p * 64, (t ? nx.qt1 : nx.qt0) * kTile, nx.bh);
        }
      }
      for (int i = ti > L::kQBufs ? ti - L::kQBufs : 0; i < ti; ++i)
        wait_drain(bar(L::bQFull + i % L::kQBufs), (i / L::kQBufs) & 1, ctl);
      (void)ok;
    } else if (warp == 1 && PAIR && !leader) {
      // ---------------- relay (odd CTA of a pair) ----------------
      // Forwards the completion of this CTA's Q and K / V copies to the leader's
      // barriers, in the order in which the leader consumes them.
      int gk = 0, ti = 0;
      bool ok = true;
      for (int k = 0, item = item0; ok && item < n_items; ++k, item = item_at(k), ++ti) {
        const Item it = decode(item);
        const int qb = ti % L::kQBufs;
        if (!(ok = wait_warp(bar(L::bQFull + qb), (ti / L::kQBufs) & 1, ctl))) break;
        if (lane == 0) mbar_arrive_cluster(mapa_shared(bar(L::bQFull + qb), 0));
        for (int j = 0; ok && j < it.n_iter; ++j) {
          const int s = (gk + j) % L::kStages;
          if (!(ok = wait_warp(bar(L::bKVFull + s), ((gk + j) / L::kStages) & 1, ctl))) break;
          if (lane == 0) mbar_arrive_cluster(mapa_shared(bar(L::bKVFull + s), 0));
        }
        gk += it.n_iter;
      }
    } else if (warp == 1) {
      // ---------------- MMA issuer (whole warp, one elected lane issues) ----------------
      // PAIR: M = 256 over the pair's two tiles t; each CTA supplies half of the
      // B operand (K: 64 keys; V: 64 of the d columns) and holds its 128 rows of
      // S_t and Obar_t in its own TMEM. Every commit arrives in both CTAs.
      constexpr int kM = PAIR ? 256 : 128;
      constexpr uint32_t idS = idesc_bf16(kM, 128, false, false);
      constexpr uint32_t idPV = idesc_bf16(kM, D, false, true);
      auto commit = [&](uint32_t b) {
        if constexpr (PAIR) umma_pair_commit_mc_warp(b, 3);
        else umma_commit_warp(b);
      };
      // S_t = Q_t K_j^T from Q buffer qb and K/V stage s.
      auto issue_s = [&](int t, int qb, int s) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t qoff = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
          const uint32_t koff = (kk >> 2) * L::kKPanelBytes + (kk & 3) * 32;
          const uint64_t a = sdesc_sw128(sbase + L::kQ + (qb * 2 + t) * L::kTileBytes + qoff, 16, 1024);
          const uint64_t b = sdesc_sw128(sbase + L::kK + s * L::kKBytes + koff, 16, 1024);
          if constexpr (PAIR) umma_pair_bf16_warp(tmem + 128 * t, a, b, idS, kk > 0);
          else umma_bf16_warp(tmem + 128 * t, a, b, idS, kk > 0);
        }
        commit(bar(L::bSFull + t));
      };
      // Obar_t (+)= Pbar_t V_j; Pbar_t is 64 BF16-pair columns (its own with the
      // split layout, else the first 64 of S_t), 8 columns per K step.
      // The profile's product of each key tile starts afresh in U_t. PAIR: this
      // CTA's V half is one 64-column block, so the block stride is not used (0
      // keeps every address inside that block).
      auto issue_pv = [&](int t, int s, int j) {
        const uint32_t tp = tmem + (L::kSplitP ? L::kColP + 64u * t : 128u * t);
        const uint32_t td = tmem + (PROFILE ? L::kColU + 64u * t : 256u + D * t);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint64_t b = sdesc_sw128(sbase + L::kV + s * L::kVBytes + kk * 2048, PAIR ? 0u : L::kPanelBytes, 1024);
          const uint32_t acc = ((!PROFILE && j > 0) || kk > 0) ? 1u : 0u;
          if constexpr (PAIR) umma_pair_bf16_tmem_a_warp(td, tp + 8 * kk, b, idPV, acc);
          else umma_bf16_tmem_a_warp(td, tp + 8 * kk, b, idPV, acc);
        }
      };
      // Phases across items: gk key tiles so far (the K/V ring), c_t scores of
      // tile t so far (SFull_t and PFull_t), ti items (the Q buffers).
      int gk = 0, c0 = 0, c1 = 0, ti = 0;
      bool ok = true;
      if constexpr (L::kSplitP) {
        // Split Pbar: per key tile j, S_0(j) and S_1(j) (each once its softmax
        // holds the previous scores of its tile), then the products of key tile
        // j - 1 with each tile's Pbar. The scores of the next key tile are thus
        // computed while the softmax works on the current one.
        for (int k = 0, item = item0; ok && item < n_items; ++k, item = item_at(k), ++ti) {
          const Item it = decode(item);
          const int last0 = it.last0, last1 = it.last1, n_iter = it.n_iter;
          const int qb = ti % L::kQBufs;
          if (!(ok = wait_warp<PAIR>(bar(L::bQFull + qb), (ti / L::kQBufs) & 1, ctl))) break;
          for (int j = 0; ok && j <= n_iter; ++j) {
            if (j < n_iter) {
              const int s = (gk + j) % L::kStages;
              if (!(ok = wait_warp<PAIR>(bar(L::bKVFull + s), ((gk + j) / L::kStages) & 1, ctl))) break;
              if (lane == 0) PFA_FWD_TRACE(0, 1, j);
              if (j <= last0) {
                if (c0 + j > 0 && !(ok = wait_warp(bar(L::bSFree + 0), (c0 + j - 1) & 1, ctl))) break;
                tc_fence_after();
                issue_s(0, qb, s);
              }
              if (j <= last1) {
                if (c1 + j > 0 && !(ok = wait_warp(bar(L::bSFree + 1), (c1 + j - 1) & 1, ctl))) break;
                tc_fence_after();
                issue_s(1, qb, s);
              }
            }
            if (j > 0) {
              const int jp = j - 1;
              const int sp = (gk + jp) % L::kStages;
              if (jp <= last0) {
                if (!(ok = wait_warp<PAIR>(bar(L::bPFull + 0), (c0 + jp) & 1, ctl))) break;
                if (lane == 0) PFA_FWD_TRACE(0, 3, jp);
                tc_fence_after();
                issue_pv(0, sp, jp);
                commit(bar(L::bPVDone + 0));
                if (jp == last0) commit(bar(L::bODone + 0));
              }
              if (jp <= last1) {
                if (!(ok = wait_warp<PAIR>(bar(L::bPFull + 1), (c1 + jp) & 1, ctl))) break;
                if (lane == 0) PFA_FWD_TRACE(0, 2, jp);
                tc_fence_after();
                issue_pv(1, sp, jp);
                commit(bar(L::bPVDone + 1));
                if (jp == last1) commit(bar(L::bODone + 1));
              }
              commit(bar(L::bKVEmpty + sp));
            }
          }
          // The item's products are done once this arrives: its Q buffer is free.
          commit(bar(L::bQEmpty + qb));
          gk += n_iter;
          c0 += last0 + 1;
          c1 += last1 + 1;
        }
      } else {
      for (int k = 0, item = item0; ok && item < n_items; ++k, item = item_at(k), ++ti) {
        const Item it = decode(item);
        const int last0 = it.last0, last1 = it.last1, n_iter = it.n_iter;
        const int qb = ti % L::kQBufs;
        if (!(ok = wait_warp<PAIR>(bar(L::bQFull + qb), (ti / L::kQBufs) & 1, ctl))) break;
        for (int j = 0; ok && j < n_iter; ++j) {
          const int s = (gk + j) % L::kStages;
          if (!(ok = wait_warp<PAIR>(bar(L::bKVFull + s), ((gk + j) / L::kStages) & 1, ctl))) break;
          const bool act0 = j <= last0, act1 = j <= last1;
          if (lane == 0) PFA_FWD_TRACE(0, 1, j);
          tc_fence_after();
          if (act0) issue_s(0, qb, s);
          if (j > 0 && j - 1 <= last1) {
            if (!(ok = wait_warp<PAIR>(bar(L::bPFull + 1), (c1 + j - 1) & 1, ctl))) break;
            if (lane == 0) PFA_FWD_TRACE(0, 2, j - 1);
            tc_fence_after();
            const int sp = (gk + j - 1) % L::kStages;
            issue_pv(1, sp, j - 1);
            commit(bar(L::bKVEmpty + sp));
            if (j - 1 == last1) commit(bar(L::bODone + 1));
          }
          if (act1) issue_s(1, qb, s);
          if (act0) {
            if (!(ok = wait_warp<PAIR>(bar(L::bPFull + 0), (c0 + j) & 1, ctl))) break;
            if (lane == 0) PFA_FWD_TRACE(0, 3, j);
            tc_fence_after();
            issue_pv(0, s, j);
            if (j == last0) commit(bar(L::bODone + 0));
            if (!act1) commit(bar(L::bKVEmpty + s));
          }
        }
        if (ok && last1 == n_iter - 1) {
          const int j = n_iter - 1;
          if ((ok = wait_warp<PAIR>(bar(L::bPFull + 1), (c1 + j) & 1, ctl))) {
            tc_fence_after();
            issue_pv(1, (gk + j) % L::kStages, j);
            commit(bar(L::bKVEmpty + (gk + j) % L::kStages));
            commit(bar(L::bODone + 1));
          }
        }
        // The item's products are done once this arrives: its Q buffer is free.
        commit(bar(L::bQEmpty + qb));
        gk += n_iter;
        c0 += last0 + 1;
        c1 += last1 + 1;
      }
      }
      // Drain: no MMA may still read shared memory or write TMEM at teardown.
      if constexpr (PAIR) umma_pair_commit_warp(bar(L::bDrain));
      else umma_commit_warp(bar(L::bDrain));
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
      // ---------------- softmax warps ----------------
      const int t = (warp - 4) >> 2;  // query tile of this warpgroup
      const uint32_t quarter = warp & 3;
      const int r = quarter * 32 + lane;  // row within the tile == TMEM lane
      const uint32_t lane_off = (quarter * 32u) << 16;
      const uint32_t tS = tmem + 128 * t + lane_off;
      const uint32_t tO = tmem + 256 + D * t + lane_off;
      const uint32_t tP = L::kSplitP ? tmem + L::kColP + 64 * t + lane_off : tS;   // Pbar_t
      const uint32_t tU = tmem + L::kColU + 64 * t + lane_off;                      // profile: Pbar_t V
      const float sl2 = sh.scale_log2;
      const float alpha = sh.scale;

      // Profile: Obar (BF16 values held in the FP32 Obar columns) becomes
      // bf16(bf16(Obar x c) + bf16(U)), U the last tile's product; `acc` is false
      // while Obar holds nothing yet.
      auto fold_profile = [&](bool acc, float c) {
        if constexpr (PROFILE) {
#pragma unroll 1
          for (int cc = 0; cc < D; cc += 32) {
            uint32_t u[32], o[32];
            tmem_ld32(tU + cc, u);
            tmem_ld32(tO + cc, o);
            tmem_ld_wait32(u);
            tmem_ld_wait32(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const float ub = bf16_round(__uint_as_float(u[e]));
              const float ob = acc ? bf16_round(__uint_as_float(o[e]) * c) : 0.f;
              o[e] = __float_as_uint(bf16_round(ob + ub));
            }
            tmem_st32(tO + cc, o);
          }
        }
      };

      // Shift rule (paper §4 equation; Algorithm 1): only rows whose maximum
      // repeats within eps change their shift.
      auto shift_of = [&](float mx, bool repeated) {
        const float r_m = mx * alpha;
        if (MODE == 0 || !repeated) return r_m;
        if (MODE == 1) return r_m > 0.f ? args.beta * r_m : (r_m < 0.f ? 0.f : kEpsShift);
        return r_m + kEpsShift;
      };
      bool ok = true;
      int ct = 0, ot = 0;   // phases across items: scores of this tile, items with this tile
      for (int k = 0, item = item0; ok && item < n_items; ++k, item = item_at(k)) {
      const Item itm = decode(item);
      const int last = t ? itm.last1 : itm.last0;
      if (last < 0) continue;             // the pair has no second tile
      const int bh = itm.bh;
      const int q0 = (t ? itm.qt1 : itm.qt0) * kTile;
      const int qrow = q0 + r;
      const bool row_ok = qrow < N;
      float m1 = -INFINITY;                  // running maximum of raw scores
      bool rep = false;                      // two entries within eps of m1
      float m_sh = -INFINITY;                // current shift, natural units
      float l0 = 0.f, l1 = 0.f;              // row sum of Pbar (two partial sums)
      int cnt = 0;                           // entries within tau of m1 (raw)
      int cnt_eps = 0;                       // entries within eps of m1 (raw; monitor)
      long long ones_op = 0;                 // BF16 Pbar == 1 handed to the product (monitor)
      float corr_prev = 1.f;                 // profile: the rescale of the previous tile

      for (int j = 0; j <= last; ++j) {
        const int k0 = j * kTile;
        const bool need_mask = (CAUSAL && k0 + kTile > q0) || (k0 + kTile > N);
        if (!(ok = wait_warp(bar(L::bSFull + t), (ct + j) & 1, ctl))) break;
        if (lane == 0 && quarter == 0) PFA_FWD_TRACE(1 + t, 4, j);
        tc_fence_after();
        uint32_t v[128];
        tmem_ld64(tS, v);
        tmem_ld64(tS + 64, v + 64);
        tmem_ld_wait64(v);
        tmem_ld_wait64(v + 64);
        if constexpr (L::kSplitP) {
          // The scores are in registers: the next S_t may overwrite them.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(L::bSFree + t));
        }
        if (need_mask) {
#pragma unroll
          for (int c = 0; c < kTile; ++c) {
            const int key = k0 + c;
            if (!(key < N && (!CAUSAL || key <= qrow))) v[c] = __float_as_uint(-INFINITY);
          }
        }
        // Tile maximum, as the maxima of eight blocks of 16 columns.
        float bm[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          auto x = [&](int e) { return __uint_as_float(v[16 * k + e]); };
          const float u0 = fmax3(x(0), x(1), x(2)), u1 = fmax3(x(3), x(4), x(5));
          const float u2 = fmax3(x(6), x(7), x(8)), u3 = fmax3(x(9), x(10), x(11));
          const float u4 = fmax3(x(12), x(13), x(14));
          bm[k] = fmaxf(fmax3(u0, u1, u2), fmax3(u3, u4, x(15)));
        }
        const float t1 = fmax3(fmax3(bm[0], bm[1], bm[2]), fmax3(bm[3], bm[4], bm[5]), fmaxf(bm[6], bm[7]));
        // Repetition flag of the running row (at least two entries within eps of
        // its maximum), kept exactly tile by tile without a second maximum:
        //   new maximum t1 > m1: repeated iff m1 >= t1 - eps or this tile holds two
        //                        entries >= t1 - eps;
        //   m1 - eps <= t1 <= m1: repeated (an entry of this tile ties the maximum);
        //   otherwise the flag is unchanged.
        // Two entries of the tile reach a threshold iff two of the eight 16-column
        // blocks do or two of the sixteen column classes (column mod 16) do: a
        // single qualifying entry lies in one block and one class, and two
        // distinct entries differ in their block or in their class. The block
        // count is known with the maximum, and only warps where some row jumps
        // count it. Only warps where some row's new maximum is alone in its block
        // take the class maxima, before the exponentials, so every tile is
        // exponentiated once, under its final shift, and the scores can die as
        // the exponentials consume them.
        bool jump = false;
        int nb = 0;
        float thr_eps = 0.f;
        bool rep_use = rep;
        if (kTies) {
          thr_eps = t1 - args.eps_raw;
          jump = t1 > m1 && m1 < thr_eps;
          if (__any_sync(0xFFFFFFFFu, jump)) {
#pragma unroll
            for (int k = 0; k < 8; ++k) nb += bm[k] >= thr_eps ? 1 : 0;
          }
          if (t1 > m1) {
            rep_use = jump ? nb >= 2 : true;
          } else if (t1 >= m1 - args.eps_raw && t1 > -INFINITY) {
            rep_use = true;
          }
          if (__any_sync(0xFFFFFFFFu, jump && nb < 2)) {
            // Class maxima (column mod 16) over the whole tile.
            int ne = 0;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              auto x = [&](int k) { return __uint_as_float(v[16 * k + e]); };
              const float c = fmax3(fmax3(x(0), x(1), x(2)), fmax3(x(3), x(4), x(5)), fmaxf(x(6), x(7)));
              ne += c >= thr_eps ? 1 : 0;
            }
            if (jump && nb < 2 && ne >= 2) rep_use = true;
          }
        }
        const float m1_old = m1;
        m1 = fmaxf(m1, t1);
        if (lane == 0 && quarter == 0) PFA_FWD_TRACE(1 + t, 5, j);

        // Pbar = exp(S - m) in FP32; l sums it (the profile sums its BF16 cast); the
        // BF16 casts go to TMEM.
        const float m_new = shift_of(m1, rep_use);
        const bool changed = (j > 0) && (m_new != m_sh);
        const float corr = changed ? ex2_approx((m_sh - m_new) * kLog2e) : 1.f;
        l0 *= corr;
        l1 *= corr;
        int cnt_tile = 0, eps_tile = 0, ones_tile = 0;
        {
          const float nml2 = -m_new * kLog2e;
          const float thr = m1 - args.tau_raw;
          const float thr_e = m1 - args.eps_raw;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t pk[32];
            // Pbar pair u (FP32) into the BF16 operand, the row sum and the monitor. With
            // a narrow Pbar format the pair arrives already rounded to it (its values are
            // exact in BF16) and l sums those values, the weights the product uses.
            auto finish = [&](int u, float p0, float p1) {
              pk[u] = pack_bf16x2(p0, p1);
              if constexpr (PBAR != kPbarBf16) {
                add2(l0, l1, p0, p1);
                if (kMonitor) ones_tile += (p0 == 1.f) + (p1 == 1.f);
              } else {
                if constexpr (PROFILE) {
                  // The profile normalises by the weights its product uses: BF16 Pbar.
                  add2(l0, l1, bf16lo_to_f32(pk[u]), bf16hi_to_f32(pk[u]));
                } else {
                  add2(l0, l1, p0, p1);
                }
                // BF16(Pbar) == 1 exactly when Pbar >= 1 - 2^-9 (Pbar <= 1 here).
                if (kMonitor) ones_tile += (p0 >= kBf16OneThreshold) + (p1 >= kBf16OneThreshold);
              }
            };
            [[maybe_unused]] float pm[PBAR == kPbarMxfp4 ? 64 : 1];
#pragma unroll
            for (int u = 0; u < 32; ++u) {
              const float x0 = __uint_as_float(v[64 * half + 2 * u]);
              const float x1 = __uint_as_float(v[64 * half + 2 * u + 1]);
              if (kCount) cnt_tile += (x0 >= thr) + (x1 >= thr);
              if (kMonitor) eps_tile += (x0 >= thr_e) + (x1 >= thr_e);
              float y0, y1;
              if constexpr (PBAR != kPbarBf16) {
                // The exponent as (alpha x - m) log2 e, so that it is exactly 0 where the score
                // is the shift: a narrow format's rounding (and MXFP4's power-of-two scale)
                // turns on whether Pbar is 1 or just below it.
                // Rounded operations that are never contracted into an FMA.
                y0 = __fmul_rn(__fsub_rn(__fmul_rn(x0, alpha), m_new), kLog2e);
                y1 = __fmul_rn(__fsub_rn(__fmul_rn(x1, alpha), m_new), kLog2e);
              } else {
                fma2(y0, y1, x0, x1, sl2, nml2);
              }
              float p0 = ex2_approx(y0), p1 = ex2_approx(y1);
              if constexpr (PBAR == kPbarMxfp4) {
                pm[2 * u] = p0;
                pm[2 * u + 1] = p1;
              } else {
                if constexpr (PBAR == kPbarE4m3) e4m3_round2(p0, p1);
                finish(u, p0, p1);
              }
            }
            if constexpr (PBAR == kPbarMxfp4) {
              // MXFP4: 32 consecutive keys share the scale X = 2^(floor(log2 amax) - 2);
              // each Pbar becomes X E2M1(Pbar / X), saturating at 6 X.
#pragma unroll
              for (int blk = 0; blk < 2; ++blk) {
                float amax = 0.f;
#pragma unroll
                for (int e = 0; e < 32; e += 2) amax = fmax3(amax, pm[32 * blk + e], pm[32 * blk + e + 1]);
                const int ex = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu) - 127;
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                  float a = 0.f, b = 0.f;
                  if (amax > 0.f) {
                    a = ldexpf(pm[32 * blk + e], 2 - ex);
                    b = ldexpf(pm[32 * blk + e + 1], 2 - ex);
                    e2m1_round2(a, b);
                    a = ldexpf(a, ex - 2);
                    b = ldexpf(b, ex - 2);
                  }
                  finish(16 * blk + e / 2, a, b);
                }
              }
            }
            if constexpr (L::kSplitP) {
              // Obar_t and the Pbar_t columns are free once the previous key
              // tile's product has completed (tile 0 of an item: its epilogue
              // waited for the last product of the previous item). Without split
              // Pbar, S_t of this tile was committed after that product.
              // A failed wait ends the loop at the bottom of this iteration.
              if (half == 0 && j > 0) {
                ok = wait_warp(bar(L::bPVDone + t), (ct + j - 1) & 1, ctl);
                tc_fence_after();
              }
            }
            tmem_st32(tP + 32 * half, pk);
          }
        }
        rep = rep_use;
        if (kCount) cnt = (m1 - m1_old > args.tau_raw) ? cnt_tile : cnt + cnt_tile;
        if (kMonitor) {
          cnt_eps = (m1 - m1_old > args.eps_raw) ? eps_tile : cnt_eps + eps_tile;
          ones_op += row_ok ? ones_tile : 0;
        }
        if (lane == 0 && quarter == 0) PFA_FWD_TRACE(1 + t, 6, j);
        if constexpr (PROFILE) {
          // Fold the previous tile's product, complete since S_t of this tile was
          // committed after it: Obar = bf16(bf16(Obar x corr) + bf16(P V)), the
          // rescale being the one that tile computed.
          if (j > 0) fold_profile(j > 1, corr_prev);
          corr_prev = corr;
        } else if (__any_sync(0xFFFFFFFFu, changed)) {
          // Rescale Obar where the shift moved: the scores are dead, so one TMEM
          // round trip covers 64 columns.
#pragma unroll 1
          for (int c = 0; c < D; c += 64) {
            uint32_t o[64];
            tmem_ld64(tO + c, o);
            tmem_ld_wait64(o);
#pragma unroll
            for (int u = 0; u < 64; u += 2) {
              float y0 = __uint_as_float(o[u]), y1 = __uint_as_float(o[u + 1]);
              mul2(y0, y1, corr);
              o[u] = __float_as_uint(y0);
              o[u + 1] = __float_as_uint(y1);
            }
            tmem_st64(tO + c, o);
          }
        }
        m_sh = m_new;
        tmem_st_wait();
        if (lane == 0 && quarter == 0) PFA_FWD_TRACE(1 + t, 7, j);
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && ok) {
          // PAIR: the leader's PFull_t, which counts both CTAs' softmax warps; only
          // the odd CTA's arrivals need the release at cluster scope.
          if (PAIR && !leader) mbar_arrive_cluster(mapa_shared(bar(L::bPFull + t), 0));
          else mbar_arrive(bar(L::bPFull + t));
        }

        if (lane == 0 && quarter == 0) PFA_FWD_TRACE(1 + t, 8, j);
        if (!ok) break;
      }

      // ---------------- epilogue ----------------
      if (ok) ok = wait_warp(bar(L::bODone + t), ot & 1, ctl);
      if (lane == 0 && quarter == 0) PFA_FWD_TRACE(1 + t, 9, ot);
      if (ok) {
        tc_fence_after();
        if constexpr (PROFILE) {
          fold_profile(last > 0, corr_prev);   // the last tile's product
          tmem_st_wait();
        }
        // The flag is exact after every tile, so the shift in use is the final one.
        const float m_fin = m_sh;
        const float l = l0 + l1;
        const float inv_l = 1.f / l;
        __nv_bfloat16* orow =
            reinterpret_cast<__nv_bfloat16*>(args.o) + (static_cast<size_t>(bh) * N + qrow) * D;
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c, o);
          tmem_ld_wait32(o);
          uint32_t pk[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            float y0 = __uint_as_float(o[2 * u]), y1 = __uint_as_float(o[2 * u + 1]);
            mul2(y0, y1, inv_l);
            pk[u] = pack_bf16x2(y0, y1);
          }
          if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
            for (int qd = 0; qd < 4; ++qd)
              dst[qd] = make_uint4(pk[4 * qd], pk[4 * qd + 1], pk[4 * qd + 2], pk[4 * qd + 3]);
          }
        }
        if (lane == 0 && quarter == 0) PFA_FWD_TRACE(1 + t, 10, ot);
        if (row_ok) args.lse[static_cast<size_t>(bh) * N + qrow] = m_fin + lg2_approx(l) * kLn2;
        if (kCount) {
          // BF16(Pbar) == 1 under the final shift: entries within tau of m1,
          // unless the shift moved the maximum more than tau below zero.
          const float moved = m_fin - m1 * alpha;
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
        if (kMonitor && args.monitor) {
          // Operational ones of this row over all its tiles, and the row's tie
          // multiplicity (entries within eps of its maximum) into bins 1..7, >= 8.
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) ones_op += __shfl_xor_sync(0xFFFFFFFFu, ones_op, o);
          if (lane == 0 && ones_op)
            atomicAdd(reinterpret_cast<unsigned long long*>(args.monitor), static_cast<unsigned long long>(ones_op));
          const int bin = min(max(cnt_eps, 1), kTieBins) - 1;
#pragma unroll
          for (int b = 0; b < kTieBins; ++b) {
            const unsigned nbin = __popc(__ballot_sync(0xFFFFFFFFu, row_ok && bin == b));
            if (lane == 0 && nbin)
              atomicAdd(reinterpret_cast<unsigned long long*>(args.monitor + 1 + b), static_cast<unsigned long long>(nbin));
          }
        }
      }
      ct += last + 1;
      ++ot;
      }
    }
    asm volatile("setmaxnreg.dec.sync.aligned.u32 168;" ::: "memory");
  }

  tc_fence_before();
  __syncthreads();
  // PAIR: neither CTA frees its TMEM or leaves while the leader's products or
  // the other CTA's arrivals may still reach it.
  if constexpr (PAIR) cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem, 512);
    else tmem_dealloc(tmem, 512);
  }
}

template <int D, int MODE, bool CAUSAL, int MON, bool PROFILE, int PBAR = kPbarBf16>
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const FwdArgs& a, cudaStream_t stream) {
  using L = FwdLayout<D, PROFILE>;
  auto kern = attn_fwd_kernel<D, MODE, CAUSAL, MON, PROFILE, PBAR>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  if (e != cudaSuccess) return e;
  // Persistent: one CTA per SM (at most one per work item).
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int n_kt = (a.s.N + kTile - 1) / kTile;
  const long long n_items = static_cast<long long>((n_kt + 1) / 2) * a.s.B * a.s.Hq;
  const dim3 grid(static_cast<unsigned>(n_items < sms ? n_items : sms));
  return launch_pdl(kern, grid, dim3(kThreads), L::kBytes, stream, tq, tk, tv, a);
}

// The paired fused path at d = 128: clusters of two CTAs, as many as the device
// holds at once (at most one per item of four query tiles), launched as a
// programmatic dependent like the others. `tk` maps K with 64-row boxes.
template <int MODE, bool CAUSAL, int MON>
cudaError_t launch_fwd_pair_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const FwdArgs& a, cudaStream_t stream) {
  using L = FwdLayout<128, false, true>;
  auto kern = attn_fwd_kernel<128, MODE, CAUSAL, MON, false, kPbarBf16, true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if ((e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg)) != cudaSuccess) return e;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  const int n_kt = (a.s.N + kTile - 1) / kTile;
  const long long n_items = static_cast<long long>((n_kt + 3) / 4) * a.s.B * a.s.Hq;
  cfg.gridDim = dim3(2u * static_cast<unsigned>(n_items < clusters ? n_items : clusters));
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, a);
}

}  // namespace fwd
}  // namespace pfa
