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
// Persistent: one CTA per SM works through items = (batch, query head, 128-row
// query tile), heaviest causal tiles first, dealt in serpentine rounds of
// gridDim.x. Barrier phases count across items: the K / V ring (2 stages), the
// half-tile buffers and the Q / dO buffers (2 at d = 64, 1 at d = 128) run on from
// one item to the next, and dQ is double-buffered in TMEM, so an item's epilogue
// overlaps the next item's products.
// 320 threads: warp 0 TMA producer, warp 1 TMEM owner and MMA issuer, warps 2..9
// compute. Each 128-key tile is processed as two 64-key halves, in two TMEM
// buffers b = (half-tile count) % 2 at [128 b, 128 b + 128): S_u = Q K_u^T in the
// first 64 columns, dP_u = dO V_u^T in the next 64; the dQ buffers sit at
// [256 + d db, 256 + d db + d). Compute warp w handles TMEM lane quarter w % 4
// (32 query rows) and the 32 keys [32 c, 32 c + 32) of each half, c = (w - 2) / 4,
// so each SM sub-partition runs two compute warps. dS (BF16, two keys per 32-bit
// column) is written over the S columns the warp has read: its 32 keys occupy
// [32 c, 32 c + 32) of the half's S, hi in the first 16 columns and lo in the
// next 16, so key step kk (16 keys) of the dQ product reads hi at
// 32 (kk / 2) + 8 (kk % 2).
// Tensor-core order per item: S, dP of its first two halves, then per half u:
// dQ_u, S_(u+2), dP_(u+2). The compute warps form dS_(u+1) while the tensor core
// runs dQ_u and S_(u+2), and in-order execution keeps S_(u+2) (same buffer) from
// overwriting dS_u before dQ_u has read it.
#include "pfa_device.cuh"

namespace pfa {
namespace {

constexpr int kThreads = 320;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kHalf = kTile / 2;   // keys of one half-tile

template <int D>
struct DqLayout {
  static constexpr int kStages = 2;                      // K / V ring
  static constexpr int kQBufs = (D == 64) ? 2 : 1;       // Q / dO buffers
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kPanelBytes = kTile * 128;
  static constexpr int kQ = 0;                           // + buffer * 2 tiles: Q, then dO
  static constexpr int kK = kQBufs * 2 * kTileBytes;     // + stage * tile
  static constexpr int kV = kK + kStages * kTileBytes;   // + stage * tile
  static constexpr int kBars = kV + kStages * kTileBytes;
  static constexpr int bQFull = 0;                       // + Q buffer
  static constexpr int bQEmpty = bQFull + kQBufs;        // + Q buffer: the item's S, dP products are done
  static constexpr int bKVFull = bQEmpty + kQBufs;       // + stage
  static constexpr int bKVEmpty = bKVFull + kStages;     // + stage
  static constexpr int bSFull = bKVEmpty + kStages;      // + half buffer: S_u and dP_u are in TMEM
  static constexpr int bDSReady = bSFull + 2;            // + half buffer: the compute warps wrote dS_u
  static constexpr int bDQFull = bDSReady + 2;           // + dQ buffer: the item's last dQ product completed
  static constexpr int bDQFree = bDQFull + 2;            // + dQ buffer: the compute warps read it out
  static constexpr int bDrain = bDQFree + 2;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kTmemSlot = kBars + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kBytes = kAbort + 4;
  static constexpr uint32_t kColDQ = 256;                // + D * dQ buffer
  static_assert(kColDQ + 2 * D <= 512, "TMEM columns");
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
  const int n_items = n_t * BHq;
  const int item0 = static_cast<int>(blockIdx.x);
  const int stride = static_cast<int>(gridDim.x);
  // The k-th item of this CTA: rounds of gridDim.x items, taken left to right in
  // even rounds and right to left in odd ones, so that a CTA given a heavy item
  // early gets a light one in the next round.
  auto item_at = [&](int k) { return k * stride + ((k & 1) ? stride - 1 - item0 : item0); };
  // Work item -> (query tile, batch and query head); query tiles heaviest first.
  struct Item {
    int bh, bh_kv, q0, n_kt;
  };
  auto decode = [&](int item) {
    Item it;
    it.bh = item % BHq;
    const int qt = n_t - 1 - item / BHq;
    const int b = it.bh / sh.Hq, h = it.bh % sh.Hq;
    it.bh_kv = b * sh.Hkv + h / (sh.Hq / sh.Hkv);
    it.q0 = qt * kTile;
    it.n_kt = CAUSAL ? qt + 1 : n_t;
    return it;
  };

  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  auto bar = [&](int i) { return sbase + L::kBars + 8u * static_cast<uint32_t>(i); };
  const WaitCtl ctl{abort_flag, args.err, args.err_site, sbase, 5u};

  if (threadIdx.x == 0) {
    *abort_flag = (sbase & 1023u) ? 1 : 0;
    if (sbase & 1023u) atomicOr(args.err, PFA_DEVERR_SMEM_ALIGN);
    for (int qb = 0; qb < L::kQBufs; ++qb) {
      mbar_init(bar(L::bQFull + qb), 1);
      mbar_init(bar(L::bQEmpty + qb), 1);
    }
    for (int st = 0; st < L::kStages; ++st) {
      mbar_init(bar(L::bKVFull + st), 1);
      mbar_init(bar(L::bKVEmpty + st), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(L::bSFull + x), 1);
      mbar_init(bar(L::bDSReady + x), 8);
      mbar_init(bar(L::bDQFull + x), 1);
      mbar_init(bar(L::bDQFree + x), 8);
    }
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
      int gk = 0;   // key tiles issued (all items): the K / V ring
      int ti = 0;   // items issued: the Q / dO buffers
      bool ok = true;
      for (int k = 0, item = item0; ok && item < n_items; ++k, item = item_at(k), ++ti) {
        const Item it = decode(item);
        const int qb = ti % L::kQBufs;
        if (!(ok = wait_warp(bar(L::bQEmpty + qb), ((ti / L::kQBufs) & 1) ^ 1, ctl))) break;
        mbar_arrive_expect_tx_warp(bar(L::bQFull + qb), 2 * L::kTileBytes);
        for (int p = 0; p < D / 64; ++p) {
          tma_load_3d_warp(sbase + L::kQ + (2 * qb) * L::kTileBytes + p * L::kPanelBytes, &tmQ,
                           bar(L::bQFull + qb), p * 64, it.q0, it.bh);
          tma_load_3d_warp(sbase + L::kQ + (2 * qb + 1) * L::kTileBytes + p * L::kPanelBytes, &tmdO,
                           bar(L::bQFull + qb), p * 64, it.q0, it.bh);
        }
        for (int j = 0; j < it.n_kt; ++j, ++gk) {
          const int st = gk % L::kStages;
          if (!(ok = wait_warp(bar(L::bKVEmpty + st), ((gk / L::kStages) & 1) ^ 1, ctl))) break;
          mbar_arrive_expect_tx_warp(bar(L::bKVFull + st), 2 * L::kTileBytes);
          for (int p = 0; p < D / 64; ++p) {
            tma_load_3d_warp(sbase + L::kK + st * L::kTileBytes + p * L::kPanelBytes, &tmK,
                             bar(L::bKVFull + st), p * 64, j * kTile, it.bh_kv);
            tma_load_3d_warp(sbase + L::kV + st * L::kTileBytes + p * L::kPanelBytes, &tmV,
                             bar(L::bKVFull + st), p * 64, j * kTile, it.bh_kv);
          }
        }
      }
      // Every issued copy has landed before shared memory is released (earlier
      // ones were consumed before later ones could reuse their buffer).
      for (int i = ti > L::kQBufs ? ti - L::kQBufs : 0; i < ti; ++i)
        wait_drain(bar(L::bQFull + i % L::kQBufs), (i / L::kQBufs) & 1, ctl);
      for (int j = gk > L::kStages ? gk - L::kStages : 0; j < gk; ++j)
        wait_drain(bar(L::bKVFull + j % L::kStages), (j / L::kStages) & 1, ctl);
    } else if (warp == 1) {
      // ---------------- MMA issuer (whole warp, one elected lane issues) ----------------
      constexpr uint32_t idS = idesc_bf16(128, kHalf, false, false);  // S_u, dP_u: N = 64 keys
      constexpr uint32_t idDQ = idesc_bf16(128, D, false, true);      // dQ: A = dS in TMEM, B = K MN-major
      // Global counters: g half-tiles (their buffer and phases), gk key tiles (the
      // K / V ring), ti items (the Q / dO and dQ buffers).
      int g = 0, gk = 0, ti = 0;
      // S_u = Q K_u^T and dP_u = dO V_u^T into half buffer g_u % 2; K_u, V_u are rows
      // [64 (u % 2), 64 (u % 2) + 64) of the key tile in stage st.
      auto issue_sdp = [&](int gu, int u, int qb, int st) {
        const uint32_t tb = tmem + 128u * static_cast<uint32_t>(gu & 1);
        const uint32_t hoff = static_cast<uint32_t>(u & 1) * kHalf * 128;
        const uint32_t sQ = sbase + L::kQ + (2 * qb) * L::kTileBytes;
        const uint32_t sDO = sbase + L::kQ + (2 * qb + 1) * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
          umma_bf16_warp(tb, sdesc_sw128(sQ + koff, 16, 1024),
                         sdesc_sw128(sbase + L::kK + st * L::kTileBytes + hoff + koff, 16, 1024), idS, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
          umma_bf16_warp(tb + kHalf, sdesc_sw128(sDO + koff, 16, 1024),
                         sdesc_sw128(sbase + L::kV + st * L::kTileBytes + hoff + koff, 16, 1024), idS, kk > 0);
        }
        umma_commit_warp(bar(L::bSFull + (gu & 1)));
      };
      // Q and dO are read only by S and dP: the item's last pair frees their buffer.
      auto sdp = [&](int gu, int u, int n_u, int qb, int st) {
        issue_sdp(gu, u, qb, st);
        if (u == n_u - 1) umma_commit_warp(bar(L::bQEmpty + qb));
      };
      // dQ (+)= dS_u K_u into dQ buffer db: hi, then lo into the same accumulator.
      auto issue_dq = [&](int gu, int u, int db, int st) {
        const uint32_t tb = tmem + 128u * static_cast<uint32_t>(gu & 1);
        const uint32_t sK = sbase + L::kK + st * L::kTileBytes;
        const uint32_t td = tmem + L::kColDQ + static_cast<uint32_t>(D * db);
        const int h4 = 4 * (u & 1);   // the half's first key step within the tile
#pragma unroll
        for (int kk = 0; kk < kHalf / 16; ++kk)
          umma_bf16_tmem_a_warp(td, tb + ds_col(kk), sdesc_sw128(sK + (h4 + kk) * 2048, L::kPanelBytes, 1024),
                                idDQ, (u > 0 || kk > 0) ? 1u : 0u);
        if constexpr (SPLIT) {
#pragma unroll
          for (int kk = 0; kk < kHalf / 16; ++kk)
            umma_bf16_tmem_a_warp(td, tb + ds_col(kk) + 16u,
                                  sdesc_sw128(sK + (h4 + kk) * 2048, L::kPanelBytes, 1024), idDQ, 1u);
        }
        // The second half's product is the last reader of the tile's K and V.
        if (u & 1) umma_commit_warp(bar(L::bKVEmpty + st));
      };
      // The first half of key tile j waits for the tile in shared memory.
      auto tile_ready = [&](int u) {
        if (u & 1) return true;
        const int gj = gk + (u >> 1);
        return wait_warp(bar(L::bKVFull + gj % L::kStages), (gj / L::kStages) & 1, ctl);
      };
      bool ok = true;
      for (int k = 0, item = item0; ok && item < n_items; ++k, item = item_at(k), ++ti) {
        const Item it = decode(item);
        const int qb = ti % L::kQBufs, db = ti & 1;
        const int n_u = 2 * it.n_kt;
        if (!(ok = wait_warp(bar(L::bQFull + qb), (ti / L::kQBufs) & 1, ctl))) break;
        for (int u = 0; ok && u < 2; ++u) {
          if (!(ok = tile_ready(u))) break;
          tc_fence_after();
          sdp(g + u, u, n_u, qb, (gk + (u >> 1)) % L::kStages);
        }
        // The dQ buffer is free once the compute warps have read out the item two back.
        if (ok && ti >= 2) ok = wait_warp(bar(L::bDQFree + db), ((ti >> 1) - 1) & 1, ctl);
        for (int u = 0; ok && u < n_u; ++u) {
          if (!(ok = wait_warp(bar(L::bDSReady + ((g + u) & 1)), ((g + u) >> 1) & 1, ctl))) break;
          tc_fence_after();
          issue_dq(g + u, u, db, (gk + (u >> 1)) % L::kStages);
          if (u + 2 < n_u) {
            if (!(ok = tile_ready(u + 2))) break;
            tc_fence_after();
            sdp(g + u + 2, u + 2, n_u, qb, (gk + ((u + 2) >> 1)) % L::kStages);
          }
        }
        if (!ok) break;
        umma_commit_warp(bar(L::bDQFull + db));   // the item's dQ is complete
        g += n_u;
        gk += it.n_kt;
      }
      // No MMA may still read shared memory or write TMEM at teardown.
      umma_commit_warp(bar(L::bDrain));
      wait_drain(bar(L::bDrain), 0, ctl);
    } else {
      // ---------------- compute warps ----------------
      const uint32_t quarter = warp & 3;
      const int c = (warp - 2) >> 2;             // keys [32 c, 32 c + 32) of each half
      const int r = quarter * 32 + lane;         // query row within the tile == TMEM lane
      const uint32_t lane_off = (quarter * 32u) << 16;
      const float sl2 = sh.scale_log2;
      bool ok = true;
      int g = 0, ti = 0;
      for (int k = 0, item = item0; ok && item < n_items; ++k, item = item_at(k), ++ti) {
        const Item it = decode(item);
        const int db = ti & 1;
        const int n_u = 2 * it.n_kt;
        const int qrow = it.q0 + r;
        const bool row_ok = qrow < N;
        const size_t rowi = static_cast<size_t>(it.bh) * N + qrow;
        // -lse (log2 units) and -delta of this row; rows past N take no part.
        const float nlse2 = row_ok ? -args.lse[rowi] * kLog2e : -INFINITY;
        const float ndelta = row_ok ? -args.delta[rowi] : 0.f;
        for (int u = 0; u < n_u; ++u) {
          const int gu = g + u;
          const int k0 = (u >> 1) * kTile + (u & 1) * kHalf + 32 * c;   // this warp's first key
          const bool need_mask = (CAUSAL && k0 + 32 > it.q0) || (k0 + 32 > N);
          const uint32_t tb = tmem + 128u * static_cast<uint32_t>(gu & 1) + lane_off + 32u * c;
          if (!(ok = wait_warp(bar(L::bSFull + (gu & 1)), (gu >> 1) & 1, ctl))) break;
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
          if (lane == 0) mbar_arrive(bar(L::bDSReady + (gu & 1)));
        }
        // ---------------- epilogue: dQ = alpha (sum of dS K) -> BF16 ----------------
        if (ok) ok = wait_warp(bar(L::bDQFull + db), (ti >> 1) & 1, ctl);
        if (!ok) break;
        tc_fence_after();
        constexpr int kCols = D / 2;   // this warp's dQ columns [kCols c, kCols c + kCols)
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(args.dq) + rowi * D + kCols * c;
        const uint32_t td = tmem + L::kColDQ + static_cast<uint32_t>(D * db) + lane_off + kCols * c;
#pragma unroll 1
        for (int cc = 0; cc < kCols; cc += 32) {
          uint32_t v[32];
          tmem_ld32(td + cc, v);
          tmem_ld_wait32(v);
          if (cc + 32 >= kCols) {
            // The buffer is read out: the item two on may accumulate into it.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::bDQFree + db));
          }
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
        g += n_u;
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
  // Persistent: one CTA per SM (at most one per work item).
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int n_t = (a.s.N + kTile - 1) / kTile;
  const long long n_items = static_cast<long long>(n_t) * a.s.B * a.s.Hq;
  const dim3 grid(static_cast<unsigned>(n_items < sms ? n_items : sms));
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
