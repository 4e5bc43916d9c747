// Short-query backward (all activations), sm_103a.
//
// "GEM Training ..." GDPA paragraph (PMA: a few seed queries over long jagged
// keys; kernels reworked for short / asymmetric shapes) and JFA paragraph
// (efficient backward passes).  The gradients are those of the main backward
// kernels:
//   dV = P^T dO,  dP = dO V^T,  dS = act'(S) dP  or  P (dP - D),
//   dQ = scale dS K,  dK = scale dS^T Q.
//
// Work item: one (sample, head) with Lq <= 32 queries (the scheduler's
// short-query list).  Q, dO, lse and D of the item stay in shared memory;
// the sample's 128-key K/V tiles stream through a two-stage ring.  Per tile,
// with TMEM lanes = keys and the queries as the MMA's N:
//   S^T = K Q^T, dP^T = V dO^T       (M = 128, N = 32, K = d)
//   P^T, dS^T                        activation warps: packed bf16 into TMEM
//                                    (A operands), dS also into shared memory;
//                                    for GDPA activations each as bf16 hi + lo
//                                    (two MMAs): the terms of dK and dQ are large
//                                    and cancel, so a single bf16 rounding of dS
//                                    shows in the sums
//   dV = P^T dO, dK = dS^T Q         (M = 128, N = d, K = 32): complete for the
//                                    tile, since every query is present; the
//                                    epilogue warps store them
//   dQ^T += K^T dS^T                 (M = d, N = 32, K = 128) in TMEM across all
//                                    key tiles of the item, stored once at the
//                                    end with plain stores: no reduce-add.  When
//                                    every sample is short, dQ goes out in bf16
//                                    and the fp32 accumulator is not used at all.
//
// Warps: 0-3 activation, 4-7 epilogue (dK / dV rows; dQ at the item's end),
// 8 producer, 9 MMA.  Every wait is bounded.
#include "common.cuh"

namespace gdpa {
namespace {

using namespace ptx;

constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kStages = 2;
constexpr float kLog2e = 1.4426950408889634f;
// TMEM columns: S^T, dP^T; P^T and dS^T as packed bf16 (16 columns each for
// hi, then 16 for lo); dQ^T; dV; dK
constexpr uint32_t kColS = 0, kColDP = 32, kColP = 64, kColDS = 96, kColDQ = 128, kColDV = 256,
                   kColDK = 384;

template <int D>
struct BsqCfg {
  static constexpr int kAtomsD = D / 64;
  static constexpr int kQBytes = kShortQ * D * 2;        // Q or dO: [atom][32 rows][128 B]
  static constexpr int kKvTile = kKvRows * D * 2;        // K or V tile
  static constexpr int kDsPart = kShortQ * kKvRows * 2;  // dS: [2 atoms of 64 keys][32 rows][128 B]
  static constexpr int kQ = 0;
  static constexpr int kO = kQBytes;
  static constexpr int kKV = 2 * kQBytes;                // + s * 2 * kKvTile (K, then V)
  static constexpr int kDs = kKV + kStages * 2 * kKvTile;  // hi, lo
  static constexpr int kStats = kDs + 2 * kDsPart;       // lse * log2e [32], D [32]
  static constexpr int kBar = kStats + 2 * kShortQ * 4;
  static constexpr int kQFull = 0, kQEmpty = 1;
  static constexpr int kKvFull = 2;                      // + s
  static constexpr int kKvEmpty = kKvFull + kStages;     // + s
  static constexpr int kSFull = kKvEmpty + kStages;
  static constexpr int kPFull = kSFull + 1;
  static constexpr int kDsEmpty = kPFull + 1;
  static constexpr int kDkvFull = kDsEmpty + 1;
  static constexpr int kDkvEmpty = kDkvFull + 1;
  static constexpr int kDqFull = kDkvEmpty + 1;
  static constexpr int kDqEmpty = kDqFull + 1;
  static constexpr int kItemFull = kDqEmpty + 1;         // + slot
  static constexpr int kItemEmpty = kItemFull + 2;
  static constexpr int kDrain = kItemEmpty + 2;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kItemSlots = kBar + 8 * kNumBars;
  static constexpr int kTmemSlot = kItemSlots + 16;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kUsed = kAbort + 4;
  static constexpr int kSmemBytes = kUsed + 1024;
};

template <int D, int ACT>
__global__ void __launch_bounds__(kThreads, 1)
bwd_sq_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
              const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
              const BwdParams p, __nv_bfloat16* dq_out) {
  using C = BsqCfg<D>;
  constexpr bool kSoftmax = (ACT == GDPA_ACT_SOFTMAX);
  constexpr bool kSplit = !kSoftmax;  // GDPA: dS for dQ as bf16 hi + lo
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  auto bar = [&](int i) -> uint32_t { return sbase + C::kBar + 8u * i; };
  int2* item_slot = reinterpret_cast<int2*>(gbase + C::kItemSlots);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kAbort);
  float* stats = reinterpret_cast<float*>(gbase + C::kStats);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(C::kQFull), 1);
    mbar_init(bar(C::kQEmpty), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(C::kKvFull + s), 1);
      mbar_init(bar(C::kKvEmpty + s), 1);
    }
    mbar_init(bar(C::kSFull), 1);
    mbar_init(bar(C::kPFull), 4);
    mbar_init(bar(C::kDsEmpty), 1);
    mbar_init(bar(C::kDkvFull), 1);
    mbar_init(bar(C::kDkvEmpty), 4);
    mbar_init(bar(C::kDqFull), 1);
    mbar_init(bar(C::kDqEmpty), 4);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::kItemFull + s), 1);
      mbar_init(bar(C::kItemEmpty + s), 1 + 8);
    }
    mbar_init(bar(C::kDrain), 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&tmap_q);
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
    prefetch_tmap(&tmap_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto fail = [&]() {
    *abort_flag = 1;
    set_status(p.status, GDPA_ERR_TIMEOUT);
  };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer (whole warp)
    const int n_items = *p.n_items;
    uint32_t it = 0, g = 0, qi = 0, inflight = 0, last_g[kStages] = {};
    bool q_inflight = false, ok = true;
    while (ok) {
      int2 item = make_int2(-1, 0);
      if (lane == 0) {
        const int t = atomicAdd(p.ticket, 1);
        if (t < n_items) item = p.items[t];
      }
      item.x = __shfl_sync(0xffffffffu, item.x, 0);
      item.y = __shfl_sync(0xffffffffu, item.y, 0);
      const uint32_t slot = it & 1u;
      bool w = mbar_wait(bar(C::kItemEmpty + slot), ((it >> 1) & 1u) ^ 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      if (lane == 0) {
        item_slot[slot] = item;
        mbar_arrive(bar(C::kItemFull + slot));
      }
      ++it;
      if (item.x < 0) break;
      const int b = item.x, head = item.y;
      const int q0 = p.qo[b], Lq = p.qo[b + 1] - q0;
      const int k0 = p.ko[b], Lkv = p.ko[b + 1] - k0;
      const int nkv = (Lkv + kKvRows - 1) / kKvRows;
      // Q, dO and the row statistics of the item (the stats buffer is rewritten
      // only after the previous item's last tile has been processed)
      w = mbar_wait(bar(C::kQEmpty), (qi & 1u) ^ 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      if (kSoftmax) {
        const long long gi = static_cast<long long>(head) * p.Tq + q0 + lane;
        stats[lane] = lane < Lq ? __ldg(p.lse + gi) * kLog2e : 0.0f;
        stats[kShortQ + lane] = lane < Lq ? __ldg(p.delta + gi) : 0.0f;
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(C::kQFull), 2 * C::kQBytes);
        for (int a = 0; a < C::kAtomsD; ++a) {
          tma_load_3d(sbase + C::kQ + a * (kShortQ * 128), &tmap_q, bar(C::kQFull), 64 * a, head, q0);
          tma_load_3d(sbase + C::kO + a * (kShortQ * 128), &tmap_do, bar(C::kQFull), 64 * a, head, q0);
        }
        q_inflight = true;
      }
      ++qi;
      for (int j = 0; j < nkv; ++j, ++g) {
        const uint32_t s = g % kStages;
        w = mbar_wait(bar(C::kKvEmpty + s), ((g / kStages) & 1u) ^ 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { ok = false; if (lane == 0) fail(); break; }
        if (lane == 0) {
          const uint32_t kdst = sbase + C::kKV + s * 2 * C::kKvTile;
          mbar_arrive_expect_tx(bar(C::kKvFull + s), 2 * C::kKvTile);
          for (int a = 0; a < C::kAtomsD; ++a) {
            tma_load_3d(kdst + a * (kKvRows * 128), &tmap_k, bar(C::kKvFull + s), 64 * a, head,
                        k0 + j * kKvRows);
            tma_load_3d(kdst + C::kKvTile + a * (kKvRows * 128), &tmap_v, bar(C::kKvFull + s),
                        64 * a, head, k0 + j * kKvRows);
          }
          inflight |= 1u << s;
          last_g[s] = g;
        }
      }
    }
    if (lane == 0 && *abort_flag) {  // let every copy this warp started land
      for (int s = 0; s < kStages; ++s)
        if (inflight & (1u << s))
          mbar_wait(bar(C::kKvFull + s), (last_g[s] / kStages) & 1u, nullptr, 50000000ull);
      if (q_inflight) mbar_wait(bar(C::kQFull), (qi - 1) & 1u, nullptr, 50000000ull);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16(128, kShortQ, true, false, false);   // S^T, dP^T
      constexpr uint32_t idesc_kv = idesc_f16(128, D, true, false, true);         // dV, dK
      constexpr uint32_t idesc_dq = idesc_f16(128, kShortQ, true, true, false);   // dQ^T
      const uint64_t dsc_q = sdesc(sbase + C::kQ, 0, 1024, kSwizzle128B);  // B of S^T (K-major)
      const uint64_t dsc_o = sdesc(sbase + C::kO, 0, 1024, kSwizzle128B);  // B of dP^T (K-major)
      // Q, dO as the MN-major B of dK, dV: 64-channel atoms 32 rows apart
      const uint64_t dsc_qmn = sdesc(sbase + C::kQ, kShortQ * 128, 1024, kSwizzle128B);
      const uint64_t dsc_omn = sdesc(sbase + C::kO, kShortQ * 128, 1024, kSwizzle128B);
      const uint64_t dsc_k = sdesc(sbase + C::kKV, 0, 1024, kSwizzle128B);            // A of S^T
      const uint64_t dsc_v = sdesc(sbase + C::kKV + C::kKvTile, 0, 1024, kSwizzle128B);  // A of dP^T
      // K as the MN-major A of dQ^T; d = 64: the second 64-row half repeats the
      // first (LBO 0) and its output lanes 64..127 are never read.
      const uint64_t dsc_kt = sdesc(sbase + C::kKV, D == 128 ? kKvRows * 128 : 0, 1024, kSwizzle128B);
      const uint64_t dsc_ds = sdesc(sbase + C::kDs, 0, 1024, kSwizzle128B);  // B of dQ^T (K-major)
      uint32_t it = 0, g = 0, qi = 0, pc = 0, kvc = 0, dqc = 0;
      bool issued_any = false, ok = true;
      while (ok) {
        const uint32_t slot = it & 1u;
        if (!mbar_wait(bar(C::kItemFull + slot), (it >> 1) & 1u, abort_flag)) { fail(); break; }
        const int2 item = item_slot[slot];
        mbar_arrive(bar(C::kItemEmpty + slot));
        ++it;
        if (item.x < 0) break;
        const int b = item.x;
        const int Lkv = p.ko[b + 1] - p.ko[b];
        const int nkv = (Lkv + kKvRows - 1) / kKvRows;
        if (!mbar_wait(bar(C::kQFull), qi & 1u, abort_flag)) { fail(); break; }
        ++qi;
        tc_fence_after();
        for (int j = 0; j < nkv; ++j) {
          const uint32_t gj = g + j;
          const uint32_t s = gj % kStages;
          if (!mbar_wait(bar(C::kKvFull + s), (gj / kStages) & 1u, abort_flag)) { ok = false; fail(); break; }
          tc_fence_after();
          const uint32_t koff = s * 2 * C::kKvTile;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t a_off = koff + (ks / 4) * (kKvRows * 128) + (ks % 4) * 32;
            const uint32_t b_off = (ks / 4) * (kShortQ * 128) + (ks % 4) * 32;
            mma_f16_ss(tmem + kColS, dadd(dsc_k, a_off), dadd(dsc_q, b_off), idesc_s, ks > 0 ? 1u : 0u);
            mma_f16_ss(tmem + kColDP, dadd(dsc_v, a_off), dadd(dsc_o, b_off), idesc_s, ks > 0 ? 1u : 0u);
          }
          mma_commit(bar(C::kSFull));
          issued_any = true;
          if (!mbar_wait(bar(C::kPFull), pc & 1u, abort_flag)) { ok = false; fail(); break; }
          ++pc;
          // the previous tile's dK / dV have been read out of TMEM
          if (!mbar_wait(bar(C::kDkvEmpty), (kvc & 1u) ^ 1u, abort_flag)) { ok = false; fail(); break; }
          ++kvc;
          tc_fence_after();
          // dV = P^T dO, dK = dS^T Q: A from TMEM (queries 16 ks .. +15 in 8 columns;
          // the lo parts 16 columns further)
#pragma unroll
          for (int part = 0; part < (kSplit ? 2 : 1); ++part)
#pragma unroll
            for (int ks = 0; ks < kShortQ / 16; ++ks) {
              mma_f16_ts(tmem + kColDV, tmem + kColP + 16 * part + 8 * ks, dadd(dsc_omn, ks * 2048),
                         idesc_kv, (part > 0 || ks > 0) ? 1u : 0u);
              mma_f16_ts(tmem + kColDK, tmem + kColDS + 16 * part + 8 * ks, dadd(dsc_qmn, ks * 2048),
                         idesc_kv, (part > 0 || ks > 0) ? 1u : 0u);
            }
          mma_commit(bar(C::kDkvFull));
          if (j == 0) {
            // the previous item's dQ^T has been read out of TMEM
            if (!mbar_wait(bar(C::kDqEmpty), (dqc & 1u) ^ 1u, abort_flag)) { ok = false; fail(); break; }
            ++dqc;
            tc_fence_after();
          }
          // dQ^T += K^T dS^T (hi, then lo for GDPA activations)
#pragma unroll
          for (int part = 0; part < (kSplit ? 2 : 1); ++part)
#pragma unroll
            for (int ks = 0; ks < kKvRows / 16; ++ks)
              mma_f16_ss(tmem + kColDQ, dadd(dsc_kt, koff + ks * 2048),
                         dadd(dsc_ds, part * C::kDsPart + (ks / 4) * (kShortQ * 128) + (ks % 4) * 32),
                         idesc_dq, (j == 0 && part == 0 && ks == 0) ? 0u : 1u);
          mma_commit(bar(C::kDsEmpty));
          mma_commit(bar(C::kKvEmpty + s));
        }
        if (!ok) break;
        g += nkv;
        if (nkv > 0) mma_commit(bar(C::kDqFull));
        mma_commit(bar(C::kQEmpty));
      }
      if (issued_any) {
        mma_commit(bar(C::kDrain));
        mbar_wait(bar(C::kDrain), 0, nullptr, 100000000ull);
      }
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ activation (lanes = keys)
    const int r = warp * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const float c_s = kSoftmax ? p.scale * kLog2e : p.scale;
    // dS element (query q, key r) of the B operand: atom r / 64, row q, 16-byte
    // chunk ((r % 64) / 8) ^ (q % 8), 2 bytes at (r % 8)
    uint8_t* dsbase = gbase + C::kDs + (r >> 6) * (kShortQ * 128) + (r & 7) * 2;
    const int chunk = (r & 63) >> 3;
    uint32_t it = 0, sc = 0, qi = 0;
    bool abort_now = false;
    while (!abort_now) {
      const uint32_t slot = it & 1u;
      bool w = mbar_wait(bar(C::kItemFull + slot), (it >> 1) & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      const int2 item = item_slot[slot];
      warp_arrive(bar(C::kItemEmpty + slot), lane);
      ++it;
      if (item.x < 0) break;
      const int b = item.x;
      const int Lq = p.qo[b + 1] - p.qo[b];
      const int Lkv = p.ko[b + 1] - p.ko[b];
      const int nkv = (Lkv + kKvRows - 1) / kKvRows;
      // the producer's row statistics of this item (written before it arrived here)
      w = mbar_wait(bar(C::kQFull), qi & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      ++qi;
      for (int j = 0; j < nkv; ++j, ++sc) {
        w = mbar_wait(bar(C::kSFull), sc & 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); abort_now = true; break; }
        tc_fence_after();
        uint32_t sr[32], dr[32];
        tmem_ld32(tmem + lane_off + kColS, sr);
        tmem_ld32(tmem + lane_off + kColDP, dr);
        const bool key_ok = j * kKvRows + r < Lkv;
        float pv[kShortQ], dsv[kShortQ];
#pragma unroll
        for (int q = 0; q < kShortQ; ++q) {
          const bool valid = key_ok && q < Lq;  // queries past the sample: no term
          const float x = __uint_as_float(sr[q]) * c_s;
          const float dpv = __uint_as_float(dr[q]);
          if (kSoftmax) {
            const float pq = valid ? ex2_approx(x - stats[q]) : 0.0f;  // stats: lse * log2e
            pv[q] = pq;
            dsv[q] = pq * (dpv - stats[kShortQ + q]);                   // D
          } else {
            float a, gr;
            act_and_grad<ACT>(x, a, gr);
            pv[q] = valid ? a : 0.0f;
            dsv[q] = valid ? gr * dpv : 0.0f;
          }
        }
        uint32_t pp[16], dd[16], pl[16], dl[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          pp[i] = pack_bf16x2(pv[2 * i], pv[2 * i + 1]);
          dd[i] = pack_bf16x2(dsv[2 * i], dsv[2 * i + 1]);
          if (kSplit) {  // the rounding remainders
            pl[i] = pack_bf16x2(pv[2 * i] - __uint_as_float(pp[i] << 16),
                                pv[2 * i + 1] - __uint_as_float(pp[i] & 0xFFFF0000u));
            dl[i] = pack_bf16x2(dsv[2 * i] - __uint_as_float(dd[i] << 16),
                                dsv[2 * i + 1] - __uint_as_float(dd[i] & 0xFFFF0000u));
          }
        }
        // the previous tile's dV / dK / dQ^T products have read their operands
        w = mbar_wait(bar(C::kDsEmpty), (sc & 1u) ^ 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); abort_now = true; break; }
        tc_fence_after();
        tmem_st16(tmem + lane_off + kColP, pp);
        tmem_st16(tmem + lane_off + kColDS, dd);
        if (kSplit) {
          tmem_st16(tmem + lane_off + kColP + 16, pl);
          tmem_st16(tmem + lane_off + kColDS + 16, dl);
        }
#pragma unroll
        for (int q = 0; q < kShortQ; ++q) {
          const int off = q * 128 + ((chunk ^ (q & 7)) << 4);
          *reinterpret_cast<uint16_t*>(dsbase + off) =
              static_cast<uint16_t>(q & 1 ? dd[q >> 1] >> 16 : dd[q >> 1] & 0xFFFFu);
          if (kSplit)
            *reinterpret_cast<uint16_t*>(dsbase + C::kDsPart + off) =
                static_cast<uint16_t>(q & 1 ? dl[q >> 1] >> 16 : dl[q >> 1] & 0xFFFFu);
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        warp_arrive(bar(C::kPFull), lane);
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ epilogue
    const int r = (warp & 3) * 32 + lane;  // TMEM lane: key (dK, dV) or channel (dQ^T)
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const bool out32 = aligned32(p.dk, p.dv);
    // every sample is short: dq in bf16 (the accumulator is neither zeroed nor
    // converted); otherwise the item's finished rows go to the accumulator,
    // whose conversion follows
    const bool direct = *p.all_short != 0;
    uint32_t it = 0, kvc = 0, dqc = 0;
    while (true) {
      const uint32_t slot = it & 1u;
      bool w = mbar_wait(bar(C::kItemFull + slot), (it >> 1) & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      const int2 item = item_slot[slot];
      warp_arrive(bar(C::kItemEmpty + slot), lane);
      ++it;
      if (item.x < 0) break;
      const int b = item.x, head = item.y;
      const int q0 = p.qo[b], Lq = p.qo[b + 1] - q0;
      const int k0 = p.ko[b], Lkv = p.ko[b + 1] - k0;
      const int nkv = (Lkv + kKvRows - 1) / kKvRows;
      bool abort_now = false;
      for (int j = 0; j < nkv; ++j) {
        w = mbar_wait(bar(C::kDkvFull), kvc & 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); abort_now = true; break; }
        ++kvc;
        tc_fence_after();
        const int key = j * kKvRows + r;
        const long long grow = (static_cast<long long>(k0 + key) * p.H + head) * D;
#pragma unroll 1
        for (int which = 0; which < 2; ++which) {
          const float mul = which ? p.scale : 1.0f;
          __nv_bfloat16* dst = (which ? p.dk : p.dv) + grow;
          const uint32_t col = which ? kColDK : kColDV;
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 64) {
            uint32_t o[64];
            tmem_ld64(tmem + lane_off + col + c0, o);
            uint32_t pk[32];
#pragma unroll
            for (int i = 0; i < 32; ++i)
              pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * mul, __uint_as_float(o[2 * i + 1]) * mul);
            if (key < Lkv) store_words(dst + c0, pk, out32);
          }
        }
        tc_fence_before();
        warp_arrive(bar(C::kDkvEmpty), lane);
      }
      if (abort_now) break;
      // dQ of the item's queries: TMEM lane = channel r, column = query
      if (nkv > 0) {
        w = mbar_wait(bar(C::kDqFull), dqc & 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
        ++dqc;
        tc_fence_after();
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + kColDQ, o);
        tc_fence_before();
        warp_arrive(bar(C::kDqEmpty), lane);
        if (r < D)
          for (int q = 0; q < Lq; ++q) {
            const long long at = (static_cast<long long>(q0 + q) * p.H + head) * D + r;
            if (direct) dq_out[at] = __float2bfloat16_rn(__uint_as_float(o[q]) * p.scale);
            else p.dq_acc[at] = __uint_as_float(o[q]);
          }
      } else if (r < D) {
        for (int q = 0; q < Lq; ++q) {  // no key: dQ is zero
          const long long at = (static_cast<long long>(q0 + q) * p.H + head) * D + r;
          if (direct) dq_out[at] = __float2bfloat16_rn(0.0f);
          else p.dq_acc[at] = 0.0f;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int ACT>
cudaError_t launch_bsq_one(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const CUtensorMap& tdo, __nv_bfloat16* dq,
                           int grid, cudaStream_t stream) {
  using C = BsqCfg<D>;
  static_assert(C::kSmemBytes <= 232448, "shared memory budget");
  cudaError_t e = cudaFuncSetAttribute(bwd_sq_kernel<D, ACT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  bwd_sq_kernel<D, ACT><<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, tdo, p, dq);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_bsq_d(const BwdParams& p, int act, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, const CUtensorMap& tdo, __nv_bfloat16* dq,
                         int grid, cudaStream_t stream) {
  switch (act) {
    case GDPA_ACT_SOFTMAX:
      return launch_bsq_one<D, GDPA_ACT_SOFTMAX>(p, tq, tk, tv, tdo, dq, grid, stream);
    case GDPA_ACT_SILU:
      return launch_bsq_one<D, GDPA_ACT_SILU>(p, tq, tk, tv, tdo, dq, grid, stream);
    case GDPA_ACT_GELU_TANH:
      return launch_bsq_one<D, GDPA_ACT_GELU_TANH>(p, tq, tk, tv, tdo, dq, grid, stream);
    case GDPA_ACT_GELU_ERF:
      return launch_bsq_one<D, GDPA_ACT_GELU_ERF>(p, tq, tk, tv, tdo, dq, grid, stream);
    default:
      return launch_bsq_one<D, GDPA_ACT_IDENTITY>(p, tq, tk, tv, tdo, dq, grid, stream);
  }
}

}  // namespace

cudaError_t launch_bwd_short_q(const BwdParams& p, int act, const CUtensorMap& tq,
                               const CUtensorMap& tk, const CUtensorMap& tv,
                               const CUtensorMap& tdo, void* dq, int grid, cudaStream_t stream) {
  __nv_bfloat16* d = static_cast<__nv_bfloat16*>(dq);
  return p.d == 64 ? launch_bsq_d<64>(p, act, tq, tk, tv, tdo, d, grid, stream)
                   : launch_bsq_d<128>(p, act, tq, tk, tv, tdo, d, grid, stream);
}

}  // namespace gdpa
