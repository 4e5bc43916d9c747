// Short-key forward (GDPA activations), sm_103a.
//
// "GEM Training ..." GDPA paragraph: production traffic has short and
// asymmetric key/value sequences (long query sequences attending over a few
// hundred keys), and large batches of them broke the occupancy assumptions of
// kernels tiled for long self-attention; the kernels were reworked for those
// shapes.  Here a sample with at most kShortKv keys keeps its K and V in
// shared memory while its queries stream past in 128-row tiles:
//   S = Q K^T           (M = 128 queries, N = keys, K = d) -> TMEM
//   P = act(scale S)    activation warps; keys past the sample give 0
//   O = P V             (P read from TMEM, N = d, K = keys) -> TMEM
// P is split into bf16 hi + lo parts (two products each), as in the other
// GDPA kernels.
//
// The unit of the pipeline is a 128-column block of scores: a whole tile when
// the sample has at most 128 keys, else one of the tile's two key halves
// ([0, 128) and the rest).  Unit u goes to S buffer u % 3 and to activation
// warpgroup u % 2; the scores of unit u + 2 are computed while units u and
// u + 1 are activated, and unit u's share of the value product follows its
// activation, so neither warpgroup waits for the other's products.  O (one
// TMEM buffer; two when d = 64) is read out by the epilogue warps, which
// store the tile while the next one is computed.
//
// Work item: (sample, head, chunk of up to kShortKvChunk queries) from the
// scheduler's short-key list.  K and V are loaded once per item (K before the
// first Q tile, V after it); the Q tiles go through a ring of stages.
//
// Warps: 0-7 activation (warp w: TMEM lane quarter w % 4, warpgroup w / 4),
// 8-11 epilogue (O -> bf16 rows in global memory), 12 producer (tickets, TMA),
// 13 MMA issuer.  TMEM: S buffers [0, 128), [128, 256), [256, 384); O from
// column 384.  Every wait is bounded.
#include <type_traits>

#include "common.cuh"

namespace gdpa {
namespace {

using namespace ptx;

constexpr int kThreads = 448;
constexpr int kActWarps = 8;
constexpr int kEpiWarps = 4;
constexpr int kProducerWarp = kActWarps + kEpiWarps;
constexpr int kMmaWarp = kProducerWarp + 1;
constexpr uint32_t kColS = 0, kColO = 384;
constexpr int kSBufs = 3;
static_assert(kShortKv == 2 * kKvRows, "K / V of a short-key sample: at most two 128-row tiles");

template <int D>
struct KvCfg {
  static constexpr int kAtoms = D / 64;                     // 64-channel atoms
  static constexpr int kQStages = D == 128 ? 3 : 4;
  static constexpr int kQTile = kHalfRows * D * 2;          // [atom][128 rows][128 B]
  static constexpr int kKvBytes = kShortKv * D * 2;         // [atom][256 rows][128 B]
  static constexpr int kK = 0;
  static constexpr int kV = kKvBytes;
  static constexpr int kQ = 2 * kKvBytes;                   // + s * kQTile
  static constexpr int kBar = kQ + kQStages * kQTile;
  static constexpr int kKFull = 0, kKEmpty = 1, kVFull = 2, kVEmpty = 3;
  static constexpr int kQFull = 4;                          // + stage
  static constexpr int kQEmpty = kQFull + kQStages;         // + stage
  static constexpr int kOBufs = D == 64 ? 2 : 1;           // O buffers in TMEM columns [384, 512)
  static constexpr int kSFull = kQEmpty + kQStages;         // + S buffer
  static constexpr int kPFull = kSFull + kSBufs;            // + S buffer
  static constexpr int kOFull = kPFull + kSBufs;            // + O buffer
  static constexpr int kOEmpty = kOFull + 2;                // + O buffer
  static constexpr int kItemFull = kOEmpty + 2;             // + slot
  static constexpr int kItemEmpty = kItemFull + 2;          // + slot
  static constexpr int kDrain = kItemEmpty + 2;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kItemSlots = kBar + 8 * kNumBars;
  static constexpr int kTmemSlot = kItemSlots + 16;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kUsed = kAbort + 4;
  static constexpr int kSmemBytes = kUsed + 1024;           // + alignment slack
};

struct KvItem {
  int b, head;
  int q0, rows;   // first query row (global) and queries of the item
  int k0, Lkv;    // first key row (global) and keys of the sample
  int nt;         // 128-query tiles
  int ns;         // score columns: Lkv rounded up to 16 (the MMA's N)
  int nc;         // 32-key column chunks of the activation
  bool dbl;       // Lkv <= 128: one unit per tile (else two: the key halves)
  int nu;         // units of the item
  bool valid;     // 1 <= Lkv <= kShortKv and rows >= 1 (else the item is skipped)
};

__device__ __forceinline__ KvItem decode_kv(int2 it, const FwdParams& p) {
  KvItem r;
  r.b = it.x;
  r.head = item_head(it);
  const int chunk = item_block(it);
  const int qs = p.qo[r.b];
  const int Lq = p.qo[r.b + 1] - qs;
  r.q0 = qs + chunk * kShortKvChunk;
  r.rows = min(kShortKvChunk, Lq - chunk * kShortKvChunk);
  r.k0 = p.ko[r.b];
  r.Lkv = p.ko[r.b + 1] - r.k0;
  r.valid = r.rows >= 1 && r.Lkv >= 1 && r.Lkv <= kShortKv;
  r.nt = r.valid ? (r.rows + kHalfRows - 1) / kHalfRows : 0;
  r.ns = (r.Lkv + 15) & ~15;
  r.nc = (r.Lkv + 31) / 32;
  r.dbl = r.Lkv <= kKvRows;
  r.nu = r.dbl ? r.nt : 2 * r.nt;
  return r;
}

template <int D, int ACT>
__global__ void __launch_bounds__(kThreads, 1)
fwd_kv_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
              const __grid_constant__ CUtensorMap tmap_v, const FwdParams p) {
  using C = KvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  auto bar = [&](int i) -> uint32_t { return sbase + C::kBar + 8u * i; };
  int2* item_slot = reinterpret_cast<int2*>(gbase + C::kItemSlots);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kAbort);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(C::kKFull), 1);
    mbar_init(bar(C::kKEmpty), 1);
    mbar_init(bar(C::kVFull), 1);
    mbar_init(bar(C::kVEmpty), 1);
    for (int s = 0; s < C::kQStages; ++s) {
      mbar_init(bar(C::kQFull + s), 1);
      mbar_init(bar(C::kQEmpty + s), 1);
    }
    for (int u = 0; u < kSBufs; ++u) {
      mbar_init(bar(C::kSFull + u), 1);
      mbar_init(bar(C::kPFull + u), kActWarps / 2);
    }
    for (int u = 0; u < 2; ++u) {
      mbar_init(bar(C::kOFull + u), 1);
      mbar_init(bar(C::kOEmpty + u), kEpiWarps);
      mbar_init(bar(C::kItemFull + u), 1);
      mbar_init(bar(C::kItemEmpty + u), 1 + kActWarps + kEpiWarps);
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
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const int n_items = *p.n_items;
      uint32_t it = 0, kvi = 0, qg = 0;
      uint32_t q_inflight = 0, q_last[C::kQStages] = {};
      bool k_inflight = false, v_inflight = false, ok = true;
      while (ok) {
        const int t = atomicAdd(p.ticket, 1);
        const int2 item = t < n_items ? p.items[t] : make_int2(-1, 0);
        const uint32_t slot = it & 1u;
        if (!mbar_wait(bar(C::kItemEmpty + slot), ((it >> 1) & 1u) ^ 1u, abort_flag)) { fail(); break; }
        item_slot[slot] = item;
        mbar_arrive(bar(C::kItemFull + slot));
        ++it;
        if (item.x < 0) break;
        const KvItem in = decode_kv(item, p);
        if (!in.valid) continue;
        const int nkt = in.Lkv > kKvRows ? 2 : 1;
        const uint32_t kv_bytes = static_cast<uint32_t>(nkt) * kKvRows * D * 2;
        // K: free once the previous item's last score product has completed
        if (!mbar_wait(bar(C::kKEmpty), (kvi & 1u) ^ 1u, abort_flag)) { fail(); break; }
        mbar_arrive_expect_tx(bar(C::kKFull), kv_bytes);
        for (int kt = 0; kt < nkt; ++kt)
          for (int a = 0; a < C::kAtoms; ++a)
            tma_load_3d(sbase + C::kK + a * (kShortKv * 128) + kt * (kKvRows * 128), &tmap_k,
                        bar(C::kKFull), 64 * a, in.head, in.k0 + kt * kKvRows);
        k_inflight = true;
        for (int tq = 0; tq < in.nt; ++tq, ++qg) {
          const uint32_t s = qg % C::kQStages;
          if (!mbar_wait(bar(C::kQEmpty + s), ((qg / C::kQStages) & 1u) ^ 1u, abort_flag)) {
            ok = false;
            fail();
            break;
          }
          mbar_arrive_expect_tx(bar(C::kQFull + s), C::kQTile);
          for (int a = 0; a < C::kAtoms; ++a)
            tma_load_3d(sbase + C::kQ + s * C::kQTile + a * (kHalfRows * 128), &tmap_q,
                        bar(C::kQFull + s), 64 * a, in.head, in.q0 + tq * kHalfRows);
          q_inflight |= 1u << s;
          q_last[s] = qg;
          if (tq == 0) {
            // V: free once the previous item's last value product has completed
            if (!mbar_wait(bar(C::kVEmpty), (kvi & 1u) ^ 1u, abort_flag)) { ok = false; fail(); break; }
            mbar_arrive_expect_tx(bar(C::kVFull), kv_bytes);
            for (int kt = 0; kt < nkt; ++kt)
              for (int a = 0; a < C::kAtoms; ++a)
                tma_load_3d(sbase + C::kV + a * (kShortKv * 128) + kt * (kKvRows * 128), &tmap_v,
                            bar(C::kVFull), 64 * a, in.head, in.k0 + kt * kKvRows);
            v_inflight = true;
          }
        }
        ++kvi;
      }
      if (*abort_flag) {  // let every copy this thread started land
        for (int s = 0; s < C::kQStages; ++s)
          if (q_inflight & (1u << s))
            mbar_wait(bar(C::kQFull + s), (q_last[s] / C::kQStages) & 1u, nullptr, 50000000ull);
        if (k_inflight) mbar_wait(bar(C::kKFull), (kvi - 1) & 1u, nullptr, 50000000ull);
        if (v_inflight) mbar_wait(bar(C::kVFull), (kvi - 1) & 1u, nullptr, 50000000ull);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // S: A = Q (K-major), B = K (K-major, up to 256 rows per atom).
      // O: A = P from TMEM, B = V (MN-major: channels contiguous, 256-row atoms).
      constexpr uint32_t idesc_o = idesc_f16(128, D, true, false, true);
      const uint64_t dsc_q = sdesc(sbase + C::kQ, 0, 1024, kSwizzle128B);
      const uint64_t dsc_k = sdesc(sbase + C::kK, 0, 1024, kSwizzle128B);
      const uint64_t dsc_v = sdesc(sbase + C::kV, kShortKv * 128, 1024, kSwizzle128B);
      uint32_t it = 0, kvi = 0, qg = 0, og = 0, gu = 0;
      bool issued_any = false, ok = true;
      while (ok) {
        const uint32_t slot = it & 1u;
        if (!mbar_wait(bar(C::kItemFull + slot), (it >> 1) & 1u, abort_flag)) { fail(); break; }
        const int2 item = item_slot[slot];
        mbar_arrive(bar(C::kItemEmpty + slot));
        ++it;
        if (item.x < 0) break;
        const KvItem in = decode_kv(item, p);
        if (!in.valid) continue;
        const int nk = (in.Lkv + 15) / 16;  // 16-key steps of the value product
        // Scores of unit v (buffer (gu + v) % 3): a tile's first unit waits
        // for its Q tile, its last one releases it; the item's last unit
        // releases K.
        auto issue_s = [&](int v) -> bool {
          const int half = in.dbl ? 0 : (v & 1);
          if (half == 0) {
            if (!mbar_wait(bar(C::kQFull + qg % C::kQStages), (qg / C::kQStages) & 1u, abort_flag))
              return false;
            tc_fence_after();
          }
          const uint32_t buf = (gu + v) % kSBufs;
          const int n = in.dbl ? in.ns : (half ? in.ns - kKvRows : kKvRows);
          const uint32_t idesc_s = idesc_f16(128, n, true, false, false);
          const uint64_t qb = dadd(dsc_q, (qg % C::kQStages) * C::kQTile);
          const uint64_t kb = dadd(dsc_k, half * (kKvRows * 128));
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            mma_f16_ss(tmem + kColS + 128 * buf,
                       dadd(qb, (ks / 4) * (kHalfRows * 128) + (ks % 4) * 32),
                       dadd(kb, (ks / 4) * (kShortKv * 128) + (ks % 4) * 32), idesc_s,
                       ks > 0 ? 1u : 0u);
          mma_commit(bar(C::kSFull + buf));
          if (in.dbl || half == 1) {
            mma_commit(bar(C::kQEmpty + qg % C::kQStages));
            ++qg;
          }
          if (v + 1 == in.nu) mma_commit(bar(C::kKEmpty));
          issued_any = true;
          return true;
        };
        if (!mbar_wait(bar(C::kKFull), kvi & 1u, abort_flag)) { fail(); break; }
        tc_fence_after();
        for (int v = 0; v < 2 && v < in.nu; ++v)
          if (!issue_s(v)) { ok = false; break; }
        for (int u = 0; u < in.nu && ok; ++u) {
          // buffer (gu + u + 2) % 3 was last read by unit u - 1's value product
          if (u + 2 < in.nu && !issue_s(u + 2)) { ok = false; break; }
          const uint32_t guu = gu + u;
          const uint32_t buf = guu % kSBufs;
          const int half = in.dbl ? 0 : (u & 1);
          const int tile = in.dbl ? u : (u >> 1);
          const uint32_t ob = og % C::kOBufs;
          if (!mbar_wait(bar(C::kPFull + buf), (guu / kSBufs) & 1u, abort_flag)) { ok = false; break; }
          if (half == 0 &&
              !mbar_wait(bar(C::kOEmpty + ob), ((og / C::kOBufs) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
          if (u == 0 && !mbar_wait(bar(C::kVFull), kvi & 1u, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t tp = tmem + kColS + 128 * buf;
          const uint32_t to = tmem + kColO + D * ob;
          const int ks0 = in.dbl ? 0 : 8 * half;
          const int ks1 = in.dbl ? nk : (half ? nk : 8);
          for (int ks = ks0; ks < ks1; ++ks) {
            const int j = ks - ks0;  // 16-key step within the unit
            const uint32_t pcol = 32 * (j / 2) + 8 * (j % 2);
            const uint64_t vb = dadd(dsc_v, ks * 2048);
            mma_f16_ts(to, tp + pcol, vb, idesc_o, ks > 0 ? 1u : 0u);
            mma_f16_ts(to, tp + pcol + 16, vb, idesc_o, 1u);
          }
          if (in.dbl || half == 1) {
            mma_commit(bar(C::kOFull + ob));
            ++og;
            if (tile + 1 == in.nt) mma_commit(bar(C::kVEmpty));
          }
        }
        if (!ok) { fail(); break; }
        gu += in.nu;
        ++kvi;
      }
      // Every MMA this thread issued must complete before TMEM is freed.
      if (issued_any) {
        mma_commit(bar(C::kDrain));
        mbar_wait(bar(C::kDrain), 0, nullptr, 100000000ull);
      }
    }
  } else if (warp < kActWarps) {
    // ------------------------------------------------------------ activation warpgroups
    // Warpgroup w activates the units u with u % 2 == w (counted over the
    // CTA's whole run): all 32-key chunks of the unit's S buffer.
    const int wq = warp & 3;
    const int wg = warp >> 2;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    uint32_t it = 0, gu = 0;
    bool abort_now = false;
    while (!abort_now) {
      const uint32_t slot = it & 1u;
      bool w = mbar_wait(bar(C::kItemFull + slot), (it >> 1) & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      const int2 item = item_slot[slot];
      warp_arrive(bar(C::kItemEmpty + slot), lane);
      ++it;
      if (item.x < 0) break;
      const KvItem in = decode_kv(item, p);
      if (!in.valid) continue;
      for (int u = (gu & 1u) == static_cast<uint32_t>(wg) ? 0 : 1; u < in.nu; u += 2) {
        const uint32_t guu = gu + u;
        const uint32_t buf = guu % kSBufs;
        const int half = in.dbl ? 0 : (u & 1);
        const int kbase = half * kKvRows;   // first key of the unit
        const int nch = in.dbl ? in.nc : (half ? in.nc - 4 : 4);
        w = mbar_wait(bar(C::kSFull + buf), (guu / kSBufs) & 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); abort_now = true; break; }
        tc_fence_after();
        const uint32_t t_s = tmem + lane_off + kColS + 128 * buf;
#pragma unroll 1
        for (int c = 0; c < nch; ++c) {
          uint32_t sr[32];
          tmem_ld32(t_s + 32 * c, sr);
          const int kin = in.Lkv - kbase - 32 * c;  // keys of this chunk inside the sample (>= 1)
          uint32_t hi[16], lo[16];
          // the last chunk of a sample masks the keys past it (stale columns
          // there are replaced, not multiplied)
          auto body = [&](auto masked) {
            constexpr bool kMask = decltype(masked)::value;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float a0, a1, g_;
              act_and_grad<ACT>(__uint_as_float(sr[2 * i]) * p.scale, a0, g_);
              act_and_grad<ACT>(__uint_as_float(sr[2 * i + 1]) * p.scale, a1, g_);
              if (kMask && 2 * i >= kin) a0 = 0.0f;
              if (kMask && 2 * i + 1 >= kin) a1 = 0.0f;
              const uint32_t h = pack_bf16x2(a0, a1);
              hi[i] = h;
              lo[i] = pack_bf16x2(a0 - __uint_as_float(h << 16), a1 - __uint_as_float(h & 0xFFFF0000u));
            }
          };
          if (kin >= 32) body(std::false_type{}); else body(std::true_type{});
          tmem_st16(t_s + 32 * c, hi);
          tmem_st16(t_s + 32 * c + 16, lo);
        }
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(bar(C::kPFull + buf), lane);
      }
      gu += in.nu;
    }
  } else if (warp < kActWarps + kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // TMEM lane: query row of the tile
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const bool out32 = aligned32(p.out);
    uint32_t it = 0, og = 0;
    bool abort_now = false;
    while (!abort_now) {
      const uint32_t slot = it & 1u;
      bool w = mbar_wait(bar(C::kItemFull + slot), (it >> 1) & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      const int2 item = item_slot[slot];
      warp_arrive(bar(C::kItemEmpty + slot), lane);
      ++it;
      if (item.x < 0) break;
      const KvItem in = decode_kv(item, p);
      for (int t = 0; t < in.nt; ++t, ++og) {
        const uint32_t ob = og % C::kOBufs;
        w = mbar_wait(bar(C::kOFull + ob), (og / C::kOBufs) & 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); abort_now = true; break; }
        tc_fence_after();
        uint32_t pk[D / 64][32];
#pragma unroll
        for (int chunk = 0; chunk < D / 64; ++chunk) {
          uint32_t o[64];
          tmem_ld64(tmem + lane_off + kColO + D * ob + 64 * chunk, o);
#pragma unroll
          for (int i = 0; i < 32; ++i)
            pk[chunk][i] = pack_bf16x2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1]));
        }
        tc_fence_before();
        warp_arrive(bar(C::kOEmpty + ob), lane);
        const int row = t * kHalfRows + r;
        if (row < in.rows) {
          __nv_bfloat16* orow = p.out + (static_cast<long long>(in.q0 + row) * p.H + in.head) * D;
#pragma unroll
          for (int chunk = 0; chunk < D / 64; ++chunk) store_words(orow + 64 * chunk, pk[chunk], out32);
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
cudaError_t launch_kv_one(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, int grid, cudaStream_t stream) {
  using C = KvCfg<D>;
  static_assert(C::kSmemBytes <= 232448, "shared memory budget");
  cudaError_t e = cudaFuncSetAttribute(fwd_kv_kernel<D, ACT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  fwd_kv_kernel<D, ACT><<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_kv_d(const FwdParams& p, int act, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, int grid, cudaStream_t stream) {
  switch (act) {
    case GDPA_ACT_SILU: return launch_kv_one<D, GDPA_ACT_SILU>(p, tq, tk, tv, grid, stream);
    case GDPA_ACT_GELU_TANH: return launch_kv_one<D, GDPA_ACT_GELU_TANH>(p, tq, tk, tv, grid, stream);
    case GDPA_ACT_GELU_ERF: return launch_kv_one<D, GDPA_ACT_GELU_ERF>(p, tq, tk, tv, grid, stream);
    case GDPA_ACT_IDENTITY: return launch_kv_one<D, GDPA_ACT_IDENTITY>(p, tq, tk, tv, grid, stream);
    default: return cudaErrorInvalidValue;  // softmax takes the general kernel
  }
}

}  // namespace

cudaError_t launch_fwd_short_kv(const FwdParams& p, int act, const CUtensorMap& tq,
                                const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                                cudaStream_t stream) {
  return p.d == 64 ? launch_kv_d<64>(p, act, tq, tk, tv, grid, stream)
                   : launch_kv_d<128>(p, act, tq, tk, tv, grid, stream);
}

}  // namespace gdpa
