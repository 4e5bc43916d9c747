// Backward kernels of jagged attention with a pluggable activation, sm_103a.
//
// "GEM Training ..." JFA paragraph ("efficient backward passes") and GDPA
// paragraph (1.6x backward speedup).  The gradients follow from the chain
// rule on s = scale q.k + bias, p = act(s) (or softmax), o = sum p v:
//   dV = P^T dO,  dP = dO V^T,  dS = P*(dP - D) (softmax, D = rowsum(dO*O))
//   or act'(S)*dP (GDPA),  dQ = scale dS K,  dK = scale dS^T Q.
//
// Main kernel: key/value-major.  A work item is one 128-row key/value block
// of one (sample, head); the CTA keeps K and V of the block in shared memory
// and streams the sample's queries past it in 64-row tiles.  Everything is
// computed transposed so that TMEM lanes are key rows:
//   S^T = K Q^T, dP^T = V dO^T           (M = 128 keys, N = 64 queries)
//   dV += P^T dO, dK += dS^T Q           (accumulated in TMEM over the tiles)
//   dQ^T = K^T dS^T                      (M = d, N = 64) -> TMA reduce-add into fp32 dQ
// P^T goes back into the S^T columns of TMEM (A operand of dV); dS^T is
// written to a swizzled shared-memory tile that is both the K-major A
// operand of dK and the MN-major B operand of dQ^T.
//
// Warp roles (448 threads, one CTA per SM, persistent over the cost-sorted
// work list):
//   warps 0-3  activation group A: P^T, dS^T for query columns [0,32) of a tile
//   warps 4-7  activation group B: the same for query columns [32,64)
//   warps 8-11 dQ group: dQ^T tile -> shared memory -> bulk tensor reduce-add
//              (each warp its own 32 channels, no group barrier)
//              into the fp32 dQ accumulator; dK/dV epilogue
//   warp  12   producer: TMA loads of K/V, Q/dO tiles; lse, D and bias values
//   warp  13   MMA issuer
// TMEM columns: S^T/P^T buffers [0,64) [64,128), dP^T [128,192),
// dQ^T [192,256), dV [256,256+d), dK [384,384+d).
//
// Small kernels: preprocess (zero the dQ accumulator, D = rowsum(dO*O)) and
// the dQ conversion (fp32 accumulator * scale -> bf16).
#include "common.cuh"

namespace gdpa {
namespace {

using namespace ptx;

constexpr int kThreads = 448;
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int kActThreads = 256;  // both activation groups
constexpr float kLog2e = 1.4426950408889634f;

template <int D, bool SPLIT>
struct BwdCfg {
  static constexpr int kKvTileBytes = kBwdKvRows * D * 2;     // K or V block
  static constexpr int kQTileBytes = kBwdQRows * D * 2;       // Q or dO tile
  static constexpr int kDsBytes = kBwdKvRows * kBwdQRows * 2;  // one dS^T tile (16 KB)
  static constexpr int kDsParts = SPLIT ? 2 : 1;
  // Q/dO stages: three where shared memory allows (hides the TMA round trip
  // behind two tiles of work), two for the split-P/dS variants.
  static constexpr int kStages = SPLIT ? 2 : 3;
  static constexpr int kK = 0;
  static constexpr int kV = kKvTileBytes;
  static constexpr int kQ = 2 * kKvTileBytes;                  // + s * 2 * qtile ; dO = Q + qtile
  static constexpr int kDs = kQ + kStages * 2 * kQTileBytes;   // + buf * parts * ds + part * ds
  // per stage: float lse2[64], D[64], bias window[192]
  static constexpr int kStatFloats = 2 * kBwdQRows + kBwdQRows + kBwdKvRows;
  static constexpr int kStats = kDs + 2 * kDsParts * kDsBytes;
  // dQ staging: per warp, three [16 queries][32 channels] fp32 buffers (each
  // warp reduces its own channels)
  static constexpr int kDqChunk = 16;
  static constexpr int kDqWarpBufs = 3;
  static constexpr int kDqStageBytes = 4 * kDqWarpBufs * kDqChunk * 32 * 4;
  static constexpr int kDqStage = kStats + kStages * kStatFloats * 4;
  // bias-table gradient: per tile, dS summed along its 191 diagonals (two
  // buffers of 192 floats, then {first diagonal, head})
  static constexpr int kDbBuf = 192 * 4 + 16;
  static constexpr int kDb = kDqStage + kDqStageBytes;
  static constexpr int kBar = kDb + 2 * kDbBuf;
  static constexpr int kKvFull = 0, kKvEmpty = 1;
  static constexpr int kQdFull = 2;                 // + s
  static constexpr int kQdEmpty = kQdFull + kStages;
  static constexpr int kSFull = kQdEmpty + kStages; // + buffer
  static constexpr int kPFull = kSFull + 2;
  static constexpr int kDqFull = kPFull + 1;
  static constexpr int kDqEmpty = kDqFull + 1;
  static constexpr int kDkvFull = kDqEmpty + 1;
  static constexpr int kDkvEmpty = kDkvFull + 1;
  static constexpr int kItemFull = kDkvEmpty + 1;   // + slot
  static constexpr int kItemEmpty = kItemFull + 2;
  static constexpr int kDrain = kItemEmpty + 2;
  static constexpr int kDbAcc = kDrain + 1;     // + buffer: the activation threads added a tile
  static constexpr int kDbFree = kDbAcc + 2;    // + buffer: flushed to the table and zeroed
  static constexpr int kNumBars = kDbFree + 2;
  static constexpr int kItemSlots = kBar + 8 * kNumBars;
  static constexpr int kTmemSlot = kItemSlots + 16;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kGroupOk = kAbort + 4;   // int[4]: dQ-group vote on a wait's result
  static constexpr int kUsed = kGroupOk + 16;
  static constexpr int kSmemBytes = kUsed + 1024;
};

// TMEM column bases
constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 192, kColDV = 256, kColDK = 384;

struct BwdItem {
  int b, head, kb;
  int q0, k0, Lq, Lkv;
  int qt0;  // first query tile (64 rows) visited
  int nq;   // number of query tiles visited
};

__device__ __forceinline__ BwdItem decode_bwd(int2 it, const BwdParams& p) {
  BwdItem r;
  r.b = it.x;
  r.head = item_head(it);
  r.kb = item_block(it);
  r.q0 = p.qo[r.b];
  r.Lq = p.qo[r.b + 1] - r.q0;
  r.k0 = p.ko[r.b];
  r.Lkv = p.ko[r.b + 1] - r.k0;
  // query tiles that see some key of the block (causal / sliding-window band)
  // (items exist only for blocks that start inside the sample, and every
  // such key is seen by some query unless the sample has no query rows)
  const int kb0 = r.kb * kBwdKvRows;
  const int qb = band_query_begin(kb0, p.causal, p.window);
  const int qe = band_query_end(min(r.Lkv, kb0 + kBwdKvRows) - 1, p.window, r.Lq);
  r.qt0 = qb / kBwdQRows;
  r.nq = (qe + kBwdQRows - 1) / kBwdQRows - r.qt0;  // 0 when qe == qb == 0 (no query rows)
  return r;
}

// With a bias-table gradient one more warp (14) adds each tile's diagonal
// sums to the table.  kDense: a dense jagged bias (p.bias_dense) instead of
// the relative-position table, read from global memory by the activation
// warps (the warp's lanes are consecutive keys: coalesced row segments); with
// p.dbias its gradient goes back the same way, one reduction per pair.
template <int D, int ACT, bool kDBias, bool kDense>
__global__ void __launch_bounds__(kThreads + (kDBias && !kDense ? 32 : 0), 1)
bwd_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
           const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
           const __grid_constant__ CUtensorMap tmap_dq, const BwdParams p) {
  constexpr bool kSoftmax = (ACT == GDPA_ACT_SOFTMAX);
  constexpr bool kSplit = !kSoftmax;
  using C = BwdCfg<D, kSplit>;
  // kDBias: the bias's gradient, of the table (diagonal sums in shared memory,
  // flushed by warp 14) or of the dense bias (reduced straight to memory)
  constexpr bool kTableGrad = kDBias && !kDense;
  constexpr bool kDenseGrad = kDBias && kDense;

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
    mbar_init(bar(C::kKvFull), 1);
    mbar_init(bar(C::kKvEmpty), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kQdFull + s), 1);
      mbar_init(bar(C::kQdEmpty + s), 1);
    }
    mbar_init(bar(C::kSFull + 0), 1);
    mbar_init(bar(C::kSFull + 1), 1);
    mbar_init(bar(C::kPFull), kActThreads);
    mbar_init(bar(C::kDqFull), 1);
    mbar_init(bar(C::kDqEmpty), 128);
    mbar_init(bar(C::kDkvFull), 1);
    mbar_init(bar(C::kDkvEmpty), 128);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::kItemFull + s), 1);
      mbar_init(bar(C::kItemEmpty + s), 1 + kActThreads + 128 + (kTableGrad ? 1 : 0));
    }
    mbar_init(bar(C::kDrain), 1);
    for (int u = 0; u < 2; ++u) {
      mbar_init(bar(C::kDbAcc + u), kActThreads);
      mbar_init(bar(C::kDbFree + u), 1);
    }
    fence_mbar_init();
  }
  if (kTableGrad)
    for (int i = threadIdx.x; i < 2 * C::kDbBuf / 4; i += blockDim.x)
      reinterpret_cast<float*>(gbase + C::kDb)[i] = 0.0f;
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&tmap_q);
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
    prefetch_tmap(&tmap_do);
    prefetch_tmap(&tmap_dq);
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
    uint32_t it = 0, g = 0, kvi = 0;
    bool kv_inflight = false;
    uint32_t inflight = 0, last_g[C::kStages] = {};
    bool ok = true;
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
      const BwdItem in = decode_bwd(item, p);
      if (in.nq == 0) continue;
      w = mbar_wait(bar(C::kKvEmpty), (kvi & 1u) ^ 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      ++kvi;
      const int krow = in.k0 + in.kb * kBwdKvRows;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(C::kKvFull), 2 * C::kKvTileBytes);
        for (int x = 0; x < D; x += 64) {
          tma_load_3d(sbase + C::kK + (x / 64) * (kBwdKvRows * 128), &tmap_k, bar(C::kKvFull), x,
                      in.head, krow);
          tma_load_3d(sbase + C::kV + (x / 64) * (kBwdKvRows * 128), &tmap_v, bar(C::kKvFull), x,
                      in.head, krow);
        }
        kv_inflight = true;
      }
      // Per-lane values of one query tile: lse*log2e and D for columns lane and
      // lane+32, and bias-window entries lane + 32k.  They are fetched one tile
      // ahead, so the global-load latency overlaps the wait for a free stage.
      const int rel_w = 2 * p.max_rel - 1;
      const float* brow =
          p.bias_table ? p.bias_table + static_cast<long long>(in.head) * rel_w : nullptr;
      constexpr int kWin = kBwdQRows + kBwdKvRows - 1;  // 191 relative positions
      auto fetch = [&](int t, float (&v)[10]) {
        const int qloc = (in.qt0 + t) * kBwdQRows;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int ql = qloc + lane + 32 * k;
          float l2 = 0.0f, dd = 0.0f;
          if (kSoftmax && ql < in.Lq) {
            const long long gi = static_cast<long long>(in.head) * p.Tq + in.q0 + ql;
            l2 = __ldg(p.lse + gi) * kLog2e;
            dd = __ldg(p.delta + gi);
          }
          v[2 * k] = l2;
          v[2 * k + 1] = dd;
        }
        // bias(i - j) for query column c and key row jj of the tile is window
        // entry c - jj + 127
        const int w0 = qloc - in.kb * kBwdKvRows - (kBwdKvRows - 1) + p.max_rel - 1;
#pragma unroll
        for (int k = 0; k < 6; ++k) {
          const int e = lane + 32 * k;
          v[4 + k] = (brow != nullptr && e < kWin) ? __ldg(brow + min(max(w0 + e, 0), rel_w - 1))
                                                   : 0.0f;
        }
      };
      float cur[10];
      fetch(0, cur);
      for (int t = 0; t < in.nq; ++t, ++g) {
        const uint32_t s = g % C::kStages;
        const uint32_t ph = (g / C::kStages) & 1u;
        w = mbar_wait(bar(C::kQdEmpty + s), ph ^ 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { ok = false; if (lane == 0) fail(); break; }
        const int qloc = (in.qt0 + t) * kBwdQRows;  // first local query row of the tile
        float* st = stats + s * C::kStatFloats;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          st[lane + 32 * k] = cur[2 * k];
          st[kBwdQRows + lane + 32 * k] = cur[2 * k + 1];
        }
        if (brow != nullptr) {
#pragma unroll
          for (int k = 0; k < 6; ++k)
            if (lane + 32 * k < kWin) st[2 * kBwdQRows + lane + 32 * k] = cur[4 + k];
        }
        float nxt[10];
        if (t + 1 < in.nq) {
          fetch(t + 1, nxt);
        } else {
#pragma unroll
          for (int k = 0; k < 10; ++k) nxt[k] = 0.0f;
        }
        __syncwarp();
        if (lane == 0) {
          const uint32_t qd = sbase + C::kQ + s * 2 * C::kQTileBytes;
          mbar_arrive_expect_tx(bar(C::kQdFull + s), 2 * C::kQTileBytes);
          for (int x = 0; x < D; x += 64) {
            tma_load_3d(qd + (x / 64) * (kBwdQRows * 128), &tmap_q, bar(C::kQdFull + s), x,
                        in.head, in.q0 + qloc);
            tma_load_3d(qd + C::kQTileBytes + (x / 64) * (kBwdQRows * 128), &tmap_do,
                        bar(C::kQdFull + s), x, in.head, in.q0 + qloc);
          }
          inflight |= 1u << s;
          last_g[s] = g;
        }
#pragma unroll
        for (int k = 0; k < 10; ++k) cur[k] = nxt[k];
      }
    }
    if (lane == 0 && *abort_flag) {
      for (int s = 0; s < C::kStages; ++s)
        if (inflight & (1u << s))
          mbar_wait(bar(C::kQdFull + s), (last_g[s] / C::kStages) & 1u, nullptr, 50000000ull);
      if (kv_inflight) mbar_wait(bar(C::kKvFull), (kvi - 1) & 1u, nullptr, 50000000ull);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16(128, kBwdQRows, true, false, false);
      constexpr uint32_t idesc_acc = idesc_f16(128, D, true, false, true);
      constexpr uint32_t idesc_dq = idesc_f16(128, kBwdQRows, true, true, true);
      uint32_t it = 0, g = 0, kvi = 0, pc = 0, dqc = 0, dkvc = 0;
      uint32_t suse[2] = {0, 0};
      bool issued_any = false;
      auto issue_sdp = [&](int t, uint32_t s) {
        const uint32_t buf = t & 1;
        const uint32_t qd = sbase + C::kQ + s * 2 * C::kQTileBytes;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t aoff = (ks / 4) * (kBwdKvRows * 128) + (ks % 4) * 32;
          const uint32_t boff = (ks / 4) * (kBwdQRows * 128) + (ks % 4) * 32;
          mma_f16_ss(tmem + kColS + buf * 64, sdesc(sbase + C::kK + aoff, 0, 1024, kSwizzle128B),
                     sdesc(qd + boff, 0, 1024, kSwizzle128B), idesc_s, ks > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t aoff = (ks / 4) * (kBwdKvRows * 128) + (ks % 4) * 32;
          const uint32_t boff = (ks / 4) * (kBwdQRows * 128) + (ks % 4) * 32;
          mma_f16_ss(tmem + kColDP, sdesc(sbase + C::kV + aoff, 0, 1024, kSwizzle128B),
                     sdesc(qd + C::kQTileBytes + boff, 0, 1024, kSwizzle128B), idesc_s,
                     ks > 0 ? 1u : 0u);
        }
        mma_commit(bar(C::kSFull + buf));
        issued_any = true;
      };
      bool ok = true;
      while (ok) {
        const uint32_t slot = it & 1u;
        if (!mbar_wait(bar(C::kItemFull + slot), (it >> 1) & 1u, abort_flag)) { fail(); break; }
        const int2 item = item_slot[slot];
        mbar_arrive(bar(C::kItemEmpty + slot));
        ++it;
        if (item.x < 0) break;
        const BwdItem in = decode_bwd(item, p);
        if (in.nq == 0) continue;
        if (!mbar_wait(bar(C::kKvFull), kvi & 1u, abort_flag)) { fail(); break; }
        ++kvi;
        {
          const uint32_t s = g % C::kStages;
          if (!mbar_wait(bar(C::kQdFull + s), (g / C::kStages) & 1u, abort_flag)) { fail(); break; }
          tc_fence_after();
          issue_sdp(0, s);
        }
        for (int t = 0; t < in.nq; ++t) {
          const uint32_t gt = g + t;
          const uint32_t s = gt % C::kStages;
          const uint32_t buf = t & 1;
          if (!mbar_wait(bar(C::kPFull), pc & 1u, abort_flag)) { ok = false; fail(); break; }
          ++pc;
          tc_fence_after();
          if (t + 1 < in.nq) {
            const uint32_t s1 = (gt + 1) % C::kStages;
            if (!mbar_wait(bar(C::kQdFull + s1), ((gt + 1) / C::kStages) & 1u, abort_flag)) { ok = false; fail(); break; }
            tc_fence_after();
            issue_sdp(t + 1, s1);
          }
          if (t == 0) {
            // previous item's dK/dV must have been read out before we overwrite them
            if (!mbar_wait(bar(C::kDkvEmpty), (dkvc & 1u) ^ 1u, abort_flag)) { ok = false; fail(); break; }
            tc_fence_after();
          }
          const uint32_t qd = sbase + C::kQ + s * 2 * C::kQTileBytes;
          const uint32_t ds = sbase + C::kDs + buf * C::kDsParts * C::kDsBytes;
          // dV += P^T dO   (A = P^T in TMEM, B = dO tile, MN-major)
#pragma unroll
          for (int ks = 0; ks < kBwdQRows / 16; ++ks) {
            const uint64_t bd = sdesc(qd + C::kQTileBytes + ks * 2048, kBwdQRows * 128, 1024,
                                      kSwizzle128B);
            const uint32_t pcol = tmem + kColS + buf * 64 + 32 * (ks / 2) + 8 * (ks % 2);
            mma_f16_ts(tmem + kColDV, pcol, bd, idesc_acc, (t == 0 && ks == 0) ? 0u : 1u);
            if (kSplit) mma_f16_ts(tmem + kColDV, pcol + 16, bd, idesc_acc, 1u);
          }
          // dK += dS^T Q   (A = dS^T smem K-major, B = Q tile MN-major)
#pragma unroll
          for (int ks = 0; ks < kBwdQRows / 16; ++ks) {
            const uint64_t bd = sdesc(qd + ks * 2048, kBwdQRows * 128, 1024, kSwizzle128B);
#pragma unroll
            for (int part = 0; part < C::kDsParts; ++part) {
              const uint64_t ad = sdesc(ds + part * C::kDsBytes + ks * 32, 0, 1024, kSwizzle128B);
              mma_f16_ss(tmem + kColDK, ad, bd, idesc_acc, (t == 0 && ks == 0 && part == 0) ? 0u : 1u);
            }
          }
          mma_commit(bar(C::kQdEmpty + s));
          // dQ^T = K^T dS^T  (A = K block MN-major, B = dS^T MN-major); wait until
          // the dQ group has drained the previous tile's dQ^T.
          if (!mbar_wait(bar(C::kDqEmpty), (dqc & 1u) ^ 1u, abort_flag)) { ok = false; fail(); break; }
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < kBwdKvRows / 16; ++ks) {
            // d = 64: the second 64-row half of A repeats the first (LBO 0); its
            // output lanes 64..127 are ignored.
            const uint64_t ad = sdesc(sbase + C::kK + ks * 2048, D == 128 ? kBwdKvRows * 128 : 0,
                                      1024, kSwizzle128B);
#pragma unroll
            for (int part = 0; part < C::kDsParts; ++part) {
              const uint64_t bd = sdesc(ds + part * C::kDsBytes + ks * 2048, 0, 1024, kSwizzle128B);
              mma_f16_ss(tmem + kColDQ, ad, bd, idesc_dq, (ks == 0 && part == 0) ? 0u : 1u);
            }
          }
          mma_commit(bar(C::kDqFull));
          ++dqc;
          suse[buf]++;
        }
        if (!ok) break;
        mma_commit(bar(C::kDkvFull));
        mma_commit(bar(C::kKvEmpty));
        ++dkvc;
        g += in.nq;
      }
      if (issued_any) {
        mma_commit(bar(C::kDrain));
        mbar_wait(bar(C::kDrain), 0, nullptr, 100000000ull);
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ activation groups
    const int wq = warp & 3;
    const int cbase = (warp >> 2) * 32;  // this group's 32 query columns of the tile
    const int j = wq * 32 + lane;        // key row within the block = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const float c_s = kSoftmax ? p.scale * kLog2e : p.scale;
    const float c_b = kSoftmax ? kLog2e : 1.0f;
    const bool has_bias = p.bias_table != nullptr;
    uint32_t it = 0, g = 0;
    uint32_t suse[2] = {0, 0};
    while (true) {
      const uint32_t slot = it & 1u;
      bool w = mbar_wait(bar(C::kItemFull + slot), (it >> 1) & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      const int2 item = item_slot[slot];
      mbar_arrive(bar(C::kItemEmpty + slot));
      ++it;
      if (item.x < 0) break;
      const BwdItem in = decode_bwd(item, p);
      const int kb0 = in.kb * kBwdKvRows;   // first local key row of the block
      const int jl = kb0 + j;               // this thread's local key row
      // queries that see this key: [vis_lo, vis_hi) (none for a key past the sample)
      const int vis_lo = band_query_begin(jl, p.causal, p.window);
      const int vis_hi = jl < in.Lkv ? band_query_end(jl, p.window, in.Lq) : 0;
      // Query tiles inside [full_lo, full_hi) pair with every key of a full
      // block and need no mask (the band's bounds grow with the key, so the
      // block's last key bounds the first such query and its first key the last).
      const int full_lo = band_query_begin(kb0 + kBwdKvRows - 1, p.causal, p.window);
      const int full_hi = kb0 + kBwdKvRows <= in.Lkv ? band_query_end(kb0, p.window, in.Lq) : 0;
      // dense bias of this key for query i: dcol[i * Lkv] (a key past the sample reads none)
      const float* dcol = (kDense && jl < in.Lkv)
                              ? p.bias_dense + p.bias_off[in.b] +
                                    static_cast<long long>(in.head) * in.Lq * in.Lkv + jl
                              : nullptr;
      // its gradient (p.dbias given with a dense bias), same layout: gcol[i * Lkv]
      float* gcol = (kDenseGrad && dcol != nullptr)
                        ? p.dbias + (dcol - p.bias_dense)
                        : nullptr;
      bool abort_now = false;
      for (int t = 0; t < in.nq; ++t, ++g) {
        const uint32_t s = g % C::kStages;
        const uint32_t buf = t & 1;
        w = mbar_wait(bar(C::kQdFull + s), (g / C::kStages) & 1u, abort_flag);
        w = w && mbar_wait(bar(C::kSFull + buf), suse[buf] & 1u, abort_flag);
        // the diagonal buffer of this tile was flushed two tiles ago
        if (kTableGrad) w = w && mbar_wait(bar(C::kDbFree + (g & 1u)), ((g >> 1) & 1u) ^ 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); abort_now = true; break; }
        suse[buf]++;
        tc_fence_after();
        const float* st = stats + s * C::kStatFloats;
        const float* bwin = st + 2 * kBwdQRows + (kBwdKvRows - 1) - j;  // bwin[c] = bias(q c, key j)
        const int qloc = (in.qt0 + t) * kBwdQRows;
        const bool full = qloc >= full_lo && qloc + kBwdQRows <= full_hi;
        int c_lo = 0, c_hi = kBwdQRows;  // valid query columns: c_lo <= c < c_hi
        if (!full) {
          c_hi = min(kBwdQRows, vis_hi - qloc);
          c_lo = max(0, vis_lo - qloc);
        }
        const uint32_t t_s = tmem + lane_off + kColS + buf * 64;
        const uint32_t t_dp = tmem + lane_off + kColDP;
        uint8_t* dsrow = gbase + C::kDs + buf * C::kDsParts * C::kDsBytes + j * 128;
        uint32_t sr[32];
        tmem_ld32(t_s + cbase, sr);  // all 32 scores first: P overwrites them in place
        // bias-table gradient: this lane's sums along four diagonals of the tile
        float diag[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int c0 = cbase + half * 16;
          uint32_t dr[16];
          tmem_ld16(t_dp + c0, dr);
          uint32_t phi[8], plo[8], dhi[8], dlo[8];
          float xd[16];  // dS of the 16 columns (bias-table gradient only)
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            float pv[2], dv[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int c = c0 + i + e;
              const float sv = __uint_as_float(sr[half * 16 + i + e]);
              const float dp = __uint_as_float(dr[i + e]);
              float bv = 0.0f;
              if (kDense) {
                if (dcol != nullptr && c >= c_lo && c < c_hi)
                  bv = __ldg(dcol + static_cast<long long>(qloc + c) * in.Lkv);
              } else if (has_bias) {
                bv = bwin[c];
              }
              if (kSoftmax) {
                const float pp = ex2_approx(fmaf(bv, c_b, fmaf(sv, c_s, -st[c])));
                pv[e] = pp;
                dv[e] = pp * (dp - st[kBwdQRows + c]);
              } else {
                float a, gr;
                act_and_grad<ACT>(fmaf(sv, c_s, bv), a, gr);
                pv[e] = a;
                dv[e] = gr * dp;
              }
              if (!full && (c < c_lo || c >= c_hi)) {
                pv[e] = 0.0f;
                dv[e] = 0.0f;
              }
              // dense-bias gradient: each pair is visited once, its dS added
              // straight to its entry
              if (kDenseGrad && gcol != nullptr && c >= c_lo && c < c_hi)
                atomicAdd(gcol + static_cast<long long>(qloc + c) * in.Lkv, dv[e]);
              if (kTableGrad) xd[i + e] = dv[e];
            }
            const uint32_t ph = pack_bf16x2(pv[0], pv[1]);
            const uint32_t dh = pack_bf16x2(dv[0], dv[1]);
            phi[i / 2] = ph;
            dhi[i / 2] = dh;
            if (kSplit) {
              plo[i / 2] = pack_bf16x2(pv[0] - __uint_as_float(ph << 16),
                                       pv[1] - __uint_as_float(ph & 0xFFFF0000u));
              dlo[i / 2] = pack_bf16x2(dv[0] - __uint_as_float(dh << 16),
                                       dv[1] - __uint_as_float(dh & 0xFFFF0000u));
            }
          }
          if (kTableGrad) {
            // dS(query c0 + i, key j = 32 wq + lane) lies on diagonal
            // (c0 - 32 wq + 127) + (i - lane).  Lane l gathers the warp's values
            // with i - src = l (mod 32): at step i it reads column i of lane
            // (i - l) mod 32, whose offset is l when i >= l and l - 32 otherwise.
            float up = 0.0f, down = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float v = __shfl_sync(0xffffffffu, xd[i], (i - lane) & 31);
              if (i >= lane) up += v; else down += v;
            }
            diag[2 * half] += down;
            diag[2 * half + 1] += up;
          }
          // P^T: query pair c/2 of the 32-column chunk lives at column chunk*32 + c/2 (hi)
          // and chunk*32 + 16 + c/2 (lo), where the dV MMA reads it.
          const uint32_t pc = t_s + cbase + half * 8;
          tmem_st8(pc, phi);
          if (kSplit) tmem_st8(pc + 16, plo);
          // dS^T row j, 128-byte swizzle: 16-byte chunk cc of the row lives at (cc ^ (j % 8))
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            const int cc = c0 / 8 + v;
            const int phys = (cc ^ (j & 7)) * 16;
            *reinterpret_cast<uint4*>(dsrow + phys) =
                make_uint4(dhi[4 * v], dhi[4 * v + 1], dhi[4 * v + 2], dhi[4 * v + 3]);
            if (kSplit)
              *reinterpret_cast<uint4*>(dsrow + C::kDsBytes + phys) =
                  make_uint4(dlo[4 * v], dlo[4 * v + 1], dlo[4 * v + 2], dlo[4 * v + 3]);
          }
        }
        if (kTableGrad) {
          // window entry (query - key + 127); a warp's lanes hit consecutive words
          float* win = reinterpret_cast<float*>(gbase + C::kDb + (g & 1u) * C::kDbBuf) +
                       (cbase - 32 * wq + 127 + lane);
          if (lane > 0) {  // some column lies left of this lane's diagonal
            atomicAdd(win - 32, diag[0]);
            atomicAdd(win - 16, diag[2]);
          }
          if (lane < 16) {  // some column lies on or right of it
            atomicAdd(win, diag[1]);
            atomicAdd(win + 16, diag[3]);
          }
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(C::kPFull));
        if (kTableGrad) {
          if (j == 0 && cbase == 0) {
            int* meta = reinterpret_cast<int*>(gbase + C::kDb + (g & 1u) * C::kDbBuf + 192 * 4);
            meta[0] = qloc - kb0 - 127;  // diagonal (query - key) of window entry 0
            meta[1] = in.head;
          }
          mbar_arrive(bar(C::kDbAcc + (g & 1u)));
        }
      }
      if (abort_now) break;
    }
  } else if (kTableGrad && warp == kMmaWarp + 1) {
    // ------------------------------------------------------------ bias-table gradient
    // Per tile: wait for the activation threads' diagonal sums, add them to the
    // table (entry = clamp(query - key + max_rel - 1)), zero the buffer.
    const int width = 2 * p.max_rel - 1;
    uint32_t it = 0, g = 0;
    while (true) {
      const uint32_t slot = it & 1u;
      bool w = mbar_wait(bar(C::kItemFull + slot), (it >> 1) & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      const int2 item = item_slot[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::kItemEmpty + slot));
      ++it;
      if (item.x < 0) break;
      const BwdItem in = decode_bwd(item, p);
      bool abort_now = false;
      for (int t = 0; t < in.nq; ++t, ++g) {
        const uint32_t u = g & 1u;
        w = mbar_wait(bar(C::kDbAcc + u), (g >> 1) & 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); abort_now = true; break; }
        float* win = reinterpret_cast<float*>(gbase + C::kDb + u * C::kDbBuf);
        const int* meta = reinterpret_cast<const int*>(win + 192);
        const int delta0 = meta[0];
        float* row = p.dbias + static_cast<long long>(meta[1]) * width;
        for (int e = lane; e < 191; e += 32) {
          const float v = win[e];
          if (v != 0.0f) atomicAdd(row + min(max(e + delta0 + p.max_rel - 1, 0), width - 1), v);
          win[e] = 0.0f;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::kDbFree + u));
      }
      if (abort_now) break;
    }
  } else if (warp < 12) {
    // ------------------------------------------------------------ dQ group + dK/dV epilogue
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // TMEM lane: channel (dQ^T) or key row (dK, dV)
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const bool out32 = aligned32(p.dk, p.dv);
    uint32_t it = 0, dqc = 0, dkvc = 0, dq_issue = 0;
    volatile int* group_ok = reinterpret_cast<volatile int*>(gbase + C::kGroupOk);
    while (true) {
      const uint32_t slot = it & 1u;
      bool w = mbar_wait(bar(C::kItemFull + slot), (it >> 1) & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      const int2 item = item_slot[slot];
      mbar_arrive(bar(C::kItemEmpty + slot));
      ++it;
      if (item.x < 0) break;
      const BwdItem in = decode_bwd(item, p);
      // every key of the sample is in this block: dQ goes out once, in bf16
      const bool direct = p.dq_direct_kv > 0 && in.Lkv <= p.dq_direct_kv;
      bool abort_now = false;
      for (int t = 0; t < in.nq; ++t) {
        w = mbar_wait(bar(C::kDqFull), dqc & 1u, abort_flag);
        // The group syncs on named barriers below, so its four warps must agree
        // on whether the wait succeeded before any of them can leave.
        w = __all_sync(0xffffffffu, w);
        if (lane == 0) group_ok[wq] = w ? 1 : 0;
        named_bar_sync(1, 128);
        const bool all_ok = group_ok[0] && group_ok[1] && group_ok[2] && group_ok[3];
        if (!all_ok) { if (lane == 0) fail(); abort_now = true; break; }
        ++dqc;
        tc_fence_after();
        uint32_t v0[32], v1[32];
        tmem_ld32(tmem + lane_off + kColDQ, v0);
        tmem_ld32(tmem + lane_off + kColDQ + 32, v1);
        tc_fence_before();
        mbar_arrive(bar(C::kDqEmpty));
        // Stage the tile as [query][channel] and add it into the fp32 dQ rows with
        // bulk tensor reduces: each warp its own 32 channels, 16 queries at a
        // time, from three buffers of its own (no group barrier).  Columns of
        // queries outside the sample carry exact zeros (their dS is masked to 0),
        // so a box that runs into the next sample's rows adds nothing; rows past
        // Tq are skipped.
        const int qrow = in.q0 + (in.qt0 + t) * kBwdQRows;
        const uint32_t wstage = sbase + C::kDqStage + wq * C::kDqWarpBufs * (C::kDqChunk * 32 * 4);
        float* wstg = reinterpret_cast<float*>(gbase + C::kDqStage) + wq * C::kDqWarpBufs * (C::kDqChunk * 32);
        if (direct) {
          // A sample whose keys fit one block: this item saw every key, so the
          // tile is dQ itself.  Each warp stages its 32 channels of 16 queries
          // as bf16 (times the scale) and writes them back as 16-byte row
          // pieces, only for the sample's own rows.
          if (lane == 0) bulk_wait_group_read<0>();  // no earlier reduce still reads the buffers
          __syncwarp();
          uint16_t* sb = reinterpret_cast<uint16_t*>(wstg);
#pragma unroll
          for (int ch = 0; ch < kBwdQRows / C::kDqChunk; ++ch) {
            if (32 * wq >= D) break;  // d = 64: warps 2 and 3 hold no channels
#pragma unroll
            for (int c = 0; c < C::kDqChunk; ++c) {
              const int q = ch * C::kDqChunk + c;
              sb[c * 32 + lane] = __bfloat16_as_ushort(
                  __float2bfloat16_rn(__uint_as_float(q < 32 ? v0[q & 31] : v1[q & 31]) * p.scale));
            }
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const int row = (lane >> 2) + 8 * k;  // query of the 16, 16-byte piece lane % 4
              const int qloc = (in.qt0 + t) * kBwdQRows + ch * C::kDqChunk + row;
              if (qloc < in.Lq)
                *reinterpret_cast<uint4*>(p.dq + (static_cast<long long>(in.q0 + qloc) * p.H + in.head) * D +
                                          32 * wq + 8 * (lane & 3)) =
                    *reinterpret_cast<const uint4*>(sb + row * 32 + 8 * (lane & 3));
            }
            __syncwarp();
          }
          continue;
        }
#pragma unroll
        for (int ch = 0; ch < kBwdQRows / C::kDqChunk; ++ch) {
          const int buf = dq_issue % C::kDqWarpBufs;
          if (lane == 0) bulk_wait_group_read<C::kDqWarpBufs - 1>();  // buffer `buf` is free again
          __syncwarp();
          if (32 * wq < D) {
            float* stg = wstg + buf * (C::kDqChunk * 32);
#pragma unroll
            for (int c = 0; c < C::kDqChunk; ++c) {
              const int q = ch * C::kDqChunk + c;
              stg[c * 32 + lane] = __uint_as_float(q < 32 ? v0[q & 31] : v1[q & 31]);
            }
            fence_proxy_async_smem();
          }
          __syncwarp();
          if (lane == 0 && 32 * wq < D) {
            tma_reduce_add_3d(&tmap_dq, wstage + buf * (C::kDqChunk * 32 * 4), 32 * wq, in.head,
                              qrow + ch * C::kDqChunk);
            bulk_commit_group();
          }
          ++dq_issue;
        }
      }
      if (abort_now) break;
      // epilogue: dV and dK rows of this key block
      const int jl = in.kb * kBwdKvRows + r;
      const bool row_ok = jl < in.Lkv;
      const long long grow = (static_cast<long long>(in.k0 + jl) * p.H + in.head) * D;
      if (in.nq > 0) {
        w = mbar_wait(bar(C::kDkvFull), dkvc & 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
        ++dkvc;
        tc_fence_after();
#pragma unroll 1
        for (int which = 0; which < 2; ++which) {
          const uint32_t col = which ? kColDK : kColDV;
          const float mul = which ? p.scale : 1.0f;
          __nv_bfloat16* dst = (which ? p.dk : p.dv) + grow;
          if (which == 1 && p.rope_base > 0.0f) {  // dK back through the rotary embedding
            rope_bwd_row<D>(tmem + lane_off + col, mul, jl, -2.0f * log2f(p.rope_base) / D, dst,
                            row_ok);
            continue;
          }
#pragma unroll 1
          for (int chunk = 0; chunk < D / 32; ++chunk) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_off + col + chunk * 32, o);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * mul, __uint_as_float(o[2 * i + 1]) * mul);
            if (row_ok) store_words(dst + chunk * 32, pk, out32);
          }
        }
        tc_fence_before();
        mbar_arrive(bar(C::kDkvEmpty));
      } else if (row_ok) {
        uint4* a4 = reinterpret_cast<uint4*>(p.dv + grow);
        uint4* b4 = reinterpret_cast<uint4*>(p.dk + grow);
        for (int v = 0; v < D / 8; ++v) {
          a4[v] = make_uint4(0, 0, 0, 0);
          b4[v] = make_uint4(0, 0, 0, 0);
        }
      }
    }
    if (lane == 0) bulk_wait_group_all();  // every dQ reduce issued by this thread has landed
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Zero the fp32 dQ accumulator and (softmax) compute D = rowsum(dO * O).
// A row of d bf16 values is d/8 16-byte vectors: each lane takes one vector of
// O and of dO, and 16 (d = 128) or 8 (d = 64) lanes share a row, so a warp
// covers 2 or 4 rows per step with full-width loads and stores.
template <int D>
__global__ void __launch_bounds__(256)
bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ out, const __nv_bfloat16* __restrict__ dout,
                      float* __restrict__ delta, float* __restrict__ dq_acc, long long Tq, int H,
                      int softmax, const int* __restrict__ all_short) {
  constexpr int kLanesPerRow = D / 8;
  // no sample reduces into the accumulator: leave it alone
  const bool zero_acc = all_short == nullptr || *all_short == 0;
  if (!zero_acc && !softmax) return;
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  const long long nrows = Tq * H;
  const int lane = threadIdx.x & 31;
  const int sub = lane / kLanesPerRow;   // row of the warp's group
  const int v = lane % kLanesPerRow;     // 16-byte vector within the row
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
  for (long long row0 = (blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32) * kRowsPerWarp;
       row0 < nrows; row0 += warps * kRowsPerWarp) {
    const long long row = row0 + sub;
    const bool ok = row < nrows;
    if (ok && zero_acc) {
      float4* acc = reinterpret_cast<float4*>(dq_acc + row * D) + 2 * v;
      acc[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      acc[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (softmax) {
      float s = 0.f;
      if (ok) {
        const uint4 a = reinterpret_cast<const uint4*>(out + row * D)[v];
        const uint4 b = reinterpret_cast<const uint4*>(dout + row * D)[v];
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          s = fmaf(__uint_as_float(aw[k] << 16), __uint_as_float(bw[k] << 16), s);
          s = fmaf(__uint_as_float(aw[k] & 0xFFFF0000u), __uint_as_float(bw[k] & 0xFFFF0000u), s);
        }
      }
#pragma unroll
      for (int off = kLanesPerRow / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      if (ok && v == 0) {
        const long long t = row / H, h = row % H;
        delta[h * Tq + t] = s;
      }
    }
  }
}

// dq = bf16(dq_acc * scale), eight values (two 16-byte loads, one 16-byte
// store) per thread and step.
__global__ void __launch_bounds__(256)
dq_convert_kernel(const float4* __restrict__ acc, uint4* __restrict__ dq, long long n8, float scale,
                  const int* __restrict__ skip) {
  if (skip != nullptr && *skip != 0) return;  // dq was written directly
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 a = acc[2 * i];
    const float4 b = acc[2 * i + 1];
    dq[i] = make_uint4(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale),
                       pack_bf16x2(b.x * scale, b.y * scale), pack_bf16x2(b.z * scale, b.w * scale));
  }
}

// With dQ written directly for some samples (BwdParams::dq_direct_kv) the
// accumulator is zeroed and converted only for the others.  Each block takes
// kSegTokens consecutive tokens, finds the sample holding the first one (one
// binary search over the offsets) and walks the samples of its range, handing
// the accumulated pieces [a, b) of tokens to f: whole rows of H * d values,
// contiguous in memory, so the block's stores stay coalesced.
constexpr int kSegTokens = 64;
template <typename F>
__device__ __forceinline__ void acc_segments(const int32_t* __restrict__ qo,
                                             const int32_t* __restrict__ ko, int B, long long Tq,
                                             int direct_kv, int short_q_max, F&& f) {
  const long long t0 = static_cast<long long>(blockIdx.x) * kSegTokens;
  const long long t1 = min(Tq, t0 + kSegTokens);
  if (t0 >= t1) return;
  int lo = 0, hi = B - 1;  // the last sample starting at or before t0
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(qo + mid) <= t0) lo = mid; else hi = mid - 1;
  }
  long long t = t0;
  for (int s = lo; s < B && t < t1; ++s) {
    const long long e = min(t1, static_cast<long long>(__ldg(qo + s + 1)));
    if (e <= t) continue;
    const int Lq = __ldg(qo + s + 1) - __ldg(qo + s);
    const int Lkv = __ldg(ko + s + 1) - __ldg(ko + s);
    if (!(Lkv >= 1 && Lkv <= direct_kv && Lq > short_q_max)) f(t, e);
    t = e;
  }
}

__global__ void __launch_bounds__(256)
dq_zero_segments_kernel(float4* __restrict__ acc, const int32_t* __restrict__ qo,
                        const int32_t* __restrict__ ko, int B, long long Tq, int H, int d,
                        int direct_kv, int short_q_max, const int* __restrict__ all_short) {
  if (all_short != nullptr && *all_short != 0) return;  // nothing reduces into the accumulator
  const long long row4 = static_cast<long long>(H) * d / 4;  // float4 per token
  acc_segments(qo, ko, B, Tq, direct_kv, short_q_max, [&](long long a, long long b) {
    for (long long i = a * row4 + threadIdx.x; i < b * row4; i += blockDim.x)
      acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  });
}

__global__ void __launch_bounds__(256)
dq_convert_segments_kernel(const float4* __restrict__ acc, uint4* __restrict__ dq, float scale,
                           const int32_t* __restrict__ qo, const int32_t* __restrict__ ko, int B,
                           long long Tq, int H, int d, int direct_kv, int short_q_max,
                           const int* __restrict__ skip) {
  if (skip != nullptr && *skip != 0) return;  // dq was written directly
  const long long row8 = static_cast<long long>(H) * d / 8;  // 8-value groups per token
  acc_segments(qo, ko, B, Tq, direct_kv, short_q_max, [&](long long a, long long b) {
    for (long long i = a * row8 + threadIdx.x; i < b * row8; i += blockDim.x) {
      const float4 x = acc[2 * i];
      const float4 y = acc[2 * i + 1];
      dq[i] = make_uint4(pack_bf16x2(x.x * scale, x.y * scale), pack_bf16x2(x.z * scale, x.w * scale),
                         pack_bf16x2(y.x * scale, y.y * scale), pack_bf16x2(y.z * scale, y.w * scale));
    }
  });
}

// dq = bf16 of the rotary backward of scale * acc: each thread takes channels
// c..c+3 of one (token, head) row and their partners c + d/2 .. c + d/2 + 3,
// the token's position found by a binary search over the sample offsets.
__global__ void __launch_bounds__(256)
dq_convert_rope_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq,
                       const int32_t* __restrict__ offsets, int B, long long T, int H, int d,
                       float scale, float rope_k) {
  const int per_row = d / 8;
  const long long units = T * H * per_row;
  for (long long u = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; u < units;
       u += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = u / per_row;          // (token, head) row
    const int c = 4 * static_cast<int>(u % per_row);
    const long long t = row / H;
    int lo = 0, hi = B - 1;  // last sample starting at or before t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (offsets[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int pos = static_cast<int>(t - offsets[lo]);
    const float4 g1 = *reinterpret_cast<const float4*>(acc + row * d + c);
    const float4 g2 = *reinterpret_cast<const float4*>(acc + row * d + d / 2 + c);
    const float a1[4] = {g1.x * scale, g1.y * scale, g1.z * scale, g1.w * scale};
    const float a2[4] = {g2.x * scale, g2.y * scale, g2.z * scale, g2.w * scale};
    float r1[4], r2[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float sn, cs;
      sincosf(static_cast<float>(pos) * exp2f(static_cast<float>(c + e) * rope_k), &sn, &cs);
      r1[e] = fmaf(a1[e], cs, a2[e] * sn);
      r2[e] = fmaf(a2[e], cs, -a1[e] * sn);
    }
    *reinterpret_cast<uint2*>(dq + row * d + c) = make_uint2(pack_bf16x2(r1[0], r1[1]), pack_bf16x2(r1[2], r1[3]));
    *reinterpret_cast<uint2*>(dq + row * d + d / 2 + c) =
        make_uint2(pack_bf16x2(r2[0], r2[1]), pack_bf16x2(r2[2], r2[3]));
  }
}

template <int D, int ACT, bool kDBias, bool kDense>
cudaError_t launch_main_db(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                           int grid, cudaStream_t s) {
  using C = BwdCfg<D, ACT != GDPA_ACT_SOFTMAX>;
  cudaError_t e = cudaFuncSetAttribute(bwd_kernel<D, ACT, kDBias, kDense>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  bwd_kernel<D, ACT, kDBias, kDense><<<grid, kThreads + (kDBias && !kDense ? 32 : 0),
                                      C::kSmemBytes, s>>>(
      tq, tk, tv, tdo, tdq, p);
  return cudaGetLastError();
}

template <int D, int ACT>
cudaError_t launch_main(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                        int grid, cudaStream_t s) {
  if (p.bias_dense != nullptr) {
    return p.dbias != nullptr ? launch_main_db<D, ACT, true, true>(p, tq, tk, tv, tdo, tdq, grid, s)
                              : launch_main_db<D, ACT, false, true>(p, tq, tk, tv, tdo, tdq, grid, s);
  }
  return p.dbias != nullptr ? launch_main_db<D, ACT, true, false>(p, tq, tk, tv, tdo, tdq, grid, s)
                            : launch_main_db<D, ACT, false, false>(p, tq, tk, tv, tdo, tdq, grid, s);
}

template <int D>
cudaError_t launch_main_d(const BwdParams& p, int act, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                          int grid, cudaStream_t s) {
  switch (act) {
    case GDPA_ACT_SILU: return launch_main<D, GDPA_ACT_SILU>(p, tq, tk, tv, tdo, tdq, grid, s);
    case GDPA_ACT_GELU_TANH:
      return launch_main<D, GDPA_ACT_GELU_TANH>(p, tq, tk, tv, tdo, tdq, grid, s);
    case GDPA_ACT_GELU_ERF: return launch_main<D, GDPA_ACT_GELU_ERF>(p, tq, tk, tv, tdo, tdq, grid, s);
    default: return launch_main<D, GDPA_ACT_IDENTITY>(p, tq, tk, tv, tdo, tdq, grid, s);
  }
}

}  // namespace

cudaError_t launch_bwd(const BwdParams& p, int act, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                       int grid,
                       cudaStream_t stream, int* launches, cudaEvent_t ev_begin,
                       cudaEvent_t ev_end, const ShortBwd* sq) {
  // 1) zero dQ accumulator, D = rowsum(dO * O)
  cudaError_t e = launch_bwd_preprocess(p, act == GDPA_ACT_SOFTMAX, stream);
  if (e != cudaSuccess) return e;
  ++*launches;
  // 2) main kernel (optionally bracketed by timing events)
  if (ev_begin != nullptr && (e = cudaEventRecord(ev_begin, stream)) != cudaSuccess) return e;
  if (act == GDPA_ACT_SOFTMAX)
    e = launch_bwd_softmax_main(p, tq, tk, tv, tdo, tdq, grid, stream);
  else
    e = (p.d == 64) ? launch_main_d<64>(p, act, tq, tk, tv, tdo, tdq, grid, stream)
                    : launch_main_d<128>(p, act, tq, tk, tv, tdo, tdq, grid, stream);
  if (e != cudaSuccess) return e;
  ++*launches;
  if (sq != nullptr) {
    // the short-query items (an empty list makes the kernel return at once)
    e = launch_bwd_short_q(sq->p, act, sq->tq, tk, tv, sq->tdo, sq->dq, sq->grid, stream);
    if (e != cudaSuccess) return e;
    ++*launches;
  }
  if (ev_end != nullptr && (e = cudaEventRecord(ev_end, stream)) != cudaSuccess) return e;
  return cudaSuccess;
}

cudaError_t launch_bwd_preprocess(const BwdParams& p, bool softmax, cudaStream_t stream) {
  if (!softmax && p.dq_direct_kv > 0) {  // only the accumulated samples' rows need zeros
    const long long blocks = (p.Tq + kSegTokens - 1) / kSegTokens;
    if (blocks == 0) return cudaSuccess;
    dq_zero_segments_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        reinterpret_cast<float4*>(p.dq_acc), p.qo, p.ko, p.B, p.Tq, p.H, p.d, p.dq_direct_kv,
        p.short_q_max, p.all_short);
    return cudaGetLastError();
  }
  const long long rows = p.Tq * p.H;
  const int pre_blocks = static_cast<int>(rows / 8 + 1 < 4096 ? rows / 8 + 1 : 4096);
  if (p.d == 64)
    bwd_preprocess_kernel<64><<<pre_blocks, 256, 0, stream>>>(p.out, p.dout, p.delta, p.dq_acc,
                                                              p.Tq, p.H, softmax ? 1 : 0,
                                                              p.all_short);
  else
    bwd_preprocess_kernel<128><<<pre_blocks, 256, 0, stream>>>(p.out, p.dout, p.delta, p.dq_acc,
                                                               p.Tq, p.H, softmax ? 1 : 0,
                                                               p.all_short);
  return cudaGetLastError();
}

cudaError_t launch_dq_convert_rope(const float* acc, void* dq, const int32_t* offsets, int B,
                                   long long T, int H, int d, float scale, float rope_base,
                                   cudaStream_t stream) {
  const long long units = T * H * (d / 8);  // 4 channels of the first half and their partners
  const int blocks = static_cast<int>(units / 256 + 1 < 8192 ? units / 256 + 1 : 8192);
  dq_convert_rope_kernel<<<blocks, 256, 0, stream>>>(acc, static_cast<__nv_bfloat16*>(dq), offsets,
                                                     B, T, H, d, scale,
                                                     -2.0f * log2f(rope_base) / d);
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(const float* acc, void* dq, long long n, float scale,
                              cudaStream_t stream, const int* skip, const BwdParams* direct) {
  if (direct != nullptr && direct->dq_direct_kv > 0) {  // the accumulated samples' rows only
    const long long blocks = (direct->Tq + kSegTokens - 1) / kSegTokens;
    if (blocks == 0) return cudaSuccess;
    dq_convert_segments_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        reinterpret_cast<const float4*>(acc), reinterpret_cast<uint4*>(dq), scale, direct->qo,
        direct->ko, direct->B, direct->Tq, direct->H, direct->d, direct->dq_direct_kv,
        direct->short_q_max, skip);
    return cudaGetLastError();
  }
  const long long n8 = n / 8;  // n = Tq * H * d with d in {64, 128}
  const int blocks = static_cast<int>(n8 / 256 + 1 < 8192 ? n8 / 256 + 1 : 8192);
  dq_convert_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(acc),
                                                reinterpret_cast<uint4*>(dq), n8, scale, skip);
  return cudaGetLastError();
}

}  // namespace gdpa
