// Forward kernel of jagged attention with a pluggable activation, sm_103a.
//
// "GEM Training ..." GDPA paragraph: two matrix multiplications with an
// elementwise activation in between (softmax -> JFA, GELU / SiLU -> GDPA).
// JFA paragraph: operate directly on jagged tensors with no padding, with
// custom attention biases and asymmetric query / key lengths.
//
// Design (one persistent CTA per SM, warp-specialised, 384 threads = three
// warpgroups):
//   warps 0-3   "softmax group 0": query rows [0,128) of the item
//   warps 4-7   "softmax group 1": query rows [128,256) of the item
//   warp  8     TMA producer: pulls work items from the cost-sorted list
//               (atomic ticket), loads Q once per item and K/V tiles into a
//               ring of shared-memory stages
//   warp  9     MMA issuer: tcgen05.mma S_h = Q_h K^T into TMEM, then
//               O_h += P_h V with P_h read from TMEM
//   warps 10-11 idle
// Registers: each SM sub-partition holds 16384; the launch gives every thread
// 168 (three warps per sub-partition), then the activation warpgroups rise to
// 200 and the producer / MMA warpgroup drops to 104 (setmaxnreg), so a row's
// 128 scores and their exponentials stay in registers without spilling.
// TMEM (512 columns): half h owns S/P columns [256h, 256h+128) and O columns
// [256h+128, 256h+128+d).  The activation group reads S row by row (TMEM lane
// = query row), applies scale, bias, mask and the activation in registers
// and writes P back into the same columns as packed bf16.  Softmax keeps an
// online row max / sum and rescales O in TMEM only when the max grows by
// more than 2^8 (stale maxima are exact after the final division).  GDPA
// activations need no normalisation; their P is split into bf16 hi + lo
// parts (two MMAs) because a single 16-bit P loses too much precision when
// thousands of unnormalised terms are summed.
//
// Issue order per item (MMA warp):  S0(0) S1(0) | PV0(j) S0(j+1) PV1(j) S1(j+1) ...
// so that while one group runs its activation the tensor core works on the
// other group's tile.  tcgen05 MMAs from one thread complete in order, which
// makes S_h(j+1) overwriting P_h(j) safe and guarantees that when S_h(j) is
// complete, PV_h(j-1) is too (so O may be rescaled then).
//
// Every mbarrier wait is bounded; on a timeout the CTA records
// GDPA_ERR_TIMEOUT in the status word, drains its own copies and MMAs with a
// short bounded wait, frees TMEM and exits.
#include "common.cuh"

namespace gdpa {
namespace {

using namespace ptx;

constexpr int kThreads = 384;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kActWarps = 8;
constexpr int kRegsAct = 200;  // activation warpgroups
constexpr int kRegsLow = 104;  // producer / MMA warpgroup
static_assert(2 * kRegsAct + kRegsLow == 3 * 168, "register split must keep the launch total");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct FwdCfg {
  static constexpr int kQHalfBytes = kHalfRows * D * 2;
  static constexpr int kTileBytes = kKvRows * D * 2;
  static constexpr int kStages = (D == 128) ? 2 : 4;
  static constexpr int kQ0 = 0;
  static constexpr int kQ1 = kQHalfBytes;
  static constexpr int kKV = 2 * kQHalfBytes;                          // K[s] = kKV + s*2*tile
  // per stage and half: the bias window (255 relative positions, in reverse
  // order, times log2e for softmax) in two copies shifted by 0 and 1 entries,
  // kBiasCopy floats apart: every query row finds its 128 entries of a key
  // tile 8-byte aligned in one copy, and with this stride the 64-bit loads of
  // a warp hit every bank once
  static constexpr int kBiasCopy = 270;
  static constexpr int kBiasBlock = 2 * kBiasCopy;                     // floats per stage and half
  static constexpr int kBias = kKV + kStages * 2 * kTileBytes;
  static constexpr int kBar = kBias + kStages * 2 * kBiasBlock * 4;   // barriers after tiles
  // barrier block layout (8 bytes each)
  static constexpr int kQFull = 0, kQEmpty = 1;
  static constexpr int kKFull = 2;                                     // + s
  static constexpr int kVFull = kKFull + kStages;
  static constexpr int kKEmpty = kVFull + kStages;                     // K tile consumed
  static constexpr int kVEmpty = kKEmpty + kStages;                    // V tile (+ bias window) consumed
  static constexpr int kSFull = kVEmpty + kStages;                     // + half
  static constexpr int kPFull = kSFull + 2;
  static constexpr int kODone = kPFull + 2;
  static constexpr int kItemFull = kODone + 2;                         // + slot
  static constexpr int kItemEmpty = kItemFull + 2;
  static constexpr int kDrain = kItemEmpty + 2;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kItemSlots = kBar + 8 * kNumBars;               // int2[2]
  static constexpr int kTmemSlot = kItemSlots + 16;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kUsed = kAbort + 4;
  static constexpr int kSmemBytes = kUsed + 1024;                      // + alignment slack
};

__device__ __forceinline__ float act_apply(int act, float x) {
  if (act == GDPA_ACT_SILU) {
    const float h = 0.5f * x;
    return fmaf(h, tanh_approx(h), h);
  }
  if (act == GDPA_ACT_GELU_TANH) {
    // 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))
    const float k0 = 0.7978845608028654f, k1 = 0.7978845608028654f * 0.044715f;
    const float u = x * fmaf(k1, x * x, k0);
    const float h = 0.5f * x;
    return fmaf(h, tanh_approx(u), h);
  }
  if (act == GDPA_ACT_GELU_ERF) return 0.5f * x * (1.0f + erff(x * 0.7071067811865476f));
  return x;  // identity
}

struct ItemInfo {
  int b, head, blk;
  int q0, k0, Lq, Lkv;
  // Key tiles visited: half h covers [lo_h, hi_h) (empty when lo_h == hi_h);
  // the item streams their union [jb, je), which is contiguous because the
  // causal / window band of consecutive rows is.
  int lo0, hi0, lo1, hi1;
  int jb, je;
  __device__ __forceinline__ int lo(int h) const { return h ? lo1 : lo0; }
  __device__ __forceinline__ int hi(int h) const { return h ? hi1 : hi0; }
  __device__ __forceinline__ bool visits(int h, int j) const { return j >= lo(h) && j < hi(h); }
  __device__ __forceinline__ bool has_half1() const { return hi1 > lo1; }
};

// kBand: a sliding window is set (p.window > 0).  Without one every half
// starts at key tile 0, which keeps the common path's arithmetic minimal.
template <bool kBand>
__device__ __forceinline__ ItemInfo decode_item(int2 it, const FwdParams& p) {
  ItemInfo r;
  r.b = it.x;
  r.head = item_head(it);
  r.blk = item_block(it);
  r.q0 = p.qo[r.b];
  r.Lq = p.qo[r.b + 1] - r.q0;
  r.k0 = p.ko[r.b];
  r.Lkv = p.ko[r.b + 1] - r.k0;
  const int r0 = r.blk * kItemRows;
  if (kBand) {
    band_key_tiles(r0, min(r.Lq, r0 + kHalfRows), p.causal, p.window, r.Lkv, kKvRows, &r.lo0,
                   &r.hi0);
    if (r0 + kHalfRows < r.Lq)
      band_key_tiles(r0 + kHalfRows, min(r.Lq, r0 + kItemRows), p.causal, p.window, r.Lkv,
                     kKvRows, &r.lo1, &r.hi1);
    else
      r.lo1 = r.hi1 = r.hi0;
  } else {
    const int nkv = (r.Lkv + kKvRows - 1) / kKvRows;
    const bool h1 = r0 + kHalfRows < r.Lq;
    r.lo0 = r.lo1 = 0;
    if (!p.causal) {
      r.hi0 = nkv;
      r.hi1 = h1 ? nkv : 0;
    } else {
      r.hi0 = min(nkv, (min(r.Lq, r0 + kHalfRows) + kKvRows - 1) / kKvRows);
      r.hi1 = h1 ? min(nkv, (min(r.Lq, r0 + kItemRows) + kKvRows - 1) / kKvRows) : 0;
    }
  }
  // Half 0 starts no later and half 1 ends no earlier; with half 0 empty
  // (no key at all) both are.
  r.jb = r.lo0;
  r.je = max(r.hi0, r.hi1);
  return r;
}

// kDense: a dense jagged bias (p.bias_dense) instead of the relative-position
// table; its rows are read from global memory by the activation warps.
template <int D, int ACT, bool kBand, bool kDense>
__global__ void __launch_bounds__(kThreads, 1)
fwd_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
           const __grid_constant__ CUtensorMap tmap_v, const FwdParams p) {
  using C = FwdCfg<D>;
  constexpr bool kSoftmax = (ACT == GDPA_ACT_SOFTMAX);
  constexpr bool kSplit = !kSoftmax;  // GDPA: P = hi + lo

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
    mbar_init(bar(C::kQFull), 1);
    mbar_init(bar(C::kQEmpty), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kKFull + s), 1);
      mbar_init(bar(C::kVFull + s), 1);
      mbar_init(bar(C::kKEmpty + s), 1);
      mbar_init(bar(C::kVEmpty + s), 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(bar(C::kSFull + h), 1);
      mbar_init(bar(C::kPFull + h), kHalfRows);
      mbar_init(bar(C::kODone + h), 1);
      mbar_init(bar(C::kItemFull + h), 1);
      mbar_init(bar(C::kItemEmpty + h), 1 + 2 * kHalfRows);
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
    // ------------------------------------------------------------ producer (whole warp)
    setmaxnreg_dec<kRegsLow>();
    // Lane 0 takes tickets and issues the TMA copies; all lanes stage the
    // bias windows of each key tile (when there is a bias).
    const int n_items = *p.n_items;
    const int rel_w = 2 * p.max_rel - 1;
    float* bias_win = reinterpret_cast<float*>(gbase + C::kBias);
    uint32_t it = 0, g = 0, qi = 0;
    uint32_t inflight = 0;  // stages whose K/V load may still be in flight (abort drain)
    bool q_inflight = false;
    uint32_t last_g[C::kStages] = {};
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
      const ItemInfo in = decode_item<kBand>(item, p);
      const int n = in.je - in.jb;
      if (n == 0) continue;
      w = mbar_wait(bar(C::kQEmpty), (qi & 1u) ^ 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      const int row0 = in.q0 + in.blk * kItemRows;
      const int n_halves = in.has_half1() ? 2 : 1;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(C::kQFull), n_halves * C::kQHalfBytes);
        for (int half = 0; half < n_halves; ++half)
          for (int x = 0; x < D; x += 64)
            tma_load_3d(sbase + (half ? C::kQ1 : C::kQ0) + (x / 64) * (kHalfRows * 128),
                        &tmap_q, bar(C::kQFull), x, in.head, row0 + half * kHalfRows);
        q_inflight = true;
      }
      ++qi;
      const float* brow =
          p.bias_table ? p.bias_table + static_cast<long long>(in.head) * rel_w : nullptr;
      // Window entry e of half h for key tile j holds bias(i - j') with
      // (i - r_h) - (j' - c0) = e - 127 (r_h: the half's first local row, c0: the
      // tile's first local column).  Each lane holds entries lane + 32k of both
      // halves, fetched one tile ahead so the load latency overlaps the wait for
      // a free stage.
      constexpr float kBiasMul = kSoftmax ? kLog2e : 1.0f;  // exponents are in log2 units
      auto fetch = [&](int j, float (&v)[16]) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int w0 = in.blk * kItemRows + h * kHalfRows - j * kKvRows - (kKvRows - 1) +
                         p.max_rel - 1;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int e = lane + 32 * k;
            v[8 * h + k] = (brow != nullptr && e < 255)
                               ? __ldg(brow + min(max(w0 + e, 0), rel_w - 1)) * kBiasMul
                               : 0.0f;
          }
        }
      };
      float cur[16];
      if (brow != nullptr) fetch(in.jb, cur);
      for (int j = in.jb; j < in.je; ++j, ++g) {
        const uint32_t s = g % C::kStages;
        const uint32_t ph = (g / C::kStages) & 1u;
        const uint32_t kdst = sbase + C::kKV + s * 2 * C::kTileBytes;
        const int krow = in.k0 + j * kKvRows;
        w = mbar_wait(bar(C::kKEmpty + s), ph ^ 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { ok = false; if (lane == 0) fail(); break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(C::kKFull + s), C::kTileBytes);
          for (int x = 0; x < D; x += 64)
            tma_load_3d(kdst + (x / 64) * (kKvRows * 128), &tmap_k, bar(C::kKFull + s), x,
                        in.head, krow);
          inflight |= 1u << s;
          last_g[s] = g;
        }
        // The V slot (and this tile's bias windows) frees up after the tile's
        // value products, later than the K slot.
        w = mbar_wait(bar(C::kVEmpty + s), ph ^ 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { ok = false; if (lane == 0) fail(); break; }
        float nxt[16];
        if (brow != nullptr) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float* win = bias_win + (s * 2 + h) * C::kBiasBlock;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int e = lane + 32 * k;
              if (e < 255) {
#pragma unroll
                for (int cp = 0; cp < 2; ++cp)  // entry e at position (254 - e) + cp of copy cp
                  win[cp * C::kBiasCopy + cp + 254 - e] = cur[8 * h + k];
              }
            }
          }
          if (j + 1 < in.je) fetch(j + 1, nxt);
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(C::kVFull + s), C::kTileBytes);
          for (int x = 0; x < D; x += 64)
            tma_load_3d(kdst + C::kTileBytes + (x / 64) * (kKvRows * 128), &tmap_v,
                        bar(C::kVFull + s), x, in.head, krow);
        }
        if (brow != nullptr && j + 1 < in.je) {
#pragma unroll
          for (int k = 0; k < 16; ++k) cur[k] = nxt[k];
        }
      }
    }
    if (lane == 0 && *abort_flag) {
      // Drain: wait (briefly, bounded) for copies this thread issued.
      for (int s = 0; s < C::kStages; ++s)
        if (inflight & (1u << s)) {
          const uint32_t ph = (last_g[s] / C::kStages) & 1u;
          mbar_wait(bar(C::kKFull + s), ph, nullptr, 50000000ull);
          mbar_wait(bar(C::kVFull + s), ph, nullptr, 50000000ull);
        }
      if (q_inflight) mbar_wait(bar(C::kQFull), (qi - 1) & 1u, nullptr, 50000000ull);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    setmaxnreg_dec<kRegsLow>();
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16(128, 128, true, false, false);
      constexpr uint32_t idesc_pv = idesc_f16(128, D, true, false, true);
      uint32_t it = 0, g = 0, qi = 0;
      uint32_t tcount[2] = {0, 0};
      bool issued_any = false;
      // Descriptors at each operand's first byte; stages, halves and k-steps
      // are added to the start-address field (see dadd), keeping the issue
      // loop short: this warp shares its sub-partition with busy warps.
      const uint64_t dsc_q = sdesc(sbase + C::kQ0, 0, 1024, kSwizzle128B);   // A of S (K-major)
      const uint64_t dsc_k = sdesc(sbase + C::kKV, 0, 1024, kSwizzle128B);   // B of S (K-major)
      const uint64_t dsc_v = sdesc(sbase + C::kKV + C::kTileBytes, kKvRows * 128, 1024,
                                   kSwizzle128B);                             // B of PV (MN-major)
      auto issue_s = [&](int half, uint32_t stage) {
        const uint64_t qb = dadd(dsc_q, half ? C::kQ1 - C::kQ0 : 0);
        const uint64_t kb = dadd(dsc_k, stage * 2 * C::kTileBytes);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t qoff = (ks / 4) * (kHalfRows * 128) + (ks % 4) * 32;
          const uint32_t koff = (ks / 4) * (kKvRows * 128) + (ks % 4) * 32;
          mma_f16_ss(tmem + half * 256, dadd(qb, qoff), dadd(kb, koff), idesc_s, ks > 0 ? 1u : 0u);
        }
        mma_commit(bar(C::kSFull + half));
        issued_any = true;
      };
      auto issue_pv = [&](int half, uint32_t stage, bool first) {
        const uint64_t vb = dadd(dsc_v, stage * 2 * C::kTileBytes);
        const uint32_t tp = tmem + half * 256;
        const uint32_t to = tmem + half * 256 + 128;
#pragma unroll
        for (int ks = 0; ks < kKvRows / 16; ++ks) {
          const uint32_t pcol = 32 * (ks / 2) + 8 * (ks % 2);
          mma_f16_ts(to, tp + pcol, dadd(vb, ks * 2048), idesc_pv, (first && ks == 0) ? 0u : 1u);
          if (kSplit) mma_f16_ts(to, tp + pcol + 16, dadd(vb, ks * 2048), idesc_pv, 1u);
        }
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
        const ItemInfo in = decode_item<kBand>(item, p);
        const int n = in.je - in.jb;
        if (n == 0) continue;
        if (!mbar_wait(bar(C::kQFull), qi & 1u, abort_flag)) { fail(); break; }
        ++qi;
        tc_fence_after();
        // Key tile j's last score product is half 1's when half 1 visits j;
        // the item's last score product is that of tile je - 1.
        const int last_s_half = in.visits(1, in.je - 1) ? 1 : 0;
        {
          const uint32_t s = g % C::kStages;
          if (!mbar_wait(bar(C::kKFull + s), (g / C::kStages) & 1u, abort_flag)) { fail(); break; }
          tc_fence_after();
          if (in.visits(0, in.jb)) issue_s(0, s);
          if (in.visits(1, in.jb)) issue_s(1, s);
          mma_commit(bar(C::kKEmpty + s));  // the first K tile has all its readers
          if (n == 1) mma_commit(bar(C::kQEmpty));
        }
        for (int j = in.jb; j < in.je; ++j) {
          const uint32_t gj = g + (j - in.jb);
          const uint32_t s = gj % C::kStages;
          const uint32_t s_next = (gj + 1) % C::kStages;
          const uint32_t ph_next = ((gj + 1) / C::kStages) & 1u;
          if (!mbar_wait(bar(C::kVFull + s), (gj / C::kStages) & 1u, abort_flag)) { ok = false; fail(); break; }
          const int last_half_j = in.visits(1, j) ? 1 : 0;  // last user of stage s
          const int last_half_next = in.visits(1, j + 1) ? 1 : 0;
          for (int half = 0; half < 2; ++half) {
            if (in.visits(half, j)) {
              if (!mbar_wait(bar(C::kPFull + half), tcount[half] & 1u, abort_flag)) { ok = false; fail(); break; }
              ++tcount[half];
              tc_fence_after();
              issue_pv(half, s, j == in.lo(half));
              if (j == in.hi(half) - 1) mma_commit(bar(C::kODone + half));
              if (half == last_half_j) mma_commit(bar(C::kVEmpty + s));
            }
            // S of the next tile (a half may start there: a sliding window
            // moves half 1's first tile past half 0's)
            if (in.visits(half, j + 1)) {
              if (!mbar_wait(bar(C::kKFull + s_next), ph_next, abort_flag)) { ok = false; fail(); break; }
              tc_fence_after();
              issue_s(half, s_next);
              if (half == last_half_next) mma_commit(bar(C::kKEmpty + s_next));
              if (j + 1 == in.je - 1 && half == last_s_half) mma_commit(bar(C::kQEmpty));
            }
          }
          if (!ok) break;
        }
        g += n;
      }
      // Make sure every MMA this thread issued has completed before TMEM is freed.
      if (issued_any) {
        mma_commit(bar(C::kDrain));
        mbar_wait(bar(C::kDrain), 0, nullptr, 100000000ull);
      }
    }
  } else if (warp < kActWarps) {
    // ------------------------------------------------------------ activation groups
    setmaxnreg_inc<kRegsAct>();
    const int half = warp >> 2;                 // 0 or 1
    const int wq = warp & 3;                    // TMEM lane quarter
    const int row_in_half = wq * 32 + lane;     // TMEM lane = query row of the half
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_off + half * 256;
    const uint32_t t_o = t_s + 128;
    const float c_s = kSoftmax ? p.scale * kLog2e : p.scale;   // score multiplier
    const float* bias_win = reinterpret_cast<const float*>(gbase + C::kBias);
    const bool out32 = aligned32(p.out);
    uint32_t it = 0, tcount = 0, ocount = 0, g = 0;
    while (true) {
      const uint32_t slot = it & 1u;
      bool ok = mbar_wait(bar(C::kItemFull + slot), (it >> 1) & 1u, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) { if (lane == 0) fail(); break; }
      const int2 item = item_slot[slot];
      mbar_arrive(bar(C::kItemEmpty + slot));
      ++it;
      if (item.x < 0) break;
      const ItemInfo in = decode_item<kBand>(item, p);
      const int j_lo = in.lo(half), j_hi = in.hi(half);
      const int nh = j_hi - j_lo;
      const uint32_t g_item = g;  // key-tile counter at this item's first tile
      g += in.je - in.jb;
      const int r = in.blk * kItemRows + half * kHalfRows + row_in_half;  // local row
      if (half == 1 && in.blk * kItemRows + kHalfRows >= in.Lq) continue;
      const bool row_valid = r < in.Lq;
      // visible key columns of this row: [col_lo, col_lim)
      const int col_lo = kBand ? band_key_begin(r, p.window) : 0;
      const int col_lim = kBand ? band_key_end(r, p.causal, p.window, in.Lkv)
                                : (p.causal ? min(in.Lkv, r + 1) : in.Lkv);
      const bool has_bias = p.bias_table != nullptr;
      // dense bias row of this query: one value per key (none past the sample)
      const float* drow = nullptr;
      if (kDense && row_valid)
        drow = p.bias_dense + p.bias_off[in.b] +
               (static_cast<long long>(in.head) * in.Lq + r) * in.Lkv;
      float m = -INFINITY;  // running max (log2 units), possibly stale
      float l = 0.0f;       // running sum relative to m
      bool abort_now = false;
      // dense bias: the row segment of key tile j is pulled into L2 one tile
      // ahead (4 lines of 32 values; only columns the row sees)
      auto prefetch_dense = [&](int jt) {
        if (kDense && drow != nullptr && jt < j_hi) {
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int c = jt * kKvRows + 32 * k4;
            if (c < col_lim) prefetch_l2(drow + c);
          }
        }
      };
      prefetch_dense(j_lo);
      for (int j = j_lo; j < j_hi; ++j) {
        const uint32_t gj = g_item + (j - in.jb);
        prefetch_dense(j + 1);
        // softmax with a dense bias: the row's 128 values of this key tile (times
        // log2e; 0 where the row does not see the key) are requested before the
        // score wait, so that one load latency overlaps the products instead of
        // one per 32-column chunk
        float dz[(kDense && kSoftmax) ? kKvRows : 1];
        if constexpr (kDense && kSoftmax) {
          // 16-byte loads from the aligned position at or before the tile's first
          // column (a load instruction costs one L1 wavefront per row either way,
          // so four columns per load cut them fourfold), then each lane shifts
          // its window by its own misalignment sh; a 16-byte group not wholly
          // inside the row's visible columns is read element by element
          const int cb = j * kKvRows;
          const int lo = kBand ? max(col_lo, 0) : 0;
          const int sh = drow != nullptr ? static_cast<int>((reinterpret_cast<uintptr_t>(drow + cb) >> 2) & 3u) : 0;
          float w[kKvRows + 4];
#pragma unroll
          for (int q = 0; q < kKvRows / 4 + 1; ++q) {
            const int ca = cb + 4 * q - sh;  // column of the group's first element
            if (drow != nullptr && ca >= lo && ca + 4 <= col_lim) {
              const float4 t = __ldg(reinterpret_cast<const float4*>(drow + ca));
              w[4 * q] = t.x;
              w[4 * q + 1] = t.y;
              w[4 * q + 2] = t.z;
              w[4 * q + 3] = t.w;
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int c = ca + e;
                w[4 * q + e] = (drow != nullptr && c >= lo && c < col_lim) ? __ldg(drow + c) : 0.0f;
              }
            }
          }
#pragma unroll
          for (int i = 0; i < kKvRows; ++i) {
            const float t01 = (sh & 1) ? w[i + 1] : w[i];
            const float t23 = (sh & 1) ? w[i + 3] : w[i + 2];
            dz[i] = ((sh & 2) ? t23 : t01) * kLog2e;
          }
        }
        bool okw = mbar_wait(bar(C::kSFull + half), tcount & 1u, abort_flag);
        // the value-tile stage also carries this tile's bias window
        if (has_bias)
          okw = okw && mbar_wait(bar(C::kVFull + gj % C::kStages), (gj / C::kStages) & 1u, abort_flag);
        okw = __all_sync(0xffffffffu, okw);
        if (!okw) { if (lane == 0) fail(); abort_now = true; break; }
        ++tcount;
        tc_fence_after();
        const int c0 = j * kKvRows;
        const bool need_mask = (kBand && c0 < col_lo) || (c0 + kKvRows > col_lim);
        // Scores need only the scale when no row of the warp needs a mask, there
        // is no bias and the scale is positive (the raw maximum times the scale is
        // then the scaled maximum).  Decided per warp: the tcgen05.ld below is
        // .sync.aligned, so the lanes of a warp must not split between the two paths.
        const bool plain =
            !has_bias && !kDense && c_s > 0.0f && __all_sync(0xffffffffu, !need_mask);
        // bwin[cc] = bias(row, tile column cc) (times log2e for softmax): the
        // window copy shifted by (row + 1) % 2 holds this row's 128 entries in
        // increasing column order from an 8-byte aligned position.
        const int cp = (row_in_half + 1) & 1;
        const float* bwin = bias_win + ((gj % C::kStages) * 2 + half) * C::kBiasBlock +
                            cp * C::kBiasCopy + cp + (kKvRows - 1) - row_in_half;
        // x = score * c_s + bias, with masked entries set to `fill` (pairs of
        // columns per packed fp32 instruction)
        auto load_x = [&](int chunk, float fill, float (&x)[32]) {
          float db[32];  // dense bias of the chunk's visible columns (times log2e for softmax)
          if (kDense) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int c = c0 + chunk * 32 + i;
              db[i] = (drow != nullptr && (!kBand || c >= col_lo) && c < col_lim)
                          ? __ldg(drow + c) * (kSoftmax ? kLog2e : 1.0f)
                          : 0.0f;
            }
          }
          uint32_t sr[32];
          tmem_ld32_nc(t_s + chunk * 32, sr);  // lets the bias loads overlap the TMEM load
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            float4 b4 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (kDense) {
              b4 = make_float4(db[4 * q4], db[4 * q4 + 1], db[4 * q4 + 2], db[4 * q4 + 3]);
            } else if (has_bias) {
              const float2 b01 = *reinterpret_cast<const float2*>(bwin + chunk * 32 + 4 * q4);
              const float2 b23 = *reinterpret_cast<const float2*>(bwin + chunk * 32 + 4 * q4 + 2);
              b4 = make_float4(b01.x, b01.y, b23.x, b23.y);
            }
            const float2 x01 = fma_f32x2(make_float2(__uint_as_float(sr[4 * q4]), __uint_as_float(sr[4 * q4 + 1])),
                                         make_float2(c_s, c_s), make_float2(b4.x, b4.y));
            const float2 x23 = fma_f32x2(make_float2(__uint_as_float(sr[4 * q4 + 2]), __uint_as_float(sr[4 * q4 + 3])),
                                         make_float2(c_s, c_s), make_float2(b4.z, b4.w));
            x[4 * q4] = x01.x;
            x[4 * q4 + 1] = x01.y;
            x[4 * q4 + 2] = x23.x;
            x[4 * q4 + 3] = x23.y;
          }
          if (need_mask) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int c = c0 + chunk * 32 + i;
              if ((kBand && c < col_lo) || c >= col_lim) x[i] = fill;
            }
          }
        };
        if (kSoftmax) {
          // The row's 128 scores stay in registers: TMEM and the bias window are
          // read once.  Plain tiles keep raw scores (scale folded into the exponent).
          float xs[kKvRows];
          float mt = -INFINITY;
          if (!kDense) {
            // One TMEM load of all 128 columns (one wait), scale and bias in
            // place, then the row maximum with three-input max instructions in
            // four independent chains.
            uint32_t sr[kKvRows];
            tmem_ld128(t_s, sr);
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (plain) {
#pragma unroll
              for (int i = 0; i < kKvRows; ++i) xs[i] = __uint_as_float(sr[i]);
#pragma unroll
              for (int i = 0; i < kKvRows; i += 2)
                m4[(i >> 1) & 3] = fmax3(m4[(i >> 1) & 3], xs[i], xs[i + 1]);
              mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * c_s;
            } else {
              const float2 cc = make_float2(c_s, c_s);
#pragma unroll
              for (int q4 = 0; q4 < kKvRows / 4; ++q4) {
                float2 b01 = make_float2(0.f, 0.f), b23 = make_float2(0.f, 0.f);
                if (has_bias) {
                  b01 = *reinterpret_cast<const float2*>(bwin + 4 * q4);
                  b23 = *reinterpret_cast<const float2*>(bwin + 4 * q4 + 2);
                }
                const float2 x01 = fma_f32x2(make_float2(__uint_as_float(sr[4 * q4]), __uint_as_float(sr[4 * q4 + 1])), cc, b01);
                const float2 x23 = fma_f32x2(make_float2(__uint_as_float(sr[4 * q4 + 2]), __uint_as_float(sr[4 * q4 + 3])), cc, b23);
                xs[4 * q4] = x01.x;
                xs[4 * q4 + 1] = x01.y;
                xs[4 * q4 + 2] = x23.x;
                xs[4 * q4 + 3] = x23.y;
              }
              if (need_mask) {
#pragma unroll
                for (int i = 0; i < kKvRows; ++i) {
                  const int c = c0 + i;
                  if ((kBand && c < col_lo) || c >= col_lim) xs[i] = -INFINITY;
                }
              }
#pragma unroll
              for (int i = 0; i < kKvRows; i += 2)
                m4[(i >> 1) & 3] = fmax3(m4[(i >> 1) & 3], xs[i], xs[i + 1]);
              mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            }
          } else {
            // dense bias: scores plus the values requested before the wait
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int chunk = 0; chunk < 4; ++chunk) {
              uint32_t sr[32];
              tmem_ld32(t_s + chunk * 32, sr);
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const int c = c0 + chunk * 32 + i;
                float x = fmaf(__uint_as_float(sr[i]), c_s, dz[chunk * 32 + i]);
                if (need_mask && ((kBand && c < col_lo) || c >= col_lim)) x = -INFINITY;
                xs[chunk * 32 + i] = x;
                m4[i & 3] = fmaxf(m4[i & 3], x);
              }
            }
            mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
          }
          const float m_new = fmaxf(m, mt);
          bool rescale = false;
          float factor = 1.0f;
          if (m == -INFINITY) {
            m = m_new;
          } else if (m_new - m > kRescaleThreshold) {
            factor = ex2_approx(m - m_new);
            l *= factor;
            m = m_new;
            rescale = true;
          }
          if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
            for (int chunk = 0; chunk < D / 32; ++chunk) {
              uint32_t o[32];
              tmem_ld32(t_o + chunk * 32, o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * factor);
              tmem_st32(t_o + chunk * 32, o);
            }
          }
          const float m_ref = (m == -INFINITY) ? 0.0f : m;
          // exponent = xs * xm - m_ref (plain: raw scores times the scale)
          const float xm = plain ? c_s : 1.0f;
          float2 l2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
          for (int chunk = 0; chunk < 4; ++chunk) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 e = fma_f32x2(make_float2(xs[chunk * 32 + 2 * i], xs[chunk * 32 + 2 * i + 1]),
                                         make_float2(xm, xm), make_float2(-m_ref, -m_ref));
              const float2 pv = make_float2(ex2_approx(e.x), ex2_approx(e.y));
              l2[i & 1] = add_f32x2(l2[i & 1], pv);
              pk[i] = pack_bf16x2(pv.x, pv.y);
            }
            tmem_st16(t_s + chunk * 32, pk);
          }
          l += (l2[0].x + l2[0].y) + (l2[1].x + l2[1].y);
        } else {
#pragma unroll 1
          for (int chunk = 0; chunk < 4; ++chunk) {
            float x[32];
            load_x(chunk, 0.0f, x);
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float p0 = act_apply(ACT, x[2 * i]);
              const float p1 = act_apply(ACT, x[2 * i + 1]);
              const uint32_t h = pack_bf16x2(p0, p1);
              const float h0 = __uint_as_float(h << 16);
              const float h1 = __uint_as_float(h & 0xFFFF0000u);
              hi[i] = h;
              lo[i] = pack_bf16x2(p0 - h0, p1 - h1);
            }
            tmem_st16(t_s + chunk * 32, hi);
            tmem_st16(t_s + chunk * 32 + 16, lo);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::kPFull + half));
      }
      if (abort_now) break;
      // ---------------------------------------------------------- epilogue
      const float inv_l = kSoftmax ? (l > 0.0f ? 1.0f / l : 0.0f) : 1.0f;
      __nv_bfloat16* orow = p.out + (static_cast<long long>(in.q0 + r) * p.H + in.head) * D;
      if (nh > 0) {
        bool okw = mbar_wait(bar(C::kODone + half), ocount & 1u, abort_flag);
        okw = __all_sync(0xffffffffu, okw);
        if (!okw) { if (lane == 0) fail(); break; }
        ++ocount;
        tc_fence_after();
#pragma unroll 1
        for (int chunk = 0; chunk < D / 64; ++chunk) {
          uint32_t o[64];
          tmem_ld64(t_o + chunk * 64, o);
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
          if (row_valid) store_words(orow + chunk * 64, pk, out32);
        }
        tc_fence_before();
      } else if (row_valid) {
        uint4* dst = reinterpret_cast<uint4*>(orow);
        for (int v = 0; v < D / 8; ++v) dst[v] = make_uint4(0, 0, 0, 0);
      }
      if (kSoftmax && row_valid && p.lse != nullptr) {
        const float lse = (l > 0.0f) ? (m * kLn2 + __logf(l)) : -INFINITY;
        p.lse[static_cast<long long>(in.head) * p.Tq + in.q0 + r] = lse;
      }
    }
  } else {
    setmaxnreg_dec<kRegsLow>();  // warps 10-11: no role
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int ACT, bool kBand, bool kDense>
cudaError_t launch_one(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, int grid, cudaStream_t stream) {
  const int smem = FwdCfg<D>::kSmemBytes;
  // The register split (setmaxnreg) hands out exactly the launch's pool of
  // 168 per thread: a build that launched with fewer would leave the
  // activation warps waiting for registers, so refuse to launch it.
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, fwd_kernel<D, ACT, kBand, kDense>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != (2 * kRegsAct + kRegsLow) / 3) return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(fwd_kernel<D, ACT, kBand, kDense>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  fwd_kernel<D, ACT, kBand, kDense><<<grid, kThreads, smem, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

template <int D, bool kBand, bool kDense>
cudaError_t launch_d(const FwdParams& p, int act, const CUtensorMap& tq, const CUtensorMap& tk,
                     const CUtensorMap& tv, int grid, cudaStream_t stream) {
  switch (act) {
    case GDPA_ACT_SOFTMAX:
      return launch_one<D, GDPA_ACT_SOFTMAX, kBand, kDense>(p, tq, tk, tv, grid, stream);
    case GDPA_ACT_SILU:
      return launch_one<D, GDPA_ACT_SILU, kBand, kDense>(p, tq, tk, tv, grid, stream);
    case GDPA_ACT_GELU_TANH:
      return launch_one<D, GDPA_ACT_GELU_TANH, kBand, kDense>(p, tq, tk, tv, grid, stream);
    case GDPA_ACT_GELU_ERF:
      return launch_one<D, GDPA_ACT_GELU_ERF, kBand, kDense>(p, tq, tk, tv, grid, stream);
    default: return launch_one<D, GDPA_ACT_IDENTITY, kBand, kDense>(p, tq, tk, tv, grid, stream);
  }
}

}  // namespace

int fwd_smem_bytes(int d) { return d == 64 ? FwdCfg<64>::kSmemBytes : FwdCfg<128>::kSmemBytes; }

cudaError_t launch_fwd(const FwdParams& p, int act, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, int grid, cudaStream_t stream) {
  const bool band = p.window > 0;
  if (p.bias_dense != nullptr) {
    if (p.d == 64)
      return band ? launch_d<64, true, true>(p, act, tq, tk, tv, grid, stream)
                  : launch_d<64, false, true>(p, act, tq, tk, tv, grid, stream);
    return band ? launch_d<128, true, true>(p, act, tq, tk, tv, grid, stream)
                : launch_d<128, false, true>(p, act, tq, tk, tv, grid, stream);
  }
  if (p.d == 64)
    return band ? launch_d<64, true, false>(p, act, tq, tk, tv, grid, stream)
                : launch_d<64, false, false>(p, act, tq, tk, tv, grid, stream);
  return band ? launch_d<128, true, false>(p, act, tq, tk, tv, grid, stream)
              : launch_d<128, false, false>(p, act, tq, tk, tv, grid, stream);
}

}  // namespace gdpa
