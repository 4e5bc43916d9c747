// MXFP8 forward kernel of jagged softmax attention (JFA), sm_103a.
//
// "GEM Training ..." low-precision paragraph: attention with end-to-end
// MXFP8 block-scaled MMA.  Both products run on the block-scaled tensor
// cores (tcgen05.mma kind::mxf8f6f4.block_scale): E4M3 operands, one E8M0
// scale per 32 elements of the contraction, fp32 accumulation.
//   S = Q K^T   Q, K quantised along channels (scales per 32 of d)
//   O = P V     V quantised along tokens in 32-token blocks aligned to each
//               sample's start; P quantised in registers per 32 keys (with a
//               saturation-free block scale, see e8m0_nosat)
// (gdpa_quantize_mxfp8 produces the Q, K and V operands.)
//
// Structure: the bf16 forward's (persistent CTAs over the cost-sorted work
// list, two 128-row query halves per item, online softmax with lazy O
// rescale), with 96-row key tiles (three 32-token scale blocks) so that the
// scale factors fit in TMEM beside S and O:
//   columns [0,96) S/P of half 0, [128,256) O of half 0,
//           [256,352) S/P of half 1, [384,512) O of half 1,
//   scale columns in the gaps [96,128) and [352,384).
// A scale factor of row r (of A) or column r (of B^T) for the 32-element
// block k of one MMA is byte k of a 32-bit word held in TMEM column
// base + r/32, lane r%32 of every 32-lane quarter.
//
// Warp roles (448 threads):
//   warps 0-3 / 4-7  activation groups of half 0 / half 1: scale, bias,
//                    mask, online softmax, P -> E4M3 codes + block scales
//   warps 8-11       scale group: writes the Q, K and V scale words to TMEM
//   warp  12         producer: tickets, TMA copies of Q/K/V codes, bias windows
//   warp  13         MMA issuer
#include "common.cuh"
#include "mx.cuh"

namespace gdpa {
namespace {

using namespace ptx;
using mx::e4m3x4;
using mx::e8m0_nosat;

constexpr int kThreads = 448;
constexpr int kScaleWarp0 = 8;
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int kD = 128;
constexpr int kTile = 96;        // key rows per tile
constexpr int kStages = 2;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;

// TMEM columns: S/P and O of half h, Q and P scale words of half h, K and
// V scale words of stage s.
__device__ __forceinline__ uint32_t col_s(int h) { return 256u * h; }
__device__ __forceinline__ uint32_t col_o(int h) { return 128u + 256u * h; }
__device__ __forceinline__ uint32_t col_sfq(int h) { return 96u + 8u * h; }
__device__ __forceinline__ uint32_t col_sfp(int h) { return 112u + 8u * h; }
__device__ __forceinline__ uint32_t col_sfk(int s) { return 352u + 8u * s; }
__device__ __forceinline__ uint32_t col_sfv(int s) { return 368u + 8u * s; }

struct Cfg {
  static constexpr int kQHalfBytes = kHalfRows * kD;   // 16 KB of E4M3 codes
  static constexpr int kTileBytes = kTile * kD;        // 12 KB
  static constexpr int kQ0 = 0, kQ1 = kQHalfBytes;
  static constexpr int kKV = 2 * kQHalfBytes;          // K[s] = kKV + s*2*tile, V = K + tile
  // per stage and half: the bias window (kTile + 127 relative positions, in
  // reverse order, times log2e) in two copies shifted by 0 and 1 entries,
  // kBiasCopy floats apart: every query row finds its entries of a key tile
  // 8-byte aligned in one copy, and with this stride the 64-bit loads of a
  // warp hit every bank once
  static constexpr int kBiasCopy = 270;
  static constexpr int kBiasBlock = 2 * kBiasCopy;
  static constexpr int kBias = kKV + kStages * 2 * kTileBytes;
  static constexpr int kSfp = kBias + kStages * 2 * kBiasBlock * 4;  // [half][buf][128] u32 P-scale words
  static constexpr int kBar = kSfp + 2 * 2 * kHalfRows * 4;
  static constexpr int kQFull = 0, kQEmpty = 1;
  static constexpr int kKFull = 2;                      // + s
  static constexpr int kVFull = kKFull + kStages;
  static constexpr int kKEmpty = kVFull + kStages;
  static constexpr int kVEmpty = kKEmpty + kStages;
  static constexpr int kSfkvFull = kVEmpty + kStages;   // K and V scale words in TMEM
  static constexpr int kSfqFull = kSfkvFull + kStages;  // Q scale words in TMEM
  static constexpr int kSFull = kSfqFull + 1;           // + half
  static constexpr int kPFull = kSFull + 2;
  static constexpr int kODone = kPFull + 2;
  static constexpr int kItemFull = kODone + 2;          // + slot
  static constexpr int kItemEmpty = kItemFull + 2;
  static constexpr int kDrain = kItemEmpty + 2;
  static constexpr int kSfpBar = kDrain + 1;            // + half * 2 + buf: P-scale words staged
  static constexpr int kNumBars = kSfpBar + 4;
  static constexpr int kItemSlots = kBar + 8 * kNumBars;
  static constexpr int kTmemSlot = kItemSlots + 16;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kUsed = kAbort + 4;
  static constexpr int kSmemBytes = kUsed + 1024;
};

__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c,
                                         uint32_t d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(a),
               "r"(b), "r"(c), "r"(d)
               : "memory");
}

struct ItemInfo {
  int b, head, blk;
  int q0, k0, Lq, Lkv;
  // Key tiles visited: half h covers [lo_h, hi_h); the item streams their
  // (contiguous) union [jb, je).
  int lo0, hi0, lo1, hi1;
  int jb, je;
  __device__ __forceinline__ int lo(int h) const { return h ? lo1 : lo0; }
  __device__ __forceinline__ int hi(int h) const { return h ? hi1 : hi0; }
  __device__ __forceinline__ bool visits(int h, int j) const { return j >= lo(h) && j < hi(h); }
  __device__ __forceinline__ bool has_half1() const { return hi1 > lo1; }
};

// kBand: a sliding window is set (p.window > 0).
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
    band_key_tiles(r0, min(r.Lq, r0 + kHalfRows), p.causal, p.window, r.Lkv, kTile, &r.lo0,
                   &r.hi0);
    if (r0 + kHalfRows < r.Lq)
      band_key_tiles(r0 + kHalfRows, min(r.Lq, r0 + kItemRows), p.causal, p.window, r.Lkv, kTile,
                     &r.lo1, &r.hi1);
    else
      r.lo1 = r.hi1 = r.hi0;
  } else {
    const int nkv = (r.Lkv + kTile - 1) / kTile;
    const bool h1 = r0 + kHalfRows < r.Lq;
    r.lo0 = r.lo1 = 0;
    if (!p.causal) {
      r.hi0 = nkv;
      r.hi1 = h1 ? nkv : 0;
    } else {
      r.hi0 = min(nkv, (min(r.Lq, r0 + kHalfRows) + kTile - 1) / kTile);
      r.hi1 = h1 ? min(nkv, (min(r.Lq, r0 + kItemRows) + kTile - 1) / kTile) : 0;
    }
  }
  r.jb = r.lo0;
  r.je = max(r.hi0, r.hi1);
  return r;
}

// kDense: a dense jagged bias (p.bias_dense) instead of the relative-position
// table; each activation thread reads its row's values of the key tile.
template <bool kBand, bool kDense>
__global__ void __launch_bounds__(kThreads, 1)
fwd_mx_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
              const __grid_constant__ CUtensorMap tmap_v, const FwdParams p,
              const uint8_t* __restrict__ q_sc, const uint8_t* __restrict__ k_sc,
              const uint8_t* __restrict__ v_sc, long long v_sc_rows) {
  using C = Cfg;
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
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(C::kKFull + s), 1);
      mbar_init(bar(C::kVFull + s), 1);
      mbar_init(bar(C::kKEmpty + s), 1);
      mbar_init(bar(C::kVEmpty + s), 1);
      mbar_init(bar(C::kSfkvFull + s), 128);
    }
    mbar_init(bar(C::kSfqFull), 128);
    for (int h = 0; h < 2; ++h) {
      mbar_init(bar(C::kSFull + h), 1);
      mbar_init(bar(C::kPFull + h), kHalfRows);
      mbar_init(bar(C::kODone + h), 1);
      mbar_init(bar(C::kItemFull + h), 1);
      mbar_init(bar(C::kItemEmpty + h), 1 + 3 * 128);
    }
    mbar_init(bar(C::kDrain), 1);
    for (int i = 0; i < 4; ++i) mbar_init(bar(C::kSfpBar + i), 4);  // one arrival per warp
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
  const int rel_w = 2 * p.max_rel - 1;
  constexpr int kWin = kHalfRows + kTile - 1;  // relative positions a (half, tile) pair spans

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer (whole warp)
    const int n_items = *p.n_items;
    float* bias_win = reinterpret_cast<float*>(gbase + C::kBias);
    uint32_t it = 0, g = 0, qi = 0;
    uint32_t inflight = 0, last_g[kStages] = {};
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
          tma_load_3d(sbase + (half ? C::kQ1 : C::kQ0), &tmap_q, bar(C::kQFull), 0, in.head,
                      row0 + half * kHalfRows);
        q_inflight = true;
      }
      ++qi;
      const float* brow =
          p.bias_table ? p.bias_table + static_cast<long long>(in.head) * rel_w : nullptr;
      for (int j = in.jb; j < in.je; ++j, ++g) {
        const uint32_t s = g % kStages;
        const uint32_t ph = (g / kStages) & 1u;
        const uint32_t kdst = sbase + C::kKV + s * 2 * C::kTileBytes;
        const int krow = in.k0 + j * kTile;
        w = mbar_wait(bar(C::kKEmpty + s), ph ^ 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { ok = false; if (lane == 0) fail(); break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(C::kKFull + s), C::kTileBytes);
          tma_load_3d(kdst, &tmap_k, bar(C::kKFull + s), 0, in.head, krow);
          inflight |= 1u << s;
          last_g[s] = g;
        }
        w = mbar_wait(bar(C::kVEmpty + s), ph ^ 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { ok = false; if (lane == 0) fail(); break; }
        if (brow != nullptr) {
          // entry e of half h: bias(i - j') with (i - r_h) - (j' - c0) = e - (kTile - 1)
          for (int h = 0; h < 2; ++h) {
            const int w0 = in.blk * kItemRows + h * kHalfRows - j * kTile - (kTile - 1) +
                           p.max_rel - 1;
            float* win = bias_win + (s * 2 + h) * C::kBiasBlock;
            for (int e = lane; e < kWin; e += 32) {
              const float b = __ldg(brow + min(max(w0 + e, 0), rel_w - 1)) * kLog2e;
              win[(kWin - 1) - e] = b;                  // copy 0: entry e at kWin - 1 - e
              win[C::kBiasCopy + kWin - e] = b;         // copy 1: one position later
            }
          }
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(C::kVFull + s), C::kTileBytes);
          tma_load_3d(kdst + C::kTileBytes, &tmap_v, bar(C::kVFull + s), 0, in.head, krow);
        }
      }
    }
    if (lane == 0 && *abort_flag) {
      for (int s = 0; s < kStages; ++s)
        if (inflight & (1u << s)) {
          const uint32_t ph = (last_g[s] / kStages) & 1u;
          mbar_wait(bar(C::kKFull + s), ph, nullptr, 50000000ull);
          mbar_wait(bar(C::kVFull + s), ph, nullptr, 50000000ull);
        }
      if (q_inflight) mbar_wait(bar(C::kQFull), (qi - 1) & 1u, nullptr, 50000000ull);
    }
  } else if (warp >= kScaleWarp0 && warp < kScaleWarp0 + 4) {
    // ------------------------------------------------------------ scale group
    // Lane L = 32q + i of this group writes, in scale column c, the word of
    // row / column i + 32c (every quarter holds the same words).
    const int wq = warp & 3;
    const int i = lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const int H = p.H;
    uint32_t it = 0, g = 0, qi = 0;
    while (true) {
      const uint32_t slot = it & 1u;
      bool w = mbar_wait(bar(C::kItemFull + slot), (it >> 1) & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      const int2 item = item_slot[slot];
      mbar_arrive(bar(C::kItemEmpty + slot));
      ++it;
      if (item.x < 0) break;
      const ItemInfo in = decode_item<kBand>(item, p);
      const int n = in.je - in.jb;
      if (n == 0) continue;
      // Q scale words of both halves: the previous item's score products must be done
      w = mbar_wait(bar(C::kQEmpty), (qi & 1u) ^ 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      ++qi;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t wv[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const long long row = static_cast<long long>(in.q0) + in.blk * kItemRows + h * kHalfRows + i + 32 * c;
          wv[c] = row < p.Tq ? __ldg(reinterpret_cast<const uint32_t*>(q_sc) + row * H + in.head)
                             : 0x7F7F7F7Fu;
        }
        tmem_st4(tmem + lane_off + col_sfq(h), wv[0], wv[1], wv[2], wv[3]);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::kSfqFull));
      const long long vrow0 = static_cast<long long>(in.b) + in.k0 / 32;  // first scale row of the sample
      const int nblk = (in.Lkv + 31) / 32;
      bool abort_now = false;
      for (int j = in.jb; j < in.je; ++j, ++g) {
        const uint32_t s = g % kStages;
        const uint32_t ph = (g / kStages) & 1u;
        // both scale columns of stage s are free once that stage's value products are done
        w = mbar_wait(bar(C::kVEmpty + s), ph ^ 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); abort_now = true; break; }
        uint32_t kw[4], vw[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int n_row = i + 32 * c;  // key row of the tile (c < 3) / channel (V)
          const long long krow = static_cast<long long>(in.k0) + j * kTile + n_row;
          kw[c] = (c < 3 && krow < p.Tkv)
                      ? __ldg(reinterpret_cast<const uint32_t*>(k_sc) + krow * H + in.head)
                      : 0x7F7F7F7Fu;
          uint32_t v = 0;
#pragma unroll
          for (int kb = 0; kb < 3; ++kb) {
            const int blk = 3 * j + kb;
            uint32_t byte = 127u;
            if (blk < nblk && vrow0 + blk < v_sc_rows)
              byte = __ldg(v_sc + ((vrow0 + blk) * H + in.head) * kD + n_row);
            v |= byte << (8 * kb);
          }
          vw[c] = v | (127u << 24);
        }
        tmem_st4(tmem + lane_off + col_sfk(s), kw[0], kw[1], kw[2], kw[3]);
        tmem_st4(tmem + lane_off + col_sfv(s), vw[0], vw[1], vw[2], vw[3]);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::kSfkvFull + s));
      }
      if (abort_now) break;
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t it = 0, g = 0, qi = 0;
      uint32_t tcount[2] = {0, 0};
      bool issued_any = false;
      // descriptors at each operand's first byte; offsets go into the
      // start-address field (see dadd)
      const uint64_t dsc_q = sdesc(sbase + C::kQ0, 0, 1024, kSwizzle128B);
      const uint64_t dsc_kv = sdesc(sbase + C::kKV, 0, 1024, kSwizzle128B);
      auto issue_s = [&](int half, uint32_t stage) {
        const uint64_t qb = dadd(dsc_q, half ? C::kQ1 - C::kQ0 : 0);
        const uint64_t kb = dadd(dsc_kv, stage * 2 * C::kTileBytes);
#pragma unroll
        for (int ks = 0; ks < kD / 32; ++ks) {
          mx::mma_ss(tmem + col_s(half), dadd(qb, ks * 32), dadd(kb, ks * 32), mx::idesc(kTile, false, false, ks),
                    tmem + col_sfq(half), tmem + col_sfk(stage), ks > 0 ? 1u : 0u);
        }
        mma_commit(bar(C::kSFull + half));
        issued_any = true;
      };
      auto issue_pv = [&](int half, uint32_t stage, bool first) {
        const uint64_t vb = dadd(dsc_kv, stage * 2 * C::kTileBytes + C::kTileBytes);
#pragma unroll
        for (int ks = 0; ks < kTile / 32; ++ks) {
          const uint64_t bd = dadd(vb, ks * 4096);
          mx::mma_ts(tmem + col_o(half), tmem + col_s(half) + 8 * ks, bd, mx::idesc(kD, false, true, ks),
                    tmem + col_sfp(half), tmem + col_sfv(stage), (first && ks == 0) ? 0u : 1u);
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
        if (!mbar_wait(bar(C::kSfqFull), qi & 1u, abort_flag)) { fail(); break; }
        ++qi;
        tc_fence_after();
        const int last_s_half = in.visits(1, in.je - 1) ? 1 : 0;
        {
          const uint32_t s = g % kStages;
          const uint32_t ph = (g / kStages) & 1u;
          if (!mbar_wait(bar(C::kKFull + s), ph, abort_flag)) { fail(); break; }
          if (!mbar_wait(bar(C::kSfkvFull + s), ph, abort_flag)) { fail(); break; }
          tc_fence_after();
          if (in.visits(0, in.jb)) issue_s(0, s);
          if (in.visits(1, in.jb)) issue_s(1, s);
          mma_commit(bar(C::kKEmpty + s));
          if (n == 1) mma_commit(bar(C::kQEmpty));
        }
        for (int j = in.jb; j < in.je; ++j) {
          const uint32_t gj = g + (j - in.jb);
          const uint32_t s = gj % kStages;
          const uint32_t s_next = (gj + 1) % kStages;
          const uint32_t ph_next = ((gj + 1) / kStages) & 1u;
          if (!mbar_wait(bar(C::kVFull + s), (gj / kStages) & 1u, abort_flag)) { ok = false; fail(); break; }
          const int last_half_j = in.visits(1, j) ? 1 : 0;
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
            if (in.visits(half, j + 1)) {
              if (!mbar_wait(bar(C::kKFull + s_next), ph_next, abort_flag) ||
                  !mbar_wait(bar(C::kSfkvFull + s_next), ph_next, abort_flag)) { ok = false; fail(); break; }
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
      if (issued_any) {
        mma_commit(bar(C::kDrain));
        mbar_wait(bar(C::kDrain), 0, nullptr, 100000000ull);
      }
    }
  } else {
    // ------------------------------------------------------------ activation groups
    const int half = warp >> 2;
    const int wq = warp & 3;
    const int row_in_half = wq * 32 + lane;
    const bool out32 = aligned32(p.out);
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_off + col_s(half);
    const uint32_t t_o = tmem + lane_off + col_o(half);
    const float c_s = p.scale * kLog2e;
    const float* bias_win = reinterpret_cast<const float*>(gbase + C::kBias);
    uint32_t* sfp_base = reinterpret_cast<uint32_t*>(gbase + C::kSfp) + half * 2 * kHalfRows;
    uint32_t it = 0, tcount = 0, ocount = 0, g = 0, ptile = 0;
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
      const uint32_t g_item = g;
      g += in.je - in.jb;
      const int r = in.blk * kItemRows + half * kHalfRows + row_in_half;
      if (half == 1 && in.blk * kItemRows + kHalfRows >= in.Lq) continue;
      const bool row_valid = r < in.Lq;
      // visible key columns of this row: [col_lo, col_lim)
      const int col_lo = kBand ? band_key_begin(r, p.window) : 0;
      const int col_lim = kBand ? band_key_end(r, p.causal, p.window, in.Lkv)
                                : (p.causal ? min(in.Lkv, r + 1) : in.Lkv);
      const bool has_bias = p.bias_table != nullptr;
      // dense bias row of this query: one value per key
      const float* drow = nullptr;
      if (kDense && row_valid)
        drow = p.bias_dense + p.bias_off[in.b] +
               (static_cast<long long>(in.head) * in.Lq + r) * in.Lkv;
      float m = -INFINITY, l = 0.0f;
      bool abort_now = false;
      for (int j = j_lo; j < j_hi; ++j) {
        const uint32_t gj = g_item + (j - in.jb);
        bool okw = mbar_wait(bar(C::kSFull + half), tcount & 1u, abort_flag);
        if (has_bias)
          okw = okw && mbar_wait(bar(C::kVFull + gj % kStages), (gj / kStages) & 1u, abort_flag);
        okw = __all_sync(0xffffffffu, okw);
        if (!okw) { if (lane == 0) fail(); abort_now = true; break; }
        ++tcount;
        tc_fence_after();
        const int c0 = j * kTile;
        const bool need_mask = (kBand && c0 < col_lo) || (c0 + kTile > col_lim);
        // bwin[cc] = bias(row, tile column cc) * log2e, from the window copy in
        // which this row's entries start 8-byte aligned
        const int cp = (row_in_half + 1) & 1;
        const float* bwin = bias_win + ((gj % kStages) * 2 + half) * C::kBiasBlock +
                            cp * C::kBiasCopy + cp + 127 - row_in_half;
        // x = score * c_s + bias - sub, two columns per packed instruction
        auto load_x = [&](int chunk, float sub, float (&x)[32]) {
          uint32_t sr[32];
          tmem_ld32_nc(t_s + chunk * 32, sr);
#pragma unroll
          for (int q2 = 0; q2 < 16; ++q2) {
            float2 b = make_float2(-sub, -sub);
            if (kDense) {  // the row's value of each visible column
              const int c = c0 + chunk * 32 + 2 * q2;
              if (drow != nullptr && (!kBand || c >= col_lo) && c < col_lim)
                b.x = fmaf(__ldg(drow + c), kLog2e, -sub);
              if (drow != nullptr && (!kBand || c + 1 >= col_lo) && c + 1 < col_lim)
                b.y = fmaf(__ldg(drow + c + 1), kLog2e, -sub);
            } else if (has_bias) {
              const float2 bb = *reinterpret_cast<const float2*>(bwin + chunk * 32 + 2 * q2);
              b = make_float2(bb.x - sub, bb.y - sub);
            }
            const float2 v = fma_f32x2(make_float2(__uint_as_float(sr[2 * q2]), __uint_as_float(sr[2 * q2 + 1])),
                                       make_float2(c_s, c_s), b);
            x[2 * q2] = v.x;
            x[2 * q2 + 1] = v.y;
          }
          if (need_mask) {
#pragma unroll
            for (int q = 0; q < 32; ++q) {
              const int c = c0 + chunk * 32 + q;
              if ((kBand && c < col_lo) || c >= col_lim) x[q] = -INFINITY;
            }
          }
        };
        float mt = -INFINITY;
#pragma unroll 1
        for (int chunk = 0; chunk < kTile / 32; ++chunk) {
          float x[32];
          load_x(chunk, 0.0f, x);
#pragma unroll
          for (int q = 0; q < 32; ++q) mt = fmaxf(mt, x[q]);
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
          for (int chunk = 0; chunk < kD / 32; ++chunk) {
            uint32_t o[32];
            tmem_ld32(t_o + chunk * 32, o);
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * factor);
            tmem_st32(t_o + chunk * 32, o);
          }
        }
        const float m_ref = (m == -INFINITY) ? 0.0f : m;
        uint32_t sfw = 127u << 24;  // byte kb = scale of keys [32kb, 32kb+32) of the tile
#pragma unroll 1
        for (int chunk = 0; chunk < kTile / 32; ++chunk) {
          float x[32];
          load_x(chunk, m_ref, x);
          float amax = 0.0f;
          float2 l2 = make_float2(0.0f, 0.0f);
#pragma unroll
          for (int q = 0; q < 32; q += 2) {
            x[q] = ex2_approx(x[q]);
            x[q + 1] = ex2_approx(x[q + 1]);
            l2 = add_f32x2(l2, make_float2(x[q], x[q + 1]));
            amax = fmaxf(amax, fmaxf(x[q], x[q + 1]));
          }
          l += l2.x + l2.y;
          const int code = e8m0_nosat(amax);
          const float inv = __uint_as_float(static_cast<uint32_t>(254 - code) << 23);
          uint32_t pk[8];
#pragma unroll
          for (int q = 0; q < 8; ++q)
            pk[q] = e4m3x4(x[4 * q] * inv, x[4 * q + 1] * inv, x[4 * q + 2] * inv,
                           x[4 * q + 3] * inv);
          tmem_st8(t_s + chunk * 8, pk);  // E4M3 codes: 4 keys per column
          sfw |= static_cast<uint32_t>(code) << (8 * chunk);
        }
        // P scale words: row r of the half goes to column r/32, lane r%32 of every
        // quarter, so the words are exchanged through shared memory (double
        // buffered: a buffer is rewritten only after every thread has passed the
        // next tile's exchange, i.e. finished reading it).
        const uint32_t pbuf = ptile & 1u;
        uint32_t* words = sfp_base + pbuf * kHalfRows;
        words[row_in_half] = sfw;
        warp_arrive(bar(C::kSfpBar + half * 2 + pbuf), lane);
        okw = mbar_wait(bar(C::kSfpBar + half * 2 + pbuf), (ptile >> 1) & 1u, abort_flag);
        okw = __all_sync(0xffffffffu, okw);
        ++ptile;
        if (!okw) { if (lane == 0) fail(); abort_now = true; break; }
        tmem_st4(tmem + lane_off + col_sfp(half), words[lane], words[32 + lane], words[64 + lane],
                 words[96 + lane]);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::kPFull + half));
      }
      if (abort_now) break;
      const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
      __nv_bfloat16* orow = p.out + (static_cast<long long>(in.q0 + r) * p.H + in.head) * kD;
      if (nh > 0) {
        bool okw = mbar_wait(bar(C::kODone + half), ocount & 1u, abort_flag);
        okw = __all_sync(0xffffffffu, okw);
        if (!okw) { if (lane == 0) fail(); break; }
        ++ocount;
        tc_fence_after();
#pragma unroll 1
        for (int chunk = 0; chunk < kD / 32; ++chunk) {
          uint32_t o[32];
          tmem_ld32(t_o + chunk * 32, o);
          uint32_t pk[16];
#pragma unroll
          for (int q = 0; q < 16; ++q)
            pk[q] = pack_bf16x2(__uint_as_float(o[2 * q]) * inv_l, __uint_as_float(o[2 * q + 1]) * inv_l);
          if (row_valid) store_words(orow + chunk * 32, pk, out32);
        }
        tc_fence_before();
      } else if (row_valid) {
        uint4* dst = reinterpret_cast<uint4*>(orow);
        for (int v = 0; v < kD / 8; ++v) dst[v] = make_uint4(0, 0, 0, 0);
      }
      if (row_valid && p.lse != nullptr) {
        const float lse = (l > 0.0f) ? (m * kLn2 + __logf(l)) : -INFINITY;
        p.lse[static_cast<long long>(in.head) * p.Tq + in.q0 + r] = lse;
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

}  // namespace

int fwd_mx_tile_rows() { return kTile; }

cudaError_t launch_fwd_mx(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const uint8_t* q_sc, const uint8_t* k_sc,
                          const uint8_t* v_sc, long long v_sc_rows, int grid, cudaStream_t s) {
  const bool dense = p.bias_dense != nullptr;
  auto kernel = p.window > 0 ? (dense ? fwd_mx_kernel<true, true> : fwd_mx_kernel<true, false>)
                             : (dense ? fwd_mx_kernel<false, true> : fwd_mx_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  kernel<<<grid, kThreads, Cfg::kSmemBytes, s>>>(tq, tk, tv, p, q_sc, k_sc, v_sc, v_sc_rows);
  return cudaGetLastError();
}

}  // namespace gdpa
