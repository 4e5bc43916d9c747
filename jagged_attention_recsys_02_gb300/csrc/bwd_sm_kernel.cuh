// Backward of jagged softmax attention (JFA) with 128-query tiles, sm_103a.
//
// "GEM Training ..." JFA paragraph (jagged softmax attention with a custom
// bias and efficient backward passes).  The gradients are those of
//   s = scale q.k + bias,  p = softmax_j(s),  o = sum_j p v:
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D)  (D = rowsum(dO * O)),
//   dQ = scale dS K,  dK = scale dS^T Q.
//
// Key/value-major like the general backward kernel: a work item is one
// 128-row key/value block of one (sample, head), the CTA keeps K and V in
// shared memory and streams the sample's queries past them, everything
// transposed so that TMEM lanes are key rows.  This kernel is the softmax
// specialisation with 128-query tiles: every product is a 128 x 128 (x d)
// tile, so a tile takes 40 tcgen05.mma instructions for twice the work that
// 32 instructions do with 64-query tiles.  The instruction count matters on
// this part: an MMA-issuing warp shares its SM sub-partition with activation
// warps (TMEM lane quarters tie each activation warp to one sub-partition),
// and while they compute, the issuing warp gets few issue slots.
//
// TMEM (512 columns): S^T, later P^T as bf16 pairs [0,128); dP^T, later
// dQ^T [128,256); dV [256,256+d); dK [384,384+d).
//
// Per tile t, on the tensor pipe (one issuing thread, in this order):
//   P(t) ready   -> dV(t) += P^T dO,  S(t+1) = K Q(t+1)^T
//   dS(t) ready  -> dQ^T(t) = K^T dS^T (into the dP columns),  dK(t) += dS^T Q
//   dQ^T read    -> dP(t+1) = V dO(t+1)^T  (the read overlaps dK(t))
// The dQ group reads the whole dQ^T tile into registers (128 per thread, from
// a register reallocation between warpgroups) so the dP columns free up at
// once, then adds it into the fp32 dQ accumulator with bulk tensor
// reduce-adds: each warp stages its own 32 channels of 16 queries in one of
// three small shared buffers and issues its own reduce, so the four warps
// never wait for each other.
// The activation warps run two phases per tile: P from S (stored back into
// TMEM for the dV product, kept in registers as bf16), then dS from dP
// (stored to shared memory for the dK and dQ products).
//
// Warp roles (512 threads = four warpgroups, one CTA per SM, persistent over
// the cost-sorted work list): warps 0-3 and 4-7 activation (query columns
// [0,64) and [64,128) of a tile), warps 8-11 dQ group (dQ^T drain; dK/dV
// epilogue), warp 12 producer (TMA K/V, Q, dO; lse, D and bias values), warp
// 13 MMA issuer, warps 14-15 idle.  Registers: 128 per thread at launch; the
// dQ group rises to 152 and the last warpgroup drops to 104 (4 x 32 x (128 +
// 128 + 152 + 104) = 65536, the whole register file).
#pragma once
#include <type_traits>

#include "common.cuh"

namespace gdpa {
namespace {

using namespace ptx;

constexpr int kThreads = 512;
constexpr int kDqChunk = kBwdSmDqRows;  // queries per dQ reduce box
constexpr int kRegsDq = 152;       // dQ warpgroup (the activation warpgroups keep 128)
constexpr int kRegsLow = 104;      // producer / MMA warpgroup
static_assert(2 * 128 + kRegsDq + kRegsLow == 4 * 128, "register split must keep the launch total");
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int kActWarps = 8;
constexpr int kQRows = kBwdSmQRows;  // 128 queries per tile
constexpr int kKRows = kBwdKvRows;   // 128 keys per item
constexpr float kLog2e = 1.4426950408889634f;
static_assert(kQRows == kKRows, "causal tile skipping assumes square tiles");

template <int D, bool kAug>
struct SmCfg {
  static constexpr int kKvTileBytes = kKRows * D * 2;     // K or V block
  static constexpr int kQTileBytes = kQRows * D * 2;      // Q or dO tile
  static constexpr int kAtom = 128 * 128;                 // one 64-column swizzled atom of 128 rows
  static constexpr int kDsBytes = kKRows * kQRows * 2;    // dS^T tile
  static constexpr int kQStages = 2;
  static constexpr int kK = 0;
  static constexpr int kV = kKvTileBytes;
  static constexpr int kQ = 2 * kKvTileBytes;                   // + s * kQTileBytes
  static constexpr int kO = kQ + kQStages * kQTileBytes;        // dO: one stage
  static constexpr int kDs = kO + kQTileBytes;                  // [query atom][key row][64 queries]
  // per Q stage: without the extra product step (below) -lse*log2e [128] and
  // -D [128]; then the bias window (255 entries, times log2e) in two copies
  // shifted by 0 and 1 entries, kBiasCopy floats apart (every key row finds
  // its 64 entries 8-byte aligned in one copy, and with this stride the
  // 64-bit loads of a warp hit every bank once)
  static constexpr int kBiasCopy = 270;
  static constexpr int kWinOff = kAug ? 0 : 2 * kQRows;                // floats
  static constexpr int kStatFloats = kWinOff + 2 * kBiasCopy + 4;      // (16-byte multiple)
  static constexpr int kStats = kDs + kDsBytes;
  // kAug: an extra K = 16 step of the score and dP products, per Q stage: row i holds
  // (a_hi, a_lo, d_hi, d_lo, 0, ...) in bf16, with a = -lse * log2e / c and
  // d = -D split into two bf16 terms (canonical K-major layout without
  // swizzle: core matrices of 8 rows x 16 bytes, the two k halves 128 bytes
  // apart, row groups 256 bytes apart).  Two selector operands, whose rows are
  // (1, 1, 0, ...) and (0, 0, 1, 1, 0, ...), pick a or d: the products come
  // out of TMEM as S^T - lse log2e / c and dP^T - D.
  // Taken with a relative-position table, whose window loads already fill the
  // activation's shared-memory reads (without one, the extra tensor work
  // costs more than the lse and D loads it saves).
  static constexpr int kSel = kStats + kQStages * kStatFloats * 4;     // 2 x 256 bytes
  static constexpr int kAugBytes = kQRows * 32;
  static constexpr int kAugRows = kSel + (kAug ? 512 : 0);              // + s * kAugBytes
  static constexpr int kDqStage = kAugRows + (kAug ? kQStages * kAugBytes : 0);  // per-warp buffers
  // bias-table gradient: per tile, dS summed along its 255 diagonals (two
  // buffers of 256 floats, then {first diagonal, head})
  static constexpr int kDbBuf = 256 * 4 + 16;
  static constexpr int kDqWarpBufs = kAug ? 2 : 3;         // per warp: [16 queries][32 channels]
  static constexpr int kDb = kDqStage + 4 * kDqWarpBufs * kDqChunk * 32 * 4;
  static constexpr int kBar = kDb + 2 * kDbBuf;
  static constexpr int kKvFull = 0, kKvEmpty = 1;
  static constexpr int kQFull = 2;                    // + stage
  static constexpr int kQEmpty = kQFull + kQStages;   // + stage
  static constexpr int kOFull = kQEmpty + kQStages;
  static constexpr int kOEmpty = kOFull + 1;
  static constexpr int kSFull = kOEmpty + 1;
  static constexpr int kPFull = kSFull + 1;
  static constexpr int kDpFull = kPFull + 1;
  static constexpr int kDsFull = kDpFull + 1;
  static constexpr int kDqFull = kDsFull + 1;
  static constexpr int kDqEmpty = kDqFull + 1;
  static constexpr int kDkvFull = kDqEmpty + 1;
  static constexpr int kDkvEmpty = kDkvFull + 1;
  static constexpr int kItemFull = kDkvEmpty + 1;     // + slot
  static constexpr int kItemEmpty = kItemFull + 2;
  static constexpr int kDrain = kItemEmpty + 2;
  static constexpr int kDbAcc = kDrain + 1;     // + buffer: the activation warps added a tile
  static constexpr int kDbFree = kDbAcc + 2;    // + buffer: flushed to the table and zeroed
  static constexpr int kNumBars = kDbFree + 2;
  static constexpr int kItemSlots = kBar + 8 * kNumBars;
  static constexpr int kTmemSlot = kItemSlots + 16;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kGroupOk = kAbort + 4;   // int[4]: dQ-group vote on a wait's result
  static constexpr int kUsed = kGroupOk + 16;
  static constexpr int kSmemBytes = kUsed + 1024;
};

constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384;

// Score multiplier c = scale * log2e of the exponent, kept away from 0: the
// extra product step carries -lse log2e / c, and a scale of 0 (scores that do
// not count) then leaves S * c at 1e-30 * S, which rounds away against lse.
__device__ __forceinline__ float score_mul(float scale) {
  const float c = scale * 1.4426950408889634f;
  return fabsf(c) < 1e-30f ? (c < 0.0f ? -1e-30f : 1e-30f) : c;
}

struct SmItem {
  int b, head, kb;
  int q0, k0, Lq, Lkv;
  int qt0;  // first query tile (128 rows) visited
  int nq;   // number of query tiles visited
};

// kBand: a sliding window is set; without one the query range is the
// plain causal / full one.
template <bool kBand>
__device__ __forceinline__ SmItem decode_sm(int2 it, const BwdParams& p) {
  SmItem r;
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
  if (kBand) {
    const int kb0 = r.kb * kKRows;
    const int qb = band_query_begin(kb0, p.causal, p.window);
    const int qe = band_query_end(min(r.Lkv, kb0 + kKRows) - 1, p.window, r.Lq);
    r.qt0 = qb / kQRows;
    r.nq = (qe + kQRows - 1) / kQRows - r.qt0;  // 0 when qe == qb == 0 (no query rows)
  } else {
    r.qt0 = p.causal ? r.kb : 0;  // queries before the block's first key see none of it
    const int rows = r.Lq - r.qt0 * kQRows;
    r.nq = rows > 0 ? (rows + kQRows - 1) / kQRows : 0;
  }
  return r;
}

// kDense: a dense jagged bias (p.bias_dense) instead of the relative-position
// table, read from global memory by the activation warps (the warp's lanes
// are consecutive keys, so each load is one coalesced 128-byte row segment);
// with p.dbias its gradient goes back the same way, one reduction per pair.
// kRope: dK (here) and dQ (in the accumulator's conversion) go back through
// the rotary embedding.
template <int D, bool kBand, bool kDBias, bool kDense, bool kRope, bool kAug>
__global__ void __launch_bounds__(kThreads, 1)
bwd_sm_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
              const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
              const __grid_constant__ CUtensorMap tmap_dq, const BwdParams p) {
  using C = SmCfg<D, kAug>;
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
    for (int s = 0; s < C::kQStages; ++s) {
      mbar_init(bar(C::kQFull + s), 1);
      mbar_init(bar(C::kQEmpty + s), 1);
    }
    mbar_init(bar(C::kOFull), 1);
    mbar_init(bar(C::kOEmpty), 1);
    mbar_init(bar(C::kSFull), 1);
    // consumer-side barriers count warps (one arrival per warp, see warp_arrive)
    mbar_init(bar(C::kPFull), kActWarps);
    mbar_init(bar(C::kDpFull), 1);
    mbar_init(bar(C::kDsFull), kActWarps);
    mbar_init(bar(C::kDqFull), 1);
    mbar_init(bar(C::kDqEmpty), 4);
    mbar_init(bar(C::kDkvFull), 1);
    mbar_init(bar(C::kDkvEmpty), 4);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::kItemFull + s), 1);
      mbar_init(bar(C::kItemEmpty + s), 1 + kActWarps + 4 + (kTableGrad ? 1 : 0));
    }
    mbar_init(bar(C::kDrain), 1);
    for (int u = 0; u < 2; ++u) {
      mbar_init(bar(C::kDbAcc + u), kActWarps);
      mbar_init(bar(C::kDbFree + u), 1);
    }
    fence_mbar_init();
  }
  if (kTableGrad)
    for (int i = threadIdx.x; i < 2 * C::kDbBuf / 4; i += kThreads)
      reinterpret_cast<float*>(gbase + C::kDb)[i] = 0.0f;
  // selectors and the zero columns of the extra product step (written once;
  // the producer rewrites only the first 8 bytes of each row per tile)
  if (kAug)
  for (int i = threadIdx.x; i < (512 + C::kQStages * C::kAugBytes) / 4; i += kThreads) {
    uint32_t v = 0;
    if (i < 128) {  // selector words: 8 rows x 16 bytes per k half
      const int sel = i / 64, kh = (i / 32) & 1, word = i & 3;  // 4 words per 16-byte row
      if (kh == 0 && word == sel) v = 0x3F803F80u;            // bf16 pair (1, 1)
    }
    reinterpret_cast<uint32_t*>(gbase + C::kSel)[i] = v;
  }
  fence_proxy_async_smem();
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
    setmaxnreg_dec<kRegsLow>();
    const int n_items = *p.n_items;
    uint32_t it = 0, g = 0, kvi = 0, oi = 0;
    bool kv_inflight = false, o_inflight = false;
    uint32_t q_inflight = 0, last_g[C::kQStages] = {};
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
      const SmItem in = decode_sm<kBand>(item, p);
      if (in.nq == 0) continue;
      w = mbar_wait(bar(C::kKvEmpty), (kvi & 1u) ^ 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      ++kvi;
      const int krow = in.k0 + in.kb * kKRows;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(C::kKvFull), 2 * C::kKvTileBytes);
        for (int x = 0; x < D; x += 64) {
          tma_load_3d(sbase + C::kK + (x / 64) * C::kAtom, &tmap_k, bar(C::kKvFull), x, in.head, krow);
          tma_load_3d(sbase + C::kV + (x / 64) * C::kAtom, &tmap_v, bar(C::kKvFull), x, in.head, krow);
        }
        kv_inflight = true;
      }
      // Per-lane values of one query tile, fetched one tile ahead: lse*log2e
      // and D for columns lane + 32k, bias-window entries lane + 32k.
      const int rel_w = 2 * p.max_rel - 1;
      const float inv_c = 1.0f / score_mul(p.scale);
      const float* brow =
          p.bias_table ? p.bias_table + static_cast<long long>(in.head) * rel_w : nullptr;
      constexpr int kWin = kQRows + kKRows - 1;  // 255 relative positions
      auto fetch = [&](int t, float (&v)[16]) {
        const int qloc = (in.qt0 + t) * kQRows;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int ql = qloc + lane + 32 * k;
          float l2 = 0.0f, dd = 0.0f;
          if (ql < in.Lq) {
            const long long gi = static_cast<long long>(in.head) * p.Tq + in.q0 + ql;
            l2 = -__ldg(p.lse + gi) * kLog2e;  // stored negated: added, not subtracted
            dd = -__ldg(p.delta + gi);
          }
          v[2 * k] = l2;
          v[2 * k + 1] = dd;
        }
        // bias(i - j) for query column c and key row jj of the tile is window
        // entry c - jj + 127
        const int w0 = qloc - in.kb * kKRows - (kKRows - 1) + p.max_rel - 1;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int e = lane + 32 * k;
          v[8 + k] = (brow != nullptr && e < kWin)
                         ? __ldg(brow + min(max(w0 + e, 0), rel_w - 1)) * kLog2e
                         : 0.0f;
        }
      };
      float cur[16];
      fetch(0, cur);
      for (int t = 0; t < in.nq; ++t, ++g) {
        const uint32_t s = g % C::kQStages;
        const uint32_t ph = (g / C::kQStages) & 1u;
        const int qloc = (in.qt0 + t) * kQRows;
        w = mbar_wait(bar(C::kQEmpty + s), ph ^ 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { ok = false; if (lane == 0) fail(); break; }
        float* st = stats + s * C::kStatFloats;
        if (!kAug) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            st[lane + 32 * k] = cur[2 * k];
            st[kQRows + lane + 32 * k] = cur[2 * k + 1];
          }
        } else {
        // extra product step: a = -lse log2e / c and d = -D as bf16 (hi, lo)
        // pairs in the first 8 bytes of row i (queries past the sample get 0)
        uint8_t* aug = gbase + C::kAugRows + s * C::kAugBytes;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = lane + 32 * k;
          // finite values only: the selectors' zeros multiply them too (a row
          // whose lse is -inf has no probability mass: a = 0 gives it P = 0
          // wherever its bias is -inf)
          float a = cur[2 * k] * inv_c, dd = cur[2 * k + 1];
          a = (fabsf(a) <= 1e38f) ? a : 0.0f;
          dd = (fabsf(dd) <= 1e38f) ? dd : 0.0f;
          const uint32_t ah = pack_bf16x2(a, 0.0f) & 0xFFFFu;
          const uint32_t dh = pack_bf16x2(dd, 0.0f) & 0xFFFFu;
          const float al = a - __uint_as_float(ah << 16), dl = dd - __uint_as_float(dh << 16);
          *reinterpret_cast<uint2*>(aug + (i >> 3) * 256 + (i & 7) * 16) =
              make_uint2(ah | (pack_bf16x2(al, 0.0f) << 16), dh | (pack_bf16x2(dl, 0.0f) << 16));
        }
        fence_proxy_async_smem();
        }
        if (brow != nullptr) {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (lane + 32 * k < kWin) {
#pragma unroll
              for (int cp = 0; cp < 2; ++cp)  // copy cp holds entry e at position e + cp
                st[C::kWinOff + cp * C::kBiasCopy + cp + lane + 32 * k] = cur[8 + k];
            }
        }
        float nxt[16];
        if (t + 1 < in.nq) {
          fetch(t + 1, nxt);
        } else {
#pragma unroll
          for (int k = 0; k < 16; ++k) nxt[k] = 0.0f;
        }
        __syncwarp();
        if (lane == 0) {
          const uint32_t qa = sbase + C::kQ + s * C::kQTileBytes;
          mbar_arrive_expect_tx(bar(C::kQFull + s), C::kQTileBytes);
          for (int x = 0; x < D; x += 64)
            tma_load_3d(qa + (x / 64) * C::kAtom, &tmap_q, bar(C::kQFull + s), x, in.head,
                        in.q0 + qloc);
          q_inflight |= 1u << s;
          last_g[s] = g;
        }
        // dO of this tile: its single buffer frees once dV of the previous tile is done
        w = mbar_wait(bar(C::kOEmpty), (oi & 1u) ^ 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { ok = false; if (lane == 0) fail(); break; }
        ++oi;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(C::kOFull), C::kQTileBytes);
          for (int x = 0; x < D; x += 64)
            tma_load_3d(sbase + C::kO + (x / 64) * C::kAtom, &tmap_do, bar(C::kOFull), x, in.head,
                        in.q0 + qloc);
          o_inflight = true;
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) cur[k] = nxt[k];
      }
    }
    if (lane == 0 && *abort_flag) {
      // let every copy this warp started land before the CTA exits
      for (int s = 0; s < C::kQStages; ++s)
        if (q_inflight & (1u << s))
          mbar_wait(bar(C::kQFull + s), (last_g[s] / C::kQStages) & 1u, nullptr, 50000000ull);
      if (o_inflight) mbar_wait(bar(C::kOFull), (oi - 1) & 1u, nullptr, 50000000ull);
      if (kv_inflight) mbar_wait(bar(C::kKvFull), (kvi - 1) & 1u, nullptr, 50000000ull);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    setmaxnreg_dec<kRegsLow>();
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16(128, kQRows, true, false, false);  // S^T, dP^T
      constexpr uint32_t idesc_acc = idesc_f16(128, D, true, false, true);      // dV, dK
      constexpr uint32_t idesc_dq = idesc_f16(128, kQRows, true, true, true);   // dQ^T
      // Descriptors at each operand's first byte; k-steps and stages are added
      // to the start-address field (see dadd).
      const uint64_t dsc_k = sdesc(sbase + C::kK, 0, 1024, kSwizzle128B);   // A of S^T (K-major)
      const uint64_t dsc_v = sdesc(sbase + C::kV, 0, 1024, kSwizzle128B);   // A of dP^T
      // K as the MN-major A of dQ^T; d = 64: the second 64-row half of A
      // repeats the first (LBO 0) and its output lanes 64..127 are ignored.
      const uint64_t dsc_kt = sdesc(sbase + C::kK, D == 128 ? C::kAtom : 0, 1024, kSwizzle128B);
      const uint64_t dsc_q = sdesc(sbase + C::kQ, 0, 1024, kSwizzle128B);   // B of S^T (K-major)
      const uint64_t dsc_qmn = sdesc(sbase + C::kQ, C::kAtom, 1024, kSwizzle128B);  // B of dK (MN-major)
      const uint64_t dsc_o = sdesc(sbase + C::kO, 0, 1024, kSwizzle128B);   // B of dP^T
      const uint64_t dsc_omn = sdesc(sbase + C::kO, C::kAtom, 1024, kSwizzle128B);  // B of dV
      const uint64_t dsc_ds = sdesc(sbase + C::kDs, 0, 1024, kSwizzle128B);  // A of dK (K-major)
      const uint64_t dsc_dsmn = sdesc(sbase + C::kDs, C::kAtom, 1024, kSwizzle128B);  // B of dQ^T (MN-major)
      // extra K = 16 step (no swizzle: k halves 128 bytes apart, row groups 256
      // apart; the selectors repeat one 8-row group, stride 0)
      const uint64_t dsc_aug = sdesc(sbase + C::kAugRows, 128, 256, 0);      // B
      const uint64_t dsc_sel_a = sdesc(sbase + C::kSel, 128, 0, 0);          // A: picks a
      const uint64_t dsc_sel_d = sdesc(sbase + C::kSel + 256, 128, 0, 0);    // A: picks d
      uint32_t it = 0, g = 0, kvi = 0, oc = 0, pc = 0, qe = 0, dkvc = 0;
      bool dq_pending = false, issued_any = false;
      bool ok = true;
      auto issue_s = [&](uint32_t s) {  // S^T = K Q^T (kAug: - lse log2e / c)
        const uint64_t qb = dadd(dsc_q, s * C::kQTileBytes);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks / 4) * C::kAtom + (ks % 4) * 32;
          mma_f16_ss(tmem + kColS, dadd(dsc_k, off), dadd(qb, off), idesc_s, ks > 0 ? 1u : 0u);
        }
        if (kAug) mma_f16_ss(tmem + kColS, dsc_sel_a, dadd(dsc_aug, s * C::kAugBytes), idesc_s, 1u);
        mma_commit(bar(C::kSFull));
        issued_any = true;
      };
      // dP^T = V dO^T (kAug: - D of the tile in Q stage s) into the dP columns,
      // once dO has landed and the dQ group has read the previous dQ^T out of
      // the same columns.
      auto issue_dp = [&](uint32_t s) -> bool {
        if (!mbar_wait(bar(C::kOFull), oc & 1u, abort_flag)) return false;
        ++oc;
        if (dq_pending) {
          if (!mbar_wait(bar(C::kDqEmpty), qe & 1u, abort_flag)) return false;
          ++qe;
          dq_pending = false;
        }
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks / 4) * C::kAtom + (ks % 4) * 32;
          mma_f16_ss(tmem + kColDP, dadd(dsc_v, off), dadd(dsc_o, off), idesc_s, ks > 0 ? 1u : 0u);
        }
        if (kAug) mma_f16_ss(tmem + kColDP, dsc_sel_d, dadd(dsc_aug, s * C::kAugBytes), idesc_s, 1u);
        mma_commit(bar(C::kDpFull));
        return true;
      };
      while (ok) {
        const uint32_t slot = it & 1u;
        if (!mbar_wait(bar(C::kItemFull + slot), (it >> 1) & 1u, abort_flag)) { fail(); break; }
        const int2 item = item_slot[slot];
        mbar_arrive(bar(C::kItemEmpty + slot));
        ++it;
        if (item.x < 0) break;
        const SmItem in = decode_sm<kBand>(item, p);
        if (in.nq == 0) continue;
        if (!mbar_wait(bar(C::kKvFull), kvi & 1u, abort_flag)) { fail(); break; }
        ++kvi;
        {
          const uint32_t s0 = g % C::kQStages;
          if (!mbar_wait(bar(C::kQFull + s0), (g / C::kQStages) & 1u, abort_flag)) { fail(); break; }
          tc_fence_after();
          issue_s(s0);
          if (!issue_dp(s0)) { fail(); break; }
        }
        for (int t = 0; t < in.nq; ++t) {
          const uint32_t gt = g + t;
          const uint32_t s = gt % C::kQStages;
          if (!mbar_wait(bar(C::kPFull), pc & 1u, abort_flag)) { ok = false; fail(); break; }
          tc_fence_after();
          if (t == 0) {
            // the previous item's dK/dV must have been read out before we overwrite them
            if (!mbar_wait(bar(C::kDkvEmpty), (dkvc & 1u) ^ 1u, abort_flag)) { ok = false; fail(); break; }
            tc_fence_after();
          }
          // dV += P^T dO   (A = P^T in TMEM, B = dO MN-major); queries ks*16..+15
          // of the tile sit in columns 64*(ks/4) + 8*(ks%4) as bf16 pairs.
#pragma unroll
          for (int ks = 0; ks < kQRows / 16; ++ks) {
            const uint32_t pcol = tmem + kColS + 64 * (ks / 4) + 8 * (ks % 4);
            mma_f16_ts(tmem + kColDV, pcol, dadd(dsc_omn, ks * 2048), idesc_acc,
                       (t == 0 && ks == 0) ? 0u : 1u);
          }
          mma_commit(bar(C::kOEmpty));
          // S(t+1) reuses the S columns: it follows dV(t) on the pipe
          if (t + 1 < in.nq) {
            const uint32_t s1 = (gt + 1) % C::kQStages;
            if (!mbar_wait(bar(C::kQFull + s1), ((gt + 1) / C::kQStages) & 1u, abort_flag)) { ok = false; fail(); break; }
            tc_fence_after();
            issue_s(s1);
          }
          if (!mbar_wait(bar(C::kDsFull), pc & 1u, abort_flag)) { ok = false; fail(); break; }
          ++pc;
          tc_fence_after();
          // dQ^T = K^T dS^T into the dP columns (dP(t) has been read by now).
          // Issued before dK: the dQ group drains dQ^T while dK runs, so the
          // columns are free again for dP(t+1) about when dK(t) completes.
#pragma unroll
          for (int ks = 0; ks < kKRows / 16; ++ks)
            mma_f16_ss(tmem + kColDP, dadd(dsc_kt, ks * 2048), dadd(dsc_dsmn, ks * 2048), idesc_dq,
                       ks > 0 ? 1u : 0u);
          mma_commit(bar(C::kDqFull));
          // dK += dS^T Q   (A = dS^T K-major, B = Q MN-major)
          const uint64_t qmn = dadd(dsc_qmn, s * C::kQTileBytes);
#pragma unroll
          for (int ks = 0; ks < kQRows / 16; ++ks)
            mma_f16_ss(tmem + kColDK, dadd(dsc_ds, (ks / 4) * C::kAtom + (ks % 4) * 32),
                       dadd(qmn, ks * 2048), idesc_acc, (t == 0 && ks == 0) ? 0u : 1u);
          mma_commit(bar(C::kQEmpty + s));
          dq_pending = true;
          if (t + 1 < in.nq && !issue_dp((gt + 1) % C::kQStages)) { ok = false; fail(); break; }
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
  } else if (warp < kActWarps) {
    // ------------------------------------------------------------ activation warps
    const int wq = warp & 3;
    const int grp = warp >> 2;           // query columns [64 grp, 64 grp + 64) of a tile
    const int j = wq * 32 + lane;        // key row within the block = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const float c_s = score_mul(p.scale);
    const bool has_bias = p.bias_table != nullptr;
    uint32_t it = 0, g = 0;
    while (true) {
      const uint32_t slot = it & 1u;
      bool w = mbar_wait(bar(C::kItemFull + slot), (it >> 1) & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      const int2 item = item_slot[slot];
      warp_arrive(bar(C::kItemEmpty + slot), lane);
      ++it;
      if (item.x < 0) break;
      const SmItem in = decode_sm<kBand>(item, p);
      const int kb0 = in.kb * kKRows;   // first local key row of the block
      const int jl = kb0 + j;           // this thread's local key row
      // queries that see this key: [vis_lo, vis_hi) (none for a key past the sample)
      const int vis_lo = band_query_begin(jl, p.causal, p.window);
      const int vis_hi = jl < in.Lkv ? band_query_end(jl, p.window, in.Lq) : 0;
      // Query tiles inside [full_lo, full_hi) pair with every key of a full
      // block and need no mask (the band's bounds grow with the key, so the
      // block's last key bounds the first such query and its first key the last).
      const int full_lo = band_query_begin(kb0 + kKRows - 1, p.causal, p.window);
      const int full_hi = kb0 + kKRows <= in.Lkv ? band_query_end(kb0, p.window, in.Lq) : 0;
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
        const uint32_t s = g % C::kQStages;
        w = mbar_wait(bar(C::kQFull + s), (g / C::kQStages) & 1u, abort_flag);
        w = w && mbar_wait(bar(C::kSFull), g & 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); abort_now = true; break; }
        tc_fence_after();
        const float* st = stats + s * C::kStatFloats;
        // bias(query c, key j) * log2e is window entry c - j + 127; the copy
        // shifted by (j + 1) % 2 holds entries c0 - j + 127 .. (c0 even) at an
        // 8-byte aligned position.
        const int cp = (j + 1) & 1;
        const float4* st4 = reinterpret_cast<const float4*>(st);  // 16-byte aligned
        const float* bwin = st + C::kWinOff + cp * C::kBiasCopy + cp + (kKRows - 1) - j;
        const int qloc = (in.qt0 + t) * kQRows;
        const bool full = qloc >= full_lo && qloc + kQRows <= full_hi;
        int c_lo = 0, c_hi = kQRows;  // valid query columns: c_lo <= c < c_hi
        if (!full) {
          c_hi = min(kQRows, vis_hi - qloc);
          c_lo = max(0, vis_lo - qloc);
        }
        // Phase 1: P^T = exp2(S^T scale log2e + bias log2e - lse log2e); bf16
        // pairs go back into the S columns (query pair k of the group's 64 at
        // column 64 grp + k) and stay in registers for phase 2.
        uint32_t pp[32];
        {
          const int c0 = 64 * grp;
          uint32_t sr[64];  // the group's 64 columns in one load and one wait
          tmem_ld64(tmem + lane_off + kColS + c0, sr);
          // One straight-line body per (masked, bias) case.
          auto body = [&](auto masked, auto biased) {
            constexpr bool kMask = decltype(masked)::value;
            constexpr bool kBias = decltype(biased)::value;
#pragma unroll
            for (int q4 = 0; q4 < 16; ++q4) {
              float bv[4] = {0.f, 0.f, 0.f, 0.f};
              if (kDense) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int c = c0 + 4 * q4 + e;
                  bv[e] = (dcol != nullptr && c >= c_lo && c < c_hi)
                              ? __ldg(dcol + static_cast<long long>(qloc + c) * in.Lkv) * kLog2e
                              : 0.0f;
                }
              } else if (kBias) {
                const float2 b01 = *reinterpret_cast<const float2*>(bwin + c0 + 4 * q4);
                const float2 b23 = *reinterpret_cast<const float2*>(bwin + c0 + 4 * q4 + 2);
                bv[0] = b01.x; bv[1] = b01.y; bv[2] = b23.x; bv[3] = b23.y;
              }
              // exponent pairs: S * c + (bias - lse) log2e, two lanes per
              // instruction (kAug: the product step already subtracted lse)
              float2 off[2] = {make_float2(bv[0], bv[1]), make_float2(bv[2], bv[3])};
              if (!kAug) {
                const float4 l4 = st4[(c0 >> 2) + q4];  // -lse*log2e
                off[0] = add_f32x2(make_float2(l4.x, l4.y), off[0]);
                off[1] = add_f32x2(make_float2(l4.z, l4.w), off[1]);
              }
              const uint32_t* sq = &sr[4 * q4];
              const float2 x01 = fma_f32x2(make_float2(__uint_as_float(sq[0]), __uint_as_float(sq[1])),
                                           make_float2(c_s, c_s), off[0]);
              const float2 x23 = fma_f32x2(make_float2(__uint_as_float(sq[2]), __uint_as_float(sq[3])),
                                           make_float2(c_s, c_s), off[1]);
              float pv[4] = {ex2_approx(x01.x), ex2_approx(x01.y), ex2_approx(x23.x), ex2_approx(x23.y)};
              if (kMask) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int c = c0 + 4 * q4 + e;
                  if (c < c_lo || c >= c_hi) pv[e] = 0.0f;
                }
              }
              pp[2 * q4] = pack_bf16x2(pv[0], pv[1]);
              pp[2 * q4 + 1] = pack_bf16x2(pv[2], pv[3]);
            }
          };
          using F = std::false_type;
          using T = std::true_type;
          if (full) {
            if (has_bias || kDense) body(F{}, T{}); else body(F{}, F{});
          } else {
            if (has_bias || kDense) body(T{}, T{}); else body(T{}, F{});
          }
          tmem_st16(tmem + lane_off + kColS + c0, *reinterpret_cast<uint32_t(*)[16]>(&pp[0]));
          tmem_st16(tmem + lane_off + kColS + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(&pp[16]));
        }
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(bar(C::kPFull), lane);
        // Phase 2: dS^T = P^T (dP^T - D) once dP^T - D of this tile is in TMEM
        // (the product step subtracted D).  The product is taken on bf16 pairs:
        // dS goes to the MMAs as bf16 anyway, and the extra rounding of dP - D
        // adds at most 2^-9 relative error.
        w = mbar_wait(bar(C::kDpFull), g & 1u, abort_flag);
        // the diagonal buffer of this tile was flushed two tiles ago
        if (kTableGrad) w = w && mbar_wait(bar(C::kDbFree + (g & 1u)), ((g >> 1) & 1u) ^ 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); abort_now = true; break; }
        tc_fence_after();
        // dS^T row j, query atom grp: 16-byte chunk cc (8 queries) at (cc ^ (j % 8))
        uint8_t* dsrow = gbase + C::kDs + grp * C::kAtom + j * 128;
        // bias-table gradient: this lane's sums along six diagonals of the tile
        // (see below), offsets -32, -31, 0, 1, 32, 33 from its own
        float diag[6] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int c0 = 64 * grp + 32 * half;
          uint32_t dr[32];
          tmem_ld32(tmem + lane_off + kColDP + c0, dr);
          uint32_t dh[16];
          // dP - D rounded to bf16 pairs, times the bf16 P pairs (masked P is
          // exactly 0, so masked dS is too).
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            float2 v01 = make_float2(__uint_as_float(dr[4 * q4]), __uint_as_float(dr[4 * q4 + 1]));
            float2 v23 = make_float2(__uint_as_float(dr[4 * q4 + 2]), __uint_as_float(dr[4 * q4 + 3]));
            if (!kAug) {
              const float4 d4 = st4[((kQRows + c0) >> 2) + q4];  // -D
              v01 = add_f32x2(v01, make_float2(d4.x, d4.y));
              v23 = add_f32x2(v23, make_float2(d4.z, d4.w));
            }
            dh[2 * q4] = mul_bf16x2(pp[16 * half + 2 * q4], pack_bf16x2(v01.x, v01.y));
            dh[2 * q4 + 1] = mul_bf16x2(pp[16 * half + 2 * q4 + 1], pack_bf16x2(v23.x, v23.y));
          }
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int cc = 4 * half + v;
            *reinterpret_cast<uint4*>(dsrow + ((cc ^ (j & 7)) * 16)) =
                make_uint4(dh[4 * v], dh[4 * v + 1], dh[4 * v + 2], dh[4 * v + 3]);
          }
          if (kDenseGrad && gcol != nullptr) {
            // dense-bias gradient: each pair of the tile is visited once, so
            // its dS is added straight to its entry (a warp's lanes are
            // consecutive keys: one 128-byte segment per query column)
            float* gt = gcol + static_cast<long long>(qloc + c0) * in.Lkv;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int c = c0 + 2 * e;
              if (c >= c_lo && c < c_hi) atomicAdd(gt, __uint_as_float(dh[e] << 16));
              gt += in.Lkv;
              if (c + 1 >= c_lo && c + 1 < c_hi) atomicAdd(gt, __uint_as_float(dh[e] & 0xFFFF0000u));
              gt += in.Lkv;
            }
          }
          if (kTableGrad) {
            // dS(query c0 + i, key 32 wq + lane) lies on diagonal
            // (c0 - 32 wq + 127) + (i - lane) of the tile.  Lane l gathers the
            // warp's bf16 pairs (columns 2e, 2e + 1) with 2e - src = l (mod
            // 32): at step e it reads pair e of lane (2e - l) mod 32, whose
            // columns sit at offsets l, l + 1 when 2e >= l and l - 32, l - 31
            // otherwise.  The second half is 32 columns further on.
            float up0 = 0.0f, up1 = 0.0f, dn0 = 0.0f, dn1 = 0.0f;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const uint32_t v = __shfl_sync(0xffffffffu, dh[e], (2 * e - lane) & 31);
              const float v0 = __uint_as_float(v << 16), v1 = __uint_as_float(v & 0xFFFF0000u);
              if (2 * e >= lane) {
                up0 += v0;
                up1 += v1;
              } else {
                dn0 += v0;
                dn1 += v1;
              }
            }
            diag[2 * half] += dn0;      // offset 32 half - 32
            diag[2 * half + 1] += dn1;  // 32 half - 31
            diag[2 * half + 2] += up0;  // 32 half
            diag[2 * half + 3] += up1;  // 32 half + 1
          }
        }
        if (kTableGrad) {
          // window entry (query - key + 127) of the tile; a warp's lanes hit
          // consecutive words (the sums outside the window are zero)
          const int e0 = 127 - 32 * wq + 64 * grp + lane;
          float* win = reinterpret_cast<float*>(gbase + C::kDb + (g & 1u) * C::kDbBuf);
          constexpr int kOff[6] = {-32, -31, 0, 1, 32, 33};
#pragma unroll
          for (int k = 0; k < 6; ++k)
            if (e0 + kOff[k] >= 0 && e0 + kOff[k] < 255) atomicAdd(win + e0 + kOff[k], diag[k]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        warp_arrive(bar(C::kDsFull), lane);
        if (kTableGrad) {
          if (j == 0 && grp == 0) {
            int* meta = reinterpret_cast<int*>(gbase + C::kDb + (g & 1u) * C::kDbBuf + 256 * 4);
            meta[0] = qloc - kb0 - 127;  // diagonal (query - key) of window entry 0
            meta[1] = in.head;
          }
          warp_arrive(bar(C::kDbAcc + (g & 1u)), lane);
        }
      }
      if (abort_now) break;
    }
  } else if (warp < 12) {
    // ------------------------------------------------------------ dQ group + dK/dV epilogue
    setmaxnreg_inc<kRegsDq>();
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // TMEM lane: channel (dQ^T) or key row (dK, dV)
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    uint32_t it = 0, dqc = 0, dkvc = 0, dq_issue = 0;
    volatile int* group_ok = reinterpret_cast<volatile int*>(gbase + C::kGroupOk);
    const bool out32 = aligned32(p.dk, p.dv);
    while (true) {
      const uint32_t slot = it & 1u;
      bool w = mbar_wait(bar(C::kItemFull + slot), (it >> 1) & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      const int2 item = item_slot[slot];
      warp_arrive(bar(C::kItemEmpty + slot), lane);
      ++it;
      if (item.x < 0) break;
      const SmItem in = decode_sm<kBand>(item, p);
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
        // The whole dQ^T tile (channel r, 128 queries) into registers first, in
        // two loads of 64 columns (two waits).
        uint32_t v[128];
        tmem_ld64(tmem + lane_off + kColDP, *reinterpret_cast<uint32_t(*)[64]>(&v[0]));
        tmem_ld64(tmem + lane_off + kColDP + 64, *reinterpret_cast<uint32_t(*)[64]>(&v[64]));
        tc_fence_before();
        warp_arrive(bar(C::kDqEmpty), lane);  // the dP columns are free again
        // Stage 16-query chunks as [query][channel] and add each into the fp32
        // dQ rows with one bulk tensor reduce.  Columns of queries outside the
        // sample carry exact zeros (their dS is 0), so a box that runs into the
        // next sample adds nothing; chunks past the sample are skipped and rows
        // past Tq are clipped by the copy.
        const int qloc = (in.qt0 + t) * kQRows;
        const int qrow = in.q0 + qloc;
        // each warp reduces its own 32 channels: no group barrier
        const uint32_t wstage = sbase + C::kDqStage + wq * C::kDqWarpBufs * (kDqChunk * 32 * 4);
        float* wstg = reinterpret_cast<float*>(gbase + C::kDqStage) + wq * C::kDqWarpBufs * (kDqChunk * 32);
#pragma unroll
        for (int ch = 0; ch < kQRows / kDqChunk; ++ch) {
          if (qloc + ch * kDqChunk >= in.Lq) break;  // uniform across the group
          const int buf = dq_issue % C::kDqWarpBufs;
          if (lane == 0) bulk_wait_group_read<C::kDqWarpBufs - 1>();
          __syncwarp();
          if (32 * wq < D) {
            float* stg = wstg + buf * (kDqChunk * 32);
#pragma unroll
            for (int c = 0; c < kDqChunk; ++c)
              stg[c * 32 + lane] = __uint_as_float(v[ch * kDqChunk + c]);
            fence_proxy_async_smem();
          }
          __syncwarp();
          if (lane == 0 && 32 * wq < D) {
            tma_reduce_add_3d(&tmap_dq, wstage + buf * (kDqChunk * 32 * 4), 32 * wq, in.head,
                              qrow + ch * kDqChunk);
            bulk_commit_group();
          }
          ++dq_issue;
        }
      }
      if (abort_now) break;
      // epilogue: dV and dK rows of this key block
      const int jl = in.kb * kKRows + r;
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
          if (kRope && which == 1) {  // dK back through the rotary embedding
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
        warp_arrive(bar(C::kDkvEmpty), lane);
      } else if (row_ok) {
        uint4* a4 = reinterpret_cast<uint4*>(p.dv + grow);
        uint4* b4 = reinterpret_cast<uint4*>(p.dk + grow);
        for (int q = 0; q < D / 8; ++q) {
          a4[q] = make_uint4(0, 0, 0, 0);
          b4[q] = make_uint4(0, 0, 0, 0);
        }
      }
    }
    if (lane == 0) bulk_wait_group_all();  // every dQ reduce issued by this thread has landed
  } else {
    setmaxnreg_dec<kRegsLow>();  // spare warps of the last warpgroup
    if (kTableGrad && warp == kMmaWarp + 1) {
      // ---------------------------------------------------------- bias-table gradient
      // Per tile: wait for the activation warps' diagonal sums, add them to the
      // table (entry = clamp(query - key + max_rel - 1)), zero the buffer.
      const int width = 2 * p.max_rel - 1;
      uint32_t it = 0, g = 0;
      while (true) {
        const uint32_t slot = it & 1u;
        bool w = mbar_wait(bar(C::kItemFull + slot), (it >> 1) & 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
        const int2 item = item_slot[slot];
        warp_arrive(bar(C::kItemEmpty + slot), lane);
        ++it;
        if (item.x < 0) break;
        const SmItem in = decode_sm<kBand>(item, p);
        bool abort_now = false;
        for (int t = 0; t < in.nq; ++t, ++g) {
          const uint32_t u = g & 1u;
          w = mbar_wait(bar(C::kDbAcc + u), (g >> 1) & 1u, abort_flag);
          if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); abort_now = true; break; }
          float* win = reinterpret_cast<float*>(gbase + C::kDb + u * C::kDbBuf);
          const int* meta = reinterpret_cast<const int*>(win + 256);
          const int delta0 = meta[0];
          float* row = p.dbias + static_cast<long long>(meta[1]) * width;
          for (int e = lane; e < 255; e += 32) {
            const float v = win[e];
            if (v != 0.0f) atomicAdd(row + min(max(e + delta0 + p.max_rel - 1, 0), width - 1), v);
            win[e] = 0.0f;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(C::kDbFree + u));
        }
        if (abort_now) break;
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

template <int D, bool kBand, bool kDBias, bool kDense, bool kRope, bool kAug>
cudaError_t launch_sm_cfg(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                          int grid, cudaStream_t s) {
  using C = SmCfg<D, kAug>;
  static_assert(C::kSmemBytes <= 232448, "shared memory budget");
  // The register split (setmaxnreg) hands out exactly the launch's pool of
  // 128 per thread: refuse a build that launched with fewer.
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, bwd_sm_kernel<D, kBand, kDBias, kDense, kRope, kAug>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != 128) return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(bwd_sm_kernel<D, kBand, kDBias, kDense, kRope, kAug>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  bwd_sm_kernel<D, kBand, kDBias, kDense, kRope, kAug><<<grid, kThreads, C::kSmemBytes, s>>>(
      tq, tk, tv, tdo, tdq, p);
  return cudaGetLastError();
}

// The extra product step goes with a relative-position table (always present
// with its gradient; never with a dense bias).
template <int D, bool kBand, bool kDBias, bool kDense, bool kRope>
cudaError_t launch_sm(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                      const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                      int grid, cudaStream_t s) {
  if constexpr (kDense) {
    return launch_sm_cfg<D, kBand, kDBias, true, kRope, false>(p, tq, tk, tv, tdo, tdq, grid, s);
  } else if constexpr (kDBias) {
    return launch_sm_cfg<D, kBand, true, false, kRope, true>(p, tq, tk, tv, tdo, tdq, grid, s);
  } else {
    if (p.bias_table != nullptr)
      return launch_sm_cfg<D, kBand, false, false, kRope, true>(p, tq, tk, tv, tdo, tdq, grid, s);
    return launch_sm_cfg<D, kBand, false, false, kRope, false>(p, tq, tk, tv, tdo, tdq, grid, s);
  }
}

template <bool kRope>
cudaError_t dispatch_sm(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                           int grid, cudaStream_t s) {
  const bool band = p.window > 0;
  const bool db = p.dbias != nullptr;
  const bool dense = p.bias_dense != nullptr;
#define GDPA_SM_LAUNCH(DD, BB, DBB, DNS) \
  if (p.d == DD && band == BB && db == DBB && dense == DNS) \
    return launch_sm<DD, BB, DBB, DNS, kRope>(p, tq, tk, tv, tdo, tdq, grid, s);
  GDPA_SM_LAUNCH(64, false, false, false)
  GDPA_SM_LAUNCH(64, false, true, false)
  GDPA_SM_LAUNCH(64, true, false, false)
  GDPA_SM_LAUNCH(64, true, true, false)
  GDPA_SM_LAUNCH(128, false, false, false)
  GDPA_SM_LAUNCH(128, false, true, false)
  GDPA_SM_LAUNCH(128, true, false, false)
  GDPA_SM_LAUNCH(128, true, true, false)
  GDPA_SM_LAUNCH(64, false, false, true)
  GDPA_SM_LAUNCH(64, false, true, true)
  GDPA_SM_LAUNCH(64, true, false, true)
  GDPA_SM_LAUNCH(64, true, true, true)
  GDPA_SM_LAUNCH(128, false, false, true)
  GDPA_SM_LAUNCH(128, false, true, true)
  GDPA_SM_LAUNCH(128, true, false, true)
  GDPA_SM_LAUNCH(128, true, true, true)
#undef GDPA_SM_LAUNCH
  return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace gdpa
