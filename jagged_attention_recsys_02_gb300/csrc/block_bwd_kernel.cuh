// Block-aligned attention: the backward kernel and its launch templates
// (shared pieces in block_common.cuh), compiled from block_bwd.cu (without
// a bias gradient), block_bwd_db.cu (the bias-table gradient),
// block_bwd_dense.cu (a dense jagged bias) and block_bwd_dense_db.cu (a dense
// bias and its gradient).
#pragma once
#include "block_common.cuh"

namespace gdpa {
namespace {

using namespace ptx;

// ---------------------------------------------------------------- backward
// One tile at a time per CTA (TMEM holds S, dP / dQ, dK and dV of a tile), all
// products on the tensor cores, rows of TMEM = tile rows:
//   S = Q K^T, dP = dO V^T                  (queries x keys)
//   activation: P = exact softmax of the row's block (or act(S)); D = sum P dP;
//               dS = P (dP - D) (or act'(S) dP); P, then dS, to shared memory
//   dV = P^T dO, dK = scale dS^T Q, dQ = scale dS K   (no atomics: a tile owns
//               every gradient row it touches)
// GDPA activations have no normalisation, so a 16-bit P or dS loses too much
// on near-zero gradients; their P and dS go through the buffer twice, as bf16
// hi and lo = x - hi parts, each followed by its products (accumulating).
// dS is formed once (dQ's hi part overwrites dP), its lo part kept in
// registers until the buffer is free.
// 320 threads: warps 0-3 activation (one query row each), warps 4-7
// epilogue (read dQ / dK / dV rows out of TMEM, store bf16), warp 8 TMA
// producer, warp 9 MMA issuer.  Shared memory: Q + K in two slots (the next
// tile's arrive while this one computes), V + dO in one slot (free once dP and
// dV are done), and one P / dS buffer.  TMEM: S [0,128), dP then dQ
// [128,128+d), dK [256,256+d), dV [384,384+d).
constexpr int kBwdThreads = 320;
constexpr int kBwdEpi0 = 4;
constexpr int kBwdProducer = 8;
constexpr int kBwdMma = 9;
constexpr uint32_t kColS = 0, kColDP = 128, kColDK = 256, kColDV = 384;

template <int D>
struct BbCfg {
  static constexpr int kTileBytes = kTileRows * D * 2;
  static constexpr int kAtom = kTileRows * 128;             // 64 bf16 columns of 128 rows
  static constexpr int kQK = 0;                             // slot i: Q at kQK + i*2*tile, K after it
  static constexpr int kVO = 4 * kTileBytes;                // V, then dO
  static constexpr int kPS = kVO + 2 * kTileBytes;          // P / dS: [key atom][query][64 keys]
  static constexpr int kPSBytes = kTileRows * kTileRows * 2;
  static constexpr int kBias = kPS + kPSBytes;              // bias window of the current head
  // bias-table gradient of the current tile: dS summed along the diagonals
  // query - key = e - (kBlk - 1), e in [0, 2 kBlk - 1) (a block's pairs only)
  static constexpr int kDbWin = kBias + 4 * (2 * kTileRows - 1) + 4;
  static constexpr int kBar = kDbWin + 4 * 2 * kBlk;
  static constexpr int kQKFull = 0, kQKEmpty = 2;           // + slot
  static constexpr int kVOFull = 4, kVOEmpty = 5;            // V (free after dP)
  static constexpr int kSFull = 6, kDpFull = 7, kPFull = 8, kDvDone = 9, kDsFull = 10;
  static constexpr int kGradFull = 11, kEpiDone = 12, kDrain = 13;
  static constexpr int kWinFree = 14, kWinReady = 15;      // bias window restaging
  static constexpr int kDsDone = 16;                        // GDPA: dK, dQ of dS's hi part done
  static constexpr int kOFull = 17, kOEmpty = 18;           // dO (V uses kVOFull / kVOEmpty)
  // epilogue of a full tile: each gradient is staged in the P / dS buffer and
  // leaves by TMA store; the buffer goes back to the activation warps after
  static constexpr int kEpiStaged = 19, kEpiFree = 20, kPsFree = 21;
  static constexpr int kDbAcc = 22, kDbFree = 23;           // gradient window: added, flushed
  static constexpr int kNumBars = 24;
  static constexpr int kTmemSlot = kBar + 8 * kNumBars;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kUsed = kAbort + 4;
  static constexpr int kSmemBytes = kUsed + 1024;
};

// Row r's 16*NCH packed bf16 pairs (keys cb .. cb + 32*NCH) into the P / dS
// buffer: key k of row r sits in atom k/64, 16-byte chunk (k%64)/8 swizzled
// with r%8 (the 128-byte swizzle the MMA descriptors use).
template <int NCH>
__device__ __forceinline__ void ps_store_row(uint8_t* ps, int r, int cb, const uint32_t* w) {
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    const int k0 = cb + 32 * ch;
    uint8_t* row = ps + (k0 / 64) * (kTileRows * 128) + r * 128;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int cc = (k0 % 64) / 8 + v;
      *reinterpret_cast<uint4*>(row + ((cc ^ (r & 7)) * 16)) =
          make_uint4(w[16 * ch + 4 * v], w[16 * ch + 4 * v + 1], w[16 * ch + 4 * v + 2],
                     w[16 * ch + 4 * v + 3]);
    }
  }
}

__device__ __forceinline__ void ps_zero_atom(uint8_t* ps, int r, int atom) {
  uint8_t* row = ps + atom * (kTileRows * 128) + r * 128;
  // in swizzled order, so that each store instruction of a warp spreads over
  // all banks (the row's chunks are all zero either way)
#pragma unroll
  for (int v = 0; v < 8; ++v)
    *reinterpret_cast<uint4*>(row + ((v ^ (r & 7)) * 16)) = make_uint4(0, 0, 0, 0);
}

template <int D, int ACT, bool kDBias, bool kDense>
__global__ void __launch_bounds__(kBwdThreads, 1)
block_bwd_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                 const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                 const __grid_constant__ CUtensorMap tmap_dq, const __grid_constant__ CUtensorMap tmap_dk,
                 const __grid_constant__ CUtensorMap tmap_dv, const BlockParams p) {
  using C = BbCfg<D>;
  constexpr bool kSoftmax = (ACT == GDPA_ACT_SOFTMAX);
  constexpr int kParts = kSoftmax ? 1 : 2;  // P / dS passes through the buffer per tile
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  auto bar = [&](int i) -> uint32_t { return sbase + C::kBar + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kAbort);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::kQKFull + i), 1);
      mbar_init(bar(C::kQKEmpty + i), 1);
    }
    mbar_init(bar(C::kVOFull), 1);
    mbar_init(bar(C::kVOEmpty), 1);
    mbar_init(bar(C::kSFull), 1);
    mbar_init(bar(C::kDpFull), 1);
    mbar_init(bar(C::kPFull), 4);
    mbar_init(bar(C::kDvDone), 1);
    mbar_init(bar(C::kDsFull), 4);
    mbar_init(bar(C::kGradFull), 1);
    mbar_init(bar(C::kEpiDone), 4);
    mbar_init(bar(C::kDrain), 1);
    mbar_init(bar(C::kWinFree), 4);
    mbar_init(bar(C::kWinReady), 4);
    mbar_init(bar(C::kDsDone), 1);
    mbar_init(bar(C::kOFull), 1);
    mbar_init(bar(C::kOEmpty), 1);
    mbar_init(bar(C::kEpiStaged), 4);
    mbar_init(bar(C::kEpiFree), 1);
    mbar_init(bar(C::kPsFree), 1);
    mbar_init(bar(C::kDbAcc), 4);
    mbar_init(bar(C::kDbFree), 4);
    fence_mbar_init();
  }
  if (threadIdx.x < 2 * kBlk) reinterpret_cast<float*>(gbase + C::kDbWin)[threadIdx.x] = 0.0f;
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp == kBwdProducer && lane == 0) {
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
  const int n_items = *p.n_tiles * p.H;
  auto item_of = [&](int k) { return static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x); };

  if (warp == kBwdProducer) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int last_qk[2] = {-1, -1}, last_vo = -1, last_o = -1;
      for (int k = 0;; ++k) {
        const int item = item_of(k);
        if (item >= n_items) break;
        const int head = item % p.H;
        const int row0 = p.tiles[item / p.H].x;
        const uint32_t slot = k & 1;
        if (!mbar_wait(bar(C::kQKEmpty + slot), ((k >> 1) & 1u) ^ 1u, abort_flag)) { fail(); break; }
        const uint32_t qk = sbase + C::kQK + slot * 2 * C::kTileBytes;
        mbar_arrive_expect_tx(bar(C::kQKFull + slot), 2 * C::kTileBytes);
#pragma unroll
        for (int x = 0; x < D; x += 64) {
          const uint32_t off = (x / 64) * C::kAtom;
          tma_load_3d(qk + off, &tmap_q, bar(C::kQKFull + slot), x, head, row0);
          tma_load_3d(qk + C::kTileBytes + off, &tmap_k, bar(C::kQKFull + slot), x, head, row0);
        }
        last_qk[slot] = k;
        // V frees up after dP, dO after dV: separate barriers let each load start early
        const uint32_t vo = sbase + C::kVO;
        if (!mbar_wait(bar(C::kVOEmpty), (k & 1u) ^ 1u, abort_flag)) { fail(); break; }
        mbar_arrive_expect_tx(bar(C::kVOFull), C::kTileBytes);
#pragma unroll
        for (int x = 0; x < D; x += 64)
          tma_load_3d(vo + (x / 64) * C::kAtom, &tmap_v, bar(C::kVOFull), x, head, row0);
        last_vo = k;
        if (!mbar_wait(bar(C::kOEmpty), (k & 1u) ^ 1u, abort_flag)) { fail(); break; }
        mbar_arrive_expect_tx(bar(C::kOFull), C::kTileBytes);
#pragma unroll
        for (int x = 0; x < D; x += 64)
          tma_load_3d(vo + C::kTileBytes + (x / 64) * C::kAtom, &tmap_do, bar(C::kOFull), x, head,
                      row0);
        last_o = k;
      }
      if (*abort_flag) {
        for (int i = 0; i < 2; ++i)
          if (last_qk[i] >= 0)
            mbar_wait(bar(C::kQKFull + i), (last_qk[i] >> 1) & 1u, nullptr, 50000000ull);
        if (last_vo >= 0) mbar_wait(bar(C::kVOFull), last_vo & 1u, nullptr, 50000000ull);
        if (last_o >= 0) mbar_wait(bar(C::kOFull), last_o & 1u, nullptr, 50000000ull);
      }
    }
  } else if (warp == kBwdMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16(128, kTileRows, true, false, false);    // S, dP
      constexpr uint32_t idesc_t = idesc_f16(128, D, true, true, true);              // dV, dK
      constexpr uint32_t idesc_q = idesc_f16(128, D, true, false, true);             // dQ
      const uint64_t dsc_qk = sdesc(sbase + C::kQK, 0, 1024, kSwizzle128B);         // Q / K, K-major
      const uint64_t dsc_qk_mn = sdesc(sbase + C::kQK, C::kAtom, 1024, kSwizzle128B);  // Q / K as MN-major B
      const uint64_t dsc_vo = sdesc(sbase + C::kVO, 0, 1024, kSwizzle128B);         // V / dO, K-major
      const uint64_t dsc_do_mn = sdesc(sbase + C::kVO + C::kTileBytes, C::kAtom, 1024, kSwizzle128B);
      const uint64_t dsc_ps = sdesc(sbase + C::kPS, 0, 1024, kSwizzle128B);         // dS, K-major A
      const uint64_t dsc_ps_mn = sdesc(sbase + C::kPS, C::kAtom, 1024, kSwizzle128B);  // P^T / dS^T, MN-major A
      bool issued_any = false;
      auto issue_nt = [&](uint32_t d_col, uint64_t a, uint64_t b) {  // [128 x 128] = A B^T over d
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks / 4) * C::kAtom + (ks % 4) * 32;
          mma_f16_ss(tmem + d_col, dadd(a, off), dadd(b, off), idesc_s, ks > 0 ? 1u : 0u);
        }
        issued_any = true;
      };
      auto qk_of = [&](int k) { return static_cast<uint32_t>((k & 1) * 2 * C::kTileBytes); };
      bool ok = item_of(0) < n_items;
      if (ok) {
        if (!mbar_wait(bar(C::kQKFull), 0, abort_flag)) { fail(); ok = false; }
        if (ok) {
          tc_fence_after();
          issue_nt(kColS, dsc_qk, dadd(dsc_qk, C::kTileBytes));
          mma_commit(bar(C::kSFull));
          if (!mbar_wait(bar(C::kVOFull), 0, abort_flag) || !mbar_wait(bar(C::kOFull), 0, abort_flag)) {
            fail();
            ok = false;
          }
        }
        if (ok) {
          tc_fence_after();
          issue_nt(kColDP, dadd(dsc_vo, C::kTileBytes), dsc_vo);
          mma_commit(bar(C::kDpFull));
          mma_commit(bar(C::kVOEmpty));  // V(0) is read
        }
      }
      for (int k = 0; ok; ++k) {
        const bool next = item_of(k + 1) < n_items;
        const uint32_t qk = qk_of(k);
        // P(k) in shared memory (per part): dV = P^T dO
        bool okp = true;
        for (int part = 0; part < kParts && okp; ++part) {
          if (!mbar_wait(bar(C::kPFull), (k * kParts + part) & 1u, abort_flag)) { okp = false; break; }
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < kTileRows / 16; ++ks)
            mma_f16_ss(tmem + kColDV, dadd(dsc_ps_mn, ks * 2048), dadd(dsc_do_mn, ks * 2048),
                       idesc_t, (part > 0 || ks > 0) ? 1u : 0u);
          mma_commit(bar(C::kDvDone));
        }
        if (!okp) { fail(); break; }
        mma_commit(bar(C::kOEmpty));  // dO(k) is read
        // S(k+1): softmax is done reading S(k) once P(k) is out; the GDPA
        // activations read S(k) again for act'(S), so theirs waits for dS(k)'s
        // hi part
        auto issue_next_s = [&]() -> bool {
          if (!mbar_wait(bar(C::kQKFull + ((k + 1) & 1)), ((k + 1) >> 1) & 1u, abort_flag)) return false;
          tc_fence_after();
          const uint32_t q1 = qk_of(k + 1);
          issue_nt(kColS, dadd(dsc_qk, q1), dadd(dsc_qk, q1 + C::kTileBytes));
          mma_commit(bar(C::kSFull));
          return true;
        };
        if (kSoftmax && next && !issue_next_s()) { fail(); break; }
        // dS(k) in shared memory (per part): dK = dS^T Q, dQ = dS K (into the dP columns)
        for (int part = 0; part < kParts && okp; ++part) {
          if (!mbar_wait(bar(C::kDsFull), (k * kParts + part) & 1u, abort_flag)) { okp = false; break; }
          tc_fence_after();
          // GDPA: S(k) and dP(k) are read once dS's hi part is out
          if (!kSoftmax && part == 0 && next && !issue_next_s()) { okp = false; break; }
#pragma unroll
          for (int ks = 0; ks < kTileRows / 16; ++ks)
            mma_f16_ss(tmem + kColDK, dadd(dsc_ps_mn, ks * 2048), dadd(dsc_qk_mn, qk + ks * 2048),
                       idesc_t, (part > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
          for (int ks = 0; ks < kTileRows / 16; ++ks)
            mma_f16_ss(tmem + kColDP, dadd(dsc_ps, (ks / 4) * C::kAtom + (ks % 4) * 32),
                       dadd(dsc_qk_mn, qk + C::kTileBytes + ks * 2048), idesc_q,
                       (part > 0 || ks > 0) ? 1u : 0u);
          if (part < kParts - 1) mma_commit(bar(C::kDsDone));
        }
        if (!okp) { fail(); break; }
        mma_commit(bar(C::kGradFull));
        mma_commit(bar(C::kQKEmpty + (k & 1)));
        if (!next) break;
        // dP(k+1) into the dP columns once the epilogue has read dQ(k) out of them
        if (!mbar_wait(bar(C::kEpiDone), k & 1u, abort_flag)) { fail(); break; }
        if (!mbar_wait(bar(C::kVOFull), (k + 1) & 1u, abort_flag) ||
            !mbar_wait(bar(C::kOFull), (k + 1) & 1u, abort_flag)) { fail(); break; }
        tc_fence_after();
        issue_nt(kColDP, dadd(dsc_vo, C::kTileBytes), dsc_vo);
        mma_commit(bar(C::kDpFull));
        mma_commit(bar(C::kVOEmpty));  // V(k+1) is read
      }
      if (issued_any) {
        mma_commit(bar(C::kDrain));
        mbar_wait(bar(C::kDrain), 0, nullptr, 100000000ull);
      }
    }
  } else if (warp < kBwdEpi0) {
    // ------------------------------------------------------------ activation warps
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // query row of the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_off + kColS;
    const uint32_t t_dp = tmem + lane_off + kColDP;
    uint8_t* ps = gbase + C::kPS;
    const float c_s = kSoftmax ? p.scale * kLog2e : p.scale;
    const bool has_bias = p.bias_table != nullptr;
    float* win = reinterpret_cast<float*>(gbase + C::kBias);
    const float* bwin = win + (kTileRows - 1) + r;  // bwin[-c] = bias(r - c)
    int win_head = -1;
    uint32_t n_win = 0;
    // bias-table gradient: each pair's dS (fp32) is added to the shared window
    // entry of its diagonal (a warp's 32 rows hit 32 different entries per
    // key), flushed to the table after every tile
    float* dwin = reinterpret_cast<float*>(gbase + C::kDbWin);
    constexpr bool want_db = kDBias && !kDense;
    // dense bias (kDense): row r's value of column c is drow[c]; its gradient
    // (kDBias too) goes to the same place in p.dbias, each pair's dS added
    // once by the thread that owns the pair
    constexpr bool kDenseGrad = kDBias && kDense;
    uint32_t n_db = 0;
    for (int k = 0;; ++k) {
      const int item = item_of(k);
      if (item >= n_items) break;
      const int head = item % p.H;
      const TileInfo ti = load_tile(p.tiles, item / p.H);
      if (has_bias && head != win_head) {
        // The four activation warps restage the window for a new head, once
        // all of them are done with the old one (bounded mbarrier waits, so a
        // warp that gave up cannot leave the others stuck).
        warp_arrive(bar(C::kWinFree), lane);
        bool wf = mbar_wait(bar(C::kWinFree), n_win & 1u, abort_flag);
        if (!__all_sync(0xffffffffu, wf)) { if (lane == 0) fail(); break; }
        for (int e = threadIdx.x; e < 2 * kTileRows - 1; e += 128)
          win[e] = __ldg(p.bias_table + static_cast<long long>(head) * (2 * p.max_rel - 1) +
                         min(max(e - (kTileRows - 1) + p.max_rel - 1, 0), 2 * p.max_rel - 2)) *
                   (kSoftmax ? kLog2e : 1.0f);
        warp_arrive(bar(C::kWinReady), lane);
        wf = mbar_wait(bar(C::kWinReady), n_win & 1u, abort_flag);
        if (!__all_sync(0xffffffffu, wf)) { if (lane == 0) fail(); break; }
        ++n_win;
        win_head = head;
      }
      int c_lo, c_hi;
      row_keys(ti, r, p.causal, &c_lo, &c_hi);
      const float* drow = nullptr;
      float* grow = nullptr;
      if (kDense) {
        const long long base = dense_row_base(p, ti, r, head);
        if (base >= 0) {
          drow = p.bias_dense + base;
          if (kDenseGrad) grow = p.dbias + base;
        }
      }
      // dense-bias gradient of (row r, column c), keys the row sees only
      auto add_dense = [&](int c, float v) {
        if (c >= c_lo && c < c_hi) atomicAdd(grow + c, v);
      };
      bool w = mbar_wait(bar(C::kSFull), k & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      tc_fence_after();
      bool abort_now = false;
      // dS of (row r, key column c) on its diagonal entry (keys the row sees only)
      auto add_db = [&](int c, float v) {
        if (c >= c_lo && c < c_hi) atomicAdd(dwin + (r - c + kBlk - 1), v);
      };
      // NCH 32-column chunks from column cb hold the row's keys.  P stays in
      // registers as bf16 pairs; everything else is formed one chunk at a
      // time from TMEM (S is read twice, dP twice for softmax).
      auto run = [&](auto nch, int cb) {
        constexpr int NCH = decltype(nch)::value;
        // x = S * c_s + bias (log2 units for softmax); keys outside the row's
        // block: -inf (softmax) or NaN (GDPA: P = act' = 0 there)
        auto load_x = [&](int ch, float (&x)[32]) {
          uint32_t sr[32];
          tmem_ld32(t_s + cb + 32 * ch, sr);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int c = cb + 32 * ch + i;
            float v = __uint_as_float(sr[i]) * c_s;
            if (kDense) {
              if (c >= c_lo && c < c_hi) v += __ldg(drow + c) * (kSoftmax ? kLog2e : 1.0f);
            } else if (has_bias) {
              v += bwin[-c];
            }
            x[i] = (c >= c_lo && c < c_hi) ? v : (kSoftmax ? -INFINITY : __int_as_float(0x7fffffff));
          }
        };
        auto wait_all = [&](int b, uint32_t parity) -> bool {
          const bool ok = mbar_wait(bar(b), parity, abort_flag);
          if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) fail();
            abort_now = true;
            return false;
          }
          return true;
        };
        auto publish = [&](int b) {  // the buffer rows are written: hand them to the MMAs
          if (NCH == 2) ps_zero_atom(ps, r, cb == 0 ? 1 : 0);
          fence_proxy_async_smem();
          tc_fence_before();
          warp_arrive(bar(b), lane);
        };
        if (kSoftmax) {
          uint32_t pw[16 * NCH];  // P as bf16 pairs
          // exact row softmax: max and sum in one pass (rescaling the sum per
          // chunk), then P = exp2(x - m) / l
          float m = -INFINITY, l = 0.0f;
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) {
            float x[32];
            load_x(ch, x);
            float mc = m;
#pragma unroll
            for (int i = 0; i < 32; ++i) mc = fmaxf(mc, x[i]);
            const float ref = (mc == -INFINITY) ? 0.0f : mc;
            float sum = 0.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i) sum += ex2_approx(x[i] - ref);
            l = (m == -INFINITY ? 0.0f : l * ex2_approx(m - ref)) + sum;
            m = mc;
          }
          const float m_ref = (m == -INFINITY) ? 0.0f : m;
          const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) {
            float x[32];
            load_x(ch, x);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pw[16 * ch + i] = pack_bf16x2(ex2_approx(x[2 * i] - m_ref) * inv_l,
                                            ex2_approx(x[2 * i + 1] - m_ref) * inv_l);
          }
          // P into the buffer once the previous tile's epilogue is done with it
          if (k > 0 && !wait_all(C::kPsFree, (k - 1) & 1u)) return;
          ps_store_row<NCH>(ps, r, cb, pw);
          publish(C::kPFull);
          // dS = P (dP - D), D = sum P dP
          if (!wait_all(C::kDpFull, k & 1u)) return;
          tc_fence_after();
          float dsum = 0.0f;
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) {
            uint32_t dr[32];
            tmem_ld32(t_dp + cb + 32 * ch, dr);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint32_t pv = pw[16 * ch + i];
              dsum = fmaf(__uint_as_float(pv << 16), __uint_as_float(dr[2 * i]), dsum);
              dsum = fmaf(__uint_as_float(pv & 0xFFFF0000u), __uint_as_float(dr[2 * i + 1]), dsum);
            }
          }
          // dS overwrites P once dV(k) has read it
          if (!wait_all(C::kDvDone, k & 1u)) return;
          tc_fence_after();
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) {
            uint32_t dr[32];
            tmem_ld32(t_dp + cb + 32 * ch, dr);
            uint32_t dw[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint32_t pv = pw[16 * ch + i];
              const float d0 = __uint_as_float(pv << 16) * (__uint_as_float(dr[2 * i]) - dsum);
              const float d1 = __uint_as_float(pv & 0xFFFF0000u) * (__uint_as_float(dr[2 * i + 1]) - dsum);
              dw[i] = pack_bf16x2(d0, d1);
              if (want_db) {
                add_db(cb + 32 * ch + 2 * i, d0);
                add_db(cb + 32 * ch + 2 * i + 1, d1);
              }
              if (kDenseGrad) {  // the bf16 dS the products use
                add_dense(cb + 32 * ch + 2 * i, __uint_as_float(dw[i] << 16));
                add_dense(cb + 32 * ch + 2 * i + 1, __uint_as_float(dw[i] & 0xFFFF0000u));
              }
            }
            ps_store_row<1>(ps, r, cb + 32 * ch, dw);
          }
          publish(C::kDsFull);
        } else {
          // P = act(S) and dS = act'(S) dP, each as a bf16 hi part and a lo part,
          // formed chunk by chunk from TMEM (S stays there until dS is out)
          for (int part = 0; part < 2; ++part) {
            if (part == 0 && k > 0 && !wait_all(C::kPsFree, (k - 1) & 1u)) return;
            if (part == 1 && !wait_all(C::kDvDone, (2 * k) & 1u)) return;  // dV read the hi part
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
              float x[32];
              load_x(ch, x);
              uint32_t pw[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float a0 = x[2 * i] != x[2 * i] ? 0.0f : act_fwd(ACT, x[2 * i]);
                const float a1 = x[2 * i + 1] != x[2 * i + 1] ? 0.0f : act_fwd(ACT, x[2 * i + 1]);
                const uint32_t h = pack_bf16x2(a0, a1);
                pw[i] = part == 0 ? h
                                  : pack_bf16x2(a0 - __uint_as_float(h << 16),
                                                a1 - __uint_as_float(h & 0xFFFF0000u));
              }
              ps_store_row<1>(ps, r, cb + 32 * ch, pw);
            }
            publish(C::kPFull);
          }
          // dS from S and dP (both read once: dQ's hi part lands in the dP
          // columns); the hi part goes to the buffer once dV read P's lo part,
          // the lo part waits in registers until dK and dQ read the hi part
          if (!wait_all(C::kDpFull, k & 1u)) return;
          if (!wait_all(C::kDvDone, (2 * k + 1) & 1u)) return;
          tc_fence_after();
          uint32_t dl[16 * NCH];
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) {
            float x[32];
            load_x(ch, x);
            uint32_t dr[32];
            tmem_ld32(t_dp + cb + 32 * ch, dr);
            uint32_t dw[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float a0, g0, a1, g1;
              act_and_grad<ACT>(x[2 * i], a0, g0);
              act_and_grad<ACT>(x[2 * i + 1], a1, g1);
              const float d0 = x[2 * i] != x[2 * i] ? 0.0f : g0 * __uint_as_float(dr[2 * i]);
              const float d1 = x[2 * i + 1] != x[2 * i + 1] ? 0.0f : g1 * __uint_as_float(dr[2 * i + 1]);
              if (want_db) {
                add_db(cb + 32 * ch + 2 * i, d0);
                add_db(cb + 32 * ch + 2 * i + 1, d1);
              }
              if (kDenseGrad) {
                add_dense(cb + 32 * ch + 2 * i, d0);
                add_dense(cb + 32 * ch + 2 * i + 1, d1);
              }
              const uint32_t h = pack_bf16x2(d0, d1);
              dw[i] = h;
              dl[16 * ch + i] = pack_bf16x2(d0 - __uint_as_float(h << 16),
                                            d1 - __uint_as_float(h & 0xFFFF0000u));
            }
            ps_store_row<1>(ps, r, cb + 32 * ch, dw);
          }
          publish(C::kDsFull);
          if (!wait_all(C::kDsDone, k & 1u)) return;
          ps_store_row<NCH>(ps, r, cb, dl);
          publish(C::kDsFull);
        }
      };
      if (ti.len_a == kBlk)
        run(std::integral_constant<int, 2>{}, wq >= 2 ? kBlk : 0);
      else
        run(std::integral_constant<int, 4>{}, 0);
      if (abort_now) break;
      if (want_db) {
        // all four warps have added this tile; each then flushes 32 entries to
        // the table (entry clamp(query - key + max_rel - 1)) and clears them
        warp_arrive(bar(C::kDbAcc), lane);
        bool ok = mbar_wait(bar(C::kDbAcc), n_db & 1u, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) { if (lane == 0) fail(); break; }
        const int e = 32 * wq + lane;
        if (e < 2 * kBlk - 1) {
          const float v = dwin[e];
          if (v != 0.0f)
            atomicAdd(p.dbias + static_cast<long long>(head) * (2 * p.max_rel - 1) +
                          min(max(e - (kBlk - 1) + p.max_rel - 1, 0), 2 * p.max_rel - 2),
                      v);
          dwin[e] = 0.0f;
        }
        warp_arrive(bar(C::kDbFree), lane);
        ok = mbar_wait(bar(C::kDbFree), n_db & 1u, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) { if (lane == 0) fail(); break; }
        ++n_db;
      }
    }
  } else if (warp < kBwdEpi0 + 4) {
    // ------------------------------------------------------------ epilogue warps
    // A full softmax tile's gradients leave through the P / dS buffer (free once
    // dK and dQ are done) and TMA stores, one gradient at a time: coalesced
    // writes instead of one 256-byte row per thread, which saturate the SM's
    // load/store pipe that the activation warps also use.  A partial tile's
    // rows are stored directly (a tile store would write into the next tile's
    // rows).
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // tile row: query (dQ) or key (dK, dV)
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    uint8_t* ps = gbase + C::kPS;
    const uint32_t col[3] = {kColDP, kColDK, kColDV};
    const float mul[3] = {p.scale, p.scale, 1.0f};
    const CUtensorMap* maps[3] = {&tmap_dq, &tmap_dk, &tmap_dv};
    // theta_c = base^(-2c/d) = exp2(c * rope_k)
    const float rope_k = p.rope_base > 0.0f ? -2.0f * log2f(p.rope_base) / D : 0.0f;
    // Gradient `which` (dQ, dK, dV) of this row, channels [32j, 32j+32) and the
    // matching half [d/2 + 32j, ...), scaled, as bf16 pairs.  With a rotary
    // embedding, dQ and dK go back through it here, in fp32: the pair (c, c+d/2)
    // is rotated by -pos * theta_c (the rotary backward, fused).
    auto grad_pair = [&](int which, int j, int pos, uint32_t (&pk)[2][16]) {
      uint32_t v1[32], v2[32];
      tmem_ld32(tmem + lane_off + col[which] + 32 * j, v1);
      tmem_ld32(tmem + lane_off + col[which] + 32 * j + D / 2, v2);
      const bool rot = p.rope_base > 0.0f && which < 2;
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        float a[2], b[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float g1 = __uint_as_float(v1[i + e]) * mul[which];
          float g2 = __uint_as_float(v2[i + e]) * mul[which];
          if (rot) {
            float sn, cs;
            sincosf(static_cast<float>(pos) * exp2f(static_cast<float>(32 * j + i + e) * rope_k), &sn, &cs);
            const float r1 = fmaf(g1, cs, g2 * sn);
            const float r2 = fmaf(g2, cs, -g1 * sn);
            g1 = r1;
            g2 = r2;
          }
          a[e] = g1;
          b[e] = g2;
        }
        pk[0][i / 2] = pack_bf16x2(a[0], a[1]);
        pk[1][i / 2] = pack_bf16x2(b[0], b[1]);
      }
    };
    uint32_t n_round = 0;
    bool stores_pending = false;
    for (int k = 0;; ++k) {
      const int item = item_of(k);
      if (item >= n_items) break;
      const int head = item % p.H;
      const TileInfo ti = load_tile(p.tiles, item / p.H);
      bool w = mbar_wait(bar(C::kGradFull), k & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      tc_fence_after();
      const int pos = ti.pos(r);
      // (GDPA tiles pass P and dS through the buffer twice each: there the
      // activation warps need it back sooner than a staged epilogue returns it)
      if (!kSoftmax || ti.rows < kTileRows) {
        if (r == 0) mbar_arrive(bar(C::kPsFree));  // the buffer is not needed here
        const long long g = (static_cast<long long>(ti.row0 + r) * p.H + head) * D;
        __nv_bfloat16* const dst[3] = {p.dq + g, p.dk + g, p.dv + g};
#pragma unroll
        for (int which = 0; which < 3; ++which) {
#pragma unroll 1
          for (int j = 0; j < D / 64; ++j) {
            uint32_t pk[2][16];
            grad_pair(which, j, pos, pk);
            if (r < ti.rows) {
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                uint4* out = reinterpret_cast<uint4*>(dst[which] + 32 * j + (D / 2) * h);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  out[q] = make_uint4(pk[h][4 * q], pk[h][4 * q + 1], pk[h][4 * q + 2], pk[h][4 * q + 3]);
              }
            }
          }
        }
        tc_fence_before();
        warp_arrive(bar(C::kEpiDone), lane);
        continue;
      }
      bool ok = true;
#pragma unroll 1
      for (int which = 0; which < 3 && ok; ++which) {
        // the previous gradient's store has finished reading the buffer
        if (n_round > 0) {
          w = mbar_wait(bar(C::kEpiFree), (n_round - 1) & 1u, abort_flag);
          if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); ok = false; break; }
        }
#pragma unroll 1
        for (int j = 0; j < D / 64; ++j) {
          uint32_t pk[2][16];
          grad_pair(which, j, pos, pk);
          ps_store_row<1>(ps, r, 32 * j, pk[0]);  // [channel atom][row][64 channels], swizzled
          ps_store_row<1>(ps, r, 32 * j + D / 2, pk[1]);
        }
        if (which == 2) {
          tc_fence_before();
          warp_arrive(bar(C::kEpiDone), lane);  // TMEM of this tile is read
        }
        fence_proxy_async_smem();
        warp_arrive(bar(C::kEpiStaged), lane);
        if (r == 0) {
          if (!mbar_wait(bar(C::kEpiStaged), n_round & 1u, abort_flag)) {
            fail();
          } else {
#pragma unroll
            for (int x = 0; x < D; x += 64)
              tma_store_3d(maps[which], smem_u32(ps) + (x / 64) * C::kAtom, x, head, ti.row0);
            bulk_commit_group();
            stores_pending = true;
          }
          bulk_wait_group_read<0>();
          mbar_arrive(bar(C::kEpiFree));
          if (which == 2) mbar_arrive(bar(C::kPsFree));
        }
        ++n_round;
      }
      if (!ok) break;
    }
    if (r == 0 && stores_pending) bulk_wait_group_all();  // global writes done before exit
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int ACT, bool kDBias, bool kDense>
cudaError_t launch_bwd_db(const BlockParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                          const CUtensorMap& tdk, const CUtensorMap& tdv, int grid, cudaStream_t s) {
  constexpr int smem = BbCfg<D>::kSmemBytes;
  static_assert(smem <= 232448, "shared memory budget");
  cudaError_t e = cudaFuncSetAttribute(block_bwd_kernel<D, ACT, kDBias, kDense>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  block_bwd_kernel<D, ACT, kDBias, kDense><<<grid, kBwdThreads, smem, s>>>(tq, tk, tv, tdo, tdq, tdk, tdv, p);
  return cudaGetLastError();
}


template <int D, bool kDBias, bool kDense>
cudaError_t launch_bwd_d(const BlockParams& p, int act, const CUtensorMap* m, int grid,
                         cudaStream_t s) {
  switch (act) {
    case GDPA_ACT_SOFTMAX:
      return launch_bwd_db<D, GDPA_ACT_SOFTMAX, kDBias, kDense>(p, m[0], m[1], m[2], m[3], m[4], m[5], m[6],
                                                 grid, s);
    case GDPA_ACT_SILU:
      return launch_bwd_db<D, GDPA_ACT_SILU, kDBias, kDense>(p, m[0], m[1], m[2], m[3], m[4], m[5], m[6],
                                                 grid, s);
    case GDPA_ACT_GELU_TANH:
      return launch_bwd_db<D, GDPA_ACT_GELU_TANH, kDBias, kDense>(p, m[0], m[1], m[2], m[3], m[4], m[5], m[6],
                                                 grid, s);
    case GDPA_ACT_GELU_ERF:
      return launch_bwd_db<D, GDPA_ACT_GELU_ERF, kDBias, kDense>(p, m[0], m[1], m[2], m[3], m[4], m[5], m[6],
                                                 grid, s);
    default:
      return launch_bwd_db<D, GDPA_ACT_IDENTITY, kDBias, kDense>(p, m[0], m[1], m[2], m[3], m[4], m[5], m[6],
                                                 grid, s);
  }
}

}  // namespace
}  // namespace gdpa
