// MXFP8 backward of jagged softmax attention (JFA), sm_103a.
//
// "GEM Training ..." low-precision paragraph: attention with end-to-end MXFP8
// block-scaled MMA in the forward and in the backward pass.  All five
// products of the softmax backward run on the block-scaled tensor cores
// (tcgen05.mma kind::mxf8f6f4.block_scale): E4M3 operands, one E8M0 scale
// per 32 elements of the contraction, fp32 accumulation.  Each operand is
// quantised along its own product's contraction axis:
//   S^T  = K Q^T       K, Q along channels
//   dP^T = V dO^T      V, dO along channels
//   dV  += P^T dO      P^T (in TMEM) along queries, dO along tokens
//   dK  += dS^T Q      dS^T along queries, Q along tokens
//   dQ^T = K^T dS^T    K along tokens, dS along keys
// P and dS are made here from S and dP (fp32) and rounded to E4M3 in blocks
// of 32 keys x 32 queries that share one scale, the smallest power of two
// that keeps every element at or below 448.  A 32 x 32 block contains a
// 32-element block along either axis, so one set of codes serves the dK
// product (contracted over queries) and the dQ product (over keys).
//
// Structure: the bf16 softmax backward's (persistent CTAs over the
// cost-sorted list of 128-key blocks of one (sample, head); the sample's
// queries stream past the block; everything transposed so that TMEM lanes
// are key rows), with 64-query tiles so that the scale factors fit in TMEM:
//   [0,64)    S^T, then the E4M3 codes of P^T: queries 32g..32g+31 in
//             columns 32g..32g+7 (four codes per column)
//   [64,128)  dP^T, later dQ^T (lanes = channels)
//   [128,208) scale-factor sets, 8 columns apart
//   [256,384) dV, [384,512) dK
// The word of operand row r (a row of A, or of B^T) sits in column set +
// r/32, lane r%32, and its byte k scales that row's 32 elements of k-step k.
// Scale words go from shared memory into TMEM with tcgen05.cp (32x128b,
// warpx4: 32 rows of 16 bytes, copied into every lane quarter), issued by
// the MMA thread in order with its MMAs.
//
// Warp roles (512 threads): warps 0-3 / 4-7 activation for query columns
// [0,32) / [32,64) of a tile (P, dS, their codes and block scales); warps
// 8-11 dQ group (dQ^T drain into the fp32 accumulator, dK/dV epilogue); warp
// 12 producer (TMA of the E4M3 codes, the operands' scale words, lse, D and
// bias values); warp 13 MMA issuer; warp 14 adds each tile's bias-table
// gradient (kDBias with the table) to the table; warp 15 idle.  kDense reads a
// dense jagged bias instead (a key row's lanes are consecutive keys, so each
// query column's load is one row segment), and with kDBias adds each pair's
// fp32 dS to its entry of the bias's gradient.  With rope_base > 0 the dK
// epilogue rotates the rows back through the rotary embedding (dQ is rotated
// in the accumulator's conversion).
//
// The kernel and its launch templates are compiled from bwd_mx.cu (no dense
// bias) and bwd_mx_dense.cu (a dense jagged bias).
#pragma once
#include <type_traits>

#include "common.cuh"
#include "mx.cuh"

namespace gdpa {
namespace {

using namespace ptx;
using mx::e4m3x4;
using mx::e8m0_nosat;

constexpr int kThreads = 512;
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int kActWarps = 8;
constexpr int kD = 128;
constexpr int kQRows = kBwdMxQRows;  // 64 queries per tile
constexpr int kKRows = kBwdKvRows;   // 128 keys per item
constexpr int kDqChunk = 16;         // queries per dQ reduce box
constexpr float kLog2e = 1.4426950408889634f;

// shared-memory staging sets of scale words (32 lanes x 16 bytes each)
enum SfSmem { kSmKd, kSmVd, kSmKt, kSmQd0, kSmQd1, kSmQt0, kSmQt1, kSmOd, kSmOt, kSmP, kSmDsR,
              kSmDsC, kNumSmSf };
// TMEM scale-factor sets
enum SfTmem { kTmKd, kTmVd, kTmKt, kTmQd, kTmQt, kTmOd, kTmOt, kTmP, kTmDsR, kTmDsC };

constexpr uint32_t kColS = 0, kColDP = 64, kColDV = 256, kColDK = 384;
__device__ __forceinline__ uint32_t col_sf(int set) { return 128u + 8u * set; }

struct Cfg {
  static constexpr int kKvBytes = kKRows * kD;  // 16 KB of E4M3 codes
  static constexpr int kQBytes = kQRows * kD;   // 8 KB
  static constexpr int kQStages = 2;
  static constexpr int kKd = 0;
  static constexpr int kKt = kKvBytes;
  static constexpr int kVd = 2 * kKvBytes;
  static constexpr int kQd = 3 * kKvBytes;                     // + s * kQBytes
  static constexpr int kQt = kQd + kQStages * kQBytes;         // + s * kQBytes
  static constexpr int kOd = kQt + kQStages * kQBytes;
  static constexpr int kOt = kOd + kQBytes;
  static constexpr int kDsT = kOt + kQBytes;         // dS^T codes [key row][128 B], queries in bytes 0..63
  static constexpr int kDsQ = kDsT + kKRows * 128;   // dS codes [query row][128 keys]
  // per Q stage: -lse*log2e [64], -D [64], then the bias window (191 entries,
  // times log2e) in two copies shifted by 0 and 1 entries, kBiasCopy floats
  // apart (every key row finds its entries 8-byte aligned in one copy; with a
  // stride of 14 mod 32 the 64-bit loads of a half-warp hit every bank once)
  static constexpr int kBiasCopy = 206;
  static constexpr int kStatFloats = 2 * kQRows + 2 * kBiasCopy + 4;  // 16-byte multiple
  static constexpr int kStats = kDsQ + kQRows * 128;
  static constexpr int kDqStageBytes = kDqChunk * kD * 4;     // [16 queries][128] fp32
  static constexpr int kDqStage = kStats + kQStages * kStatFloats * 4;
  static constexpr int kSfBytes = 512;
  static constexpr int kSf = kDqStage + 2 * kDqStageBytes;
  // bias-table gradient: per tile, dS summed along its 191 diagonals (two
  // buffers of 192 floats, then {first diagonal, head})
  static constexpr int kDbBuf = 192 * 4 + 16;
  static constexpr int kDb = kSf + kNumSmSf * kSfBytes;
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
  static constexpr int kGroupOk = kAbort + 4;  // int[4]: dQ-group vote on a wait's result
  static constexpr int kUsed = kGroupOk + 16;
  static constexpr int kSmemBytes = kUsed + 1024;
};
static_assert(Cfg::kDsT % 1024 == 0 && Cfg::kDsQ % 1024 == 0 && Cfg::kQd % 1024 == 0,
              "swizzled operand tiles need 1024-byte alignment");
static_assert((Cfg::kStatFloats * 4) % 16 == 0 && Cfg::kSf % 16 == 0, "alignment");
static_assert(Cfg::kSmemBytes <= 232448, "shared memory budget");

// Copies 32 rows x 16 bytes of shared memory (described by `desc`) into TMEM
// lanes 0..31 of every lane quarter, columns taddr..taddr+3.
__device__ __forceinline__ void tmem_cp_sf(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc)
               : "memory");
}

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
  uint32_t r;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}
// Largest |x| of 32 values (pairwise tree).
__device__ __forceinline__ float amax32(const float (&x)[32]) {
  float m[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) m[i] = fmaxf(fabsf(x[2 * i]), fabsf(x[2 * i + 1]));
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) m[i] = fmaxf(m[i], m[i + w]);
  return m[0];
}
// E4M3 codes of x * inv, four per word (packed fp32x2 scaling).
__device__ __forceinline__ void quant32(const float (&x)[32], float inv, uint32_t (&pk)[8]) {
  const float2 s2 = make_float2(inv, inv), z2 = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float2 a = fma_f32x2(make_float2(x[4 * q], x[4 * q + 1]), s2, z2);
    const float2 b = fma_f32x2(make_float2(x[4 * q + 2], x[4 * q + 3]), s2, z2);
    pk[q] = e4m3x4(a.x, a.y, b.x, b.y);
  }
}
// 4 x 4 byte transpose across the lanes of each aligned group of four: lane r
// holds bytes (query c = 0..3) of key r in `x`; returns bytes (key 0..3) of
// query r.
__device__ __forceinline__ uint32_t transpose4x4_bytes(uint32_t x, int lane) {
  uint32_t p = __shfl_xor_sync(0xffffffffu, x, 1);
  uint32_t t = __byte_perm(x, p, (lane & 1) ? 0x3715u : 0x6240u);
  p = __shfl_xor_sync(0xffffffffu, t, 2);
  return __byte_perm(t, p, (lane & 2) ? 0x3276u : 0x5410u);
}

struct MxItem {
  int b, head, kb;
  int q0, k0, Lq, Lkv;
  int qt0;  // first query tile (64 rows) visited
  int nq;   // number of query tiles visited
};

template <bool kBand>
__device__ __forceinline__ MxItem decode_mx(int2 it, const BwdParams& p) {
  MxItem r;
  r.b = it.x;
  r.head = item_head(it);
  r.kb = item_block(it);
  r.q0 = p.qo[r.b];
  r.Lq = p.qo[r.b + 1] - r.q0;
  r.k0 = p.ko[r.b];
  r.Lkv = p.ko[r.b + 1] - r.k0;
  const int kb0 = r.kb * kKRows;
  if (kBand) {
    const int qb = band_query_begin(kb0, p.causal, p.window);
    const int qe = band_query_end(min(r.Lkv, kb0 + kKRows) - 1, p.window, r.Lq);
    r.qt0 = qb / kQRows;
    r.nq = max(0, (qe + kQRows - 1) / kQRows - r.qt0);
  } else {
    r.qt0 = p.causal ? kb0 / kQRows : 0;  // queries before the block's first key see none of it
    const int rows = r.Lq - r.qt0 * kQRows;
    r.nq = rows > 0 ? (rows + kQRows - 1) / kQRows : 0;
  }
  return r;
}

template <bool kBand, bool kDBias, bool kRope, bool kDense>
__global__ void __launch_bounds__(kThreads, 1)
bwd_mx_kernel(const __grid_constant__ CUtensorMap tmap_qd, const __grid_constant__ CUtensorMap tmap_qt,
              const __grid_constant__ CUtensorMap tmap_dod, const __grid_constant__ CUtensorMap tmap_dot,
              const __grid_constant__ CUtensorMap tmap_kd, const __grid_constant__ CUtensorMap tmap_kt,
              const __grid_constant__ CUtensorMap tmap_vd, const __grid_constant__ CUtensorMap tmap_dq,
              const BwdParams p, const BwdMxOperands mx) {
  using C = Cfg;
  constexpr bool kTableGrad = kDBias && !kDense;  // the table's gradient (warp 14)
  constexpr bool kDenseGrad = kDBias && kDense;   // the dense bias's gradient
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  auto bar = [&](int i) -> uint32_t { return sbase + C::kBar + 8u * i; };
  int2* item_slot = reinterpret_cast<int2*>(gbase + C::kItemSlots);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kAbort);
  float* stats = reinterpret_cast<float*>(gbase + C::kStats);
  uint8_t* sf_smem = gbase + C::kSf;

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
    mbar_init(bar(C::kPFull), kActWarps);  // one arrival per warp (warp_arrive)
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
  // scale bytes that no product reads (k-steps past a tile) are still copied:
  // give them a defined value
  for (int i = threadIdx.x; i < kNumSmSf * C::kSfBytes / 4; i += kThreads)
    reinterpret_cast<uint32_t*>(sf_smem)[i] = 0x7F7F7F7Fu;
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&tmap_qd);
    prefetch_tmap(&tmap_qt);
    prefetch_tmap(&tmap_dod);
    prefetch_tmap(&tmap_dot);
    prefetch_tmap(&tmap_kd);
    prefetch_tmap(&tmap_kt);
    prefetch_tmap(&tmap_vd);
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
    const int H = p.H;
    uint32_t it = 0, g = 0, kvi = 0, oi = 0;
    bool kv_inflight = false, o_inflight = false;
    uint32_t q_inflight = 0, last_g[C::kQStages] = {};
    bool ok = true;
    // lane's 16 bytes of a staging set: the words of rows lane, 32 + lane, 64 + lane, 96 + lane
    auto sf_put = [&](int set, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3) {
      *reinterpret_cast<uint4*>(sf_smem + set * C::kSfBytes + lane * 16) = make_uint4(w0, w1, w2, w3);
    };
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
      const MxItem in = decode_mx<kBand>(item, p);
      if (in.nq == 0) continue;
      const int head = in.head;
      // channel-scale word (4 scales of d = 128) of row `row`; scale 1 past the tensor
      auto ch_word = [&](const uint8_t* sc, long long row, long long T) -> uint32_t {
        return row < T ? __ldg(reinterpret_cast<const uint32_t*>(sc) + row * H + head) : 0x7F7F7F7Fu;
      };
      // token-scale byte of channel n for 32-token block r of a sample whose
      // first block is scale row row0; scale 1 for a block past the sample
      auto tok_byte = [&](const uint8_t* sc, long long row0, int r, int L, int n) -> uint32_t {
        return 32 * r < L ? static_cast<uint32_t>(__ldg(sc + ((row0 + r) * H + head) * kD + n)) : 127u;
      };
      w = mbar_wait(bar(C::kKvEmpty), (kvi & 1u) ^ 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      ++kvi;
      const int kloc = in.kb * kKRows;
      const int krow = in.k0 + kloc;
      {
        const long long krow0 = static_cast<long long>(in.b) + in.k0 / 32;
        uint32_t wk[4], wv[4], wt[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          wk[c] = ch_word(mx.kd_sc, static_cast<long long>(krow) + 32 * c + lane, p.Tkv);
          wv[c] = ch_word(mx.vd_sc, static_cast<long long>(krow) + 32 * c + lane, p.Tkv);
          uint32_t t = 0;
#pragma unroll
          for (int kbk = 0; kbk < 4; ++kbk)
            t |= tok_byte(mx.kt_sc, krow0, kloc / 32 + kbk, in.Lkv, 32 * c + lane) << (8 * kbk);
          wt[c] = t;
        }
        sf_put(kSmKd, wk[0], wk[1], wk[2], wk[3]);
        sf_put(kSmVd, wv[0], wv[1], wv[2], wv[3]);
        sf_put(kSmKt, wt[0], wt[1], wt[2], wt[3]);
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(C::kKvFull), 3 * C::kKvBytes);
        tma_load_3d(sbase + C::kKd, &tmap_kd, bar(C::kKvFull), 0, head, krow);
        tma_load_3d(sbase + C::kKt, &tmap_kt, bar(C::kKvFull), 0, head, krow);
        tma_load_3d(sbase + C::kVd, &tmap_vd, bar(C::kKvFull), 0, head, krow);
        kv_inflight = true;
      }
      // Per-lane values of one query tile, fetched one tile ahead: -lse*log2e
      // and -D for columns lane + 32k, bias-window entries lane + 32k.
      const int rel_w = 2 * p.max_rel - 1;
      const float* brow = p.bias_table ? p.bias_table + static_cast<long long>(head) * rel_w : nullptr;
      constexpr int kWin = kQRows + kKRows - 1;  // 191 relative positions
      auto fetch = [&](int t, float (&v)[10]) {
        const int qloc = (in.qt0 + t) * kQRows;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int ql = qloc + lane + 32 * k;
          float l2 = 0.0f, dd = 0.0f;
          if (ql < in.Lq) {
            const long long gi = static_cast<long long>(head) * p.Tq + in.q0 + ql;
            l2 = -__ldg(p.lse + gi) * kLog2e;  // stored negated: added, not subtracted
            dd = -__ldg(p.delta + gi);
          }
          v[2 * k] = l2;
          v[2 * k + 1] = dd;
        }
        // bias(i - j) for query column c and key row jj of the tile is window
        // entry c - jj + 127
        const int w0 = qloc - kloc - (kKRows - 1) + p.max_rel - 1;
#pragma unroll
        for (int k = 0; k < 6; ++k) {
          const int e = lane + 32 * k;
          v[4 + k] = (brow != nullptr && e < kWin)
                         ? __ldg(brow + min(max(w0 + e, 0), rel_w - 1)) * kLog2e
                         : 0.0f;
        }
      };
      const long long qrow0 = static_cast<long long>(in.b) + in.q0 / 32;  // first token-scale row
      float cur[10];
      fetch(0, cur);
      for (int t = 0; t < in.nq; ++t, ++g) {
        const uint32_t s = g % C::kQStages;
        const uint32_t ph = (g / C::kQStages) & 1u;
        const int qloc = (in.qt0 + t) * kQRows;
        const long long qrow = static_cast<long long>(in.q0) + qloc;
        w = mbar_wait(bar(C::kQEmpty + s), ph ^ 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { ok = false; if (lane == 0) fail(); break; }
        float* st = stats + s * C::kStatFloats;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          st[lane + 32 * k] = cur[2 * k];
          st[kQRows + lane + 32 * k] = cur[2 * k + 1];
        }
        if (brow != nullptr) {
#pragma unroll
          for (int k = 0; k < 6; ++k)
            if (lane + 32 * k < kWin) {
#pragma unroll
              for (int cp = 0; cp < 2; ++cp)  // copy cp holds entry e at position e + cp
                st[2 * kQRows + cp * C::kBiasCopy + cp + lane + 32 * k] = cur[4 + k];
            }
        }
        // scale words of Q (along channels: rows = the tile's 64 queries;
        // along tokens: rows = channels, bytes = the tile's two query blocks)
        {
          uint32_t wt[4];
#pragma unroll
          for (int c = 0; c < 4; ++c)
            wt[c] = tok_byte(mx.qt_sc, qrow0, qloc / 32, in.Lq, 32 * c + lane) |
                    (tok_byte(mx.qt_sc, qrow0, qloc / 32 + 1, in.Lq, 32 * c + lane) << 8) |
                    0x7F7F0000u;
          sf_put(kSmQd0 + s, ch_word(mx.qd_sc, qrow + lane, p.Tq),
                 ch_word(mx.qd_sc, qrow + 32 + lane, p.Tq), 0x7F7F7F7Fu, 0x7F7F7F7Fu);
          sf_put(kSmQt0 + s, wt[0], wt[1], wt[2], wt[3]);
        }
        float nxt[10];
        if (t + 1 < in.nq) {
          fetch(t + 1, nxt);
        } else {
#pragma unroll
          for (int k = 0; k < 10; ++k) nxt[k] = 0.0f;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(C::kQFull + s), 2 * C::kQBytes);
          tma_load_3d(sbase + C::kQd + s * C::kQBytes, &tmap_qd, bar(C::kQFull + s), 0, head,
                      static_cast<int>(qrow));
          tma_load_3d(sbase + C::kQt + s * C::kQBytes, &tmap_qt, bar(C::kQFull + s), 0, head,
                      static_cast<int>(qrow));
          q_inflight |= 1u << s;
          last_g[s] = g;
        }
        // dO of this tile: its single buffer frees once dV of the previous tile is done
        w = mbar_wait(bar(C::kOEmpty), (oi & 1u) ^ 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { ok = false; if (lane == 0) fail(); break; }
        ++oi;
        {
          uint32_t wt[4];
#pragma unroll
          for (int c = 0; c < 4; ++c)
            wt[c] = tok_byte(mx.dot_sc, qrow0, qloc / 32, in.Lq, 32 * c + lane) |
                    (tok_byte(mx.dot_sc, qrow0, qloc / 32 + 1, in.Lq, 32 * c + lane) << 8) |
                    0x7F7F0000u;
          sf_put(kSmOd, ch_word(mx.dod_sc, qrow + lane, p.Tq),
                 ch_word(mx.dod_sc, qrow + 32 + lane, p.Tq), 0x7F7F7F7Fu, 0x7F7F7F7Fu);
          sf_put(kSmOt, wt[0], wt[1], wt[2], wt[3]);
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(C::kOFull), 2 * C::kQBytes);
          tma_load_3d(sbase + C::kOd, &tmap_dod, bar(C::kOFull), 0, head, static_cast<int>(qrow));
          tma_load_3d(sbase + C::kOt, &tmap_dot, bar(C::kOFull), 0, head, static_cast<int>(qrow));
          o_inflight = true;
        }
#pragma unroll
        for (int k = 0; k < 10; ++k) cur[k] = nxt[k];
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
    if (lane == 0) {
      // Descriptors at each operand's first byte (128-byte swizzle, 8-row
      // groups 1024 bytes apart); k-steps and stages go into the start
      // address field (see dadd).  K-major k-steps advance 32 bytes inside
      // the swizzled rows, MN-major k-steps 32 rows (4096 bytes).
      const uint64_t dsc_kd = sdesc(sbase + C::kKd, 0, 1024, kSwizzle128B);   // A of S^T
      const uint64_t dsc_vd = sdesc(sbase + C::kVd, 0, 1024, kSwizzle128B);   // A of dP^T
      const uint64_t dsc_kt = sdesc(sbase + C::kKt, 0, 1024, kSwizzle128B);   // A of dQ^T (MN-major)
      const uint64_t dsc_qd = sdesc(sbase + C::kQd, 0, 1024, kSwizzle128B);   // B of S^T
      const uint64_t dsc_qt = sdesc(sbase + C::kQt, 0, 1024, kSwizzle128B);   // B of dK (MN-major)
      const uint64_t dsc_od = sdesc(sbase + C::kOd, 0, 1024, kSwizzle128B);   // B of dP^T
      const uint64_t dsc_ot = sdesc(sbase + C::kOt, 0, 1024, kSwizzle128B);   // B of dV (MN-major)
      const uint64_t dsc_dst = sdesc(sbase + C::kDsT, 0, 1024, kSwizzle128B); // A of dK
      const uint64_t dsc_dsq = sdesc(sbase + C::kDsQ, 0, 1024, kSwizzle128B); // B of dQ^T
      // scale staging: 32 rows of 16 bytes, no swizzle, 8-row groups 128 bytes apart
      const uint64_t dsc_sf = sdesc(sbase + C::kSf, 128, 128, 0);
      auto cp_sf = [&](int sm, int tm) {
        tmem_cp_sf(tmem + col_sf(tm), dadd(dsc_sf, sm * C::kSfBytes));
      };
      uint32_t it = 0, g = 0, kvi = 0, oc = 0, pc = 0, qe = 0, dkvc = 0;
      bool dq_pending = false, issued_any = false;
      bool ok = true;
      auto issue_s = [&](uint32_t s) {  // S^T = K Q^T
        cp_sf(kSmQd0 + s, kTmQd);
        const uint64_t qb = dadd(dsc_qd, s * C::kQBytes);
#pragma unroll
        for (int ks = 0; ks < kD / 32; ++ks)
          mx::mma_ss(tmem + kColS, dadd(dsc_kd, ks * 32), dadd(qb, ks * 32),
                    mx::idesc(kQRows, false, false, ks), tmem + col_sf(kTmKd), tmem + col_sf(kTmQd),
                    ks > 0 ? 1u : 0u);
        mma_commit(bar(C::kSFull));
        issued_any = true;
      };
      // dP^T = V dO^T into the dP columns, once dO has landed and the dQ group
      // has read the previous dQ^T out of the same columns.
      auto issue_dp = [&]() -> bool {
        if (!mbar_wait(bar(C::kOFull), oc & 1u, abort_flag)) return false;
        ++oc;
        if (dq_pending) {
          if (!mbar_wait(bar(C::kDqEmpty), qe & 1u, abort_flag)) return false;
          ++qe;
          dq_pending = false;
        }
        tc_fence_after();
        cp_sf(kSmOd, kTmOd);
#pragma unroll
        for (int ks = 0; ks < kD / 32; ++ks)
          mx::mma_ss(tmem + kColDP, dadd(dsc_vd, ks * 32), dadd(dsc_od, ks * 32),
                    mx::idesc(kQRows, false, false, ks), tmem + col_sf(kTmVd), tmem + col_sf(kTmOd),
                    ks > 0 ? 1u : 0u);
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
        const MxItem in = decode_mx<kBand>(item, p);
        if (in.nq == 0) continue;
        if (!mbar_wait(bar(C::kKvFull), kvi & 1u, abort_flag)) { fail(); break; }
        ++kvi;
        tc_fence_after();
        cp_sf(kSmKd, kTmKd);
        cp_sf(kSmVd, kTmVd);
        cp_sf(kSmKt, kTmKt);
        {
          const uint32_t s0 = g % C::kQStages;
          if (!mbar_wait(bar(C::kQFull + s0), (g / C::kQStages) & 1u, abort_flag)) { fail(); break; }
          tc_fence_after();
          issue_s(s0);
          if (!issue_dp()) { fail(); break; }
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
          // dV += P^T dO   (A = P^T codes in TMEM, B = dO MN-major)
          cp_sf(kSmP, kTmP);
          cp_sf(kSmOt, kTmOt);
#pragma unroll
          for (int ks = 0; ks < kQRows / 32; ++ks)
            mx::mma_ts(tmem + kColDV, tmem + kColS + 32 * ks, dadd(dsc_ot, ks * 4096),
                      mx::idesc(kD, false, true, ks), tmem + col_sf(kTmP), tmem + col_sf(kTmOt),
                      (t == 0 && ks == 0) ? 0u : 1u);
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
          // dK += dS^T Q   (A = dS^T K-major, B = Q MN-major)
          cp_sf(kSmDsR, kTmDsR);
          cp_sf(kSmQt0 + s, kTmQt);
          const uint64_t qtb = dadd(dsc_qt, s * C::kQBytes);
#pragma unroll
          for (int ks = 0; ks < kQRows / 32; ++ks)
            mx::mma_ss(tmem + kColDK, dadd(dsc_dst, ks * 32), dadd(qtb, ks * 4096),
                      mx::idesc(kD, false, true, ks), tmem + col_sf(kTmDsR), tmem + col_sf(kTmQt),
                      (t == 0 && ks == 0) ? 0u : 1u);
          mma_commit(bar(C::kQEmpty + s));
          // dQ^T = K^T dS^T into the dP columns (A = K MN-major, B = dS K-major)
          cp_sf(kSmDsC, kTmDsC);
#pragma unroll
          for (int ks = 0; ks < kKRows / 32; ++ks)
            mx::mma_ss(tmem + kColDP, dadd(dsc_kt, ks * 4096), dadd(dsc_dsq, ks * 32),
                      mx::idesc(kQRows, true, false, ks), tmem + col_sf(kTmKt), tmem + col_sf(kTmDsC),
                      ks > 0 ? 1u : 0u);
          mma_commit(bar(C::kDqFull));
          dq_pending = true;
          if (t + 1 < in.nq && !issue_dp()) { ok = false; fail(); break; }
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
    const int grp = warp >> 2;           // query columns [32 grp, 32 grp + 32) of a tile
    const int j = wq * 32 + lane;        // key row within the block = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const float c_s = p.scale * kLog2e;
    const bool has_bias = p.bias_table != nullptr;
    uint8_t* sf_p = sf_smem + kSmP * C::kSfBytes;
    uint8_t* sf_dsr = sf_smem + kSmDsR * C::kSfBytes;
    uint8_t* sf_dsc = sf_smem + kSmDsC * C::kSfBytes;
    uint32_t it = 0, g = 0;
    while (true) {
      const uint32_t slot = it & 1u;
      bool w = mbar_wait(bar(C::kItemFull + slot), (it >> 1) & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      const int2 item = item_slot[slot];
      warp_arrive(bar(C::kItemEmpty + slot), lane);
      ++it;
      if (item.x < 0) break;
      const MxItem in = decode_mx<kBand>(item, p);
      const int kb0 = in.kb * kKRows;   // first local key row of the block
      const int jl = kb0 + j;           // this thread's local key row
      // queries that see this key: [vis_lo, vis_hi) (none for a key past the sample)
      const int vis_lo = band_query_begin(jl, p.causal, p.window);
      const int vis_hi = jl < in.Lkv ? band_query_end(jl, p.window, in.Lq) : 0;
      // query tiles inside [full_lo, full_hi) pair with every key of a full block
      const int full_lo = band_query_begin(kb0 + kKRows - 1, p.causal, p.window);
      const int full_hi = kb0 + kKRows <= in.Lkv ? band_query_end(kb0, p.window, in.Lq) : 0;
      // dense bias of this key for query i: dcol[i * Lkv] (a key past the
      // sample reads none); its gradient at the same place of p.dbias
      const float* dcol = (kDense && jl < in.Lkv)
                              ? p.bias_dense + p.bias_off[in.b] +
                                    static_cast<long long>(in.head) * in.Lq * in.Lkv + jl
                              : nullptr;
      float* gcol = (kDenseGrad && dcol != nullptr) ? p.dbias + (dcol - p.bias_dense) : nullptr;
      bool abort_now = false;
      for (int t = 0; t < in.nq; ++t, ++g) {
        const uint32_t s = g % C::kQStages;
        w = mbar_wait(bar(C::kQFull + s), (g / C::kQStages) & 1u, abort_flag);
        w = w && mbar_wait(bar(C::kSFull), g & 1u, abort_flag);
        // the diagonal buffer of this tile was flushed two tiles ago
        if (kTableGrad) w = w && mbar_wait(bar(C::kDbFree + (g & 1u)), ((g >> 1) & 1u) ^ 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); abort_now = true; break; }
        tc_fence_after();
        const float* st = stats + s * C::kStatFloats;
        const float4* st4 = reinterpret_cast<const float4*>(st);  // 16-byte aligned
        // bias(query c, key j) * log2e is window entry c - j + 127; the copy
        // shifted by (j + 1) % 2 holds it 8-byte aligned for even c
        const int cpy = (j + 1) & 1;
        const float* bwin = st + 2 * kQRows + cpy * C::kBiasCopy + cpy + (kKRows - 1) - j;
        const int qloc = (in.qt0 + t) * kQRows;
        const bool full = qloc >= full_lo && qloc + kQRows <= full_hi;
        int c_lo = 0, c_hi = kQRows;  // valid query columns: c_lo <= c < c_hi
        if (!full) {
          c_hi = min(kQRows, vis_hi - qloc);
          c_lo = max(0, vis_lo - qloc);
        }
        const int c0 = 32 * grp;
        // Phase 1: P^T = exp2(S^T scale log2e + bias log2e - lse log2e) (fp32,
        // kept for phase 2); E4M3 codes into the group's first 8 S columns.
        float pv[32];
        {
          uint32_t sr[32];
          tmem_ld32(tmem + lane_off + kColS + c0, sr);
          auto body = [&](auto masked, auto biased) {
            constexpr bool kMask = decltype(masked)::value;
            constexpr bool kBias = decltype(biased)::value;
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              const float4 l4 = st4[(c0 >> 2) + q4];
              float2 off[2] = {make_float2(l4.x, l4.y), make_float2(l4.z, l4.w)};  // -lse*log2e
              if (kDense) {
                float bv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int c = c0 + 4 * q4 + e;
                  bv[e] = (dcol != nullptr && c >= c_lo && c < c_hi)
                              ? __ldg(dcol + static_cast<long long>(qloc + c) * in.Lkv) * kLog2e
                              : 0.0f;
                }
                off[0] = add_f32x2(make_float2(bv[0], bv[1]), off[0]);
                off[1] = add_f32x2(make_float2(bv[2], bv[3]), off[1]);
              } else if (kBias) {
                const float2 b01 = *reinterpret_cast<const float2*>(bwin + c0 + 4 * q4);
                const float2 b23 = *reinterpret_cast<const float2*>(bwin + c0 + 4 * q4 + 2);
                off[0] = add_f32x2(b01, off[0]);
                off[1] = add_f32x2(b23, off[1]);
              }
              const float2 x01 = fma_f32x2(make_float2(__uint_as_float(sr[4 * q4]), __uint_as_float(sr[4 * q4 + 1])),
                                           make_float2(c_s, c_s), off[0]);
              const float2 x23 = fma_f32x2(make_float2(__uint_as_float(sr[4 * q4 + 2]), __uint_as_float(sr[4 * q4 + 3])),
                                           make_float2(c_s, c_s), off[1]);
              pv[4 * q4] = ex2_approx(x01.x);
              pv[4 * q4 + 1] = ex2_approx(x01.y);
              pv[4 * q4 + 2] = ex2_approx(x23.x);
              pv[4 * q4 + 3] = ex2_approx(x23.y);
              if (kMask) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int c = c0 + 4 * q4 + e;
                  if (c < c_lo || c >= c_hi) pv[4 * q4 + e] = 0.0f;
                }
              }
            }
          };
          using F = std::false_type;
          using T = std::true_type;
          if (full) {
            if (has_bias || kDense) body(F{}, T{}); else body(F{}, F{});
          } else {
            if (has_bias || kDense) body(T{}, T{}); else body(T{}, F{});
          }
        }
        {
          // one scale per 32 keys (this warp's lanes) x 32 queries (this group)
          const int code = e8m0_nosat(__uint_as_float(warp_max_u32(__float_as_uint(amax32(pv)))));
          const float inv = __uint_as_float(static_cast<uint32_t>(254 - code) << 23);
          uint32_t pk[8];
          quant32(pv, inv, pk);
          tmem_st8(tmem + lane_off + kColS + c0, pk);
          // word of key row 32 wq + lane, byte grp (the k-step of these queries)
          sf_p[lane * 16 + wq * 4 + grp] = static_cast<uint8_t>(code);
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        warp_arrive(bar(C::kPFull), lane);
        // Phase 2: dS^T = P^T (dP^T - D) once dP^T of this tile is in TMEM.
        w = mbar_wait(bar(C::kDpFull), g & 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); abort_now = true; break; }
        tc_fence_after();
        {
          uint32_t dr[32];
          tmem_ld32(tmem + lane_off + kColDP + c0, dr);
          const float2 z2 = make_float2(0.0f, 0.0f);
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            const float4 d4 = st4[((kQRows + c0) >> 2) + q4];  // -D
            const float2 v01 = add_f32x2(make_float2(__uint_as_float(dr[4 * q4]), __uint_as_float(dr[4 * q4 + 1])),
                                         make_float2(d4.x, d4.y));
            const float2 v23 = add_f32x2(make_float2(__uint_as_float(dr[4 * q4 + 2]), __uint_as_float(dr[4 * q4 + 3])),
                                         make_float2(d4.z, d4.w));
            // masked P is exactly 0, so masked dS is too
            const float2 a = fma_f32x2(make_float2(pv[4 * q4], pv[4 * q4 + 1]), v01, z2);
            const float2 b = fma_f32x2(make_float2(pv[4 * q4 + 2], pv[4 * q4 + 3]), v23, z2);
            pv[4 * q4] = a.x;
            pv[4 * q4 + 1] = a.y;
            pv[4 * q4 + 2] = b.x;
            pv[4 * q4 + 3] = b.y;
          }
          if (kDenseGrad && gcol != nullptr) {
            // dense-bias gradient: each pair is visited once, its fp32 dS added
            // to its entry (lanes are consecutive keys: one row segment per query)
            float* gt = gcol + static_cast<long long>(qloc + c0) * in.Lkv;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              if (c0 + i >= c_lo && c0 + i < c_hi) atomicAdd(gt, pv[i]);
              gt += in.Lkv;
            }
          }
          if (kTableGrad) {
            // dS(query c0 + i, key 32 wq + lane) lies on diagonal
            // (c0 - 32 wq + 127) + (i - lane) of the tile.  Lane l gathers the
            // warp's values with i - src = l (mod 32): at step i it reads
            // column i of lane (i - l) mod 32, whose offset is l when i >= l
            // and l - 32 otherwise; two shared atomics per lane and tile.
            float up = 0.0f, down = 0.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float v = __shfl_sync(0xffffffffu, pv[i], (i - lane) & 31);
              if (i >= lane) up += v; else down += v;
            }
            float* win = reinterpret_cast<float*>(gbase + C::kDb + (g & 1u) * C::kDbBuf) +
                         (c0 - 32 * wq + 127 + lane);
            atomicAdd(win, up);
            if (lane > 0) atomicAdd(win - 32, down);
          }
          const int code = e8m0_nosat(__uint_as_float(warp_max_u32(__float_as_uint(amax32(pv)))));
          const float inv = __uint_as_float(static_cast<uint32_t>(254 - code) << 23);
          uint32_t pk[8];
          quant32(pv, inv, pk);
          // dS^T row j (A of dK): queries c0..c0+31 are 16-byte chunks 2 grp,
          // 2 grp + 1, stored at (chunk ^ (j % 8))
          uint8_t* dsrow = gbase + C::kDsT + j * 128;
          *reinterpret_cast<uint4*>(dsrow + (((2 * grp) ^ (j & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4*>(dsrow + (((2 * grp + 1) ^ (j & 7)) << 4)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          // dS (B of dQ^T): query row i holds key j at byte j of the row, in
          // 16-byte chunk (j / 16) ^ (i % 8).  Each group of four lanes (keys
          // j4..j4+3) transposes its bytes so that lane r writes one word:
          // keys j4..j4+3 of query c0 + 4q + r.
          {
            const int j4 = j & ~3;
            const int r4 = lane & 3;
            uint8_t* dsq = gbase + C::kDsQ + (j4 & 15);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const uint32_t word = transpose4x4_bytes(pk[q], lane);
              const int i = c0 + 4 * q + r4;
              *reinterpret_cast<uint32_t*>(dsq + i * 128 + (((j4 >> 4) ^ (i & 7)) << 4)) = word;
            }
          }
          // row scales of dS^T (rows = keys, k-step = query block grp) and
          // column scales (rows = queries of block grp, k-step = key block wq)
          sf_dsr[lane * 16 + wq * 4 + grp] = static_cast<uint8_t>(code);
          sf_dsc[lane * 16 + grp * 4 + wq] = static_cast<uint8_t>(code);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        warp_arrive(bar(C::kDsFull), lane);
        if (kTableGrad) {
          if (j == 0 && grp == 0) {
            int* meta = reinterpret_cast<int*>(gbase + C::kDb + (g & 1u) * C::kDbBuf + 192 * 4);
            meta[0] = qloc - kb0 - 127;  // diagonal (query - key) of window entry 0
            meta[1] = in.head;
          }
          warp_arrive(bar(C::kDbAcc + (g & 1u)), lane);
        }
      }
      if (abort_now) break;
    }
  } else if (kTableGrad && warp == kMmaWarp + 1) {
    // ------------------------------------------------------------ bias-table gradient
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
      const MxItem in = decode_mx<kBand>(item, p);
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
      warp_arrive(bar(C::kItemEmpty + slot), lane);
      ++it;
      if (item.x < 0) break;
      const MxItem in = decode_mx<kBand>(item, p);
      bool abort_now = false;
      for (int t = 0; t < in.nq; ++t) {
        w = mbar_wait(bar(C::kDqFull), dqc & 1u, abort_flag);
        w = __all_sync(0xffffffffu, w);
        // Read dQ^T out and free the dP columns first (the next dP product
        // waits for them); a warp whose wait failed reads nothing.
        uint32_t v[2][32];
        if (w) {
          tc_fence_after();
          tmem_ld32(tmem + lane_off + kColDP, v[0]);
          tmem_ld32(tmem + lane_off + kColDP + 32, v[1]);
          tc_fence_before();
          warp_arrive(bar(C::kDqEmpty), lane);  // the dP columns are free again
        }
        // The group syncs on named barriers below, so its four warps must agree
        // on whether the wait succeeded before any of them can leave.
        if (lane == 0) group_ok[wq] = w ? 1 : 0;
        named_bar_sync(1, 128);
        const bool all_ok = group_ok[0] && group_ok[1] && group_ok[2] && group_ok[3];
        if (!all_ok) { if (lane == 0) fail(); abort_now = true; break; }
        ++dqc;
        // Stage 16-query chunks as [query][channel] and add each into the fp32
        // dQ rows with one bulk tensor reduce.  Columns of queries outside the
        // sample carry exact zeros (their dS is 0), so a box that runs into the
        // next sample adds nothing; chunks past the sample are skipped and rows
        // past Tq are clipped by the copy.
        const int qloc = (in.qt0 + t) * kQRows;
        const int qrow = in.q0 + qloc;
#pragma unroll
        for (int ch = 0; ch < kQRows / kDqChunk; ++ch) {
          if (qloc + ch * kDqChunk >= in.Lq) break;  // uniform across the group
          const int buf = dq_issue & 1;
          if (r == 0) bulk_wait_group_read<1>();  // buffer `buf` is free again
          named_bar_sync(1, 128);
          float* stg = reinterpret_cast<float*>(gbase + C::kDqStage + buf * C::kDqStageBytes);
#pragma unroll
          for (int c = 0; c < kDqChunk; ++c)
            stg[c * kD + r] = __uint_as_float(v[(ch * kDqChunk + c) / 32][(ch * kDqChunk + c) % 32]);
          fence_proxy_async_smem();
          named_bar_sync(1, 128);
          if (r == 0) {
            tma_reduce_add_3d(&tmap_dq, sbase + C::kDqStage + buf * C::kDqStageBytes, 0, in.head,
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
      const long long grow = (static_cast<long long>(in.k0 + jl) * p.H + in.head) * kD;
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
            rope_bwd_row<kD>(tmem + lane_off + col, mul, jl, -2.0f * log2f(p.rope_base) / kD, dst,
                             row_ok);
            continue;
          }
#pragma unroll 1
          for (int chunk = 0; chunk < kD / 32; ++chunk) {
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
        for (int q = 0; q < kD / 8; ++q) {
          a4[q] = make_uint4(0, 0, 0, 0);
          b4[q] = make_uint4(0, 0, 0, 0);
        }
      }
    }
    if (r == 0) bulk_wait_group_all();  // every dQ reduce issued by this thread has landed
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool kBand, bool kDBias, bool kRope, bool kDense>
cudaError_t launch_mx(const BwdParams& p, const BwdMxOperands& mx, const CUtensorMap* m, int grid,
                      cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(bwd_mx_kernel<kBand, kDBias, kRope, kDense>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  bwd_mx_kernel<kBand, kDBias, kRope, kDense><<<grid, kThreads, Cfg::kSmemBytes, s>>>(
      m[0], m[1], m[2], m[3], m[4], m[5], m[6], m[7], p, mx);
  return cudaGetLastError();
}

// The bias gradient and the rotary backward have instantiations of their own,
// so calls without them run the unchanged kernels.
template <bool kBand, bool kDense>
cudaError_t launch_mx_band(const BwdParams& p, const BwdMxOperands& mx, const CUtensorMap* m,
                           int grid, cudaStream_t s) {
  const bool db = p.dbias != nullptr, rope = p.rope_base > 0.0f;
  if (rope)
    return db ? launch_mx<kBand, true, true, kDense>(p, mx, m, grid, s)
              : launch_mx<kBand, false, true, kDense>(p, mx, m, grid, s);
  return db ? launch_mx<kBand, true, false, kDense>(p, mx, m, grid, s)
            : launch_mx<kBand, false, false, kDense>(p, mx, m, grid, s);
}

}  // namespace
}  // namespace gdpa
