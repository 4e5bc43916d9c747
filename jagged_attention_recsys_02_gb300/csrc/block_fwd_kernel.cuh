// Block-aligned attention: the forward kernel and its launch templates
// (shared pieces in block_common.cuh), compiled from block.cu (no bias or the
// relative-position table) and block_fwd_dense.cu (a dense jagged bias).
#pragma once
#include "block_common.cuh"

namespace gdpa {
namespace {

using namespace ptx;
// ---------------------------------------------------------------- forward
// 320 threads: warps 0-3 and 4-7 are two activation groups that take the
// CTA's items in turn (group u: items k with k % 2 == u, TMEM buffer u),
// warp 8 the TMA producer, warp 9 the MMA issuer.  TMEM buffer u: S / P
// columns [256u, 256u+128), O [256u+128, 256u+128+d).  Per item the MMA warp
// issues S(k) = Q K^T and, once item k-1's P is in TMEM, O(k-1) = P V (P from
// TMEM, V from shared memory); the activation group masks the scores to the
// row's block, takes the exact softmax (or the GDPA activation, P split into
// bf16 hi + lo parts for two value MMAs), writes P, then stores O / l.
constexpr int kFwdThreads = 320;
constexpr int kFwdProducer = 8;
constexpr int kFwdMma = 9;

template <int D>
struct BfCfg {
  static constexpr int kTileBytes = kTileRows * D * 2;
  static constexpr int kStages = (D == 128) ? 2 : 4;
  static constexpr int kBiasBytes = 1024;                      // 255 floats, padded
  static constexpr int kStageBytes = 3 * kTileBytes + kBiasBytes;  // Q, K, V, bias window
  static_assert(kStageBytes % 1024 == 0, "stages keep 1024-byte alignment");
  static constexpr int kQ = 0, kK = kTileBytes, kV = 2 * kTileBytes, kBias = 3 * kTileBytes;
  static constexpr int kBar = kStages * kStageBytes;
  // Q and K of a stage free up after its score product, V and the bias window
  // after the value product: the next loads start as early as they can.
  static constexpr int kQKFull = 0;               // + stage
  static constexpr int kQKEmpty = kStages;        // + stage
  static constexpr int kVFull = 2 * kStages;      // + stage (V and the bias window)
  static constexpr int kVEmpty = 3 * kStages;     // + stage
  static constexpr int kSFull = 4 * kStages;      // + buffer
  static constexpr int kPFull = kSFull + 2;       // + buffer
  static constexpr int kODone = kPFull + 2;       // + buffer
  static constexpr int kDrain = kODone + 2;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kTmemSlot = kBar + 8 * kNumBars;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kUsed = kAbort + 4;
  static constexpr int kSmemBytes = kUsed + 1024;
};

// kDense: a dense jagged bias (p.bias_dense) instead of the relative-position
// table; each activation thread reads its row's values of the keys it sees
// (its own block: at most 64 consecutive floats).
template <int D, int ACT, bool kDense>
__global__ void __launch_bounds__(kFwdThreads, 1)
block_fwd_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                 const __grid_constant__ CUtensorMap tmap_v, const BlockParams p) {
  using C = BfCfg<D>;
  constexpr bool kSoftmax = (ACT == GDPA_ACT_SOFTMAX);
  constexpr bool kSplit = !kSoftmax;
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
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kQKFull + s), 1);
      mbar_init(bar(C::kQKEmpty + s), 1);
      mbar_init(bar(C::kVFull + s), 1);
      mbar_init(bar(C::kVEmpty + s), 1);
    }
    for (int u = 0; u < 2; ++u) {
      mbar_init(bar(C::kSFull + u), 1);
      mbar_init(bar(C::kPFull + u), 4);  // one arrival per activation warp
      mbar_init(bar(C::kODone + u), 1);
    }
    mbar_init(bar(C::kDrain), 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp == kFwdProducer && lane == 0) {
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
  const int n_items = *p.n_tiles * p.H;
  auto item_of = [&](int k) { return static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x); };

  if (warp == kFwdProducer) {
    // ------------------------------------------------------------ producer
    const bool has_bias = p.bias_table != nullptr;
    uint32_t inflight = 0, last_k[C::kStages] = {};
    for (int k = 0;; ++k) {
      const int item = item_of(k);
      if (item >= n_items) break;
      const int head = item % p.H;
      const TileInfo ti = load_tile(p.tiles, item / p.H);
      const uint32_t s = k % C::kStages, ph = (k / C::kStages) & 1u;
      const uint32_t st = sbase + s * C::kStageBytes;
      bool w = mbar_wait(bar(C::kQKEmpty + s), ph ^ 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(C::kQKFull + s), 2 * C::kTileBytes);
#pragma unroll
        for (int x = 0; x < D; x += 64) {
          const uint32_t off = (x / 64) * (kTileRows * 128);
          tma_load_3d(st + C::kQ + off, &tmap_q, bar(C::kQKFull + s), x, head, ti.row0);
          tma_load_3d(st + C::kK + off, &tmap_k, bar(C::kQKFull + s), x, head, ti.row0);
        }
        inflight |= 1u << s;
        last_k[s] = k;
      }
      w = mbar_wait(bar(C::kVEmpty + s), ph ^ 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      if (has_bias)
        stage_bias(reinterpret_cast<float*>(gbase + s * C::kStageBytes + C::kBias), p.bias_table,
                   head, p.max_rel, kSoftmax ? kLog2e : 1.0f, lane);
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(C::kVFull + s), C::kTileBytes);
#pragma unroll
        for (int x = 0; x < D; x += 64)
          tma_load_3d(st + C::kV + (x / 64) * (kTileRows * 128), &tmap_v, bar(C::kVFull + s), x,
                      head, ti.row0);
      }
    }
    if (lane == 0 && *abort_flag) {
      for (int s = 0; s < C::kStages; ++s)
        if (inflight & (1u << s)) {
          mbar_wait(bar(C::kQKFull + s), (last_k[s] / C::kStages) & 1u, nullptr, 50000000ull);
          mbar_wait(bar(C::kVFull + s), (last_k[s] / C::kStages) & 1u, nullptr, 50000000ull);
        }
    }
  } else if (warp == kFwdMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16(128, kTileRows, true, false, false);
      constexpr uint32_t idesc_pv = idesc_f16(128, D, true, false, true);
      const uint64_t dsc_q = sdesc(sbase + C::kQ, 0, 1024, kSwizzle128B);
      const uint64_t dsc_k = sdesc(sbase + C::kK, 0, 1024, kSwizzle128B);
      const uint64_t dsc_v = sdesc(sbase + C::kV, kTileRows * 128, 1024, kSwizzle128B);
      bool issued_any = false;
      for (int k = 0;; ++k) {
        const bool have = item_of(k) < n_items;
        if (have) {
          const uint32_t s = k % C::kStages;
          if (!mbar_wait(bar(C::kQKFull + s), (k / C::kStages) & 1u, abort_flag)) { fail(); break; }
          tc_fence_after();
          const uint32_t so = s * C::kStageBytes;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = (ks / 4) * (kTileRows * 128) + (ks % 4) * 32;
            mma_f16_ss(tmem + (k & 1) * 256, dadd(dsc_q, so + off), dadd(dsc_k, so + off), idesc_s,
                       ks > 0 ? 1u : 0u);
          }
          mma_commit(bar(C::kSFull + (k & 1)));
          mma_commit(bar(C::kQKEmpty + s));
          issued_any = true;
        }
        if (k >= 1) {
          const int kk = k - 1;
          const uint32_t u = kk & 1, s = kk % C::kStages;
          if (!mbar_wait(bar(C::kPFull + u), (kk >> 1) & 1u, abort_flag)) { fail(); break; }
          if (!mbar_wait(bar(C::kVFull + s), (kk / C::kStages) & 1u, abort_flag)) { fail(); break; }
          tc_fence_after();
          const uint64_t vb = dadd(dsc_v, s * C::kStageBytes);
          const uint32_t tp = tmem + u * 256, to = tp + 128;
#pragma unroll
          for (int ks = 0; ks < kTileRows / 16; ++ks) {
            const uint32_t pcol = 32 * (ks / 2) + 8 * (ks % 2);
            mma_f16_ts(to, tp + pcol, dadd(vb, ks * 2048), idesc_pv, ks == 0 ? 0u : 1u);
            if (kSplit) mma_f16_ts(to, tp + pcol + 16, dadd(vb, ks * 2048), idesc_pv, 1u);
          }
          mma_commit(bar(C::kODone + u));
          mma_commit(bar(C::kVEmpty + s));
        }
        if (!have) break;
      }
      if (issued_any) {
        mma_commit(bar(C::kDrain));
        mbar_wait(bar(C::kDrain), 0, nullptr, 100000000ull);
      }
    }
  } else {
    // ------------------------------------------------------------ activation groups
    const int u = warp >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // tile row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_off + u * 256;
    const uint32_t t_o = t_s + 128;
    const float c_s = kSoftmax ? p.scale * kLog2e : p.scale;
    const bool has_bias = p.bias_table != nullptr;
    for (int k = u;; k += 2) {
      const int item = item_of(k);
      if (item >= n_items) break;
      const int head = item % p.H;
      const TileInfo ti = load_tile(p.tiles, item / p.H);
      const uint32_t s = k % C::kStages;
      bool w = mbar_wait(bar(C::kSFull + u), (k >> 1) & 1u, abort_flag);
      // the stage's bias window was written by the producer before V's barrier phase
      if (has_bias) w = w && mbar_wait(bar(C::kVFull + s), (k / C::kStages) & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      tc_fence_after();
      int c_lo, c_hi;
      row_keys(ti, r, p.causal, &c_lo, &c_hi);
      const float* bwin = reinterpret_cast<const float*>(gbase + s * C::kStageBytes + C::kBias) +
                          (kTileRows - 1) + r;  // bwin[-c] = bias(r - c)
      // dense bias of (row r, column c): drow[c], read only where the row sees c
      const float* drow = nullptr;
      if (kDense) {
        const long long base = dense_row_base(p, ti, r, head);
        if (base >= 0) drow = p.bias_dense + base;
      }
      float l = 0.0f;
      // NCH 32-column chunks from column cb (P of the other chunks is zero).
      // Every array index below is a compile-time constant, so nothing leaves
      // registers.
      auto run = [&](auto nch, int cb) {
        constexpr int NCH = decltype(nch)::value;
        constexpr float fill = kSoftmax ? -INFINITY : 0.0f;
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
            x[i] = (c < c_lo || c >= c_hi) ? fill : v;
          }
        };
        if (kSoftmax) {
          float xs[NCH][32];
          float m = -INFINITY;
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) {
            load_x(ch, xs[ch]);
#pragma unroll
            for (int i = 0; i < 32; ++i) m = fmaxf(m, xs[ch][i]);
          }
          const float m_ref = (m == -INFINITY) ? 0.0f : m;
          float2 l2 = make_float2(0.0f, 0.0f);
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) {
            uint32_t hi[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float p0 = ex2_approx(xs[ch][2 * i] - m_ref);
              const float p1 = ex2_approx(xs[ch][2 * i + 1] - m_ref);
              l2 = add_f32x2(l2, make_float2(p0, p1));
              hi[i] = pack_bf16x2(p0, p1);
            }
            tmem_st16(t_s + cb + 32 * ch, hi);
          }
          l = l2.x + l2.y;
        } else {
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) {
            float x[32];
            load_x(ch, x);
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float p0 = act_fwd(ACT, x[2 * i]), p1 = act_fwd(ACT, x[2 * i + 1]);
              const uint32_t h = pack_bf16x2(p0, p1);
              hi[i] = h;
              lo[i] = pack_bf16x2(p0 - __uint_as_float(h << 16), p1 - __uint_as_float(h & 0xFFFF0000u));
            }
            tmem_st16(t_s + cb + 32 * ch, hi);
            tmem_st16(t_s + cb + 32 * ch + 16, lo);
          }
        }
        if (NCH < kTileRows / 32) {
          // the other block's half of P
          const uint32_t zero[16] = {};
          const int zb = cb == 0 ? 32 * NCH : 0;
#pragma unroll
          for (int z = 0; z < kTileRows / 32 - NCH; ++z) {
            tmem_st16(t_s + zb + 32 * z, zero);
            if (kSplit) tmem_st16(t_s + zb + 32 * z + 16, zero);
          }
        }
      };
      // Two full blocks (the common case): warps 0-1 hold block A's rows and
      // need columns [0,64) only, warps 2-3 block B's rows and [64,128).
      if (ti.len_a == kBlk)
        run(std::integral_constant<int, 2>{}, wq >= 2 ? kBlk : 0);
      else
        run(std::integral_constant<int, 4>{}, 0);
      tmem_st_wait();
      tc_fence_before();
      warp_arrive(bar(C::kPFull + u), lane);
      w = mbar_wait(bar(C::kODone + u), (k >> 1) & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      tc_fence_after();
      const float inv_l = kSoftmax ? (l > 0.0f ? 1.0f / l : 0.0f) : 1.0f;
      __nv_bfloat16* orow = p.out + (static_cast<long long>(ti.row0 + r) * p.H + head) * D;
#pragma unroll 1
      for (int chunk = 0; chunk < D / 32; ++chunk) {
        uint32_t o[32];
        tmem_ld32(t_o + 32 * chunk, o);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
        if (r < ti.rows) {
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * chunk);
#pragma unroll
          for (int v = 0; v < 4; ++v) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int ACT, bool kDense>
cudaError_t launch_fwd_one(const BlockParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, int grid, cudaStream_t s) {
  constexpr int smem = BfCfg<D>::kSmemBytes;
  static_assert(smem <= 232448, "shared memory budget");
  cudaError_t e = cudaFuncSetAttribute(block_fwd_kernel<D, ACT, kDense>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  block_fwd_kernel<D, ACT, kDense><<<grid, kFwdThreads, smem, s>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

template <int D, bool kDense>
cudaError_t launch_fwd_d(const BlockParams& p, int act, const CUtensorMap& tq,
                         const CUtensorMap& tk, const CUtensorMap& tv, int grid, cudaStream_t s) {
  switch (act) {
    case GDPA_ACT_SOFTMAX:
      return launch_fwd_one<D, GDPA_ACT_SOFTMAX, kDense>(p, tq, tk, tv, grid, s);
    case GDPA_ACT_SILU: return launch_fwd_one<D, GDPA_ACT_SILU, kDense>(p, tq, tk, tv, grid, s);
    case GDPA_ACT_GELU_TANH:
      return launch_fwd_one<D, GDPA_ACT_GELU_TANH, kDense>(p, tq, tk, tv, grid, s);
    case GDPA_ACT_GELU_ERF:
      return launch_fwd_one<D, GDPA_ACT_GELU_ERF, kDense>(p, tq, tk, tv, grid, s);
    default: return launch_fwd_one<D, GDPA_ACT_IDENTITY, kDense>(p, tq, tk, tv, grid, s);
  }
}

}  // namespace
}  // namespace gdpa
