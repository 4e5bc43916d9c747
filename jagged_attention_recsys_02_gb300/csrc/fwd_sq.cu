// Short-query forward (GDPA activations), sm_103a.
//
// "GEM Training ..." GDPA paragraph: GDPA serves PMA, whose few learned seed
// queries attend over long jagged key sequences, and the kernels were
// reworked for the short / asymmetric shapes of production.  With 32 or
// fewer queries a 128-row query tile would be three quarters empty, so this
// kernel swaps the roles of the operands: TMEM lanes are keys and the
// queries are the MMA's N.
//
// Work item: one (sample, head) of the scheduler's short-query list (Lq <= 32).
// The CTA keeps the item's queries in shared memory and streams the sample's
// 128-key K/V tiles through a three-stage ring:
//   S^T = K Q^T                (M = 128 keys, N = 32 queries, K = d) -> TMEM
//   P^T = act(scale S^T)       activation warps, keys past the sample masked
//   O^T += V^T P^T             (M = d channels, N = 32, K = 128 keys) -> TMEM
// P^T is split into bf16 hi + lo parts (two MMAs), as in the row-major
// forward, because thousands of unnormalised terms are summed; it is written
// to shared memory as the K-major B operand: row = query, 128-byte swizzled
// atoms of 64 keys.  O^T is stored once per item (lanes = channels).
//
// Warps: 0-3 activation and epilogue, 4 producer (tickets, TMA), 5 MMA.
// TMEM: S^T buffers [0,32) [32,64); O^T [64,96).  Every wait is bounded.
#include "common.cuh"

namespace gdpa {
namespace {

using namespace ptx;

constexpr int kThreads = 192;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kStages = 3;
constexpr uint32_t kColS = 0, kColO = 64;

template <int D>
struct SqCfg {
  static constexpr int kAtomsD = D / 64;                    // 64-channel atoms
  static constexpr int kQBytes = kShortQ * D * 2;           // [atom][32 rows][128 B]
  static constexpr int kKvTile = kKvRows * D * 2;           // K or V tile
  static constexpr int kPPart = kShortQ * kKvRows * 2;      // P^T part: [2 atoms][32 rows][128 B]
  static constexpr int kQ = 0;
  static constexpr int kKV = kQBytes;                       // + s * 2 * kKvTile (K, then V)
  static constexpr int kP = kKV + kStages * 2 * kKvTile;    // hi, lo
  static constexpr int kBar = kP + 2 * kPPart;
  static constexpr int kQFull = 0, kQEmpty = 1;
  static constexpr int kKvFull = 2;                         // + s
  static constexpr int kKvEmpty = kKvFull + kStages;        // + s
  static constexpr int kSFull = kKvEmpty + kStages;         // + buffer
  static constexpr int kPFull = kSFull + 2;
  static constexpr int kPEmpty = kPFull + 1;
  static constexpr int kOFull = kPEmpty + 1;
  static constexpr int kOEmpty = kOFull + 1;
  static constexpr int kItemFull = kOEmpty + 1;             // + slot
  static constexpr int kItemEmpty = kItemFull + 2;
  static constexpr int kDrain = kItemEmpty + 2;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kItemSlots = kBar + 8 * kNumBars;
  static constexpr int kTmemSlot = kItemSlots + 16;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kUsed = kAbort + 4;
  static constexpr int kSmemBytes = kUsed + 1024;
};

template <int ACT>
__device__ __forceinline__ float act_value(float x) {
  float a, g;
  act_and_grad<ACT>(x, a, g);
  return a;
}

template <int D, int ACT>
__global__ void __launch_bounds__(kThreads, 1)
fwd_sq_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
              const __grid_constant__ CUtensorMap tmap_v, const FwdParams p) {
  using C = SqCfg<D>;
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
      mbar_init(bar(C::kKvFull + s), 1);
      mbar_init(bar(C::kKvEmpty + s), 1);
    }
    mbar_init(bar(C::kSFull), 1);
    mbar_init(bar(C::kSFull + 1), 1);
    mbar_init(bar(C::kPFull), 4);
    mbar_init(bar(C::kPEmpty), 1);
    mbar_init(bar(C::kOFull), 1);
    mbar_init(bar(C::kOEmpty), 4);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::kItemFull + s), 1);
      mbar_init(bar(C::kItemEmpty + s), 1 + 4);
    }
    mbar_init(bar(C::kDrain), 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 128);
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
      uint32_t it = 0, g = 0, qi = 0, inflight = 0, last_g[kStages] = {};
      bool q_inflight = false, ok = true;
      while (ok) {
        const int t = atomicAdd(p.ticket, 1);
        const int2 item = t < n_items ? p.items[t] : make_int2(-1, 0);
        const uint32_t slot = it & 1u;
        if (!mbar_wait(bar(C::kItemEmpty + slot), ((it >> 1) & 1u) ^ 1u, abort_flag)) { fail(); break; }
        item_slot[slot] = item;
        mbar_arrive(bar(C::kItemFull + slot));
        ++it;
        if (item.x < 0) break;
        const int b = item.x, head = item.y;
        const int q0 = p.qo[b], k0 = p.ko[b], Lkv = p.ko[b + 1] - k0;
        const int nkv = (Lkv + kKvRows - 1) / kKvRows;
        if (!mbar_wait(bar(C::kQEmpty), (qi & 1u) ^ 1u, abort_flag)) { fail(); break; }
        mbar_arrive_expect_tx(bar(C::kQFull), C::kQBytes);
        for (int a = 0; a < C::kAtomsD; ++a)
          tma_load_3d(sbase + C::kQ + a * (kShortQ * 128), &tmap_q, bar(C::kQFull), 64 * a, head, q0);
        q_inflight = true;
        ++qi;
        for (int j = 0; j < nkv; ++j, ++g) {
          const uint32_t s = g % kStages;
          if (!mbar_wait(bar(C::kKvEmpty + s), ((g / kStages) & 1u) ^ 1u, abort_flag)) { ok = false; fail(); break; }
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
      if (*abort_flag) {  // let every copy this thread started land
        for (int s = 0; s < kStages; ++s)
          if (inflight & (1u << s))
            mbar_wait(bar(C::kKvFull + s), (last_g[s] / kStages) & 1u, nullptr, 50000000ull);
        if (q_inflight) mbar_wait(bar(C::kQFull), (qi - 1) & 1u, nullptr, 50000000ull);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // S^T: A = K (K-major), B = Q (K-major), M = 128, N = 32.
      // O^T: A = V^T (V tile read M-major: channels contiguous), B = P^T (K-major).
      constexpr uint32_t idesc_s = idesc_f16(128, kShortQ, true, false, false);
      constexpr uint32_t idesc_o = idesc_f16(128, kShortQ, true, true, false);
      const uint64_t dsc_q = sdesc(sbase + C::kQ, 0, 1024, kSwizzle128B);
      const uint64_t dsc_k = sdesc(sbase + C::kKV, 0, 1024, kSwizzle128B);
      // d = 64: the second 64-row half of A repeats the first (LBO 0); its
      // output lanes 64..127 are never read.
      const uint64_t dsc_vt = sdesc(sbase + C::kKV + C::kKvTile, D == 128 ? kKvRows * 128 : 0, 1024,
                                    kSwizzle128B);
      const uint64_t dsc_p = sdesc(sbase + C::kP, 0, 1024, kSwizzle128B);
      uint32_t it = 0, g = 0, qi = 0, sc = 0, pc = 0, oc = 0;
      bool issued_any = false, ok = true;
      auto issue_s = [&](uint32_t stage, uint32_t buf) {
        const uint64_t kb = dadd(dsc_k, stage * 2 * C::kKvTile);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_f16_ss(tmem + kColS + 32 * buf,
                     dadd(kb, (ks / 4) * (kKvRows * 128) + (ks % 4) * 32),
                     dadd(dsc_q, (ks / 4) * (kShortQ * 128) + (ks % 4) * 32), idesc_s,
                     ks > 0 ? 1u : 0u);
        mma_commit(bar(C::kSFull + buf));
        issued_any = true;
      };
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
        if (nkv == 0) {
          mma_commit(bar(C::kQEmpty));
          continue;
        }
        {
          const uint32_t s0 = g % kStages;
          if (!mbar_wait(bar(C::kKvFull + s0), (g / kStages) & 1u, abort_flag)) { fail(); break; }
          tc_fence_after();
          issue_s(s0, sc & 1u);
        }
        for (int j = 0; j < nkv; ++j) {
          const uint32_t gj = g + j;
          const uint32_t s = gj % kStages;
          // S^T of the next tile into the other buffer (its previous P^T has been
          // consumed: the activation warps finished it before this tile's S^T)
          if (j + 1 < nkv) {
            const uint32_t s1 = (gj + 1) % kStages;
            if (!mbar_wait(bar(C::kKvFull + s1), ((gj + 1) / kStages) & 1u, abort_flag)) { ok = false; fail(); break; }
            tc_fence_after();
            issue_s(s1, (sc + 1 + j) & 1u);
          } else {
            mma_commit(bar(C::kQEmpty));  // every S^T of the item has been issued
          }
          if (!mbar_wait(bar(C::kPFull), pc & 1u, abort_flag)) { ok = false; fail(); break; }
          ++pc;
          if (j == 0) {
            // the previous item's O^T must have been read out before it is overwritten
            if (!mbar_wait(bar(C::kOEmpty), (oc & 1u) ^ 1u, abort_flag)) { ok = false; fail(); break; }
            ++oc;
          }
          tc_fence_after();
          const uint64_t vb = dadd(dsc_vt, s * 2 * C::kKvTile);
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int ks = 0; ks < kKvRows / 16; ++ks)
              mma_f16_ss(tmem + kColO, dadd(vb, ks * 2048),
                         dadd(dsc_p, part * C::kPPart + (ks / 4) * (kShortQ * 128) + (ks % 4) * 32),
                         idesc_o, (j == 0 && part == 0 && ks == 0) ? 0u : 1u);
          mma_commit(bar(C::kPEmpty));
          mma_commit(bar(C::kKvEmpty + s));
        }
        if (!ok) break;
        sc += nkv;
        g += nkv;
        mma_commit(bar(C::kOFull));
      }
      if (issued_any) {
        mma_commit(bar(C::kDrain));
        mbar_wait(bar(C::kDrain), 0, nullptr, 100000000ull);
      }
    }
  } else {
    // ------------------------------------------------------------ activation + epilogue
    const int r = warp * 32 + lane;                            // TMEM lane: key, or channel
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    // P^T element (query q, key r): atom r / 64, row q, 16-byte chunk
    // ((r % 64) / 8) ^ (q % 8), 2 bytes at (r % 8)
    uint8_t* pbase = gbase + C::kP + (r >> 6) * (kShortQ * 128) + (r & 7) * 2;
    const int chunk = (r & 63) >> 3;
    uint32_t it = 0, sc = 0, pc = 0, oc = 0;
    bool abort_now = false;
    while (!abort_now) {
      const uint32_t slot = it & 1u;
      bool w = mbar_wait(bar(C::kItemFull + slot), (it >> 1) & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      const int2 item = item_slot[slot];
      warp_arrive(bar(C::kItemEmpty + slot), lane);
      ++it;
      if (item.x < 0) break;
      const int b = item.x, head = item.y;
      const int q0 = p.qo[b], Lq = p.qo[b + 1] - q0;
      const int Lkv = p.ko[b + 1] - p.ko[b];
      const int nkv = (Lkv + kKvRows - 1) / kKvRows;
      for (int j = 0; j < nkv; ++j, ++sc) {
        w = mbar_wait(bar(C::kSFull + (sc & 1u)), (sc >> 1) & 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); abort_now = true; break; }
        tc_fence_after();
        uint32_t sr[32];
        tmem_ld32(tmem + lane_off + kColS + 32 * (sc & 1u), sr);
        const bool key_ok = j * kKvRows + r < Lkv;
        uint16_t hi[kShortQ], lo[kShortQ];
#pragma unroll
        for (int q = 0; q < kShortQ; ++q) {
          const float a = key_ok ? act_value<ACT>(__uint_as_float(sr[q]) * p.scale) : 0.0f;
          const __nv_bfloat16 h = __float2bfloat16_rn(a);
          hi[q] = __bfloat16_as_ushort(h);
          lo[q] = __bfloat16_as_ushort(__float2bfloat16_rn(a - __bfloat162float(h)));
        }
        // the previous tile's O^T products have read the P^T buffer (the first
        // wait on the fresh barrier returns at once)
        w = mbar_wait(bar(C::kPEmpty), (pc & 1u) ^ 1u, abort_flag);
        if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); abort_now = true; break; }
#pragma unroll
        for (int q = 0; q < kShortQ; ++q) {
          const int off = q * 128 + ((chunk ^ (q & 7)) << 4);
          *reinterpret_cast<uint16_t*>(pbase + off) = hi[q];
          *reinterpret_cast<uint16_t*>(pbase + C::kPPart + off) = lo[q];
        }
        ++pc;
        fence_proxy_async_smem();
        tc_fence_before();
        warp_arrive(bar(C::kPFull), lane);
      }
      if (abort_now) break;
      if (nkv == 0) {
        // no key: the queries' outputs are zero
        if (r < D)
          for (int q = 0; q < Lq; ++q)
            p.out[(static_cast<long long>(q0 + q) * p.H + head) * D + r] = __float2bfloat16_rn(0.0f);
        continue;
      }
      // ---------------------------------------------------------- epilogue: O^T lanes are channels
      w = mbar_wait(bar(C::kOFull), oc & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { if (lane == 0) fail(); break; }
      ++oc;
      tc_fence_after();
      uint32_t o[32];
      tmem_ld32(tmem + lane_off + kColO, o);
      tc_fence_before();
      warp_arrive(bar(C::kOEmpty), lane);
      if (r < D)
        for (int q = 0; q < Lq; ++q)
          p.out[(static_cast<long long>(q0 + q) * p.H + head) * D + r] =
              __float2bfloat16_rn(__uint_as_float(o[q]));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

template <int D, int ACT>
cudaError_t launch_sq_one(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, int grid, cudaStream_t stream) {
  using C = SqCfg<D>;
  static_assert(C::kSmemBytes <= 232448, "shared memory budget");
  cudaError_t e = cudaFuncSetAttribute(fwd_sq_kernel<D, ACT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  fwd_sq_kernel<D, ACT><<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_sq_d(const FwdParams& p, int act, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, int grid, cudaStream_t stream) {
  switch (act) {
    case GDPA_ACT_SILU: return launch_sq_one<D, GDPA_ACT_SILU>(p, tq, tk, tv, grid, stream);
    case GDPA_ACT_GELU_TANH: return launch_sq_one<D, GDPA_ACT_GELU_TANH>(p, tq, tk, tv, grid, stream);
    case GDPA_ACT_GELU_ERF: return launch_sq_one<D, GDPA_ACT_GELU_ERF>(p, tq, tk, tv, grid, stream);
    case GDPA_ACT_IDENTITY: return launch_sq_one<D, GDPA_ACT_IDENTITY>(p, tq, tk, tv, grid, stream);
    default: return cudaErrorInvalidValue;  // softmax needs row statistics across the keys
  }
}

}  // namespace

cudaError_t launch_fwd_short_q(const FwdParams& p, int act, const CUtensorMap& tq,
                               const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                               cudaStream_t stream) {
  return p.d == 64 ? launch_sq_d<64>(p, act, tq, tk, tv, grid, stream)
                   : launch_sq_d<128>(p, act, tq, tk, tv, grid, stream);
}

}  // namespace gdpa
