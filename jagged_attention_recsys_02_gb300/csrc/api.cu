// C ABI entry points (include/gdpa.h): argument checks, TMA descriptors,
// workspace carving and kernel launches.  No device memory is allocated
// here; the caller passes every buffer, including the workspace.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace gdpa {
namespace {

// Device status word: set by kernels (timeouts, malformed offsets), read and
// cleared by gdpa_get_device_status().
__device__ int g_status_word;

constexpr int kMaxDevices = 64;
struct DeviceInfo {
  bool init = false;
  int sms = 0;
  int* status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
thread_local int t_launches = 0;

// Optional timing of the main kernels (gdpa_timing_enable / _collect).
constexpr int kMaxTimed = 4096;
struct TimingRing {
  bool enabled = false;
  int n = 0;
  int kind[kMaxTimed];
  cudaEvent_t ev[2 * kMaxTimed] = {};
};
thread_local TimingRing* t_timing = nullptr;

// Returns the event pair to record around the next main kernel, or false.
bool timing_slot(int kind, cudaEvent_t* a, cudaEvent_t* b) {
  TimingRing* r = t_timing;
  if (r == nullptr || !r->enabled || r->n >= kMaxTimed) return false;
  const int i = r->n;
  for (int e = 0; e < 2; ++e)
    if (r->ev[2 * i + e] == nullptr && cudaEventCreate(&r->ev[2 * i + e]) != cudaSuccess) return false;
  r->kind[i] = kind;
  *a = r->ev[2 * i];
  *b = r->ev[2 * i + 1];
  r->n = i + 1;
  return true;
}

cudaError_t device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.init) {
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_status_word);
    if (e != cudaSuccess) return e;
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q);
      if (e != cudaSuccess) return e;
      if (q != cudaDriverEntryPointSuccess || fn == nullptr) return cudaErrorNotSupported;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    d.init = true;
  }
  *out = &d;
  return cudaSuccess;
}

// 3-D TMA map over a [T][H][d] bf16 tensor: box = 64 channels x 1 head x
// `box_rows` rows, 128-byte swizzle (the layout the tcgen05 descriptors use).
bool make_thd_map(CUtensorMap* m, const void* base, int64_t T, int H, int d, int box_rows) {
  if (T <= 0) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(H) * static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D TMA map over the fp32 dQ accumulator [T][H][d]: box = `box_ch` channels
// x 1 head x `box_rows` rows, no swizzle (the target of the backward's tile
// reduce-add).
bool make_dq_map(CUtensorMap* m, void* base, int64_t T, int H, int d, int box_ch, int box_rows) {
  if (T <= 0) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4,
                           static_cast<cuuint64_t>(H) * static_cast<cuuint64_t>(d) * 4};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_ch), 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D TMA map over E4M3 codes [T][H][d] (u8): box = d bytes x 1 head x
// `box_rows` rows, 128-byte swizzle (d = 128).
bool make_u8_map(CUtensorMap* m, const void* base, int64_t T, int H, int d, int box_rows) {
  if (T <= 0) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d),
                           static_cast<cuuint64_t>(H) * static_cast<cuuint64_t>(d)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(d), 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

gdpa_status check_common(const void* q, const int32_t* qo, const void* k, const void* v,
                         const int32_t* ko, int B, int H, int d, int64_t Tq, int64_t Tkv,
                         const gdpa_bias* bias, int act, int causal, int window) {
  if (B < 0 || H <= 0 || Tq < 0 || Tkv < 0) return GDPA_ERR_INVALID_ARG;
  if (window < 0) return GDPA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return GDPA_ERR_UNSUPPORTED;
  if (H > 256) return GDPA_ERR_UNSUPPORTED;
  if (act < GDPA_ACT_SOFTMAX || act > GDPA_ACT_GELU_ERF) return GDPA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return GDPA_ERR_INVALID_ARG;
  if (qo == nullptr || ko == nullptr) return GDPA_ERR_INVALID_ARG;
  if (Tq > 0 && q == nullptr) return GDPA_ERR_INVALID_ARG;
  if (Tkv > 0 && (k == nullptr || v == nullptr)) return GDPA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return GDPA_ERR_INVALID_ARG;
  if (Tq > (int64_t(1) << 31) - 1 || Tkv > (int64_t(1) << 31) - 1) return GDPA_ERR_UNSUPPORTED;
  if (bias != nullptr && bias->kind != GDPA_BIAS_NONE) {
    if (bias->kind == GDPA_BIAS_DENSE) {
      if (bias->table == nullptr || bias->offsets == nullptr ||
          (reinterpret_cast<uintptr_t>(bias->table) & 3u) ||
          (reinterpret_cast<uintptr_t>(bias->offsets) & 7u))
        return GDPA_ERR_INVALID_ARG;
      return GDPA_OK;
    }
    if (bias->kind != GDPA_BIAS_RELPOS) return GDPA_ERR_INVALID_ARG;
    if (bias->table == nullptr || bias->max_rel < 1 || bias->max_rel > 65536)
      return GDPA_ERR_INVALID_ARG;
  }
  return GDPA_OK;
}

bool is_dense(const gdpa_bias* bias) { return bias != nullptr && bias->kind == GDPA_BIAS_DENSE; }
int bias_kind(const gdpa_bias* bias) { return bias == nullptr ? GDPA_BIAS_NONE : bias->kind; }

// The relative-position table (nullptr for no bias or a dense bias).
const float* bias_table(const gdpa_bias* bias, int* max_rel) {
  if (bias == nullptr || bias->kind != GDPA_BIAS_RELPOS) {
    *max_rel = 1;
    return nullptr;
  }
  *max_rel = bias->max_rel;
  return bias->table;
}

// A pipeline wait that cannot complete: one mbarrier that nothing arrives
// at, waited on with the kernels' own bounded wait (limit_ns of wall time).
// When the wait gives up, the kernel records GDPA_ERR_TIMEOUT in the status
// word and returns, as every kernel of the library does on a timeout.
__global__ void selftest_timeout_kernel(int* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  const uint32_t b = ptx::smem_u32(&bar);
  if (threadIdx.x == 0) {
    ptx::mbar_init(b, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !ptx::mbar_wait(b, 0, nullptr, limit_ns))
    set_status(status, GDPA_ERR_TIMEOUT);
}

}  // namespace
}  // namespace gdpa

using namespace gdpa;

extern "C" {

// Workspace header (256 bytes): main-list count and ticket, short-query list
// count and ticket, all-short flag, short-key list count and ticket.  The main
// list follows at byte 256, the short-query list (one item per sample and
// head at most) after it, then the forward's short-key list.
size_t gdpa_fwd_workspace_size(int B, int H, int d, int64_t Tq, int64_t Tkv) {
  (void)d;
  (void)Tkv;
  if (B < 0 || H <= 0 || Tq < 0) return 0;
  return 256 + align_up(static_cast<size_t>(max_fwd_items(B, H, Tq)) * sizeof(int2), 256) +
         align_up(static_cast<size_t>(B) * H * sizeof(int2), 256) +
         align_up(static_cast<size_t>(max_kv_items(B, H, Tq)) * sizeof(int2), 256);
}

gdpa_status gdpa_fwd(const void* q, const int32_t* q_offsets, const void* k, const void* v,
                     const int32_t* kv_offsets, int B, int H, int d, int64_t Tq, int64_t Tkv,
                     const gdpa_bias* bias, int act, int causal, float scale, void* out,
                     float* lse, void* workspace, size_t ws_bytes, void* stream) {
  return gdpa_fwd_window(q, q_offsets, k, v, kv_offsets, B, H, d, Tq, Tkv, bias, act, causal, 0,
                         scale, out, lse, workspace, ws_bytes, stream);
}

gdpa_status gdpa_fwd_window(const void* q, const int32_t* q_offsets, const void* k,
                            const void* v, const int32_t* kv_offsets, int B, int H, int d,
                            int64_t Tq, int64_t Tkv, const gdpa_bias* bias, int act, int causal,
                            int window, float scale, void* out, float* lse, void* workspace,
                            size_t ws_bytes, void* stream) {
  t_launches = 0;
  gdpa_status st = check_common(q, q_offsets, k, v, kv_offsets, B, H, d, Tq, Tkv, bias, act,
                                causal, window);
  if (st != GDPA_OK) return st;
  if (Tq > 0 && (out == nullptr || !aligned16(out))) return GDPA_ERR_INVALID_ARG;
  if (act == GDPA_ACT_SOFTMAX && Tq > 0 && lse == nullptr) return GDPA_ERR_INVALID_ARG;
  const size_t need = gdpa_fwd_workspace_size(B, H, d, Tq, Tkv);
  if (workspace == nullptr || ws_bytes < need || !aligned16(workspace)) return GDPA_ERR_WORKSPACE;
  if (Tq == 0 || B == 0) return GDPA_OK;

  DeviceInfo* dev = nullptr;
  if (device_info(&dev) != cudaSuccess) return GDPA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  int max_rel = 1;
  const float* table = bias_table(bias, &max_rel);
  const int64_t* dense_off = is_dense(bias) ? bias->offsets : nullptr;
  CUtensorMap tq, tk, tv;
  if (!make_thd_map(&tq, q, Tq, H, d, kHalfRows)) return GDPA_ERR_INVALID_ARG;
  // With no key rows at all there is nothing to load; any valid map will do.
  const void* kb = Tkv > 0 ? k : q;
  const void* vb = Tkv > 0 ? v : q;
  const int64_t Tk = Tkv > 0 ? Tkv : Tq;
  if (!make_thd_map(&tk, kb, Tk, H, d, kKvRows)) return GDPA_ERR_INVALID_ARG;
  if (!make_thd_map(&tv, vb, Tk, H, d, kKvRows)) return GDPA_ERR_INVALID_ARG;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* n_items = reinterpret_cast<int*>(ws);
  int* ticket = reinterpret_cast<int*>(ws + 4);
  int2* items = reinterpret_cast<int2*>(ws + 256);
  // Samples with at most kShortQ queries go to the short-query kernel, samples
  // with more queries and at most kShortKv keys to the short-key kernel (GDPA
  // activations without mask or bias: the PMA and cross-attention shapes).
  ShortList sq;
  KvList kvl;
  CUtensorMap tq_short;
  if (act != GDPA_ACT_SOFTMAX && !causal && window == 0 && bias_kind(bias) == GDPA_BIAS_NONE) {
    if (!make_thd_map(&tq_short, q, Tq, H, d, kShortQ)) return GDPA_ERR_INVALID_ARG;
    const size_t sq_off = 256 + align_up(static_cast<size_t>(max_fwd_items(B, H, Tq)) * sizeof(int2), 256);
    sq.max_q = kShortQ;
    sq.items = reinterpret_cast<int2*>(ws + sq_off);
    sq.n_items = reinterpret_cast<int*>(ws + 8);
    sq.ticket = reinterpret_cast<int*>(ws + 12);
    sq.all_short = reinterpret_cast<int*>(ws + 16);
    kvl.max_kv = kShortKv;
    kvl.items = reinterpret_cast<int2*>(ws + sq_off + align_up(static_cast<size_t>(B) * H * sizeof(int2), 256));
    kvl.n_items = reinterpret_cast<int*>(ws + 20);
    kvl.ticket = reinterpret_cast<int*>(ws + 24);
  }

  if (launch_build_worklist(q_offsets, kv_offsets, B, H, Tq, Tkv, causal, window, 0, items,
                            n_items, ticket, dev->status, s, dense_off, sq, kvl) != cudaSuccess)
    return GDPA_ERR_CUDA;
  ++t_launches;

  FwdParams p{};
  p.qo = q_offsets;
  p.ko = kv_offsets;
  p.B = B;
  p.H = H;
  p.d = d;
  p.Tq = Tq;
  p.Tkv = Tkv;
  p.bias_table = table;
  p.max_rel = max_rel;
  p.causal = causal;
  p.window = window;
  p.scale = scale;
  p.bias_dense = dense_off != nullptr ? bias->table : nullptr;
  p.bias_off = dense_off;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.items = items;
  p.n_items = n_items;
  p.ticket = ticket;
  p.status = dev->status;
  const int64_t max_items = max_fwd_items(B, H, Tq);
  const int grid = static_cast<int>(max_items < dev->sms ? max_items : dev->sms);
  cudaEvent_t ea = nullptr, eb = nullptr;
  const bool timed = timing_slot(0, &ea, &eb);
  if (timed && cudaEventRecord(ea, s) != cudaSuccess) return GDPA_ERR_CUDA;
  if (launch_fwd(p, act, tq, tk, tv, grid, s) != cudaSuccess) return GDPA_ERR_CUDA;
  ++t_launches;
  if (sq.items != nullptr) {
    // the short-query items (an empty list makes the kernel return at once)
    FwdParams ps = p;
    ps.items = sq.items;
    ps.n_items = sq.n_items;
    ps.ticket = sq.ticket;
    const int64_t n_sq = static_cast<int64_t>(B) * H;
    const int grid_sq = static_cast<int>(n_sq < dev->sms ? n_sq : dev->sms);
    if (launch_fwd_short_q(ps, act, tq_short, tk, tv, grid_sq, s) != cudaSuccess)
      return GDPA_ERR_CUDA;
    ++t_launches;
  }
  if (kvl.items != nullptr) {
    // the short-key items (an empty list makes the kernel return at once)
    FwdParams pk = p;
    pk.items = kvl.items;
    pk.n_items = kvl.n_items;
    pk.ticket = kvl.ticket;
    const int64_t n_kv = max_kv_items(B, H, Tq);
    const int grid_kv = static_cast<int>(n_kv < dev->sms ? (n_kv > 0 ? n_kv : 1) : dev->sms);
    if (launch_fwd_short_kv(pk, act, tq, tk, tv, grid_kv, s) != cudaSuccess) return GDPA_ERR_CUDA;
    ++t_launches;
  }
  if (timed && cudaEventRecord(eb, s) != cudaSuccess) return GDPA_ERR_CUDA;
  return GDPA_OK;
}

size_t gdpa_bwd_workspace_size(int B, int H, int d, int64_t Tq, int64_t Tkv) {
  if (B < 0 || H <= 0 || Tq < 0 || Tkv < 0) return 0;
  size_t sz = 256;
  sz += align_up(static_cast<size_t>(max_bwd_items(B, H, Tkv)) * sizeof(int2), 256);
  sz += align_up(static_cast<size_t>(Tq) * H * d * sizeof(float), 256);  // dQ accumulator
  sz += align_up(static_cast<size_t>(Tq) * H * sizeof(float), 256);      // D = rowsum(dO*O)
  sz += align_up(static_cast<size_t>(B) * H * sizeof(int2), 256);        // short-query list
  return sz;
}

gdpa_status gdpa_bwd(const void* q, const int32_t* q_offsets, const void* k, const void* v,
                     const int32_t* kv_offsets, int B, int H, int d, int64_t Tq, int64_t Tkv,
                     const gdpa_bias* bias, int act, int causal, float scale, const void* out,
                     const float* lse, const void* dout, void* dq, void* dk, void* dv,
                     void* workspace, size_t ws_bytes, void* stream) {
  return gdpa_bwd_window(q, q_offsets, k, v, kv_offsets, B, H, d, Tq, Tkv, bias, act, causal, 0,
                         scale, out, lse, dout, dq, dk, dv, nullptr, workspace, ws_bytes, stream);
}

gdpa_status gdpa_bwd_window(const void* q, const int32_t* q_offsets, const void* k,
                            const void* v, const int32_t* kv_offsets, int B, int H, int d,
                            int64_t Tq, int64_t Tkv, const gdpa_bias* bias, int act, int causal,
                            int window, float scale, const void* out, const float* lse,
                            const void* dout, void* dq, void* dk, void* dv, float* dbias,
                            void* workspace, size_t ws_bytes, void* stream) {
  return gdpa_bwd_rope(q, q_offsets, k, v, kv_offsets, B, H, d, Tq, Tkv, bias, act, causal, window,
                       scale, 0.0f, out, lse, dout, dq, dk, dv, dbias, workspace, ws_bytes, stream);
}

gdpa_status gdpa_bwd_rope(const void* q, const int32_t* q_offsets, const void* k, const void* v,
                          const int32_t* kv_offsets, int B, int H, int d, int64_t Tq,
                          int64_t Tkv, const gdpa_bias* bias, int act, int causal, int window,
                          float scale, float rope_base, const void* out, const float* lse,
                          const void* dout, void* dq, void* dk, void* dv, float* dbias,
                          void* workspace, size_t ws_bytes, void* stream) {
  t_launches = 0;
  if (!(rope_base >= 0.0f) || rope_base == INFINITY) return GDPA_ERR_INVALID_ARG;  // NaN too
  gdpa_status st = check_common(q, q_offsets, k, v, kv_offsets, B, H, d, Tq, Tkv, bias, act,
                                causal, window);
  if (st != GDPA_OK) return st;
  if (dbias != nullptr) {
    // the gradient of a bias needs that bias (a relative-position table or a dense bias)
    if (bias_kind(bias) == GDPA_BIAS_NONE) return GDPA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(dbias) & 3u) return GDPA_ERR_INVALID_ARG;
  }
  if (Tq > 0 && (dout == nullptr || dq == nullptr || !aligned16(dout) || !aligned16(dq)))
    return GDPA_ERR_INVALID_ARG;
  if (Tkv > 0 && (dk == nullptr || dv == nullptr || !aligned16(dk) || !aligned16(dv)))
    return GDPA_ERR_INVALID_ARG;
  if (act == GDPA_ACT_SOFTMAX && Tq > 0 && (out == nullptr || lse == nullptr || !aligned16(out)))
    return GDPA_ERR_INVALID_ARG;
  const size_t need = gdpa_bwd_workspace_size(B, H, d, Tq, Tkv);
  if (workspace == nullptr || ws_bytes < need || !aligned16(workspace)) return GDPA_ERR_WORKSPACE;
  if (B == 0 || (Tq == 0 && Tkv == 0)) return GDPA_OK;

  DeviceInfo* dev = nullptr;
  if (device_info(&dev) != cudaSuccess) return GDPA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  int max_rel = 1;
  const float* table = bias_table(bias, &max_rel);
  const int64_t* dense_off = is_dense(bias) ? bias->offsets : nullptr;
  // Maps need at least one row; an empty side is never loaded, so any
  // valid tensor stands in for it.
  const void* qb = Tq > 0 ? q : k;
  const void* dob = Tq > 0 ? dout : k;
  const int64_t Tqm = Tq > 0 ? Tq : Tkv;
  const void* kb = Tkv > 0 ? k : q;
  const void* vb = Tkv > 0 ? v : q;
  const int64_t Tkm = Tkv > 0 ? Tkv : Tq;
  // The softmax kernel streams 128-query tiles, the general kernel 64-query
  // tiles; both reduce dQ in [16 queries x 32 channels] boxes, one warp's
  // channels each.
  const bool sm = act == GDPA_ACT_SOFTMAX;
  const int q_rows = sm ? kBwdSmQRows : kBwdQRows;
  CUtensorMap tq, tk, tv, tdo;
  if (!make_thd_map(&tq, qb, Tqm, H, d, q_rows) || !make_thd_map(&tdo, dob, Tqm, H, d, q_rows) ||
      !make_thd_map(&tk, kb, Tkm, H, d, kBwdKvRows) || !make_thd_map(&tv, vb, Tkm, H, d, kBwdKvRows))
    return GDPA_ERR_INVALID_ARG;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* n_items = reinterpret_cast<int*>(ws);
  int* ticket = reinterpret_cast<int*>(ws + 4);
  size_t off = 256;
  int2* items = reinterpret_cast<int2*>(ws + off);
  off += align_up(static_cast<size_t>(max_bwd_items(B, H, Tkv)) * sizeof(int2), 256);
  float* dq_acc = reinterpret_cast<float*>(ws + off);
  off += align_up(static_cast<size_t>(Tq) * H * d * sizeof(float), 256);
  float* delta = reinterpret_cast<float*>(ws + off);
  off += align_up(static_cast<size_t>(Tq) * H * sizeof(float), 256);
  // Without query rows there is nothing to reduce into; any valid map will do.
  CUtensorMap tdq;
  if (!make_dq_map(&tdq, Tq > 0 ? static_cast<void*>(dq_acc) : ws, Tq > 0 ? Tq : 1, H, d,
                   32, kBwdSmDqRows))
    return GDPA_ERR_INVALID_ARG;
  // Samples with at most kShortQ queries go to the short-query kernel (no
  // mask, bias, bias gradient or rotary backward).
  ShortList sql;
  ShortBwd sqb;
  const bool short_q = Tq > 0 && !causal && window == 0 && bias_kind(bias) == GDPA_BIAS_NONE &&
                       dbias == nullptr && rope_base == 0.0f;
  if (short_q) {
    if (!make_thd_map(&sqb.tq, q, Tq, H, d, kShortQ) ||
        !make_thd_map(&sqb.tdo, dout, Tq, H, d, kShortQ))
      return GDPA_ERR_INVALID_ARG;
    sql.max_q = kShortQ;
    sql.items = reinterpret_cast<int2*>(ws + off);
    sql.n_items = reinterpret_cast<int*>(ws + 8);
    sql.ticket = reinterpret_cast<int*>(ws + 12);
    sql.all_short = reinterpret_cast<int*>(ws + 16);
  }

  if (launch_build_worklist(kv_offsets, q_offsets, B, H, Tkv, Tq, causal, window, 1, items,
                            n_items, ticket, dev->status, s, dense_off, sql) != cudaSuccess)
    return GDPA_ERR_CUDA;
  ++t_launches;

  BwdParams p{};
  p.qo = q_offsets;
  p.ko = kv_offsets;
  p.B = B;
  p.H = H;
  p.d = d;
  p.Tq = Tq;
  p.Tkv = Tkv;
  p.bias_table = table;
  p.max_rel = max_rel;
  p.causal = causal;
  p.window = window;
  p.scale = scale;
  p.bias_dense = dense_off != nullptr ? bias->table : nullptr;
  p.bias_off = dense_off;
  p.out = static_cast<const __nv_bfloat16*>(out);
  p.lse = lse;
  p.dout = static_cast<const __nv_bfloat16*>(dout);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.dbias = dbias;
  p.rope_base = rope_base;
  p.dq_acc = dq_acc;
  p.delta = delta;
  p.items = items;
  p.n_items = n_items;
  p.ticket = ticket;
  p.status = dev->status;
  p.all_short = sql.all_short;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  // GDPA without the rotary backward: samples whose keys fit one key block get
  // their dQ written once, in bf16, by the main kernel
  p.dq_direct_kv = (act != GDPA_ACT_SOFTMAX && rope_base == 0.0f) ? kBwdKvRows : 0;
  p.short_q_max = short_q ? kShortQ : 0;
  if (short_q) {
    sqb.p = p;
    sqb.p.items = sql.items;
    sqb.p.n_items = sql.n_items;
    sqb.p.ticket = sql.ticket;
    sqb.dq = dq;
    const int64_t n_sq = static_cast<int64_t>(B) * H;
    sqb.grid = static_cast<int>(n_sq < dev->sms ? n_sq : dev->sms);
  }
  const int64_t max_items = max_bwd_items(B, H, Tkv);
  const int grid = static_cast<int>(max_items < dev->sms ? (max_items > 0 ? max_items : 1) : dev->sms);
  int launches = 0;
  cudaEvent_t ea = nullptr, eb = nullptr;
  const bool timed = timing_slot(1, &ea, &eb);
  cudaError_t e = launch_bwd(p, act, tq, tk, tv, tdo, tdq, grid, s, &launches,
                             timed ? ea : nullptr, timed ? eb : nullptr, short_q ? &sqb : nullptr);
  t_launches += launches;
  if (e != cudaSuccess) return GDPA_ERR_CUDA;
  if (Tq > 0) {
    const cudaError_t ce =
        rope_base > 0.0f
            ? launch_dq_convert_rope(dq_acc, dq, q_offsets, B, Tq, H, d, scale, rope_base, s)
            : launch_dq_convert(dq_acc, dq, static_cast<long long>(Tq) * H * d, scale, s,
                                p.all_short, &p);
    if (ce != cudaSuccess) return GDPA_ERR_CUDA;
    ++t_launches;
  }
  return GDPA_OK;
}

size_t gdpa_block_workspace_size(int B, int H, int d, int64_t T) {
  (void)H;
  (void)d;
  if (B < 0 || T < 0) return 0;
  return 256 + align_up(static_cast<size_t>(max_block_tiles(B, T)) * sizeof(int4), 256);
}

gdpa_status gdpa_block_fwd(const void* q, const int32_t* offsets, const void* k, const void* v,
                           int B, int H, int d, int64_t T, const gdpa_bias* bias, int act,
                           int causal, float scale, void* out, void* workspace, size_t ws_bytes,
                           void* stream) {
  t_launches = 0;
  gdpa_status st = check_common(q, offsets, k, v, offsets, B, H, d, T, T, bias, act, causal, 0);
  if (st != GDPA_OK) return st;
  if (T > 0 && (out == nullptr || !aligned16(out))) return GDPA_ERR_INVALID_ARG;
  const size_t need = gdpa_block_workspace_size(B, H, d, T);
  if (workspace == nullptr || ws_bytes < need || !aligned16(workspace)) return GDPA_ERR_WORKSPACE;
  if (T == 0 || B == 0) return GDPA_OK;
  DeviceInfo* dev = nullptr;
  if (device_info(&dev) != cudaSuccess) return GDPA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int max_rel = 1;
  const float* table = bias_table(bias, &max_rel);
  CUtensorMap tq, tk, tv;
  if (!make_thd_map(&tq, q, T, H, d, 2 * kBlockRows) ||
      !make_thd_map(&tk, k, T, H, d, 2 * kBlockRows) ||
      !make_thd_map(&tv, v, T, H, d, 2 * kBlockRows))
    return GDPA_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* n_tiles = reinterpret_cast<int*>(ws);
  int4* tiles = reinterpret_cast<int4*>(ws + 256);
  const int64_t* dense_off = is_dense(bias) ? bias->offsets : nullptr;
  if (launch_block_list(offsets, B, T, tiles, n_tiles, dev->status, s, dense_off, H) !=
      cudaSuccess)
    return GDPA_ERR_CUDA;
  ++t_launches;
  BlockParams p{};
  p.tiles = tiles;
  p.n_tiles = n_tiles;
  p.H = H;
  p.d = d;
  p.T = T;
  p.bias_table = table;
  p.max_rel = max_rel;
  p.causal = causal;
  p.scale = scale;
  p.bias_dense = dense_off != nullptr ? bias->table : nullptr;
  p.bias_off = dense_off;
  p.offsets = offsets;
  p.B = B;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.status = dev->status;
  const int64_t max_items = max_block_tiles(B, T) * H;
  const int grid = static_cast<int>(max_items < dev->sms ? max_items : dev->sms);
  cudaEvent_t ea = nullptr, eb = nullptr;
  const bool timed = timing_slot(0, &ea, &eb);
  if (timed && cudaEventRecord(ea, s) != cudaSuccess) return GDPA_ERR_CUDA;
  if (launch_block_fwd(p, act, tq, tk, tv, grid, s) != cudaSuccess) return GDPA_ERR_CUDA;
  if (timed && cudaEventRecord(eb, s) != cudaSuccess) return GDPA_ERR_CUDA;
  ++t_launches;
  return GDPA_OK;
}

gdpa_status gdpa_block_bwd(const void* q, const int32_t* offsets, const void* k, const void* v,
                           int B, int H, int d, int64_t T, const gdpa_bias* bias, int act,
                           int causal, float scale, float rope_base, const void* dout, void* dq,
                           void* dk, void* dv, void* workspace, size_t ws_bytes, void* stream) {
  return gdpa_block_bwd_dbias(q, offsets, k, v, B, H, d, T, bias, act, causal, scale, rope_base,
                              dout, dq, dk, dv, nullptr, workspace, ws_bytes, stream);
}

gdpa_status gdpa_block_bwd_dbias(const void* q, const int32_t* offsets, const void* k,
                                 const void* v, int B, int H, int d, int64_t T,
                                 const gdpa_bias* bias, int act, int causal, float scale,
                                 float rope_base, const void* dout, void* dq, void* dk, void* dv,
                                 float* dbias, void* workspace, size_t ws_bytes, void* stream) {
  t_launches = 0;
  gdpa_status st = check_common(q, offsets, k, v, offsets, B, H, d, T, T, bias, act, causal, 0);
  if (st != GDPA_OK) return st;
  if (dbias != nullptr) {  // the gradient of a bias needs that bias (a table or a dense bias)
    if (bias_kind(bias) == GDPA_BIAS_NONE) return GDPA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(dbias) & 3u) return GDPA_ERR_INVALID_ARG;
  }
  if (!(rope_base >= 0.0f) || rope_base > 3.0e38f) return GDPA_ERR_INVALID_ARG;  // NaN, < 0, inf
  if (T > 0 && (dout == nullptr || dq == nullptr || dk == nullptr || dv == nullptr ||
                !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv)))
    return GDPA_ERR_INVALID_ARG;
  const size_t need = gdpa_block_workspace_size(B, H, d, T);
  if (workspace == nullptr || ws_bytes < need || !aligned16(workspace)) return GDPA_ERR_WORKSPACE;
  if (T == 0 || B == 0) return GDPA_OK;
  DeviceInfo* dev = nullptr;
  if (device_info(&dev) != cudaSuccess) return GDPA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int max_rel = 1;
  const float* table = bias_table(bias, &max_rel);
  CUtensorMap maps[7];
  const void* bases[7] = {q, k, v, dout, dq, dk, dv};
  for (int i = 0; i < 7; ++i)
    if (!make_thd_map(&maps[i], bases[i], T, H, d, 2 * kBlockRows)) return GDPA_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* n_tiles = reinterpret_cast<int*>(ws);
  int4* tiles = reinterpret_cast<int4*>(ws + 256);
  const int64_t* dense_off = is_dense(bias) ? bias->offsets : nullptr;
  if (launch_block_list(offsets, B, T, tiles, n_tiles, dev->status, s, dense_off, H) !=
      cudaSuccess)
    return GDPA_ERR_CUDA;
  ++t_launches;
  BlockParams p{};
  p.tiles = tiles;
  p.n_tiles = n_tiles;
  p.H = H;
  p.d = d;
  p.T = T;
  p.bias_table = table;
  p.max_rel = max_rel;
  p.causal = causal;
  p.scale = scale;
  p.bias_dense = dense_off != nullptr ? bias->table : nullptr;
  p.bias_off = dense_off;
  p.offsets = offsets;
  p.B = B;
  p.dout = static_cast<const __nv_bfloat16*>(dout);
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.rope_base = rope_base;
  p.dbias = dbias;
  p.status = dev->status;
  const int64_t max_items = max_block_tiles(B, T) * H;
  const int grid = static_cast<int>(max_items < dev->sms ? max_items : dev->sms);
  cudaEvent_t ea = nullptr, eb = nullptr;
  const bool timed = timing_slot(1, &ea, &eb);
  if (timed && cudaEventRecord(ea, s) != cudaSuccess) return GDPA_ERR_CUDA;
  if (launch_block_bwd(p, act, maps, grid, s) != cudaSuccess) return GDPA_ERR_CUDA;
  if (timed && cudaEventRecord(eb, s) != cudaSuccess) return GDPA_ERR_CUDA;
  ++t_launches;
  return GDPA_OK;
}

size_t gdpa_mxfp8_scale_bytes(int B, int H, int d, int64_t T, int mode) {
  if (B < 0 || H <= 0 || T < 0 || (d != 64 && d != 128)) return 0;
  if ((mode & ~(GDPA_MX_ALONG_TOKENS | GDPA_MX_NOSAT)) != 0) return 0;
  if ((mode & GDPA_MX_ALONG_TOKENS) == 0) return static_cast<size_t>(T) * H * (d / 32);
  return (static_cast<size_t>(B) + T / 32 + 1) * H * d;
}

gdpa_status gdpa_quantize_mxfp8(const void* x, const int32_t* offsets, int B, int H, int d,
                                int64_t T, int mode, void* codes, void* scales, void* stream) {
  t_launches = 0;
  if (B < 0 || H <= 0 || T < 0) return GDPA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return GDPA_ERR_UNSUPPORTED;
  if ((mode & ~(GDPA_MX_ALONG_TOKENS | GDPA_MX_NOSAT)) != 0) return GDPA_ERR_INVALID_ARG;
  const bool tokens = (mode & GDPA_MX_ALONG_TOKENS) != 0;
  const bool nosat = (mode & GDPA_MX_NOSAT) != 0;
  if (T == 0) return GDPA_OK;
  if (x == nullptr || codes == nullptr || scales == nullptr || !aligned16(x) || !aligned16(codes))
    return GDPA_ERR_INVALID_ARG;
  if (tokens && offsets == nullptr) return GDPA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = !tokens ? launch_quant_rows(x, T * H, d, codes, scales, s, nosat)
                          : launch_quant_tokens(x, offsets, B, H, d, T, codes, scales, s, nosat);
  if (e != cudaSuccess) return GDPA_ERR_CUDA;
  ++t_launches;
  return GDPA_OK;
}

gdpa_status gdpa_fwd_mxfp8(const void* q_codes, const void* q_scales, const int32_t* q_offsets,
                           const void* k_codes, const void* k_scales, const void* v_codes,
                           const void* v_scales, const int32_t* kv_offsets, int B, int H, int d,
                           int64_t Tq, int64_t Tkv, const gdpa_bias* bias, int act, int causal,
                           float scale, void* out, float* lse, void* workspace, size_t ws_bytes,
                           void* stream) {
  return gdpa_fwd_mxfp8_window(q_codes, q_scales, q_offsets, k_codes, k_scales, v_codes, v_scales,
                               kv_offsets, B, H, d, Tq, Tkv, bias, act, causal, 0, scale, out,
                               lse, workspace, ws_bytes, stream);
}

gdpa_status gdpa_fwd_mxfp8_window(const void* q_codes, const void* q_scales,
                                  const int32_t* q_offsets, const void* k_codes,
                                  const void* k_scales, const void* v_codes, const void* v_scales,
                                  const int32_t* kv_offsets, int B, int H, int d, int64_t Tq,
                                  int64_t Tkv, const gdpa_bias* bias, int act, int causal,
                                  int window, float scale, void* out, float* lse,
                                  void* workspace, size_t ws_bytes, void* stream) {
  t_launches = 0;
  gdpa_status st = check_common(q_codes, q_offsets, k_codes, v_codes, kv_offsets, B, H, d, Tq,
                                Tkv, bias, act, causal, window);
  if (st != GDPA_OK) return st;
  if (d != 128 || act != GDPA_ACT_SOFTMAX) return GDPA_ERR_UNSUPPORTED;
  if (Tq > 0 && (q_scales == nullptr || out == nullptr || lse == nullptr || !aligned16(out)))
    return GDPA_ERR_INVALID_ARG;
  if (Tkv > 0 && (k_scales == nullptr || v_scales == nullptr)) return GDPA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q_scales) & 3u) || (reinterpret_cast<uintptr_t>(k_scales) & 3u))
    return GDPA_ERR_INVALID_ARG;  // scale words are read as 32-bit
  const size_t need = gdpa_fwd_workspace_size(B, H, d, Tq, Tkv);
  if (workspace == nullptr || ws_bytes < need || !aligned16(workspace)) return GDPA_ERR_WORKSPACE;
  if (Tq == 0 || B == 0) return GDPA_OK;

  DeviceInfo* dev = nullptr;
  if (device_info(&dev) != cudaSuccess) return GDPA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int max_rel = 1;
  const float* table = bias_table(bias, &max_rel);
  CUtensorMap tq, tk, tv;
  if (!make_u8_map(&tq, q_codes, Tq, H, d, kHalfRows)) return GDPA_ERR_INVALID_ARG;
  const void* kb = Tkv > 0 ? k_codes : q_codes;
  const void* vb = Tkv > 0 ? v_codes : q_codes;
  const int64_t Tk = Tkv > 0 ? Tkv : Tq;
  if (!make_u8_map(&tk, kb, Tk, H, d, fwd_mx_tile_rows()) ||
      !make_u8_map(&tv, vb, Tk, H, d, fwd_mx_tile_rows()))
    return GDPA_ERR_INVALID_ARG;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* n_items = reinterpret_cast<int*>(ws);
  int* ticket = reinterpret_cast<int*>(ws + 4);
  int2* items = reinterpret_cast<int2*>(ws + 256);
  const int64_t* dense_off = is_dense(bias) ? bias->offsets : nullptr;
  if (launch_build_worklist(q_offsets, kv_offsets, B, H, Tq, Tkv, causal, window, 0, items,
                            n_items, ticket, dev->status, s, dense_off) != cudaSuccess)
    return GDPA_ERR_CUDA;
  ++t_launches;
  FwdParams p{};
  p.qo = q_offsets;
  p.ko = kv_offsets;
  p.B = B;
  p.H = H;
  p.d = d;
  p.Tq = Tq;
  p.Tkv = Tkv;
  p.bias_table = table;
  p.max_rel = max_rel;
  p.bias_dense = dense_off != nullptr ? bias->table : nullptr;
  p.bias_off = dense_off;
  p.causal = causal;
  p.window = window;
  p.scale = scale;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.items = items;
  p.n_items = n_items;
  p.ticket = ticket;
  p.status = dev->status;
  const int64_t max_items = max_fwd_items(B, H, Tq);
  const int grid = static_cast<int>(max_items < dev->sms ? max_items : dev->sms);
  const long long v_rows = static_cast<long long>(B) + Tkv / 32 + 1;
  cudaEvent_t ea = nullptr, eb = nullptr;
  const bool timed = timing_slot(0, &ea, &eb);
  if (timed && cudaEventRecord(ea, s) != cudaSuccess) return GDPA_ERR_CUDA;
  if (launch_fwd_mx(p, tq, tk, tv, static_cast<const uint8_t*>(q_scales),
                    static_cast<const uint8_t*>(k_scales), static_cast<const uint8_t*>(v_scales),
                    v_rows, grid, s) != cudaSuccess)
    return GDPA_ERR_CUDA;
  if (timed && cudaEventRecord(eb, s) != cudaSuccess) return GDPA_ERR_CUDA;
  ++t_launches;
  return GDPA_OK;
}

namespace {
// Carves the MXFP8 backward's workspace; returns the bytes it needs.
struct BwdMxLayout {
  size_t items, dq_acc, delta, qd, qt, dod, dot, kd, kt, vd, qd_sc, dod_sc, kd_sc, vd_sc, qt_sc,
      dot_sc, kt_sc, total;
};
BwdMxLayout bwd_mx_layout(int B, int H, int d, int64_t Tq, int64_t Tkv) {
  BwdMxLayout l{};
  size_t off = 256;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align_up(bytes, 256);
    return at;
  };
  const size_t hd = static_cast<size_t>(H) * d;
  l.items = take(static_cast<size_t>(max_bwd_items(B, H, Tkv)) * sizeof(int2));
  l.dq_acc = take(static_cast<size_t>(Tq) * hd * sizeof(float));
  l.delta = take(static_cast<size_t>(Tq) * H * sizeof(float));
  l.qd = take(static_cast<size_t>(Tq) * hd);
  l.qt = take(static_cast<size_t>(Tq) * hd);
  l.dod = take(static_cast<size_t>(Tq) * hd);
  l.dot = take(static_cast<size_t>(Tq) * hd);
  l.kd = take(static_cast<size_t>(Tkv) * hd);
  l.kt = take(static_cast<size_t>(Tkv) * hd);
  l.vd = take(static_cast<size_t>(Tkv) * hd);
  l.qd_sc = take(static_cast<size_t>(Tq) * H * (d / 32));
  l.dod_sc = take(static_cast<size_t>(Tq) * H * (d / 32));
  l.kd_sc = take(static_cast<size_t>(Tkv) * H * (d / 32));
  l.vd_sc = take(static_cast<size_t>(Tkv) * H * (d / 32));
  l.qt_sc = take((static_cast<size_t>(B) + Tq / 32 + 1) * hd);
  l.dot_sc = take((static_cast<size_t>(B) + Tq / 32 + 1) * hd);
  l.kt_sc = take((static_cast<size_t>(B) + Tkv / 32 + 1) * hd);
  l.total = off;
  return l;
}
}  // namespace

size_t gdpa_bwd_mxfp8_workspace_size(int B, int H, int d, int64_t Tq, int64_t Tkv) {
  if (B < 0 || H <= 0 || Tq < 0 || Tkv < 0 || (d != 64 && d != 128)) return 0;
  return bwd_mx_layout(B, H, d, Tq, Tkv).total;
}

gdpa_status gdpa_bwd_mxfp8(const void* q, const int32_t* q_offsets, const void* k, const void* v,
                           const int32_t* kv_offsets, int B, int H, int d, int64_t Tq,
                           int64_t Tkv, const gdpa_bias* bias, int act, int causal, float scale,
                           const void* out, const float* lse, const void* dout, void* dq, void* dk,
                           void* dv, void* workspace, size_t ws_bytes, void* stream) {
  return gdpa_bwd_mxfp8_window(q, q_offsets, k, v, kv_offsets, B, H, d, Tq, Tkv, bias, act, causal,
                               0, scale, out, lse, dout, dq, dk, dv, workspace, ws_bytes, stream);
}

gdpa_status gdpa_bwd_mxfp8_window(const void* q, const int32_t* q_offsets, const void* k,
                                  const void* v, const int32_t* kv_offsets, int B, int H, int d,
                                  int64_t Tq, int64_t Tkv, const gdpa_bias* bias, int act,
                                  int causal, int window, float scale, const void* out,
                                  const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                  void* workspace, size_t ws_bytes, void* stream) {
  return gdpa_bwd_mxfp8_rope(q, q_offsets, k, v, kv_offsets, B, H, d, Tq, Tkv, bias, act, causal,
                             window, scale, 0.0f, out, lse, dout, dq, dk, dv, nullptr, workspace,
                             ws_bytes, stream);
}

gdpa_status gdpa_bwd_mxfp8_rope(const void* q, const int32_t* q_offsets, const void* k,
                                const void* v, const int32_t* kv_offsets, int B, int H, int d,
                                int64_t Tq, int64_t Tkv, const gdpa_bias* bias, int act, int causal,
                                int window, float scale, float rope_base, const void* out,
                                const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                float* dbias, void* workspace, size_t ws_bytes, void* stream) {
  t_launches = 0;
  if (!(rope_base >= 0.0f) || rope_base == INFINITY) return GDPA_ERR_INVALID_ARG;  // NaN too
  gdpa_status st = check_common(q, q_offsets, k, v, kv_offsets, B, H, d, Tq, Tkv, bias, act,
                                causal, window);
  if (st != GDPA_OK) return st;
  if (d != 128 || act != GDPA_ACT_SOFTMAX) return GDPA_ERR_UNSUPPORTED;
  if (dbias != nullptr) {  // the gradient of a bias needs that bias (a table or a dense bias)
    if (bias_kind(bias) == GDPA_BIAS_NONE) return GDPA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(dbias) & 3u) return GDPA_ERR_INVALID_ARG;
  }
  if (Tq > 0 && (dout == nullptr || dq == nullptr || out == nullptr || lse == nullptr ||
                 !aligned16(dout) || !aligned16(dq) || !aligned16(out)))
    return GDPA_ERR_INVALID_ARG;
  if (Tkv > 0 && (dk == nullptr || dv == nullptr || !aligned16(dk) || !aligned16(dv)))
    return GDPA_ERR_INVALID_ARG;
  const BwdMxLayout lay = bwd_mx_layout(B, H, d, Tq, Tkv);
  if (workspace == nullptr || ws_bytes < lay.total || !aligned16(workspace)) return GDPA_ERR_WORKSPACE;
  if (B == 0 || (Tq == 0 && Tkv == 0)) return GDPA_OK;

  DeviceInfo* dev = nullptr;
  if (device_info(&dev) != cudaSuccess) return GDPA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto at = [&](size_t off) { return static_cast<void*>(ws + off); };

  // 1) operand codes and scales: Q, K, dO along channels and along tokens, V along channels
  if (Tq > 0) {
    if (launch_quant_rows(q, Tq * H, d, at(lay.qd), at(lay.qd_sc), s) != cudaSuccess ||
        launch_quant_tokens(q, q_offsets, B, H, d, Tq, at(lay.qt), at(lay.qt_sc), s) != cudaSuccess ||
        launch_quant_rows(dout, Tq * H, d, at(lay.dod), at(lay.dod_sc), s) != cudaSuccess ||
        launch_quant_tokens(dout, q_offsets, B, H, d, Tq, at(lay.dot), at(lay.dot_sc), s) != cudaSuccess)
      return GDPA_ERR_CUDA;
    t_launches += 4;
  }
  if (Tkv > 0) {
    if (launch_quant_rows(k, Tkv * H, d, at(lay.kd), at(lay.kd_sc), s) != cudaSuccess ||
        launch_quant_tokens(k, kv_offsets, B, H, d, Tkv, at(lay.kt), at(lay.kt_sc), s) != cudaSuccess ||
        launch_quant_rows(v, Tkv * H, d, at(lay.vd), at(lay.vd_sc), s) != cudaSuccess)
      return GDPA_ERR_CUDA;
    t_launches += 3;
  }

  // 2) TMA maps over the codes (an empty side is never loaded; any valid tensor stands in)
  const int64_t Tqm = Tq > 0 ? Tq : Tkv;
  const int64_t Tkm = Tkv > 0 ? Tkv : Tq;
  const size_t qsrc[4] = {lay.qd, lay.qt, lay.dod, lay.dot};
  const size_t ksrc[3] = {lay.kd, lay.kt, lay.vd};
  CUtensorMap maps[8];
  for (int i = 0; i < 4; ++i)
    if (!make_u8_map(&maps[i], at(Tq > 0 ? qsrc[i] : ksrc[0]), Tqm, H, d, kBwdMxQRows))
      return GDPA_ERR_INVALID_ARG;
  for (int i = 0; i < 3; ++i)
    if (!make_u8_map(&maps[4 + i], at(Tkv > 0 ? ksrc[i] : qsrc[0]), Tkm, H, d, kBwdKvRows))
      return GDPA_ERR_INVALID_ARG;
  float* dq_acc = reinterpret_cast<float*>(ws + lay.dq_acc);
  if (!make_dq_map(&maps[7], Tq > 0 ? static_cast<void*>(dq_acc) : ws, Tq > 0 ? Tq : 1, H, d, d,
                   kBwdSmDqRows))
    return GDPA_ERR_INVALID_ARG;

  // 3) work list of 128-key blocks
  int* n_items = reinterpret_cast<int*>(ws);
  int* ticket = reinterpret_cast<int*>(ws + 4);
  int2* items = reinterpret_cast<int2*>(ws + lay.items);
  const int64_t* dense_off = is_dense(bias) ? bias->offsets : nullptr;
  if (launch_build_worklist(kv_offsets, q_offsets, B, H, Tkv, Tq, causal, window, 1, items,
                            n_items, ticket, dev->status, s, dense_off) != cudaSuccess)
    return GDPA_ERR_CUDA;
  ++t_launches;

  int max_rel = 1;
  const float* table = bias_table(bias, &max_rel);
  BwdParams p{};
  p.qo = q_offsets;
  p.ko = kv_offsets;
  p.B = B;
  p.H = H;
  p.d = d;
  p.Tq = Tq;
  p.Tkv = Tkv;
  p.bias_table = table;
  p.max_rel = max_rel;
  p.bias_dense = dense_off != nullptr ? bias->table : nullptr;
  p.bias_off = dense_off;
  p.causal = causal;
  p.window = window;
  p.scale = scale;
  p.out = static_cast<const __nv_bfloat16*>(out);
  p.lse = lse;
  p.dout = static_cast<const __nv_bfloat16*>(dout);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.dq_acc = dq_acc;
  p.dbias = dbias;
  p.rope_base = rope_base;
  p.delta = reinterpret_cast<float*>(ws + lay.delta);
  p.items = items;
  p.n_items = n_items;
  p.ticket = ticket;
  p.status = dev->status;
  // 4) zero the dQ accumulator, D = rowsum(dO * O) from the bf16 tensors
  if (Tq > 0) {
    if (launch_bwd_preprocess(p, true, s) != cudaSuccess) return GDPA_ERR_CUDA;
    ++t_launches;
  }
  BwdMxOperands mx{};
  mx.qd_sc = ws + lay.qd_sc;
  mx.kd_sc = ws + lay.kd_sc;
  mx.vd_sc = ws + lay.vd_sc;
  mx.dod_sc = ws + lay.dod_sc;
  mx.qt_sc = ws + lay.qt_sc;
  mx.kt_sc = ws + lay.kt_sc;
  mx.dot_sc = ws + lay.dot_sc;
  const int64_t max_items = max_bwd_items(B, H, Tkv);
  const int grid = static_cast<int>(max_items < dev->sms ? (max_items > 0 ? max_items : 1) : dev->sms);
  cudaEvent_t ea = nullptr, eb = nullptr;
  const bool timed = timing_slot(1, &ea, &eb);
  if (timed && cudaEventRecord(ea, s) != cudaSuccess) return GDPA_ERR_CUDA;
  if (launch_bwd_mx(p, mx, maps, grid, s) != cudaSuccess) return GDPA_ERR_CUDA;
  if (timed && cudaEventRecord(eb, s) != cudaSuccess) return GDPA_ERR_CUDA;
  ++t_launches;
  // 5) dQ = bf16(scale * accumulator), rotated back through the rotary embedding if asked
  if (Tq > 0) {
    const cudaError_t ce =
        rope_base > 0.0f
            ? launch_dq_convert_rope(dq_acc, dq, q_offsets, B, Tq, H, d, scale, rope_base, s)
            : launch_dq_convert(dq_acc, dq, static_cast<long long>(Tq) * H * d, scale, s);
    if (ce != cudaSuccess) return GDPA_ERR_CUDA;
    ++t_launches;
  }
  return GDPA_OK;
}

gdpa_status gdpa_selftest_timeout(int limit_us, void* stream) {
  t_launches = 0;
  if (limit_us < 1 || limit_us > 1000000) return GDPA_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  if (device_info(&dev) != cudaSuccess) return GDPA_ERR_CUDA;
  selftest_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      dev->status, static_cast<unsigned long long>(limit_us) * 1000ull);
  if (cudaGetLastError() != cudaSuccess) return GDPA_ERR_CUDA;
  ++t_launches;
  return GDPA_OK;
}

gdpa_status gdpa_get_device_status(void* stream) {
  DeviceInfo* dev = nullptr;
  if (device_info(&dev) != cudaSuccess) return GDPA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return GDPA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, dev->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return GDPA_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return GDPA_ERR_CUDA;
  }
  return static_cast<gdpa_status>(v);
}

const char* gdpa_status_string(int status) {
  switch (status) {
    case GDPA_OK: return "GDPA_OK";
    case GDPA_ERR_INVALID_ARG: return "GDPA_ERR_INVALID_ARG";
    case GDPA_ERR_UNSUPPORTED: return "GDPA_ERR_UNSUPPORTED";
    case GDPA_ERR_WORKSPACE: return "GDPA_ERR_WORKSPACE";
    case GDPA_ERR_CUDA: return "GDPA_ERR_CUDA";
    case GDPA_ERR_TIMEOUT: return "GDPA_ERR_TIMEOUT";
    case GDPA_ERR_BAD_OFFSETS: return "GDPA_ERR_BAD_OFFSETS";
    default: return "GDPA_ERR_UNKNOWN";
  }
}

int gdpa_last_launch_count(void) { return t_launches; }

gdpa_status gdpa_timing_enable(int enable) {
  if (t_timing == nullptr) t_timing = new TimingRing();
  if (enable) t_timing->n = 0;
  t_timing->enabled = enable != 0;
  return GDPA_OK;
}

int gdpa_timing_collect(float* ms, int* kind, int max) {
  TimingRing* r = t_timing;
  if (r == nullptr) return 0;
  const int n = r->n < max ? r->n : max;
  for (int i = 0; i < n; ++i) {
    if (cudaEventSynchronize(r->ev[2 * i + 1]) != cudaSuccess) return -1;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r->ev[2 * i], r->ev[2 * i + 1]) != cudaSuccess) return -1;
    if (ms != nullptr) ms[i] = t;
    if (kind != nullptr) kind[i] = r->kind[i];
  }
  return n;
}

}  // extern "C"
