// Forward pass for callers that cannot allocate device memory.
//
// gdpa_fwd needs a caller-provided workspace (the scheduler's work list).
// Some callers have no way to provide one: a plugin running inside a host
// framework that has already reserved the device memory for its own pool,
// or a fixed-budget service whose memory plan forbids allocations after
// start-up.  gdpa_fwd_noalloc serves them from a scratch array that is part
// of this library's image: a file-scope __device__ array of
// kNoAllocScratchBytes (1 MiB) that every GPU which loads the library holds
// until the process exits.
//
// In host code the array's name only stands for the device symbol; its
// device address is looked up once per device with cudaGetSymbolAddress and
// cached.  That look-up happens inside the first call on each device, so the
// first call on a device should come before any stream capture.
//
// Every call shares the one array and leaves the last call's work list in
// it; the scheduler kernel rewrites the item count and resets the ticket on
// every call, so nothing has to start at zero.  Calls whose kernels overlap
// on the GPU (different streams, or different host threads) race on the
// array and produce undefined outputs: serialise them.
#include <mutex>

#include "common.cuh"

namespace gdpa {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

}  // namespace
}  // namespace gdpa

extern "C" gdpa_status gdpa_fwd_noalloc(const void* q, const int32_t* q_offsets, const void* k,
                                        const void* v, const int32_t* kv_offsets, int B, int H,
                                        int d, int64_t Tq, int64_t Tkv, const gdpa_bias* bias,
                                        int act, int causal, float scale, void* out, float* lse,
                                        void* stream) {
  using namespace gdpa;
  // Sizes the static scratch cannot hold are refused before anything runs.
  const size_t need = gdpa_fwd_workspace_size(B, H, d, Tq, Tkv);
  if (need > kNoAllocScratchBytes) return GDPA_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDPA_ERR_CUDA;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
        return GDPA_ERR_CUDA;
      g_scratch_addr[dev] = p;
    }
    scratch = g_scratch_addr[dev];
  }
  return gdpa_fwd(q, q_offsets, k, v, kv_offsets, B, H, d, Tq, Tkv, bias, act, causal, scale,
                  out, lse, scratch, kNoAllocScratchBytes, stream);
}
