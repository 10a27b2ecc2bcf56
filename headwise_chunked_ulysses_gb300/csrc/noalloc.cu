// upipe_attention_bwd_noalloc: the attention backward entry point for callers
// that cannot allocate device memory.
//
// Some callers of this library have no way to obtain a scratch buffer: a host
// that reserves all device memory up front and hands out only the tensors it
// owns (a fixed-budget inference or training engine), a plugin running inside
// another framework's operator that forbids allocations on its call path, or
// code that must not call cudaMalloc because it synchronises the device and
// would stall other work.  upipe_attention_bwd needs 8*n_q*S bytes of scratch
// (the per-row D = rowsum(dO*O) and the log2-domain lse); this variant takes
// that scratch from a fixed array compiled into the library instead, so the
// caller passes only inputs and outputs.
//
// The array lives in device memory of every GPU that loads the library, for
// the life of the process.  All calls on a device share it: two calls whose
// work overlaps on the GPU (different streams, or different host threads)
// race on it.  Calls ordered on one stream are safe.  Nothing in it needs to
// start at zero: the backward's preprocessing writes every scratch entry it
// later reads, and zeroes the dQ output itself.
//
// Host code cannot use the array's name as a device address (in host code it
// names a host-side stand-in), so the first call on each device resolves the
// device address with cudaGetSymbolAddress while that device is current and
// caches it.  That first call must come before any stream capture begins.
#include <mutex>

#include "upipe.h"
#include "upipe_internal.h"

namespace upipe {
namespace {

constexpr size_t kNoAllocScratchBytes = 8u << 20;  // 8 MiB: n_q * S <= 1,048,576
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device; resolved once
// per device, with that device current.
cudaError_t scratch_for_current_device(void** scratch) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> g(g_setup_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *scratch = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace upipe

using namespace upipe;

extern "C" int upipe_attention_bwd_noalloc(const upipe_bf16* Q, const upipe_bf16* K, const upipe_bf16* V,
                                           const upipe_bf16* O, const upipe_bf16* dO, const float* lse, int n_q,
                                           int n_kv, int S, int d_head, const int32_t* kv_of_q, float* dQ,
                                           float* dK, float* dV, void* stream) {
  const int rc = attention_bwd_check(Q, K, V, O, dO, lse, n_q, n_kv, S, d_head, kv_of_q, dQ, dK, dV);
  if (rc != UPIPE_OK) return rc;
  // the fixed scratch holds D and lse*log2(e) for every (query slot, token)
  if (attention_bwd_scratch_bytes(n_q, S) > kNoAllocScratchBytes) return UPIPE_ENOSPC;
  if (!device_supported()) return UPIPE_EUNSUPPORTED;
  void* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return UPIPE_ECUDA;
  return attention_bwd_enqueue(Q, K, V, O, dO, lse, n_q, n_kv, S, d_head, kv_of_q, dQ, dK, dV, scratch,
                               static_cast<cudaStream_t>(stream));
}
