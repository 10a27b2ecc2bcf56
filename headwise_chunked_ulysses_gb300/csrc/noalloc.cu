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

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace upipe

using namespace upipe;

extern "C" int upipe_attention_bwd_noalloc(const upipe_bf16* Q, const upipe_bf16* K, const upipe_bf16* V,
                                           const upipe_bf16* O, const upipe_bf16* dO, const float* lse, int n_q,
                                           int n_kv, int S, int d_head, const int32_t* kv_of_q, float* dQ,
                                           float* dK, float* dV, void* stream) {
  const void* ptrs[] = {Q, K, V, O, dO, lse, dQ, dK, dV};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return UPIPE_EINVAL;
  if (!kv_of_q || n_q <= 0 || n_kv <= 0 || S <= 0 || S % 128) return UPIPE_EINVAL;
  if (d_head != 64 && d_head != 128) return UPIPE_EUNSUPPORTED;
  if (n_q > kMaxSlots) return UPIPE_EUNSUPPORTED;
  for (int k = 0; k < n_q; ++k)
    if (kv_of_q[k] < 0 || kv_of_q[k] >= n_kv) return UPIPE_EINVAL;
  // the fixed scratch holds D and lse*log2(e) for every (query slot, token)
  if (8ull * static_cast<unsigned long long>(n_q) * static_cast<unsigned long long>(S) > kNoAllocScratchBytes)
    return UPIPE_ENOSPC;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return UPIPE_ECUDA;
  if (major != 10 || minor != 3) return UPIPE_EUNSUPPORTED;
  void* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return UPIPE_ECUDA;
  int* status = device_status_word();  // the word upipe_sync_status() reads
  if (!status) return UPIPE_ECUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* dsum = static_cast<float*>(scratch);
  float* lse2 = dsum + static_cast<size_t>(n_q) * S;
  BwdPrepDesc pr;
  pr.dO = dO; pr.ld_do = d_head; pr.O = O; pr.ld_o = d_head; pr.lse = lse;
  pr.Dsum = dsum; pr.lse2 = lse2; pr.dQacc = dQ; pr.S = S; pr.D = d_head; pr.n_slots = n_q;
  for (int k = 0; k < n_q; ++k) {
    pr.do_unit[k] = k * S;
    pr.o_unit[k] = k * S;
    pr.lse_row[k] = static_cast<uint16_t>(k);
  }
  if (launch_bwd_prep(pr, st) != cudaSuccess) return UPIPE_ECUDA;
  AttnBwdDesc ab;
  ab.Q = Q; ab.K = K; ab.V = V; ab.dO = dO; ab.lse2 = lse2; ab.Dsum = dsum; ab.dQacc = dQ; ab.dK = dK; ab.dV = dV;
  ab.accumulate_kv = 0; ab.S = S; ab.D = d_head; ab.n_qslots = n_q; ab.n_kvslots = n_kv;
  for (int k = 0; k < n_q; ++k) ab.kv_slot[k] = static_cast<uint16_t>(kv_of_q[k]);
  return launch_attn_bwd(ab, status, st) == cudaSuccess ? UPIPE_OK : UPIPE_ECUDA;
}
