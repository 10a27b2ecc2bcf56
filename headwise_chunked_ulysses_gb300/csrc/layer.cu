// Host orchestration of the headwise-chunked attention layer and the C ABI.
//
// "Untied Ulysses" summary (paper.rainbus.top), Method steps: the layer runs
// H/U stages; stage i projects X onto the Q, K, V of its heads (1), exchanges
// them from sequence shards to head shards (2), runs causal attention (3) and
// exchanges the output back (4); buffers are reused by every stage.  Each
// stage then adds O_s W_o[rows of s] into Y.  Novelty section: the GQA
// out-of-order schedule.  The backward pass is not on the pages; it repeats
// the stages, recomputing (1) and (2), so Q, K and V never outlive a stage.
//
// Everything here runs on the host: argument checks, the head schedule, the
// workspace plan (offsets of the stage buffers, aliased by liveness), and the
// launch sequence on the caller's stream.  All arithmetic happens in the
// kernels of gemm.cu, attn_fwd.cu, attn_bwd.cu and permute.cu.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "upipe.h"
#include "upipe_internal.h"

namespace upipe {

// ---------------------------------------------------------------------------
// tensor maps, device facts, status word
// ---------------------------------------------------------------------------
namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
__device__ int g_status_word;

// Facts the library needs about each device, looked up once per device with
// that device current: a __device__ variable has one instance per device, so
// its address (like the SM count and the architecture) is a per-device fact.
constexpr int kMaxDevices = 64;
struct DeviceFacts {
  bool probed = false;
  bool supported = false;  // compute capability 10.3 (sm_103)
  int sms = 0;
  int* status = nullptr;   // this device's instance of g_status_word
  std::vector<const void*> smem_configured;  // kernels whose shared-memory limit is raised
};
std::mutex g_dev_mu;
DeviceFacts g_dev[kMaxDevices];

// The current device's facts (nullptr if the device cannot be queried).
// Caller holds g_dev_mu.
DeviceFacts* facts_locked() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceFacts& f = g_dev[dev];
  if (!f.probed) {
    int major = 0, minor = 0, sms = 0;
    void* p = nullptr;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess)
      return nullptr;  // not cached: the next call asks again
    f.supported = (major == 10 && minor == 3);
    f.sms = sms > 0 ? sms : 1;
    f.status = static_cast<int*>(p);
    f.probed = true;
  }
  return &f;
}

int* status_ptr() {
  std::lock_guard<std::mutex> g(g_dev_mu);
  const DeviceFacts* f = facts_locked();
  return f ? f->status : nullptr;
}
}  // namespace

namespace {
bool make_tmap_2d(CUtensorMap* m, CUtensorMapDataType type, uint64_t elem_bytes, const void* base, uint64_t inner,
                  uint64_t outer, uint64_t row_stride_elems, uint32_t box_inner, uint32_t box_outer) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_stride_elems * elem_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t es[2] = {1, 1};
  return g_encode(m, type, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_stride_elems,
                    uint32_t box_inner, uint32_t box_outer) {
  return make_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, inner, outer, row_stride_elems, box_inner,
                      box_outer);
}

bool make_tmap_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_stride_elems,
                  uint32_t box_inner, uint32_t box_outer) {
  return make_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, inner, outer, row_stride_elems, box_inner,
                      box_outer);
}

bool make_tmap_f32(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_stride_elems,
                   uint32_t box_inner, uint32_t box_outer) {
  return make_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, inner, outer, row_stride_elems, box_inner,
                      box_outer);
}

int* device_status_word() { return status_ptr(); }

int num_sms() {
  std::lock_guard<std::mutex> g(g_dev_mu);
  const DeviceFacts* f = facts_locked();
  return f ? f->sms : 1;
}

cudaError_t ensure_dynamic_smem(const void* kernel, int bytes) {
  std::lock_guard<std::mutex> g(g_dev_mu);
  DeviceFacts* f = facts_locked();
  if (!f) return cudaErrorInvalidDevice;
  for (const void* k : f->smem_configured)
    if (k == kernel) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) f->smem_configured.push_back(kernel);
  return e;
}

bool device_supported() {
  std::lock_guard<std::mutex> g(g_dev_mu);
  const DeviceFacts* f = facts_locked();
  return f && f->supported;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------------------
// shape, schedule and workspace plan
// ---------------------------------------------------------------------------
struct Shape {
  int S, dm, H, G, d, U, C, sched;
};

int check_shape(const Shape& s) {
  if (s.S <= 0 || s.dm <= 0 || s.H <= 0 || s.G <= 0 || s.d <= 0 || s.U <= 0 || s.C <= 0) return UPIPE_EINVAL;
  if (s.sched != UPIPE_SCHED_INORDER && s.sched != UPIPE_SCHED_GQA_OOO) return UPIPE_EINVAL;
  if (s.H % s.U || s.U % s.C || s.H % s.G || s.S % s.C) return UPIPE_EINVAL;
  if (s.sched == UPIPE_SCHED_GQA_OOO && !(s.G % s.C == 0 || s.C % s.G == 0)) return UPIPE_EINVAL;
  if (s.S % 128 || s.dm % 64) return UPIPE_EINVAL;
  if (s.d != 64 && s.d != 128) return UPIPE_EUNSUPPORTED;
  // widest stage buffer, in heads: the stage's queries plus the K and V heads it moves
  const int kv_moved = s.sched == UPIPE_SCHED_GQA_OOO ? std::max(s.G, s.C) : std::min(s.U, s.G);
  const int cols = s.U + 2 * std::max(kv_moved, s.sched == UPIPE_SCHED_GQA_OOO ? s.G : 0);
  if (3 * s.U > kMaxSlots || s.U + 2 * kv_moved > kMaxSlots || cols * s.d / 64 > kMaxMap) return UPIPE_EUNSUPPORTED;
  return UPIPE_OK;
}

inline int kv_of(const Shape& s, int h) { return h / (s.H / s.G); }

// query head of (stage i, rank r, slot j)
inline int sched_head(const Shape& s, int i, int r, int j) {
  const int qpr = s.U / s.C;
  return s.sched == UPIPE_SCHED_INORDER ? i * s.U + r * qpr + j : r * (s.H / s.C) + i * qpr + j;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct Stage {
  std::vector<int> q_heads;  // U query heads, slot k = r*(U/C) + j
  std::vector<int> kv_proj;  // KV heads this stage projects and exchanges (sorted)
  std::vector<int> k_src;    // per exchanged K (and V) slot: index into kv_proj
  std::vector<int> kv_of_q;  // per query slot: its KV slot
  int ncols() const { return static_cast<int>(q_heads.size() + 2 * kv_proj.size()); }  // in heads
};

struct Plan {
  Shape sh;
  int n_stages = 0, n_kv_slots = 0, max_cols = 0;
  std::vector<Stage> st;
  std::vector<int> resident;  // out of order: KV head of each resident slot
  // workspace layout (bytes)
  size_t off_seq = 0, off_qkvh = 0, off_doh = 0, off_dsum = 0, off_lse2 = 0, off_dacc = 0, off_acc32 = 0;
  bool prefetch = false;            // forward: a second stage-buffer set for the next stage
  size_t off_seq2 = 0, off_qkvh2 = 0;
  size_t arena = 0, persistent = 0, total = 0;
};

void build_schedule(Plan& p) {
  const Shape& s = p.sh;
  const int qpr = s.U / s.C;
  p.n_stages = s.H / s.U;
  p.st.assign(p.n_stages, Stage());
  if (s.sched == UPIPE_SCHED_GQA_OOO) {
    // rank r keeps the KV heads its query heads use, in every stage
    int kvr = 0;
    std::vector<std::vector<int>> rk(s.C);
    for (int r = 0; r < s.C; ++r) {
      for (int i = 0; i < p.n_stages; ++i)
        for (int j = 0; j < qpr; ++j) rk[r].push_back(kv_of(s, sched_head(s, i, r, j)));
      std::sort(rk[r].begin(), rk[r].end());
      rk[r].erase(std::unique(rk[r].begin(), rk[r].end()), rk[r].end());
      kvr = std::max<int>(kvr, static_cast<int>(rk[r].size()));
    }
    p.resident.assign(s.C * kvr, -1);
    for (int r = 0; r < s.C; ++r)
      for (int m = 0; m < static_cast<int>(rk[r].size()); ++m) p.resident[r * kvr + m] = rk[r][m];
    p.n_kv_slots = s.C * kvr;
    for (int i = 0; i < p.n_stages; ++i) {
      Stage& g = p.st[i];
      for (int r = 0; r < s.C; ++r)
        for (int j = 0; j < qpr; ++j) {
          const int h = sched_head(s, i, r, j);
          g.q_heads.push_back(h);
          const int m = static_cast<int>(std::find(rk[r].begin(), rk[r].end(), kv_of(s, h)) - rk[r].begin());
          g.kv_of_q.push_back(r * kvr + m);
        }
      if (i == 0) {
        for (int r = 0; r < s.C; ++r)
          for (int m = 0; m < kvr; ++m) {
            const int gh = p.resident[r * kvr + m];
            if (gh >= 0 && std::find(g.kv_proj.begin(), g.kv_proj.end(), gh) == g.kv_proj.end())
              g.kv_proj.push_back(gh);
          }
        std::sort(g.kv_proj.begin(), g.kv_proj.end());
        for (int r = 0; r < s.C * kvr; ++r) {
          const int gh = p.resident[r] >= 0 ? p.resident[r] : g.kv_proj[0];
          g.k_src.push_back(static_cast<int>(std::find(g.kv_proj.begin(), g.kv_proj.end(), gh) - g.kv_proj.begin()));
        }
      }
    }
  } else {
    p.n_kv_slots = s.U;  // every query slot receives its own copy of its KV head
    for (int i = 0; i < p.n_stages; ++i) {
      Stage& g = p.st[i];
      for (int r = 0; r < s.C; ++r)
        for (int j = 0; j < qpr; ++j) g.q_heads.push_back(sched_head(s, i, r, j));
      for (int h : g.q_heads) g.kv_proj.push_back(kv_of(s, h));
      std::sort(g.kv_proj.begin(), g.kv_proj.end());
      g.kv_proj.erase(std::unique(g.kv_proj.begin(), g.kv_proj.end()), g.kv_proj.end());
      for (int k = 0; k < s.U; ++k) {
        const int gh = kv_of(s, g.q_heads[k]);
        g.k_src.push_back(static_cast<int>(std::find(g.kv_proj.begin(), g.kv_proj.end(), gh) - g.kv_proj.begin()));
        g.kv_of_q.push_back(k);
      }
    }
  }
  p.max_cols = 0;
  for (const Stage& g : p.st) p.max_cols = std::max(p.max_cols, g.ncols());
  if (s.sched == UPIPE_SCHED_GQA_OOO) p.max_cols = std::max(p.max_cols, 2 * s.G);
}

// FP8 stage buffers inside the head-layout region of a stage: Q and K as E4M3
// codes, V in bf16, the fp32 scales of Q rows and of 128-key blocks of K
struct Fp8Stage {
  uint8_t* q = nullptr;
  uint8_t* k = nullptr;
  uint16_t* v = nullptr;
  float* qs = nullptr;
  float* ks = nullptr;
  size_t bytes = 0;
};

Fp8Stage fp8_stage_buffers(const Plan& p, uint8_t* base) {
  const Shape& s = p.sh;
  const size_t Sd = static_cast<size_t>(s.S) * s.d;
  Fp8Stage f;
  const size_t o_k = align256(s.U * Sd);
  const size_t o_v = align256(o_k + p.n_kv_slots * Sd);
  const size_t o_qs = align256(o_v + p.n_kv_slots * Sd * 2);
  const size_t o_ks = align256(o_qs + static_cast<size_t>(s.U) * s.S * 4);
  f.bytes = o_ks + static_cast<size_t>(p.n_kv_slots) * (s.S / 128) * 4;
  if (base) {
    f.q = base;
    f.k = base + o_k;
    f.v = reinterpret_cast<uint16_t*>(base + o_v);
    f.qs = reinterpret_cast<float*>(base + o_qs);
    f.ks = reinterpret_cast<float*>(base + o_ks);
  }
  return f;
}

// Workspace: [stage arena | persistent].  The stage arena holds the sequence-
// layout stage buffer (QKV, then reused for dO and dQKV) and the head-layout
// exchange buffers; the persistent part holds the fp32 Y / dX accumulator.
Plan make_plan(const Shape& s, bool backward, bool prefetch = false, bool fp8_all = false) {
  Plan p;
  p.sh = s;
  build_schedule(p);
  const size_t S = s.S, d = s.d, U = s.U;
  size_t o = 0;
  p.off_seq = o;
  o = align256(o + S * p.max_cols * d * 2);
  p.off_qkvh = o;
  // head-layout stage buffers; when every stage runs FP8 scores they hold Q
  // and K codes with their scales and bf16 V (fp8_all: backward plans only)
  o = align256(o + (fp8_all ? fp8_stage_buffers(p, nullptr).bytes : (U + 2 * p.n_kv_slots) * S * d * 2));
  if (backward) {
    p.off_doh = o;
    o = align256(o + U * S * d * 2);
    p.off_dsum = o;
    o = align256(o + U * S * 4);
    p.off_lse2 = o;
    o = align256(o + U * S * 4);
    p.off_dacc = o;
    o = align256(o + (U + 2 * p.n_kv_slots) * S * d * 4);
  }
  if (prefetch && !backward) {
    // odd stages' buffers: the sequence buffer and the head-layout Q slots,
    // plus (in order) their own K and V slots; out of order the K and V slots
    // of the first set stay resident for every stage
    p.prefetch = true;
    p.off_seq2 = o;
    o = align256(o + S * p.max_cols * d * 2);
    p.off_qkvh2 = o;
    o = align256(o + (s.sched == UPIPE_SCHED_GQA_OOO ? U : U + 2 * p.n_kv_slots) * S * d * 2);
  }
  p.arena = o;
  const int acc_gemms = backward ? p.n_stages + (s.sched == UPIPE_SCHED_GQA_OOO ? 1 : 0) : p.n_stages;
  p.off_acc32 = o;
  if (acc_gemms > 1) o = align256(o + S * s.dm * 4);
  p.persistent = o - p.arena;
  p.total = o;
  return p;
}

// Whether every stage of the plan is flagged FP8 (in-order stages).
bool all_stages_fp8(const Plan& p, const uint8_t* fp8_heads) {
  if (!fp8_heads) return false;
  for (const Stage& g : p.st)
    if (!fp8_heads[g.q_heads[0]]) return false;
  return true;
}

// Split of a long-K contraction over CTAs (partial sums added atomically):
// of the splits s <= 8 that divide its K blocks into runs of at least 8 and
// whose s fp32 partial outputs come to at most 256 MB of reduce-adds, the
// one whose s x (output tiles) work units fill the last round of the GPU's
// tile slots best (CTA pairs for 256 x 256 tiles, one CTA otherwise); a
// larger split must fill it at least 2 % better.
int choose_split_k(const GemmDesc& g) {
  const int bn = (g.N % 256 == 0) ? 256 : (g.N % 128 == 0 ? 128 : 64);
  const bool pair = bn == 256 && g.M % 256 == 0 && num_sms() >= 2;
  const long long tiles = pair ? static_cast<long long>(g.M / 256) * (g.N / bn)
                               : static_cast<long long>((g.M + 127) / 128) * (g.N / bn);
  const long long slots = pair ? num_sms() / 2 : num_sms();
  const int kb = g.K / 64;
  // a split's K range is kb/s blocks, rounded either way; the estimated time
  // is the number of rounds of work units times the longest range, and a
  // larger split is taken only when it is at least 2 % faster (its partial
  // sums add more fp32 traffic)
  int best = 1;
  double best_time = 0.0;
  for (int s = 1; s <= 8; ++s) {
    if (kb / s < 8) break;
    if (s > 1 && static_cast<long long>(s) * g.M * g.N * 4 > (1LL << 28)) break;
    const long long units = tiles * s, rounds = (units + slots - 1) / slots;
    const double time = static_cast<double>(rounds) * static_cast<double>((kb + s - 1) / s);
    if (s == 1 || time < 0.98 * best_time) {
      best = s;
      best_time = time;
    }
  }
  return best;
}

// 64-element blocks of the given heads (d columns each), in order
void head_blocks(BlockMap& m, const std::vector<int>& cols_in_heads, int d) {
  m.n = 0;
  for (int h : cols_in_heads)
    for (int b = 0; b < d / 64; ++b) m.idx[m.n++] = static_cast<uint16_t>(h * (d / 64) + b);
}

// Column heads (in units of d) of a stage's sequence buffer inside W_qkv.
std::vector<int> stage_wqkv_heads(const Shape& s, const std::vector<int>& q, const std::vector<int>& kv) {
  std::vector<int> c(q.begin(), q.end());
  for (int g : kv) c.push_back(s.H + g);
  for (int g : kv) c.push_back(s.H + s.G + g);
  return c;
}

// Optional per-launch timing: CUDA events recorded on the caller's stream
// around every kernel, summed per kernel kind by upipe_profile_read().
// A second stream per device for work that runs beside the caller's stream
// (created on first use, kept for the life of the process).
cudaStream_t side_stream() {
  static std::mutex mu;
  static cudaStream_t streams[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> g(mu);
  if (!streams[dev] && cudaStreamCreateWithFlags(&streams[dev], cudaStreamNonBlocking) != cudaSuccess)
    streams[dev] = nullptr;
  return streams[dev];
}

struct Profiler {
  bool on = false;
  std::vector<cudaEvent_t> ev;  // pairs
  std::vector<int> kind;
  size_t used = 0;
  std::mutex mu;
  int begin(cudaStream_t st, int k) {
    if (!on) return -1;
    std::lock_guard<std::mutex> g(mu);
    if (2 * used + 2 > ev.size()) {
      for (int i = 0; i < 2; ++i) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) return -1;
        ev.push_back(e);
      }
      kind.push_back(0);
    }
    const int slot = static_cast<int>(used++);
    kind[slot] = k;
    cudaEventRecord(ev[2 * slot], st);
    return slot;
  }
  void end(cudaStream_t st, int slot) {
    if (slot >= 0) cudaEventRecord(ev[2 * slot + 1], st);
  }
};
Profiler g_prof;

struct Launcher {
  cudaStream_t st;
  int* status;
  int launches = 0;
  size_t permute_bytes = 0;
  int n_kind[UPIPE_KERNEL_KINDS] = {};
  double flops[UPIPE_KERNEL_KINDS] = {};
  double bytes[UPIPE_KERNEL_KINDS] = {};
  cudaError_t err = cudaSuccess;
  bool ok() const { return err == cudaSuccess; }
  void merge(const Launcher& o) {  // counts and first error of work issued on another stream
    launches += o.launches;
    permute_bytes += o.permute_bytes;
    for (int k = 0; k < UPIPE_KERNEL_KINDS; ++k) {
      n_kind[k] += o.n_kind[k];
      flops[k] += o.flops[k];
      bytes[k] += o.bytes[k];
    }
    if (ok() && !o.ok()) err = o.err;
  }
  template <typename F>
  void run(int kind, double fl, double by, F&& f) {
    if (!ok()) return;
    const int slot = g_prof.begin(st, kind);
    err = f();
    g_prof.end(st, slot);
    ++launches;
    ++n_kind[kind];
    flops[kind] += fl;
    bytes[kind] += by;
  }
  void gemm(const GemmDesc& g) {
    const double M = g.M, N = g.N, K = g.K;
    const double out_b = (g.out_mode == kOutBf16 ? 2.0 : 4.0) * M * N;
    const double extra = (g.out_mode == kOutF32Acc || g.out_mode == kOutBf16PlusF32) ? 4.0 * M * N : 0.0;
    run(UPIPE_KERNEL_GEMM, 2.0 * M * N * K, 2.0 * (M * K + K * N) + out_b + extra,
        [&] { return launch_gemm(g, status, st); });
  }
  // visible (query, key) pairs of one query slot: query row r sees
  // min(kv_len, q_off + r + 1) keys
  static double visible_pairs(double S, double kv_len, double q_off) {
    if (q_off >= kv_len) return S * kv_len;
    const double ramp = std::min(S, kv_len - q_off);  // rows before the key range ends
    return ramp * q_off + ramp * (ramp + 1) / 2 + (S - ramp) * kv_len;
  }
  void fwd(const AttnFwdDesc& a) {
    const double S = a.S, kv = a.kv_len ? a.kv_len : a.S, pairs = visible_pairs(S, kv, a.q_off);
    const double acc = a.mode == kFwdPlain ? 0.0 : (a.mode == kFwdFirst ? 4.0 : 8.0) * a.D + 8.0;
    run(UPIPE_KERNEL_ATTN_FWD, 2.0 * 2.0 * a.D * pairs * a.n_qslots,
        2.0 * a.D * (2.0 * S * a.n_qslots + 2.0 * kv * a.n_kvslots) + 4.0 * S * a.n_qslots + acc * S * a.n_qslots,
        [&] { return launch_attn_fwd(a, status, st); });
  }
  void bwd(const AttnBwdDesc& a) {
    const double S = a.S, kv = a.kv_len ? a.kv_len : a.S, pairs = visible_pairs(S, kv, a.q_off);
    run(UPIPE_KERNEL_ATTN_BWD, 5.0 * 2.0 * a.D * pairs * a.n_qslots,
        a.D * (S * (2.0 * 2 * a.n_qslots + 4.0 * a.n_qslots) +
               kv * (2.0 * 2 * a.n_kvslots + 4.0 * (a.accumulate_kv ? 2 : 1) * 2 * a.n_kvslots)) +
            8.0 * S * a.n_qslots,
        [&] { return launch_attn_bwd(a, status, st); });
  }
  void s2h(const Seq2HeadDesc& p) {
    const double b = 2.0 * p.n_slots * p.S * p.D * 2;
    run(UPIPE_KERNEL_SEQ2HEAD, 0.0, b, [&] { return launch_seq2head(p, st); });
    permute_bytes += static_cast<size_t>(b);
  }
  void h2s(const Head2SeqDesc& p) {
    const double b = static_cast<double>(p.first[p.n_heads]) * p.S * p.D * (p.src_f32 ? 4 : 2) +
                     static_cast<double>(p.n_heads) * p.S * p.D * 2;
    run(UPIPE_KERNEL_HEAD2SEQ, 0.0, b, [&] { return launch_head2seq(p, st); });
    permute_bytes += static_cast<size_t>(b);
  }
  void quant(const QuantDesc& p) {
    const double b = static_cast<double>(p.n_slots) * p.S * p.D * (2 + 1) +
                     4.0 * p.n_slots * (p.per_row ? p.S : p.S / 128);
    run(UPIPE_KERNEL_SEQ2HEAD, 0.0, b, [&] { return launch_quant_e4m3(p, st); });
    permute_bytes += static_cast<size_t>(b);
  }
  void prep(const BwdPrepDesc& p) {
    const double b = static_cast<double>(p.n_slots) * p.S * (2.0 * 2 * p.D + 4.0 * p.D + 12.0);
    run(UPIPE_KERNEL_BWD_PREP, 0.0, b, [&] { return launch_bwd_prep(p, st); });
  }
};

// The exchange of an FP8 stage from the projected sequence buffer: Q rows and
// K blocks encoded with their scales, V moved as bf16.
void exchange_fp8(Launcher& L, const Plan& p, int i, const uint16_t* seq, const Fp8Stage& f) {
  const Shape& s = p.sh;
  const Stage& g = p.st[i];
  const long long ld = static_cast<long long>(g.ncols()) * s.d;
  const int nkv = static_cast<int>(g.kv_proj.size());
  QuantDesc q;
  q.src = seq; q.ld_src = ld; q.dst = f.q; q.scale = f.qs; q.S = s.S; q.D = s.d; q.n_slots = s.U; q.per_row = true;
  for (int k = 0; k < s.U; ++k) q.src_head[k] = static_cast<uint16_t>(k);
  L.quant(q);
  QuantDesc kq;
  kq.src = seq; kq.ld_src = ld; kq.dst = f.k; kq.scale = f.ks; kq.S = s.S; kq.D = s.d; kq.n_slots = p.n_kv_slots;
  kq.per_row = false;
  for (int k = 0; k < p.n_kv_slots; ++k) kq.src_head[k] = static_cast<uint16_t>(s.U + g.k_src[k]);
  L.quant(kq);
  Seq2HeadDesc x;
  x.src = seq; x.ld_src = ld; x.dst = f.v; x.S = s.S; x.D = s.d; x.n_slots = p.n_kv_slots;
  for (int k = 0; k < p.n_kv_slots; ++k) x.src_head[k] = static_cast<uint16_t>(s.U + nkv + g.k_src[k]);
  L.s2h(x);
}

// QKV projection of one stage into the sequence buffer, then the exchange.
void project_and_exchange(Launcher& L, const Plan& p, int i, const uint16_t* X, const uint16_t* W_qkv,
                          uint8_t* ws, int set = 0, bool fp8 = false) {
  const Shape& s = p.sh;
  const Stage& g = p.st[i];
  uint16_t* seq = reinterpret_cast<uint16_t*>(ws + (set ? p.off_seq2 : p.off_seq));
  uint16_t* qkvh = reinterpret_cast<uint16_t*>(ws + (set ? p.off_qkvh2 : p.off_qkvh));
  const int ncols = g.ncols();
  GemmDesc gd;
  gd.A = X; gd.lda = s.dm; gd.a_rows = s.S; gd.a_cols = s.dm; gd.a_mn = false;
  gd.B = W_qkv; gd.ldb = (s.H + 2 * s.G) * s.d; gd.b_rows = s.dm; gd.b_cols = gd.ldb; gd.b_mn = true;
  gd.M = s.S; gd.N = ncols * s.d; gd.K = s.dm;
  head_blocks(gd.bmap_n, stage_wqkv_heads(s, g.q_heads, g.kv_proj), s.d);
  gd.out = seq; gd.ldo = static_cast<long long>(ncols) * s.d; gd.out_mode = kOutBf16;
  L.gemm(gd);
  if (fp8) {
    exchange_fp8(L, p, i, seq, fp8_stage_buffers(p, reinterpret_cast<uint8_t*>(qkvh)));
    return;
  }
  // exchange: Q slots, then (when this stage moves KV) K slots and V slots
  Seq2HeadDesc x;
  x.src = seq; x.ld_src = static_cast<long long>(ncols) * s.d;
  x.dst = qkvh; x.S = s.S; x.D = s.d;
  int n = 0;
  for (int k = 0; k < s.U; ++k) x.src_head[n++] = static_cast<uint16_t>(k);
  if (!g.kv_proj.empty()) {
    const int nkv = static_cast<int>(g.kv_proj.size());
    for (int k = 0; k < p.n_kv_slots; ++k) x.src_head[n++] = static_cast<uint16_t>(s.U + g.k_src[k]);
    for (int k = 0; k < p.n_kv_slots; ++k) x.src_head[n++] = static_cast<uint16_t>(s.U + nkv + g.k_src[k]);
  }
  x.n_slots = n;
  L.s2h(x);
}

int finish(Launcher& L, const Plan& p, upipe_stats* stats) {
  if (stats) {
    stats->arena_peak_bytes = p.arena;
    stats->stage_closed_form_bytes = 12ull * p.sh.S * p.sh.U * p.sh.d;
    stats->persistent_bytes = p.persistent;
    stats->permute_bytes = L.permute_bytes;
    stats->launches = L.launches;
    stats->stages = p.n_stages;
    for (int k = 0; k < UPIPE_KERNEL_KINDS; ++k) {
      stats->launches_by_kind[k] = L.n_kind[k];
      stats->flops_by_kind[k] = L.flops[k];
      stats->bytes_by_kind[k] = L.bytes[k];
    }
  }
  return L.ok() ? UPIPE_OK : UPIPE_ECUDA;
}

int common_checks(const Shape& s, const void* const* ptrs, int n_ptrs, const void* ws, size_t ws_bytes, size_t need) {
  int rc = check_shape(s);
  if (rc != UPIPE_OK) return rc;
  for (int i = 0; i < n_ptrs; ++i)
    if (!ptrs[i] || !aligned16(ptrs[i])) return UPIPE_EINVAL;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return UPIPE_EINVAL;
  if (ws_bytes < need) return UPIPE_ENOSPC;
  if (!device_supported()) return UPIPE_EUNSUPPORTED;
  if (!status_ptr()) return UPIPE_ECUDA;
  return UPIPE_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// attention backward of one stage's heads: the body shared by the entry point
// that takes a workspace and the one whose scratch is a fixed array
// ---------------------------------------------------------------------------
size_t attention_bwd_scratch_bytes(int n_q, int S) {
  return 8ull * static_cast<unsigned long long>(n_q) * static_cast<unsigned long long>(S);
}

int attention_bwd_check(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* lse,
                        int n_q, int n_kv, int S, int d_head, const int32_t* kv_of_q, const float* dQ,
                        const float* dK, const float* dV) {
  const void* ptrs[] = {Q, K, V, O, dO, lse, dQ, dK, dV};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return UPIPE_EINVAL;
  if (!kv_of_q || n_q <= 0 || n_kv <= 0 || S <= 0 || S % 128) return UPIPE_EINVAL;
  if (d_head != 64 && d_head != 128) return UPIPE_EUNSUPPORTED;
  if (n_q > kMaxSlots) return UPIPE_EUNSUPPORTED;
  for (int k = 0; k < n_q; ++k)
    if (kv_of_q[k] < 0 || kv_of_q[k] >= n_kv) return UPIPE_EINVAL;
  return UPIPE_OK;
}

int attention_bwd_enqueue(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                          const float* lse, int n_q, int n_kv, int S, int d_head, const int32_t* kv_of_q, float* dQ,
                          float* dK, float* dV, void* scratch, cudaStream_t st) {
  if (!device_supported()) return UPIPE_EUNSUPPORTED;
  int* status = status_ptr();
  if (!status) return UPIPE_ECUDA;
  float* dsum = static_cast<float*>(scratch);
  float* lse2 = dsum + static_cast<size_t>(n_q) * S;
  BwdPrepDesc pr;
  pr.dO = static_cast<const uint16_t*>(dO); pr.ld_do = d_head; pr.O = static_cast<const uint16_t*>(O);
  pr.ld_o = d_head; pr.lse = lse;
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

}  // namespace upipe

using namespace upipe;

extern "C" {

size_t upipe_fwd_workspace_bytes(int S, int d_model, int H, int G, int d_head, int U, int C, int sched) {
  const Shape s{S, d_model, H, G, d_head, U, C, sched};
  if (check_shape(s) != UPIPE_OK) return 0;
  return make_plan(s, false).total;
}

size_t upipe_fwd_workspace_bytes_prefetch(int S, int d_model, int H, int G, int d_head, int U, int C, int sched) {
  const Shape s{S, d_model, H, G, d_head, U, C, sched};
  if (check_shape(s) != UPIPE_OK) return 0;
  return make_plan(s, false, true).total;
}

size_t upipe_bwd_workspace_bytes(int S, int d_model, int H, int G, int d_head, int U, int C, int sched) {
  const Shape s{S, d_model, H, G, d_head, U, C, sched};
  if (check_shape(s) != UPIPE_OK) return 0;
  return make_plan(s, true).total;
}

size_t upipe_bwd_workspace_bytes_fp8(int S, int d_model, int H, int G, int d_head, int U, int C,
                                     const uint8_t* fp8_heads) {
  const Shape s{S, d_model, H, G, d_head, U, C, UPIPE_SCHED_INORDER};
  if (check_shape(s) != UPIPE_OK || !fp8_heads) return 0;
  const Plan p = make_plan(s, true);
  return all_stages_fp8(p, fp8_heads) ? make_plan(s, true, false, true).total : p.total;
}

}  // extern "C"

namespace {

int attn_fwd_issue(const upipe_bf16* X, const upipe_bf16* W_qkv, const upipe_bf16* W_o, int S, int d_model, int H,
                   int G, int d_head, int U, int C, int sched, upipe_bf16* Y, upipe_bf16* O_saved, float* lse,
                   void* ws, size_t ws_bytes, void* stream, upipe_stats* stats, bool allow_prefetch,
                   const uint8_t* fp8_heads = nullptr) {
  const Shape s{S, d_model, H, G, d_head, U, C, sched};
  if (check_shape(s) != UPIPE_OK) return check_shape(s);
  const Plan pmin = make_plan(s, false);
  const void* ptrs[] = {X, W_qkv, W_o, Y, O_saved, lse};
  int rc = common_checks(s, ptrs, 6, ws, ws_bytes, pmin.total);
  if (rc != UPIPE_OK) return rc;
  // with room for a second stage-buffer set, stage i+1's projection and
  // exchange run on a second stream while stage i's attention runs
  const Plan ppf = pmin.n_stages > 1 ? make_plan(s, false, true) : pmin;
  const bool pf = allow_prefetch && !fp8_heads && ppf.prefetch && ws_bytes >= ppf.total;
  const Plan& p = pf ? ppf : pmin;
  cudaStream_t st0 = static_cast<cudaStream_t>(stream), st1 = nullptr;
  cudaEvent_t ev[6] = {};  // fork, join, ready[2], free[2]
  if (pf) {
    st1 = side_stream();
    if (!st1) return UPIPE_ECUDA;
    for (cudaEvent_t& e : ev)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
        for (cudaEvent_t& f : ev)
          if (f) cudaEventDestroy(f);
        return UPIPE_ECUDA;
      }
  }
  cudaEvent_t ev_fork = ev[0], ev_join = ev[1], *ev_ready = ev + 2, *ev_free = ev + 4;
  Launcher L{st0, status_ptr()};
  Launcher L2{st1, L.status};
  uint8_t* w = static_cast<uint8_t*>(ws);
  const int d = d_head;
  float* y32 = reinterpret_cast<float*>(w + p.off_acc32);
  const size_t slot_elems = static_cast<size_t>(S) * d;
  if (pf) {  // stage 0's projection and exchange, after the caller's prior work
    cudaEventRecord(ev_fork, st0);
    cudaStreamWaitEvent(st1, ev_fork, 0);
    project_and_exchange(L2, p, 0, X, W_qkv, w, 0);
    cudaEventRecord(ev_ready[0], st1);
  }
  for (int i = 0; i < p.n_stages && L.ok() && L2.ok(); ++i) {
    const Stage& g = p.st[i];
    const int set = pf ? (i & 1) : 0;
    uint16_t* qkvh = reinterpret_cast<uint16_t*>(w + (set ? p.off_qkvh2 : p.off_qkvh));
    // K and V: out of order they stay resident in the first set
    uint16_t* kvh = reinterpret_cast<uint16_t*>(w + (set && sched != UPIPE_SCHED_GQA_OOO ? p.off_qkvh2 : p.off_qkvh));
    uint16_t* oh = reinterpret_cast<uint16_t*>(w + (set ? p.off_seq2 : p.off_seq));  // dead after the exchange
    // (1) projection, (2) exchange to head shards: on the second stream, one
    // stage ahead, into the other buffer set once the stage before has left it
    if (pf) {
      if (i + 1 < p.n_stages) {
        if (i >= 1) cudaStreamWaitEvent(st1, ev_free[(i + 1) & 1], 0);
        project_and_exchange(L2, p, i + 1, X, W_qkv, w, (i + 1) & 1);
        cudaEventRecord(ev_ready[(i + 1) & 1], st1);
      }
      cudaStreamWaitEvent(st0, ev_ready[set], 0);
    }
    const bool f8 = fp8_heads && fp8_heads[g.q_heads[0]];
    if (!pf) project_and_exchange(L, p, i, X, W_qkv, w, 0, f8);
    // (3) attention of the stage's heads
    AttnFwdDesc a;
    a.Q = qkvh;
    a.K = kvh + U * slot_elems;
    a.V = kvh + (U + p.n_kv_slots) * slot_elems;
    if (f8) {
      const Fp8Stage f = fp8_stage_buffers(p, reinterpret_cast<uint8_t*>(qkvh));
      a.fp8 = true;
      a.Q = f.q; a.K = f.k; a.V = f.v; a.q_scale = f.qs; a.k_scale = f.ks;
    }
    a.O = oh;
    a.lse = lse;
    a.S = S; a.D = d; a.n_qslots = U; a.n_kvslots = p.n_kv_slots;
    for (int k = 0; k < U; ++k) {
      a.kv_slot[k] = static_cast<uint16_t>(g.kv_of_q[k]);
      a.lse_row[k] = static_cast<uint16_t>(g.q_heads[k]);
    }
    L.fwd(a);
    // (4) exchange back into the stage's columns of O_saved
    Head2SeqDesc b;
    b.src = oh; b.src_f32 = false;
    b.dst = O_saved; b.ld_dst = static_cast<long long>(H) * d;
    b.S = S; b.D = d; b.n_heads = U;
    for (int k = 0; k <= U; ++k) b.first[k] = static_cast<uint16_t>(k);
    for (int k = 0; k < U; ++k) {
      b.dst_head[k] = static_cast<uint16_t>(g.q_heads[k]);
      b.src_slot[k] = static_cast<uint16_t>(k);
    }
    L.h2s(b);
    if (pf) cudaEventRecord(ev_free[set], st0);  // this set's buffers are free again
    // (5) the stage's heads' share of the output projection accumulates into Y:
    // fp32 Y32 = O_s W_o[rows of s] for the first stage, += for the next ones
    // (TMA stores / atomic adds), bf16 Y = Y32 + the last share
    GemmDesc go;
    go.A = O_saved; go.lda = static_cast<long long>(H) * d; go.a_rows = S; go.a_cols = go.lda; go.a_mn = false;
    go.B = W_o; go.ldb = d_model; go.b_rows = static_cast<long long>(H) * d; go.b_cols = d_model; go.b_mn = true;
    go.M = S; go.N = d_model; go.K = U * d;
    head_blocks(go.amap_k, g.q_heads, d);
    go.bmap_k = go.amap_k;
    if (p.n_stages == 1) {
      go.out = Y; go.ldo = d_model; go.out_mode = kOutBf16;
    } else if (i == 0) {
      go.out = y32; go.ldo = d_model; go.out_mode = kOutF32;
    } else if (i + 1 < p.n_stages) {
      go.out = y32; go.ldo = d_model; go.out_mode = kOutF32Acc;
    } else {
      go.out = Y; go.ldo = d_model; go.out_mode = kOutBf16PlusF32; go.aux = y32; go.ld_aux = d_model;
    }
    L.gemm(go);
  }
  if (pf) {
    cudaEventRecord(ev_join, st1);
    cudaStreamWaitEvent(st0, ev_join, 0);
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
    L.merge(L2);
  }
  return finish(L, p, stats);
}

int attn_bwd_issue(const upipe_bf16* X, const upipe_bf16* W_qkv, const upipe_bf16* W_o, int S, int d_model, int H,
                   int G, int d_head, int U, int C, int sched, const upipe_bf16* O_saved, const float* lse,
                   const upipe_bf16* dY, upipe_bf16* dX, float* dW_qkv, float* dW_o, void* ws, size_t ws_bytes,
                   void* stream, upipe_stats* stats, const uint8_t* fp8_heads = nullptr) {
  const Shape s{S, d_model, H, G, d_head, U, C, sched};
  if (check_shape(s) != UPIPE_OK) return check_shape(s);
  const Plan p0 = make_plan(s, true);
  const Plan p = all_stages_fp8(p0, fp8_heads) ? make_plan(s, true, false, true) : p0;
  const void* ptrs[] = {X, W_qkv, W_o, O_saved, lse, dY, dX, dW_qkv, dW_o};
  int rc = common_checks(s, ptrs, 9, ws, ws_bytes, p.total);
  if (rc != UPIPE_OK) return rc;
  Launcher L{static_cast<cudaStream_t>(stream), status_ptr()};
  uint8_t* w = static_cast<uint8_t*>(ws);
  const int d = d_head;
  const bool ooo = sched == UPIPE_SCHED_GQA_OOO;
  const size_t slot_elems = static_cast<size_t>(S) * d;
  const long long qkv_ld = static_cast<long long>(H + 2 * G) * d;
  uint16_t* seq = reinterpret_cast<uint16_t*>(w + p.off_seq);
  uint16_t* qkvh = reinterpret_cast<uint16_t*>(w + p.off_qkvh);
  uint16_t* doh = reinterpret_cast<uint16_t*>(w + p.off_doh);
  float* dsum = reinterpret_cast<float*>(w + p.off_dsum);
  float* lse2 = reinterpret_cast<float*>(w + p.off_lse2);
  float* dacc = reinterpret_cast<float*>(w + p.off_dacc);  // [dQ: U | dK: n_kv | dV: n_kv] slots, fp32
  float* dx32 = reinterpret_cast<float*>(w + p.off_acc32);
  const int n_dx = p.n_stages + (ooo ? 1 : 0);
  int dx_done = 0;

  if (cudaMemsetAsync(dW_qkv, 0, static_cast<size_t>(d_model) * qkv_ld * 4, L.st) != cudaSuccess)
    return UPIPE_ECUDA;

  // dX (+)= dQKV_seq W_qkv[:, heads]^T ; dW_qkv[:, heads] += X^T dQKV_seq
  auto project_back = [&](const uint16_t* dseq, const std::vector<int>& wheads) {
    const int ncols = static_cast<int>(wheads.size());
    GemmDesc gx;
    gx.A = dseq; gx.lda = static_cast<long long>(ncols) * d; gx.a_rows = S; gx.a_cols = gx.lda; gx.a_mn = false;
    gx.B = W_qkv; gx.ldb = qkv_ld; gx.b_rows = d_model; gx.b_cols = qkv_ld; gx.b_mn = false;
    gx.M = S; gx.N = d_model; gx.K = ncols * d;
    head_blocks(gx.bmap_k, wheads, d);
    if (n_dx == 1) {
      gx.out = dX; gx.ldo = d_model; gx.out_mode = kOutBf16;
    } else if (dx_done == 0) {
      gx.out = dx32; gx.ldo = d_model; gx.out_mode = kOutF32;
    } else if (dx_done + 1 < n_dx) {
      gx.out = dx32; gx.ldo = d_model; gx.out_mode = kOutF32Acc;
    } else {
      gx.out = dX; gx.ldo = d_model; gx.out_mode = kOutBf16PlusF32; gx.aux = dx32; gx.ld_aux = d_model;
    }
    ++dx_done;
    L.gemm(gx);
    GemmDesc gw;
    gw.A = X; gw.lda = d_model; gw.a_rows = S; gw.a_cols = d_model; gw.a_mn = true;
    gw.B = dseq; gw.ldb = static_cast<long long>(ncols) * d; gw.b_rows = S; gw.b_cols = gw.ldb; gw.b_mn = true;
    gw.M = d_model; gw.N = ncols * d; gw.K = S;
    head_blocks(gw.omap_n, wheads, d);
    gw.out = dW_qkv; gw.ldo = qkv_ld; gw.out_mode = kOutF32Red;  // dW_qkv is zeroed above
    gw.split_k = choose_split_k(gw);
    L.gemm(gw);
  };

  for (int i = 0; i < p.n_stages && L.ok(); ++i) {
    const Stage& g = p.st[i];
    // recompute (1) and (2); an FP8 stage exchanges Q and K as the codes its
    // forward attended with
    const bool f8 = fp8_heads && fp8_heads[g.q_heads[0]];
    project_and_exchange(L, p, i, X, W_qkv, w, 0, f8);
    // dO_s = dY W_o[rows of the stage]^T in sequence layout (the QKV sequence buffer is dead)
    GemmDesc gd;
    gd.A = dY; gd.lda = d_model; gd.a_rows = S; gd.a_cols = d_model; gd.a_mn = false;
    gd.B = W_o; gd.ldb = d_model; gd.b_rows = static_cast<long long>(H) * d; gd.b_cols = d_model; gd.b_mn = false;
    gd.M = S; gd.N = U * d; gd.K = d_model;
    head_blocks(gd.bmap_n, g.q_heads, d);
    gd.out = seq; gd.ldo = static_cast<long long>(U) * d; gd.out_mode = kOutBf16;
    L.gemm(gd);
    // exchange dO to head shards
    Seq2HeadDesc xd;
    xd.src = seq; xd.ld_src = static_cast<long long>(U) * d;
    xd.dst = doh; xd.S = S; xd.D = d; xd.n_slots = U;
    for (int k = 0; k < U; ++k) xd.src_head[k] = static_cast<uint16_t>(k);
    L.s2h(xd);
    // D = rowsum(dO * O), lse in log2 units, dQ accumulator zeroed
    BwdPrepDesc pr;
    pr.dO = seq; pr.ld_do = static_cast<long long>(U) * d;
    pr.O = O_saved; pr.ld_o = static_cast<long long>(H) * d;
    pr.lse = lse; pr.Dsum = dsum; pr.lse2 = lse2; pr.dQacc = dacc;
    pr.S = S; pr.D = d; pr.n_slots = U;
    for (int k = 0; k < U; ++k) {
      pr.do_unit[k] = k;
      pr.o_unit[k] = g.q_heads[k];
      pr.lse_row[k] = static_cast<uint16_t>(g.q_heads[k]);
    }
    L.prep(pr);
    // attention backward
    AttnBwdDesc ab;
    ab.Q = qkvh;
    ab.K = qkvh + U * slot_elems;
    ab.V = qkvh + (U + p.n_kv_slots) * slot_elems;
    if (f8) {
      const Fp8Stage f = fp8_stage_buffers(p, reinterpret_cast<uint8_t*>(qkvh));
      ab.Q = f.q; ab.K = f.k; ab.V = f.v;
      ab.fp8 = true; ab.q_scale = f.qs; ab.k_scale = f.ks;
    }
    ab.dO = doh; ab.lse2 = lse2; ab.Dsum = dsum; ab.dQacc = dacc;
    ab.dK = dacc + U * slot_elems;
    ab.dV = dacc + (U + p.n_kv_slots) * slot_elems;
    ab.accumulate_kv = (ooo && i > 0) ? 1 : 0;
    ab.S = S; ab.D = d; ab.n_qslots = U; ab.n_kvslots = p.n_kv_slots;
    for (int k = 0; k < U; ++k) ab.kv_slot[k] = static_cast<uint16_t>(g.kv_of_q[k]);
    L.bwd(ab);
    // exchange back: dQ (and in order, the summed copies of dK and dV) into the sequence buffer
    std::vector<int> wheads(g.q_heads.begin(), g.q_heads.end());
    const int nkv = ooo ? 0 : static_cast<int>(g.kv_proj.size());
    for (int part = 0; part < 2; ++part)
      for (int m = 0; m < nkv; ++m) wheads.push_back((part == 0 ? H : H + G) + g.kv_proj[m]);
    const long long ld_dseq = static_cast<long long>(wheads.size()) * d;
    Head2SeqDesc qb;  // row-major fp32 dQ -> bf16
    qb.src = dacc; qb.src_f32 = true;
    qb.dst = seq; qb.ld_dst = ld_dseq; qb.S = S; qb.D = d; qb.n_heads = U;
    for (int k = 0; k <= U; ++k) qb.first[k] = static_cast<uint16_t>(k);
    for (int k = 0; k < U; ++k) {
      qb.dst_head[k] = static_cast<uint16_t>(k);
      qb.src_slot[k] = static_cast<uint16_t>(k);
    }
    L.h2s(qb);
    if (nkv > 0) {
      Head2SeqDesc hb;
      hb.src = dacc; hb.src_f32 = true;
      hb.dst = seq; hb.ld_dst = ld_dseq; hb.S = S; hb.D = d;
      int n = 0, r = 0;
      hb.first[0] = 0;
      for (int part = 0; part < 2; ++part)
        for (int m = 0; m < nkv; ++m) {
          hb.dst_head[n] = static_cast<uint16_t>(U + n);
          for (int k = 0; k < p.n_kv_slots; ++k)
            if (g.k_src[k] == m) hb.src_slot[r++] = static_cast<uint16_t>(U + part * p.n_kv_slots + k);
          hb.first[++n] = static_cast<uint16_t>(r);
        }
      hb.n_heads = n;
      L.h2s(hb);
    }
    project_back(seq, wheads);
  }
  if (ooo && L.ok()) {
    // resident dK, dV go back once, copies of a KV head summed in rank order
    Head2SeqDesc hb;
    hb.src = dacc + U * slot_elems; hb.src_f32 = true;
    hb.dst = seq; hb.S = S; hb.D = d;
    std::vector<int> wheads;
    int n = 0, r = 0;
    hb.first[0] = 0;
    for (int part = 0; part < 2; ++part)
      for (int gh = 0; gh < G; ++gh) {
        hb.dst_head[n] = static_cast<uint16_t>(n);
        for (int k = 0; k < p.n_kv_slots; ++k)
          if (p.resident[k] == gh) hb.src_slot[r++] = static_cast<uint16_t>(part * p.n_kv_slots + k);
        hb.first[++n] = static_cast<uint16_t>(r);
        wheads.push_back((part == 0 ? H : H + G) + gh);
      }
    hb.n_heads = n;
    hb.ld_dst = static_cast<long long>(n) * d;
    L.h2s(hb);
    project_back(seq, wheads);
  }
  // dW_o = O_saved^T dY (O_saved holds every head already)
  GemmDesc gwo;
  gwo.A = O_saved; gwo.lda = static_cast<long long>(H) * d; gwo.a_rows = S; gwo.a_cols = gwo.lda; gwo.a_mn = true;
  gwo.B = dY; gwo.ldb = d_model; gwo.b_rows = S; gwo.b_cols = d_model; gwo.b_mn = true;
  gwo.M = H * d; gwo.N = d_model; gwo.K = S;
  gwo.out = dW_o; gwo.ldo = d_model;
  gwo.split_k = choose_split_k(gwo);
  if (gwo.split_k > 1) {
    if (cudaMemsetAsync(dW_o, 0, static_cast<size_t>(H) * d * d_model * 4, L.st) != cudaSuccess) return UPIPE_ECUDA;
    gwo.out_mode = kOutF32Red;
  } else {
    gwo.out_mode = kOutF32;
  }
  L.gemm(gwo);
  return finish(L, p, stats);
}

#include "layer_chunked.inl"

#include "layer_graphs.inl"


}  // namespace

extern "C" {

int upipe_attn_fwd(const upipe_bf16* X, const upipe_bf16* W_qkv, const upipe_bf16* W_o, int S, int d_model, int H,
                   int G, int d_head, int U, int C, int sched, upipe_bf16* Y, upipe_bf16* O_saved, float* lse,
                   void* ws, size_t ws_bytes, void* stream, upipe_stats* stats) {
  std::vector<unsigned long long> key = {1ull, as_key(X), as_key(W_qkv), as_key(W_o), as_key(Y), as_key(O_saved),
                                         as_key(lse), as_key(ws), ws_bytes};
  for (int v : {S, d_model, H, G, d_head, U, C, sched}) key.push_back(static_cast<unsigned long long>(v));
  // a graph is replayed on one stream: the prefetching path is used only uncached
  bool graphs_on;
  {
    std::lock_guard<std::mutex> g(g_graphs.mu);
    graphs_on = g_graphs.on;
  }
  return run_graphed(std::move(key), stream, stats, [&](void* st, upipe_stats* sts) {
    return attn_fwd_issue(X, W_qkv, W_o, S, d_model, H, G, d_head, U, C, sched, Y, O_saved, lse, ws, ws_bytes, st,
                          sts, !graphs_on);
  });
}

int upipe_attn_bwd(const upipe_bf16* X, const upipe_bf16* W_qkv, const upipe_bf16* W_o, int S, int d_model, int H,
                   int G, int d_head, int U, int C, int sched, const upipe_bf16* O_saved, const float* lse,
                   const upipe_bf16* dY, upipe_bf16* dX, float* dW_qkv, float* dW_o, void* ws, size_t ws_bytes,
                   void* stream, upipe_stats* stats) {
  std::vector<unsigned long long> key = {2ull, as_key(X), as_key(W_qkv), as_key(W_o), as_key(O_saved), as_key(lse),
                                         as_key(dY), as_key(dX), as_key(dW_qkv), as_key(dW_o), as_key(ws), ws_bytes};
  for (int v : {S, d_model, H, G, d_head, U, C, sched}) key.push_back(static_cast<unsigned long long>(v));
  return run_graphed(std::move(key), stream, stats, [&](void* st, upipe_stats* sts) {
    return attn_bwd_issue(X, W_qkv, W_o, S, d_model, H, G, d_head, U, C, sched, O_saved, lse, dY, dX, dW_qkv, dW_o, ws,
                          ws_bytes, st, sts);
  });
}

int upipe_graphs_enable(int on) {
  std::vector<GraphEntry> old;
  {
    std::lock_guard<std::mutex> g(g_graphs.mu);
    g_graphs.on = on != 0;
    if (!g_graphs.on) old.swap(g_graphs.entries);
  }
  if (!old.empty()) {
    // replays may still be in flight on any stream
    if (cudaDeviceSynchronize() != cudaSuccess) return UPIPE_ECUDA;
    for (GraphEntry& e : old) cudaGraphExecDestroy(e.exec);
  }
  return UPIPE_OK;
}

size_t upipe_chunked_workspace_bytes(int S, int d_model, int H, int G, int d_head, int U, int C, int n_chunks,
                                     int backward) {
  const Shape s{S, d_model, H, G, d_head, U, C, UPIPE_SCHED_INORDER};
  if (check_chunks(s, n_chunks) != UPIPE_OK) return 0;
  return make_chunk_plan(s, n_chunks, backward != 0).total;
}

size_t upipe_chunked_store_bytes(int S, int d_model, int H, int G, int d_head, int U, int C, int n_chunks,
                                 int backward) {
  const Shape s{S, d_model, H, G, d_head, U, C, UPIPE_SCHED_INORDER};
  if (check_chunks(s, n_chunks) != UPIPE_OK) return 0;
  return make_chunk_plan(s, n_chunks, backward != 0).store;
}

int upipe_attn_fwd_chunked(const upipe_bf16* X, const upipe_bf16* W_qkv, const upipe_bf16* W_o, int S, int d_model,
                           int H, int G, int d_head, int U, int C, int n_chunks, upipe_bf16* Y, upipe_bf16* O_saved,
                           float* lse, void* ws, size_t ws_bytes, void* store, size_t store_bytes, void* stream,
                           upipe_stats* stats) {
  return attn_fwd_chunked_issue(X, W_qkv, W_o, S, d_model, H, G, d_head, U, C, n_chunks, Y, O_saved, lse, ws,
                                ws_bytes, store, store_bytes, stream, stats);
}

int upipe_attn_bwd_chunked(const upipe_bf16* X, const upipe_bf16* W_qkv, const upipe_bf16* W_o, int S, int d_model,
                           int H, int G, int d_head, int U, int C, int n_chunks, const upipe_bf16* O_saved,
                           const float* lse, const upipe_bf16* dY, upipe_bf16* dX, float* dW_qkv, float* dW_o,
                           void* ws, size_t ws_bytes, void* store, size_t store_bytes, void* stream,
                           upipe_stats* stats) {
  return attn_bwd_chunked_issue(X, W_qkv, W_o, S, d_model, H, G, d_head, U, C, n_chunks, O_saved, lse, dY, dX, dW_qkv,
                                dW_o, ws, ws_bytes, store, store_bytes, stream, stats);
}


int upipe_layout_seq2head(const upipe_bf16* src, upipe_bf16* dst, int S, int n_heads, int d_head, int C,
                          int src_row_stride, void* stream) {
  if (!src || !dst || !aligned16(src) || !aligned16(dst) || S <= 0 || n_heads <= 0 || C <= 0 || d_head <= 0)
    return UPIPE_EINVAL;
  if (n_heads % C || S % C || d_head % 8 || src_row_stride % 8 || src_row_stride < n_heads * d_head)
    return UPIPE_EINVAL;
  if (n_heads > kMaxSlots) return UPIPE_EUNSUPPORTED;
  // rank c receives heads c*n/C .. (c+1)*n/C-1, so destination slot k holds head k
  Seq2HeadDesc x;
  x.src = src; x.ld_src = src_row_stride; x.dst = dst; x.S = S; x.D = d_head; x.n_slots = n_heads;
  for (int k = 0; k < n_heads; ++k) x.src_head[k] = static_cast<uint16_t>(k);
  return launch_seq2head(x, static_cast<cudaStream_t>(stream)) == cudaSuccess ? UPIPE_OK : UPIPE_ECUDA;
}

int upipe_layout_head2seq(const upipe_bf16* src, upipe_bf16* dst, int S, int n_heads, int d_head, int C,
                          int dst_row_stride, void* stream) {
  if (!src || !dst || !aligned16(src) || !aligned16(dst) || S <= 0 || n_heads <= 0 || C <= 0 || d_head <= 0)
    return UPIPE_EINVAL;
  if (n_heads % C || S % C || d_head % 8 || dst_row_stride % 8 || dst_row_stride < n_heads * d_head)
    return UPIPE_EINVAL;
  if (n_heads > kMaxSlots) return UPIPE_EUNSUPPORTED;
  Head2SeqDesc h;
  h.src = src; h.src_f32 = false; h.dst = dst; h.ld_dst = dst_row_stride; h.S = S; h.D = d_head; h.n_heads = n_heads;
  for (int k = 0; k < n_heads; ++k) {
    h.dst_head[k] = static_cast<uint16_t>(k);
    h.first[k] = static_cast<uint16_t>(k);
    h.src_slot[k] = static_cast<uint16_t>(k);
  }
  h.first[n_heads] = static_cast<uint16_t>(n_heads);
  return launch_head2seq(h, static_cast<cudaStream_t>(stream)) == cudaSuccess ? UPIPE_OK : UPIPE_ECUDA;
}

int upipe_layout_head2seq_sum(const float* src, int n_src, const int32_t* head_of_src, upipe_bf16* dst, int S,
                              int n_heads, int d_head, int dst_row_stride, void* stream) {
  if (!src || !dst || !head_of_src || !aligned16(src) || !aligned16(dst)) return UPIPE_EINVAL;
  if (S <= 0 || n_src <= 0 || n_heads <= 0 || d_head <= 0 || d_head % 8 || dst_row_stride % 8 ||
      dst_row_stride < static_cast<long long>(n_heads) * d_head)
    return UPIPE_EINVAL;
  if (n_src > kMaxSlots || n_heads > kMaxSlots) return UPIPE_EUNSUPPORTED;
  Head2SeqDesc h;
  h.src = src; h.src_f32 = true; h.dst = dst; h.ld_dst = dst_row_stride; h.S = S; h.D = d_head; h.n_heads = n_heads;
  // CSR of the source slots of each output head, ascending slot order
  int n = 0;
  for (int k = 0; k < n_heads; ++k) {
    h.dst_head[k] = static_cast<uint16_t>(k);
    h.first[k] = static_cast<uint16_t>(n);
    for (int j = 0; j < n_src; ++j)
      if (head_of_src[j] == k) h.src_slot[n++] = static_cast<uint16_t>(j);
    if (n == h.first[k]) return UPIPE_EINVAL;  // an output head without a source
  }
  if (n != n_src) return UPIPE_EINVAL;  // a source slot naming no output head
  h.first[n_heads] = static_cast<uint16_t>(n);
  return launch_head2seq(h, static_cast<cudaStream_t>(stream)) == cudaSuccess ? UPIPE_OK : UPIPE_ECUDA;
}

int upipe_schedule_table(int H, int G, int U, int C, int sched, int32_t* host_out) {
  const Shape s{128 * (C > 0 ? C : 1), 128, H, G, 64, U, C, sched};  // only H, G, U, C matter here
  if (!host_out) return UPIPE_EINVAL;
  const int rc = check_shape(s);
  if (rc != UPIPE_OK) return rc;
  const int qpr = U / C;
  for (int i = 0; i < H / U; ++i)
    for (int r = 0; r < C; ++r)
      for (int j = 0; j < qpr; ++j) host_out[(i * C + r) * qpr + j] = sched_head(s, i, r, j);
  return UPIPE_OK;
}

int upipe_choose_u(int S, int d_model, int H, int G, int d_head, int C, int sched, size_t budget_bytes) {
  int best = 0;
  for (int U = 1; U <= H; ++U) {
    const Shape s{S, d_model, H, G, d_head, U, C, sched};
    if (check_shape(s) != UPIPE_OK) continue;
    const size_t need = std::max(make_plan(s, false).total, make_plan(s, true).total);
    if (need <= budget_bytes) best = U;
  }
  return best;
}

int upipe_choose_chunks(int S, int d_model, int H, int G, int d_head, int U, int C, size_t budget_bytes) {
  for (int n = 1; n <= S / 128; ++n) {
    const Shape s{S, d_model, H, G, d_head, U, C, UPIPE_SCHED_INORDER};
    if (check_chunks(s, n) != UPIPE_OK) continue;
    const size_t need = std::max(make_chunk_plan(s, n, false).total, make_chunk_plan(s, n, true).total);
    if (need <= budget_bytes) return n;
  }
  return 0;
}

int upipe_attention_fwd(const upipe_bf16* Q, const upipe_bf16* K, const upipe_bf16* V, int n_q, int n_kv, int S,
                        int d_head, const int32_t* kv_of_q, upipe_bf16* O, float* lse, void* stream) {
  const void* ptrs[] = {Q, K, V, O, lse};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return UPIPE_EINVAL;
  if (!kv_of_q || n_q <= 0 || n_kv <= 0 || S <= 0 || S % 128) return UPIPE_EINVAL;
  if (d_head != 64 && d_head != 128) return UPIPE_EUNSUPPORTED;
  if (n_q > kMaxSlots || n_q > 65535 / 1) return UPIPE_EUNSUPPORTED;
  for (int k = 0; k < n_q; ++k)
    if (kv_of_q[k] < 0 || kv_of_q[k] >= n_kv) return UPIPE_EINVAL;
  if (!device_supported()) return UPIPE_EUNSUPPORTED;
  int* status = status_ptr();
  if (!status) return UPIPE_ECUDA;
  AttnFwdDesc a;
  a.Q = Q; a.K = K; a.V = V; a.O = O; a.lse = lse;
  a.S = S; a.D = d_head; a.n_qslots = n_q; a.n_kvslots = n_kv;
  for (int k = 0; k < n_q; ++k) {
    a.kv_slot[k] = static_cast<uint16_t>(kv_of_q[k]);
    a.lse_row[k] = static_cast<uint16_t>(k);
  }
  return launch_attn_fwd(a, status, static_cast<cudaStream_t>(stream)) == cudaSuccess ? UPIPE_OK : UPIPE_ECUDA;
}

int upipe_quantize_e4m3(const upipe_bf16* src, int S, int n_heads, int d_head, long long src_row_stride,
                        int per_row, uint8_t* dst, float* scales, void* stream) {
  if (!src || !dst || !scales || !aligned16(src) || !aligned16(dst) || !aligned16(scales)) return UPIPE_EINVAL;
  if (S <= 0 || S % 128 || n_heads <= 0 || src_row_stride < static_cast<long long>(n_heads) * d_head ||
      src_row_stride % 8)
    return UPIPE_EINVAL;
  if (d_head != 64 && d_head != 128) return UPIPE_EUNSUPPORTED;
  if (n_heads > kMaxSlots) return UPIPE_EUNSUPPORTED;
  if (!device_supported()) return UPIPE_EUNSUPPORTED;
  QuantDesc q;
  q.src = src; q.ld_src = src_row_stride; q.dst = dst; q.scale = scales;
  q.S = S; q.D = d_head; q.n_slots = n_heads; q.per_row = per_row != 0;
  for (int k = 0; k < n_heads; ++k) q.src_head[k] = static_cast<uint16_t>(k);
  return launch_quant_e4m3(q, static_cast<cudaStream_t>(stream)) == cudaSuccess ? UPIPE_OK : UPIPE_ECUDA;
}

int upipe_attention_fwd_fp8(const uint8_t* Q, const float* q_scale, const uint8_t* K, const float* k_scale,
                            const upipe_bf16* V, int n_q, int n_kv, int S, int d_head, const int32_t* kv_of_q,
                            upipe_bf16* O, float* lse, void* stream) {
  const void* ptrs[] = {Q, q_scale, K, k_scale, V, O, lse};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return UPIPE_EINVAL;
  if (!kv_of_q || n_q <= 0 || n_kv <= 0 || S <= 0 || S % 128) return UPIPE_EINVAL;
  if (d_head != 128) return UPIPE_EUNSUPPORTED;
  if (n_q > kMaxSlots) return UPIPE_EUNSUPPORTED;
  for (int k = 0; k < n_q; ++k)
    if (kv_of_q[k] < 0 || kv_of_q[k] >= n_kv) return UPIPE_EINVAL;
  if (!device_supported()) return UPIPE_EUNSUPPORTED;
  int* status = status_ptr();
  if (!status) return UPIPE_ECUDA;
  AttnFwdDesc a;
  a.Q = Q; a.K = K; a.V = V; a.O = O; a.lse = lse;
  a.fp8 = true; a.q_scale = q_scale; a.k_scale = k_scale;
  a.S = S; a.D = d_head; a.n_qslots = n_q; a.n_kvslots = n_kv;
  for (int k = 0; k < n_q; ++k) {
    a.kv_slot[k] = static_cast<uint16_t>(kv_of_q[k]);
    a.lse_row[k] = static_cast<uint16_t>(k);
  }
  return launch_attn_fwd(a, status, static_cast<cudaStream_t>(stream)) == cudaSuccess ? UPIPE_OK : UPIPE_ECUDA;
}

int upipe_attn_fwd_fp8(const upipe_bf16* X, const upipe_bf16* W_qkv, const upipe_bf16* W_o, int S, int d_model,
                       int H, int G, int d_head, int U, int C, const uint8_t* fp8_heads, upipe_bf16* Y,
                       upipe_bf16* O_saved, float* lse, void* ws, size_t ws_bytes, void* stream, upipe_stats* stats) {
  const Shape s{S, d_model, H, G, d_head, U, C, UPIPE_SCHED_INORDER};
  int rc = check_shape(s);
  if (rc != UPIPE_OK) return rc;
  if (!fp8_heads) return UPIPE_EINVAL;
  const Plan p = make_plan(s, false);
  bool any = false;
  for (const Stage& g : p.st) {
    const uint8_t f = fp8_heads[g.q_heads[0]] ? 1 : 0;
    for (int h : g.q_heads)
      if ((fp8_heads[h] ? 1 : 0) != f) return UPIPE_EINVAL;  // a stage runs in one precision
    any = any || f;
  }
  if (any) {
    if (d_head != 128) return UPIPE_EUNSUPPORTED;
    // the FP8 buffers must fit where the stage's bf16 head-layout buffers go
    const size_t region = static_cast<size_t>(U + 2 * p.n_kv_slots) * S * d_head * 2;
    if (fp8_stage_buffers(p, nullptr).bytes > region) return UPIPE_EUNSUPPORTED;
  }
  return attn_fwd_issue(X, W_qkv, W_o, S, d_model, H, G, d_head, U, C, UPIPE_SCHED_INORDER, Y, O_saved, lse, ws,
                        ws_bytes, stream, stats, false, any ? fp8_heads : nullptr);
}

int upipe_attn_bwd_fp8(const upipe_bf16* X, const upipe_bf16* W_qkv, const upipe_bf16* W_o, int S, int d_model,
                       int H, int G, int d_head, int U, int C, const uint8_t* fp8_heads, const upipe_bf16* O_saved,
                       const float* lse, const upipe_bf16* dY, upipe_bf16* dX, float* dW_qkv, float* dW_o, void* ws,
                       size_t ws_bytes, void* stream, upipe_stats* stats) {
  const Shape s{S, d_model, H, G, d_head, U, C, UPIPE_SCHED_INORDER};
  int rc = check_shape(s);
  if (rc != UPIPE_OK) return rc;
  if (!fp8_heads) return UPIPE_EINVAL;
  const Plan p = make_plan(s, true);
  bool any = false;
  for (const Stage& g : p.st) {
    const uint8_t f = fp8_heads[g.q_heads[0]] ? 1 : 0;
    for (int h : g.q_heads)
      if ((fp8_heads[h] ? 1 : 0) != f) return UPIPE_EINVAL;  // a stage runs in one precision
    any = any || f;
  }
  if (any) {
    if (d_head != 128) return UPIPE_EUNSUPPORTED;
    const size_t region = static_cast<size_t>(U + 2 * p.n_kv_slots) * S * d_head * 2;
    if (fp8_stage_buffers(p, nullptr).bytes > region) return UPIPE_EUNSUPPORTED;
  }
  return attn_bwd_issue(X, W_qkv, W_o, S, d_model, H, G, d_head, U, C, UPIPE_SCHED_INORDER, O_saved, lse, dY, dX,
                        dW_qkv, dW_o, ws, ws_bytes, stream, stats, any ? fp8_heads : nullptr);
}

int upipe_attention_bwd_fp8(const uint8_t* Q, const float* q_scale, const uint8_t* K, const float* k_scale,
                            const upipe_bf16* V, const upipe_bf16* O, const upipe_bf16* dO, const float* lse, int n_q,
                            int n_kv, int S, int d_head, const int32_t* kv_of_q, float* dQ, float* dK, float* dV,
                            void* ws, size_t ws_bytes, void* stream) {
  if (!q_scale || !k_scale || !aligned16(q_scale) || !aligned16(k_scale)) return UPIPE_EINVAL;
  const int rc = attention_bwd_check(Q, K, V, O, dO, lse, n_q, n_kv, S, d_head, kv_of_q, dQ, dK, dV);
  if (rc != UPIPE_OK) return rc;
  if (d_head != 128) return UPIPE_EUNSUPPORTED;
  if (!ws || !aligned16(ws)) return UPIPE_EINVAL;
  if (ws_bytes < attention_bwd_scratch_bytes(n_q, S)) return UPIPE_ENOSPC;
  if (!device_supported()) return UPIPE_EUNSUPPORTED;
  int* status = status_ptr();
  if (!status) return UPIPE_ECUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* dsum = static_cast<float*>(ws);
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
  ab.fp8 = true; ab.q_scale = q_scale; ab.k_scale = k_scale;
  for (int k = 0; k < n_q; ++k) ab.kv_slot[k] = static_cast<uint16_t>(kv_of_q[k]);
  return launch_attn_bwd(ab, status, st) == cudaSuccess ? UPIPE_OK : UPIPE_ECUDA;
}

int upipe_attention_bwd(const upipe_bf16* Q, const upipe_bf16* K, const upipe_bf16* V, const upipe_bf16* O,
                        const upipe_bf16* dO, const float* lse, int n_q, int n_kv, int S, int d_head,
                        const int32_t* kv_of_q, float* dQ, float* dK, float* dV, void* ws, size_t ws_bytes,
                        void* stream) {
  const int rc = attention_bwd_check(Q, K, V, O, dO, lse, n_q, n_kv, S, d_head, kv_of_q, dQ, dK, dV);
  if (rc != UPIPE_OK) return rc;
  if (!ws || !aligned16(ws)) return UPIPE_EINVAL;
  if (ws_bytes < attention_bwd_scratch_bytes(n_q, S)) return UPIPE_ENOSPC;
  return attention_bwd_enqueue(Q, K, V, O, dO, lse, n_q, n_kv, S, d_head, kv_of_q, dQ, dK, dV, ws,
                               static_cast<cudaStream_t>(stream));
}

int upipe_gemm_bf16(const upipe_bf16* A, const upipe_bf16* B, void* D, int M, int N, int K, int a_trans, int b_trans,
                    long long lda, long long ldb, long long ldd, int out_mode, void* stream) {
  if (!A || !B || !D || !aligned16(A) || !aligned16(B) || !aligned16(D)) return UPIPE_EINVAL;
  if (M <= 0 || N <= 0 || K <= 0 || M % 64 || N % 64 || K % 64) return UPIPE_EINVAL;
  if (out_mode < 0 || out_mode > 3 || lda % 8 || ldb % 8 || ldd % 8) return UPIPE_EINVAL;
  if (!device_supported()) return UPIPE_EUNSUPPORTED;
  int* status = status_ptr();
  if (!status) return UPIPE_ECUDA;
  GemmDesc g;
  g.A = A; g.lda = lda; g.a_mn = a_trans != 0;
  g.a_rows = a_trans ? K : M; g.a_cols = a_trans ? M : K;
  g.B = B; g.ldb = ldb; g.b_mn = b_trans == 0;
  g.b_rows = b_trans ? N : K; g.b_cols = b_trans ? K : N;
  if (g.a_cols > lda || g.b_cols > ldb) return UPIPE_EINVAL;
  g.M = M; g.N = N; g.K = K;
  g.out = D; g.ldo = ldd;
  g.out_mode = out_mode == 0 ? kOutBf16 : (out_mode == 1 ? kOutF32 : (out_mode == 2 ? kOutF32Acc : kOutF32Red));
  if (out_mode == 3) g.split_k = choose_split_k(g);
  return launch_gemm(g, status, static_cast<cudaStream_t>(stream)) == cudaSuccess ? UPIPE_OK : UPIPE_ECUDA;
}

int upipe_sync_status(void* stream) {
  int* st = status_ptr();
  if (!st) return UPIPE_ECUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return UPIPE_ECUDA;
  int v = 0;
  if (cudaMemcpy(&v, st, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return UPIPE_ECUDA;
  if (v != 0) {
    const int zero = 0;
    cudaMemcpy(st, &zero, sizeof(int), cudaMemcpyHostToDevice);
    return UPIPE_ETIMEOUT;
  }
  return UPIPE_OK;
}

const char* upipe_status_str(int status) {
  switch (status) {
    case UPIPE_OK: return "ok";
    case UPIPE_EINVAL: return "invalid argument (shape, null or misaligned pointer)";
    case UPIPE_ENOSPC: return "workspace too small";
    case UPIPE_EUNSUPPORTED: return "unsupported (head width, sizes or GPU)";
    case UPIPE_ECUDA: return "CUDA launch or runtime error";
    case UPIPE_ETIMEOUT: return "a kernel wait timed out";
    default: return "unknown status";
  }
}

int upipe_version(void) { return 100; }

int upipe_profile_enable(int on) {
  std::lock_guard<std::mutex> g(g_prof.mu);
  g_prof.on = on != 0;
  g_prof.used = 0;
  return UPIPE_OK;
}

int upipe_profile_read(double* ms_by_kind, int* count_by_kind) {
  if (!ms_by_kind || !count_by_kind) return UPIPE_EINVAL;
  std::lock_guard<std::mutex> g(g_prof.mu);
  for (int k = 0; k < UPIPE_KERNEL_KINDS; ++k) {
    ms_by_kind[k] = 0.0;
    count_by_kind[k] = 0;
  }
  for (size_t i = 0; i < g_prof.used; ++i) {
    if (cudaEventSynchronize(g_prof.ev[2 * i + 1]) != cudaSuccess) return UPIPE_ECUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]) != cudaSuccess) return UPIPE_ECUDA;
    ms_by_kind[g_prof.kind[i]] += ms;
    count_by_kind[g_prof.kind[i]] += 1;
  }
  g_prof.used = 0;
  return UPIPE_OK;
}

}  // extern "C"
