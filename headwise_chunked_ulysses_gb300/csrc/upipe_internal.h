// Internal interfaces between the host orchestration and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace upipe {

constexpr int kMaxMap = 256;   // 64-wide blocks a gather map can name
constexpr int kMaxSlots = 256; // head slots one attention launch can hold

// A gather over 64-element blocks: block b of the logical operand comes from
// block idx[b] of the stored tensor.  n == 0 means identity.
struct BlockMap {
  int n = 0;
  uint16_t idx[kMaxMap];
};

enum GemmOut : int {
  kOutBf16 = 0,        // out(bf16)  = acc
  kOutF32 = 1,         // out(fp32)  = acc
  kOutF32Acc = 2,      // out(fp32) += acc
  kOutBf16PlusF32 = 3, // out(bf16)  = acc + aux(fp32)
  kOutF32Red = 4,      // out(fp32) += acc with vector atomics (split-K partial sums)
};

// D[M,N] = A[M,K] * B[K,N], bf16 operands, fp32 accumulation.
//   a_mn == false: A stored [M rows][K cols] (K contiguous), else [K rows][M cols].
//   b_mn == false: B stored [N rows][K cols],                else [K rows][N cols].
// lda/ldb are the stored row strides in elements.  amap_k / bmap_k gather
// along K, bmap_n gathers along N, omap_n scatters output column blocks.
struct GemmDesc {
  const void* A = nullptr; long long lda = 0; long long a_rows = 0; long long a_cols = 0; bool a_mn = false;
  const void* B = nullptr; long long ldb = 0; long long b_rows = 0; long long b_cols = 0; bool b_mn = false;
  int M = 0, N = 0, K = 0;
  BlockMap amap_k, bmap_k, bmap_n, omap_n;
  void* out = nullptr; long long ldo = 0; int out_mode = kOutF32;
  const float* aux = nullptr; long long ld_aux = 0;
  int split_k = 1;  // > 1 only with kOutF32Red: K is cut into split_k ranges of K/64/split_k blocks, rounded either way
};

// Epilogues of the attention forward: one launch over all keys (plain), or
// one of several launches over disjoint key chunks whose results merge by
// log-sum-exp in an fp32 accumulator (first, middle, last; the last writes O
// and lse).
enum { kFwdPlain = 0, kFwdFirst = 1, kFwdMiddle = 2, kFwdLast = 3 };

struct AttnFwdDesc {
  const void* Q = nullptr;  // [n_qslots][S][D] bf16
  const void* K = nullptr;  // [n_kvslots][kv_ld][D] bf16, rows [0, kv_len) used
  const void* V = nullptr;  // [n_kvslots][kv_ld][D] bf16
  void* O = nullptr;        // [n_qslots][S][D] bf16
  float* lse = nullptr;     // rows lse_row[slot], lse_ld apart (natural log)
  int S = 0, D = 0, n_qslots = 0, n_kvslots = 0;
  // Query row r sits at key position q_off + r (a multiple of 128, >= 0): it
  // sees the keys at positions <= q_off + r below kv_len.  Defaults (0):
  // kv_len = kv_ld = lse_ld = S, q_off = 0, the plain causal case.
  int kv_len = 0, kv_ld = 0, q_off = 0, lse_ld = 0;
  int mode = kFwdPlain;
  float* o_acc = nullptr;    // [n_qslots][S][D] fp32 running output (merge modes)
  float* lse_acc = nullptr;  // [n_qslots][S] fp32 running log-sum-exp, log2 units
  // FP8 scores (D = 128 only): Q and K hold E4M3 codes, one byte each; the
  // score of (row r, key j) is their dot product times q_scale[slot][r] times
  // k_scale[kv slot][j / 128] (k_scale rows are kv_ld / 128 long)
  bool fp8 = false;
  const float* q_scale = nullptr;
  const float* k_scale = nullptr;
  uint16_t kv_slot[kMaxSlots];
  uint16_t lse_row[kMaxSlots];
};

struct AttnBwdDesc {
  const void* Q = nullptr;   // [n_qslots][S][D] bf16
  const void* K = nullptr;   // [n_kvslots][kv_ld][D] bf16, rows [0, kv_len) used
  const void* V = nullptr;   // [n_kvslots][kv_ld][D] bf16
  const void* dO = nullptr;  // [n_qslots][S][D] bf16
  const float* lse2 = nullptr;  // [n_qslots][S]  minus the log-sum-exp in log2 units
  const float* Dsum = nullptr;  // [n_qslots][S]  rowsum(dO * O)
  // fp32 per query slot, [slot][S][D] row-major, pre-zeroed; every KV block
  // adds its share by TMA reduce-adds of 32 x 32 chunks staged in shared memory
  float* dQacc = nullptr;
  float* dK = nullptr;       // [n_kvslots][kv_ld][D] fp32
  float* dV = nullptr;       // [n_kvslots][kv_ld][D] fp32
  int accumulate_kv = 0;     // add into dK/dV instead of overwriting
  int S = 0, D = 0, n_qslots = 0, n_kvslots = 0;
  // key positions as in AttnFwdDesc (defaults: kv_len = kv_ld = S, q_off = 0)
  int kv_len = 0, kv_ld = 0, q_off = 0;
  // CTAs per KV block (1..16), each taking a contiguous share of the block's
  // (query slot, query block) items; above 1, dK and dV are ADDED atomically
  // into buffers that hold zeros or earlier partial sums (accumulate_kv is
  // then implied and nothing is zero-filled)
  int q_split = 1;
  // FP8 heads (plain launch, D = 128): Q and K hold E4M3 codes,
  // one byte each, with q_scale [n_qslots][S] and k_scale [n_kvslots][kv_ld / 128]
  bool fp8 = false;
  const float* q_scale = nullptr;
  const float* k_scale = nullptr;
  uint16_t kv_slot[kMaxSlots];  // q slot -> kv slot
};

// Copy of head blocks between sequence layout [S][row of heads] and head
// layout [slot][S][D].
struct Seq2HeadDesc {
  const uint16_t* src = nullptr; long long ld_src = 0;  // elements per token row
  uint16_t* dst = nullptr;                              // [n_slots][S][D]
  int S = 0, D = 0, n_slots = 0;
  uint16_t src_head[kMaxSlots];  // slot -> head block in a source row
};
struct Head2SeqDesc {
  const void* src = nullptr; bool src_f32 = false;       // [*][S][D]
  uint16_t* dst = nullptr; long long ld_dst = 0;         // bf16 [S][row]
  int S = 0, D = 0, n_heads = 0;
  uint16_t dst_head[kMaxSlots];     // output head -> head block in a dest row
  uint16_t first[kMaxSlots + 1];    // CSR over source slots per output head
  uint16_t src_slot[kMaxSlots];     // summed in this order (fp32)
};
struct BwdPrepDesc {
  const uint16_t* dO = nullptr; long long ld_do = 0;  // seq layout
  const uint16_t* O = nullptr; long long ld_o = 0;    // seq layout (saved forward output)
  const float* lse = nullptr;                         // [*][lse_ld] natural log
  long long lse_ld = 0;                               // 0: S
  float* Dsum = nullptr;   // [n_slots][S]
  float* lse2 = nullptr;   // [n_slots][S]  -lse * log2(e)
  float* dQacc = nullptr;  // [n_slots][S][D], zeroed here
  int S = 0, D = 0, n_slots = 0;
  // slot -> start of its d-wide block, in units of D elements: a head index
  // for sequence layout, slot*S for head layout (with ld == D)
  int32_t do_unit[kMaxSlots];
  int32_t o_unit[kMaxSlots];
  uint16_t lse_row[kMaxSlots];  // slot -> lse row
};

// Sequence layout (bf16) -> head layout in E4M3 codes, with fp32 scales
// amax/448 (1 for an all-zero group): one per row (per_row) or one per 128
// rows (per 128-key block).  S a multiple of 128, D 64 or 128.
struct QuantDesc {
  const uint16_t* src = nullptr; long long ld_src = 0;  // elements per token row
  uint8_t* dst = nullptr;                               // [n_slots][S][D]
  float* scale = nullptr;                               // [n_slots][S] or [n_slots][S/128]
  int S = 0, D = 0, n_slots = 0;
  bool per_row = true;
  uint16_t src_head[kMaxSlots];
};

// Launchers (return cudaError_t of the launch).
cudaError_t launch_gemm(const GemmDesc& g, int* status, cudaStream_t st);
cudaError_t launch_attn_fwd(const AttnFwdDesc& a, int* status, cudaStream_t st);
cudaError_t launch_attn_bwd(const AttnBwdDesc& a, int* status, cudaStream_t st);
cudaError_t launch_seq2head(const Seq2HeadDesc& p, cudaStream_t st);
cudaError_t launch_head2seq(const Head2SeqDesc& p, cudaStream_t st);
cudaError_t launch_bwd_prep(const BwdPrepDesc& p, cudaStream_t st);
cudaError_t launch_quant_e4m3(const QuantDesc& p, cudaStream_t st);

// Tensor maps (driver entry point resolved through the runtime).
bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_stride_elems,
                    uint32_t box_inner, uint32_t box_outer);
bool make_tmap_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_stride_elems,
                  uint32_t box_inner, uint32_t box_outer);
bool make_tmap_f32(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_stride_elems,
                   uint32_t box_inner, uint32_t box_outer);
// Facts of the current device, looked up once per device with it current.
int num_sms();
bool device_supported();  // compute capability 10.3
// Device address of the current device's status word that bounded waits
// write (read and cleared by upipe_sync_status).
int* device_status_word();
// Raises a kernel's dynamic shared-memory limit on the current device (once
// per device and kernel).
cudaError_t ensure_dynamic_smem(const void* kernel, int bytes);

// The attention backward of one stage's heads in head layout, shared by
// upipe_attention_bwd (scratch in the caller's workspace) and
// upipe_attention_bwd_noalloc (scratch in a fixed array of the library).
// Scratch: D = rowsum(dO * O) and -lse * log2(e), n_q * S floats each.
size_t attention_bwd_scratch_bytes(int n_q, int S);
// Argument checks of the public call (pointers, shape, KV slot map); UPIPE_* code.
int attention_bwd_check(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* lse,
                        int n_q, int n_kv, int S, int d_head, const int32_t* kv_of_q, const float* dQ,
                        const float* dK, const float* dV);
// Enqueues the preprocessing and the backward kernel on st; arguments already
// checked; scratch holds attention_bwd_scratch_bytes() bytes of device memory.
int attention_bwd_enqueue(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                          const float* lse, int n_q, int n_kv, int S, int d_head, const int32_t* kv_of_q, float* dQ,
                          float* dK, float* dV, void* scratch, cudaStream_t st);

}  // namespace upipe
