/*
 * upipe.h -- C ABI of the headwise-chunked (UPipe) causal GQA attention layer
 * on one GB300 (sm_103a).
 *
 * The operation is the attention layer of "Untied Ulysses: Memory-Efficient
 * Context Parallelism via Headwise Chunking" (summary page, paper.rainbus.top):
 *   - Core method: attention runs in H/U stages of U heads; the stage buffers
 *     are reused, so intermediate memory grows with U, not H.
 *   - Method steps (1)-(4): per stage, project X onto the Q, K, V of heads
 *     iU..(i+1)U-1; all-to-all from sequence shards (S/C tokens per rank) to
 *     head shards (U/C heads of all S tokens per rank); causal attention;
 *     all-to-all back.  Each stage then adds its heads' share of the output
 *     projection, O_s W_o[rows of s], into Y.
 *   - Novelty: the GQA schedule takes heads out of order so every KV head is
 *     exchanged once, in the first stage, and later stages move query heads only.
 *   - Background: DeepSpeed Ulysses (the all-to-all) and GQA (H query heads
 *     share G KV heads, H/G consecutive query heads per KV head).
 * The C ranks are virtual: their buffers sit side by side in one GPU's memory
 * and the all-to-all is a device permute with the same index map.
 *
 * Beyond the plain layer calls (each documented at its declaration): the next
 * stage's projection overlapped with the current attention
 * (upipe_fwd_workspace_bytes_prefetch), CUDA-graph replay for short sequences
 * (upipe_graphs_enable), stage-width and chunk-count choosers for a memory
 * budget (upipe_choose_u, upipe_choose_chunks), head stages on sequence
 * chunks with an offload store (upipe_attn_fwd_chunked / _bwd_chunked) and
 * FP8 scores for chosen stages (upipe_attn_fwd_fp8).
 *
 * Conventions for every call:
 *   - All tensors are row-major.  bf16 values are passed as upipe_bf16 bit
 *     patterns; fp32 as float.
 *   - X, Y, dY, dX: [S, d_model].  W_qkv: [d_model, (H + 2G) d_head], columns
 *     [Q head 0..H-1 | K head 0..G-1 | V head 0..G-1], d_head columns each.
 *     W_o: [H d_head, d_model].  O_saved: [S, H d_head].  lse: [H, S], natural
 *     log of each causal softmax row's normaliser (scores scaled 1/sqrt(d_head)).
 *   - Pointers named as device pointers must be device memory the caller owns
 *     and 16-byte aligned.  The library never allocates device memory and keeps
 *     no pointer after a call returns (except the graphs of
 *     upipe_graphs_enable, which hold the pointers of the calls they captured
 *     until graphs are turned off).  Work is ordered on `stream` (a
 *     cudaStream_t; NULL is the legacy default stream); calls return once the
 *     work is enqueued.  Two calls may run concurrently only with distinct
 *     workspaces and outputs.
 *   - Return value: UPIPE_OK or an error code.  Argument checks happen before
 *     any launch: on an error nothing has been enqueued, except for
 *     UPIPE_ECUDA (a launch failed) and UPIPE_ETIMEOUT.
 *   - Shape rules (method constraints and kernel tiling): U | H (stages of U
 *     heads), C | U (U/C heads per rank; the pages' Limitations section),
 *     G | H, C | S, S % 128 == 0, d_model % 64 == 0, d_head in {64, 128},
 *     H + 2G <= 256 heads in one stage; the out-of-order schedule also needs
 *     C | G or G | C.
 */
#ifndef UPIPE_H
#define UPIPE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t upipe_bf16; /* bfloat16 storage */

enum upipe_status {
  UPIPE_OK = 0,
  UPIPE_EINVAL = 1,      /* bad shape, null or misaligned pointer */
  UPIPE_ENOSPC = 2,      /* workspace smaller than *_workspace_bytes() */
  UPIPE_EUNSUPPORTED = 3,/* d_head not 64/128, or the GPU is not sm_103 */
  UPIPE_ECUDA = 4,       /* a CUDA launch or runtime call failed */
  UPIPE_ETIMEOUT = 5     /* a kernel's bounded wait gave up (device status word) */
};

enum upipe_schedule {
  UPIPE_SCHED_INORDER = 0, /* stage i holds heads iU..(i+1)U-1; each query slot gets its KV head */
  UPIPE_SCHED_GQA_OOO = 1  /* rank r keeps heads r*H/C..(r+1)*H/C-1; KV heads move once, stage 0 */
};

/* Kernel kinds, for the statistics and the optional timing below. */
enum upipe_kernel_kind {
  UPIPE_KERNEL_GEMM = 0,
  UPIPE_KERNEL_ATTN_FWD = 1,
  UPIPE_KERNEL_ATTN_BWD = 2,
  UPIPE_KERNEL_SEQ2HEAD = 3,
  UPIPE_KERNEL_HEAD2SEQ = 4,
  UPIPE_KERNEL_BWD_PREP = 5,
  UPIPE_KERNEL_KINDS = 6
};

/* Filled by the layer calls when `stats` is non-NULL. */
typedef struct {
  size_t arena_peak_bytes;        /* stage arena high-water mark of the call's slot plan */
  size_t stage_closed_form_bytes; /* 12*S*U*d_head: the pages' QKV + exchange form, summed over C ranks */
  size_t persistent_bytes;        /* workspace outside the stage arena (fp32 accumulators, resident KV) */
  size_t permute_bytes;           /* bytes read + written by the emulated all-to-alls */
  int launches;                   /* kernel launches enqueued */
  int stages;                     /* H / U */
  /* per kernel kind: launches, algorithmic FLOPs (GEMM 2MNK; attention 2*d per
   * causal (query, key) pair and matmul: 2 matmuls forward, 5 backward) and
   * algorithmic HBM bytes (operands read once, results written once) */
  int launches_by_kind[UPIPE_KERNEL_KINDS];
  double flops_by_kind[UPIPE_KERNEL_KINDS];
  double bytes_by_kind[UPIPE_KERNEL_KINDS];
  size_t offload_bytes;           /* sequence-chunked calls: size of the offload store (0 otherwise) */
  size_t offload_copy_bytes;      /* sequence-chunked calls: bytes copied between store and device */
} upipe_stats;

/* Workspace sizes in bytes for the layer calls (0 if the shape is invalid). */
size_t upipe_fwd_workspace_bytes(int S, int d_model, int H, int G, int d_head, int U, int C, int sched);
size_t upipe_bwd_workspace_bytes(int S, int d_model, int H, int G, int d_head, int U, int C, int sched);
/*
 * Forward workspace with a second stage-buffer set ("Untied Ulysses" summary,
 * paper.rainbus.top, section on weaknesses from an independent analysis:
 * fetch the next stage's QKV while the current stage's attention runs).  When
 * upipe_attn_fwd gets at least this many bytes and the layer has more than
 * one stage, stage i+1's projection and exchange run on a second stream of
 * the library while stage i's attention runs on `stream`; results are the
 * same as with the minimal workspace.  The extra set is O(U): the sequence
 * buffer and the head-layout Q slots, plus their own K and V slots in the
 * in-order schedule.  0 if the shape is invalid.
 */
size_t upipe_fwd_workspace_bytes_prefetch(int S, int d_model, int H, int G, int d_head, int U, int C, int sched);

/*
 * Forward pass of the layer (Method steps (1)-(4) per stage, plus the
 * stage's share of Y = O W_o).
 *   X, W_qkv, W_o : device, bf16, inputs.
 *   Y             : device, bf16 [S, d_model], output.
 *   O_saved       : device, bf16 [S, H*d_head], output (attention output of every
 *                   head, kept for the backward pass).
 *   lse           : device, fp32 [H, S], output.
 *   ws            : device workspace of at least upipe_fwd_workspace_bytes() bytes,
 *                   256-byte aligned; contents on entry are ignored.  With at
 *                   least upipe_fwd_workspace_bytes_prefetch() bytes the next
 *                   stage is projected and exchanged on a second stream.  The
 *                   call then orders that stream after `stream`'s prior work
 *                   and `stream` after all of it, so the caller sees one
 *                   stream's worth of ordering; calls that overlap on one
 *                   device share that second stream.
 */
int upipe_attn_fwd(const upipe_bf16* X, const upipe_bf16* W_qkv, const upipe_bf16* W_o, int S, int d_model,
                   int H, int G, int d_head, int U, int C, int sched, upipe_bf16* Y, upipe_bf16* O_saved,
                   float* lse, void* ws, size_t ws_bytes, void* stream, upipe_stats* stats);

/*
 * Backward pass: gradients of L = <Y, dY>.  The pages do not describe it; it
 * runs the same stages, recomputing each stage's projection and exchange (Q,
 * K, V are never kept), and uses O_saved and lse from the forward call.
 *   dY      : device, bf16 [S, d_model], input.
 *   dX      : device, bf16 [S, d_model], output.
 *   dW_qkv  : device, fp32 [d_model, (H+2G) d_head], output.
 *   dW_o    : device, fp32 [H d_head, d_model], output.
 *   ws      : at least upipe_bwd_workspace_bytes() bytes.
 */
int upipe_attn_bwd(const upipe_bf16* X, const upipe_bf16* W_qkv, const upipe_bf16* W_o, int S, int d_model,
                   int H, int G, int d_head, int U, int C, int sched, const upipe_bf16* O_saved,
                   const float* lse, const upipe_bf16* dY, upipe_bf16* dX, float* dW_qkv, float* dW_o, void* ws,
                   size_t ws_bytes, void* stream, upipe_stats* stats);

/*
 * Head stages combined with sequence chunks ("Untied Ulysses" summary page,
 * paper.rainbus.top, sections Limitations and Future directions: FPDT chunks
 * the sequence and keeps a memory edge through arbitrary chunk sizes, UPipe
 * chunks the heads; the two are orthogonal and may be combined).  In-order
 * schedule only.  The sequence is cut into n_chunks chunks of
 * Sc = S / n_chunks tokens (Sc a multiple of 128 and of C).  Forward: for
 * chunk i = 0, 1, ... and each stage, the chunk's rows are projected onto the
 * stage's heads and exchanged; the stage's K and V of the chunk go to the
 * offload store (one copy per KV head); the chunk's queries attend to KV
 * chunks 0..i, fetched back from the store on a copy stream of the library,
 * the partial softmax results merged by log-sum-exp; the stage's share of
 * O W_o is added to the chunk's rows of Y.  Backward: all K/V chunks are
 * recomputed into the store; query chunks run from the last to the first,
 * partial dK/dV of each KV chunk are kept in the store until their own query
 * chunk completes them.  Outputs and their layouts are those of
 * upipe_attn_fwd / upipe_attn_bwd (same lse, O_saved; the two calls pair
 * with each other only through them).
 *   ws    : device, at least upipe_chunked_workspace_bytes() bytes, 256-byte
 *           aligned; every buffer in it is O(Sc), none O(S).
 *   store : device memory or page-locked host memory (cudaHostAlloc or
 *           registered) of at least upipe_chunked_store_bytes() bytes,
 *           16-byte aligned, owned by the caller: [chunk][K,V][G][Sc][d_head]
 *           bf16 (forward), followed by the same in fp32 for dK, dV
 *           (backward).  Its contents on return are scratch.
 * The sizes return 0 for an invalid shape or chunk count.  Errors: as
 * upipe_attn_fwd / upipe_attn_bwd; UPIPE_EINVAL for a bad chunk count or
 * store pointer, UPIPE_ENOSPC for a short store; a failing copy gives
 * UPIPE_ECUDA.  stats->offload_bytes and offload_copy_bytes report the
 * store size and the bytes the call copied.
 */
size_t upipe_chunked_workspace_bytes(int S, int d_model, int H, int G, int d_head, int U, int C, int n_chunks,
                                     int backward);
size_t upipe_chunked_store_bytes(int S, int d_model, int H, int G, int d_head, int U, int C, int n_chunks,
                                 int backward);
/*
 * Chunk-count chooser for the calls below: the smallest n_chunks (the longest
 * chunks, so the fewest and largest launches) for which both
 * upipe_chunked_workspace_bytes(..., 0) and (..., 1) are at most
 * budget_bytes; 0 if no valid count fits.  The store is not counted (it may
 * live in host memory).  Host only.
 */
int upipe_choose_chunks(int S, int d_model, int H, int G, int d_head, int U, int C, size_t budget_bytes);
int upipe_attn_fwd_chunked(const upipe_bf16* X, const upipe_bf16* W_qkv, const upipe_bf16* W_o, int S, int d_model,
                           int H, int G, int d_head, int U, int C, int n_chunks, upipe_bf16* Y, upipe_bf16* O_saved,
                           float* lse, void* ws, size_t ws_bytes, void* store, size_t store_bytes, void* stream,
                           upipe_stats* stats);
int upipe_attn_bwd_chunked(const upipe_bf16* X, const upipe_bf16* W_qkv, const upipe_bf16* W_o, int S, int d_model,
                           int H, int G, int d_head, int U, int C, int n_chunks, const upipe_bf16* O_saved,
                           const float* lse, const upipe_bf16* dY, upipe_bf16* dX, float* dW_qkv, float* dW_o,
                           void* ws, size_t ws_bytes, void* store, size_t store_bytes, void* stream,
                           upipe_stats* stats);

/*
 * The Ulysses input all-to-all over C virtual ranks (Background, DeepSpeed
 * Ulysses; Method steps (2)).  src is sequence-sharded: device bf16 rows of
 * src_row_stride elements, token t at row t, head h at columns h*d_head..;
 * rank c owns tokens [c S/C, (c+1) S/C).  dst is head-sharded: device bf16
 * [C][n_heads/C][S][d_head], rank c receiving heads c*n_heads/C .. +n_heads/C-1.
 * Needs C | n_heads, C | S, d_head % 8 == 0, src_row_stride % 8 == 0.
 */
int upipe_layout_seq2head(const upipe_bf16* src, upipe_bf16* dst, int S, int n_heads, int d_head, int C,
                          int src_row_stride, void* stream);

/* The reverse exchange (Method steps (4)): head-sharded src
 * [C][n_heads/C][S][d_head] back to sequence-sharded dst rows of
 * dst_row_stride elements.  Same requirements. */
int upipe_layout_head2seq(const upipe_bf16* src, upipe_bf16* dst, int S, int n_heads, int d_head, int C,
                          int dst_row_stride, void* stream);

/*
 * The reverse exchange of the backward pass (Method steps (2) and (4) run
 * backwards): gradients held in head layout return to sequence layout, and
 * the copies of one head that several ranks hold are summed.  In the in-order
 * exchange every query slot receives its own copy of its KV head, so the
 * gradient of that KV head is the sum of the copies' gradients.
 *   src : device fp32 [n_src][S][d_head], one gradient per source slot.
 *   head_of_src : HOST int32 [n_src], the output head each source slot
 *         belongs to; every output head 0..n_heads-1 needs at least one.
 *   dst : device bf16 rows of dst_row_stride elements; head h of token t at
 *         dst[t * dst_row_stride + h * d_head ..].
 * Each output value is the fp32 sum of its sources taken in ascending source
 * slot order (the first source, plus the second, ...; ascending slot order is
 * ascending rank order), rounded once to bf16 (nearest, ties to even).  The
 * result is therefore bit-for-bit reproducible.  d_head % 8 == 0,
 * dst_row_stride % 8 == 0, n_src and n_heads <= 256.
 */
int upipe_layout_head2seq_sum(const float* src, int n_src, const int32_t* head_of_src, upipe_bf16* dst, int S,
                              int n_heads, int d_head, int dst_row_stride, void* stream);

/*
 * Head schedule (Method steps (1)-(2), Novelty): host_out[(i*C + r)*(U/C) + j]
 * receives the query head that stage i places in slot j of rank r.
 * host_out is HOST memory of H int32 entries.
 */
int upipe_schedule_table(int H, int G, int U, int C, int sched, int32_t* host_out);

/*
 * Stage width chooser ("Untied Ulysses" summary, paper.rainbus.top, section
 * on weaknesses from an independent analysis: pick U from the sequence length,
 * large U for short sequences to save launches, small U for long ones to save
 * memory).  Returns the largest U (U | H, C | U, and the schedule's own
 * constraints; U = H is plain Ulysses) for which both
 * upipe_fwd_workspace_bytes() and upipe_bwd_workspace_bytes() are at most
 * budget_bytes, or 0 if no valid U fits or the shape is invalid for every U.
 * Host only: touches no device and allocates nothing.
 */
int upipe_choose_u(int S, int d_model, int H, int G, int d_head, int C, int sched, size_t budget_bytes);

/*
 * Causal GQA attention of one stage's heads in head layout (Method steps (3)).
 *   Q   : device bf16 [n_q][S][d_head];  K, V: device bf16 [n_kv][S][d_head].
 *   kv_of_q : HOST int32 [n_q], the KV slot each query slot reads.
 *   O   : device bf16 [n_q][S][d_head];  lse: device fp32 [n_q][S] (natural log).
 * n_q <= 256, S % 128 == 0.
 */
int upipe_attention_fwd(const upipe_bf16* Q, const upipe_bf16* K, const upipe_bf16* V, int n_q, int n_kv, int S,
                        int d_head, const int32_t* kv_of_q, upipe_bf16* O, float* lse, void* stream);

/*
 * Lower-precision heads ("Untied Ulysses" summary page, paper.rainbus.top,
 * section on weaknesses from an independent analysis: heads that can run in
 * FP8 cut memory and communication further).  FP8 here is E4M3 (4 exponent
 * bits, bias 7, 3 mantissa bits, largest finite 448), round to nearest even,
 * saturating.
 *
 * upipe_quantize_e4m3: the exchange of such heads.  src: device bf16 in
 * sequence layout, token t's head h at src[t * src_row_stride + h * d_head ..]
 * (S a multiple of 128).  dst: device [n_heads][S][d_head] E4M3 codes (one
 * byte each).  scales: device fp32, [n_heads][S] (per_row != 0: one scale per
 * token and head) or [n_heads][S / 128] (one per block of 128 tokens).  Each
 * scale is amax / 448 over its group in fp32 (IEEE division; 1 for an all-zero
 * group) and each code is E4M3(x / scale) with x / scale an IEEE fp32
 * division, so a value = code * scale.  d_head 64 or 128; n_heads <= 64.
 */
int upipe_quantize_e4m3(const upipe_bf16* src, int S, int n_heads, int d_head, long long src_row_stride,
                        int per_row, uint8_t* dst, float* scales, void* stream);

/*
 * Causal GQA attention with FP8 scores: Q and K are E4M3 codes from
 * upipe_quantize_e4m3 (Q per row, K per 128-key block); the score of query i
 * and key j is (Q_i . K_j) * q_scale[i] * k_scale[j / 128] / sqrt(d_head),
 * computed on the tensor cores' FP8 path; the softmax, P (bf16) and P V (bf16
 * V) are as in upipe_attention_fwd, and so are O and lse.  d_head 128 only.
 */
int upipe_attention_fwd_fp8(const uint8_t* Q, const float* q_scale, const uint8_t* K, const float* k_scale,
                            const upipe_bf16* V, int n_q, int n_kv, int S, int d_head, const int32_t* kv_of_q,
                            upipe_bf16* O, float* lse, void* stream);

/*
 * The layer forward (in-order schedule) with the stages whose heads are
 * flagged in fp8_heads (HOST array of H bytes, nonzero = FP8; every head of a
 * stage must carry the same flag, else UPIPE_EINVAL) exchanging Q and K as
 * E4M3 codes with their scales and attending with FP8 scores; V, O, Y and the
 * other stages are as in upipe_attn_fwd, with the same workspace
 * (upipe_fwd_workspace_bytes with the in-order schedule): an FP8 stage's
 * buffers take (U + n_kv) S d_head bytes of codes plus 2 n_kv S d_head of V
 * where the bf16 stage takes 2 (U + 2 n_kv) S d_head.  FP8 stages need
 * d_head = 128 (UPIPE_EUNSUPPORTED otherwise).  O_saved and lse feed
 * upipe_attn_bwd_fp8 (the exact backward of this forward) or upipe_attn_bwd
 * (which recomputes the scores in bf16: the gradients of the bf16 layer at the
 * FP8 forward's softmax statistics).
 */
int upipe_attn_fwd_fp8(const upipe_bf16* X, const upipe_bf16* W_qkv, const upipe_bf16* W_o, int S, int d_model,
                       int H, int G, int d_head, int U, int C, const uint8_t* fp8_heads, upipe_bf16* Y,
                       upipe_bf16* O_saved, float* lse, void* ws, size_t ws_bytes, void* stream, upipe_stats* stats);

/*
 * The backward of upipe_attention_fwd_fp8 (the pages give no backward; this
 * is the exact gradient of the FP8-scored attention in its dequantized
 * operands, the rounding to E4M3 passed through as the identity): the scores
 * are recomputed from the same codes and scales the forward used, dV = P^T dO,
 * dS = P * (dO V^T - rowsum(dO * O)), dQ = dS K~ / sqrt(d), dK = dS^T Q~ /
 * sqrt(d), with K~ = codes x block scale and Q~ = codes x row scale (Q~ is
 * rounded to bf16 on the way to the tensor cores).  Q, q_scale, K, k_scale as
 * for upipe_attention_fwd_fp8; V, O, dO, lse, outputs, workspace and errors as
 * for upipe_attention_bwd.  d_head 128 only.
 */
int upipe_attention_bwd_fp8(const uint8_t* Q, const float* q_scale, const uint8_t* K, const float* k_scale,
                            const upipe_bf16* V, const upipe_bf16* O, const upipe_bf16* dO, const float* lse, int n_q,
                            int n_kv, int S, int d_head, const int32_t* kv_of_q, float* dQ, float* dK, float* dV,
                            void* ws, size_t ws_bytes, void* stream);

/*
 * The layer backward (in-order schedule) of upipe_attn_fwd_fp8: the stages
 * whose heads are flagged in fp8_heads (HOST, H bytes, the same flags as the
 * forward) recompute their projection, exchange Q and K as E4M3 codes with
 * their scales (the operands the forward attended with) and run the FP8
 * attention backward above; other stages are as in upipe_attn_bwd.
 * Gradients in X and the weights follow through the dequantized Q and K.
 * Workspace: upipe_bwd_workspace_bytes_fp8() bytes -- when every stage is
 * FP8, the head-layout stage buffers hold (U + n_kv) S d_head bytes of codes,
 * 2 n_kv S d_head of V and the scales instead of 2 (U + 2 n_kv) S d_head, and
 * the arena (stats->arena_peak_bytes) is that much smaller; otherwise it is
 * upipe_bwd_workspace_bytes() of the in-order schedule.  FP8 stages need
 * d_head = 128 (UPIPE_EUNSUPPORTED otherwise); a stage whose heads carry
 * different flags is UPIPE_EINVAL.
 */
size_t upipe_bwd_workspace_bytes_fp8(int S, int d_model, int H, int G, int d_head, int U, int C,
                                     const uint8_t* fp8_heads);
int upipe_attn_bwd_fp8(const upipe_bf16* X, const upipe_bf16* W_qkv, const upipe_bf16* W_o, int S, int d_model,
                       int H, int G, int d_head, int U, int C, const uint8_t* fp8_heads, const upipe_bf16* O_saved,
                       const float* lse, const upipe_bf16* dY, upipe_bf16* dX, float* dW_qkv, float* dW_o, void* ws,
                       size_t ws_bytes, void* stream, upipe_stats* stats);

/*
 * Its backward pass.  dO: device bf16 [n_q][S][d_head]; O, lse from the forward.
 *   dQ  : device fp32 [n_q][S][d_head], output.
 *   dK, dV : device fp32 [n_kv][S][d_head], output (summed over the query
 *            slots that share each KV slot).
 *   ws  : device workspace of 8*n_q*S bytes.
 */
int upipe_attention_bwd(const upipe_bf16* Q, const upipe_bf16* K, const upipe_bf16* V, const upipe_bf16* O,
                        const upipe_bf16* dO, const float* lse, int n_q, int n_kv, int S, int d_head,
                        const int32_t* kv_of_q, float* dQ, float* dK, float* dV, void* ws, size_t ws_bytes,
                        void* stream);

/*
 * upipe_attention_bwd for callers that cannot allocate device memory.  The
 * pages have no counterpart: this is a deployment convenience, not part of the
 * method.  Some callers own no allocator on their call path (an engine that
 * reserves all device memory up front, a plugin inside another framework's
 * operator that forbids allocations, code that must not call cudaMalloc
 * because it synchronises the device), so this variant needs no `ws`: its
 * 8*n_q*S bytes of scratch come from a fixed 8 MiB array compiled into the
 * library, present on every GPU that loads it until the process exits.
 *   Arguments, layouts and results: as upipe_attention_bwd, without ws.
 *   Limit: 8*n_q*S <= 8 MiB (n_q*S <= 1,048,576), else UPIPE_ENOSPC before any launch.
 *   The first call on each device looks up the array's device address (with
 *   that device current) and caches it; make that first call before any stream
 *   capture begins.  All calls on a device share the array, which keeps the
 *   last call's contents: calls whose work overlaps on the GPU race; calls
 *   ordered on one stream do not.  Calls no cudaMalloc, cudaFree or allocating
 *   library routine.
 */
int upipe_attention_bwd_noalloc(const upipe_bf16* Q, const upipe_bf16* K, const upipe_bf16* V, const upipe_bf16* O,
                                const upipe_bf16* dO, const float* lse, int n_q, int n_kv, int S, int d_head,
                                const int32_t* kv_of_q, float* dQ, float* dK, float* dV, void* stream);

/*
 * The dense contraction behind the projections (Method steps (1) and the
 * output projection): D[M,N] = A[M,K] B[K,N], bf16 in, fp32 accumulate.
 *   A : device bf16, stored [M][K] (a_trans == 0) or [K][M] (a_trans == 1), row stride lda.
 *   B : device bf16, stored [K][N] (b_trans == 0) or [N][K] (b_trans == 1), row stride ldb.
 *   out_mode 0: D bf16;  1: D fp32;  2: D fp32 += A B;  3: D fp32 += A B with K
 *   split across CTAs and the partial sums added by fp32 atomics (for few output
 *   tiles and a long K; the summation order varies between runs).  ldd: row stride of D.
 * M % 64 == 0, N % 64 == 0, K % 64 == 0.
 */
int upipe_gemm_bf16(const upipe_bf16* A, const upipe_bf16* B, void* D, int M, int N, int K, int a_trans, int b_trans,
                    long long lda, long long ldb, long long ldd, int out_mode, void* stream);

/*
 * Self-test of the failure detection (no counterpart on the pages): every
 * wait of the library's kernels on an mbarrier is bounded; when one runs out
 * the kernel records a timeout in the device status word and exits, and
 * upipe_sync_status() returns UPIPE_ETIMEOUT.  This call launches one CTA
 * that waits, with a limit of limit_cycles SM clocks (1000 .. 1e9), on an
 * mbarrier nothing arrives at -- with the per-thread form of the wait
 * (warp_form == 0) or the warp-collective form (1) -- so that path runs for
 * real: nothing else is in flight in that CTA, and it returns within the
 * limit.  The next upipe_sync_status() reports UPIPE_ETIMEOUT and clears the
 * word.  UPIPE_EUNSUPPORTED when the library was built without it
 * (UPIPE_SELFTEST=0).
 */
int upipe_watchdog_selftest(long long limit_cycles, int warp_form, void* stream);

/* Reads (and clears) the device status word that bounded waits write; the
 * call synchronises `stream`.  UPIPE_OK or UPIPE_ETIMEOUT. */
int upipe_sync_status(void* stream);

/* Static description of a status code. */
const char* upipe_status_str(int status);

/* Library version (major*10000 + minor*100 + patch). */
int upipe_version(void);

/*
 * Optional kernel timing, off by default.  When enabled, every kernel the
 * library enqueues is bracketed by two CUDA events on the caller's stream;
 * upipe_profile_read() waits for them and returns, per kernel kind, the summed
 * milliseconds and the launch count since the last read (or enable), then
 * clears.  Output arrays: HOST memory of UPIPE_KERNEL_KINDS entries.  The
 * events add a few microseconds per launch; leave timing off in production.
 */
int upipe_profile_enable(int on);
int upipe_profile_read(double* ms_by_kind, int* count_by_kind);

/*
 * Optional CUDA-graph replay of whole layer calls, off by default (the
 * short-sequence overhead named in the "Untied Ulysses" summary page's
 * weaknesses section: a layer call issues several dozen small launches, whose
 * host-side gaps are a visible share of a short step).  When enabled, the first
 * upipe_attn_fwd / upipe_attn_bwd call with a given argument list (every
 * pointer, size and the device) captures its launch sequence on a private
 * stream into a graph and launches that graph on the caller's stream; later
 * calls with the same argument list replay it.  Replays read the CURRENT
 * contents of the same buffers, so the caller keeps the buffers alive and
 * unmoved while graphs are on; calls with other pointers capture a new graph
 * (up to 32 are kept; further argument lists run uncached).  Results are
 * bit-identical to direct calls.  Calls run directly, without a graph, while
 * upipe_profile_enable is on, when the caller's stream is itself being
 * captured, and the forward never uses its prefetching schedule under a graph
 * (a prefetch-sized workspace is accepted and runs the single-stream plan).
 * The stats a replay reports are those of the captured call.
 * upipe_graphs_enable(0) waits for the device and destroys every cached graph.
 * Errors: UPIPE_ECUDA when capture, instantiation or launch fails.
 */
int upipe_graphs_enable(int on);

#ifdef __cplusplus
}
#endif

#endif /* UPIPE_H */
