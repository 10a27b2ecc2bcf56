// Causal GQA attention backward for the heads one stage holds.
//
// The pages describe only the forward stage; the backward pass here is the
// analytic gradient of the same attention ("Untied Ulysses" summary, Method
// steps (3)), recomputing P from the saved log-sum-exp:
//   P  = exp(Q K^T / sqrt(d) - lse)          (causal)
//   dV = sum over query heads sharing the KV head of P^T dO
//   dS = P * (dO V^T - rowsum(dO * O))
//   dQ = dS K / sqrt(d),  dK = sum over those query heads of dS^T Q / sqrt(d)
//
// FP8 heads (D = 128): Q and K arrive as E4M3 codes with fp32 scales (Q per
// row, K per 128-key block), the operands the forward's scores were formed
// from.  The codes land in the upper half of their bf16 tiles and are widened
// in place on the integer and FMA pipes (the special-function pipe is the
// softmax's): K's codes once, exactly, by warps 2 and 3 (its block scale is a
// constant of the CTA, folded into the score's exponent factor and into dQ);
// each item's Q codes times their row scale, rounded to bf16, by the first-
// half softmax warps in their idle time after the previous item's dS -- so the
// MMAs and the softmax are the bf16 ones.  The gradients in Q and K are those of the dequantized
// operands (the rounding to E4M3 passed through as the identity).
//
// One CTA per (KV slot, 128-row KV block), ordered in groups of two KV slots
// (block 0, the longest, first), so the CTAs running at one time keep two
// slots' query-side data in L2.  A CTA walks every query slot mapped to its
// KV slot and every query block at or after its KV block, so the GQA
// reduction of dK/dV happens in TMEM with no atomics.  Per step i:
//   S^T = K Q^T, dP^T = V dO^T  (tensor cores -> TMEM)
//   warps 4..11, two per TMEM lane quarter, each thread owning half of one
//     KV row (64 query columns): P^T as bf16 back into S^T's TMEM columns,
//     then dS^T = P^T * (dP^T - D) (dP^T - D in fp32, the product in packed
//     bf16) into the other half of those columns and into shared memory
//   dV += P^T dO and dK += dS^T Q (A operands read from TMEM), dQ = dS K
//     (both operands in shared memory; dQ reuses dP's TMEM columns)
//   warps 12..15, one query row per thread, move dQ_i out of TMEM and send
//     it to the global fp32 accumulator with TMA reduce-adds, staged in the
//     Q/dO buffer of step i: its dO tile is free once dV_i has run (before
//     dQ_i), its Q tile once dK_i has; the producer refills that buffer
//     after the engine has read the staged dQ, so the next dS never waits
//     for the reduce-adds.
// MMA issue order dV_i, dQ_i, dK_i, S_{i+1}, dP_{i+1}: dQ_i is drained while
// dK_i and S_{i+1} run, and dP_{i+1} waits only for dQ_i to have left TMEM.
// The tensor pipe executes one CTA's MMAs in issue order, so S_{i+1}
// overwrites P^T_i and dS^T_i only after dV_i and dK_i have read them.

#include <algorithm>
#include <cmath>
#include <type_traits>

#include "ptx.cuh"
#include "upipe_internal.h"

namespace upipe {
namespace {

constexpr int BQ = 128;
constexpr int BKV = 128;
constexpr int CH = 128 * 128;  // a 64-column chunk of a 128-row bf16 tile

struct BwdArgs {
  int S, n_qslots, n_kvslots, q_blocks;
  int kv_ld, kv_blocks, q_off_blocks;  // key positions: see AttnBwdDesc
  int q_split;  // CTAs per KV block, each a contiguous share of its items (dK, dV added atomically)
  float scale_log2, scale;
  int accumulate_kv;
  int grp_slots;  // KV slots per group of the CTA order (divides n_kvslots)
  uint16_t kv_slot[kMaxSlots];
  const float* lse2;
  const float* Dsum;
  float* dQacc;
  float* dK;
  float* dV;
  const float* q_scale;  // FP8 heads: per query row
  const float* k_scale;  // FP8 heads: per 128-key block, kv_ld / 128 per KV slot
  int* status;
};

template <int D>
struct BwdCfg {
  static constexpr int TILE = 128 * D * 2;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = TILE;
  static constexpr int Q_OFF = 2 * TILE;    // 2 stages
  static constexpr int DO_OFF = 4 * TILE;   // 2 stages
  static constexpr int DS_TILE_OFF = 6 * TILE;  // dS^T, 128 x 128 bf16
  static constexpr int LSE_OFF = DS_TILE_OFF + BKV * BQ * 2;  // 2 stages x 128 fp32
  static constexpr int DS_OFF = LSE_OFF + 2 * BQ * 4;     // 2 stages x 128 fp32
  static constexpr int BAR_OFF = DS_OFF + 2 * BQ * 4;
  static constexpr int SMEM = BAR_OFF + 256;
  // TMEM: S^T [0,128) (then P^T as bf16 pairs in [0,32) and [64,96), dS^T
  //       in [32,64) and [96,128))
  //       dP^T / dQ [128,256)  dV [256,256+D)  dK [256+D,256+2D)
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t T_S = 0, T_DP = 128, T_DV = 256, T_DK = 256 + D;
};

// The (query slot, query block) pairs a CTA visits, in order: the query
// blocks at or after its KV block (query block b sits at KV block
// b + q_off_blocks).
template <bool GEN>
struct ItemCursor {
  int qs = -1, qb = 0, qb_first = 0, q_blocks = 0;
  bool primed = false;
  __device__ bool next(const BwdArgs& a, int kvs) {
    if (GEN && primed) { primed = false; return true; }
    if (qs >= 0 && ++qb < q_blocks) return true;
    for (++qs; qs < a.n_qslots; ++qs)
      if (a.kv_slot[qs] == kvs) { qb = qb_first; return true; }
    return false;
  }
  // position on item k (0-based) of this KV slot; next() then returns it first
  __device__ void seek(const BwdArgs& a, int kvs, int k) {
    const int per_slot = q_blocks - qb_first;
    if (!GEN || k <= 0 || per_slot <= 0) return;
    int skip = k / per_slot;
    for (qs = 0; qs < a.n_qslots; ++qs)
      if (a.kv_slot[qs] == kvs && skip-- == 0) break;
    qb = qb_first + k % per_slot;
    primed = true;
  }
};

// E4M3 codes to bf16 in place.  Row r of a 128 x 128 code tile (128-byte
// swizzled rows, at offset CH of its bf16 tile) becomes row r of the tile's
// two 64-column bf16 chunks, each value code x scale rounded to bf16 (exact
// for scale 1).  The row's codes are read before any of its outputs are
// written, and only row r's bytes are written, so rows convert independently.
__device__ __forceinline__ void e4m3_row_to_bf16(uint32_t tile, int r, float scale) {
  const uint32_t sw = static_cast<uint32_t>(r & 7);
  uint4 c[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) c[u] = ld_shared_v4(tile + CH + r * 128 + ((u ^ sw) << 4));
#pragma unroll
  for (int u = 0; u < 8; ++u) {  // codes of columns 16u .. 16u + 15
    const uint32_t wds[4] = {c[u].x, c[u].y, c[u].z, c[u].w};
    uint32_t o[8];
    const uint64_t sc = f2(scale, scale);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint64_t a = mul2(e4m3x2_to_f2(wds[k] & 0xFFFFu), sc), b = mul2(e4m3x2_to_f2(wds[k] >> 16), sc);
      o[2 * k] = pack_bf16(f2_lo(a), f2_hi(a));
      o[2 * k + 1] = pack_bf16(f2_lo(b), f2_hi(b));
    }
    const uint32_t row = tile + (u >> 2) * CH + r * 128;
    st_shared_v4(row + ((static_cast<uint32_t>((2 * u) & 7) ^ sw) << 4), o[0], o[1], o[2], o[3]);
    st_shared_v4(row + ((static_cast<uint32_t>((2 * u + 1) & 7) ^ sw) << 4), o[4], o[5], o[6], o[7]);
  }
}

// GEN: key offsets, key ranges and split KV blocks (chunk pairs); without it
// the launch is the plain causal case and those paths compile away.  F8: Q
// and K as E4M3 codes (plain launch, D = 128).
template <int D, bool GEN, bool F8>
__global__ void __launch_bounds__(512, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ BwdArgs a) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* kv_full = bars + 0;
  uint64_t* qdo_full = bars + 1;   // [2]
  uint64_t* qdo_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;
  uint64_t* dp_full = bars + 6;
  uint64_t* p_ready = bars + 7;
  uint64_t* dq_staged = bars + 8;  // [2] per Q/dO stage: its item's dQ has been read out of it
  uint64_t* ds_ready = bars + 10;
  uint64_t* ds_consumed = bars + 11;  // the dS tile free again (FP8: and the dQ chunks staged in it read)
  uint64_t* dq_full = bars + 12;
  uint64_t* dq_drained = bars + 13;
  uint64_t* kv_done = bars + 14;
  uint64_t* q_ready = bars + 15;   // [2] FP8: the stage's Q codes widened (first-half softmax warps)
  uint64_t* k_ready = bars + 17;   // FP8: K's codes widened
  uint64_t* do_full = bars + 18;   // [2] FP8: a stage's dO tile loaded (qdo_full: its Q tile, lse and D)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 20);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* s_lse = reinterpret_cast<float*>(smem + C::LSE_OFF);
  float* s_D = reinterpret_cast<float*>(smem + C::DS_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Watch w{abort_flag, a.status};
  const bool aligned = (smem_u32(smem) & 1023u) == 0;

  // CTA order: KV slots in groups of grp_slots, and within a group block 0
  // (most work) first, so the CTAs running at one time share few slots'
  // query-side data
  const int grp_slots = a.grp_slots;
  const int q_split = GEN ? a.q_split : 1;
  const int q_off_blocks = GEN ? a.q_off_blocks : 0;
  const int kv_blocks = GEN ? a.kv_blocks : a.q_blocks;
  const int kv_ld = GEN ? a.kv_ld : a.S;
  // (the q_split CTAs of one KV block are adjacent in launch order)
  const int part = GEN ? static_cast<int>(blockIdx.x) % q_split : 0;
  const int cta = GEN ? static_cast<int>(blockIdx.x) / q_split : static_cast<int>(blockIdx.x);
  const int per_grp = grp_slots * kv_blocks;
  const int grp = cta / per_grp, rem = cta % per_grp;
  const int kvb = rem / grp_slots;
  const int kvs = grp * grp_slots + rem % grp_slots;
  int n_q = 0;
  for (int i = 0; i < a.n_qslots; ++i) n_q += (a.kv_slot[i] == kvs);
  const int qb_first = GEN ? max(0, kvb - q_off_blocks) : kvb;
  const int n_all = n_q * max(0, a.q_blocks - qb_first);
  const int item0 = GEN ? static_cast<int>(static_cast<long long>(n_all) * part / q_split) : 0;
  const int n_items = GEN ? static_cast<int>(static_cast<long long>(n_all) * (part + 1) / q_split) - item0 : n_all;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&qdo_full[s], 1);
      mbar_init(&qdo_empty[s], 1);
      mbar_init(&do_full[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_ready, 256);
    mbar_init(ds_ready, 256);
    mbar_init(ds_consumed, F8 ? 4 : 1);  // FP8: lane 0 of each dQ warp
    mbar_init(dq_full, 1);
    mbar_init(dq_drained, 128);
    mbar_init(&dq_staged[0], 4);  // lane 0 of each dQ warp
    mbar_init(&dq_staged[1], 4);
    mbar_init(&q_ready[0], 128);  // the four first-half softmax warps
    mbar_init(&q_ready[1], 128);
    mbar_init(k_ready, 64);       // warps 2 and 3
    mbar_init(kv_done, 1);
    *abort_flag = aligned ? 0 : 1;
    if (!aligned && a.status) atomicCAS(a.status, 0, kDevBadSmem);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (aligned && n_items > 0) {
    if (warp == 0 && lane == 0) {
      // ---------------- TMA producer ----------------
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      tma_prefetch_map(&tmdO);
      const int kv_row = kvs * kv_ld + kvb * BKV;
      mbar_arrive_expect_tx(kv_full, (F8 ? CH : C::TILE) + C::TILE);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        if (!F8) tma_load_2d(smem + C::K_OFF + c * CH, &tmK, kv_full, c * 64, kv_row);
        tma_load_2d(smem + C::V_OFF + c * CH, &tmV, kv_full, c * 64, kv_row);
      }
      if (F8) tma_load_2d(smem + C::K_OFF + CH, &tmK, kv_full, 0, kv_row);  // codes: one 128 x 128 box
      ItemCursor<GEN> cur;
      cur.qb_first = qb_first;
      cur.q_blocks = a.q_blocks;
      cur.seek(a, kvs, item0);
      for (int i = 0; i < n_items && cur.next(a, kvs); ++i) {
        const int st = i & 1;
        if (!mbar_wait(&qdo_empty[st], ((i >> 1) & 1) ^ 1, w, 40)) break;
        const long long q_row = static_cast<long long>(cur.qs) * a.S + cur.qb * BQ;
        if constexpr (F8) {
          // Q's codes, lse and D once dK_{i-2} has read the stage's Q tile;
          // dO once the half of dQ_{i-2} staged in its dO tile has left it
          mbar_arrive_expect_tx(&qdo_full[st], CH + 2 * BQ * 4);
          tma_load_2d(smem + C::Q_OFF + st * C::TILE + CH, &tmQ, &qdo_full[st], 0, (int)q_row);
          bulk_load(s_lse + st * BQ, a.lse2 + q_row, BQ * 4, &qdo_full[st]);
          bulk_load(s_D + st * BQ, a.Dsum + q_row, BQ * 4, &qdo_full[st]);
          if (!mbar_wait(&dq_staged[st], ((i >> 1) & 1) ^ 1, w, 39)) break;
          mbar_arrive_expect_tx(&do_full[st], C::TILE);
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_2d(smem + C::DO_OFF + st * C::TILE + c * CH, &tmdO, &do_full[st], c * 64, (int)q_row);
        } else {
          // the stage's previous item staged its dQ here
          if (!mbar_wait(&dq_staged[st], ((i >> 1) & 1) ^ 1, w, 39)) break;
          mbar_arrive_expect_tx(&qdo_full[st], 2 * C::TILE + 2 * BQ * 4);
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            tma_load_2d(smem + C::Q_OFF + st * C::TILE + c * CH, &tmQ, &qdo_full[st], c * 64, (int)q_row);
            tma_load_2d(smem + C::DO_OFF + st * C::TILE + c * CH, &tmdO, &qdo_full[st], c * 64, (int)q_row);
          }
          bulk_load(s_lse + st * BQ, a.lse2 + q_row, BQ * 4, &qdo_full[st]);
          bulk_load(s_D + st * BQ, a.Dsum + q_row, BQ * 4, &qdo_full[st]);
        }
      }
    } else if (warp == 1 && lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t ID_S = idesc_bf16(BKV, BQ, false, false);  // S^T, dP^T
      constexpr uint32_t ID_KV = idesc_bf16(BKV, D, false, true);   // dV, dK
      constexpr uint32_t ID_Q = idesc_bf16(BQ, D, true, true);      // dQ
      const uint32_t sK = smem_u32(smem + C::K_OFF);
      const uint32_t sV = smem_u32(smem + C::V_OFF);
      const uint32_t sDS = smem_u32(smem + C::DS_TILE_OFF);
      auto sQ = [&](int st) { return smem_u32(smem + C::Q_OFF + st * C::TILE); };
      auto sdO = [&](int st) { return smem_u32(smem + C::DO_OFF + st * C::TILE); };
      // operand descriptors are built once per tile and advanced by constants
      auto qk_mma = [&](uint32_t d_tmem, uint32_t sA, uint32_t sB) {
        const uint64_t a0 = sdesc_kmajor(sA), b0 = sdesc_kmajor(sB);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * CH + (k & 3) * 32;
          mma_ss(d_tmem, sdesc_advance(a0, off), sdesc_advance(b0, off), ID_S, k > 0);
        }
      };
      // (FP8: the converters' barriers follow the loads' completion)
      bool ok = F8 ? (mbar_wait(k_ready, 0, w, 41) && mbar_wait(&q_ready[0], 0, w, 42))
                   : (mbar_wait(kv_full, 0, w, 41) && mbar_wait(&qdo_full[0], 0, w, 42));
      if (ok) {
        tc_fence_after();
        qk_mma(tmem + C::T_S, sK, sQ(0));
        mma_commit(s_full);
        if (F8) ok = mbar_wait(&do_full[0], 0, w, 59);
        if (ok) {
          if (F8) tc_fence_after();
          qk_mma(tmem + C::T_DP, sV, sdO(0));
          mma_commit(dp_full);
        }
      }
      for (int i = 0; ok && i < n_items; ++i) {
        const int st = i & 1;
        // dV += P^T dO, P^T read from TMEM (16 bf16 of K per 8 columns): query
        // columns [0,64) at S^T columns [0,32), [64,128) at [64,96)
        if (!mbar_wait(p_ready, i & 1, w, 43)) break;
        tc_fence_after();
        {
          const uint64_t b0 = sdesc_mnmajor(sdO(st), CH);
#pragma unroll
          for (int k = 0; k < BQ / 16; ++k)
            mma_ts(tmem + C::T_DV, tmem + C::T_S + (k >> 2) * 64 + (k & 3) * 8, sdesc_advance(b0, k * 2048), ID_KV,
                   (i | k) != 0);
        }
        // dQ = dS K (into dP's columns, read already), then dK += dS^T Q with
        // dS^T read from TMEM: the softmax warps start draining dQ while dK runs
        if (!mbar_wait(ds_ready, i & 1, w, 45)) break;
        tc_fence_after();
        {
          const uint64_t a1 = sdesc_mnmajor(sDS, CH), b1 = sdesc_mnmajor(sK, CH);
#pragma unroll
          for (int k = 0; k < BKV / 16; ++k)
            mma_ss(tmem + C::T_DP, sdesc_advance(a1, k * 2048), sdesc_advance(b1, k * 2048), ID_Q, k > 0);
          mma_commit(dq_full);
          if (!F8) mma_commit(ds_consumed);
          const uint64_t b0 = sdesc_mnmajor(sQ(st), CH);
#pragma unroll
          for (int k = 0; k < BQ / 16; ++k)
            mma_ts(tmem + C::T_DK, tmem + C::T_S + 32 + (k >> 2) * 64 + (k & 3) * 8, sdesc_advance(b0, k * 2048),
                   ID_KV, (i | k) != 0);
        }
        mma_commit(&qdo_empty[st]);
        // next S^T: issued after dV_i and dK_i, so it overwrites P^T_i and dS^T_i
        // only once they have been read
        if (i + 1 < n_items) {
          if (!mbar_wait(F8 ? &q_ready[st ^ 1] : &qdo_full[st ^ 1], ((i + 1) >> 1) & 1, w, 44)) break;
          tc_fence_after();
          qk_mma(tmem + C::T_S, sK, sQ(st ^ 1));
          mma_commit(s_full);
        }
        // next dP^T once dQ has been drained out of its columns
        if (i + 1 < n_items) {
          if (!mbar_wait(dq_drained, i & 1, w, 46)) break;
          if (F8 && !mbar_wait(&do_full[st ^ 1], ((i + 1) >> 1) & 1, w, 60)) break;
          tc_fence_after();
          qk_mma(tmem + C::T_DP, sV, sdO(st ^ 1));
          mma_commit(dp_full);
        }
      }
      if (ok) mma_commit(kv_done);
    } else if (warp >= 4 && warp < 12) {
      // ---------------- softmax and dS: half a row per thread ----------------
      const int q4 = warp & 3;
      const int half = (warp - 4) >> 2;  // 0: columns [0,64), 1: [64,128)
      const int row = q4 * 32 + lane;    // TMEM lane = KV row (S^T, dP^T) or query row (dQ)
      const int kv_idx = kvb * BKV + row;
      const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
      const uint32_t sDS = smem_u32(smem + C::DS_TILE_OFF);
      // FP8: K's codes are unscaled; its block scale joins the exponent factor
      const float sl2 = F8 ? a.scale_log2 * a.k_scale[static_cast<long long>(kvs) * (kv_ld / BKV) + kvb] : a.scale_log2;
      const uint64_t sl2x2 = f2(sl2, sl2);
      ItemCursor<GEN> cur;
      cur.qb_first = qb_first;
      cur.q_blocks = a.q_blocks;
      cur.seek(a, kvs, item0);
      bool ok = true;
      // FP8: the first-half warps widen each item's Q codes (a row per
      // thread), item 0 here and item i+1 after dS_i, one item ahead of its S^T
      ItemCursor<GEN> ahead = cur;
      auto widen_q = [&](int j) -> bool {
        if (!ahead.next(a, kvs)) return true;
        if (!mbar_wait_warp(&qdo_full[j & 1], (j >> 1) & 1, w, 56)) return false;
        const float qs = a.q_scale[static_cast<long long>(ahead.qs) * a.S + ahead.qb * BQ + row];
        e4m3_row_to_bf16(smem_u32(smem + C::Q_OFF + (j & 1) * C::TILE), row, qs);
        fence_proxy_async_smem();
        mbar_arrive(&q_ready[j & 1]);
        return true;
      };
      if (F8 && half == 0 && n_items > 0) ok = widen_q(0);
      int i = 0;
      for (; ok && i < n_items && cur.next(a, kvs); ++i) {
        const int st = i & 1;
        const bool diag = (cur.qb + q_off_blocks == kvb);
        if (!mbar_wait_warp(s_full, i & 1, w, 47)) { ok = false; break; }
        if (!mbar_wait_warp(&qdo_full[st], (i >> 1) & 1, w, 48)) { ok = false; break; }
        tc_fence_after();
        const float* lse = s_lse + st * BQ + half * 64;
        const float* Dv = s_D + st * BQ + half * 64;
        uint32_t pk[32];  // P^T of query columns [64*half, 64*half+64) as bf16 pairs
        {
          // this half row of S^T in one load (one wait)
          uint32_t v[64];
          tmem_ld64(tmem + lane_off + C::T_S + half * 64, v);
          // the causal mask only on the diagonal block, outside the unrolled
          // loop, so the off-diagonal loop is straight-line code
          auto p_loop = [&](auto masked) {
#pragma unroll
            for (int q0 = 0; q0 < 64; q0 += 4) {  // within this half
              const int e = q0;
              const float4 l4 = *reinterpret_cast<const float4*>(lse + q0);
              const uint64_t xa = fma2(f2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), sl2x2, f2(l4.x, l4.y));
              const uint64_t xb =
                  fma2(f2(__uint_as_float(v[e + 2]), __uint_as_float(v[e + 3])), sl2x2, f2(l4.z, l4.w));
              float p0 = ex2(f2_lo(xa)), p1 = ex2(f2_hi(xa)), p2 = ex2(f2_lo(xb)), p3 = ex2(f2_hi(xb));
              if (decltype(masked)::value) {
                if (half * 64 + q0 < row) p0 = 0.f;
                if (half * 64 + q0 + 1 < row) p1 = 0.f;
                if (half * 64 + q0 + 2 < row) p2 = 0.f;
                if (half * 64 + q0 + 3 < row) p3 = 0.f;
              }
              pk[q0 >> 1] = pack_bf16(p0, p1);
              pk[(q0 >> 1) + 1] = pack_bf16(p2, p3);
            }
          };
          if (diag)
            p_loop(std::true_type{});
          else
            p_loop(std::false_type{});
        }
        // P^T (bf16 pairs) into the first 32 columns of this half's own S^T
        // columns, which only this thread has read
        tmem_st32(tmem + lane_off + C::T_S + half * 64, pk);
        tc_fence_before();
        mbar_arrive(p_ready);
        // dS^T = P^T * (dP^T - D)
        if (!mbar_wait_warp(dp_full, i & 1, w, 50)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + C::T_DP + half * 64 + c * 32, v);
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            // dP^T - D in fp32, rounded to bf16, times the bf16 P^T it pairs with
            const int q0 = c * 32 + e;
            const float4 d4 = *reinterpret_cast<const float4*>(Dv + q0);
            const uint64_t ta = sub2(f2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), f2(d4.x, d4.y));
            const uint64_t tb = sub2(f2(__uint_as_float(v[e + 2]), __uint_as_float(v[e + 3])), f2(d4.z, d4.w));
            pk[q0 >> 1] = mul_bf16x2(pk[q0 >> 1], pack_bf16(f2_lo(ta), f2_hi(ta)));
            pk[(q0 >> 1) + 1] = mul_bf16x2(pk[(q0 >> 1) + 1], pack_bf16(f2_lo(tb), f2_hi(tb)));
          }
        }
        // the dS^T tile is free once the previous step's dQ MMA has read it
        if (i > 0 && !mbar_wait_warp(ds_consumed, (i - 1) & 1, w, 49)) {
          ok = false;
          break;
        }
        // dS^T as bf16 pairs into the other 32 of this half's S^T columns (the A
        // operand of dK), and into shared memory (the A operand of dQ)
        tmem_st32(tmem + lane_off + C::T_S + half * 64 + 32, pk);
#pragma unroll
        for (int piece = 0; piece < 8; ++piece)
          st_shared_v4(sDS + half * CH + row * 128 + ((piece ^ (row & 7)) << 4), pk[piece * 4], pk[piece * 4 + 1],
                       pk[piece * 4 + 2], pk[piece * 4 + 3]);
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(ds_ready);
        if (F8 && half == 0 && i + 1 < n_items && !widen_q(i + 1)) {
          ok = false;
          break;
        }
      }
      // dK, dV epilogue: this thread's half of the d columns of KV row `row`
      if (ok && mbar_wait_warp(kv_done, 0, w, 52)) {
        tc_fence_after();
        const long long base = (static_cast<long long>(kvs) * kv_ld + kv_idx) * D + half * (D / 2);
#pragma unroll 1
        for (int which = 0; which < 2; ++which) {
          float* dst = (which == 0 ? a.dV : a.dK) + base;
          const float mul = which == 0 ? 1.f : a.scale;
          const uint32_t col = (which == 0 ? C::T_DV : C::T_DK) + half * (D / 2);
#pragma unroll 1
          for (int c = 0; c < D / 64; ++c) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_off + col + c * 32, v);
            float4* o = reinterpret_cast<float4*>(dst + c * 32);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              float4 x = make_float4(__uint_as_float(v[4 * e]) * mul, __uint_as_float(v[4 * e + 1]) * mul,
                                     __uint_as_float(v[4 * e + 2]) * mul, __uint_as_float(v[4 * e + 3]) * mul);
              if (GEN && q_split > 1) {  // other CTAs add to the same rows
                red_add_v4(dst + c * 32 + 4 * e, x.x, x.y, x.z, x.w);
                continue;
              }
              if (a.accumulate_kv) {
                const float4 p = o[e];
                x.x += p.x; x.y += p.y; x.z += p.z; x.w += p.w;
              }
              o[e] = x;
            }
          }
        }
      }
    } else if (F8 && (warp == 2 || warp == 3)) {
      // ---------------- FP8: widen K's codes to bf16, once ----------------
      const int t = (warp - 2) * 32 + lane;
      if (mbar_wait_warp(kv_full, 0, w, 55)) {
        e4m3_row_to_bf16(smem_u32(smem + C::K_OFF), t, 1.f);
        e4m3_row_to_bf16(smem_u32(smem + C::K_OFF), t + 64, 1.f);
        fence_proxy_async_smem();
        mbar_arrive(k_ready);
      }
    } else if (warp >= 12) {
      // ---------------- dQ: one query row per thread ----------------
      // dQ_i leaves TMEM (freeing dP's columns for dP_{i+1}) and is added into
      // the global fp32 accumulator by the TMA engine, off the softmax warps'
      // path
      const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
      // dQ = dS K / sqrt(d); FP8: K's block scale as well (K's tile holds its codes)
      const float dq_mul = F8 ? a.scale * a.k_scale[static_cast<long long>(kvs) * (kv_ld / BKV) + kvb] : a.scale;
      ItemCursor<GEN> cur;
      cur.qb_first = qb_first;
      cur.q_blocks = a.q_blocks;
      cur.seek(a, kvs, item0);
      // row-major fp32 dQ through the TMA engine: each warp stages its 32
      // rows in 32-column chunks (32 x 32 fp32, 128-byte swizzle, 4 KB)
      // in its quarter of step i's Q/dO buffer -- the first D/64 chunks in
      // the dO tile (free: dV_i, its last reader, ran before dQ_i), the
      // rest in the Q tile once dK_i has completed -- and issues element-
      // wise reduce-adds; when the engine has read them, the buffer goes
      // back to the producer
      tma_prefetch_map(&tmDQ);
      constexpr int NCH = D / 32, HALF = NCH / 2;
      const uint32_t quarter = (warp & 3) * (C::TILE / 4);
      for (int i = 0; i < n_items && cur.next(a, kvs); ++i) {
        const int st = i & 1;
        if (!mbar_wait_warp(dq_full, i & 1, w, 53)) break;
        tc_fence_after();
        const int y0 = cur.qs * a.S + cur.qb * BQ + (warp & 3) * 32;
        const uint32_t s_stage = smem_u32(smem) + st * C::TILE + quarter;
        const uint32_t s_ds = smem_u32(smem + C::DS_TILE_OFF) + (warp & 3) * (BKV * BQ * 2 / 4);
        bool ok = true;
#pragma unroll 1
        for (int c = 0; ok && c < D / 64; ++c) {
          uint32_t v[64];
          tmem_ld64(tmem + lane_off + C::T_DP + c * 64, v);
          if (c == D / 64 - 1) {
            tc_fence_before();
            mbar_arrive(dq_drained);
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int chunk = 2 * c + h;
            if (!F8 && chunk == HALF && !mbar_wait_warp(&qdo_empty[st], (i >> 1) & 1, w, 54)) {
              ok = false;
              break;
            }
            // FP8: the second half in this warp's quarter of the dS tile,
            // which dQ_i (complete at dq_full) was the last to read, so the
            // Q tile goes back to the producer as soon as dK_i has read it
            const uint32_t buf = chunk < HALF ? s_stage + C::DO_OFF + chunk * 4096
                                 : F8 ? s_ds + (chunk - HALF) * 4096
                                      : s_stage + C::Q_OFF + (chunk - HALF) * 4096;
#pragma unroll
            for (int p = 0; p < 8; ++p)
              st_shared_v4(buf + lane * 128 + ((p ^ (lane & 7)) << 4),
                           __float_as_uint(__uint_as_float(v[h * 32 + 4 * p]) * dq_mul),
                           __float_as_uint(__uint_as_float(v[h * 32 + 4 * p + 1]) * dq_mul),
                           __float_as_uint(__uint_as_float(v[h * 32 + 4 * p + 2]) * dq_mul),
                           __float_as_uint(__uint_as_float(v[h * 32 + 4 * p + 3]) * dq_mul));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_reduce_add_2d(&tmDQ, buf, chunk * 32, y0);
              bulk_commit();
            }
          }
        }
        if (!ok) break;
        if (lane == 0) {
          if constexpr (F8) {  // chunk groups in issue order: the dO tile's first
            bulk_wait_read<NCH - HALF>();
            mbar_arrive(&dq_staged[st]);
            bulk_wait_read<0>();
            mbar_arrive(ds_consumed);
          } else {
            bulk_wait_read<0>();
            mbar_arrive(&dq_staged[st]);
          }
        }
        __syncwarp();
      }
      if (lane == 0) bulk_wait_all();
      __syncwarp();
    }
  } else if (aligned && n_items == 0 && !a.accumulate_kv && q_split == 1 && warp >= 4 && warp < 12) {
    // a KV slot no query head uses in this launch: its gradient is zero
    const int row = (warp & 3) * 32 + lane;
    const int half = (warp - 4) >> 2;
    const long long base = (static_cast<long long>(kvs) * kv_ld + kvb * BKV + row) * D + half * (D / 2);
    for (int c = 0; c < D / 2; c += 4) {
      *reinterpret_cast<float4*>(a.dK + base + c) = make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4*>(a.dV + base + c) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// D = rowsum(dO * O) per (slot, token), minus lse in log2 units (the bias of the
// exponent the backward recomputes P with), dQ accumulator zeroed.
__global__ void bwd_prep_kernel(const BwdPrepDesc p) {
  const int lanes_per_row = p.D / 8;            // 16-byte vectors per row
  const int rows_per_warp = 32 / lanes_per_row;
  const int lane = threadIdx.x & 31;
  const long long warp_g = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long total = static_cast<long long>(p.n_slots) * p.S;
  const long long r = warp_g * rows_per_warp + lane / lanes_per_row;
  const int v = lane % lanes_per_row;
  float acc = 0.f;
  int slot = 0, t = 0;
  if (r < total) {
    slot = static_cast<int>(r / p.S);
    t = static_cast<int>(r % p.S);
    const uint4 x = *reinterpret_cast<const uint4*>(p.dO + t * p.ld_do +
                                                    static_cast<long long>(p.do_unit[slot]) * p.D + v * 8);
    const uint4 y = *reinterpret_cast<const uint4*>(p.O + t * p.ld_o +
                                                    static_cast<long long>(p.o_unit[slot]) * p.D + v * 8);
    const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) acc += bf16_lo(xs[i]) * bf16_lo(ys[i]) + bf16_hi(xs[i]) * bf16_hi(ys[i]);
    float4* z = reinterpret_cast<float4*>(p.dQacc + r * p.D + v * 8);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int off = lanes_per_row / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (r < total && v == 0) {
    p.Dsum[r] = acc;
    p.lse2[r] = p.lse[static_cast<long long>(p.lse_row[slot]) * (p.lse_ld ? p.lse_ld : p.S) + t] * -1.4426950408889634f;
  }
}

template <int D, bool GEN, bool F8 = false>
cudaError_t run_bwd(const CUtensorMap* tm, const BwdArgs& args, cudaStream_t st) {
  auto kern = attn_bwd_kernel<D, GEN, F8>;
  // the kernel needs more than the default 48 KB of dynamic shared memory;
  // the limit is raised once per device
  if (const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), BwdCfg<D>::SMEM); e != cudaSuccess)
    return e;
  kern<<<args.n_kvslots * args.kv_blocks * args.q_split, 512, BwdCfg<D>::SMEM, st>>>(tm[0], tm[1], tm[2], tm[3], tm[4],
                                                                                      args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_prep(const BwdPrepDesc& p, cudaStream_t st) {
  if ((p.D != 64 && p.D != 128) || p.n_slots <= 0 || p.n_slots > kMaxSlots) return cudaErrorInvalidValue;
  const long long rows = static_cast<long long>(p.n_slots) * p.S;
  const int rows_per_warp = 32 / (p.D / 8);
  const long long warps = (rows + rows_per_warp - 1) / rows_per_warp;
  const long long blocks = (warps + 7) / 8;
  bwd_prep_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd(const AttnBwdDesc& d, int* status, cudaStream_t st) {
  const int kv_len = d.kv_len ? d.kv_len : d.S;
  const int kv_ld = d.kv_ld ? d.kv_ld : kv_len;
  if ((d.D != 64 && d.D != 128) || d.S % 128 || d.n_qslots <= 0 || d.n_qslots > kMaxSlots ||
      d.n_kvslots <= 0)
    return cudaErrorInvalidValue;
  if (kv_len <= 0 || kv_len % 128 || kv_ld < kv_len || d.q_off < 0 || d.q_off % 128) return cudaErrorInvalidValue;
  if (d.q_split < 1 || d.q_split > 16) return cudaErrorInvalidValue;
  for (int i = 0; i < d.n_qslots; ++i)
    if (d.kv_slot[i] >= d.n_kvslots) return cudaErrorInvalidValue;
  CUtensorMap tm[5];
  if (d.fp8 && (d.D != 128 || !d.q_scale || !d.k_scale)) return cudaErrorInvalidValue;
  if (d.fp8) {  // Q and K codes: one 128 x 128 byte box per tile
    if (!make_tmap_u8(&tm[0], d.Q, d.D, (uint64_t)d.n_qslots * d.S, d.D, 128, 128)) return cudaErrorInvalidValue;
    if (!make_tmap_u8(&tm[1], d.K, d.D, (uint64_t)d.n_kvslots * kv_ld, d.D, 128, 128)) return cudaErrorInvalidValue;
  } else {
    if (!make_tmap_bf16(&tm[0], d.Q, d.D, (uint64_t)d.n_qslots * d.S, d.D, 64, 128)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16(&tm[1], d.K, d.D, (uint64_t)d.n_kvslots * kv_ld, d.D, 64, 128)) return cudaErrorInvalidValue;
  }
  if (!make_tmap_bf16(&tm[2], d.V, d.D, (uint64_t)d.n_kvslots * kv_ld, d.D, 64, 128)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tm[3], d.dO, d.D, (uint64_t)d.n_qslots * d.S, d.D, 64, 128)) return cudaErrorInvalidValue;
  // the dQ accumulator as fp32 rows, for the TMA reduce-adds
  if (!make_tmap_f32(&tm[4], d.dQacc, d.D, (uint64_t)d.n_qslots * d.S, d.D, 32, 32)) return cudaErrorInvalidValue;
  BwdArgs a;
  a.S = d.S;
  a.kv_ld = kv_ld;
  a.kv_blocks = kv_len / BKV;
  a.q_off_blocks = d.q_off / BQ;
  a.q_split = d.q_split;
  a.n_qslots = d.n_qslots;
  a.n_kvslots = d.n_kvslots;
  a.q_blocks = d.S / BQ;
  a.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d.D)));
  a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d.D)));
  a.accumulate_kv = d.accumulate_kv;
  // two KV slots per group of the CTA order (one beyond 2^19 tokens), a
  // divisor of n_kvslots: the CTAs running at one time then sweep the query
  // blocks of two slots, whose Q, dO and fp32 dQ rows stay in L2 between the
  // CTAs' visits, so each is read from and written to DRAM about once per
  // launch (32K, 8 slots: 0.77 GB of DRAM traffic against 3.07 GB with eight
  // slots per group, in the same time)
  int g = std::max(1, std::min(2, (1 << 20) / d.S));
  g = std::min(g, d.n_kvslots);
  while (g > 1 && d.n_kvslots % g) --g;
  a.grp_slots = g;
  for (int i = 0; i < d.n_qslots; ++i) a.kv_slot[i] = d.kv_slot[i];
  a.lse2 = d.lse2;
  a.Dsum = d.Dsum;
  a.dQacc = d.dQacc;
  a.dK = d.dK;
  a.dV = d.dV;
  a.q_scale = d.q_scale;
  a.k_scale = d.k_scale;
  a.status = status;
  const bool gen = d.q_off != 0 || kv_len != d.S || kv_ld != d.S || d.q_split > 1;
  if (d.fp8) return gen ? cudaErrorInvalidValue : run_bwd<128, false, true>(tm, a, st);
  if (gen) return d.D == 128 ? run_bwd<128, true>(tm, a, st) : run_bwd<64, true>(tm, a, st);
  return d.D == 128 ? run_bwd<128, false>(tm, a, st) : run_bwd<64, false>(tm, a, st);
}

}  // namespace upipe
