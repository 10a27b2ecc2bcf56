// Causal GQA attention forward for the heads one stage holds ("Untied
// Ulysses" summary, Method steps (3): attention of the stage's U heads).
//
// O = softmax(Q K^T / sqrt(d) + causal mask) V, with the natural-log
// log-sum-exp of every row saved for the backward pass.  Query slots map to
// KV slots through a table, so grouped-query heads read their shared K/V.
//
// One CTA per (query slot, 256 query rows) = two 128-row query tiles A and B
// that take turns on the tensor cores; CTAs with the longest causal rows are
// scheduled first.  TMEM (512 columns): S_A, S_B (128 fp32 columns each) and
// O_A, O_B (d columns each).  Warp 0 streams 128-row K/V blocks by TMA into
// two-deep rings shared by both tiles, K one block ahead of V (K_j is last read
// by the scores of block j, V_j one step later by P V); warp 1 issues, per KV
// block j,
//   S_A(j) = Q_A K_j^T, S_B(j), then O_A += P_A(j) V_j, S_A(j+1), O_B += ...
// Warps 4..7 (tile A) and 8..11 (tile B) own one query row per thread: they
// read the row of S from TMEM with one load, keep a per-row reference maximum (rescaling the
// TMEM accumulator O only when the running maximum grows by more than 2^8,
// which is exact since the same reference enters numerator and denominator),
// and write P as bf16 pairs back into the first 64 columns of their S, where
// the P V MMA reads its A operand.  The tensor pipe runs one CTA's MMAs in
// issue order, so when S_T(j) is complete, O_T += P_T(j-1) V_{j-1} is complete
// too: O is stable while the softmax warps rescale it, and P_T(j-1) has been
// consumed before S_T(j) overwrites it.
#include <cmath>

#include "ptx.cuh"
#include "upipe_internal.h"

namespace upipe {
namespace {

constexpr int BQ = 128;        // query rows per tile (two tiles per CTA)
constexpr int BKV = 128;       // key rows per block
constexpr int CH = 128 * 128;  // one 64-column chunk of a 128-row bf16 tile (bytes)
constexpr float kRescaleLog2 = 8.0f;

struct FwdArgs {
  int S, n_qslots, q_blocks, q_pairs;
  int kv_ld, kv_blocks, q_off_blocks, lse_ld, mode;
  float scale_log2;
  uint16_t kv_slot[kMaxSlots];
  uint16_t lse_row[kMaxSlots];
  uint16_t* O;
  float* lse;
  float* o_acc;
  float* lse_acc;
  const float* q_scale;  // FP8 scores: per query row
  const float* k_scale;  // FP8 scores: per 128-key block, kv_ld / 128 per KV slot
  int* status;
};

// F8: Q and K tiles hold E4M3 codes (one 128-byte swizzled row per query or
// key at D = 128) and the scores come from kind::f8f6f4 MMAs; V, P and O stay
// bf16.
template <int D, bool F8 = false>
struct FwdCfg {
  static constexpr int TILE = BQ * D * 2;           // a bf16 tile (V)
  static constexpr int QK_TILE = F8 ? BQ * D : TILE;  // a Q or K tile
  static constexpr int QK_CHUNKS = QK_TILE / CH;      // 128-byte-wide column chunks
  static constexpr int QA_OFF = 0;
  static constexpr int QB_OFF = QK_TILE;
  static constexpr int K_OFF = 2 * QK_TILE;            // 2 stages
  static constexpr int V_OFF = 2 * QK_TILE + 2 * QK_TILE;  // 2 stages
  static constexpr int BAR_OFF = V_OFF + 2 * TILE;
  static constexpr int SMEM = BAR_OFF + 256;
  static constexpr uint32_t TMEM_COLS = 512;
  // TMEM columns: S of tile t at t*128, O of tile t at 256 + t*D
  static __device__ __forceinline__ uint32_t t_s(int tile) { return static_cast<uint32_t>(tile) * 128u; }
  static __device__ __forceinline__ uint32_t t_o(int tile) { return 256u + static_cast<uint32_t>(tile) * D; }
};

// GEN: key offsets and ranges, and the merging epilogues (chunk pairs);
// without it the launch is the plain causal case and those paths compile away.
template <int D, bool F8, bool GEN>
__global__ void __launch_bounds__(384, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ FwdArgs a) {
  using C = FwdCfg<D, F8>;
  static_assert(!F8 || D == 128, "FP8 scores need 128-byte Q and K rows");
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;    // [2]
  uint64_t* v_full = bars + 3;    // [2]
  uint64_t* k_empty = bars + 5;   // [2]
  uint64_t* s_full = bars + 7;    // [2] per tile
  uint64_t* p_ready = bars + 9;   // [2] per tile
  uint64_t* o_done = bars + 11;   // [2] per tile
  uint64_t* v_empty = bars + 13;  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 15);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Watch w{abort_flag, a.status};
  const bool aligned = (smem_u32(smem) & 1023u) == 0;

  // longest causal rows first: pair index t covers query blocks 2t and 2t+1;
  // more than 8 query slots go in groups of 8 (each group longest first), so
  // the CTAs running at one time share few slots' K/V
  const int grp_slots = (a.n_qslots > 8 && a.n_qslots % 8 == 0) ? 8 : a.n_qslots;
  const int per_grp = grp_slots * a.q_pairs;
  const int grp = static_cast<int>(blockIdx.x) / per_grp, rem = static_cast<int>(blockIdx.x) % per_grp;
  const int t = a.q_pairs - 1 - rem / grp_slots;
  const int slot = grp * grp_slots + rem % grp_slots;
  const int kvs = a.kv_slot[slot];
  const int qb0 = 2 * t, qb1 = 2 * t + 1;
  const bool has_b = qb1 < a.q_blocks;
  // query block b sits at KV block b + q_off_blocks: it sees the KV blocks up
  // to that one (the diagonal, masked) or all of them when it lies beyond
  const int q_off_blocks = GEN ? a.q_off_blocks : 0;
  const int kv_blocks = GEN ? a.kv_blocks : a.q_blocks;
  const int kv_ld = GEN ? a.kv_ld : a.S;
  const int n_kv0 = GEN ? min(kv_blocks, qb0 + q_off_blocks + 1) : qb0 + 1;
  const int n_kv1 = has_b ? (GEN ? min(kv_blocks, qb1 + q_off_blocks + 1) : qb1 + 1) : 0;
  const int n_blocks = has_b ? n_kv1 : n_kv0;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&p_ready[s], 128);
      mbar_init(&o_done[s], 1);
    }
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

  if (aligned) {
    if (warp == 0 && lane == 0) {
      // ---------------- TMA producer ----------------
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      mbar_arrive_expect_tx(q_full, (has_b ? 2 : 1) * C::QK_TILE);
      for (int tile = 0; tile < (has_b ? 2 : 1); ++tile)
#pragma unroll
        for (int c = 0; c < C::QK_CHUNKS; ++c)
          tma_load_2d(smem + (tile ? C::QB_OFF : C::QA_OFF) + c * CH, &tmQ, q_full, c * (F8 ? 128 : 64),
                      slot * a.S + (tile ? qb1 : qb0) * BQ);
      // K of block j is last read by the scores of block j, one step before V of
      // block j is last read by P V: K runs one block ahead of V
      for (int j = 0; j <= n_blocks; ++j) {
        if (j < n_blocks) {
          const int s = j & 1;
          if (!mbar_wait(&k_empty[s], ((j >> 1) & 1) ^ 1, w, 20)) break;
          mbar_arrive_expect_tx(&k_full[s], C::QK_TILE);
#pragma unroll
          for (int c = 0; c < C::QK_CHUNKS; ++c)
            tma_load_2d(smem + C::K_OFF + s * C::QK_TILE + c * CH, &tmK, &k_full[s], c * (F8 ? 128 : 64),
                        kvs * kv_ld + j * BKV);
        }
        if (j > 0) {
          const int jv = j - 1, s = jv & 1;
          if (!mbar_wait(&v_empty[s], ((jv >> 1) & 1) ^ 1, w, 19)) break;
          mbar_arrive_expect_tx(&v_full[s], C::TILE);
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_2d(smem + C::V_OFF + s * C::TILE + c * CH, &tmV, &v_full[s], c * 64, kvs * kv_ld + jv * BKV);
        }
      }
    } else if (warp == 1 && lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t ID_S = F8 ? idesc_e4m3(BQ, BKV) : idesc_bf16(BQ, BKV, false, false);
      constexpr uint32_t ID_O = idesc_bf16(BQ, D, false, true);
      const uint32_t sQ[2] = {smem_u32(smem + C::QA_OFF), smem_u32(smem + C::QB_OFF)};
      bool ok = mbar_wait(q_full, 0, w, 21);
      auto issue_s = [&](int tile, int j) -> bool {
        const int s = j & 1;
        if (!mbar_wait(&k_full[s], (j >> 1) & 1, w, 22)) return false;
        tc_fence_after();
        const uint64_t a0 = sdesc_kmajor(sQ[tile]), b0 = sdesc_kmajor(smem_u32(smem + C::K_OFF + s * C::QK_TILE));
        // 32 bytes of each row per MMA: K = 16 bf16 or 32 E4M3 values
#pragma unroll
        for (int k = 0; k < C::QK_TILE / BQ / 32; ++k) {
          const uint32_t off = (k >> 2) * CH + (k & 3) * 32;
          if constexpr (F8)
            mma_ss_f8(tmem + C::t_s(tile), sdesc_advance(a0, off), sdesc_advance(b0, off), ID_S, k > 0);
          else
            mma_ss(tmem + C::t_s(tile), sdesc_advance(a0, off), sdesc_advance(b0, off), ID_S, k > 0);
        }
        mma_commit(&s_full[tile]);
        return true;
      };
      auto issue_pv = [&](int tile, int j) -> bool {
        const int s = j & 1;
        if (!mbar_wait(&p_ready[tile], j & 1, w, 23)) return false;
        if (!mbar_wait(&v_full[s], (j >> 1) & 1, w, 24)) return false;
        tc_fence_after();
        const uint64_t b0 = sdesc_mnmajor(smem_u32(smem + C::V_OFF + s * C::TILE), CH);
#pragma unroll
        for (int k = 0; k < BKV / 16; ++k)
          mma_ts(tmem + C::t_o(tile), tmem + C::t_s(tile) + k * 8, sdesc_advance(b0, k * 2048), ID_O, (j | k) != 0);
        return true;
      };
      if (ok) ok = issue_s(0, 0);
      if (ok && has_b) ok = issue_s(1, 0);
      if (ok) mma_commit(&k_empty[0]);
      for (int j = 0; ok && j < n_blocks; ++j) {
        const int s = j & 1;
        if (j < n_kv0) {
          if (!issue_pv(0, j)) break;
          if (j + 1 < n_kv0) {
            if (!issue_s(0, j + 1)) break;
          } else {
            mma_commit(&o_done[0]);
          }
        }
        if (has_b) {
          if (!issue_pv(1, j)) break;
          if (j + 1 < n_kv1) {
            if (!issue_s(1, j + 1)) break;
          } else {
            mma_commit(&o_done[1]);
          }
        }
        mma_commit(&v_empty[s]);
        if (j + 1 < n_blocks) mma_commit(&k_empty[(j + 1) & 1]);
      }
    } else if (warp >= 4) {
      // ---------------- softmax: one query row of one tile per thread ----------------
      const int tile = (warp - 4) >> 2;
      if (tile == 0 || has_b) {
        const int q4 = warp & 3;
        const int row = q4 * 32 + lane;
        const int qb = tile ? qb1 : qb0;
        const int qi = qb * BQ + row;                     // row of the query slot
        const int qk = qi + q_off_blocks * BQ;            // its position among the keys
        const bool has_diag = !GEN || qb + q_off_blocks < kv_blocks;
        const int nkv = tile ? n_kv1 : n_kv0;
        const uint32_t t_s = tmem + (static_cast<uint32_t>(q4 * 32) << 16) + C::t_s(tile);
        const uint32_t t_o = tmem + (static_cast<uint32_t>(q4 * 32) << 16) + C::t_o(tile);
        // scores times sl2 are the exponents in log2 units; FP8 scores carry the
        // row's and the key block's scales as well
        const float sl2_row = F8 ? a.scale_log2 * a.q_scale[static_cast<long long>(slot) * a.S + qi] : a.scale_log2;
        const float* ksc = F8 ? a.k_scale + static_cast<long long>(kvs) * (kv_ld / BKV) : nullptr;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < nkv; ++j) {
          if (!mbar_wait_warp(&s_full[tile], j & 1, w, 25)) { ok = false; break; }
          tc_fence_after();
          const float sl2 = F8 ? sl2_row * ksc[j] : sl2_row;
          const bool diag = has_diag && (j == nkv - 1);
          const int lim = diag ? qk - j * BKV : BKV;  // keys at column > lim are in the future
          // the whole row of S in one TMEM load: its maximum, then P from registers
          uint32_t v[BKV];
          tmem_ld128(t_s, v);
          float mx = -INFINITY;
          if (diag) {
#pragma unroll
            for (int e = 0; e < BKV; ++e)
              if (e <= lim) mx = fmaxf(mx, __uint_as_float(v[e]));
          } else {
            float m4[4] = {mx, mx, mx, mx};
#pragma unroll
            for (int e = 0; e < BKV; e += 8) {
#pragma unroll
              for (int q = 0; q < 4; ++q) m4[q] = max3(m4[q], __uint_as_float(v[e + 2 * q]), __uint_as_float(v[e + 2 * q + 1]));
            }
            mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
          }
          const float m_new = fmaxf(m_run, mx * sl2);
          float alpha = 1.f;
          bool resc = false;
          if (m_new > m_run + kRescaleLog2) {
            alpha = ex2(m_run - m_new);
            m_run = m_new;
            resc = true;
          }
          // P = 2^(s*scale - m) as bf16 pairs into S's first 64 columns (S itself
          // is already in registers)
          float rs = 0.f;
          uint64_t rs2 = f2(0.f, 0.f);
          const uint64_t sl2x2 = f2(sl2, sl2), negm2 = f2(-m_run, -m_run);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t pk[32];
            if (diag) {
#pragma unroll
              for (int e = 0; e < 64; e += 2) {
                const int col = h * 64 + e;
                const float p0 = col <= lim ? ex2(fmaf(__uint_as_float(v[col]), sl2, -m_run)) : 0.f;
                const float p1 = col + 1 <= lim ? ex2(fmaf(__uint_as_float(v[col + 1]), sl2, -m_run)) : 0.f;
                rs += p0 + p1;
                pk[e >> 1] = pack_bf16(p0, p1);
              }
            } else {
#pragma unroll
              for (int e = 0; e < 64; e += 2) {
                const int col = h * 64 + e;
                const uint64_t x = fma2(f2(__uint_as_float(v[col]), __uint_as_float(v[col + 1])), sl2x2, negm2);
                const float p0 = ex2(f2_lo(x));
                const float p1 = ex2(f2_hi(x));
                rs2 = add2(rs2, f2(p0, p1));
                pk[e >> 1] = pack_bf16(p0, p1);
              }
            }
            tmem_st32(t_s + h * 32, pk);
          }
          // O (complete up to block j-1, see above) follows a raised reference;
          // done after P so that S no longer occupies registers
          if (j > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(t_o + c * 32, o);
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tmem_st32(t_o + c * 32, o);
            }
          }
          l_run = l_run * alpha + (rs + (f2_lo(rs2) + f2_hi(rs2)));
          tc_fence_before();
          mbar_arrive(&p_ready[tile]);
        }
        if (ok && mbar_wait_warp(&o_done[tile], 0, w, 27)) {
          tc_fence_after();
          const long long orow_idx = static_cast<long long>(slot) * a.S + qi;
          uint16_t* orow = a.O + orow_idx * D;
          const float lse2_part = m_run + __log2f(l_run);  // this launch's keys, log2 units
          float* lrow = a.lse + static_cast<long long>(a.lse_row[slot]) * (GEN ? a.lse_ld : a.S) + qi;
          if (!GEN || a.mode == kFwdPlain) {
            const float inv = 1.f / l_run;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t v[32];
              tmem_ld32(t_o + c * 32, v);
              uint4* o = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                o[i] = make_uint4(pack_bf16(__uint_as_float(v[8 * i]) * inv, __uint_as_float(v[8 * i + 1]) * inv),
                                  pack_bf16(__uint_as_float(v[8 * i + 2]) * inv, __uint_as_float(v[8 * i + 3]) * inv),
                                  pack_bf16(__uint_as_float(v[8 * i + 4]) * inv, __uint_as_float(v[8 * i + 5]) * inv),
                                  pack_bf16(__uint_as_float(v[8 * i + 6]) * inv, __uint_as_float(v[8 * i + 7]) * inv));
              }
            }
            *lrow = lse2_part * 0.69314718055994531f;
          } else {
            // merge with the running result of the earlier key chunks (fp32
            // output normalised over its keys, log-sum-exp in log2 units):
            // weights 2^(lse_x - lse_union)
            float* acc = a.o_acc + orow_idx * D;
            float* lacc = a.lse_acc + orow_idx;
            float wa = 0.f, wb = 1.f / l_run, lse2_new = lse2_part;
            if (a.mode != kFwdFirst) {
              const float prev = *lacc;
              const float m = fmaxf(prev, lse2_part);
              const float ea = ex2(prev - m), eb = ex2(lse2_part - m);
              const float inv_s = 1.f / (ea + eb);
              wa = ea * inv_s;
              wb = eb * inv_s / l_run;
              lse2_new = m + __log2f(ea + eb);
            }
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t v[32];
              tmem_ld32(t_o + c * 32, v);
              float4* ac = reinterpret_cast<float4*>(acc + c * 32);
              float x[32];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                float4 p = make_float4(0.f, 0.f, 0.f, 0.f);
                if (a.mode != kFwdFirst) p = ac[i];
                x[4 * i] = fmaf(__uint_as_float(v[4 * i]), wb, p.x * wa);
                x[4 * i + 1] = fmaf(__uint_as_float(v[4 * i + 1]), wb, p.y * wa);
                x[4 * i + 2] = fmaf(__uint_as_float(v[4 * i + 2]), wb, p.z * wa);
                x[4 * i + 3] = fmaf(__uint_as_float(v[4 * i + 3]), wb, p.w * wa);
              }
              if (a.mode == kFwdLast) {
                uint4* o = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  o[i] = make_uint4(pack_bf16(x[8 * i], x[8 * i + 1]), pack_bf16(x[8 * i + 2], x[8 * i + 3]),
                                    pack_bf16(x[8 * i + 4], x[8 * i + 5]), pack_bf16(x[8 * i + 6], x[8 * i + 7]));
              } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) ac[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
              }
            }
            if (a.mode == kFwdLast)
              *lrow = lse2_new * 0.69314718055994531f;
            else
              *lacc = lse2_new;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool F8, bool GEN>
cudaError_t run_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdArgs& args,
                    cudaStream_t st) {
  auto kern = attn_fwd_kernel<D, F8, GEN>;
  // the kernel needs more than the default 48 KB of dynamic shared memory;
  // the limit is raised once per device
  if (const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), FwdCfg<D, F8>::SMEM); e != cudaSuccess)
    return e;
  kern<<<args.n_qslots * args.q_pairs, 384, FwdCfg<D, F8>::SMEM, st>>>(tq, tk, tv, args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(const AttnFwdDesc& d, int* status, cudaStream_t st) {
  const int kv_len = d.kv_len ? d.kv_len : d.S;
  const int kv_ld = d.kv_ld ? d.kv_ld : kv_len;
  if ((d.D != 64 && d.D != 128) || d.S % 128 || d.n_qslots <= 0 || d.n_qslots > kMaxSlots) return cudaErrorInvalidValue;
  if (kv_len <= 0 || kv_len % 128 || kv_ld < kv_len || d.q_off < 0 || d.q_off % 128 || d.n_kvslots <= 0)
    return cudaErrorInvalidValue;
  if (d.mode < kFwdPlain || d.mode > kFwdLast || (d.mode != kFwdPlain && (!d.o_acc || !d.lse_acc)))
    return cudaErrorInvalidValue;
  for (int i = 0; i < d.n_qslots; ++i)
    if (d.kv_slot[i] >= d.n_kvslots) return cudaErrorInvalidValue;
  if (d.fp8 && (d.D != 128 || !d.q_scale || !d.k_scale)) return cudaErrorInvalidValue;
  CUtensorMap tq, tk, tv;
  if (d.fp8) {
    if (!make_tmap_u8(&tq, d.Q, d.D, (uint64_t)d.n_qslots * d.S, d.D, 128, 128)) return cudaErrorInvalidValue;
    if (!make_tmap_u8(&tk, d.K, d.D, (uint64_t)d.n_kvslots * kv_ld, d.D, 128, 128)) return cudaErrorInvalidValue;
  } else {
    if (!make_tmap_bf16(&tq, d.Q, d.D, (uint64_t)d.n_qslots * d.S, d.D, 64, 128)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16(&tk, d.K, d.D, (uint64_t)d.n_kvslots * kv_ld, d.D, 64, 128)) return cudaErrorInvalidValue;
  }
  if (!make_tmap_bf16(&tv, d.V, d.D, (uint64_t)d.n_kvslots * kv_ld, d.D, 64, 128)) return cudaErrorInvalidValue;
  FwdArgs a;
  a.S = d.S;
  a.kv_ld = kv_ld;
  a.kv_blocks = kv_len / BKV;
  a.q_off_blocks = d.q_off / BQ;
  a.lse_ld = d.lse_ld ? d.lse_ld : d.S;
  a.mode = d.mode;
  a.o_acc = d.o_acc;
  a.lse_acc = d.lse_acc;
  a.q_scale = d.q_scale;
  a.k_scale = d.k_scale;
  a.n_qslots = d.n_qslots;
  a.q_blocks = d.S / BQ;
  a.q_pairs = (a.q_blocks + 1) / 2;
  a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d.D)));
  for (int i = 0; i < d.n_qslots; ++i) {
    a.kv_slot[i] = d.kv_slot[i];
    a.lse_row[i] = d.lse_row[i];
  }
  a.O = static_cast<uint16_t*>(d.O);
  a.lse = d.lse;
  a.status = status;
  const bool gen = d.q_off != 0 || kv_len != d.S || kv_ld != d.S || a.lse_ld != d.S || d.mode != kFwdPlain;
  if (d.fp8) return gen ? cudaErrorInvalidValue : run_fwd<128, true, false>(tq, tk, tv, a, st);
  if (gen) return d.D == 128 ? run_fwd<128, false, true>(tq, tk, tv, a, st) : run_fwd<64, false, true>(tq, tk, tv, a, st);
  return d.D == 128 ? run_fwd<128, false, false>(tq, tk, tv, a, st) : run_fwd<64, false, false>(tq, tk, tv, a, st);
}

}  // namespace upipe
