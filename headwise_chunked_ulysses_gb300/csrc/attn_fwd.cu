// Causal GQA attention forward for the heads one stage holds ("Untied
// Ulysses" summary, Method steps (3): attention of the stage's U heads).
//
// O = softmax(Q K^T / sqrt(d) + causal mask) V, with the natural-log
// log-sum-exp of every row saved for the backward pass.  Query slots map to
// KV slots through a table, so grouped-query heads read their shared K/V.
//
// One CTA per (query slot, 128-row query block); blocks with the longest
// causal rows are scheduled first.  Warp 0 streams K/V blocks of 128 rows by
// TMA into a two-deep ring; warp 1 issues S = Q K^T (M=N=128) into one of two
// TMEM score buffers while the softmax warps (4..7, one query row per
// thread) turn the other into P (bf16, written to shared memory in the MMA's
// 128-byte-swizzled K-major layout) and then O += P V accumulates in TMEM.
// The online softmax keeps a per-row reference maximum and rescales the TMEM
// accumulator only when the running maximum grows by more than 2^8, so the
// rescale is rare and exact (the same reference enters numerator and
// denominator).
#include <cmath>

#include "ptx.cuh"
#include "upipe_internal.h"

namespace upipe {
namespace {

constexpr int BQ = 128;   // query rows per CTA
constexpr int BKV = 128;  // key rows per block
constexpr int CH = 128 * 128;  // one 64-column chunk of a 128-row tile (bytes)
constexpr float kRescaleLog2 = 8.0f;

struct FwdArgs {
  int S, n_qslots, q_blocks;
  float scale_log2;
  uint16_t kv_slot[kMaxSlots];
  uint16_t lse_row[kMaxSlots];
  uint16_t* O;
  float* lse;
  int* status;
};

template <int D>
struct FwdCfg {
  static constexpr int TILE = BQ * D * 2;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = TILE;          // 2 stages
  static constexpr int V_OFF = 3 * TILE;      // 2 stages
  static constexpr int P_OFF = 5 * TILE;      // 128 x 128 bf16
  static constexpr int BAR_OFF = P_OFF + BQ * BKV * 2;
  static constexpr int SMEM = BAR_OFF + 256;
  static constexpr uint32_t TMEM_COLS = 512;  // S0 [0,128) S1 [128,256) O [256,256+D)
};

template <int D>
__global__ void __launch_bounds__(256, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ FwdArgs a) {
  using C = FwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;    // [2]
  uint64_t* v_full = bars + 3;    // [2]
  uint64_t* kv_empty = bars + 5;  // [2]
  uint64_t* s_full = bars + 7;    // [2]
  uint64_t* p_full = bars + 9;
  uint64_t* pv_done = bars + 10;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 11);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Watch w{abort_flag, a.status};
  const bool aligned = (smem_u32(smem) & 1023u) == 0;

  const int qb = a.q_blocks - 1 - static_cast<int>(blockIdx.x) / a.n_qslots;
  const int slot = static_cast<int>(blockIdx.x) % a.n_qslots;
  const int kvs = a.kv_slot[slot];
  const int n_kv = qb + 1;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
      mbar_init(&s_full[s], 1);
    }
    mbar_init(p_full, 128);
    mbar_init(pv_done, 1);
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
      mbar_arrive_expect_tx(q_full, C::TILE);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_2d(smem + C::Q_OFF + c * CH, &tmQ, q_full, c * 64, slot * a.S + qb * BQ);
      for (int j = 0; j < n_kv; ++j) {
        const int s = j & 1;
        if (!mbar_wait(&kv_empty[s], ((j >> 1) & 1) ^ 1, w, 20)) break;
        const int row = kvs * a.S + j * BKV;
        mbar_arrive_expect_tx(&k_full[s], C::TILE);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(smem + C::K_OFF + s * C::TILE + c * CH, &tmK, &k_full[s], c * 64, row);
        mbar_arrive_expect_tx(&v_full[s], C::TILE);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(smem + C::V_OFF + s * C::TILE + c * CH, &tmV, &v_full[s], c * 64, row);
      }
    } else if (warp == 1 && lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t ID_S = idesc_bf16(BQ, BKV, false, false);
      constexpr uint32_t ID_O = idesc_bf16(BQ, D, false, true);
      const uint32_t sQ = smem_u32(smem + C::Q_OFF);
      const uint32_t sP = smem_u32(smem + C::P_OFF);
      bool ok = mbar_wait(q_full, 0, w, 21);
      auto issue_s = [&](int j) -> bool {
        const int s = j & 1;
        if (!mbar_wait(&k_full[s], (j >> 1) & 1, w, 22)) return false;
        tc_fence_after();
        const uint32_t sK = smem_u32(smem + C::K_OFF + s * C::TILE);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * CH + (k & 3) * 32;
          mma_ss(tmem + s * BKV, sdesc_kmajor(sQ + off), sdesc_kmajor(sK + off), ID_S, k > 0);
        }
        mma_commit(&s_full[s]);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int s = j & 1;
        if (j + 1 < n_kv && !issue_s(j + 1)) break;
        if (!mbar_wait(p_full, j & 1, w, 23)) break;
        if (!mbar_wait(&v_full[s], (j >> 1) & 1, w, 24)) break;
        tc_fence_after();
        const uint32_t sV = smem_u32(smem + C::V_OFF + s * C::TILE);
#pragma unroll
        for (int k = 0; k < BKV / 16; ++k) {
          const uint32_t poff = (k >> 2) * CH + (k & 3) * 32;
          mma_ss(tmem + 256, sdesc_kmajor(sP + poff), sdesc_mnmajor(sV + k * 2048, CH), ID_O, (j | k) != 0);
        }
        mma_commit(pv_done);
        mma_commit(&kv_empty[s]);
      }
    } else if (warp >= 4) {
      // ---------------- softmax: one query row per thread ----------------
      const int q4 = warp & 3;
      const int row = q4 * 32 + lane;
      const int qi = qb * BQ + row;
      const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
      const float sl2 = a.scale_log2;
      float m_run = -INFINITY, l_run = 0.f;
      bool ok = true;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j & 1;
        if (!mbar_wait_warp(&s_full[s], (j >> 1) & 1, w, 25)) { ok = false; break; }
        tc_fence_after();
        float x[BKV];
#pragma unroll
        for (int c = 0; c < BKV / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + s * BKV + c * 32, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) x[c * 32 + i] = __uint_as_float(v[i]);
        }
        if (j == n_kv - 1) {
          const int lim = qi - j * BKV;  // keys with column index > lim are in the future
#pragma unroll
          for (int i = 0; i < BKV; ++i)
            if (i > lim) x[i] = -INFINITY;
        }
        float mx = x[0];
#pragma unroll
        for (int i = 1; i < BKV; ++i) mx = fmaxf(mx, x[i]);
        const float m_new = fmaxf(m_run, mx * sl2);
        float alpha = 1.f;
        bool resc = false;
        if (m_new > m_run + kRescaleLog2) {
          alpha = ex2(m_run - m_new);
          m_run = m_new;
          resc = true;
        }
        uint32_t pk[BKV / 2];
        float rs = 0.f;
#pragma unroll
        for (int i = 0; i < BKV / 2; ++i) {
          const float p0 = ex2(fmaf(x[2 * i], sl2, -m_run));
          const float p1 = ex2(fmaf(x[2 * i + 1], sl2, -m_run));
          rs += p0 + p1;
          pk[i] = pack_bf16(p0, p1);
        }
        l_run = l_run * alpha + rs;
        if (j > 0) {
          // P buffer and the O accumulator are free once P_{j-1} V_{j-1} is done.
          if (!mbar_wait_warp(pv_done, (j - 1) & 1, w, 26)) { ok = false; break; }
          tc_fence_after();
          if (__any_sync(0xffffffffu, resc)) {
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t v[32];
              const uint32_t ta = tmem + lane_off + 256 + c * 32;
              tmem_ld32(ta, v);
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
              tmem_st32(ta, v);
            }
          }
        }
        const uint32_t sP = smem_u32(smem + C::P_OFF);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int piece = 0; piece < 8; ++piece) {
            const uint32_t addr = sP + c * CH + row * 128 + ((piece ^ (row & 7)) << 4);
            const int b = c * 32 + piece * 4;
            st_shared_v4(addr, pk[b], pk[b + 1], pk[b + 2], pk[b + 3]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(p_full);
      }
      if (ok && mbar_wait_warp(pv_done, (n_kv - 1) & 1, w, 27)) {
        tc_fence_after();
        const float inv = 1.f / l_run;
        uint16_t* orow = a.O + (static_cast<long long>(slot) * a.S + qi) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + 256 + c * 32, v);
          uint4* o = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            o[i] = make_uint4(pack_bf16(__uint_as_float(v[8 * i]) * inv, __uint_as_float(v[8 * i + 1]) * inv),
                              pack_bf16(__uint_as_float(v[8 * i + 2]) * inv, __uint_as_float(v[8 * i + 3]) * inv),
                              pack_bf16(__uint_as_float(v[8 * i + 4]) * inv, __uint_as_float(v[8 * i + 5]) * inv),
                              pack_bf16(__uint_as_float(v[8 * i + 6]) * inv, __uint_as_float(v[8 * i + 7]) * inv));
          }
        }
        a.lse[static_cast<long long>(a.lse_row[slot]) * a.S + qi] = (m_run + __log2f(l_run)) * 0.69314718055994531f;
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

template <int D>
cudaError_t run_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdArgs& args,
                    cudaStream_t st) {
  auto kern = attn_fwd_kernel<D>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FwdCfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  kern<<<args.n_qslots * args.q_blocks, 256, FwdCfg<D>::SMEM, st>>>(tq, tk, tv, args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(const AttnFwdDesc& d, int* status, cudaStream_t st) {
  if ((d.D != 64 && d.D != 128) || d.S % 128 || d.n_qslots <= 0 || d.n_qslots > kMaxSlots) return cudaErrorInvalidValue;
  CUtensorMap tq, tk, tv;
  if (!make_tmap_bf16(&tq, d.Q, d.D, (uint64_t)d.n_qslots * d.S, d.D, 64, 128)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tk, d.K, d.D, (uint64_t)d.n_kvslots * d.S, d.D, 64, 128)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tv, d.V, d.D, (uint64_t)d.n_kvslots * d.S, d.D, 64, 128)) return cudaErrorInvalidValue;
  FwdArgs a;
  a.S = d.S;
  a.n_qslots = d.n_qslots;
  a.q_blocks = d.S / BQ;
  a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d.D)));
  for (int i = 0; i < d.n_qslots; ++i) {
    a.kv_slot[i] = d.kv_slot[i];
    a.lse_row[i] = d.lse_row[i];
  }
  a.O = static_cast<uint16_t*>(d.O);
  a.lse = d.lse;
  a.status = status;
  return d.D == 128 ? run_fwd<128>(tq, tk, tv, a, st) : run_fwd<64>(tq, tk, tv, a, st);
}

}  // namespace upipe
