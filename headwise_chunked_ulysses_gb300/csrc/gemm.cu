// Dense bf16 contraction on the 5th-generation tensor cores.
//
// Serves the layer's projections: the per-stage QKV projection X * W_qkv[:,
// stage heads] ("Untied Ulysses" summary, Method steps (1)), the per-stage
// output-projection share O_s * W_o[stage rows] that each stage adds into Y,
// and the matching backward contractions (dO, dX, dW_qkv, dW_o).
//
// Design: persistent CTAs (one per SM), 128 x BN output tiles, K in blocks of
// 64.  Warp 0 issues TMA loads of 64x64 bf16 boxes (128-byte swizzle) into a
// STAGES-deep shared-memory ring; warp 1 issues tcgen05.mma (M=128, N=BN,
// K=16) into one of two TMEM accumulators; warps 4..7 drain the other
// accumulator (tcgen05.ld) and write the epilogue, so the epilogue of tile t
// overlaps the main loop of tile t+1.  Every box coordinate passes through an
// optional 64-block gather map, which is how the non-contiguous head sets of
// the out-of-order schedule are read without copies; the K maps are copied
// into shared memory before the main loop, so per K block the producer only
// waits for a free stage, reads two map entries and issues its loads.  Split-K
// (few output tiles, long K) cuts K into ranges of about K/64/split_k blocks
// whose fp32 partial sums the TMA engine adds into the output.
#include <algorithm>

#include "ptx.cuh"
#include "upipe_internal.h"

namespace upipe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int BOX_BYTES = 64 * 64 * 2;  // one 64x64 bf16 box: 64 rows of 128 B

struct GemmArgs {
  int M, N, K;
  int m_tiles, n_tiles, split_k;
  int use_amap_k, use_bmap_k, use_bmap_n, use_omap_n;
  uint16_t amap_k[kMaxMap];
  uint16_t bmap_k[kMaxMap];
  uint16_t bmap_n[kMaxMap];
  uint16_t omap_n[kMaxMap];
  void* out;
  long long ldo;
  int out_mode;
  int acc_load;  // fp32 +=: old values read by TMA and the sums stored, instead of reduce-adds
  const float* aux;
  long long ld_aux;
  int* status;
};

// The K-block gather maps go to shared memory before the main loop: the
// producer thread reads one entry of each per K block, right after waiting
// for a free ring stage, and a dynamically indexed kernel parameter is a
// constant-cache load that can miss (a miss there delays every refill).
__device__ __forceinline__ void stage_k_maps(const GemmArgs& g, uint16_t* kmap, int lane) {
  const int n = g.K / BK;
  if (g.use_amap_k)
    for (int i = lane; i < n; i += 32) kmap[i] = g.amap_k[i];
  if (g.use_bmap_k)
    for (int i = lane; i < n; i += 32) kmap[kMaxMap + i] = g.bmap_k[i];
}

template <int BN>
struct Cfg {
  static constexpr int STAGES = BN == 256 ? 4 : (BN == 128 ? 6 : 8);
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr int MAP_OFF = BAR_OFF + 256;  // K-block maps of A and B: 2 x kMaxMap uint16
  static constexpr int SMEM = MAP_OFF + 2 * kMaxMap * 2;
};

__device__ __forceinline__ void store_tile_chunk(const GemmArgs& g, int m, int oc, const uint32_t (&v)[32]) {
  if (g.out_mode == kOutF32Red) {  // split-K partial sums: vector reductions
    float* o = static_cast<float*>(g.out) + (long long)m * g.ldo + oc;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      red_add_v4(o + 4 * i, __uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]), __uint_as_float(v[4 * i + 2]),
                 __uint_as_float(v[4 * i + 3]));
  } else if (g.out_mode == kOutF32 || g.out_mode == kOutF32Acc) {
    float4* o = reinterpret_cast<float4*>(static_cast<float*>(g.out) + (long long)m * g.ldo + oc);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float4 x = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]), __uint_as_float(v[4 * i + 2]),
                             __uint_as_float(v[4 * i + 3]));
      if (g.out_mode == kOutF32Acc) {
        const float4 p = o[i];
        x.x += p.x; x.y += p.y; x.z += p.z; x.w += p.w;
      }
      o[i] = x;
    }
  } else {
    float f[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
    if (g.out_mode == kOutBf16PlusF32) {
      const float4* a = reinterpret_cast<const float4*>(g.aux + (long long)m * g.ld_aux + oc);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 p = a[i];
        f[4 * i] += p.x; f[4 * i + 1] += p.y; f[4 * i + 2] += p.z; f[4 * i + 3] += p.w;
      }
    }
    uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(g.out) + (long long)m * g.ldo + oc);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[i] = make_uint4(pack_bf16(f[8 * i], f[8 * i + 1]), pack_bf16(f[8 * i + 2], f[8 * i + 3]),
                        pack_bf16(f[8 * i + 4], f[8 * i + 5]), pack_bf16(f[8 * i + 6], f[8 * i + 7]));
    }
  }
}

template <int BN, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(256, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ GemmArgs g) {
  using C = Cfg<BN>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Watch w{abort_flag, g.status};
  const bool aligned = (smem_u32(smem) & 1023u) == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    *abort_flag = aligned ? 0 : 1;
    if (!aligned && g.status) atomicCAS(g.status, 0, kDevBadSmem);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
  }
  uint16_t* kmap = reinterpret_cast<uint16_t*>(smem + C::MAP_OFF);
  if (warp == 3) stage_k_maps(g, kmap, lane);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_tiles = g.m_tiles * g.n_tiles * g.split_k;
  const int kb_all = g.K / BK;
  // tile t: split ks = t / (m_tiles*n_tiles), then m-major, n fastest; split
  // ks covers K blocks [ks*kb_all/split_k, (ks+1)*kb_all/split_k)
  auto tile_m0 = [&](int t) { return ((t % (g.m_tiles * g.n_tiles)) / g.n_tiles) * BM; };
  auto tile_n0 = [&](int t) { return (t % g.n_tiles) * BN; };
  auto tile_kb0 = [&](int t) { return (t / (g.m_tiles * g.n_tiles)) * kb_all / g.split_k; };
  auto tile_kbs = [&](int t) { return tile_kb0(t + g.m_tiles * g.n_tiles) - tile_kb0(t); };

  if (aligned) {
    if (warp == 0 && lane == 0) {
      // ---------------- TMA producer ----------------
      int s = 0;        // ring stage
      uint32_t ph = 0;  // its phase parity
      bool ok = true;
      for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
        const int m0 = tile_m0(t), n0 = tile_n0(t), kb0 = tile_kb0(t), kb1 = kb0 + tile_kbs(t);
        int nc[BN / 64];  // the tile's B columns, fixed over its K loop
#pragma unroll
        for (int i = 0; i < BN / 64; ++i) nc[i] = (g.use_bmap_n ? g.bmap_n[n0 / 64 + i] : n0 / 64 + i) * 64;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[s], ph ^ 1, w, 1)) { ok = false; break; }
          uint8_t* sa = smem + s * C::STAGE_BYTES;
          uint8_t* sb = sa + C::A_BYTES;
          mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
          const int ka = (g.use_amap_k ? kmap[kb] : kb) * BK;
          const int kbb = (g.use_bmap_k ? kmap[kMaxMap + kb] : kb) * BK;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            if (A_MN) tma_load_2d(sa + i * BOX_BYTES, &tmA, &full[s], m0 + 64 * i, ka);
            else      tma_load_2d(sa + i * BOX_BYTES, &tmA, &full[s], ka, m0 + 64 * i);
          }
#pragma unroll
          for (int i = 0; i < BN / 64; ++i) {
            if (B_MN) tma_load_2d(sb + i * BOX_BYTES, &tmB, &full[s], nc[i], kbb);
            else      tma_load_2d(sb + i * BOX_BYTES, &tmB, &full[s], kbb, nc[i]);
          }
          if (++s == STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
      }
    } else if (warp == 1 && lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t IDESC = idesc_bf16(BM, BN, A_MN, B_MN);
      int s = 0, tl = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x, ++tl) {
        const int acc = tl & 1;
        if (!mbar_wait(&tempty[acc], ((tl >> 1) & 1) ^ 1, w, 2)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * BN;
        const int kblocks = tile_kbs(t);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&full[s], ph, w, 3)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * C::STAGE_BYTES);
          const uint32_t sb = sa + C::A_BYTES;
          const uint64_t a0 = A_MN ? sdesc_mnmajor(sa, BOX_BYTES) : sdesc_kmajor(sa);
          const uint64_t b0 = B_MN ? sdesc_mnmajor(sb, BOX_BYTES) : sdesc_kmajor(sb);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = sdesc_advance(a0, A_MN ? k * 2048 : k * 32);
            const uint64_t bd = sdesc_advance(b0, B_MN ? k * 2048 : k * 32);
            mma_ss(d_tmem, ad, bd, IDESC, (kb | k) != 0);
          }
          mma_commit(&empty[s]);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
        if (ok) mma_commit(&tfull[acc]);
      }
    } else if (warp >= 4) {
      // ---------------- epilogue (4 warps, one TMEM lane quarter each) ----------------
      const int q = warp & 3;
      const int row = q * 32 + lane;
      int tl = 0;
      for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++tl) {
        const int acc = tl & 1;
        if (!mbar_wait_warp(&tfull[acc], (tl >> 1) & 1, w, 4)) break;
        tc_fence_after();
        const int m = tile_m0(t) + row;
        const int n0 = tile_n0(t);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * BN + c * 32, v);
          const int n = n0 + c * 32;
          const int oc = g.use_omap_n ? g.omap_n[n >> 6] * 64 + (n & 63) : n;
          // the last row tile of an M that is a multiple of 64 only: its A
          // rows past M were read as zeros and its rows past M are not written
          if (m < g.M) store_tile_chunk(g, m, oc, v);
        }
        tc_fence_before();
        mbar_arrive(&tempty[acc]);
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

// ---------------------------------------------------------------------------
// Paired-CTA variant: a cluster of two CTAs computes a 256 x 256 output tile
// with the M=256 form of the MMA.  CTA r of the pair loads A rows
// [m0 + 128r, +128) and B columns [n0 + 128r, +128) of each 64-deep K block
// into its own shared memory, so each SM reads and writes half of B compared
// with one CTA computing 128 x 256: the shared-memory traffic per MMA falls
// from about 1.5x to about 1x of what one SM can move.  CTA 0 issues the MMAs
// (operands at the same shared offsets in both CTAs) and owns the pair's "full"
// barriers, on which both CTAs' TMA loads complete; MMA completion is
// multicast to both CTAs' "empty" and "accumulator full" barriers; each CTA
// drains its own 128 accumulator rows and reports to CTA 0's "accumulator
// empty" barrier.
// ---------------------------------------------------------------------------
struct Cfg2 {
  static constexpr int STAGES = 6;
  static constexpr int A_BYTES = 128 * BK * 2;   // this CTA's A rows
  static constexpr int B_BYTES = 128 * BK * 2;   // this CTA's B columns
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TMEM_COLS = 512;          // two 256-column accumulators
  static constexpr int EPI_OFF = STAGES * STAGE_BYTES;  // fp32 output staging: 4 warps x 2 x (32 x 32)
  static constexpr int EPI_BYTES = 4 * 2 * 32 * 32 * 4;
  static constexpr int BAR_OFF = EPI_OFF + EPI_BYTES;
  static constexpr int MAP_OFF = BAR_OFF + 256;  // K-block maps of A and B: 2 x kMaxMap uint16
  static constexpr int SMEM = MAP_OFF + 2 * kMaxMap * 2;
};

template <bool A_MN, bool B_MN>
__global__ void __launch_bounds__(256, 1)
    gemm2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmO, const __grid_constant__ GemmArgs g) {
  using C = Cfg2;
  constexpr int STAGES = C::STAGES;
  constexpr int BNP = 256;  // output columns per pair tile
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);  // used in CTA 0
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;  // used in CTA 0
  uint64_t* aux_full = tempty + 2;  // [4 warps][2 buffers]: accumulator chunks loaded for bf16 = acc + aux
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(aux_full + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const Watch w{abort_flag, g.status};
  const bool aligned = (smem_u32(smem) & 1023u) == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 256);  // both CTAs' epilogue threads
    }
    for (int b = 0; b < 8; ++b) mbar_init(&aux_full[b], 1);
    *abort_flag = aligned ? 0 : 1;
    if (!aligned && g.status) atomicCAS(g.status, 0, kDevBadSmem);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
  }
  uint16_t* kmap = reinterpret_cast<uint16_t*>(smem + C::MAP_OFF);
  if (warp == 3) stage_k_maps(g, kmap, lane);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before any remote use
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int pair = static_cast<int>(blockIdx.x) >> 1, n_pairs = static_cast<int>(gridDim.x) >> 1;
  const int n_tiles = g.m_tiles * g.n_tiles * g.split_k;  // m_tiles counts 256-row tiles here
  const int kb_all = g.K / BK;
  auto tile_m0 = [&](int t) { return ((t % (g.m_tiles * g.n_tiles)) / g.n_tiles) * 256; };
  auto tile_n0 = [&](int t) { return (t % g.n_tiles) * BNP; };
  auto tile_kb0 = [&](int t) { return (t / (g.m_tiles * g.n_tiles)) * kb_all / g.split_k; };
  auto tile_kbs = [&](int t) { return tile_kb0(t + g.m_tiles * g.n_tiles) - tile_kb0(t); };
  const uint32_t full0 = mapa_shared(smem_u32(full), 0);     // CTA 0's full[0]
  const uint32_t tempty0 = mapa_shared(smem_u32(tempty), 0); // CTA 0's tempty[0]

  if (aligned) {
    if (warp == 0 && lane == 0) {
      // ---------------- TMA producer (both CTAs) ----------------
      int s = 0;        // ring stage
      uint32_t ph = 0;  // its phase parity
      bool ok = true;
      for (int t = pair; ok && t < n_tiles; t += n_pairs) {
        const int m0 = tile_m0(t) + 128 * static_cast<int>(rank), n0 = tile_n0(t) + 128 * static_cast<int>(rank);
        const int kb0 = tile_kb0(t), kb1 = kb0 + tile_kbs(t);
        // the tile's B columns are fixed over its K loop
        const int nc0 = (g.use_bmap_n ? g.bmap_n[n0 / 64] : n0 / 64) * 64;
        const int nc1 = (g.use_bmap_n ? g.bmap_n[n0 / 64 + 1] : n0 / 64 + 1) * 64;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[s], ph ^ 1, w, 61)) { ok = false; break; }
          uint8_t* sa = smem + s * C::STAGE_BYTES;
          uint8_t* sb = sa + C::A_BYTES;
          const uint32_t fb = full0 + s * 8;
          if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * C::STAGE_BYTES);
          const int ka = (g.use_amap_k ? kmap[kb] : kb) * BK;
          const int kbb = (g.use_bmap_k ? kmap[kMaxMap + kb] : kb) * BK;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            if (A_MN) tma_load_2d_pair(sa + i * BOX_BYTES, &tmA, fb, m0 + 64 * i, ka);
            else      tma_load_2d_pair(sa + i * BOX_BYTES, &tmA, fb, ka, m0 + 64 * i);
          }
          if (B_MN) {
            tma_load_2d_pair(sb, &tmB, fb, nc0, kbb);
            tma_load_2d_pair(sb + BOX_BYTES, &tmB, fb, nc1, kbb);
          } else {
            tma_load_2d_pair(sb, &tmB, fb, kbb, nc0);
            tma_load_2d_pair(sb + BOX_BYTES, &tmB, fb, kbb, nc1);
          }
          if (++s == STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
      }
    } else if (warp == 1 && lane == 0 && rank == 0) {
      // ---------------- MMA issuer (CTA 0 only) ----------------
      constexpr uint32_t IDESC = idesc_bf16(256, BNP, A_MN, B_MN);
      int s = 0, tl = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = pair; ok && t < n_tiles; t += n_pairs, ++tl) {
        const int acc = tl & 1;
        if (!mbar_wait(&tempty[acc], ((tl >> 1) & 1) ^ 1, w, 62)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * BNP;
        const int kblocks = tile_kbs(t);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&full[s], ph, w, 63)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * C::STAGE_BYTES);
          const uint32_t sb = sa + C::A_BYTES;
          const uint64_t a0 = A_MN ? sdesc_mnmajor(sa, BOX_BYTES) : sdesc_kmajor(sa);
          const uint64_t b0 = B_MN ? sdesc_mnmajor(sb, BOX_BYTES) : sdesc_kmajor(sb);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = sdesc_advance(a0, A_MN ? k * 2048 : k * 32);
            const uint64_t bd = sdesc_advance(b0, B_MN ? k * 2048 : k * 32);
            mma_ss_pair(d_tmem, ad, bd, IDESC, (kb | k) != 0);
          }
          mma_commit_pair(&empty[s]);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
        if (ok) mma_commit_pair(&tfull[acc]);
      }
    } else if (warp >= 4) {
      // ---------------- epilogue: this CTA's 128 rows of the pair tile ----------------
      // fp32 outputs leave through the TMA engine: each warp stages 32 x 32
      // chunks of its rows (128-byte swizzle, two buffers) and stores them, or
      // adds them atomically into the output (short-K accumulate, split-K
      // partials), with no read of the old values into the SM; a long-K
      // accumulate reads the old chunk by TMA (one ahead, the first while the
      // tile's accumulator is still being computed), adds and stores
      const int q = warp & 3;
      const int row = q * 32 + lane;
      const bool acc_in = g.out_mode == kOutF32Acc && g.acc_load;
      const bool tma_out = g.out_mode == kOutF32 || g.out_mode == kOutF32Red || (g.out_mode == kOutF32Acc && !acc_in);
      const bool tma_add = g.out_mode != kOutF32;
      // bf16 = acc + aux: the aux (fp32) chunks come in by TMA, one ahead
      const bool aux_in = g.out_mode == kOutBf16PlusF32;
      const uint32_t epi = smem_u32(smem + C::EPI_OFF) + q * (2 * 32 * 32 * 4);
      uint64_t* abar = aux_full + q * 2;
      int nb = 0;  // chunks this warp has handed to (or taken from) the TMA engine
      int tl = 0;
      for (int t = pair; t < n_tiles; t += n_pairs, ++tl) {
        const int acc = tl & 1;
        const int m = tile_m0(t) + 128 * static_cast<int>(rank) + row;
        const int n0 = tile_n0(t);
        auto out_col = [&](int c) {
          const int n = n0 + c * 32;
          return g.use_omap_n ? g.omap_n[n >> 6] * 64 + (n & 63) : n;
        };
        auto load_aux = [&](int c, int k) {  // chunk c of this warp's rows into buffer k&1
          if (lane == 0) {
            mbar_arrive_expect_tx(&abar[k & 1], 32 * 32 * 4);
            tma_load_2d(smem + C::EPI_OFF + q * (2 * 32 * 32 * 4) + (k & 1) * (32 * 32 * 4), &tmO, &abar[k & 1],
                        out_col(c), m - lane);
          }
        };
        // the tile's first input chunk comes in while its accumulator is
        // still being computed
        if (acc_in && lane == 0) bulk_wait_read<0>();  // the stores out of both buffers have been read
        __syncwarp();
        if (aux_in || acc_in) load_aux(0, nb);
        if (!mbar_wait_warp(&tfull[acc], (tl >> 1) & 1, w, 64)) break;
        tc_fence_after();
        bool ok = true;
#pragma unroll 1
        for (int c = 0; c < BNP / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * BNP + c * 32, v);
          const int oc = out_col(c);
          if (tma_out) {
            const uint32_t buf = epi + (nb & 1) * (32 * 32 * 4);
            if (nb >= 2) {  // the chunk sent two chunks ago has left this buffer
              if (lane == 0) bulk_wait_read<1>();
              __syncwarp();
            }
#pragma unroll
            for (int p = 0; p < 8; ++p)
              st_shared_v4(buf + lane * 128 + ((p ^ (lane & 7)) << 4), v[4 * p], v[4 * p + 1], v[4 * p + 2], v[4 * p + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              if (tma_add) tma_reduce_add_2d(&tmO, buf, oc, m - lane);
              else tma_store_2d(&tmO, buf, oc, m - lane);
              bulk_commit();
            }
            ++nb;
          } else if (acc_in) {
            // fp32 +=, the long-K form: the old chunk came in by TMA one chunk
            // ahead; the sum goes back through the same buffer by a TMA store
            const uint32_t buf = epi + (nb & 1) * (32 * 32 * 4);
            if (c + 1 < BNP / 32) {
              // the next chunk's buffer: its last store has been read
              if (lane == 0) bulk_wait_read<0>();
              __syncwarp();
              load_aux(c + 1, nb + 1);
            }
            if (!mbar_wait_warp(&abar[nb & 1], (nb >> 1) & 1, w, 66)) { ok = false; break; }
#pragma unroll
            for (int p = 0; p < 8; ++p) {
              const uint32_t a = buf + lane * 128 + ((p ^ (lane & 7)) << 4);
              const uint4 x = ld_shared_v4(a);
              st_shared_v4(a, __float_as_uint(__uint_as_float(v[4 * p]) + __uint_as_float(x.x)),
                           __float_as_uint(__uint_as_float(v[4 * p + 1]) + __uint_as_float(x.y)),
                           __float_as_uint(__uint_as_float(v[4 * p + 2]) + __uint_as_float(x.z)),
                           __float_as_uint(__uint_as_float(v[4 * p + 3]) + __uint_as_float(x.w)));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmO, buf, oc, m - lane);
              bulk_commit();
            }
            ++nb;
          } else if (aux_in) {
            // the next chunk's aux is on its way while this one is added
            if (c + 1 < BNP / 32) load_aux(c + 1, nb + 1);
            if (!mbar_wait_warp(&abar[nb & 1], (nb >> 1) & 1, w, 65)) { ok = false; break; }
            const uint32_t buf = epi + (nb & 1) * (32 * 32 * 4);
            uint32_t pk16[16];
#pragma unroll
            for (int p = 0; p < 8; ++p) {
              const uint4 x = ld_shared_v4(buf + lane * 128 + ((p ^ (lane & 7)) << 4));
              pk16[2 * p] = pack_bf16(__uint_as_float(v[4 * p]) + __uint_as_float(x.x),
                                      __uint_as_float(v[4 * p + 1]) + __uint_as_float(x.y));
              pk16[2 * p + 1] = pack_bf16(__uint_as_float(v[4 * p + 2]) + __uint_as_float(x.z),
                                          __uint_as_float(v[4 * p + 3]) + __uint_as_float(x.w));
            }
            __syncwarp();  // every lane has read the buffer before it is loaded again
            uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(g.out) + (long long)m * g.ldo + oc);
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] = make_uint4(pk16[4 * i], pk16[4 * i + 1], pk16[4 * i + 2], pk16[4 * i + 3]);
            ++nb;
          } else {
            store_tile_chunk(g, m, oc, v);
          }
        }
        if (!ok) break;
        tc_fence_before();
        mbar_arrive_remote(tempty0 + acc * 8);
      }
      if ((tma_out || acc_in) && lane == 0) bulk_wait_all();
      __syncwarp();
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while its pair may still touch its shared memory
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::TMEM_COLS);
  }
}

template <bool A_MN, bool B_MN>
cudaError_t run2(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to, const GemmArgs& args,
                 cudaStream_t st) {
  auto kern = gemm2_kernel<A_MN, B_MN>;
  // the kernel needs more than the default 48 KB of dynamic shared memory;
  // the limit is raised once per device
  if (const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), Cfg2::SMEM); e != cudaSuccess)
    return e;
  const int tiles = args.m_tiles * args.n_tiles * args.split_k;
  const int pairs = std::min(tiles, num_sms() / 2);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = Cfg2::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, ta, tb, to, args);
}

template <int BN, bool A_MN, bool B_MN>
cudaError_t run(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& args, cudaStream_t st) {
  auto kern = gemm_kernel<BN, A_MN, B_MN>;
  // the kernel needs more than the default 48 KB of dynamic shared memory;
  // the limit is raised once per device
  if (const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), Cfg<BN>::SMEM); e != cudaSuccess)
    return e;
  const int tiles = args.m_tiles * args.n_tiles * args.split_k;
  const int grid = std::min(tiles, num_sms());
  kern<<<grid, 256, Cfg<BN>::SMEM, st>>>(ta, tb, args);
  return cudaGetLastError();
}

template <int BN>
cudaError_t dispatch_major(const GemmDesc& d, const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a,
                           cudaStream_t st) {
  if (d.a_mn && d.b_mn) return run<BN, true, true>(ta, tb, a, st);
  if (d.a_mn) return run<BN, true, false>(ta, tb, a, st);
  if (d.b_mn) return run<BN, false, true>(ta, tb, a, st);
  return run<BN, false, false>(ta, tb, a, st);
}

void copy_map(const BlockMap& m, int& use, uint16_t* dst) {
  use = m.n > 0;
  for (int i = 0; i < m.n && i < kMaxMap; ++i) dst[i] = m.idx[i];
}

}  // namespace

cudaError_t launch_gemm(const GemmDesc& d, int* status, cudaStream_t st) {
  if (d.M % 64 || d.K % BK || d.N % 64 || d.M <= 0 || d.N <= 0 || d.K <= 0) return cudaErrorInvalidValue;
  if (d.split_k < 1 || d.K / BK < d.split_k || (d.split_k > 1 && d.out_mode != kOutF32Red))
    return cudaErrorInvalidValue;
  // a gather map names every 64-wide block of its dimension
  auto map_ok = [](const BlockMap& m, int blocks) { return m.n == 0 || (m.n == blocks && blocks <= kMaxMap); };
  if (!map_ok(d.amap_k, d.K / BK) || !map_ok(d.bmap_k, d.K / BK) || !map_ok(d.bmap_n, d.N / 64) ||
      !map_ok(d.omap_n, d.N / 64))
    return cudaErrorInvalidValue;
  const int BN = (d.N % 256 == 0) ? 256 : (d.N % 128 == 0 ? 128 : 64);
  CUtensorMap ta, tb;
  if (!make_tmap_bf16(&ta, d.A, d.a_cols, d.a_rows, d.lda, 64, 64)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, d.B, d.b_cols, d.b_rows, d.ldb, 64, 64)) return cudaErrorInvalidValue;
  GemmArgs a;
  a.M = d.M; a.N = d.N; a.K = d.K;
  a.m_tiles = (d.M + BM - 1) / BM;  // a last tile of 64 rows reads zeros past M
  a.n_tiles = d.N / BN;
  a.split_k = d.split_k;
  copy_map(d.amap_k, a.use_amap_k, a.amap_k);
  copy_map(d.bmap_k, a.use_bmap_k, a.bmap_k);
  copy_map(d.bmap_n, a.use_bmap_n, a.bmap_n);
  copy_map(d.omap_n, a.use_omap_n, a.omap_n);
  a.out = d.out; a.ldo = d.ldo; a.out_mode = d.out_mode;
  // accumulating outputs of K >= 1536 read the old values and store the sums
  // (the main loop of a tile is long enough to hide the reads); shorter K
  // adds through TMA reduce-adds (W_o at K = 1024: 241 against 256 us; dX at
  // K = 1536: 276 against 302 us)
  a.acc_load = d.out_mode == kOutF32Acc && d.K >= 1536;
  a.aux = d.aux; a.ld_aux = d.ld_aux;
  a.status = status;
  if (BN == 256 && d.M % 256 == 0 && num_sms() >= 2) {
    a.m_tiles = d.M / 256;  // pair tiles of 256 x 256
    // fp32 outputs: a map over the whole output buffer, 32 x 32 boxes
    CUtensorMap to = ta;
    if ((d.out_mode == kOutF32 || d.out_mode == kOutF32Acc || d.out_mode == kOutF32Red) &&
        !make_tmap_f32(&to, d.out, d.ldo, d.M, d.ldo, 32, 32))
      return cudaErrorInvalidValue;
    // bf16 = acc + aux: the map reads the fp32 aux in 32 x 32 boxes
    if (d.out_mode == kOutBf16PlusF32 && !make_tmap_f32(&to, d.aux, d.ld_aux, d.M, d.ld_aux, 32, 32))
      return cudaErrorInvalidValue;
    if (d.a_mn && d.b_mn) return run2<true, true>(ta, tb, to, a, st);
    if (d.a_mn) return run2<true, false>(ta, tb, to, a, st);
    if (d.b_mn) return run2<false, true>(ta, tb, to, a, st);
    return run2<false, false>(ta, tb, to, a, st);
  }
  if (BN == 256) return dispatch_major<256>(d, ta, tb, a, st);
  if (BN == 128) return dispatch_major<128>(d, ta, tb, a, st);
  return dispatch_major<64>(d, ta, tb, a, st);
}

}  // namespace upipe
