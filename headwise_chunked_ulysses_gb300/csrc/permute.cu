// The Ulysses all-to-all of C virtual ranks on one GPU, as an HBM permute.
//
// "Untied Ulysses" summary, Background (DeepSpeed Ulysses) and Method steps
// (2) and (4): before attention each rank holds S/C tokens of every head of
// the stage and needs all S tokens of U/C heads; afterwards the outputs go
// back.  With the C ranks' buffers side by side in one GPU's memory, the
// exchange is the index map
//     seq layout  [S tokens][heads][d]    (rank c owns tokens cS/C..(c+1)S/C-1)
//     head layout [slot][S tokens][d]     (rank c owns a run of slots)
// and every byte moves once.  Each thread copies one 16-byte vector (8 bf16),
// consecutive threads walk along d then along tokens, so both the reads and
// the writes are full, coalesced 128-byte lines.
//
// head2seq can sum several source slots into one output head (the copies of
// a KV head's gradient held by different ranks), in fp32, in the listed
// order starting from the first source, then rounds once to bf16 (round to
// nearest even).  A single bf16 source is moved bit for bit.
#include <algorithm>

#include "ptx.cuh"
#include "upipe_internal.h"

namespace upipe {
namespace {

__global__ void seq2head_kernel(const Seq2HeadDesc p) {
  const int vpr = p.D / 8;  // 16-byte vectors per head row
  const long long total = static_cast<long long>(p.n_slots) * p.S * vpr;
  for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < total;
       g += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int v = static_cast<int>(g % vpr);
    const long long rest = g / vpr;
    const int t = static_cast<int>(rest % p.S);
    const int k = static_cast<int>(rest / p.S);
    const uint4 x =
        *reinterpret_cast<const uint4*>(p.src + t * p.ld_src + static_cast<long long>(p.src_head[k]) * p.D + v * 8);
    *reinterpret_cast<uint4*>(p.dst + g * 8) = x;
  }
}

template <bool F32>
__global__ void head2seq_kernel(const Head2SeqDesc p) {
  const int vpr = p.D / 8;
  const long long total = static_cast<long long>(p.n_heads) * p.S * vpr;
  for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < total;
       g += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int v = static_cast<int>(g % vpr);
    const long long rest = g / vpr;
    const int t = static_cast<int>(rest % p.S);
    const int k = static_cast<int>(rest / p.S);
    uint4* out = reinterpret_cast<uint4*>(p.dst + t * p.ld_dst + static_cast<long long>(p.dst_head[k]) * p.D + v * 8);
    const int r0 = p.first[k], r1 = p.first[k + 1];
    if (!F32 && r1 - r0 == 1) {  // a plain move: copy the bits
      *out = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.src) +
                                             (static_cast<long long>(p.src_slot[r0]) * p.S + t) * p.D + v * 8);
      continue;
    }
    float f[8];
    for (int r = r0; r < r1; ++r) {
      const long long off = (static_cast<long long>(p.src_slot[r]) * p.S + t) * p.D + v * 8;
      float x[8];
      if (F32) {
        const float4* s = reinterpret_cast<const float4*>(static_cast<const float*>(p.src) + off);
        const float4 a = s[0], b = s[1];
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
      } else {
        const uint4 a = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.src) + off);
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          x[2 * i] = bf16_lo(w[i]);
          x[2 * i + 1] = bf16_hi(w[i]);
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = (r == r0) ? x[i] : f[i] + x[i];
    }
    *out = make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
  }
}

unsigned grid_for(long long work, int threads) {
  const long long want = (work + threads - 1) / threads;
  const long long cap = static_cast<long long>(num_sms()) * 16;
  return static_cast<unsigned>(std::max(1LL, std::min(want, cap)));
}

// Sequence layout bf16 -> head layout E4M3 codes with per-row or per-128-row
// fp32 scales (lower-precision heads; "Untied Ulysses" summary, weaknesses
// from an independent analysis).  One CTA per (slot, 128 rows); each thread
// holds its 16-byte vectors in registers between the amax and the encoding.
// scale = amax / 448 (IEEE division; 1 for an all-zero group), code =
// E4M3(x / scale), round to nearest even, saturating.
template <int D>
__global__ void __launch_bounds__(256) quant_e4m3_kernel(const QuantDesc p) {
  constexpr int VPR = D / 8;               // vectors per row
  constexpr int NV = 128 * VPR / 256;      // vectors per thread
  const int blocks = p.S / 128;
  const int blk = static_cast<int>(blockIdx.x) % blocks;
  const int k = static_cast<int>(blockIdx.x) / blocks;
  __shared__ float red[8];
  uint4 x[NV];
  float am[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int idx = threadIdx.x + i * 256;
    const int row = blk * 128 + idx / VPR, v = idx % VPR;
    x[i] = *reinterpret_cast<const uint4*>(p.src + row * p.ld_src + static_cast<long long>(p.src_head[k]) * D + v * 8);
    const uint32_t w[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
    float m = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[e])), fabsf(bf16_hi(w[e]))));
    am[i] = m;
  }
  float sc[NV];
  if (p.per_row) {
    // the VPR lanes of a row are consecutive lanes of one warp
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      float m = am[i];
#pragma unroll
      for (int off = VPR / 2; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      sc[i] = m > 0.f ? __fdiv_rn(m, 448.f) : 1.f;
      const int idx = threadIdx.x + i * 256;
      if (idx % VPR == 0) p.scale[static_cast<long long>(k) * p.S + blk * 128 + idx / VPR] = sc[i];
    }
  } else {
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) m = fmaxf(m, am[i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int wi = 1; wi < 8; ++wi) m = fmaxf(m, red[wi]);
    const float s = m > 0.f ? __fdiv_rn(m, 448.f) : 1.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) sc[i] = s;
    if (threadIdx.x == 0) p.scale[static_cast<long long>(k) * blocks + blk] = s;
  }
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int idx = threadIdx.x + i * 256;
    const int row = blk * 128 + idx / VPR, v = idx % VPR;
    const uint32_t w[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
    uint32_t o[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t lo = cvt_e4m3x2(__fdiv_rn(bf16_lo(w[2 * h]), sc[i]), __fdiv_rn(bf16_hi(w[2 * h]), sc[i]));
      const uint32_t hi =
          cvt_e4m3x2(__fdiv_rn(bf16_lo(w[2 * h + 1]), sc[i]), __fdiv_rn(bf16_hi(w[2 * h + 1]), sc[i]));
      o[h] = lo | (hi << 16);
    }
    *reinterpret_cast<uint2*>(p.dst + (static_cast<long long>(k) * p.S + row) * D + v * 8) = make_uint2(o[0], o[1]);
  }
}

}  // namespace

cudaError_t launch_seq2head(const Seq2HeadDesc& p, cudaStream_t st) {
  if (p.D % 8 || p.n_slots <= 0 || p.n_slots > kMaxSlots || p.S <= 0) return cudaErrorInvalidValue;
  const long long work = static_cast<long long>(p.n_slots) * p.S * (p.D / 8);
  seq2head_kernel<<<grid_for(work, 256), 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_head2seq(const Head2SeqDesc& p, cudaStream_t st) {
  if (p.D % 8 || p.n_heads <= 0 || p.n_heads > kMaxSlots || p.S <= 0) return cudaErrorInvalidValue;
  const long long work = static_cast<long long>(p.n_heads) * p.S * (p.D / 8);
  if (p.src_f32) head2seq_kernel<true><<<grid_for(work, 256), 256, 0, st>>>(p);
  else head2seq_kernel<false><<<grid_for(work, 256), 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_quant_e4m3(const QuantDesc& p, cudaStream_t st) {
  if ((p.D != 64 && p.D != 128) || p.S <= 0 || p.S % 128 || p.n_slots <= 0 || p.n_slots > kMaxSlots || !p.src ||
      !p.dst || !p.scale)
    return cudaErrorInvalidValue;
  const unsigned grid = static_cast<unsigned>(p.n_slots) * (p.S / 128);
  if (p.D == 128)
    quant_e4m3_kernel<128><<<grid, 256, 0, st>>>(p);
  else
    quant_e4m3_kernel<64><<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace upipe
