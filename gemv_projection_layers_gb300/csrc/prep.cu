// prep.cu -- prepare-time (untimed) weight transforms, all lossless:
//   * bf16 W -> 128 x 64 tiles in the swizzled shared-memory image (and back);
//   * histogram of the 7 high exponent bits, and the 12-bit exponent-window
//     encoder/decoder (muse_bf16_proj project report, "Round 5 -- lossless
//     12-bit compressed weights", "Format");
//   * router fp32 W -> 128 x 64 swizzled tiles for the FMA kernel (and back);
//   * router fp32 W -> three bf16 planes hi + mid + lo == W (exact), packed as
//     bf16 tiles of a [N, 3K] matrix whose column p K + k holds plane p of
//     W[:, k] (and back, summing the planes).
//   * bf16 W -> 16 x 16 tiles in the A-fragment order of the m16n8k16
//     warp MMA, for the few-token GEMV (and back);
//   * bf16 W -> 12-bit row-chunk records (same window, nibbles and escapes as
//     the tile records) for the register GEMV (and back).
// The tile and record layouts are defined in kernels.h.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace proj {
namespace {

__device__ __forceinline__ size_t tile_chunk_offset(int r, int c) {
  return static_cast<size_t>(r) * 128 + (static_cast<size_t>(c ^ (r & 7)) << 4);
}

// One thread per 16-byte chunk (8 bf16) of W.
__global__ void pack_bf16_kernel(const uint16_t* __restrict__ W, int N, int K,
                                 uint8_t* __restrict__ dst) {
  const int64_t chunks = static_cast<int64_t>(N) * (K / 8);
  const int KB = K / kTileK;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < chunks;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int n = static_cast<int>(i / (K / 8));
    const int k8 = static_cast<int>(i % (K / 8));
    const int t = n / kTileRows, r = n % kTileRows;
    const int kb = k8 / 8, c = k8 % 8;
    const uint4 v = *reinterpret_cast<const uint4*>(W + static_cast<size_t>(n) * K + k8 * 8);
    uint8_t* tile = dst + (static_cast<size_t>(t) * KB + kb) * kTileBytes;
    *reinterpret_cast<uint4*>(tile + tile_chunk_offset(r, c)) = v;
  }
}

__global__ void unpack_bf16_kernel(const uint8_t* __restrict__ src, int N, int K,
                                   uint16_t* __restrict__ W) {
  const int64_t chunks = static_cast<int64_t>(N) * (K / 8);
  const int KB = K / kTileK;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < chunks;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int n = static_cast<int>(i / (K / 8));
    const int k8 = static_cast<int>(i % (K / 8));
    const int t = n / kTileRows, r = n % kTileRows;
    const int kb = k8 / 8, c = k8 % 8;
    const uint8_t* tile = src + (static_cast<size_t>(t) * KB + kb) * kTileBytes;
    *reinterpret_cast<uint4*>(W + static_cast<size_t>(n) * K + k8 * 8) =
        *reinterpret_cast<const uint4*>(tile + tile_chunk_offset(r, c));
  }
}

__global__ void high7_hist_kernel(const uint16_t* __restrict__ W, int64_t n,
                                  uint32_t* __restrict__ hist) {
  __shared__ uint32_t h[128];
  for (int i = threadIdx.x; i < 128; i += blockDim.x) h[i] = 0;
  __syncthreads();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    atomicAdd(&h[(W[i] >> 8) & 0x7F], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 128; i += blockDim.x)
    if (h[i]) atomicAdd(&hist[i], h[i]);
}

// One thread per chunk of 8 weights.  The record's escape block must be
// zeroed before the launch (its count is accumulated atomically).
__global__ void encode_expwin12_kernel(const uint16_t* __restrict__ W, int N, int K, int e0,
                                       uint8_t* __restrict__ dst, uint32_t* overflow,
                                       unsigned long long* n_esc) {
  const int64_t chunks = static_cast<int64_t>(N) * (K / 8);
  const int KB = K / kTileK;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < chunks;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int n = static_cast<int>(i / (K / 8));
    const int k8 = static_cast<int>(i % (K / 8));
    const int t = n / kTileRows, r = n % kTileRows;
    const int kb = k8 / 8, c = k8 % 8;
    const uint4 v = *reinterpret_cast<const uint4*>(W + static_cast<size_t>(n) * K + k8 * 8);
    const uint16_t w[8] = {
        static_cast<uint16_t>(v.x & 0xFFFF), static_cast<uint16_t>(v.x >> 16),
        static_cast<uint16_t>(v.y & 0xFFFF), static_cast<uint16_t>(v.y >> 16),
        static_cast<uint16_t>(v.z & 0xFFFF), static_cast<uint16_t>(v.z >> 16),
        static_cast<uint16_t>(v.w & 0xFFFF), static_cast<uint16_t>(v.w >> 16)};
    uint8_t* rec = dst + (static_cast<size_t>(t) * KB + kb) * kRecBytes;
    const int ch = r * 8 + c;
    uint32_t lo0 = 0, lo1 = 0, nb = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t b = w[j];
      const uint32_t lo = b & 0xFF;
      const int h7 = static_cast<int>((b >> 8) & 0x7F);
      const uint32_t sgn = b >> 15;
      int code = h7 - e0;
      const bool esc = code < 0 || code > 7;
      code = code < 0 ? 0 : (code > 7 ? 7 : code);
      const uint32_t nib = (sgn << 3) | static_cast<uint32_t>(code);
      if (j < 4) {
        lo0 |= lo << (8 * j);
        nb |= nib << (8 * j);
      } else {
        lo1 |= lo << (8 * (j - 4));
        nb |= nib << (8 * (j - 4) + 4);
      }
      if (esc) {
        uint32_t* blk = reinterpret_cast<uint32_t*>(rec + kRecEscOff);
        const uint32_t slot = atomicAdd(blk, 1u);
        atomicAdd(n_esc, 1ull);
        if (slot < static_cast<uint32_t>(kEscCap)) {
          const uint32_t pos = static_cast<uint32_t>(r * 64 + c * 8 + j);
          blk[1 + slot] = (pos << 8) | (b >> 8);
        } else {
          atomicOr(overflow, 1u);
        }
      }
    }
    *reinterpret_cast<uint2*>(rec + kRecLowOff + ch * 8) = make_uint2(lo0, lo1);
    *reinterpret_cast<uint32_t*>(rec + kRecNibOff + ch * 4) = nb;
  }
}

// Decode records back to row-major bf16 (the same arithmetic the tensor-core
// kernel's decode warps run, then the escape patch).
__global__ void decode_expwin12_kernel(const uint8_t* __restrict__ src, int N, int K,
                                       uint32_t e0x4, uint16_t* __restrict__ W) {
  const int64_t chunks = static_cast<int64_t>(N) * (K / 8);
  const int KB = K / kTileK;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < chunks;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int n = static_cast<int>(i / (K / 8));
    const int k8 = static_cast<int>(i % (K / 8));
    const int t = n / kTileRows, r = n % kTileRows;
    const int kb = k8 / 8, c = k8 % 8;
    const uint8_t* rec = src + (static_cast<size_t>(t) * KB + kb) * kRecBytes;
    const int ch = r * 8 + c;
    const uint2 lo = *reinterpret_cast<const uint2*>(rec + kRecLowOff + ch * 8);
    const uint32_t nb = *reinterpret_cast<const uint32_t*>(rec + kRecNibOff + ch * 4);
    const uint32_t v0 = nb & 0x0F0F0F0Fu;
    const uint32_t v1 = (nb >> 4) & 0x0F0F0F0Fu;
    const uint32_t h0 = ((v0 & 0x07070707u) + e0x4) | ((v0 << 4) & 0x80808080u);
    const uint32_t h1 = ((v1 & 0x07070707u) + e0x4) | ((v1 << 4) & 0x80808080u);
    uint4 o;
    o.x = __byte_perm(lo.x, h0, 0x5140);
    o.y = __byte_perm(lo.x, h0, 0x7362);
    o.z = __byte_perm(lo.y, h1, 0x5140);
    o.w = __byte_perm(lo.y, h1, 0x7362);
    uint16_t w[8] = {
        static_cast<uint16_t>(o.x & 0xFFFF), static_cast<uint16_t>(o.x >> 16),
        static_cast<uint16_t>(o.y & 0xFFFF), static_cast<uint16_t>(o.y >> 16),
        static_cast<uint16_t>(o.z & 0xFFFF), static_cast<uint16_t>(o.z >> 16),
        static_cast<uint16_t>(o.w & 0xFFFF), static_cast<uint16_t>(o.w >> 16)};
    const uint32_t* esc = reinterpret_cast<const uint32_t*>(rec + kRecEscOff);
    const uint32_t cnt = min(esc[0], static_cast<uint32_t>(kEscCap));
    for (uint32_t e = 0; e < cnt; ++e) {
      const uint32_t ent = esc[1 + e];
      const uint32_t pos = ent >> 8;
      if (static_cast<int>(pos >> 6) == r && static_cast<int>((pos & 63) >> 3) == c) {
        const int j = pos & 7;
        w[j] = static_cast<uint16_t>((w[j] & 0x00FF) | ((ent & 0xFF) << 8));
      }
    }
    uint4 out;
    out.x = w[0] | (static_cast<uint32_t>(w[1]) << 16);
    out.y = w[2] | (static_cast<uint32_t>(w[3]) << 16);
    out.z = w[4] | (static_cast<uint32_t>(w[5]) << 16);
    out.w = w[6] | (static_cast<uint32_t>(w[7]) << 16);
    *reinterpret_cast<uint4*>(W + static_cast<size_t>(n) * K + k8 * 8) = out;
  }
}

// Router (FMA tiles): one thread per float4 of W.
__global__ void pack_router_fma_kernel(const float* __restrict__ W, int N, int K,
                                       uint8_t* __restrict__ dst) {
  const int64_t quads = static_cast<int64_t>(N) * (K / 4);
  const int KB = K / kRfK;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < quads;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int n = static_cast<int>(i / (K / 4));
    const int k4 = static_cast<int>(i % (K / 4));
    const int t = n / kRfRows, r = n % kRfRows;
    const int kb = k4 / 16, c = k4 % 16;
    const float4 v = *reinterpret_cast<const float4*>(W + static_cast<size_t>(n) * K + k4 * 4);
    uint8_t* tile = dst + (static_cast<size_t>(t) * KB + kb) * kRfBytes;
    *reinterpret_cast<float4*>(tile + r * 256 + ((c ^ (r & 15)) << 4)) = v;
  }
}

__global__ void unpack_router_fma_kernel(const uint8_t* __restrict__ src, int N, int K,
                                         float* __restrict__ W) {
  const int64_t quads = static_cast<int64_t>(N) * (K / 4);
  const int KB = K / kRfK;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < quads;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int n = static_cast<int>(i / (K / 4));
    const int k4 = static_cast<int>(i % (K / 4));
    const int t = n / kRfRows, r = n % kRfRows;
    const int kb = k4 / 16, c = k4 % 16;
    const uint8_t* tile = src + (static_cast<size_t>(t) * KB + kb) * kRfBytes;
    *reinterpret_cast<float4*>(W + static_cast<size_t>(n) * K + k4 * 4) =
        *reinterpret_cast<const float4*>(tile + r * 256 + ((c ^ (r & 15)) << 4));
  }
}

// Exact three-way split of an fp32 value into bf16 planes: each plane is the
// round-to-nearest bf16 of what the previous ones left.  A normal fp32 value
// has 24 significant bits; each rounding to 8 bits leaves a remainder that is
// exact in fp32 and at least 8 bits shorter, so the third plane is the last
// remainder exactly (for |w| >= 2^-100; subnormal remainders are not met by
// the weights here and are still split as closely as bf16 allows).
__device__ __forceinline__ void split3(float w, uint16_t& hi, uint16_t& mid, uint16_t& lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(w);
  const float r1 = w - __bfloat162float(h);
  const __nv_bfloat16 m = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(m);
  const __nv_bfloat16 l = __float2bfloat16_rn(r2);
  hi = __bfloat16_as_ushort(h);
  mid = __bfloat16_as_ushort(m);
  lo = __bfloat16_as_ushort(l);
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// One thread per 8 consecutive weights of a row.
__global__ void pack_planes_kernel(const float* __restrict__ W, int N, int K,
                                   uint8_t* __restrict__ dst) {
  const int64_t chunks = static_cast<int64_t>(N) * (K / 8);
  const int KB = K / kTileK;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < chunks;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int n = static_cast<int>(i / (K / 8));
    const int k8 = static_cast<int>(i % (K / 8));
    const int t = n / kTileRows, r = n % kTileRows;
    const int kb = k8 / 8, c = k8 % 8;
    const float* src = W + static_cast<size_t>(n) * K + k8 * 8;
    uint16_t pl[3][8];
#pragma unroll
    for (int j = 0; j < 8; ++j) split3(src[j], pl[0][j], pl[1][j], pl[2][j]);
#pragma unroll
    for (int p = 0; p < 3; ++p) {
      uint4 v;
      v.x = pl[p][0] | (static_cast<uint32_t>(pl[p][1]) << 16);
      v.y = pl[p][2] | (static_cast<uint32_t>(pl[p][3]) << 16);
      v.z = pl[p][4] | (static_cast<uint32_t>(pl[p][5]) << 16);
      v.w = pl[p][6] | (static_cast<uint32_t>(pl[p][7]) << 16);
      uint8_t* tile = dst + (static_cast<size_t>(t) * 3 * KB + p * KB + kb) * kTileBytes;
      *reinterpret_cast<uint4*>(tile + tile_chunk_offset(r, c)) = v;
    }
  }
}

__global__ void unpack_planes_kernel(const uint8_t* __restrict__ src, int N, int K,
                                     float* __restrict__ W) {
  const int64_t chunks = static_cast<int64_t>(N) * (K / 8);
  const int KB = K / kTileK;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < chunks;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int n = static_cast<int>(i / (K / 8));
    const int k8 = static_cast<int>(i % (K / 8));
    const int t = n / kTileRows, r = n % kTileRows;
    const int kb = k8 / 8, c = k8 % 8;
    uint4 v[3];
#pragma unroll
    for (int p = 0; p < 3; ++p)
      v[p] = *reinterpret_cast<const uint4*>(
          src + (static_cast<size_t>(t) * 3 * KB + p * KB + kb) * kTileBytes +
          tile_chunk_offset(r, c));
    float* o = W + static_cast<size_t>(n) * K + k8 * 8;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t wd = j / 2, sh = (j % 2) * 16;
      auto pick = [&](const uint4& q) -> uint16_t {
        const uint32_t word = wd == 0 ? q.x : (wd == 1 ? q.y : (wd == 2 ? q.z : q.w));
        return static_cast<uint16_t>(word >> sh);
      };
      o[j] = (bf16_bits_to_float(pick(v[0])) + bf16_bits_to_float(pick(v[1]))) +
             bf16_bits_to_float(pick(v[2]));
    }
  }
}

// One thread per 16-byte fragment: tile (rb, kb) of 16 rows x 16 k at
// (rb K/16 + kb) x 512 B, lane l's four words at l x 16: rows g = l / 4 and
// g + 8, columns c = 2 (l % 4) (+1) and c + 8 (+1), as kernels.h states.
__global__ void pack_frag16_kernel(const uint16_t* __restrict__ W, int N, int K,
                                   uint32_t* __restrict__ dst) {
  const int KT = K / 16;
  const int64_t frags = static_cast<int64_t>(N / 16) * KT * 32;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < frags;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tile = i / 32;
    const int l = static_cast<int>(i % 32);
    const int rb = static_cast<int>(tile / KT), kb = static_cast<int>(tile % KT);
    const int g = l >> 2, c = (l & 3) * 2;
    const uint16_t* r0 = W + static_cast<size_t>(rb * 16 + g) * K + kb * 16 + c;
    const uint16_t* r8 = r0 + static_cast<size_t>(8) * K;
    uint4 v;
    v.x = *reinterpret_cast<const uint32_t*>(r0);
    v.y = *reinterpret_cast<const uint32_t*>(r8);
    v.z = *reinterpret_cast<const uint32_t*>(r0 + 8);
    v.w = *reinterpret_cast<const uint32_t*>(r8 + 8);
    reinterpret_cast<uint4*>(dst)[i] = v;
  }
}

__global__ void unpack_frag16_kernel(const uint32_t* __restrict__ src, int N, int K,
                                     uint16_t* __restrict__ W) {
  const int KT = K / 16;
  const int64_t frags = static_cast<int64_t>(N / 16) * KT * 32;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < frags;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tile = i / 32;
    const int l = static_cast<int>(i % 32);
    const int rb = static_cast<int>(tile / KT), kb = static_cast<int>(tile % KT);
    const int g = l >> 2, c = (l & 3) * 2;
    uint16_t* r0 = W + static_cast<size_t>(rb * 16 + g) * K + kb * 16 + c;
    uint16_t* r8 = r0 + static_cast<size_t>(8) * K;
    const uint4 v = reinterpret_cast<const uint4*>(src)[i];
    *reinterpret_cast<uint32_t*>(r0) = v.x;
    *reinterpret_cast<uint32_t*>(r8) = v.y;
    *reinterpret_cast<uint32_t*>(r0 + 8) = v.z;
    *reinterpret_cast<uint32_t*>(r8 + 8) = v.w;
  }
}

// Row-run layout of the few-token GEMV (gemv_rows.cu): CTA c of G owns rows
// [r0, r1) = [c Nr / G, (c + 1) Nr / G); its run sits at byte r0 K 2 as
// [K / 32 steps][r1 - r0 rows][32 columns].  16-byte unit (row r, columns
// 8u .. 8u + 7) of the row-major source goes to
// r0 K 2 + (u / 4) (r1 - r0) 64 + (r - r0) 64 + (u % 4) 16.
__device__ __forceinline__ size_t runs_offset(int r, int u, int Nr, int K, int G) {
  const int c = static_cast<int>(part_owner(r, Nr, G));
  const int r0 = static_cast<int>(part_begin(c, Nr, G));
  const int r1 = static_cast<int>(part_begin(c + 1, Nr, G));
  return static_cast<size_t>(r0) * K * 2 + static_cast<size_t>(u >> 2) * (r1 - r0) * 64 +
         static_cast<size_t>(r - r0) * 64 + (u & 3) * 16;
}

__global__ void pack_runs_kernel(const uint16_t* __restrict__ W, int Nr, int K, int G,
                                 uint8_t* __restrict__ dst) {
  const int U = K / 8;
  const int64_t n = static_cast<int64_t>(Nr) * U;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(i / U), u = static_cast<int>(i % U);
    *reinterpret_cast<uint4*>(dst + runs_offset(r, u, Nr, K, G)) =
        *reinterpret_cast<const uint4*>(W + static_cast<size_t>(r) * K + 8 * u);
  }
}

__global__ void unpack_runs_kernel(const uint8_t* __restrict__ src, int Nr, int K, int G,
                                   uint16_t* __restrict__ W) {
  const int U = K / 8;
  const int64_t n = static_cast<int64_t>(Nr) * U;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(i / U), u = static_cast<int>(i % U);
    *reinterpret_cast<uint4*>(W + static_cast<size_t>(r) * K + 8 * u) =
        *reinterpret_cast<const uint4*>(src + runs_offset(r, u, Nr, K, G));
  }
}

constexpr int kPrepBlock = 256;
constexpr int kPrepGrid = 152 * 8;

// Row-chunk records for the register GEMV: one warp per 1024-column chunk,
// lane l encoding its groups j = 0..3 (columns 8 (l + 32 j) .. + 7); escapes
// are numbered in column order (group, then lane, then column) by a warp
// prefix sum, so the records do not depend on scheduling.
__global__ void encode_rc12_kernel(const uint16_t* __restrict__ W, int N, int K, int e0,
                                   uint8_t* __restrict__ rec, uint32_t* __restrict__ esc,
                                   uint32_t* overflow) {
  const int lane = threadIdx.x & 31;
  const int64_t chunks = static_cast<int64_t>(N) * (K / kRc12Chunk);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  for (int64_t q = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) / 32; q < chunks;
       q += nwarps) {
    const uint16_t* src = W + q * kRc12Chunk;  // chunks are contiguous in row-major W
    uint8_t* r = rec + q * kRc12Bytes;
    uint32_t* eb = esc + q * kRc12EscWords;
    uint32_t nibw[4];
    uint32_t base = 0;  // escapes numbered so far
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = (lane + 32 * j) * 8;
      const uint4 v = *reinterpret_cast<const uint4*>(src + col);
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
      uint32_t lo0 = 0, lo1 = 0, nb = 0, emask = 0;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const uint32_t wb = (wv[b >> 1] >> (16 * (b & 1))) & 0xFFFFu;
        const int h7 = static_cast<int>((wb >> 8) & 0x7F);
        int code = h7 - e0;
        if (code < 0 || code > 7) emask |= 1u << b;
        code = code < 0 ? 0 : (code > 7 ? 7 : code);
        const uint32_t nib = ((wb >> 15) << 3) | static_cast<uint32_t>(code);
        if (b < 4) {
          lo0 |= (wb & 0xFF) << (8 * b);
          nb |= nib << (8 * b);
        } else {
          lo1 |= (wb & 0xFF) << (8 * (b - 4));
          nb |= nib << (8 * (b - 4) + 4);
        }
      }
      *reinterpret_cast<uint2*>(r + (lane + 32 * (j >> 1)) * 16 + (j & 1) * 8) =
          make_uint2(lo0, lo1);
      nibw[j] = nb;
      const uint32_t cnt = __popc(emask);
      uint32_t incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      uint32_t slot = base + incl - cnt;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        if ((emask >> b) & 1u) {
          const uint32_t wb = (wv[b >> 1] >> (16 * (b & 1))) & 0xFFFFu;
          if (slot < static_cast<uint32_t>(kRc12EscCap))
            eb[1 + slot] = (static_cast<uint32_t>(col + b) << 8) | (wb >> 8);
          ++slot;
        }
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    *reinterpret_cast<uint4*>(r + kRc12Chunk + lane * 16) =
        make_uint4(nibw[0], nibw[1], nibw[2], nibw[3]);
    if (lane == 0) {
      eb[0] = min(base, static_cast<uint32_t>(kRc12EscCap));
      if (base > static_cast<uint32_t>(kRc12EscCap)) atomicOr(overflow, 1u);
    }
  }
}

// Row-chunk records back to row-major bf16: the register GEMV's decode, then
// the escape patch.
__global__ void decode_rc12_kernel(const uint8_t* __restrict__ rec,
                                   const uint32_t* __restrict__ esc, int N, int K, uint32_t e0x4,
                                   uint16_t* __restrict__ W) {
  const int lane = threadIdx.x & 31;
  const int64_t chunks = static_cast<int64_t>(N) * (K / kRc12Chunk);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  for (int64_t q = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) / 32; q < chunks;
       q += nwarps) {
    const uint8_t* r = rec + q * kRc12Bytes;
    const uint32_t* eb = esc + q * kRc12EscWords;
    const uint4 nib = *reinterpret_cast<const uint4*>(r + kRc12Chunk + lane * 16);
    const uint32_t nibw[4] = {nib.x, nib.y, nib.z, nib.w};
    const uint32_t cnt = min(eb[0], static_cast<uint32_t>(kRc12EscCap));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = (lane + 32 * j) * 8;
      const uint2 lo = *reinterpret_cast<const uint2*>(r + (lane + 32 * (j >> 1)) * 16 + (j & 1) * 8);
      const uint32_t nb = nibw[j];
      const uint32_t hl = ((nb & 0x07070707u) + e0x4) | ((nb << 4) & 0x80808080u);
      const uint32_t hh = (((nb >> 4) & 0x07070707u) + e0x4) | (nb & 0x80808080u);
      uint32_t o[4] = {__byte_perm(lo.x, hl, 0x5140), __byte_perm(lo.x, hl, 0x7362),
                       __byte_perm(lo.y, hh, 0x5140), __byte_perm(lo.y, hh, 0x7362)};
      for (uint32_t e = 0; e < cnt; ++e) {
        const uint32_t ent = eb[1 + e];
        const int b = static_cast<int>(ent >> 8) - col;
        if (b >= 0 && b < 8) {
#pragma unroll
          for (int w = 0; w < 4; ++w)
            if (w == (b >> 1)) o[w] = __byte_perm(o[w], ent, (b & 1) ? 0x4210 : 0x3240);
        }
      }
      *reinterpret_cast<uint4*>(W + q * kRc12Chunk + col) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

}  // namespace

cudaError_t pack_bf16_tiles(const uint16_t* W, int N, int K, uint8_t* dst, cudaStream_t s) {
  pack_bf16_kernel<<<kPrepGrid, kPrepBlock, 0, s>>>(W, N, K, dst);
  return cudaGetLastError();
}

cudaError_t unpack_bf16_tiles(const uint8_t* src, int N, int K, uint16_t* W, cudaStream_t s) {
  unpack_bf16_kernel<<<kPrepGrid, kPrepBlock, 0, s>>>(src, N, K, W);
  return cudaGetLastError();
}

cudaError_t high7_histogram(const uint16_t* W, int64_t n, uint32_t* hist128, cudaStream_t s) {
  high7_hist_kernel<<<kPrepGrid, kPrepBlock, 0, s>>>(W, n, hist128);
  return cudaGetLastError();
}

cudaError_t encode_expwin12(const uint16_t* W, int N, int K, int e0, uint8_t* dst,
                            uint32_t* overflow, unsigned long long* n_esc, cudaStream_t s) {
  encode_expwin12_kernel<<<kPrepGrid, kPrepBlock, 0, s>>>(W, N, K, e0, dst, overflow, n_esc);
  return cudaGetLastError();
}

cudaError_t decode_expwin12(const uint8_t* src, int N, int K, int e0, uint16_t* W,
                            cudaStream_t s) {
  const uint32_t e0x4 = static_cast<uint32_t>(e0) * 0x01010101u;
  decode_expwin12_kernel<<<kPrepGrid, kPrepBlock, 0, s>>>(src, N, K, e0x4, W);
  return cudaGetLastError();
}

cudaError_t encode_rc12(const uint16_t* W, int N, int K, int e0, uint8_t* rec, uint32_t* esc,
                        uint32_t* overflow, cudaStream_t s) {
  encode_rc12_kernel<<<kPrepGrid, kPrepBlock, 0, s>>>(W, N, K, e0, rec, esc, overflow);
  return cudaGetLastError();
}

cudaError_t decode_rc12(const uint8_t* rec, const uint32_t* esc, int N, int K, int e0,
                        uint16_t* W, cudaStream_t s) {
  const uint32_t e0x4 = static_cast<uint32_t>(e0) * 0x01010101u;
  decode_rc12_kernel<<<kPrepGrid, kPrepBlock, 0, s>>>(rec, esc, N, K, e0x4, W);
  return cudaGetLastError();
}

cudaError_t pack_frag16(const uint16_t* W, int N, int K, uint32_t* dst, cudaStream_t s) {
  pack_frag16_kernel<<<kPrepGrid, kPrepBlock, 0, s>>>(W, N, K, dst);
  return cudaGetLastError();
}

cudaError_t unpack_frag16(const uint32_t* src, int N, int K, uint16_t* W, cudaStream_t s) {
  unpack_frag16_kernel<<<kPrepGrid, kPrepBlock, 0, s>>>(src, N, K, W);
  return cudaGetLastError();
}

cudaError_t pack_runs(const uint16_t* W, int Nr, int K, int G, uint8_t* dst, cudaStream_t s) {
  pack_runs_kernel<<<kPrepGrid, kPrepBlock, 0, s>>>(W, Nr, K, G, dst);
  return cudaGetLastError();
}

cudaError_t unpack_runs(const uint8_t* src, int Nr, int K, int G, uint16_t* W, cudaStream_t s) {
  unpack_runs_kernel<<<kPrepGrid, kPrepBlock, 0, s>>>(src, Nr, K, G, W);
  return cudaGetLastError();
}

cudaError_t pack_router_fma_tiles(const float* W, int N, int K, uint8_t* dst, cudaStream_t s) {
  pack_router_fma_kernel<<<kPrepGrid, kPrepBlock, 0, s>>>(W, N, K, dst);
  return cudaGetLastError();
}

cudaError_t pack_router_planes(const float* W, int N, int K, uint8_t* dst, cudaStream_t s) {
  pack_planes_kernel<<<kPrepGrid, kPrepBlock, 0, s>>>(W, N, K, dst);
  return cudaGetLastError();
}

cudaError_t unpack_router_planes(const uint8_t* src, int N, int K, float* W, cudaStream_t s) {
  unpack_planes_kernel<<<kPrepGrid, kPrepBlock, 0, s>>>(src, N, K, W);
  return cudaGetLastError();
}

cudaError_t unpack_router_fma_tiles(const uint8_t* src, int N, int K, float* W,
                                    cudaStream_t s) {
  unpack_router_fma_kernel<<<kPrepGrid, kPrepBlock, 0, s>>>(src, N, K, W);
  return cudaGetLastError();
}

}  // namespace proj
