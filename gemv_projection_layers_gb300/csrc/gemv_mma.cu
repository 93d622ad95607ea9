// gemv_mma.cu -- the bf16 layers at 3..8 tokens: a weight-streaming GEMV
// whose multiply-adds run on the warp-level tensor-core MMA.
//
// out[i, n] = sum_k x[i, k] W[n, k]            (muse_bf16_proj guide, ch. 1, §1.1)
//
// At a few tokens the layer is still a weight stream; what it adds over the
// one-token GEMV is m products per weight, too many for the CUDA cores'
// mixed-precision FMA at the stream's rate (the pooler at m = 8 would need
// half their peak) and too few to fill a tcgen05 tile.  This is the pages'
// GEMV design (muse_bf16_proj project report, "What was built": 16-row
// blocks, warps splitting K, mma.sync, weights straight to registers) on
// GB300:
//
// * W is prepacked (lossless) into 16 x 16 tiles in the A-fragment order of
//   mma.sync m16n8k16, so one 16-byte load per lane -- 512 contiguous bytes
//   per warp -- is one tile's fragment, straight into registers.
// * CTA c owns the 16-row blocks [c NB / G, (c + 1) NB / G) (whole blocks:
//   nothing crosses CTAs).  Its sixteen warps split the blocks' k-tiles into
//   contiguous runs (a warp changes block at most once, so one accumulator
//   tile suffices), two batches of eight fragments in flight per warp.
// * x (up to 8 tokens) is staged once into shared memory in B-fragment
//   order (8 bytes per lane per k-tile), after the dependency wait, while
//   the first batch of weights is in flight.
// * Each warp accumulates a 16 x 8 fp32 tile per row block in registers;
//   the sixteen warps' tiles are summed in warp order (deterministic) and
//   rounded to bf16.
// Products are exact and accumulate in fp32 on the tensor cores.
//
// The 12-bit form reads the fragment-order copy recoded as 12-bit records
// (four consecutive fragment tiles of a block per 1536-byte record, the
// row-chunk record layout of kernels.h applied to the fragment stream, so
// that a lane's decoded words are exactly its four A fragments), decodes
// them in registers with the same byte permutes as the register GEMV,
// restores the escapes, and runs the same MMAs in the same order: its
// outputs are bit-identical to the dense form at the same partition.  Warps
// then take runs of whole records (four k-tiles).
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace proj {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kU = 8;  // fragments per batch per warp
// Shared memory for NT tiles of 8 tokens: x in B-fragment order (K / 16
// k-tiles x NT x 256 B) and the warps' partial tiles ([warp][block][NT][lane][4]).
constexpr int red_bytes(int nt) { return kWarps * kGemvMmaMaxBlocks * nt * 32 * 4 * 4; }
constexpr int smem_bytes(int nt, int K) { return K / 16 * nt * 256 + red_bytes(nt); }
constexpr int kSmemLimit = 227 * 1024;

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ld_shared_u2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_shared_f32x4(uint32_t addr, float a, float b, float c,
                                                float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

// Shared-memory slot of B-fragment word w of lane l for k-tile kt: each
// k-tile's 32 lanes x 8 bytes form one 256-byte block, lanes permuted by
// l ^ 2 (kt % 16) so that the staging stores (consecutive k-tiles per warp)
// spread over the banks; the MMA loads (one k-tile per warp) stay
// conflict-free.
__device__ __forceinline__ uint32_t xfrag_off(int kt, int l, int w) {
  return static_cast<uint32_t>(kt * 256 + ((l ^ ((kt & 15) << 1)) << 3) + w * 4);
}

// d += A (16 x 16, bf16, row) * B (16 x 8, bf16, col), fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint4& a, const uint2& b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y));
}

__device__ __forceinline__ uint32_t ldg_stream_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// Lane l's four fragments of a 12-bit record: low-byte words lo[0..1],
// nibble word nb, escape word e (lane l holds word l % 8 of the block).
__device__ __forceinline__ void decode_frag12(const uint4 (&r)[3], uint32_t e, uint32_t e0x4,
                                              int lane, uint4 (&a)[4]) {
  uint32_t pw[16];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t lo0 = (j & 1) ? r[j >> 1].z : r[j >> 1].x;
    const uint32_t lo1 = (j & 1) ? r[j >> 1].w : r[j >> 1].y;
    const uint32_t nb = j == 0 ? r[2].x : (j == 1 ? r[2].y : (j == 2 ? r[2].z : r[2].w));
    const uint32_t hl = ((nb & 0x07070707u) + e0x4) | ((nb << 4) & 0x80808080u);
    const uint32_t hh = (((nb >> 4) & 0x07070707u) + e0x4) | (nb & 0x80808080u);
    pw[4 * j + 0] = __byte_perm(lo0, hl, 0x5140);
    pw[4 * j + 1] = __byte_perm(lo0, hl, 0x7362);
    pw[4 * j + 2] = __byte_perm(lo1, hh, 0x5140);
    pw[4 * j + 3] = __byte_perm(lo1, hh, 0x7362);
  }
  const uint32_t cnt = min(__shfl_sync(0xffffffffu, e, 0), static_cast<uint32_t>(kRc12EscCap));
  for (uint32_t k = 0; k < cnt; ++k) {  // warp-uniform
    const uint32_t ent = __shfl_sync(0xffffffffu, e, static_cast<int>(1 + k));
    const uint32_t pos = ent >> 8;  // 256 (tile) + 8 (lane) + element
    if (static_cast<int>((pos >> 3) & 31) == lane) {
      const uint32_t wi = (pos >> 8) * 4 + ((pos >> 1) & 3);
      const uint32_t sel = (pos & 1) ? 0x4210u : 0x3240u;
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (static_cast<uint32_t>(i) == wi) pw[i] = __byte_perm(pw[i], ent, sel);
    }
  }
#pragma unroll
  for (int t = 0; t < 4; ++t) a[t] = make_uint4(pw[4 * t], pw[4 * t + 1], pw[4 * t + 2], pw[4 * t + 3]);
}

template <int NT, bool kX12>
__global__ void __launch_bounds__(kThreads, 1) gemv_mma_kernel(const GemvMmaParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  // [K/16 k-tiles][NT][32 lanes][2 words], fragment (kt, nt) at xfrag_off(kt NT + nt, ...)
  const uint32_t sX = smem_u32(smem_raw);
  const uint32_t sRed = sX + static_cast<uint32_t>(p.K / 16 * NT * 256);  // [warp][block][NT][lane][4]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int KT = p.K / 16;
  const int NB = p.n_rows / 16;
  const int b0 = static_cast<int>(static_cast<uint32_t>(blockIdx.x) * NB / p.G);
  const int b1 = static_cast<int>((static_cast<uint32_t>(blockIdx.x) + 1u) * NB / p.G);
  const int nu = (b1 - b0) * KT;  // units (block, k-tile) of this CTA, block-major
  // Warp w takes the contiguous units [u0, u1): consecutive k-tiles (4 KB
  // contiguous per batch), at most one block change on the way; whole
  // records of four k-tiles in the 12-bit form (KT is a multiple of 16).
  constexpr int kGran = kX12 ? 4 : 1;
  const int u0 = kGran * static_cast<int>(static_cast<uint32_t>(warp) * (nu / kGran) / kWarps);
  const int u1 = kGran * static_cast<int>(static_cast<uint32_t>(warp + 1) * (nu / kGran) / kWarps);
  // unit u: block b0 + u / KT, k-tile u % KT; its fragment for this lane
  const uint4* W = p.w + static_cast<size_t>(b0) * KT * 32 + lane;

  // The 12-bit records of this CTA's first unit onwards: record r covers
  // units 4 r .. 4 r + 3.
  const uint8_t* R = kX12 ? p.rec + static_cast<size_t>(b0) * KT / 4 * kRc12Bytes : nullptr;
  const uint32_t* E = kX12 ? p.esc + static_cast<size_t>(b0) * KT / 4 * kRc12EscWords : nullptr;
  auto load_batch = [&](int base, uint4 (&a)[kU]) {
    if constexpr (kX12) {
      // kU / 4 records: a[3 g .. 3 g + 2] their three 16-byte words, the
      // escape word in a[6 + g].x
#pragma unroll
      for (int g = 0; g < kU / 4; ++g) {
        const int u = base + 4 * g;
        if (u < u1) {
          const uint8_t* src = R + static_cast<size_t>(u / 4) * kRc12Bytes;
          a[3 * g + 0] = ldg_stream(reinterpret_cast<const uint4*>(src) + lane);
          a[3 * g + 1] = ldg_stream(reinterpret_cast<const uint4*>(src) + lane + 32);
          a[3 * g + 2] = ldg_stream(reinterpret_cast<const uint4*>(src + kRc12Chunk) + lane);
          a[6 + g].x = ldg_stream_u32(E + static_cast<size_t>(u / 4) * kRc12EscWords + (lane & 7));
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const int u = base + j;
        if (u < u1) a[j] = ldg_stream(W + static_cast<size_t>(u) * 32);
      }
    }
  };
  auto red_at = [&](int w, int q, int nt, int l) {
    return sRed + static_cast<uint32_t>((((w * kGemvMmaMaxBlocks + q) * NT + nt) * 32 + l) * 16);
  };
  // Partial tiles, zero where a warp has no unit of a block.
#pragma unroll
  for (int q = 0; q < kGemvMmaMaxBlocks; ++q)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) st_shared_f32x4(red_at(warp, q, nt, lane), 0.f, 0.f, 0.f, 0.f);
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  int cur = u0 / KT;  // block of the accumulator (local index)
  auto flush = [&]() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      st_shared_f32x4(red_at(warp, cur, nt, lane), acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
  };
  // One unit's MMAs (block change handled first).
  auto mma_unit = [&](int u, const uint4& frag) {
    const int bl = u / KT;
    const int kt = u - bl * KT;
    if (bl != cur) {  // warp-uniform; at most once per warp
      flush();
      cur = bl;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const uint2 b = ld_shared_u2(sX + xfrag_off(kt * NT + nt, lane, 0));
      mma16816(acc[nt], frag, b);
    }
  };
  auto compute_batch = [&](int base, const uint4 (&a)[kU]) {
    if constexpr (kX12) {
      // record by record: decode its four fragments, then their MMAs
#pragma unroll
      for (int g = 0; g < kU / 4; ++g) {
        if (base + 4 * g >= u1) break;
        const uint4 r[3] = {a[3 * g], a[3 * g + 1], a[3 * g + 2]};
        uint4 d[4];
        decode_frag12(r, a[6 + g].x, p.e0x4, lane, d);
#pragma unroll
        for (int t = 0; t < 4; ++t) mma_unit(base + 4 * g + t, d[t]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const int u = base + j;
        if (u >= u1) break;
        mma_unit(u, a[j]);
      }
    }
  };

  // The first batch of weights streams before the wait on the previous
  // kernel of the stream (weights are constant); x comes after it.
  uint4 wa[kU], wb[kU];
  int base = u0;
  load_batch(base, wa);
  griddep_launch_dependents();
  griddep_wait();
  {
    // x -> B fragments: 16-byte chunk (token n < m, k 8 h .. 8 h + 7) of
    // k-tile kt = h / 2 feeds lanes 4 n + q (q < 4), word h % 2 (k pairs 2 q,
    // 2 q + 1 of the tile's low or high eight).  Tokens n >= m are not staged:
    // their B columns only reach output columns that are never stored.
    // Eight loads in flight per thread per round.
    const int n8 = p.m * (p.K / 8);
    for (int r0 = 0; r0 < n8; r0 += 8 * kThreads) {
      uint4 xv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = r0 + threadIdx.x + j * kThreads;
        if (i < n8)
          xv[j] = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.x) +
                                                  static_cast<size_t>(i) * 8);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = r0 + threadIdx.x + j * kThreads;
        if (i >= n8) break;
        const int n = i / (p.K / 8);
        const int h = i - n * (p.K / 8);  // 16-byte chunk within the row
        const int f = (h >> 1) * NT + (n >> 3);  // fragment (k-tile, token tile)
        const int l4 = 4 * (n & 7);
        st_shared_u32(sX + xfrag_off(f, l4 + 0, h & 1), xv[j].x);
        st_shared_u32(sX + xfrag_off(f, l4 + 1, h & 1), xv[j].y);
        st_shared_u32(sX + xfrag_off(f, l4 + 2, h & 1), xv[j].z);
        st_shared_u32(sX + xfrag_off(f, l4 + 3, h & 1), xv[j].w);
      }
    }
  }
  __syncthreads();
  // two batches in flight: the next batch's loads go out before this one
  // is multiplied
  while (base < u1) {
    if (base + kU < u1) load_batch(base + kU, wb);
    compute_batch(base, wa);
    base += kU;
    if (base >= u1) break;
    if (base + kU < u1) load_batch(base + kU, wa);
    compute_batch(base, wb);
    base += kU;
  }
  if (u0 < u1) flush();
  __syncthreads();
  // Each (block, row, token) summed over the warps' partial tiles in warp
  // order.
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
  for (int idx = threadIdx.x; idx < (b1 - b0) * NT * 128; idx += kThreads) {
    const int q = idx / (NT * 128);   // block
    const int nt = (idx / 128) % NT;  // token tile
    const int l = (idx / 4) % 32;     // fragment lane
    const int e = idx % 4;            // fragment element
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += ld_shared_f32(red_at(w, q, nt, l) + e * 4);
    // element e of lane l: row l / 4 (+ 8 for e >= 2), token 2 (l % 4) + e % 2
    const int row = (l >> 2) + (e >= 2 ? 8 : 0);
    const int tok = nt * 8 + 2 * (l & 3) + (e & 1);
    if (tok < p.m)
      out[static_cast<size_t>(tok) * p.n_rows + (b0 + q) * 16 + row] = __float2bfloat16_rn(s);
  }
}


template <int NT>
cudaError_t set_attr() {
  cudaError_t e = cudaFuncSetAttribute(gemv_mma_kernel<NT, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(gemv_mma_kernel<NT, true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
}

template <int NT, bool kX12>
cudaError_t launch(const GemvMmaParams& p, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = gemv_mma_smem(NT, p.K);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_mma_kernel<NT, kX12>, p);
}

}  // namespace

int gemv_mma_smem(int nt, int K) { return smem_bytes(nt, K); }

bool gemv_mma_fits(int nt, int K) { return smem_bytes(nt, K) <= kSmemLimit; }

cudaError_t gemv_mma_init_attributes() {
  cudaError_t e;
  if ((e = set_attr<1>()) != cudaSuccess) return e;
  if ((e = set_attr<2>()) != cudaSuccess) return e;
  return set_attr<4>();
}

cudaError_t gemv_mma_launch(int nt, bool x12, const GemvMmaParams& p, cudaStream_t s) {
  switch (nt) {
    case 1: return x12 ? launch<1, true>(p, s) : launch<1, false>(p, s);
    case 2: return x12 ? launch<2, true>(p, s) : launch<2, false>(p, s);
    case 4: return x12 ? launch<4, true>(p, s) : launch<4, false>(p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace proj
