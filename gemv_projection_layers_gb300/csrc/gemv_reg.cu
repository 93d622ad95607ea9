// gemv_reg.cu -- streaming GEMV for m <= 2 with the weights loaded straight
// into registers (no shared-memory ring, no producer, no mbarriers).
//
// out[i, n] = sum_k x[i, k] W[n, k]            (muse_bf16_proj guide, ch. 1, §1.1)
//
// Partition: CTA c of G owns whole rows [c N / G, (c + 1) N / G) of W
// (row-major, each row cut into 1024-element chunks), so no row is shared
// between CTAs and nothing crosses CTAs: no flags, no second pass.  (The
// register form serves the short weight streams, where a CTA's rows fit in
// one or two batches of loads, so whole-row runs cost no balance.)  Sixteen
// warps take the CTA's chunks round-robin, each chunk being 16 (bf16) or 32
// (fp32) 16-byte loads across the warp, coalesced.  A warp keeps two batches
// of chunks in flight (double-buffered registers: the next batch's loads go
// out before the current batch is multiplied), so an SM has ~128 KB of loads
// outstanding with no set-up beyond the launch.  x sits in shared memory in
// the lanes' layout.  Each chunk's lane partials are reduced by a shuffle
// tree and parked in shared memory; after a CTA barrier one thread per
// (row, token) sums the row's chunks in chunk order (deterministic) and
// stores the output.  This follows the pages' "weights straight to
// registers" GEMV (project report, "What was built"; notebook n. 47), on a
// row-chunk layout instead of 16-row blocks.  A second kernel runs the same
// partition and arithmetic on the 12-bit row-chunk records, decoding each
// lane's weights in registers.
#include <cuda_bf16.h>

#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"

namespace proj {
namespace {

constexpr int kChunk = 1024;
constexpr int kMaxKs = 8;  // chunks per row: K <= 8192
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;

template <typename WT, int MT>
struct RCfgG {
  using XT = typename std::conditional<sizeof(WT) == 2, uint16_t, float>::type;
  static constexpr int kVec = 16 / static_cast<int>(sizeof(WT));       // weights per 16 B
  static constexpr int kLd = kChunk / kVec / 32;                        // 16-B loads per lane
  static constexpr int U = sizeof(WT) == 2 ? 2 : 1;                      // chunks per batch
  static constexpr int kXBytes = MT * 8192 * static_cast<int>(sizeof(XT));  // K <= 8192
  static constexpr size_t kSmem = 64 + kXBytes + static_cast<size_t>(kGemvRegMaxChunks) * MT * 4;
};

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xFFFF0000u);
}

// acc += lo(w) * lo(x), acc2 += hi(w) * hi(x): bf16 x bf16 + fp32 with the
// exact product, one instruction per weight.
__device__ __forceinline__ void fma_bf16x2(float& acc, float& acc2, uint32_t w, uint32_t x) {
  asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
      "mov.b32 {wl, wh}, %2;\n\t"
      "mov.b32 {xl, xh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, wl, xl, %0;\n\t"
      "fma.rn.f32.bf16 %1, wh, xh, %1;\n\t}"
      : "+f"(acc), "+f"(acc2)
      : "r"(w), "r"(x));
}

// (acc, acc2) += (w0, w1) * (x0, x1) in one instruction.
__device__ __forceinline__ void fma_f32x2(float& acc, float& acc2, uint32_t w0, uint32_t w1,
                                          float x0, float x1) {
  uint64_t a = (static_cast<uint64_t>(__float_as_uint(acc2)) << 32) | __float_as_uint(acc);
  const uint64_t w = (static_cast<uint64_t>(w1) << 32) | w0;
  const uint64_t x = (static_cast<uint64_t>(__float_as_uint(x1)) << 32) | __float_as_uint(x0);
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a) : "l"(w), "l"(x));
  acc = __uint_as_float(static_cast<uint32_t>(a));
  acc2 = __uint_as_float(static_cast<uint32_t>(a >> 32));
}

template <typename WT, int MT>
__global__ void __launch_bounds__(kThreads, 1) gemv_reg_kernel(const GemvParams p) {
  using C = RCfgG<WT, MT>;
  using XT = typename C::XT;
  constexpr int U = C::U;
  constexpr int L = C::kLd;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  XT* xs = reinterpret_cast<XT*>(smem_raw);
  float* cp = reinterpret_cast<float*>(smem_raw + C::kXBytes);  // [chunk][MT]
  const uint32_t xs_a = smem_u32(xs);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ks = p.K / kChunk;
  // rows [r0, r1): n_rows * G < 2^31 (n_rows <= 65536, G <= SMs)
  const int r0 = static_cast<int>(static_cast<uint32_t>(blockIdx.x) *
                                  static_cast<uint32_t>(p.n_rows) / static_cast<uint32_t>(p.G));
  const int r1 = static_cast<int>((static_cast<uint32_t>(blockIdx.x) + 1u) *
                                  static_cast<uint32_t>(p.n_rows) / static_cast<uint32_t>(p.G));
  const int64_t q0 = static_cast<int64_t>(r0) * ks;  // first chunk of the run
  const int nq = (r1 - r0) * ks;  // <= kGemvRegMaxChunks (host-checked)
  const WT* W = static_cast<const WT*>(p.w);

  // Chunk q of the run: row r0 + q / ks, columns (q % ks) * 1024 + ...
  auto load_batch = [&](int base, uint4 (&w)[U][L]) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int q = base + u * kWarps;
      if (q < nq) {
        const WT* src = W + (q0 + q) * static_cast<int64_t>(kChunk);  // chunks are contiguous
#pragma unroll
        for (int i = 0; i < L; ++i) w[u][i] = ldg_stream(src + (lane + 32 * i) * C::kVec);
      }
    }
  };
  auto compute_batch = [&](int base, const uint4 (&w)[U][L]) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int q = base + u * kWarps;
      if (q >= nq) break;
      const int col0 = (q % ks) * kChunk;
      float a8[MT][8];
#pragma unroll
      for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int c = 0; c < 8; ++c) a8[t][c] = 0.f;
#pragma unroll
      for (int i = 0; i < L; ++i) {
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          const uint4 xv = ld_shared_u4(
              xs_a + static_cast<uint32_t>((t * p.K + col0 + (lane + 32 * i) * C::kVec) *
                                           static_cast<int>(sizeof(XT))));
          float* a = a8[t];
          if constexpr (sizeof(WT) == 2) {
            fma_bf16x2(a[(i & 1) * 4 + 0], a[(i & 1) * 4 + 1], w[u][i].x, xv.x);
            fma_bf16x2(a[(i & 1) * 4 + 2], a[(i & 1) * 4 + 3], w[u][i].y, xv.y);
            fma_bf16x2(a[(i & 1) * 4 + 0], a[(i & 1) * 4 + 1], w[u][i].z, xv.z);
            fma_bf16x2(a[(i & 1) * 4 + 2], a[(i & 1) * 4 + 3], w[u][i].w, xv.w);
          } else {
            fma_f32x2(a[(i & 3) * 2 + 0], a[(i & 3) * 2 + 1], w[u][i].x, w[u][i].y,
                      __uint_as_float(xv.x), __uint_as_float(xv.y));
            fma_f32x2(a[(i & 3) * 2 + 0], a[(i & 3) * 2 + 1], w[u][i].z, w[u][i].w,
                      __uint_as_float(xv.z), __uint_as_float(xv.w));
          }
        }
      }
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        float v = ((a8[t][0] + a8[t][1]) + (a8[t][2] + a8[t][3])) +
                  ((a8[t][4] + a8[t][5]) + (a8[t][6] + a8[t][7]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == t) cp[q * MT + t] = v;
      }
    }
  };

  // The first batch of weights streams before the wait on the previous
  // kernel of the stream (weights are constant); x and every global write
  // come after it.
  uint4 wa[U][L], wb[U][L];
  int base = warp;
  load_batch(base, wa);
  griddep_launch_dependents();
  griddep_wait();
  {
    // x -> shared memory (bf16 as is, fp32 widened for fp32 weights; rows
    // beyond m are zero).  Every load is issued before the first store, so
    // staging costs one memory round trip (x is cold after a flush).
    const uint4* xg = static_cast<const uint4*>(p.x);
    const int n8 = MT * p.K / 8;
    constexpr int kXLd = (MT * 8192 / 8 + kThreads - 1) / kThreads;
    uint4 xv[kXLd];
#pragma unroll
    for (int u = 0; u < kXLd; ++u) {
      const int i = threadIdx.x + u * kThreads;
      xv[u] = (i < n8 && i / (p.K / 8) < p.m) ? xg[i] : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kXLd; ++u) {
      const int i = threadIdx.x + u * kThreads;
      if (i >= n8) break;
      const uint4 v = xv[u];
      if constexpr (sizeof(WT) == 2) {
        reinterpret_cast<uint4*>(xs)[i] = v;
      } else {
        float4 a, b;
        bf16x2_to_f32(v.x, a.x, a.y);
        bf16x2_to_f32(v.y, a.z, a.w);
        bf16x2_to_f32(v.z, b.x, b.y);
        bf16x2_to_f32(v.w, b.z, b.w);
        reinterpret_cast<float4*>(xs)[2 * i] = a;
        reinterpret_cast<float4*>(xs)[2 * i + 1] = b;
      }
    }
  }
  __syncthreads();
  constexpr int kStride = kWarps * U;
  // two batches in flight: the next batch's loads go out before this one is
  // multiplied
  while (base < nq) {
    if (base + kStride < nq) load_batch(base + kStride, wb);
    compute_batch(base, wa);
    base += kStride;
    if (base >= nq) break;
    if (base + kStride < nq) load_batch(base + kStride, wa);
    compute_batch(base, wb);
    base += kStride;
  }
  __syncthreads();

  // Rows of the run, each summed over its chunks in chunk order.
  const uint32_t cp_a = smem_u32(cp);
  for (int idx = threadIdx.x; idx < (r1 - r0) * MT; idx += kThreads) {
    const int rr = idx / MT;
    const int t = idx - rr * MT;
    float part[kMaxKs];
#pragma unroll
    for (int c = 0; c < kMaxKs; ++c)
      part[c] = c < ks ? ld_shared_f32(cp_a + static_cast<uint32_t>(((rr * ks + c) * MT + t) * 4))
                       : 0.f;
    float v = part[0];
#pragma unroll
    for (int c = 1; c < kMaxKs; ++c)
      if (c < ks) v += part[c];
    if (t < p.m) {
      const int64_t o = static_cast<int64_t>(t) * p.n_rows + r0 + rr;
      if (p.out_f32)
        static_cast<float*>(p.out)[o] = v;
      else
        static_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(v);
    }
  }
}

__device__ __forceinline__ uint32_t ldg_stream_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// The same GEMV on 12-bit row-chunk records (bf16 weights, bf16 output):
// a chunk is three 16-byte loads per lane (two of low bytes, one of nibbles)
// and one 4-byte load of its escape block (lane l reads word l % 8).  Each
// lane rebuilds its 32 bf16 weights in registers -- high byte = sign | (e0 +
// code) from the nibble, paired with the low byte by byte permutes -- patches
// the chunk's escapes (rare: a warp-uniform branch on the count), and then
// multiplies exactly as the dense kernel does, in the same order, so the
// result is bit-identical to it (muse_bf16_proj project report, "Round 5 --
// lossless 12-bit compressed weights", on a row-chunk layout).
template <int MT>
__global__ void __launch_bounds__(kThreads, 1) gemv_reg12_kernel(const GemvParams p) {
  constexpr int U = 2;  // chunks per batch
  constexpr int kXBytes = MT * 8192 * 2;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem_raw);
  float* cp = reinterpret_cast<float*>(smem_raw + kXBytes);  // [chunk][MT]
  const uint32_t xs_a = smem_u32(xs);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ks = p.K / kChunk;
  const int r0 = static_cast<int>(static_cast<uint32_t>(blockIdx.x) *
                                  static_cast<uint32_t>(p.n_rows) / static_cast<uint32_t>(p.G));
  const int r1 = static_cast<int>((static_cast<uint32_t>(blockIdx.x) + 1u) *
                                  static_cast<uint32_t>(p.n_rows) / static_cast<uint32_t>(p.G));
  const int64_t q0 = static_cast<int64_t>(r0) * ks;
  const int nq = (r1 - r0) * ks;  // <= kGemvRegMaxChunks (host-checked)
  const uint8_t* R = static_cast<const uint8_t*>(p.w);

  auto load_batch = [&](int base, uint4 (&w)[U][3], uint32_t (&e)[U]) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int q = base + u * kWarps;
      if (q < nq) {
        const uint8_t* src = R + (q0 + q) * static_cast<int64_t>(kRc12Bytes);
        w[u][0] = ldg_stream(src + lane * 16);
        w[u][1] = ldg_stream(src + (lane + 32) * 16);
        w[u][2] = ldg_stream(src + kRc12Chunk + lane * 16);
        e[u] = ldg_stream_u32(p.esc + (q0 + q) * kRc12EscWords + (lane & 7));
      }
    }
  };
  auto compute_batch = [&](int base, const uint4 (&w)[U][3], const uint32_t (&e)[U]) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int q = base + u * kWarps;
      if (q >= nq) break;
      const int col0 = (q % ks) * kChunk;
      // group j: low bytes in w[j / 2] (.x .y or .z .w), nibbles in word j of w[2]
      uint32_t pw[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t lo0 = (j & 1) ? w[u][j >> 1].z : w[u][j >> 1].x;
        const uint32_t lo1 = (j & 1) ? w[u][j >> 1].w : w[u][j >> 1].y;
        const uint32_t nb = j == 0 ? w[u][2].x : (j == 1 ? w[u][2].y : (j == 2 ? w[u][2].z : w[u][2].w));
        const uint32_t hl = ((nb & 0x07070707u) + p.e0x4) | ((nb << 4) & 0x80808080u);
        const uint32_t hh = (((nb >> 4) & 0x07070707u) + p.e0x4) | (nb & 0x80808080u);
        pw[4 * j + 0] = __byte_perm(lo0, hl, 0x5140);
        pw[4 * j + 1] = __byte_perm(lo0, hl, 0x7362);
        pw[4 * j + 2] = __byte_perm(lo1, hh, 0x5140);
        pw[4 * j + 3] = __byte_perm(lo1, hh, 0x7362);
      }
      const uint32_t cnt = min(__shfl_sync(0xffffffffu, e[u], 0), static_cast<uint32_t>(kRc12EscCap));
      for (uint32_t k = 0; k < cnt; ++k) {  // warp-uniform
        const uint32_t ent = __shfl_sync(0xffffffffu, e[u], static_cast<int>(1 + k));
        const uint32_t pos = ent >> 8;  // column in the chunk: 8 (lane + 32 j) + b
        if (static_cast<int>((pos >> 3) & 31) == lane) {
          const uint32_t wi = (pos >> 8) * 4 + ((pos >> 1) & 3);
          const uint32_t sel = (pos & 1) ? 0x4210u : 0x3240u;  // byte 3 or byte 1 <- high byte
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (static_cast<uint32_t>(i) == wi) pw[i] = __byte_perm(pw[i], ent, sel);
        }
      }
      float a8[MT][8];
#pragma unroll
      for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int c = 0; c < 8; ++c) a8[t][c] = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          const uint4 xv = ld_shared_u4(
              xs_a + static_cast<uint32_t>((t * p.K + col0 + (lane + 32 * i) * 8) * 2));
          float* a = a8[t];
          fma_bf16x2(a[(i & 1) * 4 + 0], a[(i & 1) * 4 + 1], pw[4 * i + 0], xv.x);
          fma_bf16x2(a[(i & 1) * 4 + 2], a[(i & 1) * 4 + 3], pw[4 * i + 1], xv.y);
          fma_bf16x2(a[(i & 1) * 4 + 0], a[(i & 1) * 4 + 1], pw[4 * i + 2], xv.z);
          fma_bf16x2(a[(i & 1) * 4 + 2], a[(i & 1) * 4 + 3], pw[4 * i + 3], xv.w);
        }
      }
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        float v = ((a8[t][0] + a8[t][1]) + (a8[t][2] + a8[t][3])) +
                  ((a8[t][4] + a8[t][5]) + (a8[t][6] + a8[t][7]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == t) cp[q * MT + t] = v;
      }
    }
  };

  uint4 wa[U][3], wb[U][3];
  uint32_t ea[U], eb[U];
  int base = warp;
  load_batch(base, wa, ea);
  griddep_launch_dependents();
  griddep_wait();
  {
    const uint4* xg = static_cast<const uint4*>(p.x);
    const int n8 = MT * p.K / 8;
    constexpr int kXLd = (MT * 8192 / 8 + kThreads - 1) / kThreads;
    uint4 xv[kXLd];
#pragma unroll
    for (int u = 0; u < kXLd; ++u) {
      const int i = threadIdx.x + u * kThreads;
      xv[u] = (i < n8 && i / (p.K / 8) < p.m) ? xg[i] : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kXLd; ++u) {
      const int i = threadIdx.x + u * kThreads;
      if (i >= n8) break;
      reinterpret_cast<uint4*>(xs)[i] = xv[u];
    }
  }
  __syncthreads();
  constexpr int kStride = kWarps * U;
  while (base < nq) {
    if (base + kStride < nq) load_batch(base + kStride, wb, eb);
    compute_batch(base, wa, ea);
    base += kStride;
    if (base >= nq) break;
    if (base + kStride < nq) load_batch(base + kStride, wa, ea);
    compute_batch(base, wb, eb);
    base += kStride;
  }
  __syncthreads();

  const uint32_t cp_a = smem_u32(cp);
  for (int idx = threadIdx.x; idx < (r1 - r0) * MT; idx += kThreads) {
    const int rr = idx / MT;
    const int t = idx - rr * MT;
    float part[kMaxKs];
#pragma unroll
    for (int c = 0; c < kMaxKs; ++c)
      part[c] = c < ks ? ld_shared_f32(cp_a + static_cast<uint32_t>(((rr * ks + c) * MT + t) * 4))
                       : 0.f;
    float v = part[0];
#pragma unroll
    for (int c = 1; c < kMaxKs; ++c)
      if (c < ks) v += part[c];
    if (t < p.m)
      static_cast<__nv_bfloat16*>(p.out)[static_cast<int64_t>(t) * p.n_rows + r0 + rr] =
          __float2bfloat16_rn(v);
  }
}

template <typename WT, int MT>
cudaError_t set_attr() {
  return cudaFuncSetAttribute(gemv_reg_kernel<WT, MT>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(RCfgG<WT, MT>::kSmem));
}

template <typename WT, int MT>
cudaError_t launch(const GemvParams& p, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = RCfgG<WT, MT>::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_reg_kernel<WT, MT>, p);
}

template <int MT>
cudaError_t launch12(const GemvParams& p, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = RCfgG<__nv_bfloat16, MT>::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_reg12_kernel<MT>, p);
}

}  // namespace

cudaError_t gemv_reg_init_attributes() {
  cudaError_t e;
  const int s1 = static_cast<int>(RCfgG<__nv_bfloat16, 1>::kSmem);
  const int s2 = static_cast<int>(RCfgG<__nv_bfloat16, 2>::kSmem);
  if ((e = cudaFuncSetAttribute(gemv_reg12_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                s1)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(gemv_reg12_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                s2)) != cudaSuccess)
    return e;
  if ((e = set_attr<__nv_bfloat16, 1>()) != cudaSuccess) return e;
  if ((e = set_attr<__nv_bfloat16, 2>()) != cudaSuccess) return e;
  if ((e = set_attr<float, 1>()) != cudaSuccess) return e;
  if ((e = set_attr<float, 2>()) != cudaSuccess) return e;
  return cudaSuccess;
}

cudaError_t gemv_reg_launch(bool f32w, int MT, const GemvParams& p, cudaStream_t s) {
  if (f32w) {
    switch (MT) {
      case 1: return launch<float, 1>(p, s);
      case 2: return launch<float, 2>(p, s);
    }
  } else {
    switch (MT) {
      case 1: return launch<__nv_bfloat16, 1>(p, s);
      case 2: return launch<__nv_bfloat16, 2>(p, s);
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t gemv_reg12_launch(int MT, const GemvParams& p, cudaStream_t s) {
  switch (MT) {
    case 1: return launch12<1>(p, s);
    case 2: return launch12<2>(p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace proj
