// router_gemv.cu -- the router (fp32 weights, fp32 output) at 3..16 tokens:
// a weight-streaming GEMV on FP32 fused multiply-adds.
//
// out[i, n] = sum_k x[i, k] W[n, k]            (muse_bf16_proj guide, ch. 1, §1.1)
//
// Full FP32 precision as in the router's other kernels: every product is the
// bf16 input widened exactly times the fp32 weight, summed in fp32 with
// fma.rn.f32x2 on (even k, odd k) pairs (guide ch. 1, §1.5).  At a few
// tokens the router is an 8 MB weight stream with little arithmetic, and
// the wide kernel's 128-row tiles need a deep split of K whose partials and
// barriers cost more than the stream.  Here, as in the one-token GEMV
// (gemv_reg.cu):
//
// * CTA c owns whole rows [c N / G, (c + 1) N / G) of the row-major W, each
//   row cut into 1024-element chunks; warp w takes chunk w (a CTA holds at
//   most 16 chunks), its 32 weights per lane loaded straight into registers
//   before the dependency wait.
// * The tokens go in passes of eight: x's eight rows (bf16, 16 KB each) are
//   staged in shared memory, every warp multiplies its chunk's registers by
//   them, and a transposing shuffle reduction leaves each token's chunk sum
//   in a lane; the next pass restages x and reuses the same weight
//   registers.
// * After a barrier each (row, token) is summed over its chunks in chunk
//   order (deterministic) and stored.  No row crosses CTAs.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace proj {
namespace {

constexpr int kChunk = 1024;
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kPass = 8;                             // tokens per pass
constexpr int kXBytes = kPass * 8192 * 2;             // bf16 x rows, K <= 8192
constexpr int kCpBytes = kWarps * kRouterGemvMaxM * 4;  // chunk partials [chunk][token]
constexpr int kSmem = kXBytes + kCpBytes;

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
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
__device__ __forceinline__ void st_shared_u4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}
// Two bf16 (low half first) widened exactly to an fp32 pair.
__device__ __forceinline__ uint64_t bf16x2_to_f32x2(uint32_t v) {
  return (static_cast<uint64_t>(v & 0xFFFF0000u) << 32) | (v << 16);
}
// (acc.lo, acc.hi) += (w.lo, w.hi) * (x.lo, x.hi)
__device__ __forceinline__ void ffma2(uint64_t& acc, uint64_t w, uint64_t x) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(w), "l"(x));
}
__device__ __forceinline__ float f32x2_sum(uint64_t a) {
  return __uint_as_float(static_cast<uint32_t>(a)) + __uint_as_float(static_cast<uint32_t>(a >> 32));
}

__global__ void __launch_bounds__(kThreads, 1) router_gemv_kernel(const RouterGemvParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const uint32_t sX = smem_u32(smem_raw);  // [8 tokens][K] bf16
  const uint32_t sCp = sX + kXBytes;       // [chunk][token] fp32

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ks = p.K / kChunk;
  const int r0 = static_cast<int>(static_cast<uint32_t>(blockIdx.x) * p.N / p.G);
  const int r1 = static_cast<int>((static_cast<uint32_t>(blockIdx.x) + 1u) * p.N / p.G);
  const int nq = (r1 - r0) * ks;  // chunks of the CTA (<= 16, host-checked)
  const bool has = warp < nq;
  const int col0 = has ? (warp % ks) * kChunk : 0;

  // This warp's chunk: lane l holds k = col0 + 4 l + 128 i + (0..3), i < 8.
  uint4 w[8];
  if (has) {
    const float* src = static_cast<const float*>(p.w) +
                       (static_cast<size_t>(r0) * ks + warp) * kChunk;  // chunks are contiguous
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = ldg_stream(src + (lane + 32 * i) * 4);
  }
  griddep_launch_dependents();
  griddep_wait();

  const uint16_t* X = static_cast<const uint16_t*>(p.x);
  const int n16 = p.K / 8;  // 16-byte chunks of an x row
  for (int t0 = 0; t0 < p.m; t0 += kPass) {
    const int nt = min(kPass, p.m - t0);
    // x rows t0 .. t0 + nt - 1 -> shared memory, all loads first
    {
      const int total = nt * n16;
      uint4 xv[kPass * 8192 / 8 / kThreads];  // 16
#pragma unroll
      for (int j = 0; j < kPass * 8192 / 8 / kThreads; ++j) {
        const int i = threadIdx.x + j * kThreads;
        if (i < total)
          xv[j] = *reinterpret_cast<const uint4*>(X + static_cast<size_t>(t0) * p.K +
                                                  static_cast<size_t>(i) * 8);
      }
#pragma unroll
      for (int j = 0; j < kPass * 8192 / 8 / kThreads; ++j) {
        const int i = threadIdx.x + j * kThreads;
        if (i < total) st_shared_u4(sX + static_cast<uint32_t>(i * 16), xv[j]);
      }
    }
    __syncthreads();
    if (has) {
      float s[kPass];
#pragma unroll
      for (int t = 0; t < kPass; ++t) {
        uint64_t a0 = 0ull, a1 = 0ull;
        if (t < nt) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint2 xv = ld_shared_u2(
                sX + static_cast<uint32_t>((t * p.K + col0 + (lane + 32 * i) * 4) * 2));
            ffma2(a0, (static_cast<uint64_t>(w[i].y) << 32) | w[i].x, bf16x2_to_f32x2(xv.x));
            ffma2(a1, (static_cast<uint64_t>(w[i].w) << 32) | w[i].z, bf16x2_to_f32x2(xv.y));
          }
        }
        s[t] = f32x2_sum(a0) + f32x2_sum(a1);
      }
      // Transposing reduction: after the three halving steps lane l holds
      // the partial of token ((l >> 2) & 7) summed over 8 lanes; two more
      // steps complete it over all 32.
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const bool up = lane & 16;
        const float send = up ? s[h] : s[h + 4];
        const float keep = up ? s[h + 4] : s[h];
        s[h] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const bool up = lane & 8;
        const float send = up ? s[h] : s[h + 2];
        const float keep = up ? s[h + 2] : s[h];
        s[h] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
      }
      {
        const bool up = lane & 4;
        const float send = up ? s[0] : s[1];
        const float keep = up ? s[1] : s[0];
        s[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
      }
      s[0] += __shfl_xor_sync(0xffffffffu, s[0], 2);
      s[0] += __shfl_xor_sync(0xffffffffu, s[0], 1);
      // lane l: token index from bits 4, 3, 2 (high half kept the upper
      // tokens at each step)
      const int t = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
      if ((lane & 3) == 0 && t < nt)
        st_shared_f32(sCp + static_cast<uint32_t>((warp * kRouterGemvMaxM + t0 + t) * 4), s[0]);
    }
    __syncthreads();  // x is restaged by the next pass; the partials are complete
  }
  // Rows of the CTA, each summed over its chunks in chunk order.
  for (int idx = threadIdx.x; idx < (r1 - r0) * p.m; idx += kThreads) {
    const int rr = idx / p.m;
    const int t = idx - rr * p.m;
    float v = 0.f;
    for (int c = 0; c < ks; ++c)
      v += ld_shared_f32(sCp + static_cast<uint32_t>(((rr * ks + c) * kRouterGemvMaxM + t) * 4));
    static_cast<float*>(p.out)[static_cast<size_t>(t) * p.N + r0 + rr] = v;
  }
}

}  // namespace

cudaError_t router_gemv_init_attributes() {
  return cudaFuncSetAttribute(router_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmem);
}

cudaError_t router_gemv_launch(const RouterGemvParams& p, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, router_gemv_kernel, p);
}

}  // namespace proj
