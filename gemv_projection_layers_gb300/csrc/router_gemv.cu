// router_gemv.cu -- the router (fp32 weights, fp32 output) at a few tokens:
// weight-streaming GEMVs on FP32 fused multiply-adds, whole rows per CTA
// (3..16 tokens) or K split across a thread-block cluster (up to 32).
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

// ---------------------------------------------------------------------------
// The same weight stream with K split across a thread-block cluster: at
// 3..32 tokens x, not W, dominates what a whole-row CTA must stage (all of
// K for every token: 16 KB per token at K = 8192, against the CTA's ~55 KB
// of weights).  Here cluster rank q takes chunk column q (columns
// [1024 q, 1024 q + 1024)) of 8 rows, one row per warp, so a CTA stages only
// its 2 KB slice of each x row; the ranks' per-row partials are summed in
// rank order (deterministic) through distributed shared memory.
// ---------------------------------------------------------------------------
constexpr int kCcWarps = 8;
constexpr int kCcThreads = kCcWarps * 32;
constexpr int kCcRW = 1;          // rows per warp
constexpr int kCcRows = kCcWarps * kCcRW;        // rows per cluster
constexpr int kCcMaxM = kRouterGemvCcMaxM;       // tokens
constexpr int kCcXBytes = kCcMaxM * kChunk * 2;  // bf16 [m][1024]
constexpr int kCcCpBytes = kCcRows * kCcMaxM * 4;
constexpr int kCcSmem = kCcXBytes + kCcCpBytes;

__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t cc_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cc_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cc_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

__global__ void __launch_bounds__(kCcThreads, 2) router_gemv_cc_kernel(const RouterGemvParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const uint32_t sX = smem_u32(smem_raw);  // [m][1024] bf16
  const uint32_t sCp = sX + kCcXBytes;     // [row][token] fp32

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int CS = p.K / kChunk;  // cluster size = chunk columns
  const uint32_t q = cc_rank();
  const int r0 = static_cast<int>(blockIdx.x) / CS * kCcRows;
  const int col0 = static_cast<int>(q) * kChunk;

  // This warp's rows r0 + kCcRW warp + j: lane l holds k = col0 + 4 l + 128 i
  // + (0..3), i < 8, of each.
  uint4 w[kCcRW][8];
#pragma unroll
  for (int j = 0; j < kCcRW; ++j) {
    const int row = r0 + kCcRW * warp + j;
    if (row < p.N) {
      const float* src = static_cast<const float*>(p.w) + static_cast<size_t>(row) * p.K + col0;
#pragma unroll
      for (int i = 0; i < 8; ++i) w[j][i] = ldg_stream(src + (lane + 32 * i) * 4);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) w[j][i] = make_uint4(0, 0, 0, 0);
    }
  }
  griddep_launch_dependents();
  griddep_wait();

  // x[t, col0 .. col0 + 1023] for every token -> shared memory: asynchronous
  // 16-byte copies (no registers held beside the weights), one round trip
  {
    const uint16_t* X = static_cast<const uint16_t*>(p.x);
    const int total = p.m * (kChunk / 8);  // 16-byte pieces
    for (int i = threadIdx.x; i < total; i += kCcThreads) {
      const int t = i >> 7, c = i & 127;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sX + static_cast<uint32_t>(i * 16)),
                   "l"(X + static_cast<size_t>(t) * p.K + col0 + c * 8)
                   : "memory");
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
  }
  __syncthreads();
  for (int t0 = 0; t0 < p.m; t0 += kPass) {
    const int nt = min(kPass, p.m - t0);
    float s[kCcRW * kPass];  // s[8 j + t]: row j, token t0 + t
#pragma unroll
    for (int t = 0; t < kPass; ++t) {
      uint64_t a[kCcRW][2];
#pragma unroll
      for (int j = 0; j < kCcRW; ++j) a[j][0] = a[j][1] = 0ull;
      if (t < nt) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint2 xv = ld_shared_u2(
              sX + static_cast<uint32_t>(((t0 + t) * kChunk + (lane + 32 * i) * 4) * 2));
          const uint64_t x01 = bf16x2_to_f32x2(xv.x), x23 = bf16x2_to_f32x2(xv.y);
#pragma unroll
          for (int j = 0; j < kCcRW; ++j) {
            ffma2(a[j][0], (static_cast<uint64_t>(w[j][i].y) << 32) | w[j][i].x, x01);
            ffma2(a[j][1], (static_cast<uint64_t>(w[j][i].w) << 32) | w[j][i].z, x23);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kCcRW; ++j) s[8 * j + t] = f32x2_sum(a[j][0]) + f32x2_sum(a[j][1]);
    }
    // Transposing reduction over the lanes: at each step a lane keeps the
    // half of its values whose index bit matches its lane bit and adds its
    // partner's copy of that half; with 8 RW values, lane l ends with value
    // (l >> (5 - log2(8 RW))) summed over the lanes that shared it.
    constexpr int kV = kCcRW * kPass;  // 8 or 16
#pragma unroll
    for (int m2 = 16, n2 = kV / 2; n2 >= 1; m2 >>= 1, n2 >>= 1) {
#pragma unroll
      for (int h = 0; h < n2; ++h) {
        const bool up = lane & m2;
        const float send = up ? s[h] : s[h + n2];
        const float keep = up ? s[h + n2] : s[h];
        s[h] = keep + __shfl_xor_sync(0xffffffffu, send, m2);
      }
    }
    // remaining lane bits: plain butterfly
    constexpr int kSteps = kV == 16 ? 4 : 3;  // bits consumed by the transposing steps
#pragma unroll
    for (int b = 4 - kSteps; b >= 0; --b) s[0] += __shfl_xor_sync(0xffffffffu, s[0], 1 << b);
    const int vi = lane >> (5 - kSteps);  // value index: 8 j + t
    const int j = vi >> 3, t = vi & 7;
    if ((lane & ((1 << (5 - kSteps)) - 1)) == 0 && t < nt)
      st_shared_f32(sCp + static_cast<uint32_t>(((kCcRW * warp + j) * kCcMaxM + t0 + t) * 4), s[0]);
  }
  // every rank's partials complete and visible to the cluster
  __syncthreads();
  cc_sync();
  // Rank q sums its share of the cluster's (row, token) outputs over the
  // ranks in rank order.
  {
    const int n = kCcRows * p.m;
    const int i0 = static_cast<int>(q) * n / CS;
    const int i1 = (static_cast<int>(q) + 1) * n / CS;
    for (int idx = i0 + static_cast<int>(threadIdx.x); idx < i1; idx += kCcThreads) {
      const int rr = idx / p.m;
      const int t = idx - rr * p.m;
      const uint32_t a = sCp + static_cast<uint32_t>((rr * kCcMaxM + t) * 4);
      float v = 0.f;
      for (int c = 0; c < CS; ++c) v += ld_dsmem_f32(cc_map(a, static_cast<uint32_t>(c)));
      if (r0 + rr < p.N) static_cast<float*>(p.out)[static_cast<size_t>(t) * p.N + r0 + rr] = v;
    }
  }
  cc_sync();  // no CTA leaves while its partials may still be read
}

cudaLaunchConfig_t cc_cfg(const RouterGemvParams& p, cudaStream_t s, cudaLaunchAttribute (&attr)[2]) {
  cudaLaunchConfig_t cfg = {};
  const int cs = p.K / kChunk;
  cfg.gridDim = dim3(static_cast<unsigned>((p.N + kCcRows - 1) / kCcRows * cs));
  cfg.blockDim = dim3(kCcThreads);
  cfg.dynamicSmemBytes = kCcSmem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

}  // namespace

cudaError_t router_gemv_cc_launch(const RouterGemvParams& p, cudaStream_t s) {
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = cc_cfg(p, s, attr);
  return cudaLaunchKernelEx(&cfg, router_gemv_cc_kernel, p);
}

int router_gemv_cc_max_active(int N, int K) {
  RouterGemvParams p = {};
  p.N = N;
  p.K = K;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = cc_cfg(p, nullptr, attr);
  cfg.numAttrs = 1;  // the occupancy query takes the cluster shape only
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, router_gemv_cc_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t router_gemv_init_attributes() {
  cudaError_t e = cudaFuncSetAttribute(router_gemv_cc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kCcSmem);
  if (e != cudaSuccess) return e;
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
