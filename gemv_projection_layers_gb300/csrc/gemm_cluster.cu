// gemm_cluster.cu -- tensor-core GEMM, split-K inside a thread-block
// cluster, combined through distributed shared memory: the bf16 layers at
// wide token tiles and the router (fp32 weights as three exact bf16 planes).
//
// out[i, n] = sum_k x[i, k] W[n, k]            (muse_bf16_proj guide, ch. 1, §1.1)
//
// At 128 and 256 tokens a 128-row output tile holds 64-128 KB of fp32
// partial sums, so splitting K across CTAs that meet in global memory moves
// as many partial bytes as weight bytes and serialises a long epilogue
// behind the MMAs.  Here every output tile (128 weight rows x BN tokens) is
// one cluster of CS CTAs (CS = 1 .. 16); CTA rank r computes the r-th 1/CS of
// K with the same swapped-operand tcgen05 pipeline as the narrow kernel
// (bulk copies of prepacked swizzled weight tiles, 2-D TMA for x, fp32
// accumulation in tensor memory).  After its last MMA the accumulator goes
// to the CTA's own shared memory, a cluster barrier publishes it, and rank r
// sums tokens [r BN / CS, (r + 1) BN / CS) over the cluster's CTAs in rank
// order (distributed shared memory loads), rounds to bf16 (the router keeps
// fp32) and stores.  No
// global partials, no atomics, no waits on other clusters; the sum order is
// fixed, so results are deterministic.  The pages' nearest design is the
// cluster/DSMEM split-K of a small-token QKV kernel (muse_bf16_proj notebook,
// n. 20 "Hopper pipelines and block clusters", distributed shared-memory
// reduction), here on tcgen05 and for the wide token tiles.
//
// Router: W (fp32) was split at prepare into bf16 planes hi + mid + lo == W
// exactly, stored as the tiles of a [N, 3K] bf16 matrix.  Weight k-block kb
// meets x k-block kb % KBx, so x @ [hi | mid | lo].T accumulates the three
// exact bf16 x bf16 products of every weight in fp32 -- the same sum as
// fp32 weights, without TF32 truncation -- and the result is stored as fp32.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace proj {
namespace {

constexpr int kSmemLimit = 232448;

template <int BN>
struct CCfg {
  static constexpr int kXBytes = BN * 128;
  static constexpr int kStage = kTileBytes + kXBytes;
  static constexpr int kFit = (kSmemLimit - 1024 - 1024) / kStage;
  static constexpr int S = kFit > 12 ? 12 : kFit;
  static constexpr int kThreads = 192;
  static constexpr int kTmemCols = BN < 32 ? 32 : BN;
  static constexpr size_t kRing = static_cast<size_t>(S) * kStage;
  static constexpr size_t kRed = static_cast<size_t>(BN) * kTileRows * 4;  // [BN][128] fp32
  static constexpr size_t kData = kRing > kRed ? kRing : kRed;
  static constexpr size_t kSmem = 1024 + kData + (2 * S + 2) * 8 + 16;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(128, BN);
  static_assert(S >= 3, "pipeline too shallow");
  static_assert(kSmem <= kSmemLimit, "shared memory budget");
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// Peer partials are stable between the two cluster barriers, so these loads
// carry no memory clobber and can be issued back to back.
__device__ __forceinline__ float4 ld_dsmem_v4(uint32_t addr) {
  float4 v;
  asm("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
      : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
      : "r"(addr));
  return v;
}

template <int BN>
__global__ void __launch_bounds__(192, 1)
    tc_cluster_kernel(const __grid_constant__ CUtensorMap tmap_x, const ClusterParams p) {
  using C = CCfg<BN>;
  constexpr int S = C::S;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + static_cast<size_t>(S) * kTileBytes;
  float* red = reinterpret_cast<float*>(smem);  // reuses the ring after the last MMA
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kData);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 2);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * S;
  const uint32_t accf = empty0 + 8 * S;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int tile = static_cast<int>(blockIdx.x) / p.CS;  // cluster index
  const int t = tile / p.MT;
  const int mt = tile % p.MT;
  const int kb0 = static_cast<int>((static_cast<int64_t>(rank) * p.KB) / p.CS);
  const int kb1 = static_cast<int>((static_cast<int64_t>(rank + 1) * p.KB) / p.CS);
  const int mv = min(BN, p.m - mt * BN);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(accf, 1);
    fence_mbar_init();
    prefetch_tmap(&tmap_x);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int64_t issued = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        const int s = static_cast<int>(issued % S);
        if (!mbar_wait(empty0 + 8 * s, static_cast<uint32_t>(((issued / S) & 1) ^ 1), p.status,
                       kStatusTimeoutProducer))
          break;
        const uint32_t fb = full0 + 8 * s;
        mbar_arrive_expect_tx(fb, kTileBytes + C::kXBytes);
        bulk_g2s(smem_u32(sA + s * kTileBytes),
                 p.w + (static_cast<size_t>(t) * p.KB + kb) * kTileBytes, kTileBytes, fb, pol);
        tma_load_2d(smem_u32(sB + s * C::kXBytes), &tmap_x, (kb % p.KBx) * kTileK, mt * BN,
                    fb);
        ++issued;
      }
      // Wait (bounded) for the copies still in flight before the ring is
      // reused as the reduction buffer or the CTA exits.
      const int64_t n = issued < S ? issued : S;
      for (int64_t j = 0; j < n; ++j) {
        const int64_t idx = issued - 1 - j;
        mbar_wait(full0 + 8 * static_cast<int>(idx % S), static_cast<uint32_t>((idx / S) & 1),
                  p.status, kStatusTimeoutDrain);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      int64_t j = 0;
      for (int kb = kb0; kb < kb1; ++kb, ++j) {
        const int s = static_cast<int>(j % S);
        if (!mbar_wait(full0 + 8 * s, static_cast<uint32_t>((j / S) & 1), p.status,
                       kStatusTimeoutMma))
          break;
        tc_fence_after();
        const uint32_t a = smem_u32(sA + s * kTileBytes);
        const uint32_t b = smem_u32(sB + s * C::kXBytes);
#pragma unroll
        for (int k = 0; k < kTileK / 16; ++k) {
          tc_mma_f16(tmem, smem_desc_sw128(a + 32 * k), smem_desc_sw128(b + 32 * k), C::kIdesc,
                     (kb > kb0 || k > 0) ? 1u : 0u);
        }
        tc_commit(empty0 + 8 * s);
      }
      tc_commit(accf);  // also covers an aborted loop: arrives once prior MMAs finish
    }
  } else {
    // ------------------------------------- epilogue: accumulator -> smem
    const int q = warp & 3;
    const int r = q * 32 + lane;
    if (mbar_wait(accf, 0, p.status, kStatusTimeoutEpilogue)) {
      tc_fence_after();
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float v[16];
        tmem_ld16(taddr + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) red[(c0 + jj) * kTileRows + r] = v[jj];
      }
      tc_fence_before();
    }
  }
  __syncwarp();
  // Every CTA of the cluster has its partial in shared memory.
  cluster_sync_all();
  // Rank r sums tokens [r BN / CS, (r + 1) BN / CS) over the cluster, in rank
  // order; a thread handles 4 consecutive rows of one token (float4).
  {
    const int j0 = static_cast<int>(rank) * BN / p.CS;
    const int j1 = min(static_cast<int>(rank + 1) * BN / p.CS, mv);
    const uint32_t red_base = smem_u32(red);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
    for (int idx = threadIdx.x; idx < (j1 - j0) * 32; idx += C::kThreads) {
      const int j = j0 + idx / 32;
      const int quad = idx % 32;
      const uint32_t off = static_cast<uint32_t>((j * kTileRows + quad * 4) * 4);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int r0 = 0; r0 < kClusterMaxCS; r0 += 8) {
        if (r0 >= p.CS) break;
        float4 v[8];
#pragma unroll
        for (int rr = 0; rr < 8; ++rr)
          if (r0 + rr < p.CS)
            v[rr] = ld_dsmem_v4(map_to_rank(red_base + off, static_cast<uint32_t>(r0 + rr)));
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) {
          if (r0 + rr < p.CS) {
            acc.x += v[rr].x;
            acc.y += v[rr].y;
            acc.z += v[rr].z;
            acc.w += v[rr].w;
          }
        }
      }
      const size_t o_idx = (static_cast<size_t>(mt) * BN + j) * p.n_out +
                           static_cast<size_t>(t) * kTileRows + quad * 4;
      if (p.out_f32) {
        *reinterpret_cast<float4*>(static_cast<float*>(p.out) + o_idx) = acc;
        continue;
      }
      __nv_bfloat16* o = out + o_idx;
      __nv_bfloat162 lo2, hi2;
      lo2.x = __float2bfloat16_rn(acc.x);
      lo2.y = __float2bfloat16_rn(acc.y);
      hi2.x = __float2bfloat16_rn(acc.z);
      hi2.y = __float2bfloat16_rn(acc.w);
      *reinterpret_cast<__nv_bfloat162*>(o) = lo2;
      *reinterpret_cast<__nv_bfloat162*>(o + 2) = hi2;
    }
  }
  // No CTA may leave while a peer still reads its shared memory.
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int BN>
cudaError_t set_attr() {
  cudaError_t e = cudaFuncSetAttribute(tc_cluster_kernel<BN>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(CCfg<BN>::kSmem));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(tc_cluster_kernel<BN>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                              1);
}

template <int BN>
cudaLaunchConfig_t make_cfg(const ClusterParams& p, cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.MT * p.T * p.CS);
  cfg.blockDim = dim3(CCfg<BN>::kThreads);
  cfg.dynamicSmemBytes = CCfg<BN>::kSmem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.CS);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <int BN>
cudaError_t launch(const CUtensorMap& tmap, const ClusterParams& p, cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg<BN>(p, s, attr);
  return cudaLaunchKernelEx(&cfg, tc_cluster_kernel<BN>, tmap, p);
}

template <int BN>
int max_clusters(int cs) {
  ClusterParams p = {};
  p.MT = 1;
  p.T = 1;
  p.CS = cs;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg<BN>(p, nullptr, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, tc_cluster_kernel<BN>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace

bool cluster_supported(int BN) {
  return BN == 16 || BN == 32 || BN == 64 || BN == 128 || BN == 256;
}

cudaError_t cluster_init_attributes() {
  cudaError_t e;
  if ((e = set_attr<16>()) != cudaSuccess) return e;
  if ((e = set_attr<32>()) != cudaSuccess) return e;
  if ((e = set_attr<64>()) != cudaSuccess) return e;
  if ((e = set_attr<128>()) != cudaSuccess) return e;
  if ((e = set_attr<256>()) != cudaSuccess) return e;
  return cudaSuccess;
}

int cluster_max_active(int BN, int cs) {
  switch (BN) {
    case 16: return max_clusters<16>(cs);
    case 32: return max_clusters<32>(cs);
    case 64: return max_clusters<64>(cs);
    case 128: return max_clusters<128>(cs);
    case 256: return max_clusters<256>(cs);
  }
  return 0;
}

int cluster_stages(int BN) {
  switch (BN) {
    case 16: return CCfg<16>::S;
    case 32: return CCfg<32>::S;
    case 64: return CCfg<64>::S;
    case 128: return CCfg<128>::S;
    case 256: return CCfg<256>::S;
  }
  return 0;
}

cudaError_t cluster_launch(int BN, const CUtensorMap& tmap, const ClusterParams& p,
                           cudaStream_t s) {
  switch (BN) {
    case 16: return launch<16>(tmap, p, s);
    case 32: return launch<32>(tmap, p, s);
    case 64: return launch<64>(tmap, p, s);
    case 128: return launch<128>(tmap, p, s);
    case 256: return launch<256>(tmap, p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace proj
