// cluster_common.cuh -- pieces shared by the cluster split-K kernels (the
// tensor-core GEMM and the FP32-FMA router): cluster helpers, output
// stores, and the fixed-order combine of a cluster's partial tiles.
#pragma once

#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace proj {

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

// The staging buffer is addressed through 32-bit shared-window addresses:
// the 1 KB alignment arithmetic on the dynamic shared-memory pointer hides
// its address space from the compiler, and generic accesses are slower.
__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ float4 ld_shared_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

// Peer partials are stable between the two cluster barriers: these loads
// carry no memory clobber, so they issue back to back; volatile keeps them
// after the barrier (volatile asm too).
__device__ __forceinline__ float4 ld_dsmem_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

// Token j, rows row0..row0 + 3 of output tile (t, mt): fp32 as is, or
// rounded to bf16 (round-to-nearest-even).
template <int BN>
__device__ __forceinline__ void store_out(const ClusterParams& p, int mt, int t, int j, int row0,
                                          float4 v) {
  const size_t o_idx = (static_cast<size_t>(mt) * BN + j) * p.n_out +
                       static_cast<size_t>(t) * kTileRows + row0;
  if (p.out_f32) {
    *reinterpret_cast<float4*>(static_cast<float*>(p.out) + o_idx) = v;
  } else {
    __nv_bfloat162 lo2, hi2;
    lo2.x = __float2bfloat16_rn(v.x);
    lo2.y = __float2bfloat16_rn(v.y);
    hi2.x = __float2bfloat16_rn(v.z);
    hi2.y = __float2bfloat16_rn(v.w);
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + o_idx;
    *reinterpret_cast<__nv_bfloat162*>(o) = lo2;
    *reinterpret_cast<__nv_bfloat162*>(o + 2) = hi2;
  }
}

// With KG > 1 clusters per output tile: every cluster has written its
// partial of rank r's tokens to its own workspace slab; the last of the
// tile's KG clusters to finish sums the slabs in cluster order -- the same
// order whichever finishes last -- and stores the tile.  Nothing waits:
// earlier clusters just leave.  One release per CTA after the barrier (it
// orders the CTA's partial stores before the count); its acquire, through
// the second barrier, orders the last CTA's loads after every other
// cluster's stores.
template <int BN, int kThreads>
__device__ __forceinline__ void group_finish(const ClusterParams& p, int cluster, int tile, int t,
                                             int mt, uint32_t rank, int j0, int n_items) {
  if (p.KG <= 1) return;
  __shared__ uint32_t s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t old = atom_add_acq_rel_gpu(p.counters + tile * p.CS + rank, 1u);
    s_last = old == static_cast<uint32_t>(p.KG - 1) ? 1u : 0u;
  }
  __syncthreads();
  if (s_last) {
    const float* slab0 = p.ws + static_cast<size_t>(tile) * p.KG * BN * kTileRows;
    for (int idx = threadIdx.x; idx < n_items; idx += kThreads) {
      const uint32_t o4 = static_cast<uint32_t>((j0 + idx / 32) * kTileRows + (idx % 32) * 4);
      // every group's partial in one round trip, summed in group order
      float4 v[kClusterMaxGroups];
#pragma unroll
      for (int gg = 0; gg < kClusterMaxGroups; ++gg)
        if (gg < p.KG)
          v[gg] = __ldcg(reinterpret_cast<const float4*>(
              slab0 + static_cast<size_t>(gg) * BN * kTileRows + o4));
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int gg = 0; gg < kClusterMaxGroups; ++gg)
        if (gg < p.KG) {
          acc.x += v[gg].x;
          acc.y += v[gg].y;
          acc.z += v[gg].z;
          acc.w += v[gg].w;
        }
      store_out<BN>(p, mt, t, j0 + idx / 32, (idx % 32) * 4, acc);
    }
    if (threadIdx.x == 0) p.counters[tile * p.CS + rank] = 0u;  // ready for the next call
  }
  (void)cluster;
}

__device__ __forceinline__ float4 ld_global_cg_v4(const float* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

// Combine through L2.  Every CTA has stored the tokens it does not own to its
// exchange slot (p.xch + blockIdx.x * BN * 128, [token][128 rows]) and kept
// its own tokens in shared memory (red_base, [token][128 rows]); a cluster
// barrier ordered those stores before this.  Rank r sums tokens
// [r BN / CS, (r + 1) BN / CS) over the cluster's CTAs in rank order (its
// own partial from shared memory, the others' from L2) and stores (or, with
// KG > 1, passes the cluster's partial on).  No CTA touches another's shared
// memory, so no barrier is needed before leaving.
template <int BN, int kThreads, int kItems = 4>
__device__ __forceinline__ void cluster_combine_l2(const ClusterParams& p, uint32_t red_base,
                                                   int cluster, int tile, int t, int mt,
                                                   uint32_t rank, int mv) {
  const int j0 = static_cast<int>(rank) * BN / p.CS;
  const int j1 = min(static_cast<int>(rank + 1) * BN / p.CS, mv);
  const int n_items = max(j1 - j0, 0) * 32;
  const float* slots = p.xch + static_cast<size_t>(cluster) * p.CS * BN * kTileRows;
  for (int base = threadIdx.x; base < n_items; base += kItems * kThreads) {
    float4 acc[kItems];
    uint32_t off[kItems];
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
      acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      const int idx = min(base + u * kThreads, n_items - 1);
      off[u] = static_cast<uint32_t>((j0 + idx / 32) * kTileRows + (idx % 32) * 4);
    }
    for (int r0 = 0; r0 < p.CS; r0 += 4) {
      float4 v[kItems][4];
#pragma unroll
      for (int u = 0; u < kItems; ++u)
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
          const int src = r0 + rr;
          if (src == static_cast<int>(rank))
            v[u][rr] = ld_shared_v4(red_base + off[u] * 4);
          else if (src < p.CS)
            v[u][rr] = ld_global_cg_v4(slots + static_cast<size_t>(src) * BN * kTileRows + off[u]);
        }
#pragma unroll
      for (int u = 0; u < kItems; ++u)
#pragma unroll
        for (int rr = 0; rr < 4; ++rr)
          if (r0 + rr < p.CS) {
            acc[u].x += v[u][rr].x;
            acc[u].y += v[u][rr].y;
            acc[u].z += v[u][rr].z;
            acc[u].w += v[u][rr].w;
          }
    }
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
      const int idx = base + u * kThreads;
      if (idx >= n_items) break;
      if (p.KG > 1) {
        *reinterpret_cast<float4*>(p.ws + static_cast<size_t>(cluster) * BN * kTileRows +
                                   off[u]) = acc[u];
      } else {
        store_out<BN>(p, mt, t, j0 + idx / 32, (idx % 32) * 4, acc[u]);
      }
    }
  }
  group_finish<BN, kThreads>(p, cluster, tile, t, mt, rank, j0, n_items);
}

// The combine after every CTA of the cluster has staged its fp32 partial of
// output tile (t, mt) at red_base ([BN tokens][128 rows], token-major) and
// a cluster barrier has published it.  kItems items per thread are in
// flight per round trip (fewer for kernels short of registers).
template <int BN, int kThreads, int kItems = 4>
__device__ __forceinline__ void cluster_combine(const ClusterParams& p, uint32_t red_base,
                                                int cluster, int tile, int t, int mt,
                                                uint32_t rank, int mv) {
  // Rank r sums tokens [r BN / CS, (r + 1) BN / CS) over the cluster, in rank
  // order; an item is 4 consecutive rows of one token (float4).  A thread
  // keeps kItems items x 4 ranks of loads in flight; its own rank's partial
  // comes from local shared memory, the others' through distributed shared
  // memory.  (Pushing the slices with bulk shared-to-shared copies instead
  // measured slower: the extra mbarrier round trip outweighs the copy.)
  const int j0 = static_cast<int>(rank) * BN / p.CS;
  const int j1 = min(static_cast<int>(rank + 1) * BN / p.CS, mv);
  const int n_items = max(j1 - j0, 0) * 32;
  {
    for (int base = threadIdx.x; base < n_items; base += kItems * kThreads) {
      float4 acc[kItems];
      uint32_t off[kItems];
#pragma unroll
      for (int u = 0; u < kItems; ++u) {
        acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        const int idx = min(base + u * kThreads, n_items - 1);
        off[u] = static_cast<uint32_t>(((j0 + idx / 32) * kTileRows + (idx % 32) * 4) * 4);
      }
      for (int r0 = 0; r0 < p.CS; r0 += 4) {
        float4 v[kItems][4];
#pragma unroll
        for (int u = 0; u < kItems; ++u)
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) {
            const uint32_t src = static_cast<uint32_t>(r0 + rr);
            if (src == rank)
              v[u][rr] = ld_shared_v4(red_base + off[u]);
            else if (r0 + rr < p.CS)
              v[u][rr] = ld_dsmem_v4(map_to_rank(red_base + off[u], src));
          }
#pragma unroll
        for (int u = 0; u < kItems; ++u)
#pragma unroll
          for (int rr = 0; rr < 4; ++rr)
            if (r0 + rr < p.CS) {
              acc[u].x += v[u][rr].x;
              acc[u].y += v[u][rr].y;
              acc[u].z += v[u][rr].z;
              acc[u].w += v[u][rr].w;
            }
      }
#pragma unroll
      for (int u = 0; u < kItems; ++u) {
        const int idx = base + u * kThreads;
        if (idx >= n_items) break;
        if (p.KG > 1) {
          // this cluster's partial of the tile, summed with the others below
          *reinterpret_cast<float4*>(p.ws + static_cast<size_t>(cluster) * BN * kTileRows +
                                     off[u] / 4) = acc[u];
        } else {
          store_out<BN>(p, mt, t, j0 + idx / 32, (idx % 32) * 4, acc[u]);
        }
      }
    }
  }
  group_finish<BN, kThreads>(p, cluster, tile, t, mt, rank, j0, n_items);
}

}  // namespace proj
