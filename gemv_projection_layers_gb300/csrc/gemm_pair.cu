// gemm_pair.cu -- tensor-core GEMM on CTA pairs (tcgen05 cta_group::2): the
// bf16 layers at wide token tiles (and the router's bf16 planes on request).
//
// out[i, n] = sum_k x[i, k] W[n, k]            (muse_bf16_proj guide, ch. 1, §1.1)
//
// At 128 and 256 tokens the single-CTA cluster kernel streams, per 16 KB of
// weights, BN x 128 B of x from L2 into the same SM (as many x bytes as
// weight bytes at BN = 128, twice as many at 256), so its main loop is
// bound by what one SM can take in rather than by HBM.  The project report
// meets the same wall on H200 ("Round 4": the per-SM ingest of the wgmma
// GEMM).  Here two CTAs on two SMs form one M = 256 MMA unit: each holds
// one 128-row weight tile and half of the token tile's x, and the pair's
// MMA multiplies both weight tiles by the whole token tile, so a weight byte
// costs half the x bytes it costs a single CTA.
//
// Work split: a pair tile is 256 weight rows x BN tokens; KG pairs split its
// K into equal k-block ranges.  Each CTA ends with a [BN][128] fp32 partial
// in tensor memory, staged to shared memory after the last MMA.  The KG
// pairs of a pair tile form one thread-block cluster of 2 KG CTAs (pair i =
// ranks 2i, 2i + 1).  With KG > 1 the KG CTAs that hold the same 128 rows
// combine through L2: each stores the tokens it does not own to its exchange
// slot, a cluster barrier orders those stores, and each sums its 1/KG of the
// tokens over the KG partials in split order (deterministic), rounds to bf16
// and stores.  Nothing waits on another cluster.
//
// Pipeline per CTA: warp 0 copies (one 2-D TMA of a prepacked 16 KB weight
// tile and one of the CTA's x rows per k-block, both counted on the even
// CTA's "full" barrier), warp 1 of the even CTA issues the pair MMAs and
// commits each stage to both CTAs' "empty" barriers; then all eight warps
// drain the accumulator (own tokens to shared memory, the others to the
// exchange slot), store and combine.
#include <cuda_bf16.h>

#include "cluster_common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace proj {
namespace {

constexpr int kPairSmemLimit = 232448;
constexpr int kPairEarlyStages = 2;

template <int BN>
struct PCfg {
  static constexpr int kHalf = BN / 2;            // tokens of x held by each CTA
  static constexpr int kXBytes = kHalf * 128;     // one k-block of them
  static constexpr int kStage = kTileBytes + kXBytes;
  static constexpr int kFit = (kPairSmemLimit - 1024 - 1024) / kStage;
  static constexpr int S = kFit > 12 ? 12 : kFit;
  static constexpr int kThreads = kPairThreads;
  static constexpr int kTmemCols = BN;
  static constexpr size_t kRing = static_cast<size_t>(S) * kStage;
  static constexpr size_t kRed = static_cast<size_t>(BN) * kTileRows * 4;  // own tokens, fp32
  static constexpr size_t kData = kRing > kRed ? kRing : kRed;
  static constexpr size_t kSmem = 1024 + kData + (2 * S + 2) * 8 + 16;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(256, BN);
  static_assert(S >= 4, "pipeline too shallow");
  static_assert(kSmem <= kPairSmemLimit, "shared memory budget");
};

__device__ __forceinline__ void store_out4(const PairParams& p, int token, int row, float4 v) {
  const size_t o = static_cast<size_t>(token) * p.n_out + row;
  if (p.out_f32) {
    *reinterpret_cast<float4*>(static_cast<float*>(p.out) + o) = v;
  } else {
    __nv_bfloat162 lo2, hi2;
    lo2.x = __float2bfloat16_rn(v.x);
    lo2.y = __float2bfloat16_rn(v.y);
    hi2.x = __float2bfloat16_rn(v.z);
    hi2.y = __float2bfloat16_rn(v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo2);
    u.y = *reinterpret_cast<uint32_t*>(&hi2);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + o) = u;
  }
}

template <int BN>
__global__ void __launch_bounds__(kPairThreads, 1)
    tc_pair_kernel(const __grid_constant__ CUtensorMap tmap_w,
                   const __grid_constant__ CUtensorMap tmap_x, const PairParams p) {
  using C = PCfg<BN>;
  constexpr int S = C::S;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + static_cast<size_t>(S) * kTileBytes;
  // [own tokens][128 rows] fp32 staging for the combine; reuses the ring
  // after the last MMA
  const uint32_t red_base = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kData);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 2);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * S;
  const uint32_t accf = empty0 + 8 * S;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint64_t* const stamp = p.stamps ? p.stamps + blockIdx.x * 8 : nullptr;
  if (stamp && threadIdx.x == 0) stamp[kStampEntry] = globaltimer_ns();
  const uint32_t rank = cluster_rank();
  const uint32_t h = rank & 1u;       // 0: the even CTA of the pair, which issues the MMAs
  const uint32_t lead = rank & ~1u;   // that CTA's rank
  const int g = static_cast<int>(rank >> 1);                 // K split of this pair
  const int tm = static_cast<int>(blockIdx.x) / (2 * p.KG);  // (pair tile, token tile): the cluster
  const int mt = tm % p.MT;
  const int tp = tm / p.MT;
  const int t = 2 * tp + static_cast<int>(h);  // this CTA's 128-row weight tile
  const int kb0 = static_cast<int>(static_cast<int64_t>(g) * p.KB / p.KG);
  const int kb1 = static_cast<int>(static_cast<int64_t>(g + 1) * p.KB / p.KG);
  const int nk = kb1 - kb0;
  const int mv = min(BN, p.m - mt * BN);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(accf, 1);
    fence_mbar_init();
    prefetch_tmap(&tmap_w);
    prefetch_tmap(&tmap_x);
  }
  if (warp == 1) {
    // collective with the peer CTA's warp 1: same columns in both CTAs
    tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish_pair();
  }
  // Barrier initialisation (both CTAs) and the tensor-memory address are
  // published before any copy can signal a barrier of the other CTA.
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint32_t full_lead = map_to_rank(full0, lead);  // the even CTA's barriers
      const uint64_t pol_w = p.w_evict_first ? policy_evict_first() : policy_evict_normal();
      const uint64_t pol_x = policy_evict_normal();
      const int pre = min(nk, S);
      const int pre_w = min(pre, kPairEarlyStages);
      int issued = 0;
      for (int j = 0; j < pre_w; ++j) {
        if (h == 0) mbar_arrive_expect_tx(full0 + 8 * j, 2u * C::kStage);
        tma_load_2d_pair(smem_u32(sA + j * kTileBytes), &tmap_w, 0,
                         (t * p.KB + kb0 + j) * kTileRows, full_lead + 8 * j, pol_w);
      }
      griddep_wait();
      if (stamp) stamp[kStampDepWait] = globaltimer_ns();
      for (int j = 0; j < pre_w; ++j)
        tma_load_2d_pair(smem_u32(sB + j * C::kXBytes), &tmap_x, ((kb0 + j) % p.KBx) * kTileK,
                         mt * BN + static_cast<int>(h) * C::kHalf, full_lead + 8 * j, pol_x);
      for (int j = pre_w; j < pre; ++j) {
        if (h == 0) mbar_arrive_expect_tx(full0 + 8 * j, 2u * C::kStage);
        tma_load_2d_pair(smem_u32(sA + j * kTileBytes), &tmap_w, 0,
                         (t * p.KB + kb0 + j) * kTileRows, full_lead + 8 * j, pol_w);
        tma_load_2d_pair(smem_u32(sB + j * C::kXBytes), &tmap_x, ((kb0 + j) % p.KBx) * kTileK,
                         mt * BN + static_cast<int>(h) * C::kHalf, full_lead + 8 * j, pol_x);
      }
      issued = pre;
      for (int j = pre; j < nk; ++j) {
        const int s = j % S;
        if (!mbar_wait(empty0 + 8 * s, static_cast<uint32_t>(((j / S) & 1) ^ 1), p.status,
                       kStatusTimeoutProducer))
          break;
        if (h == 0) mbar_arrive_expect_tx(full0 + 8 * s, 2u * C::kStage);
        const int kb = kb0 + j;
        tma_load_2d_pair(smem_u32(sA + s * kTileBytes), &tmap_w, 0, (t * p.KB + kb) * kTileRows,
                         full_lead + 8 * s, pol_w);
        tma_load_2d_pair(smem_u32(sB + s * C::kXBytes), &tmap_x, (kb % p.KBx) * kTileK,
                         mt * BN + static_cast<int>(h) * C::kHalf, full_lead + 8 * s, pol_x);
        ++issued;
      }
      // The even CTA's barriers count both CTAs' copies: wait (bounded) for
      // the last ring's worth before the ring can be reused or the pair can
      // leave (the odd CTA stays until then through the cluster barrier).
      if (h == 0) {
        const int n = issued < S ? issued : S;
        for (int j = issued - n; j < issued; ++j)
          mbar_wait(full0 + 8 * (j % S), static_cast<uint32_t>((j / S) & 1), p.status,
                    kStatusTimeoutDrain);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (h == 0 && lane == 0) {
      const uint16_t pair_mask = static_cast<uint16_t>(0x3u << lead);
      for (int j = 0; j < nk; ++j) {
        const int s = j % S;
        if (!mbar_wait(full0 + 8 * s, static_cast<uint32_t>((j / S) & 1), p.status,
                       kStatusTimeoutMma))
          break;
        if (stamp && j == 0) stamp[kStampFirstFull] = globaltimer_ns();
        tc_fence_after();
        const uint32_t a = smem_u32(sA + s * kTileBytes);
        const uint32_t b = smem_u32(sB + s * C::kXBytes);
#pragma unroll
        for (int k = 0; k < kTileK / 16; ++k)
          tc_mma_f16_pair(tmem, smem_desc_sw128(a + 32 * k), smem_desc_sw128(b + 32 * k),
                          C::kIdesc, (j > 0 || k > 0) ? 1u : 0u);
        tc_commit_pair(empty0 + 8 * s, pair_mask);
      }
      // arrives once every MMA issued above has completed (also after an
      // aborted loop)
      tc_commit_pair(accf, pair_mask);
      if (stamp) stamp[kStampLastMma] = globaltimer_ns();
    }
  }
  __syncwarp();
  // ------------------------------------------------------------------ drain
  // All eight warps, once every MMA has completed: warp w reads tensor-memory
  // lane quarter w & 3 (rows 32 (w & 3) ..), columns of token half w >> 2.
  // The tokens this CTA owns go to the shared-memory staging ([BN][128]
  // fp32 at red_base, the ring, free by then); with KG > 1 the others go
  // straight from registers to this CTA's exchange slot ([BN][128] fp32: one
  // warp store is 32 consecutive rows of a token, 128 contiguous bytes).
  // (A first form drained with four warps into shared memory and copied the
  // exchange out in a second pass.)
  const int jo0 = g * BN / p.KG;  // CTA g owns tokens [g BN / KG, (g + 1) BN / KG)
  const int jo1 = (g + 1) * BN / p.KG;
  {
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int c_beg = (warp >> 2) * (BN / 2);
    const int c_end = min(c_beg + BN / 2, mv);
    if (mbar_wait_sleep(accf, 0, p.status, kStatusTimeoutEpilogue)) {
      if (stamp && warp == 4 && lane == 0) stamp[kStampAccReady] = globaltimer_ns();
      tc_fence_after();
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16);
      float* const slot =
          p.KG > 1 ? p.xch + static_cast<size_t>(blockIdx.x) * BN * kTileRows : nullptr;
      // (the previous kernel of the stream may be this handle's previous
      // call, still reading the exchange: wait for it before storing)
      (void)slot;
      auto put = [&](int c, float val) {
        st_shared_f32(red_base + static_cast<uint32_t>((c * kTileRows + r) * 4), val);
      };
#pragma unroll 1
      for (int c0 = c_beg; c0 < c_end; c0 += 32) {
        float v[16], u[16];
        tmem_ld16(taddr + c0, v);
        tmem_ld16(taddr + c0 + 16, u);
        tmem_ld_wait();
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) put(c0 + jj, v[jj]);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) put(c0 + 16 + jj, u[jj]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();  // the staging is complete; every tensor-memory read is done
  if (stamp && threadIdx.x == 0) stamp[kStampDrained] = globaltimer_ns();
  griddep_wait();   // before the first global write
  const int tid = static_cast<int>(threadIdx.x);
  // An item is 4 consecutive rows of one token (float4 of the staging).
  auto staged = [&](int j, int r4) {
    return ld_shared_v4(red_base + static_cast<uint32_t>((j * kTileRows + r4) * 4));
  };
  if (p.KG == 1) {
    for (int idx = tid; idx < mv * 32; idx += kPairThreads) {
      const int j = idx >> 5, r4 = (idx & 31) * 4;
      store_out4(p, mt * BN + j, t * kTileRows + r4, staged(j, r4));
    }
  } else {
    float* slot = p.xch + static_cast<size_t>(blockIdx.x) * BN * kTileRows;
    const int lo = min(jo0, mv);
    const int n_other = lo + max(mv - jo1, 0);
    for (int idx = tid; idx < n_other * 32; idx += kPairThreads) {
      const int jj = idx >> 5, r4 = (idx & 31) * 4;
      const int j = jj < lo ? jj : jj - lo + jo1;
      *reinterpret_cast<float4*>(slot + j * kTileRows + r4) = staged(j, r4);
    }
  }
  // Every CTA of the cluster is done with its tensor memory (and the pair's
  // MMAs with both CTAs' shared memory); with KG > 1 the barrier's release /
  // acquire also orders every CTA's exchange stores before the loads below.
  cluster_sync_all();
  if (stamp && threadIdx.x == 0) stamp[kStampCombine] = globaltimer_ns();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::kTmemCols);
  }
  if (p.KG == 1 || jo0 >= mv) {
    if (stamp && threadIdx.x == 0) stamp[kStampExit] = globaltimer_ns();
    return;
  }

  // ------------------------------------- combine across the cluster's pairs
  // Sum the owned tokens over the KG partials of these 128 rows (cluster
  // ranks 2 g' + h) in split order.  No CTA reads another's shared memory,
  // so none has to wait for the others before leaving.
  const int n_items = (min(jo1, mv) - jo0) * 32;
  const float* slot0 = p.xch + static_cast<size_t>(tm) * p.KG * 2 * BN * kTileRows;
  // Items (4 rows of one token) per thread per round trip: their loads from
  // the other pairs' slots are all in flight before the first is summed
  // (8 instead of 4: the unpooler at 256 tokens, KG = 2, 22.9 -> 22.5 us).
  constexpr int kItems = 8;
  for (int base = tid; base < n_items; base += kItems * kPairThreads) {
    float4 acc[kItems];
    int jl[kItems], r4[kItems];
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
      acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      const int idx = min(base + u * kPairThreads, n_items - 1);
      jl[u] = jo0 + (idx >> 5);
      r4[u] = (idx & 31) * 4;
    }
    for (int g0 = 0; g0 < p.KG; g0 += 4) {
      float4 v[kItems][4];
#pragma unroll
      for (int u = 0; u < kItems; ++u)
#pragma unroll
        for (int gg = 0; gg < 4; ++gg) {
          const int src = g0 + gg;
          if (src == g)
            v[u][gg] = staged(jl[u], r4[u]);
          else if (src < p.KG)
            v[u][gg] = ld_global_cg_v4(slot0 +
                                       (static_cast<size_t>(src) * 2 + h) * BN * kTileRows +
                                       static_cast<size_t>(jl[u]) * kTileRows + r4[u]);
        }
#pragma unroll
      for (int u = 0; u < kItems; ++u)
#pragma unroll
        for (int gg = 0; gg < 4; ++gg)
          if (g0 + gg < p.KG) {
            acc[u].x += v[u][gg].x;
            acc[u].y += v[u][gg].y;
            acc[u].z += v[u][gg].z;
            acc[u].w += v[u][gg].w;
          }
    }
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
      const int idx = base + u * kPairThreads;
      if (idx >= n_items) break;
      store_out4(p, mt * BN + jl[u], t * kTileRows + r4[u], acc[u]);
    }
  }
  if (stamp && threadIdx.x == 0) stamp[kStampExit] = globaltimer_ns();
}

template <int BN>
cudaError_t set_attr() {
  cudaError_t e = cudaFuncSetAttribute(tc_pair_kernel<BN>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(PCfg<BN>::kSmem));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(tc_pair_kernel<BN>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                              1);
}

template <int BN>
cudaLaunchConfig_t make_cfg(int ctas, int cluster, cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = PCfg<BN>::kSmem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <int BN>
cudaError_t launch(const CUtensorMap& tw, const CUtensorMap& tx, const PairParams& p,
                   int pair_tiles, cudaStream_t s) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = make_cfg<BN>(pair_tiles * p.MT * p.KG * 2, 2 * p.KG, s, attr);
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, tc_pair_kernel<BN>, tw, tx, p);
}

template <int BN>
int max_active(int kg) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg<BN>(2 * kg, 2 * kg, nullptr, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, tc_pair_kernel<BN>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace

bool pair_supported(int BN) { return BN == 64 || BN == 128 || BN == 256; }

cudaError_t pair_init_attributes() {
  cudaError_t e;
  if ((e = set_attr<64>()) != cudaSuccess) return e;
  if ((e = set_attr<128>()) != cudaSuccess) return e;
  return set_attr<256>();
}

int pair_max_active(int BN, int kg) {
  switch (BN) {
    case 64: return max_active<64>(kg);
    case 128: return max_active<128>(kg);
    case 256: return max_active<256>(kg);
  }
  return 0;
}

int pair_stages(int BN) {
  switch (BN) {
    case 64: return PCfg<64>::S;
    case 128: return PCfg<128>::S;
    case 256: return PCfg<256>::S;
  }
  return 0;
}

cudaError_t pair_launch(int BN, const CUtensorMap& tw, const CUtensorMap& tx, const PairParams& p,
                        int pair_tiles, cudaStream_t s) {
  switch (BN) {
    case 64: return launch<64>(tw, tx, p, pair_tiles, s);
    case 128: return launch<128>(tw, tx, p, pair_tiles, s);
    case 256: return launch<256>(tw, tx, p, pair_tiles, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace proj
