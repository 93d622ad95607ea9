// gemm_cluster.cu -- tensor-core GEMM, split-K inside a thread-block
// cluster, the partials combined through L2 or distributed shared memory:
// the dispatch form of the bf16 layers above the few-token GEMVs (qkv_gate
// and the pooler from 9 tokens, o from 17 to 128, the unpooler from 9 to
// 191; the CTA-pair kernel takes o above 128 tokens and the unpooler from
// 192) and, on request only (PROJ_VARIANT_PLANES3), the router with its fp32
// weights as three exact bf16 planes.  The router's dispatch form is the
// FP32-FMA path at every token count (router_cluster.cu and the router GEMVs).
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
// Router, opt-in form: W (fp32) was split at prepare into bf16 planes
// hi + mid + lo == W exactly, stored as the tiles of a [N, 3K] bf16 matrix.
// Weight k-block kb meets x k-block kb % KBx, so x @ [hi | mid | lo].T
// accumulates the three exact bf16 x bf16 products of every weight in fp32
// -- the same sum as fp32 weights, without TF32 truncation -- and the
// result is stored as fp32.
#include <cuda_bf16.h>

#include "cluster_common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace proj {
namespace {

constexpr int kSmemLimit = 232448;
// Weight stages the producer issues before the wait on the previous kernel
// of the stream; the rest of the first ring follows x.  Measured on GB300
// (device time after an L2 flush): issuing the whole ring early queues the
// first x tiles behind every SM's weight burst -- the first MMA started
// ~2.7 us after entry at 256 tokens -- and two early stages took 1.0-1.5 us
// off each bf16 layer at 128 tokens (qkv_gate 15.2 -> 14.0 us, pooler
// 18.5 -> 17.0); zero early stages was no better than two.
constexpr int kClusterEarlyStages = 2;

template <int BN>
struct CCfg {
  static constexpr int kXBytes = BN * 128;
  static constexpr int kStage = kTileBytes + kXBytes;
  // Narrow token tiles (the weight-streaming regime) take half an SM's
  // shared memory, so that the next kernel of the stream -- launched early
  // by programmatic dependent launch -- can sit beside this one and stream
  // its first weights during this kernel's tail; wide tiles keep the SM.
  static constexpr bool kHalfSm = BN <= 64;
  static constexpr int kBlocksPerSm = kHalfSm ? 2 : 1;
  static constexpr int kBudget = kHalfSm ? 113 * 1024 : kSmemLimit;
  static constexpr int kFit = (kBudget - 1024 - 1024) / kStage;
  static constexpr int S = kFit > 12 ? 12 : kFit;
  // warp 0 copies, warp 1 issues MMAs, the next kDrainWarps drain the
  // accumulator (one or two per tensor-memory lane quarter), and every warp
  // combines the cluster's partials.
  static constexpr int kThreads = kHalfSm ? 192 : 384;
  static constexpr int kDrainWarps = kHalfSm ? 4 : 8;
  static constexpr int kTmemCols = BN < 32 ? 32 : BN;
  static constexpr size_t kRing = static_cast<size_t>(S) * kStage;
  static constexpr size_t kRed = static_cast<size_t>(BN) * kTileRows * 4;  // [BN][128] fp32
  static constexpr size_t kData = kRing > kRed ? kRing : kRed;
  static constexpr size_t kSmem = 1024 + kData + (2 * S + 2) * 8 + 16;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(128, BN);
  static_assert(S >= 3, "pipeline too shallow");
  static_assert(kSmem <= kSmemLimit, "shared memory budget");
};

// kXch: the partials are exchanged through L2 (p.xch), else through
// distributed shared memory (two instantiations, so that neither carries
// the other's code).
template <int BN, bool kXch>
__global__ void __launch_bounds__(CCfg<BN>::kThreads, CCfg<BN>::kBlocksPerSm)
    tc_cluster_kernel(const __grid_constant__ CUtensorMap tmap_x, const ClusterParams p) {
  using C = CCfg<BN>;
  constexpr int S = C::S;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + static_cast<size_t>(S) * kTileBytes;
  // [BN][128] fp32 accumulator staging; reuses the ring after the last MMA
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
  const int cluster = static_cast<int>(blockIdx.x) / p.CS;
  const int tile = cluster / p.KG;   // output tile (t, mt)
  const int grp = cluster % p.KG;    // which of the tile's KG clusters
  const int t = tile / p.MT;
  const int mt = tile % p.MT;
  const int64_t split = static_cast<int64_t>(grp) * p.CS + rank;  // K slice of this CTA
  const int64_t nsplit = static_cast<int64_t>(p.KG) * p.CS;
  const int kb0 = static_cast<int>(split * p.KB / nsplit);
  const int kb1 = static_cast<int>((split + 1) * p.KB / nsplit);
  const int mv = min(BN, p.m - mt * BN);

  // Thread 0 (the producer) sets up the barriers and issues the weights of
  // the first kClusterEarlyStages stages before the CTA barrier: they are
  // constant, so they stream before the wait on the previous kernel of the
  // stream; x and every global write come after that wait.
  const int pre = min(kb1 - kb0, S);
  const int pre_w = min(pre, kClusterEarlyStages);  // weight stages issued before the wait
  uint64_t pol = 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(accf, 1);
    fence_mbar_init();
    pol = policy_evict_first();
    for (int j = 0; j < pre_w; ++j) {
      const uint32_t fb = full0 + 8 * j;
      mbar_arrive_expect_tx(fb, kTileBytes + C::kXBytes);
      bulk_g2s(smem_u32(sA + j * kTileBytes),
               p.w + (static_cast<size_t>(t) * p.KB + kb0 + j) * kTileBytes, kTileBytes, fb,
               pol);
    }
    prefetch_tmap(&tmap_x);
  }
  griddep_launch_dependents();
  __syncwarp();
  __syncthreads();
  // The producer starts streaming at once; the tensor-memory allocation runs
  // meanwhile and is published to the MMA and epilogue warps (1..5) only.
  uint32_t tmem = 0;
  if (warp >= 1) {
    if (warp == 1) {
      tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
      tmem_relinquish();
    }
    tc_fence_before();
    named_bar_sync(1, C::kThreads - 32);
    tc_fence_after();
    tmem = *tmem_slot;
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      griddep_wait();
      if (stamp) stamp[kStampDepWait] = globaltimer_ns();
      for (int j = 0; j < pre_w; ++j)
        tma_load_2d(smem_u32(sB + j * C::kXBytes), &tmap_x, ((kb0 + j) % p.KBx) * kTileK,
                    mt * BN, full0 + 8 * j);
      for (int j = pre_w; j < pre; ++j) {  // the rest of the first ring: weights, then x
        const uint32_t fb = full0 + 8 * j;
        mbar_arrive_expect_tx(fb, kTileBytes + C::kXBytes);
        bulk_g2s(smem_u32(sA + j * kTileBytes),
                 p.w + (static_cast<size_t>(t) * p.KB + kb0 + j) * kTileBytes, kTileBytes, fb,
                 pol);
        tma_load_2d(smem_u32(sB + j * C::kXBytes), &tmap_x, ((kb0 + j) % p.KBx) * kTileK,
                    mt * BN, fb);
      }
      int64_t issued = pre;
      for (int kb = kb0 + pre; kb < kb1; ++kb) {
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
        if (stamp && j == 0) stamp[kStampFirstFull] = globaltimer_ns();
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
      if (stamp) stamp[kStampLastMma] = globaltimer_ns();
    }
  } else if (warp < 2 + C::kDrainWarps) {
    // ------------------------------------- epilogue: accumulator -> smem
    const int q = warp & 3;            // lane quarter this warp may access
    const int part = (warp - 2) >> 2;  // column part
    constexpr int kParts = (C::kDrainWarps == 8 && BN >= 32) ? 2 : 1;
    constexpr int kCols = BN / kParts;
    const int r = q * 32 + lane;
    if (part < kParts && mbar_wait(accf, 0, p.status, kStatusTimeoutEpilogue)) {
      if (stamp && warp == 2 && lane == 0) stamp[kStampAccReady] = globaltimer_ns();
      tc_fence_after();
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16);
      const int c_beg = part * kCols;
      // Tokens this rank owns stay in shared memory; with the L2 exchange the
      // others go to this CTA's exchange slot (32 rows of a token: 128
      // contiguous bytes per warp store).
      float* slot = kXch ? p.xch + static_cast<size_t>(blockIdx.x) * BN * kTileRows : nullptr;
      // (the previous kernel of the stream may be this handle's previous
      // call, still reading the exchange: wait for it before storing)
      if constexpr (kXch) griddep_wait();
      const int jo0 = static_cast<int>(rank) * BN / p.CS;
      const int jo1 = static_cast<int>(rank + 1) * BN / p.CS;
      auto drain = [&](auto put) {
        if constexpr (kCols == 16) {
          float v[16];
          tmem_ld16(taddr + c_beg, v);
          tmem_ld_wait();
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) put(c_beg + jj, v[jj]);
        } else {
          // two loads in flight per wait
#pragma unroll 1
          for (int c0 = c_beg; c0 < c_beg + kCols; c0 += 32) {
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
      };
      if constexpr (kXch) {
        drain([&](int c, float val) {
          if (c < jo0 || c >= jo1)
            slot[c * kTileRows + r] = val;
          else
            st_shared_f32(red_base + static_cast<uint32_t>((c * kTileRows + r) * 4), val);
        });
      } else {
        drain([&](int c, float val) {
          st_shared_f32(red_base + static_cast<uint32_t>((c * kTileRows + r) * 4), val);
        });
      }
      tc_fence_before();
      if (stamp && warp == 2 && lane == 0) stamp[kStampDrained] = globaltimer_ns();
    }
  }
  __syncwarp();
  // Every CTA of the cluster has its partial in shared memory (and, with the
  // L2 exchange, in its exchange slot; the barrier's release/acquire orders
  // those global stores too).
  cluster_sync_all();
  if (stamp && threadIdx.x == 0) stamp[kStampCombine] = globaltimer_ns();
  griddep_wait();  // before the first global write of this thread
  if constexpr (kXch) {
    cluster_combine_l2<BN, C::kThreads>(p, red_base, cluster, tile, t, mt, rank, mv);
  } else {
    cluster_combine<BN, C::kThreads>(p, red_base, cluster, tile, t, mt, rank, mv);
    // No CTA may leave while a peer still reads its shared memory.
    cluster_sync_all();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (stamp && threadIdx.x == 0) stamp[kStampExit] = globaltimer_ns();
}

template <int BN, bool kXch>
cudaError_t set_attr_one() {
  cudaError_t e = cudaFuncSetAttribute(tc_cluster_kernel<BN, kXch>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(CCfg<BN>::kSmem));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(tc_cluster_kernel<BN, kXch>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                              1);
}

template <int BN>
cudaError_t set_attr() {
  cudaError_t e = set_attr_one<BN, false>();
  if (e != cudaSuccess) return e;
  return set_attr_one<BN, true>();
}

template <int BN>
cudaLaunchConfig_t make_cfg(const ClusterParams& p, cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.MT * p.T * p.KG * p.CS);
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
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = make_cfg<BN>(p, s, attr);
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 2;
  return p.xch ? cudaLaunchKernelEx(&cfg, tc_cluster_kernel<BN, true>, tmap, p)
                : cudaLaunchKernelEx(&cfg, tc_cluster_kernel<BN, false>, tmap, p);
}

template <int BN>
int max_clusters(int cs) {
  ClusterParams p = {};
  p.MT = 1;
  p.T = 1;
  p.KG = 1;
  p.CS = cs;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg<BN>(p, nullptr, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, tc_cluster_kernel<BN, false>, &cfg) != cudaSuccess) {
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

int cluster_blocks_per_sm(int BN) {
  switch (BN) {
    case 16: return CCfg<16>::kBlocksPerSm;
    case 32: return CCfg<32>::kBlocksPerSm;
    case 64: return CCfg<64>::kBlocksPerSm;
    case 128: return CCfg<128>::kBlocksPerSm;
    case 256: return CCfg<256>::kBlocksPerSm;
  }
  return 1;
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
