// router_cluster.cu -- the router (fp32 weights, fp32 output) from three
// tokens on: FP32 fused multiply-adds on the CUDA cores, split-K inside a
// thread-block cluster.
//
// out[i, n] = sum_k x[i, k] W[n, k]            (muse_bf16_proj guide, ch. 1, §1.1)
//
// The router keeps full FP32 precision (no TF32, no bf16 split): every
// product is the bf16 input widened exactly times the fp32 weight, summed
// in fp32 (guide ch. 1, §1.5; the router's 1e-4 bound).  Only the work
// layout is new:
//
// * An output tile is 128 weight rows x BN tokens (BN = 16..64; two row
//   tiles cover the 256 rows).  Like the tensor-core cluster kernel, each
//   tile is one cluster of CS CTAs (and KG clusters per tile when one
//   cluster per tile leaves SMs idle) splitting K; partials are combined in
//   a fixed order through distributed shared memory (cluster_common.cuh).
// * One producer thread streams 32 KB weight tiles (128 rows x 64 k, fp32,
//   16-byte chunks swizzled by row so that 16 consecutive rows read
//   conflict-free) with one bulk copy each, and the x tile with the same
//   128-byte-swizzled 2-D TMA load as the tensor-core kernel.
// * Eight compute warps.  At each stage a warp first widens (exactly) the
//   bf16 x of its 16 tokens over its k-range to fp32 in a private
//   shared-memory scratch, k-major (one 64-byte row of 16 tokens per k).  A
//   thread owns 8 rows x 8 tokens.  Per 4 k it loads its 8 rows' weights
//   (16-byte loads from the 32 KB tiles) and, per k, its 8 tokens' x as four
//   token pairs (two 16-byte loads, one address per half-warp), and issues
//   fma.rn.f32x2 with the weight in both halves against each token pair, so
//   every output is one fp32 sum in k order.  (The previous thread tile,
//   8 rows x 4 tokens with (even k, odd k) pairs, needed 36 shared-memory
//   wavefronts per warp for 64 pair-FMAs against 40 for 128 here; the
//   token pairs measured 1-2 us faster at 128-256 tokens and 5 us at 512.)
//   Narrow token tiles split each stage's 64 k among warp groups inside the
//   CTA; their partial tiles are added in group order.  Nine warps put three
//   on one of the SM's four schedulers, whose quarter of the register file
//   then holds about 170 registers per thread: the 8 x 8 tile takes 135-160.
// The pages' router runs cross-CTA split-K on warp-level FMAs/MMAs with an
// atomic epilogue (project report, Round 4; notebook n. 28, n. 38); here the
// combine is deterministic and there is one launch.
#include <cuda_bf16.h>

#include "cluster_common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace proj {
namespace {

constexpr int kSmemMax = 232448;

template <int BN>
struct RCfg {
  static_assert(BN >= 16 && BN <= 64, "token tile");
  static constexpr int kXBytes = BN * 128;  // bf16 [BN][64]
  static constexpr int kStage = kRfBytes + kXBytes;
  static constexpr int kComputeWarps = 8;
  static constexpr int kThreads = (kComputeWarps + 1) * 32;  // warp 0: producer
  static constexpr int kWpt = BN / 16;               // warps per token tile (16 tokens each)
  static constexpr int kKGroups = kComputeWarps / kWpt;  // k-groups inside the CTA
  static constexpr int kKPerGroup = kRfK / kKGroups;     // k of a stage per warp
  // per compute warp: its 16 tokens' x for its k-range of a stage, widened
  // to fp32, k-major ([kKPerGroup][16] floats, 64 bytes per k)
  static constexpr int kScrWarp = kKPerGroup * 64;
  static constexpr int kScrAll = kComputeWarps * kScrWarp;
  static constexpr int kFit = (kSmemMax - 1024 - 1024 - kScrAll) / kStage;
  static constexpr int S = kFit > 8 ? 8 : kFit;
  static constexpr size_t kRing = static_cast<size_t>(S) * kStage;
  static constexpr size_t kPart = static_cast<size_t>(kKGroups) * BN * kTileRows * 4;
  static constexpr size_t kData = kRing > kPart ? kRing : kPart;
  static constexpr size_t kSmem = 1024 + kData + kScrAll + (2 * S) * 8 + 16;
  static_assert(S >= 3, "pipeline too shallow");
  static_assert(kSmem <= kSmemMax, "shared memory budget");
  static_assert(kKPerGroup % 8 == 0, "k step");
};

__device__ __forceinline__ void ld_shared_2x64(uint32_t addr, uint64_t& a, uint64_t& b) {
  asm volatile("ld.shared.v2.u64 {%0,%1}, [%2];" : "=l"(a), "=l"(b) : "r"(addr));
}
// (acc.lo, acc.hi) += (w, w) * (x.lo, x.hi): one weight times two tokens
__device__ __forceinline__ void ffma2_bcast(uint64_t& acc, uint32_t w, uint64_t x) {
  asm("{\n\t.reg .b64 wp;\n\tmov.b64 wp, {%1, %1};\n\t"
      "fma.rn.f32x2 %0, wp, %2, %0;\n\t}"
      : "+l"(acc)
      : "r"(w), "l"(x));
}

// kXch: the partials are exchanged through L2 (p.xch), else through
// distributed shared memory (two instantiations, so that neither carries
// the other's code).
template <int BN, bool kXch>
__global__ void __launch_bounds__(RCfg<BN>::kThreads, 1)
    router_cluster_kernel(const __grid_constant__ CUtensorMap tmap_x, const ClusterParams p) {
  using C = RCfg<BN>;
  constexpr int S = C::S;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sW = smem_u32(smem);                    // [S][32 KB] weight tiles
  const uint32_t sX = sW + static_cast<uint32_t>(S) * kRfBytes;  // [S][BN x 128 B]
  // After the main loop: [kKGroups][BN][128] fp32 partials; group 0 becomes
  // the CTA's partial tile that the combine reads.
  const uint32_t part_base = sW;
  const uint32_t red_base = sW;
  const uint32_t sScr = sW + static_cast<uint32_t>(C::kData);  // per-warp fp32 x
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kData + C::kScrAll);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * S;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int cluster = static_cast<int>(blockIdx.x) / p.CS;
  const int tile = cluster / p.KG;
  const int grp = cluster % p.KG;
  const int t = tile / p.MT;
  const int mt = tile % p.MT;
  const int64_t split = static_cast<int64_t>(grp) * p.CS + rank;
  const int64_t nsplit = static_cast<int64_t>(p.KG) * p.CS;
  const int kb0 = static_cast<int>(split * p.KB / nsplit);
  const int kb1 = static_cast<int>((split + 1) * p.KB / nsplit);
  const int mv = min(BN, p.m - mt * BN);

  // Thread 0 (the producer) sets up the barriers and issues the weights of
  // the first ring's worth of stages before the CTA barrier: they are
  // constant, so they stream before the wait on the previous kernel of the
  // stream; x comes after that wait.
  const int pre = min(kb1 - kb0, S);
  uint64_t pol = 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, C::kComputeWarps);
    }
    fence_mbar_init();
    pol = policy_evict_first();
    for (int j = 0; j < pre; ++j) {
      const uint32_t fb = full0 + 8 * j;
      mbar_arrive_expect_tx(fb, kRfBytes + C::kXBytes);
      bulk_g2s(sW + j * kRfBytes, p.w + (static_cast<size_t>(t) * p.KB + kb0 + j) * kRfBytes,
               kRfBytes, fb, pol);
    }
    prefetch_tmap(&tmap_x);
  }
  griddep_launch_dependents();
  __syncwarp();
  __syncthreads();

  bool ok = true;
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      griddep_wait();
      for (int j = 0; j < pre; ++j)
        tma_load_2d(sX + j * C::kXBytes, &tmap_x, (kb0 + j) * kRfK, mt * BN, full0 + 8 * j);
      int64_t issued = pre;
      for (int kb = kb0 + pre; kb < kb1; ++kb) {
        const int s = static_cast<int>(issued % S);
        if (!mbar_wait(empty0 + 8 * s, static_cast<uint32_t>(((issued / S) & 1) ^ 1), p.status,
                       kStatusTimeoutProducer))
          break;
        const uint32_t fb = full0 + 8 * s;
        mbar_arrive_expect_tx(fb, kRfBytes + C::kXBytes);
        bulk_g2s(sW + s * kRfBytes, p.w + (static_cast<size_t>(t) * p.KB + kb) * kRfBytes,
                 kRfBytes, fb, pol);
        tma_load_2d(sX + s * C::kXBytes, &tmap_x, kb * kRfK, mt * BN, fb);
        ++issued;
      }
      // Wait (bounded) for the copies still in flight before the ring is
      // reused for the partial tiles.
      const int64_t n = issued < S ? issued : S;
      for (int64_t j = 0; j < n; ++j) {
        const int64_t idx = issued - 1 - j;
        mbar_wait(full0 + 8 * static_cast<int>(idx % S), static_cast<uint32_t>((idx / S) & 1),
                  p.status, kStatusTimeoutDrain);
      }
    }
  }

  // ---------------------------------------------------------- compute warps
  const int cw = warp - 1;
  const int tt = cw % C::kWpt;        // token sub-tile of 16
  const int kg = cw / C::kWpt;        // k-group inside the CTA
  const int rg = lane & 15;           // rows rg + 16 i
  const int tg = lane >> 4;           // tokens 16 tt + 8 tg + 2 q + {0, 1} (pair q)
  uint64_t acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[i][q] = 0ull;
  if (warp > 0) {
    int64_t j = 0;
    for (int kb = kb0; kb < kb1; ++kb, ++j) {
      const int s = static_cast<int>(j % S);
      if (!mbar_wait_sleep(full0 + 8 * s, static_cast<uint32_t>((j / S) & 1), p.status,
                           kStatusTimeoutMma)) {
        ok = false;
        break;
      }
      const uint32_t wst = sW + s * kRfBytes;
      const uint32_t xst = sX + s * C::kXBytes;
      // Widen this warp's 16 tokens x its k-range of the stage to fp32 once,
      // k-major (16-byte chunks of the 128-byte-swizzled bf16 tile).
      const uint32_t scr = sScr + static_cast<uint32_t>(cw * C::kScrWarp);
      {
        constexpr int kCh = C::kKPerGroup / 8;  // 16-byte bf16 chunks per token
#pragma unroll
        for (int idx = lane; idx < 16 * kCh; idx += 32) {
          const int t16 = idx & 15, cc = idx >> 4;
          const int jt = 16 * tt + t16;
          const int kc = kg * kCh + cc;
          const uint4 v = ld_shared_u4(xst + jt * 128 + ((kc ^ (jt & 7)) << 4));
          const uint32_t a = scr + static_cast<uint32_t>(cc * 8 * 64 + t16 * 4);
          const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            st_shared_f32(a + (2 * e) * 64, __uint_as_float(w4[e] << 16));
            st_shared_f32(a + (2 * e + 1) * 64, __uint_as_float(w4[e] & 0xFFFF0000u));
          }
        }
        __syncwarp();
      }
#pragma unroll
      for (int kk = 0; kk < C::kKPerGroup; kk += 4) {
        const int k0 = kg * C::kKPerGroup + kk;
        const int c = k0 >> 2;  // 16-byte weight chunk
        uint4 w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = rg + 16 * i;
          w[i] = ld_shared_u4(wst + r * 256 + ((c ^ (r & 15)) << 4));
        }
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          uint64_t xq[4];  // token pairs (0,1) (2,3) (4,5) (6,7) of the lane's eight
          ld_shared_2x64(scr + (kk + k4) * 64 + tg * 32, xq[0], xq[1]);
          ld_shared_2x64(scr + (kk + k4) * 64 + tg * 32 + 16, xq[2], xq[3]);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t wk = k4 == 0 ? w[i].x : k4 == 1 ? w[i].y : k4 == 2 ? w[i].z : w[i].w;
#pragma unroll
            for (int q = 0; q < 4; ++q) ffma2_bcast(acc[i][q], wk, xq[q]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);
    }
  }
  // Every copy has landed and every stage has been read: the ring becomes
  // the partial-tile area.  (__syncthreads is an aligned barrier: warp 0,
  // whose lane 0 ran the producer loop alone, reconverges first.)
  __syncwarp();
  __syncthreads();
  if (warp > 0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int r = rg + 16 * i;
        const int jt = 16 * tt + 8 * tg + 2 * q;
        st_shared_f32(part_base + static_cast<uint32_t>(((kg * BN + jt) * kTileRows + r) * 4),
                      __uint_as_float(static_cast<uint32_t>(acc[i][q])));
        st_shared_f32(part_base + static_cast<uint32_t>(((kg * BN + jt + 1) * kTileRows + r) * 4),
                      __uint_as_float(static_cast<uint32_t>(acc[i][q] >> 32)));
      }
    }
  }
  __syncthreads();
  if constexpr (C::kKGroups > 1) {
    // the k-groups' partial tiles, added in group order into group 0's
    for (int idx = threadIdx.x; idx < BN * kTileRows / 4; idx += C::kThreads) {
      const uint32_t off = static_cast<uint32_t>(idx * 16);
      float4 a = ld_shared_v4(part_base + off);
#pragma unroll
      for (int g = 1; g < C::kKGroups; ++g) {
        const float4 b = ld_shared_v4(part_base + g * BN * kTileRows * 4 + off);
        a.x += b.x;
        a.y += b.y;
        a.z += b.z;
        a.w += b.w;
      }
      asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(red_base + off), "f"(a.x),
                   "f"(a.y), "f"(a.z), "f"(a.w)
                   : "memory");
    }
  }
  if constexpr (kXch) {
    // L2 exchange: the tokens this rank does not own go to the CTA's
    // exchange slot (after the wait: the previous kernel of the stream may
    // be this handle's previous call, still reading it).
    __syncthreads();
    griddep_wait();
    const int jo0 = static_cast<int>(rank) * BN / p.CS;
    const int jo1 = static_cast<int>(rank + 1) * BN / p.CS;
    float* slot = p.xch + static_cast<size_t>(blockIdx.x) * BN * kTileRows;
    for (int idx = threadIdx.x; idx < BN * kTileRows / 4; idx += C::kThreads) {
      const int j = idx / (kTileRows / 4);
      if (j >= jo0 && j < jo1) continue;
      *reinterpret_cast<float4*>(slot + idx * 4) = ld_shared_v4(red_base + idx * 16);
    }
  }
  __syncwarp();
  // Every CTA of the cluster has its partial in shared memory (and, with the
  // L2 exchange, in its exchange slot).
  cluster_sync_all();
  griddep_wait();  // before the first global write of this thread
  if constexpr (kXch) {
    cluster_combine_l2<BN, C::kThreads, 1>(p, red_base, cluster, tile, t, mt, rank, mv);
  } else {
    cluster_combine<BN, C::kThreads, 1>(p, red_base, cluster, tile, t, mt, rank, mv);
    // No CTA may leave while a peer still reads its shared memory.
    cluster_sync_all();
  }
  (void)ok;
}

template <int BN, bool kXch>
cudaError_t set_attr_one() {
  cudaError_t e = cudaFuncSetAttribute(router_cluster_kernel<BN, kXch>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(RCfg<BN>::kSmem));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(router_cluster_kernel<BN, kXch>,
                              cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
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
  cfg.blockDim = dim3(RCfg<BN>::kThreads);
  cfg.dynamicSmemBytes = RCfg<BN>::kSmem;
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
  return p.xch ? cudaLaunchKernelEx(&cfg, router_cluster_kernel<BN, true>, tmap, p)
                : cudaLaunchKernelEx(&cfg, router_cluster_kernel<BN, false>, tmap, p);
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
  if (cudaOccupancyMaxActiveClusters(&n, router_cluster_kernel<BN, false>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace

cudaError_t router_cluster_init_attributes() {
  cudaError_t e;
  if ((e = set_attr<16>()) != cudaSuccess) return e;
  if ((e = set_attr<32>()) != cudaSuccess) return e;
  if ((e = set_attr<64>()) != cudaSuccess) return e;
  return cudaSuccess;
}

int router_cluster_max_active(int BN, int cs) {
  switch (BN) {
    case 16: return max_clusters<16>(cs);
    case 32: return max_clusters<32>(cs);
    case 64: return max_clusters<64>(cs);
  }
  return 0;
}

int router_cluster_stages(int BN) {
  switch (BN) {
    case 16: return RCfg<16>::S;
    case 32: return RCfg<32>::S;
    case 64: return RCfg<64>::S;
  }
  return 0;
}

cudaError_t router_cluster_launch(int BN, const CUtensorMap& tmap, const ClusterParams& p,
                                  cudaStream_t s) {
  switch (BN) {
    case 16: return launch<16>(tmap, p, s);
    case 32: return launch<32>(tmap, p, s);
    case 64: return launch<64>(tmap, p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace proj
