// router.cu -- the router projection with fp32 weights, fp32 output and fp32
// fused multiply-adds (no TF32, no bf16 split of the weights).
//
// out[i, n] = sum_k float(x[i, k]) * W[n, k],  W fp32 [256, 8192]
// (muse_bf16_proj guide, ch. 1, §1.1; the router's tighter 0.01 % bound,
// §1.5, is why its weights keep full fp32 precision).
//
// Design: one CTA per SM (cooperative launch); the (m-tile, 64-row tile,
// 64-column block) units are cut into G equal ranges as in the tensor-core
// path (the router has only 256 rows, so K must be split to fill 152 SMs:
// muse_bf16_proj notebook, n. 12 "Why the router needs special care").
// Thread 0 streams the 16 KB prepacked weight tiles with bulk copies and the
// bf16 x block with a 2-D TMA load into an 8-stage ring; all 256 threads
// widen x to fp32 in a swizzled shared buffer and run a 4-row x 4-token
// register tile of FMAs per thread.  For small token tiles the threads also
// split each 64-column block into k-groups (KS = 64 / TM), reduced through
// shared memory in fixed order at the end of a segment.  Shared tiles are
// combined in fixed CTA order (splitk.cuh, owner or distributed mode).
#include "kernels.h"
#include "ptx.cuh"
#include "splitk.cuh"

namespace proj {
namespace {

constexpr int kThreads = 256;
constexpr int kStages = 8;
constexpr int kRedFloats = 4096;  // KS * 64 * TM == 4096 for every TM

template <int TM>
struct RCfg {
  static constexpr int kXbBytes = TM * 128;           // bf16 x block [TM][64]
  static constexpr int kStageBytes = kRtBytes + kXbBytes;
  static constexpr int kXfBytes = TM * 256;           // fp32 x block [TM][64]
  static constexpr int KS = 64 / TM;                  // k-groups
  static constexpr int kGroupThreads = kThreads / KS; // = 4 TM
  static constexpr int kKPerGroup = 64 / KS;          // columns per k-group per stage
  static constexpr size_t kSmem =
      1024 + kStages * kStageBytes + kXfBytes + kRedFloats * 4 + kStages * 8 + 16;
  static_assert(kSmem <= 232448, "shared memory budget");
};

template <int TM>
__global__ void __launch_bounds__(kThreads, 1)
    router_kernel(const __grid_constant__ CUtensorMap tmap_x, const RouterParams p) {
  using C = RCfg<TM>;
  constexpr int64_t kSlot = 64 * TM;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sW = smem;                                   // kStages x 16 KB
  uint8_t* sXb = sW + kStages * kRtBytes;               // kStages x TM*128
  float* sXf = reinterpret_cast<float*>(sXb + kStages * C::kXbBytes);
  float* sRed = sXf + TM * 64;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sRed + kRedFloats);
  const uint32_t full0 = smem_u32(bars);

  const int tid = threadIdx.x;
  const int kg = tid / C::kGroupThreads;
  const int g = tid % C::kGroupThreads;
  const int tr = g & 15;        // rows tr + 16 j
  const int tt = g >> 4;        // tokens tt + (TM / 4) j
  const int64_t G = p.G;
  const int64_t U = static_cast<int64_t>(p.MT) * p.T * p.KB;
  const int64_t cta = blockIdx.x;
  const int64_t u0 = part_begin(cta, U, G);
  const int64_t u1 = part_begin(cta + 1, U, G);
  const int64_t nunits = u1 - u0;
  const int64_t first_tile = u0 / p.KB;
  const bool owner_mode = (p.reduce == 0);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(full0 + 8 * s, 1);
    fence_mbar_init();
    prefetch_tmap(&tmap_x);
  }
  __syncthreads();

  const uint64_t pol = policy_evict_first();
  auto issue = [&](int64_t j) {  // unit u0 + j into stage j % kStages
    const int64_t u = u0 + j;
    const int tile = static_cast<int>(u / p.KB);
    const int kb = static_cast<int>(u % p.KB);
    const int t = tile / p.MT, mt = tile % p.MT;
    const int s = static_cast<int>(j % kStages);
    const uint32_t fb = full0 + 8 * s;
    mbar_arrive_expect_tx(fb, kRtBytes + C::kXbBytes);
    bulk_g2s(smem_u32(sW + s * kRtBytes), p.w + (static_cast<size_t>(t) * p.KB + kb) * kRtBytes,
             kRtBytes, fb, pol);
    tma_load_2d(smem_u32(sXb + s * C::kXbBytes), &tmap_x, kb * kRtK, mt * TM, fb);
  };
  int64_t issued = 0;  // meaningful in thread 0 only
  if (tid == 0) {
    for (; issued < nunits && issued < kStages; ++issued) issue(issued);
  }

  float acc[4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;

  bool ok = true;
  int seg_kb0 = 0;
  int pend[2];
  int npend = 0;
  for (int64_t j = 0; j < nunits; ++j) {
    const int64_t u = u0 + j;
    const int tile = static_cast<int>(u / p.KB);
    const int kb = static_cast<int>(u % p.KB);
    if (j == 0 || kb == 0) seg_kb0 = kb;
    const int s = static_cast<int>(j % kStages);
    if (!mbar_wait(full0 + 8 * s, static_cast<uint32_t>((j / kStages) & 1), p.status,
                   kStatusTimeoutMma)) {
      ok = false;
    }
    // Abort is uniform: a timed-out thread still joins the barriers below.
    if (__syncthreads_or(!ok)) {
      ok = false;
      break;
    }
    // Widen x (bf16 [TM][64]) to fp32, swizzled: row i, float4 q at q ^ (i & 7).
    {
      const uint16_t* xb = reinterpret_cast<const uint16_t*>(sXb + s * C::kXbBytes);
      for (int e = tid * 4; e < TM * 64; e += kThreads * 4) {
        const int i = e >> 6, k = e & 63;
        const uint2 v = *reinterpret_cast<const uint2*>(xb + e);
        float4 f;
        f.x = __uint_as_float(v.x << 16);
        f.y = __uint_as_float(v.x & 0xFFFF0000u);
        f.z = __uint_as_float(v.y << 16);
        f.w = __uint_as_float(v.y & 0xFFFF0000u);
        *reinterpret_cast<float4*>(sXf + i * 64 + (((k >> 2) ^ (i & 7)) << 2)) = f;
      }
    }
    __syncthreads();
    {
      const float* w = reinterpret_cast<const float*>(sW + s * kRtBytes);
#pragma unroll 4
      for (int qq = 0; qq < C::kKPerGroup / 4; ++qq) {
        const int q = kg * (C::kKPerGroup / 4) + qq;
        float4 wv[4], xv[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const int r = tr + 16 * a;
          wv[a] = *reinterpret_cast<const float4*>(w + r * 64 + ((q ^ (r & 7)) << 2));
        }
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int i = tt + (TM / 4) * b;
          xv[b] = *reinterpret_cast<const float4*>(sXf + i * 64 + ((q ^ (i & 7)) << 2));
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            float c = acc[a][b];
            c = fmaf(wv[a].x, xv[b].x, c);
            c = fmaf(wv[a].y, xv[b].y, c);
            c = fmaf(wv[a].z, xv[b].z, c);
            c = fmaf(wv[a].w, xv[b].w, c);
            acc[a][b] = c;
          }
      }
    }
    __syncthreads();  // stage s and sXf are free
    if (tid == 0 && issued < nunits) issue(issued++);

    const bool seg_end = (kb == p.KB - 1) || (j == nunits - 1);
    if (!seg_end) continue;

    // ---------------------------------------------------------- epilogue
    const int t = tile / p.MT, mt = tile % p.MT;
    const int mv = min(TM, p.m - mt * TM);
    const bool whole = (seg_kb0 == 0 && kb == p.KB - 1);
    const bool owner = owner_mode && !whole && seg_kb0 == 0;
    // k-group partials -> sRed[kg][row][token], then fixed-order sum over kg.
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        sRed[(kg * 64 + tr + 16 * a) * TM + tt + (TM / 4) * b] = acc[a][b];
        acc[a][b] = 0.f;
      }
    __syncthreads();
    TileSplit ts{0, 0};
    if (owner) {
      ts = tile_split(tile, p.KB, U, G);
      if (!spin_until_ge(p.counters + tile,
                         static_cast<uint32_t>(ts.c_last - ts.c_first), p.status))
        ok = false;
    }
    float* slot = p.ws + (owner_mode ? cta : 2 * cta + (tile == first_tile ? 0 : 1)) * kSlot;
    for (int o = tid; o < 64 * TM; o += kThreads) {
      const int r = o % 64, i = o / 64;
      if (i >= mv) continue;
      float v = 0.f;
      for (int gk = 0; gk < C::KS; ++gk) v += sRed[(gk * 64 + r) * TM + i];
      float* dst = p.out + (static_cast<size_t>(mt) * TM + i) * 256 + t * 64 + r;
      if (whole) {
        *dst = v;
      } else if (owner) {
        const float* base = p.ws + i * 64 + r;
        float pre = 0.f;
        for (int64_t c = ts.c_first + 1; c <= ts.c_last; c += 8) {
          float w8[8];
#pragma unroll
          for (int a = 0; a < 8; ++a) w8[a] = (c + a <= ts.c_last) ? __ldcg(base + (c + a) * kSlot) : 0.f;
#pragma unroll
          for (int a = 0; a < 8; ++a) pre += w8[a];
        }
        *dst = v + pre;
      } else {
        slot[i * 64 + r] = v;
      }
    }
    if (!whole) {
      if (owner) {
        __syncthreads();
        if (tid == 0) p.counters[tile] = 0u;
      } else {
        // the barrier orders every thread's partial stores before thread 0's
        // release (cumulative; one arrival per CTA)
        __syncthreads();
        if (tid == 0) red_release_gpu_add(p.counters + tile, 1u);
        if (!owner_mode) pend[npend++] = tile;
      }
    }
    __syncthreads();  // sRed reuse
  }

  // distributed mode: this CTA's share of each split tile it touched, as
  // float4 runs of 4 rows, 4 runs and 4 contributors in flight per thread.
  for (int i = 0; ok && i < npend; ++i) {
    const int tile = pend[i];
    const TileSplit ts = tile_split(tile, p.KB, U, G);
    const int64_t S = ts.c_last - ts.c_first + 1;
    if (!spin_until_ge(p.counters + tile, static_cast<uint32_t>(S), p.status)) break;
    const int t = tile / p.MT, mt = tile % p.MT;
    const int mv = min(TM, p.m - mt * TM);
    const int64_t nq = 16 * static_cast<int64_t>(mv);
    const int64_t me = cta - ts.c_first;
    const int64_t q0 = me * nq / S, q1 = (me + 1) * nq / S;
    const int64_t s_first =
        2 * ts.c_first + ((part_begin(ts.c_first, U, G) / p.KB) == tile ? 0 : 1);
    const float4* ws4 = reinterpret_cast<const float4*>(p.ws);
    constexpr int64_t kSlot4 = kSlot / 4;
    for (int64_t qb = q0 + tid; qb < q1; qb += kThreads * 4) {
      float4 acc[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int64_t q = qb + kThreads * b;
        acc[b] = q < q1 ? __ldcg(ws4 + s_first * kSlot4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      for (int64_t c = ts.c_first + 1; c <= ts.c_last; c += 4) {
        float4 v[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const int64_t q = qb + kThreads * b;
            v[a][b] = (c + a <= ts.c_last && q < q1) ? __ldcg(ws4 + 2 * (c + a) * kSlot4 + q)
                                                     : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            acc[b].x += v[a][b].x;
            acc[b].y += v[a][b].y;
            acc[b].z += v[a][b].z;
            acc[b].w += v[a][b].w;
          }
      }
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int64_t q = qb + kThreads * b;
        if (q < q1) {
          const int ii = static_cast<int>(q / 16), r = static_cast<int>(q % 16) * 4;
          *reinterpret_cast<float4*>(p.out + (static_cast<size_t>(mt) * TM + ii) * 256 + t * 64 + r) =
              acc[b];
        }
      }
    }
    __syncthreads();
    if (tid == 0) {
      const uint32_t old = atomicAdd(p.counters + tile, 1u);
      if (old == static_cast<uint32_t>(2 * S - 1)) p.counters[tile] = 0u;
    }
  }

  // Drain copies still in flight (only after an abort): the last kStages
  // issued units may not have been waited on.
  if (tid == 0 && !ok) {
    for (int64_t j = issued > kStages ? issued - kStages : 0; j < issued; ++j) {
      mbar_wait(full0 + 8 * static_cast<int>(j % kStages), static_cast<uint32_t>((j / kStages) & 1),
                p.status, kStatusTimeoutDrain);
    }
  }
}

template <int TM>
cudaError_t set_attr() {
  return cudaFuncSetAttribute(router_kernel<TM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(RCfg<TM>::kSmem));
}

template <int TM>
cudaError_t launch(const CUtensorMap& tmap, const RouterParams& p, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = RCfg<TM>::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, router_kernel<TM>, tmap, p);
}

}  // namespace

bool router_supported(int TM) { return TM == 4 || TM == 8 || TM == 16 || TM == 32 || TM == 64; }

size_t router_smem_bytes(int TM) {
  switch (TM) {
    case 4: return RCfg<4>::kSmem;
    case 8: return RCfg<8>::kSmem;
    case 16: return RCfg<16>::kSmem;
    case 32: return RCfg<32>::kSmem;
    case 64: return RCfg<64>::kSmem;
  }
  return 0;
}

cudaError_t router_init_attributes() {
  cudaError_t e;
  if ((e = set_attr<4>()) != cudaSuccess) return e;
  if ((e = set_attr<8>()) != cudaSuccess) return e;
  if ((e = set_attr<16>()) != cudaSuccess) return e;
  if ((e = set_attr<32>()) != cudaSuccess) return e;
  if ((e = set_attr<64>()) != cudaSuccess) return e;
  return cudaSuccess;
}

cudaError_t router_launch(int TM, const CUtensorMap& tmap, const RouterParams& p, cudaStream_t s) {
  switch (TM) {
    case 4: return launch<4>(tmap, p, s);
    case 8: return launch<8>(tmap, p, s);
    case 16: return launch<16>(tmap, p, s);
    case 32: return launch<32>(tmap, p, s);
    case 64: return launch<64>(tmap, p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace proj
