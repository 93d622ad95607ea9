// gemv.cu -- streaming GEMV for small token counts (m <= 2), bf16 or fp32
// weights, fp32 fused multiply-adds on the CUDA cores, no tensor memory.
//
// out[i, n] = sum_k x[i, k] W[n, k]            (muse_bf16_proj guide, ch. 1, §1.1)
//
// At m <= 2 the projection is a weight stream with a few FMAs per weight
// (guide ch. 1, §1.7: about m FLOPs per byte), so the design is about
// streaming and about the tail:
//
// * W stays row-major.  Each row is cut into chunks of 1024 consecutive
//   weights (k-slices: K / 1024 per row, 8 for K = 8192), and the chunks of
//   the whole matrix, in row-major order, are split into G equal contiguous
//   runs, one per CTA (one CTA per SM).  Every CTA therefore streams the same
//   number of bytes and, with runs of at least one row, only the first and
//   the last row of a run can be shared with a neighbour.
// * One producer thread streams 8-chunk stages (16 KB bf16 / 32 KB fp32)
//   with bulk copies into a 12 / 6 stage ring.  Eight compute warps: warp w
//   takes the chunk q with q % 8 == w of every stage, so its k-slice is fixed
//   (q % slices == w % slices) and its part of x lives in registers, widened
//   to fp32 once.  Each chunk is a 32-lane dot product (32 weights per lane,
//   16-byte conflict-free shared loads), reduced with a fixed shuffle tree.
// * Rows are summed over their k-slices in slice order inside the CTA.  The
//   run's last row, when it continues into the next CTA, is streamed FIRST;
//   its partial (lower slices) is published with a release flag early, and
//   the next CTA -- which holds that row's upper slices as the start of its
//   run -- adds it at its end: row = lower part + upper part, a fixed order.
//   No tensor memory, no tile-level split-K (muse_bf16_proj notebook, n. 47:
//   one-token vector reduction; project report, "What did not pay off":
//   in-CTA reduction beat cross-CTA split-K).
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "splitk.cuh"

namespace proj {
namespace {

constexpr int kComputeWarps = 8;
constexpr int kGemvThreads = (kComputeWarps + 1) * 32;
constexpr int kChunkElems = 1024;
constexpr int kRowRing = 128;   // rows in flight in the reduction ring (>= run-ahead + 1 stage)
constexpr int kMaxSlices = 8;   // K <= 8192

template <typename WT>
struct GCfg {
  static constexpr int kChunkBytes = kChunkElems * static_cast<int>(sizeof(WT));
  static constexpr int kStageBytes = 8 * kChunkBytes;
  static constexpr int S = sizeof(WT) == 2 ? 12 : 6;
  static constexpr int kVec = 16 / static_cast<int>(sizeof(WT));  // elements per 16 B
};

template <typename WT, int MT>
struct GSmem {
  static constexpr size_t kRing = static_cast<size_t>(GCfg<WT>::S) * GCfg<WT>::kStageBytes;
  static constexpr size_t kRed = static_cast<size_t>(kRowRing) * kMaxSlices * MT * 4;
  static constexpr size_t kEdge = 2 * kMaxSlices * MT * 4;
  static constexpr size_t kCnt = (kRowRing + 2) * 4;
  static constexpr size_t kBars = 2 * GCfg<WT>::S * 8;
  static constexpr size_t kTotal = 1024 + kRing + kRed + kEdge + kCnt + kBars + 64;
};

// Stage j of this CTA's processing order: chunks [qs, qs + ns).
struct StagePlan {
  int64_t tail_lo;   // first chunk of the streamed-first tail piece (== q1 if none)
  int64_t q0, q1;
  int64_t n_tail_stages;
  __device__ void stage(int64_t j, int64_t& qs, int& ns) const {
    if (j < n_tail_stages) {
      qs = tail_lo + j * 8;
      ns = static_cast<int>(q1 - qs < 8 ? q1 - qs : 8);
    } else {
      qs = q0 + (j - n_tail_stages) * 8;
      ns = static_cast<int>(tail_lo - qs < 8 ? tail_lo - qs : 8);
    }
  }
};

template <typename WT>
__device__ __forceinline__ void widen8(const uint4 v, float (&f)[8]);

template <>
__device__ __forceinline__ void widen8<__nv_bfloat16>(const uint4 v, float (&f)[8]) {
  f[0] = __uint_as_float(v.x << 16);
  f[1] = __uint_as_float(v.x & 0xFFFF0000u);
  f[2] = __uint_as_float(v.y << 16);
  f[3] = __uint_as_float(v.y & 0xFFFF0000u);
  f[4] = __uint_as_float(v.z << 16);
  f[5] = __uint_as_float(v.z & 0xFFFF0000u);
  f[6] = __uint_as_float(v.w << 16);
  f[7] = __uint_as_float(v.w & 0xFFFF0000u);
}

template <typename WT, int MT>
__global__ void __launch_bounds__(kGemvThreads, 1) gemv_kernel(const GemvParams p) {
  using C = GCfg<WT>;
  using SM = GSmem<WT, MT>;
  constexpr int S = C::S;
  constexpr int VEC = C::kVec;
  constexpr int NI = 32 / VEC;  // 16-byte loads per lane per chunk
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* ring = smem;
  float* red = reinterpret_cast<float*>(ring + SM::kRing);        // [kRowRing][slices][MT]
  float* head_red = red + kRowRing * kMaxSlices * MT;              // [slices][MT]
  float* tail_red = head_red + kMaxSlices * MT;                    // [slices][MT]
  // slices deposited per ring row; [kRowRing] = head row, [kRowRing + 1] = tail row
  uint32_t* cnt = reinterpret_cast<uint32_t*>(tail_red + kMaxSlices * MT);
  uint64_t* bars = reinterpret_cast<uint64_t*>(cnt + kRowRing + 2);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * S;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ks = p.K / kChunkElems;  // k-slices per row (1..8)
  const int64_t C_total = static_cast<int64_t>(p.n_rows) * ks;
  const int64_t cta = blockIdx.x;
  const int64_t q0 = part_begin(cta, C_total, p.G);
  const int64_t q1 = part_begin(cta + 1, C_total, p.G);
  const bool has_head = (q0 % ks) != 0;               // row q0/ks began in CTA cta-1
  const bool has_tail = (q1 % ks) != 0;               // row q1/ks continues in CTA cta+1
  const int64_t head_row = q0 / ks;
  const int64_t tail_row = q1 / ks;
  StagePlan plan;
  plan.q0 = q0;
  plan.q1 = q1;
  plan.tail_lo = has_tail ? tail_row * ks : q1;
  plan.n_tail_stages = has_tail ? (q1 - plan.tail_lo + 7) / 8 : 0;
  const int64_t n_stages = plan.n_tail_stages + (plan.tail_lo - q0 + 7) / 8;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kComputeWarps);
    }
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < kRowRing + 2; i += blockDim.x) cnt[i] = 0;
  __syncthreads();

  if (warp == kComputeWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const uint8_t* w = static_cast<const uint8_t*>(p.w);
      int64_t j = 0;
      for (; j < n_stages; ++j) {
        const int s = static_cast<int>(j % S);
        if (!mbar_wait(empty0 + 8 * s, static_cast<uint32_t>(((j / S) & 1) ^ 1), p.status,
                       kStatusTimeoutProducer))
          break;
        int64_t qs;
        int ns;
        plan.stage(j, qs, ns);
        const uint32_t bytes = static_cast<uint32_t>(ns) * C::kChunkBytes;
        mbar_arrive_expect_tx(full0 + 8 * s, bytes);
        bulk_g2s(smem_u32(ring + static_cast<size_t>(s) * C::kStageBytes),
                 w + qs * C::kChunkBytes, bytes, full0 + 8 * s, pol);
      }
      for (int64_t d = (j > S ? j - S : 0); d < j; ++d)
        mbar_wait(full0 + 8 * static_cast<int>(d % S), static_cast<uint32_t>((d / S) & 1),
                  p.status, kStatusTimeoutDrain);
    }
    return;
  }

  // ----------------------------------------------------------- compute warps
  const int tid = threadIdx.x;  // 0..255
  const int slice = warp % ks;
  // x for this warp's k-slice, widened to fp32: element (i, e) of the lane is
  // column slice*1024 + lane*VEC + 32*VEC*i + e.
  float xr[MT][32];
  {
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(p.x);
#pragma unroll
    for (int t = 0; t < MT; ++t) {
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        const int64_t col = static_cast<int64_t>(slice) * kChunkElems + lane * VEC + 32 * VEC * i;
#pragma unroll
        for (int e = 0; e < VEC; ++e) xr[t][i * VEC + e] = 0.f;
        if (t < p.m) {
          if (VEC == 8) {
            const uint4 v = *reinterpret_cast<const uint4*>(xb + t * static_cast<int64_t>(p.K) + col);
            float f[8];
            widen8<__nv_bfloat16>(v, f);
#pragma unroll
            for (int e = 0; e < 8; ++e) xr[t][i * VEC + e] = f[e];
          } else {
            const uint2 v = *reinterpret_cast<const uint2*>(xb + t * static_cast<int64_t>(p.K) + col);
            xr[t][i * VEC + 0] = __uint_as_float(v.x << 16);
            xr[t][i * VEC + 1] = __uint_as_float(v.x & 0xFFFF0000u);
            xr[t][i * VEC + 2] = __uint_as_float(v.y << 16);
            xr[t][i * VEC + 3] = __uint_as_float(v.y & 0xFFFF0000u);
          }
        }
      }
    }
  }

  const int head_nsl = has_head ? static_cast<int>(ks - (q0 - head_row * ks)) : 0;
  const int tail_nsl = has_tail ? static_cast<int>(q1 - tail_row * ks) : 0;
  auto store_out = [&](int64_t row, int t, float v) {
    if (p.out_f32)
      static_cast<float*>(p.out)[static_cast<int64_t>(t) * p.n_rows + row] = v;
    else
      static_cast<__nv_bfloat16*>(p.out)[static_cast<int64_t>(t) * p.n_rows + row] =
          __float2bfloat16_rn(v);
  };

  // Warps run independently: each waits for its stage, reduces its chunk,
  // deposits the slice sum, and the warp that deposits a row's last slice
  // sums the row in slice order.  The copy ring bounds how far one warp can
  // run ahead of another (S stages), which the row ring covers.
  bool ok = true;
  for (int64_t j = 0; j < n_stages; ++j) {
    const int s = static_cast<int>(j % S);
    int64_t qs;
    int ns;
    plan.stage(j, qs, ns);
    const int off = static_cast<int>(((warp - qs) % 8 + 8) % 8);
    const bool got = mbar_wait(full0 + 8 * s, static_cast<uint32_t>((j / S) & 1), p.status,
                               kStatusTimeoutMma);
    if (!got) {
      ok = false;
      break;
    }
    if (off < ns) {
      const uint8_t* chunk = ring + static_cast<size_t>(s) * C::kStageBytes +
                             static_cast<size_t>(off) * C::kChunkBytes;
      // 4 independent FMA chains per token (one per group of loads, mod 4)
      float acc[MT][4];
#pragma unroll
      for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[t][c] = 0.f;
      uint4 raw[NI];
#pragma unroll
      for (int i = 0; i < NI; ++i)
        raw[i] = *reinterpret_cast<const uint4*>(chunk + (lane + 32 * i) * 16);
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        float wv[VEC];
        if constexpr (VEC == 8) {
          float f[8];
          widen8<__nv_bfloat16>(raw[i], f);
#pragma unroll
          for (int e = 0; e < 8; ++e) wv[e] = f[e];
        } else {
          wv[0] = __uint_as_float(raw[i].x);
          wv[1] = __uint_as_float(raw[i].y);
          wv[2] = __uint_as_float(raw[i].z);
          wv[3] = __uint_as_float(raw[i].w);
        }
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
          for (int e = 0; e < VEC; ++e)
            acc[t][i & 3] = fmaf(wv[e], xr[t][i * VEC + e], acc[t][i & 3]);
      }
      float sum[MT];
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        sum[t] = (acc[t][0] + acc[t][1]) + (acc[t][2] + acc[t][3]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum[t] += __shfl_xor_sync(0xffffffffu, sum[t], o);
      }
      const int64_t row = (qs + off) / ks;
      const bool is_head = has_head && row == head_row;
      const bool is_tail = has_tail && row == tail_row;
      float* dst = is_head ? head_red
                 : is_tail ? tail_red
                           : red + static_cast<int>(row % kRowRing) * kMaxSlices * MT;
      uint32_t* c = is_head ? cnt + kRowRing : is_tail ? cnt + kRowRing + 1
                                                       : cnt + static_cast<int>(row % kRowRing);
      const uint32_t need = is_head ? head_nsl : is_tail ? tail_nsl : static_cast<uint32_t>(ks);
      uint32_t prev = 0;
      if (lane == 0) {
#pragma unroll
        for (int t = 0; t < MT; ++t) dst[slice * MT + t] = sum[t];
        __threadfence_block();
        prev = atomicAdd(c, 1u);
      }
      prev = __shfl_sync(0xffffffffu, prev, 0);
      if (prev + 1 == need && !is_head) {
        // last slice of the row: sum slices in order
        __threadfence_block();
        const int sl0 = is_tail ? 0 : 0;
        const int sl1 = is_tail ? tail_nsl : ks;
        if (lane < MT) {
          float v = 0.f;
          for (int sl = sl0; sl < sl1; ++sl) v += dst[sl * MT + lane];
          if (is_tail) {
            p.ws[cta * MT + lane] = v;
          } else if (lane < p.m) {
            store_out(row, lane, v);
          }
        }
        if (is_tail) {
          __syncwarp();
          if (lane == 0) {
            __threadfence();
            red_release_gpu_add(p.flags + cta, 1u);
          }
        } else if (lane == 0) {
          *c = 0u;  // ring slot free for row + kRowRing
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
  }
  // Every compute warp is done: the head row's upper slices are all deposited.
  if (named_bar_sync_or(1, kComputeWarps * 32, !ok)) ok = false;
  // The first row of the run: its lower slices come from the previous CTA,
  // which published them right after streaming them.
  if (ok && has_head && tid < MT) {
    const int t = tid;
    if (spin_until_ge(p.flags + cta - 1, 1u, p.status)) {
      const float lo = __ldcg(p.ws + (cta - 1) * MT + t);
      float up = 0.f;
      for (int sl = ks - head_nsl; sl < ks; ++sl) up += head_red[sl * MT + t];
      if (t < p.m) store_out(head_row, t, lo + up);
    }
  }
  if (has_head) {
    named_bar_sync(1, kComputeWarps * 32);
    if (tid == 0) p.flags[cta - 1] = 0u;
  }
}

template <typename WT, int MT>
cudaError_t set_attr() {
  return cudaFuncSetAttribute(gemv_kernel<WT, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(GSmem<WT, MT>::kTotal));
}

template <typename WT, int MT>
cudaError_t launch(const GemvParams& p, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = GSmem<WT, MT>::kTotal;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_kernel<WT, MT>, p);
}

}  // namespace

cudaError_t gemv_init_attributes() {
  cudaError_t e;
  if ((e = set_attr<__nv_bfloat16, 1>()) != cudaSuccess) return e;
  if ((e = set_attr<__nv_bfloat16, 2>()) != cudaSuccess) return e;
  if ((e = set_attr<float, 1>()) != cudaSuccess) return e;
  if ((e = set_attr<float, 2>()) != cudaSuccess) return e;
  return cudaSuccess;
}

cudaError_t gemv_launch(bool f32w, int MT, const GemvParams& p, cudaStream_t s) {
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

}  // namespace proj
