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
//   weights (K / 1024 "slices" per row), and the chunks of the whole matrix,
//   in row-major order, are split into G equal contiguous runs, one per CTA
//   (one CTA per SM).  Every CTA streams the same number of bytes; a run is at
//   least one row long, so only its first and last row can be shared with a
//   neighbour.
// * One producer thread streams 8-chunk stages (16 KB bf16 / 32 KB fp32)
//   with bulk copies into a ring of S slots, and there is one compute warp
//   per slot: stage j lands in slot j % S and belongs to warp j % S, so every
//   slot has a single, in-order consumer (a parity wait cannot tell one ring
//   generation from the one two laps earlier, so no slot may be shared by
//   warps that can drift apart).  The warp keeps a lane partial per row
//   across the stage's chunks and reduces each row segment once with a
//   shuffle tree; x sits in shared memory as bf16 in the same lane layout as
//   the weights (conflict-free 16-byte loads).
// * A row is summed in a fixed order: lane partials over its chunks in
//   column order, the shuffle tree, then lower segment + upper segment when
//   the row straddles two stages (the warp that deposits second finishes it).
//   The run's last row, when it continues into the next CTA, is streamed
//   FIRST and published with a release flag; the next CTA, which holds that
//   row's upper slices at the start of its run, adds it at its end.
//   No tensor memory and no tile-level split-K (muse_bf16_proj notebook,
//   n. 47: a one-token vector reduction; project report, "What did not pay
//   off": in-CTA reduction beat cross-CTA split-K).
#include <cuda_bf16.h>

#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"
#include "splitk.cuh"

namespace proj {
namespace {

constexpr int kChunkElems = 1024;
constexpr int kSplitRing = 64;  // rows straddling two stages, in flight

template <typename WT, int MT>
struct GCfg {
  static constexpr int kChunkBytes = kChunkElems * static_cast<int>(sizeof(WT));
  static constexpr int kStageBytes = 8 * kChunkBytes;
  static constexpr int kVec = 16 / static_cast<int>(sizeof(WT));  // weights per 16 B
  static constexpr int kXBytes = MT * 8192 * static_cast<int>(sizeof(WT));  // x, K <= 8192
  static constexpr int kFit = (232448 - 1024 - kXBytes - 2048) / kStageBytes;
  static constexpr int S = kFit > 12 ? 12 : kFit;  // ring slots == compute warps
  static constexpr int kThreads = (S + 1) * 32;
  static constexpr size_t kSplit = static_cast<size_t>(kSplitRing) * 2 * MT * 4;
  static constexpr size_t kSmem = 1024 + static_cast<size_t>(S) * kStageBytes + kXBytes + kSplit +
                                  kSplitRing * 4 + 2 * S * 8 + 64;
  static_assert(S >= 4, "ring too shallow");
  static_assert(kSmem <= 232448, "shared memory budget");
};

// Stage j of this CTA's processing order covers chunks [qs, qs + ns): first
// the tail piece (the run's last row, when it continues in the next CTA),
// then the run from its start.
struct StagePlan {
  int64_t tail_lo;   // first chunk of the tail piece (== q1 if none)
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

__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xFFFF0000u);
}

// x in shared memory, in the same lane layout as the weights: bf16 for bf16
// weights (16-byte loads of 8 columns), fp32 for fp32 weights (16-byte loads
// of 4 columns); a warp's loads are contiguous 512-byte runs (conflict-free).

// acc += lo(w) * lo(x) and acc2 += hi(w) * hi(x): fp32 = bf16 * bf16 + fp32
// (the product of two bf16 values is exact in fp32, so this equals widening
// both operands and a single-precision FMA), one instruction per weight.
__device__ __forceinline__ void fma_bf16x2(float& acc, float& acc2, uint32_t w, uint32_t x) {
  asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
      "mov.b32 {wl, wh}, %2;\n\t"
      "mov.b32 {xl, xh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, wl, xl, %0;\n\t"
      "fma.rn.f32.bf16 %1, wh, xh, %1;\n\t}"
      : "+f"(acc), "+f"(acc2)
      : "r"(w), "r"(x));
}

// (acc, acc2) += (w0, w1) * (x0, x1), two fp32 FMAs in one instruction.
__device__ __forceinline__ void fma_f32x2(float& acc, float& acc2, uint32_t w0, uint32_t w1,
                                          float x0, float x1) {
  uint64_t a = (static_cast<uint64_t>(__float_as_uint(acc2)) << 32) | __float_as_uint(acc);
  const uint64_t w = (static_cast<uint64_t>(w1) << 32) | w0;
  const uint64_t x = (static_cast<uint64_t>(__float_as_uint(x1)) << 32) | __float_as_uint(x0);
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a) : "l"(w), "l"(x));
  acc = __uint_as_float(static_cast<uint32_t>(a));
  acc2 = __uint_as_float(static_cast<uint32_t>(a >> 32));
}

template <typename WT>
using XT = typename std::conditional<sizeof(WT) == 2, uint16_t, float>::type;

// Lane partial of one chunk for MT tokens (col0: the chunk's first column).
// Eight independent accumulation chains; combined in a fixed order.
template <typename WT, int MT>
__device__ __forceinline__ void chunk_partial(uint32_t chunk, uint32_t xs, int K, int col0,
                                              int lane, float (&acc)[MT]) {
  constexpr int VEC = GCfg<WT, MT>::kVec;
  constexpr int NI = 32 / VEC;
  float a8[MT][8];
#pragma unroll
  for (int t = 0; t < MT; ++t)
#pragma unroll
    for (int c = 0; c < 8; ++c) a8[t][c] = 0.f;
  uint4 wraw[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) wraw[i] = ld_shared_u4(chunk + (lane + 32 * i) * 16);
#pragma unroll
  for (int i = 0; i < NI; ++i) {
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      const uint4 xv = ld_shared_u4(
          xs + static_cast<uint32_t>((t * K + col0 + (lane + 32 * i) * VEC) * sizeof(XT<WT>)));
      float* a = a8[t];
      if constexpr (VEC == 8) {
        fma_bf16x2(a[(i & 1) * 4 + 0], a[(i & 1) * 4 + 1], wraw[i].x, xv.x);
        fma_bf16x2(a[(i & 1) * 4 + 2], a[(i & 1) * 4 + 3], wraw[i].y, xv.y);
        fma_bf16x2(a[(i & 1) * 4 + 0], a[(i & 1) * 4 + 1], wraw[i].z, xv.z);
        fma_bf16x2(a[(i & 1) * 4 + 2], a[(i & 1) * 4 + 3], wraw[i].w, xv.w);
      } else {
        fma_f32x2(a[(i & 3) * 2 + 0], a[(i & 3) * 2 + 1], wraw[i].x, wraw[i].y,
                  __uint_as_float(xv.x), __uint_as_float(xv.y));
        fma_f32x2(a[(i & 3) * 2 + 0], a[(i & 3) * 2 + 1], wraw[i].z, wraw[i].w,
                  __uint_as_float(xv.z), __uint_as_float(xv.w));
      }
    }
  }
#pragma unroll
  for (int t = 0; t < MT; ++t)
    acc[t] += ((a8[t][0] + a8[t][1]) + (a8[t][2] + a8[t][3])) +
              ((a8[t][4] + a8[t][5]) + (a8[t][6] + a8[t][7]));
}

template <typename WT, int MT>
__global__ void __launch_bounds__(GCfg<WT, MT>::kThreads, 1) gemv_kernel(const GemvParams p) {
  using C = GCfg<WT, MT>;
  constexpr int S = C::S;
  constexpr int kComputeWarps = S;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* ring = smem;
  XT<WT>* xs = reinterpret_cast<XT<WT>*>(ring + static_cast<size_t>(S) * C::kStageBytes);
  float* split = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(xs) + C::kXBytes);
  uint32_t* split_cnt = reinterpret_cast<uint32_t*>(split + kSplitRing * 2 * MT);
  uint64_t* bars = reinterpret_cast<uint64_t*>(split_cnt + kSplitRing);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * S;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ks = p.K / kChunkElems;  // slices per row (1..8)
  const int64_t C_total = static_cast<int64_t>(p.n_rows) * ks;
  const int64_t cta = blockIdx.x;
  // The partition in 32-bit arithmetic when it fits (every fixed layer):
  // 64-bit divisions are software routines and delay the first copy.
  int64_t q0, q1;
  if (C_total < (int64_t{1} << 22)) {
    const uint32_t ct = static_cast<uint32_t>(C_total), g = static_cast<uint32_t>(p.G);
    q0 = static_cast<uint32_t>(blockIdx.x) * ct / g;
    q1 = (static_cast<uint32_t>(blockIdx.x) + 1u) * ct / g;
  } else {
    q0 = part_begin(cta, C_total, p.G);
    q1 = part_begin(cta + 1, C_total, p.G);
  }
  const bool has_head = (q0 % ks) != 0;  // row q0 / ks began in CTA cta - 1
  const bool has_tail = (q1 % ks) != 0;  // row q1 / ks continues in CTA cta + 1
  const int64_t head_row = q0 / ks;
  const int64_t tail_row = q1 / ks;
  StagePlan plan;
  plan.q0 = q0;
  plan.q1 = q1;
  plan.tail_lo = has_tail ? tail_row * ks : q1;
  plan.n_tail_stages = has_tail ? 1 : 0;  // the tail piece is < ks <= 8 chunks
  const int64_t n_stages = plan.n_tail_stages + (plan.tail_lo - q0 + 7) / 8;

  // The producer thread sets up the ring.  Its copies go out after the CTA
  // barrier: a bulk-copy issue blocks while the SM's copy queue is full, and
  // issuing a ring's worth first held the compute warps (and the x staging)
  // back by microseconds.
  const bool producer = warp == kComputeWarps && lane == 0;
  uint64_t pol = 0;
  int64_t issued = 0;
  auto issue = [&](int64_t j) {
    const int s = static_cast<int>(j % S);
    int64_t qs;
    int ns;
    plan.stage(j, qs, ns);
    const uint32_t bytes = static_cast<uint32_t>(ns) * C::kChunkBytes;
    mbar_arrive_expect_tx(full0 + 8 * s, bytes);
    bulk_g2s(smem_u32(ring + static_cast<size_t>(s) * C::kStageBytes),
             static_cast<const uint8_t*>(p.w) + qs * C::kChunkBytes, bytes, full0 + 8 * s, pol);
  };
  if (producer) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    fence_mbar_init();
    pol = policy_evict_first();
  }
  for (int i = threadIdx.x; i < kSplitRing; i += blockDim.x) split_cnt[i] = 0;
  griddep_launch_dependents();
  __syncwarp();
  __syncthreads();

  if (warp == kComputeWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int64_t j = issued;
      for (; j < n_stages; ++j) {
        const int s = static_cast<int>(j % S);
        if (!mbar_wait(empty0 + 8 * s, static_cast<uint32_t>(((j / S) & 1) ^ 1), p.status,
                       kStatusTimeoutProducer))
          break;
        issue(j);
      }
      for (int64_t d = (j > S ? j - S : 0); d < j; ++d)
        mbar_wait(full0 + 8 * static_cast<int>(d % S), static_cast<uint32_t>((d / S) & 1),
                  p.status, kStatusTimeoutDrain);
    }
    return;
  }

  // ----------------------------------------------------------- compute warps
  const int tid = threadIdx.x;  // 0..255
  // The producer streams W (constant) at once; x and every global write wait
  // for the previous kernel of the stream.
  griddep_wait();
  {
    // x -> shared memory (bf16 as is, or widened to fp32 for fp32 weights;
    // zero rows beyond m).  Every load is issued before the first store, so
    // staging costs one memory round trip (x is cold after a flush).
    const uint4* xg = static_cast<const uint4*>(p.x);
    const int n8 = MT * p.K / 8;  // groups of 8 columns
    constexpr int kXLd = (MT * 8192 / 8 + kComputeWarps * 32 - 1) / (kComputeWarps * 32);
    uint4 xv[kXLd];
#pragma unroll
    for (int u = 0; u < kXLd; ++u) {
      const int i = tid + u * kComputeWarps * 32;
      xv[u] = (i < n8 && i / (p.K / 8) < p.m) ? xg[i] : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kXLd; ++u) {
      const int i = tid + u * kComputeWarps * 32;
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
  named_bar_sync(1, kComputeWarps * 32);

  auto store_out = [&](int64_t row, int t, float v) {
    if (p.out_f32)
      static_cast<float*>(p.out)[static_cast<int64_t>(t) * p.n_rows + row] = v;
    else
      static_cast<__nv_bfloat16*>(p.out)[static_cast<int64_t>(t) * p.n_rows + row] =
          __float2bfloat16_rn(v);
  };

  float head_val[MT];
#pragma unroll
  for (int t = 0; t < MT; ++t) head_val[t] = 0.f;
  bool ok = true;
  bool publish_tail = false;
  for (int64_t j = warp; j < n_stages; j += kComputeWarps) {
    const int s = static_cast<int>(j % S);
    int64_t qs;
    int ns;
    plan.stage(j, qs, ns);
    // slot s == warp: this warp consumed the slot's previous generation itself
    if (!mbar_wait_sleep(full0 + 8 * s, static_cast<uint32_t>((j / S) & 1), p.status,
                         kStatusTimeoutMma)) {
      ok = false;
      break;
    }
    const uint8_t* stage = ring + static_cast<size_t>(s) * C::kStageBytes;
    // Walk the stage's chunks, one row segment at a time.
    int c = 0;
    while (c < ns) {
      const int64_t row = (qs + c) / ks;
      const int64_t seg_lo = qs + c;
      int64_t seg_hi = (row + 1) * ks;  // exclusive chunk bound of the row
      if (seg_hi > qs + ns) seg_hi = qs + ns;
      float acc[MT];
#pragma unroll
      for (int t = 0; t < MT; ++t) acc[t] = 0.f;
      const int cc0 = static_cast<int>(seg_lo - qs);
      const int cc1 = static_cast<int>(seg_hi - qs);
      const int col_base = static_cast<int>(seg_lo - row * ks) * kChunkElems - cc0 * kChunkElems;
#pragma unroll 2
      for (int cc = cc0; cc < cc1; ++cc) {
        chunk_partial<WT, MT>(smem_u32(stage + cc * C::kChunkBytes), smem_u32(xs), p.K,
                              col_base + cc * kChunkElems,
                              lane, acc);
      }
#pragma unroll
      for (int t = 0; t < MT; ++t) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
      }
      const bool whole_here = (seg_lo == row * ks) && (seg_hi == (row + 1) * ks);
      if (has_head && row == head_row) {
#pragma unroll
        for (int t = 0; t < MT; ++t) head_val[t] = acc[t];  // all of it lies in one stage
      } else if (has_tail && row == tail_row) {
        // published below, after the stage is released
#pragma unroll
        for (int t = 0; t < MT; ++t)
          if (lane == t) p.ws[cta * MT + t] = acc[t];
        publish_tail = true;
      } else if (whole_here) {
#pragma unroll
        for (int t = 0; t < MT; ++t)
          if (lane == t && t < p.m) store_out(row, t, acc[t]);
      } else {
        // the row straddles two stages: lower segment (holds its first
        // chunk) + upper segment; whichever warp deposits second sums them
        const int slot = static_cast<int>(row % kSplitRing);
        const int part = (seg_lo == row * ks) ? 0 : 1;
        uint32_t prev = 0;
        if (lane == 0) {
#pragma unroll
          for (int t = 0; t < MT; ++t) split[(slot * 2 + part) * MT + t] = acc[t];
          __threadfence_block();
          prev = atomicAdd(split_cnt + slot, 1u);
        }
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev == 1) {
          __threadfence_block();
          if (lane < MT && lane < p.m) {
            const float v = split[(slot * 2 + 0) * MT + lane] + split[(slot * 2 + 1) * MT + lane];
            store_out(row, lane, v);
          }
          if (lane == 0) split_cnt[slot] = 0u;
        }
      }
      c = static_cast<int>(seg_hi - qs);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
    if (publish_tail) {
      // the lanes' partial stores, ordered by the warp barrier above, are
      // published by one release (cumulative)
      if (lane == 0) red_release_gpu_add(p.flags + cta, 1u);
      publish_tail = false;
    }
  }
  // The head row: its upper slices were reduced by the warp that owns the
  // first main stage; its lower slices come from the previous CTA, which
  // published them right after streaming them.
  if (has_head) {
    const int64_t owner_stage = plan.n_tail_stages;
    if (warp == static_cast<int>(owner_stage % S) && ok && lane < MT) {
      if (spin_until_ge(p.flags + cta - 1, 1u, p.status)) {
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          if (lane == t) {
            const float lo = __ldcg(p.ws + (cta - 1) * MT + t);
            if (t < p.m) store_out(head_row, t, lo + head_val[t]);
          }
        }
      }
    }
    named_bar_sync(1, kComputeWarps * 32);
    if (tid == 0) p.flags[cta - 1] = 0u;
  }
}

template <typename WT, int MT>
cudaError_t set_attr() {
  return cudaFuncSetAttribute(gemv_kernel<WT, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(GCfg<WT, MT>::kSmem));
}

template <typename WT, int MT>
cudaError_t launch(const GemvParams& p, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(GCfg<WT, MT>::kThreads);
  cfg.dynamicSmemBytes = GCfg<WT, MT>::kSmem;
  cfg.stream = s;
  // No cooperative launch: a CTA waits only on its predecessor (blockIdx - 1),
  // which is dispatched no later than it, and G <= SMs at one CTA per SM,
  // so every wait ends even while the previous kernel still holds SMs.
  // Programmatic stream serialization lets this grid start under the
  // previous kernel's tail (see griddep_wait above).
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
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
