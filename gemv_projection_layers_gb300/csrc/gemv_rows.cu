// gemv_rows.cu -- the bf16 layers at 3..32 tokens: a weight stream over whole
// row runs per CTA, fed by tensor copies into a shared-memory ring and
// multiplied on the warp-level tensor-core MMA.
//
// out[i, n] = sum_k x[i, k] W[n, k]            (muse_bf16_proj guide, ch. 1, §1.1)
//
// The one-token GEMV reaches the read floor because every CTA owns whole
// rows (no split-K hand-off) and keeps its weight stream going from the
// first cycle.  This kernel keeps that partition for a few tokens, where m
// products per weight need the tensor cores:
//
// * CTA c of G owns rows [c N / G, (c + 1) N / G) of the row-major W -- the
//   register GEMV's partition, balanced to one row, so every SM streams the
//   same bytes.  Its rows form 16-row blocks for the mma.sync m16n8k16 A
//   operand; the last block may be partial (its missing rows are neither
//   loaded nor stored).
// * K is walked in 32-column steps.  Prepare lays each CTA's run out as
//   [step][row][64 B] (lossless), so one thread streams a stage of KS steps
//   of all its rows with a single contiguous bulk copy -- a sequential read,
//   like the read floor's -- into a ring of S stages.  x comes with a 3-D
//   tensor copy (64 columns, tokens, double steps) in the 128-byte swizzle;
//   tokens beyond m are zero-filled by the copy.  (For a grid other than the
//   one the layout was packed for, W comes from the row-major copy through
//   3-D tensor copies of (32 columns, rows, steps) boxes instead, one box row
//   per CTA shorter where its run is.)  The first ring's worth of weights is
//   requested before the wait on the previous kernel of the stream.
// * Within a step, lane (g, c) of a warp reads 16 bytes at columns
//   8c .. 8c + 7 of block rows g and g + 8 and of token rows g (+ 8 t).
//   The MMA's A and B fragments want columns {2c, 2c + 1, 2c + 8, 2c + 9} of
//   a 16-column k-tile; assigning those four logical columns of k-tile
//   j in {0, 1} to the physical columns 8c + 4j .. 8c + 4j + 3 -- the same
//   assignment on both operands -- makes each 16-byte read two k-tiles'
//   fragments, and the step's two MMAs still sum over exactly its 32
//   columns.  Eight consecutive rows x 64 bytes: every read is conflict-free.
// * Sixteen consumer warps: 16 / NB per 16-row block, each taking every
//   (16 / NB)-th step of a stage.  After the last stage the warps' 16 x 8
//   fp32 tiles are summed per block in warp order (deterministic), rounded
//   to bf16 and stored.
// This is the pages' GEMV (muse_bf16_proj project report, "What was built":
// 16-row blocks, warps splitting K, mma.sync) on GB300, with the one-token
// GEMV's row partition and the weights fed by bulk tensor copies.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace proj {
namespace {

constexpr int kConsumers = kGemvRowsConsumers;
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kRowPitch = kGemvRowsRowPitch;

// 3-D tiled tensor copy global -> shared (c0 innermost).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t c0,
                                            int32_t c1, int32_t c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
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

// d += A (16 x 16, bf16, row) * B (16 x 8, bf16, col), fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ldg_x(const void* p) {
  uint4 v;
  asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <int NT, int SPW>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_rows_kernel(const __grid_constant__ CUtensorMap tw_hi,
                     const __grid_constant__ CUtensorMap tw_lo, const GemvRowsParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  if (p.stamps && threadIdx.x == 0) p.stamps[blockIdx.x * 8 + kStampEntry] = globaltimer_ns();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int KS = p.KS;
  const int S = p.S;
  const uint32_t stage = gemv_rows_stage_bytes(p.KS, p.nr_hi);
  const uint32_t ring = smem_u32(smem);
  // barriers after the ring (or after the tiles' staging, which reuses it)
  const uint32_t full0 = ring + gemv_rows_bar_offset(NT, p.KS, p.S, p.nr_hi);
  const uint32_t empty0 = full0 + 8 * S;

  const int r0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * p.n_rows / p.G);
  const int r1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * p.n_rows / p.G);
  const int nr = r1 - r0;                 // nr_hi or nr_hi - 1
  const int NB = (p.nr_hi + 15) >> 4;     // 16-row blocks (of the longest run)
  const int wpb = kConsumers / gemv_rows_block_slots(p.nr_hi);  // warps per block: KS = SPW wpb
  const int nst = (p.K >> 5) / KS;        // stages of the run

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kConsumers);
    }
    fence_mbar_init();
  }
  __syncthreads();
  griddep_launch_dependents();

  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer
    // The weights are constant: they stream from the first cycle, without
    // waiting for the previous kernel of the stream.
    if (lane == 0) {
      const CUtensorMap* tw = nr == p.nr_hi ? &tw_hi : &tw_lo;
      if (!p.w_runs) prefetch_tmap(tw);
      // this CTA's run in the packed layout: stage j is one contiguous piece
      const uint8_t* run = p.w_runs ? p.w_runs + static_cast<size_t>(r0) * p.K * 2 : nullptr;
      const uint32_t wbytes = static_cast<uint32_t>(KS) * nr * 64;
      const uint64_t pol = policy_evict_first();
      int issued = 0;
      for (int j = 0; j < nst; ++j) {
        const int s = j % S;
        if (j >= S && !mbar_wait(empty0 + 8 * s, static_cast<uint32_t>(((j / S) & 1) ^ 1),
                                 p.status, kStatusTimeoutProducer))
          break;
        mbar_arrive_expect_tx(full0 + 8 * s, wbytes);
        if (run)
          bulk_g2s(ring + s * stage, run + static_cast<size_t>(j) * wbytes, wbytes, full0 + 8 * s,
                   pol);
        else
          tma_load_3d(ring + s * stage, tw, 0, r0, j * KS, full0 + 8 * s);
        issued = j + 1;
      }
      // Wait (bounded) for the copies of the last ring's worth of stages
      // before the CTA may leave (normally they are long done: the consumers
      // waited on them; after a timeout they may still be in flight).
      for (int j = issued > S ? issued - S : 0; j < issued; ++j)
        mbar_wait(full0 + 8 * (j % S), static_cast<uint32_t>((j / S) & 1), p.status,
                  kStatusTimeoutDrain);
    }
  } else {
    // ----------------------------------------------------------- consumers
    const int g = lane >> 2;
    const int c = lane & 3;
    const int q = warp / wpb;       // block of this warp (idle if q >= NB)
    const int jw = warp - q * wpb;  // its steps of every stage: jw + k wpb, k < SPW
    const int ra = 16 * q + g;      // its rows ra and ra + 8 within the run
    const bool act = q < NB;
    const bool va = act && ra < nr;
    const bool vb = act && ra + 8 < nr;
    // x: lane (g, c) reads 16 bytes of token 8 t + g at columns 8c .. of
    // each of its steps (zero beyond m), from L2 after the first touch,
    // D stages ahead of their use.
    const uint16_t* xl = p.x + 8 * c;
    auto load_x = [&](int i, uint4 (&xb)[SPW][NT]) {
#pragma unroll
      for (int k = 0; k < SPW; ++k) {
        const int col = 32 * (i * KS + jw + k * wpb);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int tok = 8 * t + g;
          xb[k][t] = (act && i < nst && tok < p.m)
                         ? ldg_x(xl + static_cast<size_t>(tok) * p.K + col)
                         : make_uint4(0, 0, 0, 0);
        }
      }
    };
    float acc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
    bool ok = true;
    auto consume = [&](int i, const uint4 (&xb)[SPW][NT]) {
      const int s = i % S;
      // One lane per warp waits (suspending: sixteen warps polling would take
      // issue slots from the producer); the warp barrier then orders the
      // other lanes' reads of the stage after that lane's acquire.
      if (lane == 0 && ok &&
          !mbar_wait_sleep(full0 + 8 * s, static_cast<uint32_t>((i / S) & 1), p.status,
                           kStatusTimeoutMma))
        ok = false;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) return;
      const uint32_t bw = ring + s * stage;
      if (act) {
#pragma unroll
        for (int k = 0; k < SPW; ++k) {
          const int j = jw + k * wpb;
          const uint32_t rw = bw + static_cast<uint32_t>((j * nr + ra) * 64 + c * 16);
          const uint4 P = va ? ld_shared_u4(rw) : make_uint4(0, 0, 0, 0);
          const uint4 Q = vb ? ld_shared_u4(rw + 8 * 64) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const uint4& X = xb[k][t];
            mma16816(acc[t], P.x, Q.x, P.y, Q.y, X.x, X.y);  // k-tile 0 of the step
            mma16816(acc[t], P.z, Q.z, P.w, Q.w, X.z, X.w);  // k-tile 1
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);
    };
    griddep_wait();  // x may be the previous kernel's output
    if (p.stamps && threadIdx.x == 0) p.stamps[blockIdx.x * 8 + kStampDepWait] = globaltimer_ns();
    // x for stages i .. i + D - 1 in flight (a static register ring: stage
    // i uses slot i % D, refilled with stage i + D right after its MMAs)
    constexpr int D = gemv_rows_x_depth(NT, SPW);
    uint4 xr[D][SPW][NT];
#pragma unroll
    for (int d = 0; d < D; ++d) load_x(d, xr[d]);
    for (int i0 = 0; i0 < nst; i0 += D) {
#pragma unroll
      for (int d = 0; d < D; ++d) {
        const int i = i0 + d;
        if (i >= nst) break;
        consume(i, xr[d]);
        load_x(i + D, xr[d]);
      }
    }
    if (p.stamps && threadIdx.x == 0) p.stamps[blockIdx.x * 8 + kStampDrained] = globaltimer_ns();
    // every stage has been consumed before the ring is reused for the tiles
    named_bar_sync(1, kConsumers * 32);
    if (act) {
      // [warp][token][kRowPitch] fp32 over the ring
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int tok = 8 * t + 2 * c;
        const uint32_t b0 = ring + static_cast<uint32_t>(((warp * 8 * NT + tok) * kRowPitch + g) * 4);
        st_shared_f32(b0, acc[t][0]);
        st_shared_f32(b0 + kRowPitch * 4, acc[t][1]);
        st_shared_f32(b0 + 8 * 4, acc[t][2]);
        st_shared_f32(b0 + kRowPitch * 4 + 8 * 4, acc[t][3]);
      }
    }
    named_bar_sync(1, kConsumers * 32);
    // Each (block, token, row): the sum over the block's warps in warp order.
    // Consecutive threads take consecutive rows of one token.
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
    const int items = NB * p.m * 16;
    for (int idx = threadIdx.x; idx < items; idx += kConsumers * 32) {
      const int row = idx & 15;
      const int tok = (idx >> 4) % p.m;
      const int qb = (idx >> 4) / p.m;
      if (16 * qb + row >= nr) continue;
      float sum = 0.f;
      for (int w = qb * wpb; w < qb * wpb + wpb; ++w)
        sum += ld_shared_f32(ring + static_cast<uint32_t>(((w * 8 * NT + tok) * kRowPitch + row) * 4));
      out[static_cast<size_t>(tok) * p.n_rows + r0 + 16 * qb + row] = __float2bfloat16_rn(sum);
    }
    if (p.stamps && threadIdx.x == 0) p.stamps[blockIdx.x * 8 + kStampExit] = globaltimer_ns();
  }
}

template <int NT, int SPW>
cudaError_t set_attr() {
  return cudaFuncSetAttribute(gemv_rows_kernel<NT, SPW>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kGemvRowsSmemMax);
}

template <int NT, int SPW>
cudaError_t launch(const CUtensorMap& tw_hi, const CUtensorMap& tw_lo, const GemvRowsParams& p,
                   cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = gemv_rows_smem(NT, p.KS, p.S, p.nr_hi);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_rows_kernel<NT, SPW>, tw_hi, tw_lo, p);
}

template <int NT>
cudaError_t launch_nt(int spw, const CUtensorMap& tw_hi, const CUtensorMap& tw_lo,
                      const GemvRowsParams& p, cudaStream_t s) {
  switch (spw) {
    case 1: return launch<NT, 1>(tw_hi, tw_lo, p, s);
    case 2: return launch<NT, 2>(tw_hi, tw_lo, p, s);
    case 4: return launch<NT, 4>(tw_hi, tw_lo, p, s);
  }
  return cudaErrorInvalidValue;
}

template <int NT>
cudaError_t set_attr_nt() {
  cudaError_t e;
  if ((e = set_attr<NT, 1>()) != cudaSuccess) return e;
  if ((e = set_attr<NT, 2>()) != cudaSuccess) return e;
  return set_attr<NT, 4>();
}

}  // namespace

size_t gemv_rows_smem(int nt, int ks, int stages, int nr_hi) {
  return 1024 + gemv_rows_bar_offset(nt, ks, stages, nr_hi) + 16 * static_cast<size_t>(stages);
}

cudaError_t gemv_rows_init_attributes() {
  cudaError_t e;
  if ((e = set_attr_nt<1>()) != cudaSuccess) return e;
  if ((e = set_attr_nt<2>()) != cudaSuccess) return e;
  return set_attr_nt<4>();
}

cudaError_t gemv_rows_launch(int nt, int spw, const CUtensorMap& tw_hi, const CUtensorMap& tw_lo,
                             const GemvRowsParams& p, cudaStream_t s) {
  switch (nt) {
    case 1: return launch_nt<1>(spw, tw_hi, tw_lo, p, s);
    case 2: return launch_nt<2>(spw, tw_hi, tw_lo, p, s);
    case 4: return launch_nt<4>(spw, tw_hi, tw_lo, p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace proj
