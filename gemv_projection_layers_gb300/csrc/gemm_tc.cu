// gemm_tc.cu -- tensor-core skinny GEMM for the bf16 layers, every token count.
//
// out[i, n] = sum_k x[i, k] W[n, k]            (muse_bf16_proj guide, ch. 1, §1.1)
//
// GB300 design (the pages' H200 kernels -- warp-level mma GEMVs with
// in-CTA split-K, wgmma GEMMs -- are prior art, not the blueprint):
//
// * Operand roles are swapped: 128 weight rows are the MMA's M side (A,
//   K-major, from shared memory), the m tokens are its N side (B, N = BN =
//   m rounded up to 16..256), so even m = 1 runs tcgen05.mma.kind::f16
//   M128 x N16 x K16 with fp32 accumulation in tensor memory.
// * Weights stream HBM -> shared memory with 1-D bulk copies of prepacked,
//   pre-swizzled 16 KB tiles (one copy per 128 x 64 tile, evict-first), x
//   with a 2-D TMA load whose out-of-range rows read as zero (ragged m).
//   A deep mbarrier ring keeps 100-200 KB in flight per SM.
// * Exactly one CTA per SM (cooperative launch) and a split-K partition
//   that gives every CTA the same number of (tile, k-block) units; tiles
//   shared by several CTAs are combined in fixed CTA order (splitk.cuh):
//   owner mode for small m (the owner pre-sums the other contributors'
//   partials while its own last segment streams), distributed mode for large
//   m (each contributor reduces 1/S of the tile).  Counters return to zero
//   on the GPU (guide ch. 1, §1.6).  One launch per call, deterministic.
// * Warp roles: warp 0 issues copies, warp 1 issues MMAs (and owns the
//   tensor memory), warps 2-5 drain the accumulators; the 12-bit variant adds
//   warps 6-9, which decode each record from a deep ring of encoded stages
//   into a short ring of swizzled bf16 tiles and patch the escapes before the
//   MMA reads them, so the MMA inputs -- and the outputs -- are bit-identical
//   to the dense kernel's (project report, "Round 5 -- lossless 12-bit
//   compressed weights").
// * The accumulator is double-buffered in tensor memory so the epilogue of
//   one tile overlaps the MMAs of the next.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "splitk.cuh"

namespace proj {
namespace {

constexpr int kSmemLimit = 232448;        // max dynamic shared memory per block
constexpr int kSmemReserve = 1024 + 512;  // alignment slack + barriers

template <int BN, bool EXPWIN>
struct Cfg {
  static constexpr int kXBytes = BN * 128;
  static constexpr int SA = EXPWIN ? 4 : 0;  // decoded-tile ring (12-bit only)
  static constexpr int kCopyStage = (EXPWIN ? kRecBytes : kTileBytes) + kXBytes;
  static constexpr int kFit = (kSmemLimit - kSmemReserve - SA * kTileBytes) / kCopyStage;
  // copy ring; with 12-bit decode a multiple of the 4 decode warps
  static constexpr int SE = EXPWIN ? (kFit >= 8 ? 8 : 4) : (kFit > 12 ? 12 : kFit);
  static constexpr int kThreads = EXPWIN ? 320 : 192;
  static constexpr int kTmemCols = (2 * BN < 32) ? 32 : 2 * BN;
  static constexpr int kABytes = (EXPWIN ? SA : SE) * kTileBytes;
  static constexpr int kBBytes = SE * kXBytes;
  static constexpr int kEBytes = EXPWIN ? SE * kRecBytes : 0;
  static constexpr int kNumBars = 2 * SE + 2 * SA + 4;
  static constexpr size_t kSmem = 1024 + kABytes + kBBytes + kEBytes + kNumBars * 8 + 16;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(128, BN);
  static_assert(SE >= 4, "pipeline too shallow");
  static_assert(kSmem <= kSmemLimit, "shared memory budget");
  static_assert((kXBytes % 1024) == 0, "x tile must keep 1024-byte alignment");
};

struct Seg {
  int tile;
  int kb0;
  int kb1;
};

__device__ __forceinline__ bool next_seg(int64_t& u, int64_t u1, int KB, Seg& s) {
  if (u >= u1) return false;
  s.tile = static_cast<int>(u / KB);
  s.kb0 = static_cast<int>(u % KB);
  const int64_t rem = u1 - u;
  s.kb1 = static_cast<int>(rem < KB - s.kb0 ? s.kb0 + rem : KB);
  u += s.kb1 - s.kb0;
  return true;
}

// Decode 8 weights (one 16-byte chunk) of a 12-bit record.
__device__ __forceinline__ uint4 expwin_decode8(uint2 lo, uint32_t nb, uint32_t e0x4) {
  const uint32_t v0 = nb & 0x0F0F0F0Fu;
  const uint32_t v1 = (nb >> 4) & 0x0F0F0F0Fu;
  const uint32_t h0 = ((v0 & 0x07070707u) + e0x4) | ((v0 << 4) & 0x80808080u);
  const uint32_t h1 = ((v1 & 0x07070707u) + e0x4) | ((v1 << 4) & 0x80808080u);
  uint4 o;
  o.x = __byte_perm(lo.x, h0, 0x5140);
  o.y = __byte_perm(lo.x, h0, 0x7362);
  o.z = __byte_perm(lo.y, h1, 0x5140);
  o.w = __byte_perm(lo.y, h1, 0x7362);
  return o;
}

// Owner mode: sum, in CTA order, the partials of contributors c_first + 1 ..
// c_last for row r and tokens [0, mv) into pre[] (ws slot = contributor).
template <int BN>
__device__ __forceinline__ void owner_presum(const float* __restrict__ ws, int64_t cf, int64_t cl,
                                             int mv, int r, float (&pre)[BN]) {
  constexpr int64_t kStride = static_cast<int64_t>(BN) * kTileRows;
#pragma unroll
  for (int j = 0; j < BN; ++j) pre[j] = 0.f;
  if (mv <= 2) {
    // few tokens: many contributors per batch
    for (int64_t c = cf + 1; c <= cl; c += 16) {
      float v[16][2];
#pragma unroll
      for (int a = 0; a < 16; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b)
          v[a][b] = (c + a <= cl && b < mv) ? __ldcg(ws + (c + a) * kStride + b * kTileRows + r)
                                            : 0.f;
#pragma unroll
      for (int a = 0; a < 16; ++a) {
        pre[0] += v[a][0];
        if (BN > 1) pre[1] += v[a][1];
      }
    }
  } else {
#pragma unroll
    for (int j0 = 0; j0 < BN; j0 += 8) {
      if (j0 < mv) {
        for (int64_t c = cf + 1; c <= cl; c += 4) {
          float v[4][8];
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 8; ++b)
              v[a][b] = (c + a <= cl && j0 + b < mv)
                            ? __ldcg(ws + (c + a) * kStride + (j0 + b) * kTileRows + r)
                            : 0.f;
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 8; ++b) pre[j0 + b] += v[a][b];
        }
      }
    }
  }
}

template <int BN, bool EXPWIN>
__global__ void __launch_bounds__(Cfg<BN, EXPWIN>::kThreads, 1)
    tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const TcParams p) {
  using C = Cfg<BN, EXPWIN>;
  constexpr int SE = C::SE;
  constexpr int SA = C::SA;
  constexpr bool kOwnerOk = (BN <= 32);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + C::kABytes;
  uint8_t* sE = sB + C::kBBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sE + C::kEBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * SE;
  const uint32_t decf0 = empty0 + 8 * SE;
  const uint32_t dece0 = decf0 + 8 * SA;
  const uint32_t accf0 = dece0 + 8 * SA;
  const uint32_t acce0 = accf0 + 16;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t G = p.G;
  const int64_t U = static_cast<int64_t>(p.MT) * p.T * p.KB;
  const int64_t cta = blockIdx.x;
  const int64_t u0 = part_begin(cta, U, G);
  const int64_t u1 = part_begin(cta + 1, U, G);
  const bool owner_mode = kOwnerOk && p.reduce == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SE; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int s = 0; s < SA; ++s) {
      mbar_init(decf0 + 8 * s, 1);
      mbar_init(dece0 + 8 * s, 1);
    }
    mbar_init(accf0, 1);
    mbar_init(accf0 + 8, 1);
    mbar_init(acce0, 128);
    mbar_init(acce0 + 8, 128);
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
      int e = 0;
      uint32_t ph = 0;
      int64_t issued = 0;
      int64_t u = u0;
      Seg sg;
      bool ok = true;
      while (ok && next_seg(u, u1, p.KB, sg)) {
        const int t = sg.tile / p.MT;
        const int mt = sg.tile % p.MT;
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
          if (!mbar_wait(empty0 + 8 * e, ph ^ 1, p.status, kStatusTimeoutProducer)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + 8 * e;
          const size_t tile_idx = static_cast<size_t>(t) * p.KB + kb;
          if (EXPWIN) {
            mbar_arrive_expect_tx(fb, kRecBytes + C::kXBytes);
            bulk_g2s(smem_u32(sE + e * kRecBytes), p.w + tile_idx * kRecBytes, kRecBytes, fb,
                     pol);
          } else {
            mbar_arrive_expect_tx(fb, kTileBytes + C::kXBytes);
            bulk_g2s(smem_u32(sA + e * kTileBytes), p.w + tile_idx * kTileBytes, kTileBytes, fb,
                     pol);
          }
          tma_load_2d(smem_u32(sB + e * C::kXBytes), &tmap_x, kb * kTileK, mt * BN, fb);
          ++issued;
          if (++e == SE) {
            e = 0;
            ph ^= 1;
          }
        }
      }
      // Drain: every copy issued must have landed before the CTA may exit.
      const int64_t n = issued < SE ? issued : SE;
      for (int64_t j = 0; j < n; ++j) {
        const int64_t idx = issued - 1 - j;
        mbar_wait(full0 + 8 * static_cast<int>(idx % SE), static_cast<uint32_t>((idx / SE) & 1),
                  p.status, kStatusTimeoutDrain);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      int64_t j = 0;  // running unit index
      int64_t u = u0;
      Seg sg;
      int segi = 0;
      bool ok = true;
      while (ok && next_seg(u, u1, p.KB, sg)) {
        const int buf = segi & 1;
        if (!mbar_wait(acce0 + 8 * buf, ((segi >> 1) & 1) ^ 1, p.status, kStatusTimeoutMma)) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * BN;
        for (int kb = sg.kb0; kb < sg.kb1; ++kb, ++j) {
          const int e = static_cast<int>(j % SE);
          if (!mbar_wait(full0 + 8 * e, static_cast<uint32_t>((j / SE) & 1), p.status,
                         kStatusTimeoutMma)) {
            ok = false;
            break;
          }
          int a_idx = e;
          if (EXPWIN) {
            constexpr int SAd = SA > 0 ? SA : 1;
            a_idx = static_cast<int>(j % SAd);
            if (!mbar_wait(decf0 + 8 * a_idx, static_cast<uint32_t>((j / SAd) & 1), p.status,
                           kStatusTimeoutMma)) {
              ok = false;
              break;
            }
          }
          tc_fence_after();
          const uint32_t a = smem_u32(sA + a_idx * kTileBytes);
          const uint32_t b = smem_u32(sB + e * C::kXBytes);
#pragma unroll
          for (int k = 0; k < kTileK / 16; ++k) {
            tc_mma_f16(d, smem_desc_sw128(a + 32 * k), smem_desc_sw128(b + 32 * k), C::kIdesc,
                       (kb > sg.kb0 || k > 0) ? 1u : 0u);
          }
          tc_commit(empty0 + 8 * e);
          if (EXPWIN) tc_commit(dece0 + 8 * a_idx);
        }
        if (!ok) break;
        tc_commit(accf0 + 8 * buf);
        ++segi;
      }
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // tensor-memory lane quarter this warp may read
    const int r = q * 32 + lane;
    const int etid = threadIdx.x - 64;  // 0..127
    const int64_t first_tile = u0 / p.KB;
    constexpr int64_t kSlot = static_cast<int64_t>(BN) * kTileRows;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
    int pend[2];
    int npend = 0;
    int64_t u = u0;
    Seg sg;
    int segi = 0;
    bool ok = true;
    while (ok && next_seg(u, u1, p.KB, sg)) {
      const int buf = segi & 1;
      const int t = sg.tile / p.MT;
      const int mt = sg.tile % p.MT;
      const int mv = min(BN, p.m - mt * BN);
      const bool whole = (sg.kb0 == 0 && sg.kb1 == p.KB);
      const bool owner = owner_mode && !whole && sg.kb0 == 0;
      __nv_bfloat16* outp = out + static_cast<size_t>(mt) * BN * p.n_out +
                            static_cast<size_t>(t) * kTileRows + r;
      float pre[kOwnerOk ? BN : 1];
      if constexpr (kOwnerOk) {
        if (owner) {
          const TileSplit ts = tile_split(sg.tile, p.KB, U, G);
          ok = spin_until_ge(p.counters + sg.tile, static_cast<uint32_t>(ts.c_last - ts.c_first),
                             p.status);
          owner_presum<BN>(p.ws, ts.c_first, ts.c_last, mv, r, pre);
        }
      }
      if (!mbar_wait(accf0 + 8 * buf, (segi >> 1) & 1, p.status, kStatusTimeoutEpilogue)) break;
      tc_fence_after();
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * BN;
      float* slot = p.ws + (owner_mode ? cta : 2 * cta + (sg.tile == first_tile ? 0 : 1)) * kSlot;
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 16) {
        if (c0 < mv) {
          float v[16];
          tmem_ld16(taddr + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int j = c0 + jj;
            if (j < mv) {
              if (whole) {
                outp[static_cast<size_t>(j) * p.n_out] = __float2bfloat16_rn(v[jj]);
              } else if (owner) {
                if constexpr (kOwnerOk)
                  outp[static_cast<size_t>(j) * p.n_out] = __float2bfloat16_rn(v[jj] + pre[j]);
              } else {
                slot[j * kTileRows + r] = v[jj];
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(acce0 + 8 * buf);
      if (!whole) {
        if (owner) {
          named_bar_sync(1, 128);
          if (etid == 0) p.counters[sg.tile] = 0u;
        } else {
          // The barrier orders the warps' partial stores before thread 0's
          // release (cumulative), which publishes them with one arrival.
          named_bar_sync(1, 128);
          if (etid == 0) red_release_gpu_add(p.counters + sg.tile, 1u);
          if (!owner_mode) pend[npend++] = sg.tile;
        }
      }
      ++segi;
    }
    // distributed mode: reduce this CTA's share of each split tile it touched.
    // Shares are runs of 4 consecutive rows (one float4 of a partial slot);
    // each thread keeps 4 of them and 4 contributors' loads in flight.
    for (int i = 0; ok && i < npend; ++i) {
      const int tile = pend[i];
      const TileSplit ts = tile_split(tile, p.KB, U, G);
      const int64_t S = ts.c_last - ts.c_first + 1;
      if (!spin_until_ge(p.counters + tile, static_cast<uint32_t>(S), p.status)) break;
      const int t = tile / p.MT;
      const int mt = tile % p.MT;
      const int mv = min(BN, p.m - mt * BN);
      const int64_t nq = static_cast<int64_t>(kTileRows / 4) * mv;  // float4 quads
      const int64_t me = cta - ts.c_first;
      const int64_t q0 = me * nq / S, q1 = (me + 1) * nq / S;
      const int64_t s_first =
          2 * ts.c_first + ((part_begin(ts.c_first, U, G) / p.KB) == tile ? 0 : 1);
      const float4* ws4 = reinterpret_cast<const float4*>(p.ws);
      constexpr int64_t kSlot4 = kSlot / 4;
      for (int64_t qb = q0 + etid; qb < q1; qb += 128 * 4) {
        float4 acc[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int64_t q = qb + 128 * b;
          acc[b] = q < q1 ? __ldcg(ws4 + s_first * kSlot4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int64_t c = ts.c_first + 1; c <= ts.c_last; c += 4) {
          float4 v[4][4];
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              const int64_t q = qb + 128 * b;
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
          const int64_t q = qb + 128 * b;
          if (q < q1) {
            const int j = static_cast<int>(q / (kTileRows / 4));
            const int rr = static_cast<int>(q % (kTileRows / 4)) * 4;
            __nv_bfloat16* o = out + (static_cast<size_t>(mt) * BN + j) * p.n_out +
                               static_cast<size_t>(t) * kTileRows + rr;
            __nv_bfloat162 lo2, hi2;
            lo2.x = __float2bfloat16_rn(acc[b].x);
            lo2.y = __float2bfloat16_rn(acc[b].y);
            hi2.x = __float2bfloat16_rn(acc[b].z);
            hi2.y = __float2bfloat16_rn(acc[b].w);
            *reinterpret_cast<__nv_bfloat162*>(o) = lo2;
            *reinterpret_cast<__nv_bfloat162*>(o + 2) = hi2;
          }
        }
      }
      named_bar_sync(1, 128);
      if (etid == 0) {
        const uint32_t old = atomicAdd(p.counters + tile, 1u);
        if (old == static_cast<uint32_t>(2 * S - 1)) p.counters[tile] = 0u;
      }
    }
  } else if (EXPWIN) {
    // -------------------------------------------------------------- decode
    // Decode warp d (0..3) owns every unit j with j % 4 == d and the decoded
    // buffer d, so stages decode in parallel with warp-local syncs only.
    constexpr int SAd = SA > 0 ? SA : 1;
    const int d = warp - 6;
    int64_t j = 0;
    int64_t u = u0;
    Seg sg;
    bool ok = true;
    while (ok && next_seg(u, u1, p.KB, sg)) {
      for (int kb = sg.kb0; kb < sg.kb1; ++kb, ++j) {
        if (static_cast<int>(j % SAd) != d) continue;
        // SE is a multiple of 4, so slot e only ever belongs to decode warp
        // e % 4, which consumes its generations in order (a parity wait
        // cannot tell one lap of the ring from the one two laps earlier).
        const int e = static_cast<int>(j % SE);
        if (!mbar_wait(full0 + 8 * e, static_cast<uint32_t>((j / SE) & 1), p.status,
                       kStatusTimeoutDecode) ||
            !mbar_wait(dece0 + 8 * d, static_cast<uint32_t>(((j / SAd) & 1) ^ 1), p.status,
                       kStatusTimeoutDecode)) {
          ok = false;
          break;
        }
        const uint8_t* rec = sE + e * kRecBytes;
        uint8_t* a = sA + d * kTileBytes;
#pragma unroll 8
        for (int ch = lane; ch < 1024; ch += 32) {
          const int rr = ch >> 3, cc = ch & 7;
          const uint2 lo = *reinterpret_cast<const uint2*>(rec + kRecLowOff + ch * 8);
          const uint32_t nb = *reinterpret_cast<const uint32_t*>(rec + kRecNibOff + ch * 4);
          *reinterpret_cast<uint4*>(a + rr * 128 + ((cc ^ (rr & 7)) << 4)) =
              expwin_decode8(lo, nb, p.e0x4);
        }
        __syncwarp();
        const uint32_t* esc = reinterpret_cast<const uint32_t*>(rec + kRecEscOff);
        const uint32_t cnt = esc[0];
        if (lane < static_cast<int>(cnt) && lane < kEscCap) {
          const uint32_t ent = esc[1 + lane];
          const uint32_t pos = ent >> 8;
          const int rr = static_cast<int>(pos >> 6), kk = static_cast<int>(pos & 63);
          a[rr * 128 + (((kk >> 3) ^ (rr & 7)) << 4) + (kk & 7) * 2 + 1] =
              static_cast<uint8_t>(ent & 0xFF);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(decf0 + 8 * d);
      }
    }
  }

  tc_fence_before();
  // __syncthreads is an aligned barrier: the producer and MMA warps, whose
  // lane 0 ran their loops alone, reconverge first.
  __syncwarp();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int BN, bool EXPWIN>
cudaError_t set_attr() {
  return cudaFuncSetAttribute(tc_kernel<BN, EXPWIN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(Cfg<BN, EXPWIN>::kSmem));
}

template <int BN, bool EXPWIN>
cudaError_t launch(const CUtensorMap& tmap, const TcParams& p, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(Cfg<BN, EXPWIN>::kThreads);
  cfg.dynamicSmemBytes = Cfg<BN, EXPWIN>::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_kernel<BN, EXPWIN>, tmap, p);
}

}  // namespace

bool tc_supported(int BN, bool expwin) {
  if (expwin) return BN == 16 || BN == 32 || BN == 64 || BN == 128;
  return BN == 16 || BN == 32 || BN == 64 || BN == 128 || BN == 256;
}

int tc_threads(bool expwin) { return expwin ? 320 : 192; }

#define PROJ_TC_SWITCH(BN, EXPWIN, ...)              \
  do {                                                  \
    if (EXPWIN) {                                       \
      switch (BN) {                                     \
        case 16: { constexpr int kB = 16; constexpr bool kE = true; __VA_ARGS__; } \
        case 32: { constexpr int kB = 32; constexpr bool kE = true; __VA_ARGS__; } \
        case 64: { constexpr int kB = 64; constexpr bool kE = true; __VA_ARGS__; } \
        case 128: { constexpr int kB = 128; constexpr bool kE = true; __VA_ARGS__; } \
      }                                                 \
    } else {                                            \
      switch (BN) {                                     \
        case 16: { constexpr int kB = 16; constexpr bool kE = false; __VA_ARGS__; } \
        case 32: { constexpr int kB = 32; constexpr bool kE = false; __VA_ARGS__; } \
        case 64: { constexpr int kB = 64; constexpr bool kE = false; __VA_ARGS__; } \
        case 128: { constexpr int kB = 128; constexpr bool kE = false; __VA_ARGS__; } \
        case 256: { constexpr int kB = 256; constexpr bool kE = false; __VA_ARGS__; } \
      }                                                 \
    }                                                   \
  } while (0)

size_t tc_smem_bytes(int BN, bool expwin) {
  PROJ_TC_SWITCH(BN, expwin, return Cfg<kB, kE>::kSmem);
  return 0;
}

int tc_stages(int BN, bool expwin) {
  PROJ_TC_SWITCH(BN, expwin, return Cfg<kB, kE>::SE);
  return 0;
}

cudaError_t tc_init_attributes() {
  cudaError_t e;
  if ((e = set_attr<16, false>()) != cudaSuccess) return e;
  if ((e = set_attr<32, false>()) != cudaSuccess) return e;
  if ((e = set_attr<64, false>()) != cudaSuccess) return e;
  if ((e = set_attr<128, false>()) != cudaSuccess) return e;
  if ((e = set_attr<256, false>()) != cudaSuccess) return e;
  if ((e = set_attr<16, true>()) != cudaSuccess) return e;
  if ((e = set_attr<32, true>()) != cudaSuccess) return e;
  if ((e = set_attr<64, true>()) != cudaSuccess) return e;
  if ((e = set_attr<128, true>()) != cudaSuccess) return e;
  return cudaSuccess;
}

cudaError_t tc_launch(int BN, bool expwin, const CUtensorMap& tmap, const TcParams& p,
                      cudaStream_t s) {
  PROJ_TC_SWITCH(BN, expwin, return (launch<kB, kE>(tmap, p, s)));
  return cudaErrorInvalidValue;
}

}  // namespace proj
