// gemm_tc.cu -- tensor-core skinny GEMM for the bf16 layers, every token count.
//
// out[i, n] = sum_k x[i, k] W[n, k]            (muse_bf16_proj guide, ch. 1, §1.1)
//
// GB300 design (the pages' H200 kernels -- warp-level mma GEMVs with
// in-CTA split-K, wgmma GEMMs -- are prior art, not the blueprint):
//
// * Operand roles are swapped: 128 weight rows are the MMA's M side (A,
//   K-major, from shared memory), the m tokens are its N side (B, N = BN =
//   m rounded up to 16..256), so even m = 1 runs one tcgen05.mma.kind::f16
//   M128 x N16 x K16 per 16 columns with fp32 accumulation in tensor memory.
// * Weights stream HBM -> shared memory with 1-D bulk copies of prepacked,
//   pre-swizzled 16 KB tiles (one copy per 128 x 64 tile, evict-first), x
//   with a 2-D TMA load whose out-of-range rows read as zero (ragged m).
//   A deep mbarrier ring (4-12 stages) keeps >= 64 KB in flight per SM,
//   enough to cover HBM latency at the per-SM share of bandwidth.
// * Exactly one CTA per SM, 152 on GB300, and a split-K partition that
//   gives every CTA the same number of (tile, k-block) units: the CTAs cut
//   the linear order of units into G equal ranges (so a tile may be shared
//   by several CTAs).  A CTA that finishes a whole tile writes bf16 output
//   directly; a shared tile's CTAs write fp32 partials, bump a per-tile
//   counter (acq_rel), and the last to arrive sums the partials in fixed CTA
//   order (= ascending k), writes the output and resets the counter to zero
//   on the GPU (muse_bf16_proj notebook, n. 19 "Split-K and the cost of
//   combining work", last-arriving-block design; guide ch. 1, §1.6: counters
//   are reset on the GPU).  No spin-wait on another CTA, one launch per call,
//   deterministic results.
// * Warp roles: warp 0 issues copies, warp 1 issues MMAs (and owns the
//   tensor memory), warps 2-5 drain the accumulators; the 12-bit variant adds
//   warps 6-9, which decode each record into the swizzled bf16 tile in shared
//   memory and patch its escapes before the MMA reads it, so the MMA inputs
//   -- and therefore the outputs -- are bit-identical to the dense kernel's
//   (project report, "Round 5 -- lossless 12-bit compressed weights").
// * The accumulator is double-buffered in tensor memory so the epilogue of
//   one tile overlaps the MMAs of the next.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace proj {
namespace {

constexpr int kSmemLimit = 232448;  // max dynamic shared memory per block
constexpr int kSmemReserve = 1024 + 512;  // alignment slack + barriers

template <int BN, bool EXPWIN>
struct Cfg {
  static constexpr int kXBytes = BN * 128;
  static constexpr int kStageBytes = kTileBytes + kXBytes + (EXPWIN ? kRecBytes : 0);
  static constexpr int kStagesFit = (kSmemLimit - kSmemReserve) / kStageBytes;
  static constexpr int kStages = kStagesFit > 12 ? 12 : kStagesFit;
  static constexpr int kThreads = EXPWIN ? 320 : 192;
  static constexpr int kTmemCols = (2 * BN < 32) ? 32 : 2 * BN;
  static constexpr int kABytes = kStages * kTileBytes;
  static constexpr int kBBytes = kStages * kXBytes;
  static constexpr int kEBytes = EXPWIN ? kStages * kRecBytes : 0;
  static constexpr int kNumBars = 3 * kStages + 4;
  static constexpr size_t kSmem = 1024 + kABytes + kBBytes + kEBytes + kNumBars * 8 + 16;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(128, BN);
  static_assert(kStages >= 3, "pipeline too shallow");
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

template <int BN, bool EXPWIN>
__global__ void __launch_bounds__(Cfg<BN, EXPWIN>::kThreads, 1)
    tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const TcParams p) {
  using C = Cfg<BN, EXPWIN>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + C::kABytes;
  uint8_t* sE = sB + C::kBBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sE + C::kEBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile uint32_t* last_flag = tmem_slot + 1;

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * S;
  const uint32_t dec0 = empty0 + 8 * S;
  const uint32_t accf0 = dec0 + 8 * S;
  const uint32_t acce0 = accf0 + 16;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t G = p.G;
  const int64_t U = static_cast<int64_t>(p.MT) * p.T * p.KB;
  const int64_t u0 = part_begin(blockIdx.x, U, G);
  const int64_t u1 = part_begin(blockIdx.x + 1, U, G);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
      mbar_init(dec0 + 8 * s, 1);
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
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      int64_t u = u0;
      Seg sg;
      bool ok = true;
      while (ok && next_seg(u, u1, p.KB, sg)) {
        const int t = sg.tile / p.MT;
        const int mt = sg.tile % p.MT;
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, p.status, kStatusTimeoutProducer)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + 8 * stage;
          const size_t tile_idx = static_cast<size_t>(t) * p.KB + kb;
          if (EXPWIN) {
            mbar_arrive_expect_tx(fb, kRecBytes + C::kXBytes);
            bulk_g2s(smem_u32(sE + stage * kRecBytes), p.w + tile_idx * kRecBytes, kRecBytes, fb,
                     pol);
          } else {
            mbar_arrive_expect_tx(fb, kTileBytes + C::kXBytes);
            bulk_g2s(smem_u32(sA + stage * kTileBytes), p.w + tile_idx * kTileBytes, kTileBytes,
                     fb, pol);
          }
          tma_load_2d(smem_u32(sB + stage * C::kXBytes), &tmap_x, kb * kTileK, mt * BN, fb);
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Drain: every copy issued must have landed before the CTA may exit.
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
      int stage = 0;
      uint32_t phase = 0;
      int64_t u = u0;
      Seg sg;
      int segi = 0;
      bool ok = true;
      while (ok && next_seg(u, u1, p.KB, sg)) {
        const int buf = segi & 1;
        if (!mbar_wait(acce0 + 8 * buf, ((segi >> 1) & 1) ^ 1, p.status, kStatusTimeoutMma)) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * BN;
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, p.status, kStatusTimeoutMma)) {
            ok = false;
            break;
          }
          if (EXPWIN && !mbar_wait(dec0 + 8 * stage, phase, p.status, kStatusTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = smem_u32(sA + stage * kTileBytes);
          const uint32_t b = smem_u32(sB + stage * C::kXBytes);
#pragma unroll
          for (int k = 0; k < kTileK / 16; ++k) {
            tc_mma_f16(d, smem_desc_sw128(a + 32 * k), smem_desc_sw128(b + 32 * k), C::kIdesc,
                       (kb > sg.kb0 || k > 0) ? 1u : 0u);
          }
          tc_commit(empty0 + 8 * stage);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
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
    int64_t u = u0;
    Seg sg;
    int segi = 0;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
    while (next_seg(u, u1, p.KB, sg)) {
      const int buf = segi & 1;
      if (!mbar_wait(accf0 + 8 * buf, (segi >> 1) & 1, p.status, kStatusTimeoutEpilogue)) break;
      tc_fence_after();
      const int t = sg.tile / p.MT;
      const int mt = sg.tile % p.MT;
      const int mv = min(BN, p.m - mt * BN);
      const bool whole = (sg.kb0 == 0 && sg.kb1 == p.KB);
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * BN;
      const size_t out_col = static_cast<size_t>(t) * kTileRows + r;
      const size_t out_row0 = static_cast<size_t>(mt) * BN;
      float* slot = p.ws + (2 * static_cast<int64_t>(blockIdx.x) + (sg.tile == first_tile ? 0 : 1)) *
                               (static_cast<int64_t>(BN) * kTileRows);
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        if (c0 >= mv) break;
        float v[16];
        tmem_ld16(taddr + c0, v);
        tmem_ld_wait();
        if (whole) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < mv)
              out[(out_row0 + c0 + j) * p.n_out + out_col] = __float2bfloat16_rn(v[j]);
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < mv) slot[(c0 + j) * kTileRows + r] = v[j];
        }
      }
      tc_fence_before();
      mbar_arrive(acce0 + 8 * buf);
      if (!whole) {
        __threadfence();
        named_bar_sync(1, 128);
        const int64_t tu0 = static_cast<int64_t>(sg.tile) * p.KB;
        const int64_t c_first = part_owner(tu0, U, G);
        const int64_t c_last = part_owner(tu0 + p.KB - 1, U, G);
        if (etid == 0) {
          const uint32_t old = atom_add_acq_rel_gpu(p.counters + sg.tile, 1u);
          *last_flag = (old == static_cast<uint32_t>(c_last - c_first)) ? 1u : 0u;
        }
        named_bar_sync(1, 128);
        if (*last_flag) {
          __threadfence();
          for (int j = 0; j < mv; ++j) {
            float acc = 0.f;
            for (int64_t c = c_first; c <= c_last; ++c) {
              const int64_t s = 2 * c + ((part_begin(c, U, G) / p.KB) == sg.tile ? 0 : 1);
              acc += __ldcg(p.ws + s * (static_cast<int64_t>(BN) * kTileRows) + j * kTileRows + r);
            }
            out[(out_row0 + j) * p.n_out + out_col] = __float2bfloat16_rn(acc);
          }
          if (etid == 0) p.counters[sg.tile] = 0u;
        }
        named_bar_sync(1, 128);
      }
      ++segi;
    }
  } else if (EXPWIN) {
    // -------------------------------------------------------------- decode
    const int dtid = threadIdx.x - 192;  // 0..127
    int stage = 0;
    uint32_t phase = 0;
    int64_t u = u0;
    Seg sg;
    bool ok = true;
    while (ok && next_seg(u, u1, p.KB, sg)) {
      for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
        if (!mbar_wait(full0 + 8 * stage, phase, p.status, kStatusTimeoutDecode)) {
          ok = false;
          break;
        }
        const uint8_t* rec = sE + stage * kRecBytes;
        uint8_t* a = sA + stage * kTileBytes;
#pragma unroll 4
        for (int ch = dtid; ch < 1024; ch += 128) {
          const int rr = ch >> 3, cc = ch & 7;
          const uint2 lo = *reinterpret_cast<const uint2*>(rec + kRecLowOff + ch * 8);
          const uint32_t nb = *reinterpret_cast<const uint32_t*>(rec + kRecNibOff + ch * 4);
          *reinterpret_cast<uint4*>(a + rr * 128 + ((cc ^ (rr & 7)) << 4)) =
              expwin_decode8(lo, nb, p.e0x4);
        }
        named_bar_sync(2, 128);
        const uint32_t* esc = reinterpret_cast<const uint32_t*>(rec + kRecEscOff);
        const uint32_t cnt = esc[0];
        if (dtid < static_cast<int>(cnt) && dtid < kEscCap) {
          const uint32_t e = esc[1 + dtid];
          const uint32_t pos = e >> 8;
          const int rr = static_cast<int>(pos >> 6), kk = static_cast<int>(pos & 63);
          a[rr * 128 + (((kk >> 3) ^ (rr & 7)) << 4) + (kk & 7) * 2 + 1] =
              static_cast<uint8_t>(e & 0xFF);
        }
        fence_proxy_async_smem();
        named_bar_sync(2, 128);
        if (dtid == 0) mbar_arrive(dec0 + 8 * stage);
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  }

  tc_fence_before();
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
  tc_kernel<BN, EXPWIN><<<p.G, Cfg<BN, EXPWIN>::kThreads, Cfg<BN, EXPWIN>::kSmem, s>>>(tmap, p);
  return cudaGetLastError();
}

}  // namespace

bool tc_supported(int BN, bool expwin) {
  if (expwin) return BN == 16 || BN == 32;
  return BN == 16 || BN == 32 || BN == 64 || BN == 128 || BN == 256;
}

int tc_threads(bool expwin) { return expwin ? 320 : 192; }

size_t tc_smem_bytes(int BN, bool expwin) {
  if (expwin) {
    switch (BN) {
      case 16: return Cfg<16, true>::kSmem;
      case 32: return Cfg<32, true>::kSmem;
    }
    return 0;
  }
  switch (BN) {
    case 16: return Cfg<16, false>::kSmem;
    case 32: return Cfg<32, false>::kSmem;
    case 64: return Cfg<64, false>::kSmem;
    case 128: return Cfg<128, false>::kSmem;
    case 256: return Cfg<256, false>::kSmem;
  }
  return 0;
}

int tc_stages(int BN, bool expwin) {
  if (expwin) {
    switch (BN) {
      case 16: return Cfg<16, true>::kStages;
      case 32: return Cfg<32, true>::kStages;
    }
    return 0;
  }
  switch (BN) {
    case 16: return Cfg<16, false>::kStages;
    case 32: return Cfg<32, false>::kStages;
    case 64: return Cfg<64, false>::kStages;
    case 128: return Cfg<128, false>::kStages;
    case 256: return Cfg<256, false>::kStages;
  }
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
  return cudaSuccess;
}

cudaError_t tc_launch(int BN, bool expwin, const CUtensorMap& tmap, const TcParams& p,
                      cudaStream_t s) {
  if (expwin) {
    switch (BN) {
      case 16: return launch<16, true>(tmap, p, s);
      case 32: return launch<32, true>(tmap, p, s);
    }
    return cudaErrorInvalidValue;
  }
  switch (BN) {
    case 16: return launch<16, false>(tmap, p, s);
    case 32: return launch<32, false>(tmap, p, s);
    case 64: return launch<64, false>(tmap, p, s);
    case 128: return launch<128, false>(tmap, p, s);
    case 256: return launch<256, false>(tmap, p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace proj
