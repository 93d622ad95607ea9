// api.cu -- the C ABI of libproj (declared in include/proj.h).
//
// prepare (untimed) validates the layer's fixed shape, repacks W into the
// kernels' tile layouts, optionally builds the 12-bit exponent-window copy,
// and allocates the split-K workspace and counters (zeroed once; the kernels
// return every counter to zero).  run validates, picks a kernel from the
// token count alone, encodes the x tensor map and launches one kernel.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>

#include "../../include/proj.h"
#include "kernels.h"

using namespace proj;

namespace {

// ------------------------------------------------------------------ errors --
thread_local int g_last_status = PROJ_OK;
thread_local char g_last_cuda[256] = "";

int fail(int status) {
  g_last_status = status;
  return status;
}

int fail_cuda(cudaError_t e, const char* what) {
  std::snprintf(g_last_cuda, sizeof g_last_cuda, "%s: %s", what, cudaGetErrorString(e));
  g_last_status = PROJ_ECUDA;
  return PROJ_ECUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// Error recording for entry points defined in other translation units.
int proj::record_status(int status, const char* text) {
  std::snprintf(g_last_cuda, sizeof g_last_cuda, "%s", text);
  return fail(status);
}

int proj::record_cuda(cudaError_t e, const char* what) { return fail_cuda(e, what); }

namespace {

// ------------------------------------------------------------ layer table --
struct LayerShape {
  int64_t N, K;
  int dtype;
};
// muse_bf16_proj guide, ch. 1, §1.1 table.
constexpr LayerShape kLayers[5] = {
    {2304, 8192, PROJ_BF16},  // qkv_gate
    {8192, 1024, PROJ_BF16},  // o
    {4096, 8192, PROJ_BF16},  // pooler
    {8192, 4096, PROJ_BF16},  // unpooler
    {256, 8192, PROJ_FP32},   // router
};
constexpr int64_t kUnpoolerSliceRows = 1024;
constexpr int64_t kUnpoolerSliceMaxM = 8;
constexpr int64_t kDefaultMMax = 1024;

// --------------------------------------------------------- tensor maps -----
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// x: bf16 [m, K] row-major; box = 64 columns x box_rows rows.
bool make_x_map(CUtensorMap* map, const void* x, int64_t m, int64_t K, int box_rows,
                bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(m)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A row-major bf16 [rows, K] matrix viewed as (32 columns, rows, K / 32
// steps): a box (32, box_rows, box_steps) lands as [step][row][64 bytes].
bool make_rows3_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int box_rows,
                    int box_steps) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {32u, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(K / 32)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, 64u};
  const cuuint32_t box[3] = {32u, static_cast<cuuint32_t>(box_rows),
                             static_cast<cuuint32_t>(box_steps)};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Ring shape of the row-run GEMV: steps per stage KS = SPW x (16 / block
// slots) for SPW in {1, 2, 4} (each consumer warp takes SPW steps of every
// stage), KS dividing K / 32, and the stages that fit shared memory (at
// most kGemvRowsMaxStages).  The longest stages that still leave three in
// the ring (or hold the whole run) win: measured on GB300, each stage costs
// a fixed hand-off (consumer release, producer re-issue) and each consumer
// warp's x loads are hidden better across more steps, so 4 steps per warp
// beat 1 by 1-4 us on every bf16 layer at 8 tokens although fewer bytes are
// in flight.
void rows_ring_shape(int nt, int nr_hi, int64_t K, int* ks_out, int* spw_out, int* s_out) {
  const int steps = static_cast<int>(K / 32);
  const int wpb = kGemvRowsConsumers / gemv_rows_block_slots(nr_hi);
  *ks_out = *spw_out = *s_out = 0;
  for (int spw = 1; spw <= 4; spw *= 2) {
    const int ks = spw * wpb;
    if (ks > steps || steps % ks) continue;
    int s = kGemvRowsMaxStages;
    while (s >= 2 && gemv_rows_smem(nt, ks, s, nr_hi) > static_cast<size_t>(kGemvRowsSmemMax)) --s;
    if (s < 2) continue;
    const int nst = steps / ks;
    if (s < 3 && nst > s) continue;
    *ks_out = ks;
    *spw_out = spw;
    *s_out = s;
  }
}

// The packed bf16 weight tiles (kTileBytes each, already the shared-memory
// image of the 128-byte swizzle) as a [tiles x 128][64] bf16 matrix: a box
// of 64 x 128 with no swizzle copies one tile verbatim.
bool make_w_map(CUtensorMap* map, const void* w, int64_t tiles) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kTileK),
                              static_cast<cuuint64_t>(tiles) * kTileRows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kTileK) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kTileK), static_cast<cuuint32_t>(kTileRows)};
  const cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int bn_for_m(int64_t m) {
  if (m <= 16) return 16;
  if (m <= 32) return 32;
  if (m <= 64) return 64;
  if (m <= 128) return 128;
  return 256;
}

// Token counts up to which the 12-bit copy is used by the dispatch table.
constexpr int64_t kExpwinAutoMaxM = 16;
// The stream-K tile kernel decodes the 12-bit tile records for any m, in
// token tiles of at most this many tokens (its decoded-tile ring, copy ring
// and x tiles fit shared memory up to 128).
constexpr int kExpwinMaxBN = 128;

// Split-K combine by token count: the owner sums the others' partials while
// its last segment streams (short tail, but one CTA reads S - 1 partials);
// the distributed form spreads that reading over the contributors.
constexpr int64_t kTcOwnerMaxM = 8;

constexpr int64_t kGemvMaxM = 2;
// The split-K router GEMV serves these token counts by default (measured on
// GB300, device time, cold L2: 1-2.2 us faster than the FP32-FMA cluster
// kernel at 9..24 tokens, slower at 32; at 5..8 tokens 0.4-1 us faster than
// the whole-row router GEMV alone, but a load with it last ran 1.5 us
// slower -- the cluster launch overlaps less with the previous kernel's
// tail -- so the whole-row form keeps 3..8).
constexpr int64_t kRouterGemvCcAutoMinM = 9;
constexpr int64_t kRouterGemvCcAutoMaxM = 24;
// m <= 2 with the 12-bit row-chunk records built: the dispatch table keeps
// the dense register GEMV (measured on GB300 at m = 1, 2 on the four bf16
// layers: the 12-bit form within +-0.6 us of it either way -- both are bound
// by the per-warp chain of load round trips, not by the bytes), so the
// records serve variant = EXPWIN12.
constexpr bool kRc12Auto = false;
// The router's few-token GEMV is the dispatch form up to this many tokens.
constexpr int64_t kRouterGemvAutoMaxM = 8;
// From three tokens to kGemvMmaMaxM the bf16 layers take the warp-MMA
// weight stream (measured faster than the tcgen05 cluster kernel there).
constexpr int64_t kGemvMmaMinM = 3;
// From three tokens on every layer goes to a cluster split-K kernel (the
// router to its FP32-FMA one); below that, the GEMV.
constexpr int64_t kClusterMinM = 3;
// The CTA-pair kernel is the dispatch form above 128 tokens on layers whose
// K needs no split (K <= 1024: o), and from kPairMinMSplit tokens on the
// wider-K layers when its shape splits K across at most two pairs (one
// cluster of four CTAs).  Measured on GB300 (device time, cold L2; pair
// against cluster kernel): o at 256 tokens 10.6 against 11.7 us; the
// unpooler at 192 and 256 tokens 21.0 / 21.6 against 22.0 / 22.5 us, at 320-512
// 27.1-28.1 against 32.0-32.8, at 1000 tokens 51.6 against 61.1; the pooler at
// 512 tokens 31.3 against 32.7.  Where the pairs must split K three or more
// ways (the pooler and qkv_gate at 256 tokens: 23.6 / 18.8 against 23.0 /
// 17.5 us), and below 192 tokens on the wider layers (unpooler at 129: 22.2
// against 21.4), the cluster kernel stays.
constexpr int64_t kPairMinM = 129;
constexpr int64_t kPairMaxK = 1024;
constexpr int64_t kPairMinMSplit = 192;
constexpr int kPairMaxAutoKG = 2;
constexpr int64_t kRouterClusterMinM = 3;
constexpr int kRouterMaxBN = 64;  // widest token tile of the FP32-FMA router kernel

int bn_for_cluster(int64_t m) {
  if (m <= 16) return 16;
  if (m <= 32) return 32;
  if (m <= 64) return 64;
  return m <= 128 ? 128 : 256;
}
int bn_index(int bn) { return bn == 16 ? 0 : bn == 32 ? 1 : bn == 64 ? 2 : bn == 128 ? 3 : 4; }

// Launch shape of the cluster kernels: token tile bn (the smallest covering m,
// or one or two halvings of it), cluster size cs and clusters per tile kg,
// chosen by a cost model calibrated on GB300 (in-kernel timestamps and a
// bulk-copy probe):
//   stream  = max(k-blocks per CTA x per-k-block time, weight bytes / HBM);
//             an SM's copy engine takes max(~160 ns, bytes / 135 GB/s) per
//             request, and a k-block is two requests (16 KB of weights, then
//             bn x 128 B of x);
//   combine = the remote part of the cluster's partials: at cs >= 3 stored
//             to and loaded from L2 (~100 GB/s per SM each way), at cs = 2
//             through distributed shared memory (~30 GB/s per SM) plus a
//             second cluster barrier;
//   groups  = kg > 1 adds a fence, an atomic and an L2 round trip (~2 us)
//             plus the last cluster's reads of the kg partials;
//   FP32 FMA router: the stream cannot beat the CUDA cores' FMA rate.
// Candidates keep every cluster resident in one wave (max_active), at most
// one CTA per SM and at least kMinKbPerCta k-blocks per CTA (the FP32-FMA
// router, whose k-blocks each carry ~1 us of FMAs at m = 16, only
// kMinKbPerCtaFma: spreading its FMAs over every SM outweighs the pipeline
// fill).
constexpr int kMinKbPerCta = 4;
constexpr int kMinKbPerCtaFma = 2;
struct ClusterShape {
  int bn, cs, kg;
};
struct ClusterCost {
  int64_t weight_bytes = 0;  // bytes of weights one call streams
  int w_request = 16384;     // bytes of one weight-tile copy (one per k-block)
  bool fma = false;          // CUDA-core FP32 FMAs instead of the tensor cores
};
ClusterShape pick_cluster(int64_t m, int T, int KB, const ClusterCost& cost, int sms, int bn0,
                          int bn_lo, const int (*max_active)[kClusterMaxCS]) {
  constexpr double kReqFloor = 160e-9;  // s per copy request, small copies
  constexpr double kReqRate = 135e9;    // bytes/s per SM, large copies
  constexpr double kHbm = 6.4e12;       // bytes/s, streaming reads
  constexpr double kDsmem = 30e9;       // bytes/s per SM, distributed shared memory
  constexpr double kL2 = 100e9;         // bytes/s per SM, partials through L2
  constexpr double kBarrier = 0.4e-6;   // s, a cluster barrier
  constexpr double kGroupFixed = 2e-6;  // s
  constexpr double kFmaRate = 150e9;    // FP32 FMAs/s per SM, fma.rn.f32x2 register tiles
  constexpr double kStageSync = 0.15e-6;  // s per stage of the FMA kernel (barriers)
  const int64_t weight_bytes = cost.weight_bytes;
  ClusterShape best{bn0, 1, 1};
  double best_t = 1e30;
  for (int bn = bn0; bn >= 16 && bn >= bn_lo; bn /= 2) {
    const int64_t tiles = static_cast<int64_t>(T) * ((m + bn - 1) / bn);
    const double part = 128.0 * bn * 4;  // one CTA's partial, bytes
    for (int kg = 1; kg <= kClusterMaxGroups; ++kg) {
      for (int cs = 1; cs <= kClusterMaxCS; ++cs) {
        if (cs * kg > 1 && KB / (cs * kg) < (cost.fma ? kMinKbPerCtaFma : kMinKbPerCta))
          continue;
        const int64_t ctas = tiles * cs * kg;
        if (ctas > sms && !(cs == 1 && kg == 1)) continue;
        const int act = max_active[bn_index(bn)][cs - 1];
        if (act > 0 && tiles * kg > act && !(cs == 1 && kg == 1)) continue;
        const double nk = static_cast<double>(KB) / (cs * kg);
        const double waves = static_cast<double>((ctas + sms - 1) / sms);
        const double t_kb = std::max(kReqFloor, cost.w_request / kReqRate) +
                            std::max(kReqFloor, 128.0 * bn / kReqRate);
        double t = std::max(nk * t_kb * waves, static_cast<double>(weight_bytes) / kHbm);
        if (cost.fma) {
          // the CTAs with the most k-blocks set the time
          const double nk_max = static_cast<double>((KB + cs * kg - 1) / (cs * kg));
          t = std::max(t, nk_max * (128.0 * bn * kTileK / kFmaRate + kStageSync) * waves);
        }
        if (cs >= 3)  // exchanged through L2: stored and loaded once each
          t += 2.0 * (cs - 1.0) / cs * part / kL2;
        else if (cs == 2)  // through distributed shared memory, and a second barrier
          t += 0.5 * part / kDsmem + kBarrier;
        if (kg > 1) t += kGroupFixed + kg * (part / cs) / kL2;
        // ties (the weight stream at the HBM rate): fewer groups, then more
        // CTAs per cluster (more streams in flight measured faster)
        if (t < best_t * 0.999 ||
            (t < best_t * 1.001 && (kg < best.kg || (kg == best.kg && cs > best.cs)))) {
          best_t = t;
          best = ClusterShape{bn, cs, kg};
        }
      }
    }
  }
  return best;
}
// The FP32-FMA router's launch shape, when one wave of clusters of four holds
// it: token tiles of 16 up to 48 tokens and of 32 above, clusters of four
// CTAs splitting K, and as many clusters per tile as fill the SMs (at most
// eight).  A device-time sweep of every shape (token tile 16/32/64 x cluster
// size 1..8 x clusters per tile 1..16, cold L2) at 25..512 tokens put
// clusters of four within 0.5 us of the best shape at every token count and
// found the cost model above 0.7-2.6 us off at 25-48, 96, 256 and 512 tokens:
// its smooth terms miss how clusters of three, six or seven CTAs pack into
// the GPU's processing clusters (144 CTAs in clusters of three or six took
// twice the time of 128 in clusters of four, though the occupancy query
// admits them).  Returns bn = 0 where the rule does not apply.
ClusterShape router_fma_shape(int64_t m, int T, int KB, int sms,
                              const int (*max_active)[kClusterMaxCS]) {
  constexpr int kCs = 4;
  constexpr int kMaxKg = 8;
  const int bn = m <= 48 ? 16 : 32;
  const int64_t tiles = static_cast<int64_t>(T) * ((m + bn - 1) / bn);
  int kg = static_cast<int>(std::min<int64_t>(kMaxKg, sms / (kCs * tiles)));
  while (kg >= 1 && KB / (kCs * kg) < kMinKbPerCtaFma) --kg;
  if (kg < 1) return ClusterShape{0, 0, 0};
  const int act = max_active[bn_index(bn)][kCs - 1];
  if (act > 0 && tiles * kg > act) return ClusterShape{0, 0, 0};
  return ClusterShape{bn, kCs, kg};
}

// Launch shape of the CTA-pair kernel: token tile bn (the smallest covering
// m, or its half) and pairs per pair tile kg (one cluster of 2 kg CTAs).
// Scored like the cluster kernels: the stream is the slower of an SM's
// ingest per k-block (16 KB of weights plus bn / 2 x 128 B of x), the pair
// MMAs per k-block (4 MMAs of 128 x bn x 16 per SM at ~4096 multiply-adds
// per clock) and the weight bytes at the HBM rate, times the waves of
// clusters; kg > 1 adds a cluster barrier and the exchange of the partials'
// remote part through L2.  At least kMinKbPerCta k-blocks per CTA.  With
// kg > 1 the grid is at most one CTA per SM: the exchange slots are indexed
// by CTA and sized for that.
struct PairShape {
  int bn, kg;
};
int pair_bn_index(int bn) { return bn == 64 ? 0 : bn == 128 ? 1 : 2; }
PairShape pick_pair(int64_t m, int T, int KB, int sms, const int (*active)[kPairMaxKG],
                    int bn_hi, int bn_lo, int kg_force) {
  constexpr double kHbm = 7.0e12;      // bytes/s, streaming reads
  constexpr double kIngest = 135e9;    // bytes/s per SM into shared memory
  constexpr double kMmaClock = 1.9e9;  // SM clock under load, Hz
  constexpr double kL2 = 100e9;        // bytes/s per SM, partials through L2
  constexpr double kBarrier = 0.4e-6;  // s, a cluster barrier
  const double weight_bytes = static_cast<double>(T) * kTileRows * KB * kTileK * 2;
  PairShape best{0, 0};
  double best_t = 1e30;
  for (int bn = bn_hi; bn >= bn_lo && bn >= 64; bn /= 2) {
    const int64_t tiles = static_cast<int64_t>(T / 2) * ((m + bn - 1) / bn);
    for (int kg = 1; kg <= kPairMaxKG; ++kg) {
      if (kg_force && kg != kg_force) continue;
      if (kg > 1 && KB / kg < kMinKbPerCta) continue;
      if (kg > 1 && tiles * kg * 2 > sms) continue;
      const int act = active[pair_bn_index(bn)][kg - 1];
      if (act <= 0) continue;
      const double waves = static_cast<double>((tiles + act - 1) / act);
      const double nk = static_cast<double>((KB + kg - 1) / kg);
      const double t_kb = std::max((kTileBytes + 64.0 * bn) / kIngest, 2.0 * bn / kMmaClock);
      double t = std::max(nk * t_kb * waves, weight_bytes / kHbm);
      if (kg > 1) t += kBarrier + 2.0 * (kg - 1.0) / kg * (128.0 * bn * 4) / kL2;
      if (t < best_t * 0.999 || (t < best_t * 1.001 && kg < best.kg)) {
        best_t = t;
        best = PairShape{bn, kg};
      }
    }
  }
  return best;
}

int mt_for_gemv(int64_t m) { return m <= 1 ? 1 : 2; }

struct Plan {
  bool gemv;
  bool gemv_reg = false;  // m <= 2: register-streaming form
  bool gemv_mma = false;  // bf16, m <= 8: warp-MMA weight stream
  bool gemv_rows = false;  // bf16, m <= 32: row-run warp-MMA weight stream
  int bpw = 1;             // gemv_rows: 32-column steps per ring stage
  bool router_gemv = false;  // router, m <= 16: FP32-FMA weight stream
  bool router_gemv_cc = false;  // router, m <= 32: the same with K split across a cluster
  bool cluster;
  bool planes = false;  // router on the tensor cores (three bf16 planes)
  bool pair = false;    // CTA-pair tensor-core kernel (bf16 layers, wide token tiles)
  int KG = 1;  // cluster kernel: clusters per output tile; pair kernel: pairs per pair tile
  bool router;
  bool expwin;
  int reduce;   // 0 owner, 1 distributed
  int bn;       // BN (tensor core) or TM (router)
  int64_t n_out;
  int T, KB, MT;
  int G;
};

}  // namespace

struct proj_ctx {
  int layer = 0, dtype = 0;
  int64_t N = 0, K = 0, m_max = 0;
  int device = 0, num_sms = 0;
  uint8_t* w_dense = nullptr;
  size_t w_dense_bytes = 0;
  void* w_rows = nullptr;          // row-major copy for the streaming GEMV
  uint32_t* gemv_flags = nullptr;  // [num_sms], zero between calls
  float* gemv_ws = nullptr;        // [num_sms][2]
  uint8_t* w_planes = nullptr;     // router: bf16 planes hi/mid/lo as [N, 3K] tiles
  uint32_t* cl_counters = nullptr; // cluster groups: [SMs][16], zero between calls
  float* xch = nullptr;            // cluster partials' exchange: [SMs][256][128] fp32
  uint32_t* w_frag = nullptr;      // bf16 layers: 16 x 16 MMA-fragment tiles (few tokens)
  uint8_t* w_runs = nullptr;       // bf16 layers: the row-run layout of all N rows over runs_G CTAs
  int runs_G = 0;
  uint8_t* w_runs_slice = nullptr; // unpooler: the same for the slice's runs_slice_rows rows
  int runs_slice_G = 0;
  int64_t runs_slice_rows = 0;
  int cluster_active[5][kClusterMaxCS] = {};   // co-resident clusters: BN 16..256 x size 1..16
  int rcluster_active[5][kClusterMaxCS] = {};  // the same for the FP32-FMA router kernel
  int rgcc_active = 0;  // co-resident clusters of the split-K router GEMV
  int pair_active[3][kPairMaxKG] = {};  // co-resident pair-kernel clusters: BN 64..256 x kg
  bool wmap_ok = false;     // tmap_w describes w_dense (bf16 layers)
  CUtensorMap tmap_w;       // the packed weight tiles as [tiles x 128][64] bf16
  uint8_t* w_exp = nullptr;
  size_t w_exp_bytes = 0;
  uint8_t* w_rc12 = nullptr;       // 12-bit row-chunk records (register GEMV, m <= 2)
  uint32_t* rc12_esc = nullptr;    // their escape blocks
  uint8_t* w_frag12 = nullptr;     // the fragment-order copy as 12-bit records (warp-MMA GEMV)
  uint32_t* frag12_esc = nullptr;  // their escape blocks
  int e0 = 0;
  int64_t n_esc = 0;
  int exp_declined = 0;
  float* ws = nullptr;
  size_t ws_bytes = 0;
  uint32_t* counters = nullptr;
  size_t counters_bytes = 0;
  uint32_t* status = nullptr;
  void* x_stage = nullptr;
  void* out_stage = nullptr;
  struct MapEntry {
    const void* x;
    int64_t m;
    int box;
    bool swz;
    CUtensorMap map;
  } maps[8];
  int n_maps = 0, next_map = 0;
  struct RowsMapEntry {
    const void* base;
    int64_t rows;
    int box_rows, box_steps;
    CUtensorMap map;
  } rmaps[16];
  int n_rmaps = 0, next_rmap = 0;
};

namespace {

void free_ctx(proj_ctx* h) {
  if (!h) return;
  cudaFree(h->w_dense);
  cudaFree(h->w_planes);
  cudaFree(h->cl_counters);
  cudaFree(h->xch);
  cudaFree(h->w_frag);
  cudaFree(h->w_runs);
  cudaFree(h->w_runs_slice);
  cudaFree(h->w_rows);
  cudaFree(h->gemv_flags);
  cudaFree(h->gemv_ws);
  cudaFree(h->w_exp);
  cudaFree(h->w_rc12);
  cudaFree(h->rc12_esc);
  cudaFree(h->w_frag12);
  cudaFree(h->frag12_esc);
  cudaFree(h->ws);
  cudaFree(h->counters);
  cudaFree(h->status);
  cudaFree(h->x_stage);
  cudaFree(h->out_stage);
  delete h;
}

const CUtensorMap* get_map(proj_ctx* h, const void* x, int64_t m, int box, bool swz) {
  for (int i = 0; i < h->n_maps; ++i) {
    auto& e = h->maps[i];
    if (e.x == x && e.m == m && e.box == box && e.swz == swz) return &e.map;
  }
  auto& e = h->maps[h->next_map];
  if (!make_x_map(&e.map, x, m, h->K, box, swz)) return nullptr;
  e.x = x;
  e.m = m;
  e.box = box;
  e.swz = swz;
  h->next_map = (h->next_map + 1) % 8;
  h->n_maps = std::min(h->n_maps + 1, 8);
  return &e.map;
}

const CUtensorMap* get_rows_map(proj_ctx* h, const void* base, int64_t rows, int box_rows,
                                int box_steps) {
  for (int i = 0; i < h->n_rmaps; ++i) {
    auto& e = h->rmaps[i];
    if (e.base == base && e.rows == rows && e.box_rows == box_rows && e.box_steps == box_steps)
      return &e.map;
  }
  auto& e = h->rmaps[h->next_rmap];
  if (!make_rows3_map(&e.map, base, rows, h->K, box_rows, box_steps)) return nullptr;
  e.base = base;
  e.rows = rows;
  e.box_rows = box_rows;
  e.box_steps = box_steps;
  h->next_rmap = (h->next_rmap + 1) % 16;
  h->n_rmaps = std::min(h->n_rmaps + 1, 16);
  return &e.map;
}

int64_t out_rows(const proj_ctx* h, int64_t m) {
  if (h->layer == PROJ_UNPOOLER && m <= kUnpoolerSliceMaxM) return kUnpoolerSliceRows;
  return h->N;
}

int make_plan(const proj_ctx* h, int64_t m, const proj_run_opts* opts, Plan* pl) {
  const int variant = opts ? opts->variant : PROJ_VARIANT_AUTO;
  const int kern = opts ? opts->kernel : PROJ_KERNEL_AUTO;
  if (kern < PROJ_KERNEL_AUTO || kern > PROJ_KERNEL_ROWS) return PROJ_EINVAL;
  if (variant < PROJ_VARIANT_AUTO || variant > PROJ_VARIANT_PLANES3) return PROJ_EINVAL;
  const int tile_n = opts ? opts->tile_n : 0;
  if (tile_n != 0 && tile_n != 16 && tile_n != 32 && tile_n != 64 && tile_n != 128 &&
      tile_n != 256)
    return PROJ_EINVAL;
  pl->router = (h->layer == PROJ_ROUTER);
  pl->n_out = out_rows(h, m);
  // Streaming GEMV: small m, uncompressed weights.
  const bool gemv_ok =
      m <= kGemvMaxM && (variant == PROJ_VARIANT_AUTO || variant == PROJ_VARIANT_DENSE ||
                         (variant == PROJ_VARIANT_EXPWIN12 && h->w_rc12));
  if ((kern == PROJ_KERNEL_GEMV || kern == PROJ_KERNEL_GEMV_REG) && !gemv_ok &&
      !(kern == PROJ_KERNEL_GEMV_REG && pl->router && m <= kRouterGemvMaxM))
    return PROJ_EUNSUPPORTED;
  if (gemv_ok && (kern == PROJ_KERNEL_GEMV || kern == PROJ_KERNEL_GEMV_REG ||
                  (kern == PROJ_KERNEL_AUTO && tile_n == 0))) {
    pl->gemv = true;
    pl->expwin = false;
    pl->reduce = 0;
    pl->bn = mt_for_gemv(m);
    pl->T = pl->KB = pl->MT = 0;
    int64_t G = h->num_sms;
    if (opts && opts->grid > 0) G = std::min<int64_t>(opts->grid, h->num_sms);
    pl->G = static_cast<int>(std::min<int64_t>(G, pl->n_out));
    // The register form (whole rows per CTA, weights straight to registers,
    // no cross-CTA step) measured faster than the ring form on every layer
    // at m = 1 and 2 on GB300; the ring form remains for the allocation-free
    // entry point and on request, and for runs longer than the register
    // form's chunk-partial buffer.
    const bool reg_ok = (pl->n_out + pl->G - 1) / pl->G * (h->K / 1024) <= kGemvRegMaxChunks;
    if (kern == PROJ_KERNEL_GEMV_REG && !reg_ok) return PROJ_EUNSUPPORTED;
    pl->gemv_reg = kern == PROJ_KERNEL_GEMV_REG || (kern == PROJ_KERNEL_AUTO && reg_ok);
    // The 12-bit records are read by the register form only.
    pl->expwin = h->w_rc12 && pl->gemv_reg &&
                 (variant == PROJ_VARIANT_EXPWIN12 || (variant == PROJ_VARIANT_AUTO && kRc12Auto));
    if (variant == PROJ_VARIANT_EXPWIN12 && !pl->expwin) return PROJ_EUNSUPPORTED;
    return PROJ_OK;
  }
  pl->gemv = false;
  pl->cluster = false;
  // The router GEMV with K split across a cluster (one 1024-column chunk
  // per CTA, eight rows per cluster): x staged per CTA is 1/8 of the
  // whole-row form's.
  if (kern == PROJ_KERNEL_GEMV_SPLITK ||
      (pl->router && kern == PROJ_KERNEL_AUTO &&
       (variant == PROJ_VARIANT_AUTO || variant == PROJ_VARIANT_DENSE) &&
       m >= kRouterGemvCcAutoMinM && m <= kRouterGemvCcAutoMaxM &&
       (!opts || (opts->grid == 0 && opts->groups == 0 && opts->tile_n == 0 &&
                  opts->reduce == PROJ_REDUCE_AUTO)))) {
    const int64_t clusters = (pl->n_out + 7) / 8;
    const bool ok = pl->router && m <= kRouterGemvCcMaxM && h->K % 1024 == 0 && h->K <= 8192 &&
                    (variant == PROJ_VARIANT_AUTO || variant == PROJ_VARIANT_DENSE) &&
                    h->rgcc_active >= clusters;
    if (ok) {
      pl->router_gemv_cc = true;
      pl->expwin = false;
      pl->reduce = 0;
      pl->bn = 8;
      pl->T = pl->KB = pl->MT = 0;
      pl->G = static_cast<int>(h->K / 1024);  // cluster size
      return PROJ_OK;
    }
    if (kern == PROJ_KERNEL_GEMV_SPLITK) return PROJ_EUNSUPPORTED;
  }
  // The router at 3..8 tokens (or on request, as the register form, to 16):
  // FP32 FMAs on a weight stream, whole rows per CTA.  (Measured on GB300:
  // 4.6-6.5 us against the cluster kernel's 8.6 at 3..8 tokens; a second
  // pass of eight tokens makes it slower than the cluster kernel.)
  if (pl->router && m <= kRouterGemvMaxM &&
      (kern == PROJ_KERNEL_GEMV_REG ||
       (kern == PROJ_KERNEL_AUTO &&
        (variant == PROJ_VARIANT_AUTO || variant == PROJ_VARIANT_DENSE) &&
        m <= kRouterGemvAutoMaxM &&
        (!opts || (opts->grid == 0 && opts->groups == 0 && opts->tile_n == 0 &&
                   opts->reduce == PROJ_REDUCE_AUTO))))) {
    int64_t G = std::min<int64_t>(pl->n_out, h->num_sms);
    if (opts && opts->grid > 0) G = std::min<int64_t>(opts->grid, pl->n_out);
    if (h->K % 1024 || h->K > 8192 || (pl->n_out + G - 1) / G * (h->K / 1024) > 16)
      return PROJ_EUNSUPPORTED;
    pl->router_gemv = true;
    pl->expwin = false;
    pl->reduce = 0;
    pl->bn = 8;
    pl->T = pl->KB = pl->MT = 0;
    pl->G = static_cast<int>(G);
    return PROJ_OK;
  }
  // A few tokens on the bf16 layers: the row-run warp-MMA weight stream
  // (whole row runs per CTA fed by tensor copies into a shared-memory ring).
  {
    int64_t G = std::min<int64_t>(pl->n_out, h->num_sms);
    if (opts && opts->grid > 0) G = std::min<int64_t>(opts->grid, pl->n_out);
    const int nt = m <= 8 ? 1 : (m <= 16 ? 2 : 4);  // tiles of 8 tokens
    const int64_t nr_hi = G > 0 ? (pl->n_out + G - 1) / G : 0;
    int ks = 0, spw = 0, stages = 0;
    if (nr_hi >= 1 && nr_hi <= kGemvRowsMaxRows && h->K % 32 == 0)
      rows_ring_shape(nt, static_cast<int>(nr_hi), h->K, &ks, &spw, &stages);
    if (opts && opts->groups > 0 && ks > 0) {  // forced steps per consumer warp and stage
      const int want = opts->groups;
      const int wpb = kGemvRowsConsumers / gemv_rows_block_slots(static_cast<int>(nr_hi));
      ks = (want == 1 || want == 2 || want == 4) && (h->K / 32) % (want * wpb) == 0 ? want * wpb
                                                                                   : 0;
      spw = want;
      if (ks) {
        stages = kGemvRowsMaxStages;
        while (stages >= 2 && gemv_rows_smem(nt, ks, stages, static_cast<int>(nr_hi)) >
                                  static_cast<size_t>(kGemvRowsSmemMax))
          --stages;
        if (stages < 2) ks = 0;
      }
    }
    const bool rows_ok = !pl->router && h->w_rows && m <= kGemvRowsMaxM && ks > 0 &&
                         (variant == PROJ_VARIANT_AUTO || variant == PROJ_VARIANT_DENSE);
    // Measured on GB300 (device time, cold L2) against the forms it replaces:
    // faster on the K = 8192 layers at 3..8 tokens (qkv_gate 10.4-10.7 us
    // against the warp-MMA GEMV's 10.6-11.6; pooler 14.6-15.0 against the
    // cluster kernel's 15.3-15.6), slower on o and the unpooler slice and
    // from 9 tokens on (each CTA reads all of x from L2: m x 16 KB at K =
    // 8192, on each consumer warp's critical path).
    const bool rows_auto = kern == PROJ_KERNEL_AUTO && m >= kGemvMmaMinM && m <= 8 &&
                           h->K >= 8192 &&
                           (!opts || (opts->grid == 0 && opts->groups == 0 &&
                                      opts->tile_n == 0 && opts->reduce == PROJ_REDUCE_AUTO));
    if (kern == PROJ_KERNEL_ROWS && !rows_ok) return PROJ_EUNSUPPORTED;
    if (rows_ok && (kern == PROJ_KERNEL_ROWS || rows_auto)) {
      pl->gemv_rows = true;
      pl->expwin = false;
      pl->reduce = 0;
      pl->bn = nt;
      pl->bpw = ks;
      pl->KG = stages;
      pl->MT = spw;
      pl->T = static_cast<int>(nr_hi);
      pl->KB = 0;
      pl->G = static_cast<int>(G);
      return PROJ_OK;
    }
  }
  // A few tokens on the bf16 layers: the warp-MMA weight stream.
  {
    const int64_t nb = pl->n_out / 16;
    int64_t G = std::min<int64_t>(nb, h->num_sms);
    if (opts && opts->grid > 0) G = std::min<int64_t>(opts->grid, nb);
    const int nt = m <= 8 ? 1 : (m <= 16 ? 2 : 4);  // tiles of 8 tokens
    // 12-bit weights: the recoded fragment copy, wherever the form fits
    const bool x12 = variant == PROJ_VARIANT_EXPWIN12 && h->w_frag12;
    const bool mma_ok = !pl->router && h->w_frag && m <= kGemvMmaMaxM &&
                        gemv_mma_fits(nt, static_cast<int>(h->K)) &&
                        (variant == PROJ_VARIANT_AUTO || variant == PROJ_VARIANT_DENSE || x12) &&
                        pl->n_out % 16 == 0 && G > 0 && (nb + G - 1) / G <= kGemvMmaMaxBlocks;
    // Measured against the cluster kernel on GB300: faster at 3..8 tokens
    // on qkv_gate (one block per CTA), o and the unpooler slice, and at 9..16
    // tokens on o (K = 1024: the cluster kernel's fixed costs dominate its
    // short stream); slower on the pooler (256 blocks over 152 CTAs, two for
    // most) and on the full unpooler (long streams over uneven blocks).
    const bool mma_shape = m <= 8 ? (nb % G == 0 || (nb + G - 1) / G == 1 || h->K <= 4096)
                                  : (m <= 16 && h->K <= 1024);
    const bool mma_auto = kern == PROJ_KERNEL_AUTO && m >= kGemvMmaMinM && mma_shape &&
                          (!opts || (opts->grid == 0 && opts->groups == 0 &&
                                     opts->tile_n == 0 && opts->reduce == PROJ_REDUCE_AUTO));
    if (kern == PROJ_KERNEL_MMA && !mma_ok) return PROJ_EUNSUPPORTED;
    if (mma_ok && (kern == PROJ_KERNEL_MMA || mma_auto ||
                   (x12 && kern == PROJ_KERNEL_AUTO && tile_n == 0))) {
      pl->gemv_mma = true;
      pl->expwin = x12;
      pl->reduce = 0;
      pl->bn = nt;
      pl->T = pl->KB = pl->MT = 0;
      pl->G = static_cast<int>(G);
      return PROJ_OK;
    }
  }
  // Wide token tiles on the bf16 layers: the CTA-pair kernel (M = 256 per
  // pair, half the x bytes per weight byte of a single CTA).
  {
    const int T = static_cast<int>(pl->n_out / kTileRows);
    const int KB = static_cast<int>(h->K / kTileK);
    const bool pair_req = kern == PROJ_KERNEL_PAIR;
    const bool pair_ok = !pl->router && h->wmap_ok && T % 2 == 0 &&
                         (variant == PROJ_VARIANT_AUTO || variant == PROJ_VARIANT_DENSE) &&
                         (tile_n == 0 || pair_supported(tile_n)) &&
                         (!opts || (opts->grid == 0 && opts->reduce == PROJ_REDUCE_AUTO &&
                                    opts->groups >= 0 && opts->groups <= kPairMaxKG));
    const bool pair_auto = kern == PROJ_KERNEL_AUTO && m >= kPairMinM &&
                           (h->K <= kPairMaxK || m >= kPairMinMSplit) &&
                           (!opts || (opts->grid == 0 && opts->groups == 0 &&
                                      opts->tile_n == 0 && opts->reduce == PROJ_REDUCE_AUTO));
    if (pair_req && !pair_ok) return PROJ_EUNSUPPORTED;
    const int bn_hi = tile_n ? tile_n : std::max(64, bn_for_cluster(m));
    // (automatic choice on the wider-K layers: the widest tile only -- the
    // 128-token pair tile measured slower there, e.g. the pooler at 256
    // tokens 26.3 us against 23.6 at 256 and 23.0 for the cluster kernel)
    const int bn_lo = tile_n ? tile_n
                      : (pair_auto && h->K > kPairMaxK) ? bn_hi
                                                         : std::max(64, bn_hi / 2);
    const PairShape ps = pair_ok && (pair_req || pair_auto)
                             ? pick_pair(m, T, KB, h->num_sms, h->pair_active, bn_hi, bn_lo,
                                         opts ? opts->groups : 0)
                             : PairShape{0, 0};
    // automatic choice on the wider-K layers: only shapes of at most two pairs per tile
    const bool pair_take =
        pair_req || (pair_auto && ps.bn != 0 && (h->K <= kPairMaxK || ps.kg <= kPairMaxAutoKG));
    if (pair_ok && pair_take) {
      if (ps.bn == 0) return PROJ_EUNSUPPORTED;  // no shape (k-blocks per CTA, residency)
      pl->pair = true;
      pl->cluster = false;
      pl->expwin = false;
      pl->reduce = 0;
      pl->bn = ps.bn;
      pl->KG = ps.kg;
      pl->T = T;
      pl->KB = KB;
      pl->MT = static_cast<int>((m + ps.bn - 1) / ps.bn);
      pl->G = (T / 2) * pl->MT * ps.kg * 2;  // CTAs
      return PROJ_OK;
    }
  }
  // The dispatch table sends wide token tiles to the cluster kernel; an
  // explicit grid or reduction mode names the global-memory split-K kernel.
  const bool auto_cluster = kern == PROJ_KERNEL_AUTO &&
                            m >= (pl->router ? kRouterClusterMinM : kClusterMinM) &&
                            (!opts || (opts->grid == 0 && opts->reduce == PROJ_REDUCE_AUTO &&
                                       opts->tile_n == 0));
  bool want_cluster;
  pl->planes = false;
  if (pl->router) {
    // From three tokens on (or when asked for) the router runs on the
    // cluster kernels: FP32 FMAs on its fp32 weights, or -- on request --
    // the tensor cores on its three exact bf16 planes.
    if (variant == PROJ_VARIANT_EXPWIN12 || kern == PROJ_KERNEL_TILE) return PROJ_EUNSUPPORTED;
    pl->planes = variant == PROJ_VARIANT_PLANES3;
    want_cluster = true;
  } else {
    if (variant == PROJ_VARIANT_PLANES3) return PROJ_EUNSUPPORTED;
    if (kern == PROJ_KERNEL_CLUSTER && variant == PROJ_VARIANT_EXPWIN12) return PROJ_EUNSUPPORTED;
    want_cluster =
        variant != PROJ_VARIANT_EXPWIN12 && (kern == PROJ_KERNEL_CLUSTER || auto_cluster);
  }
  if (want_cluster) {
    pl->cluster = true;
    pl->expwin = false;
    pl->reduce = 0;
    const bool fma = pl->router && !pl->planes;
    if (fma && tile_n > kRouterMaxBN) return PROJ_EUNSUPPORTED;
    pl->T = static_cast<int>(pl->n_out / kTileRows);
    pl->KB = static_cast<int>(h->K / kTileK) * (pl->planes ? 3 : 1);
    ClusterCost cost;
    cost.weight_bytes = pl->n_out * h->K * (pl->planes ? 6 : (pl->router ? 4 : 2));
    cost.w_request = fma ? kRfBytes : kTileBytes;
    cost.fma = fma;
    // A forced tile width, cluster size or group count keeps the token tile
    // the smallest covering m (or the forced one).
    const bool forced = opts && (opts->grid > 0 || opts->groups > 0);
    int bn0 = tile_n ? tile_n : bn_for_cluster(m);
    if (fma && bn0 > kRouterMaxBN) bn0 = kRouterMaxBN;
    ClusterShape shp =
        pick_cluster(m, pl->T, pl->KB, cost, h->num_sms, bn0, (tile_n || forced) ? bn0 : bn0 / 4,
                     fma ? h->rcluster_active : h->cluster_active);
    if (fma && !tile_n && !forced) {
      const ClusterShape r = router_fma_shape(m, pl->T, pl->KB, h->num_sms, h->rcluster_active);
      if (r.bn) shp = r;
    }
    pl->bn = shp.bn;
    pl->MT = static_cast<int>((m + pl->bn - 1) / pl->bn);
    int cs = shp.cs, kg = shp.kg;
    if (opts && (opts->grid > 0 || opts->groups > 0)) {
      cs = opts->grid > 0 ? opts->grid : 1;
      kg = opts->groups > 0 ? opts->groups : 1;
      if (cs > kClusterMaxCS || kg > kClusterMaxGroups) return PROJ_EINVAL;
      if (cs * kg > pl->KB) return PROJ_EUNSUPPORTED;
      // the group partials and counters are sized for one CTA per SM
      if (kg > 1 && static_cast<int64_t>(pl->MT) * pl->T * kg * cs > h->num_sms)
        return PROJ_EUNSUPPORTED;
    }
    pl->G = cs;  // cluster size
    pl->KG = kg;
    return PROJ_OK;
  }
  {
    bool use_exp = false;
    if (variant == PROJ_VARIANT_EXPWIN12) {
      if (!h->w_exp) return PROJ_EUNSUPPORTED;
      use_exp = true;
    } else if (variant == PROJ_VARIANT_AUTO) {
      use_exp = h->w_exp && m <= kExpwinAutoMaxM;
    } else if (variant != PROJ_VARIANT_DENSE) {
      return PROJ_EINVAL;
    }
    pl->expwin = use_exp;
    pl->bn = tile_n ? tile_n : bn_for_m(m);
    if (use_exp && !tile_n && pl->bn > kExpwinMaxBN) pl->bn = kExpwinMaxBN;
    if (use_exp && pl->bn > kExpwinMaxBN) return PROJ_EUNSUPPORTED;
    pl->T = static_cast<int>(pl->n_out / kTileRows);
    pl->KB = static_cast<int>(h->K / kTileK);
  }
  const int rq = opts ? opts->reduce : PROJ_REDUCE_AUTO;
  if (rq == PROJ_REDUCE_AUTO) {
    pl->reduce = (m <= kTcOwnerMaxM) ? 0 : 1;
  } else if (rq == PROJ_REDUCE_OWNER) {
    if (pl->bn > 32) return PROJ_EUNSUPPORTED;
    pl->reduce = 0;
  } else if (rq == PROJ_REDUCE_DISTRIBUTED) {
    pl->reduce = 1;
  } else {
    return PROJ_EINVAL;
  }
  pl->MT = static_cast<int>((m + pl->bn - 1) / pl->bn);
  const int64_t U = static_cast<int64_t>(pl->MT) * pl->T * pl->KB;
  int64_t G = h->num_sms;
  if (opts && opts->grid > 0) G = std::min<int64_t>(opts->grid, h->num_sms);
  pl->G = static_cast<int>(std::min<int64_t>(G, U));
  return PROJ_OK;
}

int choose_window(const uint32_t hist[128]) {
  int best_e0 = 0;
  int64_t best = -1;
  for (int e0 = 0; e0 <= 120; ++e0) {
    int64_t c = 0;
    for (int j = 0; j < 8; ++j) c += hist[e0 + j];
    if (c > best) {
      best = c;
      best_e0 = e0;
    }
  }
  return best_e0;
}

template <typename T>
cudaError_t dmalloc(T** p, size_t bytes) {
  return cudaMalloc(reinterpret_cast<void**>(p), bytes ? bytes : 16);
}

}  // namespace

// ============================================================================
extern "C" {

int proj_last_status(void) { return g_last_status; }

const char* proj_last_cuda_error(void) { return g_last_cuda; }

const char* proj_status_string(int status) {
  switch (status) {
    case PROJ_OK: return "ok";
    case PROJ_EINVAL: return "invalid argument";
    case PROJ_EUNSUPPORTED: return "unsupported request";
    case PROJ_EALIGN: return "pointer not 16-byte aligned";
    case PROJ_ENOMEM: return "out of memory";
    case PROJ_ECUDA: return "CUDA error";
    case PROJ_EDEVICE: return "device-side fault reported";
  }
  return "unknown status";
}

int proj_num_sms(void) {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

proj_handle proj_prepare_ex(int layer, const void* W, int64_t N, int64_t K, int dtype,
                            uint32_t flags, int64_t m_max, int* status) {
  auto bail = [&](int st) -> proj_handle {
    fail(st);
    if (status) *status = st;
    return nullptr;
  };
  if (layer < 0 || layer > 4) return bail(PROJ_EINVAL);
  const LayerShape& ls = kLayers[layer];
  if (N != ls.N || K != ls.K || dtype != ls.dtype) return bail(PROJ_EINVAL);
  if (!W) return bail(PROJ_EINVAL);
  if (!aligned16(W)) return bail(PROJ_EALIGN);
  if (flags & ~static_cast<uint32_t>(PROJ_ENCODE_EXPWIN12)) return bail(PROJ_EINVAL);
  if (m_max < 0) return bail(PROJ_EINVAL);
  if (m_max == 0) m_max = kDefaultMMax;

  proj_ctx* h = new (std::nothrow) proj_ctx();
  if (!h) return bail(PROJ_ENOMEM);
  h->layer = layer;
  h->dtype = dtype;
  h->N = N;
  h->K = K;
  h->m_max = m_max;
  auto bail_cuda = [&](cudaError_t e, const char* what) -> proj_handle {
    fail_cuda(e, what);
    free_ctx(h);
    const int st = (e == cudaErrorMemoryAllocation) ? PROJ_ENOMEM : PROJ_ECUDA;
    g_last_status = st;
    if (status) *status = st;
    return nullptr;
  };
  cudaError_t e;
  if ((e = cudaGetDevice(&h->device)) != cudaSuccess) return bail_cuda(e, "cudaGetDevice");
  if ((e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device)) !=
      cudaSuccess)
    return bail_cuda(e, "cudaDeviceGetAttribute");
  if ((e = tc_init_attributes()) != cudaSuccess) return bail_cuda(e, "tc attributes");
  if ((e = router_cluster_init_attributes()) != cudaSuccess)
    return bail_cuda(e, "router attributes");
  if ((e = gemv_init_attributes()) != cudaSuccess) return bail_cuda(e, "gemv attributes");
  if ((e = gemv_reg_init_attributes()) != cudaSuccess) return bail_cuda(e, "gemv attributes");
  if ((e = gemv_mma_init_attributes()) != cudaSuccess) return bail_cuda(e, "gemv attributes");
  if ((e = gemv_rows_init_attributes()) != cudaSuccess) return bail_cuda(e, "gemv attributes");
  if ((e = router_gemv_init_attributes()) != cudaSuccess) return bail_cuda(e, "gemv attributes");
  if ((e = cluster_init_attributes()) != cudaSuccess) return bail_cuda(e, "cluster attributes");
  if ((e = pair_init_attributes()) != cudaSuccess) return bail_cuda(e, "pair attributes");
  for (int b = 0; b < 3; ++b)
    for (int kg = 1; kg <= kPairMaxKG; ++kg) h->pair_active[b][kg - 1] = pair_max_active(64 << b, kg);
  {
    const int bns[5] = {16, 32, 64, 128, 256};
    for (int b = 0; b < 5; ++b)
      for (int c = 0; c < kClusterMaxCS; ++c) {
        // The occupancy query counts one CTA per SM for a cluster launch;
        // the narrow-tile kernel holds two per SM (measured: 18 clusters of
        // 8 such CTAs run in one wave where the query says 15).
        h->cluster_active[b][c] = cluster_max_active(bns[b], c + 1) * cluster_blocks_per_sm(bns[b]);
        h->rcluster_active[b][c] = router_cluster_max_active(bns[b], c + 1);
      }
  }
  if (layer == PROJ_ROUTER && K % 1024 == 0 && K <= 8192)
    h->rgcc_active = router_gemv_cc_max_active(static_cast<int>(N), static_cast<int>(K));
  if (!encode_fn()) return bail_cuda(cudaErrorNotSupported, "cuTensorMapEncodeTiled");

  cudaStream_t s;
  if ((e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking)) != cudaSuccess)
    return bail_cuda(e, "cudaStreamCreate");
  auto done = [&]() { cudaStreamDestroy(s); };

  const int64_t sms = h->num_sms;
  if (layer == PROJ_ROUTER) {
    h->w_dense_bytes = static_cast<size_t>(N) * K * 4;
    if ((e = dmalloc(&h->w_dense, h->w_dense_bytes)) != cudaSuccess) {
      done();
      return bail_cuda(e, "cudaMalloc(weights)");
    }
    if ((e = pack_router_fma_tiles(static_cast<const float*>(W), static_cast<int>(N),
                                   static_cast<int>(K), h->w_dense, s)) != cudaSuccess) {
      done();
      return bail_cuda(e, "pack router");
    }
    if ((e = dmalloc(&h->w_planes, static_cast<size_t>(N) * K * 6)) != cudaSuccess) {
      done();
      return bail_cuda(e, "cudaMalloc(weight planes)");
    }
    if ((e = pack_router_planes(static_cast<const float*>(W), static_cast<int>(N),
                                static_cast<int>(K), h->w_planes, s)) != cudaSuccess) {
      done();
      return bail_cuda(e, "pack router planes");
    }
    h->ws_bytes = 16;  // sized below for the cluster groups
    h->counters_bytes = 16;
  } else {
    h->w_dense_bytes = static_cast<size_t>(N) * K * 2;
    if ((e = dmalloc(&h->w_dense, h->w_dense_bytes)) != cudaSuccess) {
      done();
      return bail_cuda(e, "cudaMalloc(weights)");
    }
    if ((e = pack_bf16_tiles(static_cast<const uint16_t*>(W), static_cast<int>(N),
                             static_cast<int>(K), h->w_dense, s)) != cudaSuccess) {
      done();
      return bail_cuda(e, "pack bf16");
    }
    h->wmap_ok = make_w_map(&h->tmap_w, h->w_dense, (N / kTileRows) * (K / kTileK));
    if (!h->wmap_ok) {
      done();
      return bail_cuda(cudaErrorInvalidValue, "cuTensorMapEncodeTiled(weights)");
    }
    if (N % 16 == 0 && K % 256 == 0 && K <= 8192) {
      if ((e = dmalloc(&h->w_frag, static_cast<size_t>(N) * K * 2)) != cudaSuccess ||
          (e = pack_frag16(static_cast<const uint16_t*>(W), static_cast<int>(N),
                           static_cast<int>(K), h->w_frag, s)) != cudaSuccess) {
        done();
        return bail_cuda(e, "pack fragment tiles");
      }
    }
    // The row-run layout of the few-token GEMV, for its default partition
    // (one CTA per SM); the unpooler also for its first 1024 rows.
    if (K % 32 == 0) {
      h->runs_G = static_cast<int>(std::min<int64_t>(N, h->num_sms));
      if ((N + h->runs_G - 1) / h->runs_G <= kGemvRowsMaxRows) {
        if ((e = dmalloc(&h->w_runs, static_cast<size_t>(N) * K * 2)) != cudaSuccess ||
            (e = pack_runs(static_cast<const uint16_t*>(W), static_cast<int>(N),
                           static_cast<int>(K), h->runs_G, h->w_runs, s)) != cudaSuccess) {
          done();
          return bail_cuda(e, "pack row runs");
        }
      }
      if (layer == PROJ_UNPOOLER) {
        h->runs_slice_rows = kUnpoolerSliceRows;
        h->runs_slice_G = static_cast<int>(std::min<int64_t>(kUnpoolerSliceRows, h->num_sms));
        if ((e = dmalloc(&h->w_runs_slice, static_cast<size_t>(kUnpoolerSliceRows) * K * 2)) !=
                cudaSuccess ||
            (e = pack_runs(static_cast<const uint16_t*>(W), static_cast<int>(kUnpoolerSliceRows),
                           static_cast<int>(K), h->runs_slice_G, h->w_runs_slice, s)) !=
                cudaSuccess) {
          done();
          return bail_cuda(e, "pack row runs");
        }
      }
    }
    if (flags & PROJ_ENCODE_EXPWIN12) {
      uint32_t* dev_hist = nullptr;
      uint32_t* dev_flag = nullptr;  // [0] overflow, [2..3] escape count (u64)
      if ((e = dmalloc(&dev_hist, 128 * 4)) != cudaSuccess ||
          (e = dmalloc(&dev_flag, 16)) != cudaSuccess) {
        cudaFree(dev_hist);
        done();
        return bail_cuda(e, "cudaMalloc(hist)");
      }
      uint32_t hist[128];
      uint32_t flag[4];
      const size_t rec_bytes =
          static_cast<size_t>(N / kTileRows) * (K / kTileK) * static_cast<size_t>(kRecBytes);
      bool ok = (e = cudaMemsetAsync(dev_hist, 0, 128 * 4, s)) == cudaSuccess &&
                (e = cudaMemsetAsync(dev_flag, 0, 16, s)) == cudaSuccess &&
                (e = high7_histogram(static_cast<const uint16_t*>(W), N * K, dev_hist, s)) ==
                    cudaSuccess &&
                (e = cudaMemcpyAsync(hist, dev_hist, sizeof hist, cudaMemcpyDeviceToHost, s)) ==
                    cudaSuccess &&
                (e = cudaStreamSynchronize(s)) == cudaSuccess;
      if (ok) {
        h->e0 = choose_window(hist);
        h->w_exp_bytes = rec_bytes;
        ok = (e = dmalloc(&h->w_exp, rec_bytes)) == cudaSuccess &&
             (e = cudaMemsetAsync(h->w_exp, 0, rec_bytes, s)) == cudaSuccess &&
             (e = encode_expwin12(static_cast<const uint16_t*>(W), static_cast<int>(N),
                                  static_cast<int>(K), h->e0, h->w_exp, dev_flag,
                                  reinterpret_cast<unsigned long long*>(dev_flag + 2), s)) ==
                 cudaSuccess &&
             (e = cudaMemcpyAsync(flag, dev_flag, sizeof flag, cudaMemcpyDeviceToHost, s)) ==
                 cudaSuccess &&
             (e = cudaStreamSynchronize(s)) == cudaSuccess;
      }
      cudaFree(dev_hist);
      cudaFree(dev_flag);
      if (!ok) {
        done();
        return bail_cuda(e, "12-bit encode");
      }
      uint64_t nesc;
      std::memcpy(&nesc, &flag[2], 8);
      h->n_esc = static_cast<int64_t>(nesc);
      if (flag[0]) {  // some tile has more escapes than its block holds
        cudaFree(h->w_exp);
        h->w_exp = nullptr;
        h->w_exp_bytes = 0;
        h->exp_declined = 1;
      }
      // The register GEMV's row-chunk records, same window.
      if (K % kRc12Chunk == 0 && K <= 8192) {
        const size_t chunks = static_cast<size_t>(N) * (K / kRc12Chunk);
        uint32_t* dev_over = nullptr;
        uint32_t over = 0;
        bool ok12 = (e = dmalloc(&dev_over, 4)) == cudaSuccess &&
                    (e = dmalloc(&h->w_rc12, chunks * kRc12Bytes)) == cudaSuccess &&
                    (e = dmalloc(&h->rc12_esc, chunks * kRc12EscWords * 4)) == cudaSuccess &&
                    (e = cudaMemsetAsync(dev_over, 0, 4, s)) == cudaSuccess &&
                    (e = cudaMemsetAsync(h->rc12_esc, 0, chunks * kRc12EscWords * 4, s)) ==
                        cudaSuccess &&
                    (e = encode_rc12(static_cast<const uint16_t*>(W), static_cast<int>(N),
                                     static_cast<int>(K), h->e0, h->w_rc12, h->rc12_esc, dev_over,
                                     s)) == cudaSuccess &&
                    (e = cudaMemcpyAsync(&over, dev_over, 4, cudaMemcpyDeviceToHost, s)) ==
                        cudaSuccess &&
                    (e = cudaStreamSynchronize(s)) == cudaSuccess;
        cudaFree(dev_over);
        if (!ok12) {
          done();
          return bail_cuda(e, "12-bit row-chunk encode");
        }
        if (over) {  // some chunk has more escapes than its block holds
          cudaFree(h->w_rc12);
          cudaFree(h->rc12_esc);
          h->w_rc12 = nullptr;
          h->rc12_esc = nullptr;
        }
      }
      // The warp-MMA GEMV's fragment-order copy, recoded the same way: its
      // stream of 16 x 16 tiles viewed as rows of 1024 elements (four tiles).
      if (h->w_frag) {
        const size_t chunks = static_cast<size_t>(N) * K / kRc12Chunk;
        uint32_t* dev_over = nullptr;
        uint32_t over = 0;
        bool okf = (e = dmalloc(&dev_over, 4)) == cudaSuccess &&
                   (e = dmalloc(&h->w_frag12, chunks * kRc12Bytes)) == cudaSuccess &&
                   (e = dmalloc(&h->frag12_esc, chunks * kRc12EscWords * 4)) == cudaSuccess &&
                   (e = cudaMemsetAsync(dev_over, 0, 4, s)) == cudaSuccess &&
                   (e = cudaMemsetAsync(h->frag12_esc, 0, chunks * kRc12EscWords * 4, s)) ==
                       cudaSuccess &&
                   (e = encode_rc12(reinterpret_cast<const uint16_t*>(h->w_frag),
                                    static_cast<int>(chunks), kRc12Chunk, h->e0, h->w_frag12,
                                    h->frag12_esc, dev_over, s)) == cudaSuccess &&
                   (e = cudaMemcpyAsync(&over, dev_over, 4, cudaMemcpyDeviceToHost, s)) ==
                       cudaSuccess &&
                   (e = cudaStreamSynchronize(s)) == cudaSuccess;
        cudaFree(dev_over);
        if (!okf) {
          done();
          return bail_cuda(e, "12-bit fragment encode");
        }
        if (over) {
          cudaFree(h->w_frag12);
          cudaFree(h->frag12_esc);
          h->w_frag12 = nullptr;
          h->frag12_esc = nullptr;
        }
      }
    }
    const int bn_max = bn_for_m(std::min<int64_t>(m_max, 256));
    h->ws_bytes = static_cast<size_t>(2 * sms) * bn_max * kTileRows * 4;
    const int64_t mt_max = (m_max + 255) / 256;
    h->counters_bytes = static_cast<size_t>(std::max<int64_t>(mt_max, 1) * (N / kTileRows)) * 4;
  }
  const size_t out_elem = (layer == PROJ_ROUTER) ? 4 : 2;
  const size_t w_bytes = static_cast<size_t>(N) * K * (layer == PROJ_ROUTER ? 4 : 2);
  if ((e = dmalloc(&h->w_rows, w_bytes)) != cudaSuccess ||
      (e = cudaMemcpyAsync(h->w_rows, W, w_bytes, cudaMemcpyDeviceToDevice, s)) != cudaSuccess ||
      (e = dmalloc(&h->gemv_flags, static_cast<size_t>(sms) * 4)) != cudaSuccess ||
      (e = cudaMemsetAsync(h->gemv_flags, 0, static_cast<size_t>(sms) * 4, s)) != cudaSuccess ||
      (e = dmalloc(&h->gemv_ws, static_cast<size_t>(sms) * 2 * 4)) != cudaSuccess) {
    done();
    return bail_cuda(e, "cudaMalloc(row-major weights)");
  }
  // cluster groups: one [256][128] fp32 partial per cluster, at most one per SM
  h->ws_bytes = std::max(h->ws_bytes, static_cast<size_t>(sms) * 256 * kTileRows * 4);
  const size_t cl_counter_bytes = static_cast<size_t>(sms) * kClusterMaxCS * 4;
  if ((e = dmalloc(&h->xch, static_cast<size_t>(sms) * 256 * kTileRows * 4)) != cudaSuccess ||
      (e = dmalloc(&h->cl_counters, cl_counter_bytes)) != cudaSuccess ||
      (e = cudaMemsetAsync(h->cl_counters, 0, cl_counter_bytes, s)) != cudaSuccess) {
    done();
    return bail_cuda(e, "cudaMalloc(cluster counters)");
  }
  if ((e = dmalloc(&h->ws, h->ws_bytes)) != cudaSuccess ||
      (e = dmalloc(&h->counters, h->counters_bytes)) != cudaSuccess ||
      (e = dmalloc(&h->status, 16)) != cudaSuccess ||
      (e = dmalloc(&h->x_stage, static_cast<size_t>(m_max) * K * 2)) != cudaSuccess ||
      (e = dmalloc(&h->out_stage, static_cast<size_t>(m_max) * N * out_elem)) != cudaSuccess) {
    done();
    return bail_cuda(e, "cudaMalloc(workspace)");
  }
  if ((e = cudaMemsetAsync(h->counters, 0, h->counters_bytes, s)) != cudaSuccess ||
      (e = cudaMemsetAsync(h->status, 0, 16, s)) != cudaSuccess ||
      (e = cudaStreamSynchronize(s)) != cudaSuccess) {
    done();
    return bail_cuda(e, "prepare sync");
  }
  done();
  if (status) *status = PROJ_OK;
  return h;
}

proj_handle proj_prepare(int layer, const void* W, int64_t N, int64_t K, int dtype) {
  return proj_prepare_ex(layer, W, N, K, dtype, 0u, 0, nullptr);
}

int64_t proj_out_features(proj_handle h, int64_t m) {
  if (!h) return -1;
  return out_rows(h, m);
}

int proj_run_ex(proj_handle h, const void* x, int64_t m, void* out, proj_stream stream,
                const proj_run_opts* opts) {
  if (!h) return fail(PROJ_EINVAL);
  if (m < 0) return fail(PROJ_EINVAL);
  if (m > h->m_max) return fail(PROJ_EUNSUPPORTED);
  if (m == 0) return PROJ_OK;
  if (!x || !out) return fail(PROJ_EINVAL);
  if (!aligned16(x) || !aligned16(out)) return fail(PROJ_EALIGN);
  Plan pl;
  int st = make_plan(h, m, opts, &pl);
  if (st != PROJ_OK) return fail(st);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (pl.gemv) {
    GemvParams g;
    g.w = pl.expwin ? static_cast<const void*>(h->w_rc12) : h->w_rows;
    g.esc = h->rc12_esc;
    g.e0x4 = static_cast<uint32_t>(h->e0) * 0x01010101u;
    g.x = x;
    g.out = out;
    g.ws = h->gemv_ws;
    g.flags = h->gemv_flags;
    g.status = h->status;
    g.m = static_cast<int>(m);
    g.n_rows = static_cast<int>(pl.n_out);
    g.K = static_cast<int>(h->K);
    g.G = pl.G;
    g.out_f32 = pl.router ? 1 : 0;
    e = pl.expwin     ? gemv_reg12_launch(pl.bn, g, s)
        : pl.gemv_reg ? gemv_reg_launch(pl.router, pl.bn, g, s)
                      : gemv_launch(pl.router, pl.bn, g, s);
    if (e != cudaSuccess) return fail_cuda(e, "kernel launch");
    return PROJ_OK;
  }
  if (pl.router_gemv || pl.router_gemv_cc) {
    RouterGemvParams r;
    r.w = h->w_rows;
    r.x = x;
    r.out = out;
    r.status = h->status;
    r.m = static_cast<int>(m);
    r.N = static_cast<int>(pl.n_out);
    r.K = static_cast<int>(h->K);
    r.G = pl.G;
    e = pl.router_gemv_cc ? router_gemv_cc_launch(r, s) : router_gemv_launch(r, s);
    if (e != cudaSuccess) return fail_cuda(e, "kernel launch");
    return PROJ_OK;
  }
  if (pl.gemv_rows) {
    const int nt = pl.bn, ks = pl.bpw, nr_hi = pl.T;
    // Each map is copied out at once: a later insertion into the cache may
    // reuse the slot a hit pointed to.
    CUtensorMap tw_hi, tw_lo;
    const CUtensorMap* mp = get_rows_map(h, h->w_rows, h->N, nr_hi, ks);
    if (!mp) return fail_cuda(cudaErrorInvalidValue, "cuTensorMapEncodeTiled(rows)");
    tw_hi = *mp;
    mp = nr_hi > 1 ? get_rows_map(h, h->w_rows, h->N, nr_hi - 1, ks) : &tw_hi;
    if (!mp) return fail_cuda(cudaErrorInvalidValue, "cuTensorMapEncodeTiled(rows)");
    tw_lo = *mp;

    GemvRowsParams g;
    g.w_runs = nullptr;
    if (pl.n_out == h->N && h->w_runs && pl.G == h->runs_G) g.w_runs = h->w_runs;
    if (pl.n_out != h->N && h->w_runs_slice && pl.n_out == h->runs_slice_rows &&
        pl.G == h->runs_slice_G)
      g.w_runs = h->w_runs_slice;
    g.x = static_cast<const uint16_t*>(x);
    g.out = out;
    g.status = h->status;
    g.stamps = opts ? static_cast<uint64_t*>(opts->stamps) : nullptr;
    g.m = static_cast<int>(m);
    g.n_rows = static_cast<int>(pl.n_out);
    g.K = static_cast<int>(h->K);
    g.G = pl.G;
    g.KS = ks;
    g.S = pl.KG;
    g.nr_hi = nr_hi;
    e = gemv_rows_launch(nt, pl.MT, tw_hi, tw_lo, g, s);
    if (e != cudaSuccess) return fail_cuda(e, "kernel launch");
    return PROJ_OK;
  }
  if (pl.gemv_mma) {
    GemvMmaParams g;
    g.w = reinterpret_cast<const uint4*>(h->w_frag);
    g.rec = h->w_frag12;
    g.esc = h->frag12_esc;
    g.e0x4 = static_cast<uint32_t>(h->e0) * 0x01010101u;
    g.x = x;
    g.out = out;
    g.status = h->status;
    g.m = static_cast<int>(m);
    g.n_rows = static_cast<int>(pl.n_out);
    g.K = static_cast<int>(h->K);
    g.G = pl.G;
    e = gemv_mma_launch(pl.bn, pl.expwin, g, s);
    if (e != cudaSuccess) return fail_cuda(e, "kernel launch");
    return PROJ_OK;
  }
  if (pl.pair) {
    const CUtensorMap* xmap = get_map(h, x, m, pl.bn / 2, true);
    if (!xmap) return fail_cuda(cudaErrorInvalidValue, "cuTensorMapEncodeTiled(x)");
    PairParams q;
    q.out = out;
    q.status = h->status;
    q.xch = h->xch;
    q.m = static_cast<int>(m);
    q.n_out = static_cast<int>(pl.n_out);
    q.KB = pl.KB;
    q.KBx = static_cast<int>(h->K / kTileK);
    q.MT = pl.MT;
    q.KG = pl.KG;
    q.out_f32 = 0;
    q.w_evict_first = pl.MT == 1 ? 1 : 0;
    q.stamps = opts ? static_cast<uint64_t*>(opts->stamps) : nullptr;
    // the exchange slots hold one [256][128] fp32 partial per SM
    if (pl.KG > 1 && pl.G > h->num_sms) return fail(PROJ_EUNSUPPORTED);
    e = pair_launch(pl.bn, h->tmap_w, *xmap, q, pl.T / 2, s);
    if (e != cudaSuccess) return fail_cuda(e, "kernel launch");
    return PROJ_OK;
  }
  const CUtensorMap* map = get_map(h, x, m, pl.bn, true);
  if (!map) return fail_cuda(cudaErrorInvalidValue, "cuTensorMapEncodeTiled(x)");
  if (pl.cluster) {
    ClusterParams c;
    c.w = pl.planes ? h->w_planes : h->w_dense;
    c.KBx = static_cast<int>(h->K / kTileK);
    c.out_f32 = pl.router ? 1 : 0;
    c.out = out;
    c.status = h->status;
    c.m = static_cast<int>(m);
    c.n_out = static_cast<int>(pl.n_out);
    c.T = pl.T;
    c.KB = pl.KB;
    c.MT = pl.MT;
    c.CS = pl.G;
    c.KG = pl.KG;
    c.ws = reinterpret_cast<float*>(h->ws);
    c.counters = h->cl_counters;
    c.stamps = (opts && !(pl.router && !pl.planes)) ? static_cast<uint64_t*>(opts->stamps) : nullptr;
    // The cluster kernels exchange their partials through L2 when three or
    // more CTAs share a tile and every CTA has a slot (one wave: at most one
    // CTA per SM); otherwise through distributed shared memory (~33 GB/s per
    // SM on GB300; at two CTAs per tile the remote half is small and the L2
    // round trip measured no faster).
    const int64_t ctas = static_cast<int64_t>(pl.MT) * pl.T * pl.KG * pl.G;
    c.xch = (pl.G >= 3 && ctas <= h->num_sms) ? h->xch : nullptr;
    e = (pl.router && !pl.planes) ? router_cluster_launch(pl.bn, *map, c, s)
                                   : cluster_launch(pl.bn, *map, c, s);
    if (e != cudaSuccess) return fail_cuda(e, "kernel launch");
    return PROJ_OK;
  }
  {
    TcParams p;
    p.w = pl.expwin ? h->w_exp : h->w_dense;
    p.out = out;
    p.ws = h->ws;
    p.counters = h->counters;
    p.status = h->status;
    p.m = static_cast<int>(m);
    p.n_out = static_cast<int>(pl.n_out);
    p.K = static_cast<int>(h->K);
    p.T = pl.T;
    p.KB = pl.KB;
    p.MT = pl.MT;
    p.G = pl.G;
    p.e0x4 = static_cast<uint32_t>(h->e0) * 0x01010101u;
    p.reduce = pl.reduce;
    e = tc_launch(pl.bn, pl.expwin, *map, p, s);
  }
  if (e != cudaSuccess) return fail_cuda(e, "kernel launch");
  return PROJ_OK;
}

int proj_run(proj_handle h, const void* x, int64_t m, void* out, proj_stream stream) {
  return proj_run_ex(h, x, m, out, stream, nullptr);
}

// The device address of page-locked host memory p if it is 16-byte aligned,
// else null (pageable or unknown memory: the caller copies with the copy
// engines).
static const void* device_mapping(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer) return nullptr;
  if (reinterpret_cast<uintptr_t>(a.devicePointer) % 16 != 0) return nullptr;
  return a.devicePointer;
}

int proj_run_host(proj_handle h, const void* x_host, int64_t m, void* out_host,
                  proj_stream stream) {
  if (!h) return fail(PROJ_EINVAL);
  if (m < 0) return fail(PROJ_EINVAL);
  if (m > h->m_max) return fail(PROJ_EUNSUPPORTED);
  if (m == 0) return PROJ_OK;
  if (!x_host || !out_host) return fail(PROJ_EINVAL);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t xb = static_cast<size_t>(m) * h->K * 2;
  const size_t ob = static_cast<size_t>(m) * out_rows(h, m) * (h->layer == PROJ_ROUTER ? 4 : 2);
  // Page-locked host buffers are mapped into the device's address space: a
  // copy kernel moves x in through that mapping (a few microseconds less per
  // transfer than a copy-engine transfer of these sizes), and the projection
  // kernel stores its result straight into the mapped output (no staging and
  // no copy-out launch: measured 7-18 us less per five-layer load end to end,
  // decode-1 50.6 -> 42.1 us); anything else goes through cudaMemcpyAsync.
  const void* x_map = device_mapping(x_host);
  void* out_map = const_cast<void*>(device_mapping(out_host));
  cudaError_t e;
  if (x_map && xb % 16 == 0)
    e = copy16_launch(h->x_stage, x_map, static_cast<int64_t>(xb), h->num_sms, s);
  else
    e = cudaMemcpyAsync(h->x_stage, x_host, xb, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return fail_cuda(e, "copy x to device");
  const bool direct = out_map && ob % 16 == 0;
  int st = proj_run_ex(h, h->x_stage, m, direct ? out_map : h->out_stage, stream, nullptr);
  if (st != PROJ_OK || direct) return st;
  e = cudaMemcpyAsync(out_host, h->out_stage, ob, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return fail_cuda(e, "copy out to host");
  return PROJ_OK;
}

int proj_info(proj_handle h, proj_info_t* info) {
  if (!h || !info) return fail(PROJ_EINVAL);
  std::memset(info, 0, sizeof *info);
  info->layer = h->layer;
  info->dtype = h->dtype;
  info->N = h->N;
  info->K = h->K;
  info->m_max = h->m_max;
  info->expwin12 = h->w_exp ? 1 : 0;
  info->expwin12_declined = h->exp_declined;
  info->expwin12_e0 = h->e0;
  info->expwin12_escapes = h->n_esc;
  info->expwin12_bytes = h->w_exp ? (h->N * h->K * 3) / 2 + h->n_esc * 4 : 0;
  info->dense_bytes = static_cast<int64_t>(h->w_dense_bytes);
  info->workspace_bytes = static_cast<int64_t>(h->ws_bytes + h->counters_bytes);
  info->num_sms = h->num_sms;
  return PROJ_OK;
}

int proj_describe(proj_handle h, int64_t m, char* buf, size_t cap) {
  return proj_describe_ex(h, m, nullptr, buf, cap);
}

int proj_describe_ex(proj_handle h, int64_t m, const proj_run_opts* opts, char* buf, size_t cap) {
  if (!h || !buf || cap == 0 || m < 1) return fail(PROJ_EINVAL);
  Plan pl;
  int st = make_plan(h, m, opts, &pl);
  if (st != PROJ_OK) return fail(st);
  if (pl.gemv) {
    std::snprintf(buf, cap, "gemv%s_%s MT=%d G=%d n_rows=%lld", pl.gemv_reg ? "_reg" : "",
                  pl.router ? "f32w" : (pl.expwin ? "expwin12rc" : "bf16w"), pl.bn, pl.G,
                  static_cast<long long>(pl.n_out));
  } else if (pl.router_gemv) {
    std::snprintf(buf, cap, "router_gemv_f32w passes_of_8 G=%d n_rows=%lld", pl.G,
                  static_cast<long long>(pl.n_out));
  } else if (pl.router_gemv_cc) {
    std::snprintf(buf, cap, "router_gemv_splitk_f32w CS=%d clusters=%lld n_rows=%lld", pl.G,
                  static_cast<long long>((pl.n_out + 7) / 8), static_cast<long long>(pl.n_out));
  } else if (pl.gemv_rows) {
    std::snprintf(buf, cap,
                  "gemv_rows_mma tokens<=%d steps_per_stage=%d steps_per_warp=%d stages=%d G=%d "
                  "rows_per_cta<=%d n_rows=%lld %s",
                  8 * pl.bn, pl.bpw, pl.MT, pl.KG, pl.G, pl.T, static_cast<long long>(pl.n_out),
                  (pl.n_out == h->N ? (h->w_runs && pl.G == h->runs_G)
                                    : (h->w_runs_slice && pl.G == h->runs_slice_G))
                      ? "packed_runs" : "row_major_tma");
  } else if (pl.gemv_mma) {
    std::snprintf(buf, cap, "gemv_mma16x8%s tokens<=%d G=%d blocks_per_cta<=%lld n_rows=%lld",
                  pl.expwin ? "_expwin12rc" : "", 8 * pl.bn, pl.G,
                  static_cast<long long>((pl.n_out / 16 + pl.G - 1) / pl.G),
                  static_cast<long long>(pl.n_out));
  } else if (pl.pair) {
    std::snprintf(buf, cap,
                  "tc_pair BN=%d stages=%d KG=%d cluster=%d CTAs=%d pair_tiles=%d KB=%d MT=%d "
                  "n_out=%lld resident_clusters=%d",
                  pl.bn, pair_stages(pl.bn), pl.KG, 2 * pl.KG, pl.G, pl.T / 2, pl.KB, pl.MT,
                  static_cast<long long>(pl.n_out),
                  h->pair_active[pair_bn_index(pl.bn)][pl.KG - 1]);
  } else if (pl.cluster) {
    const bool fma = pl.router && !pl.planes;
    std::snprintf(buf, cap,
                  "%s BN=%d stages=%d CS=%d KG=%d CTAs=%d T=%d KB=%d MT=%d "
                  "n_out=%lld resident_clusters=%d",
                  fma ? "fma_cluster" : (pl.planes ? "tc_cluster_planes3" : "tc_cluster"), pl.bn,
                  fma ? router_cluster_stages(pl.bn) : cluster_stages(pl.bn), pl.G, pl.KG,
                  pl.MT * pl.T * pl.KG * pl.G, pl.T, pl.KB, pl.MT,
                  static_cast<long long>(pl.n_out),
                  (fma ? h->rcluster_active : h->cluster_active)[bn_index(pl.bn)][pl.G - 1]);
  } else {
    std::snprintf(buf, cap, "tc_%s BN=%d stages=%d G=%d T=%d KB=%d MT=%d n_out=%lld reduce=%s",
                  pl.expwin ? "expwin12" : "dense", pl.bn, tc_stages(pl.bn, pl.expwin), pl.G,
                  pl.T, pl.KB, pl.MT, static_cast<long long>(pl.n_out),
                  pl.reduce ? "distributed" : "owner");
  }
  return PROJ_OK;
}

int proj_unpack_weights(proj_handle h, int variant, void* W_out, proj_stream stream) {
  if (!h || !W_out) return fail(PROJ_EINVAL);
  if (!aligned16(W_out)) return fail(PROJ_EALIGN);
  if ((variant < PROJ_VARIANT_AUTO || variant > PROJ_VARIANT_PLANES3) &&
      variant != PROJ_UNPACK_FRAG16 && variant != PROJ_UNPACK_RC12 &&
      variant != PROJ_UNPACK_FRAG12 && variant != PROJ_UNPACK_RUNS &&
      variant != PROJ_UNPACK_RUNS_SLICE)
    return fail(PROJ_EINVAL);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (h->layer == PROJ_ROUTER) {
    if (variant == PROJ_VARIANT_EXPWIN12 || variant == PROJ_UNPACK_FRAG16 ||
        variant == PROJ_UNPACK_RC12 || variant == PROJ_UNPACK_FRAG12 ||
        variant == PROJ_UNPACK_RUNS || variant == PROJ_UNPACK_RUNS_SLICE)
      return fail(PROJ_EUNSUPPORTED);
    if (variant == PROJ_VARIANT_PLANES3)
      e = unpack_router_planes(h->w_planes, static_cast<int>(h->N), static_cast<int>(h->K),
                               static_cast<float*>(W_out), s);
    else
      e = unpack_router_fma_tiles(h->w_dense, static_cast<int>(h->N), static_cast<int>(h->K),
                                  static_cast<float*>(W_out), s);
  } else if (variant == PROJ_VARIANT_PLANES3) {
    return fail(PROJ_EUNSUPPORTED);
  } else if (variant == PROJ_UNPACK_FRAG12) {
    // records -> the fragment stream (a temporary) -> row-major
    if (!h->w_frag12) return fail(PROJ_EUNSUPPORTED);
    uint16_t* tmp = nullptr;
    const size_t nk = static_cast<size_t>(h->N) * h->K;
    if ((e = dmalloc(&tmp, nk * 2)) != cudaSuccess) return fail_cuda(e, "unpack temporary");
    if ((e = decode_rc12(h->w_frag12, h->frag12_esc, static_cast<int>(nk / kRc12Chunk), kRc12Chunk,
                         h->e0, tmp, s)) == cudaSuccess &&
        (e = unpack_frag16(reinterpret_cast<const uint32_t*>(tmp), static_cast<int>(h->N),
                           static_cast<int>(h->K), static_cast<uint16_t*>(W_out), s)) ==
            cudaSuccess)
      e = cudaStreamSynchronize(s);
    cudaFree(tmp);
  } else if (variant == PROJ_UNPACK_RC12) {
    if (!h->w_rc12) return fail(PROJ_EUNSUPPORTED);
    e = decode_rc12(h->w_rc12, h->rc12_esc, static_cast<int>(h->N), static_cast<int>(h->K), h->e0,
                    static_cast<uint16_t*>(W_out), s);
  } else if (variant == PROJ_UNPACK_RUNS) {
    if (!h->w_runs) return fail(PROJ_EUNSUPPORTED);
    e = unpack_runs(h->w_runs, static_cast<int>(h->N), static_cast<int>(h->K), h->runs_G,
                    static_cast<uint16_t*>(W_out), s);
  } else if (variant == PROJ_UNPACK_RUNS_SLICE) {
    if (!h->w_runs_slice) return fail(PROJ_EUNSUPPORTED);
    e = unpack_runs(h->w_runs_slice, static_cast<int>(h->runs_slice_rows), static_cast<int>(h->K),
                    h->runs_slice_G, static_cast<uint16_t*>(W_out), s);
  } else if (variant == PROJ_UNPACK_FRAG16) {
    if (!h->w_frag) return fail(PROJ_EUNSUPPORTED);
    e = unpack_frag16(h->w_frag, static_cast<int>(h->N), static_cast<int>(h->K),
                      static_cast<uint16_t*>(W_out), s);
  } else if (variant == PROJ_VARIANT_EXPWIN12 ||
             (variant == PROJ_VARIANT_AUTO && h->w_exp != nullptr)) {
    if (!h->w_exp) return fail(PROJ_EUNSUPPORTED);
    e = decode_expwin12(h->w_exp, static_cast<int>(h->N), static_cast<int>(h->K), h->e0,
                        static_cast<uint16_t*>(W_out), s);
  } else {
    e = unpack_bf16_tiles(h->w_dense, static_cast<int>(h->N), static_cast<int>(h->K),
                          static_cast<uint16_t*>(W_out), s);
  }
  if (e != cudaSuccess) return fail_cuda(e, "unpack");
  return PROJ_OK;
}

int proj_device_status(proj_handle h, proj_stream stream, uint32_t* code) {
  if (!h) return fail(PROJ_EINVAL);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  cudaError_t e;
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return fail_cuda(e, "sync");
  if ((e = cudaMemcpy(&word, h->status, 4, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return fail_cuda(e, "read status");
  if ((e = cudaMemset(h->status, 0, 4)) != cudaSuccess) return fail_cuda(e, "clear status");
  if (code) *code = word;
  return word ? fail(PROJ_EDEVICE) : PROJ_OK;
}

void proj_destroy(proj_handle h) {
  if (!h) return;
  cudaDeviceSynchronize();
  free_ctx(h);
}

int proj_read_floor(const void* buf, int64_t bytes, void* sink, int grid, int mode,
                    proj_stream stream) {
  if (!buf || !sink || bytes <= 0 || (bytes % 16) != 0 || grid < 0 || (mode & ~5) != 0)
    return fail(PROJ_EINVAL);
  if (!aligned16(buf) || (reinterpret_cast<uintptr_t>(sink) & 3u)) return fail(PROJ_EALIGN);
  if (grid == 0) {
    const int sms = proj_num_sms();
    if (sms <= 0) return fail_cuda(cudaErrorNoDevice, "proj_num_sms");
    grid = ((mode & 1) == 0) ? 2 * sms : sms;
  }
  cudaError_t e = read_floor_launch(buf, bytes, static_cast<uint32_t*>(sink), grid, mode,
                                    reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "read floor launch");
  return PROJ_OK;
}

int proj_fma_peak(void* sink, int iters, int grid, proj_stream stream, double* flops) {
  if (!sink || iters < 1 || iters > (1 << 24) || grid < 0) return fail(PROJ_EINVAL);
  if (reinterpret_cast<uintptr_t>(sink) & 3u) return fail(PROJ_EALIGN);
  if (grid == 0) {
    const int sms = proj_num_sms();
    if (sms <= 0) return fail_cuda(cudaErrorNoDevice, "proj_num_sms");
    grid = 8 * sms;
  }
  cudaError_t e = fma_peak_launch(static_cast<uint32_t*>(sink), iters, grid,
                                  reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "fma peak launch");
  if (flops) *flops = fma_peak_flops(grid, iters);
  return PROJ_OK;
}

}  // extern "C"
