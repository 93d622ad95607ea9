// kernels.h -- host-side interface between the C ABI (api.cu) and the kernel
// translation units.  Internal to libproj.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace proj {

// ----------------------------------------------------------------------------
// Packed bf16 weights for the tensor-core path.
//
// W [N, K] row-major is cut into tiles of 128 rows x 64 columns.  Tile (t, kb)
// covers rows [128 t, 128 t + 128) and columns [64 kb, 64 kb + 64) and is
// stored contiguously at byte offset (t * KB + kb) * 16384, already in the
// shared-memory image the MMA reads: row r at byte r * 128, its 16-byte chunk
// c (columns 8c .. 8c + 7) at chunk position c ^ (r & 7) -- the 128-byte
// swizzle.  One bulk copy per tile lands it ready for tcgen05.mma.
// ----------------------------------------------------------------------------
constexpr int kTileRows = 128;
constexpr int kTileK = 64;
constexpr int kTileBytes = kTileRows * kTileK * 2;  // 16384

// 12-bit exponent-window record of one tile (same tiling):
//   [0, 8192)      low bytes, chunk-major: chunk (r, c) at (8 r + c) * 8,
//                  bytes in column order;
//   [8192, 12288)  nibbles, chunk (r, c) at 8192 + (8 r + c) * 4: byte b of the
//                  32-bit word holds the nibble of column 8c + b in bits 0-3 and
//                  that of column 8c + 4 + b in bits 4-7; nibble = sign << 3 |
//                  code, high byte = sign << 7 | (e0 + code);
//   [12288, 12352) escape block: word 0 = count (<= kEscCap), then count
//                  words (position << 8 | original high byte), position =
//                  64 r + column within the tile.
constexpr int kRecBytes = 12352;
constexpr int kRecLowOff = 0;
constexpr int kRecNibOff = 8192;
constexpr int kRecEscOff = 12288;
constexpr int kEscCap = 15;

// 12-bit row-chunk records for the register GEMV (m <= 2), same nibble and
// escape conventions: W [N, K] row-major cut into 1024-column chunks, chunk
// q = n K / 1024 + c covering W[n, 1024 c .. 1024 c + 1023], record q at
// q x 1536 bytes.  Lane l of the warp that reads a chunk holds its groups
// j = 0..3, group j being columns 1024 c + 8 (l + 32 j) .. + 7:
//   [0, 1024)     low bytes: the 16 bytes at 16 (l + 32 i), i = 0, 1, hold
//                 groups 2i and 2i + 1 of lane l (8 bytes each, column order);
//   [1024, 1536)  nibbles: the 16 bytes at 1024 + 16 l, word j for group j,
//                 byte b holding the nibble of the group's column b in bits
//                 0-3 and that of column b + 4 in bits 4-7.
// Escapes sit in a separate array, 8 words per chunk at q x 32 bytes: word 0
// = count (<= kRc12EscCap), then (position << 8 | original high byte), the
// position being the column within the chunk, in increasing order.
constexpr int kRc12Chunk = 1024;
constexpr int kRc12Bytes = 1536;
constexpr int kRc12EscWords = 8;
constexpr int kRc12EscCap = kRc12EscWords - 1;

// Router (fp32) tiles for the FMA kernel: 128 rows x 64 columns, 32768
// bytes, tile (t, kb) at (t * K / 64 + kb) * 32768; row r at r * 256, its
// 16-byte chunk c (columns 4c .. 4c+3) at slot c ^ (r & 15).
constexpr int kRfRows = 128;
constexpr int kRfK = 64;
constexpr int kRfBytes = kRfRows * kRfK * 4;

struct TcParams {
  const uint8_t* w;     // packed tiles or 12-bit records
  void* out;            // bf16 [m, n_out]
  float* ws;            // split-K partials: [2 G][BN][128] fp32 (slot stride BN * 128)
  uint32_t* counters;   // [MT * T], zero between calls
  uint32_t* status;     // device status word
  int m;
  int n_out;            // rows of W computed (multiple of 128)
  int K;
  int T;                // n_out / 128
  int KB;               // K / 64
  int MT;               // ceil(m / BN)
  int G;                // CTAs (the split-K partition)
  uint32_t e0x4;        // 12-bit window base replicated into 4 bytes
  int reduce;           // split-K combine: 0 = owner, 1 = distributed
};


// Streaming GEMV (m <= 2): W row-major, bf16 or fp32; MT in {1, 2}.
struct GemvParams {
  const void* w;        // row-major [n_rows (+ more), K]
  const void* x;        // bf16 [m, K]
  void* out;            // [m, n_rows], bf16 or fp32
  float* ws;            // [G][MT] partial rows
  uint32_t* flags;      // [G], zero between calls
  uint32_t* status;
  int m;
  int n_rows;           // rows computed
  int K;                // multiple of 1024, <= 8192
  int G;                // CTAs, <= n_rows
  int out_f32;
  const uint32_t* esc;  // 12-bit register form: escape blocks of the records in w
  uint32_t e0x4;        // 12-bit register form: window base replicated into 4 bytes
};
cudaError_t gemv_init_attributes();
// Register-streaming GEMV (m <= 2), same parameters (ws and flags unused);
// CTA c computes rows [c n_rows / G, (c + 1) n_rows / G) and keeps at most
// kGemvRegMaxChunks chunk partials (its rows x K / 1024).
constexpr int kGemvRegMaxChunks = 2048;
cudaError_t gemv_reg_init_attributes();
cudaError_t gemv_reg_launch(bool f32w, int MT, const GemvParams& p, cudaStream_t s);
// The same form on 12-bit row-chunk records (bf16 weights, bf16 output).
cudaError_t gemv_reg12_launch(int MT, const GemvParams& p, cudaStream_t s);
// Record a failing status (and its text) for proj_last_status /
// proj_last_cuda_error; both return the status.
int record_status(int status, const char* text);
int record_cuda(cudaError_t e, const char* what);
cudaError_t gemv_launch(bool f32w, int MT, const GemvParams& p, cudaStream_t s);

// Tensor-core path: BN in {16, 32, 64, 128, 256}; expwin12 for BN in {16, 32, 64, 128}.
bool tc_supported(int BN, bool expwin);
int tc_threads(bool expwin);
size_t tc_smem_bytes(int BN, bool expwin);
int tc_stages(int BN, bool expwin);
cudaError_t tc_init_attributes();
cudaError_t tc_launch(int BN, bool expwin, const CUtensorMap& tmap_x, const TcParams& p,
                      cudaStream_t s);

// Cluster split-K tensor-core path: BN in {16, 32, 64, 128, 256}, cluster
// size 1..16.  Weight k-block kb multiplies x k-block kb % KBx, so the
// router's three bf16 planes (KB = 3 KBx) run as one bf16 GEMM.
struct ClusterParams {
  const uint8_t* w;     // packed bf16 tiles (same layout as TcParams::w), KB per tile row
  void* out;            // [m, n_out], bf16 or fp32 (out_f32)
  uint32_t* status;
  int m;
  int n_out;
  int T;                // n_out / 128
  int KB;               // weight k-blocks per tile row
  int KBx;              // x k-blocks (K / 64)
  int MT;               // ceil(m / BN)
  int CS;               // cluster size
  int KG;               // clusters per output tile (K split = KG x CS)
  int out_f32;
  float* ws;            // KG > 1: [T MT][KG][BN][128] fp32 cluster partials
  uint32_t* counters;   // KG > 1: [T MT][CS], zero between calls
  float* xch;           // CS > 1 and every CTA resident: [CTA][BN][128] fp32, the
                        // partials' exchange through L2; null: through distributed
                        // shared memory
  uint64_t* stamps;     // optional: [CTA][8] %globaltimer phase stamps (kStamp*), or null
};
// Phase stamps of the tensor-core kernels (per CTA, 8 slots).
enum : int {
  kStampEntry = 0,      // kernel entry
  kStampDepWait = 1,    // the producer passed the wait on the previous kernel
  kStampFirstFull = 2,  // the MMA issuer saw the first stage land
  kStampLastMma = 3,    // the MMA issuer committed the last stage
  kStampAccReady = 4,   // the drain saw the accumulator complete
  kStampDrained = 5,    // the accumulator is staged (and exchange stores issued)
  kStampCombine = 6,    // past the cluster barrier before the combine
  kStampExit = 7,       // after the combine's last store
};
constexpr int kClusterMaxCS = 16;      // CTAs per cluster, at most
constexpr int kClusterMaxGroups = 16;  // clusters per output tile, at most
bool cluster_supported(int BN);
cudaError_t cluster_init_attributes();
int cluster_max_active(int BN, int cs);
int cluster_blocks_per_sm(int BN);  // CTAs one SM holds (2 for the narrow tiles)
int cluster_stages(int BN);
cudaError_t cluster_launch(int BN, const CUtensorMap& tmap_x, const ClusterParams& p,
                           cudaStream_t s);

// CTA-pair tensor-core path (tcgen05 cta_group::2): BN in {64, 128, 256}.
// A pair tile is 256 weight rows (packed tiles 2 tp and 2 tp + 1) x BN
// tokens; the two CTAs of a pair each hold one 128-row tile and half of the
// tokens' x.  KG pairs split a pair tile's K and form one cluster of 2 KG
// CTAs; their fp32 partials meet in L2 (exchange slots) behind a cluster
// barrier, and each CTA sums 1/KG of the tokens in split order.
struct PairParams {
  void* out;            // [m, n_out], bf16 or fp32 (out_f32)
  uint32_t* status;
  float* xch;           // KG > 1: [CTA][BN][128] fp32 exchange slots (grid <= SMs)
  int m;
  int n_out;
  int KB;               // weight k-blocks per tile row
  int KBx;              // x k-blocks (K / 64); weight k-block kb meets x k-block kb % KBx
  int MT;               // token tiles: ceil(m / BN)
  int KG;               // pairs per pair tile (K split), 1..kPairMaxKG
  int out_f32;
  int w_evict_first;    // the weights are read once (MT == 1): evict them first from L2
  uint64_t* stamps;     // optional: [CTA][8] %globaltimer phase stamps (kStamp*), or null
};
constexpr int kPairMaxKG = 8;  // clusters of at most 16 CTAs
constexpr int kPairThreads = 256;
bool pair_supported(int BN);
cudaError_t pair_init_attributes();
int pair_max_active(int BN, int kg);  // co-resident clusters of 2 kg CTAs (occupancy query)
int pair_stages(int BN);
// tmap_w: the packed weight tiles viewed as a [tiles x 128 rows][64] bf16
// matrix (box 64 x 128, no swizzle: each tile is already the shared-memory
// image); tmap_x: x [m, K] bf16, box 64 x BN / 2, 128-byte swizzle.
cudaError_t pair_launch(int BN, const CUtensorMap& tmap_w, const CUtensorMap& tmap_x,
                        const PairParams& p, int pair_tiles, cudaStream_t s);

// FP32-FMA router on the cluster split-K skeleton: BN in {16, 32, 64}.
// The router at a few tokens: whole rows per CTA, fp32 weights straight to
// registers, x in passes of eight tokens (router_gemv.cu).
struct RouterGemvParams {
  const void* w;    // fp32 row-major [N, K]
  const void* x;    // bf16 [m, K]
  void* out;        // fp32 [m, N]
  uint32_t* status;
  int m;            // <= kRouterGemvMaxM
  int N;
  int K;            // multiple of 1024, <= 8192
  int G;            // CTAs: CTA c computes rows [c N / G, (c + 1) N / G), at most 16 chunks
};
constexpr int kRouterGemvMaxM = 16;
cudaError_t router_gemv_init_attributes();
cudaError_t router_gemv_launch(const RouterGemvParams& p, cudaStream_t s);
// The router GEMV with K split across a cluster (router_gemv.cu): cluster
// size K / 1024 (<= 8), rank q takes columns [1024 q, 1024 q + 1024) of 8
// rows (one per warp); ceil(N / 8) clusters; G unused.  m <= 32.
constexpr int kRouterGemvCcMaxM = 32;
cudaError_t router_gemv_cc_launch(const RouterGemvParams& p, cudaStream_t s);
int router_gemv_cc_max_active(int N, int K);  // co-resident clusters (occupancy query)
cudaError_t router_cluster_init_attributes();
int router_cluster_max_active(int BN, int cs);
int router_cluster_stages(int BN);
cudaError_t router_cluster_launch(int BN, const CUtensorMap& tmap_x, const ClusterParams& p,
                                  cudaStream_t s);

// Prepare-time kernels (prep.cu).
cudaError_t pack_bf16_tiles(const uint16_t* W, int N, int K, uint8_t* dst, cudaStream_t s);
cudaError_t unpack_bf16_tiles(const uint8_t* src, int N, int K, uint16_t* W, cudaStream_t s);
cudaError_t high7_histogram(const uint16_t* W, int64_t n, uint32_t* hist128, cudaStream_t s);
cudaError_t encode_expwin12(const uint16_t* W, int N, int K, int e0, uint8_t* dst,
                            uint32_t* overflow, unsigned long long* n_esc, cudaStream_t s);
cudaError_t decode_expwin12(const uint8_t* src, int N, int K, int e0, uint16_t* W,
                            cudaStream_t s);
// Row-chunk records (K % 1024 == 0); esc must be zeroed before the encode,
// *overflow is set when a chunk has more than kRc12EscCap escapes.
cudaError_t encode_rc12(const uint16_t* W, int N, int K, int e0, uint8_t* rec, uint32_t* esc,
                        uint32_t* overflow, cudaStream_t s);
cudaError_t decode_rc12(const uint8_t* rec, const uint32_t* esc, int N, int K, int e0,
                        uint16_t* W, cudaStream_t s);
// Few-token GEMV layout: bf16 W [N, K] as 16 x 16 tiles in the A-fragment
// order of mma.sync m16n8k16 (row-major A): tile (rb, kb) at
// (rb K/16 + kb) x 512 bytes, lane l's 16 bytes at l x 16 holding the pairs
// (row g, k c..c+1), (row g+8, k c..c+1), (row g, k c+8..c+9),
// (row g+8, k c+8..c+9) with g = l / 4, c = 2 (l % 4).  N % 16 == K % 16 == 0.
cudaError_t pack_frag16(const uint16_t* W, int N, int K, uint32_t* dst, cudaStream_t s);
cudaError_t unpack_frag16(const uint32_t* src, int N, int K, uint16_t* W, cudaStream_t s);
struct GemvMmaParams {
  const uint4* w;   // frag16 layout of the rows computed (and more)
  const uint8_t* rec;   // 12-bit form: the frag16 stream as row-chunk records (1024 elements each)
  const uint32_t* esc;  // 12-bit form: their escape blocks
  uint32_t e0x4;        // 12-bit form: window base replicated into 4 bytes
  const void* x;    // bf16 [m, K]
  void* out;        // bf16 [m, n_rows]
  uint32_t* status;
  int m;            // <= 8 x nt
  int n_rows;       // rows computed, multiple of 16
  int K;            // multiple of 256, <= 8192
  int G;            // CTAs: CTA c computes 16-row blocks [c NB / G, (c + 1) NB / G)
};
constexpr int kGemvMmaMaxM = 32;
constexpr int kGemvMmaMaxBlocks = 4;  // 16-row blocks per CTA, at most
int gemv_mma_smem(int nt, int K);   // dynamic shared memory at nt tiles of 8 tokens
bool gemv_mma_fits(int nt, int K);  // it fits one CTA's shared memory
cudaError_t gemv_mma_init_attributes();
cudaError_t gemv_mma_launch(int nt, bool x12, const GemvMmaParams& p, cudaStream_t s);
// Row-run warp-MMA GEMV (gemv_rows.cu): bf16 layers, m <= 8 NT (NT in
// {1, 2, 4} tiles of 8 tokens).  CTA c of G owns rows [c N / G, (c + 1) N / G)
// of W (nr_hi = ceil(N / G) rows or one fewer, at most kGemvRowsMaxRows);
// one thread streams them into a ring of S stages of KS 32-column steps:
// from the packed run layout with one bulk copy per stage, or -- for another
// grid -- through tw_hi / tw_lo, W viewed as (32 columns, N rows, K / 32
// steps) with boxes (32, nr_hi or nr_hi - 1, KS).  The 16 consumer warps
// take 16 / NB per 16-row block (NB = ceil(rows / 16)) and SPW = KS NB / 16
// steps of every stage each, loading their x fragments from global memory.
struct GemvRowsParams {
  const uint8_t* w_runs;  // the rows' run layout for this (n_rows, G) (pack_runs), or null:
                          // W through the tensor maps instead
  const uint16_t* x;    // bf16 [m, K]
  void* out;            // bf16 [m, n_rows]
  uint32_t* status;
  uint64_t* stamps;     // optional: [G][8] %globaltimer at entry (slot 0), after the
                        // dependency wait (1), after the main loop (5), at exit (7); null: none
  int m;
  int n_rows;
  int K;                // multiple of 32 KS
  int G;
  int KS;               // steps per stage
  int S;                // ring stages
  int nr_hi;            // ceil(n_rows / G)
};
constexpr int kGemvRowsMaxM = 32;
constexpr int kGemvRowsMaxRows = 64;     // rows per CTA: at most four 16-row blocks
constexpr int kGemvRowsConsumers = 16;   // consumer warps
constexpr int kGemvRowsRowPitch = 20;    // fp32 per staged tile row (bank-spread stores)
constexpr int kGemvRowsMaxStages = 16;
constexpr int kGemvRowsSmemMax = 227 * 1024;
// Consumer warps are dealt to 1, 2 or 4 block slots (the 16-row blocks of
// the longest run, rounded up to a power of two), 16 / slots per block.
__host__ __device__ inline int gemv_rows_block_slots(int nr_hi) {
  const int nb = (nr_hi + 15) >> 4;
  return nb <= 1 ? 1 : (nb <= 2 ? 2 : 4);
}
// Stages of x fragments a consumer warp keeps in flight (registers:
// D x SPW x NT x 4).
__host__ __device__ constexpr int gemv_rows_x_depth(int nt, int spw) {
  return (nt == 1 ? 8 : (nt == 2 ? 6 : 4)) / spw < 2 ? 2 : (nt == 1 ? 8 : (nt == 2 ? 6 : 4)) / spw;
}
// A stage: KS steps of the run's rows, [step][row][64 B], padded to 128 B.
__host__ __device__ inline uint32_t gemv_rows_stage_bytes(int ks, int nr_hi) {
  return (static_cast<uint32_t>(ks) * nr_hi * 64 + 127u) & ~127u;
}
// Byte offset of the barriers: after the ring, or after the accumulator
// staging that reuses it, whichever is longer.
__host__ __device__ inline uint32_t gemv_rows_bar_offset(int nt, int ks, int stages, int nr_hi) {
  const uint32_t ring = static_cast<uint32_t>(stages) * gemv_rows_stage_bytes(ks, nr_hi);
  const uint32_t red = static_cast<uint32_t>(kGemvRowsConsumers) * 8 * nt * kGemvRowsRowPitch * 4;
  return ((ring > red ? ring : red) + 7u) & ~7u;
}
size_t gemv_rows_smem(int nt, int ks, int stages, int nr_hi);
cudaError_t gemv_rows_init_attributes();
cudaError_t gemv_rows_launch(int nt, int spw, const CUtensorMap& tw_hi, const CUtensorMap& tw_lo,
                             const GemvRowsParams& p, cudaStream_t s);
// The row-run layout: rows [0, Nr) of a row-major bf16 [*, K] matrix for the
// partition over G CTAs; CTA c's run [c Nr / G, (c + 1) Nr / G) at byte
// offset (c Nr / G) K 2, laid out [K / 32 steps][run rows][32 columns].
cudaError_t pack_runs(const uint16_t* W, int Nr, int K, int G, uint8_t* dst, cudaStream_t s);
cudaError_t unpack_runs(const uint8_t* src, int Nr, int K, int G, uint16_t* W, cudaStream_t s);
cudaError_t pack_router_fma_tiles(const float* W, int N, int K, uint8_t* dst, cudaStream_t s);
cudaError_t unpack_router_fma_tiles(const uint8_t* src, int N, int K, float* W, cudaStream_t s);
// Router W -> bf16 planes hi, mid, lo (hi + mid + lo == W) packed as the bf16
// tiles of a [N, 3K] matrix: tile (t, p KB + kb) holds plane p.
cudaError_t pack_router_planes(const float* W, int N, int K, uint8_t* dst, cudaStream_t s);
cudaError_t unpack_router_planes(const uint8_t* src, int N, int K, float* W, cudaStream_t s);

// Streaming read (read.cu).
// FP32 FMA probe (read.cu): FLOPs of one launch, and the launch.
double fma_peak_flops(int grid, int iters);
cudaError_t fma_peak_launch(uint32_t* sink, int iters, int grid, cudaStream_t s);
cudaError_t read_floor_launch(const void* buf, int64_t bytes, uint32_t* sink, int grid, int mode,
                              cudaStream_t s);
// bytes / 16 16-byte words from src to dst (both 16-byte aligned, device-
// accessible: device memory or the device mapping of page-locked host memory),
// as a programmatic dependent launch that touches memory only after the
// dependency wait.
cudaError_t copy16_launch(void* dst, const void* src, int64_t bytes, int sms, cudaStream_t s);

// Split-K partition shared by every kernel: CTA c owns work units
// [c U / G, (c + 1) U / G) of the linear order (tile, k-block).
__host__ __device__ inline int64_t part_begin(int64_t c, int64_t U, int64_t G) {
  return c * U / G;
}
// The CTA whose range holds unit u.
__host__ __device__ inline int64_t part_owner(int64_t u, int64_t U, int64_t G) {
  return ((u + 1) * G - 1) / U;
}

}  // namespace proj
