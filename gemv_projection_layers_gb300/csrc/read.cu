// read.cu -- the HBM read floor: a kernel that only streams bytes into the SMs.
//
// The pages measure the practical ceiling of a weight stream with a
// hand-written cold-L2 read kernel and a bulk-copy streaming kernel, and find
// both reach the same time (muse_bf16_proj project report, "Method /
// tooling" and "Round 2").  The file also holds the FP32 FMA probe: the
// measured ceiling of the CUDA cores' fused multiply-adds, the denominator
// of the router's FP32-FMA path (guide ch. 1, §1.5: the router in full FP32).  Both forms are here: mode 0 streams with 128-bit
// non-allocating loads into registers, mode 1 with 1-D bulk copies into a
// shared-memory ring.  Each CTA reads one contiguous range; a checksum per
// CTA keeps the loads alive.  Run over a buffer larger than L2 it is also the
// flush that makes the next call's weights cold.
#include "kernels.h"
#include "ptx.cuh"

namespace proj {
namespace {

constexpr int kRegThreads = 512;
constexpr int kRegUnroll = 8;

__global__ void __launch_bounds__(kRegThreads)
    read_regs_kernel(const uint4* __restrict__ buf, int64_t n16, uint32_t* __restrict__ sink) {
  const int64_t b = part_begin(blockIdx.x, n16, gridDim.x);
  const int64_t e = part_begin(blockIdx.x + 1, n16, gridDim.x);
  uint32_t acc = 0;
  for (int64_t i = b + threadIdx.x; i < e; i += static_cast<int64_t>(kRegThreads) * kRegUnroll) {
    uint4 v[kRegUnroll];
#pragma unroll
    for (int u = 0; u < kRegUnroll; ++u) {
      const int64_t j = i + static_cast<int64_t>(u) * kRegThreads;
      v[u] = j < e ? ld_stream_v4(buf + j) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kRegUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  __shared__ uint32_t red[kRegThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t r = 0;
    for (int w = 0; w < kRegThreads / 32; ++w) r ^= red[w];
    sink[blockIdx.x] = r;
  }
}

constexpr int kBulkStages = 12;
constexpr int kBulkChunk = 16384;
constexpr size_t kBulkSmem = 1024 + kBulkStages * kBulkChunk + kBulkStages * 8;

__global__ void __launch_bounds__(32)
    read_bulk_kernel(const uint8_t* __restrict__ buf, int64_t n16, uint32_t* __restrict__ sink,
                     uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t bar0 = smem_u32(smem + kBulkStages * kBulkChunk);
  const int64_t b = part_begin(blockIdx.x, n16, gridDim.x) * 16;
  const int64_t e = part_begin(blockIdx.x + 1, n16, gridDim.x) * 16;
  const int64_t nchunks = (e - b + kBulkChunk - 1) / kBulkChunk;
  if (threadIdx.x != 0) return;
  for (int s = 0; s < kBulkStages; ++s) mbar_init(bar0 + 8 * s, 1);
  fence_mbar_init();
  const uint64_t pol = policy_evict_first();
  auto issue = [&](int64_t j) {
    const int64_t off = b + j * kBulkChunk;
    const int64_t left = e - off;
    const uint32_t bytes = static_cast<uint32_t>(left < kBulkChunk ? left : kBulkChunk);
    const int s = static_cast<int>(j % kBulkStages);
    mbar_arrive_expect_tx(bar0 + 8 * s, bytes);
    bulk_g2s(smem_u32(smem + s * kBulkChunk), buf + off, bytes, bar0 + 8 * s, pol);
  };
  int64_t issued = 0;
  for (; issued < nchunks && issued < kBulkStages; ++issued) issue(issued);
  uint32_t acc = 0;
  for (int64_t j = 0; j < nchunks; ++j) {
    const int s = static_cast<int>(j % kBulkStages);
    if (!mbar_wait(bar0 + 8 * s, static_cast<uint32_t>((j / kBulkStages) & 1), status,
                   kStatusTimeoutProducer)) {
      break;
    }
    acc ^= *reinterpret_cast<const uint32_t*>(smem + s * kBulkChunk);
    if (issued < nchunks) issue(issued++);
  }
  // Drain (normally a no-op: every issued chunk has been waited on).
  for (int64_t j = issued > kBulkStages ? issued - kBulkStages : 0; j < issued; ++j)
    mbar_wait(bar0 + 8 * static_cast<int>(j % kBulkStages),
              static_cast<uint32_t>((j / kBulkStages) & 1), status, kStatusTimeoutDrain);
  sink[blockIdx.x] = acc;
}

// 16-byte copy, grid-stride (proj_run_host: host-mapped buffers <-> device),
// launched as a programmatic dependent launch: it may start during the
// previous kernel's tail, but reads and writes only after it (the source may
// be that kernel's output, even through host memory).
__global__ void __launch_bounds__(256) copy16_kernel(uint4* __restrict__ dst,
                                                     const uint4* __restrict__ src, int64_t n16) {
  griddep_launch_dependents();
  griddep_wait();
  for (int64_t i = blockIdx.x * 256ll + threadIdx.x; i < n16; i += gridDim.x * 256ll) dst[i] = src[i];
}

// FP32 FMA probe: every thread runs kFmaChains independent dependency chains
// of packed fp32x2 fused multiply-adds (acc = acc * mul + add, both halves),
// so the FMA pipes, not latency, set the rate.  mul and add depend on the
// kernel argument, and the chains' sum decides a store the host never asks
// for, so nothing is folded or dropped.  Measured on GB300 (eight CTAs of
// 256 threads per SM, 2070 MHz): 8 chains unrolled 64 deep 78.5 TFLOP/s,
// 0.97 of SMs x 128 lanes x 2 x clock; a 4-deep unroll 68.7, 12-16 chains
// 68-72, scalar fma.rn.f32 77.
constexpr int kFmaThreads = 256;
constexpr int kFmaChains = 8;

__device__ __forceinline__ uint64_t pack_f2(float lo, float hi) {
  return (static_cast<uint64_t>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}

__global__ void __launch_bounds__(kFmaThreads)
    fma_peak_kernel(uint32_t* __restrict__ sink, int iters, float seed) {
  const float base = seed + static_cast<float>(threadIdx.x) * 1e-6f;
  uint64_t acc[kFmaChains];
#pragma unroll
  for (int c = 0; c < kFmaChains; ++c)
    acc[c] = pack_f2(base + static_cast<float>(c), base - static_cast<float>(c));
  const uint64_t mul = pack_f2(1.0f - 1e-7f * seed, 1.0f + 1e-7f * seed);
  const uint64_t add = pack_f2(1e-7f * seed, -1e-7f * seed);
#pragma unroll 64
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < kFmaChains; ++c)
      asm("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(acc[c]) : "l"(mul), "l"(add));
  }
  float sum = 0.f;
#pragma unroll
  for (int c = 0; c < kFmaChains; ++c)
    sum += __uint_as_float(static_cast<uint32_t>(acc[c])) +
           __uint_as_float(static_cast<uint32_t>(acc[c] >> 32));
  if (sum == 1.25e30f) sink[0] = __float_as_uint(sum);
}

}  // namespace

double fma_peak_flops(int grid, int iters) {
  return static_cast<double>(grid) * kFmaThreads * kFmaChains * 2.0 * 2.0 * iters;
}

cudaError_t fma_peak_launch(uint32_t* sink, int iters, int grid, cudaStream_t s) {
  fma_peak_kernel<<<grid, kFmaThreads, 0, s>>>(sink, iters, 1.0f);
  return cudaGetLastError();
}

cudaError_t copy16_launch(void* dst, const void* src, int64_t bytes, int sms, cudaStream_t s) {
  const int64_t n16 = bytes / 16;
  if (n16 == 0) return cudaSuccess;
  int64_t grid = (n16 + 255) / 256;
  if (grid > 4ll * sms) grid = 4ll * sms;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, copy16_kernel, static_cast<uint4*>(dst),
                            static_cast<const uint4*>(src), n16);
}

cudaError_t read_floor_launch(const void* buf, int64_t bytes, uint32_t* sink, int grid, int mode,
                              cudaStream_t s) {
  const int64_t n16 = bytes / 16;
  // mode bit 2: launched like the projection kernels, as a programmatic
  // dependent launch (it may start as the previous kernel's CTAs exit; it
  // reads nothing that kernel writes)
  const bool pdl = (mode & 4) != 0;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if ((mode & 3) == 0) {
    cfg.blockDim = dim3(kRegThreads);
    return cudaLaunchKernelEx(&cfg, read_regs_kernel, static_cast<const uint4*>(buf), n16, sink);
  }
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(read_bulk_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kBulkSmem));
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  // The status word for the bulk form lives in the tail of the sink buffer.
  cfg.blockDim = dim3(32);
  cfg.dynamicSmemBytes = kBulkSmem;
  return cudaLaunchKernelEx(&cfg, read_bulk_kernel, static_cast<const uint8_t*>(buf), n16, sink,
                            sink + grid);
}

}  // namespace proj
