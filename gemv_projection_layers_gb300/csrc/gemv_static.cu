// gemv_static.cu -- proj_gemv_static: the streaming GEMV (m <= 2) on the
// caller's own row-major weights, with its scratch in a static device array,
// so that a call allocates no device memory at all.
//
// Who needs it: a component that is handed only its input and output
// buffers by a host framework that owns every byte of device memory (a
// plugin or custom operator inside an inference engine, whose allocator has
// reserved the free memory up front), and latency-critical code that must not
// call cudaMalloc or cudaFree, which can block on the whole device and can
// fail at run time.  Such callers cannot create a handle (proj_prepare
// allocates the repacked weights and the split-K workspace), so this entry
// point streams W exactly as the caller stores it.
//
// The scratch of the GEMV is small and bounded by its CTA count: one
// hand-off flag and MT partial row sums per CTA, plus a status word.  It
// lives in g_gemv_scratch below (4 KB per device, held from the library's
// first use on that device until the process exits).  Host code never passes
// the array's name to a kernel -- in host code that name denotes a host-side
// stand-in, not device memory -- but the device address that
// cudaGetSymbolAddress returns, queried once per device with that device
// current.
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdio>
#include <mutex>

#include "../../include/proj.h"
#include "kernels.h"

namespace proj {
namespace {

// Scratch layout in 32-bit words.
constexpr int kStaticMaxCtas = 256;                  // CTAs of one call, at most
constexpr int kFlagsWord = 0;                        // [kStaticMaxCtas] hand-off flags
constexpr int kStatusWord = kStaticMaxCtas;          // device status word
constexpr int kWsWord = kStaticMaxCtas + 64;         // [kStaticMaxCtas][2] fp32 partials
constexpr int kScratchWords = 1024;                  // 4 KB
static_assert(kWsWord + 2 * kStaticMaxCtas <= kScratchWords, "scratch layout");

static __device__ __align__(256) uint32_t g_gemv_scratch[kScratchWords];

constexpr int kMaxDevices = 64;

struct DeviceSlot {
  std::atomic<bool> ready{false};
  uint32_t* scratch = nullptr;  // device address of g_gemv_scratch
  int sms = 0;
};

DeviceSlot g_slots[kMaxDevices];
std::mutex g_setup_mutex;

// Once per device, with that device current: the scratch's device address,
// the SM count and the GEMV kernels' shared-memory attribute.
int setup_device(int dev, DeviceSlot** out) {
  if (dev < 0 || dev >= kMaxDevices)
    return record_status(PROJ_EUNSUPPORTED, "proj_gemv_static: device ordinal above 63");
  DeviceSlot& d = g_slots[dev];
  if (!d.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!d.ready.load(std::memory_order_relaxed)) {
      void* ptr = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&ptr, g_gemv_scratch);
      if (e != cudaSuccess) return record_cuda(e, "proj_gemv_static: cudaGetSymbolAddress");
      int sms = 0;
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return record_cuda(e, "proj_gemv_static: SM count");
      e = gemv_init_attributes();
      if (e != cudaSuccess) return record_cuda(e, "proj_gemv_static: kernel attributes");
      d.scratch = static_cast<uint32_t*>(ptr);
      d.sms = sms;
      d.ready.store(true, std::memory_order_release);
    }
  }
  *out = &d;
  return PROJ_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace proj

using namespace proj;

extern "C" int proj_gemv_static(const void* W, int w_dtype, int64_t N, int64_t K, const void* x,
                                int64_t m, void* out, proj_stream stream) {
  if (!W || !x || !out || N < 1 || m < 0)
    return record_status(PROJ_EINVAL, "proj_gemv_static: null pointer, N < 1 or m < 0");
  if (w_dtype != PROJ_BF16 && w_dtype != PROJ_FP32)
    return record_status(PROJ_EINVAL, "proj_gemv_static: w_dtype is not PROJ_BF16 or PROJ_FP32");
  if (m > 2)
    return record_status(PROJ_EUNSUPPORTED,
                         "proj_gemv_static: m > 2 (the static scratch holds two token rows)");
  if (K < 1024 || K > 8192 || K % 1024 != 0)
    return record_status(PROJ_EUNSUPPORTED,
                         "proj_gemv_static: K must be a multiple of 1024 in [1024, 8192]");
  if (N > INT_MAX) return record_status(PROJ_EUNSUPPORTED, "proj_gemv_static: N > INT_MAX");
  if (!aligned16(W) || !aligned16(x) || !aligned16(out))
    return record_status(PROJ_EALIGN, "proj_gemv_static: pointer not 16-byte aligned");
  if (m == 0) return PROJ_OK;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return record_cuda(e, "proj_gemv_static: cudaGetDevice");
  DeviceSlot* d = nullptr;
  const int st = setup_device(dev, &d);
  if (st != PROJ_OK) return st;

  int64_t G = d->sms < kStaticMaxCtas ? d->sms : kStaticMaxCtas;
  if (G > N) G = N;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The flags and the status word must start at zero; the partial row sums
  // are always written before they are read.  The memset is also what keeps
  // the caller's W safe: the GEMV is a programmatic dependent launch that
  // streams its (constant) weights before its dependency wait, and W here
  // belongs to the caller, who may have written it in the kernel just before.
  // A memset node is an ordinary dependency, so the GEMV starts only after
  // everything earlier on the stream has completed.
  e = cudaMemsetAsync(d->scratch + kFlagsWord, 0, (kStatusWord + 1) * sizeof(uint32_t), s);
  if (e != cudaSuccess) return record_cuda(e, "proj_gemv_static: clearing the scratch flags");
  GemvParams g;
  g.w = W;
  g.x = x;
  g.out = out;
  g.ws = reinterpret_cast<float*>(d->scratch + kWsWord);
  g.flags = d->scratch + kFlagsWord;
  g.status = d->scratch + kStatusWord;
  g.m = static_cast<int>(m);
  g.n_rows = static_cast<int>(N);
  g.K = static_cast<int>(K);
  g.G = static_cast<int>(G);
  g.out_f32 = w_dtype == PROJ_FP32 ? 1 : 0;
  g.esc = nullptr;  // dense weights only
  g.e0x4 = 0;
  e = gemv_launch(w_dtype == PROJ_FP32, static_cast<int>(m), g, s);
  if (e != cudaSuccess) return record_cuda(e, "proj_gemv_static: kernel launch");
  return PROJ_OK;
}

extern "C" int proj_gemv_static_status(proj_stream stream, uint32_t* code) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return record_cuda(e, "proj_gemv_static_status: cudaGetDevice");
  DeviceSlot* d = nullptr;
  const int st = setup_device(dev, &d);
  if (st != PROJ_OK) return st;
  e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return record_cuda(e, "proj_gemv_static_status: stream synchronize");
  uint32_t word = 0;
  e = cudaMemcpy(&word, d->scratch + kStatusWord, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return record_cuda(e, "proj_gemv_static_status: reading the status word");
  if (code) *code = word;
  return word ? record_status(PROJ_EDEVICE, "proj_gemv_static: a bounded wait gave up")
              : PROJ_OK;
}
