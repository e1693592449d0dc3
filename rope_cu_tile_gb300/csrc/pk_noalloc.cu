// pk_noalloc.cu -- pk_attend_noalloc: the attention call for callers that must not allocate.
//
// pk_attend keeps a small per-(device, stream) workspace for the tile scheduler (tile
// records and a control word) and allocates it with cudaMalloc the first time it meets a
// stream or a larger T. Some callers cannot let a library do that: code running where every
// byte of device memory is planned up front (a serving process with a fixed memory budget,
// an inference plugin whose enqueue step is forbidden to allocate, an application whose
// own pool allocator owns the device), or code on a path where a cudaMalloc would
// synchronize the device at the wrong moment. This entry point runs the same scheduler and
// attention kernels on a scratch area that lives in the library image itself: a file-scope
// static __device__ array sized for T <= PK_NOALLOC_MAX_T tokens (about 4 MB, held by
// every GPU that loads the library until the process exits).
//
// It calls no cudaMalloc, cudaFree or other allocating routine. Its first call on a device
// does a one-time set-up with that device current (device check, the kernels' shared-memory
// attribute, and cudaGetSymbolAddress to turn the array into a device address the kernels
// can use); make that first call before any stream capture. Every call, on every stream,
// shares the one array: calls whose work overlaps on the GPU race with each other, so the
// caller must order them (one stream, or events between streams).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <mutex>

#include "pk.h"
#include "pk_dev.cuh"

namespace pk {

cudaError_t attend_tc_prepare();
cudaError_t attend_q4_prepare();
cudaError_t band_prepare();
cudaError_t schedule_prepare();

namespace {

constexpr long long kNoallocMaxT = PK_NOALLOC_MAX_T;
constexpr long long kNoallocCap = 3 * ((kNoallocMaxT + kCapUnit - 1) / kCapUnit) + 1;
constexpr long long kNoallocStage = schedule_stage_records(kNoallocMaxT);
constexpr size_t kScratchBytes = sizeof(Ctl) + static_cast<size_t>(kNoallocCap + kNoallocStage) * sizeof(TileRec);

// The scratch area: the control block, the tile records, then the scheduler's staging slots.
// Zero at load time; each call clears the control block before use.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

struct Setup {
  bool ready = false;
  bool supported = false;
  int sms = 0;
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch on this device
};

std::mutex g_noalloc_mu;
Setup g_noalloc_setup[kMaxDevices];

// once per device, with that device current
int setup_device(int dev, Setup** out) {
  if (dev < 0 || dev >= kMaxDevices) return PK_ERR_UNSUPPORTED;
  Setup& s = g_noalloc_setup[dev];
  if (!s.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return PK_ERR_CUDA;
    s.supported = prop.major == 10 && prop.minor == 3;
    s.sms = prop.multiProcessorCount;
    if (s.supported) {
      if (attend_tc_prepare() != cudaSuccess || attend_q4_prepare() != cudaSuccess || band_prepare() != cudaSuccess ||
          schedule_prepare() != cudaSuccess)
        return PK_ERR_CUDA;
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return PK_ERR_CUDA;
      s.scratch = static_cast<unsigned char*>(p);
    }
    s.ready = true;
  }
  if (!s.supported) return PK_ERR_UNSUPPORTED;
  *out = &s;
  return PK_OK;
}

unsigned long long noalloc_timeout_ns() {
  const char* e = std::getenv("PK_TIMEOUT_MS");
  const long long ms = e ? std::atoll(e) : 0;
  return static_cast<unsigned long long>(ms > 0 ? ms : 2000) * 1000000ull;
}

bool is_aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace pk

using namespace pk;

extern "C" int pk_attend_noalloc(int dtype, const void* qkv, const void* cos, const void* sin, const uint32_t* cu,
                                 int S, int64_t T, int H, int window, float scale, void* out, float* lse,
                                 int* status, struct CUstream_st* stream) {
  if (dtype != PK_F32 && dtype != PK_BF16 && dtype != PK_F16) return PK_ERR_ARG;
  if (S < 0 || T < 0 || H < 1 || H > PK_MAX_H || window < 0) return PK_ERR_ARG;
  if (T > kNoallocMaxT) return PK_ERR_TOO_LARGE;
  if (S == 0 && T != 0) return PK_ERR_ARG;
  if (T > 0 && (!qkv || !cos || !sin || !cu || !out || !lse)) return PK_ERR_ARG;
  if (T > 0 && (!is_aligned(qkv, 16) || !is_aligned(cos, 16) || !is_aligned(sin, 16) || !is_aligned(out, 16) ||
                !is_aligned(cu, 4) || !is_aligned(lse, 4) || (status && !is_aligned(status, 4))))
    return PK_ERR_ALIGN;
  cudaStream_t st = stream;
  if (T == 0) {
    if (status && cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return PK_ERR_CUDA;
    return PK_OK;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PK_ERR_CUDA;
  Setup* s = nullptr;
  int rc = setup_device(dev, &s);
  if (rc != PK_OK) return rc;
  Ctl* ctl = reinterpret_cast<Ctl*>(s->scratch);
  TileRec* tiles = reinterpret_cast<TileRec*>(s->scratch + sizeof(Ctl));
  TileRec* stage = tiles + kNoallocCap;

  // the control block starts each call at zero (the last call's counter and status stay in it)
  if (cudaMemsetAsync(ctl, 0, sizeof(Ctl), st) != cudaSuccess) return PK_ERR_CUDA;
  // the same kernels as pk_attend would run for these arguments
  // (the split kernel for fp32 inputs needs a copy of qkv's size: fp32 calls here run the
  // CUDA-core kernel)
  int kernel = select_forward_kernel(dtype, window);
  if (kernel == kKernelSplit) kernel = kKernelF32;
  rc = forward_launch(kernel, dtype, dtype, qkv, cos, sin, cu, S, static_cast<long long>(T), H, window, scale, out,
                      lse, ctl, tiles, kNoallocCap, stage, nullptr, 0, s->sms, noalloc_timeout_ns(), st, nullptr);
  if (rc != PK_OK) return rc;
  if (status && cudaMemcpyAsync(status, &ctl->status, sizeof(int), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return PK_ERR_CUDA;
  return PK_OK;
}
