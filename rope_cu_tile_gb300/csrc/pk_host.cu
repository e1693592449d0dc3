// pk_host.cu -- the C ABI of include/pk.h: argument checks, the per-(device, stream)
// workspace, the qkv tensor map, and the two launches of a call (scheduler, then the
// attention kernel of the element type).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "pk.h"
#include "pk_dev.cuh"

namespace pk {

cudaError_t schedule_launch(const uint32_t* cu, int S, long long T, int window, TileRec* tiles, long long cap,
                            TileRec* stage, Ctl* ctl, cudaStream_t stream);
cudaError_t attend_tc_prepare();
cudaError_t schedule_prepare();
cudaError_t backward_prepare();
long long backward_scratch_floats(long long T, int H);
cudaError_t backward_launch(int dtype, const void* qkv, const void* cos_t, const void* sin_t, const uint32_t* cu,
                            int S, long long T, int H, int window, float scale, const void* out, const float* lse,
                            const void* dout, void* dqkv, const TileRec* tiles, Ctl* ctl, float* scratch, int sms,
                            cudaStream_t stream);
cudaError_t attend_tc_launch(bool bf16, const CUtensorMap& tmap, const void* cos_t, const void* sin_t,
                             const uint32_t* cu, const TileRec* tiles, void* out, float* lse, Ctl* ctl, int H,
                             long long T, int window, float scale, unsigned long long timeout_ns, int grid,
                             bool singles, bool out32, bool prerotated, cudaStream_t stream);
cudaError_t rotate16_launch(int op_dtype, const float* qkv, const float* cos_t, const float* sin_t, const uint32_t* cu,
                            int S, long long T, int H, float q_mul, const Ctl* ctl, void* y, int sms,
                            cudaStream_t stream);
cudaError_t attend_q4_prepare();
cudaError_t attend_q4_launch(bool bf16, const CUtensorMap& tmap, const void* cos_t, const void* sin_t,
                             const uint32_t* cu, const TileRec* tiles, void* out, float* lse, Ctl* ctl, int H,
                             long long T, int window, float scale, unsigned long long timeout_ns, int grid,
                             cudaStream_t stream);
cudaError_t band_prepare();
long long band_first_words(long long T);
cudaError_t band_prep_launch(const uint32_t* cu, int S, long long T, uint32_t* first, Ctl* ctl, cudaStream_t stream);
cudaError_t band_launch(int dtype, int out_dtype, const void* qkv, const void* cos_t, const void* sin_t,
                        const uint32_t* cu, int S, uint32_t* first, void* out, float* lse, Ctl* ctl, int H, long long T,
                        int window, float scale, cudaStream_t stream);
cudaError_t attend_split_prepare();
cudaError_t split16_launch(const float* qkv, const float* cos_t, const float* sin_t, const uint32_t* cu, int S,
                           long long T, int H, float q_mul, const Ctl* ctl, void* y, int sms, cudaStream_t stream);
cudaError_t attend_split_launch(const CUtensorMap& tmap, const uint32_t* cu, const TileRec* tiles, float* out,
                                float* lse, Ctl* ctl, int H, long long T, int window, float scale,
                                unsigned long long timeout_ns, int grid, cudaStream_t stream);
cudaError_t attend_f32_launch(const float* qkv, const float* cos_t, const float* sin_t, const uint32_t* cu,
                              const TileRec* tiles, void* out, int out_dtype, float* lse, Ctl* ctl, int H,
                              long long T, int window, float scale, int grid, cudaStream_t stream);

namespace {

int64_t schedule_capacity(int64_t T) { return 3 * ((T + kCapUnit - 1) / kCapUnit) + 1; }

struct Workspace {
  void* base = nullptr;
  Ctl* ctl = nullptr;
  TileRec* tiles = nullptr;  // cap records
  TileRec* stage = nullptr;  // the scheduler's staging slots
  int64_t cap = 0;
  int64_t room = 0;  // tokens the workspace is sized for
  float* bwd = nullptr;    // the backward pass's fp32 scratch (allocated on its first use)
  int64_t bwd_floats = 0;
  void* ops16 = nullptr;   // pk_attend_mixed_ops: the rotated 16-bit copy of qkv (first use)
  int64_t ops16_bytes = 0;
};

struct DeviceInfo {
  bool checked = false;
  bool supported = false;
  int sms = 0;
  bool attrs_set = false;
};

// kernel timing (pk_profile_start / pk_profile_stop)
struct Profile {
  bool on = false;
  int dev = -1;
  int cap = 0;
  int used = 0;
  cudaEvent_t* ev = nullptr;  // 3 per call: before schedule, before attention, after attention
};

std::mutex g_mu;
Profile g_prof;

// Tile autotuning (hanzo-kernel packed.rs fn attend_tuned): the fastest usable kernel for a
// (device, element type, heads, window, tokens, longest sequence) key, timed once and kept.
// Like the pages' key, the window enters as w + 1 (0: every key) and the token count and the
// longest length as their next powers of two.
struct TuneKey {
  int dev, dtype, heads, window1;
  long long tokens, longest;
  bool operator<(const TuneKey& o) const {
    if (dev != o.dev) return dev < o.dev;
    if (dtype != o.dtype) return dtype < o.dtype;
    if (heads != o.heads) return heads < o.heads;
    if (window1 != o.window1) return window1 < o.window1;
    if (tokens != o.tokens) return tokens < o.tokens;
    return longest < o.longest;
  }
};
std::map<TuneKey, int> g_tune;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;
std::map<int, DeviceInfo> g_dev;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

unsigned long long timeout_ns() {
  static unsigned long long t = 0;
  if (!t) {
    const char* e = std::getenv("PK_TIMEOUT_MS");
    long long ms = e ? std::atoll(e) : 0;
    t = static_cast<unsigned long long>(ms > 0 ? ms : 2000) * 1000000ull;
  }
  return t;
}

// The forward kernels a call can run:
//   kBand  narrow windows (1 <= w <= kBandMaxW), any element type: CUDA cores, fp32 (no tile
//          records: a check of cu replaces the scheduler);
//   kF32   fp32 inputs otherwise: CUDA cores, fp32;
//   kSplit fp32 inputs otherwise: tensor cores on split bf16 operands (a pre-pass writes the
//          rotated hi / lo copy into the workspace);
//   kTc    16-bit inputs: the paired-stream tensor-core kernel (two query tiles in flight per
//          SM, 128-key stream tiles);
//   kQ4    16-bit inputs: the four-chain tensor-core kernel (two pipes of two query tiles,
//          64-key stream tiles).
// PK_ATTN=tc, q4 or tc_single picks the tensor-core kernel for 16-bit inputs; PK_ATTN=f32 or
// split the kernel for fp32 inputs.
constexpr int kBandMaxW = 16;
int tensor_kernel_choice() {
  const char* e = std::getenv("PK_ATTN");
  if (e && std::strcmp(e, "q4") == 0) return kKernelQ4;
  if (e && std::strcmp(e, "tc_single") == 0) return kKernelTcSingle;
  return kKernelTc;
}

}  // namespace

int select_forward_kernel(int dtype, int window) {
  if (window >= 1 && window <= kBandMaxW) return kKernelBand;
  if (dtype == PK_F32) {
    const char* e = std::getenv("PK_ATTN");
    return (e && std::strcmp(e, "split") == 0) ? kKernelSplit : kKernelF32;
  }
  return tensor_kernel_choice();
}

namespace {

// device checks (caller holds g_mu)
int device_info(int dev, DeviceInfo** out) {
  DeviceInfo& di = g_dev[dev];
  if (!di.checked) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return PK_ERR_CUDA;
    di.checked = true;
    di.supported = prop.major == 10 && prop.minor == 3;
    di.sms = prop.multiProcessorCount;
  }
  if (!di.supported) return PK_ERR_UNSUPPORTED;
  if (!di.attrs_set) {
    if (attend_tc_prepare() != cudaSuccess || attend_q4_prepare() != cudaSuccess || band_prepare() != cudaSuccess ||
        attend_split_prepare() != cudaSuccess || schedule_prepare() != cudaSuccess || backward_prepare() != cudaSuccess)
      return PK_ERR_CUDA;
    di.attrs_set = true;
  }
  *out = &di;
  return PK_OK;
}

// the workspace of (dev, stream) sized for T tokens: the records and the scheduler's staging
// slots (caller holds g_mu)
int workspace(int dev, cudaStream_t stream, int64_t T, Workspace** out) {
  Workspace& ws = g_ws[std::make_pair(dev, stream)];
  if (ws.base && ws.room >= T) {
    *out = &ws;
    return PK_OK;
  }
  cudaStreamCaptureStatus cap_status = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap_status) != cudaSuccess) {
    cudaGetLastError();
    return PK_ERR_CUDA;
  }
  if (cap_status != cudaStreamCaptureStatusNone) return PK_ERR_CAPTURE;
  int carried = 0;
  if (ws.base) {
    // keep the sticky status across the move
    if (cudaStreamSynchronize(stream) != cudaSuccess) return PK_ERR_CUDA;
    if (cudaMemcpy(&carried, &ws.ctl->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
      return PK_ERR_CUDA;
    cudaFree(ws.base);
    if (ws.bwd) cudaFree(ws.bwd);
    if (ws.ops16) cudaFree(ws.ops16);
    ws = Workspace();
  }
  int64_t room = T < 65536 ? 65536 : T;
  room = room + room / 4;  // headroom against regrowth
  const int64_t cap = schedule_capacity(room), stage = schedule_stage_records(room);
  const size_t bytes = sizeof(Ctl) + static_cast<size_t>(cap + stage) * sizeof(TileRec);
  void* p = nullptr;
  if (cudaMalloc(&p, bytes) != cudaSuccess) {
    cudaGetLastError();
    return PK_ERR_NOMEM;
  }
  Ctl init;
  std::memset(&init, 0, sizeof init);
  init.status = carried;
  if (cudaMemcpy(p, &init, sizeof init, cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaFree(p);
    return PK_ERR_CUDA;
  }
  ws.base = p;
  ws.ctl = static_cast<Ctl*>(p);
  ws.tiles = reinterpret_cast<TileRec*>(static_cast<char*>(p) + sizeof(Ctl));
  ws.stage = ws.tiles + cap;
  ws.cap = cap;
  ws.room = room;
  *out = &ws;
  return PK_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_args(int dtype, const void* qkv, const void* cos, const void* sin, const uint32_t* cu, int S,
               int64_t T, int H, int window, const void* out, const float* lse) {
  if (dtype != PK_F32 && dtype != PK_BF16 && dtype != PK_F16) return PK_ERR_ARG;
  if (S < 0 || T < 0 || T > PK_MAX_T || H < 1 || H > PK_MAX_H || window < 0) return PK_ERR_ARG;
  if (S == 0 && T != 0) return PK_ERR_ARG;
  if (T > 0 && (!qkv || !cos || !sin || !cu || !out || !lse)) return PK_ERR_ARG;
  if (T > 0 && (!aligned(qkv, 16) || !aligned(cos, 16) || !aligned(sin, 16) || !aligned(out, 16) ||
                !aligned(cu, 4) || !aligned(lse, 4)))
    return PK_ERR_ALIGN;
  return PK_OK;
}

int launch_schedule(const uint32_t* cu, int S, int64_t T, int window, Workspace* ws, cudaStream_t stream) {
  return schedule_launch(cu, S, static_cast<long long>(T), window, ws->tiles, static_cast<long long>(ws->cap),
                         ws->stage, ws->ctl, stream) == cudaSuccess
             ? PK_OK
             : PK_ERR_CUDA;
}

// out_dtype: the output's type (the input type, except for fp32 inputs with a 16-bit output)
int ops16_scratch(Workspace* ws, cudaStream_t stream, int64_t bytes);

int attend(int dtype, int out_dtype, const void* qkv, const void* cos, const void* sin, const uint32_t* cu, int S,
           int64_t T, int H, int window, float scale, void* out, float* lse, cudaStream_t stream) {
  int rc = check_args(dtype, qkv, cos, sin, cu, S, T, H, window, out, lse);
  if (rc != PK_OK || T == 0) return rc;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PK_ERR_CUDA;
  DeviceInfo* di = nullptr;
  if ((rc = device_info(dev, &di)) != PK_OK) return rc;
  Workspace* ws = nullptr;
  if ((rc = workspace(dev, stream, T, &ws)) != PK_OK) return rc;
  int kernel = select_forward_kernel(dtype, window);
  if (kernel == kKernelSplit && out_dtype != PK_F32) kernel = kKernelF32;  // the split kernel writes fp32
  if (kernel == kKernelSplit && (rc = ops16_scratch(ws, stream, split_copy_bytes(T, H))) != PK_OK) return rc;
  cudaEvent_t* ev = nullptr;
  if (g_prof.on && g_prof.dev == dev && g_prof.used < g_prof.cap) ev = g_prof.ev + 3 * g_prof.used++;
  return forward_launch(kernel, dtype, out_dtype, qkv, cos, sin, cu, S, static_cast<long long>(T), H, window, scale,
                        out, lse, ws->ctl, ws->tiles, ws->cap, ws->stage, ws->ops16, ws->ops16_bytes, di->sms,
                        timeout_ns(), stream, ev);
}

long long next_pow2(long long x) {
  long long p = 1;
  while (p < x) p <<= 1;
  return p;
}

TuneKey tune_key(int dev, int dtype, int H, int window, long long T, long long longest) {
  return TuneKey{dev, dtype, H, window > 0 ? window + 1 : 0, next_pow2(T), next_pow2(longest)};
}

// The kernels a call may run, fastest first unknown: narrow windows keep to the band kernel
// (fp32 arithmetic: the tensor-core kernels round q' and k' to the element type, which costs
// fp16 inputs of large magnitude their tolerance), fp32 inputs to the CUDA-core kernels.
constexpr int kMaxCandidates = 3;  // the longest list tune_candidates writes
int tune_candidates(int dtype, int window, int* c) {
  if (window >= 1 && window <= kBandMaxW) {
    c[0] = kKernelBand;
    return 1;
  }
  if (dtype == PK_F32) {
    c[0] = kKernelF32;
    c[1] = kKernelSplit;
    return 2;
  }
  c[0] = kKernelTc;
  c[1] = kKernelTcSingle;
  c[2] = kKernelQ4;
  return 3;
}

constexpr int kTuneRounds = 3;  // timing rounds over the candidates (after one untimed launch each)

int attend_tuned(int dtype, const void* qkv, const void* cos, const void* sin, const uint32_t* cu, int S, int64_t T,
                 int H, int window, float scale, int64_t longest, void* out, float* lse, cudaStream_t stream) {
  int rc = check_args(dtype, qkv, cos, sin, cu, S, T, H, window, out, lse);
  if (rc != PK_OK || T == 0) return rc;
  if (longest < 0) return PK_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PK_ERR_CUDA;
  DeviceInfo* di = nullptr;
  if ((rc = device_info(dev, &di)) != PK_OK) return rc;
  Workspace* ws = nullptr;
  if ((rc = workspace(dev, stream, T, &ws)) != PK_OK) return rc;
  auto run = [&](int kernel, cudaEvent_t* ev) {
    int r = PK_OK;
    if (kernel == kKernelSplit && (r = ops16_scratch(ws, stream, split_copy_bytes(T, H))) != PK_OK) return r;
    return forward_launch(kernel, dtype, dtype, qkv, cos, sin, cu, S, static_cast<long long>(T), H, window, scale, out,
                          lse, ws->ctl, ws->tiles, ws->cap, ws->stage, ws->ops16, ws->ops16_bytes, di->sms,
                          timeout_ns(), stream, ev);
  };
  const TuneKey key = tune_key(dev, dtype, H, window, T, longest);
  auto it = g_tune.find(key);
  int kernel;
  if (it != g_tune.end()) {
    kernel = it->second;
  } else {
    int cand[kMaxCandidates];
    const int n = tune_candidates(dtype, window, cand);
    kernel = cand[0];
    if (n > 1) {
      // timing needs the host to wait for the stream: not while it is being captured
      cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
      if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        return PK_ERR_CUDA;
      }
      if (cs != cudaStreamCaptureStatusNone) return PK_ERR_CAPTURE;
      cudaEvent_t e0, e1;
      if (cudaEventCreate(&e0) != cudaSuccess) return PK_ERR_CUDA;
      if (cudaEventCreate(&e1) != cudaSuccess) {
        cudaEventDestroy(e0);
        return PK_ERR_CUDA;
      }
      // every candidate once untimed, then kTuneRounds rounds over the candidates in turn (so
      // that clock or cache drift during the tuning touches them alike), each timing two launches;
      // a candidate's time is its best round
      float best_ms[kMaxCandidates] = {};
      for (int i = 0; i < n && rc == PK_OK; ++i) rc = run(cand[i], nullptr);
      for (int round = 0; round < kTuneRounds && rc == PK_OK; ++round) {
        for (int i = 0; i < n && rc == PK_OK; ++i) {
          if (cudaEventRecord(e0, stream) != cudaSuccess) rc = PK_ERR_CUDA;
          for (int r = 0; r < 2 && rc == PK_OK; ++r) rc = run(cand[i], nullptr);
          float ms = 0.f;
          if (rc == PK_OK && (cudaEventRecord(e1, stream) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
                              cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess))
            rc = PK_ERR_CUDA;
          if (rc == PK_OK && (round == 0 || ms < best_ms[i])) best_ms[i] = ms;
        }
      }
      int bi = 0;
      for (int i = 1; i < n; ++i)
        if (best_ms[i] < best_ms[bi]) bi = i;
      kernel = cand[bi];
      cudaEventDestroy(e0);
      cudaEventDestroy(e1);
      if (rc != PK_OK) return rc;
    }
    g_tune[key] = kernel;
  }
  cudaEvent_t* ev = nullptr;
  if (g_prof.on && g_prof.dev == dev && g_prof.used < g_prof.cap) ev = g_prof.ev + 3 * g_prof.used++;
  return run(kernel, ev);
}

// the backward scratch of a workspace, grown to `floats` (caller holds g_mu)
int backward_scratch(Workspace* ws, cudaStream_t stream, int64_t floats) {
  if (ws->bwd && ws->bwd_floats >= floats) return PK_OK;
  cudaStreamCaptureStatus cap_status = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap_status) != cudaSuccess) {
    cudaGetLastError();
    return PK_ERR_CUDA;
  }
  if (cap_status != cudaStreamCaptureStatusNone) return PK_ERR_CAPTURE;
  if (ws->bwd) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return PK_ERR_CUDA;
    cudaFree(ws->bwd);
    ws->bwd = nullptr;
    ws->bwd_floats = 0;
  }
  const int64_t want = floats + floats / 4;
  void* p = nullptr;
  if (cudaMalloc(&p, static_cast<size_t>(want) * sizeof(float)) != cudaSuccess) {
    cudaGetLastError();
    return PK_ERR_NOMEM;
  }
  ws->bwd = static_cast<float*>(p);
  ws->bwd_floats = want;
  return PK_OK;
}

// the rotated 16-bit copy of qkv of a workspace, grown to `bytes` (caller holds g_mu)
int ops16_scratch(Workspace* ws, cudaStream_t stream, int64_t bytes) {
  if (ws->ops16 && ws->ops16_bytes >= bytes) return PK_OK;
  cudaStreamCaptureStatus cap_status = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap_status) != cudaSuccess) {
    cudaGetLastError();
    return PK_ERR_CUDA;
  }
  if (cap_status != cudaStreamCaptureStatusNone) return PK_ERR_CAPTURE;
  if (ws->ops16) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return PK_ERR_CUDA;
    cudaFree(ws->ops16);
    ws->ops16 = nullptr;
    ws->ops16_bytes = 0;
  }
  const int64_t want = bytes + bytes / 4;
  void* p = nullptr;
  if (cudaMalloc(&p, static_cast<size_t>(want)) != cudaSuccess) {
    cudaGetLastError();
    return PK_ERR_NOMEM;
  }
  ws->ops16 = p;
  ws->ops16_bytes = want;
  return PK_OK;
}

// fp32 storage, 16-bit operands: the scheduler, the rotated 16-bit copy, then the paired
// tensor-core kernel on that copy (no rotation of its own) with an fp32 output
int attend_mixed_ops(int op_dtype, const float* qkv, const float* cos, const float* sin, const uint32_t* cu, int S,
                     int64_t T, int H, int window, float scale, float* out, float* lse, cudaStream_t stream) {
  if (op_dtype != PK_BF16 && op_dtype != PK_F16) return PK_ERR_ARG;
  int rc = check_args(PK_F32, qkv, cos, sin, cu, S, T, H, window, out, lse);
  if (rc != PK_OK || T == 0) return rc;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PK_ERR_CUDA;
  DeviceInfo* di = nullptr;
  if ((rc = device_info(dev, &di)) != PK_OK) return rc;
  Workspace* ws = nullptr;
  if ((rc = workspace(dev, stream, T, &ws)) != PK_OK) return rc;
  const int64_t elems = static_cast<int64_t>(T) * 3 * H * kD;
  if ((rc = ops16_scratch(ws, stream, elems * 2)) != PK_OK) return rc;
  cudaEvent_t* ev = nullptr;
  if (g_prof.on && g_prof.dev == dev && g_prof.used < g_prof.cap) ev = g_prof.ev + 3 * g_prof.used++;
  if (ev && cudaEventRecord(ev[0], stream) != cudaSuccess) return PK_ERR_CUDA;
  if ((rc = launch_schedule(cu, S, T, window, ws, stream)) != PK_OK) return rc;
  // a positive scale multiplies the scores in the attention kernel; any other the rotated q here
  if (rotate16_launch(op_dtype, qkv, cos, sin, cu, S, static_cast<long long>(T), H, scale > 0.0f ? 1.0f : scale,
                      ws->ctl, ws->ops16, di->sms, stream) != cudaSuccess)
    return PK_ERR_CUDA;
  if (ev && cudaEventRecord(ev[1], stream) != cudaSuccess) return PK_ERR_CUDA;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return PK_ERR_CUDA;
  CUtensorMap tmap;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(3) * H * kD, static_cast<cuuint64_t>(T)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(3) * H * kD * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kD), static_cast<cuuint32_t>(kBR)};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(&tmap, op_dtype == PK_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, ws->ops16,
          dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return PK_ERR_CUDA;
  if (attend_tc_launch(op_dtype == PK_BF16, tmap, cos, sin, cu, ws->tiles, out, lse, ws->ctl, H,
                       static_cast<long long>(T), window, scale, timeout_ns(), di->sms, false, true, true,
                       stream) != cudaSuccess)
    return PK_ERR_CUDA;
  if (ev && cudaEventRecord(ev[2], stream) != cudaSuccess) return PK_ERR_CUDA;
  return PK_OK;
}

int attend_backward(int dtype, const void* qkv, const void* cos, const void* sin, const uint32_t* cu, int S,
                    int64_t T, int H, int window, float scale, const void* out, const float* lse, const void* dout,
                    void* dqkv, cudaStream_t stream) {
  int rc = check_args(dtype, qkv, cos, sin, cu, S, T, H, window, out, lse);
  if (rc != PK_OK || T == 0) return rc;
  if (!dout || !dqkv) return PK_ERR_ARG;
  if (!aligned(dout, 16) || !aligned(dqkv, 16)) return PK_ERR_ALIGN;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PK_ERR_CUDA;
  DeviceInfo* di = nullptr;
  if ((rc = device_info(dev, &di)) != PK_OK) return rc;
  Workspace* ws = nullptr;
  if ((rc = workspace(dev, stream, T, &ws)) != PK_OK) return rc;
  if ((rc = backward_scratch(ws, stream, backward_scratch_floats(T, H))) != PK_OK) return rc;
  if ((rc = launch_schedule(cu, S, T, window, ws, stream)) != PK_OK) return rc;
  return backward_launch(dtype, qkv, cos, sin, cu, S, static_cast<long long>(T), H, window, scale, out, lse, dout,
                         dqkv, ws->tiles, ws->ctl, ws->bwd, di->sms, stream) == cudaSuccess
             ? PK_OK
             : PK_ERR_CUDA;
}

}  // namespace

int forward_launch(int kernel, int dtype, int out_dtype, const void* qkv, const void* cos, const void* sin,
                   const uint32_t* cu, int S, long long T, int H, int window, float scale, void* out, float* lse,
                   Ctl* ctl, TileRec* tiles, long long cap, TileRec* stage, void* copy, long long copy_bytes, int sms,
                   unsigned long long timeout, cudaStream_t stream, cudaEvent_t* ev) {
  if (ev && cudaEventRecord(ev[0], stream) != cudaSuccess) return PK_ERR_CUDA;
  cudaError_t e = cudaSuccess;
  if (kernel == kKernelBand) {
    // the band kernel needs no tile records: its block-to-sequence table goes where they would
    if (band_first_words(T) * 4 > cap * static_cast<long long>(sizeof(TileRec))) return PK_ERR_INTERNAL;
    uint32_t* first = reinterpret_cast<uint32_t*>(tiles);
    if (band_prep_launch(cu, S, T, first, ctl, stream) != cudaSuccess) return PK_ERR_CUDA;
    if (ev && cudaEventRecord(ev[1], stream) != cudaSuccess) return PK_ERR_CUDA;
    e = band_launch(dtype, out_dtype, qkv, cos, sin, cu, S, first, out, lse, ctl, H, T, window, scale, stream);
    if (e != cudaSuccess) return PK_ERR_CUDA;
    if (ev && cudaEventRecord(ev[2], stream) != cudaSuccess) return PK_ERR_CUDA;
    return PK_OK;
  }
  if (kernel == kKernelSplit &&
      (dtype != PK_F32 || out_dtype != PK_F32 || !copy || copy_bytes < split_copy_bytes(T, H)))
    return PK_ERR_INTERNAL;
  if (schedule_launch(cu, S, T, window, tiles, cap, stage, ctl, stream) != cudaSuccess) return PK_ERR_CUDA;
  // the split kernel's pre-pass: q, k rotated in fp32, then q', k', v as bf16 hi / lo pairs
  // (a positive scale multiplies the scores in the kernel, any other the rotated q here)
  if (kernel == kKernelSplit &&
      split16_launch(static_cast<const float*>(qkv), static_cast<const float*>(cos), static_cast<const float*>(sin),
                     cu, S, T, H, scale > 0.0f ? 1.0f : scale, ctl, copy, sms, stream) != cudaSuccess)
    return PK_ERR_CUDA;
  if (ev && cudaEventRecord(ev[1], stream) != cudaSuccess) return PK_ERR_CUDA;
  if (kernel == kKernelSplit) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return PK_ERR_CUDA;
    CUtensorMap tmap;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(6) * H * kD, static_cast<cuuint64_t>(T)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(6) * H * kD * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kD), static_cast<cuuint32_t>(kBR)};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, copy, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PK_ERR_CUDA;
    e = attend_split_launch(tmap, cu, tiles, static_cast<float*>(out), lse, ctl, H, T, window, scale, timeout, sms,
                            stream);
  } else if (kernel == kKernelF32) {
    e = attend_f32_launch(static_cast<const float*>(qkv), static_cast<const float*>(cos),
                          static_cast<const float*>(sin), cu, tiles, out, out_dtype, lse, ctl, H, T, window, scale,
                          sms * 4, stream);
  } else {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return PK_ERR_CUDA;
    CUtensorMap tmap;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(3) * H * kD, static_cast<cuuint64_t>(T)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(3) * H * kD * 2};
    // box: one 128-row query tile (paired kernel) or one 64-row tile (four-chain kernel)
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kD), static_cast<cuuint32_t>(kernel == kKernelQ4 ? 64 : kBR)};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt =
        dtype == PK_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (enc(&tmap, dt, 2, const_cast<void*>(qkv), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PK_ERR_CUDA;
    if (kernel == kKernelQ4)
      e = attend_q4_launch(dtype == PK_BF16, tmap, cos, sin, cu, tiles, out, lse, ctl, H, T, window, scale, timeout,
                           sms, stream);
    else
      e = attend_tc_launch(dtype == PK_BF16, tmap, cos, sin, cu, tiles, out, lse, ctl, H, T, window, scale, timeout,
                           sms, kernel == kKernelTcSingle, false, false, stream);
  }
  if (e != cudaSuccess) return PK_ERR_CUDA;
  if (ev && cudaEventRecord(ev[2], stream) != cudaSuccess) return PK_ERR_CUDA;
  return PK_OK;
}

}  // namespace pk

using namespace pk;

extern "C" {

int pk_attend_dt(int dtype, const void* qkv, const void* cos, const void* sin, const uint32_t* cu, int S,
                 int64_t T, int H, int window, float scale, void* out, float* lse, struct CUstream_st* stream) {
  return attend(dtype, dtype, qkv, cos, sin, cu, S, T, H, window, scale, out, lse, stream);
}

int pk_attend_mixed(int out_dtype, const float* qkv, const float* cos, const float* sin, const uint32_t* cu, int S,
                    int64_t T, int H, int window, float scale, void* out, float* lse, struct CUstream_st* stream) {
  if (out_dtype != PK_F32 && out_dtype != PK_BF16 && out_dtype != PK_F16) return PK_ERR_ARG;
  return attend(PK_F32, out_dtype, qkv, cos, sin, cu, S, T, H, window, scale, out, lse, stream);
}

int pk_attend_mixed_ops(int op_dtype, const float* qkv, const float* cos, const float* sin, const uint32_t* cu, int S,
                        int64_t T, int H, int window, float scale, float* out, float* lse, struct CUstream_st* stream) {
  return attend_mixed_ops(op_dtype, qkv, cos, sin, cu, S, T, H, window, scale, out, lse, stream);
}

int pk_attend_backward(int dtype, const void* qkv, const void* cos, const void* sin, const uint32_t* cu, int S,
                       int64_t T, int H, int window, float scale, const void* out, const float* lse, const void* dout,
                       void* dqkv, struct CUstream_st* stream) {
  return attend_backward(dtype, qkv, cos, sin, cu, S, T, H, window, scale, out, lse, dout, dqkv, stream);
}

int pk_attend(const void* qkv, const void* cos, const void* sin, const uint32_t* cu, int S, int64_t T, int H,
              int window, float scale, void* out, float* lse, struct CUstream_st* stream) {
  return attend(PK_BF16, PK_BF16, qkv, cos, sin, cu, S, T, H, window, scale, out, lse, stream);
}

int pk_attend_bf16(const void* qkv, const void* cos, const void* sin, const uint32_t* cu, int S, int64_t T,
                   int H, int window, float scale, void* out, float* lse, struct CUstream_st* stream) {
  return attend(PK_BF16, PK_BF16, qkv, cos, sin, cu, S, T, H, window, scale, out, lse, stream);
}

int pk_attend_f16(const void* qkv, const void* cos, const void* sin, const uint32_t* cu, int S, int64_t T,
                  int H, int window, float scale, void* out, float* lse, struct CUstream_st* stream) {
  return attend(PK_F16, PK_F16, qkv, cos, sin, cu, S, T, H, window, scale, out, lse, stream);
}

int pk_attend_f32(const void* qkv, const void* cos, const void* sin, const uint32_t* cu, int S, int64_t T,
                  int H, int window, float scale, void* out, float* lse, struct CUstream_st* stream) {
  return attend(PK_F32, PK_F32, qkv, cos, sin, cu, S, T, H, window, scale, out, lse, stream);
}

int pk_attend_tuned(int dtype, const void* qkv, const void* cos, const void* sin, const uint32_t* cu, int S, int64_t T,
                    int H, int window, float scale, int64_t longest, void* out, float* lse, struct CUstream_st* stream) {
  return attend_tuned(dtype, qkv, cos, sin, cu, S, T, H, window, scale, longest, out, lse, stream);
}

int pk_tune_pick(int dtype, int H, int window, int64_t T, int64_t longest) {
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  auto it = g_tune.find(tune_key(dev, dtype, H, window, T, longest));
  return it == g_tune.end() ? -1 : it->second;
}

int pk_tune_key(int dtype, int H, int window, int64_t T, int64_t longest, char* buf, int n) {
  if (!buf || n < 1 || T < 0 || longest < 0 || window < 0 || H < 1) return PK_ERR_ARG;
  const TuneKey k = tune_key(0, dtype, H, window, T, longest);
  const char* dt = dtype == PK_F32 ? "f32" : dtype == PK_BF16 ? "bf16" : dtype == PK_F16 ? "f16" : "?";
  const int w = std::snprintf(buf, static_cast<size_t>(n), "dtype=%s,heads=%d,window=%d,tokens=%lld,longest=%lld", dt,
                              k.heads, k.window1, k.tokens, k.longest);
  return (w < 0 || w >= n) ? PK_ERR_ARG : PK_OK;
}

int pk_tune_clear(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_tune.clear();
  return PK_OK;
}

const char* pk_kernel_name(int kernel) {
  switch (kernel) {
    case kKernelBand: return "pk_attend_band_kernel";
    case kKernelF32: return "pk_attend_f32_kernel";
    case kKernelTc: return "pk_attend_tc_kernel";
    case kKernelQ4: return "pk_attend_q4_kernel";
    case kKernelTcSingle: return "pk_attend_tc_kernel (single-record items)";
    case kKernelSplit: return "pk_attend_split_kernel";
    default: return "";
  }
}

int pk_forward_kernel(int dtype, int window) { return select_forward_kernel(dtype, window); }

int64_t pk_schedule_capacity(int64_t T) { return T < 0 ? 0 : schedule_capacity(T); }

int pk_schedule(const uint32_t* cu, int S, int64_t T, int window, uint32_t* tiles, int64_t cap, int64_t* nt,
                struct CUstream_st* stream) {
  if (!nt) return PK_ERR_ARG;
  *nt = 0;
  if (S < 0 || T < 0 || T > PK_MAX_T || window < 0 || (S == 0 && T != 0)) return PK_ERR_ARG;
  if (T == 0) return PK_OK;
  if (!cu || !tiles || !aligned(tiles, 16) || !aligned(cu, 4)) return PK_ERR_ARG;
  if (cap < schedule_capacity(T)) return PK_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PK_ERR_CUDA;
  DeviceInfo* di = nullptr;
  int rc = device_info(dev, &di);
  if (rc != PK_OK) return rc;
  Workspace* ws = nullptr;
  if ((rc = workspace(dev, stream, T, &ws)) != PK_OK) return rc;
  if ((rc = launch_schedule(cu, S, T, window, ws, stream)) != PK_OK) return rc;
  Ctl ctl;
  if (cudaMemcpyAsync(&ctl, ws->ctl, sizeof ctl, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return PK_ERR_CUDA;
  if (ctl.status == PK_ERR_BAD_CU) {
    int zero = 0;
    cudaMemcpy(&ws->ctl->status, &zero, sizeof zero, cudaMemcpyHostToDevice);
    return PK_ERR_BAD_CU;
  }
  if (ctl.ntiles > 0 &&
      cudaMemcpyAsync(tiles, ws->tiles, static_cast<size_t>(ctl.ntiles) * sizeof(TileRec), cudaMemcpyDeviceToDevice,
                      stream) != cudaSuccess)
    return PK_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return PK_ERR_CUDA;
  *nt = ctl.ntiles;
  return PK_OK;
}

int pk_last_status(struct CUstream_st* stream) {
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PK_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return PK_ERR_CUDA;
  auto it = g_ws.find(std::make_pair(dev, static_cast<cudaStream_t>(stream)));
  if (it == g_ws.end() || !it->second.base) return PK_OK;
  int st = 0, zero = 0;
  if (cudaMemcpy(&st, &it->second.ctl->status, sizeof st, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(&it->second.ctl->status, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
    return PK_ERR_CUDA;
  return st;
}

int pk_profile_start(int n) {
  if (n < 1) return PK_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PK_ERR_CUDA;
  if (g_prof.ev) {
    for (int i = 0; i < 3 * g_prof.cap; ++i) cudaEventDestroy(g_prof.ev[i]);
    delete[] g_prof.ev;
  }
  g_prof = Profile();
  g_prof.ev = new cudaEvent_t[3 * n];
  for (int i = 0; i < 3 * n; ++i)
    if (cudaEventCreate(&g_prof.ev[i]) != cudaSuccess) {
      for (int k = 0; k < i; ++k) cudaEventDestroy(g_prof.ev[k]);
      delete[] g_prof.ev;
      g_prof = Profile();
      return PK_ERR_CUDA;
    }
  g_prof.cap = n;
  g_prof.dev = dev;
  g_prof.on = true;
  return PK_OK;
}

int pk_profile_stop(double* schedule_ms, double* attend_ms, int* calls) {
  if (!schedule_ms || !attend_ms || !calls) return PK_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  *schedule_ms = 0.0;
  *attend_ms = 0.0;
  *calls = 0;
  int rc = PK_OK;
  for (int i = 0; i < g_prof.used; ++i) {
    float a = 0.f, b = 0.f;
    cudaEvent_t* e = g_prof.ev + 3 * i;
    if (cudaEventSynchronize(e[2]) != cudaSuccess || cudaEventElapsedTime(&a, e[0], e[1]) != cudaSuccess ||
        cudaEventElapsedTime(&b, e[1], e[2]) != cudaSuccess) {
      rc = PK_ERR_CUDA;
      break;
    }
    *schedule_ms += a;
    *attend_ms += b;
    ++*calls;
  }
  if (g_prof.ev) {
    for (int i = 0; i < 3 * g_prof.cap; ++i) cudaEventDestroy(g_prof.ev[i]);
    delete[] g_prof.ev;
  }
  g_prof = Profile();
  return rc;
}

const char* pk_status_string(int status) {
  switch (status) {
    case PK_OK: return "ok";
    case PK_ERR_ARG: return "invalid argument";
    case PK_ERR_ALIGN: return "pointer not aligned (see the entry point's alignment rules in pk.h)";
    case PK_ERR_CUDA: return "CUDA runtime or driver call failed";
    case PK_ERR_UNSUPPORTED: return "device is not sm_103 (GB300)";
    case PK_ERR_BAD_CU: return "cu malformed (cu[0] != 0, decreasing, or cu[S] != T), or a position past the tables";
    case PK_ERR_TIMEOUT: return "a device wait exceeded its bound; results invalid";
    case PK_ERR_NOMEM: return "workspace allocation failed";
    case PK_ERR_INTERNAL: return "schedule capacity exceeded (library bug)";
    case PK_ERR_TOO_LARGE: return "T exceeds PK_NOALLOC_MAX_T, the static scratch capacity of pk_attend_noalloc";
    case PK_ERR_CAPTURE: return "stream capture would have to allocate the workspace: make one uncaptured call first";
    default: return "unknown status";
  }
}

int pk_version(void) { return 100; }

int pk_release(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int rc = PK_OK;
  int cur = 0;
  cudaGetDevice(&cur);
  // each device with a workspace is synchronized as a whole (the streams the workspaces were
  // made for may have been destroyed by now: their handles are not used again)
  int synced = -1;
  for (auto& kv : g_ws) {
    if (!kv.second.base) continue;
    cudaSetDevice(kv.first.first);
    if (kv.first.first != synced) {
      if (cudaDeviceSynchronize() != cudaSuccess) rc = PK_ERR_CUDA;
      synced = kv.first.first;
    }
    cudaFree(kv.second.base);
    if (kv.second.bwd) cudaFree(kv.second.bwd);
    if (kv.second.ops16) cudaFree(kv.second.ops16);
  }
  g_ws.clear();
  cudaSetDevice(cur);
  return rc;
}

}  // extern "C"

static_assert(pk::kKernelBand == PK_KERNEL_BAND && pk::kKernelF32 == PK_KERNEL_F32 && pk::kKernelTc == PK_KERNEL_TC &&
                  pk::kKernelQ4 == PK_KERNEL_Q4 && pk::kKernelTcSingle == PK_KERNEL_TC_SINGLE &&
                  pk::kKernelSplit == PK_KERNEL_SPLIT,
              "kernel ids match enum pk_kernel");
