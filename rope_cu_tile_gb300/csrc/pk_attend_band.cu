// pk_attend_band.cu -- packed RoPE attention forward for narrow windows (1 <= w <= 16), on
// the CUDA cores in fp32.
//
// What it computes: hanzo-kernel 0.2.42 packed.rs fn attend with a window: each query row
// i of a sequence sees the keys j of the same sequence with |i - j| <= w (fn attend_ref:
// abs_diff <= w), q and k rotated at their in-sequence positions, q scaled, softmax of the
// scores, out = sum p v, lse = m + ln sum exp(s - m).
//
// Why a separate kernel: with a narrow window a row sees at most 2 w + 1 keys, so the
// 128 x 128 score tiles of the tensor-core kernels are almost entirely masked (the
// short-sequence batch, w = 4, uses 9 of every 128 columns at most) and the work is bound by
// moving qkv through HBM, not by any arithmetic unit. Here every product and sum is fp32 from
// the stored values (no rounding of the rotated q and k, or of the probabilities, to the
// storage type), which also keeps fp16 inputs of large magnitude inside their tolerance.
//
// Launch: one CTA per block of 32 tokens and group of four, two or one heads (one warp per
// head: as many as let two CTAs share an SM). Every global read is an asynchronous copy into shared memory, all of a CTA's in
// flight at once: each warp's raw q, k and v rows of its head over the staged tokens
// [t0 - W, t0 + 32 + W), and the CTA's cos / sin rows of those tokens' positions. Then a
// warp rotates its k rows to fp32 (rows padded so that consecutive rows start four banks
// apart) and lane l takes query row t0 + l: q' in registers, the 2 w + 1 scores (kept in
// shared memory), the softmax, and 64 fp32 output accumulators. The sequence of every staged
// token comes from the offsets cu[s0 ..] staged once per CTA, s0 being the sequence of the
// block's first staged token; pk_band_prep_kernel (launched just before, on the same stream)
// checks cu and writes s0 for every block.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pk.h"
#include "pk_dev.cuh"

namespace pk {

namespace {

constexpr int kBandRows = 32;     // query tokens per block
constexpr int kBandCu = 96;       // staged sequence offsets per CTA
constexpr int kKStride = 68;      // floats per staged k' row (64 + 4: rows 4 banks apart)

template <typename F>
struct Store;
template <>
struct Store<float> {
  static constexpr int kVStride = 68;  // elements per staged v row
  __device__ static __forceinline__ float to_f(float x) { return x; }
};
template <>
struct Store<__nv_bfloat16> {
  static constexpr int kVStride = 72;  // 144 bytes: rows 4 banks apart
  __device__ static __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
};
template <>
struct Store<__half> {
  static constexpr int kVStride = 72;
  __device__ static __forceinline__ float to_f(__half x) { return __half2float(x); }
};

// 8 stored elements (16 bytes for 16-bit types, two 16-byte loads for fp32) as fp32
template <typename F>
__device__ __forceinline__ void load8(const F* p, float (&x)[8]) {
  if constexpr (sizeof(F) == 4) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  } else {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const F* e = reinterpret_cast<const F*>(&u);
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = Store<F>::to_f(e[k]);
  }
}

template <int OUT>
__device__ __forceinline__ void store8(void* out, int64_t at, const float (&y)[8]) {
  if constexpr (OUT == PK_F32) {
    float4* d = reinterpret_cast<float4*>(static_cast<float*>(out) + at);
    d[0] = make_float4(y[0], y[1], y[2], y[3]);
    d[1] = make_float4(y[4], y[5], y[6], y[7]);
  } else {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if constexpr (OUT == PK_BF16) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(y[2 * k], y[2 * k + 1]);
        w[k] = *reinterpret_cast<const uint32_t*>(&h);
      } else {
        const __half2 h = __floats2half2_rn(y[2 * k], y[2 * k + 1]);
        w[k] = *reinterpret_cast<const uint32_t*>(&h);
      }
    }
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + at) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// The staged member (index into off[0 .. n]) holding token a: the last i < n with off[i] <= a.
__device__ __forceinline__ int staged_member(const uint32_t* off, int n, uint32_t a) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= a)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

}  // namespace

// Checks cu (cu[0] = 0, non-decreasing, cu[S] = T; otherwise PK_ERR_BAD_CU in the status word
// and ctl->ntiles = 0, so that the band kernel writes nothing) and, for every block b of 32
// tokens, writes into `first` the sequence holding token max(0, 32 b - 16): the first
// sequence a CTA of the band kernel stages. One CTA; ctl->ntiles = 1 when cu is well formed.
__global__ void __launch_bounds__(1024) pk_band_prep_kernel(const uint32_t* __restrict__ cu, int S, long long T,
                                                            uint32_t* __restrict__ first, Ctl* ctl) {
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  griddep_launch_dependents();
  if (tid == 0) s_bad = (__ldg(cu) != 0u || static_cast<long long>(__ldg(cu + S)) != T) ? 1 : 0;
  __syncthreads();
  for (int s = tid; s < S; s += blockDim.x)
    if (__ldg(cu + s + 1) < __ldg(cu + s)) s_bad = 1;
  __syncthreads();
  if (s_bad) {
    if (tid == 0) {
      ctl->ntiles = 0;
      ctl->next = 0;
      set_status(ctl, kErrBadCu);
    }
    return;
  }
  // block b's probe token max(0, 32 b - 16) lies in exactly one non-empty sequence: the last s
  // with cu[s] <= probe (cu is small and read by every thread: L1 serves the searches)
  const long long nb = (T + kBandRows - 1) / kBandRows;
  for (long long b = tid; b < nb; b += blockDim.x) {
    const uint32_t probe = static_cast<uint32_t>(b == 0 ? 0 : kBandRows * b - 16);
    first[b] = seq_of_token(cu, 0u, static_cast<uint32_t>(S), probe);
  }
  if (tid == 0) {
    ctl->ntiles = 1;
    ctl->next = 0;
  }
}

// 16-byte asynchronous copy global -> shared (through L1: table rows repeat across tokens)
__device__ __forceinline__ void band_cp16(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

// Shared-memory layout of a CTA (W: the instance's largest window; rows: 32 + 2 W staged
// tokens; VS: elements per staged 16-bit or fp32 row, padded so rows start 4 banks apart):
//   k'   [4][rows][68] fp32        rotated keys
//   v    [4][rows][VS] stored      values
//   q    [4][32][VS]   stored      raw queries (then the scores [4][2 W + 1][32] fp32)
//   kraw [4][rows][VS] stored      raw keys
//   tab  [rows][2][32] stored      cos and sin rows of each staged token's position
template <typename F, int W>
struct BandSmem {
  static constexpr int kRows = kBandRows + 2 * W;
  static constexpr int kVS = Store<F>::kVStride;
  // bytes of one head's rows (k', v, q, raw k) and of the CTA's table rows
  static constexpr size_t kPerHead = sizeof(float) * kRows * kKStride + sizeof(F) * kRows * kVS +
                                     sizeof(F) * kBandRows * kVS + sizeof(F) * kRows * kVS;
  static constexpr size_t kTabBytes = sizeof(F) * kRows * 2 * kHalf;
  // heads per CTA (one warp each): four, two or one, whichever lets two CTAs share an SM
  static constexpr size_t kTwoPerSm = 113 * 1024;
  static constexpr int kHeads = 4 * kPerHead + kTabBytes <= kTwoPerSm ? 4 : 2 * kPerHead + kTabBytes <= kTwoPerSm ? 2 : 1;
  static constexpr size_t kK = 0;
  static constexpr size_t kV = kK + sizeof(float) * kHeads * kRows * kKStride;
  static constexpr size_t kQ = kV + sizeof(F) * kHeads * kRows * kVS;
  static constexpr size_t kKraw = kQ + sizeof(F) * kHeads * kBandRows * kVS;
  static constexpr size_t kTab = kKraw + sizeof(F) * kHeads * kRows * kVS;
  static constexpr size_t kBytes = kTab + kTabBytes;
  static_assert(kBytes <= 227 * 1024, "fits the shared memory a block may use");
  static_assert(sizeof(float) * (2 * W + 1) * 32 <= sizeof(F) * kBandRows * kVS, "scores fit the q area");
};

// W: the largest window this instance serves (4, 8 or 16); the call's window is 1 .. W.
template <typename F, int OUT, int W>
__global__ void __launch_bounds__(kBandRows * BandSmem<F, W>::kHeads)
pk_attend_band_kernel(const F* __restrict__ qkv, const F* __restrict__ cos_t, const F* __restrict__ sin_t,
                      const uint32_t* __restrict__ cu, int S, const uint32_t* __restrict__ first,
                      void* __restrict__ out, float* __restrict__ lse, const Ctl* ctl, int H, long long T,
                      int window, float scale) {
  using L = BandSmem<F, W>;
  constexpr int kRowsSt = L::kRows;
  constexpr int kVS = L::kVS;
  constexpr int kChunk = 16 / sizeof(F);          // elements per 16-byte chunk
  constexpr int kRowChunks = kD / kChunk;         // chunks per 64-element row
  constexpr int kTabChunks = kHalf / kChunk;      // chunks per 32-element table row
  extern __shared__ __align__(16) unsigned char band_smem[];
  auto s_k = reinterpret_cast<float (*)[kRowsSt][kKStride]>(band_smem + L::kK);
  auto s_v = reinterpret_cast<F (*)[kRowsSt][kVS]>(band_smem + L::kV);
  auto s_q = reinterpret_cast<F (*)[kBandRows][kVS]>(band_smem + L::kQ);
  auto s_kr = reinterpret_cast<F (*)[kRowsSt][kVS]>(band_smem + L::kKraw);
  auto s_tab = reinterpret_cast<F (*)[2][kHalf]>(band_smem + L::kTab);
  __shared__ uint32_t s_cu[kBandCu + 1];
  __shared__ int s_ncu;
  __shared__ int s_seq_lo[kRowsSt], s_seq_hi[kRowsSt];  // sequence [start, end) of each staged token

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const long long b = blockIdx.x;
  const long long t0 = b * kBandRows;
  const long long base = t0 - W;  // token of staged row 0
  const int h = blockIdx.y * L::kHeads + warp;
  const int64_t ldq = 3ll * H * kD;
  // the offsets were checked (and `first` written) by the kernel launched just before
  griddep_wait();
  if (__ldcg(&ctl->ntiles) == 0u) return;

  // raw q, k and v rows of this warp's head: asynchronous copies, all in flight at once
  if (h < H) {
    for (int i = lane; i < kRowsSt * kRowChunks; i += 32) {
      const int r = i / kRowChunks, c = i % kRowChunks;
      const long long a = base + r;
      F* kd = s_kr[warp][r] + c * kChunk;
      F* vd = s_v[warp][r] + c * kChunk;
      if (a >= 0 && a < T) {
        const F* row = qkv + a * ldq;
        band_cp16(kd, row + static_cast<int64_t>(H + h) * kD + c * kChunk);
        band_cp16(vd, row + static_cast<int64_t>(2 * H + h) * kD + c * kChunk);
      } else {
        *reinterpret_cast<uint4*>(kd) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(vd) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    for (int i = lane; i < kBandRows * kRowChunks; i += 32) {
      const int r = i / kRowChunks, c = i % kRowChunks;
      const long long a = t0 + r;
      F* qd = s_q[warp][r] + c * kChunk;
      if (a < T)
        band_cp16(qd, qkv + a * ldq + static_cast<int64_t>(h) * kD + c * kChunk);
      else
        *reinterpret_cast<uint4*>(qd) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  // stage cu[s0 .. s0 + kBandCu] (the block's staged tokens start in sequence s0)
  const uint32_t s0 = __ldg(first + b);
  for (int i = tid; i <= kBandCu; i += blockDim.x)
    s_cu[i] = s0 + i <= static_cast<uint32_t>(S) ? __ldg(cu + s0 + i) : 0xFFFFFFFFu;
  if (tid == 0) s_ncu = min(kBandCu, S - static_cast<int>(s0));
  __syncthreads();
  // the sequence bounds of every staged token (from the staged offsets when they reach it)
  for (int r = tid; r < kRowsSt; r += blockDim.x) {
    const long long a = base + r;
    int lo = 0, hi = 0;
    if (a >= 0 && a < T) {
      const int n = s_ncu;
      if (static_cast<long long>(s_cu[n]) > a) {
        const int i = staged_member(s_cu, n, static_cast<uint32_t>(a));
        lo = static_cast<int>(s_cu[i]);
        hi = static_cast<int>(s_cu[i + 1]);
      } else {
        const uint32_t sq = seq_of_token(cu, s0, static_cast<uint32_t>(S) - s0, static_cast<uint32_t>(a));
        lo = static_cast<int>(__ldg(cu + sq));
        hi = static_cast<int>(__ldg(cu + sq + 1));
      }
    }
    s_seq_lo[r] = lo;
    s_seq_hi[r] = hi;
  }
  __syncthreads();
  // the cos and sin rows of every staged token's position
  for (int i = tid; i < kRowsSt * 2 * kTabChunks; i += blockDim.x) {
    const int r = i / (2 * kTabChunks), rest = i % (2 * kTabChunks);
    const int which = rest / kTabChunks, c = rest % kTabChunks;
    const long long a = base + r;
    if (a >= 0 && a < T) {
      const int64_t pos = a - s_seq_lo[r];
      band_cp16(&s_tab[r][which][c * kChunk], (which ? sin_t : cos_t) + pos * kHalf + c * kChunk);
    } else {
      *reinterpret_cast<uint4*>(&s_tab[r][which][c * kChunk]) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  if (h >= H) return;

  // k' = rot(k) in fp32: four lanes per row, lane chunk c < 4 holding elements 8 c .. 8 c + 7
  // of each half (the rotary pairs (u, u + 32))
  for (int i = lane; i < kRowsSt * 4; i += 32) {
    const int r = i >> 2, c = i & 3;
    const F* kr = s_kr[warp][r];
    const F* tc = s_tab[r][0];
    const F* ts = s_tab[r][1];
    float* kd = s_k[warp][r];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int u = 8 * c + e;
      const float x1 = Store<F>::to_f(kr[u]), x2 = Store<F>::to_f(kr[u + kHalf]);
      const float cc = Store<F>::to_f(tc[u]), ss = Store<F>::to_f(ts[u]);
      kd[u] = x1 * cc - x2 * ss;
      kd[u + kHalf] = x1 * ss + x2 * cc;
    }
  }
  // this lane's query row: q' = rot(q, pos) * scale in fp32
  const long long a = t0 + lane;
  const bool row_ok = a < T;
  float q[kD];
  int lo = 0, hi = 0;
  {
    const int r = lane + W;
    const F* qr = s_q[warp][lane];
    const F* tc = s_tab[r][0];
    const F* ts = s_tab[r][1];
#pragma unroll
    for (int u = 0; u < kHalf; ++u) {
      const float x1 = Store<F>::to_f(qr[u]), x2 = Store<F>::to_f(qr[u + kHalf]);
      const float cc = Store<F>::to_f(tc[u]), ss = Store<F>::to_f(ts[u]);
      q[u] = (x1 * cc - x2 * ss) * scale;
      q[u + kHalf] = (x1 * ss + x2 * cc) * scale;
    }
    if (row_ok) {
      lo = max(s_seq_lo[r], static_cast<int>(a) - window);
      hi = min(s_seq_hi[r], static_cast<int>(a) + window + 1);
    }
  }
  __syncwarp();

  // scores of the keys a - W .. a + W (staged rows lane .. lane + 2 W), kept per lane in shared
  // memory; invisible ones -inf. The key loops stay rolled (a small register footprint).
  // (the raw q rows are read: their area holds the scores now)
  float* sc = reinterpret_cast<float*>(s_q[warp]) + lane;  // score d of this lane at sc[32 d]
  float m = -INFINITY;
#pragma unroll 1
  for (int d = 0; d <= 2 * W; ++d) {
    const long long j = a - W + d;
    const float* kr = s_k[warp][lane + d];
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int u = 0; u < kD; u += 8) {
      const float4 x = *reinterpret_cast<const float4*>(kr + u);
      const float4 y = *reinterpret_cast<const float4*>(kr + u + 4);
      acc0 = fmaf(q[u], x.x, acc0);
      acc1 = fmaf(q[u + 1], x.y, acc1);
      acc0 = fmaf(q[u + 2], x.z, acc0);
      acc1 = fmaf(q[u + 3], x.w, acc1);
      acc0 = fmaf(q[u + 4], y.x, acc0);
      acc1 = fmaf(q[u + 5], y.y, acc1);
      acc0 = fmaf(q[u + 6], y.z, acc0);
      acc1 = fmaf(q[u + 7], y.w, acc1);
    }
    const float sv = (j >= lo && j < hi) ? acc0 + acc1 : -INFINITY;
    sc[32 * d] = sv;
    m = fmaxf(m, sv);
  }
  // softmax weights (a row past T has none) and the weighted sum of the visible values
  float l = 0.f;
  float o[kD];
#pragma unroll
  for (int u = 0; u < kD; ++u) o[u] = 0.f;
#pragma unroll 1
  for (int d = 0; d <= 2 * W; ++d) {
    const float p = row_ok ? __expf(sc[32 * d] - m) : 0.f;
    l += p;
    const F* vr = s_v[warp][lane + d];
#pragma unroll
    for (int u = 0; u < kD; u += 8) {
      float x[8];
      if constexpr (sizeof(F) == 4) {
        const float4 a4 = *reinterpret_cast<const float4*>(vr + u);
        const float4 b4 = *reinterpret_cast<const float4*>(vr + u + 4);
        x[0] = a4.x; x[1] = a4.y; x[2] = a4.z; x[3] = a4.w;
        x[4] = b4.x; x[5] = b4.y; x[6] = b4.z; x[7] = b4.w;
      } else {
        const uint4 w4 = *reinterpret_cast<const uint4*>(vr + u);
        const F* e = reinterpret_cast<const F*>(&w4);
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = Store<F>::to_f(e[k]);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) o[u + k] = fmaf(p, x[k], o[u + k]);
    }
  }
  if (row_ok) {
    const float inv = 1.0f / l;
    const int64_t at = a * static_cast<int64_t>(H) * kD + static_cast<int64_t>(h) * kD;
#pragma unroll
    for (int u = 0; u < kD; u += 8) {
      float y[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) y[k] = o[u + k] * inv;
      store8<OUT>(out, at + u, y);
    }
    lse[static_cast<int64_t>(h) * T + a] = m + logf(l);
  }
}

namespace {

template <typename F, int W>
constexpr size_t band_smem_bytes() {
  return BandSmem<F, W>::kBytes;
}

template <typename F, int OUT, int W>
cudaError_t band_attr() {
  return cudaFuncSetAttribute(pk_attend_band_kernel<F, OUT, W>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(band_smem_bytes<F, W>()));
}

template <typename F, int OUT>
cudaError_t band_attrs() {
  cudaError_t e = band_attr<F, OUT, 4>();
  if (e == cudaSuccess) e = band_attr<F, OUT, 8>();
  if (e == cudaSuccess) e = band_attr<F, OUT, 16>();
  return e;
}

template <typename F, int OUT>
cudaError_t band_launch_w(const void* qkv, const void* cos_t, const void* sin_t, const uint32_t* cu, int S,
                          const uint32_t* first, void* out, float* lse, const Ctl* ctl, int H, long long T, int window,
                          float scale, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((T + kBandRows - 1) / kBandRows));
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const F* q = static_cast<const F*>(qkv);
  const F* c = static_cast<const F*>(cos_t);
  const F* s = static_cast<const F*>(sin_t);
  auto shape = [&](int heads) {
    cfg.gridDim.y = static_cast<unsigned>((H + heads - 1) / heads);
    cfg.blockDim = dim3(kBandRows * heads);
  };
  if (window <= 4) {
    shape(BandSmem<F, 4>::kHeads);
    cfg.dynamicSmemBytes = band_smem_bytes<F, 4>();
    return cudaLaunchKernelEx(&cfg, pk_attend_band_kernel<F, OUT, 4>, q, c, s, cu, S, first, out, lse, ctl, H, T,
                              window, scale);
  }
  if (window <= 8) {
    shape(BandSmem<F, 8>::kHeads);
    cfg.dynamicSmemBytes = band_smem_bytes<F, 8>();
    return cudaLaunchKernelEx(&cfg, pk_attend_band_kernel<F, OUT, 8>, q, c, s, cu, S, first, out, lse, ctl, H, T,
                              window, scale);
  }
  shape(BandSmem<F, 16>::kHeads);
  cfg.dynamicSmemBytes = band_smem_bytes<F, 16>();
  return cudaLaunchKernelEx(&cfg, pk_attend_band_kernel<F, OUT, 16>, q, c, s, cu, S, first, out, lse, ctl, H, T,
                            window, scale);
}

}  // namespace

// Host side: opt in to the dynamic shared memory of every instance once per device.
cudaError_t band_prepare() {
  cudaError_t e = band_attrs<__nv_bfloat16, PK_BF16>();
  if (e == cudaSuccess) e = band_attrs<__half, PK_F16>();
  if (e == cudaSuccess) e = band_attrs<float, PK_F32>();
  if (e == cudaSuccess) e = band_attrs<float, PK_BF16>();
  if (e == cudaSuccess) e = band_attrs<float, PK_F16>();
  return e;
}

// Records needed in `first` (uint32 each) for T tokens.
long long band_first_words(long long T) { return (T + kBandRows - 1) / kBandRows; }

// The two launches of a narrow-window call, on `stream`: band_prep_launch (the offsets check,
// which also writes `first`), then band_launch (the attention kernel). dtype: the storage type of qkv and the tables;
// out_dtype: the output's type (the same, or a 16-bit type for fp32 inputs). 1 <= window <= 16.
cudaError_t band_prep_launch(const uint32_t* cu, int S, long long T, uint32_t* first, Ctl* ctl, cudaStream_t stream) {
  pk_band_prep_kernel<<<1, 1024, 0, stream>>>(cu, S, T, first, ctl);
  return cudaGetLastError();
}

cudaError_t band_launch(int dtype, int out_dtype, const void* qkv, const void* cos_t, const void* sin_t,
                        const uint32_t* cu, int S, uint32_t* first, void* out, float* lse, Ctl* ctl, int H, long long T,
                        int window, float scale, cudaStream_t stream) {
  if (dtype == PK_BF16) return band_launch_w<__nv_bfloat16, PK_BF16>(qkv, cos_t, sin_t, cu, S, first, out, lse, ctl, H, T, window, scale, stream);
  if (dtype == PK_F16) return band_launch_w<__half, PK_F16>(qkv, cos_t, sin_t, cu, S, first, out, lse, ctl, H, T, window, scale, stream);
  if (out_dtype == PK_BF16) return band_launch_w<float, PK_BF16>(qkv, cos_t, sin_t, cu, S, first, out, lse, ctl, H, T, window, scale, stream);
  if (out_dtype == PK_F16) return band_launch_w<float, PK_F16>(qkv, cos_t, sin_t, cu, S, first, out, lse, ctl, H, T, window, scale, stream);
  return band_launch_w<float, PK_F32>(qkv, cos_t, sin_t, cu, S, first, out, lse, ctl, H, T, window, scale, stream);
}

}  // namespace pk
