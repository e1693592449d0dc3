// pk_rope.cu -- the standalone rotary embedding of a packed qkv (pk_rope in include/pk.h).
//
// The pages' rope op (hanzo-kernel fast ops, `FastOp::Rope` and its graph fallback): the first
// `dims` features of a head vector are rotated in pairs -- the two halves (j, j + dims/2), or
// interleaved pairs (2j, 2j + 1) ("traditional") -- by the angle of pair j at the vector's
// position, forwards or inversely (the transposed rotation, the gradient); features past
// `dims` are unchanged. As kime's rope step does for a packed qkv, it is applied here to every q
// and k head vector of qkv [T, 3 H 64], the position of a token being its index in its
// sequence (cu); v is copied when the output is not the input. Tables cos/sin [P, dims/2] hold
// the angles' cosines and sines in the element type.
//
// Layout of the work: one warp per token (a contiguous run of tokens per warp, so a sequence
// is found once by a 32-way search and then followed). Lane l holds features 2l and 2l + 1 of
// a head vector (one 4-byte word in 16 bits, 8 bytes in fp32), so a head vector is one
// coalesced 128- or 256-byte access; the partner of a feature sits in another lane (halves) or
// the same lane (interleaved pairs) and comes by shuffle. Head vectors are processed twelve at a
// time so that several loads are in flight per warp; the grid is one wave of resident blocks. Arithmetic in fp32, one rounding to the
// element type.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pk.h"
#include "pk_dev.cuh"

namespace pk {

namespace {

constexpr int kRopeThreads = 256;
constexpr int kRopeBatch = 12;  // head vectors in flight per warp (measured best of 4 to 24)

// two elements of one lane as floats, and back
template <int DT>
struct Pair2;
template <>
struct Pair2<PK_F32> {
  using Word = float2;
  static __device__ __forceinline__ float2 widen(Word w) { return w; }
  static __device__ __forceinline__ Word narrow(float2 v) { return v; }
  static __device__ __forceinline__ float one(const void* t, int64_t i) { return static_cast<const float*>(t)[i]; }
};
template <>
struct Pair2<PK_BF16> {
  using Word = uint32_t;
  static __device__ __forceinline__ float2 widen(Word w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  static __device__ __forceinline__ Word narrow(float2 v) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v.x))) |
           (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v.y))) << 16);
  }
  static __device__ __forceinline__ float one(const void* t, int64_t i) {
    return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(t)[i]) << 16);
  }
};
template <>
struct Pair2<PK_F16> {
  using Word = uint32_t;
  static __device__ __forceinline__ float2 widen(Word w) {
    return make_float2(__half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu))),
                       __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16))));
  }
  static __device__ __forceinline__ Word narrow(float2 v) {
    return static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v.x))) |
           (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v.y))) << 16);
  }
  static __device__ __forceinline__ float one(const void* t, int64_t i) {
    return __half2float(static_cast<const __half*>(t)[i]);
  }
};

// The role of feature f in the rotation: its pair j, and its partner feature p (f itself when f
// is not rotated); `first` is true for the pair's first member (a), false for the second (b).
struct Role {
  int j, p;
  bool rot, first;
};
__device__ __forceinline__ Role role_of(int f, int dims, bool traditional) {
  Role r;
  const int h = dims >> 1;
  r.rot = f < dims;
  if (!r.rot) {
    r.j = 0;
    r.p = f;
    r.first = true;
  } else if (traditional) {
    r.j = f >> 1;
    r.p = f ^ 1;
    r.first = (f & 1) == 0;
  } else {
    r.first = f < h;
    r.j = r.first ? f : f - h;
    r.p = r.first ? f + h : f - h;
  }
  return r;
}

struct RopeArgs {
  const void* x;
  void* y;
  const void* cos_t;
  const void* sin_t;
  long long P;
  const uint32_t* cu;
  int S;
  long long T;
  int H;
  int dims;
  int traditional;
  int inverse;
  int copy_v;
  int* status;
};

__device__ __forceinline__ void flag(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// At most 64 registers a thread, so that four blocks are resident per SM: the kernel is bound by
// the bytes in flight per SM.
template <int DT>
__global__ void __launch_bounds__(kRopeThreads, 4) pk_rope_kernel(const RopeArgs a) {
  using P2 = Pair2<DT>;
  using Word = typename P2::Word;
  const int lane = threadIdx.x & 31;
  const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  if (gw == 0 && lane == 0 && (__ldg(a.cu) != 0u || static_cast<long long>(__ldg(a.cu + a.S)) != a.T))
    flag(a.status, kErrBadCu);
  const long long per = (a.T + nw - 1) / nw;
  const long long t0 = gw * per, t1 = min(a.T, t0 + per);
  if (t0 >= t1) return;

  // this lane's two features and their roles (fixed for the call)
  const bool trad = a.traditional != 0;
  const Role r0 = role_of(2 * lane, a.dims, trad), r1 = role_of(2 * lane + 1, a.dims, trad);
  const int h = a.dims >> 1;
  // sign of the partner term: y = x c + sign * partner * s
  const float g0 = (a.inverse != 0) == r0.first ? 1.f : -1.f;
  const float g1 = (a.inverse != 0) == r1.first ? 1.f : -1.f;

  // the sequence holding t0: the last s < S with cu[s] <= t0, by a 32-way search
  uint32_t lo = 0, hi = static_cast<uint32_t>(a.S);  // answer + 1 in (lo, hi]: first s with cu[s] > t0
  while (lo < hi) {
    const uint32_t step = (hi - lo + 31) / 32;
    const unsigned long long e = static_cast<unsigned long long>(lo) + static_cast<unsigned long long>(lane + 1) * step;
    const uint32_t q = static_cast<uint32_t>(min(e, static_cast<unsigned long long>(hi))) - 1;
    const bool pred = static_cast<unsigned long long>(lo) + static_cast<unsigned long long>(lane) * step < hi &&
                      static_cast<long long>(__ldg(a.cu + q)) > t0;
    const unsigned int m = __ballot_sync(0xffffffffu, pred);
    if (m == 0u) {
      lo = hi;
      break;
    }
    const uint32_t k = static_cast<uint32_t>(__ffs(m) - 1);
    const uint32_t qk = static_cast<uint32_t>(
        min(static_cast<unsigned long long>(lo) + static_cast<unsigned long long>(k + 1) * step,
            static_cast<unsigned long long>(hi))) - 1;
    lo += k * step;
    hi = qk;
  }
  // lo = first s with cu[s] > t0 (or S); the token's sequence is lo - 1
  uint32_t s = lo > 0 ? lo - 1 : 0;
  long long start = __ldg(a.cu + s), end = __ldg(a.cu + s + 1);

  const long long W = 3LL * a.H * kD;
  const int nqk = 2 * a.H;
  for (long long t = t0; t < t1; ++t) {
    while (t >= end && s + 1 < static_cast<uint32_t>(a.S)) {
      ++s;
      start = end;
      end = __ldg(a.cu + s + 1);
    }
    const long long pos = t - start;
    if (t >= end || pos < 0 || pos >= a.P) {
      if (lane == 0) flag(a.status, kErrBadCu);
      continue;
    }
    // this token's table entries for the lane's two pairs
    float c0 = 1.f, s0 = 0.f, c1 = 1.f, s1 = 0.f;
    if (r0.rot) {
      c0 = P2::one(a.cos_t, pos * h + r0.j);
      s0 = g0 * P2::one(a.sin_t, pos * h + r0.j);
    }
    if (r1.rot) {
      c1 = P2::one(a.cos_t, pos * h + r1.j);
      s1 = g1 * P2::one(a.sin_t, pos * h + r1.j);
    }
    const Word* xr = reinterpret_cast<const Word*>(static_cast<const char*>(a.x) + t * W * (DT == PK_F32 ? 4 : 2));
    Word* yr = reinterpret_cast<Word*>(static_cast<char*>(a.y) + t * W * (DT == PK_F32 ? 4 : 2));
    // q and k head vectors: word `lane` of vector v sits at v * 32 + lane
    for (int v0 = 0; v0 < nqk; v0 += kRopeBatch) {
      Word w[kRopeBatch];
#pragma unroll
      for (int b = 0; b < kRopeBatch; ++b)
        if (v0 + b < nqk) w[b] = xr[(v0 + b) * 32 + lane];
#pragma unroll
      for (int b = 0; b < kRopeBatch; ++b) {
        if (v0 + b >= nqk) break;  // (uniform across the warp)
        const float2 xv = P2::widen(w[b]);
        // the partners' values: both features of the partner lanes, then the right one
        const float a0 = __shfl_sync(0xffffffffu, xv.x, r0.p >> 1), b0 = __shfl_sync(0xffffffffu, xv.y, r0.p >> 1);
        const float a1 = __shfl_sync(0xffffffffu, xv.x, r1.p >> 1), b1 = __shfl_sync(0xffffffffu, xv.y, r1.p >> 1);
        const float p0 = (r0.p & 1) ? b0 : a0, p1 = (r1.p & 1) ? b1 : a1;
        float2 out;
        out.x = r0.rot ? fmaf(xv.x, c0, p0 * s0) : xv.x;
        out.y = r1.rot ? fmaf(xv.y, c1, p1 * s1) : xv.y;
        yr[(v0 + b) * 32 + lane] = P2::narrow(out);
      }
    }
    if (a.copy_v)
      for (int v0 = nqk; v0 < 3 * a.H; v0 += kRopeBatch) {
        Word w[kRopeBatch];
#pragma unroll
        for (int b = 0; b < kRopeBatch; ++b)
          if (v0 + b < 3 * a.H) w[b] = xr[(v0 + b) * 32 + lane];
#pragma unroll
        for (int b = 0; b < kRopeBatch; ++b)
          if (v0 + b < 3 * a.H) yr[(v0 + b) * 32 + lane] = w[b];
      }
  }
}

template <int DT>
cudaError_t launch_rope(const RopeArgs& a, int sms, cudaStream_t stream) {
  // one wave: as many blocks as are resident at once (each warp then takes a longer run of
  // tokens), never more warps than tokens
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pk_rope_kernel<DT>, kRopeThreads, 0);
  if (e != cudaSuccess) return e;
  const long long warps_needed = a.T;
  const long long blocks = min(static_cast<long long>(sms) * max(per_sm, 1), (warps_needed + 7) / 8);
  pk_rope_kernel<DT><<<static_cast<unsigned int>(blocks > 0 ? blocks : 1), kRopeThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

bool aligned_to(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; }

}  // namespace

}  // namespace pk

extern "C" int pk_rope(int dtype, const void* x, void* y, const void* cos, const void* sin, int64_t P,
                       const uint32_t* cu, int S, int64_t T, int H, int dims, int traditional, int inverse,
                       int* status, struct CUstream_st* stream) {
  using namespace pk;
  if (dtype != PK_F32 && dtype != PK_BF16 && dtype != PK_F16) return PK_ERR_ARG;
  if (S < 0 || T < 0 || T > PK_MAX_T || H < 1 || H > PK_MAX_H) return PK_ERR_ARG;
  if (dims < 2 || dims > kD || (dims & 1)) return PK_ERR_ARG;
  if (S == 0 && T != 0) return PK_ERR_ARG;
  cudaStream_t st = stream;
  if (T == 0) {
    if (status && cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return PK_ERR_CUDA;
    return PK_OK;
  }
  if (!x || !y || !cos || !sin || !cu || P < 1) return PK_ERR_ARG;
  const uintptr_t word = dtype == PK_F32 ? 8 : 4, elem = dtype == PK_F32 ? 4 : 2;
  if (!aligned_to(x, word) || !aligned_to(y, word) || !aligned_to(cos, elem) || !aligned_to(sin, elem) ||
      !aligned_to(cu, 4) || (status && !aligned_to(status, 4)))
    return PK_ERR_ALIGN;
  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PK_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PK_ERR_CUDA;
  if (major != 10 || minor != 3) return PK_ERR_UNSUPPORTED;
  if (status && cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return PK_ERR_CUDA;
  RopeArgs a{x, y, cos, sin, static_cast<long long>(P), cu, S, static_cast<long long>(T), H, dims,
             traditional ? 1 : 0, inverse ? 1 : 0, x != y ? 1 : 0, status};
  cudaError_t e;
  if (dtype == PK_F32)
    e = launch_rope<PK_F32>(a, sms, st);
  else if (dtype == PK_BF16)
    e = launch_rope<PK_BF16>(a, sms, st);
  else
    e = launch_rope<PK_F16>(a, sms, st);
  return e == cudaSuccess ? PK_OK : PK_ERR_CUDA;
}
