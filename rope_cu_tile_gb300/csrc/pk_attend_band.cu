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
// head: as many as let two CTAs share an SM). Every global read is in flight at once: each
// warp's raw k and v rows of its head over the staged tokens [t0 - W, t0 + 32 + W) and the
// CTA's cos / sin rows of those tokens' positions as asynchronous copies into shared memory,
// and each lane's own q features of its first rows straight into registers (q needs no
// staging: a lane reads only its own rows and features, once). A warp then rotates its k rows to fp32 in place and computes its 32 query rows in
// register tiles (R rows x 16 features a lane, so that each key and value granule it loads
// serves up to R rows; see the kernel). The sequence of every staged token comes from the
// offsets cu[s0 ..] staged once per CTA, s0 being the sequence of the block's first staged
// token; pk_band_prep_kernel (launched just before, on the same stream) checks cu and writes s0
// for every block.
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
  __device__ static __forceinline__ float to_f(float x) { return x; }
};
template <>
struct Store<__nv_bfloat16> {
  __device__ static __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
};
template <>
struct Store<__half> {
  __device__ static __forceinline__ float to_f(__half x) { return __half2float(x); }
};

template <int OUT>
__device__ __forceinline__ void store4(void* out, int64_t at, float y0, float y1, float y2, float y3) {
  if constexpr (OUT == PK_F32) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + at) = make_float4(y0, y1, y2, y3);
  } else if constexpr (OUT == PK_BF16) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(y0, y1), b = __floats2bfloat162_rn(y2, y3);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + at) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
  } else {
    const __half2 a = __floats2half2_rn(y0, y1), b = __floats2half2_rn(y2, y3);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + at) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
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
// tokens; heads: one warp each):
//   k'  [heads][rows][68] fp32     rotated keys (a 68-float row starts four banks after the
//                                  one before); the raw 16-bit row is copied into its last 128
//                                  bytes (byte 144 on) and rotated in place
//   v   [heads][rows][VS] stored   values as stored (VS: 72 16-bit or 68 fp32 elements)
//   tab [rows][2][32]     stored   cos and sin rows of each staged token's position
template <typename F, int W>
struct BandSmem {
  static constexpr int kRows = kBandRows + 2 * W;
  static constexpr int kVS = sizeof(F) == 4 ? 68 : 72;
  static constexpr size_t kRowBytes = sizeof(float) * kKStride;  // 272
  static constexpr size_t kRawAt = sizeof(F) == 4 ? 0 : 144;     // raw 16-bit k row inside its fp32 row
  static constexpr size_t kPerHead = kRows * kRowBytes + sizeof(F) * kRows * kVS;
  static constexpr size_t kTabBytes = sizeof(F) * kRows * 2 * kHalf;
  // heads per CTA (one warp each): four, two or one, whichever lets two CTAs share an SM
  static constexpr size_t kTwoPerSm = 113 * 1024;
  static constexpr int kHeads = 4 * kPerHead + kTabBytes <= kTwoPerSm ? 4 : 2 * kPerHead + kTabBytes <= kTwoPerSm ? 2 : 1;
  static constexpr size_t kK = 0;
  static constexpr size_t kV = kK + kHeads * kRows * kRowBytes;
  static constexpr size_t kTab = kV + sizeof(F) * kHeads * kRows * kVS;
  static constexpr size_t kBytes = kTab + kTabBytes;
  static_assert(kBytes <= 227 * 1024, "fits the shared memory a block may use");
  static_assert(kRawAt + 128 <= kRowBytes, "a raw 16-bit row fits inside its fp32 row");
};

// 8 stored elements (16 bytes of a 16-bit type, 32 bytes of fp32) from shared memory, as fp32
template <typename F>
__device__ __forceinline__ void lds8(const F* p, float (&x)[8]) {
  if constexpr (sizeof(F) == 4) {
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  } else {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const F* e = reinterpret_cast<const F*>(&u);
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = Store<F>::to_f(e[k]);
  }
}
// 4 stored elements (8 bytes of a 16-bit type, 16 bytes of fp32) from shared memory, as fp32
template <typename F>
__device__ __forceinline__ void lds4(const F* p, float (&x)[4]) {
  if constexpr (sizeof(F) == 4) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  } else {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const F* e = reinterpret_cast<const F*>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) x[k] = Store<F>::to_f(e[k]);
  }
}
// 4 consecutive stored elements (one feature granule) in registers: 8 bytes of a 16-bit type,
// 16 of fp32; read from global memory and widened to fp32
template <typename F>
struct Granule {
  using type = uint2;
  __device__ static __forceinline__ type load(const F* p) { return __ldg(reinterpret_cast<const uint2*>(p)); }
  __device__ static __forceinline__ type zero() { return make_uint2(0u, 0u); }
  __device__ static __forceinline__ void widen(const type& g, float (&x)[4]) {
    const F* e = reinterpret_cast<const F*>(&g);
#pragma unroll
    for (int k = 0; k < 4; ++k) x[k] = Store<F>::to_f(e[k]);
  }
};
template <>
struct Granule<float> {
  using type = float4;
  __device__ static __forceinline__ type load(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
  __device__ static __forceinline__ type zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ static __forceinline__ void widen(const type& g, float (&x)[4]) {
    x[0] = g.x; x[1] = g.y; x[2] = g.z; x[3] = g.w;
  }
};

__device__ __forceinline__ void sts8(float* p, const float (&y)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(y[0], y[1], y[2], y[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(y[4], y[5], y[6], y[7]);
}

// W: the largest window this instance serves (4, 8 or 16); the call's window is 1 .. W.
//
// The products: lane (g, e) of a warp, g = lane / 4, e = lane % 4, takes R consecutive query
// rows of its block (R = 4 for W <= 4, else 2; 8 R rows per pass) and 16 of the 64 features:
// the 4-feature granules e, e + 4, e + 8, e + 12, which hold both members of their rotary
// pairs (u, u + 32). Each key row it loads serves up to R of its rows: the partial scores
// of its features are summed over the four lanes of the group (with R = 4 by two exchange
// rounds that leave lane e the whole scores of row e, whose softmax it takes alone before
// the weights are shared again; otherwise by two shuffles of every sum), and its share of
// out accumulates from the value granules of the same features.
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
  constexpr int R = W <= 4 ? 4 : 2;               // query rows per lane
  constexpr int kKeys = R + 2 * W;                // key rows a lane's group reads
  extern __shared__ __align__(16) unsigned char band_smem[];
  auto s_k = reinterpret_cast<float (*)[kRowsSt][kKStride]>(band_smem + L::kK);
  auto s_v = reinterpret_cast<F (*)[kRowsSt][kVS]>(band_smem + L::kV);
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
  auto raw_k = [&](int r) { return reinterpret_cast<F*>(reinterpret_cast<unsigned char*>(s_k[warp][r]) + L::kRawAt); };
  // the offsets were checked (and `first` written) by the kernel launched just before
  griddep_wait();
  if (__ldcg(&ctl->ntiles) == 0u) return;

  // raw q, k and v rows of this warp's head: asynchronous copies, all in flight at once
  if (h < H) {
    for (int i = lane; i < kRowsSt * kRowChunks; i += 32) {
      const int r = i / kRowChunks, c = i % kRowChunks;
      const long long a = base + r;
      F* kd = raw_k(r) + c * kChunk;
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
  }
  // this lane's raw q granules (e, e + 4, e + 8, e + 12) of the R rows it takes first, into
  // registers while the copies are in flight
  const int g = lane >> 2, e = lane & 3;
  // scores in base-2 units: q' carries scale * log2(e), so each weight is one ex2
  const float sl2 = scale * 1.4426950408889634f;
  using QG = Granule<F>;
  typename QG::type qraw[R][4];
  auto load_q = [&](int rb) {
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const long long a = t0 + rb + i;
#pragma unroll
      for (int gi = 0; gi < 4; ++gi)
        qraw[i][gi] = (h < H && a < T) ? QG::load(qkv + a * ldq + static_cast<int64_t>(h) * kD + 4 * (e + 4 * gi))
                                       : QG::zero();
    }
  };
  load_q(R * g);
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

  // k' = rot(k) in fp32, in place: a row's raw elements are all read (by the four lanes that
  // share it: chunk pair c < 4 holds elements 8 c .. 8 c + 7 of each half) before any of its
  // fp32 values are written
#pragma unroll 1
  for (int r0 = 0; r0 < kRowsSt; r0 += 8) {
    const int r = r0 + (lane >> 2), c = lane & 3;
    float x1[8], x2[8], tc[8], ts[8];
    const bool in = r < kRowsSt;
    if (in) {
      lds8(raw_k(r) + 8 * c, x1);
      lds8(raw_k(r) + 8 * c + kHalf, x2);
      lds8(&s_tab[r][0][8 * c], tc);
      lds8(&s_tab[r][1][8 * c], ts);
    }
    __syncwarp();
    if (in) {
      float y1[8], y2[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        y1[k] = x1[k] * tc[k] - x2[k] * ts[k];
        y2[k] = x1[k] * ts[k] + x2[k] * tc[k];
      }
      sts8(s_k[warp][r] + 8 * c, y1);
      sts8(s_k[warp][r] + 8 * c + kHalf, y2);
    }
  }
  __syncwarp();

  // the lane's 16 features: granules e, e + 4 (first half of the rotary pairs), e + 8, e + 12
  // (their partners); q' and the key granules are held in that order
#pragma unroll 1
  for (int rb = R * g; rb < kBandRows; rb += 8 * R) {
    if (rb != R * g) load_q(rb);
    // q' of the lane's rows, its features, in fp32
    float qv[R][16];
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int row = rb + i, r = row + W;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float x1[4], x2[4], tc[4], ts[4];
        const int u = 4 * (e + 4 * c);
        QG::widen(qraw[i][c], x1);
        QG::widen(qraw[i][c + 2], x2);
        lds4(&s_tab[r][0][u], tc);
        lds4(&s_tab[r][1][u], ts);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          qv[i][4 * c + k] = (x1[k] * tc[k] - x2[k] * ts[k]) * sl2;
          qv[i][8 + 4 * c + k] = (x1[k] * ts[k] + x2[k] * tc[k]) * sl2;
        }
      }
    }
    // partial scores of the lane's features: row i against key rb + kk (d = kk - i)
    float ps[R][2 * W + 1];
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
      for (int d = 0; d <= 2 * W; ++d) ps[i][d] = 0.f;
#pragma unroll
    for (int kk = 0; kk < kKeys; ++kk) {
      const float* kr = s_k[warp][rb + kk];
      float kv[16];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float4 x = *reinterpret_cast<const float4*>(kr + 4 * (e + 4 * c));
        kv[4 * c] = x.x;
        kv[4 * c + 1] = x.y;
        kv[4 * c + 2] = x.z;
        kv[4 * c + 3] = x.w;
      }
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const int d = kk - i;
        if (d >= 0 && d <= 2 * W) {
          float2 acc = make_float2(0.f, 0.f);
#pragma unroll
          for (int f = 0; f < 16; f += 2)
            acc = __ffma2_rn(make_float2(qv[i][f], qv[i][f + 1]), make_float2(kv[f], kv[f + 1]), acc);
          ps[i][d] = acc.x + acc.y;
        }
      }
    }
    // whole scores (the four lanes of the group), the mask, the softmax
    float l[R], m[R];
    bool ok[R];
    if constexpr (R == 4) {
      // Lane e of a group finishes row e alone: two exchange rounds (each sends the half of its
      // partial sums it does not keep) leave it the whole scores of its row; it takes that row's
      // softmax, and the four rows' weights, maxima and sums are then shared within the group.
      const bool hi2 = (e & 2) != 0, hi1 = (e & 1) != 0;
      float h[2][2 * W + 1];
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int d = 0; d <= 2 * W; ++d) {
          const float keep = hi2 ? ps[i + 2][d] : ps[i][d];
          const float send = hi2 ? ps[i][d] : ps[i + 2][d];
          h[i][d] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
        }
      float sr[2 * W + 1];
#pragma unroll
      for (int d = 0; d <= 2 * W; ++d) {
        const float keep = hi1 ? h[1][d] : h[0][d];
        const float send = hi1 ? h[0][d] : h[1][d];
        sr[d] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
      }
      const long long a = t0 + rb + e;
      const bool oke = a < T;
      const int r = rb + e + W;
      const int aw = static_cast<int>(a) - W;
      const int dlo = oke ? max(s_seq_lo[r], static_cast<int>(a) - window) - aw : 0;
      const int dhi = oke ? min(s_seq_hi[r], static_cast<int>(a) + window + 1) - aw : 0;
      float me = -INFINITY;
#pragma unroll
      for (int d = 0; d <= 2 * W; ++d) {
        const float x = (d >= dlo && d < dhi) ? sr[d] : -INFINITY;
        sr[d] = x;
        me = fmaxf(me, x);
      }
      float le = 0.f;
#pragma unroll
      for (int d = 0; d <= 2 * W; ++d) {
        float pw;
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(pw) : "f"(sr[d] - me));
        pw = oke ? pw : 0.f;
        sr[d] = pw;
        le += pw;
      }
      const int grp = lane & ~3;
#pragma unroll
      for (int i = 0; i < R; ++i) {
#pragma unroll
        for (int d = 0; d <= 2 * W; ++d) ps[i][d] = __shfl_sync(0xffffffffu, sr[d], grp | i);
        l[i] = __shfl_sync(0xffffffffu, le, grp | i);
        m[i] = __shfl_sync(0xffffffffu, me, grp | i);
        ok[i] = t0 + rb + i < T;
      }
    } else {
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const long long a = t0 + rb + i;
        ok[i] = a < T;
        const int r = rb + i + W;
        // key a - W + d is visible for d in [dlo, dhi) (tokens < 2^31)
        const int aw = static_cast<int>(a) - W;
        const int dlo = ok[i] ? max(s_seq_lo[r], static_cast<int>(a) - window) - aw : 0;
        const int dhi = ok[i] ? min(s_seq_hi[r], static_cast<int>(a) + window + 1) - aw : 0;
        m[i] = -INFINITY;
#pragma unroll
        for (int d = 0; d <= 2 * W; ++d) {
          float x = ps[i][d];
          x += __shfl_xor_sync(0xffffffffu, x, 1);
          x += __shfl_xor_sync(0xffffffffu, x, 2);
          x = (d >= dlo && d < dhi) ? x : -INFINITY;
          ps[i][d] = x;
          m[i] = fmaxf(m[i], x);
        }
        l[i] = 0.f;
#pragma unroll
        for (int d = 0; d <= 2 * W; ++d) {
          float pw;
          asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(pw) : "f"(ps[i][d] - m[i]));
          pw = ok[i] ? pw : 0.f;
          ps[i][d] = pw;
          l[i] += pw;
        }
      }
    }
    // out: the lane's features of each row, from the value granules of key rb + kk
    float2 o[R][8];
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
      for (int f = 0; f < 8; ++f) o[i][f] = make_float2(0.f, 0.f);
#pragma unroll
    for (int kk = 0; kk < kKeys; ++kk) {
      float vv[16];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float x[4];
        lds4(s_v[warp][rb + kk] + 4 * (e + 4 * c), x);
        vv[4 * c] = x[0];
        vv[4 * c + 1] = x[1];
        vv[4 * c + 2] = x[2];
        vv[4 * c + 3] = x[3];
      }
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const int d = kk - i;
        if (d >= 0 && d <= 2 * W) {
          const float2 p2 = make_float2(ps[i][d], ps[i][d]);
#pragma unroll
          for (int f = 0; f < 8; ++f) o[i][f] = __ffma2_rn(p2, make_float2(vv[2 * f], vv[2 * f + 1]), o[i][f]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < R; ++i) {
      if (!ok[i]) continue;
      const long long a = t0 + rb + i;
      const float inv = 1.0f / l[i];
      const int64_t at = a * static_cast<int64_t>(H) * kD + static_cast<int64_t>(h) * kD;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        // granule e + 4 c: this lane's features 4 c .. 4 c + 3
        const float y0 = o[i][2 * c].x * inv, y1 = o[i][2 * c].y * inv;
        const float y2 = o[i][2 * c + 1].x * inv, y3 = o[i][2 * c + 1].y * inv;
        store4<OUT>(out, at + 4 * (e + 4 * c), y0, y1, y2, y3);
      }
      if (e == 0) lse[static_cast<int64_t>(h) * T + a] = m[i] * 0.6931471805599453f + logf(l[i]);
    }
  }
}

namespace {

template <typename F, int W>
constexpr size_t band_smem_bytes() {
  return BandSmem<F, W>::kBytes;
}

template <typename F, int OUT, int W>
cudaError_t band_attr() {
  cudaError_t e = cudaFuncSetAttribute(pk_attend_band_kernel<F, OUT, W>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(band_smem_bytes<F, W>()));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pk_attend_band_kernel<F, OUT, W>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  return e;
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
