// pk_backward.cu -- the backward pass of packed RoPE attention (pk_attend_backward in
// include/pk.h), on the CUDA cores in fp32.
//
// The pages' attend_back (hanzo-kernel packed.rs) computes, per query row i and visible key j of
// its sequence, with q'_i = rot(q_i, i), k'_j = rot(k_j, j), s_ij = scale q'_i . k'_j and the
// forward's lse: P_ij = exp(s_ij - lse_i), D_i = dout_i . out_i, dP_ij = dout_i . v_j,
// dS_ij = P_ij (dP_ij - D_i); then dv_j = sum_i P_ij dout_i, dq'_i = scale sum_j dS_ij k'_j,
// dk'_j = scale sum_i dS_ij q'_i, and the rotation is undone: dq = rot^T(dq'), dk = rot^T(dk').
//
// Three kernels over the forward's tile records (the same device schedule):
//   prep    D [H, T] = rowsum(dout * out), fp32
//   main    per work item (tile record, head), persistent CTAs of 128 threads (two per SM),
//           thread r <-> query row r (dout in registers, q' and dout in shared memory). Keys go
//           through shared memory 16 at a time (rotated once); each thread forms its row's P and
//           dS for them (key and value rows read as 16-byte broadcasts) and accumulates dq' in
//           registers; the CTA then reduces dv and dk' of the 16 keys over its rows and adds
//           them to fp32 accumulators in global memory (other records of the same sequence add
//           to the same keys). dq' of each row is written once. Shared-memory bandwidth bounds
//           this version (the column sums read two 64-float rows per row and key).
//   finish  dq = rot^T(dq'), dk = rot^T(dk'), dv, rounded once to the element type.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pk.h"
#include "pk_dev.cuh"

namespace pk {

namespace {

constexpr int kBwdThreads = 128;
constexpr int kBwdChunk = 16;  // keys per shared-memory chunk
constexpr int kRowF = kD + 4;  // shared-memory row stride in floats (rows start on 16 bytes)
constexpr int kBwdSmem =
    static_cast<int>(sizeof(float)) * ((2 * kBwdChunk + 2 * kBwdThreads) * kRowF + 2 * kBwdThreads * (kBwdChunk + 1));

template <int DT>
__device__ __forceinline__ float ldf(const void* p, int64_t i) {
  if constexpr (DT == PK_F32) {
    return __ldg(static_cast<const float*>(p) + i);
  } else if constexpr (DT == PK_BF16) {
    return __uint_as_float(static_cast<uint32_t>(__ldg(static_cast<const unsigned short*>(p) + i)) << 16);
  } else {
    return __half2float(__ushort_as_half(__ldg(static_cast<const unsigned short*>(p) + i)));
  }
}

template <int DT>
__device__ __forceinline__ void stf2(void* p, int64_t i, float a, float b) {
  if constexpr (DT == PK_F32) {
    *reinterpret_cast<float2*>(static_cast<float*>(p) + i) = make_float2(a, b);
  } else if constexpr (DT == PK_BF16) {
    *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p) + i) =
        static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(a))) |
        (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(b))) << 16);
  } else {
    *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p) + i) =
        static_cast<uint32_t>(__half_as_ushort(__float2half_rn(a))) |
        (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(b))) << 16);
  }
}

// D [h * T + t] = sum_d dout[t, h, d] out[t, h, d]
template <int DT>
__global__ void __launch_bounds__(256) pk_bwd_prep_kernel(const void* __restrict__ out, const void* __restrict__ dout,
                                                          float* __restrict__ D, int H, long long T) {
  const long long n = T * H;
  for (long long u = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; u < n;
       u += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long t = u / H;
    const int h = static_cast<int>(u % H);
    const int64_t at = t * H * kD + h * kD;
    float acc = 0.f;
#pragma unroll 8
    for (int d = 0; d < kD; ++d) acc = fmaf(ldf<DT>(dout, at + d), ldf<DT>(out, at + d), acc);
    D[static_cast<int64_t>(h) * T + t] = acc;
  }
}

template <int DT>
__global__ void __launch_bounds__(kBwdThreads, 2)
pk_bwd_main_kernel(const void* __restrict__ qkv, const void* __restrict__ cos_t, const void* __restrict__ sin_t,
                   const uint32_t* __restrict__ cu, const TileRec* __restrict__ tiles, Ctl* ctl,
                   const float* __restrict__ lse, const void* __restrict__ dout, const float* __restrict__ D,
                   float* __restrict__ dq_acc, float* __restrict__ dk_acc, float* __restrict__ dv_acc, int H,
                   long long T, int window, float scale) {
  // dynamic shared memory (kBwdSmem bytes): keys, values, the rows' q' and dout, P and dS
  extern __shared__ __align__(16) float bwd_smem[];
  float(*sk)[kRowF] = reinterpret_cast<float(*)[kRowF]>(bwd_smem);
  float(*sv)[kRowF] = sk + kBwdChunk;
  float(*sq)[kRowF] = sv + kBwdChunk;
  float(*sdo)[kRowF] = sq + kBwdThreads;
  float(*sp)[kBwdChunk + 1] = reinterpret_cast<float(*)[kBwdChunk + 1]>(sdo + kBwdThreads);
  float(*sds)[kBwdChunk + 1] = sp + kBwdThreads;
  __shared__ unsigned int s_item;
  const int tid = threadIdx.x;
  const unsigned int n_items = __ldcg(&ctl->ntiles) * static_cast<unsigned int>(H);
  const int64_t ldq = 3ll * H * kD;
  const int64_t hd = static_cast<int64_t>(H) * kD;

  for (;;) {
    if (tid == 0) s_item = atomicAdd(&ctl->next, 1u);
    __syncthreads();
    const unsigned int item = s_item;
    __syncthreads();
    if (item >= n_items) break;
    const unsigned int ti = item / static_cast<unsigned int>(H);
    const int h = static_cast<int>(item % static_cast<unsigned int>(H));
    const TileRec rec = tiles[ti];

    // this thread's row: q' (rotated), dout, lse, D and the visible key interval [lo, hi)
    const int r = tid;
    const bool row_ok = r < static_cast<int>(rec.rows);
    const uint32_t a = rec.q0 + r;
    int64_t lo = 0, hi = 0;
    float lse_r = 0.f, d_r = 0.f;
    if (row_ok) {
      const uint32_t s = rec.kind == 0 ? rec.seq : seq_of_token(cu, rec.seq, rec.nseq, a);
      const int64_t ss = __ldg(cu + s), se = __ldg(cu + s + 1);
      const int64_t pos = static_cast<int64_t>(a) - ss;
      lo = ss;
      hi = se;
      if (window > 0) {
        lo = max(ss, static_cast<int64_t>(a) - window);
        hi = min(se, static_cast<int64_t>(a) + window + 1);
      }
      const int64_t x = static_cast<int64_t>(a) * ldq + h * kD;
      for (int u = 0; u < kHalf; ++u) {
        const float c = ldf<DT>(cos_t, pos * kHalf + u), sn = ldf<DT>(sin_t, pos * kHalf + u);
        const float x1 = ldf<DT>(qkv, x + u), x2 = ldf<DT>(qkv, x + u + kHalf);
        sq[r][u] = x1 * c - x2 * sn;
        sq[r][u + kHalf] = x1 * sn + x2 * c;
      }
      const int64_t g = static_cast<int64_t>(a) * hd + h * kD;
      for (int d = 0; d < kD; ++d) sdo[r][d] = ldf<DT>(dout, g + d);
      lse_r = __ldg(lse + static_cast<int64_t>(h) * T + a);
      d_r = __ldg(D + static_cast<int64_t>(h) * T + a);
    } else {
      for (int d = 0; d < kD; ++d) sq[r][d] = sdo[r][d] = 0.f;
    }
    // this row's dout in registers as well (the shared copies serve the column sums); its q'
    // is read from shared memory 16 bytes at a time
    float dor[kD], dq[kD];
#pragma unroll
    for (int d = 0; d < kD; ++d) {
      dor[d] = sdo[r][d];
      dq[d] = 0.f;
    }
    const float4* qrow = reinterpret_cast<const float4*>(sq[r]);

    const uint32_t kend = rec.k0 + rec.nk;
    for (uint32_t j0 = rec.k0; j0 < kend; j0 += kBwdChunk) {
      __syncthreads();  // the previous chunk's reduction has read sk, sv, sp, sds
      // stage 16 keys (rotated) and values: 8 threads per key, 4 rotary pairs each
      {
        const int kk = tid >> 3, part = tid & 7;
        const uint32_t b = j0 + kk;
        if (b < kend) {
          const uint32_t sb = rec.kind == 0 ? rec.seq : seq_of_token(cu, rec.seq, rec.nseq, b);
          const int64_t pos = static_cast<int64_t>(b) - __ldg(cu + sb);
          const int64_t x = static_cast<int64_t>(b) * ldq + hd + h * kD;
          const int64_t v = static_cast<int64_t>(b) * ldq + 2 * hd + h * kD;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int u = part * 4 + e;
            const float c = ldf<DT>(cos_t, pos * kHalf + u), sn = ldf<DT>(sin_t, pos * kHalf + u);
            const float x1 = ldf<DT>(qkv, x + u), x2 = ldf<DT>(qkv, x + u + kHalf);
            sk[kk][u] = x1 * c - x2 * sn;
            sk[kk][u + kHalf] = x1 * sn + x2 * c;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) sv[kk][part * 8 + e] = ldf<DT>(qkv, v + part * 8 + e);
        }
      }
      __syncthreads();
      // this row against the chunk's keys: P, dS, and dq' += scale dS k'
      const int nc = static_cast<int>(min(static_cast<uint32_t>(kBwdChunk), kend - j0));
      for (int c = 0; c < kBwdChunk; ++c) {
        const int64_t b = static_cast<int64_t>(j0) + c;
        float p = 0.f, ds = 0.f;
        if (row_ok && c < nc && b >= lo && b < hi) {
          // key and value rows: the same address for every thread (broadcast), 16 bytes a load
          const float4* kc = reinterpret_cast<const float4*>(sk[c]);
          const float4* vc = reinterpret_cast<const float4*>(sv[c]);
          float sdot = 0.f, pdot = 0.f;
#pragma unroll
          for (int q4 = 0; q4 < kD / 4; ++q4) {
            const float4 k4 = kc[q4], v4 = vc[q4], x4 = qrow[q4];
            sdot = fmaf(x4.x, k4.x, sdot);
            sdot = fmaf(x4.y, k4.y, sdot);
            sdot = fmaf(x4.z, k4.z, sdot);
            sdot = fmaf(x4.w, k4.w, sdot);
            pdot = fmaf(dor[4 * q4], v4.x, pdot);
            pdot = fmaf(dor[4 * q4 + 1], v4.y, pdot);
            pdot = fmaf(dor[4 * q4 + 2], v4.z, pdot);
            pdot = fmaf(dor[4 * q4 + 3], v4.w, pdot);
          }
          p = __expf(scale * sdot - lse_r);
          ds = p * (pdot - d_r);
#pragma unroll
          for (int q4 = 0; q4 < kD / 4; ++q4) {
            const float4 k4 = kc[q4];
            dq[4 * q4] = fmaf(ds, k4.x, dq[4 * q4]);
            dq[4 * q4 + 1] = fmaf(ds, k4.y, dq[4 * q4 + 1]);
            dq[4 * q4 + 2] = fmaf(ds, k4.z, dq[4 * q4 + 2]);
            dq[4 * q4 + 3] = fmaf(ds, k4.w, dq[4 * q4 + 3]);
          }
        }
        sp[r][c] = p;
        sds[r][c] = ds;
      }
      __syncthreads();
      // the chunk's dv and dk' over this CTA's rows: thread (c, 8 dims)
      {
        const int c = tid >> 3, d0 = (tid & 7) * 8;
        if (c < nc) {
          float dv[8], dk[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) dv[e] = dk[e] = 0.f;
          const int nr = static_cast<int>(rec.rows);
          for (int rr = 0; rr < nr; ++rr) {
            const float p = sp[rr][c], ds = sds[rr][c];
            const float4 o0 = *reinterpret_cast<const float4*>(&sdo[rr][d0]);
            const float4 o1 = *reinterpret_cast<const float4*>(&sdo[rr][d0 + 4]);
            const float4 q0 = *reinterpret_cast<const float4*>(&sq[rr][d0]);
            const float4 q1 = *reinterpret_cast<const float4*>(&sq[rr][d0 + 4]);
            dv[0] = fmaf(p, o0.x, dv[0]); dv[1] = fmaf(p, o0.y, dv[1]);
            dv[2] = fmaf(p, o0.z, dv[2]); dv[3] = fmaf(p, o0.w, dv[3]);
            dv[4] = fmaf(p, o1.x, dv[4]); dv[5] = fmaf(p, o1.y, dv[5]);
            dv[6] = fmaf(p, o1.z, dv[6]); dv[7] = fmaf(p, o1.w, dv[7]);
            dk[0] = fmaf(ds, q0.x, dk[0]); dk[1] = fmaf(ds, q0.y, dk[1]);
            dk[2] = fmaf(ds, q0.z, dk[2]); dk[3] = fmaf(ds, q0.w, dk[3]);
            dk[4] = fmaf(ds, q1.x, dk[4]); dk[5] = fmaf(ds, q1.y, dk[5]);
            dk[6] = fmaf(ds, q1.z, dk[6]); dk[7] = fmaf(ds, q1.w, dk[7]);
          }
          const int64_t at = (static_cast<int64_t>(j0) + c) * hd + h * kD + d0;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            atomicAdd(dv_acc + at + e, dv[e]);
            atomicAdd(dk_acc + at + e, scale * dk[e]);
          }
        }
      }
    }
    if (row_ok) {
      const int64_t at = static_cast<int64_t>(a) * hd + h * kD;
#pragma unroll
      for (int d = 0; d < kD; d += 4)
        *reinterpret_cast<float4*>(dq_acc + at + d) =
            make_float4(scale * dq[d], scale * dq[d + 1], scale * dq[d + 2], scale * dq[d + 3]);
    }
    __syncthreads();
  }
}

// dqkv: dq = rot^T(dq'), dk = rot^T(dk'), dv; one warp per token, lane l holding the rotary pair
// (l, l + 32) of a head vector (the halves' pairing), positions from cu
template <int DT>
__global__ void __launch_bounds__(256)
pk_bwd_finish_kernel(const void* __restrict__ cos_t, const void* __restrict__ sin_t, const uint32_t* __restrict__ cu,
                     int S, long long T, int H, const float* __restrict__ dq_acc, const float* __restrict__ dk_acc,
                     const float* __restrict__ dv_acc, void* __restrict__ dqkv) {
  const int lane = threadIdx.x & 31;
  const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int64_t hd = static_cast<int64_t>(H) * kD, ldq = 3 * hd;
  for (long long t = gw; t < T; t += nw) {
    // the token's sequence: the last s with cu[s] <= t (binary search in global memory)
    uint32_t lo = 0, hi = static_cast<uint32_t>(S);  // first s with cu[s] > t lies in (lo, hi]
    while (lo < hi) {
      const uint32_t mid = (lo + hi) >> 1;
      if (static_cast<long long>(__ldg(cu + mid)) <= t) lo = mid + 1; else hi = mid;
    }
    const uint32_t s = lo > 0 ? lo - 1 : 0;
    const int64_t pos = t - static_cast<int64_t>(__ldg(cu + s));
    const float c = ldf<DT>(cos_t, pos * kHalf + lane), sn = ldf<DT>(sin_t, pos * kHalf + lane);
    for (int h = 0; h < H; ++h) {
      const int64_t g = t * hd + h * kD;
      // rot^T: y_a = x_a c + x_b s, y_b = x_b c - x_a s
      const float qa = dq_acc[g + lane], qb = dq_acc[g + lane + kHalf];
      const float ka = dk_acc[g + lane], kb = dk_acc[g + lane + kHalf];
      const int64_t o = t * ldq + h * kD;
      float y[4] = {fmaf(qa, c, qb * sn), fmaf(qb, c, -qa * sn), fmaf(ka, c, kb * sn), fmaf(kb, c, -ka * sn)};
      // lanes write pairs of neighbouring features: gather them by shuffle
      const float qa1 = __shfl_down_sync(0xffffffffu, y[0], 1), qb1 = __shfl_down_sync(0xffffffffu, y[1], 1);
      const float ka1 = __shfl_down_sync(0xffffffffu, y[2], 1), kb1 = __shfl_down_sync(0xffffffffu, y[3], 1);
      if ((lane & 1) == 0) {
        stf2<DT>(dqkv, o + lane, y[0], qa1);
        stf2<DT>(dqkv, o + lane + kHalf, y[1], qb1);
        stf2<DT>(dqkv, o + hd + lane, y[2], ka1);
        stf2<DT>(dqkv, o + hd + lane + kHalf, y[3], kb1);
      }
      const float2 v = *reinterpret_cast<const float2*>(dv_acc + g + 2 * lane);
      stf2<DT>(dqkv, o + 2 * hd + 2 * lane, v.x, v.y);
    }
  }
}

template <int DT>
cudaError_t launch_backward_t(const void* qkv, const void* cos_t, const void* sin_t, const uint32_t* cu, int S,
                              long long T, int H, int window, float scale, const void* out, const float* lse,
                              const void* dout, void* dqkv, const TileRec* tiles, Ctl* ctl, float* scratch, int sms,
                              cudaStream_t stream) {
  // regions start on 256-byte boundaries (dq' is stored 16 bytes at a time)
  float* D = scratch;
  float* dq = D + (static_cast<int64_t>(H) * T + 63) / 64 * 64;
  float* dk = dq + T * H * kD;
  float* dv = dk + T * H * kD;
  cudaError_t e = cudaMemsetAsync(dk, 0, static_cast<size_t>(2) * T * H * kD * sizeof(float), stream);
  if (e != cudaSuccess) return e;
  const long long prep_blocks = min(static_cast<long long>(sms) * 8, (T * H + 255) / 256);
  pk_bwd_prep_kernel<DT><<<static_cast<unsigned int>(max(prep_blocks, 1ll)), 256, 0, stream>>>(out, dout, D, H, T);
  pk_bwd_main_kernel<DT><<<sms * 2, kBwdThreads, kBwdSmem, stream>>>(qkv, cos_t, sin_t, cu, tiles, ctl, lse, dout, D,
                                                                      dq, dk, dv, H, T, window, scale);
  const long long fin_blocks = min(static_cast<long long>(sms) * 8, (T + 7) / 8);
  pk_bwd_finish_kernel<DT><<<static_cast<unsigned int>(max(fin_blocks, 1ll)), 256, 0, stream>>>(
      cos_t, sin_t, cu, S, T, H, dq, dk, dv, dqkv);
  return cudaGetLastError();
}

}  // namespace

// once per device: the main kernel's dynamic shared memory (two blocks per SM)
cudaError_t backward_prepare() {
  cudaError_t e = cudaFuncSetAttribute(pk_bwd_main_kernel<PK_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, kBwdSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pk_bwd_main_kernel<PK_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kBwdSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pk_bwd_main_kernel<PK_F16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kBwdSmem);
  return e;
}

// fp32 scratch the backward needs for T tokens and H heads: D, dq', dk', dv
long long backward_scratch_floats(long long T, int H) {
  return (static_cast<long long>(H) * T + 63) / 64 * 64 + 3LL * H * T * kD;
}

cudaError_t backward_launch(int dtype, const void* qkv, const void* cos_t, const void* sin_t, const uint32_t* cu,
                            int S, long long T, int H, int window, float scale, const void* out, const float* lse,
                            const void* dout, void* dqkv, const TileRec* tiles, Ctl* ctl, float* scratch, int sms,
                            cudaStream_t stream) {
  if (dtype == PK_F32)
    return launch_backward_t<PK_F32>(qkv, cos_t, sin_t, cu, S, T, H, window, scale, out, lse, dout, dqkv, tiles, ctl,
                                     scratch, sms, stream);
  if (dtype == PK_BF16)
    return launch_backward_t<PK_BF16>(qkv, cos_t, sin_t, cu, S, T, H, window, scale, out, lse, dout, dqkv, tiles, ctl,
                                      scratch, sms, stream);
  return launch_backward_t<PK_F16>(qkv, cos_t, sin_t, cu, S, T, H, window, scale, out, lse, dout, dqkv, tiles, ctl,
                                   scratch, sms, stream);
}

}  // namespace pk
