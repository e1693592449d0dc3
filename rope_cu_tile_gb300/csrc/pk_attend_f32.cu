// pk_attend_f32.cu -- packed RoPE attention forward for fp32 inputs, on the CUDA cores.
//
// Same operation and tile records as the tensor-core kernel (hanzo-kernel packed.rs fn
// attend: rotate and scale q, rotate k, scores of each query against its own sequence's
// keys within the window, online softmax, out = O / l, lse = m + ln l), with every product
// and sum in fp32. fp32 inputs ask for max |error| <= 1e-4 on out and lse, which one pass
// of TF32 tensor-core products (10-bit mantissas) cannot give; this kernel is exact to
// fp32 rounding.
//
// One 128-thread CTA per work item (tile record, head) at a time, persistent; thread r
// owns query row r (q' in registers, 64 output accumulators). Keys go through shared
// memory 32 at a time, rotated once by the CTA.
//
// The output may also be written in a 16-bit type (OUT: kime's attention variant with an
// FP32 qkv and a half output, which keeps q and k in FP32 because rounding them moves the
// softmax): everything stays fp32 up to one rounding of out = O / l.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pk.h"
#include "pk_dev.cuh"

namespace pk {

namespace {
constexpr int kThreadsF32 = 128;
constexpr int kChunk = 32;   // keys per shared-memory chunk
}  // namespace

namespace {
// four output values, rounded to the output type and stored together
template <int OUT>
__device__ __forceinline__ void store4(void* out, int64_t i, float a, float b, float c, float d) {
  if constexpr (OUT == PK_F32) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + i) = make_float4(a, b, c, d);
  } else if constexpr (OUT == PK_BF16) {
    const uint32_t lo = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(a))) |
                        (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(b))) << 16);
    const uint32_t hi = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(c))) |
                        (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(d))) << 16);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + i) = make_uint2(lo, hi);
  } else {
    const uint32_t lo = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(a))) |
                        (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(b))) << 16);
    const uint32_t hi = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(c))) |
                        (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(d))) << 16);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + i) = make_uint2(lo, hi);
  }
}
}  // namespace

template <int OUT>
__global__ void __launch_bounds__(kThreadsF32)
pk_attend_f32_kernel(const float* __restrict__ qkv, const float* __restrict__ cos_t,
                     const float* __restrict__ sin_t, const uint32_t* __restrict__ cu,
                     const TileRec* __restrict__ tiles, void* __restrict__ out,
                     float* __restrict__ lse, Ctl* ctl, int H, long long T, int window,
                     float scale) {
  __shared__ float sk[kChunk][kD + 1];
  __shared__ float sv[kChunk][kD + 1];
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

    const int r = tid;
    const bool row_ok = r < static_cast<int>(rec.rows);
    const uint32_t a = rec.q0 + r;
    int64_t lo = 0, hi = 0;
    float q[kD];
#pragma unroll
    for (int d = 0; d < kD; ++d) q[d] = 0.f;
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
      const float* x = qkv + static_cast<int64_t>(a) * ldq + h * kD;
#pragma unroll
      for (int u = 0; u < kHalf; ++u) {
        const float c = __ldg(cos_t + pos * kHalf + u), sn = __ldg(sin_t + pos * kHalf + u);
        const float x1 = __ldg(x + u), x2 = __ldg(x + u + kHalf);
        q[u] = (x1 * c - x2 * sn) * scale;
        q[u + kHalf] = (x1 * sn + x2 * c) * scale;
      }
    }
    float o[kD];
#pragma unroll
    for (int d = 0; d < kD; ++d) o[d] = 0.f;
    float m = -INFINITY, l = 0.f;
    const uint32_t kend = rec.k0 + rec.nk;
    for (uint32_t j0 = rec.k0; j0 < kend; j0 += kChunk) {
      // stage 32 keys (rotated) and values: 4 threads per key, 8 rotary pairs each
      {
        const int kk = tid >> 2, part = tid & 3;
        const uint32_t b = j0 + kk;
        if (b < kend) {
          const uint32_t sb = rec.kind == 0 ? rec.seq : seq_of_token(cu, rec.seq, rec.nseq, b);
          const int64_t pos = static_cast<int64_t>(b) - __ldg(cu + sb);
          const float* x = qkv + static_cast<int64_t>(b) * ldq + hd + h * kD;
          const float* v = qkv + static_cast<int64_t>(b) * ldq + 2 * hd + h * kD;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int u = part * 8 + e;
            const float c = __ldg(cos_t + pos * kHalf + u), sn = __ldg(sin_t + pos * kHalf + u);
            const float x1 = __ldg(x + u), x2 = __ldg(x + u + kHalf);
            sk[kk][u] = x1 * c - x2 * sn;
            sk[kk][u + kHalf] = x1 * sn + x2 * c;
            sv[kk][u] = __ldg(v + u);
            sv[kk][u + kHalf] = __ldg(v + u + kHalf);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int u = part * 8 + e;
            sk[kk][u] = 0.f;
            sk[kk][u + kHalf] = 0.f;
            sv[kk][u] = 0.f;
            sv[kk][u + kHalf] = 0.f;
          }
        }
      }
      __syncthreads();
      float sc[kChunk];
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < kChunk; ++c) {
        const int64_t j = static_cast<int64_t>(j0) + c;
        float acc = 0.f;
#pragma unroll
        for (int d = 0; d < kD; ++d) acc = fmaf(q[d], sk[c][d], acc);
        const bool vis = j >= lo && j < hi;
        sc[c] = vis ? acc : -INFINITY;
        mx = fmaxf(mx, sc[c]);
      }
      if (mx > -INFINITY) {
        const float m_new = fmaxf(m, mx);
        const float alpha = __expf(m - m_new);   // exp(-inf) = 0 on the first visible chunk
        float sum = 0.f;
#pragma unroll
        for (int d = 0; d < kD; ++d) o[d] *= alpha;
#pragma unroll
        for (int c = 0; c < kChunk; ++c) {
          const float p = __expf(sc[c] - m_new);
          sum += p;
#pragma unroll
          for (int d = 0; d < kD; ++d) o[d] = fmaf(p, sv[c][d], o[d]);
        }
        l = l * alpha + sum;
        m = m_new;
      }
      __syncthreads();
    }
    if (row_ok) {
      const float inv = 1.0f / l;
      const int64_t at = static_cast<int64_t>(a) * hd + h * kD;
#pragma unroll
      for (int d = 0; d < kD; d += 4) store4<OUT>(out, at + d, o[d] * inv, o[d + 1] * inv, o[d + 2] * inv, o[d + 3] * inv);
      lse[static_cast<int64_t>(h) * T + a] = m + logf(l);
    }
  }
}

// out_dtype: PK_F32, or PK_BF16 / PK_F16 for a 16-bit output
cudaError_t attend_f32_launch(const float* qkv, const float* cos_t, const float* sin_t, const uint32_t* cu,
                              const TileRec* tiles, void* out, int out_dtype, float* lse, Ctl* ctl, int H,
                              long long T, int window, float scale, int grid, cudaStream_t stream) {
  if (out_dtype == PK_BF16)
    pk_attend_f32_kernel<PK_BF16><<<grid, kThreadsF32, 0, stream>>>(qkv, cos_t, sin_t, cu, tiles, out, lse, ctl, H,
                                                                     T, window, scale);
  else if (out_dtype == PK_F16)
    pk_attend_f32_kernel<PK_F16><<<grid, kThreadsF32, 0, stream>>>(qkv, cos_t, sin_t, cu, tiles, out, lse, ctl, H,
                                                                    T, window, scale);
  else
    pk_attend_f32_kernel<PK_F32><<<grid, kThreadsF32, 0, stream>>>(qkv, cos_t, sin_t, cu, tiles, out, lse, ctl, H,
                                                                    T, window, scale);
  return cudaGetLastError();
}

}  // namespace pk
