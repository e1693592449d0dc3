// pk_mixed_ops.cu -- fp32 storage, 16-bit tensor-core operands: the rotation step of
// pk_attend_mixed_ops.
//
// hanzo-kernel packed.rs keeps the storage type F of qkv, the tables and the output apart from
// the operand type M of the matrix products (fn attend: the rotated q and k and the
// probabilities are cast to M; the tests run f32 storage with f16 operands). On this part the
// 16-bit operands are read by the tensor cores straight from shared memory, where TMA puts
// them, so an fp32 qkv is first brought to that form: this kernel rotates q and k in fp32 (q
// multiplied by `q_mul`), rounds q', k' and v once to the operand type and writes them in the
// packed layout [T, 3 H 64]. The tensor-core kernel then runs on that copy without rotating
// again, and writes an fp32 output.
//
// The rotation is the same expression, in the same order, as the tensor-core kernel's own
// (y1 = fma(x1, c, -(x2 s)), y2 = fma(x1, s, x2 c), then the multiply), so that for fp32 inputs
// holding 16-bit values the operands -- and so the whole result -- equal those of the 16-bit
// path bit for bit.
//
// One warp per token (grid-stride): lane l holds the rotary pair (l, l + 32) of every head
// vector of the token, so each fp32 row is read and each 16-bit row written in whole 128-byte
// and 64-byte runs. The token's position comes from a search in cu (small; L1 serves it). The
// tile scheduler runs before this kernel and has checked cu: after a malformed one
// (ctl->ntiles = 0) the kernel writes nothing.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pk.h"
#include "pk_dev.cuh"

namespace pk {

namespace {
template <bool BF16>
__device__ __forceinline__ uint16_t round16(float x) {
  if constexpr (BF16)
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  else
    return __half_as_ushort(__float2half_rn(x));
}
}  // namespace

template <bool BF16>
__global__ void __launch_bounds__(256)
pk_rotate16_kernel(const float* __restrict__ qkv, const float* __restrict__ cos_t, const float* __restrict__ sin_t,
                   const uint32_t* __restrict__ cu, int S, long long T, int H, float q_mul, const Ctl* ctl,
                   uint16_t* __restrict__ y) {
  if (__ldcg(&ctl->ntiles) == 0u) return;
  const int lane = threadIdx.x & 31;
  const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const int64_t ld = 3ll * H * kD;
  for (long long a = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); a < T;
       a += nwarps) {
    const uint32_t s = seq_of_token(cu, 0u, static_cast<uint32_t>(S), static_cast<uint32_t>(a));
    const int64_t pos = a - static_cast<long long>(__ldg(cu + s));
    const float c = __ldg(cos_t + pos * kHalf + lane), sn = __ldg(sin_t + pos * kHalf + lane);
    const float* x = qkv + a * ld;
    uint16_t* yo = y + a * ld;
    for (int part = 0; part < 2; ++part) {
      for (int h = 0; h < H; ++h) {
        const int64_t off = static_cast<int64_t>(part * H + h) * kD;
        const float x1 = __ldg(x + off + lane), x2 = __ldg(x + off + lane + kHalf);
        float y1 = fmaf(x1, c, -(x2 * sn));
        float y2 = fmaf(x1, sn, x2 * c);
        if (part == 0 && q_mul != 1.0f) {
          y1 *= q_mul;
          y2 *= q_mul;
        }
        yo[off + lane] = round16<BF16>(y1);
        yo[off + lane + kHalf] = round16<BF16>(y2);
      }
    }
    for (int h = 0; h < H; ++h) {
      const int64_t off = static_cast<int64_t>(2 * H + h) * kD;
      yo[off + lane] = round16<BF16>(__ldg(x + off + lane));
      yo[off + lane + kHalf] = round16<BF16>(__ldg(x + off + lane + kHalf));
    }
  }
}

// Split copy for fp32 inputs on the tensor cores: every value x of q' (rotated, times q_mul),
// k' (rotated) and v becomes two bf16 values, hi = bf16(x) and lo = bf16(x - hi), so that
// hi + lo carries 16 significant bits of x. Row a of y holds 6 H 64 values: the hi copy of
// the packed row [q' | k' | v] in columns [0, 3 H 64) and the lo copy in [3 H 64, 6 H 64).
// The products S = Qh Kh^T + Qh Kl^T + Ql Kh^T then match the fp32 scores to about 2^-16
// of their terms' size (the Ql Kl^T term, 2^-16 smaller again, is left out).
__device__ __forceinline__ void split_store(uint16_t* hi, uint16_t* lo, float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  *hi = __bfloat16_as_ushort(h);
  *lo = __bfloat16_as_ushort(__float2bfloat16_rn(x - __bfloat162float(h)));
}

__global__ void __launch_bounds__(256)
pk_split16_kernel(const float* __restrict__ qkv, const float* __restrict__ cos_t, const float* __restrict__ sin_t,
                  const uint32_t* __restrict__ cu, int S, long long T, int H, float q_mul, const Ctl* ctl,
                  uint16_t* __restrict__ y) {
  if (__ldcg(&ctl->ntiles) == 0u) return;
  const int lane = threadIdx.x & 31;
  const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const int64_t ld = 3ll * H * kD;
  for (long long a = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); a < T;
       a += nwarps) {
    const uint32_t s = seq_of_token(cu, 0u, static_cast<uint32_t>(S), static_cast<uint32_t>(a));
    const int64_t pos = a - static_cast<long long>(__ldg(cu + s));
    const float c = __ldg(cos_t + pos * kHalf + lane), sn = __ldg(sin_t + pos * kHalf + lane);
    const float* x = qkv + a * ld;
    uint16_t* yh = y + a * 2 * ld;
    uint16_t* yl = yh + ld;
    for (int part = 0; part < 2; ++part) {
      for (int h = 0; h < H; ++h) {
        const int64_t off = static_cast<int64_t>(part * H + h) * kD;
        const float x1 = __ldg(x + off + lane), x2 = __ldg(x + off + lane + kHalf);
        float y1 = fmaf(x1, c, -(x2 * sn));
        float y2 = fmaf(x1, sn, x2 * c);
        if (part == 0 && q_mul != 1.0f) {
          y1 *= q_mul;
          y2 *= q_mul;
        }
        split_store(yh + off + lane, yl + off + lane, y1);
        split_store(yh + off + lane + kHalf, yl + off + lane + kHalf, y2);
      }
    }
    for (int h = 0; h < H; ++h) {
      const int64_t off = static_cast<int64_t>(2 * H + h) * kD;
      split_store(yh + off + lane, yl + off + lane, __ldg(x + off + lane));
      split_store(yh + off + lane + kHalf, yl + off + lane + kHalf, __ldg(x + off + lane + kHalf));
    }
  }
}

// Host side: the split copy (T x 6 H 64 bf16 values) of an fp32 qkv into `y`, on `stream`
// after the tile scheduler.
cudaError_t split16_launch(const float* qkv, const float* cos_t, const float* sin_t, const uint32_t* cu, int S,
                           long long T, int H, float q_mul, const Ctl* ctl, void* y, int sms, cudaStream_t stream) {
  const int blocks = static_cast<int>(min(static_cast<long long>(sms) * 8, (T + 7) / 8));
  pk_split16_kernel<<<blocks, 256, 0, stream>>>(qkv, cos_t, sin_t, cu, S, T, H, q_mul, ctl, static_cast<uint16_t*>(y));
  return cudaGetLastError();
}

// Host side: the rotated 16-bit copy of an fp32 qkv into `y` (T x 3 H 64 elements of
// op_dtype), on `stream` after the tile scheduler.
cudaError_t rotate16_launch(int op_dtype, const float* qkv, const float* cos_t, const float* sin_t, const uint32_t* cu,
                            int S, long long T, int H, float q_mul, const Ctl* ctl, void* y, int sms,
                            cudaStream_t stream) {
  const long long warps_needed = T;
  const int blocks = static_cast<int>(min(static_cast<long long>(sms) * 8, (warps_needed + 7) / 8));
  if (op_dtype == PK_BF16)
    pk_rotate16_kernel<true><<<blocks, 256, 0, stream>>>(qkv, cos_t, sin_t, cu, S, T, H, q_mul, ctl,
                                                         static_cast<uint16_t*>(y));
  else
    pk_rotate16_kernel<false><<<blocks, 256, 0, stream>>>(qkv, cos_t, sin_t, cu, S, T, H, q_mul, ctl,
                                                          static_cast<uint16_t*>(y));
  return cudaGetLastError();
}

}  // namespace pk
