// pk_backward.cu -- the backward pass of packed RoPE attention (pk_attend_backward in
// include/pk.h): 16-bit inputs on the tensor cores (the tcgen05 kernel of pk_backward_tc.cu;
// the warp-level mma.sync kernel below when PK_BWD_MMA_SYNC=1), fp32 inputs on the CUDA cores.
//
// The pages' attend_back (hanzo-kernel packed.rs) computes, per query row i and visible key j of
// its sequence, with q'_i = rot(q_i, i), k'_j = rot(k_j, j), s_ij = scale q'_i . k'_j and the
// forward's lse: P_ij = exp(s_ij - lse_i), D_i = dout_i . out_i, dP_ij = dout_i . v_j,
// dS_ij = P_ij (dP_ij - D_i); then dv_j = sum_i P_ij dout_i, dq'_i = scale sum_j dS_ij k'_j,
// dk'_j = scale sum_i dS_ij q'_i, and the rotation is undone: dq = rot^T(dq'), dk = rot^T(dk').
//
// Three kernels over the forward's tile records (the same device schedule):
//   prep    D [H, T] = rowsum(dout * out), fp32
//   main    for 16-bit inputs pk_bwd_tc_kernel (pk_backward_tc.cu), or pk_bwd_mma_kernel
//           (below); for fp32 inputs pk_bwd_main_kernel:
//           per work item (tile record, head), persistent CTAs of 128 threads (two per SM),
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

#include <cstdlib>

#include "pk.h"
#include "pk_dev.cuh"

namespace pk {

cudaError_t backward_tc_prepare();
cudaError_t backward_tc_launch(bool bf16, const void* qkv, const void* cos_t, const void* sin_t, const uint32_t* cu,
                               long long T, int H, int window, float scale, const float* lse, const void* dout,
                               const float* D, float* dq, void* dqkv, const TileRec* tiles, Ctl* ctl, int sms,
                               cudaStream_t stream);

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

// the value of 16-bit storage bits (a shared-memory copy of an element)
template <int DT>
__device__ __forceinline__ float bits_f(uint16_t u) {
  if constexpr (DT == PK_BF16) {
    return __uint_as_float(static_cast<uint32_t>(u) << 16);
  } else {
    return __half2float(__ushort_as_half(u));
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

// D [h * T + t] = sum_d dout[t, h, d] out[t, h, d]. A row (t, h) is 64 contiguous elements of
// both arrays (rows of one token are contiguous too): L lanes read one row 16 bytes each
// (L = 8 for 16-bit types, 16 for fp32), so a warp reads 32 / L whole rows per load, and the
// row's lanes sum by shuffles.
template <int DT>
__global__ void __launch_bounds__(256) pk_bwd_prep_kernel(const void* __restrict__ out, const void* __restrict__ dout,
                                                          float* __restrict__ D, int H, long long T) {
  constexpr int kEl = DT == PK_F32 ? 4 : 8;  // elements per 16-byte piece
  constexpr int kLanes = kD / kEl;           // lanes per row
  constexpr int kRows = 32 / kLanes;         // rows per warp load
  const int lane = threadIdx.x & 31;
  const int sub = lane / kLanes, part = lane % kLanes;
  const long long n = T * H;
  const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long u0 = gw * kRows; u0 < n; u0 += nw * kRows) {
    const long long u = u0 + sub;  // row (t, h) = (u / H, u % H): element offset u * 64
    float acc = 0.f;
    if (u < n) {
      const uint4 o4 = *reinterpret_cast<const uint4*>(static_cast<const char*>(out) + (u * kD + part * kEl) * (DT == PK_F32 ? 4 : 2));
      const uint4 g4 = *reinterpret_cast<const uint4*>(static_cast<const char*>(dout) + (u * kD + part * kEl) * (DT == PK_F32 ? 4 : 2));
      const uint32_t ow[4] = {o4.x, o4.y, o4.z, o4.w}, gw4[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        if constexpr (DT == PK_F32) {
          acc = fmaf(__uint_as_float(ow[w]), __uint_as_float(gw4[w]), acc);
        } else if constexpr (DT == PK_BF16) {
          acc = fmaf(__uint_as_float(ow[w] << 16), __uint_as_float(gw4[w] << 16), acc);
          acc = fmaf(__uint_as_float(ow[w] & 0xffff0000u), __uint_as_float(gw4[w] & 0xffff0000u), acc);
        } else {
          acc = fmaf(__half2float(__ushort_as_half(static_cast<unsigned short>(ow[w] & 0xffffu))),
                     __half2float(__ushort_as_half(static_cast<unsigned short>(gw4[w] & 0xffffu))), acc);
          acc = fmaf(__half2float(__ushort_as_half(static_cast<unsigned short>(ow[w] >> 16))),
                     __half2float(__ushort_as_half(static_cast<unsigned short>(gw4[w] >> 16))), acc);
        }
      }
    }
#pragma unroll
    for (int o = kLanes / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (u < n && part == 0) D[static_cast<int64_t>(u % H) * T + u / H] = acc;
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

// ------------------------------------------------------------------------------------------
// The 16-bit backward on tensor cores (mma.sync m16n8k16, fp32 accumulation), FA2-style with
// the key tile owning the work: visibility is symmetric (same sequence, |i - j| <= w), so a
// tile record's rows serve as a key tile and its key range as the queries that see those keys.
// Per work item (record, head): 8 warps x 16 keys; the key tile's K' (rotated, rounded to the
// element type) and V stay in shared memory; queries come 32 at a time (Q', dout, lse, D).
// Per chunk each warp forms S^T = K' Q'^T and dP^T = V dout^T (16 MMAs each), P^T and dS^T in
// registers, and accumulates dV += P^T dout and dK' += dS^T Q' in registers; dS goes to shared
// memory and the CTA forms the chunk's dQ' = dS K' (warp w: dims 8w .. 8w+7), added to the fp32
// accumulator with atomics (other records' keys add to the same queries). dK' and dV of each key
// are complete at the end of the item: rotated back and written once. Fragments come by
// ldmatrix from [row][element] tiles whose rows start on 16 bytes (strides of 72 and 136
// elements keep the eight rows of each 8x8 load in distinct banks); the operands used
// transposed (dout and Q' for dV and dK', K' for dQ') come by transposing loads rather than
// transposed copies.

constexpr int kMmaWarps = 8;
constexpr int kMmaThreads = 32 * kMmaWarps;
constexpr int kQc = 32;          // queries per chunk
constexpr int kKP = kD + 8;      // row stride (16-bit elements) of [row][dim] tiles
constexpr int kKTP = kBR + 8;    // row stride of dS [query][key]
// K', V; two buffers of Q' and dout; dS; two raw staging buffers of q rows and of cos | sin rows
constexpr int kMmaSmemHalves = 2 * kBR * kKP + 4 * kQc * kKP + kQc * kKTP + 4 * kQc * kD;
constexpr int kMmaSmem = kMmaSmemHalves * 2 + 4 * kQc * 4;

template <int DT>
__device__ __forceinline__ uint16_t to16(float x) {
  if constexpr (DT == PK_BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  else return __half_as_ushort(__float2half_rn(x));
}
template <int DT>
__device__ __forceinline__ uint32_t pack16(float lo, float hi) {
  return static_cast<uint32_t>(to16<DT>(lo)) | (static_cast<uint32_t>(to16<DT>(hi)) << 16);
}
// four (two) 8x8 16-bit matrices from shared memory; lane l gives the address of one matrix row
__device__ __forceinline__ void ldsm4(const uint16_t* p, uint32_t (&r)[4]) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
// asynchronous global -> shared copy of kBytes (4 or 16) bytes; when `valid` is false nothing is
// read and the destination is filled with zeros
template <int kBytes>
__device__ __forceinline__ void cp_async(void* dst, const void* src, bool valid) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], %2, %3;" ::"r"(d), "l"(__cvta_generic_to_global(src)),
               "n"(kBytes), "r"(valid ? kBytes : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit_b() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all_b() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void ldsm4t(const uint16_t* p, uint32_t (&r)[4]) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
// the B fragments (16 x 8) of n-blocks n0 and n0 + 8 at k-step k0 from a row-major [k][n] tile
// (transposing load): r[0], r[1] for n0 and r[2], r[3] for n0 + 8
__device__ __forceinline__ void ldb2t(const uint16_t* tile, int stride, int n0, int k0, int lane, uint32_t (&r)[4]) {
  ldsm4t(tile + (k0 + (lane & 7) + 8 * ((lane >> 3) & 1)) * stride + n0 + 8 * (lane >> 4), r);
}
// the A fragment (16 x 16, row-major tile with `stride` elements per row) at (row0, col0)
__device__ __forceinline__ void lda(const uint16_t* tile, int stride, int row0, int col0, int lane, uint32_t (&r)[4]) {
  ldsm4(tile + (row0 + (lane & 7) + 8 * ((lane >> 3) & 1)) * stride + col0 + 8 * (lane >> 4), r);
}
// the B fragments (16 x 8, column-major: element (k, n) at tile[n][k]) of n-blocks n0 and n0 + 8
// at k-step k0: r[0], r[1] for n0 and r[2], r[3] for n0 + 8
__device__ __forceinline__ void ldb2(const uint16_t* tile, int stride, int n0, int k0, int lane, uint32_t (&r)[4]) {
  ldsm4(tile + (n0 + (lane & 7) + 8 * (lane >> 4)) * stride + k0 + 8 * ((lane >> 3) & 1), r);
}

// D += A B, m16n8k16, A row-major 16x16, B column-major 16x8, fp32 accumulators
template <int DT>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (DT == PK_BF16) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

template <int DT>
__global__ void __launch_bounds__(kMmaThreads, 2)
pk_bwd_mma_kernel(const void* __restrict__ qkv, const void* __restrict__ cos_t, const void* __restrict__ sin_t,
                  const uint32_t* __restrict__ cu, const TileRec* __restrict__ tiles, Ctl* ctl,
                  const float* __restrict__ lse, const void* __restrict__ dout, const float* __restrict__ D,
                  float* __restrict__ dq_acc, void* __restrict__ dqkv, int H, long long T, int window,
                  float scale) {
  extern __shared__ __align__(16) uint16_t mma_smem[];
  uint16_t* sK = mma_smem;                // [128][kKP]   K' (rotated)
  uint16_t* sV = sK + kBR * kKP;          // [128][kKP]   V
  uint16_t* sQ2 = sV + kBR * kKP;         // [2][32][kKP] Q' of the chunk (two buffers)
  uint16_t* sDO2 = sQ2 + 2 * kQc * kKP;   // [2][32][kKP] dout of the chunk
  uint16_t* sDS = sDO2 + 2 * kQc * kKP;   // [32][kKTP]   dS [query][key]
  uint16_t* rawX2 = sDS + kQc * kKTP;     // [2][32][64]  q rows as loaded
  uint16_t* rawCS2 = rawX2 + 2 * kQc * kD;  // [2][32][64]  cos (32) | sin (32) rows of the queries' positions
  float* sLse2 = reinterpret_cast<float*>(rawCS2 + 2 * kQc * kD);  // [2][32]
  float* sD2 = sLse2 + 2 * kQc;                                     // [2][32]
  __shared__ unsigned int s_item;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;
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
    const int nkeys = static_cast<int>(rec.rows);  // the record's rows are the key tile

    // stage the key tile: thread t rotates half the pairs of key row t / 2 and copies half its v
    {
      const int kr = tid >> 1, half = tid & 1;
      if (kr < nkeys) {
        const uint32_t b = rec.q0 + kr;
        const uint32_t sb = rec.kind == 0 ? rec.seq : seq_of_token(cu, rec.seq, rec.nseq, b);
        const int64_t pos = static_cast<int64_t>(b) - __ldg(cu + sb);
        const int64_t x = static_cast<int64_t>(b) * ldq + hd + h * kD;
        const int64_t v = static_cast<int64_t>(b) * ldq + 2 * hd + h * kD;
        for (int e = 0; e < 16; ++e) {
          const int u = half * 16 + e;
          const float c = ldf<DT>(cos_t, pos * kHalf + u), sn = ldf<DT>(sin_t, pos * kHalf + u);
          const float x1 = ldf<DT>(qkv, x + u), x2 = ldf<DT>(qkv, x + u + kHalf);
          const uint16_t y1 = to16<DT>(x1 * c - x2 * sn), y2 = to16<DT>(x1 * sn + x2 * c);
          sK[kr * kKP + u] = y1;
          sK[kr * kKP + u + kHalf] = y2;
        }
        for (int e = 0; e < 32; ++e)
          sV[kr * kKP + half * 32 + e] = static_cast<const uint16_t*>(qkv)[v + half * 32 + e];
      } else {
        for (int e = 0; e < 16; ++e) {
          const int u = half * 16 + e;
          sK[kr * kKP + u] = sK[kr * kKP + u + kHalf] = 0;
        }
        for (int e = 0; e < 32; ++e) sV[kr * kKP + half * 32 + e] = 0;
      }
    }
    // this thread's two keys (rows g and g + 8 of the warp's 16): validity and visible queries
    int64_t klo[2], khi[2], kstart[2];
    bool kok[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int kr = warp * 16 + g + 8 * e;
      kok[e] = kr < nkeys;
      klo[e] = khi[e] = kstart[e] = 0;
      if (kok[e]) {
        const uint32_t b = rec.q0 + kr;
        const uint32_t sb = rec.kind == 0 ? rec.seq : seq_of_token(cu, rec.seq, rec.nseq, b);
        const int64_t ss = __ldg(cu + sb), se = __ldg(cu + sb + 1);
        klo[e] = ss;
        kstart[e] = ss;
        khi[e] = se;
        if (window > 0) {
          klo[e] = max(ss, static_cast<int64_t>(b) - window);
          khi[e] = min(se, static_cast<int64_t>(b) + window + 1);
        }
      }
    }
    float dv[8][4], dk[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) dv[n][e] = dk[n][e] = 0.f;

    const uint32_t qend = rec.k0 + rec.nk;
    // chunk copies: thread (query row t / 8, 16-byte piece t % 8) copies its piece of the raw q
    // row, of the cos | sin rows at the query's position and of the dout row; lanes of piece 0
    // also copy lse and D. Chunk i + 1 is in flight while chunk i is computed.
    auto issue = [&](uint32_t qb, int buf) {
      const int qr = tid >> 3, part = tid & 7;
      const uint32_t a = qb + qr;
      const bool ok = a < qend;
      int64_t pos = 0;
      if (ok) {
        const uint32_t sa = rec.kind == 0 ? rec.seq : seq_of_token(cu, rec.seq, rec.nseq, a);
        pos = static_cast<int64_t>(a) - __ldg(cu + sa);
      }
      const int64_t ar = ok ? static_cast<int64_t>(a) : 0;
      const uint16_t* q16 = static_cast<const uint16_t*>(qkv);
      const uint16_t* c16 = static_cast<const uint16_t*>(part < 4 ? cos_t : sin_t);
      cp_async<16>(rawX2 + (buf * kQc + qr) * kD + part * 8, q16 + ar * ldq + h * kD + part * 8, ok);
      cp_async<16>(rawCS2 + (buf * kQc + qr) * kD + part * 8, c16 + pos * kHalf + (part & 3) * 8, ok);
      cp_async<16>(sDO2 + (buf * kQc + qr) * kKP + part * 8,
                   static_cast<const uint16_t*>(dout) + ar * hd + h * kD + part * 8, ok);
      if (part == 0) {
        cp_async<4>(sLse2 + buf * kQc + qr, lse + static_cast<int64_t>(h) * T + ar, ok);
        cp_async<4>(sD2 + buf * kQc + qr, D + static_cast<int64_t>(h) * T + ar, ok);
      }
      cp_async_commit_b();
    };
    if (rec.nk > 0) issue(rec.k0, 0);
    int ci = 0;
    for (uint32_t qb = rec.k0; qb < qend; qb += kQc, ++ci) {
      const int buf = ci & 1;
      uint16_t* sQ = sQ2 + buf * kQc * kKP;
      const uint16_t* sDO = sDO2 + buf * kQc * kKP;
      const float* sLse = sLse2 + buf * kQc;
      const float* sD = sD2 + buf * kQc;
      cp_async_wait_all_b();  // this chunk's copies (the only ones in flight)
      __syncthreads();        // ... visible to all; the previous chunk is done with sDS (and the key tile is staged)
      // rotate this chunk's q rows: thread (row t / 8, 4 rotary pairs)
      {
        const int qr = tid >> 3, part = tid & 7;
        const uint16_t* xr = rawX2 + (buf * kQc + qr) * kD;
        const uint16_t* cr = rawCS2 + (buf * kQc + qr) * kD;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int u = part * 4 + e;
          const float c = bits_f<DT>(cr[u]), sn = bits_f<DT>(cr[kHalf + u]);
          const float x1 = bits_f<DT>(xr[u]), x2 = bits_f<DT>(xr[u + kHalf]);
          sQ[qr * kKP + u] = to16<DT>(x1 * c - x2 * sn);
          sQ[qr * kKP + u + kHalf] = to16<DT>(x1 * sn + x2 * c);
        }
      }
      if (qb + kQc < qend) issue(qb + kQc, buf ^ 1);
      __syncthreads();  // this chunk's Q' is in place

      // S^T = K'_w Q'^T and dP^T = V_w dout^T: 16 keys x 32 queries (four n-blocks of 8)
      float st[4][4], dpt[4][4];
#pragma unroll
      for (int nb = 0; nb < 4; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e) st[nb][e] = dpt[nb][e] = 0.f;
      const int k0r = warp * 16;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t ak[4], av[4];
        lda(sK, kKP, k0r, 16 * kk, lane, ak);
        lda(sV, kKP, k0r, 16 * kk, lane, av);
#pragma unroll
        for (int nb = 0; nb < 4; nb += 2) {
          uint32_t bq[4], bo[4];
          ldb2(sQ, kKP, 8 * nb, 16 * kk, lane, bq);
          ldb2(sDO, kKP, 8 * nb, 16 * kk, lane, bo);
          mma16816<DT>(st[nb], ak, bq[0], bq[1]);
          mma16816<DT>(st[nb + 1], ak, bq[2], bq[3]);
          mma16816<DT>(dpt[nb], av, bo[0], bo[1]);
          mma16816<DT>(dpt[nb + 1], av, bo[2], bo[3]);
        }
      }
      // P^T and dS^T (element e of tile nb: key row g + 8 (e >> 1), query 8 nb + 2 t4 + (e & 1));
      // dS goes to shared memory as [query][key] for the dQ' product
#pragma unroll
      for (int nb = 0; nb < 4; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int kr = e >> 1;
          const int ql = 8 * nb + 2 * t4 + (e & 1);
          const int64_t a = static_cast<int64_t>(qb) + ql;
          float p = 0.f, ds = 0.f;
          if (kok[kr] && a < qend && a >= klo[kr] && a < khi[kr]) {
            p = __expf(scale * st[nb][e] - sLse[ql]);
            ds = p * (dpt[nb][e] - sD[ql]);
          }
          st[nb][e] = p;
          dpt[nb][e] = ds;
          sDS[ql * kKTP + k0r + g + 8 * kr] = to16<DT>(ds);
        }
      // dV += P^T dout and dK' += dS^T Q': A from the accumulators (two n-blocks = one k-step)
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        uint32_t ap[4], ad[4];
        ap[0] = pack16<DT>(st[2 * ks][0], st[2 * ks][1]);
        ap[1] = pack16<DT>(st[2 * ks][2], st[2 * ks][3]);
        ap[2] = pack16<DT>(st[2 * ks + 1][0], st[2 * ks + 1][1]);
        ap[3] = pack16<DT>(st[2 * ks + 1][2], st[2 * ks + 1][3]);
        ad[0] = pack16<DT>(dpt[2 * ks][0], dpt[2 * ks][1]);
        ad[1] = pack16<DT>(dpt[2 * ks][2], dpt[2 * ks][3]);
        ad[2] = pack16<DT>(dpt[2 * ks + 1][0], dpt[2 * ks + 1][1]);
        ad[3] = pack16<DT>(dpt[2 * ks + 1][2], dpt[2 * ks + 1][3]);
#pragma unroll
        for (int nd = 0; nd < 8; nd += 2) {
          uint32_t bo[4], bq[4];
          ldb2t(sDO, kKP, 8 * nd, 16 * ks, lane, bo);
          ldb2t(sQ, kKP, 8 * nd, 16 * ks, lane, bq);
          mma16816<DT>(dv[nd], ap, bo[0], bo[1]);
          mma16816<DT>(dv[nd + 1], ap, bo[2], bo[3]);
          mma16816<DT>(dk[nd], ad, bq[0], bq[1]);
          mma16816<DT>(dk[nd + 1], ad, bq[2], bq[3]);
        }
      }
      __syncthreads();  // every warp's dS is in shared memory
      // dQ' of the chunk, dims 8 warp .. 8 warp + 7: dS [32 x 128] K' [128 x 8]
      {
        float acc[2][4];
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[mb][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < kBR / 16; kk += 2) {
          // B of this warp's 8 dims for k-steps kk and kk + 1 (the x4 load's two "n-blocks" are
          // read here as two k-steps of one n-block: rows 8 warp .. + 7, columns 16 kk .. + 31)
          // B of this warp's 8 dims for k-steps kk and kk + 1 from K' [key][dim] (transposing
          // load): matrices at key rows 16 kk, 16 kk + 8, 16 kk + 16, 16 kk + 24
          uint32_t b[4];
          ldsm4t(sK + (16 * kk + (lane & 7) + 8 * (lane >> 3)) * kKP + 8 * warp, b);
#pragma unroll
          for (int mb = 0; mb < 2; ++mb) {
            uint32_t a4[4], a5[4];
            lda(sDS, kKTP, 16 * mb, 16 * kk, lane, a4);
            lda(sDS, kKTP, 16 * mb, 16 * kk + 16, lane, a5);
            mma16816<DT>(acc[mb], a4, b[0], b[1]);
            mma16816<DT>(acc[mb], a5, b[2], b[3]);
          }
        }
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int ql = 16 * mb + g + 8 * (e >> 1);
            const int64_t a = static_cast<int64_t>(qb) + ql;
            if (a < qend)
              atomicAdd(dq_acc + a * hd + h * kD + 8 * warp + 2 * t4 + (e & 1), scale * acc[mb][e]);
          }
      }
    }
    // dk = rot^T(dk') and dv of this warp's keys, rounded once and written to dqkv: this thread
    // holds dims 8 nd + 2 t4 + {0, 1} of its keys, so both members u and u + 32 of each rotary pair
    // (n-blocks nd and nd + 4)
#pragma unroll
    for (int kr = 0; kr < 2; ++kr) {
      if (!kok[kr]) continue;
      const int64_t b = static_cast<int64_t>(rec.q0) + warp * 16 + g + 8 * kr;
      const int64_t pos = b - kstart[kr];
      const int64_t row = b * ldq + h * kD;
#pragma unroll
      for (int nd = 0; nd < 4; ++nd) {
        float ya[2], yb[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int u = 8 * nd + 2 * t4 + i;
          const float c = ldf<DT>(cos_t, pos * kHalf + u), sn = ldf<DT>(sin_t, pos * kHalf + u);
          const float xa = scale * dk[nd][2 * kr + i], xb = scale * dk[nd + 4][2 * kr + i];
          ya[i] = fmaf(xa, c, xb * sn);
          yb[i] = fmaf(xb, c, -xa * sn);
        }
        stf2<DT>(dqkv, row + hd + 8 * nd + 2 * t4, ya[0], ya[1]);
        stf2<DT>(dqkv, row + hd + kHalf + 8 * nd + 2 * t4, yb[0], yb[1]);
      }
#pragma unroll
      for (int nd = 0; nd < 8; ++nd) stf2<DT>(dqkv, row + 2 * hd + 8 * nd + 2 * t4, dv[nd][2 * kr], dv[nd][2 * kr + 1]);
    }
  }
}

// dqkv: dq = rot^T(dq'), dk = rot^T(dk'), dv; one warp per token, lane l holding the rotary pair
// (l, l + 32) of a head vector (the halves' pairing), positions from cu
template <int DT>
__global__ void __launch_bounds__(256)
pk_bwd_finish_kernel(const void* __restrict__ cos_t, const void* __restrict__ sin_t, const uint32_t* __restrict__ cu,
                     int S, long long T, int H, const float* __restrict__ dq_acc, const float* __restrict__ dk_acc,
                     const float* __restrict__ dv_acc, void* __restrict__ dqkv, int dq_only) {
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
      const int64_t o = t * ldq + h * kD;
      const float y0 = fmaf(qa, c, qb * sn), y1 = fmaf(qb, c, -qa * sn);
      // lanes write pairs of neighbouring features: gather them by shuffle
      const float y01 = __shfl_down_sync(0xffffffffu, y0, 1), y11 = __shfl_down_sync(0xffffffffu, y1, 1);
      if ((lane & 1) == 0) {
        stf2<DT>(dqkv, o + lane, y0, y01);
        stf2<DT>(dqkv, o + lane + kHalf, y1, y11);
      }
      if (dq_only) continue;  // dk and dv were written by the main kernel
      const float ka = dk_acc[g + lane], kb = dk_acc[g + lane + kHalf];
      const float z0 = fmaf(ka, c, kb * sn), z1 = fmaf(kb, c, -ka * sn);
      const float z01 = __shfl_down_sync(0xffffffffu, z0, 1), z11 = __shfl_down_sync(0xffffffffu, z1, 1);
      if ((lane & 1) == 0) {
        stf2<DT>(dqkv, o + hd + lane, z0, z01);
        stf2<DT>(dqkv, o + hd + lane + kHalf, z1, z11);
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
  // the 16-bit types take the tensor-core kernel (dq' by atomics, dk' and dv written once); fp32
  // the CUDA-core one (dk' and dv by atomics, dq' written once)
  constexpr bool kMma = DT != PK_F32;
  cudaError_t e = kMma ? cudaMemsetAsync(dq, 0, static_cast<size_t>(T) * H * kD * sizeof(float), stream)
                       : cudaMemsetAsync(dk, 0, static_cast<size_t>(2) * T * H * kD * sizeof(float), stream);
  if (e != cudaSuccess) return e;
  const long long prep_blocks = min(static_cast<long long>(sms) * 8, (T * H + 31) / 32);
  pk_bwd_prep_kernel<DT><<<static_cast<unsigned int>(max(prep_blocks, 1ll)), 256, 0, stream>>>(out, dout, D, H, T);
  if constexpr (kMma) {
    // the tcgen05 kernel, or the mma.sync one for comparison (PK_BWD_MMA_SYNC=1)
    const char* legacy = std::getenv("PK_BWD_MMA_SYNC");
    if (legacy && legacy[0] == '1')
      pk_bwd_mma_kernel<DT><<<sms * 2, kMmaThreads, kMmaSmem, stream>>>(qkv, cos_t, sin_t, cu, tiles, ctl, lse, dout,
                                                                         D, dq, dqkv, H, T, window, scale);
    else if ((e = backward_tc_launch(DT == PK_BF16, qkv, cos_t, sin_t, cu, T, H, window, scale, lse, dout, D, dq, dqkv,
                                     tiles, ctl, sms, stream)) != cudaSuccess)
      return e;
  }
  else
    pk_bwd_main_kernel<DT><<<sms * 2, kBwdThreads, kBwdSmem, stream>>>(qkv, cos_t, sin_t, cu, tiles, ctl, lse, dout, D,
                                                                        dq, dk, dv, H, T, window, scale);
  const long long fin_blocks = min(static_cast<long long>(sms) * 8, (T + 7) / 8);
  pk_bwd_finish_kernel<DT><<<static_cast<unsigned int>(max(fin_blocks, 1ll)), 256, 0, stream>>>(
      cos_t, sin_t, cu, S, T, H, dq, dk, dv, dqkv, kMma ? 1 : 0);
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
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pk_bwd_mma_kernel<PK_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMmaSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pk_bwd_mma_kernel<PK_F16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMmaSmem);
  if (e == cudaSuccess) e = backward_tc_prepare();
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
