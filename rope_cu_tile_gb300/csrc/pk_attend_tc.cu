// pk_attend_tc.cu -- packed RoPE attention forward for bf16 / fp16 on tcgen05 (sm_103a).
//
// What it computes: hanzo-kernel 0.2.42 packed.rs fn attend -- a tile of query rows of
// one head against every key tile its window reaches, q and k rotated in the kernel
// ("the query tile, rotated and scaled"; "the key tile rotated, the value tile as is"),
// scores and the output product on the matrix units, the softmax online per row with
// masked keys weighing exactly zero, then out = O / l and lse = m + ln l.
//
// How (GB300): a persistent kernel, one 128-thread CTA per work item at a time, where an
// item is (tile record, head). For each item:
//   Q tile  : one TMA load of 128 rows x 64 columns straight from the strided qkv, 128-byte
//             swizzled; each thread rotates and scales its row in shared memory.
//   per key tile of 128 keys:
//     TMA K and V tiles; each thread rotates one key row in shared memory;
//     S = Q K^T   : tcgen05.mma kind::f16, M=128, N = keys rounded up to 16, into TMEM;
//     softmax     : thread r reads TMEM lane r (its query row), masks by its row's visible
//                   key interval, updates the running max m and sum l, writes P (rounded
//                   to the input type) to shared memory in the MMA's K-major layout;
//     O_t = P V   : tcgen05.mma with V as an MN-major operand, into TMEM; each thread adds
//                   it to its register accumulator, rescaled by exp(m_old - m_new).
//   epilogue: out row = O / l (16-byte stores), lse = m + ln l.
// Every mbarrier wait is bounded; on timeout the CTA records PK_ERR_TIMEOUT, stops
// issuing work, waits (bounded) for its own copies and MMAs in flight, frees its tensor
// memory and returns.
#include "pk_dev.cuh"

namespace pk {

namespace {

constexpr int kThreads = 128;
constexpr uint32_t kTileBytes = 128 * 128;      // 128 rows x 64 elements x 2 bytes
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileBytes;
constexpr uint32_t kOffV = kOffK + kTileBytes;
constexpr uint32_t kOffP = kOffV + kTileBytes;  // two 64-key halves
constexpr uint32_t kOffBar = kOffP + 2 * kTileBytes;
constexpr uint32_t kSmemUsed = kOffBar + 64;
constexpr uint32_t kTmemCols = 256;             // S: [0, 128), O tile: [128, 192)
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNeg = -1.0e30f;                // running-max start: exp2 of (kNeg - real) is 0

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Rotate (and scale) row r of a 128-byte-swizzled 64-column tile in place: elements u and
// u + 32 are logical 16-byte chunks c and c + 4, stored at chunks (c ^ (r & 7)) and
// ((c + 4) ^ (r & 7)).
template <bool BF16>
__device__ __forceinline__ void rope_row_sw128(uint8_t* tile, int r, const uint16_t* cos_row,
                                               const uint16_t* sin_row, float mul) {
  uint8_t* row = tile + r * 128;
  const int sw = r & 7;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4* p1 = reinterpret_cast<uint4*>(row + ((c ^ sw) << 4));
    uint4* p2 = reinterpret_cast<uint4*>(row + (((c + 4) ^ sw) << 4));
    const uint4 x1 = *p1, x2 = *p2;
    const uint4 cv = __ldg(reinterpret_cast<const uint4*>(cos_row) + c);
    const uint4 sv = __ldg(reinterpret_cast<const uint4*>(sin_row) + c);
    const uint32_t a[4] = {x1.x, x1.y, x1.z, x1.w};
    const uint32_t b[4] = {x2.x, x2.y, x2.z, x2.w};
    const uint32_t cc[4] = {cv.x, cv.y, cv.z, cv.w};
    const uint32_t ss[4] = {sv.x, sv.y, sv.z, sv.w};
    uint32_t y1[4], y2[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 xa = Elem<BF16>::unpack(a[k]);
      const float2 xb = Elem<BF16>::unpack(b[k]);
      const float2 c2 = Elem<BF16>::unpack(cc[k]);
      const float2 s2 = Elem<BF16>::unpack(ss[k]);
      const float lo1 = (xa.x * c2.x - xb.x * s2.x) * mul;
      const float hi1 = (xa.y * c2.y - xb.y * s2.y) * mul;
      const float lo2 = (xa.x * s2.x + xb.x * c2.x) * mul;
      const float hi2 = (xa.y * s2.y + xb.y * c2.y) * mul;
      y1[k] = Elem<BF16>::pack(lo1, hi1);
      y2[k] = Elem<BF16>::pack(lo2, hi2);
    }
    *p1 = make_uint4(y1[0], y1[1], y1[2], y1[3]);
    *p2 = make_uint4(y2[0], y2[1], y2[2], y2[3]);
  }
}

}  // namespace

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
pk_attend_tc_kernel(const __grid_constant__ CUtensorMap tmap_qkv,
                    const uint16_t* __restrict__ cos_t, const uint16_t* __restrict__ sin_t,
                    const uint32_t* __restrict__ cu, const TileRec* __restrict__ tiles,
                    uint16_t* __restrict__ out, float* __restrict__ lse, Ctl* ctl, int H,
                    long long T, int window, float scale, unsigned long long timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sK = smem + kOffK;
  uint8_t* sP = smem + kOffP;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffBar + 32);
  uint32_t* s_item = s_tmem + 1;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const uint32_t bar_q = smem_u32(&bars[0]);
  const uint32_t bar_kv = smem_u32(&bars[1]);
  const uint32_t bar_mma = smem_u32(&bars[2]);
  const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(smem + kOffV),
                 aP = smem_u32(sP);

  if (tid == 0) {
    tma_prefetch_desc(&tmap_qkv);
    mbar_init(bar_q, 1);
    mbar_init(bar_kv, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(s_tmem), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

  // the schedule kernel ran before this one in stream order
  const unsigned int n_items = __ldcg(&ctl->ntiles) * static_cast<unsigned int>(H);
  const int64_t hd = static_cast<int64_t>(H) * kD;
  const uint32_t idesc_pv = idesc_f16(BF16, 128, 64, false, true);

  uint32_t ph_q = 0, ph_kv = 0, ph_mma = 0;
  bool pend_q = false, pend_kv = false, pend_mma = false;  // thread 0: ops not yet waited on
  bool bad = false;

  for (;;) {
    if (tid == 0) *s_item = atomicAdd(&ctl->next, 1u);
    if (__syncthreads_or(bad)) break;
    const unsigned int item = *s_item;
    if (item >= n_items) break;
    const unsigned int ti = item / static_cast<unsigned int>(H);
    const int h = static_cast<int>(item % static_cast<unsigned int>(H));
    const TileRec rec = tiles[ti];

    if (tid == 0) {
      mbar_arrive_expect_tx(bar_q, kTileBytes);
      tma_load_2d(aQ, &tmap_qkv, bar_q, h * kD, static_cast<int32_t>(rec.q0));
      pend_q = true;
    }
    // this thread's query row: its sequence and visible key interval [lo, hi)
    const int r = tid;
    const bool row_ok = r < static_cast<int>(rec.rows);
    const uint32_t a = rec.q0 + r;
    int64_t lo = 0, hi = 0;
    uint32_t qpos = 0;
    if (row_ok) {
      const uint32_t s = rec.kind == 0 ? rec.seq : seq_of_token(cu, rec.seq, rec.nseq, a);
      const int64_t ss = __ldg(cu + s), se = __ldg(cu + s + 1);
      qpos = a - static_cast<uint32_t>(ss);
      lo = ss;
      hi = se;
      if (window > 0) {
        lo = max(ss, static_cast<int64_t>(a) - window);
        hi = min(se, static_cast<int64_t>(a) + window + 1);
      }
    }
    bad |= !mbar_wait(bar_q, ph_q, timeout_ns, bad);
    ph_q ^= 1;
    if (tid == 0) pend_q = bad;
    if (row_ok) rope_row_sw128<BF16>(sQ, r, cos_t + qpos * kHalf, sin_t + qpos * kHalf, scale);
    fence_proxy_async_smem();

    float o[kD];
#pragma unroll
    for (int d = 0; d < kD; ++d) o[d] = 0.f;
    float m = kNeg, l = 0.f;
    const uint32_t seq0_start = __ldg(cu + rec.seq);

    for (uint32_t kt = 0; kt < rec.ktiles; ++kt) {
      const uint32_t j0 = rec.k0 + kt * kBC;
      const uint32_t nkeys = min(static_cast<uint32_t>(kBC), rec.k0 + rec.nk - j0);
      const uint32_t n16 = (nkeys + 15u) & ~15u;
      if (tid == 0 && !bad) {
        mbar_arrive_expect_tx(bar_kv, 2 * kTileBytes);
        tma_load_2d(aK, &tmap_qkv, bar_kv, static_cast<int32_t>(hd + h * kD), static_cast<int32_t>(j0));
        tma_load_2d(aV, &tmap_qkv, bar_kv, static_cast<int32_t>(2 * hd + h * kD), static_cast<int32_t>(j0));
        pend_kv = true;
      }
      bad |= !mbar_wait(bar_kv, ph_kv, timeout_ns, bad);
      ph_kv ^= 1;
      if (tid == 0) pend_kv = bad;
      // rotate key row r
      if (r < static_cast<int>(nkeys)) {
        const uint32_t b = j0 + r;
        const uint32_t sk = rec.kind == 0 ? rec.seq : seq_of_token(cu, rec.seq, rec.nseq, b);
        const uint32_t kpos = b - (rec.kind == 0 ? seq0_start : __ldg(cu + sk));
        rope_row_sw128<BF16>(sK, r, cos_t + kpos * kHalf, sin_t + kpos * kHalf, 1.0f);
      }
      fence_proxy_async_smem();
      if (__syncthreads_or(bad)) break;

      // S = Q K^T
      if (tid == 0) {
        tc_fence_after();
        const uint32_t idesc = idesc_f16(BF16, 128, n16, false, false);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_f16_ss(tmem + kColS, sdesc_sw128(aQ + ks * 32, 16, 1024),
                      sdesc_sw128(aK + ks * 32, 16, 1024), idesc, ks > 0);
        umma_commit(bar_mma);
        pend_mma = true;
      }
      bad |= !mbar_wait(bar_mma, ph_mma, timeout_ns, bad);
      ph_mma ^= 1;
      if (tid == 0) pend_mma = bad;
      tc_fence_after();

      // visible columns of this row in this key tile: [c_lo, c_hi)
      const int c_lo = static_cast<int>(max(lo - static_cast<int64_t>(j0), static_cast<int64_t>(0)));
      const int c_hi = static_cast<int>(min(hi - static_cast<int64_t>(j0), static_cast<int64_t>(nkeys)));
      // pass 1: the row max over visible columns
      float mx = kNeg;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        if (ch * 32 >= static_cast<int>(n16)) break;
        float v[32];
        tmem_ld32(tmem + lane_base + kColS + ch * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int c = ch * 32 + i;
          if (c >= c_lo && c < c_hi) mx = fmaxf(mx, v[i]);
        }
      }
      const float m_new = fmaxf(m, mx);
      const float alpha = ex2((m - m_new) * kLog2e);
      const float mb = m_new * kLog2e;
      // pass 2: probabilities, their sum, P to shared memory (K-major, 128-byte swizzle)
      float sum = 0.f;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        if (ch * 32 >= static_cast<int>(n16)) break;
        float v[32];
        tmem_ld32(tmem + lane_base + kColS + ch * 32, v);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const int c = ch * 32 + i;
          const float p0 = (c >= c_lo && c < c_hi) ? ex2(fmaf(v[i], kLog2e, -mb)) : 0.f;
          const float p1 = (c + 1 >= c_lo && c + 1 < c_hi) ? ex2(fmaf(v[i + 1], kLog2e, -mb)) : 0.f;
          sum += p0 + p1;
          pk[i / 2] = Elem<BF16>::pack(p0, p1);
        }
        // 32 columns = 4 chunks of 8; column block ch covers half ch / 2, chunks (ch & 1) * 4 ..
        uint8_t* prow = sP + (ch >> 1) * kTileBytes + r * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int chunk = (ch & 1) * 4 + q;
          *reinterpret_cast<uint4*>(prow + ((chunk ^ (r & 7)) << 4)) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
      l = l * alpha + sum;
      m = m_new;
      fence_proxy_async_smem();
      tc_fence_before();
      if (__syncthreads_or(bad)) break;

      // O_t = P V
      if (tid == 0) {
        tc_fence_after();
        const int ksteps = static_cast<int>(n16 / 16);
        for (int ks = 0; ks < ksteps; ++ks)
          umma_f16_ss(tmem + kColO, sdesc_sw128(aP + (ks >> 2) * kTileBytes + (ks & 3) * 32, 16, 1024),
                      sdesc_sw128(aV + ks * 2048, 8192, 1024), idesc_pv, ks > 0);
        umma_commit(bar_mma);
        pend_mma = true;
      }
      bad |= !mbar_wait(bar_mma, ph_mma, timeout_ns, bad);
      ph_mma ^= 1;
      if (tid == 0) pend_mma = bad;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        float v[32];
        tmem_ld32(tmem + lane_base + kColO + ch * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[ch * 32 + i] = fmaf(o[ch * 32 + i], alpha, v[i]);
      }
      tc_fence_before();
    }
    if (__syncthreads_or(bad)) break;

    // epilogue
    if (row_ok) {
      const float inv = 1.0f / l;
      uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<int64_t>(a) * hd + h * kD));
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        dst[q] = make_uint4(Elem<BF16>::pack(o[8 * q + 0] * inv, o[8 * q + 1] * inv),
                            Elem<BF16>::pack(o[8 * q + 2] * inv, o[8 * q + 3] * inv),
                            Elem<BF16>::pack(o[8 * q + 4] * inv, o[8 * q + 5] * inv),
                            Elem<BF16>::pack(o[8 * q + 6] * inv, o[8 * q + 7] * inv));
      }
      lse[static_cast<int64_t>(h) * T + a] = m + lg2(l) * kLn2;
    }
  }

  if (bad) {
    if (tid == 0) {
      set_status(ctl, kErrTimeout);
      // let this CTA's own copies and MMAs land before its memory goes away
      if (pend_q) mbar_wait(bar_q, ph_q ^ 1, timeout_ns);
      if (pend_kv) mbar_wait(bar_kv, ph_kv ^ 1, timeout_ns);
      if (pend_mma) mbar_wait(bar_mma, ph_mma ^ 1, timeout_ns);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

uint32_t attend_tc_smem_bytes() { return kSmemUsed + 1024; }

// Host side: opt in to the dynamic shared memory once per device.
cudaError_t attend_tc_prepare() {
  const int smem = static_cast<int>(attend_tc_smem_bytes());
  cudaError_t e = cudaFuncSetAttribute(pk_attend_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(pk_attend_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

// Host side: one launch over `grid` persistent CTAs.
cudaError_t attend_tc_launch(bool bf16, const CUtensorMap& tmap, const void* cos_t, const void* sin_t,
                             const uint32_t* cu, const TileRec* tiles, void* out, float* lse, Ctl* ctl, int H,
                             long long T, int window, float scale, unsigned long long timeout_ns, int grid,
                             cudaStream_t stream) {
  const uint32_t smem = attend_tc_smem_bytes();
  const uint16_t* c = static_cast<const uint16_t*>(cos_t);
  const uint16_t* s = static_cast<const uint16_t*>(sin_t);
  uint16_t* o = static_cast<uint16_t*>(out);
  if (bf16)
    pk_attend_tc_kernel<true><<<grid, kThreads, smem, stream>>>(tmap, c, s, cu, tiles, o, lse, ctl, H, T, window,
                                                                scale, timeout_ns);
  else
    pk_attend_tc_kernel<false><<<grid, kThreads, smem, stream>>>(tmap, c, s, cu, tiles, o, lse, ctl, H, T, window,
                                                                 scale, timeout_ns);
  return cudaGetLastError();
}

}  // namespace pk
