// pk_attn_common.cuh -- device helpers shared by the attention kernels for sm_103a:
// bounded barrier waits that watch a CTA-wide abort flag, exp2 / log2 / max3, the staged
// member offsets of a tile record, cos / sin table rows fetched into shared memory, and the
// half-split rotation of a 128-byte-swizzled 64-column tile row in place.
//
// The rotation: packed.rs fn attend applies to the query tile "rotated and scaled" and to
// the key tile "rotated" the pair rotation (u, u + 32) at the token's in-sequence position:
//     y[u] = x[u] c - x[u + 32] s,   y[u + 32] = x[u] s + x[u + 32] c   (u < 32)
// with c, s the cos / sin table entries of that position.
#pragma once

#include "pk_dev.cuh"

namespace pk {
namespace attn {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNeg = -1.0e30f;      // running-max start: ex2 of (masked - kNeg) stays 0
constexpr float kRescale = 8.0f;      // rescale O only when the max grows by more than 2^8
constexpr uint32_t kSleepNs = 20000;  // longest sleep of a waiting thread between checks
constexpr uint32_t kRowTblBytes = 128;  // cos (64 B) + sin (64 B) of one position, 16-bit
constexpr int kCuStage = kBR + 2;       // staged member offsets of a group of up to 128 sequences

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
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float y;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}

// ------------------------------------------------------------------------------------
// bounded waits

__device__ __forceinline__ bool aborted(const int32_t* flag) { return *reinterpret_cast<const volatile int32_t*>(flag) != 0; }
__device__ __forceinline__ void raise_abort(int32_t* flag, Ctl* ctl) {
  *reinterpret_cast<volatile int32_t*>(flag) = 1;
  set_status(ctl, kErrTimeout);
}

// Wait for phase `parity` of `bar`, giving up (false) once the CTA's abort flag is up or
// after `timeout_ns` (which raises the flag and records PK_ERR_TIMEOUT).
__device__ __forceinline__ bool wait_bar(int32_t* flag, Ctl* ctl, uint64_t* bar, uint32_t parity,
                                         uint64_t timeout_ns) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_sleep(a, parity, kSleepNs)) return true;
    if ((i & 7u) == 0u) {
      if (aborted(flag)) return false;
      if (globaltimer_ns() - t0 > timeout_ns) {
        raise_abort(flag, ctl);
        return false;
      }
    }
  }
}

__device__ __forceinline__ uint32_t round16(uint32_t n) { return (n + 15u) & ~15u; }

// ------------------------------------------------------------------------------------
// member sequences of a record

// The offsets cu[rec.seq .. rec.seq + rec.nseq], copied by `nthr` threads into `dst` when
// they fit (a group can hold any number of empty sequences; past kCuStage - 1 members only
// the first offset is staged).
__device__ __forceinline__ bool staged_all(const TileRec& rec) { return rec.nseq + 1 <= kCuStage; }
__device__ __forceinline__ void stage_cu(const uint32_t* cu, const TileRec& rec, uint32_t* dst, int t, int nthr) {
  const int n = staged_all(rec) ? static_cast<int>(rec.nseq) : 0;
  for (int i = t; i <= n; i += nthr) dst[i] = __ldg(cu + rec.seq + i);
}

// The member (index into a staged offset list of n + 1 values) holding token a: the last
// i < n with off[i] <= a.
__device__ __forceinline__ int staged_seq(const uint32_t* off, int n, uint32_t a) {
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

// Start and end tokens of the member sequence of group `rec` holding token a, from the
// staged offsets when they are all there, else from cu in global memory.
__device__ __forceinline__ void group_bounds(const uint32_t* cu, const TileRec& rec, const uint32_t* off, uint32_t a,
                                             uint32_t& ss, uint32_t& se) {
  if (staged_all(rec)) {
    const int i = staged_seq(off, static_cast<int>(rec.nseq), a);
    ss = off[i];
    se = off[i + 1];
  } else {
    const uint32_t sq = seq_of_token(cu, rec.seq, rec.nseq, a);
    ss = __ldg(cu + sq);
    se = __ldg(cu + sq + 1);
  }
}

// ------------------------------------------------------------------------------------
// table rows in shared memory (cp.async, 16 bytes at a time, through L1: the rows of short
// sequences are the same few table rows for every thread)

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// The cos and sin rows of position `pos` (32 16-bit values each) into the 128-byte buffer
// `buf`: logical chunk k (cos 0..3, sin 4..7) at 16-byte slot k ^ (t & 7), so eight threads
// of a quarter warp reading the same chunk hit eight different bank groups.
__device__ __forceinline__ void fetch_table_row(const uint16_t* cos_t, const uint16_t* sin_t, uint32_t buf,
                                                uint32_t pos, int t) {
  const uint16_t* c = cos_t + static_cast<size_t>(pos) * kHalf;
  const uint16_t* s = sin_t + static_cast<size_t>(pos) * kHalf;
  const int sw = t & 7;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    cp_async16(buf + ((k ^ sw) << 4), c + 8 * k);
    cp_async16(buf + (((k + 4) ^ sw) << 4), s + 8 * k);
  }
}

// Rotation of one 16-byte chunk pair: x1 holds elements u .. u+7 of the first half of a
// row, x2 the matching elements u+32 .. u+39, tc / ts the table values of the same u;
// y1 = x1 c - x2 s, y2 = x1 s + x2 c in fp32 from the 16-bit operands, times `mul` when
// SCALED, each rounded once to the element type.
template <bool BF16, bool SCALED>
__device__ __forceinline__ void rope_chunk(const uint4& x1, const uint4& x2, const uint4& tc, const uint4& ts,
                                           float mul, uint4& y1o, uint4& y2o) {
  using E = Elem<BF16>;
  const uint32_t a[4] = {x1.x, x1.y, x1.z, x1.w};
  const uint32_t b[4] = {x2.x, x2.y, x2.z, x2.w};
  const uint32_t cc[4] = {tc.x, tc.y, tc.z, tc.w};
  const uint32_t ss[4] = {ts.x, ts.y, ts.z, ts.w};
  uint32_t y1[4], y2[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float lo1 = E::fma_lo(a[k], cc[k], -E::fma_lo(b[k], ss[k], 0.f));
    float hi1 = E::fma_hi(a[k], cc[k], -E::fma_hi(b[k], ss[k], 0.f));
    float lo2 = E::fma_lo(a[k], ss[k], E::fma_lo(b[k], cc[k], 0.f));
    float hi2 = E::fma_hi(a[k], ss[k], E::fma_hi(b[k], cc[k], 0.f));
    if (SCALED) {
      lo1 *= mul;
      hi1 *= mul;
      lo2 *= mul;
      hi2 *= mul;
    }
    y1[k] = E::pack(lo1, hi1);
    y2[k] = E::pack(lo2, hi2);
  }
  y1o = make_uint4(y1[0], y1[1], y1[2], y1[3]);
  y2o = make_uint4(y2[0], y2[1], y2[2], y2[3]);
}

// Rotate (and multiply by `mul` unless it is 1) row r of a 128-byte-swizzled 64-column tile
// in place. Elements u and u + 32 are logical 16-byte chunks c and c + 4, stored at chunks
// (c ^ (r & 7)) and ((c + 4) ^ (r & 7)); the table row is in `tbl` as fetch_table_row left
// it for thread t.
template <bool BF16>
__device__ __forceinline__ void rope_row(uint8_t* tile, int r, const uint8_t* tbl, int t, float mul) {
  uint8_t* row = tile + r * 128;
  const int sw = r & 7, tw = t & 7;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    const uint4 x1 = *reinterpret_cast<const uint4*>(row + ((c ^ sw) << 4));
    const uint4 x2 = *reinterpret_cast<const uint4*>(row + (((c + 4) ^ sw) << 4));
    const uint4 tc = *reinterpret_cast<const uint4*>(tbl + ((c ^ tw) << 4));
    const uint4 ts = *reinterpret_cast<const uint4*>(tbl + (((c + 4) ^ tw) << 4));
    uint4 y1, y2;
    if (mul == 1.0f)
      rope_chunk<BF16, false>(x1, x2, tc, ts, mul, y1, y2);
    else
      rope_chunk<BF16, true>(x1, x2, tc, ts, mul, y1, y2);
    *reinterpret_cast<uint4*>(row + ((c ^ sw) << 4)) = y1;
    *reinterpret_cast<uint4*>(row + (((c + 4) ^ sw) << 4)) = y2;
  }
}

}  // namespace attn
}  // namespace pk
