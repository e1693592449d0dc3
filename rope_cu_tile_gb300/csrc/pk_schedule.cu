// pk_schedule.cu -- device tile scheduler: cu -> tile records.
//
// Rule (hanzo-kernel packed.rs, fn layout and the key-range clipping of fn attend, with
// short sequences grouped):
//   - a sequence longer than kShort tokens is cut into 128-row pieces at rows 0, 128, ...
//     (fn layout); a piece's keys are the whole sequence, or with a window w the rows
//     [max(start, q0 - w), min(end, q0 + rows + w)) -- the union of its rows' windows;
//   - sequences of at most kShort tokens (empty ones included) whose first token falls in
//     the same kGrain-token granule form one group tile whose queries and keys are all of
//     their rows (at most 63 + 64 = 127 rows);
//   - records are listed by increasing first query token.
//
// The device computes this in parallel over granules: every record's first query token
// falls in exactly one granule [64 b, 64 b + 64), and a granule holds at most three:
// (i) a piece of the long sequence that covers the granule's first token, (ii) the group
// of short sequences starting in it, (iii) the first piece of a long sequence starting in
// it (a long sequence starting in a granule is the last one starting there, since it runs
// past the granule's end). One block of threads stages cu in shared memory (when it fits),
// takes contiguous runs of granules, counts, scans, then writes.
#include "pk_dev.cuh"

namespace pk {

namespace {

constexpr int kSchedThreads = 1024;
// cu is staged in shared memory when it has at most this many entries (192 KB); longer lists
// are searched in global memory
constexpr int kStageMax = 48 * 1024;

// cu as the caller's array in global memory (read-only path)
struct GlobalCu {
  const uint32_t* p;
};
__device__ __forceinline__ uint32_t ld_cu(GlobalCu cu, uint32_t i) { return __ldg(cu.p + i); }
// cu as the staged copy in shared memory
__device__ __forceinline__ uint32_t ld_cu(const uint32_t* cu, uint32_t i) { return cu[i]; }

// first index s in [0, n) with cu[s] >= v, or n
template <class CuPtr>
__device__ __forceinline__ uint32_t lower_bound_cu(CuPtr cu, uint32_t n, uint64_t v) {
  uint32_t lo = 0, hi = n;
  while (lo < hi) {
    const uint32_t mid = (lo + hi) >> 1;
    if (static_cast<uint64_t>(ld_cu(cu, mid)) < v) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// first index s in [0, n) with cu[s] > v, or n
template <class CuPtr>
__device__ __forceinline__ uint32_t upper_bound_cu(CuPtr cu, uint32_t n, uint64_t v) {
  uint32_t lo = 0, hi = n;
  while (lo < hi) {
    const uint32_t mid = (lo + hi) >> 1;
    if (static_cast<uint64_t>(ld_cu(cu, mid)) <= v) lo = mid + 1; else hi = mid;
  }
  return lo;
}

template <class CuPtr>
__device__ __forceinline__ TileRec piece(CuPtr cu, uint32_t s, uint32_t i0, int window) {
  const uint32_t start = ld_cu(cu, s), end = ld_cu(cu, s + 1);
  const uint32_t L = end - start;
  TileRec r;
  r.q0 = start + i0;
  r.rows = min(static_cast<uint32_t>(kBR), L - i0);
  uint64_t k0 = start, k1 = end;
  if (window > 0) {
    const uint64_t w = static_cast<uint64_t>(window);
    if (static_cast<uint64_t>(r.q0) > k0 + w) k0 = r.q0 - w;
    if (static_cast<uint64_t>(r.q0) + r.rows + w < k1) k1 = static_cast<uint64_t>(r.q0) + r.rows + w;
  }
  r.k0 = static_cast<uint32_t>(k0);
  r.nk = static_cast<uint32_t>(k1 - k0);
  r.seq = s;
  r.nseq = 1;
  r.kind = 0;
  r.ktiles = (r.nk + kBC - 1) / kBC;
  return r;
}

// Calls emit(record) for each record whose first query token falls in granule b, in
// increasing q0 (at most three; no array, so nothing goes to local memory).
template <class CuPtr, class Emit>
__device__ __forceinline__ void granule_visit(CuPtr cu, uint32_t S, int window, uint64_t b, Emit&& emit) {
  const uint64_t G0 = b * kGrain, G1 = G0 + kGrain;
  // (i) the sequence holding token G0, if it started earlier and is long
  {
    const uint32_t sc = upper_bound_cu(cu, S + 1, G0) - 1;  // largest s with cu[s] <= G0
    if (sc < S) {
      const uint64_t start = ld_cu(cu, sc), end = ld_cu(cu, sc + 1);
      if (start < G0 && end - start > static_cast<uint64_t>(kShort)) {
        const uint64_t i0 = ((G0 - start + kBR - 1) / kBR) * kBR;
        if (start + i0 < end && start + i0 < G1) emit(piece(cu, sc, static_cast<uint32_t>(i0), window));
      }
    }
  }
  // sequences whose first token falls in [G0, G1)
  const uint32_t s_lo = lower_bound_cu(cu, S, G0);
  const uint32_t s_hi = lower_bound_cu(cu, S, G1);
  if (s_lo < s_hi) {
    const uint32_t last = s_hi - 1;
    const bool last_long = ld_cu(cu, last + 1) - ld_cu(cu, last) > static_cast<uint32_t>(kShort);
    const uint32_t m_end = last_long ? last : s_hi;  // members [s_lo, m_end)
    if (m_end > s_lo) {
      const uint32_t q0 = ld_cu(cu, s_lo);
      const uint32_t rows = ld_cu(cu, m_end) - q0;
      if (rows > 0) {
        TileRec r;
        r.q0 = q0;
        r.rows = rows;
        r.k0 = q0;
        r.nk = rows;
        r.seq = s_lo;
        r.nseq = m_end - s_lo;
        r.kind = 1;
        r.ktiles = (rows + kBC - 1) / kBC;
        emit(r);
      }
    }
    if (last_long) emit(piece(cu, last, 0, window));
  }
}

// Count, scan and write the records, reading cu through `cu` (the staged shared copy or the
// caller's array; the body is instantiated for each so that loads use their own space).
template <class CuPtr>
__device__ __forceinline__ void schedule_body(CuPtr cu, int S, long long T, int window, TileRec* __restrict__ tiles,
                                              long long cap, Ctl* ctl, uint32_t* s_warp) {
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  const uint64_t NB = (static_cast<uint64_t>(T) + kGrain - 1) / kGrain;
  const uint64_t per = (NB + nthr - 1) / nthr;
  const uint64_t b0 = min(NB, per * tid), b1 = min(NB, b0 + per);
  // one granule per thread (T <= 64 x threads): its records stay in registers from the count
  // to the write; otherwise they are enumerated twice
  const bool single = per <= 1;
  TileRec g0{}, g1{}, g2{};
  uint32_t count = 0;
  if (single) {
    if (b0 < b1)
      granule_visit(cu, S, window, b0, [&](const TileRec& r) {
        if (count == 0)
          g0 = r;
        else if (count == 1)
          g1 = r;
        else
          g2 = r;
        ++count;
      });
  } else {
    for (uint64_t b = b0; b < b1; ++b) granule_visit(cu, S, window, b, [&](const TileRec&) { ++count; });
  }

  // exclusive scan of the per-thread counts
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t incl = count;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = nthr / 32;
    uint32_t x = lane < nw ? s_warp[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += v;
    }
    if (lane < nw) s_warp[lane] = x;  // inclusive over warps
  }
  __syncthreads();
  const uint32_t base = (warp ? s_warp[warp - 1] : 0u) + incl - count;
  const uint32_t total = s_warp[nthr / 32 - 1];

  uint32_t at = base;
  auto put = [&](const TileRec& r) {
    if (at < static_cast<uint64_t>(cap)) {
      uint4* d = reinterpret_cast<uint4*>(tiles + at);
      d[0] = make_uint4(r.q0, r.rows, r.k0, r.nk);
      d[1] = make_uint4(r.seq, r.nseq, r.kind, r.ktiles);
    }
    ++at;
  };
  if (single) {
    if (count > 0) put(g0);
    if (count > 1) put(g1);
    if (count > 2) put(g2);
  } else {
    for (uint64_t b = b0; b < b1; ++b) granule_visit(cu, S, window, b, put);
  }
  if (tid == 0) {
    if (total > static_cast<uint64_t>(cap)) {
      ctl->ntiles = 0;
      set_status(ctl, kErrInternal);
    } else {
      ctl->ntiles = total;
    }
    ctl->next = 0;
  }
}

}  // namespace

__global__ void __launch_bounds__(kSchedThreads)
pk_schedule_kernel(const uint32_t* __restrict__ cu_g, int S, long long T, int window,
                   TileRec* __restrict__ tiles, long long cap, Ctl* ctl) {
  extern __shared__ uint32_t s_cu[];
  __shared__ int s_bad;
  __shared__ uint32_t s_warp[kSchedThreads / 32];
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  // the attention kernel may start its set-up now; it reads the records only after this
  // grid has completed (griddep_wait)
  griddep_launch_dependents();
  const bool staged = S + 1 <= kStageMax;
  if (tid == 0) s_bad = 0;
  if (staged) {
    for (int s = tid; s <= S; s += nthr) s_cu[s] = __ldg(cu_g + s);
    __syncthreads();
    if (tid == 0 && (s_cu[0] != 0u || static_cast<long long>(s_cu[S]) != T)) s_bad = 1;
    for (int s = tid; s < S; s += nthr)
      if (s_cu[s + 1] < s_cu[s]) s_bad = 1;
  } else {
    __syncthreads();
    if (tid == 0 && (__ldg(cu_g) != 0u || static_cast<long long>(__ldg(cu_g + S)) != T)) s_bad = 1;
    for (int s = tid; s < S; s += nthr)
      if (__ldg(cu_g + s + 1) < __ldg(cu_g + s)) s_bad = 1;
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) {
      ctl->ntiles = 0;
      ctl->next = 0;
      set_status(ctl, kErrBadCu);
    }
    return;
  }
  if (staged)
    schedule_body(static_cast<const uint32_t*>(s_cu), S, T, window, tiles, cap, ctl, s_warp);
  else
    schedule_body(GlobalCu{cu_g}, S, T, window, tiles, cap, ctl, s_warp);
}

// The carve-out matches the attention kernel's (all shared memory), so that the SMs need
// no reconfiguration between the two kernels of a call.
cudaError_t schedule_prepare() {
  cudaError_t e = cudaFuncSetAttribute(pk_schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kStageMax * static_cast<int>(sizeof(uint32_t)));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(pk_schedule_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              cudaSharedmemCarveoutMaxShared);
}

cudaError_t schedule_launch(const uint32_t* cu, int S, long long T, int window, TileRec* tiles, long long cap,
                            Ctl* ctl, cudaStream_t stream) {
  const size_t smem = S + 1 <= kStageMax ? static_cast<size_t>(S + 1) * sizeof(uint32_t) : 0;
  pk_schedule_kernel<<<1, kSchedThreads, smem, stream>>>(cu, S, T, window, tiles, cap, ctl);
  return cudaGetLastError();
}

}  // namespace pk
