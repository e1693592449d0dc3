// pk_schedule.cu -- device tile scheduler: cu -> tile records.
//
// Rule (hanzo-kernel packed.rs, fn layout and the key-range clipping of fn attend, with
// short sequences grouped):
//   - a sequence longer than kShort tokens is cut into 128-row pieces at rows 0, 128, ...
//     (fn layout); a piece's keys are the whole sequence, or with a window w the rows
//     [max(start, q0 - w), min(end, q0 + rows + w)) -- the union of its rows' windows;
//   - sequences of at most kShort tokens (empty ones included) are grouped within
//     kWin-token windows, a sequence belonging to the window of its first token: in order,
//     a group takes the next sequence while that one is short, belongs to the group's
//     window and keeps the group within 128 rows (greedy packing); a group tile's queries
//     and keys are all of its rows, and a group of empty sequences only gives no record;
//   - records are listed by increasing first query token.
//
// The device computes this in parallel over windows: every record's first query token
// falls in exactly one window [kWin w, kWin w + kWin), which holds (i) the pieces of the
// long sequence that covers the window's first token, if it started earlier, then (ii) the
// records of the sequences starting in it, found by one walk over them. One block of
// threads stages cu in shared memory (when it fits); each warp walks a contiguous run of
// windows (its lanes test 32 candidate group members at once and write pieces side by
// side), counts, the warps' counts are scanned, then the warps walk again to write.
#include <cooperative_groups.h>

#include "pk_dev.cuh"

namespace cg = cooperative_groups;

namespace pk {

namespace {

constexpr int kSchedThreads = 32 * kSchedWarps;
// cu is staged in shared memory when it has at most this many entries (192 KB); longer lists
// are searched in global memory
constexpr int kStageMax = 48 * 1024;
// dynamic shared memory the scheduler may use: staged cu, then (when they fit) the record
// slots of the block's warps
constexpr int kSchedSmem = 200 * 1024;

// cu as the caller's array in global memory (read-only path)
struct GlobalCu {
  const uint32_t* p;
};
__device__ __forceinline__ uint32_t ld_cu(GlobalCu cu, uint32_t i) { return __ldg(cu.p + i); }
// cu as the staged copy in shared memory
__device__ __forceinline__ uint32_t ld_cu(const uint32_t* cu, uint32_t i) { return cu[i]; }

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

// The record sink of a warp's walk: every lane calls it with the same arguments, and the
// write position stays warp-uniform.
struct WriteSink {
  TileRec* tiles;
  uint64_t cap;
  uint32_t at;
  __device__ __forceinline__ void put(uint32_t i, const TileRec& r) const {
    if (i < cap) {
      uint4* d = reinterpret_cast<uint4*>(tiles + i);
      d[0] = make_uint4(r.q0, r.rows, r.k0, r.nk);
      d[1] = make_uint4(r.seq, r.nseq, r.kind, r.ktiles);
    }
  }
  // k pieces of sequence s at rows i0, i0 + 128, ...: lane l writes pieces l, l + 32, ...
  template <class CuPtr>
  __device__ __forceinline__ void pieces(CuPtr cu, uint32_t s, uint32_t i0, uint32_t k, int window, int lane) {
    for (uint32_t i = lane; i < k; i += 32) put(at + i, piece(cu, s, i0 + i * kBR, window));
    at += k;
  }
  __device__ __forceinline__ void group(uint32_t s, uint32_t e, uint32_t c0, uint32_t ce, int lane) {
    if (lane == 0) {
      TileRec r;
      r.q0 = c0;
      r.rows = ce - c0;
      r.k0 = c0;
      r.nk = ce - c0;
      r.seq = s;
      r.nseq = e - s;
      r.kind = 1;
      r.ktiles = (r.rows + kBC - 1) / kBC;
      put(at, r);
    }
    ++at;
  }
};

// First index i in [lo, hi) with cu[i] >= v (strict: cu[i] > v), or hi, found by the
// lanes of a warp together: each round splits [lo, hi) into 32 blocks, tests the last entry
// of each, and keeps the first block whose test holds (a 32-way search: about three
// dependent loads for 32K entries). Called by every lane with the same arguments.
template <class CuPtr>
__device__ __forceinline__ uint32_t warp_search(CuPtr cu, uint32_t lo, uint32_t hi, uint64_t v, bool strict,
                                                int lane) {
  while (lo < hi) {
    const uint32_t step = (hi - lo + 31) / 32;
    const uint64_t end = static_cast<uint64_t>(lo) + static_cast<uint64_t>(lane + 1) * step;
    const uint32_t q = static_cast<uint32_t>(min(end, static_cast<uint64_t>(hi))) - 1;  // last of block `lane`
    bool pred = false;
    if (static_cast<uint64_t>(lo) + static_cast<uint64_t>(lane) * step < hi) {
      const uint64_t c = ld_cu(cu, q);
      pred = strict ? c > v : c >= v;
    }
    const unsigned int m = __ballot_sync(0xffffffffu, pred);
    if (m == 0u) return hi;
    const uint32_t k = static_cast<uint32_t>(__ffs(m) - 1);
    const uint32_t qk = static_cast<uint32_t>(min(static_cast<uint64_t>(lo) + static_cast<uint64_t>(k + 1) * step,
                                                  static_cast<uint64_t>(hi))) - 1;
    lo += k * step;  // the answer is in [lo + k step, qk], and qk holds
    hi = qk;
  }
  return hi;
}

// One warp walks window w = [kWin w, kWin w + kWin) and hands its records to the sink in
// increasing q0. The sequences starting in the window are read 32 at a time (lane l holds
// sequence base + l); groups are closed with ballots over those registers.
template <class CuPtr, class Sink>
__device__ __forceinline__ void window_visit(CuPtr cu, uint32_t S, int window, uint64_t w, int lane, Sink& sink) {
  const uint64_t W0 = w * kWin, W1 = W0 + kWin;
  const uint32_t s_lo = warp_search(cu, 0u, S, W0, false, lane);  // first sequence starting at or after W0
  const uint32_t s_hi = warp_search(cu, s_lo, S, W1, false, lane);
  // (i) the pieces in this window of the long sequence holding token W0, if it started
  // earlier: the last sequence starting before W0, when the next one starts after W0
  if (s_lo > 0 && (s_lo == S || ld_cu(cu, s_lo) > W0)) {
    const uint32_t sc = s_lo - 1;
    const uint64_t start = ld_cu(cu, sc), end = ld_cu(cu, sc + 1);
    if (end - start > static_cast<uint64_t>(kShort)) {
      const uint64_t i0 = ((W0 - start + kBR - 1) / kBR) * kBR;
      const uint64_t lim = min(end, W1) - start;  // pieces start below lim
      if (i0 < lim)
        sink.pieces(cu, sc, static_cast<uint32_t>(i0), static_cast<uint32_t>((lim - i0 + kBR - 1) / kBR), window, lane);
    }
  }
  // (ii) the sequences starting in [W0, W1), in order
  bool open = false;    // a group is open: first member gs, first token g0
  uint32_t gs = 0, g0 = 0;
  for (uint32_t base = s_lo; base < s_hi; base += 32) {
    const uint32_t j = base + static_cast<uint32_t>(lane);
    const bool valid = j < s_hi;
    const uint32_t cj = j <= S ? ld_cu(cu, j) : 0u;       // cu[j]
    const uint32_t cj1 = valid ? ld_cu(cu, j + 1) : 0u;   // cu[j + 1]
    const bool is_long = valid && cj1 - cj > static_cast<uint32_t>(kShort);
    const unsigned int longs = __ballot_sync(0xffffffffu, is_long);
    uint32_t p = base;  // the next sequence of this chunk not yet placed
    while (p < s_hi && p < base + 32) {
      const uint32_t off = p - base;
      if (open) {
        // the open group takes p, p + 1, ... until one is outside the window, long, or ends
        // past g0 + 128
        const bool stop = lane >= static_cast<int>(off) && (!valid || is_long || cj1 - g0 > static_cast<uint32_t>(kBR));
        const unsigned int ends = __ballot_sync(0xffffffffu, stop);
        if (ends == 0u) break;  // it runs into the next chunk
        const uint32_t e_off = static_cast<uint32_t>(__ffs(ends) - 1);
        const uint32_t ce = __shfl_sync(0xffffffffu, cj, static_cast<int>(e_off));  // cu[e]
        if (ce > g0) sink.group(gs, base + e_off, g0, ce, lane);
        open = false;
        p = base + e_off;
        continue;
      }
      if ((longs >> off) & 1u) {
        // a long sequence: its pieces that start in this window
        const uint32_t c0 = __shfl_sync(0xffffffffu, cj, static_cast<int>(off));
        const uint32_t c1 = __shfl_sync(0xffffffffu, cj1, static_cast<int>(off));
        const uint64_t lim = min(static_cast<uint64_t>(c1), W1) - c0;
        sink.pieces(cu, p, 0u, static_cast<uint32_t>((lim + kBR - 1) / kBR), window, lane);
        ++p;
        continue;
      }
      // a short sequence opens a group
      open = true;
      gs = p;
      g0 = __shfl_sync(0xffffffffu, cj, static_cast<int>(off));
      ++p;
    }
  }
  // a group still open at the window's last sequence ends there
  if (open) {
    const uint32_t ce = ld_cu(cu, s_hi);
    if (ce > g0) sink.group(gs, s_hi, g0, ce, lane);
  }
}

// Walk, scan and place the records, reading cu through `cu` (the staged shared copy or the
// caller's array; the body is instantiated for each so that loads use their own space).
// The C blocks of the cluster (schedule_ctas) hold kSchedWarps warps each; global warp gw =
// warp x C + rank takes a contiguous run of windows (so consecutive runs are spread over the
// blocks) and writes their records, in order, to its own staging slots. The warps'
// counts, exchanged through distributed shared memory, give each warp the position of its
// run, which it then copies into place: the runs follow in q0 order.
template <class CuPtr>
__device__ __forceinline__ void schedule_body(CuPtr cu, int S, long long T, int window, TileRec* __restrict__ tiles,
                                              long long cap, TileRec* __restrict__ stage, TileRec* smem_slots,
                                              Ctl* ctl, uint32_t* s_warp, cg::cluster_group& cluster) {
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster.block_rank(), C = cluster.num_blocks();
  const uint32_t G = kSchedWarps * C;
  const uint32_t gw = static_cast<uint32_t>(warp) * C + rank;
  const uint64_t NB = (static_cast<uint64_t>(T) + kWin - 1) / kWin;
  const uint64_t per = (NB + G - 1) / G;
  const uint64_t b0 = min(NB, per * gw), b1 = min(NB, b0 + per);
  const uint64_t slots = per * kWinCap;
  // this warp's slots: in shared memory when the launch found room, else in the workspace
  TileRec* mine = smem_slots ? smem_slots + static_cast<uint64_t>(warp) * slots : stage + static_cast<uint64_t>(gw) * slots;
  WriteSink st{mine, slots, 0u};
  for (uint64_t b = b0; b < b1; ++b) window_visit(cu, static_cast<uint32_t>(S), window, b, lane, st);
  const uint32_t count = st.at;

  // every warp's count, then this warp's position: the sum over the warps before it
  if (lane == 0) s_warp[warp] = count;
  if (C == 1)
    __syncthreads();  // (also orders the staged records before the copies below)
  else
    cluster.sync();
  uint32_t before = 0, total = 0;
  for (uint32_t k = lane; k < G; k += 32) {
    const uint32_t v = C == 1 ? s_warp[k] : cluster.map_shared_rank(s_warp, k % C)[k / C];
    total += v;
    if (k < gw) before += v;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    total += __shfl_xor_sync(0xffffffffu, total, o);
  }
  if (C > 1) cluster.sync();  // no block leaves while another still reads its counts
  const bool fits = count <= slots && total <= static_cast<uint64_t>(cap);
  if (fits) {
    const uint4* src = reinterpret_cast<const uint4*>(mine);
    uint4* dst = reinterpret_cast<uint4*>(tiles + before);
    for (uint32_t i = lane; i < 2 * count; i += 32) dst[i] = src[i];
  }
  if (!fits && lane == 0) set_status(ctl, kErrInternal);
  if (rank == 0 && tid == 0) {
    ctl->ntiles = total <= static_cast<uint64_t>(cap) ? total : 0u;
    ctl->next = 0;
  }
}

}  // namespace

// One cluster of schedule_ctas(T) blocks. Every block stages cu (when it fits) and checks it;
// a malformed cu sends all of them out before the first cluster barrier.
__global__ void __launch_bounds__(kSchedThreads)
pk_schedule_kernel(const uint32_t* __restrict__ cu_g, int S, long long T, int window,
                   TileRec* __restrict__ tiles, long long cap, TileRec* __restrict__ stage, Ctl* ctl,
                   unsigned int slots_at) {
  extern __shared__ __align__(16) uint32_t s_cu[];
  // record slots in shared memory past the staged cu (slots_at bytes in), or none
  TileRec* smem_slots = slots_at ? reinterpret_cast<TileRec*>(reinterpret_cast<char*>(s_cu) + slots_at) : nullptr;
  __shared__ int s_bad;
  __shared__ uint32_t s_warp[kSchedWarps];
  cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  // the attention kernel may start its set-up now; it reads the records only after this
  // grid has completed (griddep_wait)
  griddep_launch_dependents();
  const bool staged = S + 1 <= kStageMax;
  if (tid == 0) s_bad = 0;
  if (staged) {
    // eight loads in flight per thread
    for (int s0 = tid; s0 <= S; s0 += 8 * nthr) {
      uint32_t v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = s0 + k * nthr <= S ? __ldg(cu_g + s0 + k * nthr) : 0u;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (s0 + k * nthr <= S) s_cu[s0 + k * nthr] = v[k];
    }
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
    if (cluster.block_rank() == 0 && tid == 0) {
      ctl->ntiles = 0;
      ctl->next = 0;
      set_status(ctl, kErrBadCu);
    }
    return;
  }
  if (staged)
    schedule_body(static_cast<const uint32_t*>(s_cu), S, T, window, tiles, cap, stage, smem_slots, ctl, s_warp,
                  cluster);
  else
    schedule_body(GlobalCu{cu_g}, S, T, window, tiles, cap, stage, smem_slots, ctl, s_warp, cluster);
}

// The carve-out matches the attention kernel's (all shared memory), so that the SMs need
// no reconfiguration between the two kernels of a call.
cudaError_t schedule_prepare() {
  cudaError_t e = cudaFuncSetAttribute(pk_schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSchedSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(pk_schedule_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              cudaSharedmemCarveoutMaxShared);
}

// `stage` holds schedule_stage_records(T) records of scratch.
cudaError_t schedule_launch(const uint32_t* cu, int S, long long T, int window, TileRec* tiles, long long cap,
                            TileRec* stage, Ctl* ctl, cudaStream_t stream) {
  const int ctas = schedule_ctas(T);
  // staged cu (when it fits), then the block's record slots (when they fit too)
  const size_t cu_bytes = S + 1 <= kStageMax ? (static_cast<size_t>(S + 1) * sizeof(uint32_t) + 15) / 16 * 16 : 0;
  const long long nb = (T + kWin - 1) / kWin;
  const long long per = (nb + kSchedWarps * ctas - 1) / (kSchedWarps * ctas);
  const size_t slot_bytes = static_cast<size_t>(kSchedWarps) * per * kWinCap * sizeof(TileRec);
  const bool in_smem = cu_bytes + slot_bytes <= static_cast<size_t>(kSchedSmem);
  const size_t smem = in_smem ? cu_bytes + slot_bytes : cu_bytes;
  const unsigned int slots_at = in_smem ? static_cast<unsigned int>(cu_bytes) : 0u;
  if (ctas == 1) {
    // a lone block is a cluster of one without the cluster launch
    pk_schedule_kernel<<<1, kSchedThreads, smem, stream>>>(cu, S, T, window, tiles, cap, stage, ctl, slots_at);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas, 1, 1);
  cfg.blockDim = dim3(kSchedThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ctas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pk_schedule_kernel, cu, S, T, window, tiles, cap, stage, ctl, slots_at);
}

}  // namespace pk
