// pk_backward_tc.cu -- the backward pass's main kernel on the tensor cores (tcgen05), bf16 / fp16.
//
// The gradient of the packed RoPE attention (hanzo-kernel packed.rs, fn attend_back): per visible
// (query a, key b) pair P = exp(scale q'_a . k'_b - lse_a), dS = P (dout_a . v_b - D_a), and
// dv_b = sum_a P dout_a, dk'_b = scale sum_a dS q'_a, dq'_a = scale sum_b dS k'_b.
//
// Work: a tile record's rows are a tile of 128 keys (visibility is symmetric, so the record's
// key range is exactly the queries that see those keys); one work item is (record, head), taken
// from the scheduler's counter by persistent CTAs, one per SM. Per item the CTA rotates K' once
// and walks the visible queries in chunks of 128:
//   S^T = K' Q'^T and dP^T = V dout^T         (M = 128 keys, N = 128 queries, K = 64)  -> TMEM
//   the row group (thread = key row) forms P^T and dS^T from both rows and writes them to
//   shared memory as 16-bit operands
//   dV += P^T dout, dK' += dS^T Q'             (M = 128 keys, N = 64, K = 128 queries) -> TMEM
//   dQ' = dS K'                                (M = 128 queries, N = 64, K = 128 keys)  -> TMEM
//   (dS read from the dS^T tiles as an MN-major operand)
// and the row group (thread = query row) adds scale dQ' to the fp32 dq accumulator. At the end of
// the item dK' and dV are complete: dk = rot^T(scale dK') and dv are rounded once and written.
//
// Roles (384 threads): warp 0 lane 0 the TMA producer, warp 1 lane 0 the MMA issuer, warp 2 owns
// the tensor memory (512 columns), warps 4-11 the row group in two halves of four warps (warp w
// reads TMEM lanes 32 (w % 4) ..): row t is shared by thread t of each half, which take half of
// the row's work each (half the chunk pairs of a rotation, 64 of a chunk's 128 queries, 32 of
// the 64 dimensions of dQ', dK', dV).
// Within an item the three roles step through the chunks in lockstep on mbarriers (each barrier
// completes once per chunk and every waiter waits for every phase, so a parity test is never two
// phases away from its barrier); items are separated by a CTA-wide barrier.
//
// Shared memory: K', V, Q', dout as 128 x 64 tiles, 128-byte swizzled as TMA lands them (row r
// at 128 r, its 16-byte chunk c at (c ^ (r & 7)) 16); P^T, dS^T as [key][query], each two such
// tiles side by side (64 queries each). K-major operands advance 32 bytes per K step of 16 inside
// a tile; the MN-major ones (dout, Q', K' as the B side of the products with N = 64, and dS^T as
// the A side of dQ' with M = 128: its two tiles are the two swizzle atoms along M) advance 2048
// bytes (16 rows).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>

#include "pk.h"
#include "pk_dev.cuh"

namespace pk {

namespace {

constexpr int kTcThreads = 384;
constexpr int kRowWarp0 = 4;              // warps 4..11: the row group, two halves of four warps
constexpr uint32_t kTile = 128u * 128u;   // 128 rows x 64 16-bit elements
constexpr uint32_t kOffK = 0;                   // K' of item buffer b at kOffK + b kKVBuf
constexpr uint32_t kOffV = kOffK + kTile;       // V of item buffer b at kOffV + b kKVBuf
constexpr uint32_t kKVBuf = 2 * kTile;          // two item buffers (K', V), taken in turn
constexpr uint32_t kOffQ = kOffK + 2 * kKVBuf;  // Q' of buffer b at kOffQ + b kQBuf
constexpr uint32_t kOffO = kOffQ + kTile;       // dout of buffer b at kOffO + b kQBuf
constexpr uint32_t kQBuf = 2 * kTile;           // two chunk buffers (Q', dout), taken in turn
constexpr uint32_t kOffPt = kOffQ + 2 * kQBuf;  // P^T  [key][query], two tiles
constexpr uint32_t kOffSt = kOffPt + 2 * kTile; // dS^T [key][query], two tiles
constexpr uint32_t kOffRow = kOffSt + 2 * kTile; // per query of the chunk: lse log2(e), D
struct TcBars {
  uint64_t kv_ready, q_ready, s_full, p_ready, c_done, drain;
  uint64_t kv_full[2];             // per item buffer: K and V loaded
  uint64_t q_full[2], q_empty[2];  // per chunk buffer: loaded; its last products have read it
};
constexpr uint32_t kOffBar = kOffRow + 2 * 128 * 4;
constexpr uint32_t kTcSmemUsed = kOffBar + sizeof(TcBars) + 16;
constexpr uint32_t kTcSmem = kTcSmemUsed + 1024;  // alignment slack
static_assert(kTcSmem <= 227u * 1024u, "fits the 227 KB a block may use");
// tensor-memory columns
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 320, kColDQ = 384;
constexpr float kLog2eTc = 1.4426950408889634f;

struct TcParams {
  const uint16_t* cos_t;
  const uint16_t* sin_t;
  const uint32_t* cu;
  const TileRec* tiles;
  Ctl* ctl;
  const float* lse;
  const float* D;
  float* dq;
  uint16_t* dqkv;
  int H;
  long long T;
  int window;
  float scale;
  unsigned long long timeout_ns;
};

__device__ __forceinline__ float ex2_tc(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// the 16-byte chunk c of row r of a 128-byte-swizzled tile
__device__ __forceinline__ uint8_t* chunk_at(uint8_t* tile, int r, int c) {
  return tile + r * 128 + ((c ^ (r & 7)) << 4);
}

// Chunk pairs c0, c0 + 1 of row r of a landed [128][64] tile rotated in place at position pos
// (pairs u, u + 32: chunk c with chunk c + 4), tables in the element type.
template <bool BF16>
__device__ __forceinline__ void rotate_row(uint8_t* tile, int r, const uint16_t* cos_t, const uint16_t* sin_t,
                                           uint32_t pos, int c0) {
  const uint4* cr = reinterpret_cast<const uint4*>(cos_t + static_cast<int64_t>(pos) * 32);
  const uint4* sr = reinterpret_cast<const uint4*>(sin_t + static_cast<int64_t>(pos) * 32);
#pragma unroll
  for (int c = c0; c < c0 + 2; ++c) {
    uint4* p1 = reinterpret_cast<uint4*>(chunk_at(tile, r, c));
    uint4* p2 = reinterpret_cast<uint4*>(chunk_at(tile, r, c + 4));
    const uint4 x1 = *p1, x2 = *p2, tc = __ldg(cr + c), ts = __ldg(sr + c);
    const uint32_t a1[4] = {x1.x, x1.y, x1.z, x1.w}, a2[4] = {x2.x, x2.y, x2.z, x2.w};
    const uint32_t ac[4] = {tc.x, tc.y, tc.z, tc.w}, as[4] = {ts.x, ts.y, ts.z, ts.w};
    uint32_t y1[4], y2[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 u = Elem<BF16>::unpack(a1[i]), w = Elem<BF16>::unpack(a2[i]);
      const float2 co = Elem<BF16>::unpack(ac[i]), si = Elem<BF16>::unpack(as[i]);
      y1[i] = Elem<BF16>::pack(u.x * co.x - w.x * si.x, u.y * co.y - w.y * si.y);
      y2[i] = Elem<BF16>::pack(u.x * si.x + w.x * co.x, u.y * si.y + w.y * co.y);
    }
    *p1 = make_uint4(y1[0], y1[1], y1[2], y1[3]);
    *p2 = make_uint4(y2[0], y2[1], y2[2], y2[3]);
  }
}

// bounded wait shared by the roles; on a timeout it records the error and raises the CTA's flag
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, const TcParams& p, volatile int* abort) {
  if (*abort) return false;
  if (mbar_wait(smem_u32(bar), parity, p.timeout_ns)) return true;
  *abort = 1;
  set_status(p.ctl, kErrTimeout);
  return false;
}

// The row group's decision to give up, taken together: a barrier over its 256 threads (named
// barrier 1) that ORs their flags, so that no warp waits at a later group barrier for a warp
// that has left.
__device__ __forceinline__ bool group_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, 256, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v ? 1u : 0u)
      : "memory");
  return r != 0;
}

template <bool BF16>
__global__ void __launch_bounds__(kTcThreads, 1)
pk_bwd_tc_kernel(const __grid_constant__ CUtensorMap tmap_qkv, const __grid_constant__ CUtensorMap tmap_dout,
                 const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  TcBars& B = *reinterpret_cast<TcBars*>(smem + kOffBar);
  float* sL2 = reinterpret_cast<float*>(smem + kOffRow);  // lse log2(e) per query of the chunk
  float* sD = sL2 + 128;
  __shared__ uint32_t s_tmem;
  __shared__ unsigned int s_item;
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H;
  const int64_t hd = static_cast<int64_t>(H) * 64;
  const int64_t ldq = 3 * hd;

  if (tid == 0) {
    mbar_init(smem_u32(&B.kv_full[0]), 1);
    mbar_init(smem_u32(&B.kv_full[1]), 1);
    mbar_init(smem_u32(&B.kv_ready), 8);
    mbar_init(smem_u32(&B.q_full[0]), 1);
    mbar_init(smem_u32(&B.q_full[1]), 1);
    mbar_init(smem_u32(&B.q_empty[0]), 1);
    mbar_init(smem_u32(&B.q_empty[1]), 1);
    mbar_init(smem_u32(&B.q_ready), 8);
    mbar_init(smem_u32(&B.s_full), 1);
    mbar_init(smem_u32(&B.p_ready), 8);
    mbar_init(smem_u32(&B.c_done), 1);
    mbar_init(smem_u32(&B.drain), 1);
    s_abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmap_qkv);
    tma_prefetch_desc(&tmap_dout);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(&s_tmem), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const unsigned int n_items = __ldcg(&p.ctl->ntiles) * static_cast<unsigned int>(H);

  // running counts: items (kv barriers) and chunks (the chunk barriers) this CTA has stepped through
  uint32_t n_it = 0, n_ch = 0;
  // the producer's loads so far; when the CTA gives up, the last K / V load and the last load of
  // each chunk buffer are the only ones that may still be in flight
  uint32_t kv_loads = 0, q_loads = 0;

  const uint32_t idS = idesc_f16(BF16, 128, 128, false, false);
  const uint32_t idG = idesc_f16(BF16, 128, 64, false, true);

  // items are claimed one ahead: the first here, each next one by the producer (thread 0) while
  // the current one runs, so that it can load the next item's K, V and first query chunk early
  if (tid == 0) s_item = atomicAdd(&p.ctl->next, 1u);
  for (;;) {
    __syncthreads();
    tc_fence_after();
    const unsigned int item = s_item;
    const bool stop = item >= n_items || s_abort;
    __syncthreads();
    if (stop) break;
    const unsigned int ti = item / static_cast<unsigned int>(H);
    const int h = static_cast<int>(item % static_cast<unsigned int>(H));
    const TileRec rec = p.tiles[ti];
    const uint32_t qend = rec.k0 + rec.nk;
    const uint32_t nchunks = (rec.nk + 127u) / 128u;

    if (warp == 0 && lane == 0) {
      // producer: K and V of an item into item buffer (item count) & 1, then Q and dout of each
      // chunk into the chunk buffers in turn (global chunk g into buffer g & 1, its (g >> 1)-th
      // use), each once the products of the chunk two back, which read that buffer, have
      // completed -- so the next chunk's copy is in flight while the current one is worked on.
      // The next item's K, V and first chunk are loaded before this item ends.
      auto load_kv = [&](const TileRec& r, int hh) {
        const uint32_t kb = kv_loads & 1u;
        mbar_arrive_expect_tx(smem_u32(&B.kv_full[kb]), 2 * kTile);
        tma_load_2d(smem_u32(smem + kOffK + kb * kKVBuf), &tmap_qkv, smem_u32(&B.kv_full[kb]),
                    static_cast<int32_t>(hd + hh * 64), static_cast<int32_t>(r.q0));
        tma_load_2d(smem_u32(smem + kOffV + kb * kKVBuf), &tmap_qkv, smem_u32(&B.kv_full[kb]),
                    static_cast<int32_t>(2 * hd + hh * 64), static_cast<int32_t>(r.q0));
        ++kv_loads;
      };
      auto load_chunk = [&](const TileRec& r, int hh, uint32_t g, uint32_t c) -> bool {
        const uint32_t b = g & 1u;
        if (g >= 2 && !tc_wait(&B.q_empty[b], ((g >> 1) - 1u) & 1u, p, &s_abort)) return false;
        const int32_t qb = static_cast<int32_t>(r.k0 + 128u * c);
        mbar_arrive_expect_tx(smem_u32(&B.q_full[b]), 2 * kTile);
        tma_load_2d(smem_u32(smem + kOffQ + b * kQBuf), &tmap_qkv, smem_u32(&B.q_full[b]), static_cast<int32_t>(hh * 64), qb);
        tma_load_2d(smem_u32(smem + kOffO + b * kQBuf), &tmap_dout, smem_u32(&B.q_full[b]), static_cast<int32_t>(hh * 64), qb);
        ++q_loads;
        return true;
      };
      const bool first = n_it == 0;  // nothing of this item was loaded ahead
      bool ok = true;
      if (first) load_kv(rec, h);
      for (uint32_t c = first ? 0u : 1u; ok && c < nchunks; ++c) ok = load_chunk(rec, h, n_ch + c, c);
      const unsigned int nxt = atomicAdd(&p.ctl->next, 1u);
      if (ok && nxt < n_items) {
        const TileRec rn = p.tiles[nxt / static_cast<unsigned int>(H)];
        const int hn = static_cast<int>(nxt % static_cast<unsigned int>(H));
        load_kv(rn, hn);
        load_chunk(rn, hn, n_ch + nchunks, 0u);
      }
      s_item = nxt;  // read by every thread after the next CTA-wide barrier
    } else if (warp == 1 && lane == 0) {
      // MMA issuer
      const uint32_t kvo = (n_it & 1u) * kKVBuf;  // this item's K / V buffer
      const uint64_t aK = sdesc_sw128(smem_u32(smem + kOffK + kvo), 16, 1024);
      const uint64_t aV = sdesc_sw128(smem_u32(smem + kOffV + kvo), 16, 1024);
      const uint64_t bQ = sdesc_sw128(smem_u32(smem + kOffQ), 16, 1024);
      const uint64_t bO = sdesc_sw128(smem_u32(smem + kOffO), 16, 1024);
      const uint64_t mO = sdesc_sw128(smem_u32(smem + kOffO), 8192, 1024);  // dout as MN-major B
      const uint64_t mQ = sdesc_sw128(smem_u32(smem + kOffQ), 8192, 1024);  // Q' as MN-major B
      const uint64_t mK = sdesc_sw128(smem_u32(smem + kOffK + kvo), 8192, 1024);  // K' as MN-major B
      const uint64_t aPt0 = sdesc_sw128(smem_u32(smem + kOffPt), 16, 1024);
      const uint64_t aPt1 = sdesc_sw128(smem_u32(smem + kOffPt + kTile), 16, 1024);
      const uint64_t aSt0 = sdesc_sw128(smem_u32(smem + kOffSt), 16, 1024);
      const uint64_t aSt1 = sdesc_sw128(smem_u32(smem + kOffSt + kTile), 16, 1024);
      // dS as the A side of dQ' = dS K' (M = 128 queries, K = keys), read from the dS^T tiles
      // [key][query] as an MN-major operand: queries 64 .. 127 are the next swizzle atom along M
      // (the second tile, kTile bytes on), 8-key row groups 1024 bytes apart, a K step of 16 keys
      // 2048 bytes
      const uint64_t mSt = sdesc_sw128(smem_u32(smem + kOffSt), kTile, 1024);
      const uint32_t idQ = idesc_f16(BF16, 128, 64, true, true);
      bool ok = tc_wait(&B.kv_ready, n_it & 1u, p, &s_abort);
      for (uint32_t c = 0; ok && c < nchunks; ++c) {
        const uint32_t ph = (n_ch + c) & 1u;
        const uint32_t b = ph;                              // the chunk's buffer
        const uint64_t boff = static_cast<uint64_t>(b) * (kQBuf >> 4);  // descriptor offset of buffer b
        if (!(ok = tc_wait(&B.q_ready, ph, p, &s_abort))) break;
        tc_fence_after();
#pragma unroll
        for (uint32_t ks = 0; ks < 4; ++ks)
          umma_f16_ss(tmem + kColS, aK + 2 * ks, bQ + boff + 2 * ks, idS, ks > 0 ? 1u : 0u);
#pragma unroll
        for (uint32_t ks = 0; ks < 4; ++ks)
          umma_f16_ss(tmem + kColDP, aV + 2 * ks, bO + boff + 2 * ks, idS, ks > 0 ? 1u : 0u);
        umma_commit(smem_u32(&B.s_full));
        if (!(ok = tc_wait(&B.p_ready, ph, p, &s_abort))) break;
        tc_fence_after();
#pragma unroll
        for (uint32_t ks = 0; ks < 8; ++ks) {
          const uint64_t aP = (ks < 4 ? aPt0 : aPt1) + 2 * (ks & 3u);
          const uint64_t aT = (ks < 4 ? aSt0 : aSt1) + 2 * (ks & 3u);

          const uint32_t acc = (c > 0 || ks > 0) ? 1u : 0u;
          umma_f16_ss(tmem + kColDV, aP, mO + boff + 128 * ks, idG, acc);
          umma_f16_ss(tmem + kColDK, aT, mQ + boff + 128 * ks, idG, acc);
          umma_f16_ss(tmem + kColDQ, mSt + 128 * ks, mK + 128 * ks, idQ, ks > 0 ? 1u : 0u);
        }
        umma_commit(smem_u32(&B.c_done));
        umma_commit(smem_u32(&B.q_empty[b]));
      }
      // every product issued has completed before the item ends (and before tensor memory is freed)
      umma_commit(smem_u32(&B.drain));
      mbar_wait(smem_u32(&B.drain), n_it & 1u, p.timeout_ns);
    } else if (warp >= kRowWarp0) {
      // the row group: thread t is key row t (rotation, P^T / dS^T, dK / dV) and query row t
      // of each chunk (rotation of Q', lse and D, dQ')
      const int t = (tid - kRowWarp0 * 32) & 127;   // the row
      const int hf = (tid - kRowWarp0 * 32) >> 7;   // the half of its work
      const uint32_t lanes = static_cast<uint32_t>((warp & 3) * 32) << 16;
      const bool kok = t < static_cast<int>(rec.rows);
      const uint32_t b = rec.q0 + static_cast<uint32_t>(t);
      int64_t klo = 0, khi = 0, kstart = 0;
      if (kok) {
        const uint32_t sb = rec.kind == 0 ? rec.seq : seq_of_token(p.cu, rec.seq, rec.nseq, b);
        const int64_t ss = __ldg(p.cu + sb), se = __ldg(p.cu + sb + 1);
        kstart = klo = ss;
        khi = se;
        if (p.window > 0) {
          klo = max(ss, static_cast<int64_t>(b) - p.window);
          khi = min(se, static_cast<int64_t>(b) + p.window + 1);
        }
      }
      bool bad = group_any(!tc_wait(&B.kv_full[n_it & 1u], (n_it >> 1) & 1u, p, &s_abort));
      if (!bad) {
        if (kok)
          rotate_row<BF16>(smem + kOffK + (n_it & 1u) * kKVBuf, t, p.cos_t, p.sin_t, static_cast<uint32_t>(b - kstart),
                           2 * hf);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&B.kv_ready));
      }
      const float c1 = p.scale * kLog2eTc;
      // Q' row t of chunk c (rotated in its buffer), its lse and D; then q_ready. Chunk c + 1 is
      // staged as soon as chunk c's P^T and dS are written, so its rotation runs while chunk c's
      // products do (lse and D are single-buffered: every thread has read chunk c's by then).
      auto stage_chunk = [&](uint32_t c) -> bool {
        const uint32_t g = n_ch + c, bq = g & 1u;
        if (group_any(!tc_wait(&B.q_full[bq], (g >> 1) & 1u, p, &s_abort))) return true;
        const uint32_t a = rec.k0 + 128u * c + static_cast<uint32_t>(t);
        float l2 = 0.f, d = 0.f;
        if (a < qend) {
          const uint32_t sa = rec.kind == 0 ? rec.seq : seq_of_token(p.cu, rec.seq, rec.nseq, a);
          rotate_row<BF16>(smem + kOffQ + bq * kQBuf, t, p.cos_t, p.sin_t, a - __ldg(p.cu + sa), 2 * hf);
          if (hf == 0) {
            l2 = __ldg(p.lse + static_cast<int64_t>(h) * p.T + a) * kLog2eTc;
            d = __ldg(p.D + static_cast<int64_t>(h) * p.T + a);
          }
        }
        if (hf == 0) {
          sL2[t] = l2;
          sD[t] = d;
        }
        fence_proxy_async_smem();
        asm volatile("bar.sync 1, 256;" ::: "memory");  // the row group's lse / D are in place
        if (lane == 0) mbar_arrive(smem_u32(&B.q_ready));
        return false;
      };
      if (!bad && nchunks > 0) bad = stage_chunk(0);
      for (uint32_t c = 0; !bad && c < nchunks; ++c) {
        const uint32_t ph = (n_ch + c) & 1u;
        const uint32_t qb = rec.k0 + 128u * c;
        // P^T and dS^T of key row t (32 queries at a time), and dS's column t
        bad = group_any(!tc_wait(&B.s_full, ph, p, &s_abort));
        if (bad) break;
        tc_fence_after();
        // the chunk's queries q this key row sees: [v_lo, v_hi) (same sequence, window, q < qend)
        int v_lo = 0, v_hi = 0;
        if (kok) {
          v_lo = static_cast<int>(min(max(klo - static_cast<int64_t>(qb), static_cast<int64_t>(0)), static_cast<int64_t>(128)));
          v_hi = static_cast<int>(min(max(min(khi, static_cast<int64_t>(qend)) - static_cast<int64_t>(qb),
                                          static_cast<int64_t>(0)), static_cast<int64_t>(128)));
          v_hi = max(v_hi, v_lo);
        }
        const float2 c1c1 = make_float2(c1, c1);
#pragma unroll 1
        for (int cb = 2 * hf; cb < 2 * hf + 2; ++cb) {
          float s[32], dp[32];
          tmem_ld32(tmem + lanes + kColS + 32 * cb, s);
          tmem_ld32(tmem + lanes + kColDP + 32 * cb, dp);
          uint32_t pw[16], dw[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const int q = 32 * cb + i;
            const float2 l2 = *reinterpret_cast<const float2*>(sL2 + q);
            const float2 dd = *reinterpret_cast<const float2*>(sD + q);
            const float2 x = __ffma2_rn(make_float2(s[i], s[i + 1]), c1c1, make_float2(-l2.x, -l2.y));
            float p0 = ex2_tc(x.x), p1 = ex2_tc(x.y);
            p0 = static_cast<unsigned>(q - v_lo) < static_cast<unsigned>(v_hi - v_lo) ? p0 : 0.f;
            p1 = static_cast<unsigned>(q + 1 - v_lo) < static_cast<unsigned>(v_hi - v_lo) ? p1 : 0.f;
            const float2 dv = __fmul2_rn(make_float2(p0, p1),
                                         __fadd2_rn(make_float2(dp[i], dp[i + 1]), make_float2(-dd.x, -dd.y)));
            pw[i / 2] = Elem<BF16>::pack(p0, p1);
            dw[i / 2] = Elem<BF16>::pack(dv.x, dv.y);
          }
          // rows of P^T and dS^T: queries 32 cb .. 32 cb + 31 are chunks 4 (cb & 1) .. + 3 of tile cb / 2
          uint8_t* tp = smem + kOffPt + (cb >> 1) * kTile;
          uint8_t* tt = smem + kOffSt + (cb >> 1) * kTile;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int ch = 4 * (cb & 1) + j;
            *reinterpret_cast<uint4*>(chunk_at(tp, t, ch)) = make_uint4(pw[4 * j], pw[4 * j + 1], pw[4 * j + 2], pw[4 * j + 3]);
            *reinterpret_cast<uint4*>(chunk_at(tt, t, ch)) = make_uint4(dw[4 * j], dw[4 * j + 1], dw[4 * j + 2], dw[4 * j + 3]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();  // (each warp writes only its own rows: its lanes' writes precede its arrival)
        if (lane == 0) mbar_arrive(smem_u32(&B.p_ready));
        if (c + 1 < nchunks) {
          bad = stage_chunk(c + 1);
          if (bad) break;
        }
        // dQ' of query row t, added to the fp32 accumulator
        bad = group_any(!tc_wait(&B.c_done, ph, p, &s_abort));
        if (bad) break;
        tc_fence_after();
        {
          float v[32];
          tmem_ld32(tmem + lanes + kColDQ + 32 * hf, v);
          const uint32_t a = qb + static_cast<uint32_t>(t);
          if (a < qend) {
            float4* dst = reinterpret_cast<float4*>(p.dq + static_cast<int64_t>(a) * hd + h * 64 + 32 * hf);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              atomicAdd(dst + j, make_float4(p.scale * v[4 * j], p.scale * v[4 * j + 1], p.scale * v[4 * j + 2],
                                             p.scale * v[4 * j + 3]));
          }
        }
        tc_fence_before();
      }
      // dk = rot^T(scale dK') and dv of key row t, rounded once
      if (!bad) {
        // this half: the pairs u in [16 hf, 16 hf + 16) of dk (columns u and u + 32) and the
        // dimensions [32 hf, 32 hf + 32) of dv
        float ka[16], kb[16], v2[32];
        tmem_ld16(tmem + lanes + kColDK + 16 * hf, ka);
        tmem_ld16(tmem + lanes + kColDK + 32 + 16 * hf, kb);
        tmem_ld32(tmem + lanes + kColDV + 32 * hf, v2);
        if (kok) {
          const uint32_t pos = static_cast<uint32_t>(b - kstart);
          const uint16_t* cr = p.cos_t + static_cast<int64_t>(pos) * 32;
          const uint16_t* sr = p.sin_t + static_cast<int64_t>(pos) * 32;
          uint16_t* rowk = p.dqkv + static_cast<int64_t>(b) * ldq + hd + h * 64;
          uint16_t* rowv = p.dqkv + static_cast<int64_t>(b) * ldq + 2 * hd + h * 64;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int c = 2 * hf + cc;
            const uint4 tc4 = __ldg(reinterpret_cast<const uint4*>(cr) + c);
            const uint4 ts4 = __ldg(reinterpret_cast<const uint4*>(sr) + c);
            const uint32_t ac[4] = {tc4.x, tc4.y, tc4.z, tc4.w}, as[4] = {ts4.x, ts4.y, ts4.z, ts4.w};
            uint32_t ya[4], yb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 co = Elem<BF16>::unpack(ac[i]), si = Elem<BF16>::unpack(as[i]);
              const int u = 8 * cc + 2 * i;  // index into this half's 16 pairs
              const float xa0 = p.scale * ka[u], xb0 = p.scale * kb[u];
              const float xa1 = p.scale * ka[u + 1], xb1 = p.scale * kb[u + 1];
              ya[i] = Elem<BF16>::pack(fmaf(xa0, co.x, xb0 * si.x), fmaf(xa1, co.y, xb1 * si.y));
              yb[i] = Elem<BF16>::pack(fmaf(xb0, co.x, -xa0 * si.x), fmaf(xb1, co.y, -xa1 * si.y));
            }
            reinterpret_cast<uint4*>(rowk)[c] = make_uint4(ya[0], ya[1], ya[2], ya[3]);
            reinterpret_cast<uint4*>(rowk)[c + 4] = make_uint4(yb[0], yb[1], yb[2], yb[3]);
          }
#pragma unroll
          for (int c = 0; c < 4; ++c)
            reinterpret_cast<uint4*>(rowv)[4 * hf + c] =
                make_uint4(Elem<BF16>::pack(v2[8 * c], v2[8 * c + 1]), Elem<BF16>::pack(v2[8 * c + 2], v2[8 * c + 3]),
                           Elem<BF16>::pack(v2[8 * c + 4], v2[8 * c + 5]), Elem<BF16>::pack(v2[8 * c + 6], v2[8 * c + 7]));
        }
        tc_fence_before();
      }
    }
    ++n_it;
    n_ch += nchunks;
  }

  // the producer's copies in flight land before the CTA's shared memory goes away
  if (warp == 0 && lane == 0 && s_abort) {
    // K / V loads go to item buffer (load count) & 1: the last load of each buffer
    for (uint32_t k = kv_loads >= 2 ? kv_loads - 2 : 0; k < kv_loads; ++k)
      mbar_wait(smem_u32(&B.kv_full[k & 1u]), (k >> 1) & 1u, p.timeout_ns);
    // chunk loads go to buffer g & 1 in the order of the CTA's global chunk index g, as
    // q_loads counts them: the last load of each buffer
    for (uint32_t g = q_loads >= 2 ? q_loads - 2 : 0; g < q_loads; ++g)
      mbar_wait(smem_u32(&B.q_full[g & 1u]), (g >> 1) & 1u, p.timeout_ns);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, 512);
}

typedef CUresult (*EncodeTiledTc)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledTc encode_tc() {
  static EncodeTiledTc fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* q = nullptr;
    cudaDriverEntryPointQueryResult r;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q, 12000, cudaEnableDefault, &r) == cudaSuccess &&
        r == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledTc>(q);
  }
  return fn;
}

bool tile_map(CUtensorMap* m, bool bf16, const void* base, uint64_t cols, uint64_t rows) {
  EncodeTiledTc enc = encode_tc();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base),
             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

unsigned long long tc_timeout_ns() {
  const char* e = std::getenv("PK_TIMEOUT_MS");
  const long long ms = e ? std::atoll(e) : 0;
  return static_cast<unsigned long long>(ms > 0 ? ms : 2000) * 1000000ull;
}

}  // namespace

cudaError_t backward_tc_prepare() {
  cudaError_t e = cudaFuncSetAttribute(pk_bwd_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pk_bwd_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
  return e;
}

// The main kernel for 16-bit types: dq' added to `dq` (zeroed by the caller), dk and dv written to dqkv.
cudaError_t backward_tc_launch(bool bf16, const void* qkv, const void* cos_t, const void* sin_t, const uint32_t* cu,
                               long long T, int H, int window, float scale, const float* lse, const void* dout,
                               const float* D, float* dq, void* dqkv, const TileRec* tiles, Ctl* ctl, int sms,
                               cudaStream_t stream) {
  CUtensorMap mq, mo;
  if (!tile_map(&mq, bf16, qkv, 3ull * H * 64, static_cast<uint64_t>(T)) ||
      !tile_map(&mo, bf16, dout, 1ull * H * 64, static_cast<uint64_t>(T)))
    return cudaErrorInvalidValue;
  TcParams p;
  p.cos_t = static_cast<const uint16_t*>(cos_t);
  p.sin_t = static_cast<const uint16_t*>(sin_t);
  p.cu = cu;
  p.tiles = tiles;
  p.ctl = ctl;
  p.lse = lse;
  p.D = D;
  p.dq = dq;
  p.dqkv = static_cast<uint16_t*>(dqkv);
  p.H = H;
  p.T = T;
  p.window = window;
  p.scale = scale;
  p.timeout_ns = tc_timeout_ns();
  if (bf16)
    pk_bwd_tc_kernel<true><<<sms, kTcThreads, kTcSmem, stream>>>(mq, mo, p);
  else
    pk_bwd_tc_kernel<false><<<sms, kTcThreads, kTcSmem, stream>>>(mq, mo, p);
  return cudaGetLastError();
}

}  // namespace pk
