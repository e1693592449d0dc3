// pk_attend_tc.cu -- packed RoPE attention forward for bf16 / fp16 on tcgen05 (sm_103a).
//
// What it computes: hanzo-kernel 0.2.42 packed.rs fn attend -- a tile of query rows of
// one head against every key tile its window reaches, q and k rotated in the kernel
// ("the query tile, rotated and scaled"; "the key tile rotated, the value tile as is"),
// scores and the output product on the matrix units, the softmax online per row with
// masked keys weighing exactly zero, then out = O / l and lse = m + ln l.
//
// How (GB300): one persistent 512-thread CTA per SM. A work item is a PAIR of consecutive
// tile records (A, B) of one head (or, in the single-record mode, one record alone). When both are pieces of the same sequence they share
// one key stream -- key tiles of 128 tokens from A's first key to the last key either can
// see -- so every K / V tile is loaded and rotated once for two query tiles; otherwise B's
// key tiles follow A's in the stream. A uses stream tiles [0, a1), B uses [b0, b1).
//
// Shared memory: Q tiles A and B, double-buffered across items (the next item's Q is
// fetched and rotated while the current one runs), a K ring and a V ring over the stream,
// and per rotation thread two 128-byte cos / sin table rows. Tensor memory (512 columns):
//     S_A, S_B [128 x 128] fp32    scores of the current key tile
//     P_A, P_B [128 x 128] 16-bit  probabilities, the A operand of the PV product
//     O_A, O_B [128 x  64] fp32    output accumulators
// Warpgroups (each warp's TMEM lane quarter is its index mod 4):
//   WG0  warp 0: producer (one lane): claims items, TMA-loads Q_A, Q_B and the stream's
//        K and V tiles (128-byte swizzle, straight from the strided qkv), K two tiles ahead
//        of V; warps 1, 2: MMA issuers of A, B (one lane each): per stream tile j,
//        S_X(j) = Q_X K(j)^T when X uses j, then O_X += P_X(j-1) V(j-1); warp 3 idle.
//   WG1  rotation: thread t rotates row t of every Q and K tile in shared memory as soon
//        as it lands, from table rows it prefetched with cp.async (q is multiplied by the
//        scale here only when the scale is not positive).
//   WG2, WG3  softmax of A, B: thread r owns query row r. It reads its S row from TMEM
//        twice (the row max by quarters, then the probabilities by halves), masks it by the
//        row's visible key interval, applies a positive scale inside exp2, keeps a running
//        max (O is rescaled only when the max grows by more than a factor 2^8), writes P to
//        TMEM, and at the end of the item writes out = O / l and lse = m + ln l.
// The loops of the rotation and softmax roles stay rolled: the four code streams sharing
// an SM sub-partition run out of instruction cache when they are unrolled.
// Every wait is bounded. A wait that times out records PK_ERR_TIMEOUT and raises the
// CTA's abort flag, which every other wait watches; the producer then waits (bounded)
// for its copies in flight, the MMA issuers for their MMAs, and the CTA frees its tensor
// memory and returns.
#include <cstdlib>

#include "pk_dev.cuh"

namespace pk {

namespace {

constexpr int kThreads = 512;
constexpr int kKStages = 4;  // a power of two (the rotation warps step the stage with a mask)
constexpr int kVStages = 3;
constexpr int kWarpProd = 0;
constexpr int kWarpMma = 1;  // warps 1 (A), 2 (B)
constexpr int kWarpRot = 4;  // warps 4..7
constexpr int kWarpSm = 8;   // warps 8..11 (A), 12..15 (B)

constexpr uint32_t kTileBytes = 128 * 128;  // 128 rows x 64 x 16-bit
constexpr uint32_t kRowTblBytes = 128;      // cos (64 B) + sin (64 B) of one position
// shared-memory map (offsets from the 1024-aligned base)
constexpr uint32_t kOffQ = 0;                                      // [X][buffer] tiles
constexpr uint32_t kOffK = kOffQ + 4 * kTileBytes;                 // K ring
constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;          // V ring
constexpr uint32_t kOffTbl = kOffV + kVStages * kTileBytes;        // [thread][2] table rows
constexpr uint32_t kOffMeta = kOffTbl + 128 * 2 * kRowTblBytes;

// One work item as the producer hands it to the other roles.
struct ItemBox {
  TileRec a, b;
  int32_t head;
  int32_t valid;     // 0: no more work
  uint32_t has_b;    // 1: B is a record
  uint32_t shared;   // 1: B reads A's key stream
  uint32_t nstream;  // key tiles in the stream
  uint32_t a1;       // A uses stream tiles [0, a1)
  uint32_t b0, b1;   // B uses stream tiles [b0, b1) (empty without B)
  uint32_t end;      // shared stream: one past its last key token
  uint32_t ss_a, se_a, ss_b, se_b;  // a piece's sequence [start, end) (A, B; unused for a group)
  uint32_t pad[3];
};
static_assert(sizeof(ItemBox) % 16 == 0, "item box keeps 16-byte alignment");

struct Bars {
  uint64_t item_full[2], item_empty[2];
  uint64_t q_full[2][2], q_ready[2][2], q_empty[2][2];  // [X][buffer]
  uint64_t k_full[kKStages], k_ready[kKStages], k_empty[kKStages];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t s_full[2], s_consumed[2], p_ready[2], pv_done[2];  // [X]
  uint64_t cu_rot[2], cu_sm[2][2];  // staged offsets ready: [item parity], [X][item parity]
  uint64_t drain[2];
};

// Member sequence offsets of an item's records, staged by the rotation warpgroup (A's and
// B's) and by each softmax warpgroup (its own record's).
constexpr int kCuStage = kBR + 2;  // a group of up to 128 non-empty sequences
struct Meta {
  Bars bars;
  ItemBox box[2];
  uint32_t cu_rot[2][2][kCuStage];  // [item parity][X]
  uint32_t cu_sm[2][2][kCuStage];   // [X][item parity]
  uint32_t tmem;
  int32_t abort;
};

constexpr uint32_t kSmemUsed = kOffMeta + sizeof(Meta);
static_assert(kSmemUsed + 1024 <= 227u * 1024u, "fits the 227 KB a block may use");
constexpr uint32_t kTmemCols = 512;
// tensor-memory columns of query tile X
__host__ __device__ constexpr uint32_t col_s(int x) { return 128u * x; }
__host__ __device__ constexpr uint32_t col_p(int x) { return 256u + 64u * x; }
__host__ __device__ constexpr uint32_t col_o(int x) { return 384u + 64u * x; }
constexpr uint32_t kItemConsumers = 2 + 4 + 4 + 4;  // MMA issuers + rotation, softmax A, B warps

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNeg = -1.0e30f;      // running-max start: ex2 of (masked - kNeg) stays 0
constexpr float kRescale = 8.0f;      // rescale O only when the max grows by more than 2^8
constexpr uint32_t kSleepNs = 20000;  // longest sleep of a waiting thread between checks

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

__device__ __forceinline__ uint8_t* q_tile(uint8_t* smem, int x, uint32_t b) {
  return smem + kOffQ + kTileBytes * (2 * x + b);
}
__device__ __forceinline__ uint8_t* k_tile(uint8_t* smem, uint32_t st) { return smem + kOffK + kTileBytes * st; }
__device__ __forceinline__ uint8_t* v_tile(uint8_t* smem, uint32_t st) { return smem + kOffV + kTileBytes * st; }

__device__ __forceinline__ bool aborted(const Meta* meta) {
  return *reinterpret_cast<const volatile int32_t*>(&meta->abort) != 0;
}
__device__ __forceinline__ void raise_abort(Meta* meta, Ctl* ctl) {
  *reinterpret_cast<volatile int32_t*>(&meta->abort) = 1;
  set_status(ctl, kErrTimeout);
}

// Bounded wait on phase `parity` of `bar` that also gives up once the CTA has aborted.
__device__ __forceinline__ bool wait_bar(Meta* meta, Ctl* ctl, uint64_t* bar, uint32_t parity,
                                         uint64_t timeout_ns) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_sleep(a, parity, kSleepNs)) return true;
    if ((i & 7u) == 0u) {
      if (aborted(meta)) return false;
      if (globaltimer_ns() - t0 > timeout_ns) {
        raise_abort(meta, ctl);
        return false;
      }
    }
  }
}

// A ring position: uses so far, giving stage and phase parity.
struct Ring {
  uint32_t n = 0;
  __device__ __forceinline__ uint32_t stage(uint32_t depth) const { return n % depth; }
  __device__ __forceinline__ uint32_t phase(uint32_t depth) const { return (n / depth) & 1u; }
};


// The key stream of an item, as every role keeps it in registers.
struct Stream {
  uint32_t a_k0, a_nk, b_k0, b_nk;
  uint32_t end;     // shared stream: one past its last key token
  uint32_t a1;      // A uses stream tiles [0, a1)
  uint32_t b0, b1;  // B uses stream tiles [b0, b1)
  uint32_t n;       // stream tiles
  uint32_t shared;  // 1: B reads A's key stream; 0: B's tiles follow A's
};
__device__ __forceinline__ Stream stream_of(const ItemBox& bx) {
  Stream s;
  s.a_k0 = bx.a.k0;
  s.a_nk = bx.a.nk;
  s.b_k0 = bx.b.k0;
  s.b_nk = bx.b.nk;
  s.end = bx.end;
  s.a1 = bx.a1;
  s.b0 = bx.b0;
  s.b1 = bx.b1;
  s.n = bx.nstream;
  s.shared = bx.shared;
  return s;
}

// Stream tile j of an item: its first key token, its key count, and whether it is one of
// B's own tiles (a concatenated stream past A's tiles).
struct StreamTile {
  uint32_t j0, nkeys;
  bool from_b;
};
__device__ __forceinline__ StreamTile stream_tile(const Stream& s, uint32_t j) {
  StreamTile st;
  if (s.shared) {
    st.j0 = s.a_k0 + j * kBC;
    st.nkeys = min(static_cast<uint32_t>(kBC), s.end - st.j0);
    st.from_b = false;
  } else if (j < s.a1) {
    st.j0 = s.a_k0 + j * kBC;
    st.nkeys = min(static_cast<uint32_t>(kBC), s.a_nk - j * kBC);
    st.from_b = false;
  } else {
    st.j0 = s.b_k0 + (j - s.a1) * kBC;
    st.nkeys = min(static_cast<uint32_t>(kBC), s.b_nk - (j - s.a1) * kBC);
    st.from_b = true;
  }
  return st;
}

struct Params {
  const uint16_t* cos_t;
  const uint16_t* sin_t;
  const uint32_t* cu;
  const TileRec* tiles;
  void* out;    // 16-bit of the element type, or fp32 (OUT32)
  float* lse;
  Ctl* ctl;
  int H;
  long long T;
  int window;
  float q_mul;  // multiplies the rotated q (the scale when it is not positive, else 1)
  float s_mul;  // multiplies the scores in the softmax (the scale when it is positive, else 1)
  unsigned long long timeout_ns;
  int skip_first_item_arrive;  // test hook: the producer withholds its first item hand-off
  int singles;                 // 1: a work item is one tile record (no B), 0: a pair of records
  int prerotated;              // 1: q and k arrive rotated (and q multiplied): no rotation here
};

// The member sequence offsets cu[rec.seq .. rec.seq + rec.nseq] of a record, copied by the
// `nthr` threads of a warpgroup into `dst` when they fit (a group can hold any number of
// empty sequences; past kCuStage - 1 members only the first offset is staged).
__device__ __forceinline__ bool staged_all(const TileRec& rec) { return rec.nseq + 1 <= kCuStage; }
__device__ __forceinline__ void stage_cu(const Params& p, const TileRec& rec, uint32_t* dst, int t, int nthr) {
  const int n = staged_all(rec) ? static_cast<int>(rec.nseq) : 0;
  for (int i = t; i <= n; i += nthr) dst[i] = __ldg(p.cu + rec.seq + i);
}

// The sequence (index into a staged offset list of n + 1 values) holding token a:
// the last i < n with off[i] <= a.
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

// Start and end tokens of the sequence of record `rec` that holds token a, from the staged
// offsets when they are all there, else from cu in global memory.
__device__ __forceinline__ void seq_bounds(const Params& p, const TileRec& rec, const uint32_t* off, uint32_t a,
                                           uint32_t& ss, uint32_t& se) {
  if (rec.kind == 0) {
    ss = off[0];
    se = off[1];
  } else if (staged_all(rec)) {
    const int i = staged_seq(off, static_cast<int>(rec.nseq), a);
    ss = off[i];
    se = off[i + 1];
  } else {
    const uint32_t sq = seq_of_token(p.cu, rec.seq, rec.nseq, a);
    ss = __ldg(p.cu + sq);
    se = __ldg(p.cu + sq + 1);
  }
}

// ------------------------------------------------------------------------------------
// table rows in shared memory (cp.async, 16 bytes at a time, no registers held; through L1,
// since the rows of short sequences are the same few table rows for every thread)

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Copies the cos and sin rows of position `pos` (32 16-bit values each) into the 128-byte
// row buffer `buf`: logical chunk k (cos 0..3, sin 4..7) at 16-byte slot k ^ (t & 7), so the
// eight threads of a quarter warp reading the same chunk hit eight different bank groups.
__device__ __forceinline__ void fetch_table_row(const Params& p, uint32_t buf, uint32_t pos, int t) {
  const uint16_t* c = p.cos_t + static_cast<size_t>(pos) * kHalf;
  const uint16_t* s = p.sin_t + static_cast<size_t>(pos) * kHalf;
  const int sw = t & 7;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    cp_async16(buf + ((k ^ sw) << 4), c + 8 * k);
    cp_async16(buf + (((k + 4) ^ sw) << 4), s + 8 * k);
  }
}

// Rotation of one 16-byte chunk pair: x1 holds elements u .. u+7 of the first half of a
// row, x2 the matching elements u+32 .. u+39, tc / ts the cos / sin table values of the
// same u; y1 = x1 c - x2 s, y2 = x1 s + x2 c in fp32 from the 16-bit operands, times `mul`
// when SCALED.
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
// it. Two chunk pairs per step, all their loads issued before the arithmetic.
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

// ------------------------------------------------------------------------------------
// producer (one thread): work items and TMA loads. Per item: Q_A, Q_B into their buffers,
// then K(0), K(1), V(0), K(2), V(1), ... over the key stream.

__device__ void producer(const CUtensorMap* tmap, const Params& p, uint8_t* smem, Meta* meta,
                         unsigned int n_items) {
  Bars& B = meta->bars;
  const int32_t hd = p.H * kD;
  const unsigned int ntiles = __ldcg(&p.ctl->ntiles);
  uint32_t it = 0;
  Ring q0r, q1r, k, v;
  bool bad = false;

  for (;;) {
    const unsigned int item = atomicAdd(&p.ctl->next, 1u);
    const uint32_t mb = it & 1u;
    if (!wait_bar(meta, p.ctl, &B.item_empty[mb], ((it >> 1) & 1u) ^ 1u, p.timeout_ns)) {
      bad = true;
      break;
    }
    ItemBox& bx = meta->box[mb];
    if (item >= n_items) {
      bx.valid = 0;
      mbar_arrive(smem_u32(&B.item_full[mb]));
      break;
    }
    const unsigned int pair = item / static_cast<unsigned int>(p.H);
    const int h = static_cast<int>(item % static_cast<unsigned int>(p.H));
    const unsigned int first_rec = p.singles ? pair : 2 * pair;
    const TileRec ra = p.tiles[first_rec];
    const bool has_b = !p.singles && 2 * pair + 1 < ntiles;
    TileRec rb = ra;
    if (has_b) rb = p.tiles[2 * pair + 1];
    const bool shared = has_b && ra.kind == 0 && rb.kind == 0 && ra.seq == rb.seq;
    uint32_t nstream, b0, b1, end = 0;
    if (shared) {
      end = max(ra.k0 + ra.nk, rb.k0 + rb.nk);
      nstream = (end - ra.k0 + kBC - 1) / kBC;
      b0 = (rb.k0 - ra.k0) / kBC;
      b1 = (rb.k0 + rb.nk - ra.k0 + kBC - 1) / kBC;
    } else {
      nstream = ra.ktiles + (has_b ? rb.ktiles : 0u);
      b0 = ra.ktiles;
      b1 = nstream;
    }
    bx.a = ra;
    bx.b = rb;
    bx.head = h;
    bx.valid = 1;
    bx.has_b = has_b;
    bx.shared = shared;
    bx.nstream = nstream;
    bx.a1 = ra.ktiles;
    bx.b0 = b0;
    bx.b1 = b1;
    bx.end = end;
    // a piece's sequence bounds travel with the item (only a group's rows need the offsets
    // of its member sequences staged)
    bx.ss_a = ra.kind == 0 ? __ldg(p.cu + ra.seq) : 0u;
    bx.se_a = ra.kind == 0 ? __ldg(p.cu + ra.seq + 1) : 0u;
    bx.ss_b = has_b && rb.kind == 0 ? __ldg(p.cu + rb.seq) : 0u;
    bx.se_b = has_b && rb.kind == 0 ? __ldg(p.cu + rb.seq + 1) : 0u;
    // (the test hook leaves the consumers waiting: their bounded waits time out and the CTA
    // unwinds with PK_ERR_TIMEOUT)
    if (!(p.skip_first_item_arrive && it == 0)) mbar_arrive(smem_u32(&B.item_full[mb]));
    ++it;

    // Q_X into its next buffer once the item two back has issued its last S_X
    auto load_q = [&](int x, Ring& qr, uint32_t q0) -> bool {
      const uint32_t qb = qr.stage(2);
      if (!wait_bar(meta, p.ctl, &B.q_empty[x][qb], qr.phase(2) ^ 1u, p.timeout_ns)) return false;
      mbar_arrive_expect_tx(smem_u32(&B.q_full[x][qb]), kTileBytes);
      tma_load_2d(smem_u32(q_tile(smem, x, qb)), tmap, smem_u32(&B.q_full[x][qb]), h * kD, static_cast<int32_t>(q0));
      ++qr.n;
      return true;
    };
    bad = !load_q(0, q0r, ra.q0) || (has_b && !load_q(1, q1r, rb.q0));
    if (bad) break;
    // the stream: K two tiles ahead of V
    const Stream sm = stream_of(bx);
    for (uint32_t t = 0; t < nstream + 2 && !bad; ++t) {
      if (t < nstream) {
        const uint32_t st = k.stage(kKStages);
        if (!wait_bar(meta, p.ctl, &B.k_empty[st], k.phase(kKStages) ^ 1u, p.timeout_ns)) {
          bad = true;
          break;
        }
        mbar_arrive_expect_tx(smem_u32(&B.k_full[st]), kTileBytes);
        tma_load_2d(smem_u32(k_tile(smem, st)), tmap, smem_u32(&B.k_full[st]), hd + h * kD,
                    static_cast<int32_t>(stream_tile(sm, t).j0));
        ++k.n;
      }
      if (t >= 2) {
        const uint32_t st = v.stage(kVStages);
        if (!wait_bar(meta, p.ctl, &B.v_empty[st], v.phase(kVStages) ^ 1u, p.timeout_ns)) {
          bad = true;
          break;
        }
        mbar_arrive_expect_tx(smem_u32(&B.v_full[st]), kTileBytes);
        tma_load_2d(smem_u32(v_tile(smem, st)), tmap, smem_u32(&B.v_full[st]), 2 * hd + h * kD,
                    static_cast<int32_t>(stream_tile(sm, t - 2).j0));
        ++v.n;
      }
    }
    if (bad) break;
  }
  if (bad || aborted(meta)) {
    // let the copies in flight land before the CTA's shared memory goes away
    for (uint32_t t = q0r.n > 2 ? q0r.n - 2 : 0; t < q0r.n; ++t)
      mbar_wait(smem_u32(&B.q_full[0][t % 2]), (t / 2) & 1u, p.timeout_ns);
    for (uint32_t t = q1r.n > 2 ? q1r.n - 2 : 0; t < q1r.n; ++t)
      mbar_wait(smem_u32(&B.q_full[1][t % 2]), (t / 2) & 1u, p.timeout_ns);
    for (uint32_t t = k.n > kKStages ? k.n - kKStages : 0; t < k.n; ++t)
      mbar_wait(smem_u32(&B.k_full[t % kKStages]), (t / kKStages) & 1u, p.timeout_ns);
    for (uint32_t t = v.n > kVStages ? v.n - kVStages : 0; t < v.n; ++t)
      mbar_wait(smem_u32(&B.v_full[t % kVStages]), (t / kVStages) & 1u, p.timeout_ns);
  }
}

// ------------------------------------------------------------------------------------
// MMA issuer of query tile X (one thread; one issuer per query tile, on different SM
// sub-partitions, so that each keeps its share of the tensor pipe fed). For every stream
// tile t: once K(t) is rotated, S_X(t) = Q_X K(t)^T if X's range holds t (after Q_X is
// rotated and S_X's previous scores were read); then, once V(t - 1) has landed,
// O_X += P_X(t - 1) V(t - 1) if X's range holds t - 1 (after P_X is written); a tile outside
// X's range is seen after that product, so the last PV of the range does not wait for the
// rotation of the next tile. K and V ring stages are released by both issuers (barriers of
// count 2): by a commit after the MMAs that read them, or by a plain arrival for a tile
// outside X's range -- made only after the tile's own ready / full phase was seen. Every
// stage's phases are waited for in order: a parity wait is only sound one phase at a time.

__device__ void mma_issuer(const Params& p, uint8_t* smem, Meta* meta, uint32_t tmem, bool bf16, int x) {
  Bars& B = meta->bars;
  // Every S product is 128 keys wide and every PV product runs over all 128 keys of its tile:
  // the columns past a tile's keys are masked scores and zero probabilities, so the extra
  // work changes no result, and the issue sequence carries no per-tile arithmetic or branch
  // (an MMA issued behind scalar code waits for it: a fixed sequence keeps the tensor pipe fed).
  const uint32_t idesc_s = idesc_f16(bf16, 128, 128, false, false);
  const uint32_t idesc_pv = idesc_f16(bf16, 128, 64, false, true);
  // operand descriptors of the first buffer of each kind; a K step of 16 adds 32 bytes (Q,
  // K) or 2048 bytes (V) to the start address field (address >> 4), and the next 16 KB tile
  // of a kind is 1024 further
  const uint64_t dq0 = sdesc_sw128(smem_u32(q_tile(smem, x, 0)), 16, 1024);
  const uint64_t dk0 = sdesc_sw128(smem_u32(k_tile(smem, 0)), 16, 1024);
  const uint64_t dv0 = sdesc_sw128(smem_u32(v_tile(smem, 0)), 8192, 1024);
  const uint32_t tS = tmem + col_s(x), tP = tmem + col_p(x), tO = tmem + col_o(x);
  uint32_t it = 0, sc = 0, pr = 0, qn = 0;
  bool pend = false;  // an S_X was issued whose reading has not been awaited yet
  uint32_t kst = 0, kph = 0, vst = 0, vph = 0;  // ring stage and phase of the next K, V tile
  bool bad = false;

  for (;;) {
    const uint32_t mb = it & 1u;
    if (!wait_bar(meta, p.ctl, &B.item_full[mb], (it >> 1) & 1u, p.timeout_ns)) break;
    const bool valid = meta->box[mb].valid != 0;
    const uint32_t n = meta->box[mb].nstream;
    const uint32_t lo = x == 0 ? 0u : meta->box[mb].b0, hi = x == 0 ? meta->box[mb].a1 : meta->box[mb].b1;
    mbar_arrive(smem_u32(&B.item_empty[mb]));
    ++it;
    if (!valid) break;
    for (uint32_t t = 0; t <= n && !bad; ++t) {
      // a tile of X's range: S_X(t) now; any other tile: seen after O_X += P_X(t - 1) V(t - 1),
      // so that the last PV of the range is not held back by the next tile's rotation
      const bool own = t < n && t >= lo && t < hi;
      if (own) {
        if (!wait_bar(meta, p.ctl, &B.k_ready[kst], kph, p.timeout_ns)) {
          bad = true;
          break;
        }
        const uint32_t qb = qn & 1u;
        if (t == lo && !wait_bar(meta, p.ctl, &B.q_ready[x][qb], (qn >> 1) & 1u, p.timeout_ns)) {
          bad = true;
          break;
        }
        if (pend) {
          if (!wait_bar(meta, p.ctl, &B.s_consumed[x], sc & 1u, p.timeout_ns)) {
            bad = true;
            break;
          }
          ++sc;
        }
        tc_fence_after();
        const uint64_t dq = dq0 + qb * 1024, dk = dk0 + kst * 1024;
        umma_f16_ss(tS, dq, dk, idesc_s, 0u);
        umma_f16_ss(tS, dq + 2, dk + 2, idesc_s, 1u);
        umma_f16_ss(tS, dq + 4, dk + 4, idesc_s, 1u);
        umma_f16_ss(tS, dq + 6, dk + 6, idesc_s, 1u);
        umma_commit(smem_u32(&B.s_full[x]));
        umma_commit(smem_u32(&B.k_empty[kst]));
        pend = true;
        if (t + 1 == hi) {
          umma_commit(smem_u32(&B.q_empty[x][qb]));
          ++qn;
        }
        kst = (kst + 1) & (kKStages - 1);
        kph ^= kst == 0 ? 1u : 0u;
      }
      if (t >= 1) {
        const uint32_t j = t - 1;
        if (!wait_bar(meta, p.ctl, &B.v_full[vst], vph, p.timeout_ns)) {
          bad = true;
          break;
        }
        if (j >= lo && j < hi) {
          if (!wait_bar(meta, p.ctl, &B.p_ready[x], pr & 1u, p.timeout_ns)) {
            bad = true;
            break;
          }
          ++pr;
          tc_fence_after();
          const uint64_t dv = dv0 + vst * 1024;
          umma_f16_ts(tO, tP, dv, idesc_pv, j > lo ? 1u : 0u);
#pragma unroll
          for (uint32_t ks = 1; ks < 8; ++ks) umma_f16_ts(tO, tP + ks * 8, dv + ks * 128, idesc_pv, 1u);
          umma_commit(smem_u32(&B.pv_done[x]));
          umma_commit(smem_u32(&B.v_empty[vst]));
        } else {
          mbar_arrive(smem_u32(&B.v_empty[vst]));
        }
        vst = vst + 1 == kVStages ? 0u : vst + 1;
        vph ^= vst == 0 ? 1u : 0u;
      }
      if (t < n && !own) {
        if (!wait_bar(meta, p.ctl, &B.k_ready[kst], kph, p.timeout_ns)) {
          bad = true;
          break;
        }
        mbar_arrive(smem_u32(&B.k_empty[kst]));
        kst = (kst + 1) & (kKStages - 1);
        kph ^= kst == 0 ? 1u : 0u;
      }
    }
    if (bad) break;
  }
  // every MMA this thread issued has completed before the CTA frees tensor memory
  umma_commit(smem_u32(&B.drain[x]));
  mbar_wait(smem_u32(&B.drain[x]), 0, p.timeout_ns);
}

// ------------------------------------------------------------------------------------
// rotation warpgroup (128 threads; thread t rotates row t of every tile)
//
// Per item: Q_A, Q_B (when B is a record), then the key stream K(0) .. K(n - 1), each as
// soon as it lands. A row's position is its token minus the start of its sequence: one
// subtraction for a piece of a sequence, a search in the staged member offsets for a group
// of short sequences (whose key rows are its query rows). The table rows of the next job
// are in flight (cp.async) while the current one is rotated. Ring stage, phase and
// positions advance step by step: the per-job bookkeeping is a few instructions, since this
// warpgroup's time goes into dependent chains. Rows past a tile's tokens are left as
// loaded; their scores are masked.

template <bool BF16>
__device__ void rotator(const Params& p, uint8_t* smem, Meta* meta, int t) {
  Bars& B = meta->bars;
  const int lane = t & 31;
  const uint32_t tbl0 = smem_u32(smem + kOffTbl + t * 2 * kRowTblBytes);
  const uint8_t* tblp = smem + kOffTbl + t * 2 * kRowTblBytes;
  uint32_t it = 0, qn0 = 0, qn1 = 0;
  uint32_t staged = 0;        // items whose member offsets were staged (those with a group)
  uint32_t kst = 0, kph = 0;  // K ring stage and phase of the next K tile
  uint32_t buf = 0;           // table buffer of the next job
  bool bad = false;
  for (;;) {
    const uint32_t mb = it & 1u;
    bad |= !wait_bar(meta, p.ctl, &B.item_full[mb], (it >> 1) & 1u, p.timeout_ns);
    bad = __any_sync(0xffffffffu, bad);
    if (bad) break;
    const ItemBox& bx = meta->box[mb];
    const bool valid = bx.valid != 0, has_b = bx.has_b != 0;
    const TileRec ra = bx.a, rb = bx.b;
    const Stream sm = stream_of(bx);
    const uint32_t ss_a = bx.ss_a, ss_b = bx.ss_b;
    // stage the member offsets of A and B when either is a group (a group needs them to find
    // each row's sequence; a piece's bounds came with the item)
    const bool grp = valid && (ra.kind != 0 || (has_b && rb.kind != 0));
    const uint32_t sb = staged & 1u;
    uint32_t* off_a = meta->cu_rot[sb][0];
    uint32_t* off_b = meta->cu_rot[sb][1];
    if (grp) {
      stage_cu(p, ra, off_a, t, 128);
      if (has_b) stage_cu(p, rb, off_b, t, 128);
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(smem_u32(&B.item_empty[mb]));
      if (grp) mbar_arrive(smem_u32(&B.cu_rot[sb]));
    }
    ++it;
    if (!valid) break;
    if (grp) {
      bad |= !wait_bar(meta, p.ctl, &B.cu_rot[sb], (staged >> 1) & 1u, p.timeout_ns);
      ++staged;
      bad = __any_sync(0xffffffffu, bad);
      if (bad) break;
    }

    // positions of row t of Q_A and Q_B (for a group also of its key row t)
    const bool qok_a = t < static_cast<int>(ra.rows);
    const bool qok_b = has_b && t < static_cast<int>(rb.rows);
    uint32_t qpos_a = 0u, qpos_b = 0u;
    if (qok_a) {
      uint32_t ss = ss_a, se;
      if (ra.kind != 0) seq_bounds(p, ra, off_a, ra.q0 + t, ss, se);
      qpos_a = ra.q0 + t - ss;
    }
    if (qok_b) {
      uint32_t ss = ss_b, se;
      if (rb.kind != 0) seq_bounds(p, rb, off_b, rb.q0 + t, ss, se);
      qpos_b = rb.q0 + t - ss;
    }

    // row t of key tile j of the stream: segment A holds tiles [0, a1) (all of them for a
    // shared stream), segment B the rest; within a segment, tile j starts at token
    // k0 + 128 (j - j_first), its keys end at kend, and a piece's row position is the token
    // minus the sequence start (a group's is its query row's)
    const uint32_t seg_a_end = sm.shared ? sm.n : sm.a1;
    const uint32_t a_kend = sm.shared ? sm.end : sm.a_k0 + sm.a_nk;
    const uint32_t b_kend = sm.b_k0 + sm.b_nk;
    const int32_t a_pbase = ra.kind != 0 ? 0 : static_cast<int32_t>(sm.a_k0 + t) - static_cast<int32_t>(ss_a);
    const int32_t b_pbase = (!has_b || rb.kind != 0) ? 0 : static_cast<int32_t>(sm.b_k0 + t) - static_cast<int32_t>(ss_b);
    auto krow = [&](uint32_t j, uint32_t& pos) -> bool {
      const bool inb = j >= seg_a_end;
      const uint32_t jj = inb ? j - seg_a_end : j;
      const uint32_t j0 = (inb ? sm.b_k0 : sm.a_k0) + jj * kBC;
      const bool ok = static_cast<uint32_t>(t) < (inb ? b_kend : a_kend) - j0;
      const bool grp = inb ? rb.kind != 0 : ra.kind != 0;
      pos = !ok ? 0u : grp ? (inb ? qpos_b : qpos_a)
                          : static_cast<uint32_t>((inb ? b_pbase : a_pbase) + static_cast<int32_t>(jj * kBC));
      return ok;
    };

    const uint32_t nq = has_b ? 2u : 1u;
    const uint32_t njobs = nq + sm.n;
    // the first job's table rows
    {
      const bool ok0 = qok_a;
      if (ok0 && !p.prerotated) fetch_table_row(p, tbl0 + buf * kRowTblBytes, qpos_a, t);
      cp_async_commit();
    }
#pragma unroll 1
    for (uint32_t i = 0; i < njobs; ++i) {
      // this job
      const bool isq = i < nq;
      const bool xb = i == 1 && has_b;
      uint32_t pos_i;
      bool ok;
      uint8_t* tile;
      uint64_t* full;
      uint64_t* ready;
      uint32_t phase;
      if (isq) {
        const uint32_t qn = xb ? qn1 : qn0;
        const uint32_t qb = qn & 1u;
        const int x = xb ? 1 : 0;
        tile = q_tile(smem, x, qb);
        full = &B.q_full[x][qb];
        ready = &B.q_ready[x][qb];
        phase = (qn >> 1) & 1u;
        ok = xb ? qok_b : qok_a;
      } else {
        tile = k_tile(smem, kst);
        full = &B.k_full[kst];
        ready = &B.k_ready[kst];
        phase = kph;
        ok = krow(i - nq, pos_i);
      }
      // the next job's table rows into the other buffer
      if (i + 1 < njobs) {
        uint32_t pos_n = 0;
        bool ok_n;
        if (i + 1 < nq) {
          ok_n = qok_b;
          pos_n = qpos_b;
        } else {
          ok_n = krow(i + 1 - nq, pos_n);
        }
        if (ok_n && !p.prerotated) fetch_table_row(p, tbl0 + (buf ^ 1u) * kRowTblBytes, pos_n, t);
      }
      cp_async_commit();
      cp_async_wait1();  // this job's rows have landed (the next one's may still be in flight)
      bad |= !wait_bar(meta, p.ctl, full, phase, p.timeout_ns);
      bad = __any_sync(0xffffffffu, bad);
      if (bad) break;
      if (ok && !p.prerotated) rope_row<BF16>(tile, t, tblp + buf * kRowTblBytes, t, isq ? p.q_mul : 1.0f);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(ready));
      buf ^= 1u;
      if (!isq) {
        kst = (kst + 1) & (kKStages - 1);
        if (kst == 0) kph ^= 1u;
      }
    }
    cp_async_wait0();
    if (bad) break;
    ++qn0;
    if (has_b) ++qn1;
  }
  cp_async_wait0();
  if (bad && lane == 0) raise_abort(meta, p.ctl);
}

// ------------------------------------------------------------------------------------
// softmax warpgroup of query tile X (128 threads; thread <-> query row <-> TMEM lane)
//
// Each warp signals the MMA issuer on its own (barriers of count 4: after the warp's TMEM
// accesses are fenced, lane 0 arrives), so warps never wait for one another; a failed wait
// is voted across the warp before any warp-collective TMEM access, so a warp leaves
// together.

template <bool BF16, bool OUT32>
__device__ void softmax_wg(const Params& p, Meta* meta, int x, uint32_t tmem) {
  Bars& B = meta->bars;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int r = (warp & 3) * 32 + lane;
  const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t tS = tmem + lane_addr + col_s(x);
  const uint32_t tP = tmem + lane_addr + col_p(x);
  const uint32_t tO = tmem + lane_addr + col_o(x);
  const int64_t hd = static_cast<int64_t>(p.H) * kD;
  // raw scores s weigh ex2(s k2 - m k2): k2 folds the score scale into the base change
  const float k2 = p.s_mul * kLog2e;

  uint32_t it = 0, sf = 0, pvd = 0, used = 0;
  bool bad = false;
  for (;;) {
    const uint32_t mb = it & 1u;
    bad |= !wait_bar(meta, p.ctl, &B.item_full[mb], (it >> 1) & 1u, p.timeout_ns);
    bad = __any_sync(0xffffffffu, bad);
    if (bad) break;
    const ItemBox& bx = meta->box[mb];
    const bool valid = bx.valid != 0;
    const bool mine = valid && (x == 0 || bx.has_b);
    const TileRec rec = x == 0 ? bx.a : bx.b;
    const int h = bx.head;
    // this query tile's stream tiles [jlo, jhi): tile j holds keys [j0, j0 + nkeys) with
    // j0 = kbase + 128 (j - jlo) and nkeys = min(128, kend - j0)
    const uint32_t jlo = x == 0 ? 0u : bx.b0, jhi = x == 0 ? bx.a1 : bx.b1;
    const uint32_t kbase = (x == 0 || bx.shared) ? bx.a.k0 + jlo * kBC : bx.b.k0;
    const uint32_t kend = bx.shared ? bx.end : rec.k0 + rec.nk;
    // a piece's sequence bounds came with the item; a group's member offsets are staged
    const uint32_t box_ss = x == 0 ? bx.ss_a : bx.ss_b, box_se = x == 0 ? bx.se_a : bx.se_b;
    const bool grp = rec.kind != 0;
    uint32_t* off = meta->cu_sm[x][used & 1u];
    if (mine && grp) stage_cu(p, rec, off, r, 128);
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(smem_u32(&B.item_empty[mb]));
      if (mine && grp) mbar_arrive(smem_u32(&B.cu_sm[x][used & 1u]));
    }
    ++it;
    if (!valid) break;
    if (!mine) continue;
    if (grp) {
      bad |= !wait_bar(meta, p.ctl, &B.cu_sm[x][used & 1u], (used >> 1) & 1u, p.timeout_ns);
      ++used;
      bad = __any_sync(0xffffffffu, bad);
      if (bad) break;
    }

    // this thread's query row and its visible key interval [lo, hi) (tokens < 2^31)
    const bool row_ok = r < static_cast<int>(rec.rows);
    const int a = static_cast<int>(rec.q0) + r;
    int lo = 0, hi = 0;
    if (row_ok) {
      uint32_t ss = box_ss, se = box_se;
      if (grp) seq_bounds(p, rec, off, static_cast<uint32_t>(a), ss, se);
      lo = static_cast<int>(ss);
      hi = static_cast<int>(se);
      if (p.window > 0) {
        lo = max(lo, a - p.window);
        hi = static_cast<int>(min(static_cast<int64_t>(hi), static_cast<int64_t>(a) + p.window + 1));
      }
    }

    float m_ref = kNeg, l = 0.f;  // running max of the raw scores, and the row sum
    for (uint32_t j = jlo; j < jhi; ++j) {
      const int j0 = static_cast<int>(kbase + (j - jlo) * kBC);
      const int nkeys = min(kBC, static_cast<int>(kend) - j0);

      // this row of S (columns past the tile's keys hold stale values; they are masked)
      bad |= !wait_bar(meta, p.ctl, &B.s_full[x], sf & 1u, p.timeout_ns);
      ++sf;
      bad = __any_sync(0xffffffffu, bad);
      if (bad) break;
      tc_fence_after();

      // visible columns [c_lo, c_hi); every other column weighs zero
      const int c_lo = min(max(lo - j0, 0), 128);
      const int c_hi = min(max(hi - j0, 0), nkeys);
      const bool full = __all_sync(0xffffffffu, c_lo == 0 && c_hi == 128);

      // Two passes over the row in halves of 64 columns, each reading its half from tensor
      // memory (the loops stay rolled: a small code footprint for the warps that share an
      // SM sub-partition). Pass 1: the row max.
      float mx = -INFINITY;
#pragma unroll 1
      for (int qq = 0; qq < 4; ++qq) {
        float v[32];
        tmem_ld32(tS + 32 * qq, v);
        if (!full) {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (static_cast<unsigned>(c + 32 * qq - c_lo) >= static_cast<unsigned>(c_hi - c_lo)) v[c] = -INFINITY;
        }
        float m0 = fmax3(v[0], v[1], v[2]), m1 = fmax3(v[3], v[4], v[5]), m2 = fmax3(v[6], v[7], v[8]),
              m3 = fmax3(v[9], v[10], v[11]);
#pragma unroll
        for (int c = 12; c < 28; c += 8) {
          m0 = fmax3(m0, v[c], v[c + 1]);
          m1 = fmax3(m1, v[c + 2], v[c + 3]);
          m2 = fmax3(m2, v[c + 4], v[c + 5]);
          m3 = fmax3(m3, v[c + 6], v[c + 7]);
        }
        mx = fmax3(mx, fmax3(m0, m1, v[28]), fmax3(fmax3(m2, m3, v[29]), v[30], v[31]));
      }
      const float m_new = fmaxf(m_ref, mx);
      const bool grow = (m_new - m_ref) * k2 > kRescale;
      float alpha = 1.f;
      if (grow) {
        alpha = ex2((m_ref - m_new) * k2);
        l *= alpha;
        m_ref = m_new;
      }
      const float mb2 = m_ref * k2;
      const float2 c2 = make_float2(k2, k2);
      const float2 nm2 = make_float2(-mb2, -mb2);
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);

      // Pass 2: probabilities of each half, written to P (the first once the previous PV
      // has read P and written O, after the O rescale that a grown max asks for).
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        float v[64];
        tmem_ld64(tS + 64 * hh, v);
        if (hh == 1) {
          // every S column of this tile is read: the next S may be issued
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&B.s_consumed[x]));
        }
        if (!full) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (static_cast<unsigned>(c + 64 * hh - c_lo) >= static_cast<unsigned>(c_hi - c_lo)) v[c] = -INFINITY;
        }
        uint32_t pp[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float2 xx = __ffma2_rn(make_float2(v[2 * c], v[2 * c + 1]), c2, nm2);
          const float2 e = make_float2(ex2(xx.x), ex2(xx.y));
          if (c & 1)
            acc1 = __fadd2_rn(acc1, e);
          else
            acc0 = __fadd2_rn(acc0, e);
          pp[c] = Elem<BF16>::pack(e.x, e.y);
        }
        if (hh == 0 && j > jlo) {
          bad |= !wait_bar(meta, p.ctl, &B.pv_done[x], pvd & 1u, p.timeout_ns);
          ++pvd;
          bad = __any_sync(0xffffffffu, bad);
          if (bad) break;
          tc_fence_after();
          if (__any_sync(0xffffffffu, grow)) {
#pragma unroll 1
            for (int oh = 0; oh < 2; ++oh) {
              float ov[32];
              tmem_ld32(tO + 32 * oh, ov);
              uint32_t ou[32];
#pragma unroll
              for (int d = 0; d < 32; ++d) ou[d] = __float_as_uint(ov[d] * alpha);
              tmem_st32(tO + 32 * oh, ou);
            }
          }
        }
        tmem_st32(tP + 32 * hh, pp);
      }
      if (bad) break;
      const float2 accs = __fadd2_rn(acc0, acc1);
      l += accs.x + accs.y;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&B.p_ready[x]));
    }
    if (bad) break;

    // epilogue: out = O / l, lse = m + ln l
    bad |= !wait_bar(meta, p.ctl, &B.pv_done[x], pvd & 1u, p.timeout_ns);
    ++pvd;
    bad = __any_sync(0xffffffffu, bad);
    if (bad) break;
    tc_fence_after();
    float ov[64];
    tmem_ld64(tO, ov);
    tc_fence_before();
    if (row_ok) {
      const float inv = 1.0f / l;
      if constexpr (OUT32) {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + (static_cast<int64_t>(a) * hd + h * kD));
#pragma unroll
        for (int q = 0; q < 16; ++q)
          dst[q] = make_float4(ov[4 * q + 0] * inv, ov[4 * q + 1] * inv, ov[4 * q + 2] * inv, ov[4 * q + 3] * inv);
      } else {
        uint4* dst =
            reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + (static_cast<int64_t>(a) * hd + h * kD));
#pragma unroll
        for (int q = 0; q < 8; ++q)
          dst[q] = make_uint4(Elem<BF16>::pack(ov[8 * q + 0] * inv, ov[8 * q + 1] * inv),
                              Elem<BF16>::pack(ov[8 * q + 2] * inv, ov[8 * q + 3] * inv),
                              Elem<BF16>::pack(ov[8 * q + 4] * inv, ov[8 * q + 5] * inv),
                              Elem<BF16>::pack(ov[8 * q + 6] * inv, ov[8 * q + 7] * inv));
      }
      p.lse[static_cast<int64_t>(h) * p.T + a] = (m_ref * k2 + lg2(l)) * kLn2;
    }
  }
  if (bad && lane == 0) raise_abort(meta, p.ctl);
}

}  // namespace

template <bool BF16, bool OUT32>
__global__ void __launch_bounds__(kThreads, 1)
pk_attend_tc_kernel(const __grid_constant__ CUtensorMap tmap_qkv, const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Meta* meta = reinterpret_cast<Meta*>(smem + kOffMeta);
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    tma_prefetch_desc(&tmap_qkv);
    Bars& B = meta->bars;
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&B.item_full[i]), 1);
      mbar_init(smem_u32(&B.item_empty[i]), kItemConsumers);
      mbar_init(smem_u32(&B.cu_rot[i]), 4);
      for (int x = 0; x < 2; ++x) {
        mbar_init(smem_u32(&B.q_full[x][i]), 1);
        mbar_init(smem_u32(&B.q_ready[x][i]), 4);
        mbar_init(smem_u32(&B.q_empty[x][i]), 1);
        mbar_init(smem_u32(&B.cu_sm[x][i]), 4);
      }
    }
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(smem_u32(&B.k_full[i]), 1);
      mbar_init(smem_u32(&B.k_ready[i]), 4);
      mbar_init(smem_u32(&B.k_empty[i]), 2);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(smem_u32(&B.v_full[i]), 1);
      mbar_init(smem_u32(&B.v_empty[i]), 2);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(&B.s_full[x]), 1);
      mbar_init(smem_u32(&B.s_consumed[x]), 4);
      mbar_init(smem_u32(&B.p_ready[x]), 4);
      mbar_init(smem_u32(&B.pv_done[x]), 1);
    }
    mbar_init(smem_u32(&B.drain[0]), 1);
    mbar_init(smem_u32(&B.drain[1]), 1);
    meta->abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(&meta->tmem), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // Register split (warpgroup-wide): the launch gives 512 x 128 = 65536 registers; the
  // producer / MMA warpgroup drops to 80 and the rotation warpgroup to 96, and the two softmax
  // warpgroups rise to 160 (ptxas compiles the code after each change within the new count;
  // the softmax code needs no more than 128): 128 x 80 + 128 x 96 + 256 x 160 = 63488.
  if (warp < kWarpRot) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 80;" ::: "memory");
    // (each role reads what it needs after its own register change: nothing computed
    // before the split stays live across it)
    if (warp == kWarpProd) {
      if (lane == 0) {
        // the records and the work counter come from the scheduler launched just before
        griddep_wait();
        const unsigned int nt = __ldcg(&p.ctl->ntiles);
        producer(&tmap_qkv, p, smem, meta, (p.singles ? nt : (nt + 1u) / 2u) * static_cast<unsigned int>(p.H));
      }
    } else if (warp == kWarpMma || warp == kWarpMma + 1) {
      if (lane == 0) mma_issuer(p, smem, meta, meta->tmem, BF16, warp - kWarpMma);
    }
  } else if (warp < kWarpSm) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 96;" ::: "memory");
    rotator<BF16>(p, smem, meta, tid - kWarpRot * 32);
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 160;" ::: "memory");
    softmax_wg<BF16, OUT32>(p, meta, (warp - kWarpSm) >> 2, meta->tmem);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(meta->tmem, kTmemCols);
  }
}

uint32_t attend_tc_smem_bytes() { return kSmemUsed + 1024; }

// Host side: opt in to the dynamic shared memory once per device.
template <bool BF16, bool OUT32>
cudaError_t attend_tc_attrs(int smem) {
  cudaError_t e =
      cudaFuncSetAttribute(pk_attend_tc_kernel<BF16, OUT32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pk_attend_tc_kernel<BF16, OUT32>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  return e;
}

cudaError_t attend_tc_prepare() {
  const int smem = static_cast<int>(attend_tc_smem_bytes());
  cudaError_t e = attend_tc_attrs<true, false>(smem);
  if (e == cudaSuccess) e = attend_tc_attrs<false, false>(smem);
  if (e == cudaSuccess) e = attend_tc_attrs<true, true>(smem);
  if (e == cudaSuccess) e = attend_tc_attrs<false, true>(smem);
  return e;
}

// Host side: one launch of `grid` persistent CTAs (one per SM: each holds all 512 TMEM
// columns and about 210 KB of shared memory).
cudaError_t attend_tc_launch(bool bf16, const CUtensorMap& tmap, const void* cos_t, const void* sin_t,
                             const uint32_t* cu, const TileRec* tiles, void* out, float* lse, Ctl* ctl, int H,
                             long long T, int window, float scale, unsigned long long timeout_ns, int grid,
                             bool singles, bool out32, bool prerotated, cudaStream_t stream) {
  Params p;
  p.cos_t = static_cast<const uint16_t*>(cos_t);
  p.sin_t = static_cast<const uint16_t*>(sin_t);
  p.cu = cu;
  p.tiles = tiles;
  p.out = out;
  p.lse = lse;
  p.ctl = ctl;
  p.H = H;
  p.T = T;
  p.window = window;
  // a positive scale is applied to the scores in the softmax (the row max of the raw
  // scores is then the max of the scaled ones); any other scale multiplies q
  p.q_mul = scale > 0.0f ? 1.0f : scale;
  p.s_mul = scale > 0.0f ? scale : 1.0f;
  p.timeout_ns = timeout_ns;
  p.singles = singles ? 1 : 0;
  p.prerotated = prerotated ? 1 : 0;
  // test hook for the bounded waits (PK_DEBUG_SKIP_ARRIVE=1): every CTA's producer withholds
  // its first work-item hand-off, so the consumers' waits run out and the call ends with
  // PK_ERR_TIMEOUT in the stream's status word; nothing faults and the context stays usable
  {
    const char* e = std::getenv("PK_DEBUG_SKIP_ARRIVE");
    p.skip_first_item_arrive = (e && e[0] == '1') ? 1 : 0;
  }
  // programmatic stream serialization: the CTAs set up (barriers, tensor memory) while the
  // scheduler finishes; the producer waits for the scheduler before it reads the records
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = attend_tc_smem_bytes();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (out32) {
    if (bf16) return cudaLaunchKernelEx(&cfg, pk_attend_tc_kernel<true, true>, tmap, p);
    return cudaLaunchKernelEx(&cfg, pk_attend_tc_kernel<false, true>, tmap, p);
  }
  if (bf16) return cudaLaunchKernelEx(&cfg, pk_attend_tc_kernel<true, false>, tmap, p);
  return cudaLaunchKernelEx(&cfg, pk_attend_tc_kernel<false, false>, tmap, p);
}

}  // namespace pk
