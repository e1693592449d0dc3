// pk_attend_tc.cu -- packed RoPE attention forward for bf16 / fp16 on tcgen05 (sm_103a).
//
// What it computes: hanzo-kernel 0.2.42 packed.rs fn attend -- a tile of query rows of
// one head against every key tile its window reaches, q and k rotated in the kernel
// ("the query tile, rotated and scaled"; "the key tile rotated, the value tile as is"),
// scores and the output product on the matrix units, the softmax online per row with
// masked keys weighing exactly zero, then out = O / l and lse = m + ln l.
//
// How (GB300): one persistent 512-thread CTA per SM runs two independent pipelines
// ("slots"); each slot takes work items (tile record x head) from a global counter and
// owns, in shared memory, two Q buffers (the next item's Q is fetched and rotated while
// the current item runs), a 3-stage K ring and a 2-stage V ring, and 256 tensor-memory
// columns:
//     S [128 x 128] fp32    scores of the current key tile
//     P [128 x 128] 16-bit  probabilities, the A operand of the PV product
//     O [128 x  64] fp32    output accumulator
// Warpgroups (each warp's TMEM lane quarter is its index mod 4):
//   WG0  warp s (s = 0, 1): producer of slot s (one lane): claims items, TMA-loads Q, K and V
//        tiles (128-byte swizzle, straight from the strided qkv), K one tile ahead of V;
//        warp 2 + s: MMA issuer of slot s (one lane): S(j) = Q K(j)^T once K(j) is rotated
//        and the S columns were read, O += P(j) V(j) once P(j) is written.
//   WG1  warps 4 + 2s, 5 + 2s: rotation of slot s: 64 threads rotate (and for Q scale) two
//        rows each of every Q and K tile in shared memory as soon as it lands.
//   WG2, WG3  softmax of slot 0, 1: thread r owns query row r. It reads its S row from TMEM,
//        masks it by the row's visible key interval, keeps a running max (O is rescaled
//        only when the max grows by more than a factor 2^8), writes P to TMEM, and at the
//        end of the item writes out = O / l and lse = m + ln l.
// Every wait is bounded. A wait that times out records PK_ERR_TIMEOUT and raises the
// CTA's abort flag, which every other wait watches; the producers then wait (bounded)
// for their copies in flight, the MMA issuers for their MMAs, and the CTA frees its
// tensor memory and returns.
#include "pk_dev.cuh"

namespace pk {

namespace {

constexpr int kSlots = 2;
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kThreads = 512;
constexpr int kWarpMma = 2;    // warps 2, 3
constexpr int kWarpRot = 4;    // warps 4, 5 (slot 0), 6, 7 (slot 1)
constexpr int kWarpSm = 8;     // warps 8..11 (slot 0), 12..15 (slot 1)
constexpr int kRotThreads = 64;

constexpr uint32_t kTileBytes = 128 * 128;  // 128 rows x 64 x 16-bit
constexpr uint32_t kSlotBytes = kTileBytes * (2 + kKStages + kVStages);

struct ItemBox {
  TileRec rec;
  int32_t head;
  int32_t valid;
  int32_t pad[6];
};

struct SlotBars {
  uint64_t item_full[2], item_empty[2];
  uint64_t q_full[2], q_ready[2], q_empty[2];
  uint64_t k_full[kKStages], k_ready[kKStages], k_empty[kKStages];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t s_full, s_consumed, p_ready, pv_done;
  uint64_t drain;
};

struct Meta {
  SlotBars bars[kSlots];
  ItemBox box[kSlots][2];
  uint32_t tmem;
  int32_t abort;
};

constexpr uint32_t kOffMeta = kSlots * kSlotBytes;
constexpr uint32_t kSmemUsed = kOffMeta + sizeof(Meta);
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColP = 128, kColO = 192;  // within a slot's 256 columns
constexpr uint32_t kItemConsumers = 1 + kRotThreads / 32 + 4;  // MMA issuer + rotation warps + softmax warps

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

__device__ __forceinline__ uint8_t* slot_q(uint8_t* smem, int s, uint32_t b) {
  return smem + s * kSlotBytes + kTileBytes * b;
}
__device__ __forceinline__ uint8_t* slot_k(uint8_t* smem, int s, uint32_t st) {
  return smem + s * kSlotBytes + kTileBytes * (2 + st);
}
__device__ __forceinline__ uint8_t* slot_v(uint8_t* smem, int s, uint32_t st) {
  return smem + s * kSlotBytes + kTileBytes * (2 + kKStages + st);
}

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

// keys of key tile j of a record: min(128, nk - 128 j)
__device__ __forceinline__ uint32_t tile_keys(const TileRec& rec, uint32_t j) {
  return min(static_cast<uint32_t>(kBC), rec.nk - j * kBC);
}
__device__ __forceinline__ uint32_t round16(uint32_t n) { return (n + 15u) & ~15u; }

// The cos / sin table rows of one position (32 16-bit values each, four 16-byte chunks).
struct RopeRow {
  uint4 c[4], s[4];
};

__device__ __forceinline__ RopeRow load_rope_row(const uint16_t* cos_t, const uint16_t* sin_t, uint32_t pos) {
  RopeRow t;
  const uint4* c = reinterpret_cast<const uint4*>(cos_t + static_cast<size_t>(pos) * kHalf);
  const uint4* s = reinterpret_cast<const uint4*>(sin_t + static_cast<size_t>(pos) * kHalf);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    t.c[k] = __ldg(c + k);
    t.s[k] = __ldg(s + k);
  }
  return t;
}

// Rotate and multiply by `mul` row r of a 128-byte-swizzled 64-column tile in
// place: y[u] = x[u] c - x[u+32] s, y[u+32] = x[u] s + x[u+32] c, in fp32 straight from the
// 16-bit operands. Elements u and u + 32 are logical 16-byte chunks c and c + 4, stored at
// chunks (c ^ (r & 7)) and ((c + 4) ^ (r & 7)).
template <bool BF16>
__device__ __forceinline__ void rope_row_sw128(uint8_t* tile, int r, const RopeRow t, float mul) {
  using E = Elem<BF16>;
  uint8_t* row = tile + r * 128;
  const int sw = r & 7;
  // two halves of the row; within a half every chunk is read before any is written back
#pragma unroll 1
  for (int hh = 0; hh < 2; ++hh) {
    uint4 x1[2], x2[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int c = 2 * hh + q;
      x1[q] = *reinterpret_cast<const uint4*>(row + ((c ^ sw) << 4));
      x2[q] = *reinterpret_cast<const uint4*>(row + (((c + 4) ^ sw) << 4));
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int c = 2 * hh + q;
      const uint4 tc = hh ? t.c[2 + q] : t.c[q];
      const uint4 ts = hh ? t.s[2 + q] : t.s[q];
      const uint32_t a[4] = {x1[q].x, x1[q].y, x1[q].z, x1[q].w};
      const uint32_t b[4] = {x2[q].x, x2[q].y, x2[q].z, x2[q].w};
      const uint32_t cc[4] = {tc.x, tc.y, tc.z, tc.w};
      const uint32_t ss[4] = {ts.x, ts.y, ts.z, ts.w};
      uint32_t y1[4], y2[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float lo1 = E::fma_lo(a[k], cc[k], -E::fma_lo(b[k], ss[k], 0.f));
        const float hi1 = E::fma_hi(a[k], cc[k], -E::fma_hi(b[k], ss[k], 0.f));
        const float lo2 = E::fma_lo(a[k], ss[k], E::fma_lo(b[k], cc[k], 0.f));
        const float hi2 = E::fma_hi(a[k], ss[k], E::fma_hi(b[k], cc[k], 0.f));
        y1[k] = E::pack(lo1 * mul, hi1 * mul);
        y2[k] = E::pack(lo2 * mul, hi2 * mul);
      }
      *reinterpret_cast<uint4*>(row + ((c ^ sw) << 4)) = make_uint4(y1[0], y1[1], y1[2], y1[3]);
      *reinterpret_cast<uint4*>(row + (((c + 4) ^ sw) << 4)) = make_uint4(y2[0], y2[1], y2[2], y2[3]);
    }
  }
}

struct Params {
  const uint16_t* cos_t;
  const uint16_t* sin_t;
  const uint32_t* cu;
  const TileRec* tiles;
  uint16_t* out;
  float* lse;
  Ctl* ctl;
  int H;
  long long T;
  int window;
  float scale;
  unsigned long long timeout_ns;
};

// in-sequence position of token a of a record (a group's rows belong to several sequences)
__device__ __forceinline__ uint32_t position_of(const Params& p, const TileRec& rec, uint32_t a,
                                                uint32_t piece_start) {
  if (rec.kind == 0) return a - piece_start;
  const uint32_t sq = seq_of_token(p.cu, rec.seq, rec.nseq, a);
  return a - __ldg(p.cu + sq);
}

// ------------------------------------------------------------------------------------
// producer of one slot (one thread): work items and TMA loads. Per item: Q into buffer
// (item count & 1), then K(0), K(1), V(0), K(2), V(1), ... so each K tile is requested a
// tile ahead of its V.

struct Ring {
  uint32_t n = 0;  // uses so far
  __device__ __forceinline__ uint32_t stage(uint32_t depth) const { return n % depth; }
  __device__ __forceinline__ uint32_t phase(uint32_t depth) const { return (n / depth) & 1u; }
};

__device__ void producer(const CUtensorMap* tmap, const Params& p, uint8_t* smem, Meta* meta, int s,
                         unsigned int n_items) {
  SlotBars& B = meta->bars[s];
  const int32_t hd = p.H * kD;
  uint32_t it = 0;
  Ring q, k, v;
  bool bad = false;

  auto load_k = [&](const TileRec& rec, int h, uint32_t j) -> bool {
    const uint32_t st = k.stage(kKStages);
    if (!wait_bar(meta, p.ctl, &B.k_empty[st], k.phase(kKStages) ^ 1u, p.timeout_ns)) return false;
    mbar_arrive_expect_tx(smem_u32(&B.k_full[st]), kTileBytes);
    tma_load_2d(smem_u32(slot_k(smem, s, st)), tmap, smem_u32(&B.k_full[st]), hd + h * kD,
                static_cast<int32_t>(rec.k0 + j * kBC));
    ++k.n;
    return true;
  };
  auto load_v = [&](const TileRec& rec, int h, uint32_t j) -> bool {
    const uint32_t st = v.stage(kVStages);
    if (!wait_bar(meta, p.ctl, &B.v_empty[st], v.phase(kVStages) ^ 1u, p.timeout_ns)) return false;
    mbar_arrive_expect_tx(smem_u32(&B.v_full[st]), kTileBytes);
    tma_load_2d(smem_u32(slot_v(smem, s, st)), tmap, smem_u32(&B.v_full[st]), 2 * hd + h * kD,
                static_cast<int32_t>(rec.k0 + j * kBC));
    ++v.n;
    return true;
  };

  for (;;) {
    const unsigned int item = atomicAdd(&p.ctl->next, 1u);
    const uint32_t mb = it & 1u;
    if (!wait_bar(meta, p.ctl, &B.item_empty[mb], ((it >> 1) & 1u) ^ 1u, p.timeout_ns)) {
      bad = true;
      break;
    }
    ItemBox& bx = meta->box[s][mb];
    if (item >= n_items) {
      bx.valid = 0;
      mbar_arrive(smem_u32(&B.item_full[mb]));
      break;
    }
    const unsigned int ti = item / static_cast<unsigned int>(p.H);
    const int h = static_cast<int>(item % static_cast<unsigned int>(p.H));
    const TileRec rec = p.tiles[ti];
    bx.rec = rec;
    bx.head = h;
    bx.valid = 1;
    mbar_arrive(smem_u32(&B.item_full[mb]));
    ++it;
    // Q into its buffer once the item two back has finished its last S
    const uint32_t qb = q.stage(2);
    if (!wait_bar(meta, p.ctl, &B.q_empty[qb], q.phase(2) ^ 1u, p.timeout_ns)) {
      bad = true;
      break;
    }
    mbar_arrive_expect_tx(smem_u32(&B.q_full[qb]), kTileBytes);
    tma_load_2d(smem_u32(slot_q(smem, s, qb)), tmap, smem_u32(&B.q_full[qb]), h * kD, static_cast<int32_t>(rec.q0));
    ++q.n;
    const uint32_t n = rec.ktiles;
    bad = !load_k(rec, h, 0) || (n > 1 && !load_k(rec, h, 1));
    for (uint32_t j = 0; !bad && j < n; ++j)
      bad = !load_v(rec, h, j) || (j + 2 < n && !load_k(rec, h, j + 2));
    if (bad) break;
  }
  if (bad || aborted(meta)) {
    // let this slot's own copies land before the CTA's shared memory goes away
    for (uint32_t t = q.n > 2 ? q.n - 2 : 0; t < q.n; ++t)
      mbar_wait(smem_u32(&B.q_full[t % 2]), (t / 2) & 1u, p.timeout_ns);
    for (uint32_t t = k.n > kKStages ? k.n - kKStages : 0; t < k.n; ++t)
      mbar_wait(smem_u32(&B.k_full[t % kKStages]), (t / kKStages) & 1u, p.timeout_ns);
    for (uint32_t t = v.n > kVStages ? v.n - kVStages : 0; t < v.n; ++t)
      mbar_wait(smem_u32(&B.v_full[t % kVStages]), (t / kVStages) & 1u, p.timeout_ns);
  }
}

// ------------------------------------------------------------------------------------
// MMA issuer of one slot (one thread)

__device__ void mma_issuer(const Params& p, uint8_t* smem, Meta* meta, int s, uint32_t tmem, bool bf16) {
  SlotBars& B = meta->bars[s];
  const uint32_t tS = tmem + s * 256 + kColS, tP = tmem + s * 256 + kColP, tO = tmem + s * 256 + kColO;
  const uint32_t idesc_pv = idesc_f16(bf16, 128, 64, false, true);
  // operand descriptors of every buffer, computed once; a K step of 16 adds 32 bytes (Q, K)
  // or 2048 bytes (V) to the start address field (address >> 4)
  // (buffers of one kind are consecutive 16 KB tiles: the next one is 1024 further)
  const uint64_t dq0 = sdesc_sw128(smem_u32(slot_q(smem, s, 0)), 16, 1024);
  const uint64_t dk0 = sdesc_sw128(smem_u32(slot_k(smem, s, 0)), 16, 1024);
  const uint64_t dv0 = sdesc_sw128(smem_u32(slot_v(smem, s, 0)), 8192, 1024);
  uint32_t it = 0, sc = 0, pr = 0;
  Ring q, k, v;
  bool pending_sc = false;  // an S was issued whose consumption has not been seen yet

  // S(j) = Q K(j)^T: needs Q rotated (j = 0), K(j) rotated, and the S columns read
  auto issue_s = [&](const TileRec& rec, uint32_t j, uint32_t qb) -> bool {
    if (j == 0) {
      if (!wait_bar(meta, p.ctl, &B.q_ready[qb], q.phase(2), p.timeout_ns)) return false;
    }
    const uint32_t st = k.stage(kKStages);
    if (!wait_bar(meta, p.ctl, &B.k_ready[st], k.phase(kKStages), p.timeout_ns)) return false;
    if (pending_sc) {
      if (!wait_bar(meta, p.ctl, &B.s_consumed, sc & 1u, p.timeout_ns)) return false;
      ++sc;
    }
    tc_fence_after();
    const uint32_t idesc = idesc_f16(bf16, 128, round16(tile_keys(rec, j)), false, false);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      umma_f16_ss(tS, dq0 + qb * 1024 + ks * 2, dk0 + st * 1024 + ks * 2, idesc, ks > 0);
    umma_commit(smem_u32(&B.s_full));
    umma_commit(smem_u32(&B.k_empty[st]));
    if (j + 1 == rec.ktiles) umma_commit(smem_u32(&B.q_empty[qb]));
    ++k.n;
    pending_sc = true;
    return true;
  };

  for (;;) {
    const uint32_t mb = it & 1u;
    if (!wait_bar(meta, p.ctl, &B.item_full[mb], (it >> 1) & 1u, p.timeout_ns)) break;
    const ItemBox bx = meta->box[s][mb];
    mbar_arrive(smem_u32(&B.item_empty[mb]));
    ++it;
    if (!bx.valid) break;
    const TileRec rec = bx.rec;
    const uint32_t qb = q.stage(2);
    bool bad = false;
    // step t: S(t) (t < ktiles), then PV(t - 1) (t >= 1)
    for (uint32_t t = 0; !bad && t <= rec.ktiles; ++t) {
      if (t < rec.ktiles && !issue_s(rec, t, qb)) {
        bad = true;
        break;
      }
      if (t == 0) continue;
      const uint32_t j = t - 1;
      // O += P(j) V(j)
      if (!wait_bar(meta, p.ctl, &B.p_ready, pr & 1u, p.timeout_ns)) {
        bad = true;
        break;
      }
      ++pr;
      const uint32_t st = v.stage(kVStages);
      if (!wait_bar(meta, p.ctl, &B.v_full[st], v.phase(kVStages), p.timeout_ns)) {
        bad = true;
        break;
      }
      tc_fence_after();
      const uint32_t ksteps = round16(tile_keys(rec, j)) / 16;
#pragma unroll
      for (uint32_t ks = 0; ks < 8; ++ks)
        if (ks < ksteps)
          umma_f16_ts(tO, tP + ks * 8, dv0 + st * 1024 + ks * 128, idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
      umma_commit(smem_u32(&B.pv_done));
      umma_commit(smem_u32(&B.v_empty[st]));
      ++v.n;
    }
    if (bad) break;
    ++q.n;
  }
  // every MMA this thread issued has completed before the CTA frees tensor memory
  umma_commit(smem_u32(&B.drain));
  mbar_wait(smem_u32(&B.drain), 0, p.timeout_ns);
}

// ------------------------------------------------------------------------------------
// rotation warps of one slot (64 threads, rows t and t + 64 of every tile)
//
// For each item: job 0 rotates and scales the Q tile, job 1 + j rotates K tile j, each as
// soon as it lands. Each warp arrives on the ready barrier once its rows are written and
// fenced (count 2); a failed wait is voted across the warp so a warp leaves together.

template <bool BF16>
__device__ void rotator(const Params& p, uint8_t* smem, Meta* meta, int s, int t) {
  SlotBars& B = meta->bars[s];
  uint32_t it = 0;
  Ring q, k;
  bool bad = false;
  for (;;) {
    const uint32_t mb = it & 1u;
    bad |= !wait_bar(meta, p.ctl, &B.item_full[mb], (it >> 1) & 1u, p.timeout_ns);
    bad = __any_sync(0xffffffffu, bad);
    if (bad) break;
    const ItemBox bx = meta->box[s][mb];
    __syncwarp();
    if ((t & 31) == 0) mbar_arrive(smem_u32(&B.item_empty[mb]));
    ++it;
    if (!bx.valid) break;
    const TileRec rec = bx.rec;
    const uint32_t piece_start = __ldg(p.cu + rec.seq);
    // positions of this thread's two query rows (for a group tile, also of its two key rows)
    const uint32_t pos0 = t < static_cast<int>(rec.rows) ? position_of(p, rec, rec.q0 + t, piece_start) : 0u;
    const uint32_t pos1 = t + 64 < static_cast<int>(rec.rows) ? position_of(p, rec, rec.q0 + t + 64, piece_start) : 0u;

#pragma unroll 1
    for (uint32_t job = 0; job <= rec.ktiles; ++job) {
      const bool isq = job == 0;
      const uint32_t j = job - 1;
      const uint32_t nrows = isq ? rec.rows : tile_keys(rec, j);
      const uint32_t base = isq ? 0u : rec.k0 + j * kBC - piece_start;
      const uint32_t st = isq ? q.stage(2) : k.stage(kKStages);
      const uint32_t ph = isq ? q.phase(2) : k.phase(kKStages);
      uint64_t* full = isq ? &B.q_full[st] : &B.k_full[st];
      uint64_t* ready = isq ? &B.q_ready[st] : &B.k_ready[st];
      uint8_t* tile = isq ? slot_q(smem, s, st) : slot_k(smem, s, st);
      const float mul = isq ? p.scale : 1.0f;
      // table positions of the two rows (row 0 of the tables for rows past the tile)
      auto pos_of = [&](int r, uint32_t qp) -> uint32_t {
        if (r >= static_cast<int>(nrows)) return 0u;
        return (isq || rec.kind != 0) ? qp : base + r;
      };
      const uint32_t kp1 = pos_of(t + 64, pos1);
      RopeRow cur = load_rope_row(p.cos_t, p.sin_t, pos_of(t, pos0));
      bad |= !wait_bar(meta, p.ctl, full, ph, p.timeout_ns);
      bad = __any_sync(0xffffffffu, bad);
      if (bad) break;
#pragma unroll 1
      for (int rr = 0; rr < 2; ++rr) {
        const RopeRow nxt = load_rope_row(p.cos_t, p.sin_t, rr == 0 ? kp1 : 0u);
        const int r = t + 64 * rr;
        if (r < static_cast<int>(nrows)) rope_row_sw128<BF16>(tile, r, cur, mul);
        cur = nxt;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if ((t & 31) == 0) mbar_arrive(smem_u32(ready));
      if (isq)
        ++q.n;
      else
        ++k.n;
    }
    if (bad) break;
  }
  if (bad && (t & 31) == 0) raise_abort(meta, p.ctl);
}

// ------------------------------------------------------------------------------------
// softmax warpgroup of one slot (128 threads; thread <-> query row <-> TMEM lane)
//
// Each warp signals the MMA issuer on its own (barriers of count 4: after the warp's TMEM
// accesses are fenced, lane 0 arrives), so warps never wait for one another; a failed wait
// is voted across the warp before any warp-collective TMEM access, so a warp leaves
// together.

template <bool BF16>
__device__ void softmax_wg(const Params& p, Meta* meta, int s, uint32_t tmem) {
  SlotBars& B = meta->bars[s];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int r = (warp & 3) * 32 + lane;
  const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t tS = tmem + lane_addr + s * 256 + kColS;
  const uint32_t tP = tmem + lane_addr + s * 256 + kColP;
  const uint32_t tO = tmem + lane_addr + s * 256 + kColO;
  const int64_t hd = static_cast<int64_t>(p.H) * kD;

  uint32_t it = 0, sf = 0, pvd = 0;
  bool bad = false;
  for (;;) {
    const uint32_t mb = it & 1u;
    bad |= !wait_bar(meta, p.ctl, &B.item_full[mb], (it >> 1) & 1u, p.timeout_ns);
    bad = __any_sync(0xffffffffu, bad);
    if (bad) break;
    const ItemBox bx = meta->box[s][mb];
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&B.item_empty[mb]));
    ++it;
    if (!bx.valid) break;
    const TileRec rec = bx.rec;
    const int h = bx.head;

    // this thread's query row and its visible key interval [lo, hi)
    const bool row_ok = r < static_cast<int>(rec.rows);
    const uint32_t a = rec.q0 + r;
    int64_t lo = 0, hi = 0;
    if (row_ok) {
      const uint32_t sq = rec.kind == 0 ? rec.seq : seq_of_token(p.cu, rec.seq, rec.nseq, a);
      const int64_t ss = __ldg(p.cu + sq), se = __ldg(p.cu + sq + 1);
      lo = ss;
      hi = se;
      if (p.window > 0) {
        lo = max(ss, static_cast<int64_t>(a) - p.window);
        hi = min(se, static_cast<int64_t>(a) + p.window + 1);
      }
    }

    float m_ref = kNeg, l = 0.f;
    for (uint32_t j = 0; j < rec.ktiles; ++j) {
      const uint32_t j0 = rec.k0 + j * kBC;
      const uint32_t nkeys = tile_keys(rec, j);

      // this row of S (columns past the tile's keys hold stale values; they are masked)
      bad |= !wait_bar(meta, p.ctl, &B.s_full, sf & 1u, p.timeout_ns);
      ++sf;
      bad = __any_sync(0xffffffffu, bad);
      if (bad) break;
      tc_fence_after();
      float sv[128];
      tmem_ld64(tS, *reinterpret_cast<float(*)[64]>(sv));
      tmem_ld64(tS + 64, *reinterpret_cast<float(*)[64]>(sv + 64));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&B.s_consumed));

      // visible columns [c_lo, c_hi); every other column weighs zero
      const int c_lo = static_cast<int>(
          min(max(lo - static_cast<int64_t>(j0), static_cast<int64_t>(0)), static_cast<int64_t>(128)));
      const int c_hi = static_cast<int>(
          min(max(hi - static_cast<int64_t>(j0), static_cast<int64_t>(0)), static_cast<int64_t>(nkeys)));
      const bool full = __all_sync(0xffffffffu, c_lo == 0 && c_hi == 128);
      if (!full) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c < c_lo || c >= c_hi) sv[c] = -INFINITY;
      }
      // row max: eight independent chains, then a tree
      float mk[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mk[k] = fmax3(sv[k], sv[8 + k], sv[16 + k]);
#pragma unroll
      for (int c = 24; c < 128; c += 16) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mk[k] = (c + 8 + k < 128) ? fmax3(mk[k], sv[c + k], sv[c + 8 + k]) : fmaxf(mk[k], sv[c + k]);
      }
      const float mx = fmaxf(fmax3(mk[0], mk[1], mk[2]), fmax3(fmax3(mk[3], mk[4], mk[5]), mk[6], mk[7]));
      const float m_new = fmaxf(m_ref, mx);
      const bool grow = (m_new - m_ref) * kLog2e > kRescale;
      float alpha = 1.f;
      if (grow) {
        alpha = ex2((m_ref - m_new) * kLog2e);
        l *= alpha;
        m_ref = m_new;
      }
      const float mb2 = m_ref * kLog2e;
      const float2 c2 = make_float2(kLog2e, kLog2e);
      const float2 nm2 = make_float2(-mb2, -mb2);
      float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      uint32_t pp[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float2 x = __ffma2_rn(make_float2(sv[2 * c], sv[2 * c + 1]), c2, nm2);
        const float2 e = make_float2(ex2(x.x), ex2(x.y));
        acc[c & 3] = __fadd2_rn(acc[c & 3], e);
        pp[c] = Elem<BF16>::pack(e.x, e.y);
      }
      const float2 accs = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
      l += accs.x + accs.y;

      // once the previous PV has read P and written O: O rescale (rare), then P
      if (j > 0) {
        bad |= !wait_bar(meta, p.ctl, &B.pv_done, pvd & 1u, p.timeout_ns);
        ++pvd;
        bad = __any_sync(0xffffffffu, bad);
        if (bad) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, grow)) {
#pragma unroll 1
          for (int hh = 0; hh < 2; ++hh) {
            float ov[32];
            tmem_ld32(tO + 32 * hh, ov);
            uint32_t ou[32];
#pragma unroll
            for (int d = 0; d < 32; ++d) ou[d] = __float_as_uint(ov[d] * alpha);
            tmem_st32(tO + 32 * hh, ou);
          }
        }
      }
      tmem_st32(tP, pp);
      tmem_st32(tP + 32, pp + 32);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&B.p_ready));
    }
    if (bad) break;

    // epilogue: out = O / l, lse = m + ln l
    bad |= !wait_bar(meta, p.ctl, &B.pv_done, pvd & 1u, p.timeout_ns);
    ++pvd;
    bad = __any_sync(0xffffffffu, bad);
    if (bad) break;
    tc_fence_after();
    float ov[64];
    tmem_ld64(tO, ov);
    tc_fence_before();
    if (row_ok) {
      const float inv = 1.0f / l;
      uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(a) * hd + h * kD));
#pragma unroll
      for (int q = 0; q < 8; ++q)
        dst[q] = make_uint4(Elem<BF16>::pack(ov[8 * q + 0] * inv, ov[8 * q + 1] * inv),
                            Elem<BF16>::pack(ov[8 * q + 2] * inv, ov[8 * q + 3] * inv),
                            Elem<BF16>::pack(ov[8 * q + 4] * inv, ov[8 * q + 5] * inv),
                            Elem<BF16>::pack(ov[8 * q + 6] * inv, ov[8 * q + 7] * inv));
      p.lse[static_cast<int64_t>(h) * p.T + a] = m_ref + lg2(l) * kLn2;
    }
  }
  if (bad && lane == 0) raise_abort(meta, p.ctl);
}


}  // namespace

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
pk_attend_tc_kernel(const __grid_constant__ CUtensorMap tmap_qkv, Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Meta* meta = reinterpret_cast<Meta*>(smem + kOffMeta);
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    tma_prefetch_desc(&tmap_qkv);
    for (int s = 0; s < kSlots; ++s) {
      SlotBars& B = meta->bars[s];
      for (int k = 0; k < 2; ++k) {
        mbar_init(smem_u32(&B.item_full[k]), 1);
        mbar_init(smem_u32(&B.item_empty[k]), kItemConsumers);
        mbar_init(smem_u32(&B.q_full[k]), 1);
        mbar_init(smem_u32(&B.q_ready[k]), kRotThreads / 32);
        mbar_init(smem_u32(&B.q_empty[k]), 1);
      }
      for (int k = 0; k < kKStages; ++k) {
        mbar_init(smem_u32(&B.k_full[k]), 1);
        mbar_init(smem_u32(&B.k_ready[k]), kRotThreads / 32);
        mbar_init(smem_u32(&B.k_empty[k]), 1);
      }
      for (int k = 0; k < kVStages; ++k) {
        mbar_init(smem_u32(&B.v_full[k]), 1);
        mbar_init(smem_u32(&B.v_empty[k]), 1);
      }
      mbar_init(smem_u32(&B.s_full), 1);
      mbar_init(smem_u32(&B.s_consumed), 4);
      mbar_init(smem_u32(&B.p_ready), 4);
      mbar_init(smem_u32(&B.pv_done), 1);
      mbar_init(smem_u32(&B.drain), 1);
    }
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
  const uint32_t tmem = meta->tmem;
  const unsigned int n_items = __ldcg(&p.ctl->ntiles) * static_cast<unsigned int>(p.H);

  // Register split (warpgroup-wide): the launch gives 512 x 128 = 65536 registers; the
  // producer / MMA warpgroup drops to 48, the rotation warpgroup to 112, and the two softmax
  // warpgroups rise to 168: 128 x 48 + 128 x 112 + 256 x 168 = 63488, within the launch.
  if (warp < kWarpRot) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 48;" ::: "memory");
    if (warp < kWarpMma) {
      if (lane == 0) producer(&tmap_qkv, p, smem, meta, warp, n_items);
    } else {
      if (lane == 0) mma_issuer(p, smem, meta, warp - kWarpMma, tmem, BF16);
    }
  } else if (warp < kWarpSm) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 112;" ::: "memory");
    const int s = (warp - kWarpRot) >> 1;
    rotator<BF16>(p, smem, meta, s, tid - (kWarpRot + 2 * s) * 32);
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 168;" ::: "memory");
    softmax_wg<BF16>(p, meta, (warp - kWarpSm) >> 2, tmem);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
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

// Host side: one launch of `grid` persistent CTAs (one per SM: each holds all 512 TMEM
// columns and about 225 KB of shared memory).
cudaError_t attend_tc_launch(bool bf16, const CUtensorMap& tmap, const void* cos_t, const void* sin_t,
                             const uint32_t* cu, const TileRec* tiles, void* out, float* lse, Ctl* ctl, int H,
                             long long T, int window, float scale, unsigned long long timeout_ns, int grid,
                             cudaStream_t stream) {
  Params p;
  p.cos_t = static_cast<const uint16_t*>(cos_t);
  p.sin_t = static_cast<const uint16_t*>(sin_t);
  p.cu = cu;
  p.tiles = tiles;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.ctl = ctl;
  p.H = H;
  p.T = T;
  p.window = window;
  p.scale = scale;
  p.timeout_ns = timeout_ns;
  const uint32_t smem = attend_tc_smem_bytes();
  if (bf16)
    pk_attend_tc_kernel<true><<<grid, kThreads, smem, stream>>>(tmap, p);
  else
    pk_attend_tc_kernel<false><<<grid, kThreads, smem, stream>>>(tmap, p);
  return cudaGetLastError();
}

}  // namespace pk
