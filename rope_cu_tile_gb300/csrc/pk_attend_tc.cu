// pk_attend_tc.cu -- packed RoPE attention forward for bf16 / fp16 on tcgen05 (sm_103a).
//
// What it computes: hanzo-kernel 0.2.42 packed.rs fn attend -- a tile of query rows of
// one head against every key tile its window reaches, q and k rotated in the kernel
// ("the query tile, rotated and scaled"; "the key tile rotated, the value tile as is"),
// scores and the output product on the matrix units, the softmax online per row with
// masked keys weighing exactly zero, then out = O / l and lse = m + ln l.
//
// How (GB300): one persistent 384-thread CTA per SM runs two independent pipelines
// ("slots"); each slot takes work items (tile record x head) from a global counter and
// owns a Q tile, a 3-stage K/V ring in shared memory and 256 tensor-memory columns:
//     S [128 x 128] fp32    scores of the current key tile
//     P [128 x 128] 16-bit  probabilities, the A operand of the PV product
//     O [128 x  64] fp32    output accumulator
// Warps, per slot s (s = 0, 1):
//   warp s        producer (one lane): claims items, TMA-loads Q and each K/V tile
//                 (128-byte swizzle, straight from the strided qkv) into the ring;
//   warp 2 + s    MMA issuer (one lane): S(j) = Q K(j)^T once K(j) is rotated and the S
//                 columns are free; O += P(j) V(j) once P(j) is written;
//   warps 4 + 4s  softmax warpgroup: thread r owns query row r (TMEM lane r). It rotates
//   .. 7 + 4s     and scales its Q row, rotates one K row of each key tile one tile ahead
//                 (so S(j+1) runs on the tensor core while it works on S(j)), reads its S
//                 row from TMEM, masks it by the row's visible key interval, keeps a
//                 running max (the O accumulator is rescaled only when the max grows by
//                 more than a factor 2^8), writes P to TMEM, and at the end of the item
//                 writes out = O / l and lse = m + ln l.
// Every wait is bounded. A wait that times out records PK_ERR_TIMEOUT and raises the
// CTA's abort flag, which every other wait watches; the producers then wait (bounded)
// for their copies in flight, the MMA issuers for their MMAs, and the CTA frees its
// tensor memory and returns.
#include "pk_dev.cuh"

namespace pk {

namespace {

constexpr int kSlots = 2;
constexpr int kStages = 3;
constexpr int kThreads = 384;
constexpr int kWarpMma = 2;   // warps 2, 3
constexpr int kWarpWG = 4;    // warps 4..7 (slot 0), 8..11 (slot 1)

constexpr uint32_t kTileBytes = 128 * 128;                        // 128 rows x 64 x 16-bit
constexpr uint32_t kSlotBytes = kTileBytes * (1 + 2 * kStages);   // Q, K[3], V[3]

struct ItemBox {
  TileRec rec;
  int32_t head;
  int32_t valid;
  int32_t pad[6];
};

struct SlotBars {
  uint64_t item_full[2], item_empty[2];
  uint64_t q_full, q_ready, q_empty;
  uint64_t kv_full[kStages], k_ready[kStages], kv_empty[kStages];
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

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNeg = -1.0e30f;    // running-max start: ex2 of (masked - kNeg) stays 0
constexpr float kRescale = 8.0f;    // rescale O only when the max grows by more than 2^8

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

__device__ __forceinline__ uint8_t* slot_q(uint8_t* smem, int s) { return smem + s * kSlotBytes; }
__device__ __forceinline__ uint8_t* slot_k(uint8_t* smem, int s, uint32_t st) {
  return smem + s * kSlotBytes + kTileBytes * (1 + st);
}
__device__ __forceinline__ uint8_t* slot_v(uint8_t* smem, int s, uint32_t st) {
  return smem + s * kSlotBytes + kTileBytes * (1 + kStages + st);
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
    if (mbar_try_wait(a, parity)) return true;
    if ((i & 63u) == 0u) {
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

// ------------------------------------------------------------------------------------
// producer of one slot (one thread): work items and TMA loads

__device__ void producer(const CUtensorMap* tmap, const Params& p, uint8_t* smem, Meta* meta, int s,
                         unsigned int n_items) {
  SlotBars& B = meta->bars[s];
  const int32_t hd = p.H * kD;
  uint32_t it = 0, kv = 0, qn = 0;
  bool bad = false;
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
    // Q tile: the slot's Q buffer is free once the previous item's last S MMA is done
    if (!wait_bar(meta, p.ctl, &B.q_empty, (qn & 1u) ^ 1u, p.timeout_ns)) {
      bad = true;
      break;
    }
    mbar_arrive_expect_tx(smem_u32(&B.q_full), kTileBytes);
    tma_load_2d(smem_u32(slot_q(smem, s)), tmap, smem_u32(&B.q_full), h * kD, static_cast<int32_t>(rec.q0));
    ++qn;
    // K/V tiles through the ring
    for (uint32_t j = 0; j < rec.ktiles; ++j, ++kv) {
      const uint32_t st = kv % kStages;
      if (!wait_bar(meta, p.ctl, &B.kv_empty[st], ((kv / kStages) & 1u) ^ 1u, p.timeout_ns)) {
        bad = true;
        break;
      }
      const int32_t y = static_cast<int32_t>(rec.k0 + j * kBC);
      mbar_arrive_expect_tx(smem_u32(&B.kv_full[st]), 2 * kTileBytes);
      tma_load_2d(smem_u32(slot_k(smem, s, st)), tmap, smem_u32(&B.kv_full[st]), hd + h * kD, y);
      tma_load_2d(smem_u32(slot_v(smem, s, st)), tmap, smem_u32(&B.kv_full[st]), 2 * hd + h * kD, y);
    }
    if (bad) break;
  }
  if (bad || aborted(meta)) {
    // let this slot's own copies land before the CTA's shared memory goes away
    if (qn) mbar_wait(smem_u32(&B.q_full), (qn - 1) & 1u, p.timeout_ns);
    for (uint32_t t = kv > kStages ? kv - kStages : 0; t < kv; ++t)
      mbar_wait(smem_u32(&B.kv_full[t % kStages]), (t / kStages) & 1u, p.timeout_ns);
  }
}

// ------------------------------------------------------------------------------------
// MMA issuer of one slot (one thread)

__device__ void mma_issuer(const Params& p, uint8_t* smem, Meta* meta, int s, uint32_t tmem, bool bf16) {
  SlotBars& B = meta->bars[s];
  const uint32_t tS = tmem + s * 256 + kColS, tP = tmem + s * 256 + kColP, tO = tmem + s * 256 + kColO;
  const uint32_t aQ = smem_u32(slot_q(smem, s));
  const uint32_t idesc_pv = idesc_f16(bf16, 128, 64, false, true);
  uint32_t it = 0, kvc = 0, qn = 0, sc = 0, pr = 0;
  bool pending_sc = false;   // an S was issued whose consumption has not been seen yet

  // S(j) = Q K(j)^T: needs Q rotated (j = 0), K(j) rotated, and the S columns read
  auto issue_s = [&](const TileRec& rec, uint32_t j) -> bool {
    if (j == 0) {
      if (!wait_bar(meta, p.ctl, &B.q_ready, qn & 1u, p.timeout_ns)) return false;
      ++qn;
    }
    const uint32_t t = kvc + j;
    const uint32_t st = t % kStages;
    if (!wait_bar(meta, p.ctl, &B.k_ready[st], (t / kStages) & 1u, p.timeout_ns)) return false;
    if (pending_sc) {
      if (!wait_bar(meta, p.ctl, &B.s_consumed, sc & 1u, p.timeout_ns)) return false;
      ++sc;
    }
    tc_fence_after();
    const uint32_t idesc = idesc_f16(bf16, 128, round16(tile_keys(rec, j)), false, false);
    const uint32_t aK = smem_u32(slot_k(smem, s, st));
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      umma_f16_ss(tS, sdesc_sw128(aQ + ks * 32, 16, 1024), sdesc_sw128(aK + ks * 32, 16, 1024), idesc, ks > 0);
    umma_commit(smem_u32(&B.s_full));
    if (j + 1 == rec.ktiles) umma_commit(smem_u32(&B.q_empty));
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
    bool bad = !issue_s(rec, 0);
    for (uint32_t j = 0; !bad && j < rec.ktiles; ++j) {
      if (j + 1 < rec.ktiles && !issue_s(rec, j + 1)) {
        bad = true;
        break;
      }
      // O += P(j) V(j)
      if (!wait_bar(meta, p.ctl, &B.p_ready, pr & 1u, p.timeout_ns)) {
        bad = true;
        break;
      }
      ++pr;
      tc_fence_after();
      const uint32_t st = (kvc + j) % kStages;
      const uint32_t aV = smem_u32(slot_v(smem, s, st));
      const uint32_t ksteps = round16(tile_keys(rec, j)) / 16;
      for (uint32_t ks = 0; ks < ksteps; ++ks)
        umma_f16_ts(tO, tP + ks * 8, sdesc_sw128(aV + ks * 2048, 8192, 1024), idesc_pv,
                    (j > 0 || ks > 0) ? 1u : 0u);
      umma_commit(smem_u32(&B.pv_done));
      umma_commit(smem_u32(&B.kv_empty[st]));
    }
    if (bad) break;
    kvc += rec.ktiles;
  }
  // every MMA this thread issued has completed before the CTA frees tensor memory
  umma_commit(smem_u32(&B.drain));
  mbar_wait(smem_u32(&B.drain), 0, p.timeout_ns);
}

// ------------------------------------------------------------------------------------
// softmax warpgroup of one slot (128 threads; thread <-> query row <-> TMEM lane)

template <bool BF16>
__device__ void softmax_wg(const Params& p, uint8_t* smem, Meta* meta, int s, uint32_t tmem) {
  SlotBars& B = meta->bars[s];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int r = (warp & 3) * 32 + lane;  // the TMEM lane quarter of a warp is its index mod 4
  const bool elected = tid == (kWarpWG + 4 * s) * 32;
  const uint32_t bar_id = 1 + s;
  const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t tS = tmem + lane_addr + s * 256 + kColS;
  const uint32_t tP = tmem + lane_addr + s * 256 + kColP;
  const uint32_t tO = tmem + lane_addr + s * 256 + kColO;
  const int64_t hd = static_cast<int64_t>(p.H) * kD;
  uint8_t* sQ = slot_q(smem, s);

  uint32_t it = 0, kvc = 0, qn = 0, sf = 0, pvd = 0;
  bool bad = false;
  for (;;) {
    const uint32_t mb = it & 1u;
    bad |= !wait_bar(meta, p.ctl, &B.item_full[mb], (it >> 1) & 1u, p.timeout_ns);
    const ItemBox bx = meta->box[s][mb];
    bad = bar_sync_or(bar_id, 128, bad);
    if (elected && !bad) mbar_arrive(smem_u32(&B.item_empty[mb]));
    ++it;
    if (bad || !bx.valid) break;
    const TileRec rec = bx.rec;
    const int h = bx.head;

    // this thread's query row: its sequence, position and visible key interval [lo, hi)
    const bool row_ok = r < static_cast<int>(rec.rows);
    const uint32_t a = rec.q0 + r;
    int64_t lo = 0, hi = 0;
    uint32_t qpos = 0;
    if (row_ok) {
      const uint32_t sq = rec.kind == 0 ? rec.seq : seq_of_token(p.cu, rec.seq, rec.nseq, a);
      const int64_t ss = __ldg(p.cu + sq), se = __ldg(p.cu + sq + 1);
      qpos = a - static_cast<uint32_t>(ss);
      lo = ss;
      hi = se;
      if (p.window > 0) {
        lo = max(ss, static_cast<int64_t>(a) - p.window);
        hi = min(se, static_cast<int64_t>(a) + p.window + 1);
      }
    }
    const uint32_t piece_start = __ldg(p.cu + rec.seq);

    // Q: rotate and scale this thread's row
    bad |= !wait_bar(meta, p.ctl, &B.q_full, qn & 1u, p.timeout_ns);
    ++qn;
    if (row_ok && !bad) rope_row_sw128<BF16>(sQ, r, p.cos_t + qpos * kHalf, p.sin_t + qpos * kHalf, p.scale);
    fence_proxy_async_smem();
    bad = bar_sync_or(bar_id, 128, bad);
    if (bad) break;
    if (elected) mbar_arrive(smem_u32(&B.q_ready));

    // rotate key row r of key tile j (a group tile's keys are its own query rows)
    auto rotate_k = [&](uint32_t j) -> bool {
      const uint32_t st = kvc % kStages;
      bool b = !wait_bar(meta, p.ctl, &B.kv_full[st], (kvc / kStages) & 1u, p.timeout_ns);
      const uint32_t nkeys = tile_keys(rec, j);
      if (!b && r < static_cast<int>(nkeys)) {
        const uint32_t kpos = rec.kind == 0 ? rec.k0 + j * kBC + r - piece_start : qpos;
        rope_row_sw128<BF16>(slot_k(smem, s, st), r, p.cos_t + kpos * kHalf, p.sin_t + kpos * kHalf, 1.0f);
      }
      fence_proxy_async_smem();
      b = bar_sync_or(bar_id, 128, b);
      if (!b && elected) mbar_arrive(smem_u32(&B.k_ready[st]));
      ++kvc;
      return !b;
    };

    if (!rotate_k(0)) {
      bad = true;
      break;
    }
    float m_ref = kNeg, l = 0.f;
    for (uint32_t j = 0; j < rec.ktiles; ++j) {
      if (j + 1 < rec.ktiles && !rotate_k(j + 1)) {
        bad = true;
        break;
      }
      const uint32_t j0 = rec.k0 + j * kBC;
      const uint32_t nkeys = tile_keys(rec, j);

      // this row of S (columns past the tile's keys hold stale values; they are masked)
      bad |= !wait_bar(meta, p.ctl, &B.s_full, sf & 1u, p.timeout_ns);
      ++sf;
      tc_fence_after();
      float sv[128];
      tmem_ld128(tS, sv);
      tc_fence_before();
      bad = bar_sync_or(bar_id, 128, bad);
      if (bad) break;
      if (elected) mbar_arrive(smem_u32(&B.s_consumed));

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
      float mx = fmax3(sv[0], sv[1], sv[2]);
#pragma unroll
      for (int c = 3; c < 127; c += 2) mx = fmax3(mx, sv[c], sv[c + 1]);
      mx = fmaxf(mx, sv[127]);
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
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
      uint32_t pp[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float2 x = __ffma2_rn(make_float2(sv[2 * c], sv[2 * c + 1]), c2, nm2);
        const float2 e = make_float2(ex2(x.x), ex2(x.y));
        if (c & 1)
          acc1 = __fadd2_rn(acc1, e);
        else
          acc0 = __fadd2_rn(acc0, e);
        pp[c] = Elem<BF16>::pack(e.x, e.y);
      }
      const float2 acc = __fadd2_rn(acc0, acc1);
      l += acc.x + acc.y;

      // once the previous PV has read P and written O: O rescale (rare), then P
      if (j > 0) {
        bad |= !wait_bar(meta, p.ctl, &B.pv_done, pvd & 1u, p.timeout_ns);
        ++pvd;
        tc_fence_after();
        if (__any_sync(0xffffffffu, grow)) {
          float ov[64];
          tmem_ld64(tO, ov);
          uint32_t ou[64];
#pragma unroll
          for (int d = 0; d < 64; ++d) ou[d] = __float_as_uint(ov[d] * alpha);
          tmem_st32(tO, ou);
          tmem_st32(tO + 32, ou + 32);
        }
      }
      tmem_st32(tP, pp);
      tmem_st32(tP + 32, pp + 32);
      tmem_wait_st();
      tc_fence_before();
      bad = bar_sync_or(bar_id, 128, bad);
      if (bad) break;
      if (elected) mbar_arrive(smem_u32(&B.p_ready));
    }
    if (bad) break;

    // epilogue: out = O / l, lse = m + ln l
    bad |= !wait_bar(meta, p.ctl, &B.pv_done, pvd & 1u, p.timeout_ns);
    ++pvd;
    tc_fence_after();
    float ov[64];
    tmem_ld64(tO, ov);
    tc_fence_before();
    if (row_ok && !bad) {
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
    bad = bar_sync_or(bar_id, 128, bad);
    if (bad) break;
  }
  if (bad && elected) raise_abort(meta, p.ctl);
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
        mbar_init(smem_u32(&B.item_empty[k]), 2);
      }
      mbar_init(smem_u32(&B.q_full), 1);
      mbar_init(smem_u32(&B.q_ready), 1);
      mbar_init(smem_u32(&B.q_empty), 1);
      for (int k = 0; k < kStages; ++k) {
        mbar_init(smem_u32(&B.kv_full[k]), 1);
        mbar_init(smem_u32(&B.k_ready[k]), 1);
        mbar_init(smem_u32(&B.kv_empty[k]), 1);
      }
      mbar_init(smem_u32(&B.s_full), 1);
      mbar_init(smem_u32(&B.s_consumed), 1);
      mbar_init(smem_u32(&B.p_ready), 1);
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

  // Register split (warpgroup-wide): the launch gives 384 x 168 = 64512 registers; the
  // producer / MMA warpgroup drops to 56 and the two softmax warpgroups rise to 224:
  // 128 x 56 + 256 x 224 = 64512, never more than the launch holds.
  if (warp < kWarpWG) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 56;" ::: "memory");
    if (warp < kWarpMma) {
      if (lane == 0) producer(&tmap_qkv, p, smem, meta, warp, n_items);
    } else {
      if (lane == 0) mma_issuer(p, smem, meta, warp - kWarpMma, tmem, BF16);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 224;" ::: "memory");
    softmax_wg<BF16>(p, smem, meta, (warp - kWarpWG) >> 2, tmem);
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
// columns and about 220 KB of shared memory).
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
