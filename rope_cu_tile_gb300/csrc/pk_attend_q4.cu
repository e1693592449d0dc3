// pk_attend_q4.cu -- packed RoPE attention forward for bf16 / fp16 on tcgen05 (sm_103a),
// with four query tiles in flight per SM.
//
// What it computes: hanzo-kernel 0.2.42 packed.rs fn attend -- a tile of query rows of
// one head against every key tile its window reaches, q and k rotated in the kernel, the
// scores and the output product on the matrix units, the softmax online per row with
// masked keys weighing exactly zero, then out = O / l and lse = m + ln l.
//
// How (GB300): one persistent 768-thread CTA per SM running two independent PIPES. Each pipe
// claims work items on its own: a PAIR of consecutive tile records (A, B) of one head. When
// A and B are pieces of one sequence with the same key range they share one key stream
// (every 64-key K / V tile is loaded and rotated once for both query tiles); otherwise A's
// and B's key tiles alternate in the stream, so both query tiles always advance together.
// Each query tile is a CHAIN: S = Q K^T (tcgen05, M = 128, N = 64), the softmax of those
// scores by one warpgroup, P written over S in tensor memory, O += P V (tcgen05, P read from
// tensor memory), and the next S issued right behind that PV product (MMAs of one thread run
// in order, so the next S cannot overwrite P before the PV product has read it). Four
// chains per SM keep the tensor pipe busy while each chain waits for its own softmax, and
// one pipe's item start-up (Q load and rotation) runs under the other pipe's work.
//
// Shared memory: the four Q tiles (16 KB each, single-buffered), per pipe a 4-stage K ring
// and a 3-stage V ring of 64-key tiles (8 KB each), and per rotation thread two 128-byte
// cos / sin table rows. Tensor memory (512 columns): per chain c, S_c (fp32, 64 columns,
// P over its first 32) at 128 c and O_c (fp32, 64 columns) at 128 c + 64.
// Warps (each warp's TMEM lane quarter is its index mod 4):
//   WG0  warps 0, 1: producer of pipe 0, 1 (one lane): claims items, TMA-loads (128-byte
//        swizzle, straight from the strided qkv) the stream's first two K tiles, Q_A, Q_B,
//        then K two tiles ahead of V; warps 2, 3: MMA issuer of pipe 0, 1 (one lane).
//   WG1  rotation: warps 4-5 for pipe 0, 6-7 for pipe 1; thread t rotates row t of every
//        64-row K tile and rows t, t + 64 of every Q tile of its pipe, in shared memory.
//   WG2..WG5  softmax of chains (pipe 0, A), (0, B), (1, A), (1, B): thread r owns query row
//        r = TMEM lane r. It reads its 64 scores of a tile from TMEM once, masks them by the
//        row's visible key interval, applies a positive scale inside exp2, keeps a running
//        max (O is rescaled only when the max grows by more than 2^8), writes P to TMEM, and
//        at the end of the item writes out = O / l and lse = m + ln l.
// Every wait is bounded. A wait that times out records PK_ERR_TIMEOUT and raises the
// CTA's abort flag, which every other wait watches; the producers then wait (bounded) for
// their copies in flight, the MMA issuers for their MMAs, and the CTA frees its tensor
// memory and returns.
#include <cstdlib>

#include "pk_attn_common.cuh"

namespace pk {

namespace {

using namespace attn;

constexpr int kThreads = 768;
constexpr int kPipes = 2;
constexpr int kKeys = 64;    // keys per stream tile
constexpr int kKStages = 4;  // K ring depth per pipe (a power of two)
constexpr int kVStages = 3;  // V ring depth per pipe
constexpr int kWarpProd = 0;  // warps 0, 1
constexpr int kWarpMma = 2;   // warps 2, 3
constexpr int kWarpRot = 4;   // warps 4..7
constexpr int kWarpSm = 8;    // warps 8..23

constexpr uint32_t kQBytes = 128 * 128;   // 128 rows x 64 x 16-bit
constexpr uint32_t kKVBytes = 64 * 128;   // 64 rows x 64 x 16-bit
// shared-memory map (offsets from the 1024-aligned base); every tile starts on 1024 bytes
constexpr uint32_t kOffQ = 0;                                          // [chain]
constexpr uint32_t kOffK = kOffQ + 4 * kQBytes;                        // [pipe][stage]
constexpr uint32_t kOffV = kOffK + kPipes * kKStages * kKVBytes;       // [pipe][stage]
constexpr uint32_t kOffTbl = kOffV + kPipes * kVStages * kKVBytes;     // [rotation thread][2]
constexpr uint32_t kOffMeta = kOffTbl + 128 * 2 * kRowTblBytes;

// One work item of a pipe as its producer hands it to the other roles.
struct ItemBox {
  TileRec a, b;
  int32_t head;
  int32_t valid;     // 0: no more work
  uint32_t has_b;    // 1: B is a record
  uint32_t shared;   // 1: A and B read one key stream; 0: their key tiles alternate
  uint32_t na, nb;   // key tiles of A and B (64 keys each)
  uint32_t n;        // key tiles in the stream
  uint32_t ss_a, se_a, ss_b, se_b;  // first and end token of the sequence of a piece
  uint32_t pad[5];
};
static_assert(sizeof(ItemBox) % 16 == 0, "item box keeps 16-byte alignment");

struct PipeBars {
  uint64_t item_full[2], item_empty[2];  // [box slot]
  uint64_t cu_ready[2];                  // [box slot] member offsets of groups staged
  uint64_t q_full[2], q_ready[2], q_empty[2];  // [X]
  uint64_t k_full[kKStages], k_ready[kKStages], k_empty[kKStages];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t s_full[2], p_ready[2], o_done[2];  // [X]
  uint64_t drain;
};

struct Meta {
  PipeBars bars[kPipes];
  ItemBox box[kPipes][2];
  uint32_t cu_st[kPipes][2][2][kCuStage];  // [pipe][box slot][X]
  uint32_t tmem;
  int32_t abort;
};

constexpr uint32_t kSmemUsed = kOffMeta + sizeof(Meta);
static_assert(kSmemUsed + 1024 <= 227u * 1024u, "fits the 227 KB a block may use");
constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t col_s(int c) { return 128u * c; }
__host__ __device__ constexpr uint32_t col_o(int c) { return 128u * c + 64u; }
// consumers of an item box: the issuer, the two rotation warps and the eight softmax warps
constexpr uint32_t kItemConsumers = 1 + 2 + 8;

__device__ __forceinline__ uint8_t* q_tile(uint8_t* smem, int chain) { return smem + kOffQ + kQBytes * chain; }
__device__ __forceinline__ uint8_t* k_tile(uint8_t* smem, int pipe, uint32_t st) {
  return smem + kOffK + kKVBytes * (pipe * kKStages + st);
}
__device__ __forceinline__ uint8_t* v_tile(uint8_t* smem, int pipe, uint32_t st) {
  return smem + kOffV + kKVBytes * (pipe * kVStages + st);
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
  float q_mul;  // multiplies the rotated q (the scale when it is not positive, else 1)
  float s_mul;  // multiplies the scores in the softmax (the scale when it is positive, else 1)
  unsigned long long timeout_ns;
  int skip_first_item_arrive;  // test hook: the producers withhold their first item hand-off
};

// ------------------------------------------------------------------------------------
// the key stream of an item
//
// Shared: tile t holds keys [a.k0 + 64 t, ...) for both query tiles. Alternating: with
// m = min(na, nb), tiles 0 .. 2m - 1 alternate A's and B's (A first), the rest belong to
// the query tile with more tiles. A query tile's i-th own tile holds keys
// [k0 + 64 i, min(k0 + nk, k0 + 64 i + 64)) of its record.

struct Stream {
  uint32_t na, nb, n, shared, has_b;
};
__device__ __forceinline__ Stream stream_of(const ItemBox& bx) {
  Stream s;
  s.na = bx.na;
  s.nb = bx.nb;
  s.n = bx.n;
  s.shared = bx.shared;
  s.has_b = bx.has_b;
  return s;
}
// owner of stream tile t: bit 0 A, bit 1 B; `ia` / `ib` the tile's index among its owners' own
__device__ __forceinline__ uint32_t owners(const Stream& s, uint32_t t, uint32_t& ia, uint32_t& ib) {
  ia = ib = t;
  if (s.shared) return 3u;
  if (!s.has_b) return 1u;
  const uint32_t m = min(s.na, s.nb);
  if (t < 2 * m) {
    ia = ib = t >> 1;
    return (t & 1u) ? 2u : 1u;
  }
  ia = ib = m + (t - 2 * m);
  return s.na > s.nb ? 1u : 2u;
}
// stream index of query tile X's last own tile
__device__ __forceinline__ uint32_t last_of(const Stream& s, int x) {
  if (s.shared || !s.has_b) return s.n - 1;
  const uint32_t nx = x == 0 ? s.na : s.nb;
  const uint32_t m = min(s.na, s.nb);
  return nx <= m ? 2 * (nx - 1) + static_cast<uint32_t>(x) : s.n - 1;
}

// ------------------------------------------------------------------------------------
// producer of pipe `pipe` (one thread): work items and TMA loads. Per item: K(0), K(1),
// Q_A, Q_B, then K(t) and V(t - 2) in turn.

__device__ __forceinline__ void producer(const CUtensorMap* tmap, const Params& p, uint8_t* smem, Meta* meta, int pipe,
                         unsigned int n_items) {
  PipeBars& B = meta->bars[pipe];
  const int32_t hd = p.H * kD;
  const unsigned int ntiles = __ldcg(&p.ctl->ntiles);
  uint32_t it = 0, qn[2] = {0u, 0u};
  uint32_t kn = 0, vn = 0;  // K and V tiles loaded so far
  bool bad = false;

  for (;;) {
    const unsigned int item = atomicAdd(&p.ctl->next, 1u);
    const uint32_t mb = it & 1u;
    if (!wait_bar(&meta->abort, p.ctl, &B.item_empty[mb], ((it >> 1) & 1u) ^ 1u, p.timeout_ns)) {
      bad = true;
      break;
    }
    ItemBox& bx = meta->box[pipe][mb];
    if (item >= n_items) {
      bx.valid = 0;
      mbar_arrive(smem_u32(&B.item_full[mb]));
      break;
    }
    const unsigned int pair = item / static_cast<unsigned int>(p.H);
    const int h = static_cast<int>(item % static_cast<unsigned int>(p.H));
    const TileRec ra = p.tiles[2 * pair];
    const bool has_b = 2 * pair + 1 < ntiles;
    TileRec rb = ra;
    if (has_b) rb = p.tiles[2 * pair + 1];
    const uint32_t ss_a = ra.kind == 0 ? __ldg(p.cu + ra.seq) : 0u;
    const uint32_t se_a = ra.kind == 0 ? __ldg(p.cu + ra.seq + 1) : 0u;
    const uint32_t ss_b = has_b && rb.kind == 0 ? __ldg(p.cu + rb.seq) : 0u;
    const uint32_t se_b = has_b && rb.kind == 0 ? __ldg(p.cu + rb.seq + 1) : 0u;
    const bool shared = has_b && ra.kind == 0 && rb.kind == 0 && ra.seq == rb.seq && ra.k0 == rb.k0 && ra.nk == rb.nk;
    const uint32_t na = (ra.nk + kKeys - 1) / kKeys;
    const uint32_t nb = has_b ? (rb.nk + kKeys - 1) / kKeys : 0u;
    bx.a = ra;
    bx.b = rb;
    bx.head = h;
    bx.valid = 1;
    bx.has_b = has_b;
    bx.shared = shared;
    bx.na = na;
    bx.nb = nb;
    bx.n = shared ? na : na + nb;
    bx.ss_a = ss_a;
    bx.se_a = se_a;
    bx.ss_b = ss_b;
    bx.se_b = se_b;
    // (the test hook leaves the consumers waiting: their bounded waits time out and the CTA
    // unwinds with PK_ERR_TIMEOUT)
    if (!(p.skip_first_item_arrive && it == 0)) mbar_arrive(smem_u32(&B.item_full[mb]));
    ++it;

    const Stream sm = stream_of(bx);
    auto load_k = [&](uint32_t t) -> bool {
      const uint32_t st = kn % kKStages;
      if (!wait_bar(&meta->abort, p.ctl, &B.k_empty[st], ((kn / kKStages) & 1u) ^ 1u, p.timeout_ns)) return false;
      uint32_t ia, ib;
      const uint32_t o = owners(sm, t, ia, ib);
      const uint32_t j0 = (o & 1u) ? ra.k0 + ia * kKeys : rb.k0 + ib * kKeys;
      mbar_arrive_expect_tx(smem_u32(&B.k_full[st]), kKVBytes);
      tma_load_2d(smem_u32(k_tile(smem, pipe, st)), tmap, smem_u32(&B.k_full[st]), hd + h * kD,
                  static_cast<int32_t>(j0));
      ++kn;
      return true;
    };
    auto load_v = [&](uint32_t t) -> bool {
      const uint32_t st = vn % kVStages;
      if (!wait_bar(&meta->abort, p.ctl, &B.v_empty[st], ((vn / kVStages) & 1u) ^ 1u, p.timeout_ns)) return false;
      uint32_t ia, ib;
      const uint32_t o = owners(sm, t, ia, ib);
      const uint32_t j0 = (o & 1u) ? ra.k0 + ia * kKeys : rb.k0 + ib * kKeys;
      mbar_arrive_expect_tx(smem_u32(&B.v_full[st]), kKVBytes);
      tma_load_2d(smem_u32(v_tile(smem, pipe, st)), tmap, smem_u32(&B.v_full[st]), 2 * hd + h * kD,
                  static_cast<int32_t>(j0));
      ++vn;
      return true;
    };
    // Q_X into its buffer once the previous item's last S_X has completed (two boxes of 64 rows)
    auto load_q = [&](int x, uint32_t q0) -> bool {
      const int c = 2 * pipe + x;
      if (!wait_bar(&meta->abort, p.ctl, &B.q_empty[x], (qn[x] & 1u) ^ 1u, p.timeout_ns)) return false;
      mbar_arrive_expect_tx(smem_u32(&B.q_full[x]), kQBytes);
      tma_load_2d(smem_u32(q_tile(smem, c)), tmap, smem_u32(&B.q_full[x]), h * kD, static_cast<int32_t>(q0));
      tma_load_2d(smem_u32(q_tile(smem, c) + kKVBytes), tmap, smem_u32(&B.q_full[x]), h * kD,
                  static_cast<int32_t>(q0 + 64));
      ++qn[x];
      return true;
    };
    const uint32_t n = sm.n;
    const uint32_t qs = min(2u, n);
    for (uint32_t t = 0; t < qs && !bad; ++t) bad = !load_k(t);
    if (!bad) bad = !load_q(0, ra.q0) || (has_b && !load_q(1, rb.q0));
    for (uint32_t t = qs; t < n + 2 && !bad; ++t) {
      if (t < n) bad = !load_k(t);
      if (!bad && t >= 2) bad = !load_v(t - 2);
    }
    if (bad) break;
  }
  if (bad || aborted(&meta->abort)) {
    // let the copies in flight land before the CTA's shared memory goes away
    for (int x = 0; x < 2; ++x)
      if (qn[x] > 0) mbar_wait(smem_u32(&B.q_full[x]), (qn[x] - 1) & 1u, p.timeout_ns);
    for (uint32_t t = kn > kKStages ? kn - kKStages : 0; t < kn; ++t)
      mbar_wait(smem_u32(&B.k_full[t % kKStages]), (t / kKStages) & 1u, p.timeout_ns);
    for (uint32_t t = vn > kVStages ? vn - kVStages : 0; t < vn; ++t)
      mbar_wait(smem_u32(&B.v_full[t % kVStages]), (t / kVStages) & 1u, p.timeout_ns);
  }
}

// ------------------------------------------------------------------------------------
// MMA issuer of pipe `pipe` (one thread) for its query tiles A and B. Per stream tile t,
// for each owner X of t: O_X += P_X V(t_prev) for X's previous tile t_prev (once P_X is
// written and V(t_prev) has landed), then S_X = Q_X K(t)^T (once K(t) is rotated and, on X's
// first tile, Q_X). A query tile whose own tiles have ended gets its last PV product at the
// next stream tile (so V tiles are released in step with the stream); the rest at the end
// of the item, each followed by a commit to o_done[X] for the epilogue. K(t) is released by
// a commit after the last S that reads it, V(t) after the last PV product that reads it.

// per query tile state of an issuer
struct IssChain {
  uint64_t dq;      // descriptor of its Q tile
  uint32_t pr, qn;  // p_ready phases seen, items whose Q it has used
  int32_t pend_t;   // stream tile of its pending PV product (-1: none)
  uint32_t pend_i, pend_n;  // that tile's index among the query tile's own, its key count
  uint32_t last;    // stream index of its last own tile in the current item
  uint32_t k0, kend;  // its record's key range
};

__device__ __forceinline__ void mma_issuer(const Params& p, uint8_t* smem, Meta* meta, uint32_t tmem, bool bf16, int pipe) {
  PipeBars& B = meta->bars[pipe];
  const uint32_t idesc_pv = idesc_f16(bf16, 128, 64, false, true);
  // operand descriptors: a K step of 16 adds 32 bytes (Q, K) or 2048 bytes (V) to the start
  // address (field units of 16 bytes); successive 8 KB K / V stages are 512 units apart
  const uint64_t dk0 = sdesc_sw128(smem_u32(k_tile(smem, pipe, 0)), 16, 1024);
  const uint64_t dv0 = sdesc_sw128(smem_u32(v_tile(smem, pipe, 0)), 8192, 1024);
  IssChain ca, cb;
  ca.dq = sdesc_sw128(smem_u32(q_tile(smem, 2 * pipe)), 16, 1024);
  cb.dq = sdesc_sw128(smem_u32(q_tile(smem, 2 * pipe + 1)), 16, 1024);
  ca.pr = cb.pr = ca.qn = cb.qn = 0u;
  uint32_t it = 0;
  uint32_t kn = 0, vbase = 0;  // K tiles consumed; V tiles of earlier items
  bool bad = false;

  // O_X += P_X V(s) for X's pending stream tile s; V(s) is released once its last reader has
  // been issued (`release`; in a shared stream B reads after A)
  auto pv = [&](int x, IssChain& c, bool release) -> bool {
    const uint32_t vq = vbase + static_cast<uint32_t>(c.pend_t);
    const uint32_t st = vq % kVStages;
    if (!wait_bar(&meta->abort, p.ctl, &B.v_full[st], (vq / kVStages) & 1u, p.timeout_ns)) return false;
    if (!wait_bar(&meta->abort, p.ctl, &B.p_ready[x], c.pr & 1u, p.timeout_ns)) return false;
    ++c.pr;
    tc_fence_after();
    const int cc = 2 * pipe + x;
    const uint32_t tO = tmem + col_o(cc), tP = tmem + col_s(cc);
    const uint32_t ksteps = round16(c.pend_n) / 16;
    const uint64_t dv = dv0 + st * (kKVBytes >> 4);
    umma_f16_ts(tO, tP, dv, idesc_pv, c.pend_i > 0 ? 1u : 0u);
#pragma unroll
    for (uint32_t ks = 1; ks < 4; ++ks)
      if (ks < ksteps) umma_f16_ts(tO, tP + ks * 8, dv + ks * 128, idesc_pv, 1u);
    if (release) umma_commit(smem_u32(&B.v_empty[st]));
    c.pend_t = -1;
    return true;
  };

  for (;;) {
    const uint32_t mb = it & 1u;
    if (!wait_bar(&meta->abort, p.ctl, &B.item_full[mb], (it >> 1) & 1u, p.timeout_ns)) break;
    const ItemBox& bx = meta->box[pipe][mb];
    const bool valid = bx.valid != 0;
    const Stream sm = stream_of(bx);
    ca.k0 = bx.a.k0;
    ca.kend = bx.a.k0 + bx.a.nk;
    cb.k0 = bx.b.k0;
    cb.kend = bx.b.k0 + bx.b.nk;
    mbar_arrive(smem_u32(&B.item_empty[mb]));
    ++it;
    if (!valid) break;
    ca.last = last_of(sm, 0);
    cb.last = sm.has_b ? last_of(sm, 1) : 0u;
    ca.pend_t = cb.pend_t = -1;
    // in a shared stream V(t) is released by B's product, A's leaves it
    const bool rel_a = !sm.shared || !sm.has_b;

    // stream tile t for query tile X (a constant after inlining): its pending PV product and
    // S = Q K(t)^T when X owns t, else the last PV product once X's own tiles have ended
    auto step = [&](int x, IssChain& c, uint32_t t, uint32_t own, uint32_t i, uint32_t kst, bool& k_seen) -> bool {
      if (own & (1u << x)) {
        if (c.pend_t >= 0 && !pv(x, c, x == 1 || rel_a)) return false;
        if (i == 0 && !wait_bar(&meta->abort, p.ctl, &B.q_ready[x], c.qn & 1u, p.timeout_ns)) return false;
        if (!k_seen && !wait_bar(&meta->abort, p.ctl, &B.k_ready[kst], (kn / kKStages) & 1u, p.timeout_ns))
          return false;
        k_seen = true;
        tc_fence_after();
        const uint32_t nkeys = min(static_cast<uint32_t>(kKeys), c.kend - (c.k0 + i * kKeys));
        const uint32_t idesc = idesc_f16(bf16, 128, round16(nkeys), false, false);
        const uint64_t dk = dk0 + kst * (kKVBytes >> 4);
        const uint32_t tS = tmem + col_s(2 * pipe + x);
        umma_f16_ss(tS, c.dq, dk, idesc, 0u);
#pragma unroll
        for (int ks = 1; ks < 4; ++ks) umma_f16_ss(tS, c.dq + ks * 2, dk + ks * 2, idesc, 1u);
        umma_commit(smem_u32(&B.s_full[x]));
        if (t == c.last) {
          umma_commit(smem_u32(&B.q_empty[x]));
          ++c.qn;
        }
        c.pend_t = static_cast<int32_t>(t);
        c.pend_i = i;
        c.pend_n = nkeys;
      } else if (c.pend_t >= 0 && c.last < t) {
        // X's own tiles have ended: its last PV product now, then the epilogue may read O
        if (!pv(x, c, true)) return false;
        umma_commit(smem_u32(&B.o_done[x]));
      }
      return true;
    };

#pragma unroll 1
    for (uint32_t t = 0; t < sm.n; ++t) {
      uint32_t ia, ib;
      const uint32_t own = owners(sm, t, ia, ib);
      const uint32_t kst = kn % kKStages;
      bool k_seen = false;
      if (!step(0, ca, t, own, ia, kst, k_seen) || !step(1, cb, t, own, ib, kst, k_seen)) {
        bad = true;
        break;
      }
      // K(t) is released after the S products that read it
      if (k_seen)
        umma_commit(smem_u32(&B.k_empty[kst]));
      else
        mbar_arrive(smem_u32(&B.k_empty[kst]));
      ++kn;
    }
    if (bad) break;
    // the last PV products of the item, each followed by the epilogue's signal
    if (ca.pend_t >= 0) {
      if (!pv(0, ca, rel_a)) break;
      umma_commit(smem_u32(&B.o_done[0]));
    }
    if (cb.pend_t >= 0) {
      if (!pv(1, cb, true)) break;
      umma_commit(smem_u32(&B.o_done[1]));
    }
    vbase += sm.n;
  }
  // every MMA this thread issued has completed before the CTA frees tensor memory
  umma_commit(smem_u32(&B.drain));
  mbar_wait(smem_u32(&B.drain), 0, p.timeout_ns);
}

// ------------------------------------------------------------------------------------
// rotation of pipe `pipe` (64 threads; thread t rotates row t of every K tile and rows t,
// t + 64 of every Q tile of the pipe)
//
// Per item: K(0), K(1), then Q_A's two halves, Q_B's, then the other K tiles, each as soon
// as it lands (the producer's load order). A row's position is its token minus the start of
// its sequence: one subtraction for a piece of a sequence, a search in the staged member
// offsets for a group of short sequences (whose key rows are its query rows). The table
// rows of the next job are in flight (cp.async) while the current one is rotated. Rows past
// a tile's tokens are left as loaded; their scores are masked.

template <bool BF16>
__device__ __forceinline__ void rotator(const Params& p, uint8_t* smem, Meta* meta, int pipe, int t) {
  PipeBars& B = meta->bars[pipe];
  const int lane = t & 31;
  const int tt = pipe * 64 + t;  // table buffer index
  const uint32_t tbl0 = smem_u32(smem + kOffTbl + tt * 2 * kRowTblBytes);
  const uint8_t* tblp = smem + kOffTbl + tt * 2 * kRowTblBytes;
  uint32_t it = 0, qn[2] = {0u, 0u};
  uint32_t kn = 0;  // K tiles rotated so far
  uint32_t buf = 0;
  bool bad = false;
  for (;;) {
    const uint32_t mb = it & 1u;
    bad |= !wait_bar(&meta->abort, p.ctl, &B.item_full[mb], (it >> 1) & 1u, p.timeout_ns);
    bad = __any_sync(0xffffffffu, bad);
    if (bad) break;
    const ItemBox& bx = meta->box[pipe][mb];
    const bool valid = bx.valid != 0, has_b = bx.has_b != 0;
    if (!valid) {
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&B.item_empty[mb]));
      break;
    }
    const TileRec ra = bx.a, rb = bx.b;
    const Stream sm = stream_of(bx);
    const uint32_t ss_a = bx.ss_a, ss_b = bx.ss_b;
    // stage the member offsets of groups (the softmax warps read them too)
    uint32_t* off_a = meta->cu_st[pipe][mb][0];
    uint32_t* off_b = meta->cu_st[pipe][mb][1];
    if (ra.kind != 0) stage_cu(p.cu, ra, off_a, t, 64);
    if (has_b && rb.kind != 0) stage_cu(p.cu, rb, off_b, t, 64);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&B.cu_ready[mb]));
    bad |= !wait_bar(&meta->abort, p.ctl, &B.cu_ready[mb], (it >> 1) & 1u, p.timeout_ns);
    ++it;
    bad = __any_sync(0xffffffffu, bad);
    if (bad) break;

    // positions of rows t and t + 64 of Q_A and Q_B (for a group also of its key rows)
    uint32_t qpos[2][2] = {{0u, 0u}, {0u, 0u}};
    bool qok[2][2] = {{false, false}, {false, false}};
    for (int x = 0; x < 2; ++x) {
      if (x == 1 && !has_b) break;
      const TileRec& rec = x == 0 ? ra : rb;
      for (int hh = 0; hh < 2; ++hh) {
        const uint32_t r = static_cast<uint32_t>(t + 64 * hh);
        qok[x][hh] = r < rec.rows;
        if (!qok[x][hh]) continue;
        const uint32_t a = rec.q0 + r;
        uint32_t ss;
        if (rec.kind == 0) {
          ss = x == 0 ? ss_a : ss_b;
        } else {
          uint32_t se;
          group_bounds(p.cu, rec, x == 0 ? off_a : off_b, a, ss, se);
        }
        qpos[x][hh] = a - ss;
      }
    }
    // row t of stream tile s: its owner's i-th own tile holds keys from k0 + 64 i; a piece's
    // position is the token minus the sequence start, a group's that of its query row
    auto krow = [&](uint32_t s, uint32_t& pos) -> bool {
      uint32_t ia, ib;
      const uint32_t o = owners(sm, s, ia, ib);
      const int x = (o & 1u) ? 0 : 1;
      const TileRec& rec = x == 0 ? ra : rb;
      const uint32_t i = x == 0 ? ia : ib;
      const uint32_t j0 = rec.k0 + i * kKeys;
      const bool ok = static_cast<uint32_t>(t) < rec.k0 + rec.nk - j0;
      if (!ok) {
        pos = 0u;
        return false;
      }
      pos = rec.kind != 0 ? qpos[x][i & 1u] : j0 + static_cast<uint32_t>(t) - (x == 0 ? ss_a : ss_b);
      return true;
    };

    // jobs: K(0 .. qs - 1), then Q_A rows t / t + 64, Q_B rows t / t + 64, then K(qs ..)
    const uint32_t qs = min(2u, sm.n);
    const uint32_t nq = has_b ? 4u : 2u;
    const uint32_t njobs = nq + sm.n;
    auto job = [&](uint32_t i, bool& isq, int& x, int& hh, uint32_t& s) {
      isq = i >= qs && i < qs + nq;
      if (isq) {
        x = static_cast<int>((i - qs) >> 1);
        hh = static_cast<int>((i - qs) & 1u);
        s = 0;
      } else {
        x = 0;
        hh = 0;
        s = i < qs ? i : i - nq;
      }
    };
    auto job_pos = [&](uint32_t i, uint32_t& pos) -> bool {
      bool isq;
      int x, hh;
      uint32_t s;
      job(i, isq, x, hh, s);
      if (isq) {
        pos = qpos[x][hh];
        return qok[x][hh];
      }
      return krow(s, pos);
    };
    {
      uint32_t pos0;
      if (job_pos(0, pos0)) fetch_table_row(p.cos_t, p.sin_t, tbl0 + buf * kRowTblBytes, pos0, tt);
      cp_async_commit();
    }
#pragma unroll 1
    for (uint32_t i = 0; i < njobs; ++i) {
      bool isq;
      int x, hh;
      uint32_t s;
      job(i, isq, x, hh, s);
      uint32_t pos_i;
      const bool ok = job_pos(i, pos_i);
      uint8_t* tile;
      uint64_t* full;
      uint32_t phase;
      int row;
      if (isq) {
        tile = q_tile(smem, 2 * pipe + x);
        full = &B.q_full[x];
        phase = qn[x] & 1u;
        row = t + 64 * hh;
      } else {
        const uint32_t kst = kn % kKStages;
        tile = k_tile(smem, pipe, kst);
        full = &B.k_full[kst];
        phase = (kn / kKStages) & 1u;
        row = t;
      }
      // the next job's table rows into the other buffer
      if (i + 1 < njobs) {
        uint32_t pos_n;
        if (job_pos(i + 1, pos_n)) fetch_table_row(p.cos_t, p.sin_t, tbl0 + (buf ^ 1u) * kRowTblBytes, pos_n, tt);
      }
      cp_async_commit();
      cp_async_wait1();  // this job's rows have landed (the next one's may still be in flight)
      bad |= !wait_bar(&meta->abort, p.ctl, full, phase, p.timeout_ns);
      bad = __any_sync(0xffffffffu, bad);
      if (bad) break;
      if (ok) rope_row<BF16>(tile, row, tblp + buf * kRowTblBytes, tt, isq ? p.q_mul : 1.0f);
      fence_proxy_async_smem();
      __syncwarp();
      if (isq) {
        if (hh == 1) {
          if (lane == 0) mbar_arrive(smem_u32(&B.q_ready[x]));
          ++qn[x];
        }
      } else {
        if (lane == 0) mbar_arrive(smem_u32(&B.k_ready[kn % kKStages]));
        ++kn;
      }
      buf ^= 1u;
    }
    cp_async_wait0();
    if (bad) break;
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&B.item_empty[mb]));
  }
  cp_async_wait0();
  if (bad && lane == 0) raise_abort(&meta->abort, p.ctl);
}

// ------------------------------------------------------------------------------------
// softmax warpgroup of query tile X of pipe `pipe` (128 threads; thread <-> query row <->
// TMEM lane). Each warp signals the MMA issuer on its own (barriers of count 4), so warps
// never wait for one another; a failed wait is voted across the warp before any
// warp-collective TMEM access, so a warp leaves together.

template <bool BF16>
__device__ __forceinline__ void softmax_wg(const Params& p, Meta* meta, int pipe, int x, uint32_t tmem) {
  PipeBars& B = meta->bars[pipe];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int r = (warp & 3) * 32 + lane;
  const int c = 2 * pipe + x;
  const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t tS = tmem + lane_addr + col_s(c);
  const uint32_t tP = tS;
  const uint32_t tO = tmem + lane_addr + col_o(c);
  const int64_t hd = static_cast<int64_t>(p.H) * kD;
  // raw scores s weigh ex2(s k2 - m k2): k2 folds the score scale into the base change
  const float k2 = p.s_mul * kLog2e;

  uint32_t it = 0, sf = 0, od = 0;
  bool bad = false;
  for (;;) {
    const uint32_t mb = it & 1u;
    bad |= !wait_bar(&meta->abort, p.ctl, &B.item_full[mb], (it >> 1) & 1u, p.timeout_ns);
    bad = __any_sync(0xffffffffu, bad);
    if (bad) break;
    const ItemBox& bx = meta->box[pipe][mb];
    const bool valid = bx.valid != 0;
    const bool mine = valid && (x == 0 || bx.has_b);
    const TileRec rec = x == 0 ? bx.a : bx.b;
    const int h = bx.head;
    const uint32_t nx = x == 0 ? bx.na : bx.nb;
    const uint32_t ss_p = x == 0 ? bx.ss_a : bx.ss_b, se_p = x == 0 ? bx.se_a : bx.se_b;
    const uint32_t* off = meta->cu_st[pipe][mb][x];
    ++it;
    if (!mine) {
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&B.item_empty[mb]));
      if (!valid) break;
      continue;
    }
    // a group's member offsets are staged by the rotation warps
    if (rec.kind != 0) bad |= !wait_bar(&meta->abort, p.ctl, &B.cu_ready[mb], ((it - 1) >> 1) & 1u, p.timeout_ns);
    bad = __any_sync(0xffffffffu, bad);
    if (bad) break;

    // this thread's query row and its visible key interval [lo, hi) (tokens < 2^31)
    const bool row_ok = r < static_cast<int>(rec.rows);
    const int a = static_cast<int>(rec.q0) + r;
    int lo = 0, hi = 0;
    if (row_ok) {
      uint32_t ss = ss_p, se = se_p;
      if (rec.kind != 0) group_bounds(p.cu, rec, off, static_cast<uint32_t>(a), ss, se);
      lo = static_cast<int>(ss);
      hi = static_cast<int>(se);
      if (p.window > 0) {
        lo = max(lo, a - p.window);
        hi = static_cast<int>(min(static_cast<int64_t>(hi), static_cast<int64_t>(a) + p.window + 1));
      }
    }

    float m_ref = kNeg, l = 0.f;  // running max of the raw scores, and the row sum
#pragma unroll 1
    for (uint32_t i = 0; i < nx; ++i) {
      const int j0 = static_cast<int>(rec.k0 + i * kKeys);
      const int nkeys = min(kKeys, static_cast<int>(rec.k0 + rec.nk) - j0);

      // this row of S (columns past the tile's keys hold stale values; they are masked)
      bad |= !wait_bar(&meta->abort, p.ctl, &B.s_full[x], sf & 1u, p.timeout_ns);
      ++sf;
      bad = __any_sync(0xffffffffu, bad);
      if (bad) break;
      tc_fence_after();

      // visible columns [c_lo, c_hi); every other column weighs zero
      const int c_lo = min(max(lo - j0, 0), kKeys);
      const int c_hi = min(max(hi - j0, 0), nkeys);
      const bool full = __all_sync(0xffffffffu, c_lo == 0 && c_hi == kKeys);

      // Two passes over the row in halves of 32 columns, each reading its half from tensor
      // memory (the whole kernel is compiled within 80 registers a thread). Pass 1: the max.
      float mx = m_ref;
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        float v[32];
        tmem_ld32(tS + 32 * hh, v);
        if (!full) {
#pragma unroll
          for (int cc = 0; cc < 32; ++cc)
            if (static_cast<unsigned>(cc + 32 * hh - c_lo) >= static_cast<unsigned>(c_hi - c_lo)) v[cc] = -INFINITY;
        }
        float m0 = fmax3(v[0], v[1], v[2]), m1 = fmax3(v[3], v[4], v[5]), m2 = fmax3(v[6], v[7], v[8]),
              m3 = fmax3(v[9], v[10], v[11]);
#pragma unroll
        for (int cc = 12; cc < 28; cc += 8) {
          m0 = fmax3(m0, v[cc], v[cc + 1]);
          m1 = fmax3(m1, v[cc + 2], v[cc + 3]);
          m2 = fmax3(m2, v[cc + 4], v[cc + 5]);
          m3 = fmax3(m3, v[cc + 6], v[cc + 7]);
        }
        mx = fmax3(mx, fmax3(m0, m1, v[28]), fmax3(fmax3(m2, m3, v[29]), v[30], v[31]));
      }
      const bool grow = (mx - m_ref) * k2 > kRescale;
      float alpha = 1.f;
      if (grow) {
        alpha = ex2((m_ref - mx) * k2);
        l *= alpha;
        m_ref = mx;
      }
      const float mb2 = m_ref * k2;
      const float2 c2 = make_float2(k2, k2);
      const float2 nm2 = make_float2(-mb2, -mb2);
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
      // Pass 2: the probabilities of each half, written over the first 32 columns of S (16-bit
      // pairs; half hh's P goes to columns 16 hh .. 16 hh + 15, which this thread has read).
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        float v[32];
        tmem_ld32(tS + 32 * hh, v);
        if (!full) {
#pragma unroll
          for (int cc = 0; cc < 32; ++cc)
            if (static_cast<unsigned>(cc + 32 * hh - c_lo) >= static_cast<unsigned>(c_hi - c_lo)) v[cc] = -INFINITY;
        }
        uint32_t pp[16];
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) {
          const float2 xx = __ffma2_rn(make_float2(v[2 * cc], v[2 * cc + 1]), c2, nm2);
          const float2 e = make_float2(ex2(xx.x), ex2(xx.y));
          if (cc & 1)
            acc1 = __fadd2_rn(acc1, e);
          else
            acc0 = __fadd2_rn(acc0, e);
          pp[cc] = Elem<BF16>::pack(e.x, e.y);
        }
        tmem_st16(tP + 16 * hh, pp);
      }
      const float2 accs = __fadd2_rn(acc0, acc1);
      l += accs.x + accs.y;
      // O holds the PV products of the earlier tiles (all complete: this tile's S was issued
      // after them); rescale it when the max grew
      if (i > 0 && __any_sync(0xffffffffu, grow)) {
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
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&B.p_ready[x]));
    }
    if (bad) break;

    // epilogue: out = O / l, lse = m + ln l
    bad |= !wait_bar(&meta->abort, p.ctl, &B.o_done[x], od & 1u, p.timeout_ns);
    ++od;
    bad = __any_sync(0xffffffffu, bad);
    if (bad) break;
    tc_fence_after();
    const float inv = 1.0f / l;
#pragma unroll 1
    for (int oh = 0; oh < 2; ++oh) {
      float ov[32];
      tmem_ld32(tO + 32 * oh, ov);
      if (row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(a) * hd + h * kD + 32 * oh));
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[q] = make_uint4(Elem<BF16>::pack(ov[8 * q + 0] * inv, ov[8 * q + 1] * inv),
                              Elem<BF16>::pack(ov[8 * q + 2] * inv, ov[8 * q + 3] * inv),
                              Elem<BF16>::pack(ov[8 * q + 4] * inv, ov[8 * q + 5] * inv),
                              Elem<BF16>::pack(ov[8 * q + 6] * inv, ov[8 * q + 7] * inv));
      }
    }
    tc_fence_before();
    // the item box (and the staged offsets in its slot) may be reused
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&B.item_empty[mb]));
    if (row_ok) p.lse[static_cast<int64_t>(h) * p.T + a] = (m_ref * k2 + lg2(l)) * kLn2;
  }
  if (bad && lane == 0) raise_abort(&meta->abort, p.ctl);
}

}  // namespace

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
pk_attend_q4_kernel(const __grid_constant__ CUtensorMap tmap_qkv, const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Meta* meta = reinterpret_cast<Meta*>(smem + kOffMeta);
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    tma_prefetch_desc(&tmap_qkv);
    for (int pp = 0; pp < kPipes; ++pp) {
      PipeBars& B = meta->bars[pp];
      for (int i = 0; i < 2; ++i) {
        mbar_init(smem_u32(&B.item_full[i]), 1);
        mbar_init(smem_u32(&B.item_empty[i]), kItemConsumers);
        mbar_init(smem_u32(&B.cu_ready[i]), 2);
        mbar_init(smem_u32(&B.q_full[i]), 1);
        mbar_init(smem_u32(&B.q_ready[i]), 2);
        mbar_init(smem_u32(&B.q_empty[i]), 1);
        mbar_init(smem_u32(&B.s_full[i]), 1);
        mbar_init(smem_u32(&B.p_ready[i]), 4);
        mbar_init(smem_u32(&B.o_done[i]), 1);
      }
      for (int i = 0; i < kKStages; ++i) {
        mbar_init(smem_u32(&B.k_full[i]), 1);
        mbar_init(smem_u32(&B.k_ready[i]), 2);
        mbar_init(smem_u32(&B.k_empty[i]), 1);
      }
      for (int i = 0; i < kVStages; ++i) {
        mbar_init(smem_u32(&B.v_full[i]), 1);
        mbar_init(smem_u32(&B.v_empty[i]), 1);
      }
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

  // Every role runs at the launch's 80 registers a thread (768 x 80 = 61440): ptxas compiles
  // the whole kernel within that count, so a warpgroup gains nothing from raising its share,
  // and the producer / issuer and rotation code spill when theirs is lowered.
  if (warp < kWarpRot) {
    if (warp < kWarpMma) {
      if (lane == 0) {
        // the records and the work counter come from the scheduler launched just before
        griddep_wait();
        producer(&tmap_qkv, p, smem, meta, warp - kWarpProd,
                 (__ldcg(&p.ctl->ntiles) + 1u) / 2u * static_cast<unsigned int>(p.H));
      }
    } else {
      if (lane == 0) mma_issuer(p, smem, meta, meta->tmem, BF16, warp - kWarpMma);
    }
  } else if (warp < kWarpSm) {
    const int rt = tid - kWarpRot * 32;
    rotator<BF16>(p, smem, meta, rt >> 6, rt & 63);
  } else {
    const int c = (warp - kWarpSm) >> 2;
    softmax_wg<BF16>(p, meta, c >> 1, c & 1, meta->tmem);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(meta->tmem, kTmemCols);
  }
}

uint32_t attend_q4_smem_bytes() { return kSmemUsed + 1024; }

// Host side: opt in to the dynamic shared memory once per device.
cudaError_t attend_q4_prepare() {
  const int smem = static_cast<int>(attend_q4_smem_bytes());
  cudaError_t e = cudaFuncSetAttribute(pk_attend_q4_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pk_attend_q4_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pk_attend_q4_kernel<true>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pk_attend_q4_kernel<false>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  return e;
}

// Host side: one launch of `grid` persistent CTAs (one per SM). `tmap` views qkv as
// {3 H 64, T} 16-bit elements with a {64, 64} box and 128-byte swizzle.
cudaError_t attend_q4_launch(bool bf16, const CUtensorMap& tmap, const void* cos_t, const void* sin_t,
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
  p.q_mul = scale > 0.0f ? 1.0f : scale;
  p.s_mul = scale > 0.0f ? scale : 1.0f;
  p.timeout_ns = timeout_ns;
  {
    const char* e = std::getenv("PK_DEBUG_SKIP_ARRIVE");
    p.skip_first_item_arrive = (e && e[0] == '1') ? 1 : 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = attend_q4_smem_bytes();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (bf16) return cudaLaunchKernelEx(&cfg, pk_attend_q4_kernel<true>, tmap, p);
  return cudaLaunchKernelEx(&cfg, pk_attend_q4_kernel<false>, tmap, p);
}

}  // namespace pk
