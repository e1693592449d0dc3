// pk_attend_split.cu -- packed RoPE attention forward for fp32 inputs on tcgen05 (sm_103a),
// with every operand split into two bf16 values.
//
// What it computes: hanzo-kernel 0.2.42 packed.rs fn attend for fp32 storage -- a tile of
// query rows of one head against every key tile its window reaches, the softmax online per
// row with masked keys weighing exactly zero, then out = O / l and lse = m + ln l, all in
// fp32 to within the pages' fp32 tolerance.
//
// How: the matrix units take 16-bit operands at most 2^-9 apart from fp32 values. A pre-pass
// (pk_split16_kernel) rotates q and k in fp32 and writes every value x of q', k' and v as
// hi = bf16(x) and lo = bf16(x - hi): hi + lo holds 16 significant bits of x. Each product
// is then taken as three bf16 products accumulated in fp32 (the lo x lo term, a further
// 2^-8 smaller, is left out):
//     S = Qh Kh^T + Qh Kl^T + Ql Kh^T,   O += Ph Vh + Ph Vl + Pl Vh
// with the probabilities split the same way (Ph = bf16(p), Pl = bf16(p - Ph)). The sum
// of a row is taken from the fp32 probabilities.
//
// Layout (GB300): one persistent 352-thread CTA per SM. A work item is a PAIR of
// consecutive tile records (A, B) of one head; when both are pieces of one sequence they
// share one key stream (every K / V tile pair is loaded once for both query tiles), else
// B's key tiles follow A's. Shared memory: Q_A, Q_B as hi / lo tiles, a 2-stage K ring and
// a 2-stage V ring of hi / lo tile pairs (192 KB). Tensor memory (384 of 512 columns):
//     SP_A, SP_B [128 x 128]  the scores of the current key tile (fp32); the probabilities
//                             are written over them: keys 0-63 as Ph in columns 0-31 and
//                             Pl in 32-63, keys 64-127 as Ph in 64-95 and Pl in 96-127
//     O_A, O_B   [128 x  64]  output accumulators (fp32)
// Since P lives over S, a query tile's next S product is issued after its PV product, by
// the same thread: the tensor pipe runs one thread's MMAs in order, so the PV product has
// read P before the next S overwrites it, and once an S product has completed, every
// earlier PV product of that tile has too. The two query tiles of an item keep the pipe
// busy while either one's softmax runs.
// Warps (each warp's TMEM lane quarter is its index mod 4):
//   warp 0: producer (one lane): claims items, TMA-loads Q_A, Q_B and the stream's K and V
//           tile pairs (128-byte swizzle, straight from the split copy);
//   warps 1, 10: MMA issuers of A, B (one lane each): per stream tile t, PV_X(t - 1) once
//           V(t - 1) and P_X(t - 1) are there, then S_X(t) once K(t) is there;
//   warps 2-5, 6-9: softmax of A, B: thread r owns query row r. It reads its S row twice
//           by halves of 64 columns (the row max, then the probabilities), masks it by the
//           row's visible key interval, keeps a running max (O is rescaled only when the max
//           grows by more than 2^8), writes Ph and Pl over each half's own scores, and at
//           the end of the item writes out = O / l and lse = m + ln l.
// Every wait is bounded. A wait that times out records PK_ERR_TIMEOUT and raises the CTA's
// abort flag, which every other wait watches; the producer then waits (bounded) for its
// copies in flight, the MMA issuers for their MMAs, and the CTA frees its tensor memory.
#include <cstdlib>

#include "pk_attn_common.cuh"

namespace pk {

namespace {

using namespace attn;

constexpr int kThreads = 352;  // 11 warps: 184 registers a thread
constexpr int kStages = 2;     // K ring and V ring depth (each stage holds a hi and a lo tile)
constexpr int kWarpProd = 0;
constexpr int kWarpMmaA = 1;
constexpr int kWarpSm = 2;      // warps 2..5 (A), 6..9 (B): four consecutive warps cover the lane quarters
constexpr int kWarpMmaB = 10;

constexpr uint32_t kTileBytes = 128 * 128;  // 128 rows x 64 bf16
// shared-memory map (offsets from the 1024-aligned base); every tile starts on 1024 bytes
constexpr uint32_t kOffQ = 0;                               // [X][hi / lo]
constexpr uint32_t kOffK = kOffQ + 4 * kTileBytes;          // [stage][hi / lo]
constexpr uint32_t kOffV = kOffK + 2 * kStages * kTileBytes;  // [stage][hi / lo]
constexpr uint32_t kOffMeta = kOffV + 2 * kStages * kTileBytes;

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
  uint32_t pad[7];
};
static_assert(sizeof(ItemBox) % 16 == 0, "item box keeps 16-byte alignment");

struct Bars {
  uint64_t item_full[2], item_empty[2];
  uint64_t q_full[2], q_empty[2];  // [X]
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t v_full[kStages], v_empty[kStages];
  uint64_t s_full[2], p_ready[2], o_done[2];  // [X]
  uint64_t cu_sm[2][2];                      // [X][item parity]
  uint64_t drain[2];
};

struct Meta {
  Bars bars;
  ItemBox box[2];
  uint32_t cu_sm[2][2][kCuStage];  // [X][item parity]
  uint32_t tmem;
  int32_t abort;
};

constexpr uint32_t kSmemUsed = kOffMeta + sizeof(Meta);
static_assert(kSmemUsed + 1024 <= 227u * 1024u, "fits the 227 KB a block may use");
constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t col_sp(int x) { return 128u * x; }
__host__ __device__ constexpr uint32_t col_o(int x) { return 256u + 64u * x; }
constexpr uint32_t kItemConsumers = 2 + 4 + 4;  // MMA issuers, softmax A, B warps
// tensor-memory column (from SP_X) of the Ph values of keys [16 ks, 16 ks + 16)
__host__ __device__ constexpr uint32_t ph_col(uint32_t ks) { return 8u * ks + (ks >= 4 ? 32u : 0u); }

__device__ __forceinline__ uint8_t* q_tile(uint8_t* smem, int x, int lo) { return smem + kOffQ + kTileBytes * (2 * x + lo); }
__device__ __forceinline__ uint8_t* k_tile(uint8_t* smem, uint32_t st, int lo) {
  return smem + kOffK + kTileBytes * (2 * st + lo);
}
__device__ __forceinline__ uint8_t* v_tile(uint8_t* smem, uint32_t st, int lo) {
  return smem + kOffV + kTileBytes * (2 * st + lo);
}

struct Params {
  const uint32_t* cu;
  const TileRec* tiles;
  float* out;
  float* lse;
  Ctl* ctl;
  int H;
  long long T;
  int window;
  float s_mul;  // multiplies the scores in the softmax (the scale when it is positive, else 1)
  unsigned long long timeout_ns;
  int skip_first_item_arrive;  // test hook: the producer withholds its first item hand-off
};

// Stream tile j of an item: its first key token and its key count.
__device__ __forceinline__ void stream_tile(const ItemBox& bx, uint32_t j, uint32_t& j0, uint32_t& nkeys) {
  if (bx.shared) {
    j0 = bx.a.k0 + j * kBC;
    nkeys = min(static_cast<uint32_t>(kBC), bx.end - j0);
  } else if (j < bx.a1) {
    j0 = bx.a.k0 + j * kBC;
    nkeys = min(static_cast<uint32_t>(kBC), bx.a.nk - j * kBC);
  } else {
    j0 = bx.b.k0 + (j - bx.a1) * kBC;
    nkeys = min(static_cast<uint32_t>(kBC), bx.b.nk - (j - bx.a1) * kBC);
  }
}

// ------------------------------------------------------------------------------------
// producer (one thread): per item Q_A, Q_B (hi and lo), then K(0), V(0), K(1), V(1), ...
// (the split copy's row: hi q | hi k | hi v | lo q | lo k | lo v, each H x 64 columns)

__device__ void producer(const CUtensorMap* tmap, const Params& p, uint8_t* smem, Meta* meta, unsigned int n_items) {
  Bars& B = meta->bars;
  const int32_t hd = p.H * kD;
  const int32_t lo_off = 3 * hd;  // column of the lo copy
  const unsigned int ntiles = __ldcg(&p.ctl->ntiles);
  uint32_t it = 0, qn[2] = {0u, 0u}, kn = 0, vn = 0;
  bool bad = false;
  int32_t* flag = &meta->abort;

  for (;;) {
    const unsigned int item = atomicAdd(&p.ctl->next, 1u);
    const uint32_t mb = it & 1u;
    if (!wait_bar(flag, p.ctl, &B.item_empty[mb], ((it >> 1) & 1u) ^ 1u, p.timeout_ns)) {
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
    const TileRec ra = p.tiles[2 * pair];
    const bool has_b = 2 * pair + 1 < ntiles;
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
    if (!(p.skip_first_item_arrive && it == 0)) mbar_arrive(smem_u32(&B.item_full[mb]));
    ++it;

    // Q_X (hi and lo) once the previous item's last S_X has read the old ones
    for (int x = 0; x < (has_b ? 2 : 1) && !bad; ++x) {
      const uint32_t q0 = x == 0 ? ra.q0 : rb.q0;
      if (!wait_bar(flag, p.ctl, &B.q_empty[x], (qn[x] & 1u) ^ 1u, p.timeout_ns)) {
        bad = true;
        break;
      }
      const uint32_t bar = smem_u32(&B.q_full[x]);
      mbar_arrive_expect_tx(bar, 2 * kTileBytes);
      tma_load_2d(smem_u32(q_tile(smem, x, 0)), tmap, bar, h * kD, static_cast<int32_t>(q0));
      tma_load_2d(smem_u32(q_tile(smem, x, 1)), tmap, bar, lo_off + h * kD, static_cast<int32_t>(q0));
      ++qn[x];
    }
    if (bad) break;
    // the stream: K(t), then V(t)
    for (uint32_t t = 0; t < nstream && !bad; ++t) {
      uint32_t j0, nk;
      stream_tile(bx, t, j0, nk);
      {
        const uint32_t st = kn % kStages;
        if (!wait_bar(flag, p.ctl, &B.k_empty[st], ((kn / kStages) & 1u) ^ 1u, p.timeout_ns)) {
          bad = true;
          break;
        }
        const uint32_t bar = smem_u32(&B.k_full[st]);
        mbar_arrive_expect_tx(bar, 2 * kTileBytes);
        tma_load_2d(smem_u32(k_tile(smem, st, 0)), tmap, bar, hd + h * kD, static_cast<int32_t>(j0));
        tma_load_2d(smem_u32(k_tile(smem, st, 1)), tmap, bar, lo_off + hd + h * kD, static_cast<int32_t>(j0));
        ++kn;
      }
      {
        const uint32_t st = vn % kStages;
        if (!wait_bar(flag, p.ctl, &B.v_empty[st], ((vn / kStages) & 1u) ^ 1u, p.timeout_ns)) {
          bad = true;
          break;
        }
        const uint32_t bar = smem_u32(&B.v_full[st]);
        mbar_arrive_expect_tx(bar, 2 * kTileBytes);
        tma_load_2d(smem_u32(v_tile(smem, st, 0)), tmap, bar, 2 * hd + h * kD, static_cast<int32_t>(j0));
        tma_load_2d(smem_u32(v_tile(smem, st, 1)), tmap, bar, lo_off + 2 * hd + h * kD, static_cast<int32_t>(j0));
        ++vn;
      }
    }
    if (bad) break;
  }
  if (bad || aborted(flag)) {
    // let the copies in flight land before the CTA's shared memory goes away
    for (int x = 0; x < 2; ++x)
      if (qn[x] > 0) mbar_wait(smem_u32(&B.q_full[x]), (qn[x] - 1) & 1u, p.timeout_ns);
    for (uint32_t t = kn > kStages ? kn - kStages : 0; t < kn; ++t)
      mbar_wait(smem_u32(&B.k_full[t % kStages]), (t / kStages) & 1u, p.timeout_ns);
    for (uint32_t t = vn > kStages ? vn - kStages : 0; t < vn; ++t)
      mbar_wait(smem_u32(&B.v_full[t % kStages]), (t / kStages) & 1u, p.timeout_ns);
  }
}

// ------------------------------------------------------------------------------------
// MMA issuer of query tile X (one thread). Per stream tile t: PV_X(t - 1) if X's range holds
// t - 1 (once V(t - 1) has landed and P_X(t - 1) is written), then S_X(t) if X's range holds
// t (once K(t) has landed, and Q_X for X's first tile). K and V ring stages are released by
// both issuers (barriers of count 2): by a commit after the MMAs that read them, or by a
// plain arrival for a tile outside X's range, made only after the tile's own full phase was
// seen. The MMA sequences are fixed (S 128 keys wide, PV over all 128 keys of a tile: the
// columns past a tile's keys are masked scores and zero probabilities).

__device__ void mma_issuer(const Params& p, uint8_t* smem, Meta* meta, uint32_t tmem, int x) {
  Bars& B = meta->bars;
  int32_t* flag = &meta->abort;
  const uint32_t idesc_s = idesc_f16(true, 128, 128, false, false);
  const uint32_t idesc_pv = idesc_f16(true, 128, 64, false, true);
  // K step of 16: +32 bytes (Q, K; start address field is address >> 4) or +2048 bytes (V)
  const uint64_t dqh = sdesc_sw128(smem_u32(q_tile(smem, x, 0)), 16, 1024);
  const uint64_t dql = sdesc_sw128(smem_u32(q_tile(smem, x, 1)), 16, 1024);
  const uint64_t dk0 = sdesc_sw128(smem_u32(k_tile(smem, 0, 0)), 16, 1024);  // + 1024 per tile
  const uint64_t dv0 = sdesc_sw128(smem_u32(v_tile(smem, 0, 0)), 8192, 1024);
  const uint32_t tS = tmem + col_sp(x), tO = tmem + col_o(x);
  uint32_t it = 0, pr = 0, qn = 0, kst = 0, kph = 0, vst = 0, vph = 0;
  bool bad = false;

  for (;;) {
    const uint32_t mb = it & 1u;
    if (!wait_bar(flag, p.ctl, &B.item_full[mb], (it >> 1) & 1u, p.timeout_ns)) break;
    const bool valid = meta->box[mb].valid != 0;
    const uint32_t n = meta->box[mb].nstream;
    const uint32_t lo = x == 0 ? 0u : meta->box[mb].b0, hi = x == 0 ? meta->box[mb].a1 : meta->box[mb].b1;
    mbar_arrive(smem_u32(&B.item_empty[mb]));
    ++it;
    if (!valid) break;
    for (uint32_t t = 0; t <= n && !bad; ++t) {
      if (t >= 1) {
        const uint32_t j = t - 1;
        if (!wait_bar(flag, p.ctl, &B.v_full[vst], vph, p.timeout_ns)) {
          bad = true;
          break;
        }
        if (j >= lo && j < hi) {
          if (!wait_bar(flag, p.ctl, &B.p_ready[x], pr & 1u, p.timeout_ns)) {
            bad = true;
            break;
          }
          ++pr;
          tc_fence_after();
          const uint64_t dvh = dv0 + (2 * vst) * 1024, dvl = dvh + 1024;
          // Ph of keys [16 ks, 16 ks + 16) sits at column 8 ks (+ 32 past the first 64 keys), Pl 32 further
          umma_f16_ts(tO, tS, dvh, idesc_pv, j > lo ? 1u : 0u);
#pragma unroll
          for (uint32_t ks = 1; ks < 8; ++ks) umma_f16_ts(tO, tS + ph_col(ks), dvh + ks * 128, idesc_pv, 1u);
#pragma unroll
          for (uint32_t ks = 0; ks < 8; ++ks) umma_f16_ts(tO, tS + ph_col(ks), dvl + ks * 128, idesc_pv, 1u);
#pragma unroll
          for (uint32_t ks = 0; ks < 8; ++ks) umma_f16_ts(tO, tS + ph_col(ks) + 32, dvh + ks * 128, idesc_pv, 1u);
          umma_commit(smem_u32(&B.v_empty[vst]));
          if (j + 1 == hi) umma_commit(smem_u32(&B.o_done[x]));
        } else {
          mbar_arrive(smem_u32(&B.v_empty[vst]));
        }
        vst = (vst + 1) & (kStages - 1);
        vph ^= vst == 0 ? 1u : 0u;
      }
      if (t < n) {
        if (!wait_bar(flag, p.ctl, &B.k_full[kst], kph, p.timeout_ns)) {
          bad = true;
          break;
        }
        if (t >= lo && t < hi) {
          if (t == lo && !wait_bar(flag, p.ctl, &B.q_full[x], qn & 1u, p.timeout_ns)) {
            bad = true;
            break;
          }
          tc_fence_after();
          const uint64_t dkh = dk0 + (2 * kst) * 1024, dkl = dkh + 1024;
          umma_f16_ss(tS, dqh, dkh, idesc_s, 0u);
#pragma unroll
          for (int ks = 1; ks < 4; ++ks) umma_f16_ss(tS, dqh + ks * 2, dkh + ks * 2, idesc_s, 1u);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) umma_f16_ss(tS, dqh + ks * 2, dkl + ks * 2, idesc_s, 1u);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) umma_f16_ss(tS, dql + ks * 2, dkh + ks * 2, idesc_s, 1u);
          umma_commit(smem_u32(&B.s_full[x]));
          umma_commit(smem_u32(&B.k_empty[kst]));
          if (t + 1 == hi) {
            umma_commit(smem_u32(&B.q_empty[x]));
            ++qn;
          }
        } else {
          mbar_arrive(smem_u32(&B.k_empty[kst]));
        }
        kst = (kst + 1) & (kStages - 1);
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
// softmax warpgroup of query tile X (128 threads; thread <-> query row <-> TMEM lane)

__device__ void softmax_wg(const Params& p, Meta* meta, int x, uint32_t tmem) {
  Bars& B = meta->bars;
  int32_t* flag = &meta->abort;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int r = (warp & 3) * 32 + lane;
  const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t tS = tmem + lane_addr + col_sp(x);
  const uint32_t tO = tmem + lane_addr + col_o(x);
  const int64_t hd = static_cast<int64_t>(p.H) * kD;
  // raw scores s weigh ex2(s k2 - m k2): k2 folds the score scale into the base change
  const float k2 = p.s_mul * kLog2e;

  uint32_t it = 0, sf = 0, used = 0;
  bool bad = false;
  for (;;) {
    const uint32_t mb = it & 1u;
    bad |= !wait_bar(flag, p.ctl, &B.item_full[mb], (it >> 1) & 1u, p.timeout_ns);
    bad = __any_sync(0xffffffffu, bad);
    if (bad) break;
    const ItemBox& bx = meta->box[mb];
    const bool valid = bx.valid != 0;
    const bool mine = valid && (x == 0 || bx.has_b);
    const TileRec rec = x == 0 ? bx.a : bx.b;
    const int h = bx.head;
    const uint32_t jlo = x == 0 ? 0u : bx.b0, jhi = x == 0 ? bx.a1 : bx.b1;
    // this query tile's stream tiles [jlo, jhi): tile j holds keys [j0, j0 + nkeys) with
    // j0 = kbase + 128 (j - jlo) and nkeys = min(128, kend - j0) (kept in registers: the
    // producer may refill this item box while the item's last tiles are still in work)
    const uint32_t kbase = (x == 0 || bx.shared) ? bx.a.k0 + jlo * kBC : bx.b.k0;
    const uint32_t kend = bx.shared ? bx.end : rec.k0 + rec.nk;
    uint32_t* off = meta->cu_sm[x][used & 1u];
    if (mine) stage_cu(p.cu, rec, off, r, 128);
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(smem_u32(&B.item_empty[mb]));
      if (mine) mbar_arrive(smem_u32(&B.cu_sm[x][used & 1u]));
    }
    ++it;
    if (!valid) break;
    if (!mine) continue;
    bad |= !wait_bar(flag, p.ctl, &B.cu_sm[x][used & 1u], (used >> 1) & 1u, p.timeout_ns);
    bad = __any_sync(0xffffffffu, bad);
    if (bad) break;

    // this thread's query row and its visible key interval [lo, hi) (tokens < 2^31)
    const bool row_ok = r < static_cast<int>(rec.rows);
    const int a = static_cast<int>(rec.q0) + r;
    int lo = 0, hi = 0;
    if (row_ok) {
      uint32_t ss, se;
      if (rec.kind == 0) {
        ss = off[0];
        se = off[1];
      } else {
        group_bounds(p.cu, rec, off, static_cast<uint32_t>(a), ss, se);
      }
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

      bad |= !wait_bar(flag, p.ctl, &B.s_full[x], sf & 1u, p.timeout_ns);
      ++sf;
      bad = __any_sync(0xffffffffu, bad);
      if (bad) break;
      tc_fence_after();

      // visible columns [c_lo, c_hi); every other column weighs zero
      const int c_lo = min(max(lo - j0, 0), 128);
      const int c_hi = min(max(hi - j0, 0), nkeys);
      const bool full = __all_sync(0xffffffffu, c_lo == 0 && c_hi == 128);

      // pass 1: the row max, by halves of 64 columns (once S_X(j) has completed, so has
      // PV_X(j - 1): O is final for the rescale below)
      float mx = -INFINITY;
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        float v[64];
        tmem_ld64(tS + 64 * hh, v);
        if (!full) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (static_cast<unsigned>(c + 64 * hh - c_lo) >= static_cast<unsigned>(c_hi - c_lo)) v[c] = -INFINITY;
        }
        float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; c += 8) {
          m0 = fmax3(m0, v[c], v[c + 1]);
          m1 = fmax3(m1, v[c + 2], v[c + 3]);
          m2 = fmax3(m2, v[c + 4], v[c + 5]);
          m3 = fmax3(m3, v[c + 6], v[c + 7]);
        }
        mx = fmax3(mx, fmaxf(m0, m1), fmaxf(m2, m3));
      }
      const float m_new = fmaxf(m_ref, mx);
      const bool grow = (m_new - m_ref) * k2 > kRescale;
      float alpha = 1.f;
      if (grow) {
        alpha = ex2((m_ref - m_new) * k2);
        l *= alpha;
        m_ref = m_new;
      }
      if (j > jlo && __any_sync(0xffffffffu, grow)) {
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
      const float mb2 = m_ref * k2;
      const float2 c2 = make_float2(k2, k2);
      const float2 nm2 = make_float2(-mb2, -mb2);
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
      // pass 2: probabilities in fp32, split into Ph and Pl written over the half's own
      // scores: keys [64 hh, 64 hh + 64) give Ph in columns 64 hh + [0, 32) and Pl in
      // 64 hh + [32, 64)
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        float v[64];
        tmem_ld64(tS + 64 * hh, v);
        if (!full) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (static_cast<unsigned>(c + 64 * hh - c_lo) >= static_cast<unsigned>(c_hi - c_lo)) v[c] = -INFINITY;
        }
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {
          uint32_t ph[16], pl[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float2 xx = __ffma2_rn(make_float2(v[32 * qq + 2 * c], v[32 * qq + 2 * c + 1]), c2, nm2);
            const float2 e = make_float2(ex2(xx.x), ex2(xx.y));
            if (c & 1)
              acc1 = __fadd2_rn(acc1, e);
            else
              acc0 = __fadd2_rn(acc0, e);
            ph[c] = Elem<true>::pack(e.x, e.y);
            const float2 eh = Elem<true>::unpack(ph[c]);
            pl[c] = Elem<true>::pack(e.x - eh.x, e.y - eh.y);
          }
          tmem_st16(tS + 64 * hh + 16 * qq, ph);
          tmem_st16(tS + 64 * hh + 32 + 16 * qq, pl);
        }
      }
      const float2 accs = __fadd2_rn(acc0, acc1);
      l += accs.x + accs.y;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&B.p_ready[x]));
    }
    if (bad) break;

    // epilogue: out = O / l, lse = m + ln l (once the item's last PV_X has completed)
    bad |= !wait_bar(flag, p.ctl, &B.o_done[x], used & 1u, p.timeout_ns);
    ++used;
    bad = __any_sync(0xffffffffu, bad);
    if (bad) break;
    tc_fence_after();
    float ov[64];
    tmem_ld64(tO, ov);
    tc_fence_before();
    if (row_ok) {
      const float inv = 1.0f / l;
      float4* dst = reinterpret_cast<float4*>(p.out + (static_cast<int64_t>(a) * hd + h * kD));
#pragma unroll
      for (int q = 0; q < 16; ++q)
        dst[q] = make_float4(ov[4 * q + 0] * inv, ov[4 * q + 1] * inv, ov[4 * q + 2] * inv, ov[4 * q + 3] * inv);
      p.lse[static_cast<int64_t>(h) * p.T + a] = (m_ref * k2 + lg2(l)) * kLn2;
    }
  }
  if (bad && lane == 0) raise_abort(flag, p.ctl);
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
pk_attend_split_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Meta* meta = reinterpret_cast<Meta*>(smem + kOffMeta);
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    tma_prefetch_desc(&tmap);
    Bars& B = meta->bars;
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&B.item_full[i]), 1);
      mbar_init(smem_u32(&B.item_empty[i]), kItemConsumers);
      mbar_init(smem_u32(&B.q_full[i]), 1);
      mbar_init(smem_u32(&B.q_empty[i]), 1);
      mbar_init(smem_u32(&B.s_full[i]), 1);
      mbar_init(smem_u32(&B.p_ready[i]), 4);
      mbar_init(smem_u32(&B.o_done[i]), 1);
      mbar_init(smem_u32(&B.cu_sm[i][0]), 4);
      mbar_init(smem_u32(&B.cu_sm[i][1]), 4);
      mbar_init(smem_u32(&B.drain[i]), 1);
    }
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&B.k_full[i]), 1);
      mbar_init(smem_u32(&B.k_empty[i]), 2);
      mbar_init(smem_u32(&B.v_full[i]), 1);
      mbar_init(smem_u32(&B.v_empty[i]), 2);
    }
    meta->abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMmaA) {
    tmem_alloc(smem_u32(&meta->tmem), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == kWarpProd) {
    if (lane == 0) {
      // the records, the work counter and the split copy come from the kernels launched before
      griddep_wait();
      const unsigned int nt = __ldcg(&p.ctl->ntiles);
      producer(&tmap, p, smem, meta, (nt + 1u) / 2u * static_cast<unsigned int>(p.H));
    }
  } else if (warp == kWarpMmaA || warp == kWarpMmaB) {
    if (lane == 0) mma_issuer(p, smem, meta, meta->tmem, warp == kWarpMmaA ? 0 : 1);
  } else {
    softmax_wg(p, meta, (warp - kWarpSm) >> 2, meta->tmem);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMmaA) {
    tc_fence_after();
    tmem_dealloc(meta->tmem, kTmemCols);
  }
}

uint32_t attend_split_smem_bytes() { return kSmemUsed + 1024; }

cudaError_t attend_split_prepare() {
  const int smem = static_cast<int>(attend_split_smem_bytes());
  cudaError_t e = cudaFuncSetAttribute(pk_attend_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pk_attend_split_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  return e;
}

// Host side: one launch of `grid` persistent CTAs (one per SM). `tmap` views the split copy
// as {6 H 64, T} bf16 values with a {64, 128} box and 128-byte swizzle.
cudaError_t attend_split_launch(const CUtensorMap& tmap, const uint32_t* cu, const TileRec* tiles, float* out,
                                float* lse, Ctl* ctl, int H, long long T, int window, float scale,
                                unsigned long long timeout_ns, int grid, cudaStream_t stream) {
  Params p;
  p.cu = cu;
  p.tiles = tiles;
  p.out = out;
  p.lse = lse;
  p.ctl = ctl;
  p.H = H;
  p.T = T;
  p.window = window;
  // a positive scale multiplies the scores here; any other scale multiplied q in the pre-pass
  p.s_mul = scale > 0.0f ? scale : 1.0f;
  p.timeout_ns = timeout_ns;
  {
    const char* e = std::getenv("PK_DEBUG_SKIP_ARRIVE");
    p.skip_first_item_arrive = (e && e[0] == '1') ? 1 : 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = attend_split_smem_bytes();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pk_attend_split_kernel, tmap, p);
}

}  // namespace pk
