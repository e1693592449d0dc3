// pk_dev.cuh -- device helpers of the packed RoPE attention library for sm_103a:
// inline PTX for mbarriers, TMA tiles, tcgen05 MMAs and tensor-memory access, the tile
// record and the per-stream control block shared by the scheduler and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pk {

constexpr int kD = 64;         // head dimension
constexpr int kHalf = 32;      // rotary pairs (u, u + 32)
constexpr int kBR = 128;       // query rows per tile (one tcgen05 M=128 tile)
constexpr int kBC = 128;       // keys per key tile
constexpr int kShort = 64;     // sequences of at most this length are grouped
constexpr int kWin = 1024;     // grouping window in tokens (groups never cross one)
// schedule capacity: pieces <= T/64 (a long sequence has at least 65 tokens), groups <=
// T/64 plus one per run of short sequences (two consecutive groups of a run hold more than
// 128 rows), runs <= long sequences + windows: at most 3 records per kCapUnit tokens, plus one
constexpr int kCapUnit = 64;
// Records whose first query token falls in one window: records of at least 65 rows start
// 65 apart (16), last pieces of at most 64 rows (the sequence holding the window's first
// token, plus one per long sequence starting in it: 17), groups of at most 64 rows closed by
// an overflow (each followed by a larger group: at most 16) or by a long sequence or the
// window's end (17): 66 at most. The scheduler's single walk writes a warp's records to
// slots of this many per window, then copies them into place.
constexpr int kWinCap = 72;
constexpr int kSchedWarps = 32;  // warps of each scheduler block
constexpr int kSchedCtas = 4;    // blocks of the scheduler's cluster when one block has too few warps
// blocks of the scheduler's one cluster for T tokens: one while a block has a warp per window
__host__ __device__ constexpr int schedule_ctas(long long T) {
  return (T + kWin - 1) / kWin <= kSchedWarps ? 1 : kSchedCtas;
}
// staging slots (records) the scheduler needs for T tokens
__host__ __device__ constexpr long long schedule_stage_records(long long T) {
  return ((T + kWin - 1) / kWin + kSchedWarps * schedule_ctas(T) - 1) / (kSchedWarps * schedule_ctas(T)) *
         (kSchedWarps * schedule_ctas(T)) * kWinCap;
}
constexpr int kRec = 8;        // uint32 per tile record

// Tile record, written by the scheduler (8 x uint32, 32 bytes).
struct TileRec {
  uint32_t q0, rows;   // query tokens [q0, q0 + rows)
  uint32_t k0, nk;     // key tokens [k0, k0 + nk)
  uint32_t seq, nseq;  // member sequences [seq, seq + nseq)
  uint32_t kind;       // 0: a piece of one sequence; 1: a group of short sequences
  uint32_t ktiles;     // ceil(nk / kBC)
};
static_assert(sizeof(TileRec) == 32, "tile record is 32 bytes");

// Per-stream control block: work counter, tile count, sticky status.
struct Ctl {
  unsigned int next;     // next work item (tile x head), reset by the scheduler
  unsigned int ntiles;   // records written by the scheduler
  int status;            // first device-detected error (0 = none); cleared by the host
  unsigned int pad[5];
};
static_assert(sizeof(Ctl) == 32, "control block is 32 bytes");

// The forward kernels (host-side dispatch: select_forward_kernel, forward_launch in pk_host.cu).
constexpr int kKernelBand = 0;  // narrow windows, CUDA cores, fp32
constexpr int kKernelF32 = 1;   // fp32 inputs, CUDA cores
constexpr int kKernelTc = 2;    // 16-bit inputs, paired-stream tensor-core kernel
constexpr int kKernelQ4 = 3;    // 16-bit inputs, four-chain tensor-core kernel
constexpr int kKernelTcSingle = 4;  // 16-bit inputs, paired-stream kernel with one record per item
constexpr int kKernelSplit = 5;     // fp32 inputs, tensor cores on split bf16 operands (needs a scratch copy)
int select_forward_kernel(int dtype, int window);
// bytes of the split copy kKernelSplit reads (T x 6 H 64 bf16 values)
inline long long split_copy_bytes(long long T, int H) { return T * 6 * H * kD * 2; }
// The launches of one forward call on caller-provided scratch (control block, `cap` tile
// records, the scheduler's staging slots, and for kKernelSplit the split copy `copy` of
// `copy_bytes` bytes); `ev`, when not null, gets three events recorded (before the first
// launch, between the preparation and the attention kernel, after it). Returns a pk_status code.
int forward_launch(int kernel, int dtype, int out_dtype, const void* qkv, const void* cos, const void* sin,
                   const uint32_t* cu, int S, long long T, int H, int window, float scale, void* out, float* lse,
                   Ctl* ctl, TileRec* tiles, long long cap, TileRec* stage, void* copy, long long copy_bytes, int sms,
                   unsigned long long timeout_ns, cudaStream_t stream, cudaEvent_t* ev);

// status codes (mirror enum pk_status)
constexpr int kErrBadCu = 5;
constexpr int kErrTimeout = 6;
constexpr int kErrInternal = 8;

__device__ __forceinline__ void set_status(Ctl* ctl, int code) { atomicCAS(&ctl->status, 0, code); }

// ------------------------------------------------------------------------------------
// time and addresses

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch: a kernel launched with programmatic stream serialization
// may start while the previous kernel of the stream runs; griddep_wait blocks until that
// kernel has completed and its memory operations are visible (a no-op without a
// dependency). griddep_launch_dependents lets the next kernel start early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------------------------
// mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, letting the thread sleep up to `hint_ns` while the phase is incomplete
// (it resumes as soon as the phase completes).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Bounded wait for phase `parity` of `bar`. Returns false when `timeout_ns` passes first.
// A caller that already gave up (`give_up`) does not wait at all.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                          bool give_up = false) {
  if (give_up) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0u && globaltimer_ns() - t0 > timeout_ns) return false;
  }
}

// ------------------------------------------------------------------------------------
// TMA (tensor tiles, global -> shared)

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tile load: box at (x = innermost element index, y = row), completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// ------------------------------------------------------------------------------------
// tcgen05: tensor memory, MMA, fences

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// generic-proxy writes to shared memory made visible to the async proxy (MMA, TMA)
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T  (kind::f16: bf16 or fp16 operands, fp32 accumulation)
__device__ __forceinline__ void umma_f16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// arrive on `bar` once every MMA this thread issued before has completed
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Instruction descriptor, kind::f16 with fp32 accumulation:
// bits 4-5 D format (1 = f32), 7-9 A format and 10-12 B format (0 = f16, 1 = bf16),
// 15 / 16 A / B major (0 = K-major, 1 = MN-major), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, uint32_t M, uint32_t N, bool a_mn,
                                                 bool b_mn) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) | ((N >> 3) << 17) |
         ((M >> 4) << 24);
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand whose tile starts on
// a 1024-byte boundary: bits 0-13 address >> 4, 16-29 leading byte offset >> 4,
// 32-45 stride byte offset >> 4, 46-47 version 1, 61-63 layout (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// D[tmem] (+)= A[tmem] * B[smem]  (A read from tensor memory: M lanes, K packed 2 per column)
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 consecutive 32-bit columns of this thread's TMEM lane <- r (waits for the store)
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0],"
      " {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16,"
      " %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// 16 consecutive 32-bit columns of this thread's TMEM lane <- r
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0],"
      " {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane, waited for before returning.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32"
      " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
      " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31},"
      " [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive fp32 columns of this thread's TMEM lane, waited for before returning.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32"
      " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 64 consecutive fp32 columns of this thread's TMEM lane, one load and one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// ------------------------------------------------------------------------------------
// 16-bit element helpers

template <bool BF16>
struct Elem;

// fp32 products of 16-bit operands without unpacking: lo/hi half of a packed pair times
// the matching half of another pair, accumulated in fp32 (fma.rn.f32.bf16 / .f16).
#define PK_MIXED_FMA(TY)                                                                          \
  __device__ static __forceinline__ float fma_lo(uint32_t a, uint32_t b, float c) {               \
    float d;                                                                                      \
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"      \
        "fma.rn.f32." TY " %0, al, bl, %3;\n\t}"                                                    \
        : "=f"(d)                                                                                 \
        : "r"(a), "r"(b), "f"(c));                                                                \
    return d;                                                                                     \
  }                                                                                               \
  __device__ static __forceinline__ float fma_hi(uint32_t a, uint32_t b, float c) {               \
    float d;                                                                                      \
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"      \
        "fma.rn.f32." TY " %0, ah, bh, %3;\n\t}"                                                    \
        : "=f"(d)                                                                                 \
        : "r"(a), "r"(b), "f"(c));                                                                \
    return d;                                                                                     \
  }

template <>
struct Elem<true> {
  PK_MIXED_FMA("bf16")
  __device__ static __forceinline__ float2 unpack(uint32_t u) {
    // low half is the element at the lower address
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
  }
  __device__ static __forceinline__ uint32_t pack(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
  }
};

template <>
struct Elem<false> {
  PK_MIXED_FMA("f16")
  __device__ static __forceinline__ float2 unpack(uint32_t u) {
    float lo, hi;
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(u));
    return make_float2(lo, hi);
  }
  __device__ static __forceinline__ uint32_t pack(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
  }
};

// ------------------------------------------------------------------------------------
// sequences

// The sequence holding token a among [s_lo, s_lo + n): the largest s with cu[s] <= a,
// stepping over empty sequences. Requires cu[s_lo] <= a < cu[s_lo + n].
__device__ __forceinline__ uint32_t seq_of_token(const uint32_t* __restrict__ cu, uint32_t s_lo,
                                                 uint32_t n, uint32_t a) {
  uint32_t lo = s_lo, hi = s_lo + n;  // answer in [lo, hi)
  while (hi - lo > 1) {
    const uint32_t mid = (lo + hi) >> 1;
    if (__ldg(cu + mid) <= a) lo = mid; else hi = mid;
  }
  return lo;
}

}  // namespace pk
