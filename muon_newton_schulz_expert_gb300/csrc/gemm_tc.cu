// Tensor-core GEMMs of one Newton-Schulz iteration on sm_103a.
//
// Source: "Training a 1T-Parameter MoE on EU public infrastructure with
// PyTorch and TorchTitan", section "FlexShard: Muon without communication":
// Newton-Schulz iterations on whole expert matrices, each matrix owned by one
// rank.  With X m x n (m <= n) one iteration is
//   A  = X X^T            (symmetric m x m: upper triangle computed, mirrored)
//   B  = b A + c A A      (A symmetric, so A A = A A^T: same kernel shape)
//   X' = a X + B X        (full m x n)
// The first iteration also applies the Frobenius factor s = 1/(||X||_F+eps):
// A gets s^2, X' gets s (so X0 = s X is never stored).
//
// Storage formats.  The caller's X (and the first iteration's input u) is
// bf16.  What the iteration produces is stored in 16 bits: in bf16 for
// matrices of more than 256 rows, and for smaller ones as fp16 scaled by a
// power of two, sigma * value, with sigma chosen on the host from a bound on
// the matrix's spectral norm (every entry of a matrix is at most its spectral
// norm) so that the largest possible entry sits near 2^14, well inside fp16's
// range: A, and B and X's high half from the second iteration on (the first
// iteration's B meets the bf16 u in one product, and tcgen05.mma of kind::f16
// takes both operands in one format).  fp16 keeps 11 significant bits against
// bf16's 8, so each rounding is 8x smaller; the scaling keeps fp16's narrow
// exponent range away from overflow and moves its subnormal floor ~2^-28
// below the largest entry.  The powers of two fold into the epilogues'
// existing constants, exactly.
// X is carried between iterations as a pair of halves, hi (bf16(X) or
// fp16(sigma X)) and lo, the remainder X - hi in 8 bits (e5m2 times a power
// of two S chosen from the same bound): the tensor cores read hi only, while
// the a X term of the epilogue uses hi + lo.  Rounding X itself to 16 bits
// would inject noise into every singular direction each iteration, and the
// quintic multiplies small singular values by up to a = 3.4445 per step, so
// on rank-deficient or ill-conditioned inputs that noise grows to percent
// level in the output (10% with bf16, 1-2% with fp16).  The remainder is at
// most hi's rounding unit, so its 8 bits leave about 2^-11 of |X| per entry;
// the last iteration's input, whose rounding passes through one step only,
// carries no lo.
//
// Design: persistent CTA pairs (clusters of 2), one CTA per SM, 320 threads,
// warp-specialised.  A pair computes a 256 x 256 output tile with
// tcgen05.mma.cta_group::2 (M=256, N=256, K=16, bf16 in, fp32 accumulate):
// each CTA holds 128 rows of A and a 128-row half of B in its own shared
// memory, and each CTA's TMEM receives its 128 rows of the accumulator.  Per
// SM this moves half the B bytes of a single-CTA 128 x 256 tile through
// shared memory, which is what keeps its bandwidth below the tensor cores'
// appetite.
//   warp 0 lane 0  TMA producer (both CTAs): 128x64 bf16 boxes, 128-byte
//                  swizzle, a ring of stages of two k-blocks (Layout); each
//                  k-block completes on its own "full" barrier in the even
//                  CTA, which counts the bytes of both halves;
//   warp 1         TMEM allocation of 512 columns (two 128 x 256 fp32
//                  accumulators) in both CTAs; lane 0 of the even CTA issues
//                  the MMAs and multicasts tcgen05.commit to both CTAs;
//   warps 2..9     epilogue (both CTAs): warp w reads TMEM lanes
//                  32*(w%4)..+31 and one 128-column half of the tile, and
//                  moves 32 x 32 boxes through shared memory with TMA.
// The double-buffered accumulator lets the epilogue of tile t overlap the
// main loop of tile t+1.  Every mbarrier wait is bounded: when it runs out the
// kernel records a timeout in the device error word, raises a shared abort
// flag so the other roles stop, lets in-flight copies land, frees its TMEM and
// returns.  No TMA multicast is used: each CTA loads its own tiles (a pair's
// rate does not depend on how many pairs run, so L2 reads are not the limit).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <mutex>

#include "common.cuh"

namespace muon {
namespace {

constexpr int CM = 256;    // rows of a pair tile
constexpr int BM = 128;    // rows of a pair tile held by one CTA
constexpr int BN = 256;    // columns of a pair tile
constexpr int BNH = 128;   // rows of the B operand held by one CTA
constexpr int BK = 64;     // one 128-byte swizzle row of bf16
constexpr int UMMA_K = 16;
// Operand ring and epilogue staging share the CTA's shared memory.
//  - A stage holds KSUB k-blocks of 64 (32 KB per k-block: 128 rows of A and
//    a 128-row half of B) behind one empty barrier and one full barrier per
//    k-block.  Each refill (MMA commit -> producer wait -> TMA issue) has a
//    fixed cost, so every kernel runs three stages of two k-blocks (8 MMAs per
//    refill); the MMAs of a stage's first k-block start as soon as its own
//    bytes land.  Measured against one full barrier per double stage, aX + BX
//    ran 1.5% faster; against six single stages in the same bytes (which cost
//    a refill per k-block), the update-fused aX + BX 5.6% faster (five single
//    stages before), aX + BX 3%, bA + cAA 1% and X X^T 1.1%.
//  - Each TMA round trip takes ~2000-2500 SM cycles under load, so the ring
//    must hold ~160-192 KB in flight to cover it.
//  - Epilogue slots, one per epilogue warp.  X X^T: output staging (direct
//    and mirror boxes).  bA + cAA: b*A in, result over it.  aX + BX: a 2 KB
//    box of X's high half and 1 KB of its 8-bit low half, the result written
//    over them, so 3 double stages fit.  aX + BX with the update: 2 KB boxes
//    of X's high half and W, W' written over them.
// aX + BX with the update: epilogue chunk width, 32 columns (2 KB boxes), or
// 16 (1 KB boxes)
#ifndef MUON_APPLY_CW
#define MUON_APPLY_CW 32
#endif
#ifndef MUON_AXPY_ROW_ORDER_T
#define MUON_AXPY_ROW_ORDER_T 1
#endif
#ifndef MUON_KSUB_SYRK
#define MUON_KSUB_SYRK 2
#endif
#ifndef MUON_KSUB_POLY
#define MUON_KSUB_POLY 2
#endif
#ifndef MUON_KSUB_AXPY
#define MUON_KSUB_AXPY 2
#endif
#ifndef MUON_KSUB_APPLY
#define MUON_KSUB_APPLY 2
#endif
#ifndef MUON_STAGES_SYRK
#define MUON_STAGES_SYRK 3
#endif
#ifndef MUON_SLOTS_SYRK
#define MUON_SLOTS_SYRK 1
#endif
#ifndef MUON_STAGES_POLY
#define MUON_STAGES_POLY 3
#endif
#ifndef MUON_SLOTS_POLY
#define MUON_SLOTS_POLY 1
#endif
#ifndef MUON_STAGES_AXPY
#define MUON_STAGES_AXPY 3
#endif
#ifndef MUON_SLOTS_AXPY
#define MUON_SLOTS_AXPY 1
#endif
#ifndef MUON_STAGES_APPLY
#define MUON_STAGES_APPLY 3
#endif
#ifndef MUON_SLOTS_APPLY
#define MUON_SLOTS_APPLY 1
#endif
constexpr int A_STAGE = BM * BK * 2;   // 16 KB
constexpr int B_STAGE = BNH * BK * 2;  // 16 KB
constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
// AXPY epilogue staging: per epilogue warp one 32 x 32 bf16 box of X's high
// half and one of its low half (64-byte swizzle), moved by TMA.
constexpr int EPI_BOX = 32;
constexpr int EPI_BOX_BYTES = EPI_BOX * EPI_BOX * 2;
constexpr int EPI_BUF = 2 * EPI_BOX_BYTES;   // one slot: two boxes
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * EPI_WARPS;  // producer warp, MMA warp, 8 epilogue warps
constexpr int ACC_COLS = BN;
constexpr int TMEM_COLS = 2 * ACC_COLS;
constexpr int CHUNKS = BN / 2 / 32;  // 32-column chunks per epilogue thread and tile

// EPI_APPLY is the last iteration's AXPY with the parameter update fused in:
// it reads the parameter W instead of writing X's halves, and writes
// W' = kw W + ko bf16(X') in place.
enum Epi { EPI_SYRK = 0, EPI_POLY = 1, EPI_AXPY = 2, EPI_APPLY = 3 };

template <int EPI>
struct Layout {
  static constexpr int stages = EPI == EPI_APPLY  ? MUON_STAGES_APPLY
                                : EPI == EPI_AXPY ? MUON_STAGES_AXPY
                                : EPI == EPI_POLY ? MUON_STAGES_POLY
                                                  : MUON_STAGES_SYRK;
  static constexpr int slots = EPI == EPI_APPLY  ? MUON_SLOTS_APPLY
                               : EPI == EPI_AXPY ? MUON_SLOTS_AXPY
                               : EPI == EPI_POLY ? MUON_SLOTS_POLY
                                                 : MUON_SLOTS_SYRK;
  // Bytes of one slot per epilogue warp.  SYRK/POLY: [direct box][mirror box].
  // AXPY: [X hi][X lo] (lo one byte per element), the result [X' hi][X' lo]
  // written over it; APPLY: [X hi][W] of cw-column boxes, W' written over it.
  // epilogue chunk width in columns (boxes of 32 rows x cw)
  static constexpr int cw = EPI == EPI_APPLY ? MUON_APPLY_CW : 32;
  static_assert(cw == 32 || cw == 16, "epilogue chunks of 32 or 16 columns");
  static constexpr int box_bytes = 32 * cw * 2;
  static constexpr int lo_bytes = 32 * cw;
  static constexpr int in_bytes = EPI == EPI_APPLY ? 2 * box_bytes : EPI == EPI_AXPY ? box_bytes + lo_bytes : EPI_BUF;
  static_assert(EPI >= EPI_AXPY || in_bytes == EPI_BUF, "the symmetric epilogues address slots of EPI_BUF bytes");
  static_assert(in_bytes % 1024 == 0, "slots keep the boxes' swizzle alignment");
  static constexpr int epi_bytes = EPI_WARPS * slots * in_bytes;
  // k-blocks of 64 per stage (one barrier round trip per ksub k-blocks)
  static constexpr int ksub = EPI == EPI_APPLY  ? MUON_KSUB_APPLY
                              : EPI == EPI_AXPY ? MUON_KSUB_AXPY
                              : EPI == EPI_POLY ? MUON_KSUB_POLY
                                                : MUON_KSUB_SYRK;
  static constexpr int stage_bytes = ksub * STAGE_BYTES;
  // a full barrier per k-block of each stage, an empty one per stage, two
  // accumulator pairs, the drain barrier and one per epilogue slot
  static constexpr int num_bars = stages * ksub + stages + 5 + EPI_WARPS * slots;
  static constexpr int smem_bytes = stages * stage_bytes + epi_bytes + 1024 + num_bars * 8 + 16;
  static_assert((128 / cw) % slots == 0, "chunks per tile must fill the staging slots evenly");
  static_assert(smem_bytes <= 232448, "shared memory per CTA");
};

struct Params {
  // epilogue maps, 32 x 32 boxes.  AXPY: X high half, X low half, X' high,
  // X' low.  SYRK/POLY: A (POLY's operand), the output, and the output again
  // without swizzle for the transposed (mirror) boxes.
  CUtensorMap tm_src, tm_src_lo, tm_out, tm_out_lo, tm_out_t;
  int M, N, K;                 // output M x N, reduction length K (per matrix)
  int tiles_m, tiles_n;        // pair tiles of 256 x 256
  int tiles_per_mat;
  int row_order;               // aX + BX: tiles ordered along rows (1) or down columns (0)
  long long num_tiles;
  void *out;                   // 16-bit elements
  long long out_ld, out_mat;   // row stride and matrix stride in elements
  const void *src;             // epilogue operand (A for POLY, X for AXPY), 16-bit elements
  long long src_ld, src_mat;
  const float *scale;          // per-matrix factor (SYRK: s^2, AXPY: s) or null
  float mul;                   // SYRK, AXPY: power-of-two storage factor, times scale[mat]
  // AXPY only: low halves of X as e5m2 bytes, lo = e5m2 * lo_in_mul on the way
  // in and e5m2(lo' * lo_out_mul) on the way out (powers of two); read at the
  // element the thread then writes, so one buffer serves in place
  const uint8_t *src_lo;
  uint8_t *out_lo;
  float lo_in_mul, lo_out_mul;
  float a, b, c;               // AXPY: a; POLY: b, c (with the storage factors folded in)
  float kw, ko;                // APPLY only: W' = kw W + ko O
  unsigned *err;
  unsigned long long timeout_ns;
};

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe of the same phase (never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

struct Watch {
  volatile int *abort;
  unsigned *err;
  unsigned long long limit_ns;
};

// Bounded wait for the phase of `bar` with the given parity to complete.
// Returns false (and stops waiting) on timeout or when another role aborted.
__device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, Watch w) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*w.abort) return false;
      if (global_ns() - t0 > w.limit_ns) {
        *w.abort = 1;
        atomicOr(w.err, kErrTimeout);
        return false;
      }
    }
  }
}

// The same bounded wait by polling with test_wait: the thread is never
// suspended, so it sees the phase flip without a wake-up delay, at the price
// of the issue slots its spinning takes from warps on the same scheduler.
// The producer and the MMA issuer wait on the operand ring this way: measured
// 1-2.5% faster per kernel than suspending in try_wait (and it lets the
// update-fused kernel and X X^T profit from single-k-block stages).
__device__ __forceinline__ bool wait_polled(uint32_t bar, uint32_t parity, Watch w) {
  if (mbar_test_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test_wait(bar, parity)) return true;
    if ((it & 1023u) == 0) {
      if (*w.abort) return false;
      if (global_ns() - t0 > w.limit_ns) {
        *w.abort = 1;
        atomicOr(w.err, kErrTimeout);
        return false;
      }
    }
  }
}

// Checked builds (-DMUON_DEVICE_CHECKS: the library's variant libmuon_checked.so)
// test, before each access that would fault if it broke, an invariant the
// kernels hold by construction: a TMA coordinate's x on a 16-element boundary
// (16 bytes or more), no store at a negative coordinate, a shared-memory
// offset inside its slot, a TMEM column inside the allocation.  A broken one
// sets MUON_ERR_DEVICE in the error word and the access is skipped (a skipped
// load leaves its barrier short, so the wait for it times out and the kernel
// returns).  The normal build compiles the checks away.
#ifdef MUON_DEVICE_CHECKS
__device__ __forceinline__ bool dcheck(bool ok, unsigned *err) {
  if (!ok && err) atomicOr(err, kErrDevice);
  return ok;
}
#else
__device__ __forceinline__ constexpr bool dcheck(bool, unsigned *) { return true; }
#endif

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c0, int c1,
                                            int c2, unsigned *err) {
  if (!dcheck((c0 & 15) == 0 && c2 >= 0, err)) return;
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Pair form: the completion is signalled on an mbarrier that may live in the
// peer CTA (a shared::cluster address), here always the pair's even CTA.
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c0, int c1,
                                                 int c2, unsigned *err) {
  if (!dcheck((c0 & 15) == 0 && c2 >= 0, err)) return;
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Arrive on an mbarrier given by its shared::cluster address (possibly in the
// peer CTA), with the default release semantics of mbarrier.arrive.  A
// cluster-scope release here would make every arrival wait for this thread's
// earlier global stores to drain.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// every thread of both CTAs of the cluster
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int c0, int c1, int c2,
                                             unsigned *err) {
  if (!dcheck((c0 & 15) == 0 && c0 >= 0 && c1 >= 0 && c2 >= 0, err)) return;
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the shared-memory source of every committed store has been read
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// every committed store has completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// order this thread's generic-proxy shared-memory accesses before later async-proxy (TMA) accesses
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Arrives once on the mbarrier at offset `bar` in every CTA of the pair named
// in `mask` when all MMAs issued so far by this thread have completed.
__device__ __forceinline__ void tc_commit_mc(uint32_t bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   bar),
               "h"(mask)
               : "memory");
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 lanes x 32 consecutive fp32 columns -> 32 registers per thread, waited.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Shared-memory matrix descriptor: start address, leading and stride byte
// offsets, descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: fp32 D (bit 4), A and B both bf16
// (format 1 at bits 7 and 10) or both fp16 (format 0), each operand K-major
// or MN-major (bits 15 and 16), N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t make_idesc(int m, int n, bool a_mn_major, bool b_mn_major, int tin) {
  return (1u << 4) | (tin == kBF16 ? (1u << 7) | (1u << 10) : 0u) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// Two floats to a pair of 16-bit values of format T (round to nearest even),
// as one 32-bit word, and back.
template <int T>
__device__ __forceinline__ uint32_t pack2(float x, float y) {
  if (T == kBF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    return *reinterpret_cast<uint32_t *>(&h);
  } else {
    __half2 h = __floats2half2_rn(x, y);
    return *reinterpret_cast<uint32_t *>(&h);
  }
}

template <int T>
__device__ __forceinline__ float2 unpack2(uint32_t v) {
  if (T == kBF16) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&v);
    return __bfloat1622float2(h);
  } else {
    __half2 h = *reinterpret_cast<__half2 *>(&v);
    return __half22float2(h);
  }
}

// The two e5m2 bytes in half `hi16` of `word` (first in the low byte) as two
// floats times `mul`.  e5m2 is the upper byte of an IEEE fp16, so the bytes
// widen exactly through fp16.
__device__ __forceinline__ float2 e5m2x2_to_float2(uint32_t word, int hi16, float mul) {
  const uint32_t pair = hi16 ? (word >> 16) : (word & 0xffffu);
  const uint32_t h2 = __byte_perm(pair, 0u, 0x1404);   // [0, b0, 0, b1]: fp16 pair (b0 << 8, b1 << 8)
  const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h2));
  return make_float2(f.x * mul, f.y * mul);
}

// Two floats to two e5m2 bytes (round to nearest even, saturating to the
// largest finite value), the first in the low byte.
__device__ __forceinline__ uint32_t float2_to_e5m2x2(float x, float y) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(x, y), __NV_SATFINITE, __NV_E5M2);
}

// One float to the 16-bit pattern of format T.
template <int T>
__device__ __forceinline__ uint16_t cvt16(float x) {
  if (T == kBF16) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t *>(&h);
  } else {
    __half h = __float2half_rn(x);
    return *reinterpret_cast<uint16_t *>(&h);
  }
}

// Tile t -> (matrix, row tile, column tile) of 256 x 256 pair tiles.
// aX + BX walks the tiles so that consecutive ones (which run at the same
// time on neighbouring pairs) share their block of X, the operand read by 7
// tiles: down a column when X is the B operand, along a row when it is the A
// operand (X stored transposed).  Symmetric outputs enumerate, per matrix,
// the tiles on or above the diagonal: row tile i needs column tiles j >= i.
template <int EPI>
__device__ __forceinline__ void decode_tile(const Params &p, long long t, int &mat, int &ti, int &tj) {
  mat = (int)(t / p.tiles_per_mat);
  int r = (int)(t - (long long)mat * p.tiles_per_mat);
  if (EPI >= EPI_AXPY) {
    if (p.row_order) {
      ti = r / p.tiles_n;
      tj = r - ti * p.tiles_n;
    } else {
      tj = r / p.tiles_m;
      ti = r - tj * p.tiles_m;
    }
  } else {
    int i = 0;
    for (;;) {
      const int cnt = p.tiles_n - i;
      if (r < cnt) break;
      r -= cnt;
      ++i;
    }
    ti = i;
    tj = i + r;
  }
}

union Pack8 {
  uint4 v;
  uint32_t w[4];   // pairs of 16-bit values
};

// Bounded wait used on the way out after an abort: waits for the phase of
// `bar` with the given parity to complete, for at most limit_ns, without
// looking at the abort flag (the caller has already given up).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return;
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > limit_ns) return;
}

// TIN: the 16-bit format of both tensor-core operands (which is also that of
// the epilogue's operand, A for POLY and X's high half for AXPY / APPLY);
// TOUT: the format the epilogue stores (SYRK, POLY, AXPY; APPLY stores bf16).
template <int EPI, bool A_MN, bool B_MN, int TIN, int TOUT>
__global__ void __launch_bounds__(THREADS, 1)
    ns_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int STAGES = Layout<EPI>::stages;
  constexpr int KSUB = Layout<EPI>::ksub;
  constexpr int SBYTES = Layout<EPI>::stage_bytes;
  static_assert(STAGES <= 32, "the producer tracks its stages in a 32-bit mask");
  uint8_t *epi_smem = smem + STAGES * SBYTES;  // epilogue staging slots, 1024-aligned
  uint64_t *bars = reinterpret_cast<uint64_t *>(epi_smem + Layout<EPI>::epi_bytes);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + Layout<EPI>::num_bars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();          // 0: issues the MMAs; 1: its peer
  const long long cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  constexpr int NFULL = STAGES * KSUB;
#define FULL(s, j) (bar0 + 8u * (uint32_t)((s) * KSUB + (j)))
#define EMPTY(s) (bar0 + 8u * (uint32_t)(NFULL + (s)))
#define ACCF(a) (bar0 + 8u * (uint32_t)(NFULL + STAGES + (a)))
#define ACCE(a) (bar0 + 8u * (uint32_t)(NFULL + STAGES + 2 + (a)))
#define EBAR(e) (bar0 + 8u * (uint32_t)(NFULL + STAGES + 5 + (e)))
  const uint32_t drain_bar = bar0 + 8u * (uint32_t)(NFULL + STAGES + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      for (int j = 0; j < KSUB; ++j)
        mbar_init(FULL(s, j), 1);  // used in CTA 0: its producer's expect_tx for both halves
      mbar_init(EMPTY(s), 1);      // multicast commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(ACCF(a), 1);                 // multicast commit
      mbar_init(ACCE(a), 2 * EPI_WARPS);     // used in CTA 0: every epilogue warp of the pair
    }
    mbar_init(drain_bar, 1);
    for (int e = 0; e < EPI_WARPS * Layout<EPI>::slots; ++e) mbar_init(EBAR(e), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (EPI != EPI_SYRK) tma_prefetch_desc(&p.tm_src);
    if (EPI >= EPI_AXPY) tma_prefetch_desc(&p.tm_out);
  }
  if (warp == 1) {  // one warp in each CTA of the pair allocates the same columns in both
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers are initialised before anyone signals them
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Watch w{abort_flag, p.err, p.timeout_ns};
  const int num_kb = (p.K + BK - 1) / BK;
  const int num_steps = (num_kb + KSUB - 1) / KSUB;  // stages per tile
  // a bounded wait on the way out after an abort (a fraction of the normal limit)
  const unsigned long long drain_ns = p.timeout_ns < 20000000ull ? p.timeout_ns : 20000000ull;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;   // stages ever filled, and the parity of their last fill
      for (long long t = cid; t < p.num_tiles; t += ncl) {
        int mat, ti, tj;
        decode_tile<EPI>(p, t, mat, ti, tj);
        const int arow = ti * CM + (int)rank * BM;    // this CTA's rows of A
        const int brow = tj * BN + (int)rank * BNH;   // this CTA's half of B
        // aX + BX: tiles that share an operand block start their K loop at
        // different offsets ((ti + tj) mod T of T segments, T the larger tile
        // count, so neighbouring tiles start about one k-block apart): a
        // block's first fetch from DRAM is waited on by the leading tile and
        // the ones just behind it read it from L2.  The sum over K starts and
        // wraps at the offset (a fixed order per tile).  Spreading the starts
        // over the whole K loop (T = 7) measured slower, as did any rotation
        // in the long-K symmetric kernels (reuse distances past what L2 holds).
        const int kt = p.tiles_m > p.tiles_n ? p.tiles_m : p.tiles_n;
        const int kb0 = EPI >= EPI_AXPY ? (int)((long long)((ti + tj) % kt) * num_kb / kt) : 0;
        bool ok = true;
        for (int i = 0; i < num_steps; ++i) {
          if (!wait_polled(EMPTY(stage), phase ^ 1u, w)) {
            ok = false;
            break;
          }
          const int valid = num_kb - i * KSUB < KSUB ? num_kb - i * KSUB : KSUB;
          // Each k-block of the stage completes on its own full barrier, so the
          // MMAs start on the first while the second is still landing.  CTA 0's
          // barrier counts the bytes of both halves; CTA 1's loads only complete
          // bytes on it (a stage is refilled only after the MMAs that read it
          // finished, so no load can run ahead into the next phase).  A k-block
          // past the end of K still completes its phase, with no bytes.
          if (rank == 0)
#pragma unroll
            for (int j = 0; j < KSUB; ++j) mbar_expect_tx(FULL(stage, j), j < valid ? 2 * STAGE_BYTES : 0);
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
#pragma unroll
          for (int j = 0; j < KSUB; ++j) {
            if (j >= valid) break;
            const int ki = i * KSUB + j;
            const int kb = kb0 + ki < num_kb ? kb0 + ki : kb0 + ki - num_kb;
            const uint32_t sa = sbase + stage * SBYTES + j * STAGE_BYTES, sb = sa + A_STAGE;
            const uint32_t full0 = map_to_rank(FULL(stage, j), 0);
            // K-major operands: one box of 128 rows x 64 K-columns.  MN-major
            // operands: boxes of 64 M/N-columns x 64 K-rows, one per swizzle atom.
            if (!A_MN) {
              tma_load_3d_pair(sa, &tmA, full0, kb * BK, arow, mat, p.err);
            } else {
#pragma unroll
              for (int q = 0; q < BM / 64; ++q)
                tma_load_3d_pair(sa + q * (64 * BK * 2), &tmA, full0, arow + q * 64, kb * BK, mat, p.err);
            }
            if (!B_MN) {
              tma_load_3d_pair(sb, &tmB, full0, kb * BK, brow, mat, p.err);
            } else {
#pragma unroll
              for (int q = 0; q < BNH / 64; ++q)
                tma_load_3d_pair(sb + q * (64 * BK * 2), &tmB, full0, brow + q * 64, kb * BK, mat, p.err);
            }
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      // After an abort, stages may still be filling.  CTA 0's full barriers of
      // a stage count both CTAs' bytes of every fill CTA 0 posted, so waiting
      // for the last fill of each stage to complete (at once when it already
      // did) keeps both CTAs' shared memory alive until those copies land.
      if (*abort_flag && rank == 0)
        for (int s2 = 0; s2 < STAGES; ++s2)
          if (issued & (1u << s2))
            for (int j = 0; j < KSUB; ++j) drain_wait(FULL(s2, j), (issued_parity >> s2) & 1u, drain_ns);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (CTA 0 of the pair)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = make_idesc(CM, BN, A_MN, B_MN, TIN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (long long t = cid; t < p.num_tiles; t += ncl) {
        if (!wait_bounded(ACCE(acc), acc_phase ^ 1u, w)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * ACC_COLS);
        bool ok = true;
        for (int i = 0; i < num_steps; ++i) {  // i-th stage of the tile in the producer's order
          const int valid = num_kb - i * KSUB < KSUB ? num_kb - i * KSUB : KSUB;
#pragma unroll
          for (int j = 0; j < KSUB; ++j) {
            if (j >= valid) break;
            if (!wait_polled(FULL(stage, j), phase, w)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = sbase + stage * SBYTES + j * STAGE_BYTES, sb = sa + A_STAGE;
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk) {
              // K-major: advance 16 K-elements (32 bytes) inside the swizzle row.
              // MN-major: advance 16 K-rows (two 8-row groups of 1024 bytes);
              // LBO = 8192 bytes between 64-wide atoms, SBO = 1024 between K groups.
              // The same shared-memory offsets address the peer CTA's halves.
              const uint64_t adesc = A_MN ? smem_desc(sa + kk * (UMMA_K * 128), 64 * BK * 2, 1024)
                                          : smem_desc(sa + kk * (UMMA_K * 2), 16, 1024);
              const uint64_t bdesc = B_MN ? smem_desc(sb + kk * (UMMA_K * 128), 64 * BK * 2, 1024)
                                          : smem_desc(sb + kk * (UMMA_K * 2), 16, 1024);
              tc_mma(d, adesc, bdesc, idesc, ((i * KSUB + j) | kk) != 0 ? 1u : 0u);
            }
          }
          if (!ok) break;
          tc_commit_mc(EMPTY(stage), 0x3);  // both CTAs may refill this stage
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_mc(ACCF(acc), 0x3);  // both CTAs' accumulators are ready
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // all MMAs issued by this thread have completed once drain_bar flips
      tc_commit_mc(drain_bar, 0x1);
      volatile int no_abort = 0;
      wait_bounded(drain_bar, 0, Watch{&no_abort, p.err, p.timeout_ns});
    }
  } else if (EPI >= EPI_AXPY) {
    // ---------------------------------------------------------------- AXPY epilogue (both CTAs)
    // X' = s (a (hi + lo) + acc) through shared memory: each warp stages a
    // 32 x 32 box of hi and the matching 32 x 32 bytes of lo (TMA loads,
    // zero-filled past the edges), writes hi' = TOUT(X') and lo' = e5m2(S_out
    // (X' - hi')) over them (each lane over what it has just read) and
    // TMA-stores them (clipped at the edges); the boxes of chunk g + SLOTS are
    // fetched into the slot once those stores have read it.  lo is stored as
    // an 8-bit e5m2 times a power of two: X' - hi' is at most hi's rounding
    // unit, which a bound on X' limits, so the scale S_out keeps every lo' in
    // e5m2's range (and lo = e5m2 / S_in on the way in).  APPLY stages hi and
    // the box of W instead (the last iteration's input carries no low half)
    // and writes W' = bf16(kw W + ko bf16(X')), the parameter update of the
    // unfused path, operation for operation, over the slot, in chunks of
    // MUON_APPLY_CW columns (2 KB boxes, or 1 KB ones for 16 columns).  Lane i
    // owns row i of the box, which is TMEM lane 32q + i; the swizzle spanning a
    // box row (64 or 32 bytes) makes these row reads conflict-free.
    constexpr bool APPLY = EPI == EPI_APPLY;
    constexpr int SLOTS = Layout<EPI>::slots;
    constexpr int IN_BYTES = Layout<EPI>::in_bytes;
    constexpr int CW = Layout<EPI>::cw;            // chunk width: 32 columns, or 16
    constexpr int NCH = 128 / CW;                  // chunks per warp and tile
    constexpr int BOXB = Layout<EPI>::box_bytes;   // one 32 x CW box of 16-bit values
    constexpr int LOB = Layout<EPI>::lo_bytes;     // one 32 x CW box of the 8-bit low half
    constexpr int PIECES = CW / 8;                 // 16-byte pieces per 16-bit box row
    static_assert(APPLY || CW == 32, "aX + BX moves 32-column chunks");
    // every lane's 16-byte accesses stay inside its slot's boxes, and every
    // chunk's accumulator columns inside the TMEM allocation
    static_assert(31 * (2 * CW) + (PIECES - 1) * 16 + 16 <= BOXB, "16-bit box rows stay inside the box");
    static_assert(APPLY || 31 * 32 + 16 + 16 <= LOB, "low-half box rows stay inside the box");
    static_assert(ACC_COLS + 128 + NCH * CW <= TMEM_COLS, "accumulator columns stay inside TMEM");
    const int ew = warp - 2;
    const int q = warp & 3, half = ew >> 2;
    uint8_t *ebase = epi_smem + ew * SLOTS * IN_BYTES;
    const uint32_t ebase_s = smem_u32(ebase);
    uint32_t ephase_bits = 0;                                // parity per slot
    uint32_t pending = 0;                                    // slots with a load not yet waited for
    const bool lo_in = !APPLY && p.src_lo != nullptr, lo_out = !APPLY && p.out_lo != nullptr;
    const uint32_t etx = BOXB + (lo_in ? (uint32_t)LOB : 0u) + (APPLY ? (uint32_t)BOXB : 0u);
    auto epi_load = [&](int slot, int m_, int row0_, int col0_) {  // lane 0 only
      const uint32_t dst = ebase_s + slot * IN_BYTES, bar = EBAR(ew * SLOTS + slot);
      fence_proxy_async_smem();
      mbar_expect_tx(bar, etx);
      tma_load_3d(dst, &p.tm_src, bar, col0_, row0_, m_, p.err);
      if (lo_in) tma_load_3d(dst + BOXB, &p.tm_src_lo, bar, col0_, row0_, m_, p.err);
      if (APPLY) tma_load_3d(dst + BOXB, &p.tm_out, bar, col0_, row0_, m_, p.err);  // W, stored over later
      pending |= 1u << slot;
    };
    const int rbase = (int)rank * BM + q * 32;  // this warp's rows within a pair tile
    int acc = 0;
    uint32_t acc_phase = 0;
    long long t = cid;
    int mat = 0, ti = 0, tj = 0;
    if (t < p.num_tiles) {
      decode_tile<EPI>(p, t, mat, ti, tj);
      if (lane == 0)
        for (int c = 0; c < SLOTS; ++c) epi_load(c, mat, ti * CM + rbase, tj * BN + half * 128 + c * CW);
    }
    bool alive = true;
    for (; alive && t < p.num_tiles; t += ncl) {
      const long long tn = t + ncl;
      int mat_n = 0, ti_n = 0, tj_n = 0;
      if (tn < p.num_tiles) decode_tile<EPI>(p, tn, mat_n, ti_n, tj_n);
      const bool ok = wait_bounded(ACCF(acc), acc_phase, w);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int row0 = ti * CM + rbase;
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * ACC_COLS + half * 128);
      const float sc = (p.scale ? p.scale[mat] : 1.0f) * p.mul;
#pragma unroll 1
      for (int ch = 0; ch < NCH; ++ch) {
        const int slot = ch % SLOTS;   // NCH is a multiple of SLOTS
        uint8_t *ebuf = ebase + slot * IN_BYTES;
        const uint32_t ebuf_s = ebase_s + slot * IN_BYTES;
        const int col0 = tj * BN + half * 128 + ch * CW;
        const bool got = wait_bounded(EBAR(ew * SLOTS + slot), (ephase_bits >> slot) & 1u, w);
        if (!__all_sync(0xffffffffu, got)) {
          alive = false;
          break;
        }
        ephase_bits ^= 1u << slot;
        pending &= ~(1u << slot);
        uint32_t r[32];
        __syncwarp();
        if (CW == 32)
          tmem_ld32(taddr + (uint32_t)(ch * CW), r);
        else
          tmem_ld16(taddr + (uint32_t)(ch * CW), r);
        __syncwarp();
        if (APPLY) {
#pragma unroll
          for (int c = 0; c < PIECES; ++c) {
            // 64-byte rows with the 64-byte swizzle, or 32-byte rows with the 32-byte swizzle
            const uint32_t off = CW == 32 ? (uint32_t)(lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4))
                                          : (uint32_t)(lane * 32 + ((c ^ ((lane >> 2) & 1)) << 4));
            Pack8 hv, wv, ho;
            hv.v = *reinterpret_cast<const uint4 *>(ebuf + off);
            wv.v = *reinterpret_cast<const uint4 *>(ebuf + BOXB + off);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int k = c * 8 + 2 * e;
              const float2 fh = unpack2<TIN>(hv.w[e]);
              const float v0 = sc * fmaf(p.a, fh.x, __uint_as_float(r[k]));
              const float v1 = sc * fmaf(p.a, fh.y, __uint_as_float(r[k + 1]));
              // O = bf16(X'); W' = kw W + ko O, each product and the sum rounded separately
              const float2 hh = unpack2<kBF16>(pack2<kBF16>(v0, v1));
              const float2 wf = unpack2<kBF16>(wv.w[e]);
              ho.w[e] = pack2<kBF16>(__fadd_rn(__fmul_rn(p.kw, wf.x), __fmul_rn(p.ko, hh.x)),
                                     __fadd_rn(__fmul_rn(p.kw, wf.y), __fmul_rn(p.ko, hh.y)));
            }
            *reinterpret_cast<uint4 *>(ebuf + off) = ho.v;
          }
        } else {
          // two 16-byte pieces of lo per lane row (32 bytes, 32-byte swizzle), each
          // covering two 16-byte pieces of hi (8 columns each)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const uint32_t loff = (uint32_t)(lane * 32 + ((j ^ ((lane >> 2) & 1)) << 4));
            Pack8 lv, lo;
            lv.v = lo_in ? *reinterpret_cast<const uint4 *>(ebuf + BOXB + loff) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              const int c = 2 * j + cc;
              const uint32_t off = (uint32_t)(lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4));
              Pack8 hv, ho;
              hv.v = *reinterpret_cast<const uint4 *>(ebuf + off);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int k = c * 8 + 2 * e;
                const float2 fh = unpack2<TIN>(hv.w[e]);
                const float2 fl = e5m2x2_to_float2(lv.w[cc * 2 + (e >> 1)], e & 1, p.lo_in_mul);
                const float v0 = sc * fmaf(p.a, fh.x + fl.x, __uint_as_float(r[k]));
                const float v1 = sc * fmaf(p.a, fh.y + fl.y, __uint_as_float(r[k + 1]));
                ho.w[e] = pack2<TOUT>(v0, v1);
                const float2 hh = unpack2<TOUT>(ho.w[e]);
                const uint32_t l2 = float2_to_e5m2x2((v0 - hh.x) * p.lo_out_mul, (v1 - hh.y) * p.lo_out_mul);
                // bytes 2e, 2e+1 of this hi piece's 8 lo bytes
                const int word = cc * 2 + (e >> 1);
                lo.w[word] = (e & 1) ? (lo.w[word] & 0x0000ffffu) | (l2 << 16) : l2;
              }
              *reinterpret_cast<uint4 *>(ebuf + off) = ho.v;
            }
            if (lo_out) *reinterpret_cast<uint4 *>(ebuf + BOXB + loff) = lo.v;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&p.tm_out, ebuf_s, col0, row0, mat, p.err);
          if (lo_out) tma_store_3d(&p.tm_out_lo, ebuf_s + BOXB, col0, row0, mat, p.err);
          bulk_commit();
          bulk_wait_read_all();  // the stores have read the slot the next load fills
          // every lane has read this input slot: fetch chunk ch + SLOTS into it (possibly of the next tile)
          const int nc = ch + SLOTS;
          if (nc < NCH)
            epi_load(slot, mat, row0, col0 + SLOTS * CW);
          else if (tn < p.num_tiles)
            epi_load(slot, mat_n, ti_n * CM + rbase, tj_n * BN + half * 128 + (nc - NCH) * CW);
        }
        __syncwarp();
      }
      if (!alive) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_to_rank(ACCE(acc), 0));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
      mat = mat_n;
      ti = ti_n;
      tj = tj_n;
    }
    if (lane == 0) {
      bulk_wait_all();
      // after an abort: let the loads still filling this warp's slots land
      if (*abort_flag)
        for (int s2 = 0; s2 < SLOTS; ++s2)
          if (pending & (1u << s2)) drain_wait(EBAR(ew * SLOTS + s2), (ephase_bits >> s2) & 1u, drain_ns);
    }
  } else {
    // ---------------------------------------------------------------- SYRK / POLY epilogue (both CTAs)
    // Each warp's 32 x 32 chunk (rows row0.., columns col0.., both multiples
    // of 32) lies strictly above the diagonal, strictly below it, or on it.
    // Above: the values go through shared memory to two TMA stores, the box
    // itself (64-byte swizzle) and its transpose (the mirror, written as
    // [column][row] without swizzle).  Below: nothing (the mirror of another
    // chunk covers it).  On the diagonal: element stores, (r, c >= r) and the
    // mirror (c, r) for c > r.  POLY's operand b*A arrives by TMA in the box.
    // (Reading it into registers for the whole tile before the accumulator is
    // ready measured 5% slower.)
    constexpr int SLOTS = Layout<EPI>::slots;
    static_assert(31 * 64 + 3 * 16 + 16 <= EPI_BOX_BYTES, "direct box rows stay inside the box");
    static_assert((31 * 32 + 31 + 1) * 2 <= EPI_BUF - EPI_BOX_BYTES, "mirror box entries stay inside the slot");
    static_assert(ACC_COLS + 128 + CHUNKS * 32 <= TMEM_COLS, "accumulator columns stay inside TMEM");
    const int ew = warp - 2;
    const int q = warp & 3, half = ew >> 2;
    uint8_t *ebase = epi_smem + ew * SLOTS * EPI_BUF;   // slots of [direct box][mirror box]
    const uint32_t ebase_s = smem_u32(ebase);
    uint32_t ephase_bits = 0;
    uint32_t pending = 0;                               // slots with a load not yet waited for
    const int rbase = (int)rank * BM + q * 32;
    auto needs_load = [&](int row0_, int col0_) {
      return EPI == EPI_POLY && col0_ + 32 > row0_ && row0_ < p.M && col0_ < p.N;
    };
    auto epi_load = [&](int slot, int m_, int row0_, int col0_) {  // lane 0 only
      const uint32_t bar = EBAR(ew * SLOTS + slot);
      fence_proxy_async_smem();
      mbar_expect_tx(bar, EPI_BOX_BYTES);
      tma_load_3d(ebase_s + slot * EPI_BUF, &p.tm_src, bar, col0_, row0_, m_, p.err);
      pending |= 1u << slot;
    };
    int acc = 0;
    uint32_t acc_phase = 0;
    long long t = cid;
    int mat = 0, ti = 0, tj = 0;
    if (t < p.num_tiles) {
      decode_tile<EPI>(p, t, mat, ti, tj);
      if (lane == 0)
        for (int c = 0; c < SLOTS; ++c) {
          const int r0 = ti * CM + rbase, c0 = tj * BN + half * 128 + c * 32;
          if (needs_load(r0, c0)) epi_load(c, mat, r0, c0);
        }
    }
    bool alive = true;
    for (; alive && t < p.num_tiles; t += ncl) {
      const long long tn = t + ncl;
      int mat_n = 0, ti_n = 0, tj_n = 0;
      if (tn < p.num_tiles) decode_tile<EPI>(p, tn, mat_n, ti_n, tj_n);
      const bool ok = wait_bounded(ACCF(acc), acc_phase, w);
      if (!__all_sync(0xffffffffu, ok)) break;  // warp-uniform: the TMEM loads below are .sync.aligned
      tc_fence_after();
      const int row0 = ti * CM + rbase;
      const int row = row0 + lane;
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * ACC_COLS + half * 128);
      const float sc = (p.scale ? p.scale[mat] : 1.0f) * p.mul;
      uint16_t *outm = static_cast<uint16_t *>(p.out) + (long long)mat * p.out_mat;
#pragma unroll 1
      for (int ch = 0; ch < CHUNKS; ++ch) {
        const int slot = ch % SLOTS;
        uint8_t *ebuf = ebase + slot * EPI_BUF;
        const int col0 = tj * BN + half * 128 + ch * 32;
        const bool in_range = row0 < p.M && col0 < p.N;
        const bool above = col0 >= row0 + 32, below = col0 + 32 <= row0;
        if (needs_load(row0, col0)) {
          const bool got = wait_bounded(EBAR(ew * SLOTS + slot), (ephase_bits >> slot) & 1u, w);
          if (!__all_sync(0xffffffffu, got)) {
            alive = false;
            break;
          }
          ephase_bits ^= 1u << slot;
          pending &= ~(1u << slot);
        }
        if (in_range && !below) {
          uint32_t r[32];
          __syncwarp();
          tmem_ld32(taddr + (uint32_t)(ch * 32), r);
          float v[32];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint32_t off = (uint32_t)(lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4));
            Pack8 av;
            if (EPI == EPI_POLY) av.v = *reinterpret_cast<const uint4 *>(ebuf + off);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int k = c * 8 + 2 * e;
              const float a0 = __uint_as_float(r[k]), a1 = __uint_as_float(r[k + 1]);
              if (EPI == EPI_SYRK) {
                v[k] = sc * a0;
                v[k + 1] = sc * a1;
              } else {
                const float2 f = unpack2<TIN>(av.w[e]);
                v[k] = fmaf(p.c, a0, p.b * f.x);
                v[k + 1] = fmaf(p.c, a1, p.b * f.y);
              }
            }
          }
          if (above) {
            // direct box [row][col] (swizzled) and mirror box [col][row]
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint32_t off = (uint32_t)(lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4));
              Pack8 o;
#pragma unroll
              for (int e = 0; e < 4; ++e) o.w[e] = pack2<TOUT>(v[c * 8 + 2 * e], v[c * 8 + 2 * e + 1]);
              *reinterpret_cast<uint4 *>(ebuf + off) = o.v;
            }
            uint16_t *mb = reinterpret_cast<uint16_t *>(ebuf + EPI_BOX_BYTES);
#pragma unroll
            for (int k = 0; k < 32; ++k) mb[k * 32 + lane] = cvt16<TOUT>(v[k]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              const uint32_t src = ebase_s + slot * EPI_BUF;
              tma_store_3d(&p.tm_out, src, col0, row0, mat, p.err);
              tma_store_3d(&p.tm_out_t, src + EPI_BOX_BYTES, row0, col0, mat, p.err);
              bulk_commit();
            }
          } else {
            // on the diagonal
            uint16_t *orow = outm + (long long)row * p.out_ld;
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const int c = col0 + k;
              if (row < p.M && c < p.N) {
                const uint16_t h = cvt16<TOUT>(v[k]);
                if (c >= row) orow[c] = h;
                if (c > row) outm[(long long)c * p.out_ld + row] = h;
              }
            }
          }
        }
        if (lane == 0) {
          // the slot's stores have read it: refill it with chunk ch + SLOTS
          bulk_wait_read_all();
          const int nc = ch + SLOTS;
          if (nc < CHUNKS) {
            if (needs_load(row0, col0 + SLOTS * 32)) epi_load(slot, mat, row0, col0 + SLOTS * 32);
          } else if (tn < p.num_tiles) {
            const int r0 = ti_n * CM + rbase, c0 = tj_n * BN + half * 128 + (nc - CHUNKS) * 32;
            if (needs_load(r0, c0)) epi_load(slot, mat_n, r0, c0);
          }
        }
        __syncwarp();
      }
      if (!alive) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_to_rank(ACCE(acc), 0));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
      mat = mat_n;
      ti = ti_n;
      tj = tj_n;
    }
    if (lane == 0) {
      bulk_wait_all();
      // after an abort: let the loads still filling this warp's slots land
      if (*abort_flag)
        for (int s2 = 0; s2 < SLOTS; ++s2)
          if (pending & (1u << s2)) drain_wait(EBAR(ew * SLOTS + s2), (ephase_bits >> s2) & 1u, drain_ns);
    }
  }
#undef FULL
#undef EMPTY
#undef ACCF
#undef ACCE
#undef EBAR

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA frees TMEM or exits while its peer may still use them
  if (*abort_flag) {
    // Fallback after the bounded drains above: CTA 1's operand loads signal
    // CTA 0's barrier, which counts them only for fills CTA 0 also posted,
    // so a fill CTA 1 issued alone is not covered there; a copy from L2 or
    // HBM lands within microseconds, so 200 us more leaves it ample time.
    const unsigned long long t0 = global_ns();
    while (global_ns() - t0 < 200000ull) __nanosleep(1000);
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

__global__ void selftest_wait_kernel(unsigned *err, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // phase 0 of `bar` never completes: nothing arrives on it
  wait_bounded(smem_u32(&bar), 0, Watch{&abort_flag, err, limit_ns});
}

// ------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// 3-D map over a [batch][rows][cols] stack of elements of format `fmt`
// (16-bit, or the 8-bit low half), rows `pitch` elements apart (0: dense);
// box = box_cols columns x box_rows rows x 1 matrix.
int make_map(CUtensorMap *map, const void *base, int fmt, int64_t batch, int64_t rows, int64_t cols, int box_rows,
             int box_cols = 64, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B, int64_t pitch = 0) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return MUON_ERR_CUDA;
  const cuuint64_t es = fmt == kE5M2 ? 1 : 2;   // element bytes
  const cuuint64_t ld = (cuuint64_t)(pitch > 0 ? pitch : cols);
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)batch};
  cuuint64_t strides[2] = {ld * es, (cuuint64_t)rows * ld * es};
  cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUtensorMapDataType dt = fmt == kE5M2 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : fmt == kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                               : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = enc(map, dt, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MUON_OK : MUON_ERR_CUDA;
}

template <int EPI, bool A_MN, bool B_MN, int TIN, int TOUT>
int launch(const CUtensorMap &ma, const CUtensorMap &mb, const Params &p, int trace_kind, cudaStream_t s) {
  if (p.num_tiles == 0) return MUON_OK;
  static std::once_flag attr_once[64];
  static int max_pairs[64];
  static cudaError_t attr_err[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MUON_ERR_CUDA;
  auto *kernel = ns_gemm_kernel<EPI, A_MN, B_MN, TIN, TOUT>;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(THREADS, 1, 1);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  std::call_once(attr_once[dev], [&] {
    attr_err[dev] = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Layout<EPI>::smem_bytes);
    // a persistent grid must fit at once: launch no more pairs than can be co-resident
    int n = 0;
    cfg.gridDim = dim3(2 * (unsigned)std::max(1, num_sms() / 2), 1, 1);
    cfg.dynamicSmemBytes = Layout<EPI>::smem_bytes;
    if (attr_err[dev] == cudaSuccess && cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) == cudaSuccess && n > 0)
      max_pairs[dev] = n;
    else
      max_pairs[dev] = std::max(1, num_sms() / 2);
    cudaGetLastError();
  });
  if (attr_err[dev] != cudaSuccess) return MUON_ERR_CUDA;
  // persistent CTA pairs over the tiles
  const long long pairs = std::min<long long>(p.num_tiles, max_pairs[dev]);
  cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
  cfg.dynamicSmemBytes = Layout<EPI>::smem_bytes;
  cfg.stream = s;
  trace_before(trace_kind, s);
  cudaError_t le = cudaLaunchKernelEx(&cfg, kernel, ma, mb, p);
  const int st = trace_after(trace_kind, s);
  return le == cudaSuccess ? st : MUON_ERR_CUDA;
}

Params base_params(int M, int N, int K, int64_t batch) {
  Params p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.tiles_m = (M + CM - 1) / CM;
  p.tiles_n = (N + BN - 1) / BN;
  p.err = device_error_word();
  p.timeout_ns = wait_timeout_ns();
  p.mul = 1.0f;
  (void)batch;
  return p;
}

int triangle_tiles(int tiles_m, int tiles_n) {
  int total = 0;
  for (int i = 0; i < tiles_m; ++i) total += tiles_n - i;
  return total;
}

bool valid_fmt(int f) { return f == kBF16 || f == kF16; }

}  // namespace

int ns_syrk(const void *X, int tin, void *A, int tout, int64_t batch, int64_t m, int64_t n, const float *s2,
            float mul, bool transposed, cudaStream_t s) {
  if (!valid_fmt(tin) || !valid_fmt(tout) || (tin == kF16 && tout == kBF16)) return MUON_ERR_INVALID_ARG;
  CUtensorMap ma, mb;
  int st;
  if (!transposed) {  // X stored m x n: both operands K-major, 128-row boxes
    st = make_map(&ma, X, tin, batch, m, n, BM);
    mb = ma;
  } else {            // X stored n x m (X^T): both operands MN-major, 64 x 64 boxes
    st = make_map(&ma, X, tin, batch, n, m, 64);
    mb = ma;
  }
  if (st) return st;
  Params p = base_params((int)m, (int)m, (int)n, batch);
  st = make_map(&p.tm_out, A, tout, batch, m, m, EPI_BOX, EPI_BOX, CU_TENSOR_MAP_SWIZZLE_64B);
  if (!st) st = make_map(&p.tm_out_t, A, tout, batch, m, m, EPI_BOX, EPI_BOX, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st) return st;
  p.tiles_per_mat = triangle_tiles(p.tiles_m, p.tiles_n);
  p.num_tiles = (long long)p.tiles_per_mat * batch;
  p.out = A;
  p.out_ld = m;
  p.out_mat = m * m;
  p.scale = s2;
  p.mul = mul;
  if (tin == kF16)
    return transposed ? launch<EPI_SYRK, true, true, kF16, kF16>(ma, mb, p, kTraceSyrk, s)
                      : launch<EPI_SYRK, false, false, kF16, kF16>(ma, mb, p, kTraceSyrk, s);
  if (tout == kF16)
    return transposed ? launch<EPI_SYRK, true, true, kBF16, kF16>(ma, mb, p, kTraceSyrk, s)
                      : launch<EPI_SYRK, false, false, kBF16, kF16>(ma, mb, p, kTraceSyrk, s);
  return transposed ? launch<EPI_SYRK, true, true, kBF16, kBF16>(ma, mb, p, kTraceSyrk, s)
                    : launch<EPI_SYRK, false, false, kBF16, kBF16>(ma, mb, p, kTraceSyrk, s);
}

int ns_poly(const void *A, int tin, void *B, int tout, int64_t batch, int64_t m, float b, float c, cudaStream_t s) {
  if (!valid_fmt(tin) || !valid_fmt(tout) || (tin == kBF16 && tout == kF16)) return MUON_ERR_INVALID_ARG;
  CUtensorMap ma, mb;
  int st = make_map(&ma, A, tin, batch, m, m, BM);
  mb = ma;
  if (st) return st;
  Params p = base_params((int)m, (int)m, (int)m, batch);
  st = make_map(&p.tm_src, A, tin, batch, m, m, EPI_BOX, EPI_BOX, CU_TENSOR_MAP_SWIZZLE_64B);
  if (!st) st = make_map(&p.tm_out, B, tout, batch, m, m, EPI_BOX, EPI_BOX, CU_TENSOR_MAP_SWIZZLE_64B);
  if (!st) st = make_map(&p.tm_out_t, B, tout, batch, m, m, EPI_BOX, EPI_BOX, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st) return st;
  p.tiles_per_mat = triangle_tiles(p.tiles_m, p.tiles_n);
  p.num_tiles = (long long)p.tiles_per_mat * batch;
  p.out = B;
  p.out_ld = m;
  p.out_mat = m * m;
  p.src = A;
  p.src_ld = m;
  p.src_mat = m * m;
  p.b = b;
  p.c = c;
  if (tin == kBF16) return launch<EPI_POLY, false, false, kBF16, kBF16>(ma, mb, p, kTracePoly, s);
  return tout == kBF16 ? launch<EPI_POLY, false, false, kF16, kBF16>(ma, mb, p, kTracePoly, s)
                       : launch<EPI_POLY, false, false, kF16, kF16>(ma, mb, p, kTracePoly, s);
}

namespace {

// X' = mul s1 (a X + B X) with X' written as Xn (+ Xn_lo), or, for EPI_APPLY,
// folded into W' = kw W + ko bf16(X') with W in place of Xn.
template <int EPI, int TIN, int TOUT>
int axpy_launch(const void *B, const void *X, const uint8_t *X_lo, float lo_in_mul, void *Xn, uint8_t *Xn_lo,
                float lo_out_mul, int64_t batch, int64_t m, int64_t n, float a, const float *s1, float mul, float kw,
                float ko, bool transposed, int trace_kind, cudaStream_t s) {
  CUtensorMap ma, mb;
  int st;
  Params p;
  if (!transposed) {
    // X' (m x n) = a X + B X: A operand B (K-major), B operand X (MN-major)
    st = make_map(&ma, B, TIN, batch, m, m, BM);
    if (!st) st = make_map(&mb, X, TIN, batch, m, n, 64);
    p = base_params((int)m, (int)n, (int)m, batch);
    p.out_ld = n;
  } else {
    // X stored n x m: X'^T = a X^T + X^T B (B symmetric), both operands K-major
    st = make_map(&ma, X, TIN, batch, n, m, BM);
    if (!st) st = make_map(&mb, B, TIN, batch, m, m, BNH);
    p = base_params((int)n, (int)m, (int)m, batch);
    p.out_ld = m;
  }
  if (st) return st;
  // epilogue boxes over X, X_lo, Xn, Xn_lo, all stored p.M x p.N: 32 rows x cw
  // columns, the swizzle spanning one box row
  const int eb = EPI_BOX, ecw = Layout<EPI>::cw;
  const CUtensorMapSwizzle sw64 = ecw == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
  st = make_map(&p.tm_src, X, TIN, batch, p.M, p.N, eb, ecw, sw64);
  // the low half: one byte per element, rows padded to 16 bytes (TMA strides);
  // boxes of 32 rows x 32 bytes, the 32-byte swizzle spanning a row
  const int64_t lo_pitch = (p.N + 15) & ~int64_t(15);
  if (!st && X_lo)
    st = make_map(&p.tm_src_lo, X_lo, kE5M2, batch, p.M, p.N, eb, 32, CU_TENSOR_MAP_SWIZZLE_32B, lo_pitch);
  if (!st) st = make_map(&p.tm_out, Xn, EPI == EPI_APPLY ? kBF16 : TOUT, batch, p.M, p.N, eb, ecw, sw64);
  if (!st && Xn_lo)
    st = make_map(&p.tm_out_lo, Xn_lo, kE5M2, batch, p.M, p.N, eb, 32, CU_TENSOR_MAP_SWIZZLE_32B, lo_pitch);
  if (st) return st;
  p.tiles_per_mat = p.tiles_m * p.tiles_n;
  p.num_tiles = (long long)p.tiles_per_mat * batch;
  p.out = Xn;
  p.out_mat = m * n;
  p.src = X;
  p.src_ld = p.out_ld;
  p.src_mat = m * n;
  p.a = a;
  p.scale = s1;
  p.mul = mul;
  p.src_lo = X_lo;
  p.out_lo = Xn_lo;
  p.lo_in_mul = lo_in_mul;
  p.lo_out_mul = lo_out_mul;
  p.kw = kw;
  p.ko = ko;
  p.row_order = transposed ? MUON_AXPY_ROW_ORDER_T : 0;
  return transposed ? launch<EPI, false, false, TIN, TOUT>(ma, mb, p, trace_kind, s)
                    : launch<EPI, false, true, TIN, TOUT>(ma, mb, p, trace_kind, s);
}

}  // namespace

int ns_axpy(const void *B, const void *X, int tin, const uint8_t *X_lo, float lo_in_mul, void *Xn, int tout,
            uint8_t *Xn_lo, float lo_out_mul, int64_t batch, int64_t m, int64_t n, float a, const float *s1, float mul,
            bool transposed, cudaStream_t s) {
  if (!valid_fmt(tin) || !valid_fmt(tout)) return MUON_ERR_INVALID_ARG;
#define MUON_AXPY(TI, TO)                                                                                          \
  axpy_launch<EPI_AXPY, TI, TO>(B, X, X_lo, lo_in_mul, Xn, Xn_lo, lo_out_mul, batch, m, n, a, s1, mul, 0.f, 0.f, \
                                transposed, kTraceAxpy, s)
  if (tin == kBF16) return tout == kBF16 ? MUON_AXPY(kBF16, kBF16) : MUON_AXPY(kBF16, kF16);
  return tout == kBF16 ? MUON_AXPY(kF16, kBF16) : MUON_AXPY(kF16, kF16);
#undef MUON_AXPY
}

int ns_axpy_apply(const void *B, const void *X, int tin, __nv_bfloat16 *W, int64_t batch, int64_t m, int64_t n,
                  float a, const float *s1, float mul, float kw, float ko, bool transposed, cudaStream_t s) {
  if (!valid_fmt(tin)) return MUON_ERR_INVALID_ARG;
  return tin == kBF16 ? axpy_launch<EPI_APPLY, kBF16, kBF16>(B, X, nullptr, 1.f, W, nullptr, 1.f, batch, m, n, a, s1,
                                                             mul, kw, ko, transposed, kTraceAxpyApply, s)
                      : axpy_launch<EPI_APPLY, kF16, kBF16>(B, X, nullptr, 1.f, W, nullptr, 1.f, batch, m, n, a, s1,
                                                            mul, kw, ko, transposed, kTraceAxpyApply, s);
}

int selftest_wait(unsigned long long timeout_ns, cudaStream_t s) {
  trace_before(kTraceSelftest, s);
  selftest_wait_kernel<<<1, 32, 0, s>>>(device_error_word(), timeout_ns);
  return trace_after(kTraceSelftest, s);
}

}  // namespace muon
