// Thin inline-PTX wrappers for sm_103a: mbarriers, TMA tile loads, tcgen05 tensor
// memory (alloc, load, store), tcgen05 MMA with shared-memory matrix descriptors,
// and bounded waits that give up with an error flag instead of hanging.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace attn {

// Device-side status bits, OR-ed into the library's status word.
enum : int { DEV_OK = 0, DEV_TIMEOUT = 1, DEV_BAD_INPUT = 2 };

// A wait gives up after this many nanoseconds of %globaltimer (each wait in these
// kernels is on work of the same CTA and normally lasts microseconds).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t lane_id() {
  uint32_t l;
  asm volatile("mov.u32 %0, %%laneid;" : "=r"(l));
  return l;
}

__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(pred));
  return pred != 0;
}

// Register reallocation between warpgroups: every warp of a warpgroup executes the same
// instruction. An increase waits until decreases elsewhere in the CTA have returned enough
// registers to the pool the CTA was launched with, so the counts must add up to at most
// that pool (threads x registers per thread at launch).
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  static_assert(N >= 24 && N <= 256 && N % 8 == 0, "register count");
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  static_assert(N >= 24 && N <= 256 && N % 8 == 0, "register count");
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Shared state every bounded wait of a CTA consults: a CTA-local abort flag (set by
// the first wait that gives up) and the library's global status word.
struct WaitCtx {
  volatile int* abort_smem;
  int* status_gmem;
};

// Waits for the phase with the given parity to complete. Returns false, after
// raising the abort flag and the global status, if the wait exceeds kWaitLimitNs
// or if another wait of this CTA already gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*w.abort_smem) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *w.abort_smem = 1;
        atomicOr(w.status_gmem, DEV_TIMEOUT);
        return false;
      }
    }
  }
}

// Waits for a copy this CTA issued, ignoring the abort flag (shared memory must not be
// left while a copy into it is in flight), for at most kDrainLimitNs.
constexpr unsigned long long kDrainLimitNs = 200000000ull;
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return;
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kDrainLimitNs) return;
}

// ---------------------------------------------------------------- named barriers
// Hardware CTA barriers 1..15 (0 is __syncthreads). Waiting on one touches no shared
// memory, so a thread that issues tcgen05.mma can wait on it without stalling the
// tensor pipe (a shared-memory access from that thread costs about 480 cycles while
// the pipe streams operands from shared memory). `count` is in threads, a multiple of
// 32, and every warp that takes part executes the instruction converged.
// Producers arrive (non-blocking); the consumer syncs. A producer may arrive again
// only after the consumer has synced the previous phase; the kernels guarantee this
// through their data dependencies, and after an abort they switch to nb_sync so that
// every arrival pairs with one consumer sync.
__device__ __forceinline__ void nb_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void nb_arrive(uint32_t id, uint32_t count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load of one box into shared memory, completing on `bar` (tx bytes).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Same, with an L2 eviction-priority hint (createpolicy result).
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar, int x, int y, int z,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "l"(policy)
      : "memory");
}

// Plain bulk copy global -> this CTA's shared memory, completing on `bar` (transaction
// bytes). Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Orders this thread's ordinary shared-memory writes before later TMA (async-proxy)
// accesses of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------- tcgen05: TMEM
// Allocation and release are warp-wide (.sync.aligned): call from one full warp.
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
__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// TMEM address: lane in bits 31..16, column in bits 15..0.
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col) {
  return base + (lane << 16) + col;
}

// tcgen05.ld / tcgen05.st / tcgen05.wait are warp-collective (.sync.aligned): every
// lane of the warp must execute them together. Each wrapper first reconverges the
// warp with __syncwarp(); a caller must still reach it from warp-uniform control flow.

// 32 lanes x 32 columns of 32-bit: thread t of the warp gets lane (base lane + t),
// columns col .. col+31 in r[0..31]. The values are valid only after tmem_wait_ld().
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  __syncwarp();
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}

// 32 lanes x 16 columns of 32-bit (thread t gets lane base + t).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  __syncwarp();
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() {
  __syncwarp();
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  __syncwarp();
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Ties the 32 registers to a point after tmem_wait_ld(), so that the compiler cannot
// move their first use above the wait.
__device__ __forceinline__ void reg_fence32(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

__device__ __forceinline__ void reg_fence16(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// 32 lanes x 8 columns store (thread t writes lane base+t, columns col..col+7).
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  __syncwarp();
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}

// 32 lanes x 16 columns store (thread t writes lane base+t, columns col..col+15).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  __syncwarp();
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  __syncwarp();
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// ---------------------------------------------------------------- tcgen05: MMA
// Shared-memory matrix descriptor for a tile written by TMA with 128-byte swizzle:
// rows of 128 bytes, 8-row (1024-byte) swizzle atoms. The start address must lie
// in a 1024-byte aligned atom (a +32/64/96-byte offset selects a 16-element K slice).
//   K-major operand : lbo unused (16 B), sbo = 1024 (next 8 rows of M/N).
//   MN-major operand: lbo = bytes to the next 64-element block of M/N,
//                     sbo = 1024 (next 8 rows of K).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;  // descriptor version for tcgen05
  d |= (uint64_t)2u << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16 with bf16 A and B, fp32 D.
// a_mn / b_mn: operand stored MN-major (transposed) instead of K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4)                       // D format f32
         | (1u << 7)                     // A format bf16
         | (1u << 10)                    // B format bf16
         | ((a_mn ? 1u : 0u) << 15)      // A major
         | ((b_mn ? 1u : 0u) << 16)      // B major
         | ((uint32_t)(N >> 3) << 17)    // N / 8
         | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// D(tmem) (+)= A(smem) * B(smem)^T-ish per the descriptors; accumulate if acc != 0.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}

// Same with A read from tensor memory (128 lanes = rows, K/2 columns of bf16 pairs).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                       uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}

// Predicated forms: every lane of the warp executes the instruction (no divergence, so
// the warp can go straight on to a warp-wide barrier); only lanes with `pred` issue.
__device__ __forceinline__ void mma_ss_if(bool pred, uint32_t d_tmem, uint64_t adesc,
                                          uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.b32 p, %4, 0;\n setp.ne.b32 q, %5, 0;\n"
      " @q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc), "r"((uint32_t)pred)
      : "memory");
}
__device__ __forceinline__ void mma_ts_if(bool pred, uint32_t d_tmem, uint32_t a_tmem,
                                          uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.b32 p, %4, 0;\n setp.ne.b32 q, %5, 0;\n"
      " @q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(acc), "r"((uint32_t)pred)
      : "memory");
}
__device__ __forceinline__ void mma_commit_if(bool pred, uint32_t bar) {
  asm volatile(
      "{\n .reg .pred q;\n setp.ne.b32 q, %1, 0;\n"
      " @q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(
          bar),
      "r"((uint32_t)pred)
      : "memory");
}

// Arrive once on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// ---------------------------------------------------------------- 8-bit (e4m3) MMAs
// Instruction descriptor for kind::f8f6f4 with e4m3 A and B (format code 0), f32 D,
// both operands K-major (8-bit operands are only used K-major here).
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4)                       // D format f32
         | (0u << 7) | (0u << 10)        // A, B format e4m3
         | ((uint32_t)(N >> 3) << 17)    // N / 8
         | ((uint32_t)(M >> 4) << 24);   // M / 16
}
// D (+)= A B^T, K = 32 per instruction, A and B in shared memory.
__device__ __forceinline__ void mma_f8_ss_if(bool pred, uint32_t d_tmem, uint64_t adesc,
                                             uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.b32 p, %4, 0;\n setp.ne.b32 q, %5, 0;\n"
      " @q tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc), "r"((uint32_t)pred)
      : "memory");
}
// Same with A in tensor memory: four e4m3 values per 32-bit column, the lowest byte
// holding the lowest K index, so K = 32 spans 8 columns.
__device__ __forceinline__ void mma_f8_ts_if(bool pred, uint32_t d_tmem, uint32_t a_tmem,
                                             uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.b32 p, %4, 0;\n setp.ne.b32 q, %5, 0;\n"
      " @q tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(acc), "r"((uint32_t)pred)
      : "memory");
}

// ---------------------------------------------------------------- Philox4x32-10
// The counter-based generator of Salmon, Moraes, Dror and Shaw ("Parallel random
// numbers: as easy as 1, 2, 3", SC 2011): ten rounds of
//   (hi0, lo0) = M0 x0, (hi1, lo1) = M1 x2, (x0, x1, x2, x3) <- (hi1^x1^k0, lo1, hi0^x3^k1, lo0)
// with the key (k0, k1) advanced by (W0, W1) after each round.
// The round keys of one seed (k0 + r W0, k1 + r W1 for rounds r = 0 .. 9): the same for
// every call with that seed, so a thread computes them once.
struct PhiloxKeys {
  uint32_t k0[10], k1[10];
};
__device__ __forceinline__ PhiloxKeys philox_keys(uint32_t k0, uint32_t k1) {
  constexpr uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  PhiloxKeys k;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    k.k0[r] = k0 + (uint32_t)r * W0;
    k.k1[r] = k1 + (uint32_t)r * W1;
  }
  return k;
}
__device__ __forceinline__ uint4 philox4x32_10(uint32_t x0, uint32_t x1, uint32_t x2,
                                               uint32_t x3, const PhiloxKeys& k) {
  constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = (uint64_t)M0 * x0, p1 = (uint64_t)M1 * x2;  // one wide multiply each
    const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    x0 = hi1 ^ x1 ^ k.k0[r];
    x1 = lo1;
    x2 = hi0 ^ x3 ^ k.k1[r];
    x3 = lo0;
  }
  return make_uint4(x0, x1, x2, x3);
}

// Dropout keep flags of four mask bytes at once. Byte b is kept iff b >= t, i.e. iff
// b + (255 - t) + 1 carries out of the byte. With y = 255 - t in every byte and
// ylo = (y & 0x7F7F7F7F) + 0x01010101, the low seven bits of every byte are added with
// the carry-in in one 32-bit add (at most 0x7F + 0x7F + 1: nothing crosses into the next
// byte), so bit 7 of the sum is the carry into bit 7, and the carry out of the byte is
// the majority of that and the two bit-7 inputs. Returns the flags in bit 7 of each byte
// (the other bits are don't-care).
struct DropThr {
  uint32_t y, ylo;
};
__host__ __device__ __forceinline__ DropThr drop_thr_words(int t) {
  const uint32_t y = 0x01010101u * (uint32_t)(255 - t);
  return {y, (y & 0x7F7F7F7Fu) + 0x01010101u};
}
__device__ __forceinline__ uint32_t keep_flags4(uint32_t w, const DropThr& th) {
  const uint32_t a = (w & 0x7F7F7F7Fu) + th.ylo;
  return (w & th.y) | ((w | th.y) & a);
}
// prmt with a selector: each selector nibble n picks byte n & 7 of {b, a} (a = bytes 0-3)
// and, when n & 8, replicates that byte's top bit over the whole result byte.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
// All-ones iff flag byte k (k = 0..3) of keep_flags4's result is set: an element mask.
// k is a constant after unrolling, so the selector is too.
__device__ __forceinline__ uint32_t keep_mask_elem(uint32_t flags, int k) {
  return prmt(flags, 0u, 0x8888u | (0x1111u * (uint32_t)k));
}
// Mask of a bf16 pair: bytes 0-1 from flag byte k, bytes 2-3 from flag byte k + 1.
__device__ __forceinline__ uint32_t keep_mask_pair(uint32_t flags, int k) {
  return prmt(flags, 0u, (0x88u | (0x11u * (uint32_t)k)) | ((0x88u | (0x11u * (uint32_t)(k + 1))) << 8));
}

// 16 x 16 byte transpose within each half-warp: lane s of a half (s = lane % 16) holds
// row s as w[0..3] (byte b of w[q] = column 4q + b) and ends with column s (byte c of
// the result = row c). One butterfly stage per bit of the column index: lanes s and
// s ^ m swap the bytes whose column bit differs from their own lane bit, and the
// partner's bytes land in the positions just vacated.
__device__ __forceinline__ void transpose16x16_bytes(uint32_t (&w)[4], int lane) {
  {  // column bit 3: words 2, 3 against words 0, 1
    const bool hi = lane & 8;
    const uint32_t r0 = __shfl_xor_sync(0xffffffffu, hi ? w[0] : w[2], 8);
    const uint32_t r1 = __shfl_xor_sync(0xffffffffu, hi ? w[1] : w[3], 8);
    w[0] = hi ? r0 : w[0];
    w[1] = hi ? r1 : w[1];
    w[2] = hi ? w[2] : r0;
    w[3] = hi ? w[3] : r1;
  }
  {  // column bit 2: words 1, 3 against words 0, 2
    const bool hi = lane & 4;
    const uint32_t r0 = __shfl_xor_sync(0xffffffffu, hi ? w[0] : w[1], 4);
    const uint32_t r1 = __shfl_xor_sync(0xffffffffu, hi ? w[2] : w[3], 4);
    w[0] = hi ? r0 : w[0];
    w[2] = hi ? r1 : w[2];
    w[1] = hi ? w[1] : r0;
    w[3] = hi ? w[3] : r1;
  }
  {  // column bit 1: the high half of each word against the low half
    const bool hi = lane & 2;
    const uint32_t ps = hi ? 0x5410u : 0x7632u;
    const uint32_t r0 = __shfl_xor_sync(0xffffffffu, prmt(w[0], w[1], ps), 2);
    const uint32_t r1 = __shfl_xor_sync(0xffffffffu, prmt(w[2], w[3], ps), 2);
    const uint32_t ue = hi ? 0x3254u : 0x5410u, uo = hi ? 0x3276u : 0x7610u;
    w[0] = prmt(w[0], r0, ue);
    w[1] = prmt(w[1], r0, uo);
    w[2] = prmt(w[2], r1, ue);
    w[3] = prmt(w[3], r1, uo);
  }
  {  // column bit 0: odd bytes against even bytes
    const bool hi = lane & 1;
    const uint32_t ps = hi ? 0x6420u : 0x7531u;
    const uint32_t r0 = __shfl_xor_sync(0xffffffffu, prmt(w[0], w[1], ps), 1);
    const uint32_t r1 = __shfl_xor_sync(0xffffffffu, prmt(w[2], w[3], ps), 1);
    const uint32_t ue = hi ? 0x3514u : 0x5240u, uo = hi ? 0x3716u : 0x7260u;
    w[0] = prmt(w[0], r0, ue);
    w[1] = prmt(w[1], r0, uo);
    w[2] = prmt(w[2], r1, ue);
    w[3] = prmt(w[3], r1, uo);
  }
}

// ---------------------------------------------------------------- math
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// tanh.approx.f32, one MUFU operation (16 per clock per SM). Measured on GB300 against
// float64 tanh on a grid of |x| < 24: at most 7.8e-6 absolute and 1e-5 relative error, so
// the soft-cap c tanh(s / c) it feeds is off by at most 7.8e-6 c.
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Packed fp32 pairs (sm_100 and later): two independent round-to-nearest operations per
// instruction, each bit for bit the scalar one. `lo` is the first element of a pair.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f32x2_split(uint64_t r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t sub_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Two floats to a bf16x2 word, round to nearest even; `lo` lands in bits 15..0.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two floats to two e4m3 bytes, round to nearest even, saturating at +-448; `lo` lands
// in bits 7..0.
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

}  // namespace attn
