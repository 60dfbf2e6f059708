// Inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA
// tile loads, and the tcgen05 tensor-core / tensor-memory instructions.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace fa {

// ---------------------------------------------------------------------------
// Device status word: the first wait that gives up records where it was.
// code = 0x80000000 | kernel << 16 | role << 8 | site.

struct StatusSlot {
  unsigned int *word;   // global status word (per library), may be null
  int *abort_flag;      // shared-memory abort flag of this CTA
  uint64_t limit_ns;    // wall-clock limit of one wait
};

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// ---------------------------------------------------------------------------
// mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
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

// The wall-clock limit of one wait comes with the status slot. A healthy wait
// lasts microseconds; the limit only turns a logic error into an error code
// instead of a hung GPU.

// Waits for the phase of parity `parity` of barrier `bar` to complete.
// Returns false (and records `code`) if it gives up or if another role of
// this CTA already gave up.
__device__ __forceinline__ bool mbar_wait_loop(uint32_t bar, uint32_t parity, StatusSlot st,
                                               uint32_t code) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u) {
      if (*(volatile int *)st.abort_flag) return false;
      if (global_timer_ns() - t0 > st.limit_ns) {
        *(volatile int *)st.abort_flag = 1;
        if (st.word) atomicCAS(st.word, 0u, code);
        return false;
      }
    }
  }
}

// The loop out of line: the callers' hot loops keep their registers.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, StatusSlot st,
                                                   uint32_t code) {
  return mbar_wait_loop(bar, parity, st, code);
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, StatusSlot st,
                                          uint32_t code) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, st, code);
}

// The same wait with the loop inlined, for kernels whose warpgroups set their
// own register counts (setmaxnreg): there every call is inlined.
__device__ __forceinline__ bool mbar_wait_inl(uint32_t bar, uint32_t parity, StatusSlot st,
                                              uint32_t code) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_loop(bar, parity, st, code);
}

// Teardown wait for copies and MMAs this CTA has already issued. Unlike
// mbar_wait it keeps waiting after another role of the CTA has given up:
// work in flight still writes this CTA's shared and tensor memory, so the CTA
// must not free its tensor memory or exit before that work is done. Only its
// own time limit ends it (recording `code` if no earlier failure did).
__device__ __forceinline__ bool mbar_wait_drain_inl(uint32_t bar, uint32_t parity, StatusSlot st,
                                                   uint32_t code) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u && global_timer_ns() - t0 > st.limit_ns) {
      *(volatile int *)st.abort_flag = 1;
      if (st.word) atomicCAS(st.word, 0u, code);
      return false;
    }
  }
}

static __device__ __noinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, StatusSlot st,
                                                    uint32_t code) {
  return mbar_wait_drain_inl(bar, parity, st, code);
}

// Register count of this warp's warpgroup: every warp of a warpgroup runs the
// same one. An increase takes registers that other warpgroups of the CTA have
// given up with a decrease, so the counts must add up to the launch's total
// (the kernel compiled to exactly its launch bound: see check_kernel_regs).
template <uint32_t kRegs>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs));
}
template <uint32_t kRegs>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs));
}

// ---------------------------------------------------------------------------
// TMA (bulk tensor copies)

__device__ __forceinline__ void tma_prefetch_desc(const void *tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 4-D tile load from a map over [B][H][rows][d]: x = column, y = row within
// the head, z = head, w = batch. Rows past the map's extent read zeros.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void *tmap, int x, int y, int z,
                                            int w, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}

// 4-D tile store from shared memory (a 128-byte-swizzled box) to a map over
// [B][H][rows][d]; rows past the tensor's extent are not written. Completion
// is tracked with bulk groups (bulk_commit_group / bulk_wait_group_read).
__device__ __forceinline__ void tma_store_4d(const void *tmap, uint32_t src, int x, int y, int z,
                                             int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];"
      ::"l"(reinterpret_cast<uint64_t>(tmap)), "r"(src), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until the committed bulk stores of this thread have finished reading
// shared memory (their global writes may still be in flight).
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// 1-D bulk copy global -> shared; both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void *src, uint32_t bytes,
                                             uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory allocation

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   dst_smem),
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

// ---------------------------------------------------------------------------
// tcgen05: MMA issue (one thread) and completion tracking

// D[tmem] (+)= A[smem] * B[smem]; kind::f16 (bf16 or f16 inputs as the instruction
// descriptor says, fp32 accumulate).
__device__ __forceinline__ void mma_f16kind_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem].
__device__ __forceinline__ void mma_f16kind_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 op issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Instruction descriptor for kind::f16 with fp32 D and A, B both bf16
// (f16 = false) or both f16 (f16 = true).
//   bits 4-5 D format (1 = f32), 7-9 A format (0 = f16, 1 = bf16), 10-12 B
//   format, 15 A major (0 = K-major, 1 = MN-major), 16 B major, 17-22 N >> 3,
//   24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_f32acc(int M, int N, int a_mn_major, int b_mn_major,
                                                    bool f16) {
  return (1u << 4) | ((f16 ? 0u : 1u) << 7) | ((f16 ? 0u : 1u) << 10) |
         (uint32_t(a_mn_major) << 15) | (uint32_t(b_mn_major) << 16) |
         (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle.
//   bits 0-13 start >> 4, 16-29 leading byte offset >> 4, 32-45 stride byte
//   offset >> 4, 46-47 version (1), 61-63 layout (2 = 128B swizzle).
// K-major operand: rows of 128 bytes (64 bf16 along K), 8-row groups `sbo`
// bytes apart; `lbo` unused. MN-major operand: K-rows of 128 bytes (64 bf16
// along M/N), 8-row groups `sbo` apart, next 64 M/N elements `lbo` apart.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((smem_addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory <-> registers. Shape 32x32b: warp w (w % 4 = q)
// reaches lanes 32q..32q+31; thread t of the warp gets lane 32q+t, and .xN
// moves N consecutive 32-bit columns starting at the address's column.

#define FA_REG8(a, i) \
  "=r"(a[i + 0]), "=r"(a[i + 1]), "=r"(a[i + 2]), "=r"(a[i + 3]), "=r"(a[i + 4]), \
      "=r"(a[i + 5]), "=r"(a[i + 6]), "=r"(a[i + 7])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : FA_REG8(r, 0), FA_REG8(r, 8), FA_REG8(r, 16), FA_REG8(r, 24)
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : FA_REG8(r, 0), FA_REG8(r, 8)
      : "r"(taddr));
}

#define FA_IN8(a, i) \
  "r"(a[i + 0]), "r"(a[i + 1]), "r"(a[i + 2]), "r"(a[i + 3]), "r"(a[i + 4]), "r"(a[i + 5]), \
      "r"(a[i + 6]), "r"(a[i + 7])

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      FA_IN8(r, 0), FA_IN8(r, 8), FA_IN8(r, 16), FA_IN8(r, 24)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      FA_IN8(r, 0), FA_IN8(r, 8)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Numerics helpers (hardware instructions)

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Pairs of fp32 values in one 64-bit register pair, for the packed fp32
// arithmetic of sm_100-class GPUs (one instruction for two lanes' worth).
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void f2unpack(uint64_t r, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}

__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ uint64_t fsub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// max(a, b, c) in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 -> packed bf16x2 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two fp32 values rounded to the 16-bit element type (round to nearest even)
// and packed, `lo` in the low half.
template <bool kF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return kF16 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi);
}

// The two 16-bit elements of `w` widened to fp32 (exact), low half first.
template <bool kF16>
__device__ __forceinline__ void unpack2(uint32_t w, float &lo, float &hi) {
  if (kF16) {
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %2; cvt.f32.f16 %0, l; cvt.f32.f16 %1, h; }"
        : "=f"(lo), "=f"(hi)
        : "r"(w));
  } else {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xffff0000u);
  }
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

}  // namespace fa
