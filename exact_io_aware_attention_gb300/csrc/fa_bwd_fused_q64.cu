// One-pass attention backward for head dimension 128 with 64-query steps, for
// sm_103a.
//
// The same method as fa_bwd_fused.cu (the pages regenerate S and P block by
// block in the backward pass: "Paper Notes: FlashAttention", "Background" and
// "Key Ideas"; aicassindra page "FlashAttention", "The backward pass:
// recompute instead of store"; the gradients are the analytic ones of
// O = softmax(scale QK^T) V): one CTA owns a 128-key K/V tile, loops over the
// Q tiles that see it, recomputes S^T and P^T once per (query, key) pair, and
// runs all five products; dK and dV accumulate in tensor memory and the dQ
// partials are added into the fp32 accumulator in the workspace.
//
// At d = 128 a 128-query step needs S^T, dP^T, dV, dK and a dQ partial of 128
// columns each: 640 of the 512 tensor-memory columns. Here each 128-row Q tile
// is processed as two steps of 64 queries, which halves S^T, dP^T and dQ:
//   [0,64)    K_j as 16-bit pairs (the A operand of S^T = K Q^T: TS form)
//   [64,128)  S^T (128 keys x 64 queries); P^T packed over it
//   [128,192) dP^T
//   [192,320) dV     [320,448) dK
//   [448,512) dQ^T = K^T dS^T (128 head-dimension rows x 64 queries)
// so every product has columns of its own. The products of a step (M = 128
// keys, or the head dimension for dQ^T):
//   S^T   TS  A = K (tensor memory), B = Q rows of the step (K-major)      N = 64
//   dP^T  SS  A = V, B = dO rows of the step (both K-major)                 N = 64
//   dV    TS  A = P^T (tensor memory), B = dO rows (MN-major)               N = 128
//   dK    SS  A = dS^T (shared, K-major), B = Q rows (MN-major)             N = 128
//   dQ^T  SS  A = K^T (K_j read MN-major), B = dS^T (shared, MN-major)      N = 64
// dQ^T has the head dimension on the tensor-memory lanes, so the reducer's
// lane holds one column of dQ for 64 query rows: a warp stages 32 rows x 32
// columns at a time and adds them with one TMA tensor reduction.
//
// 16 warps: warp 0 TMA producer (K_j, V_j once; per Q tile Q_i with LSE_i and
// dO_i with D_i, two slots each); warp 1 MMA issuer; warps 4-7 and 8-11 the
// softmax warpgroups (thread = key row, queries 0..31 and 32..63 of each step;
// warpgroup 0 first copies K_j into tensor memory); warps 12-15 the dQ
// reducer (thread = head-dimension column).
// Shared memory: K_j, V_j, Q_i[2] with LSE_i, dO_i[2] with D_i, the dS^T tile
// and the reducer's staging (4 KB per warp): 231,584 bytes.
// MMA order per step s: dV(s), S^T(s+1), dP^T(s+1), dK(s), dQ^T(s). MMAs
// issued by one thread execute in issue order, so S^T(s+1) overwrites P^T(s)
// after dV(s) has read it. dP^T(s+1) goes out as soon as the softmax warps
// have read dP^T(s) (they announce dS^T(s) after that), ahead of dK(s) and
// dQ^T(s): the softmax warps form dS^T(s+1) while those run, and write it into
// the shared tile once dK(s) and dQ^T(s) have read dS^T(s) (ds_empty).
#include <math.h>

#include "fa_internal.h"
#include "ptx.cuh"
#include "tile_store.cuh"

namespace fa {
namespace {

constexpr int kThreads = 512;
constexpr int kD = 128;
constexpr int kChunkBytes = kTile * 128;     // 128 rows x 128 bytes
constexpr int kTileBytes = 2 * kChunkBytes;  // a 128 x 128 16-bit tile (K_j, V_j)
constexpr int kStep = 64;                    // queries per step
constexpr int kHalfChunk = kStep * 128;      // 64 rows x 128 bytes
constexpr int kHalfBytes = 2 * kHalfChunk;   // 64 rows of Q or dO (16 KB)
constexpr int kQSlots = 4, kdOSlots = 3, kdSBufs = 2;
constexpr int kKOff = 0;
constexpr int kVOff = kKOff + kTileBytes;
constexpr int kQOff = kVOff + kTileBytes;                  // Q half-tiles
constexpr int kdOOff = kQOff + kQSlots * kHalfBytes;       // dO half-tiles
constexpr int kdSOff = kdOOff + kdOSlots * kHalfBytes;     // dS^T buffers: 128 keys x 64 queries
constexpr int kStageOff = kdSOff + kdSBufs * kTile * 128;  // the reducer's 4 KB per warp
constexpr int kLseOff = kStageOff + 4 * 4096;              // [kQSlots][64] LSE * log2(e)
constexpr int kDeltaOff = kLseOff + kQSlots * kStep * 4;   // [kdOSlots][64] D
constexpr int kBarOff = kDeltaOff + kdOSlots * kStep * 4;
constexpr int kNumBars = 1 + 2 * kQSlots + 2 * kdOSlots + 10 + kdSBufs;
constexpr int kMiscOff = kBarOff + kNumBars * 8;
constexpr int kBytes = kMiscOff + 16;
static_assert(kBytes <= 232448, "shared memory budget");
constexpr uint32_t kColK = 0, kColS = 64, kColDP = 128, kColDV = 192, kColDK = 320, kColDQ = 448;

struct Bars {
  uint32_t base;
  __device__ uint32_t kv_full() const { return base; }
  __device__ uint32_t q_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t q_empty(int s) const { return base + 8 * (1 + kQSlots + s); }
  __device__ uint32_t do_full(int s) const { return base + 8 * (1 + 2 * kQSlots + s); }
  __device__ uint32_t do_empty(int s) const { return base + 8 * (1 + 2 * kQSlots + kdOSlots + s); }
  static constexpr int kX = 1 + 2 * kQSlots + 2 * kdOSlots;
  __device__ uint32_t s_full() const { return base + 8 * (kX + 0); }
  __device__ uint32_t p_full() const { return base + 8 * (kX + 1); }
  __device__ uint32_t dp_full() const { return base + 8 * (kX + 2); }
  __device__ uint32_t ds_full() const { return base + 8 * (kX + 3); }
  __device__ uint32_t dq_full() const { return base + 8 * (kX + 4); }
  __device__ uint32_t dq_free() const { return base + 8 * (kX + 5); }
  __device__ uint32_t k_tmem() const { return base + 8 * (kX + 6); }  // K_j is in tensor memory
  __device__ uint32_t acc_done() const { return base + 8 * (kX + 7); }
  __device__ uint32_t teardown() const { return base + 8 * (kX + 8); }
  __device__ uint32_t spare() const { return base + 8 * (kX + 9); }
  // dK and dQ^T have read dS^T buffer b
  __device__ uint32_t ds_empty(int b) const { return base + 8 * (kX + 10 + b); }
};

enum Role : uint32_t { kRoleLoad = 1, kRoleMma = 2, kRoleSoftmax = 3, kRoleInit = 5 };

__device__ __forceinline__ int next_q(const Shape &sh, int i, int j) {
  if (sh.mask)
    while (i < sh.tq && sh.mask[(size_t)i * sh.tk + j] == 0) ++i;
  return i;
}

__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t &a, uint32_t &b, uint32_t &c,
                                             uint32_t &d) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
               : "r"(addr)
               : "memory");
}

// Adds the 32 x 32 fp32 box at `src` (shared memory, 128-byte swizzle) into
// the map's tensor at column x, row y: a TMA tensor reduction performed in L2.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap *tm, uint32_t src, int x,
                                                  int y) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];"
      ::"l"(reinterpret_cast<uint64_t>(tm)), "r"(src), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void st_shared_b32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Rows 128 i + 64 hs .. + 63 of Q with their LSE * log2(e) into Q slot s.
__device__ __forceinline__ void load_qh(const BwdParams &p, const Bars &bars, int s, int i, int hs,
                                        uint32_t s_base, size_t stat_head, int h_idx, int b_idx) {
  mbar_arrive_expect_tx(bars.q_full(s), kHalfBytes + kStep * 4);
  for (int c = 0; c < 2; ++c)
    tma_load_4d(s_base + kQOff + s * kHalfBytes + c * kHalfChunk, &p.tm_qh, c * 64,
                i * kTile + hs * kStep, h_idx, b_idx, bars.q_full(s));
  bulk_load_1d(s_base + kLseOff + s * kStep * 4,
               p.lse2 + stat_head + (size_t)i * kTile + hs * kStep, kStep * 4, bars.q_full(s));
}

// The same rows of dO with their D into dO slot s.
__device__ __forceinline__ void load_doh(const BwdParams &p, const Bars &bars, int s, int i, int hs,
                                         uint32_t s_base, size_t stat_head, int h_idx, int b_idx) {
  mbar_arrive_expect_tx(bars.do_full(s), kHalfBytes + kStep * 4);
  for (int c = 0; c < 2; ++c)
    tma_load_4d(s_base + kdOOff + s * kHalfBytes + c * kHalfChunk, &p.tm_doh, c * 64,
                i * kTile + hs * kStep, h_idx, b_idx, bars.do_full(s));
  bulk_load_1d(s_base + kDeltaOff + s * kStep * 4,
               p.delta + stat_head + (size_t)i * kTile + hs * kStep, kStep * 4, bars.do_full(s));
}

template <bool kF16>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_fused_q64(const __grid_constant__ BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t s_base = smem_u32(smem);
  int *misc = reinterpret_cast<int *>(smem + kMiscOff);  // [0] tmem [2] abort
  if (s_base & 1023u) {  // the 128-byte swizzle needs 1024-byte aligned tiles
    if (threadIdx.x == 0 && p.status)
      atomicCAS(p.status, 0u, status_code(kKernBwdFused, kRoleInit, 2));
    return;
  }
  const uint32_t sK = s_base + kKOff, sV = s_base + kVOff;
  const uint32_t sQ = s_base + kQOff, sdO = s_base + kdOOff, sdS = s_base + kdSOff;
  // slots and buffers of step s
  auto q_slot = [](int s) { return s % kQSlots; };
  auto do_slot = [](int s) { return s % kdOSlots; };
  const float *lse_s = reinterpret_cast<const float *>(smem + kLseOff);
  const float *delta_s = reinterpret_cast<const float *>(smem + kDeltaOff);
  Bars bars{s_base + kBarOff};
  StatusSlot st{p.status, &misc[2], p.wait_limit_ns};

  const int warp = threadIdx.x >> 5;
  const Shape &sh = p.sh;
  const int T = sh.tq;
  // CTA order as in the other backward kernels: head groups, heavy K/V tiles first
  const int hg = p.head_group;
  const int group = blockIdx.x / (hg * sh.tk);
  const int g_base = group * hg;
  const int g_size = min(hg, sh.bh - g_base);
  const int g_rank = blockIdx.x - group * hg * sh.tk;
  const int j = g_rank / g_size;
  const int bh = g_base + g_rank % g_size;
  const int b_idx = bh / sh.heads, h_idx = bh % sh.heads;
  const int first = next_q(sh, sh.first_q_tile(j), j);
  const bool any = first < T;
  const size_t stat_head = (size_t)bh * T * kTile;

  if (warp == 0 && (threadIdx.x & 31) == 0) {
    mbar_init(bars.kv_full(), 1);
    for (int s = 0; s < kQSlots; ++s) {
      mbar_init(bars.q_full(s), 1);
      mbar_init(bars.q_empty(s), 1);
    }
    // a dO slot is free once dV of its step has read it (one commit) and the
    // softmax warps have read D (256 threads)
    for (int s = 0; s < kdOSlots; ++s) {
      mbar_init(bars.do_full(s), 1);
      mbar_init(bars.do_empty(s), 257);
    }
    for (int b = 0; b < kdSBufs; ++b) mbar_init(bars.ds_empty(b), 1);
    mbar_init(bars.s_full(), 1);
    mbar_init(bars.p_full(), 256);
    mbar_init(bars.dp_full(), 1);
    mbar_init(bars.ds_full(), 256);
    mbar_init(bars.dq_full(), 1);
    mbar_init(bars.dq_free(), 128);
    mbar_init(bars.k_tmem(), 128);
    mbar_init(bars.acc_done(), 1);
    mbar_init(bars.teardown(), 1);
    mbar_init(bars.spare(), 1);
    misc[2] = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tm_qh);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
    tma_prefetch_desc(&p.tm_doh);
    tma_prefetch_desc(&p.tm_dqacc);
    if (any && !(p.debug_flags & kDebugSkipLoads)) {
      mbar_arrive_expect_tx(bars.kv_full(), 2 * kTileBytes);
      for (int c = 0; c < 2; ++c) {
        tma_load_4d(sK + c * kChunkBytes, &p.tm_k, c * 64, j * kTile, h_idx, b_idx, bars.kv_full());
        tma_load_4d(sV + c * kChunkBytes, &p.tm_v, c * 64, j * kTile, h_idx, b_idx, bars.kv_full());
      }
      load_qh(p, bars, 0, first, 0, s_base, stat_head, h_idx, b_idx);
      load_doh(p, bars, 0, first, 0, s_base, stat_head, h_idx, b_idx);
    }
  } else if (warp == 1) {
    tmem_alloc(smem_u32(&misc[0]), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);

  if (warp == 0) {
    // ---- TMA producer: Q and dO half-tiles, one per step ------------------------
    if (elect_one() && any && !(p.debug_flags & kDebugSkipLoads)) {
      int nq = 1, ndo = 1;  // halves issued: the first step's came with the set-up
      bool ok = true;
      for (int i = first; i < T && ok; i = next_q(sh, i + 1, j)) {
        for (int hs = (i == first ? 1 : 0); hs < 2 && ok; ++hs) {
          const int qs = nq % kQSlots;
          ok = mbar_wait(bars.q_empty(qs), ((nq / kQSlots) & 1u) ^ 1u, st,
                         status_code(kKernBwdFused, kRoleLoad, 1));
          if (!ok) break;
          load_qh(p, bars, qs, i, hs, s_base, stat_head, h_idx, b_idx);
          ++nq;
          const int ds = ndo % kdOSlots;
          ok = mbar_wait(bars.do_empty(ds), ((ndo / kdOSlots) & 1u) ^ 1u, st,
                         status_code(kKernBwdFused, kRoleLoad, 4));
          if (!ok) break;
          load_doh(p, bars, ds, i, hs, s_base, stat_head, h_idx, b_idx);
          ++ndo;
        }
      }
      // teardown: every copy issued has landed
      mbar_wait_drain(bars.kv_full(), 0, st, status_code(kKernBwdFused, kRoleLoad, 2));
      for (int s = 0; s < kQSlots && s < nq; ++s) {
        const int last = s + ((nq - 1 - s) / kQSlots) * kQSlots;
        mbar_wait_drain(bars.q_full(s), (last / kQSlots) & 1u, st,
                        status_code(kKernBwdFused, kRoleLoad, 3));
      }
      for (int s = 0; s < kdOSlots && s < ndo; ++s) {
        const int last = s + ((ndo - 1 - s) / kdOSlots) * kdOSlots;
        mbar_wait_drain(bars.do_full(s), (last / kdOSlots) & 1u, st,
                        status_code(kKernBwdFused, kRoleLoad, 5));
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- tcgen05 issuer ----------------------------------------------------
    if (elect_one()) {
      constexpr uint32_t kIdS = idesc_f32acc(kTile, 64, 0, 0, kF16);    // S^T, dP^T
      constexpr uint32_t kIdAcc = idesc_f32acc(kTile, kD, 0, 1, kF16);   // dV, dK: B MN-major
      constexpr uint32_t kIdDq = idesc_f32acc(kD, 64, 1, 1, kF16);       // dQ^T: A, B MN-major
      bool ok = !any || (mbar_wait(bars.kv_full(), 0, st, status_code(kKernBwdFused, kRoleMma, 1)) &&
                         mbar_wait(bars.k_tmem(), 0, st, status_code(kKernBwdFused, kRoleMma, 11)));
      // S^T = K Q^T over a step's 64 queries (Q slot qs): A = K in tensor
      // memory (8 columns per 16-element K-step), B = the Q rows (K-major)
      auto issue_s = [&](int qs) {
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_f16kind_ts(tmem + kColS, tmem + kColK + kk * 8,
                         sdesc_sw128(sQ + qs * kHalfBytes + (kk >> 2) * kHalfChunk + (kk & 3) * 32,
                                     16, 1024),
                         kIdS, kk > 0);
      };
      // dP^T = V dO^T over a step's 64 queries (dO slot ds): both K-major
      auto issue_dp = [&](int ds) {
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_f16kind_ss(tmem + kColDP,
                         sdesc_sw128(sV + (kk >> 2) * kChunkBytes + (kk & 3) * 32, 16, 1024),
                         sdesc_sw128(sdO + ds * kHalfBytes + (kk >> 2) * kHalfChunk + (kk & 3) * 32,
                                     16, 1024),
                         kIdS, kk > 0);
      };
      // dV += P^T dO: P^T packed in tensor memory (queries 32h.. of the step
      // at kColS + 32h), dO rows of the step's slot (MN-major, 16 per K-step)
      auto issue_dv = [&](int ds, bool first_step) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f16kind_ts(tmem + kColDV, tmem + kColS + (kk >> 1) * 32 + (kk & 1) * 8,
                         sdesc_sw128(sdO + ds * kHalfBytes + kk * 2048, kHalfChunk, 1024), kIdAcc,
                         (!first_step || kk > 0) ? 1u : 0u);
      };
      // dK += dS^T Q: A = dS^T buffer b (K-major: rows = keys), B = the Q rows
      // of the step's slot (MN-major)
      auto issue_dk = [&](int b, int qs, bool first_step) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f16kind_ss(tmem + kColDK, sdesc_sw128(sdS + b * kChunkBytes + kk * 32, 16, 1024),
                         sdesc_sw128(sQ + qs * kHalfBytes + kk * 2048, kHalfChunk, 1024), kIdAcc,
                         (!first_step || kk > 0) ? 1u : 0u);
      };
      // dQ^T = K^T dS^T: A = K_j read MN-major (M = head dimension along a
      // row, K = keys down the rows), B = dS^T buffer b (N = 64 queries along
      // a row, K = keys)
      auto issue_dq = [&](int b) {
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_f16kind_ss(tmem + kColDQ, sdesc_sw128(sK + kk * 2048, kChunkBytes, 1024),
                         sdesc_sw128(sdS + b * kChunkBytes + kk * 2048, kChunkBytes, 1024), kIdDq,
                         kk > 0);
      };
      if (ok && any) {
        ok = mbar_wait(bars.q_full(0), 0, st, status_code(kKernBwdFused, kRoleMma, 2));
        if (ok) {
          tc_fence_after();
          issue_s(0);
          mma_commit(bars.s_full());
          ok = mbar_wait(bars.do_full(0), 0, st, status_code(kKernBwdFused, kRoleMma, 7));
        }
        if (ok) {
          tc_fence_after();
          issue_dp(0);
          mma_commit(bars.dp_full());
        }
      }
      int s = 0;  // steps: 64 queries each, two per Q tile
      for (int i = first; i < T && ok;) {
        const int inext = next_q(sh, i + 1, j);
        for (int hs = 0; hs < 2 && ok; ++hs, ++s) {
          const bool more = hs == 0 || inext < T;  // a step s + 1 follows
          const int b = s & 1;                     // dS^T buffer of step s
          ok = mbar_wait(bars.p_full(), s & 1, st, status_code(kKernBwdFused, kRoleMma, 3));
          if (!ok) break;
          tc_fence_after();
          issue_dv(do_slot(s), s == 0);
          mma_commit(bars.do_empty(do_slot(s)));  // dP^T(s) and dV(s) are done with dO
          if (more) {
            ok = mbar_wait(bars.q_full(q_slot(s + 1)), ((s + 1) / kQSlots) & 1, st,
                           status_code(kKernBwdFused, kRoleMma, 4));
            if (!ok) break;
            tc_fence_after();
            issue_s(q_slot(s + 1));
            mma_commit(bars.s_full());
          }
          ok = mbar_wait(bars.ds_full(), s & 1, st, status_code(kKernBwdFused, kRoleMma, 5));
          if (!ok) break;
          tc_fence_after();
          // the softmax warps have read dP^T(s): dP^T(s+1) may take its columns
          if (more) {
            ok = mbar_wait(bars.do_full(do_slot(s + 1)), ((s + 1) / kdOSlots) & 1, st,
                           status_code(kKernBwdFused, kRoleMma, 7));
            if (!ok) break;
            tc_fence_after();
            issue_dp(do_slot(s + 1));
            mma_commit(bars.dp_full());
          }
          issue_dk(b, q_slot(s), s == 0);
          mma_commit(bars.q_empty(q_slot(s)));  // S^T(s) and dK(s) are done with Q
          if (s > 0) {  // the reducer has read dQ^T(s-1)
            ok = mbar_wait(bars.dq_free(), (s - 1) & 1, st, status_code(kKernBwdFused, kRoleMma, 10));
            if (!ok) break;
            tc_fence_after();
          }
          issue_dq(b);
          mma_commit(bars.dq_full());
          mma_commit(bars.ds_empty(b));  // dK(s) and dQ^T(s) have read dS^T buffer b
        }
        i = inext;
      }
      if (ok) mma_commit(bars.acc_done());
      mma_commit(bars.teardown());
      mbar_wait_drain(bars.teardown(), 0, st, status_code(kKernBwdFused, kRoleMma, 8));
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 12) {
    // ---- K_j into tensor memory, then P^T and dS^T (thread = key row) ----------
    const int h = (warp - 4) >> 2;       // queries 32h..32h+31 of each step
    const int kr = threadIdx.x & 127;    // key row = TMEM lane
    const uint32_t t = tmem + (uint32_t((warp & 3) * 32) << 16);
    const float c = p.scale_log2;
    bool ok = true;
    if (h == 0 && any) {
      // row kr of K_j as 16-bit pairs: chunk cc holds the head-dimension
      // columns 64cc.., 16-byte piece u at position u ^ (kr & 7)
      ok = __all_sync(0xffffffffu, mbar_wait(bars.kv_full(), 0, st,
                                             status_code(kKernBwdFused, kRoleSoftmax, 10)));
      if (ok) {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t kw[32];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            ld_shared_v4(sK + cc * kChunkBytes + kr * 128 + ((uint32_t(u) ^ uint32_t(kr & 7)) << 4),
                         kw[4 * u], kw[4 * u + 1], kw[4 * u + 2], kw[4 * u + 3]);
          tmem_st32(t + kColK + 32 * cc, kw);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bars.k_tmem());
      }
    }
    int s = 0;  // steps: 64 queries each, two per Q tile
    for (int i = first; i < T && ok; i = next_q(sh, i + 1, j)) {
      const bool cross = sh.causal && kTile * j + kTile - 1 > kTile * i + sh.causal_off;
      for (int hs = 0; hs < 2 && ok; ++hs, ++s) {
        const int q0 = 64 * hs + 32 * h;  // this warpgroup's first query of the step in Q tile i
        const float *lse2 = lse_s + q_slot(s) * kStep + 32 * h;
        const float *delta = delta_s + do_slot(s) * kStep + 32 * h;
        ok = __all_sync(0xffffffffu, mbar_wait(bars.s_full(), s & 1, st,
                                               status_code(kKernBwdFused, kRoleSoftmax, 1)));
        if (ok)
          ok = __all_sync(0xffffffffu, mbar_wait(bars.q_full(q_slot(s)), (s / kQSlots) & 1, st,
                                                 status_code(kKernBwdFused, kRoleSoftmax, 2)));
        if (!ok) break;
        tc_fence_after();
        // P^T_kq = exp2(s_kq * scale * log2e - LSE_q * log2e) for this
        // warpgroup's 32 queries, packed over its first 16 S^T columns
        float pr[32];
        {
          uint32_t sr[32];
          tmem_ld32(t + kColS + 32 * h, sr);
          tmem_wait_ld();
#pragma unroll
          for (int x = 0; x < 32; ++x)
            pr[x] = ex2_approx(fmaf(__uint_as_float(sr[x]), c, -lse2[x]));
          if (cross) {  // key kr sees query q0 + x only if x >= lo
            const int lo = kTile * (j - i) + kr - sh.causal_off - q0;
#pragma unroll
            for (int x = 0; x < 32; ++x)
              if (x < lo) pr[x] = 0.f;
          }
          uint32_t pk[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) pk[x] = pack2<kF16>(pr[2 * x], pr[2 * x + 1]);
          tmem_st16(t + kColS + 32 * h, pk);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bars.p_full());
        }
        // dS^T_kq = P^T_kq (dP^T_kq - D_q) into dS^T buffer s & 1 (the A
        // operand of dK, the B operand of dQ^T): row kr, queries 32h.. of the
        // step = 16-byte pieces 4h..4h+3
        ok = __all_sync(0xffffffffu, mbar_wait(bars.dp_full(), s & 1, st,
                                               status_code(kKernBwdFused, kRoleSoftmax, 4)));
        if (ok)
          ok = __all_sync(0xffffffffu, mbar_wait(bars.do_full(do_slot(s)), (s / kdOSlots) & 1, st,
                                                 status_code(kKernBwdFused, kRoleSoftmax, 5)));
        if (!ok) break;
        tc_fence_after();
        uint32_t dsp[16];
        {
          uint32_t dr[32];
          tmem_ld32(t + kColDP + 32 * h, dr);
          tmem_wait_ld();
#pragma unroll
          for (int x = 0; x < 32; x += 2)
            dsp[x / 2] = pack2<kF16>(pr[x] * (__uint_as_float(dr[x]) - delta[x]),
                                     pr[x + 1] * (__uint_as_float(dr[x + 1]) - delta[x + 1]));
        }
        // dK(s-2) and dQ^T(s-2) have read the buffer
        if (s >= kdSBufs) {
          ok = __all_sync(0xffffffffu, mbar_wait(bars.ds_empty(s & 1), ((s >> 1) - 1) & 1, st,
                                                 status_code(kKernBwdFused, kRoleSoftmax, 7)));
          if (!ok) break;
        }
        {
          const uint32_t row = sdS + (s & 1) * kChunkBytes + kr * 128;
#pragma unroll
          for (int u = 0; u < 4; ++u)
            st_shared_v4(row + ((uint32_t(4 * h + u) ^ uint32_t(kr & 7)) << 4), dsp[4 * u],
                         dsp[4 * u + 1], dsp[4 * u + 2], dsp[4 * u + 3]);
        }
        fence_proxy_async_smem();  // the tensor core reads dS^T through the async proxy
        tc_fence_before();         // dP^T(s) has been read: dP^T(s+1) may take its columns
        mbar_arrive(bars.ds_full());
        mbar_arrive(bars.do_empty(do_slot(s)));  // D has been read
      }
    }
    // epilogue: warps 4-7 write dV, warps 8-11 write dK (scaled), through the
    // K_j and V_j buffers once every MMA has completed
    if (ok && any)
      ok = __all_sync(0xffffffffu, mbar_wait(bars.acc_done(), 0, st,
                                             status_code(kKernBwdFused, kRoleSoftmax, 6)));
    if (ok) {
      tc_fence_after();
      store_rows_tma<kD, kF16>(h ? &p.tm_dk : &p.tm_dv, t + (h ? kColDK : kColDV), h ? sV : sK,
                               kr, j * kTile, 0, h ? p.scale : 1.f, any, sh.d, sh.nk, h_idx, b_idx);
    }
  } else if (warp >= 12) {
    // ---- dQ reducer (thread = head-dimension column) ---------------------------
    // Lane = column 32qw + lane of dQ; each step's 64 query rows leave in two
    // 32 x 32 boxes staged in this warp's 4 KB (row x at 128 x, 16-byte piece
    // lane / 4 at position (lane / 4) ^ (x & 7): the map's 128-byte swizzle,
    // free of bank conflicts) and added into the accumulator by TMA tensor
    // reductions, which one thread can keep in flight at L2's rate.
    const int qw = warp & 3;
    const int lane = threadIdx.x & 31;
    const uint32_t t = tmem + (uint32_t(qw * 32) << 16);
    const uint32_t slot = s_base + kStageOff + qw * 4096;
    const uint32_t col_off = uint32_t(lane & 3) * 4;
    const int row_base = (int)stat_head;  // this head's first accumulator row
    bool ok = true;
    int s = 0;
    for (int i = first; i < T && ok; i = next_q(sh, i + 1, j)) {
      for (int hs = 0; hs < 2; ++hs, ++s) {
        ok = __all_sync(0xffffffffu, mbar_wait(bars.dq_full(), s & 1, st,
                                               status_code(kKernBwdFused, kRoleSoftmax, 8)));
        if (!ok) break;
        tc_fence_after();
        uint32_t v[2][32];
        tmem_ld32(t + kColDQ, v[0]);
        tmem_ld32(t + kColDQ + 32, v[1]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bars.dq_free());
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          if (lane == 0) bulk_wait_group_read0();  // the slot's previous box has been read
          __syncwarp();
#pragma unroll
          for (int x = 0; x < 32; ++x)
            st_shared_b32(slot + x * 128 + (((uint32_t(lane) >> 2) ^ uint32_t(x & 7)) << 4) + col_off,
                          v[r][x]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_reduce_add_2d(&p.tm_dqacc, slot, 32 * qw, row_base + kTile * i + 64 * hs + 32 * r);
            bulk_commit_group();
          }
        }
      }
    }
    // the CTA's shared memory must outlive the reductions' reads of it
    if (lane == 0) bulk_wait_group_read0();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool kF16>
cudaError_t launch_q64(const BwdParams &p, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(fa_bwd_fused_q64<kF16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  {
    LaunchProbe probe(kKindBwdFused, stream);
    fa_bwd_fused_q64<kF16><<<p.sh.tk * p.sh.bh, kThreads, kBytes, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward_fused_q64(const BwdParams &p, cudaStream_t stream) {
  return p.sh.f16 ? launch_q64<true>(p, stream) : launch_q64<false>(p, stream);
}

}  // namespace fa
