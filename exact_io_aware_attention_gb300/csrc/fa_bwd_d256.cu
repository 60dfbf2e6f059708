// Attention backward for head dimension 256 on sm_103a.
//
// The gradients are those of fa_bwd.cu: the analytic gradients of
// O = softmax(scale QK^T) V, with P recomputed block by block from Q, K and
// the stored LSE (the pages keep only O and the softmax statistics and
// regenerate S and P in the backward pass: "Paper Notes: FlashAttention",
// "Key Ideas"; aicassindra page, "The backward pass: recompute instead of
// store"):
//
//   P_ij = exp(scale s_ij - LSE_i), dV_j = sum_i P_ij dO_i, dP_ij = dO_i . V_j,
//   dS_ij = P_ij (dP_ij - D_i), dQ_i = scale sum_j dS_ij K_j,
//   dK_j = scale sum_i dS_ij Q_i, D_i = dO_i . O_i.
//
// Only the split of the work differs. A 128-row accumulator of 256 fp32
// columns takes half of the 512 tensor-memory columns, so dK and dV cannot
// live in one CTA beside the S^T and dP^T tiles, and a 128 x 256 tile of 16-bit
// elements is 64 KB of shared memory. Three kernels follow fa_bwd_pre on the
// caller's stream, each owning its output tile (no cross-CTA reduction):
//
//   fa_bwd256_dv            CTA = one 128-key K/V tile, looping over the Q
//                           tiles that see it: S^T = K Q_i^T,
//                           P^T = exp2(S^T scale log2e - LSE_i log2e),
//                           dV += P^T dO_i
//   fa_bwd256_grad<true>    CTA = one 128-key tile: S^T = K Q_i^T,
//                           dP^T = V dO_i^T, dS^T = P^T (dP^T - D_i),
//                           dK += dS^T Q_i
//   fa_bwd256_grad<false>   CTA = one 128-row Q tile, looping over its K/V
//                           tiles: S = Q K_j^T, dP = dO V_j^T,
//                           dS = P (dP - D), dQ += dS K_j
//
// The CTA's own 128 x 256 operands stay in shared memory; the other tiles
// stream through a ring of 32 KB slots, each holding 128 columns (one half)
// of a 128-row tile, in the order the MMAs consume them. A streamed tile that
// is needed twice in a step (Q_i for S^T and dK, K_j for S and dQ) is loaded
// twice: the ring has no room to keep it, and the second copy comes from L2.
// S^T is recomputed by fa_bwd256_dv and fa_bwd256_grad<true>, so the kernels
// execute 8 of the method's GEMM units where it counts 5 (d <= 128: 7).
//
// Rows past the end of a sequence arrive as zeros; a missing query row has
// LSE log2e = +inf in the workspace, so its P is exactly 0; keys past the end
// and keys above the causal boundary are masked element-wise where a tile
// needs it; a missing key row only feeds its own dK/dV row, which is not
// stored.
#include <math.h>

#include "fa_internal.h"
#include "ptx.cuh"
#include "tile_store.cuh"

namespace fa {
namespace {

constexpr int kThreads = 384;
constexpr int kChunkBytes = kTile * 128;     // 128 rows x 64 columns of 16-bit elements
constexpr int kTileBytes = 4 * kChunkBytes;  // 128 rows x 256 columns
constexpr int kHalfBytes = 2 * kChunkBytes;  // 128 rows x 128 columns: one ring slot

enum Role : uint32_t { kRoleLoad = 1, kRoleMma = 2, kRoleSoftmax = 3, kRoleInit = 5 };

// Tensor-memory column of the packed A operand (P^T, dS^T or dS) for MMA
// step kk (columns 16kk..16kk+15 of the 128 x 128 tile): the warpgroup that
// owns columns 64h..64h+63 packs them at column 64h.
__device__ __forceinline__ uint32_t packed_col(int kk) { return (kk >> 2) * 64 + (kk & 3) * 8; }

// Next Q tile at or after i that the block mask lets see K/V tile j (tq if none).
__device__ __forceinline__ int next_q(const Shape &sh, int i, int j) {
  if (sh.mask)
    while (i < sh.tq && sh.mask[(size_t)i * sh.tk + j] == 0) ++i;
  return i;
}

// Next K/V tile at or after j, up to jmax, that the block mask lets Q tile i
// see (tk if none).
__device__ __forceinline__ int next_k(const Shape &sh, int i, int j, int jmax) {
  while (j <= jmax && !sh.mask_allows(i, j)) ++j;
  return j <= jmax ? j : sh.tk;
}

// Half h (columns 128h .. 128h+127) of rows row .. row+127 of one head.
__device__ __forceinline__ void load_half(uint32_t dst, const CUtensorMap *tm, int h, int row,
                                          int h_idx, int b_idx, uint32_t bar) {
  for (int c = 0; c < 2; ++c)
    tma_load_4d(dst + c * kChunkBytes, tm, h * 128 + c * 64, row, h_idx, b_idx, bar);
}

// D (128 x 128 fp32 at d_tmem) (+)= A[:, 128h .. 128h+127] B^T: A is a
// resident 128 x 256 tile, B one ring slot (128 rows x 128 columns); both
// K-major, 8 k-steps of 16 columns.
__device__ __forceinline__ void mma_half_ss(uint32_t d_tmem, uint32_t a, uint32_t b, int h,
                                            uint32_t idesc, bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
    mma_f16kind_ss(d_tmem, sdesc_sw128(a + h * kHalfBytes + off, 16, 1024),
                   sdesc_sw128(b + off, 16, 1024), idesc, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// D (128 x 128 fp32 at d_tmem) (+)= E B: E is a 128 x 128 tile of packed
// 16-bit pairs in tensor memory at e_tmem (packed_col layout), B one ring
// slot with its 128 rows as the reduction dimension (MN-major, 16 rows per
// k-step).
__device__ __forceinline__ void mma_half_ts(uint32_t d_tmem, uint32_t e_tmem, uint32_t b,
                                            uint32_t idesc, bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_f16kind_ts(d_tmem, e_tmem + packed_col(kk), sdesc_sw128(b + kk * 2048, kChunkBytes, 1024),
                   idesc, (accumulate || kk > 0) ? 1u : 0u);
}

// ---------------------------------------------------------------------------
// fa_bwd256_dv, 12 warps:
//   warp 0      TMA producer: K_j once; per step LSE_i log2e (2 stages), and the
//               halves of Q_i and dO_i through a ring of 5 slots in the order
//               Q_0, Q_1, dO_0, Q_2, dO_1, Q_3, ...
//   warp 1      tcgen05 issuer (one lane) and tensor-memory owner
//   warps 4-7   thread = key row: P^T for queries 0..63 of each Q tile
//   warps 8-11  thread = key row: P^T for queries 64..127; then both
//               warpgroups store dV (128 columns each)
// Tensor memory: S^T in two buffers [0,128) and [128,256), dV in [256,512).
// P^T (16-bit pairs) goes over the first 32 of each warpgroup's 64 S^T
// columns. MMA order: S^T(0), S^T(1), then per step n: dV += P^T(n) dO(n),
// S^T(n+2) (into the buffer of n, after the MMA that reads P^T(n)).
struct DvLayout {
  static constexpr int kSlots = 5;
  static constexpr int kKOff = 0;
  static constexpr int kRingOff = kTileBytes;
  static constexpr int kStatOff = kRingOff + kSlots * kHalfBytes;  // [2 stages][128] LSE log2e
  static constexpr int kStatBytes = kTile * 4;
  static constexpr int kBarOff = kStatOff + 2 * kStatBytes;
  // k_full, full[5], empty[5], x_full[2], p_full[2], stat_full[2], stat_empty[2],
  // acc_done, teardown
  static constexpr int kNumBars = 1 + 2 * kSlots + 2 + 2 + 2 + 2 + 2;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  static_assert(kBytes <= 232448, "shared memory budget");
  static constexpr uint32_t kColAcc = 256;
};

struct DvBars {
  uint32_t base;
  __device__ uint32_t k_full() const { return base; }
  __device__ uint32_t full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t empty(int s) const { return base + 8 * (6 + s); }
  __device__ uint32_t x_full(int b) const { return base + 8 * (11 + b); }
  __device__ uint32_t p_full(int b) const { return base + 8 * (13 + b); }
  __device__ uint32_t stat_full(int b) const { return base + 8 * (15 + b); }
  __device__ uint32_t stat_empty(int b) const { return base + 8 * (17 + b); }
  __device__ uint32_t acc_done() const { return base + 8 * 19; }
  __device__ uint32_t teardown() const { return base + 8 * 20; }
};

template <bool kF16>
__global__ void __launch_bounds__(kThreads, 1) fa_bwd256_dv(const __grid_constant__ BwdParams p) {
  using L = DvLayout;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t s_base = smem_u32(smem);
  int *misc = reinterpret_cast<int *>(smem + L::kMiscOff);  // [0] tmem [2] abort [3] loads in set-up
  // the 128-byte swizzle needs 1024-byte aligned tiles; the layout has no
  // room for alignment slack, so a misaligned base is reported
  if (s_base & 1023u) {
    if (threadIdx.x == 0 && p.status) atomicCAS(p.status, 0u, status_code(kKernBwd256Dv, kRoleInit, 1));
    return;
  }
  const uint32_t sK = s_base + L::kKOff, sRing = s_base + L::kRingOff;
  const float *stat = reinterpret_cast<const float *>(smem + L::kStatOff);
  DvBars bars{s_base + L::kBarOff};
  StatusSlot st{p.status, &misc[2], p.wait_limit_ns};
  const int warp = threadIdx.x >> 5;

  // CTA order as in fa_bwd_dkdv: head groups of p.head_group heads, heavy
  // (early, under causal masking) key tiles first within a group
  const Shape &sh = p.sh;
  const int T = sh.tq;
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
    mbar_init(bars.k_full(), 1);
    for (int s = 0; s < L::kSlots; ++s) {
      mbar_init(bars.full(s), 1);
      mbar_init(bars.empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.x_full(b), 1);
      mbar_init(bars.p_full(b), 256);
      mbar_init(bars.stat_full(b), 1);
      mbar_init(bars.stat_empty(b), 256);
    }
    mbar_init(bars.acc_done(), 1);
    mbar_init(bars.teardown(), 1);
    misc[2] = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_do);
    // K_j and the operands of the first two S^T (LSE log2e, both Q halves)
    // depend on blockIdx only: load them now, while the other warps set up
    int pre = 0;
    if (any && !(p.debug_flags & kDebugSkipLoads)) {
      mbar_arrive_expect_tx(bars.k_full(), kTileBytes);
      for (int c = 0; c < 4; ++c)
        tma_load_4d(sK + c * kChunkBytes, &p.tm_k, c * 64, j * kTile, h_idx, b_idx, bars.k_full());
      for (int i = first; i < T && pre < 2; i = next_q(sh, i + 1, j), ++pre) {
        mbar_arrive_expect_tx(bars.stat_full(pre), L::kStatBytes);
        bulk_load_1d(s_base + L::kStatOff + pre * L::kStatBytes, p.lse2 + stat_head + (size_t)i * kTile,
                     L::kStatBytes, bars.stat_full(pre));
        for (int h = 0; h < 2; ++h) {  // ring positions 2 pre + h
          mbar_arrive_expect_tx(bars.full(2 * pre + h), kHalfBytes);
          load_half(sRing + (2 * pre + h) * kHalfBytes, &p.tm_q, h, i * kTile, h_idx, b_idx,
                    bars.full(2 * pre + h));
        }
      }
    }
    misc[3] = pre;  // S^T steps whose operands were issued during set-up
  } else if (warp == 1) {
    tmem_alloc(smem_u32(&misc[0]), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);

  if (warp == 0) {
    // ---- TMA producer ------------------------------------------------------
    if (elect_one() && any && !(p.debug_flags & kDebugSkipLoads)) {
      bool ok = true;
      int issued = 0;  // ring position of the next half
      int nst = 0;     // statistics stages issued
      auto ring_load = [&](const CUtensorMap *tm, int i, int h) {
        if (!ok) return;
        const int s = issued % L::kSlots;
        ok = mbar_wait(bars.empty(s), ((issued / L::kSlots) & 1u) ^ 1u, st,
                       status_code(kKernBwd256Dv, kRoleLoad, 1));
        if (!ok) return;
        mbar_arrive_expect_tx(bars.full(s), kHalfBytes);
        load_half(sRing + s * kHalfBytes, tm, h, i * kTile, h_idx, b_idx, bars.full(s));
        ++issued;
      };
      // step nst's LSE log2e, then both halves of Q_i (already issued during
      // set-up for the first misc[3] steps)
      const int pre = misc[3];
      auto load_x = [&](int i) {
        if (nst < pre) {
          ++nst;
          issued += 2;
          return;
        }
        const int b = nst & 1;
        ok = ok && mbar_wait(bars.stat_empty(b), ((nst >> 1) & 1u) ^ 1u, st,
                             status_code(kKernBwd256Dv, kRoleLoad, 2));
        if (!ok) return;
        mbar_arrive_expect_tx(bars.stat_full(b), L::kStatBytes);
        bulk_load_1d(s_base + L::kStatOff + b * L::kStatBytes, p.lse2 + stat_head + (size_t)i * kTile,
                     L::kStatBytes, bars.stat_full(b));
        ++nst;
        ring_load(&p.tm_q, i, 0);
        ring_load(&p.tm_q, i, 1);
      };
      int ix = first;  // Q tile of the next S^T
      load_x(ix);
      ix = next_q(sh, ix + 1, j);
      if (ix < T) {
        load_x(ix);
        ix = next_q(sh, ix + 1, j);
      }
      for (int i = first; i < T && ok; i = next_q(sh, i + 1, j)) {
        ring_load(&p.tm_do, i, 0);
        ring_load(&p.tm_do, i, 1);
        if (ix < T) {
          load_x(ix);
          ix = next_q(sh, ix + 1, j);
        }
      }
      // teardown: every copy issued has landed
      mbar_wait_drain(bars.k_full(), 0, st, status_code(kKernBwd256Dv, kRoleLoad, 3));
      for (int s = 0; s < L::kSlots && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / L::kSlots) * L::kSlots;
        mbar_wait_drain(bars.full(s), (last / L::kSlots) & 1u, st, status_code(kKernBwd256Dv, kRoleLoad, 4));
      }
      for (int b = 0; b < 2 && b < nst; ++b) {
        const int last = b + ((nst - 1 - b) / 2) * 2;
        mbar_wait_drain(bars.stat_full(b), (last >> 1) & 1u, st, status_code(kKernBwd256Dv, kRoleLoad, 5));
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- tcgen05 issuer ----------------------------------------------------
    if (elect_one()) {
      constexpr uint32_t kIdX = idesc_f32acc(kTile, kTile, 0, 0, kF16);    // S^T: K-major
      constexpr uint32_t kIdAcc = idesc_f32acc(kTile, kTile, 0, 1, kF16);  // dV half: dO MN-major
      bool ok = !any || mbar_wait(bars.k_full(), 0, st, status_code(kKernBwd256Dv, kRoleMma, 1));
      int pos = 0;  // ring position of the next half
      // the next ring slot once its copy has landed, or -1
      auto next_slot = [&](uint32_t site) -> int {
        const int s = pos % L::kSlots;
        if (!mbar_wait(bars.full(s), (pos / L::kSlots) & 1u, st,
                       status_code(kKernBwd256Dv, kRoleMma, site)))
          return -1;
        tc_fence_after();
        return s;
      };
      // S^T(n) = K Q^T into buffer b: 8 k-steps per Q half
      auto issue_x = [&](int b) -> bool {
        for (int h = 0; h < 2; ++h) {
          const int s = next_slot(2);
          if (s < 0) return false;
          mma_half_ss(tmem + b * kTile, sK, sRing + s * kHalfBytes, h, kIdX, h > 0);
          mma_commit(bars.empty(s));
          ++pos;
        }
        mma_commit(bars.x_full(b));
        return true;
      };
      if (ok && any) {
        int ix = first;
        ok = issue_x(0);
        ix = next_q(sh, ix + 1, j);
        if (ok && ix < T) {
          ok = issue_x(1);
          ix = next_q(sh, ix + 1, j);
        }
        int n = 0;
        for (int i = first; i < T && ok; i = next_q(sh, i + 1, j), ++n) {
          const int b = n & 1;
          ok = mbar_wait(bars.p_full(b), (n >> 1) & 1u, st, status_code(kKernBwd256Dv, kRoleMma, 3));
          if (!ok) break;
          tc_fence_after();
          // dV[:, 128h ..] += P^T(n) dO_i[:, 128h ..]
          for (int h = 0; h < 2 && ok; ++h) {
            const int s = next_slot(4);
            if (s < 0) {
              ok = false;
              break;
            }
            mma_half_ts(tmem + L::kColAcc + h * kTile, tmem + b * kTile, sRing + s * kHalfBytes,
                        kIdAcc, n > 0);
            mma_commit(bars.empty(s));
            ++pos;
          }
          if (ok && ix < T) {
            ok = issue_x(b);
            ix = next_q(sh, ix + 1, j);
          }
        }
      }
      if (ok && any) mma_commit(bars.acc_done());
      mma_commit(bars.teardown());
      mbar_wait_drain(bars.teardown(), 0, st, status_code(kKernBwd256Dv, kRoleMma, 8));
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---- P^T for one half of the queries (thread = key row) ------------------
    const int h = (warp - 4) >> 2;                 // queries 64h .. 64h+63
    const int kr = threadIdx.x & 127;              // key row = TMEM lane
    const uint32_t t = tmem + (uint32_t((warp & 3) * 32) << 16);
    const float c = p.scale_log2;
    bool ok = true;
    int n = 0;
    for (int i = first; i < T && ok; i = next_q(sh, i + 1, j), ++n) {
      const int b = n & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(bars.x_full(b), (n >> 1) & 1u, st,
                                             status_code(kKernBwd256Dv, kRoleSoftmax, 1)));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bars.stat_full(b), (n >> 1) & 1u, st,
                                                     status_code(kKernBwd256Dv, kRoleSoftmax, 2)));
      if (!ok) break;
      tc_fence_after();
      const float *lse2 = stat + b * kTile + 64 * h;
      float pr[64];
      {
        // both loads in flight before the one wait
        uint32_t sr[2][32];
        tmem_ld32(t + b * kTile + 64 * h, sr[0]);
        tmem_ld32(t + b * kTile + 64 * h + 32, sr[1]);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 64; ++x)
          pr[x] = ex2_approx(fmaf(__uint_as_float(sr[x >> 5][x & 31]), c, -lse2[x]));
      }
      // only on a tile that the causal boundary crosses: key kr sees query
      // 64h + x only if x >= lo
      if (sh.causal && kTile * j + kTile - 1 > kTile * i + sh.causal_off) {
        const int lo = kTile * (j - i) + kr - sh.causal_off - 64 * h;
#pragma unroll
        for (int x = 0; x < 64; ++x)
          if (x < lo) pr[x] = 0.f;
      }
      uint32_t pk[32];
#pragma unroll
      for (int x = 0; x < 32; ++x) pk[x] = pack2<kF16>(pr[2 * x], pr[2 * x + 1]);
      // P^T over the first 32 of this warpgroup's S^T columns (already read)
      tmem_st32(t + b * kTile + 64 * h, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bars.stat_empty(b));
      mbar_arrive(bars.p_full(b));
    }
    if (ok && any)
      ok = __all_sync(0xffffffffu, mbar_wait(bars.acc_done(), 0, st,
                                             status_code(kKernBwd256Dv, kRoleSoftmax, 3)));
    // dV, 128 columns per warpgroup, through the K buffer (no MMA reads it
    // any more; with no Q tile it was never loaded)
    if (ok) {
      tc_fence_after();
      store_rows_tma<128, kF16>(&p.tm_dv, t + L::kColAcc + h * 128, sK + h * kHalfBytes, kr,
                                j * kTile, h * 128, 1.f, any, sh.d, sh.nk, h_idx, b_idx);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// fa_bwd256_grad<kKeys>: dK (kKeys, the CTA owns a key tile and loops over Q
// tiles) or dQ (the CTA owns a Q tile and loops over K/V tiles). In the
// CTA's own terms: rows = its tile, X = A1 B1^T and Y = A2 B2^T are the score
// and score-gradient tiles, E = P (Y - D) and acc += E B1, with
//   dK: A1 = K_j, A2 = V_j, B1 = Q_i, B2 = dO_i, LSE and D per column
//   dQ: A1 = Q_i, A2 = dO_i, B1 = K_j, B2 = V_j, LSE and D per row.
// 12 warps:
//   warp 0      TMA producer: A1 and A2 once; per step (dK) LSE_i log2e and D_i
//               (2 stages), and the halves of B1 and B2 through a ring of 3
//               slots in the order B1_0, B2_0, then per step n: B1_{n+1},
//               B1_n (again, for acc), B2_{n+1}
//   warp 1      tcgen05 issuer (one lane) and tensor-memory owner
//   warps 4-7   thread = row: P and E for columns 0..63 of each tile
//   warps 8-11  thread = row: columns 64..127; then both warpgroups store
//               the output (128 columns each)
// Tensor memory: X [0,128), Y [128,256) with E (16-bit pairs) written over
// the first 32 of each warpgroup's 64 Y columns, acc [256,512). MMA order:
// X(0), Y(0), then per step n: X(n+1) once X(n) has been read, acc += E(n)
// B1_n once E(n) is in tensor memory, Y(n+1) (after the MMA that reads E(n)).
template <bool kKeys>
struct GradLayout {
  static constexpr int kSlots = 3;
  static constexpr int kA1Off = 0;
  static constexpr int kA2Off = kTileBytes;
  static constexpr int kRingOff = 2 * kTileBytes;
  static constexpr int kStatOff = kRingOff + kSlots * kHalfBytes;  // dK: [2][LSE log2e 128 | D 128]
  static constexpr int kStatBytes = 2 * kTile * 4;
  static constexpr int kBarOff = kStatOff + (kKeys ? 2 * kStatBytes : 0);
  // a_full, full[3], empty[3], x_full, x_free, y_full, e_full, acc_done,
  // teardown, stat_full[2], stat_empty[2]
  static constexpr int kNumBars = 1 + 2 * kSlots + 6 + 4;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  static_assert(kBytes <= 232448, "shared memory budget");
  static constexpr uint32_t kColX = 0, kColY = 128, kColAcc = 256;
};

struct GradBars {
  uint32_t base;
  __device__ uint32_t a_full() const { return base; }
  __device__ uint32_t full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t empty(int s) const { return base + 8 * (4 + s); }
  __device__ uint32_t x_full() const { return base + 8 * 7; }
  __device__ uint32_t x_free() const { return base + 8 * 8; }
  __device__ uint32_t y_full() const { return base + 8 * 9; }
  __device__ uint32_t e_full() const { return base + 8 * 10; }
  __device__ uint32_t acc_done() const { return base + 8 * 11; }
  __device__ uint32_t teardown() const { return base + 8 * 12; }
  __device__ uint32_t stat_full(int b) const { return base + 8 * (13 + b); }
  __device__ uint32_t stat_empty(int b) const { return base + 8 * (15 + b); }
};

template <bool kKeys, bool kF16>
__global__ void __launch_bounds__(kThreads, 1) fa_bwd256_grad(const __grid_constant__ BwdParams p) {
  using L = GradLayout<kKeys>;
  constexpr uint32_t kKern = kKeys ? kKernBwd256Dk : kKernBwd256Dq;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t s_base = smem_u32(smem);
  int *misc = reinterpret_cast<int *>(smem + L::kMiscOff);  // [0] tmem [2] abort [3] loads in set-up
  if (s_base & 1023u) {  // the 128-byte swizzle needs 1024-byte aligned tiles
    if (threadIdx.x == 0 && p.status) atomicCAS(p.status, 0u, status_code(kKern, kRoleInit, 1));
    return;
  }
  const uint32_t sA1 = s_base + L::kA1Off, sA2 = s_base + L::kA2Off;
  const uint32_t sRing = s_base + L::kRingOff;
  const float *stat = reinterpret_cast<const float *>(smem + L::kStatOff);
  GradBars bars{s_base + L::kBarOff};
  StatusSlot st{p.status, &misc[2], p.wait_limit_ns};
  const int warp = threadIdx.x >> 5;
  const CUtensorMap *tm_a1 = kKeys ? &p.tm_k : &p.tm_q;
  const CUtensorMap *tm_a2 = kKeys ? &p.tm_v : &p.tm_do;
  const CUtensorMap *tm_b1 = kKeys ? &p.tm_q : &p.tm_k;
  const CUtensorMap *tm_b2 = kKeys ? &p.tm_do : &p.tm_v;

  // CTA order: head groups of p.head_group heads; within a group the heavy
  // tiles first (causal: early key tiles for dK, late Q tiles for dQ)
  const Shape &sh = p.sh;
  const int n_rows = kKeys ? sh.tk : sh.tq;  // row tiles per head
  const int hg = p.head_group;
  const int group = blockIdx.x / (hg * n_rows);
  const int g_base = group * hg;
  const int g_size = min(hg, sh.bh - g_base);
  const int g_rank = blockIdx.x - group * hg * n_rows;
  const int rt = kKeys ? g_rank / g_size : n_rows - 1 - g_rank / g_size;  // this CTA's row tile
  const int bh = g_base + g_rank % g_size;
  const int b_idx = bh / sh.heads, h_idx = bh % sh.heads;
  // column tiles, ascending: dK: Q tiles with a row that sees a key of tile
  // rt; dQ: K/V tiles up to the last one a row of tile rt sees; both where
  // the block mask allows
  const int jmax = kKeys ? 0 : sh.last_kv_tile(rt);
  const int col_end = kKeys ? sh.tq : sh.tk;
  auto next_col = [&](int x) { return kKeys ? next_q(sh, x, rt) : next_k(sh, rt, x, jmax); };
  const int first = next_col(kKeys ? sh.first_q_tile(rt) : 0);
  const bool any = first < col_end;
  const size_t stat_head = (size_t)bh * sh.tq * kTile;  // this head's workspace rows

  if (warp == 0 && (threadIdx.x & 31) == 0) {
    mbar_init(bars.a_full(), 1);
    for (int s = 0; s < L::kSlots; ++s) {
      mbar_init(bars.full(s), 1);
      mbar_init(bars.empty(s), 1);
    }
    mbar_init(bars.x_full(), 1);
    mbar_init(bars.x_free(), 256);
    mbar_init(bars.y_full(), 1);
    mbar_init(bars.e_full(), 256);
    mbar_init(bars.acc_done(), 1);
    mbar_init(bars.teardown(), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.stat_full(b), 1);
      mbar_init(bars.stat_empty(b), 256);
    }
    misc[2] = 0;
    fence_mbar_init();
    tma_prefetch_desc(tm_a1);
    tma_prefetch_desc(tm_a2);
    tma_prefetch_desc(tm_b1);
    tma_prefetch_desc(tm_b2);
    // A1, A2 and the first ring positions (both halves of B1 and the first
    // half of B2 of the first column tile, with its statistics) depend on
    // blockIdx only: load them now
    int pre = 0;
    if (any && !(p.debug_flags & kDebugSkipLoads)) {
      mbar_arrive_expect_tx(bars.a_full(), 2 * kTileBytes);
      for (int c = 0; c < 4; ++c) {
        tma_load_4d(sA1 + c * kChunkBytes, tm_a1, c * 64, rt * kTile, h_idx, b_idx, bars.a_full());
        tma_load_4d(sA2 + c * kChunkBytes, tm_a2, c * 64, rt * kTile, h_idx, b_idx, bars.a_full());
      }
      if constexpr (kKeys) {
        const uint32_t dst = s_base + L::kStatOff;
        const size_t row = stat_head + (size_t)first * kTile;
        mbar_arrive_expect_tx(bars.stat_full(0), L::kStatBytes);
        bulk_load_1d(dst, p.lse2 + row, kTile * 4, bars.stat_full(0));
        bulk_load_1d(dst + kTile * 4, p.delta + row, kTile * 4, bars.stat_full(0));
      }
      for (int q = 0; q < L::kSlots; ++q) {  // positions 0, 1: B1 halves; 2: B2 half 0
        mbar_arrive_expect_tx(bars.full(q), kHalfBytes);
        load_half(sRing + q * kHalfBytes, q < 2 ? tm_b1 : tm_b2, q & 1, first * kTile, h_idx, b_idx,
                  bars.full(q));
      }
      pre = L::kSlots;
    }
    misc[3] = pre;  // ring positions issued during set-up
  } else if (warp == 1) {
    tmem_alloc(smem_u32(&misc[0]), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);

  if (warp == 0) {
    // ---- TMA producer ------------------------------------------------------
    if (elect_one() && any && !(p.debug_flags & kDebugSkipLoads)) {
      bool ok = true;
      int issued = 0, nst = 0;
      const int pre = misc[3];  // positions (and the first statistics) issued in set-up
      auto ring_load = [&](const CUtensorMap *tm, int x) {
        for (int h = 0; h < 2 && ok; ++h) {
          if (issued < pre) {
            ++issued;
            continue;
          }
          const int s = issued % L::kSlots;
          ok = mbar_wait(bars.empty(s), ((issued / L::kSlots) & 1u) ^ 1u, st,
                         status_code(kKern, kRoleLoad, 1));
          if (!ok) return;
          mbar_arrive_expect_tx(bars.full(s), kHalfBytes);
          load_half(sRing + s * kHalfBytes, tm, h, x * kTile, h_idx, b_idx, bars.full(s));
          ++issued;
        }
      };
      // dK: LSE_i log2e and D_i of step nst (Q tile i)
      auto load_stats = [&](int i) {
        if constexpr (kKeys) {
          if (nst == 0 && pre > 0) {
            nst = 1;
            return;
          }
          const int b = nst & 1;
          ok = ok && mbar_wait(bars.stat_empty(b), ((nst >> 1) & 1u) ^ 1u, st,
                               status_code(kKern, kRoleLoad, 2));
          if (!ok) return;
          const uint32_t dst = s_base + L::kStatOff + b * L::kStatBytes;
          const size_t row = stat_head + (size_t)i * kTile;
          mbar_arrive_expect_tx(bars.stat_full(b), L::kStatBytes);
          bulk_load_1d(dst, p.lse2 + row, kTile * 4, bars.stat_full(b));
          bulk_load_1d(dst + kTile * 4, p.delta + row, kTile * 4, bars.stat_full(b));
          ++nst;
        }
      };
      load_stats(first);
      ring_load(tm_b1, first);
      ring_load(tm_b2, first);
      for (int x = first; x < col_end && ok;) {
        const int xn = next_col(x + 1);
        if (xn < col_end) {
          load_stats(xn);
          ring_load(tm_b1, xn);
        }
        ring_load(tm_b1, x);
        if (xn < col_end) ring_load(tm_b2, xn);
        x = xn;
      }
      // teardown: every copy issued has landed
      mbar_wait_drain(bars.a_full(), 0, st, status_code(kKern, kRoleLoad, 3));
      for (int s = 0; s < L::kSlots && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / L::kSlots) * L::kSlots;
        mbar_wait_drain(bars.full(s), (last / L::kSlots) & 1u, st, status_code(kKern, kRoleLoad, 4));
      }
      for (int b = 0; b < 2 && b < nst; ++b) {
        const int last = b + ((nst - 1 - b) / 2) * 2;
        mbar_wait_drain(bars.stat_full(b), (last >> 1) & 1u, st, status_code(kKern, kRoleLoad, 5));
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- tcgen05 issuer ----------------------------------------------------
    if (elect_one()) {
      constexpr uint32_t kIdX = idesc_f32acc(kTile, kTile, 0, 0, kF16);    // X, Y: K-major
      constexpr uint32_t kIdAcc = idesc_f32acc(kTile, kTile, 0, 1, kF16);  // acc half: B1 MN-major
      bool ok = !any || mbar_wait(bars.a_full(), 0, st, status_code(kKern, kRoleMma, 1));
      int pos = 0;
      auto next_slot = [&](uint32_t site) -> int {
        const int s = pos % L::kSlots;
        if (!mbar_wait(bars.full(s), (pos / L::kSlots) & 1u, st, status_code(kKern, kRoleMma, site)))
          return -1;
        tc_fence_after();
        return s;
      };
      // X = A1 B1^T (a = sA1, col = X) or Y = A2 B2^T, over the two halves
      auto issue_sq = [&](uint32_t a, uint32_t col, uint32_t done_bar) -> bool {
        for (int h = 0; h < 2; ++h) {
          const int s = next_slot(2);
          if (s < 0) return false;
          mma_half_ss(tmem + col, a, sRing + s * kHalfBytes, h, kIdX, h > 0);
          mma_commit(bars.empty(s));
          ++pos;
        }
        mma_commit(done_bar);
        return true;
      };
      if (ok && any) {
        ok = issue_sq(sA1, L::kColX, bars.x_full());
        if (ok) ok = issue_sq(sA2, L::kColY, bars.y_full());
        int n = 0;
        for (int x = first; x < col_end && ok; ++n) {
          const int xn = next_col(x + 1);
          if (xn < col_end) {
            ok = mbar_wait(bars.x_free(), n & 1, st, status_code(kKern, kRoleMma, 3));
            if (ok) ok = issue_sq(sA1, L::kColX, bars.x_full());
            if (!ok) break;
          }
          ok = mbar_wait(bars.e_full(), n & 1, st, status_code(kKern, kRoleMma, 4));
          if (!ok) break;
          tc_fence_after();
          // acc[:, 128h ..] += E(n) B1_x[:, 128h ..]
          for (int h = 0; h < 2 && ok; ++h) {
            const int s = next_slot(5);
            if (s < 0) {
              ok = false;
              break;
            }
            mma_half_ts(tmem + L::kColAcc + h * kTile, tmem + L::kColY, sRing + s * kHalfBytes,
                        kIdAcc, n > 0);
            mma_commit(bars.empty(s));
            ++pos;
          }
          if (ok && xn < col_end) ok = issue_sq(sA2, L::kColY, bars.y_full());
          x = xn;
        }
      }
      if (ok && any) mma_commit(bars.acc_done());
      mma_commit(bars.teardown());
      mbar_wait_drain(bars.teardown(), 0, st, status_code(kKern, kRoleMma, 8));
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---- P and E for one half of the columns (thread = row) ----------------
    const int h = (warp - 4) >> 2;                 // columns 64h .. 64h+63 of each tile
    const int r = threadIdx.x & 127;               // row = TMEM lane
    const uint32_t t = tmem + (uint32_t((warp & 3) * 32) << 16);
    const float c = p.scale_log2;
    float lse2_row = 0.f, d_row = 0.f;             // dQ: this query row's LSE log2e and D
    if constexpr (!kKeys) {
      const size_t grow = stat_head + (size_t)rt * kTile + r;
      lse2_row = p.lse2[grow];
      d_row = p.delta[grow];
    }
    bool ok = true;
    int n = 0;
    for (int x = first; x < col_end && ok; x = next_col(x + 1), ++n) {
      ok = __all_sync(0xffffffffu, mbar_wait(bars.x_full(), n & 1, st,
                                             status_code(kKern, kRoleSoftmax, 1)));
      if constexpr (kKeys)
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bars.stat_full(n & 1), (n >> 1) & 1u, st,
                                                       status_code(kKern, kRoleSoftmax, 2)));
      if (!ok) break;
      tc_fence_after();
      const float *lse2c = stat + (n & 1) * 2 * kTile + 64 * h;  // dK: per-column statistics
      const float *dc = lse2c + kTile;
      float pr[64];
      {
        // both loads in flight before the one wait
        uint32_t sr[2][32];
        tmem_ld32(t + L::kColX + 64 * h, sr[0]);
        tmem_ld32(t + L::kColX + 64 * h + 32, sr[1]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bars.x_free());
#pragma unroll
        for (int k = 0; k < 64; ++k)
          pr[k] = ex2_approx(fmaf(__uint_as_float(sr[k >> 5][k & 31]), c,
                                  kKeys ? -lse2c[k] : -lse2_row));
      }
      // the mask, only on the tiles it touches
      if constexpr (kKeys) {
        // key row r of tile rt sees query 64h + k of tile x iff k >= lo
        if (sh.causal && kTile * rt + kTile - 1 > kTile * x + sh.causal_off) {
          const int lo = kTile * (rt - x) + r - sh.causal_off - 64 * h;
#pragma unroll
          for (int k = 0; k < 64; ++k)
            if (k < lo) pr[k] = 0.f;
        }
      } else {
        // keys 64h + k >= key_limit of tile x are hidden from query row r
        if (sh.partial(rt, x)) {
          const int lim = sh.key_limit(rt, r, x) - 64 * h;
#pragma unroll
          for (int k = 0; k < 64; ++k)
            if (k >= lim) pr[k] = 0.f;
        }
      }
      ok = __all_sync(0xffffffffu, mbar_wait(bars.y_full(), n & 1, st,
                                             status_code(kKern, kRoleSoftmax, 3)));
      if (!ok) break;
      tc_fence_after();
      uint32_t ep[32];
      {
        uint32_t dr[2][32];
        tmem_ld32(t + L::kColY + 64 * h, dr[0]);
        tmem_ld32(t + L::kColY + 64 * h + 32, dr[1]);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 64; k += 2) {
          const float d0 = kKeys ? dc[k] : d_row;
          const float d1 = kKeys ? dc[k + 1] : d_row;
          ep[k / 2] = pack2<kF16>(pr[k] * (__uint_as_float(dr[k >> 5][k & 31]) - d0),
                                  pr[k + 1] * (__uint_as_float(dr[k >> 5][(k + 1) & 31]) - d1));
        }
      }
      // E over the first 32 of this warpgroup's Y columns (already read)
      tmem_st32(t + L::kColY + 64 * h, ep);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bars.e_full());
      if constexpr (kKeys) mbar_arrive(bars.stat_empty(n & 1));
    }
    if (ok && any)
      ok = __all_sync(0xffffffffu, mbar_wait(bars.acc_done(), 0, st,
                                             status_code(kKern, kRoleSoftmax, 4)));
    // dK or dQ (times scale), 128 columns per warpgroup, through the A1
    // buffer (no MMA reads it any more; with no column tile it was never loaded)
    if (ok) {
      tc_fence_after();
      store_rows_tma<128, kF16>(kKeys ? &p.tm_dk : &p.tm_dq, t + L::kColAcc + h * 128,
                                sA1 + h * kHalfBytes, r, rt * kTile, h * 128, p.scale, any, sh.d,
                                kKeys ? sh.nk : sh.nq, h_idx, b_idx);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool kF16>
cudaError_t launch_d256(const BwdParams &p, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(fa_bwd256_dv<kF16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, DvLayout::kBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fa_bwd256_grad<true, kF16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, GradLayout<true>::kBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fa_bwd256_grad<false, kF16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, GradLayout<false>::kBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const unsigned key_ctas = unsigned(p.sh.tk) * unsigned(p.sh.bh);
  {
    LaunchProbe probe(kKindBwd256Dv, stream);
    fa_bwd256_dv<kF16><<<key_ctas, kThreads, DvLayout::kBytes, stream>>>(p);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    LaunchProbe probe(kKindBwd256Dk, stream);
    fa_bwd256_grad<true, kF16><<<key_ctas, kThreads, GradLayout<true>::kBytes, stream>>>(p);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    LaunchProbe probe(kKindBwd256Dq, stream);
    fa_bwd256_grad<false, kF16><<<unsigned(p.sh.tq) * unsigned(p.sh.bh), kThreads,
                                  GradLayout<false>::kBytes, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward_d256(const BwdParams &p, cudaStream_t stream) {
  return p.sh.f16 ? launch_d256<true>(p, stream) : launch_d256<false>(p, stream);
}

}  // namespace fa
