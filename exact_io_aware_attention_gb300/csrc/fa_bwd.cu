// Attention backward for sm_103a, by recomputation: preprocess and dK/dV.
//
// The pages store only O and the softmax statistics and regenerate S and P
// block by block in the backward pass ("Paper Notes: FlashAttention",
// "Background" and "Key Ideas"; aicassindra page, "The backward pass:
// recompute instead of store"). They do not print the gradient formulas; the
// kernels evaluate the analytic gradients of O = softmax(scale QK^T) V:
//
//   P_ij  = exp(scale s_ij - LSE_i)        (recomputed from Q, K and LSE)
//   dV_j  = sum_i P_ij dO_i
//   dP_ij = dO_i . V_j
//   D_i   = dO_i . O_i                     (= sum_j P_ij dP_ij)
//   dS_ij = P_ij (dP_ij - D_i)
//   dQ_i  = scale sum_j dS_ij K_j,   dK_j = scale sum_i dS_ij Q_i
//
// The two-kernel backward, three kernels on the caller's stream (the one-pass
// backward of fa_bwd_fused.cu shares fa_bwd_pre and replaces the other two):
//   fa_bwd_pre        D_i and LSE_i * log2(e), padded to whole Q tiles
//   fa_bwd_dkdv       one CTA per 128-key K/V tile, looping over the Q tiles
//                     that see it (causal: a row of the tile sees one of its
//                     keys; block-sparse: mask[i][j]); dK and dV accumulate in
//                     tensor memory (this file)
//   fa_bwd_dq_kernel  one CTA per Q tile, looping over its K/V tiles; dQ
//                     accumulates in tensor memory (fa_bwd_dq.cu)
// Each gradient is owned by one CTA, so no cross-CTA reduction is needed;
// the price is that S and dP are recomputed by both kernels. Head dimension
// 256 shares fa_bwd_pre and then runs the kernels of fa_bwd_d256.cu.
//
// Rows past the end of a sequence (the last, partial Q or K/V tile) arrive
// as zeros from the tensor maps. A missing query row has LSE * log2(e) = +inf
// in the workspace, so its P row is exactly 0 and it adds nothing; a missing
// key row only feeds its own dK/dV row, which is not stored.
//
// fa_bwd_dkdv, 12 warps:
//   warp 0      TMA producer: K_j, V_j once; per step Q_i with LSE_i (3 slots) and
//               dO_i with D_i (2 slots)
//   warp 1      tcgen05 issuer (one lane) and tensor-memory owner
//   warps 4-7   thread = key row: P^T and dS^T for queries 0..63; then dV out
//               (once the last dV MMA has completed: dv_done)
//   warps 8-11  thread = key row: P^T and dS^T for queries 64..127; then dK out
// Tensor memory (512 columns): [0,128) S^T, [128,256) dP^T, then dV and dK
// (d columns each). P^T and dS^T (16-bit pairs) are the tensor-memory A
// operands of dV += P^T dO and dK += dS^T Q: the warpgroup for queries
// 64h..64h+63 writes them over the first 32 of its own 64 S^T (dP^T)
// columns once it has read them. P^T goes out in two halves of 32 queries,
// each on its own barrier, and dV(n) is issued in the same two halves.
// Shared memory: K_j, V_j, Q_i[3] with LSE_i, dO_i[2] with D_i. A Q slot is
// free once dK has read it; a dO slot once dV has read dO_i and the softmax
// warps have read D_i, so Q_{n+2} loads while step n is still running.
// MMA order per step n: dV(n), S^T(n+1), dK(n), dP^T(n+1); MMAs issued by
// one thread execute in issue order, so S^T(n+1) and dP^T(n+1) overwrite
// P^T(n) and dS^T(n) only after dV(n) and dK(n) have read them.
#include <math.h>

#include "fa_internal.h"
#include "ptx.cuh"
#include "tile_store.cuh"

namespace fa {
namespace {

constexpr int kThreads = 384;

template <int D>
struct DkdvLayout {
  static constexpr int kChunks = (D + 63) / 64;  // d = 96: 2, the last half zeros
  static constexpr int kChunkBytes = kTile * 128;
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static constexpr int kQSlots = 3, kdOSlots = 2;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kTileBytes;
  static constexpr int kQOff = kVOff + kTileBytes;
  static constexpr int kdOOff = kQOff + kQSlots * kTileBytes;
  static constexpr int kLseOff = kdOOff + kdOSlots * kTileBytes;  // [kQSlots][128] LSE * log2(e)
  static constexpr int kDeltaOff = kLseOff + kQSlots * kTile * 4;  // [kdOSlots][128] D
  static constexpr int kBarOff = kDeltaOff + kdOSlots * kTile * 4;
  static constexpr int kNumBars = 19;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  static_assert(kBytes <= 232448, "shared memory budget");
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
};

struct Bars {
  uint32_t base;
  __device__ uint32_t kv_full() const { return base; }
  // Q slot s (Q_i with LSE_i) and dO slot s (dO_i with D_i)
  __device__ uint32_t q_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t q_empty(int s) const { return base + 8 * (4 + s); }
  __device__ uint32_t do_full(int s) const { return base + 8 * (7 + s); }
  __device__ uint32_t do_empty(int s) const { return base + 8 * (9 + s); }
  __device__ uint32_t s_full() const { return base + 8 * 11; }
  // P^T of queries 64h + 32u .. 64h + 32u + 31 of both warpgroups h (u = 0, 1)
  __device__ uint32_t p_full(int u) const { return base + 8 * (12 + u); }
  __device__ uint32_t dp_full() const { return base + 8 * 14; }
  __device__ uint32_t ds_full() const { return base + 8 * 15; }
  __device__ uint32_t acc_done() const { return base + 8 * 16; }
  __device__ uint32_t teardown() const { return base + 8 * 17; }
  __device__ uint32_t dv_done() const { return base + 8 * 18; }
};

enum Role : uint32_t { kRoleLoad = 1, kRoleMma = 2, kRoleSoftmax = 3, kRoleInit = 5 };

// Next Q tile at or after i that the block mask lets see K/V tile j (tq if none).
__device__ __forceinline__ int next_q(const Shape &sh, int i, int j) {
  if (sh.mask)
    while (i < sh.tq && sh.mask[(size_t)i * sh.tk + j] == 0) ++i;
  return i;
}

// Tensor-memory column of the packed A operand (P^T or dS^T) for MMA step kk
// (queries 16kk..16kk+15): queries 64h.. are packed at column 64h.
__device__ __forceinline__ uint32_t packed_col(int kk) { return (kk >> 2) * 64 + (kk & 3) * 8; }

// Q tile i with LSE_i * log2(e) into Q slot s, onto q_full(s).
template <int D>
__device__ __forceinline__ void load_q(const BwdParams &p, const Bars &bars, int s, int i,
                                       uint32_t s_base, size_t stat_head, int h_idx, int b_idx) {
  using L = DkdvLayout<D>;
  mbar_arrive_expect_tx(bars.q_full(s), L::kTileBytes + kTile * 4);
  for (int c = 0; c < L::kChunks; ++c)
    tma_load_4d(s_base + L::kQOff + s * L::kTileBytes + c * L::kChunkBytes, &p.tm_q, c * 64,
                i * kTile, h_idx, b_idx, bars.q_full(s));
  bulk_load_1d(s_base + L::kLseOff + s * kTile * 4, p.lse2 + stat_head + (size_t)i * kTile,
               kTile * 4, bars.q_full(s));
}

// dO tile i with D_i into dO slot s, onto do_full(s).
template <int D>
__device__ __forceinline__ void load_do(const BwdParams &p, const Bars &bars, int s, int i,
                                        uint32_t s_base, size_t stat_head, int h_idx, int b_idx) {
  using L = DkdvLayout<D>;
  mbar_arrive_expect_tx(bars.do_full(s), L::kTileBytes + kTile * 4);
  for (int c = 0; c < L::kChunks; ++c)
    tma_load_4d(s_base + L::kdOOff + s * L::kTileBytes + c * L::kChunkBytes, &p.tm_do, c * 64,
                i * kTile, h_idx, b_idx, bars.do_full(s));
  bulk_load_1d(s_base + L::kDeltaOff + s * kTile * 4, p.delta + stat_head + (size_t)i * kTile,
               kTile * 4, bars.do_full(s));
}

// kF16: f16 elements instead of bf16. D is 64, 96 or 128: at 96 the tiles keep two 64-column
// chunks (the tensor maps read zeros in columns 96..127), the MMAs run 6 K-steps over the head
// dimension and N = 96, and 96 columns of dK and dV are stored.
template <int D, bool kF16>
__global__ void __launch_bounds__(kThreads, 1) fa_bwd_dkdv(const __grid_constant__ BwdParams p) {
  using L = DkdvLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t s_base = smem_u32(smem);
  int *misc = reinterpret_cast<int *>(smem + L::kMiscOff);  // [0] tmem [2] abort
  // The 128-byte swizzle patterns need 1024-byte aligned tiles; the layout
  // has no room for alignment slack, so a misaligned base is reported.
  if (s_base & 1023u) {
    if (threadIdx.x == 0 && p.status) atomicCAS(p.status, 0u, status_code(kKernBwd, kRoleInit, 1));
    return;
  }
  const uint32_t sK = s_base + L::kKOff, sV = s_base + L::kVOff;
  const uint32_t sQ = s_base + L::kQOff, sdO = s_base + L::kdOOff;
  const float *lse_s = reinterpret_cast<const float *>(smem + L::kLseOff);
  const float *delta_s = reinterpret_cast<const float *>(smem + L::kDeltaOff);
  Bars bars{s_base + L::kBarOff};
  StatusSlot st{p.status, &misc[2], p.wait_limit_ns};

  const int warp = threadIdx.x >> 5;
  const Shape &sh = p.sh;
  const int T = sh.tq;
  // CTAs are ordered head group by head group (p.head_group heads at a
  // time); within a group the heavy K/V tiles come first (causal: the early
  // key tiles are seen by the most Q tiles).
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
  const size_t stat_head = (size_t)bh * T * kTile;  // this head's rows in the workspace

  if (warp == 0 && (threadIdx.x & 31) == 0) {
    mbar_init(bars.kv_full(), 1);
    for (int s = 0; s < L::kQSlots; ++s) {
      mbar_init(bars.q_full(s), 1);
      mbar_init(bars.q_empty(s), 1);
    }
    // a dO slot is free once dV has read dO_i (one commit) and the softmax
    // warps have read D_i (256 threads)
    for (int s = 0; s < L::kdOSlots; ++s) {
      mbar_init(bars.do_full(s), 1);
      mbar_init(bars.do_empty(s), 257);
    }
    mbar_init(bars.s_full(), 1);
    mbar_init(bars.p_full(0), 256);
    mbar_init(bars.p_full(1), 256);
    mbar_init(bars.dp_full(), 1);
    mbar_init(bars.ds_full(), 256);
    mbar_init(bars.acc_done(), 1);
    mbar_init(bars.teardown(), 1);
    mbar_init(bars.dv_done(), 1);
    misc[2] = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
    tma_prefetch_desc(&p.tm_do);
    // K_j, V_j and the first Q tile's stage depend on blockIdx only: load
    // them now, while the other warps set up
    if (any && !(p.debug_flags & kDebugSkipLoads)) {
      mbar_arrive_expect_tx(bars.kv_full(), 2 * L::kTileBytes);
      for (int c = 0; c < L::kChunks; ++c) {
        tma_load_4d(sK + c * L::kChunkBytes, &p.tm_k, c * 64, j * kTile, h_idx, b_idx,
                    bars.kv_full());
        tma_load_4d(sV + c * L::kChunkBytes, &p.tm_v, c * 64, j * kTile, h_idx, b_idx,
                    bars.kv_full());
      }
      load_q<D>(p, bars, 0, first, s_base, stat_head, h_idx, b_idx);
      load_do<D>(p, bars, 0, first, s_base, stat_head, h_idx, b_idx);
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
    // ---- TMA producer ------------------------------------------------------
    if (elect_one() && any && !(p.debug_flags & kDebugSkipLoads)) {
      int nq = 1, ndo = 1;  // tiles issued: the first Q tile's Q and dO came with the set-up
      bool ok = true;
      for (int i = next_q(sh, first + 1, j); i < T && ok; i = next_q(sh, i + 1, j)) {
        const int qs = nq % L::kQSlots;
        ok = mbar_wait(bars.q_empty(qs), ((nq / L::kQSlots) & 1u) ^ 1u, st,
                       status_code(kKernBwd, kRoleLoad, 1));
        if (!ok) break;
        load_q<D>(p, bars, qs, i, s_base, stat_head, h_idx, b_idx);
        ++nq;
        const int ds = ndo % L::kdOSlots;
        ok = mbar_wait(bars.do_empty(ds), ((ndo / L::kdOSlots) & 1u) ^ 1u, st,
                       status_code(kKernBwd, kRoleLoad, 4));
        if (!ok) break;
        load_do<D>(p, bars, ds, i, s_base, stat_head, h_idx, b_idx);
        ++ndo;
      }
      // teardown: every copy issued has landed
      mbar_wait_drain(bars.kv_full(), 0, st, status_code(kKernBwd, kRoleLoad, 2));
      for (int s = 0; s < L::kQSlots && s < nq; ++s) {
        const int last = s + ((nq - 1 - s) / L::kQSlots) * L::kQSlots;
        mbar_wait_drain(bars.q_full(s), (last / L::kQSlots) & 1u, st, status_code(kKernBwd, kRoleLoad, 3));
      }
      for (int s = 0; s < L::kdOSlots && s < ndo; ++s) {
        const int last = s + ((ndo - 1 - s) / L::kdOSlots) * L::kdOSlots;
        mbar_wait_drain(bars.do_full(s), (last / L::kdOSlots) & 1u, st, status_code(kKernBwd, kRoleLoad, 5));
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- tcgen05 issuer ----------------------------------------------------
    if (elect_one()) {
      constexpr uint32_t kIdSq = idesc_f32acc(kTile, kTile, 0, 0, kF16);  // S^T, dP^T
      constexpr uint32_t kIdAcc = idesc_f32acc(kTile, D, 0, 1, kF16);     // dV, dK: B MN-major
      bool ok = !any || mbar_wait(bars.kv_full(), 0, st, status_code(kKernBwd, kRoleMma, 1));
      // X^T = A Y^T with A in {K_j, V_j} and Y in {Q_i, dO_i}: K-major over d
      auto issue_sq = [&](uint32_t a_base, uint32_t b_base, uint32_t col) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::kChunkBytes + (kk & 3) * 32;
          mma_f16kind_ss(tmem + col, sdesc_sw128(a_base + off, 16, 1024),
                      sdesc_sw128(b_base + off, 16, 1024), kIdSq, kk > 0);
        }
      };
      // acc += X Y with X = P^T (or dS^T) packed in tensor memory at a_col and
      // Y with queries as K (MN-major, 16 query rows per step), over the
      // queries 64h + 32u .. 64h + 32u + 31 of both warpgroups h
      auto issue_acc = [&](uint32_t a_col, uint32_t y_base, uint32_t col, bool first, int u) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int kk = (e >> 1) * 4 + 2 * u + (e & 1);
          mma_f16kind_ts(tmem + col, tmem + a_col + packed_col(kk),
                      sdesc_sw128(y_base + kk * 2048, L::kChunkBytes, 1024), kIdAcc,
                      (!first || u > 0 || e > 0) ? 1u : 0u);
        }
      };
      if (ok && any) {
        ok = mbar_wait(bars.q_full(0), 0, st, status_code(kKernBwd, kRoleMma, 2));
        if (ok) {
          tc_fence_after();
          issue_sq(sK, sQ, L::kColS);
          mma_commit(bars.s_full());
          ok = mbar_wait(bars.do_full(0), 0, st, status_code(kKernBwd, kRoleMma, 7));
        }
        if (ok) {
          tc_fence_after();
          issue_sq(sV, sdO, L::kColDP);
          mma_commit(bars.dp_full());
        }
      }
      int n = 0, qs = 0, qph = 0;  // Q slot of step n and the parity of its phase
      for (int i = first; i < T && ok; ++n) {
        const int ds = n & 1, ds1 = ds ^ 1;  // dO slots of steps n and n + 1
        const int qs1 = qs + 1 == L::kQSlots ? 0 : qs + 1;
        const int qph1 = qs + 1 == L::kQSlots ? qph ^ 1 : qph;
        const int inext = next_q(sh, i + 1, j);
        // dV(n) in two halves: the first runs while the softmax warps finish
        // the second half of P^T(n)
        ok = mbar_wait(bars.p_full(0), n & 1, st, status_code(kKernBwd, kRoleMma, 3));
        if (!ok) break;
        tc_fence_after();
        issue_acc(L::kColS, sdO + ds * L::kTileBytes, L::kColDV, n == 0, 0);
        ok = mbar_wait(bars.p_full(1), n & 1, st, status_code(kKernBwd, kRoleMma, 6));
        if (!ok) break;
        tc_fence_after();
        issue_acc(L::kColS, sdO + ds * L::kTileBytes, L::kColDV, n == 0, 1);
        mma_commit(bars.do_empty(ds));  // dV(n) has read dO_n
        // dV is final after the last step's dV MMA: its epilogue need not
        // wait for the last dK
        if (inext >= T) mma_commit(bars.dv_done());
        if (inext < T) {
          ok = mbar_wait(bars.q_full(qs1), qph1, st, status_code(kKernBwd, kRoleMma, 4));
          if (!ok) break;
          tc_fence_after();
          issue_sq(sK, sQ + qs1 * L::kTileBytes, L::kColS);
          mma_commit(bars.s_full());
        }
        ok = mbar_wait(bars.ds_full(), n & 1, st, status_code(kKernBwd, kRoleMma, 5));
        if (!ok) break;
        tc_fence_after();
        issue_acc(L::kColDP, sQ + qs * L::kTileBytes, L::kColDK, n == 0, 0);
        issue_acc(L::kColDP, sQ + qs * L::kTileBytes, L::kColDK, n == 0, 1);
        mma_commit(bars.q_empty(qs));
        if (inext < T) {
          ok = mbar_wait(bars.do_full(ds1), ((n + 1) >> 1) & 1, st, status_code(kKernBwd, kRoleMma, 7));
          if (!ok) break;
          tc_fence_after();
          issue_sq(sV, sdO + ds1 * L::kTileBytes, L::kColDP);
          mma_commit(bars.dp_full());
        }
        i = inext;
        qs = qs1;
        qph = qph1;
      }
      if (ok) mma_commit(bars.acc_done());
      mma_commit(bars.teardown());
      mbar_wait_drain(bars.teardown(), 0, st, status_code(kKernBwd, kRoleMma, 8));
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---- P^T and dS^T for one half of the queries (thread = key row) --------
    const int h = (warp - 4) >> 2;                 // query half: 64h .. 64h+63
    const int kr = threadIdx.x & 127;              // key row = TMEM lane
    const uint32_t t = tmem + (uint32_t((warp & 3) * 32) << 16);
    const float c = p.scale_log2;
    bool ok = true;
    int n = 0, qs = 0, qph = 0;  // Q slot of step n and the parity of its phase
    for (int i = first; i < T && ok; i = next_q(sh, i + 1, j), ++n) {
      const int ds = n & 1;  // dO slot
      ok = __all_sync(0xffffffffu, mbar_wait(bars.s_full(), n & 1, st,
                                             status_code(kKernBwd, kRoleSoftmax, 1)));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bars.q_full(qs), qph, st,
                                                     status_code(kKernBwd, kRoleSoftmax, 2)));
      if (!ok) break;
      tc_fence_after();
      const float *lse2 = lse_s + qs * kTile + 64 * h;
      const float *delta = delta_s + ds * kTile + 64 * h;
      qph = qs + 1 == L::kQSlots ? qph ^ 1 : qph;
      qs = qs + 1 == L::kQSlots ? 0 : qs + 1;
      // P^T_kq = exp2(s_kq * scale * log2e - LSE_q * log2e), in two halves of
      // 32 queries, each written to tensor memory (over this warpgroup's
      // first 32 S^T columns, already read) and announced on its own barrier
      // so that dV's MMAs over the first half can start early
      float pr[64];
      {
        uint32_t sr[2][32];
        tmem_ld32(t + L::kColS + 64 * h, sr[0]);
        tmem_ld32(t + L::kColS + 64 * h + 32, sr[1]);
        tmem_wait_ld();
        // only on a tile that the causal boundary crosses (one per K/V
        // tile): key kr sees query 64h + x only if x >= lo
        const bool cross = sh.causal && kTile * j + kTile - 1 > kTile * i + sh.causal_off;
        const int lo = kTile * (j - i) + kr - sh.causal_off - 64 * h;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
#pragma unroll
          for (int x = 32 * u; x < 32 * u + 32; ++x)
            pr[x] = ex2_approx(fmaf(__uint_as_float(sr[u][x & 31]), c, -lse2[x]));
          if (cross) {
#pragma unroll
            for (int x = 32 * u; x < 32 * u + 32; ++x)
              if (x < lo) pr[x] = 0.f;
          }
          uint32_t pk[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) pk[x] = pack2<kF16>(pr[32 * u + 2 * x], pr[32 * u + 2 * x + 1]);
          tmem_st16(t + L::kColS + 64 * h + 16 * u, pk);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bars.p_full(u));
        }
      }
      // dS^T_kq = P^T_kq (dP^T_kq - D_q) into tensor memory over dP^T
      ok = __all_sync(0xffffffffu, mbar_wait(bars.dp_full(), n & 1, st,
                                             status_code(kKernBwd, kRoleSoftmax, 4)));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bars.do_full(ds), (n >> 1) & 1, st,
                                                     status_code(kKernBwd, kRoleSoftmax, 5)));
      if (!ok) break;
      tc_fence_after();
      uint32_t dsp[32];
      {
        uint32_t dr[2][32];
        tmem_ld32(t + L::kColDP + 64 * h, dr[0]);
        tmem_ld32(t + L::kColDP + 64 * h + 32, dr[1]);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 64; x += 2)
          dsp[x / 2] = pack2<kF16>(pr[x] * (__uint_as_float(dr[x >> 5][x & 31]) - delta[x]),
                                   pr[x + 1] * (__uint_as_float(dr[x >> 5][(x + 1) & 31]) - delta[x + 1]));
      }
      tmem_st32(t + L::kColDP + 64 * h, dsp);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bars.ds_full());
      mbar_arrive(bars.do_empty(ds));  // D_i has been read
    }
    // epilogue: warps 4-7 write dV, warps 8-11 write dK (scaled)
    if (ok && any)
      ok = __all_sync(0xffffffffu, mbar_wait(h ? bars.acc_done() : bars.dv_done(), 0, st,
                                             status_code(kKernBwd, kRoleSoftmax, 6)));
    // dV (warps 4-7) and dK (warps 8-11, times scale) leave through the K and
    // V buffers, which no MMA reads any more
    if (ok) {
      tc_fence_after();
      store_rows_tma<D, kF16>(h ? &p.tm_dk : &p.tm_dv, t + (h ? L::kColDK : L::kColDV),
                              h ? sV : sK, kr, j * kTile, 0, h ? p.scale : 1.f, any, sh.d, sh.nk,
                              h_idx, b_idx);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// D_i = dO_i . O_i and LSE_i * log2(e) for every row of every Q tile: a row
// past the end of the sequence, or one that sees no key (LSE = -inf), gets
// D = 0 and LSE * log2(e) = +inf, which makes its P row exactly 0. For the
// one-pass backward it also zeroes the block's rows of the fp32 dQ
// accumulator.
// Block = 64 rows of one head (blockIdx.x = (b * H + h) * chunks + chunk), so
// the index arithmetic is done once per block; a row is read by 16 threads with
// 16-byte loads (8 elements each; with a head dimension of 96, run as
// D = 128, the last 4 threads of a row add nothing), two rows per warp step.
constexpr int kPreRows = 64;

template <int D, bool kF16>
__global__ void __launch_bounds__(256) fa_bwd_pre(const __grid_constant__ BwdParams p) {
  constexpr int kLanesPerRow = D / 8;            // 8 or 16
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  const Shape &sh = p.sh;
  const int chunks = sh.tq * kTile / kPreRows;  // row chunks per head
  const int bh = int(blockIdx.x / chunks), chunk = int(blockIdx.x % chunks);
  const int b_idx = bh / sh.heads, h_idx = bh % sh.heads;
  const uint16_t *o_head = static_cast<const uint16_t *>(p.o) + p.so.row(b_idx, h_idx, 0);
  const uint16_t *g_head = static_cast<const uint16_t *>(p.dout) + p.sdo.row(b_idx, h_idx, 0);
  const size_t stat_head = (size_t)bh * sh.tq * kTile;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int part = lane % kLanesPerRow;
  const bool col_live = part * 8 < sh.d;
  for (int k = 0; k < kPreRows / (8 * kRowsPerWarp); ++k) {
    const int n = chunk * kPreRows + (k * 8 + warp) * kRowsPerWarp + lane / kLanesPerRow;
    const bool live = n < sh.nq;
    float acc = 0.f;
    if (live && col_live) {
      const uint4 o = *reinterpret_cast<const uint4 *>(o_head + (long long)n * p.so.n_ + part * 8);
      const uint4 g = *reinterpret_cast<const uint4 *>(g_head + (long long)n * p.sdo.n_ + part * 8);
      const uint32_t ow[4] = {o.x, o.y, o.z, o.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        float o0, o1, g0, g1;
        unpack2<kF16>(ow[h], o0, o1);
        unpack2<kF16>(gw[h], g0, g1);
        acc = fmaf(o0, g0, acc);
        acc = fmaf(o1, g1, acc);
      }
    }
#pragma unroll
    for (int off = kLanesPerRow / 2; off > 0; off >>= 1)
      acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (part == 0 && n < sh.tq * kTile) {
      const float l = live ? p.lse[(size_t)bh * sh.nq + n] : -INFINITY;
      const bool empty = isinf(l);  // also the rows past the end
      p.delta[stat_head + n] = empty ? 0.f : acc;
      p.lse2[stat_head + n] = empty ? INFINITY : l * 1.4426950408889634f;
    }
  }
  if (p.dq_acc) {  // rows chunk*64 .. chunk*64+63 of the head, sh.d floats each
    float4 *z = reinterpret_cast<float4 *>(p.dq_acc + (stat_head + (size_t)chunk * kPreRows) * sh.d);
    const int n4 = kPreRows * sh.d / 4;
    for (int x = threadIdx.x; x < n4; x += blockDim.x) z[x] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

template <int D, bool kF16>
cudaError_t launch_bwd_d(const BwdParams &p, cudaStream_t stream) {
  {
    LaunchProbe probe(kKindBwdPre, stream);
    const unsigned blocks = unsigned(p.sh.tq * kTile / kPreRows) * unsigned(p.sh.bh);
    // the preprocess reduces a row over a power-of-two number of lanes: a
    // head dimension of 96 runs its d = 128 form (the last 4 lanes of a row
    // add nothing)
    fa_bwd_pre<(D == 96 ? 128 : D), kF16><<<blocks, 256, 0, stream>>>(p);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if constexpr (D == 256) {
    return launch_backward_d256(p, stream);  // fa_bwd_d256.cu
  } else {
    if (p.dq_acc) return launch_backward_fused(p, stream);  // fa_bwd_fused.cu
    using L = DkdvLayout<D>;
    static bool configured = false;
    if (!configured) {
      e = cudaFuncSetAttribute(fa_bwd_dkdv<D, kF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               L::kBytes);
      if (e != cudaSuccess) return e;
      configured = true;
    }
    {
      LaunchProbe probe(kKindBwdDkdv, stream);
      fa_bwd_dkdv<D, kF16><<<p.sh.tk * p.sh.bh, kThreads, L::kBytes, stream>>>(p);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_backward_dq(p, stream);
  }
}

}  // namespace

cudaError_t launch_backward(const BwdParams &p, cudaStream_t stream) {
  const bool f16 = p.sh.f16 != 0;
  if (p.sh.d == 64) return f16 ? launch_bwd_d<64, true>(p, stream) : launch_bwd_d<64, false>(p, stream);
  if (p.sh.d == 96) return f16 ? launch_bwd_d<96, true>(p, stream) : launch_bwd_d<96, false>(p, stream);
  if (p.sh.d == 128)
    return f16 ? launch_bwd_d<128, true>(p, stream) : launch_bwd_d<128, false>(p, stream);
  if (p.sh.d == 256)
    return f16 ? launch_bwd_d<256, true>(p, stream) : launch_bwd_d<256, false>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
