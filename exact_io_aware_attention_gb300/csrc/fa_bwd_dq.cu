// Attention backward, dQ part, for sm_103a.
//
// dQ_i = scale * sum_j dS_ij K_j with dS_ij = P_ij (dP_ij - D_i),
// P_ij = exp(scale s_ij - LSE_i), dP_ij = dO_i . V_j (the analytic gradient
// of the definition; the pages leave the backward formulas to a companion
// article, aicassindra page "The backward pass: recompute instead of
// store"). One CTA owns a 128-row Q tile and recomputes S and dP for every
// K/V tile it sees (causal: a row of the tile sees one of the tile's keys;
// block-sparse: mask[i][j] != 0), so dQ accumulates in tensor memory and is
// written once, in 16 bits, without any cross-CTA reduction. Keys past the end
// of the sequence (zeros from the tensor map) and keys above the causal
// boundary get P = 0 on the tiles that need it.
//
// 12 warps:
//   warp 0      TMA producer: Q_i and dO_i once; K_j (3-slot ring) and V_j
//               (2 slots), interleaved
//   warp 1      tcgen05 issuer (one lane) and tensor-memory owner
//   warp 2      builds the list of K/V tiles to visit
//   warps 4-7   thread = query row; keys 0..63 of each tile
//   warps 8-11  thread = query row; keys 64..127 of each tile
// Tensor memory: [0,128) S_ij, [128,256) dP_ij, [256,384) dS_ij as packed
// 16-bit pairs in two buffers of 64 columns (the A operand of the dQ MMA;
// step n uses buffer n & 1), [384,384+d) dQ accumulator. MMA order per step
// n: S(n+1) once S(n) has been read, dP(n+1) once dP(n) has been read, then
// dQ += dS(n) K_n once dS(n) is in tensor memory, so that the tensor core
// computes S(n+1) and dP(n+1) while P and dS of step n are formed; with two
// dS buffers dS(n+1) does not wait for dQ(n).
#include <math.h>

#include "fa_internal.h"
#include "ptx.cuh"
#include "tile_store.cuh"

namespace fa {
namespace {

constexpr int kThreads = 384;

template <int D>
struct DqLayout {
  static constexpr int kChunks = (D + 63) / 64;  // d = 96: 2, the last half zeros
  static constexpr int kChunkBytes = kTile * 128;
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static constexpr int kKSlots = 3, kVSlots = 2;
  static constexpr int kQOff = 0;
  static constexpr int kdOOff = kQOff + kTileBytes;
  static constexpr int kKOff = kdOOff + kTileBytes;
  static constexpr int kVOff = kKOff + kKSlots * kTileBytes;
  static constexpr int kListOff = kVOff + kVSlots * kTileBytes;
  static constexpr int kBarOff = kListOff + kMaxTiles * 2;
  // q_full, k_full[3], k_empty[3], v_full[2], v_empty[2], s_full, s_free,
  // dp_full, ds_full[2][2], dq_step[2], dq_final, teardown, dp_free
  static constexpr int kNumBars = 1 + 2 * kKSlots + 2 * kVSlots + 12;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  static_assert(kBytes <= 232448, "shared memory budget");
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDS = 256, kColDQ = 384;
};

struct Bars {
  uint32_t base;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t k_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t k_empty(int s) const { return base + 8 * (4 + s); }
  __device__ uint32_t v_full(int s) const { return base + 8 * (7 + s); }
  __device__ uint32_t v_empty(int s) const { return base + 8 * (9 + s); }
  __device__ uint32_t s_full() const { return base + 8 * 11; }
  __device__ uint32_t s_free() const { return base + 8 * 12; }
  __device__ uint32_t dp_full() const { return base + 8 * 13; }
  // dS buffer b holds keys 64h + 32u .. 64h + 32u + 31 of both warpgroups h
  __device__ uint32_t ds_full(int b, int u) const {
    return base + 8 * (u ? 21 + b : (b ? 18 : 14));
  }
  __device__ uint32_t dq_step(int b) const { return base + 8 * (b ? 19 : 15); }
  __device__ uint32_t dq_final() const { return base + 8 * 16; }
  __device__ uint32_t teardown() const { return base + 8 * 17; }
  __device__ uint32_t dp_free() const { return base + 8 * 20; }
};

enum Role : uint32_t { kRoleLoad = 1, kRoleMma = 2, kRoleSoftmax = 3, kRoleInit = 5 };

// TMEM load of 32 consecutive fp32 columns into floats.
__device__ __forceinline__ void ld_cols32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  tmem_ld32(taddr, r);
  tmem_wait_ld();
#pragma unroll
  for (int x = 0; x < 32; ++x) v[x] = __uint_as_float(r[x]);
}

// kF16: f16 elements instead of bf16. D is 64, 96 or 128: at 96 the tiles keep two 64-column
// chunks (the tensor maps read zeros in columns 96..127), the MMAs run 6 K-steps over the head
// dimension and N = 96, and 96 columns of dQ are stored.
template <int D, bool kF16>
__global__ void __launch_bounds__(kThreads, 1) fa_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  using L = DqLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t s_base = smem_u32(smem);
  int *misc = reinterpret_cast<int *>(smem + L::kMiscOff);  // [0] tmem [1] count [2] abort [3] set-up loads
  if (s_base & 1023u) {  // the 128-byte swizzle needs 1024-byte aligned tiles
    if (threadIdx.x == 0 && p.status) atomicCAS(p.status, 0u, status_code(kKernBwdDq, kRoleInit, 1));
    return;
  }
  const uint32_t sQ = s_base + L::kQOff, sdO = s_base + L::kdOOff;
  const uint32_t sK = s_base + L::kKOff, sV = s_base + L::kVOff;
  uint16_t *list = reinterpret_cast<uint16_t *>(smem + L::kListOff);
  Bars bars{s_base + L::kBarOff};
  StatusSlot st{p.status, &misc[2], p.wait_limit_ns};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // CTA order: head groups of p.head_group heads; heavy Q tiles (late i for
  // causal masking) first within a group.
  const Shape &sh = p.sh;
  const int T = sh.tq;
  const int hg = p.head_group;
  const int group = blockIdx.x / (hg * T);
  const int g_base = group * hg;
  const int g_size = min(hg, sh.bh - g_base);
  const int g_rank = blockIdx.x - group * hg * T;
  const int i = T - 1 - g_rank / g_size;
  const int bh = g_base + g_rank % g_size;
  const int b_idx = bh / sh.heads, h_idx = bh % sh.heads;

  if (warp == 0 && lane == 0) {
    mbar_init(bars.q_full(), 1);
    for (int s = 0; s < L::kKSlots; ++s) {
      mbar_init(bars.k_full(s), 1);
      mbar_init(bars.k_empty(s), 1);
    }
    for (int s = 0; s < L::kVSlots; ++s) {
      mbar_init(bars.v_full(s), 1);
      mbar_init(bars.v_empty(s), 1);
    }
    mbar_init(bars.s_full(), 1);
    mbar_init(bars.s_free(), 256);
    mbar_init(bars.dp_full(), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.ds_full(b, 0), 256);
      mbar_init(bars.ds_full(b, 1), 256);
      mbar_init(bars.dq_step(b), 1);
    }
    mbar_init(bars.dp_free(), 256);
    mbar_init(bars.dq_final(), 1);
    mbar_init(bars.teardown(), 1);
    misc[2] = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
    tma_prefetch_desc(&p.tm_do);
    // Q_i and dO_i depend on blockIdx only: load them now, while the other
    // warps set up (the producer waits for them even if the list is empty);
    // so do K and V of the first list entry (the smallest visible key tile),
    // into K slot 0 and V slot 0
    int pre = 0;
    if (!(p.debug_flags & kDebugSkipLoads)) {
      mbar_arrive_expect_tx(bars.q_full(), 2 * L::kTileBytes);
      for (int c = 0; c < L::kChunks; ++c) {
        tma_load_4d(sQ + c * L::kChunkBytes, &p.tm_q, c * 64, i * kTile, h_idx, b_idx,
                    bars.q_full());
        tma_load_4d(sdO + c * L::kChunkBytes, &p.tm_do, c * 64, i * kTile, h_idx, b_idx,
                    bars.q_full());
      }
      const int jmax = sh.last_kv_tile(i);
      int j0 = -1;
      for (int j = 0; j <= jmax && j0 < 0; ++j)
        if (sh.mask_allows(i, j)) j0 = j;
      if (j0 >= 0) {
        mbar_arrive_expect_tx(bars.k_full(0), L::kTileBytes);
        mbar_arrive_expect_tx(bars.v_full(0), L::kTileBytes);
        for (int c = 0; c < L::kChunks; ++c) {
          tma_load_4d(sK + c * L::kChunkBytes, &p.tm_k, c * 64, j0 * kTile, h_idx, b_idx,
                      bars.k_full(0));
          tma_load_4d(sV + c * L::kChunkBytes, &p.tm_v, c * 64, j0 * kTile, h_idx, b_idx,
                      bars.v_full(0));
        }
        pre = 1;
      }
    }
    misc[3] = pre;  // list entries whose K and V were loaded during set-up
  } else if (warp == 1) {
    tmem_alloc(smem_u32(&misc[0]), 512);
    tmem_relinquish();
  } else if (warp == 2) {
    // K/V tiles this Q tile sees, ascending; bit 15: needs element-wise masking
    const int jmax = sh.last_kv_tile(i);
    int count = 0;
    for (int base = 0; base <= jmax; base += 32) {
      const int j = base + lane;
      const bool a = j <= jmax && sh.mask_allows(i, j);
      const uint32_t ball = __ballot_sync(0xffffffffu, a);
      if (a)
        list[count + __popc(ball & ((1u << lane) - 1u))] =
            uint16_t(j | (sh.partial(i, j) ? 1u << 15 : 0u));
      count += __popc(ball);
    }
    if (lane == 0) misc[1] = count;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  const int count = misc[1];

  if (warp == 0) {
    // ---- TMA producer: Q, dO; then K_0, and per step K_{n+1}, V_n ------------
    if (elect_one() && !(p.debug_flags & kDebugSkipLoads)) {
      bool ok = true;
      const int pre = misc[3];
      int nk = pre, nv = pre;  // tiles issued so far (entry 0's K and V may be in already)
      auto load_k = [&](int n) {
        const int s = n % L::kKSlots;
        const uint32_t u = n / L::kKSlots;
        ok = mbar_wait(bars.k_empty(s), (u & 1u) ^ 1u, st, status_code(kKernBwdDq, kRoleLoad, 1));
        if (!ok) return;
        mbar_arrive_expect_tx(bars.k_full(s), L::kTileBytes);
        const int row = (list[n] & 0x7FFF) * kTile;
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_4d(sK + s * L::kTileBytes + c * L::kChunkBytes, &p.tm_k, c * 64, row, h_idx,
                      b_idx, bars.k_full(s));
        ++nk;
      };
      auto load_v = [&](int n) {
        const int s = n % L::kVSlots;
        const uint32_t u = n / L::kVSlots;
        ok = mbar_wait(bars.v_empty(s), (u & 1u) ^ 1u, st, status_code(kKernBwdDq, kRoleLoad, 2));
        if (!ok) return;
        mbar_arrive_expect_tx(bars.v_full(s), L::kTileBytes);
        const int row = (list[n] & 0x7FFF) * kTile;
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_4d(sV + s * L::kTileBytes + c * L::kChunkBytes, &p.tm_v, c * 64, row, h_idx,
                      b_idx, bars.v_full(s));
        ++nv;
      };
      // K_j and V_j in the order the MMAs consume them: S(n+1) and dP(n+1)
      // are issued before dQ(n), so V_{n+1} must not wait behind K_{n+2}
      for (int n = pre; n < count && ok; ++n) {
        load_k(n);
        if (ok) load_v(n);
      }
      // teardown: every copy issued has landed
      mbar_wait_drain(bars.q_full(), 0, st, status_code(kKernBwdDq, kRoleLoad, 3));
      for (int s = 0; s < L::kKSlots && s < nk; ++s) {
        const int last = s + ((nk - 1 - s) / L::kKSlots) * L::kKSlots;
        mbar_wait_drain(bars.k_full(s), (last / L::kKSlots) & 1u, st, status_code(kKernBwdDq, kRoleLoad, 4));
      }
      for (int s = 0; s < L::kVSlots && s < nv; ++s) {
        const int last = s + ((nv - 1 - s) / L::kVSlots) * L::kVSlots;
        mbar_wait_drain(bars.v_full(s), (last / L::kVSlots) & 1u, st, status_code(kKernBwdDq, kRoleLoad, 5));
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- tcgen05 issuer ----------------------------------------------------
    if (elect_one()) {
      constexpr uint32_t kIdSq = idesc_f32acc(kTile, kTile, 0, 0, kF16);  // S, dP: K-major over d
      constexpr uint32_t kIdDq = idesc_f32acc(kTile, D, 0, 1, kF16);      // dS (TMEM) x K (MN-major)
      bool ok = count == 0 || mbar_wait(bars.q_full(), 0, st, status_code(kKernBwdDq, kRoleMma, 1));
      // S = Q K_n^T and dP = dO V_n^T, both operands K-major over d
      auto issue_sq = [&](uint32_t a_base, uint32_t b_base, uint32_t col) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::kChunkBytes + (kk & 3) * 32;
          mma_f16kind_ss(tmem + col, sdesc_sw128(a_base + off, 16, 1024),
                      sdesc_sw128(b_base + off, 16, 1024), kIdSq, kk > 0);
        }
      };
      if (ok && count > 0) {
        ok = mbar_wait(bars.k_full(0), 0, st, status_code(kKernBwdDq, kRoleMma, 2));
        if (ok) {
          tc_fence_after();
          issue_sq(sQ, sK, L::kColS);
          mma_commit(bars.s_full());
          ok = mbar_wait(bars.v_full(0), 0, st, status_code(kKernBwdDq, kRoleMma, 3));
        }
        if (ok) {
          tc_fence_after();
          issue_sq(sdO, sV, L::kColDP);
          mma_commit(bars.dp_full());
          mma_commit(bars.v_empty(0));
        }
      }
      for (int n = 0; n < count && ok; ++n) {
        const int ks = n % L::kKSlots;
        if (n + 1 < count) {
          // S(n+1) once the softmax warps have read S(n)
          const int ks1 = (n + 1) % L::kKSlots;
          ok = mbar_wait(bars.s_free(), n & 1, st, status_code(kKernBwdDq, kRoleMma, 4));
          if (ok) ok = mbar_wait(bars.k_full(ks1), ((n + 1) / L::kKSlots) & 1, st,
                                 status_code(kKernBwdDq, kRoleMma, 5));
          if (!ok) break;
          tc_fence_after();
          issue_sq(sQ, sK + ks1 * L::kTileBytes, L::kColS);
          mma_commit(bars.s_full());
        }
        if (n + 1 < count) {
          const int vs = (n + 1) % L::kVSlots;
          ok = mbar_wait(bars.dp_free(), n & 1, st, status_code(kKernBwdDq, kRoleMma, 9));
          if (ok) ok = mbar_wait(bars.v_full(vs), ((n + 1) / L::kVSlots) & 1, st,
                                 status_code(kKernBwdDq, kRoleMma, 7));
          if (!ok) break;
          tc_fence_after();
          issue_sq(sdO, sV + vs * L::kTileBytes, L::kColDP);
          mma_commit(bars.dp_full());
          mma_commit(bars.v_empty(vs));
        }
        const int b = n & 1;
        const uint32_t kb = sK + ks * L::kTileBytes;
        // dQ(n) in the two halves of dS(n): the first runs while the softmax
        // warps form the second
        for (int u = 0; u < 2 && ok; ++u) {
          ok = mbar_wait(bars.ds_full(b, u), (n >> 1) & 1, st,
                         status_code(kKernBwdDq, kRoleMma, u ? 10 : 6));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int kk = (e >> 1) * 4 + 2 * u + (e & 1);
            mma_f16kind_ts(tmem + L::kColDQ, tmem + L::kColDS + 64 * b + kk * 8,
                        sdesc_sw128(kb + kk * 2048, L::kChunkBytes, 1024), kIdDq,
                        (n > 0 || kk > 0) ? 1u : 0u);
          }
        }
        if (!ok) break;
        mma_commit(bars.dq_step(b));
        mma_commit(bars.k_empty(ks));
      }
      if (ok && count > 0) mma_commit(bars.dq_final());
      mma_commit(bars.teardown());
      mbar_wait_drain(bars.teardown(), 0, st, status_code(kKernBwdDq, kRoleMma, 8));
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---- P, dS for one half of the keys (thread = query row) ---------------
    const int h = (warp - 4) >> 2;                 // key half: 64h .. 64h+63
    const int r = threadIdx.x & 127;               // query row = TMEM lane
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const uint32_t t = tmem + lane_off;
    const int qrow = i * kTile + r;                // query row within the head
    const size_t grow = (size_t)bh * T * kTile + qrow;  // its workspace row
    const float c = p.scale_log2;
    const float lse2 = p.lse2[grow];               // LSE_r * log2(e)
    const float dd = p.delta[grow];                // D_r = dO_r . O_r
    bool ok = true;
    for (int n = 0; n < count && ok; ++n) {
      ok = __all_sync(0xffffffffu, mbar_wait(bars.s_full(), n & 1, st,
                                             status_code(kKernBwdDq, kRoleSoftmax, 1)));
      if (!ok) break;
      tc_fence_after();
      float pr[64];
      {
        // both loads in flight before the one wait
        uint32_t sr[2][32];
        tmem_ld32(t + L::kColS + 64 * h, sr[0]);
        tmem_ld32(t + L::kColS + 64 * h + 32, sr[1]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bars.s_free());
#pragma unroll
        for (int x = 0; x < 64; ++x) pr[x] = ex2_approx(fmaf(__uint_as_float(sr[x >> 5][x & 31]), c, -lse2));
      }
      {
        const uint32_t e = list[n];
        if (e >> 15) {  // a partial tile: keys x >= lim of this half are hidden from this row
          const int lim = sh.key_limit(i, r, int(e & 0x7FFF)) - 64 * h;
#pragma unroll
          for (int x = 0; x < 64; ++x)
            if (x >= lim) pr[x] = 0.f;
        }
      }
      ok = __all_sync(0xffffffffu, mbar_wait(bars.dp_full(), n & 1, st,
                                             status_code(kKernBwdDq, kRoleSoftmax, 2)));
      if (!ok) break;
      tc_fence_after();
      const int b = n & 1;
      {
        uint32_t dr[2][32];
        tmem_ld32(t + L::kColDP + 64 * h, dr[0]);
        tmem_ld32(t + L::kColDP + 64 * h + 32, dr[1]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bars.dp_free());
        // dS as packed 16-bit pairs (keys 2x, 2x+1 of this half), in two
        // halves of 32 keys, each announced on its own barrier
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          uint32_t dsp[16];
#pragma unroll
          for (int x = 0; x < 32; x += 2)
            dsp[x / 2] = pack2<kF16>(pr[32 * u + x] * (__uint_as_float(dr[u][x]) - dd),
                                     pr[32 * u + x + 1] * (__uint_as_float(dr[u][x + 1]) - dd));
          if (u == 0 && n >= 2) {
            // buffer b is free once the dQ MMAs of step n - 2 have read it
            ok = __all_sync(0xffffffffu, mbar_wait(bars.dq_step(b), ((n >> 1) + 1) & 1, st,
                                                   status_code(kKernBwdDq, kRoleSoftmax, 3)));
            if (!ok) break;
            tc_fence_after();
          }
          tmem_st16(t + L::kColDS + 64 * b + 32 * h + 16 * u, dsp);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bars.ds_full(b, u));
        }
      }
      if (!ok) break;
    }
    // epilogue: dQ = scale * accumulator, this half of the d columns
    if (ok && count > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(bars.dq_final(), 0, st,
                                             status_code(kKernBwdDq, kRoleSoftmax, 4)));
    // tensor-memory loads are warp-wide; rows past the sequence end store nothing
    const bool live = qrow < sh.nq;
    if (ok && D >= 96 && count > 0) {
      // each warpgroup's 64 columns leave through its chunk of the Q buffer,
      // which no MMA reads any more (count > 0: its Q load has landed; an
      // empty list stores its zeros directly below)
      tc_fence_after();
      store_rows_tma<64, kF16>(&p.tm_dq, t + L::kColDQ + h * 64, sQ + h * L::kChunkBytes, r,
                               i * kTile, h * 64, p.scale, count > 0, sh.d, sh.nq, h_idx, b_idx);
    } else if (ok) {
      tc_fence_after();
      // the first warpgroup takes columns [0, kHalf), the second [kHalf, D)
      constexpr int kHalf = D == 64 ? 32 : 64;
      uint16_t *dst_row =
          static_cast<uint16_t *>(p.dq) + p.sdq.row(b_idx, h_idx, qrow) + h * kHalf;
      const float sc = p.scale;
#pragma unroll
      for (int q = 0; q < kHalf / 32; ++q) {
        if (h * kHalf + q * 32 >= D) break;  // head dimension 96: 32 columns in the second half
        float v[32];
        if (count > 0) {
          ld_cols32(t + L::kColDQ + h * kHalf + 32 * q, v);
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) v[x] = 0.f;
        }
        uint4 *dst = reinterpret_cast<uint4 *>(dst_row + 32 * q);
#pragma unroll
        for (int x = 0; x < 4; ++x)
          if (live)
            dst[x] = make_uint4(pack2<kF16>(v[8 * x] * sc, v[8 * x + 1] * sc),
                                pack2<kF16>(v[8 * x + 2] * sc, v[8 * x + 3] * sc),
                                pack2<kF16>(v[8 * x + 4] * sc, v[8 * x + 5] * sc),
                                pack2<kF16>(v[8 * x + 6] * sc, v[8 * x + 7] * sc));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool kF16>
cudaError_t launch_dq_d(const BwdParams &p, cudaStream_t stream) {
  using L = DqLayout<D>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(fa_bwd_dq_kernel<D, kF16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  LaunchProbe probe(kKindBwdDq, stream);
  fa_bwd_dq_kernel<D, kF16><<<p.sh.tq * p.sh.bh, kThreads, L::kBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward_dq(const BwdParams &p, cudaStream_t stream) {
  const bool f16 = p.sh.f16 != 0;
  if (p.sh.d == 64) return f16 ? launch_dq_d<64, true>(p, stream) : launch_dq_d<64, false>(p, stream);
  if (p.sh.d == 96) return f16 ? launch_dq_d<96, true>(p, stream) : launch_dq_d<96, false>(p, stream);
  if (p.sh.d == 128)
    return f16 ? launch_dq_d<128, true>(p, stream) : launch_dq_d<128, false>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
