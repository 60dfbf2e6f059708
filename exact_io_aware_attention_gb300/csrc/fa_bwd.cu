// Attention backward for sm_103a, by recomputation.
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
// Three kernels on the caller's stream:
//   fa_bwd_pre   D_i, LSE_i * log2(e), and a zeroed fp32 dQ accumulator
//   fa_bwd_main  one CTA per 128-key K/V tile; loops over the Q tiles that
//                see it (causal: i >= j; block-sparse: mask[i][j] != 0)
//   fa_bwd_dq    dQ = bf16(scale * dQ accumulator)
//
// fa_bwd_main, 12 warps:
//   warp 0      TMA producer: K_j, V_j once; Q_i, dO_i, LSE_i, D_i per step (2 stages)
//   warp 1      tcgen05 issuer (one lane) and tensor-memory owner
//   warps 4-7   thread = key row: P^T from S^T, dS^T from dP^T, then dV out
//   warps 8-11  dQ partial of each step -> fp32 reductions into global; then dK out
// Tensor memory (512 columns): [0,128) S^T, [128,256) dP^T, then dV and dK
// (d columns each). With d = 128 the dQ^T partial (d lanes x 128 queries)
// reuses the dP^T columns once dS^T has been formed; with d = 64 the dQ
// partial (128 queries x 64) has its own columns at 384.
// Shared memory: K_j, V_j, Q_i[2], dO_i[2], one bf16 [keys][queries] tile that
// holds P^T and then dS^T of the current step, LSE and D of the current step.
#include <math.h>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 384;

template <int D>
struct BwdLayout {
  static constexpr int kChunks = D / 64;
  static constexpr int kChunkBytes = kTile * 128;
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kTileBytes;
  static constexpr int kQOff = kVOff + kTileBytes;       // 2 stages
  static constexpr int kdOOff = kQOff + 2 * kTileBytes;  // 2 stages
  static constexpr int kDSOff = kdOOff + 2 * kTileBytes; // bf16 [128 keys][128 queries]
  static constexpr int kDSBytes = kTile * kTile * 2;
  static constexpr int kStatOff = kDSOff + kDSBytes;     // [2 stages][lse2 128 | delta 128] fp32
  static constexpr int kStatBytes = 2 * kTile * 4;
  static constexpr int kBarOff = kStatOff + 2 * kStatBytes;
  static constexpr int kNumBars = 14;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  static_assert(kBytes <= 232448, "shared memory budget");
  // tensor memory columns
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
  static constexpr bool kDqAlias = (D == 128);          // dQ^T in the dP^T columns
  static constexpr uint32_t kColDQ = kDqAlias ? kColDP : 384;
};

struct Bars {
  uint32_t base;
  __device__ uint32_t kv_full() const { return base; }
  __device__ uint32_t q_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t q_empty(int s) const { return base + 8 * (3 + s); }
  __device__ uint32_t s_full() const { return base + 8 * 5; }
  __device__ uint32_t p_full() const { return base + 8 * 6; }
  __device__ uint32_t dp_full() const { return base + 8 * 7; }
  __device__ uint32_t dv_done() const { return base + 8 * 8; }
  __device__ uint32_t ds_full() const { return base + 8 * 9; }
  __device__ uint32_t dq_full() const { return base + 8 * 10; }
  __device__ uint32_t dq_free() const { return base + 8 * 11; }
  __device__ uint32_t acc_done() const { return base + 8 * 12; }
  __device__ uint32_t teardown() const { return base + 8 * 13; }
};

enum Role : uint32_t { kRoleLoad = 1, kRoleMma = 2, kRoleSoftmax = 3, kRoleDq = 4, kRoleInit = 5 };

// Next Q tile at or after i that sees K/V tile j (T if none).
__device__ __forceinline__ int next_q(const BwdParams &p, int i, int j, int T) {
  if (p.mask)
    while (i < T && p.mask[(size_t)i * T + j] == 0) ++i;
  return i;
}

__device__ __forceinline__ uint32_t ds_addr(uint32_t base, int row, int unit16) {
  // bf16 [row][128 cols] as two 64-column chunks, 128-byte swizzle
  return base + (unit16 >> 3) * (kTile * 128) + row * 128 + (((unit16 & 7) ^ (row & 7)) << 4);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) fa_bwd_main(const __grid_constant__ BwdParams p) {
  using L = BwdLayout<D>;
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
  const uint32_t sDS = s_base + L::kDSOff;
  const float *stat = reinterpret_cast<const float *>(smem + L::kStatOff);
  Bars bars{s_base + L::kBarOff};
  StatusSlot st{p.status, &misc[2]};

  const int warp = threadIdx.x >> 5;
  const int T = p.n / kTile;
  // CTAs are ordered head group by head group (p.head_group heads at a time),
  // so that the fp32 dQ rows being accumulated by concurrent CTAs stay in L2;
  // within a group the heavy K/V tiles come first (causal: tile j sees T - j
  // Q tiles).
  const int hg = p.head_group;
  const int group = blockIdx.x / (hg * T);
  const int g_base = group * hg;
  const int g_size = min(hg, p.bh - g_base);
  const int g_rank = blockIdx.x - group * hg * T;
  const int j = g_rank / g_size;
  const int bh = g_base + g_rank % g_size;
  const int first = next_q(p, p.causal ? j : 0, j, T);
  const bool any = first < T;
  const size_t kvrow = (size_t)bh * p.n + (size_t)j * kTile;

  if (warp == 0 && (threadIdx.x & 31) == 0) {
    mbar_init(bars.kv_full(), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bars.q_full(s), 1);
      mbar_init(bars.q_empty(s), 1);
    }
    mbar_init(bars.s_full(), 1);
    mbar_init(bars.p_full(), 128);
    mbar_init(bars.dp_full(), 1);
    mbar_init(bars.dv_done(), 1);
    mbar_init(bars.ds_full(), 128);
    mbar_init(bars.dq_full(), 1);
    mbar_init(bars.dq_free(), 128);
    mbar_init(bars.acc_done(), 1);
    mbar_init(bars.teardown(), 1);
    misc[2] = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
    tma_prefetch_desc(&p.tm_do);
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
    if (elect_one() && any) {
      mbar_arrive_expect_tx(bars.kv_full(), 2 * L::kTileBytes);
      for (int c = 0; c < L::kChunks; ++c) {
        tma_load_2d(sK + c * L::kChunkBytes, &p.tm_k, c * 64, (int)kvrow, bars.kv_full());
        tma_load_2d(sV + c * L::kChunkBytes, &p.tm_v, c * 64, (int)kvrow, bars.kv_full());
      }
      int n = 0;
      bool ok = true;
      for (int i = first; i < T && ok; i = next_q(p, i + 1, j, T), ++n) {
        const int s = n & 1;
        const uint32_t u = n >> 1;
        ok = mbar_wait(bars.q_empty(s), (u & 1u) ^ 1u, st, status_code(kKernBwd, kRoleLoad, 1));
        if (!ok) break;
        const size_t qrow = (size_t)bh * p.n + (size_t)i * kTile;
        mbar_arrive_expect_tx(bars.q_full(s), 2 * L::kTileBytes + L::kStatBytes);
        for (int c = 0; c < L::kChunks; ++c) {
          tma_load_2d(sQ + s * L::kTileBytes + c * L::kChunkBytes, &p.tm_q, c * 64, (int)qrow,
                      bars.q_full(s));
          tma_load_2d(sdO + s * L::kTileBytes + c * L::kChunkBytes, &p.tm_do, c * 64, (int)qrow,
                      bars.q_full(s));
        }
        const uint32_t sst = s_base + L::kStatOff + s * L::kStatBytes;
        bulk_load_1d(sst, p.lse2 + qrow, kTile * 4, bars.q_full(s));
        bulk_load_1d(sst + kTile * 4, p.delta + qrow, kTile * 4, bars.q_full(s));
      }
      // teardown: every copy issued has landed
      mbar_wait(bars.kv_full(), 0, st, status_code(kKernBwd, kRoleLoad, 2));
      for (int s = 0; s < 2 && s < n; ++s) {
        const int last = s + ((n - 1 - s) / 2) * 2;
        mbar_wait(bars.q_full(s), (last >> 1) & 1u, st, status_code(kKernBwd, kRoleLoad, 3));
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- tcgen05 issuer ----------------------------------------------------
    if (elect_one()) {
      constexpr uint32_t kIdSq = idesc_bf16_f32(kTile, kTile, 0, 0);  // S^T, dP^T
      constexpr uint32_t kIdAcc = idesc_bf16_f32(kTile, D, 0, 1);     // dV, dK: B MN-major
      // dQ^T = K^T dS^T (M = d) for d = 128; dQ = dS K (M = 128 queries) for d = 64
      constexpr uint32_t kIdDq = L::kDqAlias ? idesc_bf16_f32(kTile, kTile, 1, 1)
                                             : idesc_bf16_f32(kTile, D, 1, 1);
      bool ok = !any || mbar_wait(bars.kv_full(), 0, st, status_code(kKernBwd, kRoleMma, 1));
      // S^T(i) = K_j Q_i^T: both operands K-major over d
      auto issue_s = [&](int s) {
        const uint32_t q = sQ + s * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::kChunkBytes + (kk & 3) * 32;
          mma_bf16_ss(tmem + L::kColS, sdesc_sw128(sK + off, 16, 1024),
                      sdesc_sw128(q + off, 16, 1024), kIdSq, kk > 0);
        }
      };
      int n = 0;
      if (ok && any) {
        ok = mbar_wait(bars.q_full(0), 0, st, status_code(kKernBwd, kRoleMma, 2));
        if (ok) {
          tc_fence_after();
          issue_s(0);
          mma_commit(bars.s_full());
        }
      }
      for (int i = first; i < T && ok; ++n) {
        const int s = n & 1;
        const int inext = next_q(p, i + 1, j, T);
        const uint32_t q = sQ + s * L::kTileBytes, dO = sdO + s * L::kTileBytes;
        // dP^T = V_j dO_i^T (its columns hold the previous dQ^T when aliased)
        if (L::kDqAlias && n > 0) {
          ok = mbar_wait(bars.dq_free(), (n - 1) & 1, st, status_code(kKernBwd, kRoleMma, 3));
          if (!ok) break;
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::kChunkBytes + (kk & 3) * 32;
          mma_bf16_ss(tmem + L::kColDP, sdesc_sw128(sV + off, 16, 1024),
                      sdesc_sw128(dO + off, 16, 1024), kIdSq, kk > 0);
        }
        mma_commit(bars.dp_full());
        // dV += P^T dO_i once P^T is in shared memory
        ok = mbar_wait(bars.p_full(), n & 1, st, status_code(kKernBwd, kRoleMma, 4));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint32_t a_off = (kk >> 2) * L::kChunkBytes + (kk & 3) * 32;
          mma_bf16_ss(tmem + L::kColDV, sdesc_sw128(sDS + a_off, 16, 1024),
                      sdesc_sw128(dO + kk * 2048, L::kChunkBytes, 1024), kIdAcc,
                      (n > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bars.dv_done());
        // S^T of the next Q tile, overlapping the dS^T work of this one
        if (inext < T) {
          const int s1 = (n + 1) & 1;
          ok = mbar_wait(bars.q_full(s1), ((n + 1) >> 1) & 1, st, status_code(kKernBwd, kRoleMma, 5));
          if (!ok) break;
          tc_fence_after();
          issue_s(s1);
          mma_commit(bars.s_full());
        }
        // dK += dS^T Q_i and the dQ partial once dS^T is in shared memory
        ok = mbar_wait(bars.ds_full(), n & 1, st, status_code(kKernBwd, kRoleMma, 6));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint32_t a_off = (kk >> 2) * L::kChunkBytes + (kk & 3) * 32;
          mma_bf16_ss(tmem + L::kColDK, sdesc_sw128(sDS + a_off, 16, 1024),
                      sdesc_sw128(q + kk * 2048, L::kChunkBytes, 1024), kIdAcc,
                      (n > 0 || kk > 0) ? 1u : 0u);
        }
        if (!L::kDqAlias && n > 0) {
          ok = mbar_wait(bars.dq_free(), (n - 1) & 1, st, status_code(kKernBwd, kRoleMma, 7));
          if (!ok) break;
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          // K dimension = keys: both operands are MN-major, 16 key rows per step
          if (L::kDqAlias)
            mma_bf16_ss(tmem + L::kColDQ, sdesc_sw128(sK + kk * 2048, L::kChunkBytes, 1024),
                        sdesc_sw128(sDS + kk * 2048, L::kChunkBytes, 1024), kIdDq, kk > 0);
          else
            mma_bf16_ss(tmem + L::kColDQ, sdesc_sw128(sDS + kk * 2048, L::kChunkBytes, 1024),
                        sdesc_sw128(sK + kk * 2048, L::kChunkBytes, 1024), kIdDq, kk > 0);
        }
        mma_commit(bars.dq_full());
        mma_commit(bars.q_empty(s));
        i = inext;
      }
      if (ok) mma_commit(bars.acc_done());
      mma_commit(bars.teardown());
      mbar_wait(bars.teardown(), 0, st, status_code(kKernBwd, kRoleMma, 8));
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 8) {
    // ---- P^T and dS^T (thread = key row) -----------------------------------
    const int kr = threadIdx.x - 128;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const float c = p.scale_log2;
    bool ok = true;
    int n = 0;
    for (int i = first; i < T && ok; i = next_q(p, i + 1, j, T), ++n) {
      const int s = n & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(bars.s_full(), n & 1, st,
                                             status_code(kKernBwd, kRoleSoftmax, 1)));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bars.q_full(s), (n >> 1) & 1, st,
                                                     status_code(kKernBwd, kRoleSoftmax, 2)));
      if (!ok) break;
      tc_fence_after();
      const float *lse2 = stat + s * 2 * kTile;
      const float *delta = lse2 + kTile;
      // P^T_kq = exp2(s_kq * scale * log2e - LSE_q * log2e); hidden entries 0.
      // S^T is read 32 columns at a time to keep register pressure low.
      const bool diag = p.causal && i == j;
      uint32_t pk[64];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t sr[32];
        tmem_ld32(tmem + lane_off + L::kColS + q * 32, sr);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 32; x += 2) {
          const int col = 32 * q + x;
          const float2 l2 = *reinterpret_cast<const float2 *>(lse2 + col);
          float p0 = ex2_approx(fmaf(__uint_as_float(sr[x]), c, -l2.x));
          float p1 = ex2_approx(fmaf(__uint_as_float(sr[x + 1]), c, -l2.y));
          if (diag) {
            if (col < kr) p0 = 0.f;
            if (col + 1 < kr) p1 = 0.f;
          }
          pk[col >> 1] = pack_bf16x2(p0, p1);
        }
      }
      // the shared P^T/dS^T tile is free once the previous dK/dQ MMAs are done
      if (n > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(bars.dq_full(), (n - 1) & 1, st,
                                               status_code(kKernBwd, kRoleSoftmax, 3)));
        if (!ok) break;
      }
#pragma unroll
      for (int u = 0; u < 16; ++u)
        st_shared_v4(ds_addr(sDS, kr, u), pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bars.p_full());
      // dS^T_kq = P^T_kq (dP^T_kq - D_q), written over P^T once dV has read it
      ok = __all_sync(0xffffffffu, mbar_wait(bars.dp_full(), n & 1, st,
                                             status_code(kKernBwd, kRoleSoftmax, 4)));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bars.dv_done(), n & 1, st,
                                                     status_code(kKernBwd, kRoleSoftmax, 5)));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t dp[32];
        tmem_ld32(tmem + lane_off + L::kColDP + q * 32, dp);
        tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 4; ++u) {  // 16-byte unit 4q+u: queries 32q+8u .. +7
          uint32_t w[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const int x = 32 * q + 8 * u + 2 * h;
            const uint32_t pp = pk[x >> 1];
            const float p0 = __uint_as_float(pp << 16), p1 = __uint_as_float(pp & 0xffff0000u);
            const float d0 = p0 * (__uint_as_float(dp[8 * u + 2 * h]) - delta[x]);
            const float d1 = p1 * (__uint_as_float(dp[8 * u + 2 * h + 1]) - delta[x + 1]);
            w[h] = pack_bf16x2(d0, d1);
          }
          st_shared_v4(ds_addr(sDS, kr, 4 * q + u), w[0], w[1], w[2], w[3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bars.ds_full());
    }
    // epilogue: dV rows of this K/V tile
    if (ok && any)
      ok = __all_sync(0xffffffffu, mbar_wait(bars.acc_done(), 0, st,
                                             status_code(kKernBwd, kRoleSoftmax, 6)));
    if (ok) {
      tc_fence_after();
      uint16_t *dst_row = static_cast<uint16_t *>(p.dv) + (kvrow + kr) * D;
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        uint32_t v[32];
        if (any) {
          tmem_ld32(tmem + lane_off + L::kColDV + q * 32, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) v[x] = 0u;
        }
        uint4 *dst = reinterpret_cast<uint4 *>(dst_row + q * 32);
#pragma unroll
        for (int x = 0; x < 4; ++x)
          dst[x] = make_uint4(
              pack_bf16x2(__uint_as_float(v[8 * x + 0]), __uint_as_float(v[8 * x + 1])),
              pack_bf16x2(__uint_as_float(v[8 * x + 2]), __uint_as_float(v[8 * x + 3])),
              pack_bf16x2(__uint_as_float(v[8 * x + 4]), __uint_as_float(v[8 * x + 5])),
              pack_bf16x2(__uint_as_float(v[8 * x + 6]), __uint_as_float(v[8 * x + 7])));
      }
    }
  } else if (warp >= 8) {
    // ---- dQ partials -> fp32 reductions; then dK rows ------------------------
    const int ln = threadIdx.x - 256;  // TMEM lane
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    bool ok = true;
    int n = 0;
    for (int i = first; i < T && ok; i = next_q(p, i + 1, j, T), ++n) {
      ok = __all_sync(0xffffffffu, mbar_wait(bars.dq_full(), n & 1, st,
                                             status_code(kKernBwd, kRoleDq, 1)));
      if (!ok) break;
      tc_fence_after();
      const size_t qrow = (size_t)bh * p.n + (size_t)i * kTile;
      if (L::kDqAlias) {
        // lane = d index, columns = the 128 queries: one 128-byte line per warp and query
        float *acc = p.dq_acc + qrow * D + ln;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + L::kColDQ + q * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int x = 0; x < 32; ++x) atomicAdd(acc + (size_t)(32 * q + x) * D, __uint_as_float(v[x]));
        }
      } else {
        // lane = query row, columns = d
        float4 *acc = reinterpret_cast<float4 *>(p.dq_acc + (qrow + ln) * D);
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + L::kColDQ + q * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int x = 0; x < 8; ++x)
            atomicAdd(acc + q * 8 + x,
                      make_float4(__uint_as_float(v[4 * x]), __uint_as_float(v[4 * x + 1]),
                                  __uint_as_float(v[4 * x + 2]), __uint_as_float(v[4 * x + 3])));
        }
      }
      tc_fence_before();
      mbar_arrive(bars.dq_free());
    }
    // epilogue: dK rows of this K/V tile (scaled)
    if (ok && any)
      ok = __all_sync(0xffffffffu, mbar_wait(bars.acc_done(), 0, st,
                                             status_code(kKernBwd, kRoleDq, 2)));
    if (ok) {
      tc_fence_after();
      uint16_t *dst_row = static_cast<uint16_t *>(p.dk) + (kvrow + ln) * D;
      const float sc = p.scale;
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        uint32_t v[32];
        if (any) {
          tmem_ld32(tmem + lane_off + L::kColDK + q * 32, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) v[x] = 0u;
        }
        uint4 *dst = reinterpret_cast<uint4 *>(dst_row + q * 32);
#pragma unroll
        for (int x = 0; x < 4; ++x)
          dst[x] = make_uint4(
              pack_bf16x2(__uint_as_float(v[8 * x + 0]) * sc, __uint_as_float(v[8 * x + 1]) * sc),
              pack_bf16x2(__uint_as_float(v[8 * x + 2]) * sc, __uint_as_float(v[8 * x + 3]) * sc),
              pack_bf16x2(__uint_as_float(v[8 * x + 4]) * sc, __uint_as_float(v[8 * x + 5]) * sc),
              pack_bf16x2(__uint_as_float(v[8 * x + 6]) * sc, __uint_as_float(v[8 * x + 7]) * sc));
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

// D_i = dO_i . O_i, LSE_i * log2(e) (0 for a row that sees no key), zero dQ_acc.
// Thread = 8 consecutive elements of a row (16-byte loads).
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre(const __grid_constant__ BwdParams p) {
  constexpr int kLanesPerRow = D / 8;
  const size_t rows = (size_t)p.bh * p.n;
  const size_t gt = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t row = gt / kLanesPerRow;
  const int part = int(gt % kLanesPerRow);
  float acc = 0.f;
  if (row < rows) {
    const uint4 o = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.o) + row * D + part * 8);
    const uint4 g = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.dout) + row * D + part * 8);
    const uint32_t ow[4] = {o.x, o.y, o.z, o.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      acc = fmaf(__uint_as_float(ow[h] << 16), __uint_as_float(gw[h] << 16), acc);
      acc = fmaf(__uint_as_float(ow[h] & 0xffff0000u), __uint_as_float(gw[h] & 0xffff0000u), acc);
    }
    float4 *z = reinterpret_cast<float4 *>(p.dq_acc + row * D + part * 8);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int off = kLanesPerRow / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && part == 0) {
    p.delta[row] = acc;
    const float l = p.lse[row];
    p.lse2[row] = isinf(l) ? 0.f : l * 1.4426950408889634f;
  }
}

// dQ = bf16(scale * dQ_acc), 8 elements per thread.
__global__ void __launch_bounds__(256) fa_bwd_dq(const __grid_constant__ BwdParams p) {
  const size_t total8 = (size_t)p.bh * p.n * p.d / 8;
  const size_t gt = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gt >= total8) return;
  const float4 *src = reinterpret_cast<const float4 *>(p.dq_acc) + 2 * gt;
  const float4 a = src[0], b = src[1];
  const float sc = p.scale;
  reinterpret_cast<uint4 *>(p.dq)[gt] =
      make_uint4(pack_bf16x2(a.x * sc, a.y * sc), pack_bf16x2(a.z * sc, a.w * sc),
                 pack_bf16x2(b.x * sc, b.y * sc), pack_bf16x2(b.z * sc, b.w * sc));
}

template <int D>
cudaError_t launch_bwd_d(const BwdParams &p, cudaStream_t stream) {
  using L = BwdLayout<D>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(fa_bwd_main<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::kBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const size_t rows = (size_t)p.bh * p.n;
  const size_t pre_threads = rows * (D / 8);
  {
    LaunchProbe probe(kKindBwdPre, stream);
    fa_bwd_pre<D><<<(unsigned)((pre_threads + 255) / 256), 256, 0, stream>>>(p);
  }
  const int T = p.n / kTile;
  {
    LaunchProbe probe(kKindBwdMain, stream);
    fa_bwd_main<D><<<T * p.bh, kThreads, L::kBytes, stream>>>(p);
  }
  const size_t total8 = rows * D / 8;
  {
    LaunchProbe probe(kKindBwdDq, stream);
    fa_bwd_dq<<<(unsigned)((total8 + 255) / 256), 256, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward(const BwdParams &p, cudaStream_t stream) {
  if (p.d == 64) return launch_bwd_d<64>(p, stream);
  if (p.d == 128) return launch_bwd_d<128>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
