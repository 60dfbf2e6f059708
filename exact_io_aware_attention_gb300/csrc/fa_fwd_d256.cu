// Attention forward for head dimension 256 on sm_103a.
//
// The method is the one of fa_fwd.cu: the tiled forward pass with online
// softmax of "Paper Notes: FlashAttention" ("Tiling: Block-by-Block Softmax"),
// in the unnormalised-accumulator form of the numpy flash_attention in "flash
// attention" (muhibwaqar.com, "build it from scratch") and of the aicassindra
// page ("Rescale and accumulate: the forward pass in one loop"), with the same
// masks, statistics, split over the keys and epilogue. Only the tiling
// differs, because a 128 x 256 output takes half of the tensor memory:
//
// CTA = one 128-row Q tile of one head. 8 warps:
//   warp 0      TMA producer: Q once (4 boxes of 64 columns), then K_j and
//               V_j as 128-column halves through a ring of 5 32 KB slots, in
//               the order the MMAs consume them: K_0, K_1, V_0, K_2, V_1, ...
//               (Q and K_0 are issued during set-up, before the CTA barrier)
//   warp 1      tcgen05 issuer (one lane) and tensor-memory owner
//   warp 2      builds the list of K/V tiles to visit
//   warps 4-7   softmax, thread = query row = TMEM lane
// Tensor memory (512 columns): S in two buffers [0,128) and [128,256), O in
// [256,512). P (16-bit pairs) is written over the first 64 columns of its S
// buffer. MMA order: S(0), S(1), then per tile n: PV(n), S(n+2); the tensor
// core computes S(n+1) while the softmax of tile n runs, and S(n+2) is issued
// after PV(n) has been issued, so it overwrites P(n) only after PV(n) read it.
// A 16-bit O leaves through the Q buffer with TMA stores (tile_store.cuh).
#include <math.h>

#include "fa_internal.h"
#include "ptx.cuh"
#include "tile_store.cuh"

namespace fa {
namespace {

constexpr int kThreads = 256;
constexpr int D = 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units, as in fa_fwd.cu

struct Layout {
  static constexpr int kChunkBytes = kTile * 128;        // 128 rows x 64 columns
  static constexpr int kQBytes = 4 * kChunkBytes;        // Q tile: 4 chunks
  static constexpr int kSlotBytes = 2 * kChunkBytes;     // half a K or V tile: 128 columns
  static constexpr int kSlots = 5;
  static constexpr int kQOff = 0;
  static constexpr int kRingOff = kQOff + kQBytes;
  static constexpr int kListOff = kRingOff + kSlots * kSlotBytes;
  static constexpr int kBarOff = kListOff + kMaxTiles * 2;
  // q_full, full[5], empty[5], s_full[2], p_full[2], pv_done, o_done, teardown
  static constexpr int kNumBars = 1 + 2 * kSlots + 2 + 2 + 3;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes + 1024;           // slack to align the base to 1024 B
  static_assert(kAlloc <= 232448, "shared memory budget");
  static constexpr uint32_t kColO = 256;
};

struct Bars {
  uint32_t base;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t empty(int s) const { return base + 8 * (1 + Layout::kSlots + s); }
  __device__ uint32_t s_full(int b) const { return base + 8 * (1 + 2 * Layout::kSlots + b); }
  __device__ uint32_t p_full(int b) const { return base + 8 * (3 + 2 * Layout::kSlots + b); }
  __device__ uint32_t pv_done() const { return base + 8 * (5 + 2 * Layout::kSlots); }
  __device__ uint32_t o_done() const { return base + 8 * (6 + 2 * Layout::kSlots); }
  __device__ uint32_t teardown() const { return base + 8 * (7 + 2 * Layout::kSlots); }
};

enum Role : uint32_t { kRoleLoad = 1, kRoleMma = 2, kRoleSoftmax = 3 };

// Ring positions (loads and MMAs take the halves in one order: K_0, then per
// tile n K_{n+1} (if any) and V_n) of half h of K_j and of V_n, with `count`
// tiles in the list.
__device__ __forceinline__ int kpos(int j, int h) { return j == 0 ? h : 4 * j - 2 + h; }
__device__ __forceinline__ int vpos(int n, int h, int count) {
  return (n + 1 < count ? 4 * n + 4 : 4 * n + 2) + h;
}

template <bool kSplit, bool kF16>
__global__ void __launch_bounds__(kThreads, 1) fa_fwd_d256_kernel(const __grid_constant__ FwdParams p) {
  using L = Layout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = smem_u32(smem);
  const uint32_t sQ = s_base + L::kQOff;
  const uint32_t sRing = s_base + L::kRingOff;
  uint16_t *list = reinterpret_cast<uint16_t *>(smem + L::kListOff);
  int *misc = reinterpret_cast<int *>(smem + L::kMiscOff);  // [0] tmem base [1] count [2] abort [3] loads in set-up
  Bars bars{s_base + L::kBarOff};
  StatusSlot st{p.status, &misc[2], p.wait_limit_ns};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // work item: head groups, heavy (late) Q tiles first within a group; splits adjacent
  const Shape &sh = p.sh;
  const int n_split = kSplit ? p.n_split : 1;
  const int split = kSplit ? int(blockIdx.x % n_split) : 0;
  const int cta = kSplit ? int(blockIdx.x / n_split) : int(blockIdx.x);
  int i;  // Q tile
  const int bh = fwd_item_head(cta, sh.bh, sh.tq, p.head_group, &i);
  const int b_idx = bh / sh.heads, h_idx = bh % sh.heads;

  // ---- setup -------------------------------------------------------------
  if (warp == 0 && lane == 0) {
    mbar_init(bars.q_full(), 1);
    for (int s = 0; s < L::kSlots; ++s) {
      mbar_init(bars.full(s), 1);
      mbar_init(bars.empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.s_full(b), 1);
      mbar_init(bars.p_full(b), 128);
    }
    mbar_init(bars.pv_done(), 1);
    mbar_init(bars.o_done(), 1);
    mbar_init(bars.teardown(), 1);
    misc[2] = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
    // Q and the first K tile of the list (the smallest key tile this Q tile
    // sees) do not depend on the list: load them now, while the other warps
    // set up. A split CTA starts further into the list, known only later.
    int pre = 0;
    if constexpr (!kSplit) {
      const int jmax = sh.last_kv_tile(i);
      int j0 = -1;
      for (int j = 0; j <= jmax && j0 < 0; ++j)
        if (sh.mask_allows(i, j)) j0 = j;
      if (j0 >= 0 && !(p.debug_flags & kDebugSkipLoads)) {
        mbar_arrive_expect_tx(bars.q_full(), L::kQBytes);
        for (int c = 0; c < 4; ++c)
          tma_load_4d(sQ + c * L::kChunkBytes, &p.tm_q, c * 64, i * kTile, h_idx, b_idx,
                      bars.q_full());
        for (int h = 0; h < 2; ++h) {  // ring positions 0 and 1: K_{j0}, both halves
          mbar_arrive_expect_tx(bars.full(h), L::kSlotBytes);
          for (int c = 0; c < 2; ++c)
            tma_load_4d(sRing + h * L::kSlotBytes + c * L::kChunkBytes, &p.tm_k, h * 128 + c * 64,
                        j0 * kTile, h_idx, b_idx, bars.full(h));
        }
        pre = 2;
      }
    }
    misc[3] = pre;  // ring positions (and Q) already issued
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
    if constexpr (kSplit) {
      // this CTA's share, entries [lo, hi), moves to the front (ascending
      // chunks: a chunk's writes land below every later source)
      const int lo = int((long long)count * split / n_split);
      const int hi = int((long long)count * (split + 1) / n_split);
      __syncwarp();
      for (int base = 0; lo > 0 && base < hi - lo; base += 32) {
        const bool in = base + lane < hi - lo;
        const uint16_t v = in ? list[lo + base + lane] : uint16_t(0);
        __syncwarp();
        if (in) list[base + lane] = v;
        __syncwarp();
      }
      count = hi - lo;
    }
    if (lane == 0) misc[1] = count;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  const int count = misc[1];

  if (warp == 0) {
    // ---- TMA producer ------------------------------------------------------
    if (elect_one() && count > 0 && !(p.debug_flags & kDebugSkipLoads)) {
      const int pre = misc[3];
      if (pre == 0) {
        mbar_arrive_expect_tx(bars.q_full(), L::kQBytes);
        for (int c = 0; c < 4; ++c)
          tma_load_4d(sQ + c * L::kChunkBytes, &p.tm_q, c * 64, i * kTile, h_idx, b_idx,
                      bars.q_full());
      }
      bool ok = true;
      int issued = pre;  // == the ring position of the next load
      // one half (h) of K_j or V_j into the next ring slot
      auto load_half = [&](const CUtensorMap *tm, int j, int h) {
        const int s = issued % L::kSlots;
        ok = mbar_wait(bars.empty(s), ((issued / L::kSlots) & 1u) ^ 1u, st,
                       status_code(kKernFwd, kRoleLoad, 1));
        if (!ok) return;
        mbar_arrive_expect_tx(bars.full(s), L::kSlotBytes);
        const int row = (list[j] & 0x7FFF) * kTile;
        for (int c = 0; c < 2; ++c)
          tma_load_4d(sRing + s * L::kSlotBytes + c * L::kChunkBytes, tm, h * 128 + c * 64, row,
                      h_idx, b_idx, bars.full(s));
        ++issued;
      };
      for (int h = pre; h < 2 && ok; ++h) load_half(&p.tm_k, 0, h);
      for (int n = 0; n < count && ok; ++n) {
        for (int h = 0; h < 2 && ok && n + 1 < count; ++h) load_half(&p.tm_k, n + 1, h);
        for (int h = 0; h < 2 && ok; ++h) load_half(&p.tm_v, n, h);
      }
      // teardown: every copy issued has landed
      mbar_wait_drain(bars.q_full(), 0, st, status_code(kKernFwd, kRoleLoad, 2));
      for (int s = 0; s < L::kSlots && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / L::kSlots) * L::kSlots;
        mbar_wait_drain(bars.full(s), (last / L::kSlots) & 1u, st, status_code(kKernFwd, kRoleLoad, 3));
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- tcgen05 issuer ----------------------------------------------------
    if (elect_one()) {
      constexpr uint32_t kIdS = idesc_f32acc(kTile, kTile, 0, 0, kF16);   // Q K^T, K-major
      constexpr uint32_t kIdPV = idesc_f32acc(kTile, kTile, 0, 1, kF16);  // P V-half, V MN-major
      bool ok = count == 0 || mbar_wait(bars.q_full(), 0, st, status_code(kKernFwd, kRoleMma, 1));

      // S(n) = Q K_n^T over 256 columns: 8 k-steps per K half
      auto issue_s = [&](int n) -> bool {
        const uint32_t d_col = tmem + (n & 1) * kTile;
        for (int h = 0; h < 2; ++h) {
          const int pos = kpos(n, h);
          const int s = pos % L::kSlots;
          if (!mbar_wait(bars.full(s), (pos / L::kSlots) & 1u, st,
                         status_code(kKernFwd, kRoleMma, 2 + h)))
            return false;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * L::kChunkBytes + (kk & 3) * 32;
            mma_f16kind_ss(d_col, sdesc_sw128(sQ + h * 2 * L::kChunkBytes + off, 16, 1024),
                           sdesc_sw128(sRing + s * L::kSlotBytes + off, 16, 1024), kIdS,
                           (h > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bars.empty(s));
        }
        mma_commit(bars.s_full(n & 1));
        return true;
      };
      // O[:, 128h .. 128h+127] += P(n) V_n[:, 128h ..]: A = P from tensor
      // memory (8 columns per 16 keys), B = the V half with keys as K
      auto issue_pv = [&](int n) -> bool {
        const uint32_t p_col = tmem + (n & 1) * kTile;
        for (int h = 0; h < 2; ++h) {
          const int pos = vpos(n, h, count);
          const int s = pos % L::kSlots;
          if (!mbar_wait(bars.full(s), (pos / L::kSlots) & 1u, st,
                         status_code(kKernFwd, kRoleMma, 4 + h)))
            return false;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_f16kind_ts(tmem + L::kColO + h * kTile, p_col + kk * 8,
                           sdesc_sw128(sRing + s * L::kSlotBytes + kk * 2048, L::kChunkBytes, 1024),
                           kIdPV, (n > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bars.empty(s));
        }
        mma_commit(bars.pv_done());
        return true;
      };

      if (ok && count > 0) ok = issue_s(0);
      if (ok && count > 1) ok = issue_s(1);
      for (int n = 0; n < count && ok; ++n) {
        ok = mbar_wait(bars.p_full(n & 1), (n >> 1) & 1u, st, status_code(kKernFwd, kRoleMma, 6));
        if (!ok) break;
        tc_fence_after();
        ok = issue_pv(n);
        if (ok && n + 2 < count) ok = issue_s(n + 2);
      }
      if (ok && count > 0) mma_commit(bars.o_done());
      // teardown: every MMA this thread issued has completed
      mma_commit(bars.teardown());
      mbar_wait_drain(bars.teardown(), 0, st, status_code(kKernFwd, kRoleMma, 8));
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---- softmax -----------------------------------------------------------
    const int r = threadIdx.x - 128;               // row within the tile = TMEM lane
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const uint32_t tO = tmem + lane_off + L::kColO;
    const float c = p.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;

    for (int n = 0; n < count && ok; ++n) {
      const uint32_t tS = tmem + lane_off + (n & 1) * kTile;
      ok = __all_sync(0xffffffffu, mbar_wait(bars.s_full(n & 1), (n >> 1) & 1u, st,
                                             status_code(kKernFwd, kRoleSoftmax, 1)));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld32(tS + q * 32, sr[q]);
      tmem_wait_ld();
      float s[kTile];
#pragma unroll
      for (int x = 0; x < kTile; ++x) s[x] = __uint_as_float(sr[x >> 5][x & 31]);
      const uint32_t e = list[n];
      if (e >> 15) {  // keys x >= lim are hidden from this row
        const int lim = sh.key_limit(i, r, int(e & 0x7FFF));
#pragma unroll
        for (int x = 0; x < kTile; ++x)
          if (x >= lim) s[x] = -INFINITY;
      }
      // row max: 4 independent partial maxima, two new keys per three-input max
      float mp[4];
#pragma unroll
      for (int y = 0; y < 4; ++y) mp[y] = fmaxf(s[2 * y], s[2 * y + 1]);
#pragma unroll
      for (int x = 8; x < kTile; x += 8)
#pragma unroll
        for (int y = 0; y < 4; ++y) mp[y] = fmax3(mp[y], s[x + 2 * y], s[x + 2 * y + 1]);
      const float m_tile = fmax3(mp[0], mp[1], fmaxf(mp[2], mp[3])) * c;
      const bool need = m_tile > m_used + kRescaleThreshold;
      float alpha = 1.f;
      if (need) {
        alpha = ex2_approx(m_used - m_tile);  // 0 on the first tile (m_used = -inf)
        m_used = m_tile;
      }
      const float m_sub = (m_used == -INFINITY) ? 0.f : m_used;
      // P = exp2(s*c - m), the scaling and the row sum on packed fp32 pairs
      // (one instruction per two keys; the sum in 4 partial sums)
      const uint64_t c2 = f2pack(c, c), nm2 = f2pack(-m_sub, -m_sub);
      uint64_t lp2[2] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
      uint32_t pk0[32], pk1[32];
      auto p_pair = [&](int x, float s0, float s1) {
        float p0, p1;
        f2unpack(ffma2(f2pack(s0, s1), c2, nm2), p0, p1);
        p0 = ex2_approx(p0);
        p1 = ex2_approx(p1);
        lp2[x & 1] = fadd2(lp2[x & 1], f2pack(p0, p1));
        return pack2<kF16>(p0, p1);
      };
#pragma unroll
      for (int x = 0; x < 32; ++x) pk0[x] = p_pair(x, s[2 * x], s[2 * x + 1]);
#pragma unroll
      for (int x = 0; x < 32; ++x) pk1[x] = p_pair(x, s[64 + 2 * x], s[64 + 2 * x + 1]);
      float lp[2];
      f2unpack(fadd2(lp2[0], lp2[1]), lp[0], lp[1]);
      // P into the first 64 columns of this S buffer
      tmem_st32(tS, pk0);
      tmem_st32(tS + 32, pk1);
      l = l * alpha + (lp[0] + lp[1]);
      if (n > 0 && __any_sync(0xffffffffu, need)) {
        // O *= alpha for this row, once PV(n-1) has completed (PV(n) cannot
        // have: it needs this P)
        ok = __all_sync(0xffffffffu, mbar_wait(bars.pv_done(), (n - 1) & 1u, st,
                                               status_code(kKernFwd, kRoleSoftmax, 2)));
        if (!ok) break;
        tc_fence_after();
#pragma unroll 4
        for (int q = 0; q < D / 16; ++q) {
          uint32_t o[16];
          tmem_ld16(tO + q * 16, o);
          tmem_wait_ld();
#pragma unroll
          for (int x = 0; x < 16; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
          tmem_st16(tO + q * 16, o);
        }
      }
      tmem_wait_st();  // P (and a rescaled O) are in tensor memory
      tc_fence_before();
      mbar_arrive(bars.p_full(n & 1));
    }
    // epilogue: O / l and LSE
    if (ok && count > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(bars.o_done(), 0, st,
                                             status_code(kKernFwd, kRoleSoftmax, 3)));
    const int qrow = i * kTile + r;  // query row within the head
    const bool live = qrow < sh.nq;
    if (ok) {
      tc_fence_after();
      const size_t prow = ((size_t)split * sh.bh + bh) * sh.nq + qrow;
      const size_t row = kSplit ? prow * D : p.so.row(b_idx, h_idx, qrow);
      float *const o32 = kSplit ? p.o_part : static_cast<float *>(p.o);
      const float inv_l = (count > 0 && l > 0.f) ? 1.f / l : 0.f;
      // a 16-bit O leaves through the Q buffer (no MMA reads it any more;
      // count > 0: its load has landed) with TMA stores
      const bool via_tma = !kSplit && !p.o_f32 && count > 0;
      if (via_tma)
        store_rows_tma<D, kF16>(&p.tm_o, tO, sQ, r, i * kTile, 0, inv_l, true, sh.d, sh.nq, h_idx,
                                b_idx);
#pragma unroll 1
      for (int q = 0; q < D / 32 && !via_tma; ++q) {
        uint32_t o[32];
        if (count > 0) {
          tmem_ld32(tO + q * 32, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = 0u;
        }
        if (!live) {
        } else if (kSplit || p.o_f32) {
          float4 *dst = reinterpret_cast<float4 *>(o32 + row + q * 32);
#pragma unroll
          for (int x = 0; x < 8; ++x)
            dst[x] = make_float4(__uint_as_float(o[4 * x]) * inv_l,
                                 __uint_as_float(o[4 * x + 1]) * inv_l,
                                 __uint_as_float(o[4 * x + 2]) * inv_l,
                                 __uint_as_float(o[4 * x + 3]) * inv_l);
        } else {
          uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.o) + row + q * 32);
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            uint4 v;
            v.x = pack2<kF16>(__uint_as_float(o[8 * x + 0]) * inv_l, __uint_as_float(o[8 * x + 1]) * inv_l);
            v.y = pack2<kF16>(__uint_as_float(o[8 * x + 2]) * inv_l, __uint_as_float(o[8 * x + 3]) * inv_l);
            v.z = pack2<kF16>(__uint_as_float(o[8 * x + 4]) * inv_l, __uint_as_float(o[8 * x + 5]) * inv_l);
            v.w = pack2<kF16>(__uint_as_float(o[8 * x + 6]) * inv_l, __uint_as_float(o[8 * x + 7]) * inv_l);
            dst[x] = v;
          }
        }
      }
      // LSE = ln(sum_j exp(scale s_ij)) = ln2 * (m + log2 l)
      if (live)
        (kSplit ? p.lse_part[prow] : p.lse[(size_t)bh * sh.nq + qrow]) =
            (count > 0 && l > 0.f) ? (m_used + lg2_approx(l)) * 0.69314718055994531f : -INFINITY;
    }
  }

  // ---- teardown ------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool kF16>
cudaError_t launch_d256(const FwdParams &p, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(fa_fwd_d256_kernel<false, kF16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Layout::kAlloc);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fa_fwd_d256_kernel<true, kF16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, Layout::kAlloc);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int grid = p.sh.tq * p.sh.bh * p.n_split;
  LaunchProbe probe(kKindFwd, stream);
  if (p.n_split > 1)
    fa_fwd_d256_kernel<true, kF16><<<grid, kThreads, Layout::kAlloc, stream>>>(p);
  else
    fa_fwd_d256_kernel<false, kF16><<<grid, kThreads, Layout::kAlloc, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_forward_d256(const FwdParams &p, cudaStream_t stream) {
  return p.sh.f16 ? launch_d256<true>(p, stream) : launch_d256<false>(p, stream);
}

}  // namespace fa
