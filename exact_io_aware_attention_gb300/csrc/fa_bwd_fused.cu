// Attention backward in one pass over the (Q tile, K/V tile) pairs, for
// sm_103a.
//
// The pages keep only O and the softmax statistics and regenerate S and P
// block by block in the backward pass ("Paper Notes: FlashAttention",
// "Background" and "Key Ideas"; aicassindra page "FlashAttention", "The
// backward pass: recompute instead of store"). The gradients are the
// analytic ones of O = softmax(scale QK^T) V:
//
//   P_ij = exp(scale s_ij - LSE_i),  dV_j = sum_i P_ij dO_i,  dP_ij = dO_i . V_j,
//   D_i = dO_i . O_i,  dS_ij = P_ij (dP_ij - D_i),
//   dQ_i = scale sum_j dS_ij K_j,  dK_j = scale sum_i dS_ij Q_i.
//
// Here each (Q tile, K/V tile) pair has S and P recomputed once, and all five
// products of the pair run on the tensor cores of one CTA. This file's kernel
// serves head dimensions 64 and 96 (128-query steps); head dimension 128 has a
// kernel of its own with 64-query steps (fa_bwd_fused_q64.cu), because at 128
// the five products of a 128-query step do not fit in tensor memory side by
// side. The CTA owns a
// 128-key K/V tile and loops over the Q tiles that see it (causal: a row of
// the tile sees one of its keys; block-sparse: mask[i][j]); dK and dV
// accumulate in tensor memory, and each step's dQ_i partial (dS K_j, fp32) is
// added into an fp32 accumulator in the workspace with reductions in L2. fa_bwd_pre zeroes that accumulator and fa_bwd_dq_convert scales it and
// rounds it into dQ afterwards.
//
// 16 warps:
//   warp 0      TMA producer: K_j, V_j once; per step Q_i with LSE_i (ring of
//               kQSlots) and dO_i with D_i (2 slots)
//   warp 1      tcgen05 issuer (one lane) and tensor-memory owner
//   warps 4-7   thread = key row: P^T and dS^T over queries 0..63; then dV out
//   warps 8-11  the same for queries 64..127; then dK out
//   warps 12-15 dQ reducer, thread = query row: reads dQ_i's partial out of
//               tensor memory, transposes it through shared memory in 32 x 32
//               chunks and adds it into the fp32 accumulator with vector
//               reductions (red.global.add.v4.f32) that each cover four whole
//               128-byte lines; the TMA unit stays free for the tile loads
// Registers are moved between the warpgroups with setmaxnreg: the producer /
// issuer warpgroup and the reducer give some up, the softmax warpgroups take
// them (88 + 2 x 160 + 104 per thread of each warpgroup: the 65536 the launch
// holds). Every wait and store helper is inlined here: ptxas does not finish
// compiling calls to out-of-line functions from such regions.
// Tensor memory (512 columns): [0,128) S^T (P^T as packed 16-bit pairs over
// the first 32 columns of each warpgroup's half: the A operand of dV), [128,256)
// dP^T, [256,256+d) dV, [256+d,256+2d) dK. dQ_i's partial (M = queries, N = d)
// needs d more columns: at d = 64 it has two buffers of its own in [384,512);
// at d = 96 and 128 it reuses the dP^T columns, which are free once the
// softmax warps have read dP^T(n), and dP^T(n+1) waits until the reducer has
// read dQ(n) out.
// Shared memory: K_j, V_j, Q_i ring, dO_i[2], the reducer's staging (two 4 KB
// chunk slots per warp) and dS^T (128 keys x 128 queries, 16-bit, 128-byte
// swizzle). dS^T is the A operand of both dK += dS^T Q (read K-major: rows =
// keys) and dQ_i = dS K_j (read MN-major: M = queries along a row, K = keys
// down the rows), so dS leaves the softmax warps once, through shared memory.
// At d = 96 and 128 dS^T(n) is written into dO_n's slot once dV(n) has read
// it (dP^T(n) has already), and the slot takes dO_{n+2} once dK(n) and dQ(n)
// have read dS^T(n); at d = 64 it has a tile of its own.
// MMA order per step n: dV(n) (two halves, as P^T(n) arrives), S^T(n+1),
// then at d = 64 dP^T(n+1), dQ(n), dK(n), and at d = 96 (dQ in dP^T's
// columns) dQ(n), dK(n), dP^T(n+1). MMAs issued by one thread execute in issue
// order, so S^T(n+1) overwrites P^T(n) only after dV(n) has read it.
#include <math.h>

#include "fa_internal.h"
#include "ptx.cuh"
#include "tile_store.cuh"

namespace fa {
namespace {

constexpr int kThreads = 512;

template <int D, bool kList = false>
struct FusedLayout {
  static constexpr int kChunks = (D + 63) / 64;  // d = 96: 2, the last half zeros
  static constexpr int kChunkBytes = kTile * 128;
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static constexpr int kQSlots = D == 64 ? 3 : 2, kdOSlots = 2;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kTileBytes;
  static constexpr int kQOff = kVOff + kTileBytes;
  static constexpr int kdOOff = kQOff + kQSlots * kTileBytes;
  // dS^T (128 x 128, two chunks) of step n goes into dO_n's slot when that
  // holds 32 KB (d = 96, 128): dV(n) and dP^T(n) have read dO_n by then.
  // Otherwise it has a tile of its own.
  static constexpr bool kDsInDo = kTileBytes >= 2 * kChunkBytes;
  static constexpr int kdSOff = kdOOff + kdOSlots * kTileBytes;
  // the reducer's staging: two 4 KB chunk slots per warp
  static constexpr int kStageOff = kdSOff + (kDsInDo ? 0 : 2 * kChunkBytes);
  static constexpr int kLseOff = kStageOff + 4 * 2 * 4096;          // [kQSlots][128] LSE * log2(e)
  static constexpr int kDeltaOff = kLseOff + kQSlots * kTile * 4;  // [kdOSlots][128] D
  // kList (d = 64 under a block mask): the Q tiles that see this CTA's K/V
  // tile, ascending (warp 2 at set-up); without it every role walks the mask
  // (d = 96 has no room for the list)
  static constexpr bool kQList = kList;
  static_assert(!kList || D == 64, "Q-tile list: d = 64 only");
  static constexpr int kListOff = kDeltaOff + kdOSlots * kTile * 4;
  static constexpr int kBarOff = kListOff + (kQList ? kMaxTiles * 2 : 0);
  static constexpr int kNumBars = 26;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  static_assert(kBytes <= 232448, "shared memory budget");
  // dQ's partial shares the dP^T columns unless 3 d-wide accumulators fit
  // beside S^T and dP^T
  static constexpr bool kDqShare = 3 * D > 256;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
  static constexpr uint32_t kColDQ0 = kDqShare ? kColDP : 256 + 2 * D;
  static constexpr uint32_t kColDQ1 = kDqShare ? kColDP : 256 + 3 * D;
  static_assert(kDqShare || 256 + 4 * D <= 512, "two dQ buffers");
};

struct Bars {
  uint32_t base;
  __device__ uint32_t kv_full() const { return base; }
  __device__ uint32_t q_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t q_empty(int s) const { return base + 8 * (4 + s); }
  __device__ uint32_t do_full(int s) const { return base + 8 * (7 + s); }
  __device__ uint32_t do_empty(int s) const { return base + 8 * (9 + s); }
  __device__ uint32_t s_full() const { return base + 8 * 11; }
  // P^T of queries 64h + 32u .. 64h + 32u + 31 of both warpgroups h (u = 0, 1)
  __device__ uint32_t p_full(int u) const { return base + 8 * (12 + u); }
  __device__ uint32_t dp_full() const { return base + 8 * 14; }
  __device__ uint32_t ds_full() const { return base + 8 * 15; }   // dS^T in shared memory
  __device__ uint32_t ds_empty() const { return base + 8 * 16; }  // dK and dQ have read it
  __device__ uint32_t dv_step() const { return base + 8 * 23; }   // dV(n) has read dO_n
  __device__ uint32_t dq_full(int b) const { return base + 8 * (17 + b); }
  __device__ uint32_t dq_free(int b) const { return base + 8 * (19 + b); }
  __device__ uint32_t acc_done() const { return base + 8 * 21; }
  __device__ uint32_t dv_done() const { return base + 8 * 24; }
  __device__ uint32_t dk_done() const { return base + 8 * 25; }
  __device__ uint32_t teardown() const { return base + 8 * 22; }
};

enum Role : uint32_t { kRoleLoad = 1, kRoleMma = 2, kRoleSoftmax = 3, kRoleInit = 5 };

// Next Q tile at or after i that the block mask lets see K/V tile j (tq if none).
__device__ __forceinline__ int next_q(const Shape &sh, int i, int j) {
  if (sh.mask)
    while (i < sh.tq && sh.mask[(size_t)i * sh.tk + j] == 0) ++i;
  return i;
}

// Tensor-memory column of the packed P^T for MMA step kk (queries
// 16kk..16kk+15): queries 64h.. are packed at column 64h.
__device__ __forceinline__ uint32_t packed_col(int kk) { return (kk >> 2) * 64 + (kk & 3) * 8; }

// Four fp32 values added into global memory at `addr` (16-byte aligned) by
// one vector reduction performed in L2.
__device__ __forceinline__ void red_add_v4(float *addr, uint32_t a, uint32_t b, uint32_t c,
                                           uint32_t d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr),
               "f"(__uint_as_float(a)), "f"(__uint_as_float(b)), "f"(__uint_as_float(c)),
               "f"(__uint_as_float(d))
               : "memory");
}

__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t &a, uint32_t &b, uint32_t &c,
                                             uint32_t &d) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
               : "r"(addr)
               : "memory");
}

// This thread's row of 32 fp32 values into a 4 KB chunk slot (32 rows x 128
// bytes, 16-byte pieces swizzled by row & 7, so that neither this write nor
// the read-back by rows conflicts on shared-memory banks).
__device__ __forceinline__ void stage_row32(uint32_t slot, int row, const uint32_t (&v)[32]) {
  const uint32_t base = slot + row * 128;
#pragma unroll
  for (int p = 0; p < 8; ++p)
    st_shared_v4(base + ((uint32_t(p) ^ uint32_t(row & 7)) << 4), v[4 * p], v[4 * p + 1],
                 v[4 * p + 2], v[4 * p + 3]);
}

template <int D>
__device__ __forceinline__ void load_q(const BwdParams &p, const Bars &bars, int s, int i,
                                       uint32_t s_base, size_t stat_head, int h_idx, int b_idx) {
  using L = FusedLayout<D>;
  mbar_arrive_expect_tx(bars.q_full(s), L::kTileBytes + kTile * 4);
  for (int c = 0; c < L::kChunks; ++c)
    tma_load_4d(s_base + L::kQOff + s * L::kTileBytes + c * L::kChunkBytes, &p.tm_q, c * 64,
                i * kTile, h_idx, b_idx, bars.q_full(s));
  bulk_load_1d(s_base + L::kLseOff + s * kTile * 4, p.lse2 + stat_head + (size_t)i * kTile,
               kTile * 4, bars.q_full(s));
}

template <int D>
__device__ __forceinline__ void load_do(const BwdParams &p, const Bars &bars, int s, int i,
                                        uint32_t s_base, size_t stat_head, int h_idx, int b_idx) {
  using L = FusedLayout<D>;
  mbar_arrive_expect_tx(bars.do_full(s), L::kTileBytes + kTile * 4);
  for (int c = 0; c < L::kChunks; ++c)
    tma_load_4d(s_base + L::kdOOff + s * L::kTileBytes + c * L::kChunkBytes, &p.tm_do, c * 64,
                i * kTile, h_idx, b_idx, bars.do_full(s));
  bulk_load_1d(s_base + L::kDeltaOff + s * kTile * 4, p.delta + stat_head + (size_t)i * kTile,
               kTile * 4, bars.do_full(s));
}

// kF16: f16 elements instead of bf16. D is 64, 96 or 128 (at 96 the tiles keep
// two 64-column chunks whose columns 96..127 the tensor maps fill with zeros).
template <int D, bool kF16, bool kList>
__global__ void __launch_bounds__(kThreads, 1) fa_bwd_fused(const __grid_constant__ BwdParams p) {
  using L = FusedLayout<D, kList>;
  // d = 64: the epilogue stores dV once its last product has completed and
  // dK once its own has (issued ahead of the last dQ), staged through V's
  // buffer and a dO slot, which no MMA reads by then
  constexpr bool kEarlyEpi = !L::kDsInDo && !L::kDqShare;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t s_base = smem_u32(smem);
  int *misc = reinterpret_cast<int *>(smem + L::kMiscOff);  // [0] tmem [2] abort [3] list length
  uint16_t *qlist = reinterpret_cast<uint16_t *>(smem + L::kListOff);
  // the 128-byte swizzle patterns need 1024-byte aligned tiles; the layout
  // has no room for alignment slack, so a misaligned base is reported
  if (s_base & 1023u) {
    if (threadIdx.x == 0 && p.status)
      atomicCAS(p.status, 0u, status_code(kKernBwdFused, kRoleInit, 1));
    return;
  }
  const uint32_t sK = s_base + L::kKOff, sV = s_base + L::kVOff;
  const uint32_t sQ = s_base + L::kQOff, sdO = s_base + L::kdOOff;
  // dS^T of step n
  auto ds_tile = [&](int n) -> uint32_t {
    return L::kDsInDo ? sdO + (n & 1) * L::kTileBytes : s_base + L::kdSOff;
  };
  const float *lse_s = reinterpret_cast<const float *>(smem + L::kLseOff);
  const float *delta_s = reinterpret_cast<const float *>(smem + L::kDeltaOff);
  Bars bars{s_base + L::kBarOff};
  StatusSlot st{p.status, &misc[2], p.wait_limit_ns};

  const int warp = threadIdx.x >> 5;
  const Shape &sh = p.sh;
  const int T = sh.tq;
  // CTAs in head groups of p.head_group heads, heavy K/V tiles (causal: the
  // early ones, seen by the most Q tiles) first within a group, so that the
  // CTAs in flight touch few heads and those heads' dQ accumulators stay in L2
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
    // a dO slot is free once the MMAs are done with it (one commit: after
    // dV, or after dK and dQ where dS^T goes into the slot) and the softmax
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
    mbar_init(bars.ds_empty(), 1);
    mbar_init(bars.dv_step(), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.dq_full(b), 1);
      mbar_init(bars.dq_free(b), 128);
    }
    mbar_init(bars.acc_done(), 1);
    mbar_init(bars.dv_done(), 1);
    mbar_init(bars.dk_done(), 1);
    mbar_init(bars.teardown(), 1);
    misc[2] = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
    tma_prefetch_desc(&p.tm_do);
    // K_j, V_j and the first Q tile's Q and dO depend on blockIdx only: load
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
  } else if (L::kQList && warp == 2) {
    // the Q tiles that see K/V tile j under the block mask, ascending, so that
    // no role walks the mask in its loop (5.8 % faster at B4 H16 N8192 with
    // 26 % of the tiles kept)
    const int lane = threadIdx.x & 31;
    int count = 0;
    for (int base = sh.first_q_tile(j); base < T; base += 32) {
      const int i = base + lane;
      const bool a = i < T && (!sh.mask || sh.mask[(size_t)i * sh.tk + j] != 0);
      const uint32_t ball = __ballot_sync(0xffffffffu, a);
      if (a) qlist[count + __popc(ball & ((1u << lane) - 1u))] = uint16_t(i);
      count += __popc(ball);
    }
    if (lane == 0) misc[3] = count;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  const int nlist = L::kQList ? misc[3] : 0;  // qlist[0] == first
  // Q tile x of this CTA's sequence, after tile i (tile x - 1); tq: none left
  auto next_tile = [&](int i, int x) -> int {
    if constexpr (L::kQList)
      return x < nlist ? int(qlist[x]) : T;
    else
      return next_q(sh, i + 1, j);
  };
  // registers per thread by warpgroup (every warp of a warpgroup runs the same
  // setmaxnreg at the head of its branch): 88 + 160 + 160 + 104 = 512 =
  // 65536 / 128, the launch's 128 per thread (checked with -Xptxas -v: the
  // kernel is compiled to exactly 128 registers, without spills)
  if (warp < 4) {
  setmaxnreg_dec<88>();
  if (warp == 0) {
    // ---- TMA producer ------------------------------------------------------
    if (elect_one() && any && !(p.debug_flags & kDebugSkipLoads)) {
      int nq = 1, ndo = 1;  // tiles issued: the first Q tile's Q and dO came with the set-up
      bool ok = true;
      for (int x = 1, i = next_tile(first, 1); i < T && ok; ++x, i = next_tile(i, x)) {
        const int qs = nq % L::kQSlots;
        ok = mbar_wait_inl(bars.q_empty(qs), ((nq / L::kQSlots) & 1u) ^ 1u, st,
                       status_code(kKernBwdFused, kRoleLoad, 1));
        if (!ok) break;
        load_q<D>(p, bars, qs, i, s_base, stat_head, h_idx, b_idx);
        ++nq;
        const int ds = ndo % L::kdOSlots;
        ok = mbar_wait_inl(bars.do_empty(ds), ((ndo / L::kdOSlots) & 1u) ^ 1u, st,
                       status_code(kKernBwdFused, kRoleLoad, 4));
        if (!ok) break;
        load_do<D>(p, bars, ds, i, s_base, stat_head, h_idx, b_idx);
        ++ndo;
      }
      // teardown: every copy issued has landed
      mbar_wait_drain_inl(bars.kv_full(), 0, st, status_code(kKernBwdFused, kRoleLoad, 2));
      for (int s = 0; s < L::kQSlots && s < nq; ++s) {
        const int last = s + ((nq - 1 - s) / L::kQSlots) * L::kQSlots;
        mbar_wait_drain_inl(bars.q_full(s), (last / L::kQSlots) & 1u, st,
                        status_code(kKernBwdFused, kRoleLoad, 3));
      }
      for (int s = 0; s < L::kdOSlots && s < ndo; ++s) {
        const int last = s + ((ndo - 1 - s) / L::kdOSlots) * L::kdOSlots;
        mbar_wait_drain_inl(bars.do_full(s), (last / L::kdOSlots) & 1u, st,
                        status_code(kKernBwdFused, kRoleLoad, 5));
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- tcgen05 issuer ----------------------------------------------------
    if (elect_one()) {
      constexpr uint32_t kIdSq = idesc_f32acc(kTile, kTile, 0, 0, kF16);  // S^T, dP^T
      constexpr uint32_t kIdAcc = idesc_f32acc(kTile, D, 0, 1, kF16);     // dV, dK: B MN-major
      constexpr uint32_t kIdDq = idesc_f32acc(kTile, D, 1, 1, kF16);      // dQ: A, B MN-major
      bool ok = !any || mbar_wait_inl(bars.kv_full(), 0, st, status_code(kKernBwdFused, kRoleMma, 1));
      // X^T = A Y^T with A in {K_j, V_j} and Y in {Q_i, dO_i}: K-major over d
      auto issue_sq = [&](uint32_t a_base, uint32_t b_base, uint32_t col) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::kChunkBytes + (kk & 3) * 32;
          mma_f16kind_ss(tmem + col, sdesc_sw128(a_base + off, 16, 1024),
                         sdesc_sw128(b_base + off, 16, 1024), kIdSq, kk > 0);
        }
      };
      // dV += P^T dO_i with P^T packed in tensor memory, over the queries
      // 64h + 32u .. 64h + 32u + 31 of both warpgroups h
      auto issue_dv = [&](uint32_t do_base, bool first_step, int u) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int kk = (e >> 1) * 4 + 2 * u + (e & 1);
          mma_f16kind_ts(tmem + L::kColDV, tmem + L::kColS + packed_col(kk),
                         sdesc_sw128(do_base + kk * 2048, L::kChunkBytes, 1024), kIdAcc,
                         (!first_step || u > 0 || e > 0) ? 1u : 0u);
        }
      };
      // dK += dS^T Q_i: dS^T K-major (rows = keys), Q_i MN-major (rows = queries)
      auto issue_dk = [&](uint32_t sdS, uint32_t q_base, bool first_step) {
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_f16kind_ss(tmem + L::kColDK,
                         sdesc_sw128(sdS + (kk >> 2) * L::kChunkBytes + (kk & 3) * 32, 16, 1024),
                         sdesc_sw128(q_base + kk * 2048, L::kChunkBytes, 1024), kIdAcc,
                         (!first_step || kk > 0) ? 1u : 0u);
      };
      // dQ_i partial = dS K_j: dS read MN-major from the dS^T tile (M =
      // queries along a row), K_j MN-major (N = d along a row); K = keys
      auto issue_dq = [&](uint32_t sdS, uint32_t col) {
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_f16kind_ss(tmem + col, sdesc_sw128(sdS + kk * 2048, L::kChunkBytes, 1024),
                         sdesc_sw128(sK + kk * 2048, L::kChunkBytes, 1024), kIdDq, kk > 0);
      };
      if (ok && any) {
        ok = mbar_wait_inl(bars.q_full(0), 0, st, status_code(kKernBwdFused, kRoleMma, 2));
        if (ok) {
          tc_fence_after();
          issue_sq(sK, sQ, L::kColS);
          mma_commit(bars.s_full());
          ok = mbar_wait_inl(bars.do_full(0), 0, st, status_code(kKernBwdFused, kRoleMma, 7));
        }
        if (ok) {
          tc_fence_after();
          issue_sq(sV, sdO, L::kColDP);
          mma_commit(bars.dp_full());
        }
      }
      int n = 0, qs = 0, qph = 0;  // Q slot of step n and the parity of its phase
      for (int x = 0, i = first; i < T && ok; ++n, ++x) {
        const int ds = n & 1, ds1 = ds ^ 1;  // dO slots of steps n and n + 1
        const int qs1 = qs + 1 == L::kQSlots ? 0 : qs + 1;
        const int qph1 = qs + 1 == L::kQSlots ? qph ^ 1 : qph;
        const int inext = next_tile(i, x + 1);
        ok = mbar_wait_inl(bars.p_full(0), n & 1, st, status_code(kKernBwdFused, kRoleMma, 3));
        if (!ok) break;
        tc_fence_after();
        issue_dv(sdO + ds * L::kTileBytes, n == 0, 0);
        ok = mbar_wait_inl(bars.p_full(1), n & 1, st, status_code(kKernBwdFused, kRoleMma, 6));
        if (!ok) break;
        tc_fence_after();
        issue_dv(sdO + ds * L::kTileBytes, n == 0, 1);
        if (kEarlyEpi && inext >= T) mma_commit(bars.dv_done());
        if (L::kDsInDo)
          mma_commit(bars.dv_step());  // dV(n) has read dO_n: dS^T(n) may go there
        else
          mma_commit(bars.do_empty(ds));  // dV(n) has read dO_n
        if (inext < T) {
          ok = mbar_wait_inl(bars.q_full(qs1), qph1, st, status_code(kKernBwdFused, kRoleMma, 4));
          if (!ok) break;
          tc_fence_after();
          issue_sq(sK, sQ + qs1 * L::kTileBytes, L::kColS);
          mma_commit(bars.s_full());
        }
        ok = mbar_wait_inl(bars.ds_full(), n & 1, st, status_code(kKernBwdFused, kRoleMma, 5));
        if (!ok) break;
        tc_fence_after();
        // d = 64 (dQ has columns of its own): dP^T(n+1) goes ahead of dQ(n) and
        // dK(n), since the softmax warps have read dP^T(n); they form dS^T(n+1)
        // while dQ(n) and dK(n) run (3 % faster on dense and block-sparse)
        if (!L::kDqShare && inext < T) {
          ok = mbar_wait_inl(bars.do_full(ds1), ((n + 1) >> 1) & 1, st,
                         status_code(kKernBwdFused, kRoleMma, 7));
          if (!ok) break;
          tc_fence_after();
          issue_sq(sV, sdO + ds1 * L::kTileBytes, L::kColDP);
          mma_commit(bars.dp_full());
        }
        const int b = L::kDqShare ? 0 : (n & 1);
        // d = 64, the item's last step: dK ahead of dQ, so that the epilogue
        // need not wait for the last dQ
        const bool dk_first = kEarlyEpi && inext >= T;
        if (dk_first) {
          issue_dk(ds_tile(n), sQ + qs * L::kTileBytes, n == 0);
          mma_commit(bars.q_empty(qs));
          mma_commit(bars.dk_done());
        }
        if (!L::kDqShare && n >= 2) {  // buffer b was last used by step n - 2
          ok = mbar_wait_inl(bars.dq_free(b), ((n >> 1) - 1) & 1, st,
                         status_code(kKernBwdFused, kRoleMma, 9));
          if (!ok) break;
        }
        tc_fence_after();
        issue_dq(ds_tile(n), b ? L::kColDQ1 : L::kColDQ0);
        mma_commit(bars.dq_full(b));
        if (!dk_first) {
          issue_dk(ds_tile(n), sQ + qs * L::kTileBytes, n == 0);
          mma_commit(bars.q_empty(qs));
        }
        if (L::kDsInDo)
          mma_commit(bars.do_empty(ds));  // dK(n) and dQ(n) have read dS^T(n) in dO_n's slot
        else
          mma_commit(bars.ds_empty());
        if (L::kDqShare && inext < T) {
          if (L::kDqShare) {  // dP^T(n+1) goes where dQ(n) is until it has been read
            ok = mbar_wait_inl(bars.dq_free(0), n & 1, st, status_code(kKernBwdFused, kRoleMma, 10));
            if (!ok) break;
          }
          ok = mbar_wait_inl(bars.do_full(ds1), ((n + 1) >> 1) & 1, st,
                         status_code(kKernBwdFused, kRoleMma, 7));
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
      mbar_wait_drain_inl(bars.teardown(), 0, st, status_code(kKernBwdFused, kRoleMma, 8));
    }
    __syncwarp();
  }
  } else if (warp < 12) {
    setmaxnreg_inc<160>();
    // ---- P^T and dS^T (thread = key row) ---------------------------------------
    const int h = (warp - 4) >> 2;                 // query half 64h..64h+63
    const int kr = threadIdx.x & 127;              // key row = TMEM lane
    const uint32_t t = tmem + (uint32_t((warp & 3) * 32) << 16);
    const float c = p.scale_log2;
    bool ok = true;
    int n = 0, qs = 0, qph = 0;  // Q slot of step n and the parity of its phase
    for (int x = 0, i = first; i < T && ok; ++x, i = next_tile(i, x), ++n) {
      const int ds = n & 1;  // dO slot
      ok = __all_sync(0xffffffffu, mbar_wait_inl(bars.s_full(), n & 1, st,
                                             status_code(kKernBwdFused, kRoleSoftmax, 1)));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait_inl(bars.q_full(qs), qph, st,
                                                     status_code(kKernBwdFused, kRoleSoftmax, 2)));
      if (!ok) break;
      tc_fence_after();
      const float *lse2 = lse_s + qs * kTile + 64 * h;
      const float *delta = delta_s + ds * kTile + 64 * h;
      qph = qs + 1 == L::kQSlots ? qph ^ 1 : qph;
      qs = qs + 1 == L::kQSlots ? 0 : qs + 1;
      // P^T_kq = exp2(s_kq * scale * log2e - LSE_q * log2e) in two halves of
      // 32 queries, each written to tensor memory over this warpgroup's first
      // 32 S^T columns (already read) and announced on its own barrier
      float pr[64];
      {
        uint32_t sr[2][32];
        tmem_ld32(t + L::kColS + 64 * h, sr[0]);
        tmem_ld32(t + L::kColS + 64 * h + 32, sr[1]);
        tmem_wait_ld();
        // only on a tile that the causal boundary crosses: key kr sees query
        // 64h + x only if x >= lo
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
      // dS^T_kq = P^T_kq (dP^T_kq - D_q), rounded to 16 bits, into the dS^T
      // tile: row kr, queries 64h.. = chunk h, 16-byte pieces swizzled by kr & 7
      ok = __all_sync(0xffffffffu, mbar_wait_inl(bars.dp_full(), n & 1, st,
                                             status_code(kKernBwdFused, kRoleSoftmax, 4)));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait_inl(bars.do_full(ds), (n >> 1) & 1, st,
                                                     status_code(kKernBwdFused, kRoleSoftmax, 5)));
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
      // where dS^T(n) goes must be free: dO_n's slot once dV(n) has read it,
      // or the own tile once dK(n-1) and dQ(n-1) have read it
      if (L::kDsInDo || n > 0) {
        ok = __all_sync(0xffffffffu,
                        L::kDsInDo ? mbar_wait_inl(bars.dv_step(), n & 1, st,
                                                   status_code(kKernBwdFused, kRoleSoftmax, 9))
                                   : mbar_wait_inl(bars.ds_empty(), (n - 1) & 1, st,
                                                   status_code(kKernBwdFused, kRoleSoftmax, 7)));
        if (!ok) break;
      }
      {
        const uint32_t row = ds_tile(n) + h * L::kChunkBytes + kr * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          st_shared_v4(row + ((uint32_t(u) ^ uint32_t(kr & 7)) << 4), dsp[4 * u], dsp[4 * u + 1],
                       dsp[4 * u + 2], dsp[4 * u + 3]);
      }
      fence_proxy_async_smem();  // the tensor core reads dS^T through the async proxy
      tc_fence_before();         // dP^T has been read: dQ(n) may take its columns
      mbar_arrive(bars.ds_full());
      mbar_arrive(bars.do_empty(ds));  // D_i has been read
    }
    // epilogue: warps 4-7 write dV, warps 8-11 write dK (scaled); at d = 96
    // through the K_j and V_j buffers once every MMA has completed, at d = 64
    // each as soon as its own last product has (V's buffer and dO slot 0)
    if (ok && any)
      ok = __all_sync(0xffffffffu, mbar_wait_inl(kEarlyEpi ? (h ? bars.dk_done() : bars.dv_done())
                                                           : bars.acc_done(), 0, st,
                                             status_code(kKernBwdFused, kRoleSoftmax, 6)));
    if (ok) {
      tc_fence_after();
      store_rows_tma_inl<D, kF16>(h ? &p.tm_dk : &p.tm_dv, t + (h ? L::kColDK : L::kColDV),
                              kEarlyEpi ? (h ? sdO : sV) : (h ? sV : sK), kr, j * kTile, 0,
                              h ? p.scale : 1.f, any, sh.d, sh.nk, h_idx, b_idx);
    }
  } else {
    setmaxnreg_dec<104>();
    // ---- dQ reducer (thread = query row) ---------------------------------------
    const int qw = warp & 3;                        // rows 32qw..32qw+31 of the Q tile
    const int lane = threadIdx.x & 31;
    const uint32_t t = tmem + (uint32_t(qw * 32) << 16);
    constexpr int kParts = D / 32;                  // 32-column chunks of a dQ row: 2, 3, 4
    float *dq_head = p.dq_acc + stat_head * D;      // this head's [tq*128][D] accumulator
    const uint32_t slot = s_base + L::kStageOff + qw * 8192;  // this warp's two 4 KB slots
    // Adds a staged 32 x 32 chunk (columns col0..col0+31 of the warp's rows)
    // into the accumulator: lane l reads 16 bytes of row 4k + l/8, so each
    // reduction instruction covers 4 rows x 128 bytes, whole L2 lines.
    auto flush = [&](uint32_t sl, int i, int col0) {
      __syncwarp();
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int r = 4 * k + (lane >> 3), pc = lane & 7;
        uint32_t a, b, c, d;
        ld_shared_v4(sl + r * 128 + ((uint32_t(pc) ^ uint32_t(r & 7)) << 4), a, b, c, d);
        const int row = kTile * i + 32 * qw + r;
        if (row < sh.nq) red_add_v4(dq_head + (size_t)row * D + col0 + 4 * pc, a, b, c, d);
      }
      __syncwarp();  // the slot may be written again
    };
    bool ok = true;
    int n = 0;
    for (int x = 0, i = first; i < T && ok; ++x, i = next_tile(i, x), ++n) {
      const int b = L::kDqShare ? 0 : (n & 1);
      ok = __all_sync(0xffffffffu,
                      mbar_wait_inl(bars.dq_full(b), L::kDqShare ? (n & 1) : ((n >> 1) & 1), st,
                                    status_code(kKernBwdFused, kRoleSoftmax, 8)));
      if (!ok) break;
      tc_fence_after();
      const uint32_t tq = t + (b ? L::kColDQ1 : L::kColDQ0);
      // columns 0..63 into the two slots; the rest into registers before the
      // tensor-memory columns are released, so that dQ's buffer frees early
      {
        uint32_t v[2][32];
        tmem_ld32(tq, v[0]);
        tmem_ld32(tq + 32, v[1]);
        tmem_wait_ld();
        if (kParts == 2) {
          tc_fence_before();
          mbar_arrive(bars.dq_free(b));
        }
        stage_row32(slot, lane, v[0]);
        stage_row32(slot + 4096, lane, v[1]);
      }
      if (kParts > 2) {
        uint32_t v[2][32];
        tmem_ld32(tq + 64, v[0]);
        if (kParts > 3) tmem_ld32(tq + 96, v[1]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bars.dq_free(b));
        flush(slot, i, 0);
        stage_row32(slot, lane, v[0]);
        flush(slot + 4096, i, 32);
        if (kParts > 3) stage_row32(slot + 4096, lane, v[1]);
        flush(slot, i, 64);
        if (kParts > 3) flush(slot + 4096, i, 96);
      } else {
        flush(slot, i, 0);
        flush(slot + 4096, i, 32);
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

// dQ = scale * dQ_acc rounded to the 16-bit type: thread = 8 columns of a row.
template <int D, bool kF16>
__global__ void __launch_bounds__(256) fa_bwd_dq_convert(const __grid_constant__ BwdParams p) {
  constexpr int kGroups = D / 8;
  const Shape &sh = p.sh;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long total = (long long)sh.bh * sh.nq * kGroups;
  if (idx >= total) return;
  const int g = int(idx % kGroups);
  const long long rowf = idx / kGroups;
  const int n = int(rowf % sh.nq), bh = int(rowf / sh.nq);
  const int b_idx = bh / sh.heads, h_idx = bh % sh.heads;
  const float4 *src = reinterpret_cast<const float4 *>(
      p.dq_acc + ((size_t)bh * sh.tq * kTile + n) * D + 8 * g);
  const float4 a = src[0], b = src[1];
  const float s = p.scale;
  uint4 o;
  o.x = pack2<kF16>(a.x * s, a.y * s);
  o.y = pack2<kF16>(a.z * s, a.w * s);
  o.z = pack2<kF16>(b.x * s, b.y * s);
  o.w = pack2<kF16>(b.z * s, b.w * s);
  *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.dq) + p.sdq.row(b_idx, h_idx, n) + 8 * g) = o;
}

// dQ = bf16(scale * dQ_acc) after the one-pass kernel
template <int D, bool kF16>
cudaError_t launch_dq_convert(const BwdParams &p, cudaStream_t stream) {
  {
    LaunchProbe probe(kKindBwdConvert, stream);
    const long long total = (long long)p.sh.bh * p.sh.nq * (D / 8);
    fa_bwd_dq_convert<D, kF16><<<unsigned((total + 255) / 256), 256, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

template <int D, bool kF16, bool kList>
cudaError_t launch_fused_kernel(const BwdParams &p, cudaStream_t stream) {
  using L = FusedLayout<D, kList>;
  static const cudaError_t configured = [] {
    cudaError_t e = cudaFuncSetAttribute(fa_bwd_fused<D, kF16, kList>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e == cudaSuccess) e = check_kernel_regs(fa_bwd_fused<D, kF16, kList>, 65536 / kThreads);
    return e;
  }();
  if (configured != cudaSuccess) return configured;
  LaunchProbe probe(kKindBwdFused, stream);
  fa_bwd_fused<D, kF16, kList><<<p.sh.tk * p.sh.bh, kThreads, L::kBytes, stream>>>(p);
  return cudaGetLastError();
}

template <int D, bool kF16>
cudaError_t launch_fused_d(const BwdParams &p, cudaStream_t stream) {
  cudaError_t e;
  if constexpr (D == 128) {
    e = launch_backward_fused_q64(p, stream);  // 64-query steps (fa_bwd_fused_q64.cu)
  } else if constexpr (D == 64) {
    // under a block mask with the list of the Q tiles that see each K/V tile
    e = p.sh.mask ? launch_fused_kernel<D, kF16, true>(p, stream)
                  : launch_fused_kernel<D, kF16, false>(p, stream);
  } else {
    e = launch_fused_kernel<D, kF16, false>(p, stream);
  }
  if (e != cudaSuccess) return e;
  return launch_dq_convert<D, kF16>(p, stream);
}

}  // namespace

cudaError_t launch_backward_fused(const BwdParams &p, cudaStream_t stream) {
  const bool f16 = p.sh.f16 != 0;
  if (p.sh.d == 64) return f16 ? launch_fused_d<64, true>(p, stream) : launch_fused_d<64, false>(p, stream);
  if (p.sh.d == 96) return f16 ? launch_fused_d<96, true>(p, stream) : launch_fused_d<96, false>(p, stream);
  if (p.sh.d == 128)
    return f16 ? launch_fused_d<128, true>(p, stream) : launch_fused_d<128, false>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
