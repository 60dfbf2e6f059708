// Fused attention forward for sm_103a: TMA loads, tcgen05 MMAs accumulating in
// tensor memory, online softmax in registers.
//
// Method: the tiled forward pass with online softmax of "Paper Notes:
// FlashAttention" (sections "Tiling: Block-by-Block Softmax" and "The Complete
// Algorithm in Pseudocode"), in the corrected form of the numpy
// flash_attention in "flash attention" (muhibwaqar.com, "build it from
// scratch") and of the aicassindra page ("Rescale and accumulate: the forward
// pass in one loop"): running max m and sum l per row, an unnormalised output
// accumulator rescaled by exp(m_old - m_new), one division by l at the end.
// Causal masking is applied per tile (aicassindra page, "Common pitfalls"):
// tiles above the diagonal are never visited, tiles that the diagonal crosses
// are masked element-wise, and so is the last K/V tile when the key count is
// not a multiple of 128 (its missing rows arrive as zeros from the tensor
// map and are hidden). Block-sparse attention ("Paper Notes: FlashAttention",
// "Experiments & Results") visits only the tiles whose mask byte is set.
//
// CTA = one head, two consecutive 128-row Q tiles (t = 0, 1) sharing one
// stream of K/V tiles; at d = 64 (without the key split) also one Q tile per
// CTA with two CTAs per SM (kNT = 1: warps 0-7, 256 tensor-memory columns;
// the launch chooses, see fwd_one_tile). 12 warps:
//   warp 0      TMA producer: Q tiles once, then K_j, V_j through a smem ring
//               (Q and the first K/V tile are issued during set-up)
//   warp 1      tcgen05 issuer (one lane) and tensor-memory owner
//   warp 2      builds the list of K/V tiles to visit and the last entry
//               each Q tile is active in, then idles
//   warps 4-7   softmax of Q tile 0 (thread = query row = TMEM lane)
//   warps 8-11  softmax of Q tile 1
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   [0,128) S_0   [128,256) S_1   [256,256+d) O_0   [256+d,256+2d) O_1
//   P_t (16-bit pairs): the first 64 columns of S_t (d >= 96) or [384+64t, +64) (d = 64)
// The MMA issue order PV_0(n), S_0(n+1), PV_1(n), S_1(n+1) lets the tensor
// core work on one Q tile while the other tile's softmax runs; at d = 64,
// where P_t has columns of its own, S_t(n+1) goes out once the softmax warps
// have read S_t(n), ahead of PV_t(n). Each Q tile's epilogue starts once its
// own last PV has completed (o_done[t]).
//
// Split over the keys (few Q tiles, many keys, e.g. decoding against a long
// cache): n_split CTAs share one Q-tile pair, each taking a contiguous share
// of its K/V tile list, and write their normalised partial O and their LSE.
// fa_fwd_combine then merges the partials with the block-merge rule of "Paper
// Notes: FlashAttention" ("Tiling: Block-by-Block Softmax": the merged max is
// the larger max, each block's sum and output are rescaled by exp(m_block -
// m), and the sums add), written with LSE_s = m_s + ln l_s:
//   LSE = ln sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) O_s.
#include <math.h>

#include "fa_internal.h"
#include "ptx.cuh"
#include "tile_store.cuh"

namespace fa {
namespace {

// kNT Q tiles per CTA: two (the general form), or one at d = 64 without the
// key split, where two CTAs share an SM
template <int kNT>
constexpr int kThreadsFor = 128 * (1 + kNT);
template <int kNT>
constexpr int kCtasPerSm = kNT == 1 ? 2 : 1;
// registers per thread: the launch bound (65536 / threads per SM, rounded down
// to 8) and, where the warpgroups move registers (d = 64), the split of it
// between the producer / MMA warpgroup and each softmax warpgroup
template <int kNT>
constexpr int kRegsLaunch = kNT == 2 ? 168 : 128;
template <int kNT>
constexpr int kRegsLoadMma = kNT == 2 ? 88 : 56;
template <int kNT>
constexpr int kRegsSoftmax = kNT == 2 ? 208 : 200;
static_assert(kRegsLoadMma<2> * 128 + kRegsSoftmax<2> * 256 == kRegsLaunch<2> * kThreadsFor<2>,
              "warpgroup register split");
static_assert(kRegsLoadMma<1> * 128 + kRegsSoftmax<1> * 128 == kRegsLaunch<1> * kThreadsFor<1>,
              "warpgroup register split");
static_assert(kRegsLaunch<1> * kThreadsFor<1> * kCtasPerSm<1> <= 65536, "registers per SM");
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale only if the max grows by > 2^8

template <int D, int kNT>
struct FwdLayout {
  static constexpr int kChunks = (D + 63) / 64;       // 128-byte column chunks per row (d = 96: 2, the last half zeros)
  static constexpr int kChunkBytes = kTile * 128;     // 128 rows x 128 B
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  // K/V ring slots (K and V alternate); one Q tile: half of the SM's shared
  // memory per CTA
  static constexpr int kStages = kNT == 1 ? 5 : (kChunks == 2) ? 5 : 10;
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQOff + kNT * kTileBytes;
  static constexpr int kListOff = kKVOff + kStages * kTileBytes;
  static constexpr int kBarOff = kListOff + kMaxTiles * 2;
  // barriers: q_full, kv_full[S], kv_empty[S], s_full[2], p_full[2][2], o_done[2], teardown,
  // s_read[2], pv_done[2]
  static constexpr int kNumBars = 1 + 2 * kStages + 2 + 4 + 2 + 1 + 4;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 32;
  static constexpr int kAlloc = kBytes + 1024;        // slack to align the base to 1024 B
  static_assert(kAlloc <= 232448, "shared memory budget");
  // P_t (16-bit pairs, 64 columns) lives in tensor memory as the A operand of
  // O_t += P_t V. With d = 128 the 512 columns hold S_0, S_1, O_0, O_1 and P_t
  // takes the first half of S_t's columns once S_t has been read; with d = 64
  // it has columns of its own.
  // tensor memory: S_t at 128t, O_t after all S, P_t (d = 64) after all O;
  // at d >= 96 P_t overlays S_t
  static constexpr uint32_t kTmemCols = 256 * kNT;
  __host__ __device__ static constexpr uint32_t col_o(int t) { return kTile * kNT + t * D; }
  __host__ __device__ static constexpr uint32_t col_p(int t) {
    return D >= 96 ? t * kTile : kTile * kNT + kNT * D + 64 * t;
  }
};

struct Bars {
  uint32_t base;
  int stages;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t kv_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t kv_empty(int s) const { return base + 8 * (1 + stages + s); }
  __device__ uint32_t s_full(int t) const { return base + 8 * (1 + 2 * stages + t); }
  // P_t for keys 64u .. 64u + 63 is in tensor memory (and O_t rescaled)
  __device__ uint32_t p_full(int t, int u) const { return base + 8 * ((u ? 8 : 3) + 2 * stages + t); }
  __device__ uint32_t o_done(int t) const { return base + 8 * (5 + 2 * stages + t); }
  __device__ uint32_t teardown() const { return base + 8 * (7 + 2 * stages); }
  // d = 64: the softmax warps of Q tile t have read S_t (128 arrivals), and
  // PV_t has completed, so its P_t columns may be rewritten
  __device__ uint32_t s_read(int t) const { return base + 8 * (10 + 2 * stages + t); }
  __device__ uint32_t pv_done(int t) const { return base + 8 * (12 + 2 * stages + t); }
};

// list entry: bits 0-11 key tile j; bits 12/13: Q tile 0/1 needs element-wise
// masking on it; bits 14/15: visited by Q tile 0/1
__device__ __forceinline__ int entry_j(uint32_t e) { return int(e & 0xFFFu); }
__device__ __forceinline__ bool entry_partial(uint32_t e, int t) { return (e >> (12 + t)) & 1u; }
__device__ __forceinline__ bool entry_act(uint32_t e, int t) { return (e >> (14 + t)) & 1u; }

enum Role : uint32_t { kRoleLoad = 1, kRoleMma = 2, kRoleSoftmax = 3 };

// kSplit: the keys are split over p.n_split CTAs per Q-tile pair and the epilogue writes this
// split's partial result (a separate instantiation, so the plain forward carries none of it).
// kF16: f16 elements instead of bf16 (Q, K, V, P and a 16-bit O). D is 64, 96 or 128: at 96 the
// tiles keep two 64-column chunks (the tensor maps read zeros in columns 96..127), the MMAs run 6
// K-steps over the head dimension and N = 96 (the PV MMA), and 96 columns of O are stored.
template <int D, bool kSplit, bool kF16, int kNT>
__global__ void __launch_bounds__(kThreadsFor<kNT>, kCtasPerSm<kNT>)
    fa_fwd_kernel(const __grid_constant__ FwdParams p) {
  using L = FwdLayout<D, kNT>;
  static_assert(kNT == 2 || (D == 64 && !kSplit), "one Q tile per CTA: d = 64 only");
  // d = 64 moves registers between the warpgroups (setmaxnreg, below)
  constexpr bool kMoveRegs = D == 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = smem_u32(smem);
  const uint32_t sQ = s_base + L::kQOff;
  const uint32_t sKV = s_base + L::kKVOff;
  uint16_t *list = reinterpret_cast<uint16_t *>(smem + L::kListOff);
  // [0] tmem base [1] count [2] abort [3] ring positions loaded in set-up
  // [4], [5] last list entry of Q tile 0 / 1 [6] head b * H + h (for the epilogue)
  int *misc = reinterpret_cast<int *>(smem + L::kMiscOff);
  Bars bars{s_base + L::kBarOff, L::kStages};
  StatusSlot st{p.status, &misc[2], p.wait_limit_ns};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // work item: head groups, heavy (late) Q-tile pairs first within a group;
  // the splits of one pair are adjacent, so they run together and share Q in L2
  const Shape &sh = p.sh;
  const int npairs = kNT == 2 ? (sh.tq + 1) >> 1 : sh.tq;  // work units per head
  const int n_split = kSplit ? p.n_split : 1;
  const int split = kSplit ? int(blockIdx.x % n_split) : 0;
  const int cta = kSplit ? int(blockIdx.x / n_split) : int(blockIdx.x);
  int pair;
  const int bh = fwd_item_head(cta, sh.bh, npairs, p.head_group, &pair);
  const int i0 = kNT * pair;
  const bool has1 = kNT == 2 && (i0 + 1) < sh.tq;
  const int b_idx = bh / sh.heads, h_idx = bh % sh.heads;

  // ---- setup -------------------------------------------------------------
  if (warp == 0 && lane == 0) {
    mbar_init(bars.q_full(), 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bars.kv_full(s), 1);
      mbar_init(bars.kv_empty(s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bars.s_full(t), 1);
      mbar_init(bars.p_full(t, 0), 128);
      mbar_init(bars.p_full(t, 1), 128);
    }
    for (int t = 0; t < 2; ++t) mbar_init(bars.o_done(t), 1);
    mbar_init(bars.teardown(), 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(bars.s_read(t), 128);
      mbar_init(bars.pv_done(t), 1);
    }
    misc[2] = 0;
    misc[6] = bh;
    fence_mbar_init();
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
    // the Q tiles do not depend on the tile list: load them now, while the
    // other warps set up
    if (!(p.debug_flags & kDebugSkipLoads)) {
      mbar_arrive_expect_tx(bars.q_full(), (has1 ? 2u : 1u) * L::kTileBytes);
      for (int c = 0; c < L::kChunks; ++c)
        tma_load_4d(sQ + c * L::kChunkBytes, &p.tm_q, c * 64, i0 * kTile, h_idx, b_idx,
                    bars.q_full());
      if (has1)
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_4d(sQ + L::kTileBytes + c * L::kChunkBytes, &p.tm_q, c * 64,
                      (i0 + 1) * kTile, h_idx, b_idx, bars.q_full());
    }
    // and the first K/V tile of the list (the smallest key tile either Q
    // tile sees) into ring positions 0 and 1; a split CTA starts further
    // into the list, which is known only after the list is built
    int pre = 0;
    if constexpr (!kSplit) {
      const int jmax0 = sh.last_kv_tile(i0);
      const int jmax1 = has1 ? sh.last_kv_tile(i0 + 1) : -1;
      int j0 = -1;
      for (int j = 0; j <= max(jmax0, jmax1) && j0 < 0; ++j)
        if ((j <= jmax0 && sh.mask_allows(i0, j)) || (j <= jmax1 && sh.mask_allows(i0 + 1, j)))
          j0 = j;
      if (j0 >= 0 && !(p.debug_flags & kDebugSkipLoads)) {
        for (int which = 0; which < 2; ++which) {
          mbar_arrive_expect_tx(bars.kv_full(which), L::kTileBytes);
          for (int c = 0; c < L::kChunks; ++c)
            tma_load_4d(sKV + which * L::kTileBytes + c * L::kChunkBytes,
                        which ? &p.tm_v : &p.tm_k, c * 64, j0 * kTile, h_idx, b_idx,
                        bars.kv_full(which));
        }
        pre = 2;
      }
    }
    misc[3] = pre;  // ring positions already issued
  } else if (warp == 1) {
    tmem_alloc(smem_u32(&misc[0]), L::kTmemCols);
    tmem_relinquish();
  } else if (warp == 2) {
    // K/V tiles visited by either Q tile, ascending, with per-tile flags
    const int i1 = i0 + 1;
    const int jmax0 = sh.last_kv_tile(i0);
    const int jmax1 = has1 ? sh.last_kv_tile(i1) : -1;
    const int jmax = max(jmax0, jmax1);
    int count = 0;
    for (int base = 0; base <= jmax; base += 32) {
      const int j = base + lane;
      const bool a0 = j <= jmax0 && sh.mask_allows(i0, j);
      const bool a1 = j <= jmax1 && sh.mask_allows(i1, j);
      const uint32_t ball = __ballot_sync(0xffffffffu, a0 || a1);
      if (a0 || a1) {
        const int slot = count + __popc(ball & ((1u << lane) - 1u));
        const uint32_t part = (a0 && sh.partial(i0, j) ? 1u << 12 : 0u) |
                              (a1 && sh.partial(i1, j) ? 1u << 13 : 0u);
        list[slot] = uint16_t(j | part | (a0 ? 1u << 14 : 0u) | (a1 ? 1u << 15 : 0u));
      }
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
    // the last entry each Q tile is active in (-1: none)
    __syncwarp();
    int last0 = -1, last1 = -1;
    for (int base = 0; base < count; base += 32) {
      const int n = base + lane;
      if (n < count) {
        const uint32_t e = list[n];
        if (entry_act(e, 0)) last0 = n;
        if (entry_act(e, 1)) last1 = n;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      last0 = max(last0, __shfl_xor_sync(0xffffffffu, last0, off));
      last1 = max(last1, __shfl_xor_sync(0xffffffffu, last1, off));
    }
    if (lane == 0) {
      misc[1] = count;
      misc[4] = last0;
      misc[5] = last1;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  const int count = misc[1];
  // d = 64: registers per thread by warpgroup, 88 for the producer / MMA
  // warpgroup and 208 for each softmax warpgroup (88 * 128 + 208 * 256 =
  // 168 * 384, the launch's total; one Q tile: 56 + 200 = 2 * 128), which
  // keeps the softmax loop free of spills; at d >= 96 the MMA issuer, with
  // twice the MMAs per step, runs slower with fewer registers and the split is
  // not made. Every wait and store below is inlined: an out-of-line call in a
  // kernel with its own register counts is not compiled, and the inlined
  // waits also measured faster at d >= 96.
  if (warp < 4) {
    if constexpr (kMoveRegs) setmaxnreg_dec<kRegsLoadMma<kNT>>();
    if (warp == 0) {
      // ---- TMA producer ------------------------------------------------------
      if (elect_one() && !(p.debug_flags & kDebugSkipLoads)) {
        int pos = misc[3];  // K and V of list[0] may have been issued during set-up
        bool ok = true;
        for (int n = pos / 2; n < count && ok; ++n) {
          const int kvrow = entry_j(list[n]) * kTile;
          for (int which = 0; which < 2 && ok; ++which, ++pos) {
            const int s = pos % L::kStages;
            const uint32_t u = pos / L::kStages;
            ok = mbar_wait_inl(bars.kv_empty(s), (u & 1u) ^ 1u, st, status_code(kKernFwd, kRoleLoad, 1));
            if (!ok) break;
            mbar_arrive_expect_tx(bars.kv_full(s), L::kTileBytes);
            const CUtensorMap *tm = which ? &p.tm_v : &p.tm_k;
            for (int c = 0; c < L::kChunks; ++c)
              tma_load_4d(sKV + s * L::kTileBytes + c * L::kChunkBytes, tm, c * 64, kvrow, h_idx,
                          b_idx, bars.kv_full(s));
          }
        }
        // teardown: wait (bounded) until every copy issued has landed (the Q
        // tiles were loaded during set-up)
        mbar_wait_drain_inl(bars.q_full(), 0, st, status_code(kKernFwd, kRoleLoad, 2));
        for (int s = 0; s < L::kStages && s < pos; ++s) {
          const int last = s + ((pos - 1 - s) / L::kStages) * L::kStages;  // last pos used on s
          mbar_wait_drain_inl(bars.kv_full(s), (last / L::kStages) & 1u, st,
                    status_code(kKernFwd, kRoleLoad, 3));
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ---- tcgen05 issuer ----------------------------------------------------
      if (elect_one()) {
        constexpr uint32_t kIdS = idesc_f32acc(kTile, kTile, 0, 0, kF16);  // Q K^T, both K-major
        constexpr uint32_t kIdPV = idesc_f32acc(kTile, D, 0, 1, kF16);     // P V, V is MN-major
        bool ok = count == 0 || mbar_wait_inl(bars.q_full(), 0, st, status_code(kKernFwd, kRoleMma, 1));
        uint32_t pcount[2] = {0, 0};
        bool first_pv[2] = {true, true};
        // d = 64: P_t has tensor-memory columns of its own, so S_t(n+1) waits
        // only until the softmax warps have read S_t(n) (s_read) and is issued
        // ahead of PV_t(n): the tensor core computes it while P_t(n) is formed,
        // which shortens the chain S -> P -> PV of a Q tile that runs alone
        // (block-sparse masks, causal edges)
        constexpr bool kEarlyS = D == 64 && !kSplit;
        uint32_t s_issued[2] = {0, 0};
        // misc[4 + t]: the last list entry Q tile t is active in (from warp 2)

        auto issue_s = [&](int t, int kslot) {
          const uint32_t q_base = sQ + t * L::kTileBytes;
          const uint32_t k_base = sKV + kslot * L::kTileBytes;
  #pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * L::kChunkBytes + (kk & 3) * 32;
            mma_f16kind_ss(tmem + t * kTile, sdesc_sw128(q_base + off, 16, 1024),
                        sdesc_sw128(k_base + off, 16, 1024), kIdS, kk > 0);
          }
        };
        // O_t += P_t V: A = P_t from tensor memory (8 columns per 16 keys),
        // B = V with keys as K (MN-major, 16 key rows per step). With d = 128,
        // S_t(n+1) is issued after this MMA into the columns P_t occupies; MMAs
        // issued by one thread execute in issue order, so P_t is read first.
        // (keys 64u .. 64u + 63: half u of P_t)
        auto issue_pv = [&](int t, int vslot, bool first, int u) {
          const uint32_t v_base = sKV + vslot * L::kTileBytes;
  #pragma unroll
          for (int kk = 4 * u; kk < 4 * u + 4; ++kk)
            mma_f16kind_ts(tmem + L::col_o(t), tmem + L::col_p(t) + kk * 8,
                        sdesc_sw128(v_base + kk * 16 * 128, L::kChunkBytes, 1024), kIdPV,
                        (kk > 0 || !first) ? 1u : 0u);
        };

        if (ok && count > 0) {
          // prologue: S for the first K tile
          ok = mbar_wait_inl(bars.kv_full(0), 0, st, status_code(kKernFwd, kRoleMma, 2));
          if (ok) {
            tc_fence_after();
            const uint32_t e = list[0];
            for (int t = 0; t < kNT; ++t)
              if (entry_act(e, t)) {
                issue_s(t, 0);
                mma_commit(bars.s_full(t));
                ++s_issued[t];
              }
            mma_commit(bars.kv_empty(0));
          }
        }
        for (int n = 0; n < count && ok; ++n) {
          const uint32_t e = list[n];
          const int vpos = 2 * n + 1, kpos = 2 * n + 2;
          const int vslot = vpos % L::kStages, kslot = kpos % L::kStages;
          const bool has_next = n + 1 < count;
          const uint32_t en = has_next ? list[n + 1] : 0u;
          ok = mbar_wait_inl(bars.kv_full(vslot), (vpos / L::kStages) & 1u, st,
                         status_code(kKernFwd, kRoleMma, 3));
          if (ok && has_next)
            ok = mbar_wait_inl(bars.kv_full(kslot), (kpos / L::kStages) & 1u, st,
                           status_code(kKernFwd, kRoleMma, 4));
          if (!ok) break;
          tc_fence_after();
          if constexpr (kEarlyS) {
            for (int t = 0; t < kNT && ok; ++t) {
              if (!(has_next && entry_act(en, t))) continue;
              // the previous S_t has been read out of its columns
              ok = mbar_wait_inl(bars.s_read(t), (s_issued[t] - 1) & 1u, st,
                                 status_code(kKernFwd, kRoleMma, 11 + t));
              if (!ok) break;
              tc_fence_after();
              issue_s(t, kslot);
              mma_commit(bars.s_full(t));
              ++s_issued[t];
            }
            if (!ok) break;
          }
          for (int t = 0; t < kNT && ok; ++t) {
            if (entry_act(e, t)) {
              // PV_t in two halves: the first runs while the softmax warps
              // form the second half of P_t (the split-key instantiation waits
              // for all of P_t on p_full(t, 1))
              if constexpr (!kSplit) {
                ok = mbar_wait_inl(bars.p_full(t, 0), pcount[t] & 1u, st,
                               status_code(kKernFwd, kRoleMma, 5 + t));
                if (!ok) break;
                tc_fence_after();
                issue_pv(t, vslot, first_pv[t], 0);
              }
              ok = mbar_wait_inl(bars.p_full(t, 1), pcount[t] & 1u, st,
                             status_code(kKernFwd, kRoleMma, 9 + t));
              if (!ok) break;
              ++pcount[t];
              tc_fence_after();
              if constexpr (kSplit) issue_pv(t, vslot, first_pv[t], 0);
              issue_pv(t, vslot, first_pv[t], 1);
              first_pv[t] = false;
              // O_t is final once this entry's PV has completed: under causal
              // masking Q tile 0 usually ends one K/V tile before Q tile 1, and
              // its epilogue then overlaps tile 1's last step
              if (n == *reinterpret_cast<volatile int *>(&misc[4 + t])) mma_commit(bars.o_done(t));
              if constexpr (kEarlyS) mma_commit(bars.pv_done(t));
            }
            if (!kEarlyS && has_next && entry_act(en, t)) {
              issue_s(t, kslot);
              mma_commit(bars.s_full(t));
            }
          }
          if (!ok) break;
          mma_commit(bars.kv_empty(vslot));
          if (has_next) mma_commit(bars.kv_empty(kslot));
        }
        // teardown: every MMA this thread issued has completed
        mma_commit(bars.teardown());
        mbar_wait_drain_inl(bars.teardown(), 0, st, status_code(kKernFwd, kRoleMma, 8));
      }
      __syncwarp();
    }
  } else {
    if constexpr (kMoveRegs) setmaxnreg_inc<kRegsSoftmax<kNT>>();
    // ---- softmax -----------------------------------------------------------
    const int t = (warp - 4) >> 2;                 // Q tile of this warpgroup
    const int r = threadIdx.x - 128 * (1 + t);     // row within the tile = TMEM lane
    const int qi = i0 + t;                         // Q tile index
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * kTile;
    const uint32_t tO = tmem + lane_off + L::col_o(t);
    const uint32_t tP = tmem + lane_off + L::col_p(t);
    const float c = p.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    uint32_t scount = 0;
    bool ok = true, any = false;

    if (t == 0 || has1) {
      for (int n = 0; n < count; ++n) {
        const uint32_t e = list[n];
        if (!entry_act(e, t)) continue;
        ok = __all_sync(0xffffffffu, mbar_wait_inl(bars.s_full(t), scount & 1u, st,
                                               status_code(kKernFwd, kRoleSoftmax, 1 + t)));
        // d = 64: S_t(n) was issued ahead of PV_t(n-1), so its completion no
        // longer implies that PV_t(n-1) has read P_t and written O_t; wait for
        // that before this step rewrites them
        constexpr bool kEarlyS = D == 64 && !kSplit;
        if (kEarlyS && ok && any)
          ok = __all_sync(0xffffffffu, mbar_wait_inl(bars.pv_done(0) + ((~threadIdx.x & 128u) >> 4),
                                                     (scount - 1) & 1u, st,
                                                     status_code(kKernFwd, kRoleSoftmax, 4)));
        if (!ok) break;
        ++scount;
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32(tS + q * 32, sr[q]);
        tmem_wait_ld();
        if constexpr (kEarlyS) {  // S_t's columns may take S_t(n+1)
          tc_fence_before();
          mbar_arrive(bars.s_read(0) + ((~threadIdx.x & 128u) >> 4));
        }
        float s[kTile];
#pragma unroll
        for (int x = 0; x < kTile; ++x) s[x] = __uint_as_float(sr[x >> 5][x & 31]);
        if (entry_partial(e, t)) {  // keys x >= lim are hidden from this row
          const int lim = sh.key_limit(qi, r, entry_j(e));
#pragma unroll
          for (int x = 0; x < kTile; ++x)
            if (x >= lim) s[x] = -INFINITY;
        }
        // row max with 4 independent partial maxima (short dependency chains),
        // two new elements per three-input max
        float mp[4];
#pragma unroll
        for (int y = 0; y < 4; ++y) mp[y] = fmaxf(s[2 * y], s[2 * y + 1]);
#pragma unroll
        for (int x = 8; x < kTile; x += 8)
#pragma unroll
          for (int y = 0; y < 4; ++y) mp[y] = fmax3(mp[y], s[x + 2 * y], s[x + 2 * y + 1]);
        const float mx = fmax3(mp[0], mp[1], fmaxf(mp[2], mp[3]));
        const float m_tile = mx * c;
        const bool need = m_tile > m_used + kRescaleThreshold;
        float alpha = 1.f;
        if (need) {
          alpha = ex2_approx(m_used - m_tile);  // 0 on the first tile (m_used = -inf)
          m_used = m_tile;
        }
        const float m_sub = (m_used == -INFINITY) ? 0.f : m_used;
        // (the split-key instantiation announces all of P_t at once: the
        // early announcement costs it spills at the register limit)
        const bool resc = kSplit || (any && __any_sync(0xffffffffu, need));
        // P = exp2(s*c - m) -> 16-bit pairs (keys 2x, 2x+1 in column x) in tensor
        // memory; the scaling and the row sum on packed fp32 pairs (one
        // instruction per two keys; the row sum in 4 independent partial sums)
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
        tmem_st32(tP, pk0);
        // keys 0..63 of P_t go to the MMA now, unless this warp's rows must
        // first rescale O_t (then both halves are announced below); the
        // barrier of this warpgroup's tile from threadIdx (fewer live registers)
        if (!resc) {
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bars.p_full(0, 0) + ((~threadIdx.x & 128u) >> 4));
        }
#pragma unroll
        for (int x = 0; x < 32; ++x) pk1[x] = p_pair(x, s[64 + 2 * x], s[64 + 2 * x + 1]);
        tmem_st32(tP + 32, pk1);
        float lp[2];
        f2unpack(fadd2(lp2[0], lp2[1]), lp[0], lp[1]);
        l = l * alpha + (lp[0] + lp[1]);
        if (resc && any && __any_sync(0xffffffffu, need)) {
          // O *= alpha for this row. The PV MMA of the previous tile has
          // completed: it was issued before this S tile, whose completion we
          // waited for (d = 64: pv_done, waited for above).
#pragma unroll
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
        if (resc && !kSplit) mbar_arrive(bars.p_full(0, 0) + ((~threadIdx.x & 128u) >> 4));
        if constexpr (kSplit)
          mbar_arrive(bars.p_full(t, 1));
        else
          mbar_arrive(bars.p_full(0, 1) + ((~threadIdx.x & 128u) >> 4));
        any = true;
      }
      // epilogue: O / l and LSE
      if (ok && any)
        // this warpgroup's o_done(t), its address from threadIdx (an address
        // computed from t here costs the softmax loop registers and spills)
        ok = __all_sync(0xffffffffu, mbar_wait_inl(bars.o_done(0) + ((~threadIdx.x & 128u) >> 4), 0, st,
                                               status_code(kKernFwd, kRoleSoftmax, 3)));
      // tensor-memory loads are warp-wide; rows past the sequence end store nothing
      const int qrow = qi * kTile + r;  // query row within the head
      const bool live = qrow < sh.nq;
      if (ok) {
        tc_fence_after();
        // destination of this row (indices recomputed here: fewer live registers):
        // O itself, or this split's fp32 partial
        const int bh_e = *reinterpret_cast<volatile int *>(&misc[6]);
        constexpr bool to_part = kSplit;
        const size_t prow = ((size_t)split * sh.bh + bh_e) * sh.nq + qrow;
        const size_t row = to_part ? prow * D : p.so.row(bh_e / sh.heads, bh_e % sh.heads, qrow);
        float *const o32 = to_part ? p.o_part : static_cast<float *>(p.o);
        const float inv_l = (any && l > 0.f) ? 1.f / l : 0.f;
        if (!kSplit && !p.o_f32 && any) {
          // 16-bit O through this tile's Q buffer, which the MMAs no longer
          // read (any: its Q load has landed, since the MMAs used it; a tile
          // without keys stores its zeros directly below)
          store_rows_tma_inl<D, kF16>(&p.tm_o, tO, sQ + t * L::kTileBytes, r, qi * kTile, 0, inv_l,
                                  any, sh.d, sh.nq, bh_e % sh.heads, bh_e / sh.heads);
        } else {
#pragma unroll
          for (int q = 0; q < D / 32; ++q) {
            uint32_t o[32];
            if (any) {
              tmem_ld32(tO + q * 32, o);
              tmem_wait_ld();
            } else {
#pragma unroll
              for (int x = 0; x < 32; ++x) o[x] = 0u;
            }
            if (!live) {
            } else if (to_part || p.o_f32) {
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
        }
        // LSE = ln(sum_j exp(scale s_ij)) = ln2 * (m + log2 l)
        if (live)
          (to_part ? p.lse_part[prow] : p.lse[(size_t)bh_e * sh.nq + qrow]) =
              (any && l > 0.f) ? (m_used + lg2_approx(l)) * 0.69314718055994531f : -INFINITY;

      }
    }
  }

  // ---- teardown ------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// Merge of the n_split partial results of one query row (see the top of the
// file): thread = 8 consecutive columns of a row; the row's n_split LSE values
// are read by each of its D/8 threads (L1 broadcast). HBM-bound:
// n_split * (4d + 4) bytes read and 2d + 4 (16-bit O) written per row.
template <int D, bool kF16>
__global__ void __launch_bounds__(256) fa_fwd_combine(const __grid_constant__ FwdParams p) {
  constexpr int kLanes = D / 8;
  const Shape &sh = p.sh;
  const size_t rows = (size_t)sh.bh * sh.nq;
  const size_t gt = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t row = gt / kLanes;  // bh * nq + n
  const int part = int(gt % kLanes);
  if (row >= rows || part * 8 >= sh.d) return;
  float m = -INFINITY;
  for (int s = 0; s < p.n_split; ++s) m = fmaxf(m, p.lse_part[s * rows + row]);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float l = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < p.n_split; ++s) {
      const float w = expf(p.lse_part[s * rows + row] - m);  // e^(m_s - m) l_s
      const float4 *src = reinterpret_cast<const float4 *>(p.o_part + (s * rows + row) * D + part * 8);
      const float4 a = src[0], b = src[1];
      l += w;
      acc[0] = fmaf(w, a.x, acc[0]); acc[1] = fmaf(w, a.y, acc[1]);
      acc[2] = fmaf(w, a.z, acc[2]); acc[3] = fmaf(w, a.w, acc[3]);
      acc[4] = fmaf(w, b.x, acc[4]); acc[5] = fmaf(w, b.y, acc[5]);
      acc[6] = fmaf(w, b.z, acc[6]); acc[7] = fmaf(w, b.w, acc[7]);
    }
  }
  const float inv_l = l > 0.f ? 1.f / l : 0.f;
  const int bh = int(row / sh.nq), n = int(row % sh.nq);
  const size_t dst = p.so.row(bh / sh.heads, bh % sh.heads, n) + part * 8;
  if (p.o_f32) {
    float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(p.o) + dst);
    o[0] = make_float4(acc[0] * inv_l, acc[1] * inv_l, acc[2] * inv_l, acc[3] * inv_l);
    o[1] = make_float4(acc[4] * inv_l, acc[5] * inv_l, acc[6] * inv_l, acc[7] * inv_l);
  } else {
    *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.o) + dst) =
        make_uint4(pack2<kF16>(acc[0] * inv_l, acc[1] * inv_l), pack2<kF16>(acc[2] * inv_l, acc[3] * inv_l),
                   pack2<kF16>(acc[4] * inv_l, acc[5] * inv_l), pack2<kF16>(acc[6] * inv_l, acc[7] * inv_l));
  }
  if (part == 0) p.lse[row] = l > 0.f ? m + logf(l) : -INFINITY;
}

template <int D, bool kF16>
cudaError_t launch_combine(const FwdParams &p, cudaStream_t stream) {
  const size_t threads = (size_t)p.sh.bh * p.sh.nq * (D / 8);
  LaunchProbe probe(kKindFwdCombine, stream);
  fa_fwd_combine<D, kF16><<<(unsigned)((threads + 255) / 256), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

// Sets the kernel's shared-memory size and checks its register count, once.
template <int D, bool kSplit, bool kF16, int kNT>
cudaError_t configure_fwd() {
  static cudaError_t status = [] {
    cudaError_t e = cudaFuncSetAttribute(fa_fwd_kernel<D, kSplit, kF16, kNT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         FwdLayout<D, kNT>::kAlloc);
    if (e == cudaSuccess) e = check_kernel_regs(fa_fwd_kernel<D, kSplit, kF16, kNT>, kRegsLaunch<kNT>);
    return e;
  }();
  return status;
}

template <int D, bool kSplit, bool kF16, int kNT>
cudaError_t launch_fwd_kernel(const FwdParams &p, cudaStream_t stream) {
  const cudaError_t e = configure_fwd<D, kSplit, kF16, kNT>();
  if (e != cudaSuccess) return e;
  const int units = kNT == 2 ? (p.sh.tq + 1) / 2 : p.sh.tq;
  const int grid = units * p.sh.bh * (kSplit ? p.n_split : 1);
  LaunchProbe probe(kKindFwd, stream);
  fa_fwd_kernel<D, kSplit, kF16, kNT>
      <<<grid, kThreadsFor<kNT>, FwdLayout<D, kNT>::kAlloc, stream>>>(p);
  return cudaGetLastError();
}

// d = 64 without the key split: one Q tile per CTA (two CTAs per SM) under a
// block mask, where a pair of Q tiles walks the union of its two tile lists
// and often has one tile idle, and where the pairs would fill at most four
// waves of the GPU, whose CTAs' set-up and epilogue then overlap the other
// CTA's steps; pairs otherwise (measured at B4 H16 N4096: dense 8 % and causal
// 1.5 % faster with pairs; block-sparse N8192 19 % and B8 H12 N1024 causal
// 10 % faster with one tile).
bool fwd_one_tile(const FwdParams &p) {
  if (p.q_tiles) return p.q_tiles == 1;
  if (p.sh.mask) return true;
  const long long pairs = (long long)((p.sh.tq + 1) / 2) * p.sh.bh;
  return p.sms > 0 && pairs <= 4LL * p.sms;
}

template <int D, bool kF16>
cudaError_t launch_fwd_d(const FwdParams &p, cudaStream_t stream) {
  cudaError_t e;
  if (p.n_split > 1)
    e = launch_fwd_kernel<D, true, kF16, 2>(p, stream);
  else if constexpr (D == 64)
    e = fwd_one_tile(p) ? launch_fwd_kernel<D, false, kF16, 1>(p, stream)
                        : launch_fwd_kernel<D, false, kF16, 2>(p, stream);
  else
    e = launch_fwd_kernel<D, false, kF16, 2>(p, stream);
  if (e != cudaSuccess || p.n_split == 1) return e;
  return launch_combine<D, kF16>(p, stream);
}

}  // namespace

cudaError_t launch_forward(const FwdParams &p, cudaStream_t stream) {
  const bool f16 = p.sh.f16 != 0;
  if (p.sh.d == 64) return f16 ? launch_fwd_d<64, true>(p, stream) : launch_fwd_d<64, false>(p, stream);
  if (p.sh.d == 96) return f16 ? launch_fwd_d<96, true>(p, stream) : launch_fwd_d<96, false>(p, stream);
  if (p.sh.d == 128)
    return f16 ? launch_fwd_d<128, true>(p, stream) : launch_fwd_d<128, false>(p, stream);
  if (p.sh.d == 256) {  // its own kernel (fa_fwd_d256.cu); the merge is shared
    cudaError_t e = launch_forward_d256(p, stream);
    if (e != cudaSuccess || p.n_split == 1) return e;
    return f16 ? launch_combine<256, true>(p, stream) : launch_combine<256, false>(p, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace fa
