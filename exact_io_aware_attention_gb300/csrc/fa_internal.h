// Internal interface between the C-ABI layer (fa_api.cu) and the kernel
// translation units. Not installed; not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

constexpr int kTile = 128;            // rows of a Q tile and keys of a K/V tile
constexpr int kMaxTiles = 512;        // tiles per sequence the kernels accept (N <= 65536)
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // default limit of one kernel-side wait

// Element strides of one [B][H][rows][d] operand: element (b, h, n, c) is at
// base + b * b_ + h * h_ + n * n_ + c.
struct RowStrides {
  long long b_, h_, n_;
  __host__ __device__ size_t row(int bi, int hi, int n) const {
    return (size_t)((long long)bi * b_ + (long long)hi * h_ + (long long)n * n_);
  }
};

// Shape of one attention problem per (batch, head): nq query rows, nk keys,
// in tq = ceil(nq/128) Q tiles and tk = ceil(nk/128) K/V tiles. Query i sees
// key j iff j < nk, (!causal || j <= i + causal_off) and the block mask
// allows tile (i/128, j/128); causal_off = nk - nq aligns the last query with
// the last key.
struct Shape {
  int bh, heads;                      // B*H and H (bh = b * heads + h)
  int nq, nk, tq, tk;
  int d, causal, causal_off;          // d: the head dimension (64, 96, 128 or 256)
  int f16;                            // 16-bit element type: 1 = f16, 0 = bf16
  const uint8_t *mask;                // [tq][tk] or null

  // Largest K/V tile with a key visible to some row of Q tile i, or -1.
  __host__ __device__ int last_kv_tile(int i) const {
    if (!causal) return tk - 1;
    const int last_q = min(kTile * i + kTile - 1, nq - 1);
    const int last_k = last_q + causal_off;             // last visible key of that row
    if (last_k < 0) return -1;
    return min(last_k / kTile, tk - 1);
  }
  // Smallest Q tile with a row that sees a key of K/V tile j, or tq if none.
  __host__ __device__ int first_q_tile(int j) const {
    if (!causal) return 0;
    const int first_q = kTile * j - causal_off;         // first row that sees key 128 j
    if (first_q > nq - 1) return tq;
    return first_q <= 0 ? 0 : first_q / kTile;
  }
  // Whether some (query, key) pair of tile (i, j) is hidden by the key count
  // or by causality, so that the tile needs element-wise masking.
  __host__ __device__ bool partial(int i, int j) const {
    if (kTile * j + kTile > nk) return true;
    return causal && kTile * j + kTile - 1 > kTile * i + causal_off;
  }
  // Keys x < key_limit(i, r, j) of K/V tile j are visible to row r of Q tile i.
  __host__ __device__ int key_limit(int i, int r, int j) const {
    int lim = nk - kTile * j;
    if (causal) lim = min(lim, kTile * (i - j) + r + causal_off + 1);
    return lim;
  }
  __host__ __device__ bool mask_allows(int i, int j) const {
    return !mask || mask[(size_t)i * tk + j] != 0;
  }
};

// Work order of a forward grid: item `cta` (0 .. units*bh - 1; the split
// CTAs of one item share it) runs unit `*unit` (a Q-tile pair, or a Q tile)
// of head `bh`. Heads go in groups of `hg`; within a group the heavy units
// (late Q tiles under causal masking) come first, so the CTAs in flight at
// any time cover only a few heads and those heads' K and V stay in L2.
__host__ __device__ inline int fwd_item_head(int cta, int bh, int units, int hg, int *unit) {
  const int group = cta / (hg * units);
  const int g_base = group * hg;
  const int g_size = min(hg, bh - g_base);
  const int g_rank = cta - group * hg * units;
  *unit = units - 1 - g_rank / g_size;
  return g_base + g_rank % g_size;
}

struct FwdParams {
  // 4-D maps over [B][H][rows][d] (dims d, rows, H, B) of bf16 or f16 elements,
  // box 64 x 128 x 1 x 1, 128-byte swizzle; rows past the end of a head and
  // columns past d read zeros
  CUtensorMap tm_q, tm_k, tm_v;
  CUtensorMap tm_o;                   // map over O (16-bit O only) with a 64 x 32 box, for TMA stores
  Shape sh;
  void *o;                            // 16-bit (the inputs' type) or fp32 rows, strides so
  RowStrides so;
  float *lse;                         // [B*H][nq]
  int o_f32;                          // 1: O stored as fp32
  // Split over the keys: n_split CTAs share the K/V tiles of one Q-tile pair
  // and write partial results, which fa_fwd_combine merges into O and LSE.
  int n_split;                        // 1: no split (o_part, lse_part unused)
  float *o_part;                      // [n_split][B*H][nq][d]: O of each split, normalised
  float *lse_part;                    // [n_split][B*H][nq]: LSE of each split (-inf: no key)
  float scale_log2;                   // scale * log2(e)
  unsigned int *status;               // device status word
  uint32_t debug_flags;               // kDebug* bits (tests of the failure path only)
  uint64_t wait_limit_ns;             // limit of one kernel-side wait
  int head_group;                     // CTA order: heads per group (1..bh), fwd_item_head
  int q_tiles;                        // d = 64 without a split: Q tiles per CTA, 1 or 2 (0: the
                                      // launch chooses)
  int sms;                            // SM count (0: unknown)
};

struct BwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do; // as in FwdParams
  CUtensorMap tm_dq, tm_dk, tm_dv;     // maps over the gradients, 64 x 32 boxes (TMA stores)
  CUtensorMap tm_dqacc;                // one-pass backward at d = 128: 2-D map over dq_acc
                                       // ([rows][128] fp32), 32 x 32 boxes, 128-byte swizzle
  CUtensorMap tm_qh, tm_doh;           // one-pass backward at d = 128: Q and dO with 64-row boxes
  Shape sh;
  const void *o, *dout;               // 16-bit rows, strides so / sdo
  RowStrides so, sdo;
  const float *lse;                   // [B*H][nq]
  float *delta;                       // workspace: D_i, [B*H][tq*128]
  float *lse2;                        // workspace: LSE_i * log2(e), [B*H][tq*128]
  float *dq_acc;                      // workspace: fp32 dQ accumulator [B*H][tq*128][d] of the
                                      // one-pass backward (null: the two-kernel backward)
  void *dq, *dk, *dv;                 // 16-bit outputs, strides sdq / sdk / sdv
  RowStrides sdq, sdk, sdv;
  int head_group;                     // CTA order: heads per group (1..bh)
  float scale, scale_log2;
  unsigned int *status;
  uint32_t debug_flags;
  uint64_t wait_limit_ns;
};

// Kernel ids of the measurement hooks (names in fa_kernel_name()).
enum KernelKind : int { kKindFwd = 0, kKindBwdPre = 1, kKindBwdDkdv = 2, kKindBwdDq = 3,
                        kKindFwdCombine = 4, kKindBwd256Dv = 5, kKindBwd256Dk = 6,
                        kKindBwd256Dq = 7, kKindBwdFused = 8, kKindBwdConvert = 9,
                        kNumKinds = 10 };

// Brackets one launch with CUDA events when measurement is enabled
// (fa_profile_enable); a no-op otherwise.
// A kernel whose warpgroups move registers between them (setmaxnreg) must be
// compiled to exactly the register count its split assumes: with fewer, an
// increase would wait for registers the launch never allocated. The launch
// functions check the compiled count once per kernel and refuse to launch on
// a mismatch (cudaErrorInvalidKernelImage).
template <typename Kernel>
inline cudaError_t check_kernel_regs(Kernel kernel, int expected) {
  cudaFuncAttributes a;
  const cudaError_t e = cudaFuncGetAttributes(&a, reinterpret_cast<const void *>(kernel));
  if (e != cudaSuccess) return e;
  return a.numRegs == expected ? cudaSuccess : cudaErrorInvalidKernelImage;
}

class LaunchProbe {
 public:
  LaunchProbe(int kind, cudaStream_t stream);
  ~LaunchProbe();
 private:
  int slot_;
  cudaStream_t stream_;
};

// Debug flags (fa_debug_configure): the TMA producers issue no copy, so the
// consumers' bounded waits run out and report through the status word.
constexpr uint32_t kDebugSkipLoads = 1u;

cudaError_t launch_forward(const FwdParams &p, cudaStream_t stream);  // + the merge when split
cudaError_t launch_forward_d256(const FwdParams &p, cudaStream_t stream);  // fa_fwd_d256.cu
cudaError_t launch_backward(const BwdParams &p, cudaStream_t stream);
cudaError_t launch_backward_dq(const BwdParams &p, cudaStream_t stream);  // fa_bwd_dq.cu
// dK, dV and the dQ partials in one kernel, then the dQ conversion, after
// fa_bwd_pre has zeroed p.dq_acc; head dimensions 64, 96, 128 (fa_bwd_fused.cu)
cudaError_t launch_backward_fused(const BwdParams &p, cudaStream_t stream);
// The one-pass kernel for head dimension 128 in 64-query steps (fa_bwd_fused_q64.cu)
cudaError_t launch_backward_fused_q64(const BwdParams &p, cudaStream_t stream);
// dV, dK and dQ for head dimension 256, after fa_bwd_pre (fa_bwd_d256.cu)
cudaError_t launch_backward_d256(const BwdParams &p, cudaStream_t stream);

// Status word codes: 0x80000000 | kernel << 16 | role << 8 | site.
enum KernelId : uint32_t { kKernFwd = 1, kKernBwdPre = 2, kKernBwd = 3, kKernBwdDq = 4,
                           kKernBwd256Dv = 5, kKernBwd256Dk = 6, kKernBwd256Dq = 7,
                           kKernBwdFused = 8 };
__host__ __device__ constexpr uint32_t status_code(uint32_t kernel, uint32_t role, uint32_t site) {
  return 0x80000000u | (kernel << 16) | (role << 8) | site;
}

}  // namespace fa
