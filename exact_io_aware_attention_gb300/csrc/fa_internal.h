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

struct FwdParams {
  CUtensorMap tm_q, tm_k, tm_v;       // 2-D bf16 maps [B*H*N rows][d], box 64 x 128, 128B swizzle
  void *o;                            // bf16 or fp32 [B*H*N][d]
  float *lse;                         // [B*H*N]
  const uint8_t *mask;                // [T][T] or null
  int bh, n, d, causal;
  int o_f32;                          // 1: O stored as fp32
  float scale_log2;                   // scale * log2(e)
  unsigned int *status;               // device status word
  uint32_t debug_flags;               // kDebug* bits (tests of the failure path only)
  uint64_t wait_limit_ns;             // limit of one kernel-side wait
};

struct BwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do; // as in FwdParams
  const void *o, *dout;               // bf16 [B*H*N][d]
  const float *lse;                   // [B*H*N]
  float *delta;                       // workspace: D_i [B*H*N]
  float *lse2;                        // workspace: LSE_i * log2(e) [B*H*N]
  void *dq, *dk, *dv;                 // bf16 outputs
  const uint8_t *mask;
  int bh, n, d, causal;
  int head_group;                     // CTA order: heads per group (1..bh)
  float scale, scale_log2;
  unsigned int *status;
  uint32_t debug_flags;
  uint64_t wait_limit_ns;
};

// Kernel ids of the measurement hooks (names in fa_kernel_name()).
enum KernelKind : int { kKindFwd = 0, kKindBwdPre = 1, kKindBwdDkdv = 2, kKindBwdDq = 3,
                        kNumKinds = 4 };

// Brackets one launch with CUDA events when measurement is enabled
// (fa_profile_enable); a no-op otherwise.
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

cudaError_t launch_forward(const FwdParams &p, cudaStream_t stream);
cudaError_t launch_backward(const BwdParams &p, cudaStream_t stream);
cudaError_t launch_backward_dq(const BwdParams &p, cudaStream_t stream);  // fa_bwd_dq.cu

// Status word codes: 0x80000000 | kernel << 16 | role << 8 | site.
enum KernelId : uint32_t { kKernFwd = 1, kKernBwdPre = 2, kKernBwd = 3, kKernBwdDq = 4 };
__host__ __device__ constexpr uint32_t status_code(uint32_t kernel, uint32_t role, uint32_t site) {
  return 0x80000000u | (kernel << 16) | (role << 8) | site;
}

}  // namespace fa
