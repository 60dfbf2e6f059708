// C-ABI layer: argument validation, TMA tensor-map encoding and kernel launch.
// The declarations and the contract of every entry point are in include/fa.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

// NVTX range around the work an entry point enqueues (visible in profilers
// that record NVTX; a no-op otherwise).
struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

// Device status word written by kernel-side bounded waits that give up.
__device__ unsigned int g_status_word = 0u;

// Process-wide debug settings (fa_debug_configure).
std::atomic<uint32_t> g_debug_flags{0};
std::atomic<unsigned long long> g_wait_limit_ns{0};  // 0: the default limit

// Text of the last FA_ERR_CUDA failure of the calling thread.
thread_local char g_last_error[256] = "";

fa_status cuda_fail(const char *where, cudaError_t e) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", where, cudaGetErrorString(e),
           (int)e);
  return FA_ERR_CUDA;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encoder() {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}

cudaError_t status_word(unsigned int **out) {
  // looked up on the calling thread's current device at every call
  void *ptr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&ptr, g_status_word);
  *out = static_cast<unsigned int *>(ptr);
  return e;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Element strides of an operand, validated: every stride of a dimension
// longer than 1 is positive, a multiple of 16 bytes and below 2^40 bytes
// (the tensor-map limits, which the 16-byte vector loads and stores of the
// kernels also need); a dimension of length 1 gets a placeholder stride.
fa_status operand_strides(const fa_tensor *t, int B, int H, int rows, int d, int elem_bytes,
                          const char *name, fa::RowStrides *out) {
  if (!t || !t->data) {
    snprintf(g_last_error, sizeof(g_last_error), "%s: null tensor", name);
    return FA_ERR_INVALID_ARG;
  }
  if (t->reserved != 0) {
    snprintf(g_last_error, sizeof(g_last_error), "%s: reserved field is not 0", name);
    return FA_ERR_INVALID_ARG;
  }
  if (!aligned16(t->data)) {
    snprintf(g_last_error, sizeof(g_last_error), "%s: data %p is not 16-byte aligned", name,
             t->data);
    return FA_ERR_MISALIGNED;
  }
  const long long ext[3] = {B, H, rows};
  long long st[3] = {t->stride_b, t->stride_h, t->stride_n};
  const long long unit = 16 / elem_bytes;
  for (int k = 0; k < 3; ++k) {
    if (ext[k] <= 1) {
      st[k] = d;  // never multiplied by a non-zero index
      continue;
    }
    if (st[k] <= 0 || st[k] >= (1LL << 40) / elem_bytes) {
      snprintf(g_last_error, sizeof(g_last_error), "%s: stride %lld of dimension %d unsupported",
               name, st[k], k);
      return FA_ERR_UNSUPPORTED;
    }
    if (st[k] % unit != 0) {
      snprintf(g_last_error, sizeof(g_last_error),
               "%s: stride %lld of dimension %d is not a multiple of 16 bytes", name, st[k], k);
      return FA_ERR_MISALIGNED;
    }
  }
  *out = fa::RowStrides{st[0], st[1], st[2]};
  return FA_OK;
}

// 4-D map of 16-bit elements (bf16 or f16) over [B][H][rows][d] (dims d, rows,
// H, B): box = 64 columns (128 bytes) x 128 rows x 1 x 1, 128-byte swizzle. A
// box that runs past `rows` reads zeros there and never the next head; one
// that runs past column d (d = 96) reads zeros in the missing columns.
bool encode_operand(CUtensorMap *m, const void *base, const fa::RowStrides &st, int B, int H,
                    int rows, int d, bool f16, int box_rows = fa::kTile) {
  EncodeTiledFn enc = encoder();
  if (!enc) {
    snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled unavailable");
    return false;
  }
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)H, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)st.n_ * 2, (cuuint64_t)st.h_ * 2,
                                 (cuuint64_t)st.b_ * 2};
  const cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, 1};
  const cuuint32_t elem[4] = {1, 1, 1, 1};
  const CUresult r =
      enc(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
          const_cast<void *>(base), dims, strides, box,
          elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    snprintf(g_last_error, sizeof(g_last_error),
             "cuTensorMapEncodeTiled(base=%p, B=%d, H=%d, rows=%d, d=%d, strides=%lld/%lld/%lld)"
             " failed: CUresult %d",
             base, B, H, rows, d, st.b_, st.h_, st.n_, (int)r);
  return r == CUDA_SUCCESS;
}

// 2-D map over the one-pass backward's fp32 dQ accumulator: `rows` rows of d
// floats, 32 x 32 boxes (128 bytes wide) in the 128-byte swizzle, for the
// kernels' TMA tensor reductions.
bool encode_dq_acc(CUtensorMap *m, float *base, long long rows, int d) {
  EncodeTiledFn enc = encoder();
  if (!enc) {
    snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled unavailable");
    return false;
  }
  const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d * 4};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t elem[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, elem,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    snprintf(g_last_error, sizeof(g_last_error),
             "cuTensorMapEncodeTiled(dQ accumulator %p, rows=%lld, d=%d) failed: CUresult %d",
             (void *)base, rows, d, (int)r);
  return r == CUDA_SUCCESS;
}

int sm_count();

// Heads per CTA group of the backward grid, whose CTAs run heavy K/V tiles
// first within each group. Groups are kept small so that the fp32 dQ rows
// the CTAs in flight accumulate stay in L2: 8 heads. With at most 8 K/V tiles
// per head (N <= 1024) a group of 8 holds less than half a wave of CTAs and
// the heavy-first order no longer balances the SMs, so a group holds two
// waves there (measured at N = 1024, d = 64 and 128: 2-5 % faster than 8;
// the dQ rows in flight stay near 2 * SMs * 128). Longer sequences keep 8:
// at N = 4096, groups of 8 and 16 measured level and 10 measured 4.7 %
// slower. FA_BWD_HEAD_GROUP overrides it for tuning runs.
int backward_head_group(int bh, int tk) {
  const char *e = getenv("FA_BWD_HEAD_GROUP");
  const int from_env = e ? atoi(e) : 0;
  int g = from_env;
  if (g <= 0) {
    const int sms = sm_count();
    g = 8;
    if (tk > 0 && tk <= 8 && sms > 0) {
      const int two_waves = (2 * sms + tk - 1) / tk;
      if (two_waves > g) g = two_waves;
    }
  }
  return g < bh ? g : bh;
}

// Heads per CTA group of the forward grid (fwd_item_head). When the K and V
// of all heads exceed half of L2, groups of 8 heads keep the CTAs in flight on
// a few heads, whose K and V then stay in L2 (measured at B4 H16 N4096 d128:
// DRAM reads 2.6x -> 1.0x the algorithmic bytes, 2.6-3.5 % faster). Smaller
// problems fit in L2 anyway and run best with every head's heavy Q tiles
// first (one group). FA_FWD_HEAD_GROUP overrides it for tuning runs.
int forward_head_group(int bh, int nk, int d) {
  const char *e = getenv("FA_FWD_HEAD_GROUP");
  const int from_env = e ? atoi(e) : 0;
  const double kv_bytes = 4.0 * bh * (double)nk * d;  // K and V, 16-bit
  const int g = from_env > 0 ? from_env : (kv_bytes > 64.0 * (1 << 20) ? 8 : bh);
  return g < bh ? g : bh;
}

// Makes the device that owns `ptr` current on the calling thread, which also
// gives a thread that has not used CUDA yet (e.g. an autograd worker) a
// current context for the driver calls that follow.
fa_status bind_device(const void *ptr) {
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, ptr);
  if (e != cudaSuccess) return cuda_fail("cudaPointerGetAttributes", e);
  if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) {
    snprintf(g_last_error, sizeof(g_last_error), "tensor at %p is not device memory", ptr);
    return FA_ERR_INVALID_ARG;
  }
  e = cudaSetDevice(a.device);
  return e == cudaSuccess ? FA_OK : cuda_fail("cudaSetDevice", e);
}

constexpr size_t kAlign = 256;
size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Shape checks shared by every entry point; `*empty` is set for a no-op call.
fa_status check_shape(int B, int H, int Nq, int Nk, int d, float scale, bool *empty) {
  *empty = false;
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || d <= 0) return FA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 96 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  if ((long long)B * H * Nq == 0) {
    *empty = true;
    return FA_OK;
  }
  const int n_max = Nq > Nk ? Nq : Nk;
  if (Nk == 0 || n_max > fa::kTile * fa::kMaxTiles) return FA_ERR_UNSUPPORTED;
  if ((long long)B * H * n_max > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

fa::Shape make_shape(int B, int H, int Nq, int Nk, int d, int causal, const uint8_t *mask,
                     bool f16 = false) {
  fa::Shape sh;
  sh.bh = B * H;
  sh.heads = H;
  sh.nq = Nq;
  sh.nk = Nk;
  sh.tq = (Nq + fa::kTile - 1) / fa::kTile;
  sh.tk = (Nk + fa::kTile - 1) / fa::kTile;
  sh.d = d;
  sh.causal = causal ? 1 : 0;
  sh.causal_off = Nk - Nq;
  sh.f16 = f16 ? 1 : 0;
  sh.mask = mask;
  return sh;
}

// The inputs' element type: Q decides (bf16 or f16) and every other 16-bit
// operand must match it; O may also be fp32 where `f32_ok`.
fa_status check_dtype(const fa_tensor *t, int elem, bool f32_ok, const char *name) {
  if (t->dtype == elem || (f32_ok && t->dtype == FA_F32)) return FA_OK;
  snprintf(g_last_error, sizeof(g_last_error), "%s: dtype %d unsupported with Q of dtype %d",
           name, (int)t->dtype, elem);
  return FA_ERR_UNSUPPORTED;
}

fa_status input_dtype(const fa_tensor *Q, int *elem) {
  if (Q->dtype != FA_BF16 && Q->dtype != FA_F16) {
    snprintf(g_last_error, sizeof(g_last_error), "Q: dtype %d unsupported (bf16 or f16)",
             (int)Q->dtype);
    return FA_ERR_UNSUPPORTED;
  }
  *elem = Q->dtype;
  return FA_OK;
}

// Columns per row the split-forward workspace reserves: 128 for a head
// dimension of 96 (the kernels use the first 96).
int padded_d(int d) { return d == 96 ? 128 : d; }

// Bytes of one part of the split-forward workspace (256-byte aligned parts).
size_t split_o_bytes(int B, int H, int Nq, int d, int ns) {
  return round_up((size_t)ns * B * H * Nq * padded_d(d) * sizeof(float));
}
size_t split_lse_bytes(int B, int H, int Nq, int ns) {
  return round_up((size_t)ns * B * H * Nq * sizeof(float));
}

constexpr int kMaxSplits = 128;

// SM count of the calling thread's current device, looked up once per device
// (0 if unknown).
int sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < 64) cache[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

fa_status forward_impl(const fa_tensor *Q, const fa_tensor *K, const fa_tensor *V,
                       const fa_tensor *O, float *LSE, int B, int H, int Nq, int Nk, int d,
                       int causal, float scale, const uint8_t *block_mask, int n_split,
                       void *workspace, size_t ws_bytes, void *stream) {
  bool empty;
  fa_status s = check_shape(B, H, Nq, Nk, d, scale, &empty);
  if (s != FA_OK || empty) return s;
  if (!Q || !K || !V || !O || !LSE) return FA_ERR_INVALID_ARG;
  if (n_split < 1) return FA_ERR_INVALID_ARG;
  if (n_split > kMaxSplits) return FA_ERR_UNSUPPORTED;
  if (n_split > 1) {
    if (!workspace) return FA_ERR_INVALID_ARG;
    if (ws_bytes < split_o_bytes(B, H, Nq, d, n_split) + split_lse_bytes(B, H, Nq, n_split))
      return FA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return FA_ERR_MISALIGNED;
  }
  fa::FwdParams p;
  memset(&p, 0, sizeof(p));
  fa::RowStrides sq, sk, sv;
  const int o_bytes = O->dtype == FA_F32 ? 4 : 2;
  int elem = FA_BF16;
  if ((s = input_dtype(Q, &elem)) != FA_OK || (s = check_dtype(K, elem, false, "K")) != FA_OK ||
      (s = check_dtype(V, elem, false, "V")) != FA_OK ||
      (s = check_dtype(O, elem, true, "O")) != FA_OK ||
      (s = operand_strides(Q, B, H, Nq, d, 2, "Q", &sq)) != FA_OK ||
      (s = operand_strides(K, B, H, Nk, d, 2, "K", &sk)) != FA_OK ||
      (s = operand_strides(V, B, H, Nk, d, 2, "V", &sv)) != FA_OK ||
      (s = operand_strides(O, B, H, Nq, d, o_bytes, "O", &p.so)) != FA_OK)
    return s;
  if (!aligned16(LSE)) return FA_ERR_MISALIGNED;
  if ((s = bind_device(Q->data)) != FA_OK) return s;
  const bool f16 = elem == FA_F16;
  if (!encode_operand(&p.tm_q, Q->data, sq, B, H, Nq, d, f16) ||
      !encode_operand(&p.tm_k, K->data, sk, B, H, Nk, d, f16) ||
      !encode_operand(&p.tm_v, V->data, sv, B, H, Nk, d, f16))
    return FA_ERR_CUDA;
  // O is stored by TMA, one 32-row box per warp
  if (O->dtype != FA_F32 && !encode_operand(&p.tm_o, O->data, p.so, B, H, Nq, d, f16, 32))
    return FA_ERR_CUDA;
  p.sh = make_shape(B, H, Nq, Nk, d, causal, block_mask, f16);
  p.o = O->data;
  p.lse = LSE;
  p.o_f32 = O->dtype == FA_F32 ? 1 : 0;
  p.n_split = n_split;
  if (n_split > 1) {
    p.o_part = static_cast<float *>(workspace);
    p.lse_part = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                           split_o_bytes(B, H, Nq, d, n_split));
  }
  p.scale_log2 = scale * 1.4426950408889634f;  // log2(e)
  p.head_group = forward_head_group(p.sh.bh, Nk, d);
  p.sms = sm_count();
  {
    // FA_FWD_Q_TILES=1 or 2 fixes the Q tiles per CTA of the d = 64 forward
    // (tuning and tests); otherwise the launch chooses
    const char *e = getenv("FA_FWD_Q_TILES");
    const int q = e ? atoi(e) : 0;
    p.q_tiles = (q == 1 || q == 2) ? q : 0;
  }
  p.debug_flags = g_debug_flags.load();
  p.wait_limit_ns = g_wait_limit_ns.load() ? g_wait_limit_ns.load() : fa::kWaitLimitNs;
  cudaError_t e = status_word(&p.status);
  if (e != cudaSuccess) return cuda_fail("cudaGetSymbolAddress", e);
  NvtxRange range(n_split > 1 ? "fa_forward (split)" : "fa_forward");
  e = fa::launch_forward(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail("forward launch", e);
}

// Backward workspace: fp32 D and LSE * log2(e) per padded query row (both
// forms), then, for the one-pass backward (head dimensions up to 128), the fp32
// dQ accumulator of d floats per padded query row.
size_t stats_workspace_bytes(int B, int H, int Nq) {
  const size_t rows = (size_t)B * H * (size_t)((Nq + fa::kTile - 1) / fa::kTile) * fa::kTile;
  return 2 * round_up(rows * sizeof(float));
}

size_t dq_acc_bytes(int B, int H, int Nq, int d) {
  if (d > 128) return 0;
  const size_t rows = (size_t)B * H * (size_t)((Nq + fa::kTile - 1) / fa::kTile) * fa::kTile;
  return round_up(rows * (size_t)d * sizeof(float));
}

// The default form by head dimension, from interleaved A/B timings of both
// forms on GB300: the one-pass kernels are 18-25 % faster at d = 64, 3-4 % at
// d = 96 and 1-7.5 % at d = 128 (64-query steps); d = 256 has the two-kernel
// form only.
bool one_pass_by_default(int d) { return d <= 128; }

// Whether a backward with this much workspace runs the one-pass kernel: the
// workspace holds the dQ accumulator too, and FA_BWD_ALGO=split (a tuning and
// A/B switch) does not ask for the two-kernel form.
bool use_one_pass(int B, int H, int Nq, int d, size_t ws_bytes) {
  if (d > 128) return false;
  // the accumulator's rows are addressed with 32-bit TMA coordinates
  if ((long long)B * H * ((Nq + fa::kTile - 1) / fa::kTile) * fa::kTile > 0x7fffffffLL)
    return false;
  const char *e = getenv("FA_BWD_ALGO");
  if (e && strcmp(e, "split") == 0) return false;
  return ws_bytes >= stats_workspace_bytes(B, H, Nq) + dq_acc_bytes(B, H, Nq, d);
}

fa_status backward_impl(const fa_tensor *Q, const fa_tensor *K, const fa_tensor *V,
                        const fa_tensor *O, const fa_tensor *dO, const float *LSE,
                        const fa_tensor *dQ, const fa_tensor *dK, const fa_tensor *dV, int B,
                        int H, int Nq, int Nk, int d, int causal, float scale,
                        const uint8_t *block_mask, void *workspace, size_t ws_bytes,
                        void *stream) {
  bool empty;
  fa_status s = check_shape(B, H, Nq, Nk, d, scale, &empty);
  if (s != FA_OK || empty) return s;
  if (!Q || !K || !V || !O || !dO || !LSE || !dQ || !dK || !dV || !workspace)
    return FA_ERR_INVALID_ARG;
  if (ws_bytes < stats_workspace_bytes(B, H, Nq)) return FA_ERR_INVALID_ARG;
  fa::BwdParams p;
  memset(&p, 0, sizeof(p));
  fa::RowStrides sq, sk, sv;
  const fa_tensor *all[8] = {Q, K, V, O, dO, dQ, dK, dV};
  const char *names[8] = {"Q", "K", "V", "O", "dO", "dQ", "dK", "dV"};
  int elem = FA_BF16;
  if ((s = input_dtype(Q, &elem)) != FA_OK) return s;
  for (int k = 1; k < 8; ++k)
    if ((s = check_dtype(all[k], elem, false, names[k])) != FA_OK) return s;
  if ((s = operand_strides(Q, B, H, Nq, d, 2, "Q", &sq)) != FA_OK ||
      (s = operand_strides(K, B, H, Nk, d, 2, "K", &sk)) != FA_OK ||
      (s = operand_strides(V, B, H, Nk, d, 2, "V", &sv)) != FA_OK ||
      (s = operand_strides(O, B, H, Nq, d, 2, "O", &p.so)) != FA_OK ||
      (s = operand_strides(dO, B, H, Nq, d, 2, "dO", &p.sdo)) != FA_OK ||
      (s = operand_strides(dQ, B, H, Nq, d, 2, "dQ", &p.sdq)) != FA_OK ||
      (s = operand_strides(dK, B, H, Nk, d, 2, "dK", &p.sdk)) != FA_OK ||
      (s = operand_strides(dV, B, H, Nk, d, 2, "dV", &p.sdv)) != FA_OK)
    return s;
  if (!aligned16(LSE) || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
    return FA_ERR_MISALIGNED;
  if ((s = bind_device(Q->data)) != FA_OK) return s;
  const bool f16 = elem == FA_F16;
  if (!encode_operand(&p.tm_q, Q->data, sq, B, H, Nq, d, f16) ||
      !encode_operand(&p.tm_k, K->data, sk, B, H, Nk, d, f16) ||
      !encode_operand(&p.tm_v, V->data, sv, B, H, Nk, d, f16) ||
      !encode_operand(&p.tm_do, dO->data, p.sdo, B, H, Nq, d, f16) ||
      !encode_operand(&p.tm_dq, dQ->data, p.sdq, B, H, Nq, d, f16, 32) ||
      !encode_operand(&p.tm_dk, dK->data, p.sdk, B, H, Nk, d, f16, 32) ||
      !encode_operand(&p.tm_dv, dV->data, p.sdv, B, H, Nk, d, f16, 32))
    return FA_ERR_CUDA;
  p.sh = make_shape(B, H, Nq, Nk, d, causal, block_mask, f16);
  p.o = O->data;
  p.dout = dO->data;
  p.lse = LSE;
  const size_t stat_bytes = stats_workspace_bytes(B, H, Nq) / 2;
  p.delta = static_cast<float *>(workspace);
  p.lse2 = reinterpret_cast<float *>(static_cast<char *>(workspace) + stat_bytes);
  p.dq_acc = use_one_pass(B, H, Nq, d, ws_bytes)
                 ? reinterpret_cast<float *>(static_cast<char *>(workspace) + 2 * stat_bytes)
                 : nullptr;
  if (p.dq_acc && d == 128 &&
      (!encode_dq_acc(&p.tm_dqacc, p.dq_acc, (long long)B * H * p.sh.tq * fa::kTile, d) ||
       !encode_operand(&p.tm_qh, Q->data, sq, B, H, Nq, d, f16, 64) ||
       !encode_operand(&p.tm_doh, dO->data, p.sdo, B, H, Nq, d, f16, 64)))
    return FA_ERR_CUDA;
  p.dq = dQ->data;
  p.dk = dK->data;
  p.dv = dV->data;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.head_group = backward_head_group(p.sh.bh, p.sh.tk);
  p.debug_flags = g_debug_flags.load();
  p.wait_limit_ns = g_wait_limit_ns.load() ? g_wait_limit_ns.load() : fa::kWaitLimitNs;
  cudaError_t e = status_word(&p.status);
  if (e != cudaSuccess) return cuda_fail("cudaGetSymbolAddress", e);
  NvtxRange range("fa_backward");
  e = fa::launch_backward(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail("backward launch", e);
}

// Descriptor of a contiguous [B][H][N][d] tensor.
fa_tensor contiguous(const void *data, int H, int N, int d, int dtype) {
  fa_tensor t;
  t.data = const_cast<void *>(data);
  t.stride_n = d;
  t.stride_h = (int64_t)N * d;
  t.stride_b = (int64_t)H * N * d;
  t.dtype = dtype;
  t.reserved = 0;
  return t;
}

// ---- measurement hooks ------------------------------------------------------

struct ProbeRecord {
  int kind;
  cudaEvent_t start, stop;
};

std::atomic<bool> g_prof_on{false};
std::mutex g_prof_mu;
std::vector<ProbeRecord> g_prof_records;
std::vector<cudaEvent_t> g_prof_pool;

cudaEvent_t pooled_event() {
  if (!g_prof_pool.empty()) {
    cudaEvent_t e = g_prof_pool.back();
    g_prof_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// ---- fixed scratch for fa_backward_noalloc ----------------------------------

// The backward workspace of fa_backward_noalloc: a fixed area in the module's
// global memory, so that call needs no allocation. Every device that loads
// the library reserves it until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the calling thread's current device.
// In host code the symbol's name is only a host-side handle; its device
// address has to be asked for. It is looked up at every call, like the status
// word's, so that it stays right after a cudaDeviceReset reloads the module.
fa_status noalloc_scratch(void **out) {
  void *ptr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (e != cudaSuccess) return cuda_fail("cudaGetSymbolAddress(noalloc scratch)", e);
  *out = ptr;
  return FA_OK;
}

// ---- measurement: the SFU exp2 rate ----------------------------------------

constexpr int kExpProbeThreads = 1024;
constexpr int kExpProbeIters = 4096;
constexpr int kExpProbeChains = 8;  // independent ex2 chains per thread
__device__ float g_exp_probe_sink;

// One CTA of 1024 threads per SM, each thread running kExpProbeChains
// independent chains of ex2.approx; the host times the launch with events.
// `key` is a runtime value the sum is compared with, so the compiler cannot
// prove the chains' results unused.
__global__ void __launch_bounds__(kExpProbeThreads, 1) fa_exp2_probe(float key) {
  float a[kExpProbeChains];
#pragma unroll
  for (int c = 0; c < kExpProbeChains; ++c) a[c] = -1e-3f * float(threadIdx.x % 97 + c);
  for (int it = 0; it < kExpProbeIters; ++it) {
#pragma unroll
    for (int c = 0; c < kExpProbeChains; ++c) {
      float y;
      asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(a[c]));
      a[c] = -y;  // stays in [-1, 0): no overflow, and a true dependency
    }
  }
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < kExpProbeChains; ++c) s += a[c];
  if (s == key) g_exp_probe_sink = s;  // keeps the chains alive
}

}  // namespace

namespace fa {

LaunchProbe::LaunchProbe(int kind, cudaStream_t stream) : slot_(-1), stream_(stream) {
  if (!g_prof_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  ProbeRecord r{kind, pooled_event(), pooled_event()};
  if (!r.start || !r.stop) return;
  if (cudaEventRecord(r.start, stream) != cudaSuccess) return;
  slot_ = (int)g_prof_records.size();
  g_prof_records.push_back(r);
}

LaunchProbe::~LaunchProbe() {
  if (slot_ < 0) return;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  cudaEventRecord(g_prof_records[slot_].stop, stream_);
}

}  // namespace fa

extern "C" {

int fa_num_kernels(void) { return fa::kNumKinds; }

const char *fa_kernel_name(int kind) {
  switch (kind) {
    case fa::kKindFwd: return "fa_fwd_kernel";
    case fa::kKindBwdPre: return "fa_bwd_pre";
    case fa::kKindBwdDkdv: return "fa_bwd_dkdv";
    case fa::kKindBwdDq: return "fa_bwd_dq";
    case fa::kKindFwdCombine: return "fa_fwd_combine";
    case fa::kKindBwd256Dv: return "fa_bwd256_dv";
    case fa::kKindBwd256Dk: return "fa_bwd256_dk";
    case fa::kKindBwd256Dq: return "fa_bwd256_dq";
    case fa::kKindBwdFused: return "fa_bwd_fused";
    case fa::kKindBwdConvert: return "fa_bwd_dq_convert";
    default: return "";
  }
}

fa_status fa_profile_enable(int enable) {
  g_prof_on.store(enable != 0);
  return FA_OK;
}

fa_status fa_profile_collect(float *total_ms, int *launches, int n) {
  if ((!total_ms || !launches) && n > 0) return FA_ERR_INVALID_ARG;
  for (int k = 0; k < n; ++k) {
    total_ms[k] = 0.f;
    launches[k] = 0;
  }
  std::lock_guard<std::mutex> lock(g_prof_mu);
  fa_status rc = FA_OK;
  for (const ProbeRecord &r : g_prof_records) {
    float ms = 0.f;
    cudaError_t e = cudaEventSynchronize(r.stop);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.start, r.stop);
    if (e != cudaSuccess) rc = cuda_fail("cudaEventElapsedTime", e);
    if (r.kind >= 0 && r.kind < n) {
      total_ms[r.kind] += ms;
      launches[r.kind] += 1;
    }
    g_prof_pool.push_back(r.start);
    g_prof_pool.push_back(r.stop);
  }
  g_prof_records.clear();
  return rc;
}


int fa_abi_version(void) { return 2; }

const char *fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    default: return "FA_ERR_UNKNOWN";
  }
}

fa_status fa_forward(const void *Q, const void *K, const void *V, void *O, float *LSE, int B,
                     int H, int N, int d, int causal, float scale, const uint8_t *block_mask,
                     void *stream) {
  if (!Q || !K || !V || !O) return (long long)B * H * N == 0 ? FA_OK : FA_ERR_INVALID_ARG;
  const fa_tensor q = contiguous(Q, H, N, d, FA_BF16), k = contiguous(K, H, N, d, FA_BF16),
                  v = contiguous(V, H, N, d, FA_BF16), o = contiguous(O, H, N, d, FA_BF16);
  return forward_impl(&q, &k, &v, &o, LSE, B, H, N, N, d, causal, scale, block_mask, 1, nullptr,
                      0, stream);
}

fa_status fa_forward_f32(const void *Q, const void *K, const void *V, float *O, float *LSE,
                         int B, int H, int N, int d, int causal, float scale,
                         const uint8_t *block_mask, void *stream) {
  if (!Q || !K || !V || !O) return (long long)B * H * N == 0 ? FA_OK : FA_ERR_INVALID_ARG;
  const fa_tensor q = contiguous(Q, H, N, d, FA_BF16), k = contiguous(K, H, N, d, FA_BF16),
                  v = contiguous(V, H, N, d, FA_BF16), o = contiguous(O, H, N, d, FA_F32);
  return forward_impl(&q, &k, &v, &o, LSE, B, H, N, N, d, causal, scale, block_mask, 1, nullptr,
                      0, stream);
}

fa_status fa_forward_ex(const fa_tensor *Q, const fa_tensor *K, const fa_tensor *V,
                        const fa_tensor *O, float *LSE, int B, int H, int Nq, int Nk, int d,
                        int causal, float scale, const uint8_t *block_mask, void *stream) {
  return forward_impl(Q, K, V, O, LSE, B, H, Nq, Nk, d, causal, scale, block_mask, 1, nullptr, 0,
                      stream);
}

int fa_forward_num_splits(int B, int H, int Nq, int Nk, int d, int causal) {
  bool empty;
  if (check_shape(B, H, Nq, Nk, 64, 1.f, &empty) != FA_OK || empty) return 1;
  const int sms = sm_count();
  if (sms <= 0) return 1;
  const fa::Shape sh = make_shape(B, H, Nq, Nk, 64, causal, nullptr);
  // CTAs of the plain forward (one per SM is resident): a pair of Q tiles
  // per CTA, one with head dimension 256
  const long long ctas = (long long)(d == 256 ? sh.tq : (sh.tq + 1) / 2) * sh.bh;
  // K/V tiles the pair with the most work visits
  const int tiles = sh.last_kv_tile(sh.tq - 1) + 1;
  if (ctas >= sms || tiles < 4) return 1;
  long long n = sms / ctas;                 // one wave
  if (n > tiles / 2) n = tiles / 2;         // at least two K/V tiles per split
  if (n > kMaxSplits) n = kMaxSplits;
  return n < 1 ? 1 : (int)n;
}

size_t fa_forward_split_workspace_bytes(int B, int H, int Nq, int d, int num_splits) {
  if (B < 0 || H < 0 || Nq < 0 || d <= 0 || num_splits < 1) return 0;
  if (num_splits == 1) return 0;
  return split_o_bytes(B, H, Nq, d, num_splits) + split_lse_bytes(B, H, Nq, num_splits);
}

fa_status fa_forward_split_ex(const fa_tensor *Q, const fa_tensor *K, const fa_tensor *V,
                              const fa_tensor *O, float *LSE, int B, int H, int Nq, int Nk,
                              int d, int causal, float scale, const uint8_t *block_mask,
                              int num_splits, void *workspace, size_t workspace_bytes,
                              void *stream) {
  return forward_impl(Q, K, V, O, LSE, B, H, Nq, Nk, d, causal, scale, block_mask, num_splits,
                      workspace, workspace_bytes, stream);
}

size_t fa_backward_workspace_bytes(int B, int H, int N, int d) {
  if (B < 0 || H < 0 || N < 0 || d <= 0) return 0;
  return stats_workspace_bytes(B, H, N) + (one_pass_by_default(d) ? dq_acc_bytes(B, H, N, d) : 0);
}

size_t fa_backward_min_workspace_bytes(int B, int H, int N, int d) {
  if (B < 0 || H < 0 || N < 0 || d <= 0) return 0;
  return stats_workspace_bytes(B, H, N);
}

size_t fa_backward_one_pass_workspace_bytes(int B, int H, int N, int d) {
  if (B < 0 || H < 0 || N < 0 || d <= 0 || d > 128) return 0;
  return stats_workspace_bytes(B, H, N) + dq_acc_bytes(B, H, N, d);
}

fa_status fa_backward(const void *Q, const void *K, const void *V, const void *O,
                      const void *dO, const float *LSE, void *dQ, void *dK, void *dV, int B,
                      int H, int N, int d, int causal, float scale, const uint8_t *block_mask,
                      void *workspace, size_t workspace_bytes, void *stream) {
  if (!Q || !K || !V || !O || !dO || !dQ || !dK || !dV)
    return (long long)B * H * N == 0 ? FA_OK : FA_ERR_INVALID_ARG;
  const fa_tensor q = contiguous(Q, H, N, d, FA_BF16), k = contiguous(K, H, N, d, FA_BF16),
                  v = contiguous(V, H, N, d, FA_BF16), o = contiguous(O, H, N, d, FA_BF16),
                  g = contiguous(dO, H, N, d, FA_BF16), gq = contiguous(dQ, H, N, d, FA_BF16),
                  gk = contiguous(dK, H, N, d, FA_BF16), gv = contiguous(dV, H, N, d, FA_BF16);
  return backward_impl(&q, &k, &v, &o, &g, LSE, &gq, &gk, &gv, B, H, N, N, d, causal, scale,
                       block_mask, workspace, workspace_bytes, stream);
}

fa_status fa_backward_ex(const fa_tensor *Q, const fa_tensor *K, const fa_tensor *V,
                         const fa_tensor *O, const fa_tensor *dO, const float *LSE,
                         const fa_tensor *dQ, const fa_tensor *dK, const fa_tensor *dV, int B,
                         int H, int Nq, int Nk, int d, int causal, float scale,
                         const uint8_t *block_mask, void *workspace, size_t workspace_bytes,
                         void *stream) {
  return backward_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Nq, Nk, d, causal, scale,
                       block_mask, workspace, workspace_bytes, stream);
}

fa_status fa_device_status(void *stream, unsigned int *code) {
  if (!code) return FA_ERR_INVALID_ARG;
  *code = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail("cudaStreamSynchronize", e);
  unsigned int w = 0, zero = 0;
  e = cudaMemcpyFromSymbol(&w, g_status_word, sizeof(w));
  if (e != cudaSuccess) return cuda_fail("cudaMemcpyFromSymbol", e);
  if (w && (e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero))) != cudaSuccess)
    return cuda_fail("cudaMemcpyToSymbol", e);
  *code = w;
  return w ? FA_ERR_TIMEOUT : FA_OK;
}

const char *fa_last_error(void) { return g_last_error; }

fa_status fa_debug_configure(unsigned int flags, unsigned long long wait_limit_ns) {
  if (flags & ~fa::kDebugSkipLoads) return FA_ERR_INVALID_ARG;
  g_debug_flags.store(flags);
  g_wait_limit_ns.store(wait_limit_ns);
  return FA_OK;
}

size_t fa_backward_noalloc_max_bytes(void) { return kNoAllocScratchBytes; }

fa_status fa_measure_exp2_rate(double *exps_per_second) {
  if (!exps_per_second) return FA_ERR_INVALID_ARG;
  *exps_per_second = 0.0;
  const int sms = sm_count();
  if (sms <= 0) return cuda_fail("SM count", cudaErrorInvalidDevice);
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  cudaError_t e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  float ms = 0.f;
  for (int rep = 0; rep < 2 && e == cudaSuccess; ++rep) {  // the first launch warms up
    e = cudaEventRecord(e0, 0);
    if (e == cudaSuccess) {
      fa_exp2_probe<<<sms, kExpProbeThreads, 0, 0>>>(1.0e30f);
      e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaEventRecord(e1, 0);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (e != cudaSuccess) return cuda_fail("exp2 probe", e);
  if (!(ms > 0.f)) return cuda_fail("exp2 probe time", cudaErrorUnknown);
  *exps_per_second =
      (double)sms * kExpProbeThreads * kExpProbeIters * kExpProbeChains / (ms * 1e-3);
  return FA_OK;
}

fa_status fa_backward_noalloc(const void *Q, const void *K, const void *V, const void *O,
                              const void *dO, const float *LSE, void *dQ, void *dK, void *dV,
                              int B, int H, int N, int d, int causal, float scale,
                              const uint8_t *block_mask, void *stream) {
  bool empty;
  fa_status s = check_shape(B, H, N, N, d, scale, &empty);
  if (s != FA_OK || empty) return s;
  if (!Q || !K || !V || !O || !dO || !LSE || !dQ || !dK || !dV) return FA_ERR_INVALID_ARG;
  // the one-pass backward when its accumulator fits in the area, else the
  // two-kernel backward, which needs only the row statistics
  size_t need = fa_backward_workspace_bytes(B, H, N, d);
  if (need > kNoAllocScratchBytes) need = fa_backward_min_workspace_bytes(B, H, N, d);
  if (need > kNoAllocScratchBytes) {
    snprintf(g_last_error, sizeof(g_last_error),
             "fa_backward_noalloc: B=%d H=%d N=%d d=%d needs %zu bytes of scratch; the fixed "
             "area holds %zu",
             B, H, N, d, need, kNoAllocScratchBytes);
    return FA_ERR_UNSUPPORTED;
  }
  if ((s = bind_device(Q)) != FA_OK) return s;
  void *scratch = nullptr;
  if ((s = noalloc_scratch(&scratch)) != FA_OK) return s;
  return fa_backward(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, causal, scale, block_mask,
                     scratch, need, stream);
}

}  // extern "C"
