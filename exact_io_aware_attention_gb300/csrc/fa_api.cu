// C-ABI layer: argument validation, TMA tensor-map encoding and kernel launch.
// The declarations and the contract of every entry point are in include/fa.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

// Device status word written by kernel-side bounded waits that give up.
__device__ unsigned int g_status_word = 0u;

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

unsigned int *status_word() {
  // per device: the symbol address is looked up on the current device each call
  void *ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_status_word) != cudaSuccess) return nullptr;
  return static_cast<unsigned int *>(ptr);
}

// 2-D bf16 map over [rows][d]: box = 64 columns (128 bytes) x 128 rows, 128-byte swizzle.
bool encode_rows(CUtensorMap *m, const void *base, long long rows, int d) {
  EncodeTiledFn enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)fa::kTile};
  const cuuint32_t elem[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
             elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr size_t kAlign = 256;
size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Shape checks shared by every entry point; `*empty` is set for a no-op call.
fa_status check_shape(int B, int H, int N, int d, float scale, bool *empty) {
  *empty = false;
  if (B < 0 || H < 0 || N < 0 || d <= 0) return FA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if ((long long)B * H * N == 0) {
    *empty = true;
    return FA_OK;
  }
  if (N % fa::kTile != 0 || N / fa::kTile > fa::kMaxTiles) return FA_ERR_UNSUPPORTED;
  if ((long long)B * H * N > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

fa_status forward_impl(const void *Q, const void *K, const void *V, void *O, float *LSE, int B,
                       int H, int N, int d, int causal, float scale, const uint8_t *block_mask,
                       void *stream, int o_f32) {
  bool empty;
  fa_status s = check_shape(B, H, N, d, scale, &empty);
  if (s != FA_OK || empty) return s;
  if (!Q || !K || !V || !O || !LSE) return FA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(LSE))
    return FA_ERR_MISALIGNED;
  fa::FwdParams p;
  memset(&p, 0, sizeof(p));
  const long long rows = (long long)B * H * N;
  if (!encode_rows(&p.tm_q, Q, rows, d) || !encode_rows(&p.tm_k, K, rows, d) ||
      !encode_rows(&p.tm_v, V, rows, d))
    return FA_ERR_CUDA;
  p.o = O;
  p.lse = LSE;
  p.mask = block_mask;
  p.bh = B * H;
  p.n = N;
  p.d = d;
  p.causal = causal ? 1 : 0;
  p.o_f32 = o_f32;
  p.scale_log2 = scale * 1.4426950408889634f;  // log2(e)
  p.status = status_word();
  if (!p.status) return FA_ERR_CUDA;
  return fa::launch_forward(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK
                                                                                 : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

int fa_abi_version(void) { return 1; }

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
  return forward_impl(Q, K, V, O, LSE, B, H, N, d, causal, scale, block_mask, stream, 0);
}

fa_status fa_forward_f32(const void *Q, const void *K, const void *V, float *O, float *LSE,
                         int B, int H, int N, int d, int causal, float scale,
                         const uint8_t *block_mask, void *stream) {
  return forward_impl(Q, K, V, O, LSE, B, H, N, d, causal, scale, block_mask, stream, 1);
}

size_t fa_backward_workspace_bytes(int B, int H, int N, int d) {
  if (B < 0 || H < 0 || N < 0 || d <= 0) return 0;
  const size_t rows = (size_t)B * H * N;
  return round_up(rows * sizeof(float)) + round_up(rows * (size_t)d * sizeof(float));
}

fa_status fa_backward(const void *Q, const void *K, const void *V, const void *O,
                      const void *dO, const float *LSE, void *dQ, void *dK, void *dV, int B,
                      int H, int N, int d, int causal, float scale, const uint8_t *block_mask,
                      void *workspace, size_t workspace_bytes, void *stream) {
  bool empty;
  fa_status s = check_shape(B, H, N, d, scale, &empty);
  if (s != FA_OK || empty) return s;
  if (!Q || !K || !V || !O || !dO || !LSE || !dQ || !dK || !dV || !workspace)
    return FA_ERR_INVALID_ARG;
  if (workspace_bytes < fa_backward_workspace_bytes(B, H, N, d)) return FA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(dO) ||
      !aligned16(LSE) || !aligned16(dQ) || !aligned16(dK) || !aligned16(dV) ||
      (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
    return FA_ERR_MISALIGNED;
  fa::BwdParams p;
  memset(&p, 0, sizeof(p));
  const long long rows = (long long)B * H * N;
  if (!encode_rows(&p.tm_q, Q, rows, d) || !encode_rows(&p.tm_k, K, rows, d) ||
      !encode_rows(&p.tm_v, V, rows, d) || !encode_rows(&p.tm_do, dO, rows, d))
    return FA_ERR_CUDA;
  p.o = O;
  p.dout = dO;
  p.lse = LSE;
  p.delta = static_cast<float *>(workspace);
  p.dq_acc = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                       round_up((size_t)rows * sizeof(float)));
  p.dq = dQ;
  p.dk = dK;
  p.dv = dV;
  p.mask = block_mask;
  p.bh = B * H;
  p.n = N;
  p.d = d;
  p.causal = causal ? 1 : 0;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = status_word();
  if (!p.status) return FA_ERR_CUDA;
  return fa::launch_backward(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK
                                                                                  : FA_ERR_CUDA;
}

fa_status fa_device_status(void *stream, unsigned int *code) {
  if (!code) return FA_ERR_INVALID_ARG;
  *code = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return FA_ERR_CUDA;
  unsigned int w = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&w, g_status_word, sizeof(w)) != cudaSuccess) return FA_ERR_CUDA;
  if (w && cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess)
    return FA_ERR_CUDA;
  *code = w;
  return w ? FA_ERR_TIMEOUT : FA_OK;
}

}  // extern "C"
