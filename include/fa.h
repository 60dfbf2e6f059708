/*
 * fa.h: C ABI of the exact IO-aware attention library for NVIDIA GB300
 * (sm_103a).
 *
 * The library computes exact scaled dot-product attention
 *
 *     O = softmax(scale * Q K^T) V            per batch b and head h,
 *
 * as defined in "Paper Notes: FlashAttention" (bv003me.vercel.app), section
 * "What Are We Computing?", with the 1/sqrt(d) score scale of the numpy
 * attention_naive in "flash attention" (muhibwaqar.com), section "build it
 * from scratch" (here an explicit argument). The forward pass is one fused
 * tiled kernel with online softmax (same page, section "Tiling: Block-by-Block
 * Softmax"; aicassindra page "FlashAttention", section "Rescale and
 * accumulate") that writes only O and the per-row log-sum-exp; the backward
 * pass recomputes the score tiles from Q, K and the log-sum-exp (aicassindra
 * page, section "The backward pass: recompute instead of store").
 *
 * Conventions shared by every entry point
 *  - Tensors are contiguous row-major [B][H][N][d]; Q, K, V, O, dO, dQ, dK, dV
 *    hold bf16 values (raw 16-bit storage, passed as void*); LSE is fp32
 *    [B][H][N], the natural-log log-sum-exp of the scaled scores of each row.
 *  - All tensor pointers are DEVICE pointers, 16-byte aligned, owned by the
 *    caller. The library never allocates, frees or synchronises; all work is
 *    enqueued on `stream` (a cudaStream_t passed as void*; NULL = the legacy
 *    default stream), which must belong to the device that holds Q. Each call
 *    makes that device current on the calling thread. Inputs are only read.
 *  - Supported: d in {64, 128}; N a positive multiple of 128; B, H >= 1;
 *    B*H*N <= 2^31 - 1; scale finite and > 0. B*H*N == 0 is a no-op that
 *    returns FA_OK.
 *  - causal != 0: query i sees key j iff j <= i (0-based, equal lengths).
 *  - block_mask: NULL for dense attention, else a DEVICE uint8 array
 *    [T][T], T = N/128, shared by every (b, h); tile (i/128, j/128) is kept
 *    iff its byte is non-zero. With causal also set, both must allow a key.
 *    The pages name a block-sparse variant only ("Paper Notes:
 *    FlashAttention", section "Experiments & Results"); this tile semantics
 *    is this library's reading. A query row that sees no key gets O = 0 and
 *    LSE = -inf.
 *  - Host-detectable errors return at once, before anything is enqueued. A
 *    failed launch returns FA_ERR_CUDA. Kernel-side bounded waits that give up
 *    record FA_ERR_TIMEOUT in a device status word that fa_device_status()
 *    reads.
 */
#ifndef FA_H
#define FA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad scale, host memory */
  FA_ERR_UNSUPPORTED = 2, /* valid but outside the supported set (d, N) */
  FA_ERR_MISALIGNED = 3,  /* a tensor pointer is not 16-byte aligned */
  FA_ERR_CUDA = 4,        /* a CUDA runtime/driver call or launch failed */
  FA_ERR_TIMEOUT = 5      /* a kernel-side wait gave up (device status word) */
} fa_status;

/* Version of this ABI; bumped on any incompatible change. */
int fa_abi_version(void);

/* Human-readable name of a status code (static storage, never NULL). */
const char *fa_status_string(int status);

/*
 * Description of the last failure reported to the calling thread: for
 * FA_ERR_CUDA the failing CUDA call and its error text, for a size that
 * fa_backward_noalloc cannot hold the bytes needed and available ("" if
 * none). Thread-local storage, valid until the thread's next failing call;
 * never NULL.
 */
const char *fa_last_error(void);

/*
 * Forward pass. Reads Q, K, V; writes O (bf16 [B,H,N,d]) and LSE
 * (fp32 [B,H,N]). S and P never reach global memory.
 */
fa_status fa_forward(const void *Q, const void *K, const void *V, void *O, float *LSE, int B,
                     int H, int N, int d, int causal, float scale, const uint8_t *block_mask,
                     void *stream);

/*
 * Forward pass with an fp32 O store: the same kernel and arithmetic as
 * fa_forward, but O is written as fp32 [B,H,N,d] before any bf16 rounding.
 * It exists so that accuracy can be checked without the output rounding.
 */
fa_status fa_forward_f32(const void *Q, const void *K, const void *V, float *O, float *LSE,
                         int B, int H, int N, int d, int causal, float scale,
                         const uint8_t *block_mask, void *stream);

/*
 * Bytes of device workspace fa_backward needs: fp32 D [B,H,N] (D_i = dO_i.O_i)
 * and fp32 LSE*log2(e) [B,H,N], each starting on a 256-byte boundary: O(N),
 * 8 bytes per query row. Returns 0 for invalid sizes.
 */
size_t fa_backward_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward pass. Reads Q, K, V, O, dO (bf16) and LSE (fp32, as written by the
 * forward pass with the same arguments); writes dQ, dK, dV (bf16 [B,H,N,d]).
 * `workspace` is a caller-owned device buffer of at least
 * fa_backward_workspace_bytes(B,H,N,d) bytes, 256-byte aligned; its contents
 * on entry do not matter and are clobbered. The score and probability tiles
 * are recomputed on chip and never reach global memory.
 */
fa_status fa_backward(const void *Q, const void *K, const void *V, const void *O,
                      const void *dO, const float *LSE, void *dQ, void *dK, void *dV, int B,
                      int H, int N, int d, int causal, float scale, const uint8_t *block_mask,
                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * Backward pass without a caller-supplied workspace. The pages have no
 * counterpart: this entry point exists for callers of this library that
 * cannot allocate device memory where they run the backward pass, e.g. a
 * plug-in inside a host application that owns all device memory and gives
 * plug-ins no allocator, or a runtime whose rules forbid allocating once it
 * has started. Such a caller cannot provide fa_backward's workspace, so this
 * call uses a scratch area of fixed size built into the library instead.
 *
 * Arguments, layouts, results and errors are those of fa_backward, minus
 * the workspace. The scratch is a global-memory area of
 * fa_backward_noalloc_max_bytes() bytes (64 MiB) that every device which
 * loads the library reserves until the process exits. A call whose
 * fa_backward_workspace_bytes(B,H,N,d) exceeds it returns FA_ERR_UNSUPPORTED
 * before doing anything, and fa_last_error() states both sizes. The call
 * allocates no memory (no cudaMalloc, no cudaFree, no allocating library
 * routine) as long as the measurement hooks are off, which is the default.
 *
 * The first call on a device looks up the scratch area's device address on
 * that device; make that first call before any stream capture. All calls on
 * a device share the one area, and it keeps the last call's contents (each
 * call re-initialises what must start at zero itself). Calls that overlap
 * on the GPU, e.g. on two streams at once, race on the area: serialise them.
 */
fa_status fa_backward_noalloc(const void *Q, const void *K, const void *V, const void *O,
                              const void *dO, const float *LSE, void *dQ, void *dK, void *dV,
                              int B, int H, int N, int d, int causal, float scale,
                              const uint8_t *block_mask, void *stream);

/* Size in bytes of fa_backward_noalloc's fixed scratch area. */
size_t fa_backward_noalloc_max_bytes(void);

/*
 * Debug/status query: synchronises `stream`, reads the device status word
 * that kernel-side bounded waits set when they give up, clears it, and
 * stores it in *code (0 = no failure; otherwise an encoded kernel/role/wait
 * site). Returns FA_ERR_TIMEOUT if a wait gave up, FA_ERR_CUDA if the stream
 * reports an error, else FA_OK.
 */
fa_status fa_device_status(void *stream, unsigned int *code);

/*
 * Failure-path testing (process-wide; not for production use).
 * flags = FA_DEBUG_SKIP_LOADS makes every kernel's TMA producer issue no
 * copy, so the kernel's bounded waits run out: each CTA records
 * 0x80000000 | kernel << 16 | role << 8 | site in the status word that
 * fa_device_status() reads, frees its tensor memory and exits, and the CUDA
 * context stays usable. wait_limit_ns sets the limit of one wait (0 restores
 * the default of 2 s). fa_debug_configure(0, 0) restores normal operation.
 * Returns FA_ERR_INVALID_ARG for unknown flag bits.
 */
#define FA_DEBUG_SKIP_LOADS 1u
fa_status fa_debug_configure(unsigned int flags, unsigned long long wait_limit_ns);

/*
 * Measurement hooks. Kernels are numbered 0 .. fa_num_kernels()-1:
 * 0 forward, 1 backward preprocess (D_i, LSE*log2 e, zeroed dQ accumulator),
 * 2 backward main, 3 backward dQ conversion; fa_kernel_name() names them
 * ("" for an unknown id).
 *
 * fa_profile_enable(1): from then on every kernel launch is bracketed by two
 * CUDA events recorded on its stream (no synchronisation, no device memory).
 * fa_profile_enable(0) stops recording. Thread-safe.
 *
 * fa_profile_collect: waits for the recorded events, writes the summed
 * event-timed duration (ms) and the launch count of kernel k into
 * total_ms[k] and launches[k] for k < n, and forgets the records. Returns
 * FA_ERR_CUDA if an event could not be read (fa_last_error() says which).
 */
int fa_num_kernels(void);
const char *fa_kernel_name(int kernel);
fa_status fa_profile_enable(int enable);
fa_status fa_profile_collect(float *total_ms, int *launches, int n);

#ifdef __cplusplus
}
#endif

#endif /* FA_H */
