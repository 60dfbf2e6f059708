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
 *  - Each batch b and head h has Nq query rows (Q, O, dO, dQ: [Nq][d]) and
 *    Nk key rows (K, V, dK, dV: [Nk][d]). The plain entry points take
 *    contiguous row-major [B][H][N][d] tensors with Nq = Nk = N; the _ex entry
 *    points take an fa_tensor descriptor per operand (any strides over b, h
 *    and the row, e.g. the [B][N][H][d] layout) and separate Nq and Nk.
 *    Q, K, V, dO, dQ, dK, dV hold 16-bit values of one type: bf16 (the plain
 *    entry points; FA_BF16) or f16 (FA_F16, _ex entry points only). O has
 *    that type too, or fp32 (fa_forward_f32 or an FA_F32 descriptor). The
 *    tensor cores multiply in that 16-bit type (P and dS are rounded to it)
 *    and accumulate in fp32. LSE is fp32 contiguous [B][H][Nq], the
 *    natural-log log-sum-exp of the scaled scores of each query row.
 *  - All tensor pointers are DEVICE pointers, 16-byte aligned, owned by the
 *    caller. The library never allocates, frees or synchronises; all work is
 *    enqueued on `stream` (a cudaStream_t passed as void*; NULL = the legacy
 *    default stream), which must belong to the device that holds Q. Each call
 *    makes that device current on the calling thread and leaves it current
 *    on return (the caller's previous current device is not restored; a
 *    caller that drives several devices from one thread sets its own device
 *    again after the call). Inputs are only read;
 *    outputs must not overlap one another or an input.
 *  - Supported: d in {64, 96, 128, 256}; 1 <= Nq, Nk <= 65536 (any length: a last,
 *    partial tile of 128 rows is handled inside the kernels); B, H >= 1;
 *    B*H*max(Nq, Nk) <= 2^31 - 1; scale finite and > 0. B*H*Nq == 0 is a
 *    no-op that returns FA_OK; Nk == 0 with Nq > 0 is FA_ERR_UNSUPPORTED.
 *  - causal != 0: query i sees key j iff j <= i + Nk - Nq (0-based): with
 *    Nq = Nk this is the pages' j <= i; with Nq != Nk the last query is
 *    aligned with the last key, so the queries are the last Nq positions of a
 *    sequence of Nk keys (this library's reading; the pages treat one
 *    sequence only). Queries with i < Nq - Nk see no key.
 *  - block_mask: NULL for dense attention, else a DEVICE uint8 array
 *    [Tq][Tk], Tq = ceil(Nq/128), Tk = ceil(Nk/128), shared by every (b, h);
 *    tile (i/128, j/128) is kept iff its byte is non-zero. With causal also
 *    set, both must allow a key. The pages name a block-sparse variant only
 *    ("Paper Notes: FlashAttention", section "Experiments & Results"); this
 *    tile semantics is this library's reading. A query row that sees no key
 *    gets O = 0 and LSE = -inf, and its rows of dQ are 0.
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

/* Element types of an fa_tensor. */
typedef enum fa_dtype {
  FA_BF16 = 0, /* bfloat16, raw 16-bit storage */
  FA_F32 = 1,  /* IEEE fp32 (accepted for O only) */
  FA_F16 = 2   /* IEEE binary16, raw 16-bit storage */
} fa_dtype;

/*
 * One operand of logical shape [B][H][rows][d]: element (b, h, n, c) is at
 * data + b*stride_b + h*stride_h + n*stride_n + c (strides in ELEMENTS; the
 * d elements of a row are contiguous). `data` is a device pointer, 16-byte
 * aligned. Every stride of a dimension longer than 1 must be positive, a
 * multiple of 16 bytes (8 bf16 or 4 fp32 elements) and below 2^40 bytes;
 * strides of dimensions of length 1 are ignored. `reserved` must be 0.
 */
typedef struct fa_tensor {
  void *data;
  int64_t stride_b;
  int64_t stride_h;
  int64_t stride_n;
  int32_t dtype; /* fa_dtype */
  int32_t reserved;
} fa_tensor;

typedef enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad scale, host memory */
  FA_ERR_UNSUPPORTED = 2, /* valid but outside the supported set (d, N, dtype, stride) */
  FA_ERR_MISALIGNED = 3,  /* a pointer or a stride is not a multiple of 16 bytes */
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
 * Forward pass, contiguous [B,H,N,d] tensors, Nq = Nk = N. Reads Q, K, V;
 * writes O (bf16 [B,H,N,d]) and LSE (fp32 [B,H,N]). S and P never reach
 * global memory.
 *
 * At d = 64 (without a split over the keys) a CTA holds one or two Q tiles:
 * one under a block mask and when pairs of tiles would fill at most four
 * waves of the GPU, two otherwise. The environment variable FA_FWD_Q_TILES=1
 * or 2 fixes the choice (tuning and tests); results agree to rounding order.
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
 * Forward pass on strided operands with Nq query rows and Nk keys per
 * (batch, head). Q, K, V are all FA_BF16 or all FA_F16; O has their type or
 * is FA_F32; LSE is fp32
 * contiguous [B,H,Nq]. Errors as for fa_forward, plus FA_ERR_UNSUPPORTED or
 * FA_ERR_MISALIGNED for a descriptor outside the rules of fa_tensor
 * (fa_last_error() names the operand).
 */
fa_status fa_forward_ex(const fa_tensor *Q, const fa_tensor *K, const fa_tensor *V,
                        const fa_tensor *O, float *LSE, int B, int H, int Nq, int Nk, int d,
                        int causal, float scale, const uint8_t *block_mask, void *stream);

/*
 * Forward pass with the keys split over several CTAs, for shapes with few
 * query tiles per (batch, head), e.g. decoding against a long cache, where
 * the plain forward would leave most SMs idle. Each of the num_splits shares
 * of a query tile's K/V tiles yields a normalised partial output O_s and its
 * LSE_s in `workspace`; a second kernel merges them with the block-merge rule
 * of "Paper Notes: FlashAttention", section "Tiling: Block-by-Block Softmax"
 * (merged max = larger max; each block's sum and output rescaled by
 * exp(m_block - m); the sums add), in LSE form:
 *     LSE = ln sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) O_s.
 * The result equals fa_forward_ex's up to rounding. Arguments and errors are
 * those of fa_forward_ex, plus: num_splits in [1, 128] (1: no split, the
 * workspace is not used; FA_ERR_INVALID_ARG below 1, FA_ERR_UNSUPPORTED
 * above 128); workspace: a device buffer of at least
 * fa_forward_split_workspace_bytes(B,H,Nq,d,num_splits) bytes, 256-byte
 * aligned, clobbered.
 */
fa_status fa_forward_split_ex(const fa_tensor *Q, const fa_tensor *K, const fa_tensor *V,
                              const fa_tensor *O, float *LSE, int B, int H, int Nq, int Nk,
                              int d, int causal, float scale, const uint8_t *block_mask,
                              int num_splits, void *workspace, size_t workspace_bytes,
                              void *stream);

/* Workspace bytes of fa_forward_split_ex: fp32 [num_splits][B][H][Nq][d]
 * partial outputs and fp32 [num_splits][B][H][Nq] partial LSE, each on a
 * 256-byte boundary (0 for num_splits = 1 or invalid sizes). */
size_t fa_forward_split_workspace_bytes(int B, int H, int Nq, int d, int num_splits);

/* The library's choice of num_splits for this shape on the calling thread's
 * current device: 1 when the plain forward already gives every SM a CTA (or
 * on any error), else about SM count / CTAs, with at least two K/V tiles per
 * split, at most 128. */
int fa_forward_num_splits(int B, int H, int Nq, int Nk, int d, int causal);

/*
 * Bytes of device workspace fa_backward and fa_backward_ex need for N query
 * rows per (batch, head) in their default form for head dimension d: fp32 D
 * (D_i = dO_i.O_i) and fp32 LSE*log2(e), each [B,H,ceil(N/128)*128], and for
 * d <= 128 (where the one-pass backward is the default) an fp32 dQ
 * accumulator [B,H,ceil(N/128)*128,d], each part on a 256-byte boundary:
 * O(N*d), 8 + 4d bytes per query row for d <= 128, 8 for d = 256. Returns 0
 * for invalid sizes.
 */
size_t fa_backward_workspace_bytes(int B, int H, int N, int d);

/*
 * The smallest workspace fa_backward and fa_backward_ex accept: the two
 * statistics only, 8 bytes per query row (O(N)). It selects the two-kernel
 * backward, which recomputes S and dP in a second kernel that owns dQ instead
 * of accumulating dQ in the workspace: a few percent (d = 128) to 25 % (d = 64)
 * slower, bitwise reproducible, and with 4d fewer bytes of workspace per row.
 * Returns 0 for invalid sizes.
 */
size_t fa_backward_min_workspace_bytes(int B, int H, int N, int d);

/*
 * The workspace that selects the one-pass backward (d <= 128): the statistics
 * and the fp32 dQ accumulator, 8 + 4d bytes per query row; equal to
 * fa_backward_workspace_bytes for d <= 128. Returns 0 for d = 256 (two-kernel
 * form only) and for invalid sizes.
 */
size_t fa_backward_one_pass_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward pass. Reads Q, K, V, O, dO (bf16) and LSE (fp32, as written by the
 * forward pass with the same arguments); writes dQ, dK, dV (bf16 [B,H,N,d]).
 * `workspace` is a caller-owned device buffer of at least
 * fa_backward_min_workspace_bytes(B,H,N,d) bytes, 256-byte aligned; its
 * contents on entry do not matter and are clobbered. The score and
 * probability tiles are recomputed on chip and never reach global memory.
 *
 * The workspace size selects the form. With at least
 * fa_backward_one_pass_workspace_bytes(B,H,N,d) bytes (d <= 128) one kernel
 * recomputes S and P once per (Q tile, K/V tile) pair and runs all five
 * products there: dK and dV accumulate on chip, and each pair's dQ partial
 * is added into the fp32 accumulator in the workspace by atomic reductions,
 * so dQ's rounding can differ from run to run in the last bits. With less
 * (at least fa_backward_min_workspace_bytes), the two-kernel form runs, whose
 * results are bitwise reproducible. fa_backward_workspace_bytes gives the
 * faster form's size for each head dimension. The environment variable
 * FA_BWD_ALGO=split selects the two-kernel form whatever the workspace (a
 * tuning switch).
 */
fa_status fa_backward(const void *Q, const void *K, const void *V, const void *O,
                      const void *dO, const float *LSE, void *dQ, void *dK, void *dV, int B,
                      int H, int N, int d, int causal, float scale, const uint8_t *block_mask,
                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * Backward pass on strided operands with Nq query rows and Nk keys per
 * (batch, head): Q, O, dO, dQ have Nq rows, K, V, dK, dV have Nk rows, all
 * FA_BF16 or all FA_F16; LSE is fp32 contiguous [B,H,Nq] as written by fa_forward_ex with
 * the same arguments. The workspace holds at least
 * fa_backward_workspace_bytes(B,H,Nq,d) bytes, 256-byte aligned.
 */
fa_status fa_backward_ex(const fa_tensor *Q, const fa_tensor *K, const fa_tensor *V,
                         const fa_tensor *O, const fa_tensor *dO, const float *LSE,
                         const fa_tensor *dQ, const fa_tensor *dK, const fa_tensor *dV, int B,
                         int H, int Nq, int Nk, int d, int causal, float scale,
                         const uint8_t *block_mask, void *workspace, size_t workspace_bytes,
                         void *stream);

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
 * loads the library reserves until the process exits. The call runs the
 * default form when fa_backward_workspace_bytes(B,H,N,d) fits in the area,
 * else the two-kernel form; a call whose
 * fa_backward_min_workspace_bytes(B,H,N,d) exceeds it returns
 * FA_ERR_UNSUPPORTED before doing anything, and fa_last_error() states both
 * sizes. The call
 * allocates no memory (no cudaMalloc, no cudaFree, no allocating library
 * routine) as long as the measurement hooks are off, which is the default.
 *
 * Every call looks up the scratch area's device address on the device that
 * holds Q (cudaGetSymbolAddress; the first such lookup on a device loads the
 * library's device code there). Make the first call on a device before any
 * stream capture. All calls on a device share the one area, and it keeps the
 * last call's contents (each call re-initialises what must start at zero
 * itself). Calls that overlap on the GPU, e.g. on two streams at once, race
 * on the area: serialise them. Like every entry point, the call leaves the
 * device that holds Q current on the calling thread.
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
 * 0 forward, 1 backward preprocess (D_i and LSE*log2 e), 2 backward dK/dV,
 * 3 backward dQ, 4 merge of a split forward, for head dimension 256 the
 * backward's 5 dV, 6 dK and 7 dQ kernels, 8 the one-pass backward and 9 its
 * dQ conversion; fa_kernel_name() names them ("" for an unknown id).
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

/*
 * Measurement helper for the exponential-rate ceiling of the softmax: runs
 * one CTA of 1024 threads per SM on the calling thread's current device (on
 * the legacy default stream), each thread evaluating 8 independent chains of
 * ex2.approx.ftz.f32, times the second of two launches with CUDA events, and
 * stores the ex2 operations per second of the whole GPU, at the clocks of
 * that moment, in *exps_per_second. Synchronises; allocates no device memory.
 */
fa_status fa_measure_exp2_rate(double *exps_per_second);
const char *fa_kernel_name(int kernel);
fa_status fa_profile_enable(int enable);
fa_status fa_profile_collect(float *total_ms, int *launches, int n);

#ifdef __cplusplus
}
#endif

#endif /* FA_H */
