/*
 * qlora.h -- C ABI of libqlora.so: the QLoRA-adapted linear layer on one
 * GB300 (sm_103a), forward and hand-derived backward.
 *
 * The operation (web pages this follows):
 *   "Introducing Unsloth: LLM 训练提速 30 倍", section 手动 Autograd --
 *       the adapted projection X(W + A B) with W frozen and only A, B trained;
 *       the backward needs dA, dB and the input gradient; the chain product is
 *       bracketed through the skinny rank-r side, i.e. (X A) B, never X (A B).
 *   "利用 Unsloth 和 NVIDIA 硬件加速 LLM 训练", section 1 (4-bit) -- the frozen
 *       weight is stored in 4 bits and dequantised to 16 bits at compute time
 *       so the product runs on tensor cores.
 *   "UnSloth极速微调" -- the LoRA branch is fused with the main linear; bf16
 *       is the 16-bit format.
 *   "Unsloth如何实现2倍速训练", section 2.2 -- the frozen weight receives no
 *       gradient (no dW is ever computed).
 *
 * With Wd = deq(W) [N,K], X [M,K], A [K,R], B [r,N], s the LoRA scale:
 *   forward :  XA = X A                         (saved for the backward)
 *              Y  = X Wd^T + s (X A) B
 *   backward:  G  = dY B^T
 *              dX = dY Wd + s G A^T
 *              dA = s X^T G
 *              dB = s (X A)^T dY
 * Several adapters may sit side by side over N ("segments", e.g. fused
 * Q/K/V): segment j owns columns [off_j, off_j + seg_n[j]) of Y / B / dY and
 * columns [j r, (j+1) r) of A, XA, G and dA; R = n_seg * r.
 *
 * Conventions shared by every entry point
 *   - Every tensor is row-major and dense (row stride = its last dimension).
 *   - "bf16" buffers hold IEEE bfloat16 bit patterns (2 bytes / element).
 *   - Tensor pointers are DEVICE pointers, 16-byte aligned, owned by the
 *     caller; the library allocates nothing and keeps no state between calls
 *     (apart from the optional profiler and the wait-limit setting below).
 *   - Calls are asynchronous and ordered on the given stream.  Argument
 *     errors are detected on the host before anything is launched.
 *   - Device-side failures (a bounded wait that ran out) set a flag in the
 *     workspace; qlora_check_device_error() reports it.
 */
#ifndef QLORA_H_
#define QLORA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QLORA_OK = 0,
  QLORA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bad rank, ... */
  QLORA_ERR_UNSUPPORTED = 2,  /* valid in principle, not handled (e.g. K % 64) */
  QLORA_ERR_ALIGNMENT = 3,    /* a pointer is not 16-byte aligned */
  QLORA_ERR_WORKSPACE = 4,    /* workspace missing or too small */
  QLORA_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed */
  QLORA_ERR_TIMEOUT = 6       /* a device-side bounded wait ran out */
} qlora_status;

/* Frozen 4-bit weight W [N,K] ("load_in_4bit" storage).
 *   idx      device, uint8 [N, K/2]: two 4-bit codes per byte, element (n,k)
 *            is in byte (n*K+k)/2, low nibble for even k, high for odd k.
 *   absmax   device, fp32 [N*K/64]: one scale per 64 consecutive elements of
 *            the row-major flattening (blocks never straddle rows: K % 64 == 0).
 *   codebook device, fp32 [16].
 *   deq(W)[n,k] = bf16_rne( fp32( codebook[code(n,k)] * absmax[(n*K+k)/64] ) ) */
typedef struct {
  const uint8_t* idx;
  const float* absmax;
  const float* codebook;
  int64_t N;
  int64_t K;
  int32_t block; /* must be 64 */
} qlora_w4;

/* Dequantise W to bf16 [N,K] (out_bf16, may be NULL) and/or to the exact fp32
 * products [N,K] (out_f32, may be NULL; at least one must be given).
 * Page: "利用 Unsloth 和 NVIDIA 硬件加速 LLM 训练", section 1.
 * Errors: INVALID_ARG (null W fields, both outputs NULL, negative sizes,
 * block != 64), UNSUPPORTED (K % 64 != 0), ALIGNMENT, CUDA. */
qlora_status dequant_4bit(const qlora_w4* w, void* out_bf16, float* out_f32, cudaStream_t stream);

/* Quantise a weight W [N,K] to the storage above (the models are loaded with
 * load_in_4bit=True: page "利用 Unsloth 和 NVIDIA 硬件加速 LLM 训练", section
 * 代码实战, and its section 1 on 4-bit weights).  W: device, row-major, fp32
 * (w_is_bf16 == 0) or bf16 bit patterns (w_is_bf16 != 0); finite values.
 * For each 64-block of the row-major flattening absmax = max |w|, and each
 * element takes the first code i minimising |w/absmax - codebook[i]|, both
 * the quotient and the differences in double precision (a zero block takes
 * the code nearest 0).  The codebook (device, fp32 [16]) need not be sorted.
 * Writes idx (device, uint8 [N, K/2], layout as in qlora_w4) and absmax
 * (device, fp32 [N*K/64]).  The caller owns every buffer.
 * Errors: INVALID_ARG (null pointer with N > 0, N < 0, K <= 0),
 * UNSUPPORTED (K % 64 != 0), ALIGNMENT (W, idx or absmax not 16-byte
 * aligned), CUDA. */
qlora_status quantize_4bit(const void* W, int32_t w_is_bf16, int64_t N, int64_t K, const float* codebook,
                           uint8_t* idx, float* absmax, cudaStream_t stream);

/* Forward: XA = X A (saved for the backward), Y = X Wd^T + s (X A) B.
 * Pages: "Introducing Unsloth: LLM 训练提速 30 倍", section 手动 Autograd (the
 * adapted projection X(W + AB), bracketed through the rank-r side);
 * "利用 Unsloth 和 NVIDIA 硬件加速 LLM 训练", section 1 (the 4-bit weight
 * dequantised to 16 bits for the tensor-core product); "UnSloth极速微调" (the
 * LoRA branch fused with the main linear).
 * X bf16 [M,K]; A bf16 [K, n_seg*r]; B bf16 [r,N]; seg_n HOST int64
 * [n_seg] summing to N (may be NULL when n_seg == 1); s the LoRA scale.
 * Writes Y bf16 [M,N] and XA_save bf16 [M, n_seg*r] = bf16(X A) (pass it to
 * qlora_linear_bwd).  ws / ws_bytes: device workspace of at least
 * qlora_workspace_bytes(M, N, K, r, n_seg) bytes, 256-byte aligned, whose
 * first 256 bytes were zeroed once before first use (they hold the device
 * error flag).  M == 0 is a no-op.
 * Preconditions: K % 64 == 0, N % 8 == 0, 8 <= r <= 128, r % 8 == 0,
 * n_seg * r <= 256, 1 <= n_seg <= 8, every segment but the last a multiple
 * of 128 columns, W->N == N.
 * Errors: INVALID_ARG, UNSUPPORTED, ALIGNMENT, WORKSPACE, CUDA. */
qlora_status qlora_linear_fwd(const void* X, int64_t M, const qlora_w4* W, const void* A, const void* B,
                              int32_t r, int32_t n_seg, const int64_t* seg_n, float s, void* Y,
                              void* XA_save, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Backward.  dY bf16 [M,N]; X bf16 [M,K]; XA_saved bf16 [M, n_seg*r] from the
 * forward; the other inputs as in the forward.  Writes dX bf16 [M,K] (skipped
 * when dX is NULL), dA fp32 [K, n_seg*r] and dB fp32 [r,N]; dA and dB are
 * overwritten, not accumulated (M == 0 writes zeros).  Page: "Introducing
 * Unsloth", section 手动 Autograd.  Errors as for the forward. */
qlora_status qlora_linear_bwd(const void* dY, const void* X, const void* XA_saved, int64_t M,
                              const qlora_w4* W, const void* A, const void* B, int32_t r, int32_t n_seg,
                              const int64_t* seg_n, float s, void* dX, float* dA, float* dB, void* ws,
                              size_t ws_bytes, cudaStream_t stream);

/* Backward for gradient accumulation over micro-batches: as qlora_linear_bwd
 * (same arguments, same dX), but the adapter gradients are added into dA and
 * dB instead of overwriting them: dA += s X^T G, dB += s XA^T dY, each element
 * updated as fl32(old + fl32(s * sum)).  M == 0 leaves dA and dB unchanged.
 * Page: "Introducing Unsloth", section 手动 Autograd (the adapter gradients);
 * errors as for the forward. */
qlora_status qlora_linear_bwd_accumulate(const void* dY, const void* X, const void* XA_saved, int64_t M,
                                         const qlora_w4* W, const void* A, const void* B, int32_t r,
                                         int32_t n_seg, const int64_t* seg_n, float s, void* dX, float* dA,
                                         float* dB, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Workspace bytes needed by qlora_linear_fwd / qlora_linear_bwd for these
 * sizes (the larger of the two); 0 for invalid sizes. */
size_t qlora_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t r, int32_t n_seg);

/* Synchronise `stream`, read and clear the workspace's device error flag.
 * Returns OK, TIMEOUT (a kernel's bounded wait ran out; its outputs are not
 * valid) or CUDA (a pending CUDA error, e.g. a failed launch). */
qlora_status qlora_check_device_error(void* ws, cudaStream_t stream);

/* Upper bound, in nanoseconds, on every barrier wait inside the kernels
 * (default 2e9).  Values below 1e6 are raised to 1e6. */
void qlora_set_wait_limit_ns(uint64_t ns);

/* Test hook for the failure path: the next launch of the GEMM with this label
 * ("gemm_xa", "gemm_fwd", "gemm_g", "gemm_dx", "gemm_dadb" or
 * "gemm_xa_static")
 * leaves the first shared-memory stage of its first CTA (CTA pair) unfilled,
 * so that CTA's consumer wait runs out after the wait limit; the kernel then
 * winds down, frees its tensor memory and sets the workspace error flag, and
 * qlora_check_device_error (qlora_linear_xa_static_status for the
 * static-scratch entry point) returns QLORA_ERR_TIMEOUT.  That call's outputs
 * are not valid; later calls work normally.  NULL clears a pending request. */
void qlora_debug_stall_next_launch(const char* label);

/* Human-readable name of a status code (static storage). */
const char* qlora_status_str(qlora_status status);

/* ---- Profiler: CUDA events around every kernel the library launches ---- */
typedef struct {
  const char* name;    /* kernel label (static storage) */
  int64_t launches;    /* launches recorded since the last collect */
  double total_ms;     /* summed event-measured duration */
} qlora_kernel_stat;

/* Turn event recording on (1) or off (0).  Off by default. */
void qlora_profiler_enable(int on);
/* Wait for every recorded launch, fold the timings per kernel into `out`
 * (up to max_entries, ordered by first launch) and reset the records.
 * Returns the number of distinct kernels (may exceed max_entries). */
int qlora_profiler_collect(qlora_kernel_stat* out, int max_entries);
/* Number of kernels launched by this library since load (profiler or not). */
uint64_t qlora_launch_counter(void);

/* ---- XA = X A without a caller-provided workspace ----
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory themselves -- for example a plug-in
 * whose host application owns every device allocation, or a loop that must
 * not go through the allocator -- and so cannot provide the workspace the
 * other entry points need.
 * Computes XA bf16 [M,R] = bf16(X A) for X bf16 [M,K] and A bf16 [K,R], the
 * same values qlora_linear_fwd writes to XA_save (R = n_seg * r there).
 * Its scratch is a static device array of QLORA_XA_STATIC_SCRATCH_BYTES
 * (8 MiB) that every GPU which loads the library holds until the process
 * exits.  The first call on a device (and in each further CUDA context of
 * that device) looks the array's address up with that device current; make
 * that first call before any stream capture.  The cached address assumes the
 * device is not reset while the library is loaded.  All calls share the array
 * and it keeps the last call's contents: calls that can overlap on the GPU
 * (different streams, or several host threads) race -- order them on one
 * stream.  Only the array's failure word has to start at zero (it is zero
 * when the library loads, and qlora_linear_xa_static_status clears it).  The
 * call allocates nothing.  Sizes whose A^T (2 R K bytes) plus the fp32
 * partial sums of 128 rows do not fit in the array (less a 256-byte header)
 * are rejected with QLORA_ERR_WORKSPACE (for example K = 16384 with R = 256);
 * larger M is processed in row chunks.
 * Preconditions: K % 64 == 0, 8 <= R <= 256, R % 8 == 0, 16-byte aligned
 * pointers.  Errors: INVALID_ARG, UNSUPPORTED, ALIGNMENT, WORKSPACE, CUDA. */
#define QLORA_XA_STATIC_SCRATCH_BYTES (8u * 1024u * 1024u)
qlora_status qlora_linear_xa_static(const void* X, int64_t M, int64_t K, const void* A, int32_t R, void* XA,
                                    cudaStream_t stream);

/* Device-side outcome of the qlora_linear_xa_static calls on the current
 * device since the last query: synchronises `stream`, then returns OK,
 * TIMEOUT (a kernel's bounded wait ran out; that call's XA is not valid) or
 * CUDA, and clears the failure word.  Allocates nothing. */
qlora_status qlora_linear_xa_static_status(cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QLORA_H_ */
