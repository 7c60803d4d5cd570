/*
 * wq.h -- C ABI of libwq, weight-only quantized matrix multiply on GB300 (sm_103a).
 *
 *   y[m, n] = sum_k x[m, k] * w[k, n],   w[k, n] = (q[k, n] - zero[g, n]) * scale[g, n],
 *   g = k / group_size,
 *
 * with q an unsigned w_bit-bit code (w_bit 2 or 4) packed 32/w_bit per int32
 * along K, as stated by BitDistiller, quantization/triton_kernels.py,
 * quant_matmul_kernel (docstring: "a: (M, K), qw: (K // pack_num, N),
 * scales: (K // group_size, N), qzeros: (K // group_size // pack_num, N)";
 * K loop: field = (packed >> ((k % pack_num) * w_bit)) & offset).  That page is
 * cut off before the scale/zero step; this library takes (q - zero) * scale.
 * Two special cases are covered:
 *   - symmetric int4 with the zero fixed at 8 (zeros == NULL), as in the
 *     dequant() of aphrodite-engine marlin_cuda_kernel.cu, which folds "-8"
 *     into its subtraction; symmetric int2 takes zero 2;
 *   - int8 weights with one fp32 scale per output channel, y[m, n] =
 *     scale[n] * sum_k x[m, k] * q[n, k] (tiny-llm kernels/int8_gemv.py,
 *     int8_matmul docstring: x (M, K) bf16/fp16, q (N, K) int8, scale (N,) fp32
 *     -> y (M, N) fp32).
 *
 * Conventions shared by every entry point.
 *   - Every array pointer is a DEVICE pointer owned by the caller.  The library
 *     allocates nothing, never synchronises (except wq_check_device), and
 *     enqueues its kernels on `stream` (a cudaStream_t passed as void*; NULL is
 *     the legacy default stream).
 *   - Arguments are validated on the host before anything is launched; an
 *     invalid call returns a status and enqueues nothing.  No exception or
 *     longjmp crosses this ABI.
 *   - Layouts are row-major and dense (no strides).
 *   - Launch failures are reported as WQ_ERR_CUDA.  A device-side wait that
 *     gives up (bounded spin on a shared-memory barrier) records a flag that
 *     wq_check_device() turns into WQ_ERR_TIMEOUT; the kernel then returns
 *     without faulting.
 *   - The library keeps no state besides per-device caches (SM count,
 *     kernel attributes, launch plans, tensor maps, the device addresses of
 *     its own __device__ variables).  cudaDeviceReset while the library is
 *     in use is not supported: those cached addresses would be stale.
 */
#ifndef WQ_H
#define WQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define WQ_API __attribute__((visibility("default")))
#else
#define WQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    WQ_OK = 0,
    WQ_ERR_NULL = 1,       /* a required pointer is NULL                               */
    WQ_ERR_SHAPE = 2,      /* M, N, K negative, zero where not allowed, or not divisible */
    WQ_ERR_WBIT = 3,       /* w_bit not in {2, 4, 8}                                   */
    WQ_ERR_GROUP = 4,      /* group_size does not divide K or is not a multiple of 16  */
    WQ_ERR_DTYPE = 5,      /* unsupported x or scale dtype for this w_bit              */
    WQ_ERR_ALIGN = 6,      /* a pointer is not 16-byte aligned                         */
    WQ_ERR_WORKSPACE = 7,  /* workspace NULL or smaller than wq_workspace_bytes()      */
    WQ_ERR_ARCH = 8,       /* current device is not compute capability 10.3            */
    WQ_ERR_CUDA = 9,       /* a CUDA runtime call or kernel launch failed              */
    WQ_ERR_TIMEOUT = 10    /* a kernel gave up waiting on one of its own barriers      */
} wq_status;

typedef enum { WQ_F16 = 0, WQ_BF16 = 1, WQ_F32 = 2 } wq_dtype;

/*
 * Human-readable name of a status; never NULL.
 * The statuses stand for the argument checks the pages make before a launch:
 * the TORCH_CHECKs of marlin_gemm and marlin_cuda (aphrodite-engine
 * marlin_cuda_kernel.cu: shape mismatches, K and N not divisible by the tile,
 * group size, workspace below its minimum) and the ValueError of tiny-llm
 * int8_matmul (kernels/int8_gemv.py: M above MAX_M, K mismatch, x not
 * bf16/fp16).  Here they are returned as codes, since no exception may cross
 * a C ABI.
 */
WQ_API const char *wq_status_string(wq_status s);

/*
 * Number of values along K that one packed chunk row spans: 256 / w_bit
 * (128 for w_bit 2, 64 for 4, 32 for 8).  K must be a multiple of it.  It
 * plays the part of Marlin's tile_size check on size_k (marlin_gemm,
 * aphrodite-engine marlin_cuda_kernel.cu): the tiled layout is only defined
 * for whole chunk rows.
 */
WQ_API int wq_chunk_k(int w_bit);

/*
 * Bytes of the packed weight buffer that wq_pack writes: K * N * w_bit / 8,
 * the same count as the input, whose shape the BitDistiller
 * quant_matmul_kernel docstring gives as qw: (K // pack_num, N) int32 with
 * pack_num = 32 / w_bit (and tiny-llm int8_matmul as q: (N, K) int8).
 * Returns 0 for an invalid shape or w_bit.
 */
WQ_API size_t wq_packed_bytes(int K, int N, int w_bit);

/*
 * wq_pack -- repack weights once, offline, into the tiled layout wq_matmul reads.
 *
 * q_in, w_bit 2 or 4: int32 (K / pack_num, N), pack_num = 32 / w_bit, in the
 *   layout of BitDistiller quant_matmul_kernel (field k % pack_num of word
 *   [k / pack_num][n], least significant field first).
 * q_in, w_bit 8: int8 (N, K), K contiguous, as in tiny-llm int8_matmul.
 * packed_out: wq_packed_bytes(K, N, w_bit) bytes.  The result is a pure bit
 *   permutation of the input (bit-exact and invertible by wq_unpack): chunk
 *   rows of KC = wq_chunk_k(w_bit) values along K, each holding N/16 tiles of
 *   16 output channels x KC, 512 bytes per tile, ordered so that one 16-byte
 *   load per thread of a warp yields whole tensor-core A fragments.
 * Requirements: N % 16 == 0, N <= 262144, K % KC == 0, both > 0; both
 *   pointers 16-byte aligned; q_in and packed_out must not overlap.
 */
WQ_API wq_status wq_pack(const void *q_in, int K, int N, int w_bit, void *packed_out, void *stream);

/*
 * wq_unpack -- inverse of wq_pack for tests and tooling.
 * codes_out: uint8 (K, N) row-major; code of (k, n) for w_bit 2/4, and the
 *   two's-complement byte of q[n, k] for w_bit 8.
 * The code of (k, n) is the field the K loop of BitDistiller
 * quant_matmul_kernel extracts from qw (K // pack_num, N):
 * (qw[k / pack_num][n] >> ((k % pack_num) * w_bit)) & (2^w_bit - 1).
 * Same requirements and statuses as wq_pack (packed 16-byte aligned).
 */
WQ_API wq_status wq_unpack(const void *packed, int K, int N, int w_bit, uint8_t *codes_out, void *stream);

/*
 * Bytes of scratch memory wq_matmul needs for this problem (0 if none).
 * It stands for the workspace of marlin_gemm (aphrodite-engine
 * marlin_cuda_kernel.cu), whose size check requires at least
 * (size_n / min_thread_n) * max_par ints of zero-filled lock counters for its
 * reduction across thread blocks along K; here the counters are followed by
 * fp32 partial sums (see below) and most shapes need none at all.
 * The workspace holds a fixed 16 KiB block of int32 arrival counters (one per
 * column block) followed by the fp32 partial sums of a split along K.  It
 * must be zero-filled before its first use; every completed call leaves the
 * counters at zero again, so one zero-fill at allocation is enough for any
 * later call, whatever its shape, as long as the buffer is large enough.  Calls that share a workspace must not
 * run concurrently (they would race on the counters and partials).
 * The split along K (and so this size) is chosen with the runtime's occupancy
 * calculator for the current device; the answer covers both the asymmetric
 * (zeros given) and the symmetric case and every x / scale dtype, so it may
 * exceed what a given call needs (a call on the tensor-core path for many
 * tokens needs none).
 */
WQ_API size_t wq_workspace_bytes(int M, int N, int K, int w_bit, int group_size);

/*
 * wq_matmul -- y = x * dequant(W), fp32 accumulation, fp32 output.
 *
 * x        (M, K) row-major, x_dtype WQ_F16 or WQ_BF16.
 * packed_w output of wq_pack for the same (K, N, w_bit).
 * scales   w_bit 2/4: (K / group_size, N), s_dtype WQ_F16 or WQ_BF16.
 *          w_bit 8:   (N,), s_dtype WQ_F32.
 * zeros    w_bit 2/4: int32 (ceil(G / pack_num), N), G = K / group_size, zero
 *          of group g in field g % pack_num of word [g / pack_num][n] (packed
 *          along the group axis like the weights along K); NULL selects the
 *          symmetric case, zero = 2^(w_bit - 1).  Unused high fields of the
 *          last row are ignored.  w_bit 8: must be NULL (zero is 0, codes signed).
 * group_size  w_bit 2/4: divides K, multiple of 16; -1 or K means one group per
 *          column.  w_bit 8: ignored (per output channel).
 * out      (M, N) fp32, fully overwritten.
 * x, packed_w, scales, zeros, out and workspace must be 16-byte aligned.
 * workspace / workspace_bytes: see wq_workspace_bytes (may be NULL/0 when it returns 0).
 *
 * M == 0 or N == 0 (with valid pointers) is a no-op returning WQ_OK, like the
 * early return of Marlin's host launcher.  K == 0 is WQ_ERR_SHAPE.
 * Precision: the weight codes and zeros enter the tensor cores exactly; the
 * group scale and zero are applied to the fp32 partial sum of each group (small
 * M) or to the weight, rounded once to the x dtype (large M).
 * The first call for a problem shape on a device asks the runtime's occupancy
 * calculator (host-side queries, cached per device and shape) and sets kernel
 * attributes; make that first call outside stream capture.
 */
WQ_API wq_status wq_matmul(const void *x, wq_dtype x_dtype, const void *packed_w,
                    const void *scales, wq_dtype s_dtype, const int32_t *zeros,
                    int M, int N, int K, int w_bit, int group_size,
                    float *out, void *workspace, size_t workspace_bytes, void *stream);

/*
 * wq_matmul_ex -- wq_matmul with a choice of output element type.
 *
 * out (M, N) row-major of out_dtype: WQ_F32 (the same as wq_matmul), WQ_F16
 * or WQ_BF16.  The result is accumulated in fp32 exactly as for wq_matmul and
 * rounded once, to nearest even, when it is stored: the fp16 output of
 * Marlin's write_result (aphrodite-engine marlin_cuda_kernel.cu, C allocated
 * in the activation dtype by marlin_gemm), without its fp16 reduction buffer.
 * A 16-bit output halves the bytes the epilogue writes.  Any other out_dtype
 * is WQ_ERR_DTYPE.  Every other argument, requirement and status as wq_matmul.
 */
WQ_API wq_status wq_matmul_ex(const void *x, wq_dtype x_dtype, const void *packed_w,
                              const void *scales, wq_dtype s_dtype, const int32_t *zeros,
                              int M, int N, int K, int w_bit, int group_size,
                              void *out, wq_dtype out_dtype,
                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * wq_matmul_noalloc -- wq_matmul for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point.  It exists for callers
 * that must not allocate at call time and cannot hand the library a
 * workspace: for example a plugin inside a host framework that owns every
 * device allocation, or a latency-critical path that cannot afford
 * cudaMalloc (which may synchronise the device).
 *
 * Same arguments and result as wq_matmul, without the workspace.  Its scratch
 * is a fixed 8 MiB array inside the library image that every GPU which loads
 * the library keeps until the process exits; no call allocates or frees
 * anything.  A problem on the few-token kernel (wq_matmul_path 0) whose
 * wq_workspace_bytes() exceeds 8 MiB returns WQ_ERR_WORKSPACE (use wq_matmul
 * with a workspace instead); the tensor-core kernels need no scratch here (the
 * many-token kernel runs one tile per thread block).
 *  - The first call on a device (made with that device current) looks up the
 *    array's device address; make that first call before any stream capture.
 *  - All calls share the one array and it keeps the previous call's
 *    contents; each call clears the part that must start at zero.  Calls whose
 *    kernels overlap on the GPU (different streams, or different host
 *    threads) race on the array: serialise them.
 */
WQ_API wq_status wq_matmul_noalloc(const void *x, wq_dtype x_dtype, const void *packed_w,
                                   const void *scales, wq_dtype s_dtype, const int32_t *zeros,
                                   int M, int N, int K, int w_bit, int group_size,
                                   float *out, void *stream);

/*
 * Ternary int2 (Liger kernels, ops/experimental/mm_int8int2.py):
 * weights in {-1, 0, 1} stored plus one as 2-bit fields of uint8, planar
 * along K (pack_weights: with R = K / 4 byte rows, bits 2i, 2i + 1 of byte
 * [k - i R][n] hold row k = i R + (k - i R)); int8 activations; the product
 * accumulated in int32 (matmul_kernel):
 *   y[m, n] = sum_k x[m, k] * (((q[k mod R][n] >> (2 (k div R))) & 3) - 1).
 * A field value of 3 stands for weight 2 (unpack_weights subtracts 1 from
 * every field).
 *
 * wq_t2_pack -- repack the planar bytes (K / 4, N) uint8 into the tiled
 * 2-bit layout wq_t2_matmul reads (K * N / 4 bytes, wq_packed_bytes(K, N, 2)).
 * Requirements: K % 128 == 0, K <= 65536, N % 16 == 0, N <= 262144; both
 * pointers 16-byte aligned and not overlapping.
 */
WQ_API wq_status wq_t2_pack(const void *q_in, int K, int N, void *packed_out, void *stream);

/*
 * Bytes of scratch wq_t2_matmul needs: the activations converted to bf16
 * (exact for int8), after any split-K partial sums of the few-token kernel
 * (same conventions as wq_workspace_bytes: zero-filled once before first use,
 * left reusable by every completed call, not shared by concurrent calls).
 */
WQ_API size_t wq_t2_workspace_bytes(int M, int N, int K);

/*
 * wq_t2_matmul -- y (M, N) int32 = x (M, K) int8 times the ternary weights
 * (output of wq_t2_pack).  Every product and partial sum is an integer below
 * 2^24 in magnitude (|x| <= 128, |w| <= 2, K <= 65536), so the tensor cores'
 * fp32 accumulation is exact and y equals the int32 result bit for bit.
 * x, packed_w, out and workspace 16-byte aligned; statuses as wq_matmul.
 */
WQ_API wq_status wq_t2_matmul(const int8_t *x, const void *packed_w, int M, int N, int K,
                              int32_t *out, void *workspace, size_t workspace_bytes, void *stream);

/*
 * wq_matmul_path -- which kernel family wq_matmul runs for this problem:
 * 0 the few-token kernel (TMA ring, register dequant, mma.sync, split-K in
 * clusters), 1 the exact tensor-core kernel (tcgen05, q - zero exact, group
 * scale in fp32), 2 the many-token tensor-core kernel (weight rounded once to
 * the x dtype), 3 the same kernel with each weight as two terms in the x
 * dtype (the rounded weight and its rounded residue: bf16 below K = 4096,
 * where one rounding could exceed the accepted error, on problems with
 * enough tiles to fill the GPU); -1 if wq_matmul would reject the arguments'
 * sizes, w_bit or dtypes.  The split by token count plays the part of tiny-llm's MAX_M
 * (kernels/int8_gemv.py: up to 64 rows per call on the few-token kernel,
 * more left to a GEMM) and of Marlin's small- and large-batch thread
 * configurations (aphrodite-engine marlin_cuda_kernel.cu).  No device is
 * touched.
 */
WQ_API int wq_matmul_path(int M, int N, int K, int w_bit, int group_size, wq_dtype x_dtype, wq_dtype s_dtype);

/*
 * wq_check_device -- synchronise `stream`, then read and clear the device
 * word in which kernels record a barrier wait that gave up.  Returns
 * WQ_ERR_TIMEOUT if one did, WQ_ERR_CUDA on a runtime error, else WQ_OK.
 * The pages have no status path of this kind: the barrier_acquire of
 * Marlin's cross-block reduction (aphrodite-engine marlin_cuda_kernel.cu)
 * spins on its lock without a limit.  Every wait of this library is bounded
 * and reports here instead of hanging the device.
 */
WQ_API wq_status wq_check_device(void *stream);

#ifdef __cplusplus
}
#endif
#endif /* WQ_H */
