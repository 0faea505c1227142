/*
 * w4a16.h - C ABI of the GB300 (sm_103a) int4 weight-only affine linear layer.
 *
 * The operation: a linear layer Y = X * W^T whose weight W[N][K] is stored as
 * 4-bit codes q in 0..15 with one binary16 scale and one binary16 bias per
 * group of G consecutive k (G = 64 by default), so that
 *     w[n][k] = scale[n][k/G]*q[n][k] + bias[n][k/G]          (affine), or,
 *     w[n][k] = scale[n][k/G]*(q[n][k] - 8)                   (symmetric),
 * when the weight has no biases.  Sources (page title, section):
 *   "The inference engine - Mojo 1.0 on Metal", "Crossing Mojo 1.0": decode
 *     is a weight-streaming multi-row GEMV plus on-device token selection;
 *     prefill dequantises each weight once into a transposed half-precision
 *     scratch and runs a half-precision GEMM.
 *   same page, "What's inside the engine today": int4 projections and LM
 *     head; greedy and top-k selection on the device.
 *   "engine-mlx", "Tech details": MLX 4-bit quantised format.
 *   "Engineering investigation ... 10x faster?", "Selective quantization":
 *     affine quantisation with group size 64.
 *   "The inference engine - Mojo 1.0 on Metal", "What's inside the engine
 *     today" and the appendix on porting MLX's kernels: that engine's own
 *     weights are symmetric int4 with group 128 (scale only).
 *
 * Storage format (shared by every call):
 *   qweight  uint32 [N][K/8], row-major.  Word j of row n holds q[n][8j+i]
 *            in bits 4i..4i+3 (lowest nibble = lowest k).
 *   scales   binary16 [N][K/G], row-major.
 *   biases   binary16 [N][K/G], row-major; NULL selects symmetric codes.
 *   group    G, a power of two with 32 <= G <= K and K % G == 0 (every call
 *            that takes `group`; 64 is the affine format above, 128 with
 *            NULL biases the symmetric group-128 format).
 *   Activations and outputs are binary16 (IEEE half, passed as uint16_t bit
 *   patterns), row-major.
 *
 * Conventions:
 *   - Every pointer is a DEVICE pointer on the current CUDA device, owned by
 *     the caller.  The library allocates no device memory and keeps no
 *     per-call state.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *     only enqueues work and returns before it completes.
 *   - The return value is a status code (W4A16_OK = 0).  All argument checks
 *     happen on the host before anything is enqueued; a failing check
 *     enqueues nothing.  W4_ERR_LAUNCH reports a launch error from the CUDA
 *     runtime.  No kernel traps.
 *   - Pointers must be 16-byte aligned.
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define W4A16_API __attribute__((visibility("default")))
#else
#define W4A16_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define W4A16_OK          0
#define W4_ERR_NULL       1  /* a required pointer is NULL */
#define W4_ERR_SHAPE      2  /* a dimension is out of the supported range */
#define W4_ERR_ALIGN      3  /* a pointer or row stride is not 16-byte aligned */
#define W4_ERR_GROUP      4  /* group not a power of two in 32..K dividing K */
#define W4_ERR_LAUNCH     5  /* the CUDA runtime rejected a launch */
#define W4_ERR_WORKSPACE  6  /* workspace missing or smaller than required */
#define W4_ERR_DEVICE     7  /* current device is not sm_103 or lacks a needed driver entry point */
#define W4_ERR_TIMEOUT    8  /* a device-side bounded wait expired (reported by w4a16_device_status) */

/*
 * Launch flag of the *_ex calls.  W4A16_OVERLAP_PREVIOUS lets the call's
 * kernel start while the previous kernel on the same stream is still running
 * (programmatic dependent launch): it streams its weights (qweight, scales,
 * biases) at once and waits for the previous kernel only before it reads its
 * activations and writes its outputs.  Use it when the weights are not
 * written by the preceding kernel on the stream (the usual case: weights are
 * loaded once).  Without the flag the call follows ordinary stream order.
 */
#define W4A16_OVERLAP_PREVIOUS 1u

/*
 * w4_gemv - decode GEMV, y[m][n] = sum_k w[n][k] * x[m][k].
 *   ("The inference engine - Mojo 1.0 on Metal", "Crossing Mojo 1.0": the
 *   multi-row weight-streaming GEMV.)
 *   x       binary16 [M][K]          activations
 *   qweight, scales, biases          int4 weight in the format above
 *   y       binary16 [M][N]          output; fp32 accumulation, rounded to
 *                                     nearest even once at the end
 *   M       1..16 activation rows, all sharing one pass over the weights
 *   N       >= 1 output features;  K  multiple of 64, >= 64;
 *   group   quantisation group (see the format); biases may be NULL
 * Errors: W4_ERR_NULL, W4_ERR_SHAPE, W4_ERR_GROUP, W4_ERR_ALIGN, W4_ERR_LAUNCH.
 */
W4A16_API int w4_gemv(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
            const uint16_t *biases, uint16_t *y, int M, int N, int K, int group,
            void *stream);

/* w4_gemv with launch flags (W4A16_OVERLAP_PREVIOUS or 0); otherwise identical. */
W4A16_API int w4_gemv_ex(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
            const uint16_t *biases, uint16_t *y, int M, int N, int K, int group,
            unsigned flags, void *stream);

/*
 * w4_gemv_seq - a list of GEMVs in one persistent launch (decode projection
 * list).
 *   ("The inference engine - Mojo 1.0 on Metal", "Appendix: the remaining
 *   gap": the per-token floor of some 250 small launches binds decode.)
 *   Runs ops[0..nops) in order, each exactly as w4_gemv would (same format,
 *   same results).  An operation with wait_prev != 0 reads activations that
 *   earlier operations of the list write: it starts only after they are
 *   complete and visible.  Weights are streamed without waiting, so they
 *   must not be written by the operations of the list.
 *   M       1..16 activation rows, shared by all operations.
 *   Each operation: N >= 1, K a multiple of 256, group (0 means 64) and
 *   biases (NULL: symmetric) as for w4_gemv, pointers 16-byte aligned.
 *   workspace  device buffer, 16-byte aligned, ZERO-FILLED before its first
 *              use and then passed unchanged to every later call (the library
 *              keeps its counters consistent: the last CTA of each launch
 *              resets them and advances an epoch).  With at least
 *              w4_gemv_seq_workspace_bytes_ex(ops, nops, M) bytes, an operation
 *              whose x lies inside the output of the latest earlier operation
 *              that writes any of x reads a tagged copy of that output (each
 *              word carries a 16-bit (epoch, operation) tag and the reader
 *              polls the words themselves); other waits, and every wait when
 *              the workspace holds only w4_gemv_seq_workspace_bytes() bytes,
 *              use a completion counter.  A workspace is used by one call at
 *              a time.  After an expired wait its contents are undefined:
 *              zero it again.
 *   flags   0.
 *   Long lists run as several launches of up to 96 operations; a launch is
 *   cooperative (one CTA per SM) and waits inside it are bounded (2 s; an
 *   expiry is reported by w4a16_device_status).
 * Errors: as w4_gemv, plus W4_ERR_WORKSPACE.
 */
typedef struct {
    const uint16_t *x;        /* binary16 [M][K] */
    const uint32_t *qweight;  /* [N][K/8] */
    const uint16_t *scales;   /* binary16 [N][K/G] */
    const uint16_t *biases;   /* binary16 [N][K/G], or NULL: symmetric codes */
    uint16_t *y;              /* binary16 [M][N] */
    int N, K;
    int wait_prev;            /* nonzero: x is written by an earlier operation */
    int group;                /* G of this operation's weight; 0 means 64 */
} w4_gemv_op;

/* Minimum workspace (completion counters only). */
W4A16_API size_t w4_gemv_seq_workspace_bytes(void);

/* Workspace for the tagged activation exchange of this operation list:
 * the counters plus, per launch of up to 96 operations, one uint32 word per
 * output element of every operation whose output a later one reads. */
W4A16_API size_t w4_gemv_seq_workspace_bytes_ex(const w4_gemv_op *ops, int nops, int M);

W4A16_API int w4_gemv_seq(const w4_gemv_op *ops, int nops, int M, void *workspace,
            size_t workspace_bytes, unsigned flags, void *stream);

/*
 * lm_head_argmax_topk - LM-head GEMV fused with token selection.
 *   ("The inference engine - Mojo 1.0 on Metal", "Crossing Mojo 1.0" and
 *   "What's inside the engine today": greedy / top-k selection on the GPU so
 *   that no logits vector crosses to the host.)
 *   Computes the fp32 logits l[m][n] = sum_k w[n][k] * x[m][k] for every
 *   n < N and returns, for each activation row m, the k largest:
 *   idx int32 [M][k] and val float32 [M][k], ordered by value descending,
 *   ties broken by the lowest index (k == 1 is greedy argmax).  No logits
 *   tensor is written: a first pass leaves per-block candidates in
 *   `workspace`, a second pass merges them.
 *   M 1..16;  N >= k;  K multiple of 64;  group and biases as for w4_gemv;
 *   1 <= k <= 64;
 *   N * k must not exceed 16,777,216.
 *   workspace  device buffer of at least lm_head_workspace_bytes(M, N, k)
 *              bytes, 16-byte aligned; contents on entry are ignored.
 * Errors: as w4_gemv, plus W4_ERR_WORKSPACE.
 */
W4A16_API int lm_head_argmax_topk(const uint16_t *x, const uint32_t *qweight,
                        const uint16_t *scales, const uint16_t *biases,
                        int M, int N, int K, int group, int k,
                        int32_t *idx, float *val,
                        void *workspace, size_t workspace_bytes, void *stream);

/* lm_head_argmax_topk with launch flags (W4A16_OVERLAP_PREVIOUS or 0). */
W4A16_API int lm_head_argmax_topk_ex(const uint16_t *x, const uint32_t *qweight,
                        const uint16_t *scales, const uint16_t *biases,
                        int M, int N, int K, int group, int k,
                        int32_t *idx, float *val,
                        void *workspace, size_t workspace_bytes, unsigned flags, void *stream);

/*
 * lm_head_argmax_topk_noalloc - lm_head_argmax_topk without a workspace
 * argument, for callers that cannot allocate device memory where they call it
 * (inside an allocator or memory-pool callback, under a fixed memory budget,
 * or in an embedding with no allocator of its own).  None of the pages has a
 * counterpart; it is a packaging variant of the call above.
 *   Arguments, results and limits are those of lm_head_argmax_topk; the
 *   candidate buffer is a 2 MiB array inside this library's device image,
 *   which covers every size lm_head_argmax_topk accepts (M <= 16, k * blocks
 *   <= 16384 keys per row).  Every GPU that loads the library holds the array
 *   until the process exits.  This call allocates nothing (no cudaMalloc, no
 *   library allocator).
 *   Set-up: the first call on a device looks up the array's device address on
 *   that device (cudaGetSymbolAddress) and caches it with the id of the CUDA
 *   context it belongs to; the first call in a new context (e.g. after
 *   cudaDeviceReset) looks it up again.  Make the first call on a device, and
 *   in each new context, before any stream capture on it.
 *   Sharing: all calls use the same array and it keeps the last call's
 *   contents.  Nothing in it has to start at zero: pass 1 writes every slot
 *   pass 2 reads, so a smaller call after a larger one never sees the
 *   larger call's leftovers.  Calls whose kernels overlap on the GPU (other
 *   streams, other host threads) race on the array: order them on one
 *   stream.
 * Errors: as lm_head_argmax_topk; W4_ERR_WORKSPACE if a size would need more
 * than the built-in 2 MiB; W4_ERR_DEVICE if the address lookup fails.
 */
W4A16_API int lm_head_argmax_topk_noalloc(const uint16_t *x, const uint32_t *qweight,
                        const uint16_t *scales, const uint16_t *biases,
                        int M, int N, int K, int group, int k,
                        int32_t *idx, float *val, void *stream);

/* Bytes of workspace lm_head_argmax_topk needs for these sizes (0 if the
 * sizes are invalid).  Depends only on its arguments. */
W4A16_API size_t lm_head_workspace_bytes(int M, int N, int k);

/*
 * w4_dequant_f16 - dequantise once into the transposed half scratch.
 *   ("The inference engine - Mojo 1.0 on Metal", "Crossing Mojo 1.0": each
 *   weight is dequantised once per prefill into a transposed half-precision
 *   scratch.)
 *   w16  binary16 [K][N] (= W transposed), w16[k][n] = the correctly rounded
 *        (nearest, ties to even) binary16 of the exact scale*q + bias, or of
 *        scale*(q - 8) when biases is NULL (a zero keeps the sign of the
 *        IEEE product scale*(q - 8)).
 *   N >= 1;  K multiple of 64;  group as for w4_gemv.
 * Errors: W4_ERR_NULL, W4_ERR_SHAPE, W4_ERR_GROUP, W4_ERR_ALIGN, W4_ERR_LAUNCH.
 */
W4A16_API int w4_dequant_f16(const uint32_t *qweight, const uint16_t *scales,
                   const uint16_t *biases, uint16_t *w16, int N, int K, int group,
                   void *stream);

/* w4_dequant_f16_ex - w4_dequant_f16 with flags (0 or W4A16_OVERLAP_PREVIOUS).
 * For this call W4A16_OVERLAP_PREVIOUS states more than for the GEMVs: the
 * call reads nothing the previous kernel on the stream writes and writes
 * nothing it reads or writes (e.g. one of many dequantisations of distinct
 * weights into distinct scratch buffers).  The kernel is then launched as a
 * programmatic dependent without any wait and may run concurrently with the
 * previous kernel. */
W4A16_API int w4_dequant_f16_ex(const uint32_t *qweight, const uint16_t *scales,
                                const uint16_t *biases, uint16_t *w16, int N, int K,
                                int group, unsigned flags, void *stream);

/*
 * w4_gemm - int4 GEMM with the dequantisation fused into the tensor-core
 * pipeline, for prefill with few activation rows:
 *   y[m][n] = sum_k w[n][k] * x[m][k],  w[n][k] = RNE_binary16(scale*q + bias)
 *   (or of scale*(q - 8) without biases): the weight values of
 *   w4_dequant_f16, multiplied without writing a scratch.
 *   ("The inference engine - Mojo 1.0 on Metal", "Crossing Mojo 1.0": the
 *   prefill GEMM over dequantised weights; here the weights are dequantised
 *   tile by tile into tensor memory and read from HBM only as 4-bit codes.)
 *   x        binary16 [M][K]   activations
 *   qweight, scales, biases, group    the int4 weight (format above)
 *   y        binary16 [M][N]   output; fp32 accumulation, one rounding
 *   M 1..128;  N >= 8, N % 8 == 0;  K >= 64, K % 64 == 0.
 *   workspace  device buffer of at least w4_gemm_workspace_bytes(M, N, K)
 *              bytes, 16-byte aligned, ZERO-FILLED before its first use and
 *              then passed unchanged to later calls (its grid-barrier
 *              counters are left ready for the next call).  Calls ordered on
 *              one stream may share it, also with W4A16_OVERLAP_PREVIOUS (a
 *              call touches it only after its dependency wait); calls that
 *              may run concurrently need separate workspaces.
 *              It holds the fp32 partial sums of the 128-row weight tiles
 *              whose k steps are shared by several blocks (the tiles left
 *              over after every block has taken whole tiles).
 *   The products are those of f16_gemm on the w4_dequant_f16 scratch (the
 *   same binary16 weight values); the 64-k steps of a tile are accumulated
 *   in fp32 starting from a per-tile rotation, and a tile shared by several
 *   blocks adds their partial sums in ascending k.  Results are
 *   deterministic.  For M <= 32 the last block to bring a shared tile's
 *   partial sums adds them all.  For M > 32 the launch is cooperative
 *   (every block resident): the blocks sharing a tile wait for each other's
 *   partial sums and each adds a slice (bounded: on expiry the call leaves
 *   that tile unwritten and w4a16_device_status reports W4_ERR_TIMEOUT).
 * Errors: W4_ERR_NULL, W4_ERR_SHAPE, W4_ERR_GROUP, W4_ERR_ALIGN,
 * W4_ERR_WORKSPACE, W4_ERR_DEVICE, W4_ERR_LAUNCH.
 */
W4A16_API int w4_gemm(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                      const uint16_t *biases, uint16_t *y, int M, int N, int K, int group,
                      void *workspace, size_t workspace_bytes, void *stream);

/* w4_gemm with launch flags (W4A16_OVERLAP_PREVIOUS: the weights are not
 * written by the previous kernel; their first tiles are fetched and
 * converted before it finishes). */
W4A16_API int w4_gemm_ex(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                         const uint16_t *biases, uint16_t *y, int M, int N, int K, int group,
                         void *workspace, size_t workspace_bytes, unsigned flags, void *stream);

/* Workspace bytes for w4_gemm (0 if the sizes are invalid): 3328 bytes of
 * counters and flags and 2 x min(256, ceil(N / 128) x K / 64) fp32 tiles of
 * M x 128.  Depends only on its arguments. */
W4A16_API size_t w4_gemm_workspace_bytes(int M, int N, int K);

/*
 * f16_gemm - dense half GEMM for prefill, y = x16 * w16.
 *   ("The inference engine - Mojo 1.0 on Metal", "Crossing Mojo 1.0": the
 *   half-precision GEMM that follows the dequantise-once step.)
 *   x16  binary16 [M][K] row-major;  w16  binary16 [K][N] row-major;
 *   y    binary16 [M][N] row-major; fp32 accumulation on the tensor cores,
 *        rounded to nearest even once at the end.
 *   M >= 1;  N >= 8 and a multiple of 8;  K >= 8 and a multiple of 8
 *   (row strides must be 16-byte multiples for the tensor-memory copies).
 * Errors: W4_ERR_NULL, W4_ERR_SHAPE, W4_ERR_ALIGN, W4_ERR_DEVICE, W4_ERR_LAUNCH.
 */
W4A16_API int f16_gemm(const uint16_t *x16, const uint16_t *w16, uint16_t *y,
             int M, int N, int K, void *stream);

/* f16_gemm_ex - f16_gemm with flags (0 or W4A16_OVERLAP_PREVIOUS).  With the
 * flag the kernel is a programmatic dependent of the previous kernel on the
 * stream: it sets up and copies the w16 tiles of its first stages at once and
 * waits for the previous kernel before it reads x16 or writes y.  w16 must
 * therefore be complete when the call is issued (not written by the previous
 * kernel, nor by any kernel still running beside it). */
W4A16_API int f16_gemm_ex(const uint16_t *x16, const uint16_t *w16, uint16_t *y, int M, int N,
                          int K, unsigned flags, void *stream);

/* Human-readable name of a status code (static string). */
W4A16_API const char *w4a16_status_string(int status);

/*
 * Synchronises the current device and reports whether any kernel of this
 * library gave up a bounded device-side wait since the last call
 * (W4_ERR_TIMEOUT), then clears the record.  W4A16_OK otherwise.
 */
W4A16_API int w4a16_device_status(void);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
