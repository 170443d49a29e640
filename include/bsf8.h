/*
 * bsf8.h -- C ABI of libbsf8, a block-scaled FP8 weight library for GB300 (sm_103a).
 *
 * The method (pages "recipes/docker-images/mia-tp4/adapter/wo_a_w8.py" and
 * "recipes/docker-images/mia-tp4/adapter/shared_pad_k.py"):
 *   A bf16 weight W[G][N][K] is kept as an fp8 "twin": one e4m3 code per element plus
 *   one exponent byte (ue8m0, byte = e + 127) per 32x32 block.  The small-batch linear
 *   y[m][g][n] = sum_k x[m][g*K + k] * W[g][n][k] reads the twin, rebuilds each bf16
 *   weight exactly as bf16(e4m3 * 2^(byte-127)) in registers and accumulates in fp32;
 *   split-K partials are summed in a fixed order, so results are deterministic.
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers owned by the caller, except where a parameter says
 *     "host".  The library never allocates, and every buffer a call touches is named in its
 *     argument list -- with one exception: bsf8_gemm_static_scratch keeps its partials in a
 *     buffer compiled into the library (BSF8_STATIC_SCRATCH_BYTES, 8 MiB on every GPU that
 *     loads it), which calls that can overlap on the GPU must not use at the same time.
 *   - bf16 tensors are passed as void* holding IEEE bfloat16 bit patterns.
 *   - Row-major layouts:  w8[G][N][K] (uint8 e4m3fn codes),  exp[G][N/32][K/32]
 *     (uint8, byte = e + 127),  x[M][ldx] (bf16; group g uses columns [g*K, (g+1)*K)),
 *     y[M][G][N] (bf16),  partials[S][M][G][N] (fp32).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream), do not synchronise the host, and allocate nothing.
 *   - Every call validates its arguments on the host first and returns a status code
 *     without launching anything when they are invalid; on success it returns BSF8_OK
 *     once the work is enqueued.  Faults found by the kernels themselves (a bounded
 *     wait that ran out) are recorded in a device status word read by
 *     bsf8_device_status().
 *   - Shapes: N and K are multiples of 32 (one exponent per 32x32 block); G >= 1.
 *
 * This library needs an sm_103a GPU (GB300); it has no CPU fallback.
 */
#ifndef BSF8_H
#define BSF8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t without pulling in the CUDA headers. */
typedef struct CUstream_st *bsf8_stream_t;

/* Status codes. */
enum {
    BSF8_OK = 0,
    BSF8_ERR_SHAPE = 1,     /* N or K not a multiple of 32, a size < 1, M out of range  */
    BSF8_ERR_ALIGN = 2,     /* a pointer or stride breaks the 16-byte rule of the call  */
    BSF8_ERR_STRIDE = 3,    /* ldx < G*K                                                */
    BSF8_ERR_WORKSPACE = 4, /* workspace missing or smaller than the call needs         */
    BSF8_ERR_NULL = 5,      /* a required pointer is NULL                               */
    BSF8_ERR_CUDA = 6,      /* a CUDA runtime call failed (launch, attribute, copy)     */
    BSF8_ERR_TIMEOUT = 7,   /* a kernel gave up a bounded wait (device status only)     */
    BSF8_ERR_DEVICE = 8,    /* the current device is not sm_103 / cannot run the kernels */
    BSF8_ERR_VALUE = 9      /* an option or scalar argument is out of range             */
};

/* Largest row count a single bsf8_gemm call accepts.  The pages serve 2..8 and 9..192
 * decode / verify / draft rows from the twin and prefill through a rebuilt bf16 copy (the
 * drop mode); here prefill-sized calls run from the twin too: past 192 rows the
 * tensor-core kernel takes the tokens in tiles of 192. */
#define BSF8_MAX_M 16384

/* Returns a static, human-readable name for a status code. */
const char *bsf8_strerror(int status);

/* Library version as major*10000 + minor*100 + patch. */
int bsf8_version(void);

/* The CUDA runtime error code (a cudaError_t value) behind the most recent
 * BSF8_ERR_CUDA or BSF8_ERR_DEVICE returned by any call of this process, 0 if none
 * has occurred.  Kept process-wide (not per thread); for diagnostics only. */
int bsf8_last_cuda_error(void);

/* --------------------------------------------------------------------- make_twin
 * "wo_a_w8.py", make_twin(): per 32x32 block of the bf16 weight w[G][N][K]
 *   amax = max |w| (raised to at least 2^-126),  e = ceil(log2(amax/448)) in [-127,127],
 *   w8   = e4m3 round-to-nearest-even of w / 2^e,  exp = e + 127,
 *   block_ok = 1 iff bf16(e4m3 * 2^e) == w for all 1024 elements (value equality),
 * and *accepted = 1 iff every block is ok (the pages keep the twin only then).
 * Blocks holding NaN or Inf get block_ok = 0, exp = 0xFF and codes 0x7F (the pages
 * leave them undefined; the tensor is rejected either way).
 *   w        device, bf16 [G][N][K], 16-byte aligned
 *   w8       device, out, uint8 [G][N][K], 16-byte aligned
 *   exp      device, out, uint8 [G][N/32][K/32]
 *   block_ok device, out, uint8 [G][N/32][K/32], or NULL
 *   accepted device, out, one int32 (written 1 or 0 on the stream)
 * Errors: BSF8_ERR_NULL, BSF8_ERR_SHAPE, BSF8_ERR_ALIGN, BSF8_ERR_CUDA. */
int bsf8_make_twin(const void *w, uint8_t *w8, uint8_t *exp, uint8_t *block_ok,
                   int32_t *accepted, int G, int N, int K, bsf8_stream_t stream);

/* ----------------------------------------------------------------------- dequant
 * "wo_a_w8.py", _dequant_kernel(): out[g][n][k] = bf16( e4m3(w8[g][n][k]) *
 * 2^(exp[g][n/32][k/32] - 127) ), rounded to nearest even; exact for every code and
 * exponent byte (byte 255 is a +inf scale: 0 -> NaN, others -> +-inf; e4m3 NaN codes
 * give NaN).  The page's drop mode serves prefill from such a per-call copy.
 *   w8  device, uint8 [G][N][K], 16-byte aligned
 *   exp device, uint8 [G][N/32][K/32]
 *   out device, out, bf16 [G][N][K], 16-byte aligned
 * Errors: BSF8_ERR_NULL, BSF8_ERR_SHAPE, BSF8_ERR_ALIGN, BSF8_ERR_CUDA. */
int bsf8_dequant(const uint8_t *w8, const uint8_t *exp, void *out, int G, int N, int K,
                 bsf8_stream_t stream);

/* -------------------------------------------------------------------------- GEMM
 * "wo_a_w8.py", _wo_a_partial_w8() / _wo_a_mid_kernel() and their fixed-order
 * reduction (module docstring: "Split-K partials are summed in a fixed order"):
 *   y[m][g][n] = bf16( sum_{s=0..S-1} P[s][m][g][n] ),  summed s = 0, 1, ... in fp32,
 *   P[s][m][g][n] = sum over split s's columns of x[m][g*K+k] * bf16(W8[g][n][k]*2^e),
 * with the products accumulated in fp32 on the tensor cores.  Split s covers columns
 * [s*c*32, min(K, (s+1)*c*32)) with c = ceil((K/32)/S) (it may be empty).
 *   x         device, bf16 [M][ldx], 16-byte aligned, ldx a multiple of 8, ldx >= G*K
 *   w8, exp   the twin (layouts above); w8 16-byte aligned
 *   y         device, out, bf16 [M][G][N]
 *   M         1 .. BSF8_MAX_M
 *   split_k   0 = the library chooses (bsf8_gemm_auto_split), else 1 .. K/32
 *   workspace device scratch of at least bsf8_gemm_workspace_bytes(...) bytes, or
 *             NULL when that is 0: fp32 partials between the two passes, which the call
 *             runs when its kernel writes partials (the tensor-core kernel, M > 16, with
 *             more than 8 splits, or 2..8 splits whose blocks take more than one wave of
 *             the device's SMs -- past 192 rows at least ceil(K/2048) splits, as a token
 *             tile's accumulators must fit tensor memory; the other kernels when a slab of
 *             16 rows needs more than 64 column tasks, e.g. split_k > 64).  No zeroing is
 *             needed; it must not be shared by calls that can overlap.
 * The splits are summed inside one thread block, across a cluster of up to 8 blocks (16
 * for the decode-ahead tensor-core kernel, where the device schedules such clusters)
 * through distributed shared memory, or by the fixed-order reduce of a second pass, always
 * in the same fixed order as bsf8_gemm_partials followed by bsf8_splitk_reduce, which run
 * the same kernel (bsf8_gemm_kernel) and give the same bits.
 * The twin is treated as a static parameter: with programmatic dependent launch
 * (BSF8_OPT_PDL) the kernel starts reading w8 and exp while the kernel before it on the
 * stream may still run, if that kernel allows it (the library's kernels that write a
 * twin -- make_twin, pad_k -- never do; a caller's kernel that writes w8 or exp must not
 * trigger its dependents early).  x is read and y written only after that kernel ends
 * (before, x's rows may be prefetched into L2, which reads nothing into the call).
 * Errors: BSF8_ERR_NULL, BSF8_ERR_SHAPE, BSF8_ERR_ALIGN, BSF8_ERR_STRIDE,
 *         BSF8_ERR_WORKSPACE, BSF8_ERR_CUDA; BSF8_ERR_VALUE when BSF8_OPT_GEMM_PATH forces a
 *         kernel that cannot run the call. */
int bsf8_gemm(const void *x, const uint8_t *w8, const uint8_t *exp, void *y,
              int M, int N, int K, int G, int split_k, int64_t ldx,
              void *workspace, size_t workspace_bytes, bsf8_stream_t stream);

/* Workspace bsf8_gemm needs for these sizes (0 for most shapes; see bsf8_gemm). */
size_t bsf8_gemm_workspace_bytes(int M, int N, int K, int G, int split_k);

/* The split count bsf8_gemm uses for split_k = 0.  Returns a value in 1 .. K/32, or a
 * negative status for invalid sizes.  1 up to 8 rows, and for 9..32 rows where the
 * decode-ahead tensor-core kernel takes the call in one split (its one-split grid fits the
 * device's SMs); otherwise 1 up to 16 rows, and past 16 (the tensor-core kernel) as many
 * splits as keep its blocks in one wave of the current device's SMs, then enough that a
 * split's accumulators fit tensor memory.  With no device, past 16 rows a size-only rule
 * (at most 8) applies. */
int bsf8_gemm_auto_split(int M, int N, int K, int G);

/* Kernels of bsf8_gemm, as bsf8_gemm_kernel reports them and BSF8_OPT_GEMM_PATH forces them. */
enum {
    BSF8_KERNEL_STREAM = 2,          /* cp.async weight streaming, mma.sync (any M)          */
    BSF8_KERNEL_DECODE_AHEAD = 4,    /* weights rebuilt into tensor memory before the        */
                                     /* dependency wait, mma.sync (M <= 8)                   */
    BSF8_KERNEL_TENSOR_CORE = 5,     /* tcgen05 MMAs on 128-row blocks (any M, token tiles   */
                                     /* of 192)                                              */
    BSF8_KERNEL_WIDE = 6,            /* wide weights, codes widened to f16 (M <= 8)          */
    BSF8_KERNEL_DECODE_AHEAD_TC = 7  /* weights rebuilt into tensor memory as the tcgen05 A  */
                                     /* operand before the dependency wait (M <= 32)         */
};

/* The kernel bsf8_gemm -- and bsf8_gemm_partials, bsf8_gemm_static_scratch -- runs for these
 * sizes and split count (0 = the library's choice) under the current options and device: a
 * BSF8_KERNEL_* value.  Negative: -BSF8_ERR_SHAPE for invalid sizes, -BSF8_ERR_VALUE when
 * BSF8_OPT_GEMM_PATH forces a kernel that cannot run the call.  The choice never depends on
 * whether the caller asks for y or for the fp32 partials. */
int bsf8_gemm_kernel(int M, int N, int K, int G, int split_k);

/* First pass alone: writes the fp32 partials P[S][M][G][N] (S = split_k >= 1, every
 * split written, empty splits as +0) with the kernel bsf8_gemm runs for the same sizes and
 * split count.  Same arguments as bsf8_gemm.
 *   partials device, out, fp32 [S][M][G][N], 16-byte aligned
 * Errors: as bsf8_gemm. */
int bsf8_gemm_partials(const void *x, const uint8_t *w8, const uint8_t *exp,
                       float *partials, int M, int N, int K, int G, int split_k,
                       int64_t ldx, bsf8_stream_t stream);

/* Second pass alone ("wo_a_w8.py", the reduce after _partial_w8): for i < count,
 *   y[i] = bf16_rne( ((P[0][i] + P[1][i]) + P[2][i]) + ... + P[S-1][i] )
 * in fp32, left to right.
 *   partials device, fp32 [S][count]
 *   y        device, out, bf16 [count]
 * While the device status word holds BSF8_ERR_TIMEOUT (a first pass gave up a wait and
 * left incomplete partials) the kernel writes nothing; bsf8_device_status reads and
 * clears the word.
 * Errors: BSF8_ERR_NULL, BSF8_ERR_SHAPE, BSF8_ERR_CUDA. */
int bsf8_splitk_reduce(const float *partials, void *y, int S, int64_t count,
                       bsf8_stream_t stream);

/* The same fixed-order sum kept in fp32: y[i] = ((P[0][i] + P[1][i]) + ...) + P[S-1][i],
 * y a device float array of `count` values.  With bsf8_gemm_partials it gives the GEMM's
 * fp32 output -- the head variant of "docs/tp4-adapters.md" (draft_head_fp8: the block
 * logits of up to 64..128 rows as fp32, the head streamed once per call); with one split
 * the partials are that output already.  Errors and the timeout rule as bsf8_splitk_reduce. */
int bsf8_splitk_reduce_f32(const float *partials, float *y, int S, int64_t count,
                           bsf8_stream_t stream);

/* ------------------------------------- per-(row, 32-column) scales (1 x 32 blocks)
 * The adapter table of "docs/tp4-adapters.md" (draft_main_proj): e4m3 codes with one
 * power-of-two scale per (weight row, 32 columns), checked to reproduce the bf16 weight
 * exactly, for the draft's projection of up to 16 rows.  The pages give no formula for it;
 * these entry points take make_twin's rule with the block narrowed to 1 x 32.  Layouts as
 * above except the exponents (and make_twin_rows' flags): exp[G][N][K/32], byte e + 127.
 *   bsf8_make_twin_rows: as bsf8_make_twin, per 1 x 32 segment.
 *   bsf8_dequant_rows:   as bsf8_dequant with the per-row exponents.
 *   bsf8_gemm_rows:      as bsf8_gemm (same x, y, split rule and fixed-order sum) with the
 *                        per-row exponents, on the decode-ahead kernel for M <= 8 and on the
 *                        decode-ahead tensor-core kernel for 9..32 rows where bsf8_gemm uses
 *                        them, else on the cp.async streaming kernel (every M
 *                        up to BSF8_MAX_M; meant for the pages' <= 16 rows); split_k 0 means
 *                        1 up to 8 rows and where the decode-ahead tensor-core kernel takes
 *                        the call in one split, else the streaming kernel's choice; workspace per
 *                        bsf8_gemm_rows_workspace_bytes (0 unless a slab needs more than
 *                        64 column tasks).
 * Errors as the block-scale counterparts. */
int bsf8_make_twin_rows(const void *w, uint8_t *w8, uint8_t *exp, uint8_t *block_ok,
                        int32_t *accepted, int G, int N, int K, bsf8_stream_t stream);
int bsf8_dequant_rows(const uint8_t *w8, const uint8_t *exp, void *out, int G, int N, int K,
                      bsf8_stream_t stream);
size_t bsf8_gemm_rows_workspace_bytes(int M, int N, int K, int G, int split_k);
int bsf8_gemm_rows(const void *x, const uint8_t *w8, const uint8_t *exp, void *y, int M,
                   int N, int K, int G, int split_k, int64_t ldx, void *workspace,
                   size_t workspace_bytes, bsf8_stream_t stream);

/* --------------------------------------------------- GEMM without a workspace
 * The pages have no counterpart for this entry point; it serves callers that cannot
 * allocate device memory for a workspace -- e.g. a serving engine that has reserved all of
 * the GPU's memory for its own arena, or a plugin running inside one that may not call
 * the allocator.  With the split count bsf8_gemm uses (split_k 0: bsf8_gemm_auto_split):
 * where bsf8_gemm needs no workspace for the call (bsf8_gemm_workspace_bytes = 0: most
 * shapes, whose kernels sum their splits on chip) it is bsf8_gemm; otherwise it runs
 * bsf8_gemm_partials and then bsf8_splitk_reduce -- the same kernel and the same fixed-order
 * sum -- so its result equals bsf8_gemm's bit for bit, with the partials held in a buffer
 * compiled into the library:
 *   - the buffer is BSF8_STATIC_SCRATCH_BYTES (8 MiB) of device memory that every GPU
 *     which loads the library holds until the process exits;
 *   - a call that needs partials whose S*M*G*N*4 bytes (S = the split count used) exceed
 *     it returns BSF8_ERR_WORKSPACE without launching anything;
 *   - nothing is allocated and nothing needs clearing: every split writes all of its
 *     partials before the reduce reads them;
 *   - every call on a device shares that one buffer, so calls that can overlap on the GPU
 *     (on different streams, or on several host threads) race and must be serialised by
 *     the caller;
 *   - the first call on a device looks up the buffer's device address (a host call,
 *     cudaGetSymbolAddress), so make that first call before any stream capture.
 * Errors: as bsf8_gemm (BSF8_ERR_WORKSPACE as described: a call at exactly the limit runs). */
#define BSF8_STATIC_SCRATCH_BYTES (8u * 1024u * 1024u)

int bsf8_gemm_static_scratch(const void *x, const uint8_t *w8, const uint8_t *exp, void *y,
                             int M, int N, int K, int G, int split_k, int64_t ldx,
                             bsf8_stream_t stream);

/* --------------------------------------------------------------- L2 prefetch
 * "docs/tp4-adapters.md", adapter table, l2_prefetch row: pull a twin -- the codes
 * w8[G][N][K] and the exponents exp[G][N/32][K/32] -- into L2 ahead of the GEMM that reads
 * it, typically on a side stream while other work runs (collectives, kernels that do not
 * let the GEMM start early).  A hint: it reads nothing into the program and writes
 * nothing, so results are the same with or without it; the lines may be evicted again
 * before the GEMM runs if other traffic passes through L2 meanwhile.
 *   w8, exp  device, 16-byte aligned (exp's last partial 16 bytes are not prefetched)
 * Errors: BSF8_ERR_NULL, BSF8_ERR_SHAPE, BSF8_ERR_ALIGN, BSF8_ERR_CUDA. */
int bsf8_prefetch_l2(const uint8_t *w8, const uint8_t *exp, int G, int N, int K,
                     bsf8_stream_t stream);

/* ------------------------------------------------------------------------- pad-K
 * "shared_pad_k.py", _pad_weight(): the twin [G][N][K] becomes [G][N][Kp] with code 0
 * (+0) in the new columns and its exponents [G][N/32][K/32] become [G][N/32][Kp/32]
 * with pad_exp in the new block columns (127 = scale 1.0, the page's choice; any byte
 * but 255 leaves every output unchanged, since 0 * 2^e = 0).
 *   w8, exp           device, the input twin; w8 16-byte aligned
 *   w8_out, exp_out   device, out; w8_out 16-byte aligned
 *   Kp                a multiple of 32, >= K;  pad_exp  0 .. 255
 * Errors: BSF8_ERR_NULL, BSF8_ERR_SHAPE, BSF8_ERR_ALIGN, BSF8_ERR_VALUE, BSF8_ERR_CUDA. */
int bsf8_pad_k(const uint8_t *w8, const uint8_t *exp, uint8_t *w8_out, uint8_t *exp_out,
               int G, int N, int K, int Kp, int pad_exp, bsf8_stream_t stream);

/* "shared_pad_k.py", _pad_input(): x[M][ldx] (group g in columns [g*K, (g+1)*K))
 * becomes x_out[M][G*Kp] with +0 in the new columns of every group.
 *   x      device, bf16, 16-byte aligned, ldx a multiple of 8, ldx >= G*K
 *   x_out  device, out, bf16 [M][G*Kp], 16-byte aligned
 * Errors: BSF8_ERR_NULL, BSF8_ERR_SHAPE, BSF8_ERR_ALIGN, BSF8_ERR_STRIDE, BSF8_ERR_CUDA. */
int bsf8_pad_x(const void *x, int64_t ldx, void *x_out, int M, int G, int K, int Kp,
               bsf8_stream_t stream);

/* ------------------------------------------------------------------ diagnostics
 * Not part of the method: a measurement aid.  Launches 2*nsm one-warp blocks on `stream`;
 * the block on SM i writes out[2i] = the global nanosecond timer and out[2i+1] = SM i's
 * cycle counter (slots of SMs no block reached keep their contents).  Two samples around
 * a timed region give each SM's average clock over it.
 *   out  device, uint64 [nsm][2];  nsm  1 .. 4096 (the device's SM count)
 * Errors: BSF8_ERR_NULL, BSF8_ERR_SHAPE, BSF8_ERR_CUDA, BSF8_ERR_DEVICE. */
int bsf8_sm_clock_sample(uint64_t *out, int nsm, bsf8_stream_t stream);

/* --------------------------------------------------------------- status, options
 * Synchronises `stream`, then reads into *status (host) and clears the device status
 * word of the current device: BSF8_OK, or BSF8_ERR_TIMEOUT if a kernel gave up a
 * bounded wait since the last read (its outputs are then undefined).
 * Errors: BSF8_ERR_NULL, BSF8_ERR_CUDA. */
int bsf8_device_status(int *status, bsf8_stream_t stream);

/* Process-wide options (host state, read at each launch). */
enum {
    BSF8_OPT_PDL = 1,              /* 1 (default): programmatic dependent launch on    */
    BSF8_OPT_WAIT_TIMEOUT_NS = 2,  /* bound of every in-kernel wait (default 2e9 ns)   */
    BSF8_OPT_DEBUG_SKIP_LOADS = 3, /* test only: the GEMM kernels that wait on         */
                                   /* mbarriers (decode-ahead, decode-ahead tensor-    */
                                   /* core, tensor-core, wide-weight) issue no weight  */
                                   /* loads, so their bounded waits run out and the    */
                                   /* call ends with BSF8_ERR_TIMEOUT in the status    */
    BSF8_OPT_GEMM_PATH = 4         /* 0 (default): the kernel chosen by shape:         */
                                   /*  - up to 8 token rows: the decode-ahead kernel   */
                                   /*    when its grid fits two blocks an SM, else the */
                                   /*    wide-weight kernel at split_k 1, else the     */
                                   /*    cp.async streaming kernel;                    */
                                   /*  - 9..32 rows: the decode-ahead tensor-core      */
                                   /*    kernel when its plan holds (S x tasks of at   */
                                   /*    most 512 columns <= 16, past 8 where the      */
                                   /*    device schedules such clusters) and its grid  */
                                   /*    fits one block an SM;                         */
                                   /*  - else 9..16 rows: the tensor-core kernel at    */
                                   /*    split_k 1 over at least one 128-row block per */
                                   /*    SM, the streaming kernel otherwise;           */
                                   /*  - beyond 16 rows: the tensor-core kernel.       */
                                   /* Else a BSF8_KERNEL_* value forces that kernel:   */
                                   /* 2 streaming (any call); 4 decode-ahead (M <= 8); */
                                   /* 5 tensor-core; 6 wide-weight (M <= 8; K and the  */
                                   /* split's columns multiples of 128, at most 6144   */
                                   /* columns a split); 7 decode-ahead tensor-core     */
                                   /* (M <= 32, S x ceil(split columns / 512) <= 16).  */
                                   /* A call the forced kernel cannot run returns      */
                                   /* BSF8_ERR_VALUE (see bsf8_gemm_kernel).           */
};
/* Errors: BSF8_ERR_VALUE for an unknown option or a negative value. */
int bsf8_set_option(int option, int64_t value);
int64_t bsf8_get_option(int option);

#ifdef __cplusplus
}
#endif

#endif /* BSF8_H */
