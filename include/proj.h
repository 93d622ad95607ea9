/*
 * proj.h -- C ABI of libproj: weight-bandwidth-bound dense projections on
 * GB300 (sm_103a).
 *
 * The operation (muse_bf16_proj guide, ch. 1, §1.1 "What is computed"):
 *
 *     out[i, n] = sum over k of x[i, k] * W[n, k]        (out = x @ W.T, no bias)
 *
 * for five fixed layers (§1.1 table):
 *
 *     layer      N x K         W dtype   out dtype
 *     qkv_gate   2304 x 8192   bf16      bf16
 *     o          8192 x 1024   bf16      bf16
 *     pooler     4096 x 8192   bf16      bf16
 *     unpooler   8192 x 4096   bf16      bf16   (only rows 0..1023 at m <= 8)
 *     router      256 x 8192   fp32      fp32
 *
 * Accumulation is in fp32; the dense layers round the fp32 sum to bf16
 * (round-to-nearest-even) on output.  The router keeps fp32 weights and an
 * fp32 sum: at every token count the dispatch runs it on the CUDA cores, the
 * bf16 input (widened exactly) meeting the fp32 weights in fp32 fused
 * multiply-adds (no TF32 truncation anywhere).  On request only
 * (PROJ_VARIANT_PLANES3) the router runs on the tensor cores instead, its
 * weights split at prepare into three bf16 planes with hi + mid + lo == W
 * exactly, so every product x * plane is exact and only the fp32
 * accumulation rounds.
 *
 * Interface shape (guide ch. 1, §1.6 "Rules that shaped the code"):
 * prepare(weights) runs once, untimed, and may repack or losslessly recode
 * W; the timed call is replayed as a CUDA graph, so it branches on shapes
 * only, performs no host synchronisation, no allocation and no memset, and
 * caches nothing derived from x.  Split-K bookkeeping is reset on the GPU.
 *
 * Threading: a handle is not thread-safe and must not run on two streams
 * at the same time (its split-K workspace and counters are shared by calls).
 * Different handles are independent.
 *
 * Errors: every call validates its arguments before touching the GPU and
 * returns a proj_status (or NULL + proj_last_status() for constructors).
 * A CUDA error raised while enqueuing maps to PROJ_ECUDA.  Nothing aborts
 * the process and no C++ exception crosses this boundary.
 */
#ifndef PROJ_H_
#define PROJ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque, library-owned state of one prepared layer. */
typedef struct proj_ctx *proj_handle;

/* A CUDA stream (cudaStream_t / CUstream).  NULL means the legacy default
 * stream of the calling thread. */
typedef struct CUstream_st *proj_stream;

enum proj_layer {
    PROJ_QKV_GATE = 0,
    PROJ_O = 1,
    PROJ_POOLER = 2,
    PROJ_UNPOOLER = 3,
    PROJ_ROUTER = 4
};

enum proj_dtype { PROJ_BF16 = 0, PROJ_FP32 = 1 };

enum proj_flags {
    /* Also keep a lossless 12-bit exponent-window copy of a bf16 W and use
     * it for the token counts its kernel covers (project report, "Round 5 --
     * lossless 12-bit compressed weights", "Format"): per weight the raw low
     * byte plus a 4-bit (sign, 3-bit window code) field; the 8 window values
     * of the 7 high exponent bits are chosen per matrix to cover the most
     * weights; weights outside the window are restored exactly from a
     * per-tile escape list.  Results are bit-identical to the uncompressed
     * kernel.  If any tile holds more escapes than the format's per-tile
     * capacity, the encoding is declined and the handle runs uncompressed
     * (proj_info reports it).  Where K is a multiple of 1024 (<= 8192) a
     * second 12-bit copy in 1024-column row chunks (same window, escapes per
     * chunk, at most 7, else that copy is declined) serves the register GEMV
     * at m <= 2, and the same format over the warp-MMA GEMV's fragment-order
     * copy serves that GEMV from 3 tokens; both are bit-identical to their
     * dense forms, and proj_describe_ex names them "expwin12rc". */
    PROJ_ENCODE_EXPWIN12 = 1u << 0
};

enum proj_status {
    PROJ_OK = 0,
    PROJ_EINVAL = 1,        /* bad argument (NULL, wrong shape or dtype, m < 0) */
    PROJ_EUNSUPPORTED = 2,  /* valid request this build does not serve (m > m_max) */
    PROJ_EALIGN = 3,        /* a pointer is not 16-byte aligned */
    PROJ_ENOMEM = 4,        /* device or host allocation failed (prepare only) */
    PROJ_ECUDA = 5,         /* a CUDA call failed; see proj_last_cuda_error() */
    PROJ_EDEVICE = 6        /* a kernel reported a fault in its status word */
};

/* Variant selection for proj_run_ex (testing and tuning). */
enum proj_variant {
    PROJ_VARIANT_AUTO = 0,      /* the dispatch table's choice */
    PROJ_VARIANT_DENSE = 1,     /* uncompressed weights */
    PROJ_VARIANT_EXPWIN12 = 2,  /* 12-bit weights (handle must hold them): the row-chunk
                                   copy on the register GEMV at m <= 2, the recoded
                                   fragment copy on the warp-MMA GEMV where x fits its
                                   shared memory (m <= 32), else the tile records on the
                                   tensor cores (stream-K tile kernel, token tiles of
                                   at most 128: any m); each where it was built */
    PROJ_VARIANT_PLANES3 = 3    /* router only: the fp32 weights as three bf16 planes,
                                   hi + mid + lo == W exactly, on the tensor cores */
};

/* How CTAs sharing a tile combine their fp32 partials (both deterministic:
 * the summation order depends only on the partition). */
enum proj_reduce {
    PROJ_REDUCE_AUTO = 0,        /* the dispatch table's choice */
    PROJ_REDUCE_OWNER = 1,       /* the CTA holding the tile's first k-range sums
                                    the others' partials (small m) */
    PROJ_REDUCE_DISTRIBUTED = 2  /* every contributor sums 1/S of the tile */
};

/* Kernel family for proj_run_ex (testing and tuning). */
enum proj_kernel {
    PROJ_KERNEL_AUTO = 0,   /* the dispatch table's choice */
    PROJ_KERNEL_GEMV = 1,   /* row-streaming CUDA-core GEMV, m <= 2 */
    PROJ_KERNEL_TILE = 2,   /* tiled kernels: tensor cores (bf16) / FMA tiles (router),
                               split-K across CTAs through global memory */
    PROJ_KERNEL_MMA = 5,    /* bf16 layers, m <= 32 (as far as x fits shared memory: K <=
                               8192 / 4096 / 1024 at 8 / 16 / 32 tokens): weight-streaming
                               GEMV on the warp-level tensor-core MMA (mma.sync m16n8k16)
                               from a copy of W in fragment order; CTAs own whole 16-row
                               blocks (at most 4), proj_run_opts.grid = CTAs; the dispatch
                               form at 3 <= m <= 8 (not the pooler) and on o to 16 */
    PROJ_KERNEL_GEMV_REG = 4, /* m <= 2 (the router: m <= 16): CUDA-core GEMV with the
                                 weights loaded straight into registers, whole rows per
                                 CTA (PROJ_KERNEL_GEMV: through a shared-memory ring fed
                                 by bulk copies); for the router at 3 <= m <= 16, FP32
                                 FMAs with x in passes of eight tokens (the dispatch
                                 form at 3 <= m <= 8) */
    PROJ_KERNEL_GEMV_SPLITK = 6, /* router, m <= 32: the FP32-FMA weight-streaming GEMV with K
                                    split across a thread-block cluster (K / 1024 CTAs, one
                                    1024-column chunk of eight rows each, x staged per CTA for
                                    its chunk only), partials summed in rank order through
                                    distributed shared memory; the dispatch form at
                                    9 <= m <= 24; PROJ_EUNSUPPORTED elsewhere */
    PROJ_KERNEL_CLUSTER = 3, /* tensor cores (dense bf16 weights; the router's bf16 planes),
                               split-K inside a thread-block cluster combined through
                               distributed shared memory, and optionally across several
                               clusters per tile through global memory:
                               proj_run_opts.grid = cluster size (1..16),
                               proj_run_opts.groups = clusters per tile (1..8) */
    PROJ_KERNEL_ROWS = 8,   /* bf16 layers, m <= 32: weight-streaming GEMV on the warp-level
                               tensor-core MMA over whole row runs per CTA (CTA c of
                               proj_run_opts.grid, default the SM count, owns rows
                               [c N / grid, (c + 1) N / grid), at most 64), W and x
                               brought from their row-major layouts into a shared-memory
                               ring by tensor copies; proj_run_opts.groups = 32-column
                               steps per ring stage (a power of two dividing K / 32, at
                               most 64; 0 = chosen for the most bytes in flight);
                               PROJ_EUNSUPPORTED elsewhere */
    PROJ_KERNEL_PAIR = 7    /* bf16 layers (dense weights): tensor cores on CTA pairs
                               (tcgen05 cta_group::2, 256 weight rows per MMA, each CTA
                               holding half of the token tile's x), K split across
                               proj_run_opts.groups pairs per 256-row tile (1..8; 0 = cost
                               model), one thread-block cluster of 2 x groups CTAs whose
                               partials meet in L2; proj_run_opts.tile_n = 64, 128 or 256
                               tokens per tile; grid and reduce must be 0; groups > 1
                               needs the grid within one CTA per SM (the partials'
                               exchange is sized for that), else PROJ_EUNSUPPORTED; the
                               dispatch form on o above 128 tokens and on the unpooler
                               from 192 */
};

typedef struct proj_run_opts {
    int variant;    /* enum proj_variant */
    int grid;       /* CTAs of the partition (1 .. SMs), or the cluster size for
                       PROJ_KERNEL_CLUSTER; 0 = dispatch table */
    int reduce;     /* enum proj_reduce (tiled kernels); owner needs m <= 32 on bf16 */
    int kernel;     /* enum proj_kernel */
    int groups;     /* PROJ_KERNEL_CLUSTER: clusters sharing one output tile's K
                       (1..16); PROJ_KERNEL_PAIR: pairs sharing one 256-row tile's K
                       (1..8); 0 = dispatch table */
    int tile_n;     /* token tile width of the tensor-core kernels (16, 32, 64, 128
                       or 256; the 12-bit kernel 16 or 32); 0 = dispatch table */
    void *stamps;   /* optional, for measurement: a device buffer of 8 uint64 per
                       CTA of the launch that the row-run kernel (PROJ_KERNEL_ROWS)
                       and the tensor-core cluster and CTA-pair kernels fill with
                       %globaltimer readings (ns): [0] entry, [1] the wait on the
                       previous kernel of the stream passed, [2] first stage landed
                       (tensor-core issuer), [3] last MMA issued, [4] accumulator
                       complete, [5] accumulator staged (row-run: main loop done),
                       [6] past the cluster barrier before the combine, [7] exit;
                       slots a kernel has no phase for are left as they are;
                       NULL = none; ignored by the other kernels */
} proj_run_opts;

typedef struct proj_info_t {
    int layer;               /* enum proj_layer */
    int dtype;               /* enum proj_dtype of W */
    int64_t N, K;
    int64_t m_max;
    int expwin12;            /* 1 if the 12-bit copy is present and used */
    int expwin12_declined;   /* 1 if requested but declined (escape overflow) */
    int expwin12_e0;         /* window base: high7 in [e0, e0 + 7] */
    int64_t expwin12_escapes;        /* weights outside the window */
    int64_t expwin12_bytes;          /* bytes of the 12-bit stream incl. escapes */
    int64_t dense_bytes;             /* bytes of the packed uncompressed W */
    int64_t workspace_bytes;         /* split-K partials + counters */
    int num_sms;
    int reserved[7];
} proj_info_t;

/*
 * Prepare a layer.  Untimed; may allocate and synchronise.
 *   layer : enum proj_layer.
 *   W     : device pointer to row-major [N, K] weights, 16-byte aligned;
 *           bf16 for every layer but the router, fp32 for the router.  It is
 *           only read, and fully consumed before return: the caller may free
 *           it afterwards.
 *   N, K  : must equal the layer's fixed shape (table above).
 *   dtype : PROJ_FP32 for the router, PROJ_BF16 otherwise.
 * Returns NULL on error; proj_last_status() then says why.
 */
proj_handle proj_prepare(int layer, const void *W, int64_t N, int64_t K, int dtype);

/*
 * As proj_prepare, plus:
 *   flags  : enum proj_flags.
 *   m_max  : largest token count proj_run will be called with; sizes the
 *            workspace.  0 selects the default, 1024.
 *   status : optional out-parameter (may be NULL).
 */
proj_handle proj_prepare_ex(int layer, const void *W, int64_t N, int64_t K, int dtype,
                            uint32_t flags, int64_t m_max, int *status);

/*
 * Timed call.  Enqueues the projection on `stream` and returns; no
 * allocation, no host synchronisation, no memset; capturable in a CUDA graph.
 * Branches on m only.
 *   x   : device pointer, bf16 row-major [m, K], contiguous, 16-byte aligned.
 *   m   : token count, 0 <= m <= m_max (m = 0 returns PROJ_OK, no launch).
 *   out : device pointer, row-major [m, proj_out_features(h, m)], contiguous,
 *         16-byte aligned; bf16 for the dense layers, fp32 for the router.
 *         Every element is written.
 * x and out must not overlap.  Returns PROJ_OK or an error status.
 */
int proj_run(proj_handle h, const void *x, int64_t m, void *out, proj_stream stream);

/* proj_run with an explicit variant and split-K grid (opts may be NULL). */
int proj_run_ex(proj_handle h, const void *x, int64_t m, void *out, proj_stream stream,
                const proj_run_opts *opts);

/*
 * End-to-end call on HOST buffers: copies x_host [m, K] bf16 to a
 * handle-owned device buffer, runs the projection, and delivers the result to
 * out_host [m, proj_out_features(h, m)], all enqueued on `stream`.  For a
 * page-locked x_host (16-byte aligned) the copy in is a copy kernel reading
 * the buffer's device mapping; for a page-locked out_host the projection
 * kernel stores the result straight into its device mapping (every element
 * written once, as on device memory); other host memory goes through
 * cudaMemcpyAsync and a handle-owned staging buffer (asynchronous only for
 * page-locked memory).  The caller synchronises `stream` before reading
 * out_host.  Same m rules as proj_run.
 */
int proj_run_host(proj_handle h, const void *x_host, int64_t m, void *out_host,
                  proj_stream stream);

/* Output width at m tokens: N, except the unpooler's 1024 at m <= 8
 * (guide ch. 1, §1.1 table).  Returns -1 for a NULL handle. */
int64_t proj_out_features(proj_handle h, int64_t m);

/* Fill *info with the handle's facts.  Returns PROJ_OK or PROJ_EINVAL. */
int proj_info(proj_handle h, proj_info_t *info);

/*
 * Describe the kernel and launch shape proj_run would use at m (for
 * reports): writes a NUL-terminated string of at most `cap` bytes to `buf`.
 */
int proj_describe(proj_handle h, int64_t m, char *buf, size_t cap);

/* The same for proj_run_ex with these options (opts may be NULL): the kernel
 * and launch shape that call would use, or the status it would refuse with
 * (PROJ_EINVAL / PROJ_EUNSUPPORTED, nothing written). */
int proj_describe_ex(proj_handle h, int64_t m, const proj_run_opts *opts, char *buf, size_t cap);

/*
 * Decode the handle's packed weights back to row-major [N, K] at W_out
 * (device, same dtype as prepared).  With the 12-bit copy present it
 * decodes that copy, so a bitwise comparison with the original W checks
 * that the recode is lossless.  For the router, PROJ_VARIANT_PLANES3 sums
 * the three bf16 planes back to fp32 (the same check for the plane split).
 * variant = PROJ_UNPACK_FRAG16 decodes the bf16 layers' copy in warp-MMA
 * fragment order (the few-token GEMV's layout; PROJ_EUNSUPPORTED where it
 * was not built), and variant = PROJ_UNPACK_RC12 the 12-bit row-chunk copy
 * (bf16 layers with PROJ_ENCODE_EXPWIN12; PROJ_EUNSUPPORTED where it was
 * not built or was declined), and variant = PROJ_UNPACK_FRAG12 the 12-bit
 * recode of the fragment-order copy (same conditions; it uses a temporary
 * device buffer of N x K bf16 and synchronises `stream`).  variant =
 * PROJ_UNPACK_RUNS decodes the row-run copy of the few-token GEMV
 * (PROJ_KERNEL_ROWS: each CTA's rows as [K / 32 steps][rows][32 columns])
 * into all N rows, and PROJ_UNPACK_RUNS_SLICE the unpooler's copy of its
 * first 1024 rows into [1024, K] (PROJ_EUNSUPPORTED where not built).
 * Otherwise enqueued on `stream`.
 */
#define PROJ_UNPACK_FRAG16 16
#define PROJ_UNPACK_RC12 32
#define PROJ_UNPACK_FRAG12 64
#define PROJ_UNPACK_RUNS 128
#define PROJ_UNPACK_RUNS_SLICE 256
int proj_unpack_weights(proj_handle h, int variant, void *W_out, proj_stream stream);

/* Read and clear the handle's device status word (synchronises `stream`).
 * Returns PROJ_OK or PROJ_EDEVICE; *code receives the raw word if non-NULL. */
int proj_device_status(proj_handle h, proj_stream stream, uint32_t *code);

/* Free everything the handle owns (synchronises the device first). */
void proj_destroy(proj_handle h);

/* Status of the last failing call on this thread, and its text. */
int proj_last_status(void);
const char *proj_status_string(int status);
/* Last error text recorded on this thread: a CUDA error, or the reason an
 * argument was rejected ("" if none). */
const char *proj_last_cuda_error(void);

/*
 * Streaming read of `bytes` bytes at device pointer `buf` (16-byte aligned,
 * bytes a multiple of 16), with every byte reaching the SMs: the HBM read
 * floor of the timing harness, and, on a buffer larger than L2, the flush
 * that makes the next call cold.  Writes one 32-bit checksum per CTA to
 * `sink` (device, >= grid + 1 words; the last one is a status word).
 * grid = 0 picks two CTAs per SM for mode 0 and one for mode 1.
 * mode 0 = 128-bit register loads, mode 1 = bulk copies into shared memory;
 * adding PROJ_READ_PDL (4) launches it the way proj_run launches the
 * projection kernels, as a programmatic dependent launch (it may start as
 * the previous kernel's CTAs exit; it reads nothing that kernel writes).
 * Any other mode is PROJ_EINVAL.
 */
#define PROJ_READ_PDL 4
int proj_read_floor(const void *buf, int64_t bytes, void *sink, int grid, int mode,
                    proj_stream stream);

/*
 * FP32 FMA probe: the measured ceiling of the CUDA cores' fp32 fused
 * multiply-adds, the denominator for the router's FP32-FMA path (guide ch. 1,
 * §1.5).  Launches `grid` CTAs of 256 threads (grid = 0: eight per SM), each
 * thread running 8 independent chains of packed `fma.rn.f32x2` for `iters`
 * steps (1 <= iters <= 2^24); enqueued on `stream`, time it with events
 * there.  `sink` (device, >= 4 bytes, 4-byte aligned) is never written in
 * practice: it keeps the arithmetic alive.  *flops (if non-NULL) receives the
 * launch's floating-point operations, grid x 256 x 8 x 2 x 2 x iters.
 * Returns PROJ_OK; PROJ_EINVAL (NULL sink, iters or grid out of range);
 * PROJ_EALIGN; PROJ_ECUDA.
 */
int proj_fma_peak(void *sink, int iters, int grid, proj_stream stream, double *flops);

/* Number of SMs of the current device (0 on error). */
int proj_num_sms(void);

/*
 * Allocation-free GEMV for one or two tokens on caller-owned weights.
 * The method's pages have no counterpart of this call: it exists for callers
 * that may not allocate device memory -- a plugin or custom operator that a
 * host framework hands only its input and output buffers while that
 * framework's allocator owns the device memory, or latency-critical code
 * that must not call cudaMalloc/cudaFree (they can stall the whole device and
 * can fail at run time).  Such callers cannot use proj_prepare, which
 * allocates repacked weights and a workspace.
 *
 *   out[i, n] = sum over k of x[i, k] * W[n, k],  0 <= i < m,  0 <= n < N
 *
 *   W       : device, row-major [N, K], contiguous, 16-byte aligned; any N >= 1.
 *   w_dtype : PROJ_BF16 (out is bf16, fp32 sum rounded to nearest even) or
 *             PROJ_FP32 (out is fp32).
 *   K       : a multiple of 1024 in [1024, 8192].
 *   x       : device, bf16 row-major [m, K], 16-byte aligned.
 *   m       : 0, 1 or 2 (0 returns PROJ_OK and launches nothing).
 *   out     : device, row-major [m, N], 16-byte aligned; every element written.
 *
 * The kernel is the ring-form streaming GEMV that proj_run_ex runs with
 * kernel = PROJ_KERNEL_GEMV: with grid = min(SMs, 256) that call splits W over
 * the same min(SMs, 256, N) CTAs and gives bit-identical results (on devices
 * of at most 256 SMs the default grid is the same).  Its scratch is a
 * 4 KB static device array inside the library (hand-off flags, partial row
 * sums and a status word for at most 256 CTAs); each device that loads the
 * library holds it until the process exits.  Nothing is allocated by any
 * call: the first call on a device (the current device when it is made) looks
 * up the array's device address and sets the kernels' shared-memory limit, so
 * make that first call before capturing any stream.  Every call then clears
 * the flags and status word with an asynchronous memset on `stream` and
 * launches one kernel.  All calls on a device share the one array, so calls
 * that overlap on the GPU (different streams, or threads without ordering)
 * race and give wrong results; serialise them.  A stall of the kernel's
 * bounded waits is recorded in that array's status word, which this call
 * does not report: read it with proj_gemv_static_status.
 *
 * Returns PROJ_OK; PROJ_EINVAL for NULL pointers, N < 1, m < 0 or a bad
 * w_dtype; PROJ_EUNSUPPORTED for m > 2 or K outside the rule above (the
 * static scratch is sized for those limits); PROJ_EALIGN; PROJ_ECUDA.  The
 * reason for a rejection is readable through proj_last_cuda_error().
 */
int proj_gemv_static(const void *W, int w_dtype, int64_t N, int64_t K, const void *x,
                     int64_t m, void *out, proj_stream stream);

/* The status word of the last proj_gemv_static call on the current device
 * (each call clears it when it starts; its kernel sets it if a bounded wait
 * gave up, in which case some rows of `out` are not written).  Synchronises
 * `stream` -- the stream of that call -- then reads the word; not for use
 * while `stream` is being captured.  *code receives the raw word if
 * non-NULL.  Returns PROJ_OK (word zero), PROJ_EDEVICE (non-zero) or
 * PROJ_ECUDA; allocates nothing. */
int proj_gemv_static_status(proj_stream stream, uint32_t *code);

#ifdef __cplusplus
}
#endif

#endif /* PROJ_H_ */
