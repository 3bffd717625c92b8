/*
 * santa.h -- C ABI of libsanta.so: GB300-native (sm_103a) SANTA decode-step attention.
 *
 * The operation ("Stochastic Sparse Attention for Memory-Bound Inference", abstract):
 * one autoregressive decode step of attention over a long KV cache.  For every batch
 * row b and query head h (KV head g = h / (H_q / H_kv), grouped-query attention), the
 * score stage reads all n_b cached keys and forms p = softmax(scale * q K^T).  The value
 * stage does not compute the dense p.V product.  It draws S << n_b key indices from p by
 * stratified or systematic sampling and returns (1/S) * sum of the S sampled V rows:
 * a gather-and-add with no multiply per key, and an unbiased estimator of p.V.
 * SANTA_DENSE computes the exact p.V with the same score machinery, as the
 * like-for-like baseline (the pages compare against split-K decode kernels).
 *
 * Conventions for every entry point:
 *  - Device pointers are plain CUDA device addresses; ownership stays with the caller.
 *    The library allocates nothing.  Between calls it keeps only the caller's workspace
 *    contents, a per-device cache of device attributes and kernel settings, and the
 *    wait limit of santa_set_wait_limit (santa_decode_static adds its own static
 *    scratch).
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  All work is enqueued
 *    asynchronously on it; the library never synchronises the host, except in
 *    santa_device_status.
 *  - Return value: SANTA_OK (0) or a negative status; see santa_status_string.  Argument
 *    errors are detected on the host before anything is enqueued.
 */
#ifndef SANTA_H_
#define SANTA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define SANTA_OK 0
#define SANTA_ERR_INVALID_ARG (-1)  /* null pointer, bad shape, bad S or mode */
#define SANTA_ERR_MISALIGNED (-2)   /* a pointer is not 16-byte aligned */
#define SANTA_ERR_WORKSPACE (-3)    /* workspace missing or smaller than required */
#define SANTA_ERR_UNSUPPORTED (-4)  /* valid but outside the compiled limits (d, G, S, B) */
#define SANTA_ERR_CUDA (-5)         /* a CUDA launch or runtime call failed */
#define SANTA_ERR_DEVICE (-6)       /* the device reported an error (santa_device_status) */
#define SANTA_ERR_SCRATCH (-7)      /* santa_decode_static: the problem needs more scratch than
                                       SANTA_STATIC_SCRATCH_BYTES */

/* Value-stage modes ("stratified and systematic sampling", abstract; iid is plain
 * multinomial sampling, the estimator before variance reduction). */
#define SANTA_DENSE 0
#define SANTA_STRATIFIED 1
#define SANTA_SYSTEMATIC 2
#define SANTA_IID 3

/* Flag, or-ed into a sampling mode: gather each distinct V row once per group of query
 * heads that share a KV head (the G heads run as one thread-block cluster and exchange
 * their sample lists), instead of once per head.  It saves V traffic when S is large,
 * but ties each head's value stage to the slowest head of its group: at S = 256 on the
 * Llama-shaped batch it is slower, so it is off unless asked for.  It applies when
 * G > 1 and G * S <= 8192; otherwise it is ignored.  Results agree with the default
 * to fp32 rounding of the sums. */
#define SANTA_GROUP_DEDUP 0x100

/* Flag, or-ed into any mode: write `out` as bf16 [B, H_q, d] instead of fp32 (the caller
 * passes a bf16 buffer through the float* parameter).  Each element is the fp32 result
 * rounded once to the nearest bf16 (ties to even), so it equals the fp32 output rounded.
 * For a caller whose next layer consumes bf16 activations. */
#define SANTA_OUT_BF16 0x200

/* Flag, or-ed into any mode: Bernoulli qK^T ("Stochastic Sparse Attention for
 * Memory-Bound Inference", abstract, last sentences: stochastic ternary queries sparsify
 * the score stage).  Before scoring, every query head q is replaced by one ternary draw
 * q~ (santa_ternary_query, seeded by `seed`): q~_i = sign(q_i) * a with probability
 * |q_i| / a and 0 otherwise, a = max_i |q_i|, so E[q~] = q and every score is unbiased.
 * A score then depends only on the key features where q~_i != 0.  With this library's
 * row-major cache ([..., n_max, d], 256-byte rows for d = 128) those features are
 * spread over every row, so the call still reads whole rows: the flag changes the
 * arithmetic, not the bytes read.  The softmax of unbiased scores is itself not
 * unbiased, so the output estimates attention under the drawn query. */
#define SANTA_BERNOULLI_QK 0x400

/* Flag, or-ed into a sampling mode: always use the two launches of the score and value
 * stages.  By default a small problem runs as one launch of the single-pass kernel
 * instead: one thread-block cluster of up to 16 CTAs per (batch row, KV head), with the
 * softmax weights and CDF kept in shared memory and the value stage done inside the
 * cluster.  It applies when the B * H_kv clusters fit the GPU at once with at most 4096
 * keys per CTA and G * S <= 2048 (for example B = 1 up to about 48k keys, or B = 4 up to
 * 8k keys, at H_kv = 8 on a GB300); santa_call_info reports which one runs.  Indices
 * are the same either way; outputs differ only by the order of the fp32 additions of
 * the gather. */
#define SANTA_TWO_PASS 0x800

/* Device error bits (santa_device_status). */
#define SANTA_DEV_BAD_SEQLEN 1      /* some seq_lens[b] outside [0, n_max]; treated as 0 */
#define SANTA_DEV_TIMEOUT 2         /* a bounded wait on a shared-memory barrier gave up */

/* Problem shape.  scale = 0 selects 1/sqrt(d) rounded to fp32. */
typedef struct {
    int32_t B;      /* batch rows, 1..1024 */
    int32_t H_q;    /* query heads */
    int32_t H_kv;   /* KV heads; G = H_q / H_kv must be 1, 2, 4 or 8 */
    int32_t d;      /* head dimension: 64 or 128 */
    int32_t n_max;  /* KV-cache capacity per (b, h_kv), 1..524288; B * H_kv * n_max < 2^31
                     * (cache rows are addressed with 32-bit tensor-copy coordinates) */
    float scale;    /* score scale */
} santa_shape;

/*
 * santa_workspace_size -- bytes of device workspace santa_decode needs for this shape,
 * S and mode.  Pure host computation.
 * Returns SANTA_OK, SANTA_ERR_INVALID_ARG or SANTA_ERR_UNSUPPORTED.
 */
int santa_workspace_size(const santa_shape *shape, int32_t S, int32_t mode, size_t *bytes);

/*
 * santa_workspace_init -- zero the workspace's control block (counters and the device
 * error word) on `stream`.  Call once after allocating a workspace; every completed
 * santa_decode leaves the counters at zero again.  Call it again after an error.
 */
int santa_workspace_init(void *workspace, size_t workspace_bytes, void *stream);

/*
 * santa_decode -- one decode step of SANTA attention (or dense attention).
 *
 *  q         device bf16 [B, H_q, d], contiguous
 *  k_cache   device bf16 [B, H_kv, n_max, d], contiguous; keys j >= seq_lens[b] unused
 *  v_cache   device bf16 [B, H_kv, n_max, d], contiguous
 *  seq_lens  device int32 [B], each in [0, n_max]; out-of-range values are treated as 0
 *            and set SANTA_DEV_BAD_SEQLEN in the device error word
 *  S         samples per (b, h): 1..4096 (ignored for SANTA_DENSE)
 *  mode      SANTA_DENSE, SANTA_STRATIFIED, SANTA_SYSTEMATIC or SANTA_IID, optionally
 *            or-ed with SANTA_GROUP_DEDUP, SANTA_OUT_BF16, SANTA_BERNOULLI_QK and
 *            SANTA_TWO_PASS
 *  seed      Philox4x64-10 key word 0 (ignored for SANTA_DENSE, except for the ternary
 *            query draws of SANTA_BERNOULLI_QK)
 *  out       device fp32 [B, H_q, d] (bf16 with SANTA_OUT_BF16); n_b = 0 gives zeros
 *  idx_out   device int32 [B, H_q, S] or NULL: the sampled key indices of each (b, h),
 *            ascending, with repeats; n_b = 0 gives -1 (ignored for SANTA_DENSE)
 *  workspace device buffer of at least santa_workspace_size bytes, 256-byte aligned,
 *            initialised once by santa_workspace_init; one call at a time per workspace
 *
 * The sample points of (b, h) are t_s = (u + s) * r_S (systematic, one uniform u) or
 * t_s = (s + u_s) * r_S (stratified, one uniform per stratum), s = 0..S-1, with r_S the
 * fp64 value nearest 1/S; iid draws S uniforms and sorts them.  Uniforms are the top 32
 * bits of Philox4x64-10 words (Salmon et al., SC'11) times 2^-32, keyed (seed, 0) with
 * counter (block, b, h, 1 | 2 | 3 for stratified | systematic | iid).  Index
 * i_s = min{ j : C_j > t_s } on the CDF of p, i.e. point s selects key j when
 * t_s lies in [C_{j-1}, C_j).
 */
int santa_decode(const santa_shape *shape, const void *q, const void *k_cache,
                 const void *v_cache, const int32_t *seq_lens, int32_t S, int32_t mode,
                 uint64_t seed, float *out, int32_t *idx_out, void *workspace,
                 size_t workspace_bytes, void *stream);

/*
 * santa_call_info -- *launches = the kernel launches one santa_decode call with this
 * shape, S and mode enqueues on the current device (for sizing CUDA graphs and counting
 * work): 1 for the single-pass cluster kernel, else 2 (the score and value stages, or
 * the dense kernel and its merge), plus 1 for the ternary query draw of
 * SANTA_BERNOULLI_QK.  Reads device attributes; enqueues nothing.  Returns SANTA_OK or
 * the argument errors of santa_decode.
 */
int santa_call_info(const santa_shape *shape, int32_t S, int32_t mode, int32_t *launches);

/*
 * santa_set_wait_limit -- how long a kernel's pipeline wait (a thread waiting on a
 * shared-memory barrier for a copy, an MMA or another warp) may last before the kernel
 * gives up: it sets SANTA_DEV_TIMEOUT in the device error word, winds its roles down
 * (asynchronous copies and MMAs still in flight are always waited for, up to 2 s) and
 * exits, leaving the context usable.  Applies to calls made after it, process-wide.
 * limit_ns = 0 restores the default of 2 s.  A diagnostic: a short limit makes the
 * timeout path run (the library's tests do that), normal use never needs it.
 * Returns SANTA_OK.
 */
int santa_set_wait_limit(uint64_t limit_ns);

/*
 * santa_sample_points -- the fp64 sample points t [B, H_q, S] (device) that santa_decode
 * uses for (mode, seed), computed by the same device code.  For checking the sampler's
 * random stream against an independent implementation.  mode must be a sampling mode.
 */
int santa_sample_points(int32_t B, int32_t H_q, int32_t S, int32_t mode, uint64_t seed,
                        double *t_out, void *stream);

/*
 * santa_ternary_query -- the Bernoulli qK^T draws that santa_decode uses with
 * SANTA_BERNOULLI_QK for this seed, computed by the same device code (for checking the
 * draw against an independent implementation, and for callers that want q~ itself).
 *  q       device bf16 [B, H_q, d], contiguous, 16-byte aligned (d = 64 or 128)
 *  q_out   device bf16 [B, H_q, d]: q~_i in {-a, 0, +a}, a = max_i |q_i| of the head
 * The uniform of feature i of head (b, h) is the top 32 bits x of word i%4 of the
 * Philox4x64-10 block with counter (i/4, b, h, 4) and key (seed, 0); the feature keeps
 * its sign and becomes +-a when x * a < |q_i| * 2^32 (an exact comparison), else 0.
 */
int santa_ternary_query(int32_t B, int32_t H_q, int32_t d, const void *q, uint64_t seed, void *q_out,
                        void *stream);

/*
 * santa_device_status -- synchronise `stream`, read the device error word of the
 * workspace into *code (0 = no error; SANTA_DEV_* bits otherwise) and clear it.
 * workspace = NULL reads the error word of santa_decode_static's scratch on the current
 * device instead (*code = 0 when no static call has run on that device).
 * Returns SANTA_OK, or SANTA_ERR_DEVICE when *code != 0.
 */
int santa_device_status(void *workspace, int32_t *code, void *stream);

/*
 * santa_decode_static -- santa_decode without a caller-provided workspace.  (The pages
 * have no counterpart: this is an interface convenience of this library.)
 *
 * For callers that cannot allocate device memory themselves: code that runs where the
 * device allocator belongs to someone else (a serving runtime with its own fixed pool,
 * a plugin that may not call cudaMalloc), or on a path where an allocation would stall
 * or is not allowed.  The library keeps one scratch buffer of SANTA_STATIC_SCRATCH_BYTES
 * in a file-scope device array instead; every GPU that loads the library holds that
 * buffer until the process exits.  This call allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.
 *
 * Arguments and results are those of santa_decode, minus the workspace.  The caller
 * still passes q, the caches, seq_lens, out and idx_out.
 *
 *  - Size limit: the call returns SANTA_ERR_SCRATCH, before touching the device, when
 *    santa_workspace_size(shape, S, mode) exceeds SANTA_STATIC_SCRATCH_BYTES (for
 *    example B=1, H_q=32, d=128 fits up to about 110k keys).  Every other argument
 *    error is also returned before anything is enqueued.
 *  - Device errors (out-of-range seq_lens, a wait that gave up) set the scratch's own
 *    error word; santa_device_status(NULL, &code, stream) reads and clears it.  A call
 *    does not clear it, so it accumulates until read.
 *  - First call per device: it looks up the device address of the scratch array
 *    (cudaGetSymbolAddress, with that device current), which can load the library's
 *    device code.  Make that first call before any stream capture.
 *  - Every call on a device shares the one buffer.  Each call clears the work counters
 *    of the buffer's control block (an asynchronous memset on `stream`; the error word is
 *    left for santa_device_status) and overwrites the rest, so contents left by an
 *    earlier call, of any shape or mode, do no harm.  Calls that can overlap on the GPU
 *    (different streams without ordering, or several host threads) race on the buffer:
 *    order them on one stream.
 */
#define SANTA_STATIC_SCRATCH_BYTES ((size_t)16 << 20)
int santa_decode_static(const santa_shape *shape, const void *q, const void *k_cache,
                        const void *v_cache, const int32_t *seq_lens, int32_t S, int32_t mode,
                        uint64_t seed, float *out, int32_t *idx_out, void *stream);

/*
 * santa_timeline_buffer -- for reading where a call's time goes: in a library built with
 * -DSANTA_TIMELINE (libsanta_timeline.so; stochastic_sparse_kv_gb300/timeline.py builds
 * and reads it), later calls write %globaltimer stamps (ns) into buf, a device buffer of
 * at least 16 * 8 * (1024 + B * H_q) bytes: 16 stamps per row, one row per CTA of the score
 * or single-pass kernel (rows 0..1023) and per value-stage CTA (row 1024 + b * H_q + h).
 * Rows beyond `bytes` are not written.  buf = NULL stops it.  Errors: INVALID_ARG when
 * bytes hold fewer than 1024 rows, MISALIGNED when buf is not 8-byte aligned.  The normal
 * build has no stamps and returns SANTA_ERR_UNSUPPORTED.
 * Not for production use: the buffer is shared by every later call, process-wide.
 */
int santa_timeline_buffer(void *buf, size_t bytes);

/* santa_status_string -- static description of a status code. */
const char *santa_status_string(int status);

/* santa_version -- library version as 10000*major + 100*minor + patch. */
int santa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SANTA_H_ */
