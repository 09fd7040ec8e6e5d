/*
 * attn.h -- C ABI of the GB300 (sm_103a) fused attention forward.
 *
 * The library computes, for every query row, the forward pass of softmax
 * attention with a fixed set of score and mask modifications:
 *
 *     s_ij  = scale * <q_i, k_j>                       (scale first)
 *     s_ij += -m_h * (qpos_i - j)                     (ALiBi, optional)
 *     s_ij  = cap * tanh(s_ij / cap)                  (soft-capping, optional)
 *     O_i   = sum_{j visible} softmax_j(s_i.) * v_j
 *     LSE_i = ln sum_{j visible} exp(s_ij)             (natural log)
 *
 * The score matrix never reaches device memory: tiles of K and V stream
 * through shared memory and the softmax is computed online (running max and
 * running sum, with the output rescaled only when the max grows by more
 * than a threshold).
 *
 * Sources:
 *  - "FlashAttention-4 explained" (theneuron.ai), section "Enter Tri Dao and
 *    FlashAttention": keep tiles in on-chip memory, write no intermediate
 *    score matrix to HBM, exact result;
 *  - same page, section "FlashAttention-4: Built for Blackwell", "Forward
 *    pass fixes": ping-pong over two query tiles, exponentials split between
 *    the hardware unit and a polynomial, conditional rescaling;
 *  - same page, section "PyTorch Gets the Upgrade Too": sliding window,
 *    ALiBi, soft-capping as custom variants;
 *  - "PyTorch 2.5 Introduces FlexAttention and TorchDynamo C++ Runtime",
 *    section "What Happened?": sliding window, document packing, prefix
 *    masking; body: modifications are functions of (q_idx, k_idx) and no
 *    quadratic score matrix is materialised.
 *
 * Conventions for every entry point:
 *  - All tensors are dense, row-major and contiguous:
 *      q   [B][H][S_q][D]     bf16
 *      k,v [B][H_kv][S_k][D]  bf16
 *      out [B][H][S_q][D]     bf16 (round to nearest even)
 *      lse [B][H][S_q]        fp32
 *    Query head h reads key/value head h / (H / H_kv) (grouped-query
 *    attention, consecutive grouping).
 *  - Device pointers are pointers to device memory of the current CUDA
 *    device; the caller owns every buffer passed in.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream).  Argument errors are detected on the host
 *    before anything is enqueued and leave device memory untouched.
 *  - Errors detected on the device (a prebuilt block mask that does not
 *    match the call, a pipeline wait that ran out of time) never trap: the
 *    kernel records a code in a per-device status word and returns.  Read it
 *    with attn_get_device_status().
 */
#ifndef ATTN_GB300_ATTN_H
#define ATTN_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so the header needs no CUDA
 * headers. */
typedef struct CUstream_st *attn_stream_t;

typedef enum attn_status {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,  /* bad pointer, size, flag or descriptor     */
    ATTN_ERR_UNSUPPORTED = 2,  /* valid request the library does not serve  */
    ATTN_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed          */
    ATTN_ERR_TIMEOUT = 4,      /* a device pipeline wait ran out of time     */
    ATTN_ERR_DEVICE_CHECK = 5  /* a device-side consistency check failed     */
} attn_status;

/* Descriptor layout version.  Version 2 appended the block-map and
 * relative-position-bias fields; a version-1 descriptor (without them) is
 * still accepted and reads as if those fields were zero. */
#define ATTN_MOD_DESC_VERSION 2u

/* Mask modifications.  Enabled masks are combined with AND.  With
 * qpos = i + q_offset for query row i and kpos = j for key j:
 *   CAUSAL     key visible iff kpos <= qpos
 *   WINDOW     key visible iff qpos - window < kpos <= qpos
 *              (so a row sees at most `window` keys, itself included)
 *   DOCUMENT   key visible iff doc_ids[b][i] == doc_ids[b][j]
 *              (packed sequences; requires S_q == S_k)
 *   PREFIX_LM  key visible iff kpos <= qpos or kpos < prefix_len[b]
 *              (already causal outside the prefix; combining it with
 *              CAUSAL gives plain causal)
 *   BLOCKS     key visible iff blocks[b'][i / 128][j / 128] != 0, a user
 *              block map over 128 x 128 tiles (b' = b when blocks_batched,
 *              else 0): block-sparse attention
 * A row that sees no key gets O = 0 and LSE = -inf. */
enum {
    ATTN_MASK_CAUSAL = 1u,
    ATTN_MASK_WINDOW = 2u,
    ATTN_MASK_DOCUMENT = 4u,
    ATTN_MASK_PREFIX_LM = 8u,
    ATTN_MASK_BLOCKS = 16u
};

/* Edge of a block-map tile, in query rows and keys. */
#define ATTN_BLOCK 128

/* Score modifications, applied after the scale in this order:
 *   ALIBI    s += -m_h * (qpos - kpos), with m_h = alibi_slopes[h] or, when
 *            alibi_slopes is NULL, m_h = 2^(-8 (h + 1) / H) for 0-based
 *            query head h;
 *   RELBIAS  s += rel_bias[h][clamp(kpos - qpos, -R, R) + R] with
 *            R = rel_max: a learned relative-position bias table per head;
 *   SOFTCAP  s = softcap * tanh(s / softcap). */
enum {
    ATTN_SCORE_ALIBI = 1u,
    ATTN_SCORE_SOFTCAP = 2u,
    ATTN_SCORE_RELBIAS = 4u
};

/* Fixed descriptor of score and mask modifications (replaces a JIT).
 * Zero-initialise it, set `version`, then the fields the flags use. */
typedef struct attn_mod_desc {
    uint32_t version;          /* 1 or ATTN_MOD_DESC_VERSION (2), else
                                  INVALID_ARG                                */
    uint32_t mask_flags;       /* ATTN_MASK_* bits                           */
    uint32_t score_flags;      /* ATTN_SCORE_* bits                          */
    int32_t window;            /* WINDOW: > 0                                */
    int32_t q_offset;          /* qpos = i + q_offset; |q_offset| < 2^30.
                                  0 aligns masks top-left, S_k - S_q
                                  bottom-right                               */
    float softcap;             /* SOFTCAP: finite, > 0                       */
    const int32_t *doc_ids;    /* DOCUMENT: device, [B][S_k]                 */
    const int32_t *prefix_len; /* PREFIX_LM: device, [B]                     */
    const float *alibi_slopes; /* ALIBI: device [H] or NULL for the default  */
    const void *block_mask;    /* optional device buffer filled by
                                  attn_build_block_mask() for exactly these
                                  B, S_q, S_k, mask fields and mask arrays;
                                  NULL: the library builds one internally    */
    size_t block_mask_bytes;   /* size of block_mask                         */
    /* version >= 2 */
    const uint8_t *blocks;     /* BLOCKS: device, [B or 1][ceil(S_q/128)]
                                  [ceil(S_k/128)], nonzero = tile may be
                                  visible                                    */
    int32_t blocks_batched;    /* BLOCKS: 1 = one map per batch entry,
                                  0 = one map for all                        */
    int32_t rel_max;           /* RELBIAS: R >= 0, R < 2^30                  */
    const float *rel_bias;     /* RELBIAS: device, [H][2 R + 1]              */
} attn_mod_desc;

/*
 * attn_fwd -- fused attention forward: O and LSE for every query row.
 *
 * Defined by: "FlashAttention-4 explained" (theneuron.ai), sections "What Is
 * Attention, and Why Is It Expensive?" and "Enter Tri Dao and
 * FlashAttention" (the exact softmax attention, tiled so no score matrix is
 * written), and "FlashAttention-4: Built for Blackwell" (the forward
 * pipeline).  Modifications: see attn_mod_desc.
 *
 *  q, k, v  device, bf16, layouts above, 16-byte aligned
 *  out      device, bf16 [B][H][S_q][D], 16-byte aligned, must not overlap
 *           the inputs; 32-byte aligned is faster (each row is written in
 *           32-byte stores, else in 16-byte ones; the results are the same)
 *  lse      device, fp32 [B][H][S_q], 4-byte aligned, or NULL to skip it
 *  B, H, H_kv, S_q, S_k  > 0, H % H_kv == 0, S_q and S_k < 2^30
 *  D        head dimension, 64 or 128 (others: ATTN_ERR_UNSUPPORTED)
 *  scale    finite and > 0 (usually 1/sqrt(D))
 *  mod      NULL for plain (dense, unmodified) attention
 *  stream   stream the work is enqueued on
 *
 * Returns ATTN_OK once the work is enqueued, ATTN_ERR_INVALID_ARG /
 * ATTN_ERR_UNSUPPORTED without enqueuing anything, or ATTN_ERR_CUDA when a
 * launch failed.  When mod->block_mask is NULL the block mask is built on
 * the stream into a library-owned per-device buffer (allocated or grown on
 * first need): calls that rely on it must not run concurrently on
 * different streams of one device.
 */
attn_status attn_fwd(const void *q, const void *k, const void *v, void *out,
                     float *lse, int B, int H, int H_kv, int S_q, int S_k,
                     int D, float scale, const attn_mod_desc *mod,
                     attn_stream_t stream);

/*
 * attn_block_mask_bytes -- size of the block-mask buffer for a problem.
 *
 * Defined by: the tile classification of the block-sparse forward (tiles
 * that no visible pair touches are skipped; the mask is evaluated only on
 * tiles that are partly visible) -- "PyTorch 2.5 Introduces FlexAttention
 * and TorchDynamo C++ Runtime", body text on masks that never materialise
 * the quadratic matrix.
 *
 * Returns 0 when the arguments are invalid (same rules as attn_fwd).
 */
size_t attn_block_mask_bytes(int B, int H, int S_q, int S_k,
                             const attn_mod_desc *mod);

/*
 * attn_build_block_mask -- classify every (128-row query tile, 128-key tile)
 * pair as EMPTY (no visible pair), FULL (every pair visible: no per-element
 * mask needed) or PARTIAL, compact the non-empty key tiles of every pair of
 * query tiles, and order the work by descending tile count.
 *
 * Defined by: as attn_block_mask_bytes.
 *
 *  B, H, S_q, S_k, mod  as in attn_fwd (mod->block_mask is ignored)
 *  dst      device buffer of at least attn_block_mask_bytes() bytes,
 *           16-byte aligned, owned by the caller; its contents are opaque
 *  bytes    size of dst
 *
 * The result stays valid while B, S_q, S_k, the mask fields of `mod` and the
 * contents of doc_ids / prefix_len stay the same; pass it to attn_fwd in
 * mod->block_mask to skip the rebuild.  Asynchronous on `stream`.
 */
attn_status attn_build_block_mask(int B, int H, int S_q, int S_k,
                                  const attn_mod_desc *mod, void *dst,
                                  size_t bytes, attn_stream_t stream);

/*
 * attn_block_mask_stats -- read back, synchronously, the tile counts of a
 * block mask built by attn_build_block_mask: the number of computed
 * (query-tile pair, key tile) entries and of FULL / PARTIAL / EMPTY
 * (query tile, key tile) classes among them.  Any pointer may be NULL.
 * Synchronises `stream`.  Intended for tests and measurements.
 */
attn_status attn_block_mask_stats(const void *block_mask, size_t bytes,
                                  attn_stream_t stream, int64_t *n_entries,
                                  int64_t *n_full, int64_t *n_partial,
                                  int64_t *n_empty);

/*
 * attn_get_device_status -- synchronise `stream`, then return and clear the
 * status word that the kernels of the current device write instead of
 * trapping (ATTN_OK when nothing was recorded).
 */
attn_status attn_get_device_status(attn_stream_t stream);

/*
 * attn_fwd_noalloc -- attn_fwd for callers that must not allocate device
 * memory on the call path.
 *
 * No counterpart on the pages this library follows: this entry point exists
 * for callers, not for the method.  attn_fwd allocates a status word and a
 * block-mask buffer on first use (and grows the buffer, with a device-wide
 * synchronisation, when a larger problem arrives).  Callers that cannot do
 * that -- code running while a stream is captured into a CUDA graph,
 * runtimes that own all device memory through their own pool or budget,
 * latency-critical paths that cannot take the synchronisation of
 * cudaMalloc/cudaFree -- use this entry point instead.  It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 * Arguments, layouts, results and errors are those of attn_fwd, except:
 *  - mod->block_mask must be NULL (the block mask is always built by the
 *    call), else ATTN_ERR_INVALID_ARG;
 *  - its scratch (status word and block mask) lives in one fixed array of
 *    ATTN_NOALLOC_SCRATCH_BYTES bytes in the library, which every GPU that
 *    loads the library holds until the process exits.  The first
 *    ATTN_NOALLOC_STATUS_BYTES hold the status word, the rest the block
 *    mask.  A problem is served when attn_block_mask_bytes() for the same
 *    arguments, asked under the same options, is at most
 *    ATTN_NOALLOC_SCRATCH_BYTES - ATTN_NOALLOC_STATUS_BYTES; anything
 *    larger is rejected with ATTN_ERR_UNSUPPORTED before anything is
 *    enqueued.  For orientation: the tile lists take 4 * nP * nK bytes per
 *    mask batch (nK = ceil(S_k / 128), nP = ceil(S_q / 256), or
 *    ceil(S_q / 512) under the CTA-pair option), and document masks add
 *    8 * S_k + 8 * nK + 4 * ceil(S_k / 1024) bytes per batch entry; a mask
 *    batch is the whole batch for document, prefix-LM and per-batch block
 *    maps, else one.  So causal S_q = S_k = 131072 needs 2 MiB, and
 *    documents over B = 3 sequences of 131072 tokens need about 9 MiB and
 *    are rejected;
 *  - the first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress, which may load the library's device code);
 *    make that first call before any stream capture begins;
 *  - every call on a device shares the one array and leaves its contents
 *    behind (each call clears the status word and rewrites the block mask
 *    before its forward kernel runs), so calls whose work overlaps on the
 *    GPU -- on different streams, or from different threads without
 *    ordering -- race and may produce wrong results;
 *  - device-side failures (a pipeline wait that ran out of time, a failed
 *    device check) are recorded in that array's status word, which
 *    attn_get_noalloc_status reads and clears (attn_get_device_status reads
 *    attn_fwd's word, not this one); the outputs of such a call are
 *    unspecified.  Each call clears the word before its kernels run, so it
 *    reports on the latest attn_fwd_noalloc call on the device.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)
#define ATTN_NOALLOC_STATUS_BYTES 256u
attn_status attn_fwd_noalloc(const void *q, const void *k, const void *v,
                             void *out, float *lse, int B, int H, int H_kv,
                             int S_q, int S_k, int D, float scale,
                             const attn_mod_desc *mod, attn_stream_t stream);

/*
 * attn_get_noalloc_status -- synchronise `stream`, then return and clear the
 * status word of attn_fwd_noalloc's fixed array on the current device
 * (ATTN_OK when the latest attn_fwd_noalloc call recorded nothing).  Like
 * that entry point it has no counterpart on the pages and allocates no
 * device memory: it copies the word out of the array and, when it is set,
 * zeroes it, both synchronously.  Not for use while `stream` is captured.
 */
attn_status attn_get_noalloc_status(attn_stream_t stream);

/*
 * attn_fwd_host -- attn_fwd on tensors in host memory.  The pages define
 * only the on-device computation; this entry point has no counterpart there.
 * It is the same forward (same kernels, same results bit for bit) with the
 * copies in and out made by the library:
 *
 *  q, k, v, out, lse   host memory, same layouts and sizes as attn_fwd; no
 *                      alignment needed; page-locked memory (cudaHostAlloc,
 *                      torch pin_memory) for full copy speed, pageable
 *                      memory works but its copies are synchronous
 *  mod                 as for attn_fwd, except that doc_ids, prefix_len,
 *                      alibi_slopes, blocks and rel_bias are host memory too
 *                      and block_mask must be NULL (else
 *                      ATTN_ERR_INVALID_ARG)
 *  stream              the call starts after the work already enqueued on
 *                      `stream`, and work enqueued on `stream` afterwards
 *                      starts once O and LSE are in host memory
 *
 * Asynchronous like cudaMemcpyAsync: the inputs must stay unchanged and the
 * outputs unread until `stream` has passed the call (synchronise it).  The
 * copies and the kernels run on three streams owned by the library (per
 * device), alternating between two device buffers of the library, so the
 * input copy of one call overlaps the compute of the previous one and the
 * output copy of the one before.  Those buffers are allocated on first use,
 * grown (after the calls that use them finish) when a larger problem
 * arrives, and kept until the process exits.  Calls on one device are
 * serialised by a lock.  Errors as for attn_fwd; device-side failures are
 * read with attn_get_device_status(stream).
 */
attn_status attn_fwd_host(const void *q, const void *k, const void *v,
                          void *out, float *lse, int B, int H, int H_kv,
                          int S_q, int S_k, int D, float scale,
                          const attn_mod_desc *mod, attn_stream_t stream);

/*
 * attn_bwd -- gradients of attn_fwd: dQ, dK and dV for a given dO.
 *
 * Defined by the forward's definition and the chain rule; "FlashAttention-4
 * explained", section "FlashAttention-4: Built for Blackwell", names the
 * backward pass as the step after the forward and prints no formula:
 *   P = softmax of the modified, masked scores (recomputed from the forward's
 *   LSE), dP = dO V^T, dS = P * (dP - rowsum(dO * O)) * (derivative of the
 *   score mod), dQ = scale * dS K, dK = scale * dS^T Q, dV = P^T dO; dK and dV
 *   of a K/V head sum over the query heads that share it.
 *
 *  q, k, v, out, lse   the forward's inputs and outputs (out and lse exactly
 *                      as attn_fwd wrote them for these q, k, v, scale, mod)
 *  dout                device, bf16 [B][H][S_q][D], the gradient of out
 *  dq                  device, bf16 [B][H][S_q][D]
 *  dk, dv              device, bf16 [B][H_kv][S_k][D]
 *  others              as attn_fwd; mod->block_mask must be NULL (the masks
 *                      are rebuilt, forward and transposed, into a
 *                      library-owned per-device buffer)
 *
 * All tensors 16-byte aligned (lse 4-byte), outputs overlapping nothing;
 * dq, dk and dv 32-byte aligned take 32-byte stores (same results).
 * Deterministic: no atomics, every output row is written once.  Errors as
 * for attn_fwd; device-side failures are read with attn_get_device_status.
 * Calls that share the library's buffer must not run concurrently on
 * different streams of one device.
 */
attn_status attn_bwd(const void *q, const void *k, const void *v,
                     const void *out, const float *lse, const void *dout,
                     void *dq, void *dk, void *dv, int B, int H, int H_kv,
                     int S_q, int S_k, int D, float scale,
                     const attn_mod_desc *mod, attn_stream_t stream);

/* Tuning options.  Process-wide; set them before enqueuing work. */
typedef enum attn_option {
    /* Rescale O only when the running row max grows by more than this many
     * units of log2 (default 8; 0 gives the textbook online softmax).  The
     * result is mathematically independent of it.  "FlashAttention-4
     * explained", "Forward pass fixes", "Conditional rescaling". */
    ATTN_OPT_RESCALE_THRESHOLD = 1,
    /* 1: classify every non-empty tile as PARTIAL (the per-element mask runs
     * everywhere).  Must not change any output bit.  Default 0. */
    ATTN_OPT_FORCE_PARTIAL = 2,
    /* Upper bound, in milliseconds, on any single pipeline wait inside a
     * kernel before it gives up with ATTN_ERR_TIMEOUT (default 2000). */
    ATTN_OPT_WAIT_BUDGET_MS = 3,
    /* Persistent CTAs to launch; 0 (default) = one per SM. */
    ATTN_OPT_NUM_CTAS = 4,
    /* Fraction of the softmax exponentials evaluated with an FMA polynomial
     * instead of the hardware exp2 unit, in [0, 1] (default 0), applied in
     * steps of 1/8 of each row's 128 columns.  Relative error of the
     * polynomial is below 1e-4, far under the bf16 rounding of P.
     * "FlashAttention-4 explained", "Forward pass fixes",
     * "Software-emulated exponentials". */
    ATTN_OPT_EXP_POLY_FRACTION = 5,
    /* Test hook, default 0.  Nonzero: the forward kernel's MMA issuers wait
     * on a barrier that nothing ever arrives on, so their bounded wait runs
     * out after ATTN_OPT_WAIT_BUDGET_MS: the kernel records ATTN_ERR_TIMEOUT,
     * lets its in-flight copies land, frees Tensor Memory and returns, with
     * unspecified outputs.  In attn_bwd, 1 does the same to the dQ kernel's
     * MMA issuer and 2 to the dK/dV kernel's.  Values other than 0, 1 and
     * 2 are rejected.  Lets tests exercise the timeout paths without any
     * real fault or hang. */
    ATTN_OPT_DEBUG_STALL = 6,
    /* 1: forwards with D = 128 run on CTA pairs (thread-block clusters of
     * two): the two CTAs of a pair issue their score and output products
     * as single 256-row tcgen05 MMAs (cta_group::2), each CTA staging its
     * own 128 query rows and half of every key / value tile ("FlashAttention-4
     * explained", "TMEM and 2-CTA MMA", "2-CTA MMA mode").  Block masks built
     * while the option is 1 group four query tiles per entry instead of two
     * (attn_block_mask_bytes changes accordingly); a block mask must be used
     * under the setting it was built with, else the forward records
     * ATTN_ERR_DEVICE_CHECK.  Forwards with D = 64 use the one-CTA kernel
     * on such masks.  Both settings meet the same accuracy bounds against
     * exact attention.  Default 0. */
    ATTN_OPT_CTA_PAIR = 7
} attn_option;

attn_status attn_set_option(attn_option opt, double value);
attn_status attn_get_option(attn_option opt, double *value);

/* Human-readable name of a status code (static storage). */
const char *attn_status_string(attn_status status);

/* ABI version of this header: ATTN_ABI_VERSION. */
#define ATTN_ABI_VERSION 1
int attn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_ATTN_H */
