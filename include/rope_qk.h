/*
 * rope_qk.h -- C ABI of the packed variable-length QK rotary position embedding
 * (RoPE) library for GB300 (sm_103a), librope_qk.so.
 *
 * The operation.  Q and K of one padding-free pack of samples are rotated in place in
 * one pass (unsloth.ai, "3x faster training with packing", section "Kernel Triton QK
 * RoPE fusionné avec packing"):
 *
 *     y = x*cos + rotate_half(x)*sin  ==  x*cos + (x @ R)*sin,  R = [[0, I], [-I, 0]]
 *
 * with the half-split pairing (element i pairs with element i + d/2 of the same head).
 * The backward is the same rotation with sin negated, dX = dY*cos + (dY @ R^T)*sin.
 * Positions restart at every packed-sample boundary (same page, section "Packing non
 * contaminé"): token t of sample s has position t - cu_seqlens[s].  Flat offsets
 * switch to 64-bit arithmetic when an element count reaches 2^31 (same page, section
 * "Indexage int64 pour les kernels Triton").  The rotary base theta is the model's
 * `rope_theta` (TRL "training beyond 1M tokens", YaRN section).
 *
 * Arithmetic, exactly (identical bits to a plain CPU evaluation of the same steps):
 *   w_j   = (float) pow(theta, -(2.0*j)/d)            binary64 on the host, j < d/2
 *   phi   = (float)pos * w_j                          one binary32 multiply
 *   c, s  = cos(phi), sin(phi) in binary64, each rounded once to binary32 (the kernels
 *           reach the same bits in binary32 double-float arithmetic where its rounding
 *           is certain, and evaluate in binary64 only for the rest; rope_cos_sin_eval)
 *   y_i     = bf16( (a*c) - (b*s) ),  y_{i+d/2} = bf16( (b*c) + (a*s) )
 *           every product and sum rounded to binary32, no fused multiply-add,
 *           one round-to-nearest-even to bf16; a = x_i, b = x_{i+d/2}.
 *
 * Layouts.  Q is bf16 [total_tokens, n_q_heads, head_dim], K is bf16
 * [total_tokens, n_kv_heads, head_dim], both row-major and contiguous.  cu_seqlens is
 * int32 [n_seqs + 1], non-decreasing, cu_seqlens[n_seqs] <= total_tokens.  A token
 * with no sample (t < cu_seqlens[0] or t >= cu_seqlens[n_seqs]) is outside the pack:
 * in place it is left untouched; out of place its rows are copied unchanged.
 *
 * Ownership.  Every pointer is owned by the caller.  Q, K, outputs, cu_seqlens,
 * position ids, seq_used, the cos/sin table and pos/err buffers are DEVICE pointers;
 * descriptors (rope_qk_desc, rope_cos_sin_cache, segment lists) are HOST memory read
 * during the call.  The library keeps no pointer after a call returns, allocates no
 * device memory, and never synchronises.  Calls are asynchronous on `stream` (a
 * cudaStream_t; NULL = the legacy default stream).
 *
 * Errors.  Every entry point returns ROPE_OK (0) or a negative rope_status.  Arguments
 * are checked on the host before anything is launched or copied; a rejected call
 * launches and copies nothing.  The values inside cu_seqlens are not read on the host
 * (that would need a synchronisation): rope_validate_cu_seqlens checks them on the
 * device.  With invalid values the kernels still stay inside the Q/K/cache bounds and
 * skip the tokens whose position cannot be derived.  No kernel traps, asserts or spins.
 */
#ifndef ROPE_QK_H
#define ROPE_QK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ROPE_QK_ABI_VERSION 5

typedef enum rope_status {
    ROPE_OK = 0,
    ROPE_ERR_NULL = -1,         /* a required pointer is NULL */
    ROPE_ERR_SHAPE = -2,        /* negative count, stride or offset; a head count < 1; a
                                   segment list not starting at row 0, not increasing or
                                   with a token offset beside it */
    ROPE_ERR_HEAD_DIM = -3,     /* head_dim not a multiple of 16 in [16, 256] */
    ROPE_ERR_ALIGN = -4,        /* a pointer not 16-byte aligned, a stride not a multiple of 8 */
    ROPE_ERR_OVERLAP = -5,      /* Q and K share elements, a view overlaps itself, or an
                                   output overlaps an input */
    ROPE_ERR_UNSUPPORTED = -6,  /* a global token index or cache row beyond 2^24 (positions
                                   are exact in binary32 only up to there); an unknown
                                   flag bit or a nonzero reserved field; segments with
                                   position ids; a host-call workspace below 8 tokens */
    ROPE_ERR_LAUNCH = -7,       /* the CUDA runtime refused a launch or copy */
    ROPE_ERR_THETA = -8,        /* theta or position_scale not finite and > 0 */
    ROPE_ERR_KIND = -9,         /* unknown activation kind (glu.h) */
    ROPE_ERR_WORKSPACE = -10,   /* one token's Q and K rows do not fit the static staging */
    ROPE_ERR_CACHE = -11        /* the cos/sin cache was built for another theta, head_dim,
                                   position_scale or device, or its descriptor was not
                                   written by rope_cos_sin_cache_build */
} rope_status;

/* Bits of rope_qk_desc.flags. */
#define ROPE_FLAG_POSITION_IDS_INT64 0x1   /* position_ids points to int64 values */

/* Bits of the word rope_validate_cu_seqlens writes. */
#define ROPE_CU_NEGATIVE_START   0x1   /* cu_seqlens[0] < 0 */
#define ROPE_CU_DECREASING       0x2   /* cu_seqlens[s+1] < cu_seqlens[s] for some s */
#define ROPE_CU_PAST_END         0x4   /* cu_seqlens[n_seqs] > total_tokens */
#define ROPE_CU_NONZERO_START    0x8   /* cu_seqlens[0] != 0 (allowed; tokens before it are outside) */

/*
 * A cos/sin cache: the (c, s) pairs of every position below `rows`, evaluated once by
 * rope_cos_sin_cache_build for one (theta, head_dim, position_scale), so that the
 * rotations read them instead of evaluating them (the pages take cos and sin as
 * precomputed inputs; unsloth.ai page, section "Kernel Triton QK RoPE fusionné avec
 * packing").  The rows are a function of theta alone (TRL "training beyond 1M
 * tokens", YaRN section: `rope_theta` must match the model), so the descriptor records
 * what they were built for and every call that reads them checks it.
 *
 * Only rope_cos_sin_cache_build writes this struct; treat it as read-only.  A call
 * rejects (ROPE_ERR_CACHE) a cache whose theta, head_dim or position_scale differs
 * from the call's, that was built on another device, or whose fields were changed
 * after the build (the `check` word no longer matches them).  The struct is host
 * memory owned by the caller and read during the call only; `data` is the device
 * table, owned by the caller, 16-byte aligned, float[rows][4][head_dim/16][4]: entry
 * [p][q][c] holds (c_j, s_j, c_{j+1}, s_{j+1}) of position p for j = 8c + 2q (chunk c
 * covers frequencies 8c..8c+7, the order in which the rotation kernel consumes them).
 */
typedef struct rope_cos_sin_cache {
    const float *data;             /* device table, rows * head_dim floats             */
    int64_t rows;                  /* positions 0 .. rows-1 (at most 2^24)             */
    int32_t head_dim;
    int32_t device;                /* CUDA device ordinal current at the build         */
    double theta;
    double position_scale;
    uint64_t check;                /* written by the build from the fields above       */
} rope_cos_sin_cache;

/*
 * Forward: rotate Q and K of every token of the pack (unsloth.ai page, section "Kernel
 * Triton QK RoPE fusionné avec packing"; positions per section "Packing non contaminé").
 *
 *   q, k            device bf16 [total_tokens, n_q_heads, head_dim] and
 *                   [total_tokens, n_kv_heads, head_dim]; 16-byte aligned; disjoint.
 *   cu_seqlens      device int32 [n_seqs + 1] sample offsets in the token stream.
 *   n_seqs          number of samples (>= 0; 0 means nothing is inside the pack).
 *   total_tokens    T, rows of Q and K (0 <= T <= 2^24, so that every position is an
 *                   exact binary32 integer).  T == 0 launches nothing, reads no
 *                   pointer and returns ROPE_OK (NULL pointers allowed).
 *   n_q_heads, n_kv_heads   >= 1 (grouped-query attention: any ratio).
 *   head_dim        d, a multiple of 16 in [16, 256].
 *   theta           rotary base (> 0, finite).
 *   in_place        nonzero: write the result over q and k (q_out/k_out ignored);
 *                   zero: write to q_out/k_out (same shapes, 16-byte aligned, disjoint
 *                   from q and k); q and k are then only read.
 *   cos_sin_cache   optional (NULL: none) cache built for the same theta and head_dim
 *                   with position_scale 1, on the current device.  Positions >= its
 *                   rows, and every position without a cache, are evaluated on the fly
 *                   with identical results.
 *   stream          cudaStream_t or NULL.
 */
int rope_qk_fwd(void *q, void *k, const int32_t *cu_seqlens, int32_t n_seqs,
                int64_t total_tokens, int32_t n_q_heads, int32_t n_kv_heads,
                int32_t head_dim, double theta, int32_t in_place,
                void *q_out, void *k_out, const rope_cos_sin_cache *cos_sin_cache,
                void *stream);

/*
 * Backward: q and k hold dL/dY for Q and K and receive dL/dX, the transpose rotation
 * (sin negated; unsloth.ai page, same section, the backward note with R^T).
 * Arguments exactly as rope_qk_fwd.
 */
int rope_qk_bwd(void *q, void *k, const int32_t *cu_seqlens, int32_t n_seqs,
                int64_t total_tokens, int32_t n_q_heads, int32_t n_kv_heads,
                int32_t head_dim, double theta, int32_t in_place,
                void *q_out, void *k_out, const rope_cos_sin_cache *cos_sin_cache,
                void *stream);

/*
 * General form: any strided Q/K views, explicit positions or a global token offset, a
 * linear position rescale, forward or backward, in place or out of place.
 *
 * Views.  Each of q, k, q_out, k_out is a bf16 [total_tokens, heads, head_dim] view with
 * head_dim contiguous and element strides for tokens and heads (multiples of 8, >= 0;
 * pointers 16-byte aligned; the view's span, (tokens - 1) * token stride + (heads - 1)
 * * head stride + head_dim, below 2^56 elements, else ROPE_ERR_SHAPE).  No two
 * (token, head) rows of one view may share an element (else ROPE_ERR_OVERLAP).  Q and
 * K must share no element: either their address
 * ranges are disjoint, or they step tokens by the same stride and each token's Q block
 * and K block are disjoint -- the Q and K slices of one fused QKV projection output,
 * e.g. qkv[T, Hq + 2*Hkv, d] with q = qkv[:, :Hq], k = qkv[:, Hq:Hq+Hkv], are accepted
 * and rotated in place without a copy (unsloth.ai page, "Kernel Triton QK RoPE
 * fusionné avec packing": no clones, no contiguous transposes).  q_out and k_out both
 * NULL = in place; else both set, disjoint from each other (same rule) and with address
 * ranges disjoint from q and k.
 *
 * Positions.  If position_ids is non-NULL (device int32 [total_tokens], the per-example
 * position ids a 1-D pack carries in databricks.com "Reducing Qwen training time 6x",
 * section on 1-D packing), row r has position position_ids[r]; a value outside
 * [0, 2^24) leaves the row out (in place: untouched; out of place: copied).  With
 * ROPE_FLAG_POSITION_IDS_INT64 in flags, position_ids points to int64 values instead
 * (8-byte aligned; the dtype of the position ids a Hugging Face collator builds), with
 * the same rule for values outside [0, 2^24).  Otherwise row r is token
 * token_offset + r of the stream cu_seqlens describes and its position
 * is derived as for rope_qk_fwd; token_offset lets a context-parallel shard holding
 * tokens [a, b) of a pack pass the whole pack's cu_seqlens with token_offset = a
 * (token_offset + total_tokens <= 2^24).
 *
 * Segments.  A context-parallel rank of the load-balanced layout (TRL "training beyond
 * 1M tokens", context-parallel section: the sequence cut into 2 * cp_size chunks, rank
 * r holding chunks r and 2 * cp_size - 1 - r) keeps rows that are not consecutive in
 * the pack.  With n_segments > 0 (at most ROPE_MAX_SEGMENTS), segments[i] says that
 * rows row_start[i] .. row_start[i+1] - 1 (the last segment: up to total_tokens - 1)
 * are tokens token_start[i], token_start[i] + 1, ... of cu_seqlens' stream, so one call
 * rotates all of a rank's shards.  segments is a HOST array read during the call;
 * segments[0].row_start == 0, row_start strictly increasing and below total_tokens,
 * token_start >= 0 and every segment's last token below 2^24 (else ROPE_ERR_SHAPE or
 * ROPE_ERR_UNSUPPORTED).  It needs cu_seqlens (not position_ids) and token_offset 0.
 *
 * seq_used.  Optional, with cu_seqlens: sample s uses only its first seq_used[s]
 * tokens; the rest of its rows (the padding of a padded batch laid out with uniform
 * cu_seqlens) are left out like tokens outside the pack.  Ignored with position_ids.
 *
 * position_scale.  Linear position rescale (> 0; 1.0 = none): every frequency is
 * divided by it in binary64 before the rounding to binary32, i.e. position p acts as
 * p / position_scale.  A cos/sin cache must have been built with the same theta,
 * head_dim and position_scale (else ROPE_ERR_CACHE).
 */
#define ROPE_MAX_SEGMENTS 16

typedef struct rope_qk_segment {
    int64_t row_start;             /* first row (of q and k) of the segment           */
    int64_t token_start;           /* its token index in cu_seqlens' stream           */
} rope_qk_segment;

typedef struct rope_qk_desc {
    void *q;                       /* bf16 view [total_tokens, n_q_heads, head_dim]  */
    int64_t q_stride_token;        /* elements between consecutive tokens             */
    int64_t q_stride_head;         /* elements between consecutive heads              */
    void *k;                       /* bf16 view [total_tokens, n_kv_heads, head_dim] */
    int64_t k_stride_token;
    int64_t k_stride_head;
    void *q_out;                   /* NULL (with k_out NULL): in place                */
    int64_t q_out_stride_token;
    int64_t q_out_stride_head;
    void *k_out;
    int64_t k_out_stride_token;
    int64_t k_out_stride_head;
    const int32_t *cu_seqlens;     /* device int32 [n_seqs + 1]; unused with position_ids */
    int32_t n_seqs;
    int32_t n_q_heads;
    int32_t n_kv_heads;
    int32_t head_dim;              /* multiple of 16 in [16, 256]                     */
    const int32_t *position_ids;   /* optional device int32 [total_tokens]            */
    int64_t total_tokens;
    int64_t token_offset;          /* >= 0; global index of row 0 in cu_seqlens' stream */
    double theta;
    double position_scale;         /* 1.0 = plain rotation                            */
    const rope_cos_sin_cache *cos_sin_cache;   /* optional (NULL: none)               */
    int32_t backward;              /* 0: rotation; nonzero: transpose (sin negated)   */
    int32_t flags;                 /* ROPE_FLAG_* bits, 0 for none; an unknown bit is
                                      ROPE_ERR_UNSUPPORTED                             */
    const int32_t *seq_used;       /* optional device int32 [n_seqs], with cu_seqlens */
    const rope_qk_segment *segments;   /* optional HOST array [n_segments]            */
    int32_t n_segments;            /* 0: no segments (row r is token token_offset + r) */
    int32_t reserved;              /* 0 */
} rope_qk_desc;

/* Apply the rotation a descriptor describes (asynchronous on `stream`). */
int rope_qk_apply(const rope_qk_desc *desc, void *stream);

/*
 * What rope_qk_apply would launch for `desc`, without launching it and without any
 * CUDA call: the rotation kernel's compile-time instance (head_dim 64, 96, 128 or 256,
 * or 0 for the generic one), whether it uses 64-bit element offsets (some view spans
 * 2^31 elements or more; unsloth.ai page, section "Indexage int64 pour les kernels
 * Triton"), how many 16-byte pair units each thread keeps in flight (4 for launches of
 * at least 32,768 tiles with 32-bit offsets, a compile-time head_dim and a cos/sin
 * cache; 3 for smaller such launches without seq_used whose tile holds at most 384
 * units, and for launches with 64-bit offsets, a compile-time head_dim and a cache but
 * no seq_used; 2 otherwise), and its grid: one CTA of `threads` threads per tile of
 * `tile_tokens` consecutive tokens.  Returns the
 * status rope_qk_apply's argument checks give (the cache's device is not checked);
 * grid == 0 when there is nothing to launch.
 */
typedef struct rope_qk_launch {
    int32_t head_dim_instance;
    int32_t long_index;
    int32_t grid;
    int32_t tile_tokens;
    int32_t threads;
    int32_t smem_bytes;            /* dynamic shared memory per CTA (cos/sin rows)    */
    int32_t unroll;                /* pair units in flight per thread                 */
} rope_qk_launch;

int rope_qk_launch_info(const rope_qk_desc *desc, rope_qk_launch *info);

/*
 * Host-buffer form of rope_qk_apply, for Q and K that live in host memory.  desc->q,
 * k, q_out, k_out are HOST pointers to contiguous bf16 [total_tokens, heads, head_dim]
 * (q_out, k_out both NULL: results go back into q and k).  Pinned memory makes the
 * copies asynchronous and overlapped; pageable memory works, with synchronous copies.
 * Every other field is as for rope_qk_apply (cu_seqlens, position_ids and the cache
 * are DEVICE pointers).
 *
 * workspace: DEVICE staging memory of workspace_bytes, 256-byte aligned, owned by the
 * caller.  It holds two slots of `chunk` tokens' Q and K rows, chunk =
 * workspace_bytes / (2 * (n_q_heads + n_kv_heads) * head_dim * 2) rounded down to a
 * multiple of 8 (ROPE_ERR_UNSUPPORTED below 8).  The pack is walked chunk by chunk:
 * the host-to-device copy of one chunk, the rotation of the previous one and the
 * device-to-host copy of the one before overlap, the copies on two streams the library
 * creates per device on first use and keeps.  Each chunk is rotated with its global
 * token offset (or its slice of position_ids, or of the segment list), so the result
 * is that of one rotation of the whole pack.
 *
 * `stream` runs the rotations and then waits for the last copy to the host: once it
 * reaches that point, the host outputs are complete.  The host buffers and the
 * workspace must stay untouched until then.  Enqueueing is serialised by a lock.
 * Every argument is checked for the whole pack before the first copy is queued, so a
 * rejected call copies and launches nothing; only a failure of the CUDA runtime itself
 * (ROPE_ERR_LAUNCH) can come after copies were queued, and `stream` is then still
 * ordered after all of them.
 */
int rope_qk_host(const rope_qk_desc *desc, void *workspace, int64_t workspace_bytes, void *stream);

/*
 * rope_qk_host for callers that cannot allocate device memory.  The source pages
 * describe nothing like it; it exists for code that may not call cudaMalloc/cudaFree
 * or any allocating routine: a plugin or embedding runtime that hands out no device
 * allocator, a process whose device memory is entirely reserved by another allocator
 * (a framework's caching allocator), or a loop that must not add the implicit
 * synchronisation of cudaMalloc/cudaFree.  It takes no workspace: it stages the chunks
 * in a 32 MiB device array that is part of this library (every GPU that loads the
 * library keeps those 32 MiB until the process exits), and it allocates nothing.
 *
 * Same descriptor and results as rope_qk_host.  Chunks of up to
 * 32 MiB / ((n_q_heads + n_kv_heads) * head_dim * 2) tokens are copied in, rotated and
 * copied out one after the other, all on `stream` (no overlap of copies and rotation).
 * A shape whose single token does not fit is rejected with ROPE_ERR_WORKSPACE.  As for
 * rope_qk_host, every argument is checked for the whole pack before the first copy: a
 * rejected call leaves the host buffers untouched.
 *
 * The first call on a device looks up the array's device address (once per device,
 * that device current); make that first call before any stream capture.  Every call
 * uses the same array, which keeps whatever the last call left in it (nothing in it
 * needs to start at zero).  Calls that overlap on the GPU (on different streams
 * without ordering between them, or from several host threads at once) race on it:
 * order them.
 */
int rope_qk_host_static(const rope_qk_desc *desc, void *stream);

/*
 * Build a cos/sin cache: fill `data` with (c, s) of every position p < rows and
 * frequency j < head_dim/2 by the arithmetic above, the frequencies divided by
 * position_scale (> 0, finite; 1.0 for the plain rotation) before their rounding to
 * binary32 (the linear rescale of TRL "training beyond 1M tokens", YaRN section: with
 * factor 4, position 100,000 is read as 25,000), and write the descriptor `cache` that
 * the rotations take.  data: device float[rows * head_dim], 16-byte aligned, owned by
 * the caller (rope_cos_sin_cache_bytes).  rows <= 2^24; build it once per (theta,
 * head_dim, position_scale) with rows >= the longest sample, on the device that runs
 * the rotations (the current device); every layer and step can reuse it.  The
 * descriptor is written only when the fill was queued (ROPE_OK); it is usable on
 * `stream`, or after it, once the fill has run.
 */
int rope_cos_sin_cache_build(rope_cos_sin_cache *cache, float *data, int64_t rows,
                             int32_t head_dim, double theta, double position_scale,
                             void *stream);

/* Bytes a cache of `cache_rows` rows takes (cache_rows * head_dim * 4), or -1. */
int64_t rope_cos_sin_cache_bytes(int64_t cache_rows, int32_t head_dim);

/*
 * Positions exactly as the rotation kernels derive them from cu_seqlens (section
 * "Packing non contaminé": reset at each boundary): pos_out[t] = t - cu_seqlens[s]
 * for the last s with cu_seqlens[s] <= t, or -1 for a token outside the pack.
 * pos_out: device int32 [total_tokens].
 */
int rope_qk_positions(const int32_t *cu_seqlens, int32_t n_seqs, int64_t total_tokens,
                      int32_t *pos_out, void *stream);

/*
 * Check the values of cu_seqlens on the device.  Writes to the device word *err_word
 * the OR of the ROPE_CU_* bits that apply (0 = valid).  The word is cleared on
 * `stream` first; read it after the stream reaches this point.
 */
int rope_validate_cu_seqlens(const int32_t *cu_seqlens, int32_t n_seqs, int64_t total_tokens,
                             int32_t *err_word, void *stream);

/*
 * cos and sin of n binary32 angles (device arrays phi, cos_out, sin_out), the values the
 * rotation uses for phi = pos * w_j: the binary64 cosine and sine rounded once to
 * binary32.  mode ROPE_COS_SIN_AS_ROTATION evaluates them as the rotation kernels and
 * the cache build do (binary32 double-float arithmetic where its rounding is certain,
 * binary64 for the rest); ROPE_COS_SIN_BINARY64 in binary64 only;
 * ROPE_COS_SIN_BINARY32_ONLY in binary32 only, writing NaN where that evaluation leaves
 * the rounding to binary64.  The first two give identical bits for every angle; the
 * third shows how often the binary64 path is taken.  ROPE_ERR_KIND for another mode.
 */
#define ROPE_COS_SIN_AS_ROTATION 0
#define ROPE_COS_SIN_BINARY64 1
#define ROPE_COS_SIN_BINARY32_ONLY 2

int rope_cos_sin_eval(const float *phi, float *cos_out, float *sin_out, int64_t n, int32_t mode,
                      void *stream);

/* Host-side inverse frequencies w_j = (float)(pow(theta, -(2.0*j)/d) / position_scale)
 * (head_dim/2 floats) exactly as the kernels use them; position_scale is 1.0 for the
 * plain rotation.  w_out: HOST float[head_dim/2].  No CUDA call. */
int rope_qk_inv_freq(double theta, int32_t head_dim, double position_scale, float *w_out);

/* Static text for a status code. */
const char *rope_strerror(int status);

/* ROPE_QK_ABI_VERSION of the loaded library. */
int rope_qk_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ROPE_QK_H */
