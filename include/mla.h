/*
 * mla.h -- C ABI of the GB300 (sm_103a) weight-absorbed MLA decode library.
 *
 * One decode step of one attention layer, with the key up-projection folded
 * into the query and the value up-projection applied after the latent-space sum
 * ("MLA, dim by dim", section "MLA Decode": decode score order and decode value
 * order; "Why MLA and MTP Fight Each Other: Attention Through Arithmetic
 * Intensity", sections 3.1-3.3 and Appendix A):
 *
 *   mla_absorb_q     q_cat = [ q_nope . W_UK^T | q_rope ]          per head
 *   mla_decode_attn  o_lat, lse = softmax(scale * q_cat . [c_kv|k_rope]^T) . c_kv
 *                    over a contiguous or paged latent cache, split along the
 *                    history and merged with a log-sum-exp combine
 *   mla_out_proj     out = o_lat . W_UV                               per head
 *   mla_decode_step  the three above as one call, the kernels overlapping
 *   mla_decode_attn_sparse  the same attention over k listed cached tokens
 *                    per query token (sparse top-k decode)
 *   mla_cache_append c_kv = x . W_DKV of the new tokens, written with their
 *                    (already rotated) RoPE keys into the latent cache
 *   mla_prefill      prefill / chunked prefill of s_q new tokens: the absorbed path above
 *                    below the crossover S*, the expand form (per-head K, V
 *                    re-expanded from the latent, then per-head attention) at or
 *                    above it ("Why MLA and MTP Fight Each Other", 5.5-5.8)
 *   mla_naive_decode the decompress-then-attend form, a comparison point only
 *                    ("The MLA decode speedup hiding in your model card",
 *                    section "The naive form, written out")
 * The latent cache is bf16 or FP8 (E4M3 codes with one scale per cache), see
 * mla_cache.
 *
 * Conventions for every entry point:
 *  - Pointers named for tensors are DEVICE pointers owned by the caller; the
 *    library never allocates, frees or keeps them.  Scratch memory is the
 *    caller's `workspace`, sized by the matching *_workspace_size query.
 *  - Tensors are dense row-major in the layouts stated, bf16 unless stated.
 *    Every tensor base pointer and the workspace must be 16-byte aligned.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and never synchronise, except mla_read_status.
 *  - Every argument is checked on the host before anything is launched.  A
 *    non-zero return means nothing was launched, except MLA_ERR_CUDA, which
 *    reports a failed launch.  Problems only the device can see (a sequence
 *    length or block-table entry out of range, a bounded wait that ran out) are
 *    written to the status word at the start of the workspace; read it with
 *    mla_read_status.  A sequence with an invalid length gets zero outputs and
 *    lse = -inf; tokens on a page outside the pool are skipped.  Nothing faults
 *    and nothing reads outside the caller's buffers.
 *  - Dimensions: H >= 1, s_q >= 1, d_c a multiple of 64 up to 512, d_rope a
 *    multiple of 16 up to 64, d_nope and d_v multiples of 16 from 16 to 256,
 *    s_q * H <= 65536 (the prefill entry points: s_q <= 2^20 on the expand
 *    path), B and H at most 65535, B * s_q at most 65535 * 128, and on the
 *    expand path B * H at most 65535 (launch grid limits).  Other shapes return
 *    MLA_ERR_UNSUPPORTED.
 */
#ifndef MLA_H
#define MLA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

typedef enum {
    MLA_OK = 0,
    MLA_ERR_NULL = 1,        /* a required pointer is NULL */
    MLA_ERR_SHAPE = 2,       /* a size is negative or sizes disagree */
    MLA_ERR_SEQLEN = 3,      /* device: seq_lens[b] outside [s_q, capacity] */
    MLA_ERR_ALIGN = 4,       /* a pointer or stride is not 16-byte aligned */
    MLA_ERR_WORKSPACE = 5,   /* workspace smaller than the size query returned */
    MLA_ERR_UNSUPPORTED = 6, /* shape outside the supported envelope above */
    MLA_ERR_CUDA = 7,        /* a CUDA runtime call or launch failed */
    MLA_ERR_TIMEOUT = 8,     /* device: a bounded wait gave up (no hang, no fault) */
    MLA_ERR_PAGE = 9         /* device: a block-table entry outside [0, num_pages) */
} mla_status;

/* Problem sizes ("MLA, dim by dim", Notation and Preliminaries; the decoupled
 * RoPE width is Appendix A's d_s).  scale multiplies every score; callers use
 * 1/sqrt(d_nope + d_rope). */
typedef struct {
    int B;        /* sequences in the batch */
    int H;        /* query heads */
    int s_q;      /* new query tokens per sequence (1 = decode, >1 = verify) */
    int d_c;      /* latent width (c_kv), 512 for DeepSeek-V3 */
    int d_rope;   /* decoupled RoPE key width, 64 for DeepSeek-V3 */
    int d_nope;   /* per-head no-RoPE query/key width absorbed through W_UK */
    int d_v;      /* per-head value width produced by W_UV */
    float scale;  /* softmax scale */
} mla_dims;

/* Element formats of the latent cache (mla_cache.kv_dtype). */
typedef enum {
    MLA_KV_BF16 = 0,  /* bf16 values */
    MLA_KV_E4M3 = 1   /* OCP FP8 E4M3 codes (1 sign, 4 exponent bits with bias 7,
                         3 mantissa bits, no infinities, S.1111.111 = NaN); the
                         value is kv_scale * code */
} mla_kv_dtype;

/* The latent cache: one row [c_kv (d_c) | k_rope (d_rope)] per cached token,
 * shared by every head ("Decode attention intensity is fixed at the
 * query-to-KV head ratio...", "A strong answer": 512 + 64 = 576 values, 1,152 B
 * in bf16, 576 B with an FP8 latent).  seq_lens[b] counts the s_q new tokens,
 * which are already appended; query i (0-based) of sequence b sees tokens
 * j <= seq_lens[b] - s_q + i.
 * FP8 cache ("Decode attention intensity...", the FP8 row of the per-token
 * table: one byte per element doubles the arithmetic intensity to 484 FLOP/B;
 * the kernel dequantises on chip and computes in 16-bit): every element of
 * every row, RoPE key included, is an E4M3 code, with one fp32 scale for the
 * whole cache.  The attention kernels fold the scale into the query and the
 * final normalisation, so |q_cat| * scale * log2(e) * kv_scale must stay below
 * 65504 (the queries are carried in fp16).  d_c + d_rope must be a multiple of
 * 16 and seq_stride a multiple of 16.  mla_naive_decode takes bf16 caches only. */
typedef struct {
    const void *kv;          /* kv_dtype elements. block_table == NULL: contiguous, sequence b's
                                token j at kv + b*seq_stride + j*(d_c+d_rope).
                                Otherwise the pool [num_pages][page_size][d_c+d_rope]. */
    long long seq_stride;    /* contiguous: elements between sequences, a multiple of 8
                                (16 for FP8), >= capacity*(d_c+d_rope) */
    int capacity;            /* contiguous: tokens each sequence may hold */
    const int *block_table;  /* NULL => contiguous; else device int32 [B][max_pages]:
                                token j of sequence b lives in pool page
                                block_table[b*max_pages + j/page_size], row j%page_size */
    int max_pages;           /* paged: columns of block_table */
    int page_size;           /* paged: tokens per page, a multiple of 64 */
    int num_pages;           /* paged: pages in the pool (entries are checked against it) */
    const int *seq_lens;     /* device int32 [B] */
    int max_seq_len;         /* host upper bound of seq_lens used to plan the split;
                                0 means capacity (contiguous) or max_pages*page_size */
    int kv_dtype;            /* mla_kv_dtype; 0 (a zero-initialised descriptor) is bf16 */
    float kv_scale;          /* MLA_KV_E4M3: value = kv_scale * code (finite, > 0); ignored for bf16 */
} mla_cache;

/* Human-readable name of a status code (static storage, never NULL). */
MLA_API const char *mla_status_string(int status);

/* ABI version of this header: bumps when a signature or struct changes. */
MLA_API int mla_abi_version(void);

/* Absorb W_UK into the query and append the RoPE query ("MLA, dim by dim",
 * "MLA Decode", decode score order; "Why MLA and MTP Fight Each Other", 3.1):
 *   q_cat[b,i,h, 0:d_c]          = sum_n q_nope[b,i,h,n] * W_UK[h,c,n]  (fp32 accumulate)
 *   q_cat[b,i,h, d_c:d_c+d_rope] = q_rope[b,i,h,:]
 * q_nope [B][s_q][H][d_nope], q_rope [B][s_q][H][d_rope], w_uk [H][d_c][d_nope],
 * q_cat [B][s_q][H][d_c+d_rope]; all bf16, outputs rounded to nearest even. */
MLA_API int mla_absorb_q(const mla_dims *dims, const void *q_nope, const void *q_rope,
                         const void *w_uk, void *q_cat, void *stream);

/* num_splits value that asks mla_decode_attn (and mla_decode_step) for the
 * balanced plan: the batch's 64-token tiles, in batch order, dealt out in equal
 * contiguous ranges to every CTA-pair slot of the GPU, each 128-row block of the
 * queries its share of the slots (d_c > 256, bf16 cache, at most 4095
 * sequences, no more 128-row blocks than slots; otherwise MLA_ERR_UNSUPPORTED).
 * A sequence held by one range is written directly; the pieces of one cut
 * between ranges are merged in the same launch with the same log-sum-exp
 * combine as split pieces. */
#define MLA_SPLITS_BALANCED (-1)

/* Bytes of workspace mla_decode_attn needs for this problem and split count
 * (num_splits 0 = the library's choice, MLA_SPLITS_BALANCED the balanced plan).
 * Returns 0 for invalid or unsupported arguments. */
MLA_API size_t mla_decode_workspace_size(const mla_dims *dims, const mla_cache *cache,
                                         int num_splits);

/* Split count mla_decode_attn uses for num_splits == 0 (a function of the dims,
 * B and the max_seq_len hint only): the pieces per sequence, or, when the plan
 * splits only the sequences of a last, partly filled wave (see mla_decode_attn),
 * the pieces of those; when the choice is the balanced plan, the number of
 * equal tile ranges per 128-row block.  Returns 0 for invalid arguments. */
MLA_API int mla_decode_num_splits(const mla_dims *dims, const mla_cache *cache);

/* Latent-space attention of every head against the shared latent cache
 * ("MLA, dim by dim", "Why RoPE Gets in the Way", decoupled score, and "MLA
 * Decode", fused decode kernel; "Why MLA and MTP Fight Each Other", 3.2 and
 * section 4's fused streaming condition: each latent tile is read once and
 * serves both the score and the weighted sum):
 *   s_j   = scale * q_cat[b,i,h,:] . kv_row_j                (all d_c+d_rope columns)
 *   lse   = log sum_j exp(s_j)          over visible j      (natural log, fp32)
 *   o_lat = sum_j exp(s_j - lse) * kv_row_j[0:d_c]           (bf16, fp32 accumulate)
 * The history of each sequence is cut into num_splits pieces processed in
 * parallel, each keeping an online softmax; the pieces are merged with a
 * log-sum-exp combine.  q_cat [B][s_q][H][d_c+d_rope]; o_lat [B][s_q][H][d_c];
 * lse fp32 [B][s_q][H].  num_splits 0 = the library's choice, else 1..64: every
 * sequence in num_splits pieces; MLA_SPLITS_BALANCED the balanced plan (see
 * there).  The library's choice splits every sequence while the pieces fit one
 * wave of the GPU, or, with CTA pairs and a contiguous bf16 cache, takes the
 * balanced plan when, with every sequence at max_seq_len, it gives the busiest
 * pair at least 16 tiles fewer than the split plans below; with more 128-row work items than a
 * wave holds, it leaves them whole except those of a last, partly filled wave,
 * whose sequences (the last ones of the batch) are split to fill that wave; their
 * pieces are the last work items of the same grid.  With a bf16 cache, up to
 * 1024 sequences and more than one wave, the work order is longest sequence
 * first (ties by index), ranked on the device from seq_lens; the "last"
 * sequences above are then the shortest.  A sequence's result depends only on
 * how many pieces it runs in, not on its place in the order. */
MLA_API int mla_decode_attn(const mla_dims *dims, const void *q_cat, const mla_cache *cache,
                            void *o_lat, float *lse, void *workspace, size_t ws_bytes,
                            int num_splits, void *stream);

/* Project the latent-space output to each head's value width ("MLA, dim by dim",
 * "MLA Decode", decode value order; "Why MLA and MTP Fight Each Other", 3.2):
 *   out[b,i,h,v] = sum_c o_lat[b,i,h,c] * W_UV[h,c,v]   (fp32 accumulate, bf16 out)
 * o_lat [B][s_q][H][d_c], w_uv [H][d_c][d_v], out [B][s_q][H][d_v]. */
MLA_API int mla_out_proj(const mla_dims *dims, const void *o_lat, const void *w_uv,
                         void *out, void *stream);

/* Bytes of workspace mla_decode_attn_sparse needs for this problem, list length
 * and split count (0 = the library's choice).  Returns 0 for invalid arguments. */
MLA_API size_t mla_decode_sparse_workspace_size(const mla_dims *dims, const mla_cache *cache, int topk,
                                                int num_splits);

/* Sparse top-k decode ("Why MLA and MTP Fight Each Other", 6: a selector keeps
 * k cached tokens per query token; the latents are gathered by index and the
 * scoring and the weighted sum run over those only, so the cost is flat in the
 * history length).  Same inputs, outputs, workspace and status word as
 * mla_decode_attn, plus indices int32 [B][s_q][topk] (device): the token
 * positions each query token attends to, shared by all heads.  An entry takes
 * part when it names a token the query may see (0 <= j <= L_b - s_q + i) on a
 * page inside the pool; others (e.g. -1 padding, future tokens) are skipped,
 * and a query with no such entry gets o_lat = 0 and lse = -inf.  Each entry
 * counts once per listing.  The learned selector itself is not part of the
 * library.  Requires s_q == 1 or H a multiple of 128 (every 128-row block of
 * query rows belongs to one query token), and, for a contiguous cache,
 * seq_stride a multiple of d_c + d_rope; otherwise MLA_ERR_UNSUPPORTED. */
MLA_API int mla_decode_attn_sparse(const mla_dims *dims, const void *q_cat, const mla_cache *cache,
                                   const int *indices, int topk, void *o_lat, float *lse, void *workspace,
                                   size_t ws_bytes, int num_splits, void *stream);

/* Bytes of workspace mla_cache_append needs: the status word (256 B) and the
 * fp32 partial sums of the split down-projection (a few MB at DeepSeek-V3
 * widths).  Returns 0 for invalid arguments. */
MLA_API size_t mla_cache_append_workspace_size(const mla_dims *dims, int d_model);

/* The step before attention: compress the new tokens' hidden states into
 * latents and append them to the cache ("MLA, dim by dim", "MLA Decode": the
 * current token's x . W_DKV, of 2*d*d_c FLOPs, is appended to the latent cache;
 * "Why MLA and MTP Fight Each Other", 4.1: the history-independent part of a
 * decode step):
 *   c[b,i,:] = sum_k x[b,i,k] * W_DKV[k,:]     (fp32 accumulate, bf16 in the cache)
 * and row L_b - s_q + i of sequence b (L_b = seq_lens[b], which already counts
 * the s_q new tokens) becomes [c[b,i,:] | k_rope[b,i,:]].  x [B][s_q][d_model],
 * w_dkv [d_model][d_c], k_rope [B][s_q][d_rope] (already rotated; the library
 * does no rotation).  The cache is described as for mla_decode_attn and its kv
 * buffer is WRITTEN (it must be writable device memory); only the new rows
 * change.  An FP8 cache receives the E4M3 code of value / kv_scale, rounded to
 * nearest even and saturated to +-448, for every element of the row.  d_model must be a multiple of 8.  A length outside [s_q, capacity]
 * (MLA_ERR_SEQLEN) or a block-table entry outside the pool (MLA_ERR_PAGE) is
 * recorded in the workspace's status word and that token's row is not
 * written.  The weight is streamed once, split along d_model over the GPU. */
MLA_API int mla_cache_append(const mla_dims *dims, int d_model, const void *x, const void *w_dkv,
                             const void *k_rope, const mla_cache *cache, void *workspace, size_t ws_bytes,
                             void *stream);

/* Bytes of workspace mla_naive_decode needs: the materialised per-head K and V
 * of every cached token plus the status word (with the tensor-core expansion,
 * rows [V_h | K_h | k_rope] of B*H*capacity*(d_v+d_nope+d_rope) bf16 and the
 * concatenated queries; otherwise B*H*capacity*(d_nope+d_v) bf16).  Returns 0
 * for invalid arguments, or when B*H exceeds 65535. */
MLA_API size_t mla_naive_workspace_size(const mla_dims *dims, const mla_cache *cache);

/* Decompress-then-attend, the comparison path ("The MLA decode speedup hiding
 * in your model card", "The naive form, written out"; "Decode attention
 * intensity...", the 33.6 MFLOP per cached token decompression): for every head
 * and every cached token, K = c_kv . W_UK[h] and V = c_kv . W_UV[h] are written
 * to the workspace, then standard attention runs with the RoPE key appended:
 *   s_j = scale * (q_nope . K_j + q_rope . k_rope_j),  out = sum_j softmax(s)_j V_j.
 * Same tensors as the absorbed path; out [B][s_q][H][d_v] bf16, lse fp32 [B][s_q][H].
 * Where the prefill expansion takes the shape (bf16 cache, d_v and d_nope multiples
 * of 64, d_v + d_nope <= 256, d_v + d_nope + d_rope <= 320) the decompression is
 * that tcgen05 GEMM and the attention runs per head on the tensor cores, the same
 * launches as mla_prefill_expand; other shapes use CUDA-core kernels.  B*H above
 * 65535 (one grid slice per sequence and head) returns MLA_ERR_UNSUPPORTED. */
MLA_API int mla_naive_decode(const mla_dims *dims, const void *q_nope, const void *q_rope,
                             const mla_cache *cache, const void *w_uk, const void *w_uv,
                             void *out, float *lse, void *workspace, size_t ws_bytes,
                             void *stream);

/* mla_decode_attn for callers that cannot allocate scratch memory.  The pages
 * have no counterpart of this entry point; it exists for hosts that hold only
 * their input and output buffers, such as a plain C or FFI caller with no
 * device allocator, or a serving loop whose device memory belongs to a
 * framework pool and where a cudaMalloc (which may synchronise the device) is
 * not allowed while decoding.
 * Same computation, arguments and outputs as mla_decode_attn, without the
 * workspace: the status word and the split partials live in one 32 MiB array
 * compiled into the library (a file-scope __device__ array; every GPU on which
 * the library's kernels are loaded holds it until the process exits).  Nothing
 * is allocated or freed by this call.
 *  - Every call looks the array's device address up (cudaGetSymbolAddress,
 *    with the device current); the first call on a device loads the library's
 *    module there, so make that first call before any stream capture.
 *  - num_splits 0 takes the library's split count (its partials stay near one
 *    wave of work items, about 20 MB, within the array); an explicit
 *    num_splits whose partials exceed 32 MiB returns MLA_ERR_WORKSPACE.
 *  - Every call shares the one array and overwrites it: calls that overlap on
 *    the GPU (other streams, other host threads, without ordering between them)
 *    race and corrupt each other's results.  Order them on one stream.
 *  - device_status (optional, device int32): receives this call's device status
 *    word (as mla_read_status would report it) once the call has run. */
MLA_API int mla_decode_attn_noalloc(const mla_dims *dims, const void *q_cat, const mla_cache *cache,
                                    void *o_lat, float *lse, int num_splits, int *device_status,
                                    void *stream);

/* Diagnostics (the pages have no counterpart): the bound, in nanoseconds, of
 * every wait for work inside the attention kernels launched from now on by this
 * process (mla_decode_attn, mla_decode_step, the sparse, prefill and no-alloc
 * entry points).  A wait that runs out records MLA_ERR_TIMEOUT in the status
 * word; the kernel then drains the copies and MMAs it has in flight (those waits
 * keep the default bound) and returns, outputs undefined.  0 restores the
 * default, 2 s.  For tests of the timeout path and for diagnosing a stalled GPU;
 * not for production use.  Always returns MLA_OK. */
MLA_API int mla_set_wait_limit_ns(unsigned long long ns);

/* One whole absorbed decode step: mla_absorb_q -> mla_decode_attn ->
 * mla_out_proj with one call, the same arguments and results (q_cat and o_lat
 * are the caller's intermediate buffers, the workspace is sized by
 * mla_decode_workspace_size).  The status word is reset first, then the three
 * kernels are launched back to back; the attention and out_proj grids are
 * launched programmatically (CUDA programmatic dependent launch), so each starts
 * while its predecessor runs -- the attention streaming its first cache tiles,
 * out_proj its W_UV tiles -- and reads the predecessor's output only once that
 * grid has completed. */
MLA_API int mla_decode_step(const mla_dims *dims, const void *q_nope, const void *q_rope, const mla_cache *cache,
                            const void *w_uk, const void *w_uv, void *q_cat, void *o_lat, void *out, float *lse,
                            void *workspace, size_t ws_bytes, int num_splits, void *stream);

/* Which path mla_prefill took. */
typedef enum { MLA_PATH_ABSORB = 0, MLA_PATH_EXPAND = 1 } mla_path;

/* The query count S* at which the absorbed and the expanded bracketings of one
 * layer cost the same FLOPs for a history of L cached tokens ("Why MLA and MTP
 * Fight Each Other", 5.3 and 5.6; H cancels):
 *   S* = L d_c (d_nope + d_v) / (d_c (d_nope + d_v) + L (2 d_c - d_nope - d_v)),
 * 128 at L = 512 rising to 171 at L = 128K for DeepSeek-V3 widths.  Host only;
 * returns 0 for invalid dims or L < 1. */
MLA_API double mla_prefill_crossover(const mla_dims *dims, long long L);

/* Bytes of workspace mla_prefill_expand needs: the status word, the queries
 * [q_nope | q_rope] (B*s_q*H*(d_nope+d_rope) bf16) and the expanded rows
 * (B*H*capacity*(d_v+d_nope+d_rope) bf16: 671 MB for one 8K-token sequence at
 * DeepSeek-V3 widths).  0 for invalid arguments or an unsupported shape. */
MLA_API size_t mla_prefill_expand_workspace_size(const mla_dims *dims, const mla_cache *cache);

/* Prefill in the expand form ("Why MLA and MTP Fight Each Other", 5.5: with
 * many query tokens the per-token expansion is amortised; "MLA, dim by dim",
 * MLA prefill: materialise K and V from the latent, then standard attention):
 *   K_h[j] = c_kv[j] . W_UK[h],  V_h[j] = c_kv[j] . W_UV[h]       for every cached j < L_b
 *   s_ij = scale * (q_nope[i,h] . K_h[j] + q_rope[i,h] . k_rope[j]),  j <= L_b - s_q + i
 *   out[b,i,h,:] = sum_j softmax_j(s_ij) V_h[j],  lse[b,i,h] = log sum_j exp(s_ij)
 * Inputs as mla_naive_decode (q_nope [B][s_q][H][d_nope], q_rope [B][s_q][H][d_rope],
 * W_UK [H][d_c][d_nope], W_UV [H][d_c][d_v], a bf16 cache); out bf16
 * [B][s_q][H][d_v], lse fp32 [B][s_q][H].  The same numbers as the absorbed path
 * (which equals it in exact arithmetic), computed with tensor-core GEMMs for the
 * expansion and per-head attention over 64-token tiles.  Requires d_v and
 * d_nope multiples of 64 with d_v + d_nope <= 256 and d_v + d_nope + d_rope <=
 * 320, and a bf16 cache; else MLA_ERR_UNSUPPORTED. */
MLA_API int mla_prefill_expand(const mla_dims *dims, const void *q_nope, const void *q_rope, const mla_cache *cache,
                               const void *w_uk, const void *w_uv, void *out, float *lse, void *workspace,
                               size_t ws_bytes, void *stream);

/* Bytes of workspace mla_prefill needs (enough for either path). */
MLA_API size_t mla_prefill_workspace_size(const mla_dims *dims, const mla_cache *cache);

/* Prefill or chunked prefill of s_q new tokens per sequence, dispatched on the
 * crossover ("Why MLA and MTP Fight Each Other", 5.6 and 5.8): with L the
 * longest history (cache->max_seq_len, else the capacity), s_q >= S*(L) takes
 * mla_prefill_expand, s_q below it (decode, verification) the absorbed path
 * mla_absorb_q -> mla_decode_attn -> mla_out_proj; shapes the expand form does
 * not support always take the absorbed path.  Same inputs and outputs as
 * mla_prefill_expand; *path (optional) receives the mla_path taken.  The
 * status word is at the start of the workspace for both paths. */
MLA_API int mla_prefill(const mla_dims *dims, const void *q_nope, const void *q_rope, const mla_cache *cache,
                        const void *w_uk, const void *w_uv, void *out, float *lse, void *workspace, size_t ws_bytes,
                        int *path, void *stream);

/* Wait for `stream`, then copy the device status word at the start of
 * `workspace` (written by the last mla_decode_attn / mla_naive_decode that used
 * it) into *status: MLA_OK, MLA_ERR_SEQLEN, MLA_ERR_PAGE or MLA_ERR_TIMEOUT.
 * Returns MLA_ERR_CUDA if the copy or the wait fails. */
MLA_API int mla_read_status(const void *workspace, int *status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H */
