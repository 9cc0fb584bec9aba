// C ABI of the MLA decode library: argument checks, workspace layout, launches.
// Declarations and the contract live in include/mla.h.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>

#include "common.cuh"
#include "launch.h"

namespace {

constexpr int kAbiVersion = 2;
constexpr int kMaxSplits = 64;
// Bound of the attention kernels' waits for work, set by mla_set_wait_limit_ns
// (0: the kernels' default).
std::atomic<unsigned long long> g_wait_ns{0};

// SMs of the current device (split planning only), looked up once per device
int num_sms() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 152;
    if (dev < 64 && cached[dev] > 0) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 2) n = 152;
    if (dev < 64) cached[dev] = n;
    return n;
}
constexpr size_t kStatusBytes = 256;  // status word + padding at the workspace start
constexpr int kMaxOrdered = 1024;     // longest-first work order up to this many sequences
constexpr int kMaxGridZ = 65535;      // largest third grid dimension of a launch
constexpr int kMaxPersistB = 4095;    // balanced plan: the kernel keeps the batch's tile prefix in 16 KB
constexpr long long kBalancedMinGain = 16;  // tiles a pair the library's choice wants the balanced plan to save

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Shapes every entry point supports (the absorbed kernels add a row limit).
int check_shape(const mla_dims *d) {
    if (!d) return MLA_ERR_NULL;
    if (d->B < 0 || d->H < 1 || d->s_q < 1 || d->d_c < 1 || d->d_rope < 0 || d->d_nope < 1 || d->d_v < 1)
        return MLA_ERR_SHAPE;
    if (d->d_c % 64 || d->d_c > 512) return MLA_ERR_UNSUPPORTED;
    if (d->d_rope % 16 || d->d_rope > 64) return MLA_ERR_UNSUPPORTED;
    if (d->d_nope % 16 || d->d_nope > 256) return MLA_ERR_UNSUPPORTED;
    if (d->d_v % 16 || d->d_v > 256) return MLA_ERR_UNSUPPORTED;
    if (d->s_q > (1 << 20)) return MLA_ERR_UNSUPPORTED;
    // grid limits: heads index the projections' third grid dimension, sequences
    // the attention's (65535 at most in either)
    if (d->H > kMaxGridZ || d->B > kMaxGridZ) return MLA_ERR_UNSUPPORTED;
    if ((long long)d->B * d->s_q > (long long)kMaxGridZ * 128) return MLA_ERR_UNSUPPORTED;  // 128-token GEMM tiles
    if (!(d->scale == d->scale)) return MLA_ERR_SHAPE;  // NaN scale
    return MLA_OK;
}

int check_dims(const mla_dims *d) {
    const int s = check_shape(d);
    if (s) return s;
    if ((long long)d->s_q * d->H > 65536) return MLA_ERR_UNSUPPORTED;
    return MLA_OK;
}

// Capacity (tokens per sequence) of a checked cache.
long long cache_capacity(const mla_cache *c) {
    return c->block_table ? (long long)c->max_pages * c->page_size : (long long)c->capacity;
}

int check_cache(const mla_dims *d, const mla_cache *c) {  // d already passed check_shape
    if (!c) return MLA_ERR_NULL;
    if (d->B == 0) return MLA_OK;
    if (!c->kv || !c->seq_lens) return MLA_ERR_NULL;
    if (!aligned16(c->kv) || ((uintptr_t)c->seq_lens & 3u)) return MLA_ERR_ALIGN;
    const long long W = d->d_c + d->d_rope;
    if (c->kv_dtype != MLA_KV_BF16 && c->kv_dtype != MLA_KV_E4M3) return MLA_ERR_UNSUPPORTED;
    if (c->kv_dtype == MLA_KV_E4M3) {
        // a positive, finite scale; rows and sequence strides of whole 16-byte units
        if (!(c->kv_scale > 0.f) || c->kv_scale > 3.0e38f) return MLA_ERR_SHAPE;
        if (W % 16 || (!c->block_table && c->seq_stride % 16)) return MLA_ERR_ALIGN;
    }
    if (c->block_table) {
        if ((uintptr_t)c->block_table & 3u) return MLA_ERR_ALIGN;
        if (c->max_pages < 1 || c->page_size < 1 || c->num_pages < 1) return MLA_ERR_SHAPE;
        if (c->page_size % 64) return MLA_ERR_UNSUPPORTED;
    } else {
        if (c->capacity < 1) return MLA_ERR_SHAPE;
        if (c->seq_stride < (long long)c->capacity * W) return MLA_ERR_SHAPE;
        if (c->seq_stride % 8) return MLA_ERR_ALIGN;
    }
    if (c->max_seq_len < 0 || c->max_seq_len > cache_capacity(c)) return MLA_ERR_SHAPE;
    if (cache_capacity(c) > (1ll << 30)) return MLA_ERR_UNSUPPORTED;
    return MLA_OK;
}

// maxL: the longest token range one work item streams (sequence length, or the
// sparse list length)
int plan_splits_len(const mla_dims *d, long long maxL, int requested) {
    if (requested > 0) return requested;
    long long tiles = (maxL + 63) / 64;
    long long row_blocks = ((long long)d->s_q * d->H + 127) / 128;
    long long units = (long long)d->B * row_blocks;  // work items before splitting
    if (units <= 0) return 1;
    // One work item runs on a pair of SMs when d_c > 256, else on one SM.  Split
    // the history only while the pieces still fit in one wave of the GPU (more
    // pieces would add a partial wave and the cross-split merge), and keep every
    // piece at least 8 tiles long.
    const long long slots = d->d_c > 256 ? num_sms() / 2 : num_sms();
    long long want = slots / units;
    long long cap = tiles / 8;
    if (want > cap) want = cap;
    if (want < 1) want = 1;
    if (want > kMaxSplits) want = kMaxSplits;
    return (int)want;
}

// Sparse decode: the index list must be shared by all rows of a 128-row block
// (one query token per block, or a single query token), and the contiguous
// cache must be a stack of whole rows (gathered through a 2-D view).
int check_sparse(const mla_dims *d, const mla_cache *c, const int *indices, int topk) {
    if (topk < 1) return MLA_ERR_SHAPE;
    if (d->s_q > 1 && d->H % 128) return MLA_ERR_UNSUPPORTED;
    if (!c->block_table && c->seq_stride % (d->d_c + d->d_rope)) return MLA_ERR_UNSUPPORTED;
    if (d->B > 0 && !indices) return MLA_ERR_NULL;
    if ((uintptr_t)indices & 3u) return MLA_ERR_ALIGN;
    return MLA_OK;
}

size_t attn_workspace_bytes(const mla_dims *d, int splits) {
    if (splits <= 1) return kStatusBytes;
    size_t rows = (size_t)d->B * splits * d->s_q * d->H;
    // per row: (m, l) of each CTA half, then the fp32 accumulator
    return kStatusBytes + round_up(rows * 4 * sizeof(float), 256) + rows * (size_t)d->d_c * sizeof(float);
}

cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

// ---------------------------------------------------------------- prefill (expand form)
// Expanded row width: [V_h (d_v) | K_h (d_nope) | k_rope (d_rope)].
long long expanded_width(const mla_dims *d) { return (long long)d->d_v + d->d_nope + d->d_rope; }

int check_expand(const mla_dims *d, const mla_cache *c) {
    if (c->kv_dtype != MLA_KV_BF16) return MLA_ERR_UNSUPPORTED;
    if (d->d_v % 64 || d->d_nope % 64 || d->d_v + d->d_nope > 256 || expanded_width(d) > 320) return MLA_ERR_UNSUPPORTED;
    if ((long long)d->B * d->H > kMaxGridZ) return MLA_ERR_UNSUPPORTED;  // one work item per (sequence, head)
    return MLA_OK;
}

size_t expand_q_bytes(const mla_dims *d) {
    return round_up((size_t)d->B * d->s_q * d->H * (d->d_nope + d->d_rope) * 2, 256);
}

size_t expand_workspace_bytes(const mla_dims *d, const mla_cache *c) {
    return kStatusBytes + expand_q_bytes(d) +
           (size_t)d->B * d->H * (size_t)cache_capacity(c) * (size_t)expanded_width(d) * 2;
}

// Work plan of a dense decode attention: sequences [0, B - b_tail) run in
// `splits` pieces each, the last b_tail sequences in tail_splits pieces.
struct DecodePlan {
    int splits;
    int b_tail;
    int tail_splits;
    bool lpt;  // longest sequences first (several waves of whole sequences)
    // balanced plan (attn_persist.cu): groups of CTA pairs, each an equal range of
    // the batch's tiles; 0 for the plans above
    int persist_groups;
};

// The balanced plan (attn_persist.cu, CTA pairs, bf16 cache): every pair slot gets
// the same share of the batch's tiles whatever the lengths and the batch size.  The
// groups launched per 128-row block are capped by the tiles the max_seq_len hint
// allows (at least 8 a range); the device deals out the tiles it finds.
bool balanced_supported(const mla_dims *d, const mla_cache *c) {
    const long long maxL = c->max_seq_len > 0 ? c->max_seq_len : cache_capacity(c);
    const long long row_blocks = ((long long)d->s_q * d->H + 127) / 128;
    const long long max_tiles = (long long)d->B * ((maxL + 63) / 64);
    return d->d_c > 256 && c->kv_dtype == MLA_KV_BF16 && d->B <= kMaxPersistB && row_blocks <= num_sms() / 2 &&
           max_tiles < (1ll << 31);
}
DecodePlan balanced_plan(const mla_dims *d, const mla_cache *c) {
    const long long maxL = c->max_seq_len > 0 ? c->max_seq_len : cache_capacity(c);
    const long long row_blocks = ((long long)d->s_q * d->H + 127) / 128;
    const long long max_tiles = (long long)d->B * ((maxL + 63) / 64);
    return DecodePlan{1, 0, 1, false, mla::persist_groups((int)(num_sms() / 2 / row_blocks), max_tiles)};
}

// The library's plan (requested == 0), else `requested` pieces for every
// sequence (MLA_SPLITS_BALANCED: the balanced plan, which the caller checked is
// supported).  In one wave of work items, the history is split to fill the wave.
// With CTA pairs and a bf16 cache the balanced plan replaces the split plans when,
// with every sequence at max_seq_len, it gives the busiest pair slot at least
// kBalancedMinGain tiles fewer (the balanced kernel's own costs, a later first
// score, the hand-overs and the in-launch merge, come to about that many tiles;
// measured: 128 -> 108 tiles a pair wins 8 %, 64 -> 54 loses 6 %, spec's 448 ->
// 432 wins 3 %), on a contiguous cache.  When the work items fill more than one wave of clusters and
// the last wave is only partly used, the sequences of that last wave are split
// over the whole of it instead: the ones before run unsplit and write their rows
// directly, and only the tail's pieces are merged.  The wave arithmetic assumes
// sequences of about equal length (only max_seq_len is known here); with ragged
// lengths the tail's pieces simply start as slots free.  Over several waves of
// whole sequences the work order is longest first (the kernel ranks the lengths,
// which only the device knows; up to 1024 sequences, bf16 caches), so that a long
// sequence does not start in the last wave; with equal lengths the order is the
// batch order.
// The split plans alone (requested > 0: that many pieces; 0: the choice above
// without the balanced plan).
DecodePlan split_plan(const mla_dims *d, const mla_cache *c, int requested) {
    const long long maxL = c->max_seq_len > 0 ? c->max_seq_len : cache_capacity(c);
    const long long tiles = (maxL + 63) / 64;
    const long long row_blocks = ((long long)d->s_q * d->H + 127) / 128;
    const long long units = (long long)d->B * row_blocks;
    const long long slots = d->d_c > 256 ? num_sms() / 2 : num_sms();
    DecodePlan pl{plan_splits_len(d, maxL, requested), 0, 1, false, 0};
    pl.lpt = pl.splits == 1 && units > slots && d->B <= kMaxOrdered && c->kv_dtype == MLA_KV_BF16;
    if (requested > 0) return pl;
    const long long rem = units % slots;
    if (units <= slots || pl.splits > 1 || rem == 0) return pl;
    const long long b_tail = (rem + row_blocks - 1) / row_blocks;
    if (b_tail >= d->B) return pl;
    long long k = slots / (b_tail * row_blocks);
    const long long cap = tiles / 8;  // pieces of at least 8 tiles
    if (k > cap) k = cap;
    if (k > kMaxSplits) k = kMaxSplits;
    if (k < 2 || d->B - b_tail + b_tail * k > kMaxGridZ) return pl;
    pl.b_tail = (int)b_tail;
    pl.tail_splits = (int)k;
    return pl;
}

DecodePlan plan_decode(const mla_dims *d, const mla_cache *c, int requested) {
    if (requested == MLA_SPLITS_BALANCED) return balanced_plan(d, c);
    const DecodePlan pl = split_plan(d, c, requested);
    const long long row_blocks = ((long long)d->s_q * d->H + 127) / 128;
    const long long units = (long long)d->B * row_blocks;
    const long long slots = d->d_c > 256 ? num_sms() / 2 : num_sms();
    // only with a contiguous cache: on a paged one the balanced kernel measured
    // slower at equal tiles (ragged paged 766 against 700 us, dsv3 paged 118.7
    // against 111.1 contiguous)
    if (requested != 0 || units == 0 || c->block_table != nullptr || !balanced_supported(d, c)) return pl;
    const long long maxL = c->max_seq_len > 0 ? c->max_seq_len : cache_capacity(c);
    const long long tiles = (maxL + 63) / 64;
    // tiles the busiest slot streams, every sequence at max_seq_len
    long long per_split;
    if (units <= slots) {
        per_split = (tiles + pl.splits - 1) / pl.splits;
    } else {
        per_split = (units / slots) * tiles;
        if (units % slots) per_split += pl.b_tail ? (tiles + pl.tail_splits - 1) / pl.tail_splits : tiles;
    }
    const DecodePlan bp = balanced_plan(d, c);
    const long long per_balanced = (d->B * tiles + bp.persist_groups - 1) / bp.persist_groups;
    return per_split - per_balanced >= kBalancedMinGain ? bp : pl;
}

// Bytes of the work order (sequence of each work-order position) after the status word.
size_t order_bytes(const mla_dims *d, const DecodePlan &pl) {
    return pl.lpt ? round_up((size_t)d->B * sizeof(int), 256) : 0;
}

// Status word, the work order, then the split pieces' partials (only the tail's,
// if the plan has one).
// Balanced plan's workspace after the status block: the merge counters ([B][row
// blocks][2], zeroed with the status word), the tile prefix (B + 1 ints), the
// (m, l) hand-over ([pair][2 CTAs][2 item parities][128 rows][3]), the pieces'
// (m, l) ([pair][2 slots][128 rows][2 halves][2]) and rows (bf16, [pair][2
// slots][128 rows][d_c]).
struct PersistLayout {
    size_t counters, prefix, ml, part_ml, part_o, total;
};
PersistLayout persist_layout(const mla_dims *d, const DecodePlan &pl) {
    const size_t n_rb = ((size_t)d->s_q * d->H + 127) / 128;
    const size_t pairs = (size_t)pl.persist_groups * n_rb;
    PersistLayout l;
    l.counters = kStatusBytes;
    l.prefix = l.counters + round_up((size_t)d->B * n_rb * 2 * sizeof(int), 256);
    l.ml = l.prefix + round_up(((size_t)d->B + 1) * sizeof(int), 256);
    l.part_ml = l.ml + round_up(pairs * 2 * 2 * 128 * 3 * sizeof(float), 256);
    l.part_o = l.part_ml + round_up(pairs * 2 * 128 * 2 * 2 * sizeof(float), 256);
    l.total = l.part_o + pairs * 2 * 128 * (size_t)d->d_c * 2;
    return l;
}

// Bytes at the workspace start that every call zeroes first: the status word,
// and the balanced plan's merge counters.
size_t plan_zero_bytes(const mla_dims *d, const DecodePlan &pl) {
    return pl.persist_groups > 0 ? persist_layout(d, pl).prefix : sizeof(int);
}

size_t plan_workspace_bytes(const mla_dims *d, const DecodePlan &pl) {
    if (pl.persist_groups > 0) return persist_layout(d, pl).total;
    if (pl.b_tail == 0) return attn_workspace_bytes(d, pl.splits) + order_bytes(d, pl);
    mla_dims t = *d;
    t.B = pl.b_tail;
    return attn_workspace_bytes(&t, pl.tail_splits) + order_bytes(d, pl);
}

// absorbed prefill: the attention's own workspace first (so that the status word
// sits at the start, as for every entry point), then q_cat and o_lat
size_t absorbed_workspace_bytes(const mla_dims *d, size_t attn_ws) {
    const size_t rows = (size_t)d->B * d->s_q * d->H;
    return round_up(attn_ws, 256) + round_up(rows * (d->d_c + d->d_rope) * 2, 256) + rows * d->d_c * 2;
}

// Points p's split partials into the workspace (past `skip` bytes of work order),
// for nb sequences in `splits` pieces.
void set_partials(mla::AttnParams &p, const mla_dims *d, int nb, int splits, void *workspace, size_t skip = 0) {
    p.num_splits = splits;
    if (splits > 1) {
        const size_t rows = (size_t)nb * splits * d->s_q * d->H;
        char *base = (char *)workspace + kStatusBytes + skip;
        p.part_ml = (float *)base;
        p.part_acc = (float *)(base + round_up(rows * 4 * sizeof(float), 256));
    }
}

// The attention launch of plan pl (and the merge of split pieces); p carries the
// whole batch.  A tail is one grid with the rest: its pieces are the grid's last
// work items, so the hardware starts them as the whole sequences before them
// leave the SMs, and only they are merged.
cudaError_t launch_decode_plan(const mla_dims *d, const DecodePlan &pl, mla::AttnParams p, void *workspace,
                               cudaStream_t st) {
    if (pl.persist_groups > 0) {
        const PersistLayout l = persist_layout(d, pl);
        char *base = (char *)workspace;
        p.counters = (int *)(base + l.counters);
        p.prefix = (int *)(base + l.prefix);
        p.ml = (float *)(base + l.ml);
        p.part_ml = (float *)(base + l.part_ml);
        p.part_acc = (float *)(base + l.part_o);
        p.num_splits = 1;
        p.persist_groups = pl.persist_groups;
        return mla::launch_attn_persist(p, st);
    }
    const size_t ob = order_bytes(d, pl);
    if (pl.lpt) {
        p.lpt = 1;
        p.order = (int *)((char *)workspace + kStatusBytes);
    }
    if (pl.b_tail == 0) {
        set_partials(p, d, d->B, pl.splits, workspace, ob);
        return mla::launch_attn_tc(p, st);
    }
    set_partials(p, d, pl.b_tail, pl.tail_splits, workspace, ob);
    p.num_splits = 1;
    p.tail_b0 = d->B - pl.b_tail;
    p.tail_splits = pl.tail_splits;
    return mla::launch_attn_tc(p, st);
}

mla::AttnParams make_params(const mla_dims *d, const mla_cache *c) {
    mla::AttnParams p;
    memset(&p, 0, sizeof p);
    p.B = d->B; p.H = d->H; p.s_q = d->s_q; p.d_c = d->d_c; p.d_rope = d->d_rope; p.scale = d->scale;
    p.kv = c->kv;
    p.kv_fp8 = c->kv_dtype == MLA_KV_E4M3;
    p.kv_scale = p.kv_fp8 ? c->kv_scale : 1.f;
    p.seq_stride = c->seq_stride;
    p.capacity = (int)cache_capacity(c);
    p.block_table = c->block_table;
    p.max_pages = c->max_pages; p.page_size = c->page_size; p.num_pages = c->num_pages;
    p.seq_lens = c->seq_lens;
    p.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    return p;
}

// The expand form ("Why MLA and MTP Fight Each Other", 5.3/5.5: materialise K_h,
// V_h, then attend per head): expansion GEMM into the workspace, query concat,
// per-head attention.  Arguments already checked; the status word is reset.
int run_expand(const mla_dims *dims, const void *q_nope, const void *q_rope, const mla_cache *cache,
               const void *w_uk, const void *w_uv, void *out, float *lse, void *workspace, cudaStream_t st) {
    char *base = (char *)workspace + kStatusBytes;
    void *q_exp = base;
    void *expd = base + expand_q_bytes(dims);
    mla::AttnParams p = make_params(dims, cache);
    p.status = (int *)workspace;
    cudaError_t e = mla::launch_expand_kv(p, dims->d_nope, dims->d_v, w_uk, w_uv, expd, st);
    if (e == cudaSuccess) e = mla::launch_concat_q(*dims, q_nope, q_rope, q_exp, st);
    if (e != cudaSuccess) return MLA_ERR_CUDA;
    // per-head attention: (sequence, head) pairs over the expanded rows
    mla::AttnParams a = p;
    a.B = dims->B * dims->H;
    a.H = 1;
    a.d_c = dims->d_v;
    a.d_rope = dims->d_nope + dims->d_rope;
    a.kv = expd;
    a.block_table = nullptr;
    a.capacity = (int)cache_capacity(cache);
    a.seq_stride = (long long)a.capacity * expanded_width(dims);
    a.q_cat = (const __nv_bfloat16 *)q_exp;
    a.q_w = dims->d_nope + dims->d_rope;
    a.heads_per_seq = dims->H;
    a.o_lat = (__nv_bfloat16 *)out;
    a.lse = lse;
    a.num_splits = 1;
    e = mla::launch_attn_expand(a, st);
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

// The naive comparison path runs on the tensor cores (the expand form) where
// those kernels take the shape, else on the CUDA-core kernels of naive.cu.
bool naive_on_expand(const mla_dims *d, const mla_cache *c) { return check_expand(d, c) == MLA_OK; }

size_t naive_cuda_core_bytes(const mla_dims *d, const mla_cache *c) {
    size_t per = (size_t)d->B * d->H * (size_t)cache_capacity(c);
    return kStatusBytes + round_up(per * d->d_nope * 2, 256) + per * d->d_v * 2;
}

}  // namespace

extern "C" {

MLA_API const char *mla_status_string(int status) {
    switch (status) {
        case MLA_OK: return "MLA_OK";
        case MLA_ERR_NULL: return "MLA_ERR_NULL: a required pointer is NULL";
        case MLA_ERR_SHAPE: return "MLA_ERR_SHAPE: a size is negative or sizes disagree";
        case MLA_ERR_SEQLEN: return "MLA_ERR_SEQLEN: a sequence length is outside [s_q, capacity]";
        case MLA_ERR_ALIGN: return "MLA_ERR_ALIGN: a pointer or stride is not 16-byte aligned";
        case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE: workspace too small";
        case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED: shape outside the supported envelope";
        case MLA_ERR_CUDA: return "MLA_ERR_CUDA: a CUDA call failed";
        case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT: a bounded device wait gave up";
        case MLA_ERR_PAGE: return "MLA_ERR_PAGE: a block-table entry is outside the pool";
        default: return "unknown mla status";
    }
}

MLA_API int mla_abi_version(void) { return kAbiVersion; }

MLA_API int mla_set_wait_limit_ns(unsigned long long ns) {
    g_wait_ns.store(ns, std::memory_order_relaxed);
    return MLA_OK;
}

MLA_API int mla_absorb_q(const mla_dims *dims, const void *q_nope, const void *q_rope, const void *w_uk,
                         void *q_cat, void *stream) {
    int s = check_dims(dims);
    if (s) return s;
    if (dims->B == 0) return MLA_OK;
    if (!q_nope || !w_uk || !q_cat || (dims->d_rope && !q_rope)) return MLA_ERR_NULL;
    if (!aligned16(q_nope) || !aligned16(w_uk) || !aligned16(q_cat) || (q_rope && !aligned16(q_rope)))
        return MLA_ERR_ALIGN;
    cudaError_t e = mla::launch_absorb_q_tc(*dims, q_nope, q_rope, w_uk, q_cat, as_stream(stream));
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

MLA_API int mla_decode_num_splits(const mla_dims *dims, const mla_cache *cache) {
    if (check_dims(dims) || check_cache(dims, cache)) return 0;
    const DecodePlan pl = plan_decode(dims, cache, 0);
    if (pl.persist_groups > 0) return pl.persist_groups;
    return pl.b_tail ? pl.tail_splits : pl.splits;
}

MLA_API size_t mla_decode_workspace_size(const mla_dims *dims, const mla_cache *cache, int num_splits) {
    if (check_dims(dims) || check_cache(dims, cache)) return 0;
    if (num_splits < MLA_SPLITS_BALANCED || num_splits > kMaxSplits) return 0;
    if (num_splits == MLA_SPLITS_BALANCED && !balanced_supported(dims, cache)) return 0;
    return plan_workspace_bytes(dims, plan_decode(dims, cache, num_splits));
}

MLA_API int mla_decode_attn(const mla_dims *dims, const void *q_cat, const mla_cache *cache, void *o_lat,
                            float *lse, void *workspace, size_t ws_bytes, int num_splits, void *stream) {
    int s = check_dims(dims);
    if (s) return s;
    if (!cache) return MLA_ERR_NULL;
    if ((s = check_cache(dims, cache))) return s;
    if (num_splits < MLA_SPLITS_BALANCED || num_splits > kMaxSplits) return MLA_ERR_SHAPE;
    if (num_splits == MLA_SPLITS_BALANCED && !balanced_supported(dims, cache)) return MLA_ERR_UNSUPPORTED;
    if (!workspace) return MLA_ERR_NULL;
    if (!aligned16(workspace)) return MLA_ERR_ALIGN;
    const DecodePlan pl = plan_decode(dims, cache, num_splits);
    if (ws_bytes < plan_workspace_bytes(dims, pl)) return MLA_ERR_WORKSPACE;
    if (dims->B > 0) {
        if (!q_cat || !o_lat || !lse) return MLA_ERR_NULL;
        if (!aligned16(q_cat) || !aligned16(o_lat) || !aligned16(lse)) return MLA_ERR_ALIGN;
    }
    cudaStream_t st = as_stream(stream);
    if (cudaMemsetAsync(workspace, 0, plan_zero_bytes(dims, pl), st) != cudaSuccess) return MLA_ERR_CUDA;
    if (dims->B == 0) return MLA_OK;

    mla::AttnParams p = make_params(dims, cache);
    p.q_cat = (const __nv_bfloat16 *)q_cat;
    p.o_lat = (__nv_bfloat16 *)o_lat;
    p.lse = lse;
    p.status = (int *)workspace;
    cudaError_t e = launch_decode_plan(dims, pl, p, workspace, st);
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

MLA_API size_t mla_cache_append_workspace_size(const mla_dims *dims, int d_model) {
    if (check_dims(dims) || d_model < 1) return 0;
    const int M = dims->B * dims->s_q;
    const mla::AppendPlan plan = mla::append_plan(M, dims->d_c, d_model);
    return kStatusBytes + (size_t)plan.splits * M * dims->d_c * sizeof(float);
}

MLA_API int mla_cache_append(const mla_dims *dims, int d_model, const void *x, const void *w_dkv, const void *k_rope,
                             const mla_cache *cache, void *workspace, size_t ws_bytes, void *stream) {
    int s = check_dims(dims);
    if (s) return s;
    if (d_model < 1) return MLA_ERR_SHAPE;
    if (d_model % 8) return MLA_ERR_ALIGN;  // rows of x must be whole 16-byte units
    s = check_cache(dims, cache);
    if (s) return s;
    if (!workspace) return MLA_ERR_NULL;
    if (!aligned16(workspace)) return MLA_ERR_ALIGN;
    if (ws_bytes < mla_cache_append_workspace_size(dims, d_model)) return MLA_ERR_WORKSPACE;
    if (dims->B > 0) {
        if (!x || !w_dkv || (dims->d_rope && !k_rope)) return MLA_ERR_NULL;
        if (!aligned16(x) || !aligned16(w_dkv) || (k_rope && !aligned16(k_rope))) return MLA_ERR_ALIGN;
    }
    cudaStream_t st = as_stream(stream);
    if (cudaMemsetAsync(workspace, 0, sizeof(int), st) != cudaSuccess) return MLA_ERR_CUDA;
    if (dims->B == 0) return MLA_OK;
    mla::AttnParams p = make_params(dims, cache);
    p.status = (int *)workspace;
    float *part = (float *)((char *)workspace + kStatusBytes);
    cudaError_t e = mla::launch_cache_append_tc(p, d_model, x, w_dkv, k_rope, part, st);
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

MLA_API size_t mla_decode_sparse_workspace_size(const mla_dims *dims, const mla_cache *cache, int topk,
                                                int num_splits) {
    if (check_dims(dims) || check_cache(dims, cache) || topk < 1) return 0;
    return attn_workspace_bytes(dims, plan_splits_len(dims, topk, num_splits));
}

MLA_API int mla_decode_attn_sparse(const mla_dims *dims, const void *q_cat, const mla_cache *cache,
                                   const int *indices, int topk, void *o_lat, float *lse, void *workspace,
                                   size_t ws_bytes, int num_splits, void *stream) {
    int s = check_dims(dims);
    if (s) return s;
    s = check_cache(dims, cache);
    if (s) return s;
    s = check_sparse(dims, cache, indices, topk);
    if (s) return s;
    if (num_splits < 0 || num_splits > kMaxSplits) return MLA_ERR_SHAPE;
    if (!workspace) return MLA_ERR_NULL;
    if (!aligned16(workspace)) return MLA_ERR_ALIGN;
    const int splits = plan_splits_len(dims, topk, num_splits);
    if (ws_bytes < attn_workspace_bytes(dims, splits)) return MLA_ERR_WORKSPACE;
    if (dims->B > 0) {
        if (!q_cat || !o_lat || !lse) return MLA_ERR_NULL;
        if (!aligned16(q_cat) || !aligned16(o_lat) || !aligned16(lse)) return MLA_ERR_ALIGN;
    }
    cudaStream_t st = as_stream(stream);
    if (cudaMemsetAsync(workspace, 0, sizeof(int), st) != cudaSuccess) return MLA_ERR_CUDA;
    if (dims->B == 0) return MLA_OK;
    mla::AttnParams p = make_params(dims, cache);
    p.q_cat = (const __nv_bfloat16 *)q_cat;
    p.o_lat = (__nv_bfloat16 *)o_lat;
    p.lse = lse;
    p.num_splits = splits;
    p.status = (int *)workspace;
    p.indices = indices;
    p.topk = topk;
    if (splits > 1) {
        size_t rows = (size_t)dims->B * splits * dims->s_q * dims->H;
        char *base = (char *)workspace + kStatusBytes;
        p.part_ml = (float *)base;
        p.part_acc = (float *)(base + round_up(rows * 4 * sizeof(float), 256));
    }
    cudaError_t e = mla::launch_attn_tc(p, st);
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

MLA_API int mla_out_proj(const mla_dims *dims, const void *o_lat, const void *w_uv, void *out, void *stream) {
    int s = check_dims(dims);
    if (s) return s;
    if (dims->B == 0) return MLA_OK;
    if (!o_lat || !w_uv || !out) return MLA_ERR_NULL;
    if (!aligned16(o_lat) || !aligned16(w_uv) || !aligned16(out)) return MLA_ERR_ALIGN;
    cudaError_t e = mla::launch_out_proj_tc(*dims, o_lat, w_uv, out, as_stream(stream));
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

MLA_API size_t mla_naive_workspace_size(const mla_dims *dims, const mla_cache *cache) {
    if (check_dims(dims) || check_cache(dims, cache)) return 0;
    if ((long long)dims->B * dims->H > kMaxGridZ) return 0;  // one (sequence, head) per grid slice
    return naive_on_expand(dims, cache) ? expand_workspace_bytes(dims, cache) : naive_cuda_core_bytes(dims, cache);
}

MLA_API int mla_naive_decode(const mla_dims *dims, const void *q_nope, const void *q_rope,
                             const mla_cache *cache, const void *w_uk, const void *w_uv, void *out, float *lse,
                             void *workspace, size_t ws_bytes, void *stream) {
    int s = check_dims(dims);
    if (s) return s;
    if (!cache) return MLA_ERR_NULL;
    if ((s = check_cache(dims, cache))) return s;
    if (cache->kv_dtype != MLA_KV_BF16) return MLA_ERR_UNSUPPORTED;
    if ((long long)dims->B * dims->H > kMaxGridZ) return MLA_ERR_UNSUPPORTED;
    if (!workspace) return MLA_ERR_NULL;
    if (!aligned16(workspace)) return MLA_ERR_ALIGN;
    if (ws_bytes < mla_naive_workspace_size(dims, cache)) return MLA_ERR_WORKSPACE;
    if (dims->B > 0) {
        if (!q_nope || !w_uk || !w_uv || !out || !lse || (dims->d_rope && !q_rope)) return MLA_ERR_NULL;
        if (!aligned16(q_nope) || !aligned16(w_uk) || !aligned16(w_uv) || !aligned16(out) || !aligned16(lse) ||
            (q_rope && !aligned16(q_rope)))
            return MLA_ERR_ALIGN;
    }
    cudaStream_t st = as_stream(stream);
    if (cudaMemsetAsync(workspace, 0, sizeof(int), st) != cudaSuccess) return MLA_ERR_CUDA;
    if (dims->B == 0) return MLA_OK;
    if (naive_on_expand(dims, cache)) return run_expand(dims, q_nope, q_rope, cache, w_uk, w_uv, out, lse, workspace, st);
    mla::AttnParams p = make_params(dims, cache);
    p.status = (int *)workspace;
    char *kbuf = (char *)workspace + kStatusBytes;
    cudaError_t e = mla::launch_naive(p, dims->d_nope, dims->d_v, q_nope, q_rope, w_uk, w_uv, out, lse, kbuf, st);
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

MLA_API double mla_prefill_crossover(const mla_dims *dims, long long L) {
    if (check_shape(dims) || L < 1) return 0.0;
    // "Why MLA and MTP Fight Each Other", 5.3 and 5.6: both bracketings cost
    //   absorb: S * [2 d_c (d_k + d_v) + L (4 d_c)]           (per head, MACs x 2)
    //   expand: L * 2 d_c (d_k + d_v) + S * L * 2 (d_k + d_v)
    // and they tie at S* = L d_c (d_k + d_v) / (d_c (d_k + d_v) + L (2 d_c - d_k - d_v)).
    const double dc = dims->d_c, dk = dims->d_nope, dv = dims->d_v, l = (double)L;
    const double denom = dc * (dk + dv) + l * (2.0 * dc - dk - dv);
    return denom > 0.0 ? l * dc * (dk + dv) / denom : INFINITY;
}

MLA_API size_t mla_prefill_expand_workspace_size(const mla_dims *dims, const mla_cache *cache) {
    if (check_shape(dims) || check_cache(dims, cache) || check_expand(dims, cache)) return 0;
    return expand_workspace_bytes(dims, cache);
}

MLA_API int mla_prefill_expand(const mla_dims *dims, const void *q_nope, const void *q_rope, const mla_cache *cache,
                               const void *w_uk, const void *w_uv, void *out, float *lse, void *workspace,
                               size_t ws_bytes, void *stream) {
    int s = check_shape(dims);
    if (s) return s;
    if (!cache) return MLA_ERR_NULL;
    if ((s = check_cache(dims, cache))) return s;
    if ((s = check_expand(dims, cache))) return s;
    if (!workspace) return MLA_ERR_NULL;
    if (!aligned16(workspace)) return MLA_ERR_ALIGN;
    if (ws_bytes < expand_workspace_bytes(dims, cache)) return MLA_ERR_WORKSPACE;
    if (dims->B > 0) {
        if (!q_nope || !w_uk || !w_uv || !out || !lse || (dims->d_rope && !q_rope)) return MLA_ERR_NULL;
        if (!aligned16(q_nope) || !aligned16(w_uk) || !aligned16(w_uv) || !aligned16(out) || !aligned16(lse) ||
            (q_rope && !aligned16(q_rope)))
            return MLA_ERR_ALIGN;
    }
    cudaStream_t st = as_stream(stream);
    if (cudaMemsetAsync(workspace, 0, sizeof(int), st) != cudaSuccess) return MLA_ERR_CUDA;
    if (dims->B == 0) return MLA_OK;
    return run_expand(dims, q_nope, q_rope, cache, w_uk, w_uv, out, lse, workspace, st);
}

MLA_API size_t mla_prefill_workspace_size(const mla_dims *dims, const mla_cache *cache) {
    if (check_shape(dims) || check_cache(dims, cache)) return 0;
    size_t n = check_dims(dims) ? 0 : absorbed_workspace_bytes(dims, plan_workspace_bytes(dims, plan_decode(dims, cache, 0)));
    if (!check_expand(dims, cache)) {
        const size_t e = expand_workspace_bytes(dims, cache);
        if (e > n) n = e;
    }
    return n;
}

MLA_API int mla_prefill(const mla_dims *dims, const void *q_nope, const void *q_rope, const mla_cache *cache,
                        const void *w_uk, const void *w_uv, void *out, float *lse, void *workspace, size_t ws_bytes,
                        int *path, void *stream) {
    int s = check_shape(dims);
    if (s) return s;
    if (!cache) return MLA_ERR_NULL;
    if ((s = check_cache(dims, cache))) return s;
    const long long L = cache->max_seq_len > 0 ? cache->max_seq_len : cache_capacity(cache);
    const bool expand = !check_expand(dims, cache) && (double)dims->s_q >= mla_prefill_crossover(dims, L);
    if (path) *path = expand ? MLA_PATH_EXPAND : MLA_PATH_ABSORB;
    if (expand) return mla_prefill_expand(dims, q_nope, q_rope, cache, w_uk, w_uv, out, lse, workspace, ws_bytes, stream);
    if ((s = check_dims(dims))) return s;
    const size_t attn_ws_bytes = plan_workspace_bytes(dims, plan_decode(dims, cache, 0));
    if (!workspace) return MLA_ERR_NULL;
    if (!aligned16(workspace)) return MLA_ERR_ALIGN;
    if (ws_bytes < absorbed_workspace_bytes(dims, attn_ws_bytes)) return MLA_ERR_WORKSPACE;
    const size_t rows = (size_t)dims->B * dims->s_q * dims->H;
    char *attn_ws = (char *)workspace;
    char *q_cat = attn_ws + round_up(attn_ws_bytes, 256);
    char *o_lat = q_cat + round_up(rows * (dims->d_c + dims->d_rope) * 2, 256);
    if ((s = mla_absorb_q(dims, q_nope, q_rope, w_uk, q_cat, stream))) return s;
    if ((s = mla_decode_attn(dims, q_cat, cache, o_lat, lse, attn_ws, attn_ws_bytes, 0, stream))) return s;
    return mla_out_proj(dims, o_lat, w_uv, out, stream);
}

MLA_API int mla_decode_step(const mla_dims *dims, const void *q_nope, const void *q_rope, const mla_cache *cache,
                            const void *w_uk, const void *w_uv, void *q_cat, void *o_lat, void *out, float *lse,
                            void *workspace, size_t ws_bytes, int num_splits, void *stream) {
    int s = check_dims(dims);
    if (s) return s;
    if (!cache) return MLA_ERR_NULL;
    if ((s = check_cache(dims, cache))) return s;
    if (num_splits < MLA_SPLITS_BALANCED || num_splits > kMaxSplits) return MLA_ERR_SHAPE;
    if (num_splits == MLA_SPLITS_BALANCED && !balanced_supported(dims, cache)) return MLA_ERR_UNSUPPORTED;
    if (!workspace) return MLA_ERR_NULL;
    if (!aligned16(workspace)) return MLA_ERR_ALIGN;
    const DecodePlan pl = plan_decode(dims, cache, num_splits);
    if (ws_bytes < plan_workspace_bytes(dims, pl)) return MLA_ERR_WORKSPACE;
    if (dims->B > 0) {
        if (!q_nope || !w_uk || !w_uv || !q_cat || !o_lat || !out || !lse || (dims->d_rope && !q_rope))
            return MLA_ERR_NULL;
        if (!aligned16(q_nope) || !aligned16(w_uk) || !aligned16(w_uv) || !aligned16(q_cat) || !aligned16(o_lat) ||
            !aligned16(out) || !aligned16(lse) || (q_rope && !aligned16(q_rope)))
            return MLA_ERR_ALIGN;
    }
    cudaStream_t st = as_stream(stream);
    // the status reset comes first, so that nothing but kernels separates the three
    // launches: the attention and out_proj grids are launched programmatically and
    // start while their predecessor runs, reading its output only once it completed
    if (cudaMemsetAsync(workspace, 0, plan_zero_bytes(dims, pl), st) != cudaSuccess) return MLA_ERR_CUDA;
    if (dims->B == 0) return MLA_OK;
    cudaError_t e = mla::launch_absorb_q_tc(*dims, q_nope, q_rope, w_uk, q_cat, st, true);
    if (e != cudaSuccess) return MLA_ERR_CUDA;
    mla::AttnParams p = make_params(dims, cache);
    p.q_cat = (const __nv_bfloat16 *)q_cat;
    p.o_lat = (__nv_bfloat16 *)o_lat;
    p.lse = lse;
    p.status = (int *)workspace;
    p.pdl = 1;
    if ((e = launch_decode_plan(dims, pl, p, workspace, st)) != cudaSuccess) return MLA_ERR_CUDA;
    e = mla::launch_out_proj_tc(*dims, o_lat, w_uv, out, st, true);
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

MLA_API int mla_read_status(const void *workspace, int *status, void *stream) {
    if (!workspace || !status) return MLA_ERR_NULL;
    int v = 0;
    cudaStream_t st = as_stream(stream);
    if (cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MLA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MLA_ERR_CUDA;
    *status = v;
    return MLA_OK;
}

}  // extern "C"
