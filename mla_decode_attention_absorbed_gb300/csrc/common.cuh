// Shared device helpers of the MLA decode library (no method arithmetic here).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mla.h"

namespace mla {

// Parameters every attention kernel receives (plain values and device pointers).
struct AttnParams {
    int B, H, s_q, d_c, d_rope;
    float scale;
    const __nv_bfloat16 *q_cat;   // [B][s_q][H][W]
    const void *kv;               // contiguous or pool, rows of W elements (bf16, or E4M3 codes)
    int kv_fp8;                   // 1: E4M3 codes, value = kv_scale * code
    float kv_scale;
    long long seq_stride;         // contiguous: elements between sequences
    int capacity;                 // tokens a sequence may hold
    const int *block_table;       // NULL => contiguous
    int max_pages, page_size, num_pages;
    const int *seq_lens;
    __nv_bfloat16 *o_lat;         // [B][s_q][H][d_c]
    float *lse;                   // [B][s_q][H]
    int num_splits;
    // tail pieces (tail_splits > 1, with num_splits == 1): grid items below tail_b0
    // are whole sequences, item tail_b0 + i is piece i % tail_splits of sequence
    // tail_b0 + i / tail_splits; partials are kept for those sequences only,
    // indexed from tail_b0
    int tail_b0, tail_splits;
    // longest-first work order (dense decode over several waves): work-order
    // position i runs the sequence of rank i by length; order[i] records it for
    // the merge (workspace, B ints)
    int lpt;
    int *order;
    // merge: partial sequence j is work-order position combine_b0 + j
    int combine_b0;
    float *part_acc;              // [B][splits][s_q*H][d_c] (num_splits > 1)
    float *part_ml;               // [B][splits][s_q*H][2 CTA halves][2]   (m, l)
    int *status;                  // device status word
    const int *indices;           // sparse: [B][s_q][topk] token positions (NULL => dense)
    int topk;
    // expanded (per-head) attention: the B "sequences" are (sequence, head) pairs
    // b = seq * heads_per_seq + head; lengths are read at seq_lens[seq] and the
    // query / output / lse rows are [seq][s_q][heads_per_seq] (0 or 1: plain)
    int heads_per_seq;
    int q_w;                      // elements per q_cat row (0: d_c + d_rope)
    // launched programmatically right after the grid that writes q_cat (a fused
    // decode step): q_cat is read only once that grid has completed, and the next
    // grid (out_proj) may start its CTAs at once
    int pdl;
    // bound of the kernel's waits for work (0: the default, 2 s); a wait that runs
    // out records MLA_ERR_TIMEOUT and the CTA unwinds (the waits that drain copies
    // and MMAs still in flight keep the default)
    unsigned long long wait_ns;
    // persistent decode (attn_persist.cu): persist_groups x (128-row blocks) CTA
    // pairs, each group an equal contiguous range of the batch's sequence tiles
    // (in batch order); a sequence one range holds whole is written out directly,
    // the others leave normalised bf16 pieces in part_acc ([pair][2 slots][128
    // rows][d_c]) with their (m, l) in part_ml, and the CTA that writes a
    // sequence's last piece merges them (counters: [B][row blocks][2 CTAs],
    // zeroed with the status word).  prefix: the batch's tile prefix (B + 1 ints);
    // ml: the (m, l) the softmax warps hand to the epilogue warps.
    int persist_groups;
    int *counters;
    int *prefix;
    float *ml;
};

// Persistent decode: groups of CTA pairs in use for T sequence tiles (at most
// max_groups, each range at least kMinGroupTiles tiles long), group g's range
// [group_first_tile(g), group_first_tile(g + 1)) of the tiles, the group whose
// range holds tile t, and the partial slot a sequence starting at tile S takes
// in group g (0: it began at or before the range, the group's first item; 1: it
// began inside and runs past it, the group's last item).
constexpr int kMinGroupTiles = 8;
__host__ __device__ __forceinline__ int persist_groups(int max_groups, long long T) {
    long long g = T / kMinGroupTiles;
    if (g > max_groups) g = max_groups;
    return g < 1 ? 1 : (int)g;
}
__host__ __device__ __forceinline__ long long group_first_tile(int g, int G, long long T) { return (long long)g * T / G; }
__host__ __device__ __forceinline__ int group_of_tile(long long t, int G, long long T) {
    int g = (int)((t * G) / T);
    while (g + 1 < G && group_first_tile(g + 1, G, T) <= t) ++g;
    while (g > 0 && group_first_tile(g, G, T) > t) --g;
    return g;
}
__host__ __device__ __forceinline__ int persist_slot(long long S, int g, int G, long long T) {
    return S <= group_first_tile(g, G, T) ? 0 : 1;
}

// Record the first device-side error; later ones keep the first.
__device__ __forceinline__ void set_status(int *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// Whether sequence b's length is usable; records MLA_ERR_SEQLEN otherwise.
__device__ __forceinline__ bool seq_len_ok(const AttnParams &p, int L) {
    return L >= p.s_q && L <= p.capacity;
}

// Row of cached token j of sequence b in a bf16 cache, or nullptr if its page
// id is out of range.
__device__ __forceinline__ const __nv_bfloat16 *kv_row(const AttnParams &p, int b, int j) {
    const long long W = p.d_c + p.d_rope;
    const __nv_bfloat16 *kv = static_cast<const __nv_bfloat16 *>(p.kv);
    if (p.block_table == nullptr) return kv + (long long)b * p.seq_stride + (long long)j * W;
    int page = __ldg(p.block_table + (long long)b * p.max_pages + j / p.page_size);
    if (page < 0 || page >= p.num_pages) return nullptr;
    return kv + ((long long)page * p.page_size + j % p.page_size) * W;
}

// Token range [t0, t1) of split `split` for a history of L tokens: the
// ceil(L/64) 64-token tiles are dealt out in equal contiguous runs.
__device__ __forceinline__ void split_range(int L, int splits, int split, int &t0, int &t1) {
    int tiles = (L + 63) / 64;
    int per = (tiles + splits - 1) / splits;
    t0 = min(L, split * per * 64);
    t1 = min(L, (split + 1) * per * 64);
}

}  // namespace mla
