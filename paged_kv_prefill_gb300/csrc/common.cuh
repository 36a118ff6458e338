// common.cuh -- parameters, constants and the per-item geometry shared by
// the scheduler, the tensor-core attention kernel and the debug gather.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/b2pa.h"

namespace b2pa {

constexpr int kKvTile = 128;      // keys per kv tile (MMA N of Q K^T, K of P V)
constexpr int kQRows = 128;       // MMA M rows per query tile (tokens x heads of one kv group)
constexpr int kQTiles = 2;        // query tiles per work item (they share every K/V tile)
constexpr int kCostCap = 1023;    // scheduler buckets: costs >= this share the top bucket
constexpr int kSchedBuckets = kCostCap + 1;
constexpr int kSchedThreads = 1024;
constexpr int kSchedMaxBatch = 4096;   // scheduler keeps 3 words per request in shared memory
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s: default pipeline wait limit; drains always use it

// Where request b's query rows start: cum_q[b], or b * q_per_req for a decode
// batch, whose requests all have q_per_req query tokens (cum_q null).
struct QStarts {
    const int* cum_q;
    int q_per_req;
    __device__ __forceinline__ int operator[](int b) const { return cum_q != nullptr ? cum_q[b] : b * q_per_req; }
};

// A request is processed only if its lengths are consistent with the bounds
// the caller gave; otherwise the scheduler sets B2PA_DEV_BAD_REQUEST.
struct RequestView {
    int q_start;
    int q_len;
    int kv_len;
    bool ok;
};

__device__ __forceinline__ RequestView load_request(QStarts cum_q, const int* seq_lens, int b, int max_q_len,
                                                    int max_kv_len, int page_size, int max_pages, int num_tokens)
{
    RequestView r;
    int q0 = cum_q[b], q1 = cum_q[b + 1];
    r.q_start = q0;
    r.q_len = q1 - q0;
    r.kv_len = seq_lens[b];
    long long pages = ((long long)r.kv_len + page_size - 1) / page_size;
    r.ok = r.q_len >= 0 && r.q_len <= r.kv_len && r.q_len <= max_q_len && r.kv_len <= max_kv_len &&
           pages <= max_pages && q0 >= 0 && q1 <= num_tokens;
    return r;
}

// Geometry of work item `it` of a request: which query tokens it covers and
// which kv tiles their visible keys touch.  Query i sits at position
// kv_len - q_len + i and sees keys lo(pos) .. pos, lo = 0 for a negative
// window, else max(0, pos - window).
struct ItemGeom {
    int tok0;   // first query token (index within the request)
    int nq;     // query tiles with at least one token (1 .. kQTiles)
    int n_lo;   // first kv tile
    int n_hi;   // last kv tile
};

__device__ __forceinline__ ItemGeom item_geometry(int q_len, int kv_len, int it, int rows_per_tile, int window)
{
    ItemGeom g;
    const int per_item = rows_per_tile * kQTiles;
    g.tok0 = it * per_item;
    int i1 = min(g.tok0 + per_item, q_len) - 1;
    static_assert(kQTiles == 2, "query tiles per item");
    g.nq = i1 - g.tok0 >= rows_per_tile ? 2 : 1;  // (i1 - tok0) / rows_per_tile + 1, without a division
    int prefix = kv_len - q_len;
    int p_min = prefix + g.tok0, p_max = prefix + i1;
    int lo = window < 0 ? 0 : max(0, p_min - window);
    g.n_lo = lo / kKvTile;
    g.n_hi = p_max / kKvTile;
    return g;
}

// The page ids of request b: a row of a [B, max_pages] block table, or (the
// ragged form) the slice ids[indptr[b] .. indptr[b + 1]) of one flat array
// (FlashInfer's paged_kv_indices / paged_kv_indptr).
__device__ __forceinline__ const int* page_row(const int* ids, long long row_stride, const int* indptr, int b)
{
    return indptr != nullptr ? ids + indptr[b] : ids + (long long)b * row_stride;
}

// Kv tile j of a request as per-page TMA boxes, for page sizes that are
// powers of two: lane l of a warp loads page column (j * kKvTile >> log2 P) + l,
// from in-page slot slot0 (nonzero only when P > kKvTile).  A lane is valid if
// l < pages per tile and its column is below the request's page count.  The
// attention producer and the debug gather both address pages through this.
struct TileLoad {
    int page;
    int slot0;
    bool valid;
};

__device__ __forceinline__ TileLoad tile_load(const int* row, int j, int lane, int log2_p, int n_pages)
{
    const int P = 1 << log2_p;
    const int ppt = P >= kKvTile ? 1 : kKvTile >> log2_p;  // pages per kv tile
    TileLoad t;
    const int first_col = (int)(((long long)j * kKvTile) >> log2_p);
    t.slot0 = P > kKvTile ? (int)(((long long)j * kKvTile) & (P - 1)) : 0;
    const int col = first_col + lane;
    t.valid = lane < ppt && col < n_pages;
    t.page = t.valid ? row[col] : 0;
    return t;
}

// Split-KV (decode batches): a request's single work item per kv head is cut
// into chunks of `split_tiles` kv tiles; chunk s covers tiles
// n_lo + s * split_tiles .. (clipped to n_hi).
__device__ __forceinline__ int split_count(const ItemGeom& g, int split_tiles)
{
    return (g.n_hi - g.n_lo + split_tiles) / split_tiles;
}
__device__ __forceinline__ void split_range(ItemGeom* g, int s, int split_tiles)
{
    g->n_lo += s * split_tiles;
    g->n_hi = min(g->n_hi, g->n_lo + split_tiles - 1);
}

// The scales a kernel computes with: the host values, or the ones in device
// memory when the call passed them as tensors (read once per thread;
// bmm1_scale * log2(e) is formed in double and rounded once, as on the host).
// ok = false when bmm1_scale is not finite and > 0 or bmm2_scale not finite.
struct Scales {
    float scale_log2;
    float bmm2;
    bool ok;
};

__device__ __forceinline__ Scales load_scales(float scale_log2, float bmm2, const float* bmm1_dev, const float* bmm2_dev)
{
    Scales sc{scale_log2, bmm2, true};
    if (bmm1_dev != nullptr) {
        const float b1 = *bmm1_dev;
        sc.ok = isfinite(b1) && b1 > 0.f;
        sc.scale_log2 = (float)((double)b1 * 1.4426950408889634);
    }
    if (bmm2_dev != nullptr) {
        sc.bmm2 = *bmm2_dev;
        sc.ok = sc.ok && isfinite(sc.bmm2);
    }
    return sc;
}

struct SchedParams {
    const int* cum_q;         // null: q_per_req query tokens per request (decode batch)
    int q_per_req;
    const int* kv_indptr;     // non-null: ragged page table (block_tables = the flat page ids)
    const int* seq_lens;
    const int* cum_kv;        // may be null
    const int* block_tables;  // read only when debug != 0
    long long bt_stride;
    int B, Hkv, rows_per_tile, window, max_q_len, max_kv_len, page_size, max_pages, num_tokens, num_pages;
    int debug;
    int cap;
    int nbuckets;             // cost buckets in use: min(kSchedBuckets, largest possible cost + 1)
    int split_tiles;          // > 0: split-KV items (one query item per request and kv head, cut in chunks)
    int* nsplit;              // split-KV: chunks per request (0 for a request without work), for the combine
    int4* items;
    int* count;
    unsigned* err;
};

struct AttnParams {  // 128-byte aligned through its CUtensorMap members
    CUtensorMap tm_q;   // 3-D: (D, H, T), box (64, G, rows_per_tile)
    CUtensorMap tm_k;   // 4-D: (D, P, Hkv, pages), box (64 | 128 bytes, min(P,128), 1, 1)
    CUtensorMap tm_v;
    CUtensorMap tm_o;   // 3-D: (D, H, T), box (64, min(G, 32), max(1, 32 / G)): one warp's 32 rows
    int out_tma;        // 1: tm_o is valid and a warp's 32 rows are whole boxes (G divides 32 or 32 divides G)
    const int* cum_q;    // null: q_per_req query tokens per request
    int q_per_req;
    const int* seq_lens;
    const int* block_tables;
    const int* kv_indptr;  // non-null: ragged page table (block_tables = the flat page ids)
    const float* sinks;  // may be null
    uint16_t* out;       // bf16 bits
    int split_tiles;     // > 0: items are kv chunks; a chunk of a request cut in several writes partials
    int part_slots;      // chunks per row in the partial buffers
    float* part_o;       // [(token * H + head) * part_slots + chunk][D] unnormalised O (f32)
    float* part_ml;      // [(token * H + head) * part_slots + chunk][2] running maximum (log2 units) and sum
    unsigned long long wait_limit_ns;  // pipeline waits give up after this long (B2PA_DEV_TIMEOUT)
    int inject_stall;                  // failure-detection tests: one wait that nothing completes
    long long bt_stride;
    long long out_stride_tok;
    long long out_stride_head;
    // Work distribution.  Every CTA builds the longest-first list itself
    // (sched: its inputs) and starts with item blockIdx.x; the first CTA to
    // win `claim` also writes the list to `items` and then sets `ready`; later
    // items are taken in order from gridDim.x on through `counter`.  The last
    // CTA to finish (`done`) sets all four words back to zero for the next launch.
    SchedParams sched;
    const int4* items;
    int* counter;
    int* claim;
    int* ready;
    int* done;
    unsigned* err;
    int cap;
    int H, Hkv, G, rows_per_tile, page_size, num_pages;
    int window;
    float scale_log2;    // bmm1_scale * log2(e)
    float bmm2;
    const float* bmm1_dev;  // non-null: bmm1_scale is read from device memory (scale_log2 unused)
    const float* bmm2_dev;  // non-null: bmm2_scale is read from device memory (bmm2 unused)
};

struct GatherParams {
    CUtensorMap tm_k;
    CUtensorMap tm_v;
    const int* seq_lens;
    const int* cum_kv;
    const int* block_tables;
    const int* kv_indptr;  // non-null: ragged page table
    long long bt_stride;
    uint8_t* k_out;
    uint8_t* v_out;
    long long out_rows;
    int B, Hkv, D, page_size, max_pages, num_pages, esize;
    unsigned* err;
};

struct GenericParams {
    const uint16_t* q;
    const void* k;
    const void* v;
    const int* cum_q;    // null: q_per_req query tokens per request
    int q_per_req;
    const int* seq_lens;
    const int* block_tables;
    const int* kv_indptr;  // non-null: ragged page table
    const float* sinks;
    uint16_t* out;
    long long q_st_tok, q_st_head;
    long long out_st_tok, out_st_head;
    long long k_st_page, k_st_head, k_st_slot;  // element strides by logical dim
    long long v_st_page, v_st_head, v_st_slot;
    long long bt_stride;
    int B, T, H, Hkv, D, page_size, max_pages, num_pages, max_q_len, max_kv_len;
    int window;
    float scale_log2;
    float bmm2;
    const float* bmm1_dev;  // as in AttnParams
    const float* bmm2_dev;
    unsigned* err;
};

// Merging the chunks of split-KV rows (decode batches): one warp per output row.
struct CombineParams {
    const float* part_o;
    const float* part_ml;
    const int* nsplit;   // chunks per request (<= 1: the attention kernel wrote the row)
    const float* sinks;  // may be null
    uint16_t* out;
    long long out_st_tok, out_st_head;
    int B, q_per_req, H, D, part_slots;
    float bmm2;
    const float* bmm2_dev;
};

// Host launchers (one translation unit each).
cudaError_t launch_schedule(const SchedParams& p, cudaStream_t stream);
cudaError_t launch_attention_tc(const AttnParams& p, int head_dim, bool fp8, int grid, cudaStream_t stream, bool pdl);
// the one-window-tile kernel for short left windows at head_dim 64 (attn_win.cu)
cudaError_t launch_attention_win(const AttnParams& p, int grid, cudaStream_t stream);
int win_max_keys();
cudaError_t launch_gather(const GatherParams& p, bool fp8, int max_kv_len, cudaStream_t stream);
cudaError_t launch_attention_generic(const GenericParams& p, bool fp8, cudaStream_t stream);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream);
// Ragged page table: kv_len[b] = (pages_b - 1) * page_size + last_page_len[b]
// (0 without pages); a malformed request gets kv_len -1 and B2PA_DEV_BAD_REQUEST.
cudaError_t launch_ragged_lengths(const int* indptr, const int* last_page_len, int B, int page_size, int* kv_len,
                                  unsigned* err, cudaStream_t stream);

}  // namespace b2pa
