// worklist.cuh -- the longest-first work list of the tensor-core path, built
// by one CTA with all its threads.  The scheduler kernel runs it for the debug
// entry point that returns the list; the attention kernel runs it in every
// CTA at its start (each CTA learns its own first item from it, and the first
// CTA to claim the job also writes the list for the others).
//
// The sort runs over units (request b, query item it): every kv head of a
// unit has the same tile range and cost, so each unit is decoded once and
// expands to Hkv consecutive items (b, 0 .. Hkv-1, it) of the list.
// 1. Validate each request (load_request) and count its units:
//    ceil(q_len / (rows_per_tile * kQTiles)), or, for split-KV (decode)
//    batches, the number of kv chunks of its one query item (cut in chunks
//    of split_tiles kv tiles; it = the chunk index there).
// 2. Enumerate units in (b, it) order; cost = kv tiles x non-empty query
//    tiles (item_geometry), bucket = min(cost, nbuckets - 1).
// 3. Stable counting sort by bucket, descending: each warp owns a contiguous
//    slice of the enumeration and counts per bucket with __match_any_sync,
//    a warp-shuffle scan over the warps gives each warp's offset within a
//    bucket, a block scan over the buckets (descending) gives their starts,
//    and a second pass gives each unit its rank r: items Hkv * r .. + Hkv - 1.
// The list is thus ordered by cost (descending), then b, it, kv head; it is
// fully deterministic.
#pragma once

#include <climits>

#include "common.cuh"

namespace b2pa {

// shared-memory ints the build needs with `warps` warps, nb buckets, B requests
__host__ __device__ constexpr size_t worklist_smem_ints(int warps, int nb, int B)
{
    return (size_t)warps * nb + 64 + nb + 3 * (size_t)B + 1 + 8;
}

struct WorklistResult {
    int n_items;  // items in the list (at most cap)
    int4 want;    // the item at the position asked for (x = -1: there is none)
    bool emit;    // this CTA wrote the list
};

template <int kWarps>
__device__ __forceinline__ int block_exclusive_scan(int v, int* scratch /* >= 33 ints */, int* total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        scratch[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int s = lane < kWarps ? scratch[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o)
                s += y;
        }
        scratch[lane] = s;  // inclusive warp totals
    }
    __syncthreads();
    const int before = warp > 0 ? scratch[warp - 1] : 0;
    if (total)
        *total = scratch[kWarps - 1];
    const int r = before + x - v;
    __syncthreads();
    return r;
}

// Run by all kWarps * 32 threads of the CTA.  sm: worklist_smem_ints(kWarps,
// p.nbuckets, p.B) ints of shared memory.  want_pos: a list position whose
// item is returned (< 0: none).  claim: read by thread 0 only; 0 means this
// CTA writes the list (items, count, per-request chunk counts, error bits),
// anything else that it only computes it.
template <int kWarps>
__device__ __noinline__ WorklistResult build_worklist(const SchedParams& p, int* sm, int want_pos, int claim)
{
    constexpr int kThreads = kWarps * 32;
    const int B = p.B;
    const int nb = p.nbuckets;
    const int Hkv = p.Hkv;
    int* hist = sm;                    // [kWarps][nb]
    int* scratch = hist + kWarps * nb;  // 64
    int* tot = scratch + 64;           // [nb]
    int* req_start = tot + nb;         // [B + 1] first unit of each request
    int* req_q = req_start + B + 1;    // [B] q_len
    int* req_kv = req_q + B;           // [B] kv_len
    int* misc = req_kv + B;            // error bits, emit flag, the wanted item (4 ints)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per_item = p.rows_per_tile * kQTiles;
    if (tid == 0) {
        misc[0] = 0;
        misc[2] = -1;
    }

    // 1. per-request unit counts, as a block-wide scan over contiguous chunks
    unsigned my_err = 0;
    const int chunk = (B + kThreads - 1) / kThreads;
    const int b_begin = min(B, tid * chunk), b_end = min(B, b_begin + chunk);
    int local = 0;
    for (int b = b_begin; b < b_end; ++b) {
        const RequestView r = load_request(QStarts{p.cum_q, p.q_per_req}, p.seq_lens, b, p.max_q_len, p.max_kv_len,
                                           p.page_size, p.max_pages, p.num_tokens);
        if (!r.ok)
            my_err |= (unsigned)B2PA_DEV_BAD_REQUEST;
        int n_it = (r.ok && r.q_len > 0) ? (r.q_len + per_item - 1) / per_item : 0;  // units (per kv head: items)
        if (p.split_tiles > 0)  // one query item per kv head (the host makes q_len fit), cut in kv chunks
            n_it = n_it > 0 ? split_count(item_geometry(r.q_len, r.kv_len, 0, p.rows_per_tile, p.window),
                                          p.split_tiles)
                            : 0;
        req_start[b] = n_it;  // count for now
        req_q[b] = r.q_len;
        req_kv[b] = r.kv_len;
        local += n_it;
        if (p.debug) {
            if (p.cum_kv != nullptr && r.ok && p.cum_kv[b + 1] - p.cum_kv[b] != r.kv_len)
                my_err |= (unsigned)B2PA_DEV_BAD_CUM_KV;
            if (r.ok) {
                const int pages = (r.kv_len + p.page_size - 1) / p.page_size;
                const int* row = page_row(p.block_tables, p.bt_stride, p.kv_indptr, b);
                for (int col = 0; col < pages; ++col) {
                    const int id = row[col];
                    if (id < 0 || id >= p.num_pages)
                        my_err |= (unsigned)B2PA_DEV_BAD_PAGE;
                }
            }
        }
    }
    for (int k = tid; k < kWarps * nb; k += kThreads)
        hist[k] = 0;
    int n_units = 0;
    int run = block_exclusive_scan<kWarps>(local, scratch, &n_units);
    if (my_err)
        atomicOr(reinterpret_cast<unsigned*>(&misc[0]), my_err);
    for (int b = b_begin; b < b_end; ++b) {
        const int n = req_start[b];
        req_start[b] = run;
        run += n;
    }
    const long long n_total = (long long)n_units * Hkv;
    if (tid == 0)
        req_start[B] = n_units;
    __syncthreads();

    // unit u -> (b, it, cost, bucket)
    auto decode = [&](int u, int4& unit, int& bucket) {
        int lo = 0, hi = B - 1;  // last b with req_start[b] <= u
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (req_start[mid] <= u)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int b = lo;
        const int it = u - req_start[b];  // split-KV: the chunk index (the query item is 0)
        ItemGeom g = item_geometry(req_q[b], req_kv[b], p.split_tiles > 0 ? 0 : it, p.rows_per_tile, p.window);
        if (p.split_tiles > 0)
            split_range(&g, it, p.split_tiles);
        const int cost = (g.n_hi - g.n_lo + 1) * g.nq;
        unit = make_int4(b, 0, it, cost);
        bucket = min(cost, nb - 1);
    };

    const int seg = (n_units + kWarps - 1) / kWarps;
    const int s_begin = min(n_units, warp * seg), s_end = min(n_units, s_begin + seg);
    int* my_hist = hist + warp * nb;

    // 2. per-warp bucket counts.  The first kKeep rounds of 32 units stay in
    // registers for the scatter; later rounds are decoded again there.
    constexpr int kKeep = 2;
    int4 kept_unit[kKeep];
    int kept_bucket[kKeep];
    auto count_round = [&](int bucket) {
        const unsigned grp = __match_any_sync(0xffffffffu, bucket);
        if (bucket >= 0 && lane == __ffs(grp) - 1)
            my_hist[bucket] += __popc(grp);
        __syncwarp();
    };
#pragma unroll
    for (int k = 0; k < kKeep; ++k) {
        const int u = s_begin + 32 * k + lane;
        kept_unit[k] = make_int4(0, 0, 0, 0);
        kept_bucket[k] = -1;
        if (u < s_end)
            decode(u, kept_unit[k], kept_bucket[k]);
        if (s_begin + 32 * k < s_end)  // warp-uniform
            count_round(kept_bucket[k]);
    }
    for (int base = s_begin + 32 * kKeep; base < s_end; base += 32) {
        const int u = base + lane;
        int4 unit;
        int bucket = -1;
        if (u < s_end)
            decode(u, unit, bucket);
        count_round(bucket);
    }
    __syncthreads();

    // 3. offsets: buckets in descending order, warps in ascending order.
    // Within a bucket, the warps' counts are scanned by one warp (lane w holds
    // warp w's count); warp u takes buckets u, u + kWarps, ...
    for (int cb = warp; cb < nb; cb += kWarps) {
        const int v = lane < kWarps ? hist[lane * nb + cb] : 0;
        int x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o)
                x += y;
        }
        if (lane < kWarps)
            hist[lane * nb + cb] = x - v;
        if (lane == 31)
            tot[cb] = x;
    }
    if (tid == 0)
        misc[1] = claim == 0 ? 1 : 0;  // the claim's answer is first needed here
    __syncthreads();
    // exclusive scan over the buckets from the top: thread t takes the
    // descending positions t * per .. t * per + per - 1 (bucket nb - 1 - d);
    // tot then holds each bucket's start
    {
        const int per = (nb + kThreads - 1) / kThreads;
        const int d0 = min(nb, tid * per), d1 = min(nb, d0 + per);
        int sum = 0;
        for (int d = d0; d < d1; ++d)
            sum += tot[nb - 1 - d];
        int start = block_exclusive_scan<kWarps>(sum, scratch, nullptr);
        for (int d = d0; d < d1; ++d) {
            const int n = tot[nb - 1 - d];
            tot[nb - 1 - d] = start;
            start += n;
        }
    }
    __syncthreads();
    const bool emit = misc[1] != 0;

    // 4. ranks, in the same order as the counts: a unit of rank r fills items
    // Hkv * r .. Hkv * r + Hkv - 1, one per kv head
    auto scatter_round = [&](const int4& unit, int bucket) {
        const unsigned grp = __match_any_sync(0xffffffffu, bucket);
        const unsigned lower = grp & ((1u << lane) - 1u);
        if (bucket >= 0) {
            const long long pos = (long long)(tot[bucket] + my_hist[bucket] + __popc(lower)) * Hkv;
            if (emit)
                for (int h = 0; h < Hkv; ++h)
                    if (pos + h < p.cap)
                        p.items[pos + h] = make_int4(unit.x, h, unit.z, unit.w);
            if (want_pos >= pos && want_pos < pos + Hkv) {
                misc[2] = unit.x;
                misc[3] = (int)(want_pos - pos);
                misc[4] = unit.z;
                misc[5] = unit.w;
            }
        }
        __syncwarp();
        if (bucket >= 0 && lane == __ffs(grp) - 1)
            my_hist[bucket] += __popc(grp);
        __syncwarp();
    };
#pragma unroll
    for (int k = 0; k < kKeep; ++k)
        if (s_begin + 32 * k < s_end)  // warp-uniform
            scatter_round(kept_unit[k], kept_bucket[k]);
    for (int base = s_begin + 32 * kKeep; base < s_end; base += 32) {
        const int u = base + lane;
        int4 unit = make_int4(0, 0, 0, 0);
        int bucket = -1;
        if (u < s_end)
            decode(u, unit, bucket);
        scatter_round(unit, bucket);
    }
    if (emit) {
        if (p.split_tiles > 0)
            for (int b = tid; b < B; b += kThreads)
                p.nsplit[b] = req_start[b + 1] - req_start[b];
        if (tid == 0) {
            *p.count = (int)min(n_total, (long long)INT_MAX);
            const unsigned e = (unsigned)misc[0] | (n_total > p.cap ? (unsigned)B2PA_DEV_OVERFLOW : 0u);
            if (e)
                atomicOr(p.err, e);
        }
    }
    __syncthreads();
    WorklistResult r;
    r.n_items = (int)min(n_total, (long long)p.cap);
    r.want = misc[2] >= 0 ? make_int4(misc[2], misc[3], misc[4], misc[5]) : make_int4(-1, 0, 0, 0);
    r.emit = emit;
    return r;
}

}  // namespace b2pa
