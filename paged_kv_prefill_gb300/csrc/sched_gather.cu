// sched_gather.cu -- the work-list scheduler of the tensor-core path and the
// debug gather that exercises its paged K/V loads.
#include <climits>
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace b2pa {

// ---------------------------------------------------------------------------
// Scheduler: one CTA of 1024 threads.
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
//    and a second pass scatters each unit's Hkv items to Hkv * its rank.
// The list is thus ordered by cost (descending), then b, it, kv head; it is
// fully deterministic.  Writes items[0 .. n) and *count = n; sets
// B2PA_DEV_BAD_REQUEST for rejected requests (their items are not emitted).
// ---------------------------------------------------------------------------
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
        int s = lane < (int)(blockDim.x >> 5) ? scratch[lane] : 0;
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
        *total = scratch[(blockDim.x >> 5) - 1];
    const int r = before + x - v;
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kSchedThreads, 1) schedule_kernel(const SchedParams p)
{
    // let the attention kernel start its prologue while the list is built
    pdl_launch_dependents();
    extern __shared__ int sm[];
    const int B = p.B;
    const int nb = p.nbuckets;
    const int Hkv = p.Hkv;
    int* hist = sm;                                  // [32 warps][nb]
    int* scratch = hist + 32 * nb;                   // 64
    int* tot = scratch + 64;                         // [nb]
    int* req_start = tot + nb;                       // [B + 1] first unit of each request
    int* req_q = req_start + B + 1;                  // [B] q_len
    int* req_kv = req_q + B;                         // [B] kv_len
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per_item = p.rows_per_tile * kQTiles;
    if (tid == 0)
        *p.counter = 0;

    // 1. per-request unit counts, as a block-wide scan over contiguous chunks
    const int chunk = (B + kSchedThreads - 1) / kSchedThreads;
    const int b_begin = min(B, tid * chunk), b_end = min(B, b_begin + chunk);
    int local = 0;
    for (int b = b_begin; b < b_end; ++b) {
        const RequestView r = load_request(QStarts{p.cum_q, p.q_per_req}, p.seq_lens, b, p.max_q_len, p.max_kv_len,
                                           p.page_size, p.max_pages, p.num_tokens);
        if (!r.ok)
            atomicOr(p.err, (unsigned)B2PA_DEV_BAD_REQUEST);
        int n_it = (r.ok && r.q_len > 0) ? (r.q_len + per_item - 1) / per_item : 0;  // units (per kv head: items)
        if (p.split_tiles > 0) {
            // one query item per kv head (the host makes q_len fit), cut in kv chunks
            const int ns = n_it > 0 ? split_count(item_geometry(r.q_len, r.kv_len, 0, p.rows_per_tile, p.window),
                                                  p.split_tiles)
                                    : 0;
            p.nsplit[b] = ns;
            n_it = ns;
        }
        req_start[b] = n_it;  // count for now
        req_q[b] = r.q_len;
        req_kv[b] = r.kv_len;
        local += n_it;
        if (p.debug) {
            if (p.cum_kv != nullptr && r.ok && p.cum_kv[b + 1] - p.cum_kv[b] != r.kv_len)
                atomicOr(p.err, (unsigned)B2PA_DEV_BAD_CUM_KV);
            if (r.ok) {
                const int pages = (r.kv_len + p.page_size - 1) / p.page_size;
                const int* row = page_row(p.block_tables, p.bt_stride, p.kv_indptr, b);
                for (int col = 0; col < pages; ++col) {
                    const int id = row[col];
                    if (id < 0 || id >= p.num_pages)
                        atomicOr(p.err, (unsigned)B2PA_DEV_BAD_PAGE);
                }
            }
        }
    }
    for (int k = tid; k < 32 * nb; k += kSchedThreads)
        hist[k] = 0;
    int n_units = 0;
    int run = block_exclusive_scan(local, scratch, &n_units);
    for (int b = b_begin; b < b_end; ++b) {
        const int n = req_start[b];
        req_start[b] = run;
        run += n;
    }
    const long long n_total = (long long)n_units * Hkv;
    if (tid == 0) {
        req_start[B] = n_units;
        if (n_total > p.cap)
            atomicOr(p.err, (unsigned)B2PA_DEV_OVERFLOW);
    }
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

    const int seg = (n_units + 31) / 32;
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
    // warp w's count); warp u takes buckets u, u + 32, ...
    for (int c = warp; c < nb; c += 32) {
        const int v = hist[lane * nb + c];
        int x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o)
                x += y;
        }
        hist[lane * nb + c] = x - v;
        if (lane == 31)
            tot[c] = x;
    }
    __syncthreads();
    // exclusive scan over buckets from the top: thread t takes bucket nb - 1 - t
    // (nb <= kSchedBuckets == kSchedThreads); tot then holds each bucket's start
    const int start = block_exclusive_scan(tid < nb ? tot[nb - 1 - tid] : 0, scratch, nullptr);
    if (tid < nb)
        tot[nb - 1 - tid] = start;
    __syncthreads();

    // 4. scatter, in the same order as the counts: a unit of rank r fills
    // items Hkv * r .. Hkv * r + Hkv - 1, one per kv head
    auto scatter_round = [&](const int4& unit, int bucket) {
        const unsigned grp = __match_any_sync(0xffffffffu, bucket);
        const unsigned lower = grp & ((1u << lane) - 1u);
        if (bucket >= 0) {
            const long long pos = (long long)(tot[bucket] + my_hist[bucket] + __popc(lower)) * Hkv;
            for (int h = 0; h < Hkv; ++h)
                if (pos + h < p.cap)
                    p.items[pos + h] = make_int4(unit.x, h, unit.z, unit.w);
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
    if (tid == 0)
        *p.count = (int)min(n_total, (long long)INT_MAX);
}

cudaError_t launch_schedule(const SchedParams& p, cudaStream_t stream)
{
    const size_t nb = (size_t)p.nbuckets;
    const size_t smem = sizeof(int) * (32 * nb + 64 + nb + 3 * (size_t)p.B + 1);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    // opt in once per device to the most shared memory any call can need
    // (every bucket in use and the largest batch), not on every call
    static std::once_flag attr_once[64];
    static cudaError_t attr_err[64];
    std::call_once(attr_once[dev], [&] {
        const size_t most = sizeof(int) * (32 * (size_t)kSchedBuckets + 64 + kSchedBuckets + 3 * (size_t)kSchedMaxBatch + 1);
        attr_err[dev] = cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most);
    });
    if (attr_err[dev] != cudaSuccess)
        return attr_err[dev];
    schedule_kernel<<<1, kSchedThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Debug gather: one CTA per (kv tile, kv head, request).  Warp 0 issues the
// same per-page tensor-map loads as the attention producer into a
// 128-row tile, then the CTA writes the rows below kv_len out contiguously,
// undoing the 128-byte swizzle.
// ---------------------------------------------------------------------------
template <bool FP8>
__global__ void __launch_bounds__(128) gather_kernel(const __grid_constant__ GatherParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* tile = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int D = p.D;
    const int halves = FP8 ? 1 : D / 64;
    const int half_bytes = kKvTile * 128;
    uint64_t* bar = reinterpret_cast<uint64_t*>(tile + halves * half_bytes);
    const int j = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int kv_len = p.seq_lens[b];
    if (kv_len < 0 || (long long)j * kKvTile >= kv_len)
        return;
    const int P = p.page_size;
    if (p.kv_indptr == nullptr && (kv_len + P - 1) / P > p.max_pages) {
        if (threadIdx.x == 0)
            atomicOr(p.err, (unsigned)B2PA_DEV_BAD_REQUEST);
        return;
    }
    const long long row0 = p.cum_kv[b];
    if (p.cum_kv[b + 1] - row0 != kv_len || row0 < 0 || row0 + kv_len > p.out_rows) {
        if (threadIdx.x == 0)
            atomicOr(p.err, (unsigned)B2PA_DEV_BAD_CUM_KV);
        return;
    }
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    const int rows = min(kKvTile, kv_len - j * kKvTile);
    const int box_rows = P >= kKvTile ? kKvTile : P;
    const int log2_p = 31 - __clz(P);  // page sizes of the tensor-core loads are powers of two
    const int* bt_row = page_row(p.block_tables, p.bt_stride, p.kv_indptr, b);
    for (int kind = 0; kind < 2; ++kind) {
        if (threadIdx.x < 32) {
            // the attention producer's page addressing
            const int lane = threadIdx.x;
            const TileLoad tl = tile_load(bt_row, j, lane, log2_p, (kv_len + P - 1) >> log2_p);
            const int slot0 = tl.slot0, page = tl.page;
            const bool valid = tl.valid;
            if (valid && (page < 0 || page >= p.num_pages))
                atomicOr(p.err, (unsigned)B2PA_DEV_BAD_PAGE);
            const uint32_t nvalid = __popc(__ballot_sync(0xffffffffu, valid));
            if (lane == 0)
                mbar_arrive_expect_tx(bar, nvalid * (uint32_t)box_rows * 128u * (uint32_t)halves);
            __syncwarp();
            if (valid) {
                const uint32_t dst = smem_u32(tile) + (uint32_t)(lane * box_rows * 128);
                for (int h = 0; h < halves; ++h)
                    tma_load_4d(dst + h * half_bytes, kind ? &p.tm_v : &p.tm_k, bar, h * 64, slot0, kvh, page);
            }
        }
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(smem_u32(bar), kind)) {
            if (global_ns() - t0 > kWaitLimitNs) {
                if (threadIdx.x == 0)
                    atomicOr(p.err, (unsigned)B2PA_DEV_TIMEOUT);
                break;
            }
        }
        uint8_t* out = kind ? p.v_out : p.k_out;
        const int row_bytes = D * p.esize;       // bytes of one (token, head) row
        const int chunks = row_bytes / 16;        // 16-byte chunks per row
        for (int k = threadIdx.x; k < rows * chunks; k += blockDim.x) {
            const int r = k / chunks, q = k % chunks;
            const int h = q / 8, cq = q % 8;       // column block, chunk inside its 128-byte row
            const uint4 v = *reinterpret_cast<const uint4*>(tile + h * half_bytes + r * 128 + ((cq ^ (r & 7)) << 4));
            const long long orow = (row0 + (long long)j * kKvTile + r) * p.Hkv + kvh;
            *reinterpret_cast<uint4*>(out + orow * row_bytes + q * 16) = v;
        }
        __syncthreads();
    }
}

cudaError_t launch_gather(const GatherParams& p, bool fp8, int max_kv_len, cudaStream_t stream)
{
    const int tiles = (max_kv_len + kKvTile - 1) / kKvTile;
    if (tiles == 0 || p.B == 0)
        return cudaSuccess;
    const int halves = fp8 ? 1 : p.D / 64;
    const size_t smem = (size_t)halves * kKvTile * 128 + 64 + 1024;
    auto kern = fp8 ? gather_kernel<true> : gather_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    kern<<<dim3(tiles, p.Hkv, p.B), 128, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace b2pa

namespace b2pa {

// ---------------------------------------------------------------------------
// Ragged page table (FlashInfer's paged_kv_indices / paged_kv_indptr /
// paged_kv_last_page_len): each request's kv length from its page count and
// the valid tokens of its last page.  A request with a negative page count, or
// with pages and a last_page_len outside [1, page_size], is malformed: its
// length becomes -1, which every later check rejects.
// ---------------------------------------------------------------------------
__global__ void ragged_lengths_kernel(const int* indptr, const int* last, int B, int P, int* kv_len, unsigned* err)
{
    for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < B; b += gridDim.x * blockDim.x) {
        const int pages = indptr[b + 1] - indptr[b];
        int len = 0;
        if (pages < 0 || indptr[b] < 0) {
            len = -1;
        } else if (pages > 0) {
            const int lp = last[b];
            len = (lp < 1 || lp > P) ? -1 : (int)min((long long)(pages - 1) * P + lp, 0x7FFFFFFFLL);
        }
        if (len < 0)
            atomicOr(err, (unsigned)B2PA_DEV_BAD_REQUEST);
        kv_len[b] = len;
    }
}

cudaError_t launch_ragged_lengths(const int* indptr, const int* last_page_len, int B, int page_size, int* kv_len,
                                  unsigned* err, cudaStream_t stream)
{
    if (B == 0)
        return cudaSuccess;
    const int blocks = (B + 255) / 256;
    ragged_lengths_kernel<<<blocks < 64 ? blocks : 64, 256, 0, stream>>>(indptr, last_page_len, B, page_size, kv_len,
                                                                           err);
    return cudaGetLastError();
}

}  // namespace b2pa
