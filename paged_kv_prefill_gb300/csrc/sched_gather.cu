// sched_gather.cu -- the work-list scheduler of the tensor-core path and the
// debug gather that exercises its paged K/V loads.
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"
#include "worklist.cuh"

namespace b2pa {

// ---------------------------------------------------------------------------
// Scheduler kernel: one CTA of 1024 threads builds and writes the work list
// (build_worklist), for b2pa_debug_worklist.  The attention kernel builds the
// same list itself at its start.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSchedThreads, 1) schedule_kernel(const SchedParams p)
{
    extern __shared__ int sm[];
    build_worklist<kSchedThreads / 32>(p, sm, -1, 0);
}

cudaError_t launch_schedule(const SchedParams& p, cudaStream_t stream)
{
    const size_t nb = (size_t)p.nbuckets;
    const size_t smem = sizeof(int) * worklist_smem_ints(kSchedThreads / 32, (int)nb, p.B);
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
        const size_t most = sizeof(int) * worklist_smem_ints(kSchedThreads / 32, kSchedBuckets, kSchedMaxBatch);
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
