// append.cu -- the write of new tokens' K and V into the paged pools, the
// step before the attention (TokenSpeed trtllm backend, _save_kv_and_prepare_q:
// fused_fp8_set_kv_buffer for an e4m3 cache, set_kv_buffer otherwise).
//
// Token n's rows k[n, h, :] and v[n, h, :] go to cache slot cache_loc[n] =
// page * page_size + slot of the pools.  A bf16 pool gets the bf16 bits; an
// e4m3 pool gets x / scale (one IEEE binary32 division) converted by
// cvt.rn.satfinite: round to nearest even, saturating at +-448.
//
// HBM-bound: a thread moves 8-element chunks (16 bytes in; 16 bytes out for
// bf16, 8 for e4m3) of (token, kv head) rows of K and the same chunks of V;
// consecutive threads take consecutive chunks of a row, so a warp reads and
// writes whole rows.  One grid covers all T * Hkv * D / 8 chunks.
#include "../../include/b2pa.h"
#include "append.cuh"

namespace b2pa {

// two binary32 values -> two e4m3 codes, `lo` in the low byte
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// eight bf16 (four words, element 2i in the low half of word i) / scale -> eight e4m3 codes
__device__ __forceinline__ uint2 quantise8(uint4 x, float scale)
{
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lo = __fdiv_rn(__uint_as_float(w[i] << 16), scale);
        const float hi = __fdiv_rn(__uint_as_float(w[i] & 0xFFFF0000u), scale);
        c[i] = e4m3x2(lo, hi);
    }
    return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// Each thread moves kUnroll chunks, kUnroll * 256 apart, issuing every load
// before its first store so that the copies overlap (one chunk per thread for
// an e4m3 pool, whose 16 divisions per chunk are better spread over more
// threads).  Idx: 32-bit index math when the chunk count allows it, else 64-bit.
constexpr int kAppendThreads = 256;
template <bool FP8>
constexpr int append_unroll() { return FP8 ? 1 : 4; }

template <bool FP8, typename Idx>
__global__ void __launch_bounds__(kAppendThreads) append_kv_kernel(const AppendParams p, const Idx total)
{
    constexpr int kUnroll = append_unroll<FP8>();
    const Idx chunks = (Idx)(p.D >> 3);
    const long long slots = (long long)p.num_pages * p.page_size;
    const Idx base = (Idx)blockIdx.x * (kAppendThreads * kUnroll) + (Idx)threadIdx.x;
    uint4 kx[kUnroll], vx[kUnroll];
    int loc[kUnroll], h[kUnroll], c[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const Idx i = base + (Idx)u * kAppendThreads;
        loc[u] = -1;
        if (i < total) {
            c[u] = (int)(i % chunks);
            const Idx r = i / chunks;
            h[u] = (int)(r % (Idx)p.Hkv);
            const Idx n = r / (Idx)p.Hkv;
            loc[u] = p.cache_loc[n];
            const long long src = (long long)n * p.new_st_tok + (long long)h[u] * p.new_st_head + 8 * c[u];
            kx[u] = *reinterpret_cast<const uint4*>(p.k_new + src);
            vx[u] = *reinterpret_cast<const uint4*>(p.v_new + src);
        }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const Idx i = base + (Idx)u * kAppendThreads;
        if (i >= total)
            continue;
        if (loc[u] < 0 || (long long)loc[u] >= slots) {
            if (h[u] == 0 && c[u] == 0)
                atomicOr(p.err, (unsigned)B2PA_DEV_BAD_SLOT);
            continue;
        }
        const long long page = loc[u] / p.page_size, slot = loc[u] - page * p.page_size;
        const long long dk = page * p.k_st[0] + h[u] * p.k_st[1] + slot * p.k_st[2] + 8 * c[u];
        const long long dv = page * p.v_st[0] + h[u] * p.v_st[1] + slot * p.v_st[2] + 8 * c[u];
        if constexpr (FP8) {
            *reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.k_pool) + dk) = quantise8(kx[u], p.k_scale);
            *reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.v_pool) + dv) = quantise8(vx[u], p.v_scale);
        } else {
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.k_pool) + dk) = kx[u];
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.v_pool) + dv) = vx[u];
        }
    }
}

template <bool FP8>
static cudaError_t launch_typed(const AppendParams& p, long long total, cudaStream_t stream)
{
    const long long per_block = (long long)kAppendThreads * append_unroll<FP8>();
    const long long blocks = (total + per_block - 1) / per_block;
    if (blocks > 0x7FFFFFFFLL)
        return cudaErrorInvalidConfiguration;
    if (total <= 0x7FFFFFFFLL - per_block)
        append_kv_kernel<FP8, unsigned><<<(unsigned)blocks, kAppendThreads, 0, stream>>>(p, (unsigned)total);
    else
        append_kv_kernel<FP8, unsigned long long><<<(unsigned)blocks, kAppendThreads, 0, stream>>>(
            p, (unsigned long long)total);
    return cudaGetLastError();
}

cudaError_t launch_append(const AppendParams& p, bool fp8, cudaStream_t stream)
{
    const long long total = (long long)p.T * p.Hkv * (p.D >> 3);
    if (total == 0)
        return cudaSuccess;
    return fp8 ? launch_typed<true>(p, total, stream) : launch_typed<false>(p, total, stream);
}

}  // namespace b2pa
