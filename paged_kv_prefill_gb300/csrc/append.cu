// append.cu -- the write of new tokens' K and V into the paged pools, the
// step before the attention (TokenSpeed trtllm backend, _save_kv_and_prepare_q:
// fused_fp8_set_kv_buffer for an e4m3 cache, set_kv_buffer otherwise).
//
// Token n's rows k[n, h, :] and v[n, h, :] go to cache slot cache_loc[n] =
// page * page_size + slot of the pools.  A bf16 pool gets the bf16 bits; an
// e4m3 pool gets x / scale (one IEEE binary32 division) converted by
// cvt.rn.satfinite: round to nearest even, saturating at +-448.
//
// HBM-bound: one thread moves one 8-element chunk (16 bytes in; 16 bytes out
// for bf16, 8 for e4m3) of a (token, kv head) row of K and the same chunk of
// V; consecutive threads take consecutive chunks of a row, so a warp reads and
// writes whole rows.  Grid-stride over T * Hkv * D / 8 chunks.
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

template <bool FP8>
__global__ void __launch_bounds__(256) append_kv_kernel(const AppendParams p)
{
    const int chunks = p.D >> 3;
    const long long total = (long long)p.T * p.Hkv * chunks;
    const long long slots = (long long)p.num_pages * p.page_size;
    const long long step = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += step) {
        const int c = (int)(i % chunks);
        const long long r = i / chunks;
        const int h = (int)(r % p.Hkv);
        const long long n = r / p.Hkv;
        const int loc = p.cache_loc[n];
        if (loc < 0 || (long long)loc >= slots) {
            if (h == 0 && c == 0)
                atomicOr(p.err, (unsigned)B2PA_DEV_BAD_SLOT);
            continue;
        }
        const long long page = loc / p.page_size, slot = loc - page * p.page_size;
        const long long src = n * p.new_st_tok + (long long)h * p.new_st_head + 8 * c;
        const uint4 kx = *reinterpret_cast<const uint4*>(p.k_new + src);
        const uint4 vx = *reinterpret_cast<const uint4*>(p.v_new + src);
        const long long dk = page * p.k_st[0] + h * p.k_st[1] + slot * p.k_st[2] + 8 * c;
        const long long dv = page * p.v_st[0] + h * p.v_st[1] + slot * p.v_st[2] + 8 * c;
        if constexpr (FP8) {
            *reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.k_pool) + dk) = quantise8(kx, p.k_scale);
            *reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.v_pool) + dv) = quantise8(vx, p.v_scale);
        } else {
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.k_pool) + dk) = kx;
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.v_pool) + dv) = vx;
        }
    }
}

cudaError_t launch_append(const AppendParams& p, bool fp8, int grid, cudaStream_t stream)
{
    if (p.T == 0 || grid <= 0)
        return cudaSuccess;
    if (fp8)
        append_kv_kernel<true><<<grid, 256, 0, stream>>>(p);
    else
        append_kv_kernel<false><<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace b2pa
