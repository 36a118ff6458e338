// generic.cu -- CUDA-core paged-KV context attention for any shape: head_dim
// 1..256, any page size, any GQA ratio, any strides, bf16 or e4m3 pools.
// It serves the shapes the tensor-core path does not take.
//
// One warp per output row (token, query head).  The warp walks the row's
// visible keys 32 at a time: lane l scores key (chunk + l) against the query
// (held in shared memory), the warp takes the running maximum and sum (an
// online softmax in log2 units), and each lane accumulates the output
// dimensions d = lane, lane + 32, ... for the chunk's 32 keys.  A key whose
// page id lies outside the pool reads as K = V = 0, as a tensor-map load
// outside the tensor would, and raises B2PA_DEV_BAD_PAGE.
#include <cuda_fp8.h>

#include "common.cuh"

namespace b2pa {

constexpr int kGenericWarps = 8;
constexpr int kGenericMaxD = 256;

template <bool FP8>
__device__ __forceinline__ float load_elem(const void* base, long long off)
{
    if (FP8) {
        const __nv_fp8_storage_t x = static_cast<const __nv_fp8_storage_t*>(base)[off];
        return __half2float(__half(__nv_cvt_fp8_to_halfraw(x, __NV_E4M3)));
    } else {
        const unsigned short x = static_cast<const unsigned short*>(base)[off];
        return __uint_as_float(static_cast<uint32_t>(x) << 16);
    }
}

__device__ __forceinline__ uint16_t to_bf16(float f)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(0.f), "f"(f));
    return static_cast<uint16_t>(r & 0xFFFFu);
}

template <bool FP8>
__global__ void __launch_bounds__(kGenericWarps * 32) generic_attention_kernel(const GenericParams p)
{
    extern __shared__ float qs_all[];
    constexpr float kLog2e = 1.4426950408889634f;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float* qs = qs_all + warp * p.D;
    if (blockIdx.x == 0) {
        for (int b = threadIdx.x; b < p.B; b += blockDim.x)
            if (!load_request(QStarts{p.cum_q, p.q_per_req}, p.seq_lens, b, p.max_q_len, p.max_kv_len, p.page_size,
                              p.max_pages, p.T)
                     .ok)
                atomicOr(p.err, (unsigned)B2PA_DEV_BAD_REQUEST);
    }
    const long long rowid = (long long)blockIdx.x * kGenericWarps + warp;
    if (rowid >= (long long)p.T * p.H)
        return;
    const int tok = (int)(rowid / p.H), h = (int)(rowid % p.H);

    // the request owning this token: last b with cum_q[b] <= tok
    const QStarts cq{p.cum_q, p.q_per_req};
    int lo_b = 0, hi_b = p.B - 1;
    if (p.cum_q == nullptr) {
        lo_b = hi_b = min(p.B - 1, tok / p.q_per_req);
    }
    while (lo_b < hi_b) {
        const int mid = (lo_b + hi_b + 1) >> 1;
        if (cq[mid] <= tok)
            lo_b = mid;
        else
            hi_b = mid - 1;
    }
    const int b = lo_b;
    const RequestView r = load_request(cq, p.seq_lens, b, p.max_q_len, p.max_kv_len, p.page_size, p.max_pages, p.T);
    if (!r.ok)
        return;
    if (tok < r.q_start || tok >= r.q_start + r.q_len)
        return;  // a token no request owns
    const int i = tok - r.q_start;
    const int pos = r.kv_len - r.q_len + i;
    const int lo = p.window < 0 ? 0 : max(0, pos - p.window);
    const int G = p.H / p.Hkv;
    const int hk = h / G;
    const Scales scl = load_scales(p.scale_log2, p.bmm2, p.bmm1_dev, p.bmm2_dev);
    if (!scl.ok) {
        if (lane == 0)
            atomicOr(p.err, (unsigned)B2PA_DEV_BAD_SCALE);
        return;
    }
    const float sl2 = scl.scale_log2;

    const uint16_t* qrow = p.q + (long long)tok * p.q_st_tok + (long long)h * p.q_st_head;
    for (int d = lane; d < p.D; d += 32)
        qs[d] = __uint_as_float(static_cast<uint32_t>(qrow[d]) << 16);
    __syncwarp();

    constexpr int kPer = kGenericMaxD / 32;
    float o[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k)
        o[k] = 0.f;
    float m = -INFINITY, l = 0.f;
    const int* bt_row = page_row(p.block_tables, p.bt_stride, p.kv_indptr, b);

    for (int base = lo; base <= pos; base += 32) {
        const int key = base + lane;
        const bool vis = key <= pos;
        long long k_off = -1, v_off = -1;
        float s = -INFINITY;
        if (vis) {
            const int page = bt_row[key / p.page_size];
            const int slot = key % p.page_size;
            if (page >= 0 && page < p.num_pages) {
                k_off = (long long)page * p.k_st_page + (long long)hk * p.k_st_head + (long long)slot * p.k_st_slot;
                v_off = (long long)page * p.v_st_page + (long long)hk * p.v_st_head + (long long)slot * p.v_st_slot;
                float dot = 0.f;
                for (int d = 0; d < p.D; ++d)
                    dot = fmaf(qs[d], load_elem<FP8>(p.k, k_off + d), dot);
                s = dot * sl2;
            } else {
                atomicOr(p.err, (unsigned)B2PA_DEV_BAD_PAGE);
                s = 0.f;  // K = 0
            }
        }
        float cm = s;
#pragma unroll
        for (int w = 16; w > 0; w >>= 1)
            cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, w));
        const float m_new = fmaxf(m, cm);
        const float alpha = m == -INFINITY ? 0.f : exp2f(m - m_new);
        const float pj = vis ? exp2f(s - m_new) : 0.f;
        float ps = pj;
#pragma unroll
        for (int w = 16; w > 0; w >>= 1)
            ps += __shfl_xor_sync(0xffffffffu, ps, w);
        l = l * alpha + ps;
#pragma unroll
        for (int k = 0; k < kPer; ++k)
            o[k] *= alpha;
        const int n = min(32, pos - base + 1);
        for (int kk = 0; kk < n; ++kk) {
            const float pk = __shfl_sync(0xffffffffu, pj, kk);
            const long long vo = __shfl_sync(0xffffffffu, v_off, kk);
            if (vo < 0)
                continue;  // V = 0
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                const int d = lane + 32 * k;
                if (d < p.D)
                    o[k] = fmaf(pk, load_elem<FP8>(p.v, vo + d), o[k]);
            }
        }
        m = m_new;
    }
    float total = l;
    if (p.sinks != nullptr && m != -INFINITY)
        total += exp2f(fmaf(p.sinks[h], kLog2e, -m));
    const float inv = (m != -INFINITY && total > 0.f) ? scl.bmm2 / total : 0.f;
    uint16_t* orow = p.out + (long long)tok * p.out_st_tok + (long long)h * p.out_st_head;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int d = lane + 32 * k;
        if (d < p.D)
            orow[d] = to_bf16(o[k] * inv);
    }
}

cudaError_t launch_attention_generic(const GenericParams& p, bool fp8, cudaStream_t stream)
{
    const long long rows = (long long)p.T * p.H;
    if (rows == 0)
        return cudaSuccess;
    const long long blocks = (rows + kGenericWarps - 1) / kGenericWarps;
    if (blocks > 0x7FFFFFFFLL)
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(float) * kGenericWarps * p.D;
    if (fp8)
        generic_attention_kernel<true><<<(unsigned)blocks, kGenericWarps * 32, smem, stream>>>(p);
    else
        generic_attention_kernel<false><<<(unsigned)blocks, kGenericWarps * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace b2pa
