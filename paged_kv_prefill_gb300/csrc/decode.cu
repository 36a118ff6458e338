// decode.cu -- the combine step of split-KV decode batches.
//
// A decode batch (every request has the same small number of query tokens,
// the TokenSpeed trtllm backend's q_len_per_req) gives too few query rows to
// fill the GPU with one work item per request and kv head, so the attention
// kernel cuts each request's kv range into chunks and writes, for every chunk,
// the unnormalised partial output O_c = sum_j 2^(s_j - m_c) V_j, its running
// maximum m_c (log2 units of the scaled scores) and its sum
// l_c = sum_j 2^(s_j - m_c).  With m = max_c m_c and w_c = 2^(m_c - m):
//
//   out = bmm2_scale * sum_c w_c O_c / (sum_c w_c l_c + [sinks] 2^(sink_h log2(e) - m))
//
// which is the softmax of the whole row (FlashInfer API reference, parameter
// list: sinks join the denominator once).  One warp per output row.
#include "common.cuh"
#include "ptx.cuh"

namespace b2pa {

constexpr int kCombineWarps = 8;

__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const CombineParams p)
{
    constexpr float kLog2e = 1.4426950408889634f;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kCombineWarps + warp;  // token * H + head
    const long long rows = (long long)p.B * p.q_per_req * p.H;
    if (row >= rows)
        return;
    const int tok = (int)(row / p.H), h = (int)(row % p.H);
    const int b = tok / p.q_per_req;
    const int ns = p.nsplit[b];
    if (ns <= 1)
        return;  // written by the attention kernel (or a request without work)
    const float bmm2 = p.bmm2_dev != nullptr ? *p.bmm2_dev : p.bmm2;
    const float* ml = p.part_ml + row * p.part_slots * 2;
    // the largest chunk maximum
    float m = -INFINITY;
    for (int c = lane; c < ns; c += 32)
        m = fmaxf(m, ml[2 * c]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float den = 0.f;
    for (int c = lane; c < ns; c += 32) {
        const float mc = ml[2 * c];
        den += mc == -INFINITY ? 0.f : ex2_approx(mc - m) * ml[2 * c + 1];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        den += __shfl_xor_sync(0xffffffffu, den, o);
    if (p.sinks != nullptr && m != -INFINITY)
        den += ex2_approx(fmaf(p.sinks[h], kLog2e, -m));
    const float inv = (m != -INFINITY && den > 0.f) ? bmm2 / den : 0.f;
    uint16_t* orow = p.out + (long long)tok * p.out_st_tok + (long long)h * p.out_st_head;
    const float* po = p.part_o + row * p.part_slots * p.D;
    // lane takes 2 consecutive dimensions at a time
    for (int d = 2 * lane; d < p.D; d += 64) {
        float a0 = 0.f, a1 = 0.f;
        for (int c = 0; c < ns; ++c) {
            const float mc = ml[2 * c];
            const float w = mc == -INFINITY ? 0.f : ex2_approx(mc - m);
            const float2 v = *reinterpret_cast<const float2*>(po + (long long)c * p.D + d);
            a0 = fmaf(w, v.x, a0);
            a1 = fmaf(w, v.y, a1);
        }
        *reinterpret_cast<uint32_t*>(orow + d) = pack_bf16x2(a0 * inv, a1 * inv);
    }
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream)
{
    const long long rows = (long long)p.B * p.q_per_req * p.H;
    if (rows == 0)
        return cudaSuccess;
    const long long blocks = (rows + kCombineWarps - 1) / kCombineWarps;
    combine_kernel<<<(unsigned)blocks, kCombineWarps * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace b2pa
