// append.cuh -- parameters of the K/V write kernel (append.cu), filled by
// b2pa_append_kv in b2pa.cu.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace b2pa {

struct AppendParams {
    const uint16_t* k_new;  // bf16 [T, Hkv, D]
    const uint16_t* v_new;
    long long new_st_tok, new_st_head;  // element strides of k_new and v_new (head_dim contiguous)
    void* k_pool;                       // bf16 or e4m3 elements
    void* v_pool;
    long long k_st[3], v_st[3];         // element strides by (page, kv head, slot); head_dim contiguous
    const int* cache_loc;               // [T]: page * page_size + slot
    int T, Hkv, D, page_size, num_pages;
    float k_scale, v_scale;             // e4m3 pools only
    unsigned* err;
};

// one launch over every chunk; each thread moves 8 elements of K and of V per chunk
cudaError_t launch_append(const AppendParams& p, bool fp8, cudaStream_t stream);

}  // namespace b2pa
