// b2pa.cu -- host side of the C ABI declared in include/b2pa.h: argument
// checks, kernel-path choice, tensor-map encoding, per-stream workspaces and
// launches.  No entry point of the attention call synchronises the host.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/b2pa.h"
#include "append.cuh"
#include "common.cuh"

using namespace b2pa;

namespace {

thread_local std::string g_last_error;
std::atomic<int> g_path{B2PA_PATH_AUTO};
std::atomic<int> g_debug{0};
std::atomic<void*> g_ev_start{nullptr};
std::atomic<void*> g_ev_stop{nullptr};
std::atomic<unsigned long long> g_wait_limit_ns{kWaitLimitNs};
std::atomic<int> g_inject_stall{0};

int fail(int status, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int status, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return status;
}

int cuda_fail(cudaError_t e, const char* what)
{
    return fail(B2PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ------------------------------------------------------------------ device info

struct DevInfo {
    bool init = false;
    int sms = 0;
    int major = 0, minor = 0;
};
std::mutex g_dev_mu;
DevInfo g_dev[64];

int device_info(int* dev_out, DevInfo* info)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64)
        return fail(B2PA_ERR_UNSUPPORTED, "device ordinal %d", dev);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevInfo& d = g_dev[dev];
    if (!d.init) {
        if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        d.init = true;
    }
    *dev_out = dev;
    *info = d;
    return B2PA_OK;
}

// ------------------------------------------------------------------ workspaces

// Per (device, stream): [0] error word, [4] item count, [8] work counter,
// [12] list claim, [16] list ready, [20] CTAs done (the attention kernel's
// work distribution; zero between launches), [256 ..) work items.
struct Workspace {
    int dev;
    cudaStream_t stream;
    uint8_t* mem;
    size_t bytes;
};
std::mutex g_ws_mu;
std::vector<Workspace> g_ws;
constexpr size_t kWsHeader = 256;

int get_workspace_bytes(int dev, cudaStream_t stream, size_t need, Workspace* out);

int get_workspace(int dev, cudaStream_t stream, size_t items, Workspace* out)
{
    return get_workspace_bytes(dev, stream, kWsHeader + items * sizeof(int4), out);
}

int get_workspace_bytes(int dev, cudaStream_t stream, size_t need, Workspace* out)
{
    std::lock_guard<std::mutex> lk(g_ws_mu);
    for (auto& w : g_ws) {
        if (w.dev == dev && w.stream == stream) {
            if (w.bytes >= need) {
                *out = w;
                return B2PA_OK;
            }
            cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
            cudaStreamIsCapturing(stream, &cs);
            if (cs != cudaStreamCaptureStatusNone)
                return fail(B2PA_ERR_CUDA,
                            "the workspace of this stream must grow during stream capture; make one call with "
                            "the largest shapes before capturing");
            cudaError_t e = cudaStreamSynchronize(stream);
            if (e != cudaSuccess)
                return cuda_fail(e, "cudaStreamSynchronize");
            uint32_t err_word = 0;
            cudaMemcpy(&err_word, w.mem, sizeof err_word, cudaMemcpyDeviceToHost);
            cudaFree(w.mem);
            w.mem = nullptr;
            const size_t bytes = need * 2;
            if ((e = cudaMalloc(&w.mem, bytes)) != cudaSuccess) {
                w.bytes = 0;
                return cuda_fail(e, "cudaMalloc(workspace)");
            }
            w.bytes = bytes;
            cudaMemset(w.mem, 0, kWsHeader);
            cudaMemcpy(w.mem, &err_word, sizeof err_word, cudaMemcpyHostToDevice);  // keep pending error bits
            *out = w;
            return B2PA_OK;
        }
    }
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(stream, &cs);
    if (cs != cudaStreamCaptureStatusNone)
        return fail(B2PA_ERR_CUDA,
                    "this stream has no workspace yet and is being captured; make one call before capturing");
    Workspace w{dev, stream, nullptr, 0};
    const size_t bytes = need < (1u << 20) ? (1u << 20) : need * 2;
    cudaError_t e = cudaMalloc(&w.mem, bytes);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMalloc(workspace)");
    w.bytes = bytes;
    if ((e = cudaMemset(w.mem, 0, kWsHeader)) != cudaSuccess)
        return cuda_fail(e, "cudaMemset(workspace)");
    g_ws.push_back(w);
    *out = w;
    return B2PA_OK;
}

bool find_workspace(int dev, cudaStream_t stream, Workspace* out)
{
    std::lock_guard<std::mutex> lk(g_ws_mu);
    for (auto& w : g_ws)
        if (w.dev == dev && w.stream == stream) {
            *out = w;
            return true;
        }
    return false;
}

// ------------------------------------------------------------------ tensor maps

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// ------------------------------------------------------------------ argument parsing

bool is_vec(const b2pa_tensor* t, int dtype, int64_t n)
{
    return t && t->data && t->dtype == dtype && t->ndim == 1 && t->shape[0] == n && (n <= 1 || t->stride[0] == 1);
}

struct Problem {
    int T, H, D, B, Hkv, P, N, max_pages, layout;
    bool fp8;
    long long q_st_tok, q_st_head, out_st_tok, out_st_head, bt_stride;
    long long k_st[3], v_st[3];  // page, head, slot (elements)
    const void *q, *k, *v;
    const int *bt, *seq, *cum_q, *cum_kv;
    int q_per_req;  // > 0: decode batch, request b owns query rows b * q_per_req .. (cum_q null)
    const int* kv_indptr;      // ragged page table: bt = the flat page ids, seq = derived on the device
    const int* last_page_len;
    const float* sinks;
    void* out;
};

int parse_pools(const b2pa_tensor* k, const b2pa_tensor* v, int32_t layout, Problem* pr)
{
    if (!k || !v || !k->data || !v->data)
        return fail(B2PA_ERR_INVALID_ARG, "k_pool / v_pool: null");
    if (k->ndim != 4 || v->ndim != 4)
        return fail(B2PA_ERR_INVALID_ARG, "k_pool / v_pool must be 4-D");
    if (k->dtype != v->dtype || (k->dtype != B2PA_BF16 && k->dtype != B2PA_FP8_E4M3))
        return fail(B2PA_ERR_INVALID_ARG, "k_pool / v_pool dtype must be bf16 or fp8_e4m3 and equal");
    for (int i = 0; i < 4; ++i)
        if (k->shape[i] != v->shape[i] || k->shape[i] < 0)
            return fail(B2PA_ERR_INVALID_ARG, "k_pool and v_pool shapes differ");
    if (layout != B2PA_HND && layout != B2PA_NHD)
        return fail(B2PA_ERR_INVALID_ARG, "layout must be B2PA_HND or B2PA_NHD");
    if ((k->shape[3] > 1 && k->stride[3] != 1) || (v->shape[3] > 1 && v->stride[3] != 1))
        return fail(B2PA_ERR_INVALID_ARG, "pools must be contiguous in head_dim");
    const int hi = layout == B2PA_HND ? 1 : 2, si = layout == B2PA_HND ? 2 : 1;
    pr->layout = layout;
    pr->fp8 = k->dtype == B2PA_FP8_E4M3;
    pr->N = (int)k->shape[0];
    pr->Hkv = (int)k->shape[hi];
    pr->P = (int)k->shape[si];
    pr->D = (int)k->shape[3];
    if (k->shape[0] > 0x7FFFFFFF || pr->N < 1 || pr->Hkv < 1 || pr->P < 1 || pr->D < 1)
        return fail(B2PA_ERR_INVALID_ARG, "pool extents must be >= 1 (pages < 2^31)");
    pr->k_st[0] = k->stride[0];
    pr->k_st[1] = k->stride[hi];
    pr->k_st[2] = k->stride[si];
    pr->v_st[0] = v->stride[0];
    pr->v_st[1] = v->stride[hi];
    pr->v_st[2] = v->stride[si];
    pr->k = k->data;
    pr->v = v->data;
    return B2PA_OK;
}

int parse_problem(const b2pa_tensor* q, const b2pa_tensor* k_pool, const b2pa_tensor* v_pool,
                  const b2pa_tensor* block_tables, const b2pa_tensor* seq_lens, const b2pa_tensor* cum_q,
                  const b2pa_tensor* cum_kv, const b2pa_tensor* sinks, int32_t layout, const b2pa_tensor* out,
                  Problem* pr, int32_t q_per_req = 0, const b2pa_tensor* kv_indptr = nullptr,
                  const b2pa_tensor* last_page_len = nullptr)
{
    std::memset(pr, 0, sizeof *pr);
    int st = parse_pools(k_pool, v_pool, layout, pr);
    if (st)
        return st;
    if (!q || !q->data || q->ndim != 3 || q->dtype != B2PA_BF16)
        return fail(B2PA_ERR_INVALID_ARG, "q must be a 3-D bf16 tensor [T, H, D]");
    if (q->shape[2] != pr->D)
        return fail(B2PA_ERR_INVALID_ARG, "q head_dim %lld != pool head_dim %d", (long long)q->shape[2], pr->D);
    if (q->shape[0] < 0 || q->shape[0] > 0x7FFFFFFF || q->shape[1] < 1 || q->shape[1] > 0x7FFFFFFF)
        return fail(B2PA_ERR_INVALID_ARG, "q extents");
    if (q->shape[2] > 1 && q->stride[2] != 1)
        return fail(B2PA_ERR_INVALID_ARG, "q must be contiguous in head_dim");
    pr->T = (int)q->shape[0];
    pr->H = (int)q->shape[1];
    if (pr->H % pr->Hkv != 0)
        return fail(B2PA_ERR_INVALID_ARG, "num_heads %d is not a multiple of num_kv_heads %d", pr->H, pr->Hkv);
    if (pr->D > 256)
        return fail(B2PA_ERR_UNSUPPORTED, "head_dim %d > 256", pr->D);
    pr->q_st_tok = q->stride[0];
    pr->q_st_head = q->stride[1];
    pr->q = q->data;
    if (!out || !out->data || out->ndim != 3 || out->dtype != B2PA_BF16 || out->shape[0] != q->shape[0] ||
        out->shape[1] != q->shape[1] || out->shape[2] != q->shape[2] || (out->shape[2] > 1 && out->stride[2] != 1))
        return fail(B2PA_ERR_INVALID_ARG, "out must be bf16 with q's shape and contiguous in head_dim");
    pr->out_st_tok = out->stride[0];
    pr->out_st_head = out->stride[1];
    pr->out = out->data;
    int64_t B = 0;
    if (kv_indptr != nullptr) {
        // ragged page table: paged_kv_indptr [B + 1], paged_kv_last_page_len [B],
        // block_tables = paged_kv_indices, the flat page ids [nnz]
        if (kv_indptr->ndim != 1 || kv_indptr->shape[0] < 1)
            return fail(B2PA_ERR_INVALID_ARG, "paged_kv_indptr must be 1-D int32 [B + 1]");
        B = kv_indptr->shape[0] - 1;
        if (B > 0x7FFFFFF || !is_vec(kv_indptr, B2PA_INT32, B + 1))
            return fail(B2PA_ERR_INVALID_ARG, "paged_kv_indptr must be contiguous int32 [B + 1]");
        if (B > 0 && !is_vec(last_page_len, B2PA_INT32, B))
            return fail(B2PA_ERR_INVALID_ARG, "paged_kv_last_page_len must be contiguous int32 [B]");
        if (!block_tables || block_tables->ndim != 1 || block_tables->dtype != B2PA_INT32 ||
            block_tables->shape[0] < 0 || block_tables->shape[0] > 0x7FFFFFFF ||
            (block_tables->shape[0] > 1 && block_tables->stride[0] != 1))
            return fail(B2PA_ERR_INVALID_ARG, "paged_kv_indices must be contiguous int32 [nnz]");
        if (block_tables->shape[0] > 0 && !block_tables->data)
            return fail(B2PA_ERR_INVALID_ARG, "paged_kv_indices: null");
        pr->kv_indptr = static_cast<const int*>(kv_indptr->data);
        pr->last_page_len = B > 0 ? static_cast<const int*>(last_page_len->data) : nullptr;
        pr->max_pages = 0x7FFFFFFF;  // each request's page count comes from the indptr
        pr->bt_stride = 0;
        pr->bt = static_cast<const int*>(block_tables->data);
        pr->B = (int)B;
    } else {
        if (!seq_lens || seq_lens->ndim != 1)
            return fail(B2PA_ERR_INVALID_ARG, "seq_lens must be 1-D int32 [B]");
        B = seq_lens->shape[0];
        if (B < 0 || B > 0x7FFFFFF)
            return fail(B2PA_ERR_INVALID_ARG, "batch size");
        pr->B = (int)B;
        if (B > 0 && !is_vec(seq_lens, B2PA_INT32, B))
            return fail(B2PA_ERR_INVALID_ARG, "seq_lens must be contiguous int32 [B]");
    }
    if (q_per_req > 0) {
        if ((long long)B * q_per_req != (long long)pr->T)
            return fail(B2PA_ERR_INVALID_ARG, "q must hold batch x q_len_per_req = %lld x %d tokens, not %d",
                        (long long)B, q_per_req, pr->T);
    } else if (!is_vec(cum_q, B2PA_INT32, B + 1)) {
        return fail(B2PA_ERR_INVALID_ARG, "cum_q must be contiguous int32 [B + 1]");
    }
    if (cum_kv && !is_vec(cum_kv, B2PA_INT32, B + 1))
        return fail(B2PA_ERR_INVALID_ARG, "cum_kv must be contiguous int32 [B + 1] (or NULL)");
    if (kv_indptr == nullptr) {
        if (!block_tables || block_tables->ndim != 2 || block_tables->dtype != B2PA_INT32 ||
            block_tables->shape[0] != B || block_tables->shape[1] < 0 ||
            (block_tables->shape[1] > 1 && block_tables->stride[1] != 1) || block_tables->shape[1] > 0x7FFFFFFF)
            return fail(B2PA_ERR_INVALID_ARG, "block_tables must be int32 [B, max_pages] with unit column stride");
        if (B > 0 && block_tables->shape[1] > 0 && !block_tables->data)
            return fail(B2PA_ERR_INVALID_ARG, "block_tables: null");
        pr->max_pages = (int)block_tables->shape[1];
        pr->bt_stride = block_tables->stride[0];
        pr->bt = static_cast<const int*>(block_tables->data);
    }
    pr->seq = (kv_indptr == nullptr && B > 0) ? static_cast<const int*>(seq_lens->data) : nullptr;
    pr->cum_q = q_per_req > 0 ? nullptr : static_cast<const int*>(cum_q->data);
    pr->q_per_req = q_per_req > 0 ? q_per_req : 0;
    pr->cum_kv = cum_kv ? static_cast<const int*>(cum_kv->data) : nullptr;
    if (sinks) {
        if (!is_vec(sinks, B2PA_FP32, pr->H))
            return fail(B2PA_ERR_INVALID_ARG, "sinks must be contiguous fp32 [H] (or NULL)");
        pr->sinks = static_cast<const float*>(sinks->data);
    }
    return B2PA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

// Why the tensor-core path cannot take this problem (nullptr if it can).
const char* tc_reject(const Problem& pr, const DevInfo& di)
{
    if (!(di.major == 10 && di.minor == 3))
        return "the tensor-core path is built for sm_103a only";
    if (pr.fp8 ? pr.D != 128 : (pr.D != 64 && pr.D != 128))
        return "head_dim must be 64 or 128 (128 for fp8 pools)";
    if (!pow2(pr.P) || pr.P < 8)
        return "page_size must be a power of two >= 8";
    if (pr.H / pr.Hkv > kQRows)
        return "more than 128 query heads per kv head";
    if (pr.B > kSchedMaxBatch)
        return "batch larger than the scheduler handles";
    const int es = pr.fp8 ? 1 : 2;
    if (!aligned16(pr.q) || (pr.q_st_tok * 2) % 16 || (pr.q_st_head * 2) % 16)
        return "q must be 16-byte aligned with 16-byte-multiple strides";
    if (!aligned16(pr.out) || (pr.out_st_tok * 2) % 16 || (pr.out_st_head * 2) % 16)
        return "out must be 16-byte aligned with 16-byte-multiple strides";
    if (!aligned16(pr.k) || !aligned16(pr.v))
        return "pools must be 16-byte aligned";
    const int ext[3] = {pr.N, pr.Hkv, pr.P};
    for (int i = 0; i < 3; ++i)
        if (ext[i] > 1 && (((pr.k_st[i] * es) % 16) || ((pr.v_st[i] * es) % 16) || pr.k_st[i] <= 0 || pr.v_st[i] <= 0))
            return "pool strides must be positive multiples of 16 bytes";
    return nullptr;
}

// Encode the 4-D (D, P, Hkv, pages) map of one pool, box = one page (at most
// 128 slots) by one 128-byte column block.
int encode_pool_map(CUtensorMap* m, const Problem& pr, const void* base, const long long st[3])
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return fail(B2PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const int es = pr.fp8 ? 1 : 2;
    // canonical strides for extent-1 dims (their value is never used)
    long long s_slot = st[2] * es, s_head = st[1] * es, s_page = st[0] * es;
    const long long row = (long long)pr.D * es;
    if (pr.P == 1)
        s_slot = row;
    if (pr.Hkv == 1)
        s_head = s_slot * pr.P;
    if (pr.N == 1)
        s_page = s_head * pr.Hkv > s_slot * pr.P ? s_head * pr.Hkv : s_slot * pr.P;
    s_slot = (s_slot + 15) / 16 * 16;
    s_head = (s_head + 15) / 16 * 16;
    s_page = (s_page + 15) / 16 * 16;
    cuuint64_t dims[4] = {(cuuint64_t)pr.D, (cuuint64_t)pr.P, (cuuint64_t)pr.Hkv, (cuuint64_t)pr.N};
    cuuint64_t strides[3] = {(cuuint64_t)s_slot, (cuuint64_t)s_head, (cuuint64_t)s_page};
    cuuint32_t box[4] = {(cuuint32_t)(pr.fp8 ? 128 : 64), (cuuint32_t)(pr.P < kKvTile ? pr.P : kKvTile), 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(m, pr.fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(B2PA_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled(pool) failed with %d", (int)r);
    return B2PA_OK;
}

int encode_q_map(CUtensorMap* m, const Problem& pr, int rows_per_tile)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return fail(B2PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const int G = pr.H / pr.Hkv;
    long long s_head = pr.q_st_head * 2, s_tok = pr.q_st_tok * 2;
    if (pr.H == 1)
        s_head = (long long)pr.D * 2;
    if (pr.T <= 1)
        s_tok = s_head * pr.H;
    cuuint64_t dims[3] = {(cuuint64_t)pr.D, (cuuint64_t)pr.H, (cuuint64_t)(pr.T > 0 ? pr.T : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)s_head, (cuuint64_t)s_tok};
    cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)rows_per_tile};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pr.q), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(B2PA_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled(q) failed with %d", (int)r);
    return B2PA_OK;
}

// The output as a 3-D (D, H, T) map whose box is one softmax warp's 32 rows
// (64 columns at a time): {64, min(G, 32), max(1, 32 / G)}.  Only when 32
// rows are whole boxes (G divides 32 or 32 divides G); *ok = false otherwise or
// if the driver rejects the map, and the kernel then stores the rows itself.
int encode_o_map(CUtensorMap* m, const Problem& pr, bool* ok)
{
    *ok = false;
    EncodeTiledFn fn = encode_fn();
    const int G = pr.H / pr.Hkv;
    if (!fn || !(32 % G == 0 || G % 32 == 0))
        return B2PA_OK;
    long long s_head = pr.out_st_head * 2, s_tok = pr.out_st_tok * 2;
    if (pr.H == 1)
        s_head = (long long)pr.D * 2;
    if (pr.T <= 1)
        s_tok = s_head * pr.H;
    cuuint64_t dims[3] = {(cuuint64_t)pr.D, (cuuint64_t)pr.H, (cuuint64_t)(pr.T > 0 ? pr.T : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)s_head, (cuuint64_t)s_tok};
    cuuint32_t box[3] = {64, (cuuint32_t)(G < 32 ? G : 32), (cuuint32_t)(G < 32 ? 32 / G : 1)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, pr.out, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    *ok = r == CUDA_SUCCESS;
    return B2PA_OK;
}

int rows_per_tile_of(const Problem& pr) { return kQRows / (pr.H / pr.Hkv); }

// The one-window-tile kernel takes a tensor-core shape at head_dim 64 with a
// 16-bit cache, a left window, no kv chunks and pages of at most 32 keys, when
// every row of a work item (two query tiles) sees keys within one tile of
// win_max_keys() keys that starts at a page boundary.
bool win_eligible(const Problem& pr, int window, bool split)
{
    return !pr.fp8 && pr.D == 64 && window >= 0 && !split && pr.P <= 32 &&
           2LL * rows_per_tile_of(pr) + window + pr.P - 1 <= win_max_keys();
}

cudaError_t launch_tc_kernel(const AttnParams& ap, const Problem& pr, int window, bool split, int sms,
                             cudaStream_t stream)
{
    return win_eligible(pr, window, split) ? launch_attention_win(ap, sms, stream)
                                           : launch_attention_tc(ap, pr.D, pr.fp8, sms, stream, true);
}

// Everything the tensor-core kernel takes: tensor maps, pointers, geometry and
// scales; the work list and its counters come from the scheduler's parameters.
int fill_attn_params(AttnParams* ap, const Problem& pr, const SchedParams& sp, size_t cap, int window,
                     float bmm1_scale, float bmm2_scale, const float* bmm1_dev = nullptr,
                     const float* bmm2_dev = nullptr)
{
    std::memset(ap, 0, sizeof *ap);
    const int rpt = rows_per_tile_of(pr);
    int st;
    if ((st = encode_q_map(&ap->tm_q, pr, rpt)) || (st = encode_pool_map(&ap->tm_k, pr, pr.k, pr.k_st)) ||
        (st = encode_pool_map(&ap->tm_v, pr, pr.v, pr.v_st)))
        return st;
    bool o_ok = false;
    encode_o_map(&ap->tm_o, pr, &o_ok);
    ap->out_tma = o_ok ? 1 : 0;
    ap->cum_q = pr.cum_q;
    ap->q_per_req = pr.q_per_req;
    ap->seq_lens = pr.seq;
    ap->block_tables = pr.bt;
    ap->kv_indptr = pr.kv_indptr;
    ap->sinks = pr.sinks;
    ap->out = static_cast<uint16_t*>(pr.out);
    ap->bt_stride = pr.bt_stride;
    ap->out_stride_tok = pr.out_st_tok;
    ap->out_stride_head = pr.out_st_head;
    ap->sched = sp;  // callers that change sp afterwards copy it again
    ap->items = sp.items;
    uint8_t* hdr = reinterpret_cast<uint8_t*>(sp.err);  // the workspace header
    ap->counter = reinterpret_cast<int*>(hdr + 8);
    ap->claim = reinterpret_cast<int*>(hdr + 12);
    ap->ready = reinterpret_cast<int*>(hdr + 16);
    ap->done = reinterpret_cast<int*>(hdr + 20);
    ap->err = sp.err;
    ap->cap = (int)cap;
    ap->H = pr.H;
    ap->Hkv = pr.Hkv;
    ap->G = pr.H / pr.Hkv;
    ap->rows_per_tile = rpt;
    ap->page_size = pr.P;
    ap->num_pages = pr.N;
    ap->window = window;
    ap->scale_log2 = (float)((double)bmm1_scale * 1.4426950408889634);
    ap->bmm2 = bmm2_scale;
    ap->bmm1_dev = bmm1_dev;
    ap->bmm2_dev = bmm2_dev;
    ap->wait_limit_ns = g_wait_limit_ns.load();
    ap->inject_stall = g_inject_stall.load();
    return B2PA_OK;
}

// A one-element fp32 device tensor holding a scale (the FlashInfer API's
// "float | Tensor" bmm scales); its pointer, or nullptr with an error set.
const float* scale_tensor(const b2pa_tensor* t, const char* what)
{
    if (!t || !t->data || t->dtype != B2PA_FP32 || t->ndim < 0 || t->ndim > 1 || (t->ndim == 1 && t->shape[0] != 1)) {
        fail(B2PA_ERR_INVALID_ARG, "%s must be a one-element fp32 device tensor", what);
        return nullptr;
    }
    if ((reinterpret_cast<uintptr_t>(t->data) & 3u) != 0) {
        fail(B2PA_ERR_INVALID_ARG, "%s must be 4-byte aligned", what);
        return nullptr;
    }
    return static_cast<const float*>(t->data);
}

size_t items_needed(const Problem& pr, int max_q_len)
{
    const long long per = (long long)rows_per_tile_of(pr) * kQTiles;
    const long long n = (long long)pr.B * pr.Hkv * ((max_q_len + per - 1) / per);
    return (size_t)(n > 0 ? n : 1);
}

int choose_path(const Problem& pr, const DevInfo& di, bool* use_tc)
{
    const int want = g_path.load();
    const char* why = tc_reject(pr, di);
    if (want == B2PA_PATH_GENERIC) {
        *use_tc = false;
        return B2PA_OK;
    }
    if (want == B2PA_PATH_TCGEN05 && why)
        return fail(B2PA_ERR_UNSUPPORTED, "tensor-core path: %s", why);
    *use_tc = why == nullptr;
    return B2PA_OK;
}

SchedParams make_sched(const Problem& pr, const Workspace& ws, int max_q_len, int max_kv_len, int window,
                       size_t cap)
{
    SchedParams sp;
    std::memset(&sp, 0, sizeof sp);
    sp.cum_q = pr.cum_q;
    sp.q_per_req = pr.q_per_req;
    sp.seq_lens = pr.seq;
    sp.kv_indptr = pr.kv_indptr;
    sp.cum_kv = pr.cum_kv;
    sp.block_tables = pr.bt;
    sp.bt_stride = pr.bt_stride;
    sp.B = pr.B;
    sp.Hkv = pr.Hkv;
    sp.rows_per_tile = rows_per_tile_of(pr);
    sp.window = window;
    sp.max_q_len = max_q_len;
    sp.max_kv_len = max_kv_len;
    sp.page_size = pr.P;
    sp.max_pages = pr.max_pages;
    sp.num_tokens = pr.T;
    sp.num_pages = pr.N;
    sp.debug = g_debug.load();
    sp.cap = (int)cap;
    // an item touches at most ceil(max_kv_len / kKvTile) kv tiles of each of its
    // query tiles; with that many buckets no cost is capped below kCostCap
    const long long max_cost = (long long)((max_kv_len + kKvTile - 1) / kKvTile) * kQTiles;
    sp.nbuckets = (int)(max_cost + 1 < kSchedBuckets ? (max_cost + 1 > 2 ? max_cost + 1 : 2) : kSchedBuckets);
    sp.items = reinterpret_cast<int4*>(ws.mem + kWsHeader);
    sp.count = reinterpret_cast<int*>(ws.mem + 4);
    sp.err = reinterpret_cast<unsigned*>(ws.mem);
    return sp;
}

// Split-KV geometry of a decode batch on the tensor-core path: chunks of
// split_tiles kv tiles, at most `slots` chunks per request (split_tiles = 0:
// no split).  The chunk size gives the batch about two work items per SM on
// its longest possible rows (the lengths themselves are on the device), and
// never fewer than two kv tiles per chunk.
struct SplitPlan {
    int split_tiles = 0;
    int slots = 1;
};

SplitPlan plan_split(const Problem& pr, int max_kv_len, int sms)
{
    SplitPlan sp;
    const int G = pr.H / pr.Hkv;
    // the e4m3 split kernel holds one query tile per item
    const int per_item = (kQRows / G) * (pr.fp8 ? 1 : kQTiles);
    if (pr.q_per_req <= 0 || pr.q_per_req > per_item)
        return sp;  // several query items per request: no split (as a context batch)
    const long long tiles = (max_kv_len + kKvTile - 1) / kKvTile;
    const long long total = (long long)pr.B * pr.Hkv * tiles;
    const long long want = 2LL * sms;
    long long chunk = (total + want - 1) / want;
    if (chunk < 2)
        chunk = 2;
    if (chunk >= tiles)
        return sp;  // enough items without cutting any request
    sp.split_tiles = (int)chunk;
    sp.slots = (int)((tiles + chunk - 1) / chunk);
    return sp;
}

// Every attention entry point: a context batch (cum_q) or a decode batch
// (q_per_req > 0, cum_q null); scales as host floats, or (bmm1_dev, bmm2_dev
// non-null) as device fp32 values read by the kernels.
int context_attention_impl(const b2pa_tensor* q, const b2pa_tensor* k_pool, const b2pa_tensor* v_pool,
                           const b2pa_tensor* block_tables, const b2pa_tensor* seq_lens, const b2pa_tensor* cum_q,
                           const b2pa_tensor* cum_kv, int32_t max_q_len, int32_t max_kv_len, float bmm1_scale,
                           float bmm2_scale, const float* bmm1_dev, const float* bmm2_dev, int32_t window_left,
                           const b2pa_tensor* sinks, int32_t layout, b2pa_tensor* out, cudaStream_t stream,
                           int32_t q_per_req = 0, const b2pa_tensor* kv_indptr = nullptr,
                           const b2pa_tensor* last_page_len = nullptr)
{
    Problem pr;
    int st = parse_problem(q, k_pool, v_pool, block_tables, seq_lens, cum_q, cum_kv, sinks, layout, out, &pr,
                           q_per_req, kv_indptr, last_page_len);
    if (st)
        return st;
    if (max_q_len < 0 || max_kv_len < 0)
        return fail(B2PA_ERR_INVALID_ARG, "max_q_len / max_kv_len must be >= 0");
    if (!std::isfinite(bmm1_scale) || !(bmm1_scale > 0.f) || !std::isfinite(bmm2_scale))
        return fail(B2PA_ERR_INVALID_ARG, "bmm1_scale must be finite and > 0, bmm2_scale finite");
    const int window = window_left < 0 ? -1 : window_left;
    if (pr.B == 0 || pr.T == 0)
        return B2PA_OK;
    int dev;
    DevInfo di;
    if ((st = device_info(&dev, &di)))
        return st;
    bool use_tc = false;
    if ((st = choose_path(pr, di, &use_tc)))
        return st;
    if (use_tc) {
        const SplitPlan split = plan_split(pr, max_kv_len, di.sms);
        const size_t cap = split.split_tiles > 0 ? (size_t)pr.B * pr.Hkv * split.slots : items_needed(pr, max_q_len);
        // workspace: header, work list, then (split-KV) chunks per request and the partial rows
        const size_t rows = (size_t)pr.T * pr.H * split.slots;
        const size_t off_nsplit = kWsHeader + cap * sizeof(int4);
        const size_t off_ml = (off_nsplit + (size_t)pr.B * sizeof(int) + 255) / 256 * 256;
        const size_t off_o = (off_ml + rows * 2 * sizeof(float) + 255) / 256 * 256;
        const size_t body = split.split_tiles > 0 ? off_o + rows * pr.D * sizeof(float) : off_nsplit;
        // ragged page table: the kv lengths derived on the device, last
        const size_t off_seq = (body + 255) / 256 * 256;
        const size_t need = pr.kv_indptr ? off_seq + (size_t)pr.B * sizeof(int) : body;
        Workspace ws;
        if ((st = get_workspace_bytes(dev, stream, need, &ws)))
            return st;
        if (pr.kv_indptr) {
            int* kv_len = reinterpret_cast<int*>(ws.mem + off_seq);
            cudaError_t e = launch_ragged_lengths(pr.kv_indptr, pr.last_page_len, pr.B, pr.P, kv_len,
                                                  reinterpret_cast<unsigned*>(ws.mem), stream);
            if (e != cudaSuccess)
                return cuda_fail(e, "ragged page-table lengths launch");
            pr.seq = kv_len;
        }
        SchedParams sp = make_sched(pr, ws, max_q_len, max_kv_len, window, cap);
        AttnParams ap;
        // a shape the tensor-core path accepts must encode; a failure is an
        // error of the call, never a silent switch to the other kernel
        if ((st = fill_attn_params(&ap, pr, sp, cap, window, bmm1_scale, bmm2_scale, bmm1_dev, bmm2_dev)))
            return st;
        if (split.split_tiles > 0) {
            sp.split_tiles = split.split_tiles;
            sp.nsplit = reinterpret_cast<int*>(ws.mem + off_nsplit);
            // chunk costs are at most split_tiles * kQTiles
            const int nb = split.split_tiles * kQTiles + 1;
            sp.nbuckets = nb < sp.nbuckets ? nb : sp.nbuckets;
            ap.split_tiles = split.split_tiles;
            ap.part_slots = split.slots;
            ap.part_ml = reinterpret_cast<float*>(ws.mem + off_ml);
            ap.part_o = reinterpret_cast<float*>(ws.mem + off_o);
        }
        ap.sched = sp;
        cudaError_t e;
        cudaEvent_t ev0 = static_cast<cudaEvent_t>(g_ev_start.load());
        cudaEvent_t ev1 = static_cast<cudaEvent_t>(g_ev_stop.load());
        const bool timed = ev0 != nullptr && ev1 != nullptr;
        if (timed && (e = cudaEventRecord(ev0, stream)) != cudaSuccess)
            return cuda_fail(e, "cudaEventRecord");
        // launched as every call launches it; with the events around it the
        // kernel follows the start event, not an earlier kernel
        e = launch_tc_kernel(ap, pr, window, split.split_tiles > 0, di.sms, stream);
        if (e != cudaSuccess)
            return cuda_fail(e, "attention kernel launch");
        if (timed && (e = cudaEventRecord(ev1, stream)) != cudaSuccess)
            return cuda_fail(e, "cudaEventRecord");
        if (split.split_tiles > 0) {
            CombineParams cp;
            std::memset(&cp, 0, sizeof cp);
            cp.part_o = ap.part_o;
            cp.part_ml = ap.part_ml;
            cp.nsplit = sp.nsplit;
            cp.sinks = pr.sinks;
            cp.out = static_cast<uint16_t*>(pr.out);
            cp.out_st_tok = pr.out_st_tok;
            cp.out_st_head = pr.out_st_head;
            cp.B = pr.B;
            cp.q_per_req = pr.q_per_req;
            cp.H = pr.H;
            cp.D = pr.D;
            cp.part_slots = split.slots;
            cp.bmm2 = bmm2_scale;
            cp.bmm2_dev = bmm2_dev;
            if ((e = launch_combine(cp, stream)) != cudaSuccess)
                return cuda_fail(e, "combine launch");
        }
        return B2PA_OK;
    }
    Workspace ws;
    if ((st = get_workspace_bytes(dev, stream, kWsHeader + (size_t)pr.B * sizeof(int), &ws)))
        return st;
    if (pr.kv_indptr) {
        int* kv_len = reinterpret_cast<int*>(ws.mem + kWsHeader);
        cudaError_t e = launch_ragged_lengths(pr.kv_indptr, pr.last_page_len, pr.B, pr.P, kv_len,
                                              reinterpret_cast<unsigned*>(ws.mem), stream);
        if (e != cudaSuccess)
            return cuda_fail(e, "ragged page-table lengths launch");
        pr.seq = kv_len;
    }
    GenericParams gp;
    std::memset(&gp, 0, sizeof gp);
    gp.q = static_cast<const uint16_t*>(pr.q);
    gp.k = pr.k;
    gp.v = pr.v;
    gp.cum_q = pr.cum_q;
    gp.q_per_req = pr.q_per_req;
    gp.seq_lens = pr.seq;
    gp.block_tables = pr.bt;
    gp.kv_indptr = pr.kv_indptr;
    gp.sinks = pr.sinks;
    gp.out = static_cast<uint16_t*>(pr.out);
    gp.q_st_tok = pr.q_st_tok;
    gp.q_st_head = pr.q_st_head;
    gp.out_st_tok = pr.out_st_tok;
    gp.out_st_head = pr.out_st_head;
    gp.k_st_page = pr.k_st[0];
    gp.k_st_head = pr.k_st[1];
    gp.k_st_slot = pr.k_st[2];
    gp.v_st_page = pr.v_st[0];
    gp.v_st_head = pr.v_st[1];
    gp.v_st_slot = pr.v_st[2];
    gp.bt_stride = pr.bt_stride;
    gp.B = pr.B;
    gp.T = pr.T;
    gp.H = pr.H;
    gp.Hkv = pr.Hkv;
    gp.D = pr.D;
    gp.page_size = pr.P;
    gp.max_pages = pr.max_pages;
    gp.num_pages = pr.N;
    gp.max_q_len = max_q_len;
    gp.max_kv_len = max_kv_len;
    gp.window = window;
    gp.scale_log2 = (float)((double)bmm1_scale * 1.4426950408889634);
    gp.bmm2 = bmm2_scale;
    gp.bmm1_dev = bmm1_dev;
    gp.bmm2_dev = bmm2_dev;
    gp.err = reinterpret_cast<unsigned*>(ws.mem);
    cudaError_t e = launch_attention_generic(gp, pr.fp8, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "generic attention launch");
    return B2PA_OK;
}

}  // namespace

// ====================================================================== C ABI

extern "C" {

int b2pa_context_attention(const b2pa_tensor* q, const b2pa_tensor* k_pool, const b2pa_tensor* v_pool,
                           const b2pa_tensor* block_tables, const b2pa_tensor* seq_lens, const b2pa_tensor* cum_q,
                           const b2pa_tensor* cum_kv, int32_t max_q_len, int32_t max_kv_len, float bmm1_scale,
                           float bmm2_scale, int32_t window_left, const b2pa_tensor* sinks, int32_t layout,
                           b2pa_tensor* out, b2pa_stream_t stream_h)
{
    g_last_error.clear();
    return context_attention_impl(q, k_pool, v_pool, block_tables, seq_lens, cum_q, cum_kv, max_q_len, max_kv_len,
                                  bmm1_scale, bmm2_scale, nullptr, nullptr, window_left, sinks, layout, out,
                                  reinterpret_cast<cudaStream_t>(stream_h));
}

int b2pa_context_attention_ragged(const b2pa_tensor* q, const b2pa_tensor* k_pool, const b2pa_tensor* v_pool,
                                  const b2pa_tensor* paged_kv_indices, const b2pa_tensor* paged_kv_indptr,
                                  const b2pa_tensor* paged_kv_last_page_len, const b2pa_tensor* cum_q,
                                  int32_t max_q_len, int32_t max_kv_len, float bmm1_scale, float bmm2_scale,
                                  int32_t window_left, const b2pa_tensor* sinks, int32_t layout, b2pa_tensor* out,
                                  b2pa_stream_t stream_h)
{
    g_last_error.clear();
    if (!paged_kv_indptr)
        return fail(B2PA_ERR_INVALID_ARG, "paged_kv_indptr: null");
    return context_attention_impl(q, k_pool, v_pool, paged_kv_indices, nullptr, cum_q, nullptr, max_q_len, max_kv_len,
                                  bmm1_scale, bmm2_scale, nullptr, nullptr, window_left, sinks, layout, out,
                                  reinterpret_cast<cudaStream_t>(stream_h), 0, paged_kv_indptr,
                                  paged_kv_last_page_len);
}

int b2pa_batch_decode(const b2pa_tensor* q, const b2pa_tensor* k_pool, const b2pa_tensor* v_pool,
                      const b2pa_tensor* block_tables, const b2pa_tensor* seq_lens, int32_t q_len_per_req,
                      int32_t max_seq_len, float bmm1_scale, float bmm2_scale, int32_t window_left,
                      const b2pa_tensor* sinks, int32_t layout, b2pa_tensor* out, b2pa_stream_t stream_h)
{
    g_last_error.clear();
    if (q_len_per_req < 1)
        return fail(B2PA_ERR_INVALID_ARG, "q_len_per_req must be >= 1");
    return context_attention_impl(q, k_pool, v_pool, block_tables, seq_lens, nullptr, nullptr, q_len_per_req,
                                  max_seq_len, bmm1_scale, bmm2_scale, nullptr, nullptr, window_left, sinks, layout,
                                  out, reinterpret_cast<cudaStream_t>(stream_h), q_len_per_req);
}

int b2pa_context_attention_tensor_scales(const b2pa_tensor* q, const b2pa_tensor* k_pool, const b2pa_tensor* v_pool,
                                         const b2pa_tensor* block_tables, const b2pa_tensor* seq_lens,
                                         const b2pa_tensor* cum_q, const b2pa_tensor* cum_kv, int32_t max_q_len,
                                         int32_t max_kv_len, const b2pa_tensor* bmm1_scale,
                                         const b2pa_tensor* bmm2_scale, int32_t window_left, const b2pa_tensor* sinks,
                                         int32_t layout, b2pa_tensor* out, b2pa_stream_t stream_h)
{
    g_last_error.clear();
    const float* b1 = scale_tensor(bmm1_scale, "bmm1_scale");
    if (!b1)
        return B2PA_ERR_INVALID_ARG;
    const float* b2 = scale_tensor(bmm2_scale, "bmm2_scale");
    if (!b2)
        return B2PA_ERR_INVALID_ARG;
    // the host values are placeholders that pass the host checks; the kernels use b1, b2
    return context_attention_impl(q, k_pool, v_pool, block_tables, seq_lens, cum_q, cum_kv, max_q_len, max_kv_len,
                                  1.0f, 1.0f, b1, b2, window_left, sinks, layout, out,
                                  reinterpret_cast<cudaStream_t>(stream_h));
}

int b2pa_debug_worklist(const b2pa_tensor* q, const b2pa_tensor* k_pool, const b2pa_tensor* block_tables,
                        const b2pa_tensor* seq_lens, const b2pa_tensor* cum_q, int32_t max_q_len, int32_t max_kv_len,
                        int32_t window_left, int32_t layout, int32_t* host_items_out, int32_t cap, int32_t* n_out,
                        int32_t* geometry_out, b2pa_stream_t stream_h)
{
    g_last_error.clear();
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_h);
    Problem pr;
    // out is not needed: describe it as q
    int st = parse_problem(q, k_pool, k_pool, block_tables, seq_lens, cum_q, nullptr, nullptr, layout, q, &pr);
    if (st)
        return st;
    if (!n_out || (cap > 0 && !host_items_out) || max_q_len < 0 || max_kv_len < 0)
        return fail(B2PA_ERR_INVALID_ARG, "n_out / host_items_out / bounds");
    int dev;
    DevInfo di;
    if ((st = device_info(&dev, &di)))
        return st;
    if (pr.B > kSchedMaxBatch)
        return fail(B2PA_ERR_UNSUPPORTED, "batch larger than the scheduler handles");
    const int rpt = rows_per_tile_of(pr);
    if (geometry_out) {
        geometry_out[0] = rpt;
        geometry_out[1] = kQTiles;
        geometry_out[2] = kKvTile;
        geometry_out[3] = kCostCap;
    }
    *n_out = 0;
    if (pr.B == 0)
        return B2PA_OK;
    const size_t need = items_needed(pr, max_q_len);
    Workspace ws;
    if ((st = get_workspace(dev, stream, need, &ws)))
        return st;
    SchedParams sp = make_sched(pr, ws, max_q_len, max_kv_len, window_left < 0 ? -1 : window_left, need);
    cudaError_t e = launch_schedule(sp, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "scheduler launch");
    int count = 0;
    if ((e = cudaMemcpyAsync(&count, sp.count, sizeof count, cudaMemcpyDeviceToHost, stream)) != cudaSuccess ||
        (e = cudaStreamSynchronize(stream)) != cudaSuccess)
        return cuda_fail(e, "reading the work list");
    *n_out = count;
    const int ncopy = count < cap ? count : cap;
    const int navail = (size_t)ncopy > need ? (int)need : ncopy;
    if (navail > 0) {
        if ((e = cudaMemcpyAsync(host_items_out, sp.items, sizeof(int4) * (size_t)navail, cudaMemcpyDeviceToHost,
                                 stream)) != cudaSuccess ||
            (e = cudaStreamSynchronize(stream)) != cudaSuccess)
            return cuda_fail(e, "reading the work list");
    }
    return B2PA_OK;
}

}  // extern "C"

namespace {

// Both debug gathers: a [B, max_pages] block table with seq_lens, or the
// ragged page table (kv_indptr non-null; block_tables = the flat page ids).
int debug_gather_impl(const b2pa_tensor* k_pool, const b2pa_tensor* v_pool, const b2pa_tensor* block_tables,
                      const b2pa_tensor* seq_lens, const b2pa_tensor* kv_indptr, const b2pa_tensor* last_page_len,
                      const b2pa_tensor* cum_kv, int32_t layout, b2pa_tensor* k_out, b2pa_tensor* v_out,
                      cudaStream_t stream)
{
    Problem pr;
    std::memset(&pr, 0, sizeof pr);
    int st = parse_pools(k_pool, v_pool, layout, &pr);
    if (st)
        return st;
    int64_t B = 0;
    if (kv_indptr != nullptr) {
        if (kv_indptr->ndim != 1 || kv_indptr->shape[0] < 1 || kv_indptr->shape[0] - 1 > 0x7FFFFFF ||
            !is_vec(kv_indptr, B2PA_INT32, kv_indptr->shape[0]))
            return fail(B2PA_ERR_INVALID_ARG, "paged_kv_indptr must be contiguous int32 [B + 1]");
        B = kv_indptr->shape[0] - 1;
        if ((B > 0 && !is_vec(last_page_len, B2PA_INT32, B)) || !is_vec(cum_kv, B2PA_INT32, B + 1))
            return fail(B2PA_ERR_INVALID_ARG, "paged_kv_last_page_len [B] / cum_kv [B + 1] must be contiguous int32");
        if (!block_tables || block_tables->ndim != 1 || block_tables->dtype != B2PA_INT32 ||
            (block_tables->shape[0] > 1 && block_tables->stride[0] != 1))
            return fail(B2PA_ERR_INVALID_ARG, "paged_kv_indices must be contiguous int32 [nnz]");
    } else {
        if (!seq_lens || seq_lens->ndim != 1)
            return fail(B2PA_ERR_INVALID_ARG, "seq_lens must be 1-D int32 [B]");
        B = seq_lens->shape[0];
        if (B < 0 || B > 0x7FFFFFF || (B > 0 && !is_vec(seq_lens, B2PA_INT32, B)) ||
            !is_vec(cum_kv, B2PA_INT32, B + 1))
            return fail(B2PA_ERR_INVALID_ARG, "seq_lens [B] / cum_kv [B + 1] must be contiguous int32");
        if (!block_tables || block_tables->ndim != 2 || block_tables->dtype != B2PA_INT32 ||
            block_tables->shape[0] != B || (block_tables->shape[1] > 1 && block_tables->stride[1] != 1))
            return fail(B2PA_ERR_INVALID_ARG, "block_tables must be int32 [B, max_pages]");
    }
    const int dt = k_pool->dtype;
    for (const b2pa_tensor* o : {static_cast<const b2pa_tensor*>(k_out), static_cast<const b2pa_tensor*>(v_out)}) {
        if (!o || !o->data || o->ndim != 3 || o->dtype != dt || o->shape[1] != pr.Hkv || o->shape[2] != pr.D ||
            o->stride[2] != 1 || o->stride[1] != pr.D || o->stride[0] != (int64_t)pr.Hkv * pr.D || !aligned16(o->data))
            return fail(B2PA_ERR_INVALID_ARG, "k_out / v_out must be contiguous [rows, Hkv, D] of the pool dtype");
    }
    if (k_out->shape[0] != v_out->shape[0])
        return fail(B2PA_ERR_INVALID_ARG, "k_out and v_out rows differ");
    pr.B = (int)B;
    pr.max_pages = kv_indptr ? 0x7FFFFFFF : (int)block_tables->shape[1];
    pr.bt_stride = kv_indptr ? 0 : block_tables->stride[0];
    // borrow the tensor-core checks with q/out stand-ins that always pass
    static const uint4 dummy = {0, 0, 0, 0};
    pr.q = &dummy;
    pr.out = const_cast<uint4*>(&dummy);
    pr.H = pr.Hkv;
    int dev;
    DevInfo di;
    if ((st = device_info(&dev, &di)))
        return st;
    if (const char* why = tc_reject(pr, di))
        return fail(B2PA_ERR_UNSUPPORTED, "gather uses the tensor-core loads: %s", why);
    if (B == 0)
        return B2PA_OK;
    Workspace ws;
    if ((st = get_workspace_bytes(dev, stream, kWsHeader + (size_t)B * sizeof(int), &ws)))
        return st;
    GatherParams gp;
    std::memset(&gp, 0, sizeof gp);
    if ((st = encode_pool_map(&gp.tm_k, pr, pr.k, pr.k_st)) || (st = encode_pool_map(&gp.tm_v, pr, pr.v, pr.v_st)))
        return st;
    if (kv_indptr != nullptr) {
        int* kv_len = reinterpret_cast<int*>(ws.mem + kWsHeader);
        cudaError_t e = launch_ragged_lengths(static_cast<const int*>(kv_indptr->data),
                                              static_cast<const int*>(last_page_len->data), (int)B, pr.P, kv_len,
                                              reinterpret_cast<unsigned*>(ws.mem), stream);
        if (e != cudaSuccess)
            return cuda_fail(e, "ragged page-table lengths launch");
        gp.seq_lens = kv_len;
        gp.kv_indptr = static_cast<const int*>(kv_indptr->data);
    } else {
        gp.seq_lens = static_cast<const int*>(seq_lens->data);
    }
    gp.cum_kv = static_cast<const int*>(cum_kv->data);
    gp.block_tables = static_cast<const int*>(block_tables->data);
    gp.bt_stride = pr.bt_stride;
    gp.k_out = static_cast<uint8_t*>(k_out->data);
    gp.v_out = static_cast<uint8_t*>(v_out->data);
    gp.out_rows = k_out->shape[0];
    gp.B = pr.B;
    gp.Hkv = pr.Hkv;
    gp.D = pr.D;
    gp.page_size = pr.P;
    gp.max_pages = pr.max_pages;
    gp.num_pages = pr.N;
    gp.esize = pr.fp8 ? 1 : 2;
    gp.err = reinterpret_cast<unsigned*>(ws.mem);
    const long long rows = k_out->shape[0];
    cudaError_t e = launch_gather(gp, pr.fp8, (int)(rows < 0x7FFFFFFF ? rows : 0x7FFFFFFF), stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "gather launch");
    return B2PA_OK;
}

}  // namespace

extern "C" {

int b2pa_debug_gather(const b2pa_tensor* k_pool, const b2pa_tensor* v_pool, const b2pa_tensor* block_tables,
                      const b2pa_tensor* seq_lens, const b2pa_tensor* cum_kv, int32_t layout, b2pa_tensor* k_out,
                      b2pa_tensor* v_out, b2pa_stream_t stream_h)
{
    g_last_error.clear();
    return debug_gather_impl(k_pool, v_pool, block_tables, seq_lens, nullptr, nullptr, cum_kv, layout, k_out, v_out,
                             reinterpret_cast<cudaStream_t>(stream_h));
}

int b2pa_debug_gather_ragged(const b2pa_tensor* k_pool, const b2pa_tensor* v_pool,
                             const b2pa_tensor* paged_kv_indices, const b2pa_tensor* paged_kv_indptr,
                             const b2pa_tensor* paged_kv_last_page_len, const b2pa_tensor* cum_kv, int32_t layout,
                             b2pa_tensor* k_out, b2pa_tensor* v_out, b2pa_stream_t stream_h)
{
    g_last_error.clear();
    if (!paged_kv_indptr)
        return fail(B2PA_ERR_INVALID_ARG, "paged_kv_indptr: null");
    return debug_gather_impl(k_pool, v_pool, paged_kv_indices, nullptr, paged_kv_indptr, paged_kv_last_page_len,
                             cum_kv, layout, k_out, v_out, reinterpret_cast<cudaStream_t>(stream_h));
}

int b2pa_append_kv(const b2pa_tensor* k_new, const b2pa_tensor* v_new, const b2pa_tensor* k_pool,
                   const b2pa_tensor* v_pool, const b2pa_tensor* cache_loc, float k_scale, float v_scale,
                   int32_t layout, b2pa_stream_t stream_h)
{
    g_last_error.clear();
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_h);
    Problem pr;
    std::memset(&pr, 0, sizeof pr);
    int st = parse_pools(k_pool, v_pool, layout, &pr);
    if (st)
        return st;
    if (!k_new || !v_new || k_new->ndim != 3 || v_new->ndim != 3 || k_new->dtype != B2PA_BF16 ||
        v_new->dtype != B2PA_BF16)
        return fail(B2PA_ERR_INVALID_ARG, "k_new / v_new must be bf16 [T, Hkv, D]");
    const int64_t T = k_new->shape[0];
    for (int i = 0; i < 3; ++i)
        if (k_new->shape[i] != v_new->shape[i] || k_new->stride[i] != v_new->stride[i])
            return fail(B2PA_ERR_INVALID_ARG, "k_new and v_new must have equal shapes and strides");
    if (T < 0 || T > 0x7FFFFFFF || k_new->shape[1] != pr.Hkv || k_new->shape[2] != pr.D)
        return fail(B2PA_ERR_INVALID_ARG, "k_new must be [T, Hkv, D] with the pools' Hkv and D (T < 2^31)");
    if (pr.D % 8 != 0)
        return fail(B2PA_ERR_UNSUPPORTED, "head_dim must be a multiple of 8");
    if (!cache_loc || cache_loc->ndim != 1 || cache_loc->dtype != B2PA_INT32 || cache_loc->shape[0] != T)
        return fail(B2PA_ERR_INVALID_ARG, "cache_loc must be int32 [T]");
    if (pr.fp8 && (!std::isfinite(k_scale) || !(k_scale > 0.f) || !std::isfinite(v_scale) || !(v_scale > 0.f)))
        return fail(B2PA_ERR_INVALID_ARG, "k_scale / v_scale must be finite and > 0");
    if (T == 0)
        return B2PA_OK;  // empty tensors may carry null data pointers
    if (!k_new->data || !v_new->data)
        return fail(B2PA_ERR_INVALID_ARG, "k_new / v_new: null data");
    if ((pr.D > 1 && k_new->stride[2] != 1) || k_new->stride[0] % 8 != 0 || k_new->stride[1] % 8 != 0 ||
        !aligned16(k_new->data) || !aligned16(v_new->data))
        return fail(B2PA_ERR_INVALID_ARG,
                    "k_new / v_new: head_dim contiguous, token and head strides multiples of 8, 16-byte aligned");
    for (int i = 0; i < 3; ++i)
        if (pr.k_st[i] % 8 != 0 || pr.v_st[i] % 8 != 0)
            return fail(B2PA_ERR_INVALID_ARG, "pool page / head / slot strides must be multiples of 8 elements");
    if (!aligned16(pr.k) || !aligned16(pr.v))
        return fail(B2PA_ERR_INVALID_ARG, "pools must be 16-byte aligned");
    if ((long long)pr.N * pr.P > 0x7FFFFFFFLL)
        return fail(B2PA_ERR_UNSUPPORTED, "num_pages * page_size must be < 2^31 (int32 slots)");
    if (!is_vec(cache_loc, B2PA_INT32, T))
        return fail(B2PA_ERR_INVALID_ARG, "cache_loc must be contiguous int32 [T]");
    int dev;
    DevInfo di;
    if ((st = device_info(&dev, &di)))
        return st;
    Workspace ws;
    if ((st = get_workspace(dev, stream, 1, &ws)))
        return st;
    AppendParams ap;
    std::memset(&ap, 0, sizeof ap);
    ap.k_new = static_cast<const uint16_t*>(k_new->data);
    ap.v_new = static_cast<const uint16_t*>(v_new->data);
    ap.new_st_tok = k_new->stride[0];
    ap.new_st_head = k_new->stride[1];
    ap.k_pool = const_cast<void*>(pr.k);
    ap.v_pool = const_cast<void*>(pr.v);
    for (int i = 0; i < 3; ++i) {
        ap.k_st[i] = pr.k_st[i];
        ap.v_st[i] = pr.v_st[i];
    }
    ap.cache_loc = static_cast<const int*>(cache_loc->data);
    ap.T = (int)T;
    ap.Hkv = pr.Hkv;
    ap.D = pr.D;
    ap.page_size = pr.P;
    ap.num_pages = pr.N;
    ap.k_scale = k_scale;
    ap.v_scale = v_scale;
    ap.err = reinterpret_cast<unsigned*>(ws.mem);
    cudaError_t e = launch_append(ap, pr.fp8, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "append launch");
    return B2PA_OK;
}

int b2pa_get_device_status(b2pa_stream_t stream_h, uint32_t* bits_out)
{
    g_last_error.clear();
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_h);
    if (bits_out)
        *bits_out = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    Workspace ws;
    if (!find_workspace(dev, stream, &ws)) {
        if ((e = cudaStreamSynchronize(stream)) != cudaSuccess)
            return cuda_fail(e, "cudaStreamSynchronize");
        return B2PA_OK;
    }
    uint32_t bits = 0;
    if ((e = cudaMemcpyAsync(&bits, ws.mem, sizeof bits, cudaMemcpyDeviceToHost, stream)) != cudaSuccess ||
        (e = cudaMemsetAsync(ws.mem, 0, sizeof bits, stream)) != cudaSuccess ||
        (e = cudaStreamSynchronize(stream)) != cudaSuccess)
        return cuda_fail(e, "reading the device error word");
    if (bits_out)
        *bits_out = bits;
    return bits ? B2PA_ERR_DEVICE : B2PA_OK;
}

int b2pa_set_kernel_path(int32_t path)
{
    if (path != B2PA_PATH_AUTO && path != B2PA_PATH_TCGEN05 && path != B2PA_PATH_GENERIC)
        return fail(B2PA_ERR_INVALID_ARG, "unknown kernel path %d", path);
    g_path.store(path);
    return B2PA_OK;
}

int b2pa_query_path(const b2pa_tensor* q, const b2pa_tensor* k_pool, const b2pa_tensor* v_pool, const b2pa_tensor* out,
                    int32_t layout)
{
    g_last_error.clear();
    Problem pr;
    std::memset(&pr, 0, sizeof pr);
    int st = parse_pools(k_pool, v_pool, layout, &pr);
    if (st)
        return st;
    if (!q || !q->data || q->ndim != 3 || q->dtype != B2PA_BF16 || q->shape[2] != pr.D || q->shape[1] < 1 ||
        q->shape[1] % pr.Hkv)
        return fail(B2PA_ERR_INVALID_ARG, "q");
    if (!out || !out->data || out->ndim != 3)
        return fail(B2PA_ERR_INVALID_ARG, "out");
    pr.T = (int)q->shape[0];
    pr.H = (int)q->shape[1];
    pr.q = q->data;
    pr.q_st_tok = q->stride[0];
    pr.q_st_head = q->stride[1];
    pr.out = out->data;
    pr.out_st_tok = out->stride[0];
    pr.out_st_head = out->stride[1];
    int dev;
    DevInfo di;
    if ((st = device_info(&dev, &di)))
        return st;
    bool use_tc = false;
    if ((st = choose_path(pr, di, &use_tc)))
        return st;
    return use_tc ? B2PA_PATH_TCGEN05 : B2PA_PATH_GENERIC;
}

int b2pa_set_timing_events(void* start_event, void* stop_event)
{
    const bool on = start_event != nullptr && stop_event != nullptr;
    g_ev_start.store(on ? start_event : nullptr);
    g_ev_stop.store(on ? stop_event : nullptr);
    return B2PA_OK;
}

int b2pa_set_wait_limit_ns(uint64_t limit_ns)
{
    g_wait_limit_ns.store(limit_ns == 0 ? kWaitLimitNs : (unsigned long long)limit_ns);
    return B2PA_OK;
}

int b2pa_debug_inject_stall(int32_t on)
{
    g_inject_stall.store(on ? 1 : 0);
    return B2PA_OK;
}

int b2pa_set_debug_checks(int32_t on)
{
    g_debug.store(on ? 1 : 0);
    return B2PA_OK;
}

const char* b2pa_status_string(int32_t status)
{
    switch (status) {
    case B2PA_OK:
        return "B2PA_OK";
    case B2PA_ERR_INVALID_ARG:
        return "B2PA_ERR_INVALID_ARG";
    case B2PA_ERR_UNSUPPORTED:
        return "B2PA_ERR_UNSUPPORTED";
    case B2PA_ERR_CUDA:
        return "B2PA_ERR_CUDA";
    case B2PA_ERR_DEVICE:
        return "B2PA_ERR_DEVICE";
    default:
        return "B2PA_UNKNOWN_STATUS";
    }
}

const char* b2pa_last_error_message(void) { return g_last_error.c_str(); }

void b2pa_release(void)
{
    std::lock_guard<std::mutex> lk(g_ws_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    for (auto& w : g_ws) {
        cudaSetDevice(w.dev);
        cudaFree(w.mem);
    }
    cudaSetDevice(cur);
    g_ws.clear();
}

}  // extern "C"

// ====================================================================== allocation-free entry point
//
// b2pa_context_attention_noalloc runs the same tensor-core attention kernel
// as b2pa_context_attention, but the scratch it needs (the error word, the
// work-distribution words and the work list) lives in the fixed array below
// instead of a cudaMalloc'd per-stream workspace.

namespace {

constexpr size_t kNoAllocItems = 65536;                                 // work items at most
constexpr size_t kNoAllocBytes = kWsHeader + kNoAllocItems * sizeof(int4);  // 1 MiB + 256 B

}  // namespace

// Shared by every call of the allocation-free entry point on a device; each
// GPU that loads this library holds one copy until the process exits.  Host
// code must not use this name as an address: it resolves it per device with
// cudaGetSymbolAddress (noalloc_scratch below).
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocBytes];

namespace {

std::mutex g_noalloc_mu;
uint8_t* g_noalloc_ptr[64] = {};  // device address of g_noalloc_scratch, per device ordinal

// Device address of the scratch on device `dev` (which must be current);
// looked up once per device.
int noalloc_scratch(int dev, uint8_t** out)
{
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaGetSymbolAddress(allocation-free scratch)");
        g_noalloc_ptr[dev] = static_cast<uint8_t*>(ptr);
    }
    *out = g_noalloc_ptr[dev];
    return B2PA_OK;
}

}  // namespace

extern "C" {

int b2pa_context_attention_noalloc(const b2pa_tensor* q, const b2pa_tensor* k_pool, const b2pa_tensor* v_pool,
                                   const b2pa_tensor* block_tables, const b2pa_tensor* seq_lens,
                                   const b2pa_tensor* cum_q, const b2pa_tensor* cum_kv, int32_t max_q_len,
                                   int32_t max_kv_len, float bmm1_scale, float bmm2_scale, int32_t window_left,
                                   const b2pa_tensor* sinks, int32_t layout, b2pa_tensor* out,
                                   uint32_t* dev_status, b2pa_stream_t stream_h)
{
    g_last_error.clear();
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_h);
    Problem pr;
    int st = parse_problem(q, k_pool, v_pool, block_tables, seq_lens, cum_q, cum_kv, sinks, layout, out, &pr);
    if (st)
        return st;
    if (max_q_len < 0 || max_kv_len < 0)
        return fail(B2PA_ERR_INVALID_ARG, "max_q_len / max_kv_len must be >= 0");
    if (!std::isfinite(bmm1_scale) || !(bmm1_scale > 0.f) || !std::isfinite(bmm2_scale))
        return fail(B2PA_ERR_INVALID_ARG, "bmm1_scale must be finite and > 0, bmm2_scale finite");
    const size_t cap = items_needed(pr, max_q_len);
    if (cap > kNoAllocItems)
        return fail(B2PA_ERR_INVALID_ARG,
                    "these bounds need %zu work items; the allocation-free entry point holds at most %zu "
                    "(batch x kv heads x ceil(max_q_len / (2 x 128 / group size))); use b2pa_context_attention",
                    cap, kNoAllocItems);
    if (pr.B == 0 || pr.T == 0) {
        if (dev_status) {
            cudaError_t e = cudaMemsetAsync(dev_status, 0, sizeof(uint32_t), stream);
            if (e != cudaSuccess)
                return cuda_fail(e, "cudaMemsetAsync(dev_status)");
        }
        return B2PA_OK;
    }
    int dev;
    DevInfo di;
    if ((st = device_info(&dev, &di)))
        return st;
    if (const char* why = tc_reject(pr, di))
        return fail(B2PA_ERR_UNSUPPORTED, "the allocation-free entry point runs the tensor-core path only: %s", why);
    uint8_t* mem = nullptr;
    if ((st = noalloc_scratch(dev, &mem)))
        return st;
    const Workspace ws{dev, stream, mem, kNoAllocBytes};
    const int window = window_left < 0 ? -1 : window_left;
    SchedParams sp = make_sched(pr, ws, max_q_len, max_kv_len, window, cap);
    AttnParams ap;
    if ((st = fill_attn_params(&ap, pr, sp, cap, window, bmm1_scale, bmm2_scale)))
        return st;
    // the error word must start at zero (the kernel leaves its work-distribution words at zero itself)
    cudaError_t e = cudaMemsetAsync(mem, 0, sizeof(uint32_t), stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemsetAsync(error word)");
    if ((e = launch_tc_kernel(ap, pr, window, false, di.sms, stream)) != cudaSuccess)
        return cuda_fail(e, "attention kernel launch");
    if (dev_status && (e = cudaMemcpyAsync(dev_status, mem, sizeof(uint32_t), cudaMemcpyDeviceToDevice, stream)) !=
                          cudaSuccess)
        return cuda_fail(e, "cudaMemcpyAsync(dev_status)");
    return B2PA_OK;
}

}  // extern "C"
