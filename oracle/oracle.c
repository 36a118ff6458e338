/*
 * oracle.c -- plain, slow fp64 CPU oracle for batched context (prefill)
 * attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  It shares no code, header, table
 * or helper with the CUDA path; both take their inputs from the seeded
 * generator module (workload.py) and nothing else.
 *
 * What it computes, and where each step comes from:
 *
 *  - The call and its arguments: flashinfer.prefill.trtllm_batch_context_with_kv_cache
 *    (FlashInfer API reference, parameter list): query [num_tokens, num_heads,
 *    head_dim]; K and V pools [num_pages, num_kv_heads, page_size, head_dim]
 *    (HND) or [num_pages, page_size, num_kv_heads, head_dim] (NHD); page table
 *    block_tables [batch, max_pages]; seq_lens = kv length per request;
 *    cum_seq_lens_q delimiting each request's query tokens; window_left = the
 *    left, inclusive window (-1 = whole sequence); bmm1_scale on Q K^T,
 *    bmm2_scale on P V; sinks = one extra per-head term of the softmax
 *    denominator.
 *  - Addressing: a table entry is a page id; token t of a request lives on
 *    page block_tables[b][t / page_size] in slot t % page_size
 *    (TensorRT-LLM teardown (6), "Attention Backend 的 prepare() 内部",
 *    sections "块偏移张量的四维布局" and "句柄到偏移的物理含义": address =
 *    pool base + block id x block stride).
 *  - The attention itself: gather the first kv_len logical tokens of a
 *    request into a contiguous [tokens, kv_heads, head_dim] K and V and run
 *    plain masked softmax attention on them (same page, section
 *    "三条路径之一：VanillaAttention", _gather_paged_kv).
 *  - Causal alignment: query i of a request with q_len queries and kv_len keys
 *    sits at position kv_len - q_len + i, because the kv length is cached
 *    prefix plus new tokens and the queries are the new tokens (TokenSpeed
 *    backends/trtllm.py, _init_extend_metadata; TensorRT-LLM teardown (6),
 *    section "步骤三" kv_lens = cached + new).
 *
 * Readings taken where the pages leave a point open:
 *  - a query head h uses kv head h / (num_heads / num_kv_heads);
 *  - window_left = W >= 0 keeps keys j with pos - W <= j <= pos (W + 1 keys);
 *  - sinks are in the units of the scaled logits (after bmm1_scale) and add
 *    exp(sink - m) to the denominator only; bmm2_scale multiplies the
 *    normalised output;
 *  - FP8 e4m3 elements are decoded exactly (OCP 8-bit floating point format:
 *    1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,
 *    S.1111.111 = NaN).
 *
 * Everything is computed in double precision from the caller's bytes.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_BF16 1
#define OR_FP8_E4M3 2
#define OR_HND 0
#define OR_NHD 1

typedef struct {
    const void* data;
    int32_t dtype;        /* OR_BF16 or OR_FP8_E4M3 */
    int32_t pad_;
    int64_t shape[4];     /* in the tensor's own order (HND: N,Hkv,P,D; NHD: N,P,Hkv,D) */
    int64_t stride[4];    /* element strides in the same order */
} oracle_pool;

/* bf16 is the upper half of an IEEE binary32. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3: bias 7; exponent field 0 is subnormal (m/8 * 2^-6);
 * S.1111.111 is NaN; there is no infinity. */
double oracle_e4m3_value(uint8_t x)
{
    int sign = x >> 7;
    int e = (x >> 3) & 0xF;
    int m = x & 0x7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

double oracle_bf16_value(uint16_t bits) { return bf16_value(bits); }

static int pool_page_size(const oracle_pool* p, int layout)
{
    return (int)(layout == OR_HND ? p->shape[2] : p->shape[1]);
}

static int pool_kv_heads(const oracle_pool* p, int layout)
{
    return (int)(layout == OR_HND ? p->shape[1] : p->shape[2]);
}

/* element offset of (page, kv head, slot, d) */
static int64_t pool_offset(const oracle_pool* p, int layout, int64_t page, int64_t head,
                           int64_t slot, int64_t d)
{
    if (layout == OR_HND)
        return page * p->stride[0] + head * p->stride[1] + slot * p->stride[2] + d * p->stride[3];
    return page * p->stride[0] + slot * p->stride[1] + head * p->stride[2] + d * p->stride[3];
}

static double pool_value(const oracle_pool* p, int64_t off)
{
    if (p->dtype == OR_BF16)
        return bf16_value(((const uint16_t*)p->data)[off]);
    return oracle_e4m3_value(((const uint8_t*)p->data)[off]);
}

/* Logical key t of request b -> element offset of (t, kv head, d), through the
 * page table.  Returns -1 if the page id is outside the pool. */
static int64_t key_offset(const oracle_pool* p, int layout, const int32_t* block_tables,
                          int64_t bt_stride, int b, int64_t t, int head, int d)
{
    int P = pool_page_size(p, layout);
    int32_t page = block_tables[(int64_t)b * bt_stride + t / P];
    if (page < 0 || page >= p->shape[0])
        return -1;
    return pool_offset(p, layout, page, head, t % P, d);
}

/*
 * Gather: write the first seq_lens[b] logical K (or V) tokens of every
 * request, raw element bytes, to out[(cum_kv[b] + t) * Hkv * D + h * D + d].
 * This is the Vanilla backend's _gather_paged_kv, for every request.
 * Returns 0, or -1 if a referenced page id is outside the pool.
 */
int oracle_gather(const oracle_pool* pool, int layout, const int32_t* block_tables,
                  int64_t bt_stride, const int32_t* seq_lens, const int32_t* cum_kv, int B,
                  void* out)
{
    int Hkv = pool_kv_heads(pool, layout);
    int D = (int)pool->shape[3];
    int esize = pool->dtype == OR_BF16 ? 2 : 1;
    int bad = 0;
    for (int b = 0; b < B; ++b) {
        for (int64_t t = 0; t < seq_lens[b]; ++t) {
            for (int h = 0; h < Hkv; ++h) {
                for (int d = 0; d < D; ++d) {
                    int64_t src = key_offset(pool, layout, block_tables, bt_stride, b, t, h, d);
                    int64_t dst = ((int64_t)cum_kv[b] + t) * Hkv * D + (int64_t)h * D + d;
                    if (src < 0) {
                        bad = 1;
                        memset((char*)out + dst * esize, 0, esize);
                        continue;
                    }
                    memcpy((char*)out + dst * esize, (const char*)pool->data + src * esize, esize);
                }
            }
        }
    }
    return bad ? -1 : 0;
}

/*
 * The ragged page table (FlashInfer's paged_kv_indices / paged_kv_indptr /
 * paged_kv_last_page_len; TensorRT-LLM teardown (6), section "三条路径之二:
 * FlashInferAttentionMetadata——page table 三件套"): the page ids of every
 * request concatenated into one flat array, indptr[b] .. indptr[b + 1] the
 * slice of request b, and last_page_len[b] the valid tokens in its last page.
 *
 * Kv length of request b: its pages hold P tokens each except the last, which
 * holds last_page_len[b]: (pages - 1) * P + last_page_len[b], or 0 without
 * pages.  A negative page count, or a last_page_len outside [1, P] with pages,
 * is malformed: length -1.
 */
void oracle_ragged_lengths(const int32_t* indptr, const int32_t* last_page_len, int B, int P, int32_t* kv_len)
{
    for (int b = 0; b < B; ++b) {
        int64_t pages = (int64_t)indptr[b + 1] - indptr[b];
        if (pages < 0 || indptr[b] < 0) {
            kv_len[b] = -1;
        } else if (pages == 0) {
            kv_len[b] = 0;
        } else {
            int last = last_page_len[b];
            kv_len[b] = (last < 1 || last > P) ? -1 : (int32_t)((pages - 1) * P + last);
        }
    }
}

/*
 * Gather through the ragged page table: token t of request b lives on page
 * indices[indptr[b] + t / P], slot t % P; the first kv_len(b) tokens go to
 * out[(cum_kv[b] + t) * Hkv * D + h * D + d] (raw element bytes).  Returns 0,
 * or -1 if a request is malformed or a page id is outside the pool.
 */
int oracle_gather_ragged(const oracle_pool* pool, int layout, const int32_t* indices, const int32_t* indptr,
                         const int32_t* last_page_len, const int32_t* cum_kv, int B, void* out)
{
    int Hkv = pool_kv_heads(pool, layout);
    int D = (int)pool->shape[3];
    int P = pool_page_size(pool, layout);
    int esize = pool->dtype == OR_BF16 ? 2 : 1;
    int bad = 0;
    int32_t* kv_len = (int32_t*)malloc(sizeof(int32_t) * (size_t)(B > 0 ? B : 1));
    oracle_ragged_lengths(indptr, last_page_len, B, P, kv_len);
    for (int b = 0; b < B; ++b) {
        if (kv_len[b] < 0) {
            bad = 1;
            continue;
        }
        for (int64_t t = 0; t < kv_len[b]; ++t) {
            int32_t page = indices[indptr[b] + t / P];
            for (int h = 0; h < Hkv; ++h) {
                for (int d = 0; d < D; ++d) {
                    int64_t dst = ((int64_t)cum_kv[b] + t) * Hkv * D + (int64_t)h * D + d;
                    if (page < 0 || page >= pool->shape[0]) {
                        bad = 1;
                        memset((char*)out + dst * esize, 0, esize);
                        continue;
                    }
                    int64_t src = pool_offset(pool, layout, page, h, t % P, d);
                    memcpy((char*)out + dst * esize, (const char*)pool->data + src * esize, esize);
                }
            }
        }
    }
    free(kv_len);
    return bad ? -1 : 0;
}

/*
 * Attention for a list of output rows.
 *
 * rows[r] = token * H + h selects output row r (rows == NULL: every row in
 * order).  out[r * D + d] receives, in double precision,
 *
 *     o = bmm2_scale * sum_j e^{s_j - m} V_j / (sum_j e^{s_j - m} + [sinks] e^{sink_h - m})
 *     s_j = bmm1_scale * <q[token, h, :], K_j>,   m = max_j s_j,
 *
 * over the visible keys j of that row: with i the row's index inside its
 * request, pos = kv_len - q_len + i, keys lo..pos with lo = 0 (W < 0) or
 * max(0, pos - W).  A row with no visible key gets 0.  status_out[r] is 0,
 * or 1 if the row's request is malformed (q_len > kv_len or negative), or 2
 * if a visible key points at a page outside the pool.
 *
 * nthreads <= 0 uses OpenMP's default thread count.  Returns the number of
 * threads used.
 */
int oracle_attention(const uint16_t* q, int64_t q_stride_tok, int64_t q_stride_head, int T, int H,
                     int D, const oracle_pool* k_pool, const oracle_pool* v_pool, int layout,
                     const int32_t* block_tables, int64_t bt_stride, const int32_t* seq_lens,
                     const int32_t* cum_q, int B, double bmm1_scale, double bmm2_scale,
                     int window_left, const float* sinks, const int64_t* rows, int64_t n_rows,
                     double* out, int32_t* status_out, int nthreads)
{
    int Hkv = pool_kv_heads(k_pool, layout);
    int G = H / Hkv;
    int threads = 1;
    if (rows == NULL)
        n_rows = (int64_t)T * H;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#else
    nthreads = 1;
#endif
    (void)nthreads;

#pragma omp parallel num_threads(nthreads)
    {
#ifdef _OPENMP
#pragma omp single
        threads = omp_get_num_threads();
#endif
        double* s = NULL;
        int64_t s_cap = 0;
        double* acc = (double*)malloc(sizeof(double) * (size_t)D);

#pragma omp for schedule(dynamic, 8)
        for (int64_t r = 0; r < n_rows; ++r) {
            int64_t row = rows ? rows[r] : r;
            int tok = (int)(row / H);
            int h = (int)(row % H);
            double* o = out + r * D;
            int32_t st = 0;
            for (int d = 0; d < D; ++d)
                o[d] = 0.0;

            /* the request that owns this token */
            int b = -1;
            for (int bb = 0; bb < B; ++bb)
                if (cum_q[bb] <= tok && tok < cum_q[bb + 1]) {
                    b = bb;
                    break;
                }
            if (b < 0) {
                status_out[r] = 1;
                continue;
            }
            int64_t q_len = cum_q[b + 1] - cum_q[b];
            int64_t kv_len = seq_lens[b];
            if (q_len > kv_len || kv_len < 0) {
                status_out[r] = 1;
                continue;
            }
            int64_t i = tok - cum_q[b];
            int64_t pos = kv_len - q_len + i;
            int64_t lo = window_left < 0 ? 0 : (pos - window_left > 0 ? pos - window_left : 0);
            int64_t n = pos - lo + 1;
            int hk = h / G;
            if (n <= 0) {
                status_out[r] = 0;
                continue;
            }
            if (n > s_cap) {
                free(s);
                s_cap = n;
                s = (double*)malloc(sizeof(double) * (size_t)s_cap);
            }

            /* s_j = bmm1 * q . K_j */
            const uint16_t* qrow = q + (int64_t)tok * q_stride_tok + (int64_t)h * q_stride_head;
            double m = -INFINITY;
            for (int64_t j = 0; j < n; ++j) {
                int64_t key = lo + j;
                double dot = 0.0;
                for (int d = 0; d < D; ++d) {
                    int64_t off = key_offset(k_pool, layout, block_tables, bt_stride, b, key, hk, d);
                    if (off < 0) {
                        st = 2;
                        break;
                    }
                    dot += bf16_value(qrow[d]) * pool_value(k_pool, off);
                }
                s[j] = bmm1_scale * dot;
                if (s[j] > m)
                    m = s[j];
            }

            /* denominator, with the sink term */
            double den = 0.0;
            for (int64_t j = 0; j < n; ++j)
                den += exp(s[j] - m);
            if (sinks)
                den += exp((double)sinks[h] - m);

            /* numerator */
            for (int d = 0; d < D; ++d)
                acc[d] = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                int64_t key = lo + j;
                double w = exp(s[j] - m);
                for (int d = 0; d < D; ++d) {
                    int64_t off = key_offset(v_pool, layout, block_tables, bt_stride, b, key, hk, d);
                    if (off < 0) {
                        st = 2;
                        break;
                    }
                    acc[d] += w * pool_value(v_pool, off);
                }
            }
            for (int d = 0; d < D; ++d)
                o[d] = bmm2_scale * acc[d] / den;
            status_out[r] = st;
        }
        free(s);
        free(acc);
    }
    return threads;
}

/*
 * Work list of the tiled GPU schedule, written out from its definition so
 * the scheduler kernel's list can be checked bit for bit.
 *
 * One item per (request b, kv head, group of n_qtiles query tiles); a query
 * tile holds rows_per_tile consecutive tokens of one request (all the
 * num_heads/num_kv_heads query heads of the kv head for each token).  Item it
 * of request b starts at token it * n_qtiles * rows_per_tile.  For its tokens
 * i0..i1 (i1 clipped to q_len - 1) the visible keys span
 * [lo(prefix + i0), prefix + i1] with lo as in oracle_attention, so the kv
 * tiles of width kv_tile touched are lo / kv_tile .. (prefix + i1) / kv_tile.
 * cost = (number of those kv tiles) * (number of non-empty query tiles).
 *
 * Items of requests that violate q_len <= kv_len, q_len <= max_q_len,
 * kv_len <= max_kv_len, ceil(kv_len / page_size) <= max_pages,
 * cum_q[b] >= 0 or cum_q[b+1] <= num_tokens are not emitted.
 *
 * Order: by min(cost, cost_cap) descending; ties keep the enumeration order
 * (b ascending, then it, then kv head: the kv heads of one query item share
 * its cost and sit side by side).  items_out gets 4 ints per item:
 * b, kv head, it, cost.  Returns the number of items (or -1 if more than
 * cap would be written).
 */
int oracle_worklist(const int32_t* cum_q, const int32_t* seq_lens, int B, int num_kv_heads,
                    int rows_per_tile, int n_qtiles, int kv_tile, int window_left, int max_q_len,
                    int max_kv_len, int page_size, int max_pages, int num_tokens, int cost_cap,
                    int32_t* items_out, int cap)
{
    /* enumerate */
    int64_t n = 0;
    int64_t alloc = 1024;
    int32_t* tmp = (int32_t*)malloc(sizeof(int32_t) * 4 * (size_t)alloc);
    int per_item = rows_per_tile * n_qtiles;
    for (int b = 0; b < B; ++b) {
        int64_t q_len = (int64_t)cum_q[b + 1] - cum_q[b];
        int64_t kv_len = seq_lens[b];
        int ok = q_len >= 0 && q_len <= kv_len && q_len <= max_q_len && kv_len <= max_kv_len &&
                 (kv_len + page_size - 1) / page_size <= max_pages && cum_q[b] >= 0 &&
                 cum_q[b + 1] <= num_tokens;
        if (!ok || q_len == 0)
            continue;
        int64_t prefix = kv_len - q_len;
        int64_t n_items = (q_len + per_item - 1) / per_item;
        for (int64_t it = 0; it < n_items; ++it) {
            for (int hk = 0; hk < num_kv_heads; ++hk) {
                int64_t i0 = it * per_item;
                int64_t i1 = i0 + per_item - 1;
                if (i1 > q_len - 1)
                    i1 = q_len - 1;
                int64_t nq = (i1 - i0) / rows_per_tile + 1;
                int64_t p_min = prefix + i0, p_max = prefix + i1;
                int64_t lo = window_left < 0 ? 0 : (p_min - window_left > 0 ? p_min - window_left : 0);
                int64_t tiles = p_max / kv_tile - lo / kv_tile + 1;
                if (n == alloc) {
                    alloc *= 2;
                    tmp = (int32_t*)realloc(tmp, sizeof(int32_t) * 4 * (size_t)alloc);
                }
                tmp[4 * n + 0] = b;
                tmp[4 * n + 1] = hk;
                tmp[4 * n + 2] = (int32_t)it;
                tmp[4 * n + 3] = (int32_t)(tiles * nq);
                ++n;
            }
        }
    }
    if (n > cap) {
        free(tmp);
        return -1;
    }
    /* stable order by capped cost, descending: one pass per cost value */
    int64_t w = 0;
    for (int c = cost_cap; c >= 0; --c) {
        for (int64_t k = 0; k < n; ++k) {
            int cost = tmp[4 * k + 3];
            int key = cost < cost_cap ? cost : cost_cap;
            if (key == c) {
                memcpy(items_out + 4 * w, tmp + 4 * k, 4 * sizeof(int32_t));
                ++w;
            }
        }
    }
    free(tmp);
    return (int)n;
}

/*
 * Writing new tokens' K and V into the paged pools: the step before the
 * attention in the TokenSpeed trtllm backend (_save_kv_and_prepare_q), which
 * calls fused_fp8_set_kv_buffer(k, v, k_cache, v_cache, cache_loc, k_scale,
 * v_scale, page_size) for an e4m3 cache and set_kv_buffer otherwise.  Token n's
 * rows k[n, h, :] and v[n, h, :] go to cache slot cache_loc[n]: page
 * cache_loc[n] / page_size, slot cache_loc[n] % page_size (the page / slot
 * addressing of the attention's gather above).
 *
 * Readings (the pages print the call, not its kernel):
 *  - a bf16 pool receives the bf16 values unchanged; the scales apply to an
 *    e4m3 pool only;
 *  - an e4m3 pool receives x / scale, the quotient taken in IEEE binary32,
 *    rounded to the nearest e4m3 value with ties to the even code; magnitudes
 *    above the largest finite value, 448, saturate to it;
 *  - a slot outside [0, num_pages * page_size) is not written.
 */

/* Nearest e4m3 code to x.  The non-negative finite codes 0x00 .. 0x7E have
 * increasing values, so a binary search finds the largest code whose value is
 * not above |x|; the answer is the nearer of it and the next code, the even
 * one on a tie.  NaN maps to 0x7F. */
uint8_t oracle_e4m3_encode(float x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7E;
    int lo = 0, hi = 0x7E; /* value(lo) <= a < value(hi) */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (oracle_e4m3_value((uint8_t)mid) <= a)
            lo = mid;
        else
            hi = mid;
    }
    double below = a - oracle_e4m3_value((uint8_t)lo), above = oracle_e4m3_value((uint8_t)hi) - a;
    int c = below < above ? lo : (above < below ? hi : ((lo & 1) ? hi : lo));
    return sign | (uint8_t)c;
}

static void store_elem(const oracle_pool* p, int64_t off, uint16_t bits, float scale)
{
    if (p->dtype == OR_BF16) {
        ((uint16_t*)p->data)[off] = bits;
    } else {
        float x = (float)bf16_value(bits); /* exact */
        float q = x / scale;               /* one binary32 division */
        ((uint8_t*)p->data)[off] = oracle_e4m3_encode(q);
    }
}

/* k_new / v_new: bf16 [T, num_kv_heads, head_dim], element strides st_tok,
 * st_head, head_dim contiguous.  The pools are written in place.  Returns the
 * number of tokens whose slot lies outside the pool. */
int64_t oracle_append_kv(const uint16_t* k_new, const uint16_t* v_new, int64_t T, int64_t st_tok,
                         int64_t st_head, const int32_t* cache_loc, const oracle_pool* k_pool,
                         const oracle_pool* v_pool, int layout, float k_scale, float v_scale)
{
    int P = pool_page_size(k_pool, layout);
    int H = pool_kv_heads(k_pool, layout);
    int D = (int)k_pool->shape[3];
    int64_t slots = k_pool->shape[0] * (int64_t)P;
    int64_t outside = 0;
    for (int64_t n = 0; n < T; ++n) {
        int64_t loc = cache_loc[n];
        if (loc < 0 || loc >= slots) {
            ++outside;
            continue;
        }
        int64_t page = loc / P, slot = loc % P;
        for (int h = 0; h < H; ++h)
            for (int d = 0; d < D; ++d) {
                int64_t src = n * st_tok + (int64_t)h * st_head + d;
                store_elem(k_pool, pool_offset(k_pool, layout, page, h, slot, d), k_new[src], k_scale);
                store_elem(v_pool, pool_offset(v_pool, layout, page, h, slot, d), v_new[src], v_scale);
            }
    }
    return outside;
}
