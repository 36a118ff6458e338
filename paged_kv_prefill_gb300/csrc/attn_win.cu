// attn_win.cu -- the sliding-window variant of the tensor-core attention for
// head_dim 64 (16-bit KV): one kv "window tile" per work item.
//
// Same operation as attn_tc.cu (flashinfer.prefill.trtllm_batch_context_with_kv_cache,
// FlashInfer API reference, parameter list; window_left as there).  A work item
// is again (request b, kv head, item index) with two query tiles of 128 MMA
// rows.  With a left window W, the keys any row of the item can see lie in
// [p_first - W, p_last], at most 2 * rows_per_tile + W keys.  When that span,
// widened to whole pages, fits in kWinKeys = 192 keys, the item needs one tile
// of 192 keys starting at a page boundary instead of two or three 128-key
// tiles: S_t = Q_t K^T is one MMA group of N = 192, the softmax makes one
// pass for the maximum and one for the exponentials (no running rescale), and
// O_t = P_t V is one MMA group of 12 steps.  The host takes this kernel for
// such windows (b2pa.cu, win_eligible); the multi-tile kernel stays the path
// for everything else.
//
//   warp 0      producer: item fetch (as attn_tc.cu), TMA of Q into a ring of
//               two Q buffers, TMA of the item's K and V window pages into a
//               ring of two K/V pairs (one box per page).
//   warp 1      MMA issuer: S_0(n+1) after P_0 V(n), S_1(n+1) after P_1 V(n).
//   warps 4-7   softmax and epilogue of query tile 0; warps 8-11 of tile 1.
//
// TMEM (512 columns): S0 [0,192), S1 [192,384), O0 [384,448), O1 [448,512);
// P_t (bf16, two keys per column) overwrites the first 96 columns of S_t.
#include <mutex>

#include "attn_common.cuh"
#include "common.cuh"
#include "ptx.cuh"
#include "worklist.cuh"

namespace b2pa {

struct WinCfg {
    static constexpr int D = 64;
    static constexpr int kWinKeys = 192;
    static constexpr int kQBufs = 2;
    static constexpr int kQTileBytes = kQRows * 128;            // 128 rows x 64 bf16
    static constexpr int kKvBytes = kWinKeys * 128;             // 192 key rows x 64 bf16
    static constexpr int kPairs = 2;                            // items whose K/V are in the ring
    static constexpr int kThreads = 384;
    static constexpr int kItemSlots = 4;
    static constexpr int kItemConsumerWarps = 1 + 8;
    static constexpr int kTmemCols = 512;
    static constexpr int kOCol = 2 * kWinKeys;
    static constexpr int kOffQ = 0;
    static constexpr int kOffRing = kOffQ + kQBufs * kQTiles * kQTileBytes;
    static constexpr int kStageWarpBytes = 32 * 128;
    static constexpr int kOffStage = kOffRing + kPairs * 2 * kKvBytes;
    static constexpr int kOffBar = kOffStage + 8 * kStageWarpBytes;
    static constexpr int kNumBars = 2 * kPairs + 2 * kQBufs + 3 * kQTiles + 1 + 2 * kItemSlots + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kOffFirst = (kOffMisc + 16 + kItemSlots * kItemRecWords * 4 + 15) / 16 * 16;
    static constexpr int kSmemBytes = kOffFirst + 16 + 1024;
    static_assert(kOCol + kQTiles * D <= kTmemCols, "tmem");
    static_assert(kSmemBytes <= 232448, "shared memory");
    // the work list is sorted in the K/V ring and the output staging at the start
    static_assert(worklist_smem_ints(kThreads / 32, kSchedBuckets, kSchedMaxBatch) * sizeof(int) <=
                      (size_t)(kOffBar - kOffRing),
                  "work-list scratch");
};

// First key of an item's window tile: the first row's window start, rounded
// down to its page.
__device__ __forceinline__ int win_first_key(const ItemInfo& it, int window, int log2_p)
{
    const int p_first = it.kv_len - it.q_len + it.g.tok0;
    const int lo = max(0, p_first - window);
    return (lo >> log2_p) << log2_p;
}

// ---------------------------------------------------------------------------
// Producer: warp 0.
// ---------------------------------------------------------------------------
__device__ void win_producer(const AttnParams& p, const Ctx& c)
{
    using C = WinCfg;
    const int lane = threadIdx.x & 31;
    const uint32_t q_smem = smem_u32(c.base + C::kOffQ);
    const uint32_t ring = smem_u32(c.base + C::kOffRing);
    const int P = p.page_size;
    const int log2_p = 31 - __clz(P);
    const int pages = C::kWinKeys >> log2_p;  // pages per window tile (P <= 32 here)
    const uint32_t q_box_bytes = (uint32_t)(p.G * p.rows_per_tile * 128);
    uint32_t kv_loads = 0, q_loads = 0;
    bool list_ready = false;
    bool ok = true;
    const bool scales_ok = load_scales(p.scale_log2, p.bmm2, p.bmm1_dev, p.bmm2_dev).ok;
    if (!scales_ok && blockIdx.x == 0 && lane == 0)
        atomicOr(p.err, (unsigned)B2PA_DEV_BAD_SCALE);
    for (uint32_t n = 0; ok; ++n) {
        const uint32_t slot = n % C::kItemSlots;
        if (!wait_bar(&c.bar.it_empty[slot], ((n / C::kItemSlots) & 1) ^ 1, c))
            break;
        volatile int* rec = c.item_slot + slot * kItemRecWords;
        if (lane == 0) {
            int w = -1;
            int4 item = *reinterpret_cast<const int4*>(c.base + C::kOffFirst);
            if (scales_ok && n == 0) {
                w = item.x >= 0 && (int)blockIdx.x < c.n_items ? (int)blockIdx.x : -1;
            } else if (scales_ok) {
                w = (int)gridDim.x + atomicAdd(p.counter, 1);
                if (w >= c.n_items)
                    w = -1;
                if (w >= 0 && !list_ready) {
                    list_ready = wait_list_ready(p.ready, c);
                    if (!list_ready)
                        w = -1;
                }
                if (w >= 0)
                    item = p.items[w];
            }
            rec[0] = w;
            if (w >= 0) {
                const ItemInfo r = read_item<false>(p, item);
                rec[1] = r.b;
                rec[2] = r.kvh;
                rec[3] = r.q0;
                rec[4] = r.q_len;
                rec[5] = r.kv_len;
                rec[6] = r.g.tok0;
                rec[7] = r.g.nq;
                rec[8] = r.g.n_lo;
                rec[9] = r.g.n_hi;
                rec[10] = r.chunk;
                rec[11] = r.chunks;
            }
            mbar_arrive(&c.bar.it_full[slot]);
        }
        __syncwarp();
        const int w = rec[0];
        if (w < 0)
            break;
        ItemInfo it;
        it.b = rec[1];
        it.kvh = rec[2];
        it.q0 = rec[3];
        it.q_len = rec[4];
        it.kv_len = rec[5];
        it.g.tok0 = rec[6];
        it.g.nq = rec[7];
        // Q tiles into buffer n % 2 once its previous item's last Q K^T is done
        const uint32_t qb = n % C::kQBufs, qph = (n / C::kQBufs) & 1;
        if (!wait_bar(&c.bar.q_empty[qb], qph ^ 1, c))
            break;
        if (lane == 0)
            mbar_arrive_expect_tx(&c.bar.q_full[qb], (uint32_t)it.g.nq * q_box_bytes);
        __syncwarp();
        if (lane < it.g.nq)
            tma_load_3d(q_smem + (qb * kQTiles + lane) * C::kQTileBytes, &p.tm_q, &c.bar.q_full[qb], 0,
                        it.kvh * p.G, it.q0 + it.g.tok0 + lane * p.rows_per_tile);
        q_loads = n + 1;
        // the window's pages: lane l loads page column k0 / P + l of K and of V
        const uint32_t m = n % C::kPairs, ph = (n / C::kPairs) & 1;
        if (!wait_bar(&c.bar.empty[m], ph ^ 1, c))
            break;
        const int* bt_row = page_row(p.block_tables, p.bt_stride, p.kv_indptr, it.b);
        const int n_pages_valid = (it.kv_len + P - 1) >> log2_p;
        const int col = (win_first_key(it, p.window, log2_p) >> log2_p) + lane;
        const bool valid = lane < pages && col < n_pages_valid;
        const int page = valid ? bt_row[col] : 0;
        if (valid && (page < 0 || page >= p.num_pages))
            atomicOr(p.err, (unsigned)B2PA_DEV_BAD_PAGE);
        const uint32_t nvalid = __popc(__ballot_sync(0xffffffffu, valid));
        mbar_arrive_expect_tx_p(&c.bar.full[m], nvalid * (uint32_t)P * 128u * 2u, lane == 0 ? 1u : 0u);
        __syncwarp();
        const uint32_t dst = ring + 2 * m * C::kKvBytes + (uint32_t)(lane * P * 128);
        tma_load_4d_p(dst, &p.tm_k, &c.bar.full[m], 0, 0, it.kvh, page, valid ? 1u : 0u);
        tma_load_4d_p(dst + C::kKvBytes, &p.tm_v, &c.bar.full[m], 0, 0, it.kvh, page, valid ? 1u : 0u);
        kv_loads = n + 1;
    }
    if (*c.abort_flag) {
        // let the copies this warp started land before the CTA releases its memory
        const uint32_t q_first = q_loads > (uint32_t)C::kQBufs ? q_loads - C::kQBufs : 0;
        for (uint32_t k = q_first; k < q_loads; ++k)
            drain_wait(&c.bar.q_full[k % C::kQBufs], (k / C::kQBufs) & 1);
        const uint32_t kv_first = kv_loads > (uint32_t)C::kPairs ? kv_loads - C::kPairs : 0;
        for (uint32_t k = kv_first; k < kv_loads; ++k)
            drain_wait(&c.bar.full[k % C::kPairs], (k / C::kPairs) & 1);
    }
}

// ---------------------------------------------------------------------------
// MMA issuer: warp 1 (issue predicated on lane 0; the warp stays converged).
// ---------------------------------------------------------------------------
__device__ void win_mma(const AttnParams& p, const Ctx& c)
{
    using C = WinCfg;
    constexpr int D = C::D;
    constexpr uint32_t kIdescS = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(C::kWinKeys >> 3) << 17) |
                                 ((uint32_t)(kQRows >> 4) << 24);
    constexpr uint32_t kIdescO = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((uint32_t)(D >> 3) << 17) |
                                 ((uint32_t)(kQRows >> 4) << 24);
    const int lane = threadIdx.x & 31;
    const uint32_t issue = lane == 0 ? 1u : 0u;
    constexpr uint32_t kHi = sdesc_hi_sw128(1024);
    const uint32_t q_lo = sdesc_lo(smem_u32(c.base + C::kOffQ), 16);
    const uint32_t k_lo = sdesc_lo(smem_u32(c.base + C::kOffRing), 16);
    const uint32_t v_lo = sdesc_lo(smem_u32(c.base + C::kOffRing), kQRows * 128);  // MN-major: LBO unused at D = 64
    constexpr uint32_t kKvW = C::kKvBytes >> 4;
    constexpr uint32_t kQTileW = C::kQTileBytes >> 4;

    auto issue_s = [&](uint32_t qb, int t, uint32_t m) {
        const uint32_t a0 = q_lo + (qb * kQTiles + t) * kQTileW;
        const uint32_t b0 = k_lo + 2 * m * kKvW;
        const uint32_t d = c.tmem + (uint32_t)(t * C::kWinKeys);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
            mma_ss_wp(d, a0 + (uint32_t)(k * 2), b0 + (uint32_t)(k * 2), kHi, kIdescS, k > 0 ? 1u : 0u, issue);
    };
    auto issue_pv = [&](int t, uint32_t m) {
        const uint32_t b0 = v_lo + (2 * m + 1) * kKvW;
        const uint32_t d = c.tmem + (uint32_t)(C::kOCol + t * D);
        const uint32_t a = c.tmem + (uint32_t)(t * C::kWinKeys);
#pragma unroll
        for (int k = 0; k < C::kWinKeys / 16; ++k)
            mma_ts_wp(d, a + (uint32_t)(k * 8), b0 + (uint32_t)(k * 128), kHi, kIdescO, k > 0 ? 1u : 0u, issue);
    };
    // an item whose Q and K/V landed: V rows past kv_len zeroed, then its S MMAs
    struct Open {
        int nq;
        uint32_t qb, m;
        bool ok;
    };
    auto open_item = [&](const ItemInfo& it, uint32_t n) -> Open {
        Open o;
        o.nq = it.g.nq;
        o.qb = n % C::kQBufs;
        o.m = n % C::kPairs;
        o.ok = wait_bar(&c.bar.q_full[o.qb], (n / C::kQBufs) & 1, c) &&
               wait_bar(&c.bar.full[o.m], (n / C::kPairs) & 1, c);
        if (o.ok) {
            // keys >= kv_len: V rows may hold any bits (or a page that was not
            // loaded); zero them so that P = 0 there cannot meet a NaN
            const int r0 = it.kv_len - win_first_key(it, p.window, 31 - __clz(p.page_size));
            if (r0 < C::kWinKeys) {
                uint4* dst = reinterpret_cast<uint4*>(c.base + C::kOffRing + (2 * o.m + 1) * C::kKvBytes + r0 * 128);
                const int n16 = (C::kWinKeys - r0) * 8;
                for (int q = lane; q < n16; q += 32)
                    dst[q] = make_uint4(0u, 0u, 0u, 0u);
                fence_proxy_async_smem();
                __syncwarp();
            }
        }
        return o;
    };
    auto first_s = [&](const Open& o, int t) {
        issue_s(o.qb, t, o.m);
        mma_commit_p(&c.bar.s_full[t], issue);
        if (t == o.nq - 1)
            mma_commit_p(&c.bar.q_empty[o.qb], issue);
    };

    bool ok = true;
    uint32_t p_cnt[kQTiles] = {0, 0};  // P hand-offs of tile t seen so far
    if (p.inject_stall && !wait_bar(c.bar.never, 0, c))
        ok = false;
    ItemInfo info;
    int w = ok ? take_item<C::kItemSlots>(p, c, 0, &ok, &info) : -1;
    Open cur;
    if (w >= 0) {
        cur = open_item(info, 0);
        ok = cur.ok;
        for (int t = 0; ok && t < cur.nq; ++t)
            first_s(cur, t);
    }
    for (uint32_t n = 0; ok && w >= 0; ++n) {
        Open nxt;
        int w_next = -1;
#pragma unroll
        for (int t = 0; t < kQTiles; ++t) {
            if (t < cur.nq) {
                if (!wait_bar(&c.bar.p_full[t], p_cnt[t] & 1, c)) {
                    ok = false;
                    break;
                }
                ++p_cnt[t];
                tc_fence_after();
                issue_pv(t, cur.m);
                mma_commit_p(&c.bar.o_full[t], issue);
                if (t == cur.nq - 1)
                    mma_commit_p(&c.bar.empty[cur.m], issue);  // the item's K and V consumed
            }
            if (t == 0) {
                // the next item: its S_0 may overwrite P_0 of this one now
                w_next = take_item<C::kItemSlots>(p, c, n + 1, &ok, &info);
                if (!ok)
                    break;
                if (w_next >= 0) {
                    nxt = open_item(info, n + 1);
                    if (!nxt.ok) {
                        ok = false;
                        break;
                    }
                    first_s(nxt, 0);
                    if (cur.nq == 1 && nxt.nq > 1)
                        first_s(nxt, 1);
                }
            } else if (w_next >= 0 && nxt.nq > 1 && cur.nq > 1) {
                first_s(nxt, 1);
            }
        }
        if (!ok)
            break;
        w = w_next;
        cur = nxt;
    }
    if (lane == 0)
        mma_commit(c.bar.drain);
    __syncwarp();
    drain_wait(c.bar.drain, 0);
}

// ---------------------------------------------------------------------------
// Softmax and epilogue of query tile t: warps 4 + 4t .. 7 + 4t, one thread per
// row.  Per item: one pass over S_t's 192 columns for the row maximum, one for
// the exponentials (P written over the first 96 columns as it goes).
// ---------------------------------------------------------------------------
__device__ void win_softmax(const AttnParams& p, const Ctx& c, int t)
{
    using C = WinCfg;
    constexpr int D = C::D;
    constexpr float kLog2e = 1.4426950408889634f;
    const int wq = (threadIdx.x >> 5) & 3;
    const int lane = threadIdx.x & 31;
    const int row = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t s_tmem = c.tmem + lane_off + (uint32_t)(t * C::kWinKeys);
    const uint32_t o_tmem = c.tmem + lane_off + (uint32_t)(C::kOCol + t * D);
    const int G = p.G, Tq = p.rows_per_tile;
    const int r_tok = row / G, r_head = row % G;
    const bool row_real = row < G * Tq;
    const int log2_p = 31 - __clz(p.page_size);
    const Scales scl = load_scales(p.scale_log2, p.bmm2, p.bmm1_dev, p.bmm2_dev);
    bool ok = true;
    uint32_t n_mine = 0;  // items with a tile t (the phase of s_full / o_full)
    for (uint32_t n = 0; ok; ++n) {
        ItemInfo it;
        const int w = take_item<C::kItemSlots>(p, c, n, &ok, &it);
        if (w < 0)
            break;
        if (t >= it.g.nq)
            continue;
        const uint32_t ph = n_mine & 1;
        ++n_mine;
        const float sl2 = scl.scale_log2;
        const int k0 = win_first_key(it, p.window, log2_p);
        const int i_first = it.g.tok0 + t * Tq;
        const int i = i_first + r_tok;
        const bool valid = row_real && i < it.q_len;
        const int pos = it.kv_len - it.q_len + i;
        // the row's visible keys relative to the tile: [lo_r, hi_r]
        // the row's sink, read now so that its latency hides behind the passes
        const float sink = (p.sinks != nullptr && row_real) ? p.sinks[it.kvh * G + r_head] : 0.f;
        const int lo_r = (p.window < 0 ? 0 : max(0, pos - p.window)) - k0;
        const int hi_r = valid ? pos - k0 : -1;
        if (!wait_bar(&c.bar.s_full[t], ph, c)) {
            ok = false;
            break;
        }
        tc_fence_after();
        // Both passes read S_t in groups of two 32-column chunks, the two
        // loads of a group in flight together; the loop over groups is not
        // unrolled (measured: the smaller code runs 12 % faster).  Per chunk, decided for the
        // whole warp: every row sees all of it (its tcgen05.ld.red maximum
        // stands; plain exponentials), no row sees any of it (skipped; P = 0),
        // or masked element by element.
        constexpr int kGroup = 2;
        constexpr int kChunks = C::kWinKeys / 32;
        // pass 1: the row maximum over the visible keys
        float mx = -INFINITY;
#pragma unroll 1
        for (int g0 = 0; g0 < kChunks; g0 += kGroup) {
            uint32_t r[kGroup][32];
            float mq[kGroup];
#pragma unroll
            for (int u = 0; u < kGroup; ++u)
                tmem_ld32_max(s_tmem + (uint32_t)(32 * (g0 + u)), r[u], &mq[u]);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < kGroup; ++u) {
                const int c0 = 32 * (g0 + u);
                if (__all_sync(0xffffffffu, c0 >= lo_r && c0 + 31 <= hi_r)) {
                    mx = fmaxf(mx, mq[u]);
                } else if (!__all_sync(0xffffffffu, c0 > hi_r || c0 + 31 < lo_r)) {
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        if (c0 + k >= lo_r && c0 + k <= hi_r)
                            mx = fmaxf(mx, __uint_as_float(r[u][k]));
                }
            }
        }
        const float m = mx * sl2;  // log2 units
        const float neg = m == -INFINITY ? 0.f : -m;
        const float2 sc2 = make_float2(sl2, sl2), ng2 = make_float2(neg, neg);
        // pass 2: P = 2^(s * scale - m) for the visible keys, 0 elsewhere
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll 1
        for (int g0 = 0; g0 < kChunks; g0 += kGroup) {
            uint32_t r[kGroup][32];
#pragma unroll
            for (int u = 0; u < kGroup; ++u)
                tmem_ld32(s_tmem + (uint32_t)(32 * (g0 + u)), r[u]);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < kGroup; ++u) {
                const int c0 = 32 * (g0 + u);
                uint32_t pk[16];
                if (__all_sync(0xffffffffu, c0 >= lo_r && c0 + 31 <= hi_r)) {
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const float2 x = __ffma2_rn(
                            make_float2(__uint_as_float(r[u][2 * k]), __uint_as_float(r[u][2 * k + 1])), sc2, ng2);
                        const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                        acc = __fadd2_rn(acc, e);
                        pk[k] = pack_bf16x2(e.x, e.y);
                    }
                } else if (__all_sync(0xffffffffu, c0 > hi_r || c0 + 31 < lo_r)) {
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        pk[k] = 0u;
                } else {
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const int k2 = c0 + 2 * k;
                        const float2 x = __ffma2_rn(
                            make_float2(__uint_as_float(r[u][2 * k]), __uint_as_float(r[u][2 * k + 1])), sc2, ng2);
                        const float e0 = (k2 >= lo_r && k2 <= hi_r) ? ex2_approx(x.x) : 0.f;
                        const float e1 = (k2 + 1 >= lo_r && k2 + 1 <= hi_r) ? ex2_approx(x.y) : 0.f;
                        acc = __fadd2_rn(acc, make_float2(e0, e1));
                        pk[k] = pack_bf16x2(e0, e1);
                    }
                }
                tmem_st16(s_tmem + (uint32_t)(16 * (g0 + u)), pk);
            }
        }
        const float l = acc.x + acc.y;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        mbar_arrive_p(&c.bar.p_full[t], lane == 0 ? 1u : 0u);

        // epilogue: out = bmm2_scale * O / (l + e^{sink - m})
        if (!wait_bar(&c.bar.o_full[t], ph, c)) {
            ok = false;
            break;
        }
        tc_fence_after();
        const int h = it.kvh * G + r_head;
        float total = l;
        if (p.sinks != nullptr && m != -INFINITY && row_real)
            total += ex2_approx(fmaf(sink, kLog2e, -m));
        const float inv = (m != -INFINITY && total > 0.f) ? scl.bmm2 / total : 0.f;
        const float2 inv2 = make_float2(inv, inv);
        uint16_t* orow = p.out + (long long)(it.q0 + (valid ? i : 0)) * p.out_stride_tok + (long long)h * p.out_stride_head;
        // the warp's 32 rows x 64 columns through shared memory (128-byte
        // swizzle of the output tensor map), then one TMA store when the rows
        // are whole boxes, else 16-byte stores of whole rows
        const uint32_t stage = smem_u32(c.base + C::kOffStage + (t * 4 + wq) * C::kStageWarpBytes);
        const unsigned long long my_row = reinterpret_cast<unsigned long long>(orow);
        const bool by_tma = p.out_tma != 0 && __all_sync(0xffffffffu, valid);
        const int r0 = wq * 32;
        const int c1 = it.kvh * G + r0 % G, c2 = it.q0 + i_first + r0 / G;
        if (lane == 0)
            bulk_wait_read_all();  // the previous store has read the staging
        __syncwarp();
        uint32_t oa[32], ob[32];
        tmem_ld32(o_tmem, oa);
        tmem_ld32(o_tmem + 32u, ob);
        tmem_wait_ld();
        uint32_t pk[32];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const float2 va = __fmul2_rn(make_float2(__uint_as_float(oa[2 * k]), __uint_as_float(oa[2 * k + 1])), inv2);
            const float2 vb = __fmul2_rn(make_float2(__uint_as_float(ob[2 * k]), __uint_as_float(ob[2 * k + 1])), inv2);
            pk[k] = pack_bf16x2(va.x, va.y);
            pk[16 + k] = pack_bf16x2(vb.x, vb.y);
        }
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
            st_shared_v4(stage + (uint32_t)(lane * 128 + ((cc ^ (lane & 7)) << 4)), pk[4 * cc], pk[4 * cc + 1],
                         pk[4 * cc + 2], pk[4 * cc + 3]);
        if (by_tma) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_3d(&p.tm_o, stage, 0, c1, c2);
                bulk_commit_group();
            }
        } else {
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int rr = 4 * k + (lane >> 3), cc = lane & 7;
                const uint4 v = ld_shared_v4(stage + (uint32_t)(rr * 128 + ((cc ^ (rr & 7)) << 4)));
                const unsigned long long a = __shfl_sync(0xffffffffu, my_row, rr);
                const int vr = __shfl_sync(0xffffffffu, valid ? 1 : 0, rr);
                if (vr)
                    *reinterpret_cast<uint4*>(a + (unsigned long long)(cc * 16)) = v;
            }
            __syncwarp();
        }
    }
    if (lane == 0)
        bulk_wait_all();  // this warp's output stores are complete before the CTA exits
    tc_fence_before();
}

// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(WinCfg::kThreads, 1) attention_win_kernel(const __grid_constant__ AttnParams p)
{
    using C = WinCfg;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::kOffBar);
    Ctx c;
    c.base = base;
    c.bar.full = bars;
    c.bar.empty = c.bar.full + C::kPairs;
    c.bar.q_full = c.bar.empty + C::kPairs;
    c.bar.q_empty = c.bar.q_full + C::kQBufs;
    c.bar.s_full = c.bar.q_empty + C::kQBufs;
    c.bar.p_full = c.bar.s_full + kQTiles;
    c.bar.o_full = c.bar.p_full + kQTiles;
    c.bar.drain = c.bar.o_full + kQTiles;
    c.bar.it_full = c.bar.drain + 1;
    c.bar.it_empty = c.bar.it_full + C::kItemSlots;
    c.bar.never = c.bar.it_empty + C::kItemSlots;
    c.bar.vfull = c.bar.vempty = c.bar.f8full = c.bar.f8empty = c.bar.q_conv = nullptr;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base + C::kOffMisc);
    c.abort_flag = reinterpret_cast<volatile int*>(base + C::kOffMisc + 4);
    c.err = p.err;
    c.wait_limit_ns = p.wait_limit_ns;
    c.item_slot = reinterpret_cast<volatile int*>(base + C::kOffMisc + 16);
    const int warp = threadIdx.x >> 5;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kPairs; ++s) {
            mbar_init(&c.bar.full[s], 1);
            mbar_init(&c.bar.empty[s], 1);
        }
        for (int b = 0; b < C::kQBufs; ++b) {
            mbar_init(&c.bar.q_full[b], 1);
            mbar_init(&c.bar.q_empty[b], 1);
        }
        for (int t = 0; t < kQTiles; ++t) {
            mbar_init(&c.bar.s_full[t], 1);
            mbar_init(&c.bar.p_full[t], 4);
            mbar_init(&c.bar.o_full[t], 1);
        }
        mbar_init(c.bar.drain, 1);
        for (int s = 0; s < C::kItemSlots; ++s) {
            mbar_init(&c.bar.it_full[s], 1);
            mbar_init(&c.bar.it_empty[s], C::kItemConsumerWarps);
        }
        mbar_init(c.bar.never, 1);
        *c.abort_flag = 0;
        fence_mbar_init();
    }
    if (threadIdx.x == 32) {
        prefetch_tmap(&p.tm_q);
        prefetch_tmap(&p.tm_k);
        prefetch_tmap(&p.tm_v);
        if (p.out_tma)
            prefetch_tmap(&p.tm_o);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, C::kTmemCols);
        tmem_relinquish();
    }
    {
        // Q rows past G * rows_per_tile are never written by TMA: keep them zero
        const int used = p.G * p.rows_per_tile * 128;
        const int pad = C::kQTileBytes - used;
        if (pad > 0) {
            const int n16 = pad / 16;
            for (int k = threadIdx.x; k < C::kQBufs * kQTiles * n16; k += blockDim.x) {
                const int blk = k / n16, q = k % n16;
                *reinterpret_cast<uint4*>(base + C::kOffQ + blk * C::kQTileBytes + used + q * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    c.tmem = *tmem_holder;

    // inputs may come from the kernel this launch follows (and the work
    // distribution words from the previous launch)
    pdl_wait();
    {
        // every CTA sorts the work itself (in the K/V ring and the output
        // staging, before any copy lands there); the first to win the claim
        // also writes the list
        int claim = 1;
        if (threadIdx.x == 0)
            claim = atomicCAS(p.claim, 0, 1);
        const WorklistResult wl =
            build_worklist<C::kThreads / 32>(p.sched, reinterpret_cast<int*>(base + C::kOffRing), blockIdx.x, claim);
        if (wl.emit && threadIdx.x == 0) {
            __threadfence();
            st_release_gpu(p.ready, 1);
        }
        c.n_items = wl.n_items;
        if (threadIdx.x == 0)
            *reinterpret_cast<int4*>(base + C::kOffFirst) = wl.want;
        fence_proxy_async_smem();
        __syncthreads();
    }

    // 384 threads launch with 168 registers each (104 + 200 + 200 = 504 = 3 x 168)
    if (warp < 4) {
        regs_dec<104>();
        if (warp == 0)
            win_producer(p, c);
        else if (warp == 1)
            win_mma(p, c);
    } else {
        regs_inc<200>();
        win_softmax(p, c, (warp - 4) >> 2);
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) {
        // the last CTA out leaves the work-distribution words at zero
        __threadfence();
        if (atomicAdd(p.done, 1) == (int)gridDim.x - 1) {
            *p.counter = 0;
            *p.claim = 0;
            *p.ready = 0;
            *p.done = 0;
        }
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(c.tmem, C::kTmemCols);
    }
}

int win_max_keys() { return WinCfg::kWinKeys; }

cudaError_t launch_attention_win(const AttnParams& p, int grid, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    static std::once_flag attr_once[64];
    static cudaError_t attr_err[64];
    std::call_once(attr_once[dev], [&] {
        attr_err[dev] = cudaFuncSetAttribute(attention_win_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             WinCfg::kSmemBytes);
    });
    if (attr_err[dev] != cudaSuccess)
        return attr_err[dev];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(WinCfg::kThreads);
    cfg.dynamicSmemBytes = WinCfg::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attention_win_kernel, p);
}

}  // namespace b2pa
