// attn_common.cuh -- the pieces both tensor-core attention kernels (attn_tc.cu
// and attn_win.cu) share: the barrier set and per-CTA context, bounded
// mbarrier waits, and the item records the producer posts for the other roles.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace b2pa {

constexpr int kItemRecWords = 12;  // a posted item: w, b, kvh, q0, q_len, kv_len, tok0, nq, n_lo, n_hi, chunk, chunks

struct Bars {
    uint64_t* full;      // [kPairs]   16-bit K of a kv tile landed (merged release: K and V)
    uint64_t* empty;     // [kPairs]   K of the tile consumed, its last Q K^T done (merged: K and V, last P V)
    uint64_t* vfull;     // [kPairs]   16-bit V of the tile landed (split release and FP8)
    uint64_t* vempty;    // [kPairs]   V of the tile consumed, its last P V done (split release)
    uint64_t* f8full;    // [kF8Stages]
    uint64_t* f8empty;   // [kF8Stages]
    uint64_t* q_full;    // [kQBufs]   Q tiles landed
    uint64_t* q_empty;   // [kQBufs]   last Q K^T of the item done
    uint64_t* q_conv;    // [kQBufs]   (FP8) Q rows scaled and converted to f16, their exponents posted
    uint64_t* s_full;    // [2]        S_t in TMEM
    uint64_t* p_full;    // [2][kPParts] part h of P_t in TMEM (4 softmax warps)
    uint64_t* o_full;    // [2]        last P V of the item done
    uint64_t* drain;
    uint64_t* it_full;   // [kItemSlots] item index posted
    uint64_t* it_empty;  // [kItemSlots] item index read by every consumer warp
    uint64_t* never;     // [1]        nothing arrives: the injected stall of failure-detection tests
};

struct Ctx {
    uint8_t* base;
    Bars bar;
    uint32_t tmem;
    int n_items;
    volatile int* item_slot;
    volatile int* abort_flag;
    unsigned* err;
    unsigned long long wait_limit_ns;  // a pipeline wait longer than this gives up
};

// Bounded wait on a barrier phase; false if this CTA gave up (another role
// raised the abort flag, or c.wait_limit_ns of %globaltimer passed: then this
// wait raises it and sets B2PA_DEV_TIMEOUT).
// Every caller is a whole warp.  The lanes of a converged warp see the same
// barrier state, so they leave a satisfied wait together; giving up is decided
// as a warp (a vote, taken only between unsuccessful tries), so that a lane
// reading the timer a cycle later cannot split the warp before
// warp-collective instructions (tcgen05.ld.sync.aligned, __syncwarp).
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const Ctx& c)
{
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity))
        return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try_wait(a, parity))
            return true;
        const bool timed_out = global_ns() - t0 > c.wait_limit_ns;
        if (__any_sync(0xffffffffu, *c.abort_flag != 0 || timed_out)) {
            if (timed_out && (threadIdx.x & 31) == 0) {
                *c.abort_flag = 1;
                atomicOr(c.err, (unsigned)B2PA_DEV_TIMEOUT);
            }
            __syncwarp();
            return false;
        }
    }
}

// Wait without looking at the abort flag (used when draining after an abort).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity)
{
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(a, parity)) {
        if (global_ns() - t0 > kWaitLimitNs)
            return;
    }
}

// Wait (lane 0 of the producer alone) until the work list that another CTA
// of this launch writes is complete; false if this CTA gave up (abort flag,
// or the wait limit ran out: then it raises both).
__device__ __forceinline__ bool wait_list_ready(const int* ready, const Ctx& c)
{
    if (ld_acquire_gpu(ready) != 0)
        return true;
    const uint64_t t0 = global_ns();
    while (ld_acquire_gpu(ready) == 0) {
        if (*c.abort_flag != 0)
            return false;
        if (global_ns() - t0 > c.wait_limit_ns) {
            *c.abort_flag = 1;
            atomicOr(c.err, (unsigned)B2PA_DEV_TIMEOUT);
            return false;
        }
        __nanosleep(128);
    }
    return true;
}

struct ItemInfo {
    int b, kvh, q0, q_len, kv_len;
    ItemGeom g;
    int chunk, chunks;  // split-KV: this item's kv chunk and the request's chunk count (else 0, 1)
};

template <bool SPLIT>
__device__ __forceinline__ ItemInfo read_item(const AttnParams& p, const int4 it)
{
    ItemInfo r;
    r.b = it.x;
    r.kvh = it.y;
    const QStarts cq{p.cum_q, p.q_per_req};
    r.q0 = cq[r.b];
    r.q_len = cq[r.b + 1] - r.q0;
    r.kv_len = p.seq_lens[r.b];
    r.chunk = 0;
    r.chunks = 1;
    if (SPLIT) {
        r.g = item_geometry(r.q_len, r.kv_len, 0, p.rows_per_tile, p.window);
        r.chunk = it.z;
        r.chunks = split_count(r.g, p.split_tiles);
        split_range(&r.g, it.z, p.split_tiles);
    } else {
        r.g = item_geometry(r.q_len, r.kv_len, it.z, p.rows_per_tile, p.window);
    }
    return r;
}

// The n-th item of this CTA (index -1: no more work) and its description, as
// posted by the producer in shared memory (no global reads in the consumers).
template <int kSlots>
__device__ __forceinline__ int take_item(const AttnParams& p, const Ctx& c, uint32_t n, bool* ok, ItemInfo* it)
{
    const uint32_t s = n % kSlots;
    if (!wait_bar(&c.bar.it_full[s], (n / kSlots) & 1, c)) {
        *ok = false;
        return -1;
    }
    const volatile int* rec = c.item_slot + s * kItemRecWords;
    const int w = rec[0];
    it->b = rec[1];
    it->kvh = rec[2];
    it->q0 = rec[3];
    it->q_len = rec[4];
    it->kv_len = rec[5];
    it->g.tok0 = rec[6];
    it->g.nq = rec[7];
    it->g.n_lo = rec[8];
    it->g.n_hi = rec[9];
    it->chunk = rec[10];
    it->chunks = rec[11];
    __syncwarp();
    if ((threadIdx.x & 31) == 0)
        mbar_arrive(&c.bar.it_empty[s]);
    return w;
}

}  // namespace b2pa
