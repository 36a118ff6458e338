// attn_tc.cu -- persistent, warp-specialised paged-KV context attention on
// the 5th-generation tensor cores (tcgen05) of sm_103a.
//
// What it computes is fixed by flashinfer.prefill.trtllm_batch_context_with_kv_cache
// (FlashInfer API reference, parameter list) with the end-aligned causal
// rule of the TokenSpeed trtllm backend (_init_extend_metadata); see the
// header of include/b2pa.h.  The design below is ours.
//
// One CTA per SM.  Work items come from the scheduler's longest-first list;
// the producer warp takes the next one with an atomic counter and hands its
// index to the other roles through a small shared-memory ring.  A work item
// is (request b, kv head, item index): two query tiles of 128 MMA rows, a row
// being one (token, query head) pair of the kv head's group (rows_per_tile
// tokens x G heads).  Both query tiles stream the same K/V tiles of 128 keys.
//
//   warp 0        producer: item fetch; TMA loads of Q (3-D map, double
//                 buffered across items where shared memory allows) and of
//                 K/V pages (4-D map, one box per page and 128-byte column
//                 block) through a ring that holds K and V of a kv tile side
//                 by side.  At head_dim 128 (16-bit KV), whose ring holds only
//                 two tiles, K and V land and are released separately: a K
//                 entry is free once the tile's last Q K^T has completed, one
//                 softmax earlier than its V, so the next K is fetched that
//                 much sooner.  Elsewhere a tile's K and V are released
//                 together after its last P V (one barrier less per tile;
//                 measured faster there).
//   warp 1        MMA issuer (one lane): S_t = Q_t K^T into TMEM, then
//                 O_t += P_t V with P_t read from TMEM, for t = 0, 1, in the
//                 order PV_0(j), S_0(j+1), PV_1(j), S_1(j+1) so the tensor
//                 core works on one tile while the other tile's softmax runs.
//                 Owns the TMEM allocation.
//   warps 4-7     softmax of query tile 0 (one thread per row), O rescale,
//                 and the epilogue (bmm2_scale / denominator, bf16 stores).
//   warps 8-11    the same for query tile 1.
//   warps 12-15   (FP8 KV only) convert e4m3 K/V tiles to f16 in the MMA
//                 layout (exact), and each Q row from bf16 to f16 after
//                 scaling it by a power of two into f16's range (exact); the
//                 softmax divides that power of two out of the row's scale.
//
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [256+D,256+2D).
// P_t (16-bit, two per column) overwrites the first 64 columns of S_t and is
// handed to the MMA warp in kPParts parts (one: each extra hand-off costs the
// MMA warp more than the overlap gains).
//
// The row maximum of an S tile comes with its TMEM load (tcgen05.ld.red, an
// sm_103a instruction) except on tiles that need masking.
//
// Every wait is bounded: after the call's wait limit (2 s of %globaltimer unless
// b2pa_set_wait_limit_ns changed it) the CTA raises B2PA_DEV_TIMEOUT, every
// role leaves its loop, in-flight TMA loads (K/V and Q), TMA stores and MMAs
// are drained (those drains keep the 2 s limit), and TMEM is freed before the
// CTA exits.
#include <mutex>

#include "attn_common.cuh"
#include "common.cuh"
#include "ptx.cuh"
#include "worklist.cuh"

namespace b2pa {


// SPLIT: the variant for split-KV work lists (decode batches), whose items are
// kv chunks and whose split rows end in partial outputs
template <int D, bool FP8, bool SPLIT>
struct TcCfg {
    static constexpr int kHalves = D / 64;            // 128-byte column blocks per 16-bit row
    static constexpr int kHalfBytes = kQRows * 128;   // one column block of a 128-row tile
    static constexpr int kQTileBytes = kHalves * kHalfBytes;
    static constexpr int kKvTileBytes = kHalves * kHalfBytes;
    // The 16-bit K/V ring holds K and V of a kv tile side by side (entries 2m
    // and 2m + 1) under one full and one empty barrier: a tile is in use from
    // S(j) to P V(j), and the next tile lands meanwhile.
    static constexpr int kQBufs = D == 128 ? 1 : 2;                 // Q buffers (items in flight)
    static constexpr int kStages = D == 128 ? 4 : 8;                // 16-bit ring entries
    static constexpr int kPairs = kStages / 2;                      // tiles in the ring
    static constexpr bool kSplitKV = D == 128 && !FP8;              // K and V released separately
    // Query tiles held per Q buffer.  A split-KV (decode) batch on the e4m3 path
    // runs with one query tile per item (the host splits only such batches), and
    // the room goes to a deeper e4m3 staging ring: there the K/V stream, not the
    // tensor core, sets the rate, and two tiles in flight hide more of HBM's latency.
    static constexpr int kQTilesAlloc = FP8 && SPLIT ? 1 : kQTiles;
    static constexpr int kF8Stages = FP8 ? (SPLIT ? 4 : 2) : 0;     // e4m3 staging ring
    static constexpr int kF8TileBytes = kKvTile * D;  // e4m3 tile: 128 rows of D bytes
    static constexpr int kThreads = FP8 ? 512 : 384;
    static constexpr int kItemSlots = 4;
    static constexpr int kItemConsumerWarps = 1 + 8 + (FP8 ? 4 : 0);
    static constexpr int kTmemCols = 512;
    static constexpr int kOCol = 2 * kKvTile;
    static constexpr int kOffQ = 0;
    static constexpr int kOffRing = kOffQ + kQBufs * kQTilesAlloc * kQTileBytes;
    static constexpr int kOffF8 = kOffRing + kStages * kKvTileBytes;
    // output staging (16-bit KV paths; the e4m3 path has no room): per softmax
    // warp, 32 rows x 64 columns of bf16, so that the output leaves in whole
    // 128-byte lines instead of one 16-byte piece per row and instruction
    static constexpr bool kStageOut = !FP8;
    static constexpr int kStageWarpBytes = 32 * 128;
    static constexpr int kOffStage = kOffF8 + kF8Stages * kF8TileBytes;
    static constexpr int kOffBar = kOffStage + (kStageOut ? 8 * kStageWarpBytes : 0);
    // P_t is handed to the MMA warp in kPParts parts of kKvTile / kPParts keys
    static constexpr int kPParts = 1;
    static constexpr int kNumBars = 4 * kPairs + 2 * kF8Stages + 3 * kQBufs + (2 + kPParts) * kQTiles + 1 + 2 * kItemSlots + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    // FP8: the power-of-two exponent of each Q row (int8), for the items of
    // both parities (a row's exponent is read by the softmax while the next
    // item's Q is being converted)
    static constexpr int kOffQExp = kOffMisc + 64 + kItemSlots * kItemRecWords * 4;
    // this CTA's first item (int4; x = -1: none), from its own copy of the work list
    static constexpr int kOffFirst = (kOffMisc + 16 + kItemSlots * kItemRecWords * 4 + 15) / 16 * 16;
    static_assert(kOffFirst % 16 == 0 && kOffFirst + 16 <= kOffQExp, "misc layout");
    static constexpr int kQExpBytes = FP8 ? 2 * kQTiles * kQRows : 0;
    static constexpr int kSmemBytes = kOffQExp + kQExpBytes + 1024;  // + slack to align the base to 1024
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(!FP8 || D == 128, "fp8 path is D = 128");
    static_assert(kOCol + kQTiles * D <= kTmemCols, "tmem");
    static_assert(kSmemBytes <= 232448, "shared memory");
    // the work list is sorted in the K/V ring at the kernel's start
    static_assert(worklist_smem_ints(kThreads / 32, kSchedBuckets, kSchedMaxBatch) * sizeof(int) <=
                      (size_t)kStages * kKvTileBytes,
                  "work-list scratch");
};

// ---------------------------------------------------------------------------
// Producer: warp 0.  Lane 0 takes items; lane l loads page l of a kv tile (one
// TMA box per 128-byte column block) after lane 0 posted the byte count.
// ---------------------------------------------------------------------------
template <int D, bool FP8, bool SPLIT>
__device__ void producer_role(const AttnParams& p, const Ctx& c)
{
    using C = TcCfg<D, FP8, SPLIT>;
    constexpr int kRingStages = FP8 ? C::kF8Stages : C::kStages;
    constexpr int kRingTileBytes = FP8 ? C::kF8TileBytes : C::kKvTileBytes;
    constexpr int kBoxes = FP8 ? 1 : C::kHalves;  // 128-byte-wide boxes per page
    uint64_t* rfull = FP8 ? c.bar.f8full : c.bar.full;
    uint64_t* rempty = FP8 ? c.bar.f8empty : c.bar.empty;
    const int lane = threadIdx.x & 31;
    const uint32_t q_smem = smem_u32(c.base + C::kOffQ);
    const uint32_t ring = smem_u32(c.base + (FP8 ? C::kOffF8 : C::kOffRing));
    const int P = p.page_size;
    const int log2_p = 31 - __clz(P);                 // the tensor-core path takes powers of two only
    const int box_rows = P >= kKvTile ? kKvTile : P;
    const uint32_t q_box_bytes = (uint32_t)(p.G * p.rows_per_tile * 128);

    uint32_t ring_idx = 0;
    uint32_t ring_kv[2] = {0, 0};  // 16-bit path: K and V tiles whose copies were started
    uint32_t q_loads = 0;          // items whose Q copies were started
    bool list_ready = false;       // lane 0: the shared work list was seen complete
    bool ok = true;
    // scales passed as device tensors are checked here: if they are unusable,
    // no item is taken, so every role finishes without writing anything
    const bool scales_ok = load_scales(p.scale_log2, p.bmm2, p.bmm1_dev, p.bmm2_dev).ok;
    if (!scales_ok && blockIdx.x == 0 && lane == 0)
        atomicOr(p.err, (unsigned)B2PA_DEV_BAD_SCALE);
    for (uint32_t n = 0; ok; ++n) {
        // post the next item index
        const uint32_t slot = n % C::kItemSlots;
        if (!wait_bar(&c.bar.it_empty[slot], ((n / C::kItemSlots) & 1) ^ 1, c))
            break;
        volatile int* rec = c.item_slot + slot * kItemRecWords;
        if (lane == 0) {
            // the first item from this CTA's own copy of the list, later ones in
            // list order from gridDim.x on, once the shared list is written
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
                const ItemInfo r = read_item<SPLIT>(p, item);
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
        it.g.n_lo = rec[8];
        it.g.n_hi = rec[9];
        it.chunk = rec[10];
        it.chunks = rec[11];
        // Q tiles, into the buffer of this item once its previous user is done
        const uint32_t qb = n % C::kQBufs, qph = (n / C::kQBufs) & 1;
        if (!wait_bar(&c.bar.q_empty[qb], qph ^ 1, c))
            break;
        if (lane == 0)
            mbar_arrive_expect_tx(&c.bar.q_full[qb], (uint32_t)(it.g.nq * C::kHalves) * q_box_bytes);
        __syncwarp();
        if (lane < it.g.nq * C::kHalves) {
            const int t = lane / C::kHalves, h = lane % C::kHalves;
            tma_load_3d(q_smem + (qb * C::kQTilesAlloc + t) * C::kQTileBytes + h * C::kHalfBytes, &p.tm_q, &c.bar.q_full[qb],
                        h * 64, it.kvh * p.G, it.q0 + it.g.tok0 + t * p.rows_per_tile);
        }
        q_loads = n + 1;
        const int* bt_row = page_row(p.block_tables, p.bt_stride, p.kv_indptr, it.b);
        const int n_pages_valid = (it.kv_len + P - 1) >> log2_p;
        for (int j = it.g.n_lo; ok && j <= it.g.n_hi; ++j) {
            const TileLoad tl = tile_load(bt_row, j, lane, log2_p, n_pages_valid);
            const int slot0 = tl.slot0, page = tl.page;
            const bool valid = tl.valid;
            if (valid && (page < 0 || page >= p.num_pages))
                atomicOr(p.err, (unsigned)B2PA_DEV_BAD_PAGE);
            const uint32_t nvalid = __popc(__ballot_sync(0xffffffffu, valid));
            const uint32_t bytes = nvalid * (uint32_t)box_rows * 128u * kBoxes;
            if constexpr (!FP8) {
                // K into ring entry 2m, V into 2m + 1: with the split release each
                // once its previous K (or V) is consumed, under its own barrier;
                // otherwise both once the pair is free, under one barrier
                const uint32_t m = ring_idx % C::kPairs, ph = (ring_idx / C::kPairs) & 1;
#pragma unroll
                for (int kind = 0; kind < 2; ++kind) {
                    const bool own = C::kSplitKV || kind == 0;  // this kind waits and posts its bytes
                    uint64_t* fb = (C::kSplitKV && kind) ? &c.bar.vfull[m] : &c.bar.full[m];
                    if (own && !wait_bar((C::kSplitKV && kind) ? &c.bar.vempty[m] : &c.bar.empty[m], ph ^ 1, c)) {
                        ok = false;
                        break;
                    }
                    // predicated rather than branched: the warp stays converged
                    if (own)
                        mbar_arrive_expect_tx_p(fb, C::kSplitKV ? bytes : 2 * bytes, lane == 0 ? 1u : 0u);
                    __syncwarp();
                    const uint32_t dst = ring + (2 * m + kind) * kRingTileBytes + (uint32_t)(lane * box_rows * 128);
#pragma unroll
                    for (int h = 0; h < kBoxes; ++h)
                        tma_load_4d_p(dst + h * C::kHalfBytes, kind ? &p.tm_v : &p.tm_k, fb, h * 64, slot0, it.kvh,
                                      page, valid ? 1u : 0u);
                    ++ring_kv[kind];
                }
                if (!ok)
                    break;
                ++ring_idx;
            } else {
                for (int kind = 0; kind < 2; ++kind) {
                    const uint32_t s = ring_idx % kRingStages, ph = (ring_idx / kRingStages) & 1;
                    if (!wait_bar(&rempty[s], ph ^ 1, c)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0)
                        mbar_arrive_expect_tx(&rfull[s], bytes);
                    __syncwarp();
                    if (valid) {
                        const uint32_t dst = ring + s * kRingTileBytes + (uint32_t)(lane * box_rows * 128);
#pragma unroll
                        for (int h = 0; h < kBoxes; ++h)
                            tma_load_4d(dst + h * C::kHalfBytes, kind ? &p.tm_v : &p.tm_k, &rfull[s], h * 64, slot0,
                                        it.kvh, page);
                    }
                    ++ring_idx;
                }
            }
        }
    }
    if (*c.abort_flag) {
        // let the copies this warp started land before the CTA releases its
        // memory: the Q tiles of the last items (one buffer each), then K/V
        const uint32_t q_first = q_loads > (uint32_t)C::kQBufs ? q_loads - C::kQBufs : 0;
        for (uint32_t k = q_first; k < q_loads; ++k)
            drain_wait(&c.bar.q_full[k % C::kQBufs], (k / C::kQBufs) & 1);
        if constexpr (FP8) {
            const uint32_t first = ring_idx > (uint32_t)kRingStages ? ring_idx - kRingStages : 0;
            for (uint32_t k = first; k < ring_idx; ++k)
                drain_wait(&rfull[k % kRingStages], (k / kRingStages) & 1);
        } else {
            for (int kind = 0; kind < 2; ++kind) {
                uint64_t* fb = (C::kSplitKV && kind) ? c.bar.vfull : c.bar.full;
                const uint32_t n_kv = C::kSplitKV || kind == 0 ? ring_kv[kind] : 0;
                const uint32_t first = n_kv > (uint32_t)C::kPairs ? n_kv - C::kPairs : 0;
                for (uint32_t k = first; k < n_kv; ++k)
                    drain_wait(&fb[k % C::kPairs], (k / C::kPairs) & 1);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// MMA issuer: warp 1.  The whole warp waits and runs the issue code; the
// MMAs and commits are predicated on lane 0, so the warp never diverges.
// ---------------------------------------------------------------------------
template <int D, bool FP8, bool SPLIT>
__device__ void mma_role(const AttnParams& p, const Ctx& c)
{
    using C = TcCfg<D, FP8, SPLIT>;
    // kind::f16; bf16 operands (f16 on the e4m3 path), f32 accumulators
    constexpr uint32_t kFmt = FP8 ? 0u : 1u;
    constexpr uint32_t kIdescS = (1u << 4) | (kFmt << 7) | (kFmt << 10) | ((uint32_t)(kKvTile >> 3) << 17) |
                                 ((uint32_t)(kQRows >> 4) << 24);
    constexpr uint32_t kIdescO = (1u << 4) | (kFmt << 7) | (kFmt << 10) | (1u << 16) | ((uint32_t)(D >> 3) << 17) |
                                 ((uint32_t)(kQRows >> 4) << 24);
    const int lane = threadIdx.x & 31;
    const bool leader = lane == 0;
    const uint32_t issue = leader ? 1u : 0u;  // lane 0 issues; the warp stays converged
    const uint32_t q_smem = smem_u32(c.base + C::kOffQ);
    const uint32_t ring = smem_u32(c.base + C::kOffRing);
    uint64_t* const full = c.bar.full;
    uint64_t* const empty = c.bar.empty;

    // descriptor words: only the low word (start address) moves between MMAs
    constexpr uint32_t kHi = sdesc_hi_sw128(1024);                 // 8 rows x 128 B per core group
    const uint32_t q_lo = sdesc_lo(q_smem, 16);                    // K-major: LBO unused
    const uint32_t k_lo = sdesc_lo(ring, 16);
    const uint32_t v_lo = sdesc_lo(ring, C::kHalfBytes);           // MN-major: LBO = next 64 columns of d
    constexpr uint32_t kStageW = C::kKvTileBytes >> 4;             // descriptor units per ring stage
    constexpr uint32_t kQTileW = C::kQTileBytes >> 4;
    constexpr uint32_t kHalfW = C::kHalfBytes >> 4;

    auto issue_s = [&](uint32_t qb, int t, uint32_t slot) {
        const uint32_t a0 = q_lo + (qb * C::kQTilesAlloc + t) * kQTileW;
        const uint32_t b0 = k_lo + slot * kStageW;
        const uint32_t d = c.tmem + (uint32_t)(t * kKvTile);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (uint32_t)((k / 4) * kHalfW + (k % 4) * 2);  // 16 elements = 32 B
            mma_ss_wp(d, a0 + off, b0 + off, kHi, kIdescS, k > 0 ? 1u : 0u, issue);
        }
    };
    // P V over the keys of part `part` of the tile
    auto issue_pv = [&](int t, int part, uint32_t slot, bool acc) {
        constexpr int kSteps = kKvTile / 16 / C::kPParts;
        const uint32_t b0 = v_lo + slot * kStageW;
        const uint32_t d = c.tmem + (uint32_t)(C::kOCol + t * D);
        const uint32_t a = c.tmem + (uint32_t)(t * kKvTile);
#pragma unroll
        for (int kk = 0; kk < kSteps; ++kk) {
            const int k = part * kSteps + kk;                          // 16 keys = 16 rows of 128 B
            mma_ts_wp(d, a + (uint32_t)(k * 8), b0 + (uint32_t)(k * 128), kHi, kIdescO, (acc || k > 0) ? 1u : 0u,
                      issue);
        }
    };
    // ring pair r % kPairs holds K (entry 2m) and V (entry 2m + 1) of the r-th tile
    auto wait_full = [&](uint32_t r) -> bool {
        return wait_bar(&full[r % C::kPairs], (r / C::kPairs) & 1, c);
    };
    auto k_slot = [](uint32_t r) { return 2u * (r % C::kPairs); };
    auto v_slot = [](uint32_t r) { return 2u * (r % C::kPairs) + 1u; };

    uint32_t ring_idx = 0;
    uint32_t p_cnt[kQTiles] = {0, 0};
    bool ok = true;

    // An open item: its Q landed and its first kv tile (ring entry `first`) too.
    struct Open {
        int n_lo, n_hi, nq, kv_len;
        uint32_t qb, first;
        bool ok;
    };
    auto open_item = [&](const ItemInfo& it, uint32_t n) -> Open {
        Open o;
        o.n_lo = it.g.n_lo;
        o.n_hi = it.g.n_hi;
        o.nq = it.g.nq;
        o.kv_len = it.kv_len;
        o.qb = n % C::kQBufs;
        // TMA (and converter) writes reach the MMA through the mbarrier alone:
        // no tcgen05 fence is needed after these waits
        o.ok = wait_bar(FP8 ? &c.bar.q_conv[o.qb] : &c.bar.q_full[o.qb], (n / C::kQBufs) & 1, c);
        o.first = ring_idx++;
        o.ok = o.ok && wait_full(o.first);
        return o;
    };
    // S_t of an open item's first kv tile
    auto first_s = [&](const Open o, int t) {
        issue_s(o.qb, t, k_slot(o.first));
        mma_commit_p(&c.bar.s_full[t], issue);
        if (t == o.nq - 1) {
            if (C::kSplitKV)
                mma_commit_p(&empty[o.first % C::kPairs], issue);  // K of the tile consumed
            if (o.n_lo == o.n_hi)
                mma_commit_p(&c.bar.q_empty[o.qb], issue);
        }
    };

    // The next item is opened while the current one's last kv tile finishes:
    // its S_0 right after the last P_0 V, its S_1 after the last P_1 V, the
    // same order as between two kv tiles of one item.
    // failure-detection tests: a wait on a barrier nothing arrives on, which runs
    // the wait limit out and sends the whole CTA down its abort path
    if (p.inject_stall && !wait_bar(c.bar.never, 0, c))
        ok = false;
    Open cur_item;
    ItemInfo info;
    int w = ok ? take_item<C::kItemSlots>(p, c, 0, &ok, &info) : -1;
    if (w >= 0) {
        cur_item = open_item(info, 0);
        ok = cur_item.ok;
        for (int t = 0; ok && t < cur_item.nq; ++t)
            first_s(cur_item, t);
    }
    for (uint32_t n = 0; ok && w >= 0; ++n) {
        const int n_lo = cur_item.n_lo, n_hi = cur_item.n_hi, kv_len = cur_item.kv_len;
        const int nq = cur_item.nq;
        const uint32_t qb = cur_item.qb;
        uint32_t cur = cur_item.first;
        Open nxt;
        int w_next = -1;
        for (int j = n_lo; ok && j <= n_hi; ++j) {
            const bool last = j == n_hi;
            const uint32_t next = last ? 0u : ring_idx++;
            if ((FP8 || C::kSplitKV) &&
                !wait_bar(&c.bar.vfull[cur % C::kPairs], (cur / C::kPairs) & 1, c)) {
                ok = false;
                break;
            }
            if (!FP8) {
                // keys >= kv_len: V rows may hold any bits (or a page that was not
                // loaded); zero them so that P = 0 there cannot meet a NaN.
                const int r0 = kv_len - j * kKvTile;
                if (r0 < kKvTile) {
                    uint8_t* vt = c.base + C::kOffRing + v_slot(cur) * C::kKvTileBytes;
                    const int n16 = (kKvTile - r0) * 8;  // 16-byte chunks per column block
                    for (int h = 0; h < C::kHalves; ++h) {
                        uint4* dst = reinterpret_cast<uint4*>(vt + h * C::kHalfBytes + r0 * 128);
                        for (int q = lane; q < n16; q += 32)
                            dst[q] = make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
            }
            // unrolled over the two query tiles, so p_cnt[t] stays in registers
#pragma unroll
            for (int t = 0; t < kQTiles; ++t) {
                if (!ok || t >= nq)
                    break;
                for (int part = 0; part < C::kPParts; ++part) {
                    if (!wait_bar(&c.bar.p_full[C::kPParts * t + part], p_cnt[t] & 1, c)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_pv(t, part, v_slot(cur), j > n_lo);
                }
                if (!ok)
                    break;
                ++p_cnt[t];
                if (t == nq - 1)  // V of tile j consumed (merged release: K and V)
                    mma_commit_p(C::kSplitKV ? &c.bar.vempty[cur % C::kPairs] : &empty[cur % C::kPairs], issue);
                if (last)
                    mma_commit_p(&c.bar.o_full[t], issue);
                if (!last) {
                    if (t == 0) {
                        if (!wait_full(next)) {
                            ok = false;
                            break;
                        }
                    }
                    issue_s(qb, t, k_slot(next));
                    mma_commit_p(&c.bar.s_full[t], issue);
                    if (t == nq - 1) {
                        if (C::kSplitKV)
                            mma_commit_p(&empty[next % C::kPairs], issue);  // K of tile j + 1 consumed
                        if (j + 1 == n_hi)
                            mma_commit_p(&c.bar.q_empty[qb], issue);
                    }
                } else if (t == (D == 128 ? nq - 1 : 0)) {
                    // D = 128 (and FP8): after the item's last P V of both tiles, so
                    // neither tile's epilogue waits behind the next item's start
                    // (measured faster there); D = 64: right after the last P_0 V
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
                        if ((D == 128 || nq == 1) && nxt.nq > 1)
                            first_s(nxt, 1);  // no P_1 V left to wait for in this item
                    }
                } else if (D != 128 && w_next >= 0 && nxt.nq > 1) {
                    first_s(nxt, 1);
                }
            }
            cur = next;
        }
        if (!ok)
            break;
        w = w_next;
        cur_item = nxt;
    }
    // every MMA this thread issued has completed once the drain barrier flips
    if (leader)
        mma_commit(c.bar.drain);
    __syncwarp();
    drain_wait(c.bar.drain, 0);
}

// ---------------------------------------------------------------------------
// Softmax / correction / epilogue for query tile t: warps 4+4t .. 7+4t, one
// thread per TMEM lane (= MMA row).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

template <int D, bool FP8, bool SPLIT>
__device__ void softmax_role(const AttnParams& p, const Ctx& c, int t)
{
    using C = TcCfg<D, FP8, SPLIT>;
    constexpr float kLog2e = 1.4426950408889634f;
    const int wq = (threadIdx.x >> 5) & 3;
    const int lane = threadIdx.x & 31;
    const int row = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t s_tmem = c.tmem + lane_off + (uint32_t)(t * kKvTile);
    const uint32_t o_tmem = c.tmem + lane_off + (uint32_t)(C::kOCol + t * D);
    const int G = p.G, Tq = p.rows_per_tile;
    const int r_tok = row / G, r_head = row % G;
    const bool row_real = row < G * Tq;
    const Scales scl = load_scales(p.scale_log2, p.bmm2, p.bmm1_dev, p.bmm2_dev);

    uint32_t s_cnt = 0, o_cnt = 0;
    bool ok = true;
    for (uint32_t n = 0; ok; ++n) {
        ItemInfo it;
        const int w = take_item<C::kItemSlots>(p, c, n, &ok, &it);
        if (w < 0)
            break;
        // FP8: every item's Q conversion is awaited (also by a warpgroup with no
        // query tile in it: a waiter that skipped phases could mistake a later
        // one for an earlier one); the row's Q was scaled by 2^k before its
        // conversion to f16, so its scores carry 2^k, taken out here
        if (FP8 && !wait_bar(&c.bar.q_conv[n % C::kQBufs], (n / C::kQBufs) & 1, c)) {
            ok = false;
            break;
        }
        if (t >= it.g.nq)
            continue;
        float sl2 = scl.scale_log2;
        if constexpr (FP8) {
            const int k = reinterpret_cast<const int8_t*>(c.base + C::kOffQExp)[(n & 1) * kQTiles * kQRows + t * kQRows + row];
            sl2 *= __int_as_float((127 - k) << 23);
        }
        const int prefix = it.kv_len - it.q_len;
        const int i_first = it.g.tok0 + t * Tq;
        const int i = i_first + r_tok;
        const bool valid = row_real && i < it.q_len;
        const int pos = prefix + i;
        const int lo = p.window < 0 ? 0 : max(0, pos - p.window);
        const int hi = valid ? pos : -1;
        const int i_last = min(i_first + Tq, it.q_len) - 1;
        const int p_first = prefix + i_first, p_last = prefix + i_last;
        const int lo_last = p.window < 0 ? 0 : max(0, p_last - p.window);

        float m_used = -INFINITY;
        float l = 0.f;
        for (int j = it.g.n_lo; j <= it.g.n_hi; ++j) {
            if (!wait_bar(&c.bar.s_full[t], s_cnt & 1, c)) {
                ok = false;
                break;
            }
            ++s_cnt;
            tc_fence_after();
            float s[kKvTile];
            float mq[4];  // maxima of the four 32-key loads
            {
                uint32_t r[32];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    tmem_ld32_max(s_tmem + (uint32_t)(q * 32), r, &mq[q]);
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        s[q * 32 + k] = __uint_as_float(r[k]);
                }
                tmem_wait_ld();
            }
            const int k0 = j * kKvTile;
            const bool interior = k0 >= lo_last && k0 + kKvTile - 1 <= p_first;
            float mx;
            if (interior) {
                mx = fmax3(fmax3(mq[0], mq[1], mq[2]), mq[3], -INFINITY);
            } else if constexpr (D == 64 && !SPLIT) {
                // head_dim 64 (measured faster there): every key masked against the
                // row's own range, without branches, then one maximum over the tile
#pragma unroll
                for (int k = 0; k < kKvTile; ++k) {
                    const int key = k0 + k;
                    if (key < lo || key > hi)
                        s[k] = -INFINITY;
                }
                float m0 = fmax3(s[0], s[1], s[2]), m1 = fmax3(s[3], s[4], s[5]);
                float m2 = fmax3(s[6], s[7], s[8]), m3 = fmax3(s[9], s[10], s[11]);
#pragma unroll
                for (int k = 12; k < 120; k += 8) {
                    m0 = fmax3(m0, s[k], s[k + 1]);
                    m1 = fmax3(m1, s[k + 2], s[k + 3]);
                    m2 = fmax3(m2, s[k + 4], s[k + 5]);
                    m3 = fmax3(m3, s[k + 6], s[k + 7]);
                }
                m0 = fmax3(m0, s[120], s[121]);
                m1 = fmax3(m1, s[122], s[123]);
                m2 = fmax3(m2, s[124], s[125]);
                m3 = fmax3(m3, s[126], s[127]);
                mx = fmax3(fmaxf(m0, m1), m2, m3);
            } else {
                // per 32-key chunk, decided for the whole warp: every row sees all of
                // it (its ld.red maximum stands), no row sees any of it (maximum
                // -inf; the exponential loop below skips it on the same test, so
                // its scores are never read), or mask element by element
                float cm[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int c0 = k0 + 32 * q;
                    if (__all_sync(0xffffffffu, c0 >= lo && c0 + 31 <= hi)) {
                        cm[q] = mq[q];
                    } else if (__all_sync(0xffffffffu, c0 > hi || c0 + 31 < lo)) {
                        cm[q] = -INFINITY;
                    } else {
#pragma unroll
                        for (int k = 0; k < 32; ++k) {
                            const int key = c0 + k;
                            if (key < lo || key > hi)
                                s[32 * q + k] = -INFINITY;
                        }
                        // two independent 3-input max chains over the chunk
                        float m0 = fmax3(s[32 * q], s[32 * q + 1], s[32 * q + 2]);
                        float m1 = fmax3(s[32 * q + 16], s[32 * q + 17], s[32 * q + 18]);
#pragma unroll
                        for (int k = 3; k < 15; k += 2) {
                            m0 = fmax3(m0, s[32 * q + k], s[32 * q + k + 1]);
                            m1 = fmax3(m1, s[32 * q + 16 + k], s[32 * q + 16 + k + 1]);
                        }
                        cm[q] = fmax3(m0, m1, fmaxf(s[32 * q + 15], s[32 * q + 31]));
                    }
                }
                mx = fmax3(fmax3(cm[0], cm[1], cm[2]), cm[3], -INFINITY);
            }
            const float m_tile = mx * sl2;
            // keep a stale maximum until the row maximum grows by more than 2^8:
            // exact, since the denominator uses the same stale maximum
            const bool need = m_tile > m_used + 8.0f;
            // branch-free, so the warp does not diverge on rows whose maximum grew
            const float alpha = need ? ex2_approx(m_used - m_tile) : 1.f;
            l *= alpha;
            m_used = need ? m_tile : m_used;
            const float neg = m_used == -INFINITY ? 0.f : -m_used;
            const float2 sc = make_float2(sl2, sl2), ng = make_float2(neg, neg);
            float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
            const bool rescale = __any_sync(0xffffffffu, need) && j > it.g.n_lo;
            // P in kPParts parts (two keys per column, part h in columns
            // h * 64 / kPParts ..), each stored 16 columns at a time as produced
            constexpr int kPartPairs = kKvTile / 2 / C::kPParts;
#pragma unroll
            for (int part = 0; part < C::kPParts; ++part) {
#pragma unroll
                for (int q = 0; q < kPartPairs / 16; ++q) {
                    uint32_t pk[16];
                    // on a masked tile, 32 keys that no row of this warp sees give P = 0
                    // without any exponential
                    const int c0 = k0 + 2 * (part * kPartPairs + q * 16);
                    // (head_dim 64: every chunk, its masked scores giving 0)
                    if (!(D == 64 && !SPLIT) && !interior && __all_sync(0xffffffffu, c0 > hi || c0 + 31 < lo)) {
#pragma unroll
                        for (int kk = 0; kk < 16; ++kk)
                            pk[kk] = 0u;
                    } else {
#pragma unroll
                        for (int kk = 0; kk < 16; ++kk) {
                            const int k = part * kPartPairs + q * 16 + kk;
                            const float2 x = __ffma2_rn(make_float2(s[2 * k], s[2 * k + 1]), sc, ng);
                            const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                            acc[kk & 3] = __fadd2_rn(acc[kk & 3], e);
                            if (FP8) {
                                uint32_t r;
                                asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(e.y), "f"(e.x));
                                pk[kk] = r;
                            } else {
                                pk[kk] = pack_bf16x2(e.x, e.y);
                            }
                        }
                    }
                    tmem_st16(s_tmem + (uint32_t)(part * kPartPairs + q * 16), pk);
                }
                if (part == 0 && rescale) {
                    // O holds this item's sum up to tile j-1 (S(j) was issued after
                    // PV(j-1)); rescale it before the first P V of tile j
                    const float f = need ? alpha : 1.f;
                    const float2 ff = make_float2(f, f);
#pragma unroll 1  // rare; kept small (the softmax's code size costs time)
                    for (int q = 0; q < D / 16; ++q) {
                        uint32_t o[16];
                        tmem_ld16(o_tmem + (uint32_t)(q * 16), o);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 16; k += 2) {
                            const float2 v =
                                __fmul2_rn(make_float2(__uint_as_float(o[k]), __uint_as_float(o[k + 1])), ff);
                            o[k] = __float_as_uint(v.x);
                            o[k + 1] = __float_as_uint(v.y);
                        }
                        tmem_st16(o_tmem + (uint32_t)(q * 16), o);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                mbar_arrive_p(&c.bar.p_full[C::kPParts * t + part], lane == 0 ? 1u : 0u);
            }
            const float2 a01 = __fadd2_rn(acc[0], acc[1]), a23 = __fadd2_rn(acc[2], acc[3]);
            const float2 a = __fadd2_rn(a01, a23);
            l += a.x + a.y;
        }
        if (!ok)
            break;
        // epilogue: out = bmm2_scale * O / (l + e^{sink - m})
        if (!wait_bar(&c.bar.o_full[t], o_cnt & 1, c)) {
            ok = false;
            break;
        }
        ++o_cnt;
        tc_fence_after();
        const int h = it.kvh * G + r_head;
        float total = l;
        if (p.sinks != nullptr && m_used != -INFINITY && row_real)
            total += ex2_approx(fmaf(p.sinks[h], kLog2e, -m_used));
        const float inv = (m_used != -INFINITY && total > 0.f) ? scl.bmm2 / total : 0.f;
        const float2 inv2 = make_float2(inv, inv);
        uint16_t* orow = p.out + (long long)(it.q0 + (valid ? i : 0)) * p.out_stride_tok + (long long)h * p.out_stride_head;
        if (SPLIT && it.chunks > 1) {
            // one kv chunk of a split row: the unnormalised O and (m, l) in the
            // running maximum's log2 units; the combine kernel merges the chunks,
            // adds the sink term and applies bmm2_scale / denominator
            const long long slot = ((long long)(it.q0 + (valid ? i : 0)) * p.H + h) * p.part_slots + it.chunk;
            float4* po = reinterpret_cast<float4*>(p.part_o + slot * D);
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
                uint32_t o[32];
                tmem_ld32(o_tmem + (uint32_t)(q * 32), o);
                tmem_wait_ld();
                if (valid) {
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        po[q * 8 + v] = make_float4(__uint_as_float(o[4 * v]), __uint_as_float(o[4 * v + 1]),
                                                    __uint_as_float(o[4 * v + 2]), __uint_as_float(o[4 * v + 3]));
                }
            }
            if (valid)
                *reinterpret_cast<float2*>(p.part_ml + slot * 2) = make_float2(m_used, l);
        } else if constexpr (C::kStageOut) {
            // each 64-column half of the warp's 32 rows goes through shared
            // memory (row r in 128 bytes, 16-byte chunks swizzled by r % 8: the
            // 128-byte swizzle of the output tensor map).  When all 32 rows are
            // written and form whole boxes, lane 0 sends them with one TMA store
            // (asynchronous; nothing else waits for it); otherwise the warp
            // copies them out itself, four whole rows per store instruction.
            const uint32_t stage = smem_u32(c.base + C::kOffStage + (t * 4 + wq) * C::kStageWarpBytes);
            const unsigned long long my_row = reinterpret_cast<unsigned long long>(orow);
            const bool by_tma = p.out_tma != 0 && __all_sync(0xffffffffu, valid);
            const int r0 = wq * 32;  // first row of the warp: token r0 / G, head r0 % G
            const int c1 = it.kvh * G + r0 % G, c2 = it.q0 + i_first + r0 / G;
#pragma unroll 1  // the softmax's code size costs time: measured 1-2 % faster rolled
            for (int hh = 0; hh < D / 64; ++hh) {
                if (lane == 0)
                    bulk_wait_read_all();  // the previous store has read the staging
                __syncwarp();
                uint32_t oa[32], ob[32];
                tmem_ld32(o_tmem + (uint32_t)(hh * 64), oa);
                tmem_ld32(o_tmem + (uint32_t)(hh * 64 + 32), ob);
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
                        tma_store_3d(&p.tm_o, stage, hh * 64, c1, c2);
                        bulk_commit_group();
                    }
                } else {
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int r = 4 * k + (lane >> 3), cc = lane & 7;
                        const uint4 v = ld_shared_v4(stage + (uint32_t)(r * 128 + ((cc ^ (r & 7)) << 4)));
                        const unsigned long long a = __shfl_sync(0xffffffffu, my_row, r);
                        const int vr = __shfl_sync(0xffffffffu, valid ? 1 : 0, r);
                        if (vr)
                            *reinterpret_cast<uint4*>(a + (unsigned long long)(hh * 128 + cc * 16)) = v;
                    }
                    __syncwarp();
                }
            }
        } else {
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
                uint32_t o[32];
                tmem_ld32(o_tmem + (uint32_t)(q * 32), o);
                tmem_wait_ld();
                if (valid) {
                    uint32_t pkd[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const float2 v =
                            __fmul2_rn(make_float2(__uint_as_float(o[2 * k]), __uint_as_float(o[2 * k + 1])), inv2);
                        pkd[k] = pack_bf16x2(v.x, v.y);
                    }
                    uint4* dst = reinterpret_cast<uint4*>(orow + q * 32);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_uint4(pkd[4 * v], pkd[4 * v + 1], pkd[4 * v + 2], pkd[4 * v + 3]);
                }
            }
        }
    }
    if (C::kStageOut && lane == 0)
        bulk_wait_all();  // this warp's output stores are complete before the CTA exits
    tc_fence_before();
}

// ---------------------------------------------------------------------------
// e4m3 -> f16 conversion (FP8 KV path): warps 12-15, one thread per tile row.
// ---------------------------------------------------------------------------
// Two e4m3 values (low 16 bits of `two`) to two f16: exact, since every
// e4m3 value (subnormals included) is a normal f16 or zero.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two)
{
    uint32_t r;
    const uint16_t in = (uint16_t)two;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(in));
    return r;
}

// Power-of-two exponent k that brings a Q row with largest magnitude `mx`
// (bf16 bits, sign cleared) to [2^14, 2^15): then every element of the row at
// least 2^-31 of the largest is an exact f16 after scaling by 2^k (a bf16
// value has 8 significant bits, an f16 11, and f16 is exact down to 2^-17 at
// that precision).  Clamped to [-30, 100] so that 2^k and 2^-k stay normal
// floats; 0 for an all-zero row.
__device__ __forceinline__ int q_row_exponent(uint32_t mx)
{
    if (mx == 0)
        return 0;
    const int e = (int)((mx >> 7) & 0xFFu) - 127;  // unbiased exponent of the largest element
    return min(100, max(-30, 14 - e));
}


template <int D, bool FP8, bool SPLIT>
__device__ void convert_role(const AttnParams& p, const Ctx& c)
{
    using C = TcCfg<D, FP8, SPLIT>;
    const int ct = threadIdx.x - 12 * 32;  // 0..127: tile row
    const int lane = threadIdx.x & 31;
    const int sw = ct & 7;                 // 128-byte swizzle phase of this row
    uint32_t r8 = 0, r = 0;
    bool ok = true;
    for (uint32_t n = 0; ok; ++n) {
        ItemInfo it;
        const int w = take_item<C::kItemSlots>(p, c, n, &ok, &it);
        if (w < 0)
            break;
        // Q: thread ct takes row ct of each query tile: scale by 2^k into f16's
        // range, convert in place (same swizzled positions), post k
        const uint32_t qb = n % C::kQBufs, qph = (n / C::kQBufs) & 1;
        if (!wait_bar(&c.bar.q_full[qb], qph, c))
            break;
        int8_t* qexp = reinterpret_cast<int8_t*>(c.base + C::kOffQExp) + (n & 1) * kQTiles * kQRows;
        for (int t = 0; t < it.g.nq; ++t) {
            uint8_t* qrow = c.base + C::kOffQ + (qb * C::kQTilesAlloc + t) * C::kQTileBytes + ct * 128;
            uint32_t mx = 0;  // largest magnitude of the row, as bf16 bits
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint4 v = *reinterpret_cast<const uint4*>(qrow + h * C::kHalfBytes + (q << 4));
                    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        mx = max(mx, max(w4[e] & 0x7FFFu, (w4[e] >> 16) & 0x7FFFu));
                }
            const int k = q_row_exponent(mx);
            const float sc = __int_as_float((127 + k) << 23);
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint4 v = *reinterpret_cast<const uint4*>(qrow + h * C::kHalfBytes + (q << 4));
                    uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float lo = __uint_as_float(w4[e] << 16) * sc, hi = __uint_as_float(w4[e] & 0xFFFF0000u) * sc;
                        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(w4[e]) : "f"(hi), "f"(lo));
                    }
                    *reinterpret_cast<uint4*>(qrow + h * C::kHalfBytes + (q << 4)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
            qexp[t * kQRows + ct] = (int8_t)k;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&c.bar.q_conv[qb]);
        for (int j = it.g.n_lo; ok && j <= it.g.n_hi; ++j) {
            const bool zero = j * kKvTile + ct >= it.kv_len;
            // the ring pair of this tile: K into entry 2m, V into 2m + 1
            const uint32_t m = r % C::kPairs;
            if (!wait_bar(&c.bar.empty[m], ((r / C::kPairs) & 1) ^ 1, c)) {
                ok = false;
                break;
            }
            for (int kind = 0; kind < 2; ++kind) {
                const uint32_t s8 = r8 % C::kF8Stages;
                if (!wait_bar(&c.bar.f8full[s8], (r8 / C::kF8Stages) & 1, c)) {
                    ok = false;
                    break;
                }
                const uint8_t* src = c.base + C::kOffF8 + s8 * C::kF8TileBytes + ct * 128;
                uint8_t* dst = c.base + C::kOffRing + (2 * m + kind) * C::kKvTileBytes + ct * 128;
#pragma unroll
                for (int q = 0; q < 8; ++q) {  // 16 e4m3 values = d 16q .. 16q+15
                    uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = make_uint4(0u, 0u, 0u, 0u);
                    if (!zero) {
                        const uint4 x = *reinterpret_cast<const uint4*>(src + ((q ^ sw) << 4));
                        lo.x = e4m3x2_to_f16x2(x.x);
                        lo.y = e4m3x2_to_f16x2(x.x >> 16);
                        lo.z = e4m3x2_to_f16x2(x.y);
                        lo.w = e4m3x2_to_f16x2(x.y >> 16);
                        hi.x = e4m3x2_to_f16x2(x.z);
                        hi.y = e4m3x2_to_f16x2(x.z >> 16);
                        hi.z = e4m3x2_to_f16x2(x.w);
                        hi.w = e4m3x2_to_f16x2(x.w >> 16);
                    }
                    const int hb = q >> 2, cc = (2 * q) & 7;
                    uint8_t* rowp = dst + hb * C::kHalfBytes;
                    *reinterpret_cast<uint4*>(rowp + ((cc ^ sw) << 4)) = lo;
                    *reinterpret_cast<uint4*>(rowp + (((cc + 1) ^ sw) << 4)) = hi;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(kind == 0 ? &c.bar.full[m] : &c.bar.vfull[m]);  // K lets Q K^T start early
                    mbar_arrive(&c.bar.f8empty[s8]);
                }
                ++r8;
            }
            ++r;  // one ring pair per tile
        }
    }
}

// ---------------------------------------------------------------------------
template <int D, bool FP8, bool SPLIT>
__global__ void __launch_bounds__(TcCfg<D, FP8, SPLIT>::kThreads, 1) attention_tc_kernel(const __grid_constant__ AttnParams p)
{
    using C = TcCfg<D, FP8, SPLIT>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::kOffBar);
    Ctx c;
    c.base = base;
    c.bar.full = bars;
    c.bar.empty = c.bar.full + C::kPairs;
    c.bar.vfull = c.bar.empty + C::kPairs;
    c.bar.vempty = c.bar.vfull + C::kPairs;
    c.bar.f8full = c.bar.vempty + C::kPairs;
    c.bar.f8empty = c.bar.f8full + C::kF8Stages;
    c.bar.q_full = c.bar.f8empty + C::kF8Stages;
    c.bar.q_empty = c.bar.q_full + C::kQBufs;
    c.bar.q_conv = c.bar.q_empty + C::kQBufs;
    c.bar.s_full = c.bar.q_conv + C::kQBufs;
    c.bar.p_full = c.bar.s_full + kQTiles;
    c.bar.o_full = c.bar.p_full + C::kPParts * kQTiles;
    c.bar.drain = c.bar.o_full + kQTiles;
    c.bar.it_full = c.bar.drain + 1;
    c.bar.it_empty = c.bar.it_full + C::kItemSlots;
    c.bar.never = c.bar.it_empty + C::kItemSlots;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base + C::kOffMisc);
    c.abort_flag = reinterpret_cast<volatile int*>(base + C::kOffMisc + 4);
    c.err = p.err;
    c.wait_limit_ns = p.wait_limit_ns;
    c.item_slot = reinterpret_cast<volatile int*>(base + C::kOffMisc + 16);
    const int warp = threadIdx.x >> 5;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kPairs; ++s) {
            mbar_init(&c.bar.full[s], FP8 ? 4 : 1);
            mbar_init(&c.bar.empty[s], 1);
            mbar_init(&c.bar.vfull[s], FP8 ? 4 : 1);
            mbar_init(&c.bar.vempty[s], 1);
        }
        for (int s = 0; s < C::kF8Stages; ++s) {
            mbar_init(&c.bar.f8full[s], 1);
            mbar_init(&c.bar.f8empty[s], 4);
        }
        for (int b = 0; b < C::kQBufs; ++b) {
            mbar_init(&c.bar.q_full[b], 1);
            mbar_init(&c.bar.q_empty[b], 1);
            mbar_init(&c.bar.q_conv[b], 4);
        }
        for (int t = 0; t < kQTiles; ++t) {
            mbar_init(&c.bar.s_full[t], 1);
            for (int h = 0; h < C::kPParts; ++h)
                mbar_init(&c.bar.p_full[C::kPParts * t + h], 4);
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
        const int pad = C::kHalfBytes - used;
        if (pad > 0) {
            const int n16 = pad / 16;
            for (int k = threadIdx.x; k < C::kQBufs * C::kQTilesAlloc * C::kHalves * n16; k += blockDim.x) {
                const int blk = k / n16, q = k % n16;
                *reinterpret_cast<uint4*>(base + C::kOffQ + blk * C::kHalfBytes + used + q * 16) =
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
        // every CTA sorts the work itself, in the K/V ring before any copy
        // lands there; the first to win the claim also writes the list
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
        fence_proxy_async_smem();  // the ring's next writes come through the async proxy
        __syncthreads();
    }

    if constexpr (FP8) {
        // 512 threads launch with 128 registers each; the softmax warpgroups
        // take registers from the others (88 + 176 + 176 + 72 = 512 = 4 x 128)
        if (warp < 4) {
            regs_dec<88>();
            if (warp == 0)
                producer_role<D, FP8, SPLIT>(p, c);
            else if (warp == 1)
                mma_role<D, FP8, SPLIT>(p, c);
        } else if (warp < 12) {
            regs_inc<176>();
            softmax_role<D, FP8, SPLIT>(p, c, (warp - 4) >> 2);
        } else {
            regs_dec<72>();
            convert_role<D, FP8, SPLIT>(p, c);
        }
    } else {
        // 384 threads launch with 168 registers each (104 + 200 + 200 = 504 = 3 x 168)
        if (warp < 4) {
            regs_dec<104>();
            if (warp == 0)
                producer_role<D, FP8, SPLIT>(p, c);
            else if (warp == 1)
                mma_role<D, FP8, SPLIT>(p, c);
        } else {
            regs_inc<200>();
            softmax_role<D, FP8, SPLIT>(p, c, (warp - 4) >> 2);
        }
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

template <int D, bool FP8, bool SPLIT>
static cudaError_t launch_one(const AttnParams& p, int grid, cudaStream_t stream, bool pdl)
{
    using C = TcCfg<D, FP8, SPLIT>;
    auto kern = attention_tc_kernel<D, FP8, SPLIT>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    // the shared-memory opt-in, once per device and instantiation (any host thread)
    static std::once_flag attr_once[64];
    static cudaError_t attr_err[64];
    std::call_once(attr_once[dev], [&] {
        attr_err[dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    });
    if (attr_err[dev] != cudaSuccess)
        return attr_err[dev];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <bool SPLIT>
static cudaError_t launch_variant(const AttnParams& p, int head_dim, bool fp8, int grid, cudaStream_t stream, bool pdl)
{
    if (fp8)
        return head_dim == 128 ? launch_one<128, true, SPLIT>(p, grid, stream, pdl) : cudaErrorInvalidValue;
    if (head_dim == 128)
        return launch_one<128, false, SPLIT>(p, grid, stream, pdl);
    if (head_dim == 64)
        return launch_one<64, false, SPLIT>(p, grid, stream, pdl);
    return cudaErrorInvalidValue;
}

cudaError_t launch_attention_tc(const AttnParams& p, int head_dim, bool fp8, int grid, cudaStream_t stream, bool pdl)
{
    return p.split_tiles > 0 ? launch_variant<true>(p, head_dim, fp8, grid, stream, pdl)
                             : launch_variant<false>(p, head_dim, fp8, grid, stream, pdl);
}

}  // namespace b2pa
