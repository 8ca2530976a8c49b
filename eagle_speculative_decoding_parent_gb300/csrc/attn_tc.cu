// tree_verify_attention, bfloat16 path on the 5th-generation tensor cores.
//
// Used for head size 128 (the warp-MMA kernel serves head size 64).  A group
// is (sequence, kv head, row tile).  Two schedules:
//   balanced split (groups too few to give every SM one, but at least half
//            as many, and the caller's workspace holds the partial results):
//            the grid is QT CTAs (one per row tile) times `lanes`; the key
//            tiles of all (sequence, kv head) pairs, laid end to end with a
//            fixed cost per piece, are cut into `lanes` runs of equal length,
//            so every CTA streams the same work.  A group cut by a run
//            boundary leaves one partial result (running max, sum, normalised
//            O) per run in global memory; a second kernel, launched under
//            programmatic dependent launch, merges them.
//   clusters (otherwise): groups go dynamically, longest first, to clusters of
//            CS CTAs that split the group's keys and merge through distributed
//            shared memory.
// A row tile holds npt = floor(128 / G) whole nodes (all G query heads of the
// kv head for each), rows r = node * G + head, so one TMA box loads it.
//
// CTA roles (288 threads, one CTA per SM)
//   warp 0   producer of pages 0-1 of each 64-key K/V tile; warp 2 loads
//            pages 2-3.  A 16-key page is one K box ([row group][half][8 rows]
//            [128 B], so the 8-key groups of a tile are 2 KB apart for the S
//            product) and one V box ([half][16 rows][128 B]); a warp's four copies
//            of a tile are issued by four lanes at once.  The ring has 5 stages (4 when a
//            cluster splits the group).  Neither producer ever waits for data:
//            the rows of a group's last, partial tile past the sequence end are
//            zeroed in V by the PV issuer just before its product.
//            Warp 2 allocates / frees 512 tensor-memory columns: S double buffer
//            (2 x 64), O (128), P (2 x 32).
//   warp 8   work items (cluster schedule, rank 0): takes the next group from
//            the counter, checks its sequence's block table and resolves each
//            rank's first 32 pages into cache rows, one group ahead of the
//            producers, so a new group's copies start without a global-memory
//            round trip.  Under the balanced split the pieces are listed in the
//            prologue and warp 0 hands them out.
//   warp 1   S issuer: loads each group's Q tile (3-D TMA box) once the
//            previous group's S products are done with it, so the K/V stream
//            runs on across groups; S = Q K^T into tensor memory (M=128, N=64,
//            K=16 steps, both operands in shared memory), double-buffered S.
//   warp 3   PV issuer: O += P V (M=128, N=128, P read from tensor memory, V
//            N-major in shared memory), in tile order; releases the K/V stage.
//            Completion is signalled with tcgen05.commit (it covers only the
//            issuing thread's products, so each issuer commits its own).  Every
//            tcgen05 and TMA instruction is issued by an elect.sync-chosen lane
//            of a converged warp.
//   warps 4-7 softmax: thread i owns row i (tensor-memory lane i); reads S,
//            applies scale and tree mask, keeps a running max that is only
//            raised (and O rescaled in tensor memory) when it grows by more
//            than 2^8, writes P (bf16 pairs) to tensor memory for the PV
//            product, and finally normalises O.
// Balanced split: before the roles start, the CTA lists its run's pieces (up
// to MAXI) and checks the block tables of their sequences with every warp at
// once; the producers load each next piece's first block ids while the
// current one streams.  So no global-memory round trip sits between pieces
// but the K/V data itself.
#include <algorithm>

#include "tv_device.cuh"
#include "tv_internal.h"
#include "tv_tc.cuh"

namespace tv {

namespace {

constexpr int KT = 64;        // keys per tile
constexpr int STAGES = 5;           // K/V ring depth when a CTA owns whole groups
constexpr int STAGES_CLUSTER = 4;   // with a cluster split the fifth stage holds the merge rows
constexpr int GQ = 4;
constexpr int THREADS = 288;
constexpr int SOFTMAX_WARP0 = 4;  // softmax warps 4-7
constexpr int FETCH_WARP = 8;
// Cluster schedule: the next group is claimed when this many key tiles of the
// current one are left to issue (enough to hide the claim and the block-table
// checks, late enough to keep the longest-first balance of the counter).
constexpr int FETCH_LEAD = 6;
constexpr int MAX_CS = 8;
constexpr int D = 128;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_O = 128;         // O at columns 128..255, S buffers at 0 and 64
constexpr uint32_t TMEM_P = 256;         // P buffers (packed bf16 pairs) at 256 and 288
constexpr float LOG2E = 1.4426950408889634f;
constexpr float RESCALE_LOG2 = 8.0f;     // raise the running max only past 2^8 growth

constexpr uint32_t IDESC_QK = idesc_bf16(128, KT, false);
constexpr uint32_t IDESC_PV = idesc_bf16(128, D, true);

// shared memory layout (offsets from a 1024-byte aligned base)
constexpr int TILE_BYTES = KT * D * 2;                 // 16 KB: one K or V tile
constexpr int OFF_RING = 0;                            // STAGES x (K, V)
// fp16 normalised O rows for the cluster merge (128 x 128 x 2 = one stage) in the fifth stage
constexpr int OFF_XO = OFF_RING + STAGES_CLUSTER * 2 * TILE_BYTES;
static_assert(128 * D * 2 <= 2 * TILE_BYTES, "merge rows fit in one ring stage");
constexpr int OFF_Q = OFF_RING + STAGES * 2 * TILE_BYTES;
constexpr int Q_BYTES = 128 * D * 2;                   // 32 KB
constexpr int OFF_XML = OFF_Q + Q_BYTES;               // (max, sum) per row
constexpr int OFF_WTS = OFF_XML + 128 * 8;             // merge weights [128][MAX_CS]
constexpr int OFF_BARS = OFF_WTS + 128 * MAX_CS * 4;
constexpr int NUM_BARS = 2 * STAGES + 2 + 2 * 4 + 2 + 2 * GQ + 2;
constexpr int OFF_MISC = OFF_BARS + NUM_BARS * 8;
constexpr int OFF_LPT = OFF_MISC + 64;                 // sequence order: lens, order
constexpr int OFF_CUM = OFF_LPT + 2 * LPT_MAX * 4;     // balanced split: int64 [LPT_MAX + 1]
constexpr int OFF_GQ4 = OFF_CUM + (LPT_MAX + 1) * 8 + 8;  // queue slots [GQ] x (word, first tile, end tile, -)
constexpr int MAXI = 64;                               // balanced split: pieces listed up front
constexpr int OFF_ITEMS = OFF_GQ4 + GQ * 16;           // [MAXI] x (word, first tile, end tile, bad)
constexpr int OFF_NITEMS = OFF_ITEMS + MAXI * 16;
constexpr int OFF_WIN = OFF_NITEMS + 16;               // [GQ][32] first-window cache rows
constexpr int OFF_CNT = OFF_WIN + GQ * 32 * 4;         // node count per sequence [LPT_MAX]
constexpr int SMEM_BYTES = OFF_CNT + LPT_MAX * 4 + 1024;  // + alignment slack
static_assert(OFF_CUM % 8 == 0, "int64 prefix sums");
static_assert(OFF_ITEMS % 16 == 0 && OFF_GQ4 % 16 == 0, "int4 slots");
// Balanced split: cost of starting a piece (Q tile, pipeline fill and drain,
// epilogue), in key-tile times.
constexpr int SPLIT_C0 = 4;
// one partial result in the workspace: fp16 normalised O rows, then (max, sum) per row
constexpr int SLOT_O_BYTES = 128 * D * 2;
constexpr int SLOT_BYTES = SLOT_O_BYTES + 128 * 8;

struct Params {
    const int32_t* table;
    const int32_t* prefix_lens;
    const uint64_t* mask;
    const int32_t* counts;  // nullable: nodes per sequence (its tree: the first counts[b] of N)
    __nv_bfloat16* out;
    int32_t* status;
    int32_t* sched;
    uint8_t* part;         // balanced split: 2 partial-result slots per CTA
    int max_blocks, B, N, Hq, Hkv, G, npt, bs, num_blocks, QT, groups;
    int lanes;             // balanced split: grid = lanes * QT, no clusters
    int c0;                // balanced split: fixed cost of a piece, in key tiles
    float scale_log2;
};

struct Group {
    int b, g, qt, P, n, L, t_lo, t_hi;  // n nodes, L = P + n keys
    bool ok;
    bool whole;            // the piece covers all of the group's key tiles
};

// A fetched work item: group word and, for the balanced split, its key tiles.
struct Item {
    int word, t_lo, t_hi;
};

// Node count of sequence b (cnts: the counts staged in shared memory, or null).
__device__ __forceinline__ int seq_nodes(const Params& p, const int* cnts, int b) {
    return cnts ? cnts[b] : (p.counts ? p.counts[b] : p.N);
}
// A sequence is usable when its node count is in [1, N] and its P + n keys
// fit the block table.
__device__ __forceinline__ bool seq_shape_ok(const Params& p, int P, int n) {
    return P >= 0 && n >= 1 && n <= p.N && (int64_t)P + n <= (int64_t)p.max_blocks * p.bs;
}

// Balanced split: the run space.  Group (b, g) takes c0 + T_b units, c0 for
// the fixed cost of starting a piece and then one per key tile; cum[0..B] is
// the exclusive prefix sum over sequences (Hkv groups each), and lens[b] the
// prefix length, cnts[b] the node count.  A sequence whose prefix length or
// node count is out of range counts one tile, so that one CTA owns it and
// reports it.  Called by every thread of the CTA; B <= LPT_MAX.
__device__ __forceinline__ void split_prefix(const Params& p, int64_t* cum, int* lens, int* cnts) {
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int64_t v[LPT_MAX / 32];
#pragma unroll
        for (int u = 0; u < LPT_MAX / 32; ++u) {
            const int b = u * 32 + lane;
            v[u] = 0;
            if (b < p.B) {
                const int P = p.prefix_lens[b];
                const int n = p.counts ? p.counts[b] : p.N;
                lens[b] = P;
                cnts[b] = n;
                const bool ok = seq_shape_ok(p, P, n);
                v[u] = (int64_t)((ok ? (P + n + KT - 1) / KT : 1) + p.c0) * p.Hkv;
            }
        }
        int64_t run = 0;
#pragma unroll
        for (int u = 0; u < LPT_MAX / 32; ++u) {
            int64_t x = v[u];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            const int b = u * 32 + lane;
            if (b < p.B) cum[b + 1] = run + x;
            run += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) cum[0] = 0;
    }
    __syncthreads();
}

// Balanced split: first tile of lane l's run among U tiles cut into L runs, and
// the lane whose run holds tile x.
__device__ __forceinline__ int64_t run_start(int64_t l, int64_t U, int64_t L) { return l * U / L; }
__device__ __forceinline__ int64_t run_owner(int64_t x, int64_t U, int64_t L) {
    return ((x + 1) * L - 1) / U;
}

__device__ __forceinline__ bool seq_ok_warp(const Params& p, int b, int P, int n) {
    const int lane = threadIdx.x & 31;
    bool ok = seq_shape_ok(p, P, n);
    if (ok) {
        // four independent loads per lane in flight per round
        const int nb = (P + n + p.bs - 1) / p.bs;
        const int32_t* row = p.table + (int64_t)b * p.max_blocks;
        for (int j0 = 0; j0 < nb; j0 += 128) {
            int blk[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = j0 + u * 32 + lane;
                blk[u] = (j < nb) ? row[j] : 0;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) ok = ok && blk[u] >= 0 && blk[u] < p.num_blocks;
        }
    }
    return __all_sync(0xffffffffu, ok);
}

// Group ids travel with a validity bit: the fetching warp checks the group's
// sequence once (seq_ok_warp) and marks a bad one with GROUP_BAD.
constexpr int GROUP_BAD = 1 << 30;

__device__ __forceinline__ int group_seq(const Params& p, const int* order, int gi) {
    const int r = gi / (p.QT * p.Hkv);
    return order ? order[r] : r;
}

// Fetched word -> group: sequence (in longest-first order when `order` is
// given), kv head, row tile; this CTA's share of its key tiles.
template <bool SPLIT>
__device__ __forceinline__ Group decode_group(const Params& p, const int* order, const int* lens,
                                             const int* cnts, const int64_t* cum, const Item& it,
                                             int rank, int cs) {
    Group gr;
    const int word = it.word;
    const int gi = word & (GROUP_BAD - 1);
    gr.qt = gi % p.QT;
    gr.g = (gi / p.QT) % p.Hkv;
    gr.b = group_seq(p, order, gi);
    gr.P = lens ? lens[gr.b] : p.prefix_lens[gr.b];
    gr.ok = (word & GROUP_BAD) == 0;
    gr.n = gr.ok ? seq_nodes(p, cnts, gr.b) : p.N;  // a bad sequence: every row gets zeros
    gr.L = gr.P + gr.n;
    const int T = gr.ok ? (gr.L + KT - 1) / KT : 0;
    if constexpr (SPLIT) {
        // a piece of a bad sequence reads nothing: a whole one writes zeros, a
        // partial one an empty partial result (zero weight in the merge)
        const int T_run = (int)((cum[gr.b + 1] - cum[gr.b]) / p.Hkv) - p.c0;
        gr.t_lo = gr.ok ? it.t_lo : 0;
        gr.t_hi = gr.ok ? it.t_hi : 0;
        gr.whole = (it.t_lo == 0 && it.t_hi == T_run);
    } else {
        gr.t_lo = (int)((int64_t)T * rank / cs);
        gr.t_hi = (int)((int64_t)T * (rank + 1) / cs);
        gr.whole = (cs == 1);
    }
    return gr;
}

// SPLIT: the balanced split (else the cluster schedule); one instantiation
// each, so that neither carries the other's code.
template <bool SPLIT>
__global__ void __launch_bounds__(THREADS, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
               const __grid_constant__ CUtensorMap vmap, Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BARS);
    uint64_t* kfull = bars;                   // [STAGES]
    uint64_t* kempty = kfull + STAGES;        // [STAGES]
    uint64_t* qfull = kempty + STAGES;
    uint64_t* qempty = qfull + 1;
    uint64_t* sfull = qempty + 1;             // [2]
    uint64_t* sfree = sfull + 2;              // [2]
    uint64_t* pfull = sfree + 2;              // [2]
    uint64_t* pfree = pfull + 2;              // [2] PV product of tile t done (by t & 1)
    uint64_t* ofree = pfree + 2;
    uint64_t* ptake = ofree + 1;              // producer took item k (phase k & 1)
    uint64_t* gq_full = ptake + 1;            // [GQ]
    uint64_t* gq_empty = gq_full + GQ;        // [GQ]
    uint64_t* xready = gq_empty + GQ;
    uint64_t* xfree = xready + 1;
    int* misc = reinterpret_cast<int*>(smem + OFF_MISC);
    // queue slot: the group word (stored into every cluster rank) and, for the
    // balanced split, the piece's key tiles; read with one 16-byte load
    int4* gq4 = reinterpret_cast<int4*>(smem + OFF_GQ4);
    uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(misc + GQ);
    int* flags = misc + GQ + 1;               // [0] abort

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_rank(), cs = cluster_size();
    const uint32_t sbase = smem_u32(smem);
    const uint32_t nst = (cs == 1) ? STAGES : STAGES_CLUSTER;  // K/V ring depth
    pdl_launch_dependents();

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&kfull[s], 2);              // both producers
            mbar_init(&kempty[s], 1);
        }
        mbar_init(qfull, 1);
        mbar_init(qempty, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sfull[i], 1);
            mbar_init(&sfree[i], 4);
            mbar_init(&pfull[i], 4);
            mbar_init(&pfree[i], 1);
        }
        mbar_init(ofree, 4);
        mbar_init(ptake, 1);
        for (int s = 0; s < GQ; ++s) {
            mbar_init(&gq_full[s], 1);
            mbar_init(&gq_empty[s], cs * 8);      // 2 producers, 2 MMA issuers, 4 softmax warps
        }
        mbar_init(xready, cs * 4);
        mbar_init(xfree, cs * 4);
        flags[0] = 0;
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc(tmem_base_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    cluster_barrier_all();
    tc_fence_after();
    pdl_wait();  // everything above touched only shared memory and TMEM
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_base_slot);
    const int* order = nullptr;
    const int64_t* cum = reinterpret_cast<const int64_t*>(smem + OFF_CUM);
    // prefix lengths in shared memory (every sequence fits the table)
    int* lens_w = reinterpret_cast<int*>(smem + OFF_LPT);
    const int* lens = (SPLIT || (p.B > 1 && p.B <= LPT_MAX)) ? lens_w : nullptr;
    // node counts in shared memory alongside (raw: checked where used)
    int* cnts_w = reinterpret_cast<int*>(smem + OFF_CNT);
    const int* cnts = lens ? cnts_w : nullptr;
    // balanced split: the run's pieces listed up front
    int4* items = reinterpret_cast<int4*>(smem + OFF_ITEMS);  // word, first tile, end tile, bad
    int* n_items = reinterpret_cast<int*>(smem + OFF_NITEMS);
    int* items_more = n_items + 1;
    // cluster schedule: per queue slot, lane l's page l of the first window as a cache row
    int* win0 = reinterpret_cast<int*>(smem + OFF_WIN);
    // balanced split: this CTA's run [x_lo, x_hi) of the run space and its row tile
    int64_t U = 0, L = 0, x_lo = 0, x_hi = 0;
    int qt_me = 0;
    if constexpr (SPLIT) {
        split_prefix(p, reinterpret_cast<int64_t*>(smem + OFF_CUM), lens_w, cnts_w);
        U = cum[p.B];
        L = min((int64_t)p.lanes, U);  // every run holds at least one tile
        const int64_t lane_me = blockIdx.x / p.QT;
        qt_me = (int)(blockIdx.x % p.QT);
        if (lane_me < L) {
            x_lo = run_start(lane_me, U, L);
            x_hi = run_start(lane_me + 1, U, L);
        }
    } else if (p.B > 1 && p.B <= LPT_MAX) {
        lpt_order(p.prefix_lens, p.B, lens_w, lens_w + LPT_MAX);
        for (int b = threadIdx.x; b < p.B; b += blockDim.x) cnts_w[b] = p.counts ? p.counts[b] : p.N;
        __syncthreads();
        order = lens_w + LPT_MAX;
    }
    // balanced split: the run's pieces as (group, first tile, end tile).  A piece
    // that starts in the run and continues into the next one goes first, so
    // that the groups cut at both ends of the run are finished (and merged)
    // early; then the rest of the run in order.  Group p.groups once done.
    // (the fetching warp only)
    int64_t x_next = x_lo, x_stop = x_hi;
    bool z_first = false;
    int z_word = 0, z_thi = 0;
    auto split_locate = [&](int64_t x, int& b, int64_t& w, int64_t& g0) {
        int lo = 0, hi = p.B;  // cum[lo] <= x < cum[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cum[mid] <= x) lo = mid;
            else hi = mid;
        }
        b = lo;
        w = (cum[lo + 1] - cum[lo]) / p.Hkv;   // c0 + tiles
        g0 = x - (x - cum[lo]) % w;            // the group's first unit
    };
    if (SPLIT && x_hi > x_lo) {
        int b;
        int64_t w, g0;
        split_locate(x_hi - 1, b, w, g0);
        const int64_t f = g0 + p.c0, tb = w - p.c0;  // first tile unit, tiles
        if (f >= x_lo && f < x_hi && f + tb > x_hi) {
            z_first = true;
            z_word = (b * p.Hkv + (int)((g0 - cum[b]) / w)) * p.QT + qt_me;
            z_thi = (int)(x_hi - f);
            x_stop = g0;
        }
    }
    auto split_next = [&](int& word, int& tlo, int& thi) {
        word = p.groups;
        tlo = thi = 0;
        if (z_first) {
            z_first = false;
            word = z_word;
            thi = z_thi;
            return;
        }
        while (x_next < x_stop) {
            int b;
            int64_t w, g0;
            split_locate(x_next, b, w, g0);
            const int64_t f = g0 + p.c0, tb = w - p.c0;
            if (x_next < f) {
                if (f >= x_stop) {  // the group's tiles all lie past this run
                    x_next = x_stop;
                    break;
                }
                x_next = f;
            }
            const int64_t t = x_next - f;
            const int64_t take = min(tb - t, x_stop - x_next);
            word = (b * p.Hkv + (int)((g0 - cum[b]) / w)) * p.QT + qt_me;
            tlo = (int)t;
            thi = (int)(t + take);
            x_next += take;
            return;
        }
    };

    if constexpr (SPLIT) {
        // the run's pieces, in the order they will be handed out (warp 0 keeps the
        // state for any pieces past the list)
        if (warp == 0) {
            int n = 0;
            while (n < MAXI) {
                int gi, tlo, thi;
                split_next(gi, tlo, thi);
                if (gi >= p.groups) break;
                if (lane == 0) items[n] = make_int4(gi, tlo, thi, 0);
                ++n;
            }
            if (lane == 0) {
                *n_items = n;
                *items_more = (n == MAXI) ? 1 : 0;
            }
        }
        __syncthreads();
        // block tables of the listed pieces' sequences, in units of 512 block ids
        // spread over all warps (16 loads per lane in flight)
        {
            const int n = *n_items;
            int u = 0;
            for (int i = 0; i < n; ++i) {
                const int b = group_seq(p, nullptr, items[i].x);
                const int P = lens[b], nn = cnts[b];
                const bool pok = seq_shape_ok(p, P, nn);
                const int nb = pok ? (P + nn + p.bs - 1) / p.bs : 0;
                const int chunks = max(1, (nb + 511) / 512);
                for (int c = 0; c < chunks; ++c, ++u) {
                    if (u % (THREADS / 32) != warp) continue;
                    bool ok = pok;
                    if (ok) {
                        const int32_t* row = p.table + (int64_t)b * p.max_blocks;
                        int blk[16];
#pragma unroll
                        for (int v = 0; v < 16; ++v) {
                            const int j = c * 512 + v * 32 + lane;
                            blk[v] = (j < nb) ? row[j] : 0;
                        }
#pragma unroll
                        for (int v = 0; v < 16; ++v) ok = ok && blk[v] >= 0 && blk[v] < p.num_blocks;
                    }
                    if (!__all_sync(0xffffffffu, ok) && lane == 0) atomicOr(&items[i].w, 1);
                }
            }
        }
        __syncthreads();
        if (tid < *n_items && items[tid].w) items[tid].x |= GROUP_BAD;
        __syncthreads();
    }

    // Work item k: the fetching warp publishes it into every cluster rank's
    // queue slot (fetch_item), every role reads it from its own (take_item).
    // The fetcher is a whole warp: it also validates the group's sequence and,
    // under the cluster schedule, resolves each rank's first window of 32 pages
    // into cache rows (win0).  Returns the group index (>= p.groups: the end).
    auto fetch_item = [&](uint32_t k) -> int {
        const int slot = k % GQ;
        int gi = p.groups, tlo = 0, thi = 0, word = p.groups;
        const bool free_slot = __all_sync(
            0xffffffffu, lane != 0 || mbar_wait_cluster(&gq_empty[slot], ((k / GQ) & 1u) ^ 1u));
        if (!free_slot) {
            // timed out: hand out the end marker
        } else if (SPLIT && (int)k < *n_items) {
            word = items[k].x;  // listed and checked in the prologue
            gi = word & (GROUP_BAD - 1);
            tlo = items[k].y;
            thi = items[k].z;
        } else {
            if constexpr (SPLIT) {
                if (!*items_more) gi = p.groups;
                else split_next(gi, tlo, thi);
            } else {
                // the first group of every cluster is its cluster index; later ones
                // come from the counter, after the clusters' first groups
                const int nclusters = (int)(gridDim.x / cs);
                if (lane == 0)
                    gi = (k == 0) ? (int)(blockIdx.x / cs) : nclusters + atomicAdd(&p.sched[0], 1);
                gi = __shfl_sync(0xffffffffu, gi, 0);
            }
            word = gi;
            if (gi < p.groups) {
                const int b = group_seq(p, order, gi);
                const int P = lens ? lens[b] : p.prefix_lens[b];
                const int nn = seq_nodes(p, cnts, b);
                if (!seq_ok_warp(p, b, P, nn)) {
                    word |= GROUP_BAD;
                } else if (!SPLIT) {
                    // each rank's first window: page `lane` of its share of the keys
                    const int g = (gi / p.QT) % p.Hkv, Lg = P + nn, T = (Lg + KT - 1) / KT;
                    for (uint32_t r = 0; r < cs; ++r) {
                        const int tk = ((int)((int64_t)T * r / cs) * (KT / 16) + lane) * 16;
                        int y = 0;
                        if (tk < Lg)
                            y = (__ldg(p.table + (int64_t)b * p.max_blocks + tk / p.bs) * p.Hkv + g) * p.bs +
                                tk % p.bs;
                        remote_st_u32(&win0[slot * 32 + lane], r, y);
                    }
                    asm volatile("fence.acq_rel.cluster;" ::: "memory");
                }
            }
        }
        __syncwarp();
        if (lane == 0) {
            gq4[slot].y = tlo;  // balanced split only: no cluster peers
            gq4[slot].z = thi;
            for (uint32_t r = 0; r < cs; ++r) {
                remote_st_u32(&gq4[slot].x, r, word);
                remote_arrive(&gq_full[slot], r);
            }
        }
        return gi;
    };
    // y0 (nullable): this lane's page of the first window, as a cache row
    auto take_item = [&](uint32_t k, int* y0) -> Item {
        const int slot = k % GQ;
        const bool got = __all_sync(0xffffffffu, mbar_wait_cluster(&gq_full[slot], (k / GQ) & 1u));
        const int4 v = lds_v4_volatile(&gq4[slot]);
        Item it;
        it.word = got ? v.x : p.groups;
        it.t_lo = v.y;
        it.t_hi = v.z;
        int dep = got ? v.x : 0;
        if (y0) {
            *y0 = *reinterpret_cast<volatile int*>(&win0[slot * 32 + lane]);
            // the slot may be refilled only after every lane's row was read
            if (__any_sync(0xffffffffu, *y0 < 0)) dep |= INT_MIN;
        }
        __syncwarp();
        // "slot read": no release needed, and a release here would wait for the
        // softmax warps' output stores of the previous group
        if (lane == 0) remote_arrive_relaxed_after(&gq_empty[slot], 0, dep);
        return it;
    };

    auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity));
    };

    if (warp == 0 || warp == 2) {
        // ==== producers: warp 0 loads pages 0-1 of each tile, warp 2 pages 2-3 ====
        // (two warps on different schedulers: each issues half of a tile's copies;
        // a page is two K boxes, one per 64-column half, and one V box)
        const bool kprod = (warp == 0);
        const int pg0 = kprod ? 0 : KT / 32;
        if (lane == 0) {
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
        }
        const uint64_t policy = (p.QT == 1) ? l2_policy_evict_first() : l2_policy_evict_normal();
        uint32_t gt = 0;
        bool alive = true;
        // balanced split: block id of page `lane` of listed piece pf_k, loaded one
        // piece ahead
        int pf_blk = 0, pf_k = -1;
        for (uint32_t k = 0; alive; ++k) {
            int y0 = 0;
            if (SPLIT && kprod && rank == 0) fetch_item(k);
            const Item it = take_item(k, SPLIT ? nullptr : &y0);
            if ((it.word & (GROUP_BAD - 1)) >= p.groups) break;
            const Group gr = decode_group<SPLIT>(p, order, lens, cnts, cum, it, rank, cs);
            const int n = gr.t_hi - gr.t_lo;
            // cluster schedule: let the fetch warp claim item k + 1 once FETCH_LEAD
            // tiles of this one are left to issue (at once for an empty one)
            const bool signals = !SPLIT && kprod && rank == 0;
            const int t_signal = max(gr.t_lo, gr.t_hi - FETCH_LEAD);
            if (n == 0) {
                if (signals && lane == 0) mbar_arrive(ptake);
                continue;
            }
            // cache rows of the group's 16-key pages, 32 pages (8 tiles) per window:
            // lane l holds page l of the current window as a row index, and the
            // block id (loaded 8 tiles ahead) and row-in-block of the next window
            constexpr int WIN_TILES = 32 / (KT / 16);
            int nxt_blk = 0, nxt_off = 0;
            auto load_window = [&](int w) {
                const int tk = (gr.t_lo * (KT / 16) + w * 32 + lane) * 16;
                nxt_blk = (tk < gr.L) ? __ldg(p.table + (int64_t)gr.b * p.max_blocks + tk / p.bs) : 0;
                nxt_off = tk % p.bs;
            };
            auto row_of = [&]() -> int { return (nxt_blk * p.Hkv + gr.g) * p.bs + nxt_off; };
            int win_y = y0;  // cluster schedule: resolved by the fetch warp
            if (SPLIT && gr.t_lo < gr.t_hi) {
                if (pf_k == (int)k) {  // loaded while the previous piece streamed
                    nxt_blk = pf_blk;
                    nxt_off = ((gr.t_lo * (KT / 16) + lane) * 16) % p.bs;
                } else {
                    load_window(0);
                }
                win_y = row_of();
            }
            if (SPLIT && (int)k + 1 < *n_items) {
                const int4 nx = items[k + 1];
                if (!(nx.x & GROUP_BAD)) {
                    const int gi = nx.x;
                    const int nb_ = group_seq(p, nullptr, gi);
                    const int tk = (nx.y * (KT / 16) + lane) * 16;
                    pf_blk = (tk < lens[nb_] + cnts[nb_])
                                 ? __ldg(p.table + (int64_t)nb_ * p.max_blocks + tk / p.bs)
                                 : 0;
                    pf_k = (int)k + 1;
                }
            }
            if (gr.t_lo + WIN_TILES < gr.t_hi) load_window(1);
            for (int t = gr.t_lo; t < gr.t_hi; ++t, ++gt) {
                const int s = gt % nst;
                const uint32_t ph = (gt / nst) & 1u;
                bool freed = !*(volatile int*)&flags[0];
                if (lane == 0 && freed) freed = mbar_wait(&kempty[s], ph ^ 1u);
                freed = __shfl_sync(0xffffffffu, freed, 0);
                if (!freed) {
                    if (lane == 0) {
                        flags[0] = 1;
                        p.status[gr.b] = TV_ERR_TIMEOUT;
                    }
                    alive = false;
                    break;
                }
                if (signals && t == t_signal && lane == 0) mbar_arrive(ptake);
                const int t0 = t * KT;
                const int nv = min(KT, gr.L - t0);
                const int pages = (nv + 15) >> 4;
                const int mine = max(0, min(KT / 32, pages - pg0));  // this warp's pages
                const uint32_t bytes = (uint32_t)mine * 16u * D * 2u * 2u;
                uint64_t* bar = &kfull[s];
                uint8_t* kt = smem + OFF_RING + s * 2 * TILE_BYTES;
                uint8_t* vt = kt + TILE_BYTES;
                // the window holds every page's cache row.  One elected lane posts the
                // byte count, then lanes 0-3 issue the warp's four copies at once: lane
                // 2 jj + c copies page pg0 + jj of K (c = 0) or V (c = 1), one box each
                mbar_arrive_expect_tx_relaxed_elect(bar, bytes);
                {
                    const int jj = lane >> 1, c = lane & 1;
                    const int j = pg0 + jj;
                    const int y = __shfl_sync(0xffffffffu, win_y,
                                              ((t - gr.t_lo) % WIN_TILES) * (KT / 16) + j);
                    if (lane < 2 * (KT / 32) && j < pages) {
                        if (c == 0) tma_load_4d_hint(kt + j * 4096, &kmap, bar, 0, 0, 0, y >> 3, policy);
                        else tma_load_3d_hint(vt + j * 4096, &vmap, bar, 0, y, 0, policy);
                    }
                    __syncwarp();
                }
                if ((t - gr.t_lo) % WIN_TILES == WIN_TILES - 1 && t + 1 < gr.t_hi) {
                    const int w = (t - gr.t_lo) / WIN_TILES + 1;   // window of tile t + 1
                    win_y = row_of();
                    if (gr.t_lo + (w + 1) * WIN_TILES < gr.t_hi) load_window(w + 1);
                }
            }
        }
    } else if (warp == 1) {
        // ===================== S issuer: S = Q K^T per tile =====================
        uint32_t gt = 0, qi = 0;
        const uint32_t tS = tmem;
        const uint64_t qpol = l2_policy_evict_normal();
        if (lane == 0) tma_prefetch_desc(&qmap);
        bool alive = true;
        for (uint32_t k = 0; alive; ++k) {
            const Item it = take_item(k, nullptr);
            if ((it.word & (GROUP_BAD - 1)) >= p.groups) break;
            const Group gr = decode_group<SPLIT>(p, order, lens, cnts, cum, it, rank, cs);
            const int n = gr.t_hi - gr.t_lo;
            if (n == 0) continue;
            // Q tile (npt nodes x G heads x 128 columns) of this group, loaded here
            // once the previous group's S products are done with the buffer, so
            // the K/V producers never wait for it
            if (!wait_all(qempty, (qi & 1u) ^ 1u)) { alive = false; break; }
            {
                const uint32_t qbytes = 2u * 64u * (uint32_t)(p.G * p.npt) * 2u;
                const int node0 = gr.b * p.N + gr.qt * p.npt;
                mbar_arrive_expect_tx_elect(qfull, qbytes);
                for (int hf = 0; hf < 2; ++hf)
                    tma_load_3d_elect(smem + OFF_Q + hf * (128 * 128), &qmap, qfull, hf * 64,
                                      gr.g * p.G, node0, qpol);
            }
            if (!wait_all(qfull, qi & 1u)) { alive = false; break; }
            ++qi;
            for (int j = 0; j < n; ++j, ++gt) {
                const int s = gt % nst, sb = gt & 1;
                if (!wait_all(&kfull[s], (gt / nst) & 1u) ||
                    !wait_all(&sfree[sb], ((gt >> 1) & 1u) ^ 1u)) {
                    alive = false;
                    break;
                }
                tc_fence_after();
                const uint32_t qa = sbase + OFF_Q;
                const uint32_t ka = sbase + OFF_RING + s * 2 * TILE_BYTES;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t ad = smem_desc_sw128(qa + (kk >> 2) * (128 * 128) + (kk & 3) * 32, 16, 1024);
                    // K is [page][row group][half][8 rows][128 bytes]: the 8-key groups
                    // of the tile are 2 KB apart, the halves 1 KB
                    const uint64_t bd = smem_desc_sw128(ka + (kk >> 2) * 1024 + (kk & 3) * 32, 16, 2048);
                    tc_mma_bf16_elect(tS + sb * KT, ad, bd, IDESC_QK, kk > 0 ? 1u : 0u);
                }
                tc_commit_elect(&sfull[sb]);
                if (j == n - 1) tc_commit_elect(qempty);
                __syncwarp();
            }
        }
        if (!alive && lane == 0) flags[0] = 1;
    } else if (warp == 3) {
        // ============ PV issuer: O += P V per tile, in tile order ============
        // (its own warp, so PV products never queue behind a wait for K data)
        uint32_t gt = 0, og = 0;
        const uint32_t tO = tmem + TMEM_O;
        bool alive = true;
        for (uint32_t k = 0; alive; ++k) {
            const Item it = take_item(k, nullptr);
            if ((it.word & (GROUP_BAD - 1)) >= p.groups) break;
            const Group gr = decode_group<SPLIT>(p, order, lens, cnts, cum, it, rank, cs);
            const int n = gr.t_hi - gr.t_lo;
            if (n == 0) continue;
            for (int j = 0; j < n; ++j, ++gt) {
                const int pb = gt & 1, s = gt % nst;
                const int nv = min(KT, gr.L - (gr.t_lo + j) * KT);
                if (nv < KT) {
                    // the group's last tile: V rows past the sequence end may hold
                    // anything (NaN times a zero weight is NaN), so zero them as soon
                    // as the tile has landed, while the softmax still works on it
                    if (!wait_all(&kfull[s], (gt / nst) & 1u)) {
                        alive = false;
                        break;
                    }
                    uint8_t* vt = smem + OFF_RING + s * 2 * TILE_BYTES + TILE_BYTES;
                    // V is [page][half][16 rows][128 bytes]: one (row, half) per lane
                    for (int e = lane; e < 2 * (KT - nv); e += 32) {
                        const int r = nv + (e >> 1);
                        uint4* dst = reinterpret_cast<uint4*>(vt + (r >> 4) * 4096 + (e & 1) * 2048 +
                                                              (r & 15) * 128);
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch) dst[ch] = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();  // the tensor core reads V through the async proxy
                    __syncwarp();
                }
                if (!wait_all(&pfull[pb], (gt >> 1) & 1u) ||
                    (j == 0 && og > 0 && !wait_all(ofree, (og - 1) & 1u))) {
                    alive = false;
                    break;
                }
                tc_fence_after();
                const uint32_t pa = tmem + TMEM_P + pb * (KT / 2);
                const uint32_t va = sbase + OFF_RING + s * 2 * TILE_BYTES + TILE_BYTES;
#pragma unroll
                for (int kk = 0; kk < KT / 16; ++kk) {
                    const uint64_t bd = smem_desc_sw128(va + kk * 4096, 2048, 1024);
                    tc_mma_bf16_ts_elect(tO, pa + kk * 8, bd, IDESC_PV, (j == 0 && kk == 0) ? 0u : 1u);
                }
                tc_commit_elect(&kempty[s]);
                tc_commit_elect(&pfree[pb]);
                __syncwarp();
            }
            if (!alive) break;
            ++og;
        }
        if (!alive && lane == 0) flags[0] = 1;
    } else if (warp == FETCH_WARP) {
        // ===== work items (cluster schedule): one group ahead of the producers =====
        if (!SPLIT && rank == 0) {
            for (uint32_t k = 0;; ++k) {
                if (k > 0 && !__all_sync(0xffffffffu, mbar_wait_sleep(ptake, (k - 1) & 1u))) break;
                if (fetch_item(k) >= p.groups) break;
            }
        }
    } else {
        // ======================== softmax (warps 4-7) ========================
        const int row = tid - SOFTMAX_WARP0 * 32;           // tensor-memory lane
        const uint32_t lane_off = (uint32_t)(32 * (warp - SOFTMAX_WARP0)) << 16;
        const uint32_t tS = tmem + lane_off, tO = tmem + lane_off + TMEM_O;
        uint8_t* xo = smem + OFF_XO;
        float2* xml = reinterpret_cast<float2*>(smem + OFF_XML);
        float* wts = reinterpret_cast<float*>(smem + OFF_WTS);
        uint32_t gt = 0, merges = 0;
        bool alive = true;
        // waits until the PV product of tile t (and so every earlier one) is complete:
        // that is phase t / 2 of pfree[t & 1].  Called only while P(t + 2) is not yet
        // published, so the barrier cannot have moved a second phase past it.
        auto wait_pv = [&](uint32_t t) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(&pfree[t & 1u], (t >> 1) & 1u));
        };
        for (uint32_t k = 0;; ++k) {
            const Item it = take_item(k, nullptr);
            if ((it.word & (GROUP_BAD - 1)) >= p.groups) break;
            const Group gr = decode_group<SPLIT>(p, order, lens, cnts, cum, it, rank, cs);
            if (rank == 0 && row == 0 && gr.g == 0 && gr.qt == 0)
                p.status[gr.b] = gr.ok ? TV_OK : TV_ERR_OUT_OF_RANGE;
            const int n = gr.t_hi - gr.t_lo;
            const int node_l = row / p.G, head = row % p.G;
            const int node = gr.qt * p.npt + node_l;
            const bool valid = (node_l < p.npt) && (node < gr.n);  // absent nodes: no output
            // the node's ancestor bits (bits at or above N are never used: the
            // visibility word is cut at the sequence end); loaded now, first
            // needed by the group's last key tile
            const uint64_t mk = valid ? ldg_nc_u64_early(p.mask + (int64_t)gr.b * p.N + node) : 0ull;
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; j < n && alive; ++j, ++gt) {
                const int sb = gt & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(&sfull[sb], (gt >> 1) & 1u))) {
                    alive = false;
                    break;
                }
                tc_fence_after();
                float sv[KT];
                {
                    uint32_t r[32], r2[32];
                    tmem_ld32(tS + sb * KT, r);
                    tmem_ld32(tS + sb * KT + 32, r2);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        sv[c] = __uint_as_float(r[c]);
                        sv[32 + c] = __uint_as_float(r2[c]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_relaxed(&sfree[sb]);
                const int t0 = (gr.t_lo + j) * KT;
                if (t0 + KT > gr.P) {
                    // visible keys of this tile as one word: bit c for key t0 + c, the
                    // prefix (t < P) and the node's ancestors (t = P + a, bit a of mk)
                    const int sh = gr.P - t0;  // tile bit of the first tree key, > -N
                    const uint64_t pre = (sh >= KT) ? ~0ull : (sh <= 0 ? 0ull : (1ull << sh) - 1ull);
                    const uint64_t tree = (sh >= KT) ? 0ull : (sh >= 0 ? mk << sh : mk >> -sh);
                    const int in_seq = gr.L - t0;  // keys t < L: bit a of mk only for a < N
                    const uint64_t seq = (in_seq >= KT) ? ~0ull : (1ull << in_seq) - 1ull;
                    const uint64_t vis = pre | (tree & seq);
#pragma unroll
                    for (int c = 0; c < KT; ++c) sv[c] = ((vis >> c) & 1ull) ? sv[c] : -INFINITY;
                }
                const float csc = p.scale_log2;
                // row maximum of the raw scores (four chains of three-input maxima); the
                // scale is folded into the exponent, so the scaled maximum is tmax * csc
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < KT; c += 8)
#pragma unroll
                    for (int i = 0; i < 4; ++i) mx[i] = fmax3(mx[i], sv[c + i], sv[c + 4 + i]);
                const float tmax = fmaxf(fmax3(mx[0], mx[1], mx[2]), mx[3]) * csc;
                // The running max m_used is raised only when a score passes it by more
                // than 2^8 (or a row has none yet); a warp with such a row rescales O.
                const bool need = (m_used == -INFINITY) ? (tmax > -INFINITY)
                                                        : (tmax > m_used + RESCALE_LOG2);
                if (__any_sync(0xffffffffu, need)) {
                    const float f = (need && m_used > -INFINITY) ? exp2f(m_used - tmax) : 1.f;
                    if (j > 0) {
                        // O holds the products of earlier tiles: rescale it once they are done
                        if (!wait_pv(gt - 1)) {
                            alive = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int c = 0; c < D; c += 32) {
                            uint32_t r[32];
                            tmem_ld32(tO + c, r);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f);
                            tmem_st32(tO + c, r);
                        }
                        tmem_wait_st();
                    }
                    l *= f;
                    if (need) m_used = tmax;
                }
                // P = 2^(s * csc - m_used), two keys per packed fp32 pair instruction
                const float nbase = (m_used == -INFINITY) ? 0.f : -m_used;
                const uint64_t sc2 = f2_pack(csc, csc), nb2 = f2_pack(nbase, nbase);
                uint32_t pk[KT / 2];
                uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};  // packed (0.f, 0.f)
#pragma unroll
                for (int c = 0; c < KT; c += 2) {
                    float xa, xb;
                    f2_unpack(f2_fma(f2_pack(sv[c], sv[c + 1]), sc2, nb2), xa, xb);
                    const float a = ex2_approx(xa);
                    const float b2 = ex2_approx(xb);
                    acc[(c >> 1) & 3] = f2_add(acc[(c >> 1) & 3], f2_pack(a, b2));
                    pk[c / 2] = pack_bf16x2(a, b2);
                }
                {
                    float lo, hi;
                    f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), lo, hi);
                    l += lo + hi;
                }
                // P row -> tensor memory (this thread's lane) once its buffer is free
                const int pb = gt & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(&pfree[pb], ((gt >> 1) & 1u) ^ 1u))) {
                    alive = false;
                    break;
                }
                tmem_st32(tmem + lane_off + TMEM_P + pb * (KT / 2), pk);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_relaxed(&pfull[pb]);
            }
            if (!alive) break;
            // ---- epilogue: O / l
            float o_inv = (l > 0.f) ? 1.f / l : 0.f;
            __nv_bfloat16* orow = nullptr;
            if (valid)
                orow = p.out + (((int64_t)gr.b * p.N + node) * p.Hq + gr.g * p.G + head) * D;
            // balanced split, a piece of a group: its slot (the first piece of this
            // run if the group began in an earlier run, else the last)
            const bool spiece = SPLIT && !gr.whole;
            uint8_t* pbase = nullptr;
            if (spiece) {
                const int64_t w = (cum[gr.b + 1] - cum[gr.b]) / p.Hkv;
                const int64_t F = cum[gr.b] + (int64_t)gr.g * w + p.c0;  // first tile unit
                const int64_t lane_me = blockIdx.x / p.QT;
                const int64_t slot = 2 * (int64_t)blockIdx.x + (F < run_start(lane_me, U, L) ? 0 : 1);
                pbase = p.part + slot * SLOT_BYTES;
            }
            if (cs > 1 && merges > 0 &&
                !__all_sync(0xffffffffu, mbar_wait_cluster(xfree, (merges - 1) & 1u))) {
                alive = false;
                break;
            }
            if (n > 0) {
                if (!wait_pv(gt - 1)) {
                    alive = false;
                    break;
                }
                tc_fence_after();
            }
#pragma unroll
            for (int c = 0; c < D; c += 32) {
                uint32_t r[32];
                if (n > 0) {
                    tmem_ld32(tO + c, r);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = 0u;
                }
                if (gr.whole) {
                    if (valid) {
#pragma unroll
                        for (int e = 0; e < 32; e += 8) {
                            uint4 v;
                            v.x = pack_bf16x2(__uint_as_float(r[e]) * o_inv, __uint_as_float(r[e + 1]) * o_inv);
                            v.y = pack_bf16x2(__uint_as_float(r[e + 2]) * o_inv, __uint_as_float(r[e + 3]) * o_inv);
                            v.z = pack_bf16x2(__uint_as_float(r[e + 4]) * o_inv, __uint_as_float(r[e + 5]) * o_inv);
                            v.w = pack_bf16x2(__uint_as_float(r[e + 6]) * o_inv, __uint_as_float(r[e + 7]) * o_inv);
                            *reinterpret_cast<uint4*>(orow + c + e) = v;
                        }
                    }
                } else {
                    // normalised row, fp16, into this CTA's exchange buffer (16-byte chunks)
                    // or, for a balanced-split piece, into its workspace slot
                    uint8_t* xr = spiece ? pbase + row * (D * 2) : xo + row * (D * 2);
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        __half2 h0 = __floats2half2_rn(__uint_as_float(r[e]) * o_inv, __uint_as_float(r[e + 1]) * o_inv);
                        __half2 h1 = __floats2half2_rn(__uint_as_float(r[e + 2]) * o_inv, __uint_as_float(r[e + 3]) * o_inv);
                        __half2 h2 = __floats2half2_rn(__uint_as_float(r[e + 4]) * o_inv, __uint_as_float(r[e + 5]) * o_inv);
                        __half2 h3 = __floats2half2_rn(__uint_as_float(r[e + 6]) * o_inv, __uint_as_float(r[e + 7]) * o_inv);
                        uint4 v;
                        v.x = *reinterpret_cast<uint32_t*>(&h0);
                        v.y = *reinterpret_cast<uint32_t*>(&h1);
                        v.z = *reinterpret_cast<uint32_t*>(&h2);
                        v.w = *reinterpret_cast<uint32_t*>(&h3);
                        *reinterpret_cast<uint4*>(xr + (c + e) * 2) = v;
                    }
                }
            }
            if (n > 0) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_relaxed(ofree);  // O may be overwritten by the next group
            }
            if (gr.whole) continue;
            if (spiece) {
                // balanced split: the piece is complete; the merge kernel that follows
                // combines the group's pieces
                reinterpret_cast<float2*>(pbase + SLOT_O_BYTES)[row] = make_float2(m_used, l);
                continue;
            }
            // ---- cluster merge: this CTA finishes rows [rank*128/cs, (rank+1)*128/cs)
            xml[row] = make_float2(m_used, l);
            asm volatile("fence.acq_rel.cluster;" ::: "memory");
            named_bar_sync(2, 128);
            if (lane == 0)
                for (uint32_t r = 0; r < cs; ++r) remote_arrive(xready, r);
            if (!__all_sync(0xffffffffu, mbar_wait_cluster(xready, merges & 1u))) {
                alive = false;
                break;
            }
            const int rows_per = 128 / (int)cs;
            const int rb = (int)rank * rows_per;
            if (row < rows_per) {
                // every rank's (max, sum) of this row, all loads in flight at once
                const int lr = rb + row;
                float2 ml[MAX_CS];
#pragma unroll
                for (int c = 0; c < MAX_CS; ++c)
                    ml[c] = (c < (int)cs) ? remote_ld_f2(reinterpret_cast<const float*>(&xml[lr]), c)
                                          : make_float2(-INFINITY, 0.f);
                float mx = -INFINITY;
#pragma unroll
                for (int c = 0; c < MAX_CS; ++c) mx = fmaxf(mx, ml[c].x);
                const float bz = (mx == -INFINITY) ? 0.f : mx;
                float w[MAX_CS];
                float den = 0.f;
#pragma unroll
                for (int c = 0; c < MAX_CS; ++c) {
                    w[c] = (c < (int)cs) ? exp2f(ml[c].x - bz) * ml[c].y : 0.f;
                    den += w[c];
                }
                const float inv = (den > 0.f) ? 1.f / den : 0.f;
#pragma unroll
                for (int c = 0; c < MAX_CS; ++c)
                    if (c < (int)cs) wts[lr * MAX_CS + c] = w[c] * inv;
            }
            named_bar_sync(2, 128);
            for (int e = row; e < rows_per * (D / 8); e += 128) {
                const int lr = rb + e / (D / 8);
                const int c8 = (e % (D / 8)) * 8;
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                uint4 xv[MAX_CS];
#pragma unroll
                for (int c = 0; c < MAX_CS; ++c)  // every rank's 16 bytes in flight at once
                    xv[c] = (c < (int)cs) ? remote_ld_u4(xo + lr * (D * 2) + c8 * 2, c)
                                          : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int c = 0; c < MAX_CS; ++c) {
                    if (c >= (int)cs) break;
                    const float w = wts[lr * MAX_CS + c];
                    const __half2* h = reinterpret_cast<const __half2*>(&xv[c]);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 f2 = __half22float2(h[q]);
                        acc[2 * q] += w * f2.x;
                        acc[2 * q + 1] += w * f2.y;
                    }
                }
                const int nl = lr / p.G, hd = lr % p.G;
                const int nd = gr.qt * p.npt + nl;
                if (nl < p.npt && nd < gr.n) {
                    __nv_bfloat16* dst = p.out + (((int64_t)gr.b * p.N + nd) * p.Hq + gr.g * p.G + hd) * D + c8;
                    uint4 v;
                    v.x = pack_bf16x2(acc[0], acc[1]);
                    v.y = pack_bf16x2(acc[2], acc[3]);
                    v.z = pack_bf16x2(acc[4], acc[5]);
                    v.w = pack_bf16x2(acc[6], acc[7]);
                    *reinterpret_cast<uint4*>(dst) = v;
                }
            }
            __syncwarp();
            if (lane == 0)
                for (uint32_t r = 0; r < cs; ++r) remote_arrive(xfree, r);
            ++merges;
        }
        if (!alive && lane == 0) {
            flags[0] = 1;
        }
        if (cs > 1 && merges > 0) mbar_wait_cluster(xfree, (merges - 1) & 1u);
        __syncwarp();
    }
    // every role meets here once done
    tc_fence_before();
    cluster_barrier_all();
    tc_fence_after();
    if (warp == 2) tmem_dealloc(tmem, TMEM_COLS);
    if (tid == 0) {
        __threadfence();
        const int done = atomicAdd(&p.sched[1], 1);
        if (done == (int)gridDim.x - 1) {
            p.sched[0] = 0;
            p.sched[1] = 0;
        }
    }
}


// Balanced split, second kernel: one CTA per (run boundary l = 1 .. L-1, row
// tile).  The boundary at run_start(l) cuts at most one group's key tiles; the
// CTA of the first boundary inside a group merges all of the group's pieces,
// row by row: weights 2^(m_k - max) l_k / (sum over the pieces) on their
// normalised partial outputs.
constexpr int MERGE_THREADS = 256;
constexpr int MERGE_MW = 16;  // pieces whose weights sit in shared memory

__global__ void __launch_bounds__(MERGE_THREADS)
attn_split_merge_kernel(Params p) {
    __shared__ int64_t cum[LPT_MAX + 1];
    __shared__ int lens[LPT_MAX];
    __shared__ int cnts[LPT_MAX];
    __shared__ float2 nz[128];                // per row: max, 1 / weighted sum
    __shared__ float pw[MERGE_MW][128];       // weights of the first MERGE_MW pieces
    __shared__ int pslot[MERGE_MW];
    pdl_launch_dependents();
    split_prefix(p, cum, lens, cnts);  // from the call's inputs: overlaps the attention kernel
    const int tid = threadIdx.x;
    const int64_t U = cum[p.B];
    const int64_t L = min((int64_t)p.lanes, U);
    const int64_t l = blockIdx.x / p.QT + 1;
    const int qt = (int)(blockIdx.x % p.QT);
    // every path waits for the attention grid before it ends: under programmatic
    // dependent launch the next kernel waits only for this grid
    if (l >= L) {
        pdl_wait();
        return;
    }
    const int64_t x = run_start(l, U, L);
    int b = 0, hi = p.B;  // cum[b] <= x < cum[hi]
    while (hi - b > 1) {
        const int mid = (b + hi) >> 1;
        if (cum[mid] <= x) b = mid;
        else hi = mid;
    }
    const int64_t w = (cum[b + 1] - cum[b]) / p.Hkv;
    const int64_t g0 = x - (x - cum[b]) % w;
    const int64_t F = g0 + p.c0, tb = w - p.c0;  // the group's first tile unit, tiles
    if (x <= F || run_start(l - 1, U, L) > F) {  // not cut here first
        pdl_wait();
        return;
    }
    const int g = (int)((g0 - cum[b]) / w);
    const int64_t l1 = run_owner(F + tb - 1, U, L);
    const int pieces = (int)(l1 - (l - 1) + 1);
    auto slot_of = [&](int k) -> int64_t {
        const int64_t ln = l - 1 + k;
        return 2 * (ln * p.QT + qt) + (F < run_start(ln, U, L) ? 0 : 1);
    };
    for (int k = tid; k < pieces && k < MERGE_MW; k += MERGE_THREADS) pslot[k] = (int)slot_of(k);
    pdl_wait();  // the attention kernel's partial results are complete
    __syncthreads();
    const uint8_t* part = p.part;
    auto slot_k = [&](int k) -> int64_t { return (k < MERGE_MW) ? pslot[k] : slot_of(k); };
    auto ml_of = [&](int k, int r) -> float2 {
        return __ldcg(reinterpret_cast<const float2*>(part + slot_k(k) * SLOT_BYTES + SLOT_O_BYTES) + r);
    };
    if (tid < 128) {
        // row tid: max over the pieces, then the pieces' weights
        const int r = tid;
        float2 m8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) m8[u] = (u < pieces) ? ml_of(u, r) : make_float2(-INFINITY, 0.f);
        float mx = -INFINITY;
#pragma unroll
        for (int u = 0; u < 8; ++u) mx = fmaxf(mx, m8[u].x);
        for (int k = 8; k < pieces; ++k) mx = fmaxf(mx, ml_of(k, r).x);
        const float bz = (mx == -INFINITY) ? 0.f : mx;
        float e8[8], den = 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            e8[u] = exp2f(m8[u].x - bz) * m8[u].y;
            den += e8[u];
        }
        for (int k = 8; k < pieces; ++k) {
            const float2 ml = ml_of(k, r);
            den += exp2f(ml.x - bz) * ml.y;
        }
        const float inv = (den > 0.f) ? 1.f / den : 0.f;
        nz[r] = make_float2(bz, inv);
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (u < pieces) pw[u][r] = e8[u] * inv;
        for (int k = 8; k < pieces && k < MERGE_MW; ++k) {
            const float2 ml = ml_of(k, r);
            pw[k][r] = exp2f(ml.x - bz) * ml.y * inv;
        }
    }
    __syncthreads();
    // 16-byte chunks of the 128 x D output tile: thread t takes t + 256 i (i < 8),
    // with two pieces' loads of all eight chunks in flight together
    constexpr int CH = 128 * (D / 8) / MERGE_THREADS;
    constexpr int KB = 2;
    int lr[CH], c8[CH];
    bool ok[CH];
#pragma unroll
    for (int v = 0; v < CH; ++v) {
        const int e = tid + MERGE_THREADS * v;
        lr[v] = e / (D / 8);
        c8[v] = (e % (D / 8)) * 8;
        const int nl = lr[v] / p.G;
        // rows of present nodes (a bad sequence: every row, zeros)
        const int nb_ = seq_shape_ok(p, lens[b], cnts[b]) ? cnts[b] : p.N;
        ok[v] = nl < p.npt && qt * p.npt + nl < nb_;
    }
    float acc[CH][8];
#pragma unroll
    for (int v = 0; v < CH; ++v)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[v][q] = 0.f;
    for (int k0 = 0; k0 < pieces; k0 += KB) {
        uint4 xv[KB][CH];
#pragma unroll
        for (int u = 0; u < KB; ++u) {
            const int k = k0 + u;
            const uint8_t* sb = (k < pieces) ? part + slot_k(k) * SLOT_BYTES : nullptr;
#pragma unroll
            for (int v = 0; v < CH; ++v)
                xv[u][v] = (sb && ok[v]) ? __ldcg(reinterpret_cast<const uint4*>(sb + lr[v] * (D * 2) + c8[v] * 2))
                                         : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < KB; ++u) {
            const int k = k0 + u;
            if (k >= pieces) break;
#pragma unroll
            for (int v = 0; v < CH; ++v) {
                float wt;
                if (k < MERGE_MW) {
                    wt = pw[k][lr[v]];
                } else {
                    const float2 ml = ml_of(k, lr[v]);
                    wt = exp2f(ml.x - nz[lr[v]].x) * ml.y * nz[lr[v]].y;
                }
                const __half2* h = reinterpret_cast<const __half2*>(&xv[u][v]);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 f2 = __half22float2(h[q]);
                    acc[v][2 * q] += wt * f2.x;
                    acc[v][2 * q + 1] += wt * f2.y;
                }
            }
        }
    }
#pragma unroll
    for (int v = 0; v < CH; ++v) {
        if (!ok[v]) continue;
        const int nl = lr[v] / p.G, hd = lr[v] % p.G;
        const int nd = qt * p.npt + nl;
        __nv_bfloat16* dst = p.out + (((int64_t)b * p.N + nd) * p.Hq + g * p.G + hd) * D + c8[v];
        uint4 o;
        o.x = pack_bf16x2(acc[v][0], acc[v][1]);
        o.y = pack_bf16x2(acc[v][2], acc[v][3]);
        o.z = pack_bf16x2(acc[v][4], acc[v][5]);
        o.w = pack_bf16x2(acc[v][6], acc[v][7]);
        *reinterpret_cast<uint4*>(dst) = o;
    }
}

// ---------------------------------------------------------------- host side
// Both instantiations may use SMEM_BYTES of dynamic shared memory; set before
// any launch or occupancy query (a query without it finds no room).
bool tc_attrs_set() {
    static bool done = false;
    if (!done) {
        if (cudaFuncSetAttribute(attn_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(attn_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_BYTES) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        done = true;
    }
    return true;
}

int resident_clusters_tc(int cs) {
    static int cache[9] = {-1, -1, -1, -1, -1, -1, -1, -1, -1};
    if (cs < 1 || cs > 8) return 0;
    if (cache[cs] >= 0) return cache[cs];
    if (!tc_attrs_set()) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = cs;
    at.val.clusterDim.y = 1;
    at.val.clusterDim.z = 1;
    cfg.attrs = &at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, attn_tc_kernel<false>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;  // not cached: a later query may succeed
    }
    cache[cs] = n;
    return n;
}

}  // namespace

// Every head-size-128 shape.  Even a row tile of a few dozen rows (a chain of
// 6 nodes x 4 heads) is faster here, padded to 128 rows, than on the warp-MMA
// kernel: the tensor cores leave the tile loop bound by the K/V stream, while
// the warp-MMA kernel's per-tile chain of dependent steps bounds it well below
// that (llama3-8B b128 chain5: 274 against 331 us).
bool attn_tc_applicable(int N, int Hq, int Hkv, int d) {
    (void)N;
    const int G = Hq / Hkv;
    return d == D && G <= 128;
}

namespace {
constexpr size_t kSchedBytes = 256;  // group counter and exit counter, padded

int device_sms() {
    static int sms = 0;
    if (sms == 0) {
        int dev = 0, n = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
            sms = n;
        else
            cudaGetLastError();
    }
    return sms;
}
}  // namespace

// Workspace: scheduler counters (zero between calls), then two partial-result
// slots per CTA of a balanced-split grid (at most one CTA per SM).
size_t attn_tc_zeroed_prefix(int B, int N, int Hq, int Hkv) {
    (void)B; (void)N; (void)Hq; (void)Hkv;
    return kSchedBytes;
}
size_t attn_tc_workspace(int B, int N, int Hq, int Hkv) {
    return attn_tc_zeroed_prefix(B, N, Hq, Hkv) + (size_t)2 * device_sms() * SLOT_BYTES;
}

// The schedule a call takes: the balanced split (lanes CTAs per row tile) or 0
// for clusters.  Balanced split when the groups are too few to give every SM
// one (whole groups would leave SMs idle) but not so few that clusters split
// them better, the workspace holds the partial results and the sequence count
// fits the in-kernel prefix sum.  Otherwise groups go to clusters dynamically,
// longest first.
int tc_split_lanes(int B, int N, int Hq, int Hkv, size_t ws_bytes) {
    const int npt = 128 / (Hq / Hkv);
    const int QT = (N + npt - 1) / npt;
    const int64_t groups = (int64_t)B * Hkv * QT;
    const int ncta = resident_clusters_tc(1);
    const int lanes = ncta / QT;
    const size_t need = attn_tc_zeroed_prefix(B, N, Hq, Hkv) + (size_t)2 * lanes * QT * SLOT_BYTES;
    const char* env = getenv("TV_SPLIT");
    const bool want = env ? (env[0] != '0') : (groups < ncta && 2 * groups >= ncta);
    return (want && lanes >= 1 && B <= LPT_MAX && ws_bytes >= need) ? lanes : 0;
}

int attn_tc_kernels(int B, int N, int Hq, int Hkv, size_t ws_bytes) {
    const int lanes = tc_split_lanes(B, N, Hq, Hkv, ws_bytes);
    return lanes >= 2 ? 2 : 1;
}

tv_status launch_attn_tc(const AttnArgs& a) {
    if (!tc_attrs_set()) return TV_ERR_CUDA;
    const int G = a.Hq / a.Hkv;
    const int npt = 128 / G;
    const int64_t rows = (int64_t)a.num_blocks * a.Hkv * a.bs;
    if (rows >= (1LL << 31)) return TV_ERR_UNSUPPORTED;
    CUtensorMap qm, km, vm;
    if (!make_q_map(&qm, a.q, D, a.Hq, (int64_t)a.B * a.N, G, npt) ||
        !make_kpage_map(&km, a.k_cache, rows) || !make_page_map(&vm, a.v_cache, rows))
        return TV_ERR_CUDA;
    Params prm{};
    prm.table = a.block_table;
    prm.prefix_lens = a.prefix_lens;
    prm.mask = a.mask;
    prm.counts = a.counts;
    prm.out = static_cast<__nv_bfloat16*>(a.out);
    prm.status = a.status;
    prm.sched = static_cast<int32_t*>(a.ws);
    prm.max_blocks = a.max_blocks;
    prm.B = a.B;
    prm.N = a.N;
    prm.Hq = a.Hq;
    prm.Hkv = a.Hkv;
    prm.G = G;
    prm.npt = npt;
    prm.bs = a.bs;
    prm.num_blocks = a.num_blocks;
    prm.QT = (a.N + npt - 1) / npt;
    const int64_t groups = (int64_t)a.B * a.Hkv * prm.QT;
    if (groups >= (1LL << 30)) return TV_ERR_UNSUPPORTED;
    prm.groups = (int)groups;
    prm.scale_log2 = a.scale * LOG2E;
    {
        const int lanes = tc_split_lanes(a.B, a.N, a.Hq, a.Hkv, a.ws_bytes);
        if (lanes > 0) {
            const size_t zeroed = attn_tc_zeroed_prefix(a.B, a.N, a.Hq, a.Hkv);
            prm.lanes = lanes;
            const char* c0e = getenv("TV_SPLIT_C0");
            prm.c0 = c0e ? std::max(0, atoi(c0e)) : SPLIT_C0;
            prm.part = static_cast<uint8_t*>(a.ws) + zeroed;
            LaunchCfg lc(dim3((unsigned)(lanes * prm.QT)), dim3(THREADS), SMEM_BYTES, a.stream, 1u);
            if (cudaLaunchKernelEx(&lc.cfg, attn_tc_kernel<true>, qm, km, vm, prm) != cudaSuccess)
                return TV_ERR_CUDA;
            if (lanes < 2) return TV_OK;  // one run: nothing is cut
            LaunchCfg lm(dim3((unsigned)((lanes - 1) * prm.QT)), dim3(MERGE_THREADS), 0, a.stream, 1u);
            return cudaLaunchKernelEx(&lm.cfg, attn_split_merge_kernel, prm) == cudaSuccess
                       ? TV_OK
                       : TV_ERR_CUDA;
        }
    }
    // cluster size: minimise rounds x (tiles per CTA + one tile of merge cost)
    const int64_t tiles_max = ((int64_t)a.max_blocks * a.bs + KT - 1) / KT;
    int best_cs = 1, best_ncl = 0;
    double best = 1e300;
    for (int cs = 1; cs <= MAX_CS; cs *= 2) {
        if (cs > 1 && tiles_max < 2 * cs) break;
        const int ncl = resident_clusters_tc(cs);
        if (ncl <= 0) continue;
        const int64_t rounds = (groups + ncl - 1) / ncl;
        const double cost = (double)rounds * ((double)tiles_max / cs + (cs > 1 ? 1.0 : 0.0));
        if (cost < best * 0.97) {
            best = cost;
            best_cs = cs;
            best_ncl = ncl;
        }
    }
    if (best_ncl <= 0) return TV_ERR_CUDA;
    const int clusters = (int)std::min<int64_t>(best_ncl, groups);
    LaunchCfg lc(dim3((unsigned)(clusters * best_cs)), dim3(THREADS), SMEM_BYTES, a.stream,
                 (unsigned)best_cs);
    return cudaLaunchKernelEx(&lc.cfg, attn_tc_kernel<false>, qm, km, vm, prm) == cudaSuccess
               ? TV_OK
               : TV_ERR_CUDA;
}

}  // namespace tv
