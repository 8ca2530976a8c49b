// tree_verify_attention, bfloat16 path on warp-level MMA: head size 64 (head
// size 128 runs on the tensor-memory kernel, attn_tc.cu).
//
// Work decomposition
//   All query heads of one KV group times all tree nodes form one packed row
//   block: row r = node * G + head-in-group (G = Hq / Hkv), M = N * G rows,
//   cut into row tiles of QROWS rows.  A "group" is (sequence, kv head, row
//   tile).  Groups are handed out dynamically (a global atomic counter) to
//   thread-block clusters of CS CTAs, one CTA per SM; the CS CTAs of a
//   cluster split the group's KV range 0 .. P+N-1 into CS equal runs of
//   64-key tiles, and merge their partial softmax results through
//   distributed shared memory (no partials in global memory).  CS is chosen
//   on the host so that small batches still cover the GPU.
//
// CTA roles
//   warp 8 (producer): streams 64-key K and V tiles through a 4-stage shared
//   memory ring with 2-D TMA copies (one 16-key page = one 16 x 64-element
//   box per 64-column half, 128-byte swizzle), resolving pages through the
//   block table.  In the cluster's rank-0 CTA its lane 0 also fetches the
//   next group id and broadcasts it to every CTA of the cluster.
//   warps 0..7 (consumers): WM row warps (16 rows each) times WK key groups
//   (group k takes tiles k, k+WK, ...).  S = Q K^T and O += P V with
//   mma.sync m16n8k16 (bf16 in, fp32 accumulate), online softmax in
//   registers (base 2), tree mask on the tiles that reach the tree's own
//   positions.
#include <algorithm>

#include "tv_device.cuh"
#include "tv_internal.h"

namespace tv {

namespace {

constexpr int KT = 64;        // keys per tile
constexpr int STAGES = 4;     // TMA ring depth
constexpr int GQ = 4;         // group-id ring depth
constexpr int CONSUMER_WARPS = 8;
constexpr int THREADS = (CONSUMER_WARPS + 1) * 32;
constexpr int MAX_CS = 16;
constexpr float LOG2E = 1.4426950408889634f;

struct Params {
    const __nv_bfloat16* q;
    const int32_t* table;
    const int32_t* prefix_lens;
    const uint64_t* mask;
    const int32_t* counts;  // nullable: nodes per sequence (the first counts[b] of N)
    __nv_bfloat16* out;
    int32_t* status;
    int32_t* sched;      // [0] next group, [1] CTAs finished (both return to 0)
    int max_blocks, B, N, Hq, Hkv, G, M, bs, num_blocks;
    int QT, groups;
    float scale_log2;    // scale * log2(e)
};

template <int D>
struct Layout {
    static constexpr int TILE_BYTES = KT * D * 2;  // one K or V tile
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    static constexpr int XO_STRIDE = D + 4;        // floats per exchanged row (O, m, l, pad)
};

// Nodes of sequence b (its tree is the first n of the N node slots).
__device__ __forceinline__ int seq_nodes(const Params& p, int b) {
    return p.counts ? p.counts[b] : p.N;
}

// Validity of sequence b, evaluated by one warp: node count in [1, N], prefix
// length in range and every block id covering positions 0..P+n-1 inside the cache.
__device__ __forceinline__ bool seq_ok_warp(const Params& p, int b, int P) {
    const int lane = threadIdx.x & 31;
    const int n = seq_nodes(p, b);
    bool ok = P >= 0 && n >= 1 && n <= p.N && (int64_t)P + n <= (int64_t)p.max_blocks * p.bs;
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

struct Group {
    int b, g, qt, P, n, L, t_lo, t_hi;  // n nodes, L = P + n keys; this CTA's tiles [t_lo, t_hi)
    bool ok;
};

// Group ids travel with a validity bit: the fetching warp checks the group's
// sequence once (seq_ok_warp) and marks a bad one with GROUP_BAD.
constexpr int GROUP_BAD = 1 << 30;

__device__ __forceinline__ int group_seq(const Params& p, const int* order, int gi) {
    const int r = gi / (p.QT * p.Hkv);
    return order ? order[r] : r;
}

// Fetched word -> group: sequence (in longest-first order when `order` is
// given), kv head, row tile; this CTA's share of its key tiles.
__device__ __forceinline__ Group decode_group(const Params& p, const int* order, int word, int rank,
                                             int cs) {
    Group gr;
    const int gi = word & (GROUP_BAD - 1);
    gr.qt = gi % p.QT;
    gr.g = (gi / p.QT) % p.Hkv;
    gr.b = group_seq(p, order, gi);
    gr.P = p.prefix_lens[gr.b];
    gr.ok = (word & GROUP_BAD) == 0;
    gr.n = gr.ok ? seq_nodes(p, gr.b) : p.N;  // a bad sequence: every row gets zeros
    gr.L = gr.P + gr.n;
    const int T = gr.ok ? (gr.L + KT - 1) / KT : 0;
    gr.t_lo = (int)((int64_t)T * rank / cs);
    gr.t_hi = (int)((int64_t)T * (rank + 1) / cs);
    return gr;
}

template <int D, int WM, int WK>
__global__ void __launch_bounds__(THREADS, 1)
attn_bf16_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                 Params p) {
    static_assert(WM * WK == CONSUMER_WARPS, "consumer warp grid");
    constexpr int QROWS = WM * 16;
    constexpr int NT = D / 8;   // O n-tiles
    constexpr int KC = D / 16;  // k-chunks of the QK^T product
    using LY = Layout<D>;
    constexpr int XS = LY::XO_STRIDE;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* ring = smem;
    float* scratch = reinterpret_cast<float*>(smem + LY::RING_BYTES);  // WK merge
    constexpr int SCRATCH_FLOATS = (WK - 1) * QROWS * (D + 2);
    float* xo = scratch + SCRATCH_FLOATS;                               // cluster exchange
    float* wts = xo + QROWS * XS;                                       // [QROWS][MAX_CS]
    float* inv_den = wts + QROWS * MAX_CS;                              // [QROWS]
    uint64_t* bars = reinterpret_cast<uint64_t*>(inv_den + QROWS);
    uint64_t* full_bar = bars;
    uint64_t* empty_bar = bars + STAGES;
    uint64_t* tail_bar = bars + 2 * STAGES;
    uint64_t* gq_full = tail_bar + 1;
    uint64_t* gq_empty = gq_full + GQ;
    uint64_t* xready = gq_empty + GQ;
    uint64_t* xfree = xready + 1;
    int* gq = reinterpret_cast<int*>(xfree + 1);  // [GQ]
    int* flags = gq + GQ;                          // [0] abort
    int* lpt = flags + 4;                          // [2][LPT_MAX] sequence lengths, order

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_rank(), cs = cluster_size();

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], WM);
        }
        mbar_init(tail_bar, 1);
        for (int s = 0; s < GQ; ++s) {
            mbar_init(&gq_full[s], 1);
            mbar_init(&gq_empty[s], cs * (1 + CONSUMER_WARPS));
        }
        mbar_init(xready, cs * CONSUMER_WARPS);
        mbar_init(xfree, cs * CONSUMER_WARPS);
        flags[0] = 0;
        fence_mbar_init();
    }
    pdl_launch_dependents();
    // every CTA of the cluster has initialised its barriers before any remote arrive
    cluster_barrier_all();
    pdl_wait();  // everything above touched only shared memory
    const int* order = nullptr;
    if (p.B > 1 && p.B <= LPT_MAX) {
        lpt_order(p.prefix_lens, p.B, lpt, lpt + LPT_MAX);
        order = lpt + LPT_MAX;
    }

    if (warp == CONSUMER_WARPS) {
        // =========================== producer ===========================
        if (lane == 0) {
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
        }
        const uint64_t policy = (p.QT == 1) ? l2_policy_evict_first() : l2_policy_evict_normal();
        uint32_t gt = 0, tail_phase = 0;
        bool alive = true;
        for (uint32_t k = 0; alive; ++k) {
            const int slot = k % GQ;
            // rank 0 fetches the next group id and hands it to the whole cluster
            // (the producer warp also validates the group's sequence, once)
            if (rank == 0) {
                // the first group of every cluster is its cluster index; later ones
                // come from the counter, after the clusters' first groups
                int gi = p.groups;
                if (lane == 0 && mbar_wait_cluster(&gq_empty[slot], ((k / GQ) & 1u) ^ 1u))
                    gi = (k == 0) ? (int)(blockIdx.x / cs)
                                  : (int)(gridDim.x / cs) + atomicAdd(&p.sched[0], 1);
                gi = __shfl_sync(0xffffffffu, gi, 0);
                int word = gi;
                if (gi < p.groups) {
                    const int b = group_seq(p, order, gi);
                    if (!seq_ok_warp(p, b, p.prefix_lens[b])) word |= GROUP_BAD;
                }
                if (lane == 0) {
                    for (uint32_t r = 0; r < cs; ++r) {
                        remote_st_u32(&gq[slot], r, word);
                        remote_arrive(&gq_full[slot], r);
                    }
                }
            }
            // every lane acquires the slot written by rank 0 before reading it
            const bool got = __all_sync(0xffffffffu, mbar_wait_cluster(&gq_full[slot], (k / GQ) & 1u));
            const int gi = got ? *(volatile int*)&gq[slot] : p.groups;
            __syncwarp();
            if (lane == 0) remote_arrive(&gq_empty[slot], 0);
            if ((gi & (GROUP_BAD - 1)) >= p.groups) break;
            const Group gr = decode_group(p, order, gi, rank, cs);
            // block id of the page holding logical position tk (0 past the sequence end)
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
            int win_y = 0;
            if (gr.t_lo < gr.t_hi) {
                load_window(0);
                win_y = row_of();
            }
            if (gr.t_lo + WIN_TILES < gr.t_hi) load_window(1);
            for (int t = gr.t_lo; t < gr.t_hi; ++t, ++gt) {
                const int s = gt % STAGES;
                const uint32_t ph = (gt / STAGES) & 1u;
                bool freed = !*(volatile int*)&flags[0];
                if (lane == 0 && freed) freed = mbar_wait(&empty_bar[s], ph ^ 1u);
                freed = __shfl_sync(0xffffffffu, freed, 0);
                if (!freed) {
                    if (lane == 0) {
                        flags[0] = 1;
                        p.status[gr.b] = TV_ERR_TIMEOUT;
                    }
                    alive = false;
                    break;
                }
                const int t0 = t * KT;
                const int nv = min(KT, gr.L - t0);  // valid keys in this tile
                const int pages = (nv + 15) >> 4;
                const uint32_t bytes = (uint32_t)pages * 16u * D * 2u * 2u;
                const bool tail = nv < KT;
                uint64_t* bar = tail ? tail_bar : &full_bar[s];
                uint8_t* kt = ring + s * LY::STAGE_BYTES;
                uint8_t* vt = kt + LY::TILE_BYTES;
                // the window holds every page's cache row; the warp walks the pages with
                // that row broadcast and one elected lane issues the byte count and copies
                mbar_arrive_expect_tx_elect(bar, bytes);
#pragma unroll
                for (int j = 0; j < KT / 16; ++j) {
                    const int y = __shfl_sync(0xffffffffu, win_y,
                                              ((t - gr.t_lo) % WIN_TILES) * (KT / 16) + j);
                    if (j < pages) {
#pragma unroll
                        for (int hf = 0; hf < D / 64; ++hf) {
                            tma_load_2d_elect(kt + hf * (KT * 128) + j * 2048, &kmap, bar, hf * 64, y, policy);
                            tma_load_2d_elect(vt + hf * (KT * 128) + j * 2048, &vmap, bar, hf * 64, y, policy);
                        }
                    }
                }
                if ((t - gr.t_lo) % WIN_TILES == WIN_TILES - 1 && t + 1 < gr.t_hi) {
                    const int w = (t - gr.t_lo) / WIN_TILES + 1;   // window of tile t + 1
                    win_y = row_of();
                    if (gr.t_lo + (w + 1) * WIN_TILES < gr.t_hi) load_window(w + 1);
                }
                if (tail) {
                    // wait for the partial tile, zero the V rows past the sequence end
                    // (they may hold anything), then publish the stage
                    const bool landed = __all_sync(0xffffffffu, mbar_wait(tail_bar, tail_phase));
                    tail_phase ^= 1u;
                    if (!landed) {
                        if (lane == 0) {
                            flags[0] = 1;
                            p.status[gr.b] = TV_ERR_TIMEOUT;
                        }
                        alive = false;
                        break;
                    }
                    const int zrows = KT - nv;
                    for (int e = lane; e < (D / 64) * zrows * 8; e += 32) {
                        const int hf = e / (zrows * 8);
                        const int r = nv + (e / 8) % zrows;
                        const int ch = e % 8;
                        *reinterpret_cast<uint4*>(vt + hf * (KT * 128) + r * 128 + ch * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&full_bar[s]);
                }
            }
        }
    } else {
        // ============================= consumers =============================
        const int wm = warp % WM, wk = warp / WM;
        const int gq4 = lane >> 2, cq = lane & 3;
        const uint32_t ring_u32 = smem_u32(ring);
        uint32_t gt_base = 0, merges = 0;
        for (uint32_t k = 0;; ++k) {
            const int slot = k % GQ;
            const bool got = __all_sync(0xffffffffu, mbar_wait_cluster(&gq_full[slot], (k / GQ) & 1u));
            const int gi = got ? *(volatile int*)&gq[slot] : p.groups;
            __syncwarp();
            if (lane == 0) remote_arrive(&gq_empty[slot], 0);
            if ((gi & (GROUP_BAD - 1)) >= p.groups) break;
            const Group gr = decode_group(p, order, gi, rank, cs);
            if (rank == 0 && tid == 0 && gr.g == 0 && gr.qt == 0)
                p.status[gr.b] = gr.ok ? TV_OK : TV_ERR_OUT_OF_RANGE;
            const int ntiles = gr.t_hi - gr.t_lo;

            // rows of this thread within the packed block
            const int r0 = gr.qt * QROWS + wm * 16 + gq4, r1 = r0 + 8;
            const int m_rows = gr.n * p.G;  // rows of present nodes
            const bool v0 = r0 < m_rows, v1 = r1 < m_rows;
            const int i0 = v0 ? r0 / p.G : 0, i1 = v1 ? r1 / p.G : 0;
            const uint64_t nmask = (gr.n >= 64) ? ~0ull : ((1ull << gr.n) - 1);
            const uint64_t mk0 = v0 ? (p.mask[(int64_t)gr.b * p.N + i0] & nmask) : 0;
            const uint64_t mk1 = v1 ? (p.mask[(int64_t)gr.b * p.N + i1] & nmask) : 0;

            uint32_t qa[KC][4];
            {
                const __nv_bfloat16* q0 =
                    p.q + (((int64_t)gr.b * p.N + i0) * p.Hq + gr.g * p.G + (r0 % p.G)) * D;
                const __nv_bfloat16* q1 =
                    p.q + (((int64_t)gr.b * p.N + i1) * p.Hq + gr.g * p.G + (r1 % p.G)) * D;
#pragma unroll
                for (int kk = 0; kk < KC; ++kk) {
                    const int c0 = kk * 16 + 2 * cq;
                    qa[kk][0] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + c0) : 0u;
                    qa[kk][1] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + c0) : 0u;
                    qa[kk][2] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + c0 + 8) : 0u;
                    qa[kk][3] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + c0 + 8) : 0u;
                }
            }

            float o[NT][4];
#pragma unroll
            for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
            float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

            for (int lt = wk; lt < ntiles; lt += WK) {
                const uint32_t gtile = gt_base + lt;
                const int s = gtile % STAGES;
                const uint32_t ph = (gtile / STAGES) & 1u;
                bool ready = !*(volatile int*)&flags[0];
                ready = __all_sync(0xffffffffu, ready && mbar_wait(&full_bar[s], ph));
                if (!ready) {
                    if (lane == 0) {
                        flags[0] = 1;
                        p.status[gr.b] = TV_ERR_TIMEOUT;
                    }
                    break;
                }
                const uint32_t ku = ring_u32 + s * LY::STAGE_BYTES;
                const uint32_t vu = ku + LY::TILE_BYTES;
                const int t0 = (gr.t_lo + lt) * KT;

                // ---- S = Q K^T (16 rows x 64 keys per warp)
                float sc[8][4];
#pragma unroll
                for (int j = 0; j < 8; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
                for (int jp = 0; jp < 4; ++jp) {
                    const uint32_t key = jp * 16 + (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
                    for (int kk = 0; kk < KC; ++kk) {
                        const uint32_t dcol = kk * 16 + ((lane >> 3) & 1) * 8;
                        const uint32_t addr =
                            ku + (dcol >> 6) * (KT * 128) + sw128(key, (dcol & 63) >> 3);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(addr, b0, b1, b2, b3);
                        mma_bf16_16816(sc[2 * jp], qa[kk], b0, b1);
                        mma_bf16_16816(sc[2 * jp + 1], qa[kk], b2, b3);
                    }
                }
                // ---- scale, tree mask, online softmax
                const bool need_mask = (t0 + KT > gr.P);
                float tmax0 = -INFINITY, tmax1 = -INFINITY;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int t = t0 + j * 8 + 2 * cq + e;
                        float s0 = sc[j][e] * p.scale_log2, s1 = sc[j][2 + e] * p.scale_log2;
                        if (need_mask) {
                            const bool tree = t >= gr.P && t < gr.L;
                            const int a = t - gr.P;
                            const bool vis0 = (t < gr.P) || (tree && ((mk0 >> a) & 1ull));
                            const bool vis1 = (t < gr.P) || (tree && ((mk1 >> a) & 1ull));
                            s0 = vis0 ? s0 : -INFINITY;
                            s1 = vis1 ? s1 : -INFINITY;
                        }
                        sc[j][e] = s0;
                        sc[j][2 + e] = s1;
                        tmax0 = fmaxf(tmax0, s0);
                        tmax1 = fmaxf(tmax1, s1);
                    }
                }
#pragma unroll
                for (int off = 1; off <= 2; off <<= 1) {
                    tmax0 = fmaxf(tmax0, __shfl_xor_sync(0xffffffffu, tmax0, off));
                    tmax1 = fmaxf(tmax1, __shfl_xor_sync(0xffffffffu, tmax1, off));
                }
                const float mn0 = fmaxf(m0, tmax0), mn1 = fmaxf(m1, tmax1);
                const float base0 = (mn0 == -INFINITY) ? 0.f : mn0;
                const float base1 = (mn1 == -INFINITY) ? 0.f : mn1;
                const float corr0 = exp2f(m0 - base0), corr1 = exp2f(m1 - base1);
                m0 = mn0;
                m1 = mn1;
                float rs0 = 0.f, rs1 = 0.f;
                uint32_t pa[4][4];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float p00 = exp2f(sc[j][0] - base0), p01 = exp2f(sc[j][1] - base0);
                    const float p10 = exp2f(sc[j][2] - base1), p11 = exp2f(sc[j][3] - base1);
                    rs0 += p00 + p01;
                    rs1 += p10 + p11;
                    const int kk2 = j >> 1, hi = j & 1;
                    pa[kk2][hi * 2 + 0] = pack_bf16x2(p00, p01);
                    pa[kk2][hi * 2 + 1] = pack_bf16x2(p10, p11);
                }
                l0 = l0 * corr0 + rs0;
                l1 = l1 * corr1 + rs1;
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    o[j][0] *= corr0;
                    o[j][1] *= corr0;
                    o[j][2] *= corr1;
                    o[j][3] *= corr1;
                }
                // ---- O += P V
#pragma unroll
                for (int kk2 = 0; kk2 < 4; ++kk2) {
                    const uint32_t key = kk2 * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                    for (int jd = 0; jd < NT; jd += 2) {
                        const uint32_t dcol = jd * 8 + (lane >> 4) * 8;
                        const uint32_t addr =
                            vu + (dcol >> 6) * (KT * 128) + sw128(key, (dcol & 63) >> 3);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(addr, b0, b1, b2, b3);
                        mma_bf16_16816(o[jd], pa[kk2], b0, b1);
                        mma_bf16_16816(o[jd + 1], pa[kk2], b2, b3);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty_bar[s]);
            }
            gt_base += ntiles;

#pragma unroll
            for (int off = 1; off <= 2; off <<= 1) {
                l0 += __shfl_xor_sync(0xffffffffu, l0, off);
                l1 += __shfl_xor_sync(0xffffffffu, l1, off);
            }

            // ---- merge the WK key groups of this CTA into group 0
            const int lr0 = wm * 16 + gq4, lr1 = lr0 + 8;
            if (WK > 1) {
                if (wk > 0) {
                    float* sc0 = scratch + ((wk - 1) * QROWS + lr0) * (D + 2);
                    float* sc1 = scratch + ((wk - 1) * QROWS + lr1) * (D + 2);
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        const int c = j * 8 + 2 * cq;
                        sc0[c] = o[j][0];
                        sc0[c + 1] = o[j][1];
                        sc1[c] = o[j][2];
                        sc1[c + 1] = o[j][3];
                    }
                    if (cq == 0) {
                        sc0[D] = m0;
                        sc0[D + 1] = l0;
                        sc1[D] = m1;
                        sc1[D + 1] = l1;
                    }
                }
                named_bar_sync(1, CONSUMER_WARPS * 32);
                if (wk == 0) {
#pragma unroll
                    for (int kg = 1; kg < WK; ++kg) {
                        const float* sc0 = scratch + ((kg - 1) * QROWS + lr0) * (D + 2);
                        const float* sc1 = scratch + ((kg - 1) * QROWS + lr1) * (D + 2);
                        const float mk0v = sc0[D], lk0 = sc0[D + 1];
                        const float mk1v = sc1[D], lk1 = sc1[D + 1];
                        const float n0 = fmaxf(m0, mk0v), n1 = fmaxf(m1, mk1v);
                        const float bz0 = (n0 == -INFINITY) ? 0.f : n0;
                        const float bz1 = (n1 == -INFINITY) ? 0.f : n1;
                        const float a0 = exp2f(m0 - bz0), b0 = exp2f(mk0v - bz0);
                        const float a1 = exp2f(m1 - bz1), b1 = exp2f(mk1v - bz1);
#pragma unroll
                        for (int j = 0; j < NT; ++j) {
                            const int c = j * 8 + 2 * cq;
                            o[j][0] = o[j][0] * a0 + sc0[c] * b0;
                            o[j][1] = o[j][1] * a0 + sc0[c + 1] * b0;
                            o[j][2] = o[j][2] * a1 + sc1[c] * b1;
                            o[j][3] = o[j][3] * a1 + sc1[c + 1] * b1;
                        }
                        l0 = l0 * a0 + lk0 * b0;
                        l1 = l1 * a1 + lk1 * b1;
                        m0 = n0;
                        m1 = n1;
                    }
                }
                named_bar_sync(1, CONSUMER_WARPS * 32);
            }

            const int hq0 = gr.g * p.G + (r0 % p.G), hq1 = gr.g * p.G + (r1 % p.G);
            if (cs == 1) {
                if (wk == 0) {
                    const float inv0 = (l0 > 0.f) ? 1.f / l0 : 0.f;
                    const float inv1 = (l1 > 0.f) ? 1.f / l1 : 0.f;
                    __nv_bfloat16* o0 = p.out + (((int64_t)gr.b * p.N + i0) * p.Hq + hq0) * D;
                    __nv_bfloat16* o1 = p.out + (((int64_t)gr.b * p.N + i1) * p.Hq + hq1) * D;
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        const int c = j * 8 + 2 * cq;
                        if (v0) *reinterpret_cast<uint32_t*>(o0 + c) = pack_bf16x2(o[j][0] * inv0, o[j][1] * inv0);
                        if (v1) *reinterpret_cast<uint32_t*>(o1 + c) = pack_bf16x2(o[j][2] * inv1, o[j][3] * inv1);
                    }
                }
                continue;
            }

            // ---- cluster merge through distributed shared memory
            // (1) the previous exchange buffer has been read by every peer
            bool fine = true;
            if (merges > 0) fine = __all_sync(0xffffffffu, mbar_wait_cluster(xfree, (merges - 1) & 1u));
            // (2) publish this CTA's unnormalised rows with their (max, sum)
            if (wk == 0) {
                float* x0 = xo + lr0 * XS;
                float* x1 = xo + lr1 * XS;
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const int c = j * 8 + 2 * cq;
                    *reinterpret_cast<float2*>(x0 + c) = make_float2(o[j][0], o[j][1]);
                    *reinterpret_cast<float2*>(x1 + c) = make_float2(o[j][2], o[j][3]);
                }
                if (cq == 0) {
                    *reinterpret_cast<float2*>(x0 + D) = make_float2(m0, l0);
                    *reinterpret_cast<float2*>(x1 + D) = make_float2(m1, l1);
                }
            }
            asm volatile("fence.acq_rel.cluster;" ::: "memory");
            named_bar_sync(1, CONSUMER_WARPS * 32);
            if (lane == 0)
                for (uint32_t r = 0; r < cs; ++r) remote_arrive(xready, r);
            fine = __all_sync(0xffffffffu, fine && mbar_wait_cluster(xready, merges & 1u));
            if (!fine && lane == 0) {
                flags[0] = 1;
                p.status[gr.b] = TV_ERR_TIMEOUT;
            }
            // (3) this CTA finishes rows [rank*QROWS/cs, (rank+1)*QROWS/cs): per-row
            //     weights 2^(m_c - max) of each peer's partial, then the weighted sum
            const int rows_per = QROWS / (int)cs;
            const int rbase = (int)rank * rows_per;
            for (int lr = rbase + tid; lr < rbase + rows_per; lr += CONSUMER_WARPS * 32) {
                float mx = -INFINITY;
                for (uint32_t c = 0; c < cs; ++c) mx = fmaxf(mx, remote_ld_f2(xo + lr * XS + D, c).x);
                const float bz = (mx == -INFINITY) ? 0.f : mx;
                float den = 0.f;
                for (uint32_t c = 0; c < cs; ++c) {
                    const float2 ml = remote_ld_f2(xo + lr * XS + D, c);
                    const float w = exp2f(ml.x - bz);
                    wts[lr * MAX_CS + c] = w;
                    den += w * ml.y;
                }
                inv_den[lr] = (den > 0.f) ? 1.f / den : 0.f;
            }
            named_bar_sync(1, CONSUMER_WARPS * 32);
            for (int e = tid; e < rows_per * (D / 4); e += CONSUMER_WARPS * 32) {
                const int lr = rbase + e / (D / 4);
                const int c4 = (e % (D / 4)) * 4;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (uint32_t c = 0; c < cs; ++c) {
                    const float w = wts[lr * MAX_CS + c];
                    const float4 x = remote_ld_f4(xo + lr * XS + c4, c);
                    acc.x += w * x.x;
                    acc.y += w * x.y;
                    acc.z += w * x.z;
                    acc.w += w * x.w;
                }
                const int r = gr.qt * QROWS + lr;
                if (r < gr.n * p.G) {
                    const float inv = inv_den[lr];
                    const int node = r / p.G, hq = gr.g * p.G + r % p.G;
                    __nv_bfloat16* dst = p.out + (((int64_t)gr.b * p.N + node) * p.Hq + hq) * D + c4;
                    uint2 pk;
                    pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
                    pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
                    *reinterpret_cast<uint2*>(dst) = pk;
                }
            }
            // (4) tell every peer this CTA is done reading their buffers
            __syncwarp();
            if (lane == 0)
                for (uint32_t r = 0; r < cs; ++r) remote_arrive(xfree, r);
            ++merges;
        }
        // the last exchange must be read by every peer before any CTA leaves
        if (merges > 0) mbar_wait_cluster(xfree, (merges - 1) & 1u);
        __syncwarp();
    }

    // no CTA may exit while a peer can still arrive on its barriers
    cluster_barrier_all();
    if (tid == 0) {
        __threadfence();
        const int done = atomicAdd(&p.sched[1], 1);
        if (done == (int)gridDim.x - 1) {  // last CTA: return the counters to zero
            p.sched[0] = 0;
            p.sched[1] = 0;
        }
    }
}

// ---------------------------------------------------------------- host side
constexpr size_t kSchedBytes = 256;  // two counters, padded

void warp_grid(int M, int* WM, int* WK) {
    if (M <= 16) { *WM = 1; *WK = 8; }
    else if (M <= 32) { *WM = 2; *WK = 4; }
    else if (M <= 64) { *WM = 4; *WK = 2; }
    else { *WM = 8; *WK = 1; }
}

template <int D, int WM, int WK>
size_t smem_bytes() {
    constexpr int QROWS = WM * 16;
    return 1024 + Layout<D>::RING_BYTES + (size_t)(WK - 1) * QROWS * (D + 2) * 4 +
           (size_t)QROWS * Layout<D>::XO_STRIDE * 4 + (size_t)QROWS * MAX_CS * 4 +
           (size_t)QROWS * 4 + (2 * STAGES + 1 + 2 * GQ + 2) * 8 + GQ * 4 + 16 +
           2 * LPT_MAX * 4;
}

// Clusters resident at once for cluster size cs (0 if the launch cannot fit).
template <int D, int WM, int WK>
int resident_clusters(int cs, size_t smem) {
    static int cache[17] = {-1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1};
    if (cs >= 1 && cs <= 16 && cache[cs] >= 0) return cache[cs];
    auto kern = attn_bf16_kernel<D, WM, WK>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = cs;
    at.val.clusterDim.y = 1;
    at.val.clusterDim.z = 1;
    cfg.attrs = &at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    if (cs >= 1 && cs <= 16) cache[cs] = n;
    return n;
}

// Cluster size minimising rounds * (tiles per CTA + a one-tile merge cost).
template <int D, int WM, int WK>
int pick_cluster_size(int groups, int64_t tiles_max, size_t smem, int* ncl_out) {
    int best_cs = 1, best_ncl = 0;
    double best = 1e300;
    for (int cs = 1; cs <= 8; cs *= 2) {
        if (cs > 1 && tiles_max < 2 * cs) break;
        const int ncl = resident_clusters<D, WM, WK>(cs, smem);
        if (ncl <= 0) continue;
        const int64_t rounds = (groups + ncl - 1) / ncl;
        const double cost = (double)rounds * ((double)tiles_max / cs + (cs > 1 ? 1.0 : 0.0));
        if (cost < best * 0.97) {
            best = cost;
            best_cs = cs;
            best_ncl = ncl;
        }
    }
    *ncl_out = best_ncl;
    return best_cs;
}

template <int D, int WM, int WK>
tv_status launch_typed(const AttnArgs& a, const CUtensorMap& km, const CUtensorMap& vm,
                       Params prm) {
    auto kern = attn_bf16_kernel<D, WM, WK>;
    const size_t smem = smem_bytes<D, WM, WK>();
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return TV_ERR_CUDA;
        attr_set = true;
    }
    const int64_t tiles_max = ((int64_t)a.max_blocks * a.bs + KT - 1) / KT;
    int ncl = 0;
    const int cs = pick_cluster_size<D, WM, WK>(prm.groups, tiles_max, smem, &ncl);
    if (ncl <= 0) return TV_ERR_CUDA;
    const int clusters = std::min<int64_t>(ncl, prm.groups);
    LaunchCfg lc(dim3((unsigned)(clusters * cs)), dim3(THREADS), smem, a.stream, (unsigned)cs);
    return cudaLaunchKernelEx(&lc.cfg, kern, km, vm, prm) == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

}  // namespace

size_t attn_bf16_workspace(int B, int N, int Hq, int Hkv, int d, int max_blocks, int bs) {
    (void)max_blocks; (void)bs;
    if (attn_tc_applicable(N, Hq, Hkv, d)) return attn_tc_workspace(B, N, Hq, Hkv);
    return kSchedBytes;
}

size_t attn_bf16_workspace_zeroed_prefix(int B, int N, int Hq, int Hkv, int d, int max_blocks,
                                         int bs) {
    (void)max_blocks; (void)bs;
    if (attn_tc_applicable(N, Hq, Hkv, d)) return attn_tc_zeroed_prefix(B, N, Hq, Hkv);
    return kSchedBytes;
}

tv_status launch_attn_bf16(const AttnArgs& a) {
    if (a.B == 0) return TV_OK;
    if (a.ws_bytes < kSchedBytes || a.ws == nullptr) return TV_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(a.ws) & 255) != 0) return TV_ERR_WORKSPACE;
    if (attn_tc_applicable(a.N, a.Hq, a.Hkv, a.d)) return launch_attn_tc(a);
    const int64_t rows = (int64_t)a.num_blocks * a.Hkv * a.bs;
    if (rows >= (1LL << 31)) return TV_ERR_UNSUPPORTED;
    CUtensorMap km, vm;
    if (!make_cache_map(&km, a.k_cache, a.d, rows) || !make_cache_map(&vm, a.v_cache, a.d, rows))
        return TV_ERR_CUDA;
    const int G = a.Hq / a.Hkv, M = a.N * G;
    int WM, WK;
    warp_grid(M, &WM, &WK);
    const int qrows = WM * 16;
    Params prm{};
    prm.q = static_cast<const __nv_bfloat16*>(a.q);
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
    prm.M = M;
    prm.bs = a.bs;
    prm.num_blocks = a.num_blocks;
    prm.QT = (M + qrows - 1) / qrows;
    const int64_t groups = (int64_t)a.B * a.Hkv * prm.QT;
    if (groups >= (1LL << 30)) return TV_ERR_UNSUPPORTED;
    prm.groups = (int)groups;
    prm.scale_log2 = a.scale * LOG2E;
#define TV_ATTN_CASE(D_, WM_, WK_)                                   \
    if (a.d == D_ && WM == WM_ && WK == WK_) return launch_typed<D_, WM_, WK_>(a, km, vm, prm);
    TV_ATTN_CASE(128, 1, 8)
    TV_ATTN_CASE(128, 2, 4)
    TV_ATTN_CASE(128, 4, 2)
    TV_ATTN_CASE(128, 8, 1)
    TV_ATTN_CASE(64, 1, 8)
    TV_ATTN_CASE(64, 2, 4)
    TV_ATTN_CASE(64, 4, 2)
    TV_ATTN_CASE(64, 8, 1)
#undef TV_ATTN_CASE
    return TV_ERR_UNSUPPORTED;
}

}  // namespace tv
