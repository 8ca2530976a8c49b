// tree_verify_attention, bfloat16 path.
//
// Work decomposition
//   All query heads of one KV group times all tree nodes form one packed row
//   block: row r = node * G + head-in-group (G = Hq / Hkv), M = N * G rows.
//   The KV range 0 .. P+N-1 of a sequence is cut into fixed chunks of C keys
//   (a multiple of the 64-key tile).  A work item is (sequence, chunk, kv
//   head, row tile); items are enumerated chunk-major so the row tiles that
//   share a chunk run side by side and share its K/V through L2.  One
//   persistent CTA per SM walks the items with a static stride.
//
// CTA roles
//   warp 8 (producer): one lane streams 64-key K and V tiles through a
//   4-stage shared-memory ring with 2-D TMA copies (one 16-key page = one
//   16 x 64-element box per 64-column half, 128-byte swizzle), resolving
//   pages through the block table.  Full/empty mbarriers pair it with
//   warps 0..7 (consumers), arranged as WM row warps (16 rows each) times WK
//   key groups (group k takes tiles k, k+WK, ...).
//   Consumers: S = Q K^T and O += P V with mma.sync m16n8k16 (bf16 in, fp32
//   accumulate), online softmax in registers (base 2), tree mask applied on
//   the tiles that reach the tree's own positions.
//
// Split-KV: a sequence with more than one chunk writes per-chunk partials
//   (unnormalised O, running max, running sum) to the workspace; the last
//   CTA to finish a (sequence, kv head, row tile) — found with an atomic
//   ticket — merges them and resets the ticket to zero.
#include <algorithm>

#include "tv_device.cuh"
#include "tv_internal.h"

namespace tv {

namespace {

constexpr int KT = 64;       // keys per tile
constexpr int STAGES = 4;    // TMA ring depth
constexpr int CONSUMER_WARPS = 8;
constexpr int THREADS = (CONSUMER_WARPS + 1) * 32;
constexpr int MAX_B = 4096;  // prefix table lives in shared memory
constexpr float LOG2E = 1.4426950408889634f;

struct Params {
    const __nv_bfloat16* q;
    const int32_t* table;
    const int32_t* prefix_lens;
    const uint64_t* mask;
    __nv_bfloat16* out;
    int32_t* status;
    int32_t* counters;   // [B][Hkv][QT]
    float* part_o;       // [B][max_nc][Hkv][QT*QROWS][D]
    float* part_ml;      // [B][max_nc][Hkv][QT*QROWS][2]
    int max_blocks, B, N, Hq, Hkv, G, M, bs, num_blocks;
    int chunk;           // keys per chunk (multiple of KT)
    int max_nc;          // chunks per sequence upper bound
    int QT;              // row tiles
    float scale_log2;    // scale * log2(e)
};

template <int D>
struct Layout {
    static constexpr int TILE_BYTES = KT * D * 2;           // one K or V tile
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
};

__device__ __forceinline__ int num_chunks(int P, int N, int cap, int chunk) {
    if (P < 0 || (int64_t)P + N > cap) return 1;  // invalid: one item that writes zeros
    return (P + N + chunk - 1) / chunk;
}

// Sequence validity: prefix length in range and every block id covering
// positions 0..P+N-1 inside the cache.  Evaluated by a group of `nthr`
// threads starting at thread `t0`; the result is combined with `combine`.
__device__ __forceinline__ bool seq_blocks_ok(const Params& p, int b, int P, int tid, int nthr) {
    if (P < 0 || (int64_t)P + p.N > (int64_t)p.max_blocks * p.bs) return false;
    const int nb = (P + p.N + p.bs - 1) / p.bs;
    bool ok = true;
    for (int j = tid; j < nb; j += nthr) {
        const int blk = p.table[(int64_t)b * p.max_blocks + j];
        ok = ok && blk >= 0 && blk < p.num_blocks;
    }
    return ok;
}

struct Item {
    int b, c, g, qt, P, L, kbeg, kend;
};

__device__ __forceinline__ Item decode_item(const Params& p, const int* pref, int idx) {
    // pref[b] = first item of sequence b (pref[B] = total); binary search
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pref[mid] <= idx) lo = mid; else hi = mid - 1;
    }
    Item it;
    it.b = lo;
    int r = idx - pref[lo];
    it.qt = r % p.QT;
    r /= p.QT;
    it.g = r % p.Hkv;
    it.c = r / p.Hkv;
    it.P = p.prefix_lens[it.b];
    it.L = it.P + p.N;
    it.kbeg = it.c * p.chunk;
    it.kend = min(it.L, it.kbeg + p.chunk);
    return it;
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

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* ring = smem;
    float* scratch = reinterpret_cast<float*>(smem + LY::RING_BYTES);
    constexpr int SCRATCH_FLOATS = (WK - 1) * QROWS * (D + 2);
    int* pref = reinterpret_cast<int*>(scratch + SCRATCH_FLOATS);
    uint64_t* bars = reinterpret_cast<uint64_t*>(
        (reinterpret_cast<uintptr_t>(pref + p.B + 1) + 7) & ~uintptr_t(7));
    uint64_t* full_bar = bars;
    uint64_t* empty_bar = bars + STAGES;
    uint64_t* tail_bar = bars + 2 * STAGES;
    int* flags = reinterpret_cast<int*>(bars + 2 * STAGES + 1);  // [0] abort, [1] ticket

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cap = p.max_blocks * p.bs;

    // ---- prologue: item prefix table, barriers ------------------------------
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], WM);
        }
        mbar_init(tail_bar, 1);
        flags[0] = 0;
        fence_mbar_init();
    }
    // exclusive scan of items per sequence (chunks * Hkv * QT), chunked by THREADS
    {
        __shared__ int carry;
        __shared__ int wsum[THREADS / 32];
        if (tid == 0) carry = 0;
        __syncthreads();
        for (int base = 0; base < p.B; base += THREADS) {
            const int b = base + tid;
            int v = 0;
            if (b < p.B) v = num_chunks(p.prefix_lens[b], p.N, cap, p.chunk) * p.Hkv * p.QT;
            int x = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off) x += y;
            }
            if (lane == 31) wsum[warp] = x;
            __syncthreads();
            int wpre = 0;
            for (int w = 0; w < warp; ++w) wpre += wsum[w];
            if (b < p.B) pref[b] = carry + wpre + x - v;
            __syncthreads();
            if (tid == THREADS - 1) carry += wpre + x;
            __syncthreads();
        }
        if (tid == 0) pref[p.B] = carry;
        __syncthreads();
    }
    const int total_items = pref[p.B];

    if (warp == CONSUMER_WARPS) {
        // =========================== producer ===========================
        if (lane == 0) {
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
        }
        const uint64_t policy = (p.QT == 1) ? l2_policy_evict_first() : l2_policy_evict_normal();
        uint32_t gt = 0;         // tiles issued by this CTA
        uint32_t tail_phase = 0;
        bool alive = true;
        for (int idx = blockIdx.x; idx < total_items && alive; idx += gridDim.x) {
            const Item it = decode_item(p, pref, idx);
            const bool ok = __all_sync(0xffffffffu, seq_blocks_ok(p, it.b, it.P, lane, 32));
            if (!ok) continue;
            const int ntiles = (it.kend - it.kbeg + KT - 1) / KT;
            for (int lt = 0; lt < ntiles; ++lt, ++gt) {
                const int s = gt % STAGES;
                const uint32_t ph = (gt / STAGES) & 1u;
                bool got = true;
                if (lane == 0) got = mbar_wait(&empty_bar[s], ph ^ 1u);
                got = __shfl_sync(0xffffffffu, got, 0);
                if (!got || *(volatile int*)&flags[0]) {
                    if (lane == 0) {
                        flags[0] = 1;
                        p.status[it.b] = TV_ERR_TIMEOUT;
                    }
                    alive = false;
                    break;
                }
                const int t0 = it.kbeg + lt * KT;
                const int nv = min(KT, it.L - t0);           // valid keys in this tile
                const int pages = (nv + 15) >> 4;
                const uint32_t bytes = (uint32_t)pages * 16u * D * 2u * 2u;
                const bool tail = nv < KT;
                uint64_t* bar = tail ? tail_bar : &full_bar[s];
                uint8_t* kt = ring + s * LY::STAGE_BYTES;
                uint8_t* vt = kt + LY::TILE_BYTES;
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar, bytes);
                    for (int pg = 0; pg < pages; ++pg) {
                        const int t = t0 + pg * 16;
                        const int blk = p.table[(int64_t)it.b * p.max_blocks + t / p.bs];
                        const int y = (blk * p.Hkv + it.g) * p.bs + (t % p.bs);
#pragma unroll
                        for (int hf = 0; hf < D / 64; ++hf) {
                            tma_load_2d(kt + hf * (KT * 128) + pg * 2048, &kmap, bar, hf * 64, y, policy);
                            tma_load_2d(vt + hf * (KT * 128) + pg * 2048, &vmap, bar, hf * 64, y, policy);
                        }
                    }
                }
                if (tail) {
                    // wait for the partial tile, zero the V rows past the sequence end
                    // (they may hold anything), then publish the stage.
                    bool landed = true;
                    if (lane == 0) landed = mbar_wait(tail_bar, tail_phase);
                    landed = __shfl_sync(0xffffffffu, landed, 0);
                    tail_phase ^= 1u;
                    if (!landed) {
                        if (lane == 0) {
                            flags[0] = 1;
                            p.status[it.b] = TV_ERR_TIMEOUT;
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
        return;
    }

    // ============================= consumers =============================
    const int wm = warp % WM, wk = warp / WM;
    const int gq = lane >> 2, cq = lane & 3;
    uint32_t gt_base = 0;
    const uint32_t ring_u32 = smem_u32(ring);

    for (int idx = blockIdx.x; idx < total_items; idx += gridDim.x) {
        const Item it = decode_item(p, pref, idx);
        // validity, evaluated by all consumer threads
        bool ok = seq_blocks_ok(p, it.b, it.P, tid, CONSUMER_WARPS * 32);
        ok = __all_sync(0xffffffffu, ok);
        {
            __shared__ int okw[CONSUMER_WARPS];
            if (lane == 0) okw[warp] = ok;
            named_bar_sync(1, CONSUMER_WARPS * 32);
            for (int w = 0; w < CONSUMER_WARPS; ++w) ok = ok && okw[w];
            named_bar_sync(1, CONSUMER_WARPS * 32);
        }
        const int nc = num_chunks(it.P, p.N, cap, p.chunk);
        if (tid == 0 && it.c == 0 && it.g == 0 && it.qt == 0)
            p.status[it.b] = ok ? TV_OK : TV_ERR_OUT_OF_RANGE;
        const int ntiles = ok ? (it.kend - it.kbeg + KT - 1) / KT : 0;

        // rows of this thread within the packed block
        const int r0 = it.qt * QROWS + wm * 16 + gq, r1 = r0 + 8;
        const bool v0 = r0 < p.M, v1 = r1 < p.M;
        const int i0 = v0 ? r0 / p.G : 0, i1 = v1 ? r1 / p.G : 0;
        const uint64_t nmask = (p.N >= 64) ? ~0ull : ((1ull << p.N) - 1);
        const uint64_t mk0 = v0 ? (p.mask[(int64_t)it.b * p.N + i0] & nmask) : 0;
        const uint64_t mk1 = v1 ? (p.mask[(int64_t)it.b * p.N + i1] & nmask) : 0;

        // Q fragments (A operand), straight from global memory
        uint32_t qa[KC][4];
        {
            const __nv_bfloat16* q0 =
                p.q + (((int64_t)it.b * p.N + i0) * p.Hq + it.g * p.G + (r0 % p.G)) * D;
            const __nv_bfloat16* q1 =
                p.q + (((int64_t)it.b * p.N + i1) * p.Hq + it.g * p.G + (r1 % p.G)) * D;
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
            bool got = !*(volatile int*)&flags[0];
            if (lane == 0 && got) got = mbar_wait(&full_bar[s], ph);
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) {
                if (lane == 0) {
                    flags[0] = 1;
                    p.status[it.b] = TV_ERR_TIMEOUT;
                }
                break;
            }
            const uint32_t ku = ring_u32 + s * LY::STAGE_BYTES;
            const uint32_t vu = ku + LY::TILE_BYTES;
            const int t0 = it.kbeg + lt * KT;

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
                    const uint32_t addr = ku + (dcol >> 6) * (KT * 128) + sw128(key, (dcol & 63) >> 3);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(addr, b0, b1, b2, b3);
                    mma_bf16_16816(sc[2 * jp], qa[kk], b0, b1);
                    mma_bf16_16816(sc[2 * jp + 1], qa[kk], b2, b3);
                }
            }
            // ---- scale, tree mask, online softmax
            const bool need_mask = (t0 + KT > it.P);
            float tmax0 = -INFINITY, tmax1 = -INFINITY;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int t = t0 + j * 8 + 2 * cq + e;
                    float s0 = sc[j][e] * p.scale_log2, s1 = sc[j][2 + e] * p.scale_log2;
                    if (need_mask) {
                        const bool tree = t >= it.P && t < it.L;
                        const int a = t - it.P;
                        const bool vis0 = (t < it.P) || (tree && ((mk0 >> a) & 1ull));
                        const bool vis1 = (t < it.P) || (tree && ((mk1 >> a) & 1ull));
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
                    const uint32_t addr = vu + (dcol >> 6) * (KT * 128) + sw128(key, (dcol & 63) >> 3);
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

        // row sums across the quad
#pragma unroll
        for (int off = 1; off <= 2; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }

        // ---- merge the WK key groups into group 0
        if (WK > 1) {
            const int lr0 = wm * 16 + gq, lr1 = lr0 + 8;
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
                for (int k = 1; k < WK; ++k) {
                    const float* sc0 = scratch + ((k - 1) * QROWS + lr0) * (D + 2);
                    const float* sc1 = scratch + ((k - 1) * QROWS + lr1) * (D + 2);
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

        // ---- epilogue
        const int hq0 = it.g * p.G + (r0 % p.G), hq1 = it.g * p.G + (r1 % p.G);
        if (nc == 1) {
            if (wk == 0) {
                const float inv0 = (l0 > 0.f) ? 1.f / l0 : 0.f;
                const float inv1 = (l1 > 0.f) ? 1.f / l1 : 0.f;
                __nv_bfloat16* o0 = p.out + (((int64_t)it.b * p.N + i0) * p.Hq + hq0) * D;
                __nv_bfloat16* o1 = p.out + (((int64_t)it.b * p.N + i1) * p.Hq + hq1) * D;
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const int c = j * 8 + 2 * cq;
                    if (v0) *reinterpret_cast<uint32_t*>(o0 + c) = pack_bf16x2(o[j][0] * inv0, o[j][1] * inv0);
                    if (v1) *reinterpret_cast<uint32_t*>(o1 + c) = pack_bf16x2(o[j][2] * inv1, o[j][3] * inv1);
                }
            }
            continue;
        }
        // split: write this chunk's partial, take a ticket, the last CTA merges
        const int rows_all = p.QT * QROWS;
        const int64_t slot = ((int64_t)it.b * p.max_nc + it.c) * p.Hkv + it.g;
        if (wk == 0) {
            float* po = p.part_o + slot * rows_all * D;
            float* pml = p.part_ml + slot * rows_all * 2;
            const int lr0 = it.qt * QROWS + wm * 16 + gq, lr1 = lr0 + 8;
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int c = j * 8 + 2 * cq;
                *reinterpret_cast<float2*>(po + (int64_t)lr0 * D + c) = make_float2(o[j][0], o[j][1]);
                *reinterpret_cast<float2*>(po + (int64_t)lr1 * D + c) = make_float2(o[j][2], o[j][3]);
            }
            if (cq == 0) {
                pml[lr0 * 2] = m0;
                pml[lr0 * 2 + 1] = l0;
                pml[lr1 * 2] = m1;
                pml[lr1 * 2 + 1] = l1;
            }
        }
        __threadfence();
        named_bar_sync(1, CONSUMER_WARPS * 32);
        int32_t* ctr = p.counters + ((int64_t)it.b * p.Hkv + it.g) * p.QT + it.qt;
        if (tid == 0) flags[1] = atomicAdd(ctr, 1);
        named_bar_sync(1, CONSUMER_WARPS * 32);
        if (flags[1] != nc - 1) continue;
        __threadfence();
        // merge all nc partials of this (sequence, kv head, row tile)
        for (int e = tid; e < QROWS * D; e += CONSUMER_WARPS * 32) {
            const int lr = e / D, col = e % D;
            const int r = it.qt * QROWS + lr;
            if (r >= p.M) continue;
            float mx = -INFINITY;
            for (int c = 0; c < nc; ++c) {
                const int64_t sl = ((int64_t)it.b * p.max_nc + c) * p.Hkv + it.g;
                mx = fmaxf(mx, __ldcg(p.part_ml + (sl * rows_all + r) * 2));
            }
            const float bz = (mx == -INFINITY) ? 0.f : mx;
            float acc = 0.f, den = 0.f;
            for (int c = 0; c < nc; ++c) {
                const int64_t sl = ((int64_t)it.b * p.max_nc + c) * p.Hkv + it.g;
                const float mc = __ldcg(p.part_ml + (sl * rows_all + r) * 2);
                const float lc = __ldcg(p.part_ml + (sl * rows_all + r) * 2 + 1);
                const float w = exp2f(mc - bz);
                den += lc * w;
                acc += __ldcg(p.part_o + (sl * rows_all + r) * D + col) * w;
            }
            const int node = r / p.G, hq = it.g * p.G + r % p.G;
            p.out[(((int64_t)it.b * p.N + node) * p.Hq + hq) * D + col] =
                __float2bfloat16_rn(den > 0.f ? acc / den : 0.f);
        }
        if (tid == 0) *ctr = 0;  // leave the workspace zeroed for the next call
    }
}

// ---------------------------------------------------------------- host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

bool make_cache_map(CUtensorMap* map, const void* base, int d, int64_t rows) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)d * 2};
    cuuint32_t box[2] = {64, 16};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Plan {
    int WM, WK, QT, chunk, max_nc;
    size_t ws_counters, ws_part_o, ws_part_ml, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

Plan make_plan(int B, int N, int Hq, int Hkv, int d, int max_blocks, int bs, int num_sms) {
    Plan pl{};
    const int G = Hq / Hkv, M = N * G;
    if (M <= 16) { pl.WM = 1; pl.WK = 8; }
    else if (M <= 32) { pl.WM = 2; pl.WK = 4; }
    else if (M <= 64) { pl.WM = 4; pl.WK = 2; }
    else { pl.WM = 8; pl.WK = 1; }
    const int qrows = pl.WM * 16;
    pl.QT = (M + qrows - 1) / qrows;
    const int64_t cap = (int64_t)max_blocks * bs;
    const int64_t tiles_max = (cap + KT - 1) / KT;
    // enough items for ~4 per SM, each at least 2 tiles long
    const int64_t total_tiles = (int64_t)B * Hkv * pl.QT * tiles_max;
    int64_t tpi = (total_tiles + 4LL * num_sms - 1) / (4LL * num_sms);
    tpi = std::max<int64_t>(tpi, 2);
    tpi = std::min<int64_t>(tpi, std::max<int64_t>(tiles_max, 1));
    pl.chunk = (int)(tpi * KT);
    pl.max_nc = (int)std::max<int64_t>(1, (cap + pl.chunk - 1) / pl.chunk);
    const int rows_all = pl.QT * qrows;
    pl.ws_counters = align256((size_t)B * Hkv * pl.QT * sizeof(int32_t));
    if (pl.max_nc > 1) {
        pl.ws_part_o = align256((size_t)B * pl.max_nc * Hkv * rows_all * d * sizeof(float));
        pl.ws_part_ml = align256((size_t)B * pl.max_nc * Hkv * rows_all * 2 * sizeof(float));
    }
    pl.total = pl.ws_counters + pl.ws_part_o + pl.ws_part_ml;
    return pl;
}

template <int D, int WM, int WK>
size_t smem_bytes(int B) {
    return 1024 + Layout<D>::RING_BYTES + (size_t)(WK - 1) * WM * 16 * (D + 2) * 4 +
           (size_t)(B + 1) * 4 + 8 + (2 * STAGES + 1) * 8 + 16;
}

template <int D, int WM, int WK>
tv_status launch_typed(const AttnArgs& a, const Plan& pl, const CUtensorMap& km,
                       const CUtensorMap& vm, const Params& prm, int num_sms) {
    auto kern = attn_bf16_kernel<D, WM, WK>;
    const size_t smem = smem_bytes<D, WM, WK>(a.B);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return TV_ERR_CUDA;
    int total_max = 0;
    {
        // upper bound on items: every sequence at full table capacity
        const int64_t t = (int64_t)a.B * pl.max_nc * a.Hkv * pl.QT;
        total_max = (int)std::min<int64_t>(t, 0x7fffffff);
    }
    const int grid = std::max(1, std::min(num_sms, total_max));
    kern<<<grid, THREADS, smem, a.stream>>>(km, vm, prm);
    return cudaGetLastError() == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

}  // namespace

size_t attn_bf16_workspace(int B, int N, int Hq, int Hkv, int d, int max_blocks, int bs) {
    return make_plan(B, N, Hq, Hkv, d, max_blocks, bs, device_sm_count()).total;
}

tv_status launch_attn_bf16(const AttnArgs& a) {
    if (a.B == 0) return TV_OK;
    if (a.B > MAX_B) return TV_ERR_UNSUPPORTED;
    const int num_sms = device_sm_count();
    const Plan pl = make_plan(a.B, a.N, a.Hq, a.Hkv, a.d, a.max_blocks, a.bs, num_sms);
    if (a.ws_bytes < pl.total || (pl.total > 0 && a.ws == nullptr)) return TV_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(a.ws) & 255) != 0) return TV_ERR_WORKSPACE;
    const int64_t rows = (int64_t)a.num_blocks * a.Hkv * a.bs;
    if (rows >= (1LL << 31)) return TV_ERR_UNSUPPORTED;
    CUtensorMap km, vm;
    if (!make_cache_map(&km, a.k_cache, a.d, rows) || !make_cache_map(&vm, a.v_cache, a.d, rows))
        return TV_ERR_CUDA;
    Params prm{};
    prm.q = static_cast<const __nv_bfloat16*>(a.q);
    prm.table = a.block_table;
    prm.prefix_lens = a.prefix_lens;
    prm.mask = a.mask;
    prm.out = static_cast<__nv_bfloat16*>(a.out);
    prm.status = a.status;
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    prm.counters = reinterpret_cast<int32_t*>(ws);
    prm.part_o = pl.ws_part_o ? reinterpret_cast<float*>(ws + pl.ws_counters) : nullptr;
    prm.part_ml = pl.ws_part_ml ? reinterpret_cast<float*>(ws + pl.ws_counters + pl.ws_part_o)
                                : nullptr;
    prm.max_blocks = a.max_blocks;
    prm.B = a.B;
    prm.N = a.N;
    prm.Hq = a.Hq;
    prm.Hkv = a.Hkv;
    prm.G = a.Hq / a.Hkv;
    prm.M = a.N * prm.G;
    prm.bs = a.bs;
    prm.num_blocks = a.num_blocks;
    prm.chunk = pl.chunk;
    prm.max_nc = pl.max_nc;
    prm.QT = pl.QT;
    prm.scale_log2 = a.scale * LOG2E;
#define TV_ATTN_CASE(D_, WM_, WK_)                                               \
    if (a.d == D_ && pl.WM == WM_ && pl.WK == WK_)                              \
        return launch_typed<D_, WM_, WK_>(a, pl, km, vm, prm, num_sms);
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
