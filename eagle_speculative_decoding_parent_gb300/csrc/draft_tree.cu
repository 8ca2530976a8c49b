// draft_tree_expand: one layer of draft-tree construction per launch
// ("vLLM-TreeEagle", 核心组件 / 3. EnhancedEagleProposer: candidates generated
// over several levels, paths pruned; "EAGLE code principles", 树结构缓冲:
// high-probability paths kept, low-probability branches cut).  Filled in
// EAGLE-2 style: top-k children per expanded node by draft logit, scores are
// cumulative log-probabilities in binary32, the k best new nodes are expanded
// next, and the last layer keeps the N - 1 best nodes.
//
// The draft rows of a layer ([B][F][V] fp32 logits, F = 1 at the first layer,
// then k) are cut into chunks of the vocabulary, one CTA per (row, chunk).
// Each CTA streams its chunk once (16-byte loads when the row allows) and
// reduces it to a running (max, sum of exp) pair and its KP largest logits,
// each kept as one 64-bit word: an order-preserving key of the value above the
// complemented token id, so "larger word" is "larger logit, then lower id".
// The partial results go to the workspace; the CTA whose arrival completes a
// sequence (arrival counter, no waiting) merges the chunks of every row of the
// sequence, appends the F x k new nodes with score = parent score + logit -
// logsumexp(row), ranks them into the next frontier and, on the last layer,
// keeps the root and the N - 1 best nodes (bitonic sort of the node words)
// and labels them breadth-first, level by level.
// All ranking is by exact comparisons of those 64-bit words.
#include <algorithm>

#include "tv_device.cuh"
#include "tv_internal.h"

namespace tv {

namespace {

constexpr int DT_THREADS = 256;
constexpr int DT_WARPS = DT_THREADS / 32;
constexpr int DT_HDR = 32;  // int32 header words of a sequence's state
constexpr int DT_FRONT = 8;  // header word where the frontier ids start

struct DtParams {
    const float* logits;  // [B][F][V]
    const int32_t* root_tokens;
    int B, V, k, F, layer, layers, N, c, per, cmax;
    int32_t* front_tokens;  // [B][k] or null
    int32_t* front_src;     // [B][k] or null
    int32_t* parents;       // [B][N], last layer
    int32_t* tokens;        // [B][N], last layer
    float* scores;          // [B][N] or null, last layer
    int32_t* status;
    int32_t* tick;      // [B] arrival counters
    int32_t* state;     // [B][DT_HDR + 4 * cmax]
    float2* ms;         // [B * k][DT_CH_MAX] (max, sum of exp); sum -1 marks bad values
    uint64_t* top;      // [B * k][DT_CH_MAX][KP]
};

// Order-preserving 32-bit key of a float (-0 taken as +0): larger key, larger value.
__device__ __forceinline__ uint32_t dt_key(float v) {
    uint32_t u = __float_as_uint(v);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float dt_unkey(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
// (value, id) as one word: higher value first, then lower id.  Never 0.
__device__ __forceinline__ uint64_t dt_word(float v, int id) {
    return ((uint64_t)dt_key(v) << 32) | (uint32_t)~(uint32_t)id;
}
__device__ __forceinline__ int dt_word_id(uint64_t w) { return (int)~(uint32_t)w; }

// A warp's KP largest words, spread over its lanes in descending order: lane j
// < KP holds the j-th largest (0 = empty), lanes >= KP hold 0.  An insertion is
// one ballot (how many held words beat the new one) and one shuffle (the words
// below it move down a lane), so keeping the list costs the warp a few
// instructions per word that enters, and nothing per word that does not: a
// value filter (one comparison per logit against the value of the last word)
// lets through a superset of the words that beat it, and the exact 64-bit
// comparison decides.
template <int KP>
struct DtWarpList {
    uint64_t w = 0;
    float thr = -INFINITY;  // value of the last word once the list is full, warp-uniform
    uint64_t last = 0;      // the last word (0 while the list is not full), warp-uniform

    // x is distinct from every held word; it enters when it beats the last one
    __device__ __forceinline__ void insert(uint64_t x, int lane) {
        const int pos = __popc(__ballot_sync(0xffffffffu, lane < KP && w > x));
        if (pos >= KP) return;
        const uint64_t up = __shfl_up_sync(0xffffffffu, w, 1);
        if (lane < KP) w = (lane < pos) ? w : (lane == pos ? x : up);
        last = __shfl_sync(0xffffffffu, w, KP - 1);
        if (last != 0) thr = dt_unkey((uint32_t)(last >> 32));
    }
    // every lane's logit v of token id, where `has` is set; after each insertion
    // the lanes still to come are filtered again against the raised threshold
    __device__ __forceinline__ void offer(float v, int id, bool has, int lane) {
        unsigned hits = __ballot_sync(0xffffffffu, has && v >= thr);
        while (hits) {
            const int src = __ffs(hits) - 1;
            insert(dt_word(__shfl_sync(0xffffffffu, v, src), __shfl_sync(0xffffffffu, id, src)),
                   lane);
            hits &= __ballot_sync(0xffffffffu, has && v >= thr) & ~((2u << src) - 1u);
        }
    }
};

// (m, s) <- the pair of the union: max, and sum of exp(x - max).
__device__ __forceinline__ void dt_combine(float& m, float& s, float m2, float s2) {
    const float M = fmaxf(m, m2);
    if (M == -INFINITY) return;
    s = (m == -INFINITY ? 0.f : s * expf(m - M)) + (m2 == -INFINITY ? 0.f : s2 * expf(m2 - M));
    m = M;
}
__device__ __forceinline__ void dt_warp_combine(float& m, float& s) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
        dt_combine(m, s, m2, s2);
    }
}

// The k-th largest (k <= 32) of the warp's values x, by a bitonic sort of their
// order-preserving keys (NaN keys sort as values; a NaN bound lets nothing
// through, and a row holding NaN is reported as bad values anyway).
__device__ __forceinline__ float dt_warp_kth(float x, int k, int lane) {
    uint32_t key = dt_key(x);
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int j = size >> 1; j > 0; j >>= 1) {
            const uint32_t other = __shfl_xor_sync(0xffffffffu, key, j);
            // descending overall: the lower lane of a pair keeps the larger key
            // in blocks of `size` whose bit is clear, the smaller where it is set
            const bool lower = (lane & j) == 0;
            const bool desc = (lane & size) == 0;
            const uint32_t hi = max(key, other), lo = min(key, other);
            key = (lower == desc) ? hi : lo;
        }
    }
    return dt_unkey(__shfl_sync(0xffffffffu, key, k - 1));
}

// Descending bitonic sort of the warp's 32 words: lane i ends with the i-th largest.
__device__ __forceinline__ uint64_t dt_sort32(uint64_t key, int lane) {
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int j = size >> 1; j > 0; j >>= 1) {
            const uint64_t other = __shfl_xor_sync(0xffffffffu, key, j);
            const bool keep_hi = ((lane & j) == 0) == ((lane & size) == 0);
            key = keep_hi ? (key > other ? key : other) : (key < other ? key : other);
        }
    }
    return key;
}
// Lanes 0-15 and lanes 16-31 each hold a descending run: the 32 words in
// descending order (the upper run reversed makes one bitonic sequence, then
// five half-cleaner stages).
__device__ __forceinline__ uint64_t dt_merge32(uint64_t key, int lane) {
    key = __shfl_sync(0xffffffffu, key, lane < 16 ? lane : 47 - lane);
#pragma unroll
    for (int j = 16; j > 0; j >>= 1) {
        const uint64_t other = __shfl_xor_sync(0xffffffffu, key, j);
        key = ((lane & j) == 0) ? (key > other ? key : other) : (key < other ? key : other);
    }
    return key;
}
// The 16 largest of words ld(0 .. n) (0 = none), descending in lanes 0-15 of the
// calling warp.  The words come in runs of `run` (a power of two <= 16), each
// descending: runs of 16 are merged into the best 16 so far, shorter runs
// sorted together with them.  Eight loads a lane are in flight.
template <class Load>
__device__ __forceinline__ uint64_t dt_top16(int n, int run, int lane, Load ld) {
    uint64_t top = 0;  // lanes 0-15: the best so far
    for (int g0 = 0; g0 < n; g0 += 16 * 8) {
        uint64_t nw[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = g0 + 16 * j + lane - 16;
            nw[j] = (lane >= 16 && e < n) ? ld(e) : 0ull;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (g0 + 16 * j >= n) break;  // uniform across the warp
            const uint64_t x = (lane < 16) ? top : nw[j];
            top = (run == 16) ? dt_merge32(x, lane) : dt_sort32(x, lane);
        }
    }
    return top;
}

// One CTA's pass over logits [lo, hi) of a row: each thread keeps a running
// (max, sum of exp) of the logits it loads, its warp keeps the warp's KP best
// words.  Every thread loads DT_U 16-byte vectors (4 * DT_U scalars without
// them) before it uses any, and the block steps through the range in lock step
// so the warp-wide list operations see converged warps.  The sum of exp uses
// the hardware exponential (arguments <= 0; a few units in the last place for
// the terms near the maximum, which carry the sum).
constexpr int DT_U = 4;
constexpr float DT_LOG2E = 1.4426950408889634f;

template <int KP, bool VEC>
__device__ __forceinline__ void dt_stream(const float* x, int lo, int hi, int tid, int lane,
                                          DtWarpList<KP>& L, float& m, float& s, bool& bad) {
    constexpr int E = 4 * DT_U;  // logits per thread per step
    const int nstep = (hi - lo + E * DT_THREADS - 1) / (E * DT_THREADS);
    for (int st = 0; st < nstep; ++st) {
        float a[E];
        int t0[DT_U];
        bool in[DT_U];
        if (VEC) {
#pragma unroll
            for (int u = 0; u < DT_U; ++u) {
                const int i = lo + st * E * DT_THREADS + (u * DT_THREADS + tid) * 4;
                t0[u] = i;
                in[u] = i < hi;  // the chunk length is a multiple of 4
                const float4 v = in[u] ? __ldcs(reinterpret_cast<const float4*>(x + i))
                                       : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                a[4 * u] = v.x;
                a[4 * u + 1] = v.y;
                a[4 * u + 2] = v.z;
                a[4 * u + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int u = 0; u < DT_U; ++u) {
                t0[u] = lo + st * E * DT_THREADS + u * 4 * DT_THREADS + tid;
                in[u] = true;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int i = t0[u] + c * DT_THREADS;
                    a[4 * u + c] = (i < hi) ? __ldcs(x + i) : -INFINITY;
                }
            }
        }
        float mx = a[0];
#pragma unroll
        for (int e = 0; e < E; ++e) mx = fmaxf(mx, a[e]);  // ignores NaN
        // first step: the KP-th largest of the lanes' maxima bounds the KP-th
        // largest logit from below (the KP largest maxima are KP distinct
        // logits), so nothing below it can enter; a warp sort of the maxima
        if (st == 0) L.thr = dt_warp_kth(mx, KP, lane);
        if (mx > m) {
            s = (m == -INFINITY) ? 0.f : s * expf(m - mx);
            m = mx;
        }
        if (m > -INFINITY) {
            // exp(a - m) = 2^(a log2 e - m log2 e), one fma per logit; a NaN logit
            // makes the step's sum NaN, +inf makes the maximum +inf
            const float ml = m * DT_LOG2E;
            float s2 = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) s2 += ex2_approx(fmaf(a[e], DT_LOG2E, -ml));
            s += s2;
            bad |= !(s2 == s2) || mx == INFINITY;
        } else {
            // nothing finite yet: every value still needs its own NaN / +inf check
#pragma unroll
            for (int e = 0; e < E; ++e) bad |= !(a[e] < INFINITY);
        }
        // the warp looks at the step's logits only when one of them can enter
        if (__any_sync(0xffffffffu, mx >= L.thr)) {
#pragma unroll
            for (int u = 0; u < DT_U; ++u)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int id = VEC ? t0[u] + c : t0[u] + c * DT_THREADS;
                    L.offer(a[4 * u + c], id, VEC ? in[u] : id < hi, lane);
                }
        }
    }
}

template <int KP, bool VEC>
__global__ void __launch_bounds__(DT_THREADS) draft_expand_kernel(DtParams p) {
    pdl_launch_dependents();
    pdl_wait();
    const int row = blockIdx.x / p.c, chunk = blockIdx.x % p.c;
    const int b = row / p.F;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    __shared__ uint64_t s_wtop[DT_WARPS * KP];
    __shared__ float2 s_wms[DT_WARPS];
    __shared__ int s_last, s_err, s_count;
    __shared__ int s_front[DT_K_MAX];
    __shared__ uint64_t s_rtop[DT_K_MAX][KP];
    __shared__ float s_lse[DT_K_MAX];
    __shared__ int s_rowbad[DT_K_MAX];
    __shared__ uint64_t s_cand[DT_K_MAX * DT_K_MAX];
    __shared__ uint64_t s_next[KP];
    __shared__ uint64_t s_fr[DT_WARPS * 16];
    __shared__ uint64_t s_sort[DT_NODES_MAX];
    __shared__ int s_kid[64], s_kdep[64], s_kpar[64], s_kpn[64], s_knew[64];

    // ---- this CTA's chunk of the row ------------------------------------
    {
        const float* x = p.logits + (int64_t)row * p.V;
        const int lo = chunk * p.per;
        const int hi = min(p.V, lo + p.per);
        DtWarpList<KP> L;
        float m = -INFINITY, s = 0.f;
        bool bad_t = false;
        dt_stream<KP, VEC>(x, lo, hi, tid, lane, L, m, s, bad_t);
        const bool bad = __syncthreads_or(bad_t ? 1 : 0) != 0;
        dt_warp_combine(m, s);
        if (lane == 0) s_wms[warp] = make_float2(m, s);
        if (lane < KP) s_wtop[warp * KP + lane] = L.w;
        __syncthreads();
        if (warp == 0) {
            // the warps' lists (descending runs of KP) into the chunk's KP best
            const uint64_t t = dt_top16(DT_WARPS * KP, KP, lane, [&](int e) { return s_wtop[e]; });
            const int64_t slot = (int64_t)row * DT_CH_MAX + chunk;
            if (lane < KP) p.top[slot * KP + lane] = t;
            float bm = (lane < DT_WARPS) ? s_wms[lane].x : -INFINITY;
            float bs = (lane < DT_WARPS) ? s_wms[lane].y : 0.f;
            dt_warp_combine(bm, bs);
            if (lane == 0) {
                p.ms[slot] = make_float2(bm, bad ? -1.f : bs);
                __threadfence();
                s_last = (atomicAdd(&p.tick[b], 1) == p.F * p.c - 1) ? 1 : 0;
            }
        }
        __syncthreads();
        if (!s_last) return;
    }

    // ---- the CTA that completed sequence b ------------------------------
    __threadfence();
    int32_t* st = p.state + (int64_t)b * (DT_HDR + 4 * p.cmax);
    int32_t* tok = st + DT_HDR;
    int32_t* par = tok + p.cmax;
    int32_t* dep = par + p.cmax;
    float* score = reinterpret_cast<float*>(dep + p.cmax);
    if (tid == 0) {
        p.tick[b] = 0;  // ready for the next layer
        int err = TV_OK, count = 0;
        if (p.layer == 0) {
            const int r = p.root_tokens[b];
            if (r < 0 || r >= p.V) err = TV_ERR_OUT_OF_RANGE;
            tok[0] = r;
            par[0] = -1;
            dep[0] = 0;
            score[0] = 0.f;
            count = 1;
            s_front[0] = 0;
        } else {
            const int64_t want = 1 + p.k + (int64_t)(p.layer - 1) * p.k * p.k;
            count = st[1];
            err = st[2];
            if (err == TV_OK && (st[0] != p.layer || count != want)) err = TV_ERR_WORKSPACE;
            for (int f = 0; f < p.F; ++f) {
                const int id = st[DT_FRONT + f];
                if (err == TV_OK && (id < 0 || id >= count)) err = TV_ERR_WORKSPACE;
                s_front[f] = (err == TV_OK) ? id : 0;
            }
        }
        s_err = err;
        s_count = count;
    }
    __syncthreads();
    if (s_err == TV_OK) {
        // every row of the sequence: logsumexp and top-k over its chunks (warp per row)
        for (int f = warp; f < p.F; f += DT_WARPS) {
            const int64_t r = (int64_t)b * p.F + f;
            float m = -INFINITY, s = 0.f;
            bool bad = false;
            for (int c = lane; c < p.c; c += 32) {
                const float2 v = __ldcg(p.ms + r * DT_CH_MAX + c);
                bad |= !(v.y >= 0.f);
                dt_combine(m, s, v.x, v.y);
            }
            dt_warp_combine(m, s);
            bad = __any_sync(0xffffffffu, bad);
            // every chunk's list (descending runs of KP)
            const uint64_t* src = p.top + r * DT_CH_MAX * KP;
            const uint64_t t = dt_top16(p.c * KP, KP, lane, [&](int e) { return __ldcg(src + e); });
            if (lane < KP) s_rtop[f][lane] = t;
            if (lane == 0) {
                s_lse[f] = m + logf(s);
                s_rowbad[f] = (bad || !(m > -INFINITY)) ? 1 : 0;
            }
        }
        __syncthreads();
        if (tid == 0) {
            for (int f = 0; f < p.F; ++f)
                if (s_rowbad[f]) s_err = TV_ERR_BAD_VALUES;
        }
        __syncthreads();
    }
    const bool last_layer = (p.layer == p.layers - 1);
    if (s_err != TV_OK) {
        const int err = s_err;
        if (tid == 0) {
            st[0] = p.layer + 1;
            st[2] = err;
            p.status[b] = err;
        }
        if (tid < p.k) {
            if (p.front_tokens) p.front_tokens[(int64_t)b * p.k + tid] = -1;
            if (p.front_src) p.front_src[(int64_t)b * p.k + tid] = -1;
        }
        if (last_layer && tid < p.N) {
            p.parents[(int64_t)b * p.N + tid] = -1;
            p.tokens[(int64_t)b * p.N + tid] = -1;
            if (p.scores) p.scores[(int64_t)b * p.N + tid] = -INFINITY;
        }
        return;
    }

    // ---- the F x k new nodes, f-major, child rank minor -----------------
    const int count0 = s_count;
    const int nnew = p.F * p.k;
    if (tid < nnew) {
        const int f = tid / p.k, j = tid % p.k;
        const uint64_t w = s_rtop[f][j];
        const int t = dt_word_id(w);
        const float v = dt_unkey((uint32_t)(w >> 32));
        const int pf = s_front[f];
        const float sc = score[pf] + (v - s_lse[f]);
        const int id = count0 + tid;
        tok[id] = t;
        par[id] = pf;
        dep[id] = dep[pf] + 1;
        score[id] = sc;
        s_cand[tid] = dt_word(sc, id);
    }
    __syncthreads();
    // ---- next frontier: the k best new nodes, best first -----------------
    // each warp sorts 32 candidates, then warp 0 merges the warps' best 16
    static_assert(DT_K_MAX * DT_K_MAX <= 32 * DT_WARPS, "one sort round per warp");
    {
        const int e = warp * 32 + lane;
        const uint64_t t = dt_sort32(e < nnew ? s_cand[e] : 0ull, lane);
        if (lane < 16) s_fr[warp * 16 + lane] = t;
    }
    __syncthreads();
    if (warp == 0) {
        const uint64_t t = dt_top16(DT_WARPS * 16, 16, lane, [&](int e) { return s_fr[e]; });
        if (lane < KP) s_next[lane] = t;
    }
    __syncthreads();
    if (tid < p.k) {
        const int id = dt_word_id(s_next[tid]);
        st[DT_FRONT + tid] = id;
        if (p.front_tokens) p.front_tokens[(int64_t)b * p.k + tid] = tok[id];
        if (p.front_src) p.front_src[(int64_t)b * p.k + tid] = (id - count0) / p.k;
    }
    const int C = count0 + nnew;
    if (tid == 0) {
        st[0] = p.layer + 1;
        st[1] = C;
        st[2] = TV_OK;
        p.status[b] = TV_OK;
    }
    if (!last_layer) return;

    // ---- last layer: keep the root and the N - 1 best nodes -------------
    const int M = C - 1;  // candidates: nodes 1 .. C-1
    int P2 = 1;
    while (P2 < M) P2 <<= 1;
    for (int i = tid; i < P2; i += DT_THREADS) s_sort[i] = (i < M) ? dt_word(score[i + 1], i + 1) : 0ull;
    __syncthreads();
    for (int size = 2; size <= P2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = tid; i < (P2 >> 1); i += DT_THREADS) {
                const int lo = 2 * i - (i & (stride - 1));
                const int hi = lo + stride;
                const uint64_t a = s_sort[lo], c = s_sort[hi];
                const bool desc = (lo & size) == 0;
                if (desc ? (a < c) : (a > c)) {
                    s_sort[lo] = c;
                    s_sort[hi] = a;
                }
            }
            __syncthreads();
        }
    }
    const int N = p.N;
    if (tid < N) {
        const int id = (tid == 0) ? 0 : dt_word_id(s_sort[tid - 1]);
        s_kid[tid] = id;
        s_kdep[tid] = dep[id];
        s_kpar[tid] = par[id];
        s_knew[tid] = (tid == 0) ? 0 : -1;
        s_kpn[tid] = -1;
    }
    // breadth-first labels, one depth at a time: a node's label is the number of
    // kept nodes above its depth plus its rank at its depth by (parent's label,
    // creation id)
    for (int d = 1; d <= p.layers; ++d) {
        __syncthreads();
        if (tid < N && s_kdep[tid] == d) {
            int pn = -1;
            for (int j = 0; j < N; ++j)
                if (s_kid[j] == s_kpar[tid]) pn = s_knew[j];
            s_kpn[tid] = pn;
        }
        __syncthreads();
        if (tid < N && s_kdep[tid] == d) {
            int lab = 0;
            for (int j = 0; j < N; ++j) {
                if (s_kdep[j] < d) ++lab;
                else if (s_kdep[j] == d && (s_kpn[j] < s_kpn[tid] ||
                                            (s_kpn[j] == s_kpn[tid] && s_kid[j] < s_kid[tid])))
                    ++lab;
            }
            s_knew[tid] = lab;
        }
    }
    __syncthreads();
    // a kept node whose parent was not kept (cannot happen: a child never
    // scores above its parent) or a label outside [0, N) fails the sequence
    bool ok = true;
    if (tid < N) ok = (s_knew[tid] >= 0 && s_knew[tid] < N) && (tid == 0 || s_kpn[tid] >= 0);
    ok = __syncthreads_and(ok ? 1 : 0) != 0;
    if (!ok) {
        if (tid == 0) {
            st[2] = TV_ERR_BAD_TREE;
            p.status[b] = TV_ERR_BAD_TREE;
        }
        if (tid < N) {
            p.parents[(int64_t)b * N + tid] = -1;
            p.tokens[(int64_t)b * N + tid] = -1;
            if (p.scores) p.scores[(int64_t)b * N + tid] = -INFINITY;
        }
        return;
    }
    if (tid < N) {
        const int n = s_knew[tid];
        const int id = s_kid[tid];
        p.parents[(int64_t)b * N + n] = (tid == 0) ? -1 : s_kpn[tid];
        p.tokens[(int64_t)b * N + n] = tok[id];
        if (p.scores) p.scores[(int64_t)b * N + n] = score[id];
    }
}

int dt_kp(int k) { return k <= 4 ? 4 : (k <= 8 ? 8 : 16); }

size_t dt_align(size_t x) { return (x + 255) & ~(size_t)255; }

struct DtLayout {
    size_t tick, state, ms, top, total;
};

DtLayout dt_layout(int B, int k, int layers) {
    const int64_t cmax = draft_tree_nodes(k, layers);
    const int64_t rows = (int64_t)B * k;
    DtLayout l;
    l.tick = 0;
    l.state = dt_align((size_t)B * 4);
    l.ms = l.state + dt_align((size_t)B * (DT_HDR + 4 * cmax) * 4);
    l.top = l.ms + dt_align((size_t)rows * DT_CH_MAX * 8);
    l.total = l.top + dt_align((size_t)rows * DT_CH_MAX * dt_kp(k) * 8);
    return l;
}

template <int KP>
tv_status dt_launch(const DtParams& p, bool vec, cudaStream_t stream) {
    LaunchCfg lc(dim3((unsigned)((int64_t)p.B * p.F * p.c)), dim3(DT_THREADS), 0, stream);
    const cudaError_t e = vec ? cudaLaunchKernelEx(&lc.cfg, draft_expand_kernel<KP, true>, p)
                              : cudaLaunchKernelEx(&lc.cfg, draft_expand_kernel<KP, false>, p);
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

}  // namespace

int64_t draft_tree_nodes(int k, int layers) {
    return 1 + (int64_t)k + (int64_t)(layers - 1) * k * k;
}

size_t draft_tree_ws_bytes(int B, int k, int layers) { return dt_layout(B, k, layers).total; }

// Chunks per row: enough CTAs to cover the GPU about four times, at least
// DT_CHUNK_MIN logits per chunk (every warp's list costs a few dozen
// insertions to fill, so short chunks spend more on their lists than on the
// stream), at most DT_CH_MAX chunks; `per` is the chunk length (a multiple of
// 4 for 16-byte loads).
constexpr int DT_CHUNK_MIN = 16384;
void draft_tree_chunks(int rows, int V, bool vec, int* c_out, int* per_out) {
    const int64_t target = 4 * (int64_t)device_sm_count();
    int64_t c = (target + rows - 1) / rows;
    c = std::min<int64_t>(c, (V + DT_CHUNK_MIN - 1) / DT_CHUNK_MIN);
    c = std::max<int64_t>(1, std::min<int64_t>(c, DT_CH_MAX));
    int64_t per = (V + c - 1) / c;
    if (vec) per = (per + 3) / 4 * 4;
    c = (V + per - 1) / per;
    *c_out = (int)c;
    *per_out = (int)per;
}

tv_status launch_draft_expand(const DraftArgs& a) {
    const DtLayout l = dt_layout(a.B, a.k, a.layers);
    if (!a.ws || a.ws_bytes < l.total) return TV_ERR_WORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    DtParams p;
    p.logits = a.logits;
    p.root_tokens = a.root_tokens;
    p.B = a.B;
    p.V = a.V;
    p.k = a.k;
    p.F = (a.layer == 0) ? 1 : a.k;
    p.layer = a.layer;
    p.layers = a.layers;
    p.N = a.N;
    p.cmax = (int)draft_tree_nodes(a.k, a.layers);
    const bool vec = (a.V % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.logits) & 15) == 0);
    draft_tree_chunks(a.B * p.F, a.V, vec, &p.c, &p.per);
    p.front_tokens = a.front_tokens;
    p.front_src = a.front_src;
    p.parents = a.parents;
    p.tokens = a.tokens;
    p.scores = a.scores;
    p.status = a.status;
    p.tick = reinterpret_cast<int32_t*>(ws + l.tick);
    p.state = reinterpret_cast<int32_t*>(ws + l.state);
    p.ms = reinterpret_cast<float2*>(ws + l.ms);
    p.top = reinterpret_cast<uint64_t*>(ws + l.top);
    switch (dt_kp(a.k)) {
        case 4: return dt_launch<4>(p, vec, a.stream);
        case 8: return dt_launch<8>(p, vec, a.stream);
        default: return dt_launch<16>(p, vec, a.stream);
    }
}

}  // namespace tv
