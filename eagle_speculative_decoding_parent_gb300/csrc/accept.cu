// tree_accept kernels.
//
//   greedy walk   (large batches) one thread-block cluster per sequence; each
//                 CTA owns a slice of the vocabulary.  A level-by-level walk
//                 from the root: the argmax of every row on the current
//                 frontier of fully matching nodes (usually one) is reduced
//                 inside each CTA, exchanged through distributed shared memory,
//                 and the matching children form the next frontier; the walk
//                 stops at the deepest accepted level, whose argmax is the bonus
//                 token.  Rows read ~ accepted depth + 1.
//   greedy rows   (small batches) every row's argmax in parallel: each row is
//                 cut into chunks, one CTA per chunk; partial results go to the
//                 workspace and the CTA that completes a sequence (arrival
//                 counter) reduces them and walks its tree.  Reads every row
//                 once, without the walk's latency.
//   stochastic    the accept tests touch two scalars per draft (all evaluated at
//                 once, the first failure wins); only the row(s) the emitted
//                 token is drawn from are read, cut into chunks, one CTA per
//                 chunk, each warp streaming whole 2048-element pieces with
//                 16-byte loads.  Integer weights make the sums exact (the draw
//                 does not depend on summation order; they are formed as two
//                 exact parts with packed fp32 arithmetic); the CTA that
//                 completes a sequence picks the piece holding the target
//                 prefix sum and searches it.
// Cluster kernels: all CTAs of a cluster take identical control-flow decisions
// (same inputs, same exchanged values), so every cluster barrier is reached by
// every CTA.  Arrival counters return to zero when a call completes.
#include <algorithm>
#include <cstdlib>

#include <cooperative_groups.h>

#include "tv_device.cuh"
#include "tv_internal.h"

namespace cg = cooperative_groups;

namespace tv {

namespace {

constexpr int NO_INDEX = 0x7fffffff;
constexpr int TIMED_OUT = -2;      // a row argmax whose data did not arrive in time

struct AccParams {
    const int32_t* parents;
    const int32_t* tokens;
    const float* target;
    const float* draft;
    int B, N, V;
    uint64_t seed, offset;
    int32_t* accept_len;
    int32_t* path;
    int32_t* out_tokens;
    int max_path;
    int32_t* status;
    uint64_t data_wait_ns;  // row scan: limit of a wait for streamed data (TV_WAIT_NS)
    const int32_t* counts;  // nullable: nodes per sequence (its tree: the first counts[b] of N)
};

// Node count of sequence b; nodes n..N-1 are absent (never checked or accepted).
__device__ __forceinline__ int seq_count(const AccParams& p, int b) {
    return p.counts ? p.counts[b] : p.N;
}

struct ArgBest {
    float v;
    int i;
};

// (v, i) beats (w, j): larger value, ties to the lower index.  Entries with
// i == NO_INDEX carry no candidate (v is -inf there).
__device__ __forceinline__ bool beats(float v, int i, float w, int j) {
    return (v > w) || (v == w && i < j);
}

__device__ __forceinline__ void take(ArgBest& a, float x, int i) {
    const bool better = !isnan(x) && beats(x, i, a.v, a.i);
    a.v = better ? x : a.v;
    a.i = better ? i : a.i;
}

// Four consecutive elements i..i+3 at once: one maximum, and only when it
// beats the running best (or is the first non-NaN value seen) the lowest
// component equal to it is located.  Same result as four take() calls
// (NaNs skipped, ties to the lower index), at a fraction of the instructions.
__device__ __forceinline__ void take4(ArgBest& a, const float4& x, int i) {
    const float m = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
    if (m > a.v || (a.i == NO_INDEX && m == m)) {
        a.v = m;
        a.i = i + ((x.x == m) ? 0 : (x.y == m) ? 1 : (x.z == m) ? 2 : 3);
    }
}

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11), written from the published
// round function: two 32x32 -> 64-bit products per round, Weyl key schedule.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
        k.x += 0x9E3779B9u;
        k.y += 0xBB67AE85u;
    }
    return c;
}

__device__ __forceinline__ uint4 draw(const AccParams& p, int b, int k) {
    return philox4x32_10(make_uint4((uint32_t)k, (uint32_t)b, (uint32_t)p.offset,
                                    (uint32_t)(p.offset >> 32)),
                         make_uint2((uint32_t)p.seed, (uint32_t)(p.seed >> 32)));
}

// Fixed-point weight floor(min(x, 1) * 2^40); 0 for NaN and x <= 0.  Taken
// from the bits with integer shifts (x * 2^40 = mantissa * 2^(exponent - 110)),
// which equals the truncating float-to-integer conversion of x * 2^40 but
// stays off the slow 64-bit conversion path.
__device__ __forceinline__ uint64_t weight(float x) {
    const uint32_t u = __float_as_uint(x);
    if ((int32_t)u <= 0) return 0ull;                                  // +0, negative, -NaN
    if (u >= 0x3F800000u) return (u > 0x7F800000u) ? 0ull : (1ull << 40);  // NaN; >= 1
    const int sh = (int)(u >> 23) - 110;
    const uint64_t m = (uint64_t)((u & 0x7FFFFFu) | 0x800000u);
    return (sh >= 0) ? (m << sh) : (sh > -24 ? (m >> -sh) : 0ull);
}

__device__ __forceinline__ uint64_t elem_weight(const float* a, const float* bq, int t, bool resid) {
    return resid ? weight(__fsub_rn(__ldg(a + t), __ldg(bq + t))) : weight(__ldg(a + t));
}

__device__ void write_fail(const AccParams& p, int b, int st) {
    for (int j = threadIdx.x; j < p.max_path; j += blockDim.x) {
        p.path[(int64_t)b * p.max_path + j] = (j == 0) ? 0 : -1;
        p.out_tokens[(int64_t)b * p.max_path + j] = -1;
    }
    if (threadIdx.x == 0) {
        p.accept_len[b] = 0;
        p.status[b] = st;
    }
}

// Emits root..chosen and the tokens; rank-0 CTA only (all its threads).
__device__ void write_path(const AccParams& p, int b, const int* spar, const int* stok,
                           int chosen, int last) {
    __shared__ int spath[64];
    __shared__ int sdep;
    if (threadIdx.x == 0) {
        int dep = 0;
        for (int j = chosen; spar[j] >= 0; j = spar[j]) ++dep;
        int j = chosen;
        for (int k = dep; k >= 0; --k) {
            spath[k] = j;
            j = spar[j];
        }
        sdep = dep;
    }
    __syncthreads();
    const int dep = sdep;
    if (dep + 1 > p.max_path) {
        write_fail(p, b, TV_ERR_OUT_OF_RANGE);
        return;
    }
    for (int j = threadIdx.x; j < p.max_path; j += blockDim.x) {
        p.path[(int64_t)b * p.max_path + j] = (j <= dep) ? spath[j] : -1;
        int tok = -1;
        if (j < dep) tok = stok[spath[j + 1]];
        else if (j == dep) tok = last;
        p.out_tokens[(int64_t)b * p.max_path + j] = tok;
    }
    if (threadIdx.x == 0) {
        p.accept_len[b] = dep;
        p.status[b] = TV_OK;
    }
}

// Checks in the order the acceptance rule states them (node count in [1, Nmax],
// then structure, then token range) over the sequence's N nodes.  One full
// warp; result in every lane.
__device__ int check_inputs(const int* spar, const int* stok, int N, int V, int Nmax) {
    const int lane = threadIdx.x & 31;
    if (N < 1 || N > Nmax) return TV_ERR_OUT_OF_RANGE;
    bool tree_bad = false, tok_bad = false;
    for (int i = lane; i < N; i += 32) {
        const int pa = spar[i];
        tree_bad |= (i == 0 && pa != -1) || (i > 0 && (pa < 0 || pa >= i));
        tok_bad |= (i > 0 && (stok[i] < 0 || stok[i] >= V));
    }
    const bool any_tree = __any_sync(0xffffffffu, tree_bad);
    const bool any_tok = __any_sync(0xffffffffu, tok_bad);
    if (any_tree) return TV_ERR_BAD_TREE;
    if (any_tok) return TV_ERR_OUT_OF_RANGE;
    return TV_OK;
}


constexpr int CH_THREADS = 256;            // CTA size of the chunked kernels
constexpr int CH_WARPS = CH_THREADS / 32;
constexpr int CH_MAX = 128;                // chunks per row at most

// Elements per chunk when a row of V entries is cut into ch chunks (multiple of 4).
__device__ __host__ __forceinline__ int chunk_len(int V, int ch) {
    int per = (V + ch - 1) / ch;
    return (per + 3) & ~3;
}

// Rows are streamed through shared memory in pieces of PIECE floats per
// operand with bulk asynchronous copies, STG pieces in flight per CTA.
constexpr int PIECE = 2048;
constexpr int STG = 4;

struct Ring {
    float* buf;        // [stg][ops][PIECE]
    uint64_t* full;    // [stg]
    uint32_t pc;       // pieces this CTA has consumed (ring position and phase)
    int stg;           // pieces in flight
    uint64_t wait_ns;  // limit of a wait for a piece's data
};

// Calls f(x, y, i) for x = a[i..i+3] and y = b[i..i+3] (zeros without b), for
// every i = lo + 4k < hi, each thread a strided subset.  lo and hi - lo are
// multiples of 4 and the rows 16-byte aligned.  Every thread of the CTA calls
// it.  Returns false if a piece did not arrive in time (after waiting, with a
// limit, for the copies still in flight).
template <typename F>
__device__ bool stream_rows(const float* a, const float* b, int lo, int hi, Ring& r, F f) {
    const int tid = threadIdx.x;
    const int ops = b ? 2 : 1;
    const int np = (hi - lo + PIECE - 1) / PIECE;
    const uint64_t pol = l2_policy_evict_first();
    auto issue = [&](int k) {
        const int s = (int)((r.pc + k) % r.stg);
        const int off = lo + k * PIECE;
        const uint32_t bytes = (uint32_t)min(PIECE, hi - off) * 4u;
        mbar_arrive_expect_tx(&r.full[s], bytes * ops);
        bulk_load(r.buf + (size_t)s * ops * PIECE, a + off, bytes, &r.full[s], pol);
        if (b) bulk_load(r.buf + (size_t)s * ops * PIECE + PIECE, b + off, bytes, &r.full[s], pol);
    };
    if (tid == 0)
        for (int k = 0; k < min(r.stg, np); ++k) issue(k);
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (np <= r.stg) {
        // everything is in flight at once: consume the pieces as they land, one
        // barrier at the end
        bool got = true;
        for (int k = 0; k < np; ++k) {
            const uint32_t g = r.pc + k;
            const int s = (int)(g % r.stg);
            got = got && mbar_wait_for(&r.full[s], (g / r.stg) & 1u, r.wait_ns);
            if (got) {
                const int off = lo + k * PIECE, n4 = min(PIECE, hi - off) >> 2;
                const float4* x4 = reinterpret_cast<const float4*>(r.buf + (size_t)s * ops * PIECE);
                const float4* y4 = x4 + PIECE / 4;
                for (int e = tid; e < n4; e += blockDim.x) f(x4[e], b ? y4[e] : z4, off + 4 * e);
            }
        }
        const bool ok = __syncthreads_and(got) != 0;
        if (!ok && tid == 0) {
            for (int k = 0; k < np; ++k) {
                const uint32_t g = r.pc + k;
                mbar_wait(&r.full[g % r.stg], (g / r.stg) & 1u);
            }
        }
        r.pc += np;
        return ok;
    }
    bool ok = true;
    int k = 0;
    for (; k < np; ++k) {
        const uint32_t g = r.pc + k;
        const int s = (int)(g % r.stg);
        const bool got = mbar_wait_for(&r.full[s], (g / r.stg) & 1u, r.wait_ns);
        if (got) {
            const int off = lo + k * PIECE, n4 = min(PIECE, hi - off) >> 2;
            const float4* x4 = reinterpret_cast<const float4*>(r.buf + (size_t)s * ops * PIECE);
            const float4* y4 = x4 + PIECE / 4;
            for (int e = tid; e < n4; e += blockDim.x) f(x4[e], b ? y4[e] : z4, off + 4 * e);
        }
        ok = __syncthreads_and(got) != 0;  // every thread is done with stage s
        if (!ok) break;
        if (tid == 0 && k + r.stg < np) issue(k + r.stg);
    }
    if (!ok && tid == 0) {
        // let the copies still in flight (piece k and the ones issued after it)
        // land before the shared memory is released; these waits keep the full limit
        for (int j = k; j < min(np, k + r.stg); ++j) {
            const uint32_t g = r.pc + j;
            mbar_wait(&r.full[g % r.stg], (g / r.stg) & 1u);
        }
    }
    r.pc += np;
    return ok;
}

// Argmax of row[lo, hi) with every thread's loads in flight at once (twelve
// 16-byte loads per thread per round): for short, latency-bound slices.
// lo and hi - lo are multiples of 4 and the row 16-byte aligned.
__device__ ArgBest slice_argmax_ldg(const float* __restrict__ row, int lo, int hi, ArgBest* red) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    ArgBest a{-INFINITY, NO_INDEX};
    const int n4 = (hi - lo) >> 2;
    const float4* r4 = reinterpret_cast<const float4*>(row + lo);
    constexpr int T = CH_THREADS, U = 12;
    for (int e0 = 0; e0 < n4; e0 += U * T) {
        float4 x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = e0 + u * T + tid;
            x[u] = (e < n4) ? __ldg(r4 + e) : make_float4(NAN, NAN, NAN, NAN);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) take4(a, x[u], lo + 4 * (e0 + u * T + tid));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float w = __shfl_xor_sync(0xffffffffu, a.v, off);
        const int j = __shfl_xor_sync(0xffffffffu, a.i, off);
        if (beats(w, j, a.v, a.i)) {
            a.v = w;
            a.i = j;
        }
    }
    if (lane == 0) red[warp] = a;
    __syncthreads();
    ArgBest r = red[0];
    for (int w = 1; w < CH_WARPS; ++w)
        if (beats(red[w].v, red[w].i, r.v, r.i)) r = red[w];
    return r;
}

// Argmax of row[lo, hi) over the CTA (CH_THREADS threads); valid in every thread.
template <bool VEC>
__device__ ArgBest chunk_argmax(const float* __restrict__ row, int lo, int hi, ArgBest* red,
                                Ring& ring, bool& ok) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    ArgBest a{-INFINITY, NO_INDEX};
    ok = true;
    if (VEC) {
        ok = stream_rows(row, nullptr, lo, hi, ring,
                         [&](const float4& x, const float4&, int i) { take4(a, x, i); });
    } else {
        for (int i = lo + tid; i < hi; i += CH_THREADS) take(a, __ldg(row + i), i);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float w = __shfl_xor_sync(0xffffffffu, a.v, off);
        const int j = __shfl_xor_sync(0xffffffffu, a.i, off);
        if (beats(w, j, a.v, a.i)) {
            a.v = w;
            a.i = j;
        }
    }
    if (lane == 0) red[warp] = a;
    __syncthreads();
    ArgBest r = red[0];
    for (int w = 1; w < CH_WARPS; ++w)
        if (beats(red[w].v, red[w].i, r.v, r.i)) r = red[w];
    return r;
}

// Walks sequence b's tree given every row's argmax (sam[], -1 for none) and
// writes the result: accepted(c) = accepted(parent) and token(c) == argmax of
// the parent's row; the deepest accepted node is emitted with its argmax.
__device__ void walk_and_write(const AccParams& p, int b, const int* spar, const int* stok,
                               const int* sam, int N) {
    __shared__ int schosen;
    if (threadIdx.x < 32) {
        // node c is accepted when every edge on its root path matches; lane takes
        // nodes lane and lane + 32: key = depth, then the lower index on ties
        const int lane = threadIdx.x;
        int best = -1;
        for (int c = lane; c < N; c += 32) {
            bool acc = true;
            int d = 0;
            for (int j = c; j > 0; j = spar[j], ++d) {
                const int pj = spar[j];
                acc = acc && sam[pj] >= 0 && stok[j] == sam[pj];
            }
            if (acc) best = max(best, (d << 8) | (255 - c));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, off));
        if (lane == 0) schosen = 255 - (best & 255);
    }
    __syncthreads();
    const int chosen = schosen;
    if (sam[chosen] < 0) write_fail(p, b, TV_ERR_BAD_VALUES);
    else write_path(p, b, spar, stok, chosen, sam[chosen]);
}

// Greedy acceptance, every row in parallel: CTA (row, c) takes chunk c of the
// row; ws: part[row][CH_MAX] (value bits, index of the chunk's argmax),
// seq_tick[b] (arrivals of the sequence's N x ch CTAs).
template <bool VEC>
__global__ void __launch_bounds__(CH_THREADS)
accept_rows_kernel(AccParams p, int ch, int2* __restrict__ part, int32_t* __restrict__ seq_tick) {
    pdl_launch_dependents();
    pdl_wait();
    const int N = p.N;
    const int row = blockIdx.x / ch, c = blockIdx.x % ch;
    const int b = row / N;
    const int n = seq_count(p, b);     // rows of absent nodes are not scanned
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    __shared__ ArgBest red[CH_WARPS];
    __shared__ int last;
    __shared__ int spar[64], stok[64], sam[64];
    __shared__ int sflag;
    extern __shared__ __align__(1024) float ring_buf[];  // [STG][PIECE]
    __shared__ uint64_t full[STG];
    // the tree is only needed by the CTA that completes the sequence; its loads
    // are issued now so they are in flight while the row streams
    int par_v = 0, tok_v = 0;
    if (tid < N) {
        par_v = p.parents[(int64_t)b * N + tid];
        tok_v = p.tokens[(int64_t)b * N + tid];
    }
    if (tid == 0) {
        for (int k = 0; k < STG; ++k) mbar_init(&full[k], 1);
        fence_mbar_init();
    }
    __syncthreads();
    Ring ring{ring_buf, full, 0u, STG, p.data_wait_ns};
    const int per = chunk_len(p.V, ch);
    const int lo = min(p.V, c * per), hi = min(p.V, lo + per);
    bool ok;
    ArgBest a{-INFINITY, NO_INDEX};
    ok = true;
    if (row - b * N < n) a = chunk_argmax<VEC>(p.target + (int64_t)row * p.V, lo, hi, red, ring, ok);
    if (tid == 0) {
        part[(int64_t)row * CH_MAX + c] = make_int2(__float_as_int(a.v), ok ? a.i : TIMED_OUT);
        __threadfence();
        last = (atomicAdd(&seq_tick[b], 1) == N * ch - 1);
    }
    __syncthreads();
    if (!last) return;
    // this CTA completed sequence b: reduce every row's chunks (warp w takes
    // rows w, w + 8, ...), then walk the tree
    __threadfence();
    if (tid < N) {
        spar[tid] = par_v;
        stok[tid] = tok_v;
    }
    // lane k holds chunk k (ch <= 32) of each of the warp's rows; all loads are
    // issued before any is used
    int2 pv[64 / CH_WARPS];
#pragma unroll
    for (int q = 0; q < 64 / CH_WARPS; ++q) {
        const int r = warp + q * CH_WARPS;
        pv[q] = (r < N && lane < ch) ? __ldcg(part + ((int64_t)b * N + r) * CH_MAX + lane)
                                     : make_int2(0, NO_INDEX);
    }
#pragma unroll
    for (int q = 0; q < 64 / CH_WARPS; ++q) {
        const int r = warp + q * CH_WARPS;
        if (r >= N) break;
        const int2 v = pv[q];
        ArgBest x{-INFINITY, NO_INDEX};
        if (v.y >= 0 && v.y != NO_INDEX) {
            x.v = __int_as_float(v.x);
            x.i = v.y;
        }
        const bool late = __any_sync(0xffffffffu, v.y == TIMED_OUT);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float w = __shfl_xor_sync(0xffffffffu, x.v, off);
            const int j = __shfl_xor_sync(0xffffffffu, x.i, off);
            if (beats(w, j, x.v, x.i)) {
                x.v = w;
                x.i = j;
            }
        }
        if (lane == 0) sam[r] = late ? TIMED_OUT : (x.i == NO_INDEX) ? -1 : x.i;
    }
    __syncthreads();
    if (tid < 32) {
        int f = check_inputs(spar, stok, n, p.V, N);
        bool late = false;
        for (int k = tid; k < n && f == TV_OK; k += 32) late |= (sam[k] == TIMED_OUT);
        const bool any_late = __any_sync(0xffffffffu, late);
        if (f == TV_OK && any_late) f = TV_ERR_TIMEOUT;
        if (tid == 0) {
            seq_tick[b] = 0;  // leave the workspace ready for the next call
            sflag = f;
        }
    }
    __syncthreads();
    if (sflag != TV_OK) {
        write_fail(p, b, sflag);
        return;
    }
    walk_and_write(p, b, spar, stok, sam, n);
}

// Greedy acceptance, level by level: one cluster of C CTAs per sequence, CTA
// `rank` owns vocabulary slice [rank * per, ...).  Each level streams the
// slice of every frontier row, exchanges the per-CTA argmax through
// distributed shared memory, and keeps the children whose token equals their
// parent's argmax.  All CTAs see the same exchanged values, so they take the
// same decisions and reach every cluster barrier.
template <bool VEC>
__global__ void __launch_bounds__(CH_THREADS)
accept_walk_kernel(AccParams p) {
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    pdl_launch_dependents();
    pdl_wait();
    const int b = blockIdx.x / C;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, Nmax = p.N;
    const int N = seq_count(p, b);  // the sequence's nodes; the rest are absent
    __shared__ int spar[64], stok[64], sam[64];
    __shared__ ArgBest exch[2][64];
    __shared__ ArgBest red[CH_WARPS];
    __shared__ int sflag;
    __shared__ unsigned long long snext;
    if (tid < 64) {
        spar[tid] = (tid < N && tid < Nmax) ? p.parents[(int64_t)b * Nmax + tid] : 0;
        stok[tid] = (tid < N && tid < Nmax) ? p.tokens[(int64_t)b * Nmax + tid] : 0;
        sam[tid] = -1;
    }
    __syncthreads();
    if (tid < 32) {
        const int f = check_inputs(spar, stok, N, p.V, Nmax);
        if (tid == 0) sflag = f;
    }
    __syncthreads();
    if (sflag != TV_OK) {
        if (rank == 0) write_fail(p, b, sflag);
        return;  // uniform across the cluster: no cluster barrier has been issued
    }
    const int per = chunk_len(p.V, C);
    const int lo = min(p.V, rank * per), hi = min(p.V, lo + per);
    uint64_t frontier = 1ull;  // node 0
    int par = 0, chosen = 0, status = TV_OK;
    // each level is one depth deeper, so the walk ends within N levels
    for (int level = 0; level < N; ++level) {
        for (uint64_t f = frontier; f; f &= f - 1) {
            const int u = __ffsll((long long)f) - 1;
            const float* row = p.target + ((int64_t)b * Nmax + u) * p.V;
            ArgBest a;
            if (VEC) {
                a = slice_argmax_ldg(row, lo, hi, red);
            } else {
                a = ArgBest{-INFINITY, NO_INDEX};
                for (int i = lo + tid; i < hi; i += CH_THREADS) take(a, __ldg(row + i), i);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const float w = __shfl_xor_sync(0xffffffffu, a.v, off);
                    const int j = __shfl_xor_sync(0xffffffffu, a.i, off);
                    if (beats(w, j, a.v, a.i)) {
                        a.v = w;
                        a.i = j;
                    }
                }
                if (lane == 0) red[warp] = a;
                __syncthreads();
                a = red[0];
                for (int w = 1; w < CH_WARPS; ++w)
                    if (beats(red[w].v, red[w].i, a.v, a.i)) a = red[w];
            }
            if (tid == 0) exch[par][u] = a;
            __syncthreads();  // red is reused by the next row
        }
        cluster.sync();
        // combine across the cluster: warp w takes frontier nodes w, w + 8, ...;
        // lane r reads rank r's candidate, then a warp argmax
        {
            int idx = 0;
            for (uint64_t f = frontier; f; f &= f - 1, ++idx) {
                if (idx % CH_WARPS != warp) continue;
                const int u = __ffsll((long long)f) - 1;
                ArgBest x{-INFINITY, NO_INDEX};
                if (lane < C) x = *cluster.map_shared_rank(&exch[par][u], lane);
                const bool late = __any_sync(0xffffffffu, x.i == TIMED_OUT);
                if (x.i == TIMED_OUT) x.i = NO_INDEX;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const float w = __shfl_xor_sync(0xffffffffu, x.v, off);
                    const int j = __shfl_xor_sync(0xffffffffu, x.i, off);
                    if (beats(w, j, x.v, x.i)) {
                        x.v = w;
                        x.i = j;
                    }
                }
                if (lane == 0) sam[u] = late ? TIMED_OUT : (x.i == NO_INDEX) ? -1 : x.i;
            }
        }
        __syncthreads();
        // next frontier: children whose token equals their (frontier) parent's argmax
        if (warp == 0) {
            uint64_t next = 0;
            bool late = false;
            for (int c0 = 0; c0 < N; c0 += 32) {
                const int c = c0 + lane;
                bool hit = false;
                if (c < N) {
                    late |= ((frontier >> c) & 1ull) && sam[c] == TIMED_OUT;
                    if (c >= 1) {
                        const int pc = spar[c];
                        hit = ((frontier >> pc) & 1ull) && sam[pc] >= 0 && stok[c] == sam[pc];
                    }
                }
                next |= (uint64_t)__ballot_sync(0xffffffffu, hit) << c0;
            }
            const bool any_late = __any_sync(0xffffffffu, late);  // every lane votes
            if (lane == 0) snext = any_late ? ~0ull : next;
        } 
        __syncthreads();
        const uint64_t next = snext;
        if (next == ~0ull) {
            status = TV_ERR_TIMEOUT;
            break;
        }
        if (next == 0) {
            chosen = __ffsll((long long)frontier) - 1;
            break;
        }
        frontier = next;
        par ^= 1;
    }
    cluster.sync();  // no CTA leaves while others may still read its exchange slots
    if (rank == 0) {
        if (status != TV_OK) write_fail(p, b, status);
        else if (sam[chosen] < 0) write_fail(p, b, TV_ERR_BAD_VALUES);
        else write_path(p, b, spar, stok, chosen, sam[chosen]);
    }
}

// Weights of a pair of values (x0, x1) added to the running part sums, exactly:
// with y = min(max(x, 0), 1) (NaN -> 0) and t = y * 2^16, the weight
// floor(y * 2^40) = H * 2^24 + L, H = floor(t) and L = floor((t - H) * 2^24) < 2^24.
// H is taken with one round-down add of 2^23 (t <= 2^16, so the sum's unit is
// 1); (t - H) * 2^24 is exact (one fma), and L its truncation.  H sums stay
// exact in fp32 for up to 256 values, L sums in 32 bits for up to 256.
__device__ __forceinline__ void weight_pair_acc(float x0, float x1, uint64_t& hacc, uint32_t& lacc) {
    const uint64_t C23 = 0x4B0000004B000000ull;                  // (2^23, 2^23)
    const uint64_t y = f2_pack(fminf(fmaxf(x0, 0.f), 1.f), fminf(fmaxf(x1, 0.f), 1.f));
    const uint64_t t = f2_mul(y, 0x4780000047800000ull);        // * 2^16
    const uint64_t h = f2_add(f2_add_rm(t, C23), 0xCB000000CB000000ull);  // floor(t)
    const uint64_t r = f2_fma(h, 0xCB800000CB800000ull, f2_mul(t, 0x4B8000004B800000ull));  // (t - H) 2^24
    float r0, r1;
    f2_unpack(r, r0, r1);
    lacc += __float2uint_rz(r0) + __float2uint_rz(r1);
    hacc = f2_add(hacc, h);
}

// Piece sums of the weights of a (RESID: of a - b) over [lo, hi), each warp
// taking whole pieces: eight 16-byte streaming loads per row and lane in
// flight, exact part sums per lane (64 values each), one 64-bit shuffle
// reduction per piece.
template <bool RESID>
__device__ __forceinline__ void warp_piece_sums(const float* a, const float* bq, int lo, int hi,
                                                int np, uint64_t* psum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float4* a4 = reinterpret_cast<const float4*>(a);
    const float4* b4 = reinterpret_cast<const float4*>(bq);
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = warp; k < np; k += CH_WARPS) {
        const int off = lo + k * PIECE;
        const int n4 = min(PIECE, hi - off) >> 2;  // float4s in this piece
        const int o4 = off >> 2;
        uint64_t hacc = 0;  // (0.f, 0.f)
        uint32_t lacc = 0;
#pragma unroll 1
        for (int r0 = 0; r0 < PIECE / 128; r0 += 8) {
            float4 x[8], y[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = lane + 32 * (r0 + i);
                x[i] = (e < n4) ? __ldcs(a4 + o4 + e) : z4;
                if (RESID) y[i] = (e < n4) ? __ldcs(b4 + o4 + e) : z4;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (RESID) {
                    weight_pair_acc(__fsub_rn(x[i].x, y[i].x), __fsub_rn(x[i].y, y[i].y), hacc, lacc);
                    weight_pair_acc(__fsub_rn(x[i].z, y[i].z), __fsub_rn(x[i].w, y[i].w), hacc, lacc);
                } else {
                    weight_pair_acc(x[i].x, x[i].y, hacc, lacc);
                    weight_pair_acc(x[i].z, x[i].w, hacc, lacc);
                }
            }
        }
        float h0, h1;
        f2_unpack(hacc, h0, h1);
        uint64_t w = (((uint64_t)__float2uint_rz(h0) + __float2uint_rz(h1)) << 24) + lacc;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
        if (lane == 0) psum[off / PIECE] = w;
    }
}

// Integer weights of row a over [lo, hi) (weight(a - b) when b is given, the
// residual; weight(a) otherwise): the sum of every PIECE-element piece k goes
// to psum[k] (global).  lo is a multiple of PIECE.  Every thread of the CTA
// calls it.  VEC (rows 16-byte aligned, lengths multiples of 4): each warp
// owns whole pieces (k = warp, warp + 8, ...), every lane keeps eight 16-byte
// streaming loads per row in flight and the warp reduces its sums with
// shuffles, so no piece waits on a CTA barrier and no shared memory is used.
template <bool VEC>
__device__ void piece_weight_sums(const float* a, const float* bq, int lo, int hi,
                                  uint64_t (*red)[CH_WARPS], uint64_t* psum) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool resid = bq != nullptr;
    const int np = (hi - lo + PIECE - 1) / PIECE;
    if (!VEC) {
        for (int k = 0; k < np; ++k) {
            const int off = lo + k * PIECE, end = min(hi, off + PIECE);
            uint64_t w = 0;
            for (int i = off + tid; i < end; i += CH_THREADS) w += elem_weight(a, bq, i, resid);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
            if (lane == 0) red[0][warp] = w;
            __syncthreads();
            if (tid == 0) {
                uint64_t t = 0;
                for (int q = 0; q < CH_WARPS; ++q) t += red[0][q];
                psum[(off) / PIECE] = t;
            }
            __syncthreads();
        }
        return;
    }
    if (resid) warp_piece_sums<true>(a, bq, lo, hi, np, psum);
    else warp_piece_sums<false>(a, bq, lo, hi, np, psum);
    __syncthreads();  // every piece sum of the CTA is written
}

// Picks the index holding the draw among n values v(k) from `get` (a prefix
// of k = 0.. in order); one full warp; returns the index (-1 when the total is
// zero) and the offset T inside it, in every lane.
template <typename Get>
__device__ int pick_index(int n, uint32_t x1, Get get, uint64_t& T) {
    const int lane = threadIdx.x & 31;
    uint64_t tot = 0;
    for (int k = lane; k < n; k += 32) tot += get(k);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
    T = 0;
    if (tot == 0) return -1;
    const uint64_t hi = __umul64hi((uint64_t)x1, tot), lo = (uint64_t)x1 * tot;
    uint64_t t = (hi << 32) | (lo >> 32);
    for (int k0 = 0; k0 < n; k0 += 32) {
        const uint64_t v = (k0 + lane < n) ? get(k0 + lane) : 0ull;
        uint64_t x = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint64_t y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        const uint64_t grp = __shfl_sync(0xffffffffu, x, 31);
        if (t < grp) {
            const int l = __ffs(__ballot_sync(0xffffffffu, x > t)) - 1;
            T = t - __shfl_sync(0xffffffffu, x - v, l);
            return k0 + l;
        }
        t -= grp;
    }
    return -1;  // not reached: t < total
}

// Smallest index i in [lo, hi) whose inclusive prefix sum of weights (from lo)
// exceeds T, for T below the range's sum; the whole CTA searches, the result
// is valid in thread 0.  Level 1: sums of 256-element tiles (one warp per
// tile); level 2: one warp scans the tile sums, then the chosen tile's
// elements, eight per lane.
__device__ int chunk_find(const float* a, const float* bq, int lo, int hi, uint64_t T,
                          uint64_t* tsum /* [>= ceil((hi-lo)/256)] */) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool resid = bq != nullptr;
    constexpr int TILE = 256;
    const int nt = (hi - lo + TILE - 1) / TILE;
    for (int t = warp; t < nt; t += CH_WARPS) {
        const int base = lo + t * TILE + lane * 8;
        uint64_t acc = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (base + k < hi) acc += elem_weight(a, bq, base + k, resid);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) tsum[t] = acc;
    }
    __syncthreads();
    __shared__ int sfound;
    if (warp == 0) {
        // tile containing T: lane-strided partial sums, then a warp scan
        int tile = -1;
        uint64_t rem = T;
        for (int t0 = 0; t0 < nt && tile < 0; t0 += 32) {
            const uint64_t v = (t0 + lane < nt) ? tsum[t0 + lane] : 0ull;
            uint64_t x = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint64_t y = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off) x += y;
            }
            const uint64_t tot = __shfl_sync(0xffffffffu, x, 31);
            if (rem < tot) {
                const unsigned hit = __ballot_sync(0xffffffffu, x > rem);
                const int l = __ffs(hit) - 1;
                const uint64_t before = __shfl_sync(0xffffffffu, x - v, l);
                tile = t0 + l;
                rem -= before;
            } else {
                rem -= tot;
            }
        }
        int found = -1;
        if (tile >= 0) {
            // eight consecutive elements per lane, a warp scan over the lane sums
            const int base = lo + tile * TILE + lane * 8;
            uint64_t wv[8];
            uint64_t ls = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                wv[k] = (base + k < hi) ? elem_weight(a, bq, base + k, resid) : 0ull;
                ls += wv[k];
            }
            uint64_t x = ls;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint64_t y = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off) x += y;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, x > rem);
            const int l = __ffs(hit) - 1;
            if (lane == l) {
                uint64_t run = x - ls;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    run += wv[k];
                    if (found < 0 && run > rem) found = base + k;
                }
            }
            found = __shfl_sync(0xffffffffu, found, l < 0 ? 0 : l);
        }
        if (lane == 0) sfound = found;
    }
    __syncthreads();
    return sfound;
}

// Stochastic acceptance on a branching tree (multi-candidate rejection
// sampling: the children of the current node are tried in node order), one
// cluster of C CTAs per sequence, CTA `rank` owning vocabulary slice
// [rank * per, ...).  The first child of a node takes the chain's exact test;
// after a rejection the target is the residual max(0, p - q) kept as exact
// integer weights: after the first rejected child c, w_t = weight(p_cur,t -
// q_c,t); after each further one c', w_t <- max(0, w_t - floor(weight(q_c',t)
// * S / 2^40)) with S the sum before.  A later child c' is accepted iff u24 *
// weight(q_c'(x)) * S < w_x * 2^64.  All children rejected: the token is drawn
// from the residual (from the target row when it has no mass) with word 1 of
// the last rejected child's draw; a leaf: the bonus token from the target row
// with word 1 of draw N (leaf N-1) or N + leaf.  N: the sequence's node count
// (rows keep the batch's stride p.N).
//
// The residual is recomputed entry by entry from the rows.  Every pass over the
// vocabulary (a residual sum, the draw) is split over the cluster: each CTA
// reduces its slice, the partial sums are exchanged through distributed shared
// memory and added in rank order, so every CTA holds the same exact integer
// sums, takes the same decisions and reaches every cluster barrier.  The CTA
// whose slice holds the draw finds the token with block scans and posts it to
// rank 0, which writes the result.  Chains and invalid inputs are left to
// accept_stochastic_kernel, launched just before on the same stream.
constexpr int TW_U = 8;                         // 16-byte positions per thread per tile
constexpr int TW_TILE = TW_U * CH_THREADS * 4;  // vocabulary entries per tile

template <bool VEC>
__global__ void __launch_bounds__(CH_THREADS)
accept_stochastic_tree_kernel(AccParams p) {
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    pdl_launch_dependents();
    pdl_wait();
    const int b = blockIdx.x / C;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, Nmax = p.N, V = p.V;
    const int N = seq_count(p, b);
    __shared__ int spar[64], stok[64];
    __shared__ int sflag, schain, sfound, xtok;
    __shared__ int rj[64];          // rejected children of the current node, in order
    __shared__ uint64_t rS[64];     // residual sum after each of those rejections
    __shared__ uint64_t tred[CH_WARPS];
    __shared__ uint64_t xpart[2];   // this slice's sum, by pass parity (read by the cluster)
    __shared__ uint64_t gsum[CH_WARPS * TW_U];  // the draw: each warp's total of each group
    if (tid < 64) {
        spar[tid] = (tid < N && tid < Nmax) ? p.parents[(int64_t)b * Nmax + tid] : 0;
        stok[tid] = (tid < N && tid < Nmax) ? p.tokens[(int64_t)b * Nmax + tid] : 0;
    }
    if (tid == 0) xtok = -1;
    __syncthreads();
    if (tid < 32) {
        const int f = check_inputs(spar, stok, N, V, Nmax);
        bool branch = false;
        if (f == TV_OK)
            for (int i = lane; i < N; i += 32) branch |= (i > 0 && spar[i] != i - 1);
        branch = __any_sync(0xffffffffu, branch);
        if (tid == 0) {
            sflag = f;
            schain = !branch;
        }
    }
    __syncthreads();
    // uniform across the cluster, before its first barrier
    if (sflag != TV_OK || schain) return;

    const int per = chunk_len(V, C);
    const int lo = min(V, rank * per), hi = min(V, lo + per);
    const float* tgt = p.target + (int64_t)b * Nmax * V;
    const float* drf = p.draft + (int64_t)b * Nmax * V;
    auto sub_floor = [](uint64_t w, uint64_t qw, uint64_t S) -> uint64_t {
        const uint64_t d = (__umul64hi(qw, S) << 24) | ((qw * S) >> 40);  // floor(qw * S / 2^40)
        return w > d ? w - d : 0ull;
    };
    // weight of entry t: the target row pc (m == 0) or the residual after m rejections
    auto wt = [&](const float* pc, int m, int t) -> uint64_t {
        if (m == 0) return weight(__ldg(pc + t));
        uint64_t w = weight(__fsub_rn(__ldg(pc + t), __ldg(drf + (int64_t)rj[0] * V + t)));
        for (int j = 1; j < m; ++j)
            w = sub_floor(w, weight(__ldg(drf + (int64_t)rj[j] * V + t)), rS[j - 1]);
        return w;
    };
    // this thread's entries of the tile at `base`: position u holds entries
    // base + (u * CH_THREADS + tid) * 4 + 0..3, read as 0 outside [lo, hi); one
    // row's loads are all issued before any is used
    auto load_tile = [&](const float* row, int base, float (&a)[TW_U][4]) {
#pragma unroll
        for (int u = 0; u < TW_U; ++u) {
            const int t = base + (u * CH_THREADS + tid) * 4;
            if (VEC) {  // hi is a multiple of 4 here
                const float4 v = (t < hi) ? __ldg(reinterpret_cast<const float4*>(row + t))
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
                a[u][0] = v.x;
                a[u][1] = v.y;
                a[u][2] = v.z;
                a[u][3] = v.w;
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) a[u][c] = (t + c < hi) ? __ldg(row + t + c) : 0.f;
            }
        }
    };
    auto tile_weights = [&](const float* pc, int m, int base, uint64_t (&w)[TW_U][4]) {
        float a[TW_U][4];
        load_tile(pc, base, a);
        if (m == 0) {
#pragma unroll
            for (int u = 0; u < TW_U; ++u)
#pragma unroll
                for (int c = 0; c < 4; ++c) w[u][c] = weight(a[u][c]);
            return;
        }
        float q[TW_U][4];
        load_tile(drf + (int64_t)rj[0] * V, base, q);
#pragma unroll
        for (int u = 0; u < TW_U; ++u)
#pragma unroll
            for (int c = 0; c < 4; ++c) w[u][c] = weight(__fsub_rn(a[u][c], q[u][c]));
        for (int j = 1; j < m; ++j) {
            load_tile(drf + (int64_t)rj[j] * V, base, q);
            const uint64_t S = rS[j - 1];
#pragma unroll
            for (int u = 0; u < TW_U; ++u)
#pragma unroll
                for (int c = 0; c < 4; ++c) w[u][c] = sub_floor(w[u][c], weight(q[u][c]), S);
        }
    };
    // the sum over the vocabulary of the weights (pc, m); `before`: the sum over
    // the slices of lower ranks, `mine`: over this slice
    int par = 0;
    auto cluster_sum = [&](const float* pc, int m, uint64_t& before, uint64_t& mine) -> uint64_t {
        uint64_t acc = 0;
        for (int base = lo; base < hi; base += TW_TILE) {
            uint64_t w[TW_U][4];
            tile_weights(pc, m, base, w);
#pragma unroll
            for (int u = 0; u < TW_U; ++u) acc += (w[u][0] + w[u][1]) + (w[u][2] + w[u][3]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) tred[warp] = acc;
        __syncthreads();
        uint64_t own = 0;
#pragma unroll
        for (int i = 0; i < CH_WARPS; ++i) own += tred[i];
        if (tid == 0) xpart[par] = own;
        cluster.sync();  // also orders every thread's reads of tred before its next writes
        const uint64_t x = (lane < C) ? *cluster.map_shared_rank(&xpart[par], lane) : 0ull;
        uint64_t tot = x, bef = (lane < rank) ? x : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            tot += __shfl_xor_sync(0xffffffffu, tot, o);
            bef += __shfl_xor_sync(0xffffffffu, bef, o);
        }
        par ^= 1;  // the slot read here is rewritten only after the next barrier
        before = bef;
        mine = own;
        return tot;
    };
    // the draw from weights (pc, m) with sum S > 0: the smallest t whose
    // inclusive prefix sum exceeds T = floor(x * S / 2^32), returned to rank 0
    auto sample = [&](const float* pc, int m, uint64_t S, uint64_t before, uint64_t mine,
                      uint32_t x) -> int {
        const uint64_t T = (uint64_t)x * (S >> 32) + (((uint64_t)x * (S & 0xffffffffull)) >> 32);
        if (before <= T && T - before < mine) {  // this slice holds it (one CTA does)
            if (tid == 0) sfound = -1;
            uint64_t run = before;
            for (int base = lo; base < hi; base += TW_TILE) {
                uint64_t w[TW_U][4];
                tile_weights(pc, m, base, w);
                // the tile's groups (group u: entries base + u * 4 * CH_THREADS onwards,
                // four a thread) are totalled in one reduction, and only the group
                // holding T is scanned
                uint64_t s4[TW_U];
#pragma unroll
                for (int u = 0; u < TW_U; ++u) {
                    s4[u] = (w[u][0] + w[u][1]) + (w[u][2] + w[u][3]);
                    uint64_t v = s4[u];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == 0) gsum[warp * TW_U + u] = v;
                }
                __syncthreads();
                int gu = -1;
                uint64_t gbase = 0;
#pragma unroll
                for (int u = 0; u < TW_U; ++u) {
                    uint64_t t = 0;
#pragma unroll
                    for (int i = 0; i < CH_WARPS; ++i) t += gsum[i * TW_U + u];
                    if (gu < 0 && run <= T && T - run < t) {
                        gu = u;
                        gbase = run;
                    }
                    run += t;
                }
                __syncthreads();  // every read of gsum and tred is done
                if (gu < 0) continue;  // uniform: T lies in a later tile
                uint64_t e4[4] = {0ull, 0ull, 0ull, 0ull}, t4 = 0;
#pragma unroll
                for (int u = 0; u < TW_U; ++u) {
                    if (u == gu) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) e4[c] = w[u][c];
                        t4 = s4[u];
                    }
                }
                uint64_t incl = t4;  // inclusive scan over the warp's lanes
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint64_t y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                if (lane == 31) tred[warp] = incl;
                __syncthreads();
                uint64_t wpre = 0;
#pragma unroll
                for (int i = 0; i < CH_WARPS; ++i) wpre += (i < warp) ? tred[i] : 0ull;
                const uint64_t ex = gbase + wpre + (incl - t4);
                if (ex <= T && T - ex < t4) {  // this thread's four entries hold it
                    uint64_t r = ex;
                    int hit = -1;  // the first entry whose inclusive prefix exceeds T
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        r += e4[c];
                        if (hit < 0 && r > T) hit = c;
                    }
                    sfound = base + (gu * CH_THREADS + tid) * 4 + hit;
                }
                __syncthreads();
                break;  // uniform
            }
            if (tid == 0) *cluster.map_shared_rank(&xtok, 0) = sfound;
        }
        cluster.sync();
        return xtok;
    };

    int cur = 0, token = -1;
    for (;;) {
        const float* pc = tgt + (int64_t)cur * V;
        int m = 0, next = -1, last_rej = -1;
        uint64_t S = 0, before = 0, mine = 0;
        for (int c = cur + 1; c < N; ++c) {
            if (spar[c] != cur) continue;
            const uint32_t u24 = draw(p, b, c).x >> 8;
            const int x = stok[c];
            const float qx = __ldg(drf + (int64_t)c * V + x);
            bool acc;
            if (m == 0) {
                acc = __dmul_rn((double)u24, (double)qx) < __dmul_rn((double)__ldg(pc + x), 16777216.0);
            } else {
                const uint64_t A = (uint64_t)u24 * weight(qx);  // < 2^64
                acc = __umul64hi(A, S) < wt(pc, m, x);
            }
            if (acc) {
                next = c;
                break;
            }
            __syncthreads();  // earlier readers of rj / rS are done
            if (tid == 0) rj[m] = c;
            __syncthreads();
            S = cluster_sum(pc, m + 1, before, mine);
            if (tid == 0) rS[m] = S;
            __syncthreads();
            ++m;
            last_rej = c;
            if (S == 0) break;
        }
        if (next >= 0) {
            cur = next;
            continue;
        }
        // a leaf: the bonus token from the target row; all children rejected: from
        // the residual, or from the target row when the residual has no mass
        const uint32_t x1 = (last_rej < 0) ? draw(p, b, (cur == N - 1) ? N : N + cur).y
                                           : draw(p, b, last_rej).y;
        if (last_rej < 0 || S == 0) {
            m = 0;
            S = cluster_sum(pc, 0, before, mine);
        }
        token = (S > 0) ? sample(pc, m, S, before, mine, x1) : -1;
        break;
    }
    cluster.sync();  // no CTA leaves while another may still read its shared memory
    if (rank == 0) {
        if (token < 0) write_fail(p, b, TV_ERR_BAD_VALUES);
        else write_path(p, b, spar, stok, cur, token);
    }
}

// Stochastic chain acceptance: CTA (b, c) takes chunk c of the row the token
// is drawn from; ws: sums[b][ceil(V / PIECE)] (weight sum of every piece), seq_tick[b].
// A sequence whose tree is not a chain is left to accept_stochastic_tree_kernel.
template <bool VEC>
__global__ void __launch_bounds__(CH_THREADS, 3)
accept_stochastic_kernel(AccParams p, int ch, uint64_t* __restrict__ sums,
                         int32_t* __restrict__ seq_tick) {
    pdl_launch_dependents();
    pdl_wait();
    const int b = blockIdx.x / ch, c = blockIdx.x % ch;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, Nmax = p.N;
    const int N = seq_count(p, b);  // the sequence's nodes; the rest are absent
    __shared__ int spar[64], stok[64];
    __shared__ int sflag, skstar, last, schain;
    __shared__ uint64_t red[STG][CH_WARPS];
    __shared__ uint64_t tsum[PIECE / 256];
    if (tid < N && tid < Nmax) {
        spar[tid] = p.parents[(int64_t)b * Nmax + tid];
        stok[tid] = p.tokens[(int64_t)b * Nmax + tid];
    }
    __syncthreads();
    if (tid < 32) {
        const int f = check_inputs(spar, stok, N, p.V, Nmax);
        bool branch = false;
        for (int i = lane; i < N; i += 32) branch |= (i > 0 && spar[i] != i - 1);
        branch = __any_sync(0xffffffffu, branch);
        if (tid == 0) {
            sflag = f;
            schain = !branch;
        }
    }
    __syncthreads();
    if (sflag != TV_OK) {
        if (c == 0) write_fail(p, b, sflag);
        return;  // every CTA of the sequence returns here: its counter is untouched
    }
    if (!schain) return;  // the tree kernel walks it; the counter is untouched
    // accept tests k = 1..K, all at once (counter-based draws); the first failure wins
    const int K = N - 1;
    if (warp == 0) {
        int kst = K + 1;  // first rejected position, K+1 = none
        for (int k0 = 1; k0 <= K && kst > K; k0 += 32) {
            const int k = k0 + lane;
            bool acc = true;
            if (k <= K) {
                const uint32_t u24 = draw(p, b, k).x >> 8;
                const int x = stok[k];
                const float pk = __ldg(p.target + ((int64_t)b * Nmax + (k - 1)) * p.V + x);
                const float qk = __ldg(p.draft + ((int64_t)b * Nmax + k) * p.V + x);
                acc = __dmul_rn((double)u24, (double)qk) < __dmul_rn((double)pk, 16777216.0);
            }
            const unsigned rej = __ballot_sync(0xffffffffu, !acc);
            if (rej) kst = k0 + __ffs(rej) - 1;
        }
        if (lane == 0) skstar = kst;
    }
    __syncthreads();
    const int kstar = skstar;
    const bool rejected = kstar <= K;
    const float* rowa = p.target + ((int64_t)b * Nmax + (rejected ? kstar - 1 : K)) * p.V;
    const float* rowb = rejected ? p.draft + ((int64_t)b * Nmax + kstar) * p.V : nullptr;
    // chunk c: whole pieces [lo, hi); piece sums of sequence b at psum[b][*]
    const int np_all = (p.V + PIECE - 1) / PIECE;
    const int per = ((np_all + ch - 1) / ch) * PIECE;
    uint64_t* psum = sums + (int64_t)b * np_all;
    {
        const int lo = min(p.V, c * per), hi = min(p.V, lo + per);
        piece_weight_sums<VEC>(rowa, rowb, lo, hi, red, psum);
        if (tid == 0) {
            __threadfence();
            last = (atomicAdd(&seq_tick[b], 1) == ch - 1);
        }
    }
    __syncthreads();
    if (!last) return;
    // this CTA completed sequence b: pick the piece holding the draw
    __threadfence();
    __shared__ int spiece, sresid;
    __shared__ uint64_t sT;
    const uint32_t x1 = draw(p, b, rejected ? kstar : K + 1).y;
    if (warp == 0) {
        uint64_t T = 0;
        const int pi = pick_index(np_all, x1, [&](int k) { return __ldcg(psum + k); }, T);
        if (lane == 0) {
            seq_tick[b] = 0;  // leave the workspace ready for the next call
            spiece = pi;
            sT = T;
            sresid = rejected;
        }
    }
    __syncthreads();
    if (rejected && spiece < 0) {
        // the residual has no mass: draw from the target row itself (rare: this
        // CTA sums every piece of it)
        piece_weight_sums<VEC>(rowa, nullptr, 0, p.V, red, psum);
        __threadfence();
        __syncthreads();  // thread 0's piece sums are visible to warp 0
        if (warp == 0) {
            uint64_t T = 0;
            const int pi = pick_index(np_all, x1, [&](int k) { return __ldcg(psum + k); }, T);
            if (lane == 0) {
                spiece = pi;
                sT = T;
                sresid = 0;
            }
        }
        __syncthreads();
    }
    int token = -1;
    if (spiece >= 0) {
        const int lo = spiece * PIECE, hi = min(p.V, lo + PIECE);
        token = chunk_find(rowa, sresid ? rowb : nullptr, lo, hi, sT, tsum);
    }
    if (token < 0) write_fail(p, b, TV_ERR_BAD_VALUES);
    else write_path(p, b, spar, stok, rejected ? kstar - 1 : K, token);
}

// The row scan pays for every row once at full bandwidth; the walk pays a few
// microseconds of latency per tree level (at most 8 levels assumed).
bool prefer_rowscan(int B, int N, int V) {
    const double bytes = (double)B * N * V * 4.0;
    const double t_scan = bytes / 6.0e12 + 3.0e-6;
    const double t_walk = (double)(N < 8 ? N : 8) * 2.5e-6;
    return t_scan < t_walk;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// CTAs of `kern` resident on the whole device with `smem` dynamic bytes.
template <typename K>
int64_t resident_ctas(K kern, size_t smem, int sms) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, CH_THREADS, smem) != cudaSuccess) {
        cudaGetLastError();
        n = 1;
    }
    return (int64_t)std::max(n, 1) * sms;
}

// Chunks per row: as many as keep all `rows` x chunks CTAs resident at once
// (one wave), with at least one piece per chunk.
int chunks_for(int64_t rows, int V, int64_t resident) {
    int64_t ch = std::max<int64_t>(1, resident / rows);
    ch = std::min<int64_t>(ch, std::max(1, (V + PIECE - 1) / PIECE));
    return (int)std::min<int64_t>(ch, CH_MAX);
}

struct RowsWs {
    size_t part, seq_tick, total;
};
RowsWs rows_ws(int B, int N) {
    const size_t R = (size_t)B * N;
    RowsWs w;
    w.part = 0;
    w.seq_tick = w.part + align256(R * CH_MAX * 8);
    w.total = w.seq_tick + align256((size_t)B * 4);
    return w;
}
constexpr size_t ROWS_SMEM = (size_t)STG * PIECE * 4 + 1024;       // ring, one operand

using AccKernel = void (*)(AccParams);

// Clusters of cs CTAs of a cluster kernel (given by its two instantiations)
// that can be resident at once (0: cannot launch); cache[cs] keeps the answer.
int resident_clusters(AccKernel kv, AccKernel ks, int cs, int* cache) {
    if (cs < 1 || cs > 16) return 0;
    if (cache[cs] >= 0) return cache[cs];
    int n = 0;
    bool ok = true;
    if (cs > 8)
        ok = cudaFuncSetAttribute(kv, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                 cudaSuccess &&
             cudaFuncSetAttribute(ks, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                 cudaSuccess;
    if (ok) {
        LaunchCfg lc(dim3(cs), dim3(CH_THREADS), 0, nullptr, (unsigned)cs);
        lc.cfg.numAttrs = 1;  // the cluster shape only
        if (cudaOccupancyMaxActiveClusters(&n, kv, &lc.cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
    cache[cs] = n;
    return n;
}

// Largest cluster (at most 16 CTAs, at least PIECE vocabulary entries per CTA)
// whose B clusters are resident at once; else the largest that launches.
int cluster_size_for(AccKernel kv, AccKernel ks, int* cache, int B, int V) {
    int fallback = 0;
    for (int cs = 16; cs >= 1; cs >>= 1) {
        if (cs > 1 && (int64_t)V < (int64_t)cs * PIECE) continue;
        const int n = resident_clusters(kv, ks, cs, cache);
        if (n <= 0) continue;
        if (n >= B) return cs;
        if (fallback == 0) fallback = cs;
    }
    return fallback;
}

int walk_cluster_size(int B, int V) {
    static int cache[17] = {-1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1};
    return cluster_size_for(accept_walk_kernel<true>, accept_walk_kernel<false>, cache, B, V);
}

int tree_cluster_size(int B, int V) {
    static int cache[17] = {-1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1};
    return cluster_size_for(accept_stochastic_tree_kernel<true>,
                            accept_stochastic_tree_kernel<false>, cache, B, V);
}

size_t stoch_ws_sums(int B, int V) { return align256((size_t)B * ((V + PIECE - 1) / PIECE) * 8); }

}  // namespace

size_t accept_workspace(tv_accept_mode mode, int B, int N, int V) {
    if (B <= 0) return 0;
    if (mode == TV_ACCEPT_GREEDY)
        return prefer_rowscan(B, N, V) ? rows_ws(B, N).total : 0;
    return stoch_ws_sums(B, V) + align256((size_t)B * 4);
}

tv_status launch_accept(const AcceptArgs& a) {
    if (a.B == 0) return TV_OK;
    AccParams p;
    p.parents = a.parents;
    p.tokens = a.tokens;
    p.target = a.target;
    p.draft = a.draft;
    p.B = a.B;
    p.N = a.N;
    p.V = a.V;
    p.seed = a.seed;
    p.offset = a.offset;
    p.accept_len = a.accept_len;
    p.path = a.path;
    p.out_tokens = a.out_tokens;
    p.max_path = a.max_path;
    p.status = a.status;
    p.counts = a.counts;
    // Test-only: TV_TEST_DATA_WAIT_NS shortens the row scan's waits for streamed
    // data (never the waits that drain copies still in flight), so a test can
    // make a legitimate wait run out and check the TV_ERR_TIMEOUT status.
    p.data_wait_ns = TV_WAIT_NS;
    if (const char* e = getenv("TV_TEST_DATA_WAIT_NS")) {
        const unsigned long long v = strtoull(e, nullptr, 10);
        if (v > 0 && v < TV_WAIT_NS) p.data_wait_ns = v;
    }
    const int sms = device_sm_count();
    const bool aligned = (reinterpret_cast<uintptr_t>(a.target) & 15) == 0 &&
                         (reinterpret_cast<uintptr_t>(a.draft) & 15) == 0;
    const bool vec = (a.V % 4 == 0) && aligned;
    const size_t need = accept_workspace(a.mode, a.B, a.N, a.V);
    if (need > 0 && (a.ws == nullptr || a.ws_bytes < need)) return TV_ERR_WORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    cudaError_t e;
    if (a.mode == TV_ACCEPT_GREEDY && need > 0) {
        const int64_t R = (int64_t)a.B * a.N;
        static int64_t cap = -1;
        if (cap < 0) cap = resident_ctas(accept_rows_kernel<true>, ROWS_SMEM, sms);
        const int ch = std::min(32, chunks_for(R, a.V, cap));  // one chunk per lane when reduced
        if (R * ch > 0x7fffffff) return TV_ERR_UNSUPPORTED;
        const RowsWs w = rows_ws(a.B, a.N);
        int2* part = reinterpret_cast<int2*>(ws + w.part);
        int32_t* st = reinterpret_cast<int32_t*>(ws + w.seq_tick);
        LaunchCfg lc(dim3((unsigned)(R * ch)), dim3(CH_THREADS), vec ? ROWS_SMEM : 0, a.stream);
        e = vec ? cudaLaunchKernelEx(&lc.cfg, accept_rows_kernel<true>, p, ch, part, st)
                : cudaLaunchKernelEx(&lc.cfg, accept_rows_kernel<false>, p, ch, part, st);
    } else if (a.mode == TV_ACCEPT_GREEDY) {
        const int C = walk_cluster_size(a.B, a.V);
        if (C <= 0) return TV_ERR_CUDA;
        if ((int64_t)a.B * C > 0x7fffffff) return TV_ERR_UNSUPPORTED;
        LaunchCfg lc(dim3((unsigned)(a.B * C)), dim3(CH_THREADS), 0, a.stream, (unsigned)C);
        e = vec ? cudaLaunchKernelEx(&lc.cfg, accept_walk_kernel<true>, p)
                : cudaLaunchKernelEx(&lc.cfg, accept_walk_kernel<false>, p);
    } else {
        static int64_t cap = -1;
        if (cap < 0) cap = resident_ctas(accept_stochastic_kernel<true>, 0, sms);
        const int ch = chunks_for(a.B, a.V, cap);
        if ((int64_t)a.B * ch > 0x7fffffff) return TV_ERR_UNSUPPORTED;
        uint64_t* sums = reinterpret_cast<uint64_t*>(ws);
        int32_t* st = reinterpret_cast<int32_t*>(ws + stoch_ws_sums(a.B, a.V));
        LaunchCfg lc(dim3((unsigned)(a.B * ch)), dim3(CH_THREADS), 0, a.stream);
        e = vec ? cudaLaunchKernelEx(&lc.cfg, accept_stochastic_kernel<true>, p, ch, sums, st)
                : cudaLaunchKernelEx(&lc.cfg, accept_stochastic_kernel<false>, p, ch, sums, st);
        // branching trees: one cluster per sequence, after the chains (every tree
        // of at most two nodes is a chain)
        if (e == cudaSuccess && a.N > 2) {
            const int C = tree_cluster_size(a.B, a.V);
            if (C <= 0) return TV_ERR_CUDA;
            if ((int64_t)a.B * C > 0x7fffffff) return TV_ERR_UNSUPPORTED;
            LaunchCfg lt(dim3((unsigned)(a.B * C)), dim3(CH_THREADS), 0, a.stream, (unsigned)C);
            e = vec ? cudaLaunchKernelEx(&lt.cfg, accept_stochastic_tree_kernel<true>, p)
                    : cudaLaunchKernelEx(&lt.cfg, accept_stochastic_tree_kernel<false>, p);
        }
    }
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

}  // namespace tv
