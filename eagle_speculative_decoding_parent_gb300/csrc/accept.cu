// tree_accept: one thread-block cluster per sequence.
//
// Each CTA of the cluster owns a contiguous slice of the vocabulary.  Only
// the rows the acceptance rule needs are read:
//   greedy      a level-by-level walk from the root: the argmax of every row
//               on the current frontier of fully matching nodes (usually one)
//               is reduced inside each CTA, exchanged through distributed
//               shared memory, and the matching children form the next
//               frontier; the walk stops at the deepest accepted level, whose
//               argmax is the bonus token.  Rows read ~ accepted depth + 1.
//   stochastic  the accept tests touch two scalars per draft; only the row(s)
//               the emitted token is drawn from are read: integer weights
//               (exact sums, so the draw does not depend on summation order),
//               slice sums exchanged across the cluster, and the CTA holding
//               the target prefix sum scans its slice.
// All CTAs of a cluster take identical control-flow decisions (they read the
// same inputs and the same exchanged values), so every cluster barrier is
// reached by every CTA.
#include <cooperative_groups.h>

#include "tv_device.cuh"
#include "tv_internal.h"

namespace cg = cooperative_groups;

namespace tv {

namespace {

constexpr int ACC_THREADS = 512;
constexpr int ACC_WARPS = ACC_THREADS / 32;
constexpr int NO_INDEX = 0x7fffffff;

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
};

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

__device__ __forceinline__ void take4(ArgBest& a, const float4& x, int i) {
    take(a, x.x, i);
    take(a, x.y, i + 1);
    take(a, x.z, i + 2);
    take(a, x.w, i + 3);
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

// Fixed-point weight floor(min(x, 1) * 2^40); 0 for NaN and x <= 0.
__device__ __forceinline__ uint64_t weight(float x) {
    if (!(x > 0.f)) return 0ull;
    if (x >= 1.f) return 1ull << 40;
    return __float2ull_rz(__fmul_rn(x, 1099511627776.f));
}

__device__ __forceinline__ uint64_t elem_weight(const float* a, const float* bq, int t, bool resid) {
    return resid ? weight(__fsub_rn(__ldg(a + t), __ldg(bq + t))) : weight(__ldg(a + t));
}

struct Slice {
    int lo, hi;      // this CTA's vocabulary range
    int seg;         // elements per warp segment (multiple of 4)
};

__device__ __forceinline__ Slice make_slice(int V, int C, int rank) {
    int per = (V + C - 1) / C;
    per = (per + 3) & ~3;
    Slice s;
    s.lo = min(V, rank * per);
    s.hi = min(V, s.lo + per);
    int seg = (s.hi - s.lo + ACC_WARPS - 1) / ACC_WARPS;
    s.seg = (seg + 3) & ~3;
    return s;
}

// Block-wide argmax of row[lo, hi); result valid in every thread.
template <bool VEC>
__device__ ArgBest block_argmax(const float* __restrict__ row, int lo, int hi, ArgBest* red) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    ArgBest a{-INFINITY, NO_INDEX};
    if (VEC) {
        const int nv = (hi - lo) >> 2;
        const float4* r4 = reinterpret_cast<const float4*>(row + lo);
        constexpr int T = ACC_THREADS;
        int e = tid;
        // four independent 16-byte loads in flight before any compare
        for (; e + 3 * T < nv; e += 4 * T) {
            const float4 x0 = __ldg(r4 + e), x1 = __ldg(r4 + e + T);
            const float4 x2 = __ldg(r4 + e + 2 * T), x3 = __ldg(r4 + e + 3 * T);
            take4(a, x0, lo + 4 * e);
            take4(a, x1, lo + 4 * (e + T));
            take4(a, x2, lo + 4 * (e + 2 * T));
            take4(a, x3, lo + 4 * (e + 3 * T));
        }
        for (; e < nv; e += T) take4(a, __ldg(r4 + e), lo + 4 * e);
        for (int i = lo + 4 * nv + tid; i < hi; i += ACC_THREADS) take(a, __ldg(row + i), i);
    } else {
        for (int i = lo + tid; i < hi; i += ACC_THREADS) take(a, __ldg(row + i), i);
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
    __syncthreads();
    if (lane == 0) red[warp] = a;
    __syncthreads();
    ArgBest r = red[0];
    for (int w = 1; w < ACC_WARPS; ++w)
        if (beats(red[w].v, red[w].i, r.v, r.i)) r = red[w];
    return r;
}

// Sum of integer weights over this CTA's slice, per warp segment (kept in
// wsum[]) and in total.  resid: weight(a - b); otherwise weight(a).
__device__ uint64_t slice_weight_sum(const float* a, const float* bq, bool resid, const Slice& s,
                                     uint64_t* wsum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int slo = min(s.hi, s.lo + warp * s.seg), shi = min(s.hi, slo + s.seg);
    uint64_t acc = 0;
    const bool vec = ((reinterpret_cast<uintptr_t>(a + slo) | (bq ? reinterpret_cast<uintptr_t>(bq + slo) : 0)) & 15) == 0;
    int t = slo;
    if (vec) {
        // four floats per lane per step, four steps in flight
        const int nv4 = (shi - slo) >> 2;
        const float4* a4 = reinterpret_cast<const float4*>(a + slo);
        const float4* b4 = resid ? reinterpret_cast<const float4*>(bq + slo) : nullptr;
        auto wsum4 = [&](const float4& x, const float4& y) -> uint64_t {
            if (resid)
                return weight(__fsub_rn(x.x, y.x)) + weight(__fsub_rn(x.y, y.y)) +
                       weight(__fsub_rn(x.z, y.z)) + weight(__fsub_rn(x.w, y.w));
            return weight(x.x) + weight(x.y) + weight(x.z) + weight(x.w);
        };
        const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
        int e = lane;
        // four independent loads per operand in flight before any use
        for (; e + 96 < nv4; e += 128) {
            const float4 x0 = __ldg(a4 + e), x1 = __ldg(a4 + e + 32);
            const float4 x2 = __ldg(a4 + e + 64), x3 = __ldg(a4 + e + 96);
            const float4 y0 = resid ? __ldg(b4 + e) : zero4, y1 = resid ? __ldg(b4 + e + 32) : zero4;
            const float4 y2 = resid ? __ldg(b4 + e + 64) : zero4, y3 = resid ? __ldg(b4 + e + 96) : zero4;
            acc += wsum4(x0, y0) + wsum4(x1, y1) + wsum4(x2, y2) + wsum4(x3, y3);
        }
        for (; e < nv4; e += 32) acc += wsum4(__ldg(a4 + e), resid ? __ldg(b4 + e) : zero4);
        t = slo + 4 * nv4;
    }
    for (t += lane; t < shi; t += 32) acc += elem_weight(a, bq, t, resid);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    __syncthreads();
    if (lane == 0) wsum[warp] = acc;
    __syncthreads();
    uint64_t tot = 0;
    for (int w = 0; w < ACC_WARPS; ++w) tot += wsum[w];
    return tot;
}

// Within this CTA's slice, the smallest index whose inclusive prefix sum of
// weights exceeds T (0 <= T < slice sum).  Run by one warp; returns in lane 0.
__device__ int slice_find(const float* a, const float* bq, bool resid, const Slice& s,
                          const uint64_t* wsum, uint64_t T) {
    const int lane = threadIdx.x & 31;
    int w = 0;
    while (w < ACC_WARPS - 1 && T >= wsum[w]) {
        T -= wsum[w];
        ++w;
    }
    const int slo = min(s.hi, s.lo + w * s.seg), shi = min(s.hi, slo + s.seg);
    for (int base = slo; base < shi; base += 32) {
        const int t = base + lane;
        uint64_t x = (t < shi) ? elem_weight(a, bq, t, resid) : 0ull;
        // inclusive warp scan
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint64_t y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        const uint64_t chunk = __shfl_sync(0xffffffffu, x, 31);
        if (T < chunk) {
            const unsigned hit = __ballot_sync(0xffffffffu, x > T);
            return base + __ffs(hit) - 1;
        }
        T -= chunk;
    }
    return -1;  // not reached when T < slice sum
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

// Tree and token checks in the order the acceptance rule states them
// (structure first, then token range).  One thread.
__device__ int check_inputs(const int* spar, const int* stok, int N, int V, bool chain) {
    for (int i = 0; i < N; ++i) {
        const int pa = spar[i];
        if ((i == 0 && pa != -1) || (i > 0 && (pa < 0 || pa >= i))) return TV_ERR_BAD_TREE;
    }
    if (chain)
        for (int i = 1; i < N; ++i)
            if (spar[i] != i - 1) return TV_ERR_UNSUPPORTED;
    for (int i = 1; i < N; ++i)
        if (stok[i] < 0 || stok[i] >= V) return TV_ERR_OUT_OF_RANGE;
    return TV_OK;
}

template <bool VEC>
__global__ void __launch_bounds__(ACC_THREADS)
accept_greedy_kernel(AccParams p) {
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    pdl_launch_dependents();
    pdl_wait();
    const int b = blockIdx.x / C;
    __shared__ int spar[64], stok[64], sam[64];
    __shared__ ArgBest exch[2][64];
    __shared__ ArgBest red[ACC_WARPS];
    __shared__ int sflag;
    const int tid = threadIdx.x, N = p.N;
    if (tid < N) {
        spar[tid] = p.parents[(int64_t)b * N + tid];
        stok[tid] = p.tokens[(int64_t)b * N + tid];
        sam[tid] = -1;
    }
    __syncthreads();
    if (tid == 0) sflag = check_inputs(spar, stok, N, p.V, false);
    __syncthreads();
    if (sflag != TV_OK) {
        if (rank == 0) write_fail(p, b, sflag);
        return;  // uniform across the cluster: no cluster barrier has been issued
    }
    const Slice sl = make_slice(p.V, C, rank);
    uint64_t frontier = 1ull;  // node 0
    int par = 0, chosen = 0;
    // each level is one depth deeper, so the walk ends within N levels
    for (int level = 0; level < N; ++level) {
        // local argmax of each frontier row
        for (uint64_t f = frontier; f; f &= f - 1) {
            const int u = __ffsll((long long)f) - 1;
            const float* row = p.target + ((int64_t)b * N + u) * p.V;
            const ArgBest a = block_argmax<VEC>(row, sl.lo, sl.hi, red);
            if (tid == 0) exch[par][u] = a;
        }
        cluster.sync();
        // combine across the cluster: warp w takes frontier nodes w, w+16, ...;
        // lane r reads rank r's candidate, then a warp argmax
        {
            const int warp = tid >> 5, lane = tid & 31;
            int idx = 0;
            for (uint64_t f = frontier; f; f &= f - 1, ++idx) {
                if (idx % ACC_WARPS != warp) continue;
                const int u = __ffsll((long long)f) - 1;
                ArgBest x{-INFINITY, NO_INDEX};
                if (lane < C) x = *cluster.map_shared_rank(&exch[par][u], lane);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const float w = __shfl_xor_sync(0xffffffffu, x.v, off);
                    const int j = __shfl_xor_sync(0xffffffffu, x.i, off);
                    if (beats(w, j, x.v, x.i)) {
                        x.v = w;
                        x.i = j;
                    }
                }
                if (lane == 0) sam[u] = (x.i == NO_INDEX) ? -1 : x.i;
            }
        }
        __syncthreads();
        // next frontier: children whose token equals their (frontier) parent's argmax
        __shared__ unsigned long long snext;
        if (tid == 0) snext = 0ull;
        __syncthreads();
        if (tid >= 1 && tid < N) {
            const int pc = spar[tid];
            if (((frontier >> pc) & 1ull) && sam[pc] >= 0 && stok[tid] == sam[pc])
                atomicOr(&snext, 1ull << tid);
        }
        __syncthreads();
        const uint64_t next = snext;
        if (next == 0) {
            chosen = __ffsll((long long)frontier) - 1;
            break;
        }
        frontier = next;
        par ^= 1;
        __syncthreads();  // snext is reset at the next level
    }
    cluster.sync();  // no CTA leaves while others may still read its exchange slots
    if (rank == 0) {
        if (sam[chosen] < 0) write_fail(p, b, TV_ERR_BAD_VALUES);
        else write_path(p, b, spar, stok, chosen, sam[chosen]);
    }
}

// Greedy acceptance for small batches: every row's argmax is computed in
// parallel (one cluster per row, DSMEM reduction), written to the workspace,
// and the CTA that completes a sequence's last row (atomic ticket) walks the
// tree.  Reads every row once, but without the walk's level-by-level latency.
template <bool VEC>
__global__ void __launch_bounds__(ACC_THREADS)
accept_rowscan_kernel(AccParams p, int32_t* __restrict__ am_ws, int32_t* __restrict__ tickets) {
    cg::cluster_group cluster = cg::this_cluster();
    const int S = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    pdl_launch_dependents();
    pdl_wait();
    const int cl = blockIdx.x / S;
    const int N = p.N;
    const int b = cl / N, row = cl % N;
    const int tid = threadIdx.x;
    __shared__ ArgBest red[ACC_WARPS];
    __shared__ ArgBest exch;
    __shared__ int last;
    __shared__ int spar[64], stok[64], sam[64];
    __shared__ int sflag;
    const Slice sl = make_slice(p.V, S, rank);
    const ArgBest a = block_argmax<VEC>(p.target + ((int64_t)b * N + row) * p.V, sl.lo, sl.hi, red);
    if (tid == 0) exch = a;
    cluster.sync();
    if (rank == 0 && tid < 32) {
        ArgBest x{-INFINITY, NO_INDEX};
        if (tid < S) x = *cluster.map_shared_rank(&exch, tid);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float w = __shfl_xor_sync(0xffffffffu, x.v, off);
            const int j = __shfl_xor_sync(0xffffffffu, x.i, off);
            if (beats(w, j, x.v, x.i)) {
                x.v = w;
                x.i = j;
            }
        }
        if (tid == 0) {
            am_ws[(int64_t)b * N + row] = (x.i == NO_INDEX) ? -1 : x.i;
            __threadfence();
            last = (atomicAdd(&tickets[b], 1) == N - 1);
        }
    }
    cluster.sync();  // peers' exchange slots stay alive until rank 0 has read them
    if (rank != 0) return;
    __syncthreads();
    if (!last) return;
    // this CTA completed sequence b: walk its tree
    __threadfence();
    if (tid < N) {
        spar[tid] = p.parents[(int64_t)b * N + tid];
        stok[tid] = p.tokens[(int64_t)b * N + tid];
        sam[tid] = __ldcg(am_ws + (int64_t)b * N + tid);
    }
    __syncthreads();
    if (tid == 0) {
        tickets[b] = 0;  // leave the workspace ready for the next call
        sflag = check_inputs(spar, stok, N, p.V, false);
    }
    __syncthreads();
    if (sflag != TV_OK) {
        write_fail(p, b, sflag);
        return;
    }
    __shared__ int schosen;
    if (tid == 0) {
        // accepted(c) = accepted(parent) and token(c) == argmax(parent row); topological order
        uint64_t acc = 1ull;
        int dep[64];
        dep[0] = 0;
        int chosen = 0;
        for (int c = 1; c < N; ++c) {
            const int pc = spar[c];
            dep[c] = dep[pc] + 1;
            if (((acc >> pc) & 1ull) && sam[pc] >= 0 && stok[c] == sam[pc]) {
                acc |= 1ull << c;
                if (dep[c] > dep[chosen]) chosen = c;
            }
        }
        schosen = chosen;
    }
    __syncthreads();
    const int chosen = schosen;
    if (sam[chosen] < 0) write_fail(p, b, TV_ERR_BAD_VALUES);
    else write_path(p, b, spar, stok, chosen, sam[chosen]);
}

__global__ void __launch_bounds__(ACC_THREADS)
accept_stochastic_kernel(AccParams p) {
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    pdl_launch_dependents();
    pdl_wait();
    const int b = blockIdx.x / C;
    __shared__ int spar[64], stok[64];
    __shared__ uint64_t wsum[ACC_WARPS];
    __shared__ uint64_t xsum[2];   // this CTA's slice sum, per attempt
    __shared__ int xidx;           // token found by this CTA (-1: none)
    __shared__ int sflag;
    const int tid = threadIdx.x, N = p.N;
    if (tid == 0) {
        sflag = 0;
        xidx = -1;
    }
    __syncthreads();
    if (tid < N) {
        spar[tid] = p.parents[(int64_t)b * N + tid];
        stok[tid] = p.tokens[(int64_t)b * N + tid];
    }
    __syncthreads();
    if (tid == 0) sflag = check_inputs(spar, stok, N, p.V, true);
    __syncthreads();
    if (sflag != TV_OK) {
        if (rank == 0) write_fail(p, b, sflag);
        return;
    }
    // accept tests (every CTA, redundantly: a few scalars)
    const int K = N - 1;
    int kstar = K + 1;  // first rejected position, K+1 = none
    for (int k = 1; k <= K; ++k) {
        const uint4 w = draw(p, b, k);
        const uint32_t u24 = w.x >> 8;
        const int x = stok[k];
        const float pk = __ldg(p.target + ((int64_t)b * N + (k - 1)) * p.V + x);
        const float qk = __ldg(p.draft + ((int64_t)b * N + k) * p.V + x);
        const bool acc = __dmul_rn((double)u24, (double)qk) < __dmul_rn((double)pk, 16777216.0);
        if (!acc) {
            kstar = k;
            break;
        }
    }
    const bool rejected = kstar <= K;
    const float* rowa = p.target + ((int64_t)b * N + (rejected ? kstar - 1 : K)) * p.V;
    const float* rowb = rejected ? p.draft + ((int64_t)b * N + kstar) * p.V : nullptr;
    const uint32_t x1 = draw(p, b, rejected ? kstar : K + 1).y;
    const Slice sl = make_slice(p.V, C, rank);

    bool resid = rejected;
    int token = -1;
    for (int attempt = 0; attempt < 2; ++attempt) {
        const uint64_t mine = slice_weight_sum(rowa, rowb, resid, sl, wsum);
        if (tid == 0) xsum[attempt] = mine;
        cluster.sync();
        uint64_t S = 0, before = 0;
        for (int r = 0; r < C; ++r) {
            const uint64_t v = *cluster.map_shared_rank(&xsum[attempt], r);
            if (r < rank) before += v;
            S += v;
        }
        if (S == 0) {
            if (resid) {
                resid = false;  // residual has no mass: draw from the target row itself
                continue;
            }
            break;  // zero-mass target row
        }
        const uint64_t hi = __umul64hi((uint64_t)x1, S), lo = (uint64_t)x1 * S;
        const uint64_t T = (hi << 32) | (lo >> 32);
        if (T >= before && T < before + mine && tid < 32) {
            const int t = slice_find(rowa, rowb, resid, sl, wsum, T - before);
            if (tid == 0) xidx = t;
        }
        cluster.sync();
        if (rank == 0) {
            for (int r = 0; r < C; ++r) {
                const int v = *cluster.map_shared_rank(&xidx, r);
                if (v >= 0) token = v;
            }
        }
        break;
    }
    cluster.sync();  // exchange slots stay alive until every CTA has read them
    if (rank == 0) {
        __shared__ int stoken;
        if (tid == 0) stoken = token;
        __syncthreads();
        if (stoken < 0) write_fail(p, b, TV_ERR_BAD_VALUES);
        else write_path(p, b, spar, stok, rejected ? kstar - 1 : K, stoken);
    }
}

// Allows 16-CTA clusters for every kernel here when the device supports it.
bool enable_large_clusters() {
    static int state = -1;
    if (state < 0) {
        state = 0;
        bool ok = cudaFuncSetAttribute(accept_greedy_kernel<true>,
                                       cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
        ok = ok && cudaFuncSetAttribute(accept_greedy_kernel<false>,
                                        cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
        ok = ok && cudaFuncSetAttribute(accept_rowscan_kernel<true>,
                                        cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
        ok = ok && cudaFuncSetAttribute(accept_rowscan_kernel<false>,
                                        cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
        ok = ok && cudaFuncSetAttribute(accept_stochastic_kernel,
                                        cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
        if (ok) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(16);
            cfg.blockDim = dim3(ACC_THREADS);
            cudaLaunchAttribute at;
            at.id = cudaLaunchAttributeClusterDimension;
            at.val.clusterDim.x = 16;
            at.val.clusterDim.y = 1;
            at.val.clusterDim.z = 1;
            cfg.attrs = &at;
            cfg.numAttrs = 1;
            int n = 0;
            ok = cudaOccupancyMaxActiveClusters(&n, accept_greedy_kernel<true>, &cfg) == cudaSuccess &&
                 n > 0;
        }
        cudaGetLastError();
        state = ok ? 1 : 0;
    }
    return state == 1;
}

int pow2_at_least(int64_t x) {
    int c = 1;
    while (c < x && c < 16) c <<= 1;
    return c;
}

// Row-scan pays for every row once at full bandwidth; the walk pays a few
// microseconds of latency per tree level (at most 8 levels assumed).
bool prefer_rowscan(int B, int N, int V) {
    const double bytes = (double)B * N * V * 4.0;
    const double t_scan = bytes / 6.0e12 + 3.0e-6;
    const double t_walk = (double)(N < 8 ? N : 8) * 2.5e-6;
    return t_scan < t_walk;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

size_t accept_workspace(tv_accept_mode mode, int B, int N, int V) {
    if (mode != TV_ACCEPT_GREEDY || B <= 0 || !prefer_rowscan(B, N, V)) return 0;
    return align256((size_t)B * N * 4) + align256((size_t)B * 4);
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
    const bool large = enable_large_clusters();
    const int cmax = large ? 16 : 8;
    const int sms = device_sm_count();
    const bool vec = (a.V % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.target) & 15) == 0);
    const size_t need = accept_workspace(a.mode, a.B, a.N, a.V);
    if (need > 0 && (a.ws == nullptr || a.ws_bytes < need)) return TV_ERR_WORKSPACE;
    const bool rowscan = need > 0;

    int C;
    int64_t units;
    if (rowscan) {
        units = (int64_t)a.B * a.N;
        C = pow2_at_least((2LL * sms + units - 1) / units);
    } else {
        units = a.B;
        C = ((int64_t)a.B * 16 <= 2LL * sms) ? 16 : 8;
    }
    if (C > cmax) C = cmax;
    while (C > 1 && C > a.V / 4) C >>= 1;  // keep every slice non-trivial on tiny vocabularies
    if (units * C > 0x7fffffff) return TV_ERR_UNSUPPORTED;
    LaunchCfg lc(dim3((unsigned)(units * C)), dim3(ACC_THREADS), 0, a.stream, (unsigned)C);
    const cudaLaunchConfig_t& cfg = lc.cfg;
    cudaError_t e;
    if (a.mode == TV_ACCEPT_GREEDY && rowscan) {
        int32_t* am = static_cast<int32_t*>(a.ws);
        int32_t* tickets = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(a.ws) +
                                                       align256((size_t)a.B * a.N * 4));
        e = vec ? cudaLaunchKernelEx(&cfg, accept_rowscan_kernel<true>, p, am, tickets)
                : cudaLaunchKernelEx(&cfg, accept_rowscan_kernel<false>, p, am, tickets);
    } else if (a.mode == TV_ACCEPT_GREEDY) {
        e = vec ? cudaLaunchKernelEx(&cfg, accept_greedy_kernel<true>, p)
                : cudaLaunchKernelEx(&cfg, accept_greedy_kernel<false>, p);
    } else {
        e = cudaLaunchKernelEx(&cfg, accept_stochastic_kernel, p);
    }
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

}  // namespace tv
