// tree_kv_append: the draft tree's K/V rows into the paged cache, keys
// optionally rotated by their tree position.
// One CTA per (node, sequence).  Every CTA of a sequence first checks that all
// of the sequence's positions have valid blocks (and depths, with rotation),
// so a bad sequence is left untouched by all of them.  Keys: rotate-half pairs
// (j, j + d/2) with angle (P + depth) * theta^(-2j/d); every product and sum
// is rounded separately in double (no fused multiply-add), then the result is
// rounded to binary32 and to the cache type; a node's (cos, sin) pairs are
// computed once and shared by its kv heads.  Values (and keys without
// rotation) are copied with 16-byte vectors.  With node counts only the first
// counts[b] nodes of a sequence exist: the others are not appended, and a
// count outside [1, N] is TV_ERR_OUT_OF_RANGE.
#include <cuda_bf16.h>

#include "tv_device.cuh"
#include "tv_internal.h"

namespace tv {

namespace {

constexpr int AP_THREADS = 128;

struct ApParams {
    const uint8_t* k_new;
    const uint8_t* v_new;
    const int32_t* depth;
    uint8_t* k_cache;
    uint8_t* v_cache;
    const int32_t* table;
    const int32_t* prefix_lens;
    const int32_t* counts;  // nullable
    int32_t* status;
    int N, Hkv, d, elem, max_blocks, bs, num_blocks;
    double theta;  // <= 0: no rotation
    bool table_cs;  // the node's (cos, sin) table is in dynamic shared memory
};

constexpr int AP_TABLE_MAX = 3072;  // pairs per table: 48 KB of shared memory

__device__ __forceinline__ int64_t ap_slot(const ApParams& p, int b, int64_t t) {
    if (t < 0) return -1;
    const int64_t lb = t / p.bs;
    if (lb >= p.max_blocks) return -1;
    const int blk = p.table[(int64_t)b * p.max_blocks + lb];
    if (blk < 0 || blk >= p.num_blocks) return -1;
    return (int64_t)blk * p.bs + t % p.bs;
}

__device__ __forceinline__ double ap_load(const ApParams& p, const uint8_t* base, int64_t idx) {
    if (p.elem == 4) return (double)reinterpret_cast<const float*>(base)[idx];
    return (double)__bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
}
__device__ __forceinline__ void ap_store(const ApParams& p, uint8_t* base, int64_t idx, double x) {
    const float f = __double2float_rn(x);
    if (p.elem == 4) reinterpret_cast<float*>(base)[idx] = f;
    else reinterpret_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(f);
}

__global__ void __launch_bounds__(AP_THREADS) kv_append_kernel(ApParams p) {
    const int i = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    pdl_launch_dependents();
    pdl_wait();
    const int P = p.prefix_lens[b];
    const int cnt = p.counts ? p.counts[b] : p.N;  // nodes cnt..N-1 are absent
    bool ok = P >= 0 && cnt >= 1 && cnt <= p.N;
    for (int n = tid; ok && n < cnt; n += AP_THREADS) {
        ok = ap_slot(p, b, (int64_t)P + n) >= 0;
        if (ok && p.theta > 0.0) {
            const int dp = p.depth[(int64_t)b * p.N + n];
            ok = dp >= 0 && dp < cnt;
        }
    }
    ok = __syncthreads_and(ok ? 1 : 0) != 0;
    if (i == 0 && tid == 0) p.status[b] = ok ? TV_OK : TV_ERR_OUT_OF_RANGE;
    if (!ok || i >= cnt) return;
    const int64_t slot = ap_slot(p, b, (int64_t)P + i);
    const int64_t blk = slot / p.bs, row = slot % p.bs;
    const int64_t row_bytes = (int64_t)p.d * p.elem;
    const int vec = (int)(row_bytes / 16);
    // values (and keys without rotation): 16-byte vectors, all heads
    for (int e = tid; e < p.Hkv * vec; e += AP_THREADS) {
        const int g = e / vec, c = e % vec;
        const int64_t src = (((int64_t)b * p.N + i) * p.Hkv + g) * row_bytes + c * 16;
        const int64_t dst = ((blk * p.Hkv + g) * p.bs + row) * row_bytes + c * 16;
        *reinterpret_cast<uint4*>(p.v_cache + dst) = *reinterpret_cast<const uint4*>(p.v_new + src);
        if (p.theta <= 0.0)
            *reinterpret_cast<uint4*>(p.k_cache + dst) = *reinterpret_cast<const uint4*>(p.k_new + src);
    }
    if (p.theta <= 0.0) return;
    const int h = p.d / 2;
    const double pos = (double)(P + p.depth[(int64_t)b * p.N + i]);
    // the angle depends on the pair, not on the kv head: each (cos, sin) is
    // computed once per node into shared memory when the table fits
    extern __shared__ double2 cs_tab[];  // [h] (cos, sin)
    auto angle = [&](int j, double& sn, double& cs) {
        sincos(__dmul_rn(pos, pow(p.theta, -2.0 * (double)j / (double)p.d)), &sn, &cs);
    };
    if (p.table_cs) {
        for (int j = tid; j < h; j += AP_THREADS) {
            double sn, cs;
            angle(j, sn, cs);
            cs_tab[j] = make_double2(cs, sn);
        }
        __syncthreads();
    }
    for (int e = tid; e < p.Hkv * h; e += AP_THREADS) {
        const int g = e / h, j = e % h;
        const int64_t src = (((int64_t)b * p.N + i) * p.Hkv + g) * p.d;
        const int64_t dst = ((blk * p.Hkv + g) * p.bs + row) * p.d;
        double sn, cs;
        if (p.table_cs) {
            const double2 t = cs_tab[j];
            cs = t.x;
            sn = t.y;
        } else {
            angle(j, sn, cs);
        }
        const double x1 = ap_load(p, p.k_new, src + j), x2 = ap_load(p, p.k_new, src + j + h);
        ap_store(p, p.k_cache, dst + j, __dsub_rn(__dmul_rn(x1, cs), __dmul_rn(x2, sn)));
        ap_store(p, p.k_cache, dst + j + h, __dadd_rn(__dmul_rn(x2, cs), __dmul_rn(x1, sn)));
    }
}

}  // namespace

tv_status launch_kv_append(const void* k_new, const void* v_new, const int32_t* depth, int B,
                           int N, const int32_t* counts, int Hkv, int d, float rope_theta,
                           void* k_cache, void* v_cache,
                           const int32_t* block_table, int max_blocks, const int32_t* prefix_lens,
                           int bs, int num_blocks, int elem, int32_t* status, cudaStream_t stream) {
    if (B == 0) return TV_OK;
    ApParams p;
    p.k_new = static_cast<const uint8_t*>(k_new);
    p.v_new = static_cast<const uint8_t*>(v_new);
    p.depth = depth;
    p.k_cache = static_cast<uint8_t*>(k_cache);
    p.v_cache = static_cast<uint8_t*>(v_cache);
    p.table = block_table;
    p.prefix_lens = prefix_lens;
    p.counts = counts;
    p.status = status;
    p.N = N;
    p.Hkv = Hkv;
    p.d = d;
    p.elem = elem;
    p.max_blocks = max_blocks;
    p.bs = bs;
    p.num_blocks = num_blocks;
    p.theta = (rope_theta > 0.f) ? (double)rope_theta : 0.0;
    p.table_cs = p.theta > 0.0 && d / 2 <= AP_TABLE_MAX;
    const size_t smem = p.table_cs ? (size_t)(d / 2) * sizeof(double2) : 0;
    LaunchCfg lc(dim3((unsigned)N, (unsigned)B), dim3(AP_THREADS), smem, stream);
    return cudaLaunchKernelEx(&lc.cfg, kv_append_kernel, p) == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

}  // namespace tv
