// tree_verify_attention, float32 path: CUDA-core FMA, one warp per
// (sequence, node, query head).  Keys are visited in groups of 32 (one per
// lane) with an online softmax across groups; the value rows are accumulated
// with lane-parallel output columns (coalesced).  Used for float32 caches,
// where tensor cores would change the arithmetic.  With node counts, sequence
// b's keys are its P + counts[b] positions and the rows of absent nodes are
// not written.
#include "tv_device.cuh"
#include "tv_internal.h"

namespace tv {

template <int DPL>  // output columns per lane (d / 32)
__global__ void __launch_bounds__(128)
attn_f32_kernel(const float* __restrict__ q, const float* __restrict__ kc,
                const float* __restrict__ vc, const int32_t* __restrict__ table, int max_blocks,
                const int32_t* __restrict__ prefix_lens, const uint64_t* __restrict__ mask,
                const int32_t* __restrict__ counts, int B, int N, int Hq, int Hkv, int bs,
                int num_blocks, float scale,
                float* __restrict__ out, int32_t* __restrict__ status) {
    constexpr int D = DPL * 32;
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    pdl_launch_dependents();
    pdl_wait();
    if (gw >= (int64_t)B * N * Hq) return;
    const int h = (int)(gw % Hq);
    const int64_t bi = gw / Hq;
    const int i = (int)(bi % N), b = (int)(bi / N);
    const int g = h / (Hq / Hkv);
    const int P = prefix_lens[b];
    const int n = counts ? counts[b] : N;  // nodes n..N-1 are absent
    const int64_t L = (int64_t)P + n;
    bool ok = P >= 0 && n >= 1 && n <= N && L <= (int64_t)max_blocks * bs;
    if (ok) {
        const int nb = (int)((L + bs - 1) / bs);
        for (int j = lane; j < nb; j += 32) {
            const int blk = table[(int64_t)b * max_blocks + j];
            ok = ok && blk >= 0 && blk < num_blocks;
        }
    }
    ok = __all_sync(0xffffffffu, ok);
    float* o = out + gw * D;
    if (i == 0 && h == 0 && lane == 0) status[b] = ok ? TV_OK : TV_ERR_OUT_OF_RANGE;
    if (!ok) {
#pragma unroll
        for (int k = 0; k < DPL; ++k) o[lane + 32 * k] = 0.f;
        return;
    }
    if (i >= n) return;  // absent node: no output row
    const uint64_t m_tree = (n >= 64) ? mask[bi] : (mask[bi] & ((1ull << n) - 1));
    const float* qr = q + gw * D;
    float acc[DPL];
#pragma unroll
    for (int k = 0; k < DPL; ++k) acc[k] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;
    auto row_of = [&](int64_t t) -> int64_t {
        const int blk = table[(int64_t)b * max_blocks + t / bs];
        return (((int64_t)blk * Hkv + g) * bs + t % bs) * D;
    };
    for (int64_t t0 = 0; t0 < L; t0 += 32) {
        const int64_t t = t0 + lane;
        const bool vis = (t < P) || (t < L && ((m_tree >> (t - P)) & 1ull));
        float s = -INFINITY;
        if (vis) {
            const float4* kr = reinterpret_cast<const float4*>(kc + row_of(t));
            const float4* q4 = reinterpret_cast<const float4*>(qr);
            float dot = 0.f;
#pragma unroll 8
            for (int c = 0; c < D / 4; ++c) {
                const float4 a = q4[c], k4 = kr[c];
                dot = fmaf(a.x, k4.x, dot);
                dot = fmaf(a.y, k4.y, dot);
                dot = fmaf(a.z, k4.z, dot);
                dot = fmaf(a.w, k4.w, dot);
            }
            s = dot * scale;
        }
        float tmax = s;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
        if (tmax == -INFINITY) continue;  // no visible key in this group
        const float m_new = fmaxf(m_run, tmax);
        const float corr = (m_run == -INFINITY) ? 0.f : expf(m_run - m_new);
        const float p = vis ? expf(s - m_new) : 0.f;
        float psum = p;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
        l_run = l_run * corr + psum;
#pragma unroll
        for (int k = 0; k < DPL; ++k) acc[k] *= corr;
        // value rows of the visible keys, eight keys per batch of independent loads
        const uint32_t vmask = __ballot_sync(0xffffffffu, vis);
        const int64_t my_row = vis ? row_of(t) : 0;
#pragma unroll 1
        for (int j0 = 0; j0 < 32; j0 += 8) {
            float vv[8][DPL];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int64_t rj = __shfl_sync(0xffffffffu, my_row, j0 + jj);
                const bool use = (vmask >> (j0 + jj)) & 1u;
#pragma unroll
                for (int k = 0; k < DPL; ++k) vv[jj][k] = use ? __ldg(vc + rj + lane + 32 * k) : 0.f;
            }
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const float pj = __shfl_sync(0xffffffffu, p, j0 + jj);
#pragma unroll
                for (int k = 0; k < DPL; ++k) acc[k] = fmaf(pj, vv[jj][k], acc[k]);
            }
        }
        m_run = m_new;
    }
    const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
#pragma unroll
    for (int k = 0; k < DPL; ++k) o[lane + 32 * k] = acc[k] * inv;
}

tv_status launch_attn_f32(const AttnArgs& a) {
    const int64_t warps = (int64_t)a.B * a.N * a.Hq;
    if (warps == 0) return TV_OK;
    const int threads = 128;
    const int64_t blocks = (warps * 32 + threads - 1) / threads;
    if (blocks > 0x7fffffff) return TV_ERR_UNSUPPORTED;
    LaunchCfg lc(dim3((unsigned)blocks), dim3(threads), 0, a.stream);
    cudaError_t e = cudaSuccess;
#define TV_F32_CASE(DPL)                                                                       \
    case DPL:                                                                                  \
        e = cudaLaunchKernelEx(&lc.cfg, attn_f32_kernel<DPL>, (const float*)a.q,              \
                               (const float*)a.k_cache, (const float*)a.v_cache, a.block_table, \
                               a.max_blocks, a.prefix_lens, a.mask, a.counts, a.B, a.N, a.Hq, \
                               a.Hkv,                                                           \
                               a.bs, a.num_blocks, a.scale, (float*)a.out, a.status);           \
        break;
    switch (a.d / 32) {
        TV_F32_CASE(1)
        TV_F32_CASE(2)
        TV_F32_CASE(3)
        TV_F32_CASE(4)
        TV_F32_CASE(5)
        TV_F32_CASE(6)
        TV_F32_CASE(7)
        TV_F32_CASE(8)
        default:
            return TV_ERR_UNSUPPORTED;
    }
#undef TV_F32_CASE
    return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

}  // namespace tv
