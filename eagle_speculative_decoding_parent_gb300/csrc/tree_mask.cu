// tree_mask_build: parent array -> ancestor-or-self bitmask and depth.
// One warp per sequence; lanes own nodes lane and lane + 32.  The parent
// array is staged in shared memory and each node walks its root path there
// (at most 63 steps: parents strictly decrease along the walk).  With node
// counts, sequence b's tree is its first counts[b] nodes: the others get no
// bits and depth -1, and a count outside [1, N] is TV_ERR_OUT_OF_RANGE.
#include "tv_device.cuh"
#include "tv_internal.h"

namespace tv {

constexpr int kMaskWarps = 4;

__global__ void __launch_bounds__(32 * kMaskWarps)
tree_mask_kernel(const int32_t* __restrict__ parents, int B, int N,
                 const int32_t* __restrict__ counts, uint64_t* __restrict__ mask,
                 int32_t* __restrict__ depth, int32_t* __restrict__ status) {
    __shared__ int32_t spar[kMaskWarps][64];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * kMaskWarps + w;
    pdl_launch_dependents();
    pdl_wait();
    if (b >= B) return;
    const int32_t* par = parents + (int64_t)b * N;
    const int n = counts ? counts[b] : N;  // nodes n..N-1 are absent
    const bool n_ok = n >= 1 && n <= N;
    bool ok = n_ok;
    for (int i = lane; i < 64; i += 32) {
        int p = (i < n) ? par[i] : 0;
        spar[w][i] = p;
        if (i < n) ok = ok && ((i == 0) ? (p == -1) : (p >= 0 && p < i));
    }
    __syncwarp();
    ok = __all_sync(0xffffffffu, ok);
    for (int i = lane; i < N; i += 32) {
        uint64_t m = 0;
        int dep = -1;
        if (ok && i < n) {
            for (int j = i; j >= 0; j = spar[w][j]) {
                m |= 1ull << j;
                ++dep;
            }
        }
        mask[(int64_t)b * N + i] = m;
        if (depth) depth[(int64_t)b * N + i] = (ok && i < n) ? dep : -1;
    }
    if (lane == 0) status[b] = ok ? TV_OK : (n_ok ? TV_ERR_BAD_TREE : TV_ERR_OUT_OF_RANGE);
}

tv_status launch_tree_mask(const int32_t* parents, int B, int N, const int32_t* counts,
                           uint64_t* mask, int32_t* depth, int32_t* status, cudaStream_t stream) {
    if (B == 0) return TV_OK;
    dim3 grid((B + kMaskWarps - 1) / kMaskWarps);
    LaunchCfg lc(grid, dim3(32 * kMaskWarps), 0, stream);
    return cudaLaunchKernelEx(&lc.cfg, tree_mask_kernel, parents, B, N, counts, mask, depth, status) ==
                   cudaSuccess
               ? TV_OK
               : TV_ERR_CUDA;
}

}  // namespace tv
