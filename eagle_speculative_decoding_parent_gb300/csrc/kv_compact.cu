// kv_compact: gather-then-scatter of the accepted rows.
// One CTA per (kv head, sequence, layer x {K, V}): the accepted path's rows
// (at most 64 of d elements) are first read into shared memory with 16-byte
// vector loads, the CTA synchronises, then the rows are written to the
// contiguous positions P .. P + accept_len.  Reading everything before
// writing anything gives the same result as index_select followed by copy_,
// even when a destination row is the source of another.
#include "tv_device.cuh"
#include "tv_internal.h"

namespace tv {

namespace {

constexpr int CP_THREADS = 128;
constexpr int CP_MAX_ROWS = 64;

struct CpParams {
    uint8_t* k;
    uint8_t* v;
    int64_t layer_stride_bytes;
    const int32_t* table;
    const int32_t* prefix_lens;
    const int32_t* path;
    const int32_t* accept_len;
    int max_blocks, max_path, Hkv, bs, num_blocks, row_bytes;
    int32_t* new_lens;
    int64_t* src_slots;
    int64_t* dst_slots;
    int32_t* status;
};

__device__ __forceinline__ int64_t slot_of(const CpParams& p, int b, int64_t t) {
    if (t < 0) return -1;
    const int64_t lb = t / p.bs;
    if (lb >= p.max_blocks) return -1;
    const int blk = p.table[(int64_t)b * p.max_blocks + lb];
    if (blk < 0 || blk >= p.num_blocks) return -1;
    return (int64_t)blk * p.bs + t % p.bs;
}

__global__ void __launch_bounds__(CP_THREADS) kv_compact_kernel(CpParams p) {
    extern __shared__ uint4 rows[];  // [A+1][row_bytes / 16]
    __shared__ int64_t ssrc[CP_MAX_ROWS], sdst[CP_MAX_ROWS];
    __shared__ int sok;
    const int g = blockIdx.x, b = blockIdx.y;
    const int layer = blockIdx.z >> 1, which = blockIdx.z & 1;
    const int tid = threadIdx.x;
    pdl_launch_dependents();
    pdl_wait();
    const int P = p.prefix_lens[b];
    const int A = p.accept_len[b];
    if (tid == 0) sok = (P >= 0 && A >= 0 && A < p.max_path && A < CP_MAX_ROWS) ? 1 : 0;
    __syncthreads();
    bool ok = sok != 0;
    if (ok) {
        for (int j = tid; j <= A; j += CP_THREADS) {
            const int pj = p.path[(int64_t)b * p.max_path + j];
            const int64_t s = (pj < 0) ? -1 : slot_of(p, b, (int64_t)P + pj);
            const int64_t d = slot_of(p, b, (int64_t)P + j);
            ssrc[j] = s;
            sdst[j] = d;
            if (s < 0 || d < 0) ok = false;
        }
    }
    ok = __syncthreads_and(ok) != 0;
    const bool writer = (g == 0 && blockIdx.z == 0);
    if (writer) {
        for (int j = tid; j < p.max_path; j += CP_THREADS) {
            const bool in = ok && j <= A;
            if (p.src_slots) p.src_slots[(int64_t)b * p.max_path + j] = in ? ssrc[j] : -1;
            if (p.dst_slots) p.dst_slots[(int64_t)b * p.max_path + j] = in ? sdst[j] : -1;
        }
        if (tid == 0) {
            p.status[b] = ok ? TV_OK : TV_ERR_OUT_OF_RANGE;
            p.new_lens[b] = ok ? P + A + 1 : P;
        }
    }
    if (!ok) return;
    uint8_t* base = (which ? p.v : p.k) + (int64_t)layer * p.layer_stride_bytes;
    const int vecs = p.row_bytes >> 4;
    const int total = (A + 1) * vecs;
    auto row_ptr = [&](int64_t slot) -> uint4* {
        const int64_t blk = slot / p.bs, r = slot % p.bs;
        return reinterpret_cast<uint4*>(base + ((blk * p.Hkv + g) * p.bs + r) * p.row_bytes);
    };
    for (int e = tid; e < total; e += CP_THREADS) {
        const int j = e / vecs, c = e % vecs;
        rows[e] = row_ptr(ssrc[j])[c];
    }
    __syncthreads();
    for (int e = tid; e < total; e += CP_THREADS) {
        const int j = e / vecs, c = e % vecs;
        row_ptr(sdst[j])[c] = rows[e];
    }
}

}  // namespace

tv_status launch_compact(const CompactArgs& a) {
    if (a.B == 0 || a.Hkv == 0 || a.num_layers == 0) return TV_OK;
    CpParams p;
    p.k = static_cast<uint8_t*>(a.k_cache);
    p.v = static_cast<uint8_t*>(a.v_cache);
    p.layer_stride_bytes = a.layer_stride * a.elem_bytes;
    p.table = a.block_table;
    p.prefix_lens = a.prefix_lens;
    p.path = a.path;
    p.accept_len = a.accept_len;
    p.max_blocks = a.max_blocks;
    p.max_path = a.max_path;
    p.Hkv = a.Hkv;
    p.bs = a.bs;
    p.num_blocks = a.num_blocks;
    p.row_bytes = a.d * a.elem_bytes;
    p.new_lens = a.new_lens;
    p.src_slots = a.src_slots;
    p.dst_slots = a.dst_slots;
    p.status = a.status;
    const int rows = a.max_path < CP_MAX_ROWS ? a.max_path : CP_MAX_ROWS;
    const size_t smem = (size_t)rows * p.row_bytes;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kv_compact_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return TV_ERR_CUDA;
    dim3 grid(a.Hkv, a.B, 2 * a.num_layers);
    if (grid.y > 65535 || grid.z > 65535) return TV_ERR_UNSUPPORTED;
    LaunchCfg lc(grid, dim3(CP_THREADS), smem, a.stream);
    return cudaLaunchKernelEx(&lc.cfg, kv_compact_kernel, p) == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

}  // namespace tv
