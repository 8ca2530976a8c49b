// tree_verify_attention_noalloc: the attention step for callers that cannot
// allocate device memory themselves.
//
// Some callers have no way to hand the library a scratch buffer: code that
// runs where device allocation is forbidden or would stall the pipeline (for
// example an engine that reserved all of HBM for its KV pool up front and
// never calls cudaMalloc while decoding, or a plugin host that exposes no
// allocator to its plugins).  This entry point serves them by using a
// scratch region that is part of the library image itself: a file-scope
// __device__ array of TV_NOALLOC_SCRATCH_BYTES, which every GPU that loads
// the library keeps for the life of the process.  The caller still owns
// inputs and outputs; nothing here calls cudaMalloc, cudaFree or an
// allocating library routine.
#include <mutex>

#include "tv_device.cuh"
#include "tv_internal.h"

namespace {

constexpr size_t kScratchBytes = TV_NOALLOC_SCRATCH_BYTES;

// The shared scratch.  In host code this name is only a stand-in for the
// symbol, never a device address: its address on a device comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch on the current device; looked up once per
// device (the first call on that device), with that device current.
tv_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_attn_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return TV_ERR_CUDA;
        }
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return TV_OK;
}

}  // namespace

extern "C" size_t tree_verify_attention_noalloc_capacity(void) { return kScratchBytes; }

extern "C" tv_status tree_verify_attention_noalloc(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
    int max_blocks_per_seq, const int32_t* prefix_lens, const uint64_t* mask, int B, int N,
    const int32_t* node_counts, int Hq, int Hkv, int d, int block_size, int num_blocks, tv_dtype dt,
    float scale, void* out, int32_t* status, tv_stream_t stream) {
    if (dt != TV_F32 && dt != TV_BF16) return TV_ERR_INVALID_ARG;
    if (B < 0 || N < 1 || N > 64 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || max_blocks_per_seq < 1 ||
        block_size < 1 || num_blocks < 1)
        return TV_ERR_INVALID_ARG;
    const size_t need = tree_verify_attention_workspace(B, N, Hq, Hkv, d, max_blocks_per_seq,
                                                        block_size, dt);
    if (need > kScratchBytes) return TV_ERR_WORKSPACE;  // shape needs more than the fixed scratch
    void* scratch = nullptr;
    if (need > 0) {
        const tv_status st = scratch_address(&scratch);
        if (st != TV_OK) return st;
        // Calls share the scratch and it keeps the previous call's contents:
        // clear the arrival counters, which must start at zero.
        const size_t zero = tv::attn_bf16_workspace_zeroed_prefix(B, N, Hq, Hkv, d,
                                                                  max_blocks_per_seq, block_size);
        if (zero > 0 && cudaMemsetAsync(scratch, 0, zero, (cudaStream_t)stream) != cudaSuccess)
            return TV_ERR_CUDA;
    }
    // The workspace size passed on is exactly `need`, the size the workspace
    // query gives for this shape, so this call takes the same schedule as a
    // tree_verify_attention call whose caller sized its workspace by that query.
    return tree_verify_attention(q, k_cache, v_cache, block_table, max_blocks_per_seq,
                                 prefix_lens, mask, B, N, node_counts, Hq, Hkv, d, block_size,
                                 num_blocks, dt, scale, out, status, scratch, need, stream);
}
