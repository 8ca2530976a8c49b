// Host-side interfaces between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "treeverify.h"

namespace tv {

// Launch configuration used for every kernel: programmatic stream
// serialisation (the kernel may be scheduled while the previous kernel in the
// stream drains; each kernel waits with griddepcontrol.wait before touching
// global memory) plus an optional cluster shape.  Setting TV_PDL=0 in the
// environment launches with plain stream order instead.
inline bool pdl_enabled() {
    static const bool on = [] {
        const char* e = getenv("TV_PDL");
        return !(e && strcmp(e, "0") == 0);
    }();
    return on;
}

struct LaunchCfg {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    LaunchCfg(dim3 grid, dim3 block, size_t smem, cudaStream_t stream, unsigned cluster = 0) {
        memset(&cfg, 0, sizeof(cfg));
        memset(attr, 0, sizeof(attr));
        cfg.gridDim = grid;
        cfg.blockDim = block;
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        unsigned n = 0;
        if (cluster > 0) {
            attr[n].id = cudaLaunchAttributeClusterDimension;
            attr[n].val.clusterDim.x = cluster;
            attr[n].val.clusterDim.y = 1;
            attr[n].val.clusterDim.z = 1;
            ++n;
        }
        if (pdl_enabled()) {
            attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[n].val.programmaticStreamSerializationAllowed = 1;
            ++n;
        }
        cfg.attrs = attr;
        cfg.numAttrs = n;
    }
};

// Multiprocessor count and opt-in shared memory of the current device (cached per device).
int device_sm_count();
int device_smem_optin();

struct AttnArgs {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_table;
    int max_blocks;
    const int32_t* prefix_lens;
    const uint64_t* mask;
    const int32_t* counts;  // nullable: nodes per sequence (first counts[b] of N)
    int B, N, Hq, Hkv, d, bs, num_blocks;
    float scale;
    void* out;
    int32_t* status;
    void* ws;
    size_t ws_bytes;
    cudaStream_t stream;
};

// TMA descriptors (cuTensorMapEncodeTiled through the runtime's driver entry point).
// K or V cache viewed as rows of d bf16 elements: box 64 columns x 16 rows, 128-byte swizzle.
bool make_cache_map(CUtensorMap* map, const void* base, int d, int64_t rows);
// Same cache with d = 128 viewed as 16-row pages: one box holds a page's two
// 64-column halves, [half][16 rows][64 columns], 128-byte swizzle.
bool make_page_map(CUtensorMap* map, const void* base, int64_t rows);
bool make_kpage_map(CUtensorMap* map, const void* base, int64_t rows);
// Q [B*N][Hq][d] bf16: box 64 columns x G heads x npt nodes, 128-byte swizzle.
bool make_q_map(CUtensorMap* map, const void* base, int d, int Hq, int64_t nodes, int G,
                int npt);

tv_status launch_tree_mask(const int32_t* parents, int B, int N, const int32_t* counts,
                           uint64_t* mask, int32_t* depth, int32_t* status, cudaStream_t stream);
tv_status launch_attn_f32(const AttnArgs& a);
size_t attn_bf16_workspace(int B, int N, int Hq, int Hkv, int d, int max_blocks, int bs);
// tensor-core (tcgen05) variant for row tiles wider than 64 rows; same workspace
bool attn_tc_applicable(int N, int Hq, int Hkv, int d);
tv_status launch_attn_tc(const AttnArgs& a);
// its workspace (balanced split: counters and partial results) and the leading
// bytes of it that must be zero when a call starts
size_t attn_tc_workspace(int B, int N, int Hq, int Hkv);
size_t attn_tc_zeroed_prefix(int B, int N, int Hq, int Hkv);
tv_status launch_kv_append(const void* k_new, const void* v_new, const int32_t* depth, int B,
                           int N, const int32_t* counts, int Hkv, int d, float rope_theta,
                           void* k_cache, void* v_cache,
                           const int32_t* block_table, int max_blocks, const int32_t* prefix_lens,
                           int bs, int num_blocks, int elem, int32_t* status, cudaStream_t stream);
// kernels one tensor-core attention call launches with this workspace size
int attn_tc_kernels(int B, int N, int Hq, int Hkv, size_t ws_bytes);
// Leading bytes of that workspace that must be zero when a call starts.
size_t attn_bf16_workspace_zeroed_prefix(int B, int N, int Hq, int Hkv, int d, int max_blocks,
                                         int bs);
tv_status launch_attn_bf16(const AttnArgs& a);

struct AcceptArgs {
    tv_accept_mode mode;
    const int32_t* parents;
    const int32_t* tokens;
    const float* target;
    const float* draft;
    const int32_t* counts;  // nullable: nodes per sequence
    int B, N, V;
    uint64_t seed, offset;
    int32_t* accept_len;
    int32_t* path;
    int32_t* out_tokens;
    int max_path;
    int32_t* status;
    void* ws;
    size_t ws_bytes;
    cudaStream_t stream;
};
size_t accept_workspace(tv_accept_mode mode, int B, int N, int V);
tv_status launch_accept(const AcceptArgs& a);

struct CompactArgs {
    void* k_cache;
    void* v_cache;
    int num_layers;
    int64_t layer_stride;
    const int32_t* block_table;
    int max_blocks;
    const int32_t* prefix_lens;
    const int32_t* path;
    const int32_t* accept_len;
    int max_path, B, Hkv, d, bs, num_blocks, elem_bytes;
    int32_t* new_lens;
    int64_t* src_slots;
    int64_t* dst_slots;
    int32_t* status;
    cudaStream_t stream;
};
tv_status launch_compact(const CompactArgs& a);

// Draft-tree construction limits: chunks per vocabulary row, top-k, nodes
// created per tree (1 + k + (layers - 1) k^2).
constexpr int DT_CH_MAX = 64;
constexpr int DT_K_MAX = 16;
constexpr int DT_NODES_MAX = 2048;

struct DraftArgs {
    const float* logits;
    const int32_t* root_tokens;
    int B, V, k, layer, layers, N;
    int32_t* front_tokens;
    int32_t* front_src;
    int32_t* parents;
    int32_t* tokens;
    float* scores;
    int32_t* status;
    void* ws;
    size_t ws_bytes;
    cudaStream_t stream;
};
int64_t draft_tree_nodes(int k, int layers);
size_t draft_tree_ws_bytes(int B, int k, int layers);
// chunks per row and chunk length of one layer's launch
void draft_tree_chunks(int rows, int V, bool vec, int* c, int* per);
tv_status launch_draft_expand(const DraftArgs& a);

}  // namespace tv
