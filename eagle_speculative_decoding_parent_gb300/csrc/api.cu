// C-ABI entry points of libtreeverify: argument checks on the host, then one
// launch per call on the caller's stream.  See include/treeverify.h for the
// contract of each call.
#include <math.h>

#include "tv_device.cuh"
#include "tv_internal.h"

namespace tv {

static int cached_attr(cudaDeviceAttr attr, int* cache) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, attr, dev) == cudaSuccess) cache[dev] = v;
    }
    return cache[dev];
}

int device_sm_count() {
    static int cache[64] = {0};
    const int v = cached_attr(cudaDevAttrMultiProcessorCount, cache);
    return v > 0 ? v : 1;
}

int device_smem_optin() {
    static int cache[64] = {0};
    return cached_attr(cudaDevAttrMaxSharedMemoryPerBlockOptin, cache);
}

}  // namespace tv

using namespace tv;

extern "C" {

const char* tv_status_string(int s) {
    switch (s) {
        case TV_OK: return "ok";
        case TV_ERR_INVALID_ARG: return "invalid argument";
        case TV_ERR_BAD_TREE: return "parent array is not a valid topologically ordered tree";
        case TV_ERR_OUT_OF_RANGE: return "block id, position, token id or length out of range";
        case TV_ERR_UNSUPPORTED: return "unsupported shape, dtype or mode";
        case TV_ERR_CUDA: return "CUDA runtime or launch failure";
        case TV_ERR_TIMEOUT: return "bounded device wait ran out";
        case TV_ERR_BAD_VALUES: return "all-NaN logits or zero-mass distribution";
        case TV_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        default: return "unknown status";
    }
}

int tv_abi_version(void) { return 2; }

tv_status tree_mask_build(const int32_t* parents, int B, int N, const int32_t* node_counts,
                          uint64_t* mask, int32_t* depth, int32_t* status, tv_stream_t stream) {
    if (B < 0 || N < 1 || N > 64) return TV_ERR_INVALID_ARG;
    if (B > 0 && (!parents || !mask || !status)) return TV_ERR_INVALID_ARG;
    return launch_tree_mask(parents, B, N, node_counts, mask, depth, status, (cudaStream_t)stream);
}

static bool attn_shape_ok(int B, int N, int Hq, int Hkv, int d, int max_blocks, int bs,
                          tv_dtype dt) {
    if (B < 0 || N < 1 || N > 64 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return false;
    if (max_blocks < 1 || bs < 1) return false;
    if (dt == TV_BF16) return (d == 64 || d == 128) && bs % 16 == 0;
    if (dt == TV_F32) return d >= 32 && d <= 256 && d % 32 == 0;
    return false;
}

size_t tree_verify_attention_workspace(int B, int N, int Hq, int Hkv, int d,
                                       int max_blocks_per_seq, int block_size, tv_dtype dt) {
    if (!attn_shape_ok(B, N, Hq, Hkv, d, max_blocks_per_seq, block_size, dt)) return 0;
    if (dt != TV_BF16 || B == 0) return 0;
    return attn_bf16_workspace(B, N, Hq, Hkv, d, max_blocks_per_seq, block_size);
}

int tree_verify_attention_kernels(int B, int N, int Hq, int Hkv, int d, int max_blocks_per_seq,
                                  int block_size, tv_dtype dt, size_t workspace_bytes) {
    if (dt != TV_F32 && dt != TV_BF16) return -1;
    if (B < 0 || N < 1 || N > 64 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || max_blocks_per_seq < 1 ||
        block_size < 1)
        return -1;
    if (!attn_shape_ok(B, N, Hq, Hkv, d, max_blocks_per_seq, block_size, dt)) return -1;
    if (B == 0) return 0;
    if (dt == TV_BF16 && attn_tc_applicable(N, Hq, Hkv, d))
        return attn_tc_kernels(B, N, Hq, Hkv, workspace_bytes);
    return 1;
}

tv_status tree_verify_attention(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_table, int max_blocks_per_seq,
                                const int32_t* prefix_lens, const uint64_t* mask, int B, int N,
                                const int32_t* node_counts, int Hq, int Hkv, int d,
                                int block_size, int num_blocks, tv_dtype dt, float scale,
                                void* out, int32_t* status, void* workspace,
                                size_t workspace_bytes, tv_stream_t stream) {
    if (dt != TV_F32 && dt != TV_BF16) return TV_ERR_INVALID_ARG;
    if (B < 0 || N < 1 || N > 64 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || max_blocks_per_seq < 1 ||
        block_size < 1 || num_blocks < 1)
        return TV_ERR_INVALID_ARG;
    if (!attn_shape_ok(B, N, Hq, Hkv, d, max_blocks_per_seq, block_size, dt))
        return TV_ERR_UNSUPPORTED;
    if (B == 0) return TV_OK;
    if (!q || !k_cache || !v_cache || !block_table || !prefix_lens || !mask || !out || !status)
        return TV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(k_cache) & 15) || (reinterpret_cast<uintptr_t>(v_cache) & 15) ||
        (reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
        return TV_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) scale = 1.0f / sqrtf((float)d);
    AttnArgs a;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_table = block_table;
    a.max_blocks = max_blocks_per_seq;
    a.prefix_lens = prefix_lens;
    a.mask = mask;
    a.counts = node_counts;
    a.B = B;
    a.N = N;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.d = d;
    a.bs = block_size;
    a.num_blocks = num_blocks;
    a.scale = scale;
    a.out = out;
    a.status = status;
    a.ws = workspace;
    a.ws_bytes = workspace_bytes;
    a.stream = (cudaStream_t)stream;
    return dt == TV_F32 ? launch_attn_f32(a) : launch_attn_bf16(a);
}

size_t tree_accept_workspace(tv_accept_mode mode, int B, int N, int V) {
    if (B <= 0 || N < 1 || N > 64 || V < 1 || V > (1 << 24)) return 0;
    return accept_workspace(mode, B, N, V);
}

tv_status tree_accept(tv_accept_mode mode, const int32_t* parents, const int32_t* draft_tokens,
                      const float* target, const float* draft_probs, int B, int N,
                      const int32_t* node_counts, int V, uint64_t seed, uint64_t offset,
                      int32_t* accept_len, int32_t* path,
                      int32_t* out_tokens, int max_path, int32_t* status, void* workspace,
                      size_t workspace_bytes, tv_stream_t stream) {
    if (mode != TV_ACCEPT_GREEDY && mode != TV_ACCEPT_STOCHASTIC) return TV_ERR_INVALID_ARG;
    if (B < 0 || N < 1 || N > 64 || V < 1 || V > (1 << 24) || max_path < 1)
        return TV_ERR_INVALID_ARG;
    if ((int64_t)B * 16 > 0x7fffffff) return TV_ERR_UNSUPPORTED;
    if (B == 0) return TV_OK;
    if (!parents || !draft_tokens || !target || !accept_len || !path || !out_tokens || !status)
        return TV_ERR_INVALID_ARG;
    if (mode == TV_ACCEPT_STOCHASTIC && !draft_probs) return TV_ERR_INVALID_ARG;
    AcceptArgs a;
    a.mode = mode;
    a.parents = parents;
    a.tokens = draft_tokens;
    a.target = target;
    a.draft = draft_probs;
    a.counts = node_counts;
    a.B = B;
    a.N = N;
    a.V = V;
    a.seed = seed;
    a.offset = offset;
    a.accept_len = accept_len;
    a.path = path;
    a.out_tokens = out_tokens;
    a.max_path = max_path;
    a.status = status;
    a.ws = workspace;
    a.ws_bytes = workspace_bytes;
    a.stream = (cudaStream_t)stream;
    return launch_accept(a);
}

tv_status tree_kv_append(const void* k_new, const void* v_new, const int32_t* depth, int B, int N,
                         const int32_t* node_counts, int Hkv, int d, float rope_theta,
                         void* k_cache, void* v_cache,
                         const int32_t* block_table, int max_blocks_per_seq,
                         const int32_t* prefix_lens, int block_size, int num_blocks, tv_dtype dt,
                         int32_t* status, tv_stream_t stream) {
    if (dt != TV_F32 && dt != TV_BF16) return TV_ERR_INVALID_ARG;
    const int eb = dt == TV_F32 ? 4 : 2;
    if (B < 0 || N < 1 || N > 64 || Hkv < 1 || d < 2 || (d & 1) || block_size < 1 ||
        num_blocks < 1 || max_blocks_per_seq < 1 || !(rope_theta == rope_theta))
        return TV_ERR_INVALID_ARG;
    if ((d * eb) % 16 != 0) return TV_ERR_UNSUPPORTED;
    if (B == 0) return TV_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !block_table || !prefix_lens || !status ||
        (rope_theta > 0.f && !depth))
        return TV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(k_new) & 15) || (reinterpret_cast<uintptr_t>(v_new) & 15) ||
        (reinterpret_cast<uintptr_t>(k_cache) & 15) || (reinterpret_cast<uintptr_t>(v_cache) & 15))
        return TV_ERR_INVALID_ARG;
    return launch_kv_append(k_new, v_new, depth, B, N, node_counts, Hkv, d, rope_theta, k_cache, v_cache,
                            block_table, max_blocks_per_seq, prefix_lens, block_size, num_blocks,
                            eb, status, (cudaStream_t)stream);
}

tv_status kv_compact(void* k_cache, void* v_cache, int num_layers, int64_t layer_stride,
                     const int32_t* block_table, int max_blocks_per_seq,
                     const int32_t* prefix_lens, const int32_t* path, const int32_t* accept_len,
                     int max_path, int B, int Hkv, int d, int block_size, int num_blocks,
                     tv_dtype dt, int32_t* new_lens, int64_t* src_slots, int64_t* dst_slots,
                     int32_t* status, tv_stream_t stream) {
    if (dt != TV_F32 && dt != TV_BF16) return TV_ERR_INVALID_ARG;
    const int eb = dt == TV_F32 ? 4 : 2;
    if (B < 0 || Hkv < 1 || d < 1 || block_size < 1 || num_blocks < 1 || max_blocks_per_seq < 1 ||
        max_path < 1 || num_layers < 0 || layer_stride < 0)
        return TV_ERR_INVALID_ARG;
    if ((d * eb) % 16 != 0 || d * eb > 1024) return TV_ERR_UNSUPPORTED;
    if (num_layers > 1 && layer_stride < (int64_t)num_blocks * Hkv * block_size * d)
        return TV_ERR_INVALID_ARG;
    if (B == 0 || num_layers == 0) return TV_OK;
    if (!k_cache || !v_cache || !block_table || !prefix_lens || !path || !accept_len ||
        !new_lens || !status)
        return TV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(k_cache) & 15) || (reinterpret_cast<uintptr_t>(v_cache) & 15) ||
        ((layer_stride * eb) & 15))
        return TV_ERR_INVALID_ARG;
    CompactArgs a;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.num_layers = num_layers;
    a.layer_stride = layer_stride;
    a.block_table = block_table;
    a.max_blocks = max_blocks_per_seq;
    a.prefix_lens = prefix_lens;
    a.path = path;
    a.accept_len = accept_len;
    a.max_path = max_path;
    a.B = B;
    a.Hkv = Hkv;
    a.d = d;
    a.bs = block_size;
    a.num_blocks = num_blocks;
    a.elem_bytes = eb;
    a.new_lens = new_lens;
    a.src_slots = src_slots;
    a.dst_slots = dst_slots;
    a.status = status;
    a.stream = (cudaStream_t)stream;
    return launch_compact(a);
}

size_t draft_tree_workspace(int B, int topk, int layers) {
    if (B < 1 || topk < 1 || topk > DT_K_MAX || layers < 1) return 0;
    if (draft_tree_nodes(topk, layers) > DT_NODES_MAX) return 0;
    return draft_tree_ws_bytes(B, topk, layers);
}

tv_status draft_tree_expand(const float* logits, const int32_t* root_tokens, int B, int V, int topk,
                            int layer, int layers, int N, int32_t* front_tokens,
                            int32_t* front_src, int32_t* parents, int32_t* tokens, float* scores,
                            int32_t* status, void* workspace, size_t workspace_bytes,
                            tv_stream_t stream) {
    if (B < 0 || V < 1 || V > (1 << 30) || topk < 1 || topk > DT_K_MAX || topk > V || layers < 1 ||
        layer < 0 || layer >= layers || N < 1 || N > 64)
        return TV_ERR_INVALID_ARG;
    const int64_t nodes = draft_tree_nodes(topk, layers);
    if (nodes > DT_NODES_MAX) return TV_ERR_UNSUPPORTED;
    if (N > nodes) return TV_ERR_INVALID_ARG;
    if (B == 0) return TV_OK;
    const bool last = (layer == layers - 1);
    if (!logits || !status || (layer == 0 && !root_tokens) || (last && (!parents || !tokens)))
        return TV_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 15) ||
        workspace_bytes < draft_tree_ws_bytes(B, topk, layers))
        return TV_ERR_WORKSPACE;
    // grid: B x F rows x at most DT_CH_MAX chunks
    if ((int64_t)B * topk * DT_CH_MAX > 0x7fffffff) return TV_ERR_UNSUPPORTED;
    DraftArgs a;
    a.logits = logits;
    a.root_tokens = root_tokens;
    a.B = B;
    a.V = V;
    a.k = topk;
    a.layer = layer;
    a.layers = layers;
    a.N = N;
    a.front_tokens = front_tokens;
    a.front_src = front_src;
    a.parents = parents;
    a.tokens = tokens;
    a.scores = scores;
    a.status = status;
    a.ws = workspace;
    a.ws_bytes = workspace_bytes;
    a.stream = (cudaStream_t)stream;
    return launch_draft_expand(a);
}

}  // extern "C"
