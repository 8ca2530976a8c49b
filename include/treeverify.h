/*
 * treeverify — target-side verification of an EAGLE draft-token tree on one
 * NVIDIA GB300 (sm_103a).  C ABI.
 *
 * One decode step of speculative decoding, as the pages on EAGLE describe it:
 * the draft head proposes a tree of candidate tokens, and the target model
 * verifies every root-to-leaf path in ONE forward pass under a tree-shaped
 * attention mask ("vLLM-TreeEagle", section 核心组件 / TreeAttentionLayer and
 * 技术创新点 / 1. Tree Attention并行验证), keeps the longest verified path and
 * truncates at the first rejection ("P-EAGLE in vLLM", 技术原理和实现方式,
 * steps 3-4), and then moves the kept entries of the KV cache into place
 * ("EAGLE code principles", KV缓存优化: KVCache.copy with index_select /
 * narrow / copy_).  The four calls below are those steps, in order:
 *
 *   tree_mask_build        parent array -> ancestor bitmask, depth
 *   tree_verify_attention  tree-masked, split-KV, paged GQA attention
 *   tree_accept            greedy argmax or rejection-sampling acceptance
 *   kv_compact             gather-then-scatter of the accepted K/V rows
 *
 * Conventions shared by all calls
 * -------------------------------
 * - Tree: N nodes (1 <= N <= 64).  Node 0 is the root: the last token the
 *   target already emitted, parent -1.  Nodes are in topological order:
 *   0 <= parents[i] < i for i >= 1.  Node i's K/V rows were written into the
 *   paged cache at logical position prefix_len + i before attention runs; its
 *   rotary position is prefix_len + depth(i) (applied by the caller).
 * - Paged KV cache: [num_blocks][Hkv][block_size][d] elements, row-major.
 *   Logical position t of sequence b lives in block block_table[b][t / bs],
 *   row t % bs.  block_table is [B][max_blocks_per_seq] int32.
 * - All pointer arguments are DEVICE pointers owned by the caller, unless a
 *   parameter says otherwise.  The library never allocates device memory:
 *   calls that need scratch take a caller-provided workspace whose size is
 *   given by the matching *_workspace() query.
 * - Every call is asynchronous on `stream` (NULL = the legacy default
 *   stream) and never synchronises with the host.
 * - The return value reports argument/shape errors (checked on the host
 *   before anything is launched: nothing is launched when it is not TV_OK)
 *   and launch failures (TV_ERR_CUDA).  Data-dependent errors are written to
 *   the per-sequence device array `status[B]` (TV_OK or an error code), and
 *   the affected sequence's outputs take a documented, defined value.  No
 *   kernel traps, asserts or waits without bound: a wait that runs out
 *   (about one second) records TV_ERR_TIMEOUT in status.
 * - Calls that overlap on the GPU must not share a workspace.
 */
#ifndef TREEVERIFY_H
#define TREEVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* Identical to cudaStream_t. */
typedef struct CUstream_st* tv_stream_t;

typedef enum {
    TV_OK = 0,
    TV_ERR_INVALID_ARG = 1,  /* host: null pointer, bad size or shape            */
    TV_ERR_BAD_TREE = 2,     /* device: parent array violates the conventions     */
    TV_ERR_OUT_OF_RANGE = 3, /* device: block id, position, token id or length    */
    TV_ERR_UNSUPPORTED = 4,  /* host: shape/dtype not built                       */
    TV_ERR_CUDA = 5,         /* host: a CUDA runtime call or launch failed        */
    TV_ERR_TIMEOUT = 6,      /* device: a bounded wait ran out                    */
    TV_ERR_BAD_VALUES = 7,   /* device: an all-NaN logit row or a zero-mass
                                distribution where a token must be chosen         */
    TV_ERR_WORKSPACE = 8     /* host: workspace missing or too small; device
                                (draft_tree_expand): no state from the previous
                                layer in the workspace                          */
} tv_status;

typedef enum { TV_F32 = 0, TV_BF16 = 1 } tv_dtype;
typedef enum { TV_ACCEPT_GREEDY = 0, TV_ACCEPT_STOCHASTIC = 1 } tv_accept_mode;

/* Static description of a status code.  Never NULL. */
const char* tv_status_string(int status);

/* ABI version of this header (incremented on any signature change). */
int tv_abi_version(void);

/* ------------------------------------------------------------------------
 * Node counts ("P-EAGLE in vLLM", practice 5: shapes are kept fixed so that
 * CUDA graphs stay valid while the drafts change).  tree_mask_build,
 * tree_verify_attention(_noalloc), tree_accept and tree_kv_append take
 * node_counts: a device int32 [B] array, or NULL for trees of N nodes.  With
 * it, sequence b's tree is its first node_counts[b] nodes (node_counts[b] in
 * [1, N]; the other slots are absent and may hold anything): absent nodes get
 * no mask bits and depth -1, no attention output row (their rows of `out` are
 * not written) and are never attended (the keys are positions
 * 0 .. P_b + node_counts[b] - 1), are never accepted (a chain of
 * node_counts[b] nodes has node_counts[b] - 1 drafts, and the draw indices
 * that the rules below write as N read node_counts[b]), and are not
 * appended.  A count outside [1, N] gives the sequence TV_ERR_OUT_OF_RANGE
 * with that call's error outputs.  The values are read on the device, so one
 * captured graph serves every count vector.
 * ------------------------------------------------------------------------ */

/* ------------------------------------------------------------------------
 * tree_mask_build — "vLLM-TreeEagle", 核心组件 / 1. TreeAttentionLayer: the
 * tree attention mask is built dynamically for an arbitrary path structure.
 *
 *   mask[b][i]  bit j set  <=>  node j is node i or one of its ancestors
 *   depth[b][i] number of edges from the root to node i
 *
 * parents: int32 [B][N]; mask: uint64 [B][N]; depth: int32 [B][N] or NULL;
 * status: int32 [B].  A sequence whose parent array breaks the conventions
 * gets status TV_ERR_BAD_TREE, mask 0 and depth -1 for every node.
 * Host errors: B < 0, N outside [1, 64], a NULL required pointer.
 * ------------------------------------------------------------------------ */
tv_status tree_mask_build(const int32_t* parents, int B, int N, const int32_t* node_counts,
                          uint64_t* mask, int32_t* depth, int32_t* status, tv_stream_t stream);

/* ------------------------------------------------------------------------
 * tree_verify_attention — "vLLM-TreeEagle", 技术创新点 / 1. Tree Attention
 * 并行验证 (one forward pass verifies all candidate paths under the tree
 * mask) and "P-EAGLE in vLLM", 技术原理和实现方式 step 3.
 *
 * For node i of sequence b and query head h (kv head g = h / (Hq / Hkv)):
 *   keys   K = { logical positions 0 .. P_b-1 } U { P_b + a : bit a of mask[b][i], a < N }
 *   O[b][i][h] = sum_{t in K} softmax_t(scale * q . k_t) v_t
 * with P_b = prefix_lens[b]; mask bits >= N are ignored; a node with no
 * visible key gets a zero output.
 *
 * q: [B][N][Hq][d] and out: [B][N][Hq][d], same dtype as the caches.
 * dt = TV_BF16: bfloat16 inputs/outputs, float32 accumulation and softmax;
 *   requires d in {64, 128} and block_size a multiple of 16.
 * dt = TV_F32: float32 throughout; requires d <= 256 and d % 32 == 0.
 * scale <= 0 selects 1/sqrt(d).
 * mask: uint64 [B][N] (from tree_mask_build).  status: int32 [B]; a sequence
 * with P_b < 0, P_b + N > max_blocks_per_seq * block_size, or a block id
 * outside [0, num_blocks) among the blocks covering positions 0..P_b+N-1 gets
 * TV_ERR_OUT_OF_RANGE and zero outputs.  Positions beyond P_b + N - 1 in the
 * last block are never read into the result (they may hold anything, NaN
 * included).
 * workspace: device scratch of tree_verify_attention_workspace() bytes,
 * 256-byte aligned.  Its leading bytes are scheduler counters and
 * per-(sequence, kv head, row tile) arrival counters that must be zero
 * before the first call (zero the whole buffer once); every call that
 * completes leaves them at zero again.  The rest holds split-KV partial
 * results (per row: softmax max and sum, normalised output) of the
 * balanced schedule, which gives every SM the same number of key tiles.
 * A smaller workspace of at least 256 bytes is accepted and selects a
 * schedule without partial results in global memory (groups of sequences
 * handed to clusters of SMs); below 256 bytes the call returns
 * TV_ERR_WORKSPACE.
 * ------------------------------------------------------------------------ */
size_t tree_verify_attention_workspace(int B, int N, int Hq, int Hkv, int d,
                                       int max_blocks_per_seq, int block_size, tv_dtype dt);

/* Kernels one tree_verify_attention call with these sizes and this workspace
 * size launches on the current device (launch accounting: the balanced
 * schedule adds a merge kernel); 0 when B = 0, -1 for arguments the call
 * rejects before launching. */
int tree_verify_attention_kernels(int B, int N, int Hq, int Hkv, int d, int max_blocks_per_seq,
                                  int block_size, tv_dtype dt, size_t workspace_bytes);

tv_status tree_verify_attention(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_table, int max_blocks_per_seq,
                                const int32_t* prefix_lens, const uint64_t* mask, int B, int N,
                                const int32_t* node_counts, int Hq, int Hkv, int d,
                                int block_size, int num_blocks,
                                tv_dtype dt, float scale, void* out, int32_t* status,
                                void* workspace, size_t workspace_bytes, tv_stream_t stream);

/* ------------------------------------------------------------------------
 * tree_accept — "P-EAGLE in vLLM", 技术原理和实现方式 step 4 (accept the
 * verified drafts, truncate at the first rejection) and "vLLM EAGLE in
 * practice", 无损性保障 (greedy speculation reproduces greedy decoding;
 * rejection sampling reproduces the target distribution).
 *
 * Row i of `target` ([B][N][V] float32) is the target model's output for the
 * token that FOLLOWS node i: logits for TV_ACCEPT_GREEDY, probabilities for
 * TV_ACCEPT_STOCHASTIC.  draft_tokens: int32 [B][N] (entry 0 unused).
 *
 * TV_ACCEPT_GREEDY: node c >= 1 matches iff draft_tokens[c] equals the argmax
 *   of row parents[c] (lowest index on ties; NaN never wins).  Accepted nodes
 *   are those whose whole root path matches; the chosen node is the deepest
 *   accepted node (ties: smallest id).  The bonus token is the argmax of the
 *   chosen node's row.  draft_probs is ignored (may be NULL).
 * TV_ACCEPT_STOCHASTIC: draft_probs [B][N][V] row k is the draft
 *   distribution node k's token was drawn from.  On a chain (parents[i] =
 *   i - 1):
 *   For k = 1..N-1, with (w0, w1, w2, w3) = Philox4x32-10(counter = (k, b,
 *   offset_lo, offset_hi), key = (seed_lo, seed_hi)) and u = w0 >> 8:
 *   accept x_k iff u * draft_probs[k][x_k] < target[k-1][x_k] * 2^24 (exact).
 *   At the first rejection the emitted token is drawn from the residual
 *   max(0, target[k-1] - draft_probs[k]) (one float32 subtraction per entry),
 *   or from target[k-1] if the residual has zero mass; after N-1 acceptances
 *   it is drawn from target[N-1] with the draw for k = N.  A draw from
 *   weights r uses integer weights floor(min(r,1) * 2^40) (0 for NaN or
 *   r <= 0), their exact sum S, T = floor(w1 * S / 2^32), and returns the
 *   smallest index whose inclusive prefix sum exceeds T.
 *   On a branching tree (this rule is the library's: the pages fix only that
 *   the result follows the target distribution) the children of the current
 *   node cur are tried in node order.  The first is tested as above against
 *   target[cur].  After a rejection the target is the residual, kept as the
 *   integer weights w (sum S): after the first rejected child c, w_t =
 *   weight(target[cur][t] - draft_probs[c][t]); after each further rejected
 *   child c', w_t -= min(w_t, floor(weight(draft_probs[c'][t]) * S / 2^40))
 *   with S before the update.  A later child c' (token x) is accepted iff
 *   u * weight(draft_probs[c'][x]) * S < w_x * 2^64.  An accepted child
 *   becomes cur.  When every child is rejected the token is drawn from w
 *   (from target[cur] if S = 0, and then no later child is tried) with w1
 *   of the last rejected child's draw; when cur is a leaf the bonus token is
 *   drawn from target[cur] with w1 of the draw for k = N (leaf N-1) or
 *   k = N + cur.  On a chain both descriptions agree.  A tree is walked by
 *   one thread-block cluster per sequence, launched after the chain kernel
 *   on the same stream (so a stochastic call launches two kernels when
 *   N > 2).
 *
 * Outputs: accept_len int32 [B] = depth of the chosen node (number of
 * accepted drafts); path int32 [B][max_path] = node ids root..chosen, then
 * -1; out_tokens int32 [B][max_path] = the accepted drafts' tokens followed
 * by the bonus/correction token, then -1.  status int32 [B].  On a data
 * error (TV_ERR_BAD_TREE, TV_ERR_OUT_OF_RANGE for a token outside [0, V) or
 * a path longer than max_path, TV_ERR_BAD_VALUES) the sequence gets accept_len 0, path
 * [0, -1, ...] and out_tokens all -1.
 * workspace: at least tree_accept_workspace() bytes (0 means none is needed
 * and NULL is allowed).  Greedy acceptance on small batches reads every row
 * once in parallel, cut into chunks, and keeps per-chunk and per-row argmax
 * results plus per-row and per-sequence arrival counters there; stochastic
 * acceptance keeps per-chunk weight sums and a per-sequence arrival counter.
 * The counters must be zero before the first call (zero the whole buffer
 * once) and every completed call leaves them at zero; calls sharing one
 * workspace must not run concurrently.
 * Host errors: N outside [1, 64], V outside [1, 2^24], max_path < 1;
 * TV_ERR_WORKSPACE when the workspace is missing or too small.
 * ------------------------------------------------------------------------ */
size_t tree_accept_workspace(tv_accept_mode mode, int B, int N, int V);

tv_status tree_accept(tv_accept_mode mode, const int32_t* parents, const int32_t* draft_tokens,
                      const float* target, const float* draft_probs, int B, int N,
                      const int32_t* node_counts, int V,
                      uint64_t seed, uint64_t offset, int32_t* accept_len, int32_t* path,
                      int32_t* out_tokens, int max_path, int32_t* status, void* workspace,
                      size_t workspace_bytes, tv_stream_t stream);

/* ------------------------------------------------------------------------
 * tree_kv_append — "EAGLE code principles", KV缓存优化: KVCache.cat appends
 * the new tokens' K/V after the prefix.  The step before
 * tree_verify_attention ("write then attend"): node i of sequence b sits at
 * logical position t = P_b + i (physical slot block_table[b][t / block_size]
 * * block_size + t % block_size).
 *
 * k_new, v_new: [B][N][Hkv][d] (dt elements), the tree's keys and values.
 * For every node and kv head the value row, and the key row when
 * rope_theta <= 0, is copied to the node's slot of v_cache / k_cache
 * ([num_blocks][Hkv][block_size][d]).  With rope_theta > 0 the key is first
 * rotated by its tree position P_b + depth[b][i] (depth int32 [B][N], e.g.
 * from tree_mask_build): rotate-half pairs (j, j + d/2), j < d/2, angle
 * pos * rope_theta^(-2j/d):
 *   k'_j = k_j cos - k_{j+d/2} sin,  k'_{j+d/2} = k_{j+d/2} cos + k_j sin,
 * every product and sum in double, rounded to float32, then to dt.
 * status int32 [B]: TV_ERR_OUT_OF_RANGE for P_b < 0, a position
 * P_b .. P_b+N-1 without a valid block, or (rotation only) a depth outside
 * [0, N); such a sequence's cache is left unchanged.
 * Host errors: N outside [1, 64], d odd, d * element size not a multiple of
 * 16 bytes (TV_ERR_UNSUPPORTED), a NULL depth with rope_theta > 0, NaN
 * rope_theta, pointers not 16-byte aligned.
 * ------------------------------------------------------------------------ */
tv_status tree_kv_append(const void* k_new, const void* v_new, const int32_t* depth, int B, int N,
                         const int32_t* node_counts, int Hkv, int d, float rope_theta,
                         void* k_cache, void* v_cache,
                         const int32_t* block_table, int max_blocks_per_seq,
                         const int32_t* prefix_lens, int block_size, int num_blocks, tv_dtype dt,
                         int32_t* status, tv_stream_t stream);

/* ------------------------------------------------------------------------
 * kv_compact — "EAGLE code principles", KV缓存优化: KVCache.copy(indices,
 * prev_length) selects the kept rows (index_select), locates the
 * destination (narrow at prev_length) and copies them there; "P-EAGLE in
 * vLLM", 技术难点: roll back on rejection, append on acceptance.
 *
 * For every layer l < num_layers (caches at k_cache/v_cache + l *
 * layer_stride elements), every kv head and both caches: first read the rows
 * at logical positions P_b + path[b][j], j = 0..accept_len[b], then write them
 * to positions P_b + j (gather-then-scatter, so a destination may be the
 * source of another row).  new_lens[b] = P_b + accept_len[b] + 1.
 * src_slots / dst_slots (int64 [B][max_path], nullable) receive the physical
 * slots block * block_size + row, padded with -1.
 * A sequence with P_b < 0, accept_len outside [0, max_path), a negative path
 * entry, or a position not covered by a valid block gets TV_ERR_OUT_OF_RANGE,
 * new_lens = P_b, slots -1 and no cache change.  Positions P_b .. P_b+N-1
 * must map to blocks that no other sequence writes in the same call.
 * dt selects the element size (TV_BF16: 2 bytes, TV_F32: 4 bytes);
 * d * element size must be a multiple of 16 bytes.
 * ------------------------------------------------------------------------ */
tv_status kv_compact(void* k_cache, void* v_cache, int num_layers, int64_t layer_stride,
                     const int32_t* block_table, int max_blocks_per_seq,
                     const int32_t* prefix_lens, const int32_t* path, const int32_t* accept_len,
                     int max_path, int B, int Hkv, int d, int block_size, int num_blocks,
                     tv_dtype dt, int32_t* new_lens, int64_t* src_slots, int64_t* dst_slots,
                     int32_t* status, tv_stream_t stream);

/* ------------------------------------------------------------------------
 * draft_tree_expand — "vLLM-TreeEagle", 核心组件 / 3. EnhancedEagleProposer
 * (candidates generated over several levels, paths pruned) and "EAGLE code
 * principles", 树结构缓冲 (likely paths precomputed, high-probability paths
 * kept, low-probability branches cut).  The step before verification: the
 * draft tree is grown one layer per call from the draft model's logits (the
 * draft model runs between calls, on the frontier each call returns).
 *
 * logits: fp32 [B][F][V]; F = 1 at layer 0 (the row after the root, whose
 * token is root_tokens[b]), F = topk at later layers (row f follows frontier
 * entry f of the previous call).  Each row's topk largest logits (ties: lowest
 * token id) become children, scored score(parent) + logit - logsumexp(row) in
 * fp32 (the root scores 0).  Nodes are numbered in creation order: row-major,
 * then rank.  The next frontier is the topk best new nodes by (score
 * descending, creation id ascending): front_tokens int32 [B][topk] (their
 * tokens, best first) and front_src int32 [B][topk] (the row each came from);
 * both nullable.  The call for the last layer (layer == layers - 1) also
 * writes the tree: the root and the N - 1 best of all created nodes, same
 * order, labelled breadth-first from the root with each node's children in
 * creation order (so 0 <= parents[i] < i, the order tree_mask_build and
 * tree_accept expect): parents int32 [B][N] (-1 at the root), tokens int32
 * [B][N] (tokens[b][0] = root token), scores fp32 [B][N] (nullable).
 * status int32 [B], written by every call: TV_ERR_OUT_OF_RANGE for a root
 * token outside [0, V) (layer 0), TV_ERR_BAD_VALUES for a NaN or +inf logit
 * or a row without a finite one, TV_ERR_WORKSPACE when the workspace does not
 * hold the sequence's state after layer - 1.  An error sticks for the later
 * layers of the tree; the sequence's frontier outputs become -1, its tree
 * parents and tokens -1 and its scores -inf.
 * workspace: draft_tree_workspace() bytes, 16-byte aligned.  It holds
 * per-sequence arrival counters that must be zero before the first call (zero
 * the whole buffer once; every completed call leaves them at zero), the tree
 * state carried from layer to layer, and per-chunk partial results.  The
 * calls of one tree go in order layer 0, 1, ..., layers - 1 on one workspace;
 * calls sharing a workspace must not run concurrently.
 * Host errors: TV_ERR_INVALID_ARG for topk outside [1, 16] or above V, V
 * outside [1, 2^30], layers < 1, layer outside [0, layers), N outside [1, 64]
 * or above the number of created nodes 1 + topk + (layers - 1) * topk^2, a
 * NULL logits or status, a NULL root_tokens at layer 0, a NULL parents or
 * tokens at the last layer; TV_ERR_UNSUPPORTED for more than 2048 created
 * nodes; TV_ERR_WORKSPACE for a missing, misaligned or small workspace.
 * draft_tree_workspace returns 0 for unsupported sizes.
 * ------------------------------------------------------------------------ */
size_t draft_tree_workspace(int B, int topk, int layers);

tv_status draft_tree_expand(const float* logits, const int32_t* root_tokens, int B, int V,
                            int topk, int layer, int layers, int N, int32_t* front_tokens,
                            int32_t* front_src, int32_t* parents, int32_t* tokens, float* scores,
                            int32_t* status, void* workspace, size_t workspace_bytes,
                            tv_stream_t stream);

/* ------------------------------------------------------------------------
 * tree_verify_attention_noalloc — no counterpart on the pages describing the
 * method; an addition of this library for callers that cannot allocate.
 *
 * Some callers cannot provide device scratch memory: an engine that reserved
 * all of HBM for its own pools up front and does not allocate while decoding,
 * or a plugin host that gives its plugins no allocator.  This call computes
 * exactly what tree_verify_attention computes (same arguments, minus the
 * workspace) but takes its scratch from a fixed array inside the library,
 * and picks the schedule a tree_verify_attention call would pick with a
 * workspace of exactly tree_verify_attention_workspace(...) bytes, so the
 * two give bit-identical outputs.  The array is
 * TV_NOALLOC_SCRATCH_BYTES of device memory that every GPU loading the
 * library holds until the process exits.  It never calls cudaMalloc,
 * cudaFree or any allocating routine.
 *
 * - Sizes whose workspace (tree_verify_attention_workspace) exceeds
 *   TV_NOALLOC_SCRATCH_BYTES are rejected with TV_ERR_WORKSPACE before
 *   anything is launched.
 * - The first call on a device looks up the array's device address (with
 *   that device current) and caches it; make that first call before any
 *   stream capture begins.
 * - All calls share the one array, and it keeps the previous call's
 *   contents: each call first clears (cudaMemsetAsync on `stream`) the part
 *   that must start at zero.  Calls that overlap on the GPU (different
 *   streams, or concurrent host threads) race on the array and must not be
 *   issued.
 * ------------------------------------------------------------------------ */
#define TV_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

size_t tree_verify_attention_noalloc_capacity(void);

tv_status tree_verify_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* block_table, int max_blocks_per_seq,
                                        const int32_t* prefix_lens, const uint64_t* mask, int B,
                                        int N, const int32_t* node_counts, int Hq, int Hkv, int d,
                                        int block_size,
                                        int num_blocks, tv_dtype dt, float scale, void* out,
                                        int32_t* status, tv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TREEVERIFY_H */
