/*
 * CPU oracle for EAGLE draft-tree verification — TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously-correct C.  Only tests/, the smoke check and the
 * benchmark's CPU-baseline leg may load this library; the product path never
 * does.  It shares no code, header, table or helper with the CUDA library.
 *
 * Sources (four web pages on EAGLE speculative decoding):
 *   [P1] "vLLM-TreeEagle: Tree Attention optimised EAGLE3 speculative
 *        decoding framework" — section "核心组件 / TreeAttentionLayer" and
 *        "技术创新点 1. Tree Attention并行验证": one forward pass verifies every
 *        candidate path; the tree attention mask is built dynamically for an
 *        arbitrary path structure.
 *   [P2] "EAGLE code principles: tree buffers and KV cache" — section
 *        "KV缓存优化": KVCache.copy(indices, prev_length) selects the kept
 *        entries (index_select), locates the destination (narrow at
 *        prev_length) and copies them there.
 *   [P3] "P-EAGLE in vLLM" — section "技术原理和实现方式" steps 3-4: all
 *        drafts verified in one target pass with a tree mask; acceptance
 *        truncates at the first rejected token; section "技术难点": rollback
 *        on failure, append on success.
 *   [P4] "vLLM EAGLE in practice" — section "无损性保障": greedy speculative
 *        decoding equals greedy decoding; rejection sampling converges to the
 *        target distribution.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - node 0 is the root (parent -1), nodes are in topological order
 *     (0 <= parent[i] < i), N <= 64, a node attends to itself;
 *   - tree node i sits at logical cache position prefix_len + i; logical
 *     position t lives in physical slot block_table[t / bs] * bs + t % bs;
 *   - attention scale 1/sqrt(d) unless given; q-head h reads kv-head
 *     h / (Hq / Hkv); masked keys are excluded (not down-weighted);
 *   - greedy: argmax takes the lowest index on ties and NaN never wins;
 *     the accepted node is the deepest fully matching one, ties to the
 *     smallest id;
 *   - stochastic: Philox4x32-10 (Salmon et al., SC'11) keyed by the seed,
 *     counter (k, b, offset_lo, offset_hi); accept iff u24 * q < p * 2^24
 *     exactly; residual max(0, p - q) sampled through an integer CDF with
 *     2^-40 resolution; on a branching tree the children of a node are tried
 *     in node order with the residual carried in exact integer weights; see
 *     orc_accept_stochastic and orc_accept_stochastic_tree;
 *   - draft-tree construction: top-k children per expanded node by draft
 *     logit, cumulative log-probability scores, the k best new nodes expanded
 *     next, the N - 1 best nodes kept and labelled breadth-first; see
 *     orc_draft_expand and orc_draft_finalize.
 *
 * Parity pins live in tests/test_oracle_*.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_BAD_TREE 2
#define ORC_OUT_OF_RANGE 3
#define ORC_UNSUPPORTED 4
#define ORC_BAD_VALUES 7

/* ------------------------------------------------------------------ */
/* element access                                                      */
/* ------------------------------------------------------------------ */

/* elem == 0: IEEE binary32; elem == 1: bfloat16 bit patterns (the upper 16
 * bits of a binary32), widened exactly. */
static double orc_load(int elem, const void* base, int64_t idx) {
    if (elem == 0) return (double)((const float*)base)[idx];
    uint32_t bits = ((uint32_t)((const uint16_t*)base)[idx]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------ */
/* tree mask ([P1] "动态构建树形注意力掩码")                           */
/* ------------------------------------------------------------------ */

/* Validates one parent array; returns ORC_OK or ORC_BAD_TREE. */
static int orc_check_tree(const int32_t* par, int64_t N) {
    if (N < 1 || N > 64) return ORC_BAD_TREE;
    if (par[0] != -1) return ORC_BAD_TREE;
    for (int64_t i = 1; i < N; ++i)
        if (par[i] < 0 || par[i] >= i) return ORC_BAD_TREE;
    return ORC_OK;
}

/* Node count of sequence b in a batch whose trees may have fewer than N nodes
 * ("P-EAGLE in vLLM", practice 5: shapes are kept fixed, so a sequence's tree
 * occupies the first counts[b] of the N slots and the rest are absent);
 * counts == NULL means every tree has N nodes.  Returns -1 for a count
 * outside [1, N]. */
static int64_t orc_count(const int32_t* counts, int64_t b, int64_t N) {
    if (!counts) return N;
    const int64_t n = counts[b];
    return (n >= 1 && n <= N) ? n : -1;
}

/* mask[b][i] bit j set  <=>  node j is node i or an ancestor of node i.
 * depth[b][i] = number of edges from the root.  A sequence with an invalid
 * parent array gets status ORC_BAD_TREE, mask 0 and depth -1 for all its
 * nodes; with counts, only the first counts[b] nodes exist (the others get
 * mask 0 and depth -1) and a count outside [1, N] gives ORC_OUT_OF_RANGE. */
int orc_tree_mask(const int32_t* parents, int64_t B, int64_t N,
                  uint64_t* mask, int32_t* depth, int32_t* status, const int32_t* counts) {
    for (int64_t b = 0; b < B; ++b) {
        const int32_t* par = parents + b * N;
        const int64_t n = orc_count(counts, b, N);
        int st = (n < 0) ? ORC_OUT_OF_RANGE : orc_check_tree(par, n);
        status[b] = st;
        for (int64_t i = 0; i < N; ++i) {
            if (st != ORC_OK || i >= n) {  /* absent nodes: no bits, depth -1 */
                mask[b * N + i] = 0;
                if (depth) depth[b * N + i] = -1;
                continue;
            }
            /* walk from i up to the root, collecting every node visited */
            uint64_t m = 0;
            int32_t dep = -1;
            for (int64_t j = i; j >= 0; j = par[j]) {
                m |= (uint64_t)1 << j;
                dep += 1;
            }
            mask[b * N + i] = m;
            if (depth) depth[b * N + i] = dep;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* tree-masked paged GQA attention ([P1] TreeAttentionLayer; [P3] step 3) */
/* ------------------------------------------------------------------ */

/* Physical slot of logical position t of sequence b, or -1 when the block
 * table does not cover t or names a block outside [0, num_blocks). */
static int64_t orc_slot(const int32_t* block_table, int64_t max_blocks, int64_t b,
                        int64_t t, int64_t bs, int64_t num_blocks) {
    int64_t lb = t / bs;
    if (t < 0 || lb >= max_blocks) return -1;
    int64_t blk = block_table[b * max_blocks + lb];
    if (blk < 0 || blk >= num_blocks) return -1;
    return blk * bs + t % bs;
}

/* Per node (b, i) and query head h (kv head g = h / (Hq / Hkv)):
 *   visible keys: logical positions 0..P-1 and P+a for every bit a < N set
 *   in mask[b][i];
 *   s_t = scale * <q, k_t>;  O = sum_t softmax(s)_t v_t
 * computed in double: first the maximum, then the exponentials and their
 * sum, then the weighted sum of values.
 *
 * sel lists flat node indices b*N+i to compute (NULL: all B*N, in order);
 * out is [n_sel][Hq][d] doubles.  A sequence whose prefix_len is negative,
 * whose P+N positions are not covered by valid blocks, gets status
 * ORC_OUT_OF_RANGE and zero outputs.  A node with no visible key gets zero.
 * With counts, sequence b has counts[b] nodes: its keys are the P + counts[b]
 * positions, only mask bits below counts[b] are read, and absent nodes get
 * zero outputs (a count outside [1, N]: ORC_OUT_OF_RANGE).
 * The K/V cache layout is [num_blocks][Hkv][bs][d]. */
int orc_attention(int elem, const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_table, int64_t max_blocks,
                  const int32_t* prefix_lens, const uint64_t* mask,
                  int64_t B, int64_t N, int64_t Hq, int64_t Hkv, int64_t d, int64_t bs,
                  int64_t num_blocks, double scale, const int64_t* sel, int64_t n_sel,
                  double* out, int32_t* status, int nthreads, const int32_t* counts) {
    if (Hkv <= 0 || Hq % Hkv != 0) return -1;
    int64_t G = Hq / Hkv;
    if (!(scale > 0.0)) scale = 1.0 / sqrt((double)d);
    /* per-sequence validity */
    for (int64_t b = 0; b < B; ++b) {
        int64_t P = prefix_lens[b];
        const int64_t n = orc_count(counts, b, N);
        int st = ORC_OK;
        if (P < 0 || n < 0) st = ORC_OUT_OF_RANGE;
        for (int64_t t = 0; st == ORC_OK && t < P + n; ++t)
            if (orc_slot(block_table, max_blocks, b, t, bs, num_blocks) < 0) st = ORC_OUT_OF_RANGE;
        status[b] = st;
    }
    int64_t count = sel ? n_sel : B * N;
    (void)nthreads;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
    for (int64_t s = 0; s < count; ++s) {
        int64_t flat = sel ? sel[s] : s;
        int64_t b = flat / N, i = flat % N;
        double* o_node = out + s * Hq * d;
        memset(o_node, 0, sizeof(double) * Hq * d);
        const int64_t n = orc_count(counts, b, N);
        if (status[b] != ORC_OK || i >= n) continue;
        int64_t P = prefix_lens[b];
        /* visible logical positions */
        int64_t nvis = 0;
        int64_t* vis = (int64_t*)malloc(sizeof(int64_t) * (P + n));
        for (int64_t t = 0; t < P; ++t) vis[nvis++] = t;
        for (int64_t a = 0; a < n; ++a)
            if ((mask[b * N + i] >> a) & 1u) vis[nvis++] = P + a;
        double* sc = (double*)malloc(sizeof(double) * (nvis > 0 ? nvis : 1));
        for (int64_t h = 0; h < Hq; ++h) {
            int64_t g = h / G;
            if (nvis == 0) continue;
            const int64_t qoff = ((b * N + i) * Hq + h) * d;
            for (int64_t v = 0; v < nvis; ++v) {
                int64_t slot = orc_slot(block_table, max_blocks, b, vis[v], bs, num_blocks);
                int64_t blk = slot / bs, r = slot % bs;
                int64_t koff = ((blk * Hkv + g) * bs + r) * d;
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c)
                    dot += orc_load(elem, q, qoff + c) * orc_load(elem, k_cache, koff + c);
                sc[v] = scale * dot;
            }
            double mx = -INFINITY;
            for (int64_t v = 0; v < nvis; ++v)
                if (sc[v] > mx) mx = sc[v];
            double den = 0.0;
            for (int64_t v = 0; v < nvis; ++v) {
                sc[v] = exp(sc[v] - mx);
                den += sc[v];
            }
            double* o = o_node + h * d;
            for (int64_t v = 0; v < nvis; ++v) {
                int64_t slot = orc_slot(block_table, max_blocks, b, vis[v], bs, num_blocks);
                int64_t blk = slot / bs, r = slot % bs;
                int64_t voff = ((blk * Hkv + g) * bs + r) * d;
                double w = sc[v] / den;
                for (int64_t c = 0; c < d; ++c) o[c] += w * orc_load(elem, v_cache, voff + c);
            }
        }
        free(sc);
        free(vis);
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* greedy acceptance ([P3] step 4; [P4] 无损性保障: greedy == greedy)   */
/* ------------------------------------------------------------------ */

/* Lowest index of the largest non-NaN value, -1 when every value is NaN. */
static int64_t orc_argmax(const float* row, int64_t V) {
    int64_t best = -1;
    for (int64_t t = 0; t < V; ++t) {
        if (isnan(row[t])) continue;
        if (best < 0 || row[t] > row[best]) best = t;
    }
    return best;
}

static void orc_accept_fail(int64_t b, int64_t max_path, int32_t* accept_len, int32_t* path,
                            int32_t* out_tokens) {
    accept_len[b] = 0;
    for (int64_t j = 0; j < max_path; ++j) {
        path[b * max_path + j] = (j == 0) ? 0 : -1;
        out_tokens[b * max_path + j] = -1;
    }
}

/* Writes the root-to-`chosen` path and the emitted tokens (accepted drafts,
 * then `last`), or fails the sequence when the path does not fit. */
static int orc_emit(int64_t b, const int32_t* par, const int32_t* tok, int64_t chosen,
                    int32_t last, int64_t max_path, int32_t* accept_len, int32_t* path,
                    int32_t* out_tokens) {
    int64_t dep = 0;
    for (int64_t j = chosen; par[j] >= 0; j = par[j]) dep += 1;
    if (dep + 1 > max_path) return ORC_OUT_OF_RANGE;
    accept_len[b] = (int32_t)dep;
    for (int64_t j = 0; j < max_path; ++j) {
        path[b * max_path + j] = -1;
        out_tokens[b * max_path + j] = -1;
    }
    int64_t j = chosen;
    for (int64_t k = dep; k >= 0; --k) {
        path[b * max_path + k] = (int32_t)j;
        j = par[j];
    }
    for (int64_t k = 1; k <= dep; ++k) out_tokens[b * max_path + k - 1] = tok[path[b * max_path + k]];
    out_tokens[b * max_path + dep] = last;
    return ORC_OK;
}

/* Node c >= 1 matches iff draft_tokens[c] == argmax(logits row parent[c]).
 * A node is accepted iff every node on its root path matches (the root is
 * always accepted).  The chosen node is the deepest accepted node, ties to
 * the smallest id.  Outputs: accept_len = depth of the chosen node; path =
 * node ids root..chosen padded with -1; out_tokens = tokens of the accepted
 * drafts followed by argmax of the chosen node's row, padded with -1.
 * Data errors (status != 0) give accept_len 0, path [0,-1,..], tokens -1. */
int orc_accept_greedy(const int32_t* parents, const int32_t* tokens, const float* logits,
                      int64_t B, int64_t N, int64_t V, int64_t max_path,
                      int32_t* accept_len, int32_t* path, int32_t* out_tokens,
                      int32_t* status, const int32_t* counts) {
    int64_t* am = (int64_t*)malloc(sizeof(int64_t) * N);
    int* acc = (int*)malloc(sizeof(int) * N);
    int* dep = (int*)malloc(sizeof(int) * N);
    for (int64_t b = 0; b < B; ++b) {
        const int32_t* par = parents + b * N;
        const int32_t* tok = tokens + b * N;
        const int64_t n = orc_count(counts, b, N);  /* nodes n..N-1 are absent */
        int st = (n < 0) ? ORC_OUT_OF_RANGE : orc_check_tree(par, n);
        for (int64_t c = 1; st == ORC_OK && c < n; ++c)
            if (tok[c] < 0 || tok[c] >= V) st = ORC_OUT_OF_RANGE;
        if (st == ORC_OK && max_path < 1) st = ORC_OUT_OF_RANGE;
        if (st != ORC_OK) {
            status[b] = st;
            orc_accept_fail(b, max_path, accept_len, path, out_tokens);
            continue;
        }
        for (int64_t i = 0; i < n; ++i) am[i] = orc_argmax(logits + (b * N + i) * V, V);
        acc[0] = 1;
        dep[0] = 0;
        for (int64_t c = 1; c < n; ++c) {
            dep[c] = dep[par[c]] + 1;
            acc[c] = acc[par[c]] && ((int64_t)tok[c] == am[par[c]]);
        }
        int64_t chosen = 0;
        for (int64_t c = 1; c < n; ++c)
            if (acc[c] && dep[c] > dep[chosen]) chosen = c;
        if (am[chosen] < 0) st = ORC_BAD_VALUES;
        if (st == ORC_OK)
            st = orc_emit(b, par, tok, chosen, (int32_t)am[chosen], max_path, accept_len, path,
                          out_tokens);
        status[b] = st;
        if (st != ORC_OK) orc_accept_fail(b, max_path, accept_len, path, out_tokens);
    }
    free(am);
    free(acc);
    free(dep);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As  */
/* Easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies with    */
/* the published multipliers and Weyl key increments.                      */
/* ------------------------------------------------------------------ */

void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    const uint64_t mul0 = 0xD2511F53u, mul1 = 0xCD9E8D57u;
    const uint32_t weyl0 = 0x9E3779B9u, weyl1 = 0xBB67AE85u;
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t p0 = mul0 * (uint64_t)c0;
        uint64_t p1 = mul1 * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
        k0 += weyl0;
        k1 += weyl1;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

/* Draw for position k of sequence b: counter (k, b, offset_lo, offset_hi),
 * key (seed_lo, seed_hi). */
static void orc_draw(uint64_t seed, uint64_t offset, int64_t b, int64_t k, uint32_t w[4]) {
    uint32_t ctr[4] = {(uint32_t)k, (uint32_t)b, (uint32_t)offset, (uint32_t)(offset >> 32)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    orc_philox4x32_10(ctr, key, w);
}

/* Fixed-point weight of a probability-like value: values that are NaN or
 * not positive weigh 0, values >= 1 weigh 2^40, others floor(x * 2^40). */
static uint64_t orc_weight(float x) {
    if (!(x > 0.0f)) return 0;
    if (x >= 1.0f) return (uint64_t)1 << 40;
    return (uint64_t)(x * 1099511627776.0f); /* exact power-of-two scaling, then truncation */
}

/* Samples an index with probability w_t / S, S = sum w (exact integers):
 * T = floor(x * S / 2^32) for a uniform 32-bit word x; the result is the
 * smallest t whose inclusive prefix sum exceeds T.  Returns -1 when S = 0. */
static int64_t orc_sample_weights(const uint64_t* w, int64_t V, uint32_t x) {
    uint64_t S = 0;
    for (int64_t t = 0; t < V; ++t) S += w[t];
    if (S == 0) return -1;
    uint64_t T = (uint64_t)(((unsigned __int128)x * (unsigned __int128)S) >> 32);
    uint64_t run = 0;
    for (int64_t t = 0; t < V; ++t) {
        run += w[t];
        if (run > T) return t;
    }
    return -1; /* unreachable: T < S */
}

/* Rejection sampling on a branching draft tree, generalising the chain rule
 * (multi-candidate speculative sampling: the children of the current node are
 * tried in node order, and after each rejection the target is replaced by
 * the normalised residual max(0, p - q); [P4] 无损性保障 states only that the
 * result follows the target distribution, so the rule is ours).  Node c >= 1
 * carries token x_c drawn from q row c; p row c is the target for the token
 * after node c.  Starting at the root (cur = 0):
 *   - the first child c of cur is tested as in the chain: u24 = word0 >> 8 of
 *     draw (b, c), accept iff u24 * q_c(x_c) < p_cur(x_c) * 2^24 (exact in
 *     double);
 *   - after a rejection the residual is kept as exact integer weights w_t with
 *     sum S: after the first rejected child c, w_t = weight(max(0, p_cur,t -
 *     q_c,t)) (one binary32 subtraction); after each further rejected child
 *     c', w_t <- max(0, w_t - floor(weight(q_c',t) * S / 2^40)) with the S
 *     before the update;
 *   - a later child c' is accepted iff u24 * weight(q_c'(x)) * S < w_x * 2^64,
 *     i.e. u24/2^24 * q_c'(x) < w_x / S in exact integers (the left product
 *     u24 * weight < 2^64, times S is formed in 128 bits);
 *   - accepted child: it becomes cur, and its children are tried next;
 *   - every child rejected: the emitted token is drawn from the residual
 *     weights with word1 of the last rejected child's draw; if the residual
 *     sums to 0 (then no later child is tried) it is drawn from
 *     weight(p_cur,t) with that word instead;
 *   - cur has no children: the bonus token is drawn from weight(p_cur,t) with
 *     word1 of draw (b, N) when cur is node N-1, else of draw (b, N + cur), so
 *     that no draw is used twice.
 * On a chain this is exactly orc_accept_stochastic.  Rows p, q, outputs and
 * status for one sequence (the caller offsets them); b keys the draws. */
int orc_accept_stochastic_tree(const int32_t* par, const int32_t* tok, const float* p,
                               const float* q, int64_t one, int64_t N, int64_t V, uint64_t seed,
                               uint64_t offset, int64_t max_path, int32_t* accept_len,
                               int32_t* path, int32_t* out_tokens, int32_t* status, int64_t b) {
    (void)one;
    int st = orc_check_tree(par, N);
    for (int64_t c = 1; st == ORC_OK && c < N; ++c)
        if (tok[c] < 0 || tok[c] >= V) st = ORC_OUT_OF_RANGE;
    if (st == ORC_OK && max_path < 1) st = ORC_OUT_OF_RANGE;
    if (st != ORC_OK) {
        status[0] = st;
        orc_accept_fail(0, max_path, accept_len, path, out_tokens);
        return 0;
    }
    uint64_t* w = (uint64_t*)malloc(sizeof(uint64_t) * V);
    int64_t cur = 0;
    int64_t emitted = -1;
    for (;;) {
        int64_t last_rej = -1;
        uint64_t S = 0;
        int accepted = 0;
        const float* pc = p + cur * V;
        for (int64_t c = cur + 1; c < N; ++c) {
            if (par[c] != cur) continue;
            uint32_t dw[4];
            orc_draw(seed, offset, b, c, dw);
            const uint32_t u24 = dw[0] >> 8;
            const int64_t x = tok[c];
            const float* qc = q + c * V;
            int acc;
            if (last_rej < 0) {
                acc = (double)u24 * (double)qc[x] < (double)pc[x] * 16777216.0;
            } else {
                const unsigned __int128 lhs =
                    (unsigned __int128)((uint64_t)u24 * orc_weight(qc[x])) * S;
                acc = lhs < ((unsigned __int128)w[x] << 64);
            }
            if (acc) {
                cur = c;
                accepted = 1;
                break;
            }
            /* residual update */
            if (last_rej < 0) {
                S = 0;
                for (int64_t t = 0; t < V; ++t) {
                    const float r = pc[t] - qc[t];
                    w[t] = orc_weight(r);
                    S += w[t];
                }
            } else {
                uint64_t S2 = 0;
                for (int64_t t = 0; t < V; ++t) {
                    const uint64_t d =
                        (uint64_t)(((unsigned __int128)orc_weight(qc[t]) * S) >> 40);
                    w[t] = w[t] > d ? w[t] - d : 0;
                    S2 += w[t];
                }
                S = S2;
            }
            last_rej = c;
            if (S == 0) break;
        }
        if (accepted) continue;
        if (last_rej < 0) {
            /* a leaf: bonus token from the target row */
            uint32_t dw[4];
            orc_draw(seed, offset, b, (cur == N - 1) ? N : N + cur, dw);
            for (int64_t t = 0; t < V; ++t) w[t] = orc_weight(pc[t]);
            emitted = orc_sample_weights(w, V, dw[1]);
        } else {
            uint32_t dw[4];
            orc_draw(seed, offset, b, last_rej, dw);
            if (S > 0) {
                emitted = orc_sample_weights(w, V, dw[1]);
            } else {
                for (int64_t t = 0; t < V; ++t) w[t] = orc_weight(pc[t]);
                emitted = orc_sample_weights(w, V, dw[1]);
            }
        }
        break;
    }
    free(w);
    if (emitted < 0) st = ORC_BAD_VALUES;
    if (st == ORC_OK)
        st = orc_emit(0, par, tok, cur, (int32_t)emitted, max_path, accept_len, path, out_tokens);
    status[0] = st;
    if (st != ORC_OK) orc_accept_fail(0, max_path, accept_len, path, out_tokens);
    return 0;
}

/* Rejection sampling along a chain draft ([P3] step 4; [P4] 无损性保障).
 * Node k (1..K, K = N-1) carries draft token x_k drawn from q row k; p row
 * k-1 is the target distribution for that position.  For k = 1..K:
 *   u24 = word0 >> 8 of draw (b, k);  accept iff u24 * q_k(x_k) < p_{k-1}(x_k) * 2^24
 * (both products are exact in double).  At the first rejection k the emitted
 * token is sampled from w_t = weight(max(0, p_{k-1,t} - q_{k,t})) (one binary32
 * subtraction) using word1 of the same draw; if those weights sum to 0 it is
 * sampled from weight(p_{k-1,t}) instead.  When all K drafts are accepted,
 * the bonus token is sampled from weight(p_{K,t}) with word1 of draw (b, K+1).
 * Trees that are not chains go to orc_accept_stochastic_tree. */
int orc_accept_stochastic(const int32_t* parents, const int32_t* tokens, const float* p,
                          const float* q, int64_t B, int64_t N, int64_t V, uint64_t seed,
                          uint64_t offset, int64_t max_path, int32_t* accept_len, int32_t* path,
                          int32_t* out_tokens, int32_t* status, const int32_t* counts) {
    uint64_t* w = (uint64_t*)malloc(sizeof(uint64_t) * V);
    for (int64_t b = 0; b < B; ++b) {
        const int32_t* par = parents + b * N;
        const int32_t* tok = tokens + b * N;
        const int64_t n = orc_count(counts, b, N);  /* nodes n..N-1 are absent */
        int st = (n < 0) ? ORC_OUT_OF_RANGE : orc_check_tree(par, n);
        int is_chain = 1;
        for (int64_t i = 1; i < n; ++i)
            if (par[i] != i - 1) is_chain = 0;
        if (st == ORC_OK && !is_chain) {
            /* the sequence's first n rows are its whole tree */
            orc_accept_stochastic_tree(parents + b * N, tokens + b * N, p + b * N * V,
                                       q + b * N * V, 1, n, V, seed, offset, max_path,
                                       accept_len + b, path + b * max_path,
                                       out_tokens + b * max_path, status + b, b);
            continue;
        }
        for (int64_t c = 1; st == ORC_OK && c < n; ++c)
            if (tok[c] < 0 || tok[c] >= V) st = ORC_OUT_OF_RANGE;
        if (st == ORC_OK && max_path < 1) st = ORC_OUT_OF_RANGE;
        if (st != ORC_OK) {
            status[b] = st;
            orc_accept_fail(b, max_path, accept_len, path, out_tokens);
            continue;
        }
        int64_t K = n - 1;
        int64_t k;
        int64_t emitted = -1;
        for (k = 1; k <= K; ++k) {
            uint32_t dw[4];
            orc_draw(seed, offset, b, k, dw);
            uint32_t u24 = dw[0] >> 8;
            int64_t x = tok[k];
            float pk = p[(b * N + (k - 1)) * V + x];
            float qk = q[(b * N + k) * V + x];
            int accept = (double)u24 * (double)qk < (double)pk * 16777216.0;
            if (accept) continue;
            const float* prow = p + (b * N + (k - 1)) * V;
            const float* qrow = q + (b * N + k) * V;
            for (int64_t t = 0; t < V; ++t) {
                float r = prow[t] - qrow[t];
                w[t] = orc_weight(r);
            }
            emitted = orc_sample_weights(w, V, dw[1]);
            if (emitted < 0) {
                for (int64_t t = 0; t < V; ++t) w[t] = orc_weight(prow[t]);
                emitted = orc_sample_weights(w, V, dw[1]);
            }
            break;
        }
        int64_t chosen; /* last accepted node */
        if (k > K) {
            chosen = K;
            uint32_t dw[4];
            orc_draw(seed, offset, b, K + 1, dw);
            const float* prow = p + (b * N + K) * V;
            for (int64_t t = 0; t < V; ++t) w[t] = orc_weight(prow[t]);
            emitted = orc_sample_weights(w, V, dw[1]);
        } else {
            chosen = k - 1;
        }
        if (emitted < 0) st = ORC_BAD_VALUES;
        if (st == ORC_OK)
            st = orc_emit(b, par, tok, chosen, (int32_t)emitted, max_path, accept_len, path,
                          out_tokens);
        status[b] = st;
        if (st != ORC_OK) orc_accept_fail(b, max_path, accept_len, path, out_tokens);
    }
    free(w);
    return 0;
}

/* ------------------------------------------------------------------ */
/* tree K/V append ([P2] KVCache.cat; the tree's rows go after the prefix) */
/* ------------------------------------------------------------------ */

/* Round a double to binary32 (nearest even), then to the cache element type
 * (elem 1: bfloat16, nearest even on the binary32 bits; NaN kept quiet). */
static void orc_store(int elem, void* base, int64_t idx, double x) {
    float f = (float)x;
    if (elem == 0) {
        ((float*)base)[idx] = f;
        return;
    }
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t h;
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) {
        h = (uint16_t)((u >> 16) | 0x0040u);
    } else {
        u += 0x7FFFu + ((u >> 16) & 1u);
        h = (uint16_t)(u >> 16);
    }
    ((uint16_t*)base)[idx] = h;
}

/* Node i of sequence b goes to logical position t = P_b + i of both caches
 * ([num_blocks][Hkv][bs][d]), every kv head.  With rope_theta > 0 the key is
 * first rotated by position P_b + depth[b][i] (rotate-half pairs (j, j + d/2),
 * j < d/2, angle pos * rope_theta^(-2j/d), in double):
 *   k'_j = k_j cos - k_{j+d/2} sin,   k'_{j+d/2} = k_{j+d/2} cos + k_j sin;
 * values (and keys when rope_theta <= 0) are copied unchanged.  A sequence
 * with P_b < 0, a depth outside [0, N) (rope only) or a position without a
 * valid block gets ORC_OUT_OF_RANGE and no write.  With counts only the first
 * counts[b] nodes are appended (N above reads counts[b]). */
int orc_tree_kv_append(int64_t elem, const void* k_new, const void* v_new, const int32_t* depth,
                       int64_t B, int64_t N, int64_t Hkv, int64_t d, double rope_theta,
                       void* k_cache, void* v_cache, const int32_t* block_table,
                       int64_t max_blocks, const int32_t* prefix_lens, int64_t bs,
                       int64_t num_blocks, int32_t* status, const int32_t* counts) {
    for (int64_t b = 0; b < B; ++b) {
        const int64_t P = prefix_lens[b];
        const int64_t n = orc_count(counts, b, N);  /* only nodes < n are appended */
        int st = ORC_OK;
        if (P < 0 || n < 0) st = ORC_OUT_OF_RANGE;
        for (int64_t i = 0; st == ORC_OK && i < n; ++i) {
            if (orc_slot(block_table, max_blocks, b, P + i, bs, num_blocks) < 0) st = ORC_OUT_OF_RANGE;
            if (rope_theta > 0.0 && (depth[b * N + i] < 0 || depth[b * N + i] >= n))
                st = ORC_OUT_OF_RANGE;
        }
        status[b] = st;
        if (st != ORC_OK) continue;
        for (int64_t i = 0; i < n; ++i) {
            const int64_t slot = orc_slot(block_table, max_blocks, b, P + i, bs, num_blocks);
            const int64_t blk = slot / bs, row = slot % bs;
            for (int64_t g = 0; g < Hkv; ++g) {
                const int64_t src = ((b * N + i) * Hkv + g) * d;
                const int64_t dst = ((blk * Hkv + g) * bs + row) * d;
                for (int64_t e = 0; e < d; ++e)
                    orc_store((int)elem, v_cache, dst + e, orc_load((int)elem, v_new, src + e));
                if (rope_theta <= 0.0) {
                    for (int64_t e = 0; e < d; ++e)
                        orc_store((int)elem, k_cache, dst + e, orc_load((int)elem, k_new, src + e));
                    continue;
                }
                const double pos = (double)(P + depth[b * N + i]);
                const int64_t h = d / 2;
                for (int64_t j = 0; j < h; ++j) {
                    const double ang = pos * pow(rope_theta, -2.0 * (double)j / (double)d);
                    const double c = cos(ang), sn = sin(ang);
                    const double x1 = orc_load((int)elem, k_new, src + j);
                    const double x2 = orc_load((int)elem, k_new, src + j + h);
                    orc_store((int)elem, k_cache, dst + j, x1 * c - x2 * sn);
                    orc_store((int)elem, k_cache, dst + j + h, x2 * c + x1 * sn);
                }
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* KV compaction ([P2] KVCache.copy: index_select -> narrow -> copy_)   */
/* ------------------------------------------------------------------ */

/* For every layer l < num_layers (caches at base + l * layer_stride elements),
 * every kv head and both caches: first gather the rows at logical positions
 * P + path[j], j = 0..accept_len, then write them to positions P + j.
 * new_lens = P + accept_len + 1.  src_slots / dst_slots (nullable) receive
 * the physical slots, padded with -1.  A sequence whose accept_len is outside
 * [0, max_path) or whose positions are not covered by valid blocks gets
 * status ORC_OUT_OF_RANGE, new_len = P and no cache change. */
int orc_kv_compact(int64_t elem_bytes, void* k_cache, void* v_cache, int64_t num_layers,
                   int64_t layer_stride, const int32_t* block_table, int64_t max_blocks,
                   const int32_t* prefix_lens, const int32_t* path, const int32_t* accept_len,
                   int64_t max_path, int64_t B, int64_t Hkv, int64_t d, int64_t bs,
                   int64_t num_blocks, int32_t* new_lens, int64_t* src_slots,
                   int64_t* dst_slots, int32_t* status) {
    for (int64_t b = 0; b < B; ++b) {
        int64_t P = prefix_lens[b];
        int64_t A = accept_len[b];
        int st = ORC_OK;
        if (P < 0 || A < 0 || A >= max_path) st = ORC_OUT_OF_RANGE;
        int64_t* src = (int64_t*)malloc(sizeof(int64_t) * max_path);
        int64_t* dst = (int64_t*)malloc(sizeof(int64_t) * max_path);
        for (int64_t j = 0; st == ORC_OK && j <= A; ++j) {
            int64_t pj = path[b * max_path + j];
            if (pj < 0) { st = ORC_OUT_OF_RANGE; break; }
            src[j] = orc_slot(block_table, max_blocks, b, P + pj, bs, num_blocks);
            dst[j] = orc_slot(block_table, max_blocks, b, P + j, bs, num_blocks);
            if (src[j] < 0 || dst[j] < 0) st = ORC_OUT_OF_RANGE;
        }
        status[b] = st;
        new_lens[b] = (int32_t)(st == ORC_OK ? P + A + 1 : P);
        for (int64_t j = 0; j < max_path; ++j) {
            int ok = (st == ORC_OK && j <= A);
            if (src_slots) src_slots[b * max_path + j] = ok ? src[j] : -1;
            if (dst_slots) dst_slots[b * max_path + j] = ok ? dst[j] : -1;
        }
        if (st == ORC_OK) {
            int64_t row = d * elem_bytes;
            unsigned char* tmp = (unsigned char*)malloc((size_t)((A + 1) * row));
            for (int64_t l = 0; l < num_layers; ++l) {
                for (int kv = 0; kv < 2; ++kv) {
                    unsigned char* cache = (unsigned char*)(kv == 0 ? k_cache : v_cache) +
                                           l * layer_stride * elem_bytes;
                    for (int64_t g = 0; g < Hkv; ++g) {
                        /* gather all sources first (index_select makes a copy) ... */
                        for (int64_t j = 0; j <= A; ++j) {
                            int64_t blk = src[j] / bs, r = src[j] % bs;
                            memcpy(tmp + j * row, cache + ((blk * Hkv + g) * bs + r) * row,
                                   (size_t)row);
                        }
                        /* ... then write the destinations */
                        for (int64_t j = 0; j <= A; ++j) {
                            int64_t blk = dst[j] / bs, r = dst[j] % bs;
                            memcpy(cache + ((blk * Hkv + g) * bs + r) * row, tmp + j * row,
                                   (size_t)row);
                        }
                    }
                }
            }
            free(tmp);
        }
        free(src);
        free(dst);
    }
    return 0;
}

/* Exposes the integer-CDF sampler to the tests (pinned exhaustively there). */
int64_t orc_sample_weights_u32(const uint64_t* w, int64_t V, uint32_t x) {
    return orc_sample_weights(w, V, x);
}

/* ------------------------------------------------------------------ */
/* draft-tree construction ([P1] EnhancedEagleProposer: multi-level    */
/* candidate generation and path pruning; [P2] tree buffers: keep the  */
/* high-probability paths, prune the low-probability branches)         */
/* ------------------------------------------------------------------ */

/* Readings (the pages give the outline only):
 *   - a node's draft row is log-softmax'ed; its candidate children are the k
 *     tokens with the largest logits (ties: lowest token id);
 *   - a node's score is its path's cumulative draft log-probability,
 *     score(child) = score(parent) + (logit - logsumexp(row)).  Which nodes
 *     are kept, and in which order, is an integer result decided by
 *     comparing these scores; the pages fix no precision for it, so the
 *     scores are formed in binary32, the precision the draft logits come
 *     in: the logsumexp accumulated in double and rounded once, then one
 *     binary32 subtraction and one binary32 addition;
 *   - nodes are numbered in creation order: frontier node f's children are
 *     created f-major, child rank j minor;
 *   - the next frontier is the k best nodes created in this layer, by
 *     (score descending, creation id ascending), in that rank order;
 *   - the final tree keeps the root and the N - 1 best other nodes by the
 *     same order, relabelled breadth-first from the root with every node's
 *     children visited in creation order.
 * `margin` (in/out) takes the minimum over every ranking decision of the
 * score gap that decided it, so a caller can tell when another precision
 * could rank differently. */

/* The k largest entries of row[0..V) by (value desc, index asc). */
static void orc_row_topk(const float* row, int64_t V, int64_t k, int64_t* idx) {
    int64_t n = 0;
    for (int64_t t = 0; t < V; ++t) {
        if (n == k && !((double)row[t] > (double)row[idx[k - 1]])) continue;
        int64_t pos = (n < k) ? n++ : k - 1;
        while (pos > 0 && (double)row[t] > (double)row[idx[pos - 1]]) {
            idx[pos] = idx[pos - 1];
            --pos;
        }
        idx[pos] = t;
    }
}

static const double* orc_sort_score;
static int orc_by_score(const void* a, const void* b) {
    const int32_t u = *(const int32_t*)a, v = *(const int32_t*)b;
    if (orc_sort_score[u] > orc_sort_score[v]) return -1;
    if (orc_sort_score[u] < orc_sort_score[v]) return 1;
    return (u > v) - (u < v);
}

/* One layer: rows[F][V] are the draft logits after frontier nodes
 * front[0..F) (creation ids).  Appends F*k nodes at ids count.. and writes
 * the next frontier (min(k, F*k) ids, best first) and, per frontier entry,
 * the row it came from.  Returns ORC_OK, or ORC_BAD_VALUES for a NaN or +inf
 * logit or a row without a finite logit (nothing is appended then). */
int orc_draft_expand(int64_t V, int64_t k, int64_t F, const float* rows, const int32_t* front,
                     int32_t* tok, int32_t* par, double* score, int64_t count,
                     int32_t* new_front, int32_t* new_src, double* margin) {
    double* lse = (double*)malloc(sizeof(double) * F);
    for (int64_t f = 0; f < F; ++f) {
        const float* row = rows + f * V;
        double m = -INFINITY;
        for (int64_t t = 0; t < V; ++t) {
            if (isnan(row[t]) || row[t] == INFINITY) { free(lse); return ORC_BAD_VALUES; }
            if ((double)row[t] > m) m = row[t];
        }
        if (m == -INFINITY) { free(lse); return ORC_BAD_VALUES; }
        double s = 0.0;
        for (int64_t t = 0; t < V; ++t) s += exp((double)row[t] - m);
        lse[f] = m + log(s);
    }
    int64_t* idx = (int64_t*)malloc(sizeof(int64_t) * k);
    for (int64_t f = 0; f < F; ++f) {
        orc_row_topk(rows + f * V, V, k, idx);
        for (int64_t j = 0; j < k; ++j) {
            const int64_t id = count + f * k + j;
            tok[id] = (int32_t)idx[j];
            par[id] = front[f];
            /* ranked in binary32: logsumexp rounded once, then two binary32 operations */
            const float logp = rows[f * V + idx[j]] - (float)lse[f];
            score[id] = (double)((float)score[front[f]] + logp);
        }
    }
    const int64_t M = F * k;
    int32_t* ord = (int32_t*)malloc(sizeof(int32_t) * M);
    for (int64_t i = 0; i < M; ++i) ord[i] = (int32_t)(count + i);
    orc_sort_score = score;
    qsort(ord, (size_t)M, sizeof(int32_t), orc_by_score);
    const int64_t nf = M < k ? M : k;
    for (int64_t r = 0; r < nf; ++r) {
        new_front[r] = ord[r];
        new_src[r] = (int32_t)((ord[r] - count) / k);
    }
    /* the frontier's order decides later creation ids, its boundary decides membership */
    for (int64_t r = 0; r + 1 < M && r < nf; ++r) {
        const double gap = score[ord[r]] - score[ord[r + 1]];
        if (gap < *margin) *margin = gap;
    }
    free(ord);
    free(idx);
    free(lse);
    return ORC_OK;
}

/* Final tree from the C created nodes (node 0 = root): the root plus the N - 1
 * best others, breadth-first.  parents/tokens [N], scores [N].  Returns
 * ORC_OK, or ORC_BAD_TREE when a kept node's parent was not kept. */
int orc_draft_finalize(int64_t C, const int32_t* tok, const int32_t* par, const double* score,
                       int64_t N, int32_t* parents, int32_t* tokens, double* scores,
                       double* margin) {
    int32_t* ord = (int32_t*)malloc(sizeof(int32_t) * (C > 1 ? C - 1 : 1));
    for (int64_t i = 1; i < C; ++i) ord[i - 1] = (int32_t)i;
    orc_sort_score = score;
    qsort(ord, (size_t)(C - 1), sizeof(int32_t), orc_by_score);
    if (N - 1 < C - 1 && N > 1) {
        const double gap = score[ord[N - 2]] - score[ord[N - 1]];
        if (gap < *margin) *margin = gap;
    }
    char* kept = (char*)calloc((size_t)C, 1);
    kept[0] = 1;
    for (int64_t r = 0; r < N - 1; ++r) kept[ord[r]] = 1;
    /* breadth-first from the root: a queue, children in creation order */
    int32_t* queue = (int32_t*)malloc(sizeof(int32_t) * N);
    int32_t* label = (int32_t*)malloc(sizeof(int32_t) * C);
    for (int64_t i = 0; i < C; ++i) label[i] = -1;
    int64_t head = 0, tail = 0;
    queue[tail++] = 0;
    label[0] = 0;
    while (head < tail) {
        const int32_t u = queue[head++];
        for (int64_t v = 1; v < C; ++v) {
            if (kept[v] && par[v] == u && tail < N) {
                label[v] = (int32_t)tail;
                queue[tail++] = (int32_t)v;
            }
        }
    }
    int st = (tail == N) ? ORC_OK : ORC_BAD_TREE;
    for (int64_t i = 0; i < N; ++i) {
        parents[i] = -1;
        tokens[i] = -1;
        scores[i] = -INFINITY;
    }
    if (st == ORC_OK) {
        for (int64_t i = 0; i < N; ++i) {
            const int32_t u = queue[i];
            parents[i] = (u == 0) ? -1 : label[par[u]];
            tokens[i] = tok[u];
            scores[i] = score[u];
        }
    }
    free(label);
    free(queue);
    free(kept);
    free(ord);
    return st;
}
