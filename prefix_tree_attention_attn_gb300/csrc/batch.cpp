// Host-side batching of rollout trees: per-tree ancestor-pair work, LPT
// assignment to data-parallel replicas, token-capped microbatches and the
// packed forest of a group of trees (see include/tree_batch.h).
//
// Work of a tree.  Query token i in node w attends the tokens of every
// ancestor of w in full and the tokens of w up to itself.  Summed over the
// queries, node u contributes L_u (L_u + 1) / 2 pairs from its own segment
// and L_u * D_u pairs from the queries below it (D_u = tokens strictly below
// u) -- the same count as the plan's sum over keys of (subend[j] - j).
#include <algorithm>
#include <new>
#include <numeric>
#include <vector>

#include "tree_attn.h"
#include "tree_batch.h"

namespace {

// Validates tree k (parent range, self-parent, seg_len > 0, acyclic) and
// returns its pairs and tokens.
int tree_work(const int32_t* parent, const int32_t* seg_len, int32_t n, int64_t* pairs, int64_t* tokens) {
    if (n <= 0) return TREE_ATTN_ERR_INVALID_TREE;
    int64_t tok = 0;
    for (int32_t v = 0; v < n; ++v) {
        if (parent[v] < -1 || parent[v] >= n || parent[v] == v || seg_len[v] <= 0) return TREE_ATTN_ERR_INVALID_TREE;
        tok += seg_len[v];
    }
    // children-first order by repeated peeling of nodes whose children are done
    std::vector<int32_t> pending(n, 0), order;
    order.reserve(n);
    for (int32_t v = 0; v < n; ++v)
        if (parent[v] >= 0) pending[parent[v]]++;
    for (int32_t v = 0; v < n; ++v)
        if (pending[v] == 0) order.push_back(v);
    for (size_t k = 0; k < order.size(); ++k) {
        const int32_t p = parent[order[k]];
        if (p >= 0 && --pending[p] == 0) order.push_back(p);
    }
    if ((int32_t)order.size() != n) return TREE_ATTN_ERR_INVALID_TREE;   // a cycle never peels
    std::vector<int64_t> below(n, 0);   // tokens strictly below each node
    int64_t pr = 0;
    for (int32_t v : order) {
        const int64_t L = seg_len[v];
        pr += L * (L + 1) / 2 + L * below[v];
        if (parent[v] >= 0) below[parent[v]] += below[v] + L;
    }
    *pairs = pr;
    *tokens = tok;
    return TREE_ATTN_OK;
}

int check_ptr(int32_t n_trees, const int32_t* node_ptr) {
    if (n_trees < 0 || !node_ptr || node_ptr[0] != 0) return TREE_ATTN_ERR_INVALID_ARG;
    for (int32_t k = 0; k < n_trees; ++k)
        if (node_ptr[k + 1] < node_ptr[k]) return TREE_ATTN_ERR_INVALID_ARG;
    return TREE_ATTN_OK;
}

// Indices in descending work, ties by ascending index.
std::vector<int32_t> lpt_order(int32_t n, const int64_t* work) {
    std::vector<int32_t> idx(n);
    std::iota(idx.begin(), idx.end(), 0);
    std::stable_sort(idx.begin(), idx.end(), [&](int32_t a, int32_t b) { return work[a] > work[b]; });
    return idx;
}

}  // namespace

extern "C" {

int tree_attn_batch_work(int32_t n_trees, const int32_t* node_ptr, const int32_t* parent, const int32_t* seg_len,
                         int64_t* tree_pairs, int64_t* tree_tokens) {
    int st = check_ptr(n_trees, node_ptr);
    if (st) return st;
    if (n_trees > 0 && node_ptr[n_trees] > 0 && (!parent || !seg_len)) return TREE_ATTN_ERR_INVALID_ARG;
    try {
        for (int32_t k = 0; k < n_trees; ++k) {
            int64_t pr = 0, tok = 0;
            const int32_t b = node_ptr[k];
            st = tree_work(parent + b, seg_len + b, node_ptr[k + 1] - b, &pr, &tok);
            if (st) return st;
            if (tree_pairs) tree_pairs[k] = pr;
            if (tree_tokens) tree_tokens[k] = tok;
        }
    } catch (const std::bad_alloc&) {
        return TREE_ATTN_ERR_OUT_OF_MEMORY;
    }
    return TREE_ATTN_OK;
}

int tree_attn_batch_assign(int32_t n_trees, const int64_t* tree_work, int32_t n_replicas, int32_t* replica_of,
                           int64_t* replica_work) {
    if (n_trees < 0 || n_replicas <= 0 || (n_trees > 0 && (!tree_work || !replica_of)))
        return TREE_ATTN_ERR_INVALID_ARG;
    for (int32_t k = 0; k < n_trees; ++k)
        if (tree_work[k] < 0) return TREE_ATTN_ERR_INVALID_ARG;
    try {
        std::vector<int64_t> load(n_replicas, 0);
        for (int32_t k : lpt_order(n_trees, tree_work)) {
            int32_t best = 0;
            for (int32_t r = 1; r < n_replicas; ++r)
                if (load[r] < load[best]) best = r;
            replica_of[k] = best;
            load[best] += tree_work[k];
        }
        if (replica_work) std::copy(load.begin(), load.end(), replica_work);
    } catch (const std::bad_alloc&) {
        return TREE_ATTN_ERR_OUT_OF_MEMORY;
    }
    return TREE_ATTN_OK;
}

int tree_attn_batch_microbatches(int32_t n_trees, const int64_t* tree_work, const int64_t* tree_tokens,
                                 const int32_t* replica_of, int32_t replica, int64_t max_tokens,
                                 int32_t* microbatch_of, int32_t* n_microbatches) {
    if (n_trees < 0 || max_tokens <= 0 || !n_microbatches ||
        (n_trees > 0 && (!tree_work || !tree_tokens || !replica_of || !microbatch_of)))
        return TREE_ATTN_ERR_INVALID_ARG;
    try {
        std::vector<int64_t> fill;   // tokens per open microbatch
        for (int32_t k = 0; k < n_trees; ++k) microbatch_of[k] = -1;
        for (int32_t k : lpt_order(n_trees, tree_work)) {
            if (replica_of[k] != replica) continue;
            if (tree_tokens[k] < 0) return TREE_ATTN_ERR_INVALID_ARG;
            int32_t m = 0;
            while (m < (int32_t)fill.size() && fill[m] + tree_tokens[k] > max_tokens) ++m;
            if (m == (int32_t)fill.size()) fill.push_back(0);
            fill[m] += tree_tokens[k];
            microbatch_of[k] = m;
        }
        *n_microbatches = (int32_t)fill.size();
    } catch (const std::bad_alloc&) {
        return TREE_ATTN_ERR_OUT_OF_MEMORY;
    }
    return TREE_ATTN_OK;
}

int tree_attn_batch_forest(int32_t n_trees, const int32_t* node_ptr, const int32_t* parent, const int32_t* seg_len,
                           const uint8_t* select, int32_t* out_parent, int32_t* out_seg_len, int32_t* out_tree,
                           int32_t* out_n_nodes) {
    int st = check_ptr(n_trees, node_ptr);
    if (st) return st;
    if (!select || !out_n_nodes || (n_trees > 0 && node_ptr[n_trees] > 0 && (!parent || !seg_len)))
        return TREE_ATTN_ERR_INVALID_ARG;
    int64_t total = 0;
    for (int32_t k = 0; k < n_trees; ++k)
        if (select[k]) total += node_ptr[k + 1] - node_ptr[k];
    if (total > 0 && (!out_parent || !out_seg_len)) return TREE_ATTN_ERR_INVALID_ARG;
    int32_t o = 0;
    for (int32_t k = 0; k < n_trees; ++k) {
        if (!select[k]) continue;
        const int32_t b = node_ptr[k], n = node_ptr[k + 1] - b;
        for (int32_t v = 0; v < n; ++v) {
            const int32_t p = parent[b + v];
            if (p < -1 || p >= n) return TREE_ATTN_ERR_INVALID_TREE;
            out_parent[o + v] = p < 0 ? -1 : p + o;
            out_seg_len[o + v] = seg_len[b + v];
            if (out_tree) out_tree[o + v] = k;
        }
        o += n;
    }
    *out_n_nodes = o;
    return TREE_ATTN_OK;
}

}  // extern "C"
