// Tree plan (host).  Everything here follows from one lemma about the packed
// (depth-first pre-order) layout:
//
//   In pre-order the tokens of subtree(u) occupy one contiguous range
//   [off(u), subtree_end(u)).  Let key j lie in node u and query i in node w.
//   Query i attends key j  <=>  u is w or an ancestor of w, and (u != w or
//   j <= i)  <=>  j <= i  and  i < subend[j],  with subend[j] = subtree_end(u).
//
//   (=>) if u is an ancestor-or-self of w then i lies in subtree(u), so
//   i < subtree_end(u); and j <= i because an ancestor's tokens come before its
//   descendants' in pre-order.  (<=) j <= i < subtree_end(u) with j in u puts
//   i inside u's own segment at or after j, or inside subtree(u) after u's
//   segment, i.e. in a descendant of u.
//
// Consequences used below: the queries of key j are the contiguous range
// [j, subend[j]); the q-tiles that use a kv-tile form one contiguous range
// starting at the kv-tile's own index, and none inside it is empty; a
// (q-tile, kv-tile) block with rows [a, b) and columns [c0, c1) is full iff
// c1 - 1 <= a and b <= min subend over the block's keys.
//
// The pages fix the tree and the DFS order (AReaL-DTA abstract: DFS-based
// execution over the rollout prefix tree) and ask for per-q-tile ancestor key
// intervals with full / partial / empty tiles; children are visited in
// ascending node id.

#include "plan.h"

#include <algorithm>
#include <climits>
#include <new>
#include <utility>

namespace treeattn {

namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

int build_plan(const int32_t* parent, const int32_t* seg_len, int32_t n, const tree_attn_plan_opts_t* opts,
               tree_attn_plan_s** out) {
    if (!parent || !seg_len || !out || n <= 0) return TREE_ATTN_ERR_INVALID_ARG;
    *out = nullptr;
    int32_t B = 128;
    int32_t chunk_opt = 0, order_opt = 0;
    if (opts) {
        if (opts->block != 0) B = opts->block;
        chunk_opt = opts->bwd_chunk_qtiles;
        order_opt = opts->bwd_cta_order;
    }
    if (B < 1 || B > 1024 || chunk_opt < 0 || order_opt < 0 || order_opt > 2) return TREE_ATTN_ERR_INVALID_ARG;

    // ---- validate -----------------------------------------------------------
    int64_t N = 0;
    for (int32_t v = 0; v < n; ++v) {
        if (parent[v] < -1 || parent[v] >= n || parent[v] == v) return TREE_ATTN_ERR_INVALID_TREE;
        if (seg_len[v] <= 0) return TREE_ATTN_ERR_INVALID_TREE;
        N += seg_len[v];
    }
    if (N + 2LL * B > INT32_MAX) return TREE_ATTN_ERR_TOO_LARGE;

    tree_attn_plan_s* P = new (std::nothrow) tree_attn_plan_s();
    if (!P) return TREE_ATTN_ERR_OUT_OF_MEMORY;
    try {
        P->n_nodes = n;
        P->cta_order = order_opt;
        P->parent.assign(parent, parent + n);
        P->seg_len.assign(seg_len, seg_len + n);
        P->block = B;
        P->N = N;
        const int32_t T = (int32_t)ceil_div(N, B);
        P->T = T;

        // children in ascending id (CSR, filled in id order)
        std::vector<int32_t> ch_ptr(n + 1, 0), ch(n > 0 ? n : 1);
        for (int32_t v = 0; v < n; ++v)
            if (parent[v] >= 0) ch_ptr[parent[v] + 1]++;
        for (int32_t v = 0; v < n; ++v) ch_ptr[v + 1] += ch_ptr[v];
        {
            std::vector<int32_t> fill(ch_ptr.begin(), ch_ptr.end() - 1);
            for (int32_t v = 0; v < n; ++v)
                if (parent[v] >= 0) ch[fill[parent[v]]++] = v;
        }

        // iterative pre-order: roots ascending, children ascending
        P->node_order.reserve(n);
        std::vector<int32_t> stack;
        stack.reserve(n);
        for (int32_t r = 0; r < n; ++r) {
            if (parent[r] != -1) continue;
            stack.push_back(r);
            while (!stack.empty()) {
                int32_t u = stack.back();
                stack.pop_back();
                P->node_order.push_back(u);
                if ((int32_t)P->node_order.size() > n) break;
                for (int32_t k = ch_ptr[u + 1] - 1; k >= ch_ptr[u]; --k) stack.push_back(ch[k]);
            }
        }
        // a cycle is unreachable from every root, so some node is never visited
        if ((int32_t)P->node_order.size() != n) {
            delete P;
            return TREE_ATTN_ERR_INVALID_TREE;
        }

        // offsets and subtree ends
        P->node_off.assign(n, 0);
        std::vector<int32_t> pos_of(n);
        {
            int64_t o = 0;
            for (int32_t k = 0; k < n; ++k) {
                int32_t u = P->node_order[k];
                pos_of[u] = k;
                P->node_off[u] = (int32_t)o;
                o += seg_len[u];
            }
        }
        std::vector<int32_t> sub_end(n);
        for (int32_t k = n - 1; k >= 0; --k) {
            int32_t u = P->node_order[k];
            if (ch_ptr[u + 1] == ch_ptr[u]) {
                sub_end[u] = P->node_off[u] + seg_len[u];
            } else {
                // the last child in pre-order closes the subtree
                int32_t last = ch[ch_ptr[u + 1] - 1];
                sub_end[u] = sub_end[last];
            }
        }
        P->subend.resize(N);
        for (int32_t u = 0; u < n; ++u)
            std::fill(P->subend.begin() + P->node_off[u], P->subend.begin() + P->node_off[u] + seg_len[u],
                      sub_end[u]);

        int64_t pairs = 0;
        for (int64_t j = 0; j < N; ++j) pairs += P->subend[j] - j;
        P->pairs = pairs;

        // per kv-tile min / max subend
        P->kv_minsub.assign(T, INT32_MAX);
        std::vector<int32_t> kv_maxsub(T, 0);
        for (int64_t j = 0; j < N; ++j) {
            int32_t c = (int32_t)(j / B);
            P->kv_minsub[c] = std::min(P->kv_minsub[c], P->subend[j]);
            kv_maxsub[c] = std::max(kv_maxsub[c], P->subend[j]);
        }
        P->kv_qlo.resize(T);
        P->kv_qhi.resize(T);
        for (int32_t c = 0; c < T; ++c) {
            P->kv_qlo[c] = c;
            P->kv_qhi[c] = (int32_t)((kv_maxsub[c] - 1) / B + 1);
        }

        // per q-tile key intervals and tile classes
        P->qi_ptr.assign(T + 1, 0);
        P->qt_ptr.assign(T + 1, 0);
        std::vector<int32_t> stamp(n, -1);
        std::vector<std::pair<int32_t, int32_t>> iv;
        int32_t pos = 0;  // packed position of the node holding row a
        int64_t n_full = 0;
        for (int32_t t = 0; t < T; ++t) {
            const int32_t a = t * B;
            const int32_t b = (int32_t)std::min<int64_t>(N, (int64_t)a + B);
            while (P->node_off[P->node_order[pos]] + seg_len[P->node_order[pos]] <= a) ++pos;
            iv.clear();
            for (int32_t k = pos; k < n; ++k) {
                const int32_t w = P->node_order[k];
                const int32_t off = P->node_off[w];
                if (off >= b) break;
                // rows of w inside the tile attend [off(w), last row + 1) of w itself
                iv.emplace_back(off, std::min(b, off + seg_len[w]));
                for (int32_t u = parent[w]; u >= 0 && stamp[u] != t; u = parent[u]) {
                    stamp[u] = t;
                    iv.emplace_back(P->node_off[u], P->node_off[u] + seg_len[u]);
                }
            }
            std::sort(iv.begin(), iv.end());
            int32_t cur_lo = -1, cur_hi = -1;
            auto flush = [&]() {
                if (cur_lo < 0) return;
                P->qi_lo.push_back(cur_lo);
                P->qi_hi.push_back(cur_hi);
            };
            for (auto& x : iv) {
                if (cur_lo >= 0 && x.first <= cur_hi) {
                    cur_hi = std::max(cur_hi, x.second);
                } else {
                    flush();
                    cur_lo = x.first;
                    cur_hi = x.second;
                }
            }
            flush();
            P->qi_ptr[t + 1] = (int32_t)P->qi_lo.size();

            int32_t last_c = -1;
            for (int32_t k = P->qi_ptr[t]; k < P->qi_ptr[t + 1]; ++k) {
                for (int32_t c = P->qi_lo[k] / B; c <= (P->qi_hi[k] - 1) / B; ++c) {
                    if (c == last_c) continue;
                    last_c = c;
                    const int64_t c1 = std::min<int64_t>(N, (int64_t)(c + 1) * B);
                    const bool full = (c1 - 1 <= a) && (b <= P->kv_minsub[c]);
                    P->qt_kv.push_back(c);
                    P->qt_cls.push_back(full ? TREE_ATTN_TILE_FULL : TREE_ATTN_TILE_PARTIAL);
                    n_full += full;
                }
            }
            if (P->qt_kv.size() > (size_t)INT32_MAX || P->qi_lo.size() > (size_t)INT32_MAX) {
                delete P;
                return TREE_ATTN_ERR_TOO_LARGE;
            }
            P->qt_ptr[t + 1] = (int32_t)P->qt_kv.size();
        }
        P->n_full = n_full;

        // forward schedule: heaviest q-tile first (stable)
        P->fwd_order.resize(T);
        for (int32_t t = 0; t < T; ++t) P->fwd_order[t] = t;
        std::stable_sort(P->fwd_order.begin(), P->fwd_order.end(), [&](int32_t x, int32_t y) {
            return P->qt_ptr[x + 1] - P->qt_ptr[x] > P->qt_ptr[y + 1] - P->qt_ptr[y];
        });

        // backward schedule: each kv-tile's q-range [c, kv_qhi) cut at the global
        // multiples of S, so that the items of every kv-tile that feed the same
        // q-tiles share one chunk index; items run chunk by chunk (then longest
        // first), which keeps the dQ rows they accumulate into resident in L2.
        // Auto size: 24 q-tiles below 64 q-tiles, 48 below 256, 64 above, doubled
        // while the split kv-tiles would need more than max(2048, 8 T) partial
        // dK/dV slots.  Longer chunks mean fewer partial slots to write and sum
        // but fewer, longer items to spread over the SMs; measured backward main
        // pass + partial sum (ms) at 24 / 48 / 64: segment tree (T = 54) 0.396 /
        // 0.593 / 0.648, GRPO star (T = 88) 0.743 / 0.727 / 0.790, agentic tree
        // (T = 463) 11.93 / 11.75 / 11.58.  On the long shared-context tree the old
        // rule (ceil(tile blocks / 600) = 1,775 q-tiles) gave a 2.07 s backward,
        // 32-96 give 1.28-1.34 s; the slot cap bounds the partials' memory.
        auto slots_for = [&](int64_t S) {
            int64_t n = 0;
            for (int32_t c = 0; c < T; ++c) {
                const int64_t nc = (P->kv_qhi[c] - 1) / S - P->kv_qlo[c] / S + 1;
                if (nc > 1) n += nc;
            }
            return n;
        };
        int64_t S64 = chunk_opt;
        if (S64 <= 0) {
            S64 = T < 64 ? 24 : (T < 256 ? 48 : 64);
            while (S64 < T && slots_for(S64) > std::max<int64_t>(2048, 8 * (int64_t)T)) S64 *= 2;
        }
        const int32_t S = (int32_t)std::min<int64_t>(S64, INT32_MAX);
        P->chunk = S;
        std::vector<int32_t> items;   // {c, t0, t1, slot} plus a sort key below
        std::vector<int32_t> chunk_of;
        for (int32_t c = 0; c < T; ++c) {
            const int32_t lo = P->kv_qlo[c], hi = P->kv_qhi[c];
            const int32_t k0 = lo / S, k1 = (hi - 1) / S;
            const int32_t nc = k1 - k0 + 1;
            int32_t base = -1;
            if (nc > 1) {
                base = (int32_t)P->n_slots;
                P->splits.insert(P->splits.end(), {c, base, nc, 0});
                P->n_slots += nc;
            }
            for (int32_t k = k0; k <= k1; ++k) {
                const int32_t t0 = std::max(lo, k * S), t1 = std::min(hi, (k + 1) * S);
                items.insert(items.end(), {c, t0, t1, nc > 1 ? base + (k - k0) : -1});
                chunk_of.push_back(k);
            }
        }
        const int32_t n_items = (int32_t)(items.size() / 4);
        std::vector<int32_t> idx(n_items);
        for (int32_t i = 0; i < n_items; ++i) idx[i] = i;
        std::stable_sort(idx.begin(), idx.end(), [&](int32_t x, int32_t y) {
            if (chunk_of[x] != chunk_of[y]) return chunk_of[x] < chunk_of[y];
            return items[4 * x + 2] - items[4 * x + 1] > items[4 * y + 2] - items[4 * y + 1];
        });
        P->bwd_items.resize(items.size());
        for (int32_t i = 0; i < n_items; ++i)
            for (int f = 0; f < 4; ++f) P->bwd_items[4 * i + f] = items[4 * idx[i] + f];
        // CSR of the items of each chunk (chunks with no item are empty ranges)
        const int32_t n_chunks = (T + S - 1) / S;
        P->chunk_ptr.assign(n_chunks + 1, 0);
        for (int32_t i = 0; i < n_items; ++i) P->chunk_ptr[chunk_of[idx[i]] + 1]++;
        for (int32_t k = 0; k < n_chunks; ++k) P->chunk_ptr[k + 1] += P->chunk_ptr[k];
    } catch (const std::bad_alloc&) {
        delete P;
        return TREE_ATTN_ERR_OUT_OF_MEMORY;
    }
    *out = P;
    return TREE_ATTN_OK;
}

int build_traj(tree_attn_plan_s* P) {
    TrajInfo& X = P->traj;
    if (X.ready) return TREE_ATTN_OK;
    try {
        const int32_t n = P->n_nodes;
        const int64_t N = P->N;
        std::vector<int32_t> n_child(n, 0), pos_of(n);
        for (int32_t v = 0; v < n; ++v)
            if (P->parent[v] >= 0) n_child[P->parent[v]]++;
        for (int32_t k = 0; k < n; ++k) pos_of[P->node_order[k]] = k;
        // tokens on the path above each node (parents come first in packed order)
        std::vector<int64_t> above(n, 0);
        for (int32_t k = 0; k < n; ++k) {
            const int32_t u = P->node_order[k], p = P->parent[u];
            above[u] = p < 0 ? 0 : above[p] + P->seg_len[p];
        }
        // leaves in packed order, per-node leaf ranges [lo, hi) in that order
        std::vector<int32_t> size(n, 1), before(n + 1, 0);
        for (int32_t k = n - 1; k >= 0; --k) {
            const int32_t u = P->node_order[k], p = P->parent[u];
            if (p >= 0) size[p] += size[u];
        }
        for (int32_t k = 0; k < n; ++k) before[k + 1] = before[k] + (n_child[P->node_order[k]] == 0 ? 1 : 0);
        X.leaves.clear();
        for (int32_t v = 0; v < n; ++v)
            if (n_child[v] == 0) X.leaves.push_back(v);
        const int32_t L = (int32_t)X.leaves.size();
        std::vector<int32_t> id_index(n, -1);
        for (int32_t i = 0; i < L; ++i) id_index[X.leaves[i]] = i;
        X.nodes.assign(6 * (size_t)n, 0);
        X.leaf_of.assign(2 * (size_t)L, 0);
        X.pos_id.assign(N, 0);
        X.mult.assign(N, 0);
        for (int32_t k = 0; k < n; ++k) {
            const int32_t u = P->node_order[k], p = P->parent[u];
            const int32_t lo = before[k], hi = before[k + size[u]];
            int32_t* e = &X.nodes[6 * (size_t)k];
            e[0] = p < 0 ? -1 : pos_of[p];
            e[1] = lo;
            e[2] = hi;
            e[3] = P->node_off[u];
            e[4] = P->seg_len[u];
            e[5] = u;
            for (int32_t i = 0; i < P->seg_len[u]; ++i) {
                X.pos_id[P->node_off[u] + i] = (int32_t)(above[u] + i);
                X.mult[P->node_off[u] + i] = hi - lo;
            }
            if (n_child[u] == 0) {
                X.leaf_of[2 * (size_t)lo] = k;
                X.leaf_of[2 * (size_t)lo + 1] = id_index[u];
            }
        }
        // trajectories, leaves ascending id
        X.traj_ptr.assign(L + 1, 0);
        for (int32_t i = 0; i < L; ++i) {
            const int32_t u = X.leaves[i];
            X.traj_ptr[i + 1] = X.traj_ptr[i] + above[u] + P->seg_len[u];
        }
        if (X.traj_ptr[L] > INT32_MAX) return TREE_ATTN_ERR_TOO_LARGE;
        X.traj_tok.assign(X.traj_ptr[L], 0);
        std::vector<int32_t> path;
        for (int32_t i = 0; i < L; ++i) {
            path.clear();
            for (int32_t u = X.leaves[i]; u >= 0; u = P->parent[u]) path.push_back(u);
            int64_t o = X.traj_ptr[i];
            for (auto it = path.rbegin(); it != path.rend(); ++it)
                for (int32_t t = 0; t < P->seg_len[*it]; ++t) X.traj_tok[o++] = P->node_off[*it] + t;
        }
        X.ready = true;
    } catch (const std::bad_alloc&) {
        return TREE_ATTN_ERR_OUT_OF_MEMORY;
    }
    return TREE_ATTN_OK;
}

}  // namespace treeattn
