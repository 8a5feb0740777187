/*
 * tree_batch.h -- host-side batching of many rollout trees for libtreeattn:
 * per-tree attention work, longest-processing-time assignment of trees to
 * data-parallel replicas, token-capped microbatches, and the packed forest of
 * a group of trees (one tree_attn_plan / fwd / bwd call per microbatch).
 *
 * Sections: AReaL-DTA abstract (a load-balanced distributed batching strategy
 * that assigns trees to GPUs to balance work); HARTS abstract (a planner that
 * builds microbatches and data-parallel replica assignments from compact-token
 * work).  The pages give no formula for the balancing; this library balances
 * ancestor pairs -- the (query, key) pairs the attention computes, which set
 * the kernels' work -- with the classic LPT rule (largest job first, onto the
 * least-loaded replica).
 *
 * Trees are passed back to back: tree k owns nodes [node_ptr[k], node_ptr[k+1])
 * of parent[] and seg_len[], and its parent indices are local to the tree
 * (0 .. size-1, -1 for a root; a "tree" may itself be a forest).  All arrays
 * are host memory, read during the call only; outputs are caller-allocated.
 * Status codes are those of tree_attn.h (0 = success).  Nothing here needs a
 * GPU.
 */
#ifndef TREE_BATCH_H
#define TREE_BATCH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Work of each tree.  tree_pairs[k] = its ancestor pairs (the plan's n_pairs:
 * sum over nodes u of L_u (L_u + 1) / 2 + L_u * (tokens strictly below u));
 * tree_tokens[k] = its compact tokens.  Either output may be NULL.
 * TREE_ATTN_ERR_INVALID_TREE names a malformed tree (as tree_attn_plan);
 * node_ptr must start at 0 and not decrease. */
int tree_attn_batch_work(int32_t n_trees, const int32_t* node_ptr, const int32_t* parent,
                         const int32_t* seg_len, int64_t* tree_pairs, int64_t* tree_tokens);

/* LPT assignment of n_trees jobs with work tree_work[k] >= 0 to n_replicas
 * replicas: jobs in descending work (ties: ascending index), each onto the
 * replica with the least work so far (ties: lowest replica index).
 * replica_of[k] receives tree k's replica; replica_work[r] (may be NULL) the
 * summed work of replica r.  The largest load is at most 4/3 - 1/(3 R) times
 * the optimum (Graham's bound). */
int tree_attn_batch_assign(int32_t n_trees, const int64_t* tree_work, int32_t n_replicas,
                           int32_t* replica_of, int64_t* replica_work);

/* Microbatches of one replica's trees under a compact-token cap: the trees of
 * replica_of == replica, in descending work (ties: ascending index), go first
 * fit into microbatches of at most max_tokens tokens (a tree above the cap
 * gets a microbatch of its own).  microbatch_of[k] receives the 0-based
 * microbatch of each of the replica's trees and -1 for the other trees;
 * *n_microbatches the count. */
int tree_attn_batch_microbatches(int32_t n_trees, const int64_t* tree_work, const int64_t* tree_tokens,
                                 const int32_t* replica_of, int32_t replica, int64_t max_tokens,
                                 int32_t* microbatch_of, int32_t* n_microbatches);

/* The forest of the selected trees (select[k] != 0), concatenated in
 * ascending tree index with parent indices rebased: out_parent / out_seg_len
 * receive the forest (size = the selected trees' total node count) and
 * out_tree (may be NULL) the source tree of each forest node; *out_n_nodes its
 * size.  The forest's packed order is that of its trees one after another, so
 * one plan over it serves every selected tree at once. */
int tree_attn_batch_forest(int32_t n_trees, const int32_t* node_ptr, const int32_t* parent,
                           const int32_t* seg_len, const uint8_t* select, int32_t* out_parent,
                           int32_t* out_seg_len, int32_t* out_tree, int32_t* out_n_nodes);

#ifdef __cplusplus
}
#endif
#endif /* TREE_BATCH_H */
