/*
 * tree_loss.h -- the calls around the attention at the loss boundary of
 * packed-tree training (libtreeattn): per-trajectory views of a plan, token
 * weights folded into a gradient, per-trajectory next-token log-probs from
 * compact logits, and subtree (segment-level) advantages.
 *
 * Trajectories.  One per leaf of the tree or forest, in ascending leaf node
 * id; trajectory l is the compact tokens of the nodes on the root-to-leaf path,
 * in path order.  A compact token belongs to every trajectory through its node
 * (its multiplicity) and sits at the same position in each of them (its
 * position id, for rotary embeddings) -- the HARTS abstract's compact-token
 * view of trajectories that share histories.
 *
 * Conventions are those of tree_attn.h: status 0 = success, negative =
 * TREE_ATTN_ERR_*; host outputs are caller-allocated; device pointers belong to
 * the caller, are 16-byte aligned and are used asynchronously on `stream`.
 * The first device call with a plan on a device uploads its trajectory tables
 * (allocates and synchronises once).
 */
#ifndef TREE_LOSS_H
#define TREE_LOSS_H

#include <stddef.h>
#include <stdint.h>

#include "tree_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Trajectory counts: n_leaves, and n_expanded = sum of trajectory lengths
 * (the tokens training every trajectory on its own would process). */
int tree_attn_plan_trajectory_info(tree_attn_plan_t plan, int32_t* n_leaves, int64_t* n_expanded);

/* Host copies: leaf_ids [n_leaves] (ascending), traj_ptr [n_leaves+1] offsets
 * into traj_tokens [n_expanded] = compact (packed) token index of every
 * trajectory position.  Any pointer may be NULL. */
int tree_attn_plan_trajectories(tree_attn_plan_t plan, int32_t* leaf_ids, int64_t* traj_ptr, int32_t* traj_tokens);

/* Host copies, [n_tokens] each, packed order: multiplicity = trajectories
 * containing the token (leaves under its node); position id = its 0-based
 * position along those trajectories.  Either pointer may be NULL. */
int tree_attn_plan_token_info(tree_attn_plan_t plan, int32_t* multiplicity, int32_t* position_ids);

/* Token weights folded into a gradient (HARTS abstract: compact tokens stand
 * for several trajectory tokens; a loss weights each compact token by how
 * many trajectory tokens it stands for, or by any other per-token weight):
 *   y[t, e] = bf16(x[t, e] * w[t])   for t < n_rows, e < row_elems
 * x, y bf16 [n_rows, row_elems] (may be the same buffer), w fp32 [n_rows];
 * row_elems a multiple of 8.  Device pointers, asynchronous on `stream`. */
int tree_attn_scale_rows(const void* x, const float* w, void* y, int64_t n_rows, int64_t row_elems, void* stream);

/* Per-trajectory next-token log-probs from compact logits.  logits bf16
 * [n_tokens, vocab] in packed order (vocab a multiple of 8); tokens int32
 * [n_tokens] = the token id at each compact position.  Writes
 *   row_lse[t]  = ln sum_v exp(logits[t, v])                    [n_tokens]
 *   logprobs[k] = logits[r, tokens[s]] - row_lse[r]             [n_expanded - n_leaves]
 * where prediction k is the k-th (position p, p+1) pair of the trajectories in
 * order, r = the compact token at p and s = the one at p+1.  At the end of a
 * shared segment r is the same for every child trajectory and s differs: the
 * one compact row predicts each child's first token.  A token id outside
 * [0, vocab) gives NaN.  Device pointers, asynchronous on `stream`. */
int tree_attn_traj_logprobs(tree_attn_plan_t plan, const void* logits, int64_t vocab, const int32_t* tokens,
                            float* row_lse, float* logprobs, void* stream);

/* Subtree (segment-level) advantages.  Section: TreePO (Approach: advantages
 * estimated over sub-trees from collective descendant outcomes; tree-based
 * advantage estimation with trajectory subgroups that share predecessor nodes;
 * discussion: simple subgroup averaging vs size-weighted aggregation, root
 * group removable).  Reading of this library (the pages give no formula):
 *   group G(u) = the leaves under node u; mean_u, std_u their rewards' mean and
 *   population standard deviation;
 *   for leaf l, the subgroups are the nodes u on its root path (u = l included)
 *   with |G(u)| >= 2 (without roots if TREE_ADV_NO_ROOT);
 *   a_u(l) = R_l - mean_u, divided by (std_u + eps) with TREE_ADV_NORM_STD;
 *   A(l)   = sum_u w_u a_u(l) / sum_u w_u with w_u = 1, or |G(u)| with
 *            TREE_ADV_SIZE_WEIGHTED; 0 when l has no subgroup;
 *   node_coef[u] = sum of A(l) over G(u); token_coef[t] = node_coef of t's node
 *   (the policy-gradient weight of a compact token: the advantages of every
 *   trajectory through it).
 * leaf_reward / leaf_adv: fp32 [n_leaves], leaves in ascending node id;
 * node_coef fp32 [n_nodes] by node id; token_coef fp32 [n_tokens], packed
 * order.  Device pointers, asynchronous on `stream`; n_nodes <= 16384. */
#define TREE_ADV_NORM_STD      1
#define TREE_ADV_SIZE_WEIGHTED 2
#define TREE_ADV_NO_ROOT       4
int tree_attn_subtree_advantage(tree_attn_plan_t plan, const float* leaf_reward, int32_t flags, float eps,
                                float* leaf_adv, float* node_coef, float* token_coef, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* TREE_LOSS_H */
