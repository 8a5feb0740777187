/*
 * tree_linear.h -- linear attention over a packed rollout tree, chunk by
 * chunk, with the recurrent state handed from each node to its children
 * (libtreeattn).
 *
 * Section: HARTS abstract -- hybrid models interleave softmax attention with
 * linear attention; on a rollout tree the linear layers' recurrent state has to
 * be carried from a shared prefix into every branch.  The pages give no
 * formula; this library computes, per q-head h (kv-head g = h / (hq / hkv)) and
 * a decay gamma_g in (0, 1] per kv-head,
 *
 *   O_i = scale * sum_{j on i's root-to-node path, j <= i} gamma_g^(pos_i - pos_j) (q_i . k_j) v_j
 *
 * (pos = position along the trajectory; gamma = 1 is plain causal linear
 * attention).  Equivalently S_j = gamma S_{j-1} + k_j v_j^T along each
 * trajectory and O_i = scale q_i^T S_i; a child's first token continues from
 * its parent's last state.
 *
 * Chunked form: every node's segment is cut into chunks of at most 128
 * tokens.  Per chunk and kv-head the state increment
 *   dS_c = sum_{m < L} gamma^(L-1-m) k_m v_m^T               (tensor cores)
 * then, every node after its parent, the state entering each chunk
 *   S_in(first chunk of u) = S_out(parent(u)),  S_in(next) = gamma^L S_in + dS_c
 * (an elementwise scan in fp32, parallel over the d x d state entries and over
 * the nodes of one depth; S_in is kept as bf16, the precision the next
 * products read it in), then per chunk
 * and q-head
 *   O = scale (diag(gamma^(m+1)) Q S_in + ((Q K^T) o D) V),  D[m, m'] = gamma^(m-m') for m' <= m
 * (Q K^T, then one accumulation of the masked scores times V and the scaled
 * query rows, rounded to bf16, times S_in on the tensor cores; the decay mask
 * in registers).
 *
 * Tensors as in tree_attn.h: Q, O [N, hq, d] bf16, K, V [N, hkv, d] bf16 in
 * packed order; decay fp32 [hkv] (device), every entry in (0, 1].  The decay
 * lives on the device, so the host cannot check it: a value outside (0, 1]
 * (0, negative, above 1, NaN) records TREE_ATTN_ERR_INVALID_DECAY in the
 * device status word (tree_attn_get_device_status) and leaves the call's
 * outputs undefined.  d = 128.  The workspace holds the per-chunk increments
 * (fp32), entering states (bf16) and the per-node exit states (fp32);
 * contents on entry ignored.  Asynchronous on `stream`.
 */
#ifndef TREE_LINEAR_H
#define TREE_LINEAR_H

#include <stddef.h>
#include <stdint.h>

#include "tree_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Chunks of the plan (<= 128 tokens, inside one node each) and the workspace
 * bytes tree_attn_linear_fwd needs for hkv kv-heads of head_dim d. */
int tree_attn_linear_workspace_size(tree_attn_plan_t plan, int32_t hkv, int32_t d, int64_t* n_chunks,
                                    size_t* ws_bytes);

int tree_attn_linear_fwd(tree_attn_plan_t plan, const void* q, const void* k, const void* v, void* o,
                         const float* decay, int32_t hq, int32_t hkv, int32_t d, float scale,
                         void* workspace, size_t ws_bytes, void* stream);

/* Backward of tree_attn_linear_fwd for the compact output gradient dout
 * ([N, hq, d] bf16, the gradient of one scalar loss; per-trajectory weights
 * are folded into it by the caller):
 *
 *   dQ_i = scale sum_{j on i's path, j <= i} gamma^(pos_i - pos_j) (dO_i . v_j) k_j
 *   dK_j = scale sum_h sum_{i: j on i's path, i >= j} gamma^(pos_i - pos_j) (dO_i^h . v_j) q_i^h
 *   dV_j = scale sum_h sum_{i: j on i's path, i >= j} gamma^(pos_i - pos_j) (q_i^h . k_j) dO_i^h
 *
 * (h over the q-heads of j's kv-head).  dQ is the forward with (q, k, v) =
 * (dO, V, K).  For dK and dV the adjoint of the state runs the other way from
 * the forward's handoff: per chunk F = scale sum_h Q_h^T diag(gamma^(m+1))
 * dO_h, then in reverse packed order Rsum(chunk) = the sum of the entering
 * adjoints of the chunks that continue it (the next chunk of its node, or the
 * first chunk of every child node), R_in = F + gamma^L Rsum, and per chunk
 * dK = diag(gamma^(L-1-m)) V Rsum^T + sum_h dA_h^T Q_h,
 * dV = diag(gamma^(L-1-m)) K Rsum + sum_h P_h^T dO_h (tensor cores, the decay
 * masks in registers).  Outputs dq [N, hq, d], dk / dv [N, hkv, d] bf16,
 * written (not accumulated).  Same workspace as the forward (contents on entry
 * ignored), same argument rules.  Asynchronous on `stream`. */
int tree_attn_linear_bwd(tree_attn_plan_t plan, const void* q, const void* k, const void* v, const void* dout,
                         void* dq, void* dk, void* dv, const float* decay, int32_t hq, int32_t hkv, int32_t d,
                         float scale, void* workspace, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* TREE_LINEAR_H */
