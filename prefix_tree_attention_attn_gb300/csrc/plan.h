// Host-side tree plan: packed layout, per-token subtree ends, per-q-tile key
// intervals and tile classes, and the forward / backward work schedules.
#pragma once

#include <cstdint>
#include <mutex>
#include <vector>

#include <cuda.h>

#include "tree_attn.h"

namespace treeattn {

constexpr int kMaxDevices = 64;

// Device copy of the plan tables (one per device; pointers into one buffer).
struct DevicePlan {
    void* base = nullptr;
    int32_t* subend = nullptr;     // [T*block], zero past N
    int32_t* qt_ptr = nullptr;     // [T+1]
    int32_t* qt_ent = nullptr;     // [entries] kv_tile*2 + (partial ? 1 : 0)
    int32_t* fwd_order = nullptr;  // [T]
    int32_t* kv_minsub = nullptr;  // [T]
    int32_t* bwd_items = nullptr;  // [4*items]
    int32_t* splits = nullptr;     // [4*splits] {kv-tile, first slot, n slots, 0}
    int32_t* chunk_ptr = nullptr;  // [n_chunks+1] first backward item of each q-range chunk
    bool ready = false;
    // trajectory tables of the loss-boundary calls (uploaded on their first use)
    void* traj_base = nullptr;
    int32_t* pred = nullptr;       // [2*n_pred] {row, target row} per next-token prediction
    int32_t* nodes = nullptr;      // [6*n_nodes] per packed node: parent's packed index, leaf range lo, hi,
                                   //             first token, tokens, node id
    int32_t* leaf_of = nullptr;    // [2*n_leaves] per leaf in packed order: packed node index, id-order index
    bool traj_ready = false;
    // chunk tables of the linear-attention calls (uploaded on their first use)
    void* lin_base = nullptr;
    int32_t* chunks = nullptr;     // [4*n_chunks] {first token, tokens, packed node, 0}
    int32_t* lnodes = nullptr;     // [4*n_nodes] per packed node {parent's packed index, first chunk, chunks,
                                   //   1 if the last child of its parent}
    int32_t* lvl_nodes = nullptr;  // packed nodes by depth (LinInfo::lvl_ptr gives each depth's range)
    int32_t* kids = nullptr;       // [n_nodes+1] child offsets, then the children in packed order
    bool lin_ready = false;
};

// Chunks of at most 128 tokens inside each node's segment, in packed order.
struct LinInfo {
    std::vector<int32_t> chunks;   // as DevicePlan::chunks
    std::vector<int32_t> lnodes;   // as DevicePlan::lnodes
    std::vector<int32_t> lvl_ptr;  // [depths+1] ranges of lvl_nodes; empty for trees too deep to scan by depth
    std::vector<int32_t> lvl_nodes;
    std::vector<int32_t> kids;     // as DevicePlan::kids
    bool ready = false;
};

// Per-trajectory view of a plan (built on first use): leaves in ascending node
// id, each trajectory's compact tokens, per-token position ids and
// multiplicities, and per-node leaf ranges in packed order.
struct TrajInfo {
    std::vector<int32_t> leaves;      // leaf node ids, ascending
    std::vector<int64_t> traj_ptr;    // [n_leaves+1]
    std::vector<int32_t> traj_tok;    // [n_expanded] compact token of each trajectory position
    std::vector<int32_t> pos_id;      // [N] position of the token along its trajectories
    std::vector<int32_t> mult;        // [N] trajectories containing the token
    std::vector<int32_t> nodes;       // [6*n_nodes] as DevicePlan::nodes
    std::vector<int32_t> leaf_of;     // [2*n_leaves] as DevicePlan::leaf_of
    bool ready = false;
};

struct Plan {
    int32_t n_nodes = 0;
    int32_t block = 128;
    int64_t N = 0;
    int32_t T = 0;
    int64_t pairs = 0;
    int64_t n_full = 0;
    int32_t chunk = 0;
    int32_t cta_order = 0;   // backward CTA order: 0 auto, 1 item-major, 2 head-major
    std::vector<int32_t> node_order, node_off, subend;
    std::vector<int32_t> qi_ptr, qi_lo, qi_hi;
    std::vector<int32_t> qt_ptr, qt_kv;
    std::vector<uint8_t> qt_cls;
    std::vector<int32_t> kv_qlo, kv_qhi, kv_minsub;
    std::vector<int32_t> fwd_order;
    std::vector<int32_t> bwd_items;   // 4 per item
    std::vector<int32_t> splits;      // 4 per split kv-tile
    std::vector<int32_t> chunk_ptr;   // items of chunk k: [chunk_ptr[k], chunk_ptr[k+1])
    int64_t n_slots = 0;
    std::vector<int32_t> parent, seg_len;   // the tree as given
    TrajInfo traj;                          // guarded by mu
    LinInfo lin;                            // guarded by mu

    std::mutex mu;
    DevicePlan dev[kMaxDevices];
};

}  // namespace treeattn

struct tree_attn_plan_s : public treeattn::Plan {};

namespace treeattn {
// Builds *out (a new plan); returns a TREE_ATTN_* status.
int build_plan(const int32_t* parent, const int32_t* seg_len, int32_t n_nodes,
               const tree_attn_plan_opts_t* opts, tree_attn_plan_s** out);
// Fills P->traj (call with P->mu held); returns a TREE_ATTN_* status.
int build_traj(tree_attn_plan_s* P);
// The current device if it is a usable sm_103 device.
int current_device(int* dev);
// TMA map of a bf16 [rows, heads, d] tensor: boxes of 64 features x 1 head x
// 128 rows, 128-byte swizzle.
int make_tensor_map(CUtensorMap* m, const void* base, int64_t rows, int heads, int d);
// Device address of the current device's status word (kernels' bounded waits).
int get_status_ptr(int dev, int** out);
}  // namespace treeattn
