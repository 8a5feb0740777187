// Host-side tree plan: packed layout, per-token subtree ends, per-q-tile key
// intervals and tile classes, and the forward / backward work schedules.
#pragma once

#include <cstdint>
#include <mutex>
#include <vector>

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
    std::vector<int32_t> node_order, node_off, subend;
    std::vector<int32_t> qi_ptr, qi_lo, qi_hi;
    std::vector<int32_t> qt_ptr, qt_kv;
    std::vector<uint8_t> qt_cls;
    std::vector<int32_t> kv_qlo, kv_qhi, kv_minsub;
    std::vector<int32_t> fwd_order;
    std::vector<int32_t> bwd_items;   // 4 per item
    std::vector<int32_t> splits;      // 4 per split kv-tile
    int64_t n_slots = 0;

    std::mutex mu;
    DevicePlan dev[kMaxDevices];
};

}  // namespace treeattn

struct tree_attn_plan_s : public treeattn::Plan {};

namespace treeattn {
// Builds *out (a new plan); returns a TREE_ATTN_* status.
int build_plan(const int32_t* parent, const int32_t* seg_len, int32_t n_nodes,
               const tree_attn_plan_opts_t* opts, tree_attn_plan_s** out);
}  // namespace treeattn
