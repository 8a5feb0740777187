// Kernel parameter blocks and launch entry points (internal to libtreeattn).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace treeattn {

struct FwdParams {
    const int32_t* qt_ptr;     // [T+1]
    const int32_t* qt_ent;     // kv_tile*2 + partial
    const int32_t* fwd_order;  // [T]
    const int32_t* subend;     // [T*128], 0 past N
    const int32_t* kv_minsub;  // [T] min subend over each kv-tile's keys
    float* lse;                // [hq, N]
    int32_t N, hq, group;
    float scale_log2;          // softmax_scale * log2(e)
    int* status;               // device status word
};

struct BwdPreParams {
    const uint16_t* o;         // [N, hq, d] bf16 bits
    const uint16_t* dout;
    const float* lse;          // [hq, N]
    float* delta;              // [hq, Npad]
    float* lse2;               // [hq, Npad]  LSE * log2(e); +inf past N
    float* dq_acc;             // [N, hq, d] fp32, zeroed here
    int32_t N, Npad, hq, d;
};

struct BwdParams {
    const int32_t* items;      // 4 per item
    const int32_t* subend;     // [T*128]
    const int32_t* kv_minsub;  // [T]
    const float* delta;        // [hq, Npad]
    const float* lse2;         // [hq, Npad]
    float* dq_acc;             // [N, hq, d]
    uint16_t* dk;              // [N, hkv, d] bf16 bits
    uint16_t* dv;
    float* part;               // [slots, hkv, 2, 128, d] fp32
    int32_t N, Npad, hq, hkv, group;
    float scale;               // softmax_scale
    float scale_log2;          // softmax_scale * log2(e)
    int* status;               // device status word
};

struct BwdPostParams {
    const float* dq_acc;       // [N, hq, d]
    uint16_t* dq;              // [N, hq, d] bf16
    const int32_t* splits;     // 4 per split kv-tile
    const float* part;
    uint16_t* dk;
    uint16_t* dv;
    int32_t N, hq, hkv, d, n_splits;
};

// Launchers return cudaSuccess or the launch error.
// nstream q-heads per CTA; per_sm = 2 (only with nstream = 1): the two-CTAs-per-SM shape
cudaError_t launch_fwd(int d, int nstream, int per_sm, const CUtensorMap* tq, const CUtensorMap* tk,
                       const CUtensorMap* tv, const CUtensorMap* to, const FwdParams& p, int grid,
                       cudaStream_t stream);
cudaError_t launch_bwd_pre(const BwdPreParams& p, cudaStream_t stream);
cudaError_t launch_bwd(int d, const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                       const CUtensorMap* tdo, const CUtensorMap* tdq, const BwdParams& p, int grid,
                       cudaStream_t stream);
cudaError_t launch_bwd_fs(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv, const CUtensorMap* tdo,
                          const CUtensorMap* tdq, const BwdParams& p, int grid, cudaStream_t stream);
cudaError_t launch_bwd_post(const BwdPostParams& p, cudaStream_t stream);
// a bounded wait that runs out on purpose (site 99)
void launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t stream);

}  // namespace treeattn
