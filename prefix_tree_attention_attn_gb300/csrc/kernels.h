// Kernel parameter blocks and launch entry points (internal to libtreeattn).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

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
    int32_t kv_major;          // CTA order: 1 = kv-head group, q-tile, head slice; 0 = q-tile, head slice
    int32_t T;                 // q-tiles (= kv-tiles)          } sizes of the tables,
    int64_t n_ent;             // entries of qt_ent             } for the debug checks
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
    const int32_t* chunk_ptr;  // [n_chunks+1] items of each q-range chunk (head-major order only)
    int32_t n_chunks;
    int32_t head_major;        // CTA order: 0 = item-major (kv-heads of an item side by side),
                               // 1 = within each chunk, every item of kv-head 0, then kv-head 1, ...
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
    int32_t T, n_items;        // q-tiles, work items            } sizes of the tables,
    int64_t n_slots;           // partial dK/dV slots            } for the debug checks
};

struct BwdPostParams {
    const float* dq_acc;       // [N, hq, d]
    uint16_t* dq;              // [N, hq, d] bf16
    const int32_t* splits;     // 4 per split kv-tile
    const float* part;
    uint16_t* dk;
    uint16_t* dv;
    int32_t N, hq, hkv, d, n_splits;
    int32_t T;                 // kv-tiles                 } for the debug checks
    int64_t n_slots;           // partial dK/dV slots      }
    int* status;               // device status word (debug checks)
};

// The (work item, kv-head) of backward CTA b.  Item-major: b = item * hkv +
// kv-head.  Head-major: the CTAs of chunk k occupy [ptr[k] * hkv, ptr[k+1] *
// hkv), kv-head by kv-head, so the CTAs that run at the same time add into the
// dQ rows of one kv-head group only (fewer distinct rows live in L2 at once).
__device__ __forceinline__ void bwd_cta_work(const BwdParams& p, int b, int& item, int& hk) {
    if (!p.head_major) {
        item = b / p.hkv;
        hk = b % p.hkv;
        if (!ta_ok(p.status, 200, item, 0, p.n_items)) item = -1;
        return;
    }
    const int i = b / p.hkv;   // chunk_ptr[k] <= i < chunk_ptr[k+1] for b's chunk k
    if (!ta_ok(p.status, 200, i, 0, p.n_items)) {   // never in a well-formed launch
        item = -1;
        hk = 0;
        return;
    }
    int lo = 0, hi = p.n_chunks - 1;
    while (lo < hi) {           // last k with chunk_ptr[k] <= i
        const int mid = (lo + hi + 1) >> 1;
        if (p.chunk_ptr[mid] <= i) lo = mid;
        else hi = mid - 1;
    }
    const int base = p.chunk_ptr[lo], n = p.chunk_ptr[lo + 1] - base;
    const int r = b - base * p.hkv;
    hk = r / n;
    item = base + r % n;
}

// Launch with programmatic stream serialization (see grid_dep_wait in ptx.cuh):
// the kernel may begin while the previous kernel on the stream finishes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

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
// a debug bounds check that fails on purpose (site 98; *out is written only
// when the check passes, i.e. in builds without the checks)
void launch_bounds_selftest(int* status, int* out, cudaStream_t stream);

}  // namespace treeattn
