// Loss-boundary calls around the tree attention (include/tree_loss.h):
// trajectory views of a plan, per-token weights folded into a gradient,
// per-trajectory next-token log-probs from compact logits, and subtree
// (segment-level) advantages.
//
// All memory-bound or tiny.  The log-prob path is one pass over the logits
// (row logsumexp: n_tokens x vocab bf16 read once, 16 bytes per load) plus a
// gather of one logit per prediction; the gather needs the (row, target row)
// pair of every trajectory position, uploaded once per plan and device.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "plan.h"
#include "tree_loss.h"

namespace treeattn {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaxAdvNodes = 16384;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ---- y = x * w (per row) -------------------------------------------------
// The tensor as one run of 16-byte vectors: each thread takes kScalePer of
// them, a block's vectors contiguous, all loads issued before the first store.
constexpr int kScalePer = 4;
__global__ void __launch_bounds__(256) scale_rows_kernel(const uint4* __restrict__ x, const float* __restrict__ w,
                                                        uint4* __restrict__ y, int64_t n_vec, int64_t vec_per_row) {
    const int64_t base = (int64_t)blockIdx.x * blockDim.x * kScalePer + threadIdx.x;
    uint4 a[kScalePer];
    float s[kScalePer];
#pragma unroll
    for (int u = 0; u < kScalePer; ++u) {
        const int64_t k = base + (int64_t)u * blockDim.x;
        if (k < n_vec) {
            a[u] = x[k];
            s[u] = w[k / vec_per_row];
        }
    }
#pragma unroll
    for (int u = 0; u < kScalePer; ++u) {
        const int64_t k = base + (int64_t)u * blockDim.x;
        if (k < n_vec) {
            uint4 b;
            b.x = pack2(bf16_lo(a[u].x) * s[u], bf16_hi(a[u].x) * s[u]);
            b.y = pack2(bf16_lo(a[u].y) * s[u], bf16_hi(a[u].y) * s[u]);
            b.z = pack2(bf16_lo(a[u].z) * s[u], bf16_hi(a[u].z) * s[u]);
            b.w = pack2(bf16_lo(a[u].w) * s[u], bf16_hi(a[u].w) * s[u]);
            y[k] = b;
        }
    }
}

// ---- row logsumexp over the vocabulary ------------------------------------
// One CTA per row; each thread keeps a running (max, sum of exp(x - max)) over
// its 8-element vectors, four loads in flight; the block merges the pairs.
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
    const float mm = fmaxf(m, m2);
    if (mm == -INFINITY) return;
    s = s * exp2f((m - mm) * kLog2e) + s2 * exp2f((m2 - mm) * kLog2e);
    m = mm;
}

__device__ __forceinline__ void lse_add8(float& m, float& s, const uint4 v) {
    const float x[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                        bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
    float lm = x[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) lm = fmaxf(lm, x[i]);
    const float mm = fmaxf(m, lm);
    float acc = (m == -INFINITY) ? 0.f : s * exp2f((m - mm) * kLog2e);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc += exp2f((x[i] - mm) * kLog2e);
    m = mm;
    s = acc;
}

__global__ void __launch_bounds__(256) row_lse_kernel(const uint16_t* __restrict__ logits, int64_t vocab,
                                                     float* __restrict__ lse) {
    const int64_t row = blockIdx.x;
    const uint4* r = reinterpret_cast<const uint4*>(logits + row * vocab);
    const int64_t nvec = vocab / 8;
    float m = -INFINITY, s = 0.f;
    int64_t i = threadIdx.x;
    for (; i + 3 * 256 < nvec; i += 4 * 256) {
        const uint4 a = __ldg(r + i), b = __ldg(r + i + 256), c = __ldg(r + i + 512), d = __ldg(r + i + 768);
        lse_add8(m, s, a);
        lse_add8(m, s, b);
        lse_add8(m, s, c);
        lse_add8(m, s, d);
    }
    for (; i < nvec; i += 256) lse_add8(m, s, __ldg(r + i));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
        lse_merge(m, s, m2, s2);
    }
    __shared__ float sm[8], ss[8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        sm[warp] = m;
        ss[warp] = s;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float M = sm[0], S = ss[0];
        for (int k = 1; k < 8; ++k) lse_merge(M, S, sm[k], ss[k]);
        lse[row] = M + log2f(S) * kLn2;
    }
}

__global__ void __launch_bounds__(256) gather_kernel(const int32_t* __restrict__ pred, int64_t n_pred,
                                                    const uint16_t* __restrict__ logits, int64_t vocab,
                                                    const int32_t* __restrict__ tokens, const float* __restrict__ lse,
                                                    float* __restrict__ out) {
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n_pred; k += (int64_t)gridDim.x * blockDim.x) {
        const int32_t r = pred[2 * k], s = pred[2 * k + 1];
        const int32_t y = tokens[s];
        out[k] = (y >= 0 && y < vocab) ? __uint_as_float((uint32_t)logits[(int64_t)r * vocab + y] << 16) - lse[r]
                                       : __int_as_float(0x7fc00000);
    }
}

// ---- subtree advantages -----------------------------------------------------
// nodes: 6 ints per packed node {parent's packed index or -1, leaf range lo,
// hi (leaves in packed order), first token, tokens, node id}; leaf_of: 2 ints
// per packed leaf {packed node index, index in ascending-id leaf order}.
// One CTA: per-node mean / std, then per-leaf aggregation, then per-node sums.
__global__ void __launch_bounds__(1024) adv_kernel(const int32_t* __restrict__ nodes,
                                                  const int32_t* __restrict__ leaf_of, int32_t n, int32_t L,
                                                  const float* __restrict__ reward, int32_t flags, float eps,
                                                  float* __restrict__ leaf_adv, float* __restrict__ node_coef) {
    extern __shared__ float sh[];
    float* mean = sh;             // [n]
    float* sdev = sh + n;         // [n]
    float* adv = sh + 2 * n;      // [L], packed leaf order
    for (int k = threadIdx.x; k < n; k += blockDim.x) {
        const int lo = nodes[6 * k + 1], hi = nodes[6 * k + 2];
        float sum = 0.f;
        for (int m = lo; m < hi; ++m) sum += reward[leaf_of[2 * m + 1]];
        const float mu = sum / (float)(hi - lo);
        float sq = 0.f;
        for (int m = lo; m < hi; ++m) {
            const float d = reward[leaf_of[2 * m + 1]] - mu;
            sq += d * d;
        }
        mean[k] = mu;
        sdev[k] = sqrtf(sq / (float)(hi - lo));
    }
    __syncthreads();
    for (int m = threadIdx.x; m < L; m += blockDim.x) {
        const int i = leaf_of[2 * m + 1];
        const float R = reward[i];
        float num = 0.f, den = 0.f;
        for (int u = leaf_of[2 * m]; u >= 0; u = nodes[6 * u]) {
            const int cnt = nodes[6 * u + 2] - nodes[6 * u + 1];
            if (cnt < 2) continue;
            if ((flags & TREE_ADV_NO_ROOT) && nodes[6 * u] < 0) continue;
            float a = R - mean[u];
            if (flags & TREE_ADV_NORM_STD) a /= sdev[u] + eps;
            const float w = (flags & TREE_ADV_SIZE_WEIGHTED) ? (float)cnt : 1.f;
            num += w * a;
            den += w;
        }
        const float A = den > 0.f ? num / den : 0.f;
        adv[m] = A;
        leaf_adv[i] = A;
    }
    __syncthreads();
    for (int k = threadIdx.x; k < n; k += blockDim.x) {
        float c = 0.f;
        for (int m = nodes[6 * k + 1]; m < nodes[6 * k + 2]; ++m) c += adv[m];
        node_coef[nodes[6 * k + 5]] = c;
    }
}

// token_coef over each node's segment; one CTA per packed node.
__global__ void __launch_bounds__(256) expand_kernel(const int32_t* __restrict__ nodes,
                                                    const float* __restrict__ node_coef, float* __restrict__ token_coef) {
    const int k = blockIdx.x;
    const int off = nodes[6 * k + 3], len = nodes[6 * k + 4];
    const float c = node_coef[nodes[6 * k + 5]];
    for (int i = threadIdx.x; i < len; i += blockDim.x) token_coef[off + i] = c;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host trajectory view (built once per plan).
int ensure_traj_host(tree_attn_plan_s* P) {
    std::lock_guard<std::mutex> lk(P->mu);
    return build_traj(P);
}

// Device trajectory tables of the current device (uploaded once).
int ensure_traj_device(tree_attn_plan_s* P, DevicePlan** out) {
    int dev;
    int st = current_device(&dev);
    if (st) return st;
    std::lock_guard<std::mutex> lk(P->mu);
    st = build_traj(P);
    if (st) return st;
    DevicePlan& D = P->dev[dev];
    if (D.traj_ready) {
        *out = &D;
        return TREE_ATTN_OK;
    }
    const TrajInfo& X = P->traj;
    const int64_t L = (int64_t)X.leaves.size();
    const int64_t n_pred = (int64_t)X.traj_tok.size() - L;
    const int64_t sizes[3] = {2 * std::max<int64_t>(n_pred, 1), (int64_t)X.nodes.size(),
                              std::max<int64_t>((int64_t)X.leaf_of.size(), 1)};
    int64_t offs[3], total = 0;
    for (int k = 0; k < 3; ++k) {
        offs[k] = total;
        total += (sizes[k] + 63) / 64 * 64;
    }
    std::vector<int32_t> h;
    try {
        h.assign(total, 0);
    } catch (const std::bad_alloc&) {
        return TREE_ATTN_ERR_OUT_OF_MEMORY;
    }
    int64_t k = 0;
    for (int64_t i = 0; i < L; ++i)
        for (int64_t p = X.traj_ptr[i]; p + 1 < X.traj_ptr[i + 1]; ++p) {
            h[offs[0] + 2 * k] = X.traj_tok[p];
            h[offs[0] + 2 * k + 1] = X.traj_tok[p + 1];
            ++k;
        }
    std::copy(X.nodes.begin(), X.nodes.end(), h.begin() + offs[1]);
    std::copy(X.leaf_of.begin(), X.leaf_of.end(), h.begin() + offs[2]);
    void* buf = nullptr;
    if (cudaMalloc(&buf, total * sizeof(int32_t)) != cudaSuccess) {
        cudaGetLastError();
        return TREE_ATTN_ERR_OUT_OF_MEMORY;
    }
    if (cudaMemcpy(buf, h.data(), total * sizeof(int32_t), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaFree(buf);
        return TREE_ATTN_ERR_CUDA;
    }
    int32_t* b = static_cast<int32_t*>(buf);
    D.traj_base = buf;
    D.pred = b + offs[0];
    D.nodes = b + offs[1];
    D.leaf_of = b + offs[2];
    D.traj_ready = true;
    *out = &D;
    return TREE_ATTN_OK;
}

int grid_for(int64_t work, int64_t per_block) {
    const int64_t g = (work + per_block - 1) / per_block;
    return (int)std::min<int64_t>(std::max<int64_t>(g, 1), 152 * 32);
}

}  // namespace

}  // namespace treeattn

using namespace treeattn;

extern "C" {

int tree_attn_plan_trajectory_info(tree_attn_plan_t P, int32_t* n_leaves, int64_t* n_expanded) {
    if (!P) return TREE_ATTN_ERR_INVALID_ARG;
    int st = ensure_traj_host(P);
    if (st) return st;
    if (n_leaves) *n_leaves = (int32_t)P->traj.leaves.size();
    if (n_expanded) *n_expanded = (int64_t)P->traj.traj_tok.size();
    return TREE_ATTN_OK;
}

int tree_attn_plan_trajectories(tree_attn_plan_t P, int32_t* leaf_ids, int64_t* traj_ptr, int32_t* traj_tokens) {
    if (!P) return TREE_ATTN_ERR_INVALID_ARG;
    int st = ensure_traj_host(P);
    if (st) return st;
    const TrajInfo& X = P->traj;
    if (leaf_ids) std::copy(X.leaves.begin(), X.leaves.end(), leaf_ids);
    if (traj_ptr) std::copy(X.traj_ptr.begin(), X.traj_ptr.end(), traj_ptr);
    if (traj_tokens) std::copy(X.traj_tok.begin(), X.traj_tok.end(), traj_tokens);
    return TREE_ATTN_OK;
}

int tree_attn_plan_token_info(tree_attn_plan_t P, int32_t* multiplicity, int32_t* position_ids) {
    if (!P) return TREE_ATTN_ERR_INVALID_ARG;
    int st = ensure_traj_host(P);
    if (st) return st;
    if (multiplicity) std::copy(P->traj.mult.begin(), P->traj.mult.end(), multiplicity);
    if (position_ids) std::copy(P->traj.pos_id.begin(), P->traj.pos_id.end(), position_ids);
    return TREE_ATTN_OK;
}

int tree_attn_scale_rows(const void* x, const float* w, void* y, int64_t n_rows, int64_t row_elems, void* stream) {
    if (n_rows < 0 || row_elems <= 0 || row_elems % 8 != 0) return TREE_ATTN_ERR_INVALID_ARG;
    if (n_rows == 0) return TREE_ATTN_OK;
    if (!x || !w || !y) return TREE_ATTN_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y) || (reinterpret_cast<uintptr_t>(w) & 3u)) return TREE_ATTN_ERR_ALIGNMENT;
    int dev;
    int st = current_device(&dev);
    if (st) return st;
    const int64_t vpr = row_elems / 8;
    const int64_t n_vec = n_rows * vpr;
    const int64_t blocks = (n_vec + 256 * kScalePer - 1) / (256 * kScalePer);
    if (blocks > INT32_MAX) return TREE_ATTN_ERR_TOO_LARGE;
    scale_rows_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(x), w, static_cast<uint4*>(y), n_vec, vpr);
    return cudaGetLastError() == cudaSuccess ? TREE_ATTN_OK : TREE_ATTN_ERR_CUDA;
}

int tree_attn_traj_logprobs(tree_attn_plan_t P, const void* logits, int64_t vocab, const int32_t* tokens,
                            float* row_lse, float* logprobs, void* stream) {
    if (!P || !logits || !tokens || !row_lse || vocab <= 0 || vocab % 8 != 0) return TREE_ATTN_ERR_INVALID_ARG;
    if (!aligned16(logits) || !aligned16(tokens) || !aligned16(row_lse)) return TREE_ATTN_ERR_ALIGNMENT;
    if (P->N > INT32_MAX) return TREE_ATTN_ERR_TOO_LARGE;
    DevicePlan* D = nullptr;
    int st = ensure_traj_device(P, &D);
    if (st) return st;
    const int64_t n_pred = (int64_t)P->traj.traj_tok.size() - (int64_t)P->traj.leaves.size();
    if (n_pred > 0 && !logprobs) return TREE_ATTN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    row_lse_kernel<<<(unsigned)P->N, 256, 0, s>>>(static_cast<const uint16_t*>(logits), vocab, row_lse);
    if (cudaGetLastError() != cudaSuccess) return TREE_ATTN_ERR_CUDA;
    if (n_pred > 0) {
        gather_kernel<<<grid_for(n_pred, 256), 256, 0, s>>>(D->pred, n_pred, static_cast<const uint16_t*>(logits),
                                                           vocab, tokens, row_lse, logprobs);
        if (cudaGetLastError() != cudaSuccess) return TREE_ATTN_ERR_CUDA;
    }
    return TREE_ATTN_OK;
}

int tree_attn_subtree_advantage(tree_attn_plan_t P, const float* leaf_reward, int32_t flags, float eps,
                                float* leaf_adv, float* node_coef, float* token_coef, void* stream) {
    if (!P || !leaf_reward || !leaf_adv || !node_coef || !token_coef) return TREE_ATTN_ERR_INVALID_ARG;
    if ((flags & ~(TREE_ADV_NORM_STD | TREE_ADV_SIZE_WEIGHTED | TREE_ADV_NO_ROOT)) || !(eps >= 0.f))
        return TREE_ATTN_ERR_INVALID_ARG;
    if (P->n_nodes > kMaxAdvNodes) return TREE_ATTN_ERR_TOO_LARGE;
    for (const void* p : {(const void*)leaf_reward, (const void*)leaf_adv, (const void*)node_coef,
                          (const void*)token_coef})
        if (reinterpret_cast<uintptr_t>(p) & 3u) return TREE_ATTN_ERR_ALIGNMENT;
    DevicePlan* D = nullptr;
    int st = ensure_traj_device(P, &D);
    if (st) return st;
    const int32_t n = P->n_nodes, L = (int32_t)P->traj.leaves.size();
    const size_t shm = (size_t)(2 * n + L) * sizeof(float);
    if (shm > 48 * 1024 &&
        cudaFuncSetAttribute(adv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)shm) != cudaSuccess)
        return TREE_ATTN_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    adv_kernel<<<1, 1024, shm, s>>>(D->nodes, D->leaf_of, n, L, leaf_reward, flags, eps, leaf_adv, node_coef);
    if (cudaGetLastError() != cudaSuccess) return TREE_ATTN_ERR_CUDA;
    expand_kernel<<<n, 256, 0, s>>>(D->nodes, node_coef, token_coef);
    return cudaGetLastError() == cudaSuccess ? TREE_ATTN_OK : TREE_ATTN_ERR_CUDA;
}

}  // extern "C"
