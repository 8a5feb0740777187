// C ABI of libtreeattn (see include/tree_attn.h): argument checks, the plan's
// device copy, TMA tensor maps, and kernel launches.  No CPU fallback exists:
// without a usable device every compute call returns an error.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "kernels.h"
#include "plan.h"

namespace treeattn {

// Device status word written by the kernels' bounded waits and, in debug
// builds, their bounds checks (0 = fine).
__device__ int g_device_status = 0;
// Output word of the bounds self-test kernel.
__device__ int g_selftest_word = 0;

namespace {

constexpr int kBlock = 128;
// mean kv-tiles per q-tile up to which the forward runs one q-head per CTA, two CTAs per SM
constexpr int kFwdShortList = 24;
// K/V bytes one q-tile streams over every kv-head above which the forward runs
// its CTAs kv-head group by kv-head group (half of the 129 MB L2)
constexpr double kFwdKvMajorBytes = 64.0 * 1024 * 1024;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---- driver entry point for tensor-map encoding (no link-time libcuda) ------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// [rows, heads, d] bf16 (or fp32), boxes of 128 bytes of d x 1 head x 128 rows,
// 128-byte swizzle.
int make_tmap(CUtensorMap* m, const void* base, int64_t rows, int heads, int d, bool fp32 = false,
              int box_rows = kBlock) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return TREE_ATTN_ERR_CUDA;
    const cuuint64_t es = fp32 ? 4 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)d * es, (cuuint64_t)heads * d * es};
    cuuint32_t box[3] = {(cuuint32_t)(128 / es), 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                     const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? TREE_ATTN_OK : TREE_ATTN_ERR_CUDA;
}

// Backward tensor-core pass: the full-step kernel for head_dim 128 (every MMA
// at N = 128), the general kernel for head_dim 64.
int launch_main(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                const CUtensorMap& tdq, const BwdParams& p, int grid, cudaStream_t s) {
    const cudaError_t e = d == 128 ? launch_bwd_fs(&tq, &tk, &tv, &tdo, &tdq, p, grid, s)
                                   : launch_bwd(d, &tq, &tk, &tv, &tdo, &tdq, p, grid, s);
    return e == cudaSuccess ? TREE_ATTN_OK : TREE_ATTN_ERR_CUDA;
}

}  // namespace

int make_tensor_map(CUtensorMap* m, const void* base, int64_t rows, int heads, int d) {
    return make_tmap(m, base, rows, heads, d);
}

int current_device(int* dev) {
    if (cudaGetDevice(dev) != cudaSuccess) return TREE_ATTN_ERR_NO_DEVICE;
    if (*dev < 0 || *dev >= kMaxDevices) return TREE_ATTN_ERR_NO_DEVICE;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev);
    if (major != 10 || minor != 3) return TREE_ATTN_ERR_NO_DEVICE;
    return TREE_ATTN_OK;
}

namespace {

// Upload (once per device) the tables the kernels read.
int ensure_device(tree_attn_plan_s* P, DevicePlan** out) {
    int dev;
    int st = current_device(&dev);
    if (st) return st;
    std::lock_guard<std::mutex> lk(P->mu);
    DevicePlan& D = P->dev[dev];
    if (D.ready) {
        *out = &D;
        return TREE_ATTN_OK;
    }
    const int64_t T = P->T;
    const int64_t n_ent = (int64_t)P->qt_kv.size();
    const int64_t n_items = (int64_t)P->bwd_items.size() / 4;
    const int64_t n_splits = (int64_t)P->splits.size() / 4;
    // one int32 buffer: subend | qt_ptr | qt_ent | fwd_order | kv_minsub | items | splits | chunk_ptr
    const int64_t sizes[8] = {T * kBlock, T + 1, n_ent, T, T, 4 * n_items, 4 * std::max<int64_t>(n_splits, 1),
                              (int64_t)P->chunk_ptr.size()};
    int64_t offs[8], total = 0;
    for (int k = 0; k < 8; ++k) {
        offs[k] = total;
        total += (sizes[k] + 63) / 64 * 64;   // 256-byte aligned sections
    }
    std::vector<int32_t> h(total, 0);
    std::copy(P->subend.begin(), P->subend.end(), h.begin() + offs[0]);
    std::copy(P->qt_ptr.begin(), P->qt_ptr.end(), h.begin() + offs[1]);
    for (int64_t e = 0; e < n_ent; ++e) {
        const int32_t c = P->qt_kv[e];
        // a kv-tile reaching past N is masked per element whatever its class
        const bool tail = (int64_t)(c + 1) * kBlock > P->N;
        const bool partial = P->qt_cls[e] == TREE_ATTN_TILE_PARTIAL || tail;
        h[offs[2] + e] = c * 2 + (partial ? 1 : 0);
    }
    std::copy(P->fwd_order.begin(), P->fwd_order.end(), h.begin() + offs[3]);
    std::copy(P->kv_minsub.begin(), P->kv_minsub.end(), h.begin() + offs[4]);
    std::copy(P->bwd_items.begin(), P->bwd_items.end(), h.begin() + offs[5]);
    std::copy(P->splits.begin(), P->splits.end(), h.begin() + offs[6]);
    std::copy(P->chunk_ptr.begin(), P->chunk_ptr.end(), h.begin() + offs[7]);
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
    D.base = buf;
    D.subend = b + offs[0];
    D.qt_ptr = b + offs[1];
    D.qt_ent = b + offs[2];
    D.fwd_order = b + offs[3];
    D.kv_minsub = b + offs[4];
    D.bwd_items = b + offs[5];
    D.splits = b + offs[6];
    D.chunk_ptr = b + offs[7];
    D.ready = true;
    *out = &D;
    return TREE_ATTN_OK;
}

// Address of the status word on the current device (looked up once per device).
int status_ptr(int dev, int** out) {
    static int* ptrs[kMaxDevices] = {};
    static std::mutex mu;
    std::lock_guard<std::mutex> lk(mu);
    if (!ptrs[dev]) {
        void* a = nullptr;
        if (cudaGetSymbolAddress(&a, g_device_status) != cudaSuccess) return TREE_ATTN_ERR_CUDA;
        ptrs[dev] = static_cast<int*>(a);
    }
    *out = ptrs[dev];
    return TREE_ATTN_OK;
}

int check_heads(const tree_attn_plan_s* P, int hq, int hkv, int d) {
    if (hq <= 0 || hkv <= 0 || hq % hkv != 0) return TREE_ATTN_ERR_UNSUPPORTED;
    if (d != 64 && d != 128) return TREE_ATTN_ERR_UNSUPPORTED;
    if (P->block != kBlock) return TREE_ATTN_ERR_UNSUPPORTED;
    if ((int64_t)P->N * hq * d > ((int64_t)1 << 40)) return TREE_ATTN_ERR_TOO_LARGE;
    // grid dimension limit of the forward launch
    if ((int64_t)P->T * hq > INT32_MAX) return TREE_ATTN_ERR_TOO_LARGE;
    return TREE_ATTN_OK;
}

struct WsLayout {
    size_t dq_acc, delta, lse2, part, total;
};

WsLayout bwd_layout(const tree_attn_plan_s* P, int hq, int hkv, int d) {
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t Npad = (size_t)P->T * kBlock;
    WsLayout w;
    w.dq_acc = 0;
    w.delta = w.dq_acc + up((size_t)P->N * hq * d * 4);
    w.lse2 = w.delta + up(Npad * hq * 4);
    w.part = w.lse2 + up(Npad * hq * 4);
    w.total = w.part + up((size_t)P->n_slots * hkv * 2 * kBlock * d * 4);
    return w;
}

// Backward CTA order.  Item-major spreads the CTAs running at one time over
// every kv-head's dQ rows (and Q / dO tiles) of the current chunk; head-major
// runs one kv-head group at a time.  Measured backward main pass: long-context
// root with 4 branches at 64 q-heads, chunk 64 (268 MB of fp32 dQ rows per
// chunk): 108.8 ms head-major vs 115.2 item-major (the full long context:
// 1,288 vs 1,326 ms at chunk 48); agentic tree, chunk 64 (134 MB): 11.32 vs
// 11.23 ms; GRPO star, chunk 48 (100 MB): 0.956 vs 0.663 ms.  So head-major
// above 192 MB of rows per chunk.
constexpr size_t kHeadMajorRowBytes = 192ull << 20;

void set_cta_order(BwdParams& p, const tree_attn_plan_s* P, const int32_t* chunk_ptr, int hq, int d) {
    p.chunk_ptr = chunk_ptr;
    p.n_chunks = (int32_t)P->chunk_ptr.size() - 1;
    const size_t rows = (size_t)P->chunk * kBlock * hq * d * 4;
    const bool head_major = P->cta_order == 0 ? rows > kHeadMajorRowBytes : P->cta_order == 2;
    p.head_major = (head_major && p.n_chunks > 0) ? 1 : 0;
}

}  // namespace

int get_status_ptr(int dev, int** out) { return status_ptr(dev, out); }

}  // namespace treeattn

using namespace treeattn;

extern "C" {

int tree_attn_plan(const int32_t* parent, const int32_t* seg_len, int32_t n_nodes, const tree_attn_plan_opts_t* opts,
                   tree_attn_plan_t* out) {
    if (!out) return TREE_ATTN_ERR_INVALID_ARG;
    *out = nullptr;
    tree_attn_plan_s* P = nullptr;
    int st = build_plan(parent, seg_len, n_nodes, opts, &P);
    if (st) return st;
    *out = P;
    return TREE_ATTN_OK;
}

int tree_attn_plan_info(tree_attn_plan_t P, tree_attn_plan_info_t* info) {
    if (!P || !info) return TREE_ATTN_ERR_INVALID_ARG;
    info->n_tokens = P->N;
    info->n_nodes = P->n_nodes;
    info->block = P->block;
    info->n_qtiles = P->T;
    info->n_bwd_items = (int32_t)(P->bwd_items.size() / 4);
    info->n_pairs = P->pairs;
    info->n_intervals = (int64_t)P->qi_lo.size();
    info->n_tile_entries = (int64_t)P->qt_kv.size();
    info->n_full_tiles = P->n_full;
    info->n_split_kv_tiles = (int32_t)(P->splits.size() / 4);
    info->bwd_chunk_qtiles = P->chunk;
    info->n_partial_slots = P->n_slots;
    return TREE_ATTN_OK;
}

int tree_attn_plan_export(tree_attn_plan_t P, const tree_attn_plan_arrays_t* d) {
    if (!P || !d) return TREE_ATTN_ERR_INVALID_ARG;
    auto cp = [](int32_t* dst, const std::vector<int32_t>& v) {
        if (dst && !v.empty()) std::memcpy(dst, v.data(), v.size() * sizeof(int32_t));
    };
    cp(d->node_order, P->node_order);
    cp(d->node_off, P->node_off);
    cp(d->subend, P->subend);
    cp(d->qi_ptr, P->qi_ptr);
    cp(d->qi_lo, P->qi_lo);
    cp(d->qi_hi, P->qi_hi);
    cp(d->qt_ptr, P->qt_ptr);
    cp(d->qt_kv, P->qt_kv);
    if (d->qt_cls && !P->qt_cls.empty()) std::memcpy(d->qt_cls, P->qt_cls.data(), P->qt_cls.size());
    cp(d->kv_qlo, P->kv_qlo);
    cp(d->kv_qhi, P->kv_qhi);
    cp(d->fwd_order, P->fwd_order);
    cp(d->bwd_items, P->bwd_items);
    return TREE_ATTN_OK;
}

int tree_attn_plan_upload(tree_attn_plan_t P) {
    if (!P) return TREE_ATTN_ERR_INVALID_ARG;
    DevicePlan* D = nullptr;
    return ensure_device(P, &D);
}

int tree_attn_workspace_size(tree_attn_plan_t P, int32_t hq, int32_t hkv, int32_t d, size_t* fwd_bytes,
                             size_t* bwd_bytes) {
    if (!P) return TREE_ATTN_ERR_INVALID_ARG;
    int st = check_heads(P, hq, hkv, d);
    if (st) return st;
    if (fwd_bytes) *fwd_bytes = 0;
    if (bwd_bytes) *bwd_bytes = bwd_layout(P, hq, hkv, d).total;
    return TREE_ATTN_OK;
}

int tree_attn_fwd(tree_attn_plan_t P, const void* q, const void* k, const void* v, void* o, float* lse, int32_t hq,
                  int32_t hkv, int32_t d, float softmax_scale, void* workspace, size_t ws_bytes, void* stream) {
    (void)workspace;
    (void)ws_bytes;
    if (!P || !q || !k || !v || !o || !lse) return TREE_ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(softmax_scale) || !(softmax_scale > 0.f)) return TREE_ATTN_ERR_INVALID_ARG;
    int st = check_heads(P, hq, hkv, d);
    if (st) return st;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return TREE_ATTN_ERR_ALIGNMENT;
    DevicePlan* D = nullptr;
    st = ensure_device(P, &D);
    if (st) return st;
    CUtensorMap tq, tk, tv, to;
    if ((st = make_tmap(&tq, q, P->N, hq, d)) || (st = make_tmap(&tk, k, P->N, hkv, d)) ||
        (st = make_tmap(&tv, v, P->N, hkv, d)) || (st = make_tmap(&to, o, P->N, hq, d)))
        return st;
    const int group = hq / hkv;
    // Short kv-tile lists (at most 24 per q-tile on average): one q-head per CTA,
    // two CTAs per SM, so CTA prologues and epilogues overlap other CTAs' tiles.
    // Longer lists: two q-heads per CTA share every K/V tile (even group size).
    const bool short_lists = (int64_t)P->qt_kv.size() <= kFwdShortList * (int64_t)P->T;
    const int ns = (!short_lists && group % 2 == 0) ? 2 : 1;
    const int per_sm = short_lists ? 2 : 1;
    // The K and V one q-tile's CTAs stream, over every kv-head: above half of L2
    // (64 MB), take the CTAs kv-head group by kv-head group.  Measured on the long
    // shared context (149 MB): forward 425 -> 413 ms, DRAM reads 530 -> 64 GB; on
    // the short-list trees the q-tile-major order keeps the longest lists first
    // across all heads and is 5-7 % faster.
    const double kv_stream = (double)P->qt_kv.size() / P->T * 128.0 * hkv * d * 4.0;
    const int kv_major = kv_stream > kFwdKvMajorBytes ? 1 : 0;
    FwdParams p;
    p.qt_ptr = D->qt_ptr;
    p.qt_ent = D->qt_ent;
    p.fwd_order = D->fwd_order;
    p.subend = D->subend;
    p.kv_minsub = D->kv_minsub;
    p.lse = lse;
    p.N = (int32_t)P->N;
    p.hq = hq;
    p.group = group;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.kv_major = kv_major;
    p.T = P->T;
    p.n_ent = (int64_t)P->qt_kv.size();
    int dev = 0;
    cudaGetDevice(&dev);
    if ((st = status_ptr(dev, &p.status))) return st;
    const int grid = P->T * (hq / ns);
    cudaError_t e = launch_fwd(d, ns, per_sm, &tq, &tk, &tv, &to, p, grid, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TREE_ATTN_OK : TREE_ATTN_ERR_CUDA;
}

int tree_attn_bwd(tree_attn_plan_t P, const void* q, const void* k, const void* v, const void* o, const float* lse,
                  const void* dout, void* dq, void* dk, void* dv, int32_t hq, int32_t hkv, int32_t d,
                  float softmax_scale, void* workspace, size_t ws_bytes, void* stream) {
    return tree_attn_bwd_stages(P, q, k, v, o, lse, dout, dq, dk, dv, hq, hkv, d, softmax_scale, workspace, ws_bytes,
                                stream, TREE_ATTN_BWD_PRE | TREE_ATTN_BWD_MAIN | TREE_ATTN_BWD_POST);
}

int tree_attn_bwd_stages(tree_attn_plan_t P, const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dout, void* dq, void* dk, void* dv, int32_t hq, int32_t hkv,
                         int32_t d, float softmax_scale, void* workspace, size_t ws_bytes, void* stream,
                         int32_t stages) {
    if (stages <= 0 || stages > 7) return TREE_ATTN_ERR_INVALID_ARG;
    if (!P || !q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return TREE_ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(softmax_scale) || !(softmax_scale > 0.f)) return TREE_ATTN_ERR_INVALID_ARG;
    int st = check_heads(P, hq, hkv, d);
    if (st) return st;
    for (const void* ptr : {q, k, v, o, (const void*)lse, dout, (const void*)dq, (const void*)dk, (const void*)dv})
        if (!aligned16(ptr)) return TREE_ATTN_ERR_ALIGNMENT;
    const WsLayout w = bwd_layout(P, hq, hkv, d);
    if (!workspace || ws_bytes < w.total) return TREE_ATTN_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return TREE_ATTN_ERR_ALIGNMENT;
    DevicePlan* D = nullptr;
    st = ensure_device(P, &D);
    if (st) return st;
    char* ws = static_cast<char*>(workspace);
    CUtensorMap tq, tk, tv, tdo, tdq;
    if ((st = make_tmap(&tq, q, P->N, hq, d)) || (st = make_tmap(&tk, k, P->N, hkv, d)) ||
        (st = make_tmap(&tv, v, P->N, hkv, d)) || (st = make_tmap(&tdo, dout, P->N, hq, d)) ||
        (st = make_tmap(&tdq, ws + w.dq_acc, P->N, hq, d, true)))
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int32_t Npad = P->T * kBlock;

    BwdPreParams pre;
    pre.o = static_cast<const uint16_t*>(o);
    pre.dout = static_cast<const uint16_t*>(dout);
    pre.lse = lse;
    pre.delta = reinterpret_cast<float*>(ws + w.delta);
    pre.lse2 = reinterpret_cast<float*>(ws + w.lse2);
    pre.dq_acc = reinterpret_cast<float*>(ws + w.dq_acc);
    pre.N = (int32_t)P->N;
    pre.Npad = Npad;
    pre.hq = hq;
    pre.d = d;
    cudaError_t e = cudaSuccess;
    if (stages & TREE_ATTN_BWD_PRE) {
        e = launch_bwd_pre(pre, s);
        if (e != cudaSuccess) return TREE_ATTN_ERR_CUDA;
    }

    BwdParams p;
    p.items = D->bwd_items;
    set_cta_order(p, P, D->chunk_ptr, hq, d);
    p.subend = D->subend;
    p.kv_minsub = D->kv_minsub;
    p.delta = pre.delta;
    p.lse2 = pre.lse2;
    p.dq_acc = pre.dq_acc;
    p.dk = static_cast<uint16_t*>(dk);
    p.dv = static_cast<uint16_t*>(dv);
    p.part = reinterpret_cast<float*>(ws + w.part);
    p.N = (int32_t)P->N;
    p.Npad = Npad;
    p.hq = hq;
    p.hkv = hkv;
    p.group = hq / hkv;
    p.scale = softmax_scale;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.T = P->T;
    p.n_items = (int32_t)(P->bwd_items.size() / 4);
    p.n_slots = P->n_slots;
    int dev = 0;
    cudaGetDevice(&dev);
    if ((st = status_ptr(dev, &p.status))) return st;
    const int64_t n_items = (int64_t)P->bwd_items.size() / 4;
    if (n_items * hkv > INT32_MAX) return TREE_ATTN_ERR_TOO_LARGE;
    if (stages & TREE_ATTN_BWD_MAIN) {
        if ((st = launch_main(d, tq, tk, tv, tdo, tdq, p, (int)(n_items * hkv), s)))
            return st;
    }

    BwdPostParams post;
    post.dq_acc = pre.dq_acc;
    post.dq = static_cast<uint16_t*>(dq);
    post.splits = D->splits;
    post.part = p.part;
    post.dk = p.dk;
    post.dv = p.dv;
    post.N = (int32_t)P->N;
    post.hq = hq;
    post.hkv = hkv;
    post.d = d;
    post.n_splits = (int32_t)(P->splits.size() / 4);
    post.T = P->T;
    post.n_slots = P->n_slots;
    post.status = p.status;
    if (stages & TREE_ATTN_BWD_POST) e = launch_bwd_post(post, s);
    return e == cudaSuccess ? TREE_ATTN_OK : TREE_ATTN_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Backward without any allocation: the scratch lives in a fixed device array.
// ---------------------------------------------------------------------------

namespace treeattn {
namespace {

// One shared scratch array per device that loads this library; it holds the
// plan's device tables and the backward workspace of one call at a time.
constexpr size_t kNoAllocScratchBytes = 32u << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device, looked up once
// per device (with that device current); host code must not use the symbol
// itself as a device pointer.
int noalloc_scratch_ptr(int dev, unsigned char** out) {
    static unsigned char* ptrs[kMaxDevices] = {};
    static std::mutex mu;
    std::lock_guard<std::mutex> lk(mu);
    if (!ptrs[dev]) {
        void* a = nullptr;
        if (cudaGetSymbolAddress(&a, g_noalloc_scratch) != cudaSuccess) return TREE_ATTN_ERR_CUDA;
        ptrs[dev] = static_cast<unsigned char*>(a);
    }
    *out = ptrs[dev];
    return TREE_ATTN_OK;
}

}  // namespace
}  // namespace treeattn

extern "C" {

int tree_attn_bwd_noalloc(tree_attn_plan_t P, const void* q, const void* k, const void* v, const void* o,
                          const float* lse, const void* dout, void* dq, void* dk, void* dv, int32_t hq,
                          int32_t hkv, int32_t d, float softmax_scale, void* stream) {
    if (!P || !q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return TREE_ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(softmax_scale) || !(softmax_scale > 0.f)) return TREE_ATTN_ERR_INVALID_ARG;
    int st = check_heads(P, hq, hkv, d);
    if (st) return st;
    for (const void* ptr : {q, k, v, o, (const void*)lse, dout, (const void*)dq, (const void*)dk, (const void*)dv})
        if (!aligned16(ptr)) return TREE_ATTN_ERR_ALIGNMENT;
    int dev = 0;
    if ((st = current_device(&dev))) return st;

    // plan tables (the same layout the uploaded plan uses), then the workspace
    const int64_t T = P->T;
    const int64_t n_ent = (int64_t)P->qt_kv.size();
    const int64_t n_items = (int64_t)P->bwd_items.size() / 4;
    const int64_t n_splits = (int64_t)P->splits.size() / 4;
    const int64_t sizes[6] = {T * kBlock, T, 4 * n_items, 4 * std::max<int64_t>(n_splits, 1),
                              (int64_t)P->chunk_ptr.size(), 0};
    int64_t offs[6], words = 0;
    for (int i = 0; i < 6; ++i) {
        offs[i] = words;
        words += (sizes[i] + 63) / 64 * 64;
    }
    const size_t table_bytes = (size_t)words * sizeof(int32_t);
    const WsLayout w = bwd_layout(P, hq, hkv, d);
    if (table_bytes + w.total > kNoAllocScratchBytes) return TREE_ATTN_ERR_SCRATCH_TOO_SMALL;
    if (n_items * hkv > INT32_MAX) return TREE_ATTN_ERR_TOO_LARGE;

    unsigned char* scratch = nullptr;
    if ((st = noalloc_scratch_ptr(dev, &scratch))) return st;
    int* status = nullptr;
    if ((st = status_ptr(dev, &status))) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    std::vector<int32_t> h((size_t)words, 0);
    std::copy(P->subend.begin(), P->subend.end(), h.begin() + offs[0]);
    std::copy(P->kv_minsub.begin(), P->kv_minsub.end(), h.begin() + offs[1]);
    std::copy(P->bwd_items.begin(), P->bwd_items.end(), h.begin() + offs[2]);
    std::copy(P->splits.begin(), P->splits.end(), h.begin() + offs[3]);
    std::copy(P->chunk_ptr.begin(), P->chunk_ptr.end(), h.begin() + offs[4]);
    // pageable source: the copy is staged before the call returns
    if (cudaMemcpyAsync(scratch, h.data(), table_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return TREE_ATTN_ERR_CUDA;
    const int32_t* tab = reinterpret_cast<const int32_t*>(scratch);
    char* ws = reinterpret_cast<char*>(scratch) + table_bytes;   // 256-byte aligned

    CUtensorMap tq, tk, tv, tdo, tdq;
    if ((st = make_tmap(&tq, q, P->N, hq, d)) || (st = make_tmap(&tk, k, P->N, hkv, d)) ||
        (st = make_tmap(&tv, v, P->N, hkv, d)) || (st = make_tmap(&tdo, dout, P->N, hq, d)) ||
        (st = make_tmap(&tdq, ws + w.dq_acc, P->N, hq, d, true)))
        return st;
    const int32_t Npad = P->T * kBlock;

    BwdPreParams pre;
    pre.o = static_cast<const uint16_t*>(o);
    pre.dout = static_cast<const uint16_t*>(dout);
    pre.lse = lse;
    pre.delta = reinterpret_cast<float*>(ws + w.delta);
    pre.lse2 = reinterpret_cast<float*>(ws + w.lse2);
    pre.dq_acc = reinterpret_cast<float*>(ws + w.dq_acc);   // zeroed by the pre kernel
    pre.N = (int32_t)P->N;
    pre.Npad = Npad;
    pre.hq = hq;
    pre.d = d;
    if (launch_bwd_pre(pre, s) != cudaSuccess) return TREE_ATTN_ERR_CUDA;

    BwdParams p;
    p.items = tab + offs[2];
    set_cta_order(p, P, tab + offs[4], hq, d);
    p.subend = tab + offs[0];
    p.kv_minsub = tab + offs[1];
    p.delta = pre.delta;
    p.lse2 = pre.lse2;
    p.dq_acc = pre.dq_acc;
    p.dk = static_cast<uint16_t*>(dk);
    p.dv = static_cast<uint16_t*>(dv);
    p.part = reinterpret_cast<float*>(ws + w.part);
    p.N = (int32_t)P->N;
    p.Npad = Npad;
    p.hq = hq;
    p.hkv = hkv;
    p.group = hq / hkv;
    p.scale = softmax_scale;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.T = P->T;
    p.n_items = (int32_t)(P->bwd_items.size() / 4);
    p.n_slots = P->n_slots;
    p.status = status;
    if ((st = launch_main(d, tq, tk, tv, tdo, tdq, p, (int)(n_items * hkv), s)))
        return st;

    BwdPostParams post;
    post.dq_acc = pre.dq_acc;
    post.dq = static_cast<uint16_t*>(dq);
    post.splits = tab + offs[3];
    post.part = p.part;
    post.dk = p.dk;
    post.dv = p.dv;
    post.N = (int32_t)P->N;
    post.hq = hq;
    post.hkv = hkv;
    post.d = d;
    post.n_splits = (int32_t)n_splits;
    post.T = P->T;
    post.n_slots = P->n_slots;
    post.status = status;
    return launch_bwd_post(post, s) == cudaSuccess ? TREE_ATTN_OK : TREE_ATTN_ERR_CUDA;
}

size_t tree_attn_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int tree_attn_selftest_wait_timeout(int32_t limit_ms, void* stream) {
    if (limit_ms < 1 || limit_ms > 2000) return TREE_ATTN_ERR_INVALID_ARG;
    int dev;
    int st = current_device(&dev);
    if (st) return st;
    int* status = nullptr;
    if ((st = status_ptr(dev, &status))) return st;
    treeattn::launch_wait_selftest(status, (uint64_t)limit_ms * 1000000ull, static_cast<cudaStream_t>(stream));
    return cudaGetLastError() == cudaSuccess ? TREE_ATTN_OK : TREE_ATTN_ERR_CUDA;
}

int tree_attn_debug_checks(void) { return treeattn::kDebugChecks ? 1 : 0; }

int tree_attn_selftest_bounds(void* stream) {
    if (!treeattn::kDebugChecks) return TREE_ATTN_ERR_UNSUPPORTED;
    int dev;
    int st = current_device(&dev);
    if (st) return st;
    int* status = nullptr;
    if ((st = status_ptr(dev, &status))) return st;
    // the word the kernel would write if its check passed
    int* out = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&out), g_selftest_word) != cudaSuccess) return TREE_ATTN_ERR_CUDA;
    treeattn::launch_bounds_selftest(status, out, static_cast<cudaStream_t>(stream));
    return cudaGetLastError() == cudaSuccess ? TREE_ATTN_OK : TREE_ATTN_ERR_CUDA;
}

int tree_attn_get_device_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return TREE_ATTN_ERR_CUDA;
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return TREE_ATTN_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess) return TREE_ATTN_ERR_CUDA;
    return v;
}

void tree_attn_plan_destroy(tree_attn_plan_t P) {
    if (!P) return;
    int cur = -1;
    bool have = cudaGetDevice(&cur) == cudaSuccess;
    for (int dev = 0; dev < kMaxDevices; ++dev) {
        if (!P->dev[dev].ready && !P->dev[dev].traj_ready && !P->dev[dev].lin_ready) continue;
        if (cudaSetDevice(dev) == cudaSuccess) {
            if (P->dev[dev].ready) cudaFree(P->dev[dev].base);
            if (P->dev[dev].traj_ready) cudaFree(P->dev[dev].traj_base);
            if (P->dev[dev].lin_ready) cudaFree(P->dev[dev].lin_base);
        }
    }
    if (have) cudaSetDevice(cur);
    cudaGetLastError();
    delete P;
}

const char* tree_attn_strerror(int s) {
    switch (s) {
        case TREE_ATTN_OK: return "ok";
        case TREE_ATTN_ERR_INVALID_ARG: return "invalid argument";
        case TREE_ATTN_ERR_INVALID_TREE: return "invalid tree (parent out of range, self-parent, cycle or seg_len <= 0)";
        case TREE_ATTN_ERR_TOO_LARGE: return "problem too large";
        case TREE_ATTN_ERR_UNSUPPORTED: return "unsupported head configuration or block size";
        case TREE_ATTN_ERR_ALIGNMENT: return "pointer not aligned (16 bytes; workspace 256 bytes)";
        case TREE_ATTN_ERR_WORKSPACE: return "workspace missing or too small";
        case TREE_ATTN_ERR_CUDA: return "CUDA runtime or driver error";
        case TREE_ATTN_ERR_NO_DEVICE: return "no usable sm_103 device";
        case TREE_ATTN_ERR_OUT_OF_MEMORY: return "out of memory";
        case TREE_ATTN_ERR_SCRATCH_TOO_SMALL:
            return "problem too large for the fixed scratch of tree_attn_bwd_noalloc "
                   "(see tree_attn_noalloc_scratch_bytes)";
        case TREE_ATTN_ERR_DEVICE_TIMEOUT: return "a bounded device wait ran out";
        case TREE_ATTN_ERR_INVALID_DECAY: return "linear-attention decay outside (0, 1]";
        case TREE_ATTN_ERR_DEVICE_BOUNDS: return "a debug bounds check failed";
        default:
            // status words with a site: code - 1000 * site
            if (s <= -1000 && (-s) % 1000 == -TREE_ATTN_ERR_DEVICE_TIMEOUT) return "a bounded device wait ran out";
            if (s <= -1000 && (-s) % 1000 == -TREE_ATTN_ERR_DEVICE_BOUNDS) return "a debug bounds check failed";
            return "unknown status";
    }
}

}  // extern "C"
