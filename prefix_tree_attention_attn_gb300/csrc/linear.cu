// Linear attention over a packed rollout tree, chunk by chunk, with the
// recurrent state handed from every node to its children
// (include/tree_linear.h).
//
// Forward, three steps per call:
//   lin_delta_kernel  per (chunk, kv-head): dS = K^T diag(gamma^(L-1-m)) V on
//                     the tensor core (M = 128 key features, N = 128 value
//                     features, K = the chunk's tokens), read out of TMEM to
//                     an fp32 workspace;
//   the scan          the entering state of each chunk
//                     S_in = gamma^L S_in(prev) + dS(prev) in fp32, a node's
//                     first chunk starting from its parent's exit state -- the
//                     branch-point handoff; S_in leaves as bf16, the operand
//                     precision of the next kernel.  lin_scan_depth_kernel
//                     runs one launch per tree depth (each node of that depth,
//                     4 state entries per thread); trees deeper than
//                     kMaxScanDepths take lin_scan_kernel, one walk over every
//                     chunk in packed order per state entry;
//   lin_out_kernel    persistent, per (chunk, kv-head) and the group's q-heads
//                     in turn: S = Q K^T, then P = S o decay mask and the
//                     query rows scaled by scale * gamma^(m+1) (registers,
//                     written back over S as packed bf16), O = P V + (f Q) S_in
//                     in one accumulation (S_in TMA-loaded like a value
//                     tile); O out as bf16.
// The backward (below) reuses these for dQ and adds three more for dK, dV.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <vector>

#include "kernels.h"
#include "plan.h"
#include "ptx.cuh"
#include "tree_linear.h"

namespace treeattn {

namespace {

constexpr int kChunk = 128;
constexpr int kD = 128;
constexpr int kTile = kChunk * kD * 2;   // 32 KB bf16 tile

__device__ __forceinline__ void bulk_store_s2g(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}

// A 128 x 128 fp32 TMEM accumulator (TMEM lane = row) -> 128 contiguous fp32
// rows of 512 bytes at `dst`, by warps 0-3 (32 rows each).  Each thread stages
// its row in shared memory at a 528-byte row stride (16 bytes more than a row,
// so the 32 rows of a warp fall on different bank groups); lane 0 of each warp
// then copies the warp's rows out with one bulk copy per row, so rows leave as
// whole lines rather than as one 16-byte piece of 32 rows per store.
constexpr uint32_t kRowStage = 528;
constexpr int kRowStageBytes = 128 * kRowStage;

__device__ __forceinline__ void store_rows_f32(uint32_t tmem_rows, uint32_t stage, float* __restrict__ dst, int warp,
                                               int lane) {
    const uint32_t my = stage + (uint32_t)(warp * 32 + lane) * kRowStage;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
        float v[32];
        tmem_ld32(tmem_rows + cc * 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 8; ++q)
            st_shared_v4(my + cc * 128 + q * 16, __float_as_uint(v[4 * q]), __float_as_uint(v[4 * q + 1]),
                         __float_as_uint(v[4 * q + 2]), __float_as_uint(v[4 * q + 3]));
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        for (int rr = 0; rr < 32; ++rr) {
            const int row = warp * 32 + rr;
            bulk_store_s2g(dst + (size_t)row * 128, stage + (uint32_t)row * kRowStage, 512);
        }
        bulk_commit();
        bulk_wait_all();
    }
    __syncwarp();
}

// The scans hand each chunk's d x d state to the tensor-core kernels as bf16,
// laid out [chunk][row][kv-head][col] (row = key feature), i.e. as a token-major
// [chunks * 128, hkv, 128] tensor that the kernels TMA-load like a value tile.
__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
    const __nv_bfloat16 h = __float2bfloat16_rn(f);   // round to nearest even, as pack_bf16x2
    return *reinterpret_cast<const uint16_t*>(&h);
}

__device__ __forceinline__ size_t state16_index(int chunk, int e, int g, int hkv) {
    return (((size_t)chunk * kChunk + (e >> 7)) * hkv + g) * kD + (e & 127);
}

// ---- dS per (chunk, kv-head) -------------------------------------------------
// warps 0-3: lane r = token row r (scaling V) and key feature r (read-out);
// warp 4: TMEM owner, lane 0 issues the loads and the MMA.
constexpr int kDeltaSmem = 1024 + kRowStageBytes;   // K, V; then the fp32 staging rows over them

__global__ void __launch_bounds__(160, 1)
    lin_delta_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const int32_t* __restrict__ chunks, const float* __restrict__ decay, int hkv,
                     float* __restrict__ ds, int* status) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    if (sb & 1023u) {
        if (threadIdx.x == 0) report_status(status, -5);
        return;
    }
    const int chunk = blockIdx.x / hkv, g = blockIdx.x % hkv;
    const int off = chunks[4 * chunk], L = chunks[4 * chunk + 1];
    // a decay outside (0, 1] has no meaning here (its log2 would be NaN or
    // -inf); say so in the status word, once per kv-head (the call's outputs
    // are then undefined)
    if (chunk == 0 && threadIdx.x == 0 && !(decay[g] > 0.f && decay[g] <= 1.f))
        report_status(status, TREE_ATTN_ERR_INVALID_DECAY);
    const uint32_t b_full = sb, b_done = sb + 8, holder = sb + 16;
    const uint32_t ka = sb + 1024, va = ka + kTile;
    if (threadIdx.x == 0) {
        mbar_init(b_full, 1);
        mbar_init(b_done, 1);
        fence_mbar_init();
    }
    if (warp == 4) tmem_alloc(holder, 128);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + 16);
    if (threadIdx.x == 128) {
        mbar_expect_tx(b_full, 2 * kTile);
        for (int blk = 0; blk < 2; ++blk) {
            tma_load_3d(ka + blk * 16384, &tm_k, blk * 64, g, off, b_full);
            tma_load_3d(va + blk * 16384, &tm_v, blk * 64, g, off, b_full);
        }
    }
    bool ok = mbar_wait(b_full, 0, status, 81);
    if (warp < 4 && ok) {
        // V row r times gamma^(L-1-r) (0 past the chunk): the row's 128 bytes in
        // each 64-feature block stay inside that row under the 128-byte swizzle
        const int r = threadIdx.x;
        const float lg = log2f(decay[g]);
        const float w = r < L ? exp2f((float)(L - 1 - r) * lg) : 0.f;
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
            uint4* row = reinterpret_cast<uint4*>(smem + 1024 + kTile + blk * 16384 + r * 128);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                // the row's 16-byte pieces in an order rotated by the row, so that the
                // 32 rows of a warp spread over every bank group instead of one
                const int cr = (c + r) & 7;
                uint4 x = row[cr];
                uint32_t* u = reinterpret_cast<uint32_t*>(&x);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    u[e] = pack_bf16x2(__uint_as_float(u[e] << 16) * w, __uint_as_float(u[e] & 0xffff0000u) * w);
                row[cr] = x;
            }
        }
        fence_proxy_async_smem();
    }
    ok = __syncthreads_and(ok);
    if (ok && threadIdx.x == 128) {
        tc_fence_after();
        constexpr uint32_t ID = idesc_bf16(128, 128, true, true);   // K^T (MN-major) x V_w (MN-major)
#pragma unroll
        for (int k = 0; k < kChunk / 16; ++k)
            mma_bf16_ss(tmem, sdesc_sw128(ka + k * 2048, 16384, 1024), sdesc_sw128(va + k * 2048, 16384, 1024), ID,
                        k > 0);
        mma_commit(b_done);
    }
    if (warp < 4) {
        if (ok) ok = mbar_wait(b_done, 0, status, 82);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            tc_fence_after();
            // row = key feature; K and V have been read by the product, so their
            // tiles hold the staging rows
            store_rows_f32(tmem + ((uint32_t)(warp << 5) << 16), sb + 1024, ds + ((size_t)chunk * hkv + g) * kD * kD,
                           warp, threadIdx.x & 31);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}

// ---- entering states, chunk by chunk in packed order -------------------------
// One thread per (state entry, kv-head) walks every chunk of the tree in packed
// order; a node's chunks are consecutive, and a node's first chunk starts from
// its parent's exit state (0 at a root), which is final by then because the
// parent precedes the node.  With one thread per entry there are few threads
// per SM, so each keeps kScanBatch increments in flight (loaded before the
// recurrence uses the first of them); chunk lengths and node ids, the same for
// every thread, are staged in shared memory a window at a time.
constexpr int kScanBatch = 16;
constexpr int kScanWin = 1024;
constexpr int kMaxScanDepths = 32;   // deeper trees use the one-walk scans (one launch per depth otherwise)

__global__ void __launch_bounds__(256) lin_scan_kernel(const int32_t* __restrict__ lnodes, int n_chunks,
                                                     const int32_t* __restrict__ chunks,
                                                     const float* __restrict__ decay, int hkv,
                                                     const float* __restrict__ ds, uint16_t* __restrict__ s_in16,
                                                     float* __restrict__ s_out) {
    __shared__ int w_len[kScanWin], w_node[kScanWin];
    const int e = blockIdx.x * blockDim.x + threadIdx.x;   // state entry (row * d + col)
    const int g = blockIdx.y;
    const size_t dd = (size_t)kD * kD;
    const float lg = log2f(decay[g]);
    float S = 0.f;
    int cur = -1;   // the node whose chunks are being walked
    for (int w0 = 0; w0 < n_chunks; w0 += kScanWin) {
        const int nw = min(kScanWin, n_chunks - w0);
        __syncthreads();   // the previous window has been read
        for (int t = threadIdx.x; t < nw; t += blockDim.x) {
            w_len[t] = chunks[4 * (w0 + t) + 1];
            w_node[t] = chunks[4 * (w0 + t) + 2];
        }
        __syncthreads();
        for (int c = 0; c < nw; c += kScanBatch) {
            float dsv[kScanBatch];
#pragma unroll
            for (int u = 0; u < kScanBatch; ++u)
                if (c + u < nw) dsv[u] = ds[((size_t)(w0 + c + u) * hkv + g) * dd + e];
#pragma unroll
            for (int u = 0; u < kScanBatch; ++u)
                if (c + u < nw) {
                    const int node = w_node[c + u];
                    if (node != cur) {   // first chunk of a node
                        const int par = lnodes[4 * node];
                        if (cur >= 0) s_out[((size_t)cur * hkv + g) * dd + e] = S;
                        // the node right after its parent continues from S itself
                        if (par != cur) S = par < 0 ? 0.f : s_out[((size_t)par * hkv + g) * dd + e];
                        cur = node;
                    }
                    s_in16[state16_index(w0 + c + u, e, g, hkv)] = float_to_bf16_bits(S);
                    S = exp2f((float)w_len[c + u] * lg) * S + dsv[u];
                }
        }
    }
    if (cur >= 0) s_out[((size_t)cur * hkv + g) * dd + e] = S;
}

// ---- outputs per (chunk, kv-head): the group's q-heads one after another ------
// Persistent: a CTA keeps one kv-head g and walks the chunks j0, j0 + lanes,
// j0 + 2 lanes, ... (grid = lanes x hkv, about one CTA per SM); every
// (chunk, q-head) pair it meets is one "unit" u.  K is loaded once per chunk,
// V and the bf16 copy of S_in together once per chunk, for the G q-heads of the
// group; Q comes through two slots.  TMEM holds two units (buffer b = u & 1):
// S at [256b, 256b + 128), O at [256b + 128, 256b + 256).
// Per unit: S = Q K^T; the element-wise warps turn S into the masked P and
// write, next to it, the query rows scaled by the carried-in weight
// f(m) = scale * gamma^(m+1), both as packed bf16 (P of keys [64 j, 64 j + 64)
// at columns [64 j, 64 j + 32), f Q of features [64 j, 64 j + 64) at
// [64 j + 32, 64 j + 64), over S columns the same threads have read); then one
// accumulation O = P V + (f Q) S_in of 256 K-steps' worth (A from TMEM).  S of
// unit u is issued before the products of unit u - 1 (the tensor core runs
// them in issue order, so P of unit u - 2 in the same buffer has been read),
// and the products of unit u wait only until unit u - 2's output has left.
// warps 0-7: query row m = 32 (w % 4) + lane (the TMEM lanes warp w may
// access), columns [64 (w / 4), 64 (w / 4) + 64) of S and of O -- two warps per
// row, so that each SM sub-partition has two warps of element-wise work.
// warp 8: loads; warp 9: TMEM owner, lane 0 issues the MMAs.  The decay mask
// gamma^(m - m') depends on m - m' alone: its 128 values (and zeros for
// m' > m) are tabulated once per CTA in shared memory.
constexpr int kOutSmem = 2048 + 5 * kTile;   // barriers, mask table, K, V, S_in (bf16), Q x 2
constexpr int kLinWarps = 10;                // 8 element-wise warps, loader, MMA issuer
constexpr int kLinThreads = 32 * kLinWarps;

__global__ void __launch_bounds__(kLinThreads, 1)
    lin_out_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_s,
                   const int32_t* __restrict__ chunks, int n_chunks, int lanes, const float* __restrict__ decay,
                   uint16_t* __restrict__ out, int hq, int hkv, float scale, int* status) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (sb & 1023u) {
        if (threadIdx.x == 0) report_status(status, -5);
        return;
    }
    const int G = hq / hkv;
    const int j0 = blockIdx.x / hkv, g = blockIdx.x % hkv;
    if (j0 >= n_chunks) return;   // uniform: nothing set up yet
    const int n_items = (n_chunks - 1 - j0) / lanes + 1;   // chunks j0 + i lanes < n_chunks
    const int U = n_items * G;                              // units of this CTA
    auto chunk_of = [&](int i) { return j0 + i * lanes; };
    // barriers: K, V with S_in, their free signals, then per buffer b: qfull,
    // qempty (S has read Q), sfull, qread (the element-wise warps have read Q),
    // p, o2, oempty
    auto bar = [&](int i) { return sb + 8u * (uint32_t)i; };
    const uint32_t b_k = bar(0), b_v = bar(1), b_kfree = bar(18), b_vfree = bar(19);
    auto b_qf = [&](int b) { return bar(2 + b); };
    auto b_qe = [&](int b) { return bar(4 + b); };
    auto b_sf = [&](int b) { return bar(6 + b); };
    auto b_qr = [&](int b) { return bar(8 + b); };
    auto b_p = [&](int b) { return bar(10 + b); };
    auto b_o2 = [&](int b) { return bar(12 + b); };
    auto b_oe = [&](int b) { return bar(14 + b); };
    const uint32_t b_drain = bar(16), holder = bar(17);
    const uint32_t ka = sb + 2048, va = ka + kTile, sina = va + kTile, qa0 = sina + kTile;
    // mtab[128 + t] = gamma^t for t = m - m' in [0, 128), 0 for t < 0
    float* mtab = reinterpret_cast<float*>(smem + 1024);
    if (threadIdx.x < 128) {
        mtab[threadIdx.x] = 0.f;
        mtab[128 + threadIdx.x] = exp2f((float)threadIdx.x * log2f(decay[g]));
    }
    if (threadIdx.x == 0) {
        mbar_init(b_k, 1);
        mbar_init(b_v, 1);
        mbar_init(b_kfree, 1);
        mbar_init(b_vfree, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(b_qf(b), 1);
            mbar_init(b_qe(b), 1);
            mbar_init(b_sf(b), 1);
            mbar_init(b_qr(b), 256);
            mbar_init(b_p(b), 256);
            mbar_init(b_o2(b), 1);
            mbar_init(b_oe(b), 256);
        }
        mbar_init(b_drain, 1);
        fence_mbar_init();
    }
    if (warp == 9) tmem_alloc(holder, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + 8 * 17);

    if (warp == 8) {
        if (lane == 0) {
            bool ok = true;
            for (int i = 0; i < n_items && ok; ++i) {
                const int chunk = chunk_of(i), off = chunks[4 * chunk];
                // K: once the previous chunk's last S product has read it
                if (i > 0) ok = mbar_wait(b_kfree, (i - 1) & 1, status, 94);
                if (!ok) break;
                mbar_expect_tx(b_k, kTile);
                for (int blk = 0; blk < 2; ++blk) tma_load_3d(ka + blk * 16384, &tm_k, blk * 64, g, off, b_k);
                for (int n = 0; n < G && ok; ++n) {
                    const int u = i * G + n, b = u & 1, w = u >> 1;
                    if (w > 0) {   // Q slot b: read by unit u - 2's S product and element-wise warps
                        ok = mbar_wait(b_qe(b), (w - 1) & 1, status, 89);
                        if (ok) ok = mbar_wait(b_qr(b), (w - 1) & 1, status, 97);
                    }
                    if (!ok) break;
                    mbar_expect_tx(b_qf(b), kTile);
                    for (int blk = 0; blk < 2; ++blk)
                        tma_load_3d(qa0 + b * kTile + blk * 16384, &tm_q, blk * 64, g * G + n, off, b_qf(b));
                    // V and S_in after the second q-head's Q (the first with one q-head):
                    // the previous chunk's last products, which must have read them, are
                    // issued before this chunk's second S product
                    if (n == (G > 1 ? 1 : 0)) {
                        if (i > 0) ok = mbar_wait(b_vfree, (i - 1) & 1, status, 95);
                        if (!ok) break;
                        mbar_expect_tx(b_v, 2 * kTile);
                        for (int blk = 0; blk < 2; ++blk) {
                            tma_load_3d(va + blk * 16384, &tm_v, blk * 64, g, off, b_v);
                            tma_load_3d(sina + blk * 16384, &tm_s, blk * 64, g, chunk * kChunk, b_v);
                        }
                    }
                }
            }
        }
    } else if (warp == 9) {
        if (lane == 0) {
            constexpr uint32_t ID_S = idesc_bf16(128, 128, false, false);   // Q K^T
            constexpr uint32_t ID_O = idesc_bf16(128, 128, false, true);    // P V, (f Q) S_in
            bool ok = true;
            auto issue_o = [&](int u) {
                const int b = u & 1, w = u >> 1, i = u / G, n = u % G;
                if (w > 0) ok = mbar_wait(b_oe(b), (w - 1) & 1, status, 90);   // unit u - 2's output read
                if (ok && n == 0) ok = mbar_wait(b_v, i & 1, status, 96);      // this chunk's V and S_in
                if (!ok) return;
                tc_fence_after();
                // keys 16k .. 16k + 15 of P packed at 64 (k / 4) + 8 (k % 4); features
                // 16k .. 16k + 15 of f Q 32 columns further
#pragma unroll
                for (int k = 0; k < kChunk / 16; ++k)
                    mma_bf16_ts(tmem + 256 * b + 128, tmem + 256 * b + (k >> 2) * 64 + (k & 3) * 8,
                                sdesc_sw128(va + k * 2048, 16384, 1024), ID_O, k > 0 ? 1u : 0u);
#pragma unroll
                for (int k = 0; k < kD / 16; ++k)
                    mma_bf16_ts(tmem + 256 * b + 128, tmem + 256 * b + 32 + (k >> 2) * 64 + (k & 3) * 8,
                                sdesc_sw128(sina + k * 2048, 16384, 1024), ID_O, 1u);
                mma_commit(b_o2(b));
                if (n == G - 1) mma_commit(b_vfree);   // V and S_in read by the chunk's last products
            };
            for (int u = 0; u < U && ok; ++u) {
                const int b = u & 1, w = u >> 1, i = u / G, n = u % G;
                ok = mbar_wait(b_qf(b), w & 1, status, 91);
                if (ok && n == 0) ok = mbar_wait(b_k, i & 1, status, 83);   // this chunk's K
                if (!ok) break;
                tc_fence_after();
                const uint32_t qa = qa0 + b * kTile;
#pragma unroll
                for (int k = 0; k < kD / 16; ++k) {
                    const uint32_t o = (k >> 2) * 16384 + (k & 3) * 32;
                    mma_bf16_ss(tmem + 256 * b, sdesc_sw128(qa + o, 16, 1024), sdesc_sw128(ka + o, 16, 1024), ID_S,
                                k > 0);
                }
                mma_commit(b_sf(b));
                mma_commit(b_qe(b));                       // Q slot b no longer read by the tensor core
                if (n == G - 1) mma_commit(b_kfree);       // K read by the chunk's last S product
                if (u > 0) {                               // the previous unit's products
                    ok = mbar_wait(b_p((u - 1) & 1), ((u - 1) >> 1) & 1, status, 85);
                    if (!ok) break;
                    issue_o(u - 1);
                }
            }
            if (ok) {
                ok = mbar_wait(b_p((U - 1) & 1), ((U - 1) >> 1) & 1, status, 92);
                if (ok) issue_o(U - 1);
            }
            mma_commit(b_drain);
            mbar_wait(b_drain, 0, status, 93);
        }
        __syncwarp();
    } else {
        const int m = ((warp & 3) << 5) + lane;   // query row
        const int grp = warp >> 2;                 // this warp's 64 columns of S and O, 64 features of Q
        const int col0 = grp * 64;
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) << 5) << 16);
        const float lg = log2f(decay[g]);
        const float fo = scale * exp2f((float)(m + 1) * lg);   // weight of the carried-in part
        const float* wt = mtab + 128 + m;   // wt[-m'] = gamma^(m - m'), 0 past the diagonal
        bool ok = true;
        // Unit u's output is stored after unit u+1's mask, so the products of
        // unit u run while the element-wise warps mask the next unit.
        int prev_off = 0, prev_L = 0, prev_h = 0;
        for (int u = 0; u <= U; ++u) {
            if (u < U) {
                const int b = u & 1, w = u >> 1;
                const uint32_t tS = lane_base + 256 * b;
                if (ok) ok = mbar_wait(b_sf(b), w & 1, status, 86);
                ok = __all_sync(0xffffffffu, ok);
                if (ok) {
                    tc_fence_after();
                    // P[m, m'] = scale * S[m, m'] * gamma^(m - m') for m' <= m (rows m >= L
                    // are never stored, and for m < L every m' <= m lies in the chunk)
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        float v[32];
                        tmem_ld32(tS + col0 + cc * 32, v);
                        tmem_wait_ld();
                        uint32_t pw[16];
#pragma unroll
                        for (int x = 0; x < 16; ++x) {
                            const int c0 = col0 + cc * 32 + 2 * x, c1 = c0 + 1;
                            pw[x] = pack_bf16x2(scale * v[2 * x] * wt[-c0], scale * v[2 * x + 1] * wt[-c1]);
                        }
                        tmem_st16(tS + col0 + cc * 16, pw);
                    }
                    // f(m) q_m over features [col0, col0 + 64), from the 128B-swizzled Q
                    // slot (block grp holds those features, row m at 128 m)
                    const uint8_t* qrow = smem + (qa0 - sb) + b * kTile + grp * 16384 + m * 128;
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        uint32_t qw[16];
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const int ch = h2 * 4 + c;   // 16-byte chunk: features 8 ch .. 8 ch + 7
                            const uint4 x = *reinterpret_cast<const uint4*>(qrow + ((ch ^ (m & 7)) << 4));
                            const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                qw[4 * c + e] = pack_bf16x2(fo * __uint_as_float(xs[e] << 16),
                                                            fo * __uint_as_float(xs[e] & 0xffff0000u));
                        }
                        tmem_st16(tS + col0 + 32 + h2 * 16, qw);
                    }
                    mbar_arrive(b_qr(b));   // Q slot b read (the values are in registers)
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(b_p(b));
                }
            }
            if (u > 0) {   // unit u-1's output
                const int b = (u - 1) & 1, w = (u - 1) >> 1;
                const uint32_t tO = lane_base + 256 * b + 128;
                if (ok) ok = mbar_wait(b_o2(b), w & 1, status, 88);
                ok = __all_sync(0xffffffffu, ok);
                if (ok) {
                    tc_fence_after();
                    uint4* dst = reinterpret_cast<uint4*>(out + ((size_t)(prev_off + m) * hq + prev_h) * kD + col0);
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        float v[32];
                        tmem_ld32(tO + col0 + cc * 32, v);
                        tmem_wait_ld();
                        if (m < prev_L) {
#pragma unroll
                            for (int x = 0; x < 4; ++x) {
                                uint4 y;
                                y.x = pack_bf16x2(v[8 * x], v[8 * x + 1]);
                                y.y = pack_bf16x2(v[8 * x + 2], v[8 * x + 3]);
                                y.z = pack_bf16x2(v[8 * x + 4], v[8 * x + 5]);
                                y.w = pack_bf16x2(v[8 * x + 6], v[8 * x + 7]);
                                dst[cc * 4 + x] = y;
                            }
                        }
                    }
                    tc_fence_before();
                    mbar_arrive(b_oe(b));   // buffer b's O may take the unit after next
                }
            }
            if (u < U) {
                const int chunk = chunk_of(u / G);
                prev_off = chunks[4 * chunk];
                prev_L = chunks[4 * chunk + 1];
                prev_h = g * G + u % G;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

int build_lin(tree_attn_plan_s* P) {
    LinInfo& X = P->lin;
    if (X.ready) return TREE_ATTN_OK;
    try {
        const int32_t n = P->n_nodes;
        std::vector<int32_t> pos_of(n);
        for (int32_t k = 0; k < n; ++k) pos_of[P->node_order[k]] = k;
        X.chunks.clear();
        X.lnodes.assign(4 * (size_t)n, 0);
        int32_t nc = 0;
        for (int32_t k = 0; k < n; ++k) {
            const int32_t u = P->node_order[k], p = P->parent[u];
            const int32_t first = nc;
            for (int32_t o = 0; o < P->seg_len[u]; o += kChunk) {
                X.chunks.insert(X.chunks.end(), {P->node_off[u] + o, std::min(kChunk, P->seg_len[u] - o), k, 0});
                ++nc;
            }
            X.lnodes[4 * (size_t)k] = p < 0 ? -1 : pos_of[p];
            X.lnodes[4 * (size_t)k + 1] = first;
            X.lnodes[4 * (size_t)k + 2] = nc - first;
        }
        // fourth field: 1 for the last child of its parent in packed order (the
        // first one the reverse scan leaves), else 0
        std::vector<int32_t> last_child(n, -1);
        for (int32_t k = 0; k < n; ++k) {
            const int32_t pp = X.lnodes[4 * (size_t)k];
            if (pp >= 0) last_child[pp] = k;   // children in increasing packed position
        }
        for (int32_t k = 0; k < n; ++k)
            if (last_child[k] >= 0) X.lnodes[4 * (size_t)last_child[k] + 3] = 1;
        // children of every node in packed order (CSR), and the nodes grouped by
        // depth (a parent precedes its children in packed order, so its depth is
        // known first); depth-by-depth scans only for trees of at most
        // kMaxScanDepths depths
        X.kids.assign((size_t)n + 1, 0);
        for (int32_t k = 0; k < n; ++k)
            if (X.lnodes[4 * (size_t)k] >= 0) ++X.kids[(size_t)X.lnodes[4 * (size_t)k] + 1];
        for (int32_t k = 0; k < n; ++k) X.kids[(size_t)k + 1] += X.kids[k];
        X.kids.resize((size_t)n + 1 + X.kids[n]);
        {
            std::vector<int32_t> fill(X.kids.begin(), X.kids.begin() + n);
            for (int32_t k = 0; k < n; ++k) {
                const int32_t pp = X.lnodes[4 * (size_t)k];
                if (pp >= 0) X.kids[(size_t)n + 1 + fill[pp]++] = k;
            }
        }
        std::vector<int32_t> depth(n, 0);
        int32_t n_depths = 0;
        for (int32_t k = 0; k < n; ++k) {
            const int32_t pp = X.lnodes[4 * (size_t)k];
            depth[k] = pp < 0 ? 0 : depth[pp] + 1;
            n_depths = std::max(n_depths, depth[k] + 1);
        }
        X.lvl_ptr.clear();
        X.lvl_nodes.clear();
        if (n_depths <= kMaxScanDepths) {
            X.lvl_ptr.assign((size_t)n_depths + 1, 0);
            for (int32_t k = 0; k < n; ++k) ++X.lvl_ptr[(size_t)depth[k] + 1];
            for (int32_t l = 0; l < n_depths; ++l) X.lvl_ptr[(size_t)l + 1] += X.lvl_ptr[l];
            X.lvl_nodes.resize(n);
            std::vector<int32_t> fill(X.lvl_ptr.begin(), X.lvl_ptr.end() - 1);
            for (int32_t k = 0; k < n; ++k) X.lvl_nodes[fill[depth[k]]++] = k;
        }
        X.ready = true;
    } catch (const std::bad_alloc&) {
        return TREE_ATTN_ERR_OUT_OF_MEMORY;
    }
    return TREE_ATTN_OK;
}

int ensure_lin_device(tree_attn_plan_s* P, DevicePlan** out) {
    int dev;
    int st = current_device(&dev);
    if (st) return st;
    std::lock_guard<std::mutex> lk(P->mu);
    if ((st = build_lin(P))) return st;
    DevicePlan& D = P->dev[dev];
    if (!D.lin_ready) {
        const size_t a = (P->lin.chunks.size() + 63) / 64 * 64, b = P->lin.lnodes.size(),
                     c = P->lin.lvl_nodes.size(), k = P->lin.kids.size();
        std::vector<int32_t> h(a + b + c + k, 0);
        std::copy(P->lin.chunks.begin(), P->lin.chunks.end(), h.begin());
        std::copy(P->lin.lnodes.begin(), P->lin.lnodes.end(), h.begin() + a);
        std::copy(P->lin.lvl_nodes.begin(), P->lin.lvl_nodes.end(), h.begin() + a + b);
        std::copy(P->lin.kids.begin(), P->lin.kids.end(), h.begin() + a + b + c);
        void* buf = nullptr;
        if (cudaMalloc(&buf, h.size() * sizeof(int32_t)) != cudaSuccess) {
            cudaGetLastError();
            return TREE_ATTN_ERR_OUT_OF_MEMORY;
        }
        if (cudaMemcpy(buf, h.data(), h.size() * sizeof(int32_t), cudaMemcpyHostToDevice) != cudaSuccess) {
            cudaFree(buf);
            return TREE_ATTN_ERR_CUDA;
        }
        D.lin_base = buf;
        D.chunks = static_cast<int32_t*>(buf);
        D.lnodes = static_cast<int32_t*>(buf) + a;
        D.lvl_nodes = static_cast<int32_t*>(buf) + a + b;
        D.kids = static_cast<int32_t*>(buf) + a + b + c;
        D.lin_ready = true;
    }
    *out = &D;
    return TREE_ATTN_OK;
}

struct LinWs {
    size_t ds, s_in, s_out, total;
};

LinWs lin_layout(const tree_attn_plan_s* P, int32_t hkv) {
    const size_t per = (size_t)hkv * kD * kD * sizeof(float);
    const size_t nc = P->lin.chunks.size() / 4;
    LinWs w;
    w.ds = 0;
    w.s_in = nc * per;
    w.s_out = 2 * nc * per;
    w.total = (2 * nc + (size_t)P->n_nodes) * per;
    return w;
}

// ============================== backward ======================================
// dQ is itself a tree linear attention: scale * sum over the path of
// gamma^(distance) (dO_i . v_j) k_j -- the three forward kernels with
// (q, k, v) = (dO, V, K).  dK and dV need the adjoint of the state, which flows
// the other way, from every node into its parent (summed over the children):
//   F_c      = scale sum_h Q_h^T diag(gamma^(m+1)) dO_h      (lin_bwd_f_kernel)
//   Rsum(c)  = sum over the chunks c' that continue c of R_in(c'),
//   R_in(c)  = F_c + gamma^L Rsum(c)                          (lin_bwd_scan_kernel)
//   dK rows  = gamma^(L-1-m') Rsum v_m'  + sum_h (dA_h^T Q_h)
//   dV rows  = gamma^(L-1-m') Rsum^T k_m' + sum_h (P_h^T dO_h) (lin_bwd_kv_kernel)
// with P_h^T[m', m] = scale (k_m' . q_m) gamma^(m-m') and dA_h^T[m', m] =
// scale (v_m' . dO_m) gamma^(m-m') for m' <= m < L.

// ---- F per (chunk, kv-head), the group's q-heads accumulated in TMEM ----------
// warps 0-3: lane r = token row r (scaling dO) and key feature r (read-out);
// warp 4: TMEM owner, lane 0 loads and issues.
constexpr int kAdjSmem = 1024 + kRowStageBytes;   // Q, dO; then the fp32 staging rows over them

__global__ void __launch_bounds__(160, 1)
    lin_bwd_f_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                     const int32_t* __restrict__ chunks, const float* __restrict__ decay, int hq, int hkv,
                     float scale, float* __restrict__ f_out, int* status) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    if (sb & 1023u) {
        if (threadIdx.x == 0) report_status(status, -5);
        return;
    }
    const int G = hq / hkv;
    const int chunk = blockIdx.x / hkv, g = blockIdx.x % hkv;
    const int off = chunks[4 * chunk], L = chunks[4 * chunk + 1];
    const uint32_t b_full = sb, b_scaled = sb + 8, b_mma = sb + 16, holder = sb + 24;
    const uint32_t qa = sb + 1024, da = qa + kTile;
    if (threadIdx.x == 0) {
        mbar_init(b_full, 1);
        mbar_init(b_scaled, 128);
        mbar_init(b_mma, 1);
        fence_mbar_init();
    }
    if (warp == 4) tmem_alloc(holder, 128);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + 24);
    const float lg = log2f(decay[g]);
    bool ok = true;
    for (int n = 0; n < G; ++n) {
        if (threadIdx.x == 128 && ok) {
            // Q and dO of the previous head must have been read by its MMAs
            if (n > 0) ok = mbar_wait(b_mma, (n - 1) & 1, status, 94);
            if (ok) {
                mbar_expect_tx(b_full, 2 * kTile);
                for (int blk = 0; blk < 2; ++blk) {
                    tma_load_3d(qa + blk * 16384, &tm_q, blk * 64, g * G + n, off, b_full);
                    tma_load_3d(da + blk * 16384, &tm_do, blk * 64, g * G + n, off, b_full);
                }
            }
        }
        if (warp < 4) {
            if (ok) ok = mbar_wait(b_full, n & 1, status, 95);
            if (ok) {
                // dO row r times scale * gamma^(r+1) (0 past the chunk), in place
                const int r = threadIdx.x;
                const float w = r < L ? scale * exp2f((float)(r + 1) * lg) : 0.f;
#pragma unroll
                for (int blk = 0; blk < 2; ++blk) {
                    uint4* row = reinterpret_cast<uint4*>(smem + 1024 + kTile + blk * 16384 + r * 128);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const int cr = (c + r) & 7;   // rotated by the row: no bank conflicts
                        uint4 x = row[cr];
                        uint32_t* u = reinterpret_cast<uint32_t*>(&x);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            u[e] = pack_bf16x2(__uint_as_float(u[e] << 16) * w,
                                               __uint_as_float(u[e] & 0xffff0000u) * w);
                        row[cr] = x;
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(b_scaled);
            }
        }
        if (threadIdx.x == 128 && ok) {
            ok = mbar_wait(b_scaled, n & 1, status, 96);
            if (ok) {
                tc_fence_after();
                constexpr uint32_t ID = idesc_bf16(128, 128, true, true);   // Q^T (MN-major) x dO_w (MN-major)
#pragma unroll
                for (int k = 0; k < kChunk / 16; ++k)
                    mma_bf16_ss(tmem, sdesc_sw128(qa + k * 2048, 16384, 1024),
                                sdesc_sw128(da + k * 2048, 16384, 1024), ID, (n > 0 || k > 0) ? 1u : 0u);
                mma_commit(b_mma);
            }
        }
    }
    if (warp < 4) {
        if (ok) ok = mbar_wait(b_mma, (G - 1) & 1, status, 97);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            tc_fence_after();
            // row = key feature; the last head's Q and dO have been read, so their
            // tiles hold the staging rows
            store_rows_f32(tmem + ((uint32_t)(warp << 5) << 16), sb + 1024,
                           f_out + ((size_t)chunk * hkv + g) * kD * kD, warp, threadIdx.x & 31);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}

// ---- adjoints, chunk by chunk in reverse packed order ------------------------
// One thread per (state entry, kv-head).  Walking the chunks backwards, a node
// is left (its first chunk done) with its entering adjoint, which adds into its
// parent's sum of children; the parent is entered (its last chunk reached)
// right after its first child is left, since the first child follows its parent
// in packed order.  The running sum of the parent whose children are being left
// stays in a register (`pend`, for node `ppar`): a child of another parent
// stores it to `csum` and starts that parent's sum -- from 0 for its last child,
// the first one met, else from the partial sum stored earlier -- and entering a
// node with children takes `pend` as its entering sum.  The additions run in
// the same order as one read-modify-write per child would.  kBwdScanBatch
// increments are loaded at a time, as in the forward scan; the sums run in fp32
// and Rsum leaves as bf16, the dK/dV kernel's operand precision.
constexpr int kBwdScanBatch = 16;

__global__ void __launch_bounds__(256) lin_bwd_scan_kernel(const int32_t* __restrict__ lnodes, int n_chunks,
                                                         const int32_t* __restrict__ chunks,
                                                         const float* __restrict__ decay, int hkv,
                                                         const float* __restrict__ f_in, uint16_t* __restrict__ rsum16,
                                                         float* __restrict__ csum) {
    __shared__ float w_fac[kScanWin];
    __shared__ int w_node[kScanWin], w_par[kScanWin], w_last[kScanWin];
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    const int g = blockIdx.y;
    const size_t dd = (size_t)kD * kD;
    const float lg = log2f(decay[g]);
    auto sum_at = [&](int node) { return ((size_t)node * hkv + g) * dd + e; };
    float acc = 0.f, pend = 0.f;
    int cur = -1, cur_par = -1, cur_last = 0, ppar = -1;
    // node `cur` has been walked down to its first chunk: its entering adjoint
    // `acc` goes to its parent
    auto leave = [&]() {
        if (cur < 0 || cur_par < 0) return;
        if (ppar == cur_par) {
            pend += acc;
        } else {
            if (ppar >= 0) csum[sum_at(ppar)] = pend;
            pend = cur_last ? acc : csum[sum_at(cur_par)] + acc;
            ppar = cur_par;
        }
    };
    // windows [w0 - nw, w0) from the end; inside a window, chunk w0 - 1 - t is t
    for (int w0 = n_chunks; w0 > 0; w0 -= kScanWin) {
        const int nw = min(kScanWin, w0);
        __syncthreads();
        for (int t = threadIdx.x; t < nw; t += blockDim.x) {
            const int node = chunks[4 * (w0 - 1 - t) + 2];
            w_fac[t] = exp2f((float)chunks[4 * (w0 - 1 - t) + 1] * lg);
            w_node[t] = node;
            w_par[t] = lnodes[4 * node];
            w_last[t] = lnodes[4 * node + 3];
        }
        __syncthreads();
        for (int c = 0; c < nw; c += kBwdScanBatch) {
            float fv[kBwdScanBatch];
#pragma unroll
            for (int u = 0; u < kBwdScanBatch; ++u)
                if (c + u < nw) fv[u] = f_in[((size_t)(w0 - 1 - c - u) * hkv + g) * dd + e];
#pragma unroll
            for (int u = 0; u < kBwdScanBatch; ++u)
                if (c + u < nw) {
                    const int node = w_node[c + u];
                    if (node != cur) {   // last chunk of a node
                        leave();
                        cur = node;
                        cur_par = w_par[c + u];
                        cur_last = w_last[c + u];
                        if (ppar == node) {   // its children's sum (none: a leaf, 0)
                            acc = pend;
                            ppar = -1;
                        } else {
                            acc = 0.f;
                        }
                    }
                    rsum16[state16_index(w0 - 1 - c - u, e, g, hkv)] = float_to_bf16_bits(acc);
                    acc = fv[u] + w_fac[c + u] * acc;
                }
        }
    }
    leave();
}

// ---- the same scans, depth by depth ---------------------------------------------
// For trees of at most kMaxScanDepths depths the scans run one launch per depth
// (roots first forward, deepest first backward), one thread per (node of that
// depth, 4 state entries, kv-head): the nodes of a depth are independent, so a
// thread walks only its own node's chunks instead of every chunk of the tree,
// four entries at a time (16-byte loads, 8-byte bf16 stores) so that a wide
// depth needs few waves.  Each entry's arithmetic, and its order, is that of
// the scans above.
constexpr int kEntryBlocks = kD * kD / 1024;   // blocks of 256 threads x 4 entries per node
constexpr int kDepthBatch = 8;

__device__ __forceinline__ uint2 bf16x4(float4 v) {
    return make_uint2((uint32_t)float_to_bf16_bits(v.x) | ((uint32_t)float_to_bf16_bits(v.y) << 16),
                      (uint32_t)float_to_bf16_bits(v.z) | ((uint32_t)float_to_bf16_bits(v.w) << 16));
}

__global__ void __launch_bounds__(256) lin_scan_depth_kernel(const int32_t* __restrict__ lnodes,
                                                           const int32_t* __restrict__ nodes,
                                                           const int32_t* __restrict__ chunks,
                                                           const float* __restrict__ decay, int hkv,
                                                           const float* __restrict__ ds,
                                                           uint16_t* __restrict__ s_in16, float* __restrict__ s_out) {
    const int k = nodes[blockIdx.x / kEntryBlocks];
    const int e = ((blockIdx.x % kEntryBlocks) * 256 + threadIdx.x) * 4;   // first of 4 state entries
    const int g = blockIdx.y;
    const size_t dd = (size_t)kD * kD;
    const float lg = log2f(decay[g]);
    const int par = lnodes[4 * k], c0 = lnodes[4 * k + 1], nc = lnodes[4 * k + 2];
    float4 S = par < 0 ? make_float4(0.f, 0.f, 0.f, 0.f)
                       : *reinterpret_cast<const float4*>(s_out + ((size_t)par * hkv + g) * dd + e);
    for (int c = c0; c < c0 + nc; c += kDepthBatch) {
        float4 dsv[kDepthBatch];
        int len[kDepthBatch];
#pragma unroll
        for (int u = 0; u < kDepthBatch; ++u)
            if (c + u < c0 + nc) {
                dsv[u] = *reinterpret_cast<const float4*>(ds + ((size_t)(c + u) * hkv + g) * dd + e);
                len[u] = chunks[4 * (c + u) + 1];
            }
#pragma unroll
        for (int u = 0; u < kDepthBatch; ++u)
            if (c + u < c0 + nc) {
                *reinterpret_cast<uint2*>(s_in16 + state16_index(c + u, e, g, hkv)) = bf16x4(S);
                const float f = exp2f((float)len[u] * lg);
                S = make_float4(f * S.x + dsv[u].x, f * S.y + dsv[u].y, f * S.z + dsv[u].z, f * S.w + dsv[u].w);
            }
    }
    *reinterpret_cast<float4*>(s_out + ((size_t)k * hkv + g) * dd + e) = S;
}

// Backward: a node's entering sum is its children's entering adjoints, added in
// reverse packed order from 0 (the order of the scan above); its own entering
// adjoint goes to `ent` for its parent.
__global__ void __launch_bounds__(256) lin_bwd_scan_depth_kernel(const int32_t* __restrict__ lnodes,
                                                               const int32_t* __restrict__ kids, int n_nodes,
                                                               const int32_t* __restrict__ nodes,
                                                               const int32_t* __restrict__ chunks,
                                                               const float* __restrict__ decay, int hkv,
                                                               const float* __restrict__ f_in,
                                                               uint16_t* __restrict__ rsum16, float* __restrict__ ent) {
    const int k = nodes[blockIdx.x / kEntryBlocks];
    const int e = ((blockIdx.x % kEntryBlocks) * 256 + threadIdx.x) * 4;
    const int g = blockIdx.y;
    const size_t dd = (size_t)kD * kD;
    const float lg = log2f(decay[g]);
    const int c0 = lnodes[4 * k + 1], nc = lnodes[4 * k + 2];
    const int32_t* kid = kids + n_nodes + 1;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int x = kids[k + 1] - 1; x >= kids[k]; --x) {
        const float4 a = *reinterpret_cast<const float4*>(ent + ((size_t)kid[x] * hkv + g) * dd + e);
        acc = make_float4(acc.x + a.x, acc.y + a.y, acc.z + a.z, acc.w + a.w);
    }
    for (int c = c0 + nc - 1; c >= c0; c -= kDepthBatch) {
        float4 fv[kDepthBatch];
        int len[kDepthBatch];
#pragma unroll
        for (int u = 0; u < kDepthBatch; ++u)
            if (c - u >= c0) {
                fv[u] = *reinterpret_cast<const float4*>(f_in + ((size_t)(c - u) * hkv + g) * dd + e);
                len[u] = chunks[4 * (c - u) + 1];
            }
#pragma unroll
        for (int u = 0; u < kDepthBatch; ++u)
            if (c - u >= c0) {
                *reinterpret_cast<uint2*>(rsum16 + state16_index(c - u, e, g, hkv)) = bf16x4(acc);
                const float f = exp2f((float)len[u] * lg);
                acc = make_float4(fv[u].x + f * acc.x, fv[u].y + f * acc.y, fv[u].z + f * acc.z, fv[u].w + f * acc.w);
            }
    }
    *reinterpret_cast<float4*>(ent + ((size_t)k * hkv + g) * dd + e) = acc;
}

// ---- dK, dV per (chunk, kv-head) ------------------------------------------------
// Persistent like the output kernel: a CTA keeps kv-head g and walks chunks
// j0, j0 + lanes, ...; unit u = one (chunk, q-head) pair.
// TMEM: dK [0, 128), dV [128, 256), S^T -> P^T [256, 384), A^T -> dA^T [384, 512).
// warps 0-7: key row m' = 32 (w % 4) + lane (the TMEM lanes warp w may access);
// warp w < 4 takes queries [0, 64) of S^T and A^T (packed over their first 32
// columns) and dK, warp w >= 4 queries [64, 128) (packed at [64, 96)) and dV;
// warp 8: loads; warp 9: TMEM owner, lane 0 issues the MMAs.  The q-heads run
// one after another through two Q / dO slot pairs, so the next unit's tiles
// arrive while the current unit is worked on; its S^T and A^T products are
// issued right after the current unit's dV and dK products, which the tensor
// core completes first (products issued by one thread run in issue order), so
// P^T and dA^T are read before they are overwritten.  The two query halves are
// masked by different warps, and each half's dV and dK products start as soon
// as that half is done.  At a chunk boundary the next chunk's K, V and Rsum
// load once the last unit's S^T and A^T products have read them, and its first
// S^T and A^T products run while the element-wise warps store the finished
// chunk's dK and dV; its carried-in products wait for that store.  The mask
// weight scale * gamma^(m - m') depends on m - m' alone and is tabulated per CTA.
constexpr int kKvSmem = 2048 + 7 * kTile;   // barriers, mask table, K, V, Rsum (bf16), (Q, dO) x 2

__global__ void __launch_bounds__(kLinThreads, 1)
    lin_bwd_kv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                      const __grid_constant__ CUtensorMap tm_r, const int32_t* __restrict__ chunks, int n_chunks,
                      int lanes, const float* __restrict__ decay, uint16_t* __restrict__ dk,
                      uint16_t* __restrict__ dv, int hq, int hkv, float scale, int* status) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (sb & 1023u) {
        if (threadIdx.x == 0) report_status(status, -5);
        return;
    }
    const int G = hq / hkv;
    const int j0 = blockIdx.x / hkv, g = blockIdx.x % hkv;
    if (j0 >= n_chunks) return;   // uniform: nothing set up yet
    const int n_items = (n_chunks - 1 - j0) / lanes + 1;
    auto chunk_of = [&](int i) { return j0 + i * lanes; };
    auto bar = [&](int i) { return sb + 8u * (uint32_t)i; };
    const uint32_t b_kv = bar(0), b_kvfree = bar(1), b_inter = bar(2), b_scaled = bar(3), b_sa = bar(8),
                   b_done = bar(11), b_drain = bar(12), holder = bar(13), b_dkvfree = bar(14);
    auto b_qf = [&](int b) { return bar(4 + b); };   // slot b's Q and dO have arrived
    auto b_qe = [&](int b) { return bar(6 + b); };   // slot b's Q and dO have been read
    auto b_pa = [&](int h) { return bar(9 + h); };   // query half h masked
    const uint32_t ka = sb + 2048, va = ka + kTile, ra = va + kTile;
    auto qa = [&](int b) { return ra + kTile + 2u * kTile * (uint32_t)b; };
    auto da = [&](int b) { return qa(b) + kTile; };
    // wtab[128 + t] = scale * gamma^t for t = m - m' in [0, 128), 0 for t < 0
    float* wtab = reinterpret_cast<float*>(smem + 1024);
    if (threadIdx.x < 128) {
        wtab[threadIdx.x] = 0.f;
        wtab[128 + threadIdx.x] = scale * exp2f((float)threadIdx.x * log2f(decay[g]));
    }
    if (threadIdx.x == 0) {
        mbar_init(b_kv, 1);
        mbar_init(b_kvfree, 1);
        mbar_init(b_inter, 1);
        mbar_init(b_scaled, 256);
        for (int b = 0; b < 2; ++b) {
            mbar_init(b_qf(b), 1);
            mbar_init(b_qe(b), 1);
            mbar_init(b_pa(b), 128);
        }
        mbar_init(b_sa, 1);
        mbar_init(b_done, 1);
        mbar_init(b_dkvfree, 256);
        mbar_init(b_drain, 1);
        fence_mbar_init();
    }
    if (warp == 9) tmem_alloc(holder, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + 8 * 13);

    if (warp == 8) {
        if (lane == 0) {
            bool ok = true;
            for (int i = 0; i < n_items && ok; ++i) {
                const int chunk = chunk_of(i), off = chunks[4 * chunk];
                if (i > 0) ok = mbar_wait(b_kvfree, (i - 1) & 1, status, 110);   // the previous chunk's done with them
                if (!ok) break;
                mbar_expect_tx(b_kv, 3 * kTile);
                for (int blk = 0; blk < 2; ++blk) {
                    tma_load_3d(ka + blk * 16384, &tm_k, blk * 64, g, off, b_kv);
                    tma_load_3d(va + blk * 16384, &tm_v, blk * 64, g, off, b_kv);
                    tma_load_3d(ra + blk * 16384, &tm_r, blk * 64, g, chunk * kChunk, b_kv);
                }
                for (int n = 0; n < G && ok; ++n) {
                    const int u = i * G + n, b = u & 1, w = u >> 1;
                    if (w > 0) ok = mbar_wait(b_qe(b), (w - 1) & 1, status, 100);
                    if (!ok) break;
                    mbar_expect_tx(b_qf(b), 2 * kTile);
                    for (int blk = 0; blk < 2; ++blk) {
                        tma_load_3d(qa(b) + blk * 16384, &tm_q, blk * 64, g * G + n, off, b_qf(b));
                        tma_load_3d(da(b) + blk * 16384, &tm_do, blk * 64, g * G + n, off, b_qf(b));
                    }
                }
            }
        }
    } else if (warp == 9) {
        if (lane == 0) {
            constexpr uint32_t ID_KK = idesc_bf16(128, 128, false, false);   // B K-major
            constexpr uint32_t ID_KM = idesc_bf16(128, 128, false, true);    // B MN-major
            bool ok = true;
            for (int i = 0; i < n_items && ok; ++i) {
                for (int n = 0; n < G && ok; ++n) {
                    const int u = i * G + n, b = u & 1;
                    if (n == 0) ok = mbar_wait(b_kv, i & 1, status, 101);   // this chunk's K, V, Rsum
                    if (ok) ok = mbar_wait(b_qf(b), (u >> 1) & 1, status, 103);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t q_s = qa(b), do_s = da(b);
#pragma unroll
                    for (int k = 0; k < kD / 16; ++k) {   // S^T = K Q^T
                        const uint32_t o = (k >> 2) * 16384 + (k & 3) * 32;
                        mma_bf16_ss(tmem + 256, sdesc_sw128(ka + o, 16, 1024), sdesc_sw128(q_s + o, 16, 1024),
                                    ID_KK, k > 0);
                    }
#pragma unroll
                    for (int k = 0; k < kD / 16; ++k) {   // A^T = V dO^T
                        const uint32_t o = (k >> 2) * 16384 + (k & 3) * 32;
                        mma_bf16_ss(tmem + 384, sdesc_sw128(va + o, 16, 1024), sdesc_sw128(do_s + o, 16, 1024),
                                    ID_KK, k > 0);
                    }
                    mma_commit(b_sa);
                    if (n == 0) {
                        // carried-in parts: dK = V Rsum^T (Rsum rows = key features, i.e.
                        // K-major for this product), dV = K Rsum (the same tile read
                        // MN-major), over TMEM the previous chunk's dK, dV have left
                        if (i > 0) ok = mbar_wait(b_dkvfree, (i - 1) & 1, status, 102);
                        if (!ok) break;
                        tc_fence_after();
#pragma unroll
                        for (int k = 0; k < kD / 16; ++k) {
                            const uint32_t o = (k >> 2) * 16384 + (k & 3) * 32;
                            mma_bf16_ss(tmem, sdesc_sw128(va + o, 16, 1024), sdesc_sw128(ra + o, 16, 1024), ID_KK,
                                        k > 0);
                        }
#pragma unroll
                        for (int k = 0; k < kD / 16; ++k) {
                            const uint32_t o = (k >> 2) * 16384 + (k & 3) * 32;
                            mma_bf16_ss(tmem + 128, sdesc_sw128(ka + o, 16, 1024),
                                        sdesc_sw128(ra + k * 2048, 16384, 1024), ID_KM, k > 0);
                        }
                        mma_commit(b_inter);
                    }
                    if (n == G - 1) mma_commit(b_kvfree);   // K, V, Rsum read by the chunk's last products
                    for (int h = 0; h < 2 && ok; ++h) {
                        ok = mbar_wait(b_pa(h), u & 1, status, 104);
                        if (ok && n == 0 && h == 0) ok = mbar_wait(b_scaled, i & 1, status, 105);   // carried-in scaled
                        if (!ok) break;
                        tc_fence_after();
#pragma unroll
                        for (int k = 4 * h; k < 4 * h + 4; ++k)   // dV += P^T dO (queries 16k .. 16k + 15,
                            mma_bf16_ts(tmem + 128, tmem + 256 + h * 64 + (k & 3) * 8,   // packed at 64h + 8 (k % 4))
                                        sdesc_sw128(do_s + k * 2048, 16384, 1024), ID_KM, 1u);
#pragma unroll
                        for (int k = 4 * h; k < 4 * h + 4; ++k)   // dK += dA^T Q
                            mma_bf16_ts(tmem, tmem + 384 + h * 64 + (k & 3) * 8,
                                        sdesc_sw128(q_s + k * 2048, 16384, 1024), ID_KM, 1u);
                    }
                    if (!ok) break;
                    mma_commit(b_qe(b));   // slot b free again once these products have read it
                }
                if (ok) mma_commit(b_done);   // this chunk's dK, dV complete
            }
            mma_commit(b_drain);
            mbar_wait(b_drain, 0, status, 106);
        }
        __syncwarp();
    } else {
        const int m = ((warp & 3) << 5) + lane;   // key row m'
        const int hc = warp >> 2;                  // query half; dK (0) or dV (1)
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) << 5) << 16);
        const float lg = log2f(decay[g]);
        const float* wt = wtab + 128 - m;   // wt[m] = scale * gamma^(m - m'), 0 for m < m'
        bool ok = true;
        for (int i = 0; i < n_items; ++i) {
            const int chunk = chunk_of(i), off = chunks[4 * chunk], L = chunks[4 * chunk + 1];
            if (ok) ok = mbar_wait(b_inter, i & 1, status, 107);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) {
                // carried-in rows weigh gamma^(L-1-m') (0 past the chunk)
                tc_fence_after();
                const float w = m < L ? exp2f((float)(L - 1 - m) * lg) : 0.f;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {   // dK (half 0) or dV (half 1)
                    float v[32];
                    tmem_ld32(lane_base + hc * 128 + cc * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int x = 0; x < 32; ++x) v[x] *= w;
                    tmem_st32(lane_base + hc * 128 + cc * 32, v);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(b_scaled);
            }
            for (int n = 0; n < G; ++n) {
                const int u = i * G + n;
                if (ok) ok = mbar_wait(b_sa, u & 1, status, 108);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) continue;
                tc_fence_after();
                // P^T[m', m] = scale S^T gamma^(m-m'), dA^T[m', m] = scale A^T gamma^(m-m'),
                // for m' <= m < L; this half's 64 queries packed as bf16 over the first
                // 32 of its columns in each region
#pragma unroll 2
                for (int cq = 0; cq < 4; ++cq) {   // 16 columns at a time
                    const int cc = 4 * hc + cq;
                    float s[16], a[16];
                    tmem_ld16(lane_base + 256 + cc * 16, s);
                    tmem_ld16(lane_base + 384 + cc * 16, a);
                    tmem_wait_ld();
                    uint32_t pw[8], aw[8];
#pragma unroll
                    for (int w2 = 0; w2 < 8; ++w2) {
                        const int c0 = cc * 16 + 2 * w2, c1 = c0 + 1;
                        const float w0 = c0 < L ? wt[c0] : 0.f;
                        const float w1 = c1 < L ? wt[c1] : 0.f;
                        pw[w2] = pack_bf16x2(s[2 * w2] * w0, s[2 * w2 + 1] * w1);
                        aw[w2] = pack_bf16x2(a[2 * w2] * w0, a[2 * w2 + 1] * w1);
                    }
                    // over columns this thread has already read
                    tmem_st8(lane_base + 256 + hc * 64 + cq * 8, pw);
                    tmem_st8(lane_base + 384 + hc * 64 + cq * 8, aw);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(b_pa(hc));
            }
            if (ok) ok = mbar_wait(b_done, i & 1, status, 109);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) {
                tc_fence_after();
                uint4* dst = reinterpret_cast<uint4*>((hc ? dv : dk) + ((size_t)(off + m) * hkv + g) * kD);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    float v[32];
                    tmem_ld32(lane_base + hc * 128 + cc * 32, v);
                    tmem_wait_ld();
                    if (m < L) {
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            uint4 y;
                            y.x = pack_bf16x2(v[8 * x], v[8 * x + 1]);
                            y.y = pack_bf16x2(v[8 * x + 2], v[8 * x + 3]);
                            y.z = pack_bf16x2(v[8 * x + 4], v[8 * x + 5]);
                            y.w = pack_bf16x2(v[8 * x + 6], v[8 * x + 7]);
                            dst[cc * 4 + x] = y;
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(b_dkvfree);   // TMEM dK, dV may take the next chunk's carried-in parts
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// The forward scan: depth by depth where the plan has the depth tables, else
// one walk over every chunk.
int launch_scan(const tree_attn_plan_s* P, const DevicePlan* D, int64_t nc, const float* decay, int hkv,
                const float* ds, uint16_t* s_in16, float* s_out, cudaStream_t s) {
    const LinInfo& X = P->lin;
    if (X.lvl_ptr.empty()) {
        lin_scan_kernel<<<dim3(kD * kD / 256, hkv), 256, 0, s>>>(D->lnodes, (int)nc, D->chunks, decay, hkv, ds,
                                                                 s_in16, s_out);
        return cudaGetLastError() == cudaSuccess ? TREE_ATTN_OK : TREE_ATTN_ERR_CUDA;
    }
    for (size_t l = 0; l + 1 < X.lvl_ptr.size(); ++l) {
        const int64_t blocks = (int64_t)(X.lvl_ptr[l + 1] - X.lvl_ptr[l]) * kEntryBlocks;
        if (blocks > INT32_MAX) return TREE_ATTN_ERR_TOO_LARGE;
        lin_scan_depth_kernel<<<dim3((unsigned)blocks, hkv), 256, 0, s>>>(D->lnodes, D->lvl_nodes + X.lvl_ptr[l],
                                                                         D->chunks, decay, hkv, ds, s_in16, s_out);
        if (cudaGetLastError() != cudaSuccess) return TREE_ATTN_ERR_CUDA;
    }
    return TREE_ATTN_OK;
}

// The reverse scan: deepest nodes first where the plan has the depth tables.
int launch_bwd_scan(const tree_attn_plan_s* P, const DevicePlan* D, int64_t nc, const float* decay, int hkv,
                    const float* f_in, uint16_t* rsum16, float* csum, cudaStream_t s) {
    const LinInfo& X = P->lin;
    if (X.lvl_ptr.empty()) {
        lin_bwd_scan_kernel<<<dim3(kD * kD / 256, hkv), 256, 0, s>>>(D->lnodes, (int)nc, D->chunks, decay, hkv,
                                                                     f_in, rsum16, csum);
        return cudaGetLastError() == cudaSuccess ? TREE_ATTN_OK : TREE_ATTN_ERR_CUDA;
    }
    for (size_t l = X.lvl_ptr.size() - 1; l-- > 0;) {
        const int64_t blocks = (int64_t)(X.lvl_ptr[l + 1] - X.lvl_ptr[l]) * kEntryBlocks;
        if (blocks > INT32_MAX) return TREE_ATTN_ERR_TOO_LARGE;
        lin_bwd_scan_depth_kernel<<<dim3((unsigned)blocks, hkv), 256, 0, s>>>(
            D->lnodes, D->kids, P->n_nodes, D->lvl_nodes + X.lvl_ptr[l], D->chunks, decay, hkv, f_in, rsum16, csum);
        if (cudaGetLastError() != cudaSuccess) return TREE_ATTN_ERR_CUDA;
    }
    return TREE_ATTN_OK;
}

// Chunk lanes of the persistent output kernel: about one CTA per SM in all
// (lanes x hkv CTAs), at least one lane, at most one per chunk.
int out_lanes(int dev, int64_t n_chunks, int hkv) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 1;
    return (int)std::max<int64_t>(1, std::min<int64_t>(n_chunks, sms / hkv));
}

}  // namespace

}  // namespace treeattn

using namespace treeattn;

extern "C" {

int tree_attn_linear_workspace_size(tree_attn_plan_t P, int32_t hkv, int32_t d, int64_t* n_chunks, size_t* ws_bytes) {
    if (!P || hkv <= 0) return TREE_ATTN_ERR_INVALID_ARG;
    if (d != kD) return TREE_ATTN_ERR_UNSUPPORTED;
    {
        std::lock_guard<std::mutex> lk(P->mu);
        int st = build_lin(P);
        if (st) return st;
    }
    if (n_chunks) *n_chunks = (int64_t)(P->lin.chunks.size() / 4);
    if (ws_bytes) *ws_bytes = lin_layout(P, hkv).total;
    return TREE_ATTN_OK;
}

int tree_attn_linear_fwd(tree_attn_plan_t P, const void* q, const void* k, const void* v, void* o,
                         const float* decay, int32_t hq, int32_t hkv, int32_t d, float scale, void* workspace,
                         size_t ws_bytes, void* stream) {
    if (!P || !q || !k || !v || !o || !decay || hq <= 0 || hkv <= 0 || hq % hkv != 0) return TREE_ATTN_ERR_INVALID_ARG;
    if (d != kD || P->block != kChunk) return TREE_ATTN_ERR_UNSUPPORTED;
    if (!(scale > 0.f) || !std::isfinite(scale)) return TREE_ATTN_ERR_INVALID_ARG;
    for (const void* p : {q, k, v, (const void*)o})
        if (!aligned(p, 16)) return TREE_ATTN_ERR_ALIGNMENT;
    if (!aligned(decay, 4) || !aligned(workspace, 256)) return TREE_ATTN_ERR_ALIGNMENT;
    DevicePlan* D = nullptr;
    int st = ensure_lin_device(P, &D);
    if (st) return st;
    const LinWs w = lin_layout(P, hkv);
    if (!workspace || ws_bytes < w.total) return TREE_ATTN_ERR_WORKSPACE;
    const int64_t nc = (int64_t)(P->lin.chunks.size() / 4);
    if (nc * hq > INT32_MAX || nc * hkv > INT32_MAX) return TREE_ATTN_ERR_TOO_LARGE;
    CUtensorMap tq, tk, tv;
    if ((st = make_tensor_map(&tq, q, P->N, hq, d)) || (st = make_tensor_map(&tk, k, P->N, hkv, d)) ||
        (st = make_tensor_map(&tv, v, P->N, hkv, d)))
        return st;
    int dev = 0;
    cudaGetDevice(&dev);
    int* status = nullptr;
    if ((st = get_status_ptr(dev, &status))) return st;
    char* ws = static_cast<char*>(workspace);
    float* ds = reinterpret_cast<float*>(ws + w.ds);
    uint16_t* s_in16 = reinterpret_cast<uint16_t*>(ws + w.s_in);   // bf16 entering states
    CUtensorMap ts;
    if ((st = make_tensor_map(&ts, s_in16, nc * kChunk, hkv, kD))) return st;
    float* s_out = reinterpret_cast<float*>(ws + w.s_out);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaFuncSetAttribute(lin_delta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDeltaSmem) != cudaSuccess ||
        cudaFuncSetAttribute(lin_out_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kOutSmem) != cudaSuccess)
        return TREE_ATTN_ERR_CUDA;
    lin_delta_kernel<<<(unsigned)(nc * hkv), 160, kDeltaSmem, s>>>(tk, tv, D->chunks, decay, hkv, ds, status);
    if (cudaGetLastError() != cudaSuccess) return TREE_ATTN_ERR_CUDA;
    if ((st = launch_scan(P, D, nc, decay, hkv, ds, s_in16, s_out, s))) return st;
    const int lanes = out_lanes(dev, nc, hkv);
    lin_out_kernel<<<(unsigned)(lanes * hkv), kLinThreads, kOutSmem, s>>>(tq, tk, tv, ts, D->chunks, (int)nc, lanes,
                                                                      decay, static_cast<uint16_t*>(o), hq, hkv,
                                                                      scale, status);
    return cudaGetLastError() == cudaSuccess ? TREE_ATTN_OK : TREE_ATTN_ERR_CUDA;
}


int tree_attn_linear_bwd(tree_attn_plan_t P, const void* q, const void* k, const void* v, const void* dout,
                         void* dq, void* dk, void* dv, const float* decay, int32_t hq, int32_t hkv, int32_t d,
                         float scale, void* workspace, size_t ws_bytes, void* stream) {
    if (!P || !q || !k || !v || !dout || !dq || !dk || !dv || !decay || hq <= 0 || hkv <= 0 || hq % hkv != 0)
        return TREE_ATTN_ERR_INVALID_ARG;
    if (d != kD || P->block != kChunk) return TREE_ATTN_ERR_UNSUPPORTED;
    if (!(scale > 0.f) || !std::isfinite(scale)) return TREE_ATTN_ERR_INVALID_ARG;
    for (const void* p : {q, k, v, dout, (const void*)dq, (const void*)dk, (const void*)dv})
        if (!aligned(p, 16)) return TREE_ATTN_ERR_ALIGNMENT;
    if (!aligned(decay, 4) || !aligned(workspace, 256)) return TREE_ATTN_ERR_ALIGNMENT;
    DevicePlan* D = nullptr;
    int st = ensure_lin_device(P, &D);
    if (st) return st;
    const LinWs w = lin_layout(P, hkv);
    if (!workspace || ws_bytes < w.total) return TREE_ATTN_ERR_WORKSPACE;
    const int64_t nc = (int64_t)(P->lin.chunks.size() / 4);
    if (nc * hq > INT32_MAX || nc * hkv > INT32_MAX) return TREE_ATTN_ERR_TOO_LARGE;
    CUtensorMap tq, tk, tv, tdo;
    if ((st = make_tensor_map(&tq, q, P->N, hq, d)) || (st = make_tensor_map(&tk, k, P->N, hkv, d)) ||
        (st = make_tensor_map(&tv, v, P->N, hkv, d)) || (st = make_tensor_map(&tdo, dout, P->N, hq, d)))
        return st;
    int dev = 0;
    cudaGetDevice(&dev);
    int* status = nullptr;
    if ((st = get_status_ptr(dev, &status))) return st;
    char* ws = static_cast<char*>(workspace);
    float* r0 = reinterpret_cast<float*>(ws + w.ds);      // dS', then F
    uint16_t* r1 = reinterpret_cast<uint16_t*>(ws + w.s_in);   // bf16 S'_in, then bf16 Rsum
    CUtensorMap tr1;
    if ((st = make_tensor_map(&tr1, r1, nc * kChunk, hkv, kD))) return st;
    float* r2 = reinterpret_cast<float*>(ws + w.s_out);   // S'_out, then the per-node child sums
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaFuncSetAttribute(lin_delta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDeltaSmem) != cudaSuccess ||
        cudaFuncSetAttribute(lin_out_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kOutSmem) != cudaSuccess ||
        cudaFuncSetAttribute(lin_bwd_f_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAdjSmem) != cudaSuccess ||
        cudaFuncSetAttribute(lin_bwd_kv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kKvSmem) != cudaSuccess)
        return TREE_ATTN_ERR_CUDA;
    // dQ: the forward with (q, k, v) = (dO, V, K)
    lin_delta_kernel<<<(unsigned)(nc * hkv), 160, kDeltaSmem, s>>>(tv, tk, D->chunks, decay, hkv, r0, status);
    if (cudaGetLastError() != cudaSuccess) return TREE_ATTN_ERR_CUDA;
    if ((st = launch_scan(P, D, nc, decay, hkv, r0, r1, r2, s))) return st;
    const int lanes = out_lanes(dev, nc, hkv);
    lin_out_kernel<<<(unsigned)(lanes * hkv), kLinThreads, kOutSmem, s>>>(tdo, tv, tk, tr1, D->chunks, (int)nc, lanes,
                                                                      decay, static_cast<uint16_t*>(dq), hq, hkv,
                                                                      scale, status);
    if (cudaGetLastError() != cudaSuccess) return TREE_ATTN_ERR_CUDA;
    // dK, dV: adjoint increments, the reverse scan, then the per-chunk products
    lin_bwd_f_kernel<<<(unsigned)(nc * hkv), 160, kAdjSmem, s>>>(tq, tdo, D->chunks, decay, hq, hkv, scale, r0, status);
    if (cudaGetLastError() != cudaSuccess) return TREE_ATTN_ERR_CUDA;
    if ((st = launch_bwd_scan(P, D, nc, decay, hkv, r0, r1, r2, s))) return st;
    lin_bwd_kv_kernel<<<(unsigned)(lanes * hkv), kLinThreads, kKvSmem, s>>>(tq, tk, tv, tdo, tr1, D->chunks, (int)nc,
                                                                         lanes, decay,
                                                                 static_cast<uint16_t*>(dk), static_cast<uint16_t*>(dv),
                                                                 hq, hkv, scale, status);
    return cudaGetLastError() == cudaSuccess ? TREE_ATTN_OK : TREE_ATTN_ERR_CUDA;
}

}  // extern "C"
