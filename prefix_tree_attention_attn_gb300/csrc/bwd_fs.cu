// Backward kernel for head_dim 128: dQ, dK, dV of tree attention on the
// sm_103a tensor cores, full 128-query steps with every MMA at N = 128.
//
// KV-major: one CTA = one work item (kv-tile c, a chunk [t0, t1) of its
// contiguous descendant q-range) x one kv-head.  K_c and V_c stay in shared
// memory, dV and dK in TMEM; steps (q-tile t ascending, then q-head h of the
// group) run in a fixed order, so dK and dV are bitwise reproducible.
//
// TMEM (512 columns):
//   [0, 128)    S^T = K Q^T; the compute warps write P^T over it as packed
//               bf16, each warp into the first half of the W columns it read
//               per half-tile (W = 32 with 8 compute warps, 16 with 16)
//   [128, 256)  dP^T = V dO^T; after dS^T is written, dQ = dS K (lane = query)
//   [256, 384)  dV += P^T dO      (A operand P^T read from TMEM)
//   [384, 512)  dK += dS^T Q      (dS^T from shared memory)
//
// Tensor-core order per step n:
//   dV(n) | S(n+1) | dQ(n) dK(n) | dP(n+1)
// dV(n) waits for P^T(n); S(n+1) reuses the S^T columns right after it; dQ(n)
// and dK(n) wait for dS^T(n); dP(n+1) waits until dQ(n) has left TMEM.  The
// compute warps alternate P(n), dS(n), P(n+1), ... and find S(n+1) and dP(n+1)
// ready (or nearly) when they get there, so the tensor core and the compute
// warps overlap without splitting a step into narrower MMAs.
//
// dQ leaves TMEM through the registers of a dedicated readout warpgroup, in
// two rounds of 64 features.  Each round goes out as two 32-feature halves
// through a 32 KB shared staging tile laid out like the fp32 dQ accumulator
// ([query][feature], 128B-swizzled, one 16 KB half per 32 features); an
// asynchronous TMA reduce-add carries each half to the accumulator.  A half is
// rewritten as soon as the reduce issued two halves earlier has read it, so
// one reduce is always in flight while the next half is written.  TMEM is
// released as soon as the second round's columns are in registers.  With every
// SM adding 64 KB of dQ per step into L2, this reduce stream is what bounds a
// step.
//
// Q tiles go through a 2-slot ring (Q(n) serves S(n), issued during step n-1,
// and dK(n)); dO tiles through one slot, refilled as soon as dV(n) has read
// it, long before dP(n+1) needs the next one.
//
// Warp roles (NCW + 6 warps): warps 0 .. NCW-1 compute P^T and dS^T (warp w
// owns TMEM lanes 32*(w%4).. -- one key each -- and query columns
// [W*(w/4), +W) and [64 + W*(w/4), +W) of every step); the next 4 warps read
// dQ out of TMEM (lane = query) and issue the reduce; then the TMA producer
// (K, V once; Q and dO per step, the next tiles prefetched into L2; LSE and
// Delta rows by bulk copy) and the MMA issuer, which owns TMEM.
#include "kernels.h"
#include "ptx.cuh"

namespace treeattn {

namespace {

// Optional clock64 event trace of a few CTAs (build with -DTREE_ATTN_TRACE;
// off in normal builds): every 128th CTA, up to 8 of them, first 32 steps.
#ifdef TREE_ATTN_TRACE
constexpr int kTrCtas = 8, kTrSteps = 32, kTrEv = 24;
__device__ unsigned long long g_bwd_trace[kTrCtas][kTrSteps][kTrEv];
#define BWD_TRACE(ev, n)                                                                        \
    do {                                                                                         \
        if ((blockIdx.x & 127u) == 0 && (blockIdx.x >> 7) < kTrCtas && (n) < kTrSteps)          \
            g_bwd_trace[blockIdx.x >> 7][(n)][(ev)] = clock64();                                 \
    } while (0)
#else
#define BWD_TRACE(ev, n) \
    do {                 \
    } while (0)
#endif

// Wait until every bulk group this thread committed, except the most recent one,
// has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[N]) {
    static_assert(N == 16 || N == 32, "columns");
    if constexpr (N == 32) tmem_ld32(taddr, v);
    else tmem_ld16(taddr, v);
}
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&v)[N]) {
    static_assert(N == 8 || N == 16, "columns");
    if constexpr (N == 16) tmem_st16(taddr, v);
    else tmem_st8(taddr, v);
}

template <int NCW_>
struct FsCfg {
    static constexpr int D = 128;
    static constexpr int TILE = 128 * D * 2;                  // 32 KB
    static constexpr int SMALL = 3072;
    static constexpr int OFF_K = SMALL;
    static constexpr int OFF_V = OFF_K + TILE;
    static constexpr int OFF_DST = OFF_V + TILE;              // dS^T: 128 keys x 128 queries bf16 (2 blocks)
    static constexpr int OFF_Q = OFF_DST + TILE;              // [2] Q tiles
    static constexpr int OFF_DO = OFF_Q + 2 * TILE;           // dO tile
    static constexpr int OFF_STAGE = OFF_DO + TILE;           // dQ staging: 2 halves of 128 queries x 32 features fp32
    static constexpr int BYTES = OFF_STAGE + 32768;
    static constexpr int NCW = NCW_;                          // compute warps 0 .. NCW-1
    static constexpr int W = 256 / NCW;                       // query columns per compute warp per half-tile
    static constexpr int EW = 512 / NCW;                      // dK / dV columns per compute warp
    static constexpr int NCOMPUTE = NCW * 32;
    static constexpr int READOUT0 = NCW;                      // 4 readout warps
    static constexpr int NREADOUT = 128;
    static constexpr int PRODUCER = NCW + 4;
    static constexpr int MMA = NCW + 5;
    static constexpr int NWARPS = NCW + 6;
    static constexpr int TMEM_COLS = 512;
    static constexpr int T_S = 0, T_DP = 128, T_DQ = 128, T_DV = 256, T_DK = 384;
    // small region
    static constexpr int B_KVFULL = 0;
    static constexpr int B_QFULL = 8;                     // [2]
    static constexpr int B_QEMPTY = B_QFULL + 16;         // [2]
    static constexpr int B_DOFULL = B_QEMPTY + 16;
    static constexpr int B_DOEMPTY = B_DOFULL + 8;
    static constexpr int B_LFULL = B_DOEMPTY + 8;         // [2]
    static constexpr int B_LEMPTY = B_LFULL + 16;         // [2]
    static constexpr int B_SFULL = B_LEMPTY + 16;         // S^T(n) ready
    static constexpr int B_DPFULL = B_SFULL + 8;          // dP^T(n) ready
    static constexpr int B_PFULL = B_DPFULL + 8;          // P^T(n) written
    static constexpr int B_DSFULL = B_PFULL + 8;          // dS^T(n) written, dP^T(n) read
    static constexpr int B_DQFULL = B_DSFULL + 8;         // dQ(n) ready
    static constexpr int B_DQEMPTY = B_DQFULL + 8;        // dQ(n) read out
    static constexpr int B_DKVFULL = B_DQEMPTY + 8;
    static constexpr int B_DRAIN = B_DKVFULL + 8;
    static constexpr int HOLDER = B_DRAIN + 8;
    static constexpr int LSD = 1024;                      // 2 stages x {lse2[128], delta[128]}
    static_assert(HOLDER + 4 <= LSD, "barriers");
    static_assert(LSD + 2 * 1024 <= SMALL, "small region");
    static_assert(BYTES <= 232448, "shared memory");
};

template <int NCW>
__global__ void __launch_bounds__(FsCfg<NCW>::NWARPS * 32, 1)
    bwd_fs_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
    using C = FsCfg<NCW>;
    constexpr int D = C::D;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (sb & 1023u) {
        if (threadIdx.x == 0) report_status(p.status, -5);
        return;
    }
    int item, hk;
    bwd_cta_work(p, blockIdx.x, item, hk);
    if (item < 0) return;   // debug builds: the CTA index maps to no item
    const int4 it = reinterpret_cast<const int4*>(p.items)[item];
    const int c = it.x, t0 = it.y, t1 = it.z, slot = it.w;
    // debug builds: the item's kv-tile, q-range, slot and kv-head must lie inside
    // the plan's tables (a uniform return, before any barrier or TMEM is set up)
    if (!(ta_ok(p.status, 211, c, 0, p.T) && ta_ok(p.status, 212, t0, c, p.T) &&
          ta_ok(p.status, 213, t1, t0 + 1, (long long)p.T + 1) && ta_ok(p.status, 214, slot, -1, p.n_slots) &&
          ta_ok(p.status, 215, hk, 0, p.hkv)))
        return;
    const int G = p.group;
    const int nsteps = (t1 - t0) * G;

    auto bar = [&](int off) { return sb + (uint32_t)off; };
    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_KVFULL), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(C::B_QFULL + 8 * s), 1);
            mbar_init(bar(C::B_QEMPTY + 8 * s), 1);
            mbar_init(bar(C::B_LFULL + 8 * s), 1);
            mbar_init(bar(C::B_LEMPTY + 8 * s), C::NCOMPUTE);
        }
        mbar_init(bar(C::B_DOFULL), 1);
        mbar_init(bar(C::B_DOEMPTY), 1);
        mbar_init(bar(C::B_SFULL), 1);
        mbar_init(bar(C::B_DPFULL), 1);
        mbar_init(bar(C::B_PFULL), C::NCOMPUTE);
        mbar_init(bar(C::B_DSFULL), C::NCOMPUTE);
        mbar_init(bar(C::B_DQFULL), 1);
        mbar_init(bar(C::B_DQEMPTY), C::NREADOUT);
        mbar_init(bar(C::B_DKVFULL), 1);
        mbar_init(bar(C::B_DRAIN), 1);
        fence_mbar_init();
    }
    if (warp == C::MMA) tmem_alloc(sb + C::HOLDER, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::HOLDER);
    // Delta, LSE and the zeroed dQ accumulator come from the pre kernel just before
    grid_dep_wait();
    grid_dep_launch();
    if (threadIdx.x == 0) BWD_TRACE(20, 0);

    if (warp == C::PRODUCER) {
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_do);
            mbar_expect_tx(bar(C::B_KVFULL), 2 * C::TILE);
            for (int blk = 0; blk < D / 64; ++blk) {
                tma_load_3d(sb + C::OFF_K + blk * 16384, &tm_k, blk * 64, hk, c * 128, bar(C::B_KVFULL));
                tma_load_3d(sb + C::OFF_V + blk * 16384, &tm_v, blk * 64, hk, c * 128, bar(C::B_KVFULL));
            }
            auto prefetch = [&](int n) {
                if (n >= nsteps) return;
                const int t = t0 + n / G, h = hk * G + n % G;
                for (int blk = 0; blk < D / 64; ++blk) {
                    tma_prefetch_3d(&tm_q, blk * 64, h, t * 128);
                    tma_prefetch_3d(&tm_do, blk * 64, h, t * 128);
                }
            };
            prefetch(1);
            bool ok = true;
            for (int n = 0; n < nsteps && ok; ++n) {
                const int t = t0 + n / G, h = hk * G + n % G;
                prefetch(n + 2);
                // Q(n) into slot n % 2, once dK(n-2) has read it
                const int qs = n & 1;
                if (n >= 2) ok = mbar_wait(bar(C::B_QEMPTY + 8 * qs), ((n >> 1) - 1) & 1, p.status, 61);
                if (!ok) break;
                mbar_expect_tx(bar(C::B_QFULL + 8 * qs), C::TILE);
                for (int blk = 0; blk < D / 64; ++blk)
                    tma_load_3d(sb + C::OFF_Q + qs * C::TILE + blk * 16384, &tm_q, blk * 64, h, t * 128,
                                bar(C::B_QFULL + 8 * qs));
                BWD_TRACE(18, n);
                // LSE and Delta rows of step n, once step n-2 is done with the stage
                const int ls = n & 1;
                if (n >= 2) ok = mbar_wait(bar(C::B_LEMPTY + 8 * ls), ((n >> 1) - 1) & 1, p.status, 62);
                if (!ok) break;
                mbar_expect_tx(bar(C::B_LFULL + 8 * ls), 1024);
                const size_t off = (size_t)ta_clamp(p.status, 216, (long long)h * p.Npad + (long long)t * 128, 0,
                                                    (long long)p.hq * p.Npad - 127);
                bulk_load(sb + C::LSD + ls * 1024, p.lse2 + off, 512, bar(C::B_LFULL + 8 * ls));
                bulk_load(sb + C::LSD + ls * 1024 + 512, p.delta + off, 512, bar(C::B_LFULL + 8 * ls));
                // dO(n), once dV(n-1) has read dO(n-1)
                if (n >= 1) ok = mbar_wait(bar(C::B_DOEMPTY), (n - 1) & 1, p.status, 63);
                if (!ok) break;
                mbar_expect_tx(bar(C::B_DOFULL), C::TILE);
                for (int blk = 0; blk < D / 64; ++blk)
                    tma_load_3d(sb + C::OFF_DO + blk * 16384, &tm_do, blk * 64, h, t * 128, bar(C::B_DOFULL));
                BWD_TRACE(19, n);
            }
        }
    } else if (warp == C::MMA) {
        if (lane == 0) {
            constexpr uint32_t ID_S = idesc_bf16(128, 128, false, false);   // K Q^T, V dO^T
            constexpr uint32_t ID_KV = idesc_bf16(128, D, false, true);     // P^T (TMEM) dO, dS^T Q
            constexpr uint32_t ID_DQ = idesc_bf16(128, D, true, true);      // dS K
            const uint32_t ka = sb + C::OFF_K, va = sb + C::OFF_V, dsa = sb + C::OFF_DST, doa = sb + C::OFF_DO;
            auto q_addr = [&](int n) { return sb + C::OFF_Q + (n & 1) * C::TILE; };
            auto wait_q = [&](int n) {
                return mbar_wait(bar(C::B_QFULL + 8 * (n & 1)), (n >> 1) & 1, p.status, 64);
            };
            auto wait_do = [&](int n) { return mbar_wait(bar(C::B_DOFULL), n & 1, p.status, 65); };
            auto issue_s = [&](int n) {   // S^T = K Q_n^T
                const uint32_t qa = q_addr(n);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
                    mma_bf16_ss(tmem + C::T_S, sdesc_sw128(ka + off, 16, 1024), sdesc_sw128(qa + off, 16, 1024),
                                ID_S, k > 0);
                }
                mma_commit(bar(C::B_SFULL));
            };
            auto issue_dp = [&]() {   // dP^T = V dO^T
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
                    mma_bf16_ss(tmem + C::T_DP, sdesc_sw128(va + off, 16, 1024), sdesc_sw128(doa + off, 16, 1024),
                                ID_S, k > 0);
                }
                mma_commit(bar(C::B_DPFULL));
            };
            bool ok = mbar_wait(bar(C::B_KVFULL), 0, p.status, 66);
            if (ok) ok = wait_q(0);
            if (ok) {
                tc_fence_after();
                issue_s(0);
                ok = wait_do(0);
            }
            if (ok) {
                tc_fence_after();
                issue_dp();
            }
            for (int n = 0; n < nsteps && ok; ++n) {
                // dV += P^T dO: the W-query group g of P^T is packed at TMEM columns
                // [g*W, g*W + W/2), so queries 16k.. start at (16k/W)*W + (16k%W)/2
                ok = mbar_wait(bar(C::B_PFULL), n & 1, p.status, 67);
                if (!ok) break;
                BWD_TRACE(4, n);
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_bf16_ts(tmem + C::T_DV, tmem + C::T_S + (16 * k / C::W) * C::W + (16 * k % C::W) / 2,
                                sdesc_sw128(doa + k * 2048, 16384, 1024),
                                ID_KV, (n > 0 || k > 0) ? 1u : 0u);
                mma_commit(bar(C::B_DOEMPTY));
                BWD_TRACE(5, n);
                if (n + 1 < nsteps) {   // S^T(n+1) over P^T(n): after dV(n) in issue order
                    ok = wait_q(n + 1);
                    if (!ok) break;
                    BWD_TRACE(6, n);
                    tc_fence_after();
                    issue_s(n + 1);
                    BWD_TRACE(7, n);
                }
                ok = mbar_wait(bar(C::B_DSFULL), n & 1, p.status, 68);
                if (!ok) break;
                BWD_TRACE(8, n);
                tc_fence_after();
                // dQ = dS K   (M = queries: A is dS^T read MN-major; K dimension = 128 keys)
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_bf16_ss(tmem + C::T_DQ, sdesc_sw128(dsa + k * 2048, 16384, 1024),
                                sdesc_sw128(ka + k * 2048, 16384, 1024), ID_DQ, k > 0);
                mma_commit(bar(C::B_DQFULL));
                BWD_TRACE(9, n);
                // dK += dS^T Q   (K dimension = 128 queries)
                const uint32_t qa = q_addr(n);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_bf16_ss(tmem + C::T_DK, sdesc_sw128(dsa + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024),
                                sdesc_sw128(qa + k * 2048, 16384, 1024), ID_KV, (n > 0 || k > 0) ? 1u : 0u);
                mma_commit(bar(C::B_QEMPTY + 8 * (n & 1)));
                BWD_TRACE(10, n);
                if (n + 1 < nsteps) {   // dP^T(n+1) over dQ(n), once it has been read out
                    ok = wait_do(n + 1);
                    BWD_TRACE(11, n);
                    if (ok) ok = mbar_wait(bar(C::B_DQEMPTY), n & 1, p.status, 69);
                    if (!ok) break;
                    BWD_TRACE(12, n);
                    tc_fence_after();
                    issue_dp();
                }
                BWD_TRACE(13, n);
            }
            if (ok) mma_commit(bar(C::B_DKVFULL));
            mma_commit(bar(C::B_DRAIN));
            mbar_wait(bar(C::B_DRAIN), 0, p.status, 70);
        }
        __syncwarp();
    } else if (warp >= C::READOUT0) {
        // ------------------------------ dQ readout ------------------------------
        const int quarter = warp & 3;
        const int rrow = (quarter << 5) + lane;                                 // query row of the tile
        const uint32_t lane_base = tmem + ((uint32_t)(quarter << 5) << 16);
        const int rtid = threadIdx.x - C::READOUT0 * 32;                        // 0..127
        const uint32_t stage = sb + C::OFF_STAGE;
        bool ok = true;
        // loops run to the end after a failed wait (work skipped), so the named
        // barriers of this warpgroup always line up
        for (int n = 0; n < nsteps; ++n) {
            const int t = t0 + n / G, h = hk * G + n % G;
            const int q0 = t * 128;
            if (ok) ok = mbar_wait(bar(C::B_DQFULL), n & 1, p.status, 71);
            if (lane == 0 && warp == C::READOUT0) BWD_TRACE(14, n);
            ok = __all_sync(0xffffffffu, ok);
#pragma unroll
            for (int rd = 0; rd < 2; ++rd) {
                float v[64];
                if (ok) {
                    tc_fence_after();
                    tmem_ld32(lane_base + C::T_DQ + 64 * rd, *reinterpret_cast<float(*)[32]>(&v[0]));
                    tmem_ld32(lane_base + C::T_DQ + 64 * rd + 32, *reinterpret_cast<float(*)[32]>(&v[32]));
                    tmem_wait_ld();
                    if (rd == 1) {
                        tc_fence_before();
                        mbar_arrive(bar(C::B_DQEMPTY));   // dQ(n) has left TMEM
                        if (lane == 0 && warp == C::READOUT0) BWD_TRACE(15, n);
                    }
                }
#pragma unroll
                for (int blk = 0; blk < 2; ++blk) {
                    // half blk of the staging tile: the reduce issued two halves ago has read it
                    if (rtid == 0) bulk_wait_read_1();
                    ok = named_bar_and(2, C::NREADOUT, ok);
                    if (ok) {
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const float* s = &v[blk * 32 + 4 * k];
                            st_shared_v4(stage + blk * 16384 + sw128_offset(rrow, k), __float_as_uint(s[0] * p.scale),
                                         __float_as_uint(s[1] * p.scale), __float_as_uint(s[2] * p.scale),
                                         __float_as_uint(s[3] * p.scale));
                        }
                    }
                    fence_proxy_async_smem();
                    ok = named_bar_and(2, C::NREADOUT, ok);
                    if (ok && rtid == 0) {
                        tma_reduce_add_3d(&tm_dq, stage + blk * 16384, rd * 64 + blk * 32, h, q0);
                        bulk_commit();
                        BWD_TRACE(16 + rd, n);
                    }
                }
            }
        }
        if (rtid == 0) bulk_wait_all();
    } else {
        // ------------------------------ compute -------------------------------
        constexpr int W = C::W;
        const int quarter = warp & 3, cs = warp >> 2;  // TMEM lane quarter, W-column slice of each half
        const int r = (quarter << 5) + lane;           // TMEM lane = this thread's key
        const uint32_t lane_base = tmem + ((uint32_t)(quarter << 5) << 16);
        const int j = c * 128 + r;
        const int sub_j = p.subend[ta_clamp(p.status, 217, j, 0, (long long)p.T * 128)];   // 0 past N
        const float sl2 = p.scale_log2;
        const uint32_t dsa = sb + C::OFF_DST;
        bool ok = true;
        for (int n = 0; n < nsteps; ++n) {
            const int t = t0 + n / G;
            const int q0 = t * 128;
            const int lo = max(j - q0, 0), hi = min(sub_j - q0, 128);
            const int ls = n & 1;
            if (ok) ok = mbar_wait(bar(C::B_LFULL + 8 * ls), (n >> 1) & 1, p.status, 72);
            if (ok) ok = mbar_wait(bar(C::B_SFULL), n & 1, p.status, 73);
            if (threadIdx.x == 0) BWD_TRACE(0, n);
            ok = __all_sync(0xffffffffu, ok);
            const float4* lse4 = reinterpret_cast<const float4*>(smem + C::LSD + ls * 1024);
            const float4* del4 = reinterpret_cast<const float4*>(smem + C::LSD + ls * 1024 + 512);
            // P^T for this thread's 2W query columns (W per half-tile), fp32 for dS
            // and packed bf16 for TMEM (the dV MMA's A operand)
            float pk[2][W];
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    const int cbase = 64 * x + W * cs;
                    float sv[W];
                    tmem_ld_cols(lane_base + C::T_S + cbase, sv);
                    tmem_wait_ld();
                    if (lo <= cbase && hi >= cbase + W) {   // every column of this row attends
#pragma unroll
                        for (int u4 = 0; u4 < W / 4; ++u4) {
                            const float4 l4 = lse4[cbase / 4 + u4];
                            pk[x][u4 * 4 + 0] = fast_exp2(fmaf(sv[u4 * 4 + 0], sl2, -l4.x));
                            pk[x][u4 * 4 + 1] = fast_exp2(fmaf(sv[u4 * 4 + 1], sl2, -l4.y));
                            pk[x][u4 * 4 + 2] = fast_exp2(fmaf(sv[u4 * 4 + 2], sl2, -l4.z));
                            pk[x][u4 * 4 + 3] = fast_exp2(fmaf(sv[u4 * 4 + 3], sl2, -l4.w));
                        }
                    } else {
#pragma unroll
                        for (int u4 = 0; u4 < W / 4; ++u4) {
                            const float4 l4 = lse4[cbase / 4 + u4];
                            const float la[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                            for (int w = 0; w < 4; ++w) {
                                const int col = cbase + u4 * 4 + w;
                                const float e = fast_exp2(fmaf(sv[u4 * 4 + w], sl2, -la[w]));
                                pk[x][u4 * 4 + w] = (col >= lo && col < hi) ? e : 0.f;
                            }
                        }
                    }
                    uint32_t pw[W / 2];
#pragma unroll
                    for (int u = 0; u < W / 2; ++u) pw[u] = pack_bf16x2(pk[x][2 * u], pk[x][2 * u + 1]);
                    // over the first W/2 of the W S^T columns this thread has just read
                    tmem_st_cols(lane_base + C::T_S + cbase, pw);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(C::B_PFULL));
                if (threadIdx.x == 0) BWD_TRACE(1, n);
                ok = mbar_wait(bar(C::B_DPFULL), n & 1, p.status, 74);
                if (threadIdx.x == 0) BWD_TRACE(2, n);
            }
            ok = __all_sync(0xffffffffu, ok);
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    const int cbase = 64 * x + W * cs;
                    float dp[W];
                    tmem_ld_cols(lane_base + C::T_DP + cbase, dp);
                    tmem_wait_ld();
                    uint32_t dw[W / 2];
#pragma unroll
                    for (int u4 = 0; u4 < W / 4; ++u4) {
                        const float4 d4 = del4[cbase / 4 + u4];
                        const float da[4] = {d4.x, d4.y, d4.z, d4.w};
                        float dv[4];
#pragma unroll
                        for (int w = 0; w < 4; ++w) dv[w] = pk[x][u4 * 4 + w] * (dp[u4 * 4 + w] - da[w]);
                        dw[u4 * 2] = pack_bf16x2(dv[0], dv[1]);
                        dw[u4 * 2 + 1] = pack_bf16x2(dv[2], dv[3]);
                    }
                    // dS^T block x (queries [64x, 64x+64)), this thread's W query columns
#pragma unroll
                    for (int g = 0; g < W / 8; ++g)
                        st_shared_v4(dsa + x * 16384 + sw128_offset(r, (W / 8) * cs + g), dw[4 * g], dw[4 * g + 1],
                                     dw[4 * g + 2], dw[4 * g + 3]);
                }
                mbar_arrive(bar(C::B_LEMPTY + 8 * ls));
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bar(C::B_DSFULL));
                if (threadIdx.x == 0) BWD_TRACE(3, n);
            }
        }
        // ------------------------------ dK, dV ---------------------------------
        if (ok) ok = mbar_wait(bar(C::B_DKVFULL), 0, p.status, 75);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            tc_fence_after();
            for (int which = 0; which < 2; ++which) {   // 0: dK, 1: dV; this warp's EW columns
                const float mul = which == 0 ? p.scale : 1.f;
#pragma unroll
                for (int cc = 0; cc < C::EW / 32; ++cc) {
                    const int col0 = C::EW * cs + 32 * cc;
                    float v[32];
                    tmem_ld32(lane_base + (which == 0 ? C::T_DK : C::T_DV) + col0, v);
                    tmem_wait_ld();
                    if (slot < 0) {
                        uint16_t* out = (which == 0 ? p.dk : p.dv) + ((size_t)j * p.hkv + hk) * D + col0;
                        if (j < p.N) {
#pragma unroll
                            for (int u = 0; u < 32; u += 8) {
                                uint4 w;
                                w.x = pack_bf16x2(v[u] * mul, v[u + 1] * mul);
                                w.y = pack_bf16x2(v[u + 2] * mul, v[u + 3] * mul);
                                w.z = pack_bf16x2(v[u + 4] * mul, v[u + 5] * mul);
                                w.w = pack_bf16x2(v[u + 6] * mul, v[u + 7] * mul);
                                *reinterpret_cast<uint4*>(out + u) = w;
                            }
                        }
                    } else {
                        float* out = p.part + ((((size_t)slot * p.hkv + hk) * 2 + which) * 128 + r) * D + col0;
#pragma unroll
                        for (int u = 0; u < 32; u += 4)
                            *reinterpret_cast<float4*>(out + u) =
                                make_float4(v[u] * mul, v[u + 1] * mul, v[u + 2] * mul, v[u + 3] * mul);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) BWD_TRACE(21, 0);
    if (warp == C::MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int NCW>
cudaError_t launch_fs(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv, const CUtensorMap* tdo,
                      const CUtensorMap* tdq, const BwdParams& p, int grid, cudaStream_t stream) {
    using C = FsCfg<NCW>;
    auto kern = bwd_fs_kernel<NCW>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::BYTES);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(C::NWARPS * 32), C::BYTES, stream, *tq, *tk, *tv, *tdo, *tdq, p);
}

}  // namespace

// 8 compute warps (64 query columns per thread and step) or 16 (32 columns)
#ifndef TREE_ATTN_BWD_NCW
#define TREE_ATTN_BWD_NCW 8
#endif

cudaError_t launch_bwd_fs(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv, const CUtensorMap* tdo,
                          const CUtensorMap* tdq, const BwdParams& p, int grid, cudaStream_t stream) {
    if (grid <= 0) return cudaSuccess;
    return launch_fs<TREE_ATTN_BWD_NCW>(tq, tk, tv, tdo, tdq, p, grid, stream);
}

#ifdef TREE_ATTN_TRACE
extern "C" int tree_attn_bwd_trace_read(void* host, size_t bytes) {
    if (bytes > sizeof(g_bwd_trace)) bytes = sizeof(g_bwd_trace);
    return cudaMemcpyFromSymbol(host, g_bwd_trace, bytes) == cudaSuccess ? 0 : -1;
}
#endif

}  // namespace treeattn
