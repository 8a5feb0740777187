// Backward kernel for head_dim 128: dQ, dK, dV of tree attention on the
// sm_103a tensor cores, with the q-tile split into two 64-query halves that
// ping-pong between the compute warps and the tensor core.
//
// KV-major, as the d = 64 kernel: one CTA = one work item (kv-tile c, a chunk
// [t0, t1) of its contiguous descendant q-range) x one kv-head; K_c, V_c stay
// in shared memory, dV and dK in TMEM; steps (q-tile t ascending, then q-head
// h of the group) run in a fixed order, so dK and dV are bitwise reproducible.
//
// Each step is two half-steps (queries [0,64) and [64,128) of the q-tile).
// TMEM (512 columns): half x owns columns [128x, 128x+128):
//   [128x,    +64)  S^T_x = K Q_x^T            (then P^T_x, packed bf16, in
//                                              the first 32 of them)
//   [128x+64, +64)  dP^T_x = V dO_x^T          (then dQ^T_x = K^T dS^T_x)
//   [256, 384)      dV += P^T_x dO_x           (P^T_x read from TMEM)
//   [384, 512)      dK += dS^T_x Q_x           (dS^T_x from shared memory)
// While the compute warps turn half x into P^T_x and dS^T_x, the tensor core
// runs the other half's MMAs.
//
// dQ^T_x (lane = feature, column = query) leaves TMEM through registers into a
// 32 KB staging tile laid out like the fp32 dQ accumulator [query][feature]
// (128B-swizzled), and reaches the accumulator by TMA bulk reduce-add.  The
// reduce runs asynchronously; the staging tile is reused one half-step later.
//
// Warp roles (448 threads): warps 0-7 compute P^T and dS^T (warp w owns TMEM
// lanes 32*(w%4).. -- one key each -- and 32 of the 64 query columns of a
// half: [32*(w/4), +32)); warps 8-11 read dQ^T out of TMEM (lane = feature, all
// 64 query columns) into the staging tile and issue the TMA reduce, so the
// compute warps never wait for dQ; warp 12 is the TMA producer (K, V once; Q
// and dO per half-step, 64 rows each, through a 6-slot ring so that each half
// releases its own slots; the next tiles prefetched into L2; LSE and Delta rows
// by bulk copy); warp 13 issues the MMAs and owns TMEM.
#include "kernels.h"
#include "ptx.cuh"

namespace treeattn {

namespace {

struct PpCfg {
    static constexpr int D = 128;
    static constexpr int TILE = 128 * D * 2;                  // 32 KB (K, V)
    static constexpr int HTILE = 64 * D * 2;                  // 16 KB (half of a Q or dO tile)
    static constexpr int NSLOT = 6;
    static constexpr int SMALL = 3072;
    static constexpr int OFF_K = SMALL;
    static constexpr int OFF_V = OFF_K + TILE;
    static constexpr int OFF_RING = OFF_V + TILE;
    static constexpr int OFF_DST = OFF_RING + NSLOT * HTILE;  // dS^T: 128 keys x 128 queries bf16 (2 blocks)
    static constexpr int OFF_STAGE = OFF_DST + 32768;         // dQ staging: 64 queries x 128 features fp32
    static constexpr int BYTES = OFF_STAGE + 32768;
    static constexpr int NWARPS = 14;
    static constexpr int NCOMPUTE = 256;                      // warps 0-7
    static constexpr int READOUT0 = 8;                        // warps 8-11
    static constexpr int NREADOUT = 128;
    static constexpr int PRODUCER = 12;
    static constexpr int MMA = 13;
    static constexpr int TMEM_COLS = 512;
    static constexpr int T_DV = 256, T_DK = 384;
    // small region
    static constexpr int B_KVFULL = 0;
    static constexpr int B_FULL = 8;                      // [NSLOT]
    static constexpr int B_EMPTY = B_FULL + 8 * NSLOT;    // [NSLOT]
    static constexpr int B_LFULL = B_EMPTY + 8 * NSLOT;   // [2]
    static constexpr int B_LEMPTY = B_LFULL + 16;         // [2]
    static constexpr int B_SDP = B_LEMPTY + 16;           // [2] S^T_x and dP^T_x ready
    static constexpr int B_PFULL = B_SDP + 16;            // [2] P^T_x, dS^T_x written
    static constexpr int B_DQFULL = B_PFULL + 16;         // [2] dQ^T_x ready
    static constexpr int B_DQEMPTY = B_DQFULL + 16;       // [2] dQ^T_x read out
    static constexpr int B_DKVFULL = B_DQEMPTY + 16;
    static constexpr int B_DRAIN = B_DKVFULL + 8;
    static constexpr int HOLDER = B_DRAIN + 8;
    static constexpr int LSD = 1024;                      // 2 stages x {lse2[128], delta[128]}
    static_assert(HOLDER + 4 <= LSD, "barriers");
    static_assert(LSD + 2 * 1024 <= SMALL, "small region");
    static_assert(BYTES <= 232448, "shared memory");
};

__global__ void __launch_bounds__(PpCfg::NWARPS * 32, 1)
    bwd_pp_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_dq64, const __grid_constant__ CUtensorMap tm_q64,
                  const __grid_constant__ CUtensorMap tm_do64, const BwdParams p) {
    using C = PpCfg;
    constexpr int D = C::D;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (sb & 1023u) {
        if (threadIdx.x == 0) report_status(p.status, -5);
        return;
    }
    const int item = blockIdx.x / p.hkv;
    const int hk = blockIdx.x % p.hkv;
    const int4 it = reinterpret_cast<const int4*>(p.items)[item];
    const int c = it.x, t0 = it.y, t1 = it.z, slot = it.w;
    const int G = p.group;
    const int nsteps = (t1 - t0) * G;

    auto bar = [&](int off) { return sb + (uint32_t)off; };
    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_KVFULL), 1);
        for (int s = 0; s < C::NSLOT; ++s) {
            mbar_init(bar(C::B_FULL + 8 * s), 1);
            mbar_init(bar(C::B_EMPTY + 8 * s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(C::B_LFULL + 8 * s), 1);
            mbar_init(bar(C::B_LEMPTY + 8 * s), C::NCOMPUTE);
            mbar_init(bar(C::B_SDP + 8 * s), 1);
            mbar_init(bar(C::B_PFULL + 8 * s), C::NCOMPUTE);
            mbar_init(bar(C::B_DQFULL + 8 * s), 1);
            mbar_init(bar(C::B_DQEMPTY + 8 * s), C::NREADOUT);
        }
        mbar_init(bar(C::B_DKVFULL), 1);
        mbar_init(bar(C::B_DRAIN), 1);
        fence_mbar_init();
    }
    if (warp == C::MMA) tmem_alloc(sb + C::HOLDER, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::HOLDER);

    // ring position of step n, half x: Q (w = 0) or dO (w = 1), 64 rows each
    auto ring_pos = [](int n, int x, int w) { return 4 * n + 2 * x + w; };

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
                for (int x = 0; x < 2 && ok; ++x) {
                    for (int w = 0; w < 2 && ok; ++w) {   // w = 0: Q, 1: dO
                        const int pos = ring_pos(n, x, w), s = pos % C::NSLOT, use = pos / C::NSLOT;
                        if (use > 0) ok = mbar_wait(bar(C::B_EMPTY + 8 * s), (use - 1) & 1, p.status, 41);
                        if (!ok) break;
                        mbar_expect_tx(bar(C::B_FULL + 8 * s), C::HTILE);
                        for (int blk = 0; blk < D / 64; ++blk)
                            tma_load_3d(sb + C::OFF_RING + s * C::HTILE + blk * 8192, w ? &tm_do64 : &tm_q64,
                                        blk * 64, h, t * 128 + 64 * x, bar(C::B_FULL + 8 * s));
                        if (x == 0 && w == 0) {
                            const int ls = n & 1, luse = n >> 1;
                            if (luse > 0) ok = mbar_wait(bar(C::B_LEMPTY + 8 * ls), (luse - 1) & 1, p.status, 42);
                            if (!ok) break;
                            mbar_expect_tx(bar(C::B_LFULL + 8 * ls), 1024);
                            const size_t off = (size_t)h * p.Npad + (size_t)t * 128;
                            bulk_load(sb + C::LSD + ls * 1024, p.lse2 + off, 512, bar(C::B_LFULL + 8 * ls));
                            bulk_load(sb + C::LSD + ls * 1024 + 512, p.delta + off, 512, bar(C::B_LFULL + 8 * ls));
                        }
                    }
                }
            }
        }
    } else if (warp == C::MMA) {
        if (lane == 0) {
            constexpr uint32_t ID_SDP = idesc_bf16(128, 64, false, false);  // K Q_x^T, V dO_x^T
            constexpr uint32_t ID_DQT = idesc_bf16(128, 64, true, true);    // K^T dS^T_x
            constexpr uint32_t ID_KV = idesc_bf16(128, 128, false, true);   // dS^T_x Q_x, P^T_x dO_x
            const uint32_t ka = sb + C::OFF_K, va = sb + C::OFF_V, dsa = sb + C::OFF_DST;
            auto slot_addr = [&](int n, int x, int w) {
                return sb + C::OFF_RING + (ring_pos(n, x, w) % C::NSLOT) * C::HTILE;
            };
            auto wait_full = [&](int n, int x, int w, int where) {
                const int pos = ring_pos(n, x, w);
                return mbar_wait(bar(C::B_FULL + 8 * (pos % C::NSLOT)), (pos / C::NSLOT) & 1, p.status, where);
            };
            // S^T_x = K Q_x^T  (N = 64 queries; a half tile holds two 8 KB feature blocks)
            auto issue_s = [&](int n, int x) {
                const uint32_t qa = slot_addr(n, x, 0);
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
                    mma_bf16_ss(tmem + 128 * x, sdesc_sw128(ka + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024),
                                sdesc_sw128(qa + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024), ID_SDP, k > 0);
            };
            auto issue_dp = [&](int n, int x) {
                const uint32_t doa = slot_addr(n, x, 1);
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
                    mma_bf16_ss(tmem + 128 * x + 64, sdesc_sw128(va + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024),
                                sdesc_sw128(doa + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024), ID_SDP, k > 0);
                mma_commit(bar(C::B_SDP + 8 * x));
            };
            bool ok = mbar_wait(bar(C::B_KVFULL), 0, p.status, 43);
            for (int x = 0; x < 2 && ok; ++x) {
                ok = wait_full(0, x, 0, 44);
                if (ok) ok = wait_full(0, x, 1, 45);
                if (!ok) break;
                tc_fence_after();
                issue_s(0, x);
                issue_dp(0, x);
            }
            for (int n = 0; n < nsteps && ok; ++n) {
                for (int x = 0; x < 2 && ok; ++x) {
                    ok = mbar_wait(bar(C::B_PFULL + 8 * x), n & 1, p.status, 46);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t qa = slot_addr(n, x, 0), doa = slot_addr(n, x, 1);
                    // dQ^T_x = K^T dS^T_x   (M = 128 features, N = 64 queries, K = 128 keys)
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mma_bf16_ss(tmem + 128 * x + 64, sdesc_sw128(ka + k * 2048, 16384, 1024),
                                    sdesc_sw128(dsa + x * 16384 + k * 2048, 16384, 1024), ID_DQT, k > 0);
                    mma_commit(bar(C::B_DQFULL + 8 * x));
                    // dK += dS^T_x Q_x ; dV += P^T_x dO_x   (K dimension = 64 queries)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_bf16_ss(tmem + C::T_DK, sdesc_sw128(dsa + x * 16384 + k * 32, 16, 1024),
                                    sdesc_sw128(qa + k * 2048, 8192, 1024), ID_KV, (n > 0 || x > 0 || k > 0) ? 1u : 0u);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_bf16_ts(tmem + C::T_DV, tmem + 128 * x + 8 * k, sdesc_sw128(doa + k * 2048, 8192, 1024),
                                    ID_KV, (n > 0 || x > 0 || k > 0) ? 1u : 0u);
                    mma_commit(bar(C::B_EMPTY + 8 * (ring_pos(n, x, 0) % C::NSLOT)));
                    mma_commit(bar(C::B_EMPTY + 8 * (ring_pos(n, x, 1) % C::NSLOT)));
                    if (n + 1 < nsteps) {
                        ok = wait_full(n + 1, x, 0, 44);
                        if (ok) ok = wait_full(n + 1, x, 1, 45);
                        if (!ok) break;
                        tc_fence_after();
                        issue_s(n + 1, x);   // over P^T_x: after dV_x in issue order
                        ok = mbar_wait(bar(C::B_DQEMPTY + 8 * x), n & 1, p.status, 47);
                        if (!ok) break;
                        tc_fence_after();
                        issue_dp(n + 1, x);  // over dQ^T_x, which has been read out
                    }
                }
            }
            if (ok) mma_commit(bar(C::B_DKVFULL));
            mma_commit(bar(C::B_DRAIN));
            mbar_wait(bar(C::B_DRAIN), 0, p.status, 48);
        }
        __syncwarp();
    } else if (warp >= C::READOUT0) {
        // ------------------------------ dQ readout ------------------------------
        const int quarter = warp & 3;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter << 5) << 16);   // lane = feature
        const uint32_t stage = sb + C::OFF_STAGE;
        const int rtid = threadIdx.x - C::READOUT0 * 32;                        // 0..127
        bool ok = true;
        // loops run to the end after a failed wait (work skipped), so the named
        // barriers of this warpgroup always line up
        for (int n = 0; n < nsteps; ++n) {
            const int t = t0 + n / G, h = hk * G + n % G;
            const int q0 = t * 128;
            for (int x = 0; x < 2; ++x) {
                if (ok) ok = mbar_wait(bar(C::B_DQFULL + 8 * x), n & 1, p.status, 51);
                ok = __all_sync(0xffffffffu, ok);
                float v[64];
                if (ok) {
                    tc_fence_after();
                    tmem_ld32(lane_base + 128 * x + 64, *reinterpret_cast<float(*)[32]>(&v[0]));
                    tmem_ld32(lane_base + 128 * x + 96, *reinterpret_cast<float(*)[32]>(&v[32]));
                    tmem_wait_ld();
                    tc_fence_before();
                    mbar_arrive(bar(C::B_DQEMPTY + 8 * x));   // dQ^T_x has left TMEM
                }
                // the previous reduce has finished reading the staging tile
                if (rtid == 0) bulk_wait_read_all();
                ok = named_bar_and(2, C::NREADOUT, ok);
                if (ok) {
                    // staging [64 queries][128 features] fp32: 4 blocks of 32 features x 64 rows
                    const uint32_t blk = stage + (uint32_t)quarter * 8192 + ((lane & 3) << 2);
#pragma unroll
                    for (int u = 0; u < 64; ++u)
                        st_shared_f32(blk + u * 128 + ((((uint32_t)lane >> 2) ^ ((uint32_t)u & 7u)) << 4),
                                      v[u] * p.scale);
                }
                fence_proxy_async_smem();
                ok = named_bar_and(2, C::NREADOUT, ok);
                if (ok && rtid == 0) {
                    for (int b = 0; b < 4; ++b) tma_reduce_add_3d(&tm_dq64, stage + b * 8192, b * 32, h, q0 + 64 * x);
                    bulk_commit();
                }
            }
        }
        if (rtid == 0) bulk_wait_all();
    } else {
        // ------------------------------ compute -------------------------------
        const int quarter = warp & 3, ch = warp >> 2;  // TMEM lane quarter, column half of a half-step
        const int r = (quarter << 5) + lane;           // TMEM lane: key (S^T, dP^T) or feature (dQ^T)
        const uint32_t lane_base = tmem + ((uint32_t)(quarter << 5) << 16);
        const int j = c * 128 + r;                     // this thread's key
        const int sub_j = p.subend[j];                 // 0 past N
        const float sl2 = p.scale_log2;
        const uint32_t dsa = sb + C::OFF_DST;
        bool ok = true;
        // After a failed wait the loops keep running with the work skipped, so all
        // compute threads meet the named barriers of every half-step.
        for (int n = 0; n < nsteps; ++n) {
            const int t = t0 + n / G, h = hk * G + n % G;
            const int q0 = t * 128;
            const int lo = max(j - q0, 0), hi = min(sub_j - q0, 128);
            const int ls = n & 1;
            if (ok) ok = mbar_wait(bar(C::B_LFULL + 8 * ls), (n >> 1) & 1, p.status, 49);
            const float4* lse4 = reinterpret_cast<const float4*>(smem + C::LSD + ls * 1024);
            const float4* del4 = reinterpret_cast<const float4*>(smem + C::LSD + ls * 1024 + 512);
            for (int x = 0; x < 2; ++x) {
                const int cbase = 64 * x + 32 * ch;     // this thread's first query column in the step
                if (ok) ok = mbar_wait(bar(C::B_SDP + 8 * x), n & 1, p.status, 50);
                ok = __all_sync(0xffffffffu, ok);
                float pk[32];      // P^T for this thread's 32 query columns (fp32, for dS)
                uint32_t pw[16];   // the same, packed bf16 (for TMEM and the dV MMA)
                if (ok) {
                    tc_fence_after();
                    float sv[32];
                    tmem_ld32(lane_base + 128 * x + 32 * ch, sv);
                    tmem_wait_ld();
                    if (lo <= cbase && hi >= cbase + 32) {   // every column of this row attends
#pragma unroll
                        for (int u4 = 0; u4 < 8; ++u4) {
                            const float4 l4 = lse4[cbase / 4 + u4];
                            pk[u4 * 4 + 0] = fast_exp2(fmaf(sv[u4 * 4 + 0], sl2, -l4.x));
                            pk[u4 * 4 + 1] = fast_exp2(fmaf(sv[u4 * 4 + 1], sl2, -l4.y));
                            pk[u4 * 4 + 2] = fast_exp2(fmaf(sv[u4 * 4 + 2], sl2, -l4.z));
                            pk[u4 * 4 + 3] = fast_exp2(fmaf(sv[u4 * 4 + 3], sl2, -l4.w));
                        }
                    } else {
#pragma unroll
                        for (int u4 = 0; u4 < 8; ++u4) {
                            const float4 l4 = lse4[cbase / 4 + u4];
                            const float la[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                            for (int w = 0; w < 4; ++w) {
                                const int col = cbase + u4 * 4 + w;
                                const float e = fast_exp2(fmaf(sv[u4 * 4 + w], sl2, -la[w]));
                                pk[u4 * 4 + w] = (col >= lo && col < hi) ? e : 0.f;
                            }
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 16; ++u) pw[u] = pack_bf16x2(pk[2 * u], pk[2 * u + 1]);
                    tc_fence_before();
                }
                // every thread has read its S^T_x columns before P^T_x overwrites them
                ok = named_bar_and(1, C::NCOMPUTE, ok);
                if (ok) {
                    tc_fence_after();
                    tmem_st16(lane_base + 128 * x + 16 * ch, pw);
                    float dp[32];
                    tmem_ld32(lane_base + 128 * x + 64 + 32 * ch, dp);
                    tmem_wait_ld();
                    uint32_t dw[16];
#pragma unroll
                    for (int u4 = 0; u4 < 8; ++u4) {
                        const float4 d4 = del4[cbase / 4 + u4];
                        const float da[4] = {d4.x, d4.y, d4.z, d4.w};
                        float dv[4];
#pragma unroll
                        for (int w = 0; w < 4; ++w) dv[w] = pk[u4 * 4 + w] * (dp[u4 * 4 + w] - da[w]);
                        dw[u4 * 2] = pack_bf16x2(dv[0], dv[1]);
                        dw[u4 * 2 + 1] = pack_bf16x2(dv[2], dv[3]);
                    }
                    // dS^T_x: block x of the dS^T tile, this thread's 32 query columns
#pragma unroll
                    for (int g = 0; g < 4; ++g)
                        st_shared_v4(dsa + x * 16384 + sw128_offset(r, 4 * ch + g), dw[4 * g], dw[4 * g + 1],
                                     dw[4 * g + 2], dw[4 * g + 3]);
                    if (x == 1) mbar_arrive(bar(C::B_LEMPTY + 8 * ls));
                    tmem_wait_st();
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(bar(C::B_PFULL + 8 * x));
                }
            }
        }
        // ------------------------------ dK, dV ---------------------------------
        if (ok) ok = mbar_wait(bar(C::B_DKVFULL), 0, p.status, 52);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            tc_fence_after();
            for (int which = 0; which < 2; ++which) {   // 0: dK, 1: dV
                const uint32_t tcol = which == 0 ? C::T_DK : C::T_DV;
                const float mul = which == 0 ? p.scale : 1.f;
                if (slot < 0) {
                    uint16_t* out = (which == 0 ? p.dk : p.dv) + ((size_t)j * p.hkv + hk) * D;
#pragma unroll
                    for (int cc = ch * 2; cc < ch * 2 + 2; ++cc) {
                        float v[32];
                        tmem_ld32(lane_base + tcol + cc * 32, v);
                        tmem_wait_ld();
                        if (j < p.N) {
#pragma unroll
                            for (int u = 0; u < 32; u += 8) {
                                uint4 w;
                                w.x = pack_bf16x2(v[u] * mul, v[u + 1] * mul);
                                w.y = pack_bf16x2(v[u + 2] * mul, v[u + 3] * mul);
                                w.z = pack_bf16x2(v[u + 4] * mul, v[u + 5] * mul);
                                w.w = pack_bf16x2(v[u + 6] * mul, v[u + 7] * mul);
                                *reinterpret_cast<uint4*>(out + cc * 32 + u) = w;
                            }
                        }
                    }
                } else {
                    float* out = p.part + ((((size_t)slot * p.hkv + hk) * 2 + which) * 128 + r) * D;
#pragma unroll
                    for (int cc = ch * 2; cc < ch * 2 + 2; ++cc) {
                        float v[32];
                        tmem_ld32(lane_base + tcol + cc * 32, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int u = 0; u < 32; u += 4)
                            *reinterpret_cast<float4*>(out + cc * 32 + u) =
                                make_float4(v[u] * mul, v[u + 1] * mul, v[u + 2] * mul, v[u + 3] * mul);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == C::MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace

cudaError_t launch_bwd_pp(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                          const CUtensorMap* tdo, const CUtensorMap* tdq64, const CUtensorMap* tq64,
                          const CUtensorMap* tdo64, const BwdParams& p, int grid, cudaStream_t stream) {
    if (grid <= 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(bwd_pp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PpCfg::BYTES);
    if (e != cudaSuccess) return e;
    bwd_pp_kernel<<<grid, PpCfg::NWARPS * 32, PpCfg::BYTES, stream>>>(*tq, *tk, *tv, *tdo, *tdq64, *tq64, *tdo64,
                                                                      p);
    return cudaGetLastError();
}

}  // namespace treeattn
