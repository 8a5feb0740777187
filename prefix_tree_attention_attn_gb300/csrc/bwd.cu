// Backward kernel for head_dim 64: dQ, dK, dV of tree attention on the sm_103a
// tensor cores (head_dim 128 has its own kernel, bwd_fs.cu).
//
// KV-major.  A work unit is one item (kv-tile c, a chunk [t0, t1) of its
// contiguous descendant q-range) x one kv-head; the kernel is persistent, each
// CTA taking work units w = blockIdx.x, blockIdx.x + gridDim.x, ... in order.
// For a unit the CTA keeps K_c and V_c in shared memory and dV, dK in TMEM, and
// walks every step (q-tile t, q-head h of the group) in a fixed order -- t
// ascending, then h ascending -- so dK and dV are summed in the same order on
// every run.  Per step n:
//
//   S^T  = K Q^T                TMEM cols [0,128)
//   dP^T = V dO^T               TMEM cols [128,256)
//   P^T  = exp2(S^T*scale*log2e - LSE*log2e), masked j <= i < subend[j];
//          written back over S^T as packed bf16 (TMEM cols [0,64))
//   dS^T = P^T * (dP^T - Delta) shared memory, bf16, K-major 128B-swizzled
//          (P^T here is the bf16-rounded value that also feeds dV)
//   dQ   = dS K                 TMEM cols [128,192) (over dP^T), issued first
//   dK  += dS^T Q               TMEM cols [320, 384)
//   dV  += P^T dO               TMEM cols [256, 320), P^T read from TMEM
//   S^T(n+1)                    issued right after, overlapping the dQ readout
//   dP^T(n+1)                   once dQ(n) has left TMEM
//
// Steps are counted across the units of a CTA, so step n+1 may be the first
// step of the next unit: its K and V sit in the other of two K/V buffers
// (loaded while the current unit runs), its S^T and dP^T run while the compute
// warps store the finished unit's dK and dV, and its first dK / dV products
// (which overwrite the accumulators) come after that store in the compute
// warps' own order.  With the tiny trees this kernel serves (items of one or
// two steps), this hides most of a unit's set-up.
//
// dQ leaves TMEM through registers into a 32 KB shared staging tile (fp32,
// 128B-swizzled) and reaches the fp32 dQ accumulator by TMA bulk reduce-add
// while the tensor core runs dK and dV.
//
// Warp roles (320 threads): warps 0-7 compute (warp w owns TMEM lanes
// 32*(w%4).. and query / dQ columns of half w/4); warp 8 is the TMA producer
// (K, V per unit into two buffers; Q and dO per step through a 4-slot ring,
// the next tiles prefetched into L2; LSE and Delta rows by bulk copy); warp 9
// issues the MMAs and owns TMEM.
#include "kernels.h"
#include "ptx.cuh"

namespace treeattn {

namespace {

struct BwdCfg {
    static constexpr int D = 64;
    static constexpr int TILE = 128 * D * 2;
    static constexpr int NSLOT = 4;
    static constexpr int NKV = 2;                             // K/V buffers
    static constexpr int SMALL = 3072;
    static constexpr int OFF_KV = SMALL;                      // buffer b: K at OFF_KV + 2b TILE, V after it
    static constexpr int OFF_RING = OFF_KV + NKV * 2 * TILE;
    static constexpr int OFF_DST = OFF_RING + NSLOT * TILE;   // dS^T, 128 x 128 bf16
    static constexpr int OFF_STAGE = OFF_DST + 32768;         // dQ staging, 128 x 64 fp32
    static constexpr int BYTES = OFF_STAGE + 32768;
    static constexpr int NWARPS = 10;
    static constexpr int NCOMPUTE = 256;                      // warps 0-7
    static constexpr int PRODUCER = 8;
    static constexpr int MMA = 9;
    static constexpr int TMEM_COLS = 512;
    static constexpr int T_S = 0, T_P = 0, T_DP = 128, T_DQ = 128, T_DV = 256, T_DK = 256 + D;
    // small region
    static constexpr int B_KVFULL = 0;                    // [NKV]
    static constexpr int B_KVEMPTY = B_KVFULL + 8 * NKV;  // [NKV]
    static constexpr int B_FULL = B_KVEMPTY + 8 * NKV;    // [NSLOT]
    static constexpr int B_EMPTY = B_FULL + 8 * NSLOT;    // [NSLOT]
    static constexpr int B_LFULL = B_EMPTY + 8 * NSLOT;   // [2]
    static constexpr int B_LEMPTY = B_LFULL + 16;         // [2]
    static constexpr int B_SFULL = B_LEMPTY + 16;
    static constexpr int B_DPFULL = B_SFULL + 8;
    static constexpr int B_PFULL = B_DPFULL + 8;
    static constexpr int B_DQFULL = B_PFULL + 8;
    static constexpr int B_DQEMPTY = B_DQFULL + 8;
    static constexpr int B_DKVFULL = B_DQEMPTY + 8;
    static constexpr int B_DRAIN = B_DKVFULL + 8;
    static constexpr int HOLDER = B_DRAIN + 8;
    static constexpr int LSD = 1024;   // 2 stages x {lse2[128], delta[128]} fp32
    static_assert(HOLDER + 4 <= LSD, "barriers");
    static_assert(LSD + 2 * 1024 <= SMALL, "small region");
    static_assert(BYTES <= 232448, "shared memory");
};

// The work unit w of the launch (item, kv-head, the item's fields) and whether
// it lies inside the plan (debug builds check; a uniform decision, taken the
// same way by every role).
struct Unit {
    int item, hk, c, t0, t1, slot;
};

__device__ __forceinline__ bool unit_of(const BwdParams& p, int w, Unit& u) {
    bwd_cta_work(p, w, u.item, u.hk);
    if (u.item < 0) return false;
    const int4 it = reinterpret_cast<const int4*>(p.items)[u.item];
    u.c = it.x;
    u.t0 = it.y;
    u.t1 = it.z;
    u.slot = it.w;
    return ta_ok(p.status, 231, u.c, 0, p.T) && ta_ok(p.status, 232, u.t0, u.c, p.T) &&
           ta_ok(p.status, 233, u.t1, u.t0 + 1, (long long)p.T + 1) && ta_ok(p.status, 234, u.slot, -1, p.n_slots) &&
           ta_ok(p.status, 235, u.hk, 0, p.hkv);
}

__global__ void __launch_bounds__(BwdCfg::NWARPS * 32, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
    using C = BwdCfg;
    constexpr int D = C::D;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (sb & 1023u) {
        if (threadIdx.x == 0) report_status(p.status, -5);
        return;
    }
    const int G = p.group;
    const int n_work = p.n_items * p.hkv;

    auto bar = [&](int off) { return sb + (uint32_t)off; };
    if (threadIdx.x == 0) {
        for (int b = 0; b < C::NKV; ++b) {
            mbar_init(bar(C::B_KVFULL + 8 * b), 1);
            mbar_init(bar(C::B_KVEMPTY + 8 * b), 1);
        }
        for (int s = 0; s < C::NSLOT; ++s) {
            mbar_init(bar(C::B_FULL + 8 * s), 1);
            mbar_init(bar(C::B_EMPTY + 8 * s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(C::B_LFULL + 8 * s), 1);
            mbar_init(bar(C::B_LEMPTY + 8 * s), C::NCOMPUTE);
        }
        mbar_init(bar(C::B_SFULL), 1);
        mbar_init(bar(C::B_DPFULL), 1);
        mbar_init(bar(C::B_PFULL), C::NCOMPUTE);
        mbar_init(bar(C::B_DQFULL), 1);
        mbar_init(bar(C::B_DQEMPTY), C::NCOMPUTE);
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

    // ring position of (CTA-wide) step g's Q (x = 0) or dO (x = 1)
    auto ring_pos = [](int g, int x) { return 2 * g + x; };
    auto k_of = [&](int kb) { return sb + C::OFF_KV + kb * 2 * C::TILE; };
    auto v_of = [&](int kb) { return k_of(kb) + C::TILE; };

    if (warp == C::PRODUCER) {
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_do);
            bool ok = true;
            int ic = 0, gs = 0;   // units and steps of this CTA so far
            for (int w = blockIdx.x; w < n_work && ok; w += gridDim.x) {
                Unit u;
                if (!unit_of(p, w, u)) continue;
                const int nsteps = (u.t1 - u.t0) * G;
                const int kb = ic % C::NKV, kuse = ic / C::NKV;
                if (kuse > 0) ok = mbar_wait(bar(C::B_KVEMPTY + 8 * kb), (kuse - 1) & 1, p.status, 20);
                if (!ok) break;
                mbar_expect_tx(bar(C::B_KVFULL + 8 * kb), 2 * C::TILE);
                tma_load_3d(k_of(kb), &tm_k, 0, u.hk, u.c * 128, bar(C::B_KVFULL + 8 * kb));
                tma_load_3d(v_of(kb), &tm_v, 0, u.hk, u.c * 128, bar(C::B_KVFULL + 8 * kb));
                auto prefetch = [&](int n) {
                    if (n >= nsteps) return;
                    const int t = u.t0 + n / G, h = u.hk * G + n % G;
                    tma_prefetch_3d(&tm_q, 0, h, t * 128);
                    tma_prefetch_3d(&tm_do, 0, h, t * 128);
                };
                prefetch(1);
                for (int n = 0; n < nsteps && ok; ++n) {
                    const int g = gs + n;
                    const int t = u.t0 + n / G, h = u.hk * G + n % G;
                    prefetch(n + 2);
                    for (int x = 0; x < 2 && ok; ++x) {   // x = 0: Q, 1: dO
                        const int pos = ring_pos(g, x), s = pos % C::NSLOT, use = pos / C::NSLOT;
                        if (use > 0) ok = mbar_wait(bar(C::B_EMPTY + 8 * s), (use - 1) & 1, p.status, 21);
                        if (!ok) break;
                        mbar_expect_tx(bar(C::B_FULL + 8 * s), C::TILE);
                        tma_load_3d(sb + C::OFF_RING + s * C::TILE, x ? &tm_do : &tm_q, 0, h, t * 128,
                                    bar(C::B_FULL + 8 * s));
                        if (x == 0) {
                            const int ls = g & 1, luse = g >> 1;
                            if (luse > 0) ok = mbar_wait(bar(C::B_LEMPTY + 8 * ls), (luse - 1) & 1, p.status, 22);
                            if (!ok) break;
                            mbar_expect_tx(bar(C::B_LFULL + 8 * ls), 1024);
                            const size_t off = (size_t)ta_clamp(p.status, 236, (long long)h * p.Npad + (long long)t * 128,
                                                                0, (long long)p.hq * p.Npad - 127);
                            bulk_load(sb + C::LSD + ls * 1024, p.lse2 + off, 512, bar(C::B_LFULL + 8 * ls));
                            bulk_load(sb + C::LSD + ls * 1024 + 512, p.delta + off, 512, bar(C::B_LFULL + 8 * ls));
                        }
                    }
                }
                ++ic;
                gs += nsteps;
            }
        }
    } else if (warp == C::MMA) {
        if (lane == 0) {
            constexpr uint32_t ID_S = idesc_bf16(128, 128, false, false);   // K Q^T, V dO^T
            constexpr uint32_t ID_DV = idesc_bf16(128, D, false, true);     // P^T (TMEM) dO
            constexpr uint32_t ID_DK = idesc_bf16(128, D, false, true);     // dS^T Q
            constexpr uint32_t ID_DQ = idesc_bf16(128, D, true, true);      // dS K
            const uint32_t dsa = sb + C::OFF_DST;
            auto slot_of = [&](int g, int x) { return ring_pos(g, x) % C::NSLOT; };
            auto wait_full = [&](int g, int x, int where) {
                const int pos = ring_pos(g, x);
                return mbar_wait(bar(C::B_FULL + 8 * (pos % C::NSLOT)), (pos / C::NSLOT) & 1, p.status, where);
            };
            auto issue_s = [&](int g, uint32_t ka) {   // S^T = K Q_g^T
                const uint32_t qa = sb + C::OFF_RING + slot_of(g, 0) * C::TILE;
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
                    mma_bf16_ss(tmem + C::T_S, sdesc_sw128(ka + k * 32, 16, 1024), sdesc_sw128(qa + k * 32, 16, 1024),
                                ID_S, k > 0);
                mma_commit(bar(C::B_SFULL));
            };
            auto issue_dp = [&](int g, uint32_t va) {   // dP^T = V dO_g^T
                const uint32_t doa = sb + C::OFF_RING + slot_of(g, 1) * C::TILE;
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
                    mma_bf16_ss(tmem + C::T_DP, sdesc_sw128(va + k * 32, 16, 1024), sdesc_sw128(doa + k * 32, 16, 1024),
                                ID_S, k > 0);
                mma_commit(bar(C::B_DPFULL));
            };
            bool ok = true;
            int ic = 0, gs = 0;
            for (int w = blockIdx.x; w < n_work && ok; w += gridDim.x) {
                Unit u;
                if (!unit_of(p, w, u)) continue;
                const int nsteps = (u.t1 - u.t0) * G;
                const int kb = ic % C::NKV;
                const uint32_t ka = k_of(kb), va = v_of(kb);
                // the unit's first S^T and dP^T; S^T goes over the previous step's P^T,
                // whose dV product was issued before, and dP^T over its dQ, which must
                // have left TMEM
                ok = mbar_wait(bar(C::B_KVFULL + 8 * kb), (ic / C::NKV) & 1, p.status, 23);
                if (ok) ok = wait_full(gs, 0, 24);
                if (ok) {
                    tc_fence_after();
                    issue_s(gs, ka);
                    ok = wait_full(gs, 1, 25);
                }
                if (ok && gs > 0) ok = mbar_wait(bar(C::B_DQEMPTY), (gs - 1) & 1, p.status, 26);
                if (ok) {
                    tc_fence_after();
                    issue_dp(gs, va);
                }
                for (int n = 0; n < nsteps && ok; ++n) {
                    const int g = gs + n;
                    ok = mbar_wait(bar(C::B_PFULL), g & 1, p.status, 27);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t qa = sb + C::OFF_RING + slot_of(g, 0) * C::TILE;
                    const uint32_t doa = sb + C::OFF_RING + slot_of(g, 1) * C::TILE;
                    // dQ = dS K   (M = queries: A is dS^T read MN-major; K dimension = 128 keys)
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mma_bf16_ss(tmem + C::T_DQ, sdesc_sw128(dsa + k * 2048, 16384, 1024),
                                    sdesc_sw128(ka + k * 2048, 16384, 1024), ID_DQ, k > 0);
                    mma_commit(bar(C::B_DQFULL));
                    // dK += dS^T Q   (K dimension = 128 queries); the unit's first step
                    // overwrites the accumulators, after the compute warps have stored
                    // the previous unit's (they arrived on P_FULL after that store)
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t aoff = (k >> 2) * 16384 + (k & 3) * 32;
                        mma_bf16_ss(tmem + C::T_DK, sdesc_sw128(dsa + aoff, 16, 1024),
                                    sdesc_sw128(qa + k * 2048, 16384, 1024), ID_DK, (n > 0 || k > 0) ? 1u : 0u);
                    }
                    mma_commit(bar(C::B_EMPTY + 8 * slot_of(g, 0)));
                    // dV += P^T dO   (P^T from TMEM: 8 packed columns per 16 queries)
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mma_bf16_ts(tmem + C::T_DV, tmem + C::T_P + k * 8, sdesc_sw128(doa + k * 2048, 16384, 1024),
                                    ID_DV, (n > 0 || k > 0) ? 1u : 0u);
                    mma_commit(bar(C::B_EMPTY + 8 * slot_of(g, 1)));
                    if (n + 1 < nsteps) {
                        ok = wait_full(g + 1, 0, 24);
                        if (!ok) break;
                        tc_fence_after();
                        issue_s(g + 1, ka);
                        ok = wait_full(g + 1, 1, 25);
                        if (ok) ok = mbar_wait(bar(C::B_DQEMPTY), g & 1, p.status, 26);
                        if (!ok) break;
                        tc_fence_after();
                        issue_dp(g + 1, va);
                    }
                }
                if (!ok) break;
                mma_commit(bar(C::B_KVEMPTY + 8 * kb));   // K, V of this unit no longer read
                mma_commit(bar(C::B_DKVFULL));            // dK, dV of this unit complete
                ++ic;
                gs += nsteps;
            }
            mma_commit(bar(C::B_DRAIN));
            mbar_wait(bar(C::B_DRAIN), 0, p.status, 28);
        }
        __syncwarp();
    } else {
        // --------------------- P^T / dS^T, then dQ readout ---------------------
        const int quarter = warp & 3, half = warp >> 2;
        const int r = (quarter << 5) + lane;          // TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(quarter << 5) << 16);
        const float sl2 = p.scale_log2;
        const uint32_t dsa = sb + C::OFF_DST;
        const uint32_t stage = sb + C::OFF_STAGE;
        bool ok = true;
        int ic = 0, gs = 0;
        // After a failed wait the loops keep running with the work skipped, so all
        // compute threads meet the named barriers of every step.
        for (int w = blockIdx.x; w < n_work; w += gridDim.x) {
            Unit u;
            if (!unit_of(p, w, u)) continue;
            const int nsteps = (u.t1 - u.t0) * G;
            const int j = u.c * 128 + r;   // this thread's key
            const int sub_j = p.subend[ta_clamp(p.status, 237, j, 0, (long long)p.T * 128)];   // 0 past N
            for (int n = 0; n < nsteps; ++n) {
                const int g = gs + n;
                const int t = u.t0 + n / G, h = u.hk * G + n % G;
                const int q0 = t * 128;
                const int lo = max(j - q0, 0), hi = min(sub_j - q0, 128);
                const int ls = g & 1;
                if (ok) ok = mbar_wait(bar(C::B_LFULL + 8 * ls), (g >> 1) & 1, p.status, 29);
                if (ok) ok = mbar_wait(bar(C::B_SFULL), g & 1, p.status, 30);
                ok = __all_sync(0xffffffffu, ok);
                const float4* lse4 = reinterpret_cast<const float4*>(smem + C::LSD + ls * 1024);
                const float4* del4 = reinterpret_cast<const float4*>(smem + C::LSD + ls * 1024 + 512);
                // P^T for this thread's 64 query columns, kept in registers as the packed
                // bf16 pairs that also feed the dV MMA (dS below uses the same values)
                uint32_t pw[2][16];
                if (ok) {
                    tc_fence_after();
#pragma unroll
                    for (int cq = 0; cq < 2; ++cq) {
                        const int cc = half * 2 + cq;
                        float sv[32];
                        tmem_ld32(lane_base + C::T_S + cc * 32, sv);
                        tmem_wait_ld();
#pragma unroll
                        for (int u4 = 0; u4 < 8; ++u4) {
                            const float4 l4 = lse4[cc * 8 + u4];
                            const float la[4] = {l4.x, l4.y, l4.z, l4.w};
                            float pe[4];
#pragma unroll
                            for (int x = 0; x < 4; ++x) {
                                const int col = cc * 32 + u4 * 4 + x;
                                const float e = fast_exp2(fmaf(sv[u4 * 4 + x], sl2, -la[x]));
                                pe[x] = (col >= lo && col < hi) ? e : 0.f;
                            }
                            pw[cq][u4 * 2] = pack_bf16x2(pe[0], pe[1]);
                            pw[cq][u4 * 2 + 1] = pack_bf16x2(pe[2], pe[3]);
                        }
                    }
                    tc_fence_before();
                }
                // every thread has read its S^T columns before P^T overwrites them
                ok = named_bar_and(1, C::NCOMPUTE, ok);
                if (ok) {
                    tc_fence_after();
#pragma unroll
                    for (int cq = 0; cq < 2; ++cq) tmem_st16(lane_base + C::T_P + (half * 2 + cq) * 16, pw[cq]);
                    ok = mbar_wait(bar(C::B_DPFULL), g & 1, p.status, 33);
                }
                ok = __all_sync(0xffffffffu, ok);
                if (ok) {
                    tc_fence_after();
#pragma unroll
                    for (int cq = 0; cq < 2; ++cq) {
                        const int cc = half * 2 + cq;
                        float dp[32];
                        tmem_ld32(lane_base + C::T_DP + cc * 32, dp);
                        tmem_wait_ld();
                        uint32_t dw[16];
#pragma unroll
                        for (int u4 = 0; u4 < 8; ++u4) {
                            const float4 d4 = del4[cc * 8 + u4];
                            const float da[4] = {d4.x, d4.y, d4.z, d4.w};
                            const float pv[4] = {__uint_as_float(pw[cq][u4 * 2] << 16),
                                                 __uint_as_float(pw[cq][u4 * 2] & 0xffff0000u),
                                                 __uint_as_float(pw[cq][u4 * 2 + 1] << 16),
                                                 __uint_as_float(pw[cq][u4 * 2 + 1] & 0xffff0000u)};
                            float dv[4];
#pragma unroll
                            for (int x = 0; x < 4; ++x) dv[x] = pv[x] * (dp[u4 * 4 + x] - da[x]);
                            dw[u4 * 2] = pack_bf16x2(dv[0], dv[1]);
                            dw[u4 * 2 + 1] = pack_bf16x2(dv[2], dv[3]);
                        }
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int col = cc * 32 + q * 8;
                            st_shared_v4(dsa + (col >> 6) * 16384 + sw128_offset(r, (col & 63) >> 3), dw[4 * q],
                                         dw[4 * q + 1], dw[4 * q + 2], dw[4 * q + 3]);
                        }
                    }
                    mbar_arrive(bar(C::B_LEMPTY + 8 * ls));
                    tmem_wait_st();
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(bar(C::B_PFULL));
                    ok = mbar_wait(bar(C::B_DQFULL), g & 1, p.status, 31);
                }
                ok = __all_sync(0xffffffffu, ok);
                // dQ rows: this thread's TMEM lane is now query q0 + r, columns of its half
                float qv[D / 2];
                if (ok) {
                    tc_fence_after();
                    float v[32];
                    tmem_ld32(lane_base + C::T_DQ + half * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int x = 0; x < 32; ++x) qv[x] = v[x] * p.scale;
                    tc_fence_before();
                    mbar_arrive(bar(C::B_DQEMPTY));   // dQ has left TMEM
                }
                // one staging round: the 32-column block of this half
                if (ok) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        st_shared_v4(stage + half * 16384 + sw128_offset(r, k), __float_as_uint(qv[4 * k]),
                                     __float_as_uint(qv[4 * k + 1]), __float_as_uint(qv[4 * k + 2]),
                                     __float_as_uint(qv[4 * k + 3]));
                }
                fence_proxy_async_smem();
                ok = named_bar_and(1, C::NCOMPUTE, ok);
                if (ok && threadIdx.x == 0) {
                    for (int blk = 0; blk < 2; ++blk) tma_reduce_add_3d(&tm_dq, stage + blk * 16384, blk * 32, h, q0);
                    bulk_commit();
                    bulk_wait_read_all();   // the staging tile may be written again
                }
            }
            // ------------------------------ dK, dV ---------------------------------
            if (ok) ok = mbar_wait(bar(C::B_DKVFULL), ic & 1, p.status, 32);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) {
                tc_fence_after();
                for (int which = 0; which < 2; ++which) {   // 0: dK, 1: dV
                    const uint32_t tcol = which == 0 ? C::T_DK : C::T_DV;
                    const float mul = which == 0 ? p.scale : 1.f;
                    float v[32];
                    tmem_ld32(lane_base + tcol + half * 32, v);
                    tmem_wait_ld();
                    if (u.slot < 0) {
                        uint16_t* out = (which == 0 ? p.dk : p.dv) + ((size_t)j * p.hkv + u.hk) * D + half * 32;
                        if (j < p.N) {
#pragma unroll
                            for (int x = 0; x < 32; x += 8) {
                                uint4 y;
                                y.x = pack_bf16x2(v[x] * mul, v[x + 1] * mul);
                                y.y = pack_bf16x2(v[x + 2] * mul, v[x + 3] * mul);
                                y.z = pack_bf16x2(v[x + 4] * mul, v[x + 5] * mul);
                                y.w = pack_bf16x2(v[x + 6] * mul, v[x + 7] * mul);
                                *reinterpret_cast<uint4*>(out + x) = y;
                            }
                        }
                    } else {
                        float* out = p.part + ((((size_t)u.slot * p.hkv + u.hk) * 2 + which) * 128 + r) * D + half * 32;
#pragma unroll
                        for (int x = 0; x < 32; x += 4)
                            *reinterpret_cast<float4*>(out + x) =
                                make_float4(v[x] * mul, v[x + 1] * mul, v[x + 2] * mul, v[x + 3] * mul);
                    }
                }
                tc_fence_before();
            }
            ++ic;
            gs += nsteps;
        }
        if (threadIdx.x == 0) bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == C::MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace

cudaError_t launch_bwd(int d, const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                       const CUtensorMap* tdo, const CUtensorMap* tdq, const BwdParams& p, int grid,
                       cudaStream_t stream) {
    if (grid <= 0) return cudaSuccess;
    if (d != 64) return cudaErrorInvalidValue;
    using C = BwdCfg;
    cudaError_t e = cudaFuncSetAttribute(bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::BYTES);
    if (e != cudaSuccess) return e;
    // persistent: about one CTA per SM, each taking work units grid-stride
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || sms <= 0)
        sms = 1;
    const int ctas = grid < sms ? grid : sms;
    return launch_pdl(bwd_kernel, dim3(ctas), dim3(C::NWARPS * 32), C::BYTES, stream, *tq, *tk, *tv, *tdo, *tdq, p);
}

}  // namespace treeattn
