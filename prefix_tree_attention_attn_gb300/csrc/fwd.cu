// Forward kernel: O and LSE of causal softmax attention over a packed prefix
// tree, on the sm_103a tensor cores.
//
// One CTA = one 128-row q-tile x NS q-heads of the same kv-head group.  The CTA
// visits only the kv-tiles in the q-tile's ancestor interval list; empty tiles
// are never loaded.  Three shapes, chosen per plan and head layout:
//  * NS = 2 (even group size, long kv-tile lists): the two q-heads read the same
//    key tiles, so every K/V tile is loaded once for both; one CTA per SM with a
//    deep K/V ring.
//  * NS = 1, two CTAs per SM (short lists): a 2-slot ring and 256 TMEM columns
//    per CTA, so two CTAs share an SM and one CTA's prologue (Q and first K
//    load, first S) and epilogue overlap the other's tiles.  With a handful of
//    kv-tiles per q-tile that overlap is worth more than loading each K/V tile
//    once per head pair.
//  * NS = 1, one CTA per SM: long lists with an odd group size.
//
// Warp roles (NS = 2; 320 threads):
//   warps 0-3  softmax for q-head 0 (one query row per thread)
//   warps 4-7  softmax for q-head 1
//   warp  8    TMA producer: Q once, then K_j, V_j through a ring of slots
//   warp  9    tcgen05 issuer (one thread) + TMEM owner
// TMEM (per q-head s): S = Q K^T at columns [256 s, 256 s + 128), the output
// accumulator O at [256 s + 128, 256 s + 128 + D).
//
// Pipeline on the tensor core:  S0(0) S1(0) | PV0(0) S0(1) | PV1(0) S1(1) | ...
// While softmax group 0 turns S0(j) into P0(j), the tensor core runs q-head 1's
// MMAs, and the other way round.  P is written back over S in TMEM (packed
// bf16) and feeds O += P V as the A operand, so it never goes through shared
// memory.  The softmax warps, not the MMAs, set the pace (their instruction
// issue), so pass 1 takes the maximum of the raw logits (the scale is
// positive) three at a time and pass 2 is one packed FFMA per two elements
// into ex2.  O is rescaled in TMEM only when a
// row's running maximum grows by more than 2^8 (the accumulated sum and O keep
// one common reference maximum, so the result is unchanged).
//
// Masking: a full block needs none; a partial block keeps key j for row i iff
// j <= i and i < subend[j] (the packed-layout lemma; see plan.cpp).  Inside a
// partial block, a warp whose 32 rows all satisfy j_max <= i < min subend
// needs no mask either.
#include "kernels.h"
#include "ptx.cuh"

namespace treeattn {

namespace {

template <int D, int NS, int PER_SM>
struct FwdCfg {
    static_assert(PER_SM == 1 || NS == 1, "two CTAs per SM only with one q-head per CTA");
    static constexpr int TILE = 128 * D * 2;          // Q/K/V tile bytes
    static constexpr int SMALL = 3072;                // barriers + subend staging
    // K/V ring: every slot that fits next to Q (at most 8)
    // (two CTAs per SM: 2 slots, 101 KB per CTA)
    static constexpr int NSLOT =
        PER_SM == 2 ? 2 : ((229376 - NS * TILE) / TILE < 8 ? (229376 - NS * TILE) / TILE : 8);
    static constexpr int OFF_Q = SMALL;
    static constexpr int OFF_KV = OFF_Q + NS * TILE;
    static constexpr int BYTES = OFF_KV + NSLOT * TILE;
    static constexpr int NWARPS = 4 * NS + 2;
    static constexpr int PRODUCER = 4 * NS;
    static constexpr int MMA = 4 * NS + 1;
    static constexpr int TMEM_COLS = NS == 2 ? 512 : 256;
    // small-region offsets
    static constexpr int B_QFULL = 0;
    static constexpr int B_KVFULL = 8;
    static constexpr int B_KVEMPTY = B_KVFULL + 8 * NSLOT;
    static constexpr int B_SFULL = B_KVEMPTY + 8 * NSLOT;
    static constexpr int B_PFULL = B_SFULL + 8 * NS;
    static constexpr int B_OFULL = B_PFULL + 8 * NS;
    static constexpr int B_DRAIN = B_OFULL + 8 * NS;
    static constexpr int HOLDER = B_DRAIN + 8;
    static constexpr int SUB = 1024;                  // NS x 128 int32
    static_assert(SUB + NS * 512 <= SMALL, "small region");
    static_assert(HOLDER + 4 <= SUB, "barriers");
    static_assert(BYTES <= 232448, "shared memory");
    static_assert(NSLOT >= NS && NSLOT >= 2, "the epilogue stages O in ring slots");
    static_assert(PER_SM * BYTES <= 232448, "CTAs per SM");
};

constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows by > 2^8

template <int D, int NS, int PER_SM>
__global__ void __launch_bounds__(FwdCfg<D, NS, PER_SM>::NWARPS * 32, PER_SM)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
               const FwdParams p) {
    using C = FwdCfg<D, NS, PER_SM>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (sb & 1023u) {
        if (threadIdx.x == 0) report_status(p.status, -5);
        return;
    }

    // CTA order (q-tiles in the planner's order, longest kv-tile list first):
    // q-tile, then head slice; or, when one q-tile's K/V stream over every kv-head
    // would crowd L2, kv-head group, then q-tile, then the group's head slices, so
    // the CTAs running at one time read one kv-head's K/V.
    int t, h0;
    if (p.kv_major) {
        const int per_g = p.group / NS;
        const int grp = blockIdx.x / (p.T * per_g);
        const int rem = blockIdx.x - grp * p.T * per_g;
        t = p.fwd_order[rem / per_g];
        h0 = grp * p.group + (rem % per_g) * NS;
    } else {
        const int n_hg = p.hq / NS;
        t = p.fwd_order[blockIdx.x / n_hg];
        h0 = (blockIdx.x % n_hg) * NS;
    }
    const int hk = h0 / p.group;
    const int q0 = t * 128;
    // debug builds: the q-tile, its kv-tile list and the heads must lie inside
    // the plan's tables (a uniform return, before any barrier or TMEM is set up)
    if (!(ta_ok(p.status, 101, t, 0, p.T) && ta_ok(p.status, 102, h0 + NS - 1, 0, p.hq)))
        return;
    const int e0 = p.qt_ptr[t];
    const int n_kv = p.qt_ptr[t + 1] - e0;  // >= 1: the diagonal block is never empty
    if (!(ta_ok(p.status, 103, e0, 0, p.n_ent) && ta_ok(p.status, 104, (long long)e0 + n_kv - 1, e0, p.n_ent)))
        return;

    const uint32_t b_qfull = sb + C::B_QFULL;
    auto b_kvfull = [&](int s) { return sb + C::B_KVFULL + 8 * s; };
    auto b_kvempty = [&](int s) { return sb + C::B_KVEMPTY + 8 * s; };
    auto b_sfull = [&](int s) { return sb + C::B_SFULL + 8 * s; };
    auto b_pfull = [&](int s) { return sb + C::B_PFULL + 8 * s; };
    auto b_ofull = [&](int s) { return sb + C::B_OFULL + 8 * s; };
    const uint32_t b_drain = sb + C::B_DRAIN;

    if (threadIdx.x == 0) {
        mbar_init(b_qfull, 1);
        for (int s = 0; s < C::NSLOT; ++s) {
            mbar_init(b_kvfull(s), 1);
            mbar_init(b_kvempty(s), 1);
        }
        for (int s = 0; s < NS; ++s) {
            mbar_init(b_sfull(s), 1);
            mbar_init(b_pfull(s), 128);
            mbar_init(b_ofull(s), 1);
        }
        mbar_init(b_drain, 1);
        fence_mbar_init();
    }
    if (warp == C::MMA) tmem_alloc(sb + C::HOLDER, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::HOLDER);
    // Q, K, V may come from the previous kernel, and O / LSE may still be read by it
    grid_dep_wait();
    grid_dep_launch();

    if (warp == C::PRODUCER) {
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            mbar_expect_tx(b_qfull, NS * C::TILE);
            for (int s = 0; s < NS; ++s)
                for (int blk = 0; blk < D / 64; ++blk)
                    tma_load_3d(sb + C::OFF_Q + s * C::TILE + blk * 16384, &tm_q, blk * 64, h0 + s, q0, b_qfull);
            bool ok = true;
            for (int j = 0; j < n_kv && ok; ++j) {
                // debug builds: an out-of-range kv-tile is reported and kv-tile 0 loaded instead
                const int c = (int)ta_clamp(p.status, 105, p.qt_ent[e0 + j] >> 1, 0, p.T);
                for (int kv = 0; kv < 2 && ok; ++kv) {
                    const int pos = 2 * j + kv, slot = pos % C::NSLOT, use = pos / C::NSLOT;
                    if (use > 0) ok = mbar_wait(b_kvempty(slot), (use - 1) & 1, p.status, 1);
                    if (!ok) break;
                    mbar_expect_tx(b_kvfull(slot), C::TILE);
                    for (int blk = 0; blk < D / 64; ++blk)
                        tma_load_3d(sb + C::OFF_KV + slot * C::TILE + blk * 16384, kv ? &tm_v : &tm_k, blk * 64, hk,
                                    c * 128, b_kvfull(slot));
                }
            }
        }
    } else if (warp == C::MMA) {
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
            constexpr uint32_t IDESC_PV = idesc_bf16(128, D, false, true);
            auto issue_s = [&](int s, int slot) {
                const uint32_t qa = sb + C::OFF_Q + s * C::TILE, ka = sb + C::OFF_KV + slot * C::TILE;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
                    mma_bf16_ss(tmem + s * 256, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024),
                                IDESC_S, k > 0);
                }
            };
            auto issue_pv = [&](int s, int slot, bool acc) {   // O += P V, P from TMEM
                const uint32_t va = sb + C::OFF_KV + slot * C::TILE;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_bf16_ts(tmem + s * 256 + 128, tmem + s * 256 + k * 8, sdesc_sw128(va + k * 2048, 16384, 1024),
                                IDESC_PV, (acc || k > 0) ? 1u : 0u);
            };
            bool ok = mbar_wait(b_qfull, 0, p.status, 2);
            if (ok) ok = mbar_wait(b_kvfull(0), 0, p.status, 3);
            if (ok) {
                tc_fence_after();
                for (int s = 0; s < NS; ++s) {
                    issue_s(s, 0);
                    mma_commit(b_sfull(s));
                }
                mma_commit(b_kvempty(0));
            }
            for (int j = 0; j < n_kv && ok; ++j) {
                const int vpos = 2 * j + 1, vslot = vpos % C::NSLOT;
                ok = mbar_wait(b_kvfull(vslot), (vpos / C::NSLOT) & 1, p.status, 4);
                tc_fence_after();
                for (int s = 0; s < NS && ok; ++s) {
                    ok = mbar_wait(b_pfull(s), j & 1, p.status, 5);
                    if (!ok) break;
                    tc_fence_after();
                    issue_pv(s, vslot, j > 0);
                    if (s == NS - 1) mma_commit(b_kvempty(vslot));
                    // O is final for every head once the last head's last PV is done;
                    // only then may the epilogue reuse ring slots for staging
                    if (j == n_kv - 1 && s == NS - 1)
                        for (int ss = 0; ss < NS; ++ss) mma_commit(b_ofull(ss));
                    if (j + 1 < n_kv) {
                        const int kpos = 2 * (j + 1), kslot = kpos % C::NSLOT;
                        if (s == 0) {
                            ok = mbar_wait(b_kvfull(kslot), (kpos / C::NSLOT) & 1, p.status, 6);
                            if (!ok) break;
                            tc_fence_after();
                        }
                        issue_s(s, kslot);
                        mma_commit(b_sfull(s));
                        if (s == NS - 1) mma_commit(b_kvempty(kslot));
                    }
                }
            }
            // every MMA this thread issued must be finished before TMEM is freed
            mma_commit(b_drain);
            mbar_wait(b_drain, 0, p.status, 7);
        }
        __syncwarp();
    } else {
        // ------------------------------ softmax ------------------------------
        const int s = warp >> 2;
        const int r = ((warp & 3) << 5) + lane;  // row in tile == TMEM lane
        const int i = q0 + r;
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) << 5) << 16);
        const uint32_t tS = lane_base + s * 256;
        const uint32_t tO = tS + 128;
        int32_t* sub_sm = reinterpret_cast<int32_t*>(smem + C::SUB + s * 512);
        const uint32_t o_stage = sb + C::OFF_KV + s * C::TILE;   // ring slot s, idle once O is final
        const float sl2 = p.scale_log2;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        // The tile list, this row's subtree end of each partial tile's keys and the
        // tile's minimum subtree end are loaded a tile ahead (the list entry two
        // ahead), so no global-memory latency sits on a tile's critical path.
        // (debug builds: subtree ends and minima read at clamped kv-tiles)
        auto kv_of = [&](int ent) { return (int)ta_clamp(p.status, 106, ent >> 1, 0, p.T); };
        int ent_next = p.qt_ent[e0];
        int sub_next = 0, min_next = 0;
        if (ent_next & 1) {
            sub_next = p.subend[kv_of(ent_next) * 128 + r];
            min_next = p.kv_minsub[kv_of(ent_next)];
        }
        int ent_after = n_kv > 1 ? p.qt_ent[e0 + 1] : 0;
        for (int j = 0; j < n_kv; ++j) {
            const int ent = ent_next;
            const int c = ent >> 1;
            const bool partial = ent & 1;
            const int my_sub = sub_next, kv_min = min_next;
            ent_next = ent_after;
            if (j + 1 < n_kv && (ent_next & 1)) {
                sub_next = p.subend[kv_of(ent_next) * 128 + r];
                min_next = p.kv_minsub[kv_of(ent_next)];
            }
            if (j + 2 < n_kv) ent_after = p.qt_ent[e0 + j + 2];
            // After a failed wait the loop keeps running (work skipped) so that every
            // thread of the group meets the same named barriers in the same order.
            if (ok) ok = mbar_wait(b_sfull(s), j & 1, p.status, 8);
            ok = __all_sync(0xffffffffu, ok);
            // One barrier publishes the staged subtree ends and makes `ok` uniform.
            // Overwriting the staging row is safe without a barrier before it: S of
            // this tile exists only after every thread of the group has arrived on
            // the previous tile's P barrier, i.e. finished reading the old values.
            if (partial) {
                if (ok) sub_sm[r] = my_sub;
                ok = named_bar_and(1 + s, 128, ok);
            }
            if (!ok) continue;
            tc_fence_after();
            // pass 1: row maximum of the raw logits over the 128 key columns.  A warp
            // whose rows all see every key of the tile (j_max <= i < min subend) skips
            // the mask; otherwise masked logits are set to -inf and written back to
            // TMEM, so pass 2 never masks.
            const int kbase = c * 128;
            const bool need_mask =
                partial && !__all_sync(0xffffffffu, kbase + 127 <= i && i < kv_min);
            auto mask = [&](float (&v)[32], int cc) {
#pragma unroll
                for (int u4 = 0; u4 < 8; ++u4) {
                    const int4 sv = reinterpret_cast<const int4*>(sub_sm)[cc * 8 + u4];
                    const int sa[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const int u = u4 * 4 + w;
                        const bool keep = (kbase + cc * 32 + u <= i) && (i < sa[w]);
                        v[u] = keep ? v[u] : -INFINITY;
                    }
                }
            };
            float mraw = -INFINITY;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                float v[32];
                tmem_ld32(tS + cc * 32, v);
                tmem_wait_ld();
                if (need_mask) {
                    mask(v, cc);
                    tmem_st32(tS + cc * 32, v);
                }
#pragma unroll
                for (int u = 0; u < 32; u += 2) mraw = fmax3(mraw, v[u], v[u + 1]);
            }
            if (need_mask) tmem_wait_st();
            const float mx = mraw * sl2;   // softmax_scale > 0, so the maximum commutes with it
            const float m_new = fmaxf(m_run, mx);
            const bool need = m_new > m_run + kRescaleThreshold;   // false while both are -inf
            const float factor = need ? fast_exp2(m_run - m_new) : 1.f;
            if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    float v[32];
                    tmem_ld32(tO + cc * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int u = 0; u < 32; ++u) v[u] *= factor;
                    tmem_st32(tO + cc * 32, v);
                }
                tmem_wait_st();
            }
            if (need) {
                l_run *= factor;
                m_run = m_new;
            }
            const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
            // pass 2: P = 2^(s * scale*log2e - m) -> packed bf16 over S's first 64
            // columns (each store lands on columns this thread has already read).
            // The softmax warps are bound by instruction issue, so the argument and
            // the row sum go through packed fp32 pairs (one instruction per two
            // columns); the per-lane results equal the scalar fmaf / add.
            const uint64_t scale2 = f32x2(sl2, sl2), negm2 = f32x2(-m_use, -m_use);
            uint64_t lsum2 = f32x2(0.f, 0.f);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                float v[32];
                tmem_ld32(tS + cc * 32, v);
                tmem_wait_ld();
                uint32_t pw[16];
#pragma unroll
                for (int h = 0; h < 16; ++h) {
                    float ta, tb;
                    f32x2_split(fma_f32x2(f32x2(v[2 * h], v[2 * h + 1]), scale2, negm2), ta, tb);
                    const float a = fast_exp2(ta), b = fast_exp2(tb);
                    lsum2 = add_f32x2(lsum2, f32x2(a, b));
                    pw[h] = pack_bf16x2(a, b);
                }
                tmem_st16(tS + cc * 16, pw);
            }
            float lsa, lsb;
            f32x2_split(lsum2, lsa, lsb);
            l_run += lsa + lsb;
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(b_pfull(s));
        }
        // ------------------------------ epilogue -----------------------------
        if (ok) ok = mbar_wait(b_ofull(s), 0, p.status, 9);
        ok = named_bar_and(1 + s, 128, ok);
        if (ok) {
            tc_fence_after();
            const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
            // O (bf16) into ring slot s (every load has been consumed by then),
            // laid out like a TMA tile of Q
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                float v[32];
                tmem_ld32(tO + cc * 32, v);
                tmem_wait_ld();
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const int col = cc * 32 + g * 8;   // first of 8 columns
                    st_shared_v4(o_stage + (col >> 6) * 16384 + sw128_offset(r, (col & 63) >> 3),
                                 pack_bf16x2(v[g * 8 + 0] * inv_l, v[g * 8 + 1] * inv_l),
                                 pack_bf16x2(v[g * 8 + 2] * inv_l, v[g * 8 + 3] * inv_l),
                                 pack_bf16x2(v[g * 8 + 4] * inv_l, v[g * 8 + 5] * inv_l),
                                 pack_bf16x2(v[g * 8 + 6] * inv_l, v[g * 8 + 7] * inv_l));
                }
            }
            if (i < p.N) p.lse[(size_t)(h0 + s) * p.N + i] = (m_run + __log2f(l_run)) * 0.69314718055994531f;
            fence_proxy_async_smem();
            named_bar_sync(1 + s, 128);
            if (r == 0) {
                for (int blk = 0; blk < D / 64; ++blk) tma_store_3d(&tm_o, o_stage + blk * 16384, blk * 64, h0 + s, q0);
                bulk_commit();
                bulk_wait_all();
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

template <int D, int NS, int PER_SM>
cudaError_t launch_cfg(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv, const CUtensorMap* to,
                       const FwdParams& p, int grid, cudaStream_t stream) {
    using C = FwdCfg<D, NS, PER_SM>;
    auto kern = fwd_kernel<D, NS, PER_SM>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::BYTES);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(C::NWARPS * 32), C::BYTES, stream, *tq, *tk, *tv, *to, p);
}

}  // namespace

cudaError_t launch_fwd(int d, int nstream, int per_sm, const CUtensorMap* tq, const CUtensorMap* tk,
                       const CUtensorMap* tv, const CUtensorMap* to, const FwdParams& p, int grid,
                       cudaStream_t stream) {
    if (d == 128) {
        if (nstream == 2) return launch_cfg<128, 2, 1>(tq, tk, tv, to, p, grid, stream);
        return per_sm == 2 ? launch_cfg<128, 1, 2>(tq, tk, tv, to, p, grid, stream)
                           : launch_cfg<128, 1, 1>(tq, tk, tv, to, p, grid, stream);
    }
    if (nstream == 2) return launch_cfg<64, 2, 1>(tq, tk, tv, to, p, grid, stream);
    return per_sm == 2 ? launch_cfg<64, 1, 2>(tq, tk, tv, to, p, grid, stream)
                       : launch_cfg<64, 1, 1>(tq, tk, tv, to, p, grid, stream);
}

}  // namespace treeattn
