// Memory-bound helpers around the backward tensor-core kernel.
//
// bwd_pre : Delta[h, i] = sum_d dO[i,h,d] * O[i,h,d] (the row term of the
//           softmax gradient, dS = P * (dP - Delta)); LSE rescaled to log2
//           units and padded with +inf past N (so padded queries get P = 0);
//           the fp32 dQ accumulator zeroed.
// bwd_post: dQ accumulator -> bf16; for kv-tiles whose descendant q-range was
//           split over several work items, the fp32 dK / dV partials summed in
//           ascending chunk order (a fixed order, so the result is
//           reproducible bit for bit) and rounded to bf16.
#include "kernels.h"
#include "ptx.cuh"

namespace treeattn {

namespace {

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t*>(&h);
}

// d/8 lanes per (row i, head h), 8 features (16 bytes of O and of dO) each;
// rows [0, Npad), last rows first: the first q-tiles' dQ accumulator rows and
// dO rows, which the backward's first work items touch, are then the ones
// written or read most recently and still in L2.
__global__ void __launch_bounds__(256) bwd_pre_kernel(const BwdPreParams p) {
    grid_dep_wait();   // O and LSE come from the forward
    grid_dep_launch();
    const int lanes = p.d >> 3;                                   // 16 (d = 128) or 8 (d = 64)
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t total = (int64_t)p.Npad * p.hq;
    const int64_t pair = total - 1 - gid / lanes;
    const int sub = (int)(gid % lanes);
    const bool live = pair >= 0;
    const int i = live ? (int)(pair / p.hq) : 0, h = live ? (int)(pair % p.hq) : 0;
    float acc = 0.f;
    if (live && i < p.N) {
        const size_t off = ((size_t)i * p.hq + h) * p.d + sub * 8;
        const uint4 ow = *reinterpret_cast<const uint4*>(p.o + off);
        const uint4 dw = *reinterpret_cast<const uint4*>(p.dout + off);
        const uint32_t ov[4] = {ow.x, ow.y, ow.z, ow.w}, dv[4] = {dw.x, dw.y, dw.z, dw.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            acc += bf16_bits_to_float(ov[k] & 0xffff) * bf16_bits_to_float(dv[k] & 0xffff);
            acc += bf16_bits_to_float(ov[k] >> 16) * bf16_bits_to_float(dv[k] >> 16);
        }
        float4* z = reinterpret_cast<float4*>(p.dq_acc + off);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // sum over the lanes of this (row, head): aligned groups of `lanes` lanes
    for (int o = lanes >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (live && sub == 0) {
        const size_t k = (size_t)h * p.Npad + i;
        p.delta[k] = acc;
        p.lse2[k] = i < p.N ? p.lse[(size_t)h * p.N + i] * 1.4426950408889634f : INFINITY;
    }
}

// dQ: kConvertPer groups of 4 elements per thread, a block's groups contiguous
// (each of the thread's loads is one coalesced row of the block), all loads
// issued before the first store.
constexpr int kConvertPer = 4;
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ src, uint16_t* __restrict__ dst,
                                                         int64_t n4) {
    grid_dep_wait();   // the accumulator is complete once the main pass has finished
    grid_dep_launch();
    const int64_t base = (int64_t)blockIdx.x * blockDim.x * kConvertPer + threadIdx.x;
    float4 v[kConvertPer];
#pragma unroll
    for (int u = 0; u < kConvertPer; ++u) {
        const int64_t k = base + (int64_t)u * blockDim.x;
        if (k < n4) v[u] = reinterpret_cast<const float4*>(src)[k];
    }
#pragma unroll
    for (int u = 0; u < kConvertPer; ++u) {
        const int64_t k = base + (int64_t)u * blockDim.x;
        if (k < n4) {
            uint2 w;
            w.x = (uint32_t)float_to_bf16_bits(v[u].x) | ((uint32_t)float_to_bf16_bits(v[u].y) << 16);
            w.y = (uint32_t)float_to_bf16_bits(v[u].z) | ((uint32_t)float_to_bf16_bits(v[u].w) << 16);
            reinterpret_cast<uint2*>(dst)[k] = w;
        }
    }
}

// One block per (split kv-tile, kv-head, dK|dV, group of 16 rows); thread = 4
// consecutive elements of the group's 16 x d slice of the 128 x d tile.
constexpr int kDkvRowGroups = 8;
__global__ void __launch_bounds__(256) dkv_reduce_kernel(const BwdPostParams p) {
    grid_dep_wait();   // the partial slots come from the main pass (the dQ conversion runs between)
    grid_dep_launch();
    const int rg = blockIdx.x % kDkvRowGroups;
    const int rest = blockIdx.x / kDkvRowGroups;
    const int which = rest & 1;
    const int hk = (rest >> 1) % p.hkv;
    const int si = (rest >> 1) / p.hkv;
    const int4 sp = reinterpret_cast<const int4*>(p.splits)[si];
    const int c = sp.x, base = sp.y, nslot = sp.z;
    // debug builds: the split's kv-tile and slot range must lie inside the plan
    if (!(ta_ok(p.status, 401, c, 0, p.T) && ta_ok(p.status, 402, base, 0, p.n_slots) &&
          ta_ok(p.status, 403, (long long)base + nslot - 1, base, p.n_slots)))
        return;
    const int per_tile = 128 * p.d;
    const int per_group = per_tile / kDkvRowGroups;
    uint16_t* out = which == 0 ? p.dk : p.dv;
    for (int e = rg * per_group + threadIdx.x * 4; e < (rg + 1) * per_group; e += blockDim.x * 4) {
        const int r = e / p.d, x = e % p.d;
        const int j = c * 128 + r;
        // ascending chunk order (the same additions on every run); loads are issued
        // four at a time so that they overlap
        const size_t stride = (size_t)p.hkv * 2 * per_tile;
        const float* src = p.part + (((size_t)base * p.hkv + hk) * 2 + which) * per_tile + e;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        int k = 0;
        for (; k + 4 <= nslot; k += 4) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = __ldg(reinterpret_cast<const float4*>(src + (size_t)(k + u) * stride));
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                acc.x += v[u].x;
                acc.y += v[u].y;
                acc.z += v[u].z;
                acc.w += v[u].w;
            }
        }
        for (; k < nslot; ++k) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(src + (size_t)k * stride));
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        if (j < p.N) {
            uint2 w;
            w.x = (uint32_t)float_to_bf16_bits(acc.x) | ((uint32_t)float_to_bf16_bits(acc.y) << 16);
            w.y = (uint32_t)float_to_bf16_bits(acc.z) | ((uint32_t)float_to_bf16_bits(acc.w) << 16);
            *reinterpret_cast<uint2*>(out + ((size_t)j * p.hkv + hk) * p.d + x) = w;
        }
    }
}

// One thread waits, with the given limit, on a barrier that no one completes:
// the timeout path of every bounded wait in the kernels, run on purpose.  The
// wait ends by itself and the kernel returns; nothing faults.
__global__ void wait_selftest_kernel(int* status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar_mem;
    const uint32_t bar = smem_u32(&bar_mem);
    mbar_init(bar, 1);
    fence_mbar_init();
    if (mbar_try_wait(bar, 0)) return;
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 <= limit_ns)
        if (mbar_try_wait(bar, 0)) return;
    report_status(status, -10 - 1000 * 99);
}

// One thread checks an index that lies outside its range on purpose: in debug
// builds the check records site 98 and the (never made) access is skipped.
__global__ void bounds_selftest_kernel(int* status, int* out) {
    const int index = 5, size = 4;
    if (ta_ok(status, 98, index, 0, size)) *out = index;
}

}  // namespace

void launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 1, 0, stream>>>(status, limit_ns);
}

void launch_bounds_selftest(int* status, int* out, cudaStream_t stream) {
    bounds_selftest_kernel<<<1, 1, 0, stream>>>(status, out);
}

cudaError_t launch_bwd_pre(const BwdPreParams& p, cudaStream_t stream) {
    const int64_t threads = (int64_t)p.Npad * p.hq * (p.d / 8);
    const int64_t blocks = (threads + 255) / 256;
    if (blocks > INT32_MAX) return cudaErrorInvalidValue;
    return launch_pdl(bwd_pre_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, p);
}

cudaError_t launch_bwd_post(const BwdPostParams& p, cudaStream_t stream) {
    const int64_t n4 = (int64_t)p.N * p.hq * p.d / 4;
    const int64_t blocks = (n4 + 256 * kConvertPer - 1) / (256 * kConvertPer);
    if (blocks > INT32_MAX) return cudaErrorInvalidValue;
    cudaError_t e = cudaSuccess;
    if (blocks > 0) e = launch_pdl(dq_convert_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, p.dq_acc, p.dq, n4);
    if (e != cudaSuccess) return e;
    if (p.n_splits > 0)
        e = launch_pdl(dkv_reduce_kernel, dim3(p.n_splits * p.hkv * 2 * kDkvRowGroups), dim3(256), 0, stream, p);
    return e;
}

}  // namespace treeattn
