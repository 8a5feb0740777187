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

// One warp per (row i, head h); rows [0, Npad).
__global__ void __launch_bounds__(256) bwd_pre_kernel(const BwdPreParams p) {
    const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t total = (int64_t)p.Npad * p.hq;
    if (wid >= total) return;
    const int i = (int)(wid / p.hq), h = (int)(wid % p.hq);
    float acc = 0.f;
    if (i < p.N) {
        const size_t base = ((size_t)i * p.hq + h) * p.d;
        for (int x = lane * 4; x < p.d; x += 128) {
            const uint2 ow = *reinterpret_cast<const uint2*>(p.o + base + x);
            const uint2 dw = *reinterpret_cast<const uint2*>(p.dout + base + x);
            acc += bf16_bits_to_float(ow.x & 0xffff) * bf16_bits_to_float(dw.x & 0xffff);
            acc += bf16_bits_to_float(ow.x >> 16) * bf16_bits_to_float(dw.x >> 16);
            acc += bf16_bits_to_float(ow.y & 0xffff) * bf16_bits_to_float(dw.y & 0xffff);
            acc += bf16_bits_to_float(ow.y >> 16) * bf16_bits_to_float(dw.y >> 16);
            *reinterpret_cast<float4*>(p.dq_acc + base + x) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
        const size_t k = (size_t)h * p.Npad + i;
        p.delta[k] = acc;
        p.lse2[k] = i < p.N ? p.lse[(size_t)h * p.N + i] * 1.4426950408889634f : INFINITY;
    }
}

// dQ: 4 elements per thread.
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ src, uint16_t* __restrict__ dst,
                                                         int64_t n4) {
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= n4) return;
    const float4 v = reinterpret_cast<const float4*>(src)[k];
    uint2 w;
    w.x = (uint32_t)float_to_bf16_bits(v.x) | ((uint32_t)float_to_bf16_bits(v.y) << 16);
    w.y = (uint32_t)float_to_bf16_bits(v.z) | ((uint32_t)float_to_bf16_bits(v.w) << 16);
    reinterpret_cast<uint2*>(dst)[k] = w;
}

// One block per (split kv-tile, kv-head, dK|dV); thread = 4 consecutive
// elements of the 128 x d tile.
__global__ void __launch_bounds__(256) dkv_reduce_kernel(const BwdPostParams p) {
    const int which = blockIdx.x & 1;
    const int hk = (blockIdx.x >> 1) % p.hkv;
    const int si = (blockIdx.x >> 1) / p.hkv;
    const int4 sp = reinterpret_cast<const int4*>(p.splits)[si];
    const int c = sp.x, base = sp.y, nslot = sp.z;
    const int per_tile = 128 * p.d;
    uint16_t* out = which == 0 ? p.dk : p.dv;
    for (int e = threadIdx.x * 4; e < per_tile; e += blockDim.x * 4) {
        const int r = e / p.d, x = e % p.d;
        const int j = c * 128 + r;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k = 0; k < nslot; ++k) {
            const float4 v = *reinterpret_cast<const float4*>(
                p.part + (((size_t)(base + k) * p.hkv + hk) * 2 + which) * per_tile + e);
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

}  // namespace

cudaError_t launch_bwd_pre(const BwdPreParams& p, cudaStream_t stream) {
    const int64_t warps = (int64_t)p.Npad * p.hq;
    const int64_t blocks = (warps * 32 + 255) / 256;
    if (blocks > INT32_MAX) return cudaErrorInvalidValue;
    bwd_pre_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_bwd_post(const BwdPostParams& p, cudaStream_t stream) {
    const int64_t n4 = (int64_t)p.N * p.hq * p.d / 4;
    const int64_t blocks = (n4 + 255) / 256;
    if (blocks > INT32_MAX) return cudaErrorInvalidValue;
    if (blocks > 0) dq_convert_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p.dq_acc, p.dq, n4);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (p.n_splits > 0) {
        dkv_reduce_kernel<<<p.n_splits * p.hkv * 2, 256, 0, stream>>>(p);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace treeattn
