// gdn_decode.cu -- the gated delta rule step by step for a few tokens per
// sequence: the decode step after a prefill, or a short run of speculative
// tokens, on the same [rows, H, V, K] fp32 state (or pool) the prefill writes
// ("GDN 与 Chunked Prefill", section "块内 state 和块间 final state": decode
// carries the final state forward one token at a time; "FlashInfer GDN Prefill
// 完全指南", the state-pool section: sequences address pool rows through
// state_indices).  Per token, with k and q normalised when asked:
//
//     u = S k,   S <- alpha S + beta (v - alpha u) k^T,   o = scale S q
//
// which is S <- alpha S (I - beta k k^T) + beta v k^T read after the update.
//
// The step is bound by the state's bytes (64 KiB read and 64 KiB written per
// (sequence, head), a few hundred bytes of q/k/v/o per token), so it runs on
// CUDA cores with the state in registers: one CTA of 1024 threads per
// (sequence, state head); warp w owns state rows 4w..4w+3 and lane l columns
// 4l..4l+3, so every state row moves as one 512-byte coalesced access, and the
// row products S k and S q are four warp-wide sums.
#include <cuda_bf16.h>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kDecThreads = 1024;

template <typename T>
__device__ __forceinline__ void load4(const T* p, float (&x)[4]);

template <>
__device__ __forceinline__ void load4<float>(const float* p, float (&x)[4]) {
    const float4 f = *reinterpret_cast<const float4*>(p);
    x[0] = f.x;
    x[1] = f.y;
    x[2] = f.z;
    x[3] = f.w;
}

template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p, float (&x)[4]) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    x[0] = __uint_as_float(u.x << 16);
    x[1] = __uint_as_float(u.x & 0xffff0000u);
    x[2] = __uint_as_float(u.y << 16);
    x[3] = __uint_as_float(u.y & 0xffff0000u);
}

template <typename T>
__device__ __forceinline__ void store4(T* p, const float (&x)[4]);

template <>
__device__ __forceinline__ void store4<float>(float* p, const float (&x)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
}

template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, const float (&x)[4]) {
    __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]), b = __floats2bfloat162_rn(x[2], x[3]);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <typename T>
__global__ void __launch_bounds__(kDecThreads) gdn_decode_kernel(const DecodeParams p) {
    const int64_t unit = blockIdx.x;
    const int32_t seq = static_cast<int32_t>(unit / p.H), h = static_cast<int32_t>(unit % p.H);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int v0 = 4 * warp, c0 = 4 * lane;
    int64_t srow = seq;
    if (p.state_indices) {
        srow = load_index(p.state_indices, p.idx_i64, seq);
        if (srow < 0 || srow >= p.n_pool) {  // uniform over the CTA: nothing is read or written
            if (threadIdx.x == 0 && p.status) atomicOr(p.status, static_cast<int32_t>(GDN_DEVICE_ERR_STATE_INDEX_RANGE));
            return;
        }
    }
    const size_t sbase = (static_cast<size_t>(srow) * p.H + h) * kHead * kHead;
    float S[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        if (p.initial_state) {
            load4(p.initial_state + sbase + static_cast<size_t>(v0 + r) * kHead + c0, S[r]);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) S[r][j] = 0.f;
        }
    }
    const T* q = static_cast<const T*>(p.q);
    const T* k = static_cast<const T*>(p.k);
    const T* v = static_cast<const T*>(p.v);
    T* out = static_cast<T*>(p.output);
    const int32_t qh = h / (p.H / p.hq), kh = h / (p.H / p.hk), vh = h / (p.H / p.hv);
    for (int32_t t = 0; t < p.m; ++t) {
        const int64_t tok = static_cast<int64_t>(seq) * p.m + t;
        float kx[4], qx[4], vx[4];
        load4(k + (static_cast<size_t>(tok) * p.hk + kh) * kHead + c0, kx);
        load4(q + (static_cast<size_t>(tok) * p.hq + qh) * kHead + c0, qx);
        load4(v + (static_cast<size_t>(tok) * p.hv + vh) * kHead + v0, vx);
        const size_t gi = static_cast<size_t>(tok) * p.H + h;
        const float a = p.g ? p.g[gi] : 1.f;
        const float b = p.beta ? p.beta[gi] : 1.f;
        if (p.l2norm) {
            const float rk = rsqrtf(warp_sum(kx[0] * kx[0] + kx[1] * kx[1] + kx[2] * kx[2] + kx[3] * kx[3]) + 1e-6f);
            const float rq = rsqrtf(warp_sum(qx[0] * qx[0] + qx[1] * qx[1] + qx[2] * qx[2] + qx[3] * qx[3]) + 1e-6f);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                kx[j] *= rk;
                qx[j] *= rq;
            }
        }
        float o[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float u = warp_sum(S[r][0] * kx[0] + S[r][1] * kx[1] + S[r][2] * kx[2] + S[r][3] * kx[3]);
            const float w = b * (vx[r] - a * u);
#pragma unroll
            for (int j = 0; j < 4; ++j) S[r][j] = a * S[r][j] + w * kx[j];
            o[r] = p.scale * warp_sum(S[r][0] * qx[0] + S[r][1] * qx[1] + S[r][2] * qx[2] + S[r][3] * qx[3]);
        }
        if (lane == 0) store4(out + (static_cast<size_t>(tok) * p.H + h) * kHead + v0, o);
    }
    if (p.output_state) {
#pragma unroll
        for (int r = 0; r < 4; ++r) store4(p.output_state + sbase + static_cast<size_t>(v0 + r) * kHead + c0, S[r]);
    }
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, bool bf16, cudaStream_t stream) {
    const int64_t blocks = static_cast<int64_t>(p.N) * p.H;
    if (blocks == 0) return cudaSuccess;
    if (bf16)
        gdn_decode_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), kDecThreads, 0, stream>>>(p);
    else
        gdn_decode_kernel<float><<<static_cast<unsigned>(blocks), kDecThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
