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
// CUDA cores with the state in registers: persistent CTAs of 1024 threads,
// one (sequence, state head) unit at a time, with the next unit's state loads
// in flight behind the current unit's arithmetic; warp w owns state rows
// 4w..4w+3 and lane l columns 4l..4l+3, so every state row moves as one
// 512-byte coalesced access, and the row products S k and S q are four
// warp-wide sums.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

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

template <>
__device__ __forceinline__ void load4<__half>(const __half* p, float (&x)[4]) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    __half2 a, b;
    memcpy(&a, &u.x, 4);
    memcpy(&b, &u.y, 4);
    const float2 fa = __half22float2(a), fb = __half22float2(b);
    x[0] = fa.x;
    x[1] = fa.y;
    x[2] = fb.x;
    x[3] = fb.y;
}

// fp8 state elements (storage only): one byte each, converted with the shared fp8 helpers
struct F8E4M3 {
    uint8_t bits;
};
struct F8E5M2 {
    uint8_t bits;
};

template <>
__device__ __forceinline__ void load4<F8E4M3>(const F8E4M3* p, float (&x)[4]) {
    state_load4(p, 0, GDN_DTYPE_F8E4M3, x);
}

template <>
__device__ __forceinline__ void load4<F8E5M2>(const F8E5M2* p, float (&x)[4]) {
    state_load4(p, 0, GDN_DTYPE_F8E5M2, x);
}

template <typename T>
__device__ __forceinline__ void store4(T* p, const float (&x)[4]);

template <>
__device__ __forceinline__ void store4<F8E4M3>(F8E4M3* p, const float (&x)[4]) {
    state_store4(p, 0, GDN_DTYPE_F8E4M3, x);
}

template <>
__device__ __forceinline__ void store4<F8E5M2>(F8E5M2* p, const float (&x)[4]) {
    state_store4(p, 0, GDN_DTYPE_F8E5M2, x);
}

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

template <>
__device__ __forceinline__ void store4<__half>(__half* p, const float (&x)[4]) {
    const __half2 a = __floats2half2_rn(x[0], x[1]), b = __floats2half2_rn(x[2], x[3]);
    uint2 u;
    memcpy(&u.x, &a, 4);
    memcpy(&u.y, &b, 4);
    *reinterpret_cast<uint2*>(p) = u;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Loads of one token: this lane's 4 columns of k and q, the warp's 4 rows of v, and alpha, beta.
struct TokenIn {
    float k[4], q[4], v[4], a, b;
};

template <typename T>
__device__ __forceinline__ void load_token(const DecodeParams& p, int64_t tok, int32_t h, int32_t qh, int32_t kh,
                                           int32_t vh, int v0, int c0, TokenIn& x) {
    load4(static_cast<const T*>(p.k) + (static_cast<size_t>(tok) * p.hk + kh) * kHead + c0, x.k);
    load4(static_cast<const T*>(p.q) + (static_cast<size_t>(tok) * p.hq + qh) * kHead + c0, x.q);
    load4(static_cast<const T*>(p.v) + (static_cast<size_t>(tok) * p.hv + vh) * kHead + v0, x.v);
    const size_t gi = static_cast<size_t>(tok) * p.H + h;
    x.a = p.g ? p.g[gi] : 1.f;
    x.b = p.beta ? p.beta[gi] : 1.f;
}

// This thread's 16 state values of unit u (sequence u / H, head u % H), states of element type SD; false
// when its pool row is out of range (then the unit is skipped and flagged).
template <typename SD>
__device__ __forceinline__ bool load_state(const DecodeParams& p, int64_t u, int v0, int c0, float (&S)[4][4],
                                           int64_t& sbase) {
    const int32_t seq = static_cast<int32_t>(u / p.H), h = static_cast<int32_t>(u % p.H);
    int64_t srow = seq;
    if (p.state_indices) {
        srow = load_index(p.state_indices, p.idx_i64, seq);
        if (srow < 0 || srow >= p.n_pool) return false;
    }
    sbase = state_offset(p.state, srow, h, v0) + c0;  // element offset of this thread's first value
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        if (p.initial_state) {
            load4(static_cast<const SD*>(p.initial_state) + sbase + r * static_cast<int32_t>(p.state.s_v), S[r]);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) S[r][j] = 0.f;
        }
    }
    return true;
}

// Persistent CTAs walk the (sequence, head) units.  With one token per
// sequence (kNextUnit) the next unit's state loads are issued before the
// current unit's arithmetic; with several, the next token's inputs are loaded
// before the current token's arithmetic instead (the registers hold one of the
// two prefetches, not both).  Either way memory latency overlaps work.
template <typename T, typename SD, bool kNextUnit>
__global__ void __launch_bounds__(kDecThreads) gdn_decode_kernel(const DecodeParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int v0 = 4 * warp, c0 = 4 * lane;
    const int64_t units = static_cast<int64_t>(p.N) * p.H;
    int64_t u = blockIdx.x;
    float Sn[4][4];
    int64_t sbase_n = 0;
    bool ok_n = kNextUnit && u < units && load_state<SD>(p, u, v0, c0, Sn, sbase_n);
    for (; u < units; u += gridDim.x) {
        float S[4][4];
        int64_t sbase;
        bool ok;
        if (kNextUnit) {
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int j = 0; j < 4; ++j) S[r][j] = Sn[r][j];
            sbase = sbase_n;
            ok = ok_n;
            const int64_t un = u + gridDim.x;
            if (un < units) ok_n = load_state<SD>(p, un, v0, c0, Sn, sbase_n);
        } else {
            ok = load_state<SD>(p, u, v0, c0, S, sbase);
        }
        if (!ok) {  // uniform over the CTA: nothing is read or written for this unit
            if (threadIdx.x == 0 && p.status) atomicOr(p.status, static_cast<int32_t>(GDN_DEVICE_ERR_STATE_INDEX_RANGE));
            continue;
        }
        const int32_t seq = static_cast<int32_t>(u / p.H), h = static_cast<int32_t>(u % p.H);
        const int32_t qh = h / (p.H / p.hq), kh = h / (p.H / p.hk), vh = h / (p.H / p.hv);
        T* out = static_cast<T*>(p.output);
        TokenIn x, xn;
        if (!kNextUnit) load_token<T>(p, static_cast<int64_t>(seq) * p.m, h, qh, kh, vh, v0, c0, xn);
        for (int32_t t = 0; t < p.m; ++t) {
            const int64_t tok = static_cast<int64_t>(seq) * p.m + t;
            if (kNextUnit) {
                load_token<T>(p, tok, h, qh, kh, vh, v0, c0, x);
            } else {
                x = xn;
                if (t + 1 < p.m) load_token<T>(p, tok + 1, h, qh, kh, vh, v0, c0, xn);
            }
            if (p.l2norm) {
                const float rk = rsqrtf(
                    warp_sum(x.k[0] * x.k[0] + x.k[1] * x.k[1] + x.k[2] * x.k[2] + x.k[3] * x.k[3]) + 1e-6f);
                const float rq = rsqrtf(
                    warp_sum(x.q[0] * x.q[0] + x.q[1] * x.q[1] + x.q[2] * x.q[2] + x.q[3] * x.q[3]) + 1e-6f);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    x.k[j] *= rk;
                    x.q[j] *= rq;
                }
            }
            float o[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float su = warp_sum(S[r][0] * x.k[0] + S[r][1] * x.k[1] + S[r][2] * x.k[2] + S[r][3] * x.k[3]);
                const float w = x.b * (x.v[r] - x.a * su);
#pragma unroll
                for (int j = 0; j < 4; ++j) S[r][j] = x.a * S[r][j] + w * x.k[j];
                o[r] = p.scale * warp_sum(S[r][0] * x.q[0] + S[r][1] * x.q[1] + S[r][2] * x.q[2] + S[r][3] * x.q[3]);
            }
            if (lane == 0) store4(out + (static_cast<size_t>(tok) * p.H + h) * kHead + v0, o);
        }
        if (p.output_state) {
#pragma unroll
            for (int r = 0; r < 4; ++r)
                store4(static_cast<SD*>(p.output_state) + sbase + r * static_cast<int32_t>(p.state.s_v), S[r]);
        }
    }
}

template <typename T, typename SD>
void launch_decode_ts(const DecodeParams& p, unsigned grid, cudaStream_t stream) {
    if (p.m == 1) gdn_decode_kernel<T, SD, true><<<grid, kDecThreads, 0, stream>>>(p);
    else gdn_decode_kernel<T, SD, false><<<grid, kDecThreads, 0, stream>>>(p);
}

template <typename T>
void launch_decode_t(const DecodeParams& p, unsigned grid, cudaStream_t stream) {
    if (p.state.dtype == GDN_DTYPE_BF16) launch_decode_ts<T, __nv_bfloat16>(p, grid, stream);
    else if (p.state.dtype == GDN_DTYPE_F16) launch_decode_ts<T, __half>(p, grid, stream);
    else if (p.state.dtype == GDN_DTYPE_F8E4M3) launch_decode_ts<T, F8E4M3>(p, grid, stream);
    else if (p.state.dtype == GDN_DTYPE_F8E5M2) launch_decode_ts<T, F8E5M2>(p, grid, stream);
    else launch_decode_ts<T, float>(p, grid, stream);
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, gdn_dtype dtype, cudaStream_t stream) {
    const int64_t units = static_cast<int64_t>(p.N) * p.H;
    if (units == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                   cudaSuccess)
        return cudaErrorUnknown;
    const int64_t blocks = units < sms ? units : sms;  // persistent: one CTA of 1024 threads per SM
    const unsigned grid = static_cast<unsigned>(blocks);
    if (dtype == GDN_DTYPE_BF16) launch_decode_t<__nv_bfloat16>(p, grid, stream);
    else if (dtype == GDN_DTYPE_F16) launch_decode_t<__half>(p, grid, stream);
    else launch_decode_t<float>(p, grid, stream);
    return cudaGetLastError();
}

}  // namespace gdn
