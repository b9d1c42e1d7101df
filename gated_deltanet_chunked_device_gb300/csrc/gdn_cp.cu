// gdn_cp.cu -- context parallelism inside one GPU for batches with few
// (sequence, head) units ("FlashInfer GDN Prefill 完全指南", the CP routing and
// max_seqlen rows of the API table; "GDN与线性注意力GPU并行实现", the
// per-block transfer (M, N) and the scan over the blocks of section 3.3).
//
// Each sequence is cut into P segments of Ls tokens (Ls a multiple of 64, or
// of the checkpoint interval).  Over one segment the chunk recurrence is
// affine in the state it starts from, S_end = S_start M + N, because every
// chunk maps S to S (gamma_63 I - W~^T D K) + U~^T D K.  So:
//   1. a transfer pass (the chunk kernel's kTransfer instance) runs segments
//      0 .. P-2 of every sequence twice: from zero (N) and from the identity
//      with U = 0 (M); the units are independent, so they fill the GPU;
//   2. cp_fixup_kernel scans the segments in order on CUDA cores in fp32:
//      S_start(0) = the initial state, S_start(s+1) = S_start(s) M_s + N_s;
//   3. the ordinary chunk kernel runs all P segments as separate sequences
//      from those start states (outputs and checkpoints land where the whole
//      sequence would put them), and cp_final_kernel copies each sequence's
//      last segment's final state to the caller's output state.
// The work is about (2 (P-1) + P) / P times a plain pass, spread over
// P times as many units.
#include <atomic>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kCpThreads = 256;
constexpr int kLdS = kHead + 1;  // padded rows of the running state in shared memory

// Segments of every sequence, the segment pass's cu_seqlens and checkpoint
// starts, and the transfer pass's work order.  One CTA (N <= 256 here).
__global__ void __launch_bounds__(kCpThreads) cp_prepare_kernel(const CpParams p) {
    const int P = p.P;
    for (int i = threadIdx.x; i < p.num_seqs; i += blockDim.x) {
        const int64_t t0 = load_index(p.cu_seqlens, p.cu_i64, i);
        int64_t L = load_index(p.cu_seqlens, p.cu_i64, i + 1) - t0;
        if (L < 0) L = 0;  // a bad cu_seqlens is flagged by the prepare kernel; keep the segments sane
        const int64_t per = (L + P - 1) / P;
        const int64_t Ls = (per + p.align - 1) / p.align * p.align;
        const int64_t c0 = p.ckpt_n > 0 ? load_index(p.ckpt_cu_starts, p.ckpt_i64, i) : 0;
        for (int s = 0; s < P; ++s) {
            const int64_t a = s * Ls < L ? s * Ls : L;
            const int64_t b = (s + 1) * Ls < L ? (s + 1) * Ls : L;
            if (s < P - 1) {
                const int j = i * (P - 1) + s;
                p.seg_a[2 * j] = t0 + a;
                p.seg_a[2 * j + 1] = b - a;
                p.order_a[j] = j;
            }
            p.cu_c[i * P + s] = static_cast<int32_t>(t0 + a);
            p.ckpt_c[i * P + s] = p.ckpt_n > 0 ? c0 + a / p.ckpt_n : 0;
        }
    }
    if (threadIdx.x == 0) {
        p.cu_c[p.num_seqs * P] = static_cast<int32_t>(load_index(p.cu_seqlens, p.cu_i64, p.num_seqs));
        p.ckpt_c[p.num_seqs * P] = p.ckpt_n > 0 ? load_index(p.ckpt_cu_starts, p.ckpt_i64, p.num_seqs) : 0;
        *p.counter_a = 0;
    }
}

__device__ __forceinline__ int64_t real_row(const CpParams& p, int32_t i) {
    return p.state_indices ? load_index(p.state_indices, p.idx_i64, i) : i;
}

// One CTA per (sequence, state head): the start states of its P segments, in
// fp32.  Thread t owns row v = t / 2, columns 64 (t % 2) .. + 63 of S.
__global__ void __launch_bounds__(kCpThreads) cp_fixup_kernel(const CpParams p) {
    extern __shared__ float cp_smem[];
    float* S = cp_smem;                 // [128][kLdS]
    float* M = cp_smem + kHead * kLdS;  // [128][128]
    if (*reinterpret_cast<volatile int32_t*>(p.status)) return;
    const int32_t i = blockIdx.x / p.H, h = blockIdx.x % p.H;
    const int P = p.P;
    const int64_t nA = static_cast<int64_t>(p.num_seqs) * (P - 1);  // transfer rows per kind
    const size_t plane = static_cast<size_t>(kHead) * kHead;
    const int t = threadIdx.x, v = t >> 1, c0 = (t & 1) * 64;
    // S_start(0): the caller's initial state (or zeros), in any layout and type
    const int64_t srow = real_row(p, i);
    float* out0 = p.start + (static_cast<size_t>(i) * P * p.H + h) * plane;
    for (int e = 4 * t; e < kHead * kHead; e += 4 * kCpThreads) {
        const int r = e / kHead, k = e % kHead;
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        if (p.initial_state) state_load4(p.initial_state, state_offset(p.state, srow, h, r) + k, p.state.dtype, x);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            S[r * kLdS + k + j] = x[j];
            out0[static_cast<size_t>(r) * kHead + k + j] = x[j];
        }
    }
    __syncthreads();
    for (int s = 0; s + 1 < P; ++s) {
        const int64_t j = static_cast<int64_t>(i) * (P - 1) + s;
        const float* Nm = p.trans + (static_cast<size_t>(j) * p.H + h) * plane;
        const float* Mm = p.trans + (static_cast<size_t>(nA + j) * p.H + h) * plane;
        for (int e = 4 * t; e < kHead * kHead; e += 4 * kCpThreads)
            *reinterpret_cast<float4*>(M + e) = *reinterpret_cast<const float4*>(Mm + e);
        __syncthreads();
        float acc[64];
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
            const float4 n4 = *reinterpret_cast<const float4*>(Nm + static_cast<size_t>(v) * kHead + c0 + c);
            acc[c] = n4.x;
            acc[c + 1] = n4.y;
            acc[c + 2] = n4.z;
            acc[c + 3] = n4.w;
        }
#pragma unroll 2
        for (int k = 0; k < kHead; ++k) {
            const float sv = S[v * kLdS + k];
            const float4* mr = reinterpret_cast<const float4*>(M + k * kHead + c0);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const float4 m4 = mr[c];
                acc[4 * c] = fmaf(sv, m4.x, acc[4 * c]);
                acc[4 * c + 1] = fmaf(sv, m4.y, acc[4 * c + 1]);
                acc[4 * c + 2] = fmaf(sv, m4.z, acc[4 * c + 2]);
                acc[4 * c + 3] = fmaf(sv, m4.w, acc[4 * c + 3]);
            }
        }
        __syncthreads();  // every row of S has been read
        float* outs = p.start + ((static_cast<size_t>(i) * P + s + 1) * p.H + h) * plane + static_cast<size_t>(v) * kHead;
#pragma unroll
        for (int c = 0; c < 64; ++c) S[v * kLdS + c0 + c] = acc[c];
#pragma unroll
        for (int c = 0; c < 64; c += 4)
            *reinterpret_cast<float4*>(outs + c0 + c) = make_float4(acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
        __syncthreads();
    }
}

// One CTA per (sequence, state head): the last segment's final state (left in
// place by the segment pass) to the caller's output state.
__global__ void __launch_bounds__(kCpThreads) cp_final_kernel(const CpParams p) {
    if (*reinterpret_cast<volatile int32_t*>(p.status)) return;
    const int32_t i = blockIdx.x / p.H, h = blockIdx.x % p.H;
    const size_t plane = static_cast<size_t>(kHead) * kHead;
    const float* src = p.start + ((static_cast<size_t>(i) * p.P + p.P - 1) * p.H + h) * plane;
    const int64_t srow = real_row(p, i);
    for (int e = 4 * threadIdx.x; e < kHead * kHead; e += 4 * kCpThreads) {
        const int r = e / kHead, k = e % kHead;
        const float4 f = *reinterpret_cast<const float4*>(src + e);
        const float x[4] = {f.x, f.y, f.z, f.w};
        state_store4(p.output_state, state_offset(p.state, srow, h, r) + k, p.state.dtype, x);
    }
}

constexpr size_t kFixupSmem = sizeof(float) * (kHead * kLdS + kHead * kHead);

}  // namespace

cudaError_t launch_cp_prepare(const CpParams& p, cudaStream_t stream) {
    cp_prepare_kernel<<<1, kCpThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_cp_fixup(const CpParams& p, cudaStream_t stream) {
    // One flag per device: the attribute is set once, and concurrent first calls from several host threads
    // each set it at most once more (the same value).
    constexpr int kMaxDevices = 64;
    static std::atomic<uint8_t> configured[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!configured[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(cp_fixup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kFixupSmem));
        if (e != cudaSuccess) return e;
        configured[dev].store(1, std::memory_order_release);
    }
    cp_fixup_kernel<<<p.num_seqs * p.H, kCpThreads, kFixupSmem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_cp_final(const CpParams& p, cudaStream_t stream) {
    if (!p.output_state) return cudaSuccess;
    cp_final_kernel<<<p.num_seqs * p.H, kCpThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
