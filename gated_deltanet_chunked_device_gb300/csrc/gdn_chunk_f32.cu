// gdn_chunk_f32.cu -- chunked Gated DeltaNet prefill for fp32 q/k/v: the same
// 64-token chunk algebra as the tensor-core kernel, in fp32 on CUDA cores.
//
// fp32 inputs are held to a 1e-3 bar; tf32 tensor-core operands (10-bit
// mantissa) would sit close to it, and 4-byte operand tiles of the fused
// tensor-core kernel do not fit in shared memory.  This kernel keeps every
// product in fp32.  One CTA owns (sequence, state head, a slice of the V rows):
// rows of the state are independent (S[v,:] only meets v_t[v] and Delta[:,v]),
// so the slices of a head run in parallel and each recomputes the
// slice-independent parts (A, T, W, P).
//
// Per chunk ("GDN 与 Chunked Prefill": cumsum, triangular solve, recompute):
//   G = running sum of log alpha, gamma = e^G
//   A_ij = beta_i e^{G_i - G_j} (k_i.k_j)  j < i;   T = (I + A)^-1
//   W = T diag(beta gamma) K,  U = T diag(beta) V
//   Delta = U - W S^T
//   O_i = scale (gamma_i S q_i + sum_{j<=i} e^{G_i - G_j} (q_i.k_j) Delta_j)
//   S <- gamma_63 S + sum_j e^{G_63 - G_j} Delta_j k_j^T
#include <atomic>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kF32Threads = 512;
static_assert(kF32Threads == 2 * 64 * 4, "the q/k norms take four threads for each of the 2 x 64 rows");
constexpr int kLdK = 132;        // padded row stride for 128-wide rows: 16-byte aligned, and eight rows of a
                                 // 16-byte column fall in eight different bank groups
constexpr int kLdV = 65;         // padded row stride for rows of up to 64

// shared memory layout (floats) for kVs rows of V (and of the state) per CTA
template <int kVs>
struct F32Layout {
    static constexpr int kOffK = 0;                       // K  [64][kLdK]
    static constexpr int kOffQ = kOffK + 64 * kLdK;       // Q  [64][kLdK]
    static constexpr int kOffW = kOffQ + 64 * kLdK;       // W  [64][kLdK]
    static constexpr int kOffS = kOffW + 64 * kLdK;       // S slice [kVs v][kLdK]
    static constexpr int kOffV = kOffS + kVs * kLdK;      // V slice [64 j][kLdV]
    static constexpr int kOffX = kOffV + 64 * kLdV;       // U, then Delta [64 j][kLdV]
    static constexpr int kOffA = kOffX + 64 * kLdV;       // A, then P [64][kLdV]
    static constexpr int kOffT = kOffA + 64 * kLdV;       // T = (I + A)^-1 [64][kLdV]
    static constexpr int kOffG = kOffT + 64 * kLdV;       // G[64], gamma[64], beta[64], dec[64], beta gamma[64]
    static constexpr size_t kBytes = sizeof(float) * (kOffG + 5 * 64);
};

// x . y over the kHead elements of two rows (16-byte aligned), four elements per load.
__device__ __forceinline__ float dot_rows(const float* x, const float* y) {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll 4
    for (int d = 0; d < kHead; d += 4) {
        const float4 a = *reinterpret_cast<const float4*>(x + d);
        const float4 b = *reinterpret_cast<const float4*>(y + d);
        s0 += a.x * b.x + a.y * b.y;
        s1 += a.z * b.z + a.w * b.w;
    }
    return s0 + s1;
}

// dot[a] = X[i0 + a] . Y[j] over the kHead elements of rows of stride kLdK (zero when `live` is false): the four
// X rows are the same for the whole warp (broadcast loads), the Y row is the lane's own, 16 bytes per load.
__device__ __forceinline__ void row4_dots(const float* X, int i0, const float* Y, int j, bool live, float (&dot)[4]) {
#pragma unroll
    for (int a = 0; a < 4; ++a) dot[a] = 0.f;
    if (!live) return;
#pragma unroll 2
    for (int d = 0; d < kHead; d += 4) {
        const float4 y = *reinterpret_cast<const float4*>(Y + j * kLdK + d);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const float4 x = *reinterpret_cast<const float4*>(X + (i0 + a) * kLdK + d);
            dot[a] += x.x * y.x + x.y * y.y + x.z * y.z + x.w * y.w;
        }
    }
}

// kSlices CTAs per (sequence, state head), each owning kHead / kSlices rows of the state.
template <int kSlices>
__global__ void __launch_bounds__(kF32Threads, 1) gdn_chunk_f32_kernel(const ChunkParams p) {
    constexpr int kVs = kHead / kSlices;
    using Lay = F32Layout<kVs>;
    extern __shared__ float sf[];
    __shared__ int s_bad;
    const int tid = threadIdx.x;
    if (tid == 0) s_bad = *reinterpret_cast<volatile int32_t*>(p.status);
    __syncthreads();
    if (s_bad) return;

    const int32_t H = p.H;
    const int64_t unit = blockIdx.x / kSlices;
    const int v0 = static_cast<int>(blockIdx.x % kSlices) * kVs;
    const int32_t seq = static_cast<int32_t>(unit / H);
    const int32_t h = static_cast<int32_t>(unit % H);
    const int qh = h / (H / p.hq), kh = h / (H / p.hk), vh = h / (H / p.hv);
    const int64_t t0 = load_index(p.cu_seqlens, p.cu_i64, seq);
    const int64_t L = load_index(p.cu_seqlens, p.cu_i64, seq + 1) - t0;
    const int64_t srow = p.state_indices ? load_index(p.state_indices, p.idx_i64, seq) : seq;
    const int64_t state_base = state_offset(p.state, srow, h, 0);  // element offset of v row 0
    const float* qg = static_cast<const float*>(p.q);
    const float* kg = static_cast<const float*>(p.k);
    const float* vg = static_cast<const float*>(p.v);
    float* og = static_cast<float*>(p.output);

    float* Ks = sf + Lay::kOffK;
    float* Qs = sf + Lay::kOffQ;
    float* Ws = sf + Lay::kOffW;
    float* Ss = sf + Lay::kOffS;
    float* Vs = sf + Lay::kOffV;
    float* Xs = sf + Lay::kOffX;
    float* Am = sf + Lay::kOffA;
    float* Ts = sf + Lay::kOffT;
    float* sG = sf + Lay::kOffG;
    float* sGam = sG + 64;
    float* sBeta = sG + 128;
    float* sDec = sG + 192;   // e^{G_63 - G_j}
    float* sWc = sG + 256;    // beta_j gamma_j

    // state slice: rows v0..v0+63 of [V][K]
    for (int e = 4 * tid; e < kVs * kHead; e += 4 * kF32Threads) {
        const int vv = e / kHead, kk = e % kHead;
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        if (p.initial_state) state_load4(p.initial_state, state_base + (v0 + vv) * p.state.s_v + kk, p.state.dtype, x);
#pragma unroll
        for (int j = 0; j < 4; ++j) Ss[vv * kLdK + kk + j] = x[j];
    }
    __syncthreads();

    const int64_t nC = (L + kChunk - 1) / kChunk;
    for (int64_t c = 0; c < nC; ++c) {
        const int64_t tc = t0 + c * kChunk;
        const int Lc = static_cast<int>(L - c * kChunk < kChunk ? L - c * kChunk : kChunk);
        // ---- load the chunk (padded rows: zeros), L2-normalise q and k rows when asked
        {   // 16 bytes per load, every load of the thread issued before its stores
            constexpr int kPer = kChunk * kHead / 4 / kF32Threads;
            float4 kv[kPer], qv[kPer];
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int e = 4 * (tid + u * kF32Threads), r = e / kHead, d = e % kHead;
                const bool ok = r < Lc;
                const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
                kv[u] = ok ? *reinterpret_cast<const float4*>(kg + (static_cast<size_t>(tc + r) * p.hk + kh) * kHead + d) : z;
                qv[u] = ok ? *reinterpret_cast<const float4*>(qg + (static_cast<size_t>(tc + r) * p.hq + qh) * kHead + d) : z;
            }
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int e = 4 * (tid + u * kF32Threads), r = e / kHead, d = e % kHead;
                *reinterpret_cast<float4*>(Ks + r * kLdK + d) = kv[u];
                *reinterpret_cast<float4*>(Qs + r * kLdK + d) = qv[u];
            }
        }
        for (int e = tid; e < kChunk * kVs; e += kF32Threads) {
            const int r = e / kVs, d = e % kVs;
            Vs[r * kLdV + d] = r < Lc ? vg[(static_cast<size_t>(tc + r) * p.hv + vh) * kHead + v0 + d] : 0.f;
        }
        __syncthreads();
        if (p.l2norm) {
            // four threads per row (elements d = part, part + 4, ...: the rows' 4-float stride offset keeps the
            // 32 lanes of a load in 32 banks), combined by shuffles
            const int row = tid >> 2, part = tid & 3;
            float* r = (row < kChunk ? Ks : Qs) + (row & 63) * kLdK + part;
            float ss = 0.f;
#pragma unroll 8
            for (int d = 0; d < kHead; d += 4) ss += r[d] * r[d];
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            ss += __shfl_xor_sync(0xffffffffu, ss, 2);
            const float inv = 1.0f / sqrtf(ss + 1e-6f);
#pragma unroll 8
            for (int d = 0; d < kHead; d += 4) r[d] *= inv;
        }
        // ---- gates (warp 0: two rows per lane, shuffle scan of log alpha)
        if (tid < 32) {
            const int r0 = 2 * tid, r1 = r0 + 1;
            float la0 = 0.f, la1 = 0.f, b0 = 0.f, b1 = 0.f;
            if (r0 < Lc) {
                const size_t gi = static_cast<size_t>(tc + r0) * H + h;
                la0 = p.g ? logf(p.g[gi]) : 0.f;
                b0 = p.beta ? p.beta[gi] : 1.f;
            }
            if (r1 < Lc) {
                const size_t gi = static_cast<size_t>(tc + r1) * H + h;
                la1 = p.g ? logf(p.g[gi]) : 0.f;
                b1 = p.beta ? p.beta[gi] : 1.f;
            }
            float incl = la0 + la1;
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, o);
                if (tid >= o) incl += y;
            }
            const float g63 = __shfl_sync(0xffffffffu, incl, 31);
            sG[r0] = incl - la1;
            sG[r1] = incl;
            sGam[r0] = expf(incl - la1);
            sGam[r1] = expf(incl);
            sBeta[r0] = b0;
            sBeta[r1] = b1;
            sDec[r0] = expf(g63 - (incl - la1));
            sDec[r1] = expf(g63 - incl);
            sWc[r0] = b0 * sGam[r0];
            sWc[r1] = b1 * sGam[r1];
        }
        __syncthreads();
        // ---- A (strictly lower): rows i0 .. i0 + 3 against row j per thread, four k elements per load
        for (int e = tid; e < kChunk * kChunk / 4; e += kF32Threads) {
            const int i0 = 4 * (e / kChunk), j = e % kChunk;
            float dot[4];
            row4_dots(Ks, i0, Ks, j, j < i0 + 3, dot);
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int i = i0 + a;
                Am[i * kLdV + j] = j < i ? sBeta[i] * expf(sG[i] - sG[j]) * dot[a] : 0.f;
            }
        }
        __syncthreads();
        // ---- T = (I + A)^-1 by forward substitution, column j on thread j, held in registers (the loops are
        //      unrolled, so the row's A entries, the same for every thread, load ahead of the running sums; the
        //      terms above the diagonal are exact zeros)
        if (tid < kChunk) {
            const int j = tid;
            float t[kChunk];
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                float a0 = (i == j) ? 1.f : 0.f, a1 = 0.f;
#pragma unroll
                for (int m = 0; m + 1 < i; m += 2) {
                    a0 -= Am[i * kLdV + m] * t[m];
                    a1 -= Am[i * kLdV + m + 1] * t[m + 1];
                }
                if (i & 1) a0 -= Am[i * kLdV + i - 1] * t[i - 1];
                t[i] = (i < j) ? 0.f : a0 + a1;
            }
#pragma unroll
            for (int i = 0; i < kChunk; ++i) Ts[i * kLdV + j] = t[i];
        }
        __syncthreads();
        // ---- W = T diag(beta gamma) K: rows i0 .. i0 + 3 and four k elements per thread (T is zero above its
        //      diagonal, so every row of the group runs to i0 + 3),  U = T diag(beta) V_slice
        for (int e = tid; e < kChunk * kHead / 16; e += kF32Threads) {
            const int i0 = 4 * (e / (kHead / 4)), d = 4 * (e % (kHead / 4));
            float4 acc[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) acc[a] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
            for (int j = 0; j <= i0 + 3; ++j) {
                const float wc = sWc[j];
                const float4 kj = *reinterpret_cast<const float4*>(Ks + j * kLdK + d);
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    const float t = Ts[(i0 + a) * kLdV + j] * wc;
                    acc[a].x += t * kj.x;
                    acc[a].y += t * kj.y;
                    acc[a].z += t * kj.z;
                    acc[a].w += t * kj.w;
                }
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) *reinterpret_cast<float4*>(Ws + (i0 + a) * kLdK + d) = acc[a];
        }
        for (int e = tid; e < kChunk * kVs; e += kF32Threads) {
            const int i = e / kVs, d = e % kVs;
            float acc = 0.f;
#pragma unroll 4
            for (int j = 0; j <= i; ++j) acc += Ts[i * kLdV + j] * sBeta[j] * Vs[j * kLdV + d];
            Xs[i * kLdV + d] = acc;
        }
        __syncthreads();
        if (p.intra_w && v0 == 0) {
            const size_t base = (static_cast<size_t>(p.chunk_offsets[seq] + c) * H + h) * kChunk * kHead;
            for (int e = tid; e < kChunk * kHead; e += kF32Threads)
                p.intra_w[base + e] = Ws[(e / kHead) * kLdK + e % kHead];
        }
        if (p.intra_u) {
            const size_t base = (static_cast<size_t>(p.chunk_offsets[seq] + c) * H + h) * kChunk * kHead;
            for (int e = tid; e < kChunk * kVs; e += kF32Threads)
                p.intra_u[base + (e / kVs) * kHead + v0 + e % kVs] = Xs[(e / kVs) * kLdV + e % kVs];
        }
        if (p.intra_g && v0 == 0 && tid < kChunk)
            p.intra_g[(static_cast<size_t>(p.chunk_offsets[seq] + c) * H + h) * kChunk + tid] = sG[tid];
        // ---- Delta = U - W S^T (slice columns), in place over U; four k elements per load
        for (int e = tid; e < kChunk * kVs; e += kF32Threads) {
            const int i = e / kVs, vv = e % kVs;
            Xs[i * kLdV + vv] -= dot_rows(Ws + i * kLdK, Ss + vv * kLdK);
        }
        __syncthreads();
        // ---- P_ij = e^{G_i - G_j} (q_i . k_j) for j <= i, over A: rows i0 .. i0 + 3 per thread
        for (int e = tid; e < kChunk * kChunk / 4; e += kF32Threads) {
            const int i0 = 4 * (e / kChunk), j = e % kChunk;
            float dot[4];
            row4_dots(Qs, i0, Ks, j, j <= i0 + 3, dot);
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int i = i0 + a;
                Am[i * kLdV + j] = j <= i ? expf(sG[i] - sG[j]) * dot[a] : 0.f;
            }
        }
        __syncthreads();
        // ---- output rows of the slice
        for (int e = tid; e < kChunk * kVs; e += kF32Threads) {
            const int i = e / kVs, vv = e % kVs;
            if (i >= Lc) continue;
            float acc = sGam[i] * dot_rows(Ss + vv * kLdK, Qs + i * kLdK);
#pragma unroll 4
            for (int j = 0; j <= i; ++j) acc += Am[i * kLdV + j] * Xs[j * kLdV + vv];
            og[(static_cast<size_t>(tc + i) * H + h) * kHead + v0 + vv] = p.scale * acc;
        }
        __syncthreads();
        // ---- state: S <- gamma_63 S + sum_j e^{G_63 - G_j} Delta_j k_j^T, four k elements per thread
        {
            const float eg63 = sGam[kChunk - 1];
            for (int e = tid; e < kVs * kHead / 4; e += kF32Threads) {
                const int vv = e / (kHead / 4), d = 4 * (e % (kHead / 4));
                float4 acc = *reinterpret_cast<const float4*>(Ss + vv * kLdK + d);
                acc = make_float4(eg63 * acc.x, eg63 * acc.y, eg63 * acc.z, eg63 * acc.w);
#pragma unroll 4
                for (int j = 0; j < kChunk; ++j) {
                    const float x = sDec[j] * Xs[j * kLdV + vv];
                    const float4 kj = *reinterpret_cast<const float4*>(Ks + j * kLdK + d);
                    acc.x += x * kj.x;
                    acc.y += x * kj.y;
                    acc.z += x * kj.z;
                    acc.w += x * kj.w;
                }
                *reinterpret_cast<float4*>(Ss + vv * kLdK + d) = acc;
            }
        }
        __syncthreads();
        // ---- checkpoint at the chunk end
        const int64_t pend = (c + 1) * kChunk;
        if (p.checkpoints && p.ckpt_n > 0 && pend % p.ckpt_n == 0 && pend <= L) {
            const int64_t slot = load_index(p.ckpt_cu_starts, p.ckpt_i64, seq) + pend / p.ckpt_n - 1;
            const int64_t ck = (slot * H + h) * static_cast<int64_t>(kHead * kHead);  // dense row, ckpt_dtype
            for (int e = 4 * tid; e < kVs * kHead; e += 4 * kF32Threads) {
                const int vv = e / kHead, kk = e % kHead;
                const float x[4] = {Ss[vv * kLdK + kk], Ss[vv * kLdK + kk + 1], Ss[vv * kLdK + kk + 2],
                                    Ss[vv * kLdK + kk + 3]};
                state_store4(p.checkpoints, ck + static_cast<int64_t>(v0 + vv) * kHead + kk, p.ckpt_dtype, x);
            }
        }
    }
    if (p.output_state) {
        for (int e = 4 * tid; e < kVs * kHead; e += 4 * kF32Threads) {
            const int vv = e / kHead, kk = e % kHead;
            const float x[4] = {Ss[vv * kLdK + kk], Ss[vv * kLdK + kk + 1], Ss[vv * kLdK + kk + 2],
                                Ss[vv * kLdK + kk + 3]};
            state_store4(p.output_state, state_base + (v0 + vv) * p.state.s_v + kk, p.state.dtype, x);
        }
    }
}

template <int kSlices>
cudaError_t launch_slices(const ChunkParams& p, int64_t units, cudaStream_t stream) {
    // One flag per device and instance: the attribute is set once, and concurrent first calls from several host
    // threads each set it at most once more (the same value).
    constexpr int kMaxDevices = 64;
    constexpr size_t kSmem = F32Layout<kHead / kSlices>::kBytes;
    static std::atomic<uint8_t> configured[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!configured[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(gdn_chunk_f32_kernel<kSlices>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmem));
        if (e != cudaSuccess) return e;
        configured[dev].store(1, std::memory_order_release);
    }
    if (units * kSlices > 0x7fffffffLL) return cudaErrorInvalidValue;
    gdn_chunk_f32_kernel<kSlices><<<static_cast<int>(units * kSlices), kF32Threads, kSmem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_f32(const ChunkParams& p, int64_t units, int slices, cudaStream_t stream) {
    switch (slices) {
        case 2: return launch_slices<2>(p, units, stream);
        case 4: return launch_slices<4>(p, units, stream);
        case 8: return launch_slices<8>(p, units, stream);
        case 16: return launch_slices<16>(p, units, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
