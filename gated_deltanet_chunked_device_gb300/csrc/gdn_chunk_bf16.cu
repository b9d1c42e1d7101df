// gdn_chunk_bf16.cu -- chunked Gated DeltaNet prefill, bf16 q/k/v, fp32 state,
// tcgen05 tensor cores with TMEM accumulators and TMA-fed operands (sm_103a).
//
// One CTA runs one work unit (sequence i, state head h) at a time and walks
// the sequence's 64-token chunks in order; persistent CTAs take units from an
// atomic counter in longest-first order.  Per chunk (notation: C = 64 rows,
// G_r = sum_{m<=r} log alpha_m inside the chunk, gamma_r = exp(G_r)):
//
//   intra-chunk step ("GDN 与 Chunked Prefill": cumsum, triangular solve,
//   recompute; the 4-token table generalised to the 64 x 64 decay table):
//     D1 = [K; Q] K^T                                  (tcgen05, M=128 N=64 K=128)
//     A_ij = beta_i e^{G_i-G_j} (k_i.k_j), j < i      (CUDA cores)
//     P_ij = e^{G_i-G_j} (q_i.k_j), j <= i            (CUDA cores)
//     T = (I + A)^-1                                   (blocked forward substitution)
//     W^T = K^T (T diag(beta gamma))^T,  U^T = V^T (T diag(beta))^T   (tcgen05)
//   state pass ("块内 state 和块间 final state": only the chunk's last state
//   crosses the boundary):
//     Delta^T = U^T - S W^T                            (tcgen05, A negated)
//     S <- gamma_63 S + (Delta^T diag(e^{G_63-G_j})) K (tcgen05, accumulate in TMEM)
//   output ("GDN与线性注意力GPU并行实现" section 3.3: O_init = Q S plus a
//   triangular-masked product):
//     O^T = scale (S Q^T diag(gamma) + Delta^T P^T)    (tcgen05, two accumulators)
//
// Operand layouts (all 128-byte swizzled, verified against torch matmul):
//   K, Q, V tiles arrive by TMA as [64 rows][64 cols] boxes; the same K tile
//   serves as K-major A/B ([K;Q]K^T), MN-major A (K^T ...) and MN-major B
//   (... K), so no transposed copy is made.  S, Delta^T, P and T' are written
//   by threads in K-major form; W^T is written MN-major.
// TMEM (512 columns): S [0,128), D1 [128,192), W^T [192,256), Delta^T [256,320),
//   S Q^T [320,384), Delta^T P^T [384,448).  Thread t owns TMEM lane t.
#include <cuda_bf16.h>

#include "gdn_internal.cuh"
#include "sm103_ptx.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 128;

// Shared memory map (bytes from a 1024-aligned base).
constexpr uint32_t kStageBytes = 49152;          // K_h0 | Q_h0 | K_h1 | Q_h1 | V_h0 | V_h1 (8 KB each)
constexpr uint32_t kOffKQ = 0;                   // inside a stage
constexpr uint32_t kOffV = 32768;                // inside a stage
constexpr uint32_t kSmTp = 2 * kStageBytes;      // T diag(beta gamma), bf16 [64 i][64 j] K-major
constexpr uint32_t kSmTpp = kSmTp + 8192;        // T diag(beta)
constexpr uint32_t kSmP = kSmTpp + 8192;         // P, bf16 [64 i][64 j] K-major
constexpr uint32_t kSmWb = kSmP + 8192;          // W^T bf16 MN-major B: [128 k rows][64 i]
constexpr uint32_t kSmSb = kSmWb + 16384;        // S bf16 K-major: 2 halves of [128 v][64 k]
constexpr uint32_t kSmDb = kSmSb + 32768;        // Delta^T bf16 K-major [128 v][64 j]; A fp32 before
constexpr uint32_t kSmDtb = kSmDb + 16384;       // decayed Delta^T; T fp32 before
constexpr uint32_t kSmSmall = kSmDtb + 16384;
constexpr uint32_t kSmG = kSmSmall;              // float[64]
constexpr uint32_t kSmGam = kSmG + 256;          // float[64]
constexpr uint32_t kSmBeta = kSmGam + 256;       // float[64]
constexpr uint32_t kSmBar = kSmBeta + 256;       // 3 x uint64 mbarriers: tma[0], tma[1], mma
constexpr uint32_t kSmMisc = kSmBar + 32;        // tmem base, unit id, abort flag
constexpr uint32_t kSmemBytes = kSmMisc + 32;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;

constexpr uint32_t kTmS = 0, kTmD1 = 128, kTmW = 192, kTmDelta = 256, kTmO1 = 320, kTmO2 = 384;
constexpr uint32_t kTmCols = 512;

constexpr uint32_t kIdescD1 = idesc_bf16_f32(128, 64);                       // [K;Q] K^T, S Q^T
constexpr uint32_t kIdescWU = idesc_bf16_f32(128, 64, true, false);          // K^T T'^T, V^T T''^T
constexpr uint32_t kIdescDelta = idesc_bf16_f32(128, 64, false, true, true); // -S W^T
constexpr uint32_t kIdescO2 = idesc_bf16_f32(128, 64);                       // Delta^T P^T
constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, true);          // Delta~^T K

__device__ __forceinline__ void tmem_ld16_f(uint32_t taddr, float* out) {
    uint32_t r[16];
    tmem_ld16(taddr, r);
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15])
                 :
                 : "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) out[j] = __uint_as_float(r[j]);
}

// Write 8 floats as one bf16 16-byte chunk of a 128B-swizzled row.
__device__ __forceinline__ void st_chunk_bf16(uint8_t* tile, uint32_t row, uint32_t chunk, const float* x) {
    uint4 v;
    v.x = pack_bf16x2(x[0], x[1]);
    v.y = pack_bf16x2(x[2], x[3]);
    v.z = pack_bf16x2(x[4], x[5]);
    v.w = pack_bf16x2(x[6], x[7]);
    *reinterpret_cast<uint4*>(tile + sw128_offset(row, chunk)) = v;
}

__device__ __forceinline__ void bf16x8_to_float(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        f[2 * j] = __uint_as_float(w[j] << 16);
        f[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
}

// A row of 128 bf16 values held as two 64-column swizzled halves 16 KB apart
// (the stage layout K_h0 | Q_h0 | K_h1 | Q_h1 puts K_h1 16 KB after K_h0).
// Zero it when `zero`, else L2-normalise it in place when `norm`.
__device__ __forceinline__ void fix_row(uint8_t* half0, uint32_t half_stride, uint32_t row, bool zero, bool norm) {
    if (zero) {
        const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int c = 0; c < 16; ++c)
            *reinterpret_cast<uint4*>(half0 + (c >> 3) * half_stride + sw128_offset(row, c & 7)) = z;
        return;
    }
    if (!norm) return;
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        float f[8];
        bf16x8_to_float(*reinterpret_cast<const uint4*>(half0 + (c >> 3) * half_stride + sw128_offset(row, c & 7)), f);
#pragma unroll
        for (int j = 0; j < 8; ++j) ss += f[j] * f[j];
    }
    const float inv = rsqrtf(ss + 1e-6f);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        uint8_t* p = half0 + (c >> 3) * half_stride + sw128_offset(row, c & 7);
        float f[8];
        bf16x8_to_float(*reinterpret_cast<const uint4*>(p), f);
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] *= inv;
        st_chunk_bf16(half0 + (c >> 3) * half_stride, row, c & 7, f);
    }
}

// T = (I + A)^-1 for a strictly lower 64 x 64 A (fp32, row-major): 16 x 16
// diagonal blocks by forward substitution, then the block formula
// T_ab = -T_aa A_ab T_bb at 16 and at 32 granularity.  Upper-triangular
// storage of T is used as scratch and is garbage on return.
__device__ void tri_inverse_64(const float* __restrict__ A, float* __restrict__ T, int tid) {
    if (tid < 64) {
        const int o = (tid >> 4) * 16, col = tid & 15;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = (r == col) ? 1.f : 0.f;
#pragma unroll
            for (int m = 0; m < r; ++m) acc -= A[(o + r) * 64 + o + m] * x[m];
            x[r] = (r < col) ? 0.f : acc;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) T[(o + r) * 64 + o + col] = x[r];
    }
    __syncthreads();
    {   // level 1, step 1: X_ab = A_ab T_bb for (a, b) = (1, 0), (3, 2); kept at block (b, a)
        const int pr = tid >> 6, a = 2 * pr + 1, b = 2 * pr;
        const int idx = tid & 63, r = idx >> 2, c0 = (idx & 3) * 4;
        float x[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const float av = A[(16 * a + r) * 64 + 16 * b + m];
#pragma unroll
            for (int q = 0; q < 4; ++q) x[q] += av * T[(16 * b + m) * 64 + 16 * b + c0 + q];
        }
        __syncthreads();
#pragma unroll
        for (int q = 0; q < 4; ++q) T[(16 * b + r) * 64 + 16 * a + c0 + q] = x[q];
        __syncthreads();
        // step 2: T_ab = -T_aa X_ab
        float y[4] = {0.f, 0.f, 0.f, 0.f};
        for (int m = 0; m <= r; ++m) {
            const float tv = T[(16 * a + r) * 64 + 16 * a + m];
#pragma unroll
            for (int q = 0; q < 4; ++q) y[q] += tv * T[(16 * b + m) * 64 + 16 * a + c0 + q];
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) T[(16 * a + r) * 64 + 16 * b + c0 + q] = -y[q];
    }
    __syncthreads();
    {   // level 2: T_21 = -T_22 A_21 T_11 on 32 x 32 blocks; X kept at rows 0..31, cols 32..63
        const int r = tid >> 2, c0 = (tid & 3) * 8;
        float x[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) x[q] = 0.f;
        for (int m = 0; m < 32; ++m) {
            const float av = A[(32 + r) * 64 + m];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float tv = (m >= c0 + q) ? T[m * 64 + c0 + q] : 0.f;  // T_11 is lower triangular
                x[q] += av * tv;
            }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) T[r * 64 + 32 + c0 + q] = x[q];
        __syncthreads();
        float y[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) y[q] = 0.f;
        for (int m = 0; m <= r; ++m) {
            const float tv = T[(32 + r) * 64 + 32 + m];
#pragma unroll
            for (int q = 0; q < 8; ++q) y[q] += tv * T[m * 64 + 32 + c0 + q];
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) T[(32 + r) * 64 + c0 + q] = -y[q];
    }
    __syncthreads();
}

struct Bars {
    uint64_t* tma[2];
    uint64_t* mma;
};

__device__ __forceinline__ void issue_chunk_loads(uint8_t* stage, uint64_t* bar, const CUtensorMap* tq,
                                                  const CUtensorMap* tk, const CUtensorMap* tv, int qh, int kh, int vh,
                                                  int32_t t) {
    mbar_arrive_expect_tx(bar, kStageBytes);
    tma_load_3d(stage + kOffKQ + 0, tk, bar, 0, kh, t);
    tma_load_3d(stage + kOffKQ + 8192, tq, bar, 0, qh, t);
    tma_load_3d(stage + kOffKQ + 16384, tk, bar, 64, kh, t);
    tma_load_3d(stage + kOffKQ + 24576, tq, bar, 64, qh, t);
    tma_load_3d(stage + kOffV + 0, tv, bar, 0, vh, t);
    tma_load_3d(stage + kOffV + 8192, tv, bar, 64, vh, t);
}

__global__ void __launch_bounds__(kThreads, 1)
    gdn_chunk_bf16_kernel(const ChunkParams p, const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5;

    float* sG = reinterpret_cast<float*>(sm + kSmG);
    float* sGam = reinterpret_cast<float*>(sm + kSmGam);
    float* sBeta = reinterpret_cast<float*>(sm + kSmBeta);
    Bars bars;
    bars.tma[0] = reinterpret_cast<uint64_t*>(sm + kSmBar);
    bars.tma[1] = bars.tma[0] + 1;
    bars.mma = bars.tma[0] + 2;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + kSmMisc);
    int32_t* s_unit = reinterpret_cast<int32_t*>(sm + kSmMisc + 4);
    int32_t* s_abort = reinterpret_cast<int32_t*>(sm + kSmMisc + 8);
    uint8_t* stage[2] = {sm, sm + kStageBytes};
    uint8_t* sTp = sm + kSmTp;
    uint8_t* sTpp = sm + kSmTpp;
    uint8_t* sP = sm + kSmP;
    uint8_t* sWb = sm + kSmWb;
    uint8_t* sSb = sm + kSmSb;
    uint8_t* sDb = sm + kSmDb;
    uint8_t* sDtb = sm + kSmDtb;
    float* sA = reinterpret_cast<float*>(sm + kSmDb);   // aliases Delta^T (dead by then)
    float* sT = reinterpret_cast<float*>(sm + kSmDtb);  // aliases decayed Delta^T

    // Bad input flagged by the prepare kernel: every thread sees one copy of the word.
    if (tid == 0) *s_abort = *reinterpret_cast<volatile int32_t*>(p.status);
    __syncthreads();
    if (*reinterpret_cast<volatile int32_t*>(s_abort) != 0) return;
    __syncthreads();
    if (tid == 0) {
        mbar_init(bars.tma[0], 1);
        mbar_init(bars.tma[1], 1);
        mbar_init(bars.mma, 1);
        fence_mbar_init();
        *s_abort = 0;
        if (p.has_tokens) {
            prefetch_tensormap(&tm_q);
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
        }
    }
    if (warp == 0) {
        tmem_alloc(s_tmem, kTmCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tm_row = tmem + lane_base;  // this thread's TMEM lane, column 0

    uint32_t tma_phase[2] = {0u, 0u};
    uint32_t mma_phase = 0u;
    int pending[2] = {0, 0};  // TMA loads issued and not yet waited on (thread 0's view)
    const int32_t H = p.H;
    const int64_t units = static_cast<int64_t>(p.num_seqs) * H;
    bool abort = false;

    auto fail = [&](void) {
        atomicOr(p.status, static_cast<int32_t>(GDN_DEVICE_ERR_TIMEOUT));
        atomicExch(s_abort, 1);
    };
    auto wait_mma = [&](void) {
        if (!mbar_wait(bars.mma, mma_phase & 1u)) fail();
        ++mma_phase;
        tc_fence_after();
    };

    for (;;) {
        if (tid == 0) *s_unit = atomicAdd(p.counter, 1);
        __syncthreads();
        const int64_t u = *s_unit;
        const bool stop = u >= units || *reinterpret_cast<volatile int32_t*>(s_abort) != 0;
        __syncthreads();  // everyone has read s_unit before thread 0 may overwrite it
        if (stop) break;
        const int32_t seq = p.seq_order[u / H];
        const int32_t h = static_cast<int32_t>(u % H);
        const int64_t t0 = load_index(p.cu_seqlens, p.cu_i64, seq);
        const int64_t L = load_index(p.cu_seqlens, p.cu_i64, seq + 1) - t0;
        const int32_t nC = static_cast<int32_t>((L + kChunk - 1) / kChunk);
        const int qh = h / (H / p.hq), kh = h / (H / p.hk), vh = h / (H / p.hv);
        const int64_t srow = p.state_indices ? load_index(p.state_indices, p.idx_i64, seq) : seq;
        const size_t state_off = (static_cast<size_t>(srow) * H + h) * kHead * kHead;
        const int32_t flat0 = p.chunk_offsets[seq];

        // ---- start loads of the first two chunks
        if (tid == 0) {
            for (int c = 0; c < 2 && c < nC; ++c) {
                issue_chunk_loads(stage[c], bars.tma[c], &tm_q, &tm_k, &tm_v, qh, kh, vh,
                                  static_cast<int32_t>(t0 + c * kChunk));
                pending[c] = 1;
            }
        }
        // ---- initial state: row v = tid into TMEM (fp32) and smem (bf16, K-major)
        {
            const float* src = p.initial_state ? p.initial_state + state_off + static_cast<size_t>(tid) * kHead
                                               : nullptr;
            float* dst_final = (nC == 0 && p.output_state)
                                   ? p.output_state + state_off + static_cast<size_t>(tid) * kHead
                                   : nullptr;
#pragma unroll 1
            for (int c0 = 0; c0 < kHead; c0 += 16) {
                float x[16];
                if (src) {
#pragma unroll
                    for (int j = 0; j < 16; j += 4) {
                        const float4 f = *reinterpret_cast<const float4*>(src + c0 + j);
                        x[j] = f.x; x[j + 1] = f.y; x[j + 2] = f.z; x[j + 3] = f.w;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) x[j] = 0.f;
                }
                if (dst_final) {
#pragma unroll
                    for (int j = 0; j < 16; j += 4)
                        *reinterpret_cast<float4*>(dst_final + c0 + j) = make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
                }
                if (nC > 0) {
                    uint32_t r[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(x[j]);
                    tmem_st16(tm_row + kTmS + c0, r);
                    uint8_t* half = sSb + (c0 >> 6) * 16384;
                    st_chunk_bf16(half, tid, (c0 & 63) >> 3, x);
                    st_chunk_bf16(half, tid, ((c0 & 63) >> 3) + 1, x + 8);
                }
            }
            if (nC > 0) tmem_wait_st();
        }
        if (nC == 0) continue;  // zero-length sequence: state passed through

        for (int32_t c = 0; c < nC && !abort; ++c) {
            const int s = c & 1;
            uint8_t* st = stage[s];
            const int64_t tc = t0 + static_cast<int64_t>(c) * kChunk;
            const int32_t Lc = static_cast<int32_t>(L - static_cast<int64_t>(c) * kChunk < kChunk
                                                        ? L - static_cast<int64_t>(c) * kChunk
                                                        : kChunk);
            // ---- P1: gates; masking and L2 norm of the staged tiles; MMA D1 and S Q^T
            if (tid < kChunk) {
                const int r = tid;
                float la = 0.f, b = 0.f;
                if (r < Lc) {
                    const size_t gi = static_cast<size_t>(tc + r) * H + h;
                    la = p.g ? logf(p.g[gi]) : 0.f;
                    b = p.beta ? p.beta[gi] : 1.f;
                }
                float run = la;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, run, o);
                    if ((tid & 31) >= o) run += y;
                }
                sG[r] = run;
                sBeta[r] = b;
            }
            __syncthreads();
            if (tid >= 32 && tid < kChunk) sG[tid] += sG[31];
            __syncthreads();
            if (tid < kChunk) sGam[tid] = expf(sG[tid]);

            if (!mbar_wait(bars.tma[s], tma_phase[s] & 1u)) fail();
            ++tma_phase[s];
            if (tid == 0) pending[s] = 0;
            if (tid < kChunk) {
                const int r = tid;
                fix_row(st + kOffKQ, 16384, r, r >= Lc, p.l2norm != 0);   // K row
                if (r >= Lc) fix_row(st + kOffV, 8192, r, true, false);  // V row
            } else {
                const int r = tid - kChunk;
                fix_row(st + kOffKQ + 8192, 16384, r, r >= Lc, p.l2norm != 0);  // Q row
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            abort = *reinterpret_cast<volatile int32_t*>(s_abort) != 0;
            if (abort) break;
            if (tid == 0) {
                tc_fence_after();
                const uint32_t kq = smem_u32(st + kOffKQ);
                const uint32_t sb = smem_u32(sSb);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                    // [K; Q] (128 rows) x K^T (64 rows)
                    mma_bf16_ss(tmem + kTmD1, desc_kmajor_sw128(kq + off), desc_kmajor_sw128(kq + off), kIdescD1,
                                ks > 0);
                    // S (128 rows v) x Q^T (64 rows i)
                    mma_bf16_ss(tmem + kTmO1, desc_kmajor_sw128(sb + off), desc_kmajor_sw128(kq + 8192 + off),
                                kIdescD1, ks > 0);
                }
                mma_commit(bars.mma);
            }
            __syncwarp();
            wait_mma();

            // ---- P2: A (strictly lower, beta and decay) and P (causal, decay)
            {
                const int i = tid & 63;
                const float Gi = sG[i];
                const float bi = sBeta[i];
                if (tid < kChunk) {
#pragma unroll 1
                    for (int j0 = 0; j0 < kChunk; j0 += 16) {
                        float d[16];
                        tmem_ld16_f(tm_row + kTmD1 + j0, d);
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int jj = j0 + j;
                            d[j] = (jj < i) ? bi * expf(Gi - sG[jj]) * d[j] : 0.f;
                        }
#pragma unroll
                        for (int j = 0; j < 16; j += 4)
                            *reinterpret_cast<float4*>(sA + i * 64 + j0 + j) = make_float4(d[j], d[j + 1], d[j + 2], d[j + 3]);
                    }
                } else {
#pragma unroll 1
                    for (int j0 = 0; j0 < kChunk; j0 += 16) {
                        float d[16];
                        tmem_ld16_f(tm_row + kTmD1 + j0, d);
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int jj = j0 + j;
                            d[j] = (jj <= i) ? expf(Gi - sG[jj]) * d[j] : 0.f;
                        }
                        st_chunk_bf16(sP, i, j0 >> 3, d);
                        st_chunk_bf16(sP, i, (j0 >> 3) + 1, d + 8);
                    }
                }
            }
            __syncthreads();

            // ---- P3: T = (I + A)^-1; T' = T diag(beta gamma), T'' = T diag(beta); W^T, U^T
            tri_inverse_64(sA, sT, tid);
            {
                const int i = tid & 63;
                const bool wpart = tid < kChunk;
                uint8_t* dst = wpart ? sTp : sTpp;
#pragma unroll 1
                for (int j0 = 0; j0 < kChunk; j0 += 8) {
                    float x[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int jj = j0 + j;
                        const float sc = wpart ? sBeta[jj] * sGam[jj] : sBeta[jj];
                        x[j] = (jj <= i) ? sT[i * 64 + jj] * sc : 0.f;
                    }
                    st_chunk_bf16(dst, i, j0 >> 3, x);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            if (tid == 0) {
                tc_fence_after();
                const uint32_t kq = smem_u32(st + kOffKQ);
                const uint32_t vv = smem_u32(st + kOffV);
                const uint32_t tp = smem_u32(sTp), tpp = smem_u32(sTpp);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    // A = K^T: K tile read MN-major (d halves 16 KB apart); B = T' rows i, K-major over j
                    mma_bf16_ss(tmem + kTmW, desc_mnmajor_sw128(kq + ks * 2048, 16384),
                                desc_kmajor_sw128(tp + ks * 32), kIdescWU, ks > 0);
                    mma_bf16_ss(tmem + kTmDelta, desc_mnmajor_sw128(vv + ks * 2048, 8192),
                                desc_kmajor_sw128(tpp + ks * 32), kIdescWU, ks > 0);
                }
                mma_commit(bars.mma);
            }
            __syncwarp();
            wait_mma();

            // ---- P4: W^T to smem (MN-major B for -S W^T); optional dumps of G, W, U
            {
#pragma unroll 1
                for (int i0 = 0; i0 < kChunk; i0 += 16) {
                    float w[16];
                    tmem_ld16_f(tm_row + kTmW + i0, w);
                    st_chunk_bf16(sWb, tid, i0 >> 3, w);
                    st_chunk_bf16(sWb, tid, (i0 >> 3) + 1, w + 8);
                    if (p.intra_w) {
                        float* dw = p.intra_w + (static_cast<size_t>(flat0 + c) * H + h) * kChunk * kHead;
#pragma unroll
                        for (int j = 0; j < 16; ++j) dw[static_cast<size_t>(i0 + j) * kHead + tid] = w[j];
                    }
                    if (p.intra_u) {
                        float uu[16];
                        tmem_ld16_f(tm_row + kTmDelta + i0, uu);
                        float* du = p.intra_u + (static_cast<size_t>(flat0 + c) * H + h) * kChunk * kHead;
#pragma unroll
                        for (int j = 0; j < 16; ++j) du[static_cast<size_t>(i0 + j) * kHead + tid] = uu[j];
                    }
                }
                if (p.intra_g && tid < kChunk)
                    p.intra_g[(static_cast<size_t>(flat0 + c) * H + h) * kChunk + tid] = sG[tid];
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            if (tid == 0) {
                tc_fence_after();
                const uint32_t sb = smem_u32(sSb), wb = smem_u32(sWb);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t aoff = (ks >> 2) * 16384 + (ks & 3) * 32;
                    mma_bf16_ss(tmem + kTmDelta, desc_kmajor_sw128(sb + aoff), desc_mnmajor_sw128(wb + ks * 2048, 8192),
                                kIdescDelta, 1);
                }
                mma_commit(bars.mma);
            }
            __syncwarp();
            wait_mma();

            // ---- P5: Delta^T and decayed Delta^T to smem; S *= gamma_63 in TMEM
            {
                const float Glast = sG[kChunk - 1];
#pragma unroll 1
                for (int j0 = 0; j0 < kChunk; j0 += 16) {
                    float d[16], e[16];
                    tmem_ld16_f(tm_row + kTmDelta + j0, d);
#pragma unroll
                    for (int j = 0; j < 16; ++j) e[j] = d[j] * expf(Glast - sG[j0 + j]);
                    st_chunk_bf16(sDb, tid, j0 >> 3, d);
                    st_chunk_bf16(sDb, tid, (j0 >> 3) + 1, d + 8);
                    st_chunk_bf16(sDtb, tid, j0 >> 3, e);
                    st_chunk_bf16(sDtb, tid, (j0 >> 3) + 1, e + 8);
                }
                const float gl = sGam[kChunk - 1];
#pragma unroll 1
                for (int c0 = 0; c0 < kHead; c0 += 16) {
                    float x[16];
                    tmem_ld16_f(tm_row + kTmS + c0, x);
                    uint32_t r[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(x[j] * gl);
                    tmem_st16(tm_row + kTmS + c0, r);
                }
                tmem_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            if (tid == 0) {
                tc_fence_after();
                const uint32_t db = smem_u32(sDb), dtb = smem_u32(sDtb), pp = smem_u32(sP);
                const uint32_t kq = smem_u32(st + kOffKQ);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    mma_bf16_ss(tmem + kTmO2, desc_kmajor_sw128(db + ks * 32), desc_kmajor_sw128(pp + ks * 32),
                                kIdescO2, ks > 0);
                    // B = K tile read MN-major: rows j (K dim), d contiguous (N), d halves 16 KB apart
                    mma_bf16_ss(tmem + kTmS, desc_kmajor_sw128(dtb + ks * 32), desc_mnmajor_sw128(kq + ks * 2048, 16384),
                                kIdescS, 1);
                }
                mma_commit(bars.mma);
            }
            __syncwarp();
            wait_mma();

            // ---- P6: output rows, next S operand, checkpoints, final state
            {
                const float sc = p.scale;
                __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.output);
#pragma unroll 1
                for (int i0 = 0; i0 < kChunk; i0 += 16) {
                    float o1[16], o2[16];
                    tmem_ld16_f(tm_row + kTmO1 + i0, o1);
                    tmem_ld16_f(tm_row + kTmO2 + i0, o2);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int i = i0 + j;
                        if (i < Lc) {
                            const float o = sc * (sGam[i] * o1[j] + o2[j]);
                            out[(static_cast<size_t>(tc + i) * H + h) * kHead + tid] = __float2bfloat16_rn(o);
                        }
                    }
                }
                const int64_t pend = static_cast<int64_t>(c + 1) * kChunk;
                float* ck = nullptr;
                if (p.checkpoints && p.ckpt_n > 0 && pend % p.ckpt_n == 0 && pend <= L) {
                    const int64_t slot = load_index(p.ckpt_cu_starts, p.ckpt_i64, seq) + pend / p.ckpt_n - 1;
                    ck = p.checkpoints + (static_cast<size_t>(slot) * H + h) * kHead * kHead +
                         static_cast<size_t>(tid) * kHead;
                }
                float* fin = (c == nC - 1 && p.output_state)
                                 ? p.output_state + state_off + static_cast<size_t>(tid) * kHead
                                 : nullptr;
                const bool need_sb = c + 1 < nC;
#pragma unroll 1
                for (int c0 = 0; c0 < kHead; c0 += 16) {
                    float x[16];
                    tmem_ld16_f(tm_row + kTmS + c0, x);
                    if (need_sb) {
                        uint8_t* half = sSb + (c0 >> 6) * 16384;
                        st_chunk_bf16(half, tid, (c0 & 63) >> 3, x);
                        st_chunk_bf16(half, tid, ((c0 & 63) >> 3) + 1, x + 8);
                    }
                    if (ck) {
#pragma unroll
                        for (int j = 0; j < 16; j += 4)
                            *reinterpret_cast<float4*>(ck + c0 + j) = make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
                    }
                    if (fin) {
#pragma unroll
                        for (int j = 0; j < 16; j += 4)
                            *reinterpret_cast<float4*>(fin + c0 + j) = make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            if (tid == 0 && c + 2 < nC) {
                issue_chunk_loads(stage[s], bars.tma[s], &tm_q, &tm_k, &tm_v, qh, kh, vh,
                                  static_cast<int32_t>(t0 + static_cast<int64_t>(c + 2) * kChunk));
                pending[s] = 1;
            }
            abort = *reinterpret_cast<volatile int32_t*>(s_abort) != 0;
        }
        if (abort) break;
    }

    // ---- clean up: drain TMA loads still in flight (bounded), free TMEM
    if (tid == 0) {
        for (int s = 0; s < 2; ++s)
            if (pending[s]) {
                if (!mbar_wait(bars.tma[s], tma_phase[s] & 1u)) atomicOr(p.status, GDN_DEVICE_ERR_TIMEOUT);
                ++tma_phase[s];
            }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmCols);
}

}  // namespace

size_t chunk_bf16_smem_bytes() { return kSmemAlloc; }

cudaError_t launch_chunk_bf16(const ChunkParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                              const CUtensorMap& tm_v, int grid, cudaStream_t stream) {
    static int configured = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured != dev) {
        e = cudaFuncSetAttribute(gdn_chunk_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemAlloc));
        if (e != cudaSuccess) return e;
        configured = dev;
    }
    gdn_chunk_bf16_kernel<<<grid, kThreads, kSmemAlloc, stream>>>(p, tm_q, tm_k, tm_v);
    return cudaGetLastError();
}

}  // namespace gdn
