// gdn_decode.cu -- the gated delta rule step by step for a few tokens per
// sequence: the decode step after a prefill, or a short run of speculative
// tokens, on the same [rows, H, V, K] state (or pool) the prefill writes
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
// (sequence, head) in fp32, a few hundred bytes of q/k/v/o per token), so it
// runs on CUDA cores: persistent CTAs, one per SM, walk the (sequence, head)
// units.  One producer warp fills a ring of up to three shared-memory stages
// with TMA bulk copies -- a unit's state rows (raw bytes of the storage type)
// and all its tokens -- and refills a stage's state part as soon as the
// consumers hold that unit's state in registers (per-stage full / empty
// mbarriers), so the HBM reads of later units overlap this one's arithmetic.
// Sixteen consumer warps hold the state, four rows by eight columns per
// thread, so that each k or q value read from shared memory serves four rows;
// the 16 threads of a row group close their eight partial sums (S k and S q
// for four rows) with a reduce-scatter of eight shuffles.  k and q are widened
// to fp32 once per token (eight tokens per window, two window buffers, one
// consumer barrier per window), and their L2 norms enter as scalars:
// S k^ = |k|^-1 S k, the rank-one update adds (w |k|^-1) k, and the output is
// o = scale |q|^-1 (alpha S q + w k . q) from the state before the update.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "gdn_internal.cuh"
#include "sm103_ptx.cuh"

namespace gdn {
namespace {

constexpr int kDecConsumers = 512;                 // sixteen consumer warps
constexpr int kDecThreads = kDecConsumers + 32;    // and one producer warp
constexpr int kDecMaxStages = 3;                   // units in flight per CTA
constexpr int kDecWin = 8;                         // tokens widened to fp32 per window
constexpr int kDecStaticSmem = 512;                // bound of the kernel's static shared memory
constexpr uint32_t kDecBarWin = 1;                 // named barrier of the consumer warps
constexpr long long kDecWaitCycles = 2000000000LL; // about a second: a wait that runs this long gives up

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

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <>
__device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// A unit's place in the walk: u = seq * H + h, advanced by the grid stride without divisions.
struct UnitPos {
    int32_t u, seq, h;
    __device__ __forceinline__ void advance(int32_t du, int32_t dseq, int32_t dh, int32_t H) {
        u += du;
        seq += dseq;
        h += dh;
        if (h >= H) {
            h -= H;
            ++seq;
        }
    }
};

struct DecodeShared {
    uint64_t full_s[kDecMaxStages], full_t[kDecMaxStages];    // the stage's state part / token part landed
    uint64_t empty_s[kDecMaxStages], empty_t[kDecMaxStages];  // ... and was released by the consumers
    int64_t row[kDecMaxStages];                               // the unit's state row
    int32_t ok[kDecMaxStages];                                // 0: that row is out of the pool's range
    int32_t abort;                                            // a wait ran out: everybody leaves
};
static_assert(sizeof(DecodeShared) + 64 <= kDecStaticSmem, "static shared memory bound");

// Bounded wait on one phase of an mbarrier that also gives up when another warp has aborted.
__device__ __forceinline__ bool dec_wait(uint64_t* bar, uint32_t parity, const volatile int32_t* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 1000)) return true;
        if (*abort) return false;
        if (clock64() - t0 > kDecWaitCycles) return false;
    }
}

// The producer warp: for each of this CTA's units in order, the stage's state part (once the consumers
// released it) by bulk copies -- the whole (row, head) plane when its v rows are contiguous, else row by
// row; a bare arrival without an initial state or for a pool row out of range -- then the token part: q, k,
// v rows by bulk copies (lane 0) and g, beta by plain loads (all lanes), every lane arriving once.
template <typename T, typename SD, bool kAhead>
__device__ void decode_producer(const DecodeParams& p, DecodeShared& sh, uint8_t* dsm, UnitPos x, int32_t units,
                                int32_t grid, int32_t gseq, int32_t gh) {
    const int lane = threadIdx.x & 31, m = p.m, stages = p.stages;
    constexpr uint32_t kRowBytes = kHead * sizeof(SD), kVecBytes = kHead * sizeof(T);
    int s = 0;
    uint32_t use = 0;  // how many times stage s has been filled before
    int32_t issued = 0;
    bool ok_run = true;
    // The pool row (lane 0) and the first 32 gate values (one per lane) of a unit are read one unit ahead, so
    // that their global-memory latency overlaps the previous unit's waits and copies instead of sitting between
    // a stage turning free and its state copy.  Not for one token on fp32 states: that step runs at the HBM
    // roofline, and there the earlier copies measured slower (0.322 -> 0.346 ms on 512 sequences x 32 heads):
    // that case runs the instance without the lookahead (kAhead false).
    constexpr bool ahead = kAhead;
    auto row_of = [&](const UnitPos& y) -> int64_t {
        return p.state_indices ? load_index(p.state_indices, p.idx_i64, y.seq) : y.seq;
    };
    auto gate_of = [&](const UnitPos& y, int i) -> float {  // i < m: g of token i, else beta of token i - m
        const float* src = i < m ? p.g : p.beta;
        const int t = i < m ? i : i - m;
        return src ? src[(static_cast<int64_t>(y.seq) * m + t) * p.H + y.h] : 1.f;
    };
    int64_t row_next = 0;
    float gate_next = 1.f;
    if (ahead && x.u < units) {
        if (lane == 0) row_next = row_of(x);
        if (lane < 2 * m) gate_next = gate_of(x, lane);
    }
    for (; x.u < units; ++issued) {
        const int64_t row_pre = row_next;
        const float gate_pre = gate_next;
        UnitPos nx = x;
        nx.advance(grid, gseq, gh, p.H);
        if (ahead && nx.u < units) {
            if (lane == 0) row_next = row_of(nx);
            if (lane < 2 * m) gate_next = gate_of(nx, lane);
        }
        uint8_t* st = dsm + static_cast<size_t>(s) * p.stage_bytes;
        if (use > 0) ok_run = dec_wait(&sh.empty_s[s], (use - 1) & 1, &sh.abort);
        if (!__all_sync(0xffffffffu, ok_run)) break;
        if (lane == 0) {
            const int64_t srow = ahead ? row_pre : row_of(x);
            const bool ok = !p.state_indices || (srow >= 0 && srow < p.n_pool);
            sh.row[s] = srow;
            sh.ok[s] = ok ? 1 : 0;
            if (!ok || !p.initial_state) {
                mbar_arrive_expect_tx(&sh.full_s[s], 0);
            } else {
                mbar_arrive_expect_tx(&sh.full_s[s], kHead * kRowBytes);
                const uint8_t* base = static_cast<const uint8_t*>(p.initial_state) +
                                      state_offset(p.state, srow, x.h, 0) * static_cast<int64_t>(sizeof(SD));
                if (p.state.s_v == kHead) {
                    constexpr uint32_t kPiece = 16384;  // a few copies in flight rather than one long one
                    for (uint32_t off = 0; off < kHead * kRowBytes; off += kPiece)
                        bulk_load(st + off, base + off, kPiece, &sh.full_s[s]);
                } else {
                    for (int row = 0; row < kHead; ++row)
                        bulk_load(st + row * kRowBytes, base + row * p.state.s_v * static_cast<int64_t>(sizeof(SD)),
                                  kRowBytes, &sh.full_s[s]);
                }
            }
        }
        if (use > 0) ok_run = dec_wait(&sh.empty_t[s], (use - 1) & 1, &sh.abort);
        if (!__all_sync(0xffffffffu, ok_run)) break;
        uint8_t* tk = st + kHead * kRowBytes;
        float* gb = reinterpret_cast<float*>(tk + 3 * m * kVecBytes);  // g [m], then beta [m]
        for (int i = lane; i < 2 * m; i += 32) gb[i] = ahead && i < 32 ? gate_pre : gate_of(x, i);
        if (lane == 0) {
            mbar_arrive_expect_tx(&sh.full_t[s], 3 * m * kVecBytes);
            for (int which = 0; which < 3; ++which) {
                const void* src = which == 0 ? p.q : (which == 1 ? p.k : p.v);
                const int32_t heads = which == 0 ? p.hq : (which == 1 ? p.hk : p.hv);
                const int32_t hh = x.h / (p.H / heads);
                for (int t = 0; t < m; ++t) {
                    const int64_t row = (static_cast<int64_t>(x.seq) * m + t) * heads + hh;
                    bulk_load(tk + (which * m + t) * kVecBytes,
                              static_cast<const uint8_t*>(src) + row * static_cast<int64_t>(kVecBytes), kVecBytes,
                              &sh.full_t[s]);
                }
            }
        } else {
            mbar_arrive(&sh.full_t[s]);  // after this lane's g / beta stores
        }
        x.advance(grid, gseq, gh, p.H);
        if (++s == stages) {
            s = 0;
            ++use;
        }
    }
    if (!ok_run && lane == 0) {
        sh.abort = 1;
        if (p.status) atomicOr(p.status, static_cast<int32_t>(GDN_DEVICE_ERR_TIMEOUT));
    }
    // Nothing may land in shared memory after the CTA exits: after an abort, wait (bounded) for the last
    // fill of every stage that was filled.
    if (sh.abort && lane == 0) {
        for (int k = 0; k < stages && k < issued; ++k) {
            const int32_t last = issued - 1 - ((issued - 1 - k) % stages);  // last fill of stage k
            const uint32_t par = static_cast<uint32_t>((last / stages) & 1);
            mbar_wait(&sh.full_s[k], par);
            mbar_wait(&sh.full_t[k], par);
        }
    }
}

template <typename T, typename SD>
__global__ void __launch_bounds__(kDecThreads, 1) gdn_decode_kernel(const DecodeParams p) {
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ DecodeShared sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t H = p.H, units = p.N * H;  // below 2^31 (checked on the host)
    const int stages = p.stages, m = p.m;
    const int32_t grid = gridDim.x, gseq = grid / H, gh = grid % H;
    const UnitPos first{static_cast<int32_t>(blockIdx.x), static_cast<int32_t>(blockIdx.x) / H,
                        static_cast<int32_t>(blockIdx.x) % H};
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&sh.full_s[s], 1);
            mbar_init(&sh.full_t[s], 32);
            mbar_init(&sh.empty_s[s], kDecConsumers / 32);
            mbar_init(&sh.empty_t[s], kDecConsumers / 32);
        }
        sh.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == kDecConsumers / 32) {
        if (sizeof(SD) < 4 || m > 1)
            decode_producer<T, SD, true>(p, sh, dsm, first, units, grid, gseq, gh);
        else
            decode_producer<T, SD, false>(p, sh, dsm, first, units, grid, gseq, gh);
        return;
    }

    // ---- consumers: thread (row group rh of warp w, column group cg) holds rows 8 w + 4 rh + i (i < 4),
    //      columns 4 cg + e and 64 + 4 cg + e (e < 4)
    constexpr int kVecBytes = kHead * static_cast<int>(sizeof(T));
    const int cg = lane & 15, rh = lane >> 4, r0 = 8 * warp + 4 * rh;
    const int b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1, b1 = (lane >> 1) & 1;
    const int my_i = 2 * b2 + b1;  // after the reduce-scatter: S k (b3 = 0) or S q (b3 = 1) of row r0 + my_i
    uint8_t* conv = dsm + static_cast<size_t>(stages) * p.stage_bytes;
    constexpr int kConvBytes = (2 * kDecWin * kHead + 4 * kDecWin) * 4;
    UnitPos cur = first;
    int s = 0;
    uint32_t par = 0;
    uint32_t wc = 0;  // windows so far (selects the fp32 buffer)
    bool alive = true;
    for (; cur.u < units && alive;) {
        const bool landed = dec_wait(&sh.full_s[s], par, &sh.abort) && dec_wait(&sh.full_t[s], par, &sh.abort);
        const uint8_t* st = dsm + static_cast<size_t>(s) * p.stage_bytes;
        const bool ok = sh.ok[s] != 0;
        const int64_t srow = sh.row[s];
        float S[4][8];
        if (ok && p.initial_state) {
            const SD* ss = reinterpret_cast<const SD*>(st) + r0 * kHead + 4 * cg;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float a4[4], b4[4];
                load4(ss + i * kHead, a4);
                load4(ss + i * kHead + 64, b4);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    S[i][e] = a4[e];
                    S[i][4 + e] = b4[e];
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int c = 0; c < 8; ++c) S[i][c] = 0.f;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.empty_s[s]);  // this warp is done with the stage's state part
        const uint8_t* tk = st + kHead * kHead * sizeof(SD);
        const T* vv = reinterpret_cast<const T*>(tk + 2 * m * kVecBytes);
        const float* gb = reinterpret_cast<const float*>(tk + 3 * m * kVecBytes);
        T* out = static_cast<T*>(p.output) + (static_cast<int64_t>(cur.seq) * m * H + cur.h) * kHead;
        // The window loop runs for every unit (m is the same for all threads), so that its barrier settles
        // first whether every wait landed; only then is `ok` (read from the stage) the same for all.
        for (int w0 = 0; w0 < m; w0 += kDecWin, ++wc) {
            const int W = m - w0 < kDecWin ? m - w0 : kDecWin;
            float* k32 = reinterpret_cast<float*>(conv + (wc & 1) * kConvBytes);  // [kDecWin][128]
            float* q32 = k32 + kDecWin * kHead;                                    // [kDecWin][128]
            float* tok_f = q32 + kDecWin * kHead;  // [kDecWin][4]: 1/|k|, 1/|q| (1 without the norm), k . q
            // widen this window's k and q rows to fp32 (one warp per token); the buffer was last read two
            // windows ago, before every consumer passed the previous window's barrier
            if (landed && warp < W) {
                const int t = warp;
                float xk[4], xq[4];
                load4(reinterpret_cast<const T*>(tk + (m + w0 + t) * kVecBytes) + 4 * lane, xk);
                load4(reinterpret_cast<const T*>(tk + (w0 + t) * kVecBytes) + 4 * lane, xq);
                *reinterpret_cast<float4*>(k32 + t * kHead + 4 * lane) = make_float4(xk[0], xk[1], xk[2], xk[3]);
                *reinterpret_cast<float4*>(q32 + t * kHead + 4 * lane) = make_float4(xq[0], xq[1], xq[2], xq[3]);
                float kk = 0.f, qq = 0.f, kq = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    kk = fmaf(xk[e], xk[e], kk);
                    qq = fmaf(xq[e], xq[e], qq);
                    kq = fmaf(xk[e], xq[e], kq);
                }
                kq = warp_sum(kq);
                float rk = 1.f, rq = 1.f;
                if (p.l2norm) {
                    rk = rsqrtf(warp_sum(kk) + 1e-6f);
                    rq = rsqrtf(warp_sum(qq) + 1e-6f);
                }
                if (lane == 0) *reinterpret_cast<float4*>(tok_f + 4 * t) = make_float4(rk, rq, kq, 0.f);
            }
            // every consumer decides together: go on, or leave because some wait ran out
            if (!named_bar_and(kDecBarWin, kDecConsumers, landed)) {
                alive = false;
                break;
            }
            if (!ok) continue;  // a pool row out of range: no outputs, no state (flagged below)
            for (int t = 0; t < W; ++t) {
                const int tt = w0 + t;
                const float* kt = k32 + t * kHead + 4 * cg;
                const float* qt = q32 + t * kHead + 4 * cg;
                const float4 ka = *reinterpret_cast<const float4*>(kt), kb = *reinterpret_cast<const float4*>(kt + 64);
                const float4 qa = *reinterpret_cast<const float4*>(qt), qb = *reinterpret_cast<const float4*>(qt + 64);
                const float kx[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
                const float qx[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
                float v8[8];  // S k of the four rows, then S q, over this thread's eight columns
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float su = 0.f, sq = 0.f;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        su = fmaf(S[i][c], kx[c], su);
                        sq = fmaf(S[i][c], qx[c], sq);
                    }
                    v8[i] = su;
                    v8[4 + i] = sq;
                }
                // reduce-scatter over the 16 threads of the row group: halve the values at every step
                float x4[4], x2[2];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float send = b3 ? v8[i] : v8[4 + i];
                    x4[i] = (b3 ? v8[4 + i] : v8[i]) + __shfl_xor_sync(0xffffffffu, send, 8);
                }
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float send = b2 ? x4[i] : x4[2 + i];
                    x2[i] = (b2 ? x4[2 + i] : x4[i]) + __shfl_xor_sync(0xffffffffu, send, 4);
                }
                float x1 = (b1 ? x2[1] : x2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? x2[0] : x2[1], 2);
                x1 += __shfl_xor_sync(0xffffffffu, x1, 1);
                const float4 tf = *reinterpret_cast<const float4*>(tok_f + 4 * t);  // rk, rq, k . q
                const float a = gb[tt], b = gb[m + tt];
                // lanes with b3 = 0 hold S k of row r0 + my_i: w = beta (v - alpha S k^) / |k| (w scales raw k)
                const float wmine = b * (to_f32(vv[tt * kHead + r0 + my_i]) - a * (tf.x * x1)) * tf.x;
                const float wrow = __shfl_xor_sync(0xffffffffu, wmine, 8);  // lanes with b3 = 1: w of their row
                if (b3 && !(lane & 1))  // o = scale / |q| (alpha S q + w k . q), S q from before the update
                    out[static_cast<int64_t>(tt) * H * kHead + r0 + my_i] =
                        from_f32<T>(p.scale * tf.y * fmaf(a, x1, wrow * tf.z));
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float wi = __shfl_sync(0xffffffffu, wmine, (lane & 16) + 2 * i);
#pragma unroll
                    for (int c = 0; c < 8; ++c) S[i][c] = fmaf(wi, kx[c], a * S[i][c]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.empty_t[s]);  // this warp is done with the stage's token part
        if (!alive) break;
        if (ok && p.output_state) {
            SD* dst = static_cast<SD*>(p.output_state) + state_offset(p.state, srow, cur.h, r0) + 4 * cg;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float a4[4] = {S[i][0], S[i][1], S[i][2], S[i][3]};
                const float b4[4] = {S[i][4], S[i][5], S[i][6], S[i][7]};
                store4(dst + i * p.state.s_v, a4);
                store4(dst + i * p.state.s_v + 64, b4);
            }
        } else if (!ok && tid == 0 && p.status) {
            atomicOr(p.status, static_cast<int32_t>(GDN_DEVICE_ERR_STATE_INDEX_RANGE));
        }
        cur.advance(grid, gseq, gh, H);
        if (++s == stages) {
            s = 0;
            par ^= 1u;
        }
    }
    if (!alive && tid == 0) {
        sh.abort = 1;  // the producer stops, then waits for what it has in flight
        if (p.status) atomicOr(p.status, static_cast<int32_t>(GDN_DEVICE_ERR_TIMEOUT));
    }
}

template <typename T, typename SD>
cudaError_t launch_decode_ts(const DecodeParams& p, unsigned grid, size_t smem, cudaStream_t stream) {
    // One flag per device: the attribute is set once (to the device's opt-in maximum less the kernel's static
    // slots, so one setting serves every token count), and concurrent first calls each set it at most once more.
    constexpr int kMaxDevices = 64;
    static std::atomic<uint8_t> configured[kMaxDevices];
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!configured[dev].load(std::memory_order_acquire)) {
        e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(gdn_decode_kernel<T, SD>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - kDecStaticSmem);
        if (e != cudaSuccess) return e;
        configured[dev].store(1, std::memory_order_release);
    }
    gdn_decode_kernel<T, SD><<<grid, kDecThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_decode_t(const DecodeParams& p, unsigned grid, size_t smem, cudaStream_t stream) {
    if (p.state.dtype == GDN_DTYPE_BF16) return launch_decode_ts<T, __nv_bfloat16>(p, grid, smem, stream);
    if (p.state.dtype == GDN_DTYPE_F16) return launch_decode_ts<T, __half>(p, grid, smem, stream);
    if (p.state.dtype == GDN_DTYPE_F8E4M3) return launch_decode_ts<T, F8E4M3>(p, grid, smem, stream);
    if (p.state.dtype == GDN_DTYPE_F8E5M2) return launch_decode_ts<T, F8E5M2>(p, grid, smem, stream);
    return launch_decode_ts<T, float>(p, grid, smem, stream);
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p_in, gdn_dtype dtype, cudaStream_t stream) {
    const int64_t units = static_cast<int64_t>(p_in.N) * p_in.H;
    if (units == 0) return cudaSuccess;
    int dev = 0, sms = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return cudaErrorUnknown;
    DecodeParams p = p_in;
    const size_t tsize = dtype == GDN_DTYPE_F32 ? 4 : 2;
    const size_t state_bytes = static_cast<size_t>(kHead) * kHead * static_cast<size_t>(dtype_bytes(p.state.dtype));
    const size_t tok_bytes = 3 * static_cast<size_t>(p.m) * kHead * tsize + 2 * static_cast<size_t>(p.m) * 4;
    const size_t stage = (state_bytes + tok_bytes + 15) / 16 * 16;
    const size_t fixed = 2 * (2 * static_cast<size_t>(kDecWin) * kHead + 4 * kDecWin) * 4;  // two fp32 windows
    // the kernel's static shared memory comes out of the same opt-in budget
    const size_t budget = static_cast<size_t>(optin) - kDecStaticSmem;
    if (fixed + stage > budget) return cudaErrorInvalidValue;
    int stages = static_cast<int>((budget - fixed) / stage);
    if (stages > kDecMaxStages) stages = kDecMaxStages;
    p.stages = stages;
    p.stage_bytes = static_cast<int32_t>(stage);
    const size_t smem = fixed + static_cast<size_t>(stages) * stage;
    const int64_t blocks = units < sms ? units : sms;  // persistent: one CTA per SM
    const unsigned grid = static_cast<unsigned>(blocks);
    if (dtype == GDN_DTYPE_BF16) return launch_decode_t<__nv_bfloat16>(p, grid, smem, stream);
    if (dtype == GDN_DTYPE_F16) return launch_decode_t<__half>(p, grid, smem, stream);
    return launch_decode_t<float>(p, grid, smem, stream);
}

}  // namespace gdn
