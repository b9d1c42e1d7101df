// gdn_cp.cu -- context parallelism inside one GPU ("FlashInfer GDN Prefill
// 完全指南", the CP routing and max_seqlen rows of the API table and the CP
// backend's routing rules; "GDN与线性注意力GPU并行实现", the per-block transfer
// (M, N) and the scan over the blocks of section 3.3).
//
// Sequences long enough to dominate the run are cut into segments of tau
// chunks (tau a multiple of the checkpoint interval); the others run whole.
// The choice is made on the device from cu_seqlens (cp_prepare_kernel, with
// the load model of gdn_internal.cuh).  Over one segment the chunk recurrence
// is affine in the state it starts from, S_end = S_start M + N, because every
// chunk maps S to S (gamma_63 I - W~^T D K) + U~^T D K.  So:
//   1. a transfer pass (the chunk kernel's kTransfer instance) runs segments
//      0 .. P_i-2 of every segmented sequence twice: from zero (N) and from
//      the identity with U = 0 (M); the units are independent;
//   2. cp_fixup_kernel scans the segments in order on CUDA cores in fp32:
//      S_start(0) = the initial state, S_start(s+1) = S_start(s) M_s + N_s
//      (rows of S are independent, so four CTAs share one (sequence, head));
//   3. the ordinary chunk kernel runs every segment, and every whole
//      sequence, as sequences of one batch: segments from their start states
//      in a scratch buffer (in place), whole sequences straight from and to
//      the caller's state; outputs and checkpoints land where one pass over
//      the whole sequences puts them;
//   4. cp_final_kernel copies each segmented sequence's last segment's final
//      state to the caller's output state.
// A segmented sequence costs about (2 (P-1) + P) / P times its plain work,
// spread over P times as many units; when the model finds no gain every
// sequence runs whole and steps 1, 2 and 4 have nothing to do.
#include <atomic>

#include "gdn_internal.cuh"
#include "sm103_ptx.cuh"

namespace gdn {
namespace {

constexpr int kCpThreads = 256;
constexpr int kCpWarps = kCpThreads / 32;
constexpr int kCand = kCpMaxSegments - 1;  // candidates P = 2 .. kCpMaxSegments
constexpr int kSlots = 8;                   // candidate slots per group of eight threads (the last: one pass)
static_assert(kCand < kSlots && kCpThreads % kSlots == 0, "one candidate per thread of a group of eight");
constexpr int kFixRows = 32;                // rows of S per fixup or final CTA
constexpr int kFixSplit = kHead / kFixRows; // fixup or final CTAs per (sequence, head)
constexpr int kLdS = kHead + 1;             // padded rows of the running state in shared memory
constexpr int kPlaneVec = kHead * kHead / (4 * kCpThreads);   // float4 per thread of a 128 x 128 plane
constexpr int kRowsVec = kFixRows * kHead / (4 * kCpThreads); // float4 per thread of a CTA's 32 rows

__device__ __forceinline__ int64_t seq_chunks(const CpParams& p, int32_t i, int64_t& t0, int64_t& L) {
    t0 = load_index(p.cu_seqlens, p.cu_i64, i);
    L = load_index(p.cu_seqlens, p.cu_i64, i + 1) - t0;
    if (L < 0) L = 0;  // a bad cu_seqlens is flagged by the prepare kernel; keep the segments sane
    return (L + kChunk - 1) / kChunk;
}

// Exclusive scan of one value per thread over the CTA; *total gets the sum.
__device__ int32_t cp_excl_scan(int32_t x, int32_t* warp_sums, int32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t inc = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) warp_sums[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int32_t w = lane < kCpThreads / 32 ? warp_sums[lane] : 0;
        int32_t wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        if (lane < kCpThreads / 32) warp_sums[lane] = wi - w;
        if (lane == 31) *total = wi;
    }
    __syncthreads();
    const int32_t r = warp_sums[warp] + inc - x;
    __syncthreads();
    return r;
}

__device__ __forceinline__ int64_t real_row(const CpParams& p, int32_t i) {
    return p.state_indices ? load_index(p.state_indices, p.idx_i64, i) : i;
}

__device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

// The segmentation, the transfer pass's segments and order, the fixup's list
// of segmented sequences and the segment pass's batch.  One CTA.  The load
// model's candidates are evaluated side by side: thread t scores candidate
// P = 2 + t % 8 on every 32nd sequence, and eight threads cost the candidates
// and one pass, so that no thread runs the 64-bit divisions of all of them.
__global__ void __launch_bounds__(kCpThreads) cp_prepare_kernel(const CpParams p) {
    __shared__ int64_t s_red[kCpWarps][2];             // per warp: longest sequence, total chunks
    __shared__ int64_t s_cand[kCpWarps][kSlots][4];    // per warp and slot: nA, nS, longest whole, largest P
    __shared__ int64_t s_cost[kSlots], s_tauc[kSlots]; // per candidate (slot 7: one pass)
    __shared__ int64_t s_tau;
    __shared__ int32_t warp_sums[kCpWarps];
    __shared__ int32_t tile_total;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t N = p.num_seqs;
    // the batch's ends, which the tail of the segment pass's batch repeats
    const int32_t end = static_cast<int32_t>(load_index(p.cu_seqlens, p.cu_i64, N));
    const int64_t ck_end = p.ckpt_n > 0 ? load_index(p.ckpt_cu_starts, p.ckpt_i64, N) : 0;
    // ---- chunk counts: longest and total
    {
        int64_t cmax = 0, sumc = 0;
        for (int32_t i = tid; i < N; i += kCpThreads) {
            int64_t t0, L;
            const int64_t c = seq_chunks(p, i, t0, L);
            cmax = max64(cmax, c);
            sumc += c;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            cmax = max64(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
            sumc += __shfl_xor_sync(0xffffffffu, sumc, o);
        }
        if (lane == 0) {
            s_red[warp][0] = cmax;
            s_red[warp][1] = sumc;
        }
    }
    __syncthreads();
    int64_t c_max = 0, sum_c = 0;
#pragma unroll
    for (int w = 0; w < kCpWarps; ++w) {
        c_max = max64(c_max, s_red[w][0]);
        sum_c += s_red[w][1];
    }
    // ---- every candidate's sums: slot j = t % 8 is candidate P = j + 2
    {
        const int j = tid % kSlots;
        const int64_t tau_j = j < kCand ? cp_tau(c_max, j + 2, p.align_chunks) : 0;
        CpSums loc{0, 0, 0, 0};
        if (j < kCand)
            for (int32_t i = tid / kSlots; i < N; i += kCpThreads / kSlots) {
                int64_t t0, L;
                cp_add_sequence(loc, seq_chunks(p, i, t0, L), tau_j);
            }
#pragma unroll
        for (int o = kSlots; o < 32; o <<= 1) {  // lanes of one slot: lane % 8 equal
            loc.nA += __shfl_xor_sync(0xffffffffu, loc.nA, o);
            loc.nS += __shfl_xor_sync(0xffffffffu, loc.nS, o);
            loc.max_whole = max64(loc.max_whole, __shfl_xor_sync(0xffffffffu, loc.max_whole, o));
            loc.max_p = max64(loc.max_p, __shfl_xor_sync(0xffffffffu, loc.max_p, o));
        }
        if (lane < kSlots) {
            s_cand[warp][lane][0] = loc.nA;
            s_cand[warp][lane][1] = loc.nS;
            s_cand[warp][lane][2] = loc.max_whole;
            s_cand[warp][lane][3] = loc.max_p;
        }
        __syncthreads();
        if (tid < kSlots) {
            CpSums s{0, 0, 0, 0};
#pragma unroll
            for (int w = 0; w < kCpWarps; ++w) {
                s.nA += s_cand[w][tid][0];
                s.nS += s_cand[w][tid][1];
                s.max_whole = max64(s.max_whole, s_cand[w][tid][2]);
                s.max_p = max64(s.max_p, s_cand[w][tid][3]);
            }
            s_tauc[tid] = tau_j;
            s_cost[tid] = tid < kCand ? cp_candidate_cost(s, tau_j, sum_c, p.H, p.sms)
                                      : cp_one_pass_cost(c_max, sum_c, p.H, p.sms);
        }
        __syncthreads();
        if (tid == 0) s_tau = (p.nA_max > 0 && p.sms > 0) ? cp_choose_tau(s_cost, s_tauc, s_cost[kCand]) : 0;
        __syncthreads();
    }
    const int64_t tau = s_tau, tau_tok = tau * kChunk;
    // Segment s of a cut sequence starts s tau_tok tokens in (that is inside
    // the sequence: (P - 1) tau < c), a whole multiple of the checkpoint interval.
    const int64_t ck_step = p.ckpt_n > 0 ? tau_tok / p.ckpt_n : 0;
    // ---- per sequence: segments, offsets (exclusive scans), lists
    int32_t carry_a = 0, carry_k = 0, carry_s = 0;
    for (int32_t base = 0; base < N; base += kCpThreads) {
        const int32_t i = base + tid;
        int64_t t0 = 0, L = 0, c0 = 0, row = 0;
        int32_t P = 1;
        if (i < N) {
            P = cp_seq_segments(seq_chunks(p, i, t0, L), tau);
            if (p.ckpt_n > 0) c0 = load_index(p.ckpt_cu_starts, p.ckpt_i64, i);
            row = real_row(p, i);
        }
        const int32_t segd = P >= 2 ? 1 : 0;
        const int32_t ta = carry_a + cp_excl_scan(P - 1, warp_sums, &tile_total);
        carry_a += tile_total;
        const int32_t k = carry_k + cp_excl_scan(segd, warp_sums, &tile_total);
        carry_k += tile_total;
        const int32_t sb = carry_s + cp_excl_scan(segd ? P : 0, warp_sums, &tile_total);
        carry_s += tile_total;
        if (i < N) {
            if (segd) {
                p.seg_seq[4 * k] = i;
                p.seg_seq[4 * k + 1] = P;
                p.seg_seq[4 * k + 2] = ta;
                p.seg_seq[4 * k + 3] = sb;
                for (int32_t s = 0; s + 1 < P; ++s) {
                    p.seg_a[2 * (ta + s)] = t0 + s * tau_tok;
                    p.seg_a[2 * (ta + s) + 1] = tau_tok;
                }
            }
            const int32_t v = i + ta;  // first entry of this sequence in the segment pass's batch
            for (int32_t s = 0; s < P; ++s) {
                p.cu_c[v + s] = static_cast<int32_t>(t0 + s * tau_tok);
                p.ckpt_c[v + s] = p.ckpt_n > 0 ? c0 + s * ck_step : 0;
                p.vrow[v + s] = segd ? static_cast<int64_t>(sb + s) : -1 - row;
            }
        }
    }
    // ---- the batch's tail of empty entries, the transfer order, the counts
    const int32_t V = N + carry_a;
    for (int32_t v = V + tid; v <= p.V_max; v += kCpThreads) {
        p.cu_c[v] = end;
        p.ckpt_c[v] = ck_end;
        if (v < p.V_max) p.vrow[v] = 0;
    }
    for (int32_t j = tid; j < p.nA_max; j += kCpThreads) p.order_a[j] = j;
    if (tid == 0) {
        p.counts[0] = carry_a;
        p.counts[1] = V;
        p.counts[2] = carry_k;
        *p.counter_a = 0;
    }
}

// Four CTAs per (segmented sequence, state head), 32 rows of S each: the
// start states of its P segments, in fp32.  Thread t owns row v = t / 8 of
// the CTA's rows and columns 4 (t % 8) + 32 q + j (q, j < 4), so that eight
// neighbouring threads read 128 contiguous bytes of M and N.  The M planes
// arrive by asynchronous copies into two buffers: M_{s+1} is in flight while
// step s multiplies by M_s.
__global__ void __launch_bounds__(kCpThreads) cp_fixup_kernel(const CpParams p) {
    extern __shared__ __align__(16) float cp_smem[];
    float* S = cp_smem;                            // [32][kLdS]
    float* Mbuf = cp_smem + kFixRows * kLdS;       // two [128][128] planes
    if (*reinterpret_cast<volatile int32_t*>(p.status)) return;
    const int32_t part = blockIdx.x % kFixSplit, uh = blockIdx.x / kFixSplit;
    const int32_t k = uh / p.H, h = uh % p.H;
    if (k >= p.counts[2]) return;
    const int32_t i = p.seg_seq[4 * k], P = p.seg_seq[4 * k + 1], ta = p.seg_seq[4 * k + 2], sb = p.seg_seq[4 * k + 3];
    const size_t plane = static_cast<size_t>(kHead) * kHead;
    const int r0 = part * kFixRows;
    const int t = threadIdx.x, v = t >> 3, cl = 4 * (t & 7);
    // One commit group per step (empty past the last M), so that waiting for
    // all but the newest group always means "M_s has landed".
    auto copy_m = [&](int32_t s) {
        if (s + 1 < P) {
            const float* Mm = p.trans + (static_cast<size_t>(p.nA_max + ta + s) * p.H + h) * plane;
            float* dst = Mbuf + (s & 1) * plane;
#pragma unroll
            for (int it = 0; it < kPlaneVec; ++it) {
                const int e = 4 * (t + it * kCpThreads);
                cp_async16(dst + e, Mm + e);
            }
        }
        cp_async_commit();
    };
    copy_m(0);
    copy_m(1);
    // S_start(0): the caller's initial state (or zeros), in any layout and type
    const int64_t srow = real_row(p, i);
    float* out0 = p.start + (static_cast<size_t>(sb) * p.H + h) * plane;
    {
        float x[kRowsVec][4];
#pragma unroll
        for (int it = 0; it < kRowsVec; ++it) {
            const int e = 4 * (t + it * kCpThreads), r = e / kHead, c = e % kHead;
#pragma unroll
            for (int j = 0; j < 4; ++j) x[it][j] = 0.f;
            if (p.initial_state)
                state_load4(p.initial_state, state_offset(p.state, srow, h, r0 + r) + c, p.state.dtype, x[it]);
        }
#pragma unroll
        for (int it = 0; it < kRowsVec; ++it) {
            const int e = 4 * (t + it * kCpThreads), r = e / kHead, c = e % kHead;
#pragma unroll
            for (int j = 0; j < 4; ++j) S[r * kLdS + c + j] = x[it][j];
            *reinterpret_cast<float4*>(out0 + static_cast<size_t>(r0 + r) * kHead + c) =
                make_float4(x[it][0], x[it][1], x[it][2], x[it][3]);
        }
    }
    for (int32_t s = 0; s + 1 < P; ++s) {
        const float* Nm = p.trans + (static_cast<size_t>(ta + s) * p.H + h) * plane;
        float acc[16];
        const float* nrow = Nm + static_cast<size_t>(r0 + v) * kHead + cl;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 n4 = *reinterpret_cast<const float4*>(nrow + 32 * q);
            acc[4 * q] = n4.x;
            acc[4 * q + 1] = n4.y;
            acc[4 * q + 2] = n4.z;
            acc[4 * q + 3] = n4.w;
        }
        cp_async_wait<1>();  // this thread's pieces of M_s
        __syncthreads();     // everyone's pieces, and S
        const float* M = Mbuf + (s & 1) * plane;
#pragma unroll 4
        for (int c = 0; c < kHead; ++c) {
            const float sv = S[v * kLdS + c];
            const float* mr = M + c * kHead + cl;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 m4 = *reinterpret_cast<const float4*>(mr + 32 * q);
                acc[4 * q] = fmaf(sv, m4.x, acc[4 * q]);
                acc[4 * q + 1] = fmaf(sv, m4.y, acc[4 * q + 1]);
                acc[4 * q + 2] = fmaf(sv, m4.z, acc[4 * q + 2]);
                acc[4 * q + 3] = fmaf(sv, m4.w, acc[4 * q + 3]);
            }
        }
        __syncthreads();  // every row of S and all of M_s have been read
        copy_m(s + 2);    // into the buffer M_s leaves
        float* outs = p.start + (static_cast<size_t>(sb + s + 1) * p.H + h) * plane +
                      static_cast<size_t>(r0 + v) * kHead + cl;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int j = 0; j < 4; ++j) S[v * kLdS + cl + 32 * q + j] = acc[4 * q + j];
            *reinterpret_cast<float4*>(outs + 32 * q) =
                make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
        }
    }
    cp_async_wait<0>();  // nothing is left in flight when the CTA ends (the groups past the last M are empty)
}

// Four CTAs per (segmented sequence, state head), 32 rows each: the last
// segment's final state (left in place by the segment pass) to the caller's
// output state.  Every load is issued before the first store.
__global__ void __launch_bounds__(kCpThreads) cp_final_kernel(const CpParams p) {
    if (*reinterpret_cast<volatile int32_t*>(p.status)) return;
    const int32_t part = blockIdx.x % kFixSplit, uh = blockIdx.x / kFixSplit;
    const int32_t k = uh / p.H, h = uh % p.H;
    if (k >= p.counts[2]) return;
    const int32_t i = p.seg_seq[4 * k], P = p.seg_seq[4 * k + 1], sb = p.seg_seq[4 * k + 3];
    const size_t plane = static_cast<size_t>(kHead) * kHead;
    const int r0 = part * kFixRows;
    const float* src = p.start + (static_cast<size_t>(sb + P - 1) * p.H + h) * plane + static_cast<size_t>(r0) * kHead;
    const int64_t srow = real_row(p, i);
    float4 f[kRowsVec];
#pragma unroll
    for (int it = 0; it < kRowsVec; ++it)
        f[it] = *reinterpret_cast<const float4*>(src + 4 * (threadIdx.x + it * kCpThreads));
#pragma unroll
    for (int it = 0; it < kRowsVec; ++it) {
        const int e = 4 * (threadIdx.x + it * kCpThreads), r = e / kHead, c = e % kHead;
        const float x[4] = {f[it].x, f[it].y, f[it].z, f[it].w};
        state_store4(p.output_state, state_offset(p.state, srow, h, r0 + r) + c, p.state.dtype, x);
    }
}

constexpr size_t kFixupSmem = sizeof(float) * (kFixRows * kLdS + 2 * kHead * kHead);
static_assert(kFixRows * kLdS % 4 == 0, "the M planes start on a 16-byte boundary");

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
    if (p.nA_max <= 0) return cudaSuccess;
    cp_fixup_kernel<<<p.nA_max * p.H * kFixSplit, kCpThreads, kFixupSmem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_cp_final(const CpParams& p, cudaStream_t stream) {
    if (!p.output_state || p.nA_max <= 0) return cudaSuccess;
    cp_final_kernel<<<p.nA_max * p.H * kFixSplit, kCpThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
