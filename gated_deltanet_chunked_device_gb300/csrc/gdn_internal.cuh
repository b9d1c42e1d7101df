// gdn_internal.cuh -- parameters shared by the host code and the kernels of the
// chunked Gated DeltaNet prefill.  Not part of the public C ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/gdn_prefill.h"

namespace gdn {

constexpr int kChunk = 64;     // tokens per chunk
constexpr int kHead = 128;     // head size (K = V = 128)

// Initial / output state layout: element type and element strides of
// [row][state head][v]; the 128 k elements of a v row are contiguous.
struct StateLayout {
    int32_t dtype;                 // a gdn_dtype: F32, BF16, F16, F8E4M3 or F8E5M2
    int64_t s_row, s_head, s_v;
};

__host__ __device__ inline int64_t dtype_bytes(int32_t dt) {
    return dt == GDN_DTYPE_F32 ? 4 : (dt == GDN_DTYPE_BF16 || dt == GDN_DTYPE_F16) ? 2 : 1;
}

// fp8 pairs <-> fp32 (PTX cvt: widening is exact; narrowing rounds to
// nearest, ties to even, and saturates to the finite range).  Element 0 is
// the low byte.
__device__ __forceinline__ void fp8x2_to_f32(uint16_t b, int32_t dt, float& lo, float& hi) {
    uint32_t h2;
    if (dt == GDN_DTYPE_F8E4M3)
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(b));
    else
        asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h2) : "h"(b));
    __half2 h;
    memcpy(&h, &h2, 4);
    const float2 f = __half22float2(h);
    lo = f.x;
    hi = f.y;
}

__device__ __forceinline__ uint16_t f32_to_fp8x2(float lo, float hi, int32_t dt) {
    uint16_t b;
    if (dt == GDN_DTYPE_F8E4M3)
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(b) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(b) : "f"(hi), "f"(lo));
    return b;
}

__host__ __device__ inline int64_t state_offset(StateLayout L, int64_t row, int64_t h, int64_t v) {
    return row * L.s_row + h * L.s_head + v * L.s_v;
}

// Four consecutive k elements of a state at element offset `off` (a multiple
// of 4), converted to or from fp32.
__device__ __forceinline__ void state_load4(const void* base, int64_t off, int32_t dt, float (&x)[4]) {
    if (dt == GDN_DTYPE_F32) {
        const float4 f = *reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
        x[0] = f.x;
        x[1] = f.y;
        x[2] = f.z;
        x[3] = f.w;
    } else if (dt == GDN_DTYPE_F8E4M3 || dt == GDN_DTYPE_F8E5M2) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(base) + off);
        fp8x2_to_f32(static_cast<uint16_t>(w & 0xffffu), dt, x[0], x[1]);
        fp8x2_to_f32(static_cast<uint16_t>(w >> 16), dt, x[2], x[3]);
    } else {
        const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + off);
        if (dt == GDN_DTYPE_BF16) {
            x[0] = __uint_as_float(u.x << 16);
            x[1] = __uint_as_float(u.x & 0xffff0000u);
            x[2] = __uint_as_float(u.y << 16);
            x[3] = __uint_as_float(u.y & 0xffff0000u);
        } else {
            __half2 a, b;
            memcpy(&a, &u.x, 4);
            memcpy(&b, &u.y, 4);
            const float2 fa = __half22float2(a), fb = __half22float2(b);
            x[0] = fa.x;
            x[1] = fa.y;
            x[2] = fb.x;
            x[3] = fb.y;
        }
    }
}

__device__ __forceinline__ void state_store4(void* base, int64_t off, int32_t dt, const float (&x)[4]) {
    if (dt == GDN_DTYPE_F32) {
        *reinterpret_cast<float4*>(static_cast<float*>(base) + off) = make_float4(x[0], x[1], x[2], x[3]);
    } else if (dt == GDN_DTYPE_F8E4M3 || dt == GDN_DTYPE_F8E5M2) {
        const uint32_t w = static_cast<uint32_t>(f32_to_fp8x2(x[0], x[1], dt)) |
                           (static_cast<uint32_t>(f32_to_fp8x2(x[2], x[3], dt)) << 16);
        *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(base) + off) = w;
    } else {
        uint2 u;
        if (dt == GDN_DTYPE_BF16) {
            const __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]), b = __floats2bfloat162_rn(x[2], x[3]);
            memcpy(&u.x, &a, 4);
            memcpy(&u.y, &b, 4);
        } else {
            const __half2 a = __floats2half2_rn(x[0], x[1]), b = __floats2half2_rn(x[2], x[3]);
            memcpy(&u.x, &a, 4);
            memcpy(&u.y, &b, 4);
        }
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(base) + off) = u;
    }
}

// Workspace layout (computed on the host from the plan).
struct WorkspaceLayout {
    size_t status;         // int32
    size_t counter;        // int32: next work unit for persistent CTAs
    size_t n_chunks;       // int32
    size_t chunk_offsets;  // int32 [max_seqs + 1]
    size_t chunk_map;      // int32 [max_chunks, 2]
    size_t seq_order;      // int32 [max_seqs]
    size_t pool_bitmap;    // uint32 [ceil(max_pool/32)]
    size_t total;
    int64_t max_chunks;
    int32_t bitmap_words;
};

// Arguments of the prepare kernel (chunk map, validation, work order).
struct PrepareParams {
    const void* cu_seqlens;
    int cu_i64;
    int32_t num_seqs;
    int64_t total_tokens;
    int64_t max_seqlen;            // 0 = no bound check
    int32_t ckpt_n;                // 0 = no checkpoints
    const void* ckpt_cu_starts;
    int ckpt_i64;
    int64_t num_checkpoints;
    const void* state_indices;     // nullptr = no pool
    int idx_i64;
    int32_t n_pool;
    int32_t* status;
    int32_t* counter;
    int32_t* n_chunks;
    int32_t* chunk_offsets;
    int32_t* chunk_map;
    int64_t max_chunks;
    int32_t* seq_order;
    uint32_t* pool_bitmap;
    int32_t bitmap_words;
    int keep_status;               // 1: add to the status word of an earlier prepare instead of clearing it
};

// Arguments of the chunk kernels (intra-chunk solve, state pass and output).
struct ChunkParams {
    const void* q;
    const void* k;
    const void* v;
    const float* g;                // nullptr = ones
    const float* beta;             // nullptr = ones
    float scale;
    int32_t hq, hk, hv, H;
    int l2norm;
    const void* cu_seqlens;
    int cu_i64;
    int32_t num_seqs;
    const void* initial_state;     // nullptr = zeros
    void* output_state;            // nullptr = no final state
    StateLayout state;             // type and strides of both
    const void* state_indices;     // nullptr = dense [N, H, V, K]
    int idx_i64;
    void* checkpoints;             // nullptr = none; dense [rows][H][128][128] of ckpt_dtype
    int32_t ckpt_dtype;            // a gdn_dtype
    int32_t ckpt_n;
    const void* ckpt_cu_starts;
    int ckpt_i64;
    void* output;
    int32_t* status;
    int32_t* counter;
    const int32_t* chunk_offsets;
    const int32_t* seq_order;
    float* intra_g;                // optional per-chunk dumps
    float* intra_w;
    float* intra_u;
    int has_tokens;                // 0: the TMA maps are blank (T == 0) and never used
    const int64_t* seg;            // transfer pass: [num_seqs][2] segment start token and length (else null)
    const int32_t* num_seqs_dev;   // non-null: the run's sequence count, read on the device (<= num_seqs)
    // Segment pass of context parallelism: a negative row r of state_indices names row -1 - r of the
    // caller's own state (initial_state2 / output_state2 in layout state2) instead of the start buffer.
    int split_state;
    const void* initial_state2;
    void* output_state2;
    StateLayout state2;
};

// Context parallelism with a segment count per sequence.  Sequence i of c_i
// chunks is cut into P_i segments of tau chunks (the last one shorter) when
// c_i > tau, else it runs whole (P_i = 1).  One tau serves the whole batch;
// it is chosen from a load model in chunk periods (one chunk of one
// (sequence, head) unit on one SM) over the three launches:
//   transfer pass  ceil(2 H nA / S) tau                 nA = sum (P_i - 1)
//   segment pass   max(ceil(H nS / S) tau, ceil(H sum c_i / S), longest whole c_i)
//                                                       nS = sum of P_i over segmented sequences
//   fixup + launches  (max P_i - 1) + 4
// against one pass, max(c_max, ceil(H sum c_i / S)); the segments are taken
// only when they cost at most 85 % of it.  Candidates: tau = c_max / P
// rounded up to the segment granularity, P = 2 .. kCpMaxSegments; ties go to
// the smaller P.  The device (cp_prepare_kernel) and the host query
// (gdn_prefill_cp_segments) both evaluate it with these functions.
constexpr int32_t kCpMaxSegments = 8;
constexpr int64_t kCpMaxPlanes = 256;  // 128 x 128 fp32 planes of transfer output, and of start states

__host__ __device__ inline int64_t cp_tau(int64_t c_max, int32_t P, int64_t align_chunks) {
    const int64_t t = (c_max + P - 1) / P;
    return (t + align_chunks - 1) / align_chunks * align_chunks;
}

__host__ __device__ inline int32_t cp_seq_segments(int64_t c, int64_t tau) {
    return (tau > 0 && c > tau) ? static_cast<int32_t>((c + tau - 1) / tau) : 1;
}

// Per-candidate sums over the batch (one per P = 2 .. kCpMaxSegments).
struct CpSums {
    int64_t nA, nS, max_whole, max_p;
};

__host__ __device__ inline void cp_add_sequence(CpSums& s, int64_t c, int64_t tau) {
    const int32_t P = cp_seq_segments(c, tau);
    if (P >= 2) {
        s.nA += P - 1;
        s.nS += P;
    } else if (c > s.max_whole) {
        s.max_whole = c;
    }
    if (P > s.max_p) s.max_p = P;
}

__host__ __device__ inline int64_t cp_ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Cost of a candidate in chunk periods, or -1 when it does not fit the scratch planes.
__host__ __device__ inline int64_t cp_cost(const CpSums& s, int64_t tau, int64_t sum_c, int32_t H, int32_t sms) {
    if (2 * H * s.nA > kCpMaxPlanes || H * s.nS > kCpMaxPlanes) return -1;
    const int64_t ta = cp_ceil_div(2 * H * s.nA, sms) * tau;
    int64_t tc = cp_ceil_div(H * s.nS, sms) * tau;
    const int64_t bal = cp_ceil_div(H * sum_c, sms);
    if (bal > tc) tc = bal;
    if (s.max_whole > tc) tc = s.max_whole;
    return ta + tc + (s.max_p - 1) + 4;
}

__host__ __device__ inline int64_t cp_one_pass_cost(int64_t c_max, int64_t sum_c, int32_t H, int32_t sms) {
    const int64_t bal = cp_ceil_div(H * sum_c, sms);
    return c_max > bal ? c_max : bal;
}

// Cost of candidate P (its tau from cp_tau) from its sums, or -1 when it cuts no
// sequence or does not fit the scratch planes.
__host__ __device__ inline int64_t cp_candidate_cost(const CpSums& s, int64_t tau, int64_t sum_c, int32_t H,
                                                     int32_t sms) {
    if (s.max_p < 2) return -1;
    return cp_cost(s, tau, sum_c, H, sms);
}

// The chosen tau from the candidates' costs and taus (index P - 2) and the
// cost of one pass: the cheapest feasible candidate (ties to the smaller P)
// when it costs at most 85 % of one pass, else 0 (one pass).
__host__ __device__ inline int64_t cp_choose_tau(const int64_t* cost, const int64_t* tau, int64_t one) {
    int64_t best = -1, t = 0;
    for (int32_t j = 0; j < kCpMaxSegments - 1; ++j) {
        if (cost[j] < 0) continue;
        if (best < 0 || cost[j] < best) {
            best = cost[j];
            t = tau[j];
        }
    }
    return (best >= 0 && 100 * best <= 85 * one) ? t : 0;
}

// The chosen tau from the candidates' sums (0: one pass).
__host__ __device__ inline int64_t cp_pick_tau(const CpSums (&s)[kCpMaxSegments - 1], int64_t c_max, int64_t sum_c,
                                               int32_t H, int32_t sms, int64_t align_chunks) {
    int64_t cost[kCpMaxSegments - 1], tau[kCpMaxSegments - 1];
    for (int32_t j = 0; j < kCpMaxSegments - 1; ++j) {
        tau[j] = cp_tau(c_max, j + 2, align_chunks);
        cost[j] = cp_candidate_cost(s[j], tau[j], sum_c, H, sms);
    }
    return cp_choose_tau(cost, tau, cp_one_pass_cost(c_max, sum_c, H, sms));
}

// Context-parallel arguments: the real batch, its segments and the scratch
// buffers of the transfer pass (A), the fp32 scan and the segment pass (C).
struct CpParams {
    const void* cu_seqlens;        // real [N+1]
    int cu_i64;
    int32_t num_seqs;              // N
    int32_t H;
    int32_t sms;                   // SMs of the device (the load model's S)
    int32_t align_chunks;          // segment length granularity in chunks (1, or the checkpoint interval / 64)
    int32_t nA_max;                // bound of transfer segments: rows per kind of the transfer output
    int32_t V_max;                 // bound of the segment pass's sequences (N + nA_max)
    int32_t ckpt_n;                // 0 = no checkpoints
    const void* ckpt_cu_starts;    // real [N+1]
    int ckpt_i64;
    int64_t* seg_a;                // [nA_max][2] transfer segments (start token, length)
    int32_t* order_a;              // [nA_max] identity work order of the transfer pass
    int32_t* counter_a;            // work counter of the transfer pass
    int32_t* counts;               // [0] transfer segments nA, [1] segment-pass sequences V, [2] segmented sequences
    int32_t* seg_seq;              // [nA_max][4] per segmented sequence: index, P, first transfer row, first start row
    int32_t* cu_c;                 // [V_max+1] cu_seqlens of the segment pass (a tail of empty entries)
    int64_t* ckpt_c;               // [V_max+1] its checkpoint starts
    int64_t* vrow;                 // [V_max] its state rows: start plane row, or -1 - row of the caller's state
    const float* trans;            // transfer output [2*nA_max][H][128][128]: N_s rows, then M_s rows
    float* start;                  // segment start states [nS][H][128][128] (the segment pass runs in place)
    const void* initial_state;     // real initial state (null: zeros)
    void* output_state;            // real output state (null: none)
    StateLayout state;             // its layout
    const void* state_indices;     // real pool rows (null: row = sequence)
    int idx_i64;
    int32_t* status;
};

// Arguments of the decode-step kernel (a few tokens per sequence, no chunking).
struct DecodeParams {
    const void* q;
    const void* k;
    const void* v;
    const float* g;                // nullptr: alpha = 1
    const float* beta;             // nullptr: beta = 1
    float scale;
    const void* initial_state;     // nullptr: zero state
    void* output_state;            // nullptr: state not written back
    StateLayout state;
    const void* state_indices;     // nullptr: row = sequence
    int idx_i64;
    int32_t n_pool;
    void* output;
    int32_t* status;               // nullptr: out-of-range pool rows are skipped silently
    int32_t N, H, hq, hk, hv;
    int32_t m;                     // tokens per sequence
    int l2norm;
    int32_t stages;                // shared-memory stages of the unit ring (set by the launcher)
    int32_t stage_bytes;           // bytes of one stage: state rows, then the unit's tokens
};

__host__ __device__ inline int64_t load_index(const void* p, int i64, int64_t i) {
    return i64 ? static_cast<const int64_t*>(p)[i] : static_cast<int64_t>(static_cast<const int32_t*>(p)[i]);
}

// Launchers (each file defines its own).
cudaError_t launch_prepare(const PrepareParams& p, cudaStream_t stream);
cudaError_t launch_chunk_16bit(const ChunkParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                               const CUtensorMap& tm_v, const CUtensorMap& tm_o, bool f16, bool transfer, int grid,
                               cudaStream_t stream);
// fp32 inputs: `slices` (2, 4, 8 or 16) CTAs per (sequence, state head) unit, each owning kHead / slices rows of
// the state (the rows are independent; every slice recomputes the slice-independent parts).
cudaError_t launch_chunk_f32(const ChunkParams& p, int64_t units, int slices, cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams& p, gdn_dtype dtype, cudaStream_t stream);
cudaError_t launch_cp_prepare(const CpParams& p, cudaStream_t stream);
cudaError_t launch_cp_fixup(const CpParams& p, cudaStream_t stream);
cudaError_t launch_cp_final(const CpParams& p, cudaStream_t stream);
size_t chunk_bf16_smem_bytes();
size_t plan_workspace_bytes(gdn_prefill_plan_t plan);

}  // namespace gdn
