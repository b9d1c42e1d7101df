// gdn_chunk_bf16.cu -- chunked Gated DeltaNet prefill, bf16 q/k/v, fp32 state,
// on sm_103a: tcgen05 tensor cores with TMEM accumulators, TMA-fed operands,
// warp-specialised and pipelined across chunks.
//
// Per chunk of C = 64 tokens (G_r = sum_{m<=r} log alpha_m inside the chunk,
// gamma_r = e^{G_r}; n_j, m_i = 1/|k_j|, 1/|q_i| when the L2 norm is on, else 1):
//
//   intra-chunk step ("GDN 与 Chunked Prefill": cumsum, triangular solve,
//   recompute; the 4-token expansion table generalised to a 64 x 64 table):
//     D1 = [K; Q] K^T                               tcgen05, M=128 N=64 K=128
//     A_ij = beta_i e^{G_i-G_j} n_i n_j (k_i.k_j), j < i
//     P_ij = e^{G_i-G_j} m_i n_j (q_i.k_j),       j <= i
//     T = (I + A)^-1                                blocked substitution, CUDA cores
//     W^T = K^T (T diag(beta gamma n))^T,  U^T = V^T (T diag(beta))^T   tcgen05
//   state pass ("块内 state 和块间 final state": only the chunk's last state
//   crosses the boundary):
//     Delta^T = U^T - S W^T                         tcgen05, A negated
//     S <- gamma_63 S + (Delta^T diag(e^{G_63-G_j} n_j)) K     tcgen05, in TMEM
//   output ("GDN与线性注意力GPU并行实现" section 3.3: O_init = Q S plus a
//   triangular-masked product):
//     O^T = scale (S Q^T diag(gamma m) + Delta^T P^T)           tcgen05
//
// The L2 norm of q and k ("FlashInfer GDN Prefill 完全指南", API table) enters
// only as the per-row factors n and m above, applied in fp32: the same values
// as normalising the rows first, without re-rounding them to bf16.
//
// Roles (384 threads, one work unit = (sequence, state head) at a time,
// units taken longest first from an atomic counter):
//   warp 0      TMA: K, Q tiles (2 stages) and V tile; unit scheduler
//   warp 1      tcgen05 issue for the intra-chunk products (D1, W, U)
//   warp 2      tcgen05 issue for the state chain (Delta, S Q^T, Delta P^T, S)
//   warp 3      TMEM allocation
//   warps 4-7   intra warpgroup: gates, A and P, T, W to shared memory,
//               one chunk ahead of the state warpgroup
//   warps 8-11  state warpgroup: Delta epilogue, state epilogue (next S
//               operand, checkpoints, final state), output epilogue
// Every wait is bounded; a timeout sets GDN_DEVICE_ERR_TIMEOUT, raises a
// shared abort flag that every other wait polls, drains the CTA's in-flight
// copies and tensor-core work, frees TMEM and returns.
#include <cuda_bf16.h>

#include "gdn_internal.cuh"
#include "sm103_ptx.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 640;
constexpr int kStateThreads = 256;  // two state warpgroups
constexpr int kIntraThreads = 256;  // two intra warpgroups
constexpr uint32_t kRegsLaunch = 96, kRegsSched = 64, kRegsIntra = 96, kRegsState = 104;  // per thread
constexpr uint32_t kBarIntra = 1, kBarState = 2;  // named barrier ids

// ---- shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t kKQ = 0;           // 2 stages x 32 KB: K_h0 | Q_h0 | K_h1 | Q_h1 (64 rows x 128 B each)
constexpr uint32_t kKQStage = 32768;
constexpr uint32_t kV = 65536;        // V_h0 | V_h1
constexpr uint32_t kTp = 81920;       // T diag(beta gamma n) bf16 [64 i][64 j] K-major
constexpr uint32_t kTpp = 90112;      // T diag(beta)
constexpr uint32_t kPb = 98304;       // 2 x P bf16 [64 i][64 j] K-major
constexpr uint32_t kWb = 114688;      // W^T bf16 as MN-major B: [128 k][64 i]
constexpr uint32_t kSb = 131072;      // S bf16 K-major: 2 halves of [128 v][64 k]
constexpr uint32_t kAbuf = 163840;    // A fp32 [64][kLd]
constexpr uint32_t kTbuf = 181248;    // T fp32 [64][kLd]
constexpr uint32_t kXs = 198656;      // inverse scratch: [2][16][20] then [32][36] fp32
constexpr uint32_t kOutT = 205824;    // output tile bf16 [64 i][128 v]
constexpr uint32_t kGbuf = 222208;    // 2 x kGFloats floats of per-row / per-column factors (see kG*)
constexpr uint32_t kBars = 229504;    // 32 mbarriers
constexpr uint32_t kRing = 229760;    // 2 unit descriptors
constexpr uint32_t kMisc = 229888;    // tmem base, abort flag
constexpr uint32_t kSmemBytes = 229952;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;
constexpr int kLd = 68;               // fp32 row stride of A and T (bank-conflict free rows)

// gbuf field offsets (floats), one 64-vector each, per chunk:
//   G      running sum of log alpha            gamma  e^G
//   beta   beta (0 on padded rows)             rn, rm 1/|k_j|, 1/|q_i| (1 without the L2 norm)
//   cw     beta_j gamma_j rn_j (T' columns)    dec    e^{G_63 - G_j} rn_j (decayed Delta columns)
//   orow   scale gamma_i rm_i (output rows)    ra     beta_i rn_i (A rows)
//   colf   rn_j e^{G_16b - G_j}, b = j / 16      rowf   [4][64] e^{G_i - G_16b} (i >= 16 b, else 0)
//   safe   1 when the chunk's G range is small enough for e^{G_i - G_j} = rowf * colf
constexpr int kGG = 0, kGGam = 64, kGBeta = 128, kGRn = 192, kGRm = 256, kGCw = 320, kGDec = 384, kGOr = 448,
              kGRa = 512, kGColf = 576, kGRowf = 640, kGSafe = 896, kGFloats = 912;
static_assert(2 * kGFloats * 4 <= kBars - kGbuf, "gbuf overflows");

// ---- barriers
enum {
    B_KQ_FULL = 0, B_KQ_EMPTY = 2, B_V_FULL = 4, B_V_EMPTY = 5, B_D1_FULL = 6, B_D1_EMPTY = 7, B_T_FULL = 8,
    B_WU_FULL = 9, B_WB_FULL = 10, B_SB_FULL = 12, B_DELTA_FULL = 14, B_DD_FULL = 16, B_S_FULL = 18,
    B_O_EMPTY = 20, B_GATES_FULL = 22, B_GATES_EMPTY = 24, B_UNIT_FULL = 26, B_UNIT_EMPTY = 28,
    B_DRAIN_I = 30, B_DRAIN_S = 31, B_COUNT = 32
};

// ---- TMEM columns
constexpr uint32_t kTmS = 0, kTmDelta = 128 /* 2 x 64 */, kTmW = 256, kTmD1 = 320, kTmO1 = 384, kTmO2 = 448;
constexpr uint32_t kTmCols = 512;

constexpr uint32_t kIdescD1 = idesc_bf16_f32(128, 64);
constexpr uint32_t kIdescWU = idesc_bf16_f32(128, 64, true, false);
constexpr uint32_t kIdescDelta = idesc_bf16_f32(128, 64, false, true, true);
constexpr uint32_t kIdescO = idesc_bf16_f32(128, 64);
constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, true);

constexpr long long kWaitCycles = 2000000000LL;  // about one second

struct UnitInfo {
    int32_t valid, seq, h, nC;
    int32_t qh, kh, vh, flat0;
    int64_t t0, L, srow, ckpt_base;
};
static_assert(sizeof(UnitInfo) <= 64, "unit descriptor slot");

struct Ctx {
    uint8_t* sm;
    uint64_t* bars;
    volatile int32_t* abort;
    int32_t* status;
};

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_bar(const Ctx& cx, int b, uint32_t parity) {
    uint64_t* bar = cx.bars + b;
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 2000)) return true;
        if (*cx.abort) return false;
        if (clock64() - t0 > kWaitCycles) {
            atomicOr(cx.status, static_cast<int32_t>(GDN_DEVICE_ERR_TIMEOUT));
            *cx.abort = 1;
            return false;
        }
    }
}

// Bounded wait used while draining (ignores the abort flag).
__device__ __forceinline__ void drain_bar(const Ctx& cx, int b, uint32_t parity) {
    if (!mbar_wait(cx.bars + b, parity, kWaitCycles)) atomicOr(cx.status, static_cast<int32_t>(GDN_DEVICE_ERR_TIMEOUT));
}

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

__device__ __forceinline__ UnitInfo read_unit(const uint8_t* sm, int slot) {
    return *reinterpret_cast<const UnitInfo*>(sm + kRing + slot * 64);
}

// ===========================================================================
// Triangular inverse T = (I + A)^-1 of a strictly lower 64 x 64 A (fp32,
// rows of kLd floats), by the two intra warpgroups (256 threads, 8 warps):
//   level 0: the four 16 x 16 diagonal blocks by forward substitution, one
//            column per thread (fp32);
//   level 1: T_ab = -T_aa A_ab T_bb for (a, b) = (1, 0), (3, 2);
//   level 2: T_21 = -T_22 A_21 T_11 on 32 x 32 blocks.
// The level 1 and 2 products are 16- and 32-row matrices, below the 64-row
// minimum of tcgen05.mma, so they run as warp-level m16n8k8 tf32 MMAs (fp32
// accumulate); T is later rounded to bf16 for the W and U products anyway.
// On return T holds the lower triangle including the diagonal; the upper
// triangle is unspecified.
// ===========================================================================
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// D (16 x 8) += A (16 x 8, row-major, stride lda) * B (8 x 8, row-major K x N, stride ldb)
__device__ __forceinline__ void mma_tf32_16x8x8(float (&d)[4], const float* A, int lda, const float* B, int ldb,
                                                int lane) {
    const int g = lane >> 2, t = lane & 3;
    const uint32_t a0 = to_tf32(A[g * lda + t]), a1 = to_tf32(A[(g + 8) * lda + t]);
    const uint32_t a2 = to_tf32(A[g * lda + t + 4]), a3 = to_tf32(A[(g + 8) * lda + t + 4]);
    const uint32_t b0 = to_tf32(B[t * ldb + g]), b1 = to_tf32(B[(t + 4) * ldb + g]);
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Store a 16 x 8 accumulator tile (times `sign`) to row-major C.
__device__ __forceinline__ void store_tile_16x8(float* C, int ldc, const float (&d)[4], float sign, int lane) {
    const int g = lane >> 2, t = lane & 3;
    *reinterpret_cast<float2*>(C + g * ldc + 2 * t) = make_float2(sign * d[0], sign * d[1]);
    *reinterpret_cast<float2*>(C + (g + 8) * ldc + 2 * t) = make_float2(sign * d[2], sign * d[3]);
}

__device__ void tri_inverse_64(const float* __restrict__ A, float* __restrict__ T, float* __restrict__ X1,
                               float* __restrict__ X2, int t) {
    const int wi = t >> 5, lane = t & 31;  // warp index 0..7 within the intra groups
    if (t < 64) {
        const int o = (t >> 4) * 16, col = t & 15;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const float* arow = A + (o + r) * kLd + o;
            float acc0 = (r == col) ? 1.f : 0.f, acc1 = 0.f;
#pragma unroll
            for (int m = 0; m + 1 < r; m += 2) {
                acc0 -= arow[m] * x[m];
                acc1 -= arow[m + 1] * x[m + 1];
            }
            if (r & 1) acc0 -= arow[r - 1] * x[r - 1];
            x[r] = (r < col) ? 0.f : acc0 + acc1;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) T[(o + r) * kLd + o + col] = x[r];
    } else if (t < 128) {
        // zero the upper blocks (0,1) and (2,3) so that T_11, T_22 read as triangular
        const int idx = t - 64;            // 64 threads x 8 values = 2 blocks x 256
        const int blk = idx >> 5, r = (idx & 31) >> 1, c0 = (idx & 1) * 8;
        const int ro = blk * 32, co = blk * 32 + 16;
#pragma unroll
        for (int q = 0; q < 8; ++q) T[(ro + r) * kLd + co + c0 + q] = 0.f;
    }
    named_bar_sync(kBarIntra, kIntraThreads);
    // level 1: warps 0..3 each own one 16 x 8 output tile: block pair pr = wi >> 1, columns nt = wi & 1
    if (wi < 4) {
        const int pr = wi >> 1, nt = (wi & 1) * 8, a = 2 * pr + 1, b = 2 * pr;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k0 = 0; k0 < 16; k0 += 8)   // X_ab = A_ab T_bb
            mma_tf32_16x8x8(d, A + (16 * a) * kLd + 16 * b + k0, kLd, T + (16 * b + k0) * kLd + 16 * b + nt, kLd, lane);
        store_tile_16x8(X1 + pr * 16 * 20 + nt, 20, d, 1.f, lane);
    }
    named_bar_sync(kBarIntra, kIntraThreads);
    if (wi < 4) {
        const int pr = wi >> 1, nt = (wi & 1) * 8, a = 2 * pr + 1, b = 2 * pr;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k0 = 0; k0 < 16; k0 += 8)   // T_ab = -T_aa X_ab
            mma_tf32_16x8x8(d, T + (16 * a) * kLd + 16 * a + k0, kLd, X1 + pr * 16 * 20 + k0 * 20 + nt, 20, lane);
        store_tile_16x8(T + (16 * a) * kLd + 16 * b + nt, kLd, d, -1.f, lane);
    }
    named_bar_sync(kBarIntra, kIntraThreads);
    // level 2: eight warps, one 16 x 8 tile each of the 32 x 32 products
    {
        const int mt = (wi >> 2) * 16, nt = (wi & 3) * 8;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k0 = 0; k0 < 32; k0 += 8)   // X = A_21 T_11
            mma_tf32_16x8x8(d, A + (32 + mt) * kLd + k0, kLd, T + k0 * kLd + nt, kLd, lane);
        store_tile_16x8(X2 + mt * 36 + nt, 36, d, 1.f, lane);
        named_bar_sync(kBarIntra, kIntraThreads);
        float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k0 = 0; k0 < 32; k0 += 8)   // T_21 = -T_22 X
            mma_tf32_16x8x8(e, T + (32 + mt) * kLd + 32 + k0, kLd, X2 + k0 * 36 + nt, 36, lane);
        store_tile_16x8(T + (32 + mt) * kLd + nt, kLd, e, -1.f, lane);
    }
    named_bar_sync(kBarIntra, kIntraThreads);
}

// ===========================================================================
// Gates of one chunk (one warp; lane l owns rows 2l, 2l+1).  load_gates issues
// the global loads early (alpha = 1, beta = 0 on padded rows); compute_gates
// forms G = running sum of log alpha, gamma = e^G and the factor vectors as
// they are without the L2 norm (rn = rm = 1).
// ===========================================================================
struct GatePrefetch {
    float a0, a1, b0, b1;
};

__device__ __forceinline__ GatePrefetch load_gates(const ChunkParams& p, int64_t tc, int32_t Lc, int32_t h, int lane) {
    GatePrefetch g{1.f, 1.f, 0.f, 0.f};
    const int r0 = 2 * lane, r1 = r0 + 1;
    if (r0 < Lc) {
        const size_t gi = static_cast<size_t>(tc + r0) * p.H + h;
        g.a0 = p.g ? p.g[gi] : 1.f;
        g.b0 = p.beta ? p.beta[gi] : 1.f;
    }
    if (r1 < Lc) {
        const size_t gi = static_cast<size_t>(tc + r1) * p.H + h;
        g.a1 = p.g ? p.g[gi] : 1.f;
        g.b1 = p.beta ? p.beta[gi] : 1.f;
    }
    return g;
}

// Sum of squares of row r of a staged 64 x 128 bf16 tile (two 64-column
// halves 16 KB apart, 128-byte swizzle).
__device__ __forceinline__ float row_sumsq(const uint8_t* half0, int r) {
    float ss = 0.f;
#pragma unroll 4
    for (int c = 0; c < 16; ++c) {
        float f[8];
        bf16x8_to_float(*reinterpret_cast<const uint4*>(half0 + (c >> 3) * 16384 + sw128_offset(r, c & 7)), f);
#pragma unroll
        for (int j = 0; j < 8; ++j) ss += f[j] * f[j];
    }
    return ss;
}

// The vectors of one chunk (see kG*): G, gamma, beta, and cw, dec, ra, colf
// as they are with unit key norms (rn = 1), orow and rm with the query norms
// when `q` (the staged Q tile) is given, else with rm = 1.  The intra
// warpgroups multiply the key norms in once the K K^T diagonal is known.
// Rows at or past Lc are padding (alpha = 1, beta = 0, rm = 0).
__device__ void compute_gates(const GatePrefetch& g, float* gb, float scale, const uint8_t* q, int32_t Lc, int lane) {
    const int r0 = 2 * lane, r1 = r0 + 1;
    const float la0 = __logf(g.a0), la1 = __logf(g.a1);
    float incl = la0 + la1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const float G1 = incl, G0 = incl - la1;
    const float G63 = __shfl_sync(0xffffffffu, incl, 31);
    float Gb[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) Gb[b] = __shfl_sync(0xffffffffu, G0, 8 * b);  // G at row 16 b
    float rm0 = 1.f, rm1 = 1.f;
    if (q) {
        rm0 = r0 < Lc ? rsqrtf(row_sumsq(q, r0) + 1e-6f) : 0.f;
        rm1 = r1 < Lc ? rsqrtf(row_sumsq(q, r1) + 1e-6f) : 0.f;
    }
    const float Gv[2] = {G0, G1}, bv[2] = {g.b0, g.b1}, rmv[2] = {rm0, rm1};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int r = r0 + k;
        const float e = __expf(Gv[k]);
        gb[kGG + r] = Gv[k];
        gb[kGGam + r] = e;
        gb[kGBeta + r] = bv[k];
        gb[kGRn + r] = 1.f;
        gb[kGRm + r] = rmv[k];
        gb[kGCw + r] = bv[k] * e;
        gb[kGDec + r] = __expf(G63 - Gv[k]);
        gb[kGOr + r] = scale * e * rmv[k];
        gb[kGRa + r] = bv[k];
        gb[kGColf + r] = __expf(Gb[r >> 4] - Gv[k]);
#pragma unroll
        for (int b = 0; b < 4; ++b) gb[kGRowf + b * 64 + r] = (r >= 16 * b) ? __expf(Gv[k] - Gb[b]) : 0.f;
    }
    float gmax = fmaxf(G0, G1), gmin = fminf(G0, G1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
        gmin = fminf(gmin, __shfl_xor_sync(0xffffffffu, gmin, o));
    }
    if (lane == 0) gb[kGSafe] = (gmax - gmin < 60.f) ? 1.f : 0.f;
}

__device__ __forceinline__ void tmem_ld16_wait(uint32_t taddr, uint32_t (&r)[16]) {
    tmem_ld16(taddr, r);
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15])
                 :
                 : "memory");
}

__device__ __forceinline__ void lds16(const float* src, float* x) {
#pragma unroll
    for (int q = 0; q < 16; q += 4) {
        const float4 v = *reinterpret_cast<const float4*>(src + q);
        x[q] = v.x;
        x[q + 1] = v.y;
        x[q + 2] = v.z;
        x[q + 3] = v.w;
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    gdn_chunk_bf16_kernel(const ChunkParams p, const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_o) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    Ctx cx;
    cx.sm = sm;
    cx.bars = reinterpret_cast<uint64_t*>(sm + kBars);
    cx.abort = reinterpret_cast<volatile int32_t*>(sm + kMisc + 4);
    cx.status = p.status;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + kMisc);

    // Bad input flagged by the prepare kernel: every thread sees one copy of the word.
    if (tid == 0) *cx.abort = *reinterpret_cast<volatile int32_t*>(p.status);
    __syncthreads();
    if (*cx.abort != 0) return;
    __syncthreads();

    if (tid == 0) {
        for (int b = 0; b < B_COUNT; ++b) mbar_init(cx.bars + b, 1);
        mbar_init(cx.bars + B_UNIT_EMPTY + 0, 5);
        mbar_init(cx.bars + B_UNIT_EMPTY + 1, 5);
        fence_mbar_init();
        if (p.has_tokens) {
            prefetch_tensormap(&tm_q);
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
            prefetch_tensormap(&tm_o);
        }
    }
    for (uint32_t off = tid * 16; off < 32768; off += kThreads * 16)  // T', T'' and both P buffers
        *reinterpret_cast<uint4*>(sm + kTp + off) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp == 3) {
        tmem_alloc(s_tmem, kTmCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const int32_t H = p.H;
    // register split: launch 640 x 96; the scheduling warpgroup gives up 32 a thread, the state ones take 8 more
    // (128 x 64 + 256 x 96 + 256 x 104 <= 640 x 96)
    static_assert(128 * kRegsSched + kIntraThreads * kRegsIntra + kStateThreads * kRegsState <= kThreads * kRegsLaunch,
                  "register split exceeds the launch budget");
    const int64_t units = static_cast<int64_t>(p.num_seqs) * H;

    if (warp < 4) {
        // the scheduling warpgroup: TMA producer, two MMA issuers, gates warp
        regs_dec<kRegsSched>();
        if (warp == 0) {
            // ================= TMA producer and unit scheduler =================
            if (lane == 0) {
                uint32_t n = 0, u = 0;
                int issued_kq[2] = {-1, -1};
                int issued_v = -1;
                for (;;) {
                    const int64_t uid = atomicAdd(p.counter, 1);
                    const int slot = u & 1;
                    if (u >= 2 && !wait_bar(cx, B_UNIT_EMPTY + slot, ((u - 2) >> 1) & 1)) break;
                    UnitInfo info;
                    info.valid = uid < units ? 1 : 0;
                    int32_t nC = 0;
                    if (info.valid) {
                        const int32_t seq = p.seq_order[uid / H];
                        const int32_t h = static_cast<int32_t>(uid % H);
                        info.seq = seq;
                        info.h = h;
                        info.t0 = load_index(p.cu_seqlens, p.cu_i64, seq);
                        info.L = load_index(p.cu_seqlens, p.cu_i64, seq + 1) - info.t0;
                        nC = static_cast<int32_t>((info.L + kChunk - 1) / kChunk);
                        info.nC = nC;
                        info.qh = h / (H / p.hq);
                        info.kh = h / (H / p.hk);
                        info.vh = h / (H / p.hv);
                        info.flat0 = p.chunk_offsets[seq];
                        info.srow = p.state_indices ? load_index(p.state_indices, p.idx_i64, seq) : seq;
                        info.ckpt_base = p.ckpt_n > 0 ? load_index(p.ckpt_cu_starts, p.ckpt_i64, seq) : 0;
                    }
                    *reinterpret_cast<UnitInfo*>(sm + kRing + slot * 64) = info;
                    mbar_arrive(cx.bars + B_UNIT_FULL + slot);
                    ++u;
                    if (!info.valid) break;
                    bool ok = true;
                    for (int32_t c = 0; c < nC && ok; ++c, ++n) {
                        const int s = n & 1;
                        const int32_t t = static_cast<int32_t>(info.t0 + static_cast<int64_t>(c) * kChunk);
                        if (n >= 2 && !(ok = wait_bar(cx, B_KQ_EMPTY + s, ((n - 2) >> 1) & 1))) break;
                        uint8_t* st = sm + kKQ + s * kKQStage;
                        uint64_t* fb = cx.bars + B_KQ_FULL + s;
                        mbar_arrive_expect_tx(fb, kKQStage);
                        tma_load_3d(st + 0, &tm_k, fb, 0, info.kh, t);
                        tma_load_3d(st + 8192, &tm_q, fb, 0, info.qh, t);
                        tma_load_3d(st + 16384, &tm_k, fb, 64, info.kh, t);
                        tma_load_3d(st + 24576, &tm_q, fb, 64, info.qh, t);
                        issued_kq[s] = static_cast<int>(n);
                        if (n >= 1 && !(ok = wait_bar(cx, B_V_EMPTY, (n - 1) & 1))) break;
                        uint64_t* vb = cx.bars + B_V_FULL;
                        mbar_arrive_expect_tx(vb, 16384);
                        tma_load_3d(sm + kV, &tm_v, vb, 0, info.vh, t);
                        tma_load_3d(sm + kV + 8192, &tm_v, vb, 64, info.vh, t);
                        issued_v = static_cast<int>(n);
                    }
                    if (!ok) break;
                }
                // drain: every issued load has landed before the CTA may exit
                for (int s = 0; s < 2; ++s)
                    if (issued_kq[s] >= 0) drain_bar(cx, B_KQ_FULL + s, (issued_kq[s] >> 1) & 1);
                if (issued_v >= 0) drain_bar(cx, B_V_FULL, issued_v & 1);
            }
        } else if (warp == 1) {
            // ================= tcgen05 issue: D1, W, U =================
            if (lane == 0) {
                uint32_t n = 0, u = 0;
                bool ok = true;
                for (; ok;) {
                    const int slot = u & 1;
                    if (!(ok = wait_bar(cx, B_UNIT_FULL + slot, (u >> 1) & 1))) break;
                    const UnitInfo info = read_unit(sm, slot);
                    mbar_arrive(cx.bars + B_UNIT_EMPTY + slot);
                    ++u;
                    if (!info.valid) break;
                    for (int32_t c = 0; c < info.nC; ++c, ++n) {
                        const int s = n & 1;
                        if (!(ok = wait_bar(cx, B_KQ_FULL + s, (n >> 1) & 1))) break;
                        if (n >= 1 && !(ok = wait_bar(cx, B_D1_EMPTY, (n - 1) & 1))) break;
                        tc_fence_after();
                        const uint32_t kq = smem_u32(sm + kKQ + s * kKQStage);
    #pragma unroll
                        for (int ks = 0; ks < 8; ++ks) {
                            const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                            mma_bf16_ss(tmem + kTmD1, desc_kmajor_sw128(kq + off), desc_kmajor_sw128(kq + off), kIdescD1,
                                        ks > 0);
                        }
                        mma_commit(cx.bars + B_D1_FULL);
                        if (!(ok = wait_bar(cx, B_T_FULL, n & 1))) break;
                        if (!(ok = wait_bar(cx, B_V_FULL, n & 1))) break;
                        if (n >= 2 && !(ok = wait_bar(cx, B_S_FULL + s, ((n - 2) >> 1) & 1))) break;
                        tc_fence_after();
                        const uint32_t vv = smem_u32(sm + kV);
                        const uint32_t tp = smem_u32(sm + kTp), tpp = smem_u32(sm + kTpp);
                        const uint32_t dbuf = tmem + kTmDelta + s * 64;
    #pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            mma_bf16_ss(tmem + kTmW, desc_mnmajor_sw128(kq + ks * 2048, 16384),
                                        desc_kmajor_sw128(tp + ks * 32), kIdescWU, ks > 0);
                            mma_bf16_ss(dbuf, desc_mnmajor_sw128(vv + ks * 2048, 8192), desc_kmajor_sw128(tpp + ks * 32),
                                        kIdescWU, ks > 0);
                        }
                        mma_commit(cx.bars + B_WU_FULL);
                        mma_commit(cx.bars + B_V_EMPTY);
                    }
                }
                mma_commit(cx.bars + B_DRAIN_I);
                drain_bar(cx, B_DRAIN_I, 0);
            }
        } else if (warp == 2) {
            // ================= tcgen05 issue: Delta, S Q^T, Delta P^T, S =================
            if (lane == 0) {
                uint32_t n = 0, u = 0;
                bool ok = true;
                for (; ok;) {
                    const int slot = u & 1;
                    if (!(ok = wait_bar(cx, B_UNIT_FULL + slot, (u >> 1) & 1))) break;
                    const UnitInfo info = read_unit(sm, slot);
                    mbar_arrive(cx.bars + B_UNIT_EMPTY + slot);
                    ++u;
                    if (!info.valid) break;
                    for (int32_t c = 0; c < info.nC; ++c, ++n) {
                        const int s = n & 1;
                        const uint32_t ph = (n >> 1) & 1;
                        if (!(ok = wait_bar(cx, B_WB_FULL + s, ph))) break;
                        if (!(ok = wait_bar(cx, B_SB_FULL + s, ph))) break;
                        if (!(ok = wait_bar(cx, B_KQ_FULL + s, ph))) break;
                        tc_fence_after();
                        const uint32_t kq = smem_u32(sm + kKQ + s * kKQStage);
                        const uint32_t sb = smem_u32(sm + kSb), wb = smem_u32(sm + kWb);
                        const uint32_t dbuf = tmem + kTmDelta + s * 64;
    #pragma unroll
                        for (int ks = 0; ks < 8; ++ks) {
                            const uint32_t aoff = (ks >> 2) * 16384 + (ks & 3) * 32;
                            mma_bf16_ss(dbuf, desc_kmajor_sw128(sb + aoff), desc_mnmajor_sw128(wb + ks * 2048, 8192),
                                        kIdescDelta, 1);
                        }
                        mma_commit(cx.bars + B_DELTA_FULL + s);
                        if (n >= 1 && !(ok = wait_bar(cx, B_O_EMPTY + ((n - 1) & 1), ((n - 1) >> 1) & 1))) break;
                        tc_fence_after();
    #pragma unroll
                        for (int ks = 0; ks < 8; ++ks) {
                            const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                            mma_bf16_ss(tmem + kTmO1, desc_kmajor_sw128(sb + off), desc_kmajor_sw128(kq + 8192 + off),
                                        kIdescO, ks > 0);
                        }
                        if (!(ok = wait_bar(cx, B_DD_FULL + s, ph))) break;
                        tc_fence_after();
                        const uint32_t pb = smem_u32(sm + kPb + s * 8192);
    #pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            const uint32_t acol = dbuf + 32 * (ks >> 1) + 8 * (ks & 1);  // packed j = 16 ks .. 16 ks + 15
                            mma_bf16_ts(tmem + kTmO2, acol, desc_kmajor_sw128(pb + ks * 32), kIdescO, ks > 0);
                            mma_bf16_ts(tmem + kTmS, acol + 16, desc_mnmajor_sw128(kq + ks * 2048, 16384), kIdescS, 1);
                        }
                        mma_commit(cx.bars + B_S_FULL + s);
                        mma_commit(cx.bars + B_KQ_EMPTY + s);
                    }
                }
                mma_commit(cx.bars + B_DRAIN_S);
                drain_bar(cx, B_DRAIN_S, 0);
            }
        } else if (warp == 3) {
            // ================= gates warp: G, gamma, beta and factor vectors per chunk =================
            uint32_t n = 0, u = 0;
            bool ok = true;
            for (; ok;) {
                const int slot = u & 1;
                if (!(ok = wait_bar(cx, B_UNIT_FULL + slot, (u >> 1) & 1))) break;
                const UnitInfo info = read_unit(sm, slot);
                __syncwarp();
                if (lane == 0) mbar_arrive(cx.bars + B_UNIT_EMPTY + slot);
                ++u;
                if (!info.valid) break;
                GatePrefetch gpf{1.f, 1.f, 0.f, 0.f};
                if (info.nC > 0)
                    gpf = load_gates(p, info.t0, info.L < kChunk ? static_cast<int32_t>(info.L) : kChunk, info.h, lane);
                for (int32_t c = 0; c < info.nC; ++c, ++n) {
                    const int gs = n & 1;
                    const GatePrefetch cur = gpf;
                    if (c + 1 < info.nC) {
                        const int64_t rem1 = info.L - static_cast<int64_t>(c + 1) * kChunk;
                        gpf = load_gates(p, info.t0 + static_cast<int64_t>(c + 1) * kChunk,
                                         rem1 < kChunk ? static_cast<int32_t>(rem1) : kChunk, info.h, lane);
                    }
                    if (n >= 2 && !(ok = wait_bar(cx, B_GATES_EMPTY + gs, ((n - 2) >> 1) & 1))) break;
                    const uint8_t* qt = nullptr;
                    if (p.l2norm) {
                        if (!(ok = wait_bar(cx, B_KQ_FULL + gs, (n >> 1) & 1))) break;
                        qt = sm + kKQ + gs * kKQStage + 8192;
                    }
                    const int64_t rem = info.L - static_cast<int64_t>(c) * kChunk;
                    compute_gates(cur, reinterpret_cast<float*>(sm + kGbuf) + gs * kGFloats, p.scale, qt,
                                  rem < kChunk ? static_cast<int32_t>(rem) : kChunk, lane);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(cx.bars + B_GATES_FULL + gs);
                }
            }
        }
    } else if (warp < 12) {
        if (kRegsIntra > kRegsLaunch) regs_inc<kRegsIntra>();
        // ================= intra warpgroups (two; each TMEM lane row split in column halves) =================
        const int it = tid - 128;                      // 0..255
        const int wq = warp & 3;                       // TMEM lane quarter
        const int hh = (warp - 4) >> 2;                // column half
        const int r = wq * 32 + lane;                  // TMEM lane: A row r (< 64) or P row r - 64
        const uint32_t tm_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const int imax = (wq & 1) * 32 + 31;           // last A or P row of this warp
        float* Abuf = reinterpret_cast<float*>(sm + kAbuf);
        float* Tbuf = reinterpret_cast<float*>(sm + kTbuf);
        float* X1 = reinterpret_cast<float*>(sm + kXs);
        float* X2 = X1 + 2 * 16 * 20;
        uint32_t n = 0, u = 0;
        bool ok = true;
        for (; ok;) {
            const int slot = u & 1;
            if (!(ok = wait_bar(cx, B_UNIT_FULL + slot, (u >> 1) & 1))) break;
            const UnitInfo info = read_unit(sm, slot);
            named_bar_sync(kBarIntra, kIntraThreads);
            if (it == 0) mbar_arrive(cx.bars + B_UNIT_EMPTY + slot);
            ++u;
            if (!info.valid) break;
            for (int32_t c = 0; c < info.nC && ok; ++c, ++n) {
                const int s = n & 1;
                const int64_t rem = info.L - static_cast<int64_t>(c) * kChunk;
                const int32_t Lc = rem < kChunk ? static_cast<int32_t>(rem) : kChunk;
                float* gb = reinterpret_cast<float*>(sm + kGbuf) + s * kGFloats;
                uint8_t* kqs = sm + kKQ + s * kKQStage;
                if (!(ok = wait_bar(cx, B_GATES_FULL + s, (n >> 1) & 1))) break;
                // P buffer s is free once O2 of chunk n-2 has completed
                if (n >= 2 && !(ok = wait_bar(cx, B_S_FULL + s, ((n - 2) >> 1) & 1))) break;
                if (!(ok = wait_bar(cx, B_D1_FULL, n & 1))) break;
                tc_fence_after();
                if (p.l2norm) {
                    // k norms: the diagonal of K K^T (lanes 0..63)
                    if (hh == 0 && r < 64) {
                        uint32_t rr[32];
                        tmem_ld32_wait(tm_lane + kTmD1 + 32 * wq, rr);
                        float kk = 0.f;
#pragma unroll
                        for (int j = 0; j < 32; ++j) kk = (j == lane) ? __uint_as_float(rr[j]) : kk;
                        const float rn = r < Lc ? rsqrtf(kk + 1e-6f) : 0.f;
                        gb[kGRn + r] = rn;
                        gb[kGRa + r] *= rn;
                    }
                    named_bar_sync(kBarIntra, kIntraThreads);
                    if (hh == 1 && r < 64) {  // column factors that meet n_j (read only after T')
                        const float rn = gb[kGRn + r];
                        gb[kGCw + r] *= rn;
                        gb[kGDec + r] *= rn;
                    }
                }
                // A rows (lanes 0..63) and P rows (lanes 64..127), this warp's 32 columns, 16 per step;
                // blocks entirely above the diagonal are skipped (A's upper part is never read, P's stays zero).
                // e^{G_i - G_j} = rowf[b][i] colf[j] inside column block b when the chunk's gate range is
                // moderate, else computed pairwise.
                {
                    const bool arow = r < 64;
                    const int i = r & 63;
                    const bool safe = gb[kGSafe] != 0.f;
                    const float rbase = arow ? gb[kGRa + i] : gb[kGRm + i];
                    uint8_t* pb = sm + kPb + s * 8192;
#pragma unroll 1
                    for (int jb = 32 * hh; jb < 32 * hh + 32; jb += 16) {
                        if (jb > imax) break;  // warp-uniform
                        uint32_t rr[16];
                        tmem_ld16_wait(tm_lane + kTmD1 + jb, rr);
                        float x[16];
                        if (safe) {
                            float cj[16], nj[16];
                            lds16(gb + kGColf + jb, cj);
                            lds16(gb + kGRn + jb, nj);
                            const float rf = rbase * gb[kGRowf + (jb >> 4) * 64 + i];
#pragma unroll
                            for (int q = 0; q < 16; ++q) {
                                const int j = jb + q;
                                const bool keep = arow ? (j < i) : (j <= i);
                                x[q] = keep ? rf * cj[q] * nj[q] * __uint_as_float(rr[q]) : 0.f;
                            }
                        } else {
                            float gj[16], nj[16];
                            lds16(gb + kGG + jb, gj);
                            lds16(gb + kGRn + jb, nj);
                            const float Gi = gb[kGG + i];
#pragma unroll
                            for (int q = 0; q < 16; ++q) {
                                const int j = jb + q;
                                const bool keep = arow ? (j < i) : (j <= i);
                                x[q] = keep ? rbase * __expf(Gi - gj[q]) * nj[q] * __uint_as_float(rr[q]) : 0.f;
                            }
                        }
                        if (arow) {
#pragma unroll
                            for (int q = 0; q < 16; q += 4)
                                *reinterpret_cast<float4*>(Abuf + i * kLd + jb + q) =
                                    make_float4(x[q], x[q + 1], x[q + 2], x[q + 3]);
                        } else {
                            st_chunk_bf16(pb, i, jb >> 3, x);
                            st_chunk_bf16(pb, i, (jb >> 3) + 1, x + 8);
                        }
                    }
                }
                // zero the padded rows of the K and V tiles (they hold the next
                // sequence or TMA zero fill; only exact zeros may meet them)
                if (Lc < kChunk) {
                    if (!(ok = wait_bar(cx, B_V_FULL, n & 1))) break;
                    const int zr = it & 63;
                    if (it < 128 && zr >= Lc) {
                        const uint4 z = make_uint4(0, 0, 0, 0);
                        uint8_t* base = (it < 64) ? kqs : sm + kV;
                        const uint32_t hs = (it < 64) ? 16384 : 8192;
#pragma unroll
                        for (int cch = 0; cch < 16; ++cch)
                            *reinterpret_cast<uint4*>(base + (cch >> 3) * hs + sw128_offset(zr, cch & 7)) = z;
                    }
                }
                tc_fence_before();  // P and the zeroed tile rows reach the async proxy with the T' and Wb fences
                named_bar_sync(kBarIntra, kIntraThreads);
                if (it == 0) mbar_arrive(cx.bars + B_D1_EMPTY);
                // T = (I + A)^-1, then T' = T diag(cw) (lanes 0..63), T'' = T diag(beta) (64..127)
                tri_inverse_64(Abuf, Tbuf, X1, X2, it);
                {
                    const bool wpart = r < 64;
                    const int i = r & 63;
                    uint8_t* dst = sm + (wpart ? kTp : kTpp);
                    const float* trow = Tbuf + i * kLd;
                    const float* cf = gb + (wpart ? kGCw : kGBeta);
#pragma unroll 1
                    for (int j0 = 32 * hh; j0 < 32 * hh + 32; j0 += 8) {
                        if (j0 > imax) break;  // warp-uniform; these chunks stay zero
                        const float4 t0 = *reinterpret_cast<const float4*>(trow + j0);
                        const float4 t1 = *reinterpret_cast<const float4*>(trow + j0 + 4);
                        const float4 c0 = *reinterpret_cast<const float4*>(cf + j0);
                        const float4 c1 = *reinterpret_cast<const float4*>(cf + j0 + 4);
                        const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
                        const float cv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                        float x[8];
#pragma unroll
                        for (int q = 0; q < 8; ++q) x[q] = (j0 + q <= i) ? tv[q] * cv[q] : 0.f;
                        st_chunk_bf16(dst, i, j0 >> 3, x);
                    }
                }
                fence_proxy_async_smem();
                named_bar_sync(kBarIntra, kIntraThreads);
                if (it == 0) mbar_arrive(cx.bars + B_T_FULL);
                // W^T -> shared memory (MN-major B operand of -S W^T), after Delta(n-1) read the old one
                if (!(ok = wait_bar(cx, B_WU_FULL, n & 1))) break;
                if (n >= 1 && !(ok = wait_bar(cx, B_DELTA_FULL + ((n - 1) & 1), ((n - 1) >> 1) & 1))) break;
                tc_fence_after();
                {
                    const size_t dump = (static_cast<size_t>(info.flat0 + c) * H + info.h) * kChunk * kHead;
                    const int i0 = 32 * hh;
                    uint32_t rr[32];
                    tmem_ld32_wait(tm_lane + kTmW + i0, rr);
                    float w[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) w[j] = __uint_as_float(rr[j]);
#pragma unroll
                    for (int q = 0; q < 4; ++q) st_chunk_bf16(sm + kWb, r, (i0 >> 3) + q, w + 8 * q);
                    if (p.intra_w) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) p.intra_w[dump + static_cast<size_t>(i0 + j) * kHead + r] = w[j];
                    }
                    if (p.intra_u) {
                        tmem_ld32_wait(tm_lane + kTmDelta + s * 64 + i0, rr);
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            p.intra_u[dump + static_cast<size_t>(i0 + j) * kHead + r] = __uint_as_float(rr[j]);
                    }
                    if (p.intra_g && it < 64)
                        p.intra_g[(static_cast<size_t>(info.flat0 + c) * H + info.h) * kChunk + it] = gb[kGG + it];
                }
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar_sync(kBarIntra, kIntraThreads);
                if (it == 0) mbar_arrive(cx.bars + B_WB_FULL + s);
            }
        }
    } else {
        // ================= state warpgroups (two; each TMEM lane row split in column halves) =================
        if (kRegsState > kRegsLaunch) regs_inc<kRegsState>();
        const int st = tid - 384;                      // 0..255
        const int wq = warp & 3;
        const int hh = (warp - 12) >> 2;               // column half
        const int v = wq * 32 + lane;                  // TMEM lane = state row v
        const uint32_t tm_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        uint8_t* sb = sm + kSb;
        __nv_bfloat16* outT = reinterpret_cast<__nv_bfloat16*>(sm + kOutT);
        uint32_t n = 0, u = 0;
        bool ok = true;
        for (; ok;) {
            const int slot = u & 1;
            if (!(ok = wait_bar(cx, B_UNIT_FULL + slot, (u >> 1) & 1))) break;
            const UnitInfo info = read_unit(sm, slot);
            named_bar_sync(kBarState, kStateThreads);
            if (st == 0) mbar_arrive(cx.bars + B_UNIT_EMPTY + slot);
            ++u;
            if (!info.valid) break;
            const size_t state_off = (static_cast<size_t>(info.srow) * H + info.h) * kHead * kHead +
                                     static_cast<size_t>(v) * kHead + 64 * hh;  // this thread's 64 columns
            const float* s0 = p.initial_state ? p.initial_state + state_off : nullptr;
            if (info.nC == 0) {
                if (p.output_state) {
                    float* dst = p.output_state + state_off;
#pragma unroll 4
                    for (int c0 = 0; c0 < 64; c0 += 4)
                        *reinterpret_cast<float4*>(dst + c0) =
                            s0 ? *reinterpret_cast<const float4*>(s0 + c0) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                continue;
            }
            // initial state: S0 -> Sb (bf16) and gamma_63(first chunk) * S0 -> TMEM
            {
                if (!(ok = wait_bar(cx, B_GATES_FULL + (n & 1), (n >> 1) & 1))) break;
                const float g63 = reinterpret_cast<const float*>(sm + kGbuf)[(n & 1) * kGFloats + kGGam + 63];
#pragma unroll 1
                for (int c0 = 0; c0 < 64; c0 += 32) {
                    float x[32];
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        const float4 f = s0 ? *reinterpret_cast<const float4*>(s0 + c0 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
                        x[j] = f.x; x[j + 1] = f.y; x[j + 2] = f.z; x[j + 3] = f.w;
                    }
                    uint8_t* half = sb + hh * 16384;
#pragma unroll
                    for (int q = 0; q < 4; ++q) st_chunk_bf16(half, v, (c0 >> 3) + q, x + 8 * q);
                    uint32_t r[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(x[j] * g63);
                    tmem_st32(tm_lane + kTmS + 64 * hh + c0, r);
                }
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar_sync(kBarState, kStateThreads);
                if (st == 0) mbar_arrive(cx.bars + B_SB_FULL + (n & 1));
            }
            for (int32_t c = 0; c < info.nC && ok; ++c, ++n) {
                const int s = n & 1;
                const uint32_t ph = (n >> 1) & 1;
                const int64_t tc = info.t0 + static_cast<int64_t>(c) * kChunk;
                const int64_t rem = info.L - static_cast<int64_t>(c) * kChunk;
                const int32_t Lc = rem < kChunk ? static_cast<int32_t>(rem) : kChunk;
                const float* gb = reinterpret_cast<const float*>(sm + kGbuf) + s * kGFloats;
                const uint32_t dbuf = tm_lane + kTmDelta + s * 64;
                // ---- Delta epilogue: this thread's 32 columns j in [32 hh, 32 hh + 32) go back into TMEM as
                //      16 packed bf16 Delta words followed by 16 packed decayed words (A operands of O2 and S)
                if (!(ok = wait_bar(cx, B_DELTA_FULL + s, ph))) break;
                if (!(ok = wait_bar(cx, B_WB_FULL + s, ph))) break;  // key-norm factors of chunk n are final
                tc_fence_after();
                {
                    uint32_t ra[32], pk[16];
                    tmem_ld32_wait(dbuf + 32 * hh, ra);
#pragma unroll
                    for (int q = 0; q < 16; ++q) pk[q] = pack_bf16x2(__uint_as_float(ra[2 * q]), __uint_as_float(ra[2 * q + 1]));
                    tmem_st16(dbuf + 32 * hh, pk);
                    float dv[16];
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        lds16(gb + kGDec + 32 * hh + 16 * part, dv);
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            pk[8 * part + q] = pack_bf16x2(__uint_as_float(ra[16 * part + 2 * q]) * dv[2 * q],
                                                           __uint_as_float(ra[16 * part + 2 * q + 1]) * dv[2 * q + 1]);
                    }
                    tmem_st16(dbuf + 32 * hh + 16, pk);
                    tmem_wait_st();
                }
                tc_fence_before();
                named_bar_sync(kBarState, kStateThreads);
                if (st == 0) mbar_arrive(cx.bars + B_DD_FULL + s);
                // ---- state epilogue: checkpoint / final state, next S operand, prescale (this thread's 64 columns)
                if (!(ok = wait_bar(cx, B_S_FULL + s, ph))) break;
                tc_fence_after();
                const bool last = (c + 1 == info.nC);
                float gnext = 1.f;
                if (!last) {
                    if (!(ok = wait_bar(cx, B_GATES_FULL + ((n + 1) & 1), ((n + 1) >> 1) & 1))) break;
                    gnext = reinterpret_cast<const float*>(sm + kGbuf)[((n + 1) & 1) * kGFloats + kGGam + 63];
                }
                {
                    const int64_t pend = static_cast<int64_t>(c + 1) * kChunk;
                    float* ck = nullptr;
                    if (p.checkpoints && p.ckpt_n > 0 && pend % p.ckpt_n == 0 && pend <= info.L)
                        ck = p.checkpoints + (static_cast<size_t>(info.ckpt_base + pend / p.ckpt_n - 1) * H + info.h) *
                                                 kHead * kHead + static_cast<size_t>(v) * kHead + 64 * hh;
                    float* fin = (last && p.output_state) ? p.output_state + state_off : nullptr;
#pragma unroll 1
                    for (int c0 = 0; c0 < 64; c0 += 16) {
                        uint32_t r[16];
                        tmem_ld16_wait(tm_lane + kTmS + 64 * hh + c0, r);
                        float x[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) x[j] = __uint_as_float(r[j]);
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
                        if (!last) {
                            uint8_t* half = sb + hh * 16384;
                            st_chunk_bf16(half, v, c0 >> 3, x);
                            st_chunk_bf16(half, v, (c0 >> 3) + 1, x + 8);
#pragma unroll
                            for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(x[j] * gnext);
                            tmem_st16(tm_lane + kTmS + 64 * hh + c0, r);
                        }
                    }
                    if (!last) tmem_wait_st();
                }
                if (st == 0) bulk_wait_group_read0();  // the previous chunk's output store has read outT
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar_sync(kBarState, kStateThreads);
                if (st == 0 && !last) mbar_arrive(cx.bars + B_SB_FULL + ((n + 1) & 1));
                // ---- output epilogue: o_i = orow_i (S Q^T)_i + scale (Delta^T P^T)_i, tokens i in [32 hh, 32 hh + 32)
                {
                    const float sc = p.scale;
                    uint32_t r1[32], r2[32];
                    tmem_ld32_wait(tm_lane + kTmO1 + 32 * hh, r1);
                    tmem_ld32_wait(tm_lane + kTmO2 + 32 * hh, r2);
                    float orow[16];
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        lds16(gb + kGOr + 32 * hh + 16 * part, orow);
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int jj = 16 * part + j;
                            const float o = orow[j] * __uint_as_float(r1[jj]) + sc * __uint_as_float(r2[jj]);
                            outT[(32 * hh + jj) * kHead + v] = __float2bfloat16_rn(o);
                        }
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar_sync(kBarState, kStateThreads);
                if (st == 0) {
                    mbar_arrive(cx.bars + B_O_EMPTY + s);
                    mbar_arrive(cx.bars + B_GATES_EMPTY + s);
                }
                if (Lc == kChunk) {
                    // a full chunk: one TMA store of the 64 x 128 tile (rows all belong to this sequence)
                    if (st == 0) {
                        tma_store_3d(&tm_o, sm + kOutT, 0, info.h, static_cast<int32_t>(tc));
                        bulk_commit_group();
                    }
                } else {
                    // the tail: coalesced copy of the valid rows only, 16 threads per 256-byte row
                    uint8_t* gout = static_cast<uint8_t*>(p.output);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int id = st + 256 * k, row = id >> 4, col = id & 15;
                        if (row < Lc) {
                            const uint4 val = *reinterpret_cast<const uint4*>(sm + kOutT + row * 256 + col * 16);
                            *reinterpret_cast<uint4*>(gout + ((static_cast<size_t>(tc + row) * H + info.h) * kHead) * 2 +
                                                      col * 16) = val;
                        }
                    }
                }
            }
        }
    }

    // ---- teardown
    if (tid == 384) bulk_wait_group0();  // output stores in flight have landed
    tc_fence_before();
    __syncthreads();
    if (warp == 3) tmem_dealloc(tmem, kTmCols);
}

}  // namespace

size_t chunk_bf16_smem_bytes() { return kSmemAlloc; }

cudaError_t launch_chunk_bf16(const ChunkParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                              const CUtensorMap& tm_v, const CUtensorMap& tm_o, int grid, cudaStream_t stream) {
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
    gdn_chunk_bf16_kernel<<<grid, kThreads, kSmemAlloc, stream>>>(p, tm_q, tm_k, tm_v, tm_o);
    return cudaGetLastError();
}

}  // namespace gdn
