// gdn_chunk_bf16.cu -- chunked Gated DeltaNet prefill, bf16 (or fp16) q/k/v,
// fp32 state, on sm_103a: tcgen05 tensor cores with TMEM accumulators,
// TMA-fed operands, warp-specialised and pipelined across chunks.  The two
// input types share one kernel template (gdn_chunk_kernel<__nv_bfloat16> and
// gdn_chunk_kernel<__half>): every 16-bit operand the kernel writes itself (P,
// T'', the TMEM copy of S, Delta) takes the input type, because A and B of one
// tcgen05 kind::f16 product have the same type.
//
// Per chunk of C = 64 tokens (G_r = sum_{m<=r} log alpha_m inside the chunk,
// gamma_r = e^{G_r}; n_j, m_i = 1/|k_j|, 1/|q_i| when the L2 norm is on, else
// 1; K and Q are the tiles as stored, not normalised):
//
//   intra-chunk step ("GDN 与 Chunked Prefill": cumsum, triangular solve,
//   recompute; the 4-token expansion table generalised to a 64 x 64 table):
//     D1 = [K; Q] K^T                               tcgen05, M=128 N=64 K=128
//     A~_ij = beta_i n_i^2 e^{G_i-G_j} (k_i.k_j), j < i      (n_i from diag D1)
//     P_ij = e^{G_i-G_j} (q_i.k_j),                j <= i
//     T~ = (I + A~)^-1                              blocked substitution + tf32 mma.sync
//     T' = T~ diag(beta gamma n^2) (fp32),  T'' = T~ diag(beta n) (16-bit)
//     U~^T = V^T T''^T                              tcgen05, into the Delta slot
//   state pass ("块内 state 和块间 final state": only the chunk's last state
//   crosses the boundary):
//     [X | O] = S [K; Q']^T                         tcgen05, one N = 128 product, A (16-bit S) from TMEM
//     Delta~^T = U~^T - X T'^T                      tcgen05 kind::tf32, A = X (fp32) from TMEM, negated
//     S <- gamma_63 S + (Delta~^T diag(e^{G_63-G_j})) K          tcgen05, in TMEM
//   (S W~^T with W~^T = K^T T'^T is computed as X T'^T: no W~ tile exists.)
//   output ("GDN与线性注意力GPU并行实现" section 3.3: O_init = Q S plus a
//   triangular-masked product):
//     O^T = scale (S Q'^T + Delta~^T P^T) diag(m),  Q' = diag(gamma) Q     tcgen05, one accumulator
//   A chunk whose G stays within [-8, 8] keeps Q as stored and folds gamma
//   into the other factors instead: P' = diag(1/gamma) P and m' = gamma m,
//   O^T = scale (S Q^T + Delta~^T P'^T) diag(m') -- the same product without
//   the pass that rescales Q in shared memory; the bound keeps the
//   accumulator's terms within e^8 of one another.
//
// The L2 norm of q and k ("FlashInfer GDN Prefill 完全指南", API table) enters
// only through the factors n and m, in fp32: the same values as normalising
// the rows first, without re-rounding them to bf16.  With the normalised
// matrix A = diag(beta n) M diag(n) (M_ij = e^{G_i-G_j} k_i.k_j), the
// similarity diag(n) (I + A) diag(n)^-1 = I + A~ gives T = diag(1/n) T~ diag(n);
// so U~ = diag(n) U, Delta~ = diag(n) Delta, and n cancels from the state
// update and from P: every norm factor is a row factor of the matrix that uses
// it, known to the thread that holds that row.
//
// Roles (640 threads in five warpgroups, one work unit = (sequence, state
// head) at a time, units taken longest first from an atomic counter):
//   warp 0       TMA: K, Q tiles (3 stages) and V tile; unit scheduler
//   warp 1       tcgen05 issue for the intra-chunk products (D1, U)
//   warp 2       tcgen05 issue for the state chain (X | O, Delta, Delta P^T, S)
//   warp 3       TMEM allocation; gates: G, gamma, beta, the per-row /
//                per-column factor vectors and the q norms
//   warps 4-11   two intra warpgroups (TMEM lane quarter x column half):
//                A and P, Q' = diag(gamma) Q where needed, T in place
//                with T' and T'', one chunk ahead of the state warpgroups
//   warps 12-19  two state warpgroups (lane quarter x column half): Delta
//                epilogue, state epilogue (next 16-bit S operand in TMEM,
//                checkpoints, final state, prescale), output epilogue;
//                checkpoints and final states leave through the output
//                tile's buffer, so that their stores are coalesced
// Every wait is bounded; a timeout sets GDN_DEVICE_ERR_TIMEOUT, raises a
// shared abort flag that every other wait polls, drains the CTA's in-flight
// copies and tensor-core work, frees TMEM and returns.  The intra and state
// warpgroups carry each wait's outcome to their next named barrier, which ANDs
// it over the group (bar.red.and), and leave their loops only there.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <type_traits>

#include "gdn_internal.cuh"
#include "sm103_ptx.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 640;
constexpr int kStateThreads = 256;  // two state warpgroups
constexpr int kIntraThreads = 256;  // two intra warpgroups
constexpr uint32_t kBarIntra = 1, kBarState = 2;  // named barrier ids
constexpr uint32_t kBarInverse = 3;               // the first four intra warps, inside the inverse

// ---- shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t kKQ = 0;           // 3 stages x 32 KB: K_h0 | Q_h0 | K_h1 | Q_h1 (64 rows x 128 B each)
constexpr uint32_t kKQStage = 32768;
constexpr uint32_t kKQStages = 3;
constexpr uint32_t kV = 98304;        // V_h0 | V_h1
constexpr uint32_t kTp = 114688;      // T' = T diag(cw) fp32 [64 i][64 j] K-major (halves of 32 j, 8 KB), n % 2 == 0
constexpr uint32_t kTpp = 131072;     // T'' = T diag(bn) bf16 [64 i][64 j] K-major
constexpr uint32_t kPb = 139264;      // 2 x P bf16 [64 i][64 j] K-major
constexpr uint32_t kTp1 = 155648;     // T' of chunks n % 2 == 1
constexpr uint32_t kAbuf = 172032;    // A, then T in place: fp32 [64][kLd]
constexpr uint32_t kXs = 189440;      // inverse scratch: [2][16][24] then [32][40] fp32
constexpr uint32_t kBars = 197632;    // up to 64 mbarriers
constexpr uint32_t kRing = 198144;    // 2 unit descriptors
constexpr uint32_t kMisc = 198272;    // tmem base, abort flag
constexpr uint32_t kGbuf = 198336;    // 3 x kGFloats floats of per-row / per-column factors (see kG*)
constexpr int kLd = 68;               // fp32 row stride of A and T (bank-conflict free rows)

// gbuf field offsets (floats), one 64-vector each, per chunk (n, m = 1/|k|, 1/|q| under the L2 norm, else 1).
// The gates warp writes them with n = m = 1; under the L2 norm the intra warps that hold the K K^T diagonal
// put n into rn, cw and bn (before the inverse reads them), and the gates warp later puts m into rm (RM_FULL):
//   G      running sum of log alpha            gamma  e^G
//   beta   beta (0 on padded rows)             rn     n_j (0 on padded rows under the norm)
//   rm     output row factor m_i, times gamma_i when Q is kept as stored (0 on padded rows under the norm)
//   cw     beta_j gamma_j n_j^2 (T' columns)   bn     beta_j n_j (T'' columns)
//   dec    e^{G_63 - G_j} (decayed Delta)      ra     A row factor beta_i n_i^2 e^{G_i - Gref}
//   rp     P row factor e^{G_i - Gref}, over gamma_i when Q is kept as stored
//   colf   e^{Gref - G_j}, Gref = (G_0 + G_63) / 2, so that e^{G_i - G_j} = (row factor) (colf) while the
//          chunk's G range is below kSafeRange
//   safe   1 when it is; else A and P take e^{G_i - G_j} pairwise
//   keepq  1 when every G_i of the chunk lies in [-8, 8]: Q stays as stored (no Q' pass)
constexpr int kGG = 0, kGGam = 64, kGBeta = 128, kGRn = 192, kGRm = 256, kGCw = 320, kGDec = 384, kGRp = 448,
              kGRa = 512, kGColf = 576, kGBn = 640, kGSafe = 704, kGKeepQ = 705, kGFloats = 720;
constexpr float kSafeRange = 80.f;  // e^{+-40} factors stay well inside fp32
constexpr float kKeepQRange = 8.f;  // bf16 only: fp16 would overflow on e^8 (q.k) with raw q and k
constexpr uint32_t kOutT = 207872;    // output tile: two halves [64 i][64 v] 16-bit, 128-byte swizzle
constexpr uint32_t kSmemBytes = kOutT + 16384;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;
static_assert(kGbuf >= kMisc + 64 && kXs + 4 * (2 * 16 * 24 + 32 * 40) <= kBars && kAbuf + 4 * 64 * kLd <= kXs,
              "shared memory map overlaps");
static_assert(kKQ + kKQStages * kKQStage == kV && kV + 16384 == kTp && kTp + 16384 == kTpp && kTpp + 8192 == kPb &&
                  kPb + 16384 == kTp1 && kTp1 + 16384 == kAbuf,
              "tile block overlap");
static_assert(kSmemAlloc <= 232448, "shared memory above the per-CTA limit");

// ---- barriers (single ones are safe where no waiter can fall two phases behind; see the roles)
enum {
    B_KQ_FULL = 0 /* 3 */, B_KQ_EMPTY = 3 /* 3 */, B_V_FULL = 6, B_V_EMPTY = 7, B_D1_FULL = 8, B_D1_EMPTY = 9,
    B_T_FULL = 10 /* 2 */, B_U_FULL = 12 /* 2 */, B_SB_FULL = 14 /* 2 */, B_DELTA_FULL = 16 /* 2 */,
    B_DD_FULL = 18 /* 2 */, B_S_FULL = 20 /* 2 */, B_O_EMPTY = 22 /* 2 */, B_GATES_FULL = 24 /* 3 */,
    B_GATES_EMPTY = 27 /* 3 */, B_UNIT_FULL = 30 /* 2 */, B_UNIT_EMPTY = 32 /* 2 */, B_DRAIN_I = 34, B_DRAIN_S = 35,
    B_XO_FULL = 36, B_XB_FULL = 37, B_O_FULL = 38, B_Q_READY = 39 /* 2 */, B_RM_FULL = 41 /* 3 */, B_COUNT = 44
};

// ---- TMEM columns
// S fp32 | Delta 2 x 64 | X = S K^T (fp32, the tf32 A operand of the Delta product) | O (S Q'^T + Delta^T P^T) |
// D1 | S as packed bf16 pairs (A operand of the X | O product)
constexpr uint32_t kTmS = 0, kTmDelta = 128, kTmX = 256, kTmO = 320, kTmD1 = 384, kTmSbf = 448;
constexpr uint32_t kTmCols = 512;
static_assert(kTmO == kTmX + 64, "X and O are one N = 128 accumulator");

template <bool kF16> constexpr uint32_t kIdescD1 = idesc_16bit_f32(128, 64, false, false, false, kF16);
template <bool kF16> constexpr uint32_t kIdescU = idesc_16bit_f32(128, 64, true, false, false, kF16);
template <bool kF16> constexpr uint32_t kIdescXO = idesc_16bit_f32(128, 128, false, false, false, kF16);
template <bool kF16> constexpr uint32_t kIdescX = idesc_16bit_f32(128, 64, false, false, false, kF16);
constexpr uint32_t kIdescDelta = idesc_tf32_f32(128, 64, true);  // X (fp32 in TMEM) times T' (fp32), negated
template <bool kF16> constexpr uint32_t kIdescO = idesc_16bit_f32(128, 64, false, false, false, kF16);
template <bool kF16> constexpr uint32_t kIdescS = idesc_16bit_f32(128, 128, false, true, false, kF16);

// The 16-bit element: bf16, or fp16 for fp16 inputs.
template <bool kF16>
struct Elem16;
template <>
struct Elem16<false> {
    using T = __nv_bfloat16;
    static __device__ __forceinline__ T from(float x) { return __float2bfloat16_rn(x); }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) { return pack_bf16x2(lo, hi); }
    static __device__ __forceinline__ float2 unpack(uint32_t w) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
};
template <>
struct Elem16<true> {
    using T = __half;
    static __device__ __forceinline__ T from(float x) { return __float2half_rn(x); }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) { return pack_f16x2(lo, hi); }
    static __device__ __forceinline__ float2 unpack(uint32_t w) {
        __half2 h;
        memcpy(&h, &w, 4);
        return __half22float2(h);
    }
};

constexpr long long kWaitCycles = 2000000000LL;  // about one second

struct UnitInfo {
    int32_t valid, seq, h, nC;  // valid: 0 = no more units, 1 = a unit, 2 = a transfer-matrix unit (identity, U = 0),
                                // 3 = a unit on the caller's own state (segment pass of context parallelism)
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
__device__ __forceinline__ bool wait_loop(const Ctx& cx, int b, uint32_t parity) {
    uint64_t* bar = cx.bars + b;
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

// Every role shares one out-of-line copy of the sleeping loop: the many wait
// sites stay small, which keeps the per-chunk code of all twenty warps
// resident in the instruction cache.
__device__ __noinline__ bool wait_bar_slow(const Ctx& cx, int b, uint32_t parity) { return wait_loop(cx, b, parity); }

__device__ __forceinline__ bool wait_bar(const Ctx& cx, int b, uint32_t parity) {
    if (mbar_try_wait(cx.bars + b, parity)) return true;
    return wait_bar_slow(cx, b, parity);
}

// The single-warp roles' slow path: the same bounded loop with a 100 ns suspend hint (measured a little
// faster for the issuers and the producer than the warpgroups' 2 us).
__device__ __noinline__ bool wait_bar_warp_slow(const Ctx& cx, int b, uint32_t parity) {
    uint64_t* bar = cx.bars + b;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 100)) return true;
        if (*cx.abort) return false;
        if (clock64() - t0 > kWaitCycles) {
            atomicOr(cx.status, static_cast<int32_t>(GDN_DEVICE_ERR_TIMEOUT));
            *cx.abort = 1;
            return false;
        }
    }
}

// A wait whose outcome is the same for every lane of a converged warp (the
// single-warp roles use elect.sync and full-mask shuffles after their waits).
__device__ __forceinline__ bool wait_bar_warp(const Ctx& cx, int b, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_try_wait(cx.bars + b, parity) || wait_bar_warp_slow(cx, b, parity));
}

// Bounded wait used while draining (ignores the abort flag).
__device__ __forceinline__ void drain_bar(const Ctx& cx, int b, uint32_t parity) {
    if (!mbar_wait(cx.bars + b, parity, kWaitCycles)) atomicOr(cx.status, static_cast<int32_t>(GDN_DEVICE_ERR_TIMEOUT));
}

template <bool kF16>
__device__ __forceinline__ void st_chunk16(uint8_t* tile, uint32_t row, uint32_t chunk, const float* x) {
    uint4 v;
    v.x = Elem16<kF16>::pack(x[0], x[1]);
    v.y = Elem16<kF16>::pack(x[2], x[3]);
    v.z = Elem16<kF16>::pack(x[4], x[5]);
    v.w = Elem16<kF16>::pack(x[6], x[7]);
    *reinterpret_cast<uint4*>(tile + sw128_offset(row, chunk)) = v;
}

template <bool kF16>
__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 t = Elem16<kF16>::unpack(w[j]);
        f[2 * j] = t.x;
        f[2 * j + 1] = t.y;
    }
}

__device__ __forceinline__ UnitInfo read_unit(const uint8_t* sm, int slot) {
    return *reinterpret_cast<const UnitInfo*>(sm + kRing + slot * 64);
}

// ===========================================================================
// Triangular inverse T = (I + A)^-1 of a strictly lower 64 x 64 A (fp32, rows
// of kLd floats), computed in place by the two intra warpgroups (256 threads),
// followed by the operands of the Delta and U products, T' = T diag(cw) in
// fp32 (tf32 operand) and T'' = T diag(bn) in the 16-bit type (K-major
// [64 i][64 j], 128-byte swizzle; their blocks above the diagonal are never
// written and stay zero).
//   stage 1 (warps 0, 1; warp w owns rows and columns 32w..32w+31): the two
//     16 x 16 diagonal blocks by forward substitution, one column per lane,
//     then the block under them, T_10 = -T_11 (A_10 T_00), and a zeroed block
//     above them, with no block-wide barrier;
//   stage 2 (all eight warps): T_21 = -T_22 (A_21 T_11) on the 32 x 32 halves;
//     its tiles go from the MMA fragments straight into T' and T'', while the
//     two diagonal 32 x 32 blocks are converted from shared memory.
// The 16- and 32-row products are below the 64-row minimum of tcgen05.mma, so
// they run as warp-level m16n8k8 tf32 MMAs (fp32 accumulate); T feeds the
// Delta and U products as tf32 and 16-bit operands anyway.
// ===========================================================================

// D (16 x 8) += A (16 x 8, row-major, stride lda) * B (8 x 8, row-major K x N, stride ldb).  The operands
// go to the tensor core as fp32 bits, which it reads as tf32 (the low mantissa bits dropped): a conversion
// with rounding per fragment element cost more time than the bit it saves (T is rounded to tf32 and bf16
// for the Delta and U products anyway).  A comes in with one ldmatrix (rows 16-byte aligned).
__device__ __forceinline__ void mma_tf32_16x8x8(float (&d)[4], const float* A, int lda, const float* B, int ldb,
                                                int lane) {
    const int g = lane >> 2, t = lane & 3;
    uint32_t a0, a1, a2, a3;  // ldmatrix: row (lane & 15), columns 4 (lane >> 4) .. + 3 of the 16 x 8 tile
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                 : "r"(smem_u32(A + (lane & 15) * lda + (lane >> 4) * 4)));
    const uint32_t b0 = __float_as_uint(B[t * ldb + g]), b1 = __float_as_uint(B[(t + 4) * ldb + g]);
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

// Two adjacent 16-bit values (row i, columns j, j + 1; j even) of a swizzled K-major [64][64] tile.
template <bool kF16>
__device__ __forceinline__ void st_pair16(uint8_t* tile, int i, int j, float x0, float x1) {
    *reinterpret_cast<uint32_t*>(tile + i * 128 + (((j >> 3) ^ (i & 7)) << 4) + (j & 7) * 2) =
        Elem16<kF16>::pack(x0, x1);
}

// fp32 elements of a swizzled K-major [64][64] tile stored as two halves of 32 columns (8 KB each, rows of
// 128 bytes): eight columns j0 .. j0 + 7 (j0 a multiple of 8) of row i, and two columns j, j + 1 (j even).
__device__ __forceinline__ void st_f32x8(uint8_t* tile, int i, int j0, const float* x) {
    uint8_t* half = tile + (j0 >> 5) * 8192;
    const uint32_t c = (j0 & 31) >> 2;
    *reinterpret_cast<float4*>(half + sw128_offset(i, c)) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4*>(half + sw128_offset(i, c + 1)) = make_float4(x[4], x[5], x[6], x[7]);
}

__device__ __forceinline__ void st_f32x2(uint8_t* tile, int i, int j, float x0, float x1) {
    *reinterpret_cast<float2*>(tile + (j >> 5) * 8192 + sw128_offset(i, (j & 31) >> 2) + (j & 3) * 4) =
        make_float2(x0, x1);
}

// Columns c0 .. c0 + 15 of this warp's 32 state rows (row = lane, values r) to a checkpoint or an output state,
// staged through the warp's 2 KB slice of shared memory: written row by row (float4 j of row i at slot
// j ^ ((i >> 1) & 3), so that neither the writes nor the reads meet a bank conflict) and read back with four lanes
// per row, so that each store instruction covers 64 contiguous bytes of eight rows.  Stored straight from the
// registers, each instruction would touch 32 rows a full row apart.  warp_off is the element offset of the warp's
// row 0 at column 0 of its half, ld the element stride between rows.  kStoreUnroll unrolls the store loop (four
// instructions of eight rows): fully on the per-chunk path, not at all on the once-per-unit one (whose registers
// the caller pays for across the call).
template <int kStoreUnroll>
__device__ __forceinline__ void stage_rows16(const uint32_t (&r)[16], float* slice, void* dst, int64_t warp_off,
                                             int64_t ld, int c0, int32_t dt, int lane) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
        *reinterpret_cast<float4*>(slice + lane * 16 + 4 * (j ^ ((lane >> 1) & 3))) =
            make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]), __uint_as_float(r[4 * j + 2]),
                        __uint_as_float(r[4 * j + 3]));
    __syncwarp();
#pragma unroll kStoreUnroll
    for (int q = 0; q < 4; ++q) {
        const int i = 8 * q + (lane >> 2), j = lane & 3;
        const float4 f4 = *reinterpret_cast<const float4*>(slice + i * 16 + 4 * (j ^ ((i >> 1) & 3)));
        const float f[4] = {f4.x, f4.y, f4.z, f4.w};
        state_store4(dst, warp_off + static_cast<int64_t>(i) * ld + c0 + 4 * j, dt, f);
    }
    __syncwarp();
}

constexpr int kLdX1 = 24, kLdX2 = 40;  // scratch strides: conflict-free B-fragment reads

template <bool kF16>
__device__ __forceinline__ void tri_inverse_64(float* __restrict__ A, uint8_t* __restrict__ tp,
                                               uint8_t* __restrict__ tpp, const float* __restrict__ cw,
                                               const float* __restrict__ bn, float* __restrict__ X1,
                                               float* __restrict__ X2, int t) {
    const int wi = t >> 5, lane = t & 31;  // warp index 0..7 within the intra groups
    if (wi < 2) {
        // ---- stage 1: diagonal 16 x 16 blocks, one column per lane
        const int o = (wi * 2 + (lane >> 4)) * 16, col = lane & 15;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const float* arow = A + (o + r) * kLd + o;
            float acc0 = (r == col) ? 1.f : 0.f, acc1 = 0.f;
#pragma unroll
            for (int m = 0; m + 3 < r; m += 4) {
                const float4 a4 = *reinterpret_cast<const float4*>(arow + m);
                acc0 -= a4.x * x[m];
                acc1 -= a4.y * x[m + 1];
                acc0 -= a4.z * x[m + 2];
                acc1 -= a4.w * x[m + 3];
            }
#pragma unroll
            for (int m = r & ~3; m < r; ++m) acc0 -= arow[m] * x[m];
            x[r] = (r < col) ? 0.f : acc0 + acc1;
        }
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 16; ++r) A[(o + r) * kLd + o + col] = x[r];
        {   // the block above the pair is zero: rows 32w..32w+15, columns 32w+16..32w+31
            float* z = A + (32 * wi + (lane >> 1)) * kLd + 32 * wi + 16 + (lane & 1) * 8;
            *reinterpret_cast<float4*>(z) = make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(z + 4) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    if (wi < 4) {
        // ---- T_10 = -T_11 (A_10 T_00) of the two 32 x 32 blocks: warp wi takes block wi / 2, output columns
        //      8 (wi % 2) .. + 7, so the four warps run the products side by side
        named_bar_sync(kBarInverse, 128);  // the diagonal blocks are in place
        const int b0 = 32 * (wi >> 1), b1 = b0 + 16, nt = (wi & 1) * 8;
        float* xs = X1 + (wi >> 1) * 16 * kLdX1;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k0 = 0; k0 < 16; k0 += 8)
            mma_tf32_16x8x8(d, A + b1 * kLd + b0 + k0, kLd, A + (b0 + k0) * kLd + b0 + nt, kLd, lane);
        store_tile_16x8(xs + nt, kLdX1, d, 1.f, lane);
        named_bar_sync(kBarInverse, 128);  // every read of A_10 is done before T_10 replaces it
        float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k0 = 0; k0 < 16; k0 += 8)
            mma_tf32_16x8x8(e, A + b1 * kLd + b1 + k0, kLd, xs + k0 * kLdX1 + nt, kLdX1, lane);
        store_tile_16x8(A + b1 * kLd + b0 + nt, kLd, e, -1.f, lane);
    }
    named_bar_sync(kBarIntra, kIntraThreads);
    // ---- stage 2: X = A_21 T_11 (one 16 x 8 tile per warp) and the diagonal 32 x 32 blocks of T' and T''
    const int mt = (wi >> 2) * 16, nt = (wi & 3) * 8;
    {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k0 = 0; k0 < 32; k0 += 8)
            mma_tf32_16x8x8(d, A + (32 + mt) * kLd + k0, kLd, A + k0 * kLd + nt, kLd, lane);
        store_tile_16x8(X2 + mt * kLdX2 + nt, kLdX2, d, 1.f, lane);
    }
    {
        const int blk = t >> 7, i = blk * 32 + ((t >> 2) & 31), j0 = blk * 32 + (t & 3) * 8;
        const float* trow = A + i * kLd + j0;
        const float4 t0 = *reinterpret_cast<const float4*>(trow);
        const float4 t1 = *reinterpret_cast<const float4*>(trow + 4);
        const float4 c0 = *reinterpret_cast<const float4*>(cw + j0);
        const float4 c1 = *reinterpret_cast<const float4*>(cw + j0 + 4);
        const float4 e0 = *reinterpret_cast<const float4*>(bn + j0);
        const float4 e1 = *reinterpret_cast<const float4*>(bn + j0 + 4);
        const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
        const float cv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        const float ev[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
        float x[8], y[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            x[q] = tv[q] * cv[q];
            y[q] = tv[q] * ev[q];
        }
        st_f32x8(tp, i, j0, x);
        st_chunk16<kF16>(tpp, i, j0 >> 3, y);
    }
    named_bar_sync(kBarIntra, kIntraThreads);
    // ---- T_21 = -T_22 X, written as T' and T'' tiles from the fragments
    {
        float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k0 = 0; k0 < 32; k0 += 8)
            mma_tf32_16x8x8(e, A + (32 + mt) * kLd + 32 + k0, kLd, X2 + k0 * kLdX2 + nt, kLdX2, lane);
        const int g = lane >> 2, j = nt + 2 * (lane & 3);
        const int i0 = 32 + mt + g, i1 = i0 + 8;
        const float be0 = bn[j], be1 = bn[j + 1], cw0 = cw[j], cw1 = cw[j + 1];
        st_f32x2(tp, i0, j, -e[0] * cw0, -e[1] * cw1);
        st_f32x2(tp, i1, j, -e[2] * cw0, -e[3] * cw1);
        st_pair16<kF16>(tpp, i0, j, -e[0] * be0, -e[1] * be1);
        st_pair16<kF16>(tpp, i1, j, -e[2] * be0, -e[3] * be1);
    }
}

// ===========================================================================
// Gates of one chunk (one warp; lane l owns rows 2l, 2l+1).  load_gates issues
// the global loads early (alpha = 1, beta = 0 on padded rows); compute_gates
// forms G = running sum of log alpha, gamma = e^G and the factor vectors.
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

// The vectors of one chunk (see kG*) with n = m = 1; under the L2 norm qk_norms then rewrites the
// norm-dependent ones.  Rows at or past Lc are padding (alpha = 1, beta = 0).
__device__ __forceinline__ void compute_gates(const GatePrefetch& g, float* gb, bool l2norm, float keep_range,
                                              int lane) {
    const int r0 = 2 * lane;
    const float la0 = __logf(g.a0), la1 = __logf(g.a1);
    float incl = la0 + la1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const float G1 = incl, G0 = incl - la1;
    const float G63 = __shfl_sync(0xffffffffu, incl, 31);
    const float Gfirst = __shfl_sync(0xffffffffu, G0, 0);
    const float Gref = 0.5f * (Gfirst + G63);
    float gmax = fmaxf(G0, G1), gmin = fminf(G0, G1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
        gmin = fminf(gmin, __shfl_xor_sync(0xffffffffu, gmin, o));
    }
    const bool keepq = gmax <= keep_range && gmin >= -keep_range;
    const float ekeep = __expf(-Gref);
    const float Gv[2] = {G0, G1}, bv[2] = {g.b0, g.b1};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int r = r0 + k;
        const float e = __expf(Gv[k]);
        const float rowf = __expf(Gv[k] - Gref);
        gb[kGG + r] = Gv[k];
        gb[kGGam + r] = e;
        gb[kGBeta + r] = bv[k];
        gb[kGRn + r] = 1.f;
        gb[kGCw + r] = bv[k] * e;
        gb[kGBn + r] = bv[k];
        gb[kGDec + r] = __expf(G63 - Gv[k]);
        if (!l2norm) gb[kGRm + r] = keepq ? e : 1.f;
        gb[kGRp + r] = keepq ? ekeep : rowf;  // e^{G_i - Gref} / gamma_i = e^{-Gref}
        gb[kGRa + r] = bv[k] * rowf;
        gb[kGColf + r] = __expf(Gref - Gv[k]);
    }
    if (lane == 0) {
        gb[kGSafe] = (gmax - gmin < kSafeRange) ? 1.f : 0.f;
        gb[kGKeepQ] = keepq ? 1.f : 0.f;
    }
}

// rm of the chunk's rows lane and lane + 32 under the L2 norm: 1/|q_i| from
// the Q tile as stored (K-major, 128B-swizzled halves), times gamma_i when the
// chunk keeps Q; 0 on padded rows.  Runs after compute_gates in the same warp
// (reads gamma and keepq back from its stores).  The two rows are summed side
// by side in eight partial sums each, so the dependent chains stay short.
template <bool kF16>
__device__ __forceinline__ void q_norms(const uint8_t* q0, float* gb, int32_t Lc, int lane) {
    const bool keepq = gb[kGKeepQ] != 0.f;
    float ss[2][8];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int j = 0; j < 8; ++j) ss[h][j] = 0.f;
#pragma unroll 2
    for (int cch = 0; cch < 16; ++cch) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float f[8];
            unpack8<kF16>(*reinterpret_cast<const uint4*>(q0 + (cch >> 3) * 16384 + sw128_offset(lane + 32 * h, cch & 7)),
                          f);
#pragma unroll
            for (int j = 0; j < 8; ++j) ss[h][j] = fmaf(f[j], f[j], ss[h][j]);
        }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int qr = lane + 32 * h;
        const float t = ((ss[h][0] + ss[h][1]) + (ss[h][2] + ss[h][3])) + ((ss[h][4] + ss[h][5]) + (ss[h][6] + ss[h][7]));
        const float rm = qr < Lc ? rsqrtf(t + 1e-6f) : 0.f;
        gb[kGRm + qr] = keepq ? rm * gb[kGGam + qr] : rm;
    }
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

// Intermediates for tests (only when requested): this thread's 32 values of W
// and U (row r = k or v, columns i0..i0+31) and G, in fp32.  U is read from
// its TMEM columns before the Delta product accumulates into them; W = T' K is
// not formed by the kernel (the state pass uses X = S K^T instead), so it is
// computed here on CUDA cores from the fp32 T' and the K tile the tensor cores
// read (fp32 sums).  Out of line, so the hot
// loop stays compact in the instruction cache.
template <bool kF16>
__device__ __noinline__ void dump_intra(float* intra_w, float* intra_u, float* intra_g, size_t dump, size_t gdump,
                                        const uint8_t* tp, const uint8_t* kt, uint32_t tm_u, int r, int i0, int it,
                                        const float* G) {
    uint32_t rr[32];
    tmem_ld32_wait(tm_u, rr);
    if (intra_u)
        for (int j = 0; j < 32; ++j) intra_u[dump + static_cast<size_t>(i0 + j) * kHead + r] = __uint_as_float(rr[j]);
    if (intra_w) {
        // K[j][r]: row j of the K tile, column r (halves of 64 columns, 128-byte swizzle)
        float kc[64];
        for (int j = 0; j < 64; ++j) {
            const uint8_t* row = kt + (r >> 6) * 16384;
            float f[8];
            unpack8<kF16>(*reinterpret_cast<const uint4*>(row + sw128_offset(j, (r & 63) >> 3)), f);
            kc[j] = f[r & 7];
        }
        for (int i = i0; i < i0 + 32; ++i) {  // T' row i: fp32, halves of 32 j, 128-byte swizzle
            float acc = 0.f;
            for (int j4 = 0; j4 < 16; ++j4) {
                const float4 t4 = *reinterpret_cast<const float4*>(tp + (j4 >> 3) * 8192 + sw128_offset(i, j4 & 7));
                acc += t4.x * kc[4 * j4] + t4.y * kc[4 * j4 + 1] + t4.z * kc[4 * j4 + 2] + t4.w * kc[4 * j4 + 3];
            }
            intra_w[dump + static_cast<size_t>(i) * kHead + r] = acc;
        }
    }
    if (intra_g && it < 64) intra_g[gdump + it] = G[it];
}

// Start of a unit's state: S0 (this thread's row v, 64 columns) as packed bf16
// pairs into the A operand columns, and gamma_63 S0 into the fp32 accumulator
// (S0 null: zeros).  Once per unit, so out of line.
template <bool kF16>
__device__ __noinline__ void load_initial_state(const void* s0, int64_t off, int32_t dt, uint32_t tm_sbf,
                                                uint32_t tm_s, float g63) {
    for (int c0 = 0; c0 < 64; c0 += 32) {
        float x[32];
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            float f[4] = {0.f, 0.f, 0.f, 0.f};
            if (s0) state_load4(s0, off + c0 + j, dt, f);
            x[j] = f[0]; x[j + 1] = f[1]; x[j + 2] = f[2]; x[j + 3] = f[3];
        }
        uint32_t pk[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) pk[q] = Elem16<kF16>::pack(x[2 * q], x[2 * q + 1]);
        tmem_st16(tm_sbf + c0 / 2, pk);
        uint32_t r[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(x[j] * g63);
        tmem_st32(tm_s + c0, r);
    }
    tmem_wait_st();
}

// A zero-length sequence: this thread's 64 elements of the initial state (or zeros) to the output state.
__device__ __noinline__ void pass_state_through(const void* s0, void* dst, int64_t off, int32_t dt) {
#pragma unroll 1
    for (int c0 = 0; c0 < 64; c0 += 4) {
        float f[4] = {0.f, 0.f, 0.f, 0.f};
        if (s0) state_load4(s0, off + c0, dt, f);
        state_store4(dst, off + c0, dt, f);
    }
}

// The transfer pass's identity start: this thread's 64 columns of row v of I (a 1 in column ic, when
// 0 <= ic < 64), into the bf16 operand and the accumulator (times g63), or straight to the output state
// for an empty segment (dst non-null).  Called by the transfer instance only.
template <bool kF16>
__device__ __noinline__ void identity_state(int ic, uint32_t tm_sbf, uint32_t tm_s, float g63, float* dst) {
    for (int c0 = 0; c0 < 64; c0 += 16) {
        float x[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = (c0 + j == ic) ? 1.f : 0.f;
        if (dst) {
#pragma unroll
            for (int j = 0; j < 16; j += 4)
                *reinterpret_cast<float4*>(dst + c0 + j) = make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
            continue;
        }
        uint32_t pk[8], r[16];
#pragma unroll
        for (int q = 0; q < 8; ++q) pk[q] = Elem16<kF16>::pack(x[2 * q], x[2 * q + 1]);
        tmem_st8(tm_sbf + c0 / 2, pk);
#pragma unroll
        for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(x[j] * g63);
        tmem_st16(tm_s + c0, r);
    }
    if (!dst) tmem_wait_st();
}

// The final state after a unit's last chunk, or its checkpoint: the warp's 32 rows of accumulator columns
// (tm_s: this thread's 64 columns) to `base` in type dt, this thread's row at element offset `off` and the rows
// ld elements apart, staged through the warp's slice of the output tile's buffer (free: the chunk's output
// store has read it).  Warp-uniform (tcgen05.ld is warp-collective).
__device__ __noinline__ void store_state_rows(uint32_t tm_s, void* base, int64_t off, int64_t ld, int32_t dt) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int lane = threadIdx.x & 31;
    float* slice = reinterpret_cast<float*>(sm + kOutT) + ((threadIdx.x >> 5) & 7) * 512;
    const int64_t warp_off = off - static_cast<int64_t>(lane) * ld;
#pragma unroll 1
    for (int c0 = 0; c0 < 64; c0 += 16) {
        uint32_t r[16];
        tmem_ld16_wait(tm_s + c0, r);
        stage_rows16<1>(r, slice, base, warp_off, ld, c0, dt, lane);
    }
}

// After a unit's last chunk: the checkpoint of that chunk end (ck_off >= 0) and the final state (dst non-null),
// from this thread's 64 accumulator columns.  One out-of-line call site in the state loop.
__device__ __noinline__ void finish_unit(uint32_t tm_s, void* ck, int64_t ck_off, int32_t ck_dt, void* dst,
                                         int64_t off, int64_t s_v, int32_t dt) {
    if (ck_off >= 0) store_state_rows(tm_s, ck, ck_off, kHead, ck_dt);
    if (dst) store_state_rows(tm_s, dst, off, s_v, dt);
}

// Cold paths of the per-chunk loops, out of line so that the code every chunk runs stays small in the
// instruction caches (every SM sub-partition runs intra, state and scheduler code at once).  The pairwise
// decay of A / P and the checkpoint rows of a unit's inner chunks stay inline: out of line (an array handed to
// the call, a second TMEM read) they cost registers and spills in the hot loops, and measured slower.

// Q' = diag(gamma) Q in place (a chunk that does not keep Q as stored): row it / 4, 32 values per thread.
template <bool kF16>
__device__ __noinline__ void scale_q_rows(uint8_t* kqs, int it, const float* gb) {
    const int qr = it >> 2, qq = it & 3;
    const float gam = gb[kGGam + qr];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int cch = 4 * qq + k;  // 16-byte column of the 256-byte row
        uint8_t* half = kqs + 8192 + (cch >> 3) * 16384;
        float f[8];
        unpack8<kF16>(*reinterpret_cast<const uint4*>(half + sw128_offset(qr, cch & 7)), f);
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] *= gam;
        st_chunk16<kF16>(half, qr, cch & 7, f);
    }
}

// The padded rows (>= Lc) of a tail chunk's K tile (threads 0..63) and V tile (64..127) are zeroed.
__device__ __noinline__ void zero_tail_rows(uint8_t* kqs, uint8_t* vt, int it, int Lc) {
    const int zr = it & 63;
    if (it < 128 && zr >= Lc) {
        const uint4 z = make_uint4(0, 0, 0, 0);
        uint8_t* base = (it < 64) ? kqs : vt;
        const uint32_t hs = (it < 64) ? 16384 : 8192;
#pragma unroll 1
        for (int cch = 0; cch < 16; ++cch)
            *reinterpret_cast<uint4*>(base + (cch >> 3) * hs + sw128_offset(zr, cch & 7)) = z;
    }
}

// The valid rows of a tail chunk's output tile (two swizzled halves of 64 v, as the TMA store reads them), by
// coalesced 16-byte stores (a full chunk goes by TMA).
__device__ __noinline__ void store_output_tail(const uint8_t* tile, uint8_t* gout, int st, int Lc, int64_t tc,
                                              int H, int h) {
#pragma unroll 1
    for (int k = 0; k < 4; ++k) {
        const int id = st + 256 * k, row = id >> 4, col = id & 15;  // col: 16-byte column (8 v) of the row
        if (row < Lc) {
            const uint4 val =
                *reinterpret_cast<const uint4*>(tile + (col >> 3) * 8192 + row * 128 + (((col & 7) ^ (row & 7)) << 4));
            *reinterpret_cast<uint4*>(gout + ((static_cast<size_t>(tc + row) * H + h) * kHead) * 2 + col * 16) = val;
        }
    }
}

// E16: the input element type, __nv_bfloat16 or __half.  kTransfer: the context-parallel transfer pass --
// units [0, N*H) run each sequence (a segment) from a zero state, units [N*H, 2*N*H) run it from the
// identity with U = 0 (the segment's transfer matrix), into output_state rows seq and N + seq; no output
// products, epilogue or stores.  kDump: the instance that also writes the intra-chunk intermediates (tests);
// the other instances carry no code for them.
template <typename E16, bool kTransfer, bool kDump>
__global__ void __launch_bounds__(kThreads, 1)
    gdn_chunk_kernel(const ChunkParams p, const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_o) {
    constexpr bool kF16 = std::is_same<E16, __half>::value;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    Ctx cx;
    cx.sm = sm;
    cx.bars = reinterpret_cast<uint64_t*>(sm + kBars);
    cx.abort = reinterpret_cast<volatile int32_t*>(sm + kMisc + 4);
    cx.status = p.status;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + kMisc);

    // Bad input flagged by the prepare kernel: every thread sees one copy of the word.  A run whose
    // device-side sequence count is zero (a transfer pass with no segments) has nothing to do either.  With a
    // programmatic launch the CTAs are resident while the prepare step finishes; griddep_wait orders every
    // read after it.
    griddep_wait();
    if (tid == 0)
        *cx.abort = *reinterpret_cast<volatile int32_t*>(p.status) != 0 || (p.num_seqs_dev && *p.num_seqs_dev <= 0);
    __syncthreads();
    if (*cx.abort != 0) return;
    __syncthreads();

    if (tid == 0) {
        for (int b = 0; b < B_COUNT; ++b) mbar_init(cx.bars + b, 1);
        mbar_init(cx.bars + B_UNIT_EMPTY + 0, 5);
        mbar_init(cx.bars + B_UNIT_EMPTY + 1, 5);
        for (int b = 0; b < 3; ++b) mbar_init(cx.bars + B_GATES_EMPTY + b, 8);  // one arrival per state warp
        fence_mbar_init();
        if (p.has_tokens) {
            prefetch_tensormap(&tm_q);
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
        }
    }
    for (uint32_t off = tid * 16; off < kAbuf - kTp; off += kThreads * 16)  // both T', T'' and both P buffers
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

    if (warp < 4) {
        // the scheduling warpgroup: TMA producer, two MMA issuers, gates warp
        if (warp == 0) {
            // ================= TMA producer and unit scheduler =================
            if (lane == 0) {
                const int64_t units1 = static_cast<int64_t>(p.num_seqs_dev ? *p.num_seqs_dev : p.num_seqs) * H;
                const int64_t units = kTransfer ? 2 * units1 : units1;
                uint32_t n = 0, u = 0;
                int64_t issued_kq[kKQStages] = {-1, -1, -1};
                int issued_v = -1;
                for (;;) {
                    const int64_t uid = atomicAdd(p.counter, 1);
                    const int slot = u & 1;
                    if (u >= 2 && !wait_bar(cx, B_UNIT_EMPTY + slot, ((u - 2) >> 1) & 1)) break;
                    UnitInfo info;
                    const bool second = kTransfer && uid >= units1;  // a transfer-matrix unit
                    info.valid = uid < units ? (second ? 2 : 1) : 0;
                    int32_t nC = 0;
                    if (info.valid) {
                        const int64_t ub = second ? uid - units1 : uid;
                        const int32_t seq = p.seq_order[ub / H];
                        const int32_t h = static_cast<int32_t>(ub % H);
                        info.seq = seq;
                        info.h = h;
                        if (kTransfer) {
                            info.t0 = p.seg[2 * seq];
                            info.L = p.seg[2 * seq + 1];
                        } else {
                            info.t0 = load_index(p.cu_seqlens, p.cu_i64, seq);
                            info.L = load_index(p.cu_seqlens, p.cu_i64, seq + 1) - info.t0;
                        }
                        nC = static_cast<int32_t>((info.L + kChunk - 1) / kChunk);
                        info.nC = nC;
                        info.qh = h / (H / p.hq);
                        info.kh = h / (H / p.hk);
                        info.vh = h / (H / p.hv);
                        info.flat0 = kTransfer ? 0 : p.chunk_offsets[seq];
                        info.srow = (p.state_indices ? load_index(p.state_indices, p.idx_i64, seq) : seq) +
                                    (second ? p.num_seqs : 0);
                        if (!kTransfer && p.split_state && info.srow < 0) {  // a row of the caller's own state
                            info.srow = -1 - info.srow;
                            info.valid = 3;
                        }
                        info.ckpt_base = p.ckpt_n > 0 ? load_index(p.ckpt_cu_starts, p.ckpt_i64, seq) : 0;
                    }
                    *reinterpret_cast<UnitInfo*>(sm + kRing + slot * 64) = info;
                    mbar_arrive(cx.bars + B_UNIT_FULL + slot);
                    ++u;
                    if (!info.valid) break;
                    bool ok = true;
                    for (int32_t c = 0; c < nC && ok; ++c, ++n) {
                        const uint32_t s = n % kKQStages;
                        const int32_t t = static_cast<int32_t>(info.t0 + static_cast<int64_t>(c) * kChunk);
                        if (n >= kKQStages && !(ok = wait_bar(cx, B_KQ_EMPTY + s, ((n - kKQStages) / kKQStages) & 1))) break;
                        uint8_t* st = sm + kKQ + s * kKQStage;
                        uint64_t* fb = cx.bars + B_KQ_FULL + s;
                        mbar_arrive_expect_tx(fb, kKQStage);
                        tma_load_3d(st + 0, &tm_k, fb, 0, info.kh, t);
                        tma_load_3d(st + 8192, &tm_q, fb, 0, info.qh, t);
                        tma_load_3d(st + 16384, &tm_k, fb, 64, info.kh, t);
                        tma_load_3d(st + 24576, &tm_q, fb, 64, info.qh, t);
                        issued_kq[s] = n;
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
                for (uint32_t s = 0; s < kKQStages; ++s)
                    if (issued_kq[s] >= 0) drain_bar(cx, B_KQ_FULL + s, (issued_kq[s] / kKQStages) & 1);
                if (issued_v >= 0) drain_bar(cx, B_V_FULL, issued_v & 1);
            }
        } else if (warp == 1) {
            // ================= tcgen05 issue: D1 and U (whole warp; one elected lane issues) =================
            // D1 of the next chunk of the unit needs only the intra side to be done with D1 of this one
            // (mid-chunk) and its K | Q tiles (three stages), while U of this chunk needs the full inverse: D1
            // goes first, so the intra side finds it computed when it starts the next chunk.
            uint32_t n = 0, u = 0;
            bool ok = true;
            auto next_unit = [&](UnitInfo& info) -> bool {  // next unit with chunks (or the end marker)
                for (;;) {
                    const int slot = u & 1;
                    if (!wait_bar_warp(cx, B_UNIT_FULL + slot, (u >> 1) & 1)) return false;
                    info = read_unit(sm, slot);
                    if (lane == 0) mbar_arrive(cx.bars + B_UNIT_EMPTY + slot);
                    ++u;
                    if (!info.valid || info.nC > 0) return true;
                }
            };
            auto issue_d1 = [&](uint32_t m) -> bool {  // D1 of global chunk m
                const uint32_t st = m % kKQStages;
                if (!wait_bar_warp(cx, B_KQ_FULL + st, (m / kKQStages) & 1)) return false;
                if (m >= 1 && !wait_bar_warp(cx, B_D1_EMPTY, (m - 1) & 1)) return false;
                tc_fence_after();
                const uint32_t kq = smem_u32(sm + kKQ + st * kKQStage);
#pragma unroll 1
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                    mma_ss_elect(tmem + kTmD1, desc_kmajor_sw128(kq + off), desc_kmajor_sw128(kq + off),
                                 kIdescD1<kF16>, ks > 0);
                }
                mma_commit_elect(cx.bars + B_D1_FULL);
                return true;
            };
            auto issue_u = [&](uint32_t m, bool no_u) -> bool {  // U of global chunk m (U = 0: no product)
                // the Delta slot is free once S of chunk m-2 has read it; T comes last (usually the last to complete)
                if (!wait_bar_warp(cx, B_V_FULL, m & 1)) return false;
                if (m >= 2 && !wait_bar_warp(cx, B_S_FULL + (m & 1), ((m - 2) >> 1) & 1)) return false;
                if (!wait_bar_warp(cx, B_T_FULL + (m & 1), (m >> 1) & 1)) return false;
                tc_fence_after();
                const uint32_t vv = smem_u32(sm + kV);
                const uint32_t tpp = smem_u32(sm + kTpp);
                const uint32_t dbuf = tmem + kTmDelta + (m & 1) * 64;
                if (!(kTransfer && no_u)) {
#pragma unroll 1
                    for (int ks = 0; ks < 4; ++ks)
                        mma_ss_elect(dbuf, desc_mnmajor_sw128(vv + ks * 2048, 8192), desc_kmajor_sw128(tpp + ks * 32),
                                     kIdescU<kF16>, ks > 0);
                }
                mma_commit_elect(cx.bars + B_U_FULL + (m & 1));
                mma_commit_elect(cx.bars + B_V_EMPTY);
                return true;
            };
            // Look-ahead stays inside a unit: reading the next unit early could wait on a ring slot that the
            // other roles free only after this unit's last U (two empty units in a row do that).
            while (ok) {
                UnitInfo cur;
                if (!(ok = next_unit(cur)) || !cur.valid) break;
                ok = issue_d1(n);
                for (int32_t c = 0; c < cur.nC && ok; ++c, ++n) {
                    if (c + 1 < cur.nC) ok = issue_d1(n + 1);
                    if (ok) ok = issue_u(n, kTransfer && cur.valid == 2);
                }
            }
            mma_commit_elect(cx.bars + B_DRAIN_I);
            drain_bar(cx, B_DRAIN_I, 0);
        } else if (warp == 2) {
            // ================= tcgen05 issue: X | S Q'^T, Delta, Delta P^T, S (whole warp, elected lane) =========
            uint32_t n = 0, u = 0;
            bool ok = true;
            for (; ok;) {
                const int slot = u & 1;
                if (!(ok = wait_bar_warp(cx, B_UNIT_FULL + slot, (u >> 1) & 1))) break;
                const UnitInfo info = read_unit(sm, slot);
                if (lane == 0) mbar_arrive(cx.bars + B_UNIT_EMPTY + slot);
                ++u;
                if (!info.valid) break;
                for (int32_t c = 0; c < info.nC; ++c, ++n) {
                    const int s = n & 1;
                    const uint32_t ph = (n >> 1) & 1;
                    const uint32_t st = n % kKQStages;
                    // [X | O] = S [K; Q']^T: the K and Q rows of a stage half are adjacent, one N = 128 B operand
                    // (the transfer pass forms X alone).  The O columns are free once the previous output
                    // epilogue has read them.
                    // (the waits on the intra side and the loads come first: they are usually complete; the state
                    // pass's release comes last, so one wake-up starts the issue)
                    if (!(ok = wait_bar_warp(cx, B_SB_FULL + s, ph))) break;
                    if (!(ok = wait_bar_warp(cx, B_KQ_FULL + st, (n / kKQStages) & 1))) break;
                    if (!kTransfer) {
                        if (n >= 1 && !(ok = wait_bar_warp(cx, B_O_EMPTY + ((n - 1) & 1), ((n - 1) >> 1) & 1))) break;
                        if (!(ok = wait_bar_warp(cx, B_GATES_FULL + n % 3, (n / 3) & 1))) break;
                        const float keepq = reinterpret_cast<const float*>(sm + kGbuf)[(n % 3) * kGFloats + kGKeepQ];
                        if (keepq == 0.f && !(ok = wait_bar_warp(cx, B_Q_READY + s, ph))) break;
                    }
                    tc_fence_after();
                    // descriptors advance by constants (16-byte units of the start address).  The issue loops stay
                    // rolled: unrolled, the back-to-back products slowed the whole kernel by about a tenth.
                    const uint32_t kq = smem_u32(sm + kKQ + st * kKQStage);
                    const uint64_t dkq = desc_kmajor_sw128(kq);
#pragma unroll 1
                    for (int ks = 0; ks < 8; ++ks)  // A = S (bf16 pairs in TMEM), k = 16 ks .. 16 ks + 15
                        mma_ts_elect(tmem + kTmX, tmem + kTmSbf + ks * 8, dkq + (((ks >> 2) * 16384 + (ks & 3) * 32) >> 4),
                                     kTransfer ? kIdescX<kF16> : kIdescXO<kF16>, ks > 0);
                    mma_commit_elect(cx.bars + B_XO_FULL);
                    // Delta~^T = U~^T - X T'^T: tf32 products with A = X read as fp32 straight from TMEM (negated)
                    // and T' in fp32, once X is complete (U = 0 for a transfer-matrix unit).  The test instance
                    // also waits for the state warps to have read U (XB_FULL).
                    if (!(ok = wait_bar_warp(cx, B_XO_FULL, n & 1))) break;
                    if (kDump && !(ok = wait_bar_warp(cx, B_XB_FULL, n & 1))) break;
                    if (!(ok = wait_bar_warp(cx, B_T_FULL + s, ph))) break;
                    if (!(ok = wait_bar_warp(cx, B_U_FULL + s, ph))) break;
                    tc_fence_after();
                    const uint64_t dtp = desc_kmajor_sw128(smem_u32(sm + (s ? kTp1 : kTp)));
                    const uint32_t dbuf = tmem + kTmDelta + s * 64;
                    const uint32_t acc0 = !(kTransfer && info.valid == 2);
#pragma unroll 1
                    for (int ks = 0; ks < 8; ++ks)  // j = 8 ks .. 8 ks + 7: 32 bytes of a T' row, halves of 32 j
                        mma_ts_tf32_elect(dbuf, tmem + kTmX + ks * 8, dtp + ((((ks >> 2) * 8192) + (ks & 3) * 32) >> 4),
                                          kIdescDelta, ks > 0 ? 1u : acc0);
                    mma_commit_elect(cx.bars + B_DELTA_FULL + s);
                    // O += Delta^T P^T (its own commit, so the output epilogue overlaps the S product), then
                    // S += (decayed Delta)^T K
                    if (!(ok = wait_bar_warp(cx, B_DD_FULL + s, ph))) break;
                    tc_fence_after();
                    if (!kTransfer) {
                        const uint64_t dpb = desc_kmajor_sw128(smem_u32(sm + kPb + s * 8192));
#pragma unroll 1
                        for (int ks = 0; ks < 4; ++ks)  // packed j = 16 ks .. 16 ks + 15
                            mma_ts_elect(tmem + kTmO, dbuf + 32 * (ks >> 1) + 8 * (ks & 1), dpb + ks * 2, kIdescO<kF16>,
                                         1);
                        mma_commit_elect(cx.bars + B_O_FULL);
                    }
                    const uint64_t dks = desc_mnmajor_sw128(kq, 16384);
#pragma unroll 1
                    for (int ks = 0; ks < 4; ++ks)
                        mma_ts_elect(tmem + kTmS, dbuf + 32 * (ks >> 1) + 8 * (ks & 1) + 16, dks + ks * 128, kIdescS<kF16>,
                                     1);
                    mma_commit_elect(cx.bars + B_S_FULL + s);
                    mma_commit_elect(cx.bars + B_KQ_EMPTY + st);
                }
            }
            mma_commit_elect(cx.bars + B_DRAIN_S);
            drain_bar(cx, B_DRAIN_S, 0);
        } else if (warp == 3) {
            // ================= gates warp: G, gamma, beta and factor vectors per chunk =================
            uint32_t n = 0, u = 0;
            bool ok = true;
            for (; ok;) {
                const int slot = u & 1;
                if (!(ok = wait_bar_warp(cx, B_UNIT_FULL + slot, (u >> 1) & 1))) break;
                const UnitInfo info = read_unit(sm, slot);
                __syncwarp();
                if (lane == 0) mbar_arrive(cx.bars + B_UNIT_EMPTY + slot);
                ++u;
                if (!info.valid) break;
                GatePrefetch gpf{1.f, 1.f, 0.f, 0.f};
                if (info.nC > 0)
                    gpf = load_gates(p, info.t0, info.L < kChunk ? static_cast<int32_t>(info.L) : kChunk, info.h, lane);
                for (int32_t c = 0; c < info.nC; ++c, ++n) {
                    const uint32_t gs = n % 3;  // gates slot (three in flight)
                    const GatePrefetch cur = gpf;
                    if (c + 1 < info.nC) {
                        const int64_t rem1 = info.L - static_cast<int64_t>(c + 1) * kChunk;
                        gpf = load_gates(p, info.t0 + static_cast<int64_t>(c + 1) * kChunk,
                                         rem1 < kChunk ? static_cast<int32_t>(rem1) : kChunk, info.h, lane);
                    }
                    if (n >= 3 && !(ok = wait_bar_warp(cx, B_GATES_EMPTY + gs, ((n - 3) / 3) & 1))) break;
                    float* gbw = reinterpret_cast<float*>(sm + kGbuf) + gs * kGFloats;
                    compute_gates(cur, gbw, p.l2norm != 0, kF16 ? 0.f : kKeepQRange, lane);
                    __syncwarp();
                    // The q norms (for the output epilogue only) come from the chunk's Q tile as stored: a chunk
                    // that keeps Q publishes its gates first and the norms after them (RM_FULL); one that does
                    // not keep Q computes the norms first, because the intra warps rescale Q in place once they
                    // have the gates.  (The stage is released only after this chunk's products, and this slot
                    // only after its output epilogue.)
                    const bool qn = p.l2norm && !kTransfer;
                    const bool late = qn && gbw[kGKeepQ] != 0.f;
                    if (qn) {
                        if (late && lane == 0) mbar_arrive(cx.bars + B_GATES_FULL + gs);
                        if (!(ok = wait_bar_warp(cx, B_KQ_FULL + n % kKQStages, (n / kKQStages) & 1))) break;
                        const int64_t rem = info.L - static_cast<int64_t>(c) * kChunk;
                        q_norms<kF16>(sm + kKQ + (n % kKQStages) * kKQStage + 8192, gbw,
                                      rem < kChunk ? static_cast<int32_t>(rem) : kChunk, lane);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(cx.bars + B_RM_FULL + gs);
                    }
                    if (!late && lane == 0) mbar_arrive(cx.bars + B_GATES_FULL + gs);
                }
            }
        }
    } else if (warp < 12) {
        // ================= intra warpgroups (two; each TMEM lane row split in column halves) =================
        const int it = tid - 128;                      // 0..255
        const int wq = warp & 3;                       // TMEM lane quarter
        const int hh = (warp - 4) >> 2;                // column half
        const uint32_t tm_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        float* Abuf = reinterpret_cast<float*>(sm + kAbuf);
        float* X1 = reinterpret_cast<float*>(sm + kXs);
        float* X2 = X1 + 2 * 16 * kLdX1;
        uint32_t n = 0, u = 0;
        bool ok = true;
        // Every wait's outcome is ANDed over the two warpgroups at their next named barrier
        // (named_bar_and), and the group leaves its loops only there, all together.
        for (; ok;) {
            const int slot = u & 1;
            ok = wait_bar(cx, B_UNIT_FULL + slot, (u >> 1) & 1);
            const UnitInfo info = read_unit(sm, slot);
            if (!(ok = named_bar_and(kBarIntra, kIntraThreads, ok))) break;
            if (it == 0) mbar_arrive(cx.bars + B_UNIT_EMPTY + slot);
            ++u;
            if (!info.valid) break;
            for (int32_t c = 0; c < info.nC && ok; ++c, ++n) {
                const int s = n & 1;
                const int64_t rem = info.L - static_cast<int64_t>(c) * kChunk;
                const int32_t Lc = rem < kChunk ? static_cast<int32_t>(rem) : kChunk;
                const uint32_t gs = n % 3;
                float* gb = reinterpret_cast<float*>(sm + kGbuf) + gs * kGFloats;
                uint8_t* kqs = sm + kKQ + (n % kKQStages) * kKQStage;
                ok = wait_bar(cx, B_GATES_FULL + gs, (n / 3) & 1);
                // P buffer s is free once O2 of chunk n-2 has completed (only the P-row warps write it)
                if (n >= 2 && wq >= 2) ok = ok && wait_bar(cx, B_S_FULL + s, ((n - 2) >> 1) & 1);
                ok = ok && wait_bar(cx, B_D1_FULL, n & 1);
                tc_fence_after();
                // A rows (lanes 0..63: warps with wq < 2) and P rows (lanes 64..127), row i, this warp's 32
                // columns.  A half that lies entirely above the diagonal is skipped (A's upper part and diagonal
                // are never read by the inverse, so A needs no mask; P's stays zero).  e^{G_i - G_j} is the row
                // factor times colf[j] while the chunk's gate range is moderate, else it is computed pairwise.
                {
                    const bool arow = wq < 2;
                    const int i = 32 * (wq & 1) + lane;
                    const bool active = !(hh == 1 && (wq & 1) == 0) && !(kTransfer && !arow);  // warp-uniform
                    float rn = 1.f;
                    if (arow && active && p.l2norm) {
                        // n_i = 1/|k_i|: |k_i|^2 is the diagonal of K K^T, column i of this lane's row (the warps
                        // whose half holds the diagonal find it in their main load below; warp wq = 1, hh = 0
                        // loads that half as well)
                        uint32_t rd[32];
                        tmem_ld32_wait(tm_lane + kTmD1 + 32 * (wq & 1), rd);
                        float kk = 0.f;
#pragma unroll
                        for (int j = 0; j < 32; ++j) kk = (j == lane) ? __uint_as_float(rd[j]) : kk;
                        rn = i < Lc ? rsqrtf(kk + 1e-6f) : 0.f;
                        if (hh == (wq & 1)) {  // one writer per row: the factors the inverse reads
                            gb[kGRn + i] = rn;
                            gb[kGCw + i] *= rn * rn;
                            gb[kGBn + i] *= rn;
                        }
                    }
                    if (active) {
                        uint32_t rr[32];
                        tmem_ld32_wait(tm_lane + kTmD1 + 32 * hh, rr);
                        float x[32];
                        const float rf = arow ? gb[kGRa + i] * rn * rn : gb[kGRp + i];
                        if (gb[kGSafe] != 0.f) {
#pragma unroll
                            for (int q = 0; q < 32; q += 4) {
                                const float4 cj = *reinterpret_cast<const float4*>(gb + kGColf + 32 * hh + q);
                                x[q] = rf * cj.x * __uint_as_float(rr[q]);
                                x[q + 1] = rf * cj.y * __uint_as_float(rr[q + 1]);
                                x[q + 2] = rf * cj.z * __uint_as_float(rr[q + 2]);
                                x[q + 3] = rf * cj.w * __uint_as_float(rr[q + 3]);
                            }
                        } else {
                            // pairwise: the row factor without its e^{G_i - Gref}, times e^{G_i - G_j}
                            const float rb = arow ? gb[kGBeta + i] * rn * rn
                                                  : (gb[kGKeepQ] != 0.f ? 1.f / gb[kGGam + i] : 1.f);
                            const float Gi = gb[kGG + i];
#pragma unroll
                            for (int q = 0; q < 32; ++q)
                                x[q] = rb * __expf(Gi - gb[kGG + 32 * hh + q]) * __uint_as_float(rr[q]);
                        }
                        if (arow) {
#pragma unroll
                            for (int q = 0; q < 32; q += 4)
                                *reinterpret_cast<float4*>(Abuf + i * kLd + 32 * hh + q) =
                                    make_float4(x[q], x[q + 1], x[q + 2], x[q + 3]);
                        } else {
                            uint8_t* pb = sm + kPb + s * 8192;
                            const int lim = i - 32 * hh;  // keep j <= i
#pragma unroll
                            for (int q = 0; q < 32; ++q) x[q] = q <= lim ? x[q] : 0.f;
#pragma unroll
                            for (int q = 0; q < 4; ++q) st_chunk16<kF16>(pb, i, 4 * hh + q, x + 8 * q);
                        }
                    }
                }
                // Q' = diag(gamma) Q in place, for the S Q'^T product (D1 has read Q already), unless the chunk
                // keeps Q as stored.  Four threads per row, 32 values each.
                if (gb[kGKeepQ] == 0.f && !kTransfer) scale_q_rows<kF16>(kqs, it, gb);
                // zero the padded rows of the K and V tiles (they hold the next
                // sequence or TMA zero fill; only exact zeros may meet them)
                if (Lc < kChunk) {
                    ok = ok && wait_bar(cx, B_V_FULL, n & 1);
                    zero_tail_rows(kqs, sm + kV, it, Lc);
                }
                // Q' and the zeroed K / V rows reach the async proxy before Q_READY (the X | O product reads Q')
                fence_proxy_async_smem();
                tc_fence_before();
                if (!(ok = named_bar_and(kBarIntra, kIntraThreads, ok))) break;
                // T = (I + A)^-1 in place, with T' = T diag(cw) (buffer s) and T'' = T diag(beta) in their bf16
                // tiles: U of the previous chunk has read T'', and Delta of chunk n-2 has read T' buffer s.  Only
                // the inverse's second stage writes those tiles, two group barriers later, so the hand-offs and
                // these waits run on warps 8..11, which have no work in its first stage, and warps 4 and 5 start
                // the forward substitution at once.
                if (it >= 128) {
                    if (it == 192) {
                        mbar_arrive(cx.bars + B_D1_EMPTY);
                        mbar_arrive(cx.bars + B_Q_READY + s);
                    }
                    if (n >= 1) ok = wait_bar(cx, B_U_FULL + ((n - 1) & 1), ((n - 1) >> 1) & 1);
                    if (n >= 2) ok = ok && wait_bar(cx, B_DELTA_FULL + s, ((n - 2) >> 1) & 1);
                }
                tri_inverse_64<kF16>(Abuf, sm + (s ? kTp1 : kTp), sm + kTpp, gb + kGCw, gb + kGBn, X1, X2, it);
                fence_proxy_async_smem();
                if (!(ok = named_bar_and(kBarIntra, kIntraThreads, ok))) break;
                if (it == 192) mbar_arrive(cx.bars + B_T_FULL + s);
            }
        }
    } else {
        // ================= state warpgroups (two; each TMEM lane row split in column halves) =================
        const int st = tid - 384;                      // 0..255
        const int wq = warp & 3;
        const int hh = (warp - 12) >> 2;               // column half
        const int v = wq * 32 + lane;                  // TMEM lane = state row v
        const uint32_t tm_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        using E = Elem16<kF16>;
        const int32_t ck_every = (p.checkpoints && p.ckpt_n > 0) ? p.ckpt_n / kChunk : 0;
        uint32_t n = 0, u = 0;
        bool ok = true;
        // As in the intra warpgroups: wait outcomes are ANDed over both warpgroups at the next named barrier,
        // and the loops are left only there.  (The pre-scale pass ends an iteration with a wait, so neither
        // loop condition may test `ok`: a thread whose wait ran out carries it to the next AND barrier, which
        // every thread reaches, instead of leaving alone.)
        for (;;) {
            const int slot = u & 1;
            ok = wait_bar(cx, B_UNIT_FULL + slot, (u >> 1) & 1);
            const UnitInfo info = read_unit(sm, slot);
            if (!(ok = named_bar_and(kBarState, kStateThreads, ok))) break;
            if (st == 0) mbar_arrive(cx.bars + B_UNIT_EMPTY + slot);
            ++u;
            if (!info.valid) break;
            // element offset of this thread's 64 columns in the initial / output state (the caller's own, for a
            // whole sequence in the segment pass of context parallelism)
            const bool own = !kTransfer && info.valid == 3;
            const int64_t state_off = state_offset(own ? p.state2 : p.state, info.srow, info.h, v) + 64 * hh;
            const int32_t sdt = own ? p.state2.dtype : p.state.dtype;
            // checkpoints: every ck_every-th chunk end of the unit (a multiple of 64 tokens), counted down, so the
            // chunk loop does no division
            int32_t ck_left = ck_every, ck_row = 0;
            const void* s0 = own ? p.initial_state2 : p.initial_state;
            // a transfer-matrix unit starts from the identity: a 1 in column v - 64 hh of this thread's row v
            const bool ident = kTransfer && info.valid == 2;
            if (info.nC == 0) {
                if (ident)  // the transfer output is dense fp32
                    identity_state<kF16>(v - 64 * hh, 0, 0, 1.f, static_cast<float*>(p.output_state) + state_off);
                else if (void* const s_out = own ? p.output_state2 : p.output_state)
                    pass_state_through(s0, s_out, state_off, sdt);
                continue;
            }
            // initial state: S0 -> the bf16 operand columns and gamma_63(first chunk) * S0 -> the accumulator
            // (the previous unit's last products, their readers, completed before its last state epilogue)
            {
                ok = wait_bar(cx, B_GATES_FULL + n % 3, (n / 3) & 1);
                const float g63 = reinterpret_cast<const float*>(sm + kGbuf)[(n % 3) * kGFloats + kGGam + 63];
                if (ident)
                    identity_state<kF16>(v - 64 * hh, tm_lane + kTmSbf + 32 * hh, tm_lane + kTmS + 64 * hh, g63,
                                         nullptr);
                else
                    load_initial_state<kF16>(s0, state_off, sdt, tm_lane + kTmSbf + 32 * hh,
                                             tm_lane + kTmS + 64 * hh, g63);
                tc_fence_before();
                if (!(ok = named_bar_and(kBarState, kStateThreads, ok))) break;
                if (st == 0) mbar_arrive(cx.bars + B_SB_FULL + (n & 1));
            }
            for (int32_t c = 0; c < info.nC; ++c, ++n) {
                const int s = n & 1;
                const uint32_t ph = (n >> 1) & 1;
                const int64_t tc = info.t0 + static_cast<int64_t>(c) * kChunk;
                const int64_t rem = info.L - static_cast<int64_t>(c) * kChunk;
                const int32_t Lc = rem < kChunk ? static_cast<int32_t>(rem) : kChunk;
                const uint32_t gs = n % 3;
                const float* gb = reinterpret_cast<const float*>(sm + kGbuf) + gs * kGFloats;
                const uint32_t dbuf = tm_lane + kTmDelta + s * 64;
                if constexpr (kDump) {
                    // test dumps: U before the Delta product accumulates onto it (the issuer waits for XB_FULL in
                    // this instance), W from T' and K
                    ok = wait_bar(cx, B_XO_FULL, n & 1);
                    ok = ok && wait_bar(cx, B_U_FULL + s, ph) && wait_bar(cx, B_T_FULL + s, ph);
                    tc_fence_after();
                    dump_intra<kF16>(p.intra_w, p.intra_u, p.intra_g,
                                     (static_cast<size_t>(info.flat0 + c) * H + info.h) * kChunk * kHead,
                                     (static_cast<size_t>(info.flat0 + c) * H + info.h) * kChunk,
                                     sm + (s ? kTp1 : kTp), sm + kKQ + (n % kKQStages) * kKQStage,
                                     dbuf + 32 * hh, v, 32 * hh, st,
                                     reinterpret_cast<const float*>(sm + kGbuf) + gs * kGFloats + kGG);
                    tc_fence_before();
                    if (!(ok = named_bar_and(kBarState, kStateThreads, ok))) break;
                    if (st == 0) mbar_arrive(cx.bars + B_XB_FULL);
                }
                // ---- Delta epilogue: this thread's 32 columns j in [32 hh, 32 hh + 32) go back into TMEM as
                //      16 packed bf16 Delta words followed by 16 packed decayed words (A operands of O2 and S)
                ok = ok && wait_bar(cx, B_DELTA_FULL + s, ph);
                tc_fence_after();
                {
                    uint32_t ra[32], pk[16];
                    tmem_ld32_wait(dbuf + 32 * hh, ra);
#pragma unroll
                    for (int q = 0; q < 16; ++q) pk[q] = E::pack(__uint_as_float(ra[2 * q]), __uint_as_float(ra[2 * q + 1]));
                    tmem_st16(dbuf + 32 * hh, pk);
                    float dv[16];
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        lds16(gb + kGDec + 32 * hh + 16 * part, dv);
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            pk[8 * part + q] = E::pack(__uint_as_float(ra[16 * part + 2 * q]) * dv[2 * q],
                                                       __uint_as_float(ra[16 * part + 2 * q + 1]) * dv[2 * q + 1]);
                    }
                    tmem_st16(dbuf + 32 * hh + 16, pk);
                    tmem_wait_st();
                }
                tc_fence_before();
                if (!(ok = named_bar_and(kBarState, kStateThreads, ok))) break;
                if (st == 0) mbar_arrive(cx.bars + B_DD_FULL + s);
                // ---- output, part 1: tokens i in [32 hh, 32 hh + 32) of O for this warp's 32 rows v leave TMEM, in
                //      the accumulator-fragment layout of two 16-row blocks (ro0, ro1), while the S product runs
                //      behind the output product; the arithmetic waits until after pass 1, so the next X | O
                //      product finds its O columns free as soon as the next bf16 S is ready.
                uint32_t ro0[16], ro1[16];
                if (!kTransfer) {
                    ok = ok && wait_bar(cx, B_O_FULL, n & 1);
                    tc_fence_after();
                    tmem_ld16x256_x4_pair_wait(tm_lane + kTmO + 32 * hh, tm_lane + (16u << 16) + kTmO + 32 * hh, ro0, ro1);
                }
                // ---- state epilogue, pass 1: S_n -> the bf16 operand of the next X | O product (this thread's 64
                //      columns); the checkpoint and the final state are written later, off the state chain
                ok = ok && wait_bar(cx, B_S_FULL + s, ph);
                tc_fence_after();
                const bool last = (c + 1 == info.nC);
                {
#pragma unroll 1
                    for (int c0 = 0; c0 < 64; c0 += 16) {
                        uint32_t r[16];
                        tmem_ld16_wait(tm_lane + kTmS + 64 * hh + c0, r);
                        if (!last) {  // bf16 pairs (c, c + 1) in column c / 2 of the operand
                            uint32_t pk[8];
#pragma unroll
                            for (int q = 0; q < 8; ++q) pk[q] = E::pack(__uint_as_float(r[2 * q]), __uint_as_float(r[2 * q + 1]));
                            tmem_st8(tm_lane + kTmSbf + 32 * hh + c0 / 2, pk);
                        }
                    }
                    if (!last) tmem_wait_st();
                }
                tc_fence_before();
                if (!(ok = named_bar_and(kBarState, kStateThreads, ok))) break;
                if (st == 0) {
                    if (!last) mbar_arrive(cx.bars + B_SB_FULL + ((n + 1) & 1));
                    if (!kTransfer) mbar_arrive(cx.bars + B_O_EMPTY + s);
                }
                // ---- output, part 2: o_i = scale rm_i (S Q'^T + Delta^T P^T)_i into the output tile (once the previous
                //      chunk's store has read it), then one TMA store of a full chunk, or the valid rows of a tail.
                //      (Stores straight from registers were measured slower than the tile and its bulk store.)
                if (!kTransfer) {
                    if (p.l2norm) ok = ok && wait_bar(cx, B_RM_FULL + gs, (n / 3) & 1);
                    if (st == 0) bulk_wait_group_read0();
                    ok = named_bar_and(kBarState, kStateThreads, ok);
                    // the tile is two halves of 64 v (8 KB, rows i of 128 bytes, 16-byte chunk c of row i at
                    // c ^ (i % 8): the TMA 128-byte swizzle).  Each stmatrix writes four 8 x 8 blocks transposed:
                    // block (token group k, row block vb) of fragment block b, rows i = 32 hh + 8 k + j of 8 v.
                    const int fq = lane & 3, fm = lane >> 3, fj = lane & 7;
                    float2 fac[4];  // scale rm_i for this thread's tokens 32 hh + 8 k + 2 fq (+ 1)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float2 rm = *reinterpret_cast<const float2*>(gb + kGRm + 32 * hh + 8 * k + 2 * fq);
                        fac[k] = make_float2(p.scale * rm.x, p.scale * rm.y);
                    }
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        const uint32_t(&rb)[16] = b ? ro1 : ro0;
#pragma unroll
                        for (int kp = 0; kp < 2; ++kp) {
                            uint32_t w[4];
#pragma unroll
                            for (int mm = 0; mm < 4; ++mm) {
                                const int k = 2 * kp + (mm >> 1), vb = mm & 1;
                                w[mm] = E::pack(fac[k].x * __uint_as_float(rb[4 * k + 2 * vb]),
                                                fac[k].y * __uint_as_float(rb[4 * k + 2 * vb + 1]));
                            }
                            const int k = 2 * kp + (fm >> 1), i = 32 * hh + 8 * k + fj;
                            const int v0 = 32 * wq + 16 * b + 8 * (fm & 1);
                            stmatrix_x4_trans(smem_u32(sm + kOutT) + (v0 >> 6) * 8192 + i * 128 +
                                                  ((((v0 & 63) >> 3) ^ fj) << 4),
                                              w[0], w[1], w[2], w[3]);
                        }
                    }
                    fence_proxy_async_smem();
                    if (!(ok = named_bar_and(kBarState, kStateThreads, ok))) break;
                    if (Lc == kChunk) {
                        if (st == 0) {
                            tma_store_3d(&tm_o, sm + kOutT, 0, info.h, static_cast<int32_t>(tc));
                            tma_store_3d(&tm_o, sm + kOutT + 8192, 64, info.h, static_cast<int32_t>(tc));
                            bulk_commit_group();
                        }
                    } else {
                        store_output_tail(sm + kOutT, static_cast<uint8_t*>(p.output), st, Lc, tc, H, info.h);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(cx.bars + B_GATES_EMPTY + gs);  // one arrival per state warp
                // a checkpoint where the chunk end, local token 64 (c + 1), is inside the sequence: this thread's 64
                // columns go to the dense checkpoint row in the checkpoint type
                int64_t ck_off = -1;
                if (ck_every > 0 && --ck_left == 0) {
                    ck_left = ck_every;
                    if (static_cast<int64_t>(c + 1) * kChunk <= info.L)
                        ck_off = ((info.ckpt_base + ck_row) * H + info.h) * static_cast<int64_t>(kHead * kHead) +
                                 static_cast<int64_t>(v) * kHead + 64 * hh;
                    ++ck_row;
                }
                if (!last) {
                    // pass 2: gamma_63 of the next chunk into the accumulator, before that chunk's S product (the
                    // next Delta epilogue's barrier orders it before that product's issue); S_n on its way through
                    // is the checkpoint
                    const uint32_t gn = (n + 1) % 3;
                    ok = wait_bar(cx, B_GATES_FULL + gn, ((n + 1) / 3) & 1);
                    const float gnext = reinterpret_cast<const float*>(sm + kGbuf)[gn * kGFloats + kGGam + 63];
                    // the checkpoint (S_n, before the scale), staged through the output tile's buffer once the
                    // output store has read it (not the unit's last chunk, so that store is a TMA store)
                    if (ck_off >= 0) {
                        if (st == 0) bulk_wait_group_read0();
                        ok = named_bar_and(kBarState, kStateThreads, ok);
                        float* slice = reinterpret_cast<float*>(sm + kOutT) + (st >> 5) * 512;
                        const int64_t warp_off = ck_off - static_cast<int64_t>(lane) * kHead;
#pragma unroll 1
                        for (int c0 = 0; c0 < 64; c0 += 16) {
                            uint32_t r[16];
                            tmem_ld16_wait(tm_lane + kTmS + 64 * hh + c0, r);
                            stage_rows16<4>(r, slice, p.checkpoints, warp_off, kHead, c0, p.ckpt_dtype, lane);
#pragma unroll
                            for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * gnext);
                            tmem_st16(tm_lane + kTmS + 64 * hh + c0, r);
                        }
                    } else {
#pragma unroll 1
                        for (int c0 = 0; c0 < 64; c0 += 32) {
                            uint32_t r[32];
                            tmem_ld32_wait(tm_lane + kTmS + 64 * hh + c0, r);
#pragma unroll
                            for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * gnext);
                            tmem_st32(tm_lane + kTmS + 64 * hh + c0, r);
                        }
                    }
                    tmem_wait_st();
                } else {
                    // the unit's last chunk: its checkpoint (when due) and the final state, out of line, staged
                    // through the output tile's buffer once this chunk's output (its TMA store or the tail rows)
                    // has left it
                    if (st == 0) bulk_wait_group_read0();
                    ok = named_bar_and(kBarState, kStateThreads, ok);
                    finish_unit(tm_lane + kTmS + 64 * hh, p.checkpoints, ck_off, p.ckpt_dtype,
                                own ? p.output_state2 : p.output_state, state_off,
                                own ? p.state2.s_v : p.state.s_v, own ? p.state2.dtype : p.state.dtype);
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

cudaError_t launch_chunk_16bit(const ChunkParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                               const CUtensorMap& tm_v, const CUtensorMap& tm_o, bool f16, bool transfer, int grid,
                               cudaStream_t stream) {
    // One flag per device and instance: cudaFuncSetAttribute runs once, and concurrent first calls from
    // several host threads each run it at most once more (the attribute value is the same).
    constexpr int kMaxDevices = 64;
    static std::atomic<uint8_t> configured[kMaxDevices][6];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool dump = p.intra_w || p.intra_u || p.intra_g;
    if (dump && transfer) return cudaErrorInvalidValue;
    auto* kernel = f16 ? (transfer ? gdn_chunk_kernel<__half, true, false>
                                   : (dump ? gdn_chunk_kernel<__half, false, true> : gdn_chunk_kernel<__half, false, false>))
                       : (transfer ? gdn_chunk_kernel<__nv_bfloat16, true, false>
                                   : (dump ? gdn_chunk_kernel<__nv_bfloat16, false, true>
                                           : gdn_chunk_kernel<__nv_bfloat16, false, false>));
    const int ki = (f16 ? 3 : 0) + (transfer ? 1 : (dump ? 2 : 0));
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!configured[dev][ki].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemAlloc));
        if (e != cudaSuccess) return e;
        configured[dev][ki].store(1, std::memory_order_release);
    }
    // a programmatic launch: the CTAs start while the previous kernel on the stream finishes (see griddep_wait)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p, tm_q, tm_k, tm_v, tm_o);
}

}  // namespace gdn
