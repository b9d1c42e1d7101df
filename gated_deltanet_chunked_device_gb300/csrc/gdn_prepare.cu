// gdn_prepare.cu -- device-side prepare step of the chunked GDN prefill.
//
// Builds, from cu_seqlens, the flat chunk -> (sequence, chunk) table that the
// pages' prepare_chunk_indices builds on the host ("GDN 与 Chunked Prefill",
// sections "chunked prefill 有两层含义" and "为什么 trace 里它可能看起来很贵": the
// host version forces a device-to-host copy and a sync).  Here it runs as one
// CTA on the caller's stream, so nothing crosses back to the host.
//
// It also
//  * validates what only device data can show (cu_seqlens order and total,
//    checkpoint_cu_starts against [0] + cumsum(L_i // n), state index range and
//    uniqueness, L_i <= max_seqlen) into the status word, with atomicOr;
//  * orders sequences longest first (LPT) for the persistent chunk kernel;
//  * resets the chunk kernel's work counter.
#include "gdn_internal.cuh"
#include "sm103_ptx.cuh"

namespace gdn {
namespace {

constexpr int kPrepThreads = 1024;
constexpr int kSortMax = 8192;  // sequences sorted on chip; more keep their order

__device__ __forceinline__ int32_t warp_incl_scan(int32_t x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

// Exclusive block scan of one value per thread; returns the prefix and the block total.
__device__ int32_t block_excl_scan(int32_t x, int32_t* warp_sums, int32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t inc = warp_incl_scan(x);
    if (lane == 31) warp_sums[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int32_t w = (lane < kPrepThreads / 32) ? warp_sums[lane] : 0;
        int32_t wi = warp_incl_scan(w);
        warp_sums[lane] = wi - w;
        if (lane == 31) *total = wi;
    }
    __syncthreads();
    int32_t r = warp_sums[warp] + inc - x;
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kPrepThreads) gdn_prepare_kernel(PrepareParams p) {
    extern __shared__ __align__(16) uint64_t sort_keys[];
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t tile_total;
    __shared__ int32_t s_err;
    const int tid = threadIdx.x;
    const int32_t N = p.num_seqs;
    // up to kSortMax sequences, the chunk offsets also live in shared memory, after the sort keys
    const bool on_chip = N <= kSortMax;
    int32_t n2 = 1;
    while (n2 < N) n2 <<= 1;
    int32_t* s_off = reinterpret_cast<int32_t*>(sort_keys + (on_chip ? n2 : 0));
    // the chunk kernel may start its set-up now; it reads what this kernel writes only after it completes
    griddep_launch_dependents();

    if (tid == 0) {
        s_err = 0;
        if (!p.keep_status) *p.status = 0;  // the word describes this run only
        *p.counter = 0;
    }
    for (int w = tid; w < p.bitmap_words; w += kPrepThreads) p.pool_bitmap[w] = 0u;
    __syncthreads();

    // ---- lengths, validation, chunk counts, exclusive scan of chunk counts
    int32_t carry = 0;
    int err = 0;
    if (tid == 0) {
        if (load_index(p.cu_seqlens, p.cu_i64, 0) != 0) err |= GDN_DEVICE_ERR_CU_SEQLENS;
        if (load_index(p.cu_seqlens, p.cu_i64, N) != p.total_tokens) err |= GDN_DEVICE_ERR_CU_SEQLENS;
        if (p.ckpt_n > 0) {
            if (load_index(p.ckpt_cu_starts, p.ckpt_i64, 0) != 0) err |= GDN_DEVICE_ERR_CHECKPOINT_STARTS;
            if (load_index(p.ckpt_cu_starts, p.ckpt_i64, N) > p.num_checkpoints)
                err |= GDN_DEVICE_ERR_CHECKPOINT_STARTS;
        }
    }
    for (int32_t base = 0; base < N; base += kPrepThreads) {
        const int32_t i = base + tid;
        int32_t nc = 0;
        if (i < N) {
            const int64_t L = load_index(p.cu_seqlens, p.cu_i64, i + 1) - load_index(p.cu_seqlens, p.cu_i64, i);
            if (L < 0) err |= GDN_DEVICE_ERR_CU_SEQLENS;
            if (p.max_seqlen > 0 && L > p.max_seqlen) err |= GDN_DEVICE_ERR_MAX_SEQLEN;
            const int64_t Lc = L > 0 ? L : 0;
            nc = static_cast<int32_t>((Lc + kChunk - 1) / kChunk);
            if (p.ckpt_n > 0) {
                const int64_t cnt = load_index(p.ckpt_cu_starts, p.ckpt_i64, i + 1) -
                                    load_index(p.ckpt_cu_starts, p.ckpt_i64, i);
                if (cnt != Lc / p.ckpt_n) err |= GDN_DEVICE_ERR_CHECKPOINT_STARTS;
            }
            if (p.state_indices) {
                const int64_t row = load_index(p.state_indices, p.idx_i64, i);
                if (row < 0 || row >= p.n_pool) {
                    err |= GDN_DEVICE_ERR_STATE_INDEX_RANGE;
                } else {
                    const uint32_t bit = 1u << (row & 31);
                    const uint32_t old = atomicOr(&p.pool_bitmap[row >> 5], bit);
                    if (old & bit) err |= GDN_DEVICE_ERR_STATE_INDEX_DUP;
                }
            }
        }
        const int32_t ex = block_excl_scan(nc, warp_sums, &tile_total);
        if (i < N) {
            p.chunk_offsets[i] = carry + ex;
            if (on_chip) s_off[i] = carry + ex;
        }
        carry += tile_total;  // every thread reads the same total
        __syncthreads();
    }
    if (tid == 0) {
        p.chunk_offsets[N] = carry;
        if (on_chip) s_off[N] = carry;
        *p.n_chunks = carry;
    }
    if (err) atomicOr(&s_err, err);
    __syncthreads();
    if (tid == 0 && s_err) atomicOr(p.status, s_err);

    // ---- flat chunk map: chunk f belongs to the last sequence whose offset is <= f
    const int32_t* offs = on_chip ? s_off : p.chunk_offsets;
    const int32_t total = carry < p.max_chunks ? carry : static_cast<int32_t>(p.max_chunks);
    for (int64_t f = tid; f < p.max_chunks; f += kPrepThreads) {
        int32_t seq = -1, c = -1;
        if (f < total) {
            int32_t lo = 0, hi = N;  // invariant: offsets[lo] <= f < offsets[hi]
            while (hi - lo > 1) {
                const int32_t mid = (lo + hi) >> 1;
                if (offs[mid] <= f) lo = mid;
                else hi = mid;
            }
            seq = lo;
            c = static_cast<int32_t>(f) - offs[lo];
        }
        p.chunk_map[2 * f] = seq;
        p.chunk_map[2 * f + 1] = c;
    }

    // ---- longest-first order of sequences (bitonic sort of (chunks desc, index asc))
    if (on_chip) {
        for (int32_t i = tid; i < n2; i += kPrepThreads) {
            uint64_t key = ~0ull;
            if (i < N) {
                const uint32_t nc = static_cast<uint32_t>(s_off[i + 1] - s_off[i]);
                key = (static_cast<uint64_t>(0x7fffffffu - nc) << 32) | static_cast<uint32_t>(i);
            }
            sort_keys[i] = key;
        }
        __syncthreads();
        for (int32_t k = 2; k <= n2; k <<= 1) {
            for (int32_t j = k >> 1; j > 0; j >>= 1) {
                for (int32_t i = tid; i < n2; i += kPrepThreads) {
                    const int32_t ixj = i ^ j;
                    if (ixj > i) {
                        const uint64_t a = sort_keys[i], b = sort_keys[ixj];
                        const bool up = (i & k) == 0;
                        if ((a > b) == up) {
                            sort_keys[i] = b;
                            sort_keys[ixj] = a;
                        }
                    }
                }
                __syncthreads();
            }
        }
        for (int32_t i = tid; i < N; i += kPrepThreads)
            p.seq_order[i] = static_cast<int32_t>(sort_keys[i] & 0xffffffffu);
    } else {
        for (int32_t i = tid; i < N; i += kPrepThreads) p.seq_order[i] = i;
    }
}

}  // namespace

cudaError_t launch_prepare(const PrepareParams& p, cudaStream_t stream) {
    int32_t n2 = 1;
    while (n2 < p.num_seqs && n2 < kSortMax) n2 <<= 1;
    const size_t smem = (p.num_seqs <= kSortMax)
                            ? static_cast<size_t>(n2) * sizeof(uint64_t) + static_cast<size_t>(p.num_seqs + 1) * sizeof(int32_t)
                            : 16;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(gdn_prepare_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    gdn_prepare_kernel<<<1, kPrepThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
