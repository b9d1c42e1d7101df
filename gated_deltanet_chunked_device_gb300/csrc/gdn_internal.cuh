// gdn_internal.cuh -- parameters shared by the host code and the kernels of the
// chunked Gated DeltaNet prefill.  Not part of the public C ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/gdn_prefill.h"

namespace gdn {

constexpr int kChunk = 64;     // tokens per chunk
constexpr int kHead = 128;     // head size (K = V = 128)

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
    const float* initial_state;    // nullptr = zeros
    float* output_state;           // nullptr = no final state
    const void* state_indices;     // nullptr = dense [N, H, V, K]
    int idx_i64;
    float* checkpoints;            // nullptr = none
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
};

// Arguments of the decode-step kernel (a few tokens per sequence, no chunking).
struct DecodeParams {
    const void* q;
    const void* k;
    const void* v;
    const float* g;                // nullptr: alpha = 1
    const float* beta;             // nullptr: beta = 1
    float scale;
    const float* initial_state;    // nullptr: zero state
    float* output_state;           // nullptr: state not written back
    const void* state_indices;     // nullptr: row = sequence
    int idx_i64;
    int32_t n_pool;
    void* output;
    int32_t* status;               // nullptr: out-of-range pool rows are skipped silently
    int32_t N, H, hq, hk, hv;
    int32_t m;                     // tokens per sequence
    int l2norm;
};

__host__ __device__ inline int64_t load_index(const void* p, int i64, int64_t i) {
    return i64 ? static_cast<const int64_t*>(p)[i] : static_cast<int64_t>(static_cast<const int32_t*>(p)[i]);
}

// Launchers (each file defines its own).
cudaError_t launch_prepare(const PrepareParams& p, cudaStream_t stream);
cudaError_t launch_chunk_16bit(const ChunkParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                               const CUtensorMap& tm_v, const CUtensorMap& tm_o, bool f16, int grid,
                               cudaStream_t stream);
cudaError_t launch_chunk_f32(const ChunkParams& p, int grid, cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams& p, gdn_dtype dtype, cudaStream_t stream);
size_t chunk_bf16_smem_bytes();
size_t plan_workspace_bytes(gdn_prefill_plan_t plan);

}  // namespace gdn
