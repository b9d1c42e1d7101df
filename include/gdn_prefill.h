/*
 * gdn_prefill.h -- C ABI of the chunked Gated DeltaNet prefill on one GB300 GPU.
 *
 * The operation ("FlashInfer GDN Prefill 完全指南", section
 * "chunk_gated_delta_rule API 全参数解析" gives the arguments, and
 * "GDN 与 Chunked Prefill", sections "GDN 是什么" and "块内 state 和块间 final
 * state", the recurrence and the read after the update): for every sequence i
 * of a packed variable-length batch and every state head h,
 *
 *     S_t = alpha_t * S_{t-1} * (I - beta_t k_t k_t^T) + beta_t * v_t k_t^T
 *     o_t = scale * S_t q_t
 *
 * with S a 128 x 128 fp32 matrix laid out [V][K], started from the initial
 * state (or zero), and computed in 64-token chunks: only each chunk's final
 * state crosses a chunk boundary ("GDN 与 Chunked Prefill", section "为什么要切成
 * 64-token chunk").
 *
 * Shapes (all tensors dense, row-major, device memory unless stated):
 *   q [T, HQ, 128], k [T, HK, 128], v [T, HV, 128]  bf16, fp16 or fp32 (one type)
 *   g, beta          [T, H] fp32, H = max(HQ, HV)   (g is alpha, linear space)
 *   cu_seqlens       [N+1] int32 or int64, cu_seqlens[0] = 0, cu_seqlens[N] = T;
 *                    equal neighbours are legal zero-length sequences
 *   initial_state    [N, H, 128, 128], or the pool [n_pool, H, 128, 128], in
 *                    the plan's state_dtype (fp32, bf16, fp16, fp8 e4m3 or
 *                    fp8 e5m2); element strides of the row, head and v dims
 *                    in state_strides (all 0: contiguous), the 128 k
 *                    elements contiguous
 *   output_state     same shape, type and strides; may be the same buffer
 *   state_indices    [N] int32 or int64: sequence i reads and writes pool row
 *                    state_indices[i] (unique, in [0, n_pool))
 *   state_checkpoints[sum_i floor(L_i / n), H, 128, 128] in the plan's
 *                    checkpoint_dtype (same choices as the state), dense: the
 *                    state after local token p = j * n of sequence i goes to
 *                    row checkpoint_cu_starts[i] + j - 1
 *   output           [T, H, 128], dtype of q
 * Head mapping ("FlashInfer GDN Prefill 完全指南", section on the legal CP
 * shapes): either HQ == HK and HV % HQ == 0 (GVA) or HK == HV and HQ % HK == 0
 * (GQA); state head h reads q head h / (H/HQ), k head h / (H/HK) and v head
 * h / (H/HV); g and beta are indexed by the state head.
 *
 * Ownership: the caller owns every tensor and the workspace; the library owns
 * only the opaque plan (shapes, dtypes, flags; no device pointers), so buffer
 * addresses may change from run to run.  gdn_prefill_run only enqueues work on
 * the caller's stream: it never synchronises, never allocates device memory
 * and never reads device memory on the host.
 *
 * Errors: conditions the host can check are returned synchronously and
 * nothing is launched (fail closed).  Conditions that depend on device data
 * (cu_seqlens order, checkpoint_cu_starts, state index range and uniqueness,
 * a sequence longer than max_seqlen, a timed-out wait) set bits of a device
 * status word, checked without a host round trip as the pages recommend
 * ("FlashInfer GDN Prefill 完全指南": checkpoint_cu_starts and state_indices are
 * not validated at launch to avoid a device-to-host sync); when a bit is set
 * the remaining kernels return early and the outputs are unspecified.  Read
 * the word with gdn_prefill_read_status, which synchronises the stream.
 */
#ifndef GDN_PREFILL_H
#define GDN_PREFILL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,   /* an argument breaks a documented precondition */
    GDN_ERR_UNSUPPORTED = 2,   /* legal for the API, outside this library's scope */
    GDN_ERR_CUDA = 3,          /* a CUDA runtime call failed (launch, attribute, ...) */
    GDN_ERR_DEVICE_INPUT = 4,  /* gdn_prefill_read_status: a device-checked input bit is set */
    GDN_ERR_DEVICE_TIMEOUT = 5 /* gdn_prefill_read_status: a bounded device wait ran out */
} gdn_status;

/* fp16 q/k/v run on fp16 tensor-core operands throughout (the kernel's own
 * 16-bit intermediates take the input type); values must stay inside fp16's
 * range (|x| < 65504), including raw q.k products and the state entries.
 * The two fp8 types ("FlashInfer GDN Prefill 完全指南": the initial_state row
 * of the API table and the dtype requirement of "中间状态检查点" list
 * float8_e4m3fn and float8_e5m2) are storage types of states and
 * checkpoints only: they are widened to fp32 on load, and on store rounded to
 * nearest (ties to even) and saturated to the finite range (e4m3: |x| <= 448,
 * no infinities; e5m2: |x| <= 57344); NaN stays NaN.  The recurrence itself
 * always runs in fp32. */
typedef enum gdn_dtype {
    GDN_DTYPE_F32 = 0,
    GDN_DTYPE_BF16 = 1,
    GDN_DTYPE_F16 = 2,
    GDN_DTYPE_F8E4M3 = 3, /* states and checkpoints only */
    GDN_DTYPE_F8E5M2 = 4  /* states and checkpoints only */
} gdn_dtype;

/* gdn_prefill_desc.flags */
enum {
    GDN_FLAG_HAS_G = 1u << 0,              /* g given; else alpha = 1 */
    GDN_FLAG_HAS_BETA = 1u << 1,           /* beta given; else beta = 1 */
    GDN_FLAG_HAS_SCALE = 1u << 2,          /* args.scale used; else 1/sqrt(128) */
    GDN_FLAG_QK_L2NORM = 1u << 3,          /* q, k rows -> x / sqrt(sum x^2 + 1e-6), fp32 sum, back to input dtype */
    GDN_FLAG_HAS_INITIAL_STATE = 1u << 4,  /* initial_state given; else zero */
    GDN_FLAG_OUTPUT_FINAL_STATE = 1u << 5, /* write the final state to output_state */
    GDN_FLAG_HAS_STATE_INDICES = 1u << 6,  /* initial/output state are pools addressed by state_indices */
    GDN_FLAG_CU_SEQLENS_I64 = 1u << 7,     /* cu_seqlens is int64 (else int32) */
    GDN_FLAG_STATE_INDICES_I64 = 1u << 8,  /* state_indices is int64 (else int32) */
    GDN_FLAG_CHECKPOINT_STARTS_I64 = 1u << 9, /* checkpoint_cu_starts is int64 (else int32) */
    /* Context parallelism inside the GPU ("FlashInfer GDN Prefill 完全指南",
     * the use_cp row of the API table and the CP backend's routing rules; the
     * per-segment transfer and boundary scan of "GDN与线性注意力GPU并行实现",
     * section 3.3): sequences long enough to set the run's time are cut into
     * segments whose start states come from a transfer pass and an fp32 scan,
     * so that more SMs share them, while the rest of the batch runs whole in
     * the same launches.  The device picks the segments from cu_seqlens with
     * a load model (no host sync), and picks none when they would not pay;
     * gdn_prefill_cp_segments gives the same choice on the host.  Same
     * results within rounding; the plan's workspace grows by about 32 MiB.
     * Not used with fp32 q/k/v, when intra-chunk outputs are requested, or
     * when args.max_seqlen shows that no sequence is long enough to gain. */
    GDN_FLAG_CONTEXT_PARALLEL = 1u << 10
};

/* Device status bits (gdn_prefill_read_status). */
enum {
    GDN_DEVICE_ERR_CU_SEQLENS = 1u << 0,        /* cu_seqlens[0] != 0, decreasing, or cu_seqlens[N] != T */
    GDN_DEVICE_ERR_CHECKPOINT_STARTS = 1u << 1, /* checkpoint_cu_starts != [0] + cumsum(L_i // n), or > capacity */
    GDN_DEVICE_ERR_STATE_INDEX_RANGE = 1u << 2, /* a state index outside [0, n_pool) */
    GDN_DEVICE_ERR_STATE_INDEX_DUP = 1u << 3,   /* two sequences name the same pool row */
    GDN_DEVICE_ERR_MAX_SEQLEN = 1u << 4,        /* a sequence longer than args.max_seqlen */
    GDN_DEVICE_ERR_TIMEOUT = 1u << 5            /* a bounded wait inside a kernel ran out */
};

/* Plan-time description: everything that selects kernels and sizes the
 * workspace.  Checked on the host by gdn_prefill_plan (no device needed). */
typedef struct gdn_prefill_desc {
    int32_t num_q_heads, num_k_heads, num_v_heads; /* HQ, HK, HV */
    int32_t head_size;                             /* must be 128 */
    gdn_dtype qkv_dtype;                           /* q, k, v and output: BF16, F16 or F32 */
    gdn_dtype state_dtype;                         /* initial / output states: F32, BF16, F16, F8E4M3 or F8E5M2,
                                                      widened to fp32 on load and rounded to nearest on store */
    int64_t max_total_tokens;                      /* upper bound of T over the plan's runs */
    int32_t max_num_seqs;                          /* upper bound of N */
    int32_t max_pool_rows;                         /* upper bound of n_pool (0 without state_indices) */
    int32_t checkpoint_every_n_tokens;             /* 0, or a multiple of 64 */
    uint32_t flags;                                /* GDN_FLAG_* */
    gdn_dtype checkpoint_dtype;                    /* state_checkpoints: F32 (0, the default), BF16, F16, F8E4M3
                                                      or F8E5M2, rounded to nearest on store like the states */
} gdn_prefill_desc;

typedef struct gdn_prefill_plan_s *gdn_prefill_plan_t;

/* Run-time arguments.  Pointers are device addresses; q, k, v and output must
 * be 16-byte aligned.  Unused optional pointers may be NULL. */
typedef struct gdn_prefill_args {
    const void *q, *k, *v;
    const float *g;               /* [T, H], required with GDN_FLAG_HAS_G */
    const float *beta;            /* [T, H], required with GDN_FLAG_HAS_BETA */
    float scale;                  /* used with GDN_FLAG_HAS_SCALE */
    const void *cu_seqlens;       /* [N+1] */
    int32_t num_seqs;             /* N >= 0 */
    int64_t total_tokens;         /* T >= 0 */
    int64_t max_seqlen;           /* 0 = unknown; else ceil(T/N) <= max_seqlen <= T (upper bound of L_i) */
    const void *initial_state;    /* required with GDN_FLAG_HAS_INITIAL_STATE; desc.state_dtype */
    void *output_state;           /* required with GDN_FLAG_OUTPUT_FINAL_STATE; desc.state_dtype */
    /* Element strides of [row][head][v] of both states; {0, 0, 0} = contiguous
     * (H*128*128, 128*128, 128).  Otherwise each is positive, a multiple of 16
     * bytes (16 elements of an fp8 state), and the layout does not overlap:
     * sorted by stride, each stride is at least the extent covered by the
     * smaller ones (128 for the v rows' own k elements).  Anything else is
     * GDN_ERR_INVALID_ARG. */
    int64_t state_strides[3];
    int32_t n_pool;               /* pool rows, with GDN_FLAG_HAS_STATE_INDICES */
    const void *state_indices;    /* [N], with GDN_FLAG_HAS_STATE_INDICES */
    void *state_checkpoints;      /* required when checkpoint_every_n_tokens > 0; desc.checkpoint_dtype */
    int64_t num_checkpoints;      /* rows of state_checkpoints (capacity, checked on the device) */
    const void *checkpoint_cu_starts; /* [N+1], required when checkpoint_every_n_tokens > 0 */
    void *output;                 /* [T, H, 128], dtype of q */
    int32_t *device_status;       /* optional: where to keep the status word (else in the workspace) */
    /* Optional outputs of the intra-chunk stage, indexed by flat chunk id f
     * (the order of the chunk map: sequence by sequence, chunk by chunk):
     * intra_g [F, H, 64] fp32 (G = running sum of log alpha in the chunk),
     * intra_w and intra_u [F, H, 64, 128] fp32 (W = T diag(beta*gamma) K,
     * U = T diag(beta) V with T = (I + A)^-1, for the keys as normalised; with
     * GDN_FLAG_QK_L2NORM row i of both comes multiplied by 1/|k_i|),
     * F = ceil(T/64) + N rows. */
    float *intra_g, *intra_w, *intra_u;
} gdn_prefill_args;

/* The context-parallel choice a gdn_prefill_run of this plan makes for a
 * batch of sequences with the host lengths seq_lens[num_seqs], on a GPU with
 * sm_count_hint SMs (or the current device's count when sm_count_hint <= 0):
 * the largest number of segments any sequence is cut into, 0 when every
 * sequence runs whole (also for plans without GDN_FLAG_CONTEXT_PARALLEL or
 * with fp32 q/k/v).  segments, when not NULL, receives each sequence's count
 * (1 = whole).  No launch; the device evaluates the same model from
 * cu_seqlens. */
int32_t gdn_prefill_cp_segments(gdn_prefill_plan_t plan, const int64_t *seq_lens, int32_t num_seqs,
                                int32_t sm_count_hint, int32_t *segments);

/* Validate `desc` and create a plan.  *workspace_bytes receives the device
 * workspace size gdn_prefill_run needs (16-byte aligned, caller allocated).
 * Needs no GPU.  Returns GDN_OK, GDN_ERR_INVALID_ARG or GDN_ERR_UNSUPPORTED. */
gdn_status gdn_prefill_plan(const gdn_prefill_desc *desc, gdn_prefill_plan_t *plan, size_t *workspace_bytes);

/* Enqueue one prefill on `stream` (a cudaStream_t; NULL = legacy default
 * stream).  Host-checked errors return before anything is launched. */
gdn_status gdn_prefill_run(gdn_prefill_plan_t plan, const gdn_prefill_args *args, void *workspace,
                           size_t workspace_bytes, void *stream);

/* The two halves of gdn_prefill_run, for callers that want to place events
 * or other work between them (same arguments and checks; the chunk half
 * must follow the prepare half of the same arguments on the same stream,
 * with no other run on that workspace in between):
 *   gdn_prefill_prepare -- the device-side chunk map, validation and work
 *                          order (one small kernel);
 *   gdn_prefill_chunks  -- the intra-chunk solve, state pass and output
 *                          (one persistent kernel). */
gdn_status gdn_prefill_prepare(gdn_prefill_plan_t plan, const gdn_prefill_args *args, void *workspace,
                               size_t workspace_bytes, void *stream);
gdn_status gdn_prefill_chunks(gdn_prefill_plan_t plan, const gdn_prefill_args *args, void *workspace,
                              size_t workspace_bytes, void *stream);

/* Copy the device status word of the last run on `stream` to *bits
 * (synchronises `stream`; outside the hot path).  `device_status` is the
 * pointer given in the run's args, or NULL when the word sits in the
 * workspace.  Returns GDN_OK when no bit is set, GDN_ERR_DEVICE_TIMEOUT when
 * the timeout bit is set, GDN_ERR_DEVICE_INPUT for any other bit. */
gdn_status gdn_prefill_read_status(gdn_prefill_plan_t plan, const void *workspace, const int32_t *device_status,
                                   void *stream, int32_t *bits);

/* Device buffers written by the prepare step (the chunk map), for callers
 * and tests: offsets in bytes from the workspace start.  chunk_offsets is
 * [N+1] int32 (exclusive prefix sum of ceil(L_i/64)), chunk_map is
 * [max_chunks, 2] int32 (sequence, chunk-in-sequence) padded with -1,
 * n_chunks is one int32, seq_order is [N] int32 (longest first). */
typedef struct gdn_prefill_layout {
    size_t status, n_chunks, chunk_offsets, chunk_map, seq_order;
    int64_t max_chunks;
} gdn_prefill_layout;
gdn_status gdn_prefill_workspace_layout(gdn_prefill_plan_t plan, gdn_prefill_layout *layout);

/* A run that allocates nothing.  The pages have no counterpart to this entry
 * point; it exists for callers that cannot allocate device memory when they
 * run the prefill (an allocator or memory-pool callback, or a host framework
 * that owns every allocation of the process) and so cannot supply a
 * workspace.  It runs exactly what gdn_prefill_run runs, with the workspace
 * taken from one fixed array of GDN_PREFILL_STATIC_WORKSPACE_BYTES in the
 * library's device globals; every GPU that loads the library holds that array
 * until the process exits.
 *   - Plans whose workspace is larger than the array are rejected with
 *     GDN_ERR_UNSUPPORTED before anything is launched (the plan's
 *     workspace_bytes tells in advance; 1 MiB covers, for example, 4096
 *     sequences and 6 million tokens).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is kept per device and
 *     context: after a device reset the first call on the new context looks
 *     it up again (and must again come before any capture).
 *   - All calls share the array, and the prepare kernel resets what must start
 *     at zero on every call.  Calls whose kernels overlap on the GPU (other
 *     streams, or host threads without ordering between them) race on it.
 *   - With args.device_status NULL the status word lives in the array and
 *     cannot be read back; pass a device_status pointer to read it with
 *     gdn_prefill_read_status.
 * Nothing here allocates: no cudaMalloc, no cudaFree, no library allocator. */
#define GDN_PREFILL_STATIC_WORKSPACE_BYTES (1u << 20)
gdn_status gdn_prefill_run_static(gdn_prefill_plan_t plan, const gdn_prefill_args *args, void *stream);

/* One decode step, or a short run of tokens, per sequence: N sequences of
 * exactly `tokens_per_seq` tokens each (1..GDN_DECODE_MAX_TOKENS_PER_SEQ),
 * token j of sequence i at row i * tokens_per_seq + j of q, k, v, g, beta
 * and output.  Each sequence's state is read from initial_state (its pool row
 * with state_indices, else row i; zero without GDN_FLAG_HAS_INITIAL_STATE),
 * carried through its tokens with the same recurrence and read-after-update
 * output as the prefill ("GDN 与 Chunked Prefill", section "块内 state 和块间
 * final state": after the prefill, decode carries the final state forward one
 * token at a time), and written to output_state with
 * GDN_FLAG_OUTPUT_FINAL_STATE (in place when it is the same pool).
 *   - Uses a plan made for the prefill (head mapping, dtypes, flags); the
 *     plan must have checkpoint_every_n_tokens = 0 (else
 *     GDN_ERR_UNSUPPORTED), and total_tokens must equal N * tokens_per_seq.
 *   - cu_seqlens, max_seqlen, the checkpoint arguments and the workspace are
 *     not used (checkpoint pointers must be NULL).
 *   - Needs no workspace and no prepare step.  A pool index outside
 *     [0, n_pool) skips that sequence and sets GDN_DEVICE_ERR_STATE_INDEX_RANGE
 *     in args.device_status when that pointer is given; duplicate indices are
 *     a caller error (their rows race).
 *   - q, k, v and output 16-byte aligned. */
#define GDN_DECODE_MAX_TOKENS_PER_SEQ 64
gdn_status gdn_decode_run(gdn_prefill_plan_t plan, const gdn_prefill_args *args, int32_t tokens_per_seq,
                          void *stream);

void gdn_prefill_plan_destroy(gdn_prefill_plan_t plan);

const char *gdn_status_string(gdn_status status);

#ifdef __cplusplus
}
#endif

#endif /* GDN_PREFILL_H */
