// gdn_prefill_host.cu -- host side of the C ABI declared in include/gdn_prefill.h:
// plan validation, workspace layout, run-time argument checks, TMA descriptor
// encoding and kernel launches.  Nothing here synchronises or allocates device
// memory, and nothing reads device memory except gdn_prefill_read_status.
//
// Host checks follow the pages' fail-closed rules ("FlashInfer GDN Prefill
// 完全指南": head_size 128 on SM100; the legal head mappings; checkpoint interval
// a multiple of 64; checkpoints and their starts given together; an output
// state pool is required with state_indices; max_seqlen within
// [ceil(T/N), T]).
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <cudaTypedefs.h>
#include <mutex>
#include <new>
#include <utility>

#include "gdn_internal.cuh"

// Context-parallel scratch (plans with GDN_FLAG_CONTEXT_PARALLEL): byte offsets
// in the workspace, after the main layout.
struct CpLayout {
    size_t trans, start, seg_a, order_a, counter_a, seg_seq, cu_c, ckpt_c, vrow;
    size_t prep;              // the segment pass's prepare
    gdn::WorkspaceLayout wc;  // its layout, relative to prep
};

struct gdn_prefill_plan_s {
    gdn_prefill_desc desc;
    gdn::WorkspaceLayout ws;
    int32_t H;
    bool cp;
    CpLayout cpl;
    size_t ws_total;  // the whole workspace (main layout plus the context-parallel scratch)
};

namespace {

constexpr uint32_t kKnownFlags = GDN_FLAG_HAS_G | GDN_FLAG_HAS_BETA | GDN_FLAG_HAS_SCALE | GDN_FLAG_QK_L2NORM |
                                 GDN_FLAG_HAS_INITIAL_STATE | GDN_FLAG_OUTPUT_FINAL_STATE |
                                 GDN_FLAG_HAS_STATE_INDICES | GDN_FLAG_CU_SEQLENS_I64 | GDN_FLAG_STATE_INDICES_I64 |
                                 GDN_FLAG_CHECKPOINT_STARTS_I64 | GDN_FLAG_CONTEXT_PARALLEL;

// Context-parallel bound: transfer segments per run (each takes 2 H planes
// of the transfer output, so at most kCpMaxPlanes / 2 with one head).
constexpr int32_t kCpMaxTransfer = static_cast<int32_t>(gdn::kCpMaxPlanes / 2);

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

gdn::WorkspaceLayout make_layout(const gdn_prefill_desc& d) {
    gdn::WorkspaceLayout w{};
    const int64_t max_chunks = (d.max_total_tokens + gdn::kChunk - 1) / gdn::kChunk + d.max_num_seqs;
    size_t off = 0;
    w.status = off;
    off += 16;
    w.counter = off;
    off += 16;
    w.n_chunks = off;
    off += 16;
    w.chunk_offsets = off;
    off = align_up(off + sizeof(int32_t) * (static_cast<size_t>(d.max_num_seqs) + 1), 16);
    w.chunk_map = off;
    off = align_up(off + sizeof(int32_t) * 2 * static_cast<size_t>(max_chunks > 0 ? max_chunks : 1), 16);
    w.seq_order = off;
    off = align_up(off + sizeof(int32_t) * static_cast<size_t>(d.max_num_seqs > 0 ? d.max_num_seqs : 1), 16);
    w.pool_bitmap = off;
    w.bitmap_words = (d.max_pool_rows + 31) / 32;
    off = align_up(off + sizeof(uint32_t) * static_cast<size_t>(w.bitmap_words > 0 ? w.bitmap_words : 1), 256);
    w.total = off;
    w.max_chunks = max_chunks;
    return w;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

CUtensorMapDataType tma_type(gdn_dtype t) {
    return t == GDN_DTYPE_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
}

// [T, heads, 128] bf16 or fp16 tensor as a 3-D TMA map with 64 x 1 x 64 boxes
// and the 128-byte swizzle; rows past T read as zeros.
bool encode_qkv_map(CUtensorMap* map, const void* base, int64_t T, int32_t heads, gdn_dtype t) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(gdn::kHead), static_cast<cuuint64_t>(heads),
                          static_cast<cuuint64_t>(T)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(gdn::kHead) * 2,
                             static_cast<cuuint64_t>(heads) * gdn::kHead * 2};
    cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(gdn::kChunk)};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(map, tma_type(t), 3, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The output [T, heads, 128] as a 3-D TMA map for stores: 64 x 1 x 64 boxes (half a chunk's v columns) and the
// 128-byte swizzle, the layout the chunk kernel writes its output tile in.
bool encode_out_map(CUtensorMap* map, void* base, int64_t T, int32_t heads, gdn_dtype t) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(gdn::kHead), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(T)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(gdn::kHead) * 2, static_cast<cuuint64_t>(heads) * gdn::kHead * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(map, tma_type(t), 3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// The state layout of a run: the plan's state type and the args' strides
// ({0, 0, 0}: contiguous [rows][H][128][128]).  False when the strides are not
// positive multiples of 16 bytes or may overlap (checked as nested: sorted by
// stride, each dimension starts past the span of the smaller ones).
bool make_state_layout(gdn_dtype dt, const int64_t (&st)[3], int64_t rows, int32_t H, gdn::StateLayout* L) {
    L->dtype = dt;
    const int64_t es = gdn::dtype_bytes(dt);
    if (st[0] == 0 && st[1] == 0 && st[2] == 0) {
        L->s_v = gdn::kHead;
        L->s_head = static_cast<int64_t>(gdn::kHead) * gdn::kHead;
        L->s_row = L->s_head * H;
        return true;
    }
    int64_t ext[3] = {rows, H, gdn::kHead}, str[3] = {st[0], st[1], st[2]};
    for (int i = 0; i < 3; ++i)
        if (str[i] <= 0 || (str[i] * es) % 16 != 0) return false;
    int order[3] = {0, 1, 2};
    for (int i = 0; i < 3; ++i)
        for (int j = i + 1; j < 3; ++j)
            if (str[order[j]] < str[order[i]]) std::swap(order[i], order[j]);
    int64_t span = gdn::kHead;  // the contiguous k elements of one v row
    for (int i = 0; i < 3; ++i) {
        const int d = order[i];
        if (ext[d] <= 1) continue;
        if (str[d] < span) return false;
        span += str[d] * (ext[d] - 1);
    }
    L->s_row = st[0];
    L->s_head = st[1];
    L->s_v = st[2];
    return true;
}

// Whether a run takes the context-parallel route (the device then chooses the
// segments, possibly none): plans that allow it, 16-bit inputs, no intra-chunk
// dumps, room for one transfer segment, and -- when max_seqlen is given -- a
// longest sequence that the load model could shorten at all: with
// 0.85 ceil(max_seqlen / 64) <= H T / (64 S) the segment pass alone already
// costs 85 % of one pass (see cp_pick_tau), so one pass it is.
bool cp_route(gdn_prefill_plan_t plan, const gdn_prefill_args& a, int32_t N, int64_t T, int sms) {
    if (!plan->cp || plan->desc.qkv_dtype == GDN_DTYPE_F32 || a.intra_g || a.intra_w || a.intra_u) return false;
    if (N <= 0 || T <= 0 || sms <= 0 || 2 * static_cast<int64_t>(plan->H) > gdn::kCpMaxPlanes) return false;
    if (a.max_seqlen > 0) {
        const int64_t c_bound = (a.max_seqlen + gdn::kChunk - 1) / gdn::kChunk;
        if (85 * c_bound * gdn::kChunk * sms <= 100 * static_cast<int64_t>(plan->H) * T) return false;
    }
    return true;
}

// Bound of the transfer segments of a run of N sequences.
int32_t cp_transfer_bound(gdn_prefill_plan_t plan, int32_t N) {
    const int64_t by_planes = gdn::kCpMaxPlanes / (2 * static_cast<int64_t>(plan->H));
    const int64_t by_seqs = static_cast<int64_t>(N) * (gdn::kCpMaxSegments - 1);
    return static_cast<int32_t>(by_planes < by_seqs ? by_planes : by_seqs);
}

// The types a state or a checkpoint may be stored in.
bool storage_dtype(gdn_dtype t) {
    return t == GDN_DTYPE_F32 || t == GDN_DTYPE_BF16 || t == GDN_DTYPE_F16 || t == GDN_DTYPE_F8E4M3 ||
           t == GDN_DTYPE_F8E5M2;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace

size_t gdn::plan_workspace_bytes(gdn_prefill_plan_t plan) { return plan ? plan->ws_total : 0; }

extern "C" {

gdn_status gdn_prefill_plan(const gdn_prefill_desc* desc, gdn_prefill_plan_t* plan, size_t* workspace_bytes) {
    if (!desc || !plan || !workspace_bytes) return GDN_ERR_INVALID_ARG;
    *plan = nullptr;
    const gdn_prefill_desc& d = *desc;
    if (d.flags & ~kKnownFlags) return GDN_ERR_INVALID_ARG;
    if (d.head_size != gdn::kHead) return GDN_ERR_UNSUPPORTED;
    if (d.num_q_heads <= 0 || d.num_k_heads <= 0 || d.num_v_heads <= 0) return GDN_ERR_INVALID_ARG;
    const bool gva = d.num_q_heads == d.num_k_heads && d.num_v_heads % d.num_q_heads == 0;
    const bool gqa = d.num_k_heads == d.num_v_heads && d.num_q_heads % d.num_k_heads == 0;
    if (!gva && !gqa) return GDN_ERR_INVALID_ARG;
    if (d.qkv_dtype != GDN_DTYPE_BF16 && d.qkv_dtype != GDN_DTYPE_F16 && d.qkv_dtype != GDN_DTYPE_F32)
        return GDN_ERR_UNSUPPORTED;
    if (!storage_dtype(d.state_dtype) || !storage_dtype(d.checkpoint_dtype)) return GDN_ERR_UNSUPPORTED;
    if (d.checkpoint_every_n_tokens < 0 || d.checkpoint_every_n_tokens % gdn::kChunk != 0)
        return GDN_ERR_INVALID_ARG;
    if (d.max_total_tokens < 0 || d.max_num_seqs < 0 || d.max_pool_rows < 0) return GDN_ERR_INVALID_ARG;
    if (d.max_total_tokens > 0x7fffffffLL - gdn::kChunk) return GDN_ERR_UNSUPPORTED;  // 32-bit TMA coordinates
    if ((d.flags & GDN_FLAG_HAS_STATE_INDICES) && d.max_pool_rows <= 0) return GDN_ERR_INVALID_ARG;
    gdn_prefill_plan_s* p = new (std::nothrow) gdn_prefill_plan_s;
    if (!p) return GDN_ERR_INVALID_ARG;
    p->desc = d;
    p->ws = make_layout(d);
    p->H = d.num_q_heads > d.num_v_heads ? d.num_q_heads : d.num_v_heads;
    p->cp = (d.flags & GDN_FLAG_CONTEXT_PARALLEL) != 0;
    size_t total = p->ws.total;
    if (p->cp) {
        const size_t plane = sizeof(float) * gdn::kHead * gdn::kHead;
        CpLayout& c = p->cpl;
        c.trans = total;
        total = align_up(total + plane * gdn::kCpMaxPlanes, 256);
        c.start = total;
        total = align_up(total + plane * gdn::kCpMaxPlanes, 256);
        const int64_t vmax = static_cast<int64_t>(d.max_num_seqs) + kCpMaxTransfer;  // segment-pass batch bound
        if (vmax > 0x7fffffffLL) {
            delete p;
            return GDN_ERR_UNSUPPORTED;
        }
        c.seg_a = total;
        total = align_up(total + sizeof(int64_t) * 2 * kCpMaxTransfer, 256);
        c.order_a = total;
        total = align_up(total + sizeof(int32_t) * kCpMaxTransfer, 256);
        c.counter_a = total;  // the work counter, then the three counts
        total = align_up(total + 16, 256);
        c.seg_seq = total;
        total = align_up(total + sizeof(int32_t) * 4 * kCpMaxTransfer, 256);
        c.cu_c = total;
        total = align_up(total + sizeof(int32_t) * (vmax + 1), 256);
        c.ckpt_c = total;
        total = align_up(total + sizeof(int64_t) * (vmax + 1), 256);
        c.vrow = total;
        total = align_up(total + sizeof(int64_t) * vmax, 256);
        gdn_prefill_desc dc = d;
        dc.max_num_seqs = static_cast<int32_t>(vmax);
        dc.max_pool_rows = 0;
        c.wc = make_layout(dc);
        c.prep = total;
        total = align_up(total + c.wc.total, 256);
    }
    p->ws_total = total;
    *plan = p;
    *workspace_bytes = total;
    return GDN_OK;
}

void gdn_prefill_plan_destroy(gdn_prefill_plan_t plan) { delete plan; }

int32_t gdn_prefill_cp_segments(gdn_prefill_plan_t plan, const int64_t* seq_lens, int32_t num_seqs,
                                int32_t sm_count_hint, int32_t* segments) {
    if (!plan || num_seqs < 0 || (num_seqs > 0 && !seq_lens)) return 0;
    for (int32_t i = 0; i < num_seqs && segments; ++i) segments[i] = 1;
    const int sms = sm_count_hint > 0 ? sm_count_hint : sm_count();
    int64_t T = 0, c_max = 0, sum_c = 0;
    for (int32_t i = 0; i < num_seqs; ++i) {
        const int64_t L = seq_lens[i] > 0 ? seq_lens[i] : 0;
        const int64_t c = (L + gdn::kChunk - 1) / gdn::kChunk;
        T += L;
        sum_c += c;
        if (c > c_max) c_max = c;
    }
    gdn_prefill_args a{};
    if (!cp_route(plan, a, num_seqs, T, sms)) return 0;
    const int32_t n = plan->desc.checkpoint_every_n_tokens;
    const int64_t align = n > 0 ? n / gdn::kChunk : 1;
    gdn::CpSums s[gdn::kCpMaxSegments - 1];
    for (int32_t P = 2; P <= gdn::kCpMaxSegments; ++P) {
        s[P - 2] = gdn::CpSums{0, 0, 0, 0};
        const int64_t tau = gdn::cp_tau(c_max, P, align);
        for (int32_t i = 0; i < num_seqs; ++i)
            gdn::cp_add_sequence(s[P - 2], (std::max<int64_t>(seq_lens[i], 0) + gdn::kChunk - 1) / gdn::kChunk, tau);
    }
    const int64_t tau = gdn::cp_pick_tau(s, c_max, sum_c, plan->H, sms, align);
    int32_t most = 0;
    for (int32_t i = 0; tau > 0 && i < num_seqs; ++i) {
        const int32_t P = gdn::cp_seq_segments((std::max<int64_t>(seq_lens[i], 0) + gdn::kChunk - 1) / gdn::kChunk, tau);
        if (segments) segments[i] = P;
        if (P > most) most = P;
    }
    return most >= 2 ? most : 0;
}

gdn_status gdn_prefill_workspace_layout(gdn_prefill_plan_t plan, gdn_prefill_layout* layout) {
    if (!plan || !layout) return GDN_ERR_INVALID_ARG;
    layout->status = plan->ws.status;
    layout->n_chunks = plan->ws.n_chunks;
    layout->chunk_offsets = plan->ws.chunk_offsets;
    layout->chunk_map = plan->ws.chunk_map;
    layout->seq_order = plan->ws.seq_order;
    layout->max_chunks = plan->ws.max_chunks;
    return GDN_OK;
}

}  // extern "C"

namespace {

enum : int { kStagePrepare = 1, kStageChunks = 2 };

gdn_status run_stages(gdn_prefill_plan_t plan, const gdn_prefill_args* args, void* workspace,
                      size_t workspace_bytes, void* stream_ptr, int stages) {
    if (!plan || !args) return GDN_ERR_INVALID_ARG;
    const gdn_prefill_desc& d = plan->desc;
    const gdn_prefill_args& a = *args;
    const uint32_t f = d.flags;
    const int32_t N = a.num_seqs;
    const int64_t T = a.total_tokens;
    if (N < 0 || N > d.max_num_seqs || T < 0 || T > d.max_total_tokens) return GDN_ERR_INVALID_ARG;
    if (N == 0) return T == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
    if (!a.cu_seqlens) return GDN_ERR_INVALID_ARG;
    if (T > 0 && (!a.q || !a.k || !a.v || !a.output)) return GDN_ERR_INVALID_ARG;
    if (!aligned(a.q, 16) || !aligned(a.k, 16) || !aligned(a.v, 16) || !aligned(a.output, 16))
        return GDN_ERR_INVALID_ARG;
    if (T > 0 && (((f & GDN_FLAG_HAS_G) && !a.g) || ((f & GDN_FLAG_HAS_BETA) && !a.beta)))
        return GDN_ERR_INVALID_ARG;
    if ((f & GDN_FLAG_HAS_INITIAL_STATE) && (!a.initial_state || !aligned(a.initial_state, 16)))
        return GDN_ERR_INVALID_ARG;
    if ((f & GDN_FLAG_OUTPUT_FINAL_STATE) && (!a.output_state || !aligned(a.output_state, 16)))
        return GDN_ERR_INVALID_ARG;
    if (f & GDN_FLAG_HAS_STATE_INDICES) {
        if (!a.state_indices || a.n_pool <= 0 || a.n_pool > d.max_pool_rows) return GDN_ERR_INVALID_ARG;
    }
    const int32_t n = d.checkpoint_every_n_tokens;
    if (n > 0) {
        if (!a.state_checkpoints || !a.checkpoint_cu_starts || a.num_checkpoints < 0 ||
            !aligned(a.state_checkpoints, 16))
            return GDN_ERR_INVALID_ARG;
    } else if (a.state_checkpoints || a.checkpoint_cu_starts) {
        return GDN_ERR_INVALID_ARG;
    }
    if (a.max_seqlen != 0) {
        const int64_t lo = (T + N - 1) / N;
        if (a.max_seqlen > T || a.max_seqlen < lo) return GDN_ERR_INVALID_ARG;
    }
    gdn::StateLayout sl{};
    if (!make_state_layout(d.state_dtype, a.state_strides, (f & GDN_FLAG_HAS_STATE_INDICES) ? a.n_pool : N, plan->H,
                           &sl))
        return GDN_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < plan->ws_total || !aligned(workspace, 16)) return GDN_ERR_INVALID_ARG;

    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int32_t* status = a.device_status ? a.device_status : reinterpret_cast<int32_t*>(ws + plan->ws.status);

    gdn::PrepareParams pp{};
    pp.cu_seqlens = a.cu_seqlens;
    pp.cu_i64 = (f & GDN_FLAG_CU_SEQLENS_I64) ? 1 : 0;
    pp.num_seqs = N;
    pp.total_tokens = T;
    pp.max_seqlen = a.max_seqlen;
    pp.ckpt_n = n;
    pp.ckpt_cu_starts = a.checkpoint_cu_starts;
    pp.ckpt_i64 = (f & GDN_FLAG_CHECKPOINT_STARTS_I64) ? 1 : 0;
    pp.num_checkpoints = a.num_checkpoints;
    pp.state_indices = (f & GDN_FLAG_HAS_STATE_INDICES) ? a.state_indices : nullptr;
    pp.idx_i64 = (f & GDN_FLAG_STATE_INDICES_I64) ? 1 : 0;
    pp.n_pool = a.n_pool;
    pp.status = status;
    pp.counter = reinterpret_cast<int32_t*>(ws + plan->ws.counter);
    pp.n_chunks = reinterpret_cast<int32_t*>(ws + plan->ws.n_chunks);
    pp.chunk_offsets = reinterpret_cast<int32_t*>(ws + plan->ws.chunk_offsets);
    pp.chunk_map = reinterpret_cast<int32_t*>(ws + plan->ws.chunk_map);
    pp.max_chunks = (T + gdn::kChunk - 1) / gdn::kChunk + N;
    pp.seq_order = reinterpret_cast<int32_t*>(ws + plan->ws.seq_order);
    pp.pool_bitmap = reinterpret_cast<uint32_t*>(ws + plan->ws.pool_bitmap);
    pp.bitmap_words = (f & GDN_FLAG_HAS_STATE_INDICES) ? (a.n_pool + 31) / 32 : 0;
    if ((stages & kStagePrepare) && gdn::launch_prepare(pp, stream) != cudaSuccess) return GDN_ERR_CUDA;
    if (!(stages & kStageChunks)) return GDN_OK;

    gdn::ChunkParams cp{};
    cp.q = a.q;
    cp.k = a.k;
    cp.v = a.v;
    cp.g = (f & GDN_FLAG_HAS_G) ? a.g : nullptr;
    cp.beta = (f & GDN_FLAG_HAS_BETA) ? a.beta : nullptr;
    cp.scale = (f & GDN_FLAG_HAS_SCALE) ? a.scale : 1.0f / std::sqrt(static_cast<float>(gdn::kHead));
    cp.hq = d.num_q_heads;
    cp.hk = d.num_k_heads;
    cp.hv = d.num_v_heads;
    cp.H = plan->H;
    cp.l2norm = (f & GDN_FLAG_QK_L2NORM) ? 1 : 0;
    cp.cu_seqlens = a.cu_seqlens;
    cp.cu_i64 = pp.cu_i64;
    cp.num_seqs = N;
    cp.initial_state = (f & GDN_FLAG_HAS_INITIAL_STATE) ? a.initial_state : nullptr;
    cp.state = sl;
    cp.output_state = (f & GDN_FLAG_OUTPUT_FINAL_STATE) ? a.output_state : nullptr;
    cp.state_indices = pp.state_indices;
    cp.idx_i64 = pp.idx_i64;
    cp.checkpoints = n > 0 ? a.state_checkpoints : nullptr;
    cp.ckpt_dtype = d.checkpoint_dtype;
    cp.ckpt_n = n;
    cp.ckpt_cu_starts = a.checkpoint_cu_starts;
    cp.ckpt_i64 = pp.ckpt_i64;
    cp.output = a.output;
    cp.status = status;
    cp.counter = pp.counter;
    cp.chunk_offsets = pp.chunk_offsets;
    cp.seq_order = pp.seq_order;
    cp.intra_g = a.intra_g;
    cp.intra_w = a.intra_w;
    cp.intra_u = a.intra_u;
    cp.has_tokens = T > 0 ? 1 : 0;

    if (d.qkv_dtype == GDN_DTYPE_F32) {
        // fp32 inputs: CUDA-core kernel, one CTA per (sequence, state head, slice of the V rows): the most slices
        // (up to 16) that keep the grid within about four CTAs per SM, since every slice repeats the
        // slice-independent work
        const int64_t units = static_cast<int64_t>(N) * plan->H;
        if (units * 2 > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
        int slices = 16;
        while (slices > 2 && units * slices > 4LL * std::max(sm_count(), 1)) slices /= 2;
        if (gdn::launch_chunk_f32(cp, units, slices, stream) != cudaSuccess) return GDN_ERR_CUDA;
        return GDN_OK;
    }
    CUtensorMap tq, tk, tv, to;
    std::memset(&to, 0, sizeof(to));
    std::memset(&tq, 0, sizeof(tq));
    std::memset(&tk, 0, sizeof(tk));
    std::memset(&tv, 0, sizeof(tv));
    if (T > 0) {
        const gdn_dtype t = d.qkv_dtype;
        if (!encode_qkv_map(&tq, a.q, T, d.num_q_heads, t) || !encode_qkv_map(&tk, a.k, T, d.num_k_heads, t) ||
            !encode_qkv_map(&tv, a.v, T, d.num_v_heads, t) || !encode_out_map(&to, a.output, T, plan->H, t))
            return GDN_ERR_CUDA;
    }
    const int sms = sm_count();
    if (sms <= 0) return GDN_ERR_CUDA;
    const bool f16 = d.qkv_dtype == GDN_DTYPE_F16;
    const int32_t H = plan->H;
    const int64_t units = static_cast<int64_t>(N) * H;
    if (!cp_route(plan, a, N, T, sms)) {
        const int grid = static_cast<int>(units < sms ? units : sms);
        if (gdn::launch_chunk_16bit(cp, tq, tk, tv, to, f16, false, grid, stream) != cudaSuccess) return GDN_ERR_CUDA;
        return GDN_OK;
    }

    // ---- context parallelism: segmentation on the device, transfer pass, fp32 scan, one pass over the
    //      segments and the whole sequences, final states of the segmented sequences
    const CpLayout& c = plan->cpl;
    const int32_t nA_max = cp_transfer_bound(plan, N);
    gdn::CpParams q{};
    q.cu_seqlens = a.cu_seqlens;
    q.cu_i64 = pp.cu_i64;
    q.num_seqs = N;
    q.H = H;
    q.sms = sms;
    q.align_chunks = n > 0 ? n / gdn::kChunk : 1;
    q.nA_max = nA_max;
    q.V_max = N + nA_max;
    q.ckpt_n = n;
    q.ckpt_cu_starts = a.checkpoint_cu_starts;
    q.ckpt_i64 = pp.ckpt_i64;
    q.seg_a = reinterpret_cast<int64_t*>(ws + c.seg_a);
    q.order_a = reinterpret_cast<int32_t*>(ws + c.order_a);
    q.counter_a = reinterpret_cast<int32_t*>(ws + c.counter_a);
    q.counts = q.counter_a + 1;
    q.seg_seq = reinterpret_cast<int32_t*>(ws + c.seg_seq);
    q.cu_c = reinterpret_cast<int32_t*>(ws + c.cu_c);
    q.ckpt_c = reinterpret_cast<int64_t*>(ws + c.ckpt_c);
    q.vrow = reinterpret_cast<int64_t*>(ws + c.vrow);
    q.trans = reinterpret_cast<const float*>(ws + c.trans);
    q.start = reinterpret_cast<float*>(ws + c.start);
    q.initial_state = cp.initial_state;
    q.output_state = cp.output_state;
    q.state = sl;
    q.state_indices = pp.state_indices;
    q.idx_i64 = pp.idx_i64;
    q.status = status;
    if (gdn::launch_cp_prepare(q, stream) != cudaSuccess) return GDN_ERR_CUDA;

    gdn::StateLayout dense{};
    dense.dtype = GDN_DTYPE_F32;
    dense.s_v = gdn::kHead;
    dense.s_head = static_cast<int64_t>(gdn::kHead) * gdn::kHead;
    dense.s_row = dense.s_head * H;

    gdn::ChunkParams ta = cp;  // transfer pass over segments 0 .. P_i-2 of the segmented sequences
    ta.num_seqs = nA_max;
    ta.num_seqs_dev = q.counts;
    ta.seg = q.seg_a;
    ta.seq_order = q.order_a;
    ta.counter = q.counter_a;
    ta.chunk_offsets = nullptr;
    ta.initial_state = nullptr;
    ta.output_state = ws + c.trans;
    ta.state = dense;
    ta.state_indices = nullptr;
    ta.checkpoints = nullptr;
    ta.ckpt_n = 0;
    ta.intra_g = ta.intra_w = ta.intra_u = nullptr;
    const int64_t units_a = 2 * static_cast<int64_t>(nA_max) * H;
    if (gdn::launch_chunk_16bit(ta, tq, tk, tv, to, f16, true, static_cast<int>(units_a < sms ? units_a : sms),
                                stream) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (gdn::launch_cp_fixup(q, stream) != cudaSuccess) return GDN_ERR_CUDA;

    uint8_t* wsc = ws + c.prep;  // the segment pass: segments and whole sequences as one batch
    const int32_t nc = q.V_max;
    gdn::PrepareParams pc{};
    pc.cu_seqlens = q.cu_c;
    pc.cu_i64 = 0;
    pc.num_seqs = nc;
    pc.total_tokens = T;
    pc.max_seqlen = 0;
    pc.ckpt_n = n;
    pc.ckpt_cu_starts = q.ckpt_c;
    pc.ckpt_i64 = 1;
    pc.num_checkpoints = a.num_checkpoints;
    pc.status = status;
    pc.counter = reinterpret_cast<int32_t*>(wsc + c.wc.counter);
    pc.n_chunks = reinterpret_cast<int32_t*>(wsc + c.wc.n_chunks);
    pc.chunk_offsets = reinterpret_cast<int32_t*>(wsc + c.wc.chunk_offsets);
    pc.chunk_map = reinterpret_cast<int32_t*>(wsc + c.wc.chunk_map);
    pc.max_chunks = (T + gdn::kChunk - 1) / gdn::kChunk + nc;
    pc.seq_order = reinterpret_cast<int32_t*>(wsc + c.wc.seq_order);
    pc.pool_bitmap = reinterpret_cast<uint32_t*>(wsc + c.wc.pool_bitmap);
    pc.bitmap_words = 0;
    pc.keep_status = 1;
    if (gdn::launch_prepare(pc, stream) != cudaSuccess) return GDN_ERR_CUDA;
    gdn::ChunkParams sc = cp;
    sc.cu_seqlens = q.cu_c;
    sc.cu_i64 = 0;
    sc.num_seqs = nc;
    sc.num_seqs_dev = q.counts + 1;
    sc.initial_state = q.start;
    sc.output_state = q.start;
    sc.state = dense;
    sc.state_indices = q.vrow;
    sc.idx_i64 = 1;
    sc.split_state = 1;
    sc.initial_state2 = cp.initial_state;
    sc.output_state2 = cp.output_state;
    sc.state2 = sl;
    sc.ckpt_cu_starts = q.ckpt_c;
    sc.ckpt_i64 = 1;
    sc.counter = pc.counter;
    sc.chunk_offsets = pc.chunk_offsets;
    sc.seq_order = pc.seq_order;
    const int64_t units_c = static_cast<int64_t>(nc) * H;
    if (gdn::launch_chunk_16bit(sc, tq, tk, tv, to, f16, false, static_cast<int>(units_c < sms ? units_c : sms),
                                stream) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (gdn::launch_cp_final(q, stream) != cudaSuccess) return GDN_ERR_CUDA;
    return GDN_OK;
}

}  // namespace

extern "C" {

gdn_status gdn_decode_run(gdn_prefill_plan_t plan, const gdn_prefill_args* args, int32_t tokens_per_seq,
                          void* stream_ptr) {
    if (!plan || !args) return GDN_ERR_INVALID_ARG;
    const gdn_prefill_desc& d = plan->desc;
    const gdn_prefill_args& a = *args;
    const uint32_t f = d.flags;
    if (d.checkpoint_every_n_tokens != 0) return GDN_ERR_UNSUPPORTED;
    if (tokens_per_seq < 1 || tokens_per_seq > GDN_DECODE_MAX_TOKENS_PER_SEQ) return GDN_ERR_INVALID_ARG;
    const int32_t N = a.num_seqs;
    const int64_t T = a.total_tokens;
    if (N < 0 || N > d.max_num_seqs || T != static_cast<int64_t>(N) * tokens_per_seq || T > d.max_total_tokens)
        return GDN_ERR_INVALID_ARG;
    if (a.state_checkpoints || a.checkpoint_cu_starts) return GDN_ERR_INVALID_ARG;
    if (N == 0) return GDN_OK;
    if (!a.q || !a.k || !a.v || !a.output || !aligned(a.q, 16) || !aligned(a.k, 16) || !aligned(a.v, 16) ||
        !aligned(a.output, 16))
        return GDN_ERR_INVALID_ARG;
    if (((f & GDN_FLAG_HAS_G) && !a.g) || ((f & GDN_FLAG_HAS_BETA) && !a.beta)) return GDN_ERR_INVALID_ARG;
    if ((f & GDN_FLAG_HAS_INITIAL_STATE) && (!a.initial_state || !aligned(a.initial_state, 16)))
        return GDN_ERR_INVALID_ARG;
    if ((f & GDN_FLAG_OUTPUT_FINAL_STATE) && (!a.output_state || !aligned(a.output_state, 16)))
        return GDN_ERR_INVALID_ARG;
    if ((f & GDN_FLAG_HAS_STATE_INDICES) && (!a.state_indices || a.n_pool <= 0 || a.n_pool > d.max_pool_rows))
        return GDN_ERR_INVALID_ARG;
    gdn::StateLayout sl{};
    if (!make_state_layout(d.state_dtype, a.state_strides, (f & GDN_FLAG_HAS_STATE_INDICES) ? a.n_pool : N, plan->H,
                           &sl))
        return GDN_ERR_INVALID_ARG;
    // (sequence, head) units in 32 bits, with room for the kernel's look-ahead of a few grid strides
    const int64_t units = static_cast<int64_t>(N) * plan->H;
    if (units > 0x7fffffffLL - (1 << 20)) return GDN_ERR_UNSUPPORTED;
    gdn::DecodeParams p{};
    p.q = a.q;
    p.k = a.k;
    p.v = a.v;
    p.g = (f & GDN_FLAG_HAS_G) ? a.g : nullptr;
    p.beta = (f & GDN_FLAG_HAS_BETA) ? a.beta : nullptr;
    p.scale = (f & GDN_FLAG_HAS_SCALE) ? a.scale : 1.0f / std::sqrt(static_cast<float>(gdn::kHead));
    p.initial_state = (f & GDN_FLAG_HAS_INITIAL_STATE) ? a.initial_state : nullptr;
    p.state = sl;
    p.output_state = (f & GDN_FLAG_OUTPUT_FINAL_STATE) ? a.output_state : nullptr;
    p.state_indices = (f & GDN_FLAG_HAS_STATE_INDICES) ? a.state_indices : nullptr;
    p.idx_i64 = (f & GDN_FLAG_STATE_INDICES_I64) ? 1 : 0;
    p.n_pool = a.n_pool;
    p.output = a.output;
    p.status = a.device_status;
    p.N = N;
    p.H = plan->H;
    p.hq = d.num_q_heads;
    p.hk = d.num_k_heads;
    p.hv = d.num_v_heads;
    p.m = tokens_per_seq;
    p.l2norm = (f & GDN_FLAG_QK_L2NORM) ? 1 : 0;
    return gdn::launch_decode(p, d.qkv_dtype, static_cast<cudaStream_t>(stream_ptr)) == cudaSuccess
               ? GDN_OK
               : GDN_ERR_CUDA;
}

gdn_status gdn_prefill_run(gdn_prefill_plan_t plan, const gdn_prefill_args* args, void* workspace,
                           size_t workspace_bytes, void* stream) {
    return run_stages(plan, args, workspace, workspace_bytes, stream, kStagePrepare | kStageChunks);
}

gdn_status gdn_prefill_prepare(gdn_prefill_plan_t plan, const gdn_prefill_args* args, void* workspace,
                               size_t workspace_bytes, void* stream) {
    return run_stages(plan, args, workspace, workspace_bytes, stream, kStagePrepare);
}

gdn_status gdn_prefill_chunks(gdn_prefill_plan_t plan, const gdn_prefill_args* args, void* workspace,
                              size_t workspace_bytes, void* stream) {
    return run_stages(plan, args, workspace, workspace_bytes, stream, kStageChunks);
}

gdn_status gdn_prefill_read_status(gdn_prefill_plan_t plan, const void* workspace, const int32_t* device_status,
                                   void* stream_ptr, int32_t* bits) {
    if (!plan || !bits || (!workspace && !device_status)) return GDN_ERR_INVALID_ARG;
    const int32_t* src = device_status
                             ? device_status
                             : reinterpret_cast<const int32_t*>(static_cast<const uint8_t*>(workspace) + plan->ws.status);
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, src, sizeof(v), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GDN_ERR_CUDA;
    *bits = v;
    if (v == 0) return GDN_OK;
    return (v & GDN_DEVICE_ERR_TIMEOUT) ? GDN_ERR_DEVICE_TIMEOUT : GDN_ERR_DEVICE_INPUT;
}

const char* gdn_status_string(gdn_status s) {
    switch (s) {
        case GDN_OK: return "ok";
        case GDN_ERR_INVALID_ARG: return "invalid argument";
        case GDN_ERR_UNSUPPORTED: return "unsupported configuration";
        case GDN_ERR_CUDA: return "CUDA runtime error";
        case GDN_ERR_DEVICE_INPUT: return "device-checked input error";
        case GDN_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

}  // extern "C"
