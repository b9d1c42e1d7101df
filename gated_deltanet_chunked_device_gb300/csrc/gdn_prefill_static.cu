// gdn_prefill_static.cu -- a prefill entry point that allocates nothing.
//
// Some callers cannot allocate device memory at the moment they run the
// prefill: code that runs inside another library's allocator hook, inside a
// memory-pool callback, or in a process whose allocations are owned by a
// framework that forbids side allocations.  They can still hand over their
// tensors, but not a workspace.  For them, gdn_prefill_run_static runs the
// same prepare and chunk kernels as gdn_prefill_run with the workspace taken
// from a fixed-size array that lives in this file's device globals (every GPU
// that loads the library holds it until the process exits).
//
// Everything the kernels need zeroed in the workspace (status word, work
// counter, pool bitmap) is reset by the prepare kernel at the start of every
// call, so the array's leftover contents from the previous call do no harm.
// All calls share the one array: two calls whose kernels overlap on the GPU
// (different streams, or different host threads without ordering) race on it.
#include <cstdint>
#include <mutex>

#include "gdn_internal.cuh"

namespace {

static __device__ __align__(256) uint8_t g_static_workspace[GDN_PREFILL_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
struct CachedAddress {
    unsigned long long context_id;  // the context the address belongs to (0: none yet)
    void* addr;
};
CachedAddress g_static_workspace_addr[kMaxDevices] = {};
std::mutex g_static_lock;

// The driver's cuCtxGetCurrent and cuCtxGetId, through the runtime's entry-point query (no link-time
// dependency on the driver library).  A context id is unique for the life of the process, so a context that
// a device reset re-creates gets a fresh look-up of the array's address.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the array on the current device (host code only sees a stand-in symbol, never the device
// address), looked up once per device and context.
gdn_status static_workspace(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
    std::lock_guard<std::mutex> guard(g_static_lock);
    CachedAddress& c = g_static_workspace_addr[dev];
    const unsigned long long id = current_context_id();
    if (!c.addr || id == 0 || id != c.context_id) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_workspace) != cudaSuccess || !ptr) return GDN_ERR_CUDA;
        c.addr = ptr;
        c.context_id = current_context_id();  // after the look-up, which makes the device's context current
    }
    *out = c.addr;
    return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_prefill_run_static(gdn_prefill_plan_t plan, const gdn_prefill_args* args, void* stream) {
    if (!plan || !args) return GDN_ERR_INVALID_ARG;
    if (gdn::plan_workspace_bytes(plan) > GDN_PREFILL_STATIC_WORKSPACE_BYTES) return GDN_ERR_UNSUPPORTED;
    void* ws = nullptr;
    const gdn_status st = static_workspace(&ws);
    if (st != GDN_OK) return st;
    return gdn_prefill_run(plan, args, ws, GDN_PREFILL_STATIC_WORKSPACE_BYTES, stream);
}
