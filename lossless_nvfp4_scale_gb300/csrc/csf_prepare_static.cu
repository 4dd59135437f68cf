// csf_prepare_static: the GPU prepare for callers that cannot allocate device
// memory.  The pages describe nothing like it; it exists for users of this
// library who have no way to hand it a scratch buffer.
//
// Some callers cannot call cudaMalloc: a plugin loaded into a host process
// that owns all device memory through its own caching allocator, code that
// runs where an allocation would implicitly synchronise the device or
// invalidate a stream capture in progress, and code with a fixed device
// memory budget.  csf_prepare needs a small scratch buffer (one ticket
// counter plus one look-back status word per tile of rows); this entry point
// keeps that scratch in a file-scope device array instead.  The caller still
// passes the dense input and every output buffer.
//
// The array is CSF_STATIC_SCRATCH_BYTES (256 KiB) and exists on every GPU that
// loads the library, in every CUDA context the library's module is loaded
// into, until that context is destroyed.  Its host-side name is only a
// stand-in for the device symbol, so the first call in each context (normally
// once per device, with that device current) looks up the device address with
// cudaGetSymbolAddress and caches it under the context's unique id; make that
// first call before any stream capture.  A device reset destroys the context:
// the next call sees a new context id and looks the address up again rather
// than reuse a stale one.  Every call shares the one array and clears the part
// it uses on the caller's stream before the kernel, so calls that overlap on
// the GPU (different streams without ordering) race and must not be issued.
#include <cuda.h>

#include <cstring>
#include <mutex>

#include "csf_internal.cuh"

using namespace csfk;

namespace {

static __device__ __align__(256) unsigned char g_prepare_scratch[CSF_STATIC_SCRATCH_BYTES];

// Driver calls that name the current context, fetched through the runtime
// (no link against the driver library).
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

constexpr int kSlots = 64;
struct Slot {
    unsigned long long ctx_id;   // 0: empty
    void *ptr;
};

std::mutex g_mu;
Slot g_slots[kSlots];
int g_next = 0;
CtxGetCurrentFn g_get_current = nullptr;
CtxGetIdFn g_get_id = nullptr;

bool driver_calls() {
    if (g_get_current && g_get_id) return true;
    void *a = nullptr, *b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) != cudaSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) != cudaSuccess ||
        qa != cudaDriverEntryPointSuccess || qb != cudaDriverEntryPointSuccess || !a || !b) {
        cudaGetLastError();
        return false;
    }
    g_get_current = reinterpret_cast<CtxGetCurrentFn>(a);
    g_get_id = reinterpret_cast<CtxGetIdFn>(b);
    return true;
}

// Unique id of the context current on this thread; 0 when none is current.
bool current_context_id(unsigned long long *id) {
    CUcontext ctx = nullptr;
    if (g_get_current(&ctx) != CUDA_SUCCESS) return false;
    *id = 0;
    if (ctx == nullptr) return true;
    return g_get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_prepare_scratch in the current context: looked up once
// per context (with its device current) and cached under the context id.
csf_status static_scratch(void **out) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!driver_calls()) return CSF_ERR_CUDA;
    unsigned long long id = 0;
    if (!current_context_id(&id)) return CSF_ERR_CUDA;
    if (id != 0)
        for (const Slot &s : g_slots)
            if (s.ctx_id == id) {
                *out = s.ptr;
                return CSF_OK;
            }
    // Set-up: this runtime call also makes the device's primary context
    // current when no context was, so the id is read again afterwards.
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_prepare_scratch);
    if (e != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return CSF_ERR_CUDA;
    }
    if (!current_context_id(&id) || id == 0) return CSF_ERR_CUDA;
    g_slots[g_next] = Slot{id, p};
    g_next = (g_next + 1) % kSlots;
    *out = p;
    return CSF_OK;
}

}  // namespace

extern "C" csf_status csf_prepare_static(const uint8_t *dense, csf_stack *out, uint64_t exc_capacity, void *stream) {
    // Host-only checks first: a geometry the built-in scratch cannot hold is
    // refused before any CUDA call.
    PrepPlan plan;
    csf_status st = prepare_check(dense, out, exc_capacity, &plan);
    if (st != CSF_OK) return st;
    if (plan.scratch_bytes > CSF_STATIC_SCRATCH_BYTES) return CSF_ERR_SIZE;   // too large for the built-in scratch
    st = prepare_configure(dense, out->g, &plan);
    if (st != CSF_OK) return st;
    void *scratch = nullptr;
    st = static_scratch(&scratch);
    if (st != CSF_OK) return st;
    return prepare_enqueue(dense, *out, exc_capacity, scratch, plan, static_cast<cudaStream_t>(stream));
}
