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
// loads the library until the process exits.  Its host-side name is only a
// stand-in for the device symbol, so the first call on each device looks up
// the device address with cudaGetSymbolAddress (with that device current)
// and caches it; make that first call before any stream capture.  Every call
// shares the one array and clears the part it uses on the caller's stream
// before the kernel, so calls that overlap on the GPU (different streams
// without ordering) race and must not be issued.
#include <cstring>
#include <mutex>

#include "csf_internal.cuh"

using namespace csfk;

namespace {

static __device__ __align__(256) unsigned char g_prepare_scratch[CSF_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices];

// Device address of g_prepare_scratch on the current device (set up once per
// device, with that device current).
csf_status static_scratch(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return CSF_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_prepare_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return CSF_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return CSF_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" csf_status csf_prepare_static(const uint8_t *dense, csf_stack *out, uint64_t exc_capacity, void *stream) {
    if (!dense || !out) return CSF_ERR_ARG;
    const csf_geometry &g = out->g;
    if (g.kind != CSF_NVFP4 && g.kind != CSF_MXFP4) return CSF_ERR_ARG;
    if (g.num_experts < 1 || g.rows < 1 || g.cols < 1) return CSF_ERR_ARG;
    const uint64_t rows = (uint64_t)g.num_experts * (uint64_t)g.rows;
    const uint64_t n = rows * (uint64_t)g.cols;
    if (rows >= (1ull << 31) || n >= (1ull << 40) || g.cols >= 65536) return CSF_ERR_UNSUPPORTED;
    if (!out->base || !out->offsets || !out->exc_index || !aligned16(out->offsets)) return CSF_ERR_ARG;
    if (g.kind == CSF_MXFP4 && (!out->escapes || !aligned16(out->escapes))) return CSF_ERR_ARG;
    if (exc_capacity > 0 && !out->exc_bytes) return CSF_ERR_ARG;
    const int32_t tr = prepare_tile_rows(g.kind, g.cols);
    const bool staged = prepare_stages_rows(g.kind, g.cols, dense);
    const size_t smem = prepare_smem_bytes(g.kind, g.cols, tr, staged);
    if (smem > 200 * 1024 || (uint64_t)tr * g.cols >= (1ull << 24)) return CSF_ERR_UNSUPPORTED;
    const uint64_t tiles = (rows + tr - 1) / tr;
    const uint64_t need = 16 + 8 * tiles;
    if (need > CSF_STATIC_SCRATCH_BYTES) return CSF_ERR_SIZE;   // stack too large for the built-in scratch

    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, dense) != cudaSuccess) {
        cudaGetLastError();
        return CSF_ERR_ARG;
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) return CSF_ERR_ARG;

    void *scratch = nullptr;
    csf_status st = static_scratch(&scratch);
    if (st != CSF_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(scratch, 0, need, s) != cudaSuccess) {   // ticket and status words start at zero
        cudaGetLastError();
        return CSF_ERR_CUDA;
    }
    PrepParams p;
    make_prep_params(p, dense, *out, exc_capacity, scratch, rows, n, staged);
    if (launch_prepare(p, smem, s) != cudaSuccess) {
        cudaGetLastError();
        return CSF_ERR_CUDA;
    }
    return CSF_OK;
}
