// gemv_noalloc.cu -- gdn_gemv_bf16_noalloc: the decode projection for callers that cannot
// allocate device memory. The split-K partial sums go to a fixed buffer that the library itself
// holds (a file-scope __device__ array) instead of a caller workspace; everything else is the
// gdn_gemv_bf16 call unchanged.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "gdn_decode.h"
#include "gdn_gemv.h"
#include "gemv_internal.h"

namespace {

// The fixed split-K buffer: GDN_GEMV_NOALLOC_MAX_FLOATS fp32 values (4 MiB), present on every GPU
// that loads the library until the process exits. Host code must not pass this name to a kernel:
// on the host it only stands in for the symbol; its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) float g_gemv_scratch[GDN_GEMV_NOALLOC_MAX_FLOATS];

constexpr int kMaxDevices = 64;
std::mutex g_lock;

// One remembered address per device, tagged with the id of the context it was looked up in
// (0: no id available, the address is then kept for the device).
struct ScratchEntry {
    float *ptr;
    unsigned long long ctx_id;
};
ScratchEntry g_scratch[kMaxDevices] = {};

// The current context's unique id (cuCtxGetId, CUDA 12+), through the runtime's driver entry
// points so that the library needs no link against libcuda; 0 when unavailable.
unsigned long long current_context_id()
{
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static bool looked_up = false;
    if (!looked_up) {   // under g_lock
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
        cudaGetLastError();
        looked_up = true;
    }
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the current device's buffer, looked up once per context with the device
// current (the runtime's cudaSetDevice / cudaFree(0) make the primary context current first).
int scratch_for_current_device(float **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_LAUNCH;
    std::lock_guard<std::mutex> guard(g_lock);
    void *p = nullptr;
    ScratchEntry &e = g_scratch[dev];
    if (e.ptr) {
        const unsigned long long id = current_context_id();
        if (id == e.ctx_id) {
            *out = e.ptr;
            return GDN_OK;
        }
    }
    if (cudaGetSymbolAddress(&p, g_gemv_scratch) != cudaSuccess || !p) return GDN_ERR_LAUNCH;
    e.ptr = static_cast<float *>(p);
    e.ctx_id = current_context_id();   // after the lookup, which makes the primary context current
    *out = e.ptr;
    return GDN_OK;
}

}  // namespace

extern "C" int gdn_gemv_bf16_noalloc(const gdn_gemv_args *args, gdn_stream_t stream)
{
    if (!args) return GDN_ERR_NULL;
    gdn_gemv_args a = *args;
    // The argument checks of gdn_gemv_bf16 come first, with a stand-in workspace that satisfies
    // them (never dereferenced: nothing is launched with it), so invalid calls get the same codes.
    a.workspace = reinterpret_cast<float *>(static_cast<uintptr_t>(256));
    a.workspace_bytes = SIZE_MAX;
    int splits = 0;
    const int rc_check = gdn::gemv_check(&a, &splits);
    if (rc_check != GDN_OK || splits == 0) return rc_check;
    a.splits = splits;   // resolved once, so the size check and the launch agree
    a.workspace = nullptr;
    a.workspace_bytes = 0;
    const size_t need = gdn_gemv_workspace_bytes(a.T, a.N, splits);
    if (need > 0) {   // more K ranges than one cluster holds
        if (need > sizeof(float) * (size_t)GDN_GEMV_NOALLOC_MAX_FLOATS) return GDN_ERR_SCRATCH;
        float *scratch = nullptr;
        const int rc = scratch_for_current_device(&scratch);
        if (rc != GDN_OK) return rc;
        a.workspace = scratch;
        a.workspace_bytes = sizeof(float) * (size_t)GDN_GEMV_NOALLOC_MAX_FLOATS;
    }
    // every partial sum the reduction reads is written earlier in the same call (NaN by a range
    // that gave up a bounded wait), so nothing in the shared buffer needs clearing between calls
    return gdn_gemv_bf16(&a, stream);
}
