// gemv_noalloc.cu -- gdn_gemv_bf16_noalloc: the decode projection for callers that cannot
// allocate device memory. The split-K partial sums go to a fixed buffer that the library itself
// holds (a file-scope __device__ array) instead of a caller workspace; everything else is the
// gdn_gemv_bf16 call unchanged.
#include <cstdint>
#include <mutex>

#include "gdn_decode.h"
#include "gdn_gemv.h"

namespace {

// The fixed split-K buffer: GDN_GEMV_NOALLOC_MAX_FLOATS fp32 values (4 MiB), present on every GPU
// that loads the library until the process exits. Host code must not pass this name to a kernel:
// on the host it only stands in for the symbol; its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) float g_gemv_scratch[GDN_GEMV_NOALLOC_MAX_FLOATS];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
float *g_scratch_ptr[kMaxDevices] = {};

// Device address of this device's buffer, looked up once per device with that device current.
int scratch_for_current_device(float **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_LAUNCH;
    std::lock_guard<std::mutex> guard(g_lock);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_gemv_scratch) != cudaSuccess || !p) return GDN_ERR_LAUNCH;
        g_scratch_ptr[dev] = static_cast<float *>(p);
    }
    *out = g_scratch_ptr[dev];
    return GDN_OK;
}

}  // namespace

extern "C" int gdn_gemv_bf16_noalloc(const gdn_gemv_args *args, gdn_stream_t stream)
{
    if (!args) return GDN_ERR_NULL;
    gdn_gemv_args a = *args;
    // the split count this call uses, resolved once so the size check and the launch agree
    if (a.splits == 0 && a.T > 0 && a.N > 0 && a.Kd > 0) a.splits = gdn_gemv_default_splits(a.T, a.N, a.Kd);
    a.workspace = nullptr;
    a.workspace_bytes = 0;
    const size_t need = a.T > 0 && a.N > 0 ? gdn_gemv_workspace_bytes(a.T, a.N, a.splits) : 0;
    if (need > 0) {   // more K ranges than one cluster holds
        if (need > sizeof(float) * (size_t)GDN_GEMV_NOALLOC_MAX_FLOATS) return GDN_ERR_SCRATCH;
        float *scratch = nullptr;
        const int rc = scratch_for_current_device(&scratch);
        if (rc != GDN_OK) return rc;
        a.workspace = scratch;
        a.workspace_bytes = sizeof(float) * (size_t)GDN_GEMV_NOALLOC_MAX_FLOATS;
    }
    // every partial sum the reduction reads is written earlier in the same call, so nothing in the
    // shared buffer needs clearing between calls
    return gdn_gemv_bf16(&a, stream);
}
