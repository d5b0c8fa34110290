// pkv_decode_static: decode_paged for callers that cannot allocate device
// memory.  The scratch that pkv_decode takes from the caller's workspace comes
// from a fixed array compiled into this file instead; the call allocates
// nothing and otherwise enqueues the same kernels as pkv_decode.
#include <mutex>

#include "pkv_internal.h"

namespace {

// The library's own scratch: every GPU that loads libpkv holds it until the
// process exits.  Its contents persist between calls (they need no zeroing:
// every call writes each scratch entry it reads).
__device__ __align__(256) unsigned char g_static_scratch[PKV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices];  // device address of g_static_scratch, per device, from the last lookup

// Device address of the scratch array on `dev` (the current device).  It is
// looked up afresh on every call whose stream is not being captured (so a
// module reloaded after cudaDeviceReset is seen); a call under stream capture
// uses the address the last uncaptured call on that device found, and looks it
// up only if there is none yet.
int scratch_address(int dev, cudaStream_t stream, void** out)
{
    if (dev < 0 || dev >= kMaxDevices) return PKV_EDEVICE;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        cs = cudaStreamCaptureStatusActive;  // unknown: do not touch the module
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (cs == cudaStreamCaptureStatusNone || !g_scratch_addr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            return PKV_ECUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return PKV_OK;
}

bool aligned_to(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

}  // namespace

extern "C" int pkv_decode_static(pkv_pool* pool, const void* q, const void* k, const void* v, const void* q_norm_w,
                                 const void* k_norm_w, const int32_t* positions, const int32_t* table, int rows,
                                 int pages, void* out, void* stream)
{
    pkv::NvtxRange range("pkv_decode_static");
    if (!pool || !q || !k || !v || !q_norm_w || !k_norm_w || !positions || !out) return PKV_EINVAL;
    if (rows <= 0 || pages <= 0) return PKV_EINVAL;
    if (rows > (1 << 20) || (int64_t)rows * pages > INT32_MAX) return PKV_ERANGE;
    if (!aligned_to(q, 16) || !aligned_to(k, 16) || !aligned_to(v, 16) || !aligned_to(out, 8) ||
        !aligned_to(q_norm_w, 8) || !aligned_to(k_norm_w, 8) || !aligned_to(positions, 4) || !aligned_to(table, 4))
        return PKV_EINVAL;
    if (!table && (int64_t)rows * pages > pool->num_pages) return PKV_ERANGE;
    const pkv::Plan plan = pkv::make_plan(pool, rows, pages, 0);
    if (plan.total > (size_t)PKV_STATIC_SCRATCH_BYTES) return PKV_ERANGE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != pool->device) return PKV_EDEVICE;
    void* scratch = nullptr;
    const int rc = scratch_address(dev, static_cast<cudaStream_t>(stream), &scratch);
    if (rc != PKV_OK) return rc;

    const pkv::StepArgs a = {q, k, v, q_norm_w, k_norm_w, nullptr, nullptr, nullptr, positions, table,
                             0, rows, pages, rows, out, static_cast<char*>(scratch)};
    if (pkv::check_enabled()) {  // the same debugging pre-check as pkv_decode (host memory only)
        const int pc = pkv::host_precheck(pool, a, static_cast<cudaStream_t>(stream));
        if (pc != PKV_OK) return pc;
    }
    return pkv::enqueue(pool, a, plan, static_cast<cudaStream_t>(stream));
}
