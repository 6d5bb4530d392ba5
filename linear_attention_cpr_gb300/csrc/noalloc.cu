// noalloc.cu — cpr_gdn_prefill_noalloc: the prefill entry point for callers that cannot
// allocate device memory.
//
// Some callers are not allowed to call cudaMalloc (or any allocating routine) at the
// point where they run a layer: serving runtimes that reserve the whole device memory
// for their own pool at start-up and hand out only input/output buffers, latency-bound
// loops that cannot afford the implicit device synchronisation an allocation may cause,
// and plain-C hosts that have no device allocator of their own.  cpr_gdn_prefill needs a
// workspace of cpr_gdn_prefill_workspace_size() bytes from its caller; this variant uses
// a scratch array that the library itself owns instead.
//
// The scratch is a file-scope static __device__ array of CPR_GDN_NOALLOC_SCRATCH_BYTES
// (16 MiB).  Every GPU on which this library's device code is loaded holds that memory
// until the process exits.  Host code cannot use the array's name as a device address
// (on the host it names a stand-in object), so on the first call on each device, with
// that device current, the entry point asks the runtime for the array's device address
// with cudaGetSymbolAddress, checks the result and remembers it for that device.
// Because that first call may load the library's device code, make it before any stream
// capture begins.  cudaDeviceReset on a device unloads the module and so invalidates the
// remembered address: a process that resets a device must not call these entry points
// on it afterwards.
//
// All calls share the one array and it keeps the last call's contents.  Nothing in it
// has to start at zero: every call's first kernel rewrites the status word and the chunk
// index, and each later kernel reads only what an earlier kernel of the same call wrote.
// Calls that can overlap on the GPU (different streams, or different host threads)
// race on the array and must be serialised by the caller.
//
// The prefill's device-side checks (bad cu_seqlens, boundary capacity, a bounded wait
// that gave up) set bits in a status word at the start of the scratch;
// cpr_gdn_prefill_noalloc_status reads it back, again without allocating.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/cpr_gdn.h"

namespace {

static __device__ __align__(256) unsigned char g_prefill_scratch[CPR_GDN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_prefill_scratch on the current device (looked up once per device).
cudaError_t scratch_address(void** out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_prefill_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" int32_t cpr_gdn_prefill_noalloc_status(uint32_t* status_out, void* stream)
{
    if (!status_out) return CPR_ERR_INVALID_ARG;
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return CPR_ERR_CUDA;
    return cpr_gdn_device_status(scratch, status_out, stream);
}

extern "C" int32_t cpr_gdn_prefill_noalloc(const void* q, const void* k, const void* v, const float* g,
                                           const float* beta, const int32_t* cu_seqlens, int32_t n_seqs,
                                           int64_t total_tokens, int32_t H, int32_t dk, int32_t dv, int32_t C,
                                           int32_t dtype, const float* state_in, void* out, float* state_out,
                                           float* boundary_states, int64_t boundary_capacity, void* stream)
{
    if (n_seqs < 0 || total_tokens < 0 || H <= 0 || dk <= 0 || dv <= 0 || C <= 0) return CPR_ERR_INVALID_ARG;
    if (!cpr_gdn_supported(dk, dv, C, dtype)) return CPR_ERR_UNSUPPORTED_SHAPE;
    const size_t need = cpr_gdn_prefill_workspace_size(total_tokens, n_seqs, H, dk, dv, C);
    if (need == 0) return CPR_ERR_INVALID_ARG;
    if (need > (size_t)CPR_GDN_NOALLOC_SCRATCH_BYTES) return CPR_ERR_WORKSPACE;  // beyond the static scratch
    if (n_seqs == 0) return CPR_OK;
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return CPR_ERR_CUDA;
    return cpr_gdn_prefill(q, k, v, g, beta, cu_seqlens, n_seqs, total_tokens, H, dk, dv, C, dtype, state_in, out,
                           state_out, boundary_states, boundary_capacity, scratch,
                           (size_t)CPR_GDN_NOALLOC_SCRATCH_BYTES, stream);
}
