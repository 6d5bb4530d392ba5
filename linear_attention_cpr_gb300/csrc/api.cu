// api.cu — the C ABI declared in include/cpr_gdn.h: argument checks, shape dispatch
// and launches.  No allocation, no host synchronisation (except
// cpr_gdn_device_status, which reads the status word back).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"

using namespace cpr;

namespace {

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }
// H value heads over Hk query/key heads: Hk divides H.
bool heads_ok(int32_t H, int32_t Hk) { return Hk > 0 && Hk <= H && H % Hk == 0; }

bool shape_built(int32_t dk, int32_t dv, int32_t C)
{
#define CPR_SHAPE_MATCH(DK, DV, CC) \
    if (dk == DK && dv == DV && C == CC) return true;
    CPR_FOR_EACH_SHAPE(CPR_SHAPE_MATCH)
#undef CPR_SHAPE_MATCH
    return false;
}

bool dtype_ok(int32_t dtype) { return dtype == CPR_DTYPE_BF16 || dtype == CPR_DTYPE_F32; }

int32_t from_cuda(cudaError_t e) { return e == cudaSuccess ? CPR_OK : CPR_ERR_CUDA; }

// Timeout-test hook (cpr_gdn_set_wait_test): extra publications the intra-chunk items
// wait for, and their wait limit (0: the default).
uint32_t g_wait_extra = 0;
uint64_t g_wait_limit_ns = 0;

constexpr int kMaxProfileEvents = 8;
cudaEvent_t g_profile_events[kMaxProfileEvents] = {};
int g_profile_n = 0;

}  // namespace

EncodeTiledFn cpr::tensor_map_encoder()
{
    static const EncodeTiledFn fn = [] {  // (thread-safe initialisation of a static)
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        const bool found =
            cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess;
        return found ? reinterpret_cast<EncodeTiledFn>(p) : static_cast<EncodeTiledFn>(nullptr);
    }();
    return fn;
}

cudaEvent_t cpr::profile_event(int i) { return (i >= 0 && i < g_profile_n) ? g_profile_events[i] : nullptr; }

namespace {
// SM count of the current device, cached per device (0 on error).
int num_sms()
{
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < 64 && cached[dev] > 0) return cached[dev];
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < 64) cached[dev] = sms;
    return sms;
}
}  // namespace

extern "C" {

int cpr_gdn_supported(int32_t dk, int32_t dv, int32_t C, int32_t dtype)
{
    return (dtype_ok(dtype) && shape_built(dk, dv, C)) ? 1 : 0;
}

int32_t cpr_gdn_version(void) { return 2; }

const char* cpr_gdn_strerror(int32_t code)
{
    switch (code) {
        case CPR_OK: return "ok";
        case CPR_ERR_INVALID_ARG: return "invalid argument";
        case CPR_ERR_UNSUPPORTED_SHAPE: return "unsupported (dk, dv, C) or dtype";
        case CPR_ERR_MISALIGNED: return "misaligned pointer";
        case CPR_ERR_WORKSPACE: return "workspace missing or too small";
        case CPR_ERR_CUDA: return "CUDA launch or runtime error";
        default: return "unknown error";
    }
}

int64_t cpr_gdn_num_chunks(const int32_t* cu_seqlens_host, int32_t n_seqs, int32_t C)
{
    if (!cu_seqlens_host || n_seqs < 0 || C <= 0 || cu_seqlens_host[0] != 0) return CPR_ERR_INVALID_ARG;
    int64_t total = 0;
    for (int32_t n = 0; n < n_seqs; ++n) {
        const int64_t L = (int64_t)cu_seqlens_host[n + 1] - cu_seqlens_host[n];
        if (L < 0) return CPR_ERR_INVALID_ARG;
        total += (L + C - 1) / C;
    }
    return total;
}

size_t cpr_gdn_prefill_workspace_size(int64_t total_tokens, int32_t n_seqs, int32_t H, int32_t dk, int32_t dv,
                                      int32_t C)
{
    if (total_tokens < 0 || n_seqs < 0 || H <= 0 || dk <= 0 || dv <= 0 || C <= 0) return 0;
    return PrefillLayout(total_tokens, n_seqs, H, dk, dv, C).total;
}

size_t cpr_gdn_backward_workspace_size(int64_t total_tokens, int32_t n_seqs, int32_t H, int32_t dk, int32_t dv,
                                       int32_t C)
{
    if (total_tokens < 0 || n_seqs < 0 || H <= 0 || dk <= 0 || dv <= 0 || C <= 0) return 0;
    return BackwardLayout(total_tokens, n_seqs, H, dk, dv, C).total;
}

int cpr_gdn_backward_supported(int32_t dk, int32_t dv, int32_t C, int32_t dtype)
{
    if (!dtype_ok(dtype) || !shape_built(dk, dv, C)) return 0;
    bool fits = false;
#define CPR_FITS(DK, DV, CC)                                                                        \
    if (dk == DK && dv == DV && C == CC)                                                             \
        fits = (dtype == CPR_DTYPE_BF16) ? backward_fits<DK, DV, CC, __nv_bfloat16>()                \
                                         : backward_fits<DK, DV, CC, float>();
    CPR_FOR_EACH_SHAPE(CPR_FITS)
#undef CPR_FITS
    return fits ? 1 : 0;
}

int32_t cpr_gdn_backward(const void* q, const void* k, const void* v, const float* g, const float* beta,
                         const int32_t* cu_seqlens, int32_t n_seqs, int64_t total_tokens, int32_t H, int32_t dk,
                         int32_t dv, int32_t C, int32_t dtype, const float* boundary_states,
                         int64_t boundary_capacity, const void* d_out, const float* d_state_out, float* dq,
                         float* dk_out, float* dv_out, float* dg, float* dbeta, float* d_state_in, void* workspace,
                         size_t workspace_bytes, void* stream)
{
    if (n_seqs < 0 || total_tokens < 0 || total_tokens > 0x7fffffffLL || H <= 0 || H > 65535 || !dtype_ok(dtype) ||
        boundary_capacity < 0)
        return CPR_ERR_INVALID_ARG;
    if (!shape_built(dk, dv, C) || !cpr_gdn_backward_supported(dk, dv, C, dtype)) return CPR_ERR_UNSUPPORTED_SHAPE;
    if (n_seqs == 0) return CPR_OK;
    if (!cu_seqlens || !workspace) return CPR_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !g || !beta || !d_out || !boundary_states || !dq || !dk_out ||
                             !dv_out || !dg || !dbeta))
        return CPR_ERR_INVALID_ARG;
    const BackwardLayout lay(total_tokens, n_seqs, H, dk, dv, C);
    if (workspace_bytes < lay.total) return CPR_ERR_WORKSPACE;
    const void* a16[] = {q, k, v, d_out, boundary_states, d_state_out, dq, dk_out, dv_out, d_state_in, workspace};
    for (const void* p : a16)
        if (p && !aligned(p, 16)) return CPR_ERR_MISALIGNED;
    const void* a4[] = {g, beta, cu_seqlens, dg, dbeta};
    for (const void* p : a4)
        if (p && !aligned(p, 4)) return CPR_ERR_MISALIGNED;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    BackwardArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.g = g;
    a.beta = beta;
    a.cu_seqlens = cu_seqlens;
    a.n_seqs = n_seqs;
    a.total_tokens = total_tokens;
    a.H = H;
    a.boundary = boundary_states;
    a.boundary_capacity = boundary_states ? boundary_capacity : 0;
    a.d_out = d_out;
    a.d_state_out = d_state_out;
    a.dq = dq;
    a.dk = dk_out;
    a.dv = dv_out;
    a.dg = dg;
    a.dbeta = dbeta;
    a.d_state_in = d_state_in;
    a.status = reinterpret_cast<uint32_t*>(ws);
    a.ready = reinterpret_cast<uint32_t*>(ws + lay.ready);
    a.cu_chunks = reinterpret_cast<int32_t*>(ws + lay.cu_chunks);
    a.mt = ws + lay.mt;
    a.cb = reinterpret_cast<float*>(ws + lay.cb);
    a.d_end = reinterpret_cast<float*>(ws + lay.d_end);
    a.max_chunks = max_chunks_bound(total_tokens, n_seqs, C);
    a.num_sms = num_sms();
    a.wait_extra = g_wait_extra;
    a.wait_limit_ns = g_wait_limit_ns;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaErrorInvalidValue;
#define CPR_DISPATCH(DK, DV, CC)                                                                   \
    if (dk == DK && dv == DV && C == CC)                                                           \
        e = (dtype == CPR_DTYPE_BF16) ? launch_backward<DK, DV, CC, __nv_bfloat16>(a, s)            \
                                      : launch_backward<DK, DV, CC, float>(a, s);
    CPR_FOR_EACH_SHAPE(CPR_DISPATCH)
#undef CPR_DISPATCH
    return from_cuda(e);
}

size_t cpr_gdn_decode_workspace_size(int32_t B, int32_t H, int32_t dk, int32_t dv, int32_t C)
{
    if (B < 0 || H <= 0 || dk <= 0 || dv <= 0 || C <= 0) return 0;
    return decode_workspace_bytes(B);
}

int32_t cpr_gdn_prefill_grouped(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                const int32_t* cu_seqlens, int32_t n_seqs, int64_t total_tokens, int32_t H,
                                int32_t Hk, uint32_t flags, int32_t dk, int32_t dv, int32_t C, int32_t dtype,
                                const float* state_in,
                                void* out, float* state_out, float* boundary_states, int64_t boundary_capacity,
                                void* workspace, size_t workspace_bytes, void* stream)
{
    if (n_seqs < 0 || total_tokens < 0 || total_tokens > 0x7fffffffLL || H <= 0 || H > 65535 || !dtype_ok(dtype) ||
        boundary_capacity < 0 || !heads_ok(H, Hk) || (flags & ~CPR_QK_L2NORM))
        return CPR_ERR_INVALID_ARG;
    if (!shape_built(dk, dv, C)) return CPR_ERR_UNSUPPORTED_SHAPE;
    if (n_seqs == 0) return CPR_OK;
    if (!cu_seqlens || !state_out || !workspace) return CPR_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !g || !beta || !out || !boundary_states)) return CPR_ERR_INVALID_ARG;
    const PrefillLayout lay(total_tokens, n_seqs, H, dk, dv, C);
    if (workspace_bytes < lay.total) return CPR_ERR_WORKSPACE;
    const void* a16[] = {q, k, v, out, state_out, boundary_states, workspace, state_in};
    for (const void* p : a16)
        if (p && !aligned(p, 16)) return CPR_ERR_MISALIGNED;
    const void* a4[] = {g, beta, cu_seqlens};
    for (const void* p : a4)
        if (p && !aligned(p, 4)) return CPR_ERR_MISALIGNED;

    unsigned char* ws = static_cast<unsigned char*>(workspace);
    PrefillArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.g = g;
    a.beta = beta;
    a.cu_seqlens = cu_seqlens;
    a.n_seqs = n_seqs;
    a.total_tokens = total_tokens;
    a.H = H;
    a.Hk = Hk;
    a.qk_norm = (flags & CPR_QK_L2NORM) ? 1 : 0;
    a.state_in = state_in;
    a.out = out;
    a.state_out = state_out;
    a.boundary = boundary_states;
    a.boundary_capacity = boundary_states ? boundary_capacity : 0;
    a.ws = ws;
    a.status = reinterpret_cast<uint32_t*>(ws);
    a.cu_chunks = reinterpret_cast<int32_t*>(ws + lay.cu_chunks);
    a.mt = ws + lay.mt;
    a.bt = reinterpret_cast<float*>(ws + lay.bt);
    a.ready = reinterpret_cast<uint32_t*>(ws + lay.ready);
    a.num_sms = num_sms();
    if (a.num_sms <= 0) return CPR_ERR_CUDA;
    a.max_chunks = max_chunks_bound(total_tokens, n_seqs, C);
    a.wait_extra = g_wait_extra;
    a.wait_limit_ns = g_wait_limit_ns;
    if (!boundary_states) {
        // boundary states are also the chain's hand-off to the intra-chunk kernel
        return CPR_ERR_INVALID_ARG;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaErrorInvalidValue;
#define CPR_DISPATCH(DK, DV, CC)                                                                            \
    if (dk == DK && dv == DV && C == CC)                                                                    \
        e = (dtype == CPR_DTYPE_BF16) ? launch_prefill<DK, DV, CC, __nv_bfloat16>(a, s)                      \
                                      : launch_prefill<DK, DV, CC, float>(a, s);
    CPR_FOR_EACH_SHAPE(CPR_DISPATCH)
#undef CPR_DISPATCH
    return from_cuda(e);
}

int32_t cpr_gdn_prefill_continue_grouped(const void* q, const void* k, const void* v, const float* g,
                                         const float* beta, const int32_t* cu_seqlens, int32_t n_seqs,
                                         int64_t total_tokens, int32_t H, int32_t Hk, uint32_t flags, int32_t dk,
                                         int32_t dv, int32_t C, int32_t dtype, const int32_t* pos0, float* state,
                                         const cpr_gdn_ring* ring,
                                         void* out, float* boundary_states, int64_t boundary_capacity, void* workspace,
                                         size_t workspace_bytes, void* stream)
{
    if (n_seqs < 0 || total_tokens < 0 || total_tokens > 0x7fffffffLL || H <= 0 || H > 65535 || !dtype_ok(dtype) ||
        boundary_capacity < 0 || !heads_ok(H, Hk) || (flags & ~CPR_QK_L2NORM))
        return CPR_ERR_INVALID_ARG;
    if (!shape_built(dk, dv, C)) return CPR_ERR_UNSUPPORTED_SHAPE;
    if (n_seqs == 0) return CPR_OK;
    if (!cu_seqlens || !pos0 || !state || !workspace || !boundary_states || !ring || !ring->S_b || !ring->k ||
        !ring->v || !ring->g || !ring->beta)
        return CPR_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !g || !beta || !out)) return CPR_ERR_INVALID_ARG;
    const PrefillLayout lay(total_tokens, n_seqs, H, dk, dv, C);
    if (workspace_bytes < lay.total) return CPR_ERR_WORKSPACE;
    const void* a16[] = {q, k, v, out, state, boundary_states, workspace, ring->S_b, ring->k, ring->v};
    for (const void* p : a16)
        if (p && !aligned(p, 16)) return CPR_ERR_MISALIGNED;
    const void* a4[] = {g, beta, cu_seqlens, pos0, ring->g, ring->beta};
    for (const void* p : a4)
        if (p && !aligned(p, 4)) return CPR_ERR_MISALIGNED;

    unsigned char* ws = static_cast<unsigned char*>(workspace);
    PrefillArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.g = g;
    a.beta = beta;
    a.cu_seqlens = cu_seqlens;
    a.skip = reinterpret_cast<const int32_t*>(ws + lay.skip);
    a.n_seqs = n_seqs;
    a.total_tokens = total_tokens;
    a.H = H;
    a.Hk = Hk;
    a.qk_norm = (flags & CPR_QK_L2NORM) ? 1 : 0;
    a.state_in = state;
    a.out = out;
    a.state_out = state;
    a.boundary = boundary_states;
    a.boundary_capacity = boundary_capacity;
    a.ws = ws;
    a.status = reinterpret_cast<uint32_t*>(ws);
    a.cu_chunks = reinterpret_cast<int32_t*>(ws + lay.cu_chunks);
    a.mt = ws + lay.mt;
    a.bt = reinterpret_cast<float*>(ws + lay.bt);
    a.ready = reinterpret_cast<uint32_t*>(ws + lay.ready);
    a.num_sms = num_sms();
    if (a.num_sms <= 0) return CPR_ERR_CUDA;
    a.max_chunks = max_chunks_bound(total_tokens, n_seqs, C);
    a.wait_extra = g_wait_extra;
    a.wait_limit_ns = g_wait_limit_ns;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaErrorInvalidValue;
#define CPR_DISPATCH(DK, DV, CC)                                                                             \
    if (dk == DK && dv == DV && C == CC)                                                                     \
        e = (dtype == CPR_DTYPE_BF16) ? launch_prefill_continue<DK, DV, CC, __nv_bfloat16>(a, pos0, state, *ring, s) \
                                      : launch_prefill_continue<DK, DV, CC, float>(a, pos0, state, *ring, s);
    CPR_FOR_EACH_SHAPE(CPR_DISPATCH)
#undef CPR_DISPATCH
    return from_cuda(e);
}

int32_t cpr_gdn_ring_from_prefill_grouped(const void* k, const void* v, const float* g, const float* beta,
                                          const int32_t* cu_seqlens, int32_t n_seqs, int64_t total_tokens, int32_t H,
                                          int32_t Hk, int32_t dk, int32_t dv, int32_t C, int32_t dtype,
                                          const float* boundary_states, const float* state_out,
                                          const cpr_gdn_ring* ring, void* stream)
{
    if (n_seqs < 0 || total_tokens < 0 || total_tokens > 0x7fffffffLL || H <= 0 || H > 65535 || !dtype_ok(dtype) ||
        !heads_ok(H, Hk))
        return CPR_ERR_INVALID_ARG;
    if (!shape_built(dk, dv, C)) return CPR_ERR_UNSUPPORTED_SHAPE;
    if (n_seqs == 0) return CPR_OK;
    if (!ring || !ring->S_b || !ring->k || !ring->v || !ring->g || !ring->beta || !cu_seqlens || !state_out)
        return CPR_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!boundary_states || !k || !v || !g || !beta)) return CPR_ERR_INVALID_ARG;
    const void* a16[] = {k, v, boundary_states, state_out, ring->S_b, ring->k, ring->v};
    for (const void* p : a16)
        if (p && !aligned(p, 16)) return CPR_ERR_MISALIGNED;
    const void* a4[] = {g, beta, cu_seqlens, ring->g, ring->beta};
    for (const void* p : a4)
        if (p && !aligned(p, 4)) return CPR_ERR_MISALIGNED;
    RingArgs a{};
    a.k = k;
    a.v = v;
    a.g = g;
    a.beta = beta;
    a.cu_seqlens = cu_seqlens;
    a.n_seqs = n_seqs;
    a.total_tokens = total_tokens;
    a.H = H;
    a.Hk = Hk;
    a.boundary = boundary_states;
    a.state_out = state_out;
    a.ring = *ring;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaErrorInvalidValue;
#define CPR_DISPATCH(DK, DV, CC)                                                                           \
    if (dk == DK && dv == DV && C == CC)                                                                   \
        e = (dtype == CPR_DTYPE_BF16) ? launch_ring_from_prefill<DK, DV, CC, __nv_bfloat16>(a, s)           \
                                      : launch_ring_from_prefill<DK, DV, CC, float>(a, s);
    CPR_FOR_EACH_SHAPE(CPR_DISPATCH)
#undef CPR_DISPATCH
    return from_cuda(e);
}

int32_t cpr_gdn_decode_grouped(const void* q, const void* k, const void* v, const float* g, const float* beta,
                               float* state, const cpr_gdn_ring* ring, const int32_t* pos, int32_t B, int32_t H,
                               int32_t Hk, uint32_t flags, int32_t dk, int32_t dv, int32_t C, int32_t dtype, void* out,
                               void* workspace, size_t workspace_bytes, void* stream)
{
    if (B < 0 || H <= 0 || H > 65535 || !dtype_ok(dtype) || !heads_ok(H, Hk) || (flags & ~CPR_QK_L2NORM))
        return CPR_ERR_INVALID_ARG;
    if (!shape_built(dk, dv, C)) return CPR_ERR_UNSUPPORTED_SHAPE;
    if (B == 0) return CPR_OK;
    if (!q || !k || !v || !g || !beta || !state || !ring || !pos || !out || !ring->S_b || !ring->k || !ring->v ||
        !ring->g || !ring->beta)
        return CPR_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < decode_workspace_bytes(B)) return CPR_ERR_WORKSPACE;
    const void* a16[] = {q, k, v, out, state, ring->S_b, ring->k, ring->v, workspace};
    for (const void* p : a16)
        if (!aligned(p, 16)) return CPR_ERR_MISALIGNED;
    const void* a4[] = {g, beta, pos, ring->g, ring->beta};
    for (const void* p : a4)
        if (!aligned(p, 4)) return CPR_ERR_MISALIGNED;
    DecodeArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.g = g;
    a.beta = beta;
    a.state = state;
    a.ring = *ring;
    a.pos = pos;
    a.B = B;
    a.H = H;
    a.Hk = Hk;
    a.qk_norm = (flags & CPR_QK_L2NORM) ? 1 : 0;
    a.out = out;
    a.status = static_cast<uint32_t*>(workspace);
    a.num_sms = num_sms();
    if (a.num_sms <= 0) return CPR_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaErrorInvalidValue;
#define CPR_DISPATCH(DK, DV, CC)                                                                  \
    if (dk == DK && dv == DV && C == CC)                                                          \
        e = (dtype == CPR_DTYPE_BF16) ? launch_decode<DK, DV, CC, __nv_bfloat16>(a, s)             \
                                      : launch_decode<DK, DV, CC, float>(a, s);
    CPR_FOR_EACH_SHAPE(CPR_DISPATCH)
#undef CPR_DISPATCH
    return from_cuda(e);
}

int32_t cpr_gdn_set_profile_events(void* const* events, int32_t n_events)
{
    if (!events) {
        g_profile_n = 0;
        return CPR_OK;
    }
    if (n_events < 4 || n_events > kMaxProfileEvents) return CPR_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n_events; ++i) {
        if (!events[i]) return CPR_ERR_INVALID_ARG;
        g_profile_events[i] = static_cast<cudaEvent_t>(events[i]);
    }
    g_profile_n = n_events;
    return CPR_OK;
}

int32_t cpr_gdn_set_wait_test(uint32_t extra_publications, uint64_t limit_ns)
{
    g_wait_extra = extra_publications;
    g_wait_limit_ns = limit_ns;
    return CPR_OK;
}

int32_t cpr_gdn_device_status(const void* workspace, uint32_t* status_out, void* stream)
{
    if (!workspace || !status_out) return CPR_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return CPR_ERR_CUDA;
    *status_out = v;
    return CPR_OK;
}

// The entry points with one query/key head per value head.
int32_t cpr_gdn_prefill(const void* q, const void* k, const void* v, const float* g, const float* beta,
                        const int32_t* cu_seqlens, int32_t n_seqs, int64_t total_tokens, int32_t H, int32_t dk,
                        int32_t dv, int32_t C, int32_t dtype, const float* state_in, void* out, float* state_out,
                        float* boundary_states, int64_t boundary_capacity, void* workspace,
                        size_t workspace_bytes, void* stream)
{
    return cpr_gdn_prefill_grouped(q, k, v, g, beta, cu_seqlens, n_seqs, total_tokens, H, H, 0u, dk, dv, C, dtype,
                                   state_in, out, state_out, boundary_states, boundary_capacity, workspace,
                                   workspace_bytes, stream);
}

int32_t cpr_gdn_prefill_continue(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                 const int32_t* cu_seqlens, int32_t n_seqs, int64_t total_tokens, int32_t H,
                                 int32_t dk, int32_t dv, int32_t C, int32_t dtype, const int32_t* pos0, float* state,
                                 const cpr_gdn_ring* ring, void* out, float* boundary_states,
                                 int64_t boundary_capacity, void* workspace, size_t workspace_bytes, void* stream)
{
    return cpr_gdn_prefill_continue_grouped(q, k, v, g, beta, cu_seqlens, n_seqs, total_tokens, H, H, 0u, dk, dv, C,
                                            dtype, pos0, state, ring, out, boundary_states, boundary_capacity,
                                            workspace, workspace_bytes, stream);
}

int32_t cpr_gdn_ring_from_prefill(const void* k, const void* v, const float* g, const float* beta,
                                  const int32_t* cu_seqlens, int32_t n_seqs, int64_t total_tokens, int32_t H,
                                  int32_t dk, int32_t dv, int32_t C, int32_t dtype, const float* boundary_states,
                                  const float* state_out, const cpr_gdn_ring* ring, void* stream)
{
    return cpr_gdn_ring_from_prefill_grouped(k, v, g, beta, cu_seqlens, n_seqs, total_tokens, H, H, dk, dv, C, dtype,
                                             boundary_states, state_out, ring, stream);
}

int32_t cpr_gdn_decode(const void* q, const void* k, const void* v, const float* g, const float* beta,
                       float* state, const cpr_gdn_ring* ring, const int32_t* pos, int32_t B, int32_t H, int32_t dk,
                       int32_t dv, int32_t C, int32_t dtype, void* out, void* workspace, size_t workspace_bytes,
                       void* stream)
{
    return cpr_gdn_decode_grouped(q, k, v, g, beta, state, ring, pos, B, H, H, 0u, dk, dv, C, dtype, out, workspace,
                                  workspace_bytes, stream);
}

}  // extern "C"
