// tri_attn_forward_static: the sm103 forward with its workspace in a
// file-scope device array, for callers that cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is unavailable or forbidden
// (inside a host callback or a custom allocator, in a process whose device
// memory is fully pre-reserved by another runtime, or a plugin host that owns
// all allocations) still has its input and output buffers but no way to
// obtain the workspace tri_attn_forward asks for, nor the status word that
// tri_attn_create allocates.
//
// The scratch array below is part of the module: every GPU on which the
// library's module is loaded holds it (kStaticScratchBytes, 34.3 MB)
// until the process exits.  Host code cannot use the array's name as a device
// address (it names a host-side stand-in), so the device address is looked up
// with cudaGetSymbolAddress, with the device current, and cached.  A device
// address belongs to one CUDA context (the module is loaded per context), so
// the cache is keyed by the context's process-unique id: a call made under
// another context, or after cudaDeviceReset re-created the primary context,
// looks the address up again instead of reusing a stale one.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "tri_attn_internal.h"

namespace tri_attn {
namespace {

constexpr int kStaticImax = 128;                      // largest I this entry point accepts
constexpr size_t kStaticWorkspace = sm103_layout(kStaticImax, 1).total;   // sm103 workspace at I = 128
constexpr size_t kStaticScratchBytes = kStaticWorkspace + 256;   // + the device status word

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct Cached {
    unsigned long long ctx_id = 0;   // 0: nothing cached (context ids start at 1)
    void* addr = nullptr;
};
Cached g_cache[kMaxDevices];
std::atomic<int> g_inject{0};        // one-shot test hook (tri_attn_static_debug_inject)

// The driver's current-context queries, looked up once (no libcuda link needed).
struct CtxFns {
    PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    PFN_cuCtxGetId_v12000 get_id = nullptr;
};
const CtxFns& ctx_fns() {
    static const CtxFns f = [] {
        CtxFns r;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            r.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            r.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
        return r;
    }();
    return f;
}

// Id of the context current on this thread (0 if it cannot be determined).
unsigned long long current_ctx_id() {
    const CtxFns& f = ctx_fns();
    if (!f.get_current || !f.get_id) return 0;
    CUcontext c = nullptr;
    if (f.get_current(&c) != CUDA_SUCCESS || c == nullptr) return 0;
    unsigned long long id = 0;
    if (f.get_id(c, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of the scratch array in the current context (looked up on
// the first call in each context).  Called after a runtime call has made the
// device's context current.
cudaError_t scratch_address(int dev, void** out) {
    const unsigned long long id = current_ctx_id();
    if (id == 0) return cudaErrorDeviceUninitialized;
    std::lock_guard<std::mutex> lock(g_mu);
    Cached& c = g_cache[dev];
    if (c.ctx_id != id) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        c.addr = p;
        c.ctx_id = id;
    }
    *out = c.addr;
    return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const char* pa = static_cast<const char*>(a);
    const char* pb = static_cast<const char*>(b);
    return pa < pb + nb && pb < pa + na;
}

}  // namespace
}  // namespace tri_attn

using namespace tri_attn;

extern "C" tri_attn_status tri_attn_forward_static(int node, int I, const void* Z, const uint8_t* token_mask,
                                                   const tri_attn_weights* w, float ln_eps, void* out,
                                                   void* stream) {
    if (!Z || !w || !out) return TRI_ATTN_EINVAL;
    if (node != TRI_ATTN_STARTING && node != TRI_ATTN_ENDING) return TRI_ATTN_EINVAL;
    if (I < 1) return TRI_ATTN_EINVAL;
    if (I > kStaticImax) return TRI_ATTN_EUNSUPPORTED;
    if (!(ln_eps > 0.f) || ln_eps > 1.f) return TRI_ATTN_EINVAL;
    if (!w->ln_gamma || !w->ln_beta || !w->w_q || !w->w_k || !w->w_v || !w->w_g || !w->w_b || !w->b_g || !w->w_o)
        return TRI_ATTN_EINVAL;
    if (!aligned16(Z) || !aligned16(out)) return TRI_ATTN_EINVAL;
    const void* wp[] = {w->ln_gamma, w->ln_beta, w->w_q, w->w_k, w->w_v, w->w_g, w->w_b, w->b_g, w->w_o, w->b_o};
    for (const void* p : wp)
        if (p && !aligned16(p)) return TRI_ATTN_EINVAL;
    const size_t pair_bytes = (size_t)I * I * 128 * 2;
    if (overlaps(out, pair_bytes, Z, pair_bytes)) return TRI_ATTN_EINVAL;
    if (token_mask && overlaps(token_mask, (size_t)I, out, pair_bytes)) return TRI_ATTN_EINVAL;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TRI_ATTN_ECUDA;
    if (dev < 0 || dev >= kMaxDevices) return TRI_ATTN_EUNSUPPORTED;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return TRI_ATTN_ECUDA;
    if (major != 10 || minor != 3) return TRI_ATTN_EUNSUPPORTED;

    const Workspace lay = sm103_layout(I, 1);
    if (lay.total > kStaticWorkspace) return TRI_ATTN_EUNSUPPORTED;
    void* base = nullptr;
    if (scratch_address(dev, &base) != cudaSuccess) return TRI_ATTN_ECUDA;
    char* ws = static_cast<char*>(base);
    uint32_t* status = reinterpret_cast<uint32_t*>(ws + kStaticWorkspace);
    // no input or output may lie in the library's array
    if (overlaps(out, pair_bytes, ws, kStaticScratchBytes) || overlaps(Z, pair_bytes, ws, kStaticScratchBytes) ||
        (token_mask && overlaps(token_mask, (size_t)I, ws, kStaticScratchBytes)))
        return TRI_ATTN_EINVAL;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the status word must start at zero: kernels that find it set return at once
    if (cudaMemsetAsync(status, 0, sizeof(uint32_t), s) != cudaSuccess) return TRI_ATTN_ECUDA;

    FwdArgs a;
    a.node = node;
    a.I = I;
    a.I_pad = lay.I_pad;
    a.c_z = 128;
    a.H = 4;
    a.d = 32;
    a.eps = ln_eps;
    a.Z = Z;
    a.mask = token_mask;
    a.w = *w;
    a.ws = ws;
    a.lay = &lay;
    a.out = out;
    a.key_chunks = 1;
    a.status = status;
    a.inject = g_inject.exchange(0);
    return sm103_forward(a, s, nullptr) == cudaSuccess ? TRI_ATTN_OK : TRI_ATTN_ECUDA;
}

extern "C" tri_attn_status tri_attn_static_status(void* stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TRI_ATTN_ECUDA;
    if (dev < 0 || dev >= kMaxDevices) return TRI_ATTN_EUNSUPPORTED;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return TRI_ATTN_ECUDA;
    uint32_t v = 0;
    if (cudaMemcpyFromSymbol(&v, g_static_scratch, sizeof v, kStaticWorkspace, cudaMemcpyDeviceToHost) != cudaSuccess)
        return TRI_ATTN_ECUDA;
    if (v == 0) return TRI_ATTN_OK;
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_static_scratch, &zero, sizeof zero, kStaticWorkspace, cudaMemcpyHostToDevice) != cudaSuccess)
        return TRI_ATTN_ECUDA;
    return (v & kStatusTimeoutMask) ? TRI_ATTN_ETIMEOUT : TRI_ATTN_ERANGE;
}

extern "C" tri_attn_status tri_attn_static_debug_inject(int fault) {
    if (fault != TRI_ATTN_FAULT_NONE && fault != TRI_ATTN_FAULT_SKIP_STAGE) return TRI_ATTN_EINVAL;
    g_inject.store(fault);
    return TRI_ATTN_OK;
}
