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
// address (it names a host-side stand-in), so the device address is obtained
// once per device with cudaGetSymbolAddress, with that device current, and
// cached.
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
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up on first use).
cudaError_t scratch_address(int dev, void** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

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
    {
        const char* a = static_cast<const char*>(out);
        const char* b = static_cast<const char*>(Z);
        if (a < b + pair_bytes && b < a + pair_bytes) return TRI_ATTN_EINVAL;
    }

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
    if (!(reinterpret_cast<const char*>(out) + pair_bytes <= ws || ws + kStaticScratchBytes <= static_cast<const char*>(out)))
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
    return sm103_forward(a, s, nullptr) == cudaSuccess ? TRI_ATTN_OK : TRI_ATTN_ECUDA;
}
