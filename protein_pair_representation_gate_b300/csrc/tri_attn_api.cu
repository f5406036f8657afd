// C-ABI layer: context, argument validation, workspace layout, dispatch and
// per-kernel timing.  The operation and the entry points are specified in
// include/tri_attn.h.
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "tri_attn_internal.h"

using namespace tri_attn;

struct tri_attn_ctx {
    tri_attn_config cfg;
    int device = 0;
    int path = TRI_ATTN_PATH_SIMT;
    bool msa_sm103 = false;  // MSA forwards with c_m = 256 take the sm103 path
    uint32_t* d_status = nullptr;

    // timing
    struct Rec { const char* name; cudaEvent_t a, b; };
    struct Timer : LaunchTimer {
        std::vector<Rec> pool;
        int used = 0;
        bool broken = false;
        bool on = false;
        void begin(const char* name, cudaStream_t s) override {
            on = used < 8192;
            if (!on) return;
            if ((int)pool.size() <= used) {
                Rec r{name, nullptr, nullptr};
                if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess) { broken = true; return; }
                pool.push_back(r);
            }
            pool[used].name = name;
            cudaEventRecord(pool[used].a, s);
        }
        void end(cudaStream_t s) override {
            if (broken || !on) return;
            cudaEventRecord(pool[used].b, s);
            ++used;
        }
    } timer;
    bool timing = false;
    int inject = 0;          // one-shot test hook
};

namespace {

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const char* pa = static_cast<const char*>(a);
    const char* pb = static_cast<const char*>(b);
    return pa < pb + nb && pb < pa + na;
}

bool aligned(const void* p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

Workspace layout_for(const tri_attn_ctx* c, int I) {
    const tri_attn_config& g = c->cfg;
    if (c->path == TRI_ATTN_PATH_SM103) return sm103_layout(I, g.key_chunks);
    if (c->path == TRI_ATTN_PATH_SM103_TF32) return sm103_tf32_layout(I, g.key_chunks);
    return simt_layout(I, g.c_z, g.heads, g.head_dim, g.key_chunks);
}

// The CUDA-core kernels run every fp32-storage dtype in fp32 arithmetic.
int simt_dtype(int dtype) { return dtype == TRI_ATTN_BF16 ? TRI_ATTN_BF16 : TRI_ATTN_F32; }

bool config_ok(const tri_attn_config* g) {
    if (g->c_z < 1 || g->c_z > 256) return false;
    if (g->heads < 1 || g->heads > 16) return false;
    if (g->head_dim < 1 || g->head_dim > 64 || g->heads * g->head_dim > 256) return false;
    if (g->I_max < 1 || g->I_max > 16384) return false;
    if (g->dtype != TRI_ATTN_F32 && g->dtype != TRI_ATTN_BF16 && g->dtype != TRI_ATTN_TF32) return false;
    if (!(g->ln_eps > 0.f) || g->ln_eps > 1.f) return false;
    if (g->key_chunks < 1 || g->key_chunks > 64) return false;
    return true;
}

}  // namespace

extern "C" {

const char* tri_attn_status_string(int s) {
    switch (s) {
        case TRI_ATTN_OK: return "ok";
        case TRI_ATTN_EINVAL: return "invalid argument";
        case TRI_ATTN_EUNSUPPORTED: return "unsupported shape or dtype";
        case TRI_ATTN_ENOMEM: return "workspace too small or allocation failed";
        case TRI_ATTN_ECUDA: return "CUDA error";
        case TRI_ATTN_ETIMEOUT: return "device wait timed out";
        case TRI_ATTN_ERANGE: return "f16 intermediate out of range";
        default: return "unknown status";
    }
}

tri_attn_status tri_attn_create(const tri_attn_config* cfg, tri_attn_ctx** out) {
    if (out) *out = nullptr;
    if (!cfg || !out) return TRI_ATTN_EINVAL;
    if (!config_ok(cfg)) return TRI_ATTN_EINVAL;
    const bool sm103 = !cfg->force_simt && sm103_supported(cfg->c_z, cfg->heads, cfg->head_dim, cfg->dtype);
    const bool tf32 = !cfg->force_simt && sm103_tf32_supported(cfg->c_z, cfg->heads, cfg->head_dim, cfg->dtype);
    const int d = cfg->head_dim;
    if (!sm103 && !tf32 && d != 8 && d != 16 && d != 32 && d != 64) return TRI_ATTN_EUNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TRI_ATTN_ECUDA;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return TRI_ATTN_ECUDA;
    const bool is_sm103 = major == 10 && minor == 3;                  // kernels are built for sm_103a only
    if ((sm103 || tf32) && !is_sm103) return TRI_ATTN_EUNSUPPORTED;
    tri_attn_ctx* c = new (std::nothrow) tri_attn_ctx();
    if (!c) return TRI_ATTN_ENOMEM;
    c->cfg = *cfg;
    c->device = dev;
    c->path = sm103 ? TRI_ATTN_PATH_SM103 : tf32 ? TRI_ATTN_PATH_SM103_TF32 : TRI_ATTN_PATH_SIMT;
    c->msa_sm103 = is_sm103 && !cfg->force_simt &&
                   sm103_msa_supported(kMsaCm, cfg->c_z, cfg->heads, cfg->head_dim, cfg->dtype);
    if (cudaMalloc(&c->d_status, sizeof(uint32_t)) != cudaSuccess ||
        cudaMemset(c->d_status, 0, sizeof(uint32_t)) != cudaSuccess) {
        cudaFree(c->d_status);
        delete c;
        return TRI_ATTN_ECUDA;
    }
    *out = c;
    return TRI_ATTN_OK;
}

void tri_attn_destroy(tri_attn_ctx* c) {
    if (!c) return;
    for (auto& r : c->timer.pool) {
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    cudaFree(c->d_status);
    delete c;
}

int tri_attn_path(const tri_attn_ctx* c) { return c ? c->path : -1; }

size_t tri_attn_workspace_bytes(const tri_attn_ctx* c, int I) {
    if (!c || I < 1 || I > c->cfg.I_max) return 0;
    return layout_for(c, I).total;
}

tri_attn_status tri_attn_forward(tri_attn_ctx* c, int node, int I, const void* Z, const uint8_t* mask,
                                 const tri_attn_weights* w, void* workspace, size_t workspace_bytes,
                                 void* out, void* stream) {
    return tri_attn_forward_ex(c, node, I, Z, mask, nullptr, w, workspace, workspace_bytes, out, stream);
}

tri_attn_status tri_attn_forward_ex(tri_attn_ctx* c, int node, int I, const void* Z, const uint8_t* mask,
                                    const tri_attn_options* opt, const tri_attn_weights* w, void* workspace,
                                    size_t workspace_bytes, void* out, void* stream) {
    if (!c || !Z || !w || !workspace || !out) return TRI_ATTN_EINVAL;
    const tri_attn_config& g = c->cfg;
    if (node != TRI_ATTN_STARTING && node != TRI_ATTN_ENDING) return TRI_ATTN_EINVAL;
    if (I < 1 || I > g.I_max) return TRI_ATTN_EINVAL;
    if (!w->ln_gamma || !w->ln_beta || !w->w_q || !w->w_k || !w->w_v || !w->w_g || !w->w_b || !w->b_g || !w->w_o)
        return TRI_ATTN_EINVAL;
    if (!aligned(Z, 16) || !aligned(out, 16) || !aligned(workspace, 256)) return TRI_ATTN_EINVAL;
    const void* wp[] = {w->ln_gamma, w->ln_beta, w->w_q, w->w_k, w->w_v, w->w_g, w->w_b, w->b_g, w->w_o, w->b_o};
    for (const void* p : wp)
        if (p && !aligned(p, 16)) return TRI_ATTN_EINVAL;
    const Workspace lay = layout_for(c, I);
    if (workspace_bytes < lay.total) return TRI_ATTN_ENOMEM;
    const size_t esz = g.dtype == TRI_ATTN_BF16 ? 2 : 4;
    const size_t pair_bytes = (size_t)I * I * g.c_z * esz;
    const bool residual = opt && opt->residual;
    const bool in_place = residual && out == Z;          // the one overlap allowed: Z += update
    if ((!in_place && overlaps(out, pair_bytes, Z, pair_bytes)) || overlaps(out, pair_bytes, workspace, lay.total) ||
        overlaps(Z, pair_bytes, workspace, lay.total))
        return TRI_ATTN_EINVAL;
    if (mask && (overlaps(mask, (size_t)I, out, pair_bytes) || overlaps(mask, (size_t)I, workspace, lay.total)))
        return TRI_ATTN_EINVAL;
    const uint8_t* pmask = opt ? opt->pair_mask : nullptr;
    if (pmask && (overlaps(pmask, (size_t)I * I, out, pair_bytes) || overlaps(pmask, (size_t)I * I, workspace, lay.total)))
        return TRI_ATTN_EINVAL;

    FwdArgs a;
    a.node = node;
    a.I = I;
    a.I_pad = lay.I_pad;
    a.c_z = g.c_z;
    a.H = g.heads;
    a.d = g.head_dim;
    a.eps = g.ln_eps;
    a.Z = Z;
    a.mask = mask;
    a.w = *w;
    a.ws = static_cast<char*>(workspace);
    a.lay = &lay;
    a.out = out;
    a.key_chunks = g.key_chunks;
    a.status = c->d_status;
    a.inject = c->inject;
    a.pair_mask = pmask;
    a.residual = residual ? 1 : 0;
    c->inject = 0;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    LaunchTimer* t = c->timing ? &c->timer : nullptr;
    cudaError_t e = c->path == TRI_ATTN_PATH_SM103        ? sm103_forward(a, s, t)
                    : c->path == TRI_ATTN_PATH_SM103_TF32 ? sm103_tf32_forward(a, s, t)
                                                          : simt_forward(a, simt_dtype(g.dtype), s, t);
    if (e != cudaSuccess) {
        fprintf(stderr, "tri_attn_forward: %s\n", cudaGetErrorString(e));
        return TRI_ATTN_ECUDA;
    }
    return TRI_ATTN_OK;
}

int tri_attn_msa_path(const tri_attn_ctx* c, int c_m) {
    if (!c) return -1;
    const tri_attn_config& g = c->cfg;
    return c->msa_sm103 && sm103_msa_supported(c_m, g.c_z, g.heads, g.head_dim, g.dtype) ? TRI_ATTN_PATH_SM103
                                                                                       : TRI_ATTN_PATH_SIMT;
}

size_t tri_attn_msa_workspace_bytes(const tri_attn_ctx* c, int S, int I) {
    if (!c || S < 1 || S > kMsaMaxRows || I < 1 || I > c->cfg.I_max) return 0;
    // enough for either path (the path also depends on c_m, which this call does not take)
    const size_t simt = simt_msa_layout(S, I, c->cfg.heads, c->cfg.head_dim, c->cfg.key_chunks).total;
    const size_t sm103 = c->msa_sm103 ? sm103_msa_layout(S, I, c->cfg.key_chunks).total : 0;
    return simt > sm103 ? simt : sm103;
}

tri_attn_status tri_attn_msa_forward(tri_attn_ctx* c, int S, int I, int c_m, const void* msa, const uint8_t* msa_mask,
                                     const void* Z, const tri_attn_msa_weights* w, int residual, void* workspace,
                                     size_t workspace_bytes, void* out, void* stream) {
    if (!c || !msa || !Z || !w || !workspace || !out) return TRI_ATTN_EINVAL;
    const tri_attn_config& g = c->cfg;
    if (S < 1 || S > kMsaMaxRows || I < 1 || I > g.I_max || c_m < 1 || c_m > 256) return TRI_ATTN_EINVAL;
    if (g.head_dim != 8 && g.head_dim != 16 && g.head_dim != 32 && g.head_dim != 64) return TRI_ATTN_EUNSUPPORTED;
    if (!w->ln_m_gamma || !w->ln_m_beta || !w->w_q || !w->w_k || !w->w_v || !w->w_g || !w->b_g || !w->w_o ||
        !w->ln_z_gamma || !w->ln_z_beta || !w->w_b)
        return TRI_ATTN_EINVAL;
    if (!aligned(msa, 16) || !aligned(Z, 16) || !aligned(out, 16) || !aligned(workspace, 256)) return TRI_ATTN_EINVAL;
    const void* wp[] = {w->ln_m_gamma, w->ln_m_beta, w->w_q, w->w_k, w->w_v, w->w_g, w->b_g, w->w_o, w->b_o,
                        w->ln_z_gamma, w->ln_z_beta, w->w_b};
    for (const void* p : wp)
        if (p && !aligned(p, 16)) return TRI_ATTN_EINVAL;
    const bool on_sm103 = tri_attn_msa_path(c, c_m) == TRI_ATTN_PATH_SM103;
    const Workspace lay = on_sm103 ? sm103_msa_layout(S, I, g.key_chunks)
                                   : simt_msa_layout(S, I, g.heads, g.head_dim, g.key_chunks);
    if (workspace_bytes < lay.total) return TRI_ATTN_ENOMEM;
    const size_t esz = g.dtype == TRI_ATTN_BF16 ? 2 : 4;
    const size_t msa_bytes = (size_t)S * I * c_m * esz, z_bytes = (size_t)I * I * g.c_z * esz;
    const bool in_place = residual && out == msa;        // the one overlap allowed: Ms += update
    if ((!in_place && overlaps(out, msa_bytes, msa, msa_bytes)) || overlaps(out, msa_bytes, Z, z_bytes) ||
        overlaps(out, msa_bytes, workspace, lay.total) || overlaps(msa, msa_bytes, workspace, lay.total) ||
        overlaps(Z, z_bytes, workspace, lay.total))
        return TRI_ATTN_EINVAL;
    if (msa_mask && (overlaps(msa_mask, (size_t)S * I, out, msa_bytes) ||
                     overlaps(msa_mask, (size_t)S * I, workspace, lay.total)))
        return TRI_ATTN_EINVAL;

    MsaArgs a;
    a.S = S;
    a.I = I;
    a.I_pad = lay.I_pad;
    a.c_m = c_m;
    a.c_z = g.c_z;
    a.H = g.heads;
    a.d = g.head_dim;
    a.key_chunks = g.key_chunks;
    a.residual = residual ? 1 : 0;
    a.eps = g.ln_eps;
    a.M = msa;
    a.msa_mask = msa_mask;
    a.Z = Z;
    a.w = *w;
    a.ws = static_cast<char*>(workspace);
    a.lay = &lay;
    a.out = out;
    a.status = c->d_status;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    LaunchTimer* t = c->timing ? &c->timer : nullptr;
    const cudaError_t e = on_sm103 ? sm103_msa_forward(a, s, t) : simt_msa_forward(a, simt_dtype(g.dtype), s, t);
    if (e != cudaSuccess) {
        fprintf(stderr, "tri_attn_msa_forward: %s\n", cudaGetErrorString(e));
        return TRI_ATTN_ECUDA;
    }
    return TRI_ATTN_OK;
}

tri_attn_status tri_attn_status_sync(tri_attn_ctx* c, void* stream) {
    if (!c) return TRI_ATTN_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return TRI_ATTN_ECUDA;
    uint32_t v = 0;
    if (cudaMemcpy(&v, c->d_status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return TRI_ATTN_ECUDA;
    if (v) {
        if (cudaMemset(c->d_status, 0, sizeof v) != cudaSuccess) return TRI_ATTN_ECUDA;
        return (v & kStatusTimeoutMask) ? TRI_ATTN_ETIMEOUT : TRI_ATTN_ERANGE;
    }
    return TRI_ATTN_OK;
}

tri_attn_status tri_attn_debug_inject(tri_attn_ctx* c, int fault) {
    if (!c) return TRI_ATTN_EINVAL;
    if (fault != TRI_ATTN_FAULT_NONE && fault != TRI_ATTN_FAULT_SKIP_STAGE) return TRI_ATTN_EINVAL;
    if (fault != TRI_ATTN_FAULT_NONE && c->path == TRI_ATTN_PATH_SIMT) return TRI_ATTN_EUNSUPPORTED;
    c->inject = fault;
    return TRI_ATTN_OK;
}

tri_attn_status tri_attn_set_timing(tri_attn_ctx* c, int on) {
    if (!c) return TRI_ATTN_EINVAL;
    c->timing = on != 0;
    c->timer.used = 0;
    return TRI_ATTN_OK;
}

int tri_attn_kernel_times(tri_attn_ctx* c, const char** names, float* ms, int cap) {
    if (!c || !c->timing) return -1;
    const int n = c->timer.used;
    for (int k = 0; k < n && k < cap; ++k) {
        auto& r = c->timer.pool[k];
        float v = 0.f;
        if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&v, r.a, r.b) != cudaSuccess) v = -1.f;
        if (names) names[k] = r.name;
        if (ms) ms[k] = v;
    }
    return n;
}

}  // extern "C"
