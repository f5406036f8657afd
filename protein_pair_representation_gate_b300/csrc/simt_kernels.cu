// SIMT (CUDA-core, fp32 arithmetic) path of the gated triangle attention, and
// of MSA row attention with pair bias (the same kernels over S rows of an MSA
// tensor, the bias projected from the pair tensor in a pass of its own).
//
// Three kernels per forward (per key chunk for the attention one):
//   simt_ln_proj    LayerNorm + q/k/v/gate/pair-bias projections, line-major
//   simt_attention  biased softmax attention with an online (running max/sum)
//                   softmax over key tiles, gate applied, key-chunk merge
//   simt_out_proj   output projection, output bias, pair mask, node-dependent store
// It serves fp32 storage (where the tensor-core path would not hold a 1e-4
// error bound) and shapes the sm103 kernels do not cover.
//
// The operation is the one described in tri_attn.h (Dell page, Evoformer
// paragraph; Intel page, steps 2 and 4); the key-chunk merge follows the
// Design-CP summary, Methodology 1 (keys in pieces, log-sum-exp merge).
#include <cuda_bf16.h>
#include <math.h>

#include "tri_attn_internal.h"

namespace tri_attn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kPairs = 16;        // pairs per block in the projection kernels
constexpr int kKeyTile = 32;      // keys per shared-memory tile in the attention kernel

template <typename T> __device__ __forceinline__ float ldf(const T* p, size_t i);
template <> __device__ __forceinline__ float ldf<float>(const float* p, size_t i) { return p[i]; }
template <> __device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p, size_t i) {
    return __bfloat162float(p[i]);
}
template <typename T> __device__ __forceinline__ T stf(float v);
template <> __device__ __forceinline__ float stf<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 stf<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

struct ProjArgs {
    int node, I, I_pad, c, H, d;
    float eps, qscale;
    const void* Z;
    const uint8_t* mask;
    const float *gamma, *beta, *b_g;
    const void *w_q, *w_k, *w_v, *w_g, *w_b;
    float *q, *k, *v, *g, *bias;
};

// One block: line L = blockIdx.y, positions x0 .. x0+15 (x0 = 16 * blockIdx.x).
template <typename T>
__global__ void __launch_bounds__(256) simt_ln_proj(ProjArgs a) {
    extern __shared__ float zh[];                      // [kPairs][c]
    const int L = blockIdx.y, x0 = blockIdx.x * kPairs;
    const int c = a.c, C = a.H * a.d;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const T* Z = static_cast<const T*>(a.Z);

    // LayerNorm, one warp per pair vector (two-pass mean / biased variance).
    for (int p = warp; p < kPairs; p += blockDim.x >> 5) {
        const int x = x0 + p;
        float* dst = zh + p * c;
        if (x >= a.I) {
            for (int cc = lane; cc < c; cc += 32) dst[cc] = 0.f;
            continue;
        }
        const size_t pair = a.node == TRI_ATTN_STARTING ? (size_t)L * a.I + x : (size_t)x * a.I + L;
        const size_t base = pair * c;
        float s = 0.f;
        for (int cc = lane; cc < c; cc += 32) s += ldf(Z, base + cc);
        for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        const float mu = s / c;
        float s2 = 0.f;
        for (int cc = lane; cc < c; cc += 32) {
            const float t = ldf(Z, base + cc) - mu;
            s2 += t * t;
        }
        for (int o = 16; o; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
        const float rstd = rsqrtf(s2 / c + a.eps);
        for (int cc = lane; cc < c; cc += 32) dst[cc] = (ldf(Z, base + cc) - mu) * rstd * a.gamma[cc] + a.beta[cc];
    }
    __syncthreads();

    // Projections: thread owns output column `col` for all 16 pairs.  Columns
    // 0 .. 4C-1 are q | k | v | g, the last H the pair bias; a NULL q skips the
    // former and a NULL bias the latter (the two passes of MSA row attention).
    const int col0 = a.q != nullptr ? 0 : 4 * C;
    const int ncols = a.bias != nullptr ? 4 * C + a.H : 4 * C;
    for (int col = col0 + threadIdx.x; col < ncols; col += blockDim.x) {
        const int which = col < 4 * C ? col / C : 4;
        const int cw = which < 4 ? col - which * C : col - 4 * C;
        const T* W = static_cast<const T*>(which == 0 ? a.w_q : which == 1 ? a.w_k : which == 2 ? a.w_v
                                            : which == 3 ? a.w_g : a.w_b);
        const int ldw = which < 4 ? C : a.H;
        float acc[kPairs];
#pragma unroll
        for (int p = 0; p < kPairs; ++p) acc[p] = 0.f;
        for (int cc = 0; cc < c; ++cc) {
            const float w = ldf(W, (size_t)cc * ldw + cw);
#pragma unroll
            for (int p = 0; p < kPairs; ++p) acc[p] = fmaf(zh[p * c + cc], w, acc[p]);
        }
        for (int p = 0; p < kPairs; ++p) {
            const int x = x0 + p;
            if (x >= a.I_pad) break;
            if (which < 3) {
                const int h = cw / a.d, e = cw % a.d;
                const size_t idx = (((size_t)L * a.H + h) * a.I_pad + x) * a.d + e;
                float* dst = which == 0 ? a.q : which == 1 ? a.k : a.v;
                dst[idx] = x < a.I ? (which == 0 ? acc[p] * a.qscale : acc[p]) : 0.f;
            } else if (which == 3) {
                const float t = acc[p] + a.b_g[cw];
                a.g[((size_t)L * a.I_pad + x) * C + cw] = x < a.I ? 1.f / (1.f + expf(-t)) : 0.f;
            } else {
                const bool valid = x < a.I && (a.mask == nullptr || a.mask[x] != 0);
                a.bias[((size_t)cw * a.I_pad + L) * a.I_pad + x] = valid ? acc[p] * kLog2e : -INFINITY;
            }
        }
    }
}

struct AttnArgs {
    int I, I_pad, H, d, C;
    int k_begin, k_end, first, last;
    const uint8_t* mask;
    const uint8_t* pmask;      // [I, I] pair mask over the pairs of Z, or NULL
    int node;
    const float *q, *k, *v, *g, *bias;
    float *u, *o_run, *lse_run;
};

// One thread per query position; block = 128 positions of one (line, head).
// Scores are in log2 units: q carries log2(e)/sqrt(d), the bias log2(e).
template <int D>
__global__ void __launch_bounds__(128) simt_attention(AttnArgs a) {
    __shared__ float ks[kKeyTile][D];
    __shared__ float vs[kKeyTile][D];
    const int x = blockIdx.x * 128 + threadIdx.x;
    const int h = blockIdx.y, L = blockIdx.z;
    if (a.mask && a.mask[L] == 0) return;               // whole line is written as zeros later
    const bool active = x < a.I;
    const size_t lh = (size_t)L * a.H + h;

    float q[D], acc[D];
#pragma unroll
    for (int e = 0; e < D; ++e) {
        q[e] = active ? a.q[(lh * a.I_pad + x) * D + e] : 0.f;
        acc[e] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    const float* brow = a.bias + ((size_t)h * a.I_pad + (active ? x : 0)) * a.I_pad;

    for (int y0 = a.k_begin; y0 < a.k_end; y0 += kKeyTile) {
        const int nk = min(kKeyTile, a.k_end - y0);
        __syncthreads();
        for (int t = threadIdx.x; t < kKeyTile * D; t += blockDim.x) {
            const int yy = t / D, e = t % D;
            const bool ok = yy < nk;
            ks[yy][e] = ok ? a.k[(lh * a.I_pad + y0 + yy) * D + e] : 0.f;
            vs[yy][e] = ok ? a.v[(lh * a.I_pad + y0 + yy) * D + e] : 0.f;
        }
        __syncthreads();
        if (!active) continue;
        float s[kKeyTile];
        float tmax = -INFINITY;
#pragma unroll
        for (int yy = 0; yy < kKeyTile; ++yy) {
            float t = -INFINITY;
            const int key = y0 + yy;
            const bool key_ok = a.pmask == nullptr ||
                                a.pmask[a.node == TRI_ATTN_STARTING ? (size_t)L * a.I + key : (size_t)key * a.I + L] != 0;
            if (yy < nk && key_ok) {
                t = brow[y0 + yy];
#pragma unroll
                for (int e = 0; e < D; ++e) t = fmaf(q[e], ks[yy][e], t);
            }
            s[yy] = t;
            tmax = fmaxf(tmax, t);
        }
        const float mnew = fmaxf(m, tmax);
        if (mnew == -INFINITY) continue;                 // every key so far is masked
        const float alpha = exp2f(m - mnew);             // m = -inf gives 0
        l *= alpha;
#pragma unroll
        for (int e = 0; e < D; ++e) acc[e] *= alpha;
#pragma unroll
        for (int yy = 0; yy < kKeyTile; ++yy) {
            const float p = exp2f(s[yy] - mnew);
            l += p;
#pragma unroll
            for (int e = 0; e < D; ++e) acc[e] = fmaf(p, vs[yy][e], acc[e]);
        }
        m = mnew;
    }
    if (!active) return;

    // Normalised partial result and its log2-sum-exp2 over this key range.
    float lse = l > 0.f ? m + log2f(l) : -INFINITY;
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int e = 0; e < D; ++e) acc[e] *= inv;

    const size_t srow = lh * a.I_pad + x;
    if (!a.first) {                                      // merge with the running chunk state
        const float lr = a.lse_run[srow];
        const float top = fmaxf(lr, lse);
        if (top != -INFINITY) {
            const float wr = exp2f(lr - top), wc = exp2f(lse - top);
            const float inv_t = 1.f / (wr + wc);
#pragma unroll
            for (int e = 0; e < D; ++e) acc[e] = (wr * a.o_run[srow * D + e] + wc * acc[e]) * inv_t;
            lse = top + log2f(wr + wc);
        }
    }
    if (!a.last) {
        a.lse_run[srow] = lse;
#pragma unroll
        for (int e = 0; e < D; ++e) a.o_run[srow * D + e] = acc[e];
        return;
    }
    const size_t urow = ((size_t)L * a.I_pad + x) * a.C + h * D;
#pragma unroll
    for (int e = 0; e < D; ++e) a.u[urow + e] = a.g[urow + e] * acc[e];
}

struct OutArgs {
    int node, I, I_pad, c, C;
    const uint8_t* mask;
    const uint8_t* pmask;      // [I, I] pair mask, or NULL
    const float* u;
    const void* w_o;
    const float* b_o;
    const void* Z;             // residual source (NULL: write the update only)
    void* out;
};

// One block: line L = blockIdx.y, positions x0 .. x0+15; thread = output channel.
template <typename T>
__global__ void __launch_bounds__(128) simt_out_proj(OutArgs a) {
    extern __shared__ float us[];                       // [kPairs][C]
    const int L = blockIdx.y, x0 = blockIdx.x * kPairs;
    const bool line_ok = a.mask == nullptr || a.mask[L] != 0;
    for (int t = threadIdx.x; t < kPairs * a.C; t += blockDim.x) {
        const int p = t / a.C, xx = t % a.C, x = x0 + p;
        us[t] = (line_ok && x < a.I) ? a.u[((size_t)L * a.I_pad + x) * a.C + xx] : 0.f;
    }
    __syncthreads();
    const T* W = static_cast<const T*>(a.w_o);
    T* out = static_cast<T*>(a.out);
    for (int n = threadIdx.x; n < a.c; n += blockDim.x) {
        float acc[kPairs];
#pragma unroll
        for (int p = 0; p < kPairs; ++p) acc[p] = 0.f;
        for (int xx = 0; xx < a.C; ++xx) {
            const float w = ldf(W, (size_t)xx * a.c + n);
#pragma unroll
            for (int p = 0; p < kPairs; ++p) acc[p] = fmaf(us[p * a.C + xx], w, acc[p]);
        }
        const float bo = a.b_o ? a.b_o[n] : 0.f;
        for (int p = 0; p < kPairs; ++p) {
            const int x = x0 + p;
            if (x >= a.I) break;
            const size_t pair = a.node == TRI_ATTN_STARTING ? (size_t)L * a.I + x : (size_t)x * a.I + L;
            const bool ok = line_ok && (a.mask == nullptr || a.mask[x] != 0) &&
                            (a.pmask == nullptr || a.pmask[pair] != 0);
            float v = ok ? acc[p] + bo : 0.f;
            if (a.Z) v += ldf(static_cast<const T*>(a.Z), pair * a.c + n);   // in place: read before write
            out[pair * a.c + n] = stf<T>(v);
        }
    }
}

template <int D>
cudaError_t launch_attention(const AttnArgs& aa, int I_pad, int H, int I, cudaStream_t s) {
    dim3 grid(I_pad / 128, H, I);
    simt_attention<D><<<grid, 128, 0, s>>>(aa);
    return cudaGetLastError();
}

template <typename T>
cudaError_t simt_forward_t(const FwdArgs& a, cudaStream_t s, LaunchTimer* tm) {
    const Workspace& W = *a.lay;
    const int C = a.H * a.d;
    auto f = [&](size_t off) { return reinterpret_cast<float*>(a.ws + off); };

    ProjArgs pa{a.node, a.I, a.I_pad, a.c_z, a.H, a.d, a.eps, kLog2e / sqrtf((float)a.d), a.Z, a.mask,
                a.w.ln_gamma, a.w.ln_beta, a.w.b_g, a.w.w_q, a.w.w_k, a.w.w_v, a.w.w_g, a.w.w_b,
                f(W.q), f(W.k), f(W.v), f(W.g), f(W.bias)};
    {
        dim3 grid(a.I_pad / kPairs, a.I);
        if (tm) tm->begin("simt_ln_proj", s);
        simt_ln_proj<T><<<grid, 256, kPairs * a.c_z * sizeof(float), s>>>(pa);
        if (tm) tm->end(s);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const int cs = chunk_size(a.I, a.key_chunks);
    for (int k0 = 0; k0 < a.I; k0 += cs) {
        const int k1 = k0 + cs < a.I ? k0 + cs : a.I;
        AttnArgs aa{a.I, a.I_pad, a.H, a.d, C, k0, k1, k0 == 0, k1 == a.I, a.mask, a.pair_mask, a.node,
                    f(W.q), f(W.k), f(W.v), f(W.g), f(W.bias), f(W.u),
                    W.o_run ? f(W.o_run) : nullptr, W.lse_run ? f(W.lse_run) : nullptr};
        if (tm) tm->begin("simt_attention", s);
        cudaError_t e;
        switch (a.d) {
            case 8: e = launch_attention<8>(aa, a.I_pad, a.H, a.I, s); break;
            case 16: e = launch_attention<16>(aa, a.I_pad, a.H, a.I, s); break;
            case 32: e = launch_attention<32>(aa, a.I_pad, a.H, a.I, s); break;
            case 64: e = launch_attention<64>(aa, a.I_pad, a.H, a.I, s); break;
            default: e = cudaErrorInvalidValue;
        }
        if (tm) tm->end(s);
        if (e != cudaSuccess) return e;
    }
    OutArgs oa{a.node, a.I, a.I_pad, a.c_z, C, a.mask, a.pair_mask, f(W.u), a.w.w_o, a.w.b_o,
               a.residual ? a.Z : nullptr, a.out};
    {
        dim3 grid((a.I + kPairs - 1) / kPairs, a.I);
        if (tm) tm->begin("simt_out_proj", s);
        simt_out_proj<T><<<grid, 128, kPairs * C * sizeof(float), s>>>(oa);
        if (tm) tm->end(s);
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t simt_msa_forward_t(const MsaArgs& a, cudaStream_t s, LaunchTimer* tm) {
    const Workspace& W = *a.lay;
    const int C = a.H * a.d;
    auto f = [&](size_t off) { return reinterpret_cast<float*>(a.ws + off); };
    cudaError_t e;
    // pair bias b[h, i, j] = LN_z(Z[i, j]) W_b[:, h]: lines i of Z, bias columns only
    ProjArgs pz{TRI_ATTN_STARTING, a.I, a.I_pad, a.c_z, a.H, a.d, a.eps, 0.f, a.Z, nullptr,
                a.w.ln_z_gamma, a.w.ln_z_beta, nullptr, nullptr, nullptr, nullptr, nullptr, a.w.w_b,
                nullptr, nullptr, nullptr, nullptr, f(W.bias)};
    {
        dim3 grid(a.I_pad / kPairs, a.I);
        if (tm) tm->begin("simt_ln_proj", s);
        simt_ln_proj<T><<<grid, 256, kPairs * a.c_z * sizeof(float), s>>>(pz);
        if (tm) tm->end(s);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // q, k, v, g of the MSA rows: lines s of Ms (row-major [S, I, c_m], the
    // starting orientation), no bias columns
    ProjArgs pm{TRI_ATTN_STARTING, a.I, a.I_pad, a.c_m, a.H, a.d, a.eps, kLog2e / sqrtf((float)a.d), a.M, nullptr,
                a.w.ln_m_gamma, a.w.ln_m_beta, a.w.b_g, a.w.w_q, a.w.w_k, a.w.w_v, a.w.w_g, nullptr,
                f(W.q), f(W.k), f(W.v), f(W.g), nullptr};
    {
        dim3 grid(a.I_pad / kPairs, a.S);
        if (tm) tm->begin("simt_ln_proj", s);
        simt_ln_proj<T><<<grid, 256, kPairs * a.c_m * sizeof(float), s>>>(pm);
        if (tm) tm->end(s);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // row s attends over its residues; the MSA mask acts as a pair mask over [S, I]
    const int cs = chunk_size(a.I, a.key_chunks);
    for (int k0 = 0; k0 < a.I; k0 += cs) {
        const int k1 = k0 + cs < a.I ? k0 + cs : a.I;
        AttnArgs aa{a.I, a.I_pad, a.H, a.d, C, k0, k1, k0 == 0, k1 == a.I, nullptr, a.msa_mask, TRI_ATTN_STARTING,
                    f(W.q), f(W.k), f(W.v), f(W.g), f(W.bias), f(W.u),
                    W.o_run ? f(W.o_run) : nullptr, W.lse_run ? f(W.lse_run) : nullptr};
        if (tm) tm->begin("simt_attention", s);
        switch (a.d) {
            case 8: e = launch_attention<8>(aa, a.I_pad, a.H, a.S, s); break;
            case 16: e = launch_attention<16>(aa, a.I_pad, a.H, a.S, s); break;
            case 32: e = launch_attention<32>(aa, a.I_pad, a.H, a.S, s); break;
            case 64: e = launch_attention<64>(aa, a.I_pad, a.H, a.S, s); break;
            default: e = cudaErrorInvalidValue;
        }
        if (tm) tm->end(s);
        if (e != cudaSuccess) return e;
    }
    OutArgs oa{TRI_ATTN_STARTING, a.I, a.I_pad, a.c_m, C, nullptr, a.msa_mask, f(W.u), a.w.w_o, a.w.b_o,
               a.residual ? a.M : nullptr, a.out};
    {
        dim3 grid((a.I + kPairs - 1) / kPairs, a.S);
        if (tm) tm->begin("simt_out_proj", s);
        simt_out_proj<T><<<grid, 128, kPairs * C * sizeof(float), s>>>(oa);
        if (tm) tm->end(s);
    }
    return cudaGetLastError();
}

}  // namespace

Workspace simt_msa_layout(int S, int I, int H, int d, int key_chunks) {
    Workspace w;
    w.I = I;
    w.I_pad = round_up(I, kTile);
    const size_t P = (size_t)S * w.I_pad;          // row-major (MSA row, residue) slots
    const size_t C = (size_t)H * d;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align256(off + bytes); return o; };
    w.q = take(P * C * 4);
    w.k = take(P * C * 4);
    w.v = take(P * C * 4);
    w.g = take(P * C * 4);
    w.u = take(P * C * 4);
    w.bias = take((size_t)H * w.I_pad * w.I_pad * 4);
    if (key_chunks > 1) {
        w.o_run = take(P * C * 4);
        w.lse_run = take(P * H * 4);
    }
    w.total = off;
    return w;
}

cudaError_t simt_msa_forward(const MsaArgs& a, int dtype, cudaStream_t s, LaunchTimer* t) {
    if (a.d != 8 && a.d != 16 && a.d != 32 && a.d != 64) return cudaErrorInvalidValue;
    return dtype == TRI_ATTN_F32 ? simt_msa_forward_t<float>(a, s, t) : simt_msa_forward_t<__nv_bfloat16>(a, s, t);
}

Workspace simt_layout(int I, int c_z, int H, int d, int key_chunks) {
    (void)c_z;
    Workspace w;
    w.I = I;
    w.I_pad = round_up(I, kTile);
    const size_t P = (size_t)I * w.I_pad;          // line-major pair slots
    const size_t C = (size_t)H * d;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align256(off + bytes); return o; };
    w.q = take(P * C * 4);
    w.k = take(P * C * 4);
    w.v = take(P * C * 4);
    w.g = take(P * C * 4);
    w.u = take(P * C * 4);
    w.bias = take((size_t)H * w.I_pad * w.I_pad * 4);
    if (key_chunks > 1) {
        w.o_run = take(P * C * 4);
        w.lse_run = take(P * H * 4);
    }
    w.total = off;
    return w;
}

cudaError_t simt_forward(const FwdArgs& a, int dtype, cudaStream_t s, LaunchTimer* t) {
    if (a.d != 8 && a.d != 16 && a.d != 32 && a.d != 64) return cudaErrorInvalidValue;
    return dtype == TRI_ATTN_F32 ? simt_forward_t<float>(a, s, t) : simt_forward_t<__nv_bfloat16>(a, s, t);
}

}  // namespace tri_attn
