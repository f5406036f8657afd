// sm_103a TF32 forward of the gated triangle attention: fp32 Z, weights and
// output (c_z = 128, H = 4, d = 32), the ExtraMSA-style precision mode.
//
// Source: OpenFold-TRT summary, Methodology (a BF16 Evoformer core with TF32 for
// the ExtraMSA stack, whose pair activations stay in fp32).  The operation is the
// one stated in tri_attn.h.
//
// Precision: the contractions of the LayerNorm and projection step read Z and
// the prepared weights as tf32 (10-bit significand; the tensor core drops the
// low 13 bits of an fp32 operand), accumulating in fp32; the LayerNorm statistics
// and the pair bias are fp32 on CUDA cores.  The attention step is the bf16
// path's kernel with f16 intermediates (q, k, v, gate, bias, P, u, W_o: the same
// 10-bit significand as tf32, with the f16 range checked: ERANGE) and an fp32
// epilogue (output bias, masks, fp32 residual, fp32 store).
//
// Kernels per forward:
//   sm103_tf32_prep   gamma-folded projection weights rounded to tf32 (q columns
//                     times log2(e)/sqrt(d)), their column sums and offsets
//                     (beta W, + b_g for the gate), gamma-folded W_b, W_o^T (f16).
//   sm103_tf32_stats  four threads per (line, position) slot in the node's
//                     orientation: LayerNorm statistics of the fp32 pair vector,
//                     the slot's row of the projection's LayerNorm K-step (tf32
//                     hi / lo parts of -mu and 1/rstd), and the pair bias of the
//                     4 heads (log2(e)-scaled f16; -30000 on masked and padded keys).
//   sm103_tf32_proj   persistent kind::tf32 GEMM, one 256-column half (q | k or
//                     v | g) per CTA with its 128 KB of weights resident, 128 slots
//                     per tile, K = 128 channels as 16 MMAs of 128 x 256 x 8 plus
//                     one K-step that adds -mu colsum + sd off; the epilogue scales
//                     by rstd and writes q, k, v^T and the sigmoid gate (f16) in the
//                     attention kernel's layouts.
//   sm103_attention   (fp32-output build, in sm103_kernels.cu), once per key chunk.
#include <atomic>
#include <cuda.h>
#include <cuda_fp16.h>

#include "sm103_ptx.cuh"
#include "tri_attn_internal.h"

namespace tri_attn {
namespace {

using namespace ptx;

constexpr int CZ = 128;                     // pair channels
constexpr int NH = 4;                       // heads
constexpr int HD = 32;                      // head dim
constexpr int CH = NH * HD;                 // 128 gated channels
constexpr int NPROJ = 4 * CH;               // 512 projection columns: q | k | v | g
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMaskedBias = -30000.f;

__device__ __forceinline__ void set_abort(volatile int* abort, uint32_t* status, uint32_t code) {
    *abort = 1;
    atomicOr(status, code);
}

__device__ __forceinline__ bool status_set(const uint32_t* status) {
    __shared__ int skip;
    if (threadIdx.x == 0) skip = *reinterpret_cast<const volatile uint32_t*>(status) != 0;
    __syncthreads();
    return skip != 0;
}

// x as hi + lo, both tf32 values (the sum is x to ~2^-22 relative)
__device__ __forceinline__ float2 split_tf32(float x) {
    const float h = tf32_round(x);
    return make_float2(h, tf32_round(x - h));
}

// =====================================================================================
// Weight preparation
// =====================================================================================
struct Tf32PrepArgs {
    const float *gamma, *beta, *b_g, *b_o;
    const float *w_q, *w_k, *w_v, *w_g, *w_b, *w_o;
    float* wprep;   // [512][128]: row n = tf32((gamma . W)[:, n] (x log2(e)/sqrt(d) for q)), K-major
    float* cst;     // [2][512]: column sum of the rounded row, then the offset
    float* wb;      // [128][4] gamma . W_b, then bcs[4] (column sums), bbw[4] (beta W_b)
    __half* wo_t;   // [128][128]: row n = W_o[:, n]
    float* bo;      // [128]
};

// Blocks 0..511: projection column n; 512..639: row of W_o^T; 640: the pair-bias weights.
__global__ void __launch_bounds__(128) sm103_tf32_prep(Tf32PrepArgs a) {
    __shared__ float red[2][4];
    const int n = blockIdx.x, c = threadIdx.x;
    if (n < NPROJ) {
        const int grp = n / CH, col = n % CH;      // q | k | v | g
        const float* W = grp == 0 ? a.w_q : grp == 1 ? a.w_k : grp == 2 ? a.w_v : a.w_g;
        const float sc = grp == 0 ? kLog2e * rsqrtf((float)HD) : 1.f;
        const float wv = W[c * CH + col] * sc;
        const float r = tf32_round(a.gamma[c] * wv);
        a.wprep[(size_t)n * CZ + c] = r;
        float wr = r, bw = a.beta[c] * wv;
        for (int o = 16; o; o >>= 1) {
            wr += __shfl_xor_sync(0xffffffffu, wr, o);
            bw += __shfl_xor_sync(0xffffffffu, bw, o);
        }
        if ((c & 31) == 0) {
            red[0][c >> 5] = wr;
            red[1][c >> 5] = bw;
        }
        __syncthreads();
        if (c == 0) {
            a.cst[n] = red[0][0] + red[0][1] + red[0][2] + red[0][3];
            a.cst[NPROJ + n] = red[1][0] + red[1][1] + red[1][2] + red[1][3] + (grp == 3 ? a.b_g[col] : 0.f);
        }
    } else if (n < NPROJ + CZ) {
        const int row = n - NPROJ;                 // output channel of W_o
        a.wo_t[row * CH + c] = __float2half_rn(a.w_o[(size_t)c * CZ + row]);
        if (c == 0) a.bo[row] = a.b_o ? a.b_o[row] : 0.f;
    } else {
        // gamma . W_b [128][4], its column sums and beta W_b (thread c owns channel c;
        // one warp reduction per head and a 4-way sum of the warps)
        __shared__ float part[2][4][NH];
        float* bcs = a.wb + CZ * NH;
        float* bbw = bcs + NH;
#pragma unroll
        for (int h = 0; h < NH; ++h) {
            const float wv = a.w_b[c * NH + h];
            float g = a.gamma[c] * wv, b = a.beta[c] * wv;
            a.wb[c * NH + h] = g;
            for (int o = 16; o; o >>= 1) {
                g += __shfl_xor_sync(0xffffffffu, g, o);
                b += __shfl_xor_sync(0xffffffffu, b, o);
            }
            if ((c & 31) == 0) {
                part[0][c >> 5][h] = g;
                part[1][c >> 5][h] = b;
            }
        }
        __syncthreads();
        if (c < 2 * NH) {
            const int which = c / NH, h = c % NH;
            const float t = part[which][0][h] + part[which][1][h] + part[which][2][h] + part[which][3][h];
            (which == 0 ? bcs : bbw)[h] = t;
        }
    }
}

// =====================================================================================
// LayerNorm statistics, the LayerNorm K-step rows, and the pair bias
// =====================================================================================
// Slot (L, x): position x of line L; its pair vector is Z[L, x] (starting node) or
// Z[x, L] (ending node).  Four threads per slot; thread q of a slot holds the
// 16-byte groups q, q + 4, ..., q + 28 (channels 4g .. 4g + 3 of group g), so each
// of the eight loads of a warp reads 64 contiguous bytes of each of its 8 pair
// vectors.  Partial sums are combined over the four threads; sums are shifted by
// the slot's first channel.
constexpr int kStatThreads = 256;
constexpr int kStatSlotsPerBlock = kStatThreads / 4;

__global__ void __launch_bounds__(kStatThreads) sm103_tf32_stats(const float* Z, int node, int I, int I_pad, float eps,
                                                                 const uint8_t* mask, const float* wb, float2* rowstat,
                                                                 uint4* ax0, uint4* ax1, __half* bias) {
    // (gamma W_b)[c][0..3] at c + c / 8: one 16-byte pad per 8 channels puts the four
    // channels that the four threads of a slot read at once in different banks
    __shared__ float4 swb[CZ + CZ / 8];
    __shared__ float sbc[2 * NH];
    for (int i = threadIdx.x; i < CZ; i += blockDim.x) swb[i + (i >> 3)] = reinterpret_cast<const float4*>(wb)[i];
    if (threadIdx.x < 2 * NH) sbc[threadIdx.x] = wb[CZ * NH + threadIdx.x];
    __syncthreads();
    const long long slot = (long long)blockIdx.x * kStatSlotsPerBlock + (threadIdx.x >> 2);
    const int qtr = threadIdx.x & 3;                 // 16-byte groups qtr + 4 i
    const long long n_slots = (long long)I * I_pad;
    const bool in = slot < n_slots;
    const int L = in ? (int)(slot / I_pad) : 0, x = in ? (int)(slot % I_pad) : 0;
    const bool live = in && x < I;
    const size_t pair = node == TRI_ATTN_STARTING ? (size_t)L * I + x : (size_t)x * I + L;
    const float4* src = reinterpret_cast<const float4*>(Z + pair * CZ) + qtr;
    float4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = live ? src[4 * i] : make_float4(0.f, 0.f, 0.f, 0.f);
    const float shift = __shfl_sync(0xffffffffu, v[0].x, threadIdx.x & 28);   // channel 0 of the slot
    float sd = 0.f, sq = 0.f, d[NH] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float z[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int ch = 4 * (qtr + 4 * i) + e;
            const float4 w = swb[ch + (ch >> 3)];
            const float dz = z[e] - shift;
            sd += dz;
            sq = fmaf(dz, dz, sq);
            d[0] = fmaf(z[e], w.x, d[0]);
            d[1] = fmaf(z[e], w.y, d[1]);
            d[2] = fmaf(z[e], w.z, d[2]);
            d[3] = fmaf(z[e], w.w, d[3]);
        }
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
        sd += __shfl_xor_sync(0xffffffffu, sd, o);
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
#pragma unroll
        for (int h = 0; h < NH; ++h) d[h] += __shfl_xor_sync(0xffffffffu, d[h], o);
    }
    if (!in) return;
    const float md = sd * (1.f / CZ);
    const float mu = live ? shift + md : 0.f;
    const float var = fmaxf(sq * (1.f / CZ) - md * md, 0.f) + eps;
    const float rstd = live ? rsqrtf(var) : 1.f;
    if (qtr == 0) {
        rowstat[slot] = make_float2(mu, rstd);
        const float2 m2 = split_tf32(-mu), s2 = split_tf32(live ? sqrtf(var) : 1.f);
        ax0[slot] = make_uint4(__float_as_uint(m2.x), __float_as_uint(m2.y), __float_as_uint(m2.x), __float_as_uint(m2.y));
        ax1[slot] = make_uint4(__float_as_uint(s2.x), __float_as_uint(s2.y), __float_as_uint(s2.x), __float_as_uint(s2.y));
    }
    // pair bias of head qtr (log2 units): rstd (z . gW_b - mu colsum) + beta W_b
    const bool valid = live && (mask == nullptr || mask[x] != 0);
    const float dh = qtr == 0 ? d[0] : qtr == 1 ? d[1] : qtr == 2 ? d[2] : d[3];
    const float bv = (rstd * (dh - mu * sbc[qtr]) + sbc[NH + qtr]) * kLog2e;
    bias[((size_t)qtr * I_pad + L) * I_pad + x] = __float2half_rn(valid ? bv : kMaskedBias);
}

// =====================================================================================
// Projection GEMM (kind::tf32): [128 slots x K = 128] x [128 x 256 columns], persistent
// =====================================================================================
// Same pipeline as the MSA row GEMM: A (Z, fp32) in K-chunks of 32 channels (16 KB)
// through a 5-slot ring, B resident (4 chunks x [256 rows x 128 B], 128 KB), a
// double-buffered 2 x 256-column TMEM accumulator, 8 epilogue warps of 128 columns.
// The LayerNorm K-step: ax (per tile, two 16-byte planes: (-mu hi, -mu lo) twice and
// (sd hi, sd lo) twice) against bx (per column: (cs hi, cs hi, cs lo, cs lo) and
// (off hi, off hi, off lo, off lo)); one K = 8 step covers both planes.
namespace kt {
constexpr int kThreads = 384;
constexpr int kEpiWarps = 8;
constexpr int kSlots = 5;
constexpr int kB = 0;
constexpr int kA = 131072;
constexpr int kBX = kA + kSlots * 16384;     // bx: 2 planes x [256 rows x 16 B]
constexpr int kAX = kBX + 8192;              // ax: 2 buffers x 2 planes x [128 rows x 16 B]
constexpr int kBar = kAX + 8192;
constexpr int kSmem = kBar + 256 + 1024;
static_assert(kSmem <= 232448, "dynamic shared memory above the per-block limit");
static_assert(kA % 1024 == 0 && kBX % 1024 == 0, "SW128 tiles need 1024-byte alignment");
}  // namespace kt

struct Tf32ProjParams {
    int node, I, I_pad, n_tiles;
    const float* cst;                        // [2][512]
    const float2* rowstat;                   // (mu, rstd) per slot
    const uint4 *ax0, *ax1;                  // the LayerNorm K-step rows per slot
    __half *q, *k, *vt, *g;                  // q, k, g: [I * 4][I_pad][32]; v^T: [I * 4][32][I_pad]
    uint32_t* status;
};

__global__ void __launch_bounds__(kt::kThreads, 1)
sm103_tf32_proj(const __grid_constant__ CUtensorMap mapZ, const __grid_constant__ CUtensorMap mapW,
                Tf32ProjParams p) {
    extern __shared__ uint8_t smem_raw[];
    if (status_set(p.status)) return;
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kt::kBar);
    uint64_t* b_full = bars + 0;
    uint64_t* a_full = bars + 1;      // [5]
    uint64_t* a_empty = bars + 6;     // [5]
    uint64_t* acc_full = bars + 11;   // [2]
    uint64_t* acc_empty = bars + 13;  // [2]
    uint64_t* ax_empty = bars + 15;   // [2]
    uint64_t* mma_done = bars + 17;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 18);
    volatile int* abort = reinterpret_cast<volatile int*>(bars + 19);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half_cols = blockIdx.x;         // 0: q | k, 1: v | g
    const int tpl = p.I_pad / 128;            // tiles per line
    if (threadIdx.x == 0) {
        mbar_init(b_full, 1);
        for (int q = 0; q < kt::kSlots; ++q) {
            mbar_init(a_full + q, 1);
            mbar_init(a_empty + q, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(acc_full + s, 1);
            mbar_init(acc_empty + s, kt::kEpiWarps);
            mbar_init(ax_empty + s, 1);
        }
        mbar_init(mma_done, 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp >= 4) {
        const int c = threadIdx.x - 128;      // column 0 .. 255 of this block: its bx rows
        const int n = half_cols * 256 + c;
        const float2 cs = split_tf32(p.cst[n]), of = split_tf32(p.cst[NPROJ + n]);
        reinterpret_cast<uint4*>(sm + kt::kBX)[c] =
            make_uint4(__float_as_uint(cs.x), __float_as_uint(cs.x), __float_as_uint(cs.y), __float_as_uint(cs.y));
        reinterpret_cast<uint4*>(sm + kt::kBX + 4096)[c] =
            make_uint4(__float_as_uint(of.x), __float_as_uint(of.x), __float_as_uint(of.y), __float_as_uint(of.y));
    }
    fence_proxy_async_smem();
    // Register split: launched at 168; the control warpgroup drops to 80, the two
    // epilogue warpgroups grow to 208 (128 x 80 + 256 x 208 = 63488 <= 384 x 168).
    if (warp < 4) setmaxnreg_dec<80>();
    if (warp == 1) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int issued = 0;
        bool ok = true;
        if (lane == 0) {
            prefetch_tmap(&mapZ);
            prefetch_tmap(&mapW);
            mbar_arrive_expect_tx(b_full, 131072);
            for (int kc = 0; kc < 4; ++kc)
                tma_load_2d(sm + kt::kB + kc * 32768, &mapW, b_full, kc * 32, half_cols * 256);
        }
        int j = 0;
        for (int t = blockIdx.y; ok && t < p.n_tiles; t += gridDim.y, ++j) {
            const int L = t / tpl, x0 = (t % tpl) * 128;
            ok = __all_sync(0xffffffffu, mbar_wait(ax_empty + (j & 1), ((j >> 1) & 1) ^ 1, abort));
            if (!ok) break;
            for (int kc = 0; kc < 4; ++kc) {
                const int q = issued % kt::kSlots, n = issued / kt::kSlots;
                ok = __all_sync(0xffffffffu, mbar_wait(a_empty + q, (n & 1) ^ 1, abort));
                if (!ok) break;
                if (lane == 0) {
                    uint8_t* dst = sm + kt::kA + q * 16384;
                    mbar_arrive_expect_tx(a_full + q, 16384 + (kc == 0 ? 4096 : 0));
                    if (kc == 0) {                   // this tile's ax planes ride on the first chunk
                        uint8_t* ax = sm + kt::kAX + (j & 1) * 4096;
                        bulk_load(ax, p.ax0 + (size_t)t * 128, 2048, a_full + q);
                        bulk_load(ax + 2048, p.ax1 + (size_t)t * 128, 2048, a_full + q);
                    }
                    if (p.node == TRI_ATTN_STARTING)
                        tma_load_3d(dst, &mapZ, a_full + q, kc * 32, x0, L);     // Z[L, x0 .. x0 + 127]
                    else
                        tma_load_3d(dst, &mapZ, a_full + q, kc * 32, L, x0);     // Z[x0 .. x0 + 127, L]
                }
                __syncwarp();
                ++issued;
            }
        }
        if (lane == 0) {
            volatile int keep_waiting = 0;
            mbar_wait(b_full, 0, &keep_waiting);
            if (!ok) {
                set_abort(abort, p.status, kStatusTimeoutProducer);
                for (int q = 0; q < kt::kSlots; ++q) {
                    const int cl = issued - 1 - ((issued - 1 - q) % kt::kSlots + kt::kSlots) % kt::kSlots;
                    if (cl >= 0) mbar_wait(a_full + q, (cl / kt::kSlots) & 1, &keep_waiting);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_tf32_f32(128, 256);
            bool ok = mbar_wait(b_full, 0, abort);
            const uint32_t bbase = smem_u32(sm + kt::kB);
            const uint64_t bxd = sdesc_noswizzle(smem_u32(sm + kt::kBX), 4096, 128);
            int used = 0, j = 0;
            for (int t = blockIdx.y; ok && t < p.n_tiles; t += gridDim.y, ++j) {
                const int ab = j & 1;
                if (!mbar_wait(acc_empty + ab, ((j >> 1) & 1) ^ 1, abort)) {
                    ok = false;
                    break;
                }
                for (int kc = 0; kc < 4; ++kc, ++used) {
                    const int q = used % kt::kSlots, n = used / kt::kSlots;
                    if (!mbar_wait(a_full + q, n & 1, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (kc == 0)                                    // -mu colsum + sd off
                        mma_ss_tf32(tmem + ab * 256, sdesc_noswizzle(smem_u32(sm + kt::kAX + (j & 1) * 4096), 2048, 128),
                                    bxd, idesc, 0u);
                    const uint32_t abase = smem_u32(sm + kt::kA + q * 16384);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = sdesc(abase + kk * 32, 1024, kSwizzle128);
                        const uint64_t bd = sdesc(bbase + kc * 32768 + kk * 32, 1024, kSwizzle128);
                        mma_ss_tf32(tmem + ab * 256, ad, bd, idesc, 1u);
                    }
                    tc_commit(a_empty + q);
                }
                if (!ok) break;
                tc_commit(ax_empty + (j & 1));
                tc_commit(acc_full + ab);
            }
            if (!ok) set_abort(abort, p.status, kStatusTimeoutMma);
            tc_commit(mma_done);
            volatile int keep_waiting = 0;
            mbar_wait(mma_done, 0, &keep_waiting);
        }
        __syncwarp();
    } else if (warp >= 4) {
        setmaxnreg_inc<208>();
        // ------------------------------------------------------------ epilogue: thread = slot, 128 columns
        const int wq = warp & 3, half = (warp - 4) >> 2;
        const int which = half_cols * 2 + half;   // 0 q, 1 k, 2 v, 3 gate
        const int r = wq * 32 + lane;
        const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16) + half * 128;
        float rstd = p.n_tiles > blockIdx.y ? p.rowstat[(size_t)blockIdx.y * 128 + r].y : 1.f;
        int j = 0;
        bool ok = true;
        for (int t = blockIdx.y; t < p.n_tiles; t += gridDim.y, ++j) {
            const int ab = j & 1;
            const int L = t / tpl, x = (t % tpl) * 128 + r;
            const float cur_rstd = rstd;
            if (!mbar_wait(acc_full + ab, (j >> 1) & 1, abort)) { ok = false; break; }
            tc_fence_after();
            uint32_t acc[2][64];
            tmem_ld64(tl + ab * 256, acc[0]);
            tmem_ld64(tl + ab * 256 + 64, acc[1]);
            tmem_ld_wait();
            tmem_regs_ready(acc[0]);
            tmem_regs_ready(acc[1]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty + ab);
            if (t + (int)gridDim.y < p.n_tiles) rstd = p.rowstat[(size_t)(t + gridDim.y) * 128 + r].y;
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                const uint32_t* a = &acc[h >> 1][(h & 1) * 32];
                uint32_t o[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float v0 = cur_rstd * __uint_as_float(a[e]), v1 = cur_rstd * __uint_as_float(a[e + 1]);
                    o[e >> 1] = which == 3 ? sigmoid_f16x2(v0, v1) : pack_f16(v0, v1);
                }
                const size_t lh = (size_t)L * NH + h;
                if (which == 2) {
                    unsigned short* dst = reinterpret_cast<unsigned short*>(p.vt + lh * HD * p.I_pad + x);
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        dst[(size_t)e * p.I_pad] = static_cast<unsigned short>(o[e >> 1] & 0xFFFFu);
                        dst[(size_t)(e + 1) * p.I_pad] = static_cast<unsigned short>(o[e >> 1] >> 16);
                    }
                } else {
                    __half* base = which == 0 ? p.q : which == 1 ? p.k : p.g;
                    uint4* dst = reinterpret_cast<uint4*>(base + (lh * p.I_pad + x) * HD);
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
                        dst[c4] = make_uint4(o[4 * c4], o[4 * c4 + 1], o[4 * c4 + 2], o[4 * c4 + 3]);
                }
            }
        }
        if (!ok) set_abort(abort, p.status, kStatusTimeoutEpilogue);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

int num_sms_of_device() {
    static std::atomic<int> cache[64];
    int dev = 0;
    cudaGetDevice(&dev);
    int n = (dev >= 0 && dev < 64) ? cache[dev].load(std::memory_order_relaxed) : 0;
    if (!n) {
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
        if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

}  // namespace

bool sm103_tf32_supported(int c_z, int H, int d, int dtype) {
    return dtype == TRI_ATTN_TF32 && c_z == CZ && H == NH && d == HD;
}

cudaError_t sm103_tf32_forward(const FwdArgs& a, cudaStream_t s, LaunchTimer* tm) {
    const Workspace& W = *a.lay;
    char* ws = a.ws;
    auto hf = [&](size_t off) { return reinterpret_cast<__half*>(ws + off); };
    auto f32 = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
    const int I = a.I, Ip = a.I_pad;
    const size_t P = (size_t)I * Ip;
    cudaError_t e;

    static std::atomic<uint64_t> attr_set{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t dev_bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
    if (!(attr_set.load(std::memory_order_acquire) & dev_bit)) {
        if ((e = cudaFuncSetAttribute(sm103_tf32_proj, cudaFuncAttributeMaxDynamicSharedMemorySize, kt::kSmem)) !=
            cudaSuccess)
            return e;
        attr_set.fetch_or(dev_bit, std::memory_order_release);
    }

    // ---- weights
    Tf32PrepArgs pa{a.w.ln_gamma, a.w.ln_beta, a.w.b_g, a.w.b_o,
                    static_cast<const float*>(a.w.w_q), static_cast<const float*>(a.w.w_k),
                    static_cast<const float*>(a.w.w_v), static_cast<const float*>(a.w.w_g),
                    static_cast<const float*>(a.w.w_b), static_cast<const float*>(a.w.w_o),
                    f32(W.wprep), f32(W.cst), f32(W.wb32), hf(W.wo_t), f32(W.bo)};
    if (tm) tm->begin("sm103_tf32_prep", s);
    sm103_tf32_prep<<<NPROJ + CZ + 1, 128, 0, s>>>(pa);
    if (tm) tm->end(s);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    // ---- LayerNorm statistics, K-step rows, pair bias
    uint4* ax0 = reinterpret_cast<uint4*>(ws + W.axrow);
    uint4* ax1 = ax0 + P;
    {
        const long long blocks = ((long long)P + kStatSlotsPerBlock - 1) / kStatSlotsPerBlock;
        if (tm) tm->begin("sm103_tf32_stats", s);
        sm103_tf32_stats<<<(unsigned)blocks, kStatThreads, 0, s>>>(
            static_cast<const float*>(a.Z), a.node, I, Ip, a.eps, a.mask, f32(W.wb32),
            reinterpret_cast<float2*>(ws + W.rowstat), ax0, ax1, hf(W.bias));
        if (tm) tm->end(s);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }

    // ---- projection GEMM (kind::tf32)
    {
        CUtensorMap mZ, mW;
        const uint64_t zd[3] = {CZ, (uint64_t)I, (uint64_t)I};
        const uint64_t zs[2] = {(uint64_t)CZ * 4, (uint64_t)I * CZ * 4};
        const uint32_t zb_start[3] = {32, 128, 1}, zb_end[3] = {32, 1, 128};
        const uint64_t wd[2] = {CZ, NPROJ};
        const uint64_t wst[1] = {(uint64_t)CZ * 4};
        const uint32_t wbx[2] = {32, 256};
        if (!sm103_map_f32(&mZ, a.Z, 3, zd, zs, a.node == TRI_ATTN_STARTING ? zb_start : zb_end, 128) ||
            !sm103_map_f32(&mW, f32(W.wprep), 2, wd, wst, wbx, 128))
            return cudaErrorInvalidValue;
        Tf32ProjParams pp{};
        pp.node = a.node;
        pp.I = I;
        pp.I_pad = Ip;
        pp.n_tiles = I * (Ip / 128);
        pp.cst = f32(W.cst);
        pp.rowstat = reinterpret_cast<const float2*>(ws + W.rowstat);
        pp.ax0 = ax0;
        pp.ax1 = ax1;
        pp.q = hf(W.q);
        pp.k = hf(W.k);
        pp.vt = hf(W.v);
        pp.g = hf(W.g);
        pp.status = a.status;
        const int rows = num_sms_of_device() / 2 > 0 ? num_sms_of_device() / 2 : 1;
        dim3 grid(2, rows < pp.n_tiles ? rows : pp.n_tiles);
        if (tm) tm->begin("sm103_tf32_proj", s);
        sm103_tf32_proj<<<grid, kt::kThreads, kt::kSmem, s>>>(mZ, mW, pp);
        if (tm) tm->end(s);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }

    // ---- attention, gate, output projection (fp32 out), once per key chunk
    TriAttnLaunch l;
    l.node = a.node;
    l.I = I;
    l.I_pad = Ip;
    l.key_chunks = a.key_chunks;
    l.inject = a.inject;
    l.f32 = true;
    l.mask = a.mask;
    l.pair_mask = a.pair_mask;
    l.Z_resid = a.residual ? a.Z : nullptr;
    l.out = a.out;
    l.q = hf(W.q);
    l.k = hf(W.k);
    l.vt = hf(W.v);
    l.g = hf(W.g);
    l.bias = hf(W.bias);
    l.wo_t = hf(W.wo_t);
    l.bo = f32(W.bo);
    l.o_run = W.o_run ? f32(W.o_run) : nullptr;
    l.lse_run = W.lse_run ? f32(W.lse_run) : nullptr;
    l.kbits = reinterpret_cast<uint64_t*>(ws + W.kbits);
    l.work = reinterpret_cast<int*>(ws + W.work);
    l.status = a.status;
    return sm103_triangle_attention(l, s, tm);
}

}  // namespace tri_attn
