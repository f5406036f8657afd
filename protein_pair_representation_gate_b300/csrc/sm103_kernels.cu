// sm_103a tensor-core path of the gated triangle attention (bf16 Z, weights
// and output; fp32 accumulation; c_z = 128, H = 4, d = 32).
//
// Intermediates (q, k, v, gate, pair bias, P, gated u, W_o) are stored in
// f16, not bf16: they are LayerNorm-bounded, so f16's range suffices, and its
// 11-bit significand keeps the error of the biased softmax (whose exponents
// reach |bias| ~ 30 in log2 units with the amplified-bias workload) inside the
// bf16 output's own rounding error.  Each MMA has both operands of one type:
// bf16 x bf16 for the projection GEMM, f16 x f16 for the attention.
//
// Three kernels per forward (the attention kernel once per key chunk):
//
//   sm103_prep      folds LayerNorm's gamma into the projection weights and
//                   precomputes the per-column constants that let the
//                   projection GEMM run on the raw pair vectors:
//                     LN(z) W = rstd * (z (gamma.W) - mu * colsum(gamma.W)) + beta W
//   sm103_ln_proj   persistent; per tile of 128 pair vectors on one line:
//                   TMA load of Z (128B swizzle), tcgen05 MMA z x [Wq|Wv|Wk|Wg]
//                   (M=128, N=2x256, K=128) into TMEM, LayerNorm statistics
//                   and the pair bias on CUDA cores, four epilogue warpgroups
//                   writing q (scaled by log2(e)/sqrt(d)), k and the sigmoid
//                   gate through TMA stores, v^T, and the log2(e)-scaled pair
//                   bias (a finite -30000 on masked keys), all in f16.
//   sm103_attention persistent, one CTA per SM, claiming work items (a line
//                   and 256 queries) from a counter; two softmax warpgroups
//                   (128 queries each), each with its own MMA-issuing warp:
//                   S = Q K^T + Bias I (tcgen05 into TMEM; Q copied once per
//                   head into TMEM, the staged bias tile as an A operand
//                   against an identity), online softmax with lazy rescaling,
//                   P (f16) written back into TMEM over S, O += P V (A operand
//                   from TMEM), then normalise, gate, and the output projection
//                   (u W_o, A operand from TMEM) with the token mask, stored in
//                   the node's orientation.  The I x I score matrix of a line
//                   is never materialised.  A second build of this kernel
//                   serves calls with an [I, I] pair mask (one more K-step adds
//                   -30000 on the line's excluded keys) or a residual (Z + out).
//   sm103_pair_keybits  (with a pair mask only) packs each line's admitted
//                   keys into 64-bit words for the attention kernel.
//
// Sources: the operation as stated in tri_attn.h (Dell page, Evoformer
// paragraph; Intel page, steps 2 and 4: bias term and fusing it into the
// score contraction); OpenFold-TRT summary, Methodology: 16-bit core, fused
// kernels; Design-CP summary, Methodology 1: key/value pieces with scores
// formed on the fly and a log-sum-exp merge across key chunks.
#include <atomic>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <cstdio>

#include "sm103_ptx.cuh"
#include "tri_attn_internal.h"

namespace tri_attn {
namespace {

using namespace ptx;

constexpr int CZ = 128;            // pair channels
constexpr int NH = 4;              // heads
constexpr int HD = 32;             // head dim
constexpr int CH = NH * HD;        // 128 gated channels
constexpr int NPROJ = 4 * CH;      // 512 MMA output columns in four groups of 128
// Order of the groups in the prepared weights and the accumulator: the first
// 256 columns (q | v) go to epilogue warpgroup 0, the last 256 (k | g, plus the
// pair bias computed on CUDA cores) to warpgroup 1, which balances their work.
constexpr int kGroupQ = 0, kGroupV = 1, kGroupK = 2, kGroupG = 3;
constexpr int NCONST = NPROJ + NH; // + pair bias columns
constexpr float kLog2e = 1.4426950408889634f;
// Pair bias of a masked or padded key, log2 units.  Finite (not -inf) because the
// bias enters S through an MMA with an identity matrix, where 0 x -inf would be
// NaN; 2^-30000 is exactly 0 in fp32, so such keys still get probability 0 (and
// if every key so far was masked, the first real key's rescale factor 2^-30000
// removes their contribution exactly).
constexpr float kMaskedBias = -30000.f;
constexpr float kMfloor = -1e30f;           // finite floor of the attention kernel's running max

// Block-uniform read of the device status word (one thread reads, all see the
// same value), so an early return never splits a block at a later barrier.
__device__ __forceinline__ bool status_set(const uint32_t* status) {
    __shared__ int skip;
    if (threadIdx.x == 0) skip = *reinterpret_cast<const volatile uint32_t*>(status) != 0;
    __syncthreads();
    return skip != 0;
}

__device__ __forceinline__ void set_abort(volatile int* abort, uint32_t* status, uint32_t code) {
    *abort = 1;
    atomicOr(status, code);
}

// =====================================================================================
// Weight preparation
// =====================================================================================
struct PrepArgs {
    const float *gamma, *beta, *b_o, *b_g;
    const __nv_bfloat16 *w_q, *w_k, *w_v, *w_g, *w_b, *w_o;
    __nv_bfloat16* wprep;   // [512][128]  row n = (gamma . W)[:, n], K-major for the MMA
    float* colsum;          // [516]       sum_c of the (rounded) gamma.W column
    float* betaw;           // [516]       sum_c beta_c W[c, n]
    float* wb32;            // [128][4]    gamma . W_b in fp32
    __half* wo_t;           // [128][128]  W_o transposed (f16): row n = W_o[:, n]
    float* bo;              // [128]
    float* cst;             // [256][4]    per column pair {colsum(n), colsum(n+1), off(n), off(n+1)},
                            //             off = scale * beta W (+ b_g for the gate group)
};

__global__ void __launch_bounds__(128) sm103_prep(PrepArgs a) {
    __shared__ float red[2][4];
    const int n = blockIdx.x, c = threadIdx.x;
    if (n < NCONST) {
        float wr, bw;
        if (n < NPROJ) {
            const int which = n / CH, col = n % CH;   // row groups q | v | k | g (see kGroup*)
            const __nv_bfloat16* W = which == kGroupQ ? a.w_q : which == kGroupK ? a.w_k : which == kGroupV ? a.w_v : a.w_g;
            const float wv = __bfloat162float(W[c * CH + col]);
            const __nv_bfloat16 r = __float2bfloat16_rn(a.gamma[c] * wv);
            a.wprep[n * CZ + c] = r;
            wr = __bfloat162float(r);
            bw = a.beta[c] * wv;
        } else {
            const int h = n - NPROJ;
            const float wv = __bfloat162float(a.w_b[c * NH + h]);
            wr = a.gamma[c] * wv;
            a.wb32[c * NH + h] = wr;
            bw = a.beta[c] * wv;
        }
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
            const float cs = red[0][0] + red[0][1] + red[0][2] + red[0][3];
            const float bw = red[1][0] + red[1][1] + red[1][2] + red[1][3];
            a.colsum[n] = cs;
            a.betaw[n] = bw;
            if (n < NPROJ) {
                const int which = n / CH;
                const float sc = which == kGroupQ ? kLog2e * rsqrtf((float)HD) : 1.f;
                const float off = bw * sc + (which == kGroupG ? a.b_g[n % CH] : 0.f);
                a.cst[(n >> 1) * 4 + (n & 1)] = cs;
                a.cst[(n >> 1) * 4 + 2 + (n & 1)] = off;
            }
        }
    } else {
        const int row = n - NCONST;           // output channel of W_o
        a.wo_t[row * CH + c] = __float2half_rn(__bfloat162float(a.w_o[c * CZ + row]));
        if (c == 0) a.bo[row] = a.b_o ? a.b_o[row] : 0.f;
    }
}

// =====================================================================================
// LayerNorm + projections
// =====================================================================================
struct ProjParams {
    int node, I, I_pad, ntx, ntiles;
    float eps;
    const uint8_t* mask;
    const float *colsum, *betaw, *wb32, *cst;
    __half *q, *k, *vt, *g, *bias;     // f16 intermediates
    uint32_t* status;
};

namespace k1 {
constexpr int kThreads = 576;                // 4 epilogue warpgroups + producer warp + MMA warp
constexpr int kProducerWarp = 16, kMmaWarp = 17;
constexpr int kW = 0;                        // 4 x 32 KB: [half(qk|vg)][k-half][256 rows][128 B]
constexpr int kZ = 131072;                   // 2 stages x 32 KB: [k-half][128 rows][128 B]
constexpr int kConst = kZ + 2 * 32768;       // cst[256][4], wb32[128][4], bias colsum[4], bias offset[4]
constexpr int kConstBytes = (256 * 4 + CZ * NH + 2 * NH) * 4;
constexpr int kBar = kConst + ((kConstBytes + 127) / 128) * 128;
// Output staging for the TMA stores of q, k and g: one 32-row x 64-byte box (64-byte
// swizzle) per warp of those three warpgroups.
constexpr int kStg = ((kBar + 256 + 1023) / 1024) * 1024;
constexpr int kStgWarp = 2048;
constexpr int kStat = kStg + 12 * kStgWarp;  // (mu, rstd) of the tile's 128 rows, 2 buffers (warpgroup 0 -> 1..3)
constexpr int kSmem = kStat + 2 * 128 * 8 + 1024;   // + alignment slack
static_assert(kSmem <= 232448, "dynamic shared memory above the per-block limit");
}  // namespace k1

__global__ void __launch_bounds__(k1::kThreads, 1)
sm103_ln_proj(const __grid_constant__ CUtensorMap mapZs, const __grid_constant__ CUtensorMap mapZe,
              const __grid_constant__ CUtensorMap mapW, const __grid_constant__ CUtensorMap mapQs,
              const __grid_constant__ CUtensorMap mapKs, const __grid_constant__ CUtensorMap mapGs, ProjParams p) {
    extern __shared__ uint8_t smem_raw[];
    if (status_set(p.status)) return;          // an earlier wait gave up: fail fast
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* s_cst = reinterpret_cast<float*>(sm + k1::kConst);   // [256][4]
    float* s_wbt = s_cst + 256 * 4;        // [4 heads][128 channels]: (gamma . W_b)^T
    float* s_bcs = s_wbt + CZ * NH;        // [4] pair-bias column sums
    float* s_bbw = s_bcs + NH;             // [4] pair-bias beta W
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + k1::kBar);
    uint64_t* w_full = bars + 0;
    uint64_t* z_full = bars + 1;      // [2]
    uint64_t* z_empty = bars + 3;     // [2]
    uint64_t* acc_full = bars + 5;    // [2] per half
    uint64_t* acc_empty = bars + 7;   // [2]
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 10);
    volatile int* abort = reinterpret_cast<volatile int*>(bars + 11);
    uint64_t* stat_full = bars + 12;  // [2]: warpgroup 0 has written the tile's (mu, rstd)
    float2* s_stat = reinterpret_cast<float2*>(sm + k1::kStat);   // [2][128]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < 256 * 4; i += blockDim.x) s_cst[i] = p.cst[i];
    for (int i = threadIdx.x; i < CZ * NH; i += blockDim.x) s_wbt[(i % NH) * CZ + i / NH] = p.wb32[i];
    if (threadIdx.x < NH) {
        s_bcs[threadIdx.x] = p.colsum[NPROJ + threadIdx.x];
        s_bbw[threadIdx.x] = p.betaw[NPROJ + threadIdx.x];
    }
    if (threadIdx.x == 0) {
        mbar_init(w_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(z_full + s, 1);
            mbar_init(z_empty + s, 1 + 16);       // MMA commit + 16 epilogue warps
            mbar_init(acc_full + s, 1);
            mbar_init(acc_empty + s, 8);          // the two warpgroups reading this half
            mbar_init(stat_full + s, 4);          // the four warps of warpgroup 0
        }
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == k1::kMmaWarp) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == k1::kProducerWarp) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&mapZs);
            prefetch_tmap(&mapZe);
            prefetch_tmap(&mapW);
            mbar_arrive_expect_tx(w_full, 4 * 32768);
            for (int h2 = 0; h2 < 2; ++h2)
                for (int kh = 0; kh < 2; ++kh)
                    tma_load_2d(sm + k1::kW + (h2 * 2 + kh) * 32768, &mapW, w_full, kh * 64, h2 * 256);
            int j = 0;
            for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++j) {
                const int s = j & 1;
                if (!mbar_wait(z_empty + s, ((j >> 1) & 1) ^ 1, abort)) {
                    set_abort(abort, p.status, kStatusTimeoutProducer);
                    break;
                }
                const int L = t / p.ntx, x0 = (t % p.ntx) * 128;
                mbar_arrive_expect_tx(z_full + s, 32768);
                for (int b = 0; b < 2; ++b) {
                    uint8_t* dst = sm + k1::kZ + s * 32768 + b * 16384;
                    if (p.node == TRI_ATTN_STARTING)
                        tma_load_3d(dst, &mapZs, z_full + s, b * 64, x0, L);
                    else
                        tma_load_3d(dst, &mapZe, z_full + s, b * 64, L, x0);
                }
            }
        }
    } else if (warp == k1::kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, 256);
            bool ok = mbar_wait(w_full, 0, abort);
            int j = 0;
            for (int t = blockIdx.x; ok && t < p.ntiles; t += gridDim.x, ++j) {
                const int s = j & 1;
                if (!mbar_wait(z_full + s, (j >> 1) & 1, abort)) { ok = false; break; }
                for (int h2 = 0; h2 < 2; ++h2) {
                    if (!mbar_wait(acc_empty + h2, (j & 1) ^ 1, abort)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t zbase = smem_u32(sm + k1::kZ + s * 32768);
                    const uint32_t wbase = smem_u32(sm + k1::kW + h2 * 2 * 32768);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t ad = sdesc(zbase + (kk >> 2) * 16384 + (kk & 3) * 32, 1024, kSwizzle128);
                        const uint64_t bd = sdesc(wbase + (kk >> 2) * 32768 + (kk & 3) * 32, 1024, kSwizzle128);
                        mma_ss(tmem + h2 * 256, ad, bd, idesc, kk > 0);
                    }
                    tc_commit(acc_full + h2);
                }
                if (!ok) break;
                tc_commit(z_empty + s);
            }
            if (!ok) set_abort(abort, p.status, kStatusTimeoutMma);
        }
    } else {
        // ------------------------------------------------------------ epilogue warpgroups
        // Warpgroup w owns accumulator columns 128 w .. 128 w + 127, i.e. projection
        // group w (q, v, k, g), and the pair bias of head w.
        const int wg = warp >> 2;
        const int wq = warp & 3;                 // TMEM lane quarter
        const int r = wq * 32 + lane;            // row = pair within the tile
        const int half = wg >> 1;                // accumulator half (q|v or k|g)
        const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16) + wg * 128;
        const float* wbt = s_wbt + wg * CZ;
        uint8_t* stg = sm + k1::kStg + ((wg == kGroupQ ? 0 : wg - 1) * 4 + wq) * k1::kStgWarp;   // unused by v
        int j = 0;
        for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++j) {
            const int s = j & 1;
            const int L = t / p.ntx, x = (t % p.ntx) * 128 + r;
            if (!mbar_wait(z_full + s, (j >> 1) & 1, abort)) {
                set_abort(abort, p.status, kStatusTimeoutEpilogue);
                break;
            }
            // Warpgroup 0 forms the LayerNorm statistics of the raw pair vector in one
            // pass over its SMEM row, shifted by its first channel (exact algebra; avoids
            // cancellation when the mean is large against the spread), and hands them to
            // the other three through shared memory; every warpgroup forms
            // z . (gamma W_b)[:, wg] for its head in its own pass.  The other warpgroups
            // release the Z stage only after reading the statistics, so the buffer of
            // tile j is rewritten (at tile j + 2, after that stage's release) only once
            // all have read it.
            const uint8_t* zb = sm + k1::kZ + s * 32768 + r * 128;
            float mu, rstd, bh = 0.f;
            if (wg == 0) {
                const float shift = bf16lo(*reinterpret_cast<const uint32_t*>(zb + ((0 ^ (r & 7)) << 4)));
                float sd = 0.f, sq = 0.f;
#pragma unroll 2
                for (int cc = 0; cc < 16; ++cc) {
                    const int b = cc >> 3, c = cc & 7;
                    const uint4 v = *reinterpret_cast<const uint4*>(zb + b * 16384 + ((c ^ (r & 7)) << 4));
                    const float4 wa = *reinterpret_cast<const float4*>(wbt + cc * 8);
                    const float4 wb = *reinterpret_cast<const float4*>(wbt + cc * 8 + 4);
                    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
                    const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2) {
                        const float z0 = bf16lo(w4[q2]), z1 = bf16hi(w4[q2]);
                        const float d0 = z0 - shift, d1 = z1 - shift;
                        sd += d0 + d1;
                        sq = fmaf(d0, d0, fmaf(d1, d1, sq));
                        bh = fmaf(z0, wv[2 * q2], fmaf(z1, wv[2 * q2 + 1], bh));
                    }
                }
                const float md = sd * (1.f / CZ);
                mu = shift + md;
                const float var = fmaxf(sq * (1.f / CZ) - md * md, 0.f);
                rstd = rsqrtf(var + p.eps);
                s_stat[s * 128 + r] = make_float2(mu, rstd);
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(stat_full + s);
                    mbar_arrive(z_empty + s);
                }
            } else {
#pragma unroll 2
                for (int cc = 0; cc < 16; ++cc) {
                    const int b = cc >> 3, c = cc & 7;
                    const uint4 v = *reinterpret_cast<const uint4*>(zb + b * 16384 + ((c ^ (r & 7)) << 4));
                    const float4 wa = *reinterpret_cast<const float4*>(wbt + cc * 8);
                    const float4 wb = *reinterpret_cast<const float4*>(wbt + cc * 8 + 4);
                    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
                    const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2)
                        bh = fmaf(bf16lo(w4[q2]), wv[2 * q2], fmaf(bf16hi(w4[q2]), wv[2 * q2 + 1], bh));
                }
                if (!mbar_wait(stat_full + s, (j >> 1) & 1, abort)) {
                    set_abort(abort, p.status, kStatusTimeoutEpilogue);
                    break;
                }
                const float2 st = s_stat[s * 128 + r];
                mu = st.x;
                rstd = st.y;
                __syncwarp();
                if (lane == 0) mbar_arrive(z_empty + s);
            }
            {
                // pair bias of head wg: rstd * (z . gW_b[:, h] - mu * colsum) + beta W_b, in log2 units
                const bool valid = x < p.I && (p.mask == nullptr || p.mask[x] != 0);
                const float v = (fmaf(bh, rstd, -mu * rstd * s_bcs[wg]) + s_bbw[wg]) * kLog2e;
                p.bias[((size_t)wg * p.I_pad + L) * p.I_pad + x] = __float2half_rn(valid ? v : kMaskedBias);
            }

            if (!mbar_wait(acc_full + half, j & 1, abort)) {
                set_abort(abort, p.status, kStatusTimeoutEpilogue);
                break;
            }
            tc_fence_after();
            // 32 accumulator columns (one head) -> normalised, transformed f16 values ->
            // global.  value = r * (acc - mu * colsum) + off, two columns per packed FMA,
            // with r = rstd (times log2(e)/sqrt(d) for q) and off from the prepared constants.
            const float rr = wg == kGroupQ ? rstd * (kLog2e * rsqrtf((float)HD)) : rstd;
            const float nmu = -mu;
#pragma unroll 1
            for (int h = 0; h < NH; ++h) {
                uint32_t acc[32];
                tmem_ld32(tl + h * 32, acc);
                tmem_ld_wait();
                const float4* cst = reinterpret_cast<const float4*>(s_cst) + ((wg * 128 + h * 32) >> 1);
                uint32_t o[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float4 c = cst[e >> 1];
                    float t0, t1, v0, v1;
                    fma2(t0, t1, nmu, nmu, c.x, c.y, __uint_as_float(acc[e]), __uint_as_float(acc[e + 1]));
                    fma2(v0, v1, rr, rr, t0, t1, c.z, c.w);
                    if (wg == kGroupG) {                  // sigmoid(v) = 0.5 tanh(v / 2) + 0.5
                        v0 = fmaf(0.5f, tanh_approx(0.5f * v0), 0.5f);
                        v1 = fmaf(0.5f, tanh_approx(0.5f * v1), 0.5f);
                    }
                    o[e >> 1] = pack_f16(v0, v1);
                }
                const size_t lh = (size_t)L * NH + h;
                if (wg == kGroupV) {
                    unsigned short* dst = reinterpret_cast<unsigned short*>(p.vt + lh * HD * p.I_pad + x);
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        dst[(size_t)e * p.I_pad] = static_cast<unsigned short>(o[e >> 1] & 0xFFFFu);
                        dst[(size_t)(e + 1) * p.I_pad] = static_cast<unsigned short>(o[e >> 1] >> 16);
                    }
                } else {
                    // q, k, g rows of head h: [line * 4 + h][x][32], written through this
                    // warp's staging box (row lane, 16-byte chunk c at c ^ ((lane >> 1) & 3))
                    // and one TMA store.  The box is rewritten only after the previous
                    // store has read it.
                    if (lane == 0) bulk_wait_read0();
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4*>(stg + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) =
                            make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const CUtensorMap* m = wg == kGroupQ ? &mapQs : (wg == kGroupK ? &mapKs : &mapGs);
                        tma_store_2d(m, stg, 0, static_cast<int>(lh * p.I_pad) + x - lane);
                        bulk_commit();
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty + half);
        }
        if (lane == 0) bulk_wait0();              // this warp's stores complete before exit
    }
    tc_fence_before();
    __syncthreads();
    if (warp == k1::kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// =====================================================================================
// Attention
// =====================================================================================
struct AttnParams {
    int node, I, I_pad, nk, k_begin, k_end, first, last;
    int n_xb, lines, n_items;  // work items: (256-query block, line[, head half]); item = xb + n_xb (L + lines z)
    int* work;                 // next unclaimed work item (zero at launch)
    __half* u;                 // MSA build: gated outputs [lines][I_pad][8 x 32] (f16), written per head
    int inject;                // test hook: the CTA holding item 0 skips the load of its stage 1
    const uint8_t* mask;
    const uint8_t* pmask;      // [I, I] pair mask over the pairs of Z, or NULL
    const uint64_t* kbits;     // [I][I_pad / 64 + 1] key-valid bits per line (with pmask), or NULL
    const __half* g;
    const float* bo;
    float *o_run, *lse_run;
    const void* Z;             // residual source (NULL: write the update only); may equal out
    void* out;                 // bf16, or fp32 in the kF32 build
    uint32_t* status;
};

// Key-valid bits of each line under a pair mask: bit kk of word w of line L is
// set when key w*64 + kk < I and the pair mask admits it on that line (starting
// node: M[L, key]; ending node: M[key, L]).  One extra zero word per line lets a
// key tile that starts off a 64-key boundary (key chunks) read two words.
__global__ void __launch_bounds__(256) sm103_pair_keybits(const uint8_t* pm, int node, int I, int lines, int words,
                                                          uint64_t* kbits) {
    // one warp per (line, word): lane l tests keys w*64 + 2l and + 1, two ballots
    // give the word's even and odd bits
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= (long long)lines * words) return;   // whole warps
    const int L = (int)(wid / words), w = (int)(wid % words);
    auto admitted = [&](int key) -> bool {
        if (key >= I) return false;
        return (node == TRI_ATTN_STARTING ? pm[(size_t)L * I + key] : pm[(size_t)key * I + L]) != 0;
    };
    const int key = w * 64 + 2 * lane;
    const uint32_t ev = __ballot_sync(0xffffffffu, admitted(key));
    const uint32_t od = __ballot_sync(0xffffffffu, admitted(key + 1));
    if (lane == 0) {
        auto spread = [](uint32_t v) -> uint64_t {        // bit i -> bit 2i
            uint64_t x = v;
            x = (x | (x << 16)) & 0x0000FFFF0000FFFFull;
            x = (x | (x << 8)) & 0x00FF00FF00FF00FFull;
            x = (x | (x << 4)) & 0x0F0F0F0F0F0F0F0Full;
            x = (x | (x << 2)) & 0x3333333333333333ull;
            x = (x | (x << 1)) & 0x5555555555555555ull;
            return x;
        };
        kbits[wid] = spread(ev) | (spread(od) << 1);
    }
}

namespace k2 {
constexpr int kThreads = 384;                // control warpgroup (producer, 2 MMA issuers, 1 idle) + 2 softmax warpgroups
constexpr int kKT = 64;                      // keys per stage (one S sub-tile)
// K and V' of a key tile live in a ring shared by both groups (freed when both
// groups' P V' has read it); each group's bias tiles live in a ring of its own,
// freed as soon as that group's S has read it, so the groups do not hold each
// other's loads back.
constexpr int kStages = 5;                   // K / V' ring: stage = it % 5, phase = (it / 5) & 1
constexpr int kBStages = 3;                  // bias ring per group: stage = it % 3, phase = (it / 3) & 1
constexpr int kQ = 0;                        // [2 bufs][2 tiles][128 x 64 B] (SW64)
constexpr int kStage = 32768;
constexpr int kSK = 0;                       // K tile: 64 keys x 64 B (SW64)
constexpr int kSV = 4096;                    // V' tile: 32 rows V^T + 16 more rows (below), 128 B each (SW128)
constexpr int kSM = kSV + 4096;              // rows 32..39 of V': M, the pair-mask row (64 keys x 16 B, no swizzle)
constexpr int kStageBytes = 10240;
constexpr int kStageTx = 4096 + 4096;        // bytes the TMA writes per K / V' stage
constexpr int kBias = kStage + kStages * kStageBytes;    // [2 groups][4] bias tiles: 128 rows x 128 B (SW128)
constexpr int kBiasBytes = 16384;
// The kernel comes in two builds: the plain forward (kEx = false) and the one
// with a pair mask and / or a residual (kEx = true), so that the plain forward
// carries none of their code.  With a pair mask, one more K-step adds E M^T to S,
// E (128 x 16) holding 1.0 in column 0 and the stage's M (64 x 16) 0 or -30000 in
// column 0 (the key is admitted or excluded on this line).  Both without swizzle;
// columns 8..15 of E are a block of zeros, those of M the stage's ones and zero
// rows (finite).  The ones row of V' then moves from row 32 to row 40.
template <bool kEx>
struct Lay {
    static constexpr int kME = kBias + 2 * kBStages * kBiasBytes;   // E: 128 rows x 16 B, then 2 KB of zeros
    static constexpr int kIdent = kME + (kEx ? 4096 : 0);            // 64 x 64 f16 identity (SW128, K-major)
    static constexpr int kWo = kIdent + 8192;     // W_o^T, 2 x [128 x 128 B] (SW128), loaded at CTA start
    static constexpr int kBo = kWo + 32768;       // b_o (128 fp32)
    static constexpr int kBar = kBo + 512;
    static constexpr int kSmem = kBar + 1024 + 1024;  // barriers + alignment slack
    static constexpr int kLCol = kEx ? 40 : 32;   // row of V' holding ones = column of P V' holding l
    static_assert(kIdent % 1024 == 0 && kWo % 1024 == 0, "SW128 tiles need 1024-byte alignment");
    static_assert(kSmem <= 232448, "dynamic shared memory above the per-block limit");
};
// TMEM columns
__host__ __device__ constexpr uint32_t colS(int g, int b) { return g * 128u + b * 64u; }   // S / P buffers
__host__ __device__ constexpr uint32_t colO(int g) { return 256u + g * 64u; }  // O (32), row sum l (kLCol)
__host__ __device__ constexpr uint32_t colU(int g) { return 384u + g * 64u; }  // gated u (f16 pairs)
static_assert(kBias % 1024 == 0 && kStageBytes % 1024 == 0, "SW128 tiles need 1024-byte alignment");
}  // namespace k2

// Item-end output of one 128-row query group: the projected rows (TMEM columns
// tOut .. tOut + 127 of this thread's lane) + b_o, masked, plus the residual, stored
// in the node's orientation.  out_free is signalled as soon as the last TMEM columns
// are in registers.  The bf16 builds call it out of line (attn_store_out_call), so
// that its registers do not shape the allocation of the attention loops; the fp32
// build inlines it (out of line, that build's attention launch took 12.0 instead of
// 10.7 ms at I = 2048).
// 32-byte global store (eight 32-bit words; the address must be 32-byte aligned)
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* w) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                 "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

template <bool kEx, bool kF32>
__device__ __forceinline__ void attn_store_out(int node, int I, const uint8_t* mask, const uint8_t* pmask,
                                               const void* Z, void* out, uint32_t tOut, int L, int x,
                                               const float* sbo, uint64_t* out_free) {
    constexpr int kRow = CZ * (kF32 ? 4 : 2) / 16;   // 16-byte words per pair vector
    const int lane = threadIdx.x & 31;
    const size_t pair = node == TRI_ATTN_STARTING ? (size_t)L * I + x : (size_t)x * I + L;
    const bool valid = x < I && (mask == nullptr || mask[x] != 0) && (!kEx || pmask == nullptr || pmask[pair] != 0);
    uint4* dst = reinterpret_cast<uint4*>(out) + pair * kRow;
    const uint4* zres = (kEx && Z) ? reinterpret_cast<const uint4*>(Z) + pair * kRow : nullptr;
    const bool wide = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;   // rows then start on 32 bytes
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
        uint32_t v[32];
        tmem_ld32(tOut + cb * 32, v);
        tmem_ld_wait();
        tmem_regs_ready(v);
        if (cb == 3) {                       // all of the output read: S(0), S(1) of the next item may go
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(out_free);
        }
        if constexpr (kF32) {
            // fp32 out (and residual): 32 channels = 8 16-byte words
            uint32_t w[32];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float4 zv = make_float4(0.f, 0.f, 0.f, 0.f);
                if (kEx && zres && x < I) zv = *reinterpret_cast<const float4*>(zres + cb * 8 + i);
                const int e = 4 * i;
                const float4 r4 = make_float4(
                    (valid ? __uint_as_float(v[e]) + sbo[cb * 32 + e] : 0.f) + zv.x,
                    (valid ? __uint_as_float(v[e + 1]) + sbo[cb * 32 + e + 1] : 0.f) + zv.y,
                    (valid ? __uint_as_float(v[e + 2]) + sbo[cb * 32 + e + 2] : 0.f) + zv.z,
                    (valid ? __uint_as_float(v[e + 3]) + sbo[cb * 32 + e + 3] : 0.f) + zv.w);
                w[4 * i] = __float_as_uint(r4.x);
                w[4 * i + 1] = __float_as_uint(r4.y);
                w[4 * i + 2] = __float_as_uint(r4.z);
                w[4 * i + 3] = __float_as_uint(r4.w);
            }
            if (x < I) {
                if (wide) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) st_global_v8(dst + cb * 8 + 2 * j, w + 8 * j);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[cb * 8 + i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                }
            }
        } else {
            uint32_t zw[16];                     // residual (this thread's own pair: read before write)
            if constexpr (kEx) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 zv = (zres && x < I) ? zres[cb * 4 + i] : make_uint4(0, 0, 0, 0);
                    zw[4 * i] = zv.x;
                    zw[4 * i + 1] = zv.y;
                    zw[4 * i + 2] = zv.z;
                    zw[4 * i + 3] = zv.w;
                }
            }
            uint32_t o[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                float a0 = valid ? __uint_as_float(v[e]) + sbo[cb * 32 + e] : 0.f;
                float a1 = valid ? __uint_as_float(v[e + 1]) + sbo[cb * 32 + e + 1] : 0.f;
                if constexpr (kEx) {
                    a0 += bf16lo(zw[e >> 1]);
                    a1 += bf16hi(zw[e >> 1]);
                }
                o[e >> 1] = pack_bf16(a0, a1);
            }
            if (x < I) {
                if (wide) {
                    st_global_v8(dst + cb * 4, o);
                    st_global_v8(dst + cb * 4 + 2, o + 8);
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[cb * 4 + i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                }
            }
        }
    }
}

template <bool kEx>
__device__ __noinline__ void attn_store_out_call(int node, int I, const uint8_t* mask, const uint8_t* pmask,
                                                 const void* Z, void* out, uint32_t tOut, int L, int x,
                                                 const float* sbo, uint64_t* out_free) {
    attn_store_out<kEx, false>(node, I, mask, pmask, Z, out, tOut, L, x, sbo, out_free);
}

// kMsa: the build for MSA row attention (always with kEx): a line is an MSA row,
// a work item covers heads h0 .. h0+3 of 8, h0 = 0 or 4 (q, k, v^T, g and the pair bias hold 8
// heads per line), the MSA mask arrives as the pair mask's key bits, and each
// head's gated output goes to global memory for the separate output projection
// (no W_o, no epilogue here).
// kF32: Z (residual) and out are fp32 (the TF32 forward); otherwise bf16.
template <bool kEx, bool kMsa, bool kF32 = false>
__global__ void __launch_bounds__(k2::kThreads, 1)
sm103_attention(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                const __grid_constant__ CUtensorMap mapVt, const __grid_constant__ CUtensorMap mapB,
                const __grid_constant__ CUtensorMap mapWo, AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    using LY = k2::Lay<kEx>;
    static_assert(kEx || !kMsa, "the MSA build is a pair-mask build");
    constexpr int NHT = kMsa ? 8 : NH;         // heads stored per line
    const bool fused_out = !kMsa && p.last;   // output projection and store in this kernel
    if (status_set(p.status)) return;          // an earlier wait gave up: fail fast
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Persistent (one CTA per SM): the TMA producer claims work items from a global
    // counter (each a 256-query block of one line and, in the MSA build, one head
    // half) and posts them in a 4-slot ring in shared memory; every role takes the
    // same item sequence from the ring and keeps running tile and item counters, so
    // the producers load the next item's first tiles while the current item's
    // epilogue runs, the CTA set-up (barriers, TMEM, W_o^T) is paid once, and SMs that
    // run slower simply take fewer items.  A claim past the last item posts -1 (end).
    auto item_x0 = [&](int item) { return (item % p.n_xb) * 256; };
    auto item_L = [&](int item) { return (item / p.n_xb) % p.lines; };
    auto item_h0 = [&](int item) { return kMsa ? (item / (p.n_xb * p.lines)) * NH : 0; };  // MSA: heads h0..h0+3
    auto skip_item = [&](int item) { return p.mask != nullptr && p.mask[item_L(item)] == 0; };

    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + LY::kBar);
    uint64_t* q_full = bars + 0;      // [2]
    uint64_t* q_empty = bars + 2;     // [2]
    uint64_t* kv_full = bars + 48;    // [5]
    uint64_t* kv_empty = bars + 56;   // [5]
    uint64_t* s_full = bars + 12;     // [2 groups][2 buffers]
    // P and O barriers alternate by tile parity: with two S buffers a softmax group
    // can write P(it) and P(it+1) before the MMA warp has waited for P(it), and one
    // barrier would then run two phases ahead of its waiter.
    uint64_t* p_full = bars + 16;     // [2 groups][tile parity]: P(it) of group g written
    uint64_t* o_ready = bars + 20;    // [2 groups][tile parity]: P V'(it) of group g done
    uint64_t* u_full = bars + 24;     // [2]
    uint64_t* o_full = bars + 26;     // [2]
    uint64_t* out_free = bars + 4;    // [2]: the group's output rows read from TMEM (its S columns free)
    uint64_t* it_full = bars + 64;    // [4]: work-item slot posted
    uint64_t* it_empty = bars + 68;   // [4]: slot read by all 12 readers (2 bias cursors, 2 MMA warps, 8 softmax warps)
    volatile int* sitem = reinterpret_cast<volatile int*>(bars + 72);   // [4] item indices
    // bars + 80 .. + 103: one 16-byte slot per warp (the softmax warps' current item)
    uint64_t* w_full = bars + 28;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 29);
    volatile int* abort = reinterpret_cast<volatile int*>(bars + 30);
    uint64_t* b_full = bars + 32;     // [2 groups][4]: bias tile staged
    uint64_t* b_empty = bars + 40;    // [2 groups][4]: S of that tile done (bias read)
    // the n-th item of this CTA's sequence, for a reader that has not yet taken it
    auto take_item = [&](int n, bool& okv) -> int {
        const int slot = n & 3;
        okv = __all_sync(0xffffffffu, mbar_wait(it_full + slot, (n >> 2) & 1, abort));
        if (!okv) return -1;
        const int item = sitem[slot];
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(it_empty + slot);
        return item;
    };

    // Rows 32..47 of each stage's V': a row of ones (row kLCol: gives the softmax
    // row sum as output column kLCol of P V'), the rest zero.  With kEx, rows
    // 32..39 hold the pair-mask tile M (zero without a pair mask; as rows of V'
    // they only fill columns 32..39 of P V', which nothing reads).  Same in every
    // swizzle phase.
    for (int i = threadIdx.x; i < k2::kStages * 2048 / 16; i += blockDim.x) {
        const int st = i / 128, off = (i % 128) * 16;
        uint8_t* dst = sm + k2::kStage + st * k2::kStageBytes + k2::kSM + off;
        const uint32_t one2 = (off >= (LY::kLCol - 32) * 128 && off < (LY::kLCol - 31) * 128) ? 0x3C003C00u : 0u;
        *reinterpret_cast<uint4*>(dst) = make_uint4(one2, one2, one2, one2);
    }
    // 64 x 64 identity, the B operand that adds the staged bias tile into S:
    // S = Q K^T + Bias I (row n holds 1.0 at column n; 128B-swizzled rows).
    for (int i = threadIdx.x; i < 8192 / 16; i += blockDim.x) {
        const int n = i >> 3, c = i & 7;                      // row n, physical 16-byte chunk c
        const int lc = c ^ (n & 7);                           // logical chunk: columns 8 lc .. 8 lc + 7
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if ((n >> 3) == lc) {
            const int e = n & 7;                              // column n within the chunk
            w[e >> 1] = (e & 1) ? 0x3C000000u : 0x00003C00u;
        }
        *reinterpret_cast<uint4*>(sm + LY::kIdent + i * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (fused_out)
        for (int i = threadIdx.x; i < CZ; i += blockDim.x) reinterpret_cast<float*>(sm + LY::kBo)[i] = p.bo[i];
    if (kEx && p.kbits != nullptr)             // E: 1.0 in column 0, then its columns 8..15: zeros
        for (int i = threadIdx.x; i < 4096 / 16; i += blockDim.x)
            *reinterpret_cast<uint4*>(sm + LY::kME + i * 16) = make_uint4(i < 128 ? 0x3C00u : 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();

    const int nk = p.nk;
    const int NT = NH * nk;
    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(q_full + s, 1);
            mbar_init(q_empty + s, 2);            // one commit per MMA issuer
            mbar_init(u_full + s, 4);
            mbar_init(o_full + s, 1);
            mbar_init(out_free + s, 4);
        }
        for (int s = 0; s < 4; ++s) {
            mbar_init(it_full + s, 1);
            mbar_init(it_empty + s, 12);
        }
        for (int s = 0; s < k2::kStages; ++s) {
            mbar_init(kv_full + s, 1);
            mbar_init(kv_empty + s, 2);           // one commit per MMA issuer (softmax group)
        }
        for (int s = 0; s < 2 * k2::kBStages; ++s) {
            mbar_init(b_full + s, 1);
            mbar_init(b_empty + s, 1);            // the group's MMA issuer commits after S
        }
        for (int s = 0; s < 4; ++s) {             // [2 groups][2 buffers or tile parities]
            mbar_init(s_full + s, 1);
            mbar_init(p_full + s, 4);
            mbar_init(o_ready + s, 1);
        }
        mbar_init(w_full, 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    // Register budget: launched at 168 per thread.  The control warpgroup
    // (warps 0-3, one warp per SM sub-partition) drops to 120 and each softmax
    // warp grows to 192, so every sub-partition releases exactly what it takes
    // (32 x 48 = 2 x 32 x 24 registers) and no increase can wait on another
    // sub-partition.
    // The producer and MMA warps run their loops converged (every lane waits on the
    // same barriers, so loop control and addresses stay warp-uniform) and one
    // elected lane issues each TMA copy or tcgen05 instruction.
    if (warp == 0) {
        setmaxnreg_dec<120>();
        // ------------------------------------------------------------ TMA producer
        const bool leader = elect_one();
        if (leader) {
            prefetch_tmap(&mapQ);
            prefetch_tmap(&mapK);
            prefetch_tmap(&mapVt);
            prefetch_tmap(&mapB);
        }
        bool ok = true;
        int it_issued = 0, skipped = -1, q_loads = 0;   // for the drain on the abort path
        if (leader && fused_out) {                // W_o^T for every item's output projection, loaded once
            prefetch_tmap(&mapWo);
            mbar_arrive_expect_tx(w_full, 32768);
            tma_load_2d(sm + LY::kWo, &mapWo, w_full, 0, 0);
            tma_load_2d(sm + LY::kWo + 16384, &mapWo, w_full, 64, 0);
        }
        // it: running tile count over this CTA's items (K / V' stage and phase); hq:
        // running head count (Q buffer hq & 1; with four heads per item its phases
        // match the per-item head index)
        for (int n = 0, it = 0, hq = 0; ok; ++n) {
            const int slot = n & 3;
            ok = __all_sync(0xffffffffu, mbar_wait(it_empty + slot, ((n >> 2) & 1) ^ 1, abort));
            if (!ok) break;
            if (leader) {
                const int got = atomicAdd(p.work, 1);
                sitem[slot] = got < p.n_items ? got : -1;
                mbar_arrive(it_full + slot);
            }
            __syncwarp();
            const int item = sitem[slot];
            if (item < 0) break;
            if (skip_item(item)) continue;
            const int L = item_L(item), xq0 = item_x0(item), h0 = item_h0(item);
            for (int h = 0; ok && h < NH; ++h, ++hq) {
                const int lh = L * NHT + h0 + h;
                for (int t = 0; t < nk; ++t, ++it) {
                    const int st = it % k2::kStages;
                    if (t == 0) {
                        const int qb = hq & 1;
                        ok = __all_sync(0xffffffffu, mbar_wait(q_empty + qb, ((hq >> 1) & 1) ^ 1, abort));
                        if (!ok) break;
                        if (leader) {
                            mbar_arrive_expect_tx(q_full + qb, 16384);
                            tma_load_2d(sm + k2::kQ + qb * 16384, &mapQ, q_full + qb, 0, lh * p.I_pad + xq0);
                            tma_load_2d(sm + k2::kQ + qb * 16384 + 8192, &mapQ, q_full + qb, 0,
                                        lh * p.I_pad + xq0 + 128);
                        }
                        q_loads = hq + 1;
                    }
                    uint32_t two = 0;                 // key-valid bits of keys k0 + 2 lane, + 1 (read before the wait;
                    if (kEx && p.kbits != nullptr) {  // k0 is a multiple of 8, so both bits sit in one 32-bit word)
                        const int k = p.k_begin + t * k2::kKT + 2 * static_cast<int>(lane_id());
                        const uint32_t* wrow =
                            reinterpret_cast<const uint32_t*>(p.kbits + (size_t)L * (p.I_pad / 64 + 1));
                        two = wrow[k >> 5] >> (k & 31);
                    }
                    ok = __all_sync(0xffffffffu, mbar_wait(kv_empty + st, ((it / k2::kStages) & 1) ^ 1, abort));
                    if (!ok) break;
                    if (kEx && p.kbits != nullptr) {  // M of the stage: lane writes keys 2 lane, 2 lane + 1
                        const uint32_t ln = lane_id();
                        uint8_t* mt =
                            sm + k2::kStage + st * k2::kStageBytes + k2::kSM + (ln >> 2) * 128 + (ln & 3) * 32;
                        *reinterpret_cast<uint16_t*>(mt) = (two & 1u) ? uint16_t(0) : uint16_t(0xF753u);   // f16 -30000
                        *reinterpret_cast<uint16_t*>(mt + 16) = (two & 2u) ? uint16_t(0) : uint16_t(0xF753u);
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                    const bool skip = p.inject == TRI_ATTN_FAULT_SKIP_STAGE && it == 1 && item == 0;
                    if (leader && !skip) {
                        const int k0 = p.k_begin + t * k2::kKT;
                        uint8_t* sb = sm + k2::kStage + st * k2::kStageBytes;
                        mbar_arrive_expect_tx(kv_full + st, k2::kStageTx);
                        tma_load_2d(sb + k2::kSK, &mapK, kv_full + st, 0, lh * p.I_pad + k0);
                        tma_load_2d(sb + k2::kSV, &mapVt, kv_full + st, k0, lh * HD);
                    }
                    if (skip) skipped = it;
                    it_issued = it + 1;
                    __syncwarp();
                }
            }
        }
        if (fused_out) {
            // the block must not end with the W_o^T copy still writing its shared
            // memory, even when another role gave up (bounded, ignores the abort flag)
            volatile int keep_waiting = 0;
            mbar_wait(w_full, 0, &keep_waiting);
        }
        if (!ok) {
            // gave up (or another role did): before the block ends, wait (bounded,
            // ignoring the abort flag) for the last copy issued into each K / V' stage
            // and each Q buffer, so that no TMA write lands in freed shared memory
            if (leader) set_abort(abort, p.status, kStatusTimeoutProducer);
            volatile int keep_waiting = 0;
            for (int st = 0; st < k2::kStages; ++st) {
                int j = it_issued - 1 - ((it_issued - 1 - st) % k2::kStages + k2::kStages) % k2::kStages;
                if (j == skipped) j -= k2::kStages;
                if (j >= 0) mbar_wait(kv_full + st, (j / k2::kStages) & 1, &keep_waiting);
            }
            for (int b = 0; b < 2; ++b) {
                const int hl = q_loads - 1 - ((q_loads - 1 - b) % 2 + 2) % 2;   // last head loaded into buffer b
                if (hl >= 0) mbar_wait(q_full + b, (hl >> 1) & 1, &keep_waiting);
            }
        }
    } else if (warp == 1 || warp == 2) {
        setmaxnreg_dec<120>();
        // ------------------------------------------------------------ MMA issuers
        // Warp 1 issues every MMA of softmax group 0, warp 2 those of group 1, so
        // each group's P -> P V' -> S(it+2) round trip waits only on its own group.
        const int g = warp - 1;
        const bool leader = elect_one();
        constexpr uint32_t idS = idesc_f16_f32(128, k2::kKT);
        constexpr uint32_t idO = idesc_f16_f32(128, 48);
        constexpr uint64_t tK = sdesc_tmpl(512, kSwizzle64);      // Q and K tiles: 64 B rows
        constexpr uint64_t tV = sdesc_tmpl(1024, kSwizzle128);    // V', bias, W_o^T: 128 B rows
        const uint32_t qbase = smem_u32(sm + k2::kQ), sbase = smem_u32(sm + k2::kStage);
        // descriptors of stage 0 / Q buffer 0 for this group; other stages and
        // buffers are fixed offsets in the 16-byte address field (no carry: shared
        // addresses < 256 KB)
        const uint64_t dQ0 = sdesc_at(tK, qbase + g * 8192), dK0 = sdesc_at(tK, sbase + k2::kSK);
        const uint64_t dV0 = sdesc_at(tV, sbase + k2::kSV);
        const uint64_t dB0 = sdesc_at(tV, smem_u32(sm + k2::kBias + g * k2::kBStages * k2::kBiasBytes));
        const uint64_t dI = sdesc_at(tV, smem_u32(sm + LY::kIdent));
        constexpr uint64_t kBiasStep = k2::kBiasBytes >> 4;
        constexpr uint64_t kStageStep = k2::kStageBytes >> 4;
        const uint64_t dE = sdesc_noswizzle(smem_u32(sm + LY::kME), 2048, 128);
        const uint64_t dM0 = sdesc_noswizzle(sbase + k2::kSM, 1024, 128);
        bool ok = true;
        // S_g(it) = Q_g K(it)^T + Bias_g(it) I into buffer it & 1: the pair bias is
        // added by the tensor core (the staged bias tile is the A operand of four
        // more K-steps against a 64 x 64 identity).
        // Q_g of head h is copied once from its staged tile into TMEM columns
        // colU(g) + 16 h .. + 15 (free until the head's gated output is written there
        // at the start of the next head), and Q K^T reads its A operand from TMEM.
        auto issue_s = [&](int it, int h) {
            const uint64_t st = static_cast<uint64_t>(it % k2::kStages);
            const uint32_t qt = tmem + k2::colU(g) + h * 16;
            const uint64_t kb = dK0 + st * kStageStep;
            const uint64_t bb = dB0 + static_cast<uint64_t>(it % k2::kBStages) * kBiasStep;
            const uint32_t d = tmem + k2::colS(g, it & 1);
            mma_ts(d, qt, kb, idS, 0u);
            mma_ts(d, qt + 8, kb + 2, idS, 1u);
#pragma unroll
            for (int kk = 0; kk < k2::kKT / 16; ++kk) mma_ss(d, bb + kk * 2, dI + kk * 2, idS, 1u);
            if (kEx && p.kbits != nullptr) mma_ss(d, dE, dM0 + st * kStageStep, idS, 1u);   // -30000 on excluded keys
        };
        // O_g (+)= P_g(it) V'(it); the first tile of a head (t == 0) overwrites
        auto issue_pv = [&](int it, int t) {
            const uint64_t vb = dV0 + static_cast<uint64_t>(it % k2::kStages) * kStageStep;
            const uint32_t a = tmem + k2::colS(g, it & 1), d = tmem + k2::colO(g);
            const uint32_t first = t > 0 ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < k2::kKT / 16; ++kk) mma_ts(d, a + kk * 8, vb + kk * 2, idO, kk > 0 ? 1u : first);
        };
        // operands of S(it) present: Q of its head (first tile), K and bias of its stage
        auto s_ready = [&](int it, int h, int t) -> bool {
            bool r = true;
            if (t == 0) r = mbar_wait(q_full + (h & 1), (h >> 1) & 1, abort);
            if (r) r = mbar_wait(kv_full + it % k2::kStages, (it / k2::kStages) & 1, abort);
            if (r) r = mbar_wait(b_full + g * k2::kBStages + it % k2::kBStages, (it / k2::kBStages) & 1, abort);
            return __all_sync(0xffffffffu, r);
        };
        auto issue_s_step = [&](int it, int h, int t) {   // leader only
            tc_fence_after();
            if (t == 0) {                                     // Q(h): smem -> TMEM, then release the buffer
                const uint64_t qa = dQ0 + static_cast<uint64_t>((h & 1) * 1024);
                const uint32_t qt = tmem + k2::colU(g) + h * 16;
                tmem_cp_128x256b(qt, qa);
                tmem_cp_128x256b(qt + 8, qa + 2);
                tc_commit(q_empty + (h & 1));
            }
            issue_s(it, h);
            tc_commit(s_full + g * 2 + (it & 1));
            tc_commit(b_empty + g * k2::kBStages + it % k2::kBStages);   // bias tile read
        };
        // Group 1 starts about a microsecond later, so that the two groups' exponential
        // phases and MMA bursts interleave instead of coinciding; with separate bias
        // rings nothing pulls them back into step.
        if (g == 1) {
            __nanosleep(500);
            __nanosleep(500);
        }
        // it0: running tile count of this CTA's earlier items (tile it of an item is
        // it0 + it for stages, buffers and phases; NT is a multiple of 4, so buffer and
        // barrier parities continue across items); done: items finished
        for (int n = 0, it0 = 0, done = 0; ok; ++n) {
            const int item = take_item(n, ok);
            if (!ok || item < 0) break;
            if (skip_item(item)) continue;
            // the output projection of the previous item left its result in this group's
            // S columns: S(0) and S(1) wait until the softmax warps have read it
            if (fused_out && done > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(out_free + g, (done - 1) & 1, abort));
                if (!ok) break;
            }
            // prologue: S of tiles 0 and 1
            int hn = 0, tn = 0;                       // (head, tile) of the next S to issue
            for (int it = 0; ok && it < 2 && it < NT; ++it) {
                ok = s_ready(it0 + it, hn, tn);
                if (!ok) break;
                if (leader) issue_s_step(it0 + it, hn, tn);
                __syncwarp();
                if (++tn == nk) { tn = 0; ++hn; }
            }
            // Per tile: P(it) -> P V'(it), then at once S(it+2) into the same buffer (the
            // tensor core runs one thread's MMAs in order).  The operands of S(it+2) are
            // checked while P(it) is still being computed, off the P -> S path.
            for (int it = 0, tp = 0; ok && it < NT; ++it) {
                const int nx = it + 2, gi = it0 + it;
                if (nx < NT) {
                    ok = s_ready(it0 + nx, hn, tn);
                    if (!ok) break;
                }
                ok = __all_sync(0xffffffffu, mbar_wait(p_full + g * 2 + (gi & 1), (gi >> 1) & 1, abort));
                if (!ok) break;
                if (leader) {
                    tc_fence_after();
                    issue_pv(gi, tp);
                    tc_commit(o_ready + g * 2 + (gi & 1));
                    tc_commit(kv_empty + gi % k2::kStages);   // this group is done with the K / V' stage
                    if (nx < NT) issue_s_step(it0 + nx, hn, tn);
                }
                __syncwarp();
                if (nx < NT && ++tn == nk) { tn = 0; ++hn; }
                if (++tp == nk) tp = 0;
            }
            if (ok && fused_out) {                    // output projection: out = u W_o
                constexpr uint32_t idP = idesc_f16_f32(128, 128);
                ok = __all_sync(0xffffffffu, mbar_wait(w_full, 0, abort) && mbar_wait(u_full + g, done & 1, abort));
                if (ok && leader) {
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ts(tmem + k2::colS(g, 0), tmem + k2::colU(g) + kk * 8,
                               sdesc_at(tV, smem_u32(sm + LY::kWo) + (kk >> 2) * 16384 + (kk & 3) * 32), idP,
                               kk > 0 ? 1u : 0u);
                    tc_commit(o_full + g);
                }
                __syncwarp();
            }
            it0 += NT;
            ++done;
        }
        if (!ok && leader) set_abort(abort, p.status, kStatusTimeoutMma);
    } else if (warp == 3) {
        setmaxnreg_dec<120>();
        // ------------------------------------------------------------ bias producer
        // Keeps each group's bias ring as full as that group's own progress allows,
        // polling both rings so a slower group never holds the other's loads back.
        const bool leader = elect_one();
        if (leader) prefetch_tmap(&mapB);
        // Per group: state of the item it is loading for (-2: take the next item from
        // the ring, -1: no more items), the item's first bias row, the (head, tile) of
        // the next load, and the running count of tiles loaded (ring stage and phase).
        int st_[2] = {-2, -2}, row0[2] = {0, 0}, hh[2] = {0, 0}, tt[2] = {0, 0}, ni[2] = {0, 0};
        int nb0 = 0, nb1 = 0;
        bool ok = true, idle = false;
        uint64_t t0 = 0;                           // start of the current run of polls without progress
        while (ok && (st_[0] != -1 || st_[1] != -1)) {
            bool progressed = false;
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                if (st_[g] == -2) {                // poll the ring: never block the other group's loads
                    const int slot = ni[g] & 3;
                    if (!__all_sync(0xffffffffu, mbar_test(it_full + slot, (ni[g] >> 2) & 1))) continue;
                    const int item = sitem[slot];
                    __syncwarp();
                    if (lane == 0) mbar_arrive(it_empty + slot);
                    ++ni[g];
                    progressed = true;
                    if (item < 0) {
                        st_[g] = -1;
                    } else if (!skip_item(item)) {
                        st_[g] = 0;
                        row0[g] = item_h0(item) * p.I_pad + item_x0(item) + g * 128;
                        hh[g] = 0;
                        tt[g] = 0;
                    }
                }
                if (st_[g] < 0) continue;
                const int j = g ? nb1 : nb0;
                const int bs = g * k2::kBStages + j % k2::kBStages;
                if (!__all_sync(0xffffffffu, mbar_test(b_empty + bs, ((j / k2::kBStages) & 1) ^ 1))) continue;
                if (leader) {
                    mbar_arrive_expect_tx(b_full + bs, k2::kBiasBytes);
                    tma_load_2d(sm + k2::kBias + bs * k2::kBiasBytes, &mapB, b_full + bs, p.k_begin + tt[g] * k2::kKT,
                                row0[g] + hh[g] * p.I_pad);
                }
                __syncwarp();
                if (g) ++nb1; else ++nb0;
                if (++tt[g] == nk) {
                    tt[g] = 0;
                    if (++hh[g] == NH) st_[g] = -2;
                }
                progressed = true;
            }
            if (progressed) {
                idle = false;
            } else if (!idle) {
                idle = true;
                t0 = globaltimer();
            } else if (*abort || globaltimer() - t0 > kWaitTimeoutNs) {
                ok = false;
            } else {
                __nanosleep(160);
            }
        }
        if (!ok) {
            // gave up: before the block ends, wait (bounded, ignoring the abort flag) for
            // the last bias copy issued into each stage of both rings
            if (leader) set_abort(abort, p.status, kStatusTimeoutProducer);
            volatile int keep_waiting = 0;
            for (int g = 0; g < 2; ++g) {
                const int issued = g ? nb1 : nb0;
                for (int st = 0; st < k2::kBStages; ++st) {
                    const int j = issued - 1 - ((issued - 1 - st) % k2::kBStages + k2::kBStages) % k2::kBStages;
                    if (j >= 0) mbar_wait(b_full + g * k2::kBStages + st, (j / k2::kBStages) & 1, &keep_waiting);
                }
            }
        }
    } else if (warp < 4) {
        setmaxnreg_dec<120>();                     // idle warps of the control warpgroup
    } else {
        setmaxnreg_inc<192>();
        // ------------------------------------------------------------ softmax warpgroups
        const int g = (warp - 4) >> 2;            // 0: queries xq0..+127, 1: xq0+128..+255
        const int wq = warp & 3;
        const int r = wq * 32 + lane;
        // the current item's line, first query and first head, kept in this warp's
        // shared-memory slot and read where they are needed (once per head), so that
        // they hold no registers in the tile loop
        volatile int* wslot = reinterpret_cast<volatile int*>(bars + 80) + warp * 4;
        const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const uint32_t tO = tl + k2::colO(g), tU = tl + k2::colU(g);
        const float* sbo = reinterpret_cast<const float*>(sm + LY::kBo);
        float m = kMfloor;                        // running max (log2 units)
        bool ok = true;
        constexpr int kRow = CZ * (kF32 ? 4 : 2) / 16;   // 16-byte words per pair vector
        // an item whose line is padding: its update is zero (with a residual: out = Z)
        auto fill_masked = [&](int item) {
            if (!p.last || (kEx && p.Z == p.out)) return;
            const int Lm = item_L(item), xm0 = item_x0(item);
            const size_t sL = p.node == TRI_ATTN_STARTING ? (size_t)p.I : 1;
            const size_t sX = p.node == TRI_ATTN_STARTING ? 1 : (size_t)p.I;
            for (int i = static_cast<int>(threadIdx.x) - 128; i < 256 * kRow; i += 256) {
                const int xm = xm0 + i / kRow;
                if (xm < p.I) {
                    const size_t at = (Lm * sL + xm * sX) * kRow + i % kRow;
                    reinterpret_cast<uint4*>(p.out)[at] =
                        (kEx && p.Z) ? reinterpret_cast<const uint4*>(p.Z)[at] : make_uint4(0, 0, 0, 0);
                }
            }
        };

        // normalise head hp, merge with the running chunk state, gate into u (TMEM)
        // gate of the head being finished, loaded at the head's last tile so that its
        // global-memory latency is hidden (heads of one tile load it in finalize)
        uint4 gpre[4];
        auto load_gate = [&](int hh) {
            const int L = wslot[0], h0 = wslot[2], x = wslot[1] + g * 128 + r;
            const uint4* gp = reinterpret_cast<const uint4*>(p.g + (((size_t)L * NHT + h0 + hh) * p.I_pad + x) * HD);
#pragma unroll
            for (int i = 0; i < 4; ++i) gpre[i] = gp[i];
        };
        auto finalize = [&](int hp) {
            const int L = wslot[0], h0 = wslot[2], x = wslot[1] + g * 128 + r;
            uint32_t ov[32];
            tmem_ld32(tO, ov);
            const float l = __uint_as_float(tmem_ld1(tO + LY::kLCol));
            tmem_ld_wait();
            float o[HD];
            const float inv = l > 0.f ? 1.f / l : 0.f;
            float lse = l > 0.f ? m + __log2f(l) : -INFINITY;
            // an f16 intermediate (q, k, v, pair bias) out of range shows up here as a
            // non-finite row sum or output (a NaN or an infinity anywhere makes the sum
            // non-finite): latch it in the status word.  Rows past I are padding.
            float chk = l;
#pragma unroll
            for (int e = 0; e < HD; ++e) {
                o[e] = __uint_as_float(ov[e]) * inv;
                chk += fabsf(o[e]);
            }
            if (x < p.I && !(chk < INFINITY)) atomicOr(p.status, kStatusRange);
            const size_t srow = ((size_t)(L * NHT + h0 + hp)) * p.I_pad + x;
            if (!p.first) {
                const float lr = p.lse_run[srow];
                const float top = fmaxf(lr, lse);
                if (top != -INFINITY) {
                    const float wr = ex2(lr - top), wc = ex2(lse - top);
                    const float it_ = 1.f / (wr + wc);
                    const float4* orun = reinterpret_cast<const float4*>(p.o_run + srow * HD);
#pragma unroll
                    for (int e4 = 0; e4 < HD / 4; ++e4) {
                        const float4 v = orun[e4];
                        o[4 * e4 + 0] = (wr * v.x + wc * o[4 * e4 + 0]) * it_;
                        o[4 * e4 + 1] = (wr * v.y + wc * o[4 * e4 + 1]) * it_;
                        o[4 * e4 + 2] = (wr * v.z + wc * o[4 * e4 + 2]) * it_;
                        o[4 * e4 + 3] = (wr * v.w + wc * o[4 * e4 + 3]) * it_;
                    }
                    lse = top + __log2f(wr + wc);
                }
            }
            if (!p.last) {
                p.lse_run[srow] = lse;
                float4* orun = reinterpret_cast<float4*>(p.o_run + srow * HD);
#pragma unroll
                for (int e4 = 0; e4 < HD / 4; ++e4)
                    orun[e4] = make_float4(o[4 * e4], o[4 * e4 + 1], o[4 * e4 + 2], o[4 * e4 + 3]);
            } else {
                if (nk == 1) load_gate(hp);
                uint32_t u[16];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 gv = gpre[i];
                    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const int e = 8 * i + 2 * jj;
                        u[4 * i + jj] = pack_f16(f16lo(gw[jj]) * o[e], f16hi(gw[jj]) * o[e + 1]);
                    }
                }
                if constexpr (kMsa) {
                    // 64 bytes of the slot's 512-byte row (workspace: 256-byte aligned)
                    uint4* dst = reinterpret_cast<uint4*>(p.u + ((size_t)L * p.I_pad + x) * (NHT * HD) + (h0 + hp) * HD);
                    st_global_v8(dst, u);
                    st_global_v8(dst + 2, u + 8);
                } else {
                    tmem_st16(tU + hp * 16, u);
                }
            }
        };

        // Barrier parities and phases below use the tile index within the item: NT is a
        // multiple of 4, so they equal those of the running tile count.
        for (int n = 0, done = 0; ok; ++n) {
            const int item = take_item(n, ok);
            if (!ok || item < 0) break;
            if (skip_item(item)) {
                fill_masked(item);
                continue;
            }
            if (lane == 0) {
                wslot[0] = item_L(item);
                wslot[1] = item_x0(item);
                wslot[2] = item_h0(item);
            }
            __syncwarp();
            for (int it = 0, h = 0, t = 0; it < NT; ++it, t = (t + 1 == nk) ? 0 : t + 1, h += (t == 0) ? 1 : 0) {
                const int b = it & 1;
                const uint32_t tS = tl + k2::colS(g, b);
                if (nk > 1 && t == nk - 1 && p.last) load_gate(h);
                if (!mbar_wait(s_full + g * 2 + b, (it >> 1) & 1, abort)) { ok = false; break; }
                tc_fence_after();
                // ---- scores of key tile it (bias already added by the tensor core)
                float s[k2::kKT];
                {
                    uint32_t va[32], vb[32];
                    tmem_ld32(tS, va);
                    tmem_ld32(tS + 32, vb);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        s[i] = __uint_as_float(va[i]);
                        s[32 + i] = __uint_as_float(vb[i]);
                    }
                }
                const int k0 = p.k_begin + t * k2::kKT;
                if (k0 + k2::kKT > p.k_end) {                // ragged last tile of the key range
                    const int nvalid = p.k_end - k0;
#pragma unroll
                    for (int k = 0; k < k2::kKT; ++k)
                        if (k >= nvalid) s[k] = -INFINITY;
                }

                // P V'(it-2) is long complete: observing it every tile keeps the o_ready
                // phases in step for the waits on P V'(it-1) below.  The test is issued
                // here and its result used only at the end of the tile.
                const bool pv2_done = it < 2 || mbar_test(o_ready + g * 2 + b, ((it - 2) >> 1) & 1);
                // Common case (the head continues): the exponentials against the running max
                // start at once; the tile max, needed only to detect a rescale, is computed
                // alongside them.
                const bool fast = t != 0;
                uint32_t pk[32];
                if (fast) {
                    const float negm = -m;
#pragma unroll
                    for (int k = 0; k < k2::kKT; k += 2) pk[k >> 1] = exp2_pair_f16x2(s[k], s[k + 1], negm);
                }
                // tile max: eight independent 3-input max chains
                float mx[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) mx[c] = max3(s[c], s[8 + c], s[16 + c]);
#pragma unroll
                for (int c = 0; c < 8; ++c) mx[c] = max3(mx[c], s[24 + c], s[32 + c]);
#pragma unroll
                for (int c = 0; c < 8; ++c) mx[c] = max3(mx[c], s[40 + c], s[48 + c]);
#pragma unroll
                for (int c = 0; c < 8; ++c) mx[c] = fmaxf(mx[c], s[56 + c]);
                const float mt = max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
                const bool need = mt > m + 8.f;              // rescale only when the max grew by > 2^8
                const bool redo = t == 0 || __any_sync(0xffffffffu, need);
                if (!fast || redo) {
                    if (!pv2_done && !mbar_wait(o_ready + g * 2 + b, ((it - 2) >> 1) & 1, abort)) { ok = false; break; }
                    auto wait_prev_pv = [&]() -> bool {
                        if (!mbar_wait(o_ready + g * 2 + (b ^ 1), ((it - 1) >> 1) & 1, abort)) return false;
                        tc_fence_after();
                        return true;
                    };
                    if (t == 0) {
                        if (it > 0) {
                            if (!wait_prev_pv()) { ok = false; break; }
                            finalize(h - 1);
                        }
                        m = fmaxf(mt, kMfloor);
                    } else if (redo) {
                        if (!wait_prev_pv()) { ok = false; break; }
                        uint32_t ov[32];
                        tmem_ld32(tO, ov);
                        uint32_t lv = tmem_ld1(tO + LY::kLCol);
                        tmem_ld_wait();
                        const float mn = need ? mt : m;
                        const float alpha = ex2(m - mn);
#pragma unroll
                        for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                        lv = __float_as_uint(__uint_as_float(lv) * alpha);
                        tmem_st32(tO, ov);
                        tmem_st1(tO + LY::kLCol, lv);
                        m = mn;
                    }
                    const float negm = -m;
#pragma unroll
                    for (int k = 0; k < k2::kKT; k += 2) pk[k >> 1] = exp2_pair_f16x2(s[k], s[k + 1], negm);
                } else if (!pv2_done && !mbar_wait(o_ready + g * 2 + b, ((it - 2) >> 1) & 1, abort)) {
                    ok = false;
                    break;
                }
                tmem_st32(tS, pk);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full + g * 2 + b);
            }
            if (ok && NT >= 2) ok = mbar_wait(o_ready + g * 2 + (NT & 1), ((NT - 2) >> 1) & 1, abort);
            if (ok) ok = mbar_wait(o_ready + g * 2 + ((NT - 1) & 1), ((NT - 1) >> 1) & 1, abort);
            if (ok) {
                tc_fence_after();
                finalize(NH - 1);
            }
            if (!ok) {
                set_abort(abort, p.status, kStatusTimeoutSoftmax);
                break;
            }
            if (fused_out) {
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(u_full + g);
                if (mbar_wait(o_full + g, done & 1, abort)) {
                    tc_fence_after();
                    if constexpr (kF32)
                        attn_store_out<kEx, true>(p.node, p.I, p.mask, p.pmask, p.Z, p.out, tl + k2::colS(g, 0),
                                                  wslot[0], wslot[1] + g * 128 + r, sbo, out_free + g);
                    else
                        attn_store_out_call<kEx>(p.node, p.I, p.mask, p.pmask, p.Z, p.out, tl + k2::colS(g, 0),
                                                 wslot[0], wslot[1] + g * 128 + r, sbo, out_free + g);
                } else {
                    set_abort(abort, p.status, kStatusTimeoutEpilogue);
                    ok = false;
                }
            }
            ++done;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// =====================================================================================
// Host side
// =====================================================================================
// the driver's tensor-map encoder, looked up once (thread-safe static initialisation)
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    }();
    return fn;
}

bool map2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t row_bytes, uint32_t box_cols,
           uint32_t box_rows, CUtensorMapSwizzle sw, CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_FLOAT16) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool map3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2,
           uint32_t b0, uint32_t b1, uint32_t b2, CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {s1, s2};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int current_device() {
    int dev = 0;
    cudaGetDevice(&dev);
    return dev;
}

// SM count of the current device (cached per device)
int num_sms() {
    static std::atomic<int> cache[64];
    const int dev = current_device();
    int n = (dev >= 0 && dev < 64) ? cache[dev].load(std::memory_order_relaxed) : 0;
    if (!n) {
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
        if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

}  // namespace

bool sm103_supported(int c_z, int H, int d, int dtype) {
    return dtype == TRI_ATTN_BF16 && c_z == CZ && H == NH && d == HD;
}

cudaError_t sm103_forward(const FwdArgs& a, cudaStream_t s, LaunchTimer* tm) {
    const Workspace& W = *a.lay;
    char* ws = a.ws;
    auto bf = [&](size_t off) { return reinterpret_cast<__nv_bfloat16*>(ws + off); };
    auto hf = [&](size_t off) { return reinterpret_cast<__half*>(ws + off); };
    auto f32 = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
    const int I = a.I, Ip = a.I_pad;

    // the shared-memory opt-in is a per-device function attribute: set it once per device
    static std::atomic<uint64_t> attr_set{0};
    const int dev = current_device();
    const uint64_t dev_bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
    if (!(attr_set.load(std::memory_order_acquire) & dev_bit)) {
        cudaError_t e = cudaFuncSetAttribute(sm103_ln_proj, cudaFuncAttributeMaxDynamicSharedMemorySize, k1::kSmem);
        if (e != cudaSuccess) return e;
        attr_set.fetch_or(dev_bit, std::memory_order_release);
    }

    // ---- weight preparation
    PrepArgs pa{a.w.ln_gamma, a.w.ln_beta, a.w.b_o, a.w.b_g,
                static_cast<const __nv_bfloat16*>(a.w.w_q), static_cast<const __nv_bfloat16*>(a.w.w_k),
                static_cast<const __nv_bfloat16*>(a.w.w_v), static_cast<const __nv_bfloat16*>(a.w.w_g),
                static_cast<const __nv_bfloat16*>(a.w.w_b), static_cast<const __nv_bfloat16*>(a.w.w_o),
                bf(W.wprep), f32(W.colsum), f32(W.betaw), f32(W.wb32), hf(W.wo_t), f32(W.bo), f32(W.cst)};
    if (tm) tm->begin("sm103_prep", s);
    sm103_prep<<<NCONST + CZ, 128, 0, s>>>(pa);
    if (tm) tm->end(s);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    // ---- LayerNorm + projections
    CUtensorMap mZs, mZe, mW;
    const uint64_t zrow = (uint64_t)CZ * 2, zline = (uint64_t)I * CZ * 2;
    if (!map3d(&mZs, a.Z, CZ, I, I, zrow, zline, 64, 128, 1) || !map3d(&mZe, a.Z, CZ, I, I, zrow, zline, 64, 1, 128) ||
        !map2d(&mW, bf(W.wprep), CZ, NPROJ, CZ * 2, 64, 256, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16))
        return cudaErrorInvalidValue;
    CUtensorMap mQs, mKs, mGs;
    const uint64_t rows_lh = (uint64_t)I * NH * Ip;
    if (!map2d(&mQs, hf(W.q), HD, rows_lh, HD * 2, HD, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !map2d(&mKs, hf(W.k), HD, rows_lh, HD * 2, HD, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !map2d(&mGs, hf(W.g), HD, rows_lh, HD * 2, HD, 32, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    ProjParams pp;
    pp.node = a.node;
    pp.I = I;
    pp.I_pad = Ip;
    pp.ntx = Ip / 128;
    pp.ntiles = I * pp.ntx;
    pp.eps = a.eps;
    pp.mask = a.mask;
    pp.colsum = f32(W.colsum);
    pp.betaw = f32(W.betaw);
    pp.wb32 = f32(W.wb32);
    pp.cst = f32(W.cst);
    pp.q = hf(W.q);
    pp.k = hf(W.k);
    pp.vt = hf(W.v);
    pp.g = hf(W.g);
    pp.bias = hf(W.bias);
    pp.status = a.status;
    {
        const int grid = pp.ntiles < num_sms() ? pp.ntiles : num_sms();
        if (tm) tm->begin("sm103_ln_proj", s);
        sm103_ln_proj<<<grid, k1::kThreads, k1::kSmem, s>>>(mZs, mZe, mW, mQs, mKs, mGs, pp);
        if (tm) tm->end(s);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }

    // ---- attention (+ gate, output projection), once per key chunk
    TriAttnLaunch l;
    l.node = a.node;
    l.I = I;
    l.I_pad = Ip;
    l.key_chunks = a.key_chunks;
    l.inject = a.inject;
    l.f32 = false;
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
    l.kbits = reinterpret_cast<uint64_t*>(a.ws + W.kbits);
    l.work = reinterpret_cast<int*>(a.ws + W.work);
    l.status = a.status;
    return sm103_triangle_attention(l, s, tm);
}

cudaError_t sm103_triangle_attention(const TriAttnLaunch& l, cudaStream_t s, LaunchTimer* tm) {
    const int I = l.I, Ip = l.I_pad;
    static std::atomic<uint64_t> attr_set{0};
    const int dev = current_device();
    const uint64_t dev_bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
    if (!(attr_set.load(std::memory_order_acquire) & dev_bit)) {
        cudaError_t e = cudaFuncSetAttribute(sm103_attention<false, false, false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, k2::Lay<false>::kSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(sm103_attention<true, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     k2::Lay<true>::kSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(sm103_attention<false, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     k2::Lay<false>::kSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(sm103_attention<true, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     k2::Lay<true>::kSmem);
        if (e != cudaSuccess) return e;
        attr_set.fetch_or(dev_bit, std::memory_order_release);
    }
    CUtensorMap mQ, mK, mV, mB, mWo;
    const uint64_t rows_qk = (uint64_t)I * NH * Ip;
    if (!map2d(&mQ, l.q, HD, rows_qk, HD * 2, HD, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !map2d(&mK, l.k, HD, rows_qk, HD * 2, HD, k2::kKT, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !map2d(&mV, l.vt, Ip, (uint64_t)I * NH * HD, (uint64_t)Ip * 2, 64, HD, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !map2d(&mB, l.bias, Ip, (uint64_t)NH * Ip, (uint64_t)Ip * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !map2d(&mWo, l.wo_t, CH, CZ, CH * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    cudaError_t e;
    uint64_t* kbits = nullptr;
    if (l.pair_mask != nullptr) {
        kbits = l.kbits;
        const int words = Ip / 64 + 1;
        if (tm) tm->begin("sm103_pair_keybits", s);
        sm103_pair_keybits<<<(unsigned)(((long long)I * words * 32 + 255) / 256), 256, 0, s>>>(l.pair_mask, l.node, I,
                                                                                           I, words, kbits);
        if (tm) tm->end(s);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const int cs = chunk_size(I, l.key_chunks);
    for (int k0 = 0; k0 < I; k0 += cs) {
        const int k1e = k0 + cs < I ? k0 + cs : I;
        AttnParams ap;
        ap.node = l.node;
        ap.I = I;
        ap.I_pad = Ip;
        ap.k_begin = k0;
        ap.k_end = k1e;
        ap.nk = (k1e - k0 + k2::kKT - 1) / k2::kKT;
        ap.first = k0 == 0;
        ap.last = k1e == I;
        ap.mask = l.mask;
        ap.pmask = l.pair_mask;
        ap.kbits = kbits;
        ap.Z = l.Z_resid;
        ap.g = l.g;
        ap.bo = l.bo;
        ap.o_run = l.o_run;
        ap.lse_run = l.lse_run;
        ap.out = l.out;
        ap.status = l.status;
        ap.inject = k0 == 0 ? l.inject : 0;
        ap.u = nullptr;
        ap.n_xb = Ip / 256;
        ap.lines = I;
        ap.n_items = ap.n_xb * I;
        ap.work = l.work;
        const dim3 grid(ap.n_items < num_sms() ? ap.n_items : num_sms());   // persistent: one CTA per SM
        e = cudaMemsetAsync(l.work, 0, sizeof(int), s);
        if (e != cudaSuccess) return e;
        const bool ex = ap.kbits != nullptr || ap.Z != nullptr;
        if (tm) tm->begin("sm103_attention", s);
        if (l.f32) {
            if (ex)
                sm103_attention<true, false, true><<<grid, k2::kThreads, k2::Lay<true>::kSmem, s>>>(mQ, mK, mV, mB, mWo, ap);
            else
                sm103_attention<false, false, true><<<grid, k2::kThreads, k2::Lay<false>::kSmem, s>>>(mQ, mK, mV, mB, mWo, ap);
        } else {
            if (ex)
                sm103_attention<true, false><<<grid, k2::kThreads, k2::Lay<true>::kSmem, s>>>(mQ, mK, mV, mB, mWo, ap);
            else
                sm103_attention<false, false><<<grid, k2::kThreads, k2::Lay<false>::kSmem, s>>>(mQ, mK, mV, mB, mWo, ap);
        }
        if (tm) tm->end(s);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

bool sm103_map2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t row_bytes, uint32_t box_cols,
                 uint32_t box_rows, int swizzle_bytes, bool bf16) {
    const CUtensorMapSwizzle sw = swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                        : CU_TENSOR_MAP_SWIZZLE_NONE;
    return map2d(m, base, cols, rows, row_bytes, box_cols, box_rows, sw,
                 bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
}

bool sm103_map_f32(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                   const uint32_t* box, int swizzle_bytes) {
    auto fn = encode_fn();
    if (!fn || rank < 1 || rank > 3) return false;
    cuuint64_t d[3], st[2];
    cuuint32_t b[3], es[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        if (i > 0) st[i - 1] = strides[i - 1];
    }
    const CUtensorMapSwizzle sw = swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rank, const_cast<void*>(base), d, st, b, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool sm103_map3d_bf16(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                      uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2, int swizzle_bytes) {
    return map3d(m, base, d0, d1, d2, s1, s2, b0, b1, b2,
                 swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

// MSA row attention on the attention kernel's MSA build: per key chunk, one
// launch over (query blocks, S lines, head halves 0-3 and 4-7).
cudaError_t sm103_msa_attention(const MsaAttnArgs& m, cudaStream_t s, LaunchTimer* tm) {
    static std::atomic<uint64_t> attr_set{0};
    const int dev = current_device();
    const uint64_t dev_bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
    if (!(attr_set.load(std::memory_order_acquire) & dev_bit)) {
        cudaError_t e = cudaFuncSetAttribute(sm103_attention<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             k2::Lay<true>::kSmem);
        if (e != cudaSuccess) return e;
        attr_set.fetch_or(dev_bit, std::memory_order_release);
    }
    const int Ip = m.I_pad;
    const uint64_t rows_qk = (uint64_t)m.S * 8 * Ip;
    CUtensorMap mQ, mK, mV, mB;
    if (!map2d(&mQ, m.q, HD, rows_qk, HD * 2, HD, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !map2d(&mK, m.k, HD, rows_qk, HD * 2, HD, k2::kKT, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !map2d(&mV, m.vt, Ip, (uint64_t)m.S * 8 * HD, (uint64_t)Ip * 2, 64, HD, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !map2d(&mB, m.bias, Ip, (uint64_t)8 * Ip, (uint64_t)Ip * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    cudaError_t e;
    uint64_t* kbits = nullptr;
    if (m.msa_mask != nullptr) {
        kbits = m.kbits;
        const int words = Ip / 64 + 1;
        if (tm) tm->begin("sm103_pair_keybits", s);
        sm103_pair_keybits<<<(unsigned)(((long long)m.S * words * 32 + 255) / 256), 256, 0, s>>>(m.msa_mask,
                                                                                              TRI_ATTN_STARTING, m.I, m.S, words,
                                                                    kbits);
        if (tm) tm->end(s);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const int cs = chunk_size(m.I, m.key_chunks);
    for (int k0 = 0; k0 < m.I; k0 += cs) {
        const int k1e = k0 + cs < m.I ? k0 + cs : m.I;
        {
            AttnParams ap{};
            ap.node = TRI_ATTN_STARTING;
            ap.I = m.I;
            ap.I_pad = Ip;
            ap.k_begin = k0;
            ap.k_end = k1e;
            ap.nk = (k1e - k0 + k2::kKT - 1) / k2::kKT;
            ap.first = k0 == 0;
            ap.last = k1e == m.I;
            ap.u = m.u;
            ap.mask = nullptr;
            ap.pmask = m.msa_mask;
            ap.kbits = kbits;
            ap.Z = nullptr;
            ap.g = m.g;
            ap.bo = nullptr;
            ap.o_run = m.o_run;
            ap.lse_run = m.lse_run;
            ap.out = nullptr;
            ap.status = m.status;
            ap.inject = 0;
            ap.n_xb = Ip / 256;
            ap.lines = m.S;
            ap.n_items = ap.n_xb * m.S * (8 / NH);
            ap.work = m.work;
            const dim3 grid(ap.n_items < num_sms() ? ap.n_items : num_sms());   // persistent: one CTA per SM
            if ((e = cudaMemsetAsync(m.work, 0, sizeof(int), s)) != cudaSuccess) return e;
            if (tm) tm->begin("sm103_attention", s);
            sm103_attention<true, true><<<grid, k2::kThreads, k2::Lay<true>::kSmem, s>>>(mQ, mK, mV, mB, mB, ap);
            if (tm) tm->end(s);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

}  // namespace tri_attn
