// sm_103a tensor-core path of MSA row-wise gated attention with pair bias
// (bf16 MSA, pair representation and weights; c_m = 256, c_z = 128, 8 heads of
// 32; f16 intermediates as on the triangle path).
//
// Source: "通量提升达 23.11 倍！至强® 可扩展平台助力 AlphaFold2 端到端优化"
// (Intel), step 4: the Evoformer's attention call takes the query rows of the
// MSA, a per-row (batched) mask and a bias shared by every row (non-batched,
// from the pair representation).  The operation is stated in tri_attn.h.
//
// Kernels per forward:
//   sm103_msa_prep   folds LayerNorm_m's gamma into W_q | W_k | W_v | W_g (the
//                    projection GEMM then runs on the raw MSA rows:
//                    LN(m) W = rstd * (m (gamma.W) - mu * colsum) + beta W),
//                    the gamma_z-folded pair-bias weights, and W_o^T in f16.
//   sm103_msa_bias   the pair bias of the 8 heads from Z (one warp per pair:
//                    LayerNorm_z and 8 dot products of length 128), log2(e)
//                    scaled, f16; padded keys get -30000 (finite, as on the
//                    triangle path: 2^-30000 is 0 in fp32).
//   sm103_msa_gemm<0>  persistent tcgen05 GEMM, one 128-column block of the
//                    1024 projection columns per CTA (its 64 KB of weights
//                    resident in shared memory), 128 MSA positions per tile,
//                    K = 256 in 16 MMAs of K = 16 into a double-buffered TMEM
//                    accumulator; the epilogue finishes the LayerNorm and writes
//                    q (log2(e)/sqrt(d) folded in), k, v^T and the sigmoid gate
//                    in the layouts of the attention kernel.
//   sm103_attention (MSA build, in sm103_kernels.cu): two launches of four
//                    heads over the S rows; the MSA mask excludes keys per row
//                    through the pair-mask key bits; each head's gated output
//                    u goes to global memory.
//   sm103_msa_gemm<1>  the same GEMM for out = u W_o (f16 operands), the output
//                    bias, the MSA mask (masked positions are 0, or Ms with the
//                    residual) and the residual in the epilogue.
#include <atomic>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sm103_ptx.cuh"
#include "tri_attn_internal.h"

namespace tri_attn {
namespace {

using namespace ptx;

constexpr int CM = 256;                     // MSA channels
constexpr int CZ = 128;                     // pair channels
constexpr int HM = 8;                       // heads
constexpr int HD = 32;                      // head dim
constexpr int CH = HM * HD;                 // 256 gated channels
constexpr int NPROJ = 4 * CH;               // 1024 projection columns: q | k | v | g
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMaskedBias = -30000.f;

__device__ __forceinline__ void set_abort(volatile int* abort, uint32_t* status, uint32_t code) {
    *abort = 1;
    atomicOr(status, code);
}

// Block-uniform read of the device status word.
__device__ __forceinline__ bool status_set(const uint32_t* status) {
    __shared__ int skip;
    if (threadIdx.x == 0) skip = *reinterpret_cast<const volatile uint32_t*>(status) != 0;
    __syncthreads();
    return skip != 0;
}

// =====================================================================================
// Weight preparation
// =====================================================================================
struct MsaPrepArgs {
    const float *gm, *bm, *gz, *bz, *b_g, *b_o;
    const __nv_bfloat16 *w_q, *w_k, *w_v, *w_g, *w_b, *w_o;
    __nv_bfloat16* wprep;   // [1024][256]: row n = (gamma_m . W)[:, n], K-major
    float* cst;             // [512][4]: per column pair {colsum(n), colsum(n+1), off(n), off(n+1)}
    float* wb;              // [128][8] gamma_z . W_b, then bcs[8] (column sums), bbw[8] (beta_z W_b)
    __half* wo_t;           // [256][256]: row n = W_o[:, n]
    float* bo;              // [256]
};

// Blocks 0..1023: projection column n; 1024..1279: row of W_o^T; 1280: the pair-bias weights.
__global__ void __launch_bounds__(256) sm103_msa_prep(MsaPrepArgs a) {
    __shared__ float red[2][8];
    const int n = blockIdx.x, c = threadIdx.x;
    if (n < NPROJ) {
        const int grp = n / CH, col = n % CH;     // q | k | v | g
        const __nv_bfloat16* W = grp == 0 ? a.w_q : grp == 1 ? a.w_k : grp == 2 ? a.w_v : a.w_g;
        const float wv = __bfloat162float(W[c * CH + col]);
        const __nv_bfloat16 r = __float2bfloat16_rn(a.gm[c] * wv);
        a.wprep[(size_t)n * CM + c] = r;
        float wr = __bfloat162float(r), bw = a.bm[c] * wv;
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
            float cs = 0.f, b = 0.f;
            for (int i = 0; i < 8; ++i) {
                cs += red[0][i];
                b += red[1][i];
            }
            const float sc = grp == 0 ? kLog2e * rsqrtf((float)HD) : 1.f;
            a.cst[(n >> 1) * 4 + (n & 1)] = cs;
            a.cst[(n >> 1) * 4 + 2 + (n & 1)] = b * sc + (grp == 3 ? a.b_g[col] : 0.f);
        }
    } else if (n < NPROJ + CM) {
        const int row = n - NPROJ;                // output channel of W_o
        a.wo_t[row * CH + c] = __float2half_rn(__bfloat162float(a.w_o[(size_t)c * CM + row]));
        if (c == 0) a.bo[row] = a.b_o ? a.b_o[row] : 0.f;
    } else {
        // gamma_z . W_b [128][8], its column sums and beta_z W_b
        float* bcs = a.wb + CZ * HM;
        float* bbw = bcs + HM;
        for (int i = c; i < CZ * HM; i += blockDim.x) {
            const int cc = i / HM;
            a.wb[i] = a.gz[cc] * __bfloat162float(a.w_b[i]);
        }
        __syncthreads();
        if (c < HM) {
            float cs = 0.f, b = 0.f;
            for (int cc = 0; cc < CZ; ++cc) {
                cs += a.wb[cc * HM + c];
                b += a.bz[cc] * __bfloat162float(a.w_b[cc * HM + c]);
            }
            bcs[c] = cs;
            bbw[c] = b;
        }
    }
}

// =====================================================================================
// Pair bias of the 8 heads: bias[h][i][j] = log2(e) * LN_z(Z[i, j]) . W_b[:, h]
// =====================================================================================
// One warp per pair (i, j) of the padded I_pad x I_pad grid.  Lane l holds channels
// 4l .. 4l+3.  LN(z) . W_b = rstd * (z . (gamma W_b) - mu * colsum) + beta W_b.
__global__ void __launch_bounds__(256) sm103_msa_bias(const __nv_bfloat16* Z, int I, int I_pad, float eps,
                                                      const float* wb, __half* bias) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= I_pad * I_pad) return;
    const int i = warp / I_pad, j = warp % I_pad;
    float v = 0.f;
    if (i < I && j < I) {
        const uint2 raw = reinterpret_cast<const uint2*>(Z + ((size_t)i * I + j) * CZ)[lane];
        float z[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                      __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
        float s1 = z[0] + z[1] + z[2] + z[3];
        for (int o = 16; o; o >>= 1) s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        const float mu = s1 * (1.f / CZ);
        float s2 = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) s2 = fmaf(z[e] - mu, z[e] - mu, s2);
        for (int o = 16; o; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
        const float rstd = rsqrtf(s2 * (1.f / CZ) + eps);
        const float* bcs = wb + CZ * HM;
        const float* bbw = bcs + HM;
        float part[HM];
#pragma unroll
        for (int h = 0; h < HM; ++h) {
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) acc = fmaf(z[e], wb[(4 * lane + e) * HM + h], acc);
            part[h] = acc;
        }
#pragma unroll
        for (int h = 0; h < HM; ++h)
            for (int o = 16; o; o >>= 1) part[h] += __shfl_xor_sync(0xffffffffu, part[h], o);
        if (lane < HM) {
            float dot = part[0];
#pragma unroll
            for (int h = 1; h < HM; ++h)
                if (lane == h) dot = part[h];
            v = (rstd * (dot - mu * bcs[lane]) + bbw[lane]) * kLog2e;
        }
    } else if (i < I) {
        v = kMaskedBias;                         // padded key
    }
    if (lane < HM) bias[((size_t)lane * I_pad + i) * I_pad + j] = __float2half_rn(v);
}

// =====================================================================================
// Row GEMM: [128 rows x K = 256] x [256 x 128-column block], persistent per block
// =====================================================================================
namespace kg {
constexpr int kThreads = 256;                // warp 0 TMA producer, warp 1 MMA issuer, warps 4-7 epilogue
constexpr int kB = 0;                        // B block: 4 K-chunks x [128 rows x 128 B] (SW128), 64 KB
constexpr int kA = 65536;                    // A stages: 2 x 4 K-chunks x [128 rows x 128 B] (SW128)
constexpr int kABytes = 65536;
constexpr int kBar = kA + 2 * kABytes;
constexpr int kSmem = kBar + 256 + 1024;
static_assert(kSmem <= 232448, "dynamic shared memory above the per-block limit");
}  // namespace kg

struct GemmParams {
    int S, I, I_pad, n_tiles;                // tiles of 128 (row, residue) positions over S x I_pad
    float eps;
    const float* cst;                        // mode 0
    __half *q, *k, *vt, *g;                  // mode 0 outputs
    const float* bo;                         // mode 1
    const uint8_t* mask;                     // mode 1: [S, I] or NULL
    const __nv_bfloat16* resid;              // mode 1: Ms [S, I, 256] or NULL
    __nv_bfloat16* out;                      // mode 1: [S, I, 256]
    uint32_t* status;
};

// MODE 0: the MSA projection (A = Ms, bf16, through a 3-D map [S][I][256] whose
// residue extent zero-fills the padded positions; epilogue: LayerNorm fold, q / k /
// v^T / gate).  MODE 1: the output projection (A = u, f16, [S * I_pad][256];
// epilogue: + b_o, MSA mask, residual, bf16 store).
template <int MODE>
__global__ void __launch_bounds__(kg::kThreads, 1)
sm103_msa_gemm(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB, GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    if (status_set(p.status)) return;
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kg::kBar);
    uint64_t* b_full = bars + 0;
    uint64_t* a_full = bars + 1;      // [2]
    uint64_t* a_empty = bars + 3;     // [2]: the MMA's commit (+ the 4 epilogue warps in MODE 0)
    uint64_t* acc_full = bars + 5;    // [2]
    uint64_t* acc_empty = bars + 7;   // [2]: 4 epilogue warps
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 9);
    volatile int* abort = reinterpret_cast<volatile int*>(bars + 10);
    uint64_t* mma_done = bars + 11;   // every MMA of this block retired (before the TMEM is freed)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cb = blockIdx.x;                // 128-column block of the output
    const int tpl = p.I_pad / 128;            // tiles per MSA row
    if (threadIdx.x == 0) {
        mbar_init(b_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(a_full + s, 1);
            mbar_init(a_empty + s, MODE == 0 ? 5 : 1);
            mbar_init(acc_full + s, 1);
            mbar_init(acc_empty + s, 4);
        }
        mbar_init(mma_done, 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        int issued = 0;
        bool ok = true;
        if (lane == 0) {
            prefetch_tmap(&mapA);
            prefetch_tmap(&mapB);
            mbar_arrive_expect_tx(b_full, 65536);
            for (int kc = 0; kc < 4; ++kc) tma_load_2d(sm + kg::kB + kc * 16384, &mapB, b_full, kc * 64, cb * 128);
            int j = 0;
            for (int t = blockIdx.y; t < p.n_tiles; t += gridDim.y, ++j) {
                const int st = j & 1;
                if (!mbar_wait(a_empty + st, ((j >> 1) & 1) ^ 1, abort)) {
                    ok = false;
                    break;
                }
                uint8_t* dst = sm + kg::kA + st * kg::kABytes;
                mbar_arrive_expect_tx(a_full + st, kg::kABytes);
                if (MODE == 0) {
                    const int s = t / tpl, i0 = (t % tpl) * 128;
                    for (int kc = 0; kc < 4; ++kc) tma_load_3d(dst + kc * 16384, &mapA, a_full + st, kc * 64, i0, s);
                } else {
                    for (int kc = 0; kc < 4; ++kc) tma_load_2d(dst + kc * 16384, &mapA, a_full + st, kc * 64, t * 128);
                }
                issued = j + 1;
            }
            volatile int keep_waiting = 0;
            mbar_wait(b_full, 0, &keep_waiting);
            if (!ok) {
                set_abort(abort, p.status, kStatusTimeoutProducer);
                // the last copy into each A stage lands before the block ends
                for (int st = 0; st < 2; ++st) {
                    const int jl = issued - 1 - ((issued - 1 - st) % 2 + 2) % 2;
                    if (jl >= 0) mbar_wait(a_full + st, (jl >> 1) & 1, &keep_waiting);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = MODE == 0 ? idesc_bf16_f32(128, 128) : idesc_f16_f32(128, 128);
            bool ok = mbar_wait(b_full, 0, abort);
            int j = 0;
            for (int t = blockIdx.y; ok && t < p.n_tiles; t += gridDim.y, ++j) {
                const int st = j & 1, ab = j & 1;
                if (!mbar_wait(a_full + st, (j >> 1) & 1, abort) || !mbar_wait(acc_empty + ab, ((j >> 1) & 1) ^ 1, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t abase = smem_u32(sm + kg::kA + st * kg::kABytes), bbase = smem_u32(sm + kg::kB);
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) {
                    const uint64_t ad = sdesc(abase + (kk >> 2) * 16384 + (kk & 3) * 32, 1024, kSwizzle128);
                    const uint64_t bd = sdesc(bbase + (kk >> 2) * 16384 + (kk & 3) * 32, 1024, kSwizzle128);
                    mma_ss(tmem + ab * 128, ad, bd, idesc, kk > 0 ? 1u : 0u);
                }
                tc_commit(acc_full + ab);
                tc_commit(a_empty + st);
            }
            if (!ok) set_abort(abort, p.status, kStatusTimeoutMma);
            tc_commit(mma_done);
            volatile int keep_waiting = 0;
            mbar_wait(mma_done, 0, &keep_waiting);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue (one thread per row)
        const int wq = warp - 4;
        const int r = wq * 32 + lane;
        const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        int j = 0;
        bool ok = true;
        for (int t = blockIdx.y; t < p.n_tiles; t += gridDim.y, ++j) {
            const int st = j & 1, ab = j & 1;
            const int s = t / tpl, i = (t % tpl) * 128 + r;
            float mu = 0.f, rstd = 0.f;
            if (MODE == 0) {
                // LayerNorm statistics of this row from the staged tile (4 K-chunks of 128 B),
                // shifted by its first channel
                if (!mbar_wait(a_full + st, (j >> 1) & 1, abort)) { ok = false; break; }
                const uint8_t* row = sm + kg::kA + st * kg::kABytes + r * 128;
                const float shift = bf16lo(*reinterpret_cast<const uint32_t*>(row + ((0 ^ (r & 7)) << 4)));
                float sd = 0.f, sq = 0.f;
#pragma unroll 4
                for (int cc = 0; cc < 32; ++cc) {
                    const uint4 v = *reinterpret_cast<const uint4*>(row + (cc >> 3) * 16384 + (((cc & 7) ^ (r & 7)) << 4));
                    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2) {
                        const float d0 = bf16lo(w4[q2]) - shift, d1 = bf16hi(w4[q2]) - shift;
                        sd += d0 + d1;
                        sq = fmaf(d0, d0, fmaf(d1, d1, sq));
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(a_empty + st);
                const float md = sd * (1.f / CM);
                mu = shift + md;
                rstd = rsqrtf(fmaxf(sq * (1.f / CM) - md * md, 0.f) + p.eps);
            }
            if (!mbar_wait(acc_full + ab, (j >> 1) & 1, abort)) { ok = false; break; }
            tc_fence_after();
            const uint32_t tacc = tl + ab * 128;
            if (MODE == 0) {
                const int grp = cb >> 1;                 // 0 q, 1 k, 2 v, 3 gate
                const float rr = grp == 0 ? rstd * (kLog2e * rsqrtf((float)HD)) : rstd;
                const float nmu = -mu;
#pragma unroll 1
                for (int hh = 0; hh < 4; ++hh) {
                    const int head = (cb & 1) * 4 + hh;
                    uint32_t acc[32];
                    tmem_ld32(tacc + hh * 32, acc);
                    tmem_ld_wait();
                    const float4* cst = reinterpret_cast<const float4*>(p.cst) + ((cb * 128 + hh * 32) >> 1);
                    uint32_t o[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float4 c = cst[e >> 1];
                        float t0, t1, v0, v1;
                        fma2(t0, t1, nmu, nmu, c.x, c.y, __uint_as_float(acc[e]), __uint_as_float(acc[e + 1]));
                        fma2(v0, v1, rr, rr, t0, t1, c.z, c.w);
                        if (grp == 3) {                   // sigmoid(v) = 0.5 tanh(v / 2) + 0.5
                            v0 = fmaf(0.5f, tanh_approx(0.5f * v0), 0.5f);
                            v1 = fmaf(0.5f, tanh_approx(0.5f * v1), 0.5f);
                        }
                        o[e >> 1] = pack_f16(v0, v1);
                    }
                    const size_t lh = (size_t)s * HM + head;
                    if (grp == 2) {                       // v^T: [S][8][32][I_pad]
                        unsigned short* dst = reinterpret_cast<unsigned short*>(p.vt + lh * HD * p.I_pad + i);
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            dst[(size_t)e * p.I_pad] = static_cast<unsigned short>(o[e >> 1] & 0xFFFFu);
                            dst[(size_t)(e + 1) * p.I_pad] = static_cast<unsigned short>(o[e >> 1] >> 16);
                        }
                    } else {                               // q, k, gate: [S][8][I_pad][32]
                        __half* base = grp == 0 ? p.q : grp == 1 ? p.k : p.g;
                        uint4* dst = reinterpret_cast<uint4*>(base + (lh * p.I_pad + i) * HD);
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4)
                            dst[c4] = make_uint4(o[4 * c4], o[4 * c4 + 1], o[4 * c4 + 2], o[4 * c4 + 3]);
                    }
                }
            } else {
                const bool row_ok = i < p.I;
                const size_t pos = (size_t)s * p.I + i;
                const bool valid = row_ok && (p.mask == nullptr || p.mask[pos] != 0);
#pragma unroll 1
                for (int cq = 0; cq < 4; ++cq) {
                    uint32_t acc[32];
                    tmem_ld32(tacc + cq * 32, acc);
                    tmem_ld_wait();
                    if (row_ok) {
                        const int c0 = cb * 128 + cq * 32;
                        uint32_t zr[16];
                        if (p.resid) {
                            const uint4* rp = reinterpret_cast<const uint4*>(p.resid + pos * CM + c0);
#pragma unroll
                            for (int c4 = 0; c4 < 4; ++c4) {
                                const uint4 v = rp[c4];
                                zr[4 * c4] = v.x;
                                zr[4 * c4 + 1] = v.y;
                                zr[4 * c4 + 2] = v.z;
                                zr[4 * c4 + 3] = v.w;
                            }
                        }
                        uint32_t o[16];
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            float a0 = valid ? __uint_as_float(acc[e]) + p.bo[c0 + e] : 0.f;
                            float a1 = valid ? __uint_as_float(acc[e + 1]) + p.bo[c0 + e + 1] : 0.f;
                            if (p.resid) {
                                a0 += bf16lo(zr[e >> 1]);
                                a1 += bf16hi(zr[e >> 1]);
                            }
                            o[e >> 1] = pack_bf16(a0, a1);
                        }
                        uint4* dst = reinterpret_cast<uint4*>(p.out + pos * CM + c0);
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4)
                            dst[c4] = make_uint4(o[4 * c4], o[4 * c4 + 1], o[4 * c4 + 2], o[4 * c4 + 3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty + ab);
        }
        if (!ok) set_abort(abort, p.status, kStatusTimeoutEpilogue);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
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

bool sm103_msa_supported(int c_m, int c_z, int H, int d, int dtype) {
    return dtype == TRI_ATTN_BF16 && c_m == CM && c_z == CZ && H == HM && d == HD;
}

cudaError_t sm103_msa_forward(const MsaArgs& a, cudaStream_t s, LaunchTimer* tm) {
    const Workspace& W = *a.lay;
    char* ws = a.ws;
    auto hf = [&](size_t off) { return reinterpret_cast<__half*>(ws + off); };
    auto f32 = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
    const int S = a.S, I = a.I, Ip = W.I_pad;
    cudaError_t e;

    static std::atomic<uint64_t> attr_set{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t dev_bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
    if (!(attr_set.load(std::memory_order_acquire) & dev_bit)) {
        if ((e = cudaFuncSetAttribute(sm103_msa_gemm<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kg::kSmem)) !=
                cudaSuccess ||
            (e = cudaFuncSetAttribute(sm103_msa_gemm<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kg::kSmem)) !=
                cudaSuccess)
            return e;
        attr_set.fetch_or(dev_bit, std::memory_order_release);
    }

    // ---- weights
    MsaPrepArgs pa{a.w.ln_m_gamma, a.w.ln_m_beta, a.w.ln_z_gamma, a.w.ln_z_beta, a.w.b_g, a.w.b_o,
                   static_cast<const __nv_bfloat16*>(a.w.w_q), static_cast<const __nv_bfloat16*>(a.w.w_k),
                   static_cast<const __nv_bfloat16*>(a.w.w_v), static_cast<const __nv_bfloat16*>(a.w.w_g),
                   static_cast<const __nv_bfloat16*>(a.w.w_b), static_cast<const __nv_bfloat16*>(a.w.w_o),
                   reinterpret_cast<__nv_bfloat16*>(ws + W.wprep), f32(W.cst), f32(W.wb32), hf(W.wo_t), f32(W.bo)};
    if (tm) tm->begin("sm103_msa_prep", s);
    sm103_msa_prep<<<NPROJ + CM + 1, 256, 0, s>>>(pa);
    if (tm) tm->end(s);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    // ---- pair bias of the 8 heads
    {
        const long long warps = (long long)Ip * Ip;
        if (tm) tm->begin("sm103_msa_bias", s);
        sm103_msa_bias<<<(unsigned)((warps + 7) / 8), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(a.Z), I, Ip, a.eps,
                                                                   f32(W.wb32), hf(W.bias));
        if (tm) tm->end(s);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }

    const int n_tiles = S * (Ip / 128);
    const int rows_per_block = num_sms_of_device() / 8 > 0 ? num_sms_of_device() / 8 : 1;

    // ---- projection GEMM: q | k | v^T | gate
    {
        CUtensorMap mA, mB;
        if (!sm103_map3d_bf16(&mA, a.M, CM, I, S, (uint64_t)CM * 2, (uint64_t)I * CM * 2, 64, 128, 1) ||
            !sm103_map2d(&mB, ws + W.wprep, CM, NPROJ, CM * 2, 64, 128, 128, true))
            return cudaErrorInvalidValue;
        GemmParams gp{};
        gp.S = S;
        gp.I = I;
        gp.I_pad = Ip;
        gp.n_tiles = n_tiles;
        gp.eps = a.eps;
        gp.cst = f32(W.cst);
        gp.q = hf(W.q);
        gp.k = hf(W.k);
        gp.vt = hf(W.v);
        gp.g = hf(W.g);
        gp.status = a.status;
        dim3 grid(NPROJ / 128, rows_per_block < n_tiles ? rows_per_block : n_tiles);
        if (tm) tm->begin("sm103_msa_proj", s);
        sm103_msa_gemm<0><<<grid, kg::kThreads, kg::kSmem, s>>>(mA, mB, gp);
        if (tm) tm->end(s);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }

    // ---- attention (two launches of four heads per key chunk), gated u to global memory
    {
        MsaAttnArgs m{S, I, Ip, a.key_chunks, hf(W.q), hf(W.k), hf(W.v), hf(W.g), hf(W.bias), hf(W.u),
                      W.o_run ? f32(W.o_run) : nullptr, W.lse_run ? f32(W.lse_run) : nullptr, a.msa_mask,
                      reinterpret_cast<uint64_t*>(ws + W.kbits), a.status};
        if ((e = sm103_msa_attention(m, s, tm)) != cudaSuccess) return e;
    }

    // ---- output projection: out = u W_o + b_o (MSA mask, residual)
    {
        CUtensorMap mA, mB;
        if (!sm103_map2d(&mA, ws + W.u, CH, (uint64_t)S * Ip, CH * 2, 64, 128, 128, false) ||
            !sm103_map2d(&mB, ws + W.wo_t, CH, CM, CH * 2, 64, 128, 128, false))
            return cudaErrorInvalidValue;
        GemmParams gp{};
        gp.S = S;
        gp.I = I;
        gp.I_pad = Ip;
        gp.n_tiles = n_tiles;
        gp.bo = f32(W.bo);
        gp.mask = a.msa_mask;
        gp.resid = a.residual ? static_cast<const __nv_bfloat16*>(a.M) : nullptr;
        gp.out = static_cast<__nv_bfloat16*>(a.out);
        gp.status = a.status;
        const int rpb = num_sms_of_device() / 2;
        dim3 grid(CM / 128, rpb < n_tiles ? rpb : n_tiles);
        if (tm) tm->begin("sm103_msa_out", s);
        sm103_msa_gemm<1><<<grid, kg::kThreads, kg::kSmem, s>>>(mA, mB, gp);
        if (tm) tm->end(s);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace tri_attn
