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
//   sm103_msa_front  three independent steps in one launch, block ranges side by
//                    side:
//                    - weight preparation: folds LayerNorm_m's gamma into W_q |
//                      W_k | W_v | W_g (the projection GEMM then runs on the raw
//                      MSA rows: LN(m) W = rstd * (m (gamma.W) - mu * colsum) +
//                      beta W), and W_o^T in f16;
//                    - LayerNorm_m mean and 1/std of every (row, residue) slot
//                      (four threads per slot), and its row of the LayerNorm
//                      K-step;
//                    - the pair bias of the 8 heads from Z (LayerNorm_z and 8 dot
//                      products of length 128 per pair, from a shared-memory copy
//                      of 64 pairs, with the gamma_z-folded weights formed in the
//                      block), log2(e) scaled, f16; padded keys get -30000
//                      (finite, as on the triangle path: 2^-30000 is 0 in fp32).
//   sm103_msa_gemm<0>  persistent tcgen05 GEMM, one 256-column group (q, k, v
//                    or gate) per CTA with its 128 KB of weights resident in
//                    shared memory, 128 MSA slots per tile, K = 256 in 16 MMAs of
//                    128 x 256 x 16 plus one K-step for the LayerNorm terms into a
//                    double-buffered TMEM accumulator; 8 epilogue warps scale by
//                    the slot's 1/std and write q (log2(e)/sqrt(d) folded in), k,
//                    v^T and the sigmoid gate in the layouts of the attention
//                    kernel.
//   sm103_attention (MSA build, in sm103_kernels.cu): one launch per key chunk,
//                    blockIdx.z picking heads 0-3 or 4-7 of an MSA row; the MSA
//                    mask excludes keys per row through the pair-mask key bits;
//                    each head's gated output u goes to global memory.
//   sm103_msa_gemm<1>  the same GEMM for out = u W_o + b_o (f16 operands; all
//                    256 output channels per CTA), the MSA mask (masked positions
//                    are 0, or Ms with the residual) and the residual in the
//                    epilogue.
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

// (hi, lo) split of x in bf16: two 16-bit codes whose sum is x to ~2^-16
__device__ __forceinline__ uint32_t split_bf16(float x) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    const __nv_bfloat16 l = __float2bfloat16_rn(x - __bfloat162float(h));
    return static_cast<uint32_t>(__bfloat16_as_ushort(h)) | (static_cast<uint32_t>(__bfloat16_as_ushort(l)) << 16);
}
// the same in f16
__device__ __forceinline__ uint32_t split_f16(float x) {
    const __half h = __float2half_rn(x);
    const __half l = __float2half_rn(x - __half2float(h));
    return static_cast<uint32_t>(__half_as_ushort(h)) | (static_cast<uint32_t>(__half_as_ushort(l)) << 16);
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
    __nv_bfloat16* wprep;   // [1024][256]: row n = (gamma_m . W)[:, n] (q columns x log2(e)/sqrt(d)), K-major
    float* cst;             // [2][1024]: colsum of each column, then its offset
    __half* wo_t;           // [256][256]: row n = W_o[:, n]
    float* bo;              // [256]
};

// Prep blocks 0..31: 32 projection columns each; 32..39: 32 rows of W_o^T each.
// The 32-column slab of W (all 256 input channels) is staged in shared memory
// with coalesced reads; each warp then writes 4 whole K-major rows (512 bytes,
// one 16-byte group of 8 channels per lane).
constexpr int kPrepCols = 32;
constexpr int kPrepBlocks = NPROJ / kPrepCols + CM / kPrepCols;

__device__ __forceinline__ void msa_prep_block(const MsaPrepArgs& a, int blk, float (*tile)[kPrepCols + 1]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (blk < NPROJ / kPrepCols) {
        const int n0 = blk * kPrepCols, grp = n0 / CH, col0 = n0 % CH;   // q | k | v | g
        const __nv_bfloat16* W = grp == 0 ? a.w_q : grp == 1 ? a.w_k : grp == 2 ? a.w_v : a.w_g;
        const float sc = grp == 0 ? kLog2e * rsqrtf((float)HD) : 1.f;   // q carries log2(e) / sqrt(d)
        for (int cc = warp; cc < CM; cc += 8) tile[cc][lane] = __bfloat162float(W[cc * CH + col0 + lane]) * sc;
        __syncthreads();
        for (int jj = 0; jj < kPrepCols / 8; ++jj) {
            const int j = warp * (kPrepCols / 8) + jj, n = n0 + j;
            uint32_t pk[4];
            float wr = 0.f, bw = 0.f;
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                const int cc = lane * 8 + e;
                const float w0 = tile[cc][j], w1 = tile[cc + 1][j];
                const __nv_bfloat16 r0 = __float2bfloat16_rn(a.gm[cc] * w0), r1 = __float2bfloat16_rn(a.gm[cc + 1] * w1);
                pk[e >> 1] = static_cast<uint32_t>(__bfloat16_as_ushort(r0)) |
                             (static_cast<uint32_t>(__bfloat16_as_ushort(r1)) << 16);
                wr += __bfloat162float(r0) + __bfloat162float(r1);
                bw = fmaf(a.bm[cc], w0, fmaf(a.bm[cc + 1], w1, bw));
            }
            reinterpret_cast<uint4*>(a.wprep + (size_t)n * CM)[lane] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            for (int o = 16; o; o >>= 1) {
                wr += __shfl_xor_sync(0xffffffffu, wr, o);
                bw += __shfl_xor_sync(0xffffffffu, bw, o);
            }
            if (lane == 0) {
                a.cst[n] = wr;
                a.cst[NPROJ + n] = bw + (grp == 3 ? a.b_g[col0 + j] : 0.f);
            }
        }
    } else {
        const int row0 = (blk - NPROJ / kPrepCols) * kPrepCols;   // output channels of W_o
        for (int cc = warp; cc < CH; cc += 8) tile[cc][lane] = __bfloat162float(a.w_o[(size_t)cc * CM + row0 + lane]);
        __syncthreads();
        for (int jj = 0; jj < kPrepCols / 8; ++jj) {
            const int j = warp * (kPrepCols / 8) + jj, row = row0 + j;
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) pk[e >> 1] = pack_f16(tile[lane * 8 + e][j], tile[lane * 8 + e + 1][j]);
            reinterpret_cast<uint4*>(a.wo_t + (size_t)row * CH)[lane] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            if (lane == 0) a.bo[row] = a.b_o ? a.b_o[row] : 0.f;
        }
    }
}

// =====================================================================================
// Pair bias of the 8 heads: bias[h][i][j] = log2(e) * LN_z(Z[i, j]) . W_b[:, h]
// =====================================================================================
// One block per (row i, 64 keys j0 .. j0+63).  Z[i, j0 .. j0+63, :] is one contiguous
// 16 KB run: it is staged in shared memory with coalesced 16-byte loads (rows padded
// to 264 B, which keeps the per-pair 8-byte reads below at two wavefronts a warp).  Thread (pair p, head
// pair hq) then forms the LayerNorm statistics of pair p (shifted by its first
// channel) and two of the 8 dot products:
//   LN(z) . W_b[:, h] = rstd * (z . (gamma W_b)[:, h] - mu * colsum_h) + (beta W_b)_h.
// The 8 x 64 results are staged again and leave as one 128-byte run per head.
// Each block first forms gamma_z . W_b, its column sums and beta_z . W_b itself
// (1024 products; the weight preparation runs in the same launch).
namespace kb {
constexpr int kPairs = 64;
constexpr int kRowBytes = CZ * 2 + 8;        // 264
}  // namespace kb

struct MsaBiasSmem {
    __align__(16) uint8_t zt[kb::kPairs * kb::kRowBytes];
    __align__(16) float wq[4][CZ][2];           // (gamma_z W_b) by head pair
    __align__(16) __half ob[HM][kb::kPairs];
    float part[2][32][HM];                      // partial column sums of gamma_z W_b and of beta_z W_b
    float bsum[2][HM];                          // their totals: bcs (column sums), bbw (beta_z W_b)
};

__device__ __forceinline__ void msa_bias_block(const __nv_bfloat16* Z, int I, int I_pad, float eps,
                                               const __nv_bfloat16* w_b, const float* gz, const float* bz,
                                               __half* bias, int bx, int by, MsaBiasSmem& sb) {
    auto& zt = sb.zt;
    auto& wq = sb.wq;
    auto& ob = sb.ob;
    const int tid = threadIdx.x;
    const int i = by, j0 = bx * kb::kPairs;
    if (i >= I) {                                          // padded query rows: 0
        if (tid < HM * 8) {
            const int h = tid >> 3, c = tid & 7;
            reinterpret_cast<uint4*>(bias + ((size_t)h * I_pad + i) * I_pad + j0)[c] = make_uint4(0, 0, 0, 0);
        }
        return;
    }
    const int nj = I - j0 < kb::kPairs ? I - j0 : kb::kPairs;   // valid keys in this block (may be <= 0)
    {
        const uint4* src = reinterpret_cast<const uint4*>(Z + ((size_t)i * I + j0) * CZ);
        for (int q = tid; q < kb::kPairs * (CZ / 8); q += 256) {
            const int pr = q >> 4, c = q & 15;                 // 16 x 16 B per pair
            const uint4 v = pr < nj ? src[q] : make_uint4(0, 0, 0, 0);
            uint2* dst = reinterpret_cast<uint2*>(zt + pr * kb::kRowBytes + c * 16);   // rows are 8-byte aligned
            dst[0] = make_uint2(v.x, v.y);
            dst[1] = make_uint2(v.z, v.w);
        }
        // gamma_z . W_b [128][8]: thread t owns head t % 8 over channels t / 8 + 32 k,
        // with partial column sums (and of beta_z W_b) reduced over the 32 threads of a head
        const int h = tid & (HM - 1);
        float cs = 0.f, b = 0.f;
        for (int cc = tid >> 3; cc < CZ; cc += 32) {
            const float wv = __bfloat162float(w_b[cc * HM + h]);
            const float g = gz[cc] * wv;
            wq[h >> 1][cc][h & 1] = g;
            cs += g;
            b = fmaf(bz[cc], wv, b);
        }
        sb.part[0][tid >> 3][h] = cs;
        sb.part[1][tid >> 3][h] = b;
    }
    __syncthreads();
    if (tid < 2 * HM) {
        const int hh = tid & (HM - 1), pl = tid < HM ? 0 : 1;
        float t = 0.f;
        for (int k = 0; k < 32; ++k) t += sb.part[pl][k][hh];
        sb.bsum[pl][hh] = t;
    }
    __syncthreads();
    const int pr = tid & 63, hq = tid >> 6;
    const uint8_t* row = zt + pr * kb::kRowBytes;
    const float shift = bf16lo(*reinterpret_cast<const uint32_t*>(row));
    float sd = 0.f, sq = 0.f, d0 = 0.f, d1 = 0.f;
#pragma unroll 8
    for (int c4 = 0; c4 < CZ / 4; ++c4) {
        const uint2 w = *reinterpret_cast<const uint2*>(row + c4 * 8);
        const float z[4] = {bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y)};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 wv = *reinterpret_cast<const float2*>(&wq[hq][c4 * 4 + e][0]);
            const float dz = z[e] - shift;
            sd += dz;
            sq = fmaf(dz, dz, sq);
            d0 = fmaf(z[e], wv.x, d0);
            d1 = fmaf(z[e], wv.y, d1);
        }
    }
    const float md = sd * (1.f / CZ);
    const float mu = shift + md;
    const float rstd = rsqrtf(fmaxf(sq * (1.f / CZ) - md * md, 0.f) + eps);
    const float* bcs = sb.bsum[0];
    const float* bbw = sb.bsum[1];
    const int h = 2 * hq;
    const bool valid = pr < nj;
    ob[h][pr] = __float2half_rn(valid ? (rstd * (d0 - mu * bcs[h]) + bbw[h]) * kLog2e : kMaskedBias);
    ob[h + 1][pr] = __float2half_rn(valid ? (rstd * (d1 - mu * bcs[h + 1]) + bbw[h + 1]) * kLog2e : kMaskedBias);
    __syncthreads();
    if (tid < HM * 8) {
        const int hh = tid >> 3, c = tid & 7;
        reinterpret_cast<uint4*>(bias + ((size_t)hh * I_pad + i) * I_pad + j0)[c] =
            reinterpret_cast<const uint4*>(&ob[hh][0])[c];
    }
}

// =====================================================================================
// LayerNorm_m statistics of every (row, residue) slot: rowstat[s * I_pad + i] = (mu, rstd)
// =====================================================================================
// Four threads per slot; thread q of a slot holds the 16-byte groups q, q + 4, ...,
// q + 28 of its 512-byte row (eight bf16 channels each), so each of the eight
// loads of a warp reads 64 contiguous bytes of each of its 8 slots.  Sums are
// shifted by the slot's first channel and combined over the four threads.
// Padded residues (i >= I) get (0, 1) and the K-step row of (mu, sd) = (0, 1),
// which makes their projections the plain offsets (finite; never attended to).
constexpr int kStatThreads = 256;
constexpr int kStatSlotsPerBlock = kStatThreads / 4;

__device__ __forceinline__ void msa_stats_block(const __nv_bfloat16* M, int S, int I, int I_pad, float eps,
                                                float2* rowstat, uint4* axrow, int blk) {
    const long long slot = (long long)blk * kStatSlotsPerBlock + (threadIdx.x >> 2);
    const int q = threadIdx.x & 3;
    const long long n_slots = (long long)S * I_pad;
    const bool in = slot < n_slots;
    const int s = in ? (int)(slot / I_pad) : 0, i = in ? (int)(slot % I_pad) : 0;
    const bool live = in && i < I;
    const uint4* src = reinterpret_cast<const uint4*>(M + ((size_t)s * I + i) * CM) + q;
    uint4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = live ? src[4 * k] : make_uint4(0, 0, 0, 0);
    const float shift = __shfl_sync(0xffffffffu, bf16lo(v[0].x), threadIdx.x & 28);   // channel 0
    float sd = 0.f, sq = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t w4[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float a = bf16lo(w4[e]) - shift, b = bf16hi(w4[e]) - shift;
            sd += a + b;
            sq = fmaf(a, a, fmaf(b, b, sq));
        }
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
        sd += __shfl_xor_sync(0xffffffffu, sd, o);
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
    }
    if (!in || q != 0) return;
    const float md = sd * (1.f / CM);
    const float mu = live ? shift + md : 0.f;
    const float var = fmaxf(sq * (1.f / CM) - md * md, 0.f) + eps;
    rowstat[slot] = make_float2(mu, live ? rsqrtf(var) : 1.f);
    // the slot's row of the projection's LayerNorm K-step: (-mu, -mu, sd, sd) as
    // bf16 (hi, lo) pairs, sd = sqrt(var) = 1 / rstd
    const uint32_t m2 = split_bf16(-mu), s2 = split_bf16(live ? sqrtf(var) : 1.f);
    axrow[slot] = make_uint4(m2, m2, s2, s2);
}

// =====================================================================================
// The three front steps of an MSA forward in one launch: they are independent of
// one another (each pair-bias block forms its own gamma_z-folded weights), so the
// weight preparation, the pair bias over Z and the LayerNorm_m statistics over the
// MSA rows share the GPU instead of running one after the other.  Blocks
// [0, kPrepBlocks) prepare weights, then n_stat blocks of statistics (64 slots
// each), then one pair-bias block per (64 keys, query row).
// =====================================================================================
struct MsaFrontArgs {
    MsaPrepArgs prep;
    const __nv_bfloat16 *M, *Z;
    int S, I, I_pad, n_stat, n_bias_x;
    float eps;
    float2* rowstat;
    uint4* axrow;
    __half* bias;
};
union MsaFrontSmem {
    float prep_tile[CM][kPrepCols + 1];
    MsaBiasSmem bias;
};
static_assert(kStatThreads == 256, "one block size for the fused front steps");

__global__ void __launch_bounds__(256) sm103_msa_front(MsaFrontArgs a) {
    __shared__ MsaFrontSmem sh;
    const int blk = blockIdx.x;
    if (blk < kPrepBlocks) {
        msa_prep_block(a.prep, blk, sh.prep_tile);
    } else if (blk < kPrepBlocks + a.n_stat) {
        msa_stats_block(a.M, a.S, a.I, a.I_pad, a.eps, a.rowstat, a.axrow, blk - kPrepBlocks);
    } else {
        const int b = blk - kPrepBlocks - a.n_stat;
        msa_bias_block(a.Z, a.I, a.I_pad, a.eps, a.prep.w_b, a.prep.gz, a.prep.bz, a.bias, b % a.n_bias_x,
                       b / a.n_bias_x, sh.bias);
    }
}

// =====================================================================================
// Row GEMM: [128 slots x K = 256] x [256 x 256 columns], persistent per block
// =====================================================================================
// One block owns 256 output columns (its 128 KB of K-major weights resident in
// shared memory) and walks 128-slot tiles.  N = 256 per MMA keeps the tensor
// core's shared-memory operand reads at 12 KB per 128 x 256 x 16 step (an N = 128
// step reads 8 KB for half the work, and with the TMA writes of A that saturates
// shared-memory bandwidth).  A arrives in K-chunks of 64 (16 KB) through a ring of
// 5 slots.  Per-column terms enter through one more K-step: a 16-wide A tile per
// 128 slots (`ax`) against a 16-wide B tile per column (`bx`), bf16 / f16 values
// split into a high and a low part so that the products are exact to ~2^-16:
//   MODE 0  ax = (-mu, -mu, sd, sd) as (hi, lo, hi, lo, ...), bx = (cs, cs, off, off)
//           so the accumulator holds m W' - mu cs + sd off and the epilogue
//           multiplies by rstd = 1 / sd: LN(m) W = rstd (m W' - mu cs) + off.
//   MODE 1  ax = (1, 1, 0, ...), bx = (b_o hi, b_o lo, 0, ...): the output bias.
// The epilogue (8 warps: two per TMEM lane quadrant, 128 columns each) stores
// straight from registers, so shared memory carries only operands.
namespace kg {
constexpr int kThreads = 384;                // warp 0 producer, warp 1 MMA issuer, warps 4-11 epilogue
constexpr int kEpiWarps = 8;
constexpr int kSlots = 5;                    // A ring: 5 x [128 rows x 64 K] (SW128)
constexpr int kB = 0;                        // B: 4 K-chunks x [256 rows x 128 B] (SW128), 128 KB
constexpr int kA = 131072;
constexpr int kBX = kA + kSlots * 16384;     // bx: 256 rows x 16 B (no swizzle)
constexpr int kAX = kBX + 4096;              // ax: 2 x [128 rows x 16 B]
constexpr int kZero = kAX + 4096;            // 4 KB of zeros: K columns 8 .. 15 of ax and bx
constexpr int kBar = kZero + 4096;
constexpr int kSmem = kBar + 256 + 1024;
static_assert(kSmem <= 232448, "dynamic shared memory above the per-block limit");
static_assert(kA % 1024 == 0 && kBX % 1024 == 0, "SW128 tiles need 1024-byte alignment");
}  // namespace kg

struct GemmParams {
    int S, I, I_pad, n_tiles;                // tiles of 128 (row, residue) slots over S x I_pad
    const float* cst;                        // mode 0: [2][1024] column sums, then offsets
    const float2* rowstat;                   // mode 0: (mu, rstd) per slot
    const uint4* axrow;                      // mode 0: the slot's row of the LayerNorm K-step
    __half *q, *k, *vt, *g;                  // mode 0 outputs
    const float* bo;                         // mode 1
    const uint8_t* mask;                     // mode 1: [S, I] or NULL
    const __nv_bfloat16* resid;              // mode 1: Ms [S, I, 256] or NULL
    __nv_bfloat16* out;                      // mode 1: [S, I, 256]
    uint32_t* status;
};

// MODE 0: the MSA projection (A = Ms, bf16, through a 3-D map [S][I][256] whose
// residue extent zero-fills the padded slots; block x = 0 q, 1 k, 2 v, 3 gate;
// epilogue: rstd x accumulator, sigmoid for the gate, q / k / gate as
// [S][8][I_pad][32], v^T as [S][8][32][I_pad]).  MODE 1: the output projection
// (A = u, f16, [S * I_pad][256]; epilogue: MSA mask, residual, bf16 out [S][I][256]).
template <int MODE>
__global__ void __launch_bounds__(kg::kThreads, 1)
sm103_msa_gemm(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB, GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    if (status_set(p.status)) return;
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kg::kBar);
    uint64_t* b_full = bars + 0;
    uint64_t* a_full = bars + 1;      // [5]
    uint64_t* a_empty = bars + 6;     // [5]: the MMA's commit
    uint64_t* acc_full = bars + 11;   // [2]
    uint64_t* acc_empty = bars + 13;  // [2]: the 8 epilogue warps
    uint64_t* ax_empty = bars + 15;   // [2]: MODE 0, the MMA's commit after the tile
    uint64_t* mma_done = bars + 17;   // every MMA of this block retired (before the TMEM is freed)
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 18);
    volatile int* abort = reinterpret_cast<volatile int*>(bars + 19);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = blockIdx.x;               // MODE 0: 0 q, 1 k, 2 v, 3 gate
    const int tpl = p.I_pad / 128;            // tiles per MSA row
    if (threadIdx.x == 0) {
        mbar_init(b_full, 1);
        for (int q = 0; q < kg::kSlots; ++q) {
            mbar_init(a_full + q, 1);
            mbar_init(a_empty + q, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(acc_full + s, 1);
            mbar_init(acc_empty + s, kg::kEpiWarps);
            mbar_init(ax_empty + s, 1);
        }
        mbar_init(mma_done, 1);
        *abort = 0;
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < 4096 / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(sm + kg::kZero)[i] = make_uint4(0, 0, 0, 0);
    if (warp >= 4) {
        const int c = threadIdx.x - 128;      // column 0 .. 255 of this block: its bx row
        uint4 row;
        if (MODE == 0) {
            const int n = grp * 256 + c;
            const uint32_t cs = split_bf16(p.cst[n]), of = split_bf16(p.cst[NPROJ + n]);
            row = make_uint4((cs & 0xFFFFu) * 0x10001u, (cs >> 16) * 0x10001u, (of & 0xFFFFu) * 0x10001u,
                             (of >> 16) * 0x10001u);                 // (cs_h, cs_h, cs_l, cs_l, of_h, of_h, of_l, of_l)
        } else {
            row = make_uint4(split_f16(p.bo[c]), 0u, 0u, 0u);        // (bo_h, bo_l, 0, ...)
            if (c < 128) {                                           // ax of both buffers: (1, 1, 0, ...) in f16
                const uint4 one = make_uint4(0x3C003C00u, 0u, 0u, 0u);
                reinterpret_cast<uint4*>(sm + kg::kAX)[c] = one;
                reinterpret_cast<uint4*>(sm + kg::kAX + 2048)[c] = one;
            }
        }
        reinterpret_cast<uint4*>(sm + kg::kBX)[c] = row;
    }
    fence_proxy_async_smem();
    if (warp == 1) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    // Register split: launched at 168 per thread; the control warpgroup (warps 0-3)
    // drops to 80 and the two epilogue warpgroups grow to 208 (128 x 80 + 256 x 208
    // = 63488 <= 384 x 168), room for a whole 128-column row of the accumulator.
    if (warp < 4) setmaxnreg_dec<80>();
    if (warp == 0) {
        // ------------------------------------------------------------ producer: TMA of A and B, the ax tiles
        int issued = 0;                       // A chunks issued (chunk c of the block goes to slot c % 5)
        bool ok = true;
        if (lane == 0) {
            prefetch_tmap(&mapA);
            prefetch_tmap(&mapB);
            mbar_arrive_expect_tx(b_full, 131072);
            for (int kc = 0; kc < 4; ++kc) tma_load_2d(sm + kg::kB + kc * 32768, &mapB, b_full, kc * 64, grp * 256);
        }
        int j = 0;
        for (int t = blockIdx.y; ok && t < p.n_tiles; t += gridDim.y, ++j) {
            const int s = t / tpl, i0 = (t % tpl) * 128;
            // ax of this tile (MODE 0: buffer j & 1, free once the MMAs of tile j - 2
            // retired) rides on the barrier of the tile's first A chunk
            if (MODE == 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(ax_empty + (j & 1), ((j >> 1) & 1) ^ 1, abort));
                if (!ok) break;
            }
            for (int kc = 0; kc < 4; ++kc) {
                const int q = issued % kg::kSlots, n = issued / kg::kSlots;
                ok = __all_sync(0xffffffffu, mbar_wait(a_empty + q, (n & 1) ^ 1, abort));
                if (!ok) break;
                if (lane == 0) {
                    uint8_t* dst = sm + kg::kA + q * 16384;
                    const bool with_ax = MODE == 0 && kc == 0;
                    mbar_arrive_expect_tx(a_full + q, 16384 + (with_ax ? 2048 : 0));
                    if (with_ax) bulk_load(sm + kg::kAX + (j & 1) * 2048, p.axrow + (size_t)t * 128, 2048, a_full + q);
                    if (MODE == 0)
                        tma_load_3d(dst, &mapA, a_full + q, kc * 64, i0, s);
                    else
                        tma_load_2d(dst, &mapA, a_full + q, kc * 64, t * 128);
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
                // the last copy into each A slot lands before the block ends
                for (int q = 0; q < kg::kSlots; ++q) {
                    const int cl = issued - 1 - ((issued - 1 - q) % kg::kSlots + kg::kSlots) % kg::kSlots;
                    if (cl >= 0) mbar_wait(a_full + q, (cl / kg::kSlots) & 1, &keep_waiting);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = MODE == 0 ? idesc_bf16_f32(128, 256) : idesc_f16_f32(128, 256);
            bool ok = mbar_wait(b_full, 0, abort);
            const uint32_t bbase = smem_u32(sm + kg::kB);
            const uint32_t zero = smem_u32(sm + kg::kZero), bx = smem_u32(sm + kg::kBX);
            const uint64_t bxd = sdesc_noswizzle(bx, zero - bx, 128);
            int used = 0, j = 0;
            for (int t = blockIdx.y; ok && t < p.n_tiles; t += gridDim.y, ++j) {
                const int ab = j & 1;
                if (!mbar_wait(acc_empty + ab, ((j >> 1) & 1) ^ 1, abort)) {
                    ok = false;
                    break;
                }
                for (int kc = 0; kc < 4; ++kc, ++used) {
                    const int q = used % kg::kSlots, n = used / kg::kSlots;
                    if (!mbar_wait(a_full + q, n & 1, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (kc == 0) {                                  // the per-column terms
                        const uint32_t ax = smem_u32(sm + kg::kAX + (MODE == 0 ? (j & 1) * 2048 : 0));
                        mma_ss(tmem + ab * 256, sdesc_noswizzle(ax, zero - ax, 128), bxd, idesc, 0u);
                    }
                    const uint32_t abase = smem_u32(sm + kg::kA + q * 16384);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = sdesc(abase + kk * 32, 1024, kSwizzle128);
                        const uint64_t bd = sdesc(bbase + kc * 32768 + kk * 32, 1024, kSwizzle128);
                        mma_ss(tmem + ab * 256, ad, bd, idesc, 1u);
                    }
                    tc_commit(a_empty + q);
                }
                if (!ok) break;
                if (MODE == 0) tc_commit(ax_empty + (j & 1));
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
        // The 128 columns come out of TMEM in two x64 loads and one wait per tile
        // (a TMEM load waits about as long as the tensor core keeps TMEM busy, so
        // one wait per tile instead of one per 32 columns).
        const int wq = warp & 3, half = (warp - 4) >> 2;
        const int r = wq * 32 + lane;
        const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16) + half * 128;
        // this slot's operand of a tile, loaded one tile ahead and first used a tile
        // later (a value, not a test of it, so that nothing waits on the load here)
        float rstd = 1.f;
        uint32_t mbyte = 0;
        auto fetch = [&](int t) {
            if (t >= p.n_tiles) return;
            if (MODE == 0) {
                rstd = p.rowstat[(size_t)t * 128 + r].y;
            } else {
                const int s = t / tpl, i = (t % tpl) * 128 + r;
                mbyte = i >= p.I ? 0u : p.mask == nullptr ? 1u : static_cast<uint32_t>(p.mask[(size_t)s * p.I + i]);
            }
        };
        fetch(blockIdx.y);
        int j = 0;
        bool ok = true;
        for (int t = blockIdx.y; t < p.n_tiles; t += gridDim.y, ++j) {
            const int ab = j & 1;
            const int s = t / tpl, i = (t % tpl) * 128 + r;
            const float cur_rstd = rstd;
            const uint32_t cur_mbyte = mbyte;
            if (!mbar_wait(acc_full + ab, (j >> 1) & 1, abort)) { ok = false; break; }
            tc_fence_after();
            uint32_t acc[2][64];
            tmem_ld64(tl + ab * 256, acc[0]);
            tmem_ld64(tl + ab * 256 + 64, acc[1]);
            tmem_ld_wait();
            tmem_regs_ready(acc[0]);
            tmem_regs_ready(acc[1]);
            tc_fence_before();                                   // the accumulator is in registers
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty + ab);
            fetch(t + gridDim.y);
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) {
                const uint32_t* a = &acc[hh >> 1][(hh & 1) * 32];
                if (MODE == 0) {
                    uint32_t o[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float v0 = cur_rstd * __uint_as_float(a[e]), v1 = cur_rstd * __uint_as_float(a[e + 1]);
                        o[e >> 1] = grp == 3 ? sigmoid_f16x2(v0, v1) : pack_f16(v0, v1);
                    }
                    const size_t lh = (size_t)s * HM + half * 4 + hh;
                    if (grp == 2) {                              // v^T: [S][8][32][I_pad]
                        unsigned short* dst = reinterpret_cast<unsigned short*>(p.vt + lh * HD * p.I_pad + i);
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            dst[(size_t)e * p.I_pad] = static_cast<unsigned short>(o[e >> 1] & 0xFFFFu);
                            dst[(size_t)(e + 1) * p.I_pad] = static_cast<unsigned short>(o[e >> 1] >> 16);
                        }
                    } else {                                     // q, k, gate: [S][8][I_pad][32]
                        __half* base = grp == 0 ? p.q : grp == 1 ? p.k : p.g;
                        uint4* dst = reinterpret_cast<uint4*>(base + (lh * p.I_pad + i) * HD);
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4)
                            dst[c4] = make_uint4(o[4 * c4], o[4 * c4 + 1], o[4 * c4 + 2], o[4 * c4 + 3]);
                    }
                } else if (i < p.I) {
                    const size_t pos = (size_t)s * p.I + i;
                    const int c0 = half * 128 + hh * 32;
                    uint32_t zr[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) zr[c] = 0u;
                    if (p.resid != nullptr) {
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
                    const bool cur_valid = cur_mbyte != 0;
                    uint32_t o[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float a0 = (cur_valid ? __uint_as_float(a[e]) : 0.f) + bf16lo(zr[e >> 1]);
                        const float a1 = (cur_valid ? __uint_as_float(a[e + 1]) : 0.f) + bf16hi(zr[e >> 1]);
                        o[e >> 1] = pack_bf16(a0, a1);
                    }
                    uint4* dst = reinterpret_cast<uint4*>(p.out + pos * CM + c0);
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
                   reinterpret_cast<__nv_bfloat16*>(ws + W.wprep), f32(W.cst), hf(W.wo_t), f32(W.bo)};
    {
        MsaFrontArgs fa{pa,
                        static_cast<const __nv_bfloat16*>(a.M),
                        static_cast<const __nv_bfloat16*>(a.Z),
                        S,
                        I,
                        Ip,
                        (int)(((long long)S * Ip + kStatSlotsPerBlock - 1) / kStatSlotsPerBlock),
                        Ip / kb::kPairs,
                        a.eps,
                        reinterpret_cast<float2*>(ws + W.rowstat),
                        reinterpret_cast<uint4*>(ws + W.axrow),
                        hf(W.bias)};
        const long long blocks = (long long)kPrepBlocks + fa.n_stat + (long long)fa.n_bias_x * Ip;
        if (tm) tm->begin("sm103_msa_front", s);
        sm103_msa_front<<<(unsigned)blocks, 256, 0, s>>>(fa);
        if (tm) tm->end(s);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }

    const int n_tiles = S * (Ip / 128);
    const int nsm = num_sms_of_device();

    // ---- projection GEMM: q | k | v^T | gate
    {
        CUtensorMap mA, mB;
        if (!sm103_map3d_bf16(&mA, a.M, CM, I, S, (uint64_t)CM * 2, (uint64_t)I * CM * 2, 64, 128, 1, 128) ||
            !sm103_map2d(&mB, ws + W.wprep, CM, NPROJ, CM * 2, 64, 256, 128, true))
            return cudaErrorInvalidValue;
        GemmParams gp{};
        gp.S = S;
        gp.I = I;
        gp.I_pad = Ip;
        gp.n_tiles = n_tiles;
        gp.cst = f32(W.cst);
        gp.rowstat = reinterpret_cast<const float2*>(ws + W.rowstat);
        gp.axrow = reinterpret_cast<const uint4*>(ws + W.axrow);
        gp.q = hf(W.q);
        gp.k = hf(W.k);
        gp.vt = hf(W.v);
        gp.g = hf(W.g);
        gp.status = a.status;
        const int rows = nsm / (NPROJ / 256) > 0 ? nsm / (NPROJ / 256) : 1;
        dim3 grid(NPROJ / 256, rows < n_tiles ? rows : n_tiles);
        if (tm) tm->begin("sm103_msa_proj", s);
        sm103_msa_gemm<0><<<grid, kg::kThreads, kg::kSmem, s>>>(mA, mB, gp);
        if (tm) tm->end(s);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }

    // ---- attention (one launch per key chunk), gated u to global memory
    {
        MsaAttnArgs m{S, I, Ip, a.key_chunks, hf(W.q), hf(W.k), hf(W.v), hf(W.g), hf(W.bias), hf(W.u),
                      W.o_run ? f32(W.o_run) : nullptr, W.lse_run ? f32(W.lse_run) : nullptr, a.msa_mask,
                      reinterpret_cast<uint64_t*>(ws + W.kbits), a.status, reinterpret_cast<int*>(ws + W.work)};
        if ((e = sm103_msa_attention(m, s, tm)) != cudaSuccess) return e;
    }

    // ---- output projection: out = u W_o + b_o (MSA mask, residual)
    {
        CUtensorMap mA, mB;
        if (!sm103_map2d(&mA, ws + W.u, CH, (uint64_t)S * Ip, CH * 2, 64, 128, 128, false) ||
            !sm103_map2d(&mB, ws + W.wo_t, CH, CM, CH * 2, 64, 256, 128, false))
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
        dim3 grid(1, nsm < n_tiles ? nsm : n_tiles);
        if (tm) tm->begin("sm103_msa_out", s);
        sm103_msa_gemm<1><<<grid, kg::kThreads, kg::kSmem, s>>>(mA, mB, gp);
        if (tm) tm->end(s);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace tri_attn
