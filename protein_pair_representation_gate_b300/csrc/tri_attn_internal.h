// Internal declarations shared by the C-ABI layer and the kernel files.
//
// Line-major convention used by every kernel after the projection step:
// a "line" L is the row i (starting node) or the column j (ending node) that
// one attention problem runs along, and a "position" x indexes the pairs on
// that line.  The pair that feeds (L, x) is Z[L, x] for the starting node and
// Z[x, L] for the ending node.  With the projections written in this
// orientation, and the pair bias written transposed for the ending node
// (bias'[h, a, b] = b[h, b, a]), the attention kernels are node-agnostic and
// only the read of Z and the write of out depend on the node.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/tri_attn.h"

namespace tri_attn {

constexpr int kTile = 128;          // token padding granule (one MMA tile of keys or queries)

constexpr int round_up(int a, int b) { return (a + b - 1) / b * b; }
constexpr size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

// Device status word bits (set by bounded waits that gave up).
enum : uint32_t {
    kStatusTimeoutProducer = 1u << 0,
    kStatusTimeoutMma = 1u << 1,
    kStatusTimeoutSoftmax = 1u << 2,
    kStatusTimeoutEpilogue = 1u << 3,
    kStatusTimeoutMask = 0xFu,
    kStatusRange = 1u << 4,          // a non-finite value from an f16 intermediate out of range
};

// Byte offsets of the workspace regions for one (config, I).  Every region
// starts on a 256-byte boundary.  Element types: SIMT path fp32 everywhere;
// sm103 path bf16 for q/k/vT/g/bias and fp32 for the chunk state.
struct Workspace {
    int I = 0, I_pad = 0;
    size_t q = 0, k = 0, v = 0, g = 0, bias = 0, u = 0;   // projections
    size_t o_run = 0, lse_run = 0;                          // key-chunk state (0 bytes if unchunked)
    size_t wprep = 0, colsum = 0, betaw = 0, wb32 = 0, wo_t = 0, bo = 0;  // prepared weights (sm103)
    size_t cst = 0;                                          // per column pair {colsum x2, offset x2} (sm103)
    size_t kbits = 0;                                        // [I][I_pad / 64 + 1] key-valid bits per line (sm103)
    size_t rowstat = 0;                                      // (mu, rstd) per MSA slot (sm103 MSA path)
    size_t axrow = 0;                                        // 16 B per MSA slot: its LayerNorm K-step row
    size_t work = 0;                                         // work-item counter of the attention kernel
    size_t total = 0;
};

struct Ctx;  // defined in tri_attn_api.cu

// Arguments of one forward, already validated, in device pointers.
struct FwdArgs {
    int node, I, I_pad, c_z, H, d;
    float eps;
    const void* Z;
    const uint8_t* mask;     // may be NULL (all valid)
    tri_attn_weights w;
    char* ws;                // workspace base
    const Workspace* lay;
    void* out;
    int key_chunks;
    uint32_t* status;        // device status word
    int inject = 0;          // test hook (tri_attn_debug_inject)
    const uint8_t* pair_mask = nullptr;   // [I, I] over the pairs of Z, or NULL
    int residual = 0;        // write Z + update
};

// Records an event pair around a launch when timing is on.
struct LaunchTimer {
    virtual void begin(const char* name, cudaStream_t s) = 0;
    virtual void end(cudaStream_t s) = 0;
    virtual ~LaunchTimer() {}
};

// SIMT path (any dtype/shape within the config limits).
Workspace simt_layout(int I, int c_z, int H, int d, int key_chunks);
cudaError_t simt_forward(const FwdArgs& a, int dtype, cudaStream_t s, LaunchTimer* t);

// MSA row attention with pair bias (CUDA-core kernels).
struct MsaArgs {
    int S, I, I_pad, c_m, c_z, H, d, key_chunks, residual;
    float eps;
    const void* M;                 // [S, I, c_m]
    const uint8_t* msa_mask;       // [S, I] or NULL
    const void* Z;                 // [I, I, c_z]
    tri_attn_msa_weights w;
    char* ws;
    const Workspace* lay;
    void* out;                     // [S, I, c_m]
    uint32_t* status = nullptr;    // device status word (sm103 path)
};
constexpr int kMsaMaxRows = 16384;
Workspace simt_msa_layout(int S, int I, int H, int d, int key_chunks);
cudaError_t simt_msa_forward(const MsaArgs& a, int dtype, cudaStream_t s, LaunchTimer* t);

// sm103 path (bf16, c_z = 128, H = 4, d = 32).
bool sm103_supported(int c_z, int H, int d, int dtype);

// Workspace of the sm103 path (usable at compile time: the allocation-free entry
// point sizes its device array with it).  Tokens are padded to a multiple of 256.
constexpr Workspace sm103_layout(int I, int key_chunks) {
    Workspace w;
    w.I = I;
    w.I_pad = round_up(I, 256);
    const size_t P = (size_t)I * w.I_pad;
    size_t off = 0;
    auto take = [&off](size_t bytes) { size_t o = off; off = align256(off + bytes); return o; };
    w.wprep = take((size_t)512 * 128 * 2);   // (gamma . W)^T for q | v | k | g, bf16
    w.colsum = take(516 * 4);
    w.betaw = take(516 * 4);
    w.wb32 = take(128 * 4 * 4);
    w.wo_t = take((size_t)128 * 128 * 2);    // W_o^T, f16
    w.bo = take(128 * 4);
    w.cst = take(256 * 4 * 4);
    w.kbits = take((size_t)I * (w.I_pad / 64 + 1) * 8);
    w.work = take(256);
    w.q = take(P * 128 * 2);
    w.k = take(P * 128 * 2);
    w.v = take(P * 128 * 2);
    w.g = take(P * 128 * 2);
    w.bias = take((size_t)4 * w.I_pad * w.I_pad * 2);
    if (key_chunks > 1) {
        w.o_run = take(P * 128 * 4);
        w.lse_run = take(P * 4 * 4);
    }
    w.total = off;
    return w;
}
cudaError_t sm103_forward(const FwdArgs& a, cudaStream_t s, LaunchTimer* t);

// MSA row attention on the sm103 path: bf16, c_m = 256, c_z = 128, 8 heads of 32.
constexpr int kMsaCm = 256, kMsaHeads = 8;
bool sm103_msa_supported(int c_m, int c_z, int H, int d, int dtype);

// Workspace of the sm103 MSA path (tokens padded to a multiple of 256).
constexpr Workspace sm103_msa_layout(int S, int I, int key_chunks) {
    Workspace w;
    w.I = I;
    w.I_pad = round_up(I, 256);
    const size_t P = (size_t)S * w.I_pad;            // (MSA row, residue) slots
    size_t off = 0;
    auto take = [&off](size_t bytes) { size_t o = off; off = align256(off + bytes); return o; };
    w.wprep = take((size_t)1024 * 256 * 2);           // (gamma_m . W)^T for q | k | v | g, bf16
    w.cst = take((size_t)2 * 1024 * 4);               // column sums, then offsets, of the 1024 columns
    w.wo_t = take((size_t)256 * 256 * 2);             // W_o^T, f16
    w.bo = take(256 * 4);
    w.kbits = take((size_t)S * (w.I_pad / 64 + 1) * 8);
    w.work = take(256);
    w.rowstat = take(P * 8);
    w.axrow = take(P * 16);
    w.q = take(P * 256 * 2);
    w.k = take(P * 256 * 2);
    w.v = take(P * 256 * 2);
    w.g = take(P * 256 * 2);
    w.u = take(P * 256 * 2);
    w.bias = take((size_t)8 * w.I_pad * w.I_pad * 2);
    if (key_chunks > 1) {
        w.o_run = take(P * 256 * 4);
        w.lse_run = take(P * 8 * 4);
    }
    w.total = off;
    return w;
}
cudaError_t sm103_msa_forward(const MsaArgs& a, cudaStream_t s, LaunchTimer* t);

// The attention step of the sm103 triangle path (attention, gate, output
// projection; once per key chunk) over prepared f16 intermediates in the
// layouts the projection writes: q, k, g [I * H][I_pad][d], v^T [I * H][d][I_pad],
// bias [H][I_pad][I_pad], W_o^T [c_z][H d].  Z (residual) and out are bf16, or
// fp32 with f32 set.
struct TriAttnLaunch {
    int node = 0, I = 0, I_pad = 0, key_chunks = 1, inject = 0;
    bool f32 = false;
    const uint8_t* mask = nullptr;
    const uint8_t* pair_mask = nullptr;
    const void* Z_resid = nullptr;     // residual source, or NULL
    void* out = nullptr;
    __half *q = nullptr, *k = nullptr, *vt = nullptr, *g = nullptr, *bias = nullptr, *wo_t = nullptr;
    float *bo = nullptr, *o_run = nullptr, *lse_run = nullptr;
    uint64_t* kbits = nullptr;         // [I][I_pad / 64 + 1] scratch (with a pair mask)
    int* work = nullptr;               // work-item counter (zeroed before each launch)
    uint32_t* status = nullptr;
};
cudaError_t sm103_triangle_attention(const TriAttnLaunch& l, cudaStream_t s, LaunchTimer* t);

// TF32 forward (fp32 Z, weights and out; c_z = 128, H = 4, d = 32): the LayerNorm
// and projection on kind::tf32 tensor cores, then the attention step above with
// f16 intermediates and fp32 out.
bool sm103_tf32_supported(int c_z, int H, int d, int dtype);
constexpr Workspace sm103_tf32_layout(int I, int key_chunks) {
    Workspace w;
    w.I = I;
    w.I_pad = round_up(I, 256);
    const size_t P = (size_t)I * w.I_pad;           // (line, position) slots
    size_t off = 0;
    auto take = [&off](size_t bytes) { size_t o = off; off = align256(off + bytes); return o; };
    w.wprep = take((size_t)512 * 128 * 4);          // (gamma . W)^T for q | k | v | g, tf32 values in fp32
    w.cst = take((size_t)2 * 512 * 4);              // column sums, then offsets
    w.wb32 = take((size_t)128 * 4 * 4 + 2 * 4 * 4); // gamma . W_b, its column sums, beta W_b
    w.wo_t = take((size_t)128 * 128 * 2);           // W_o^T, f16
    w.bo = take(128 * 4);
    w.kbits = take((size_t)I * (w.I_pad / 64 + 1) * 8);
    w.work = take(256);
    w.rowstat = take(P * 8);
    w.axrow = take(P * 32);                         // two planes of 16 B per slot
    w.q = take(P * 128 * 2);
    w.k = take(P * 128 * 2);
    w.v = take(P * 128 * 2);
    w.g = take(P * 128 * 2);
    w.bias = take((size_t)4 * w.I_pad * w.I_pad * 2);
    if (key_chunks > 1) {
        w.o_run = take(P * 128 * 4);
        w.lse_run = take(P * 4 * 4);
    }
    w.total = off;
    return w;
}
cudaError_t sm103_tf32_forward(const FwdArgs& a, cudaStream_t s, LaunchTimer* t);

// Pieces of the sm103 triangle kernels the MSA path shares.
struct MsaAttnArgs {
    int S, I, I_pad, key_chunks;
    __half *q, *k, *vt, *g, *bias, *u;
    float *o_run, *lse_run;
    const uint8_t* msa_mask;
    uint64_t* kbits;
    uint32_t* status;
    int* work;                 // work-item counter (zeroed before each launch)
};
cudaError_t sm103_msa_attention(const MsaAttnArgs& m, cudaStream_t s, LaunchTimer* t);
bool sm103_map2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t row_bytes, uint32_t box_cols,
                 uint32_t box_rows, int swizzle_bytes, bool bf16);
bool sm103_map3d_bf16(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                      uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2, int swizzle_bytes);
// fp32 tensor map of rank 1..3: dims and box innermost first, strides in bytes of
// dims 1.. (rank - 1 of them); swizzle 128 or none.
bool sm103_map_f32(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                   const uint32_t* box, int swizzle_bytes);

// Chunk bounds shared by both paths: size = round_up(ceil(I / n), 8).
inline int chunk_size(int I, int n) {
    if (n <= 1) return I;
    int s = (I + n - 1) / n;
    return round_up(s, 8);
}

}  // namespace tri_attn
