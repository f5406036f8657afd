/*
 * tri_attn.h -- C ABI of the B300 gated triangle self-attention library.
 *
 * The operation (pair-biased, gated triangle self-attention over a pair
 * representation Z[I, I, c_z]):
 *
 *   zh      = LayerNorm(Z)                         per pair vector, biased variance
 *   q, k, v = zh W_q, zh W_k, zh W_v               H heads x d channels, no bias
 *   g       = sigmoid(zh W_g + b_g)                H*d channels
 *   b[h]    = zh W_b[:, h]                         one pair bias per head
 *   starting node, row i, head h, query (i, j), keys (i, k) with mask[k] = 1:
 *     o[i,j,h] = sum_k softmax_k( q[i,j,h].k[i,k,h] / sqrt(d) + b[h,j,k] ) v[i,k,h]
 *   ending node, column j, head h, query (i, j), keys (k, j) with mask[k] = 1:
 *     o[i,j,h] = sum_k softmax_k( q[i,j,h].k[k,j,h] / sqrt(d) + b[h,k,i] ) v[k,j,h]
 *   out[i,j] = (g[i,j] * concat_h o[i,j,h]) W_o + b_o,   and 0 where mask[i]*mask[j] = 0.
 *
 * Sources.  None of the pages prints these formulas; they name the parts:
 *   - "戴尔PowerEdgeXE8545 强劲算力助力蛋白质模型分析" (Dell), Evoformer paragraph:
 *     the Evoformer processes the residue-pair graph with triangle attention.
 *   - "通量提升达 23.11 倍！至强可扩展平台助力 AlphaFold2 端到端优化" (Intel),
 *     step 2 (triangle-geometry constraints learnt by self-attention over the
 *     pair representation) and step 4 (the attention module carries a large
 *     bias term formed by tensor contractions; fusing the score contraction
 *     with the bias add).
 *   - "Efficient protein structure prediction ... with OpenFold-TRT",
 *     Methodology: a bf16 Evoformer core and fused kernels.
 *   - "Resumo Técnico: Design-CP", Methodology 1: scores formed on the fly
 *     from key/value pieces, never materialising the full score matrix, and
 *     self-attention recast as cross-attention over key shards (the key-chunk
 *     schedule selected by tri_attn_config.key_chunks).
 * Readings where the pages are silent: LayerNorm eps from the config (1e-5
 * by default), biased variance; no bias on the q/k/v/pair-bias projections;
 * the 1/sqrt(d) scale applies to q.k only; masked keys get -inf; pairs that
 * touch a padded token are written as exactly 0 (a fully masked row is 0,
 * never NaN); the caller adds any residual.
 *
 * Conventions for every entry point
 *   - Tensors are caller-owned DEVICE memory unless stated otherwise; the
 *     library never frees them and keeps no pointer after a call returns.
 *   - Weights are stored [in, out] row-major (x W); head h owns channels
 *     h*d .. h*d+d-1 of q, k, v, g and of the rows of W_o.
 *   - "dtype" tensors are float32 when config.dtype is TRI_ATTN_F32 or
 *     TRI_ATTN_TF32 and bf16 (raw 16-bit patterns) when it is TRI_ATTN_BF16.
 *   - Calls validate their arguments on the host first; a validation error
 *     is returned synchronously and nothing is launched.
 *   - tri_attn_forward is asynchronous on the given stream (a cudaStream_t
 *     passed as void*, NULL = legacy default stream).  Errors raised on the
 *     device (a bounded wait that gave up) are latched in a device status
 *     word that tri_attn_status_sync reads.
 *   - A context may be used by one host thread at a time.
 */
#ifndef TRI_ATTN_H
#define TRI_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TRI_ATTN_OK = 0,
    TRI_ATTN_EINVAL = 1,        /* NULL / out-of-range / misaligned / aliasing argument  */
    TRI_ATTN_EUNSUPPORTED = 2,  /* shape or dtype the library has no kernel for          */
    TRI_ATTN_ENOMEM = 3,        /* workspace too small, or host allocation failed        */
    TRI_ATTN_ECUDA = 4,         /* a CUDA runtime call or kernel launch failed           */
    TRI_ATTN_ETIMEOUT = 5,      /* a device-side bounded wait gave up (status word set)  */
    TRI_ATTN_ERANGE = 6         /* an f16 intermediate of the sm103 path (q, k, v or the */
                                /* pair bias) left the f16 range: the output is invalid  */
} tri_attn_status;

typedef enum { TRI_ATTN_STARTING = 0, TRI_ATTN_ENDING = 1 } tri_attn_node;
/* Storage type of Z, the projection weights and out, and the arithmetic it selects:
 *   F32   fp32 storage and fp32 arithmetic (CUDA-core kernels; the 1e-4 bound)
 *   BF16  bf16 storage; tensor cores with f16/bf16 operands, fp32 accumulation
 *   TF32  fp32 storage; tensor cores reading the LayerNorm/projection operands as
 *         tf32 (10-bit significand), f16 attention operands, fp32 accumulation and
 *         fp32 output: the ExtraMSA-style mode (OpenFold-TRT summary, Methodology:
 *         TF32 for ExtraMSA).  Shapes the TF32 kernels do not cover run the fp32
 *         CUDA-core kernels, which are at least as accurate. */
typedef enum { TRI_ATTN_F32 = 0, TRI_ATTN_BF16 = 1, TRI_ATTN_TF32 = 2 } tri_attn_dtype;

/* Kernel path a context runs (tri_attn_path). */
typedef enum {
    TRI_ATTN_PATH_SIMT = 0,     /* fp32 CUDA-core kernels: any supported shape, f32 or bf16 storage */
    TRI_ATTN_PATH_SM103 = 1,    /* tcgen05/TMEM/TMA kernels: bf16, c_z = 128, H = 4, d = 32           */
    TRI_ATTN_PATH_SM103_TF32 = 2 /* the same with dtype TF32: fp32 storage, c_z = 128, H = 4, d = 32  */
} tri_attn_path_kind;

typedef struct {
    int   c_z;          /* pair channels; 1..256                                         */
    int   heads;        /* H; 1..16                                                      */
    int   head_dim;     /* d; 1..64, H*d <= 256                                          */
    int   I_max;        /* largest token count forward will accept; 1..16384             */
    int   dtype;        /* tri_attn_dtype of Z, the projection weights and out           */
    float ln_eps;       /* LayerNorm epsilon (> 0; 1e-5 is the usual value)              */
    int   key_chunks;   /* 1 = one pass over the keys; n > 1 = keys processed in n       */
                        /* sequential chunks merged by log-sum-exp (Design-CP,           */
                        /* Methodology 1, on one GPU).  Chunk boundaries are multiples   */
                        /* of 8 tokens: size = round_up(ceil(I / n), 8).  1..64.         */
    int   force_simt;   /* nonzero: use the SIMT path even where the sm103 path applies  */
} tri_attn_config;

/* Device pointers to the module parameters.  Sizes with C = heads*head_dim. */
typedef struct {
    const float* ln_gamma;  /* [c_z] fp32                    */
    const float* ln_beta;   /* [c_z] fp32                    */
    const void*  w_q;       /* [c_z, C] dtype                */
    const void*  w_k;       /* [c_z, C] dtype                */
    const void*  w_v;       /* [c_z, C] dtype                */
    const void*  w_g;       /* [c_z, C] dtype                */
    const void*  w_b;       /* [c_z, H] dtype                */
    const float* b_g;       /* [C] fp32                      */
    const void*  w_o;       /* [C, c_z] dtype                */
    const float* b_o;       /* [c_z] fp32, or NULL for zero  */
} tri_attn_weights;

typedef struct tri_attn_ctx tri_attn_ctx;

/* Create a context for one configuration on the current CUDA device.
 * Owns host state and one small device allocation (the status word).
 * Returns EINVAL for a NULL argument or out-of-range field, EUNSUPPORTED when
 * no kernel covers the shape, ECUDA when the device is not usable.  On error
 * *out is set to NULL. */
tri_attn_status tri_attn_create(const tri_attn_config* cfg, tri_attn_ctx** out);

/* Release a context (NULL is a no-op).  Call after the stream work that
 * uses it has completed. */
void tri_attn_destroy(tri_attn_ctx* ctx);

/* Path the context runs (tri_attn_path_kind), or -1 for a NULL context. */
int tri_attn_path(const tri_attn_ctx* ctx);

/* Bytes of device workspace tri_attn_forward needs for I tokens (0 for an
 * invalid I or a NULL context).  The caller allocates it, 256-byte aligned,
 * and must not touch it while a forward that uses it is in flight. */
size_t tri_attn_workspace_bytes(const tri_attn_ctx* ctx, int I);

/* One forward pass.
 *   node        TRI_ATTN_STARTING or TRI_ATTN_ENDING
 *   I           tokens, 1 <= I <= cfg.I_max
 *   Z           [I, I, c_z] dtype, row-major, 16-byte aligned
 *   token_mask  [I] uint8 (nonzero = valid token), or NULL for all valid
 *   w           module parameters (struct itself is host memory)
 *   workspace   >= tri_attn_workspace_bytes(ctx, I) bytes, 256-byte aligned; must
 *               not overlap Z, token_mask or out
 *   out         [I, I, c_z] dtype, 16-byte aligned, must not overlap Z, token_mask
 *               or the workspace
 *   stream      cudaStream_t as void*
 * Writes out (the update only).  Asynchronous; returns EINVAL / EUNSUPPORTED
 * / ENOMEM from validation without launching, ECUDA if a launch fails. */
tri_attn_status tri_attn_forward(tri_attn_ctx* ctx, int node, int I,
                                 const void* Z, const uint8_t* token_mask,
                                 const tri_attn_weights* w,
                                 void* workspace, size_t workspace_bytes,
                                 void* out, void* stream);

/* Options of tri_attn_forward_ex (a host struct; NULL means all defaults).
 *   pair_mask  [I, I] uint8 device array over the pairs (i, j) of Z, row-major,
 *              nonzero = valid pair, or NULL (all valid).  Starting node: line i
 *              attends only keys (i, k) with pair_mask[i, k] != 0; ending node:
 *              line j attends only keys (k, j) with pair_mask[k, j] != 0; in both
 *              the output of a pair with pair_mask[i, j] == 0 is 0.  It acts on
 *              top of token_mask.  (The sources name masking but print no formula;
 *              this follows the token-mask reading pair by pair.)
 *   residual   nonzero: write Z + update (rounded once to the dtype) instead of the
 *              update; out may then be Z itself (in-place update Z += update). */
typedef struct {
    const uint8_t* pair_mask;
    int residual;
} tri_attn_options;

/* tri_attn_forward with options.  Arguments as for tri_attn_forward, except that
 * with opt->residual set `out` may equal Z (a partial overlap is still EINVAL).
 * tri_attn_forward(...) is tri_attn_forward_ex(..., opt = NULL, ...). */
tri_attn_status tri_attn_forward_ex(tri_attn_ctx* ctx, int node, int I,
                                    const void* Z, const uint8_t* token_mask,
                                    const tri_attn_options* opt,
                                    const tri_attn_weights* w,
                                    void* workspace, size_t workspace_bytes,
                                    void* out, void* stream);

/* MSA row-wise gated self-attention with pair bias: the same attention with
 * another batch and bias source.  For an MSA representation Ms[S, I, c_m], a
 * pair representation Z[I, I, c_z] and a mask mm[S, I]:
 *
 *   mh      = LayerNorm_m(Ms);  q, k, v = mh W_q, mh W_k, mh W_v;  g = sigmoid(mh W_g + b_g)
 *   b[h]    = LayerNorm_z(Z) W_b[:, h]                   shared by all S rows
 *   row s, head h, query (s, i), keys (s, j) with mm[s, j] != 0:
 *     o[s,i,h] = sum_j softmax_j( q[s,i,h].k[s,j,h] / sqrt(d) + b[h,i,j] ) v[s,j,h]
 *   out[s,i] = (g[s,i] * concat_h o[s,i,h]) W_o + b_o,  0 where mm[s, i] == 0
 *              (with residual: Ms + that, rounded once to the dtype).
 *
 * Source: "通量提升达 23.11 倍！至强可扩展平台助力 AlphaFold2 端到端优化" (Intel),
 * step 4: the Evoformer's attention call takes the query rows, a per-row
 * (batched) mask bias and a bias shared by all rows (non-batched, from the pair
 * representation).  Readings: the MSA and Z have LayerNorms of their own (the
 * context's ln_eps for both); the MSA mask excludes keys and zeroes outputs as
 * the pair mask of tri_attn_forward_ex does.
 *
 * The context supplies c_z (pair channels), heads, head_dim, dtype, ln_eps and
 * key_chunks.  Two paths (tri_attn_msa_path):
 *   sm103  bf16, c_m = 256, c_z = 128, 8 heads of 32 (the Evoformer's MSA row
 *          attention), on an sm_103 device without force_simt: the MSA and pair
 *          projections on tcgen05 tensor cores with f16 intermediates (q, k, v,
 *          gate, pair bias, gated output u) and fp32 accumulation; the attention
 *          kernel of tri_attn_forward; ERANGE as there.
 *   SIMT   any other supported shape (head_dim 8, 16, 32 or 64): CUDA-core
 *          kernels, fp32 arithmetic on dtype storage. */
typedef struct {
    const float* ln_m_gamma;  /* [c_m] fp32                   */
    const float* ln_m_beta;   /* [c_m] fp32                   */
    const void*  w_q;         /* [c_m, C] dtype               */
    const void*  w_k;         /* [c_m, C] dtype               */
    const void*  w_v;         /* [c_m, C] dtype               */
    const void*  w_g;         /* [c_m, C] dtype               */
    const float* b_g;         /* [C] fp32                     */
    const void*  w_o;         /* [C, c_m] dtype               */
    const float* b_o;         /* [c_m] fp32, or NULL for zero */
    const float* ln_z_gamma;  /* [c_z] fp32                   */
    const float* ln_z_beta;   /* [c_z] fp32                   */
    const void*  w_b;         /* [c_z, H] dtype               */
} tri_attn_msa_weights;

/* Path (tri_attn_path_kind) tri_attn_msa_forward takes on this context for
 * c_m MSA channels, or -1 for a NULL context. */
int tri_attn_msa_path(const tri_attn_ctx* ctx, int c_m);

/* Bytes of device workspace tri_attn_msa_forward needs for S rows of I
 * residues, whichever path it takes (0 for a NULL context, S outside 1..16384
 * or I outside 1..I_max).  Same ownership rules as tri_attn_workspace_bytes. */
size_t tri_attn_msa_workspace_bytes(const tri_attn_ctx* ctx, int S, int I);

/*   S           MSA rows, 1 <= S <= 16384
 *   I           residues, 1 <= I <= cfg.I_max
 *   c_m         MSA channels, 1 <= c_m <= 256
 *   msa         Ms [S, I, c_m] dtype, row-major, 16-byte aligned
 *   msa_mask    [S, I] uint8 (nonzero = valid), or NULL for all valid
 *   Z           [I, I, cfg.c_z] dtype, row-major, 16-byte aligned
 *   w           parameters (struct itself is host memory; device pointers)
 *   residual    nonzero: write Ms + update; out may then be msa itself
 *   workspace   >= tri_attn_msa_workspace_bytes(ctx, S, I) bytes, 256-byte aligned;
 *               must not overlap msa, msa_mask, Z or out
 *   out         [S, I, c_m] dtype, 16-byte aligned; must not overlap Z, the
 *               workspace or msa_mask, nor msa unless it is msa itself with residual
 *               (msa_mask must not lie in the workspace either)
 * Asynchronous; EINVAL / EUNSUPPORTED / ENOMEM from validation without
 * launching, ECUDA if a launch fails. */
tri_attn_status tri_attn_msa_forward(tri_attn_ctx* ctx, int S, int I, int c_m,
                                     const void* msa, const uint8_t* msa_mask, const void* Z,
                                     const tri_attn_msa_weights* w, int residual,
                                     void* workspace, size_t workspace_bytes,
                                     void* out, void* stream);

/* Synchronise `stream`, then read and clear the context's device status word.
 * Returns ETIMEOUT if a kernel gave up a bounded wait since the last call,
 * else ERANGE if a forward on the sm103 path met a non-finite value (one of its
 * f16 intermediates q, k, v or pair bias exceeded 65504 in magnitude, e.g. from
 * LayerNorm weights far beyond a trained model's scale), ECUDA if the stream
 * reports an error, else OK. */
tri_attn_status tri_attn_status_sync(tri_attn_ctx* ctx, void* stream);

/* Per-kernel timing.  tri_attn_set_timing(ctx, 1) clears the record list and
 * turns recording on: every later forward records a CUDA event pair around
 * each of its kernel launches, on the launching stream (at most 8192 records;
 * later launches are not recorded).  tri_attn_kernel_times waits for the
 * recorded events and writes up to `cap` entries: names[k] (static strings)
 * and ms[k]; it returns the number of records, or -1 if timing is off.
 * tri_attn_set_timing(ctx, 0) turns recording off and clears the list. */
tri_attn_status tri_attn_set_timing(tri_attn_ctx* ctx, int on);
int tri_attn_kernel_times(tri_attn_ctx* ctx, const char** names, float* ms, int cap);

/* Allocation-free forward, for callers that cannot allocate device memory.
 *
 * Some callers have their input and output buffers but may not call
 * cudaMalloc: code running inside a host callback or a custom allocator, a
 * plugin whose host runtime owns every device allocation, or a process whose
 * device memory is fully reserved up front.  They can use neither the
 * caller-allocated workspace of tri_attn_forward nor tri_attn_create (which
 * allocates the status word).  This entry point needs neither: its workspace
 * is a file-scope device array of the library (34.3 MB: the sm103 workspace
 * at I = 128 plus a status word), which every GPU that loads the library
 * holds until the process exits.  The paper has no counterpart of it.
 *
 *   shape       bf16 Z / weights / out, c_z = 128, H = 4, d = 32, one key chunk
 *               (the sm103 kernels; sm_103 devices only, else EUNSUPPORTED)
 *   I           1 <= I <= 128; larger I returns TRI_ATTN_EUNSUPPORTED
 *   ln_eps      LayerNorm epsilon, 0 < ln_eps <= 1
 *   other args  as for tri_attn_forward (device pointers, 16-byte aligned);
 *               out must not overlap Z or token_mask, and none of Z, token_mask
 *               and out may lie in the library's array (EINVAL, nothing launched)
 * It calls no cudaMalloc, cudaFree or other allocating routine.  The array's
 * device address belongs to the CUDA context current at the call: the first
 * call in each context (per device, and again after cudaDeviceReset re-creates
 * the primary context) looks it up with cudaGetSymbolAddress and caches it
 * under the context's id, so make that first call before any stream capture.
 * Every call shares the one array and leaves its contents behind; the status
 * word inside it is cleared (on the stream) at the start of each call, and the
 * attention kernel's work-item counter before each of its launches.  Calls
 * whose work overlaps on the GPU race on the array: issue them on one stream,
 * or otherwise order them. */
tri_attn_status tri_attn_forward_static(int node, int I, const void* Z, const uint8_t* token_mask,
                                        const tri_attn_weights* w, float ln_eps, void* out, void* stream);

/* Status of the last tri_attn_forward_static on the current device, without
 * allocating: synchronises `stream`, reads the status word in the library's
 * array and clears it.  Returns ETIMEOUT if a device-side bounded wait of that
 * call gave up (its `out` is then incomplete), else ERANGE if an f16
 * intermediate left the f16 range (as for tri_attn_status_sync), ECUDA if the
 * stream or the copy reports an error, else OK.  Call it before the next
 * static call (which clears the word). */
tri_attn_status tri_attn_static_status(void* stream);

/* Test hook for the failure path (no GPU fault is involved).
 * fault = TRI_ATTN_FAULT_SKIP_STAGE: the next tri_attn_forward of this context
 * runs its attention kernel with the producer of the CTA that takes the first
 * work item skipping one K/V stage load, so that CTA's bounded waits run out
 * (about 2 s), it records the timeout in the status word and exits (the other
 * CTAs take the remaining work items and finish; a later launch that finds the
 * status set exits at once); tri_attn_status_sync then returns
 * TRI_ATTN_ETIMEOUT and clears the word, after which the context is fully
 * usable.  The hook applies to one forward; fault = 0 clears it.
 * EUNSUPPORTED on the SIMT path. */
enum { TRI_ATTN_FAULT_NONE = 0, TRI_ATTN_FAULT_SKIP_STAGE = 1 };
tri_attn_status tri_attn_debug_inject(tri_attn_ctx* ctx, int fault);

/* The same test hook for tri_attn_forward_static: the next static call (in this
 * process) runs with the first work item's producer skipping one stage load;
 * tri_attn_static_status then returns TRI_ATTN_ETIMEOUT.  fault = 0 clears it. */
tri_attn_status tri_attn_static_debug_inject(int fault);

/* Static description of a status code. */
const char* tri_attn_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* TRI_ATTN_H */
