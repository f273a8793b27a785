/*
 * tq.h -- C ABI of the rotated-codebook quantization library (libtq.so).
 *
 * The method (TurboQuant-style weight and KV-cache quantization) as stated on
 * the page "How it works" (turboquant-mlx), sections
 *   "Quantizing a weight, with no data"   rotate, group + RMS scale, snap, pack
 *   "The ternary tier (1.58 bits)"        {-c, 0, +c}, 20 trits per 32-bit word
 *   "Running a quantized layer"           rotate the input, decode codes inline;
 *                                         the MoE kernel split by shape of work
 *   "The KV cache"                        same rotation + codebook, 8-bit K / 3-bit V
 *   "Configuration that converter and loader share"
 *                                         codebook size marks bit vs trit packing
 * and on the page "Running a 1T-Parameter Model on a Laptop" (the MoE router,
 * create_hadamard_matrix, the TurboQuant KV cache update_and_fetch).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument documented as "device" is a CUDA device pointer
 *    owned by the caller; the library allocates no memory and keeps no state.
 *    "host" pointers are ordinary CPU memory.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Device
 *    work is enqueued asynchronously on it; the call returns once enqueued.
 *  - Return value: TQ_OK, or an error found on the host before any launch
 *    (TQ_ERR_INVALID: bad argument; TQ_ERR_UNSUPPORTED: valid but not built)
 *    or a launch error (TQ_ERR_CUDA).  Nothing is launched when a host check
 *    fails.
 *  - Errors a kernel detects (an expert id out of range, a bounded wait that
 *    ran out, a codebook of the wrong shape) are OR-ed as TQ_DEVERR_* bits into
 *    the optional device word `err` (NULL: not reported).  The offending rows
 *    are written as zeros; no kernel traps.
 *  - Codes: a codebook of 3 entries means trit-packed (20 base-3 digits per
 *    uint32, digit j has weight 3^j); 2^b entries (b = 1,2,3,4,8) means
 *    bit-packed, 32/b codes per word (10 for b = 3, top two bits zero), code j
 *    of a word at bits [b*j, b*j+b).  Each row starts a fresh word; unused
 *    slots and padding words are zero.  Digit/code value i stands for the
 *    i-th centroid in ascending order.
 *  - Scales: IEEE fp16 bit patterns, one per group of `group` consecutive
 *    codes of a row, row-major [rows, cols/group].
 *  - Rotation: R = blockdiag(H_b, ..., H_b) . diag(signs) / sqrt(b), H_b the
 *    Sylvester Hadamard matrix of order b (a power of two dividing dim).
 *    Weights are stored rotated along the input dim (W_rot = W R^T), so
 *    W x = W_rot (R x).
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum tq_status {
    TQ_OK = 0,
    TQ_ERR_INVALID = 1,      /* argument rejected on the host */
    TQ_ERR_UNSUPPORTED = 2,  /* valid combination that the library does not cover */
    TQ_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
    TQ_ERR_TIMEOUT = 4,      /* a bounded device wait ran out (from tq_check_error) */
    TQ_ERR_DEVICE = 5        /* a kernel reported a bad input (from tq_check_error) */
} tq_status;

/* Bits of the device error word. */
#define TQ_DEVERR_BAD_ID 1u      /* an expert id outside [0, experts) */
#define TQ_DEVERR_TIMEOUT 2u     /* a bounded spin-wait gave up */
#define TQ_DEVERR_BAD_BOOK 4u    /* a ternary codebook that is not {c0, c0+d, c0+2d} */

typedef enum tq_dtype { TQ_F32 = 0, TQ_BF16 = 1, TQ_F16 = 2 } tq_dtype;

/* A codebook in device memory.  levels: 3, or 2^b with b in {1,2,3,4,8}.
 * centroids: device float[levels], ascending.  thresholds: device
 * float[levels-1], ascending; thresholds[i] separates centroids i and i+1
 * (the midpoints for a Lloyd-Max book). */
typedef struct tq_codebook_t {
    int32_t levels;
    const float* centroids;
    const float* thresholds;
} tq_codebook_t;

/* A rotation.  dim: length of the rotated vectors.  block: Hadamard order, a
 * power of two with 1 <= block <= 8192 dividing dim.  signs: device
 * int8[dim] holding +1 or -1. */
typedef struct tq_rotation_t {
    int32_t dim;
    int32_t block;
    const int8_t* signs;
} tq_rotation_t;

/* A bank of `experts` quantized matrices of shape [rows, cols], stored
 * rotated along cols.  Expert e, row n starts at codes + e*expert_stride_words
 * + n*row_stride_words and at scales + e*expert_stride_scales + n*(cols/group).
 * row_stride_words: >= tq_row_words(levels, cols) and a multiple of 4 (rows
 * start 16-byte aligned).  expert_stride_words: >= rows*row_stride_words,
 * multiple of 4.  expert_stride_scales >= rows*cols/group.  group: 16, 32, 64
 * or 128, dividing cols.  A dense (non-MoE) matrix is a bank with experts = 1. */
typedef struct tq_qweight_t {
    const uint32_t* codes;
    const uint16_t* scales;
    int32_t experts;
    int32_t rows;
    int32_t cols;
    int32_t group;
    int64_t row_stride_words;
    int64_t expert_stride_words;
    int64_t expert_stride_scales;
    tq_codebook_t cb;
} tq_qweight_t;

/* ------------------------------------------------------------------ host helpers */

/* Human-readable name of a status.  Never NULL. */
const char* tq_status_string(tq_status s);

/* Codes per 32-bit word for a codebook size ("The ternary tier": 3 entries =>
 * 20 trits; "Quantizing a weight", step Pack: 2^b entries => 32/b codes).
 * Returns 0 for an unsupported size. */
int32_t tq_codes_per_word(int32_t levels);

/* Words holding one row of `cols` codes (ceil(cols / codes_per_word)); 0 if invalid. */
int64_t tq_row_words(int32_t levels, int32_t cols);

/* tq_row_words rounded up to a multiple of 4 (the padded row stride). */
int64_t tq_row_stride_words(int32_t levels, int32_t cols);

/* Gaussian Lloyd-Max codebook, computed on the host in fp64.
 * "How it works", "Quantizing a weight, with no data", step "Snap to a
 * codebook": the error-minimising quantizer for a Gaussian, a fixed constant
 * per bit width; "The ternary tier": the three-level book {-c, 0, +c}.
 * levels: 2, 3, 4, 8, 16 or 256.  centroids: host double[levels];
 * thresholds: host double[levels-1] (midpoints).  Both ascending and exactly
 * symmetric about 0.  Returns TQ_ERR_INVALID for other sizes or NULL output. */
tq_status tq_codebook(int32_t levels, double* centroids, double* thresholds);

/* Rotation sign vector from a seed, on the host.
 * "How it works", "Configuration that converter and loader share": the
 * rotation's seed is recorded with the model; for a Hadamard layer the
 * rotation is a dim-length +-1 vector.  signs[i] = -1 if the top bit of the
 * i-th SplitMix64 output (Steele, Lea & Flood 2014) for `seed` is set, else +1.
 * signs: host int8[dim]. */
tq_status tq_rotation_signs(uint64_t seed, int32_t dim, int8_t* signs);

/* Dense rotation for a dimension the block Hadamard transform mixes too little.
 * Weight-reservoir page: such a layer's rotation is derived from its seed by a
 * QR decomposition of a random matrix (the QR fallback).  G[i][j] is the
 * (i*dim + j)-th standard normal draw of the seed's SplitMix64 stream through
 * the Box-Muller transform (draws 2p, 2p+1 from outputs 2p, 2p+1, u = (output
 * >> 11) / 2^53, r = sqrt(-2 ln(1 - u_2p)), cos / sin of 2 pi u_2p+1); G = QU
 * with U's diagonal positive, computed in fp64 by Householder reflections on the
 * host's threads; R = Q, written row-major to host double[dim * dim].  The layer
 * then stores W R^T and multiplies R x.  Cost: about 3 dim^3 flops on the host
 * (seconds at dim 2000).  dim: 1 .. 16384. */
tq_status tq_rotation_dense(uint64_t seed, int32_t dim, double* R);

/* ------------------------------------------------------------------ device entry points */

/* x_rot = R x for `rows` vectors.
 * "How it works", "Running a quantized layer": the layer rotates its input
 * (R orthonormal) instead of un-rotating the weights.
 * x: device [rows, rot->dim] of dtype xdt (f32, bf16 or f16).  x_rot: device
 * [rows, rot->dim] of dtype ydt (f32, bf16 or f16), may not alias x. */
tq_status tq_rotate(const tq_rotation_t* rot, const void* x, tq_dtype xdt, int64_t rows,
                    void* x_rot, tq_dtype ydt, void* stream);

/* y[r] = R x[r] for `rows` vectors with a dense rotation (the QR fallback above).
 * R: device f32 [dim, dim] row-major.  x: device [rows, dim] of xdt (f32, bf16 or
 * f16).  y: device f32 [rows, dim], may not alias x.  precise != 0 accumulates in
 * fp64 (for encoding: the rotated value then carries only its final fp32
 * rounding); 0 accumulates in fp32 (a decode input).  To encode such a layer,
 * rotate its rows with precise = 1 and pass them to tq_quantize with the
 * identity rotation (block 1, all signs +1). */
tq_status tq_rotate_dense(const float* R, int32_t dim, const void* x, tq_dtype xdt, int64_t rows, float* y,
                          int32_t precise, void* stream);

/* Fused encode of weight rows: rotate, per-group RMS, snap, pack.
 * "How it works", "Quantizing a weight, with no data" (all four steps).
 * W: device [rows, cols] of dtype wdt (f32 or bf16); rot->dim == cols.
 * Each group of `group` rotated values is divided by its RMS
 * sqrt(sum v^2 / group) computed in fp32 (a zero group gives u = 0); the
 * stored scale is that RMS rounded to fp16 (nearest even).  The code of u is
 * the number of thresholds strictly below u (fp32 compare).
 * codes: device uint32 [rows, row_stride_words] (padding written as zero);
 * scales: device fp16 [rows, cols/group].  cb->levels: 3, 4, 8 or 16. */
tq_status tq_quantize(const void* W, tq_dtype wdt, int64_t rows, int32_t cols, int32_t group,
                      const tq_rotation_t* rot, const tq_codebook_t* cb,
                      uint32_t* codes, uint16_t* scales, int64_t row_stride_words, void* stream);

/* Dense quantized matvec, codes decoded inline: y[t, n] = sum_k W_rot[n, k] x_rot[t, k]
 * with W_rot[n, k] = fp16 scale[n, k/group] * centroid[code[n, k]] of expert 0.
 * "How it works", "Running a quantized layer": fused kernels decode the packed
 * codes inline, so the full-precision weights never exist.
 * x_rot: device f32 [T, cols] (already rotated).  y: device [T, rows] of ydt
 * (f32 or bf16).  T >= 0 (0: nothing is launched).  cb->levels: 3, 4, 8 or 16.
 * Arithmetic: fp32 products and sums of the decoded weights (the three-level
 * kernels hold the input as 16-bit integers with one scale per vector);
 * tq_qmv_tc is the tensor-core form with fp16 operands. */
tq_status tq_qmv(const tq_qweight_t* w, const float* x_rot, int32_t T, void* y, tq_dtype ydt, void* stream);

/* MoE decode: every routed expert reads the shared input of its token.
 * "How it works", "Running a quantized layer", row "Decoding one token"
 * (polar_gather_qmv).  y[t, j, :] = W_{ids[t, j]} x_rot[t].
 * x_rot: device f32 [T, cols].  ids: device int32 [T, k].  y: device
 * [T, k, rows] of ydt (f32 or bf16).  Out-of-range ids zero their row of y
 * and set TQ_DEVERR_BAD_ID in *err.
 * ws: 16-byte aligned device scratch of tq_gather_qmv_workspace_bytes(w, T, k)
 * bytes, or NULL.  Three-level books with group 16 run a table-lookup kernel
 * that splits rows wider than 2560 columns among CTAs; their partial sums go
 * to ws.  With ws NULL (or too small) such rows take the single-pass kernel
 * instead (slower); a size of 0 means no scratch is needed.  Bit-packed books
 * (4, 8, 16 levels) with T >= 2 and the full scratch group the T*k pairs by
 * expert on the device, so a repeated expert's words are decoded once for up
 * to four of its pairs; its rows wider than one column chunk also keep their
 * partial sums in ws.  Without scratch the pairs run one by one (an f32 y then
 * takes the chunks' sums by atomics; a bf16 y takes the single-pass kernel).
 * Every path gives each pair the same products; only the order in which the
 * column chunks' sums are added may differ.
 * Arithmetic of the three-level kernels: the input is held as integers per
 * group of 16 columns (|xq| <= 8191, one fp32 scale per group; the
 * single-pass kernel: 16-bit, one scale per vector); products and sums of
 * those integers are exact, the group and weight scales are applied in fp32.
 * Bit-packed books: fp32 products and sums. */
tq_status tq_gather_qmv(const tq_qweight_t* w, const float* x_rot, const int32_t* ids, int32_t T, int32_t k,
                        void* y, tq_dtype ydt, void* ws, size_t ws_bytes, uint32_t* err, void* stream);
size_t tq_gather_qmv_workspace_bytes(const tq_qweight_t* w, int32_t T, int32_t k);

/* MoE with a different input for each (expert, input) pair.
 * "How it works", row "Prefill with a different input per expert"
 * (polar_multi_gather_qmv).  y[p, :] = W_{ids[p]} x_rot[p].
 * x_rot: device f32 [P, cols].  ids: device int32 [P].  y: device [P, rows]
 * of ydt (f32 or bf16).  ws / ws_bytes and the arithmetic as for
 * tq_gather_qmv (tq_multi_gather_qmv_workspace_bytes(w, P) bytes; bit-packed
 * books with the full scratch group the pairs by expert, each expert decoded
 * once per record of up to four pairs). */
tq_status tq_multi_gather_qmv(const tq_qweight_t* w, const float* x_rot, const int32_t* ids, int32_t P,
                              void* y, tq_dtype ydt, void* ws, size_t ws_bytes, uint32_t* err, void* stream);
size_t tq_multi_gather_qmv_workspace_bytes(const tq_qweight_t* w, int32_t P);

/* tq_gather_qmv with the input rotation done inside the matvec: y[t, j, :] =
 * W_{ids[t, j]} (R x[t]), R = rot (blockdiag(H_block) diag(signs) / sqrt(block),
 * "How it works": the input is rotated once per layer and shared by every
 * expert).  x: device [T, cols] of xdt (f32 or bf16); rot->dim == cols.
 * Saves the separate tq_rotate launch of a decode step.  Supported for
 * three-level books with group 16 whose banks the tensor-copy kernel can read
 * (16-byte aligned codes and scales, row and expert strides in whole 16-byte
 * chunks, cols a multiple of 32, rot->block in 32..8192); TQ_ERR_UNSUPPORTED
 * otherwise (then call tq_rotate and tq_gather_qmv). */
tq_status tq_gather_qmv_rotate(const tq_qweight_t* w, const void* x, tq_dtype xdt, const tq_rotation_t* rot,
                               const int32_t* ids, int32_t T, int32_t k, void* y, tq_dtype ydt, uint32_t* err,
                               void* stream);

/* tq_multi_gather_qmv with tq_swiglu_rotate folded in: y[p, :] = W_{ids[p]} h_rot[p]
 * with h_rot[p] = R (silu(gate_up[p, 0:cols]) * gate_up[p, cols:2 cols]).
 * gate_up: device f32 [P, 2 * cols] (an expert's gate | up outputs); rot->dim ==
 * cols.  Same support as tq_gather_qmv_rotate; TQ_ERR_UNSUPPORTED otherwise
 * (then call tq_swiglu_rotate and tq_multi_gather_qmv). */
tq_status tq_multi_gather_qmv_swiglu(const tq_qweight_t* w, const float* gate_up, const tq_rotation_t* rot,
                                     const int32_t* ids, int32_t P, void* y, tq_dtype ydt, uint32_t* err,
                                     void* stream);

/* Router: top-k experts per token, softmax weights, expert-sorted pair order.
 * "Running a 1T-Parameter Model on a Laptop": the router picks the 8 best of
 * 384 experts per token; "How it works", row "A large batch sorted by expert".
 * logits: device f32 [T, E] (E <= 1024, k <= 32, k <= E).  Ties go to the
 * lower expert id; ids[t, :] is in descending logit order.  probs: softmax over
 * the k selected logits.  Pairs f = t*k + j are sorted by (expert, f):
 * perm[i] = pair at sorted position i; pair_pos[f] = sorted position of pair f;
 * offsets[e] = first sorted position of expert e, offsets[E] = T*k.
 * ids, perm, pair_pos: device int32 [T*k]; probs: device f32 [T*k];
 * offsets: device int32 [E+1].  ws: device scratch of at least
 * tq_route_workspace_bytes(E) bytes (contents need not be initialised).
 * With perm, pair_pos and offsets all NULL only ids and probs are written
 * (one token's decode reads the experts by id and needs no sorted order);
 * ws may then be NULL.  pair_pos alone may be NULL when sorting. */
tq_status tq_moe_route(const float* logits, int32_t T, int32_t E, int32_t k, int32_t* ids, float* probs,
                       int32_t* perm, int32_t* pair_pos, int32_t* offsets, void* ws, size_t ws_bytes,
                       void* stream);
size_t tq_route_workspace_bytes(int32_t E);

/* SwiGLU between an expert's gate/up and down projections, followed by the
 * rotation of the intermediate (the down projection consumes R h).
 * gate_up: device f32 [P, 2*inter], gate in columns [0, inter), up in
 * [inter, 2*inter).  h_rot[p] = R (silu(gate) * up), silu(g) = g / (1 + e^-g).
 * rot->dim == inter.  h_rot: device [P, inter] of ydt (f32, bf16 or f16). */
tq_status tq_swiglu_rotate(const float* gate_up, int64_t P, int32_t inter, const tq_rotation_t* rot,
                           void* h_rot, tq_dtype ydt, void* stream);

/* Router-weighted sum of the experts' outputs: out[t] = sum_j probs[t*k+j] * y[row(t*k+j)],
 * row(f) = pair_pos[f] when pair_pos is not NULL (y in expert-sorted order),
 * else f (y in pair order).  y: device f32 [T*k, H].  out: device [T, H] of
 * odt (f32 or bf16). */
tq_status tq_moe_combine(const float* y, const float* probs, const int32_t* pair_pos, int32_t T, int32_t k,
                         int32_t H, void* out, tq_dtype odt, void* stream);

/* MoE prefill: expert-sorted batched gather-GEMM on the tensor cores.
 * "How it works", row "A large batch sorted by expert" (polar_gather_qmm).
 * For sorted position i with expert e (offsets[e] <= i < offsets[e+1]):
 *   y[i, :] = W_e x_src(i),  src(i) = perm[i] / k  (per_pair_input == 0: rows of
 *   x are tokens) or src(i) = i (per_pair_input != 0: rows of x are the
 *   sorted pairs' own inputs).
 * Codes are decoded to the operand type xdt (f16 or bf16) in shared memory and
 * multiplied with fp32 accumulation.  x: device [T or P, cols] of xdt (already
 * rotated, 16-byte aligned).  perm: device int32 [P] (ignored when
 * per_pair_input); an entry outside [0, P) sets TQ_DEVERR_BAD_ID and its pair
 * reads a zero input row.  offsets: device int32 [experts+1].  y: device
 * [P, rows] of ydt (f32 or bf16).  ws: 16-byte aligned device scratch of at
 * least tq_gather_qmm_workspace_bytes(P, cols, per_pair_input) bytes (the
 * token rows gathered into sorted pair order; TQ_ERR_INVALID if smaller).
 * cols must be a multiple of 64, rows a multiple of 128. */
tq_status tq_gather_qmm(const tq_qweight_t* w, const void* x, tq_dtype xdt, const int32_t* perm,
                        const int32_t* offsets, int32_t P, int32_t k, int32_t per_pair_input,
                        void* y, tq_dtype ydt, void* ws, size_t ws_bytes, uint32_t* err, void* stream);
size_t tq_gather_qmm_workspace_bytes(int32_t P, int32_t cols, int32_t per_pair_input);

/* Dense matvec on the tensor cores: y[t, :] = W x_rot[t] for expert 0 of w, as
 * tq_qmv computes it, with fp16 operands.
 * "How it works", "Running a quantized layer" (the rotated input times the
 * codes, decoded inline; the full-precision weights are never written out).
 * Each input row is scaled by the power of two 2^e_t just above its largest
 * magnitude and rounded to fp16; the decoded weights c[code] * s_group are
 * formed in fp16; products accumulate in fp32 and the outputs are scaled back
 * by 2^e_t.  The columns are split among the SMs and
 * the partial sums added with atomics (the summation order varies from run to
 * run).  x_rot: device f32 [T, cols].  y: device f32 [T, rows] (overwritten).
 * ws: 16-byte aligned device scratch of at least tq_qmv_tc_workspace_bytes(T,
 * cols) bytes (TQ_ERR_INVALID if smaller); it holds the fp16 rows and their
 * scales and must not be shared with a call running concurrently.
 * TQ_ERR_UNSUPPORTED (nothing launched) unless cb->levels is 4, 8 or 16, rows
 * is a multiple of 128, cols a multiple of 64 with at most 64 groups per row,
 * and 1 <= T <= 64; tq_qmv covers the other cases.  err: optional device word
 * (NULL: not reported); a bounded wait that ran out sets TQ_DEVERR_TIMEOUT
 * there, and y then holds partial sums. */
tq_status tq_qmv_tc(const tq_qweight_t* w, const float* x_rot, int32_t T, float* y, void* ws, size_t ws_bytes,
                    uint32_t* err, void* stream);
size_t tq_qmv_tc_workspace_bytes(int32_t T, int32_t cols);

/* Dequantize selected experts to dense rotated-domain weights, for a regular matmul.
 * "How it works", row "Anything else" (polar_dequant_experts).
 * out[i, n, c] = fp16 scale * centroid of expert ids[i]; out: device
 * [n_ids, rows, cols] of odt (f32, bf16 or f16).  The caller multiplies by the
 * rotated input. */
tq_status tq_dequant_experts(const tq_qweight_t* w, const int32_t* ids, int32_t n_ids, void* out, tq_dtype odt,
                             uint32_t* err, void* stream);

/* KV cache compression of T new tokens at positions [pos, pos+T).
 * "How it works", "The KV cache": the same rotation and codebook compress the
 * cache at run time (8-bit keys, 3-bit values recommended);
 * "Running a 1T-Parameter Model on a Laptop", update_and_fetch: rotate, then
 * quantize.  Each (token, head) vector of D is rotated by rot (dim = block =
 * D), split into groups of `group`, scaled by the group RMS and snapped.
 * k, v: device [T, Hkv, D] of dt (f32 or bf16).  Outputs, for each head h and
 * position p: kcodes + (h*capacity + p)*kw (kw = tq_row_words(kcb->levels, D)
 * words), kscales + (h*capacity + p)*(D/group), and the same for v with vw.
 * D: 128 (one warp per vector).  kcb/vcb levels: 3, 4, 8, 16 or 256. */
tq_status tq_kv_quantize(const void* k, const void* v, tq_dtype dt, int32_t T, int32_t Hkv, int32_t D,
                         int64_t pos, int64_t capacity, const tq_rotation_t* rot,
                         const tq_codebook_t* kcb, const tq_codebook_t* vcb, int32_t group,
                         uint32_t* kcodes, uint16_t* kscales, uint32_t* vcodes, uint16_t* vscales,
                         void* stream);

/* One decode step of attention read straight from the compressed cache.
 * "Running a 1T-Parameter Model on a Laptop", update_and_fetch: the cache is
 * dequantized and de-rotated and attention softmax(q K^T / sqrt(D)) V runs on
 * it.  Here the rotation is moved algebraically: q_rot = R q, scores
 * q_rot . k_rot_hat / sqrt(D), o = R^T sum_t p_t v_rot_hat(t) (one
 * de-rotation of the output instead of one per cached token).
 * q: device [Hq, D] of qdt (f32 or bf16); query head h reads kv head
 * h / (Hq/Hkv).  Cache layout as written by tq_kv_quantize, first ctx
 * positions.  o: device f32 [Hq, D].  ws: device scratch of
 * tq_kv_attend_workspace_bytes(Hq, D, ctx) bytes.  D: 128. */
tq_status tq_kv_attend(const void* q, tq_dtype qdt, int32_t Hq, int32_t Hkv, int32_t D, int64_t ctx,
                       int64_t capacity, const tq_rotation_t* rot, const tq_codebook_t* kcb, const tq_codebook_t* vcb,
                       int32_t group, const uint32_t* kcodes, const uint16_t* kscales, const uint32_t* vcodes,
                       const uint16_t* vscales, float* o, void* ws, size_t ws_bytes, void* stream);
size_t tq_kv_attend_workspace_bytes(int32_t Hq, int32_t D, int64_t ctx);

/* tq_kv_attend without a caller-supplied workspace.
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory where they run attention: for example a
 * serving process whose device memory is all handed out up front by its own
 * pool, or a plug-in inside a host framework that owns every device buffer
 * and gives the plug-in no allocator.  cudaMalloc and cudaFree can also
 * synchronise the device, which a latency-bound decode loop may not accept.
 * Arguments and results are those of tq_kv_attend minus ws / ws_bytes.  The
 * split-context partial results live instead in a fixed array of
 * tq_kv_attend_noalloc_max_scratch_bytes() bytes (4 MiB) inside the library's
 * device image: every GPU that loads the library holds it until the process
 * exits.  No memory is allocated by the call (no cudaMalloc, cudaFree or
 * allocating library routine).  The first call on each device looks up the
 * array's device address (cudaGetSymbolAddress, with that device current) and
 * caches it for the device's current CUDA context; make that first call
 * before any stream capture.  After cudaDeviceReset (a new context) the next
 * call looks the address up again, so it too belongs before any capture.  Sizes whose
 * scratch, tq_kv_attend_workspace_bytes(Hq, D, ctx), exceeds the maximum
 * return TQ_ERR_INVALID without launching.  All calls on a device share the
 * array, which keeps the previous call's contents (every slot a call reads is
 * first written by that call); calls whose kernels overlap on the GPU, e.g.
 * on two streams, race on it and must be serialised by the caller. */
tq_status tq_kv_attend_noalloc(const void* q, tq_dtype qdt, int32_t Hq, int32_t Hkv, int32_t D, int64_t ctx,
                               int64_t capacity, const tq_rotation_t* rot, const tq_codebook_t* kcb,
                               const tq_codebook_t* vcb, int32_t group, const uint32_t* kcodes,
                               const uint16_t* kscales, const uint32_t* vcodes, const uint16_t* vscales, float* o,
                               void* stream);
size_t tq_kv_attend_noalloc_max_scratch_bytes(void);

/* ------------------------------------------------------------------ fused decode layer */

/* One token through a Mixture-of-Experts layer in one launch: route (top-k of
 * the E logits, softmax over the k), rotate x (rot_h), gate||up gather, SwiGLU
 * and the intermediate rotation (rot_i) of each routed expert's output, down
 * gather, out = sum_j probs[j] * down_j.  "How it works", "Running a quantized
 * layer" and the Kimi-K2 router of "Running a 1T-Parameter Model on a Laptop".
 * One cooperative launch whose phases meet at grid barriers (each wait bounded
 * by the wait budget: TQ_DEVERR_TIMEOUT in *err on expiry), after a 4-byte
 * memset of the barrier counter in ws; the arithmetic is that of tq_moe_route,
 * tq_rotate, tq_gather_qmv, tq_swiglu_rotate, tq_multi_gather_qmv and
 * tq_moe_combine in sequence, with the same bits.
 * gate_up: ternary bank, group 16, rows = 2 * down->cols (gate rows first),
 * cols = H; down: ternary bank, group 16, rows = H, cols = I, the same expert
 * count E <= 512.  logits: device f32 [E]; x: device [H] of xdt; out: device
 * [H] of odt (f32 or bf16); k <= 32.  ws: device scratch of
 * tq_moe_decode_layer_workspace_bytes(gate_up, down, k) bytes, 256-byte
 * aligned; calls that may run at the same time must not share it.
 * TQ_ERR_UNSUPPORTED for shapes this launch does not take (then call the
 * separate entry points): H a multiple of 1024 rotated in blocks of 1024 into
 * 2 to 8 table-lookup slices, I = 2048 rotated as one block of 2048. */
size_t tq_moe_decode_layer_workspace_bytes(const tq_qweight_t* gate_up, const tq_qweight_t* down, int32_t k);
tq_status tq_moe_decode_layer(const tq_qweight_t* gate_up, const tq_qweight_t* down, const tq_rotation_t* rot_h,
                              const tq_rotation_t* rot_i, const float* logits, const void* x, tq_dtype xdt,
                              int32_t k, void* out, tq_dtype odt, void* ws, size_t ws_bytes, uint32_t* err,
                              void* stream);

/* ------------------------------------------------------------------ persisted packed layers (host) */

/* Per-layer tiers and a persisted packed format.
 * "How it works", "The ternary tier (1.58 bits)": the format marks itself (2^b
 * codebook entries = bit-packed, 3 = trit-packed), so a model mixes tiers layer
 * by layer (ternary experts, 4-bit down projections, 3-bit protected layers);
 * "Configuration that converter and loader share": bit widths are chosen per
 * layer from its name, the loader recomputes the same choice, and a layer's
 * width is recovered from the size of its saved codebook, never from a config
 * field.  The weight-reservoir page: a flat, page-aligned file of each layer's
 * packed indices and scales with a small header (shape, rotation seed), loaded
 * byte-identical to what was written.  All of this is host code: buffers are
 * host memory, and nothing touches the GPU. */

#define TQ_LAYER_NAME_BYTES 64

/* A quantized layer as stored: name (NUL-terminated), a bank of `experts`
 * matrices [rows, cols] with `group`-wide fp16 scales, codes at row_stride_words
 * words per row, the rotation (dim = cols, Hadamard block, sign seed) and the
 * codebook: `levels` fp64 centroids, ascending.  codes: host uint32
 * [experts][rows][row_stride_words]; scales: host fp16 bits
 * [experts][rows][cols/group]. */
typedef struct tq_layer_desc_t {
    char name[TQ_LAYER_NAME_BYTES];
    int32_t experts, rows, cols, group;
    int64_t row_stride_words;
    int32_t levels;
    int32_t rot_dim, rot_block;
    uint64_t rot_seed;
    const double* centroids;
    const uint32_t* codes;
    const uint16_t* scales;
} tq_layer_desc_t;

/* Tier (codebook size and group) of each layer class.  A layer belongs to the
 * first class whose marker its name contains: "down_proj", "expert", "mlp",
 * "attn"; any other layer (e.g. a protected embedding or head) is "other". */
typedef struct tq_tier_policy_t {
    int32_t down_levels, down_group;
    int32_t expert_levels, expert_group;
    int32_t mlp_levels, mlp_group;
    int32_t attn_levels, attn_group;
    int32_t other_levels, other_group;
} tq_tier_policy_t;

/* The tier of layer `name` under `policy`: *levels and *group.  TQ_ERR_INVALID
 * for NULL arguments or a policy entry that is not a supported book / group. */
tq_status tq_layer_tier(const char* name, const tq_tier_policy_t* policy, int32_t* levels, int32_t* group);

/* Writes n_layers layers to `path` (overwritten): a 64-byte header, one 256-byte
 * record per layer, then each layer's codebook, codes and scales, each blob
 * starting on a 4096-byte boundary with zero bytes between.  Writing the same
 * layers again gives the same bytes.  TQ_ERR_INVALID for an inconsistent layer
 * (levels not 3/4/8/16/256, rot_dim != cols, block not dividing cols, stride too
 * short, unterminated name, NULL data) or an I/O error. */
tq_status tq_pack_file_write(const char* path, const tq_layer_desc_t* layers, int32_t n_layers);

/* Reads the layer table of `path`: *n_layers, and the first min(cap, n) layers'
 * metadata into infos (pointers left NULL).  Each layer's levels is the number of
 * centroids stored in its codebook blob.  TQ_ERR_INVALID for a file that is not a
 * packed-layer file of this version or whose table points past its end. */
tq_status tq_pack_file_info(const char* path, int32_t* n_layers, tq_layer_desc_t* infos, int32_t cap);

/* Reads layer `index` of `path` into host buffers sized from tq_pack_file_info:
 * centroids double[levels], codes uint32[experts*rows*row_stride_words], scales
 * uint16[experts*rows*(cols/group)]. */
tq_status tq_pack_file_read_layer(const char* path, int32_t index, double* centroids, uint32_t* codes,
                                  uint16_t* scales);

/* ------------------------------------------------------------------ expert streaming (host bank, device LRU) */

/* Expert streaming from host memory.
 * "How it works", "Expert streaming": a Mixture-of-Experts bank larger than the
 * device budget stays outside it, and only the experts a step routes to are
 * brought in, through a least-recently-used cache, with results bit-identical
 * to running the whole bank resident.  "Running a 1T-Parameter Model on a
 * Laptop": expert loading reads only the routed experts.
 *
 * Here the bank is a tq_qweight_t whose codes and scales are HOST memory
 * (pinned, so that copies run asynchronously over the CPU-GPU link), experts
 * back to back (expert_stride_words = rows*row_stride_words, expert_stride_scales
 * = rows*cols/group).  The cache owns no memory on either side: dev_codes
 * (uint32 [slots][rows][row_stride_words]) and dev_scales (fp16 bits
 * [slots][rows][cols/group]) are caller-allocated device buffers that must stay
 * valid for the cache's lifetime.  A device-side view of the slots is the bank
 * with codes/scales replaced by dev_codes/dev_scales and experts = slots; the
 * gather entry points run on it with ids remapped to slots. */
typedef struct tq_expert_cache tq_expert_cache;

/* Creates a cache of `slots` device slots over `host_bank` (copied; the
 * arrays it points to are not).  TQ_ERR_INVALID for NULL arguments, slots <= 0
 * or a malformed bank; TQ_ERR_UNSUPPORTED for experts not stored back to back. */
tq_status tq_expert_cache_create(const tq_qweight_t* host_bank, int32_t slots, uint32_t* dev_codes,
                                 uint16_t* dev_scales, tq_expert_cache** out);

/* Frees the bookkeeping (not the buffers).  NULL is a no-op. */
void tq_expert_cache_destroy(tq_expert_cache* cache);

/* One step of LRU bookkeeping, host only: for ids[0..n) (host int32 expert ids,
 * repeats allowed) writes slots[i] (host int32), the slot holding expert ids[i]
 * after the step, and miss[i] (host uint8) = 1 where ids[i] is the first
 * occurrence of an expert that was not cached and must be copied into slots[i].
 * Experts used in the step are never evicted by the step; the victim of a miss is
 * the lowest empty slot if any, else the slot used least recently (the lowest
 * of equals).  TQ_ERR_INVALID for
 * an id outside [0, experts) (nothing changes) or more distinct uncached experts
 * than slots not used by the step (no slot changes content). */
tq_status tq_expert_cache_plan(tq_expert_cache* cache, const int32_t* ids, int32_t n, int32_t* slots, uint8_t* miss);

/* tq_expert_cache_plan, then the copies of every missing expert's code words
 * and scales into its slot, on `stream`: one kernel launch that reads the bank
 * directly over the CPU-GPU link when the bank is pinned memory mapped into the
 * device's address space and every expert's codes and scales are whole 16-byte
 * pieces at 16-byte aligned addresses (checked at creation), else two
 * cudaMemcpyAsync per missing expert.  Work on `stream` after the call sees the
 * experts in place.  TQ_ERR_CUDA if a copy cannot be enqueued. */
tq_status tq_expert_cache_map(tq_expert_cache* cache, const int32_t* ids, int32_t n, int32_t* slots, void* stream);

/* Counters since creation: distinct-per-step hits and misses, and bytes copied
 * (any pointer may be NULL). */
tq_status tq_expert_cache_stats(const tq_expert_cache* cache, int64_t* hits, int64_t* misses,
                                int64_t* bytes_copied);

/* Waits for `stream`, reads the device error word and clears it.
 * Returns TQ_OK if it was 0, TQ_ERR_TIMEOUT if TQ_DEVERR_TIMEOUT is set, else
 * TQ_ERR_DEVICE; *bits (host, may be NULL) receives the word. */
tq_status tq_check_error(uint32_t* err, uint32_t* bits, void* stream);

/* Test hook for the bounded waits of the tensor-core kernels (tq_gather_qmm,
 * tq_qmv_tc) and of the three-level tensor-copy matvec (the ternary kernel of
 * calls without scratch, of groups other than 16 and of the fused input
 * stages): every wait of a pipeline role on another (an mbarrier phase)
 * gives up after `cycles` SM clock cycles, raises TQ_DEVERR_TIMEOUT in the
 * call's error word (tq_check_error then returns TQ_ERR_TIMEOUT) and the CTA
 * stops: each role drains the copies and MMAs it has in flight (bounded by the
 * default budget, whatever `cycles` is), TMEM is freed and the kernel returns,
 * leaving the output incomplete.  Applies to launches after the call, process
 * wide.  cycles < 0 restores the default, 2^31 cycles (about a second); 0 makes
 * every wait whose phase has not already completed give up at once.  Not for
 * production use: a short budget aborts work that would have finished. */
tq_status tq_set_wait_budget(int64_t cycles);

/* Exhaustive self-check of the divide-free base-3 digit decoder used by the
 * ternary kernels: decodes every word in [first, first+count) (count words,
 * first+count <= 3^20) and compares each digit with plain division.
 * mismatches: device uint64 counter, incremented per wrong word (caller
 * zeroes it).  For tests. */
tq_status tq_selftest_trit_decode(uint32_t first, uint32_t count, unsigned long long* mismatches, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H_ */
