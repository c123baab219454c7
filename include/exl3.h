/*
 * exl3.h - C ABI of libexl3: fused randomized-Hadamard + bitshift-trellis
 * decode + GEMV / skinny GEMM for GB300 (sm_103a).
 *
 * What is computed (source pages):
 *   - "Trellis Quantization" (Lecture 1b), Part eight: every 16x16 weight tile
 *     is one 256-step tail-biting bitshift trellis; the state of step t is the
 *     16-bit window starting at bit K*t of the tile's circular 256*K-bit stream.
 *   - same lecture, Part nine: the lookup-free computed codes 3INST and 1MAD
 *     turn a state into a binary16 weight.
 *   - "ExLlamaV3 & EXL3 Deep Dive", Section 2: the randomized Hadamard transform
 *     applied to x on the way in and to the product on the way out, so that
 *     y = Hb(s_out (.) (scale (.) (W-hat Hb(s_in (.) x)))); Lecture 1b Part
 *     eleven: Hb is blockwise over 128-element blocks, H_128 Sylvester-ordered
 *     and normalized by 1/sqrt(128).
 *   - "EXL3 field guide": per-output-channel binary16 scales.
 *
 * Data formats (all little-endian device memory):
 *   codes   uint32 words; tile (I, J) (rows 16I..16I+15, columns 16J..16J+15)
 *           occupies words [(I*(n/16) + J) * 8K, +8K).  Stream bit j of a tile
 *           is bit 31 - (j % 32) of its word j / 32 (MSB first).  Step t of a
 *           tile is element (16I + t/16, 16J + t%16).
 *   half    IEEE-754 binary16 bit patterns (exl3_half).
 *   x       [M][n] row-major halves; y [M][m] row-major halves.
 *   signs   +-1 halves, length n (s_in) or m (s_out).  NULL = no rotation on
 *           that side (neither signs nor Hadamard).
 *   scales  length-m halves.
 *
 * Conventions:
 *   - Ownership: every pointer is caller-owned device memory; the library
 *     allocates, frees and synchronizes nothing (exl3_device_status, which
 *     waits for the stream, excepted), and keeps no per-call global state.  Calls are asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream).
 *   - Validation happens on the host before anything is launched; on any
 *     error nothing is launched and the outputs are untouched:
 *       m, n positive multiples of 128 (EXL3_ERR_SHAPE), 1 <= K <= 8
 *       (EXL3_ERR_K), known codebook (EXL3_ERR_CODEBOOK), batch M within the
 *       call's range (EXL3_ERR_BATCH), required pointers non-NULL
 *       (EXL3_ERR_NULL), every device pointer 16-byte aligned (EXL3_ERR_ALIGN),
 *       workspace large enough (EXL3_ERR_WORKSPACE).
 *   - A failed launch returns EXL3_ERR_CUDA (the CUDA error is left for
 *     cudaGetLastError to report as well).
 *   - No C++ exception crosses this interface.
 */
#ifndef EXL3_H_
#define EXL3_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/** A cudaStream_t. */
typedef struct CUstream_st *exl3_stream_t;

/** IEEE-754 binary16 bit pattern. */
typedef uint16_t exl3_half;

typedef enum {
  EXL3_OK = 0,
  EXL3_ERR_NULL = 1,
  EXL3_ERR_SHAPE = 2,
  EXL3_ERR_K = 3,
  EXL3_ERR_CODEBOOK = 4,
  EXL3_ERR_BATCH = 5,
  EXL3_ERR_ALIGN = 6,
  EXL3_ERR_WORKSPACE = 7,
  EXL3_ERR_CUDA = 8,
  EXL3_ERR_DEVICE_CHECK = 9,
  EXL3_ERR_SCRATCH = 10
} exl3_status;

/** Computed codes ("Trellis Quantization" Parts nine, eleven and twelve):
 *  3INST and 1MAD on the LCG x = A*s + B; MCG (3INST on the multiplicative
 *  generator x = A*s) and mul1 (six-bit masked byte sum of A*s, minus 126,
 *  times 1/sqrt(1365)) as far as the pages fix them; A = 0x9E3779B9,
 *  B = 0x7F4A7C15. */
typedef enum { EXL3_CB_3INST = 0, EXL3_CB_1MAD = 1, EXL3_CB_MCG = 2, EXL3_CB_MUL1 = 3 } exl3_codebook;

/** Largest batch accepted by exl3_gemm_small. */
#define EXL3_MAX_BATCH 32

/**
 * Input-side randomized Hadamard transform (Deep Dive Section 2; Lecture 1b
 * Part eleven): x_rot[b] = Hb(s_in (.) x[b]) for b < M, rounded once to binary16.
 *   x      [M][n] halves (read)      s_in  [n] +-1 halves (read, required)
 *   x_rot  [M][n] halves (written; must not overlap x)
 *   M >= 1, n a multiple of 128.
 */
exl3_status exl3_rht_in(const exl3_half *x, const exl3_half *s_in, exl3_half *x_rot,
                        int M, int n, exl3_stream_t stream);

/**
 * Output-side transform (Deep Dive Section 2, the H^T diag(s_left) factor of
 * the runtime identity; H_128 is symmetric): y[b] = Hb(s_out (.) z[b]).
 *   z [M][m] halves (read)   s_out [m] (read, required)   y [M][m] (written)
 */
exl3_status exl3_rht_out(const exl3_half *z, const exl3_half *s_out, exl3_half *y,
                         int M, int m, exl3_stream_t stream);

/**
 * Decode every tile into the unscaled binary16 W-hat (Lecture 1b Parts eight
 * and nine).  Bit-exact: each weight is one defined binary16 value.
 *   codes  (m/16)*(n/16)*8K words (read)
 *   w_out  [m][n] row-major halves (written)
 */
exl3_status exl3_decode_tiles(const uint32_t *codes, int K, int codebook, int m, int n,
                              exl3_half *w_out, exl3_stream_t stream);

/**
 * Bytes of scratch that exl3_gemv / exl3_gemm_small need for an m x n layer
 * at batch M: per-row-block counters and the status word, M*m fp32 row sums,
 * and then either the warp-shuffle kernel's x pairs (M*n 32-bit words) or the
 * decode-MMA kernel's rotated input laid out as its MMA operand (16 or 32
 * rows of n halves) with M*(n/128) fp32 block sums.
 * Returns 0 for an invalid shape or batch.  The workspace must be zero-filled
 * once after allocation; every call leaves it zero-filled again.  Two calls
 * that may run concurrently must not share a workspace.  The uint32 at byte
 * offset 4*(m/128) is a status word: the tensor-core kernel ORs 1 into it if
 * one of its bounded device-side waits timed out (its outputs are then not
 * valid); it stays set until the caller clears it.  After a call that set it,
 * zero-fill the whole workspace again before reusing it.
 */
size_t exl3_workspace_bytes(int m, int n, int M);

/**
 * Fused batch-1 layer (the decode-time quantized linear of Deep Dive
 * Sections 2-3):  y = Hb(s_out (.) (scale (.) (W-hat Hb(s_in (.) x)))),
 * W-hat decoded on the fly from `codes`, y rounded once to binary16.
 * Arithmetic: on the warp-shuffle kernel (batch 1 and 2 by default) each
 * weight-activation product is formed and summed in binary16 over the 16
 * columns of one tile, and the tile sums are accumulated in fp32; on the
 * decode-MMA kernel (batch 3 to 32 by default) binary16 weights and
 * binary16 rotated activations meet in tcgen05 MMAs that accumulate in fp32.
 * Both stay within the documented tolerance of the exact layer.
 *   x [n] halves, y [m] halves, scales [m] halves (required);
 *   s_in [n] / s_out [m] or NULL (no rotation on that side);
 *   workspace: >= exl3_workspace_bytes(m, n, 1) bytes, see there.
 */
exl3_status exl3_gemv(const uint32_t *codes, int K, int codebook, int m, int n,
                      const exl3_half *s_in, const exl3_half *s_out,
                      const exl3_half *scales, const exl3_half *x, exl3_half *y,
                      void *workspace, size_t workspace_bytes, exl3_stream_t stream);

/**
 * Same layer for a skinny batch of 1 <= M <= EXL3_MAX_BATCH rows:
 * x [M][n] -> y [M][m].  workspace >= exl3_workspace_bytes(m, n, M).
 */
exl3_status exl3_gemm_small(const uint32_t *codes, int K, int codebook, int m, int n,
                            const exl3_half *s_in, const exl3_half *s_out,
                            const exl3_half *scales, int M, const exl3_half *x,
                            exl3_half *y, void *workspace, size_t workspace_bytes,
                            exl3_stream_t stream);

/**
 * Bytes of scratch for exl3_gemm at batch M: exl3_workspace_bytes(m, n, M) for
 * M <= EXL3_MAX_BATCH; above, enough for either prefill strategy: the
 * counters and status word, fp32 row sums [M][m], the rotated x as operand
 * images (M rounded up to 256 rows, times n binary16), the decoded matrix
 * (m * n binary16) and one uint32 per (128-row block, 256-row batch tile);
 * batches of up to 128 rows run as one narrower tile inside these regions.
 * Same zero-fill contract and status word as exl3_workspace_bytes.  0 for an
 * invalid shape or M < 1.
 */
size_t exl3_gemm_workspace_bytes(int m, int n, int M);

/**
 * The layer for any batch M >= 1 (prefill): x [M][n] -> y [M][m].  Up to
 * EXL3_MAX_BATCH rows this is exl3_gemm_small.  Above, a tcgen05 GEMM (128 x
 * N x 16 MMAs, both operands in shared memory) runs over all M rows, with the
 * weights in one of two ways (exl3_set_prefill):
 *   - fused (default up to 256 rows): each CTA decodes the codes of every
 *     64-column stage into a binary16 operand image in shared memory, once
 *     per batch tile (N = 64 up to 64 rows, 128 up to 128, else tiles of 256);
 *   - decode-once (default above 256 rows): the matrix is decoded once per
 *     call into binary16 in the workspace and streamed from there (N = 64
 *     up to 64 rows, 128 up to 128, else tiles of 256): "decode a block once
 *     and reuse it", Lecture 1b Part fourteen -- at large batch the decode is
 *     amortised and the product is a plain matrix multiplication.
 * With EXL3_PATH_TENSOR selected, passes of 128 rows run the tensor-core
 * kernel with 128 batch columns per MMA instead, decoding each tile once per
 * pass into tensor memory.  All compute the layer within the documented
 * tolerance.
 */
exl3_status exl3_gemm(const uint32_t *codes, int K, int codebook, int m, int n,
                      const exl3_half *s_in, const exl3_half *s_out,
                      const exl3_half *scales, int M, const exl3_half *x, exl3_half *y,
                      void *workspace, size_t workspace_bytes, exl3_stream_t stream);

/**
 * QTIP's whole-vector randomized Hadamard transform ("Trellis Quantization"
 * Part eleven: QTIP rotates whole rows and columns where EXL3 rotates
 * 128-blocks): out[r] = binary16(H_d (signs (.) in[r]) / sqrt(d)) for each of
 * `rows` rows, H_d the Sylvester Hadamard matrix of order d.
 *   in, out [rows][d] halves; signs [d] halves of +-1 (required);
 *   d a power of two, 128 <= d <= 32768, else EXL3_ERR_SHAPE.
 * fp32 butterflies, one rounding to binary16.  Asynchronous on `stream`.
 */
exl3_status exl3_rht_whole(const exl3_half *in, const exl3_half *signs, exl3_half *out,
                           int rows, int d, exl3_stream_t stream);

/**
 * Bytes of scratch for exl3_gemm_whole: exl3_gemm_workspace_bytes(m, n, M)
 * rounded up to 256 bytes (first, so the status word is at byte 4*(m/128) as
 * for exl3_workspace_bytes), then max(m, n) halves of unit signs, M*n halves
 * of the input after the cross-block transform and M*m halves of the output
 * before it (each 256-byte aligned).  Same zero-fill contract.  0 unless m and
 * n are powers of two in [128, 32768] and M >= 1.
 */
size_t exl3_gemm_whole_workspace_bytes(int m, int n, int M);

/**
 * The layer with QTIP's whole-vector rotations on both sides ("Trellis
 * Quantization" Part eleven) instead of EXL3's 128-blocks:
 *   y = binary16(H_m (s_out (.) (scale (.) (W-hat H_n (s_in (.) x)))))
 * with H_d / sqrt(d) over the full length.  m and n must be powers of two in
 * [128, 32768] (EXL3_ERR_SHAPE); s_in / s_out NULL = no rotation on that side;
 * any M >= 1.  Computed as the blockwise layer (exl3_gemm) between two
 * transforms across the 128-blocks, since H_{128B} = H_B (x) H_128 in
 * Sylvester order; each of the two adds one binary16 rounding of an
 * intermediate vector.  Arguments, alignment and errors as exl3_gemm.
 */
exl3_status exl3_gemm_whole(const uint32_t *codes, int K, int codebook, int m, int n,
                            const exl3_half *s_in, const exl3_half *s_out,
                            const exl3_half *scales, int M, const exl3_half *x, exl3_half *y,
                            void *workspace, size_t workspace_bytes, exl3_stream_t stream);

/**
 * Bytes of workspace for exl3_encode_tiles to encode `ctas` tiles at a time:
 * 256 * 2^(16-K) bytes per tile in flight (the predecessor chosen for every
 * group of states at every step).  0 for K outside 1..8 or ctas < 1.
 */
size_t exl3_encode_workspace_bytes(int K, int ctas);

/**
 * Tail-biting Viterbi encoding of `tiles` 256-step sequences ("Trellis
 * Quantization" Part seven, the Viterbi search; Part eight, the bitshift
 * trellis with a 16-bit window moving K bits per step and the two-pass
 * tail-biting approximation).  For each tile: the stream of 256*K bits, as
 * 8K uint32 words MSB first (the layout exl3_decode_tiles reads), whose
 * states minimise sum_t (v(state_t) - target_t)^2, v the codebook's binary16
 * value of a state, and that cost.
 *   target [tiles][256] float, in code units (to quantize a unit-variance
 *          source, multiply it by the code's rms value);
 *   words  [tiles][8K] uint32 (out); cost [tiles] float (out).
 * Path costs are binary32, each evaluated as best + (v - x)^2 in that order;
 * the smallest predecessor wins ties, and the smallest state at the end.
 * The workspace holds one slot of exl3_encode_workspace_bytes(K, 1) bytes per
 * tile in flight; as many tiles run at once as slots fit, up to one per SM.
 * Errors: EXL3_ERR_SHAPE (tiles < 1), EXL3_ERR_K, EXL3_ERR_CODEBOOK,
 * EXL3_ERR_NULL, EXL3_ERR_ALIGN (target or words not 16-byte aligned),
 * EXL3_ERR_WORKSPACE (smaller than one slot).  Asynchronous on `stream`.
 */
exl3_status exl3_encode_tiles(const float *target, int tiles, int K, int codebook,
                              uint32_t *words, float *cost, void *workspace,
                              size_t workspace_bytes, exl3_stream_t stream);

/**
 * Activations to int8 for the dp4a path ("Trellis Quantization" Part
 * eleven).  Per 128-column block of each of M rows of the rotated activations
 * x_rot (binary16 [M][n]): qscale = max|x| / 127 and q = the nearest integer
 * to x / qscale, ties to even, both binary32 divisions correctly rounded; a
 * block of zeros gets qscale 0 and q 0.
 *   q [M][n] int8 (out), qscale [M][n/128] float (out).
 * n a multiple of 128 (EXL3_ERR_SHAPE); x_rot and q 16-byte aligned.
 */
exl3_status exl3_quantize_act(const exl3_half *x_rot, int M, int n, int8_t *q, float *qscale,
                              exl3_stream_t stream);

/**
 * Workspace of exl3_gemm_i8 / exl3_gemm_int8act: counters and status word as
 * for exl3_workspace_bytes, fp32 row sums [M][m], the activations replicated
 * into 32-bit words [M][n], per-tile corrections [M][n/16] and per-block
 * factors [M][n/128] (each 256-byte aligned).  Same zero-fill contract.  0
 * for an invalid shape or M outside 1..EXL3_MAX_BATCH.
 */
size_t exl3_gemm_i8_workspace_bytes(int m, int n, int M);

/**
 * The layer on int8 activations, for the byte-sum codes only (EXL3_CB_1MAD,
 * EXL3_CB_MUL1; others EXL3_ERR_CODEBOOK):
 *   y = binary16(Hb(s_out (.) (scale (.) (W-hat x-hat)))),
 *   x-hat[b][j] = q[b][j] * qscale[b][j / 128]   (already rotated).
 * The weight is C * (S - centre) for the byte sum S of a state, so each
 * product is one dp4a of the four (masked) bytes with q replicated four times
 * ("Trellis Quantization" Part eleven), accumulated exactly in int32 per
 * 16-column tile and scaled by C * qscale in binary32.  This uses the exact
 * affine weight rather than its binary16 rounding (within the layer
 * tolerance).  q [M][n] int8, qscale [M][n/128] float; 1 <= M <= 32; other
 * arguments as exl3_gemm_small (no s_in: the activations are given rotated).
 */
exl3_status exl3_gemm_i8(const uint32_t *codes, int K, int codebook, int m, int n,
                         const exl3_half *s_out, const exl3_half *scales, int M, const int8_t *q,
                         const float *qscale, exl3_half *y, void *workspace,
                         size_t workspace_bytes, exl3_stream_t stream);

/**
 * The int8-activation layer from binary16 activations: x-tilde =
 * binary16(Hb(s_in (.) x)) (x itself without s_in), quantized as by
 * exl3_quantize_act, then exl3_gemm_i8.  The result differs from exl3_gemm's
 * by the activation quantization (about 1% relative at batch 1 on Gaussian
 * activations).  Arguments as exl3_gemm_small, 1MAD or mul1 only.
 */
exl3_status exl3_gemm_int8act(const uint32_t *codes, int K, int codebook, int m, int n,
                              const exl3_half *s_in, const exl3_half *s_out,
                              const exl3_half *scales, int M, const exl3_half *x, exl3_half *y,
                              void *workspace, size_t workspace_bytes, exl3_stream_t stream);

/**
 * Kernel launches one exl3_gemm (or exl3_gemm_small / exl3_gemv, M <= 32)
 * call of this shape and batch makes on the current device under the current
 * exl3_set_path setting.  Up to 32 rows: on the decode-MMA kernel 1 at M <= 2
 * (input transform, layer and output transform in one launch) and 2 above
 * (operand image, layer kernel); on the warp-shuffle kernel 2 or 3 per batch
 * chunk (x pairs when the layer is split into sub-units, layer, output
 * transform).  Above 32 rows: 2 for the fused prefill, 3 for the decode-once
 * prefill (exl3_set_prefill); 3 per 128-row pass for the prefill passes.  0
 * for an invalid shape or M < 1.
 */
int exl3_gemm_launches(int m, int n, int M);

/** Most layers in one grouped call (exl3_gemm_grouped and its variants). */
#define EXL3_MAX_GROUP 64

/** One layer of a grouped call (the arguments of exl3_gemm_small that differ
 *  between layers; formats as above). */
typedef struct {
  const uint32_t *codes;   /* (m/16)*(n/16)*8K words */
  int m, n;                /* positive multiples of 128 */
  const exl3_half *s_in;   /* [n] or NULL */
  const exl3_half *s_out;  /* [m] or NULL */
  const exl3_half *scales; /* [m] */
  const exl3_half *x;      /* [M][n] */
  exl3_half *y;            /* [M][m] */
} exl3_layer;

/**
 * Bytes of scratch for exl3_gemm_grouped over `layers` at batch M: a status
 * word (first 256 bytes), then for every layer its per-row-block counters
 * and M*m fp32 row sums, then for every layer the larger of
 * min(M, 8)*n 32-bit x pairs and, for M > 2, the decode-MMA operand image
 * with its block sums (as for exl3_workspace_bytes); each region 256-byte
 * aligned.  Same zero-fill contract as exl3_workspace_bytes: the status word
 * is at byte 0.  Returns 0 for an invalid group.
 */
size_t exl3_group_workspace_bytes(const exl3_layer *layers, int count, int M);

/**
 * `count` (1..EXL3_MAX_GROUP) independent layers that share K, the codebook
 * and the batch M (1..EXL3_MAX_BATCH): the results equal `count` calls of
 * exl3_gemm_small, in fewer kernel launches.  The pages have no counterpart;
 * it serves decoders that apply several projections to the same step (q, k
 * and v; gate and up), and any set of independent layers of one K and code
 * (the experts of a mixture-of-experts layer, or the layers of several
 * sequences' steps), whose kernel chain it runs once for all of them.
 * `layers` is a host array read during the call.  No
 * layer may read another layer's output (x of one aliasing y of another) in the
 * same call.  On the warp-shuffle kernel the layers share one chain per batch
 * chunk (x pairs of every layer, one decode+GEMV kernel over the tiles of
 * every layer, one output kernel for every layer); on the decode-MMA kernel
 * one operand-image launch for every layer, then one layer kernel over the
 * tiles of every layer (at M <= 2, that one launch alone).  The workspace's per-layer
 * scratch is sized for either.
 */
exl3_status exl3_gemm_grouped(const exl3_layer *layers, int count, int K, int codebook, int M,
                              void *workspace, size_t workspace_bytes, exl3_stream_t stream);

/** One layer of a multi-code grouped call: a layer with its own K and code. */
typedef struct {
  exl3_layer layer;
  int K;        /* 1..8 */
  int codebook; /* EXL3_CB_* */
} exl3_layer_kc;

/**
 * Bytes of scratch for exl3_gemm_multi: exl3_group_workspace_bytes of the
 * same layers (the plain layers' shapes and M).  0 for an invalid group.
 */
size_t exl3_multi_workspace_bytes(const exl3_layer_kc *layers, int count, int M);

/**
 * `count` (1..EXL3_MAX_GROUP) independent layers of their own K and code at one
 * batch M (1..EXL3_MAX_BATCH): the results equal `count` calls of
 * exl3_gemm_small.  The pages have no counterpart; EXL3 models give each
 * tensor its own bit width ("EXL3 field guide"), so a decoder step's layers
 * differ in K.  On the warp-shuffle kernels (M <= 2 by default) the layers
 * share one kernel chain per batch chunk: one x-pair kernel over every layer,
 * one sub-unit kernel per (K, code) class over that class's layers (in order
 * of first appearance, each a programmatic dependent of the one before; in a
 * chunk of one row, one kernel for all the classes of one K when their tiles
 * give every SM at least 2048), one output kernel over every layer.  On the decode-MMA kernel each class runs
 * as exl3_gemm_grouped would run it.
 * Validation and errors as exl3_gemm_grouped, K and the code checked per
 * layer; workspace >= exl3_multi_workspace_bytes, same zero-fill contract.
 */
exl3_status exl3_gemm_multi(const exl3_layer_kc *layers, int count, int M, void *workspace,
                            size_t workspace_bytes, exl3_stream_t stream);

/**
 * Bytes of scratch for exl3_gemm_whole_grouped: exl3_group_workspace_bytes of
 * the same layers rounded up to 256 bytes (first, so the status word is at
 * byte 0), then max over the layers of max(m, n) halves of unit signs, then
 * per layer M*n halves of its transformed input and M*m halves of its output
 * before the last transform (each 256-byte aligned).  Same zero-fill
 * contract.  0 for an invalid group (count outside 1..EXL3_MAX_GROUP, M
 * outside 1..EXL3_MAX_BATCH, an m or n not a power of two in [128, 32768]).
 */
size_t exl3_gemm_whole_grouped_workspace_bytes(const exl3_layer *layers, int count, int M);

/**
 * `count` (1..EXL3_MAX_GROUP) independent layers with QTIP's whole-vector
 * rotations ("Trellis Quantization" Part eleven), sharing K, the codebook and
 * the batch M (1..EXL3_MAX_BATCH): the results equal `count` calls of
 * exl3_gemm_whole, in one chain -- one transform kernel across the
 * 128-blocks for every layer's input, exl3_gemm_grouped on the transformed
 * inputs, one transform kernel for every layer's output.  Layers as for
 * exl3_gemm_grouped (s_in / s_out NULL = no rotation on that side); m and n
 * powers of two in [128, 32768] (EXL3_ERR_SHAPE).  Other errors as
 * exl3_gemm_grouped (EXL3_ERR_BATCH for count or M out of range).
 */
exl3_status exl3_gemm_whole_grouped(const exl3_layer *layers, int count, int K, int codebook, int M,
                                    void *workspace, size_t workspace_bytes, exl3_stream_t stream);

/**
 * Workspace of exl3_gemm_int8act_grouped: a status word (first 256 bytes),
 * then per layer the regions of exl3_gemm_i8_workspace_bytes after its
 * counters (row sums, activation words, tile corrections, block factors).
 * Same zero-fill contract.  0 for an invalid group.
 */
size_t exl3_group_i8_workspace_bytes(const exl3_layer *layers, int count, int M);

/**
 * `count` (1..EXL3_MAX_GROUP) independent layers on int8 activations, as
 * `count` calls of exl3_gemm_int8act (same K, byte-sum code and batch
 * 1..EXL3_MAX_BATCH): one activation kernel for every layer's x, one layer
 * kernel over the tiles of every layer per batch chunk, one output kernel.
 * Validation and errors as exl3_gemm_grouped and exl3_gemm_int8act.
 */
exl3_status exl3_gemm_int8act_grouped(const exl3_layer *layers, int count, int K, int codebook,
                                      int M, void *workspace, size_t workspace_bytes,
                                      exl3_stream_t stream);

/**
 * Bytes of scratch for exl3_gemm_int8act_multi: exl3_group_i8_workspace_bytes
 * of the same layers.  0 for an invalid group.
 */
size_t exl3_multi_i8_workspace_bytes(const exl3_layer_kc *layers, int count, int M);

/**
 * `count` (1..EXL3_MAX_GROUP) independent layers on int8 activations, each
 * with its own K and byte-sum code (1MAD or mul1), at one batch M
 * (1..EXL3_MAX_BATCH): the results equal `count` calls of exl3_gemm_int8act.
 * One activation kernel for every layer's x (each layer's tile corrections
 * and block factors with its own code's centre and scale), per batch chunk one
 * int8 layer kernel per (K, code) class (in order of first appearance; in a
 * chunk of one row, one for both codes of one K when their tiles give every
 * SM at least 2048), one output kernel.  Validation and errors as exl3_gemm_int8act_grouped, K and the
 * code checked per layer; workspace >= exl3_multi_i8_workspace_bytes, same
 * zero-fill contract.
 */
exl3_status exl3_gemm_int8act_multi(const exl3_layer_kc *layers, int count, int M, void *workspace,
                                    size_t workspace_bytes, exl3_stream_t stream);

/** Kernel family used by exl3_gemv / exl3_gemm_small. */
typedef enum {
  EXL3_PATH_AUTO = 0,    /**< warp-shuffle kernel for M <= 2, decode-MMA kernel above */
  EXL3_PATH_SHUFFLE = 1, /**< decode + binary16 FMA per tile, fp32 across tiles, warp-shuffle reduction; any M */
  EXL3_PATH_TENSOR = 2   /**< decode-MMA: decoded tiles in TMEM feeding tcgen05 MMAs (fp32 accumulation); any M */
} exl3_path;

/** Prefill strategy of exl3_gemm above EXL3_MAX_BATCH rows. */
typedef enum {
  EXL3_PREFILL_AUTO = 0,        /**< fused up to 256 rows, decode-once above */
  EXL3_PREFILL_FUSED = 1,       /**< codes decoded into shared memory inside the GEMM, per batch tile */
  EXL3_PREFILL_DECODE_ONCE = 2  /**< the matrix decoded once per call into HBM, then a dense GEMM */
} exl3_prefill;

/**
 * Select the prefill strategy of subsequent exl3_gemm calls with M >
 * EXL3_MAX_BATCH (a process-wide setting, default EXL3_PREFILL_AUTO; ignored
 * while exl3_set_path(EXL3_PATH_TENSOR) selects 128-row passes).  Every
 * strategy computes the layer within the documented tolerance and uses the
 * workspace of exl3_gemm_workspace_bytes.  Returns EXL3_ERR_BATCH for an
 * unknown value.
 */
exl3_status exl3_set_prefill(int strategy);

/**
 * Select the kernel family for subsequent exl3_gemv / exl3_gemm_small calls
 * (a process-wide setting, default EXL3_PATH_AUTO).  Both families compute the
 * same layer within the documented tolerance.  Returns EXL3_ERR_BATCH for an
 * unknown value.
 */
exl3_status exl3_set_path(int path);

/**
 * Failure-detection test hook (no counterpart in the pages).  While `on` is
 * non-zero, the operand producers of the tensor-core kernel (operand B) and
 * of the dense prefill kernel (both operands) post nothing, so the bounded
 * device-side waits for the operands run out: every role of the kernel
 * stops, waits (bounded) for its copies in flight, frees its tensor memory,
 * and the kernel ORs 1 into the workspace status word (see
 * exl3_workspace_bytes) before it exits.  The call's outputs are then not
 * valid; later calls with the hook off are unaffected.  No GPU fault, trap or
 * unbounded wait is involved.  Process-wide, like exl3_set_path.
 */
exl3_status exl3_debug_stall_tensor_wait(int on);

/**
 * The one call that waits: reads the status word at device address
 * `status_word` once the work queued on `stream` so far has finished
 * (byte 4*(m/128) of an exl3_workspace_bytes / exl3_gemm_workspace_bytes /
 * exl3_gemm_whole_workspace_bytes workspace, byte 0 of a group's).  Returns
 * EXL3_OK if it is 0, EXL3_ERR_DEVICE_CHECK if a device-side wait of a
 * preceding call timed out (see exl3_debug_stall_tensor_wait), EXL3_ERR_NULL
 * for a NULL address, EXL3_ERR_CUDA if the copy or the synchronization
 * fails.  The word is left as it is.
 */
exl3_status exl3_device_status(const void *status_word, exl3_stream_t stream);

/** Size of the fixed device array that exl3_gemv_noalloc uses as scratch. */
#define EXL3_NOALLOC_SCRATCH_BYTES (4u << 20)

/**
 * exl3_gemv without a workspace argument, for callers that cannot allocate
 * device memory: code running where cudaMalloc is unavailable or not allowed
 * (host callbacks, allocator hooks, plugins whose host framework owns all
 * device memory, loops that must never allocate).  The source pages have no
 * counterpart; it computes exactly what exl3_gemv computes, with the same
 * arguments minus the workspace.
 *   - Scratch: a file-scope device array of EXL3_NOALLOC_SCRATCH_BYTES bytes,
 *     present on every GPU that loads the library until the process exits.
 *     A layer fits if a256(4*(m/128 + 1)) + a256(4*m) + a256(4*n) <=
 *     EXL3_NOALLOC_SCRATCH_BYTES, a256 rounding up to a multiple of 256 (the
 *     block counters and status word, m fp32 row sums, n 32-bit x pairs);
 *     a larger layer is rejected with EXL3_ERR_SCRATCH before anything is
 *     launched.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current.  `stream` must belong
 *     to the current device (EXL3_ERR_CUDA otherwise: the address is per
 *     device).  The call is not supported inside a stream capture (there it
 *     returns EXL3_ERR_CUDA).
 *   - Every call shares the one array and clears its counters and row sums
 *     with an asynchronous memset on `stream`.  Calls whose work can overlap on the
 *     GPU (other streams, other host threads) race: serialize them.
 *   - Allocates and frees nothing; asynchronous on `stream`.
 */
exl3_status exl3_gemv_noalloc(const uint32_t *codes, int K, int codebook, int m, int n,
                              const exl3_half *s_in, const exl3_half *s_out,
                              const exl3_half *scales, const exl3_half *x, exl3_half *y,
                              exl3_stream_t stream);

/**
 * Integer-throughput probe (a measurement aid; the pages have no counterpart):
 * launches `blocks` CTAs of 256 threads, each thread running 8 independent
 * dependency chains of 4*iters instructions of one kind -- 0 IMAD
 * (mad.lo.u32), 1 LOP3, 2 SHF (funnel shift), 3 IDP4A, 4 PRMT -- or an even
 * mix over the chains: 5 IMAD + LOP3, 6 IMAD + IDP4A + LOP3 + SHF.  The
 * caller times it on `stream`; it executes blocks * 8192 * iters
 * instructions.  The INT32 term of the layer roofline ("Trellis Quantization"
 * Part three counts the decode in integer instructions per weight) is checked
 * against it.  out: device array of blocks * 256 uint32 (the chains' results),
 * 16-byte aligned.  Errors: EXL3_ERR_BATCH (unknown kind), EXL3_ERR_SHAPE
 * (blocks or iters < 1), EXL3_ERR_NULL, EXL3_ERR_ALIGN, EXL3_ERR_CUDA.
 */
exl3_status exl3_probe_int(int kind, uint32_t *out, int blocks, int iters, exl3_stream_t stream);

/** Static, NUL-terminated description of a status code. */
const char *exl3_status_string(exl3_status status);

/** Static version string of the library. */
const char *exl3_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EXL3_H_ */
