/*
 * tl.h -- C ABI of the ternary projection linears for B300 (sm_103a).
 *
 * The operation (Neutrino-1 pages):
 *   every projection weight is one of {-1, 0, +1} (blog "Neutrino-1:
 *   quantization is a training decision", "What's actually ternary"), a
 *   linear multiplies the signed sum of its inputs by a scale ("state times
 *   scale", same section), there is one scale and one row sum per output row
 *   ("Neutrino-1 8B" model page, "Architecture": per-row metadata holds "row
 *   dimensions, scales, and row sums"), and the weights stay packed at rest
 *   and are decoded inside the matrix kernel (model page, "Overview").
 *
 *       y[n, m] = scale[m] * sum_k w[m, k] * x[n, k]
 *
 *   TL_MODE_BF16 (mode A): x is bf16, products are exact, sums are fp32.
 *   TL_MODE_I8   (mode B): x was quantised per token by tl_quantize_act into
 *       int8 q with step s[n] and zero point z[n]; acc = sum_k w*q is exact
 *       (int32) and y = ((float)(acc - z[n]*rowsum[m]) * s[n]) * scale[m].
 *   TL_MODE_I8_FUSED: mode B with the quantisation done inside the linear's
 *       own launch: x is bf16, and every token is quantised exactly as
 *       tl_quantize_act would (asymmetric, or symmetric with
 *       TL_FLAG_SYMMETRIC), so Y is bit for bit what tl_quantize_act
 *       followed by TL_MODE_I8 gives, with one launch instead of two.
 *
 * Batch sizes: 1 <= N <= 8 is the decode / speculative-verify path (one
 * token plus up to seven drafted ones verified "in one batched pass", wiki
 * "Neutrino-1", "What is actually new"); every token's result is bitwise
 * independent of N.  9 <= N < 256 runs as chunks of 8.  N >= 256 is the
 * prefill-sized dense contraction on the tensor cores (tcgen05).
 *
 * Conventions for every call:
 *   - The caller owns all buffers.  The library never allocates or frees
 *     device memory and keeps no state except cached device attributes.
 *   - "device" pointers are CUDA global memory of the current device; "host"
 *     pointers are ordinary process memory.
 *   - Device calls are asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  Argument errors are returned before anything
 *     is launched; a failed launch returns TL_ERR_CUDA.  Faults inside a
 *     kernel surface at the caller's next synchronisation.
 *   - Nothing aborts or throws across the ABI.
 *   - Row-major everywhere: X is [N][K], Y is [N][M].
 *
 * Packed weight format "TL2P v2" (the pages' own format is unpublished; this
 * is the library's own):
 *   W[M][K] is padded with zero weights to Mp = ceil(M/16)*16 rows and
 *   Kp = ceil(K/128)*128 columns and cut into 16 x 128 tiles of 512 bytes;
 *   tile (r, b) starts at byte (r * Kp/128 + b) * 512.  In a tile, lane
 *   L = 4g + t (g < 8, t < 4) owns the 16 bytes (4 little-endian words) at
 *   16L.  Weight (i, c) of the tile (row i < 16, column c < 128) has g = i%8,
 *   h = i/8, s = c/16, cc = c%16, u = cc/8, t = (cc%8)/2, e = cc%2; it lives
 *   in word j = 2u + h of lane 4g+t, in the 2-bit field starting at bit
 *   2s + 16e.  The field holds 1 - w as an unsigned number: 00 -> +1,
 *   01 -> 0, 10 -> -1; 11 is never written.  Padding fields hold 01, so a
 *   word of sixteen zero weights is 0x55555555.  Size:
 *   tl_packed_bytes(M, K) = Mp * Kp / 4 bytes.
 */
#ifndef TL_H
#define TL_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TL_API __attribute__((visibility("default")))
#else
#define TL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TL_OK = 0,
    TL_ERR_NULL = 1,        /* a required pointer is NULL */
    TL_ERR_SHAPE = 2,       /* M, K, N, G out of range */
    TL_ERR_ALIGN = 3,       /* packed not 16-byte aligned, or an element pointer misaligned */
    TL_ERR_BAD_VALUE = 4,   /* tl_pack: a weight outside {-1, 0, 1}; tl_validate: bad codes */
    TL_ERR_MODE = 5,        /* unknown mode / output type, or a combination that does not exist */
    TL_ERR_UNSUPPORTED = 6, /* layout tag not TL2P v2, or no device of compute capability 10.3 */
    TL_ERR_CUDA = 7,        /* a CUDA runtime call failed */
    TL_ERR_TIMEOUT = 8,     /* a bounded device-side wait gave up */
    TL_ERR_WORKSPACE = 9    /* workspace NULL or smaller than tl_workspace_bytes() */
} tl_status;

enum { TL_MODE_BF16 = 0, TL_MODE_I8 = 1, TL_MODE_I8_FUSED = 2 };
enum { TL_OUT_F32 = 0, TL_OUT_BF16 = 1, TL_OUT_I32_RAW = 2 };

/* tl_linear flags */
#define TL_FLAG_PDL 1u  /* launch with programmatic dependent launch: the kernel
                           may start, and begin streaming weights, before the
                           previous kernel on the stream has finished.  Only set
                           it when that previous kernel does not write this call's
                           weights, scales or row sums (it may write X). */
#define TL_FLAG_SYMMETRIC 2u /* TL_MODE_I8_FUSED: quantise symmetrically (as
                                tl_quantize_act with symmetric != 0); ignored in
                                the other modes */

#define TL_LAYOUT_TL2P_V2 2u
#define TL_MAX_GROUP 4
#define TL_MAX_K (1 << 20)
#define TL_MAX_M (1 << 24)

/* One packed ternary matrix, all pointers device memory owned by the caller. */
typedef struct {
    const uint32_t *packed; /* TL2P v2 words, tl_packed_bytes(M, K) bytes, 16-byte aligned */
    const float *scale;     /* [M] fp32 per-row scale */
    const int32_t *rowsum;  /* [M] int32 sum_k w[m,k]; required in mode B, ignored in mode A */
    int32_t M, K;           /* logical rows (outputs) and columns (inputs) */
    uint32_t layout;        /* TL_LAYOUT_TL2P_V2 */
} tl_weight;

/* Bytes of the TL2P v2 image of an M x K matrix (0 if M or K < 1). */
TL_API size_t tl_packed_bytes(int64_t M, int64_t K);

/* HOST.  Pack int8 W[M][K] (row-major, values in {-1, 0, 1}) into `packed`
 * (tl_packed_bytes(M, K) bytes, written completely, padding zero), compute
 * rowsum[m] = sum_k W[m][k] and copy scale_in[M] to scale_out[M] (either
 * scale pointer may be NULL to skip the copy).  Returns TL_ERR_BAD_VALUE,
 * and leaves the outputs unspecified, if any weight lies outside {-1, 0, 1}.
 * Cite: model page "Architecture" (per-row scales and row sums).  Uses all
 * host cores for large matrices. */
TL_API tl_status tl_pack(const int8_t *W, int64_t M, int64_t K, const float *scale_in,
                  uint32_t *packed, float *scale_out, int32_t *rowsum);

/* HOST.  Check a TL2P v2 image: *bad_codes receives the number of 11 fields
 * plus non-zero padding weights (NULL allowed).  TL_OK iff that is 0. */
TL_API tl_status tl_validate_packed(const uint32_t *packed, int64_t M, int64_t K,
                             int64_t *bad_codes);

/* Device workspace needed by tl_linear / tl_linear_group for these shapes
 * and this N (all matrices in Ws share K).  The workspace holds a status word,
 * per-row-tile arrival counters and exchange slots at its front, and split-K
 * partial sums (scratch) at its back, ending at the workspace's end.  It must
 * be zero-filled before its first use and 256-byte aligned; every call leaves
 * its front bytes zero again when it completes.  One workspace of the largest
 * size asked for by a set of calls may serve any sequence of those calls, of
 * any shapes, on one stream; calls that overlap on the GPU must not share it.
 * Device-side errors: the kernels cannot return a status, so a bounded wait
 * that gives up (about a second) writes a non-zero value into the
 * workspace's first int32 (the status word), and the call's outputs are then
 * invalid.  Read that word after the stream has passed the call; if it is
 * non-zero, treat the call as having failed with TL_ERR_TIMEOUT and zero-fill
 * the whole workspace before using it again. */
TL_API size_t tl_workspace_bytes(const tl_weight *Ws, int G, int N);

/* HOST.  The work split that tl_linear / tl_linear_group use for these
 * shapes at batch N (N <= 8 per launch) on a GPU with `sms` SMs; runs no GPU
 * code and needs no GPU.  It exists so that tests and tuning can check the
 * split against the kernel's invariants; the pages describe no such call.
 * plan[TL_PLAN_FIELDS] receives, in order: row tiles R, 128-column blocks KB,
 * K slices NS, slice width KW, last slice width KWL, CTAs per slice Pps,
 * CTAs P = NS * Pps, units per CTA Lc (last slice LcL), row tiles a CTA may
 * touch, warps per CTA, tiles per weight copy at this N, CTA slots per SM,
 * and the row-tile limit per CTA.  Unit u of slice s (u = r * kw + b for row
 * tile r, block b) belongs to CTA s * Pps + u / Lc (LcL in the last slice).
 * Returns TL_ERR_NULL, TL_ERR_SHAPE or TL_OK. */
#define TL_PLAN_FIELDS 14
TL_API tl_status tl_decode_plan(const tl_weight *Ws, int G, int N, int sms, int32_t *plan);

/* HOST.  The tensor-core kernel's plan for these shapes at batch N (used
 * from N = 256 on) on a GPU with `sms` SMs; runs no GPU code and needs no
 * GPU, for tests and tuning (the pages describe no such call).
 * plan[TL_PREFILL_PLAN_FIELDS] receives: tokens per tile BN (256 or 128),
 * K splits S, 128-column blocks per split KBS, output tiles (128 rows x BN
 * tokens, over the group), and CTAs launched (one per SM at most).  The
 * planner minimises rounds of items x blocks per split x the block time of
 * BN, plus a cost per extra split.  Returns TL_ERR_NULL, TL_ERR_SHAPE or
 * TL_OK. */
#define TL_PREFILL_PLAN_FIELDS 5
TL_API tl_status tl_prefill_plan(const tl_weight *Ws, int G, int N, int sms, int32_t *plan);

/* DEVICE.  Per-token activation quantisation (bf16 -> int8).  X_bf16 [N][K]
 * (2-byte aligned), Q [N][K] int8, s [N] fp32, z [N] int32.
 *   symmetric == 0: lo = min(0, min x), hi = max(0, max x),
 *       s = (hi - lo) / 255, z = -128 - rint(lo / s),
 *       q = clamp(rint(x / s) + z, -128, 127); an all-zero token gets s = 1,
 *       z = 0, q = 0.
 *   symmetric != 0: s = max|x| / 127 (1 if that is 0), z = 0,
 *       q = clamp(rint(x / s), -127, 127).
 * fp32 arithmetic with IEEE division and round-half-to-even.  The pages are
 * silent on activation quantisation; this is the library's reading. */
TL_API tl_status tl_quantize_act(const void *X_bf16, int N, int K, int8_t *Q, float *s,
                          int32_t *z, int symmetric, void *stream);

/* DEVICE.  Y = linear(W, X) for one matrix.
 *   mode TL_MODE_BF16: X is bf16 [N][K]; s, z ignored (may be NULL).
 *   mode TL_MODE_I8:   X is int8 [N][K] from tl_quantize_act; s, z [N] required;
 *                      W->rowsum required.
 *   mode TL_MODE_I8_FUSED: X is bf16 [N][K]; s, z ignored (may be NULL);
 *                      W->rowsum required.  Up to 255 tokens run on the
 *                      decode kernel (chunks of 8, each CTA reducing each
 *                      token's whole row for its step and zero point); from
 *                      256 tokens the quantiser writes the integers as bf16
 *                      into the workspace and the tensor-core kernel reads
 *                      them (two launches instead of three).
 *   out_dtype: TL_OUT_F32 (fp32 Y), TL_OUT_BF16 (bf16 Y, round to nearest
 *              even of the fp32 result), TL_OUT_I32_RAW (mode TL_MODE_I8
 *              only: the exact int32 acc = sum_k w*q, before any correction).
 *   workspace: device, >= tl_workspace_bytes(W, 1, N) bytes, 256-byte aligned.
 *   flags: 0, or TL_FLAG_PDL and / or TL_FLAG_SYMMETRIC.
 * Y must not alias X.  Deterministic: the same call gives the same bits. */
TL_API tl_status tl_linear(const tl_weight *W, const void *X, const float *s, const int32_t *z,
                    void *Y, int N, int mode, int out_dtype, void *workspace,
                    size_t workspace_bytes, unsigned flags, void *stream);

/* DEVICE.  G (1..TL_MAX_GROUP) matrices that read the same X (q/k/v, or
 * gate/up) in one launch; Ys[g] is [N][Ws[g].M].  Every Ws[g].K must be
 * equal.  Each Ys[g] equals what tl_linear(&Ws[g], ...) would write.
 * `Ws` and `Ys` are host arrays of G entries. */
TL_API tl_status tl_linear_group(const tl_weight *Ws, int G, const void *X, const float *s,
                          const int32_t *z, void *const *Ys, int N, int mode,
                          int out_dtype, void *workspace, size_t workspace_bytes,
                          unsigned flags, void *stream);

/* ---------------------------------------------------------------- block-wise scales
 * The blog ("Neutrino-1: quantization is a training decision", "What's
 * actually ternary") describes blocks of weights with one higher-precision
 * scale each, the codes being round(clamp(w / scale, -1, 1)) with scale the
 * block's mean |w|.  Here a block is TL_SCALE_BLOCK = 128 consecutive
 * columns of one row (the TL2P tile width; the pages give no size); the
 * last block of a row may be shorter. */
#define TL_SCALE_BLOCK 128

/* HOST.  Ternarise float W [M][K] by blocks: bscale[m][b] = mean of |W| over
 * the block's columns (taken in double, stored fp32), T[m][k] =
 * rint(clamp(W / bscale, -1, 1)) (in double, ties to even; 0 where the
 * block is all zero).  bscale has ceil(K / 128) entries per row.  Pack T
 * with tl_pack.  TL_ERR_BAD_VALUE for a non-finite weight. */
TL_API tl_status tl_ternarize_absmean(const float *W, int64_t M, int64_t K, int8_t *T,
                                      float *bscale);

/* DEVICE.  y[n][m] = sum_b bscale[m][b] * sum_{k in block b} w[m][k] * x[n][k]
 * on TL2P v2 codes (16-byte aligned), bscale fp32 [M][ceil(K/128)], X bf16
 * [N][K] (any N, run in chunks of 8), Y fp32 or bf16 [N][M].  fp32 sums
 * (bf16 products are exact).  Needs no workspace.  flags: 0 or TL_FLAG_PDL. */
TL_API tl_status tl_linear_blockscale(const uint32_t *packed, const float *bscale, int M, int K,
                                      const void *X, int N, void *Y, int out_dtype,
                                      unsigned flags, void *stream);

/* ---------------------------------------------------------------- int8 head and embedding
 * The projections are ternary, but the token embedding and the output head
 * stay int8 with one higher-precision scale per row (blog "Neutrino-1:
 * quantization is a training decision", "What's actually ternary"; model
 * page "Neutrino-1 8B", "Architecture": two untied int8 tensors of
 * vocabulary x hidden, one scale per row).  Greedy decoding reads the
 * head's argmax. */

/* Device workspace for tl_head_argmax (0 for invalid shapes). */
TL_API size_t tl_head_workspace_bytes(int64_t V, int D, int N);

/* DEVICE.  Output head with a fused argmax, on activations quantised per
 * token by tl_quantize_act (Q [N][D] int8, s, z [N]):
 *     acc[n,v]   = sum_d H[v,d] * Q[n,d]            (exact int32)
 *     logit[n,v] = ((float)(acc - z[n] * sum_d H[v,d]) * s[n]) * scale[v]
 *     token[n]   = the smallest v with the largest logit; best[n] = that logit.
 * H: int8 [V][D] row-major, 16-byte aligned; scale: fp32 [V].  Shapes:
 * 16 <= D <= 32768, D % 16 == 0, N * D <= 98304, 1 <= N <= 8, V < 2^31 - 1.
 * logits: fp32 [N][V] or NULL (then only token and best are written).
 * workspace: >= tl_head_workspace_bytes(V, D, N), 256-byte aligned,
 * zero-filled before first use; every call leaves its counter zero again.
 * flags: 0 or TL_FLAG_PDL (as for tl_linear). */
TL_API tl_status tl_head_argmax(const int8_t *H, const float *scale, int64_t V, int D,
                                const int8_t *Q, const float *s, const int32_t *z, int N,
                                float *logits, int32_t *token, float *best, void *workspace,
                                size_t workspace_bytes, unsigned flags, void *stream);

/* DEVICE.  Embedding lookup: X[n][d] = bf16(E[t][d] * scale[t]) for
 * t = tokens[n] (the fp32 product rounded to nearest even); E int8 [V][D],
 * scale fp32 [V], tokens int32 [N] (device), X bf16 [N][D].  A token outside
 * [0, V) gives a zero row. */
TL_API tl_status tl_embed(const int8_t *E, const float *scale, int64_t V, int D,
                          const int32_t *tokens, int N, void *X_bf16, void *stream);

/* ---------------------------------------------------------------- fused neighbours
 * Each decoder layer normalises its input with RMSNorm (eps 1e-6) before the
 * q/k/v and gate/up projections, and its feed-forward is SwiGLU ("Neutrino-1
 * 8B" model page, "Architecture").  These two calls produce a linear's input
 * in one pass: the op's bf16 output (Y, may be NULL when Q is given) and/or
 * that output quantised per token (Q int8 [N][K], s, z [N]; NULL to skip),
 * Q, s and z being bit for bit what tl_quantize_act(Y, symmetric) gives.
 * K <= 32768; a row runs on one CTA or, when long (SwiGLU beyond 1024
 * columns, RMSNorm beyond 8192), on a cluster of up to eight CTAs that
 * exchange their partial sums and ranges.  The pages fix neither the rounding
 * of these ops nor how their outputs are quantised; here the op is computed
 * in fp32 (IEEE division and square root; exp from the CUDA math library),
 * rounded once to bf16, and that bf16 row is quantised. */

/* DEVICE.  y[n,k] = bf16(x[n,k] * r[n] * gamma[k]),
 * r[n] = 1 / sqrt(sum_k x[n,k]^2 / K + eps); X bf16 [N][K], gamma bf16 [K]. */
TL_API tl_status tl_rmsnorm_quant(const void *X, const void *gamma, float eps, int N, int K,
                                  void *Y, int8_t *Q, float *s, int32_t *z, int symmetric,
                                  void *stream);

/* DEVICE.  h[n,m] = bf16(g / (1 + exp(-g)) * u) for the gate and up
 * projections' outputs G, U (bf16 [N][M]). */
TL_API tl_status tl_swiglu_quant(const void *G, const void *U, int N, int M, void *H,
                                 int8_t *Q, float *s, int32_t *z, int symmetric, void *stream);

/* ---------------------------------------------------------------- chains
 * A decoder runs its projections one after another, each reading what the
 * previous layer produced: per layer [q, k, v] -> o -> [gate, up] -> down
 * ("Neutrino-1 8B" model page, "Architecture": seven linears per layer, 36
 * layers), and single-stream decode is bound by the bytes it streams per
 * token (blog, "Serving it: the Neutrino Engine").  A chain runs such a
 * sequence of (grouped) linears in ONE persistent, cooperative launch: step
 * i reads its X only after every CTA has finished step i - 1 (so X may be
 * what step i - 1 wrote), while the weights of later steps keep streaming
 * into shared memory and L2 during that wait.  Each step computes exactly
 * what tl_linear_group computes for the same arguments (bit for bit: same
 * work split, same summation order).  In mode B the chain quantises each
 * step's bf16 X itself, per token and asymmetrically, exactly as
 * tl_quantize_act(symmetric = 0), into its workspace.
 *
 * Use: tl_chain_encode builds a host image (tl_chain_image_bytes bytes) that
 * names every pointer of the chain; the caller copies it to device memory
 * (16-byte aligned) once and calls tl_chain_run(host image, device image,
 * stream) for every pass.  The workspace (tl_chain_workspace_bytes,
 * 256-byte aligned, zero-filled before the first pass) belongs to that
 * chain: it holds the status word (its first int32), a count of completed
 * passes and per-step arrival counters that only grow from pass to pass,
 * split-K state that every pass leaves zero, and scratch.  Passes of one
 * chain must not overlap on the GPU.
 * Errors on the device: a wait for a step's inputs gives up after
 * wait_limit SM cycles (0: about a second) and writes a non-zero status
 * word; the other CTAs then stop too.  Read the word after the stream has
 * passed the run; if it is non-zero the outputs are invalid (treat it as
 * TL_ERR_TIMEOUT) and the workspace must be zero-filled again before the
 * next pass. */
#define TL_MAX_CHAIN 4096

typedef struct {
    const tl_weight *Ws;   /* host array of G matrices that read X (device pointers inside) */
    int G;                 /* 1..TL_MAX_GROUP; every Ws[g].K equal */
    const void *X;         /* device bf16 [N][K] (2-byte aligned; 16-byte for vector loads) */
    void *const *Ys;       /* host array of G device outputs [N][Ws[g].M], out_dtype */
} tl_chain_step;

/* Bytes of the image of a chain of nsteps linear steps (0 if out of range). */
TL_API size_t tl_chain_image_bytes(int nsteps, int mode);

/* Device workspace a chain needs (0 for invalid arguments). */
TL_API size_t tl_chain_workspace_bytes(const tl_chain_step *steps, int nsteps, int N, int mode);

/* HOST.  Encode a chain of nsteps steps at batch 1 <= N <= 8 into `image`
 * (host memory, >= tl_chain_image_bytes bytes).  mode, out_dtype as for
 * tl_linear (mode B: steps read bf16 X, which the chain quantises).
 * gate: NULL, or a device word that step 0 waits on (bounded) until it is
 * non-zero -- a producer outside the chain can hold the chain back with it.
 * wait_limit: SM cycles before a wait for inputs gives up (0: default).
 * Checks every argument, and that all of the launch's CTAs can be resident
 * at once (else TL_ERR_UNSUPPORTED); launches nothing. */
TL_API tl_status tl_chain_encode(const tl_chain_step *steps, int nsteps, int N, int mode,
                                 int out_dtype, const unsigned *gate, long long wait_limit,
                                 void *workspace, size_t workspace_bytes, void *image,
                                 size_t image_bytes);

/* DEVICE.  One pass of an encoded chain: `image` is the host image (read for
 * the launch shape), `image_device` its copy in device memory. */
TL_API tl_status tl_chain_run(const void *image, const void *image_device, void *stream);

/* Size of the library's fixed scratch array for tl_linear_noalloc (4 MiB):
 * enough for every 8B-shaped matrix at up to 8 tokens per chunk, and for
 * matrices of up to 32,496 rows at K <= 4096 (10,912 rows at K = 12288). */
#define TL_NOALLOC_SCRATCH_BYTES (4u << 20)

/* DEVICE.  tl_linear for callers that cannot allocate device memory.
 * The pages describe no such call; it exists for users of this library who
 * may not call cudaMalloc (or any allocating routine, torch's included) when
 * they run a linear -- code inside another runtime's memory pool, a loop
 * that must not allocate after start-up, or a host that only hands over
 * input and output buffers.  The caller still passes W, X, s, z and Y
 * exactly as for tl_linear; the split-K partial sums, arrival counters and
 * exchange slots that tl_linear keeps in the caller's workspace live instead in a
 * file-scope __device__ array of TL_NOALLOC_SCRATCH_BYTES bytes, which every
 * GPU that loads the library holds until the process exits.
 *   - Any N >= 1 runs on the decode / verify kernel in chunks of 8 tokens
 *     (never on the prefill kernel); results equal tl_linear's for N <= 255.
 *   - Shapes whose scratch would exceed TL_NOALLOC_SCRATCH_BYTES return
 *     TL_ERR_WORKSPACE before anything is launched.
 *   - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 *     routine.  Each call clears the array's status word, counters and slots with
 *     cudaMemsetAsync on `stream` before its launches.
 *   - Every call looks up the array's device address in the current context
 *     (cudaGetSymbolAddress, with that device current).  The first call in a
 *     context also loads the library's kernels there; make it before any
 *     stream capture.
 *   - All calls share the one array: calls that overlap on the GPU (other
 *     streams, other host threads) race and give wrong results; serialise
 *     them on one stream.
 *   - A bounded device-side wait that gives up (see tl_workspace_bytes)
 *     writes its status word into the library's array, which the caller
 *     cannot read, and the next call's clearing erases it: a timeout on this
 *     entry point is not reported.  Callers that must detect one use
 *     tl_linear with a workspace they own. */
TL_API tl_status tl_linear_noalloc(const tl_weight *W, const void *X, const float *s,
                                   const int32_t *z, void *Y, int N, int mode, int out_dtype,
                                   unsigned flags, void *stream);

/* Static, never NULL. */
TL_API const char *tl_status_string(tl_status status);

/* Library version, e.g. 100 for 0.1.0. */
TL_API int tl_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TL_H */
