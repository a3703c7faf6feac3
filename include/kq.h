/*
 * kq -- fused dequantize-and-multiply of block-quantized weights for GB300 (sm_103a).
 *
 * What the library computes (engine READMEs this library follows):
 *  - Kinetic README, "What makes it fast": on a personal computer a decode step is
 *    bound by memory bandwidth because a dense model reads all of its weights once
 *    per token; speculative decoding checks every guessed token in one pass over
 *    the weights; several users can share that pass. kq_gemv is that pass:
 *        Y[j][n] = sum_k deq(W)[n][k] * X[j][k],   j < M <= 16, n < N, k < K.
 *  - Same section, last paragraph: every row of a batch is summed in the same
 *    order as that token would be on its own. kq_gemv guarantees it: row j of Y
 *    has the same bits for every M in 1..16 and every slot position j.
 *  - Same section: long prompts run as tiled matrix products so that each weight
 *    block is unpacked once and used for many tokens. kq_gemm with M > 16 is that
 *    prefill product, on the tensor cores.
 *  - Same section: the next token is chosen from an output layer of up to a quarter of
 *    a million rows by bounding every row's score from a small copy and scoring exactly
 *    only the rows that can still win. kq_shortlist_build / kq_head_argmax are that head.
 *  - Kinetic README, "Switching from llama.cpp": GGUF files work unchanged, so
 *    Q8_0 and Q4_K blocks use GGUF's byte layouts. Kipp README, "How fast": its
 *    4-bit scheme is affine (scale + bias) with groups of 32 (layout below).
 *
 * Conventions: W is N x K, row-major, the blocks of one row contiguous along K
 * (GGUF order). X is M x K row-major (fp32 or bf16). Y is M x N fp32 row-major and
 * is overwritten, never accumulated. All pointers are DEVICE pointers unless a
 * function says otherwise. The caller owns every buffer; the library allocates
 * nothing per call. Its only state: a thread-local error string, per-device caches of
 * the SM count and of kernel attributes, the device error words read by
 * kq_device_errors(), and the fixed scratch array of kq_decode_step_static.
 * Every call is asynchronous on `stream` (a cudaStream_t passed as void*, NULL =
 * the legacy default stream) and never synchronises. There is no CPU fallback:
 * a call either launches the sm_103a kernels or returns an error.
 */
#ifndef KQ_H
#define KQ_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Block formats.
 * KQ_Q8_0        34 bytes / 32 weights: fp16 d, int8 q[32];            w = d*q
 * KQ_Q4_K       144 bytes / 256 weights: fp16 d, fp16 dmin, scales[12] (eight 6-bit
 *                scales sc_j and mins m_j, GGUF packing), qs[128] (byte 32c+l holds
 *                weight 64c+l in its low nibble and 64c+32+l in its high nibble);
 *                w = d*sc_j*q - dmin*m_j for sub-block j = weight/32
 * KQ_AFFINE4_G32 20 bytes / 32 weights: fp16 s, fp16 b, codes[16] (weight 2i in the
 *                low nibble of byte i, weight 2i+1 in the high nibble); w = s*q + b
 * KQ_Q5_K       176 bytes / 256 weights: Q4_K's d, dmin and scales[12], then qh[32],
 *                then Q4_K's qs[128] holding the low four code bits; the fifth bit of
 *                weight 64c+32h+l (c = 0..3, h = 0/1, l = 0..31) is bit 2c+h of qh[l];
 *                codes 0..31, w = d*sc_j*q - dmin*m_j (GGUF's Q5_K; the next k-quant
 *                that Q4_K_M model files mix in)
 * KQ_Q6_K       210 bytes / 256 weights: ql[128], qh[64], int8 scales[16], fp16 d (GGUF's
 *                Q6_K); weight 128n+32k+l takes its low 4 code bits from ql[64n+32(k%2)+l]
 *                (low nibble for k < 2, else high) and its top 2 from bits 2k..2k+1 of
 *                qh[32n+l]; w = d*scales[i/16]*(q - 32). Rows are only 2-byte aligned, so
 *                Q6_K runs on CUDA cores for both activation types. */
enum kq_fmt { KQ_Q8_0 = 1, KQ_Q4_K = 2, KQ_AFFINE4_G32 = 3, KQ_Q5_K = 4, KQ_Q6_K = 5 };

/* Activation element types. */
enum kq_dtype { KQ_F32 = 1, KQ_BF16 = 2 };

/* Status codes: 0 on success, negative on failure (text in kq_last_error()). */
enum kq_status {
  KQ_OK = 0,
  KQ_ERR_ARG = -1,         /* null pointer, size out of range, misaligned pointer */
  KQ_ERR_UNSUPPORTED = -2, /* unknown format or dtype, or a pair with no kernel */
  KQ_ERR_WORKSPACE = -3,   /* workspace missing or smaller than kq_gemm_workspace_size */
  KQ_ERR_CUDA = -4,        /* a CUDA launch or runtime call failed */
  KQ_ERR_TIMEOUT = -5      /* a bounded device-side wait gave up */
};

/* Bytes and weights per block of `fmt`; 0 for an unknown format. */
size_t kq_block_bytes(int fmt);
size_t kq_block_weights(int fmt);
/* Bytes of one row of K weights; 0 if fmt is unknown or K is not a multiple of the
 * block's weight count. */
size_t kq_row_bytes(int fmt, int K);

/* Message for the last failing call on this host thread ("" after a success). The
 * pointer stays valid until the next kq_* call on the same thread. */
const char* kq_last_error(void);
const char* kq_version(void);

/* Reads and clears the device error word of the current device; synchronises the device.
 * Every wait inside a kernel is bounded: if one gives up, the kernel records bit 0 here,
 * skips the rest of its work (its output is then invalid) and returns instead of hanging.
 * Returns the bits (0 = nothing recorded) or KQ_ERR_CUDA if the word cannot be read. */
int kq_device_errors(void);

/* Quantized GEMV / speculative-verify product (Kinetic README, "What makes it fast").
 *   fmt       KQ_Q8_0, KQ_Q4_K, KQ_AFFINE4_G32, KQ_Q5_K or KQ_Q6_K
 *   w_blocks  N * kq_row_bytes(fmt, K) bytes, 16-byte aligned
 *   x_dtype   KQ_BF16 (tensor-core path) or KQ_F32 (CUDA-core path)
 *   x         M x K activations, 16-byte aligned
 *   y         M x N fp32 output (overwritten), 8-byte aligned
 *   M         1..16 token rows; 0 returns KQ_OK without launching
 *   N         output rows, >= 0 (0 is a no-op)
 *   K         inputs per row, >= 0, a multiple of 256 (keeps every format's rows
 *             16-byte aligned for vector loads); K == 0 writes zeros
 * Row j of Y is bit-identical for every M and every position j (the kernel and its
 * work split are chosen from (fmt, x_dtype, N, K) only; M masks loads and stores).
 * Memory: w_blocks must be device memory (the weights are read by tensor copies); x and y
 * may be device memory or pinned host memory that the device can address (cudaHostAlloc /
 * cudaMallocHost under unified addressing): the kernels then read x and write y there over
 * the host link, with the same results, and need no copy before or after the call.
 * Errors: KQ_ERR_ARG, KQ_ERR_UNSUPPORTED, KQ_ERR_CUDA. */
int kq_gemv(int fmt, const void* w_blocks, int x_dtype, const void* x, float* y, int M, int N,
            int K, void* stream);

/* Flags of kq_gemv_ex. */
enum kq_flags {
  /* The kernel launched just before this call on `stream` does not write w_blocks (for
   * example the previous layer's GEMV). The GEMV may then start streaming its weights
   * before that kernel finishes (programmatic dependent launch); it still waits for it
   * before reading x or writing y. Both the tensor-core path (KQ_BF16) and the CUDA-core
   * path (KQ_F32) use it; the latter loads its first 256-weight unit before the wait. */
  KQ_OVERLAP_PREVIOUS = 1u
};

/* kq_gemv with flags (0 gives exactly kq_gemv). Unknown flag bits: KQ_ERR_ARG. Results are
 * identical with and without KQ_OVERLAP_PREVIOUS. */
int kq_gemv_ex(int fmt, const void* w_blocks, int x_dtype, const void* x, float* y, int M, int N,
               int K, unsigned flags, void* stream);

/* Quantized GEMM (Kinetic README, "What makes it fast": long prompts as tiled matrix
 * products, each weight block unpacked once for many tokens; a speculative check runs
 * all of its guesses through one pass over the weights).
 *   M <= 16: identical to kq_gemv (same kernels, same bits); the workspace is unused.
 *   16 < M <= 32 with Q4_K x bf16, and every M > 16 for the other format / dtype pairs:
 *            kq_gemv in passes of 16 token rows (rows c..c+15 in pass c/16, each pass
 *            reading W once), so every row of Y has exactly the bits kq_gemv gives it and
 *            the bit-identity across M holds for every M; the workspace is unused.
 *            (Batched verify of up to 32 guesses: below a few hundred rows the tensor-core
 *            product's time is set by unpacking W, and two passes are faster at M = 32.)
 *   M  > 32 with fmt = KQ_Q4_K, x_dtype = KQ_BF16: tensor-core (tcgen05) product. Every
 *            product the tensor cores form is exact: X
 *            goes to fp16 under an exact power-of-two scale per token; the weights enter
 *            as the integers sc*q with d applied per super-block in fp32 afterwards; the
 *            min term is a product of fp16 hi/lo splits of the sub-block sums of X and
 *            of dmin*m. The result differs from the exact fp64 value by fp32 rounding
 *            only (about 1e-6 of sum_k |w*x|). Not bit-identical to kq_gemv. Limits:
 *            64*dmin*m must be below 65504 (the fp16 range) for every sub-block.
 *   workspace/ws_bytes: device scratch of at least kq_gemm_workspace_size() bytes
 *            (tensor-core route: about M*(K + 3K/32)*2 + N*(3K/32)*2 bytes; otherwise 0),
 *            256-byte aligned, owned by the caller; may be NULL when that size is 0.
 * Other arguments as kq_gemv. Errors: as kq_gemv, plus KQ_ERR_WORKSPACE. */
int kq_gemm(int fmt, const void* w_blocks, int x_dtype, const void* x, float* y, int M, int N,
            int K, void* workspace, size_t ws_bytes, void* stream);
size_t kq_gemm_workspace_size(int fmt, int x_dtype, int M, int N, int K);

/* Quantize an N x K fp32 matrix (device memory) into N rows of blocks of `fmt`, on the
 * GPU, in fp64 arithmetic, with the same covering scheme in every call:
 *   Q8_0:    d = fp16_rn(max|w|/127), q = clamp(round_half_away(w/d), -127, 127)
 *   Q4_K:    per sub-block lo = min(0, min w), hi = max(0, max w);
 *            dmin = smallest fp16 >= max(-lo)/63, m_j = ceil(-lo_j/dmin);
 *            t_j = hi_j + dmin*m_j, d = smallest fp16 >= max(t)/945,
 *            sc_j = ceil(t_j/(15 d)), q = round_half_away((w + dmin*m_j)/(d*sc_j))
 *   Q5_K:    as Q4_K with 31 levels: d = smallest fp16 >= max(t)/1953,
 *            sc_j = ceil(t_j/(31 d)), q = round_half_away((w + dmin*m_j)/(d*sc_j)) in 0..31
 *   Q6_K:    per 16-weight sub-block a = max|w|, d = smallest fp16 >= max(a)/3937,
 *            sc = ceil(a/(31 d)), q = 32 + round_half_away(w/(d*sc)) in 1..63
 *   AFFINE4: b = largest fp16 <= min w, s = smallest fp16 >= (max w - b)/15,
 *            q = clamp(round_half_away((w - b)/s), 0, 15)
 * These make data for tests and benchmarks (the GEMV never quantizes). K must be a
 * multiple of the block's weight count; w 4-byte aligned, w_blocks 2-byte aligned.
 * Errors: KQ_ERR_ARG, KQ_ERR_CUDA. */
int kq_quantize(int fmt, const float* w, void* w_blocks, int N, int K, void* stream);

/* ---- Decode attention of a verify window over a KV cache ----
 * A speculative step checks its guesses in one pass (Kinetic README, "What makes it fast";
 * Kapitsa README verifies a tree of guesses at once): window token i (0..M-1, at position
 * L+i) attends to the cached positions 0..L-1 and to window positions L+j with j <= i, or,
 * with a tree mask, those with bit j of mask[i] set. Query head hq reads kv head
 * hq / (n_q / n_kv).
 *   q        M x (n_q*head_dim) fp32 (device, 16-byte aligned); rounded to bf16 (nearest
 *            even) before the products, as every activation between ops is bf16
 *   k_cache, v_cache  (L+M) x (n_kv*head_dim) bf16 rows (device, 16-byte aligned); rows
 *            L..L+M-1 hold the window's own keys and values (the caller appends them)
 *   o        M x (n_q*head_dim) fp32 (device, overwritten)
 *   M        1..32; L in 0..65000; head_dim 64 or 128; (n_q / n_kv) * M <= 128
 *   mask     NULL (causal within the window) or M words in device memory
 *   scale    multiplies q.k (usually 1/sqrt(head_dim))
 *   o = sum_p softmax_p(scale q.k_p) v_p over the visible positions (zeros if none).
 * Scores and sums are fp32 (products of bf16 on the tensor cores, the softmax weights
 * carried as bf16 hi + lo pairs), so o is within about 1e-5 of sum_p w_p |v_p| of the exact
 * value. Positions 0..L+M-1 are cut into chunks of 128 by absolute position and added in a
 * fixed order, and positions a token may not see add exact zeros: a token's output is
 * bit-identical for every M and every position in the batch (given its own mask row), and
 * (causal) equals the output of the same token alone at cache length L + i with the window's
 * earlier rows cached -- verifying guesses gives the bits plain decoding gives. Both
 * guarantees need finite keys and values: every row of a chunk enters its P V product, a
 * position the token may not see with weight 0, and 0 * Inf is NaN.
 * workspace: kq_attention_workspace_size() bytes, 256-byte aligned.
 * Errors: KQ_ERR_ARG, KQ_ERR_WORKSPACE, KQ_ERR_CUDA. */
size_t kq_attention_workspace_size(int M, int L, int n_q, int n_kv, int head_dim);
int kq_attention(const float* q, const void* k_cache, const void* v_cache, float* o, int M, int L, int n_q,
                 int n_kv, int head_dim, const unsigned int* mask, float scale, void* workspace, size_t ws_bytes,
                 void* stream);

/* ---- Shortlist output head: the greedy next token ----
 * Kinetic README, "What makes it fast" (choosing the next token): the output layer, up to a
 * quarter of a million rows, is read for every token; each row's score is first bounded
 * from a small copy, and exact scores are computed only for the rows that can still win.
 *
 * kq_shortlist_build makes the small copy of a Q8_0 head W (N x K, rows of blocks as for
 * kq_gemv) once, at load time, into one caller-owned buffer of kq_shortlist_bytes(N, K)
 * bytes (256-byte aligned):
 *   bytes [0, S)        N rows of K/256 Q4_K blocks (144 bytes): each 256-weight super-block
 *                       of deq(W) through the Q4_K quantizer of kq_quantize; S is that size
 *                       rounded up to a multiple of 256;
 *   bytes [S, S + 4N)   B_n (fp32): ||w_n - w'_n||_2 + K 2^-22 (||w_n||_2 + A_n), rounded up,
 *                       with A_n = sqrt(32 sum_g (15 d sc_g + dmin m_g)^2) over the row's
 *                       32-weight sub-blocks g.
 * For any x, |x.w_n - x.w'_n| <= B_n ||x||_2 (Cauchy-Schwarz), and the second term covers
 * the fp32 rounding of both the exact and the small-copy products.
 *
 * kq_head_argmax gives, for each of M (1..16) hidden states x_j, the row with the largest
 * exact score (ties: the lowest row) and that score. A row is scored exactly only if its
 * small-copy score plus B_n ||x_j|| reaches the largest small-copy score minus bound of
 * some token (bounds evaluated with directed rounding), so the row that wins is never
 * skipped. The exact score of row n is an fp32 sum in a fixed order (one warp per row: lane
 * l takes blocks l, l+32, ..., each a sequential FMA chain promoted by d; a fixed butterfly
 * across lanes). It does not depend on M, on the shortlist or on the other rows scored, so
 * the result equals the result with KQ_HEAD_ALL_ROWS (every row scored exactly, no
 * small-copy pass; shortlist may then be NULL). It can differ from the argmax of kq_gemv's
 * output only between rows whose scores lie within fp32 rounding of each other.
 *   w_q8        the Q8_0 head (device, 16-byte aligned); N >= 1; K a multiple of 256
 *   shortlist   from kq_shortlist_build for this head
 *   x           M x K, fp32 or bf16 (x_dtype), device, 16-byte aligned
 *   token       M int32 (device): the winning row (a row whose score is NaN never wins), or
 *               -1 if no row has a comparable (non-NaN) score
 *   score       M fp32 (device): its exact score
 *   rows_scored NULL or one uint32 (device): the number of rows scored exactly
 *   workspace   kq_head_argmax_workspace_size(M, N) bytes, 256-byte aligned
 * Three launches on `stream` (the small-copy GEMV, the bounds, the exact scores), no
 * synchronisation, no allocation. Errors: KQ_ERR_ARG, KQ_ERR_WORKSPACE, KQ_ERR_CUDA. */
enum { KQ_HEAD_ALL_ROWS = 1u };
size_t kq_shortlist_bytes(int N, int K);
int kq_shortlist_build(const void* w_q8, int N, int K, void* shortlist, size_t bytes, void* stream);
size_t kq_head_argmax_workspace_size(int M, int N);
int kq_head_argmax(const void* w_q8, const void* shortlist, int x_dtype, const void* x, int M, int N, int K,
                   int* token, float* score, unsigned int* rows_scored, void* workspace, size_t ws_bytes,
                   unsigned flags, void* stream);

/* ---- Decode step (composition of the GEMVs; Kinetic README, "What makes it fast": a
 * decode step is hundreds of small kernels replayed with one launch per token, and a
 * dense model reads all of its weights once per token). ----
 * Per layer: x = RMSNorm(h); [q k v] = x Wqkv^T; attention stand-in: each token attends
 * only to itself (a context of one), so query head hq outputs v of kv head
 * hq / (q_dim/kv_dim); h += o Wo^T with o that expanded v; x = RMSNorm(h);
 * [g u] = x Wgu^T; h += (silu(g) * u) Wd^T. Then logits = RMSNorm(h) Whead^T.
 * RMSNorm has unit weight: x = h / sqrt(mean(h^2) + rms_eps). Every GEMV input is rounded
 * to bf16 (nearest even); h and every GEMV output are fp32. Rows are independent, so a
 * token's logits are bit-identical for every M.
 * Weight matrices (device memory, rows of blocks as for kq_gemv):
 *   w_qkv[l]     (q_dim + 2*kv_dim) x hidden   rows q, then k, then v
 *   w_o[l]       hidden x q_dim
 *   w_gate_up[l] (2*ffn) x hidden              rows gate, then up
 *   w_down[l]    hidden x ffn
 *   w_head       vocab x hidden
 * The struct and the four pointer arrays live in HOST memory; the pointers in them are
 * device pointers. hidden, q_dim and ffn are multiples of 256. */
typedef struct kq_decode_model {
  int n_layers, hidden, q_dim, kv_dim, head_dim, ffn, vocab;
  int layer_fmt; /* format of every layer matrix */
  int head_fmt;  /* format of w_head */
  float rms_eps;
  const void* const* w_qkv;
  const void* const* w_o;
  const void* const* w_gate_up;
  const void* const* w_down;
  const void* w_head;
} kq_decode_model;

/* Device workspace bytes kq_decode_step needs for M tokens (0 on invalid arguments). */
size_t kq_decode_workspace_size(const kq_decode_model* model, int M);

/* One decode step for M (1..16) token rows: x = M x hidden bf16 (device), logits =
 * M x vocab fp32 (device, overwritten). workspace: >= kq_decode_workspace_size bytes of
 * device memory, 256-byte aligned, owned by the caller (the library allocates nothing).
 * Asynchronous on stream; can be captured in a CUDA graph. Errors: KQ_ERR_ARG,
 * KQ_ERR_UNSUPPORTED, KQ_ERR_WORKSPACE, KQ_ERR_CUDA. */
int kq_decode_step(const kq_decode_model* model, const void* x, float* logits, int M, void* workspace,
                   size_t ws_bytes, void* stream);

/* The decode step with a trace: the same launches as kq_decode_step, with a device-to-device
 * copy of every op's output into `trace` after the op, so that each op can be checked on its
 * own inputs (a test gives the oracle the GPU's input of every GEMV, RMSNorm and SwiGLU).
 * trace: kq_decode_trace_size(model, M) bytes of device memory, 256-byte aligned, owned by
 * the caller. Layout (every field starts on a 256-byte boundary, rows of M tokens):
 *   h0 (M x hidden fp32: the input as the residual stream), x0 (M x hidden bf16: its RMSNorm,
 *   the first qkv GEMV's input); then per layer, in order: qkv (M x (q_dim + 2 kv_dim) fp32),
 *   o_in (M x q_dim bf16: the Wo GEMV's input), y_o (M x hidden fp32), h_mid (fp32: h after
 *   the attention block), x_mid (bf16: its RMSNorm), gu (M x 2 ffn fp32), act (M x ffn bf16),
 *   y_d (M x hidden fp32), h_out (fp32), x_out (bf16: the next GEMV's input, the head's after
 *   the last layer). The logits are bit-identical to kq_decode_step's.
 * Errors: as kq_decode_step; KQ_ERR_ARG for a NULL, short or misaligned trace. */
size_t kq_decode_trace_size(const kq_decode_model* model, int M);
int kq_decode_step_trace(const kq_decode_model* model, const void* x, float* logits, int M, void* workspace,
                         size_t ws_bytes, void* trace, size_t trace_bytes, void* stream);

/* ---- Decode step with attention over a KV cache (a true speculative step) ----
 * kq_decode_step with its attention stand-in replaced by kq_attention's attention: per layer
 * the window's k and v (rounded to bf16) are written to rows L..L+M-1 of the layer's cache,
 * q = the first q_dim columns of [q k v], scale = 1/sqrt(head_dim) (as a float), token i sees
 * the L cached rows and window rows j <= i (or bit j of mask[i]); the attention output is
 * rounded to bf16 as it feeds Wo. A speculative decoder verifies M guesses in one step and
 * then advances `length` by the guesses it accepts (the rows after them are rewritten by the
 * next step). Model limits as kq_decode_step, plus head_dim 64 or 128 and
 * (q_dim / kv_dim) * M <= 128. */
typedef struct kq_kv_cache {
  void* const* k;  /* per layer: capacity rows of kv_dim bf16 (device, 16-byte aligned) */
  void* const* v;
  int length;      /* L: rows 0..L-1 hold the context (0..65000) */
  int capacity;    /* rows per layer array: L + M <= capacity */
} kq_kv_cache;
/* Device workspace bytes kq_decode_step_attn needs (0 on invalid arguments). */
size_t kq_decode_attn_workspace_size(const kq_decode_model* model, int M, int L);
/* x, logits, workspace as kq_decode_step; cache: HOST struct and pointer arrays of device
 * pointers; mask: NULL (causal) or M words of device memory. */
int kq_decode_step_attn(const kq_decode_model* model, const kq_kv_cache* cache, const void* x, float* logits,
                        int M, const unsigned int* mask, void* workspace, size_t ws_bytes, void* stream);

/* ---- Decode step that allocates nothing (no counterpart in the engine pages) ----
 * kq_decode_step needs a device workspace from its caller. Some callers cannot call
 * cudaMalloc or any allocating routine: code that only borrows a GPU from a host framework
 * that owns every device allocation, code on a latency-critical path where an allocation
 * could synchronise the device, or code that must not allocate while a stream is being
 * captured. kq_decode_step_static runs the same step with scratch memory that the library
 * holds in a fixed device array of KQ_DECODE_STATIC_SCRATCH_BYTES (4 MiB): every GPU that
 * loads the library keeps that array until the process exits, and nothing is allocated
 * per call (no cudaMalloc, no allocating library routine).
 *  - The caller still passes x and logits (device memory), as for kq_decode_step.
 *  - Models whose kq_decode_workspace_size(model, M) exceeds the array are rejected with
 *    KQ_ERR_WORKSPACE and a message giving both sizes.
 *  - The first call on a device looks up the array's device address (with that device
 *    current) and caches it with the device's current context; make that first call
 *    before capturing any stream. A call that finds another context current (the old
 *    one was destroyed, e.g. by cudaDeviceReset) looks the address up again.
 *  - Every call on a device shares the one array and leaves the last step's intermediate
 *    values in it; the step writes each value before reading it, so nothing needs
 *    clearing. Two calls that run at the same time on one device (for example on two
 *    streams) race on the array: serialise them.
 * Other arguments, results and errors as kq_decode_step. */
#define KQ_DECODE_STATIC_SCRATCH_BYTES (4u << 20)
int kq_decode_step_static(const kq_decode_model* model, const void* x, float* logits, int M, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KQ_H */
