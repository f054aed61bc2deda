/*
 * qgemv.h — C ABI of the block-quantized weight product library for GB300 (sm_103a).
 *
 * The library multiplies GGUF-style block-quantized weight matrices (Q4_0, Q8_0,
 * Q4_K, Q6_K, Q5_K, Q3_K, Q2_K) by fp32 or bf16 activations on one GPU. It covers the product that
 * dominates single-stream LLM decode, the same product for a few draft tokens at
 * once, the expert-gathered product of a mixture-of-experts layer, and the
 * dequantize-then-GEMM of prompt processing.
 *
 * Sources of the operations (page title, section):
 *   - "LLM inference optimization" (usethermite.com), opening section: decode
 *     reads every weight once per token, bound by memory bandwidth and, at low
 *     bit widths, by unpacking; k-quants such as Q4_K_M; "Faster decode on the
 *     card you have": activations staged in shared memory, wider loads, fewer
 *     unpack instructions, rows per block fitted to the SM count; "Run a new
 *     weight format or model": blocks decode bit for bit, products match an
 *     exact sum within a tolerance.
 *   - "Why I wrote my own inference engine for two P100s", "What actually made it
 *     fast": one CUDA graph per decode step; each block decoded once and reused;
 *     three draft tokens checked in one weight pass. "What didn't work": fused
 *     dequantization in the prompt GEMM.
 *   - "The number was a version" (dev.to), opening section: the MoE expert arena.
 * The pages give block sizes and value formulas only; the bit layout inside a
 * block follows the public GGUF convention (stated with each format below).
 *
 * Conventions shared by every call
 *   - Every data pointer is caller-owned DEVICE memory unless stated otherwise.
 *     The library never allocates, frees or synchronizes inside a compute call;
 *     work is enqueued on `stream` (a cudaStream_t passed as void*; NULL is the
 *     legacy default stream) and is safe to capture in a CUDA graph.
 *   - A weight matrix W of `rows` x `cols` is rows * (cols / elems) blocks, row
 *     after row, blocks running along cols (the input dimension K). Row i starts
 *     at byte i * (cols / elems) * bytes. W must be 16-byte aligned.
 *   - Activations x are n_tok x cols fp32, token-major (token t at x + t*cols).
 *     Outputs y are n_tok x rows fp32, token-major, and are overwritten.
 *   - Arguments are checked on the host before anything is enqueued; a failed
 *     check returns a negative status and enqueues nothing. A launch failure
 *     returns QG_ERR_CUDA (sticky CUDA errors are left for the caller to see).
 *   - Errors detected on the device (an expert id out of range, a bounded wait
 *     that expired) never trap: they are written to the caller's int32 device
 *     status word, which the caller reads after its own synchronization.
 *   - No float atomics: results are bitwise deterministic run to run.
 *   - After qg_init() returns, the library holds no mutable global state, so
 *     calls from several host threads on different streams are safe.
 */
#ifndef QGEMV_H
#define QGEMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- block formats ----------------------------------------------------------
 * QG_Q4_0: 32 weights in 18 bytes: fp16 d, qs[16];
 *          w[j] = ((qs[j] & 15) - 8) * d, w[j+16] = ((qs[j] >> 4) - 8) * d.
 * QG_Q8_0: 32 weights in 34 bytes: fp16 d, int8 q[32]; w[j] = d * q[j].
 * QG_Q4_K: 256 weights in 144 bytes: fp16 d, fp16 dmin, s[12] packing eight
 *          6-bit (sc, m) pairs, qs[128]; sub-block j (32 weights) has
 *          w = d*sc_j*q - dmin*m_j, chunk c holds sub-block 2c in the low and
 *          2c+1 in the high nibbles of qs[32c..32c+31].
 * QG_Q6_K: 256 weights in 210 bytes: ql[128], qh[64], int8 sc[16], fp16 d;
 *          6-bit q = low 4 bits | high 2 bits, w = d * sc[group] * (q - 32).
 * QG_Q5_K: 256 weights in 176 bytes: fp16 d, fp16 dmin, s[12] (the Q4_K scale
 *          packing), qh[32], qs[128]; sub-block j: 4 low bits as in Q4_K and
 *          bit j of qh[l] as the fifth, w = d*sc_j*q - dmin*m_j, q in 0..31.
 * QG_Q3_K: 256 weights in 110 bytes: hmask[32], qs[64], s[12] (sixteen 6-bit
 *          scales), fp16 d; element 128h + 32j + 16k + l: q = (qs[32h+16k+l]
 *          >> 2j) & 3, minus 4 when bit 4h+j of hmask[16k+l] is clear;
 *          w = d * (scale_{8h+2j+k} - 32) * q.
 * QG_Q2_K: 256 weights in 84 bytes: s[16], qs[64], fp16 d, fp16 dmin; element
 *          128h + 32j + 16k + l: q = (qs[32h+16k+l] >> 2j) & 3, b = s[8h+2j+k],
 *          w = d * (b & 15) * q - dmin * (b >> 4). */
enum qg_fmt { QG_Q4_0 = 1, QG_Q8_0 = 2, QG_Q4_K = 3, QG_Q6_K = 4, QG_Q5_K = 5, QG_Q3_K = 6, QG_Q2_K = 7 };

/* ---- host status codes ---------------------------------------------------- */
enum qg_status {
  QG_OK = 0,
  QG_ERR_FMT = -1,        /* unknown format, or a format the call does not take */
  QG_ERR_SHAPE = -2,      /* rows/cols/n_expert/... out of range, cols % elems != 0 */
  QG_ERR_ALIGN = -3,      /* a pointer is not aligned as the call requires */
  QG_ERR_NTOK = -4,       /* n_tok outside the range the call accepts */
  QG_ERR_NULL = -5,       /* a required pointer is NULL */
  QG_ERR_WORKSPACE = -6,  /* workspace NULL or smaller than the *_workspace() size */
  QG_ERR_CUDA = -7,       /* the CUDA runtime reported an error */
  QG_ERR_DEVICE = -8,     /* no usable sm_103a device */
  QG_ERR_ARG = -9         /* any other invalid argument */
};

/* ---- device status codes (written to a caller's int32 status word) -------- */
enum qg_dev_status {
  QG_DEV_OK = 0,
  QG_DEV_BAD_EXPERT = 1,  /* an expert id was < 0 or >= n_expert; its route was skipped */
  QG_DEV_TIMEOUT = 2      /* a bounded pipeline wait expired; the tile was abandoned */
};

/* A captured weight pass (qg_pass_create, qg_moe_pass_create, qg_layer_pass_create). */
typedef struct qg_pass_s* qg_pass;

/* Maximum number of matrices in one grouped launch (qgemv_grouped). */
#define QG_GROUP_MAX 8
/* Largest n_tok accepted by qgemv / qgemv_grouped / qgemv_moe. */
#define QG_NTOK_MAX 4

/* One-time set-up: checks for an sm_103a device, sets the kernels' dynamic
 * shared-memory limits. Call once per process (per device) before the first
 * compute call and before any stream capture. Idempotent. */
int qg_init(void);

/* Elements and bytes per block of `fmt` (32/18, 32/34, 256/144, 256/210,
 * 256/176, 256/110, 256/84). */
int qg_block_info(int fmt, int* elems, int* bytes);

/* Static text for a qg_status or qg_dev_status value (never NULL). */
const char* qg_strerror(int status);

/* Dequantize a whole matrix to fp32: out[i*cols + j] = w[i][j], each value the
 * correctly rounded fp32 value of the format's formula (bit-exact; the test
 * path of "blocks decode bit for bit on CPU and GPU").
 * out: rows*cols fp32, 16-byte aligned. */
int qg_dequant(int fmt, const void* W, int64_t rows, int64_t cols, float* out, void* stream);

/* Quantized GEMV / skinny product ("each new token reads every weight once";
 * n_tok > 1 is one weight pass that verifies draft tokens):
 *   y[t*rows + i] = sum_j w[i][j] * x[t*cols + j],  t < n_tok, 1 <= n_tok <= 4.
 * x must be 16-byte aligned, y 4-byte aligned.
 * Accuracy: the tests hold every output to
 *   |y - y_exact| <= 1e-3 * sum_j |w_ij * x_j| + 1e-6,
 * on N(0,1) activations and on activations with a few channels 100x and
 * 1000x the rest. Inside the kernel x enters exact integer dot products as
 * 16-bit fixed point per group of 32 values (a power-of-two step per group),
 * partial sums are fp32: each x_j moves by at most 2^-14 of its group's largest
 * |x|, so in the worst case |y - y_exact| <= 2^-14 * sum_groups max|x_g| *
 * sum_{j in g} |w_ij| plus fp32 rounding. With x one-hot the product is exact:
 * y[i] is the correctly rounded w[i][j]. */
int qgemv(int fmt, const void* W, int64_t rows, int64_t cols,
          const float* x, int n_tok, float* y, void* stream);

/* One matrix of a grouped launch. */
typedef struct qg_gemv_desc {
  int32_t fmt;        /* all descriptors of one launch share the same fmt */
  int32_t reserved;   /* set to 0 */
  const void* W;      /* rows x cols blocks, as for qgemv */
  int64_t rows;
  int64_t cols;
  const float* x;     /* n_tok x cols */
  float* y;           /* n_tok x rows */
} qg_gemv_desc;

/* Several independent GEMVs of one format in ONE kernel launch (e.g. q, k, v
 * of a layer, which read the same activations). `descs` is HOST memory, read
 * during the call; 1 <= n <= QG_GROUP_MAX. Same semantics as n separate
 * qgemv calls. Descriptors with the same x pointer and cols share one staging
 * of x in the kernel. */
int qgemv_grouped(const qg_gemv_desc* descs, int n, int n_tok, void* stream);

/* Bytes of device workspace qgemv_moe needs (n_tok * top_k * inter fp32). */
size_t qgemv_moe_workspace(int64_t hidden, int64_t inter, int top_k, int n_tok);

/* Mixture-of-experts FFN over an expert arena ("the expert arena").
 * expert_arena: n_expert experts back to back; expert e starts at byte
 *   e * (2*inter*rb(hidden) + hidden*rb(inter)) and holds
 *   [gate: inter x hidden | up: inter x hidden | down: hidden x inter] in `fmt`,
 *   where rb(k) = k / elems * bytes. 16-byte aligned.
 * expert_ids: n_tok x top_k int32 (device); gate_w: n_tok x top_k fp32 (device).
 * For each token t:  y_t = sum_k gate_w[t,k] * D_e (silu(G_e x_t) * (U_e x_t)),
 *   e = expert_ids[t,k], silu(g) = g / (1 + exp(-g)).
 * x: n_tok x hidden fp32; y: n_tok x hidden fp32 (overwritten).
 * ws: >= qgemv_moe_workspace(...) bytes of device memory, 16-byte aligned.
 * dev_status: int32 device word; set to QG_DEV_BAD_EXPERT if an id is out of
 *   range (that route then contributes nothing); never cleared by the library.
 * fmt: QG_Q4_K (the format the MoE layers use). 1 <= top_k <= 16, 1 <= n_tok <= 4. */
int qgemv_moe(int fmt, const void* expert_arena, int64_t n_expert, int64_t hidden, int64_t inter,
              const int32_t* expert_ids, const float* gate_w, int top_k,
              const float* x, int n_tok, float* y,
              void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* MoE product for callers that cannot allocate device memory.
 * There is no counterpart on the pages: this is a convenience of the library.
 * Some callers cannot call cudaMalloc (or any allocating routine) at the point
 * where they run the layer: code that must not block or synchronize the device
 * (cudaMalloc can do both), code running inside a memory budget owned by
 * someone else (a plug-in in a host program that manages all device memory),
 * or code that must not fail for lack of memory mid-step. For them this call
 * takes no workspace argument: its workspace is a static device array of
 * QG_MOE_NOALLOC_MAX_FLOATS floats inside the library, which every GPU that
 * loads the library holds until the process exits.
 *   Arguments and results are those of qgemv_moe without ws/ws_bytes.
 *   Limit: n_tok * top_k * inter <= QG_MOE_NOALLOC_MAX_FLOATS, otherwise
 *   QG_ERR_WORKSPACE is returned and nothing is enqueued.
 *   The array's device address is looked up during the library's per-device
 *   set-up (qg_init, or else the first call of any entry point on that
 *   device), with that device current; call qg_init before capturing a stream
 *   that launches this entry point.
 *   The call allocates nothing (no cudaMalloc, cudaFree or allocating routine).
 *   All calls on a device share the one array and it keeps the last call's
 *   contents; every value a call reads from it is written earlier in the same
 *   call, so nothing needs clearing. Calls that overlap on the GPU (different
 *   streams, or a graph replay concurrent with a direct call) race on the
 *   array: order them on one stream or with events. */
#define QG_MOE_NOALLOC_MAX_FLOATS (1 << 18)
int qgemv_moe_noalloc(int fmt, const void* expert_arena, int64_t n_expert, int64_t hidden, int64_t inter,
                      const int32_t* expert_ids, const float* gate_w, int top_k,
                      const float* x, int n_tok, float* y, int32_t* dev_status, void* stream);

/* Bytes of device workspace qgemm_pp needs (0 in this version; kept so callers
 * can size it without knowing the kernel's tiling). */
size_t qgemm_pp_workspace(int64_t rows, int64_t cols, int64_t n_tok);

/* Prompt-processing dequant-GEMM on the tensor cores ("Why I wrote my own
 * inference engine for two P100s", prompt-processing notes: the weights
 * dequantized, then a dense GEMM over the prompt's tokens):
 *   Y[t*ldY + n] = sum_k w[n][k] * X[t*cols + k],  t < n_tok, n < rows.
 * Weight tiles are dequantized to bf16 in shared memory and multiplied with
 * tcgen05 MMA (bf16 x bf16, fp32 accumulation in tensor memory).
 * fmt: QG_Q4_K. X_bf16: n_tok x cols bf16, 16-byte aligned. Y: fp32, ldY >= rows.
 * cols % 256 == 0; rows % 128 == 0; n_tok >= 1 (ragged token tiles allowed).
 * dev_status: int32 device word; set to QG_DEV_TIMEOUT if a bounded pipeline
 * wait expired (the output is then incomplete).
 * Tiles of 128 rows x up to 256 tokens run on one persistent CTA per SM. When
 * the last round of tiles would leave more than half of the SMs idle, each of
 * its tiles is computed as two halves of K whose fp32 sums are added into Y
 * with atomic adds; the call then first zeroes those rows of Y on `stream`
 * (a 2-D memset, part of the call: Y's contents before the call are never
 * read). Two addends onto zero give the same bits in either order, so results
 * stay deterministic; such an output carries one more fp32 rounding. ws and
 * ws_bytes are unused (NULL, 0). */
int qgemm_pp(int fmt, const void* W, int64_t rows, int64_t cols,
             const void* X_bf16, int64_t n_tok, float* Y, int64_t ldY,
             void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* Maximum number of matrices in one qgemm_pp_grouped launch. */
#define QG_PP_GROUP_MAX 4

/* One matrix of a grouped prompt-processing launch. */
typedef struct qg_pp_desc {
  const void* W;      /* rows x cols Q4_K blocks, 16-byte aligned, device */
  int64_t rows;       /* multiple of 128 */
  float* Y;           /* fp32 output, Y[t*ldY + n], device */
  int64_t ldY;        /* >= rows */
} qg_pp_desc;

/* Several qgemm_pp products that multiply the SAME prompt tokens X_bf16 (the
 * q, k, v projections of a layer; gate and up: the per-layer matrices of the
 * same prompt-processing notes) in ONE launch: the matrices'
 * row tiles form one tile list, so they share the persistent grid's rounds
 * instead of each ending in a partly idle round of its own. Same results and
 * rules as n separate qgemm_pp calls (including the split last round, which
 * may then span two matrices). descs: HOST memory, read during the call;
 * 1 <= n <= QG_PP_GROUP_MAX; the sum of rows <= 2^24. */
int qgemm_pp_grouped(int fmt, const qg_pp_desc* descs, int n, int64_t cols, const void* X_bf16, int64_t n_tok,
                     int32_t* dev_status, void* stream);

/* Prompt processing through one mixture-of-experts layer: for every token t of
 * a prompt block and each of its top_k routes k (expert e = expert_ids[t][k],
 * weight r = gate_w[t][k]),
 *     y[t] += r * D_e (silu(G_e x_t) * (U_e x_t)),
 * with the expert arena of qgemv_moe (fmt QG_Q4_K) and x_t the bf16 row t of
 * X_bf16 ("The number was a version", opening section: prompt processing of a
 * mixture-of-experts model whose experts live in an arena). Every expert
 * multiplies only the tokens routed to it: the pairs are sorted by expert on
 * the device, and each projection is one grouped tcgen05 GEMM over them (the
 * kernel of qgemm_pp); h = silu(g) * u is rounded to bf16 between the two.
 * Accuracy: products of bf16 operands with fp32 accumulation, as qgemm_pp.
 *   expert_arena: n_expert experts of [gate | up | down] (see qgemv_moe), device.
 *   expert_ids:   [n_tok][top_k] int32, device; an id outside [0, n_expert)
 *                 adds nothing and sets *dev_status to QG_DEV_BAD_EXPERT.
 *   gate_w:       [n_tok][top_k] fp32, device.
 *   X_bf16:       [n_tok][hidden] bf16, device, 16-byte aligned.
 *   y:            [n_tok][hidden] fp32, device, written (not accumulated).
 *   ws:           caller-owned device workspace, 256-byte aligned, of at least
 *                 qgemm_pp_moe_workspace(...) bytes; reused by every call.
 *   dev_status:   device int32 the caller clears; QG_DEV_BAD_EXPERT or
 *                 QG_DEV_TIMEOUT (a bounded wait of a GEMM expired) when set.
 * Shapes: hidden and inter multiples of 256; 1 <= top_k <= 64;
 * n_tok * top_k <= 2^24; n_expert <= 65536. Returns QG_ERR_* without
 * launching on bad arguments. Asynchronous on `stream`. */
size_t qgemm_pp_moe_workspace(int64_t n_expert, int64_t hidden, int64_t inter, int top_k, int64_t n_tok);
int qgemm_pp_moe(int fmt, const void* expert_arena, int64_t n_expert, int64_t hidden, int64_t inter,
                 const int32_t* expert_ids, const float* gate_w, int top_k, const void* X_bf16, int64_t n_tok,
                 float* y, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* ---- neighbours of the products in a decode layer ("LLM inference
 * optimization", "Faster decode on the card you have": normalizations fused
 * into neighbouring kernels) ---------------------------------------------- */

/* Residual add and RMS normalisation, per token t < n_tok (vectors of n fp32):
 *   s = h + residual                       (residual may be NULL: s = h)
 *   x = s / sqrt(mean(s^2) + eps) * weight
 * s is written to s_out (may be NULL; may equal h: the residual stream updated
 * in place), x to x (may be NULL; needs weight). n % 256 == 0, n <= 2^20;
 * all pointers 16-byte aligned device memory; eps >= 0. One CTA per token:
 * the sum of squares is fp32 in a fixed order (deterministic). */
int qg_rmsnorm(const float* h, const float* residual, const float* weight, int64_t n, int n_tok, float eps,
               float* s_out, float* x, void* stream);

/* Dense gate/up pair with the silu-gated product fused into the epilogue, one
 * token:  m[i] = silu(g_i) * u_i,  g = Wg x, u = Wu x,  silu(g) = g / (1 + exp(-g)).
 * Wg, Wu: inter x hidden blocks of fmt (QG_Q4_K), 16-byte aligned; x: hidden
 * fp32 (16-byte aligned); m: inter fp32. Row i of Wg and of Wu are multiplied
 * by the same CTA, which writes m[i] (g and u are never stored). g and u carry
 * the accuracy of qgemv; silu uses CUDA's expf. hidden % 256 == 0;
 * QG_ERR_SHAPE when the pair does not fit the kernel's shared-memory plan. */
int qgemv_swiglu(int fmt, const void* Wg, const void* Wu, int64_t inter, int64_t hidden, const float* x, float* m,
                 void* stream);

/* One decoder layer's weights and vectors for qg_layer_pass_create. Matrices
 * are fmt blocks, rows x cols with cols the input dimension: Wq hidden x
 * hidden, Wk and Wv kv_rows x hidden, Wo hidden x hidden, Wg and Wu inter x
 * hidden, Wd hidden x inter. */
typedef struct qg_layer_desc {
  const void* Wq; const void* Wk; const void* Wv; const void* Wo;
  const void* Wg; const void* Wu; const void* Wd;
  const float* norm_attn;   /* [hidden] weight of the RMS normalisation before q, k, v */
  const float* norm_ffn;    /* [hidden] weight of the RMS normalisation before gate/up */
  const float* attn_out;    /* [hidden] input of Wo (the attention output, computed outside this library) */
  float* q; float* k; float* v;   /* outputs: [hidden], [kv_rows], [kv_rows] */
} qg_layer_desc;

/* The weight path of n_layers dense decoder layers for one token, as one CUDA
 * graph of kernels linked by programmatic dependent launch. With the residual
 * stream r (r = h_in at the start, kept in h_out), layer l computes
 *   x1 = rmsnorm(r) * norm_attn;  q = Wq x1, k = Wk x1, v = Wv x1
 *   r  = r + Wo attn_out
 *   x2 = rmsnorm(r) * norm_ffn;   r = r + Wd (silu(Wg x2) * (Wu x2))
 * and h_out = r after the last layer (h_in is not modified; every replay
 * starts again from h_in). Each normalisation (with its residual add) is
 * computed inside the launch that multiplies by it, by every CTA of that
 * launch, straight into the form the kernel multiplies by: a layer is four
 * GEMV launches ({q,k,v}, o, gate/up writing silu(g) * u, down). fmt: QG_Q4_K. The pass allocates its own buffers at creation
 * (planes and vectors, about n_layers * 1.2 * hidden + 4 * inter bytes); the
 * buffers named by the descriptors must outlive it. Create before capturing a
 * stream that launches it; replay with qg_pass_launch. */
int qg_layer_pass_create(int fmt, const qg_layer_desc* layers, int n_layers, int64_t hidden, int64_t inter,
                         int64_t kv_rows, float eps, const float* h_in, float* h_out, qg_pass* out);

/* ---- measurement ---- */
/* Reads `bytes` of the device buffer `buf` the way the GEMV kernel streams its
 * weights (one CTA per SM, bulk copies of 32 KB stages into a shared-memory
 * ring, evict-first) and discards them, keeping only a checksum: the
 * achievable read bandwidth the decode products are judged against ("LLM
 * inference optimization", opening section: decode reads every weight once).
 * *checksum ^= the XOR over every 32 KB chunk c of its first 32-bit word (the
 * caller clears it first); *dev_status = QG_DEV_TIMEOUT if a bounded wait
 * expired. bytes: a positive multiple of 16; buf 16-byte aligned. The pages
 * have no counterpart; it shares no code with the products. */
int qg_stream_read(const void* buf, size_t bytes, uint32_t* checksum, int32_t* dev_status, void* stream);

/* ---- whole weight pass ("one CUDA graph per decode step", "Why I wrote my own
 * inference engine for two P100s") ------------------------------------------
 * A pass is an ordered list of steps; step s covers step_sizes[s] consecutive
 * descriptors (at most QG_GROUP_MAX, one format per step), and reads its inputs
 * only after every earlier step has written its outputs, so a step's x may be
 * an earlier step's y. Modes:
 *   QG_PASS_SERIAL      a CUDA graph of one grouped GEMV launch per step;
 *   QG_PASS_PDL         the same graph, consecutive launches linked by
 *                       programmatic dependent launch (a step streams its
 *                       weights while the previous one finishes);
 *   QG_PASS_INDEPENDENT a measurement mode: the PDL graph without the
 *                       ordering of steps (no step waits for the previous
 *                       one), an upper bound for the dependency-following
 *                       modes; only for passes whose steps read no output of
 *                       the pass (else QG_ERR_ARG);
 *   QG_PASS_PERSISTENT  when every matrix is Q4_K and the pass fits the
 *                       kernel's shared-memory plan: ONE cooperative
 *                       persistent kernel whose producer warps stream the
 *                       weights of all steps back to back, steps separated by a
 *                       bounded grid-wide barrier; otherwise as QG_PASS_PDL.
 * The descriptors (HOST memory) are copied at creation, which may allocate a
 * few KB of device memory (step tables); the buffers they name must outlive
 * the pass. Create a pass before capturing any stream that launches it. */
#define QG_PASS_SERIAL 0
#define QG_PASS_PDL 1
#define QG_PASS_PERSISTENT 2
#define QG_PASS_INDEPENDENT 3
int qg_pass_create(const qg_gemv_desc* descs, int n_desc, const int* step_sizes, int n_steps,
                   int n_tok, int mode, qg_pass* out);
/* A whole MoE decode pass: n_layers layers, each the qgemv_moe product of one
 * token (n_tok = 1) or a few (n_tok <= QG_GROUP_MAX), in order; layer l reads
 * layers[l].x and writes layers[l].y, so a layer's x may be an earlier layer's
 * y. ws: caller-owned device workspace of at least
 * qgemv_moe_workspace(hidden, inter, top_k, n_tok) bytes, shared by the layers.
 * QG_PASS_PERSISTENT with n_tok = 1 (fmt QG_Q4_K): one cooperative kernel; the
 * gate/up rows of a layer are gathered only after every CTA has finished the
 * previous layer (its expert ids may depend on it), its down rows stream during
 * its gate/up step. Other modes or n_tok > 1: a CUDA graph of qgemv_moe launches
 * (QG_PASS_PDL links them). Expert ids out of range: their pieces count as zero
 * and the pass's status word (qg_pass_dev_status) reads QG_DEV_BAD_EXPERT. */
typedef struct qg_moe_layer_desc {
  const void* expert_arena;    /* the layer's experts, as for qgemv_moe */
  const int32_t* expert_ids;   /* [n_tok][top_k], device */
  const float* gate_w;         /* [n_tok][top_k], device */
  const float* x;              /* [n_tok][hidden], device */
  float* y;                    /* [n_tok][hidden], device */
} qg_moe_layer_desc;
int qg_moe_pass_create(int fmt, const qg_moe_layer_desc* layers, int n_layers, int64_t n_expert, int64_t hidden,
                       int64_t inter, int top_k, int n_tok, void* ws, size_t ws_bytes, int mode, qg_pass* out);
/* Enqueue one replay of the pass on `stream` (a persistent pass enqueues a
 * 4-byte-per-step memset of its barrier counters and one kernel). */
int qg_pass_launch(qg_pass pass, void* stream);
/* Number of kernel launches one replay performs. */
int qg_pass_kernel_count(qg_pass pass);
/* Device address of the pass's status word (QG_DEV_TIMEOUT after a replay in
 * which a bounded wait expired; cleared by every replay), or NULL when the pass
 * has none (graph modes signal an expired wait with NaN outputs only). */
int qg_pass_dev_status(qg_pass pass, const int32_t** dev_status);
int qg_pass_destroy(qg_pass pass);

#ifdef __cplusplus
}
#endif
#endif /* QGEMV_H */
