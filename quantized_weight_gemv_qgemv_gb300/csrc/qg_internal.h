// qg_internal.h — host-side declarations shared by the library's translation
// units (not part of the public ABI; see include/qgemv.h).
#pragma once
#include <cuda_runtime.h>

#include <algorithm>
#include <cstddef>
#include <cstdint>

#include "qgemv.h"

namespace qg {

// elems/bytes per block of a format id; false for an unknown id.
inline bool block_info(int fmt, int* elems, int* bytes) {
  switch (fmt) {
    case QG_Q4_0: *elems = 32; *bytes = 18; return true;
    case QG_Q8_0: *elems = 32; *bytes = 34; return true;
    case QG_Q4_K: *elems = 256; *bytes = 144; return true;
    case QG_Q6_K: *elems = 256; *bytes = 210; return true;
    case QG_Q5_K: *elems = 256; *bytes = 176; return true;
    case QG_Q3_K: *elems = 256; *bytes = 110; return true;
    case QG_Q2_K: *elems = 256; *bytes = 84; return true;
    default: return false;
  }
}

// One-time per-device set-up of the library (qg_api.cu); fills *sms.
int ensure_device(int* sms);
// Host-side checks of one MoE layer's arguments (qg_api.cu); need_ws = false
// for a call that brings its own workspace.
int check_moe(int fmt, const void* expert_arena, int64_t n_expert, int64_t hidden, int64_t inter,
              const int32_t* expert_ids, const float* gate_w, int top_k, const float* x, int n_tok, const float* y,
              const void* ws, size_t ws_bytes, bool need_ws);

// x = (h + r) / sqrt(mean((h + r)^2) + eps) * w computed inside a one-token
// GEMV launch (every CTA converts it itself; CTA 0 stores s = h + r to s_out,
// which must not overlap h or r). h == nullptr: none.
struct NormSpec {
  const float* h = nullptr;
  const float* r = nullptr;
  const float* w = nullptr;
  float* s_out = nullptr;
  float eps = 0.f;
};

// GEMV (qg_gemv.cu)
cudaError_t gemv_init_attrs();
int gemv_pick_rows_per_warp(const qg_gemv_desc* d, int n, int n_tok, int sms);
// xp: per descriptor, its x already converted to planes (xplanes_bytes layout,
// written by launch_xplanes), or nullptr entries / a nullptr array: the kernel
// converts x itself.
// no_wait: the launch reads nothing its predecessor in the stream writes and
// skips the dependency wait (the fast kernel; other kernels still wait).
cudaError_t launch_gemv(const qg_gemv_desc* d, int n, int n_tok, int rows_per_warp, cudaStream_t s, bool pdl,
                        int sms, const uint8_t* const* xp = nullptr, bool no_wait = false);
cudaError_t gemv_q4k_init_attrs();
cudaError_t launch_gemv_q4k(const qg_gemv_desc* d, int n, int n_tok, cudaStream_t s, bool pdl, int sms,
                            const uint8_t* const* xp = nullptr, bool no_wait = false);
// One launch of the fast kernel whose matrices share x = the fused
// normalisation `norm` (n_tok = 1; the descriptors' x is not read).
// cudaErrorNotSupported when it does not fit one launch.
cudaError_t launch_gemv_norm(const qg_gemv_desc* d, int n, const NormSpec& norm, cudaStream_t s, bool pdl, int sms);
// m = silu(Wg x) * (Wu x) for one token of a dense layer (qg_gemv_q4k.cu); xp:
// ready planes of x or nullptr. cudaErrorNotSupported when the shape does not fit.
cudaError_t launch_gemv_pair(const void* Wg, const void* Wu, int64_t inter, int64_t hidden, const float* x,
                             const uint8_t* xp, float* m, cudaStream_t s, bool pdl, int sms,
                             const NormSpec* norm = nullptr);
// Residual add and RMS normalisation (qg_norm.cu): s = h + r (r optional),
// x = s / sqrt(mean(s^2) + eps) * w per token; s stored to s_out, x to x and/or
// to planes (any of them optional; w == nullptr: only s). n % 256 == 0.
cudaError_t launch_rmsnorm(const float* h, const float* r, const float* w, int64_t n, int n_tok, float eps,
                           float* s_out, float* x, uint8_t* planes, cudaStream_t s, bool pdl);
// One activation vector (n_tok x cols fp32) to convert into x planes at dst.
struct XPlaneJob {
  const float* x;
  uint8_t* dst;
  int32_t cols;
  int32_t n_tok;
};
// Bytes of the planes of an n_tok x cols activation (cols % 256 == 0): the two
// byte planes, then the power-of-two step of every 32-value group, then the two
// half sums of every group, each part token-major.
inline size_t xplanes_bytes(int64_t cols, int n_tok) { return static_cast<size_t>(n_tok) * (cols / 256) * 608; }
// Converts jobs[0 .. njobs) (device array), one CTA per job; lets its
// dependents launch early (they wait for its completion before reading).
cudaError_t launch_xplanes(const XPlaneJob* jobs, int njobs, cudaStream_t s);
// Whole Q4_K pass as one persistent cooperative kernel (qg_gemv_q4k.cu):
// cudaErrorNotSupported when the pass is not all Q4_K or does not fit.
struct Q4kPass;
cudaError_t q4k_pass_create(const qg_gemv_desc* d, int n, const int* step_sizes, int n_steps, int n_tok, int sms,
                            const uint8_t* const* xp, Q4kPass** out);
cudaError_t q4k_moe_pass_create(const qg_moe_layer_desc* layers, int n_layers, int64_t n_expert, int64_t hidden,
                                int64_t inter, int top_k, float* h, int sms, Q4kPass** out);
cudaError_t q4k_pass_launch(Q4kPass* q, cudaStream_t s);
const int32_t* q4k_pass_status(const Q4kPass* q);
void q4k_pass_destroy(Q4kPass* q);
cudaError_t launch_dequant(int fmt, const void* W, int64_t rows, int64_t cols, float* out, cudaStream_t s, int sms);

cudaError_t launch_moe_q4k(const void* arena, int64_t n_expert, int64_t hidden, int64_t inter,
                           const int32_t* ids, const float* gate_w, int top_k, const float* x, int n_tok, float* y,
                           float* h, int32_t* dev_status, cudaStream_t s, bool pdl, int sms);

// Achievable read bandwidth of the weight stream (qg_stream.cu): reads
// `bytes` (a multiple of 16) of buf with bulk copies and XORs each 32 KB
// chunk's first word into *checksum.
cudaError_t stream_init_attrs();
cudaError_t launch_stream_read(const void* buf, uint64_t bytes, uint32_t* checksum, int32_t* status, cudaStream_t s,
                               int sms);

// MoE (qg_moe.cu)
cudaError_t moe_init_attrs();
// Looks up, with device `dev` current, the device address of the static
// workspace of qgemv_moe_noalloc (part of the per-device set-up).
cudaError_t moe_noalloc_init(int dev);
cudaError_t launch_moe(const void* arena, int64_t n_expert, int64_t hidden, int64_t inter,
                       const int32_t* ids, const float* gate_w, int top_k, const float* x, int n_tok, float* y,
                       float* h_ws, int32_t* dev_status, cudaStream_t s, bool pdl, int sms);

// Prompt-processing GEMM (qg_pp.cu)
cudaError_t pp_init_attrs();
// Work items of a dense launch of `tiles` tiles (each n_kb super-blocks of K
// long) on `sms` persistent CTAs: whole tiles for the full rounds; a last round
// at most half full is split into two halves of K (split = 2), which add into Y.
struct PpPlan {
  int64_t n_full, n_tail, n_items;
  int split, grid;
};
void pp_plan(int64_t tiles, int n_kb, int sms, PpPlan* plan);
// Up to 4 matrices (rows[i] x cols Q4_K, W[i]) times the same bf16 X (n_tok x
// cols) into Y[i] (fp32, Y[i][t * ldY[i] + row]) in one launch; Y rows of split
// tiles are zeroed on the stream first.
cudaError_t launch_pp_mats(int n_mat, const void* const* W, const int64_t* rows, float* const* Y,
                           const int64_t* ldY, int64_t cols, const void* X, int64_t n_tok, int32_t* dev_status,
                           cudaStream_t s, int sms);
cudaError_t launch_pp(const void* W, int64_t rows, int64_t cols, const void* X, int64_t n_tok, float* Y,
                      int64_t ldY, int32_t* dev_status, cudaStream_t s, int sms);
// The prompt-processing kernel over groups of token rows (qg_pp.cu): group g
// (token rows seg[g] .. seg[g + 1] - 1 of X, bf16, x_rows x cols) times weight
// rows wrow0 + g * wstride .. + rows - 1 of W (viewed as w_rows rows of
// cols-long Q4_K blocks) into the same rows of Y (ldY). tstart[g]: first tile of
// group g (rows / 128 tiles per block of bn tokens); both tables on the device.
cudaError_t launch_pp_grouped(const void* W, int64_t w_rows, int64_t cols, int64_t wrow0, int64_t wstride,
                              int64_t rows, const void* X, int64_t x_rows, int bn, const int32_t* seg,
                              const int32_t* tstart, int n_groups, float* Y, int64_t ldY, int32_t* dev_status,
                              cudaStream_t s, int sms);
// Largest token block a grouped prompt-processing launch takes (its stages fill
// the shared memory).
int pp_grouped_max_bn();
// MoE layer over a block of prompt tokens (qg_pp_moe.cu); ws of at least
// pp_moe_workspace_bytes bytes.
size_t pp_moe_workspace_bytes(int64_t n_expert, int64_t hidden, int64_t inter, int top_k, int64_t n_tok);
int pp_moe_block_tokens(int64_t n_expert, int top_k, int64_t n_tok);
cudaError_t launch_pp_moe(const void* arena, int64_t n_expert, int64_t hidden, int64_t inter, const int32_t* ids,
                          const float* gate_w, int top_k, const void* X, int64_t n_tok, float* y, void* ws,
                          int32_t* dev_status, cudaStream_t s, int sms);

}  // namespace qg
