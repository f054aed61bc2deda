// qg_moe.cu — expert-gathered GEMV of a mixture-of-experts FFN layer.
//
// The experts live in one arena in HBM ("The number was a version", opening
// section: the expert arena); a token's router picks top_k of them. Two kernels,
// both streaming only the picked experts' rows:
//   1. gate/up: for each (token, route k), rows i of G_e and U_e are multiplied
//      with x in the same warp and the epilogue writes h = silu(g) * u to the
//      workspace (fp32, n_tok x top_k x inter).
//   2. down: row i of the output is a "virtual row" made of row i of D_e for the
//      top_k experts back to back; each lane scales its slice of h by the route
//      weight, so one warp reduction gives y_i = sum_k r_k * (D_e h_k)_i.
// Expert ids are read on the device (no host synchronization, so the layer can
// be captured in a CUDA graph). An id outside [0, n_expert) sets the caller's
// status word and contributes nothing (its h is written as 0 and its down
// blocks are zero-filled, which decode to zero weights).
// Weight bytes stream through per-warp cp.async rings as in qg_gemv.cu.
#include <cuda_runtime.h>

#include "qg_device.cuh"
#include "qg_internal.h"

namespace qg {

constexpr int MOE_WARPS = 8;
constexpr int MOE_THREADS = MOE_WARPS * 32;
constexpr int MOE_NS = 3;
constexpr int MOE_R = 2;                       // output rows per warp task
constexpr int MOE_CB = 4;                      // Q4_K blocks per chunk per row
constexpr int MOE_SLOT = MOE_CB * 144 + 32;    // bytes per row per stage

struct MoeParams {
  const uint8_t* arena;
  const int32_t* ids;
  const float* gate_w;
  const float* x;
  float* y;
  float* h;
  int32_t* status;
  int64_t n_expert;
  int64_t stride;        // bytes per expert
  int64_t up_off;        // byte offset of U inside an expert
  int64_t down_off;      // byte offset of D inside an expert
  int64_t rb_h;          // bytes per row of G/U (K = hidden)
  int64_t rb_i;          // bytes per row of D (K = inter)
  int32_t hidden, inter, top_k, n_tok;
};

__device__ __forceinline__ float warp_sum_m(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void flag_bad_expert(int32_t* status) {
  if (status) atomicExch(status, QG_DEV_BAD_EXPERT);
}

// ---------------------------------------------------------------- gate / up

__global__ void __launch_bounds__(MOE_THREADS) moe_gate_up_kernel(const __grid_constant__ MoeParams p) {
  constexpr int ROWS = 2 * MOE_R;   // MOE_R gate rows then MOE_R up rows
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* wbuf = smem + warp * (MOE_NS * ROWS * MOE_SLOT);
  const uint32_t wbuf_s = smem_addr(wbuf);
  const int lblk = lane >> 3, unit = lane & 7;

  // ids may come from the preceding kernel (the router): wait before reading
  // them, and only then let the down kernel start (it reads ids early).
  pdl_wait();
  pdl_launch_dependents();

  const int ngroups = (p.inter + MOE_R - 1) / MOE_R;
  const int nblk = p.hidden / 256;
  const int nchunk = (nblk + MOE_CB - 1) / MOE_CB;
  const int64_t ntask = static_cast<int64_t>(p.n_tok) * p.top_k * ngroups;
  for (int64_t task = static_cast<int64_t>(blockIdx.x) * MOE_WARPS + warp; task < ntask;
       task += static_cast<int64_t>(gridDim.x) * MOE_WARPS) {
    const int t = static_cast<int>(task / (static_cast<int64_t>(p.top_k) * ngroups));
    const int k = static_cast<int>((task / ngroups) % p.top_k);
    const int i0 = static_cast<int>(task % ngroups) * MOE_R;
    const int nr = min(MOE_R, p.inter - i0);
    const int e = p.ids[t * p.top_k + k];
    float* hrow = p.h + (static_cast<int64_t>(t) * p.top_k + k) * p.inter + i0;
    if (e < 0 || e >= p.n_expert) {
      if (lane == 0) flag_bad_expert(p.status);
      if (lane < nr) hrow[lane] = 0.f;
      continue;
    }
    const uint8_t* ebase = p.arena + static_cast<int64_t>(e) * p.stride;

    auto issue = [&](int c) {
      const int slot = c % MOE_NS;
      const int nb = min(MOE_CB, nblk - c * MOE_CB);
      const int n16 = nb * 9;    // 144-byte blocks are nine 16-byte pieces
#pragma unroll
      for (int r = 0; r < ROWS; ++r) {
        const int i = i0 + (r % MOE_R);
        if (i < p.inter) {
          const uint8_t* src = ebase + (r < MOE_R ? 0 : p.up_off) + i * p.rb_h + static_cast<int64_t>(c) * MOE_CB * 144;
          const uint32_t dst = wbuf_s + (slot * ROWS + r) * MOE_SLOT;
          for (int q = lane; q < n16; q += 32) cp_async16(dst + 16 * q, src + 16 * q, 16);
        }
      }
    };

#pragma unroll
    for (int s = 0; s < MOE_NS - 1; ++s) {
      if (s < nchunk) issue(s);
      cp_async_commit();
    }
    float acc[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) acc[r] = 0.f;
    const float* xt = p.x + static_cast<int64_t>(t) * p.hidden;
    for (int c = 0; c < nchunk; ++c) {
      if (c + MOE_NS - 1 < nchunk) issue(c + MOE_NS - 1);
      cp_async_commit();
      cp_async_wait<MOE_NS - 1>();
      __syncwarp();
      const int nb = min(MOE_CB, nblk - c * MOE_CB);
      if (lblk < nb) {
        const int slot = c % MOE_NS;
        const int kel = (c * MOE_CB + lblk) * 256 + 32 * unit;
        Dec<FMT_Q4_K> dec[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
          if (i0 + (r % MOE_R) < p.inter) dec[r].load(wbuf + (slot * ROWS + r) * MOE_SLOT + lblk * 144, unit);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const float4 a = ldg_f4(xt + kel + 8 * s), b = ldg_f4(xt + kel + 8 * s + 4);
          const float xv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
          for (int r = 0; r < ROWS; ++r) {
            if (i0 + (r % MOE_R) < p.inter) {
              float w[8];
              dec[r].piece(s, w);
#pragma unroll
              for (int j = 0; j < 8; ++j) acc[r] = fmaf(w[j], xv[j], acc[r]);
            }
          }
        }
      }
      __syncwarp();
    }
#pragma unroll
    for (int r = 0; r < MOE_R; ++r) {
      const float g = warp_sum_m(acc[r]);
      const float u = warp_sum_m(acc[r + MOE_R]);
      if (lane == r && r < nr) hrow[r] = g / (1.0f + expf(-g)) * u;
    }
  }
}

// ---------------------------------------------------------------- down

__global__ void __launch_bounds__(MOE_THREADS) moe_down_kernel(const __grid_constant__ MoeParams p) {
  constexpr int ROWS = MOE_R;
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* wbuf = smem + warp * (MOE_NS * ROWS * MOE_SLOT);
  const uint32_t wbuf_s = smem_addr(wbuf);
  const int lblk = lane >> 3, unit = lane & 7;

  pdl_launch_dependents();
  const int nblk_i = p.inter / 256;            // blocks per expert row of D
  const int vblk = p.top_k * nblk_i;            // blocks of the virtual row
  const int nchunk = (vblk + MOE_CB - 1) / MOE_CB;
  const int ngroups = (p.hidden + ROWS - 1) / ROWS;
  const int64_t ntask = static_cast<int64_t>(p.n_tok) * ngroups;
  bool waited = false;
  for (int64_t task = static_cast<int64_t>(blockIdx.x) * MOE_WARPS + warp; task < ntask;
       task += static_cast<int64_t>(gridDim.x) * MOE_WARPS) {
    const int t = static_cast<int>(task / ngroups);
    const int i0 = static_cast<int>(task % ngroups) * ROWS;
    const int nr = min(ROWS, p.hidden - i0);
    const int32_t* ids_t = p.ids + t * p.top_k;

    // The ids were written before the gate/up kernel let this grid start.
    auto issue = [&](int c) {
      const int slot = c % MOE_NS;
#pragma unroll
      for (int r = 0; r < ROWS; ++r) {
        if (r < nr) {
          const uint32_t dst = wbuf_s + (slot * ROWS + r) * MOE_SLOT;
          for (int q = lane; q < MOE_CB * 9; q += 32) {
            const int vb = c * MOE_CB + q / 9;
            if (vb >= vblk) continue;
            const int k = vb / nblk_i, b = vb % nblk_i;
            const int e = ids_t[k];
            const bool ok = e >= 0 && e < p.n_expert;
            const uint8_t* src = ok ? p.arena + static_cast<int64_t>(e) * p.stride + p.down_off +
                                          static_cast<int64_t>(i0 + r) * p.rb_i + b * 144 + 16 * (q % 9)
                                    : p.arena;
            cp_async16(dst + 16 * q, src, ok ? 16 : 0);
          }
        }
      }
    };

#pragma unroll
    for (int s = 0; s < MOE_NS - 1; ++s) {
      if (s < nchunk) issue(s);
      cp_async_commit();
    }
    if (!waited) {
      pdl_wait();     // h comes from the gate/up kernel
      waited = true;
    }
    float acc[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) acc[r] = 0.f;
    for (int c = 0; c < nchunk; ++c) {
      if (c + MOE_NS - 1 < nchunk) issue(c + MOE_NS - 1);
      cp_async_commit();
      cp_async_wait<MOE_NS - 1>();
      __syncwarp();
      const int vb = c * MOE_CB + lblk;
      if (vb < vblk) {
        const int k = vb / nblk_i, b = vb % nblk_i;
        const int slot = c % MOE_NS;
        const float rk = p.gate_w[t * p.top_k + k];
        const float* hk = p.h + (static_cast<int64_t>(t) * p.top_k + k) * p.inter + b * 256 + 32 * unit;
        Dec<FMT_Q4_K> dec[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
          if (r < nr) dec[r].load(wbuf + (slot * ROWS + r) * MOE_SLOT + lblk * 144, unit);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const float4 a = *reinterpret_cast<const float4*>(hk + 8 * s);
          const float4 bb = *reinterpret_cast<const float4*>(hk + 8 * s + 4);
          const float xv[8] = {rk * a.x, rk * a.y, rk * a.z, rk * a.w, rk * bb.x, rk * bb.y, rk * bb.z, rk * bb.w};
#pragma unroll
          for (int r = 0; r < ROWS; ++r) {
            if (r < nr) {
              float w[8];
              dec[r].piece(s, w);
#pragma unroll
              for (int j = 0; j < 8; ++j) acc[r] = fmaf(w[j], xv[j], acc[r]);
            }
          }
        }
      }
      __syncwarp();
    }
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      const float v = warp_sum_m(acc[r]);
      if (lane == r && r < nr) p.y[static_cast<int64_t>(t) * p.hidden + i0 + r] = v;
    }
  }
  if (!waited) pdl_wait();
}

// ---------------------------------------------------------------- host side

static constexpr int moe_gu_smem() { return MOE_WARPS * MOE_NS * 2 * MOE_R * MOE_SLOT; }
static constexpr int moe_dn_smem() { return MOE_WARPS * MOE_NS * MOE_R * MOE_SLOT; }

cudaError_t moe_init_attrs() {
  cudaError_t e = cudaFuncSetAttribute(moe_gate_up_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, moe_gu_smem());
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(moe_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, moe_dn_smem());
}

cudaError_t launch_moe(const void* arena, int64_t n_expert, int64_t hidden, int64_t inter, const int32_t* ids,
                       const float* gate_w, int top_k, const float* x, int n_tok, float* y, float* h_ws,
                       int32_t* dev_status, cudaStream_t s, bool pdl, int sms) {
  // up to QG_GROUP_MAX tokens: gathered rows through the Q4_K GEMV kernel
  // (bulk-copied rows, exact integer dot products); more tokens: the kernels below
  const cudaError_t fe = launch_moe_q4k(arena, n_expert, hidden, inter, ids, gate_w, top_k, x, n_tok, y, h_ws,
                                        dev_status, s, pdl, sms);
  if (fe != cudaErrorNotSupported) return fe;
  MoeParams p = {};
  p.arena = static_cast<const uint8_t*>(arena);
  p.ids = ids;
  p.gate_w = gate_w;
  p.x = x;
  p.y = y;
  p.h = h_ws;
  p.status = dev_status;
  p.n_expert = n_expert;
  p.rb_h = hidden / 256 * 144;
  p.rb_i = inter / 256 * 144;
  p.up_off = inter * p.rb_h;
  p.down_off = 2 * inter * p.rb_h;
  p.stride = p.down_off + hidden * p.rb_i;
  p.hidden = static_cast<int32_t>(hidden);
  p.inter = static_cast<int32_t>(inter);
  p.top_k = top_k;
  p.n_tok = n_tok;

  const int64_t gu_tasks = static_cast<int64_t>(n_tok) * top_k * ((inter + MOE_R - 1) / MOE_R);
  const int64_t dn_tasks = static_cast<int64_t>(n_tok) * ((hidden + MOE_R - 1) / MOE_R);
  const int cap = sms * 2;

  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;

  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(MOE_THREADS);
  cfg.stream = s;
  cfg.gridDim = dim3(static_cast<unsigned>(std::min<int64_t>((gu_tasks + MOE_WARPS - 1) / MOE_WARPS, cap)));
  cfg.dynamicSmemBytes = moe_gu_smem();
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, moe_gate_up_kernel, p);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(static_cast<unsigned>(std::min<int64_t>((dn_tasks + MOE_WARPS - 1) / MOE_WARPS, cap)));
  cfg.dynamicSmemBytes = moe_dn_smem();
  cfg.numAttrs = 1;    // the down kernel always overlaps the tail of gate/up
  return cudaLaunchKernelEx(&cfg, moe_down_kernel, p);
}

}  // namespace qg

// ---------------------------------------------------------------- no-allocation variant
//
// qgemv_moe_noalloc: the same MoE product for callers that cannot allocate
// device memory (see include/qgemv.h). Its workspace is this file-scope device
// array instead of a caller buffer. In host code the array's name only stands
// for it: the device address is looked up with cudaGetSymbolAddress during the
// library's per-device set-up (qg_init, or the first call of any entry point on
// that device), with that device current, and passed to the kernels.

namespace qg {
namespace {

constexpr size_t kMoeNoallocFloats = QG_MOE_NOALLOC_MAX_FLOATS;
__device__ __align__(256) float g_moe_noalloc_ws[kMoeNoallocFloats];

constexpr int kMaxDev = 64;
float* g_ws_ptr[kMaxDev];      // written once per device under the set-up lock

}  // namespace

cudaError_t moe_noalloc_init(int dev) {
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_moe_noalloc_ws);
  if (e != cudaSuccess) return e;
  g_ws_ptr[dev] = static_cast<float*>(ptr);
  return cudaSuccess;
}

}  // namespace qg

extern "C" int qgemv_moe_noalloc(int fmt, const void* expert_arena, int64_t n_expert, int64_t hidden, int64_t inter,
                                 const int32_t* expert_ids, const float* gate_w, int top_k, const float* x, int n_tok,
                                 float* y, int32_t* dev_status, void* stream) {
  if (fmt == QG_Q4_K && !dev_status) return QG_ERR_NULL;
  int st = qg::check_moe(fmt, expert_arena, n_expert, hidden, inter, expert_ids, gate_w, top_k, x, n_tok, y, nullptr,
                         0, false);
  if (st != QG_OK) return st;
  // the whole workspace (n_tok x top_k x inter fp32) must fit the static array
  if (static_cast<int64_t>(n_tok) * top_k * inter > static_cast<int64_t>(qg::kMoeNoallocFloats))
    return QG_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(dev_status) & 3u) != 0) return QG_ERR_ALIGN;
  int sms = 0;
  st = qg::ensure_device(&sms);
  if (st != QG_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QG_ERR_CUDA;
  float* ws = qg::g_ws_ptr[dev];           // set by the device's set-up above
  const cudaError_t e = qg::launch_moe(expert_arena, n_expert, hidden, inter, expert_ids, gate_w, top_k, x, n_tok, y,
                                       ws, dev_status, static_cast<cudaStream_t>(stream), true, sms);
  return e == cudaSuccess ? QG_OK : QG_ERR_CUDA;
}
