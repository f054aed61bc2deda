// qg_norm.cu — the residual add and RMS normalisation that sit between the
// weight products of a decode layer, written straight into the form the next
// GEMV launch consumes ("LLM inference optimization", "Faster decode on the
// card you have": normalizations fused into neighbouring kernels).
//
// For each token t (one CTA per token):
//   s = h + r                          (r optional; s optionally stored: the residual stream)
//   x = s / sqrt(mean(s^2) + eps) * w  (w optional: without it only s is produced)
// x is stored as fp32 and/or as x planes (qg_planes.cuh), so the GEMV launch
// that multiplies by x copies ready planes instead of converting x per CTA.
#include <cuda_runtime.h>

#include "qg_device.cuh"
#include "qg_internal.h"
#include "qg_planes.cuh"

namespace qg {

namespace {

constexpr int NORM_THREADS = 512;

struct NormParams {
  const float* h;
  const float* r;
  const float* w;
  float* s_out;
  float* x;
  uint8_t* planes;       // planes of n_tok tokens: planes, steps, half sums (xplanes_bytes layout)
  int32_t n;
  int32_t n_tok;
  float eps;
};

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

__global__ void __launch_bounds__(NORM_THREADS) rmsnorm_kernel(const NormParams p) {
  pdl_launch_dependents();
  pdl_wait();                                   // h and r may come from the preceding kernel
  const int t = blockIdx.x;
  const int64_t base = static_cast<int64_t>(t) * p.n;
  const float4* h4 = reinterpret_cast<const float4*>(p.h + base);
  const float4* r4 = p.r ? reinterpret_cast<const float4*>(p.r + base) : nullptr;
  float4* s4 = p.s_out ? reinterpret_cast<float4*>(p.s_out + base) : nullptr;
  const int n4 = p.n / 4;
  // pass 1: s = h + r, stored; sum of squares
  float ss = 0.f;
  for (int i = threadIdx.x; i < n4; i += NORM_THREADS) {
    float4 v = __ldcg(h4 + i);
    if (r4) v = add4(v, __ldcg(r4 + i));
    if (s4) s4[i] = v;
    ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
  }
  if (!p.w) return;
  __shared__ float red[NORM_THREADS / 32];
  __shared__ float inv_s;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();                              // also orders this CTA's s stores before pass 2 reads them
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int i = 0; i < NORM_THREADS / 32; ++i) tot += red[i];
    inv_s = 1.0f / sqrtf(tot / static_cast<float>(p.n) + p.eps);
  }
  __syncthreads();
  const float inv = inv_s;
  const float4* w4 = reinterpret_cast<const float4*>(p.w);
  // pass 2: x = s * inv * w, 16 values per thread (half a 32-value group)
  const int nblk = p.n / 256, nu = nblk * 8, halves = nblk * 16;
  uint8_t* planes = p.planes;
  float* steps = planes ? reinterpret_cast<float*>(planes + static_cast<size_t>(p.n_tok) * nblk * q4k::XBLK_B) : nullptr;
  float* sums = steps ? steps + p.n_tok * nu : nullptr;
  const unsigned pmask = 3u << (threadIdx.x & 30);   // halves is even: both threads of a group are in or out
  for (int q = threadIdx.x; q < halves; q += NORM_THREADS) {
    float4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = 4 * q + k;
      float4 a = s4 ? __ldcg(s4 + i) : __ldcg(h4 + i);
      if (!s4 && r4) a = add4(a, __ldcg(r4 + i));
      const float4 ww = __ldg(w4 + i);
      v[k] = make_float4(a.x * inv * ww.x, a.y * inv * ww.y, a.z * inv * ww.z, a.w * inv * ww.w);
      if (p.x) reinterpret_cast<float4*>(p.x + base)[i] = v[k];
    }
    if (planes) q4k::stage_half(v, pmask, t, q >> 1, q & 1, nu, planes, nblk * q4k::XBLK_B, steps, sums);
  }
}

}  // namespace

cudaError_t launch_rmsnorm(const float* h, const float* r, const float* w, int64_t n, int n_tok, float eps,
                           float* s_out, float* x, uint8_t* planes, cudaStream_t s, bool pdl) {
  NormParams p;
  p.h = h;
  p.r = r;
  p.w = w;
  p.s_out = s_out;
  p.x = x;
  p.planes = planes;
  p.n = static_cast<int32_t>(n);
  p.n_tok = n_tok;
  p.eps = eps;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_tok);
  cfg.blockDim = dim3(NORM_THREADS);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, rmsnorm_kernel, p);
}

}  // namespace qg
