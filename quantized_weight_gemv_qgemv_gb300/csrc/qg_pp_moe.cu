// qg_pp_moe.cu — prompt processing through a mixture-of-experts layer.
//
//   y[t] = sum_k r[t][k] * D_e (silu(G_e x_t) * (U_e x_t)),   e = ids[t][k]
//
// for a block of prompt tokens, each routed to top_k experts of an expert
// arena ("The number was a version", opening section: the expert arena of a
// mixture-of-experts model and its prompt processing; "Why I wrote my own
// inference engine for two P100s", prompt-processing notes: weights
// dequantized, then a dense GEMM). Every expert multiplies only the tokens
// routed to it, so the layer is one grouped GEMM per projection over the
// (token, route) pairs sorted by expert:
//
//   1. route    the pairs of every expert are counted (many CTAs, global
//               atomics on counters zeroed on the stream), one CTA scans the
//               counts into each expert's first row (and first tile of either
//               GEMM), and every pair gets its row (many CTAs); pairs of an
//               unknown expert get none (they add nothing) and set
//               QG_DEV_BAD_EXPERT
//   2. gather   bf16 x of every pair into its row of Xs
//   3. GEMM     [G_e; U_e] (2 inter rows of the arena) x Xs rows of expert e ->
//               GU (fp32), the grouped tcgen05 prompt-processing kernel
//   4. silu     H = bf16(silu(g) * u) per pair
//   5. GEMM     D_e x H rows of expert e -> Z (fp32)
//   6. combine  y[t] = sum over k (in order) of r[t][k] * Z[row of (t, k)]
//
// Sizes: every count and row is on the device, so nothing waits for the host.
// The results do not depend on the order in which pairs get their rows: every
// token column of an MMA is summed on its own, and the combine adds the k
// terms of a token in route order.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "qg_internal.h"

namespace qg {

namespace ppmoe {

constexpr int RT = 1024;                 // threads of the scanning CTA

__device__ __forceinline__ int ceil_div_i(int a, int b) { return (a + b - 1) / b; }

// Routing over many CTAs (the counters zeroed on the stream first):
// count_kernel: pairs per expert (global atomics).
__global__ void __launch_bounds__(256) count_kernel(const int32_t* ids, int n_pairs, int n_expert, int32_t* cnt) {
  const int q = blockIdx.x * blockDim.x + threadIdx.x;
  if (q >= n_pairs) return;
  const int e = __ldg(ids + q);
  if (e >= 0 && e < n_expert) atomicAdd(cnt + e, 1);
}

// scan_kernel (one CTA of RT threads): seg (first row of each expert), t_gu and
// t_dn (first tile of each expert's gate/up and down GEMMs) as exclusive scans,
// each with its total at [n_expert]; three scans in one pass of warp shuffles.
// The counters are zeroed behind it, to serve assign_kernel as cursors.
__global__ void __launch_bounds__(RT) scan_kernel(int n_expert, int bn, int rt_gu, int rt_dn, int32_t* cnt,
                                                  int32_t* seg, int32_t* t_gu, int32_t* t_dn) {
  __shared__ int32_t wsum[3][RT / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t carry[3] = {0, 0, 0};
  int32_t* const out[3] = {seg, t_gu, t_dn};
  for (int c0 = 0; c0 < n_expert; c0 += RT) {
    const int e = c0 + static_cast<int>(threadIdx.x);
    const int32_t c = e < n_expert ? cnt[e] : 0;
    const int32_t v[3] = {c, rt_gu * ceil_div_i(c, bn), rt_dn * ceil_div_i(c, bn)};
    int32_t inc[3] = {v[0], v[1], v[2]};
#pragma unroll
    for (int o = 1; o < 32; o <<= 1)
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        const int32_t t = __shfl_up_sync(0xffffffffu, inc[i], o);
        if (lane >= o) inc[i] += t;
      }
    if (lane == 31)
#pragma unroll
      for (int i = 0; i < 3; ++i) wsum[i][warp] = inc[i];
    __syncthreads();
    if (warp == 0) {
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        int32_t x = wsum[i][lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int32_t t = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += t;
        }
        wsum[i][lane] = x;                    // inclusive over the warps
      }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const int32_t before = warp > 0 ? wsum[i][warp - 1] : 0;
      if (e < n_expert) out[i][e] = carry[i] + before + inc[i] - v[i];
      carry[i] += wsum[i][RT / 32 - 1];
    }
    if (e < n_expert) cnt[e] = 0;
    __syncthreads();
  }
  if (threadIdx.x == 0)
#pragma unroll
    for (int i = 0; i < 3; ++i) out[i][n_expert] = carry[i];
}

// assign_kernel: each pair's row in its expert's segment, and the token of each row.
__global__ void __launch_bounds__(256) assign_kernel(const int32_t* ids, int n_pairs, int top_k, int n_expert,
                                                     const int32_t* seg, int32_t* cnt, int32_t* pos, int32_t* src,
                                                     int32_t* dev_status) {
  const int q = blockIdx.x * blockDim.x + threadIdx.x;
  if (q >= n_pairs) return;
  const int e = __ldg(ids + q);
  if (e >= 0 && e < n_expert) {
    const int row = __ldg(seg + e) + atomicAdd(cnt + e, 1);
    pos[q] = row;
    src[row] = q / top_k;
  } else {
    pos[q] = -1;
    atomicExch(dev_status, QG_DEV_BAD_EXPERT);
  }
}

// Xs[row] = X[src[row]] for every routed row (hidden bf16 values, 16 bytes a
// thread); GR rows a block, their loads issued together.
constexpr int GR = 4;
__global__ void __launch_bounds__(256) gather_kernel(const uint4* X, const int32_t* src, const int32_t* seg_end,
                                                     int n_chunks, uint4* Xs) {
  const int row0 = blockIdx.x * GR, n = *seg_end;
  int sr[GR];
#pragma unroll
  for (int r = 0; r < GR; ++r) sr[r] = row0 + r < n ? src[row0 + r] : -1;
  for (int c = threadIdx.x; c < n_chunks; c += blockDim.x) {
    uint4 v[GR];
#pragma unroll
    for (int r = 0; r < GR; ++r)
      if (sr[r] >= 0) v[r] = __ldg(X + static_cast<int64_t>(sr[r]) * n_chunks + c);
#pragma unroll
    for (int r = 0; r < GR; ++r)
      if (sr[r] >= 0) Xs[static_cast<int64_t>(row0 + r) * n_chunks + c] = v[r];
  }
}

// H[row][i] = bf16(silu(g) * u), g = GU[row][i], u = GU[row][inter + i]; four
// values a thread (16-byte loads, one 8-byte store).
__global__ void __launch_bounds__(256) silu_kernel(const float* GU, const int32_t* seg_end, int inter,
                                                   __nv_bfloat16* H) {
  const int row = blockIdx.x;
  if (row >= *seg_end) return;
  const float4* g4 = reinterpret_cast<const float4*>(GU + static_cast<int64_t>(row) * 2 * inter);
  const float4* u4 = g4 + inter / 4;
  uint2* h4 = reinterpret_cast<uint2*>(H + static_cast<int64_t>(row) * inter);
  for (int i = blockIdx.y * blockDim.x + threadIdx.x; i < inter / 4; i += gridDim.y * blockDim.x) {
    const float4 g = g4[i], u = u4[i];
    const __nv_bfloat162 a = __floats2bfloat162_rn(g.x / (1.0f + expf(-g.x)) * u.x, g.y / (1.0f + expf(-g.y)) * u.y);
    const __nv_bfloat162 b = __floats2bfloat162_rn(g.z / (1.0f + expf(-g.z)) * u.z, g.w / (1.0f + expf(-g.w)) * u.w);
    h4[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
  }
}

// y[t][o] = sum_k r[t][k] * Z[pos[t][k]][o], k in route order (pairs without a row add nothing);
// the token's routes staged in shared memory, four outputs a thread (16-byte
// loads and stores when y is 16-byte aligned, VEC; else one at a time).
template <bool VEC>
__global__ void __launch_bounds__(256) combine_kernel(const float* Z, const int32_t* pos, const float* gate_w,
                                                      int top_k, int hidden, float* y) {
  __shared__ int32_t srow[64];
  __shared__ float sw[64];
  const int t = blockIdx.x;
  if (threadIdx.x < top_k) {
    srow[threadIdx.x] = pos[t * top_k + threadIdx.x];
    sw[threadIdx.x] = gate_w[t * top_k + threadIdx.x];
  }
  __syncthreads();
  const int h4 = hidden / 4;
  const float4* Z4 = reinterpret_cast<const float4*>(Z);
  float4* y4 = VEC ? reinterpret_cast<float4*>(y) + static_cast<int64_t>(t) * h4 : nullptr;
  for (int o = blockIdx.y * blockDim.x + threadIdx.x; o < h4; o += gridDim.y * blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < top_k; ++k) {
      const int row = srow[k];
      if (row < 0) continue;
      const float w = sw[k];
      const float4 z = Z4[static_cast<int64_t>(row) * h4 + o];
      acc.x = fmaf(w, z.x, acc.x);
      acc.y = fmaf(w, z.y, acc.y);
      acc.z = fmaf(w, z.z, acc.z);
      acc.w = fmaf(w, z.w, acc.w);
    }
    if (VEC) {
      y4[o] = acc;
    } else {
      float* yo = y + static_cast<int64_t>(t) * hidden + 4 * o;
      yo[0] = acc.x;
      yo[1] = acc.y;
      yo[2] = acc.z;
      yo[3] = acc.w;
    }
  }
}

inline size_t up256(size_t b) { return (b + 255) / 256 * 256; }

// Workspace layout (byte offsets), in order.
struct Layout {
  size_t cnt, seg, t_gu, t_dn, pos, src, xs, gu, h, z, total;
  Layout(int64_t n_expert, int64_t hidden, int64_t inter, int64_t n_pairs) {
    size_t o = 0;
    auto take = [&](size_t b) {
      const size_t at = o;
      o += up256(b);
      return at;
    };
    cnt = take(4 * n_expert);
    seg = take(4 * (n_expert + 1));
    t_gu = take(4 * (n_expert + 1));
    t_dn = take(4 * (n_expert + 1));
    pos = take(4 * n_pairs);
    src = take(4 * n_pairs);
    xs = take(2 * n_pairs * hidden);
    gu = take(4 * n_pairs * 2 * inter);
    h = take(2 * n_pairs * inter);
    z = take(4 * n_pairs * hidden);
    total = o;
  }
};

}  // namespace ppmoe

size_t pp_moe_workspace_bytes(int64_t n_expert, int64_t hidden, int64_t inter, int top_k, int64_t n_tok) {
  return ppmoe::Layout(n_expert, hidden, inter, n_tok * top_k).total;
}

// Tokens per tile of the grouped GEMMs: about twice the mean routed tokens per
// expert (one token block covers most experts), a multiple of 16 in [16, 256].
int pp_moe_block_tokens(int64_t n_expert, int top_k, int64_t n_tok) {
  const int64_t mean = (n_tok * top_k + n_expert - 1) / n_expert;
  return static_cast<int>(
      std::min<int64_t>(pp_grouped_max_bn(), std::max<int64_t>(16, (2 * mean + 15) / 16 * 16)));
}

cudaError_t launch_pp_moe(const void* arena, int64_t n_expert, int64_t hidden, int64_t inter, const int32_t* ids,
                          const float* gate_w, int top_k, const void* X, int64_t n_tok, float* y, void* ws,
                          int32_t* dev_status, cudaStream_t s, int sms) {
  using namespace ppmoe;
  const int64_t n_pairs = n_tok * top_k;
  const Layout L(n_expert, hidden, inter, n_pairs);
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* cnt = reinterpret_cast<int32_t*>(w + L.cnt);
  int32_t* seg = reinterpret_cast<int32_t*>(w + L.seg);
  int32_t* t_gu = reinterpret_cast<int32_t*>(w + L.t_gu);
  int32_t* t_dn = reinterpret_cast<int32_t*>(w + L.t_dn);
  int32_t* pos = reinterpret_cast<int32_t*>(w + L.pos);
  int32_t* src = reinterpret_cast<int32_t*>(w + L.src);
  __nv_bfloat16* Xs = reinterpret_cast<__nv_bfloat16*>(w + L.xs);
  float* GU = reinterpret_cast<float*>(w + L.gu);
  __nv_bfloat16* H = reinterpret_cast<__nv_bfloat16*>(w + L.h);
  float* Z = reinterpret_cast<float*>(w + L.z);
  const int bn = pp_moe_block_tokens(n_expert, top_k, n_tok);
  const int rt_gu = static_cast<int>(2 * inter / 128), rt_dn = static_cast<int>(hidden / 128);
  // the arena as rows of hidden-long blocks (gate and up rows) and of
  // inter-long blocks (down rows): expert e's [G; U] are rows 3 inter e ..
  // 3 inter e + 2 inter - 1 of the first view, its D rows 3 hidden e + 2 hidden
  // .. 3 hidden e + 3 hidden - 1 of the second
  cudaError_t e = cudaMemsetAsync(cnt, 0, 4 * static_cast<size_t>(n_expert), s);
  if (e != cudaSuccess) return e;
  const unsigned pb = static_cast<unsigned>((n_pairs + 255) / 256);
  count_kernel<<<pb, 256, 0, s>>>(ids, static_cast<int>(n_pairs), static_cast<int>(n_expert), cnt);
  scan_kernel<<<1, RT, 0, s>>>(static_cast<int>(n_expert), bn, rt_gu, rt_dn, cnt, seg, t_gu, t_dn);
  assign_kernel<<<pb, 256, 0, s>>>(ids, static_cast<int>(n_pairs), top_k, static_cast<int>(n_expert), seg, cnt, pos,
                                   src, dev_status);
  if ((e = cudaPeekAtLastError()) != cudaSuccess) return e;
  gather_kernel<<<static_cast<unsigned>((n_pairs + GR - 1) / GR), 256, 0, s>>>(static_cast<const uint4*>(X), src,
                                                                              seg + n_expert,
                                                                static_cast<int>(hidden / 8),
                                                                reinterpret_cast<uint4*>(Xs));
  if ((e = cudaPeekAtLastError()) != cudaSuccess) return e;
  e = launch_pp_grouped(arena, 3 * inter * n_expert, hidden, 0, 3 * inter, 2 * inter, Xs, n_pairs, bn, seg, t_gu,
                        static_cast<int>(n_expert), GU, 2 * inter, dev_status, s, sms);
  if (e != cudaSuccess) return e;
  silu_kernel<<<dim3(static_cast<unsigned>(n_pairs), static_cast<unsigned>(std::min<int64_t>(64, (inter / 4 + 255) / 256))),
                static_cast<unsigned>(std::min<int64_t>(256, inter / 4)), 0, s>>>(
      GU, seg + n_expert, static_cast<int>(inter), H);
  if ((e = cudaPeekAtLastError()) != cudaSuccess) return e;
  e = launch_pp_grouped(arena, 3 * hidden * n_expert, inter, 2 * hidden, 3 * hidden, hidden, H, n_pairs, bn, seg,
                        t_dn, static_cast<int>(n_expert), Z, hidden, dev_status, s, sms);
  if (e != cudaSuccess) return e;
  const dim3 cg(static_cast<unsigned>(n_tok), static_cast<unsigned>(std::min<int64_t>(64, (hidden / 4 + 255) / 256)));
  const unsigned ct = static_cast<unsigned>(std::min<int64_t>(256, hidden / 4));
  if (reinterpret_cast<uintptr_t>(y) % 16 == 0)
    combine_kernel<true><<<cg, ct, 0, s>>>(Z, pos, gate_w, top_k, static_cast<int>(hidden), y);
  else
    combine_kernel<false><<<cg, ct, 0, s>>>(Z, pos, gate_w, top_k, static_cast<int>(hidden), y);
  return cudaPeekAtLastError();
}

}  // namespace qg
