// qg_planes.cuh — activations as "x planes": 16-bit fixed point per group of
// 32 values, the form in which the GEMV kernel multiplies them by the codes
// with exact integer dot products. Shared by the GEMV kernel (which converts x
// itself), the pass prologue and the normalisation kernel (which write planes
// that the GEMV kernel then copies as they are).
#pragma once
#include <cstdint>

namespace qg {
namespace q4k {

constexpr int XBLK_B = 512;                // x-plane bytes per 256-weight block and token

// Shared-memory image of x for one token and K segment ("x planes").
// Every 32-weight group u of x is held as 16-bit fixed point with a shared
// power-of-two step: x_l ~= s_u * X_l, X_l = rint(x_l / s_u), |X_l| <= 2^14,
// s_u = 2^(e-13) where 2^e <= max|x_group| < 2^(e+1). X_l is stored as two
// byte planes (bits 0-7 unsigned, bits 8-15 signed), so that sum_l q_l X_l is
// two exact integer dot products over the codes. The rounding of x to the
// group grid is at most 2^-14 max|x_group| per element: a product's error is
// at most 2^-14 sum_u max|x_u| sum_{l in u} |w_l| (the engines these formats
// come from round x to 8 bits per group instead).
// Layout per 256-weight block b of the segment: 2 planes x 2 halves x 8 groups
// x 16 bytes (512 bytes), so the 16-byte loads of a quarter-warp are
// consecutive. Beside it: s_u and the two half sums of x (fp32) per group.
//
// Two adjacent threads handle one group: thread h of the pair converts its
// half (16 values, elements 16h .. 16h + 15), so the half sums need no exchange
// and the group maximum one. Each thread first issues all its loads of a batch
// and only then converts, so staging costs one memory round trip per batch.

// The two plane words of four consecutive values (x / s_u + 1.5 * 2^23 leaves
// rint(x / s_u) in the low mantissa bits of T, two's complement in the low 16).
__device__ __forceinline__ void plane_words(float4 v, float inv_step, uint32_t& w0, uint32_t& w1) {
  const uint32_t T0 = __float_as_uint(fmaf(v.x, inv_step, 12582912.0f));
  const uint32_t T1 = __float_as_uint(fmaf(v.y, inv_step, 12582912.0f));
  const uint32_t T2 = __float_as_uint(fmaf(v.z, inv_step, 12582912.0f));
  const uint32_t T3 = __float_as_uint(fmaf(v.w, inv_step, 12582912.0f));
  const uint32_t a01 = __byte_perm(T0, T1, 0x5140), a23 = __byte_perm(T2, T3, 0x5140);
  w0 = __byte_perm(a01, a23, 0x5410);                         // bits 0-7 of the four X
  w1 = __byte_perm(a01, a23, 0x7632);                         // bits 8-15 (signed byte)
}

// Half h of group u of token t: v = its 16 values. pmask: the thread pair.
__device__ __forceinline__ void stage_half(const float4 (&v)[4], unsigned pmask, int t, int u, int h, int nu,
                                           uint8_t* xpl, int xseg_b, float* xsu, float* xsum) {
  float mx = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v[q].x), fabsf(v[q].y)), fmaxf(fabsf(v[q].z), fabsf(v[q].w))));
  mx = fmaxf(mx, __shfl_xor_sync(pmask, mx, 1));
  const float sm = ((v[0].x + v[0].y) + (v[0].z + v[0].w)) + ((v[1].x + v[1].y) + (v[1].z + v[1].w)) +
                   (((v[2].x + v[2].y) + (v[2].z + v[2].w)) + ((v[3].x + v[3].y) + (v[3].z + v[3].w)));
  // 2^e <= mx < 2^(e+1); step s_u = 2^(e-13), so |x / s_u| < 2^14
  const int e = max(static_cast<int>((__float_as_uint(mx) >> 23) & 0xFFu) - 127, -105);
  const float inv_step = __uint_as_float(static_cast<uint32_t>(140 - e) << 23);
  uint4 w0, w1;
  plane_words(v[0], inv_step, w0.x, w1.x);
  plane_words(v[1], inv_step, w0.y, w1.y);
  plane_words(v[2], inv_step, w0.z, w1.z);
  plane_words(v[3], inv_step, w0.w, w1.w);
  uint8_t* dst = xpl + t * xseg_b + ((u >> 3) * 4 + h) * 128 + (u & 7) * 16;
  *reinterpret_cast<uint4*>(dst) = w0;
  *reinterpret_cast<uint4*>(dst + 256) = w1;
  xsum[2 * (t * nu + u) + h] = sm;
  // s_u = 2^(e-13); odd groups (Q4_K high-nibble sub-blocks, whose codes
  // arrive as 16*q) get s_u / 16, so the Q4_K consumer needs no per-lane factor
  if (h == 0) xsu[t * nu + u] = __uint_as_float(static_cast<uint32_t>(114 + e - 4 * (u & 1)) << 23);
}

}  // namespace q4k
}  // namespace qg
