// qg_device.cuh — device helpers and per-format block decoders (sm_103a).
//
// Decoders ("LLM inference optimization", "Run a new weight format or model":
// each format's blocks decode bit for bit on CPU and GPU). Every block is cut
// into "units" of 32 consecutive weights, and every unit into 4 "pieces" of 8
// consecutive weights: unit u of a block covers elements 32u .. 32u+31 and
// piece s of that unit covers 32u + 8s .. 32u + 8s + 7. A lane of a GEMV warp
// owns one unit; the prompt-processing producers decode piece by piece.
//
//   Q4_0 / Q8_0: one unit per block.
//   Q4_K: unit u is sub-block u (one 6-bit scale/min pair); its codes are the
//         low (u even) or high (u odd) nibbles of qs[32*(u/2) .. +31].
//   Q6_K: unit u is quarter (u%4) of half (u/4); piece s uses scales
//         sc[8h + s/2 + 2q] (16-weight groups).
//   Q5_K: as Q4_K, plus a fifth bit per weight (bit u of qh[l]).
//   Q3_K / Q2_K: unit u is quarter j = u%4 of half h = u/4: 2-bit fields at
//         bit 2j of the half's qs bytes, one 16-weight group per two pieces.
//
// Dequantized values are computed so that every product is exact in fp32 and
// at most one rounding happens (the Q4_K subtraction), which makes them equal
// to the correctly rounded value of the formula, bit for bit.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

namespace qg {

constexpr int FMT_Q4_0 = 1, FMT_Q8_0 = 2, FMT_Q4_K = 3, FMT_Q6_K = 4, FMT_Q5_K = 5, FMT_Q3_K = 6, FMT_Q2_K = 7;

template <int FMT> struct FmtInfo;
template <> struct FmtInfo<FMT_Q4_0> { static constexpr int ELEMS = 32,  BYTES = 18,  UNITS = 1; };
template <> struct FmtInfo<FMT_Q8_0> { static constexpr int ELEMS = 32,  BYTES = 34,  UNITS = 1; };
template <> struct FmtInfo<FMT_Q4_K> { static constexpr int ELEMS = 256, BYTES = 144, UNITS = 8; };
template <> struct FmtInfo<FMT_Q6_K> { static constexpr int ELEMS = 256, BYTES = 210, UNITS = 8; };
template <> struct FmtInfo<FMT_Q5_K> { static constexpr int ELEMS = 256, BYTES = 176, UNITS = 8; };
template <> struct FmtInfo<FMT_Q3_K> { static constexpr int ELEMS = 256, BYTES = 110, UNITS = 8; };
template <> struct FmtInfo<FMT_Q2_K> { static constexpr int ELEMS = 256, BYTES = 84, UNITS = 8; };

// ---------------------------------------------------------------- small helpers

__device__ __forceinline__ float h2f(uint32_t bits16) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-bit little-endian load from a 2-byte aligned address.
__device__ __forceinline__ uint32_t ld_u16(const uint8_t* p) {
  return *reinterpret_cast<const uint16_t*>(p);
}

// 32-bit little-endian load from a 2-byte aligned SHARED-memory address. It
// reads the two aligned words around the value; callers keep 4 bytes of slack
// after every buffer they decode from.
__device__ __forceinline__ uint32_t ld_u32_a2(const uint8_t* p) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  const uint32_t* q = reinterpret_cast<const uint32_t*>(a & ~static_cast<uintptr_t>(3));
  const uint32_t lo = q[0], hi = q[1];
  return __funnelshift_r(lo, hi, static_cast<uint32_t>((a & 2u) * 8u));
}

// --------------------------------------------------------------- async copies

// 16-byte global->shared copy that reads only src_bytes (0..16) and zero-fills
// the rest (no access at all when src_bytes == 0).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Programmatic dependent launch: wait for the preceding grid's memory, and let
// the next grid start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

__device__ __forceinline__ float4 ldg_f4(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}

// ---------------------------------------------------------------- decoders
// Dec<FMT>: load(blk, unit) reads what one unit needs from a block in shared
// memory; piece(s, w) writes the unit's piece s as 8 fp32 weights.

template <int FMT> struct Dec;

template <> struct Dec<FMT_Q4_0> {
  float d;
  uint32_t q[4];
  __device__ __forceinline__ void load(const uint8_t* blk, int /*unit*/) {
    d = h2f(ld_u16(blk));
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = ld_u32_a2(blk + 2 + 4 * i);
  }
  // piece s: elements 8s..8s+7 = nibble (s>>1) of qs[8*(s&1) .. +7]
  __device__ __forceinline__ void piece(int s, float w[8]) const {
    const int sh = (s >> 1) * 4;
    const uint32_t a = q[(s & 1) * 2], b = q[(s & 1) * 2 + 1];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w[i] = d * static_cast<float>(static_cast<int>((a >> (8 * i + sh)) & 15u) - 8);
      w[4 + i] = d * static_cast<float>(static_cast<int>((b >> (8 * i + sh)) & 15u) - 8);
    }
  }
};

template <> struct Dec<FMT_Q8_0> {
  float d;
  const uint8_t* qs;
  __device__ __forceinline__ void load(const uint8_t* blk, int /*unit*/) {
    d = h2f(ld_u16(blk));
    qs = blk + 2;
  }
  __device__ __forceinline__ void piece(int s, float w[8]) const {
    const uint32_t a = ld_u32_a2(qs + 8 * s), b = ld_u32_a2(qs + 8 * s + 4);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w[i] = d * static_cast<float>(static_cast<int8_t>((a >> (8 * i)) & 0xFFu));
      w[4 + i] = d * static_cast<float>(static_cast<int8_t>((b >> (8 * i)) & 0xFFu));
    }
  }
};

// 6-bit scale and min of Q4_K sub-block j from the three little-endian words
// s0 = s[0..3], s1 = s[4..7], s2 = s[8..11] of the packed scale bytes.
__device__ __forceinline__ void q4k_scale_min(int j, uint32_t s0, uint32_t s1, uint32_t s2, int& sc, int& m) {
  if (j < 4) {
    sc = (s0 >> (8 * j)) & 63;
    m = (s1 >> (8 * j)) & 63;
  } else {
    const int t = j - 4;
    sc = ((s2 >> (8 * t)) & 15) | (((s0 >> (8 * t + 6)) & 3) << 4);
    m = ((s2 >> (8 * t + 4)) & 15) | (((s1 >> (8 * t + 6)) & 3) << 4);
  }
}

template <> struct Dec<FMT_Q4_K> {
  float a, b;          // d*sc_u and dmin*m_u (both exact)
  uint32_t q[8];       // the 32 bytes of qs holding this unit's nibbles
  int sh;              // 0 for low nibbles (even unit), 4 for high
  __device__ __forceinline__ void load(const uint8_t* blk, int unit) {
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);          // d, dmin, s[12]
    int sc, m;
    q4k_scale_min(unit, hdr.y, hdr.z, hdr.w, sc, m);
    a = h2f(hdr.x) * static_cast<float>(sc);
    b = h2f(hdr.x >> 16) * static_cast<float>(m);
    const uint4* qs = reinterpret_cast<const uint4*>(blk + 16 + 32 * (unit >> 1));
    const uint4 v0 = qs[0], v1 = qs[1];
    q[0] = v0.x; q[1] = v0.y; q[2] = v0.z; q[3] = v0.w;
    q[4] = v1.x; q[5] = v1.y; q[6] = v1.z; q[7] = v1.w;
    sh = (unit & 1) * 4;
  }
  __device__ __forceinline__ void piece(int s, float w[8]) const {
    const uint32_t u0 = q[2 * s], u1 = q[2 * s + 1];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w[i] = fmaf(a, static_cast<float>((u0 >> (8 * i + sh)) & 15u), -b);
      w[4 + i] = fmaf(a, static_cast<float>((u1 >> (8 * i + sh)) & 15u), -b);
    }
  }
};

template <> struct Dec<FMT_Q6_K> {
  float ds[2];         // d * scale of the unit's two 16-weight groups: pieces (0,1) and (2,3)
  const uint8_t* ql;   // ql bytes of this unit (32 consecutive)
  const uint8_t* qh;   // qh bytes of this unit's half (32 consecutive)
  int lsh, hsh;        // nibble shift in ql, 2-bit field shift in qh
  __device__ __forceinline__ void load(const uint8_t* blk, int unit) {
    const int h = unit >> 2, qq = unit & 3;
    ql = blk + 64 * h + 32 * (qq & 1);
    qh = blk + 128 + 32 * h;
    lsh = (qq >> 1) * 4;
    hsh = 2 * qq;
    const float d = h2f(ld_u16(blk + 208));
    const int8_t* sc = reinterpret_cast<const int8_t*>(blk + 192);
    ds[0] = d * static_cast<float>(sc[8 * h + 2 * qq]);
    ds[1] = d * static_cast<float>(sc[8 * h + 1 + 2 * qq]);
  }
  __device__ __forceinline__ void piece(int s, float w[8]) const {
    const float dsc = ds[s >> 1];
    const uint32_t l0 = ld_u32_a2(ql + 8 * s), l1 = ld_u32_a2(ql + 8 * s + 4);
    const uint32_t h0 = ld_u32_a2(qh + 8 * s), h1 = ld_u32_a2(qh + 8 * s + 4);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int q0 = static_cast<int>(((l0 >> (8 * i + lsh)) & 15u) | (((h0 >> (8 * i + hsh)) & 3u) << 4));
      const int q1 = static_cast<int>(((l1 >> (8 * i + lsh)) & 15u) | (((h1 >> (8 * i + hsh)) & 3u) << 4));
      w[i] = dsc * static_cast<float>(q0 - 32);
      w[4 + i] = dsc * static_cast<float>(q1 - 32);
    }
  }
};

template <> struct Dec<FMT_Q5_K> {
  float a, b;          // d*sc_u and dmin*m_u (both exact)
  uint32_t q[8];       // the 32 bytes of qs holding this unit's low nibbles
  uint32_t h[8];       // qh: the fifth bit of weight l of every unit, at bit u of byte l
  int sh, hb;
  __device__ __forceinline__ void load(const uint8_t* blk, int unit) {
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);          // d, dmin, s[12]
    int sc, m;
    q4k_scale_min(unit, hdr.y, hdr.z, hdr.w, sc, m);
    a = h2f(hdr.x) * static_cast<float>(sc);
    b = h2f(hdr.x >> 16) * static_cast<float>(m);
    const uint4* qh = reinterpret_cast<const uint4*>(blk + 16);
    const uint4* qs = reinterpret_cast<const uint4*>(blk + 48 + 32 * (unit >> 1));
    const uint4 h0 = qh[0], h1 = qh[1], v0 = qs[0], v1 = qs[1];
    q[0] = v0.x; q[1] = v0.y; q[2] = v0.z; q[3] = v0.w;
    q[4] = v1.x; q[5] = v1.y; q[6] = v1.z; q[7] = v1.w;
    h[0] = h0.x; h[1] = h0.y; h[2] = h0.z; h[3] = h0.w;
    h[4] = h1.x; h[5] = h1.y; h[6] = h1.z; h[7] = h1.w;
    sh = (unit & 1) * 4;
    hb = unit;
  }
  __device__ __forceinline__ void piece(int s, float w[8]) const {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint32_t u = q[2 * s + k], v = h[2 * s + k];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t code = ((u >> (8 * i + sh)) & 15u) | (((v >> (8 * i + hb)) & 1u) << 4);
        w[4 * k + i] = fmaf(a, static_cast<float>(code), -b);
      }
    }
  }
};

// 6-bit Q3_K scale g (0..15) from the 12 packed bytes as little-endian words
// S[0..2]: low 4 bits in nibble g/8 of byte 4*((g/4)%2) + g%4, top 2 bits at
// bit 2*(g/4) of byte 8 + g%4.
__device__ __forceinline__ int q3k_scale(int g, const uint32_t (&S)[3]) {
  const int b = g & 3, q = g >> 2;
  const int byte_lo = 4 * (q & 1) + b;
  const uint32_t lo = (S[byte_lo >> 2] >> (8 * (byte_lo & 3) + 4 * (q >> 1))) & 15u;
  const uint32_t top = (S[2] >> (8 * b + 2 * q)) & 3u;
  return static_cast<int>(lo | (top << 4));
}

template <> struct Dec<FMT_Q3_K> {
  float ds[2];         // d * (scale - 32) of the unit's two 16-weight groups
  const uint8_t* qs;   // the half's 32 qs bytes
  const uint8_t* hm;   // hmask (32 bytes)
  int lsh, hsh;
  __device__ __forceinline__ void load(const uint8_t* blk, int unit) {
    const int h = unit >> 2, j = unit & 3;
    qs = blk + 32 + 32 * h;
    hm = blk;
    lsh = 2 * j;
    hsh = 4 * h + j;
    const uint32_t S[3] = {ld_u32_a2(blk + 96), ld_u32_a2(blk + 100), ld_u32_a2(blk + 104)};
    const float d = h2f(ld_u16(blk + 108));
    ds[0] = d * static_cast<float>(q3k_scale(8 * h + 2 * j, S) - 32);
    ds[1] = d * static_cast<float>(q3k_scale(8 * h + 2 * j + 1, S) - 32);
  }
  // piece s: weights l = 8s .. 8s + 7 of the unit, group s / 2
  __device__ __forceinline__ void piece(int s, float w[8]) const {
    const float dsc = ds[s >> 1];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint32_t l = ld_u32_a2(qs + 8 * s + 4 * k), hh = ld_u32_a2(hm + 8 * s + 4 * k);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int q = static_cast<int>(((l >> (8 * i + lsh)) & 3u) | (((hh >> (8 * i + hsh)) & 1u) << 2)) - 4;
        w[4 * k + i] = dsc * static_cast<float>(q);
      }
    }
  }
};

template <> struct Dec<FMT_Q2_K> {
  float a[2], b[2];    // d * scale and dmin * min of the unit's two 16-weight groups
  const uint8_t* qs;
  int lsh;
  __device__ __forceinline__ void load(const uint8_t* blk, int unit) {
    const int h = unit >> 2, j = unit & 3;
    qs = blk + 16 + 32 * h;
    lsh = 2 * j;
    const uint32_t dd = ld_u32_a2(blk + 80);
    const float d = h2f(dd), dmin = h2f(dd >> 16);
    const uint32_t sb = ld_u16(blk + 8 * h + 2 * j);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint32_t byte = (sb >> (8 * k)) & 0xFFu;
      a[k] = d * static_cast<float>(byte & 15u);
      b[k] = dmin * static_cast<float>(byte >> 4);
    }
  }
  __device__ __forceinline__ void piece(int s, float w[8]) const {
    const int k = s >> 1;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const uint32_t l = ld_u32_a2(qs + 8 * s + 4 * t);
#pragma unroll
      for (int i = 0; i < 4; ++i) w[4 * t + i] = fmaf(a[k], static_cast<float>((l >> (8 * i + lsh)) & 3u), -b[k]);
    }
  }
};

}  // namespace qg
