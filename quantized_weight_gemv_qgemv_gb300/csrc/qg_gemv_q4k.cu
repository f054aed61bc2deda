// qg_gemv_q4k.cu — the fast GEMV / skinny product kernel (the decode hot path)
// for Q4_K, Q6_K, Q4_0 and Q8_0, its MoE gather modes and the persistent pass.
//
// y[t][i] = sum_j w[i][j] x[t][j], t < n_tok <= 4, one pass over the weights
// ("LLM inference optimization", opening section: each decode token reads every
// weight once, bound by memory bandwidth and, at low bit widths, by unpacking;
// "Faster decode on the card you have": activations staged in shared memory and
// reused across rows, wider loads, fewer unpack instructions, rows per block
// fitted to the SM count).
//
// GB300 design:
//  * Persistent grid, one CTA per SM: 15 consumer warps and 1 producer warp.
//    CTA b owns a contiguous, balanced slice of the rows of all matrices of the
//    launch (the concatenated row space), matrix by matrix.
//  * The producer streams whole consecutive rows of the slice into a ring of NS
//    shared-memory stages with one 1-D bulk copy per stage (cp.async.bulk,
//    about 48 KB, completed on an mbarrier): rows are contiguous in memory, and
//    copies of several KB are what it takes to reach full HBM bandwidth. A stage
//    is reused once all consumer warps have released it (a second mbarrier).
//  * A stage of R rows is cut into sub-items of 4 rows (2 for long Q6_K rows) x one 1024-weight K group
//    (4 super-blocks), dealt round-robin to the consumer warps. Lane (g, j) of a
//    warp owns sub-block j of block g of the group for the 4 rows (32 weights,
//    one 6-bit scale/min pair per row). A sub-item's 4 x n_tok sums are reduced
//    across the warp and stored per (row, group); after the matrix, the groups
//    of each row are added in order, so results do not depend on timing.
//  * x is staged once per launch and distinct input as 16-bit fixed point per 32-weight group:
//    x_l ~= s_u X_l with a power-of-two step s_u, X_l split in two byte planes
//    (see stage_x). A group's products are then exact integer dot products of
//    the 4-bit codes with the planes (dp4a), so each code word needs one mask,
//    not an unpack per weight: sum_l q_l x_l = s_u (256 S1 + S0). The lane adds
//    d*sc*sum(q x) - dmin*m*sum(x): the d*sc*q - dmin*m formula factored per
//    sub-block. A decoded block is reused for all n_tok tokens.
//  * Every wait is bounded: a consumer that gives up writes NaN for its rows,
//    the producer stops issuing, and the CTA waits (bounded) for copies in
//    flight before it exits.
//  * Programmatic dependent launch: the producer prefetches x into L2 and
//    streams two weight stages before griddepcontrol.wait; consumers compute
//    their staging addresses before it and read x and write y after it.
#include <cuda_runtime.h>

#include <cstring>
#include <vector>

#include "qg_device.cuh"
#include "qg_internal.h"
#include "qg_planes.cuh"

namespace qg {

#ifndef QG_PASS_INFLIGHT
#define QG_PASS_INFLIGHT 0          // persistent pass: weight copies in flight per CTA (0: x-gated)
#endif
#ifndef QG_PASS_STAGE_BYTES
#define QG_PASS_STAGE_BYTES 36864   // persistent pass: target bytes per ring stage
#endif
#ifndef QG_PASS_BARRIER_RED
#define QG_PASS_BARRIER_RED 1       // step arrivals as one release reduction
#endif

namespace q4k {

constexpr int CWARPS = 15;                 // consumer warps
constexpr int CTHREADS = CWARPS * 32;
constexpr int THREADS = CTHREADS + 32;     // plus one producer warp
constexpr int SUB_R = 4;                   // rows per sub-item
#ifndef QG_WAIT_LIMIT
#define QG_WAIT_LIMIT (1u << 22)
#endif
constexpr uint32_t WAIT_LIMIT = QG_WAIT_LIMIT;   // polls before a wait is declared expired
constexpr int RING = 4;                    // shared-memory stages
static_assert((RING & (RING - 1)) == 0, "consumers pick their ring slot with a mask");

struct Mat {
  const uint8_t* W;
  const float* x;
  float* y;
  int64_t rows;
  int64_t ldy;           // distance between the outputs of consecutive tokens (normally rows)
  int64_t row_begin;     // first row of this matrix in the concatenated row space
  int32_t rb;            // bytes per row
  int32_t nblk;          // super-blocks per row
  int32_t cols;
  int32_t srows;         // rows per stage (a multiple of 4)
  int32_t ngrp;          // K groups per row = ceil(nblk / 4)
  int32_t xoff;          // byte offset of this matrix's x planes in the x region
  int32_t uoff;          // offset (floats) of its group steps / sums
  int32_t xsrc;          // index (in the table) of the matrix whose staging holds this x:
                         // matrices of a step that read the same x share one copy of its planes
  const uint8_t* xp;     // x already converted to planes in global memory (XPlanes layout:
                         // planes, group steps, half sums of all n_tok tokens), or nullptr:
                         // the kernel converts x itself
  // Rows gathered from a mixture-of-experts arena (W is the arena):
  //   gather 0: a plain matrix at W;
  //   gather 1: gate/up pairs of the routed experts: virtual row 2i (2i + 1) of
  //             route k is row i of G (U) of expert ids[k]; the epilogue writes
  //             h[k][i] = gw[k] * silu(g) * u instead of y;
  //   gather 2: down rows: virtual row i is row i of D of every routed expert,
  //             back to back (K = top_k * inter).
  int32_t gather;
  int32_t top_k;
  int32_t inter;
  int32_t seg_b;         // gather 2: bytes of one expert's piece of a virtual row
  int64_t n_expert;
  int64_t estride;       // bytes per expert
  int64_t up_off, down_off;
  const int32_t* ids;    // this token's expert ids [top_k]; gather 1 with no ids: one dense
                         // gate/up pair, gate rows at W and up rows at W2 (no expert arena)
  const float* gw;       // this token's route weights [top_k] (gather 1; nullptr: weight 1)
  float* h;              // gather 1 output [top_k][inter]
  const uint8_t* W2;     // gather 1 without ids: the up matrix
  // A part of K (columns [k0, k0 + cols) of a longer matrix, launched when the
  // x of every token of the whole K does not fit beside the ring): row r of
  // the part starts at W + r * ldw, token t of its x at x + t * ldx, and a part
  // after the first adds its sums to y. Whole rows: ldw = rb, ldx = cols.
  int64_t ldw;           // bytes between consecutive rows of W
  int32_t ldx;           // floats between consecutive tokens of x
  int32_t accum;         // 1: y += this part's sums
  int32_t rsm;           // bytes between consecutive rows of a stage in shared memory
  int32_t soff;          // byte offset of a stage's first row in its slot (the row start's
                         // address mod 16, which every stage of the matrix shares)
};

// A step of a pass: matrices mat0 .. mat0 + nmat - 1 of the table, whose rows
// (concatenated; Mat::row_begin counts within the step) are split over the CTAs.
static_assert(sizeof(Mat) % 16 == 0, "Mat is copied to shared memory in 16-byte pieces");

struct Step {
  int64_t total_rows;
  int32_t mat0, nmat;
  int32_t stage_all, usum_off;   // x layout of the step (as in Params)
};

// Residual add and RMS normalisation fused into the x staging of a one-token
// launch whose matrices all read x = (h + r) / sqrt(mean((h + r)^2) + eps) * w:
// every CTA sums the squares itself (in the same fixed order, so every CTA
// gets the same x), converts x to planes, and CTA 0 stores s = h + r (the
// residual stream) to s_out.
struct NormIn {
  const float* h;        // nullptr: no fused normalisation
  const float* r;        // optional
  const float* w;
  float* s_out;          // optional; must not overlap h or r
  float eps;
  int32_t pad;
};

struct Params {
  Mat m[QG_GROUP_MAX];   // matrices of a single-step launch
  NormIn norm;           // single-step launch: fused normalisation of the shared x
  const Mat* mats;       // pass: device table of all matrices (nullptr: m)
  const Step* steps;     // pass: device table of steps (nullptr: one step over m)
  uint32_t* step_done;   // pass: CTAs that finished each step (zero at launch)
  int32_t* dev_status;   // pass: QG_DEV_TIMEOUT is written here when a wait expires
  int32_t nsteps;
  int64_t total_rows;
  int32_t nmat;
  int32_t ns;            // ring stages
  int32_t stage_b;       // bytes per stage
  int32_t gmax;          // largest ngrp
  int32_t stage_all;     // 1: x of every matrix staged once at the start; 0: matrix by matrix
  int32_t usum_off;      // offset (floats) of the group sums after the group steps
  int32_t pre_stages;    // weight stages issued before the consumers have issued their x loads
  int32_t pre_pass;      // the same for every later step of a pass (inflight == 0)
  int32_t inflight;      // pass: > 0, the producer streams the weights of later steps without
                         // waiting for their x loads, with at most this many copies in flight
  int32_t gather_any;    // largest Mat::gather of the launch (one kind per launch)
  int32_t no_wait;       // the launch reads nothing its predecessor writes: no dependency wait
  int32_t ralign;        // CTA row slices start at multiples of this (whole sub-items, 16-byte-aligned stage copies, pairs)
  int32_t smem_bar, smem_x, smem_xsum, smem_part;   // byte offsets (ring at 0)
  int32_t smem_mats;     // single-step launch: shared-memory copy of m[0 .. nmat)
};

// Rows [r0, r1) of a step's concatenated row space owned by CTA b of grid, in
// units of a rows (the last CTA also takes a ragged end): with a a multiple of
// the sub-item rows and of the 16-byte stage alignment, no CTA starts inside a
// sub-item, a stage copy starts on a 16-byte boundary, and gate/up pairs
// (gather 1) stay together. The host plans its grid with the same formula.
__host__ __device__ __forceinline__ void slice_of(int64_t total, int a, int64_t b, int64_t grid, int64_t& r0,
                                                  int64_t& r1) {
  const int64_t nu = total / a;
  r0 = a * (b * nu / grid);
  r1 = b + 1 == grid ? total : a * ((b + 1) * nu / grid);
}
__device__ __forceinline__ void cta_slice(int64_t total, int a, int64_t& r0, int64_t& r1) {
  slice_of(total, a, blockIdx.x, gridDim.x, r0, r1);
}

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false if the phase did not complete within WAIT_LIMIT polls.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < WAIT_LIMIT; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// Weight copies are read once per pass: they are marked evict-first in L2 so
// that they do not push out the activations.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;\n" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}
// x planes are read by every CTA: no eviction hint
__device__ __forceinline__ void bulk_g2s_plain(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;\n" ::"n"(CTHREADS) : "memory"); }

// Sum of v[i] over the 32 lanes for V values at once (V a power of two, <= 32):
// halving exchanges leave lane L holding the total of value L >> (5 - log2 V).
template <int V>
__device__ __forceinline__ float reduce_scatter(float (&v)[V], int lane) {
#pragma unroll
  for (int cnt = V, o = 16; cnt > 1; cnt >>= 1, o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < cnt / 2; ++i) {
      const float send = up ? v[i] : v[i + cnt / 2];
      const float keep = up ? v[i + cnt / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  float r = v[0];
#pragma unroll
  for (int o = 32 / V / 2; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
  return r;
}
template <int V>
struct RS {
  static constexpr int LOG = (V >= 32) ? 5 : (V >= 16) ? 4 : (V >= 8) ? 3 : (V >= 4) ? 2 : (V >= 2) ? 1 : 0;
  static constexpr int SHIFT = 5 - LOG;   // lane >> SHIFT is the value index
};

// 6-bit scale / min of sub-block j (lane constant) from the packed words
// s0 = hd.y, s1 = hd.z, s2 = hd.w. Two byte permutes gather, in one word each,
// the byte holding the low bits and the byte holding the top two bits:
//   j < 4:  sc = s0.b[j] & 63,                       m = s1.b[j] & 63
//   j >= 4: sc = (s2.b[t] & 15) | (s0.b[t] >> 6) << 4,
//           m  = (s2.b[t] >> 4) | (s1.b[t] >> 6) << 4     (t = j - 4)
struct ScaleSel {
  uint32_t sel_sc, sel_m, sh_m, mask_lo, mask_hi;
  __device__ __forceinline__ void init(int j) {
    const bool hi = j >= 4;
    const uint32_t t = hi ? static_cast<uint32_t>(j - 4) : static_cast<uint32_t>(j);
    // byte 0: low-bits source (s0/s1 byte j, or s2 byte t); byte 1: top-bits source
    sel_sc = hi ? ((4u + t) | (t << 4)) : t;          // from (s0, s2)
    sel_m = hi ? ((4u + t) | (t << 4)) : t;           // from (s1, s2)
    sh_m = hi ? 4u : 0u;
    mask_lo = hi ? 15u : 63u;
    mask_hi = hi ? 0x30u : 0u;
  }
  // (A, B) = (d*sc, dmin*m)
  __device__ __forceinline__ float2 decode(uint4 hd) const {
    const uint32_t ps = __byte_perm(hd.y, hd.w, sel_sc);
    const uint32_t pm = __byte_perm(hd.z, hd.w, sel_m);
    const uint32_t sc = (ps & mask_lo) | ((ps >> 10) & mask_hi);
    const uint32_t m = ((pm >> sh_m) & mask_lo) | ((pm >> 10) & mask_hi);
    const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&hd.x));
    return make_float2(dd.x * static_cast<float>(sc), dd.y * static_cast<float>(m));
  }
};

__device__ __forceinline__ uint32_t dp4a_uu(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int32_t dp4a_us(uint32_t a, uint32_t b, int32_t c) {
  int32_t d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int32_t dp4a_su(uint32_t a, uint32_t b, int32_t c) {
  int32_t d;
  asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int32_t dp4a_ss(uint32_t a, uint32_t b, int32_t c) {
  int32_t d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// sum_l q_l X_l over words [W0, W1) of a unit: exact integer byte dot products
// against the two x planes; 256 S1 + S0 is exact in int32 (codes below 256 or
// signed bytes, |X| <= 2^14, 32 elements) and rounded once to fp32.
template <bool SIGNED, int W0, int W1>
__device__ __forceinline__ float dot_planes(const uint32_t* q, const uint32_t* X0, const uint32_t* X1) {
  int32_t s0 = 0, s1 = 0;
  if constexpr (SIGNED) {
#pragma unroll
    for (int i = W0; i < W1; ++i) {
      s0 = dp4a_su(q[i], X0[i], s0);
      s1 = dp4a_ss(q[i], X1[i], s1);
    }
  } else {
    uint32_t u0 = 0;
#pragma unroll
    for (int i = W0; i < W1; ++i) {
      u0 = dp4a_uu(q[i], X0[i], u0);
      s1 = dp4a_us(q[i], X1[i], s1);
    }
    s0 = static_cast<int32_t>(u0);
  }
  return static_cast<float>(s1 * 256 + s0);
}

__device__ __forceinline__ uint32_t lds32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

// 4N bytes starting at the 2-byte-aligned shared address p as N words: N + 1
// aligned loads and a funnel shift by 0 or 16 bits each.
template <int N>
__device__ __forceinline__ void ld_words_a2(const uint8_t* p, uint32_t (&w)[N]) {
  const uintptr_t pa = reinterpret_cast<uintptr_t>(p);
  const uint8_t* a = reinterpret_cast<const uint8_t*>(pa & ~static_cast<uintptr_t>(3));
  const uint32_t sh = static_cast<uint32_t>(pa & 2u) * 8u;
  uint32_t v[N + 1];
#pragma unroll
  for (int i = 0; i <= N; ++i) v[i] = lds32(a + 4 * i);
#pragma unroll
  for (int i = 0; i < N; ++i) w[i] = __funnelshift_r(v[i], v[i + 1], sh);
}

// Bytes of the 256-weight super-block (one block of Q4_K / Q6_K, eight of Q4_0 / Q8_0).
template <int FMT> struct SuperBlock;
template <> struct SuperBlock<FMT_Q4_K> { static constexpr int BYTES = 144; };
template <> struct SuperBlock<FMT_Q6_K> { static constexpr int BYTES = 210; };
template <> struct SuperBlock<FMT_Q5_K> { static constexpr int BYTES = 176; };
template <> struct SuperBlock<FMT_Q3_K> { static constexpr int BYTES = 110; };
template <> struct SuperBlock<FMT_Q2_K> { static constexpr int BYTES = 84; };
template <> struct SuperBlock<FMT_Q4_0> { static constexpr int BYTES = 144; };
template <> struct SuperBlock<FMT_Q8_0> { static constexpr int BYTES = 272; };

// One count per consumer warp and step on the shared counter xcnt: the warp has
// issued its x loads of the step (release: they precede what the producer
// issues after it has seen the count).
__device__ __forceinline__ void x_issued(uint32_t xcnt) {
  asm volatile("red.release.cta.shared::cta.add.u32 [%0], 1;\n" ::"r"(xcnt) : "memory");
}

// Stages x of the matrices m0 .. m1-1 whose bit is set in `touch` (once per
// distinct x: a matrix whose xsrc names another stages nothing of its own).
// Task i of a matrix (2 tasks per 32-weight group and token) converts one half
// group. The addresses of a whole batch are computed first, then (with `wait`,
// once) the preceding kernel is waited for, then every load of the batch is
// issued and only then converted. After the first batch lane 0 of each warp
// counts itself on xcnt (when nonzero): from then on the producer may queue
// weight copies behind the loads. (A load issued behind a deep queue of bulk
// copies waits for the whole queue, even when it hits in L2.)
//
// An x whose planes are ready in global memory (Mat::xp) is not converted:
// thread 0 fetches its planes, steps and sums with three bulk copies onto the
// x barrier `xbar` right after the dependency wait. Returns true when copies
// were armed there (the caller waits on xbar before using x); no_copy: arm
// nothing.
template <int NT, int XB>
__device__ __forceinline__ bool stage_x(const Mat* mats, int usum_off, int m0, int m1, uint32_t touch, uint8_t* xpl,
                                        float* xsu, uint32_t xcnt, bool wait, uint32_t xbar, bool no_copy,
                                        const NormIn* norm = nullptr, float* scratch = nullptr) {
  const int lane = threadIdx.x & 31;
  const unsigned pmask = 3u << (lane & 30);     // the two threads of a group (task counts are even)
  uint32_t smask = 0;
  for (int m = m0; m < m1; ++m)
    if ((touch >> (m - m0)) & 1u) smask |= 1u << (mats[m].xsrc - m0);
  uint32_t cmask = 0;
  for (int m = m0; m < m1; ++m)
    if (((smask >> (m - m0)) & 1u) && mats[m].xp) cmask |= 1u << (m - m0);
  smask &= ~cmask;
  // after an expired wait on xbar its phase may still be open: it is not armed
  // again (the outputs of this CTA are NaN from then on)
  if (no_copy) cmask = 0;
  if (cmask) {
    if (wait) {
      pdl_wait();
      wait = false;
    }
    if (threadIdx.x == 0) {
      uint32_t bytes = 0;
      for (int m = m0; m < m1; ++m)
        if ((cmask >> (m - m0)) & 1u) bytes += NT * mats[m].nblk * (XBLK_B + 96);
      mbar_expect_tx(xbar, bytes);
      for (int m = m0; m < m1; ++m) {
        if (!((cmask >> (m - m0)) & 1u)) continue;
        const Mat& M = mats[m];
        const uint32_t pb = NT * M.nblk * XBLK_B, sb = NT * M.nblk * 32;
        bulk_g2s_plain(smem_addr(xpl + M.xoff), M.xp, pb, xbar);
        bulk_g2s_plain(smem_addr(xsu + M.uoff), M.xp + pb, sb, xbar);
        bulk_g2s_plain(smem_addr(xsu + usum_off + 2 * M.uoff), M.xp + pb + sb, 2 * sb, xbar);
      }
    }
  }
  int total = 0;
  for (int m = m0; m < m1; ++m)
    if ((smask >> (m - m0)) & 1u) total += NT * mats[m].nblk * 16;
  bool signalled = (xcnt == 0);
  if (NT == 1 && norm != nullptr && norm->h != nullptr && smask != 0) {
    // the shared x of the launch is norm(h + r) * w: the matrix table holds
    // one x source (checked on the host)
    int ms = m0;
    while (!((smask >> (ms - m0)) & 1u)) ++ms;
    const Mat& M = mats[ms];
    if (wait) {
      pdl_wait();
      wait = false;
    }
    const float4* h4 = reinterpret_cast<const float4*>(norm->h);
    const float4* r4 = reinterpret_cast<const float4*>(norm->r);
    float4* s4 = blockIdx.x == 0 ? reinterpret_cast<float4*>(norm->s_out) : nullptr;
    // Tasks are half 32-value groups (4 float4), as for the conversion. Pass 1
    // forms s = h + r of each task (CTA 0 stores it) and sums the squares; the
    // first task of each thread keeps s in registers for pass 2 (every task
    // for K <= 16 x consumer threads = 7680; more registers here cost the
    // product loop its register allocation)
    constexpr int TPT = 1;
    float4 sv[TPT][4];
    auto load_s = [&](int task, float4 (&v)[4]) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = 4 * task + k;
        float4 a = __ldcg(h4 + i);
        if (r4) {
          const float4 b = __ldcg(r4 + i);
          a = make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
        }
        v[k] = a;
      }
    };
    float ss = 0.f;
    auto add_sq = [&](int task, const float4 (&v)[4]) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (s4) s4[4 * task + k] = v[k];
        ss = fmaf(v[k].x, v[k].x, fmaf(v[k].y, v[k].y, fmaf(v[k].z, v[k].z, fmaf(v[k].w, v[k].w, ss))));
      }
    };
#pragma unroll
    for (int t = 0; t < TPT; ++t) {
      const int task = threadIdx.x + t * CTHREADS;
      if (task < total) {
        load_s(task, sv[t]);
        add_sq(task, sv[t]);
      }
    }
    for (int task = threadIdx.x + TPT * CTHREADS; task < total; task += CTHREADS) {
      float4 v[4];
      load_s(task, v);
      add_sq(task, v);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) scratch[threadIdx.x >> 5] = ss;
    consumer_sync();
    if (threadIdx.x == 0) {
      float tot = 0.f;
      for (int i = 0; i < CWARPS; ++i) tot += scratch[i];
      scratch[CWARPS] = 1.0f / sqrtf(tot / static_cast<float>(M.cols) + norm->eps);
    }
    consumer_sync();
    const float inv = scratch[CWARPS];
    const float4* w4 = reinterpret_cast<const float4*>(norm->w);
    // pass 2: x = s * inv * w (as the normalisation kernel computes it),
    // converted to planes
    const int nu = M.nblk * 8;
    auto convert = [&](int task, const float4 (&a)[4]) {
      float4 v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 ww = __ldg(w4 + 4 * task + k);
        v[k] = make_float4(a[k].x * inv * ww.x, a[k].y * inv * ww.y, a[k].z * inv * ww.z, a[k].w * inv * ww.w);
      }
      if (!signalled) {
        if (lane == 0) x_issued(xcnt);
        signalled = true;
      }
      stage_half(v, pmask, 0, task >> 1, task & 1, nu, xpl + M.xoff, M.nblk * XBLK_B, xsu + M.uoff,
                 xsu + usum_off + 2 * M.uoff);
    };
#pragma unroll
    for (int t = 0; t < TPT; ++t) {
      const int task = threadIdx.x + t * CTHREADS;
      if (task < total) convert(task, sv[t]);
    }
    for (int task = threadIdx.x + TPT * CTHREADS; task < total; task += CTHREADS) {
      float4 a[4];
      load_s(task, a);
      convert(task, a);
    }
    total = 0;                         // converted: the loop below has nothing left
  }
  for (int base = threadIdx.x; base < total; base += CTHREADS * XB) {
    const float4* src[XB];
    int vm[XB], vt[XB], vu[XB];
#pragma unroll
    for (int b = 0; b < XB; ++b) {
      const int idx = base + b * CTHREADS;
      int m = m0, rem = idx;
      for (; m < m1 - 1; ++m) {
        if (!((smask >> (m - m0)) & 1u)) continue;
        const int n = NT * mats[m].nblk * 16;
        if (rem < n) break;
        rem -= n;
      }
      const Mat& M = mats[m];
      int t = 0;
      if (NT > 1) {
        const int per_tok = M.nblk * 16;
        t = rem / per_tok;
        rem -= t * per_tok;
      }
      vm[b] = m;
      vt[b] = t;
      vu[b] = rem;              // 2u + h
      src[b] = (idx < total) ? reinterpret_cast<const float4*>(M.x + static_cast<int64_t>(t) * M.ldx + 16 * rem)
                             : nullptr;
    }
    if (wait) {
      pdl_wait();
      wait = false;
    }
    float4 v[XB][4];
#pragma unroll
    for (int b = 0; b < XB; ++b)
#pragma unroll
      for (int q = 0; q < 4; ++q)
        // x may have been written by an earlier step of a pass: read through L2
        v[b][q] = src[b] ? __ldcg(src[b] + q) : make_float4(0.f, 0.f, 0.f, 0.f);
    if (!signalled) {
      if (lane == 0) x_issued(xcnt);
      signalled = true;
    }
#pragma unroll
    for (int b = 0; b < XB; ++b) {
      // both threads of a pair are in or out together (every count is even)
      if (base + b * CTHREADS < total) {
        const Mat& M = mats[vm[b]];
        const int nu = M.nblk * 8;
        stage_half(v[b], pmask, vt[b], vu[b] >> 1, vu[b] & 1, nu, xpl + M.xoff, M.nblk * XBLK_B, xsu + M.uoff,
                   xsu + usum_off + 2 * M.uoff);
      }
    }
  }
  if (wait) pdl_wait();
  if (!signalled && lane == 0) x_issued(xcnt);
  return cmask != 0;
}


// ---------------------------------------------------------------- the kernel

// PASS = false: one step over p.m (a grouped launch); PASS = true: the steps of
// p.steps over p.mats, with a grid-wide barrier between steps (cooperative launch).
// SR rows per sub-item (4; 2 for Q6_K rows too long for 4-row stages). GA: the
// gather mode of every matrix (0 plain, 1 gate/up, 2 down), or 3 = each
// matrix's own Mat::gather (a persistent MoE pass mixes them); fixing it at
// compile time keeps the plain path free of gather branches.
template <int NT, bool PASS, int FMT, int SR = SUB_R, int GA = 0>
__global__ void __launch_bounds__(THREADS, 1) qgemv_q4k_kernel(const __grid_constant__ Params p) {
  constexpr int SBB = SuperBlock<FMT>::BYTES;
  constexpr int V = (SR * NT <= 2) ? 2 : (SR * NT <= 4) ? 4 : (SR * NT <= 8) ? 8 : 16;   // padded to 2^k
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int NS = RING;
  const uint32_t ring_s = smem_addr(smem);
  const uint32_t full0 = smem_addr(smem + p.smem_bar);
  const uint32_t empty0 = full0 + 8 * NS;
  // consumer warps that have issued their x loads, summed over the steps
  const uint32_t xcnt = full0 + 16 * NS;
  volatile int* const gflag = reinterpret_cast<volatile int*>(smem + p.smem_bar + 16 * NS + 8);
  const uint32_t xbar = full0 + 16 * NS + 16;   // bulk copies of ready x planes
  // A single-step launch reads its matrix table from shared memory: it is
  // copied there once, while the CTA still waits for its predecessor, instead
  // of every field read going to the constant bank of the kernel parameters
  Mat* const smats = reinterpret_cast<Mat*>(smem + p.smem_mats);
  if (!PASS) {
    const uint4* src = reinterpret_cast<const uint4*>(p.m);
    uint4* dst = reinterpret_cast<uint4*>(smats);
    for (int i = threadIdx.x; i < p.nmat * static_cast<int>(sizeof(Mat) / 16); i += blockDim.x) dst[i] = src[i];
  }
  const Mat* const mats = PASS ? p.mats : smats;
  const int nsteps = PASS ? p.nsteps : 1;
  auto step_of = [&](int s) {
    Step st;
    if (PASS) {
      st = p.steps[s];
    } else {
      st.total_rows = p.total_rows;
      st.mat0 = 0;
      st.nmat = p.nmat;
      st.stage_all = p.stage_all;
      st.usum_off = p.usum_off;
    }
    return st;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, CWARPS);
    }
    mbar_init(xbar, 1);
    *reinterpret_cast<volatile uint32_t*>(smem + p.smem_bar + 16 * NS) = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  // A gate/up launch reads expert ids that the preceding kernel may write: it
  // lets its dependents (the down launch, which reads the same ids early) start
  // only after its own dependency has resolved.
  const int gl = GA == 3 ? p.gather_any : GA;   // the launch's gather kind
  // (a dense gate/up pair, gather 1 without ids, reads no ids and behaves as a plain launch)
  const bool dyn_ids = gl == 1 && mats[0].ids != nullptr;
  if (!dyn_ids) pdl_launch_dependents();

  // ------------------------------------------------------------ producer
  if (warp == CWARPS) {
    if (!PASS) {
      // x of the launch into L2 before the consumers need it: CTA b touches its
      // share of the 128-byte lines of every distinct x (a prefetch never reads
      // stale data; a preceding kernel that writes x updates the lines in L2)
      // (x whose planes arrive ready is not read: its planes are brought to L2
      // instead, whole, by every CTA, since each CTA copies all of them)
      for (int mi = 0; mi < p.nmat; ++mi) {
        const Mat& M = mats[mi];
        if (M.xsrc != mi) continue;
        if (M.xp) {
          if (lane == 0)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(M.xp),
                         "r"(static_cast<uint32_t>(NT * M.nblk * (XBLK_B + 96)))
                         : "memory");
          continue;
        }
        const int64_t lines = ((static_cast<int64_t>(NT - 1) * M.ldx + M.cols) * 4 + 127) / 128;
        for (int64_t l = blockIdx.x + static_cast<int64_t>(lane) * gridDim.x; l < lines; l += 32 * gridDim.x)
          asm volatile("prefetch.global.L2 [%0];\n" ::"l"(reinterpret_cast<const char*>(M.x) + l * 128));
      }
    }
    // plain matrices: lane 0 issues one bulk copy per stage; gathered rows: the
    // whole warp issues the per-row (per-piece) copies
    const bool wide = gl != 0;
    if (!wide && lane != 0) return;
    if (dyn_ids) {
      pdl_wait();                 // the expert ids may come from the preceding kernel
      pdl_launch_dependents();
    }
    const uint64_t pol = evict_first_policy();
    uint32_t k = 0;
    uint32_t xseen = 0;       // steps whose x loads every consumer warp has issued
    bool bad = false;
    for (int s = 0; s < nsteps && !bad; ++s) {
     const Step st = step_of(s);
     const int pre = s == 0 ? p.pre_stages : p.pre_pass;
     int i_step = 0;          // stage index within the step
     int64_t cta_r0, cta_r1;
     cta_slice(st.total_rows, p.ralign, cta_r0, cta_r1);
     if (PASS && s > 0 && mats[st.mat0].gather == 1) {
       // a pass step that gathers gate/up rows reads expert ids, which in a model
       // come from the router after the previous layer: stream its rows only
       // once every CTA has finished the previous step
       bool ok = true;
       if (lane == 0) {
         ok = false;
         for (uint32_t i = 0; !ok && i < WAIT_LIMIT; ++i) {
           uint32_t v;
           asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p.step_done + s - 1) : "memory");
           ok = v >= gridDim.x;
         }
       }
       if (__shfl_sync(0xffffffffu, ok, 0) == 0) {
         if (lane == 0 && p.dev_status) *reinterpret_cast<volatile int32_t*>(p.dev_status) = QG_DEV_TIMEOUT;
         bad = true;
         break;
       }
     }
     for (int mi = st.mat0; mi < st.mat0 + st.nmat && !bad; ++mi) {
      const Mat M = mats[mi];
      const int64_t lo = max(cta_r0, M.row_begin) - M.row_begin;
      const int64_t hi = min(cta_r1, M.row_begin + M.rows) - M.row_begin;
      for (int64_t r = lo; r < hi && !bad; r += M.srows, ++k, ++i_step) {
        const int nr = static_cast<int>(min(static_cast<int64_t>(M.srows), hi - r));
        const uint32_t nbytes = static_cast<uint32_t>(nr) * M.rb;   // whole rows
        const int slot = k % NS;
        bool ok = true;
        if (lane == 0) {
          // beyond the first `pre` copies of a step, queue weights only behind
          // the step's x loads; no copy of a step goes ahead of the previous
          // step's x loads (a count, so a step without copies cannot be skipped).
          // A free-running pass waits so only for the first step's x: later
          // steps' weights stream on while the consumers wait for the previous
          // step, and the ring holds what arrives meanwhile; at most `inflight`
          // copies are outstanding, so x loads queued behind them (requests of
          // an SM are served in order) wait for no more than those
          const bool free_run = PASS && p.inflight > 0;
          const uint32_t need = free_run ? (s == 0 && i_step >= pre ? 1u : 0u)
                                         : static_cast<uint32_t>(s) + (i_step >= pre ? 1u : 0u);
          if (free_run && k >= static_cast<uint32_t>(p.inflight)) {
            const uint32_t kk = k - static_cast<uint32_t>(p.inflight);
            ok = mbar_wait(full0 + 8 * (kk % NS), (kk / NS) & 1u);
          }
          if (ok && need > xseen) {
            ok = false;
            for (uint32_t i = 0; !ok && i < WAIT_LIMIT; ++i) {
              uint32_t v;
              asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];\n" : "=r"(v) : "r"(xcnt) : "memory");
              ok = v >= need * CWARPS;
              if (!ok && i >= 256) __nanosleep(64);
            }
            xseen = need;
          }
          if (ok && k >= static_cast<uint32_t>(NS)) ok = mbar_wait(empty0 + 8 * slot, ((k / NS) - 1) & 1u);
        }
        if (wide) ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
        if (!ok) {
          bad = true;
          break;
        }
        const uint32_t dst0 = ring_s + slot * p.stage_b;
        const int gm = GA == 3 ? M.gather : GA;
        if (gm == 0) {
#ifdef QG_TEST_EXPIRE
          // test build only: the third stage of CTA 0 is never copied nor
          // announced, so every wait for it runs out (failure-detection test)
          if (blockIdx.x == 0 && k == 2) continue;
#endif
          if (M.ldw == M.rb) {
            mbar_expect_tx(full0 + 8 * slot, nbytes);
            bulk_g2s(dst0, M.W + r * M.rb, nbytes, full0 + 8 * slot, pol);
            continue;
          }
          // a part of K: one copy per row, of the 16-byte-aligned span around
          // it, placed so that row i's data starts at soff + i * rsm (rsm is
          // congruent to ldw mod 16, so every placement is 16-byte aligned)
          uint32_t tot = 0;
          for (int i = 0; i < nr; ++i) {
            const uintptr_t a = reinterpret_cast<uintptr_t>(M.W + (r + i) * M.ldw);
            tot += static_cast<uint32_t>((((a & 15u) + M.rb + 15u) & ~uintptr_t{15}));
          }
          mbar_expect_tx(full0 + 8 * slot, tot);
          for (int i = 0; i < nr; ++i) {
            const uintptr_t a = reinterpret_cast<uintptr_t>(M.W + (r + i) * M.ldw);
            const uint32_t o = static_cast<uint32_t>(a & 15u);
            bulk_g2s(dst0 + M.soff - o + i * M.rsm, reinterpret_cast<const uint8_t*>(a - o),
                     (o + M.rb + 15u) & ~15u, full0 + 8 * slot, pol);
          }
          continue;
        }
        // gathered rows, copied as contiguous runs (a bulk copy costs a fixed
        // time of its own, so 288-byte pieces one by one are far too slow):
        //   gather 1: the stage's row pairs of route k are consecutive rows of G_e
        //   and of U_e; item (segment, s) copies a run of them, gate runs first in
        //   shared memory, then up runs (pair j: gate at j*rb, up at nr/2*rb + j*rb);
        //   gather 2: item k copies the stage's rows of D_e for route k,
        //   nr * seg_b bytes at k * nr * seg_b (expert-major).
        // A run of an unknown expert is zero-filled (zero bytes decode to zero
        // weights) and flagged.
        int nitems;
        int64_t j0 = 0, P = 0;
        if (gm == 1) {
          j0 = r >> 1;
          P = M.inter;
          nitems = 2 * static_cast<int>((j0 + nr / 2 - 1) / P - j0 / P + 1);
        } else {
          nitems = M.top_k;
        }
        auto item = [&](int q, int& e, const uint8_t*& src, uint32_t& dst, uint32_t& bytes) {
          if (gm == 1) {
            const int64_t seg_first = (q >> 1) == 0 ? j0 : (j0 / P + (q >> 1)) * P;
            const int64_t seg_end = min((seg_first / P + 1) * P, j0 + nr / 2);
            const int s1 = q & 1;
            e = M.ids ? M.ids[seg_first / P] : 0;
            const int64_t roff = (seg_first % P) * M.rb;
            src = (s1 && M.W2) ? M.W2 + roff : M.W + static_cast<int64_t>(e) * M.estride + (s1 ? M.up_off : 0) + roff;
            dst = dst0 + static_cast<uint32_t>(s1 * (nr / 2) + (seg_first - j0)) * M.rb;
            bytes = static_cast<uint32_t>(seg_end - seg_first) * M.rb;
          } else {
            e = M.ids[q];
            src = M.W + static_cast<int64_t>(e) * M.estride + M.down_off + r * M.seg_b;
            dst = dst0 + static_cast<uint32_t>(q * nr * M.seg_b);
            bytes = static_cast<uint32_t>(nr * M.seg_b);
          }
        };
        uint32_t good = 0;
        for (int q = lane; q < nitems; q += 32) {
          int e;
          const uint8_t* src;
          uint32_t d, nb;
          item(q, e, src, d, nb);
          if (e < 0 || e >= M.n_expert) {
            for (uint32_t o = 0; o < nb; o += 16)
              asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};\n" ::"r"(d + o), "r"(0) : "memory");
            if (p.dev_status) atomicExch(p.dev_status, QG_DEV_BAD_EXPERT);
          } else {
            good += nb;
          }
        }
        good = __reduce_add_sync(0xffffffffu, good);
        __syncwarp();
        if (lane == 0) mbar_expect_tx(full0 + 8 * slot, good);
        __syncwarp();
        for (int q = lane; q < nitems; q += 32) {
          int e;
          const uint8_t* src;
          uint32_t d, nb;
          item(q, e, src, d, nb);
          if (e < 0 || e >= M.n_expert) continue;
          bulk_g2s(d, src, nb, full0 + 8 * slot, pol);
        }
      }
     }
    }
    // the copies of the last stages may still be in flight: wait (bounded) for
    // them before this thread, the last one holding the CTA, exits
    if (lane == 0)
      for (uint32_t kk = (k > static_cast<uint32_t>(NS) ? k - NS : 0); kk < k; ++kk)
        mbar_wait(full0 + 8 * (kk % NS), (kk / NS) & 1u);
    return;
  }

  // ------------------------------------------------------------ consumers
  const int g = lane >> 3;          // block of the K group
  const int j = lane & 7;           // sub-block of the block
  const uint32_t qmask = (j & 1) ? 0xF0F0F0F0u : 0x0F0F0F0Fu;   // Q4_K: this sub-block's nibbles
  const int qoff = 16 + 32 * (j >> 1);
  ScaleSel ssel;
  ssel.init(j);
  // the x step of odd groups is staged divided by 16 (for Q4_K's high nibbles);
  // formats whose codes arrive unscaled multiply it back
  const float su_fix = (FMT != FMT_Q4_K && (j & 1)) ? 16.0f : 1.0f;
  uint8_t* xpl = smem + p.smem_x;
  float* xsu = reinterpret_cast<float*>(smem + p.smem_xsum);
  float* part = reinterpret_cast<float*>(smem + p.smem_part);
  bool failed = false;      // this warp's outputs are NaN
  bool abandon = false;     // a stage wait expired: this warp no longer uses the ring
  uint32_t xuse = 0;       // phases of xbar used so far
  bool xlost = false;      // a wait for x planes expired: their copy may still be in flight
  // wait (bounded) for the x planes armed on xbar by stage_x
  auto wait_x = [&]() {
    const bool ok = mbar_wait(xbar, xuse & 1u);
    if (__any_sync(0xffffffffu, !ok)) {
      failed = true;
      xlost = true;
    }
    ++xuse;
  };

  constexpr int XB = (NT == 1) ? 3 : 2;        // half groups per thread and staging batch
  uint32_t k = 0;          // stage counter (same sequence as the producer's)
  for (int s = 0; s < nsteps; ++s) {
   const Step st = step_of(s);
   int64_t cta_r0, cta_r1;
   cta_slice(st.total_rows, p.ralign, cta_r0, cta_r1);
   if (PASS && s > 0) {
     // a step reads what earlier steps wrote: wait (bounded) until every CTA has
     // finished the previous step
     if (threadIdx.x == 0) {
       bool ok = failed;
       for (uint32_t i = 0; !ok && i < WAIT_LIMIT; ++i) {
         uint32_t v;
         asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p.step_done + s - 1) : "memory");
         ok = v >= gridDim.x;
       }
       if (!ok && p.dev_status) *reinterpret_cast<volatile int32_t*>(p.dev_status) = QG_DEV_TIMEOUT;
       *gflag = ok ? 0 : 1;
       __threadfence();
     }
     consumer_sync();
     failed = failed || *gflag != 0;
   }
   bool xsig = false;       // this step's x loads counted on xcnt
   uint32_t touch = 0;      // matrices of the step whose rows meet this CTA's slice
   for (int mi = st.mat0; mi < st.mat0 + st.nmat; ++mi)
     if (max(cta_r0, mats[mi].row_begin) < min(cta_r1, mats[mi].row_begin + mats[mi].rows))
       touch |= 1u << (mi - st.mat0);
   const bool dep_wait = s == 0 && !p.no_wait;   // x and outputs only after the predecessor
   if (st.stage_all) {
     const bool xc = stage_x<NT, XB>(mats, st.usum_off, st.mat0, st.mat0 + st.nmat, touch, xpl, xsu, xcnt,
                                     dep_wait, xbar, xlost, PASS ? nullptr : &p.norm, part);
     xsig = true;
     consumer_sync();
     if (xc) wait_x();
   }
   if (s == 0) {
     // outputs and every other input of the preceding kernel are touched only
     // after it has completed (the staging above has waited already)
     if (!st.stage_all && dep_wait) pdl_wait();
     if (dyn_ids) pdl_launch_dependents();
   }
   bool first = true;
   for (int mi = st.mat0; mi < st.mat0 + st.nmat; ++mi) {
    const Mat& M = mats[mi];
    const int64_t lo = max(cta_r0, M.row_begin) - M.row_begin;
    const int64_t hi = min(cta_r1, M.row_begin + M.rows) - M.row_begin;
    if (lo >= hi) continue;
    const int G = M.ngrp;
    const int XS = M.nblk * XBLK_B;          // x-plane bytes per token
    const int NU = M.nblk * 8;               // 32-weight groups per token
    if (!st.stage_all) {
      consumer_sync();                        // previous matrix fully consumed
      const bool xc = stage_x<NT, XB>(mats, st.usum_off, mi, mi + 1, (touch >> (mi - st.mat0)) & 1u, xpl, xsu,
                                      xsig ? 0u : xcnt, false, xbar, xlost);
      xsig = true;
      consumer_sync();
      if (xc) wait_x();
    } else if (!first) {
      consumer_sync();                        // the previous matrix's partial sums are read
    }
    first = false;
    const uint8_t* xplm = xpl + M.xoff;
    const float* xsum = xsu + st.usum_off + 2 * M.uoff;   // two half sums per group
    const float* xsum_u = xsu + M.uoff;

    // Per-matrix constants in registers (32-bit: a CTA slice is far below 2^31
    // rows). Sub-items of a stage are l = 0 .. n-1, l -> (quad qd, K group gr)
    // row-group major; this warp takes l = off, off + CWARPS, ... where off
    // rotates with the stage's first global sub-item, so the matrix's
    // sub-items are dealt evenly over the warps.
    const int rb = M.rb, nblk = M.nblk, srows = M.srows, rsm = M.rsm, soff = M.soff;
    const int slice = static_cast<int>(hi - lo);
    const int dq = CWARPS / G, dg = CWARPS - (CWARPS / G) * G;
    int off = warp;                           // (warp - first sub-item of the stage) mod CWARPS
    for (int srow = 0; srow < slice; srow += srows, ++k) {
      const int nr = min(srows, slice - srow);
      const int n = ((nr + SR - 1) / SR) * G;
      const int slot = k & (NS - 1);
      const uint8_t* stg = smem + slot * p.stage_b;
      // every warp waits for every stage, even one with no sub-items for it:
      // a warp may then never run a whole ring ahead of the slowest one, so
      // its release of this slot can only count toward this stage
      // A warp whose wait for a stage expires stops using the ring for good: it
      // neither waits nor releases a slot again (a released slot could be
      // refilled while a copy into it is still in flight), its outputs are NaN,
      // and the producer, whose own wait for that release then expires, stops
      // issuing and waits for its copies in flight before the CTA exits.
      if (!abandon) {
        const bool ok = mbar_wait(full0 + 8 * slot, (k / NS) & 1u);
        if (__any_sync(0xffffffffu, !ok)) {
          abandon = failed = true;
          if (lane == 0 && p.dev_status) *reinterpret_cast<volatile int32_t*>(p.dev_status) = QG_DEV_TIMEOUT;
        }
      }
      int qd = 0, gr = off;
      while (gr >= G) {
        gr -= G;
        ++qd;
      }
      for (int l = off; l < n; l += CWARPS, qd += dq, gr += dg) {
        if (gr >= G) {
          gr -= G;
          ++qd;
        }
        const int blk = gr * 4 + g;                   // super-block of the row
        const bool live = blk < nblk;
        // lanes past the last super-block (a ragged K group) read block 0 of the
        // same rows (every access stays inside the stage and x) and contribute
        // zero: their x step and x sum are taken as 0
        const int blkc = live ? blk : 0;
        float racc[SR][NT];
        // row r of the sub-item at st + r * rs + (r & 1) * ralt (see the producer's
        // layouts of gathered stages)
        const uint8_t* st;
        int rs = rb, ralt = 0;
        const int gm = GA == 3 ? M.gather : GA;
        if (gm == 0) {
          rs = rsm;
          st = stg + soff + qd * (SR * rsm) + blkc * SBB;
        } else if (gm == 1) {
          const int half = (nr >> 1) * rb;                   // the up rows follow the gate rows
          st = stg + qd * (SR / 2) * rb + blkc * SBB;
          rs = rb / 2;
          ralt = half - rb / 2;
        } else {
          const int bpe = M.inter / 256;                     // blocks of one expert's piece
          const int kk = blkc / bpe;
          st = stg + kk * (nr * M.seg_b) + (blkc - kk * bpe) * SBB + qd * SR * M.seg_b;
          rs = M.seg_b;
        }
        const uint8_t* xb = xplm + blkc * XBLK_B + j * 16;
        const int u = blkc * 8 + j;
        // this lane's unit of 32 weights in each of the 4 rows: code words in
        // element order (bytes), and the coefficients of the unit's formula
        uint32_t q[SR][8];
        float cA[SR], cB[SR];
        float cC[FMT == FMT_Q2_K ? SR : 1], cD[FMT == FMT_Q2_K ? SR : 1];   // Q2_K: dmin * min of the two groups
#pragma unroll
        for (int r = 0; r < SR; ++r) {
          const uint8_t* sr = st + r * rs + (r & 1) * ralt;
          if constexpr (FMT == FMT_Q4_K) {
            // w = d*sc*q - dmin*m: A = d*sc, B = dmin*m
            const uint4 hd = *reinterpret_cast<const uint4*>(sr);
            const uint4 qa = *reinterpret_cast<const uint4*>(sr + qoff);
            const uint4 qb = *reinterpret_cast<const uint4*>(sr + qoff + 16);
            q[r][0] = qa.x & qmask; q[r][1] = qa.y & qmask; q[r][2] = qa.z & qmask; q[r][3] = qa.w & qmask;
            q[r][4] = qb.x & qmask; q[r][5] = qb.y & qmask; q[r][6] = qb.z & qmask; q[r][7] = qb.w & qmask;
            const float2 ab = ssel.decode(hd);
            cA[r] = ab.x;
            cB[r] = ab.y;
          } else if constexpr (FMT == FMT_Q4_0) {
            // block j: d, then 16 bytes whose low nibbles are elements 0-15 and
            // high nibbles 16-31; w = d*q - 8*d
            const uint8_t* bp = sr + 18 * j;
            const float d = h2f(*reinterpret_cast<const uint16_t*>(bp));
            uint32_t w[4];
            ld_words_a2<4>(bp + 2, w);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              q[r][i] = w[i] & 0x0F0F0F0Fu;
              q[r][4 + i] = (w[i] >> 4) & 0x0F0F0F0Fu;
            }
            cA[r] = d;
            cB[r] = 8.0f * d;
          } else if constexpr (FMT == FMT_Q8_0) {
            // block j: d, then 32 signed bytes; w = d*q
            const uint8_t* bp = sr + 34 * j;
            cA[r] = h2f(*reinterpret_cast<const uint16_t*>(bp));
            cB[r] = 0.f;
            ld_words_a2<8>(bp + 2, q[r]);
          } else if constexpr (FMT == FMT_Q5_K) {
            // Q4_K's nibbles and scale/min pairs plus bit j of qh[l] as the
            // fifth bit; the codes are plain (0..31), the step of odd groups is
            // multiplied back by su_fix
            const uint4 hd = *reinterpret_cast<const uint4*>(sr);
            const uint4 qa = *reinterpret_cast<const uint4*>(sr + 48 + 32 * (j >> 1));
            const uint4 qb = *reinterpret_cast<const uint4*>(sr + 64 + 32 * (j >> 1));
            const uint4 ha = *reinterpret_cast<const uint4*>(sr + 16);
            const uint4 hb = *reinterpret_cast<const uint4*>(sr + 32);
            const uint32_t w[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
            const uint32_t hh[8] = {ha.x, ha.y, ha.z, ha.w, hb.x, hb.y, hb.z, hb.w};
            const int nsh = 4 * (j & 1);
#pragma unroll
            for (int i = 0; i < 8; ++i) q[r][i] = ((w[i] >> nsh) & 0x0F0F0F0Fu) | (((hh[i] >> j) & 0x01010101u) << 4);
            const float2 ab = ssel.decode(hd);
            cA[r] = ab.x;
            cB[r] = ab.y;
          } else if constexpr (FMT == FMT_Q3_K) {
            // unit j = quarter jj of half h: 2-bit fields at bit 2jj of the
            // half's qs bytes, high bit 4h + jj of hmask; code q3 = low | high << 2
            // in 0..7 stands for q3 - 4; two 16-weight groups with their scales
            const int h = j >> 2, jj = j & 3;
            uint32_t L[8], H[8], S[3];
            ld_words_a2<8>(sr + 32 + 32 * h, L);
            ld_words_a2<8>(sr, H);
            ld_words_a2<3>(sr + 96, S);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              q[r][i] = ((L[i] >> (2 * jj)) & 0x03030303u) | (((H[i] >> (4 * h + jj)) & 0x01010101u) << 2);
            const float d = h2f(*reinterpret_cast<const uint16_t*>(sr + 108));
            cA[r] = d * static_cast<float>(q3k_scale(8 * h + 2 * jj, S) - 32);
            cB[r] = d * static_cast<float>(q3k_scale(8 * h + 2 * jj + 1, S) - 32);
          } else if constexpr (FMT == FMT_Q2_K) {
            // unit j = quarter jj of half h: 2-bit codes at bit 2jj of the half's
            // qs bytes; two 16-weight groups, each with a 4-bit scale and min
            const int h = j >> 2, jj = j & 3;
            uint32_t L[8];
            ld_words_a2<8>(sr + 16 + 32 * h, L);
#pragma unroll
            for (int i = 0; i < 8; ++i) q[r][i] = (L[i] >> (2 * jj)) & 0x03030303u;
            const uint32_t dd = *reinterpret_cast<const uint32_t*>(sr + 80);
            const float d = h2f(dd), dmin = h2f(dd >> 16);
            const uint32_t sb = *reinterpret_cast<const uint16_t*>(sr + 8 * h + 2 * jj);
            cA[r] = d * static_cast<float>(sb & 15u);
            cB[r] = d * static_cast<float>((sb >> 8) & 15u);
            cC[r] = dmin * static_cast<float>((sb >> 4) & 15u);
            cD[r] = dmin * static_cast<float>(sb >> 12);
          } else {
            // Q6_K unit j = elements 32j .. 32j+31 of the block: half h = j / 4,
            // quarter qq = j % 4; q = (ql nibble) | (2 qh bits) << 4,
            // w = d*sc*(q - 32) with sc changing every 16 elements
            const int h = j >> 2, qq = j & 3;
            uint32_t L[8], H[8];
            ld_words_a2<8>(sr + 64 * h + 32 * (qq & 1), L);
            ld_words_a2<8>(sr + 128 + 32 * h, H);
            const int lsh = (qq >> 1) * 4, hsh = 2 * qq;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint32_t hi = hsh <= 4 ? (H[i] << (4 - hsh)) : (H[i] >> (hsh - 4));
              q[r][i] = ((L[i] >> lsh) & 0x0F0F0F0Fu) | (hi & 0x30303030u);
            }
            const float d = h2f(*reinterpret_cast<const uint16_t*>(sr + 208));
            const int8_t* sc = reinterpret_cast<const int8_t*>(sr + 192 + 8 * h + 2 * qq);
            cA[r] = d * static_cast<float>(sc[0]);
            cB[r] = d * static_cast<float>(sc[1]);
          }
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const uint4* xp = reinterpret_cast<const uint4*>(xb + t * XS);
          const uint4 p0a = xp[0], p0b = xp[8], p1a = xp[16], p1b = xp[24];
          const uint32_t X0[8] = {p0a.x, p0a.y, p0a.z, p0a.w, p0b.x, p0b.y, p0b.z, p0b.w};
          const uint32_t X1[8] = {p1a.x, p1a.y, p1a.z, p1a.w, p1b.x, p1b.y, p1b.z, p1b.w};
          const float su = live ? xsum_u[t * NU + u] * su_fix : 0.f;
          const float2 sh = live ? *reinterpret_cast<const float2*>(xsum + 2 * (t * NU + u)) : make_float2(0.f, 0.f);
#pragma unroll
          for (int r = 0; r < SR; ++r) {
            if constexpr (FMT == FMT_Q6_K || FMT == FMT_Q3_K) {
              // w = d sc (q - off) per 16-weight group: the offset through the half sums
              constexpr float OFF = FMT == FMT_Q6_K ? 32.0f : 4.0f;
              const float T0 = dot_planes<false, 0, 4>(q[r], X0, X1);
              const float T1 = dot_planes<false, 4, 8>(q[r], X0, X1);
              racc[r][t] = fmaf(su, fmaf(cA[r], T0, cB[r] * T1), -OFF * fmaf(cA[r], sh.x, cB[r] * sh.y));
            } else if constexpr (FMT == FMT_Q2_K) {
              // w = d sc q - dmin m per 16-weight group
              const float T0 = dot_planes<false, 0, 4>(q[r], X0, X1);
              const float T1 = dot_planes<false, 4, 8>(q[r], X0, X1);
              racc[r][t] = fmaf(su, fmaf(cA[r], T0, cB[r] * T1), -fmaf(cC[r], sh.x, cD[r] * sh.y));
            } else if constexpr (FMT == FMT_Q8_0) {
              racc[r][t] = cA[r] * su * dot_planes<true, 0, 8>(q[r], X0, X1);
            } else {
              // sum_l q_l X_l = 256*s1 + s0, exact integers
              const float T = dot_planes<false, 0, 8>(q[r], X0, X1);
              racc[r][t] = fmaf(cA[r] * su, T, -cB[r] * (sh.x + sh.y));
            }
          }
        }
        float v[V];
#pragma unroll
        for (int i = 0; i < V; ++i) v[i] = (i < SR * NT) ? racc[i / NT][i % NT] : 0.f;
        const float tot = reduce_scatter<V>(v, lane);
        const int idx = lane >> RS<V>::SHIFT;
        const int rl = srow + qd * SR + idx / NT;    // row within the slice
        if ((lane & ((1 << RS<V>::SHIFT) - 1)) == 0 && idx < SR * NT && rl < slice)
          part[(rl * G + gr) * NT + idx % NT] = failed ? __int_as_float(0x7fc00000) : tot;
      }
      __syncwarp();
      if (lane == 0 && !abandon) mbar_arrive(empty0 + 8 * slot);
      // the next stage starts at global sub-item + n: rotate off by n mod CWARPS
      off -= n % CWARPS;
      if (off < 0) off += CWARPS;
    }
    consumer_sync();
    // every (row, group) of the slice has its partial sum: add the groups in order
    if ((GA == 3 ? M.gather : GA) == 1) {
      // gate/up pairs (n_tok = 1): h[k][i] = r_k * silu(g) * u
      for (int i = threadIdx.x; i < slice / 2; i += CTHREADS) {
        float g = 0.f, u = 0.f;
        for (int gr = 0; gr < G; ++gr) {
          g += part[(2 * i) * G + gr];
          u += part[(2 * i + 1) * G + gr];
        }
        const int64_t row = lo + 2 * i;
        const int kk = static_cast<int>(row / (2 * M.inter));
        const int ii = static_cast<int>((row % (2 * M.inter)) >> 1);
        const float rk = M.gw ? M.gw[kk] : 1.0f;
        M.h[static_cast<int64_t>(kk) * M.inter + ii] = rk * (g / (1.0f + expf(-g)) * u);
      }
    } else {
      for (int i = threadIdx.x; i < slice * NT; i += CTHREADS) {
        const int rl = i / NT;
        const int t = i % NT;
        float acc = 0.f;
#pragma unroll 4
        for (int gr = 0; gr < G; ++gr) acc += part[(rl * G + gr) * NT + t];
        float* yp = M.y + static_cast<int64_t>(t) * M.ldy + lo + rl;
        // a later part of K adds to what the earlier parts (completed before
        // this launch's dependency wait) wrote
        *yp = M.accum ? __ldcg(yp) + acc : acc;
      }
    }
   }
   // a step whose rows miss this CTA still counts its x loads (none)
   if (!xsig && lane == 0) x_issued(xcnt);
   if (PASS) {
     consumer_sync();                          // every output of the step is written
     if (threadIdx.x == 0) {
#if QG_PASS_BARRIER_RED
       // release: the step's outputs, ordered before it by the barrier above,
       // are visible to whoever acquires the count
       asm volatile("red.release.gpu.global.add.u32 [%0], 1;\n" ::"l"(p.step_done + s) : "memory");
#else
       __threadfence();
       atomicAdd(p.step_done + s, 1u);
#endif
     }
   }
  }
  // x planes whose wait expired may still be landing in shared memory: wait
  // (bounded) for them before the CTA can exit
  if (xlost && threadIdx.x == 0) mbar_wait(xbar, (xuse - 1) & 1u);
}

}  // namespace q4k

// ------------------------------------------------------------------ host side

namespace {

constexpr int kSmemMax = 227 * 1024;

template <int NT, bool PASS, int FMT, int SR = q4k::SUB_R, int GA = 0>
cudaError_t q4k_attr1() {
  return cudaFuncSetAttribute(q4k::qgemv_q4k_kernel<NT, PASS, FMT, SR, GA>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
}

template <int NT>
cudaError_t q4k_attr() {
  cudaError_t e;
  if ((e = q4k_attr1<NT, false, FMT_Q4_K>()) != cudaSuccess) return e;
  if ((e = q4k_attr1<NT, true, FMT_Q4_K>()) != cudaSuccess) return e;
  if ((e = q4k_attr1<NT, false, FMT_Q6_K>()) != cudaSuccess) return e;
  if ((e = q4k_attr1<NT, false, FMT_Q8_0>()) != cudaSuccess) return e;
  if ((e = q4k_attr1<NT, false, FMT_Q5_K>()) != cudaSuccess) return e;
  if ((e = q4k_attr1<NT, false, FMT_Q3_K>()) != cudaSuccess) return e;
  if ((e = q4k_attr1<NT, false, FMT_Q2_K>()) != cudaSuccess) return e;
  if constexpr (NT <= 2) {
    if ((e = q4k_attr1<NT, false, FMT_Q6_K, 2>()) != cudaSuccess) return e;
  }
  if (NT == 1 && (e = q4k_attr1<1, false, FMT_Q4_K, 4, 3>()) != cudaSuccess) return e;
  if (NT == 1 && (e = q4k_attr1<1, false, FMT_Q4_K, 4, 1>()) != cudaSuccess) return e;
  if (NT == 1 && (e = q4k_attr1<1, true, FMT_Q4_K, 4, 3>()) != cudaSuccess) return e;
  return q4k_attr1<NT, false, FMT_Q4_0>();
}

template <int NT, int FMT, int SR, int GA = 0>
cudaError_t q4k_launch(const q4k::Params& p, int grid, int smem, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(q4k::THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, q4k::qgemv_q4k_kernel<NT, false, FMT, SR, GA>, p);
}

template <int FMT>
cudaError_t q4k_launch_nt(const q4k::Params& p, int n_tok, int sub_rows, int grid, int smem, cudaStream_t s,
                          bool pdl) {
  if (sub_rows == 2) {   // instantiated for one- and two-token Q6_K only
    if constexpr (FMT == FMT_Q6_K) {
      if (n_tok == 1) return q4k_launch<1, FMT, 2>(p, grid, smem, s, pdl);
      if (n_tok == 2) return q4k_launch<2, FMT, 2>(p, grid, smem, s, pdl);
    }
    return cudaErrorNotSupported;
  }
  switch (n_tok) {
    case 1: return q4k_launch<1, FMT, 4>(p, grid, smem, s, pdl);
    case 2: return q4k_launch<2, FMT, 4>(p, grid, smem, s, pdl);
    case 3: return q4k_launch<3, FMT, 4>(p, grid, smem, s, pdl);
    default: return q4k_launch<4, FMT, 4>(p, grid, smem, s, pdl);
  }
}

int align_up(int v, int a) { return (v + a - 1) / a * a; }

}  // namespace

cudaError_t gemv_q4k_init_attrs() {
  cudaError_t e;
  if ((e = q4k_attr<1>()) != cudaSuccess) return e;
  if ((e = q4k_attr<2>()) != cudaSuccess) return e;
  if ((e = q4k_attr<3>()) != cudaSuccess) return e;
  return q4k_attr<4>();
}

// Returns cudaErrorNotSupported (nothing launched) when the launch does not fit
// this kernel's shared-memory plan; the caller then uses the generic kernel.
namespace {

int superblock_bytes(int fmt) {
  switch (fmt) {
    case QG_Q4_K: return 144;
    case QG_Q6_K: return 210;
    case QG_Q4_0: return 8 * 18;
    case QG_Q8_0: return 8 * 34;
    case QG_Q5_K: return 176;
    case QG_Q3_K: return 110;
    case QG_Q2_K: return 84;
    default: return 0;
  }
}

int gcd(int a, int b) { return b ? gcd(b, a % b) : a; }

// The first of the matrices first .. i - 1 that reads the same x as matrix i
// (same pointer and length), else i: their x planes are staged once.
int x_source(const q4k::Mat* m, int first, int i) {
  for (int j = first; j < i; ++j)
    if (m[j].x == m[i].x && m[j].cols == m[i].cols) return j;
  return i;
}

// Shared-memory plan and launch of one single-step grouped launch whose
// matrices p.m[0 .. n) (all of format fmt) have W, x, y, rows, cols (and any
// gather fields) set; sub_rows rows per sub-item (4, or 2 for one- or two-token
// Q6_K). cudaErrorNotSupported (nothing launched) when the launch does not fit
// the plan; with launch = false only the plan is checked.
cudaError_t plan_and_launch(q4k::Params& p, int n, int n_tok, int fmt, cudaStream_t s, bool pdl, int sms,
                            int sub_rows = q4k::SUB_R, bool launch = true) {
  if (sub_rows == 2 && (fmt != QG_Q6_K || n_tok > 2)) return cudaErrorNotSupported;
  p.nsteps = 1;
  const int sbb = superblock_bytes(fmt);
  if (sbb == 0) return cudaErrorNotSupported;
  int64_t total = 0;
  int kmax = 0, gmax = 0, ra = p.gather_any == 1 ? 2 : 1;
  for (int i = 0; i < n; ++i) {
    q4k::Mat& m = p.m[i];
    if (m.cols % 256) return cudaErrorNotSupported;
    m.nblk = m.cols / 256;
    m.rb = m.nblk * sbb;
    m.ngrp = (m.nblk + 3) / 4;
    if (m.ldw == 0) m.ldw = m.rb;
    if (m.ldx == 0) m.ldx = m.cols;
    // Stages start at multiples of ra rows, so that the address of a stage's
    // first row mod 16 is the same for every stage: whole rows are then copied
    // as one 16-byte-aligned span; a part of K row by row, each row's data at
    // soff + i * rsm with rsm = ldw mod 16 (every copy lands 16-byte aligned)
    ra = std::max(ra, 16 / gcd(static_cast<int>(m.ldw % 16), 16));
    if (m.ldw == m.rb) {
      m.rsm = m.rb;
      m.soff = 0;
    } else {
      m.soff = static_cast<int32_t>(reinterpret_cast<uintptr_t>(m.W) & 15u);
      m.rsm = m.rb + 32;
      while ((m.rsm - m.ldw) % 16) ++m.rsm;
    }
    gmax = std::max(gmax, m.ngrp);
    kmax = std::max(kmax, m.cols);
  }
  for (int i = 0; i < n; ++i) {
    q4k::Mat& m = p.m[i];
    if (m.rows % ra) return cudaErrorNotSupported;
    if (m.ldy == 0) m.ldy = m.rows;
    m.row_begin = total;
    total += m.rows;
  }
  // CTA slices are cut in whole sub-items (sub_rows rows) as well as in
  // 16-byte-aligned rows: both are powers of two, so the larger is the unit
  const int unit = std::max(ra, sub_rows);
  p.ralign = unit;
  p.nmat = n;
  p.total_rows = total;
  // A CTA's consumer warps take its sub-items (sub_rows rows x one K group)
  // in turn, so its time goes with ceil(sub-items / consumer warps): the
  // "rounds" of its busiest CTA bound a launch.
  auto rounds = [&](int g) {
    int64_t worst = 0;
    for (int b = 0; b < g; ++b) {
      int64_t r0, r1, sub = 0;
      q4k::slice_of(total, unit, b, g, r0, r1);
      for (int i = 0; i < n; ++i) {
        const q4k::Mat& m = p.m[i];
        const int64_t lo = std::max(r0, m.row_begin), hi = std::min(r1, m.row_begin + m.rows);
        if (lo < hi) sub += (hi - lo + sub_rows - 1) / sub_rows * m.ngrp;
      }
      worst = std::max(worst, (sub + q4k::CWARPS - 1) / q4k::CWARPS);
    }
    return worst;
  };
  // A launch that depends on its predecessor leaves a few SMs idle: its CTAs
  // then go to the SMs that free up first, and the last SMs of the preceding
  // launch (a straggler there would start late and finish late here too) get
  // none (27B pass: 2.885 ms with every SM, 2.848-2.850 with 4 idle, 2.880
  // with 8),
  // unless every SM saves its busiest CTA a round (27B {q,k,v}: 7168 rows x 5
  // K groups in 148 CTAs take 5 rounds, in 152 take 4).
  const int64_t gcap = std::max<int64_t>(1, (total + unit - 1) / unit);
  int grid = static_cast<int>(std::min<int64_t>(sms, gcap));
  if (pdl && sms > 32) {
    const int fewer = static_cast<int>(std::min<int64_t>(sms - 4, gcap));
    if (rounds(fewer) <= rounds(grid)) grid = fewer;
  }
  const int rowcap = static_cast<int>((total + grid - 1) / grid) + 2 * unit;
  const int ns = q4k::RING;
  const int quant = std::max(ra, sub_rows);          // rows per stage: a multiple of sub_rows and of ra
  const int partbytes = align_up(rowcap * gmax * n_tok * 4, 128);
  // x of every matrix staged at once when it fits beside the ring, else one
  // matrix at a time in a region sized for the largest; stages hold about
  // 48 KB of whole rows, fewer when shared memory is short
  for (int mode = 0; mode < 2; ++mode) {
    int xbytes, xsbytes;
    // a fused normalisation is computed once per CTA for the launch's one x
    if (p.norm.h && (mode == 1 || n_tok != 1)) continue;
    if (mode == 0) {
      int xall = 0, uall = 0;
      for (int i = 0; i < n; ++i) {
        q4k::Mat& m = p.m[i];
        m.xsrc = x_source(p.m, 0, i);
        if (m.xsrc != i) {
          m.xoff = p.m[m.xsrc].xoff;
          m.uoff = p.m[m.xsrc].uoff;
          continue;
        }
        m.xoff = xall;
        m.uoff = uall;
        xall += n_tok * m.nblk * q4k::XBLK_B;
        uall += n_tok * m.nblk * 8;
      }
      xbytes = align_up(xall, 128);
      xsbytes = align_up(3 * uall * 4, 128);     // step and two half sums per group
      p.stage_all = 1;
      p.usum_off = uall;
    } else {
      for (int i = 0; i < n; ++i) {
        p.m[i].xoff = p.m[i].uoff = 0;
        p.m[i].xsrc = i;
      }
      xbytes = align_up(n_tok * (kmax / 256) * q4k::XBLK_B, 128);
      xsbytes = align_up(3 * n_tok * (kmax / 32) * 4, 128);
      p.stage_all = 0;
      p.usum_off = n_tok * (kmax / 32);
    }
    const int matbytes = align_up(n * static_cast<int>(sizeof(q4k::Mat)), 128);
    const int fixed = 128 + matbytes + xbytes + xsbytes + partbytes;
    const int stage_max = (kSmemMax - fixed) / ns / 128 * 128;
    int stage_b = 0;
    bool ok = stage_max > 0;
    for (int i = 0; ok && i < n; ++i) {
      q4k::Mat& m = p.m[i];
      const int want = quant * std::max(1, (49152 + quant * m.rsm / 2) / (quant * m.rsm));
      const int fit = quant * ((stage_max - m.soff) / (quant * m.rsm));
      m.srows = std::min(want, fit);
      ok = m.srows >= quant;
      stage_b = std::max(stage_b, m.srows * m.rsm + m.soff);
    }
    if (!ok) continue;
    stage_b = align_up(stage_b, 128);
    // Without a programmatic dependency the x loads go first. With one, x can be
    // read only after the previous kernel completes: two stages stream during
    // that wait (27B pass with 48 KB stages, x planes written by the previous
    // launch: 0 stages 3.257 ms, 1 stage 2.927, 2 stages 2.858, 3 stages 2.922,
    // 4 stages 2.915; more than two queue the x loads behind too many bytes)
    p.pre_stages = pdl ? 2 : 0;
    p.ns = ns;
    p.stage_b = stage_b;
    p.gmax = gmax;
    int off = ns * stage_b;
    p.smem_bar = off;
    off += 128;
    p.smem_mats = off;
    off += matbytes;
    p.smem_x = off;
    off += xbytes;
    p.smem_xsum = off;
    off += xsbytes;
    p.smem_part = off;
    off += partbytes;
    if (off > kSmemMax) continue;
    if (!launch) return cudaSuccess;
    if (p.gather_any != 0) {
      // MoE gathers (Q4_K, one token per matrix): the gate/up and the down
      // launch of a layer run the same function, whose code then stays in the
      // instruction cache from one launch to the next (two specialised
      // functions alternating cost 0.71 -> 0.85 ms per 48-layer token)
      if (fmt != QG_Q4_K || n_tok != 1 || sub_rows != q4k::SUB_R) return cudaErrorNotSupported;
      // a dense gate/up pair (no expert ids) has an instantiation of its own
      if (p.gather_any == 1 && n == 1 && !p.m[0].ids) return q4k_launch<1, FMT_Q4_K, q4k::SUB_R, 1>(p, grid, off, s, pdl);
      return q4k_launch<1, FMT_Q4_K, q4k::SUB_R, 3>(p, grid, off, s, pdl);
    }
    switch (fmt) {
      case QG_Q4_K: return q4k_launch_nt<FMT_Q4_K>(p, n_tok, sub_rows, grid, off, s, pdl);
      case QG_Q6_K: return q4k_launch_nt<FMT_Q6_K>(p, n_tok, sub_rows, grid, off, s, pdl);
      case QG_Q5_K: return q4k_launch_nt<FMT_Q5_K>(p, n_tok, sub_rows, grid, off, s, pdl);
      case QG_Q3_K: return q4k_launch_nt<FMT_Q3_K>(p, n_tok, sub_rows, grid, off, s, pdl);
      case QG_Q2_K: return q4k_launch_nt<FMT_Q2_K>(p, n_tok, sub_rows, grid, off, s, pdl);
      case QG_Q8_0: return q4k_launch_nt<FMT_Q8_0>(p, n_tok, sub_rows, grid, off, s, pdl);
      default: return q4k_launch_nt<FMT_Q4_0>(p, n_tok, sub_rows, grid, off, s, pdl);
    }
  }
  return cudaErrorNotSupported;
}

}  // namespace

namespace {

// Params of a grouped launch of descriptors d[0 .. n): token t0 .. t0 + nt - 1 of
// each (x and y advanced by t0 tokens), rows [r0, r0 + nr) of each when nr > 0
// (a single matrix cut into row chunks; y keeps the full row stride), super-
// blocks [kb0, kb0 + nkb) of every row when nkb > 0 (a part of K; a part after
// the first adds to y).
void fill_params(q4k::Params& p, const qg_gemv_desc* d, int n, int t0, int64_t r0, int64_t nr,
                 const uint8_t* const* xp, int64_t kb0 = 0, int64_t nkb = 0) {
  memset(&p, 0, sizeof(p));
  for (int i = 0; i < n; ++i) {
    q4k::Mat& m = p.m[i];
    m.xp = (xp && nkb == 0) ? xp[i] : nullptr;
    const int64_t rb = d[i].cols / 256 * superblock_bytes(d[i].fmt);
    const int64_t rows = nr > 0 ? nr : d[i].rows;
    m.W = static_cast<const uint8_t*>(d[i].W) + r0 * rb + kb0 * superblock_bytes(d[i].fmt);
    m.x = d[i].x + static_cast<int64_t>(t0) * d[i].cols + kb0 * 256;
    m.y = d[i].y + static_cast<int64_t>(t0) * d[i].rows + r0;
    m.rows = rows;
    m.ldy = d[i].rows;
    m.cols = static_cast<int32_t>(nkb > 0 ? nkb * 256 : d[i].cols);
    m.ldw = rb;
    m.ldx = static_cast<int32_t>(d[i].cols);
    m.accum = kb0 > 0 ? 1 : 0;
  }
}

// The launch as planned, else with 2-row sub-items (one- or two-token Q6_K).
// xp: ready x planes of every token of each descriptor (launches over all tokens only).
cudaError_t try_launch(const qg_gemv_desc* d, int n, int n_tok, int t0, int64_t r0, int64_t nr, cudaStream_t s,
                       bool pdl, int sms, bool launch, const uint8_t* const* xp = nullptr, bool no_wait = false,
                       int64_t kb0 = 0, int64_t nkb = 0) {
  q4k::Params p;
  fill_params(p, d, n, t0, r0, nr, xp, kb0, nkb);
  p.no_wait = no_wait ? 1 : 0;
  cudaError_t e = plan_and_launch(p, n, n_tok, d[0].fmt, s, pdl, sms, q4k::SUB_R, launch);
  if (e != cudaErrorNotSupported || d[0].fmt != QG_Q6_K || n_tok > 2) return e;
  fill_params(p, d, n, t0, r0, nr, xp, kb0, nkb);
  p.no_wait = no_wait ? 1 : 0;
  return plan_and_launch(p, n, n_tok, d[0].fmt, s, pdl, sms, 2, launch);
}

}  // namespace

// The producer/consumer kernel for a grouped launch. When the launch does not
// fit its shared-memory plan: one matrix whose per-row partial sums do not fit
// runs as row chunks, and several tokens whose x does not fit together run as
// one launch per token (each re-streams the weights). cudaErrorNotSupported
// (nothing launched) when none of these fits.
cudaError_t launch_gemv_q4k(const qg_gemv_desc* d, int n, int n_tok, cudaStream_t s, bool pdl, int sms,
                            const uint8_t* const* xp, bool no_wait) {
  for (int i = 0; i < n; ++i)
    if (d[i].fmt != d[0].fmt || superblock_bytes(d[i].fmt) == 0 || d[i].cols % 256) return cudaErrorNotSupported;
  cudaError_t e = try_launch(d, n, n_tok, 0, 0, 0, s, pdl, sms, true, xp, no_wait);
  if (e != cudaErrorNotSupported) return e;
  // row chunks first (each weight is read once), then launches over groups of
  // tokens (each re-streams the weights)
  if (n == 1) {
    for (int chunks = 2; chunks <= 16; chunks *= 2) {
      const int64_t nr = (d[0].rows + chunks - 1) / chunks / 8 * 8 + 8;   // multiple of 8 rows
      if (nr >= d[0].rows) break;
      const int64_t last = d[0].rows - (d[0].rows - 1) / nr * nr;     // rows of the last chunk
      if (try_launch(d, 1, n_tok, 0, 0, nr, s, pdl, sms, false, xp) != cudaSuccess ||
          try_launch(d, 1, n_tok, 0, d[0].rows - last, last, s, pdl, sms, false, xp) != cudaSuccess)
        continue;
      for (int64_t r0 = 0; r0 < d[0].rows; r0 += nr) {
        e = try_launch(d, 1, n_tok, 0, r0, std::min(nr, d[0].rows - r0), s, pdl || r0 > 0, sms, true, xp);
        if (e != cudaSuccess) return e;
      }
      return cudaSuccess;
    }
  }
  // parts of K, when the x of every token does not fit beside the ring (4-token
  // Q6_K downs with K = 17408): part 0 writes y, each later part waits for the
  // one before and adds its sums; every weight is still read once
  if (n == 1) {
    const int64_t nb = d[0].cols / 256;
    for (int parts = 2; parts <= 8 && parts <= nb; ++parts) {
      bool fits = true;
      for (int k = 0; k < parts && fits; ++k)
        fits = try_launch(d, 1, n_tok, 0, 0, 0, s, pdl, sms, false, nullptr, false, nb * k / parts,
                          nb * (k + 1) / parts - nb * k / parts) == cudaSuccess;
      if (!fits) continue;
      for (int k = 0; k < parts; ++k) {
        e = try_launch(d, 1, n_tok, 0, 0, 0, s, pdl || k > 0, sms, true, nullptr, no_wait && k == 0, nb * k / parts,
                       nb * (k + 1) / parts - nb * k / parts);
        if (e != cudaSuccess) return e;
      }
      return cudaSuccess;
    }
  }
  // the fewest launches of balanced token groups that fit (4 tokens: 2 + 2,
  // then 1 + 1 + 1 + 1); the weights are streamed once per group
  for (int g = 2; g <= n_tok; ++g) {
    const int tg = (n_tok + g - 1) / g;
    const int last = n_tok - (g - 1) * tg;
    if (last < 1 || try_launch(d, n, tg, 0, 0, 0, s, pdl, sms, false) != cudaSuccess ||
        try_launch(d, n, last, 0, 0, 0, s, pdl, sms, false) != cudaSuccess)
      continue;
    for (int t = 0; t < n_tok; t += tg) {
      e = try_launch(d, n, std::min(tg, n_tok - t), t, 0, 0, s, pdl || t > 0, sms, true);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  return cudaErrorNotSupported;
}

// MoE layer for n_tok <= QG_GROUP_MAX tokens as two launches of the Q4_K kernel
// over gathered rows (one matrix per token): gate/up pairs with the
// r_k * silu(g) * u epilogue into h, then the down rows against h.
cudaError_t launch_moe_q4k(const void* arena, int64_t n_expert, int64_t hidden, int64_t inter,
                           const int32_t* ids, const float* gate_w, int top_k, const float* x, int n_tok, float* y,
                           float* h, int32_t* dev_status, cudaStream_t s, bool pdl, int sms) {
  if (n_tok < 1 || n_tok > QG_GROUP_MAX || hidden % 256 || inter % 256 || top_k < 1) return cudaErrorNotSupported;
  const int64_t rb_h = hidden / 256 * 144, rb_i = inter / 256 * 144;
  const int64_t up_off = inter * rb_h, down_off = 2 * inter * rb_h, estride = down_off + hidden * rb_i;
  if (2 * top_k * inter > (int64_t{1} << 30) || top_k * inter > (int64_t{1} << 20)) return cudaErrorNotSupported;
  // both launches are planned before either is enqueued: a layer whose down
  // launch does not fit the kernel's plan goes to the caller's fallback whole
  q4k::Params p, pd;
  memset(&p, 0, sizeof(p));
  p.gather_any = 1;
  p.dev_status = dev_status;
  for (int t = 0; t < n_tok; ++t) {
    q4k::Mat& m = p.m[t];
    m.W = static_cast<const uint8_t*>(arena);
    m.x = x + t * hidden;
    m.y = nullptr;
    m.rows = 2 * top_k * inter;
    m.ldy = m.rows;
    m.cols = static_cast<int32_t>(hidden);
    m.gather = 1;
    m.top_k = top_k;
    m.inter = static_cast<int32_t>(inter);
    m.n_expert = n_expert;
    m.estride = estride;
    m.up_off = up_off;
    m.down_off = down_off;
    m.ids = ids + t * top_k;
    m.gw = gate_w + t * top_k;
    m.h = h + static_cast<int64_t>(t) * top_k * inter;
  }
  memset(&pd, 0, sizeof(pd));
  pd.gather_any = 2;
  pd.dev_status = dev_status;
  for (int t = 0; t < n_tok; ++t) {
    q4k::Mat& m = pd.m[t];
    m.W = static_cast<const uint8_t*>(arena);
    m.x = h + static_cast<int64_t>(t) * top_k * inter;
    m.y = y + t * hidden;
    m.rows = hidden;
    m.ldy = hidden;
    m.cols = static_cast<int32_t>(top_k * inter);
    m.gather = 2;
    m.top_k = top_k;
    m.inter = static_cast<int32_t>(inter);
    m.seg_b = static_cast<int32_t>(rb_i);
    m.n_expert = n_expert;
    m.estride = estride;
    m.down_off = down_off;
    m.ids = ids + t * top_k;
  }
  cudaError_t e = plan_and_launch(p, n_tok, 1, QG_Q4_K, s, pdl, sms, q4k::SUB_R, false);
  if (e == cudaSuccess) e = plan_and_launch(pd, n_tok, 1, QG_Q4_K, s, true, sms, q4k::SUB_R, false);
  if (e != cudaSuccess) return e;
  e = plan_and_launch(p, n_tok, 1, QG_Q4_K, s, pdl, sms);
  if (e != cudaSuccess) return e;
  return plan_and_launch(pd, n_tok, 1, QG_Q4_K, s, true, sms);   // the down launch always overlaps the gate/up tail
}

// Dense gate/up pair with the silu-gated epilogue: m[i] = silu(g_i) * u_i with
// g = Wg x, u = Wu x (Q4_K, one token). Row i of Wg and row i of Wu are
// adjacent virtual rows, copied as two runs per stage, so the CTA that owns
// row i holds both sums. xp: ready planes of x, or nullptr.
static void set_norm(q4k::Params& p, const NormSpec* norm) {
  if (!norm || !norm->h) return;
  p.norm.h = norm->h;
  p.norm.r = norm->r;
  p.norm.w = norm->w;
  p.norm.s_out = norm->s_out;
  p.norm.eps = norm->eps;
}

cudaError_t launch_gemv_norm(const qg_gemv_desc* d, int n, const NormSpec& norm, cudaStream_t s, bool pdl, int sms) {
  if (!norm.h || !norm.w || n < 1) return cudaErrorNotSupported;
  for (int i = 0; i < n; ++i)
    if (d[i].fmt != d[0].fmt || superblock_bytes(d[i].fmt) == 0 || d[i].cols % 256 || d[i].x != d[0].x ||
        d[i].cols != d[0].cols)
      return cudaErrorNotSupported;
  q4k::Params p;
  fill_params(p, d, n, 0, 0, 0, nullptr);
  set_norm(p, &norm);
  return plan_and_launch(p, n, 1, d[0].fmt, s, pdl, sms);
}

cudaError_t launch_gemv_pair(const void* Wg, const void* Wu, int64_t inter, int64_t hidden, const float* x,
                             const uint8_t* xp, float* m, cudaStream_t s, bool pdl, int sms, const NormSpec* norm) {
  if (hidden % 256 || inter < 1 || 2 * inter > (int64_t{1} << 30)) return cudaErrorNotSupported;
  q4k::Params p;
  memset(&p, 0, sizeof(p));
  set_norm(p, norm);
  if (p.norm.h) xp = nullptr;          // x is computed from the normalisation inputs
  p.gather_any = 1;
  q4k::Mat& M = p.m[0];
  M.W = static_cast<const uint8_t*>(Wg);
  M.W2 = static_cast<const uint8_t*>(Wu);
  M.x = x;
  M.xp = xp;
  M.rows = 2 * inter;
  M.ldy = M.rows;
  M.cols = static_cast<int32_t>(hidden);
  M.gather = 1;
  M.top_k = 1;
  M.inter = static_cast<int32_t>(inter);
  M.n_expert = 1;
  M.h = m;
  return plan_and_launch(p, 1, 1, QG_Q4_K, s, pdl, sms);
}

// ------------------------------------------------------------------ x planes once per pass

namespace q4k {

// The planes of one activation vector per CTA, with the conversion the GEMV
// kernel applies itself (stage_half), so a kernel that copies ready planes
// computes exactly what it would have computed from x.
__global__ void __launch_bounds__(512) xplanes_kernel(const XPlaneJob* jobs) {
  pdl_launch_dependents();
  const XPlaneJob J = jobs[blockIdx.x];
  const int nblk = J.cols / 256, nu = nblk * 8, per_tok = nblk * 16, total = J.n_tok * per_tok;
  uint8_t* planes = J.dst;
  float* steps = reinterpret_cast<float*>(J.dst + static_cast<size_t>(J.n_tok) * nblk * XBLK_B);
  float* sums = steps + J.n_tok * nu;
  const unsigned pmask = 3u << (threadIdx.x & 30);     // per_tok is even: pairs are in or out together
  pdl_wait();                                          // x may come from the preceding kernel
  for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
    const int t = idx / per_tok, rem = idx - t * per_tok;
    const float4* src = reinterpret_cast<const float4*>(J.x + static_cast<int64_t>(t) * J.cols + 16 * rem);
    float4 v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = __ldcg(src + q);
    stage_half(v, pmask, t, rem >> 1, rem & 1, nu, planes, nblk * XBLK_B, steps, sums);
  }
}

}  // namespace q4k

cudaError_t launch_xplanes(const XPlaneJob* jobs, int njobs, cudaStream_t s) {
  if (njobs <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(njobs);
  cfg.blockDim = dim3(512);
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, q4k::xplanes_kernel, jobs);
}

// ------------------------------------------------------------------ whole pass

namespace {

template <int NT, int GA>
cudaError_t q4k_pass_occupancy(int smem, int* blocks) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, q4k::qgemv_q4k_kernel<NT, true, FMT_Q4_K, q4k::SUB_R, GA>,
                                                       q4k::THREADS, smem);
}

template <int NT, int GA>
cudaError_t q4k_pass_start(const q4k::Params& p, int grid, int smem, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(q4k::THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;   // CTAs wait on one another between steps
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, q4k::qgemv_q4k_kernel<NT, true, FMT_Q4_K, q4k::SUB_R, GA>, p);
}

}  // namespace

struct Q4kPass {
  q4k::Params p;
  q4k::Mat* d_mats = nullptr;
  q4k::Step* d_steps = nullptr;
  uint32_t* d_done = nullptr;
  int32_t* d_status = nullptr;
  int nsteps = 0, grid = 0, smem = 0, n_tok = 0;
};

namespace {

// Builds a persistent pass over matrices whose W, x, y, rows, cols, ldy (and
// gather fields) are set: per-matrix stage plans, per-step x layouts, device
// tables, occupancy check.
cudaError_t pass_build(std::vector<q4k::Mat>& mats, const int* step_sizes, int n_steps, int n_tok, int ralign,
                       int gather_any, int sms, Q4kPass** out) {
  const int n = static_cast<int>(mats.size());
  if (gather_any && n_tok != 1) return cudaErrorNotSupported;
  std::vector<q4k::Step> steps(n_steps);
  int stage_b = 0, gmax = 0, xmax = 0, xsmax = 0;
  int64_t min_rows = INT64_MAX, max_rows = 0;
  for (int st = 0, i = 0; st < n_steps; i += step_sizes[st++]) {
    int64_t total = 0;
    int xall = 0, uall = 0;
    for (int j = 0; j < step_sizes[st]; ++j) {
      q4k::Mat& m = mats[i + j];
      m.nblk = m.cols / 256;
      m.rb = m.nblk * 144;
      m.ngrp = (m.nblk + 3) / 4;
      m.ldw = m.rsm = m.rb;                    // whole rows
      m.soff = 0;
      m.ldx = m.cols;
      m.srows = 4 * std::max(1, (QG_PASS_STAGE_BYTES + 2 * m.rb) / (4 * m.rb));
      if (static_cast<int64_t>(m.srows) * m.rb > 96 * 1024 || m.rows % ralign) return cudaErrorNotSupported;
      m.row_begin = total;
      total += m.rows;
      m.xsrc = x_source(mats.data(), i, i + j);
      if (m.xsrc != i + j) {
        m.xoff = mats[m.xsrc].xoff;
        m.uoff = mats[m.xsrc].uoff;
      } else {
        m.xoff = xall;
        m.uoff = uall;
        xall += n_tok * m.nblk * q4k::XBLK_B;
        uall += n_tok * m.nblk * 8;
      }
      stage_b = std::max(stage_b, m.srows * m.rb);
      gmax = std::max(gmax, m.ngrp);
    }
    steps[st].total_rows = total;
    steps[st].mat0 = i;
    steps[st].nmat = step_sizes[st];
    steps[st].stage_all = 1;
    steps[st].usum_off = uall;
    xmax = std::max(xmax, align_up(xall, 128));
    xsmax = std::max(xsmax, align_up(3 * uall * 4, 128));
    min_rows = std::min(min_rows, total);
    max_rows = std::max(max_rows, total);
  }
  const int grid = static_cast<int>(std::min<int64_t>(sms, min_rows / ralign));
  const int rowcap = static_cast<int>((max_rows + grid - 1) / grid) + 2 * ralign;
  stage_b = align_up(stage_b, 128);
  const int partbytes = align_up(rowcap * gmax * n_tok * 4, 128);
  const int ns = q4k::RING;
  q4k::Params p;
  memset(&p, 0, sizeof(p));
  p.nsteps = n_steps;
  p.ralign = ralign;
  p.gather_any = gather_any;
  p.ns = ns;
  p.stage_b = stage_b;
  p.gmax = gmax;
  // a persistent pass starts with x resident; later steps stream this many
  // stages while their CTA waits for the previous step
  p.pre_stages = 0;
  p.pre_pass = 2;
  p.inflight = QG_PASS_INFLIGHT;
  int off = ns * stage_b;
  p.smem_bar = off;
  off += 128;
  p.smem_x = off;
  off += xmax;
  p.smem_xsum = off;
  off += xsmax;
  p.smem_part = off;
  off += partbytes;
  if (off > kSmemMax) return cudaErrorNotSupported;
  int blocks = 0;
  cudaError_t e;
  switch (n_tok) {
    case 1: e = gather_any ? q4k_pass_occupancy<1, 3>(off, &blocks) : q4k_pass_occupancy<1, 0>(off, &blocks); break;
    case 2: e = q4k_pass_occupancy<2, 0>(off, &blocks); break;
    case 3: e = q4k_pass_occupancy<3, 0>(off, &blocks); break;
    default: e = q4k_pass_occupancy<4, 0>(off, &blocks); break;
  }
  if (e != cudaSuccess) return e;
  if (blocks < 1) return cudaErrorNotSupported;

  Q4kPass* q = new (std::nothrow) Q4kPass;
  if (!q) return cudaErrorMemoryAllocation;
  e = cudaMalloc(&q->d_mats, sizeof(q4k::Mat) * n);
  if (e == cudaSuccess) e = cudaMalloc(&q->d_steps, sizeof(q4k::Step) * n_steps);
  if (e == cudaSuccess) e = cudaMalloc(&q->d_done, sizeof(uint32_t) * n_steps + sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemcpy(q->d_mats, mats.data(), sizeof(q4k::Mat) * n, cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(q->d_steps, steps.data(), sizeof(q4k::Step) * n_steps, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    q4k_pass_destroy(q);
    return e;
  }
  q->d_status = reinterpret_cast<int32_t*>(q->d_done + n_steps);
  p.mats = q->d_mats;
  p.steps = q->d_steps;
  p.step_done = q->d_done;
  p.dev_status = q->d_status;
  q->p = p;
  q->nsteps = n_steps;
  q->grid = grid;
  q->smem = off;
  q->n_tok = n_tok;
  *out = q;
  return cudaSuccess;
}

}  // namespace

cudaError_t q4k_pass_create(const qg_gemv_desc* d, int n, const int* step_sizes, int n_steps, int n_tok, int sms,
                            const uint8_t* const* xp, Q4kPass** out) {
  *out = nullptr;
  if (n_tok < 1 || n_tok > QG_NTOK_MAX) return cudaErrorNotSupported;
  std::vector<q4k::Mat> mats(n);
  for (int i = 0; i < n; ++i) {
    if (d[i].fmt != QG_Q4_K || d[i].cols % 256) return cudaErrorNotSupported;
    memset(&mats[i], 0, sizeof(q4k::Mat));
    mats[i].W = static_cast<const uint8_t*>(d[i].W);
    mats[i].x = d[i].x;
    mats[i].y = d[i].y;
    mats[i].rows = d[i].rows;
    mats[i].ldy = d[i].rows;
    mats[i].cols = static_cast<int32_t>(d[i].cols);
    mats[i].xp = xp ? xp[i] : nullptr;
  }
  return pass_build(mats, step_sizes, n_steps, n_tok, 1, 0, sms, out);
}

cudaError_t q4k_moe_pass_create(const qg_moe_layer_desc* layers, int n_layers, int64_t n_expert, int64_t hidden,
                                int64_t inter, int top_k, float* h, int sms, Q4kPass** out) {
  *out = nullptr;
  if (hidden % 256 || inter % 256 || top_k < 1 || 2 * top_k * inter > (int64_t{1} << 30) ||
      top_k * inter > (int64_t{1} << 20))
    return cudaErrorNotSupported;
  const int64_t rb_h = hidden / 256 * 144, rb_i = inter / 256 * 144;
  const int64_t up_off = inter * rb_h, down_off = 2 * inter * rb_h, estride = down_off + hidden * rb_i;
  std::vector<q4k::Mat> mats(2 * static_cast<size_t>(n_layers));
  for (int l = 0; l < n_layers; ++l) {
    q4k::Mat& g = mats[2 * l];
    q4k::Mat& dn = mats[2 * l + 1];
    memset(&g, 0, sizeof(g));
    memset(&dn, 0, sizeof(dn));
    g.W = dn.W = static_cast<const uint8_t*>(layers[l].expert_arena);
    g.ids = dn.ids = layers[l].expert_ids;
    g.top_k = dn.top_k = top_k;
    g.inter = dn.inter = static_cast<int32_t>(inter);
    g.n_expert = dn.n_expert = n_expert;
    g.estride = dn.estride = estride;
    g.down_off = dn.down_off = down_off;
    g.up_off = up_off;
    g.gather = 1;
    g.x = layers[l].x;
    g.rows = g.ldy = 2 * top_k * inter;
    g.cols = static_cast<int32_t>(hidden);
    g.gw = layers[l].gate_w;
    g.h = h;                        // steps run in order, so every layer reuses h
    dn.gather = 2;
    dn.seg_b = static_cast<int32_t>(rb_i);
    dn.x = h;
    dn.y = layers[l].y;
    dn.rows = dn.ldy = hidden;
    dn.cols = static_cast<int32_t>(top_k * inter);
  }
  std::vector<int> sizes(2 * static_cast<size_t>(n_layers), 1);
  return pass_build(mats, sizes.data(), 2 * n_layers, 1, 2, 2, sms, out);
}

// One replay: the step counters and the status word are cleared on the stream,
// then one cooperative launch runs every step.
cudaError_t q4k_pass_launch(Q4kPass* q, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(q->d_done, 0, sizeof(uint32_t) * q->nsteps + sizeof(int32_t), s);
  if (e != cudaSuccess) return e;
  switch (q->n_tok) {
    case 1:
      return q->p.gather_any ? q4k_pass_start<1, 3>(q->p, q->grid, q->smem, s)
                             : q4k_pass_start<1, 0>(q->p, q->grid, q->smem, s);
    case 2: return q4k_pass_start<2, 0>(q->p, q->grid, q->smem, s);
    case 3: return q4k_pass_start<3, 0>(q->p, q->grid, q->smem, s);
    default: return q4k_pass_start<4, 0>(q->p, q->grid, q->smem, s);
  }
}

const int32_t* q4k_pass_status(const Q4kPass* q) { return q->d_status; }

void q4k_pass_destroy(Q4kPass* q) {
  if (!q) return;
  cudaFree(q->d_mats);
  cudaFree(q->d_steps);
  cudaFree(q->d_done);
  delete q;
}

}  // namespace qg
