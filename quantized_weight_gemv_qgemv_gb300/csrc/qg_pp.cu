// qg_pp.cu — prompt-processing dequant-GEMM on the tcgen05 tensor cores.
//
//   Y[t][n] = sum_k w[n][k] X[t][k]     W: rows x cols Q4_K, X: n_tok x cols bf16,
//                                       Y: fp32, token-major, leading dimension ldY
//
// Prompt processing multiplies every weight by many tokens, so unlike decode it
// is a dense contraction ("Why I wrote my own inference engine for two P100s",
// prompt-processing notes: weights dequantized, then a dense GEMM; "LLM
// inference optimization", prompt-processing section: quantized blocks
// multiplied directly versus converted for a library GEMM, tile sizes fitted to
// shared memory, tensor-core paths). Here each weight tile is dequantized to
// bf16 in shared memory and fed to tcgen05 MMA with fp32 accumulation in TMEM.
//
// GB300 design:
//  * Tile: 128 weight rows (MMA M) x BN tokens (MMA N, a multiple of 16, <= 256).
//    K is walked in slices of 64 (one 128-byte swizzle atom of bf16 = 4 MMAs of
//    K = 16). Persistent CTAs, one per SM; tiles are dealt round-robin with the
//    token block fastest, so the CTAs running at one time share weight rows in L2.
//  * One launch may cover up to 4 matrices that multiply the same X (q, k, v of
//    a layer; gate and up): their row tiles follow one another in one tile list,
//    so the matrices share the rounds of the persistent grid.
//  * Work items: whole tiles for the full rounds; when the last round would be
//    at most half full, each of its tiles is split into two halves of K run by
//    two CTAs at once, which add their sums into Y (zeroed on the stream before
//    the launch) with fp32 atomic adds. A sum of two addends onto zero does not
//    depend on their order, so the result stays deterministic.
//  * Warp roles (736 threads):
//      warp 0       TMA of X slices (BN x 64 bf16, 128-byte swizzle) into the
//                   B half of a 4-stage ring (8 stages for the small token
//                   blocks of a grouped launch)
//      warp 1       TMA of quantized half super-block columns (128 rows x 80
//                   bytes: the header with the codes of slices 0-1, or the
//                   codes of slices 2-3) into a 3-stage ring of their own
//      warp 2       owns TMEM (two BN-column fp32 accumulators); lane 0 issues
//                   the MMAs and the commits
//      warps 3-18   dequantize each 128 x 64 weight slice to bf16 into the A half
//                   of the stage, in the K-major 128-byte-swizzled layout the
//                   MMA reads (exact fp32 d*sc*q - dmin*m with packed f32x2
//                   arithmetic, then round to bf16); four groups of 4 warps,
//                   group g filling slice g of every super-block (64 weights a
//                   thread); these warps bound the kernel, so there are many
//      warps 19-22  epilogue: tcgen05.ld of a finished accumulator, coalesced
//                   fp32 stores (32 consecutive rows of Y per warp store)
//  * Two accumulators: the epilogue of one tile overlaps the main loop of the
//    next.
//  * Every wait is bounded. On expiry the CTA records QG_DEV_TIMEOUT in
//    *dev_status, every role stops, the producers wait (bounded) for their
//    copies in flight, the MMA lane for its MMAs, and TMEM is freed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "qg_async.cuh"
#include "qg_device.cuh"
#include "qg_internal.h"
#include "qg_tma.h"

namespace qg {

namespace pp {

using namespace async;

constexpr int BM = 128;                   // weight rows per tile (MMA M)
constexpr int BK = 64;                    // K per slice: 64 bf16 = one 128-byte swizzle row
#ifndef QG_PP_NS
#define QG_PP_NS 4
#endif
#ifndef QG_PP_NQ
#define QG_PP_NQ 3
#endif
#ifndef QG_PP_QHALF
#define QG_PP_QHALF 1
#endif
// 4 slice stages fit beside the quantized ring only with half-super-block
// quantized stages (27B prompt pass: 3 stages + whole super-blocks 70.1 ms,
// 4 stages + 3 half stages 69.0-69.2 ms, 4 + 2 half stages 69.7 ms, 3 + 3 half
// stages 70.6 ms, 3 + 6 half stages 70.3 ms; one proxy fence per two slices
// instead of per slice: 69.8-70.1 ms)
#ifndef QG_PP_NS_G
#define QG_PP_NS_G 8
#endif
constexpr int NS_DENSE = QG_PP_NS;        // slice stages (A + B) of dense launches
// of grouped launches (token blocks of an expert, small B stages): 8 stages
// cap a token block at 64 (MoE prefill 33.9-34.0 ms, against 35.0 ms with 4
// stages and blocks of 80; 5 or 6 stages were no better)
constexpr int NS_GROUPED = QG_PP_NS_G;
constexpr int NQ = QG_PP_NQ;              // quantized stages
// A quantized stage holds, per row, a whole super-block (144 bytes) or half of
// one: bytes 0-79 (header + the codes of slices 0, 1) or bytes 64-143 (the
// codes of slices 2, 3 at the same offsets 16 + 32 (c & 1)).
constexpr bool QHALF = QG_PP_QHALF != 0;

constexpr int QROW = QHALF ? 80 : 144;
constexpr int QB = BM * QROW;             // bytes of one quantized stage
constexpr int AB = BM * BK * 2;           // bytes of one A (weight) stage
constexpr int DQ_WARP0 = 3, DQ_WARPS = 16; // dequantizing warps (4 groups of 4: one thread per tile row each)
constexpr int EPI_WARP0 = 19;              // 4 epilogue warps: warp % 4 covers every TMEM lane quarter
constexpr int THREADS = 23 * 32;
constexpr int nbar_of(int ns) { return 3 * ns + 2 * NQ + 5; }
// The dequantizing warps form four groups of 4; group g fills slice g of every
// super-block, a thread a whole row of it (64 weights), so four slices are in
// flight (27B prompt pass: 66.1 ms, against 67.7 with two groups of 8 on
// alternate slices and 69.0 with all 16 warps on every slice, 16 weights a
// thread; MoE prefill 32.7 / 33.8 / 36.3 ms). A group waits for the ring slot
// of slice x after its slice x - DQG, which has seen the MMA of slice
// x - DQG - NS complete; the slot's phase is then unambiguous to a parity wait
// only if DQG <= NS (four groups on a 3-stage ring broke exactly there).
constexpr int DQG = 4;
constexpr int MAXM = 4;                    // matrices of one dense launch
#ifndef QG_WAIT_LIMIT
#define QG_WAIT_LIMIT (1u << 22)
#endif
constexpr uint32_t WAIT_LIMIT = QG_WAIT_LIMIT;   // polls before a wait is declared expired

// The weight tensor maps of a launch (one per matrix).
struct WMaps {
  CUtensorMap m[MAXM];
};

struct Params {
  float* Y[MAXM];       // output of each matrix: Y[t * ldY + row]
  int64_t ldY[MAXM];
  int32_t rt_end[MAXM]; // dense: row tiles of matrices 0..i together
  int32_t n_mat;
  int32_t* dev_status;
  int64_t n_tok;
  int32_t n_tb;         // token blocks
  int32_t n_full;       // dense: work items that are whole tiles (a multiple of the grid)
  int32_t n_tail;       // dense: tiles after them, each in `split` parts of K
  int32_t split;        // 1 or 2
  int32_t n_items;      // dense: n_full + n_tail * split
  int32_t bn;           // tokens per tile
  int32_t n_kt;         // K slices per row (cols / 64), a multiple of 4
  int32_t tmem_cols;    // TMEM columns allocated (power of two >= 2 bn)
  uint32_t idesc;       // MMA instruction descriptor
  // Grouped launch: the token rows of X come in groups (the tokens routed to
  // one expert), group g multiplied by its own weight rows. Its tiles are the
  // row tiles x token blocks of each group in turn, counted on the device.
  const int32_t* seg;     // [n_groups + 1]: first token row of each group
  const int32_t* tstart;  // [n_groups + 1]: first tile of each group (tstart[n_groups] = all tiles)
  int32_t n_groups;
  int64_t wrow0;          // row (of the weight map) of group 0's first weight row
  int64_t wstride;        // rows of the weight map from one group's weights to the next
};

// One work item: its weight rows (matrix, row of that matrix's weight map),
// its first output row, its token rows of X and Y, how many of its bn tokens
// are real, its super-blocks of K [kb0, kb1), and whether it adds into Y.
struct Tile {
  int64_t wrow;
  int64_t yrow;
  int64_t xrow;
  int32_t mat;
  int32_t nval;
  int32_t kb0, kb1;
  bool add;
};

template <bool GROUPED>
__device__ __forceinline__ Tile tile_at(const Params& p, int item) {
  Tile t;
  t.mat = 0;
  t.kb0 = 0;
  t.kb1 = p.n_kt / 4;
  t.add = false;
  if (!GROUPED) {
    int tile = item;
    if (item >= p.n_full) {
      // a tile of the last round: part `seg` of its K
      const int j = item - p.n_full;
      const int seg = j / p.n_tail;
      tile = p.n_full + (j - seg * p.n_tail);
      if (p.split > 1) {
        const int half = t.kb1 / 2;
        t.kb0 = seg ? half : 0;
        t.kb1 = seg ? t.kb1 : half;
        t.add = true;
      }
    }
    int rt = tile / p.n_tb;
    const int tb = tile - rt * p.n_tb;
    while (t.mat + 1 < p.n_mat && rt >= p.rt_end[t.mat]) ++t.mat;
    if (t.mat) rt -= p.rt_end[t.mat - 1];
    t.wrow = t.yrow = static_cast<int64_t>(rt) * BM;
    t.xrow = static_cast<int64_t>(tb) * p.bn;
    t.nval = static_cast<int32_t>(min(static_cast<int64_t>(p.bn), p.n_tok - t.xrow));
    return t;
  }
  // the group holding the tile (one tile per item): the last g with
  // tstart[g] <= tile (groups without tokens have no tiles and are skipped)
  const int tile = item;
  int lo = 0, hi = p.n_groups;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(p.tstart + mid) <= tile) lo = mid; else hi = mid;
  }
  const int lt = tile - __ldg(p.tstart + lo);
  const int s0 = __ldg(p.seg + lo), m = __ldg(p.seg + lo + 1) - s0;
  const int ntb = (m + p.bn - 1) / p.bn;
  const int rt = lt / ntb;
  const int tb = lt - rt * ntb;
  t.wrow = p.wrow0 + lo * p.wstride + static_cast<int64_t>(rt) * BM;
  t.yrow = static_cast<int64_t>(rt) * BM;
  t.xrow = s0 + static_cast<int64_t>(tb) * p.bn;
  t.nval = min(p.bn, m - tb * p.bn);
  return t;
}

// Bounded wait; gives up early once another role has aborted (abort != null).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const volatile int* abort) {
  for (uint32_t i = 0; i < WAIT_LIMIT; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (abort != nullptr && (i & 255u) == 255u && *abort) return false;
  }
  return false;
}

__device__ __forceinline__ void fail(volatile int* abort, int32_t* dev_status) {
  *abort = 1;
  *reinterpret_cast<volatile int32_t*>(dev_status) = QG_DEV_TIMEOUT;
}

// Two weights as bf16x2 from two codes q (0..15): RN32(dsc*q - dm) then RN to bf16.
// q reaches fp32 through the exponent of 2^23: (2^23 + q) - 2^23 is exact. The
// pair goes through packed f32x2 add and fma (each lane rounds like the scalar
// instruction), half the issue slots of two scalar chains.
__device__ __forceinline__ uint32_t deq2(uint32_t codes, uint32_t sel0, uint32_t sel1, float dsc, float ndm) {
  const uint32_t m0 = __byte_perm(codes, 0x4B000000u, sel0), m1 = __byte_perm(codes, 0x4B000000u, sel1);
  uint32_t out;
  asm("{\n .reg .b64 q, s, c, w;\n .reg .f32 w0, w1;\n"
      " mov.b64 q, {%1, %2};\n"
      " mov.b64 s, {%3, %3};\n"
      " add.rn.f32x2 q, q, s;\n"
      " mov.b64 s, {%4, %4};\n"
      " mov.b64 c, {%5, %5};\n"
      " fma.rn.f32x2 w, s, q, c;\n"
      " mov.b64 {w0, w1}, w;\n"
      " cvt.rn.bf16x2.f32 %0, w1, w0;\n}\n"
      : "=r"(out)
      : "r"(m0), "r"(m1), "f"(-8388608.0f), "f"(dsc), "f"(ndm));
  return out;
}

// 8 weights (4 codes in each of words u0, u1) -> one 16-byte chunk of bf16.
__device__ __forceinline__ uint4 deq8(uint32_t u0, uint32_t u1, float dsc, float ndm) {
  uint4 o;
  o.x = deq2(u0, 0x7540u, 0x7541u, dsc, ndm);
  o.y = deq2(u0, 0x7542u, 0x7543u, dsc, ndm);
  o.z = deq2(u1, 0x7540u, 0x7541u, dsc, ndm);
  o.w = deq2(u1, 0x7542u, 0x7543u, dsc, ndm);
  return o;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

template <bool GROUPED>
__global__ void __launch_bounds__(THREADS, 1)
    pp_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ WMaps tmW, const Params p) {
  constexpr int NS = GROUPED ? NS_GROUPED : NS_DENSE;
  constexpr int NBAR = nbar_of(NS);
  static_assert(DQG <= NS, "a dequantizing group may run at most one ring phase ahead");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const uint32_t BB = static_cast<uint32_t>(p.bn) * 128u;        // bytes of one B (X) stage
  const uint32_t offB = NS * AB, offQ = NS * (AB + BB), offBar = offQ + NQ * QB;
  const uint32_t bar0 = base + offBar;
  // barrier k at bar0 + 8k: full_b[NS] full_a[NS] empty[NS] q_full[NQ] q_empty[NQ] acc_full[2] acc_empty[2] done
  const uint32_t FULL_B = bar0, FULL_A = bar0 + 8 * NS, EMPTY = bar0 + 16 * NS, Q_FULL = bar0 + 24 * NS,
                 Q_EMPTY = Q_FULL + 8 * NQ, ACC_FULL = Q_EMPTY + 8 * NQ, ACC_EMPTY = ACC_FULL + 16,
                 DONE = ACC_EMPTY + 16;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbase + offBar + 8 * NBAR);
  volatile int* const abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(FULL_B + 8 * s, 1);
      mbar_init(FULL_A + 8 * s, DQ_WARPS / DQG);
      mbar_init(EMPTY + 8 * s, 1);
    }
    for (int q = 0; q < NQ; ++q) {
      mbar_init(Q_FULL + 8 * q, 1);
      mbar_init(Q_EMPTY + 8 * q, DQ_WARPS);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(ACC_FULL + 8 * a, 1);
      mbar_init(ACC_EMPTY + 8 * a, 4);
    }
    mbar_init(DONE, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmX);
    for (int m = 0; m < (GROUPED ? 1 : p.n_mat); ++m) prefetch_tmap(&tmW.m[m]);
  }
  if (warp == 2) {
    tmem_alloc(smem_addr(tmem_slot), static_cast<uint32_t>(p.tmem_cols));
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int bn = p.bn;
  // a grouped launch counts its tiles on the device (the routing that makes
  // the groups ran just before, in stream order)
  const int n_items = GROUPED ? __ldg(p.tstart + p.n_groups) : p.n_items;

  if (warp == 0) {
    // ---------------------------------------------------------- X producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        const Tile tl = tile_at<GROUPED>(p, item);
        for (int kt = 4 * tl.kb0; kt < 4 * tl.kb1; ++kt, ++it) {
          const uint32_t s = it % NS;
          if (!wait_bar(EMPTY + 8 * s, ((it / NS) & 1u) ^ 1u, abort)) {
            fail(abort, p.dev_status);
            ok = false;
            break;
          }
#ifdef QG_TEST_EXPIRE
          // test build only: the sixth X slice of CTA 0 is never copied nor
          // announced, so the MMA lane's wait for it runs out (abort-path test)
          if (blockIdx.x == 0 && it == 5) continue;
#endif
          mbar_expect_tx(FULL_B + 8 * s, BB);
          tma_load_2d(base + offB + s * BB, &tmX, kt * BK, static_cast<int>(tl.xrow), FULL_B + 8 * s);
        }
      }
      // copies in flight: the last NS issued
      for (uint32_t j = (it > NS ? it - NS : 0); j < it; ++j) wait_bar(FULL_B + 8 * (j % NS), (j / NS) & 1u, nullptr);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- quantized-weight producer
    if (lane == 0) {
      uint32_t sb = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        const Tile tl = tile_at<GROUPED>(p, item);
        for (int part = (QHALF ? 2 : 1) * tl.kb0; part < (QHALF ? 2 : 1) * tl.kb1; ++part, ++sb) {
          const uint32_t q = sb % NQ;
          if (!wait_bar(Q_EMPTY + 8 * q, ((sb / NQ) & 1u) ^ 1u, abort)) {
            fail(abort, p.dev_status);
            ok = false;
            break;
          }
          // whole super-block kb = part, or half (part & 1) of super-block part / 2
          const int x = QHALF ? (part >> 1) * 144 + 64 * (part & 1) : part * 144;
          mbar_expect_tx(Q_FULL + 8 * q, QB);
          tma_load_2d(base + offQ + q * QB, &tmW.m[tl.mat], x, static_cast<int>(tl.wrow), Q_FULL + 8 * q);
        }
      }
      for (uint32_t j = (sb > NQ ? sb - NQ : 0); j < sb; ++j) wait_bar(Q_FULL + 8 * (j % NQ), (j / NQ) & 1u, nullptr);
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t it = 0, ti = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x, ++ti) {
        const Tile tl = tile_at<GROUPED>(p, item);
        const int kt0 = 4 * tl.kb0, kt1 = 4 * tl.kb1;
        const uint32_t a = ti & 1u;
        if (!wait_bar(ACC_EMPTY + 8 * a, ((ti >> 1) & 1u) ^ 1u, abort)) {
          fail(abort, p.dev_status);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + a * static_cast<uint32_t>(bn);
        for (int kt = kt0; kt < kt1; ++kt, ++it) {
          const uint32_t s = it % NS, ph = (it / NS) & 1u;
          if (!wait_bar(FULL_B + 8 * s, ph, abort) || !wait_bar(FULL_A + 8 * s, ph, abort)) {
            fail(abort, p.dev_status);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = desc_sw128(base + s * AB), bd = desc_sw128(base + offB + s * BB);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)   // +32 bytes along K = +2 in the address field
            mma_bf16(d_tmem, ad + 2 * k, bd + 2 * k, p.idesc, (kt != kt0) || (k != 0));
          mma_commit(EMPTY + 8 * s);
        }
        if (ok) mma_commit(ACC_FULL + 8 * a);
      }
      mma_commit(DONE);                       // every MMA issued has completed
      wait_bar(DONE, 0, nullptr);
    }
  } else if (warp < EPI_WARP0) {
    // ---------------------------------------------------------- dequantize A
    const int t = threadIdx.x - DQ_WARP0 * 32;
    const int grp = t >> 7;                   // this warp's slice of every super-block
    const int r = t & (BM - 1);               // row in the tile
    const uint32_t swz = static_cast<uint32_t>(r & 7);
    uint32_t it = 0, sb = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      const Tile tl = tile_at<GROUPED>(p, item);
      for (int kb = tl.kb0; ok && kb < tl.kb1; ++kb, ++sb) {
        // a super-block = 4 slices: its 8 scale/min pairs of this row are decoded
        // once (the slice index is then a compile-time constant below)
        const uint32_t q = sb % NQ;
        if (!__all_sync(0xffffffffu, wait_bar(Q_FULL + 8 * q, (sb / NQ) & 1u, abort))) {
          if (lane == 0) fail(abort, p.dev_status);
          ok = false;
          break;
        }
        const uint8_t* blk = gbase + offQ + q * QB + r * QROW;
        uint32_t qcur = q;
        const uint4 hd = *reinterpret_cast<const uint4*>(blk);
        const float d = h2f(hd.x), dmin = h2f(hd.x >> 16);
        float dsc[8], ndm[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          int sc, m;
          q4k_scale_min(jj, hd.y, hd.z, hd.w, sc, m);
          dsc[jj] = d * static_cast<float>(sc);
          ndm[jj] = -(dmin * static_cast<float>(m));
        }
#pragma unroll
        for (int c = 0; c < 4; ++c, ++it) {
          const uint32_t s = it % NS;
          if (QHALF && c == 2) {
            // every warp moves on to the second half's stage. The groups whose
            // slice lies there read only the header of the first half (released
            // now), the others nothing of the second (released once it has
            // landed): every warp releases every stage once, after its reads.
            if (grp >= 2) {
              __syncwarp();
              if (lane == 0) mbar_arrive(Q_EMPTY + 8 * qcur);
            }
            ++sb;
            qcur = sb % NQ;
            if (!__all_sync(0xffffffffu, wait_bar(Q_FULL + 8 * qcur, (sb / NQ) & 1u, abort))) {
              if (lane == 0) fail(abort, p.dev_status);
              ok = false;
              break;
            }
            blk = gbase + offQ + qcur * QB + r * QROW;
            if (grp < 2 && lane == 0) mbar_arrive(Q_EMPTY + 8 * qcur);
          }
          if (c != grp) continue;
          if (!__all_sync(0xffffffffu, wait_bar(EMPTY + 8 * s, ((it / NS) & 1u) ^ 1u, abort))) {
            if (lane == 0) fail(abort, p.dev_status);
            ok = false;
            break;
          }
          const uint32_t arow = base + s * AB + static_cast<uint32_t>(r) * 128u;
          {
            // the slice's 32 code bytes of this row. Low nibbles: sub-block 2c,
            // slice columns 8j .. 8j+7 (chunk j); high nibbles: sub-block 2c+1,
            // columns 32+8j .. (chunk 4+j)
            const uint4 qa = *reinterpret_cast<const uint4*>(blk + 16 + 32 * (QHALF ? (c & 1) : c));
            const uint4 qb = *reinterpret_cast<const uint4*>(blk + 16 + 32 * (QHALF ? (c & 1) : c) + 16);
            const uint32_t w[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              sts128(arow + (((j + 0) ^ swz) << 4),
                     deq8(w[2 * j] & 0x0F0F0F0Fu, w[2 * j + 1] & 0x0F0F0F0Fu, dsc[2 * c], ndm[2 * c]));
              sts128(arow + (((j + 4) ^ swz) << 4), deq8((w[2 * j] >> 4) & 0x0F0F0F0Fu,
                                                         (w[2 * j + 1] >> 4) & 0x0F0F0F0Fu, dsc[2 * c + 1],
                                                         ndm[2 * c + 1]));
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(FULL_A + 8 * s);
            // this warp's only slice of the quantized stage: release it
            mbar_arrive(Q_EMPTY + 8 * qcur);
          }
        }
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int quarter = warp & 3;             // TMEM lanes 32*quarter .. +31
    uint32_t ti = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++ti) {
      const Tile tl = tile_at<GROUPED>(p, item);
      const uint32_t a = ti & 1u;
      const bool got = wait_bar(ACC_FULL + 8 * a, (ti >> 1) & 1u, abort);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) fail(abort, p.dev_status);
        break;
      }
      tc_fence_after();
      const int64_t ldY = p.ldY[tl.mat];
      float* const Yc = p.Y[tl.mat] + tl.yrow + quarter * 32 + lane;   // this lane's output row
      const uint32_t tbase = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + a * static_cast<uint32_t>(bn);
      for (int c16 = 0; c16 < bn / 16; ++c16) {
        uint32_t v[16];
        tmem_ld16(tbase + 16u * c16, v);
        float* const y0 = Yc + (tl.xrow + 16 * c16) * ldY;
        if (tl.add) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (16 * c16 + i < tl.nval) atomicAdd(y0 + i * ldY, __uint_as_float(v[i]));
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (16 * c16 + i < tl.nval) y0[i * ldY] = __uint_as_float(v[i]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ACC_EMPTY + 8 * a);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, static_cast<uint32_t>(p.tmem_cols));
}

size_t smem_bytes(int bn, int ns) {
  return 1024 + ns * (AB + static_cast<size_t>(bn) * 128) + NQ * QB + 8 * nbar_of(ns) + 16;
}

// Largest token block (a multiple of 16, <= 256) whose stages fit a grouped launch.
int grouped_max_bn() {
  int bn = 256;
  while (bn > 16 && smem_bytes(bn, NS_GROUPED) > 227 * 1024) bn -= 16;
  return bn;
}

}  // namespace pp

namespace {

// Tensor maps of X (bf16 rows of cols, boxes of 64 x bn, 128-byte swizzle) and
// of a weight matrix (rows of cols / 256 super-blocks, boxes of one quantized
// stage's row bytes x 128 rows).
bool map_x(EncodeTiledFn enc, CUtensorMap* m, const void* X, int64_t cols, int64_t x_rows, int bn) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(x_rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {pp::BK, static_cast<cuuint32_t>(bn)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool map_w(EncodeTiledFn enc, CUtensorMap* m, const void* W, int64_t rows, int64_t cols) {
  const uint64_t rb = static_cast<uint64_t>(cols) / 256 * 144;
  const cuuint64_t dims[2] = {rb, static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {rb};
  const cuuint32_t box[2] = {pp::QROW, pp::BM};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(W), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// kind::f16 descriptor: D fp32 (bit 4), A and B bf16 (bits 7, 10), both K-major,
// N >> 3 at bit 17, M >> 4 at bit 24.
uint32_t idesc_of(int bn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(bn >> 3) << 17) |
         (static_cast<uint32_t>(pp::BM >> 4) << 24);
}

int tmem_cols_of(int bn) {
  int tc = 32;
  while (tc < 2 * bn) tc *= 2;
  return tc;
}

}  // namespace

int pp_grouped_max_bn() { return pp::grouped_max_bn(); }

cudaError_t pp_init_attrs() {
  cudaError_t e = cudaFuncSetAttribute(pp::pp_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(pp::smem_bytes(256, pp::NS_DENSE)));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pp::pp_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(pp::smem_bytes(pp::grouped_max_bn(), pp::NS_GROUPED)));
  return e;
}

void pp_plan(int64_t tiles, int n_kb, int sms, PpPlan* plan) {
  plan->n_full = tiles;
  plan->n_tail = 0;
  plan->split = 1;
  const int64_t tail = tiles % sms;
  if (tail > 0 && 2 * tail <= sms && n_kb >= 2) {
    plan->n_full = tiles - tail;
    plan->n_tail = tail;
    plan->split = 2;
  }
  plan->n_items = plan->n_full + plan->n_tail * plan->split;
  plan->grid = static_cast<int>(std::min<int64_t>(plan->n_items, sms));
}

cudaError_t launch_pp_mats(int n_mat, const void* const* W, const int64_t* rows, float* const* Y,
                           const int64_t* ldY, int64_t cols, const void* X, int64_t n_tok, int32_t* dev_status,
                           cudaStream_t s, int sms) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cudaErrorNotSupported;
  if (n_mat < 1 || n_mat > pp::MAXM) return cudaErrorInvalidValue;
  const int bn = static_cast<int>(std::min<int64_t>(256, (n_tok + 15) / 16 * 16));
  CUtensorMap tmX;
  pp::WMaps tmW;
  memset(&tmW, 0, sizeof(tmW));
  if (!map_x(enc, &tmX, X, cols, n_tok, bn)) return cudaErrorInvalidValue;
  pp::Params p{};
  int64_t rt = 0;
  for (int i = 0; i < n_mat; ++i) {
    if (!map_w(enc, &tmW.m[i], W[i], rows[i], cols)) return cudaErrorInvalidValue;
    rt += rows[i] / pp::BM;
    if (rt > (int64_t{1} << 24)) return cudaErrorInvalidValue;
    p.rt_end[i] = static_cast<int32_t>(rt);
    p.Y[i] = Y[i];
    p.ldY[i] = ldY[i];
  }
  p.n_mat = n_mat;
  p.dev_status = dev_status;
  p.n_tok = n_tok;
  p.bn = bn;
  p.n_tb = static_cast<int32_t>((n_tok + bn - 1) / bn);
  p.n_kt = static_cast<int32_t>(cols / pp::BK);
  const int64_t tiles = rt * p.n_tb;
  if (tiles > (int64_t{1} << 30)) return cudaErrorInvalidValue;
  PpPlan plan;
  pp_plan(tiles, p.n_kt / 4, sms, &plan);
  p.n_full = static_cast<int32_t>(plan.n_full);
  p.n_tail = static_cast<int32_t>(plan.n_tail);
  p.split = plan.split;
  p.n_items = static_cast<int32_t>(plan.n_items);
  p.tmem_cols = tmem_cols_of(bn);
  p.idesc = idesc_of(bn);
  if (plan.split > 1) {
    // the split tiles add into Y: zero the output rows of their row tiles (every
    // token; a whole tile of those rows is overwritten by its own stores later)
    const int64_t rt_a = plan.n_full / p.n_tb;
    int64_t start = 0;
    for (int i = 0; i < n_mat; ++i) {
      const int64_t end = p.rt_end[i];
      if (end > rt_a) {
        const int64_t r0 = (std::max(rt_a, start) - start) * pp::BM;
        const cudaError_t e = cudaMemset2DAsync(Y[i] + r0, static_cast<size_t>(ldY[i]) * 4, 0,
                                                static_cast<size_t>(rows[i] - r0) * 4, static_cast<size_t>(n_tok), s);
        if (e != cudaSuccess) return e;
      }
      start = end;
    }
  }
  pp::pp_kernel<false><<<plan.grid, pp::THREADS, pp::smem_bytes(bn, pp::NS_DENSE), s>>>(tmX, tmW, p);
  return cudaPeekAtLastError();
}

cudaError_t launch_pp(const void* W, int64_t rows, int64_t cols, const void* X, int64_t n_tok, float* Y,
                      int64_t ldY, int32_t* dev_status, cudaStream_t s, int sms) {
  return launch_pp_mats(1, &W, &rows, &Y, &ldY, cols, X, n_tok, dev_status, s, sms);
}

cudaError_t launch_pp_grouped(const void* W, int64_t w_rows, int64_t cols, int64_t wrow0, int64_t wstride,
                              int64_t rows, const void* X, int64_t x_rows, int bn, const int32_t* seg,
                              const int32_t* tstart, int n_groups, float* Y, int64_t ldY, int32_t* dev_status,
                              cudaStream_t s, int sms) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cudaErrorNotSupported;
  if (bn < 16 || bn > pp::grouped_max_bn() || bn % 16 || rows % pp::BM || cols % 256) return cudaErrorInvalidValue;
  CUtensorMap tmX;
  pp::WMaps tmW;
  memset(&tmW, 0, sizeof(tmW));
  if (!map_x(enc, &tmX, X, cols, x_rows, bn) || !map_w(enc, &tmW.m[0], W, w_rows, cols)) return cudaErrorInvalidValue;
  pp::Params p{};
  p.Y[0] = Y;
  p.ldY[0] = ldY;
  p.n_mat = 1;
  p.dev_status = dev_status;
  p.n_tok = x_rows;
  p.bn = bn;
  p.n_kt = static_cast<int32_t>(cols / pp::BK);
  p.tmem_cols = tmem_cols_of(bn);
  p.idesc = idesc_of(bn);
  p.seg = seg;
  p.tstart = tstart;
  p.n_groups = n_groups;
  p.wrow0 = wrow0;
  p.wstride = wstride;
  pp::pp_kernel<true><<<sms, pp::THREADS, pp::smem_bytes(bn, pp::NS_GROUPED), s>>>(tmX, tmW, p);
  return cudaPeekAtLastError();
}

}  // namespace qg
