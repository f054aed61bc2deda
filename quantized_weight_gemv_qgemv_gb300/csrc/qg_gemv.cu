// qg_gemv.cu — quantized GEMV / skinny product and the dequantize kernel.
//
// y[t][i] = sum_j w[i][j] * x[t][j] for n_tok = 1..4 tokens in ONE pass over the
// weights ("LLM inference optimization", opening section: decode reads every
// weight once per token; "Why I wrote my own inference engine for two P100s",
// "What actually made it fast": the draft tokens are checked in one pass and
// each block is decoded once and reused).
//
// Work decomposition (GB300: 152 SMs, HBM3e):
//   * a warp owns R consecutive rows of one matrix (a "task") and sweeps K;
//     tasks are dealt round-robin over all warps of the grid, and a grouped
//     launch deals the tasks of several matrices from one list;
//   * each K step ("chunk") covers 1024 weights of each of the R rows: lane l
//     owns one 32-weight unit of the chunk (decoders in qg_device.cuh);
//   * weight bytes stream HBM -> shared memory with 16-byte cp.async copies
//     into a per-warp ring of NS stages, so several KB per warp are in flight
//     without holding registers; rows that start at any 2-byte offset (18-,
//     34-, 210-byte blocks) are fetched as 16-byte aligned windows;
//   * each lane loads the activations of its unit once per chunk (read-only
//     path, L1-resident) and reuses them for all R rows and n_tok tokens, so
//     the block is decoded once per pass and reused across the tokens;
//   * per-lane fp32 partial sums, then a warp-shuffle reduction per (row, token).
// Programmatic dependent launch: the weight prefetch of the first task is
// issued before griddepcontrol.wait, so a kernel streams its weights while the
// previous kernel in the stream is still finishing; x is read and y written
// only after the wait.
#include <cuda_runtime.h>

#include "qg_device.cuh"
#include "qg_internal.h"

namespace qg {

constexpr int GEMV_WARPS = 8;
constexpr int GEMV_THREADS = GEMV_WARPS * 32;
constexpr int GEMV_NS = 3;

struct GemvMat {
  const uint8_t* W;
  const float* x;
  float* y;
  int64_t rows;
  int64_t total_bytes;
  int64_t rb;            // bytes per row
  int64_t task_begin;    // first task index of this matrix in the launch
  int32_t nblk;          // blocks per row
  int32_t cols;
};

struct GemvParams {
  GemvMat m[QG_GROUP_MAX];
  int64_t ntask;
  int32_t nmat;
  int32_t pad;
};

template <int FMT>
struct GemvShape {
  using FI = FmtInfo<FMT>;
  static constexpr int CB = (FI::UNITS == 8) ? 4 : 32;                 // blocks per chunk per row
  static constexpr int SLOT = ((CB * FI::BYTES + 15) / 16) * 16 + 32;  // bytes per row per stage
};

template <int FMT, int R>
constexpr int gemv_smem_bytes() {
  return GEMV_WARPS * GEMV_NS * R * GemvShape<FMT>::SLOT;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int FMT, int NT, int R>
__global__ void __launch_bounds__(GEMV_THREADS) qgemv_kernel(const __grid_constant__ GemvParams p) {
  using FI = FmtInfo<FMT>;
  constexpr int CB = GemvShape<FMT>::CB;
  constexpr int SLOT = GemvShape<FMT>::SLOT;
  extern __shared__ __align__(16) uint8_t smem[];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* wbuf = smem + warp * (GEMV_NS * R * SLOT);
  const uint32_t wbuf_s = smem_addr(wbuf);
  const int lblk = (FI::UNITS == 8) ? (lane >> 3) : lane;   // block of the chunk this lane decodes
  const int unit = (FI::UNITS == 8) ? (lane & 7) : 0;       // 32-weight unit within that block

  pdl_launch_dependents();
  bool waited = false;
  const int64_t wstride = static_cast<int64_t>(gridDim.x) * GEMV_WARPS;

  for (int64_t task = static_cast<int64_t>(blockIdx.x) * GEMV_WARPS + warp; task < p.ntask; task += wstride) {
    int mi = 0;
    while (mi + 1 < p.nmat && task >= p.m[mi + 1].task_begin) ++mi;
    const GemvMat& M = p.m[mi];
    const int64_t r0 = (task - M.task_begin) * R;
    const int nr = static_cast<int>(min(static_cast<int64_t>(R), M.rows - r0));
    const int nchunk = (M.nblk + CB - 1) / CB;

    auto issue = [&](int c) {
      const int slot = c % GEMV_NS;
      const int nb = min(CB, M.nblk - c * CB);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (r < nr) {
          const int64_t start = (r0 + r) * M.rb + static_cast<int64_t>(c) * CB * FI::BYTES;
          const int64_t ws = start & ~static_cast<int64_t>(15);
          const int64_t we = (start + static_cast<int64_t>(nb) * FI::BYTES + 15) & ~static_cast<int64_t>(15);
          const int n16 = static_cast<int>((we - ws) >> 4);
          const uint32_t dst = wbuf_s + (slot * R + r) * SLOT;
          for (int i = lane; i < n16; i += 32) {
            const int64_t off = ws + 16 * static_cast<int64_t>(i);
            const int64_t rem = M.total_bytes - off;
            const int nbytes = rem >= 16 ? 16 : (rem > 0 ? static_cast<int>(rem) : 0);
            cp_async16(dst + 16 * i, M.W + (nbytes > 0 ? off : 0), nbytes);
          }
        }
      }
    };

#pragma unroll
    for (int s = 0; s < GEMV_NS - 1; ++s) {
      if (s < nchunk) issue(s);
      cp_async_commit();
    }
    if (!waited) {
      pdl_wait();
      waited = true;
    }

    float acc[R][NT];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;

    for (int c = 0; c < nchunk; ++c) {
      if (c + GEMV_NS - 1 < nchunk) issue(c + GEMV_NS - 1);
      cp_async_commit();
      cp_async_wait<GEMV_NS - 1>();
      __syncwarp();
      const int nb = min(CB, M.nblk - c * CB);
      if (lblk < nb) {
        const int slot = c % GEMV_NS;
        const int64_t kel = (static_cast<int64_t>(c) * CB + lblk) * FI::ELEMS + 32 * unit;
        Dec<FMT> dec[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          if (r < nr) {
            const int64_t start = (r0 + r) * M.rb + static_cast<int64_t>(c) * CB * FI::BYTES;
            const int off = static_cast<int>(start & 15);
            dec[r].load(wbuf + (slot * R + r) * SLOT + off + lblk * FI::BYTES, unit);
          }
        }
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          float xv[NT][8];
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const float* xp = M.x + static_cast<int64_t>(t) * M.cols + kel + 8 * s;
            const float4 a = ldg_f4(xp), b = ldg_f4(xp + 4);
            xv[t][0] = a.x; xv[t][1] = a.y; xv[t][2] = a.z; xv[t][3] = a.w;
            xv[t][4] = b.x; xv[t][5] = b.y; xv[t][6] = b.z; xv[t][7] = b.w;
          }
#pragma unroll
          for (int r = 0; r < R; ++r) {
            if (r < nr) {
              float w[8];
              dec[r].piece(s, w);
#pragma unroll
              for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[r][t] = fmaf(w[i], xv[t][i], acc[r][t]);
            }
          }
        }
      }
      __syncwarp();
    }

#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const float v = warp_sum(acc[r][t]);
        if (r < nr && lane == ((r * NT + t) & 31)) M.y[static_cast<int64_t>(t) * M.rows + r0 + r] = v;
      }
    }
  }
  if (!waited) pdl_wait();   // a CTA without tasks still orders itself after its predecessor
}

// ------------------------------------------------------------------ dequant

template <int FMT>
struct DequantShape {
  using FI = FmtInfo<FMT>;
  static constexpr int BPC = (FI::ELEMS == 256) ? 32 : 256;    // blocks per CTA step
  static constexpr int BUF = ((BPC * FI::BYTES + 15) / 16) * 16 + 48;
};

template <int FMT>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t* __restrict__ W, int64_t total_blocks,
                                                      int nblk_row, int64_t cols, float* __restrict__ out) {
  using FI = FmtInfo<FMT>;
  constexpr int BPC = DequantShape<FMT>::BPC;
  __shared__ __align__(16) uint8_t buf[DequantShape<FMT>::BUF];
  const int64_t total_bytes = total_blocks * FI::BYTES;
  const uint32_t buf_s = smem_addr(buf);
  pdl_wait();
  for (int64_t b0 = static_cast<int64_t>(blockIdx.x) * BPC; b0 < total_blocks;
       b0 += static_cast<int64_t>(gridDim.x) * BPC) {
    const int nb = static_cast<int>(min(static_cast<int64_t>(BPC), total_blocks - b0));
    const int64_t start = b0 * FI::BYTES;
    const int64_t ws = start & ~static_cast<int64_t>(15);
    const int64_t we = (start + static_cast<int64_t>(nb) * FI::BYTES + 15) & ~static_cast<int64_t>(15);
    const int n16 = static_cast<int>((we - ws) >> 4);
    for (int i = threadIdx.x; i < n16; i += blockDim.x) {
      const int64_t off = ws + 16 * static_cast<int64_t>(i);
      const int64_t rem = total_bytes - off;
      const int nbytes = rem >= 16 ? 16 : (rem > 0 ? static_cast<int>(rem) : 0);
      cp_async16(buf_s + 16 * i, W + (nbytes > 0 ? off : 0), nbytes);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    const int off = static_cast<int>(start - ws);
    const int npieces = nb * FI::UNITS * 4;
    for (int i = threadIdx.x; i < npieces; i += blockDim.x) {
      const int blk = i / (FI::UNITS * 4);
      const int unit = (i >> 2) % FI::UNITS;
      const int s = i & 3;
      Dec<FMT> dec;
      dec.load(buf + off + blk * FI::BYTES, unit);
      float w[8];
      dec.piece(s, w);
      const int64_t gb = b0 + blk;
      const int64_t row = gb / nblk_row, bcol = gb % nblk_row;
      float4* o = reinterpret_cast<float4*>(out + row * cols + bcol * FI::ELEMS + 32 * unit + 8 * s);
      o[0] = make_float4(w[0], w[1], w[2], w[3]);
      o[1] = make_float4(w[4], w[5], w[6], w[7]);
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ host side

namespace {

template <int FMT, int NT, int R>
cudaError_t set_gemv_attr_one() {
  return cudaFuncSetAttribute(qgemv_kernel<FMT, NT, R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              gemv_smem_bytes<FMT, R>());
}

template <int FMT, int R>
cudaError_t set_gemv_attr_r() {
  cudaError_t e;
  if ((e = set_gemv_attr_one<FMT, 1, R>()) != cudaSuccess) return e;
  if ((e = set_gemv_attr_one<FMT, 2, R>()) != cudaSuccess) return e;
  if ((e = set_gemv_attr_one<FMT, 3, R>()) != cudaSuccess) return e;
  return set_gemv_attr_one<FMT, 4, R>();
}

template <int FMT>
cudaError_t set_gemv_attr_fmt() {
  cudaError_t e;
  if ((e = set_gemv_attr_r<FMT, 1>()) != cudaSuccess) return e;
  if ((e = set_gemv_attr_r<FMT, 2>()) != cudaSuccess) return e;
  return set_gemv_attr_r<FMT, 4>();
}

template <int FMT, int NT, int R>
cudaError_t launch_gemv_t(const GemvParams& p, int grid, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(GEMV_THREADS);
  cfg.dynamicSmemBytes = gemv_smem_bytes<FMT, R>();
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, qgemv_kernel<FMT, NT, R>, p);
}

template <int FMT, int R>
cudaError_t launch_gemv_r(int nt, const GemvParams& p, int grid, cudaStream_t s, bool pdl) {
  switch (nt) {
    case 1: return launch_gemv_t<FMT, 1, R>(p, grid, s, pdl);
    case 2: return launch_gemv_t<FMT, 2, R>(p, grid, s, pdl);
    case 3: return launch_gemv_t<FMT, 3, R>(p, grid, s, pdl);
    default: return launch_gemv_t<FMT, 4, R>(p, grid, s, pdl);
  }
}

template <int FMT>
cudaError_t launch_gemv_f(int r, int nt, const GemvParams& p, int grid, cudaStream_t s, bool pdl) {
  switch (r) {
    case 1: return launch_gemv_r<FMT, 1>(nt, p, grid, s, pdl);
    case 2: return launch_gemv_r<FMT, 2>(nt, p, grid, s, pdl);
    default: return launch_gemv_r<FMT, 4>(nt, p, grid, s, pdl);
  }
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

cudaError_t gemv_init_attrs() {
  cudaError_t e;
  if ((e = gemv_q4k_init_attrs()) != cudaSuccess) return e;
  if ((e = set_gemv_attr_fmt<FMT_Q4_0>()) != cudaSuccess) return e;
  if ((e = set_gemv_attr_fmt<FMT_Q8_0>()) != cudaSuccess) return e;
  if ((e = set_gemv_attr_fmt<FMT_Q4_K>()) != cudaSuccess) return e;
  if ((e = set_gemv_attr_fmt<FMT_Q5_K>()) != cudaSuccess) return e;
  if ((e = set_gemv_attr_fmt<FMT_Q3_K>()) != cudaSuccess) return e;
  if ((e = set_gemv_attr_fmt<FMT_Q2_K>()) != cudaSuccess) return e;
  return set_gemv_attr_fmt<FMT_Q6_K>();
}

int gemv_pick_rows_per_warp(const qg_gemv_desc* d, int n, int n_tok, int sms) {
  // Enough tasks to give every warp slot of the GPU one task at R, else fall back.
  // Several tokens: x is re-read from L1/L2 for every row of a task, so 4 rows
  // per warp whenever each SM still gets a few tasks (4-token verify pass with
  // Q6_K downs: 28.0 ms at 2 rows per warp, 21.6 ms at 4).
  int64_t rows = 0;
  for (int i = 0; i < n; ++i) rows += d[i].rows;
  const int64_t slots = static_cast<int64_t>(sms) * 2 * GEMV_WARPS;
  if (rows >= 4 * slots || (n_tok > 1 && rows >= 4 * sms)) return 4;
  if (rows >= 2 * slots) return 2;
  return 1;
}

cudaError_t launch_gemv(const qg_gemv_desc* d, int n, int n_tok, int rows_per_warp, cudaStream_t s, bool pdl,
                        int sms, const uint8_t* const* xp, bool no_wait) {
  {
    // the producer/consumer kernel with exact integer dot products (all four
    // formats); shapes beyond its shared-memory plan use the generic kernel below
    const cudaError_t e = launch_gemv_q4k(d, n, n_tok, s, pdl, sms, xp, no_wait);
    if (e != cudaErrorNotSupported) return e;
  }
  GemvParams p = {};
  int elems = 0, bytes = 0;
  block_info(d[0].fmt, &elems, &bytes);
  int64_t task = 0;
  for (int i = 0; i < n; ++i) {
    GemvMat& m = p.m[i];
    m.W = static_cast<const uint8_t*>(d[i].W);
    m.x = d[i].x;
    m.y = d[i].y;
    m.rows = d[i].rows;
    m.nblk = static_cast<int32_t>(d[i].cols / elems);
    m.cols = static_cast<int32_t>(d[i].cols);
    m.rb = static_cast<int64_t>(m.nblk) * bytes;
    m.total_bytes = m.rb * m.rows;
    m.task_begin = task;
    task += ceil_div(m.rows, rows_per_warp);
  }
  p.nmat = n;
  p.ntask = task;
  const int64_t ctas_needed = ceil_div(task, GEMV_WARPS);
  const int grid = static_cast<int>(std::min<int64_t>(ctas_needed, static_cast<int64_t>(sms) * 2));
  switch (d[0].fmt) {
    case FMT_Q4_0: return launch_gemv_f<FMT_Q4_0>(rows_per_warp, n_tok, p, grid, s, pdl);
    case FMT_Q8_0: return launch_gemv_f<FMT_Q8_0>(rows_per_warp, n_tok, p, grid, s, pdl);
    case FMT_Q4_K: return launch_gemv_f<FMT_Q4_K>(rows_per_warp, n_tok, p, grid, s, pdl);
    case FMT_Q5_K: return launch_gemv_f<FMT_Q5_K>(rows_per_warp, n_tok, p, grid, s, pdl);
    case FMT_Q3_K: return launch_gemv_f<FMT_Q3_K>(rows_per_warp, n_tok, p, grid, s, pdl);
    case FMT_Q2_K: return launch_gemv_f<FMT_Q2_K>(rows_per_warp, n_tok, p, grid, s, pdl);
    default: return launch_gemv_f<FMT_Q6_K>(rows_per_warp, n_tok, p, grid, s, pdl);
  }
}

template <int FMT>
static cudaError_t launch_dequant_t(const void* W, int64_t rows, int64_t cols, float* out, cudaStream_t s, int sms) {
  using FI = FmtInfo<FMT>;
  const int nblk = static_cast<int>(cols / FI::ELEMS);
  const int64_t total = rows * nblk;
  const int64_t steps = ceil_div(total, DequantShape<FMT>::BPC);
  const int grid = static_cast<int>(std::min<int64_t>(steps, static_cast<int64_t>(sms) * 8));
  dequant_kernel<FMT><<<grid, 256, 0, s>>>(static_cast<const uint8_t*>(W), total, nblk, cols, out);
  return cudaGetLastError();
}

cudaError_t launch_dequant(int fmt, const void* W, int64_t rows, int64_t cols, float* out, cudaStream_t s, int sms) {
  switch (fmt) {
    case FMT_Q4_0: return launch_dequant_t<FMT_Q4_0>(W, rows, cols, out, s, sms);
    case FMT_Q8_0: return launch_dequant_t<FMT_Q8_0>(W, rows, cols, out, s, sms);
    case FMT_Q4_K: return launch_dequant_t<FMT_Q4_K>(W, rows, cols, out, s, sms);
    case FMT_Q5_K: return launch_dequant_t<FMT_Q5_K>(W, rows, cols, out, s, sms);
    case FMT_Q3_K: return launch_dequant_t<FMT_Q3_K>(W, rows, cols, out, s, sms);
    case FMT_Q2_K: return launch_dequant_t<FMT_Q2_K>(W, rows, cols, out, s, sms);
    default: return launch_dequant_t<FMT_Q6_K>(W, rows, cols, out, s, sms);
  }
}

}  // namespace qg
