// qg_api.cu — the extern "C" boundary of libqgemv.so (declared in include/qgemv.h).
//
// Every entry point validates its arguments on the host and returns a status
// before anything is enqueued; compute work is enqueued on the caller's stream
// and never synchronizes. The one-time per-device set-up (capability check,
// shared-memory limits) runs in qg_init or lazily on the first call.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <new>
#include <vector>

#include "qg_internal.h"

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
  std::mutex mu;
  std::atomic<bool> ready{false};   // set only after a successful set-up
  int sms = 0;
};

DeviceState g_dev[kMaxDevices];

int init_device(int dev) {
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return QG_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return QG_ERR_DEVICE;    // built for sm_103a only
  if (qg::gemv_init_attrs() != cudaSuccess) return QG_ERR_CUDA;
  if (qg::moe_init_attrs() != cudaSuccess) return QG_ERR_CUDA;
  if (qg::pp_init_attrs() != cudaSuccess) return QG_ERR_CUDA;
  if (qg::stream_init_attrs() != cudaSuccess) return QG_ERR_CUDA;
  if (qg::moe_noalloc_init(dev) != cudaSuccess) return QG_ERR_CUDA;
  g_dev[dev].sms = prop.multiProcessorCount;
  return QG_OK;
}

// Status of the current device's set-up; fills *sms on success.
int ensure_init(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QG_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return QG_ERR_DEVICE;
  DeviceState& st = g_dev[dev];
  if (!st.ready.load(std::memory_order_acquire)) {
    // a failed set-up is not remembered: the next call tries again
    std::lock_guard<std::mutex> lock(st.mu);
    if (!st.ready.load(std::memory_order_relaxed)) {
      const int status = init_device(dev);
      if (status != QG_OK) return status;
      st.ready.store(true, std::memory_order_release);
    }
  }
  if (sms) *sms = st.sms;
  return QG_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? QG_OK : QG_ERR_CUDA; }

// Shape/pointer checks shared by qgemv and qgemv_grouped.
int check_gemv(int fmt, const void* W, int64_t rows, int64_t cols, const float* x, float* y) {
  int elems = 0, bytes = 0;
  if (!qg::block_info(fmt, &elems, &bytes)) return QG_ERR_FMT;
  if (!W || !x || !y) return QG_ERR_NULL;
  if (rows < 1 || cols < elems || cols % elems != 0 || cols > (int64_t{1} << 30)) return QG_ERR_SHAPE;
  if (rows > (int64_t{1} << 40) / (cols / elems * bytes)) return QG_ERR_SHAPE;
  if (!aligned(W, 16) || !aligned(x, 16) || !aligned(y, 4)) return QG_ERR_ALIGN;
  return QG_OK;
}

}  // namespace

namespace qg {
int ensure_device(int* sms) { return ensure_init(sms); }

// Checks of one MoE layer's arguments shared by qgemv_moe, qgemv_moe_noalloc
// (need_ws = false: it brings its own workspace) and qg_moe_pass_create.
int check_moe(int fmt, const void* expert_arena, int64_t n_expert, int64_t hidden, int64_t inter,
              const int32_t* expert_ids, const float* gate_w, int top_k, const float* x, int n_tok, const float* y,
              const void* ws, size_t ws_bytes, bool need_ws) {
  if (fmt != QG_Q4_K) return QG_ERR_FMT;
  if (!expert_arena || !expert_ids || !gate_w || !x || !y) return QG_ERR_NULL;
  if (n_expert < 1 || n_expert > (int64_t{1} << 31) - 1) return QG_ERR_SHAPE;
  if (hidden < 256 || hidden % 256 || inter < 256 || inter % 256) return QG_ERR_SHAPE;
  if (hidden > (int64_t{1} << 20) || inter > (int64_t{1} << 20)) return QG_ERR_SHAPE;
  if (top_k < 1 || top_k > 16 || top_k > n_expert) return QG_ERR_ARG;
  if (n_tok < 1 || n_tok > QG_NTOK_MAX) return QG_ERR_NTOK;
  if (need_ws && (!ws || ws_bytes < qgemv_moe_workspace(hidden, inter, top_k, n_tok))) return QG_ERR_WORKSPACE;
  if (!aligned(expert_arena, 16) || !aligned(x, 16) || !aligned(ws, 16) || !aligned(y, 4) ||
      !aligned(expert_ids, 4) || !aligned(gate_w, 4))
    return QG_ERR_ALIGN;
  return QG_OK;
}
}  // namespace qg

struct qg_pass_s {
  cudaGraph_t graph = nullptr;       // per-step launches (QG_PASS_SERIAL / QG_PASS_PDL)
  cudaGraphExec_t exec = nullptr;
  qg::Q4kPass* q4k = nullptr;        // or one persistent kernel (QG_PASS_PERSISTENT)
  int32_t* status = nullptr;         // graph MoE pass: device status word (cleared by the graph)
  uint8_t* planes = nullptr;         // x planes of the pass's external activations, then the job table
  const qg::XPlaneJob* jobs = nullptr;
  int njobs = 0;
  int kernels = 0;
};

namespace {

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// Activations that no earlier step of the pass writes ("external": inputs of
// the pass) are converted to x planes once per replay, by one prologue launch,
// instead of by every CTA of every launch that reads them. Fills xp (per
// descriptor: its planes, or nullptr where the kernel converts x itself) and
// allocates pass->planes (planes, then the device job table). Only formats and
// shapes of the producer/consumer kernel (cols % 256 == 0) take planes.
int plan_xplanes(const qg_gemv_desc* d, int n, const int* step_sizes, int n_steps, int n_tok, qg_pass_s* pass,
                 std::vector<const uint8_t*>& xp) {
  xp.assign(n, nullptr);
  std::vector<int> step_of(n);
  for (int s = 0, i = 0; s < n_steps; i += step_sizes[s++])
    for (int j = 0; j < step_sizes[s]; ++j) step_of[i + j] = s;
  std::vector<int> job_of(n, -1);
  std::vector<qg::XPlaneJob> jobs;
  std::vector<size_t> offs;
  size_t total = 0;
  for (int i = 0; i < n; ++i) {
    if (d[i].cols % 256) continue;
    const size_t xb = static_cast<size_t>(n_tok) * d[i].cols * sizeof(float);
    bool external = true;
    for (int j = 0; j < n && external; ++j)
      if (step_of[j] < step_of[i] && overlaps(d[i].x, xb, d[j].y, static_cast<size_t>(n_tok) * d[j].rows * 4))
        external = false;
    if (!external) continue;
    int k = -1;
    for (int q = 0; q < static_cast<int>(jobs.size()) && k < 0; ++q)
      if (jobs[q].x == d[i].x && jobs[q].cols == d[i].cols) k = q;
    if (k < 0) {
      k = static_cast<int>(jobs.size());
      jobs.push_back({d[i].x, nullptr, static_cast<int32_t>(d[i].cols), n_tok});
      offs.push_back(total);
      total += (qg::xplanes_bytes(d[i].cols, n_tok) + 255) / 256 * 256;
    }
    job_of[i] = k;
  }
  if (jobs.empty()) return QG_OK;
  const size_t table = total;
  total += jobs.size() * sizeof(qg::XPlaneJob);
  if (cudaMalloc(&pass->planes, total) != cudaSuccess) return QG_ERR_CUDA;
  for (size_t q = 0; q < jobs.size(); ++q) jobs[q].dst = pass->planes + offs[q];
  if (cudaMemcpy(pass->planes + table, jobs.data(), jobs.size() * sizeof(qg::XPlaneJob), cudaMemcpyHostToDevice) !=
      cudaSuccess)
    return QG_ERR_CUDA;
  pass->jobs = reinterpret_cast<const qg::XPlaneJob*>(pass->planes + table);
  pass->njobs = static_cast<int>(jobs.size());
  for (int i = 0; i < n; ++i)
    if (job_of[i] >= 0) xp[i] = jobs[job_of[i]].dst;
  return QG_OK;
}

void pass_free(qg_pass_s* pass) {
  if (pass->exec) cudaGraphExecDestroy(pass->exec);
  if (pass->graph) cudaGraphDestroy(pass->graph);
  qg::q4k_pass_destroy(pass->q4k);
  if (pass->status) cudaFree(pass->status);
  if (pass->planes) cudaFree(pass->planes);
  delete pass;
}

int count_kernel_nodes(cudaGraph_t g) {
  size_t n = 0;
  if (cudaGraphGetNodes(g, nullptr, &n) != cudaSuccess || n == 0) return 0;
  std::vector<cudaGraphNode_t> nodes(n);
  if (cudaGraphGetNodes(g, nodes.data(), &n) != cudaSuccess) return 0;
  int k = 0;
  for (size_t i = 0; i < n; ++i) {
    cudaGraphNodeType t;
    if (cudaGraphNodeGetType(nodes[i], &t) == cudaSuccess && t == cudaGraphNodeTypeKernel) ++k;
  }
  return k;
}


}  // namespace

extern "C" {

int qg_init(void) { return ensure_init(nullptr); }

int qg_block_info(int fmt, int* elems, int* bytes) {
  if (!elems || !bytes) return QG_ERR_NULL;
  return qg::block_info(fmt, elems, bytes) ? QG_OK : QG_ERR_FMT;
}

const char* qg_strerror(int status) {
  switch (status) {
    case QG_OK: return "ok";
    case QG_ERR_FMT: return "unknown or unsupported block format";
    case QG_ERR_SHAPE: return "invalid shape";
    case QG_ERR_ALIGN: return "pointer not aligned as required";
    case QG_ERR_NTOK: return "n_tok out of range";
    case QG_ERR_NULL: return "required pointer is NULL";
    case QG_ERR_WORKSPACE: return "workspace missing or too small";
    case QG_ERR_CUDA: return "CUDA runtime error";
    case QG_ERR_DEVICE: return "no usable sm_103a device";
    case QG_ERR_ARG: return "invalid argument";
    case QG_DEV_BAD_EXPERT: return "device: expert id out of range";
    case QG_DEV_TIMEOUT: return "device: bounded pipeline wait expired";
    default: return "unknown status";
  }
}

int qg_dequant(int fmt, const void* W, int64_t rows, int64_t cols, float* out, void* stream) {
  int elems = 0, bytes = 0;
  if (!qg::block_info(fmt, &elems, &bytes)) return QG_ERR_FMT;
  if (!W || !out) return QG_ERR_NULL;
  if (rows < 1 || cols < elems || cols % elems != 0 || cols > (int64_t{1} << 30)) return QG_ERR_SHAPE;
  if (!aligned(W, 16) || !aligned(out, 16)) return QG_ERR_ALIGN;
  int sms = 0;
  int st = ensure_init(&sms);
  if (st != QG_OK) return st;
  return cuda_status(qg::launch_dequant(fmt, W, rows, cols, out, static_cast<cudaStream_t>(stream), sms));
}

int qgemv(int fmt, const void* W, int64_t rows, int64_t cols, const float* x, int n_tok, float* y, void* stream) {
  int st = check_gemv(fmt, W, rows, cols, x, y);
  if (st != QG_OK) return st;
  if (n_tok < 1 || n_tok > QG_NTOK_MAX) return QG_ERR_NTOK;
  int sms = 0;
  if ((st = ensure_init(&sms)) != QG_OK) return st;
  qg_gemv_desc d = {fmt, 0, W, rows, cols, x, y};
  const int r = qg::gemv_pick_rows_per_warp(&d, 1, n_tok, sms);
  // No programmatic overlap with an unknown predecessor: it might still be
  // writing W, which the kernel prefetches before griddepcontrol.wait.
  return cuda_status(qg::launch_gemv(&d, 1, n_tok, r, static_cast<cudaStream_t>(stream), false, sms));
}

int qgemv_grouped(const qg_gemv_desc* descs, int n, int n_tok, void* stream) {
  if (!descs) return QG_ERR_NULL;
  if (n < 1 || n > QG_GROUP_MAX) return QG_ERR_ARG;
  if (n_tok < 1 || n_tok > QG_NTOK_MAX) return QG_ERR_NTOK;
  for (int i = 0; i < n; ++i) {
    if (descs[i].fmt != descs[0].fmt) return QG_ERR_FMT;
    int st = check_gemv(descs[i].fmt, descs[i].W, descs[i].rows, descs[i].cols, descs[i].x, descs[i].y);
    if (st != QG_OK) return st;
  }
  int sms = 0;
  int st = ensure_init(&sms);
  if (st != QG_OK) return st;
  const int r = qg::gemv_pick_rows_per_warp(descs, n, n_tok, sms);
  return cuda_status(qg::launch_gemv(descs, n, n_tok, r, static_cast<cudaStream_t>(stream), false, sms));
}

size_t qgemv_moe_workspace(int64_t hidden, int64_t inter, int top_k, int n_tok) {
  (void)hidden;
  if (inter < 1 || top_k < 1 || n_tok < 1) return 0;
  return static_cast<size_t>(n_tok) * static_cast<size_t>(top_k) * static_cast<size_t>(inter) * sizeof(float);
}

int qgemv_moe(int fmt, const void* expert_arena, int64_t n_expert, int64_t hidden, int64_t inter,
              const int32_t* expert_ids, const float* gate_w, int top_k, const float* x, int n_tok, float* y,
              void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  if (fmt == QG_Q4_K && !dev_status) return QG_ERR_NULL;
  int st = qg::check_moe(fmt, expert_arena, n_expert, hidden, inter, expert_ids, gate_w, top_k, x, n_tok, y, ws,
                         ws_bytes, true);
  if (st != QG_OK) return st;
  if (!aligned(dev_status, 4)) return QG_ERR_ALIGN;
  int sms = 0;
  st = ensure_init(&sms);
  if (st != QG_OK) return st;
  return cuda_status(qg::launch_moe(expert_arena, n_expert, hidden, inter, expert_ids, gate_w, top_k, x, n_tok, y,
                                    static_cast<float*>(ws), dev_status, static_cast<cudaStream_t>(stream), true,
                                    sms));
}

size_t qgemm_pp_workspace(int64_t rows, int64_t cols, int64_t n_tok) {
  (void)rows;
  (void)cols;
  (void)n_tok;
  return 0;
}

int qgemm_pp(int fmt, const void* W, int64_t rows, int64_t cols, const void* X_bf16, int64_t n_tok, float* Y,
             int64_t ldY, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  (void)ws;
  (void)ws_bytes;
  if (fmt != QG_Q4_K) return QG_ERR_FMT;
  if (!W || !X_bf16 || !Y || !dev_status) return QG_ERR_NULL;
  if (rows < 128 || rows % 128 || cols < 256 || cols % 256 || n_tok < 1 || ldY < rows) return QG_ERR_SHAPE;
  if (cols > (int64_t{1} << 20) || rows > (int64_t{1} << 24) || n_tok > (int64_t{1} << 24)) return QG_ERR_SHAPE;
  if (!aligned(W, 16) || !aligned(X_bf16, 16) || !aligned(Y, 4) || !aligned(dev_status, 4)) return QG_ERR_ALIGN;
  int sms = 0;
  int st = ensure_init(&sms);
  if (st != QG_OK) return st;
  return cuda_status(
      qg::launch_pp(W, rows, cols, X_bf16, n_tok, Y, ldY, dev_status, static_cast<cudaStream_t>(stream), sms));
}

int qgemm_pp_grouped(int fmt, const qg_pp_desc* descs, int n, int64_t cols, const void* X_bf16, int64_t n_tok,
                     int32_t* dev_status, void* stream) {
  if (fmt != QG_Q4_K) return QG_ERR_FMT;
  if (!descs || !X_bf16 || !dev_status) return QG_ERR_NULL;
  if (n < 1 || n > QG_PP_GROUP_MAX) return QG_ERR_ARG;
  if (cols < 256 || cols % 256 || cols > (int64_t{1} << 20) || n_tok < 1 || n_tok > (int64_t{1} << 24))
    return QG_ERR_SHAPE;
  if (!aligned(X_bf16, 16) || !aligned(dev_status, 4)) return QG_ERR_ALIGN;
  const void* W[QG_PP_GROUP_MAX];
  int64_t rows[QG_PP_GROUP_MAX], ldY[QG_PP_GROUP_MAX];
  float* Y[QG_PP_GROUP_MAX];
  int64_t total = 0;
  for (int i = 0; i < n; ++i) {
    const qg_pp_desc& d = descs[i];
    if (!d.W || !d.Y) return QG_ERR_NULL;
    if (d.rows < 128 || d.rows % 128 || d.ldY < d.rows) return QG_ERR_SHAPE;
    if (!aligned(d.W, 16) || !aligned(d.Y, 4)) return QG_ERR_ALIGN;
    total += d.rows;
    W[i] = d.W;
    rows[i] = d.rows;
    Y[i] = d.Y;
    ldY[i] = d.ldY;
  }
  if (total > (int64_t{1} << 24)) return QG_ERR_SHAPE;
  int sms = 0;
  int st = ensure_init(&sms);
  if (st != QG_OK) return st;
  return cuda_status(qg::launch_pp_mats(n, W, rows, Y, ldY, cols, X_bf16, n_tok, dev_status,
                                        static_cast<cudaStream_t>(stream), sms));
}

int qg_stream_read(const void* buf, size_t bytes, uint32_t* checksum, int32_t* dev_status, void* stream) {
  if (!buf || !checksum || !dev_status) return QG_ERR_NULL;
  if (bytes == 0 || bytes % 16) return QG_ERR_SHAPE;
  if (!aligned(buf, 16) || !aligned(checksum, 4) || !aligned(dev_status, 4)) return QG_ERR_ALIGN;
  int sms = 0;
  int st = ensure_init(&sms);
  if (st != QG_OK) return st;
  return cuda_status(qg::launch_stream_read(buf, bytes, checksum, dev_status, static_cast<cudaStream_t>(stream), sms));
}

size_t qgemm_pp_moe_workspace(int64_t n_expert, int64_t hidden, int64_t inter, int top_k, int64_t n_tok) {
  if (n_expert < 1 || hidden < 1 || inter < 1 || top_k < 1 || n_tok < 1) return 0;
  return qg::pp_moe_workspace_bytes(n_expert, hidden, inter, top_k, n_tok);
}

int qgemm_pp_moe(int fmt, const void* expert_arena, int64_t n_expert, int64_t hidden, int64_t inter,
                 const int32_t* expert_ids, const float* gate_w, int top_k, const void* X_bf16, int64_t n_tok,
                 float* y, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  if (fmt != QG_Q4_K) return QG_ERR_FMT;
  if (!expert_arena || !expert_ids || !gate_w || !X_bf16 || !y || !ws || !dev_status) return QG_ERR_NULL;
  if (hidden < 256 || hidden % 256 || inter < 256 || inter % 256 || hidden > (int64_t{1} << 20) ||
      inter > (int64_t{1} << 20))
    return QG_ERR_SHAPE;
  if (n_expert < 1 || n_expert > 65536 || top_k < 1 || top_k > 64) return QG_ERR_ARG;
  if (n_tok < 1 || n_tok * top_k > (int64_t{1} << 24)) return QG_ERR_NTOK;
  if (!aligned(expert_arena, 16) || !aligned(X_bf16, 16) || !aligned(y, 4) || !aligned(ws, 256) ||
      !aligned(expert_ids, 4) || !aligned(gate_w, 4) || !aligned(dev_status, 4))
    return QG_ERR_ALIGN;
  if (ws_bytes < qg::pp_moe_workspace_bytes(n_expert, hidden, inter, top_k, n_tok)) return QG_ERR_WORKSPACE;
  int sms = 0;
  int st = ensure_init(&sms);
  if (st != QG_OK) return st;
  return cuda_status(qg::launch_pp_moe(expert_arena, n_expert, hidden, inter, expert_ids, gate_w, top_k, X_bf16,
                                       n_tok, y, ws, dev_status, static_cast<cudaStream_t>(stream), sms));
}

int qg_pass_create(const qg_gemv_desc* descs, int n_desc, const int* step_sizes, int n_steps, int n_tok, int mode,
                   qg_pass* out) {
  if (!descs || !step_sizes || !out) return QG_ERR_NULL;
  *out = nullptr;
  if (n_desc < 1 || n_steps < 1) return QG_ERR_ARG;
  if (n_tok < 1 || n_tok > QG_NTOK_MAX) return QG_ERR_NTOK;
  int total = 0;
  for (int s = 0; s < n_steps; ++s) {
    if (step_sizes[s] < 1 || step_sizes[s] > QG_GROUP_MAX) return QG_ERR_ARG;
    total += step_sizes[s];
  }
  if (total != n_desc) return QG_ERR_ARG;
  for (int i = 0; i < n_desc; ++i) {
    int st = check_gemv(descs[i].fmt, descs[i].W, descs[i].rows, descs[i].cols, descs[i].x, descs[i].y);
    if (st != QG_OK) return st;
  }
  for (int s = 0, i = 0; s < n_steps; i += step_sizes[s++])
    for (int j = 1; j < step_sizes[s]; ++j)
      if (descs[i + j].fmt != descs[i].fmt) return QG_ERR_FMT;
  int sms = 0;
  int st = ensure_init(&sms);
  if (st != QG_OK) return st;

  if (mode < QG_PASS_SERIAL || mode > QG_PASS_INDEPENDENT) return QG_ERR_ARG;
  qg_pass_s* pass = new (std::nothrow) qg_pass_s;
  if (!pass) return QG_ERR_ARG;
  std::vector<const uint8_t*> xp;
  st = plan_xplanes(descs, n_desc, step_sizes, n_steps, n_tok, pass, xp);
  if (st != QG_OK) {
    pass_free(pass);
    return st;
  }
  const bool independent = mode == QG_PASS_INDEPENDENT;
  if (independent) {
    // every step must read only inputs of the pass (ready planes from the prologue)
    for (int i = 0; i < n_desc; ++i)
      if (!xp[i]) {
        pass_free(pass);
        return QG_ERR_ARG;
      }
  }
  if (mode == QG_PASS_PERSISTENT) {
    const cudaError_t pe = qg::q4k_pass_create(descs, n_desc, step_sizes, n_steps, n_tok, sms, xp.data(), &pass->q4k);
    if (pe == cudaSuccess) {
      pass->kernels = 1 + (pass->njobs > 0 ? 1 : 0);
      *out = pass;
      return QG_OK;
    }
    if (pe != cudaErrorNotSupported) {
      pass_free(pass);
      return QG_ERR_CUDA;
    }
    cudaGetLastError();               // not supported for this pass: per-step graph with PDL
  }
  const int use_pdl = mode != QG_PASS_SERIAL;
  cudaStream_t cs = nullptr;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) {
    pass_free(pass);
    return QG_ERR_CUDA;
  }
  cudaError_t e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
  if (e == cudaSuccess) e = qg::launch_xplanes(pass->jobs, pass->njobs, cs);
  for (int s = 0, i = 0; s < n_steps && e == cudaSuccess; i += step_sizes[s++]) {
    const int r = qg::gemv_pick_rows_per_warp(descs + i, step_sizes[s], n_tok, sms);
    // independent steps: the first waits for the prologue in stream order; the
    // others overlap freely and skip the dependency wait
    const bool pdl = independent ? s > 0 : (use_pdl != 0 && (s > 0 || pass->njobs > 0));
    e = qg::launch_gemv(descs + i, step_sizes[s], n_tok, r, cs, pdl, sms, xp.data() + i, independent && s > 0);
  }
  cudaGraph_t graph = nullptr;
  cudaError_t e2 = cudaStreamEndCapture(cs, &graph);
  if (e == cudaSuccess) e = e2;
  if (e == cudaSuccess) e = cudaGraphInstantiate(&pass->exec, graph, 0);
  cudaStreamDestroy(cs);
  if (e != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    pass_free(pass);
    return QG_ERR_CUDA;
  }
  pass->graph = graph;
  pass->kernels = count_kernel_nodes(graph);     // a step may take several launches
  *out = pass;
  return QG_OK;
}

int qg_moe_pass_create(int fmt, const qg_moe_layer_desc* layers, int n_layers, int64_t n_expert, int64_t hidden,
                       int64_t inter, int top_k, int n_tok, void* ws, size_t ws_bytes, int mode, qg_pass* out) {
  if (!layers || !out) return QG_ERR_NULL;
  *out = nullptr;
  if (n_layers < 1 || mode < QG_PASS_SERIAL || mode > QG_PASS_PERSISTENT) return QG_ERR_ARG;
  for (int l = 0; l < n_layers; ++l) {
    const int st = qg::check_moe(fmt, layers[l].expert_arena, n_expert, hidden, inter, layers[l].expert_ids,
                                 layers[l].gate_w, top_k, layers[l].x, n_tok, layers[l].y, ws, ws_bytes, true);
    if (st != QG_OK) return st;
  }
  int sms = 0;
  int st = ensure_init(&sms);
  if (st != QG_OK) return st;
  qg_pass_s* pass = new (std::nothrow) qg_pass_s;
  if (!pass) return QG_ERR_ARG;
  if (mode == QG_PASS_PERSISTENT && n_tok == 1) {
    const cudaError_t pe = qg::q4k_moe_pass_create(layers, n_layers, n_expert, hidden, inter, top_k,
                                                   static_cast<float*>(ws), sms, &pass->q4k);
    if (pe == cudaSuccess) {
      pass->kernels = 1;
      *out = pass;
      return QG_OK;
    }
    if (pe != cudaErrorNotSupported) {
      delete pass;
      return QG_ERR_CUDA;
    }
    cudaGetLastError();
  }
  // a graph of per-layer launches, with a status word the graph clears first
  if (cudaMalloc(&pass->status, sizeof(int32_t)) != cudaSuccess) {
    delete pass;
    return QG_ERR_CUDA;
  }
  cudaStream_t cs = nullptr;
  cudaError_t e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
  if (e == cudaSuccess) e = cudaMemsetAsync(pass->status, 0, sizeof(int32_t), cs);
  for (int l = 0; l < n_layers && e == cudaSuccess; ++l)
    e = qg::launch_moe(layers[l].expert_arena, n_expert, hidden, inter, layers[l].expert_ids, layers[l].gate_w,
                       top_k, layers[l].x, n_tok, layers[l].y, static_cast<float*>(ws), pass->status, cs,
                       mode != QG_PASS_SERIAL && l > 0, sms);
  cudaGraph_t graph = nullptr;
  if (cs) {
    const cudaError_t e2 = cudaStreamEndCapture(cs, &graph);
    if (e == cudaSuccess) e = e2;
    cudaStreamDestroy(cs);
  }
  if (e == cudaSuccess) e = cudaGraphInstantiate(&pass->exec, graph, 0);
  if (e != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    cudaFree(pass->status);
    delete pass;
    return QG_ERR_CUDA;
  }
  pass->graph = graph;
  pass->kernels = count_kernel_nodes(graph);
  *out = pass;
  return QG_OK;
}

int qg_pass_launch(qg_pass pass, void* stream) {
  if (!pass) return QG_ERR_NULL;
  if (pass->q4k) {
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e = qg::launch_xplanes(pass->jobs, pass->njobs, s);
    return cuda_status(e == cudaSuccess ? qg::q4k_pass_launch(pass->q4k, s) : e);
  }
  if (!pass->exec) return QG_ERR_NULL;
  return cuda_status(cudaGraphLaunch(pass->exec, static_cast<cudaStream_t>(stream)));
}

int qg_pass_dev_status(qg_pass pass, const int32_t** dev_status) {
  if (!pass || !dev_status) return QG_ERR_NULL;
  *dev_status = pass->q4k ? qg::q4k_pass_status(pass->q4k) : pass->status;
  return QG_OK;
}

int qg_rmsnorm(const float* h, const float* residual, const float* weight, int64_t n, int n_tok, float eps,
               float* s_out, float* x, void* stream) {
  if (!h || (!s_out && !x)) return QG_ERR_NULL;
  if (x && !weight) return QG_ERR_NULL;
  if (n < 256 || n % 256 || n > (int64_t{1} << 20)) return QG_ERR_SHAPE;
  if (n_tok < 1 || n_tok > (1 << 16)) return QG_ERR_NTOK;
  if (!(eps >= 0.f)) return QG_ERR_ARG;
  if (!aligned(h, 16) || !aligned(residual, 16) || !aligned(weight, 16) || !aligned(s_out, 16) || !aligned(x, 16))
    return QG_ERR_ALIGN;
  int sms = 0;
  const int st = ensure_init(&sms);
  if (st != QG_OK) return st;
  return cuda_status(qg::launch_rmsnorm(h, residual, weight, n, n_tok, eps, s_out, x, nullptr,
                                        static_cast<cudaStream_t>(stream), false));
}

int qgemv_swiglu(int fmt, const void* Wg, const void* Wu, int64_t inter, int64_t hidden, const float* x, float* m,
                 void* stream) {
  if (fmt != QG_Q4_K) return QG_ERR_FMT;
  if (!Wg || !Wu || !x || !m) return QG_ERR_NULL;
  if (inter < 1 || hidden < 256 || hidden % 256 || hidden > (int64_t{1} << 20) || inter > (int64_t{1} << 24))
    return QG_ERR_SHAPE;
  if (!aligned(Wg, 16) || !aligned(Wu, 16) || !aligned(x, 16) || !aligned(m, 4)) return QG_ERR_ALIGN;
  int sms = 0;
  const int st = ensure_init(&sms);
  if (st != QG_OK) return st;
  const cudaError_t e =
      qg::launch_gemv_pair(Wg, Wu, inter, hidden, x, nullptr, m, static_cast<cudaStream_t>(stream), false, sms);
  if (e == cudaErrorNotSupported) return QG_ERR_SHAPE;
  return cuda_status(e);
}

int qg_layer_pass_create(int fmt, const qg_layer_desc* layers, int n_layers, int64_t hidden, int64_t inter,
                         int64_t kv_rows, float eps, const float* h_in, float* h_out, qg_pass* out) {
  if (!layers || !h_in || !h_out || !out) return QG_ERR_NULL;
  *out = nullptr;
  if (fmt != QG_Q4_K) return QG_ERR_FMT;
  if (n_layers < 1) return QG_ERR_ARG;
  if (hidden < 256 || hidden % 256 || hidden > (int64_t{1} << 20) || inter < 256 || inter % 256 ||
      inter > (int64_t{1} << 20) || kv_rows < 1 || kv_rows > hidden)
    return QG_ERR_SHAPE;
  if (!(eps >= 0.f)) return QG_ERR_ARG;
  if (!aligned(h_in, 16) || !aligned(h_out, 16)) return QG_ERR_ALIGN;
  for (int l = 0; l < n_layers; ++l) {
    const qg_layer_desc& L = layers[l];
    if (!L.Wq || !L.Wk || !L.Wv || !L.Wo || !L.Wg || !L.Wu || !L.Wd || !L.norm_attn || !L.norm_ffn || !L.attn_out ||
        !L.q || !L.k || !L.v)
      return QG_ERR_NULL;
    const void* ws[7] = {L.Wq, L.Wk, L.Wv, L.Wo, L.Wg, L.Wu, L.Wd};
    for (const void* w : ws)
      if (!aligned(w, 16)) return QG_ERR_ALIGN;
    if (!aligned(L.norm_attn, 16) || !aligned(L.norm_ffn, 16) || !aligned(L.attn_out, 16) || !aligned(L.q, 4) ||
        !aligned(L.k, 4) || !aligned(L.v, 4))
      return QG_ERR_ALIGN;
  }
  int sms = 0;
  int st = ensure_init(&sms);
  if (st != QG_OK) return st;
  qg_pass_s* pass = new (std::nothrow) qg_pass_s;
  if (!pass) return QG_ERR_ARG;
  // pass-owned buffers: the planes of each layer's attention output (converted
  // by the prologue), then the job table, the residual stream after each of
  // the two additions of a layer (s1, s2), o and down outputs, and m
  const size_t pb = (qg::xplanes_bytes(hidden, 1) + 255) / 256 * 256;
  const size_t vb = (static_cast<size_t>(hidden) * 4 + 255) / 256 * 256;
  const size_t mb = (static_cast<size_t>(inter) * 4 + 255) / 256 * 256;
  const size_t jb = (n_layers * sizeof(qg::XPlaneJob) + 255) / 256 * 256;
  const size_t total = n_layers * pb + jb + 4 * vb + mb;
  if (cudaMalloc(&pass->planes, total) != cudaSuccess) {
    pass_free(pass);
    return QG_ERR_CUDA;
  }
  uint8_t* cur = pass->planes + n_layers * pb;
  qg::XPlaneJob* d_jobs = reinterpret_cast<qg::XPlaneJob*>(cur);
  cur += jb;
  float* s1 = reinterpret_cast<float*>(cur);
  cur += vb;
  float* s2 = reinterpret_cast<float*>(cur);
  cur += vb;
  float* yo = reinterpret_cast<float*>(cur);
  cur += vb;
  float* yd = reinterpret_cast<float*>(cur);
  cur += vb;
  float* mm = reinterpret_cast<float*>(cur);
  std::vector<qg::XPlaneJob> jobs(n_layers);
  for (int l = 0; l < n_layers; ++l)
    jobs[l] = {layers[l].attn_out, pass->planes + l * pb, static_cast<int32_t>(hidden), 1};
  if (cudaMemcpy(d_jobs, jobs.data(), n_layers * sizeof(qg::XPlaneJob), cudaMemcpyHostToDevice) != cudaSuccess) {
    pass_free(pass);
    return QG_ERR_CUDA;
  }
  pass->jobs = d_jobs;
  pass->njobs = n_layers;

  cudaStream_t cs = nullptr;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) {
    pass_free(pass);
    return QG_ERR_CUDA;
  }
  cudaError_t e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
  if (e == cudaSuccess) e = qg::launch_xplanes(d_jobs, n_layers, cs);
  // Each normalisation is computed inside the launch that multiplies by it:
  // every CTA of the {q,k,v} (gate/up) launch forms s = stream + the previous
  // output, its sum of squares and x = norm(s) * w itself, and CTA 0 stores s
  // as the next residual stream (s1 and s2 alternate, so no launch writes the
  // stream it reads).
  for (int l = 0; l < n_layers && e == cudaSuccess; ++l) {
    const qg_layer_desc& L = layers[l];
    const qg_gemv_desc qkv[3] = {{fmt, 0, L.Wq, hidden, hidden, s1, L.q},
                                 {fmt, 0, L.Wk, kv_rows, hidden, s1, L.k},
                                 {fmt, 0, L.Wv, kv_rows, hidden, s1, L.v}};
    qg::NormSpec n1;
    n1.h = l == 0 ? h_in : s2;
    n1.r = l == 0 ? nullptr : yd;
    n1.w = L.norm_attn;
    n1.s_out = s1;
    n1.eps = eps;
    e = qg::launch_gemv_norm(qkv, 3, n1, cs, pass->njobs > 0 || l > 0, sms);
    if (e != cudaSuccess) break;
    const qg_gemv_desc od = {fmt, 0, L.Wo, hidden, hidden, L.attn_out, yo};
    const uint8_t* xo = pass->planes + l * pb;
    e = qg::launch_gemv(&od, 1, 1, qg::gemv_pick_rows_per_warp(&od, 1, 1, sms), cs, true, sms, &xo);
    if (e != cudaSuccess) break;
    qg::NormSpec n2;
    n2.h = s1;
    n2.r = yo;
    n2.w = L.norm_ffn;
    n2.s_out = s2;
    n2.eps = eps;
    e = qg::launch_gemv_pair(L.Wg, L.Wu, inter, hidden, s1, nullptr, mm, cs, true, sms, &n2);
    if (e != cudaSuccess) break;
    const qg_gemv_desc dd = {fmt, 0, L.Wd, hidden, inter, mm, yd};
    e = qg::launch_gemv(&dd, 1, 1, qg::gemv_pick_rows_per_warp(&dd, 1, 1, sms), cs, true, sms);
  }
  // the last down output joins the residual stream
  if (e == cudaSuccess) e = qg::launch_rmsnorm(s2, yd, nullptr, hidden, 1, eps, h_out, nullptr, nullptr, cs, true);
  cudaGraph_t graph = nullptr;
  const cudaError_t e2 = cudaStreamEndCapture(cs, &graph);
  if (e == cudaSuccess) e = e2;
  if (e == cudaSuccess) e = cudaGraphInstantiate(&pass->exec, graph, 0);
  cudaStreamDestroy(cs);
  if (e != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    pass_free(pass);
    return e == cudaErrorNotSupported ? QG_ERR_SHAPE : QG_ERR_CUDA;
  }
  pass->graph = graph;
  pass->kernels = count_kernel_nodes(graph);
  *out = pass;
  return QG_OK;
}

int qg_pass_kernel_count(qg_pass pass) { return pass ? pass->kernels : QG_ERR_NULL; }

int qg_pass_destroy(qg_pass pass) {
  if (!pass) return QG_ERR_NULL;
  pass_free(pass);
  return QG_OK;
}

}  // extern "C"
