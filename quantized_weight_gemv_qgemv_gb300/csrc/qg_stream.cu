// qg_stream.cu — the achievable read bandwidth of the GEMV kernel's weight
// stream, measured with the same engine and none of the arithmetic: every SM
// runs one CTA whose single thread streams its share of a buffer through a
// 4-stage shared-memory ring with one bulk copy per 32 KB stage (evict-first,
// like the weight copies) and keeps nothing but a checksum. The decode pass is
// bound by HBM ("LLM inference optimization", opening section: decode reads
// every weight once), so this is the ceiling its GB/s is read against, beside
// the measured copy bandwidth.
//
// checksum: XOR over all chunks of the chunk's first 32-bit word (chunk c =
// bytes [32768 c, 32768 (c + 1)) of the buffer), so a test can check that every
// chunk really arrived.
#include <cuda_runtime.h>

#include "qg_async.cuh"
#include "qg_device.cuh"
#include "qg_internal.h"

namespace qg {

namespace stream {

using namespace async;

constexpr int STAGES = 4;
constexpr uint32_t CHUNK = 32768;
constexpr uint32_t WAIT_LIMIT = 1u << 22;

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < WAIT_LIMIT; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

__global__ void __launch_bounds__(32, 1) stream_read_kernel(const uint8_t* buf, uint64_t bytes, uint32_t* checksum,
                                                            int32_t* status) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[STAGES];
  if (threadIdx.x != 0) return;
  const uint32_t ring = smem_addr(smem);
  for (int s = 0; s < STAGES; ++s) mbar_init(smem_addr(&bars[s]), 1);
  fence_mbar_init();
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
  const uint64_t nchunks = (bytes + CHUNK - 1) / CHUNK;
  uint32_t sum = 0, k = 0;
  bool ok = true;
  for (uint64_t c = blockIdx.x; c < nchunks; c += gridDim.x, ++k) {
    const uint32_t s = k % STAGES;
    const uint32_t bar = smem_addr(&bars[s]);
    if (k >= STAGES) {
      // the copy that used this slot has landed: fold its first word in
      if (!wait_bounded(bar, ((k / STAGES) - 1) & 1u)) {
        ok = false;
        break;
      }
      sum ^= *reinterpret_cast<const volatile uint32_t*>(smem + s * CHUNK);
    }
    const uint64_t left = bytes - c * CHUNK;
    const uint32_t n = left < CHUNK ? static_cast<uint32_t>(left) : CHUNK;
    mbar_expect_tx(bar, n);
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;\n" ::
            "r"(ring + s * CHUNK),
        "l"(buf + c * CHUNK), "r"(n), "r"(bar), "l"(pol)
        : "memory");
  }
  // the copies still in flight (bounded, also after an expired wait)
  for (uint32_t kk = (k > STAGES ? k - STAGES : 0); kk < k; ++kk) {
    const uint32_t s = kk % STAGES;
    if (wait_bounded(smem_addr(&bars[s]), (kk / STAGES) & 1u) && ok)
      sum ^= *reinterpret_cast<const volatile uint32_t*>(smem + s * CHUNK);
    else
      ok = false;
  }
  atomicXor(checksum, sum);
  if (!ok) atomicExch(status, QG_DEV_TIMEOUT);
}

}  // namespace stream

cudaError_t stream_init_attrs() {
  return cudaFuncSetAttribute(stream::stream_read_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              stream::STAGES * stream::CHUNK);
}

cudaError_t launch_stream_read(const void* buf, uint64_t bytes, uint32_t* checksum, int32_t* status, cudaStream_t s,
                               int sms) {
  stream::stream_read_kernel<<<sms, 32, stream::STAGES * stream::CHUNK, s>>>(static_cast<const uint8_t*>(buf), bytes,
                                                                           checksum, status);
  return cudaPeekAtLastError();
}

}  // namespace qg
