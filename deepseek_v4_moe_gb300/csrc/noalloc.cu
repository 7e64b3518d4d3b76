// Allocation-free variant of the hyper-connection split (HC mix + split + Sinkhorn).
//
// Some callers cannot allocate device memory when they call in: serving or real-time loops that
// forbid allocation after start-up (cudaMalloc may synchronise the whole device and its latency is
// unbounded), and hosts whose memory pool already owns all of the GPU's memory, where cudaMalloc
// fails.  This entry point takes its scratch from a fixed array compiled into the library instead
// of a handle, so it allocates nothing per call.
//
// The array is file-scope device memory: every GPU that loads the library holds its 1 MiB until
// the process exits.  Host code cannot use the array's name as a device address (on the host the
// name is a stand-in object), so the first call on each device looks the address up with
// cudaGetSymbolAddress while that device is current and caches it.  That first call may make the
// CUDA runtime load the module onto the device: make it before any stream capture begins.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "moe_ffn.h"

namespace {

constexpr size_t kScratchBytes = size_t(1) << 20;  // 1 MiB
constexpr int kTicketSlots = 1024;                 // one per group of 4 rows
constexpr int kMaxRows = 4 * kTicketSlots;         // 4096
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

int reject(int code, const char *msg) {
  moe::set_global_error(msg);
  return code;
}

}  // namespace

extern "C" int moe_ffn_hc_split_noalloc(const float *state, const uint16_t *hc_fn, const float *hc_scale,
                                        const float *hc_base, int32_t rows, int32_t hc, int32_t hidden,
                                        int32_t sinkhorn_iters, float rms_eps, float *pre, float *post,
                                        float *comb, void *stream) {
  // an error left by earlier, unrelated work would otherwise surface after this call's work was
  // enqueued; report it first, with nothing enqueued
  if (cudaPeekAtLastError() != cudaSuccess)
    return reject(MOE_FFN_ERR_CUDA, "hc_split_noalloc: a CUDA error is pending from earlier work");
  if (!state || !hc_fn || !hc_scale || !hc_base || !pre || !post || !comb)
    return reject(MOE_FFN_ERR_NULL_PTR, "hc_split_noalloc: a pointer argument is NULL");
  if (hc < 1 || hc > moe::kHcMax || hidden < 128 || hidden % 128 || hidden > 8192 || sinkhorn_iters < 0 ||
      !(rms_eps >= 0.f))
    return reject(MOE_FFN_ERR_BAD_CONFIG, "hc_split_noalloc: hc must be 1..4, hidden a multiple of 128 up to 8192");
  if (rows == 0) return reject(MOE_FFN_ERR_ROWS_ZERO, "hc_split_noalloc: rows must be at least 1");
  if (rows < 0 || rows > kMaxRows)
    return reject(MOE_FFN_ERR_ROWS_RANGE, "hc_split_noalloc: rows exceed the fixed scratch (at most 4096)");
  if ((reinterpret_cast<uintptr_t>(state) | reinterpret_cast<uintptr_t>(hc_fn)) & 15u)
    return reject(MOE_FFN_ERR_ALIGNMENT, "hc_split_noalloc: state and hc_fn must be 16-byte aligned");
  const int hcd = hc * hidden, M = (2 + hc) * hc;
  const size_t partial = (size_t)rows * moe::hc_mix_chunks(rows, hcd) * (M + 1);
  const size_t need = kTicketSlots * sizeof(unsigned) + ((size_t)rows * M + partial) * sizeof(float);
  if (need > kScratchBytes)
    return reject(MOE_FFN_ERR_ROWS_RANGE, "hc_split_noalloc: rows x (hc*hidden) exceed the fixed 1 MiB scratch");

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return reject(MOE_FFN_ERR_CUDA, "hc_split_noalloc: no usable current device");
  void *base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
      void *p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || !p) return reject(MOE_FFN_ERR_CUDA, "hc_split_noalloc: cudaGetSymbolAddress failed");
      g_scratch_ptr[dev] = p;
    }
    base = g_scratch_ptr[dev];
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned *tickets = static_cast<unsigned *>(base);
  float *mixes = reinterpret_cast<float *>(static_cast<unsigned char *>(base) + kTicketSlots * sizeof(unsigned));
  float *part = mixes + (size_t)rows * M;
  // The array keeps the previous call's contents: the tickets must start at zero.
  if (cudaMemsetAsync(tickets, 0, kTicketSlots * sizeof(unsigned), st) != cudaSuccess)
    return reject(MOE_FFN_ERR_CUDA, "hc_split_noalloc: clearing the tickets failed");
  moe::launch_hc_mix_raw(state, hc_fn, hc_scale, hc_base, rows, hc, hidden, sinkhorn_iters, rms_eps, part, tickets,
                         mixes, pre, post, comb, st);
  // a failure here comes after the memset was enqueued (the header says so)
  if (cudaGetLastError() != cudaSuccess) return reject(MOE_FFN_ERR_CUDA, "hc_split_noalloc: launch failed");
  return MOE_FFN_OK;
}
