// Attention entry point for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc: a host process whose
// device memory is entirely pre-reserved by another framework's caching
// allocator, or embedding code that is only handed fixed buffers and must not
// allocate (a cudaMalloc can also synchronise the device).  For them,
// dg_attention_noalloc runs the split-key attention of the denoising step
// with its scratch (a status word, the per-split partial outputs and their
// max / sum) in a static device array of this file instead of a caller
// workspace.
//
// The array is 16 MiB.  Every GPU that loads the library holds it until the
// process exits.  All calls share it and it keeps the contents of the last
// call.  Only the status word must start at zero: each call clears it on the
// stream before its kernels run; every split writes its whole partial tile
// before the merge reads it, so the partials need no clearing.  Calls that
// overlap on the GPU (different streams, or different host threads on one
// device) race on it.
#include <climits>
#include <mutex>

#include "dg_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;
constexpr size_t kStatusBytes = 256;  // the status word, padded to keep the partials aligned
__device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
unsigned char* g_scratch_ptr[kMaxDevices] = {};

// Device address of the static array on the current device.  The first call
// on a device looks it up with cudaGetSymbolAddress (with that device
// current); later calls reuse it.  The cached address belongs to the device's
// primary context: a caller that destroys that context (cudaDeviceReset) must
// not call these entry points again in the same process.
dg_status scratch_on_current_device(unsigned char** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DG_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) return DG_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<unsigned char*>(p);
  }
  *out = g_scratch_ptr[dev];
  return DG_OK;
}

}  // namespace

extern "C" dg_status dg_attention_noalloc(const void* q, const void* K, const void* V, int32_t cap,
                                          int32_t len, const void* k, const void* v, void* o, int32_t B,
                                          int32_t C, int32_t Hq, int32_t Hkv, int32_t hd, void* stream) {
  if (!q || !K || !V || !k || !v || !o) return DG_ERR_ARG;
  if (B <= 0 || C <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || cap < 0 || len < 0 || len > cap)
    return DG_ERR_ARG;
  if (hd != 32 && hd != 64 && hd != 128) return DG_ERR_SHAPE;
  // the same bounds the denoising step applies to its dims, and the grid's
  // second dimension (one row per canvas and head)
  if (C > 1024 || (int64_t)B * C > (1 << 20) || (int64_t)B * Hq > 65535) return DG_ERR_SHAPE;
  const int64_t T = (int64_t)len + C;
  if (T > INT32_MAX / 2) return DG_ERR_SHAPE;
  dg_dims D{};
  D.B = B;
  D.C = C;
  D.Hq = Hq;
  D.Hkv = Hkv;
  D.hd = hd;
  int ns = 1, kps = 0;
  dg::attn_split(D, (int)T, len, &ns, &kps);
  const size_t rows = (size_t)B * Hq * C;
  const size_t part_bytes = dg::align_up((size_t)ns * rows * hd * 4, 256);
  const size_t need = ns > 1 ? part_bytes + (size_t)ns * rows * 8 : 0;
  if (need > kScratchBytes - kStatusBytes) return DG_ERR_WORKSPACE;  // larger than the static scratch
  unsigned char* scratch = nullptr;
  dg_status s = scratch_on_current_device(&scratch);
  if (s != DG_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* status = reinterpret_cast<int*>(scratch);
  unsigned char* parts = scratch + kStatusBytes;
  if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return DG_ERR_CUDA;
  dg::AttnArgs a{q, K, V, k, v, o, reinterpret_cast<float*>(parts),
                 reinterpret_cast<float*>(parts + part_bytes), B, C, Hq, Hkv, hd, len, cap};
  dg::StopCtl none{nullptr, 0, 0};
  return dg::launch_attention(a, none, status, st) == cudaSuccess ? DG_OK : DG_ERR_CUDA;
}

extern "C" dg_status dg_attention_noalloc_status(int32_t* status, void* stream) {
  if (!status) return DG_ERR_ARG;
  unsigned char* scratch = nullptr;
  dg_status s = scratch_on_current_device(&scratch);
  if (s != DG_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(status, scratch, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return DG_ERR_CUDA;
  return DG_OK;
}
