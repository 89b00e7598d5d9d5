// fas_prepass_noalloc: the prepass with its scratch in a fixed static device
// array, for callers that cannot allocate device memory.  See include/fas.h.

#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "fas.h"
#include "internal.h"
#include "kernels.h"

namespace fas {
namespace {

// The scratch.  In host code `g_noalloc_scratch` is only a stand-in for the
// symbol; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FAS_NOALLOC_SCRATCH_BYTES];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

constexpr int kMaxDevices = 64;
std::mutex g_addr_mutex;
struct Cached {
  CUcontext ctx;
  void* addr;
};
Cached g_addr[kMaxDevices] = {};
CtxGetCurrentFn g_ctx_get = nullptr;

// Device address of the scratch on the current device, looked up once per
// context: after a device reset the primary context (and with it the
// array's address) is new, so the cache is keyed on the current context.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return FAS_ERR_CUDA;
  if (dev >= kMaxDevices) return FAS_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_addr_mutex);
  if (!g_ctx_get) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return FAS_ERR_CUDA;
    g_ctx_get = reinterpret_cast<CtxGetCurrentFn>(fn);
  }
  CUcontext ctx = nullptr;
  if (g_ctx_get(&ctx) != CUDA_SUCCESS) return FAS_ERR_CUDA;
  if (ctx == nullptr || g_addr[dev].addr == nullptr || g_addr[dev].ctx != ctx) {
    // The lookup also makes the device's primary context current when no
    // context is yet.
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return FAS_ERR_CUDA;
    if (g_ctx_get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return FAS_ERR_CUDA;
    g_addr[dev].ctx = ctx;
    g_addr[dev].addr = p;
  }
  *out = g_addr[dev].addr;
  return FAS_OK;
}

size_t round256(size_t b) { return (b + 255) & ~(size_t)255; }

}  // namespace
}  // namespace fas

extern "C" int fas_prepass_noalloc(const void* q, const void* k, int frame_tokens, int n_frames, int ref_frames,
                                   int window_radius, int heads, int head_dim, float* row_bound, float* stat,
                                   uint8_t* elig, void* cuda_stream) {
  using namespace fas;
  const int T = frame_tokens, F = n_frames, R0 = ref_frames, r = window_radius, H = heads, d = head_dim;
  if (T <= 0 || T % 16 != 0 || F < 1 || R0 < 0 || r < 0 || H < 1 || (d != 64 && d != 128)) return FAS_ERR_ARG;
  const int64_t Nf = (int64_t)R0 + F;
  const int64_t N = Nf * T;
  if (N > (int64_t)INT32_MAX || (int64_t)H * N > (int64_t)INT32_MAX) return FAS_ERR_ARG;
  if (!q || !k || !row_bound || !stat || !elig) return FAS_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(q) & 15u) || (reinterpret_cast<uintptr_t>(k) & 15u) ||
      (reinterpret_cast<uintptr_t>(row_bound) & 3u) || (reinterpret_cast<uintptr_t>(stat) & 3u))
    return FAS_ERR_ALIGN;

  // Scratch layout: per-item key sums, per-item centred maxima, per-item
  // slack maxima, mean key, frame sums, frame maxima, frame slack maxima,
  // window mean centred keys, window maxima (fp32), then the counters and
  // flags and the error word.
  const int chunks = (T + kPrepassRowsNoalloc - 1) / kPrepassRowsNoalloc;
  const size_t hs = (size_t)H, nf = (size_t)Nf, cs = (size_t)chunks, ds = (size_t)d;
  const size_t sizes[11] = {hs * nf * cs * ds * 4, hs * nf * cs * 4, hs * nf * cs * 4,
                            hs * ds * 4,           hs * nf * ds * 4, hs * nf * 4,
                            hs * nf * 4,           hs * nf * ds * 4, hs * nf * 4,
                            prepass_sync_words(H, (int)Nf) * 4, 4};
  size_t total = 0;
  for (size_t b : sizes) total += round256(b);
  if (total > (size_t)FAS_NOALLOC_SCRATCH_BYTES) return FAS_ERR_SCRATCH;

  void* base = nullptr;
  const int rc = scratch_address(&base);
  if (rc != FAS_OK) return rc;
  void* part[11];
  size_t off = 0;
  for (int i = 0; i < 11; ++i) {
    part[i] = static_cast<unsigned char*>(base) + off;
    off += round256(sizes[i]);
  }

  PrepassArgs a;
  a.q = q;
  a.k = k;
  a.row_stride = d;                 // head-major [H, N, d]
  a.head_stride = (int64_t)N * d;
  a.spans = nullptr;                // uniform frames of T tokens
  a.fvis = nullptr;                 // visible frames from the frame rule
  a.R0 = R0;
  a.r = r;
  a.key_sums = nullptr;             // the key items read k
  a.ksum_part = static_cast<float*>(part[0]);
  a.kmax_part = static_cast<float*>(part[1]);
  a.gmax_part = static_cast<float*>(part[2]);
  a.mu = static_cast<float*>(part[3]);
  a.fsum = static_cast<float*>(part[4]);
  a.frame_max = static_cast<float*>(part[5]);
  a.gmax_frame = static_cast<float*>(part[6]);
  a.kbarc = static_cast<float*>(part[7]);
  a.mvis = static_cast<float*>(part[8]);
  a.sync = static_cast<unsigned int*>(part[9]);
  a.err = static_cast<unsigned int*>(part[10]);
  a.row_bound = row_bound;
  a.stat = stat;
  a.elig = elig;
  a.N = N;
  a.T = T;
  a.Nf = (int)Nf;
  a.H = H;
  a.d = d;
  a.chunks_k = a.chunks_q = chunks;
  a.scale = (float)(1.0 / sqrt((double)d));
  a.limit_ns = kWaitLimitNs;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  // The error word starts clear on every call: a wait that gave up in an
  // earlier call must not stop this one.
  if (cudaMemsetAsync(a.err, 0, 4, st) != cudaSuccess) return FAS_ERR_CUDA;
  const int n = launch_prepass(a, st);
  return n > 0 ? FAS_OK : FAS_ERR_CUDA;
}
