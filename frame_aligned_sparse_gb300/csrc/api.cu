// C ABI of the library: plan state, device buffers, tensor maps, launches.
// Declarations and contracts: include/fas.h.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <vector>

#include "fas.h"
#include "internal.h"
#include "kernels.h"

namespace {

using fas::HostPlan;

struct State {
  bool planned = false;
  HostPlan plan;
  int device = -1;
  void* arena = nullptr;
  int4* work = nullptr;
  int4* table = nullptr;
  float* partial = nullptr;
  float* mu = nullptr;
  float* fsum = nullptr;
  float* mpart = nullptr;
  float* frame_max = nullptr;
  float* mvis = nullptr;
  float* kbarc = nullptr;
  float* row_bound = nullptr;
  float* gpart = nullptr;
  float* stat = nullptr;
  uint8_t* elig = nullptr;
  unsigned int* err = nullptr;
  const void* pre_q = nullptr;
  const void* pre_k = nullptr;
  int last_launches = 0;
  fas_plan_info info{};
};

State g_state;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

void fill_info(const HostPlan& p, fas_plan_info* info) {
  info->block_k = p.Bk;
  info->q_tile = fas::kQTile;
  info->n_work = p.n_work;
  info->total_frames = p.Nf;
  info->tokens = p.N;
  info->key_blocks = p.key_blocks;
  info->visible_flops = p.visible_flops;
  info->host_table = p.table.data();
}

void release() {
  if (g_state.arena) {
    int cur = -1;
    cudaGetDevice(&cur);
    if (g_state.device >= 0 && cur != g_state.device) cudaSetDevice(g_state.device);
    cudaFree(g_state.arena);
    if (cur >= 0 && cur != g_state.device) cudaSetDevice(cur);
  }
  g_state = State();
}

// Carves the library's device buffers out of one allocation.
int allocate(const HostPlan& p) {
  const size_t H = p.H, Nf = p.Nf, D = p.d, C = p.chunks, N = (size_t)p.N;
  struct Part {
    size_t bytes;
    void** dst;
  };
  State& s = g_state;
  Part parts[] = {
      {(size_t)p.n_work * sizeof(int4), (void**)&s.work},
      {Nf * sizeof(int4), (void**)&s.table},
      {H * Nf * C * D * 4, (void**)&s.partial},
      {H * D * 4, (void**)&s.mu},
      {H * Nf * D * 4, (void**)&s.fsum},
      {H * Nf * C * 4, (void**)&s.mpart},
      {H * Nf * 4, (void**)&s.frame_max},
      {H * Nf * 4, (void**)&s.mvis},
      {H * Nf * D * 4, (void**)&s.kbarc},
      {H * N * 4, (void**)&s.row_bound},
      {H * Nf * C * 4, (void**)&s.gpart},
      {H * 4, (void**)&s.stat},
      {H, (void**)&s.elig},
      {sizeof(unsigned int), (void**)&s.err},
  };
  size_t total = 0;
  for (auto& pt : parts) total += (pt.bytes + 255) & ~(size_t)255;
  void* arena = nullptr;
  if (cudaMalloc(&arena, total) != cudaSuccess) return FAS_ERR_CUDA;
  s.arena = arena;
  size_t off = 0;
  for (auto& pt : parts) {
    *pt.dst = static_cast<uint8_t*>(arena) + off;
    off += (pt.bytes + 255) & ~(size_t)255;
  }
  if (cudaMemset(arena, 0, total) != cudaSuccess) return FAS_ERR_CUDA;
  if (cudaMemcpy(s.work, p.work.data(), p.work.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess)
    return FAS_ERR_CUDA;
  if (cudaMemcpy(s.table, p.table.data(), p.table.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess)
    return FAS_ERR_CUDA;
  return FAS_OK;
}

int ensure_encoder() {
  if (g_encode) return FAS_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return FAS_ERR_CUDA;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return FAS_OK;
}

// bf16 tensor map with 128-byte swizzle; dims innermost first.
int encode(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides_bytes,
           const cuuint32_t* box) {
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides_bytes,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FAS_OK : FAS_ERR_CUDA;
}

int check_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FAS_ERR_CUDA;
  if (g_state.planned && dev != g_state.device) return FAS_ERR_STATE;
  return FAS_OK;
}

}  // namespace

extern "C" {

int fas_plan_describe(int frame_tokens, int n_frames, int ref_frames, int window_radius, int heads, int head_dim,
                      int block_k, fas_plan_info* info, int32_t* table, int32_t* work) {
  HostPlan p;
  const int rc = fas::build_plan(frame_tokens, n_frames, ref_frames, window_radius, heads, head_dim, block_k, &p);
  if (rc != FAS_OK) return rc;
  if (info) {
    fill_info(p, info);
    info->host_table = nullptr;  // p is local; the caller's table buffer holds the copy
  }
  if (table) memcpy(table, p.table.data(), p.table.size() * 4);
  if (work) memcpy(work, p.work.data(), p.work.size() * 4);
  return FAS_OK;
}

int fas_plan_ex(int frame_tokens, int n_frames, int ref_frames, int window_radius, int heads, int head_dim,
                int block_k, fas_plan_info* info) {
  HostPlan p;
  int rc = fas::build_plan(frame_tokens, n_frames, ref_frames, window_radius, heads, head_dim, block_k, &p);
  if (rc != FAS_OK) return rc;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FAS_ERR_CUDA;
  if (g_state.planned && g_state.device == dev && g_state.plan.same_geometry(p)) {
    if (info) *info = g_state.info;
    return FAS_OK;
  }
  release();
  rc = allocate(p);
  if (rc != FAS_OK) {
    release();
    return rc;
  }
  g_state.plan = std::move(p);
  g_state.device = dev;
  g_state.planned = true;
  fill_info(g_state.plan, &g_state.info);
  if (info) *info = g_state.info;
  return FAS_OK;
}

int fas_plan(int frame_tokens, int n_frames, int ref_frames, int window_radius, int heads, int head_dim,
             fas_plan_info* info) {
  return fas_plan_ex(frame_tokens, n_frames, ref_frames, window_radius, heads, head_dim, 0, info);
}

int fas_prepass(const void* q, const void* k, void* cuda_stream, uint8_t* elig_host) {
  if (!g_state.planned) return FAS_ERR_STATE;
  if (!q || !k) return FAS_ERR_ARG;
  if (!aligned16(q) || !aligned16(k)) return FAS_ERR_ALIGN;
  int rc = check_device();
  if (rc != FAS_OK) return rc;
  const HostPlan& p = g_state.plan;
  State& s = g_state;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  fas::PrepassArgs a;
  a.q = q;
  a.k = k;
  a.table = s.table;
  a.partial = s.partial;
  a.mu = s.mu;
  a.fsum = s.fsum;
  a.mpart = s.mpart;
  a.frame_max = s.frame_max;
  a.mvis = s.mvis;
  a.kbarc = s.kbarc;
  a.row_bound = s.row_bound;
  a.gpart = s.gpart;
  a.stat = s.stat;
  a.elig = s.elig;
  a.N = p.N;
  a.T = p.T;
  a.Nf = p.Nf;
  a.H = p.H;
  a.d = p.d;
  a.chunks = p.chunks;
  a.scale = (float)(1.0 / sqrt((double)p.d));
  const int n = fas::launch_prepass(a, st);
  s.last_launches = n > 0 ? n : 0;
  if (n < 0) return FAS_ERR_CUDA;
  s.pre_q = q;
  s.pre_k = k;
  if (elig_host) {
    if (cudaStreamSynchronize(st) != cudaSuccess) return FAS_ERR_CUDA;
    unsigned int e = 0;
    if (cudaMemcpy(&e, s.err, sizeof(e), cudaMemcpyDeviceToHost) != cudaSuccess) return FAS_ERR_CUDA;
    if (e) return FAS_ERR_TIMEOUT;
    if (cudaMemcpy(elig_host, s.elig, (size_t)p.H, cudaMemcpyDeviceToHost) != cudaSuccess) return FAS_ERR_CUDA;
  }
  return FAS_OK;
}

int fas_forward(const void* q, const void* k, const void* v, void* out, float* lse, int mode, void* cuda_stream) {
  if (!g_state.planned) return FAS_ERR_STATE;
  if (!q || !k || !v || !out || !lse) return FAS_ERR_ARG;
  if (mode != FAS_MODE_AUTO && mode != FAS_MODE_ONLINE && mode != FAS_MODE_BOUNDED) return FAS_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse)) return FAS_ERR_ALIGN;
  if (mode != FAS_MODE_ONLINE && (q != g_state.pre_q || k != g_state.pre_k)) return FAS_ERR_STATE;
  int rc = check_device();
  if (rc != FAS_OK) return rc;
  rc = ensure_encoder();
  if (rc != FAS_OK) return rc;
  const HostPlan& p = g_state.plan;
  State& s = g_state;
  const cuuint64_t D = (cuuint64_t)p.d;
  // Q: [H][Nf][T][d] so a tile's rows past the frame end read as zeros.
  CUtensorMap tq, tk, tv;
  {
    const cuuint64_t dims[4] = {D, (cuuint64_t)p.T, (cuuint64_t)p.Nf, (cuuint64_t)p.H};
    const cuuint64_t strides[3] = {D * 2, (cuuint64_t)p.T * D * 2, (cuuint64_t)p.N * D * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)fas::kQTile, 1, 1};
    if (encode(&tq, q, 4, dims, strides, box) != FAS_OK) return FAS_ERR_CUDA;
  }
  {
    const cuuint64_t dims[3] = {D, (cuuint64_t)p.N, (cuuint64_t)p.H};
    const cuuint64_t strides[2] = {D * 2, (cuuint64_t)p.N * D * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)p.Bk, 1};
    if (encode(&tk, k, 3, dims, strides, box) != FAS_OK) return FAS_ERR_CUDA;
    if (encode(&tv, v, 3, dims, strides, box) != FAS_OK) return FAS_ERR_CUDA;
  }
  fas::FwdParams fp;
  fp.work = s.work;
  fp.table = s.table;
  fp.row_bound = s.row_bound;
  fp.elig = s.elig;
  fp.out = static_cast<uint16_t*>(out);
  fp.lse = lse;
  fp.err = s.err;
  fp.N = p.N;
  fp.T = p.T;
  fp.Bk = p.Bk;
  fp.mode = mode;
  fp.scale_log2 = (float)(1.4426950408889634 / sqrt((double)p.d));
  fp.limit_ns = fas::kWaitLimitNs;
  const cudaError_t e = fas::launch_attention(p.d, tq, tk, tv, fp, p.n_work, static_cast<cudaStream_t>(cuda_stream));
  s.last_launches = e == cudaSuccess ? 1 : 0;
  return e == cudaSuccess ? FAS_OK : FAS_ERR_CUDA;
}

int fas_free(void) {
  release();
  return FAS_OK;
}

int fas_status(void* cuda_stream) {
  if (!g_state.planned) return FAS_ERR_STATE;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) return FAS_ERR_CUDA;
  unsigned int e = 0;
  if (cudaMemcpy(&e, g_state.err, sizeof(e), cudaMemcpyDeviceToHost) != cudaSuccess) return FAS_ERR_CUDA;
  if (e == 0) return FAS_OK;
  if (cudaMemset(g_state.err, 0, sizeof(e)) != cudaSuccess) return FAS_ERR_CUDA;
  return FAS_ERR_TIMEOUT;
}

int fas_prepass_readback(float* mu, float* frame_max, float* stat, uint8_t* elig, float* row_bound,
                         void* cuda_stream) {
  if (!g_state.planned) return FAS_ERR_STATE;
  if (!g_state.pre_q) return FAS_ERR_STATE;
  const HostPlan& p = g_state.plan;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) return FAS_ERR_CUDA;
  struct Copy {
    void* dst;
    const void* src;
    size_t bytes;
  } copies[] = {
      {mu, g_state.mu, (size_t)p.H * p.d * 4},
      {frame_max, g_state.frame_max, (size_t)p.H * p.Nf * 4},
      {stat, g_state.stat, (size_t)p.H * 4},
      {elig, g_state.elig, (size_t)p.H},
      {row_bound, g_state.row_bound, (size_t)p.H * (size_t)p.N * 4},
  };
  for (auto& c : copies)
    if (c.dst && cudaMemcpy(c.dst, c.src, c.bytes, cudaMemcpyDeviceToHost) != cudaSuccess) return FAS_ERR_CUDA;
  return FAS_OK;
}

int fas_selftest_wait_timeout(int limit_us, void* cuda_stream) {
  if (limit_us < 1 || limit_us > 1000000) return FAS_ERR_ARG;
  unsigned int* err = nullptr;
  if (cudaMalloc(&err, sizeof(unsigned int)) != cudaSuccess) return FAS_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  int rc = FAS_ERR_CUDA;
  if (cudaMemsetAsync(err, 0, sizeof(unsigned int), st) == cudaSuccess &&
      fas::launch_wait_selftest(err, (uint64_t)limit_us * 1000ull, st) == cudaSuccess &&
      cudaStreamSynchronize(st) == cudaSuccess) {
    unsigned int e = 0;
    if (cudaMemcpy(&e, err, sizeof(e), cudaMemcpyDeviceToHost) == cudaSuccess)
      rc = (e & fas::kErrWaitSelftest) ? FAS_ERR_TIMEOUT : FAS_OK;
  }
  cudaFree(err);
  return rc;
}

int fas_last_launch_count(void) { return g_state.last_launches; }

const char* fas_error_string(int status) {
  switch (status) {
    case FAS_OK: return "ok";
    case FAS_ERR_ARG: return "invalid argument";
    case FAS_ERR_STATE: return "call out of order (no plan or no matching prepass)";
    case FAS_ERR_ALIGN: return "pointer not 16-byte aligned";
    case FAS_ERR_CUDA: return "CUDA error";
    case FAS_ERR_TIMEOUT: return "device-side wait exceeded its bound";
    case FAS_ERR_UNSUPPORTED: return "unsupported";
    case FAS_ERR_SCRATCH: return "problem larger than the fixed scratch of fas_prepass_noalloc";
    default: return "unknown status";
  }
}

}  // extern "C"
