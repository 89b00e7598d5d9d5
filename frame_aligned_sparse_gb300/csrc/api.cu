// C ABI of the library: plan state, device buffers, tensor maps, launches.
// Declarations and contracts: include/fas.h.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
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
  int sms = 0;            // SMs of the plan's device
  int chunks_k = 0;       // prepass key items per frame (set by the frame span: the frame sums' order)
  size_t part_items = 0;  // per-item slots of the prepass's centred and query partials (the largest launch)
  void* arena = nullptr;
  int4* work = nullptr;
  int4* table = nullptr;
  int2* spans = nullptr;
  int4* fvis = nullptr;
  float* ksum_part = nullptr;
  float* mu = nullptr;
  float* fsum = nullptr;
  float* kmax_part = nullptr;
  float* frame_max = nullptr;
  float* gmax_frame = nullptr;
  float* kbarc = nullptr;
  float* mvis = nullptr;
  float* row_bound = nullptr;
  float* gmax_part = nullptr;
  float* stat = nullptr;
  uint8_t* elig = nullptr;
  unsigned int* sync = nullptr;
  // A second set of the prepass's per-launch scratch (centred and query
  // partials, counters), for fas_forward_host's second compute stream.
  float* kmax_part2 = nullptr;
  float* gmax_part2 = nullptr;
  unsigned int* sync2 = nullptr;
  unsigned int* err = nullptr;
  unsigned int* flags = nullptr;  // kFlagBoundRange (attention); cleared by fas_status
  const void* pre_q = nullptr;
  const void* pre_k = nullptr;
  int last_launches = 0;
  int layout = FAS_LAYOUT_HND;  // of q, k, v and out
  fas_plan_info info{};
  // fas_forward_host: library-owned device copies of q, k, v, out, lse, the
  // work list regrouped by head group, and the pipeline's streams/events.
  void* io = nullptr;
  uint16_t *dq = nullptr, *dk = nullptr, *dv = nullptr, *dout = nullptr;
  float* dlse = nullptr;
  CUtensorMap io_tq{}, io_tk{}, io_tv{};
  int4* gwork = nullptr;
  int gwork_hg = -1;                 // heads_per_group argument the regrouped list was built for
  std::vector<int> grp_h0;           // first head of each group (plus H)
  std::vector<int> gwork_off;        // first item of each group (plus the end)
  cudaStream_t st_h2d = nullptr, st_d2h = nullptr;
  cudaStream_t st_comp[2] = {nullptr, nullptr};  // head groups alternate between the two
  std::vector<cudaEvent_t> ev_qk, ev_in, ev_done;  // per group: q and k in, v in, computed
  cudaEvent_t ev_entry = nullptr, ev_exit = nullptr;
  bool exit_recorded = false;
  // fas_forward_ablation: both passes' work lists and fp32 intermediates.
  void* abl = nullptr;
  int4* abl_work[2] = {nullptr, nullptr};
  int abl_items[2] = {0, 0};
  float *abl_o[2] = {nullptr, nullptr}, *abl_lse[2] = {nullptr, nullptr};
  int64_t abl_npad = 0;
};

State g_state;
// Heads per group of fas_forward_host's default schedule in steady state:
// large enough that each group's attention launch fills the GPU many times
// over.  The schedule ramps up to it (1, 2, 4, ... heads) so that the first
// copy-in, which nothing hides, is one head, and each group's copy-in takes
// about as long as the previous group's compute; it ends with a one-head
// group so that the last copy-out is short too.
constexpr int kHostGroupHeads = 4;

// Group boundaries (first head of each group, then H) for heads_per_group
// hg > 0 (uniform groups) or 0 (the ramped default schedule).
std::vector<int> head_groups(int H, int hg) {
  std::vector<int> b(1, 0);
  if (hg > 0) {
    for (int h = hg; h < H; h += hg) b.push_back(h);
  } else if (H > 2) {
    // 1, 2, 4, 4, ... heads over the first H - 1 heads, then one head.
    int h = 0, size = 1;
    while (h < H - 1) {
      h += (H - 1 - h < size) ? H - 1 - h : size;
      b.push_back(h);
      if (size < kHostGroupHeads) size *= 2;
    }
  }
  b.push_back(H);
  return b;
}

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
  State& s = g_state;
  if (s.arena || s.io || s.st_h2d || s.abl) {
    int cur = -1;
    cudaGetDevice(&cur);
    if (s.device >= 0 && cur != s.device) cudaSetDevice(s.device);
    for (cudaStream_t st : {s.st_h2d, s.st_comp[0], s.st_comp[1], s.st_d2h})
      if (st) cudaStreamSynchronize(st);
    for (cudaStream_t st : {s.st_h2d, s.st_comp[0], s.st_comp[1], s.st_d2h})
      if (st) cudaStreamDestroy(st);
    for (auto* evs : {&s.ev_qk, &s.ev_in, &s.ev_done})
      for (cudaEvent_t e : *evs) cudaEventDestroy(e);
    for (cudaEvent_t e : {s.ev_entry, s.ev_exit})
      if (e) cudaEventDestroy(e);
    if (s.gwork) cudaFree(s.gwork);
    if (s.abl) cudaFree(s.abl);
    if (s.io) cudaFree(s.io);
    if (s.arena) cudaFree(s.arena);
    if (cur >= 0 && cur != s.device) cudaSetDevice(cur);
  }
  g_state = State();
}

// Carves the library's device buffers out of one allocation.
int allocate(const HostPlan& p) {
  const size_t H = p.H, Nf = p.Nf, D = p.d, N = (size_t)p.N;
  State& s = g_state;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&s.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FAS_ERR_CUDA;
  // Key items per frame depend on the frame span alone (so a head's frame
  // sums, added in chunk order, are the same in every launch and in every
  // plan, whatever its number of heads); a launch over nh heads holds
  // nh * Nf * chunks(nh) centred and query partials, and the host pipeline
  // launches over head groups of any size up to H.
  s.chunks_k = (p.T + fas::kPrepassRows - 1) / fas::kPrepassRows;
  s.part_items = 0;
  for (int nh = 1; nh <= p.H; ++nh) {
    const size_t items = (size_t)nh * Nf * fas::prepass_chunks(nh, p.N, p.T, s.sms);
    if (items > s.part_items) s.part_items = items;
  }
  const size_t PI = s.part_items;
  struct Part {
    size_t bytes;
    void** dst;
  };
  Part parts[] = {
      {(size_t)p.n_work * sizeof(int4), (void**)&s.work},
      {Nf * sizeof(int4), (void**)&s.table},
      {Nf * sizeof(int2), (void**)&s.spans},
      {Nf * sizeof(int4), (void**)&s.fvis},
      {H * Nf * (size_t)s.chunks_k * D * 4, (void**)&s.ksum_part},
      {H * D * 4, (void**)&s.mu},
      {H * Nf * D * 4, (void**)&s.fsum},
      {PI * 4, (void**)&s.kmax_part},
      {H * Nf * 4, (void**)&s.frame_max},
      {H * Nf * 4, (void**)&s.gmax_frame},
      {H * Nf * D * 4, (void**)&s.kbarc},
      {H * Nf * 4, (void**)&s.mvis},
      {H * N * 4, (void**)&s.row_bound},
      {PI * 4, (void**)&s.gmax_part},
      {H * 4, (void**)&s.stat},
      {H, (void**)&s.elig},
      {fas::prepass_sync_words(p.H, p.Nf) * 4, (void**)&s.sync},
      {PI * 4, (void**)&s.kmax_part2},
      {PI * 4, (void**)&s.gmax_part2},
      {fas::prepass_sync_words(p.H, p.Nf) * 4, (void**)&s.sync2},
      {sizeof(unsigned int), (void**)&s.err},
      {sizeof(unsigned int), (void**)&s.flags},
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
  if (cudaMemcpy(s.spans, p.spans.data(), p.spans.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess)
    return FAS_ERR_CUDA;
  if (cudaMemcpy(s.fvis, p.fvis.data(), p.fvis.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess)
    return FAS_ERR_CUDA;
  return FAS_OK;
}

// bf16 tensor map with 128-byte swizzle; dims innermost first.
int encode(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides_bytes,
           const cuuint32_t* box) {
  return fas::bf16_tensor_map(map, base, rank, dims, strides_bytes, box);
}

// Element strides of q, k, v and out in the current layout: between two
// tokens of one head, and between two heads.
int64_t row_stride() {
  const HostPlan& p = g_state.plan;
  return g_state.layout == FAS_LAYOUT_NHD ? (int64_t)p.H * p.d : (int64_t)p.d;
}
int64_t head_stride() {
  const HostPlan& p = g_state.plan;
  return g_state.layout == FAS_LAYOUT_NHD ? (int64_t)p.d : p.N * (int64_t)p.d;
}

// Prepass arguments for heads [h0, h0 + nh) of q and k.  Every per-head
// statistics buffer is head-major, so it is offset by h0, and so are the
// key partials (sized for every head); the centred and query partials and
// the counters are a launch's own scratch, one of two sets: launches that
// may run at once (fas_forward_host's two compute streams) use different
// sets.
fas::PrepassArgs prepass_args(const void* q, const void* k, int h0, int nh, int set = 0) {
  const HostPlan& p = g_state.plan;
  State& s = g_state;
  const size_t H0 = (size_t)h0, Nf = p.Nf, D = p.d, N = (size_t)p.N;
  fas::PrepassArgs a;
  a.q = static_cast<const uint16_t*>(q) + h0 * head_stride();
  a.k = static_cast<const uint16_t*>(k) + h0 * head_stride();
  a.row_stride = row_stride();
  a.head_stride = head_stride();
  a.spans = s.spans;
  a.fvis = s.fvis;
  a.R0 = p.R0;
  a.r = p.r;
  a.key_sums = nullptr;
  a.ksum_part = s.ksum_part + H0 * Nf * (size_t)s.chunks_k * D;
  a.kmax_part = set ? s.kmax_part2 : s.kmax_part;
  a.gmax_part = set ? s.gmax_part2 : s.gmax_part;
  a.mu = s.mu + H0 * D;
  a.fsum = s.fsum + H0 * Nf * D;
  a.frame_max = s.frame_max + H0 * Nf;
  a.gmax_frame = s.gmax_frame + H0 * Nf;
  a.kbarc = s.kbarc + H0 * Nf * D;
  a.mvis = s.mvis + H0 * Nf;
  a.row_bound = s.row_bound + H0 * N;
  a.stat = s.stat + H0;
  a.elig = s.elig + H0;
  a.sync = set ? s.sync2 : s.sync;
  a.err = s.err;
  a.N = p.N;
  a.T = p.T;
  a.Nf = p.Nf;
  a.H = nh;
  a.d = p.d;
  a.chunks_k = s.chunks_k;
  a.chunks_q = fas::prepass_chunks(nh, p.N, p.T, s.sms);
  a.scale = (float)(1.0 / sqrt((double)p.d));
  a.limit_ns = fas::kWaitLimitNs;
  return a;
}

// Tensor maps of q, k, v (device bf16, current layout).  With uniform frames
// Q is [H][Nf][T][d], so a tile's rows past the frame end read as zeros;
// with ragged frames Q is [H][N][d] and a tile's rows past the frame end
// are the next frame's (computed, never stored).
int encode_qkv(const void* q, const void* k, const void* v, CUtensorMap* tq, CUtensorMap* tk, CUtensorMap* tv) {
  const HostPlan& p = g_state.plan;
  const cuuint64_t D = (cuuint64_t)p.d;
  const cuuint64_t rs = (cuuint64_t)row_stride() * 2, hs = (cuuint64_t)head_stride() * 2;  // bytes
  const cuuint64_t dims[3] = {D, (cuuint64_t)p.N, (cuuint64_t)p.H};
  const cuuint64_t strides[2] = {rs, hs};
  if (!p.ragged) {
    const cuuint64_t qdims[4] = {D, (cuuint64_t)p.T, (cuuint64_t)p.Nf, (cuuint64_t)p.H};
    const cuuint64_t qstrides[3] = {rs, (cuuint64_t)p.T * rs, hs};
    const cuuint32_t box[4] = {64, (cuuint32_t)fas::kQTile, 1, 1};
    if (encode(tq, q, 4, qdims, qstrides, box) != FAS_OK) return FAS_ERR_CUDA;
  } else {
    const cuuint32_t box[3] = {64, (cuuint32_t)fas::kQTile, 1};
    if (encode(tq, q, 3, dims, strides, box) != FAS_OK) return FAS_ERR_CUDA;
  }
  const cuuint32_t box[3] = {64, (cuuint32_t)p.Bk, 1};
  if (encode(tk, k, 3, dims, strides, box) != FAS_OK) return FAS_ERR_CUDA;
  if (encode(tv, v, 3, dims, strides, box) != FAS_OK) return FAS_ERR_CUDA;
  return FAS_OK;
}

// Launches the attention kernel over work items [first, first + count).
cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const int4* work,
                       int count, void* out, float* lse, int mode, cudaStream_t st) {
  const HostPlan& p = g_state.plan;
  State& s = g_state;
  fas::FwdParams fp;
  fp.work = work;
  fp.table = s.table;
  fp.spans = s.spans;
  fp.q_by_frame = p.ragged ? 0 : 1;
  fp.row_bound = s.row_bound;
  fp.elig = s.elig;
  fp.out = static_cast<uint16_t*>(out);
  fp.out_row_stride = row_stride();
  fp.out_head_stride = head_stride();
  fp.lse = lse;
  fp.err = s.err;
  fp.flags = s.flags;
  fp.N = p.N;
  fp.Bk = p.Bk;
  fp.mode = mode;
  fp.scale_log2 = (float)(1.4426950408889634 / sqrt((double)p.d));
  fp.limit_ns = fas::kWaitLimitNs;
  return fas::launch_attention(p.d, tq, tk, tv, fp, count, st);
}

// Copies nh heads of a bf16 q/k/v/out tensor in the current layout; dst and
// src point at the first head's first element.
cudaError_t copy_heads(uint16_t* dst, const uint16_t* src, int nh, cudaMemcpyKind kind, cudaStream_t st) {
  const HostPlan& p = g_state.plan;
  if (g_state.layout == FAS_LAYOUT_NHD) {
    const size_t pitch = (size_t)row_stride() * 2, width = (size_t)nh * p.d * 2;
    return cudaMemcpy2DAsync(dst, pitch, src, pitch, width, (size_t)p.N, kind, st);
  }
  return cudaMemcpyAsync(dst, src, (size_t)nh * (size_t)head_stride() * 2, kind, st);
}

// fas_forward_host resources: device copies of the inputs and outputs, the
// work list regrouped by head group (heaviest items first inside a group),
// four streams (copy in, two for compute, copy out) and the per-group
// events.  Built on first use per plan.
int ensure_host_pipeline(int hg) {
  State& s = g_state;
  const HostPlan& p = s.plan;
  const size_t hnd = (size_t)p.H * (size_t)p.N * (size_t)p.d;
  if (!s.io) {
    const size_t bytes = 4 * hnd * 2 + (size_t)p.H * (size_t)p.N * 4;
    if (cudaMalloc(&s.io, bytes) != cudaSuccess) {
      s.io = nullptr;
      return FAS_ERR_CUDA;
    }
    uint16_t* b = static_cast<uint16_t*>(s.io);
    s.dq = b;
    s.dk = b + hnd;
    s.dv = b + 2 * hnd;
    s.dout = b + 3 * hnd;
    s.dlse = reinterpret_cast<float*>(b + 4 * hnd);
    if (encode_qkv(s.dq, s.dk, s.dv, &s.io_tq, &s.io_tk, &s.io_tv) != FAS_OK) return FAS_ERR_CUDA;
  }
  if (!s.st_h2d) {
    for (cudaStream_t* st : {&s.st_h2d, &s.st_comp[0], &s.st_comp[1], &s.st_d2h})
      if (cudaStreamCreateWithFlags(st, cudaStreamNonBlocking) != cudaSuccess) return FAS_ERR_CUDA;
    for (cudaEvent_t* e : {&s.ev_entry, &s.ev_exit})
      if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return FAS_ERR_CUDA;
  }
  if (s.gwork_hg != hg) s.grp_h0 = head_groups(p.H, hg);
  const int groups = (int)s.grp_h0.size() - 1;
  while ((int)s.ev_in.size() < groups) {
    for (auto* evs : {&s.ev_qk, &s.ev_in, &s.ev_done}) {
      cudaEvent_t e = nullptr;
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return FAS_ERR_CUDA;
      evs->push_back(e);
    }
  }
  if (s.gwork_hg != hg) {
    // The plan's list is heaviest first over all heads; keeping that order
    // inside each group keeps every group's launch heaviest first.
    std::vector<int32_t> grouped;
    grouped.reserve(p.work.size());
    s.gwork_off.assign(1, 0);
    for (int g = 0; g < groups; ++g) {
      for (size_t i = 0; i < p.work.size(); i += 4)
        if (p.work[i] >= s.grp_h0[g] && p.work[i] < s.grp_h0[g + 1])
          grouped.insert(grouped.end(), p.work.begin() + i, p.work.begin() + i + 4);
      s.gwork_off.push_back((int)(grouped.size() / 4));
    }
    if (!s.gwork && cudaMalloc(&s.gwork, p.work.size() * 4) != cudaSuccess) {
      s.gwork = nullptr;
      return FAS_ERR_CUDA;
    }
    if (cudaMemcpy(s.gwork, grouped.data(), grouped.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess)
      return FAS_ERR_CUDA;
    s.gwork_hg = hg;
  }
  return FAS_OK;
}

int describe(const int32_t* spans, int frame_tokens, int n_frames, int ref_frames, int window_radius, int heads,
             int head_dim, int block_k, fas_plan_info* info, int32_t* table, int32_t* work) {
  if (spans && (n_frames < 1 || ref_frames < 0)) return FAS_ERR_ARG;
  HostPlan p;
  const int rc =
      fas::build_plan(spans, frame_tokens, n_frames, ref_frames, window_radius, heads, head_dim, block_k, &p);
  if (rc != FAS_OK) return rc;
  if (info) {
    fill_info(p, info);
    info->host_table = nullptr;  // p is local; the caller's table buffer holds the copy
  }
  if (table) memcpy(table, p.table.data(), p.table.size() * 4);
  if (work) memcpy(work, p.work.data(), p.work.size() * 4);
  return FAS_OK;
}

int make_plan(const int32_t* spans, int frame_tokens, int n_frames, int ref_frames, int window_radius, int heads,
              int head_dim, int block_k, fas_plan_info* info) {
  if (spans && (n_frames < 1 || ref_frames < 0)) return FAS_ERR_ARG;
  HostPlan p;
  int rc = fas::build_plan(spans, frame_tokens, n_frames, ref_frames, window_radius, heads, head_dim, block_k, &p);
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

// The ablation's work lists: per pass, one item per (head, 128-row query
// tile of the padded sequence) with the tile's key range rounded out to
// 128 tokens: the union of its rows' windows (pass 0) or the reference
// frames (pass 1).  Heaviest items first.
void ablation_work(const HostPlan& p, int pass, std::vector<int32_t>* out) {
  const int64_t npad = (p.N + 127) / 128 * 128;
  const int64_t T = p.T;
  std::vector<int32_t> items;
  for (int h = 0; h < p.H; ++h)
    for (int64_t qt = 0; qt * 128 < npad; ++qt) {
      const int64_t r0 = qt * 128, r1 = std::min<int64_t>(r0 + 128, p.N) - 1;  // valid rows of the tile
      int64_t lo, hi;
      if (pass == 1) {
        lo = 0;
        hi = (int64_t)p.R0 * T;
      } else {
        const int fa = (int)(r0 / T), fb = (int)(r1 / T);
        if (fa < p.R0) {
          lo = (int64_t)p.R0 * T;
          hi = p.N;
        } else {
          lo = (int64_t)std::max(p.R0, fa - p.r) * T;
          hi = (int64_t)(std::min(p.Nf - 1, fb + p.r) + 1) * T;
        }
      }
      lo = lo / 128 * 128;
      hi = (hi + 127) / 128 * 128;
      if (hi <= lo) continue;
      items.insert(items.end(), {h, (int32_t)qt, (int32_t)lo, (int32_t)((hi - lo) / 128)});
    }
  const size_t n = items.size() / 4;
  std::vector<size_t> order(n);
  for (size_t i = 0; i < n; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(),
                   [&](size_t a, size_t b) { return items[a * 4 + 3] > items[b * 4 + 3]; });
  out->clear();
  for (size_t i : order) out->insert(out->end(), items.begin() + i * 4, items.begin() + i * 4 + 4);
}

int ensure_ablation() {
  State& s = g_state;
  if (s.abl) return FAS_OK;
  const HostPlan& p = s.plan;
  const int64_t npad = (p.N + 127) / 128 * 128;
  std::vector<int32_t> w[2];
  for (int pass = 0; pass < 2; ++pass) ablation_work(p, pass, &w[pass]);
  const size_t o_bytes = (size_t)p.H * npad * p.d * 4, l_bytes = (size_t)p.H * npad * 4;
  const size_t w_bytes[2] = {(w[0].size() * 4 + 255) / 256 * 256, (w[1].size() * 4 + 255) / 256 * 256};
  if (cudaMalloc(&s.abl, 2 * o_bytes + 2 * l_bytes + w_bytes[0] + w_bytes[1] + 256) != cudaSuccess) {
    s.abl = nullptr;
    return FAS_ERR_CUDA;
  }
  uint8_t* b = static_cast<uint8_t*>(s.abl);
  for (int pass = 0; pass < 2; ++pass) {
    s.abl_o[pass] = reinterpret_cast<float*>(b);
    b += o_bytes;
  }
  for (int pass = 0; pass < 2; ++pass) {
    s.abl_lse[pass] = reinterpret_cast<float*>(b);
    b += l_bytes;
  }
  for (int pass = 0; pass < 2; ++pass) {
    s.abl_work[pass] = reinterpret_cast<int4*>(b);
    s.abl_items[pass] = (int)(w[pass].size() / 4);
    if (!w[pass].empty() &&
        cudaMemcpy(s.abl_work[pass], w[pass].data(), w[pass].size() * 4, cudaMemcpyHostToDevice) != cudaSuccess)
      return FAS_ERR_CUDA;
    b += w_bytes[pass];
  }
  s.abl_npad = npad;
  return FAS_OK;
}

int check_device_plain() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FAS_ERR_CUDA;
  return dev == g_state.device ? FAS_OK : FAS_ERR_STATE;
}

// The device error word the calls that need no plan report into: the
// plan's when there is one, else one allocated on first use per device and
// kept for the process.
int error_word(unsigned int** out) {
  if (g_state.planned && check_device_plain() == FAS_OK) {
    *out = g_state.err;
    return FAS_OK;
  }
  static unsigned int* words[64] = {nullptr};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FAS_ERR_CUDA;
  if (!words[dev]) {
    if (cudaMalloc(&words[dev], sizeof(unsigned int)) != cudaSuccess) return FAS_ERR_CUDA;
    if (cudaMemset(words[dev], 0, sizeof(unsigned int)) != cudaSuccess) return FAS_ERR_CUDA;
  }
  *out = words[dev];
  return FAS_OK;
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
  return describe(nullptr, frame_tokens, n_frames, ref_frames, window_radius, heads, head_dim, block_k, info, table,
                  work);
}

int fas_plan_describe_ragged(const int32_t* frame_tokens, int n_frames, int ref_frames, int window_radius,
                             int heads, int head_dim, int block_k, fas_plan_info* info, int32_t* table,
                             int32_t* work) {
  if (!frame_tokens) return FAS_ERR_ARG;
  return describe(frame_tokens, 0, n_frames, ref_frames, window_radius, heads, head_dim, block_k, info, table, work);
}

int fas_plan_ex(int frame_tokens, int n_frames, int ref_frames, int window_radius, int heads, int head_dim,
                int block_k, fas_plan_info* info) {
  return make_plan(nullptr, frame_tokens, n_frames, ref_frames, window_radius, heads, head_dim, block_k, info);
}

int fas_plan(int frame_tokens, int n_frames, int ref_frames, int window_radius, int heads, int head_dim,
             fas_plan_info* info) {
  return fas_plan_ex(frame_tokens, n_frames, ref_frames, window_radius, heads, head_dim, 0, info);
}

int fas_plan_ragged(const int32_t* frame_tokens, int n_frames, int ref_frames, int window_radius, int heads,
                    int head_dim, int block_k, fas_plan_info* info) {
  if (!frame_tokens) return FAS_ERR_ARG;
  return make_plan(frame_tokens, 0, n_frames, ref_frames, window_radius, heads, head_dim, block_k, info);
}

namespace {

int run_prepass(const void* q, const void* k, const float* key_sums, void* cuda_stream, uint8_t* elig_host) {
  if (!g_state.planned) return FAS_ERR_STATE;
  if (!q || !k) return FAS_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || (key_sums && !aligned16(key_sums))) return FAS_ERR_ALIGN;
  int rc = check_device();
  if (rc != FAS_OK) return rc;
  const HostPlan& p = g_state.plan;
  State& s = g_state;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  fas::PrepassArgs a = prepass_args(q, k, 0, p.H);
  a.key_sums = key_sums;
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

}  // namespace

int fas_prepass(const void* q, const void* k, void* cuda_stream, uint8_t* elig_host) {
  return run_prepass(q, k, nullptr, cuda_stream, elig_host);
}

int fas_prepass_with_key_sums(const void* q, const void* k, const float* key_sums, void* cuda_stream,
                              uint8_t* elig_host) {
  if (!key_sums) return FAS_ERR_ARG;
  return run_prepass(q, k, key_sums, cuda_stream, elig_host);
}

int fas_forward(const void* q, const void* k, const void* v, void* out, float* lse, int mode, void* cuda_stream) {
  if (!g_state.planned) return FAS_ERR_STATE;
  if (!q || !k || !v || !out || !lse) return FAS_ERR_ARG;
  if (mode != FAS_MODE_AUTO && mode != FAS_MODE_ONLINE && mode != FAS_MODE_BOUNDED) return FAS_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse)) return FAS_ERR_ALIGN;
  if (mode != FAS_MODE_ONLINE && (q != g_state.pre_q || k != g_state.pre_k)) return FAS_ERR_STATE;
  int rc = check_device();
  if (rc != FAS_OK) return rc;
  const HostPlan& p = g_state.plan;
  State& s = g_state;
  CUtensorMap tq, tk, tv;
  if (encode_qkv(q, k, v, &tq, &tk, &tv) != FAS_OK) return FAS_ERR_CUDA;
  const cudaError_t e = launch_fwd(tq, tk, tv, s.work, p.n_work, out, lse, mode, static_cast<cudaStream_t>(cuda_stream));
  s.last_launches = e == cudaSuccess ? 1 : 0;
  return e == cudaSuccess ? FAS_OK : FAS_ERR_CUDA;
}

int fas_forward_host(const void* q, const void* k, const void* v, void* out, float* lse, int mode,
                     int heads_per_group, void* cuda_stream) {
  if (!g_state.planned) return FAS_ERR_STATE;
  if (!q || !k || !v || !out || !lse) return FAS_ERR_ARG;
  if (mode != FAS_MODE_AUTO && mode != FAS_MODE_ONLINE && mode != FAS_MODE_BOUNDED) return FAS_ERR_ARG;
  const HostPlan& p = g_state.plan;
  if (heads_per_group < 0 || heads_per_group > p.H) return FAS_ERR_ARG;
  const int hg = heads_per_group;
  int rc = check_device();
  if (rc != FAS_OK) return rc;
  rc = ensure_host_pipeline(hg);
  if (rc != FAS_OK) return rc;
  State& s = g_state;
  cudaStream_t caller = static_cast<cudaStream_t>(cuda_stream);
  const int groups = (int)s.grp_h0.size() - 1;
  int launches = 0;
  // Start after the caller's earlier work, and after the previous call of
  // this function has finished with the library's device copies.
  if (cudaEventRecord(s.ev_entry, caller) != cudaSuccess) return FAS_ERR_CUDA;
  for (cudaStream_t st : {s.st_h2d, s.st_comp[0], s.st_comp[1], s.st_d2h}) {
    if (cudaStreamWaitEvent(st, s.ev_entry, 0) != cudaSuccess) return FAS_ERR_CUDA;
    if (s.exit_recorded && cudaStreamWaitEvent(st, s.ev_exit, 0) != cudaSuccess) return FAS_ERR_CUDA;
  }
  // Work is submitted breadth first: group g+1's copy in, group g's
  // compute, group g-1's copy out.  Streams may share a hardware queue
  // (the driver maps them onto a few connections), and a shared queue
  // holds back whatever sits behind a command that waits.  In this order a
  // waiting command only ever waits for work that is due before what
  // follows it: a copy never sits behind compute it does not need, and
  // compute never behind the copies of later groups.
  auto copy_in = [&](int g) -> bool {
    // The group's heads, one contiguous slice in [H, N, d]; in [N, H, d] a
    // slice of every token's row, copied as a 2D block.
    const int h0 = s.grp_h0[g], nh = s.grp_h0[g + 1] - h0;
    const size_t off = (size_t)h0 * (size_t)head_stride();
    // k and q first: the group's prepass needs only those, so it starts
    // while v is still coming in (this hides part of the first group's
    // copy, which nothing else hides).
    const void* src[3] = {k, q, v};
    uint16_t* dst[3] = {s.dk, s.dq, s.dv};
    for (int t = 0; t < 3; ++t) {
      if (copy_heads(dst[t] + off, static_cast<const uint16_t*>(src[t]) + off, nh, cudaMemcpyHostToDevice,
                     s.st_h2d) != cudaSuccess)
        return false;
      if (t == 1 && cudaEventRecord(s.ev_qk[g], s.st_h2d) != cudaSuccess) return false;
    }
    return cudaEventRecord(s.ev_in[g], s.st_h2d) == cudaSuccess;
  };
  auto compute = [&](int g) -> bool {
    // Prepass and attention for the group's heads, on the group's compute
    // stream with its set of prepass scratch.  Groups alternate between the
    // two, so the next group's launches take the SMs the current group's
    // last CTAs leave idle; they share nothing but the error words.
    const int h0 = s.grp_h0[g], nh = s.grp_h0[g + 1] - h0;
    cudaStream_t st = s.st_comp[g & 1];
    if (cudaStreamWaitEvent(st, s.ev_qk[g], 0) != cudaSuccess) return false;
    const int np = fas::launch_prepass(prepass_args(s.dq, s.dk, h0, nh, g & 1), st);
    if (np < 0) return false;
    launches += np;
    if (cudaStreamWaitEvent(st, s.ev_in[g], 0) != cudaSuccess) return false;
    const int i0 = s.gwork_off[g], ni = s.gwork_off[g + 1] - i0;
    if (launch_fwd(s.io_tq, s.io_tk, s.io_tv, s.gwork + i0, ni, s.dout, s.dlse, mode, st) != cudaSuccess)
      return false;
    ++launches;
    return cudaEventRecord(s.ev_done[g], st) == cudaSuccess;
  };
  auto copy_out = [&](int g) -> bool {
    // The group's rows of out and lse.
    const int h0 = s.grp_h0[g], nh = s.grp_h0[g + 1] - h0;
    const size_t off = (size_t)h0 * (size_t)head_stride();
    return cudaStreamWaitEvent(s.st_d2h, s.ev_done[g], 0) == cudaSuccess &&
           copy_heads(static_cast<uint16_t*>(out) + off, s.dout + off, nh, cudaMemcpyDeviceToHost, s.st_d2h) ==
               cudaSuccess &&
           cudaMemcpyAsync(lse + (size_t)h0 * p.N, s.dlse + (size_t)h0 * p.N, (size_t)nh * p.N * 4,
                           cudaMemcpyDeviceToHost, s.st_d2h) == cudaSuccess;
  };
  if (!copy_in(0)) return FAS_ERR_CUDA;
  for (int g = 0; g < groups; ++g) {
    if (g + 1 < groups && !copy_in(g + 1)) return FAS_ERR_CUDA;
    if (!compute(g)) return FAS_ERR_CUDA;
    if (g >= 1 && !copy_out(g - 1)) return FAS_ERR_CUDA;
  }
  if (!copy_out(groups - 1)) return FAS_ERR_CUDA;
  // The caller's stream continues once every group's results are on the host.
  if (cudaEventRecord(s.ev_exit, s.st_d2h) != cudaSuccess) return FAS_ERR_CUDA;
  s.exit_recorded = true;
  if (cudaStreamWaitEvent(caller, s.ev_exit, 0) != cudaSuccess) return FAS_ERR_CUDA;
  s.pre_q = s.dq;
  s.pre_k = s.dk;
  s.last_launches = launches;
  return FAS_OK;
}

int fas_forward_ablation(const void* q, const void* k, const void* v, void* out, float* lse, void* cuda_stream) {
  if (!g_state.planned) return FAS_ERR_STATE;
  if (!q || !k || !v || !out || !lse) return FAS_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse)) return FAS_ERR_ALIGN;
  const HostPlan& p = g_state.plan;
  if (p.ragged || g_state.layout != FAS_LAYOUT_HND) return FAS_ERR_UNSUPPORTED;
  int rc = check_device();
  if (rc != FAS_OK) return rc;
  rc = ensure_ablation();
  if (rc != FAS_OK) return rc;
  State& s = g_state;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  // Q, K and V as [H][N][d] with 128-row boxes: tiles of the padded sequence
  // read zeros past N.
  const cuuint64_t D = (cuuint64_t)p.d;
  const cuuint64_t dims[3] = {D, (cuuint64_t)p.N, (cuuint64_t)p.H};
  const cuuint64_t strides[2] = {D * 2, (cuuint64_t)p.N * D * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  CUtensorMap tq, tk, tv;
  if (encode(&tq, q, 3, dims, strides, box) != FAS_OK || encode(&tk, k, 3, dims, strides, box) != FAS_OK ||
      encode(&tv, v, 3, dims, strides, box) != FAS_OK)
    return FAS_ERR_CUDA;
  int launches = 0;
  for (int pass = 0; pass < 2; ++pass) {
    if (s.abl_items[pass] == 0) continue;  // no reference frames: no reference pass
    fas::AblationParams a;
    a.f.work = s.abl_work[pass];
    a.f.table = nullptr;
    a.f.spans = nullptr;
    a.f.q_by_frame = 0;
    a.f.row_bound = nullptr;
    a.f.elig = nullptr;
    a.f.out = nullptr;
    a.f.out_row_stride = a.f.out_head_stride = 0;
    a.f.lse = nullptr;
    a.f.err = s.err;
    a.f.flags = s.flags;
    a.f.N = p.N;
    a.f.Bk = 128;
    a.f.mode = FAS_MODE_ONLINE;
    a.f.scale_log2 = (float)(1.4426950408889634 / sqrt((double)p.d));
    a.f.limit_ns = fas::kWaitLimitNs;
    a.o32 = s.abl_o[pass];
    a.lse32 = s.abl_lse[pass];
    a.Npad = s.abl_npad;
    a.T = p.T;
    a.R0 = p.R0;
    a.r = p.r;
    a.Nf = p.Nf;
    a.pass = pass;
    if (fas::launch_ablation_pass(p.d, tq, tk, tv, a, s.abl_items[pass], st) != cudaSuccess) return FAS_ERR_CUDA;
    ++launches;
  }
  const bool two = s.abl_items[1] > 0;
  if (fas::launch_ablation_merge(p.d, s.abl_o[0], s.abl_lse[0], two ? s.abl_o[1] : nullptr,
                                 two ? s.abl_lse[1] : nullptr, static_cast<uint16_t*>(out), lse, p.H, p.N,
                                 s.abl_npad, st) != cudaSuccess)
    return FAS_ERR_CUDA;
  s.last_launches = launches + 1;
  return FAS_OK;
}

int fas_prologue(const void* x, const void* w_folded, const float* cos_tab, const float* sin_tab, int tokens,
                 int width, int heads, int head_dim, float eps, void* q, void* k, void* v, int layout, int groups,
                 int ranks, void* cuda_stream) {
  return fas_prologue_with_key_sums(x, w_folded, cos_tab, sin_tab, tokens, width, heads, head_dim, eps, q, k, v,
                                    layout, groups, ranks, nullptr, cuda_stream);
}

int fas_prologue_with_key_sums(const void* x, const void* w_folded, const float* cos_tab, const float* sin_tab,
                               int tokens, int width, int heads, int head_dim, float eps, void* q, void* k, void* v,
                               int layout, int groups, int ranks, float* key_sums, void* cuda_stream) {
  if (!x || !w_folded || !cos_tab || !sin_tab || !q || !k || !v) return FAS_ERR_ARG;
  if (key_sums && tokens % 16 != 0) return FAS_ERR_ARG;
  if (key_sums && !aligned16(key_sums)) return FAS_ERR_ALIGN;
  if (tokens < 1 || width < 64 || width % 64 != 0 || (head_dim != 64 && head_dim != 128) || heads < 1 ||
      fas::prologue_tile_cols(heads, head_dim) == 0 || !(eps >= 0.f))
    return FAS_ERR_ARG;
  if (layout != FAS_LAYOUT_HND && layout != FAS_LAYOUT_NHD && layout != FAS_LAYOUT_A2A) return FAS_ERR_ARG;
  if (layout == FAS_LAYOUT_A2A && (groups < 1 || ranks < 1 || heads % (groups * ranks) != 0)) return FAS_ERR_ARG;
  if ((int64_t)tokens * width > (int64_t)INT32_MAX * 64) return FAS_ERR_ARG;
  for (const void* ptr : {x, w_folded, (const void*)cos_tab, (const void*)sin_tab, (const void*)q, (const void*)k,
                          (const void*)v})
    if (!aligned16(ptr)) return FAS_ERR_ALIGN;
  unsigned int* err = nullptr;
  const int rc = error_word(&err);
  if (rc != FAS_OK) return rc;
  // x: {C, N} with 64 x 128 boxes; W': {C, 3*H*d} with 64 x TN boxes (both
  // K-major, 128-byte swizzle).  Rows of the last panel past N read zeros.
  const int tn = fas::prologue_tile_cols(heads, head_dim);
  const cuuint64_t xd[2] = {(cuuint64_t)width, (cuuint64_t)tokens};
  const cuuint64_t xs[1] = {(cuuint64_t)width * 2};
  const cuuint32_t xb[2] = {64, 128};
  const cuuint64_t wd[2] = {(cuuint64_t)width, (cuuint64_t)3 * heads * head_dim};
  const cuuint32_t wb[2] = {64, (cuuint32_t)(tn / fas::prologue_cluster())};  // each CTA loads its share
  CUtensorMap tx, tw;
  if (encode(&tx, x, 2, xd, xs, xb) != FAS_OK || encode(&tw, w_folded, 2, wd, xs, wb) != FAS_OK) return FAS_ERR_CUDA;
  fas::PrologueParams pp;
  pp.q = q;
  pp.k = k;
  pp.v = v;
  pp.cos_tab = cos_tab;
  pp.sin_tab = sin_tab;
  pp.tokens = tokens;
  pp.width = width;
  pp.heads = heads;
  pp.head_dim = head_dim;
  pp.layout = layout;
  pp.groups = layout == FAS_LAYOUT_A2A ? groups : 1;
  pp.ranks = layout == FAS_LAYOUT_A2A ? ranks : 1;
  pp.key_sums = key_sums;
  pp.eps = eps;
  pp.err = err;
  pp.limit_ns = fas::kWaitLimitNs;
  const cudaError_t e = fas::launch_prologue(tx, tw, pp, static_cast<cudaStream_t>(cuda_stream));
  g_state.last_launches = e == cudaSuccess ? 1 : 0;
  return e == cudaSuccess ? FAS_OK : FAS_ERR_CUDA;
}

int fas_prologue_fold_weights(const void* w, const float* gamma, void* w_folded, int width, int out_features,
                              void* cuda_stream) {
  if (!w || !gamma || !w_folded || width < 1 || out_features < 1) return FAS_ERR_ARG;
  const cudaError_t e = fas::launch_fold_weights(static_cast<const uint16_t*>(w), gamma,
                                                 static_cast<uint16_t*>(w_folded), out_features, width,
                                                 static_cast<cudaStream_t>(cuda_stream));
  return e == cudaSuccess ? FAS_OK : FAS_ERR_CUDA;
}

int fas_set_layout(int layout) {
  if (layout != FAS_LAYOUT_HND && layout != FAS_LAYOUT_NHD) return FAS_ERR_ARG;
  if (!g_state.planned) return FAS_ERR_STATE;
  if (layout != g_state.layout) {
    g_state.layout = layout;
    // The host pipeline's tensor maps and the last prepass belong to the
    // old layout.
    if (g_state.io && encode_qkv(g_state.dq, g_state.dk, g_state.dv, &g_state.io_tq, &g_state.io_tk,
                                 &g_state.io_tv) != FAS_OK)
      return FAS_ERR_CUDA;
    g_state.pre_q = g_state.pre_k = nullptr;
  }
  return FAS_OK;
}

int fas_free(void) {
  release();
  return FAS_OK;
}

int fas_status(void* cuda_stream) {
  if (!g_state.planned) return FAS_ERR_STATE;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) return FAS_ERR_CUDA;
  unsigned int e = 0, f = 0;
  if (cudaMemcpy(&e, g_state.err, sizeof(e), cudaMemcpyDeviceToHost) != cudaSuccess) return FAS_ERR_CUDA;
  if (cudaMemcpy(&f, g_state.flags, sizeof(f), cudaMemcpyDeviceToHost) != cudaSuccess) return FAS_ERR_CUDA;
  if (e == 0 && f == 0) return FAS_OK;
  if (e && cudaMemset(g_state.err, 0, sizeof(e)) != cudaSuccess) return FAS_ERR_CUDA;
  if (f && cudaMemset(g_state.flags, 0, sizeof(f)) != cudaSuccess) return FAS_ERR_CUDA;
  return e ? FAS_ERR_TIMEOUT : FAS_ERR_BOUND;
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
    case FAS_ERR_BOUND: return "bounded softmax sums out of range (q or k changed since the prepass?)";
    default: return "unknown status";
  }
}

}  // extern "C"
