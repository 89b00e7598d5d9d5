// Prepass: mean-centred key norms, per-row bounds and per-head eligibility.
//
// "HeyGen x Google Cloud: Avatar IV on TPU", section "Unchaining the
// Softmax": a query's largest logit is at most its norm times the largest key
// norm (Cauchy-Schwarz); centring the keys on their mean tightens this and
// changes no output; a small array of precomputed norms lets every row derive
// its bound up front; heads whose bound is too loose use the online path; the
// guarantee is taken per row over the slice of keys that row sees.
//
// For row i of head h in query frame f (s = 1/sqrt(d)):
//   m_i  = s q_i.mu_h + b_i,   b_i = s |q_i| max_{g visible from f} max_{j in g} |k_j - mu_h|
//   G_i  = b_i - s q_i.kbar_c(f)          (kbar_c: mean of k_j - mu_h over visible keys)
//   stat_h = max_i G_i,  eligible <=> stat_h <= 32
// Since the mean of the visible centred logits is at most their maximum,
// G_i bounds the gap between b_i and the true centred row maximum.
//
// One persistent kernel, one CTA of sixteen warps per SM, in which every warp
// works on its own.  A work item is (phase, head, frame, chunk of the frame's
// rows) and belongs to one warp.  Key chunks are fixed by the frame span
// (about 256 rows), which fixes the order the frame's key sums are added in;
// centred and query chunks are sized (32 to 256 rows) for about one item per
// two warps of the grid in each phase.  The warp streams the
// rows through a private ring of shared-memory stages that bulk copies
// (cp.async.bulk, completing on an mbarrier) fill ahead of it, running into
// the next item's rows (input data, ready whatever the next item waits for)
// while it works on this one, so memory parallelism is set by shared
// memory, not registers.  No barrier spans more than a warp, so a warp
// waiting on memory, an atomic or a flag holds up no other.  The queue
// holds every head's items of one phase before the next phase's:
//   keys:     column sums of the chunk's keys;
//   centred:  max |k_j - mu_h|^2 over the chunk (needs mu_h);
//   queries:  m_i and the max of G_i over the chunk (needs kbar_c and the
//             window maximum of its frame: the warp that completes a head's
//             keys writes every frame's kbar_c right after mu_h, the one that
//             completes its centred maxima every frame's window maximum, and
//             the second of the two publishes the head's ready flag).
// An item's inputs come from a phase whose items all left the queue long
// before, so items practically never wait; the price is that K is read
// twice, the second time mostly from DRAM (a lag of a few heads between
// phases kept the second read in L2 but made items wait for their head's
// mean, which cost more).  Every read carries an evict-first L2 policy, so
// the stream leaves L2 to the kernels around it.  Completion is
// counted per frame and per head: the warp that completes a frame reduces
// its chunks' results, and the warp that completes a head's last frame
// reduces the frames.  A consumer item polls its head's ready flag with a
// bounded wait.
//
// A stage (6 KB; two per warp) holds up to 24 rows (d = 128) or 48 rows
// (d = 64): one bulk copy when a head's rows are contiguous (the head-major
// [H, N, d] layout), one per row otherwise (token-major [N, H, d], rows H*d
// elements apart).  Each phase keeps only its own registers (128 at most at
// d = 128), so sixteen warps fit on an SM.  Four lanes share a row, each with a fixed quarter of the columns (and the
// matching quarter of mu_h and kbar_c in registers), so a row's dot
// products and norms need two shuffle steps and the key sums none until
// the item ends; the arithmetic runs on packed fp32 pairs (fma.rn.f32x2,
// add.rn.f32x2), two elements per instruction.  Every reduction runs in a
// fixed order (no floating-point atomics), so results are bit-reproducible
// whichever warp does an item.

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fas.h"
#include "internal.h"
#include "kernels.h"
#include "ptx.cuh"

namespace fas {
namespace {

#ifndef FAS_PREPASS_STAGES
#define FAS_PREPASS_STAGES 2
#endif
#ifndef FAS_PREPASS_WARPS
#define FAS_PREPASS_WARPS 16
#endif
constexpr int kWarps = FAS_PREPASS_WARPS;
constexpr int kThreads = 32 * kWarps;
constexpr int kStages = FAS_PREPASS_STAGES;  // ring stages per warp
#ifndef FAS_PREPASS_STAGE_BYTES
#define FAS_PREPASS_STAGE_BYTES 6144
#endif
constexpr int kStageBytes = FAS_PREPASS_STAGE_BYTES;
constexpr size_t kSmemBytes = (size_t)kWarps * kStages * kStageBytes;

enum Phase { kKeys = 0, kCentred = 1, kQueries = 2 };



// Packed fp32 pairs (sm_100 family): a bf16 pair word as two fp32 lanes, and
// lane-wise add / fused multiply-add.
__device__ __forceinline__ uint64_t bf16_pair(uint32_t w) {
  uint64_t r;
  asm("{\n\t.reg .b32 lo, hi;\n\tshl.b32 lo, %1, 16;\n\tand.b32 hi, %1, 0xffff0000;\n\tmov.b64 %0, {lo, hi};\n\t}"
      : "=l"(r) : "r"(w));
  return r;
}
__device__ __forceinline__ uint64_t pair(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unpair(uint64_t v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return make_float2(lo, hi);
}
__device__ __forceinline__ void fma2(uint64_t& acc, uint64_t a, uint64_t b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}


// Streamed lines (K twice, Q once; none is reused from L2 in time): first to
// leave L2.
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from global to this CTA's shared memory, completing on the mbarrier.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait (one lane) for a ready flag.  Gives up at once when the
// error word is already set, or after limit_ns, recording kErrWaitPrepass.
__device__ bool wait_ready(const unsigned* flag, unsigned* err, uint64_t limit_ns) {
  if (ld_acquire(flag)) return true;
  const uint64_t t0 = ptx::global_timer_ns();
  for (;;) {
    __nanosleep(200);
    if (ld_acquire(flag)) return true;
    if (*reinterpret_cast<volatile unsigned*>(err) != 0u) return false;
    if (ptx::global_timer_ns() - t0 > limit_ns) {
      atomicOr(err, kErrWaitPrepass);
      return false;
    }
  }
}

// Bounded wait (every lane) for a ring stage's copies.  The waiting warp
// sleeps in the try-wait (a suspend-time hint) rather than spinning, so it
// leaves its scheduler's issue slots to the other warps.  With `give_up`,
// it returns false once the error word is set (the caller then drains).
__device__ bool stage_wait(uint32_t bar, uint32_t parity, unsigned* err, uint64_t limit_ns, bool give_up) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::global_timer_ns();
  for (;;) {
    if (ptx::mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (give_up && *reinterpret_cast<volatile unsigned*>(err) != 0u) return false;
    if (ptx::global_timer_ns() - t0 > limit_ns) {
      atomicOr(err, kErrWaitPrepass);
      return false;
    }
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Maximum of p[0 .. n-1] over the warp (order-free: max is exact), at least lo.
__device__ __forceinline__ float warp_max_of(const float* p, int n, float lo, int lane) {
  float m = lo;
  for (int i = lane; i < n; i += 32) m = fmaxf(m, __ldcg(p + i));
  return warp_max(m);
}

// s[e] = sum over i < n of p[i * stride + e], e < CPL, added in index order,
// with eight rows of loads in flight (data written by other warps of this
// launch: read at L2).
template <int CPL>
__device__ __forceinline__ void ordered_sum(const float* p, int n, int64_t stride, float (&s)[CPL]) {
#pragma unroll
  for (int e = 0; e < CPL; ++e) s[e] = 0.f;
  for (int i = 0; i < n; i += 8) {
    float v[8][CPL];
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int e = 0; e < CPL; ++e) v[u][e] = i + u < n ? __ldcg(p + (int64_t)(i + u) * stride + e) : 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int e = 0; e < CPL; ++e) s[e] += v[u][e];  // adding the 0 of a missing row leaves s exact
  }
}

// Visible frames of query frame f: [a0, a1) and [b0, b1).
__device__ __forceinline__ int4 visible(const PrepassArgs& a, int f) {
  if (a.fvis) return a.fvis[f];
  if (f < a.R0) return make_int4(0, a.Nf, 0, 0);
  return make_int4(0, a.R0, max(a.R0, f - a.r), min(a.Nf - 1, f + a.r) + 1);
}

__device__ __forceinline__ int2 span(const PrepassArgs& a, int g) {
  return a.spans ? a.spans[g] : make_int2(g * a.T, a.T);
}

struct Item {
  int phase, h, g, row0, rows;
  int C;           // items per frame of the item's phase
  int64_t hf, pi;  // per-frame and per-item slots
};

// Item `item` of the queue: every head's key items (chunks_k per frame),
// then every head's centred items, then every head's query items
// (chunks_q per frame each), heads and frames in order.  An item's inputs
// come from a phase whose items all left the queue long before it.
__device__ __forceinline__ Item decode(const PrepassArgs& a, int item) {
  const int nk = a.H * a.Nf * a.chunks_k, nq = a.H * a.Nf * a.chunks_q;
  Item it;
  int local;
  if (item < nk) {
    it.phase = kKeys, it.C = a.chunks_k, local = item;
  } else if (item < nk + nq) {
    it.phase = kCentred, it.C = a.chunks_q, local = item - nk;
  } else {
    it.phase = kQueries, it.C = a.chunks_q, local = item - nk - nq;
  }
  const int per = a.Nf * it.C;
  it.h = local / per;
  it.g = (local % per) / it.C;
  const int c = local % it.C;
  // Chunk boundaries at multiples of 8 rows of the frame (frame starts and
  // spans are multiples of 16, stages of 8 rows): row j then always meets
  // the lane of row class j % 8, whose chunk order it is reduced in, so a
  // row's results do not depend on how many items the launch cuts.  Key
  // items that read given 16-row key sums cut at multiples of 16.
  const int64_t cut = it.phase == kKeys && a.key_sums ? ~15LL : ~7LL;
  const int2 sp = span(a, it.g);
  it.row0 = sp.x + (int)((((int64_t)sp.y * c) / it.C) & cut);
  it.rows = sp.x + (int)((((int64_t)sp.y * (c + 1)) / it.C) & cut) - it.row0;
  it.hf = (int64_t)it.h * a.Nf + it.g;
  it.pi = it.hf * it.C + c;
  return it;
}

// Counts the warp's item of a group of n; true (all lanes) in the warp that
// counted the last one.  Every lane's writes of the item are made visible
// before the count, and the last warp's reads come after it.
__device__ __forceinline__ bool warp_finish(unsigned* done, int n, int lane) {
  __threadfence();
  __syncwarp();
  unsigned last = 0;
  if (lane == 0) last = atomicAdd(done, 1u) == (unsigned)(n - 1);
  last = __shfl_sync(0xffffffffu, last, 0);
  if (last) __threadfence();
  return last != 0;
}

// Publishes a ready flag once every lane's writes are visible.
__device__ __forceinline__ void warp_publish(unsigned* flag, int lane) {
  __threadfence();
  __syncwarp();
  if (lane == 0) st_release(flag, 1u);
}

// One of the two results a head's query items wait for is written (the
// window mean centred keys, or the window maxima); the second to arrive
// publishes the ready flag.
__device__ __forceinline__ void win_arrive(unsigned* count, unsigned* flag, int lane) {
  __threadfence();
  __syncwarp();
  unsigned second = 0;
  if (lane == 0) second = atomicAdd(count, 1u) == 1u;
  if (__shfl_sync(0xffffffffu, second, 0)) {
    __threadfence();
    if (lane == 0) st_release(flag, 1u);
  }
}

// v[e] = p[e], e < N (N = 2 or 4), one vector load from L2.
template <int N>
__device__ __forceinline__ void load_cols(const float* p, float (&v)[N]) {
  if constexpr (N == 4) {
    const float4 t = __ldcg(reinterpret_cast<const float4*>(p));
    v[0] = t.x, v[1] = t.y, v[2] = t.z, v[3] = t.w;
  } else {
    const float2 t = __ldcg(reinterpret_cast<const float2*>(p));
    v[0] = t.x, v[1] = t.y;
  }
}

// One warp's ring of shared-memory stages, filled and emptied in order.
template <int D>
struct Ring {
  static constexpr int kRowBytes = 2 * D;
  static constexpr int kRowsPerStage = kStageBytes / kRowBytes;  // 32 (d = 128) or 64 (d = 64)
  uint32_t buf;  // this warp's first stage (shared address)
  uint32_t bar;  // this warp's first stage barrier (shared address)
  unsigned issued, consumed;

  __device__ __forceinline__ uint32_t stage_buf(unsigned n) const { return buf + (n % kStages) * kStageBytes; }
  __device__ __forceinline__ uint32_t stage_bar(unsigned n) const { return bar + (n % kStages) * 8; }

  // Stages of the item's rows (none for key items given 16-row key sums).
  static __device__ __forceinline__ int stages(const PrepassArgs& a, const Item& it) {
    if (it.phase == kKeys && a.key_sums) return 0;
    return (it.rows + kRowsPerStage - 1) / kRowsPerStage;
  }

  // Copies stage t of the item (its rows t*kRowsPerStage ..) into the next
  // slot.  Warp-wide.
  __device__ __forceinline__ void issue(const PrepassArgs& a, const Item& it, int t, int lane, uint64_t pol) {
    const int r0 = t * kRowsPerStage;
    const int n = min(kRowsPerStage, it.rows - r0);
    const uint16_t* src = static_cast<const uint16_t*>(it.phase == kQueries ? a.q : a.k) +
                          (int64_t)it.h * a.head_stride + (int64_t)(it.row0 + r0) * a.row_stride;
    const uint32_t dst = stage_buf(issued), b = stage_bar(issued);
    if (lane == 0) ptx::mbar_arrive_expect_tx(b, (uint32_t)(n * kRowBytes));
    if (a.row_stride == D) {
      if (lane == 0) bulk_g2s(dst, src, (uint32_t)(n * kRowBytes), b, pol);
    } else {
      __syncwarp();  // the expected byte count is set before any copy lands
      for (int i = lane; i < n; i += 32)
        bulk_g2s(dst + (uint32_t)(i * kRowBytes), src + (int64_t)i * a.row_stride, kRowBytes, b, pol);
    }
    ++issued;
  }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1) prepass_kernel(const PrepassArgs a) {
  using R = Ring<D>;
  constexpr int VPR = D / 8;                   // 16-byte chunks per row
  constexpr int NCH = D / 32;                  // chunks per lane: four lanes share a row
  constexpr int STEPS = R::kRowsPerStage / 8;  // eight rows per warp-wide read
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t bars[kWarps][kStages];
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  // Lane (rl, sg) reads rows rl, rl + 8, ... of a stage and, of each, the
  // chunks sg + 4 (j ^ x), j < NCH, x = rl & 1: its columns are fixed, and
  // the eight lanes of each quarter-warp read eight different bank groups.
  const int sg = lane & 3, rl = lane >> 2, xr = rl & 1;
  int chunk[NCH];
#pragma unroll
  for (int j = 0; j < NCH; ++j) chunk[j] = sg + 4 * (j ^ xr);
  const int H = a.H, Nf = a.Nf;
  const int total = H * Nf * (a.chunks_k + 2 * a.chunks_q);
  unsigned* const queue = a.sync;
  unsigned* const keys_frame_done = a.sync + 1;  // [H, Nf] items done per frame and phase
  unsigned* const cent_frame_done = keys_frame_done + H * Nf;
  unsigned* const qry_frame_done = cent_frame_done + H * Nf;
  unsigned* const keys_done = qry_frame_done + H * Nf;  // [H] frames done per head and phase
  unsigned* const cent_done = keys_done + H;
  unsigned* const qry_done = cent_done + H;
  unsigned* const mu_ready = qry_done + H;
  unsigned* const win_ready = mu_ready + H;
  unsigned* const win_count = win_ready + H;  // [H] of the two window results written
  const uint64_t drop = evict_first_policy();  // every read is the line's last use in this kernel
  const uint32_t smem_base = ptx::smem_addr(smem);

  R ring;
  ring.buf = smem_base + (uint32_t)(warp * kStages * kStageBytes);
  ring.bar = ptx::smem_addr(&bars[warp][0]);
  ring.issued = ring.consumed = 0;
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) ptx::mbar_init(ring.bar + s * 8, 1);
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  __syncwarp();

  // Item A is worked on; item B is the next one, whose index is fetched
  // while A runs and whose rows enter the ring once A's are all issued.
  unsigned raw = 0;
  if (lane == 0) raw = atomicAdd(queue, 1u);
  const int ia = (int)__shfl_sync(0xffffffffu, raw, 0);
  if (ia < total) {
    Item A = decode(a, ia), B = A;
    int nA = R::stages(a, A), tA = 0, nB = 0, tB = 0;
    unsigned rawB = 0;
    if (lane == 0) rawB = atomicAdd(queue, 1u);
    int ib = -1;        // B's index, once looked at
    bool hasB = false;  // B decoded
    // Keeps every stage of the ring in flight: A's remaining rows, then B's.
    auto top_up = [&]() {
      while (ring.issued - ring.consumed < (unsigned)kStages) {
        if (tA < nA) {
          ring.issue(a, A, tA++, lane, drop);
          continue;
        }
        if (ib < 0) ib = (int)__shfl_sync(0xffffffffu, rawB, 0);
        if (ib >= total) break;
        if (!hasB) {
          B = decode(a, ib);
          nB = R::stages(a, B);
          tB = 0;
          hasB = true;
        }
        if (tB >= nB) break;
        ring.issue(a, B, tB++, lane, drop);
      }
    };

    for (;;) {
      top_up();
      if (A.phase != kKeys) {
        unsigned got = 1;
        if (lane == 0) got = wait_ready(A.phase == kCentred ? &mu_ready[A.h] : &win_ready[A.h], a.err, a.limit_ns);
        if (!__shfl_sync(0xffffffffu, got, 0)) break;  // the error word is set; drain below
      }
      const int64_t hbase = (int64_t)A.h * D;
      // Streams the item's stages, body(sb, r0, n) on each (sb: the stage's
      // rows, r0: its first row in the item, n: its rows); false when a
      // wait gave up.  Each phase below keeps its own registers.
      auto stream_item = [&](auto&& body) -> bool {
        for (int t = 0; t < nA; ++t) {
          top_up();
          const unsigned n_st = ring.consumed;
          if (!stage_wait(ring.stage_bar(n_st), (n_st / kStages) & 1u, a.err, a.limit_ns, true)) return false;
          const uint4* sb = reinterpret_cast<const uint4*>(smem + (ring.stage_buf(n_st) - smem_base));
          const int r0 = t * R::kRowsPerStage;
          body(sb, r0, min(R::kRowsPerStage, A.rows - r0));
          // The stage's shared-memory reads (generic proxy) are ordered
          // before the bulk copy that refills it (async proxy).
          ptx::fence_proxy_async_smem();
          __syncwarp();
          ++ring.consumed;
        }
        return true;
      };
      // This lane's quarter of a head-length vector, as packed pairs.
      auto load_pairs = [&](const float* v, uint64_t (&out)[NCH][4], float sign) {
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          const float4* vp = reinterpret_cast<const float4*>(v + chunk[j] * 8);
          const float4 lo = __ldcg(vp), hi = __ldcg(vp + 1);
          out[j][0] = pair(sign * lo.x, sign * lo.y);
          out[j][1] = pair(sign * lo.z, sign * lo.w);
          out[j][2] = pair(sign * hi.x, sign * hi.y);
          out[j][3] = pair(sign * hi.z, sign * hi.w);
        }
      };

      if (A.phase == kKeys && a.key_sums) {
        // Column sums of the chunk's keys from its 16-row group sums, added
        // in group order; lane l owns columns CPL l .. CPL l + CPL - 1.
        constexpr int CPL = D / 32;
        constexpr int U = 8;  // groups loaded ahead of their additions
        const float* src = a.key_sums + ((int64_t)A.h * (a.N / 16) + A.row0 / 16) * D + lane * CPL;
        const int ng = A.rows / 16;
        float s[CPL];
#pragma unroll
        for (int e = 0; e < CPL; ++e) s[e] = 0.f;
        for (int g0 = 0; g0 < ng; g0 += U) {
          float v[U][CPL];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            if (g0 + u < ng) {
              load_cols<CPL>(src + (int64_t)(g0 + u) * D, v[u]);
            } else {
#pragma unroll
              for (int e = 0; e < CPL; ++e) v[u][e] = 0.f;
            }
          }
#pragma unroll
          for (int u = 0; u < U; ++u)
            if (g0 + u < ng) {
#pragma unroll
              for (int e = 0; e < CPL; ++e) s[e] += v[u][e];
            }
        }
#pragma unroll
        for (int e = 0; e < CPL; ++e) a.ksum_part[A.pi * D + lane * CPL + e] = s[e];
      } else if (A.phase == kKeys) {
        // Column sums of the chunk's keys.
        uint64_t acc2[NCH][4];
#pragma unroll
        for (int j = 0; j < NCH; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc2[j][e] = 0;
        if (!stream_item([&](const uint4* sb, int, int n) {
#pragma unroll
              for (int q = 0; q < STEPS; ++q) {
                const int row = q * 8 + rl;
                if (row < n) {
#pragma unroll
                  for (int j = 0; j < NCH; ++j) {
                    const uint4 x = sb[row * VPR + chunk[j]];
                    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc2[j][e] = add2(acc2[j][e], bf16_pair(w[e]));
                  }
                }
              }
            }))
          break;
        float acc[NCH][8];
#pragma unroll
        for (int j = 0; j < NCH; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 t2 = unpair(acc2[j][e]);
            acc[j][2 * e] = t2.x;
            acc[j][2 * e + 1] = t2.y;
          }
        // Every lane's sums in chunk order sg + 4j (the odd rows' lanes read
        // the chunk pairs swapped), then the eight row lanes of each column
        // group added in a fixed tree.
#pragma unroll
        for (int j = 0; j < NCH; j += 2)
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float u0 = acc[j][e], u1 = acc[j + 1][e];
            acc[j][e] = xr ? u1 : u0;
            acc[j + 1][e] = xr ? u0 : u1;
          }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1)
#pragma unroll
          for (int j = 0; j < NCH; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[j][e] += __shfl_xor_sync(0xffffffffu, acc[j][e], o);
        if (rl == 0) {
#pragma unroll
          for (int j = 0; j < NCH; ++j) {
            float4* dst = reinterpret_cast<float4*>(a.ksum_part + A.pi * D + (sg + 4 * j) * 8);
            dst[0] = make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
            dst[1] = make_float4(acc[j][4], acc[j][5], acc[j][6], acc[j][7]);
          }
        }
      }
      if (A.phase == kKeys) {
        if (warp_finish(&keys_frame_done[A.hf], A.C, lane)) {
          // The frame's key sums, in chunk order.
          constexpr int CPL = D / 32;
          float s[CPL];
          ordered_sum<CPL>(a.ksum_part + A.hf * A.C * D + lane * CPL, A.C, D, s);
#pragma unroll
          for (int e = 0; e < CPL; ++e) a.fsum[A.hf * D + lane * CPL + e] = s[e];
          if (warp_finish(&keys_done[A.h], Nf, lane)) {
            // The head's mean key, from the frame sums in frame order.
            ordered_sum<CPL>(a.fsum + (int64_t)A.h * Nf * D + lane * CPL, Nf, D, s);
            float mu_l[CPL];
#pragma unroll
            for (int e = 0; e < CPL; ++e) {
              mu_l[e] = s[e] / (float)a.N;
              a.mu[hbase + lane * CPL + e] = mu_l[e];
            }
            warp_publish(&mu_ready[A.h], lane);
            // Per query frame: the mean centred key over the keys it sees
            // (frame sums added in frame order).
            for (int f = 0; f < Nf; ++f) {
              const int4 vis = visible(a, f);
              float kc[CPL];
#pragma unroll
              for (int e = 0; e < CPL; ++e) kc[e] = 0.f;
              int64_t cnt = 0;
#pragma unroll
              for (int part = 0; part < 2; ++part) {
                const int g0 = part == 0 ? vis.x : vis.z, g1 = part == 0 ? vis.y : vis.w;
                for (int gg = g0; gg < g1; ++gg) {
                  float fv[CPL];
                  load_cols<CPL>(a.fsum + ((int64_t)A.h * Nf + gg) * D + lane * CPL, fv);
#pragma unroll
                  for (int e = 0; e < CPL; ++e) kc[e] += fv[e];
                  cnt += span(a, gg).y;
                }
              }
#pragma unroll
              for (int e = 0; e < CPL; ++e)
                a.kbarc[((int64_t)A.h * Nf + f) * D + lane * CPL + e] = kc[e] / (float)cnt - mu_l[e];
            }
            win_arrive(&win_count[A.h], &win_ready[A.h], lane);
          }
        }
      } else if (A.phase == kCentred) {
        // Largest |k_j - mu_h|^2 over the chunk.
        uint64_t negm2[NCH][4];
        load_pairs(a.mu + hbase, negm2, -1.f);
        float best = 0.f;
        if (!stream_item([&](const uint4* sb, int, int n) {
#pragma unroll
              for (int q = 0; q < STEPS; ++q) {
                const int row = q * 8 + rl;
                const bool valid = row < n;
                uint64_t s2 = 0;
#pragma unroll
                for (int j = 0; j < NCH; ++j) {
                  const uint4 x = valid ? sb[row * VPR + chunk[j]] : make_uint4(0, 0, 0, 0);
                  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    const uint64_t dlt = add2(bf16_pair(w[e]), negm2[j][e]);
                    fma2(s2, dlt, dlt);
                  }
                }
                const float2 sp2 = unpair(s2);
                float s = sp2.x + sp2.y;
                s += __shfl_xor_sync(0xffffffffu, s, 1);
                s += __shfl_xor_sync(0xffffffffu, s, 2);
                if (valid) best = fmaxf(best, s);
              }
            }))
          break;
        best = warp_max(best);
        if (lane == 0) a.kmax_part[A.pi] = best;
        if (warp_finish(&cent_frame_done[A.hf], A.C, lane)) {
          const float mx = warp_max_of(a.kmax_part + A.hf * A.C, A.C, 0.f, lane);
          if (lane == 0) a.frame_max[A.hf] = sqrtf(mx);
          if (warp_finish(&cent_done[A.h], Nf, lane)) {
            // Per query frame: the largest maximum of the frames it sees.
            for (int f = lane; f < Nf; f += 32) {
              const int4 vis = visible(a, f);
              float mx2 = 0.f;
              for (int gg = vis.x; gg < vis.y; ++gg) mx2 = fmaxf(mx2, __ldcg(&a.frame_max[(int64_t)A.h * Nf + gg]));
              for (int gg = vis.z; gg < vis.w; ++gg) mx2 = fmaxf(mx2, __ldcg(&a.frame_max[(int64_t)A.h * Nf + gg]));
              a.mvis[(int64_t)A.h * Nf + f] = mx2;
            }
            win_arrive(&win_count[A.h], &win_ready[A.h], lane);
          }
        }
      } else {
        // Row bounds and the chunk's largest slack, with the frame's window
        // statistics (written once per frame when the head's keys and
        // centred maxima completed).
        uint64_t m2[NCH][4], kb2[NCH][4];
        load_pairs(a.mu + hbase, m2, 1.f);
        load_pairs(a.kbarc + A.hf * D, kb2, 1.f);
        const float Mv = __ldcg(&a.mvis[A.hf]);
        float* const out = a.row_bound + (int64_t)A.h * a.N + A.row0;
        float gmax = -INFINITY;
        if (!stream_item([&](const uint4* sb, int r0, int n) {
#pragma unroll
              for (int q = 0; q < STEPS; ++q) {
                const int row = q * 8 + rl;
                const bool valid = row < n;
                uint64_t qq2 = 0, qm2 = 0, qk2 = 0;
#pragma unroll
                for (int j = 0; j < NCH; ++j) {
                  const uint4 x = valid ? sb[row * VPR + chunk[j]] : make_uint4(0, 0, 0, 0);
                  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    const uint64_t f2 = bf16_pair(w[e]);
                    fma2(qq2, f2, f2);
                    fma2(qm2, f2, m2[j][e]);
                    fma2(qk2, f2, kb2[j][e]);
                  }
                }
                const float2 a2 = unpair(qq2), b2 = unpair(qm2), c2 = unpair(qk2);
                float qq = a2.x + a2.y, qm = b2.x + b2.y, qk = c2.x + c2.y;
                qq += __shfl_xor_sync(0xffffffffu, qq, 1);
                qm += __shfl_xor_sync(0xffffffffu, qm, 1);
                qk += __shfl_xor_sync(0xffffffffu, qk, 1);
                qq += __shfl_xor_sync(0xffffffffu, qq, 2);
                qm += __shfl_xor_sync(0xffffffffu, qm, 2);
                qk += __shfl_xor_sync(0xffffffffu, qk, 2);
                if (valid && sg == 0) {
                  const float b = a.scale * sqrtf(qq) * Mv;
                  out[r0 + row] = fmaf(a.scale, qm, b);
                  gmax = fmaxf(gmax, b - a.scale * qk);
                }
              }
            }))
          break;
        gmax = warp_max(gmax);
        if (lane == 0) a.gmax_part[A.pi] = gmax;
        if (warp_finish(&qry_frame_done[A.hf], A.C, lane)) {
          const float fm = warp_max_of(a.gmax_part + A.hf * A.C, A.C, -INFINITY, lane);
          if (lane == 0) a.gmax_frame[A.hf] = fm;
          if (warp_finish(&qry_done[A.h], Nf, lane)) {
            // Largest slack of the head (max is exact in any order).
            const float mx = warp_max_of(a.gmax_frame + (int64_t)A.h * Nf, Nf, -INFINITY, lane);
            if (lane == 0) {
              a.stat[A.h] = mx;
              a.elig[A.h] = mx <= FAS_ELIG_SLACK_NATS ? 1 : 0;
            }
          }
        }
      }

      // Next item: B (whose first stages may already be in the ring).
      if (ib < 0) ib = (int)__shfl_sync(0xffffffffu, rawB, 0);
      if (ib >= total) break;
      if (!hasB) {
        B = decode(a, ib);
        nB = R::stages(a, B);
        tB = 0;
      }
      A = B;
      nA = nB;
      tA = tB;
      hasB = false;
      ib = -1;
      if (lane == 0) rawB = atomicAdd(queue, 1u);
    }
  }
  // Copies still in flight land before the warp leaves (after a failure; on
  // the normal path every issued stage has been consumed).
  while (ring.consumed < ring.issued) {
    stage_wait(ring.stage_bar(ring.consumed), (ring.consumed / kStages) & 1u, a.err, a.limit_ns, false);
    ++ring.consumed;
  }
}

// CTAs of a launch: the kernel's resident CTAs per SM on the current device
// (its shared-memory opt-in is set on every call: the attribute belongs to
// the device's context), at most one item per warp.
template <int D>
int grid_size(int items) {
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaFuncSetAttribute(prepass_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, prepass_kernel<D>, kThreads, kSmemBytes) != cudaSuccess ||
      per_sm < 1)
    return -1;
  const int g = per_sm * sms;
  const int need = (items + kWarps - 1) / kWarps;  // one item per warp at least
  return g < need ? g : need;
}

template <int D>
int launch_d(const PrepassArgs& a, cudaStream_t st) {
  // The counters and flags start at zero; the eligibility bits start at 0
  // (ineligible: the online path is always correct) so that a prepass that
  // gives up on a wait leaves every head on the safe path.
  if (cudaMemsetAsync(a.sync, 0, prepass_sync_words(a.H, a.Nf) * sizeof(unsigned), st) != cudaSuccess) return -1;
  if (cudaMemsetAsync(a.elig, 0, (size_t)a.H, st) != cudaSuccess) return -1;
  const int items = a.H * a.Nf * (a.chunks_k + 2 * a.chunks_q);
  const int grid = grid_size<D>(items);
  if (grid < 1) return -1;
  prepass_kernel<D><<<grid, kThreads, kSmemBytes, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return -1;
  return 1;
}

}  // namespace

size_t prepass_sync_words(int H, int Nf) { return 1 + 3 * (size_t)H * Nf + 6 * (size_t)H; }

int prepass_chunks(int heads, int64_t rows_per_head, int span_max, int sms) {
  // Items per phase: one per two warps.  More, smaller items measured
  // slower (each item's reductions, counters and flag cost the same).
  const int64_t target = (int64_t)(sms > 0 ? sms : 1) * kWarps / 2;
  int64_t r = (int64_t)heads * rows_per_head / target / 8 * 8;
  if (r < kPrepassMinRows) r = kPrepassMinRows;
  if (r > kPrepassRows) r = kPrepassRows;
  return (int)((span_max + r - 1) / r);
}

int launch_prepass(const PrepassArgs& a, cudaStream_t stream) {
  if (a.d == 128) return launch_d<128>(a, stream);
  if (a.d == 64) return launch_d<64>(a, stream);
  return -1;
}

}  // namespace fas
