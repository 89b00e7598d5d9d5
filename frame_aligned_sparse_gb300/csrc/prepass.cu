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
// One persistent kernel, four 256-thread CTAs per SM.  Work items are
// (phase, head, frame, chunk of at most 1024 rows of that frame), taken from
// a queue in the order
//     keys(h)  centred(h-L)  queries(h-2L)    for h = 0, 1, ..., H+2L-1
//   keys:     column sums of the chunk's keys;
//   centred:  max |k_j - mu_h|^2 over the chunk (needs mu_h);
//   queries:  m_i and the max of G_i over the chunk (needs the window
//             statistics of head h).
// With a lag of L = 3 heads between phases, by the time a head's centred
// (or query) items come out of the queue its keys (or centred) items have
// finished, so items rarely wait.  Keys are first read with an evict-last
// L2 policy and read the second time (like the queries) with evict-first,
// so that the L heads' keys between their two reads (about 60 MB at the
// 720p geometry) stay in L2 while the query stream passes through: K is
// read from DRAM once, and the prepass moves one K and one Q from HBM plus
// the small outputs.  An item's fixed costs (taking it from the queue,
// waiting for its head's flag, the reductions and completion counts) are a
// chain of dependent steps; four CTAs per SM run four such chains at once,
// and large items spread each chain's cost over more bytes.
// Completion is counted per frame and per head: the item that completes a
// frame reduces its chunks' results, and the item that completes the last
// frame of a head reduces the frames and publishes the next phase's inputs:
// mu_h after the key sums (the frame sums on the way); Mvis and kbar_c
// after the centred maxima (the frame maxima on the way); stat_h and the
// eligibility bit after the queries.  These reductions sit on the critical
// path of every head, so they keep many loads in flight and add in a fixed
// order.  A consumer item polls the head's ready flag with a bounded wait.
//
// All loads are 16-byte vectors, one row shared by d/8 consecutive lanes
// (each row's d values are contiguous), consecutive rows over the block.
// Rows of one head are row_stride elements apart: d in the head-major
// [H, N, d] layout, H*d in the token-major [N, H, d] layout.  Every reduction
// runs in a fixed order (no floating-point atomics), so results are
// bit-reproducible whichever CTA completes a phase.

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fas.h"
#include "internal.h"
#include "kernels.h"

namespace fas {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;  // 16-byte loads in flight per thread in a sweep

enum Phase { kKeys = 0, kCentred = 1, kQueries = 2 };

#ifndef FAS_PREPASS_LAG
#define FAS_PREPASS_LAG 3
#endif
constexpr int kLag = FAS_PREPASS_LAG;  // heads between consecutive phases in the queue

__device__ __forceinline__ void unpack8(const uint4& x, float (&f)[8]) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    f[2 * e] = __uint_as_float(w[e] << 16);
    f[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
  }
}

// 16-byte load through L2 with an L2 eviction policy, not kept in L1 (each
// row is read once per phase).
__device__ __forceinline__ uint4 ld_policy(const uint4* p, uint64_t policy) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(policy));
  return r;
}

// Keys' first read: keep the line in L2 ahead of other lines (its second
// read comes L heads later).
__device__ __forceinline__ uint64_t evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// A line's last use (keys' second read, queries): first to leave L2.
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait (one thread) for a ready flag.  Gives up at once when the
// error word is already set, or after limit_ns, recording kErrWaitPrepass.
__device__ bool wait_ready(const unsigned* flag, unsigned* err, uint64_t limit_ns) {
  if (ld_acquire(flag)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    __nanosleep(100);
    if (ld_acquire(flag)) return true;
    if (*reinterpret_cast<volatile unsigned*>(err) != 0u) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      atomicOr(err, kErrWaitPrepass);
      return false;
    }
  }
}

// Block-wide max of one float per thread.
__device__ __forceinline__ float block_max(float v, float* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  __syncthreads();  // scratch may still be read from the previous call
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  float r = scratch[0];
  for (int w = 1; w < kThreads / 32; ++w) r = fmaxf(r, scratch[w]);
  return r;
}

constexpr int kCacheFrames = kThreads / 8;  // frames whose sums fit in `red` for the window statistics

struct Shared {
  float red[kThreads / 8][128];  // per-row-slot column sums; later the head's frame sums
  float fmax[kCacheFrames];      // the head's frame maxima
  float scratch[kThreads / 32];
  int item;
  int last;
  int ok;
};

// Sum of p[i * stride] for i = 0 .. n-1, added in index order, with eight
// loads in flight (data written by other CTAs of this launch: read at L2).
__device__ __forceinline__ float ordered_sum(const float* p, int n, int64_t stride) {
  float s = 0.f;
  for (int i = 0; i < n; i += 8) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = i + u < n ? __ldcg(p + (int64_t)(i + u) * stride) : 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) s += v[u];  // adding the 0 of a missing element leaves s exact
  }
  return s;
}

// Maximum of p[i] for i = 0 .. n-1 (order-free: max is exact), at least lo.
__device__ __forceinline__ float batched_max(const float* p, int n, float lo) {
  float m = lo;
  for (int i = 0; i < n; i += 8) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = i + u < n ? __ldcg(p + i + u) : lo;
#pragma unroll
    for (int u = 0; u < 8; ++u) m = fmaxf(m, v[u]);
  }
  return m;
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

// Signals that this CTA finished its item of (phase, head); returns true in
// the CTA that finished the last one (all threads).  Every thread's global
// writes of the item are made visible before the count.
__device__ __forceinline__ bool finish_item(unsigned* done, int n_items, Shared& sh) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned old = atomicAdd(done, 1u);
    sh.last = old == (unsigned)(n_items - 1);
    if (sh.last) __threadfence();
  }
  __syncthreads();
  return sh.last != 0;
}

// Publishes a ready flag once every thread's writes are visible.
__device__ __forceinline__ void publish(unsigned* flag) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) st_release(flag, 1u);
}

template <int D>
__global__ void __launch_bounds__(kThreads, kPrepassCtasPerSm) prepass_kernel(const PrepassArgs a) {
  constexpr int VPR = D / 8;              // 16-byte vectors per row
  constexpr int RPI = kThreads / VPR;     // rows per sweep
  __shared__ Shared sh;
  const int v = threadIdx.x % VPR, rs = threadIdx.x / VPR;
  const int H = a.H, Nf = a.Nf, C = a.chunks;
  const int per = Nf * C;                 // items per (phase, head)
  const int total = 3 * (H + 2 * kLag) * per;
  unsigned* const queue = a.sync;
  unsigned* const keys_frame_done = a.sync + 1;           // [H, Nf] items done per frame
  unsigned* const cent_frame_done = keys_frame_done + H * Nf;
  unsigned* const keys_done = cent_frame_done + H * Nf;   // [H] frames done per head
  unsigned* const cent_done = keys_done + H;
  unsigned* const qry_done = cent_done + H;                // [H] items done per head
  unsigned* const mu_ready = qry_done + H;
  unsigned* const win_ready = mu_ready + H;
  const uint4* const q = static_cast<const uint4*>(a.q);
  const uint4* const k = static_cast<const uint4*>(a.k);
  const int64_t rstride = a.row_stride / 8, hstride = a.head_stride / 8;  // in 16-byte vectors
  const uint64_t last_use = evict_first_policy();
  const uint64_t reused = evict_last_policy();

  for (;;) {
    if (threadIdx.x == 0) {
      sh.item = (*reinterpret_cast<volatile unsigned*>(a.err) != 0u) ? total : (int)atomicAdd(queue, 1u);
      sh.ok = 1;
    }
    __syncthreads();
    const int item = sh.item;
    __syncthreads();
    if (item >= total) break;
    const int seg = item / per, local = item % per;
    const int phase = seg % 3, h = seg / 3 - kLag * phase;
    if (h < 0 || h >= H) continue;  // the queue's first and last steps have fewer phases
    const int g = local / C, c = local % C;
    const int2 sp = span(a, g);
    const int row0 = sp.x + (int)(((int64_t)sp.y * c) / C);
    const int rows = sp.x + (int)(((int64_t)sp.y * (c + 1)) / C) - row0;
    const int64_t pi = ((int64_t)h * Nf + g) * C + c;  // per-item slot

    if (phase != kKeys) {
      if (threadIdx.x == 0) sh.ok = wait_ready(phase == kCentred ? &mu_ready[h] : &win_ready[h], a.err, a.limit_ns);
      __syncthreads();
      const int ok = sh.ok;
      __syncthreads();  // every thread has read the flag before thread 0 may rewrite it
      if (!ok) continue;  // the error word is set; the loop drains the queue
    }

    if (phase == kKeys) {
      // Column sums of the chunk's keys.
      const uint4* base = k + (int64_t)h * hstride + (int64_t)row0 * rstride + v;
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      int r = rs;
      for (; r + 3 * RPI < rows; r += 4 * RPI) {
        uint4 x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) x[u] = ld_policy(base + (int64_t)(r + u * RPI) * rstride, reused);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float f[8];
          unpack8(x[u], f);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[e] += f[e];
        }
      }
      for (; r < rows; r += RPI) {
        float f[8];
        unpack8(ld_policy(base + (int64_t)r * rstride, reused), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += f[e];
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) sh.red[rs][v * 8 + e] = acc[e];
      __syncthreads();
      if (threadIdx.x < D) {
        float s = 0.f;
        for (int t = 0; t < RPI; ++t) s += sh.red[t][threadIdx.x];
        a.ksum_part[pi * D + threadIdx.x] = s;
      }
      if (finish_item(&keys_frame_done[h * Nf + g], C, sh)) {
        // The frame's key sums, in chunk order.
        if (threadIdx.x < D)
          a.fsum[((int64_t)h * Nf + g) * D + threadIdx.x] =
              ordered_sum(&a.ksum_part[((int64_t)h * Nf + g) * C * D + threadIdx.x], C, D);
        if (finish_item(&keys_done[h], Nf, sh)) {
          // The head's mean key, from the frame sums in frame order.
          if (threadIdx.x < D)
            a.mu[(int64_t)h * D + threadIdx.x] =
                ordered_sum(&a.fsum[(int64_t)h * Nf * D + threadIdx.x], Nf, D) / (float)a.N;
          publish(&mu_ready[h]);
        }
      }
    } else if (phase == kCentred) {
      // Largest |k_j - mu_h|^2 over the chunk.
      float m[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) m[e] = __ldcg(&a.mu[(int64_t)h * D + v * 8 + e]);
      const uint4* base = k + (int64_t)h * hstride + (int64_t)row0 * rstride + v;
      float best = 0.f;
      // Uniform trip count across the block so the lane shuffles stay converged.
      for (int r0 = 0; r0 < rows; r0 += kUnroll * RPI) {
        uint4 x[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int r = r0 + u * RPI + rs;
          x[u] = r < rows ? ld_policy(base + (int64_t)r * rstride, last_use) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int r = r0 + u * RPI + rs;
          float f[8];
          unpack8(x[u], f);
          float s = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float t = f[e] - m[e];
            s = fmaf(t, t, s);
          }
#pragma unroll
          for (int o = VPR / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
          if (r < rows) best = fmaxf(best, s);
        }
      }
      const float bm = block_max(best, sh.scratch);
      if (threadIdx.x == 0) a.kmax_part[pi] = bm;
      if (finish_item(&cent_frame_done[h * Nf + g], C, sh)) {
        if (threadIdx.x == 0)
          a.frame_max[(int64_t)h * Nf + g] = sqrtf(batched_max(&a.kmax_part[((int64_t)h * Nf + g) * C], C, 0.f));
        if (finish_item(&cent_done[h], Nf, sh)) {
          // Per query frame: the max of the visible frames' maxima and the
          // mean centred key over the visible keys (frame sums added in
          // frame order).  The head's frame sums and maxima are staged in
          // shared memory first when they fit.
          const bool cached = Nf <= kCacheFrames;
          if (cached) {
            if (threadIdx.x < D)
              for (int g0 = 0; g0 < Nf; g0 += 8) {
                float v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                  v[u] = g0 + u < Nf ? __ldcg(&a.fsum[((int64_t)h * Nf + g0 + u) * D + threadIdx.x]) : 0.f;
#pragma unroll
                for (int u = 0; u < 8; ++u)
                  if (g0 + u < Nf) sh.red[g0 + u][threadIdx.x] = v[u];
              }
            for (int gg = threadIdx.x; gg < Nf; gg += kThreads) sh.fmax[gg] = __ldcg(&a.frame_max[(int64_t)h * Nf + gg]);
          }
          __syncthreads();
          if (threadIdx.x < D) {
            const int e = threadIdx.x;
            const float mue = __ldcg(&a.mu[(int64_t)h * D + e]);
            for (int f = 0; f < Nf; ++f) {
              const int4 vis = visible(a, f);
              float acc = 0.f, mx = 0.f;
              int64_t cnt = 0;
              for (int part = 0; part < 2; ++part) {
                const int g0 = part == 0 ? vis.x : vis.z, g1 = part == 0 ? vis.y : vis.w;
                for (int gg = g0; gg < g1; ++gg) {
                  acc += cached ? sh.red[gg][e] : __ldcg(&a.fsum[((int64_t)h * Nf + gg) * D + e]);
                  mx = fmaxf(mx, cached ? sh.fmax[gg] : __ldcg(&a.frame_max[(int64_t)h * Nf + gg]));
                  cnt += span(a, gg).y;
                }
              }
              a.kbarc[((int64_t)h * Nf + f) * D + e] = acc / (float)cnt - mue;
              if (e == 0) a.mvis[(int64_t)h * Nf + f] = mx;
            }
          }
          publish(&win_ready[h]);
        }
      }
    } else {
      // Row bounds and the chunk's largest slack.
      float m[8], kb[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        m[e] = __ldcg(&a.mu[(int64_t)h * D + v * 8 + e]);
        kb[e] = __ldcg(&a.kbarc[((int64_t)h * Nf + g) * D + v * 8 + e]);
      }
      const float Mv = __ldcg(&a.mvis[(int64_t)h * Nf + g]);
      const uint4* base = q + (int64_t)h * hstride + (int64_t)row0 * rstride + v;
      float* out = a.row_bound + (int64_t)h * a.N + row0;
      float gmax = -INFINITY;
      for (int r0 = 0; r0 < rows; r0 += kUnroll * RPI) {
        uint4 x[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int r = r0 + u * RPI + rs;
          x[u] = r < rows ? ld_policy(base + (int64_t)r * rstride, last_use) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int r = r0 + u * RPI + rs;
          float f[8];
          unpack8(x[u], f);
          float qq = 0.f, qm = 0.f, qk = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            qq = fmaf(f[e], f[e], qq);
            qm = fmaf(f[e], m[e], qm);
            qk = fmaf(f[e], kb[e], qk);
          }
#pragma unroll
          for (int o = VPR / 2; o > 0; o >>= 1) {
            qq += __shfl_xor_sync(0xffffffffu, qq, o);
            qm += __shfl_xor_sync(0xffffffffu, qm, o);
            qk += __shfl_xor_sync(0xffffffffu, qk, o);
          }
          if (r < rows && v == 0) {
            const float b = a.scale * sqrtf(qq) * Mv;
            out[r] = fmaf(a.scale, qm, b);
            gmax = fmaxf(gmax, b - a.scale * qk);
          }
        }
      }
      const float bm = block_max(gmax, sh.scratch);
      if (threadIdx.x == 0) a.gmax_part[pi] = bm;
      if (finish_item(&qry_done[h], per, sh)) {
        // Largest slack of the head over all its items (max is exact in any
        // order), with every thread loading.
        float mx = -INFINITY;
        for (int i = threadIdx.x; i < per; i += kThreads) mx = fmaxf(mx, __ldcg(&a.gmax_part[(int64_t)h * per + i]));
        mx = block_max(mx, sh.scratch);
        if (threadIdx.x == 0) {
          a.stat[h] = mx;
          a.elig[h] = mx <= FAS_ELIG_SLACK_NATS ? 1 : 0;
        }
      }
    }
  }
}

// Resident CTAs per SM of the kernel for one head dimension (looked up once
// per process; every device of one process is assumed to be a GB300).
template <int D>
int grid_size(int items) {
  static int per_sm = 0, sms = 0;
  if (per_sm == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, prepass_kernel<D>, kThreads, 0) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1, sms = sms > 0 ? sms : 1;
    if (per_sm > kPrepassCtasPerSm) per_sm = kPrepassCtasPerSm;
  }
  const int g = per_sm * sms;
  return g < items ? g : items;
}

template <int D>
int launch_d(const PrepassArgs& a, cudaStream_t st) {
  // The counters and flags start at zero; the eligibility bits start at 0
  // (ineligible: the online path is always correct) so that a prepass that
  // gives up on a wait leaves every head on the safe path.
  if (cudaMemsetAsync(a.sync, 0, prepass_sync_words(a.H, a.Nf) * sizeof(unsigned), st) != cudaSuccess) return -1;
  if (cudaMemsetAsync(a.elig, 0, (size_t)a.H, st) != cudaSuccess) return -1;
  const int items = 3 * (a.H + 2 * kLag) * a.Nf * a.chunks;
  prepass_kernel<D><<<grid_size<D>(items), kThreads, 0, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return -1;
  return 1;
}

}  // namespace

size_t prepass_sync_words(int H, int Nf) { return 1 + 2 * (size_t)H * Nf + 5 * (size_t)H; }

int launch_prepass(const PrepassArgs& a, cudaStream_t stream) {
  if (a.d == 128) return launch_d<128>(a, stream);
  if (a.d == 64) return launch_d<64>(a, stream);
  return -1;
}

}  // namespace fas
