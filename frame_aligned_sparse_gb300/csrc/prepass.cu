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
// All loads are 16-byte vectors, one row shared by d/8 consecutive lanes
// (each row's d values are contiguous), consecutive rows over the block.
// Rows of one head are row_stride elements apart: d in the head-major
// [H, N, d] layout (fully contiguous), H*d in the token-major [N, H, d]
// layout (one 2d-byte segment per row).  Every reduction runs in
// a fixed order (no floating-point atomics), so results are bit-reproducible.

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fas.h"
#include "internal.h"
#include "kernels.h"

namespace fas {
namespace {

constexpr int kPrepassThreads = 256;

__device__ __forceinline__ void unpack8(const uint4& x, float (&f)[8]) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    f[2 * e] = __uint_as_float(w[e] << 16);
    f[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Block-wide max of one float per thread (kPrepassThreads threads).
__device__ __forceinline__ float block_max(float v, float* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  float r = scratch[0];
  for (int w = 1; w < kPrepassThreads / 32; ++w) r = fmaxf(r, scratch[w]);
  return r;
}

// (1) Per (head, frame, chunk) column sums of the keys.
template <int D>
__global__ void __launch_bounds__(kPrepassThreads) key_chunk_sums(const uint4* __restrict__ k,
                                                                  float* __restrict__ partial, int64_t N,
                                                                  int64_t rstride, int64_t hstride, int T,
                                                                  int Nf, int chunks) {
  constexpr int VPR = D / 8;                   // 16-byte vectors per row
  constexpr int RPI = kPrepassThreads / VPR;   // rows per sweep
  __shared__ float red[RPI][D];
  const int c = blockIdx.x, g = blockIdx.y, h = blockIdx.z;
  const int v = threadIdx.x % VPR, rs = threadIdx.x / VPR;
  const int row0 = c * kPrepassRows;
  const int rows = min(kPrepassRows, T - row0);
  const uint4* base = k + (int64_t)h * hstride + ((int64_t)g * T + row0) * rstride + v;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  int r = rs;
  for (; r + 3 * RPI < rows; r += 4 * RPI) {
    uint4 x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) x[u] = ld_stream(base + (int64_t)(r + u * RPI) * rstride);
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
    unpack8(ld_stream(base + (int64_t)r * rstride), f);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] += f[e];
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) red[rs][v * 8 + e] = acc[e];
  __syncthreads();
  if (threadIdx.x < D) {
    float s = 0.f;
    for (int q = 0; q < RPI; ++q) s += red[q][threadIdx.x];
    partial[(((int64_t)h * Nf + g) * chunks + c) * D + threadIdx.x] = s;
  }
}

// (2) Per-frame key sums and the per-head mean key.  One block per head,
// one thread per column.
template <int D>
__global__ void __launch_bounds__(D) key_frame_sums(const float* __restrict__ partial, float* __restrict__ fsum,
                                                    float* __restrict__ mu, int64_t N, int Nf, int chunks) {
  const int h = blockIdx.x, e = threadIdx.x;
  float tot = 0.f;
  for (int g = 0; g < Nf; ++g) {
    float s = 0.f;
    for (int c = 0; c < chunks; ++c) s += partial[(((int64_t)h * Nf + g) * chunks + c) * D + e];
    fsum[((int64_t)h * Nf + g) * D + e] = s;
    tot += s;
  }
  mu[(int64_t)h * D + e] = tot / (float)N;
}

// (3) Per (head, frame, chunk) max of |k_j - mu_h|.
template <int D>
__global__ void __launch_bounds__(kPrepassThreads) key_centred_max(const uint4* __restrict__ k,
                                                                   const float* __restrict__ mu,
                                                                   float* __restrict__ mpart, int64_t N,
                                                                   int64_t rstride, int64_t hstride, int T,
                                                                   int Nf, int chunks) {
  constexpr int VPR = D / 8;
  constexpr int RPI = kPrepassThreads / VPR;
  __shared__ float scratch[kPrepassThreads / 32];
  const int c = blockIdx.x, g = blockIdx.y, h = blockIdx.z;
  const int v = threadIdx.x % VPR, rs = threadIdx.x / VPR;
  const int row0 = c * kPrepassRows;
  const int rows = min(kPrepassRows, T - row0);
  float m[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) m[e] = mu[(int64_t)h * D + v * 8 + e];
  const uint4* base = k + (int64_t)h * hstride + ((int64_t)g * T + row0) * rstride + v;
  float best = 0.f;
  // Uniform trip count across the block so the lane shuffles stay converged.
  for (int r0 = 0; r0 < rows; r0 += 2 * RPI) {
    uint4 x[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int r = r0 + u * RPI + rs;
      x[u] = r < rows ? ld_stream(base + (int64_t)r * rstride) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
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
  const float bm = block_max(best, scratch);
  if (threadIdx.x == 0) mpart[((int64_t)h * Nf + g) * chunks + c] = sqrtf(bm);
}

// (4) Per head: frame maxima, and for every query frame the max over its
// visible frames and the mean centred key over its visible keys.  Visible
// frames come from the block table (the same ranges the attention walks).
template <int D>
__global__ void __launch_bounds__(D) window_stats(const float* __restrict__ mpart, const float* __restrict__ fsum,
                                                  const float* __restrict__ mu, const int4* __restrict__ table,
                                                  float* __restrict__ frame_max, float* __restrict__ mvis,
                                                  float* __restrict__ kbarc, int T, int Nf, int chunks) {
  const int h = blockIdx.x, e = threadIdx.x;
  for (int g = e; g < Nf; g += D) {
    float mx = 0.f;
    for (int c = 0; c < chunks; ++c) mx = fmaxf(mx, mpart[((int64_t)h * Nf + g) * chunks + c]);
    frame_max[(int64_t)h * Nf + g] = mx;
  }
  __syncthreads();
  const float mue = mu[(int64_t)h * D + e];
  for (int f = 0; f < Nf; ++f) {
    const int4 t = table[f];
    const int g0 = t.x / T, g1 = (t.x + t.y) / T, g2 = t.z / T, g3 = (t.z + t.w) / T;
    float acc = 0.f, mx = 0.f;
    for (int g = g0; g < g1; ++g) {
      acc += fsum[((int64_t)h * Nf + g) * D + e];
      mx = fmaxf(mx, frame_max[(int64_t)h * Nf + g]);
    }
    for (int g = g2; g < g3; ++g) {
      acc += fsum[((int64_t)h * Nf + g) * D + e];
      mx = fmaxf(mx, frame_max[(int64_t)h * Nf + g]);
    }
    kbarc[((int64_t)h * Nf + f) * D + e] = acc / (float)(t.y + t.w) - mue;
    if (e == 0) mvis[(int64_t)h * Nf + f] = mx;
  }
}

// (4') The same statistics with the visible frames taken straight from the
// frame rule (reference frames global both ways, window clipped to the
// video frames) instead of a block table in device memory.
template <int D>
__global__ void __launch_bounds__(D) window_stats_rule(const float* __restrict__ mpart,
                                                       const float* __restrict__ fsum, const float* __restrict__ mu,
                                                       float* __restrict__ frame_max, float* __restrict__ mvis,
                                                       float* __restrict__ kbarc, int T, int Nf, int chunks, int R0,
                                                       int r) {
  const int h = blockIdx.x, e = threadIdx.x;
  for (int g = e; g < Nf; g += D) {
    float mx = 0.f;
    for (int c = 0; c < chunks; ++c) mx = fmaxf(mx, mpart[((int64_t)h * Nf + g) * chunks + c]);
    frame_max[(int64_t)h * Nf + g] = mx;
  }
  __syncthreads();
  const float mue = mu[(int64_t)h * D + e];
  for (int f = 0; f < Nf; ++f) {
    // Visible frames: [0, a) and [b, c).
    int a, b, c;
    if (f < R0) {
      a = Nf; b = Nf; c = Nf;
    } else {
      a = R0; b = max(R0, f - r); c = min(Nf - 1, f + r) + 1;
    }
    float acc = 0.f, mx = 0.f;
    for (int g = 0; g < a; ++g) {
      acc += fsum[((int64_t)h * Nf + g) * D + e];
      mx = fmaxf(mx, frame_max[(int64_t)h * Nf + g]);
    }
    for (int g = b; g < c; ++g) {
      acc += fsum[((int64_t)h * Nf + g) * D + e];
      mx = fmaxf(mx, frame_max[(int64_t)h * Nf + g]);
    }
    kbarc[((int64_t)h * Nf + f) * D + e] = acc / (float)((a + c - b) * T) - mue;
    if (e == 0) mvis[(int64_t)h * Nf + f] = mx;
  }
}

// (5) Per row: m_i, and the per-chunk max of the slack G_i.
template <int D>
__global__ void __launch_bounds__(kPrepassThreads) query_bounds(const uint4* __restrict__ q,
                                                                const float* __restrict__ mu,
                                                                const float* __restrict__ mvis,
                                                                const float* __restrict__ kbarc,
                                                                float* __restrict__ row_bound,
                                                                float* __restrict__ gpart, int64_t N,
                                                                int64_t rstride, int64_t hstride, int T,
                                                                int Nf, int chunks, float scale) {
  constexpr int VPR = D / 8;
  constexpr int RPI = kPrepassThreads / VPR;
  __shared__ float scratch[kPrepassThreads / 32];
  const int c = blockIdx.x, g = blockIdx.y, h = blockIdx.z;
  const int v = threadIdx.x % VPR, rs = threadIdx.x / VPR;
  const int row0 = c * kPrepassRows;
  const int rows = min(kPrepassRows, T - row0);
  float m[8], kb[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    m[e] = mu[(int64_t)h * D + v * 8 + e];
    kb[e] = kbarc[((int64_t)h * Nf + g) * D + v * 8 + e];
  }
  const float Mv = mvis[(int64_t)h * Nf + g];
  const uint4* base = q + (int64_t)h * hstride + ((int64_t)g * T + row0) * rstride + v;
  float* out = row_bound + (int64_t)h * N + (int64_t)g * T + row0;
  float gmax = -INFINITY;
  for (int r0 = 0; r0 < rows; r0 += 2 * RPI) {
    uint4 x[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int r = r0 + u * RPI + rs;
      x[u] = r < rows ? ld_stream(base + (int64_t)r * rstride) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
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
        const float b = scale * sqrtf(qq) * Mv;
        out[r] = fmaf(scale, qm, b);
        gmax = fmaxf(gmax, b - scale * qk);
      }
    }
  }
  const float bm = block_max(gmax, scratch);
  if (threadIdx.x == 0) gpart[((int64_t)h * Nf + g) * chunks + c] = bm;
}

// (6) Per head: stat_h = max slack, eligibility bit.
__global__ void __launch_bounds__(256) eligibility(const float* __restrict__ gpart, float* __restrict__ stat,
                                                   uint8_t* __restrict__ elig, int H, int per_head) {
  for (int h = blockIdx.x * blockDim.x + threadIdx.x; h < H; h += gridDim.x * blockDim.x) {
    float mx = -INFINITY;
    for (int i = 0; i < per_head; ++i) mx = fmaxf(mx, gpart[(int64_t)h * per_head + i]);
    stat[h] = mx;
    elig[h] = mx <= FAS_ELIG_SLACK_NATS ? 1 : 0;
  }
}

template <int D>
int launch_prepass_d(const PrepassArgs& a, cudaStream_t st) {
  const dim3 grid(a.chunks, a.Nf, a.H);
  const uint4* q = static_cast<const uint4*>(a.q);
  const uint4* k = static_cast<const uint4*>(a.k);
  const int64_t rstride = a.row_stride / 8, hstride = a.head_stride / 8;  // in 16-byte vectors
  int n = 0;
  key_chunk_sums<D><<<grid, kPrepassThreads, 0, st>>>(k, a.partial, a.N, rstride, hstride, a.T, a.Nf, a.chunks);
  ++n;
  key_frame_sums<D><<<a.H, D, 0, st>>>(a.partial, a.fsum, a.mu, a.N, a.Nf, a.chunks);
  ++n;
  key_centred_max<D><<<grid, kPrepassThreads, 0, st>>>(k, a.mu, a.mpart, a.N, rstride, hstride, a.T, a.Nf,
                                                      a.chunks);
  ++n;
  window_stats<D><<<a.H, D, 0, st>>>(a.mpart, a.fsum, a.mu, a.table, a.frame_max, a.mvis, a.kbarc, a.T, a.Nf,
                                     a.chunks);
  ++n;
  query_bounds<D><<<grid, kPrepassThreads, 0, st>>>(q, a.mu, a.mvis, a.kbarc, a.row_bound, a.gpart, a.N, rstride,
                                                    hstride, a.T, a.Nf, a.chunks, a.scale);
  ++n;
  const int blocks = (a.H + 255) / 256;
  eligibility<<<blocks, 256, 0, st>>>(a.gpart, a.stat, a.elig, a.H, a.Nf * a.chunks);
  ++n;
  if (cudaGetLastError() != cudaSuccess) return -1;
  return n;
}

template <int D>
int launch_prepass_rule_d(const PrepassArgs& a, int R0, int r, cudaStream_t st) {
  const dim3 grid(a.chunks, a.Nf, a.H);
  const uint4* q = static_cast<const uint4*>(a.q);
  const uint4* k = static_cast<const uint4*>(a.k);
  const int64_t rstride = a.row_stride / 8, hstride = a.head_stride / 8;  // in 16-byte vectors
  int n = 0;
  key_chunk_sums<D><<<grid, kPrepassThreads, 0, st>>>(k, a.partial, a.N, rstride, hstride, a.T, a.Nf, a.chunks);
  ++n;
  key_frame_sums<D><<<a.H, D, 0, st>>>(a.partial, a.fsum, a.mu, a.N, a.Nf, a.chunks);
  ++n;
  key_centred_max<D><<<grid, kPrepassThreads, 0, st>>>(k, a.mu, a.mpart, a.N, rstride, hstride, a.T, a.Nf,
                                                      a.chunks);
  ++n;
  window_stats_rule<D><<<a.H, D, 0, st>>>(a.mpart, a.fsum, a.mu, a.frame_max, a.mvis, a.kbarc, a.T, a.Nf, a.chunks,
                                          R0, r);
  ++n;
  query_bounds<D><<<grid, kPrepassThreads, 0, st>>>(q, a.mu, a.mvis, a.kbarc, a.row_bound, a.gpart, a.N, rstride,
                                                    hstride, a.T, a.Nf, a.chunks, a.scale);
  ++n;
  const int blocks = (a.H + 255) / 256;
  eligibility<<<blocks, 256, 0, st>>>(a.gpart, a.stat, a.elig, a.H, a.Nf * a.chunks);
  ++n;
  if (cudaGetLastError() != cudaSuccess) return -1;
  return n;
}

}  // namespace

int launch_prepass_rule(const PrepassArgs& a, int ref_frames, int window_radius, cudaStream_t stream) {
  if (a.d == 128) return launch_prepass_rule_d<128>(a, ref_frames, window_radius, stream);
  if (a.d == 64) return launch_prepass_rule_d<64>(a, ref_frames, window_radius, stream);
  return -1;
}

int launch_prepass(const PrepassArgs& a, cudaStream_t stream) {
  if (a.d == 128) return launch_prepass_d<128>(a, stream);
  if (a.d == 64) return launch_prepass_d<64>(a, stream);
  return -1;
}

}  // namespace fas
