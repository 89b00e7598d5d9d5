// Splash-style ablation: the frame-window + reference attention computed the
// way a general block-sparse kernel does it, for a measured "before".
//
// "HeyGen x Google Cloud: Avatar IV on TPU", section "Deleting the Mask": the
// kernel the work started from tiles the sequence in multiples of 128, so
// live blocks straddle frame boundaries; that forces a mask predicate in the
// inner loop wherever a block straddles a boundary, a padded sequence so the
// block grid tiles the full length, and the two parts of the mask (the
// frame window and the reference frame) as two attention passes that write
// full-precision intermediates, which a merge pass re-reads and combines.
//
// This file builds exactly that on the same tcgen05 machinery as the
// frame-aligned kernel (attention_core.cuh), so the two differ only in what
// the pages say changed:
//   - query tiles and key blocks of 128 tokens over the sequence padded to a
//     multiple of 128 (not frame-aligned; TMA reads zeros past the end);
//   - pass 0 covers each query tile's window keys (the union over its rows,
//     rounded out to 128), pass 1 the reference frames' keys rounded up to
//     128; in a block that is not wholly visible to a row, every element is
//     tested against the row's visible key range;
//   - online softmax only (running maximum, conditional rescale);
//   - each pass writes O / sum(P) and the natural-log LSE in fp32 for every
//     padded row; a third kernel merges the two passes by their LSEs into the
//     bf16 output and the final LSE.

#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "attention_core.cuh"
#include "fas.h"
#include "internal.h"
#include "kernels.h"
#include "ptx.cuh"

namespace fas {
namespace {

using namespace core;

constexpr int kAblBlock = 128;          // query tile and key block
constexpr int kAblChunks = kAblBlock / 16;

// Visible key tokens [lo, hi) of row `row` in one pass.
__device__ __forceinline__ int2 visible_keys(const AblationParams& a, int64_t row) {
  if (row >= a.f.N) return make_int2(0, 0);  // padding row: sees nothing
  const int fi = (int)(row / a.T);
  if (a.pass == 1) return make_int2(0, a.R0 * a.T);
  if (fi < a.R0) return make_int2(a.R0 * a.T, (int)a.f.N);
  const int lo = max(a.R0, fi - a.r), hi = min(a.Nf - 1, fi + a.r);
  return make_int2(lo * a.T, (hi + 1) * a.T);
}

// The mask predicate of a block: in a block that is not wholly inside the
// row's visible key range [lo, hi), every score is tested and the hidden
// ones set to -inf.  The test runs whenever any row of the warp needs it.
struct KeyRangeMask {
  static constexpr bool kActive = true;
  int kb;        // first key of the block
  int lo, hi;    // the row's visible keys
  bool partial;  // some row of the warp does not see the whole block
  template <int M>
  __device__ __forceinline__ void apply(uint32_t (&r)[M][16], int c0, int n) const {
    if (!partial) return;
#pragma unroll
    for (int u = 0; u < M; ++u) {
      if (u >= n) break;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int key = kb + (c0 + u) * 16 + e;
        if (key < lo || key >= hi) r[u][e] = __float_as_uint(-INFINITY);
      }
    }
  }
};

template <int D>
__device__ __forceinline__ void ablation_softmax(Barriers& bars, uint32_t tmem, int warp, int lane, int h, int qt,
                                                 int kstart, int nblk, const AblationParams& a) {
  const FwdParams& p = a.f;
  volatile int* abort_flag = &bars.abort;
  const int g = warp / 4;
  const int trow = (warp % 4) * 32 + lane;
  const uint32_t lane_base = (uint32_t)((warp % 4) * 32) << 16;
  const int64_t row = (int64_t)qt * kAblBlock + trow;  // token row, < Npad
  const int2 vis = visible_keys(a, row);
  const uint64_t sl2 = ptx::f32x2(p.scale_log2, p.scale_log2);
  OnlineRow st{-INFINITY, 0.f, 0.f, 0.f, 0.f};
  bool ok = true;
  for (int j = g; ok && j < nblk; j += kGroups) {
    const int buf = j & 1;
    const bool got = ptx::mbar_wait(ptx::smem_addr(&bars.s_full[buf]), (j >> 1) & 1, abort_flag, p.err,
                                    kErrWaitSoftmax, p.limit_ns);
    ok = __all_sync(0xffffffffu, got);
    if (!ok) break;
    ptx::tc_fence_after_sync();
    const uint32_t sbase = tmem + lane_base + s_col(buf, kAblBlock);
    const int kb = kstart + j * kAblBlock;
    const bool partial = !(kb >= vis.x && kb + kAblBlock <= vis.y);
    const KeyRangeMask mask{kb, vis.x, vis.y, __any_sync(0xffffffffu, partial) != 0};
    ok = online_block<D, kAblChunks>(bars, tmem, lane_base, sbase, j, trow, sl2, st, p, mask);
  }
  if (ok) {
    const bool got = ptx::mbar_wait(ptx::smem_addr(&bars.o_full), 0, abort_flag, p.err, kErrWaitSoftmax, p.limit_ns);
    ok = __all_sync(0xffffffffu, got);
  }
  ptx::named_barrier_sync(kSoftmaxBarrier, kSoftmaxThreads);
  if (ok) settle_sums(st, bars.mchain[(nblk - 1) & 1][trow]);
  bars.red[g][0][trow] = st.l0 + st.l1;
  bars.red[g][1][trow] = st.w0 + st.w1;
  ptx::named_barrier_sync(kSoftmaxBarrier, kSoftmaxThreads);
  const float l = bars.red[0][0][trow] + bars.red[1][0][trow];
  const float lw = bars.red[0][1][trow] + bars.red[1][1][trow];
  if (!ok) return;
  ptx::tc_fence_after_sync();
  // The pass's full-precision intermediate, for every (padded) row.
  const float inv = lw > 0.f ? 1.0f / lw : 0.0f;
  float* orow = a.o32 + ((int64_t)h * a.Npad + row) * D;
  constexpr int kOutChunks = D / 16 / kGroups;
  uint32_t o[kOutChunks][16];
#pragma unroll
  for (int u = 0; u < kOutChunks; ++u) ptx::tmem_ld16(tmem + lane_base + kColO + (g * kOutChunks + u) * 16, o[u]);
#pragma unroll
  for (int u = 0; u < kOutChunks; ++u) ptx::tmem_ld_wait(o[u]);
#pragma unroll
  for (int u = 0; u < kOutChunks; ++u) {
    float4* dst = reinterpret_cast<float4*>(orow + (g * kOutChunks + u) * 16);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4)
      dst[q4] = make_float4(__uint_as_float(o[u][4 * q4]) * inv, __uint_as_float(o[u][4 * q4 + 1]) * inv,
                            __uint_as_float(o[u][4 * q4 + 2]) * inv, __uint_as_float(o[u][4 * q4 + 3]) * inv);
  }
  if (g == 0) a.lse32[(int64_t)h * a.Npad + row] = l > 0.f ? (st.m_run + ptx::lg2(l)) * kLn2 : -INFINITY;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    ablation_fwd(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const AblationParams a) {
  const FwdParams& p = a.f;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Barriers bars;
  const uint32_t tiles = (ptx::smem_addr(smem_raw) + 1023u) & ~1023u;
  const uint32_t q_s = tiles;
  const uint32_t k_s0 = q_s + p.qslot_bytes;
  const uint32_t v_s0 = k_s0 + (uint32_t)p.kd * kAblBlock * D * 2;

  if (threadIdx.x == 0) bars.skip = *reinterpret_cast<volatile unsigned int*>(p.err) != 0u;
  __syncthreads();
  if (bars.skip) return;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int4 item = p.work[blockIdx.x];  // head, query tile, first key, key blocks
  const int h = item.x, qt = item.y, kstart = item.z, nblk = item.w;

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_addr(&bars.q_full), 1);
    ptx::mbar_init(ptx::smem_addr(&bars.q_tmem), 1);
    for (int s = 0; s < kMaxStages; ++s) {
      ptx::mbar_init(ptx::smem_addr(&bars.k_full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&bars.k_empty[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&bars.v_full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&bars.v_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_addr(&bars.s_full[b]), 1);
      ptx::mbar_init(ptx::smem_addr(&bars.pa_full[b]), 32 * 4);  // the block's warpgroup
      ptx::mbar_init(ptx::smem_addr(&bars.p_full[b]), 32 * 4);
      ptx::mbar_init(ptx::smem_addr(&bars.mchain_bar[b]), 32 * 4);
    }
    ptx::mbar_init(ptx::smem_addr(&bars.pv_done), 1);
    ptx::mbar_init(ptx::smem_addr(&bars.o_full), 1);
    ptx::mbar_init(ptx::smem_addr(&bars.drain), 1);
    bars.abort = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_addr(&bars.tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem = bars.tmem_base;

  if (warp == kKProducerWarp) {
    if (lane == 0) {
      ptx::mbar_arrive_expect_tx(ptx::smem_addr(&bars.q_full), kQTile * D * 2);
#pragma unroll
      for (int half = 0; half < D / 64; ++half)
        ptx::tma_load_3d(q_s + half * (kQTile * 128), &tm_q, ptx::smem_addr(&bars.q_full), half * 64,
                         qt * kAblBlock, h);
      ring_producer<D>(&tm_k, bars.k_full, bars.k_empty, p.kst, p.kd, k_s0, q_s, &bars.q_tmem, h,
                       make_int4(kstart, nblk * kAblBlock, 0, 0), &bars.abort, p);
      if (bars.abort) drain_wait(ptx::smem_addr(&bars.q_full), 0, p.err, p.limit_ns);
    }
  } else if (warp == kVProducerWarp) {
    if (lane == 0)
      ring_producer<D>(&tm_v, bars.v_full, bars.v_empty, p.vst, p.vst, v_s0, 0, nullptr, h,
                       make_int4(kstart, nblk * kAblBlock, 0, 0), &bars.abort, p);
  } else if (warp == kMmaWarp) {
    if (ptx::elect_one()) mma_issuer<D, kAblChunks>(bars, tmem, q_s, k_s0, v_s0, nblk, false, p);
    __syncwarp();
  } else {
    ablation_softmax<D>(bars, tmem, warp, lane, h, qt, kstart, nblk, a);
  }

  ptx::tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// The merge pass: reads both passes' fp32 intermediates and combines them by
// their LSEs (log-sum-exp of the two partial softmax sums).  One warp per
// row; each lane handles d/32 consecutive columns.
template <int D>
__global__ void __launch_bounds__(256) ablation_merge(const float* __restrict__ o0, const float* __restrict__ l0,
                                                      const float* __restrict__ o1, const float* __restrict__ l1,
                                                      uint16_t* __restrict__ out, float* __restrict__ lse, int H,
                                                      int64_t N, int64_t Npad) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x % 32;
  const int64_t rows = (int64_t)H * N;
  for (int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) / 32; w < rows;
       w += (int64_t)gridDim.x * blockDim.x / 32) {
    const int64_t h = w / N, i = w % N;
    const int64_t src = h * Npad + i;
    const float a = l0[src], b = l1 ? l1[src] : -INFINITY;
    const float m = fmaxf(a, b);
    const float wa = a == -INFINITY ? 0.f : expf(a - m), wb = b == -INFINITY ? 0.f : expf(b - m);
    const float tot = wa + wb;
    const float ca = wa / tot, cb = wb / tot;
    float x[E];
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = ca * o0[src * D + lane * E + e];
    if (l1) {
#pragma unroll
      for (int e = 0; e < E; ++e) x[e] = fmaf(cb, o1[src * D + lane * E + e], x[e]);
    }
    uint16_t* dst = out + (h * N + i) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      uint32_t pk;
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(pk) : "f"(x[e + 1]), "f"(x[e]));
      *reinterpret_cast<uint32_t*>(dst + e) = pk;
    }
    if (lane == 0) lse[h * N + i] = m + logf(tot);
  }
}

template <int D>
cudaError_t launch_ablation_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, AblationParams a,
                              int grid, cudaStream_t st) {
  const size_t smem = ring_plan(D, kAblBlock, &a.f);
  if (smem == 0) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(ablation_fwd<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  ablation_fwd<D><<<grid, kThreads, smem, st>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ablation_pass(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const AblationParams& a, int grid, cudaStream_t stream) {
  if (a.f.Bk != kAblBlock) return cudaErrorInvalidValue;
  if (d == 128) return launch_ablation_d<128>(tq, tk, tv, a, grid, stream);
  if (d == 64) return launch_ablation_d<64>(tq, tk, tv, a, grid, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_ablation_merge(int d, const float* o0, const float* l0, const float* o1, const float* l1,
                                  uint16_t* out, float* lse, int H, int64_t N, int64_t Npad, cudaStream_t stream) {
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
    return cudaErrorInvalidValue;
  const int64_t warps = (int64_t)H * N;
  int64_t blocks = (warps * 32 + 255) / 256;
  if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
  if (d == 128)
    ablation_merge<128><<<(int)blocks, 256, 0, stream>>>(o0, l0, o1, l1, out, lse, H, N, Npad);
  else if (d == 64)
    ablation_merge<64><<<(int)blocks, 256, 0, stream>>>(o0, l0, o1, l1, out, lse, H, N, Npad);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace fas
