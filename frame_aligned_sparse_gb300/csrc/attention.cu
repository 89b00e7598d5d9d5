// Frame-aligned sparse attention, single pass, for sm_103a.
//
// "HeyGen x Google Cloud: Avatar IV on TPU":
//  - "Deleting the Mask" (Fig. 3): key blocks divide the frame's token span,
//    so every visible block is full; the kernel walks the (at most two)
//    visible key ranges of its query frame block by block — the reference
//    frame's blocks are just more blocks of the same softmax.  No mask
//    predicate, no padding, no second pass, no merge.
//  - "Unchaining the Softmax" (Fig. 4): eligible heads use a fixed per-row
//    maximum m_i (precomputed Cauchy-Schwarz bound), so the inner loop has no
//    running max and no rescale; other heads run the online softmax (running
//    max, conditional rescale of the accumulator) inside the same kernel.
//  - "Proving the Pixels Didn't Change": the P.V product runs in bf16 on the
//    tensor cores with fp32 accumulation.
//
// One CTA per work item (head h, query frame f, query tile of 128 rows).
//   warps 0-7   softmax + epilogue in two warpgroups.  Thread (g, w, t) owns
//               row 32(w%4) + t of the tile, i.e. TMEM lane 32(w%4) + t (warp
//               w may only read lanes 32(w%4)..+31).  For bounded heads group
//               g handles the blocks of S buffer g (even or odd blocks): the
//               two groups ping-pong, each hiding the other's waits.  Online
//               heads ping-pong the same way and pass the running row
//               maximum from each block's group to the next block's.
//   warp 8      TMA producer of the Q tile and the K ring
//   warp 9      TMA producer of the V ring (never waits behind K)
//   warp 10     TMEM allocator and tcgen05.mma issuer (whole warp, one
//               elected lane issues)
// TMEM (512 columns): O at [0, d), S buffers at 128 and 128 + roundup32(Bk),
// and the Q tile (bf16 pairs) at [448, 512) so that S = Q.K^T reads its A
// operand from TMEM instead of shared memory.
// The bf16 P of each 16-column chunk overwrites the first 8 columns of that
// chunk (already read by the same thread) and feeds the P.V MMA straight
// from TMEM, one 16-key MMA per chunk.
// MMA issue order: S0, S1, PV0, S2, PV1, ...; the tensor pipe executes them
// in order, so S(j+2) never overwrites P(j) before PV(j) has read it.
// The kernel is instantiated per number of 16-key chunks in a block (the
// plan fixes the block size), so every loop over chunks is unrolled with no
// run-time predicate around the warp-collective tcgen05 loads, stores and
// MMAs: predicated forms of them measured ~20% slower.

#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fas.h"
#include "internal.h"
#include "kernels.h"
#include "attention_core.cuh"
#include "ptx.cuh"

namespace fas {
namespace {

using namespace core;

// Softmax and epilogue for one thread: row `trow` of the tile.  Warpgroup g
// takes the blocks j with j % 2 == g, exactly the blocks of S buffer g, so
// the two groups ping-pong, each hiding the other's waits.  Bounded heads
// use the fixed per-row maximum and the groups never talk until the
// epilogue; online heads pass the running maximum from block to block
// (online_block).
template <int D, int NCH>
__device__ __forceinline__ void softmax_epilogue(Barriers& bars, uint32_t tmem, int warp, int lane, int h, int f,
                                                 int qt, int nblk, bool bounded, const FwdParams& p) {
  volatile int* abort_flag = &bars.abort;
  const int g = warp / 4;
  const int trow = (warp % 4) * 32 + lane;
  const uint32_t lane_base = (uint32_t)((warp % 4) * 32) << 16;
  const int2 sp = p.spans[f];  // first token and span of the query frame
  const int row = qt * kQTile + trow;  // row inside the frame
  const bool valid = row < sp.y;
  const int64_t grow = (int64_t)h * p.N + sp.x + row;
  constexpr int kPa = (NCH + 1) / 2;  // chunks in the first half of a block
  const uint64_t sl2 = ptx::f32x2(p.scale_log2, p.scale_log2);
  // Bounded heads: the row maximum in log2 units of the scaled logits.  A
  // row past the frame's end (zeros, or the next frame's rows when frames
  // are ragged) is never stored; with an infinite maximum its probabilities
  // are all zero.  The sums: l of the fp32 probabilities (for the LSE) and
  // w of the bf16-rounded weights the P.V MMA actually uses (for
  // normalising O, so the output is a convex combination of V rows even
  // when the largest probability is not 1).
  OnlineRow st{-INFINITY, 0.f, 0.f, 0.f, 0.f};
  if (bounded) st.m_run = valid ? p.row_bound[grow] * kLog2e : INFINITY;
  bool ok = true;

  for (int j = g; ok && j < nblk; j += kGroups) {
    const int buf = j & 1;
    const bool got = ptx::mbar_wait(ptx::smem_addr(&bars.s_full[buf]), (j >> 1) & 1, abort_flag, p.err,
                                    kErrWaitSoftmax, p.limit_ns);
    ok = __all_sync(0xffffffffu, got);
    if (!ok) break;
    ptx::tc_fence_after_sync();
    const uint32_t sbase = tmem + lane_base + s_col(buf, NCH * 16);
    if (!bounded) {
      ok = online_block<D, NCH>(bars, tmem, lane_base, sbase, j, trow, sl2, st, p);
      continue;
    }
    // P of the block's first chunks is released as soon as it is stored, so
    // that their P.V MMAs run while the rest of the block is exponentiated.
    const uint64_t neg_m = ptx::f32x2(-st.m_run, -st.m_run);
    softmax_phase<0, kPa>(sbase, sl2, neg_m, st.l0, st.l1, st.w0, st.w1);
    ptx::tmem_st_wait();
    ptx::tc_fence_before_sync();
    ptx::mbar_arrive(ptx::smem_addr(&bars.pa_full[buf]));
    softmax_phase<kPa, NCH - kPa>(sbase, sl2, neg_m, st.l0, st.l1, st.w0, st.w1);
    ptx::tmem_st_wait();
    ptx::tc_fence_before_sync();
    ptx::mbar_arrive(ptx::smem_addr(&bars.p_full[buf]));
  }

  // Epilogue: combine the groups' row sums, then each group writes half of
  // the output columns.  Every softmax thread reaches the named barrier.
  if (ok) {
    const bool got = ptx::mbar_wait(ptx::smem_addr(&bars.o_full), 0, abort_flag, p.err, kErrWaitSoftmax, p.limit_ns);
    ok = __all_sync(0xffffffffu, got);
  }
  if (!bounded) {
    // Both groups' sums against the maximum after the last block (published
    // by its group before the named barrier below; read after a first one).
    ptx::named_barrier_sync(kSoftmaxBarrier, kSoftmaxThreads);
    if (ok) settle_sums(st, bars.mchain[(nblk - 1) & 1][trow]);
  }
  bars.red[g][0][trow] = st.l0 + st.l1;
  bars.red[g][1][trow] = st.w0 + st.w1;
  ptx::named_barrier_sync(kSoftmaxBarrier, kSoftmaxThreads);
  float l = 0.f, lw = 0.f;
#pragma unroll
  for (int q = 0; q < kGroups; ++q) {
    l += bars.red[q][0][trow];
    lw += bars.red[q][1][trow];
  }
  if (!ok) return;
  // A bound that does not hold for these q and k shows in the row's sum
  // (see kFlagBoundRange); the row is still written, the host is told.
  if (bounded && valid && g == 0 && !(l >= kBoundSumMin && l <= kBoundSumMax)) atomicOr(p.flags, kFlagBoundRange);
  ptx::tc_fence_after_sync();
  const float inv = 1.0f / lw;
  uint16_t* orow = p.out + (int64_t)h * p.out_head_stride + ((int64_t)sp.x + row) * p.out_row_stride;
  constexpr int kOutChunks = D / 16 / kGroups;
  // All of the group's O columns are loaded before one wait.
  uint32_t o[kOutChunks][16];
#pragma unroll
  for (int u = 0; u < kOutChunks; ++u) ptx::tmem_ld16(tmem + lane_base + kColO + (g * kOutChunks + u) * 16, o[u]);
#pragma unroll
  for (int u = 0; u < kOutChunks; ++u) ptx::tmem_ld_wait(o[u]);
#pragma unroll
  for (int u = 0; u < kOutChunks; ++u) {
    uint32_t pk[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
      pk[e] = ptx::pack_bf16x2(__uint_as_float(o[u][2 * e]) * inv, __uint_as_float(o[u][2 * e + 1]) * inv);
    if (valid) {
      uint4* dst = reinterpret_cast<uint4*>(orow + (g * kOutChunks + u) * 16);
      dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
    }
  }
  if (valid && g == 0) p.lse[grow] = (st.m_run + ptx::lg2(l)) * kLn2;
}

template <int D, int NCH>
__global__ void __launch_bounds__(kThreads, 1)
    attention_fwd(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Barriers bars;
  const uint32_t tiles = (ptx::smem_addr(smem_raw) + 1023u) & ~1023u;  // 128B-swizzle atoms need 1 KB alignment
  const uint32_t q_s = tiles;  // Q tile, then (once Q is in TMEM) K stage kd
  const uint32_t k_s0 = q_s + p.qslot_bytes;
  const uint32_t v_s0 = k_s0 + (uint32_t)p.kd * p.Bk * D * 2;

  // A CTA of this launch (or an earlier one) already gave up on a wait: the
  // whole CTA does nothing (the host reports FAS_ERR_TIMEOUT).  One thread
  // reads the error word so that every thread takes the same decision
  // before any barrier or TMEM is set up.
  if (threadIdx.x == 0) bars.skip = *reinterpret_cast<volatile unsigned int*>(p.err) != 0u;
  __syncthreads();
  if (bars.skip) return;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int4 item = p.work[blockIdx.x];
  const int h = item.x, f = item.y, qt = item.z, nblk = item.w;
  const bool bounded = p.mode == FAS_MODE_BOUNDED || (p.mode == FAS_MODE_AUTO && p.elig[h] != 0);

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_addr(&bars.q_full), 1);
    ptx::mbar_init(ptx::smem_addr(&bars.q_tmem), 1);  // tcgen05.commit after the Q copy
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
      const int2 sp = p.spans[f];
#pragma unroll
      for (int half = 0; half < D / 64; ++half) {
        // Uniform frames: a rank-4 map {d, T, Nf, H} reads zeros past the
        // frame's end.  Ragged frames: a rank-3 map {d, N, H}; the rows
        // past the frame's end are computed and discarded.
        if (p.q_by_frame)
          ptx::tma_load_4d(q_s + half * (kQTile * 128), &tm_q, ptx::smem_addr(&bars.q_full), half * 64, qt * kQTile,
                           f, h);
        else
          ptx::tma_load_3d(q_s + half * (kQTile * 128), &tm_q, ptx::smem_addr(&bars.q_full), half * 64,
                           sp.x + qt * kQTile, h);
      }
      ring_producer<D>(&tm_k, bars.k_full, bars.k_empty, p.kst, p.kd, k_s0, q_s, &bars.q_tmem, h, p.table[f],
                       &bars.abort, p);
      if (bars.abort) drain_wait(ptx::smem_addr(&bars.q_full), 0, p.err, p.limit_ns);
    }
  } else if (warp == kVProducerWarp) {
    if (lane == 0)
      ring_producer<D>(&tm_v, bars.v_full, bars.v_empty, p.vst, p.vst, v_s0, 0, nullptr, h, p.table[f], &bars.abort,
                       p);
  } else if (warp == kMmaWarp) {
    if (ptx::elect_one()) mma_issuer<D, NCH>(bars, tmem, q_s, k_s0, v_s0, nblk, bounded, p);
    __syncwarp();
  } else {
    softmax_epilogue<D, NCH>(bars, tmem, warp, lane, h, f, qt, nblk, bounded, p);
  }

  ptx::tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

__global__ void wait_selftest(unsigned int* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_addr(&bar), 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  // Nothing ever arrives on `bar`: the bounded wait must give up and report.
  if (threadIdx.x == 0)
    ptx::mbar_wait(ptx::smem_addr(&bar), 0, &abort_flag, err, kErrWaitSelftest, limit_ns);
  __syncthreads();
}

template <int D, int NCH>
cudaError_t launch_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, FwdParams p, int grid,
                     cudaStream_t st) {
  const size_t smem = ring_plan(D, p.Bk, &p);
  if (smem == 0) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(attention_fwd<D, NCH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  attention_fwd<D, NCH><<<grid, kThreads, smem, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

// One instantiation per (head dimension, chunks per key block): the block
// size is fixed per plan, so the kernel's loops are fully unrolled for it.
template <int D>
cudaError_t launch_dim(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                       int grid, cudaStream_t stream) {
  static_assert(kMaxBlockK == 160, "extend the dispatch below");
  if (p.Bk % 16 != 0) return cudaErrorInvalidValue;
  switch (p.Bk / 16) {
    case 1: return launch_d<D, 1>(tq, tk, tv, p, grid, stream);
    case 2: return launch_d<D, 2>(tq, tk, tv, p, grid, stream);
    case 3: return launch_d<D, 3>(tq, tk, tv, p, grid, stream);
    case 4: return launch_d<D, 4>(tq, tk, tv, p, grid, stream);
    case 5: return launch_d<D, 5>(tq, tk, tv, p, grid, stream);
    case 6: return launch_d<D, 6>(tq, tk, tv, p, grid, stream);
    case 7: return launch_d<D, 7>(tq, tk, tv, p, grid, stream);
    case 8: return launch_d<D, 8>(tq, tk, tv, p, grid, stream);
    case 9: return launch_d<D, 9>(tq, tk, tv, p, grid, stream);
    case 10: return launch_d<D, 10>(tq, tk, tv, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_attention(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const FwdParams& p, int grid, cudaStream_t stream) {
  if (d == 128) return launch_dim<128>(tq, tk, tv, p, grid, stream);
  if (d == 64) return launch_dim<64>(tq, tk, tv, p, grid, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_wait_selftest(unsigned int* err, uint64_t limit_ns, cudaStream_t stream) {
  wait_selftest<<<1, 32, 0, stream>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace fas
