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
//               two groups ping-pong, each hiding the other's waits.  For
//               online heads group 0 handles every block.
//   warp 8      TMA producer of the Q tile and the K ring
//   warp 9      TMA producer of the V ring (never waits behind K)
//   warp 10     TMEM allocator and tcgen05.mma issuer (whole warp, one
//               elected lane issues)
// TMEM (512 columns): O at [0, d), S buffers at 128 and 128 + roundup32(Bk),
// and, when Bk leaves room, the Q tile (bf16 pairs) at [448, 512) so that
// S = Q.K^T reads its A operand from TMEM instead of shared memory.
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
#include "ptx.cuh"

namespace fas {
namespace {

constexpr int kGroups = 2;  // softmax warpgroups, ping-pong over the S buffers
constexpr int kSoftmaxWarps = 4 * kGroups;
constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
constexpr int kKProducerWarp = kSoftmaxWarps;
constexpr int kVProducerWarp = kSoftmaxWarps + 1;
constexpr int kMmaWarp = kSoftmaxWarps + 2;
constexpr int kThreads = 32 * (kSoftmaxWarps + 3);
constexpr int kMaxStages = 4;  // per ring
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;
constexpr uint32_t kColS0 = 128;
constexpr uint32_t kColQ = 448;  // Q tile in TMEM (d/2 columns of bf16 pairs)
constexpr uint32_t kSoftmaxBarrier = 1;  // named barrier of all softmax warps
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Online path: keep the current maximum until a block raises it by more than
// 2^8; probabilities then stay below 256 (safe in fp32 and bf16).
constexpr float kRescaleThreshold = 8.0f;

struct Barriers {
  uint64_t q_full;
  uint64_t q_tmem;  // Q copied into TMEM, the Q slot free (used when Q lives in TMEM)
  uint64_t k_full[kMaxStages];
  uint64_t k_empty[kMaxStages];
  uint64_t v_full[kMaxStages];
  uint64_t v_empty[kMaxStages];
  uint64_t s_full[2];
  uint64_t pa_full[2];  // P of the first (NCH + 1) / 2 chunks of the block in S buffer b
  uint64_t p_full[2];   // P of the remaining chunks
  uint64_t pv_done;
  uint64_t o_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  // Per-row partial sums of the softmax warpgroups, combined in the
  // epilogue: [group][l, lw][row].
  float red[kGroups][2][kQTile];
};

__host__ __device__ constexpr uint32_t s_col(int buf, int Bk) {
  return buf == 0 ? kColS0 : kColS0 + ((uint32_t)(Bk + 31) & ~31u);
}

// Q fits in TMEM next to O and both S buffers.
__host__ __device__ constexpr bool q_fits_tmem(int Bk) { return s_col(1, Bk) + (uint32_t)Bk <= kColQ; }

// Wait with no abort check (used only to drain in-flight copies and MMAs).
__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, unsigned int* err, uint64_t limit) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::global_timer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::global_timer_ns() - t0 > limit) {
      atomicOr(err, kErrWaitDrain);
      return false;
    }
  }
  return true;
}

// One TMA ring (K or V): fills stage j % depth with block j of the visible
// key ranges, after the consumer has released the stage's previous fill.
// Stages below `dedicated` have their own slots; stage `dedicated` (when
// depth > dedicated) is the Q slot, whose first fill waits until Q has been
// copied out of it (`slot_free`).
template <int D>
__device__ __forceinline__ void ring_producer(const CUtensorMap* tm, uint64_t* full, uint64_t* empty, int depth,
                                              int dedicated, uint32_t s0, uint32_t extra_slot, uint64_t* slot_free,
                                              int h, int4 rng, volatile int* abort_flag, const FwdParams& p) {
  const uint32_t kv_bytes = (uint32_t)p.Bk * D * 2;
  const uint32_t half_bytes = (uint32_t)p.Bk * 128;
  int fills[kMaxStages] = {0, 0, 0, 0};
  bool ok = true;
  int j = 0;
  for (int part = 0; part < 2 && ok; ++part) {
    const int start = part == 0 ? rng.x : rng.z;
    const int len = part == 0 ? rng.y : rng.w;
    for (int key = start; key < start + len; key += p.Bk, ++j) {
      const int st = j % depth, u = j / depth;
      bool got = true;
      if (u >= 1)
        got = ptx::mbar_wait<true>(ptx::smem_addr(&empty[st]), (u - 1) & 1, abort_flag, p.err, kErrWaitProducer,
                                   p.limit_ns);
      else if (st >= dedicated)
        got = ptx::mbar_wait<true>(ptx::smem_addr(slot_free), 0, abort_flag, p.err, kErrWaitProducer, p.limit_ns);
      if (!got) {
        ok = false;
        break;
      }
      const uint32_t dst = st < dedicated ? s0 + st * kv_bytes : extra_slot;
      const uint32_t fb = ptx::smem_addr(&full[st]);
      ptx::mbar_arrive_expect_tx(fb, kv_bytes);
#pragma unroll
      for (int half = 0; half < D / 64; ++half)
        ptx::tma_load_3d(dst + half * half_bytes, tm, fb, half * 64, key, h);
      ++fills[st];
    }
  }
  if (!ok) {
    // Let every copy this thread started land before the CTA exits.
    for (int st = 0; st < depth; ++st)
      if (fills[st] > 0) drain_wait(ptx::smem_addr(&full[st]), (fills[st] - 1) & 1, p.err, p.limit_ns);
  }
}

// The MMA issuer: one elected lane of the MMA warp runs the whole loop,
// waits included, while the other lanes wait at the warp's reconvergence.
// An MMA is accepted several instructions ahead of its execution only while
// the issuing thread runs undisturbed: a whole warp that votes on each wait
// and reconverges around an elected lane per batch measured tens of clocks
// of pipe idle per batch.  The region is entered through elect.sync (not a
// lane-index test) so that its arithmetic stays warp-uniform; a lane-index
// branch here measured 30% slower.  Shared-memory descriptors are built once
// per CTA and advanced by constant adds: a tcgen05 shared-memory descriptor
// holds the start address >> 4 in its low 14 bits and every tile here lies
// in the first 256 KB of shared memory, so advancing a tile by b bytes adds
// b >> 4.
template <int D, bool kQTmem, int NCH>
__device__ __forceinline__ void mma_issuer(Barriers& bars, uint32_t tmem, uint32_t q_s, uint32_t k_s0,
                                           uint32_t v_s0, int nblk, bool bounded, const FwdParams& p) {
  volatile int* abort_flag = &bars.abort;
  constexpr uint32_t kBk = NCH * 16;
  constexpr uint32_t kKvBytes = kBk * D * 2;
  constexpr uint32_t kHalfBytes = kBk * 128;  // one 64-column half of a K or V tile
  constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(kQTile, kBk, false);
  constexpr uint32_t idesc_o = ptx::idesc_bf16_f32(kQTile, D, true);
  constexpr int kPa = (NCH + 1) / 2;  // chunks of P released first
  // K (K-major, 128B swizzle): stage base; the stage in the Q slot; Q itself
  // as an A operand; V (MN-major): stage base.
  const uint64_t kdesc0 = ptx::smem_desc_sw128(k_s0, 16, 1024);
  const uint64_t kdesc_qslot = ptx::smem_desc_sw128(q_s, 16, 1024);
  const uint64_t qdesc = ptx::smem_desc_sw128(q_s, 16, 1024);
  const uint64_t vdesc0 = ptx::smem_desc_sw128(v_s0, kHalfBytes, 1024);
  bool ok = ptx::mbar_wait<false>(ptx::smem_addr(&bars.q_full), 0, abort_flag, p.err, kErrWaitMma, p.limit_ns);
  if (ok && kQTmem) {
    // Q into TMEM: one 128-lane x 256-bit copy per 16-column K slice of the
    // 128B-swizzled tile, which lands in the A-operand layout of
    // tcgen05.mma (column c holds elements 2c, 2c+1 of the lane's row).  The
    // pipe runs the copies before the S MMAs issued after them; the commit
    // frees the Q slot for the K ring once the copies are done.
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      ptx::tmem_cp_128x256b(tmem + kColQ + kk * 8, qdesc + (((kk >> 2) * (kQTile * 128) + (kk & 3) * 32) >> 4));
    ptx::mma_commit(ptx::smem_addr(&bars.q_tmem));
  }
  // Ring positions (stage, phase parity) advanced incrementally.
  int ks = 0, kph = 0, vs = 0, vph = 0;
  // S(j) = Q . K(j)^T : M=128, N=Bk, K=d in d/16 MMAs.
  auto issue_s = [&](int j) {
    const uint64_t kdesc = ks < p.kd ? kdesc0 + (uint64_t)(ks * (kKvBytes >> 4)) : kdesc_qslot;
    const uint32_t d_s = tmem + s_col(j & 1, kBk);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint64_t bdesc = kdesc + (((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
      if (kQTmem) {
        ptx::mma_ts(d_s, tmem + kColQ + kk * 8, bdesc, idesc_s, kk > 0 ? 1u : 0u);
      } else {
        const uint64_t adesc = qdesc + (((kk >> 2) * (kQTile * 128) + (kk & 3) * 32) >> 4);
        ptx::mma_ss(d_s, adesc, bdesc, idesc_s, kk > 0 ? 1u : 0u);
      }
    }
    ptx::mma_commit(ptx::smem_addr(&bars.s_full[j & 1]));
    ptx::mma_commit(ptx::smem_addr(&bars.k_empty[ks]));
    if (++ks == p.kst) {
      ks = 0;
      kph ^= 1;
    }
  };
  // The first two S blocks fill both S buffers.
  for (int j = 0; ok && j < 2 && j < nblk; ++j) {
    ok = ptx::mbar_wait<false>(ptx::smem_addr(&bars.k_full[ks]), kph, abort_flag, p.err, kErrWaitMma, p.limit_ns);
    if (ok) issue_s(j);
  }
  // Then one batch per block i: O += P(i) . V(i), followed by S(i+2) into the
  // S buffer that P(i) occupied (the pipe runs them in order, so P(i) is read
  // before it is overwritten), after one wait point for V(i), P(i) and K(i+2).
  for (int i = 0; ok && i < nblk; ++i) {
    const bool more = i + 2 < nblk;
    // P(i) . V(i): M=128, N=d, one K=16 MMA per 16-key chunk; P from TMEM
    // (chunk kk's bf16 P sits in the first 8 columns of its own 16 S
    // columns), V MN-major in shared memory.  The first kPa chunks go as
    // soon as their P is released; the rest, and S(i+2), after the rest of
    // P(i) and K(i+2).
    const uint64_t vdesc = vdesc0 + (uint64_t)(vs * (kKvBytes >> 4));
    const uint32_t a_p = tmem + s_col(i & 1, kBk);
    ok = ptx::mbar_wait<false>(ptx::smem_addr(&bars.v_full[vs]), vph, abort_flag, p.err, kErrWaitMma, p.limit_ns);
    if (ok)
      ok = ptx::mbar_wait<false>(ptx::smem_addr(&bars.pa_full[i & 1]), (i >> 1) & 1, abort_flag, p.err, kErrWaitMma,
                                 p.limit_ns);
    if (!ok) break;
    ptx::tc_fence_after_sync();
#pragma unroll
    for (int kk = 0; kk < kPa; ++kk)
      ptx::mma_ts(tmem + kColO, a_p + kk * 16, vdesc + ((kk * 2048) >> 4), idesc_o, (i > 0 || kk > 0) ? 1u : 0u);
    ok = ptx::mbar_wait<false>(ptx::smem_addr(&bars.p_full[i & 1]), (i >> 1) & 1, abort_flag, p.err, kErrWaitMma,
                               p.limit_ns);
    if (ok && more)
      ok = ptx::mbar_wait<false>(ptx::smem_addr(&bars.k_full[ks]), kph, abort_flag, p.err, kErrWaitMma, p.limit_ns);
    if (!ok) break;
    ptx::tc_fence_after_sync();
#pragma unroll
    for (int kk = kPa; kk < NCH; ++kk)
      ptx::mma_ts(tmem + kColO, a_p + kk * 16, vdesc + ((kk * 2048) >> 4), idesc_o, 1u);
    ptx::mma_commit(ptx::smem_addr(&bars.v_empty[vs]));
    if (!bounded) ptx::mma_commit(ptx::smem_addr(&bars.pv_done));
    if (i == nblk - 1) ptx::mma_commit(ptx::smem_addr(&bars.o_full));
    if (++vs == p.vst) {
      vs = 0;
      vph ^= 1;
    }
    if (more) issue_s(i + 2);
  }
  // Every MMA issued above completes before TMEM is released.
  ptx::mma_commit(ptx::smem_addr(&bars.drain));
  drain_wait(ptx::smem_addr(&bars.drain), 0, p.err, p.limit_ns);
}

// Of the 8 element pairs of a 16-column chunk, this many take 2^x on the FMA
// pipe (ptx::ex2_poly_x2) and the rest on the special-function unit.  At
// d = 128 one exponential per (query, key) pair on the SFU alone takes as
// long as the pair's share of both MMAs, so moving part of them to the FMA
// pipe is what lets the tensor pipe, not the SFU, set the pace.
#ifndef FAS_EX2_POLY_PAIRS
#define FAS_EX2_POLY_PAIRS 0
#endif
constexpr int kPolyPairs = FAS_EX2_POLY_PAIRS;
static_assert(kPolyPairs >= 0 && kPolyPairs <= 8, "pairs per 16-column chunk");

// Spreads the kPolyPairs software pairs evenly over the chunk.
__host__ __device__ constexpr bool poly_pair(int e) { return ((e + 1) * kPolyPairs) / 8 != (e * kPolyPairs) / 8; }

// Softmax of one 16-column chunk held in registers: P = 2^(S*sl2 - m) (two
// lanes per packed instruction), both row sums, P packed to bf16 pairs.
__device__ __forceinline__ void exp_chunk(const uint32_t (&r)[16], uint64_t sl2, uint64_t neg_m, float& l0,
                                          float& l1, float& w0, float& w1, uint32_t (&pk)[8]) {
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    float x0, x1;
    ptx::fma_f32x2(x0, x1, __uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]), sl2, neg_m);
    float p0, p1;
    if (poly_pair(e)) {
      ptx::ex2_poly_x2(p0, p1, x0, x1);
    } else {
      p0 = ptx::ex2(x0);
      p1 = ptx::ex2(x1);
    }
    ptx::add_f32x2(l0, l1, p0, p1);
    pk[e] = ptx::pack_bf16x2(p0, p1);
    ptx::add_f32x2(w0, w1, __uint_as_float(pk[e] << 16), __uint_as_float(pk[e] & 0xFFFF0000u));
  }
}

// Row maximum of the block's raw scores (online path; one chunk at a time
// to keep the fallback's registers low).
__device__ __forceinline__ float block_max(uint32_t sbase, int nch) {
  float mx = -INFINITY;
  for (int c = 0; c < nch; ++c) {
    uint32_t r[16];
    ptx::tmem_ld16(sbase + c * 16, r);
    ptx::tmem_ld_wait(r);
#pragma unroll
    for (int e = 0; e < 16; ++e) mx = fmaxf(mx, __uint_as_float(r[e]));
  }
  return mx;
}

// P for chunks [C0, C0 + N) of an S block.  All TMEM loads of the phase go
// out before any of its stores: a TMEM load issued after a TMEM store of the
// same thread waits for that store, so loading chunk by chunk between stores
// would pay that wait once per chunk.  Each chunk's bf16 P lands in the first
// 8 columns of the chunk's own S columns (already read).
template <int C0, int N>
__device__ __forceinline__ void softmax_phase(uint32_t sbase, uint64_t sl2, uint64_t neg_m, float& l0, float& l1,
                                              float& w0, float& w1) {
  if constexpr (N > 0) {
    uint32_t r[N][16];
#pragma unroll
    for (int u = 0; u < N; ++u) ptx::tmem_ld16(sbase + (C0 + u) * 16, r[u]);
#pragma unroll
    for (int u = 0; u < N; ++u) ptx::tmem_ld_wait(r[u]);
#pragma unroll
    for (int u = 0; u < N; ++u) {
      if (u > 0) ptx::order_after(r[u], w1);
      uint32_t pk[8];
      exp_chunk(r[u], sl2, neg_m, l0, l1, w0, w1, pk);
      ptx::tmem_st8(sbase + (C0 + u) * 16, pk);
    }
  }
}

// Softmax and epilogue for one thread: row `trow` of the tile.
// Bounded heads: warpgroup g takes the blocks j with j % 2 == g, exactly the
// blocks of S buffer g, so the two groups ping-pong and neither talks to the
// other until the epilogue.  Online heads: warpgroup 0 takes every block (the
// running maximum is a serial chain); warpgroup 1 joins for the epilogue.
template <int D, bool kQTmem, int NCH>
__device__ __forceinline__ void softmax_epilogue(Barriers& bars, uint32_t tmem, uint32_t q_s, int warp, int lane,
                                                 int h, int f, int qt, int nblk, bool bounded,
                                                 const FwdParams& p) {
  volatile int* abort_flag = &bars.abort;
  const int g = warp / 4;
  const int trow = (warp % 4) * 32 + lane;
  const uint32_t lane_base = (uint32_t)((warp % 4) * 32) << 16;
  const int row = qt * kQTile + trow;  // row inside the frame
  const bool valid = row < p.T;
  const int64_t grow = (int64_t)h * p.N + (int64_t)f * p.T + row;
  constexpr int nch = NCH;
  constexpr int kPa = (NCH + 1) / 2;  // chunks in the first half of a block
  const uint64_t sl2 = ptx::f32x2(p.scale_log2, p.scale_log2);
  // Row maximum in log2 units of the scaled logits.
  float m_run = -INFINITY;
  if (bounded) m_run = valid ? p.row_bound[grow] * kLog2e : 0.0f;
  // Two row sums, each kept as two interleaved partials: l of the fp32
  // probabilities (for the LSE) and w of the bf16-rounded weights the P.V
  // MMA actually uses (for normalising O, so the output is a convex
  // combination of V rows even when the largest probability is not 1).
  float l0 = 0.f, l1 = 0.f, w0 = 0.f, w1 = 0.f;
  bool ok = true;

  const int j0 = bounded ? g : 0;
  const int jstep = bounded ? kGroups : 1;
  const bool active = bounded || g == 0;
  for (int j = j0; ok && active && j < nblk; j += jstep) {
    const int buf = j & 1;
    const bool got = ptx::mbar_wait(ptx::smem_addr(&bars.s_full[buf]), (j >> 1) & 1, abort_flag, p.err,
                                    kErrWaitSoftmax, p.limit_ns);
    ok = __all_sync(0xffffffffu, got);
    if (!ok) break;
    ptx::tc_fence_after_sync();
    const uint32_t sbase = tmem + lane_base + s_col(buf, NCH * 16);

    if (!bounded) {
      const float mx = block_max(sbase, nch);
      const float cand = mx * p.scale_log2;
      if (j == 0) {
        m_run = cand;
      } else {
        const bool need = cand > m_run + kRescaleThreshold;
        float alpha = 1.0f;
        if (need) {
          alpha = ptx::ex2(m_run - cand);
          m_run = cand;
          l0 *= alpha;
          l1 *= alpha;
          w0 *= alpha;
          w1 *= alpha;
        }
        if (__any_sync(0xffffffffu, need)) {
          // The accumulator may be rescaled only once P(j-1).V(j-1) is done.
          const bool pv = ptx::mbar_wait(ptx::smem_addr(&bars.pv_done), (j - 1) & 1, abort_flag, p.err,
                                         kErrWaitSoftmax, p.limit_ns);
          ok = __all_sync(0xffffffffu, pv);
          if (!ok) break;
          ptx::tc_fence_after_sync();
#pragma unroll 1
          for (int c = 0; c < D / 16; ++c) {
            uint32_t o[16];
            const uint32_t oaddr = tmem + lane_base + kColO + c * 16;
            ptx::tmem_ld16(oaddr, o);
            ptx::tmem_ld_wait(o);
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            ptx::tmem_st16(oaddr, o);
          }
        }
      }
    }

    // P of the block's first chunks is released as soon as it is stored, so
    // that their P.V MMAs run while the rest of the block is exponentiated.
    const uint64_t neg_m = ptx::f32x2(-m_run, -m_run);
    softmax_phase<0, kPa>(sbase, sl2, neg_m, l0, l1, w0, w1);
    ptx::tmem_st_wait();
    ptx::tc_fence_before_sync();
    ptx::mbar_arrive(ptx::smem_addr(&bars.pa_full[buf]));
    softmax_phase<kPa, NCH - kPa>(sbase, sl2, neg_m, l0, l1, w0, w1);
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
  bars.red[g][0][trow] = l0 + l1;
  bars.red[g][1][trow] = w0 + w1;
  ptx::named_barrier_sync(kSoftmaxBarrier, kSoftmaxThreads);
  float l = 0.f, lw = 0.f;
#pragma unroll
  for (int q = 0; q < kGroups; ++q) {
    l += bars.red[q][0][trow];
    lw += bars.red[q][1][trow];
  }
  if (!ok) return;
  ptx::tc_fence_after_sync();
  const float inv = 1.0f / lw;
  uint16_t* orow = p.out + (int64_t)h * p.out_head_stride + ((int64_t)f * p.T + row) * p.out_row_stride;
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
  if (valid && g == 0) p.lse[grow] = (m_run + ptx::lg2(l)) * kLn2;
}

template <int D, int NCH>
__global__ void __launch_bounds__(kThreads, 1)
    attention_fwd(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  constexpr bool kQTmem = q_fits_tmem(NCH * 16);
  extern __shared__ uint8_t smem_raw[];
  __shared__ Barriers bars;
  const uint32_t tiles = (ptx::smem_addr(smem_raw) + 1023u) & ~1023u;  // 128B-swizzle atoms need 1 KB alignment
  const uint32_t q_s = tiles;  // Q tile, then (Q in TMEM) K stage kd
  const uint32_t k_s0 = q_s + p.qslot_bytes;
  const uint32_t v_s0 = k_s0 + (uint32_t)p.kd * p.Bk * D * 2;

  // A CTA of this launch (or an earlier one) already gave up on a wait: do
  // nothing, the host reports FAS_ERR_TIMEOUT.
  if (*reinterpret_cast<volatile unsigned int*>(p.err) != 0u) return;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int4 item = p.work[blockIdx.x];
  const int h = item.x, f = item.y, qt = item.z, nblk = item.w;

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
      ptx::mbar_init(ptx::smem_addr(&bars.pa_full[b]), 32 * 4);  // one warpgroup per block
      ptx::mbar_init(ptx::smem_addr(&bars.p_full[b]), 32 * 4);
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
        ptx::tma_load_4d(q_s + half * (kQTile * 128), &tm_q, ptx::smem_addr(&bars.q_full), half * 64, qt * kQTile, f,
                         h);
      ring_producer<D>(&tm_k, bars.k_full, bars.k_empty, p.kst, p.kd, k_s0, q_s, &bars.q_tmem, h, p.table[f],
                       &bars.abort, p);
      if (bars.abort) drain_wait(ptx::smem_addr(&bars.q_full), 0, p.err, p.limit_ns);
    }
  } else if (warp == kVProducerWarp) {
    if (lane == 0)
      ring_producer<D>(&tm_v, bars.v_full, bars.v_empty, p.vst, p.vst, v_s0, 0, nullptr, h, p.table[f], &bars.abort,
                       p);
  } else if (warp == kMmaWarp) {
    const bool bounded = p.mode == FAS_MODE_BOUNDED || (p.mode == FAS_MODE_AUTO && p.elig[h] != 0);
    if (ptx::elect_one()) mma_issuer<D, kQTmem, NCH>(bars, tmem, q_s, k_s0, v_s0, nblk, bounded, p);
    __syncwarp();
  } else {
    const bool bounded = p.mode == FAS_MODE_BOUNDED || (p.mode == FAS_MODE_AUTO && p.elig[h] != 0);
    softmax_epilogue<D, kQTmem, NCH>(bars, tmem, q_s, warp, lane, h, f, qt, nblk, bounded, p);
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

constexpr size_t kSmemLimit = 232448;  // opt-in shared memory per block (sm_100 family)

template <int D, int NCH>
cudaError_t launch_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, FwdParams p, int grid,
                     cudaStream_t st) {
  // Shared memory: [Q slot][kd K stages][vst V stages].  With Q in TMEM the
  // Q slot (sized for a K stage too) becomes K stage kd once Q is copied.
  constexpr bool kQTmem = q_fits_tmem(NCH * 16);
  const size_t kv_bytes = (size_t)p.Bk * D * 2;
  const size_t q_bytes = (size_t)kQTile * D * 2;
  const size_t qslot = kQTmem ? (kv_bytes > q_bytes ? kv_bytes : q_bytes) : q_bytes;
  const size_t fixed = 1024 + qslot + sizeof(Barriers) + 256;
  int n = (int)((kSmemLimit - fixed) / kv_bytes);
  if (n > 2 * kMaxStages - 1) n = 2 * kMaxStages - 1;
  if (n < 4) return cudaErrorInvalidValue;
  int kd = n / 2;
  if (kd > kMaxStages - 1) kd = kMaxStages - 1;
  int vst = n - kd;
  if (vst > kMaxStages) vst = kMaxStages;
  p.kd = kd;
  p.kst = kd + (kQTmem ? 1 : 0);
  p.vst = vst;
  p.qslot_bytes = (uint32_t)qslot;
  const size_t smem = 1024 + qslot + (size_t)(kd + vst) * kv_bytes;
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
