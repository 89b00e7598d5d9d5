// Shared pieces of the tcgen05 attention kernels (the frame-aligned kernel
// and the splash-style ablation): warp roles, TMEM columns, the barrier
// block, the TMA ring producer, the MMA issuer and the exponentiation of S
// chunks held in registers.  See attention.cu for the design.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fas.h"
#include "internal.h"
#include "kernels.h"
#include "ptx.cuh"

namespace fas {
namespace core {

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
// Online path: keep the current maximum until a block raises it by more
// than 2^32, so every probability stays below 2^32.  bf16 keeps the same
// relative precision at any scale, and with at most 2^31 keys the fp32 sums
// stay below 2^63 |v| (far from the fp32 range), so a large threshold costs
// nothing numerically; it makes the rescale of O (which must wait for the
// previous block's P.V) rare.  With 32 rows per warp and a threshold of 2^8,
// some row of a warp raised its maximum in most early blocks.
constexpr float kRescaleThreshold = 32.0f;

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
  uint64_t mchain_bar[2];  // online heads: block j's running maximum published in mchain[j % 2]
  uint32_t tmem_base;
  int abort;
  int skip;  // an earlier CTA already recorded an error: this CTA does nothing
  // Online heads: the running row maximum after block j (log2 units), passed
  // from the group that processed block j to the one processing block j+1.
  float mchain[2][kQTile];
  // Per-row partial sums of the softmax warpgroups, combined in the
  // epilogue: [group][l, lw][row].
  float red[kGroups][2][kQTile];
};

__host__ __device__ constexpr uint32_t s_col(int buf, int Bk) {
  return buf == 0 ? kColS0 : kColS0 + ((uint32_t)(Bk + 31) & ~31u);
}

// Q lives in TMEM next to O and both S buffers for every block size the
// planner allows, so S = Q.K^T always reads its A operand from TMEM.
static_assert(s_col(1, kMaxBlockK) + (uint32_t)kMaxBlockK <= kColQ, "Q must fit in TMEM beside O and S");

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
template <int D, int NCH>
__device__ __forceinline__ void mma_issuer(Barriers& bars, uint32_t tmem, uint32_t q_s, uint32_t k_s0,
                                           uint32_t v_s0, int nblk, bool bounded, const FwdParams& p) {
  volatile int* abort_flag = &bars.abort;
  constexpr uint32_t kBk = NCH * 16;
  constexpr uint32_t kKvBytes = kBk * D * 2;
  constexpr uint32_t kHalfBytes = kBk * 128;  // one 64-column half of a K or V tile
  constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(kQTile, kBk, false);
  constexpr uint32_t idesc_o = ptx::idesc_bf16_f32(kQTile, D, true);
  constexpr int kPa = (NCH + 1) / 2;  // chunks of P released first
  // K (K-major, 128B swizzle): stage base; the stage in the Q slot; the Q
  // tile (copied into TMEM); V (MN-major): stage base.
  const uint64_t kdesc0 = ptx::smem_desc_sw128(k_s0, 16, 1024);
  const uint64_t kdesc_qslot = ptx::smem_desc_sw128(q_s, 16, 1024);
  const uint64_t qdesc = ptx::smem_desc_sw128(q_s, 16, 1024);
  const uint64_t vdesc0 = ptx::smem_desc_sw128(v_s0, kHalfBytes, 1024);
  bool ok = ptx::mbar_wait<false>(ptx::smem_addr(&bars.q_full), 0, abort_flag, p.err, kErrWaitMma, p.limit_ns);
  if (ok) {
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
  // S(j) = Q . K(j)^T (from column 16 c0 on, with the matching rows of the
  // K tile): M=128, N set by idesc, K=d in d/16 MMAs.
  auto s_part = [&](int j, int c0, uint32_t idesc) {
    const uint64_t kdesc = (ks < p.kd ? kdesc0 + (uint64_t)(ks * (kKvBytes >> 4)) : kdesc_qslot) +
                           (uint64_t)((c0 * 16 * 128) >> 4);
    const uint32_t d_s = tmem + s_col(j & 1, kBk) + c0 * 16;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint64_t bdesc = kdesc + (((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
      ptx::mma_ts(d_s, tmem + kColQ + kk * 8, bdesc, idesc, kk > 0 ? 1u : 0u);
    }
  };
  auto s_done = [&](int j) {
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
    if (!ok) break;
    s_part(j, 0, idesc_s);
    s_done(j);
  }
  // Then one batch per block i: O += P(i) . V(i), followed by S(i+2) into the
  // S buffer that P(i) occupied (the pipe runs them in order, so P(i) is read
  // before it is overwritten), after one wait point for V(i), P(i) and K(i+2).
  // (Issuing the columns of S(i+2) over P(i)'s first half right after that
  // half's P.V, before the rest of P(i) is released, measured 4% slower on
  // the 720p chunk.)
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
    if (more) {
      s_part(i + 2, 0, idesc_s);
      s_done(i + 2);
    }
  }
  // Every MMA issued above completes before TMEM is released.
  ptx::mma_commit(ptx::smem_addr(&bars.drain));
  drain_wait(ptx::smem_addr(&bars.drain), 0, p.err, p.limit_ns);
}

// Softmax of one 16-column chunk held in registers: P = 2^(S*sl2 - m) (two
// lanes per packed instruction), both row sums, P packed to bf16 pairs.
__device__ __forceinline__ void exp_chunk(const uint32_t (&r)[16], uint64_t sl2, uint64_t neg_m, float& l0,
                                          float& l1, float& w0, float& w1, uint32_t (&pk)[8]) {
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    float x0, x1;
    ptx::fma_f32x2(x0, x1, __uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]), sl2, neg_m);
    const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
    ptx::add_f32x2(l0, l1, p0, p1);
    pk[e] = ptx::pack_bf16x2(p0, p1);
    ptx::add_f32x2(w0, w1, __uint_as_float(pk[e] << 16), __uint_as_float(pk[e] & 0xFFFF0000u));
  }
}

// Exponentiates chunks [C0, C0 + N) of an S block already loaded into r and
// stores each chunk's bf16 P into the first 8 columns of the chunk's own S
// columns (already read).
template <int C0, int N, int M>
__device__ __forceinline__ void exp_store(const uint32_t (&r)[M][16], uint32_t sbase, uint64_t sl2, uint64_t neg_m,
                                          float& l0, float& l1, float& w0, float& w1) {
#pragma unroll
  for (int u = 0; u < N; ++u) {
    uint32_t x[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) x[e] = r[u][e];
    if (u > 0) ptx::order_after(x, w1);
    uint32_t pk[8];
    exp_chunk(x, sl2, neg_m, l0, l1, w0, w1, pk);
    ptx::tmem_st8(sbase + (C0 + u) * 16, pk);
  }
}

// Loads chunks [C0, C0 + N) of an S block.  All TMEM loads of a phase go out
// before any of its stores: a TMEM load issued after a TMEM store of the
// same thread waits for that store, so loading chunk by chunk between stores
// would pay that wait once per chunk.
template <int C0, int N, int M>
__device__ __forceinline__ void load_chunks(uint32_t sbase, uint32_t (&r)[M][16]) {
#pragma unroll
  for (int u = 0; u < N; ++u) ptx::tmem_ld16(sbase + (C0 + u) * 16, r[u]);
#pragma unroll
  for (int u = 0; u < N; ++u) ptx::tmem_ld_wait(r[u]);
}

// Element mask of the S chunks: NoMask keeps every score (every block the
// frame-aligned kernel visits is wholly visible); a mask with apply() sets
// hidden scores to -inf before the maximum and the exponentials.
struct NoMask {
  static constexpr bool kActive = false;
  template <int M>
  __device__ __forceinline__ void apply(uint32_t (&)[M][16], int, int) const {}
};

// P for chunks [C0, C0 + N) of an S block with a fixed maximum.
template <int C0, int N, class Mask = NoMask>
__device__ __forceinline__ void softmax_phase(uint32_t sbase, uint64_t sl2, uint64_t neg_m, float& l0, float& l1,
                                              float& w0, float& w1, const Mask& mask = Mask()) {
  if constexpr (N > 0) {
    uint32_t r[N][16];
    load_chunks<C0, N>(sbase, r);
    if constexpr (Mask::kActive) mask.apply(r, C0, N);
    exp_store<C0, N>(r, sbase, sl2, neg_m, l0, l1, w0, w1);
  }
}

// Row maximum of chunks [C0, C0 + N) of an S block (raw scores).
template <int C0, int N, class Mask>
__device__ __forceinline__ float chunk_max(uint32_t sbase, const Mask& mask) {
  float mx = -INFINITY;
  if constexpr (N > 0) {
    uint32_t r[N][16];
    load_chunks<C0, N>(sbase, r);
    if constexpr (Mask::kActive) mask.apply(r, C0, N);
#pragma unroll
    for (int u = 0; u < N; ++u)
#pragma unroll
      for (int e = 0; e < 16; ++e) mx = fmaxf(mx, __uint_as_float(r[u][e]));
  }
  return mx;
}

// Per-thread state of one row's softmax: the maximum this thread's sums are
// taken against (log2 units of the scaled logits; fixed for bounded heads)
// and its two row sums, each as two interleaved partials.
struct OnlineRow {
  float m_run;
  float l0, l1, w0, w1;
};

// Online softmax of block j for the warpgroup that owns it.  Online heads
// ping-pong over the blocks like bounded ones (group j % 2 takes block j), so
// one group's exponentials overlap the other's; the running maximum is the
// only serial link.  After its max pass over S(j) the group waits (bounded)
// for block j-1's maximum from the other group, applies the conditional
// rescale rule, and publishes block j's maximum in mchain[j % 2].  Each
// group keeps its sums against the maximum it last used and brings them to
// a new one when the chain raises it; when block j raises the maximum, this
// group rescales the whole row of O once P(j-1).V(j-1) is done (before P(j)
// is released, so P(j).V(j) accumulates onto the rescaled O).  Returns
// false when a wait gave up.
template <int D, int NCH, class Mask = NoMask>
__device__ __forceinline__ bool online_block(Barriers& bars, uint32_t tmem, uint32_t lane_base, uint32_t sbase,
                                             int j, int trow, uint64_t sl2, OnlineRow& st, const FwdParams& p,
                                             const Mask& mask = Mask()) {
  volatile int* abort_flag = &bars.abort;
  constexpr int kPa = (NCH + 1) / 2;
  const int buf = j & 1;
  const float mx = fmaxf(chunk_max<0, kPa>(sbase, mask), chunk_max<kPa, NCH - kPa>(sbase, mask));
  const float cand = mx * p.scale_log2;
  float m_prev = -INFINITY;
  if (j > 0) {
    const bool got = ptx::mbar_wait(ptx::smem_addr(&bars.mchain_bar[buf ^ 1]), ((j - 1) >> 1) & 1, abort_flag,
                                    p.err, kErrWaitSoftmax, p.limit_ns);
    if (!__all_sync(0xffffffffu, got)) return false;
    m_prev = bars.mchain[buf ^ 1][trow];
  }
  // Keep the maximum until a block raises it by more than the threshold
  // (then every probability stays below 2^threshold).
  const bool raise = j > 0 && cand > m_prev + kRescaleThreshold;
  const float m_new = (j == 0 || raise) ? cand : m_prev;
  bars.mchain[buf][trow] = m_new;
  ptx::mbar_arrive(ptx::smem_addr(&bars.mchain_bar[buf]));
  if (st.m_run != m_new) {
    // This group's sums were taken against an older (smaller) maximum.
    const float a = st.m_run == -INFINITY ? 0.f : ptx::ex2(st.m_run - m_new);
    st.l0 *= a;
    st.l1 *= a;
    st.w0 *= a;
    st.w1 *= a;
    st.m_run = m_new;
  }
  if (__any_sync(0xffffffffu, raise)) {
    // O holds P(0..j-1).V against m_prev: rescale it once P(j-1).V(j-1) is
    // done (the pipe has finished everything before S(j), so pv_done is at
    // most one phase behind and the parity wait is unambiguous).
    const bool pv = ptx::mbar_wait(ptx::smem_addr(&bars.pv_done), (j - 1) & 1, abort_flag, p.err,
                                   kErrWaitSoftmax, p.limit_ns);
    if (!__all_sync(0xffffffffu, pv)) return false;
    ptx::tc_fence_after_sync();
    const float alpha = raise ? ptx::ex2(m_prev - m_new) : 1.0f;
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
  // A row that has seen no visible key yet (masked scores only) has an
  // infinite maximum; its scores are all -inf and its P all zero.
  const float m = m_new == -INFINITY ? 0.0f : m_new;
  const uint64_t neg_m = ptx::f32x2(-m, -m);
  softmax_phase<0, kPa>(sbase, sl2, neg_m, st.l0, st.l1, st.w0, st.w1, mask);
  ptx::tmem_st_wait();
  ptx::tc_fence_before_sync();
  ptx::mbar_arrive(ptx::smem_addr(&bars.pa_full[buf]));
  softmax_phase<kPa, NCH - kPa>(sbase, sl2, neg_m, st.l0, st.l1, st.w0, st.w1, mask);
  ptx::tmem_st_wait();
  ptx::tc_fence_before_sync();
  ptx::mbar_arrive(ptx::smem_addr(&bars.p_full[buf]));
  return true;
}

// Brings a group's sums to the row's final maximum m_final (online heads:
// the maximum after the last block, published in mchain).
__device__ __forceinline__ void settle_sums(OnlineRow& st, float m_final) {
  if (st.m_run != m_final) {
    const float a = st.m_run == -INFINITY ? 0.f : ptx::ex2(st.m_run - m_final);
    st.l0 *= a;
    st.l1 *= a;
    st.w0 *= a;
    st.w1 *= a;
    st.m_run = m_final;
  }
}

// Shared-memory plan of one launch: [Q slot][kd K stages][vst V stages].  The
// Q slot (sized for a K stage too) becomes K stage kd once Q is copied into
// TMEM.  Returns the dynamic shared-memory bytes, or 0 when fewer than four
// K/V stages fit.
inline size_t ring_plan(int D, int Bk, FwdParams* p) {
  constexpr size_t kSmemLimit = 232448;  // opt-in shared memory per block (sm_100 family)
  const size_t kv_bytes = (size_t)Bk * D * 2;
  const size_t q_bytes = (size_t)kQTile * D * 2;
  const size_t qslot = kv_bytes > q_bytes ? kv_bytes : q_bytes;
  const size_t fixed = 1024 + qslot + sizeof(Barriers) + 256;
  int n = (int)((kSmemLimit - fixed) / kv_bytes);
  if (n > 2 * kMaxStages - 1) n = 2 * kMaxStages - 1;
  if (n < 4) return 0;
  int kd = n / 2;
  if (kd > kMaxStages - 1) kd = kMaxStages - 1;
  int vst = n - kd;
  if (vst > kMaxStages) vst = kMaxStages;
  p->kd = kd;
  p->kst = kd + 1;
  p->vst = vst;
  p->qslot_bytes = (uint32_t)qslot;
  return 1024 + qslot + (size_t)(kd + vst) * kv_bytes;
}

}  // namespace core
}  // namespace fas
