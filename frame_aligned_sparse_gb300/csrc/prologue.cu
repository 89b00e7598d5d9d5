// The attention prologue: RMSNorm -> QKV projection -> rotary embedding ->
// head packing, in one kernel that writes q, k and v in the layout their
// consumer reads.
//
// "HeyGen x Google Cloud: Avatar IV on TPU", section "Layout Is the ABI" and
// Fig. 5: attention's inputs are produced by normalization, rotary
// embeddings, projections and head packing; fusing that chain into one
// kernel that writes exactly the layout the next step wants makes the
// kernel's output buffer the consumer's input buffer, with no repack.
//
// For token n with hidden state x_n [C]:
//   y_n = (x_n / sqrt(mean(x_n^2) + eps) * gamma) W^T        (W [3*H*d, C])
//   q, k: each head's d values rotated pair by pair, (i, i + d/2) by the
//         angle of (n, i): (a, b) -> (a c - b s, a s + b c); v as projected.
// The norm scale is folded into the weight once (W' = gamma * W, per input
// feature, rounded to bf16: fas_prologue_fold_weights), so the contraction
// runs on the raw hidden states and each row is scaled by its 1/rms in the
// epilogue (the two are equal in exact arithmetic).
//
// One CTA per (128-token panel, part q|k|v).  The CTA sweeps the part's H*d
// output features in tiles of TN = 256 (or 128) on the tensor cores:
//   warp 0     TMA producer: x tile [128 x 64] and W' tile [TN x 64] per
//              K-step of 64 (128B-swizzled, K-major) into a 4-stage ring;
//              the CTAs of a cluster (consecutive panels of one part) load
//              a share of each W' tile and multicast it to all of them;
//   warp 1     TMEM allocator and MMA issuer (one elected lane):
//              tcgen05.mma kind::f16, M = 128, N = TN, both operands from
//              shared memory, fp32 accumulators in TMEM, two accumulator
//              buffers so one tile's epilogue overlaps the next tile's MMAs;
//   warps 2-5  one thread per row: during the first tile, the row's sum of
//              squares straight from the staged x tiles (the 128B swizzle
//              only permutes 16-byte pieces inside a row); then per tile the
//              epilogue: TMEM -> registers, times 1/rms, rotary (q, k),
//              round to bf16, stores in the output layout.
//
// Optionally the k part also writes, per head, the column sums of the
// rounded keys over each group of 16 tokens, the statistic the prepass's
// key phase would otherwise compute by reading k back ("Unchaining the
// Softmax": the mean key and the per-frame key sums).  Frames start at
// multiples of 16 tokens, so no group crosses a frame.  A group is the 16
// rows of a half-warp; its column sums are reduced by recursive halving
// across the half-warp (four exchange steps, 30 shuffles per 32 columns),
// after which each lane holds two columns' sums.

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

#ifndef FAS_PROLOGUE_CLUSTER
#define FAS_PROLOGUE_CLUSTER 2
#endif
constexpr int kClusterP = FAS_PROLOGUE_CLUSTER;  // CTAs that share each W' tile (TMA multicast)
#ifndef FAS_PROLOGUE_KEEP_X
#define FAS_PROLOGUE_KEEP_X 1
#endif
#ifndef FAS_PROLOGUE_KEEP_W
#define FAS_PROLOGUE_KEEP_W 1
#endif
#ifndef FAS_PROLOGUE_STREAM_OUT
#define FAS_PROLOGUE_STREAM_OUT 1
#endif
constexpr int kThreadsP = 192;
constexpr int kStagesP = 4;
constexpr int kKStep = 64;   // K elements per stage: one 128-byte swizzle row of bf16
constexpr int kRows = 128;   // tokens per panel (MMA M)

struct PBars {
  uint64_t full[kStagesP];
  uint64_t empty[kStagesP];   // the MMAs of the stage are done
  uint64_t rowsum[kStagesP];  // the row-sum warps have read the stage's x tile (first tile only)
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Recursive halving across the lanes of a half-warp: on entry v[0 .. W) are
// this lane's W columns; afterwards v[0 .. W/2) are column sums over lanes
// l and l ^ O of the half that this lane keeps (the upper half of the
// columns when bit O of its lane index is set).
template <int W, int O>
__device__ __forceinline__ void halve(float (&v)[32], int lane) {
  const bool up = (lane & O) != 0;
#pragma unroll
  for (int i = 0; i < W / 2; ++i) {
    const float send = up ? v[i] : v[i + W / 2];
    const float keep = up ? v[i + W / 2] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
  }
}

// Element offset of (head h, token n) in the output layout.
__device__ __forceinline__ int64_t out_offset(const PrologueParams& p, int h, int64_t n) {
  const int D = p.head_dim;
  if (p.layout == FAS_LAYOUT_NHD) return (int64_t)h * D + n * (int64_t)p.heads * D;
  if (p.layout == FAS_LAYOUT_A2A) {
    const int hg = p.heads / p.groups, hp = hg / p.ranks;
    const int g = h / hg, r = (h % hg) / hp, j = h % hp;
    return ((int64_t)(g * p.ranks + r) * p.tokens + n) * hp * D + (int64_t)j * D;
  }
  return ((int64_t)h * p.tokens + n) * D;  // FAS_LAYOUT_HND
}

template <int D, int TN, int CL>
__global__ void __launch_bounds__(kThreadsP, 1)
    prologue_qkv(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                 const PrologueParams p) {
  constexpr uint32_t kABytes = kRows * kKStep * 2;
  constexpr uint32_t kBBytes = TN * kKStep * 2;
  constexpr uint32_t kStageBytes = kABytes + kBBytes;
  constexpr uint32_t kAccCols = TN;
  constexpr uint32_t kTmemCols = 2 * TN;
  constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kRows, TN, false);
  extern __shared__ uint8_t smem_raw[];
  __shared__ PBars bars;
  const uint32_t ring = (ptx::smem_addr(smem_raw) + 1023u) & ~1023u;
  uint8_t* const ring_ptr = smem_raw + (ring - ptx::smem_addr(smem_raw));

  // The CTAs of a cluster take consecutive panels of the same part, so they
  // need the same W' tiles: each loads 1/CL of every W' tile and multicasts
  // it to all of them, and each one's MMAs free a stage in all of them.
  // (No early exit here: a CTA of a cluster must take part in the whole
  // exchange; the error word is looked at by the bounded waits.)
  const uint32_t rank = CL > 1 ? ptx::cluster_ctarank() : 0u;
  constexpr uint16_t kMask = (uint16_t)((1u << CL) - 1u);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int cid = blockIdx.x / CL;
  const int part = cid % 3, panel = (cid / 3) * CL + (int)rank;
  const int ksteps = p.width / kKStep;
  const int ncol = p.heads * D / TN;
  volatile int* abort_flag = &bars.abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesP; ++s) {
      ptx::mbar_init(ptx::smem_addr(&bars.full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&bars.empty[s]), CL);  // the MMAs of every CTA of the cluster
      ptx::mbar_init(ptx::smem_addr(&bars.rowsum[s]), kRows);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_addr(&bars.acc_full[b]), 1);
      ptx::mbar_init(ptx::smem_addr(&bars.acc_empty[b]), kRows);
    }
    ptx::mbar_init(ptx::smem_addr(&bars.drain), 1);
    bars.abort = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(&bars.tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  if (CL > 1) ptx::cluster_sync();  // every CTA's barriers exist before any multicast reaches them
  const uint32_t tmem = bars.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      // Producer: fill f goes to stage f % S after the stage's previous fill
      // is consumed by the MMAs of every CTA of the cluster (and, for
      // first-tile fills, by this CTA's row sums).
      // x (each panel read once per column tile) and W' (read by every
      // panel of the part) stay in L2 ahead of the q, k, v stream.
      const uint64_t keep_x = FAS_PROLOGUE_KEEP_X ? ptx::policy_evict_last() : ptx::policy_evict_normal();
      const uint64_t keep_w = FAS_PROLOGUE_KEEP_W ? ptx::policy_evict_last() : ptx::policy_evict_normal();
      int fill = 0;
      bool ok = true;
      for (int n = 0; ok && n < ncol; ++n)
        for (int kk = 0; ok && kk < ksteps; ++kk, ++fill) {
          const int s = fill % kStagesP, u = fill / kStagesP;
          if (u >= 1) {
            ok = ptx::mbar_wait<true>(ptx::smem_addr(&bars.empty[s]), (u - 1) & 1, abort_flag, p.err,
                                      kErrWaitProducer, p.limit_ns);
            const int prev = fill - kStagesP;
            if (ok && prev < ksteps)
              ok = ptx::mbar_wait<true>(ptx::smem_addr(&bars.rowsum[s]), (prev / kStagesP) & 1, abort_flag, p.err,
                                        kErrWaitProducer, p.limit_ns);
            if (!ok) break;
          }
          const uint32_t dst = ring + s * kStageBytes;
          const uint32_t fb = ptx::smem_addr(&bars.full[s]);
          ptx::mbar_arrive_expect_tx(fb, kStageBytes);
          ptx::tma_load_2d_hint(dst, &tm_x, fb, kk * kKStep, panel * kRows, keep_x);
          if (CL == 1)
            ptx::tma_load_2d_hint(dst + kABytes, &tm_w, fb, kk * kKStep, part * p.heads * D + n * TN, keep_w);
          else
            ptx::tma_load_2d_multicast_hint(dst + kABytes + rank * (kBBytes / CL), &tm_w, fb, kk * kKStep,
                                            part * p.heads * D + n * TN + (int)rank * (TN / CL), kMask, keep_w);
        }
      if (!ok) {
        // Let the copies already started land before the CTA exits (a
        // bounded wait that ignores the abort flag).
        for (int f = (fill > kStagesP ? fill - kStagesP : 0); f < fill; ++f) {
          const uint32_t bar = ptx::smem_addr(&bars.full[f % kStagesP]);
          const uint64_t t0 = ptx::global_timer_ns();
          while (!ptx::mbar_try_wait(bar, (f / kStagesP) & 1)) {
            if (ptx::global_timer_ns() - t0 > p.limit_ns) {
              atomicOr(p.err, kErrWaitDrain);
              break;
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    if (ptx::elect_one()) {
      int fill = 0;
      bool ok = true;
      for (int n = 0; ok && n < ncol; ++n) {
        const int b = n & 1;
        if (n >= 2)
          ok = ptx::mbar_wait<false>(ptx::smem_addr(&bars.acc_empty[b]), ((n >> 1) - 1) & 1, abort_flag, p.err,
                                     kErrWaitMma, p.limit_ns);
        for (int kk = 0; ok && kk < ksteps; ++kk, ++fill) {
          const int s = fill % kStagesP;
          ok = ptx::mbar_wait<false>(ptx::smem_addr(&bars.full[s]), (fill / kStagesP) & 1, abort_flag, p.err,
                                     kErrWaitMma, p.limit_ns);
          if (!ok) break;
          ptx::tc_fence_after_sync();
          const uint32_t a_s = ring + s * kStageBytes;
          const uint64_t adesc = ptx::smem_desc_sw128(a_s, 16, 1024);
          const uint64_t bdesc = ptx::smem_desc_sw128(a_s + kABytes, 16, 1024);
#pragma unroll
          for (int k = 0; k < kKStep / 16; ++k)
            ptx::mma_ss(tmem + b * kAccCols, adesc + (uint64_t)(k * 2), bdesc + (uint64_t)(k * 2), kIdesc,
                        (kk > 0 || k > 0) ? 1u : 0u);
          if (CL == 1)
            ptx::mma_commit(ptx::smem_addr(&bars.empty[s]));
          else
            ptx::mma_commit_multicast(ptx::smem_addr(&bars.empty[s]), kMask);
        }
        if (ok) ptx::mma_commit(ptx::smem_addr(&bars.acc_full[b]));
      }
      ptx::mma_commit(ptx::smem_addr(&bars.drain));
      ptx::mbar_wait<false>(ptx::smem_addr(&bars.drain), 0, abort_flag, p.err, kErrWaitDrain, p.limit_ns);
    }
    __syncwarp();
  } else {
    // Epilogue warps: warp w reads TMEM lanes 32 (w % 4) .. + 31.
    const int row = (warp % 4) * 32 + lane;
    const int64_t token = (int64_t)panel * kRows + row;
    const bool valid = token < p.tokens;
    const uint32_t lane_base = (uint32_t)((warp % 4) * 32) << 16;
    bool ok = true;
    // Sum of squares of the row's hidden state, from the first tile's x
    // stages (fills 0 .. ksteps-1).
    float ss0 = 0.f, ss1 = 0.f;
    for (int kk = 0; kk < ksteps; ++kk) {
      const int s = kk % kStagesP;
      const bool got = ptx::mbar_wait<false>(ptx::smem_addr(&bars.full[s]), (kk / kStagesP) & 1, abort_flag, p.err,
                                             kErrWaitSoftmax, p.limit_ns);
      ok = __all_sync(0xffffffffu, got);
      if (!ok) break;
      const uint4* src = reinterpret_cast<const uint4*>(ring_ptr + s * kStageBytes + row * 128);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        // The row's eight pieces in the order of the swizzled rows' bank
        // groups, so that eight consecutive rows read eight different ones.
        const uint4 v = src[c ^ (row & 7)];
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          ss0 = fmaf(bf16_lo(w4[e]), bf16_lo(w4[e]), ss0);
          ss1 = fmaf(bf16_hi(w4[e]), bf16_hi(w4[e]), ss1);
        }
      }
      // The stage goes back to the producer, whose next TMA write (async
      // proxy) must not land before these shared-memory reads (generic
      // proxy): the arrive waits for the values read, and the proxy fence
      // orders the reads before the async proxy's write.
      ptx::consume(ss0, ss1);
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(ptx::smem_addr(&bars.rowsum[s]));
    }
    const float rstd = rsqrtf((ss0 + ss1) / (float)p.width + p.eps);
    // q, k, v: written once here, read by later kernels.
    const uint64_t stream = FAS_PROLOGUE_STREAM_OUT ? ptx::policy_evict_first() : ptx::policy_evict_normal();
    uint16_t* const out = static_cast<uint16_t*>(part == 0 ? p.q : part == 1 ? p.k : p.v);
    // Key sums: this half-warp's group of 16 tokens.
    const bool sums = part == 1 && p.key_sums != nullptr;
    const int64_t groups16 = p.tokens / 16;
    const int64_t grp = ((int64_t)panel * kRows + (warp % 4) * 32 + (lane & 16)) / 16;
    const float* const ctab = p.cos_tab + (valid ? token : 0) * (D / 2);
    const float* const stab = p.sin_tab + (valid ? token : 0) * (D / 2);
    for (int n = 0; ok && n < ncol; ++n) {
      const int b = n & 1;
      const bool got = ptx::mbar_wait<false>(ptx::smem_addr(&bars.acc_full[b]), (n >> 1) & 1, abort_flag, p.err,
                                             kErrWaitSoftmax, p.limit_ns);
      ok = __all_sync(0xffffffffu, got);
      if (!ok) break;
      ptx::tc_fence_after_sync();
#pragma unroll 1
      for (int hh = 0; hh < TN / D; ++hh) {
        const int head = n * (TN / D) + hh;
        uint16_t* const dst = out + out_offset(p, head, token);
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          // Columns i = 16c .. 16c+15 of the head and their rotation partners
          // i + d/2.
          uint32_t a[16], bb[16];
          const uint32_t col = b * kAccCols + hh * D + c * 16;
          ptx::tmem_ld16(tmem + lane_base + col, a);
          ptx::tmem_ld16(tmem + lane_base + col + D / 2, bb);
          ptx::tmem_ld_wait(a);
          ptx::tmem_ld_wait(bb);
          float lo[16], hi[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            lo[e] = __uint_as_float(a[e]) * rstd;
            hi[e] = __uint_as_float(bb[e]) * rstd;
          }
          if (part < 2) {
            float cs[16], sn[16];
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {
              const float4 c4 = reinterpret_cast<const float4*>(ctab + c * 16)[e4];
              const float4 s4 = reinterpret_cast<const float4*>(stab + c * 16)[e4];
              cs[4 * e4] = c4.x; cs[4 * e4 + 1] = c4.y; cs[4 * e4 + 2] = c4.z; cs[4 * e4 + 3] = c4.w;
              sn[4 * e4] = s4.x; sn[4 * e4 + 1] = s4.y; sn[4 * e4 + 2] = s4.z; sn[4 * e4 + 3] = s4.w;
            }
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float x0 = lo[e], x1 = hi[e];
              lo[e] = x0 * cs[e] - x1 * sn[e];
              hi[e] = fmaf(x0, sn[e], x1 * cs[e]);
            }
          }
          uint32_t pl[8], ph[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            pl[e] = ptx::pack_bf16x2(lo[2 * e], lo[2 * e + 1]);
            ph[e] = ptx::pack_bf16x2(hi[2 * e], hi[2 * e + 1]);
          }
          if (valid) {
            uint4* d0 = reinterpret_cast<uint4*>(dst + c * 16);
            uint4* d1 = reinterpret_cast<uint4*>(dst + D / 2 + c * 16);
            ptx::st_global_hint(d0, make_uint4(pl[0], pl[1], pl[2], pl[3]), stream);
            ptx::st_global_hint(d0 + 1, make_uint4(pl[4], pl[5], pl[6], pl[7]), stream);
            ptx::st_global_hint(d1, make_uint4(ph[0], ph[1], ph[2], ph[3]), stream);
            ptx::st_global_hint(d1 + 1, make_uint4(ph[4], ph[5], ph[6], ph[7]), stream);
          }
          if (sums) {
            // The 16 rows of this half-warp, columns 16c .. 16c+15 (v[0 .. 16))
            // and d/2 + 16c .. (v[16 .. 32)), as rounded and stored; rows
            // past the last token count as zero.
            float v[32];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              v[2 * e] = valid ? bf16_lo(pl[e]) : 0.f;
              v[2 * e + 1] = valid ? bf16_hi(pl[e]) : 0.f;
              v[16 + 2 * e] = valid ? bf16_lo(ph[e]) : 0.f;
              v[16 + 2 * e + 1] = valid ? bf16_hi(ph[e]) : 0.f;
            }
            halve<32, 8>(v, lane);
            halve<16, 4>(v, lane);
            halve<8, 2>(v, lane);
            halve<4, 1>(v, lane);
            // Lane l of the half holds columns 2 (l % 16) and 2 (l % 16) + 1
            // of the 32.
            const int li = lane & 15;
            const int col = (li < 8 ? 0 : D / 2) + c * 16 + 2 * (li & 7);
            if (grp < groups16)
              *reinterpret_cast<float2*>(p.key_sums + ((int64_t)head * groups16 + grp) * D + col) =
                  make_float2(v[0], v[1]);
          }
        }
      }
      // The accumulator's values are in registers and stored: the MMAs of
      // tile n + 2 may overwrite it.
      ptx::tc_fence_before_sync();
      ptx::mbar_arrive(ptx::smem_addr(&bars.acc_empty[b]));
    }
  }

  ptx::tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
  // A CTA's shared memory must outlive the other CTAs' multicasts and
  // commits into it.
  if (CL > 1) ptx::cluster_sync();
}

// W'[o, c] = bf16(W[o, c] * gamma[c]), rounded to nearest even.
__global__ void fold_weights(const uint16_t* __restrict__ w, const float* __restrict__ gamma,
                             uint16_t* __restrict__ out, int64_t rows, int width) {
  const int64_t total = rows * width;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const float x = __uint_as_float((uint32_t)w[i] << 16) * gamma[i % width];
    const uint32_t packed = ptx::pack_bf16x2(x, 0.f);
    out[i] = (uint16_t)(packed & 0xFFFFu);
  }
}

template <int D, int TN>
cudaError_t launch_pd(const CUtensorMap& tx, const CUtensorMap& tw, const PrologueParams& p, cudaStream_t st) {
  const size_t smem = 1024 + (size_t)kStagesP * (kRows + TN) * kKStep * 2;
  auto kern = prologue_qkv<D, TN, kClusterP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t panels = (p.tokens + kRows - 1) / kRows;
  const int64_t clusters = (panels + kClusterP - 1) / kClusterP * 3;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(clusters * kClusterP));
  cfg.blockDim = dim3(kThreadsP);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kClusterP;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, tx, tw, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

int prologue_cluster() { return kClusterP; }

int prologue_tile_cols(int heads, int head_dim) {
  const int f = heads * head_dim;
  if (f % 256 == 0) return 256;
  if (f % 128 == 0) return 128;
  return 0;
}

cudaError_t launch_prologue(const CUtensorMap& tx, const CUtensorMap& tw, const PrologueParams& p,
                            cudaStream_t stream) {
  const int tn = prologue_tile_cols(p.heads, p.head_dim);
  if (p.head_dim == 128 && tn == 256) return launch_pd<128, 256>(tx, tw, p, stream);
  if (p.head_dim == 128 && tn == 128) return launch_pd<128, 128>(tx, tw, p, stream);
  if (p.head_dim == 64 && tn == 256) return launch_pd<64, 256>(tx, tw, p, stream);
  if (p.head_dim == 64 && tn == 128) return launch_pd<64, 128>(tx, tw, p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_fold_weights(const uint16_t* w, const float* gamma, uint16_t* out, int64_t rows, int width,
                                cudaStream_t stream) {
  const int64_t total = rows * width;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  fold_weights<<<(unsigned)blocks, 256, 0, stream>>>(w, gamma, out, rows, width);
  return cudaGetLastError();
}

}  // namespace fas
