// Block-table planner (host only).
//
// "HeyGen x Google Cloud: Avatar IV on TPU", section "Deleting the Mask" and
// Fig. 3: the live region of the mask snaps to frame boundaries, so a key
// block size that is a multiple of 16 and divides the frame's token span
// makes every block either fully visible or fully hidden.  The visible key
// tokens of a query frame are then at most two contiguous ranges — the
// reference frame(s) and the clipped window — and the kernel walks them
// block by block with no mask predicate, padding, second pass or merge.

#include <algorithm>
#include <numeric>

#include "fas.h"
#include "internal.h"

namespace fas {

int auto_block_k(int T) {
  for (int b = kMaxBlockK; b >= 16; b -= 16)
    if (T % b == 0) return b;
  return 0;
}

int build_plan(int T, int F, int R0, int r, int H, int d, int block_k, HostPlan* out) {
  if (T <= 0 || T % 16 != 0 || F < 1 || R0 < 0 || r < 0 || H < 1) return FAS_ERR_ARG;
  if (d != 64 && d != 128) return FAS_ERR_ARG;
  const int64_t Nf = (int64_t)R0 + F;
  const int64_t N = Nf * T;
  // Token indices and TMA coordinates are 32-bit; element offsets are 64-bit.
  if (N > (int64_t)INT32_MAX || (int64_t)H * N > (int64_t)INT32_MAX) return FAS_ERR_ARG;
  int Bk = block_k;
  if (Bk == 0) {
    Bk = auto_block_k(T);
  } else if (Bk < 16 || Bk % 16 != 0 || T % Bk != 0 || Bk > kMaxBlockK) {
    return FAS_ERR_ARG;
  }
  if (Bk == 0) return FAS_ERR_ARG;

  HostPlan p;
  p.T = T; p.F = F; p.R0 = R0; p.r = r; p.H = H; p.d = d;
  p.Nf = (int)Nf; p.N = N; p.Bk = Bk;
  p.tiles_per_frame = (T + kQTile - 1) / kQTile;
  p.chunks = (T + kPrepassRows - 1) / kPrepassRows;
  p.table.assign((size_t)Nf * 4, 0);

  int64_t pairs_frames = 0;  // visible (query frame, key frame) pairs
  for (int f = 0; f < Nf; ++f) {
    int32_t* e = &p.table[(size_t)f * 4];
    if (f < R0) {
      // Reference rows see every frame (the reference is global both ways).
      e[0] = 0; e[1] = (int32_t)N; e[2] = 0; e[3] = 0;
      pairs_frames += Nf;
      continue;
    }
    const int lo = std::max(R0, f - r);
    const int hi = (int)std::min<int64_t>(Nf - 1, (int64_t)f + r);
    if (R0 == 0 || lo == R0) {
      // Reference and window are adjacent: one range.
      e[0] = 0; e[1] = (hi + 1) * T; e[2] = 0; e[3] = 0;
      if (R0 == 0) { e[0] = lo * T; e[1] = (hi - lo + 1) * T; }
    } else {
      e[0] = 0; e[1] = R0 * T; e[2] = lo * T; e[3] = (hi - lo + 1) * T;
    }
    pairs_frames += R0 + (hi - lo + 1);
  }
  p.visible_flops = 4.0 * d * (double)H * (double)pairs_frames * (double)T * (double)T;

  // Work items: (head, query frame, query tile), heaviest first.  Within one
  // weight the order stays head-major then frame-major, so neighbouring CTAs
  // share the same key/value window in L2.
  const int64_t nw = (int64_t)H * Nf * p.tiles_per_frame;
  if (nw > (int64_t)INT32_MAX / 4) return FAS_ERR_ARG;
  p.n_work = (int)nw;
  std::vector<int32_t> items((size_t)nw * 4);
  size_t w = 0;
  for (int h = 0; h < H; ++h)
    for (int f = 0; f < Nf; ++f) {
      const int32_t* e = &p.table[(size_t)f * 4];
      const int32_t nblk = (e[1] + e[3]) / Bk;
      for (int t = 0; t < p.tiles_per_frame; ++t) {
        items[w * 4 + 0] = h; items[w * 4 + 1] = f; items[w * 4 + 2] = t; items[w * 4 + 3] = nblk;
        p.key_blocks += nblk;
        ++w;
      }
    }
  std::vector<int64_t> order((size_t)nw);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int64_t a, int64_t b) {
    return items[(size_t)a * 4 + 3] > items[(size_t)b * 4 + 3];
  });
  p.work.resize((size_t)nw * 4);
  for (size_t i = 0; i < (size_t)nw; ++i)
    for (int c = 0; c < 4; ++c) p.work[i * 4 + c] = items[(size_t)order[i] * 4 + c];

  *out = std::move(p);
  return FAS_OK;
}

}  // namespace fas
