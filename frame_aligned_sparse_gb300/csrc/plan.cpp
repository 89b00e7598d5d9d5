// Block-table planner (host only).
//
// "HeyGen x Google Cloud: Avatar IV on TPU", section "Deleting the Mask" and
// Fig. 3: the live region of the mask snaps to frame boundaries, so a key
// block size that is a multiple of 16 and divides the frame's token span
// makes every block either fully visible or fully hidden.  The visible key
// tokens of a query frame are then at most two contiguous ranges — the
// reference frame(s) and the clipped window — and the kernel walks them
// block by block with no mask predicate, padding, second pass or merge.
//
// Frames may have different spans (a ragged block table): the block then
// divides every span, so it still never straddles a frame boundary.

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

int build_plan(const int32_t* spans, int T, int F, int R0, int r, int H, int d, int block_k, HostPlan* out) {
  if (F < 1 || R0 < 0 || r < 0 || H < 1) return FAS_ERR_ARG;
  if (d != 64 && d != 128) return FAS_ERR_ARG;
  const int64_t Nf = (int64_t)R0 + F;
  if (Nf > (int64_t)INT32_MAX / 4) return FAS_ERR_ARG;
  HostPlan p;
  p.ragged = spans != nullptr;
  p.spans.assign((size_t)Nf * 2, 0);
  int64_t N = 0;
  int tmax = 0, tgcd = 0;
  for (int64_t f = 0; f < Nf; ++f) {
    const int tf = spans ? spans[f] : T;
    if (tf <= 0 || tf % 16 != 0) return FAS_ERR_ARG;
    p.spans[(size_t)f * 2] = (int32_t)std::min<int64_t>(N, INT32_MAX);
    p.spans[(size_t)f * 2 + 1] = tf;
    N += tf;
    tmax = std::max(tmax, tf);
    tgcd = std::gcd(tgcd, tf);
  }
  // Token indices and TMA coordinates are 32-bit; element offsets are 64-bit.
  if (N > (int64_t)INT32_MAX || (int64_t)H * N > (int64_t)INT32_MAX) return FAS_ERR_ARG;
  int Bk = block_k;
  if (Bk == 0) {
    Bk = auto_block_k(tgcd);
  } else if (Bk < 16 || Bk % 16 != 0 || tgcd % Bk != 0 || Bk > kMaxBlockK) {
    return FAS_ERR_ARG;
  }
  if (Bk == 0) return FAS_ERR_ARG;

  p.T = tmax; p.F = F; p.R0 = R0; p.r = r; p.H = H; p.d = d;
  p.Nf = (int)Nf; p.N = N; p.Bk = Bk;
  p.table.assign((size_t)Nf * 4, 0);
  p.fvis.assign((size_t)Nf * 4, 0);
  auto start = [&](int64_t f) -> int32_t { return f < Nf ? p.spans[(size_t)f * 2] : (int32_t)N; };

  double pairs = 0.0;  // visible (query, key) token pairs of one head
  for (int f = 0; f < Nf; ++f) {
    int32_t* e = &p.table[(size_t)f * 4];
    int32_t* v = &p.fvis[(size_t)f * 4];
    const double tf = p.spans[(size_t)f * 2 + 1];
    if (f < R0) {
      // Reference rows see every frame (the reference is global both ways).
      e[0] = 0; e[1] = (int32_t)N; e[2] = 0; e[3] = 0;
      v[0] = 0; v[1] = (int32_t)Nf; v[2] = 0; v[3] = 0;
      pairs += tf * (double)N;
      continue;
    }
    const int lo = std::max(R0, f - r);
    const int hi = (int)std::min<int64_t>(Nf - 1, (int64_t)f + r);
    v[0] = 0; v[1] = R0; v[2] = lo; v[3] = hi + 1;
    if (R0 == 0 || lo == R0) {
      // Reference and window are adjacent: one range.
      e[0] = start(R0 == 0 ? lo : 0); e[1] = start(hi + 1) - e[0]; e[2] = 0; e[3] = 0;
    } else {
      e[0] = 0; e[1] = start(R0); e[2] = start(lo); e[3] = start(hi + 1) - start(lo);
    }
    pairs += tf * (double)(e[1] + e[3]);
  }
  p.visible_flops = 4.0 * d * (double)H * pairs;

  // Work items: (head, query frame, query tile), heaviest first.  Within one
  // weight the order stays head-major then frame-major, so neighbouring CTAs
  // share the same key/value window in L2.
  int64_t nw = 0;
  for (int f = 0; f < Nf; ++f) nw += (p.spans[(size_t)f * 2 + 1] + kQTile - 1) / kQTile;
  nw *= H;
  if (nw > (int64_t)INT32_MAX / 4) return FAS_ERR_ARG;
  p.n_work = (int)nw;
  std::vector<int32_t> items((size_t)nw * 4);
  size_t w = 0;
  for (int h = 0; h < H; ++h)
    for (int f = 0; f < Nf; ++f) {
      const int32_t* e = &p.table[(size_t)f * 4];
      const int32_t nblk = (e[1] + e[3]) / Bk;
      const int tiles = (p.spans[(size_t)f * 2 + 1] + kQTile - 1) / kQTile;
      for (int t = 0; t < tiles; ++t) {
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
