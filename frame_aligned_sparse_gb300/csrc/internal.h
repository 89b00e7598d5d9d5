// Internal declarations shared by the planner, the host API and the kernels.
#pragma once

#include <stdint.h>
#include <vector>

namespace fas {

constexpr int kQTile = 128;        // query rows per work item (MMA M)
constexpr int kMaxBlockK = 160;    // largest key block: TMEM (O, two S buffers, Q) and the softmax registers
#ifndef FAS_PREPASS_ROWS
#define FAS_PREPASS_ROWS 256
#endif
constexpr int kPrepassRows = FAS_PREPASS_ROWS;  // rows per prepass work item (one warp's), at most; items never cross frames
#ifndef FAS_PREPASS_MIN_ROWS
#define FAS_PREPASS_MIN_ROWS 32
#endif
constexpr int kPrepassMinRows = FAS_PREPASS_MIN_ROWS;  // rows per prepass work item, at least (launches over few heads)
constexpr int kPrepassRowsNoalloc = 1024;       // rows per item of fas_prepass_noalloc (fewer partial results to hold)
#ifndef FAS_PREPASS_CTAS
#define FAS_PREPASS_CTAS 2
#endif
constexpr int kPrepassCtasPerSm = FAS_PREPASS_CTAS;  // resident prepass CTAs per SM (bounds its registers)

struct HostPlan {
  int T = 0, F = 0, R0 = 0, r = 0, H = 0, d = 0;  // T: the frame span (the largest one when ragged)
  bool ragged = false;                              // frames have their own spans
  int Nf = 0;
  int64_t N = 0;
  int Bk = 0;
  int n_work = 0;
  int64_t key_blocks = 0;
  double visible_flops = 0.0;
  std::vector<int32_t> spans;  // Nf x 2: first token, tokens
  std::vector<int32_t> table;  // Nf x 4: start0, len0, start1, len1 (key tokens)
  std::vector<int32_t> fvis;   // Nf x 4: visible frames [x, y) and [z, w)
  std::vector<int32_t> work;   // n_work x 4: head, query frame, query tile, key blocks

  bool same_geometry(const HostPlan& o) const {
    return T == o.T && F == o.F && R0 == o.R0 && r == o.r && H == o.H && d == o.d && Bk == o.Bk &&
           ragged == o.ragged && spans == o.spans;
  }
};

// Validates and builds the plan on the host.  Returns a FAS_* status.
// spans: null (every frame has T tokens) or R0 + F per-frame token counts.
int build_plan(const int32_t* spans, int T, int F, int R0, int r, int H, int d, int block_k, HostPlan* out);

// Largest legal key block dividing T (0 when none).
int auto_block_k(int T);

}  // namespace fas
