// Kernel launch interfaces (host side) and the parameter blocks they take.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fas {

// Device error word bits.
constexpr unsigned int kErrWaitProducer = 1u;
constexpr unsigned int kErrWaitMma = 2u;
constexpr unsigned int kErrWaitSoftmax = 4u;
constexpr unsigned int kErrWaitDrain = 8u;
constexpr unsigned int kErrWaitSelftest = 16u;

// Bound on any single device-side wait in the attention kernel.
constexpr uint64_t kWaitLimitNs = 500ull * 1000ull * 1000ull;

struct PrepassArgs {
  const void* q;        // bf16, row (h, j) at q + h * head_stride + j * row_stride
  const void* k;        // bf16, same layout as q
  int64_t row_stride;   // elements between consecutive tokens of one head
  int64_t head_stride;  // elements between heads
  const int4* table;    // [Nf] {start0, len0, start1, len1}
  float* partial;       // [H, Nf, chunks, d]  per-chunk key sums
  float* mu;            // [H, d]              mean key
  float* fsum;          // [H, Nf, d]          per-frame key sums
  float* mpart;         // [H, Nf, chunks]     per-chunk max centred key norm
  float* frame_max;     // [H, Nf]             per-frame max centred key norm
  float* mvis;          // [H, Nf]             max over the frames visible from f
  float* kbarc;         // [H, Nf, d]          mean centred key visible from f
  float* row_bound;     // [H, N]              m_i (natural-log units)
  float* gpart;         // [H, Nf, chunks]     per-chunk max slack
  float* stat;          // [H]                 max slack per head
  uint8_t* elig;        // [H]
  int64_t N;
  int T, Nf, H, d, chunks;
  float scale;          // 1/sqrt(d)
};

// Launches the six prepass kernels on `stream`; returns the number launched
// (negative on a launch error).
int launch_prepass(const PrepassArgs& a, cudaStream_t stream);

// The same six kernels, with the window statistics computed from the frame
// rule instead of the plan's block table (no library state needed).  The
// table pointer in `a` is not used.
int launch_prepass_rule(const PrepassArgs& a, int ref_frames, int window_radius, cudaStream_t stream);

struct FwdParams {
  const int4* work;        // [n_work] {head, query frame, query tile, key blocks}
  const int4* table;       // [Nf] {start0, len0, start1, len1}
  const float* row_bound;  // [H, N] or null (online mode)
  const uint8_t* elig;     // [H] or null (online mode)
  uint16_t* out;           // bf16, row (h, j) at out + h * out_head_stride + j * out_row_stride
  int64_t out_row_stride;  // elements
  int64_t out_head_stride; // elements
  float* lse;              // [H, N]
  unsigned int* err;       // device error word
  int64_t N;
  int T;
  int Bk;
  int kst, vst;            // K and V ring depths (set by the launcher from the smem budget)
  int kd;                  // K stages in their own slots; stage kd (if kst > kd) reuses the Q slot
  uint32_t qslot_bytes;    // bytes of the shared-memory slot that first holds the Q tile
  int mode;                // FAS_MODE_*
  float scale_log2;        // log2(e) / sqrt(d)
  uint64_t limit_ns;
};

cudaError_t launch_attention(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const FwdParams& p, int grid, cudaStream_t stream);

cudaError_t launch_wait_selftest(unsigned int* err, uint64_t limit_ns, cudaStream_t stream);

}  // namespace fas
