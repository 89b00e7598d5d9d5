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
constexpr unsigned int kErrWaitPrepass = 32u;

// Flag word bits (a word of its own: they report on results and stop no
// wait).  kFlagBoundRange: a bounded row's probability sum under its bound
// left [kBoundSumMin, kBoundSumMax].  A valid bound keeps every weight at or
// below 1 and, for an eligible head (slack <= 32 nats), the largest at or
// above e^-32, so the sum lies in [2^-47, keys]; outside the range the
// weights overflowed or their largest neared fp32's subnormal range, which
// a bound from other inputs (q or k changed after the prepass) causes.
constexpr unsigned int kFlagBoundRange = 1u;
constexpr float kBoundSumMin = 0x1p-100f;
constexpr float kBoundSumMax = 0x1p100f;

// Bound on any single device-side wait in the attention kernel.
constexpr uint64_t kWaitLimitNs = 500ull * 1000ull * 1000ull;

// A bf16 tensor map with 128-byte swizzle (dims innermost first); returns a
// FAS_* status.
int bf16_tensor_map(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                    const cuuint64_t* strides_bytes, const cuuint32_t* box);

struct PrepassArgs {
  const void* q;        // bf16, row (h, j) at q + h * head_stride + j * row_stride
  const void* k;        // bf16, same layout as q
  int64_t row_stride;   // elements between consecutive tokens of one head
  int64_t head_stride;  // elements between heads
  const int2* spans;    // [Nf] {first token, tokens} of each frame; null: frame g is [g*T, (g+1)*T)
  const int4* fvis;     // [Nf] frames visible from f: [x, y) and [z, w); null: the frame rule with R0, r
  int R0, r;            // reference frames and window radius (used when fvis is null)
  const float* key_sums = nullptr;  // null (the key items read k), or [H, N / 16, d] key sums per 16 rows
  float* ksum_part;     // [H, Nf, chunks_k, d] per-item key column sums
  float* kmax_part;     // [H, Nf, chunks_q]    per-item max |k - mu|^2
  float* gmax_part;     // [H, Nf, chunks_q]    per-item max slack
  float* mu;            // [H, d]              mean key
  float* fsum;          // [H, Nf, d]          per-frame key sums
  float* frame_max;     // [H, Nf]             per-frame max centred key norm
  float* gmax_frame;    // [H, Nf]             per-frame max slack
  float* kbarc;         // [H, Nf, d]          mean centred key visible from f
  float* mvis;          // [H, Nf]             max over the frames visible from f
  float* row_bound;     // [H, N]              m_i (natural-log units)
  float* stat;          // [H]                 max slack per head
  uint8_t* elig;        // [H]
  unsigned int* sync;   // prepass_sync_words(H, Nf) counters and flags (zeroed by the launcher)
  unsigned int* err;    // device error word
  int64_t N;
  int T;                // frame span when spans is null; else the largest span
  int Nf, H, d;
  int chunks_k;         // key items per frame (sets the frame sums' order: fixed by the frame span)
  int chunks_q;         // centred and query items per frame (any count >= 1)
  float scale;          // 1/sqrt(d)
  uint64_t limit_ns;    // bound on each wait for another item's result
};

// 32-bit words of the prepass's counters and ready flags for H heads.
size_t prepass_sync_words(int H, int Nf);

// Work items per frame and phase for a prepass launch over `heads` heads of
// `rows_per_head` rows (frames of at most `span_max` rows) on `sms` SMs:
// items of kPrepassMinRows .. kPrepassRows rows, about one per two warps of
// the launch per phase, so that a launch over few heads still spreads.
int prepass_chunks(int heads, int64_t rows_per_head, int span_max, int sms);

// Zeroes the counters and the eligibility bits, then launches the fused
// prepass kernel on `stream`; returns the number of kernels launched (1),
// or a negative value on a launch error.
int launch_prepass(const PrepassArgs& a, cudaStream_t stream);

struct FwdParams {
  const int4* work;        // [n_work] {head, query frame, query tile, key blocks}
  const int4* table;       // [Nf] {start0, len0, start1, len1}
  const int2* spans;       // [Nf] {first token, tokens} of each frame
  int q_by_frame;          // Q tensor map is {d, T, Nf, H} (uniform frames); else {d, N, H}
  const float* row_bound;  // [H, N] or null (online mode)
  const uint8_t* elig;     // [H] or null (online mode)
  uint16_t* out;           // bf16, row (h, j) at out + h * out_head_stride + j * out_row_stride
  int64_t out_row_stride;  // elements
  int64_t out_head_stride; // elements
  float* lse;              // [H, N]
  unsigned int* err;       // device error word
  unsigned int* flags;     // device word for kFlagBoundRange (never stops a wait)
  int64_t N;
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

// The splash-style ablation ("Deleting the Mask": 128-multiple tiles over a
// padded sequence, mask predicates, window and reference as two passes
// merged from full-precision intermediates).
struct AblationParams {
  FwdParams f;      // work (this pass's list), err, N, Bk = 128, ring depths, scale_log2, limit_ns
  float* o32;       // [H, Npad, d]  this pass's O / sum(P), fp32
  float* lse32;     // [H, Npad]     this pass's natural-log LSE (-inf: no visible key)
  int64_t Npad;     // N rounded up to a multiple of 128
  int T, R0, r, Nf;
  int pass;         // 0: window keys, 1: reference keys
};

cudaError_t launch_ablation_pass(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const AblationParams& a, int grid, cudaStream_t stream);

cudaError_t launch_ablation_merge(int d, const float* o0, const float* l0, const float* o1, const float* l1,
                                  uint16_t* out, float* lse, int H, int64_t N, int64_t Npad, cudaStream_t stream);

// The attention prologue ("Layout Is the ABI"): RMSNorm -> projection ->
// rotary -> head packing into the consumer's layout.
struct PrologueParams {
  void* q;                // bf16 outputs in `layout`
  void* k;
  void* v;
  const float* cos_tab;   // [tokens, head_dim / 2]
  const float* sin_tab;
  int64_t tokens;         // N (this rank's tokens for the all-to-all layout)
  int width;              // C, a multiple of 64
  int heads, head_dim;    // H, d; H * d a multiple of 128
  int layout;             // FAS_LAYOUT_HND, FAS_LAYOUT_NHD or FAS_LAYOUT_A2A
  int groups, ranks;      // the all-to-all layout's G and P
  float* key_sums = nullptr;  // null, or fp32 [heads, tokens / 16, head_dim]: column sums of the
                              // written k over each group of 16 tokens (tokens a multiple of 16)
  float eps;
  unsigned int* err;      // device error word
  uint64_t limit_ns;
};

// Output features per tile of the prologue kernel for H heads of d (0 when
// H * d is not a multiple of 128).
int prologue_tile_cols(int heads, int head_dim);

// CTAs per cluster of the prologue kernel (they share each weight tile).
int prologue_cluster();

cudaError_t launch_prologue(const CUtensorMap& tx, const CUtensorMap& tw, const PrologueParams& p,
                            cudaStream_t stream);

cudaError_t launch_fold_weights(const uint16_t* w, const float* gamma, uint16_t* out, int64_t rows, int width,
                                cudaStream_t stream);

cudaError_t launch_wait_selftest(unsigned int* err, uint64_t limit_ns, cudaStream_t stream);

}  // namespace fas
