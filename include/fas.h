/*
 * fas.h — frame-aligned sparse attention for GB300 (sm_103a), C ABI.
 *
 * The operation (page "HeyGen x Google Cloud: Avatar IV on TPU",
 * news.xcc.im/article/5328):
 *
 *   - section "Deleting the Mask": the queries of each video frame attend to
 *     the keys of a window of nearby frames plus one global reference frame.
 *     The live region snaps to frame boundaries, so key blocks whose size is a
 *     multiple of 16 dividing the frame span are either fully visible or fully
 *     hidden; one pass over the visible blocks covers the whole mask, with no
 *     mask predicate, padding, second pass or merge.
 *   - section "Unchaining the Softmax": the running maximum of online softmax
 *     is replaced by a per-row upper bound (Cauchy-Schwarz: |q| times the
 *     largest norm of the mean-centred keys the row can see).  Mean-centring
 *     changes no output in exact arithmetic.  Heads whose bound is too loose
 *     use the online-softmax path inside the same kernel.
 *   - section "Proving the Pixels Didn't Change": the final product P.V runs
 *     in bf16 on the matrix unit.
 *
 * Geometry.  T = frame_tokens, R0 = ref_frames, F = n_frames, Nf = R0 + F,
 * N = Nf * T.  Token j belongs to frame j / T.  Frames 0..R0-1 are reference
 * frames, R0..Nf-1 video frames in time order.  Query frame f sees
 *   - every frame, if f < R0 (the reference is global both ways);
 *   - frames 0..R0-1 and max(R0, f-r)..min(Nf-1, f+r), if f >= R0.
 *
 * Data layout (all device pointers, owned by the caller):
 *   q, k, v, out : bf16, base 16-byte aligned, contiguous [H, N, d] (the
 *                  default, FAS_LAYOUT_HND) or, after
 *                  fas_set_layout(FAS_LAYOUT_NHD), contiguous [N, H, d];
 *   lse          : fp32, contiguous [H, N] in both layouts (natural log of
 *                  the sum of exp(s * q.k) over the visible keys,
 *                  s = 1/sqrt(d)).
 * Batch is folded into H: every head is independent.
 *
 * State.  The library holds one plan at a time (not thread-safe).  fas_plan
 * owns the block table, the work list, the prepass statistics and a device
 * error word; fas_free or the next fas_plan with other arguments releases
 * them.  All device work is enqueued on the caller's stream (a cudaStream_t
 * passed as void*; NULL = legacy default stream) and is asynchronous unless
 * stated otherwise.
 *
 * Errors.  Every call returns FAS_OK (0) or a negative FAS_ERR_* code.
 * Argument and order checks are synchronous and leave the state unchanged.
 * Launch failures return FAS_ERR_CUDA.  A device-side wait that exceeds its
 * bound sets the device error word; the next synchronising call (fas_status,
 * or fas_prepass with elig_host) returns FAS_ERR_TIMEOUT.  fas_status also
 * reports FAS_ERR_BOUND (bounded softmax sums out of range, see fas_forward).  No call traps or
 * asserts on the device.
 */
#ifndef FAS_H_
#define FAS_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  FAS_OK = 0,
  FAS_ERR_ARG = -1,         /* invalid shape or argument */
  FAS_ERR_STATE = -2,       /* call out of order (no plan, no matching prepass) */
  FAS_ERR_ALIGN = -3,       /* pointer not 16-byte aligned */
  FAS_ERR_CUDA = -4,        /* CUDA runtime/driver error (no device, launch failure) */
  FAS_ERR_TIMEOUT = -5,     /* a bounded device-side wait expired */
  FAS_ERR_UNSUPPORTED = -6, /* valid request this build does not support */
  FAS_ERR_SCRATCH = -7,     /* problem needs more than fas_prepass_noalloc's fixed scratch */
  FAS_ERR_BOUND = -8        /* a bounded row's softmax sum left [2^-100, 2^100] (see fas_status) */
};

enum {
  FAS_LAYOUT_HND = 0, /* q, k, v, out contiguous [H, N, d] (head-major) */
  FAS_LAYOUT_NHD = 1, /* q, k, v, out contiguous [N, H, d] (token-major) */
  FAS_LAYOUT_A2A = 2  /* fas_prologue only: a rank's token shard in the head-grouped all-to-all
                         layout [G, P, n, H/(G*P), d] (see fas_prologue) */
};

enum {
  FAS_MODE_AUTO = 0,    /* per head: bounded softmax if eligible, else online */
  FAS_MODE_ONLINE = 1,  /* every head online softmax (running max + rescale) */
  FAS_MODE_BOUNDED = 2  /* every head bounded softmax (ablation; loose heads may underflow) */
};

/* Per-head eligibility threshold: a head keeps the bounded softmax when the
 * guaranteed gap between every row's bound and its true maximum is at most
 * this many nats (e^-32 stays far above the fp32 underflow limit e^-87). */
#define FAS_ELIG_SLACK_NATS 32.0f

typedef struct {
  int32_t block_k;       /* key block B_k: multiple of 16 that divides T */
  int32_t q_tile;        /* query rows per work item (128); tiles never cross frames */
  int32_t n_work;        /* work items = H * Nf * ceil(T / q_tile) */
  int32_t total_frames;  /* Nf */
  int64_t tokens;        /* N */
  int64_t key_blocks;    /* sum over work items of visible key blocks */
  double visible_flops;  /* 4*d per visible (query, key) pair, valid rows only */
  const int32_t* host_table; /* library-owned, Nf x 4 int32 per query frame:
                                start0, len0, start1, len1 (key tokens);
                                len1 = 0 when the two ranges merge */
} fas_plan_info;

/* Build the block table and work list for one geometry ("Deleting the Mask",
 * Fig. 3: blocks divide the frame's token span, so every block is full or
 * skipped).  Requirements: T > 0, T % 16 == 0, F >= 1, R0 >= 0, r >= 0,
 * H >= 1, d in {64, 128}.  B_k is the largest multiple of 16 dividing T that
 * fits the kernel's on-chip budget (at most 160).  Allocates the library's
 * device buffers (needs a CUDA device).  A call with the same arguments as
 * the current plan is a no-op.  info (nullable) receives library-owned
 * pointers valid until the next fas_plan or fas_free. */
int fas_plan(int frame_tokens, int n_frames, int ref_frames, int window_radius,
             int heads, int head_dim, fas_plan_info* info);

/* fas_plan with an explicit key block size (block_k = 0: automatic).  A
 * nonzero block_k must be a multiple of 16 dividing T and at most 160. */
int fas_plan_ex(int frame_tokens, int n_frames, int ref_frames, int window_radius,
                int heads, int head_dim, int block_k, fas_plan_info* info);

/* fas_plan_ex for frames of different spans (a ragged block table):
 * frame_tokens points to R0 + F host int32 token counts, frame 0 first (the
 * reference frames, then the video frames in time order); token j belongs
 * to the frame whose token range [T_0 + .. + T_{g-1}, T_0 + .. + T_g) holds
 * it.  Every count must be a positive multiple of 16.  The key block B_k is
 * the largest multiple of 16 (at most 160) that divides every span, so no
 * block straddles a frame boundary ("Deleting the Mask": blocks divide the
 * frame's token span).  Visibility is the same frame rule as fas_plan.
 * block_k = 0 chooses B_k; a nonzero block_k must divide every span.  The
 * other calls take the ragged plan unchanged (q, k, v, out and lse have
 * N = T_0 + .. + T_{Nf-1} tokens per head); fas_prepass_noalloc has no
 * ragged form.  Query tiles of 128 rows stay inside one frame. */
int fas_plan_ragged(const int32_t* frame_tokens, int n_frames, int ref_frames, int window_radius, int heads,
                    int head_dim, int block_k, fas_plan_info* info);

/* Host-only planning: the same plan fas_plan_ex would build, written to the
 * caller's buffers; touches no device and no library state.
 *   table (nullable): Nf * 4 int32 (see fas_plan_info.host_table);
 *   work  (nullable): n_work * 4 int32 per item: head, query frame,
 *                     query tile, key block count; heaviest items first. */
int fas_plan_describe(int frame_tokens, int n_frames, int ref_frames, int window_radius,
                      int heads, int head_dim, int block_k, fas_plan_info* info,
                      int32_t* table, int32_t* work);

/* fas_plan_describe for a ragged plan (frame_tokens as in fas_plan_ragged). */
int fas_plan_describe_ragged(const int32_t* frame_tokens, int n_frames, int ref_frames, int window_radius,
                             int heads, int head_dim, int block_k, fas_plan_info* info, int32_t* table,
                             int32_t* work);

/* Prepass ("Unchaining the Softmax": precomputed norms, mean-centred keys).
 * Reads q (device, bf16, in the current layout: [H, N, d] by default) once
 * and k twice (one kernel: the key sums, then, once mu_h is known, the
 * centred norms; fas_prepass_with_key_sums skips the first read) and
 * computes per head the mean key mu_h, per key frame the largest centred
 * key norm, and per row
 *   m_i = s q_i.mu_h + s |q_i| max_{visible frames g} max_{j in g} |k_j - mu_h|
 * (an upper bound on the row's largest scaled logit), plus the eligibility
 * statistic stat_h = max_i (b_i - s q_i.kbar_c(i)) where b_i is the centred
 * bound and kbar_c(i) the mean centred key visible from row i; a head is
 * eligible when stat_h <= FAS_ELIG_SLACK_NATS.  Needs a plan.  elig_host
 * (nullable, H bytes, 1 = eligible): if set, the call synchronises the
 * stream, copies the bits and reports device timeouts.  A prepass whose
 * bounded device wait gives up leaves every head ineligible (the online
 * path, correct for any input) and sets the device error word. */
int fas_prepass(const void* q, const void* k, void* cuda_stream, uint8_t* elig_host);

/* fas_prepass with the key column sums given instead of read from k: the
 * kernel's key phase adds key_sums' groups instead of reading k, so k is
 * read once (for the centred norms) and q once.  key_sums: device fp32
 * [H, N/16, d], head-major whatever the layout of q and k, row (h, t) the
 * column sums of head h's keys t*16 .. t*16 + 15, 16-byte aligned; written
 * by fas_prologue_with_key_sums for the k it writes, or by the caller.
 * Frames start at multiples of 16 tokens, so no group spans two frames.
 * The frame sums and mu_h add the groups in a fixed order (results are
 * bit-reproducible) that is not fas_prepass's, so the two calls' statistics
 * agree to fp32 rounding, not bit for bit.  Sums that are not those of k
 * give wrong bounds, which the attention's range guard (FAS_ERR_BOUND)
 * catches only when they are far off.  Null key_sums: FAS_ERR_ARG;
 * otherwise as fas_prepass (same plan, same q/k freshness rule). */
int fas_prepass_with_key_sums(const void* q, const void* k, const float* key_sums, void* cuda_stream,
                              uint8_t* elig_host);

/* Attention.  q, k, v, out: device bf16 in the current layout ([H, N, d],
 * or [N, H, d] after fas_set_layout); lse: device fp32 [H, N].  Modes AUTO
 * and BOUNDED need a prior fas_prepass on the same q and k (else
 * FAS_ERR_STATE); ONLINE does not.  "Same" is checked by pointer only: a
 * caller that overwrites q or k in place must call fas_prepass again.  If
 * it does not, the kernel still guards the result: a bounded row whose
 * probability sum under its bound falls outside [2^-100, 2^100] (weights
 * that overflowed, or whose largest neared fp32's subnormal range) sets a
 * flag that the next fas_status reports as FAS_ERR_BOUND.  Inside that range
 * the bounded softmax is accurate whatever bound it was given (the bound
 * only shifts the exponent).  With fresh bounds an eligible head's sums lie
 * in [2^-47, keys], so the flag never fires; BOUNDED mode on an ineligible
 * head can fire it.  Every output row is written exactly once; out rows are
 * rounded to bf16 (nearest even). */
int fas_forward(const void* q, const void* k, const void* v, void* out, float* lse,
                int mode, void* cuda_stream);

/* Attention with inputs and outputs in HOST memory: the call a process makes
 * when its activations live on the host.  q, k, v, out: host bf16 in the
 * current layout ([H, N, d], or [N, H, d] after fas_set_layout); lse: host
 * fp32 [H, N]; results as for fas_prepass followed by fas_forward
 * (bit-identical outputs).  The heads are independent, so the
 * call splits them into groups and pipelines the groups on four
 * library-owned streams: while group g is computed (prepass and attention),
 * group g+1 is copied in and group g-1 copied out; consecutive groups
 * compute on two alternating streams, so a group's launches can start on
 * the SMs the previous group's last CTAs leave idle.  heads_per_group > 0
 * gives groups of that many heads; 0 gives the default schedule, which
 * ramps up (1, 2, then 4 heads per group) so that the first copy-in, which
 * nothing hides, is short, and ends with a one-head group so that the last
 * copy-out is short too.  The host buffers should be page-locked
 * (cudaHostAlloc or cudaHostRegister); pageable buffers give correct
 * results without the overlap.  On first use per plan the library allocates device copies of
 * q, k, v, out and lse (4*H*N*d*2 + 4*H*N bytes, released by fas_free or
 * the next fas_plan), creates its streams and events, and regroups the work
 * list.  The work starts after everything already enqueued on cuda_stream
 * and the call returns at once: out and lse are complete when cuda_stream
 * reaches this point (synchronise it, or call fas_status, before reading
 * them).  Consecutive calls are ordered with each other.  Needs a plan;
 * heads_per_group outside 0..H returns FAS_ERR_ARG; no pointer alignment is
 * required.  Afterwards fas_prepass_readback reports this call's
 * statistics. */
int fas_forward_host(const void* q, const void* k, const void* v, void* out, float* lse,
                     int mode, int heads_per_group, void* cuda_stream);

/* The splash-style ablation of fas_forward, for measuring what the
 * frame-aligned single pass removes ("Deleting the Mask": the kernel the
 * pages started from tiled the sequence in multiples of 128, so blocks
 * straddle frame boundaries and need a mask predicate; padded the sequence
 * to the tile grid; and ran the frame window and the reference frame as two
 * attention passes writing full-precision intermediates that a merge pass
 * re-read).  Same operation and results as fas_forward in FAS_MODE_ONLINE
 * (within rounding): 128-row query tiles and 128-key blocks over the
 * sequence padded to a multiple of 128, a per-element visibility test in
 * every block a row does not see whole, online softmax, pass 1 over each
 * tile's window keys and pass 2 over the reference keys, each writing
 * O / sum(P) and the LSE in fp32 for every padded row (library-owned
 * intermediates, 2 * H * Npad * (d + 1) * 4 bytes, allocated on first use
 * per plan), then a merge kernel.  q, k, v, out: device bf16 [H, N, d];
 * lse: device fp32 [H, N].  Needs a uniform plan (FAS_ERR_STATE without a
 * plan) in the head-major layout; a ragged plan or the token-major layout
 * returns FAS_ERR_UNSUPPORTED.  No prepass is needed.  Three launches
 * (two when the plan has no reference frame), asynchronous on cuda_stream. */
int fas_forward_ablation(const void* q, const void* k, const void* v, void* out, float* lse, void* cuda_stream);

/* Memory layout of q, k, v and out for the calls that follow, on the
 * current plan: FAS_LAYOUT_HND ([H, N, d], the default of every new plan) or
 * FAS_LAYOUT_NHD ([N, H, d]: the tokens' rows of all heads side by side, as
 * a fused QKV projection writes them, so no transpose is needed before the
 * call).  The kernels read and write the strided layout directly (TMA
 * tensor maps with the layout's strides, strided prepass rows and output
 * stores); results are bit-identical to the same data in [H, N, d].  lse is
 * [H, N] in both layouts.  fas_forward_host takes host buffers in the same
 * layout.  A layout change invalidates the last prepass (AUTO and BOUNDED
 * need a new fas_prepass).  Needs a plan (FAS_ERR_STATE); an unknown layout
 * returns FAS_ERR_ARG. */
int fas_set_layout(int layout);

/* Release every library-owned device buffer and forget the plan. */
int fas_free(void);

/* Synchronise the stream and report the device words: FAS_ERR_TIMEOUT if a
 * bounded wait gave up, else FAS_ERR_BOUND if a bounded row's sum left its
 * safe range (see fas_forward), else FAS_OK; clears both words. */
int fas_status(void* cuda_stream);

/* Copy prepass results to host buffers (each nullable); synchronises the
 * stream.  mu: H*d fp32; frame_max: H*Nf fp32 (largest centred key norm per
 * key frame); stat: H fp32; elig: H bytes; row_bound: H*N fp32 (m_i). */
int fas_prepass_readback(float* mu, float* frame_max, float* stat, uint8_t* elig,
                         float* row_bound, void* cuda_stream);

/* Self-test of the bounded device waits: launches one block that waits on
 * an mbarrier nothing will complete, with the given limit in microseconds
 * (1..1000000).  Expected result: FAS_ERR_TIMEOUT, with the context intact. */
int fas_selftest_wait_timeout(int limit_us, void* cuda_stream);

/* Bytes of the fixed device array that fas_prepass_noalloc uses as scratch. */
#define FAS_NOALLOC_SCRATCH_BYTES (4u << 20)

/* fas_prepass for callers that cannot allocate device memory.  (The pages
 * have no counterpart; this is a deployment convenience.)  Some callers own
 * all device memory themselves: a serving process that reserves the GPU's
 * memory in its own pool at start-up and hands libraries only pre-sized
 * buffers, or a per-chunk streaming loop that must not stall on
 * cudaMalloc/cudaFree, which can synchronise the device.  This call needs no
 * plan and allocates nothing: its scratch is a fixed array of
 * FAS_NOALLOC_SCRATCH_BYTES in device memory that the library image holds on
 * every GPU that loads it, until the process exits.
 *   q, k       : device bf16 [H, N, d] (head-major, whatever the current
 *                layout of the plan calls), 16-byte aligned, with exactly
 *                N = (ref_frames + n_frames) * frame_tokens rows per head:
 *                the call has no plan to check the buffers against, and
 *                shorter buffers are read past their end;
 *   row_bound  : device fp32 [H, N] (the same N), receives m_i (as
 *                fas_prepass_readback);
 *   stat       : device fp32 [H], receives stat_h;
 *   elig       : device uint8 [H], receives the eligibility bits.
 * The geometry arguments follow fas_plan.  The scratch needed is about
 * 4 * H * Nf * (ceil(T/1024) * d + 2 * d) bytes; a geometry that does not fit
 * returns FAS_ERR_SCRATCH before any device work (e.g. 720p and 1080p SR
 * chunks with H up to 48, d = 128 fit; H = 96 at 720p does not).
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current, and again after the
 * device's context has changed (a device reset); make that first call
 * before any stream capture.  All calls share the one array and leave their
 * values in it; each call clears, on cuda_stream, the counters, flags and
 * error word it keeps there (and every other element is written before it
 * is read): calls that may overlap on the GPU — other streams, other host
 * threads — race and must be serialised by the caller.  Asynchronous on
 * cuda_stream; launch errors return FAS_ERR_CUDA.  If a bounded device wait
 * gives up, elig stays all zero (every head ineligible: the online path,
 * correct for any input). */
int fas_prepass_noalloc(const void* q, const void* k, int frame_tokens, int n_frames, int ref_frames,
                        int window_radius, int heads, int head_dim, float* row_bound, float* stat,
                        uint8_t* elig, void* cuda_stream);

/* The attention prologue ("Layout Is the ABI", Fig. 5: normalization,
 * rotary embeddings, projections and head packing fused into one kernel that
 * writes exactly the layout the consumer reads).  For each token n:
 *   y_n = (x_n / sqrt(mean(x_n^2) + eps) * gamma) W^T,   W: [3*H*d, C],
 * output features [0, H*d) are q, [H*d, 2*H*d) k, the rest v, head h of each
 * the d features from h*d; q and k are rotated per head, element i paired
 * with i + d/2: (a, b) -> (a*cos - b*sin, a*sin + b*cos) with
 * cos/sin[n, i]; v is as projected.  Rounded once to bf16 (nearest even).
 * The projection runs on the tensor cores on the raw hidden states with
 * the norm scale folded into the weight (fas_prologue_fold_weights) and
 * 1/rms applied per row afterwards.
 *   x         : device bf16 [tokens, width] (row-major), 16-byte aligned;
 *   w_folded  : device bf16 [3*heads*head_dim, width] from
 *               fas_prologue_fold_weights, 16-byte aligned;
 *   cos_tab,
 *   sin_tab   : device fp32 [tokens, head_dim/2], 16-byte aligned;
 *   q, k, v   : device bf16 outputs, 16-byte aligned, in `layout`:
 *               FAS_LAYOUT_HND [heads, tokens, d]; FAS_LAYOUT_NHD
 *               [tokens, heads, d]; FAS_LAYOUT_A2A [groups, ranks, tokens,
 *               heads/(groups*ranks), d], element [g, r, t, j] being token t
 *               of head g*(heads/groups) + r*(heads/(groups*ranks)) + j (the
 *               input of a head-grouped sequence-to-head all-to-all: group
 *               g's slab [ranks, tokens, ...] is sent slice r to rank r);
 *   groups,
 *   ranks     : the A2A layout's G and P (ignored for the other layouts).
 * Requirements: width a positive multiple of 64; head_dim in {64, 128};
 * heads * head_dim a multiple of 128; for A2A heads divisible by
 * groups * ranks; eps >= 0; tokens >= 1.  Otherwise FAS_ERR_ARG; pointer
 * misalignment FAS_ERR_ALIGN.  Needs no plan.  One kernel, asynchronous on
 * cuda_stream; a bounded device wait that gives up sets the error word of
 * the current plan, if any (read by fas_status), and leaves the outputs
 * incomplete. */
int fas_prologue(const void* x, const void* w_folded, const float* cos_tab, const float* sin_tab, int tokens,
                 int width, int heads, int head_dim, float eps, void* q, void* k, void* v, int layout, int groups,
                 int ranks, void* cuda_stream);

/* fas_prologue that also writes the prepass's key statistic, so that
 * fas_prepass_with_key_sums need not read k back for it ("Layout Is the
 * ABI": the producer writes what its consumer reads).  key_sums: device
 * fp32 [heads, tokens/16, head_dim], 16-byte aligned (null: as
 * fas_prologue); row (h, t) receives the column sums of head h's keys for
 * tokens t*16 .. t*16 + 15 exactly as written to k (bf16 values added in
 * fp32, in a fixed order).  In the all-to-all layout the tokens are the
 * rank's own.  tokens must be a multiple of 16 (FAS_ERR_ARG); misaligned
 * key_sums: FAS_ERR_ALIGN. */
int fas_prologue_with_key_sums(const void* x, const void* w_folded, const float* cos_tab, const float* sin_tab,
                               int tokens, int width, int heads, int head_dim, float eps, void* q, void* k, void* v,
                               int layout, int groups, int ranks, float* key_sums, void* cuda_stream);

/* Folds the RMSNorm scale into the projection weight once, for
 * fas_prologue: w_folded[o, c] = bf16(w[o, c] * gamma[c]) (nearest even).
 * w, w_folded: device bf16 [out_features, width] (may not overlap);
 * gamma: device fp32 [width].  Asynchronous on cuda_stream. */
int fas_prologue_fold_weights(const void* w, const float* gamma, void* w_folded, int width, int out_features,
                              void* cuda_stream);

/* Kernel launches issued by the last fas_prepass / fas_forward call. */
int fas_last_launch_count(void);

/* Static description of a status code. */
const char* fas_error_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* FAS_H_ */
