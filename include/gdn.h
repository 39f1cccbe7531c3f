/*
 * gdn.h -- C ABI of the Gated DeltaNet (GDN) token-mixer hot path on GB300
 * (sm_103a).
 *
 * The path has two parts, both from the Qwen3.5-style hybrid serving engine
 * that the pages "perf(gdn): dispatch exact causal-conv chunks" and "RTX 5070
 * Ti: close Qwen3.5-4B TTFT, TPOT, and VRAM gaps vs vLLM" optimise:
 *   1. a varlen depthwise causal conv1d (width 4, SiLU, rolling conv_state),
 *      dispatched over exact (sequence, 8-token chunk) descriptors that are
 *      built once per engine step and reused by every GDN layer;
 *   2. the gated delta rule
 *          S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,  o_t = S_t q_t
 *      as a single-token decode update and as a chunked (WY/UT) prefill.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every pointer argument that names a tensor is a DEVICE pointer (memory of
 *   the current CUDA device) unless its comment says "host". The caller owns
 *   all memory; the library allocates nothing. Scratch memory is passed in
 *   explicitly (the prefill "workspace").
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream). Every call is asynchronous on that stream: it validates its
 *   arguments on the host, enqueues kernels and returns. No call synchronises
 *   with the device.
 * - BF16 is IEEE bfloat16 (stored as 16-bit patterns); arithmetic is float32
 *   with round-to-nearest-even on every BF16 store.
 * - Validation happens before any launch. A failed check returns a negative
 *   gdn_status_t and enqueues nothing; outputs are then untouched. Shapes with
 *   zero tokens or zero sequences are valid and enqueue nothing. A CUDA launch
 *   failure returns GDN_ERR_CUDA (the CUDA error string is then available from
 *   gdn_last_cuda_error_string()).
 * - Vector paths need 16-byte alignment: every BF16 tensor pointer, the
 *   float32 state pointer and the conv weights must be 16-byte aligned, and
 *   row strides (in elements) must be multiples of 8.
 * - Contents of device buffers (cu_seqlens values, descriptor counts) cannot be
 *   checked on the host. Kernels that read cu_seqlens treat a decreasing or
 *   out-of-range entry as an empty sequence; gdn_build_conv_chunks also
 *   reports such input through its optional device status word.
 */
#ifndef GDN_GB300_H
#define GDN_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Option bits of the `flags` argument of the delta-rule entry points
 * (gdn_delta_rule_decode, gdn_decode_step_fused, gdn_delta_rule_prefill_chunked
 * and their variants). Other bits are GDN_ERR_INVALID_ARG.
 *
 * GDN_FLAG_QK_L2NORM: q and k are first replaced by x / sqrt(sum x^2 + 1e-6)
 *   per head (the post-conv q/k normalisation).
 * GDN_FLAG_GATE_LOGITS: the gate arrays hold raw logits z_a, z_b instead of
 *   activated gates, and the kernel computes a = exp(-softplus(z_a)) (decay)
 *   and b = sigmoid(z_b) (write strength) itself. Source: "RTX 5070 Ti: close
 *   Qwen3.5-4B TTFT, TPOT, and VRAM gaps vs vLLM", Existing evidence (the gate
 *   prep between the conv and the recurrence folded into a kernel: the
 *   post-conv tile).
 * Without GDN_FLAG_GATE_LOGITS, a and b are the activated gates. Either way a
 * decay below 1e-30 acts as 1e-30.
 */
#define GDN_FLAG_QK_L2NORM 1
#define GDN_FLAG_GATE_LOGITS 2
/* Chunked prefill only: the workspace already holds the call's chunk plan
 * (gdn_delta_rule_prefill_plan), so the call skips building it. */
#define GDN_FLAG_PLANNED 4

/* Status codes. */
typedef enum gdn_status_t {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = -1, /* NULL pointer, negative size, bad stride, half-set descriptor pair */
  GDN_ERR_UNSUPPORTED = -2, /* valid but not implemented: K != 4, head dims, channel count */
  GDN_ERR_ALIGNMENT = -3,   /* a pointer or stride breaks the 16-byte rule */
  GDN_ERR_WORKSPACE = -4,   /* workspace too small, or descriptor capacity exceeded */
  GDN_ERR_CUDA = -5,        /* a CUDA call failed */
  GDN_ERR_TIMEOUT = -6      /* a bounded device-side wait gave up (gdn_device_status) */
} gdn_status_t;

/*
 * One exact conv dispatch unit: tokens [tok_start, tok_start + len) of
 * sequence `seq`, whose first token sits at position `pos_in_seq` of that
 * sequence. 16 bytes, four int32 fields, no padding.
 * Source: "perf(gdn): dispatch exact causal-conv chunks", What changed
 * (exact (sequence, 8-token chunk) descriptors).
 */
typedef struct gdn_conv_chunk_t {
  int32_t seq;
  int32_t tok_start;
  int32_t len;
  int32_t pos_in_seq;
} gdn_conv_chunk_t;

/*
 * Build the exact (sequence, chunk) descriptors of one engine step.
 * Source: "perf(gdn): dispatch exact causal-conv chunks", What changed (built
 * once per step, uploaded once, reused across layers) and its reviewer
 * comment (mirrors the upstream causal-conv metadata builder).
 *
 *   cu_seqlens    device int32 [num_seqs + 1], packed offsets; cu[0] must be 0
 *                 and the entries non-decreasing.
 *   num_seqs      N >= 0.
 *   chunk_tokens  tokens per descriptor (8 on the engine path), at least 3
 *                 (K - 1): the conv then has exactly one descriptor per
 *                 sequence that reads the old conv_state, which lets it update
 *                 the state in place. Any value at least the longest sequence
 *                 gives whole-sequence descriptors. Smaller values return
 *                 GDN_ERR_INVALID_ARG.
 *   chunks        device gdn_conv_chunk_t [capacity], 16-byte aligned (output).
 *   capacity      entries available in `chunks`; sum_s ceil(L_s / chunk_tokens)
 *                 is at most floor(T / chunk_tokens) + N.
 *   num_chunks    device int32 [1] (output): the descriptor count.
 *   device_status device int32 [1] or NULL (output): GDN_OK, or
 *                 GDN_ERR_INVALID_ARG for malformed cu_seqlens, or
 *                 GDN_ERR_WORKSPACE when the count exceeds `capacity`. In
 *                 both error cases *num_chunks is set to 0, so conv launches
 *                 that read it do nothing.
 * Order: sequence-major, chunks ascending; fields as in gdn_conv_chunk_t;
 * empty sequences emit nothing. One kernel launch, no host synchronisation.
 */
GDN_API gdn_status_t gdn_build_conv_chunks(const int32_t* cu_seqlens, int32_t num_seqs,
                                   int32_t chunk_tokens, gdn_conv_chunk_t* chunks,
                                   int32_t capacity, int32_t* num_chunks,
                                   int32_t* device_status, void* stream);

/*
 * Varlen depthwise causal conv1d prefill (width K = 4) with SiLU and a rolling
 * state. Source: "perf(gdn): dispatch exact causal-conv chunks", What changed
 * (one program per descriptor; whole-sequence mapping kept as the rollback)
 * and "RTX 5070 Ti ...", Existing evidence (the K=4 specialisation).
 *
 * For sequence s, channel c and local position i:
 *   y[cu[s]+i, c] = SiLU(bias[c] + sum_{j=0..3} w[c, j] * xw(i - 3 + j)),
 *   xw(m) = x[cu[s]+m, c] for m >= 0; conv_state[s, c, 3+m] for m < 0 when
 *   has_initial_state[s] != 0, else 0.
 * conv_state[s] is then replaced by the last 3 entries of (initial state ++
 * x_s); sequences with no tokens keep their state.
 *
 *   x                  BF16 [T, C], row stride x_stride elements (>= C, % 8 == 0).
 *   w                  BF16 [C, 4] contiguous.   bias  BF16 [C] or NULL (zero).
 *   conv_state         BF16 [N, C, 3] contiguous, read and written.
 *   has_initial_state  uint8 [N] or NULL (all zero).
 *   cu_seqlens         int32 [N + 1].
 *   chunks, num_chunks descriptors from gdn_build_conv_chunks (chunk_tokens
 *                      8 on the engine path, any size >= 3), and their count; BOTH
 *                      NULL selects whole-sequence dispatch (one program per
 *                      sequence, byte-identical output). Exactly one NULL is
 *                      GDN_ERR_INVALID_ARG.
 *   max_chunks         the grid bound: the capacity used to build `chunks`
 *                      (ignored in whole-sequence mode).
 *   T, C, K, N         tokens, channels (% 8 == 0), taps (4 only), sequences.
 *   silu               1 applies SiLU, 0 returns the pre-activation.
 *   y                  BF16 [T, C] contiguous (output). Must not alias x.
 */
GDN_API gdn_status_t gdn_causal_conv1d_fwd(const void* x, int64_t x_stride, const void* w,
                                   const void* bias, void* conv_state,
                                   const uint8_t* has_initial_state,
                                   const int32_t* cu_seqlens,
                                   const gdn_conv_chunk_t* chunks,
                                   const int32_t* num_chunks, int32_t max_chunks,
                                   int32_t T, int32_t C, int32_t K, int32_t N,
                                   int32_t silu, void* y, void* stream);

/*
 * One decode token per sequence through the conv, rolling the state.
 * Window (conv_state[n,c,0..2], x[n,c]); y = SiLU(bias + sum_j w[c,j] win_j);
 * conv_state[n,c] <- (conv_state[n,c,1], conv_state[n,c,2], x[n,c]).
 *
 *   x           BF16 [N, C], row stride x_stride (>= C, % 8 == 0).
 *   w, bias     as for gdn_causal_conv1d_fwd.
 *   conv_state  BF16 [N, C, 3], read and written.
 *   y           BF16 [N, C] contiguous (output).
 */
GDN_API gdn_status_t gdn_causal_conv1d_update(const void* x, int64_t x_stride, const void* w,
                                      const void* bias, void* conv_state, int32_t N,
                                      int32_t C, int32_t K, int32_t silu, void* y,
                                      void* stream);

/*
 * Single-token gated delta-rule update for N sequences.
 * Source: "RTX 5070 Ti ...", Existing evidence (fused decode; the state tile
 * held in registers across the update; vector state stores).
 *
 * For sequence n and v-head h with q/k-head g = h / (Hv / Hk):
 *   S' = a S;  u = b (v - S' k);  S_new = S' + u k^T;  o = S_new q,
 * which equals a S (I - b k k^T) + b v k^T and o = S_new q. No 1/sqrt(dk) scale.
 * flags: GDN_FLAG_QK_L2NORM and / or GDN_FLAG_GATE_LOGITS (see above).
 *
 *   q, k       BF16; element (n, g, i) at n * qk_stride + g * dk + i.
 *   v          BF16; element (n, h, i) at n * v_stride + h * dv + i.
 *   a, b       float32 [N, Hv] contiguous: the decay and write gates, or their
 *              logits with GDN_FLAG_GATE_LOGITS.
 *   S          float32 [N, Hv, dv, dk] contiguous (row i of S is dk-contiguous),
 *              read and written in place.
 *   o          BF16 [N, Hv, dv] contiguous (output).
 *   dk, dv     each one of 16, 32, 64, 128.   Hv % Hk == 0.
 */
GDN_API gdn_status_t gdn_delta_rule_decode(const void* q, const void* k, int64_t qk_stride,
                                   const void* v, int64_t v_stride, const float* a,
                                   const float* b, float* S, void* o, int32_t N,
                                   int32_t Hk, int32_t Hv, int32_t dk, int32_t dv,
                                   int32_t flags, void* stream);

/*
 * One decode step of a GDN layer in a single launch: the conv update of
 * gdn_causal_conv1d_update followed by gdn_delta_rule_decode on its output,
 * without the conv output ever leaving the GPU's on-chip memory. Source: "RTX
 * 5070 Ti ...", Existing evidence (the fused decode path, the post-conv step
 * folded into its neighbours); here the conv update is the part folded in.
 *
 * The result equals the two calls in sequence, bit for bit: the conv output is
 * rounded to BF16 exactly as gdn_causal_conv1d_update stores it, and q | k | v
 * are its channels [0, Hk dk) | [Hk dk, 2 Hk dk) | [2 Hk dk, C).
 *
 *   x              BF16 [N, C] conv inputs, row stride x_stride (>= C, % 8 == 0),
 *                  C = 2 Hk dk + Hv dv.
 *   w, bias        BF16 [C, 4] taps and [C] bias or NULL, as for the conv calls.
 *   conv_state_in  BF16 [N, C, 3]: the state before the step (read only).
 *   conv_state_out BF16 [N, C, 3]: the state after it (written). The two must
 *                  not overlap: several blocks read a q/k channel's old state
 *                  while one of them writes its new one, so the update cannot be
 *                  in place (callers alternate two buffers). Overlap is
 *                  GDN_ERR_INVALID_ARG.
 *   a, b, S, o     as for gdn_delta_rule_decode (S updated in place).
 *   dk, dv         128 only (else GDN_ERR_UNSUPPORTED; use the two calls).
 *   K              4.   silu: 0 or 1.   flags: GDN_FLAG_* bits.
 * All pointers 16-byte aligned.
 */
GDN_API gdn_status_t gdn_decode_step_fused(const void* x, int64_t x_stride, const void* w,
                                   const void* bias, const void* conv_state_in,
                                   void* conv_state_out, const float* a, const float* b,
                                   float* S, void* o, int32_t N, int32_t Hk, int32_t Hv,
                                   int32_t dk, int32_t dv, int32_t K, int32_t silu,
                                   int32_t flags, void* stream);

/*
 * Bytes of device workspace that gdn_delta_rule_prefill_chunked needs for these
 * sizes (0 for invalid sizes). Pure host arithmetic.
 */
GDN_API size_t gdn_delta_rule_prefill_workspace_size(int32_t T, int32_t N, int32_t Hv,
                                             int32_t dk, int32_t dv, int32_t chunk);

/*
 * Chunked (WY/UT) prefill of the gated delta rule over packed sequences.
 * The recurrence is the one of gdn_delta_rule_decode applied token by token;
 * the chunked form reaches the same result up to rounding. Chunks of `chunk`
 * tokens start at each sequence's first token and never cross sequences; the
 * last chunk of a sequence may be partial.
 *
 *   q, k, v, qk_stride, v_stride   as for decode, indexed by packed token t.
 *   a, b        float32 [T, Hv] (gates, or logits with GDN_FLAG_GATE_LOGITS).
 *   flags       GDN_FLAG_* bits, as for decode, plus GDN_FLAG_PLANNED (the
 *               workspace holds this call's plan: gdn_delta_rule_prefill_plan).
 *   cu_seqlens  int32 [N + 1].
 *   S           float32 [N, Hv, dv, dk]: the initial state of sequence s where
 *               has_initial_state[s] != 0 (zeros otherwise), replaced by the
 *               final state. Sequences with no tokens keep S unchanged.
 *   has_initial_state  uint8 [N] or NULL (all zero).
 *   o           BF16 [T, Hv, dv] contiguous (output).
 *   chunk       64 (the only size implemented).
 *   workspace   device scratch of at least
 *               gdn_delta_rule_prefill_workspace_size(T, N, Hv, dk, dv, chunk)
 *               bytes, 256-byte aligned; contents on entry do not matter.
 *               The call owns it until the enqueued work completes. Once it
 *               has, two int32 words report device-side failures, which the
 *               host cannot see before launch: word 1 (byte offset 4) is the
 *               chunk-descriptor builder's status (GDN_OK, or
 *               GDN_ERR_INVALID_ARG for malformed cu_seqlens, which then count
 *               as no chunks at all: state and outputs are left untouched);
 *               word 2 (byte offset 8) is the state pass's status (GDN_OK;
 *               for dk = dv = 128 also GDN_ERR_INVALID_ARG when the chunks do
 *               not cover a sequence, whose state and outputs are then left
 *               untouched, or GDN_ERR_TIMEOUT when a bounded device-side wait
 *               gave up).
 */
GDN_API gdn_status_t gdn_delta_rule_prefill_chunked(const void* q, const void* k, int64_t qk_stride,
                                            const void* v, int64_t v_stride,
                                            const float* a, const float* b,
                                            const int32_t* cu_seqlens, int32_t N, int32_t T,
                                            float* S, const uint8_t* has_initial_state,
                                            void* o, int32_t Hk, int32_t Hv, int32_t dk,
                                            int32_t dv, int32_t chunk, int32_t flags,
                                            void* workspace, size_t workspace_bytes,
                                            void* stream);

/*
 * The chunk plan of a prefill step: the 64-token chunk descriptors of
 * cu_seqlens (and, for dk = dv = 128, the order in which the state pass starts
 * the sequences, longest first), written into `workspace` where
 * gdn_delta_rule_prefill_chunked reads them. Source: "perf(gdn): dispatch
 * exact causal-conv chunks", What changed (the step's descriptors are built
 * once, uploaded once and reused by every layer): every layer of an engine
 * step runs the prefill on the same cu_seqlens, so one plan per step serves
 * them all, each call passing GDN_FLAG_PLANNED.
 *
 *   cu_seqlens, N, T, Hv, dk, dv, chunk   as for gdn_delta_rule_prefill_chunked.
 *   workspace, workspace_bytes            the workspace those calls will use
 *                                         (at least the size they need).
 * Host-side validation as for the prefill (same status codes). One kernel
 * launch; device-side failures (malformed cu_seqlens) are reported in
 * workspace word 1, and every planned call then leaves its state and outputs
 * untouched. A call with GDN_FLAG_PLANNED must use the same cu_seqlens
 * contents, N, T, Hv, dk, dv and chunk as the plan (not checked), and the plan
 * region of the workspace (everything but the chunk records) must not have
 * been overwritten in between; calls without the flag rebuild the plan.
 */
GDN_API gdn_status_t gdn_delta_rule_prefill_plan(const int32_t* cu_seqlens, int32_t N, int32_t T,
                                                 int32_t Hv, int32_t dk, int32_t dv,
                                                 int32_t chunk, void* workspace,
                                                 size_t workspace_bytes, void* stream);

/*
 * The chunked prefill above, for callers that cannot allocate device memory.
 * (The pages describe no such variant; it exists for integration only.)
 *
 * Who needs it: code that must not call cudaMalloc -- a plugin running inside
 * a host framework that owns every device allocation through its own pool, or
 * a call site where an allocation could block or synchronise the device. Such
 * callers cannot provide the workspace that gdn_delta_rule_prefill_chunked
 * takes, so this entry point takes none: its scratch is a fixed 64 MiB array
 * inside the library, present on every GPU that loads the library until the
 * process exits.
 *
 * Arguments, results and layouts are those of gdn_delta_rule_prefill_chunked,
 * minus workspace / workspace_bytes; GDN_FLAG_PLANNED is GDN_ERR_INVALID_ARG
 * here (a plan would have to live in the library's array). Sizes whose workspace
 * (gdn_delta_rule_prefill_workspace_size) exceeds 64 MiB are rejected with
 * GDN_ERR_WORKSPACE before anything is enqueued (for example, 2 x 512 tokens
 * with 32 v-heads of width 128 fit; 2 x 1024 tokens do not).
 *
 * Every argument check and the size limit run before any CUDA call, so a
 * rejected call touches no CUDA state.
 *
 * Set-up: the array's device address belongs to the library's module as
 * loaded into one CUDA context. The first call made in a context (the calling
 * thread's current context; with none current, the current device's primary
 * context, which the call then makes current as any runtime call does) looks
 * the address up with cudaGetSymbolAddress and caches it under that context's
 * unique id, so another context on the same device, or the primary context
 * re-created after cudaDeviceReset, gets its own lookup. Make the first call in
 * a context before capturing a stream in it. The call never allocates: no
 * cudaMalloc, no cudaFree, no allocating library routine.
 *
 * Device-side status: the regular call reports what only the GPU can see
 * (malformed cu_seqlens, a bounded wait that gave up) in words 1 and 2 of its
 * workspace. Here those words live in the library's array, which the caller
 * cannot address; gdn_delta_rule_prefill_chunked_noalloc_status copies them
 * out.
 *
 * Sharing: every call on a device uses the same array, and the array keeps
 * whatever the last call left in it (each call writes everything it reads
 * back, and clears its own status words). Two calls whose work overlaps on the
 * GPU -- on different streams, or from different host threads -- race on the
 * array and corrupt each other's results: serialise them.
 */
GDN_API gdn_status_t gdn_delta_rule_prefill_chunked_noalloc(
    const void* q, const void* k, int64_t qk_stride, const void* v, int64_t v_stride,
    const float* a, const float* b, const int32_t* cu_seqlens, int32_t N, int32_t T, float* S,
    const uint8_t* has_initial_state, void* o, int32_t Hk, int32_t Hv, int32_t dk, int32_t dv,
    int32_t chunk, int32_t flags, void* stream);

/*
 * Status words of the last gdn_delta_rule_prefill_chunked_noalloc call in the
 * current context: enqueues, on `stream`, a copy of the two int32 words that
 * gdn_delta_rule_prefill_chunked documents as its workspace words 1 and 2 into
 * status[0] (the chunk-descriptor builder's status: GDN_OK, or
 * GDN_ERR_INVALID_ARG for malformed cu_seqlens) and status[1] (the state
 * pass's status: GDN_OK, GDN_ERR_INVALID_ARG, or GDN_ERR_TIMEOUT). Read them
 * once the copy has completed; enqueue it on the stream of the call it
 * reports on, after that call.
 *
 *   status  int32 [2]: device memory, or host memory (pinned memory keeps the
 *           copy asynchronous; pageable host memory makes this call wait for
 *           the stream).
 * NULL status is GDN_ERR_INVALID_ARG. Allocates nothing. Before any
 * noalloc prefill in this context the words read as GDN_OK.
 */
GDN_API gdn_status_t gdn_delta_rule_prefill_chunked_noalloc_status(int32_t* status, void* stream);

/*
 * State-slot variants. Source: "RTX 5070 Ti: close Qwen3.5-4B TTFT, TPOT, and
 * VRAM gaps vs vLLM", Problem (the serving engine runs 32 concurrent requests
 * out of a fixed block cache); the pages do not describe the cache layout, so this is
 * the plainest form of it: the recurrent states live in a cache of slots that
 * outlives any one batch, and each call says which slot every sequence of the
 * batch owns.
 *
 * Each *_slots call computes exactly what the call without the suffix computes,
 * with two changes:
 *   conv_state  BF16 [num_slots, C, 3] and S float32 [num_slots, Hv, dv, dk]:
 *               sequence n of the batch reads and writes slot state_indices[n]
 *               instead of entry n.
 *   state_indices  device int32 [N], 4-byte aligned. An index outside
 *               [0, num_slots) (for example -1) marks a padding entry: its
 *               state is neither read nor written and its outputs (its rows of
 *               y or o) are left as they were. The valid indices of one call
 *               must be distinct (two sequences in one slot race); this is not
 *               checked. has_initial_state stays indexed by sequence n.
 *   num_slots   >= 0 (0: every entry is padding).
 * NULL state_indices or negative num_slots is GDN_ERR_INVALID_ARG, a
 * misaligned state_indices GDN_ERR_ALIGNMENT. The results for a valid entry
 * are bit-identical to the call without the suffix on the gathered states.
 */
GDN_API gdn_status_t gdn_causal_conv1d_fwd_slots(const void* x, int64_t x_stride, const void* w,
                                         const void* bias, void* conv_state,
                                         const uint8_t* has_initial_state,
                                         const int32_t* cu_seqlens,
                                         const gdn_conv_chunk_t* chunks,
                                         const int32_t* num_chunks, int32_t max_chunks,
                                         int32_t T, int32_t C, int32_t K, int32_t N,
                                         int32_t silu, void* y,
                                         const int32_t* state_indices, int32_t num_slots,
                                         void* stream);

GDN_API gdn_status_t gdn_causal_conv1d_update_slots(const void* x, int64_t x_stride,
                                            const void* w, const void* bias,
                                            void* conv_state, int32_t N, int32_t C,
                                            int32_t K, int32_t silu, void* y,
                                            const int32_t* state_indices, int32_t num_slots,
                                            void* stream);

GDN_API gdn_status_t gdn_delta_rule_decode_slots(const void* q, const void* k, int64_t qk_stride,
                                         const void* v, int64_t v_stride, const float* a,
                                         const float* b, float* S, void* o, int32_t N,
                                         int32_t Hk, int32_t Hv, int32_t dk, int32_t dv,
                                         int32_t flags, const int32_t* state_indices,
                                         int32_t num_slots, void* stream);

GDN_API gdn_status_t gdn_delta_rule_prefill_chunked_slots(
    const void* q, const void* k, int64_t qk_stride, const void* v, int64_t v_stride,
    const float* a, const float* b, const int32_t* cu_seqlens, int32_t N, int32_t T, float* S,
    const uint8_t* has_initial_state, void* o, int32_t Hk, int32_t Hv, int32_t dk, int32_t dv,
    int32_t chunk, int32_t flags, void* workspace, size_t workspace_bytes,
    const int32_t* state_indices, int32_t num_slots, void* stream);

/*
 * Self-test of the bounded device-side waits every kernel of this library
 * uses on its mbarriers. Launches one CTA that waits, with that same wait, for
 * an mbarrier phase that nothing completes, giving up after about
 * `max_cycles` SM clock cycles (1 .. 4e9; the kernels use about 4e9, ~2 s).
 * When the wait gives up, *device_status becomes GDN_ERR_TIMEOUT, the CTA
 * records it in the sticky status that gdn_device_status reads (as every
 * kernel of the library does when one of its waits gives up) and exits
 * normally: the context stays usable. GDN_OK would mean that the wait
 * returned without its phase completing (a defect).
 *
 *   device_status  device int32 [1] (output).
 * NULL device_status or max_cycles outside the range is GDN_ERR_INVALID_ARG.
 */
GDN_API gdn_status_t gdn_selftest_bounded_wait(int32_t* device_status, int64_t max_cycles,
                                               void* stream);

/*
 * Failures that only the GPU can see. Every kernel of this library bounds its
 * device-side waits (about two seconds); a wait that gives up makes its
 * kernel stop without storing any unit of work it has not finished (the
 * call's outputs and states are then undefined; nothing faults or hangs) and
 * records GDN_ERR_TIMEOUT in a sticky device-side status of the library (one
 * per CUDA context). The chunked prefill also reports it in its workspace
 * (word 2).
 *
 * gdn_device_status enqueues, on `stream`, the read of that status into
 * *status: GDN_OK, or the first failure recorded since the last clear. With
 * clear = 1 the status is reset to GDN_OK after the read.
 *
 *   status  device int32 [1], 4-byte aligned (written by a kernel).
 *   clear   0 or 1.
 * NULL or misaligned status, or another clear value, is GDN_ERR_INVALID_ARG /
 * GDN_ERR_ALIGNMENT. Allocates nothing.
 */
GDN_API gdn_status_t gdn_device_status(int32_t* status, int32_t clear, void* stream);

/* Static description of a status code (never NULL). */
GDN_API const char* gdn_status_string(gdn_status_t status);

/* Text of the CUDA error behind the calling thread's most recent GDN_ERR_CUDA
 * ("" if none). Kept per thread, like errno: the pointer stays valid until the
 * same thread's next failing call, whatever other threads do. */
GDN_API const char* gdn_last_cuda_error_string(void);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* GDN_GB300_H */
