/*
 * dspark.h -- C ABI of the GB300 (sm_103a) DSpark ancestral draft-block
 * sampler.
 *
 * The method (brb-nv/TensorRT-LLM PR #21, "2. Golden sampling semantics";
 * brb-nv/TensorRT-LLM PR #27, "2. One fused kernel per draft position"):
 * for request b and draft position k = 0..K-1,
 *     l_k   = base_k + bias(d_{k-1}),   bias(d) = U[d] @ Wb   (rank-r head)
 *     s_k   = l_k / T                   (float32 IEEE division)
 *     d_k   = argmax_v (s_k[v] + g[v])  (Gumbel-max; g from Philox noise
 *                                        keyed by (seed, offset, k))
 *     q_k   = softmax(s_k)              (the proposal, written after the
 *                                        block from the same float32 l_k)
 * with d_{-1} = d0[b], the last accepted token.  Greedy requests take
 * d_k = argmax_v s_k[v] and store a one-hot proposal.  CUDA-graph padding
 * rows draw from the bias alone.  Verification is standard token-level
 * rejection sampling (PR #21, "2. Golden sampling semantics").
 *
 * Noise (reading of PR #27, "2. One fused kernel per draft position"):
 * Philox4x32-10 with key = (seed lo, seed hi) and counter
 * (v >> 2, k | stream << 16, offset lo, offset hi), word v & 3; stream 0
 * feeds the draft, 1 the acceptance uniforms, 2 the residual / bonus draws.
 * g = -log(-log1p(-w)), w = (x + 0.5) * 2^-32.  Ties go to the lowest index;
 * a NaN or -inf score never wins, and a row where nothing wins (every score
 * NaN or -inf) yields token 0.
 *
 * Conventions for every entry point:
 *   - All tensors are dense, row-major, and live in device memory unless
 *     stated otherwise.  The caller owns every buffer; the library does not
 *     allocate, free, print or trap, and does not synchronise except in the
 *     calls documented as synchronising (the measurement variants
 *     dspark_draft_block_profile and dspark_draft_block_timeline, and
 *     dspark_read_device_error).
 *   - Calls are asynchronous on `stream` and, except those three, may be
 *     captured in a CUDA graph (their work is kernel launches and memsets on
 *     `stream`).
 *   - Argument checks run on the host before any launch; a failing check
 *     returns a status and enqueues nothing.  A launch failure returns
 *     DSPARK_ERR_CUDA (from cudaGetLastError).
 *   - Results are bitwise deterministic given the inputs on a given GPU
 *     model (fixed reduction order, counter-based noise).
 */
#ifndef DSPARK_H_
#define DSPARK_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define DSPARK_API __attribute__((visibility("default")))
#else
#define DSPARK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { DSPARK_F32 = 0, DSPARK_BF16 = 1 } dspark_dtype;

typedef enum {
  DSPARK_OK = 0,
  DSPARK_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, bad T,
                                 misaligned pointer, out-of-range token */
  DSPARK_ERR_UNSUPPORTED = 2, /* valid but outside the supported shapes */
  DSPARK_ERR_WORKSPACE = 3,   /* workspace missing or too small */
  DSPARK_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  DSPARK_ERR_DEVICE = 5       /* a kernel recorded an error in the workspace
                                 (a bounded wait ran out); see
                                 dspark_read_device_error */
} dspark_status;

/* Supported shapes: 1 <= B <= 1024, 1 <= K <= 64, 1 <= V <= 2^26,
 * 16 <= r <= 256 with r % 16 == 0.  (PR #27, Results: B x 7 x 200064
 * logits and a rank-256 head sit inside these limits.) */
#define DSPARK_MAX_B 1024
#define DSPARK_MAX_K 64
#define DSPARK_MAX_R 256
#define DSPARK_MAX_V (1 << 26)

/*
 * Bytes of device workspace dspark_draft_block needs for these sizes
 * (0 if the sizes are unsupported).  The workspace holds a device error
 * word (its first 4 bytes), the decision keys the position kernels share
 * across CTAs, per-chunk softmax statistics (two buffers, so consecutive
 * positions do not overwrite each other's) and per-row (max, sum-exp) of
 * every position.  Its contents need not be initialised: every call first
 * clears the error word and the keys (one 2-D memset on `stream`), and
 * every other word is written before it is read.  Two calls in flight at
 * the same time must not share a workspace.
 */
DSPARK_API size_t dspark_draft_workspace_bytes(int B, int K, int V, int r);

/*
 * dspark_draft_block -- ancestral drafting of one K-token block for B
 * requests (PR #27, "2. One fused kernel per draft position").
 *
 *   base_logits  [B,K,V] base_dtype (F32 or BF16); read only, never modified
 *                (PR #27, Test Coverage: the drafter's logits are left as
 *                they are).  Rows of padding requests may hold anything,
 *                NaN included.
 *   U            [V,r] w_dtype;  Wb [r,V] w_dtype (F32 or BF16, both the
 *                same dtype).  bias(d) = U[d] @ Wb, accumulated in float32.
 *   d0           [B] int32, the last accepted token of each request, in
 *                [0, V).  An entry outside that range is replaced by 0 and
 *                the workspace's device error word is set to 1 (read it with
 *                dspark_read_device_error).
 *   seed, offset [B] uint64 each: the request's noise key and draft slot.
 *                A new offset draws anew (PR #27, Test Coverage).
 *   T            temperature, finite and > 0 (the same for every request).
 *   greedy       [B] uint8 or NULL: nonzero = greedy request (argmax chain,
 *                one-hot proposal, no noise consumed).  NULL = all sampled.
 *   pad_row      [B] uint8 or NULL: nonzero = CUDA-graph padding row; its
 *                base logits are ignored and l = bias (PR #27: padding rows
 *                draw from the bias alone).
 *   tokens       [B,K] int32 out: the drafted tokens d_k.
 *   logits       [B,K,V] float32 out: the biased logits l_k.
 *   draft_probs  [B,K,V] float32 out: the proposals q_k.
 *   workspace    device scratch of at least
 *                dspark_draft_workspace_bytes(B,K,V,r) bytes, 256-byte
 *                aligned.
 * Alignment: every device pointer must be at least 16-byte aligned
 * (DSPARK_ERR_INVALID_ARG otherwise).
 * Launches on `stream`, after one 2-D memset of the error word and the
 * decision keys: with a bf16 head, r a multiple of 16 up to 256 and
 * V % 8 == 0 the tensor-core kernel, K positions and one pick per request
 * group (ceil(B / 96) groups of near-equal size, each a chain over the same
 * heads), then one proposal writer; otherwise the FFMA kernel, K positions
 * and K picks, then the writer.  No host synchronisation; graph capturable.
 */
DSPARK_API dspark_status dspark_draft_block(
    const void* base_logits, dspark_dtype base_dtype, const void* U,
    const void* Wb, dspark_dtype w_dtype, const int32_t* d0,
    const uint64_t* seed, const uint64_t* offset, float T,
    const uint8_t* greedy, const uint8_t* pad_row, int B, int K, int V, int r,
    int32_t* tokens, float* logits, float* draft_probs, void* workspace,
    size_t workspace_bytes, cudaStream_t stream);

/*
 * dspark_draft_block_profile -- measurement variant of dspark_draft_block:
 * the same argument checks and the same launch sequence, with a pair of CUDA
 * events recorded on `stream` around every launch.  It then synchronises
 * `stream` and returns, per kernel class, the summed event time and the
 * number of launches:
 *   stage_ms[3], stage_launches[3]  (host arrays) -- [0] the position
 *   kernels (K per request group), [1] the pick kernels (one after each
 *   group's last position on the tensor-core path, one after every position
 *   on the FFMA path), [2] the proposal writer.  The events between launches remove the overlap of
 *   consecutive positions (programmatic dependent launch); see
 *   dspark_draft_block_timeline for times in the block's own schedule.
 * Outputs are identical to dspark_draft_block's.  Because it synchronises
 * and creates events, it must not be captured in a CUDA graph.
 */
DSPARK_API dspark_status dspark_draft_block_profile(
    const void* base_logits, dspark_dtype base_dtype, const void* U,
    const void* Wb, dspark_dtype w_dtype, const int32_t* d0,
    const uint64_t* seed, const uint64_t* offset, float T,
    const uint8_t* greedy, const uint8_t* pad_row, int B, int K, int V, int r,
    int32_t* tokens, float* logits, float* draft_probs, void* workspace,
    size_t workspace_bytes, float* stage_ms, int* stage_launches,
    cudaStream_t stream);

/*
 * dspark_draft_block_timeline -- measurement variant of dspark_draft_block
 * that keeps the block's own schedule (positions chained by programmatic
 * dependent launch, no event between them).  It captures one
 * dspark_draft_block launch sequence from `stream` into a CUDA graph, with
 * event nodes at its start, between the position chain (the memset, the K
 * position kernels and their picks) and the proposal writer, and at its
 * end; it then replays the graph `replays` (>= 1) times, synchronising
 * after each replay, and returns the mean duration of each segment:
 *   chain_ms[1], proposal_ms[1] (host) -- milliseconds per replay.
 * `stream` must be a created stream (not the legacy NULL stream; status
 * DSPARK_ERR_INVALID_ARG) that is not already capturing.  Outputs are
 * identical to dspark_draft_block's.  It creates three events, a graph and
 * its executable (the driver allocates for them) and destroys them before
 * returning; it synchronises and must not itself be captured.
 */
DSPARK_API dspark_status dspark_draft_block_timeline(
    const void* base_logits, dspark_dtype base_dtype, const void* U,
    const void* Wb, dspark_dtype w_dtype, const int32_t* d0,
    const uint64_t* seed, const uint64_t* offset, float T,
    const uint8_t* greedy, const uint8_t* pad_row, int B, int K, int V, int r,
    int32_t* tokens, float* logits, float* draft_probs, void* workspace,
    size_t workspace_bytes, int replays, float* chain_ms, float* proposal_ms,
    cudaStream_t stream);

/*
 * dspark_draft_block_per_request -- dspark_draft_block with a temperature
 * per request and slot-indexed proposals, as a serving batch needs them
 * (PR #27, "2. One fused kernel per draft position": the proposal writer
 * stores q_k into the slot-indexed draft_probs; the temperature of a draft
 * is its request's sampling temperature).
 *
 *   temperature  [B] float32, device, 4-byte aligned: request b's T.  A
 *                value that is not finite and positive counts as 1 and sets
 *                the device error word to 3 (DSPARK_ERR_DEVICE via
 *                dspark_read_device_error).
 *   draft_probs  [num_slots, K, V] float32 when slot is given, else [B,K,V].
 *   slot         [B] int32 device (4-byte aligned) or NULL: request b's
 *                proposals are written to draft_probs[slot[b]]; slots of
 *                different requests must differ; a slot outside
 *                [0, num_slots) writes nothing for that request and sets the
 *                device error word to 4.  Slots of no request are left as
 *                they are.
 *   num_slots    rows of draft_probs (ignored when slot is NULL).
 * Every other argument, the workspace (dspark_draft_workspace_bytes) and the
 * errors are those of dspark_draft_block; tokens and logits stay [B,K] and
 * [B,K,V].  With equal temperatures T the outputs are bitwise those of
 * dspark_draft_block with T.
 */
DSPARK_API dspark_status dspark_draft_block_per_request(
    const void* base_logits, dspark_dtype base_dtype, const void* U,
    const void* Wb, dspark_dtype w_dtype, const int32_t* d0,
    const uint64_t* seed, const uint64_t* offset, const float* temperature,
    const uint8_t* greedy, const uint8_t* pad_row, int B, int K, int V, int r,
    int32_t* tokens, float* logits, float* draft_probs, const int32_t* slot,
    int num_slots, void* workspace, size_t workspace_bytes,
    cudaStream_t stream);

/*
 * dspark_draft_block_noalloc -- dspark_draft_block for callers that cannot
 * allocate device memory: code that is handed only its input and output
 * buffers by a host runtime that owns all device memory (an inference
 * server that sizes every allocation at start-up and forbids allocation
 * afterwards), or that runs where cudaMalloc must not be called.  There is
 * no counterpart in the pages; it is the same launch sequence as
 * dspark_draft_block with the workspace replaced by library-owned scratch.
 *
 * Arguments and outputs are those of dspark_draft_block without
 * `workspace` / `workspace_bytes`.  The scratch is one file-scope device
 * array of DSPARK_NOALLOC_SCRATCH_BYTES bytes (2 MiB), held on every GPU
 * that loads the library until the process exits; sizes whose workspace
 * (dspark_draft_workspace_bytes) exceeds it are rejected with
 * DSPARK_ERR_WORKSPACE before any launch (B <= 101 fits at K = 7).
 * The call allocates nothing: no cudaMalloc, cudaFree or allocating library
 * routine.  Each call made outside stream capture looks up the scratch's
 * device address on the current device (so a device reset or a new primary
 * context is followed); a call made during a capture uses the address the
 * last uncaptured call on that device found, so the first call on a device
 * must come before any capture, and a capture must not outlive a device
 * reset.  Every call on a device shares the one scratch array and it keeps
 * the last call's contents (each call clears the device error word and the
 * decision keys it starts with); calls that overlap on the GPU, from any
 * stream or thread, race on it and must be serialised by the caller.  Device-side error codes
 * of this variant stay in the scratch and are not reported.
 */
#define DSPARK_NOALLOC_SCRATCH_BYTES (2u << 20)
DSPARK_API dspark_status dspark_draft_block_noalloc(
    const void* base_logits, dspark_dtype base_dtype, const void* U,
    const void* Wb, dspark_dtype w_dtype, const int32_t* d0,
    const uint64_t* seed, const uint64_t* offset, float T,
    const uint8_t* greedy, const uint8_t* pad_row, int B, int K, int V, int r,
    int32_t* tokens, float* logits, float* draft_probs, cudaStream_t stream);

/*
 * dspark_draft_host_workspace_bytes -- device workspace of
 * dspark_draft_block_host: that of dspark_draft_block plus room for the
 * per-request inputs and the tokens (0 if the sizes are unsupported).
 */
DSPARK_API size_t dspark_draft_host_workspace_bytes(int B, int K, int V, int r);

/*
 * dspark_draft_block_host -- dspark_draft_block with its inputs in host
 * memory and the drafted tokens returned to host memory; the call issues
 * the copies itself.
 *
 *   base_logits_host [B,K,V] base_dtype in host memory.  Page-locked memory
 *                lets the copies run asynchronously (with pageable memory
 *                each copy synchronises).
 *   d0_host, seed_host, offset_host [B]; greedy_host, pad_row_host [B] or
 *                NULL: host memory, meanings as in dspark_draft_block.
 *   U, Wb        device, as in dspark_draft_block (resident weights).
 *   base_dev     device [B,K,V] base_dtype buffer that receives the drafter
 *                logits (16-byte aligned; read by this call's kernels).
 *   tokens_host  [B,K] int32 host out, copied on `stream` after the block.
 *   logits, draft_probs  device [B,K,V] float32 outputs.
 *   workspace    device, dspark_draft_host_workspace_bytes(B,K,V,r) bytes,
 *                256-byte aligned.
 *   stream       the compute stream; copy_stream a second stream for the
 *                drafter-logit copies (must differ from stream).
 * Position k's drafter logits (B rows of V values, one 2-D copy) travel on
 * copy_stream while earlier positions compute on stream.  Position k waits
 * for its own copy only, and each position's proposals are written as soon
 * as its softmax statistics exist (after the next position on the
 * tensor-core path, after its pick otherwise), so the block's work hides
 * behind the copies.  The copies start after all
 * work issued to `stream` before the call.  Outputs are identical to
 * dspark_draft_block's.  Host buffers must stay valid until `stream` has
 * passed the end of the call.  The call creates and destroys K+1 CUDA
 * events.  It may be captured in a CUDA graph: its event waits join
 * copy_stream to the capture of `stream`.
 */
DSPARK_API dspark_status dspark_draft_block_host(
    const void* base_logits_host, dspark_dtype base_dtype, const void* U,
    const void* Wb, dspark_dtype w_dtype, const int32_t* d0_host,
    const uint64_t* seed_host, const uint64_t* offset_host, float T,
    const uint8_t* greedy_host, const uint8_t* pad_row_host, int B, int K,
    int V, int r, void* base_dev, int32_t* tokens_host, float* logits,
    float* draft_probs, void* workspace, size_t workspace_bytes,
    cudaStream_t stream, cudaStream_t copy_stream);

/*
 * dspark_verify_standard -- standard token-level rejection sampling of the
 * drafts (PR #21, "2. Golden sampling semantics": the default rule), for B
 * requests.
 *
 *   draft_probs  [B,K,V] float32: the proposals q_k the drafts came from.
 *   target_probs [B,K+1,V] float32: the target's p_k for the drafted prefix;
 *                row K is the bonus distribution.
 *   tokens       [B,K] int32 drafts, each in [0, V) (a token outside it makes
 *                that request report accepted_len = -1).
 *   seed, offset [B] uint64 (streams 1 and 2 of the counter layout above).
 *   accepted_len [B] int32 out: number of accepted drafts, 0..K.
 *   emitted_token[B] int32 out: the token emitted after the accepted prefix
 *                (the residual draw at the first rejection, or the bonus
 *                draw from p_K when all K are accepted).
 * Draft k is accepted iff float(u_k * q_k[d_k]) < p_k[d_k] with
 * u_k = ((x >> 9) + 0.5) * 2^-23 from stream 1 word 0 at position k.  The
 * residual is max(p_k - q_k, 0) (p_k itself if that is all zero); draws are
 * Gumbel-max over log(weight) with stream 2 noise at the drawing position.
 */
DSPARK_API dspark_status dspark_verify_standard(const float* draft_probs,
                                     const float* target_probs,
                                     const int32_t* tokens,
                                     const uint64_t* seed,
                                     const uint64_t* offset, int B, int K,
                                     int V, int32_t* accepted_len,
                                     int32_t* emitted_token,
                                     cudaStream_t stream);

/*
 * dspark_verify_block -- block verification of the drafts (PR #21, "2.
 * Golden sampling semantics": the block value of rejection_sample_method,
 * the block verification of Sun et al., 2024), for B requests.  Arguments,
 * layouts, outputs and errors are those of dspark_verify_standard.
 * With d_k = tokens[b,k], q_k = draft_probs[b,k], p_k = target_probs[b,k]:
 *   w_0 = 1, w_{k+1} = min(w_k * (p_k[d_k] / q_k[d_k]), 1) in float32
 *   (a NaN weight counts as 0);
 *   h_i = r_i / (r_i + 1 - w_i) for i = 1..K-1, with
 *   r_i = sum_x max(w_i p_i(x) - q_i(x), 0) (1 when r_i = 1 - w_i = 0);
 *   h_K = w_K;
 *   accepted_len = the largest i in 1..K with u_{i-1} <= h_i (0 if none),
 *   u_k the uniform of the standard rule;
 *   emitted_token: Gumbel-max with stream 2 noise at position accepted_len
 *   over p_K when accepted_len = K, else over max(w p - q, 0) at that
 *   position (over p itself if that is all zero).
 * The sums r_i run in float32 in a fixed order (results are reproducible
 * call to call).  The call reads the K-1 rows p_1..p_{K-1} and q_1..q_{K-1}
 * in full.  On average it accepts at least as many drafts as the standard
 * rule, and it is lossless.
 */
DSPARK_API dspark_status dspark_verify_block(const float* draft_probs,
                                  const float* target_probs,
                                  const int32_t* tokens, const uint64_t* seed,
                                  const uint64_t* offset, int B, int K, int V,
                                  int32_t* accepted_len, int32_t* emitted_token,
                                  cudaStream_t stream);

/*
 * dspark_sample_workspace_bytes -- device workspace of
 * dspark_sample_temperature for R rows of V logits (0 if unsupported).
 */
DSPARK_API size_t dspark_sample_workspace_bytes(int R, int V);

/*
 * dspark_sample_temperature -- temperature-only sampling of target rows
 * (PR #27, "1. Temperature-only sampling runs no filter": softmax and
 * sampling, no top-k, top-p or min-p).
 *
 *   logits       [R,V] float32 device: one row per sample.
 *   temperature  [R] float32 device (4-byte aligned) or NULL: per-row T (a
 *                value that is not finite and positive counts as 1 and sets
 *                the device error word to 3); NULL uses T (finite, > 0).
 *   greedy       [R] uint8 or NULL: 1 = argmax of s, one-hot probabilities.
 *   seed, offset [R] uint64: the row's noise key and counter words.
 *   position     [R] int32 (4-byte aligned) or NULL (0): the counter's
 *                position word, in [0, 65535] (outside: 0 is used and the
 *                device error word is set to 5).
 *   tokens       [R] int32 out; probs [R,V] float32 out, or NULL to skip.
 *   workspace    dspark_sample_workspace_bytes(R, V) bytes, 256-byte aligned.
 * Row i: s = l / T_i (float32 IEEE), token = argmax of s + g with g from
 * noise stream 3 (word v & 3 of Philox4x32-10 block (v >> 2,
 * position | 3 << 16, offset lo, offset hi) under key seed), the lowest
 * index on ties, NaN never winning (a row where nothing wins gives token 0);
 * probs = softmax(s).  R <= 65535.  Three launches on `stream` (two when
 * probs is NULL), graph capturable; results are reproducible call to call.
 */
DSPARK_API dspark_status dspark_sample_temperature(
    const float* logits, const float* temperature, float T,
    const uint8_t* greedy, const uint64_t* seed, const uint64_t* offset,
    const int32_t* position, int R, int V, int32_t* tokens, float* probs,
    void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * dspark_noise_words -- diagnostic: writes the n raw Philox words the
 * sampler uses for elements 0..n-1 of (seed, offset, position k, stream),
 * i.e. out[v] = word (v & 3) of Philox4x32-10(counter (v >> 2,
 * k | stream << 16, offset lo, offset hi), key (seed lo, seed hi)), and
 * gumbel[v] = the float32 Gumbel variate the draft kernel derives from it
 * (gumbel may be NULL).  out/gumbel are device pointers.
 */
DSPARK_API dspark_status dspark_noise_words(uint64_t seed, uint64_t offset, int k,
                                 int stream_id, int n, uint32_t* out,
                                 float* gumbel, cudaStream_t stream);

/*
 * dspark_noise_words_folded -- the same diagnostic computed the way the
 * position, verification and sampler kernels compute their noise: the parts
 * of Philox4x32-10's first two rounds that depend only on the key and the
 * fixed counter words (k | stream << 16, offset lo, offset hi) are folded
 * into per-request constants, and the round keys are precomputed.  Its
 * words must equal dspark_noise_words' (and the published Philox4x32-10's)
 * bit for bit; arguments and errors are those of dspark_noise_words.
 */
DSPARK_API dspark_status dspark_noise_words_folded(uint64_t seed, uint64_t offset,
                                        int k, int stream_id, int n,
                                        uint32_t* out, float* gumbel,
                                        cudaStream_t stream);

/*
 * dspark_read_device_error -- copies the device error word of `workspace`
 * to the host (synchronising `stream`) and clears it.  Returns DSPARK_OK if
 * no kernel of the last call on this workspace recorded an error,
 * DSPARK_ERR_DEVICE (and *code != 0) if one did.  Every draft-block and
 * sampler call clears the word when it starts, so the code describes the
 * last call only.  Codes: 1 a d0 outside [0, V) (token 0 used), 2 a bounded
 * wait inside a kernel ran out, 3 a per-request temperature that is not
 * finite and positive (1 used), 4 a proposal slot outside [0, num_slots),
 * 5 a sampler position outside [0, 65535] (0 used).  Synchronises
 * `stream`.
 */
DSPARK_API dspark_status dspark_read_device_error(void* workspace, int* code,
                                       cudaStream_t stream);

/* Human-readable name of a status. */
DSPARK_API const char* dspark_status_string(dspark_status status);

/* Library version, "major.minor.patch". */
DSPARK_API const char* dspark_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H_ */
