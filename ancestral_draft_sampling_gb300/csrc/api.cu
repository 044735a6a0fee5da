// api.cu -- the C ABI declared in include/dspark.h: argument checks,
// workspace layout and the launch sequence of one draft block.
//
// Launch sequence of dspark_draft_block (brb-nv/TensorRT-LLM PR #27,
// "2. One fused kernel per draft position"): one 2-D memset (the device
// error word and the decision keys), then for k = 0..K-1 one position
// kernel (bias, scaling, Gumbel-max, logits, chunk statistics), one pick
// (token d_k, row max and sum-exp) after the last tensor-core position or
// after every FFMA position, and one proposal writer for all positions.  No
// host synchronisation, so the whole call can be captured in a CUDA graph.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "dspark_common.cuh"

namespace dspark {
int generic_chunks_used(int V, int n_chunks);
}

namespace {

using namespace dspark;

bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

bool sizes_supported(int B, int K, int V, int r) {
  return B >= 1 && B <= DSPARK_MAX_B && K >= 1 && K <= DSPARK_MAX_K &&
         V >= 1 && V <= DSPARK_MAX_V && r >= 16 && r <= DSPARK_MAX_R &&
         r % 16 == 0;
}

// Streaming multiprocessors of the current device (cached per device).
int sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
            cudaSuccess ||
        n <= 0)
      n = 1;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

dspark_status from_cuda(cudaError_t e) {
  return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

// Checks the arguments of dspark_draft_block and fills the kernel arguments.
dspark_status prepare_draft(
    const void* base_logits, dspark_dtype base_dtype, const void* U,
    const void* Wb, dspark_dtype w_dtype, const int32_t* d0,
    const uint64_t* seed, const uint64_t* offset, float T,
    const uint8_t* greedy, const uint8_t* pad_row, int B, int K, int V, int r,
    int32_t* tokens, float* logits, float* draft_probs, void* workspace,
    size_t workspace_bytes, DraftArgs& a) {
  // ---- argument checks, before any launch
  if (B <= 0 || K <= 0 || V <= 0 || r <= 0) return DSPARK_ERR_INVALID_ARG;
  if (!base_logits || !U || !Wb || !d0 || !seed || !offset || !tokens ||
      !logits || !draft_probs)
    return DSPARK_ERR_INVALID_ARG;
  if (!(T > 0.0f) || !std::isfinite(T)) return DSPARK_ERR_INVALID_ARG;
  if ((base_dtype != DSPARK_F32 && base_dtype != DSPARK_BF16) ||
      (w_dtype != DSPARK_F32 && w_dtype != DSPARK_BF16))
    return DSPARK_ERR_INVALID_ARG;
  const void* ptrs[] = {base_logits, U, Wb, d0, seed, offset, tokens, logits,
                        draft_probs, greedy, pad_row, workspace};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return DSPARK_ERR_INVALID_ARG;
  if (!sizes_supported(B, K, V, r)) return DSPARK_ERR_UNSUPPORTED;
  const WorkspaceLayout L = workspace_layout(B, K);
  if (!workspace || workspace_bytes < L.total ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return DSPARK_ERR_WORKSPACE;

  a.base = base_logits;
  a.base_dtype = base_dtype;
  a.U = U;
  a.Wb = Wb;
  a.w_dtype = w_dtype;
  a.d0 = d0;
  a.seed = seed;
  a.offset = offset;
  a.T = T;
  a.greedy = greedy;
  a.pad_row = pad_row;
  a.B = B;
  a.K = K;
  a.V = V;
  a.r = r;
  a.tokens = tokens;
  a.logits = logits;
  a.probs = draft_probs;
  char* ws = static_cast<char*>(workspace);
  a.stats = reinterpret_cast<ChunkStat*>(ws + L.stats);
  a.rowstats = reinterpret_cast<float*>(ws + L.rowstats);
  a.hints = reinterpret_cast<unsigned long long*>(ws + L.hints);
  a.control = reinterpret_cast<int*>(ws + L.control);

  return DSPARK_OK;
}

// Event pairs around each kernel class: [0] position kernels, [1] picks,
// [2] proposal writer.  Accumulated milliseconds are returned.
struct StageTimer {
  std::vector<cudaEvent_t> ev;  // two per launch
  std::vector<int> cls;         // one per launch
  int n = 0;
};

dspark_status timed_launch(StageTimer* t, int cls, cudaStream_t stream,
                           cudaError_t (*fn)(const DraftArgs&, int, int,
                                             cudaStream_t),
                           const DraftArgs& a, int k, int n) {
  if (t) {
    if (t->n >= (int)t->cls.size()) return DSPARK_ERR_INVALID_ARG;
    if (cudaEventRecord(t->ev[2 * t->n], stream) != cudaSuccess)
      return DSPARK_ERR_CUDA;
  }
  dspark_status st = from_cuda(fn(a, k, n, stream));
  if (st != DSPARK_OK) return st;
  if (t) {
    if (cudaEventRecord(t->ev[2 * t->n + 1], stream) != cudaSuccess)
      return DSPARK_ERR_CUDA;
    t->cls[t->n++] = cls;
  }
  return DSPARK_OK;
}

// The pick of the last tensor-core position overlaps that kernel's end (both
// are launched for programmatic dependent launch) and takes d_{K-1} from the
// decision keys; after each FFMA position the pick is an ordinary launch
// and merges the winner from the statistics.
cudaError_t launch_pick_keys(const DraftArgs& a, int k, int n,
                             cudaStream_t s) {
  return launch_pick(a, k, n, k & 1, true, true, s);
}

cudaError_t launch_pick_plain(const DraftArgs& a, int k, int n,
                              cudaStream_t s) {
  return launch_pick(a, k, n, 0, false, false, s);
}

cudaError_t proposals_adapter(const DraftArgs& a, int, int, cudaStream_t s) {
  return launch_proposals(a, 0, a.K, s);
}

// Which position kernel runs: the tensor-core kernel when the shape allows
// it, else the FFMA kernel.  DSPARK_POSITION_KERNEL=generic forces the FFMA
// kernel (for comparisons); =tc fails with UNSUPPORTED where it cannot run.
int position_kernel_choice(const DraftArgs& a) {
  const char* env = std::getenv("DSPARK_POSITION_KERNEL");
  const bool tc_ok = position_tc_supported(a);
  if (env && std::strcmp(env, "generic") == 0) return 0;
  if (env && std::strcmp(env, "tc") == 0) return tc_ok ? 1 : -1;
  return tc_ok ? 1 : 0;
}

// Host-memory drafter logits of dspark_draft_block_host: position k's slice
// is copied on copy_stream into a.base and signalled by ready[k]; ready[K]
// orders the copies after the caller's earlier work on the compute stream.
struct HostFeed {
  const char* base_host;  // [B,K,V]
  size_t elt;
  cudaStream_t copy_stream;
  cudaEvent_t* ready;     // K + 1 events
};

// Requests b0 .. b0 + n - 1 of a block as a block of their own: the same
// heads, workspace statistics and error word; their rows of every other
// array (per-request slots index the full proposal array).
DraftArgs request_group(const DraftArgs& a, int b0, int n) {
  DraftArgs g = a;
  const size_t rows = (size_t)b0 * a.K;
  const size_t elt = a.base_dtype == DSPARK_F32 ? 4 : 2;
  g.B = n;
  g.base = static_cast<const char*>(a.base) + rows * a.V * elt;
  g.d0 = a.d0 + b0;
  g.seed = a.seed + b0;
  g.offset = a.offset + b0;
  if (a.greedy) g.greedy = a.greedy + b0;
  if (a.pad_row) g.pad_row = a.pad_row + b0;
  if (a.temperature) g.temperature = a.temperature + b0;
  g.tokens = a.tokens + rows;
  g.logits = a.logits + rows * a.V;
  if (a.slot) g.slot = a.slot + b0;
  else if (a.probs) g.probs = a.probs + rows * a.V;
  g.rowstats = a.rowstats + rows * 2;
  g.hints = a.hints + (size_t)b0 * kHintRowKeys;
  return g;
}

// Launches one draft block makes (an upper bound when the kernel is not
// yet known): per request group, K positions and K picks at most, then the
// proposal writer.
int block_launch_bound(int B, int K) {
  return position_tc_groups(B) * 2 * K + 1;
}

// The launch sequence of one draft block.  chain_end (measurement only):
// an event recorded as an external event node between the position chain
// (the memset, the positions and their picks) and the proposal writer.
// A block of more requests than the tensor-core kernel takes in one launch
// runs as consecutive request groups (position_tc_groups), each its own
// chain of positions over the same heads; the proposal writer then covers
// all rows at once.
dspark_status run_block(const DraftArgs& a, cudaStream_t stream,
                        StageTimer* t, const HostFeed* feed = nullptr,
                        cudaEvent_t chain_end = nullptr) {
  const int sms = sm_count() < kMaxChunks ? sm_count() : kMaxChunks;
  const int choice = position_kernel_choice(a);
  if (choice < 0) return DSPARK_ERR_UNSUPPORTED;
  const bool tc = choice == 1;
  // position kernels fill n_chunks statistics slots per request; they are
  // merged in slot order
  const int want = tc ? position_tc_chunks(a.V, sms) : sms;
  const int n_chunks = tc ? want : generic_chunks_used(a.V, want);
  // One 2-D memset over the control row and the B key rows (one pitch):
  // the device error word starts every block at 0, and the decision keys of
  // every position at zero (no winner).
  if (cudaMemset2DAsync(a.control, kHintRowBytes, 0,
                        (size_t)a.K * sizeof(uint64_t), (size_t)a.B + 1,
                        stream) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (feed) {
    // position k's drafter logits: B rows of V values, K V apart
    const size_t row = (size_t)a.V * feed->elt, pitch = (size_t)a.K * row;
    if (cudaEventRecord(feed->ready[a.K], stream) != cudaSuccess ||
        cudaStreamWaitEvent(feed->copy_stream, feed->ready[a.K], 0) != cudaSuccess)
      return DSPARK_ERR_CUDA;
    char* dst = static_cast<char*>(const_cast<void*>(a.base));
    for (int k = 0; k < a.K; ++k) {
      if (cudaMemcpy2DAsync(dst + k * row, pitch, feed->base_host + k * row,
                            pitch, row, a.B, cudaMemcpyHostToDevice,
                            feed->copy_stream) != cudaSuccess ||
          cudaEventRecord(feed->ready[k], feed->copy_stream) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    }
  }
  // Tensor-core positions follow one another directly: position k reads
  // d_{k-1} from the decision keys and merges position k-1's statistics
  // itself; one pick after the last position finishes the block.  Each
  // FFMA position is followed by its pick.
  const int n_groups = tc ? position_tc_groups(a.B) : 1;
  const int per_group = (a.B + n_groups - 1) / n_groups;
  for (int b0 = 0; b0 < a.B; b0 += per_group) {
    const DraftArgs g = n_groups == 1 ? a
                                      : request_group(a, b0, std::min(per_group, a.B - b0));
    for (int k = 0; k < g.K; ++k) {
      if (feed && cudaStreamWaitEvent(stream, feed->ready[k], 0) != cudaSuccess)
        return DSPARK_ERR_CUDA;
      dspark_status st = timed_launch(
          t, 0, stream, tc ? launch_position_tc : launch_position_generic, g, k,
          want);
      if (st != DSPARK_OK) return st;
      if (!tc || k == g.K - 1) {
        st = timed_launch(t, 1, stream, tc ? launch_pick_keys : launch_pick_plain,
                          g, k, n_chunks);
        if (st != DSPARK_OK) return st;
      }
      // with host-fed logits the GPU would idle until the next slice
      // arrives: write each position's proposals as soon as its (M, S)
      // exist (after its pick, or after the next tensor-core position has
      // merged them)
      if (feed) {
        int lo = k, hi = k;  // FFMA: position k's pick has just run
        if (tc) {            // position k merged k-1; the last pick ran for K-1
          lo = k - 1 < 0 ? 0 : k - 1;
          hi = k == g.K - 1 ? k : k - 1;
        }
        if (hi >= lo &&
            from_cuda(launch_proposals(g, lo, hi - lo + 1, stream)) != DSPARK_OK)
          return DSPARK_ERR_CUDA;
      }
    }
  }
  if (feed) return DSPARK_OK;
  if (chain_end && cudaEventRecordWithFlags(chain_end, stream,
                                            cudaEventRecordExternal) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  return timed_launch(t, 2, stream, proposals_adapter, a, 0, 0);
}

// dspark_draft_block_timeline: the block captured once into a CUDA graph
// with event nodes at its start, between the position chain and the
// proposal writer, and at its end; the graph is replayed and the two
// segments timed per replay.
dspark_status timeline(const DraftArgs& a, int replays, float* chain_ms,
                       float* proposal_ms, cudaStream_t stream) {
  cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  dspark_status st = DSPARK_OK;
  for (int i = 0; i < 3 && st == DSPARK_OK; ++i)
    if (cudaEventCreate(&ev[i]) != cudaSuccess) st = DSPARK_ERR_CUDA;
  if (st == DSPARK_OK &&
      cudaStreamBeginCapture(stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
    st = DSPARK_ERR_CUDA;
  if (st == DSPARK_OK) {
    dspark_status cap = from_cuda(
        cudaEventRecordWithFlags(ev[0], stream, cudaEventRecordExternal));
    if (cap == DSPARK_OK) cap = run_block(a, stream, nullptr, nullptr, ev[1]);
    if (cap == DSPARK_OK)
      cap = from_cuda(
          cudaEventRecordWithFlags(ev[2], stream, cudaEventRecordExternal));
    // the capture is ended in every case, so the stream leaves capture mode
    const cudaError_t end = cudaStreamEndCapture(stream, &graph);
    st = cap != DSPARK_OK ? cap : from_cuda(end);
  }
  if (st == DSPARK_OK &&
      cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess)
    st = DSPARK_ERR_CUDA;
  double chain = 0.0, prop = 0.0;
  for (int i = 0; i < replays && st == DSPARK_OK; ++i) {
    float m0 = 0.0f, m1 = 0.0f;
    if (cudaGraphLaunch(exec, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess ||
        cudaEventElapsedTime(&m0, ev[0], ev[1]) != cudaSuccess ||
        cudaEventElapsedTime(&m1, ev[1], ev[2]) != cudaSuccess) {
      st = DSPARK_ERR_CUDA;
      break;
    }
    chain += m0;
    prop += m1;
  }
  if (st == DSPARK_OK) {
    *chain_ms = (float)(chain / replays);
    *proposal_ms = (float)(prop / replays);
  }
  if (exec) cudaGraphExecDestroy(exec);
  if (graph) cudaGraphDestroy(graph);
  for (int i = 0; i < 3; ++i)
    if (ev[i]) cudaEventDestroy(ev[i]);
  return st;
}

// Device workspace of dspark_draft_block_host: the draft workspace, then the
// per-request inputs and the tokens.
struct HostLayout {
  size_t d0, seed, offset, greedy, pad_row, tokens, total;
};

HostLayout host_layout(int B, int K) {
  HostLayout H;
  size_t off = workspace_layout(B, K).total;
  H.d0 = off;
  off = align_up(off + (size_t)B * sizeof(int32_t), 256);
  H.seed = off;
  off = align_up(off + (size_t)B * sizeof(uint64_t), 256);
  H.offset = off;
  off = align_up(off + (size_t)B * sizeof(uint64_t), 256);
  H.greedy = off;
  off = align_up(off + (size_t)B, 256);
  H.pad_row = off;
  off = align_up(off + (size_t)B, 256);
  H.tokens = off;
  off = align_up(off + (size_t)B * K * sizeof(int32_t), 256);
  H.total = off;
  return H;
}

// ---------------------------------------------------- allocation-free scratch
// The scratch of dspark_draft_block_noalloc: one file-scope device array,
// loaded with the library on every GPU that uses it and held until exit.
constexpr size_t kNoallocScratchBytes = size_t(2) << 20;  // 2 MiB
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch on the current device.  The symbol
// name is a host-side stand-in, never a device address, so it is resolved
// with the device current.  Outside stream capture it is looked up on every
// call (cheap; a device reset or a new primary context moves it) and
// cached per device; during a capture the cached address is used, so the
// first call on a device must come before any capture.
cudaError_t noalloc_scratch(cudaStream_t stream, void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (cap == cudaStreamCaptureStatusNone || addr[dev] == nullptr) {
    if (cap != cudaStreamCaptureStatusNone) return cudaErrorStreamCaptureUnsupported;
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

// The argument checks and launch shared by the two verification rules.
dspark_status verify_rule(const float* draft_probs, const float* target_probs,
                          const int32_t* tokens, const uint64_t* seed,
                          const uint64_t* offset, int B, int K, int V,
                          int32_t* accepted_len, int32_t* emitted_token,
                          bool block, cudaStream_t stream) {
  if (B <= 0 || K <= 0 || V <= 0) return DSPARK_ERR_INVALID_ARG;
  if (!draft_probs || !target_probs || !tokens || !seed || !offset ||
      !accepted_len || !emitted_token)
    return DSPARK_ERR_INVALID_ARG;
  const void* ptrs[] = {draft_probs, target_probs, tokens, seed,
                        offset, accepted_len, emitted_token};
  for (const void* p : ptrs)
    if (!aligned16(p)) return DSPARK_ERR_INVALID_ARG;
  if (B > 65535 || K > DSPARK_MAX_K || V > DSPARK_MAX_V)
    return DSPARK_ERR_UNSUPPORTED;
  return from_cuda(launch_verify(draft_probs, target_probs, tokens, seed,
                                 offset, B, K, V, accepted_len, emitted_token,
                                 sm_count(), block, stream));
}

}  // namespace

extern "C" {

const char* dspark_version(void) { return "0.1.0"; }

const char* dspark_status_string(dspark_status status) {
  switch (status) {
    case DSPARK_OK: return "DSPARK_OK";
    case DSPARK_ERR_INVALID_ARG: return "DSPARK_ERR_INVALID_ARG";
    case DSPARK_ERR_UNSUPPORTED: return "DSPARK_ERR_UNSUPPORTED";
    case DSPARK_ERR_WORKSPACE: return "DSPARK_ERR_WORKSPACE";
    case DSPARK_ERR_CUDA: return "DSPARK_ERR_CUDA";
    case DSPARK_ERR_DEVICE: return "DSPARK_ERR_DEVICE";
  }
  return "DSPARK_UNKNOWN_STATUS";
}

size_t dspark_draft_workspace_bytes(int B, int K, int V, int r) {
  if (!sizes_supported(B, K, V, r)) return 0;
  return workspace_layout(B, K).total;
}

dspark_status dspark_draft_block(
    const void* base_logits, dspark_dtype base_dtype, const void* U,
    const void* Wb, dspark_dtype w_dtype, const int32_t* d0,
    const uint64_t* seed, const uint64_t* offset, float T,
    const uint8_t* greedy, const uint8_t* pad_row, int B, int K, int V, int r,
    int32_t* tokens, float* logits, float* draft_probs, void* workspace,
    size_t workspace_bytes, cudaStream_t stream) {
  DraftArgs a{};
  dspark_status st = prepare_draft(
      base_logits, base_dtype, U, Wb, w_dtype, d0, seed, offset, T, greedy,
      pad_row, B, K, V, r, tokens, logits, draft_probs, workspace,
      workspace_bytes, a);
  if (st != DSPARK_OK) return st;
  return run_block(a, stream, nullptr);
}

dspark_status dspark_draft_block_per_request(
    const void* base_logits, dspark_dtype base_dtype, const void* U,
    const void* Wb, dspark_dtype w_dtype, const int32_t* d0,
    const uint64_t* seed, const uint64_t* offset, const float* temperature,
    const uint8_t* greedy, const uint8_t* pad_row, int B, int K, int V, int r,
    int32_t* tokens, float* logits, float* draft_probs, const int32_t* slot,
    int num_slots, void* workspace, size_t workspace_bytes,
    cudaStream_t stream) {
  if (!temperature || (reinterpret_cast<uintptr_t>(temperature) & 3u) != 0)
    return DSPARK_ERR_INVALID_ARG;
  if (slot && ((reinterpret_cast<uintptr_t>(slot) & 3u) != 0 || num_slots <= 0 ||
               num_slots > 65535 * 16))
    return DSPARK_ERR_INVALID_ARG;
  DraftArgs a{};
  // T = 2 only passes the scalar check; every kernel reads temperature[b]
  dspark_status st = prepare_draft(
      base_logits, base_dtype, U, Wb, w_dtype, d0, seed, offset, 2.0f, greedy,
      pad_row, B, K, V, r, tokens, logits, draft_probs, workspace,
      workspace_bytes, a);
  if (st != DSPARK_OK) return st;
  a.temperature = temperature;
  a.slot = slot;
  a.num_slots = slot ? num_slots : 0;
  return run_block(a, stream, nullptr);
}

dspark_status dspark_draft_block_profile(
    const void* base_logits, dspark_dtype base_dtype, const void* U,
    const void* Wb, dspark_dtype w_dtype, const int32_t* d0,
    const uint64_t* seed, const uint64_t* offset, float T,
    const uint8_t* greedy, const uint8_t* pad_row, int B, int K, int V, int r,
    int32_t* tokens, float* logits, float* draft_probs, void* workspace,
    size_t workspace_bytes, float* stage_ms, int* stage_launches,
    cudaStream_t stream) {
  if (!stage_ms || !stage_launches) return DSPARK_ERR_INVALID_ARG;
  DraftArgs a{};
  dspark_status st = prepare_draft(
      base_logits, base_dtype, U, Wb, w_dtype, d0, seed, offset, T, greedy,
      pad_row, B, K, V, r, tokens, logits, draft_probs, workspace,
      workspace_bytes, a);
  if (st != DSPARK_OK) return st;
  StageTimer t;
  const int n_launch = block_launch_bound(B, K);
  const int n_ev = 2 * n_launch;
  t.ev.assign(n_ev, nullptr);
  t.cls.assign(n_launch, 0);
  int created = 0;
  for (; created < n_ev; ++created)
    if (cudaEventCreate(&t.ev[created]) != cudaSuccess) break;
  if (created == n_ev) st = run_block(a, stream, &t);
  else st = DSPARK_ERR_CUDA;
  if (st == DSPARK_OK && cudaStreamSynchronize(stream) != cudaSuccess)
    st = DSPARK_ERR_CUDA;
  for (int c = 0; c < 3; ++c) {
    stage_ms[c] = 0.0f;
    stage_launches[c] = 0;
  }
  for (int i = 0; st == DSPARK_OK && i < t.n; ++i) {
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, t.ev[2 * i], t.ev[2 * i + 1]) != cudaSuccess)
      st = DSPARK_ERR_CUDA;
    stage_ms[t.cls[i]] += ms;
    stage_launches[t.cls[i]] += 1;
  }
  for (int i = 0; i < created; ++i) cudaEventDestroy(t.ev[i]);
  return st;
}

dspark_status dspark_draft_block_timeline(
    const void* base_logits, dspark_dtype base_dtype, const void* U,
    const void* Wb, dspark_dtype w_dtype, const int32_t* d0,
    const uint64_t* seed, const uint64_t* offset, float T,
    const uint8_t* greedy, const uint8_t* pad_row, int B, int K, int V, int r,
    int32_t* tokens, float* logits, float* draft_probs, void* workspace,
    size_t workspace_bytes, int replays, float* chain_ms, float* proposal_ms,
    cudaStream_t stream) {
  if (!chain_ms || !proposal_ms || replays < 1 || stream == nullptr)
    return DSPARK_ERR_INVALID_ARG;
  DraftArgs a{};
  dspark_status st = prepare_draft(
      base_logits, base_dtype, U, Wb, w_dtype, d0, seed, offset, T, greedy,
      pad_row, B, K, V, r, tokens, logits, draft_probs, workspace,
      workspace_bytes, a);
  if (st != DSPARK_OK) return st;
  return timeline(a, replays, chain_ms, proposal_ms, stream);
}

dspark_status dspark_draft_block_noalloc(
    const void* base_logits, dspark_dtype base_dtype, const void* U,
    const void* Wb, dspark_dtype w_dtype, const int32_t* d0,
    const uint64_t* seed, const uint64_t* offset, float T,
    const uint8_t* greedy, const uint8_t* pad_row, int B, int K, int V, int r,
    int32_t* tokens, float* logits, float* draft_probs, cudaStream_t stream) {
  // host-side checks first, against a stand-in scratch address
  DraftArgs a{};
  void* const stand_in = reinterpret_cast<void*>(uintptr_t(256));
  dspark_status st = prepare_draft(
      base_logits, base_dtype, U, Wb, w_dtype, d0, seed, offset, T, greedy,
      pad_row, B, K, V, r, tokens, logits, draft_probs, stand_in,
      kNoallocScratchBytes, a);
  if (st != DSPARK_OK) return st;  // sizes past the scratch: WORKSPACE
  void* scratch = nullptr;
  if (noalloc_scratch(stream, &scratch) != cudaSuccess) return DSPARK_ERR_CUDA;
  st = prepare_draft(base_logits, base_dtype, U, Wb, w_dtype, d0, seed,
                     offset, T, greedy, pad_row, B, K, V, r, tokens, logits,
                     draft_probs, scratch, kNoallocScratchBytes, a);
  if (st != DSPARK_OK) return st;
  // the scratch keeps the previous call's contents: only the device error
  // word and the decision keys must start at zero, and the block's first
  // launch clears them (every other word is written before it is read)
  return run_block(a, stream, nullptr);
}

size_t dspark_draft_host_workspace_bytes(int B, int K, int V, int r) {
  if (!sizes_supported(B, K, V, r)) return 0;
  return host_layout(B, K).total;
}

dspark_status dspark_draft_block_host(
    const void* base_logits_host, dspark_dtype base_dtype, const void* U,
    const void* Wb, dspark_dtype w_dtype, const int32_t* d0_host,
    const uint64_t* seed_host, const uint64_t* offset_host, float T,
    const uint8_t* greedy_host, const uint8_t* pad_row_host, int B, int K,
    int V, int r, void* base_dev, int32_t* tokens_host, float* logits,
    float* draft_probs, void* workspace, size_t workspace_bytes,
    cudaStream_t stream, cudaStream_t copy_stream) {
  if (!base_logits_host || !d0_host || !seed_host || !offset_host ||
      !tokens_host || !base_dev || stream == copy_stream)
    return DSPARK_ERR_INVALID_ARG;
  if (B <= 0 || K <= 0 || V <= 0 || r <= 0) return DSPARK_ERR_INVALID_ARG;
  if (!sizes_supported(B, K, V, r)) return DSPARK_ERR_UNSUPPORTED;
  const HostLayout H = host_layout(B, K);
  if (!workspace || workspace_bytes < H.total ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return DSPARK_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  int32_t* d0 = reinterpret_cast<int32_t*>(ws + H.d0);
  uint64_t* seed = reinterpret_cast<uint64_t*>(ws + H.seed);
  uint64_t* offset = reinterpret_cast<uint64_t*>(ws + H.offset);
  uint8_t* greedy = greedy_host ? reinterpret_cast<uint8_t*>(ws + H.greedy) : nullptr;
  uint8_t* pad_row = pad_row_host ? reinterpret_cast<uint8_t*>(ws + H.pad_row) : nullptr;
  int32_t* tokens = reinterpret_cast<int32_t*>(ws + H.tokens);
  DraftArgs a{};
  dspark_status st = prepare_draft(
      base_dev, base_dtype, U, Wb, w_dtype, d0, seed, offset, T, greedy,
      pad_row, B, K, V, r, tokens, logits, draft_probs, workspace,
      workspace_bytes, a);
  if (st != DSPARK_OK) return st;
  // the per-request inputs, ahead of the first position on `stream`
  const struct { void* dst; const void* src; size_t n; } small[] = {
      {d0, d0_host, (size_t)B * sizeof(int32_t)},
      {seed, seed_host, (size_t)B * sizeof(uint64_t)},
      {offset, offset_host, (size_t)B * sizeof(uint64_t)},
      {greedy, greedy_host, (size_t)B},
      {pad_row, pad_row_host, (size_t)B}};
  for (const auto& c : small)
    if (c.src && cudaMemcpyAsync(c.dst, c.src, c.n, cudaMemcpyHostToDevice,
                                 stream) != cudaSuccess)
      return DSPARK_ERR_CUDA;
  cudaEvent_t ready[DSPARK_MAX_K + 1];
  int created = 0;
  for (; created <= K; ++created)
    if (cudaEventCreateWithFlags(&ready[created], cudaEventDisableTiming) !=
        cudaSuccess)
      break;
  if (created == K + 1) {
    const HostFeed feed{static_cast<const char*>(base_logits_host),
                        base_dtype == DSPARK_F32 ? (size_t)4 : (size_t)2,
                        copy_stream, ready};
    st = run_block(a, stream, nullptr, &feed);
    if (st == DSPARK_OK &&
        cudaMemcpyAsync(tokens_host, tokens, (size_t)B * K * sizeof(int32_t),
                        cudaMemcpyDeviceToHost, stream) != cudaSuccess)
      st = DSPARK_ERR_CUDA;
  } else {
    st = DSPARK_ERR_CUDA;
  }
  // an event still pending is released by the runtime once it completes
  for (int i = 0; i < created; ++i) cudaEventDestroy(ready[i]);
  return st;
}

dspark_status dspark_verify_standard(const float* draft_probs,
                                     const float* target_probs,
                                     const int32_t* tokens,
                                     const uint64_t* seed,
                                     const uint64_t* offset, int B, int K,
                                     int V, int32_t* accepted_len,
                                     int32_t* emitted_token,
                                     cudaStream_t stream) {
  return verify_rule(draft_probs, target_probs, tokens, seed, offset, B, K, V,
                     accepted_len, emitted_token, false, stream);
}

dspark_status dspark_verify_block(const float* draft_probs,
                                  const float* target_probs,
                                  const int32_t* tokens, const uint64_t* seed,
                                  const uint64_t* offset, int B, int K, int V,
                                  int32_t* accepted_len, int32_t* emitted_token,
                                  cudaStream_t stream) {
  return verify_rule(draft_probs, target_probs, tokens, seed, offset, B, K, V,
                     accepted_len, emitted_token, true, stream);
}

size_t dspark_sample_workspace_bytes(int R, int V) {
  if (R < 1 || R > 65535 || V < 1 || V > DSPARK_MAX_V) return 0;
  return workspace_layout(R, 1).total;
}

dspark_status dspark_sample_temperature(
    const float* logits, const float* temperature, float T,
    const uint8_t* greedy, const uint64_t* seed, const uint64_t* offset,
    const int32_t* position, int R, int V, int32_t* tokens, float* probs,
    void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (R <= 0 || V <= 0 || !logits || !seed || !offset || !tokens)
    return DSPARK_ERR_INVALID_ARG;
  if (!temperature && (!(T > 0.0f) || !std::isfinite(T)))
    return DSPARK_ERR_INVALID_ARG;
  const void* ptrs16[] = {logits, seed, offset, tokens, probs, workspace};
  for (const void* p : ptrs16)
    if (p && !aligned16(p)) return DSPARK_ERR_INVALID_ARG;
  const void* ptrs4[] = {temperature, position};
  for (const void* p : ptrs4)
    if (p && (reinterpret_cast<uintptr_t>(p) & 3u) != 0)
      return DSPARK_ERR_INVALID_ARG;
  if (R > 65535 || V > DSPARK_MAX_V) return DSPARK_ERR_UNSUPPORTED;
  const WorkspaceLayout L = workspace_layout(R, 1);
  if (!workspace || workspace_bytes < L.total ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return DSPARK_ERR_WORKSPACE;
  // rows as requests of a one-position block: the pick and the proposal
  // writer of the draft block finish the rows
  DraftArgs a{};
  a.logits = const_cast<float*>(logits);
  a.probs = probs;
  a.tokens = tokens;
  a.seed = seed;
  a.offset = offset;
  a.greedy = greedy;
  a.T = temperature ? 1.0f : T;
  a.temperature = temperature;
  a.B = R;
  a.K = 1;
  a.V = V;
  a.r = 16;
  char* ws = static_cast<char*>(workspace);
  a.stats = reinterpret_cast<ChunkStat*>(ws + L.stats);
  a.rowstats = reinterpret_cast<float*>(ws + L.rowstats);
  a.hints = reinterpret_cast<unsigned long long*>(ws + L.hints);
  a.control = reinterpret_cast<int*>(ws + L.control);
  const int sms = sm_count();
  const int n_chunks = sample_chunks(R, V, sms);
  // the device error word starts every call at 0
  if (cudaMemsetAsync(a.control, 0, sizeof(int), stream) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  dspark_status st = from_cuda(launch_sample_stats(a, position, n_chunks, stream));
  if (st != DSPARK_OK) return st;
  st = from_cuda(launch_pick(a, 0, n_chunks, 0, false, false, stream));
  if (st != DSPARK_OK || !probs) return st;
  return from_cuda(launch_proposals(a, 0, 1, stream));
}

namespace {
dspark_status noise_words(uint64_t seed, uint64_t offset, int k, int stream_id,
                          int n, uint32_t* out, float* gumbel, bool folded,
                          cudaStream_t stream) {
  if (n <= 0 || !out || k < 0 || k > 0xffff || stream_id < 0 ||
      stream_id > 0xffff)
    return DSPARK_ERR_INVALID_ARG;
  if (!aligned16(out) || (gumbel && !aligned16(gumbel)))
    return DSPARK_ERR_INVALID_ARG;
  return from_cuda(launch_noise_words(seed, offset, k, stream_id, n, out,
                                      gumbel, folded, stream));
}
}  // namespace

dspark_status dspark_noise_words(uint64_t seed, uint64_t offset, int k,
                                 int stream_id, int n, uint32_t* out,
                                 float* gumbel, cudaStream_t stream) {
  return noise_words(seed, offset, k, stream_id, n, out, gumbel, false,
                     stream);
}

dspark_status dspark_noise_words_folded(uint64_t seed, uint64_t offset, int k,
                                        int stream_id, int n, uint32_t* out,
                                        float* gumbel, cudaStream_t stream) {
  return noise_words(seed, offset, k, stream_id, n, out, gumbel, true, stream);
}

dspark_status dspark_read_device_error(void* workspace, int* code,
                                       cudaStream_t stream) {
  if (!workspace || !code) return DSPARK_ERR_INVALID_ARG;
  // the error word is the first int of the control block at offset 0
  int host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, workspace, sizeof(int),
                                  cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return DSPARK_ERR_CUDA;
  *code = host;
  if (host == 0) return DSPARK_OK;
  e = cudaMemsetAsync(workspace, 0, sizeof(int), stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return e == cudaSuccess ? DSPARK_ERR_DEVICE : DSPARK_ERR_CUDA;
}

}  // extern "C"
