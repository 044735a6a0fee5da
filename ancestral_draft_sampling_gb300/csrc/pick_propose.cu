// pick_propose.cu -- the cross-chunk pick and the post-block proposal writer.
//
// brb-nv/TensorRT-LLM PR #27, "2. One fused kernel per draft position":
// a small kernel picks the token from the per-chunk statistics, and after
// the block one kernel writes q_k = softmax(logits_k / T) for every position
// from the float32 biased logits, recomputing logits_k / T bit for bit as the
// draw used it.  Greedy requests store a one-hot proposal (PR #27, Test
// Coverage, "Also checked").
#include "dspark_common.cuh"
#include "sm100_ptx.cuh"

namespace dspark {
namespace {

constexpr int kPickThreads = 32;

// One warp per request: merge the chunk statistics of position k from
// buffer buf (merge_row's fixed order), write d_k and the row's (M, S).
// On the tensor-core path (from_keys) d_k is the request's decision key,
// the token the position kernels use; otherwise it is the merged winner,
// and the row U[d_k] that the next position gathers first is prefetched
// into L2.  When launched for programmatic dependent launch the kernel lets
// the next kernel be scheduled at once and waits for the position kernel
// before reading its statistics.
__global__ void __launch_bounds__(kPickThreads)
pick_kernel(DraftArgs a, int k, int n_chunks, int buf, bool from_keys) {
  sm100::launch_dependents();
  sm100::grid_dependency_wait();
  const int b = blockIdx.x;
  const ChunkStat st = merge_row(stat_slot(a.stats, buf, a.B, b, 0), n_chunks,
                                 (int)threadIdx.x);
  const int token = from_keys
                        ? key_token(a.hints[(size_t)b * kHintRowKeys + k])
                        : (st.idx == kNoIndex ? 0 : st.idx);
  if (threadIdx.x == 0) {
    const size_t row = (size_t)b * a.K + k;
    a.tokens[row] = token;
    a.rowstats[2 * row] = st.m;
    a.rowstats[2 * row + 1] = st.s;
  }
  if (!from_keys && k + 1 < a.K) {
    const size_t row_bytes = (size_t)a.r * (a.w_dtype == DSPARK_BF16 ? 2 : 4);
    const char* u = static_cast<const char*>(a.U) + (size_t)token * row_bytes;
    for (size_t off = (size_t)threadIdx.x * 128; off < row_bytes;
         off += (size_t)kPickThreads * 128)
      sm100::prefetch_l2(u + off);
  }
}

constexpr int kPropThreads = 256;
constexpr int kPropN4 = 4;  // float4 per thread (2 and 8 measured slower)
constexpr int kPropPerThread = 4 * kPropN4;

__device__ __forceinline__ float scale(float l, float T) {
  return T == 1.0f ? l : __fdiv_rn(l, T);
}

// One CTA per (row, segment of a row) for positions k_first .. k_first +
// k_count - 1, in a 1-D grid of B * k_count * n_seg CTAs.  The CTAs visit the
// rows of the last position first and, within a row, the highest segment
// first: the position kernel writes its vocab tiles in ascending order, so
// the logits it wrote last are re-read first, while they are still in L2.
// q = exp(s - M) * (1 / S).  Every load of a thread is issued before its
// first store.
template <bool kVec>
__global__ void __launch_bounds__(kPropThreads)
proposals_kernel(DraftArgs a, int k_first, int k_count, int n_seg) {
  const int visit = (int)blockIdx.x / n_seg;        // row in visiting order
  const int seg_idx = n_seg - 1 - ((int)blockIdx.x - visit * n_seg);
  const int kk = k_count - 1 - visit / a.B;          // last position first
  const int b = visit - (visit / a.B) * a.B;
  const int row = b * a.K + k_first + kk;
  const int V = a.V;
  const float M = a.rowstats[2 * (size_t)row];
  const float invS = __frcp_rn(a.rowstats[2 * (size_t)row + 1]);
  const bool greedy = a.greedy != nullptr && a.greedy[b] != 0;
  const int token = greedy ? a.tokens[row] : -1;
  const float* __restrict__ lrow = a.logits + (size_t)row * V;
  // per-request entry point: request b's proposals go to slot slot[b]
  const int k = row - b * a.K;
  int dst = b;
  if (a.slot != nullptr) {
    dst = a.slot[b];
    if (dst < 0 || dst >= a.num_slots) {  // nothing is written for it
      if (k == 0 && seg_idx == 0 && threadIdx.x == 0)
        a.control[0] = kDevErrBadSlot;
      return;
    }
  }
  float* __restrict__ qrow = a.probs + ((size_t)dst * a.K + k) * V;
  const float T = request_temperature(a, b);
  if (a.temperature != nullptr && k == 0 && seg_idx == 0 && threadIdx.x == 0 &&
      T == 1.0f && a.temperature[b] != 1.0f)  // not finite and positive
    a.control[0] = kDevErrBadTemperature;
  const int seg = kPropThreads * kPropPerThread;
  const int v_begin = seg_idx * seg;
  if (kVec) {
    float4 l[kPropN4];
#pragma unroll
    for (int i = 0; i < kPropN4; ++i) {
      const int v = v_begin + (i * kPropThreads + threadIdx.x) * 4;
      if (v < V) l[i] = __ldcs(reinterpret_cast<const float4*>(lrow + v));
    }
#pragma unroll
    for (int i = 0; i < kPropN4; ++i) {
      const int v = v_begin + (i * kPropThreads + threadIdx.x) * 4;
      if (v >= V) break;  // V % 4 == 0: the whole float4 is in range
      float4 q;
      if (greedy) {
        q = make_float4(v == token, v + 1 == token, v + 2 == token, v + 3 == token);
      } else {
        q.x = __fmul_rn(expf(scale(l[i].x, T) - M), invS);
        q.y = __fmul_rn(expf(scale(l[i].y, T) - M), invS);
        q.z = __fmul_rn(expf(scale(l[i].z, T) - M), invS);
        q.w = __fmul_rn(expf(scale(l[i].w, T) - M), invS);
      }
      __stcs(reinterpret_cast<float4*>(qrow + v), q);
    }
  } else {
    for (int i = 0; i < kPropPerThread; ++i) {
      const int v = v_begin + i * kPropThreads + threadIdx.x;
      if (v >= V) break;
      const float q = greedy ? (v == token ? 1.0f : 0.0f)
                             : __fmul_rn(expf(scale(lrow[v], T) - M), invS);
      qrow[v] = q;
    }
  }
}

constexpr int kNoiseThreads = 256;

// folded: the words come from philox_fold / philox_folded, the form the
// position, verification and sampler kernels run (rounds 1-2 folded into
// per-request constants); otherwise from the plain ten-round loop.
__global__ void noise_words_kernel(uint64_t seed, uint64_t offset, int k,
                                   int stream_id, int n, uint32_t* out,
                                   float* gumbel, bool folded) {
  const int v = blockIdx.x * kNoiseThreads + threadIdx.x;
  if (v >= n) return;
  uint4 w;
  if (folded) {
    uint4 pre, rk[4];
    philox_fold(pre, rk, (uint32_t)seed, (uint32_t)(seed >> 32),
                (uint32_t)k | ((uint32_t)stream_id << 16), (uint32_t)offset,
                (uint32_t)(offset >> 32));
    w = philox_folded(pre, rk, (uint32_t)v >> 2);
  } else {
    w = noise_block(seed, offset, k, stream_id, (uint32_t)v >> 2);
  }
  const uint32_t x = word_of(w, v & 3);
  out[v] = x;
  if (gumbel) gumbel[v] = gumbel_from_word(x);
}

}  // namespace

cudaError_t launch_pick(const DraftArgs& a, int k, int n_chunks, int buf,
                        bool from_keys, bool overlap_previous,
                        cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.B, 1, 1);
  cfg.blockDim = dim3(kPickThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_previous ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, pick_kernel, a, k, n_chunks, buf, from_keys);
}

cudaError_t launch_proposals(const DraftArgs& a, int k_first, int k_count,
                             cudaStream_t stream) {
  const int seg = kPropThreads * kPropPerThread;
  const int n_seg = (a.V + seg - 1) / seg;
  const long long ctas = (long long)a.B * k_count * n_seg;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const dim3 grid((unsigned)ctas);
  if (a.V % 4 == 0)
    proposals_kernel<true><<<grid, kPropThreads, 0, stream>>>(a, k_first, k_count, n_seg);
  else
    proposals_kernel<false><<<grid, kPropThreads, 0, stream>>>(a, k_first, k_count, n_seg);
  return cudaGetLastError();
}

cudaError_t launch_noise_words(uint64_t seed, uint64_t offset, int k,
                               int stream_id, int n, uint32_t* out,
                               float* gumbel, bool folded,
                               cudaStream_t stream) {
  noise_words_kernel<<<(n + kNoiseThreads - 1) / kNoiseThreads, kNoiseThreads,
                       0, stream>>>(seed, offset, k, stream_id, n, out, gumbel,
                                    folded);
  return cudaGetLastError();
}

}  // namespace dspark
