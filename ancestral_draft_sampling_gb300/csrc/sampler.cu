// sampler.cu -- temperature-only target sampling.
//
// brb-nv/TensorRT-LLM PR #27, "1. Temperature-only sampling runs no filter":
// the target side samples with the temperature alone, i.e. softmax and
// sampling, with no top-k, top-p or min-p filter.  A row of target logits is
// drawn like a draft position: s = l / T (float32 IEEE quotient), token =
// argmax of s + g with g the Gumbel variate of the row's counter-based
// Philox noise (stream 3 at the row's position), lowest index on ties
// (argmax of s for a greedy row), probabilities softmax(s).
//
// This kernel writes one chunk statistic per (row, vocab chunk) -- best
// score and index, max and sum-exp of s -- into statistics buffer 0.  The
// pick kernel merges them into the token and the row's (M, S), and the
// proposal writer writes softmax(s) (rows as requests, K = 1).  Every entry
// gets its exact Gumbel score: this is the straightforward form, without
// the position kernel's candidate test.
#include "dspark_common.cuh"

namespace dspark {
namespace {

constexpr int kSampleThreads = 256;
constexpr int kSampleWarps = kSampleThreads / 32;

// grid (n_chunks, R): chunk c of row r covers the Philox blocks (4 entries
// each) [c * chunk_blocks, (c + 1) * chunk_blocks).
template <bool kVec>
__global__ void __launch_bounds__(kSampleThreads)
sample_stats_kernel(DraftArgs a, const int32_t* __restrict__ position,
                    int chunk_blocks) {
  __shared__ uint4 s_pre, s_rk[4];
  __shared__ ChunkStat s_part[kSampleWarps];
  const int row = blockIdx.y, chunk = blockIdx.x;
  const int V = a.V;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* __restrict__ lrow = a.logits + (size_t)row * V;
  const float T = request_temperature(a, row);
  const bool greedy = a.greedy != nullptr && a.greedy[row] != 0;
  if (threadIdx.x == 0) {
    int pos = position != nullptr ? position[row] : 0;
    if (pos < 0 || pos > 0xffff) {
      if (chunk == 0) a.control[0] = kDevErrBadPosition;
      pos = 0;
    }
    const uint64_t sd = a.seed[row], off = a.offset[row];
    philox_fold(s_pre, s_rk, (uint32_t)sd, (uint32_t)(sd >> 32),
                (uint32_t)pos | ((uint32_t)kNoiseTarget << 16), (uint32_t)off,
                (uint32_t)(off >> 32));
  }
  __syncthreads();
  const int n_blk = (V + 3) / 4;
  const int lo = chunk * chunk_blocks;
  const int hi = min(lo + chunk_blocks, n_blk);
  ChunkStat st = empty_stat();
  for (int j = lo + (int)threadIdx.x; j < hi; j += kSampleThreads) {
    const int v = 4 * j;
    float l[4];
    if (kVec) {
      const float4 x = __ldcs(reinterpret_cast<const float4*>(lrow) + j);
      l[0] = x.x;
      l[1] = x.y;
      l[2] = x.z;
      l[3] = x.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) l[e] = v + e < V ? __ldcs(lrow + v + e) : 0.0f;
    }
    float s[4], score[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) s[e] = T == 1.0f ? l[e] : __fdiv_rn(l[e], T);
    if (greedy) {
#pragma unroll
      for (int e = 0; e < 4; ++e) score[e] = s[e];
    } else {
      const uint4 w = philox_folded(s_pre, s_rk, (uint32_t)j);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        score[e] = __fadd_rn(s[e], gumbel_from_word(word_of(w, e)));
    }
    fold4(st, s, score, v, V);
  }
  st = warp_reduce_stat(st);
  if (lane == 0) s_part[warp] = st;
  __syncthreads();
  if (threadIdx.x == 0) {
    ChunkStat r = s_part[0];
    for (int w = 1; w < kSampleWarps; ++w) merge_stat(r, s_part[w]);
    *stat_slot(a.stats, 0, a.B, row, chunk) = r;
  }
}

}  // namespace

// Chunks per row: enough CTAs for several waves over the SMs, at most
// kMaxChunks, and at least 64 Philox blocks (256 entries) per chunk.
int sample_chunks(int R, int V, int sm_count) {
  const int n_blk = (V + 3) / 4;
  int c = (8 * sm_count + R - 1) / R;
  if (c > n_blk / 64) c = n_blk / 64;
  if (c > kMaxChunks) c = kMaxChunks;
  return c < 1 ? 1 : c;
}

cudaError_t launch_sample_stats(const DraftArgs& a, const int32_t* position,
                                int n_chunks, cudaStream_t stream) {
  const int n_blk = (a.V + 3) / 4;
  const int chunk_blocks = (n_blk + n_chunks - 1) / n_chunks;
  const dim3 grid((unsigned)n_chunks, (unsigned)a.B, 1);
  if (a.V % 4 == 0)
    sample_stats_kernel<true><<<grid, kSampleThreads, 0, stream>>>(a, position,
                                                                  chunk_blocks);
  else
    sample_stats_kernel<false><<<grid, kSampleThreads, 0, stream>>>(a, position,
                                                                   chunk_blocks);
  return cudaGetLastError();
}

}  // namespace dspark
