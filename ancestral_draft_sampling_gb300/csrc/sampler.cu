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
// proposal writer writes softmax(s) (rows as requests, K = 1).
//
// Each thread keeps its best decision score ref (and index) and a sum
// reference m (its largest s).  One exp2 per entry, f = exp(s - m), feeds the
// sum and a conservative candidate test: an entry can beat ref only if its
// Gumbel score does, i.e. only if w < exp(s - ref) = f exp(m - ref), which
// the test (float)x < 2^32 (1 + 2^-11) f h, h = exp(m - ref), admits with
// room for the rounding of both sides.  Only admitted entries get the exact
// score s + g.
#include "dspark_common.cuh"

namespace dspark {
namespace {

constexpr int kSampleThreads = 256;
constexpr int kSampleWarps = kSampleThreads / 32;
constexpr int kSampleBatch = 2;  // blocks a thread loads before using them
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTestScale = 4297064448.0f;  // 2^32 (1 + 2^-11), exact in float32

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

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
  float ref = -INFINITY;  // best decision score of this thread
  int idx = kNoIndex;
  float m = -INFINITY;    // largest s of this thread: the sum's reference
  float sum = 0.0f;       // sum of exp(s - m)
  float h = INFINITY;     // exp(m - ref), used by the candidate test
  // kSampleBatch blocks per thread and step, every load issued first; the
  // blocks are then taken in the order j, j + threads, ... as one at a time
  for (int j0 = lo + (int)threadIdx.x; j0 < hi; j0 += kSampleBatch * kSampleThreads) {
    float lb[kSampleBatch][4];
#pragma unroll
    for (int u = 0; u < kSampleBatch; ++u) {
      const int j = j0 + u * kSampleThreads, v = 4 * j;
      if (j >= hi) {
#pragma unroll
        for (int e = 0; e < 4; ++e) lb[u][e] = -INFINITY;
      } else if (kVec) {
        const float4 x = __ldcs(reinterpret_cast<const float4*>(lrow) + j);
        lb[u][0] = x.x;
        lb[u][1] = x.y;
        lb[u][2] = x.z;
        lb[u][3] = x.w;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          lb[u][e] = v + e < V ? __ldcs(lrow + v + e) : -INFINITY;
      }
    }
#pragma unroll
    for (int u = 0; u < kSampleBatch; ++u) {
      const int j = j0 + u * kSampleThreads, v = 4 * j;
      if (j >= hi) break;
      const float* l = lb[u];
      float s[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) s[e] = T == 1.0f ? l[e] : __fdiv_rn(l[e], T);
      // the sum's reference moves to a larger s (rare)
      float m4 = m;
#pragma unroll
      for (int e = 0; e < 4; ++e) m4 = s[e] > m4 ? s[e] : m4;  // NaN ignored
      if (m4 > m) {
        sum = __fmul_rn(sum, ex2_approx((m - m4) * kLog2e));  // 0 from -inf
        m = m4;
        h = ex2_approx((m - ref) * kLog2e);
      }
      float f[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)  // -inf -> 0, NaN -> NaN
        f[e] = m == -INFINITY ? (s[e] != s[e] ? s[e] : 0.0f)
                              : ex2_approx((s[e] - m) * kLog2e);
      sum = __fadd_rn(sum, __fadd_rn(__fadd_rn(f[0], f[1]), __fadd_rn(f[2], f[3])));
      if (greedy) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (s[e] > ref) {  // NaN and -inf never win; e ascending keeps the lower
            ref = s[e];
            idx = v + e;
          }
      } else {
        const uint4 w = philox_folded(s_pre, s_rk, (uint32_t)j);
        const float c = kTestScale * h;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t x = word_of(w, e);
          if (__uint2float_rz(x) < __fmul_ru(f[e], c)) {  // a possible winner
            const float sc = __fadd_rn(s[e], gumbel_from_word(x));
            if (sc > ref) {
              ref = sc;
              idx = v + e;
              h = ex2_approx((m - ref) * kLog2e);
            }
          }
        }
      }
    }
  }
  ChunkStat st;
  st.best = ref;
  st.idx = idx;
  st.m = m;
  st.s = sum;
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
