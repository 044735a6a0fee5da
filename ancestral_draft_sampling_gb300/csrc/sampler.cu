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
// A row chunk is swept by the warp draw of gumbel_draw.cuh.  With the
// reference shared by the 32 lanes, a warp meets an admitted entry in a few
// of its steps only (a reference per lane admitted one in most steps of
// some lane, and the whole warp ran the exact path).
#include "dspark_common.cuh"
#include "gumbel_draw.cuh"

namespace dspark {
namespace {

constexpr int kSampleThreads = 256;
constexpr int kSampleWarps = kSampleThreads / 32;
constexpr int kSampleBatch = 2;  // blocks a thread loads before using them
constexpr int kSampleMinBlocks = 5;  // resident CTAs per SM (48 registers)

// Thread 0: the row's noise constants (stream 3 at the row's position).
__device__ __forceinline__ void row_noise_setup(const DraftArgs& a,
                                                const int32_t* position,
                                                int row, int chunk, uint4& pre,
                                                uint4 (&rk)[4]) {
  int pos = position != nullptr ? position[row] : 0;
  if (pos < 0 || pos > 0xffff) {
    if (chunk == 0) a.control[0] = kDevErrBadPosition;
    pos = 0;
  }
  const uint64_t sd = a.seed[row], off = a.offset[row];
  philox_fold(pre, rk, (uint32_t)sd, (uint32_t)(sd >> 32),
              (uint32_t)pos | ((uint32_t)kNoiseTarget << 16), (uint32_t)off,
              (uint32_t)(off >> 32));
}

// The chunk statistic: warps reduce by a butterfly, then thread 0 merges
// the warps in order and stores it.
__device__ __forceinline__ void chunk_stat_out(const DraftArgs& a, int row,
                                               int chunk, const SampleState& ss,
                                               ChunkStat (&part)[kSampleWarps]) {
  ChunkStat st;
  st.best = ss.ref;
  st.idx = ss.idx;
  st.m = ss.m;
  st.s = ss.sum;
  st = warp_reduce_stat(st);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = st;
  __syncthreads();
  if (threadIdx.x == 0) {
    ChunkStat r = part[0];
    for (int w = 1; w < kSampleWarps; ++w) merge_stat(r, part[w]);
    *stat_slot(a.stats, 0, a.B, row, chunk) = r;
  }
}

// grid (n_chunks, R): chunk c of row r covers the Philox blocks (4 entries
// each) [c * chunk_blocks, (c + 1) * chunk_blocks).  Thread t of the CTA
// takes the blocks lo + t, lo + t + 256, ...; a warp's 32 lanes take 32
// consecutive blocks at each step, and every warp runs the same number of
// steps (lanes past the chunk's end see -inf entries).  A thread loads its
// blocks into registers.  Streaming the chunk through a shared-memory ring
// filled by bulk copies cut the stalls on loads (long scoreboard 4.3 -> 1.6
// per issue) but the per-step barrier waits and arrivals added 19 % more
// instructions, and it measured 214 us against 192 us for 704 rows.
template <bool kVec, bool kUnitT>
__global__ void __launch_bounds__(kSampleThreads, kSampleMinBlocks)
sample_stats_kernel(DraftArgs a, const int32_t* __restrict__ position,
                    int chunk_blocks) {
  __shared__ uint4 s_pre, s_rk[4];
  __shared__ ChunkStat s_part[kSampleWarps];
  const int row = blockIdx.y, chunk = blockIdx.x;
  const int V = a.V;
  const int warp = threadIdx.x >> 5;
  const float* __restrict__ lrow = a.logits + (size_t)row * V;
  const float T = request_temperature(a, row);
  const bool greedy = a.greedy != nullptr && a.greedy[row] != 0;
  if (threadIdx.x == 0) row_noise_setup(a, position, row, chunk, s_pre, s_rk);
  __syncthreads();
  const int n_blk = (V + 3) / 4;
  const int lo = chunk * chunk_blocks;
  const int hi = min(lo + chunk_blocks, n_blk);
  SampleState st = sample_state_init();
  // kSampleBatch blocks per thread and step, every load issued first; the
  // blocks are then taken in the order j, j + threads, ... as one at a time
  for (int base = lo; base < hi; base += kSampleBatch * kSampleThreads) {
    float lb[kSampleBatch][4];
#pragma unroll
    for (int u = 0; u < kSampleBatch; ++u) {
      const int j = base + (int)threadIdx.x + u * kSampleThreads, v = 4 * j;
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
    // the blocks' noise first: independent Philox chains the scheduler
    // interleaves (greedy rows use none; 352.8 -> 342.5 us for 704 rows)
    uint4 wv[kSampleBatch];
#pragma unroll
    for (int u = 0; u < kSampleBatch; ++u)
      wv[u] = greedy ? make_uint4(0u, 0u, 0u, 0u)
                     : philox_folded(s_pre, s_rk,
                                     (uint32_t)(base + (int)threadIdx.x + u * kSampleThreads));
#pragma unroll
    for (int u = 0; u < kSampleBatch; ++u) {
      // warp-uniform: the warp's first block is past the end
      if (base + u * kSampleThreads + 32 * warp >= hi) break;
      sample_block<kUnitT>(st, lb[u], base + (int)threadIdx.x + u * kSampleThreads,
                           T, greedy, wv[u]);
    }
  }
  chunk_stat_out(a, row, chunk, st, s_part);
}

}  // namespace

// Chunks per row: enough CTAs for several waves over the SMs (8 per SM),
// chunks of at most kChunkBlocksMax Philox blocks, at most kMaxChunks, and
// at least 64 Philox blocks (256 entries) per chunk.  Measured on 200064
// entries per row: 704 rows took 368, 359 and 364 us in 2, 3 and 4 chunks;
// 88 rows did best with 7 to 14 chunks, and 8 rows with 152 to 228.
constexpr int kChunkBlocksMax = 18000;

int sample_chunks(int R, int V, int sm_count) {
  const int n_blk = (V + 3) / 4;
  int c = (8 * sm_count + R - 1) / R;
  const int by_length = (n_blk + kChunkBlocksMax - 1) / kChunkBlocksMax;
  if (c < by_length) c = by_length;
  if (c > n_blk / 64) c = n_blk / 64;
  if (c > kMaxChunks) c = kMaxChunks;
  return c < 1 ? 1 : c;
}

cudaError_t launch_sample_stats(const DraftArgs& a, const int32_t* position,
                                int n_chunks, cudaStream_t stream) {
  const int n_blk = (a.V + 3) / 4;
  const int chunk_blocks = (n_blk + n_chunks - 1) / n_chunks;
  const dim3 grid((unsigned)n_chunks, (unsigned)a.B, 1);
  const bool unit = a.temperature == nullptr && a.T == 1.0f;
  auto k = a.V % 4 == 0 ? (unit ? sample_stats_kernel<true, true>
                                : sample_stats_kernel<true, false>)
                        : (unit ? sample_stats_kernel<false, true>
                                : sample_stats_kernel<false, false>);
  k<<<grid, kSampleThreads, 0, stream>>>(a, position, chunk_blocks);
  return cudaGetLastError();
}

}  // namespace dspark
