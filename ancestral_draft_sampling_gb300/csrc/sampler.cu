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
// Each warp keeps one reference ref (the best decision score it has found,
// and its index), the same in every lane; each thread keeps a sum reference
// m (its largest s).  One exp2 per entry, f = exp(s - m), feeds the sum and a
// conservative candidate test: an entry can beat ref only if its Gumbel
// score does, i.e. only if w < exp(s - ref) = f exp(m - ref), which the test
// (float)x < 2^32 (1 + 2^-11) f h, h = exp(m - ref), admits with room for the
// rounding of both sides.  Only admitted entries get the exact score s + g,
// and the warp then adopts the best of them.  With the reference shared by
// the 32 lanes, a warp meets an admitted entry in a few of its steps only
// (a reference per lane admitted one in most steps of some lane, and the
// whole warp ran the exact path).
#include "dspark_common.cuh"

namespace dspark {
namespace {

constexpr int kSampleThreads = 256;
constexpr int kSampleWarps = kSampleThreads / 32;
constexpr int kSampleBatch = 2;  // blocks a thread loads before using them
constexpr int kSampleMinBlocks = 5;  // resident CTAs per SM (48 registers)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTestScale = 4297064448.0f;  // 2^32 (1 + 2^-11), exact in float32

__device__ __forceinline__ float word_pick(const float (&a)[4], int e) {
  return e == 0 ? a[0] : e == 1 ? a[1] : e == 2 ? a[2] : a[3];
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The best of the lanes' exact candidates (cb, ci) against the warp's
// reference (ref, idx): the largest score by a max-reduction over
// order-preserving bits, then the lowest index among the lanes that hold it.
// A lane without a candidate offers key 0 (below every score).  Ties with
// the reference keep the lower index.
__device__ __forceinline__ bool warp_adopt(float& ref, int& idx, float cb,
                                           int ci) {
  const uint32_t key = ci == kNoIndex ? 0u : ordered_bits(cb);
  const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
  if (kmax == 0u) return false;
  const uint32_t imin = __reduce_min_sync(
      0xffffffffu, key == kmax ? (uint32_t)ci : 0xffffffffu);
  const float wb = from_ordered_bits(kmax);
  if (wb > ref || (wb == ref && (int)imin < idx)) {
    ref = wb;
    idx = (int)imin;
    return true;
  }
  return false;
}

// Running state of one thread: ref and idx are the warp's (the same in every
// lane) for a sampled row, the thread's own for a greedy row.
struct SampleState {
  float ref;  // best decision score (s + g, or s for a greedy row)
  int idx;    // its vocab index (kNoIndex: none)
  float m;    // largest s of this thread: the sum's reference
  float sum;  // sum of exp(s - m)
  float h;    // exp(m - ref), used by the candidate test
};

__device__ __forceinline__ SampleState sample_state_init() {
  SampleState st;
  st.ref = -INFINITY;
  st.idx = kNoIndex;
  st.m = -INFINITY;
  st.sum = 0.0f;
  st.h = INFINITY;
  return st;
}

// Philox block j (entries v = 4j .. 4j+3, logits l, noise words w) folded
// into the state.  Every lane of the warp calls it at the same step: the
// sampled path votes across the warp.
template <bool kUnitT>
__device__ __forceinline__ void sample_block(SampleState& st, const float (&l)[4],
                                             int j, float T, bool greedy,
                                             const uint4 w) {
  const int v = 4 * j;
  float s[4];
#pragma unroll
  for (int e = 0; e < 4; ++e)
    s[e] = kUnitT || T == 1.0f ? l[e] : __fdiv_rn(l[e], T);
  // the sum's reference moves to a larger s (rare)
  const float m4 = fmaxf(fmaxf(st.m, s[0]), fmaxf(fmaxf(s[1], s[2]), s[3]));  // NaN ignored
  if (m4 > st.m) {
    st.sum = __fmul_rn(st.sum, ex2_approx((st.m - m4) * kLog2e));  // 0 from -inf
    st.m = m4;
    st.h = ex2_approx((st.m - st.ref) * kLog2e);
  }
  // exp(s - m); while m is -inf every s is -inf (term 0) or NaN (NaN),
  // which the reference -FLT_MAX (the lowest finite float) gives as well
  const float mr = fmaxf(st.m, -0x1.fffffep127f);
  float f[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) f[e] = ex2_approx((s[e] - mr) * kLog2e);
  st.sum = __fadd_rn(st.sum, __fadd_rn(__fadd_rn(f[0], f[1]), __fadd_rn(f[2], f[3])));
  if (greedy) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (s[e] > st.ref) {  // NaN and -inf never win; e ascending keeps the lower
        st.ref = s[e];
        st.idx = v + e;
      }
    return;
  }
  const float c = kTestScale * st.h;
  // the warp-wide vote needs only whether some entry passes; which ones pass
  // is worked out on the rare path
  const bool any = (__uint2float_rz(w.x) < __fmul_ru(f[0], c)) |
                   (__uint2float_rz(w.y) < __fmul_ru(f[1], c)) |
                   (__uint2float_rz(w.z) < __fmul_ru(f[2], c)) |
                   (__uint2float_rz(w.w) < __fmul_ru(f[3], c));
  if (__any_sync(0xffffffffu, any)) {  // a possible winner
    uint32_t cand = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      cand |= (__uint2float_rz(word_of(w, e)) < __fmul_ru(f[e], c) ? 1u : 0u) << e;
    float cb = -INFINITY;
    int ci = kNoIndex;
    while (cand) {
      const int e = __ffs(cand) - 1;
      cand &= cand - 1u;
      const float sc = __fadd_rn(word_pick(s, e), gumbel_from_word(word_of(w, e)));
      if (sc > cb) {  // e ascending: strict keeps the lower index
        cb = sc;
        ci = v + e;
      }
    }
    if (warp_adopt(st.ref, st.idx, cb, ci))
      st.h = ex2_approx((st.m - st.ref) * kLog2e);
  }
}

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
