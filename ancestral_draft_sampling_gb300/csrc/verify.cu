// verify.cu -- standard token-level rejection verification of a draft block.
//
// brb-nv/TensorRT-LLM PR #21, "2. Golden sampling semantics": the default
// "standard" rule verifies drafts token by token (Leviathan et al. 2023,
// Chen et al. 2023).  Draft k is accepted with probability
// min(1, p_k[d_k] / q_k[d_k]); at the first rejection the replacement is
// drawn from the residual norm(max(p_k - q_k, 0)); if all K drafts pass, a
// bonus token is drawn from p_K.
//
// One thread-block cluster of C CTAs per request (C chosen so the grid fills
// the GPU).  Every CTA of the cluster runs the K acceptance tests itself (one
// thread per draft, one uniform each from noise stream 1; the first rejection
// is a shared-memory minimum), then draws from its own slice of the drawing
// row by Gumbel-max over log(weight) with noise stream 2 at the drawing
// position; the C partial winners merge through distributed shared memory.
//
// In a slice, warps sweep 128 entries per step, lane l on one Philox block of
// 4 entries.  An entry with weight r and exponential variate E can only beat
// the warp's best score B if log r - log E > B, i.e. E < r e^-B, which needs
// w < r e^-B since E = -log(1 - w) >= w; so the test
// (float)x < 2^32 r e^-B (1 + 2^-11) admits every possible winner (the slack
// covers the float32 rounding of both scores) with a multiply and a compare,
// and only entries that pass get the exact score.  Candidates merge by a
// max-reduction over order-preserving score bits, then a min over indices.
#include <cooperative_groups.h>

#include "dspark_common.cuh"

namespace dspark {
namespace {

namespace cg = cooperative_groups;

constexpr int kVerifyThreads = 256;
constexpr int kVerifyWarps = kVerifyThreads / 32;
constexpr int kVerifyMinBlocks = 4;   // resident CTAs per SM the launch asks for
constexpr int kMaxCluster = 8;        // portable cluster size
constexpr int kMinSliceBlocks = 1024; // Philox blocks (4 entries) per CTA, at least
constexpr float kSlack = 1.000489f;   // 1 + 2^-11, rounded up
// Above this best score e^-B leaves the normal range of float32; the test
// then admits everything (still exact, only slower).  Scores that large need
// weights above e^57.
constexpr float kMaxTestScore = 80.0f;

struct Best {
  float score;
  int idx;
};

struct alignas(16) Slot {
  float score;
  int idx;
  int any;
  int pad;
};

// Keeps the better of st and the warp's candidates (larger score, then the
// lower index); lanes without a candidate offer key 0.
__device__ __forceinline__ void warp_take(Best& st, float cb, int ci) {
  const uint32_t key = ci == kNoIndex ? 0u : ordered_bits(cb);
  const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
  if (kmax == 0u) return;
  const uint32_t imin =
      __reduce_min_sync(0xffffffffu, key == kmax ? (uint32_t)ci : 0xffffffffu);
  const float wb = from_ordered_bits(kmax);
  if (better(wb, (int)imin, st.score, st.idx)) {
    st.score = wb;
    st.idx = (int)imin;
  }
}

__device__ __forceinline__ float elem(const float4 v, int e) {
  return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
}

// Loads Philox block j (entries 4j .. 4j+3) of p and, for the residual, q;
// entries at or beyond V read as 0.
template <bool kVec>
__device__ __forceinline__ void load_block(const float* __restrict__ p,
                                           const float* __restrict__ q, int V,
                                           int j, int hi, float4& pv,
                                           float4& qv) {
  pv = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  qv = pv;
  if (j >= hi) return;
  if (kVec) {
    pv = __ldcs(reinterpret_cast<const float4*>(p) + j);
    if (q) qv = __ldcs(reinterpret_cast<const float4*>(q) + j);
  } else {
    float* pp = &pv.x;
    float* qq = &qv.x;
    for (int e = 0; e < 4; ++e)
      if (4 * j + e < V) {
        pp[e] = __ldcs(p + 4 * j + e);
        if (q) qq[e] = __ldcs(q + 4 * j + e);
      }
  }
}

// The candidate test's scale for the warp's best: 2^32 (1 + slack)
// e^-best; +inf (everything is a candidate) while nothing has won or e^-best
// is out of float32's normal range.  It changes only when the best does.
__device__ __forceinline__ float test_scale(const Best& st) {
  return (st.idx == kNoIndex || st.score > kMaxTestScore)
             ? INFINITY
             : 0x1p32f * kSlack * expf(-st.score);
}

// One Philox block of the sweep, with its noise words w: weights, candidate
// test, exact scores of the candidates, warp merge.  Warp-uniform control
// flow.  c is test_scale(st), kept up to date here.
__device__ __forceinline__ void sweep_block(Best& st, float& c, bool& any, int j,
                                            float4 pv, float4 qv, bool resid,
                                            float wscale, const uint4 w) {
  float wt[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float pe = elem(pv, e);
    const float d = resid ? __fsub_rn(__fmul_rn(wscale, pe), elem(qv, e)) : pe;
    wt[e] = d > 0.0f ? d : 0.0f;  // NaN and non-positive weights: 0
    any |= wt[e] > 0.0f;
  }
  float thr[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) thr[e] = wt[e] > 0.0f ? __fmul_ru(wt[e], c) : 0.0f;
  // the vote needs only whether some entry passes; the rare path works out
  // which ones do
  const bool pass = (__uint2float_rz(w.x) < thr[0]) | (__uint2float_rz(w.y) < thr[1]) |
                    (__uint2float_rz(w.z) < thr[2]) | (__uint2float_rz(w.w) < thr[3]);
  if (__any_sync(0xffffffffu, pass)) {
    uint32_t cand = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      cand |= (__uint2float_rz(word_of(w, e)) < thr[e] ? 1u : 0u) << e;
    float cb = -INFINITY;
    int ci = kNoIndex;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (!((cand >> e) & 1u)) continue;
      const float sc = __fadd_rn(logf(wt[e]), gumbel_from_word(word_of(w, e)));
      if (ci == kNoIndex || sc > cb) {  // e ascending: keeps the lower index
        cb = sc;
        ci = 4 * j + e;
      }
    }
    warp_take(st, cb, ci);
    c = test_scale(st);
  }
}

// Gumbel-max over log(weight) on this CTA's slice [lo, hi) of Philox blocks,
// weights max(wscale p - q, 0) when q != nullptr (the residual; wscale is 1
// for the standard rule, and 1 * p is p exactly), else p; zero weights never
// win.  (pre, rk): the folded Philox constants of noise
// stream 2 at the drawing position (philox_fold).  Then the cluster-wide winner and "some weight was
// positive", identical in every CTA of the cluster.
template <bool kVec>
__device__ Slot draw_row(cg::cluster_group& cluster, const float* __restrict__ p,
                         const float* __restrict__ q, int V, int lo, int hi,
                         float wscale, const uint4& pre, const uint4 (&rk)[4],
                         Best* part, int* any_part, Slot* slot) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool resid = q != nullptr;
  Best st = {-INFINITY, kNoIndex};
  float c = test_scale(st);
  bool any = false;
  constexpr int kStride = kVerifyWarps * 32;
  // two blocks per lane in flight: j and j + kStride
  for (int base = lo + warp * 32; base < hi; base += 2 * kStride) {
    const int j0 = base + lane, j1 = base + kStride + lane;
    float4 p0, q0, p1, q1;
    load_block<kVec>(p, q, V, j0, hi, p0, q0);
    load_block<kVec>(p, q, V, j1, hi, p1, q1);
    // the two blocks' noise first: two independent Philox chains the
    // scheduler interleaves (43.1 -> 41.5 us for the B=88 block)
    const uint4 w0 = philox_folded(pre, rk, (uint32_t)j0);
    const uint4 w1 = philox_folded(pre, rk, (uint32_t)j1);
    sweep_block(st, c, any, j0, p0, q0, resid, wscale, w0);
    if (base + kStride < hi)
      sweep_block(st, c, any, j1, p1, q1, resid, wscale, w1);
  }
  any = __any_sync(0xffffffffu, any);
  if (lane == 0) {
    part[warp] = st;
    any_part[warp] = any;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    Best r = part[0];
    int a = any_part[0];
    for (int i = 1; i < kVerifyWarps; ++i) {
      if (!better(r.score, r.idx, part[i].score, part[i].idx)) r = part[i];
      a |= any_part[i];
    }
    *slot = Slot{r.score, r.idx, a, 0};
  }
  cluster.sync();  // every CTA's slot is written
  Slot all = *cluster.map_shared_rank(slot, 0u);
  for (unsigned i = 1; i < cluster.num_blocks(); ++i) {
    const Slot o = *cluster.map_shared_rank(slot, i);
    if (!better(all.score, all.idx, o.score, o.idx)) {
      all.score = o.score;
      all.idx = o.idx;
    }
    all.any |= o.any;
  }
  cluster.sync();  // every CTA has read every slot (they may be rewritten)
  return all;
}

// Block verification's sums r_i = sum_x max(w_i p_i(x) - q_i(x), 0),
// i = 1..K-1, over this CTA's slice of each row, then over the cluster.
// Every CTA ends with the same values: each thread adds its blocks in
// order, warps combine by a butterfly, the warps' sums and then the CTAs'
// are added in a fixed order.
template <bool kVec>
__device__ void block_sums(cg::cluster_group& cluster, const float* __restrict__ q,
                           const float* __restrict__ p, int b, int K, int V,
                           int lo, int hi, const float* s_w, float* s_wpart,
                           float* s_part, float* s_r) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = 1; i < K; ++i) {
    const float* prow = p + ((size_t)b * (K + 1) + i) * V;
    const float* qrow = q + ((size_t)b * K + i) * V;
    const float wi = s_w[i];
    float acc = 0.0f;
    // four blocks in flight per thread
    for (int j0 = lo + (int)threadIdx.x; j0 < hi; j0 += 4 * kVerifyThreads) {
      float4 pv[4], qv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        load_block<kVec>(prow, qrow, V, j0 + u * kVerifyThreads, hi, pv[u], qv[u]);
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float t = __fsub_rn(__fmul_rn(wi, elem(pv[u], e)), elem(qv[u], e));
          acc = __fadd_rn(acc, t > 0.0f ? t : 0.0f);  // NaN terms count as 0
        }
    }
#pragma unroll
    for (int mask = 16; mask > 0; mask >>= 1)
      acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, mask));
    if (lane == 0) s_wpart[(i - 1) * kVerifyWarps + warp] = acc;
  }
  __syncthreads();
  for (int i = 1 + (int)threadIdx.x; i < K; i += kVerifyThreads) {
    float c = 0.0f;
    for (int w = 0; w < kVerifyWarps; ++w) c = __fadd_rn(c, s_wpart[(i - 1) * kVerifyWarps + w]);
    s_part[i - 1] = c;
  }
  cluster.sync();  // every CTA's partial sums are written
  for (int i = 1 + (int)threadIdx.x; i < K; i += kVerifyThreads) {
    float r = 0.0f;
    for (unsigned c = 0; c < cluster.num_blocks(); ++c)
      r = __fadd_rn(r, cluster.map_shared_rank(s_part, c)[i - 1]);
    s_r[i] = r;
  }
  cluster.sync();  // every CTA has read them (and s_r is complete)
}

template <bool kVec, bool kBlock>
__global__ void __launch_bounds__(kVerifyThreads, kVerifyMinBlocks)
verify_kernel(const float* __restrict__ q, const float* __restrict__ p,
              const int32_t* __restrict__ tokens, const uint64_t* seed,
              const uint64_t* offset, int K, int V, int32_t* accepted_len,
              int32_t* emitted) {
  __shared__ int s_first;
  __shared__ int s_bad;
  __shared__ Best part[kVerifyWarps];
  __shared__ int any_part[kVerifyWarps];
  __shared__ Slot slot;
  __shared__ uint4 s_pre, s_rk[4];
  // block rule: ratios, weights w_0..w_K, uniforms, sums r_1..r_{K-1}
  __shared__ float s_ratio[kBlock ? DSPARK_MAX_K : 1];
  __shared__ float s_w[kBlock ? DSPARK_MAX_K + 1 : 1];
  __shared__ float s_eta[kBlock ? DSPARK_MAX_K : 1];
  __shared__ float s_wpart[kBlock ? DSPARK_MAX_K * kVerifyWarps : 1];
  __shared__ float s_part[kBlock ? DSPARK_MAX_K : 1];
  __shared__ float s_r[kBlock ? DSPARK_MAX_K : 1];
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.x / C;
  const uint64_t sd = seed[b], off = offset[b];
  if (threadIdx.x == 0) {
    s_first = K;
    s_bad = 0;
  }
  __syncthreads();
  for (int k = threadIdx.x; k < K; k += kVerifyThreads) {
    const int d = tokens[(size_t)b * K + k];
    if (d < 0 || d >= V) {
      atomicOr(&s_bad, 1);
      continue;
    }
    const float qd = q[((size_t)b * K + k) * V + d];
    const float pd = p[((size_t)b * (K + 1) + k) * V + d];
    const float u = accept_uniform(noise_block(sd, off, k, kNoiseAccept, 0u).x);
    if (kBlock) {
      s_ratio[k] = __fdiv_rn(pd, qd);
      s_eta[k] = u;
    } else if (!(__fmul_rn(u, qd) < pd)) {
      atomicMin(&s_first, k);
    }
  }
  __syncthreads();
  if (s_bad) {  // the same in every CTA of the cluster: all return here
    if (rank == 0 && threadIdx.x == 0) {
      accepted_len[b] = -1;
      emitted[b] = -1;
    }
    return;
  }
  // this CTA's slice of the row's Philox blocks
  const int n_blk = (V + 3) / 4;
  const int per = (n_blk + C - 1) / C;
  const int lo = min(rank * per, n_blk), hi = min(lo + per, n_blk);
  float wscale = 1.0f;
  if (kBlock) {
    if (threadIdx.x == 0) {  // w_{k+1} = min(w_k (p/q), 1); NaN counts as 0
      float w = 1.0f;
      s_w[0] = w;
      for (int k = 0; k < K; ++k) {
        const float t = __fmul_rn(w, s_ratio[k]);
        w = t < 1.0f ? t : (t >= 1.0f ? 1.0f : 0.0f);
        s_w[k + 1] = w;
      }
    }
    __syncthreads();
    block_sums<kVec>(cluster, q, p, b, K, V, lo, hi, s_w, s_wpart, s_part, s_r);
    if (threadIdx.x == 0) {  // the longest prefix whose uniform is under h_i
      int tau = 0;
      for (int i = 1; i <= K; ++i) {
        float h;
        if (i < K) {
          const float r = s_r[i];
          const float den = __fadd_rn(r, __fsub_rn(1.0f, s_w[i]));
          h = den > 0.0f ? __fdiv_rn(r, den) : 1.0f;
        } else {
          h = s_w[K];
        }
        if (s_eta[i - 1] <= h) tau = i;
      }
      s_first = tau;
    }
    __syncthreads();
    wscale = s_w[s_first];
  }
  const int kk = s_first;
  if (threadIdx.x == 0)
    philox_fold(s_pre, s_rk, (uint32_t)sd, (uint32_t)(sd >> 32),
                (uint32_t)kk | ((uint32_t)kNoiseResample << 16), (uint32_t)off,
                (uint32_t)(off >> 32));
  __syncthreads();
  const float* prow = p + ((size_t)b * (K + 1) + kk) * V;
  const float* qrow = kk < K ? q + ((size_t)b * K + kk) * V : nullptr;
  Slot r = draw_row<kVec>(cluster, prow, qrow, V, lo, hi, wscale, s_pre, s_rk,
                          part, any_part, &slot);
  if (qrow != nullptr && !r.any)  // residual all zero: draw from p itself
    r = draw_row<kVec>(cluster, prow, nullptr, V, lo, hi, 1.0f, s_pre, s_rk,
                       part, any_part, &slot);
  if (rank == 0 && threadIdx.x == 0) {
    accepted_len[b] = kk;
    emitted[b] = r.idx == kNoIndex ? 0 : r.idx;
  }
}

// CTAs per request: enough clusters to fill every SM's resident slots, at
// most the portable cluster size, and at least kMinSliceBlocks per slice.
int verify_cluster_size(int B, int V, int sms) {
  const int slots = sms * kVerifyMinBlocks;
  int c = slots / (B > 0 ? B : 1);
  const int n_blk = (V + 3) / 4;
  const int by_len = n_blk / kMinSliceBlocks;
  if (c > by_len) c = by_len;
  if (c > kMaxCluster) c = kMaxCluster;
  return c < 1 ? 1 : c;
}

template <bool kVec, bool kBlock>
cudaError_t launch_verify_t(const float* q, const float* p,
                            const int32_t* tokens, const uint64_t* seed,
                            const uint64_t* offset, int B, int K, int V,
                            int32_t* accepted_len, int32_t* emitted, int C,
                            cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)B * (unsigned)C, 1, 1);
  cfg.blockDim = dim3(kVerifyThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, verify_kernel<kVec, kBlock>, q, p, tokens,
                            seed, offset, K, V, accepted_len, emitted);
}

}  // namespace

cudaError_t launch_verify(const float* q, const float* p, const int32_t* tokens,
                          const uint64_t* seed, const uint64_t* offset, int B,
                          int K, int V, int32_t* accepted_len,
                          int32_t* emitted, int sms, bool block,
                          cudaStream_t stream) {
  const int C = verify_cluster_size(B, V, sms);
  const bool vec = V % 4 == 0;
  if (block)
    return vec ? launch_verify_t<true, true>(q, p, tokens, seed, offset, B, K, V,
                                             accepted_len, emitted, C, stream)
               : launch_verify_t<false, true>(q, p, tokens, seed, offset, B, K, V,
                                              accepted_len, emitted, C, stream);
  return vec ? launch_verify_t<true, false>(q, p, tokens, seed, offset, B, K, V,
                                            accepted_len, emitted, C, stream)
             : launch_verify_t<false, false>(q, p, tokens, seed, offset, B, K, V,
                                             accepted_len, emitted, C, stream);
}

}  // namespace dspark
