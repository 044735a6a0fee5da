// verify.cu -- standard token-level rejection verification of a draft block.
//
// brb-nv/TensorRT-LLM PR #21, "2. Golden sampling semantics": the default
// "standard" rule verifies drafts token by token (Leviathan et al. 2023,
// Chen et al. 2023).  Draft k is accepted with probability
// min(1, p_k[d_k] / q_k[d_k]); at the first rejection the replacement is
// drawn from the residual norm(max(p_k - q_k, 0)); if all K drafts pass, a
// bonus token is drawn from p_K.
//
// One CTA per request.  Thread 0 walks the K acceptance tests (one uniform
// each, noise stream 1); then the whole CTA does one Gumbel-max sweep over
// the drawing row (noise stream 2 at the drawing position).
#include "dspark_common.cuh"

namespace dspark {
namespace {

constexpr int kVerifyThreads = 512;

struct Cand {
  float score;
  int idx;
};

// Keeps the better of c and (score, idx): larger score, then lower index.
__device__ __forceinline__ void take(Cand& c, float score, int idx) {
  if (better(c.score, c.idx, score, idx)) return;
  c.score = score;
  c.idx = idx;
}

__device__ __forceinline__ Cand block_argmax(Cand c, Cand* part) {
#pragma unroll
  for (int mask = 16; mask > 0; mask >>= 1) {
    const float os = __shfl_xor_sync(0xffffffffu, c.score, mask);
    const int oi = __shfl_xor_sync(0xffffffffu, c.idx, mask);
    take(c, os, oi);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) part[warp] = c;
  __syncthreads();
  c = part[0];
  for (int w = 1; w < kVerifyThreads / 32; ++w) take(c, part[w].score, part[w].idx);
  return c;
}

__global__ void __launch_bounds__(kVerifyThreads)
verify_kernel(const float* __restrict__ q, const float* __restrict__ p,
              const int32_t* __restrict__ tokens, const uint64_t* seed,
              const uint64_t* offset, int K, int V, int32_t* accepted_len,
              int32_t* emitted) {
  __shared__ int s_draw_pos;
  __shared__ int s_bad;
  __shared__ Cand part[kVerifyThreads / 32];
  const int b = blockIdx.x;
  const uint64_t sd = seed[b], off = offset[b];
  if (threadIdx.x == 0) {
    int kk = K, bad = 0;
    for (int k = 0; k < K; ++k) {
      const int d = tokens[(size_t)b * K + k];
      if (d < 0 || d >= V) {
        bad = 1;
        break;
      }
      const float qd = q[((size_t)b * K + k) * V + d];
      const float pd = p[((size_t)b * (K + 1) + k) * V + d];
      const float u = accept_uniform(noise_block(sd, off, k, kNoiseAccept, 0u).x);
      if (!(__fmul_rn(u, qd) < pd)) {
        kk = k;
        break;
      }
    }
    s_draw_pos = kk;
    s_bad = bad;
  }
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x == 0) {
      accepted_len[b] = -1;
      emitted[b] = -1;
    }
    return;
  }
  const int kk = s_draw_pos;
  const float* prow = p + ((size_t)b * (K + 1) + kk) * V;
  const float* qrow = kk < K ? q + ((size_t)b * K + kk) * V : nullptr;
  Cand res = {-INFINITY, kNoIndex};  // residual draw
  Cand tgt = {-INFINITY, kNoIndex};  // draw from p itself
  const int n_blk = (V + 3) / 4;
  for (int j = threadIdx.x; j < n_blk; j += kVerifyThreads) {
    const uint4 w = noise_block(sd, off, kk, kNoiseResample, (uint32_t)j);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int v = 4 * j + e;
      if (v >= V) break;
      const float g = gumbel_from_word(word_of(w, e));
      const float pv = prow[v];
      if (pv > 0.0f) take(tgt, __fadd_rn(logf(pv), g), v);
      if (qrow) {
        const float diff = __fsub_rn(pv, qrow[v]);
        if (diff > 0.0f) take(res, __fadd_rn(logf(diff), g), v);
      }
    }
  }
  res = block_argmax(res, part);
  tgt = block_argmax(tgt, part);
  if (threadIdx.x == 0) {
    int tok = (qrow && res.idx != kNoIndex) ? res.idx : tgt.idx;
    if (tok == kNoIndex) tok = 0;
    accepted_len[b] = kk;
    emitted[b] = tok;
  }
}

}  // namespace

cudaError_t launch_verify(const float* q, const float* p, const int32_t* tokens,
                          const uint64_t* seed, const uint64_t* offset, int B,
                          int K, int V, int32_t* accepted_len,
                          int32_t* emitted, cudaStream_t stream) {
  verify_kernel<<<B, kVerifyThreads, 0, stream>>>(q, p, tokens, seed, offset,
                                                  K, V, accepted_len, emitted);
  return cudaGetLastError();
}

}  // namespace dspark
