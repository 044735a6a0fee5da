// gumbel_draw.cuh -- a warp's Gumbel-max draw over a row of scaled logits,
// with the row's sum-exp, for the kernels that sweep whole rows a warp at a
// time (the temperature-only target sampler and the FFMA draft position).
//
// brb-nv/TensorRT-LLM PR #27, "2. One fused kernel per draft position" and
// "1. Temperature-only sampling runs no filter": token = argmax of s + g
// over the row (s = l / T, g the Gumbel variate of the entry's Philox word,
// lowest index on ties), and the softmax statistics (max, sum-exp) of s.
//
// Each warp keeps one reference ref (the best decision score it has found,
// and its index), the same in every lane; each thread keeps a sum reference
// m (its largest s).  One exp2 per entry, f = exp(s - m), feeds the sum and a
// conservative candidate test: an entry can beat ref only if its Gumbel
// score does, i.e. only if w < exp(s - ref) = f exp(m - ref), which the test
// (float)x < 2^32 (1 + 2^-11) f h, h = exp(m - ref), admits with room for the
// rounding of both sides.  Only admitted entries get the exact score s + g,
// and the warp then adopts the best of them.
#pragma once

#include "dspark_common.cuh"

namespace dspark {

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

}  // namespace dspark
