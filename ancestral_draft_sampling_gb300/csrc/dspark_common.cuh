// dspark_common.cuh -- device helpers shared by the sampler's kernels:
// counter-based noise, the Gumbel transform, and the merge rules of the
// per-chunk softmax statistics.
//
// Method: brb-nv/TensorRT-LLM PR #27, "2. One fused kernel per draft
// position" (Gumbel-max with a counter-based Philox stream keyed by the
// request's (seed, offset) draft slot of position k; per-chunk softmax
// statistics; a small kernel picks the token).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/dspark.h"

namespace dspark {

// ---------------------------------------------------------------- limits
constexpr int kMaxChunks = 512;        // vocab chunks per position (grid.x)
constexpr int kNoIndex = 0x7fffffff;   // "no non-NaN candidate yet"
constexpr int kNoiseDraft = 0;         // counter stream ids
constexpr int kNoiseAccept = 1;
constexpr int kNoiseResample = 2;
constexpr int kNoiseTarget = 3;   // the temperature-only target sampler

// ---------------------------------------------------------------- Philox
// Philox4x32-10 (Salmon et al., "Parallel random numbers: as easy as 1, 2,
// 3", SC'11): ten rounds of two 32x32->64 multiplies with the published
// multipliers, the key advanced by the published Weyl constants between
// rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 ctr, uint2 key) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      key.x += 0x9E3779B9u;
      key.y += 0xBB67AE85u;
    }
    // one widening multiply gives both halves of each 64-bit product
    const unsigned long long pa = (unsigned long long)0xD2511F53u * ctr.x;
    const unsigned long long pb = (unsigned long long)0xCD9E8D57u * ctr.z;
    ctr = make_uint4((uint32_t)(pb >> 32) ^ ctr.y ^ key.x, (uint32_t)pb,
                     (uint32_t)(pa >> 32) ^ ctr.w ^ key.y, (uint32_t)pa);
  }
  return ctr;
}

// The Philox block that holds the words of elements 4*blk .. 4*blk+3 of
// stream `stream` at position k for request (seed, offset).
__device__ __forceinline__ uint4 noise_block(uint64_t seed, uint64_t offset,
                                             int k, int stream, uint32_t blk) {
  const uint4 ctr = make_uint4(blk, (uint32_t)k | ((uint32_t)stream << 16),
                               (uint32_t)offset, (uint32_t)(offset >> 32));
  const uint2 key = make_uint2((uint32_t)seed, (uint32_t)(seed >> 32));
  return philox4x32_10(ctr, key);
}

// One Philox4x32-10 round (the published multipliers) with round key k.
__device__ __forceinline__ uint4 philox_round(uint4 c, uint32_t k0, uint32_t k1) {
  const unsigned long long pa = (unsigned long long)0xD2511F53u * c.x;
  const unsigned long long pb = (unsigned long long)0xCD9E8D57u * c.z;
  return make_uint4((uint32_t)(pb >> 32) ^ c.y ^ k0, (uint32_t)pb,
                    (uint32_t)(pa >> 32) ^ c.w ^ k1, (uint32_t)pa);
}

// Philox4x32-10 along a row of counters (x0, c1, c2, c3) with only x0
// varying, under key (k0, k1).  The parts of rounds 1 and 2 that depend on
// the fixed words alone fold into constants: round 1 gives
// (A, B, hi(M0 x0) ^ C1, lo(M0 x0)) with A = hi(M1 c2) ^ c1 ^ k0,
// B = lo(M1 c2), C1 = c3 ^ k1; round 2 then gives
// (hi(M1 z) ^ D2, lo(M1 z), lo(M0 x0) ^ E2, F2) with z the third word,
// D2 = B ^ k0', E2 = hi(M0 A) ^ k1', F2 = lo(M0 A).  philox_fold computes
// pre = (C1, D2, E2, F2) and the round keys of rounds 3..10 (round r uses
// (k0 + r W0, k1 + r W1), r = 0..9); philox_folded gives the block of x0,
// bit-identical to philox4x32_10.
__device__ __forceinline__ void philox_fold(uint4& pre, uint4 (&rk)[4],
                                            uint32_t k0, uint32_t k1,
                                            uint32_t c1, uint32_t c2,
                                            uint32_t c3) {
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  const unsigned long long m1c2 = (unsigned long long)0xCD9E8D57u * c2;
  const uint32_t A = (uint32_t)(m1c2 >> 32) ^ c1 ^ k0;
  const uint32_t Bv = (uint32_t)m1c2;
  const uint32_t C1 = c3 ^ k1;
  const unsigned long long m0a = (unsigned long long)0xD2511F53u * A;
  pre = make_uint4(C1, Bv ^ (k0 + W0), (uint32_t)(m0a >> 32) ^ (k1 + W1),
                   (uint32_t)m0a);
  for (int j = 0; j < 4; ++j) {
    const uint32_t r = 2 * j + 2;
    rk[j] = make_uint4(k0 + r * W0, k1 + r * W1, k0 + (r + 1) * W0,
                       k1 + (r + 1) * W1);
  }
}

__device__ __forceinline__ uint4 philox_folded(const uint4& pre_ref,
                                               const uint4 (&rk)[4],
                                               uint32_t x0) {
  const uint4 pre = pre_ref;
  const unsigned long long pa = (unsigned long long)0xD2511F53u * x0;
  const uint32_t z = (uint32_t)(pa >> 32) ^ pre.x;
  const unsigned long long pb = (unsigned long long)0xCD9E8D57u * z;
  uint4 c = make_uint4((uint32_t)(pb >> 32) ^ pre.y, (uint32_t)pb,
                       (uint32_t)pa ^ pre.z, pre.w);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 k = rk[j];
    c = philox_round(c, k.x, k.y);
    c = philox_round(c, k.z, k.w);
  }
  return c;
}

__device__ __forceinline__ uint32_t word_of(uint4 w, int i) {
  return i == 0 ? w.x : i == 1 ? w.y : i == 2 ? w.z : w.w;
}

// Standard exponential variate E = -log(1 - w), w = (x + 0.5) * 2^-32, in
// float32 with one logarithm and no divergent branch.  Both w and 1 - w are
// formed from the word (exact up to one rounding), and the logarithm is
// taken of whichever is the better argument:
//   w >= 1/2: E = -log(1 - w), 1 - w = (~x + 0.5) * 2^-32 <= 1/2;
//   w <  1/2: E = -log1p(-w) by Kahan's identity log1p(z) = z log(u)/(u - 1)
//             with u = 1 + z rounded (u - 1 is exact for u in [1/2, 1]), and
//             E = w when u rounds to 1.
// Relative error a few ulp over the whole range, including both tails.
__device__ __forceinline__ float exponential_from_word(uint32_t x) {
  const bool lower = x < 0x80000000u;
  const float w = fmaf(__uint2float_rn(x), 0x1p-32f, 0x1p-33f);
  const float one_minus_w = fmaf(__uint2float_rn(~x), 0x1p-32f, 0x1p-33f);
  const float u = lower ? __fsub_rn(1.0f, w) : one_minus_w;
  const float L = logf(u);
  const float d = __fsub_rn(u, 1.0f);
  const float kahan = d == 0.0f ? w : __fmul_rn(L, __fdividef(w, d));
  return lower ? kahan : -L;
}

// Standard Gumbel variate g = -log(E) = -log(-log(1 - w)).
__device__ __forceinline__ float gumbel_from_word(uint32_t x) {
  return -logf(exponential_from_word(x));
}

// Uniform in (0, 1) for the acceptance test, exact in float32:
// ((x >> 9) + 0.5) * 2^-23.
__device__ __forceinline__ float accept_uniform(uint32_t x) {
  return ((float)(x >> 9) + 0.5f) * 0x1p-23f;
}

// ------------------------------------------------- chunk softmax statistics
// Per (request, vocab chunk): the best decision score and its index, and the
// running (max m, sum exp(s - m)) of the scaled logits.
struct alignas(16) ChunkStat {
  float best;  // largest decision score (s + g, or s for greedy rows)
  int idx;     // its lowest index; kNoIndex if no score beat -inf
  float m;     // max of the non-NaN scaled logits (-inf if none)
  float s;     // sum of exp(s_v - m) (NaN if any s_v was NaN)
};

// Candidate order: larger score first, then the lower index; an entry with
// idx == kNoIndex (nothing but NaN seen) loses to anything.
__device__ __forceinline__ bool better(float sa, int ia, float sb, int ib) {
  if (ib == kNoIndex) return true;
  if (ia == kNoIndex) return false;
  if (sa != sb) return sa > sb;
  return ia < ib;
}

__device__ __forceinline__ void merge_argmax(float& best, int& idx, float ob,
                                             int oi) {
  if (!better(best, idx, ob, oi)) {
    best = ob;
    idx = oi;
  }
}

// (m, s) (+) (om, os): the sum-exp of the union, relative to the larger max.
__device__ __forceinline__ void merge_sumexp(float& m, float& s, float om,
                                             float os) {
  const float mn = fmaxf(m, om);
  if (mn == -INFINITY) {
    s = __fadd_rn(s, os);  // both empty (0) or carrying a NaN
  } else {
    // explicit roundings: no FMA contraction, so (a, b) and (b, a) agree
    s = __fadd_rn(__fmul_rn(s, expf(m - mn)), __fmul_rn(os, expf(om - mn)));
  }
  m = mn;
}

__device__ __forceinline__ void merge_stat(ChunkStat& a, const ChunkStat& b) {
  merge_argmax(a.best, a.idx, b.best, b.idx);
  merge_sumexp(a.m, a.s, b.m, b.s);
}

__device__ __forceinline__ ChunkStat shfl_xor_stat(const ChunkStat& a,
                                                   int lane_mask) {
  ChunkStat o;
  o.best = __shfl_xor_sync(0xffffffffu, a.best, lane_mask);
  o.idx = __shfl_xor_sync(0xffffffffu, a.idx, lane_mask);
  o.m = __shfl_xor_sync(0xffffffffu, a.m, lane_mask);
  o.s = __shfl_xor_sync(0xffffffffu, a.s, lane_mask);
  return o;
}

// Butterfly reduction over the 32 lanes; every lane ends with the result.
// merge_stat(a, b) and merge_stat(b, a) give the same bits (max, the index
// tie-break and the two-term IEEE sum are all commutative), so partners
// agree and the result is bitwise reproducible.
__device__ __forceinline__ ChunkStat warp_reduce_stat(ChunkStat a) {
#pragma unroll
  for (int mask = 16; mask > 0; mask >>= 1) {
    const ChunkStat o = shfl_xor_stat(a, mask);
    merge_stat(a, o);
  }
  return a;
}

__device__ __forceinline__ ChunkStat empty_stat() {
  ChunkStat e;
  e.best = -INFINITY;
  e.idx = kNoIndex;
  e.m = -INFINITY;
  e.s = 0.0f;
  return e;
}

// Folds four consecutive candidates v..v+3 into a lane's running statistic.
__device__ __forceinline__ void fold4(ChunkStat& st, const float s[4],
                                      const float score[4], int v, int V) {
  float m4 = -INFINITY;
  bool any_nan = false;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if (v + e >= V) continue;
    if (score[e] > st.best) {  // NaN and -inf never win
      st.best = score[e];
      st.idx = v + e;
    }
    m4 = fmaxf(m4, s[e]);
    any_nan |= isnan(s[e]);
  }
  const float mn = fmaxf(st.m, m4);
  if (mn == -INFINITY) {
    if (any_nan) st.s = __int_as_float(0x7fc00000);
  } else {
    float acc = (st.m == mn) ? st.s : __fmul_rn(st.s, expf(st.m - mn));
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (v + e < V) acc = __fadd_rn(acc, expf(s[e] - mn));
    st.s = acc;
    st.m = mn;
  }
}

// Float32 -> uint32 map that preserves order (for finite and infinite
// values): flip every bit of negatives, set the sign bit of the others.
__device__ __forceinline__ uint32_t ordered_bits(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float from_ordered_bits(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Decision key of a winner (score, index): the score's order-preserving
// bits above the complement of the index, so the unsigned maximum of keys
// is the candidate order of better() (larger score, then lower index).  A
// winner's score is never NaN and its key never 0; 0 means "no winner".
__device__ __forceinline__ unsigned long long decision_key(float score,
                                                           int idx) {
  return ((unsigned long long)ordered_bits(score) << 32) |
         (unsigned long long)(0xffffffffu - (uint32_t)idx);
}

// The token a key selects: its index, or 0 when no entry won (the token
// the pick writes for a request whose statistics hold no winner).
__device__ __forceinline__ int key_token(unsigned long long key) {
  return key == 0ull ? 0 : (int)(0xffffffffu - (uint32_t)key);
}

// Statistics slot (buf, b, chunk) of the two-buffer array.
__device__ __forceinline__ ChunkStat* stat_slot(ChunkStat* stats, int buf,
                                                int B, int b, int chunk) {
  return stats + ((size_t)buf * B + b) * kMaxChunks + chunk;
}

// The merged statistics of request b over chunks 0..n_chunks-1, by one
// whole warp: lane l merges chunks l, l+32, ... in that order, then a
// butterfly combines the lanes (every lane returns the result).  Up to
// kMergeBatch loads of a lane are issued before its first merge.
constexpr int kMergeBatch = 8;
__device__ __forceinline__ ChunkStat merge_row(const ChunkStat* row,
                                               int n_chunks, int lane) {
  ChunkStat st = empty_stat();
  for (int c0 = lane; c0 < n_chunks; c0 += 32 * kMergeBatch) {
    ChunkStat got[kMergeBatch];
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j)
      if (c0 + 32 * j < n_chunks) got[j] = row[c0 + 32 * j];
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j)
      if (c0 + 32 * j < n_chunks) merge_stat(st, got[j]);
  }
  return warp_reduce_stat(st);
}

// --------------------------------------------------------------- bf16 load
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float((uint32_t)b << 16);
}

// ------------------------------------------------------- workspace layout
// Decision keys of the tensor-core path: request b's keys (one per
// position) start a 4 KB row of their own.  Every CTA posts and reads them
// through a position; keys packed into the same or nearby lines serialise
// at their L2 slices (4 KB apart measured 2 us faster per position than
// 128 B apart).
constexpr int kHintRowKeys = 512;
constexpr size_t kHintRowBytes = kHintRowKeys * sizeof(uint64_t);

// The control row (the device error word first) and the B key rows share
// one pitch, so a single 2-D memset of width 8 K over B + 1 rows clears the
// error word and the keys of every position at the start of a block.
struct WorkspaceLayout {
  size_t control;   // one key row at offset 0: int 0 is the device error
                    // word (the rest of the row is unused)
  size_t hints;     // [B] rows of kHintRowKeys uint64 right after it; key k
                    // of row b is the best decision key posted for
                    // (b, position k)
  size_t stats;     // [2, B, kMaxChunks] ChunkStat: two buffers, so that a
                    // position's statistics survive the next position
  size_t rowstats;  // [B, K, 2] float (M, S)
  size_t total;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) {
  return (x + a - 1) / a * a;
}

__host__ __device__ inline WorkspaceLayout workspace_layout(int B, int K) {
  WorkspaceLayout L;
  size_t off = 0;
  L.control = off;
  off += kHintRowBytes;
  L.hints = off;
  off += (size_t)B * kHintRowBytes;
  L.stats = off;
  off = align_up(off + 2 * (size_t)B * kMaxChunks * sizeof(ChunkStat), 256);
  L.rowstats = off;
  off = align_up(off + (size_t)B * K * 2 * sizeof(float), 256);
  L.total = off;
  return L;
}

// Device error codes written to the control word.
enum DeviceError : int {
  kDevErrNone = 0,
  kDevErrBadToken = 1,  // a d0 entry outside [0, V) (token 0 used instead)
  kDevErrTimeout = 2,   // a bounded wait inside a kernel ran out
  kDevErrBadTemperature = 3,  // a per-request temperature not finite and > 0
  kDevErrBadSlot = 4,   // a proposal slot outside [0, num_slots)
  kDevErrBadPosition = 5,  // a sampler position outside [0, 65535] (0 used)
};

// ------------------------------------------------------- kernel launchers
struct DraftArgs {
  const void* base;
  int base_dtype;
  const void* U;
  const void* Wb;
  int w_dtype;
  const int32_t* d0;
  const uint64_t* seed;
  const uint64_t* offset;
  float T;
  const uint8_t* greedy;
  const uint8_t* pad_row;
  int B, K, V, r;
  int32_t* tokens;
  float* logits;
  float* probs;
  ChunkStat* stats;
  float* rowstats;
  unsigned long long* hints;  // [B] x kHintRowKeys; keys 0..K-1 zeroed per block
  // per-request entry point: temperature [B] (device) replaces T; request
  // b's proposals go to draft_probs slot slot[b] of num_slots (both null /
  // 0 otherwise)
  const float* temperature;
  const int32_t* slot;
  int num_slots;
  int* control;
};

// The temperature of request b: its own when the call gives per-request
// temperatures (a value that is not finite and positive counts as 1), else
// the block's T.
__device__ __forceinline__ float request_temperature(const DraftArgs& a, int b) {
  if (a.temperature == nullptr) return a.T;
  const float t = a.temperature[b];
  return (t > 0.0f && t <= 3.40282347e38f) ? t : 1.0f;
}

// Launch helpers (each returns the cudaGetLastError of its launch).
cudaError_t launch_position_generic(const DraftArgs& a, int k, int n_chunks,
                                    cudaStream_t stream);
bool position_tc_supported(const DraftArgs& a);
int position_tc_groups(int B);
int position_tc_chunks(int V, int sm_count);
cudaError_t launch_position_tc(const DraftArgs& a, int k, int n_chunks,
                               cudaStream_t stream);
// overlap_previous: launched with programmatic stream serialisation (the
// kernel waits for the previous grid before reading its statistics).
// buf: the statistics buffer position k filled; from_keys: d_k is read from
// the decision keys (tensor-core path) instead of the merged statistics.
cudaError_t launch_pick(const DraftArgs& a, int k, int n_chunks, int buf,
                        bool from_keys, bool overlap_previous,
                        cudaStream_t stream);
// Proposals of positions k_first .. k_first + k_count - 1.
cudaError_t launch_proposals(const DraftArgs& a, int k_first, int k_count,
                             cudaStream_t stream);
// block: the block-verification rule instead of the standard one.
cudaError_t launch_verify(const float* q, const float* p, const int32_t* tokens,
                          const uint64_t* seed, const uint64_t* offset, int B,
                          int K, int V, int32_t* accepted_len,
                          int32_t* emitted, int sms, bool block,
                          cudaStream_t stream);
// Temperature-only sampler: chunk statistics of the rows of a.logits
// (a.B rows, a.K == 1) into statistics buffer 0.
int sample_chunks(int R, int V, int sm_count);
cudaError_t launch_sample_stats(const DraftArgs& a, const int32_t* position,
                                int n_chunks, cudaStream_t stream);
cudaError_t launch_noise_words(uint64_t seed, uint64_t offset, int k,
                               int stream_id, int n, uint32_t* out,
                               float* gumbel, bool folded,
                               cudaStream_t stream);

}  // namespace dspark
