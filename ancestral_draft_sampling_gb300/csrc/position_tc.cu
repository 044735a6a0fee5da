// position_tc.cu -- one draft position with the Markov bias on the 5th-gen
// tensor cores (tcgen05), for bfloat16 heads.
//
// brb-nv/TensorRT-LLM PR #27, "2. One fused kernel per draft position":
// bias(d_{k-1}) = U[d_{k-1}] @ Wb, added to the drafter logits, scaled by
// 1/T, Gumbel-max with Philox noise, float32 biased logits and per-chunk
// softmax statistics out.  The pages keep the bias GEMM on cuBLAS; here it
// is fused into the position kernel.
//
// Per CTA (one per SM; CTA c takes the 128-wide vocab tiles c, c + grid, ...):
//   warp 0, lane 0  TMA producer of Wb[r0:r0+64, v0:v0+128] stages (two
//                   64x64 boxes, 128-byte swizzle) into a ring.
//   warp 0, lane 1  TMA producer of the drafter-logit tile base[:, k,
//                   v0:v0+128] ([Bpad x 128], rows past B read as zero),
//                   straight into one of two float32 tile buffers (bf16
//                   logits go to a staging tile instead).
//   warp 1, lane 0  MMA issuer: D[v, b] = sum_j Wb[j, v] * u[b, j] with
//                   tcgen05.mma kind::f16 (M = 128 vocab rows, N = B rounded
//                   up to 16, K = r) into one of two TMEM accumulators.  A
//                   (the Wb tile) is vocab-major, B (u) is r-major.
//   warps 2..9      drain.  Warp (q, h), q = warp % 4, drains TMEM lanes
//                   32q.. (vocab) of the 16-column groups 2g+h (requests)
//                   and writes l = base + bias (l = bias on padding rows)
//                   into the tile buffer, in place; once all eight have, one
//                   thread stores the tile to global memory with a TMA tile
//                   store.  They drain tile t+1 while the decision warps
//                   work on tile t.
//   warps 10..31    decision.  Warp w takes requests w-10, w+12, ... with
//                   lane L on vocab 4L .. 4L+3 (one Philox block): scaled
//                   logits, noise, the decision and the sum-exp, all from
//                   shared memory.
// Decision: a conservative test per entry (one exp2, no logarithm) admits
// every entry that may beat a reference score; only those get the exact
// score s + g, merged over the warp by max/min reductions.  The reference
// is the larger of the request's best score in this CTA and the best score
// any CTA has posted for the request so far: a score some entry reaches, so
// an entry below it cannot win.  The posts are decision keys (the score's
// order-preserving bits above the complement of the index) combined by an
// atomic maximum in global memory and read once per tile.  The sum-exp
// reuses the test's exp2 values, relative to a reference set from the data
// alone.  The Philox rounds that depend only on the request's key and
// counter words are folded into per-request constants.
//
// Once the grid has finished, the key of each request is the winner of the
// position (largest score, lowest index on ties): the next position's
// kernel reads d_{k-1} from it directly, so consecutive positions follow
// each other with no kernel between them.  While its pipeline fills, that
// kernel's decision warps also merge the previous position's per-chunk
// statistics into tokens[:, k-1] and its softmax statistics (M, S); the
// statistics alternate between two buffers, so position k never overwrites
// those of position k-1.
//
// Every mbarrier wait is bounded; on a timeout the kernel records an error
// in the workspace control word, stops issuing work, waits (bounded) for
// its in-flight copies and MMAs, frees its TMEM and returns.
#include <cudaTypedefs.h>

#include <cstdlib>
#include <mutex>

#include "dspark_common.cuh"
#include "sm100_ptx.cuh"

namespace dspark {
namespace {

using namespace sm100;

constexpr int kTileV = 128;                        // vocab rows per tile (M)
constexpr int kKChunk = 64;                        // r per pipeline stage
constexpr int kBoxBytes = 64 * kKChunk * 2;        // one 64x64 bf16 box
constexpr int kStageBytes = 2 * kBoxBytes;         // 128 vocab x 64 r
constexpr int kDrainWarps = 8;                     // two per TMEM lane quarter
constexpr int kComputeWarps = 22;                  // the decision warps
constexpr int kWorkWarps = kDrainWarps + kComputeWarps;
constexpr int kThreads = 32 * (2 + kWorkWarps);
constexpr int kWorkThreads = 32 * kWorkWarps;      // set-up and u gather
constexpr int kDrainThreads = 32 * kDrainWarps;
constexpr int kComputeThreads = 32 * kComputeWarps;
constexpr int kMaxBpad = 96;
constexpr int kGatherBatch = 4;                    // u pieces a thread loads at once
constexpr int kMaxRows = (kMaxBpad + kComputeWarps - 1) / kComputeWarps;  // requests per compute warp
constexpr uint32_t kTmemCols = 256;                // two accumulators
constexpr uint32_t kAccCols = 128;
constexpr uint32_t kSpin = 1u << 22;
constexpr uint32_t kStallPolls = 1u << 12;  // the stalled wait's poll limit
// Fewest Wb stages the kernel runs with.  Two is what bf16 drafter logits
// leave at r = 256 and 81..96 requests (one staging tile): 519 us for a
// B=88, K=7, V=200064 block, against 4255 us on the FFMA kernel.
constexpr int kMinStages = 2;
constexpr int kMaxStages = 8;
constexpr size_t kSmemLimit = 232448;              // 227 KB per CTA
constexpr float kLog2e = 1.4426950408889634f;
// Slack of the candidate test in log2 units: the test admits entries up to a
// factor 2^(2^-11) = 1 + 3.4e-4 past the exact bound (32 + 2^-11 is exact in
// float32).
constexpr float kThrSlack = 0x1p-11f;
// exp(s - best) from the test value 2^(32 + slack) exp(s - best): the scale
// 2^-(32 + 2^-11), rounded to float32 (relative error < 2^-24)
constexpr float kSumScale = 2.3275186e-10f;

// Per-request constants in shared memory.  The Philox round keys of the
// request's key (seed) are precomputed, so a noise block costs the ten
// rounds' multiplies and XORs only.
struct alignas(16) RowConst {
  uint4 pre;     // rounds 1-2 folded: (C1, D2, E2, F2), see row_noise
  uint4 rk[4];   // round keys of rounds 3..10: rk[j] = rounds 2j+3, 2j+4
  uint32_t flags;  // bit 0: padding row, bit 1: greedy request
  float T;         // the request's temperature (per-request entry point)
  uint32_t pad[2];
};
constexpr uint32_t kRowPad = 1u, kRowGreedy = 2u;

struct TcParams {
  DraftArgs a;
  int k;
  int bpad;
  int stages;
  int stage_bufs;  // bf16 drafter-logit staging tiles (1 or 2; 0 for f32)
  int tiles_total;
  int stall_first_wait;  // failure-path test: the MMA issuer waits for a
                         // phase nothing completes, with a short limit
  int n_chunks;
  uint32_t u_off, tile_off, stage_off, rows_off, rstate_off, bar_off;
};

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Running state of one request in the compute warp that owns it:
//   sum        per lane: sum of exp(s - sref) over the lane's entries;
//   ref, idx   the same in every lane: the reference of the candidate test,
//              the largest decision score known (s + g for a sampled
//              request, s for a greedy one), and its vocab index when this
//              CTA reached it (kNoIndex when it was posted by another CTA,
//              or nothing has won).  An entry below ref cannot be the
//              request's winner, so this CTA's own best below ref is not
//              kept;
//   sref       the reference of the sum, set from the data alone (the
//              largest scaled logit of the first tile that has one above
//              -inf, moved only when a term would overflow), so that the sum
//              does not depend on when hints arrive;
//   h          exp(sref - ref), recomputed whenever ref or sref moves.
struct RowState {
  float sum, ref, sref, h;
  int idx;
};



// The constant of the candidate test for reference `ref`:
// 32 + 2^-11 - ref log2(e).  While nothing has won (ref = -inf) a huge
// finite constant stands in: every finite entry is then admitted, and a
// -inf entry adds exp2(-inf) = 0 to the sum.
__device__ __forceinline__ float thr_const(float ref) {
  return fmaf(-fmaxf(ref, -0x1p100f), kLog2e, 32.0f + kThrSlack);
}

// exp(sref - ref): turns a sum term into the candidate test value
// 2^(32+slack) exp(s - ref).  +inf while nothing has won (every finite entry
// is a candidate); clamped at 2^-100 so that it never flushes to zero (and a
// finite term times it stays finite).
__device__ __forceinline__ float ref_factor(float sref, float ref) {
  return ref == -INFINITY ? INFINITY
                          : ex2_approx(fmaxf((sref - ref) * kLog2e, -100.0f));
}

// 2^(32 + slack) exp(s - best).  A sampled entry wins only if s + g > best
// with g = -log E, E = -log(1 - w) increasing in w = (x + 0.5) 2^-32, i.e.
// only if w < 1 - exp(-(s - best)) <= exp(s - best).  The test
// (float)x < this value is therefore conservative: the slack covers the
// approximate exp2, the rounding of x and the error of the float32 score,
// and entries that pass are decided exactly.
__device__ __forceinline__ float test_value(float s, float tc) {
  return ex2_approx(fmaf(s, kLog2e, tc));
}

__device__ __forceinline__ float pick4(const float (&a)[4], int e) {
  return e == 0 ? a[0] : e == 1 ? a[1] : e == 2 ? a[2] : a[3];
}

// Scaled logit: the float32 IEEE quotient l / T; division by 1 is exact.
template <bool kUnitT>
__device__ __forceinline__ float scale(float l, float T) {
  return kUnitT ? l : __fdiv_rn(l, T);
}

// Keeps the better of st and the warp's candidates (cb, ci): the largest
// score by a max-reduction over order-preserving bits, then the lowest index
// among the lanes that hold it by a min-reduction.  Lanes without a
// candidate offer key 0 (below every score, -inf included).
__device__ __forceinline__ void warp_take_best(RowState& st, float cb, int ci) {
  const uint32_t key = ci == kNoIndex ? 0u : ordered_bits(cb);
  const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
  if (kmax == 0u) return;
  const uint32_t imin = __reduce_min_sync(
      0xffffffffu, key == kmax ? (uint32_t)ci : 0xffffffffu);
  const float wb = from_ordered_bits(kmax);
  // beats the reference, or reaches it at a lower index than a reference of
  // this CTA's own (equal to another CTA's posted score: both are reported,
  // the pick keeps the lower index)
  if (wb > st.ref ||
      (wb == st.ref && (st.idx == kNoIndex || (int)imin < st.idx))) {
    st.ref = wb;
    st.idx = (int)imin;
    st.h = ref_factor(st.sref, wb);
  }
}

// The noise block of vocab v: Philox4x32-10 of counter (v >> 2, c1, c2, c3)
// under the request's key, from the request's folded constants.
__device__ __forceinline__ uint4 row_noise(const RowConst& rc, int v) {
  return philox_folded(rc.pre, rc.rk, (uint32_t)v >> 2);
}

// The folded constants of a request with key (k0, k1) and counter words
// c1, c2, c3.
__device__ __forceinline__ void row_constants(RowConst& rc, uint32_t k0,
                                              uint32_t k1, uint32_t c1,
                                              uint32_t c2, uint32_t c3) {
  philox_fold(rc.pre, rc.rk, k0, k1, c1, c2, c3);
}

// Exact decision scores of the sampled entries in `cand`, merged into st.
__device__ __forceinline__ void decide_sampled(RowState& st, uint32_t cand,
                                               const float (&s)[4],
                                               const uint4 w, int v) {
  float cb = -INFINITY;
  int ci = kNoIndex;
  while (cand) {
    const int e = __ffs(cand) - 1;
    cand &= cand - 1u;
    const float sc =
        __fadd_rn(pick4(s, e), -logf(exponential_from_word(word_of(w, e))));
    if (sc > cb) {  // e ascending: strict keeps the lower index
      cb = sc;
      ci = v + e;
    }
  }
  warp_take_best(st, cb, ci);
}

// The largest scaled logit of the warp's 128 entries (NaN ignored; -inf if
// there is none above -inf).
__device__ __forceinline__ float warp_max_scaled(const float (&s)[4]) {
  float m = -INFINITY;
#pragma unroll
  for (int e = 0; e < 4; ++e)
    if (s[e] > m) m = s[e];
  return from_ordered_bits(__reduce_max_sync(0xffffffffu, ordered_bits(m)));
}

// The sum's terms relative to sref, scaled: f = 2^(32+slack) exp(s - sref).
// While sref is unset (-inf) every term above -inf is +inf, which makes it a
// candidate; the candidate path then sets sref (rebase_sum).
__device__ __forceinline__ void sum_terms(const RowState& st,
                                          const float (&s)[4], float (&f)[4]) {
  const float tc = thr_const(st.sref);
#pragma unroll
  for (int e = 0; e < 4; ++e) f[e] = test_value(s[e], tc);
}

// A term at or above 2^100 (always a candidate) means sref is unset or s -
// sref nears float32's range: sref moves to this tile's largest scaled
// logit (a value fixed by the data), the sum is rescaled to it (from an
// unset sref the sum is 0, or NaN after a NaN entry) and the terms are
// recomputed.  Warp-uniform.
__device__ __forceinline__ void rebase_sum(RowState& st, const float (&s)[4],
                                           float (&f)[4]) {
  const bool big = f[0] >= 0x1p100f || f[1] >= 0x1p100f ||
                   f[2] >= 0x1p100f || f[3] >= 0x1p100f;
  if (__any_sync(0xffffffffu, big)) {
    const float r = warp_max_scaled(s);
    if (r > st.sref) {
      st.sum *= ex2_approx((st.sref - r) * kLog2e);
      st.sref = r;
      st.h = ref_factor(r, st.ref);
      sum_terms(st, s, f);
    }
  }
}

// The sum-exp of four entries relative to sref: the terms, scaled back.
__device__ __forceinline__ void accumulate(RowState& st, const float (&f)[4]) {
  st.sum = fmaf(__fadd_rn(__fadd_rn(f[0], f[1]), __fadd_rn(f[2], f[3])),
                kSumScale, st.sum);
}

// A best score posted by another CTA (the order-preserving bits of a
// decision key's score, 0 = none) raises the reference of the candidate
// test.
__device__ __forceinline__ void adopt_hint(RowState& st, uint32_t h) {
  if (h > ordered_bits(st.ref)) {
    st.ref = from_ordered_bits(h);
    st.idx = kNoIndex;  // another CTA's entry
    st.h = ref_factor(st.sref, st.ref);
  }
}

// Steady state of a sampled request (its best is finite): the conservative
// test for every entry, exact scores for the few that pass.  kVote: the
// warp's vote takes the OR of the four tests and the rare path works out
// which entries pass (fewer instructions, more live registers: used where
// no division per entry competes for them).
template <bool kVote>
__device__ __forceinline__ void sampled_step(const uint4 w,
                                             const float (&s)[4], int v,
                                             RowState& st) {
  float f[4];
  sum_terms(st, s, f);
  const float h = st.h;
  uint32_t cand = 0;
  bool any;
  if (kVote) {
    any = (__uint2float_rz(w.x) < __fmul_ru(f[0], h)) |
          (__uint2float_rz(w.y) < __fmul_ru(f[1], h)) |
          (__uint2float_rz(w.z) < __fmul_ru(f[2], h)) |
          (__uint2float_rz(w.w) < __fmul_ru(f[3], h));
  } else {
    cand = (__uint2float_rz(w.x) < __fmul_ru(f[0], h) ? 1u : 0u) |
           (__uint2float_rz(w.y) < __fmul_ru(f[1], h) ? 2u : 0u) |
           (__uint2float_rz(w.z) < __fmul_ru(f[2], h) ? 4u : 0u) |
           (__uint2float_rz(w.w) < __fmul_ru(f[3], h) ? 8u : 0u);
    any = cand != 0u;
  }
  if (__any_sync(0xffffffffu, any)) {
    if (kVote)
      cand = (__uint2float_rz(w.x) < __fmul_ru(f[0], h) ? 1u : 0u) |
             (__uint2float_rz(w.y) < __fmul_ru(f[1], h) ? 2u : 0u) |
             (__uint2float_rz(w.z) < __fmul_ru(f[2], h) ? 4u : 0u) |
             (__uint2float_rz(w.w) < __fmul_ru(f[3], h) ? 8u : 0u);
    decide_sampled(st, cand, s, w, v);
    rebase_sum(st, s, f);
  }
  accumulate(st, f);
}

// Approximate decision score s - log E, used only to choose which entry of
// a chunk's first tile to decide exactly (accuracy does not matter for the
// result: every entry is then tested conservatively against the exact best).
__device__ __forceinline__ float rough_score(float s, uint32_t x) {
  const float w = fmaf(__uint2float_rz(x), 0x1p-32f, 0x1p-33f);
  const float e = w < 0x1p-10f ? w : -__logf(__fsub_rn(1.0f, w));
  return s - __logf(e);
}

// First tile of a sampled request (nothing has won yet): each lane decides
// its roughly best entry exactly, the warp keeps the best of those, then
// the remaining entries go through the conservative test.
__device__ __forceinline__ void sampled_first(const uint4 w,
                                              const float (&s)[4], int v,
                                              RowState& st) {
  uint32_t first = 0;
  float top = -INFINITY;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float a = s[e] == -INFINITY ? -INFINITY : rough_score(s[e], word_of(w, e));
    if (a > top) {
      top = a;
      first = 1u << e;
    }
  }
  decide_sampled(st, first, s, w, v);
  float f[4];
  sum_terms(st, s, f);
  rebase_sum(st, s, f);  // sets sref on the first tile with a value
  const float h = st.h;
  uint32_t cand = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e)
    cand |= (__uint2float_rz(word_of(w, e)) < __fmul_ru(f[e], h) ? 1u : 0u) << e;
  cand &= ~first;
  if (__any_sync(0xffffffffu, cand != 0u)) decide_sampled(st, cand, s, w, v);
  accumulate(st, f);
}

// sampled_first out of line: it runs once per request and CTA, and inlined
// into every row of the unrolled row loop it made the kernel's code large
// enough to slow the steady state (measured 5 us per block).  Arguments and
// result go by value, so the caller's arrays stay in registers.
__device__ __noinline__ RowState sampled_first_call(const uint4 w, const float4 s4,
                                                    int v, RowState st) {
  const float s[4] = {s4.x, s4.y, s4.z, s4.w};
  sampled_first(w, s, v, st);
  return st;
}

// A greedy request: no noise; an entry is a candidate iff s > best.
__device__ __forceinline__ void greedy_step(const float (&s)[4], int v,
                                            RowState& st) {
  const float old_best = st.ref;
  uint32_t cand = (s[0] > old_best ? 1u : 0u) | (s[1] > old_best ? 2u : 0u) |
                  (s[2] > old_best ? 4u : 0u) | (s[3] > old_best ? 8u : 0u);
  if (__any_sync(0xffffffffu, cand != 0u)) {
    float cb = -INFINITY;
    int ci = kNoIndex;
    while (cand) {
      const int e = __ffs(cand) - 1;
      cand &= cand - 1u;
      if (pick4(s, e) > cb) {
        cb = pick4(s, e);
        ci = v + e;
      }
    }
    warp_take_best(st, cb, ci);
  }
  float f[4];
  sum_terms(st, s, f);
  rebase_sum(st, s, f);
  accumulate(st, f);
}

template <bool kUnitT>
__device__ __forceinline__ void scaled4(const float4 l4, float T,
                                        float (&s)[4]) {
  s[0] = scale<kUnitT>(l4.x, T);
  s[1] = scale<kUnitT>(l4.y, T);
  s[2] = scale<kUnitT>(l4.z, T);
  s[3] = scale<kUnitT>(l4.w, T);
}

// kRowT: per-request temperatures (the per-request entry point); each row
// divides by its own T, rows whose T is 1 skip the division.
template <typename BT, bool kUnitT, bool kRowT>
__global__ void __launch_bounds__(kThreads, 1)
position_tc_kernel(const __grid_constant__ CUtensorMap wb_map,
                   const __grid_constant__ CUtensorMap base_map,
                   const __grid_constant__ CUtensorMap out_map,
                   const __grid_constant__ TcParams P) {
  constexpr bool kStaged = sizeof(BT) == 2;  // bf16 logits: via a staging tile
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* ring = smem;
  uint8_t* u_s = smem + P.u_off;
  float* tiles = reinterpret_cast<float*>(smem + P.tile_off);
  const BT* stage = reinterpret_cast<const BT*>(smem + P.stage_off);
  RowConst* rows = reinterpret_cast<RowConst*>(smem + P.rows_off);
  const int S = P.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + P.bar_off);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* base_full = acc_empty + 2;
  uint64_t* tile_free = base_full + 2;
  uint64_t* stage_free = tile_free + 2;  // [2]: staging tiles read
  uint64_t* mma_done = stage_free + 2;
  uint64_t* u_ready = mma_done + 1;
  uint64_t* drained = u_ready + 1;  // [2]: the drain warps have filled a buffer
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drained + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const DraftArgs& a = P.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x;
  // tiles chunk, chunk + n_chunks, ...: at any moment the CTAs work on
  // neighbouring tiles (measured faster than contiguous ranges)
  const int n_tiles = (P.tiles_total - 1 - chunk) / P.n_chunks + 1;
  // r-chunks of kKChunk; the last one may be partial (r % 16 == 0): its Wb
  // rows past r load as zeros (TMA fill) and the gather writes zeros into
  // its u rows past r, so the MMA's K steps there add exactly 0
  const int kchunks = (a.r + kKChunk - 1) / kKChunk;
  const int tile_floats = P.bpad * kTileV;
  // bf16 drafter logits: staging tile and phase of tile t (one or two
  // staging tiles, see make_layout)
  auto stage_of = [&](int t) { return P.stage_bufs == 2 ? (t & 1) : 0; };
  auto stage_parity = [&](int t) {
    return (uint32_t)(P.stage_bufs == 2 ? (t >> 1) : t) & 1u;
  };

  auto fail = [&](int code) {
    *abort_flag = 1;
    a.control[0] = code;
  };

  // ------------------------------------------------------------ set-up
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kDrainThreads);
      mbar_init(&base_full[i], 1);
      mbar_init(&tile_free[i], kComputeThreads + 1);  // + the storer
      mbar_init(&drained[i], kDrainThreads);
    }
    mbar_init(&stage_free[0], kDrainThreads);
    mbar_init(&stage_free[1], kDrainThreads);
    mbar_init(mma_done, 1);
    mbar_init(u_ready, kWorkThreads);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&wb_map);
    prefetch_tmap(&base_map);
    prefetch_tmap(&out_map);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  if (warp >= 2) {
    // per-request constants (inputs only: they may be read before the
    // previous position's kernel has finished)
    const int ct = threadIdx.x - 64;
    for (int b = ct; b < P.bpad; b += kWorkThreads) {
      RowConst rc;
      uint32_t k0 = 0, k1 = 0, c2 = 0, c3 = 0;
      rc.flags = 0;
      rc.T = 1.0f;
      rc.pad[0] = rc.pad[1] = 0;
      if (b < a.B) {
        k0 = (uint32_t)a.seed[b];
        k1 = (uint32_t)(a.seed[b] >> 32);
        c2 = (uint32_t)a.offset[b];
        c3 = (uint32_t)(a.offset[b] >> 32);
        rc.flags = (a.pad_row != nullptr && a.pad_row[b] != 0 ? kRowPad : 0u) |
                   (a.greedy != nullptr && a.greedy[b] != 0 ? kRowGreedy : 0u);
        if (kRowT) rc.T = request_temperature(a, b);
      }
      row_constants(rc, k0, k1, (uint32_t)P.k | ((uint32_t)kNoiseDraft << 16),
                    c2, c3);
      rows[b] = rc;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the pick kernel that follows may be scheduled now; it waits for this
  // grid to finish before it reads the statistics
  if (threadIdx.x == 0) launch_dependents();
  const uint32_t tmem_base = *tmem_holder;
  // loads issued by the two producers (warp 0, lanes 0 and 1): after an
  // abort, the teardown waits for them to land before the CTA exits
  int wb_issued = 0, base_issued = 0;

  if (warp == 0) {
    if (lane == 0) {
      // -------------------------------------------------- Wb producer
      int& g = wb_issued;
      for (int t = 0; t < n_tiles && !*abort_flag; ++t) {
        const int v0 = (chunk + t * P.n_chunks) * kTileV;
        for (int kc = 0; kc < kchunks; ++kc, ++g) {
          const int s = g % S;
          const uint32_t ph = (uint32_t)(g / S) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, kSpin)) {
            fail(kDevErrTimeout);
            break;
          }
          mbar_arrive_expect_tx(&full[s], kStageBytes);
          uint8_t* dst = ring + (size_t)s * kStageBytes;
          tma_load_2d(dst, &wb_map, &full[s], v0, kc * kKChunk);
          tma_load_2d(dst + kBoxBytes, &wb_map, &full[s], v0 + 64, kc * kKChunk);
        }
      }
    } else if (lane == 1) {
      // ----------------------------------------- drafter-logit producer
      const uint32_t bytes = (uint32_t)(tile_floats * (int)sizeof(BT));
      int& issued = base_issued;
      for (int t = 0; t < n_tiles && !*abort_flag; ++t, ++issued) {
        const int v0 = (chunk + t * P.n_chunks) * kTileV;
        if (kStaged) {
          const int sb = stage_of(t);
          if (!mbar_wait(&stage_free[sb], stage_parity(t) ^ 1u, kSpin)) {
            fail(kDevErrTimeout);
            break;
          }
          mbar_arrive_expect_tx(&base_full[sb], bytes);
          tma_load_2d(const_cast<BT*>(stage) + (size_t)sb * tile_floats, &base_map,
                      &base_full[sb], v0, 0);
        } else {
          const int buf = t & 1;
          if (!mbar_wait(&tile_free[buf], ((uint32_t)(t >> 1) & 1u) ^ 1u, kSpin)) {
            fail(kDevErrTimeout);
            break;
          }
          mbar_arrive_expect_tx(&base_full[buf], bytes);
          tma_load_2d(tiles + (size_t)buf * tile_floats, &base_map, &base_full[buf], v0, 0);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kTileV, (uint32_t)P.bpad, 1u, 0u);
      const uint32_t u_base = smem_u32(u_s);
      bool u_ok = mbar_wait(u_ready, 0u, kSpin);
      // failure-path test: once u is ready, a wait for the barrier's second
      // phase, which nothing completes (u_ready takes one round of arrivals
      // per launch)
      if (u_ok && P.stall_first_wait) u_ok = mbar_wait(u_ready, 1u, kStallPolls);
      if (!u_ok) fail(kDevErrTimeout);
      int g = 0;
      for (int t = 0; t < n_tiles && !*abort_flag; ++t) {
        const int acc = t & 1;
        const uint32_t aph = (uint32_t)(t >> 1) & 1u;
        if (!mbar_wait(&acc_empty[acc], aph ^ 1u, kSpin)) {
          fail(kDevErrTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)acc * kAccCols;
        bool ok = true;
        for (int kc = 0; kc < kchunks; ++kc, ++g) {
          const int s = g % S;
          const uint32_t ph = (uint32_t)(g / S) & 1u;
          if (!mbar_wait(&full[s], ph, kSpin)) {
            fail(kDevErrTimeout);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(ring + (size_t)s * kStageBytes);
          const uint32_t b_base = u_base + (uint32_t)(kc * P.bpad * 128);
#pragma unroll
          for (int sub = 0; sub < kKChunk / 16; ++sub) {
            // A: vocab-major, 64-vocab atoms kBoxBytes apart (LBO), 8-row r
            // groups 1024 B apart (SBO); 16 r rows = 2048 B per K step.
            const uint64_t adesc =
                smem_desc_sw128(a_base + sub * 2048, kBoxBytes, 1024);
            // B: r-major rows of 128 B, 8-row groups 1024 B apart (SBO);
            // a 16-wide K step is 32 B inside the swizzled row.
            const uint64_t bdesc = smem_desc_sw128(b_base + sub * 32, 16, 1024);
            mma_bf16(d_tmem, adesc, bdesc, idesc, (kc | sub) != 0 ? 1u : 0u);
          }
          mma_commit(&empty[s]);
        }
        if (!ok) break;
        mma_commit(&acc_full[acc]);
      }
      // all MMAs this thread issued are complete before TMEM is released
      mma_commit(mma_done);
      mbar_wait(mma_done, 0u, kSpin);
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------- compute
    // u row b = U[d_{k-1}(b)], stored r-major with the 128-byte swizzle: row
    // b of r-chunk c at c*(bpad*128) + b*128, 16-byte piece p at (p ^ (b & 7)).
    // d_{k-1} comes from the previous position's kernel: wait for it first.
    // A thread issues the token loads of kGatherBatch pieces, then their U
    // loads, then the stores: two memory round trips per batch.
    grid_dependency_wait();
    {
    const int ct = threadIdx.x - 64;
    const int pieces = kchunks * (kKChunk / 8);  // 16-byte pieces, whole chunks
    const int valid = a.r / 8;                   // pieces that hold U values
    const int total = P.bpad * pieces;
    const uint16_t* U = static_cast<const uint16_t*>(a.U);
    for (int i0 = ct; i0 < total; i0 += kWorkThreads * kGatherBatch) {
      int prev[kGatherBatch];
#pragma unroll
      for (int j = 0; j < kGatherBatch; ++j) {
        const int i = i0 + j * kWorkThreads, b = i / pieces;
        prev[j] = 0;
        if (i < total && b < a.B)
          prev[j] = (P.k == 0) ? a.d0[b]
                               : key_token(a.hints[(size_t)b * kHintRowKeys + (P.k - 1)]);
      }
      uint4 val[kGatherBatch];
#pragma unroll
      for (int j = 0; j < kGatherBatch; ++j) {
        const int i = i0 + j * kWorkThreads, b = i / pieces, piece = i - b * pieces;
        val[j] = make_uint4(0u, 0u, 0u, 0u);
        if (i < total && b < a.B && piece < valid) {
          int pv = prev[j];
          if ((unsigned)pv >= (unsigned)a.V) {
            if (piece == 0) a.control[0] = kDevErrBadToken;
            pv = 0;
          }
          val[j] = __ldg(reinterpret_cast<const uint4*>(U + (size_t)pv * a.r) + piece);
        }
      }
#pragma unroll
      for (int j = 0; j < kGatherBatch; ++j) {
        const int i = i0 + j * kWorkThreads, b = i / pieces, piece = i - b * pieces;
        const int c = piece >> 3, p = piece & 7;
        if (i < total)
          *reinterpret_cast<uint4*>(u_s + (size_t)c * (P.bpad * 128) + b * 128 +
                                    ((p ^ (b & 7)) << 4)) = val[j];
      }
    }
    }
    fence_proxy_async_smem();  // the MMA reads u through the async proxy
    mbar_arrive(u_ready);
    if (warp < 2 + kDrainWarps) {
      // ----------------------------------------------------------- drain
      // Warp q drains TMEM lanes 32q.. (vocab rows m of the tile) for every
      // request, adds the bias into the drafter-logit tile in place (l =
      // bias on padding rows), and then the tile is stored with one TMA
      // store while the compute warps take the previous tile.
      const int q = warp & 3;                // TMEM lane quarter
      const int h = (warp - 2) >> 2;         // column half: 16-column groups 2g+h
      const int m = 32 * q + lane;           // drained vocab row of the tile
      const bool storer = warp == 2 && lane == 0;
      // bit c & 31 of word c >> 5: request c is a padding row
      uint32_t pad0 = 0, pad1 = 0, pad2 = 0;
      static_assert(kMaxBpad <= 96, "three padding words");
      for (int c = 0; c < a.B; ++c)
        if (rows[c].flags & kRowPad) {
          const uint32_t bit = 1u << (c & 31);
          if (c < 32) pad0 |= bit; else if (c < 64) pad1 |= bit; else pad2 |= bit;
        }
      for (int t = 0; t < n_tiles; ++t) {
        const int buf = t & 1;
        const uint32_t ph = (uint32_t)(t >> 1) & 1u;
        const int v0 = (chunk + t * P.n_chunks) * kTileV;
        float* tile = tiles + (size_t)buf * tile_floats;
        // bf16 logits arrive in a staging tile, so the f32 buffer is
        // written here: it must be released (tile t-2 read by the compute
        // warps and the store) first; f32 logits were loaded into it by TMA
        // only after that release
        const int sb = kStaged ? stage_of(t) : buf;
        const BT* stage_t = stage + (size_t)sb * tile_floats;
        bool ok = !*abort_flag &&
                  (!kStaged || mbar_wait(&tile_free[buf], ph ^ 1u, kSpin)) &&
                  mbar_wait(&base_full[sb], kStaged ? stage_parity(t) : ph, kSpin) &&
                  mbar_wait(&acc_full[buf], ph, kSpin);
        ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld needs the whole warp
        if (ok) {
          tc_fence_after();
          const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) +
                                 (uint32_t)buf * kAccCols;
          float* col = tile + m;
#pragma unroll 1
          for (int c0 = 16 * h; c0 < a.B; c0 += 32) {
            float bias[16];
            tmem_ld16(taddr + (uint32_t)c0, bias);  // within the 128 columns
            const uint32_t pw =
                (c0 < 32 ? pad0 : (c0 < 64 ? pad1 : pad2)) >> (c0 & 31);
            if (c0 + 16 <= a.B) {
              // all 16 requests present: the drafter logits are read while
              // the TMEM load is in flight
              float x[16];
#pragma unroll
              for (int j = 0; j < 16; ++j)
                x[j] = kStaged ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(
                                                     stage_t)[(c0 + j) * kTileV + m] << 16)
                               : col[(c0 + j) * kTileV];
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 16; ++j)
                col[(c0 + j) * kTileV] =
                    ((pw >> j) & 1u) ? bias[j] : __fadd_rn(x[j], bias[j]);
            } else {
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int c = c0 + j;
                if (c >= a.B) break;
                float x;
                if (kStaged)
                  x = __uint_as_float(
                      (uint32_t)reinterpret_cast<const uint16_t*>(stage_t)[c * kTileV + m] << 16);
                else
                  x = col[c * kTileV];
                col[c * kTileV] = ((pw >> j) & 1u) ? bias[j] : __fadd_rn(x, bias[j]);
              }
            }
          }
          // the ragged last tile: vocab rows past V become -inf, which no
          // decision admits and the sum ignores (the logits store clips them)
          if (v0 + kTileV > a.V && v0 + m >= a.V) {
            for (int c = 0; c < a.B; ++c)
              if (((c >> 4) & 1) == h) col[c * kTileV] = -INFINITY;
          }
          tc_fence_before();
        } else if (!*abort_flag) {
          fail(kDevErrTimeout);
        }
        mbar_arrive(&acc_empty[buf]);
        if (kStaged) mbar_arrive(&stage_free[sb]);
        fence_proxy_async_smem();         // the tile store reads these writes
        named_sync(1, kDrainThreads);     // the whole tile is drained
        if (storer && !*abort_flag) {
          tma_store_2d(&out_map, tile, v0, 0);
          bulk_commit();
        }
        mbar_arrive(&drained[buf]);
        if (storer) {
          bulk_wait_read_all();  // the store has read the tile
          mbar_arrive(&tile_free[buf]);
        }
      }
      if (storer) bulk_wait_all();
    } else {
    // ------------------------------------------------------------- compute
    const int cw = warp - 2 - kDrainWarps;
    // lane i < kMaxRows: the decision key of this warp's row i
    unsigned long long* hint_ptr = nullptr;
    {
      const int hb = cw + kComputeWarps * lane;
      if (lane < kMaxRows && hb < a.B)
        hint_ptr = a.hints + (size_t)hb * kHintRowKeys + P.k;
    }
    uint32_t greedy_mask = 0;  // bit i: this warp's row i is greedy
#pragma unroll
    for (int i = 0; i < kMaxRows; ++i) {
      const int b = cw + kComputeWarps * i;
      if (b < a.B && (rows[b].flags & kRowGreedy)) greedy_mask |= 1u << i;
    }
    const float T = a.T;
    // The warp-uniform part of each request's state (ref, sref, h, idx)
    // lives in shared memory between row steps, the per-lane sums in
    // registers.  Every lane stores the same values and reads back its own
    // store, so only the initialisation (by lanes 0..kMaxRows-1) needs a
    // warp sync.
    float sums[kMaxRows];
    float4* rstate = reinterpret_cast<float4*>(smem + P.rstate_off) + cw * kMaxRows;
#pragma unroll
    for (int i = 0; i < kMaxRows; ++i) sums[i] = 0.0f;
    if (lane < kMaxRows)  // nothing won, no reference yet
      rstate[lane] = make_float4(-INFINITY, -INFINITY, INFINITY,
                                 __int_as_float(kNoIndex));
    __syncwarp();
    // the previous position, complete since grid_dependency_wait: d_{k-1}
    // from its decision key and (M, S) from its merged statistics, one
    // request per warp, while the first tile is still in flight
    if (P.k > 0) {
      for (int b = chunk + P.n_chunks * cw; b < a.B;
           b += P.n_chunks * kComputeWarps) {
        const ChunkStat ps = merge_row(
            stat_slot(a.stats, (P.k - 1) & 1, a.B, b, 0), P.n_chunks, lane);
        if (lane == 0) {
          const size_t row = (size_t)b * a.K + (P.k - 1);
          a.tokens[row] = key_token(a.hints[(size_t)b * kHintRowKeys + (P.k - 1)]);
          a.rowstats[2 * row] = ps.m;
          a.rowstats[2 * row + 1] = ps.s;
        }
      }
    }

    for (int t = 0; t < n_tiles; ++t) {
      const int buf = t & 1;
      const uint32_t ph = (uint32_t)(t >> 1) & 1u;
      const int v0 = (chunk + t * P.n_chunks) * kTileV;
      const float* tile = tiles + (size_t)buf * tile_floats;
      const unsigned long long hint_in = hint_ptr ? __ldcg(hint_ptr) : 0ull;
      // the drain warps have written this tile's biased logits
      const bool ok = !*abort_flag && mbar_wait(&drained[buf], ph, kSpin);
      if (!ok && !*abort_flag) fail(kDevErrTimeout);
      bool released = false;
      if (ok && !*abort_flag) {
        const int v = v0 + 4 * lane;
#pragma unroll
        for (int i0 = 0; i0 < kMaxRows; i0 += 2) {
          const int b0 = cw + kComputeWarps * i0;
          if (b0 >= a.B) break;
          const bool has1 = i0 + 1 < kMaxRows && b0 + kComputeWarps < a.B;
          // T = 1: the last pair's values go to registers first, and the
          // buffer can take the next tile while this pair is decided
          // (measured 0.6 us per launch; with a division per entry the extra
          // registers spill, so the other instantiations read the tile row
          // by row and release it at the end)
          float4 lp[2];
          if (kUnitT) {
            const bool last = !(i0 + 2 < kMaxRows && b0 + 2 * kComputeWarps < a.B);
            lp[0] = *reinterpret_cast<const float4*>(tile + b0 * kTileV + 4 * lane);
            lp[1] = *reinterpret_cast<const float4*>(
                tile + (has1 ? b0 + kComputeWarps : b0) * kTileV + 4 * lane);
            if (last) {
              mbar_arrive(&tile_free[buf]);
              released = true;
            }
          }
          // the noise of two rows first: two independent Philox chains the
          // scheduler interleaves (a row step is latency-bound; four chains
          // spill at this kernel's 64 registers)
          uint4 wn[2];
          wn[0] = row_noise(rows[b0], v);
          wn[1] = row_noise(rows[has1 ? b0 + kComputeWarps : b0], v);
#pragma unroll
          for (int i = i0; i < i0 + 2 && i < kMaxRows; ++i) {
            const int b = cw + kComputeWarps * i;
            if (b >= a.B) break;
            const uint4 w = wn[i - i0];
            const float4 l4 =
                kUnitT ? lp[i - i0]
                       : *reinterpret_cast<const float4*>(tile + b * kTileV + 4 * lane);
            float sv[4];
            if (!kRowT) {
              scaled4<kUnitT>(l4, T, sv);
            } else {
              const float Tb = rows[b].T;
              if (Tb == 1.0f)
                scaled4<true>(l4, Tb, sv);
              else
                scaled4<false>(l4, Tb, sv);
            }
            const uint32_t h = (uint32_t)(__shfl_sync(0xffffffffu, hint_in, i) >> 32);
            const float4 q = rstate[i];
            RowState st{sums[i], q.x, q.y, q.z, __float_as_int(q.w)};  // ref, sref, h, idx
            if ((greedy_mask >> i) & 1u) {
              greedy_step(sv, v, st);
            } else {
              adopt_hint(st, h);
              // first tile: bootstrap the reference; afterwards the steady
              // state (which also handles a reference still at -inf)
              if (t == 0 && st.ref == -INFINITY)
                st = sampled_first_call(w, make_float4(sv[0], sv[1], sv[2], sv[3]), v, st);
              else
                sampled_step<kUnitT>(w, sv, v, st);
            }
            sums[i] = st.sum;
            rstate[i] = make_float4(st.ref, st.sref, st.h, __int_as_float(st.idx));
          }
        }
        // post this CTA's own winners whose keys beat the key read for
        // this tile (the one that ends the grid highest is the position's
        // winner)
        __syncwarp();
        unsigned long long mine = 0;
        if (lane < kMaxRows) {
          const float4 q = rstate[lane];
          if (__float_as_int(q.w) != kNoIndex)
            mine = decision_key(q.x, __float_as_int(q.w));
        }
        if (hint_ptr && mine > hint_in) atomicMax(hint_ptr, mine);
      }
      if (!released) mbar_arrive(&tile_free[buf]);
    }
    // chunk statistics: best score and index (already warp-wide), the
    // lanes' sums (same reference) added by a butterfly
#pragma unroll
    for (int i = 0; i < kMaxRows; ++i) {
      const int b = cw + kComputeWarps * i;
      if (b >= a.B) break;
      float sum = sums[i];
      const float4 q = rstate[i];
#pragma unroll
      for (int mask = 16; mask > 0; mask >>= 1)
        sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, mask));
      if (lane == 0) {
        ChunkStat cs;
        cs.idx = __float_as_int(q.w);
        cs.best = cs.idx == kNoIndex ? -INFINITY : q.x;  // this CTA's own winner
        cs.m = q.y;  // the reference of the sum (-inf: none set)
        cs.s = sum;
        *stat_slot(a.stats, P.k & 1, a.B, b, chunk) = cs;
      }
    }
    // the next position first gathers U[d_k]: bring the rows of this CTA's
    // own winners into L2 (the position's winner is one of them)
    if (P.k + 1 < a.K) {
      const int row_bytes = a.r * 2;  // bf16 U
#pragma unroll
      for (int i = 0; i < kMaxRows; ++i) {
        const int b = cw + kComputeWarps * i;
        if (b >= a.B) break;
        const int idx = __float_as_int(rstate[i].w);
        if (idx != kNoIndex && lane * 128 < row_bytes)
          prefetch_l2(static_cast<const char*>(a.U) + (size_t)idx * row_bytes + lane * 128);
      }
    }
    }
  }

  // ---------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  if (warp == 0 && *abort_flag) {
    // after an abort, loads may have been issued that no consumer waited
    // for: let each barrier's last issued load land (bounded) before the
    // CTA's shared memory is released
    if (lane == 0) {
      for (int s = 0; s < S && s < wb_issued; ++s) {
        const int last = wb_issued - 1 - ((wb_issued - 1 - s) % S);
        mbar_wait(&full[s], (uint32_t)(last / S) & 1u, kSpin >> 4);
      }
    } else if (lane == 1 && base_issued > 0) {
      if (kStaged && P.stage_bufs == 1) {  // its last load is the latest phase
        mbar_wait(&base_full[0], (uint32_t)(base_issued - 1) & 1u, kSpin >> 4);
      } else {  // the last load of each of the two tile or staging buffers
        for (int t = base_issued - 2 < 0 ? 0 : base_issued - 2; t < base_issued; ++t)
          mbar_wait(&base_full[t & 1], (uint32_t)(t >> 1) & 1u, kSpin >> 4);
      }
    }
  }
}

// ------------------------------------------------------------ host side
// DSPARK_TEST_STALL_WAIT=1 (tests of the failure path only): once u is
// ready, the MMA issuer waits for the u barrier's second phase, which
// nothing completes, with a short poll limit, so that the wait runs out,
// the kernel records kDevErrTimeout and takes its abort path.  That wait
// guards no copy.
bool stall_first_wait_requested() {
  const char* env = std::getenv("DSPARK_TEST_STALL_WAIT");
  return env != nullptr && env[0] == '1';
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

struct Layout {
  int bpad, stages, stage_bufs;
  uint32_t u_off, tile_off, stage_off, rows_off, rstate_off, bar_off;
  size_t smem;
};

// Shared memory: the Wb ring, u, two float32 tile buffers [bpad][128], one
// or two bf16 staging tiles when the drafter logits are bf16, row info,
// barriers.  Two staging tiles let the load of tile t+1's drafter logits
// overlap the drain of tile t (a single one serialises them: measured
// 336.9 -> 321.7 us per B=44 block); they are used while the Wb ring keeps
// at least one tile of r = 256 (four stages), else one.
Layout make_layout(int B, int r, int base_elt) {
  Layout L;
  L.bpad = (B + 15) / 16 * 16;
  // u: whole r-chunks of 64 (128-byte swizzled rows)
  const size_t u = (size_t)L.bpad * ((r + kKChunk - 1) / kKChunk * kKChunk) * 2;
  const size_t tiles = 2 * (size_t)L.bpad * kTileV * 4;
  const size_t rows = align_up((size_t)L.bpad * sizeof(RowConst), 16);
  const size_t rstate = (size_t)kComputeWarps * kMaxRows * 16;
  const size_t bars = (2 * kMaxStages + 14) * 8 + 16;
  size_t stage = 0;
  for (int nsb = base_elt == 2 ? 2 : 0; nsb >= 0; --nsb) {
    stage = (size_t)nsb * L.bpad * kTileV * 2;
    L.stage_bufs = nsb;
    const size_t fixed = u + tiles + stage + rows + rstate + bars + 1024;
    L.stages = fixed < kSmemLimit ? (int)((kSmemLimit - fixed) / kStageBytes) : 0;
    if (L.stages > kMaxStages) L.stages = kMaxStages;
    if (nsb <= 1 || L.stages >= 4) break;
  }
  L.u_off = (uint32_t)((size_t)L.stages * kStageBytes);
  L.tile_off = (uint32_t)(L.u_off + u);
  L.stage_off = (uint32_t)(L.tile_off + tiles);
  L.rows_off = (uint32_t)(L.stage_off + stage);
  L.rstate_off = (uint32_t)(L.rows_off + rows);
  L.bar_off = (uint32_t)(L.rstate_off + rstate);
  L.smem = L.bar_off + bars + 1024;
  return L;
}

// A [rows, V] view of one position of a [B, K, V] tensor: dims {V, B},
// row stride K*V elements, box {128, bpad}, no swizzle.
CUresult encode_position_map(CUtensorMap* map, CUtensorMapDataType dt,
                             const void* base, int elt, int B, int K, int V,
                             int k, int bpad) {
  const cuuint64_t dims[2] = {(cuuint64_t)V, (cuuint64_t)B};
  const cuuint64_t strides[1] = {(cuuint64_t)K * V * elt};
  const cuuint32_t box[2] = {(cuuint32_t)kTileV, (cuuint32_t)bpad};
  const cuuint32_t estr[2] = {1, 1};
  void* addr = const_cast<char*>(static_cast<const char*>(base)) +
               (size_t)k * V * elt;
  return encode_fn()(map, dt, 2, addr, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// Positions after the first are launched with programmatic stream
// serialisation behind the previous position's pick kernel: their set-up
// and first Wb / drafter-logit loads overlap the end of the previous
// position; they wait for its token before the gather.
template <typename BT, bool kUnitT, bool kRowT>
cudaError_t launch_typed(const CUtensorMap& wb, const CUtensorMap& bm,
                         const CUtensorMap& om, const TcParams& P, size_t smem,
                         int n_chunks, bool overlap_previous,
                         cudaStream_t stream) {
  auto kern = position_tc_kernel<BT, kUnitT, kRowT>;
  cudaError_t err = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)n_chunks, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_previous ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, wb, bm, om, P);
}

}  // namespace

// Request groups of a block on the tensor-core kernel: one launch per
// position takes at most kMaxBpad requests, so a larger block runs as
// ceil(B / kMaxBpad) groups of near-equal size (each reads Wb once per
// position).
int position_tc_groups(int B) {
  return B <= kMaxBpad ? 1 : (B + kMaxBpad - 1) / kMaxBpad;
}

bool position_tc_supported(const DraftArgs& a) {
  const int elt = a.base_dtype == DSPARK_F32 ? 4 : 2;
  const int n = position_tc_groups(a.B);
  const int per_group = (a.B + n - 1) / n;
  return a.w_dtype == DSPARK_BF16 && a.r % 16 == 0 && a.r <= 256 &&
         a.V % 8 == 0 && per_group <= kMaxBpad &&
         make_layout(per_group, a.r, elt).stages >= kMinStages &&
         encode_fn() != nullptr;
}

// CTAs of the tensor-core kernel: one per SM, at most one per vocab tile.
int position_tc_chunks(int V, int sm_count) {
  const int tiles = (V + kTileV - 1) / kTileV;
  int n = tiles < sm_count ? tiles : sm_count;
  return n < kMaxChunks ? n : kMaxChunks;
}

cudaError_t launch_position_tc(const DraftArgs& a, int k, int n_chunks,
                               cudaStream_t stream) {
  if (!encode_fn()) return cudaErrorNotSupported;
  if (a.B > kMaxBpad) return cudaErrorInvalidValue;  // a request group at most
  const int elt = a.base_dtype == DSPARK_F32 ? 4 : 2;
  const Layout L = make_layout(a.B, a.r, elt);
  CUtensorMap wb, bm, om;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)a.V, (cuuint64_t)a.r};
    const cuuint64_t strides[1] = {(cuuint64_t)a.V * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kKChunk};
    const cuuint32_t estr[2] = {1, 1};
    if (encode_fn()(&wb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    const_cast<void*>(a.Wb), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (encode_position_map(&bm,
                          elt == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          a.base, elt, a.B, a.K, a.V, k, L.bpad) != CUDA_SUCCESS ||
      encode_position_map(&om, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.logits, 4,
                          a.B, a.K, a.V, k, L.bpad) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  TcParams P;
  P.a = a;
  P.k = k;
  P.bpad = L.bpad;
  P.stages = L.stages;
  P.stage_bufs = L.stage_bufs;
  P.stall_first_wait = stall_first_wait_requested() ? 1 : 0;
  P.tiles_total = (a.V + kTileV - 1) / kTileV;
  P.n_chunks = n_chunks;
  P.u_off = L.u_off;
  P.tile_off = L.tile_off;
  P.stage_off = L.stage_off;
  P.rows_off = L.rows_off;
  P.rstate_off = L.rstate_off;
  P.bar_off = L.bar_off;
  const bool unit = a.T == 1.0f;
  const bool pdl = k > 0;
  if (a.temperature != nullptr)
    return elt == 4
               ? launch_typed<float, false, true>(wb, bm, om, P, L.smem, n_chunks, pdl, stream)
               : launch_typed<uint16_t, false, true>(wb, bm, om, P, L.smem, n_chunks, pdl,
                                                     stream);
  if (elt == 4)
    return unit ? launch_typed<float, true, false>(wb, bm, om, P, L.smem, n_chunks, pdl, stream)
                : launch_typed<float, false, false>(wb, bm, om, P, L.smem, n_chunks, pdl, stream);
  return unit ? launch_typed<uint16_t, true, false>(wb, bm, om, P, L.smem, n_chunks, pdl, stream)
              : launch_typed<uint16_t, false, false>(wb, bm, om, P, L.smem, n_chunks, pdl,
                                                     stream);
}

}  // namespace dspark
