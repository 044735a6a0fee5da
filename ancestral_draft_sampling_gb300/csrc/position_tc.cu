// position_tc.cu -- one draft position with the Markov bias on the 5th-gen
// tensor cores (tcgen05), for bfloat16 heads.
//
// brb-nv/TensorRT-LLM PR #27, "2. One fused kernel per draft position":
// bias(d_{k-1}) = U[d_{k-1}] @ Wb, added to the drafter logits, scaled by
// 1/T, Gumbel-max with Philox noise, float32 biased logits and per-chunk
// softmax statistics out.  The pages keep the bias GEMM on cuBLAS; here it
// is fused into the position kernel.
//
// Per CTA (one per SM, a contiguous range of 128-wide vocab tiles):
//   warp 0      TMA producer: Wb[r0:r0+64, v0:v0+128] stages (two 64x64
//               boxes, 128-byte swizzle) into a ring of shared-memory stages.
//   warp 1      MMA issuer: D[v, b] = sum_j Wb[j, v] * u[b, j] with
//               tcgen05.mma kind::f16 (M = 128 vocab rows, N = B rounded up
//               to 16, K = r), accumulating in one of two TMEM buffers.
//               A (Wb tile) is vocab-major, B (u) is r-major.
//   warps 2..9  compute.  Warps 2..5 (one per TMEM lane quarter) drain the
//               finished accumulator into a [b][128] float32 shared tile;
//               then all eight take requests b = w, w+8, ... with lane l on
//               vocab entries 4l..4l+3 (one Philox block), add the drafter
//               logits, write the float32 biased logits, scale, perturb and
//               fold into per-lane running statistics, reduced per warp at
//               the end of the chunk.
// Every mbarrier wait is bounded; on a timeout the kernel records an error
// in the workspace control word, stops issuing work, waits (bounded) for
// its in-flight MMAs, frees its TMEM and returns.
#include <cudaTypedefs.h>

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
constexpr int kComputeWarps = 16;
constexpr int kThreads = 32 * (2 + kComputeWarps);
constexpr int kComputeThreads = 32 * kComputeWarps;
constexpr int kMaxBpad = 128;
constexpr int kMaxRowsPerWarp = kMaxBpad / kComputeWarps;
constexpr uint32_t kTmemCols = 256;                // two accumulators
constexpr uint32_t kAccCols = 128;
constexpr uint32_t kSpin = 1u << 22;
constexpr int kMaxStages = 8;
constexpr size_t kSmemLimit = 232448;              // 227 KB per CTA
constexpr float kLog2e = 1.4426950408889634f;

struct RowInfo {
  uint64_t seed;
  uint64_t offset;
  int pad;
  int greedy;
};

struct TcParams {
  DraftArgs a;
  int k;
  int bpad;
  int stages;
  int nbuf;  // bias tiles in shared memory (2: drain of t+1 overlaps t)
  int tiles_total;
  int n_chunks;
  uint32_t u_off, bias_off, rows_off, bar_off;
};

// Running state of one (lane, request) over the lane's vocab entries:
//   m    max of the scaled logits s seen (-inf if none);
//   sum  sum of exp(s - m);
//   key  the best candidate so far, relative to m: exp(s - m) / E for a
//        sampled request (exponential race: the largest exp(s) / E is the
//        largest s - log E = s + g), s itself for a greedy request;
//   idx  its vocab index (kNoIndex while nothing has won).
struct LaneStat {
  float m, sum, key;
  int idx;
};

__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float scale(float l, float T) {
  return T == 1.0f ? l : __fdiv_rn(l, T);
}

// Folds the four candidates v..v+3 (s[e] = -inf past V) into st.  E is the
// exponential variate of each candidate (unused for greedy requests).
template <bool kGreedy>
__device__ __forceinline__ void fold4(LaneStat& st, const float s[4],
                                      const float E[4], int v) {
  const float m4 = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
  const float mn = fmaxf(st.m, m4);
  if (mn > st.m) {  // a new running max: rescale what is kept relative to m
    const float f = ex2_approx((st.m - mn) * kLog2e);
    st.sum *= f;
    if (!kGreedy) st.key *= f;
    st.m = mn;
  }
  if (mn != -INFINITY) {
    const float nml = -mn * kLog2e;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float ee = ex2_approx(fmaf(s[e], kLog2e, nml));
      st.sum += ee;
      const float key = kGreedy ? s[e] : __fdividef(ee, E[e]);
      const bool win = key > st.key;  // strict: the lower index keeps a tie
      st.key = win ? key : st.key;
      st.idx = win ? v + e : st.idx;
    }
  } else if (isnan(s[0]) || isnan(s[1]) || isnan(s[2]) || isnan(s[3])) {
    st.sum = __int_as_float(0x7fc00000);
  }
}

// One request's four vocab entries v..v+3 of the tile: biased logits (written
// when `store`), scaled logits, noise, and the fold into the lane state.
__device__ __forceinline__ void process_row(const RowInfo& ri, size_t row,
                                            const float4 bias, const float x[4],
                                            bool valid, bool store, int v,
                                            LaneStat& st, const DraftArgs& a,
                                            int k, float T) {
  float l[4], s[4];
  l[0] = ri.pad ? bias.x : __fadd_rn(x[0], bias.x);
  l[1] = ri.pad ? bias.y : __fadd_rn(x[1], bias.y);
  l[2] = ri.pad ? bias.z : __fadd_rn(x[2], bias.z);
  l[3] = ri.pad ? bias.w : __fadd_rn(x[3], bias.w);
  if (valid && store)
    __stcs(reinterpret_cast<float4*>(a.logits + row * a.V + v),
           make_float4(l[0], l[1], l[2], l[3]));
#pragma unroll
  for (int e = 0; e < 4; ++e) s[e] = valid ? scale(l[e], T) : -INFINITY;
  if (ri.greedy) {
    const float E[4] = {1.0f, 1.0f, 1.0f, 1.0f};
    fold4<true>(st, s, E, v);
  } else {
    const uint4 w = noise_block(ri.seed, ri.offset, k, kNoiseDraft,
                                (uint32_t)v >> 2);
    float E[4];
    E[0] = exponential_from_word(w.x);
    E[1] = exponential_from_word(w.y);
    E[2] = exponential_from_word(w.z);
    E[3] = exponential_from_word(w.w);
    fold4<false>(st, s, E, v);
  }
}

template <typename BT>
__device__ __forceinline__ void load_base4(const BT* p, float out[4]) {
  if constexpr (sizeof(BT) == 4) {
    const float4 x = __ldcs(reinterpret_cast<const float4*>(p));
    out[0] = x.x; out[1] = x.y; out[2] = x.z; out[3] = x.w;
  } else {
    const uint2 x = __ldcs(reinterpret_cast<const uint2*>(p));
    out[0] = __uint_as_float(x.x << 16);
    out[1] = __uint_as_float(x.x & 0xffff0000u);
    out[2] = __uint_as_float(x.y << 16);
    out[3] = __uint_as_float(x.y & 0xffff0000u);
  }
}

template <int kN>
__device__ __forceinline__ void tmem_ld4x(uint32_t taddr, float (&v)[4 * kN],
                                          int n_valid) {
#pragma unroll
  for (int i = 0; i < kN; ++i) {
    if (i < n_valid) {
      uint32_t r0, r1, r2, r3;
      asm volatile(
          "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
          : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
          : "r"(taddr + 4u * i)
          : "memory");
      v[4 * i] = __uint_as_float(r0);
      v[4 * i + 1] = __uint_as_float(r1);
      v[4 * i + 2] = __uint_as_float(r2);
      v[4 * i + 3] = __uint_as_float(r3);
    }
  }
}

template <typename BT>
__global__ void __launch_bounds__(kThreads, 1)
position_tc_kernel(const __grid_constant__ CUtensorMap wb_map,
                   const __grid_constant__ TcParams P) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* ring = smem;
  uint8_t* u_s = smem + P.u_off;
  float* bias_s = reinterpret_cast<float*>(smem + P.bias_off);
  RowInfo* rows = reinterpret_cast<RowInfo*>(smem + P.rows_off);
  const int S = P.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + P.bar_off);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* mma_done = acc_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const DraftArgs& a = P.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x;
  const int t_begin = (int)((long long)chunk * P.tiles_total / P.n_chunks);
  const int t_end = (int)((long long)(chunk + 1) * P.tiles_total / P.n_chunks);
  const int n_tiles = t_end - t_begin;
  const int kchunks = a.r / kKChunk;

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
      mbar_init(&acc_empty[i], kComputeThreads);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) prefetch_tmap(&wb_map);
  if (warp == 1) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  if (warp >= 2) {
    // u_b = U[d_{k-1}(b)], stored r-major with the 128-byte swizzle: row n of
    // r-chunk c at c*(bpad*128) + n*128, 16-byte piece p at (p ^ (n & 7)).
    const int ct = threadIdx.x - 64;
    const int pieces = a.r / 8;
    const uint16_t* U = static_cast<const uint16_t*>(a.U);
    for (int i = ct; i < P.bpad * pieces; i += kComputeThreads) {
      const int n = i / pieces, piece = i - n * pieces;
      const int c = piece >> 3, p = piece & 7;
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      if (n < a.B) {
        int prev = (P.k == 0) ? a.d0[n] : a.tokens[(size_t)n * a.K + (P.k - 1)];
        if ((unsigned)prev >= (unsigned)a.V) {
          if (piece == 0) a.control[0] = kDevErrBadToken;
          prev = 0;
        }
        val = __ldg(reinterpret_cast<const uint4*>(U + (size_t)prev * a.r) + piece);
      }
      *reinterpret_cast<uint4*>(u_s + (size_t)c * (P.bpad * 128) + n * 128 +
                                ((p ^ (n & 7)) << 4)) = val;
    }
    for (int n = ct; n < P.bpad; n += kComputeThreads) {
      RowInfo ri;
      if (n < a.B) {
        ri.seed = a.seed[n];
        ri.offset = a.offset[n];
        ri.pad = a.pad_row != nullptr && a.pad_row[n] != 0;
        ri.greedy = a.greedy != nullptr && a.greedy[n] != 0;
      } else {
        ri.seed = ri.offset = 0;
        ri.pad = ri.greedy = 0;
      }
      rows[n] = ri;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int g = 0;
      for (int t = 0; t < n_tiles && !*abort_flag; ++t) {
        const int v0 = (t_begin + t) * kTileV;
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
      // every issued load lands before the CTA may exit: wait for the last
      // phase of each stage that was used (bounded; only matters on abort)
      if (*abort_flag) {
        for (int s = 0; s < S && s < g; ++s) {
          const int last = g - 1 - ((g - 1 - s) % S);
          mbar_wait(&full[s], (uint32_t)(last / S) & 1u, kSpin >> 4);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kTileV, (uint32_t)P.bpad, 1u, 0u);
      const uint32_t u_base = smem_u32(u_s);
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
    const int cw = warp - 2;
    const int quarter = warp & 3;        // TMEM lanes this warp may access
    const int col_group = cw >> 2;       // which quarter of the columns
    const int cols = P.bpad / 4;         // columns drained by this warp
    const int col0 = col_group * cols;
    const BT* base = static_cast<const BT*>(a.base);
    const float T = a.T;
    const int V = a.V;
    LaneStat st[kMaxRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kMaxRowsPerWarp; ++i) {
      st[i].m = -INFINITY;
      st[i].sum = 0.0f;
      st[i].key = 0.0f;
      st[i].idx = kNoIndex;
    }
#pragma unroll
    for (int i = 0; i < kMaxRowsPerWarp; ++i) {
      const int b = cw + kComputeWarps * i;
      if (b < a.B && rows[b].greedy) st[i].key = -INFINITY;
    }

    for (int t = 0; t < n_tiles; ++t) {
      const int acc = t & 1;
      const uint32_t aph = (uint32_t)(t >> 1) & 1u;
      float* bias_t = bias_s + (P.nbuf == 2 ? acc : 0) * (P.bpad * kTileV);
      // drain: lanes quarter*32.., columns col0..col0+cols of the accumulator
      bool ok = !*abort_flag && mbar_wait(&acc_full[acc], aph, kSpin);
      ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld needs the whole warp
      if (ok) {
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) +
                               (uint32_t)acc * kAccCols + (uint32_t)col0;
        float vals[kMaxBpad / 4];
        tmem_ld4x<kMaxBpad / 16>(taddr, vals, cols / 4);
        tmem_ld_wait();
        const int m = quarter * 32 + lane;
#pragma unroll
        for (int i = 0; i < kMaxBpad / 4; ++i)
          if (i < cols) bias_t[(col0 + i) * kTileV + m] = vals[i];
        tc_fence_before();
      } else if (!*abort_flag) {
        fail(kDevErrTimeout);
      }
      mbar_arrive(&acc_empty[acc]);
      // bias tile complete (and, with two tiles, the other one is free again:
      // every warp finished computing on it before arriving here)
      named_sync(1, kComputeThreads);
      if (!*abort_flag) {
        const int v = (t_begin + t) * kTileV + 4 * lane;
        const bool valid = v < V;  // V % 8 == 0: v..v+3 all in range
#pragma unroll
        for (int i = 0; i < kMaxRowsPerWarp; ++i) {
          const int b = cw + kComputeWarps * i;
          if (b >= a.B) break;
          const RowInfo ri = rows[b];
          const float4 bias =
              *reinterpret_cast<const float4*>(bias_t + b * kTileV + 4 * lane);
          const size_t row = (size_t)b * a.K + P.k;
          float x[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          if (!ri.pad && valid) load_base4<BT>(base + row * V + v, x);
          process_row(ri, row, bias, x, valid, true, v, st[i], a, P.k, T);
        }
      }
      if (P.nbuf == 1) named_sync(2, kComputeThreads);  // bias tile consumed
    }
    // chunk statistics: the lane winner's log-domain score s + g, then a
    // butterfly over the warp
#pragma unroll
    for (int i = 0; i < kMaxRowsPerWarp; ++i) {
      const int b = cw + kComputeWarps * i;
      if (b >= a.B) break;
      const RowInfo ri = rows[b];
      ChunkStat cs;
      cs.idx = st[i].idx;
      cs.m = st[i].m;
      cs.s = st[i].sum;
      cs.best = -INFINITY;
      if (cs.idx != kNoIndex) {
        if (ri.greedy) {
          cs.best = st[i].key;
        } else {
          const size_t row = (size_t)b * a.K + P.k;
          const float s_best = scale(a.logits[row * V + cs.idx], T);
          const uint4 w = noise_block(ri.seed, ri.offset, P.k, kNoiseDraft,
                                      (uint32_t)cs.idx >> 2);
          cs.best = __fadd_rn(
              s_best, -logf(exponential_from_word(word_of(w, cs.idx & 3))));
        }
      }
      const ChunkStat red = warp_reduce_stat(cs);
      if (lane == 0) a.stats[(size_t)b * kMaxChunks + chunk] = red;
    }
  }

  // ---------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------ host side
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
  int bpad, stages, nbuf;
  uint32_t u_off, bias_off, rows_off, bar_off;
  size_t smem;
};

// Shared memory: the Wb ring, u, one or two bias tiles, row info, barriers.
// Two bias tiles are used when at least four ring stages still fit.
Layout make_layout(int B, int r) {
  Layout L;
  L.bpad = (B + 15) / 16 * 16;
  const size_t u = (size_t)L.bpad * r * 2;
  const size_t bias = (size_t)L.bpad * kTileV * 4;
  const size_t rows = align_up((size_t)L.bpad * sizeof(RowInfo), 16);
  const size_t bars_max = (2 * kMaxStages + 5) * 8 + 16;
  for (L.nbuf = 2; L.nbuf >= 1; --L.nbuf) {
    const size_t fixed = u + L.nbuf * bias + rows + bars_max + 1024;
    L.stages = fixed < kSmemLimit ? (int)((kSmemLimit - fixed) / kStageBytes) : 0;
    if (L.stages > kMaxStages) L.stages = kMaxStages;
    if (L.stages >= 4 || L.nbuf == 1) break;
  }
  L.u_off = (uint32_t)((size_t)L.stages * kStageBytes);
  L.bias_off = (uint32_t)(L.u_off + u);
  L.rows_off = (uint32_t)(L.bias_off + L.nbuf * bias);
  L.bar_off = (uint32_t)(L.rows_off + rows);
  L.smem = L.bar_off + (2 * L.stages + 5) * 8 + 16 + 1024;
  return L;
}

}  // namespace

bool position_tc_supported(const DraftArgs& a) {
  return a.w_dtype == DSPARK_BF16 && a.r % kKChunk == 0 && a.r <= 256 &&
         a.V % 8 == 0 && a.B <= kMaxBpad && make_layout(a.B, a.r).stages >= 2 &&
         encode_fn() != nullptr;
}

int position_tc_chunks(int V, int sm_count) {
  const int tiles = (V + kTileV - 1) / kTileV;
  return tiles < sm_count ? tiles : sm_count;
}

cudaError_t launch_position_tc(const DraftArgs& a, int k, int n_chunks,
                               cudaStream_t stream) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)a.V, (cuuint64_t)a.r};
  const cuuint64_t strides[1] = {(cuuint64_t)a.V * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)kKChunk};
  const cuuint32_t estr[2] = {1, 1};
  CUresult cr = encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                       const_cast<void*>(a.Wb), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE,
                       CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
  const Layout L = make_layout(a.B, a.r);
  TcParams P;
  P.a = a;
  P.k = k;
  P.bpad = L.bpad;
  P.stages = L.stages;
  P.nbuf = L.nbuf;
  P.tiles_total = (a.V + kTileV - 1) / kTileV;
  P.n_chunks = n_chunks;
  P.u_off = L.u_off;
  P.bias_off = L.bias_off;
  P.rows_off = L.rows_off;
  P.bar_off = L.bar_off;
  auto kern = a.base_dtype == DSPARK_F32 ? position_tc_kernel<float>
                                         : position_tc_kernel<uint16_t>;
  cudaError_t err = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.smem);
  if (err != cudaSuccess) return err;
  kern<<<n_chunks, kThreads, L.smem, stream>>>(map, P);
  return cudaGetLastError();
}

}  // namespace dspark
