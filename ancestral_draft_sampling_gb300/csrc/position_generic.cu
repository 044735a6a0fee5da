// position_generic.cu -- one draft position, CUDA-core (FFMA) bias.
//
// brb-nv/TensorRT-LLM PR #27, "2. One fused kernel per draft position": add
// the Markov bias U[d_{k-1}] @ Wb to the drafter logits, scale by 1/T, take
// the Gumbel-max with Philox noise, write the float32 biased logits and the
// per-chunk softmax statistics.
//
// This kernel serves float32 heads (where a tensor-core contraction would
// not hold float32 accuracy) and any shape the tensor-core kernel does not
// take.  Grid: (vocab chunks, batch groups of up to kGroup requests); each
// CTA walks its chunk in 128-wide vocab tiles.  Warp w owns the requests
// w, w+8, ... of the group; lane l owns the four consecutive vocab entries
// 4l..4l+3 of the tile, which are exactly the four words of one Philox
// block.  The draw and the sum-exp are the warp draw of gumbel_draw.cuh
// (a reference shared by the warp, a conservative candidate test, exact
// scores for the admitted entries only), with each request's folded Philox
// constants in shared memory.  Against an exact score for every entry (two
// logarithms and a full Philox block each) it took B=88, K=7, V=200064
// blocks with f32 heads from 1344 to 1058 us at r = 16, 1733 to 1427 us at
// r = 64 and 4358 to 4092 us at r = 256 (where the FFMA contraction
// dominates).
#include "dspark_common.cuh"
#include "gumbel_draw.cuh"

namespace dspark {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTileV = 128;
constexpr int kGroup = 64;                 // requests per CTA
constexpr int kRowsPerWarp = kGroup / kWarps;  // 8
constexpr int kRowsPerPass = 4;            // rows sharing one sweep over Wb

template <typename WT>
__device__ __forceinline__ float4 load_w4(const WT* p);

template <>
__device__ __forceinline__ float4 load_w4<float>(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}

template <>
__device__ __forceinline__ float4 load_w4<uint16_t>(const uint16_t* p) {
  const uint2 raw = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(raw.x << 16),
                     __uint_as_float(raw.x & 0xffff0000u),
                     __uint_as_float(raw.y << 16),
                     __uint_as_float(raw.y & 0xffff0000u));
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<uint16_t>(uint16_t x) {
  return bf16_bits_to_float(x);
}

// Loads base[row, v..v+3] (any of them past V read as 0).
template <typename BT, bool kVec>
__device__ __forceinline__ void load_base4(const BT* row, int v, int V,
                                           float out[4]) {
  if (kVec && v + 3 < V) {
    if constexpr (sizeof(BT) == 4) {
      const float4 x = __ldcs(reinterpret_cast<const float4*>(row + v));
      out[0] = x.x; out[1] = x.y; out[2] = x.z; out[3] = x.w;
    } else {
      const uint2 x = __ldcs(reinterpret_cast<const uint2*>(row + v));
      out[0] = __uint_as_float(x.x << 16);
      out[1] = __uint_as_float(x.x & 0xffff0000u);
      out[2] = __uint_as_float(x.y << 16);
      out[3] = __uint_as_float(x.y & 0xffff0000u);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) out[e] = (v + e < V) ? to_f32<BT>(row[v + e]) : 0.0f;
  }
}

template <bool kVec>
__device__ __forceinline__ void store_logits4(float* row, int v, int V,
                                              const float l[4]) {
  if (kVec && v + 3 < V) {
    __stcs(reinterpret_cast<float4*>(row + v), make_float4(l[0], l[1], l[2], l[3]));
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (v + e < V) row[v + e] = l[e];
  }
}

// A request's folded Philox constants (philox_fold), its flags and its
// temperature, read once per CTA.
struct alignas(16) RowNoise {
  uint4 pre;
  uint4 rk[4];
  uint32_t pad;     // a padding row: l = bias
  uint32_t greedy;  // a greedy request
  float T;
  uint32_t unused;
};

// kMinBlocks: 2 where the shared memory lets two CTAs share an SM (the
// registers are then held to 128), else 1.  With the drafter logits of a
// pass loaded before its contraction, B=88, K=7, V=200064 blocks with f32
// heads took 1058 -> 898 us at r = 16, 1429 -> 1303 us at r = 64 and
// 4102 -> 3827 us at r = 256 (one CTA per SM by shared memory; 4171 us
// with the two-CTA bound there).  The small first configuration (f32 head)
// went from 33.5 to 36.8 us.
template <typename WT, typename BT, bool kVec, int kMinBlocks>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
position_generic_kernel(DraftArgs a, int k, int tiles_per_chunk) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int r = a.r, V = a.V, B = a.B, K = a.K;
  float* u_s = reinterpret_cast<float*>(smem_raw);             // [kGroup][r]
  WT* w_s = reinterpret_cast<WT*>(u_s + (size_t)kGroup * r);   // [r][kTileV]
  // [kGroup]: each request's folded Philox constants (noise stream 0 at
  // position k)
  RowNoise* noise_s = reinterpret_cast<RowNoise*>(w_s + (size_t)r * kTileV);

  const int chunk = blockIdx.x;
  const int g0 = blockIdx.y * kGroup;
  const int nb = min(kGroup, B - g0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WT* U = static_cast<const WT*>(a.U);
  const WT* Wb = static_cast<const WT*>(a.Wb);
  const BT* base = static_cast<const BT*>(a.base);

  // u_b = U[d_{k-1}(b)] for the group, as float32 (zero rows past B)
  for (int i = threadIdx.x; i < kGroup * r; i += kThreads) {
    const int bl = i / r, j = i - bl * r;
    float x = 0.0f;
    if (bl < nb) {
      const int b = g0 + bl;
      int prev = (k == 0) ? a.d0[b] : a.tokens[(size_t)b * K + (k - 1)];
      if ((unsigned)prev >= (unsigned)V) {  // caller's d0 out of range
        if (j == 0) a.control[0] = kDevErrBadToken;
        prev = 0;
      }
      x = to_f32<WT>(U[(size_t)prev * r + j]);
    }
    u_s[i] = x;
  }
  for (int bl = threadIdx.x; bl < nb; bl += kThreads) {
    const uint64_t sd = a.seed[g0 + bl], off = a.offset[g0 + bl];
    philox_fold(noise_s[bl].pre, noise_s[bl].rk, (uint32_t)sd, (uint32_t)(sd >> 32),
                (uint32_t)k | ((uint32_t)kNoiseDraft << 16), (uint32_t)off,
                (uint32_t)(off >> 32));
    noise_s[bl].pad = a.pad_row != nullptr && a.pad_row[g0 + bl] != 0;
    noise_s[bl].greedy = a.greedy != nullptr && a.greedy[g0 + bl] != 0;
    noise_s[bl].T = request_temperature(a, g0 + bl);
  }

  SampleState st[kRowsPerWarp];
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) st[i] = sample_state_init();

  const int n_tiles = (V + kTileV - 1) / kTileV;
  const int t_begin = chunk * tiles_per_chunk;
  const int t_end = min(n_tiles, t_begin + tiles_per_chunk);
  const bool w_vec = (V % (16 / (int)sizeof(WT))) == 0;

  for (int t = t_begin; t < t_end; ++t) {
    const int v0 = t * kTileV;
    __syncthreads();  // previous tile fully consumed (and u_s written)
    // Wb[:, v0 : v0+128] -> w_s, zero past V
    if (w_vec && v0 + kTileV <= V) {
      constexpr int kPer16 = 16 / sizeof(WT);
      for (int i = threadIdx.x; i < r * (kTileV / kPer16); i += kThreads) {
        const int j = i / (kTileV / kPer16), c = i - j * (kTileV / kPer16);
        reinterpret_cast<uint4*>(w_s + (size_t)j * kTileV)[c] =
            __ldg(reinterpret_cast<const uint4*>(Wb + (size_t)j * V + v0) + c);
      }
    } else {
      for (int i = threadIdx.x; i < r * kTileV; i += kThreads) {
        const int j = i / kTileV, c = i - j * kTileV;
        w_s[i] = (v0 + c < V) ? Wb[(size_t)j * V + v0 + c] : WT(0);
      }
    }
    __syncthreads();

    const int v = v0 + 4 * lane;
#pragma unroll
    for (int p = 0; p < kRowsPerWarp; p += kRowsPerPass) {
      if (warp + kWarps * p >= nb) break;
      // the pass's drafter logits first: their loads are in flight during
      // the contraction below
      float base4[kRowsPerPass][4];
#pragma unroll
      for (int q = 0; q < kRowsPerPass; ++q) {
        const int bl = warp + kWarps * (p + q);
#pragma unroll
        for (int e = 0; e < 4; ++e) base4[q][e] = 0.0f;
        if (bl < nb && !noise_s[bl].pad)
          load_base4<BT, kVec>(base + ((size_t)(g0 + bl) * K + k) * V, v0 + 4 * lane, V,
                               base4[q]);
      }
      float acc[kRowsPerPass][4];
#pragma unroll
      for (int q = 0; q < kRowsPerPass; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[q][e] = 0.0f;
      // bias = sum_j u_b[j] * Wb[j, v], j ascending, float32 FMA
      for (int j = 0; j < r; j += 4) {
        float4 u4[kRowsPerPass];
#pragma unroll
        for (int q = 0; q < kRowsPerPass; ++q)
          u4[q] = *reinterpret_cast<const float4*>(
              u_s + (size_t)(warp + kWarps * (p + q)) * r + j);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const float4 w = load_w4<WT>(w_s + (size_t)(j + jj) * kTileV + 4 * lane);
#pragma unroll
          for (int q = 0; q < kRowsPerPass; ++q) {
            const float u = jj == 0 ? u4[q].x : jj == 1 ? u4[q].y : jj == 2 ? u4[q].z : u4[q].w;
            acc[q][0] = fmaf(u, w.x, acc[q][0]);
            acc[q][1] = fmaf(u, w.y, acc[q][1]);
            acc[q][2] = fmaf(u, w.z, acc[q][2]);
            acc[q][3] = fmaf(u, w.w, acc[q][3]);
          }
        }
      }
      // epilogue: logits, scaled logits, noise, statistics
#pragma unroll
      for (int q = 0; q < kRowsPerPass; ++q) {
        const int bl = warp + kWarps * (p + q);
        if (bl >= nb) break;
        const int b = g0 + bl;
        const size_t row = (size_t)b * K + k;
        const bool pad = noise_s[bl].pad != 0;
        const bool greedy = noise_s[bl].greedy != 0;
        float l[4];
        const float T = noise_s[bl].T;
#pragma unroll
        for (int e = 0; e < 4; ++e) l[e] = pad ? acc[q][e] : __fadd_rn(base4[q][e], acc[q][e]);
        store_logits4<kVec>(a.logits + row * V, v, V, l);
        // entries past V take no part in the draw or the sum
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (v + e >= V) l[e] = -INFINITY;
        const uint4 w = greedy ? make_uint4(0u, 0u, 0u, 0u)
                               : philox_folded(noise_s[bl].pre, noise_s[bl].rk,
                                               (uint32_t)v >> 2);
        sample_block<false>(st[p + q], l, v >> 2, T, greedy, w);
      }
    }
  }

#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    const int bl = warp + kWarps * i;
    if (bl >= nb) break;
    ChunkStat cs;
    cs.best = st[i].ref;
    cs.idx = st[i].idx;
    cs.m = st[i].m;
    cs.s = st[i].sum;
    const ChunkStat red = warp_reduce_stat(cs);
    if (lane == 0) *stat_slot(a.stats, 0, a.B, g0 + bl, chunk) = red;
  }
}

template <typename WT, typename BT, bool kVec>
cudaError_t launch_typed(const DraftArgs& a, int k, int n_chunks,
                         cudaStream_t stream) {
  const size_t smem = (size_t)kGroup * a.r * sizeof(float) +
                      (size_t)a.r * kTileV * sizeof(WT) + kGroup * sizeof(RowNoise);
  // two CTAs per SM if their shared memory (and the 1 KB each reserves) fits
  const bool two = 2 * (smem + 1024) <= 228 * 1024;
  auto kern = two ? position_generic_kernel<WT, BT, kVec, 2>
                  : position_generic_kernel<WT, BT, kVec, 1>;
  cudaError_t err = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int n_tiles = (a.V + kTileV - 1) / kTileV;
  const int tiles_per_chunk = (n_tiles + n_chunks - 1) / n_chunks;
  const int used_chunks = (n_tiles + tiles_per_chunk - 1) / tiles_per_chunk;
  const dim3 grid(used_chunks, (a.B + kGroup - 1) / kGroup);
  kern<<<grid, kThreads, smem, stream>>>(a, k, tiles_per_chunk);
  return cudaGetLastError();
}

}  // namespace

// Number of chunks the generic kernel actually uses for n_chunks requested.
int generic_chunks_used(int V, int n_chunks) {
  const int n_tiles = (V + kTileV - 1) / kTileV;
  const int tiles_per_chunk = (n_tiles + n_chunks - 1) / n_chunks;
  return (n_tiles + tiles_per_chunk - 1) / tiles_per_chunk;
}

cudaError_t launch_position_generic(const DraftArgs& a, int k, int n_chunks,
                                    cudaStream_t stream) {
  const bool vec = (a.V % 4) == 0;
  const bool wf = a.w_dtype == DSPARK_F32, bf = a.base_dtype == DSPARK_F32;
  if (wf && bf) return vec ? launch_typed<float, float, true>(a, k, n_chunks, stream)
                           : launch_typed<float, float, false>(a, k, n_chunks, stream);
  if (wf && !bf) return vec ? launch_typed<float, uint16_t, true>(a, k, n_chunks, stream)
                            : launch_typed<float, uint16_t, false>(a, k, n_chunks, stream);
  if (!wf && bf) return vec ? launch_typed<uint16_t, float, true>(a, k, n_chunks, stream)
                            : launch_typed<uint16_t, float, false>(a, k, n_chunks, stream);
  return vec ? launch_typed<uint16_t, uint16_t, true>(a, k, n_chunks, stream)
             : launch_typed<uint16_t, uint16_t, false>(a, k, n_chunks, stream);
}

}  // namespace dspark
