// elementwise.cu -- the memory-bound steps of the path: tree combine of rank
// partials, RMSNorm, the logprob chunk tree + gather, MoE routing, permutation,
// gather and the routing-slot combine, plus the bounded-wait self test.  (SwiGLU
// runs in the epilogue of the gate/up GEMM.)
// Every reduction has a fixed shape that depends only on the problem's row
// length (H, k, C), never on the number of rows or on the launch geometry.
#include <cuda_bf16.h>

#include "iso_elementwise.h"
#include "iso_ptx.cuh"

namespace iso {

namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint16_t f2bf(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return static_cast<uint32_t>(f2bf(lo)) | (static_cast<uint32_t>(f2bf(hi)) << 16);
}

// Balanced binary tree over v[0..n) (n a power of two <= NMAX), left = lower index.
template <int NMAX>
__device__ __forceinline__ float tree_sum(float (&v)[NMAX], int n) {
#pragma unroll
  for (int w = 1; w < NMAX; w *= 2) {
#pragma unroll
    for (int p = 0; p + w < NMAX; p += 2 * w)
      if (p + w < n) v[p] = __fadd_rn(v[p], v[p + w]);
  }
  return v[0];
}

}  // namespace

// ----------------------------------------------------------------- tree combine
// C[i, j] = bf16_rn(tree_r S[r][i, j]); each thread owns 4 consecutive columns.
__global__ void tree_combine_kernel(const float* __restrict__ S, int64_t lds, int64_t rank_stride, int R,
                                    __nv_bfloat16* __restrict__ C, int64_t ldc, int M, int N) {
  grid_dependency_wait();  // launched as a dependent grid: the partials come from the grid before
  grid_launch_dependents();
  const int64_t nvec_row = N / 4;
  const int64_t total = static_cast<int64_t>(M) * nvec_row;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t i = idx / nvec_row;
    const int64_t j = (idx - i * nvec_row) * 4;
    float a[MAX_LEAVES], b[MAX_LEAVES], c[MAX_LEAVES], d[MAX_LEAVES];
#pragma unroll
    for (int r = 0; r < MAX_LEAVES; ++r) {
      if (r < R) {
        const float4 v = __ldcs(reinterpret_cast<const float4*>(S + r * rank_stride + i * lds + j));
        a[r] = v.x;
        b[r] = v.y;
        c[r] = v.z;
        d[r] = v.w;
      } else {
        a[r] = b[r] = c[r] = d[r] = 0.f;
      }
    }
    const float ra = tree_sum<MAX_LEAVES>(a, R), rb = tree_sum<MAX_LEAVES>(b, R), rc = tree_sum<MAX_LEAVES>(c, R),
                rd = tree_sum<MAX_LEAVES>(d, R);
    uint2 o = make_uint2(pack2(ra, rb), pack2(rc, rd));
    *reinterpret_cast<uint2*>(C + i * ldc + j) = o;
  }
}

// ---------------------------------------------------------------------- RMSNorm
// One warp per row.  Lane l owns the 8-element vectors v = l, l+32, l+64, ...
// and sums x^2 over them in ascending order (rn multiply, rn add); an xor
// shuffle tree 16,8,4,2,1 completes the row sum, identical in every lane.
// Two blocks (16 warps, 16 rows in flight) per SM for rows of up to 4096: with the compiler's
// free choice one 174-register block per SM kept too few bytes in flight for HBM (5.3 TB/s at
// T = 262144, H = 4096 on GB300; 6.1 TB/s with this bound, bitwise identical output).
template <int VPL>  // vectors per lane when H == 256*VPL (kept in registers); 0 = generic
__global__ void __launch_bounds__(256, (VPL > 0 && VPL <= 16) ? 2 : 1) rmsnorm_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ gamma,
                               float eps, __nv_bfloat16* __restrict__ y, int T, int H) {
  const int lane = threadIdx.x & 31;
  const int warps_per_block = blockDim.x >> 5;
  const int nvec = H / 8;
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * warps_per_block + (threadIdx.x >> 5); row < T;
       row += static_cast<int64_t>(gridDim.x) * warps_per_block) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * H);
    uint4* yr = reinterpret_cast<uint4*>(y + row * H);
    const uint4* gr = reinterpret_cast<const uint4*>(gamma);
    float acc = 0.f;
    if constexpr (VPL > 0) {
      uint4 v[VPL];
#pragma unroll
      for (int i = 0; i < VPL; ++i) v[i] = __ldcs(xr + lane + 32 * i);
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float a = bf16_lo(w[q]), b = bf16_hi(w[q]);
          acc = __fadd_rn(acc, __fmul_rn(a, a));
          acc = __fadd_rn(acc, __fmul_rn(b, b));
        }
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
      const float ms = __fdiv_rn(acc, static_cast<float>(H));
      const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const uint4 g = __ldg(gr + lane + 32 * i);
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float lo = __fmul_rn(__fmul_rn(bf16_lo(w[q]), r), bf16_lo(gw[q]));
          const float hi = __fmul_rn(__fmul_rn(bf16_hi(w[q]), r), bf16_hi(gw[q]));
          o[q] = pack2(lo, hi);
        }
        __stcs(yr + lane + 32 * i, make_uint4(o[0], o[1], o[2], o[3]));
      }
    } else {
      for (int vi = lane; vi < nvec; vi += 32) {
        const uint4 v = xr[vi];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float a = bf16_lo(w[q]), b = bf16_hi(w[q]);
          acc = __fadd_rn(acc, __fmul_rn(a, a));
          acc = __fadd_rn(acc, __fmul_rn(b, b));
        }
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
      const float ms = __fdiv_rn(acc, static_cast<float>(H));
      const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
      for (int vi = lane; vi < nvec; vi += 32) {
        const uint4 v = xr[vi];
        const uint4 g = __ldg(gr + vi);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float lo = __fmul_rn(__fmul_rn(bf16_lo(w[q]), r), bf16_lo(gw[q]));
          const float hi = __fmul_rn(__fmul_rn(bf16_hi(w[q]), r), bf16_hi(gw[q]));
          o[q] = pack2(lo, hi);
        }
        yr[vi] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
}

// ----------------------------------------------------- logprob: chunk tree
// Two-block LSE merge with (-inf, 0) as the empty block (same operations as the
// GEMM epilogue's fold).
__device__ __forceinline__ void lse_merge_into(float& m1, float& s1, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m1 == -INFINITY) {
    m1 = m2;
    s1 = s2;
    return;
  }
  const float mm = fmaxf(m1, m2);
  s1 = __fadd_rn(__fmul_rn(s1, expf(__fsub_rn(m1, mm))), __fmul_rn(s2, expf(__fsub_rn(m2, mm))));
  m1 = mm;
}

// Statistics are stored entry-major ([entry][T]: consecutive rows adjacent), so both the
// GEMM epilogue's writes and the reads here are coalesced.
//
// Tile statistics -> chunk statistics: thread (c, t) folds the tiles of chunk c for row t left
// to right -- the fold the GEMM epilogue performs when one CTA owns a whole chunk.
__global__ void lse_fold_tiles_kernel(const float2* __restrict__ tile_stats, float2* __restrict__ chunk_stats, int T,
                                      int C, int ntiles, int chunk_tiles) {
  grid_dependency_wait();  // launched as a dependent grid: the tile statistics come from the GEMM
  grid_launch_dependents();
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<int64_t>(C) * T) return;
  const int c = static_cast<int>(idx / T);
  const int t = static_cast<int>(idx - static_cast<int64_t>(c) * T);
  const int t0 = c * chunk_tiles;
  const int t1 = min(t0 + chunk_tiles, ntiles);
  float2 v = tile_stats[static_cast<int64_t>(t0) * T + t];
  for (int q = t0 + 1; q < t1; ++q) {
    const float2 w = tile_stats[static_cast<int64_t>(q) * T + t];
    lse_merge_into(v.x, v.y, w.x, w.y);
  }
  chunk_stats[idx] = v;
}

// Per row: the C chunk statistics are merged by the balanced pairwise tree with the odd node
// carried up: level by level, node i of the next level is node 2i (left, lower chunks) merged
// with node 2i+1, and an odd last node passes up unchanged.  One warp per row holds the row's
// nodes in shared memory and merges each level's pairs in parallel (log2 C levels).
// lse = m + logf(s); out = z_sel - lse.
// zsel holds one [T] array per vocab shard; a row's selected logit comes from the shard whose
// chunk range [chunk0[r], chunk0[r+1]) holds the id's chunk (one shard: chunk0 = {0, C}).
constexpr int kFinalizeWarps = 8;
constexpr int kFinalizeMaxChunks = 256;

__global__ void __launch_bounds__(32 * kFinalizeWarps)
    lse_finalize_kernel(const float2* __restrict__ stats, const float* __restrict__ zsel,
                        const int32_t* __restrict__ ids, float* __restrict__ out, int T, int C, int V,
                        ShardBounds shards, unsigned int* status) {
  __shared__ float2 node[kFinalizeWarps][kFinalizeMaxChunks];
  grid_dependency_wait();  // launched as a dependent grid: the statistics come from the grid before
  grid_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  const int t = blockIdx.x * kFinalizeWarps + w;
  if (t >= T) return;  // whole warps leave together
  float2* nd = node[w];
  for (int c = lane; c < C; c += 32) nd[c] = stats[static_cast<int64_t>(c) * T + t];
  __syncwarp();
  for (int n = C; n > 1; n = (n + 1) >> 1) {
    const int pairs = n >> 1;
    float2 res[kFinalizeMaxChunks / 64];
#pragma unroll
    for (int q = 0; q < kFinalizeMaxChunks / 64; ++q) {
      const int i = lane + 32 * q;
      if (i < pairs) {
        float2 a = nd[2 * i];
        const float2 b2 = nd[2 * i + 1];
        lse_merge_into(a.x, a.y, b2.x, b2.y);
        res[q] = a;
      }
    }
    const float2 carry = (n & 1) ? nd[n - 1] : make_float2(0.f, 0.f);
    __syncwarp();
#pragma unroll
    for (int q = 0; q < kFinalizeMaxChunks / 64; ++q) {
      const int i = lane + 32 * q;
      if (i < pairs) nd[i] = res[q];
    }
    if ((n & 1) && lane == 0) nd[pairs] = carry;
    __syncwarp();
  }
  if (lane != 0) return;
  const int id = ids[t];
  if (id < 0 || id >= V) {
    out[t] = __int_as_float(0x7fc00000);
    atomicOr(status, kDevBadToken);
    return;
  }
  const int chunk = id / (LP_TILE_COLS * LP_CHUNK_TILES);
  int owner = 0;
  for (int r = 1; r < shards.n; ++r)
    if (shards.chunk0[r] <= chunk) owner = r;
  const float lse = __fadd_rn(nd[0].x, logf(nd[0].y));
  out[t] = __fsub_rn(zsel[static_cast<int64_t>(owner) * T + t], lse);
}

// ------------------------------------------------------------------ MoE route
// One warp per token; each lane holds E/32 logits (expert e = lane + 32 i).
// k rounds of a warp argmax with ties to the lower expert id; gates are
// expf(l_j - l_0) / sum_j, the sum taken in slot order.
template <int EPL>
__global__ void moe_route_kernel(const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ ids,
                                 float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * warps + (threadIdx.x >> 5); t < T;
       t += static_cast<int64_t>(gridDim.x) * warps) {
    float v[EPL];
    bool taken[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      v[i] = e < E ? logits[t * E + e] : -INFINITY;
      taken[i] = e >= E;
    }
    // lane j keeps the j-th selection (k <= 32), so nothing goes to local memory
    float my_l = -INFINITY;
    int my_e = 0;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        if (!taken[i] && (v[i] > bv || (v[i] == bv && e < be) || be == 0x7fffffff)) {
          bv = v[i];
          be = e;
        }
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oe = __shfl_xor_sync(0xffffffffu, be, off);
        if (oe != 0x7fffffff && (be == 0x7fffffff || ov > bv || (ov == bv && oe < be))) {
          bv = ov;
          be = oe;
        }
      }
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (lane + 32 * i == be) taken[i] = true;
      if (lane == j) {
        my_l = bv;
        my_e = be;
      }
    }
    const float m = __shfl_sync(0xffffffffu, my_l, 0);
    const float ex = lane < k ? expf(__fsub_rn(my_l, m)) : 0.f;
    float s = 0.f;  // slot order: s = ((e_0 + e_1) + e_2) + ...
    for (int j = 0; j < k; ++j) s = __fadd_rn(s, __shfl_sync(0xffffffffu, ex, j));
    if (lane < k) {
      ids[t * k + lane] = my_e;
      w[t * k + lane] = __fdiv_rn(ex, s);
    }
  }
}

// ---------------------------------------------------------------- MoE permute
// A counting sort in three passes over chunks of MOE_PERM_CHUNK pairs:
//   hist     chunk c counts its pairs per expert                 -> hist[c][e]
//   scan     hist[c][e] becomes the exclusive prefix over chunks; counts, offsets
//            and the unit prefixes of the two grouped GEMMs follow from the totals
//   scatter  chunk c writes each listed pair to offsets[e] + hist[c][e] + (its rank
//            among the chunk's earlier pairs of expert e)
// Every count is an exact integer and every pair's slot is determined by the pair order
// alone, so perm lists the pairs of each expert in ascending pair order.

__global__ void moe_hist_kernel(const int32_t* __restrict__ ids, int64_t P, int E, int32_t* __restrict__ hist,
                                unsigned int* status) {
  __shared__ int h[MOE_MAX_EXPERTS];
  for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
  __syncthreads();
  const int64_t p0 = static_cast<int64_t>(blockIdx.x) * MOE_PERM_CHUNK;
  const int64_t p1 = min(P, p0 + MOE_PERM_CHUNK);
  for (int64_t p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
    const int id = ids[p];
    if (id >= 0 && id < E) atomicAdd(&h[id], 1);
    else atomicOr(status, kDevBadToken);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[static_cast<int64_t>(blockIdx.x) * E + e] = h[e];
}

// One block of 4 x MOE_MAX_EXPERTS threads: thread (g, e) walks a quarter of the chunks of
// expert e.  Then counts (zero for experts outside the partition), offsets and the unit
// prefixes (row blocks x n-tiles per expert) as exclusive scans over the experts.
__global__ void __launch_bounds__(4 * MOE_MAX_EXPERTS)
    moe_scan_kernel(int32_t* __restrict__ hist, int C, int E, const int32_t* __restrict__ part_map, int part,
                    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ up_prefix,
                    int up_nblocks, int32_t* __restrict__ down_prefix, int down_nblocks, int up_unit_rows,
                    int down_unit_rows) {
  __shared__ int part_sum[4][MOE_MAX_EXPERTS];
  __shared__ int scan[3][MOE_MAX_EXPERTS + 1];
  const int g = threadIdx.x / MOE_MAX_EXPERTS;
  const int e = threadIdx.x % MOE_MAX_EXPERTS;
  const int per = (C + 3) / 4;
  const int c0 = min(C, g * per), c1 = min(C, c0 + per);
  int sum = 0;
  if (e < E)
    for (int c = c0; c < c1; ++c) sum += hist[static_cast<int64_t>(c) * E + e];
  part_sum[g][e] = sum;
  __syncthreads();
  if (e < E) {
    int run = 0;
    for (int q = 0; q < g; ++q) run += part_sum[q][e];
    for (int c = c0; c < c1; ++c) {
      const int64_t i = static_cast<int64_t>(c) * E + e;
      const int v = hist[i];
      hist[i] = run;
      run += v;
    }
  }
  if (g == 0) {
    int cnt = 0;
    if (e < E) {
      cnt = part_sum[0][e] + part_sum[1][e] + part_sum[2][e] + part_sum[3][e];
      if (part_map != nullptr && part_map[e] != part) cnt = 0;
      counts[e] = cnt;
    }
    scan[0][e] = cnt;
    scan[1][e] = (cnt + up_unit_rows - 1) / up_unit_rows * up_nblocks;
    scan[2][e] = (cnt + down_unit_rows - 1) / down_unit_rows * down_nblocks;
  }
  __syncthreads();
  // exclusive scans over the experts: thread (g < 3, e == 0) runs array g sequentially
  if (e == 0 && g < 3) {
    int run = 0;
    for (int i = 0; i < E; ++i) {
      const int v = scan[g][i];
      scan[g][i] = run;
      run += v;
    }
    scan[g][E] = run;
  }
  __syncthreads();
  for (int i = threadIdx.x; i <= E; i += blockDim.x) {
    offsets[i] = scan[0][i];
    up_prefix[i] = scan[1][i];
    down_prefix[i] = scan[2][i];
  }
}

__global__ void __launch_bounds__(MOE_PERM_THREADS)
    moe_scatter_kernel(const int32_t* __restrict__ ids, int64_t P, int E, const int32_t* __restrict__ hist,
                       const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets,
                       int32_t* __restrict__ perm, unsigned int* status) {
  constexpr int NW = MOE_PERM_THREADS / 32;
  __shared__ int base[MOE_MAX_EXPERTS];
  __shared__ int wcnt[NW][MOE_MAX_EXPERTS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    base[e] = offsets[e] + hist[static_cast<int64_t>(blockIdx.x) * E + e];
  const int64_t p0 = static_cast<int64_t>(blockIdx.x) * MOE_PERM_CHUNK;
  for (int r = 0; r < MOE_PERM_CHUNK / MOE_PERM_THREADS; ++r) {
    for (int i = threadIdx.x; i < NW * MOE_MAX_EXPERTS; i += blockDim.x) (&wcnt[0][0])[i] = 0;
    __syncthreads();
    const int64_t p = p0 + r * MOE_PERM_THREADS + threadIdx.x;
    int id = (p < P) ? ids[p] : -1;
    if (id < 0 || id >= E || counts[id] == 0) id = -1;  // not listed (bad id, or outside the partition)
    const unsigned int same = __match_any_sync(0xffffffffu, id);
    const int rank = __popc(same & ((1u << lane) - 1u));
    if (id >= 0 && rank == 0) wcnt[warp][id] = __popc(same);
    __syncthreads();
    if (id >= 0) {
      int pos = base[id] + rank;
      for (int w = 0; w < warp; ++w) pos += wcnt[w][id];
      if (ISO_DCHECK(pos >= 0 && pos < P, status)) perm[pos] = static_cast<int32_t>(p);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int add = 0;
#pragma unroll
      for (int w = 0; w < NW; ++w) add += wcnt[w][e];
      base[e] += add;
    }
    __syncthreads();  // wcnt is cleared for the next round only after every reader is done
  }
}

// x_perm[i] = x[perm[i] / k]: one warp per row, 16-byte vectors, 8 loads per lane in flight
// before their stores (one load at a time per lane left the copy latency-bound).
__global__ void moe_gather_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ perm,
                                  const int32_t* __restrict__ total, int k, int H, __nv_bfloat16* __restrict__ xp,
                                  int64_t P, unsigned int* status) {
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  const int n = *total;
  const int nvec = H / 8;
  for (int i = blockIdx.x * warps + (threadIdx.x >> 5); i < n; i += gridDim.x * warps) {
    if (!ISO_DCHECK(i < P && perm[i] >= 0 && perm[i] < P, status)) continue;
    const int t = perm[i] / k;
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t) * H);
    uint4* dst = reinterpret_cast<uint4*>(xp + static_cast<int64_t>(i) * H);
    for (int v0 = lane; v0 < nvec; v0 += 32 * 8) {
      uint4 r[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (v0 + 32 * u < nvec) r[u] = __ldg(src + v0 + 32 * u);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (v0 + 32 * u < nvec) dst[v0 + 32 * u] = r[u];
    }
  }
}

// out[t, c] = bf16_rn(tree_j rn(w[t,j] * y[t,j,c])): 8 columns per thread.  Grid x covers a
// row's 8-column vectors, grid y strides over the tokens.  A thread first issues the k slot
// loads of its 8 columns (all in flight together), then runs the slot tree one column at a
// time, which keeps few registers live and many blocks resident (5.7 TB/s at T = 8192,
// k = 8, H = 2048 on GB300, against 2.5 TB/s for per-slot products of all columns at once).
__global__ void __launch_bounds__(256)
    moe_combine_kernel(const __nv_bfloat16* __restrict__ y, const float* __restrict__ w, int T, int k, int H,
                       __nv_bfloat16* __restrict__ out) {
  const int v = blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= H / 8) return;
  const int c = v * 8;
  for (int t = blockIdx.y; t < T; t += gridDim.y) {
    const int64_t slot0 = static_cast<int64_t>(t) * k;
    uint4 q4[8];
    float wj[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k) {
        q4[j] = __ldcs(reinterpret_cast<const uint4*>(y + (slot0 + j) * H + c));
        wj[j] = w[slot0 + j];
      } else {
        q4[j] = make_uint4(0u, 0u, 0u, 0u);
        wj[j] = 0.f;
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float lo[8], hi[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t word = q == 0 ? q4[j].x : (q == 1 ? q4[j].y : (q == 2 ? q4[j].z : q4[j].w));
        lo[j] = __fmul_rn(wj[j], bf16_lo(word));
        hi[j] = __fmul_rn(wj[j], bf16_hi(word));
      }
      o[q] = pack2(tree_sum<8>(lo, k), tree_sum<8>(hi, k));
    }
    __stcs(reinterpret_cast<uint4*>(out + static_cast<int64_t>(t) * H + c), make_uint4(o[0], o[1], o[2], o[3]));
  }
}

// ----------------------------------------------------------- bounded wait test
__global__ void bounded_wait_selftest_kernel(uint64_t timeout_ns, unsigned int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nothing ever arrives on `bar`: the wait must give up after timeout_ns
    (void)mbar_wait(&bar, 0, timeout_ns, &abort_flag, status);
  }
  __syncthreads();
}

// ================================================================== launchers
static int grid_for(int64_t work_items, int threads, int max_blocks) {
  int64_t b = (work_items + threads - 1) / threads;
  if (b < 1) b = 1;
  if (b > max_blocks) b = max_blocks;
  return static_cast<int>(b);
}

cudaError_t launch_tree_combine(const float* S, int64_t lds, int64_t rank_stride, int R, uint16_t* C, int64_t ldc,
                                int M, int N, cudaStream_t s) {
  const int64_t work = static_cast<int64_t>(M) * (N / 4);
  const cudaError_t e = launch_dependent(tree_combine_kernel, dim3(grid_for(work, 256, sm_count() * 8)), dim3(256), 0,
                                         s, 1u, S, lds, rank_stride, R, reinterpret_cast<__nv_bfloat16*>(C), ldc, M, N);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// The same RMSNorm with the rows staged in shared memory by bulk copies: one CTA per SM, 8
// warps, each warp a ring of NB row buffers.  A warp's lane 0 keeps NB - 1 row loads in flight
// (cp.async.bulk, completion on the buffer's mbarrier) and writes each finished row back with a
// bulk store from the same buffer, which it reuses once that store has read it.  Lane l reads
// the row's 8-element vectors l, l + 32, ... from shared memory and runs exactly the arithmetic
// of rmsnorm_kernel (same per-lane order, same shuffle tree), so the bits are the same; the
// copies keep ~128 KB of reads in flight per SM without holding rows in registers.
constexpr int RMS_BULK_WARPS = 8;

template <int VPL, int NB>
__global__ void __launch_bounds__(32 * RMS_BULK_WARPS, 1)
    rmsnorm_bulk_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ gamma, float eps,
                        __nv_bfloat16* __restrict__ y, int T, int H, unsigned int* status, uint64_t timeout_ns) {
  constexpr int ROWB = VPL * 32 * 16;  // bytes per row
  extern __shared__ __align__(128) uint8_t rms_smem[];
  __shared__ int abort_flag_s;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint8_t* const wbuf = rms_smem + warp * NB * ROWB;
  uint64_t* const full = reinterpret_cast<uint64_t*>(rms_smem + RMS_BULK_WARPS * NB * ROWB) + warp * NB;
  if (threadIdx.x == 0) abort_flag_s = 0;
  if (lane == 0) {
    for (int b = 0; b < NB; ++b) mbar_init(&full[b], 1);
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort_flag = &abort_flag_s;
  const int64_t G = static_cast<int64_t>(gridDim.x) * RMS_BULK_WARPS;
  const int64_t w0 = static_cast<int64_t>(blockIdx.x) * RMS_BULK_WARPS + warp;
  const int64_t n = T > w0 ? (T - w0 + G - 1) / G : 0;  // rows of this warp: w0 + i G
  const uint4* gr = reinterpret_cast<const uint4*>(gamma);
  if (lane == 0)
    for (int64_t i = 0; i < NB - 1 && i < n; ++i) {
      const int b = static_cast<int>(i % NB);
      mbar_arrive_expect_tx(&full[b], ROWB);
      bulk_load(wbuf + b * ROWB, x + (w0 + i * G) * H, ROWB, &full[b]);
    }
  for (int64_t i = 0; i < n; ++i) {
    const int b = static_cast<int>(i % NB);
    if (!mbar_wait(&full[b], static_cast<uint32_t>((i / NB) & 1), timeout_ns, abort_flag, status)) break;
    uint4* rb = reinterpret_cast<uint4*>(wbuf + b * ROWB);
    uint4 v[VPL];
#pragma unroll
    for (int k = 0; k < VPL; ++k) v[k] = rb[lane + 32 * k];
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
      const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float a = bf16_lo(w[q]), c = bf16_hi(w[q]);
        acc = __fadd_rn(acc, __fmul_rn(a, a));
        acc = __fadd_rn(acc, __fmul_rn(c, c));
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
    const float ms = __fdiv_rn(acc, static_cast<float>(H));
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
      const uint4 g = __ldg(gr + lane + 32 * k);
      const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
      const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float lo = __fmul_rn(__fmul_rn(bf16_lo(w[q]), r), bf16_lo(gw[q]));
        const float hi = __fmul_rn(__fmul_rn(bf16_hi(w[q]), r), bf16_hi(gw[q]));
        o[q] = pack2(lo, hi);
      }
      rb[lane + 32 * k] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    fence_proxy_async_smem();  // the row's generic stores become visible to the bulk store
    __syncwarp();
    if (lane == 0) {
      bulk_store(y + (w0 + i * G) * H, rb, ROWB);
      bulk_commit();
      // refill the buffer of row i - 1 with row i + NB - 1 once that row's store has read it
      if (i + NB - 1 < n) {
        bulk_wait_read<1>();
        const int bn = static_cast<int>((i + NB - 1) % NB);
        mbar_arrive_expect_tx(&full[bn], ROWB);
        bulk_load(wbuf + bn * ROWB, x + (w0 + (i + NB - 1) * G) * H, ROWB, &full[bn]);
      }
    }
    __syncwarp();
  }
  if (lane == 0) bulk_wait_all();
}

template <int VPL, int NB>
static cudaError_t launch_rmsnorm_bulk(const __nv_bfloat16* X, const __nv_bfloat16* G, float eps, __nv_bfloat16* Y,
                                       int T, int H, cudaStream_t s) {
  constexpr int ROWB = VPL * 32 * 16;
  constexpr int SMEM = RMS_BULK_WARPS * NB * (ROWB + 8);
  static_assert(SMEM <= 227 * 1024, "rows and barriers fit one CTA's shared memory");
  auto kern = rmsnorm_bulk_kernel<VPL, NB>;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  const int64_t want = (static_cast<int64_t>(T) + RMS_BULK_WARPS - 1) / RMS_BULK_WARPS;
  const int blocks = static_cast<int>(want < sm_count() ? want : sm_count());
  kern<<<blocks, 32 * RMS_BULK_WARPS, SMEM, s>>>(X, G, eps, Y, T, H, device_status_ptr(), wait_timeout_ns());
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const uint16_t* x, const uint16_t* gamma, float eps, uint16_t* y, int T, int H,
                           cudaStream_t s) {
  const int threads = 256;  // 8 rows per block
  const int blocks = grid_for(static_cast<int64_t>(T) * 32, threads, sm_count() * 16);
  auto X = reinterpret_cast<const __nv_bfloat16*>(x);
  auto G = reinterpret_cast<const __nv_bfloat16*>(gamma);
  auto Y = reinterpret_cast<__nv_bfloat16*>(y);
  // Large batches take the bulk-staged kernel (measured on GB300, bits identical: T = 262144,
  // H = 4096 0.913 -> 0.936 of the HBM copy rate, T = 65536 0.878 -> 0.930); below that the
  // register kernel's many small blocks start sooner (T = 8192, H = 2048: 16.0 vs 17.0 us).
  if (T >= 32768) {
    if (H == 1024) return launch_rmsnorm_bulk<4, 4>(X, G, eps, Y, T, H, s);
    if (H == 2048) return launch_rmsnorm_bulk<8, 4>(X, G, eps, Y, T, H, s);
    if (H == 4096) return launch_rmsnorm_bulk<16, 3>(X, G, eps, Y, T, H, s);
  }
  switch (H) {
    case 1024: rmsnorm_kernel<4><<<blocks, threads, 0, s>>>(X, G, eps, Y, T, H); break;
    case 2048: rmsnorm_kernel<8><<<blocks, threads, 0, s>>>(X, G, eps, Y, T, H); break;
    case 4096: rmsnorm_kernel<16><<<blocks, threads, 0, s>>>(X, G, eps, Y, T, H); break;
    case 8192: rmsnorm_kernel<32><<<blocks, threads, 0, s>>>(X, G, eps, Y, T, H); break;
    default: rmsnorm_kernel<0><<<blocks, threads, 0, s>>>(X, G, eps, Y, T, H); break;
  }
  return cudaGetLastError();
}

// Per-row 1 / sqrt(mean x^2 + eps) of the fused RMSNorm prologue: one warp per row with the
// reduction of rmsnorm_kernel (lane l accumulates x^2 over the 8-element vectors l, l + 32, ...
// in ascending order, low then high half of each pair; xor shuffle tree 16, 8, 4, 2, 1; IEEE
// division and square root), so the factor has the bits iso_rmsnorm uses.
__global__ void __launch_bounds__(256) rms_rows_kernel(const __nv_bfloat16* __restrict__ x, float eps,
                                                       float* __restrict__ rinv, int T, int H, int64_t ldx) {
  const int lane = threadIdx.x & 31;
  const int nvec = H / 8;
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5); row < T;
       row += static_cast<int64_t>(gridDim.x) * 8) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * ldx);
    float acc = 0.f;
    for (int vi = lane; vi < nvec; vi += 32) {
      const uint4 v = xr[vi];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float a = bf16_lo(w[q]), b = bf16_hi(w[q]);
        acc = __fadd_rn(acc, __fmul_rn(a, a));
        acc = __fadd_rn(acc, __fmul_rn(b, b));
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
    const float ms = __fdiv_rn(acc, static_cast<float>(H));
    if (lane == 0) rinv[row] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
  }
}

cudaError_t launch_rms_rows(const void* x, float eps, float* rinv, int T, int H, int64_t ldx, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  int blocks = (T + 7) / 8;
  if (blocks > sm_count() * 16) blocks = sm_count() * 16;
  rms_rows_kernel<<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x), eps, rinv, T, H, ldx);
  return cudaGetLastError();
}

cudaError_t launch_lse_finalize(const float2* tile_stats, float2* chunk_stats, const float* zsel, const int32_t* ids,
                                float* out, int T, int C, int V, int ntiles, int chunk_tiles, cudaStream_t s) {
  if (tile_stats != nullptr) {
    const cudaError_t e = launch_lse_fold_tiles(tile_stats, chunk_stats, T, C, ntiles, chunk_tiles, s);
    if (e != cudaSuccess) return e;
  }
  ShardBounds one;
  one.n = 1;
  one.chunk0[0] = 0;
  return launch_lse_combine(chunk_stats, zsel, ids, out, T, C, V, one, s);
}

cudaError_t launch_lse_combine(const float2* chunk_stats, const float* zsel, const int32_t* ids, float* out, int T,
                               int C, int V, const ShardBounds& shards, cudaStream_t s) {
  const cudaError_t e =
      launch_dependent(lse_finalize_kernel, dim3((T + kFinalizeWarps - 1) / kFinalizeWarps), dim3(32 * kFinalizeWarps),
                       0, s, 1u, chunk_stats, zsel, ids, out, T, C, V, shards, device_status_ptr());
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_lse_fold_tiles(const float2* tile_stats, float2* chunk_stats, int T, int C, int ntiles,
                                  int chunk_tiles, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(C) * T;
  if (n == 0) return cudaSuccess;
  const cudaError_t e = launch_dependent(lse_fold_tiles_kernel, dim3(static_cast<unsigned int>((n + 255) / 256)),
                                         dim3(256), 0, s, 1u, tile_stats, chunk_stats, T, C, ntiles, chunk_tiles);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_moe_route(const float* logits, int T, int E, int k, int32_t* ids, float* w, cudaStream_t s) {
  const int threads = 256;
  const int blocks = grid_for(static_cast<int64_t>(T) * 32, threads, sm_count() * 16);
  if (E <= 32) moe_route_kernel<1><<<blocks, threads, 0, s>>>(logits, T, E, k, ids, w);
  else if (E <= 64) moe_route_kernel<2><<<blocks, threads, 0, s>>>(logits, T, E, k, ids, w);
  else if (E <= 128) moe_route_kernel<4><<<blocks, threads, 0, s>>>(logits, T, E, k, ids, w);
  else moe_route_kernel<8><<<blocks, threads, 0, s>>>(logits, T, E, k, ids, w);
  return cudaGetLastError();
}

int64_t moe_perm_chunks(int64_t P) { return (P + MOE_PERM_CHUNK - 1) / MOE_PERM_CHUNK; }

cudaError_t launch_moe_permute(const int32_t* ids, int64_t P, int E, const int32_t* part_map, int part,
                               int32_t* counts, int32_t* hist, int32_t* perm, int32_t* offsets, int32_t* up_prefix,
                               int up_nblocks, int32_t* down_prefix, int down_nblocks, int up_unit_rows,
                               int down_unit_rows, cudaStream_t s) {
  const int64_t C = moe_perm_chunks(P);
  if (C > 0) {
    moe_hist_kernel<<<static_cast<unsigned int>(C), MOE_PERM_THREADS, 0, s>>>(ids, P, E, hist, device_status_ptr());
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  moe_scan_kernel<<<1, 4 * MOE_MAX_EXPERTS, 0, s>>>(hist, static_cast<int>(C), E, part_map, part, counts, offsets,
                                                    up_prefix, up_nblocks, down_prefix, down_nblocks, up_unit_rows,
                                                    down_unit_rows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || C == 0) return e;
  moe_scatter_kernel<<<static_cast<unsigned int>(C), MOE_PERM_THREADS, 0, s>>>(ids, P, E, hist, counts, offsets,
                                                                                perm, device_status_ptr());
  return cudaGetLastError();
}

cudaError_t launch_moe_gather(const uint16_t* x, const int32_t* perm, const int32_t* total, int64_t max_rows, int k,
                              int H, uint16_t* xp, cudaStream_t s) {
  const int threads = 256;
  moe_gather_kernel<<<grid_for(max_rows * 32, threads, sm_count() * 16), threads, 0, s>>>(
      reinterpret_cast<const __nv_bfloat16*>(x), perm, total, k, H, reinterpret_cast<__nv_bfloat16*>(xp), max_rows,
      device_status_ptr());
  return cudaGetLastError();
}

cudaError_t launch_moe_combine(const uint16_t* y, const float* w, int T, int k, int H, uint16_t* out,
                               cudaStream_t s) {
  const int threads = 256;
  const int gx = (H / 8 + threads - 1) / threads;
  int gy = (sm_count() * 8 + gx - 1) / gx;
  if (gy > T) gy = T;
  if (gy > 65535) gy = 65535;
  moe_combine_kernel<<<dim3(gx, gy), threads, 0, s>>>(reinterpret_cast<const __nv_bfloat16*>(y), w, T, k, H,
                                                      reinterpret_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

cudaError_t launch_bounded_wait_selftest(uint64_t timeout_ns, cudaStream_t s) {
  bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(timeout_ns, device_status_ptr());
  return cudaGetLastError();
}

}  // namespace iso
