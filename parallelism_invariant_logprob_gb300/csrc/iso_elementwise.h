// iso_elementwise.h -- launchers of the memory-bound kernels (elementwise.cu).
#pragma once
#include "iso_internal.h"

namespace iso {

cudaError_t launch_tree_combine(const float* S, int64_t lds, int64_t rank_stride, int R, uint16_t* C, int64_t ldc,
                                int M, int N, cudaStream_t s);
cudaError_t launch_rmsnorm(const uint16_t* x, const uint16_t* gamma, float eps, uint16_t* y, int T, int H,
                           cudaStream_t s);
// chunk_stats: [C][T] chunk statistics (m, s).  With tile_stats ([ntiles][T] per-tile statistics)
// the chunk entries are first formed by folding chunk_tiles tiles left to right into chunk_stats.
cudaError_t launch_lse_finalize(const float2* tile_stats, float2* chunk_stats, const float* zsel, const int32_t* ids,
                                float* out, int T, int C, int V, int ntiles, int chunk_tiles, cudaStream_t s);
// Vocab shards: shard r owns chunks [chunk0[r], chunk0[r+1]) (chunk0[n] implied = C).
constexpr int kMaxVocabShards = 64;
struct ShardBounds {
  int n;
  int chunk0[kMaxVocabShards];
};
// Tile statistics [ntiles][T] -> chunk statistics [C][T] (left fold of each chunk's tiles).
cudaError_t launch_lse_fold_tiles(const float2* tile_stats, float2* chunk_stats, int T, int C, int ntiles,
                                  int chunk_tiles, cudaStream_t s);
// Chunk tree over chunk_stats [C][T], lse, and out = zsel[owner shard][t] - lse.
cudaError_t launch_lse_combine(const float2* chunk_stats, const float* zsel, const int32_t* ids, float* out, int T,
                               int C, int V, const ShardBounds& shards, cudaStream_t s);
cudaError_t launch_moe_route(const float* logits, int T, int E, int k, int32_t* ids, float* w, cudaStream_t s);
// Chunks of the permutation's counting sort for P pairs; hist holds chunks x E int32.
int64_t moe_perm_chunks(int64_t P);
// part_map (device, [E]) selects experts with part_map[e] == part; NULL = all.  The unit
// prefixes count ceil(count / unit rows) row blocks per expert times the n-blocks (unit rows:
// 128 for single-CTA units, 256 for CTA pairs; each GEMM its own).
cudaError_t launch_moe_permute(const int32_t* ids, int64_t P, int E, const int32_t* part_map, int part,
                               int32_t* counts, int32_t* hist, int32_t* perm, int32_t* offsets, int32_t* up_prefix,
                               int up_nblocks, int32_t* down_prefix, int down_nblocks, int up_unit_rows,
                               int down_unit_rows, cudaStream_t s);
cudaError_t launch_moe_gather(const uint16_t* x, const int32_t* perm, const int32_t* total, int64_t max_rows, int k,
                              int H, uint16_t* xp, cudaStream_t s);
cudaError_t launch_moe_combine(const uint16_t* y, const float* w, int T, int k, int H, uint16_t* out,
                               cudaStream_t s);
cudaError_t launch_bounded_wait_selftest(uint64_t timeout_ns, cudaStream_t s);
// rinv[t] = 1 / sqrt(mean_i x[t, i]^2 + eps) with iso_rmsnorm's reduction (x: [T x H], leading dim ldx).
cudaError_t launch_rms_rows(const void* x, float eps, float* rinv, int T, int H, int64_t ldx, cudaStream_t s);

}  // namespace iso
