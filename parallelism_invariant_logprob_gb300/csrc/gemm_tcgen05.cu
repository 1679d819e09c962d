// gemm_tcgen05.cu -- the leaf-tree GEMM engine on 5th-generation tensor cores.
//
// What it computes [IsoExec blog, "Parallelism-invariant kernels"]: K is cut
// into L contiguous leaves; each leaf is one deterministic chain of
// tcgen05.mma (M=128, N=128, K=16, bf16 x bf16 -> fp32 in TMEM), ascending k,
// the first MMA of a leaf overwriting its accumulator; the L leaf partials are
// combined by the fixed balanced binary tree (level by level, left operand =
// lower leaf index, IEEE fp32 round-to-nearest adds) and the root is either
//   EPI_BF16    converted to bf16 once and stored [RL-Kernel blog, §2 trigger
//               table "accumulate-then-convert"; §7 "GEMM"],
//   EPI_F32     stored as fp32 (a simulated rank's subtree root), or
//   EPI_SWIGLU  for the MoE gate/up projection: a tile holds 64 gate and the
//               matching 64 up columns; the epilogue writes
//               h = bf16(silu(bf16 g) * bf16 u) [RL-Kernel blog, §6 table row 04]
//   EPI_LOGPROB reduced to per-row (max, sum exp) statistics per 128-column
//               vocab tile, folded left to right over the tiles of a vocab
//               chunk with the two-block LSE merge [RL-Kernel blog, §4
//               "Causal Chain: How Block Merge Order Alters LSE"; §7 "LogP"],
//               plus the logit of the selected token, or
//   EPI_CLUSTER one row block split into leaf groups over a thread-block
//               cluster: each CTA's group root meets the others' in
//               distributed shared memory for the tree's top levels.
//
// A row's bits depend only on that row, the B columns and the contract: the
// MMA instruction shape, the per-leaf chain and the tree are the same for
// every M, every tile position and every schedule; nothing is split along K
// beyond the contract's leaves and nothing uses atomics.
//
// Structure (one CTA per SM, persistent over work units; with PAIR two CTAs on
// neighbouring SMs run M = 256 MMAs over both, each holding 128 A rows and half of B):
//   warps 0,3 TMA producers, one elected lane each (warp 0 the stages of the even
//             leaves, warp 3 those of the odd leaves): A tile 128x64 (K-major)
//             and B tile 64x128 (MN-major, two 64-column boxes), 128-byte
//             swizzle, as many stages as shared memory holds (up to 12).
//   warps 1-2 MMA issuers, one elected lane each: warp 1 issues the even leaves and
//             warp 2 the odd leaves of every leaf pair, so one leaf's waits
//             overlap the other's MMAs (a single issuer measured slower); warp 1
//             also owns the TMEM allocation.
//   warps 4-7 epilogue: one thread per accumulator row (TMEM lane); they read
//             each finished leaf once (tcgen05.ld) and run the tree in registers
//             while the MMAs fill the next leaves, and write the output.  With
//             short leaves (bf16 and SwiGLU outputs) warps 8-11 join them: each
//             warp then takes one 64-column half of its lane quarter's rows.
// Leaves accumulate in four 128-column TMEM buffers, the CTA's s-th leaf in
// buffer s % 4, so the MMA threads and the epilogue agree on buffers and
// barrier phases without exchanging anything.
#include <cuda_bf16.h>
#include <stdio.h>
#include <stdlib.h>

#include <atomic>
#include <mutex>

#include "iso_internal.h"
#include "iso_ptx.cuh"

namespace iso {

namespace {

struct Unit {
  int a_row0;      // first A row of this unit
  int a_col0;      // first A column (the K offset of a leaf group; 0 otherwise)
  int b_row0;      // first B row (K offset of the expert in grouped mode, or of a leaf group)
  int n_tile0;     // first 128-column tile
  int n_tiles;     // tiles in this unit
  int rows_valid;  // rows of the 128 that are real
  int chunk;       // vocab chunk (logprob)
};

__device__ __forceinline__ int unit_count(const GemmParams& p) {
  if (p.unit_mode == UNIT_GROUPED) return p.g_unit_prefix[p.E];
  return p.num_units;
}

// Unit u of the launch.  With CTA pairs (cl = 2) a unit covers 2 x 128 rows: the CTA of
// rank r takes the 128-row block 2 mb + r of it (rows_valid <= 0: a block past the rows).
__device__ __forceinline__ void decode_unit(const GemmParams& p, int u, Unit& U, int cl, int rank) {
  if (p.unit_mode == UNIT_GEMM) {
    const int per_group = p.group_m * p.n_blocks;
    const int g = u / per_group;
    const int r = u - g * per_group;
    const int gm0 = g * p.group_m;
    const int gsz = min(p.group_m, p.m_blocks - gm0);
    const int mb = gm0 + r % gsz;
    const int nb = r / gsz;
    U.a_row0 = (mb * cl + rank) * BM;
    U.a_col0 = 0;
    U.b_row0 = 0;
    U.n_tile0 = nb;
    U.n_tiles = 1;
    U.rows_valid = min(BM, p.M - U.a_row0);
    U.chunk = 0;
  } else if (p.unit_mode == UNIT_LEAF_SPLIT) {
    // group-major: the n-tiles of one leaf group run together and share its A columns
    const int r = u / p.n_blocks;
    U.a_row0 = 0;
    U.a_col0 = r * p.K;
    U.b_row0 = r * p.K;
    U.n_tile0 = u - r * p.n_blocks;
    U.n_tiles = 1;
    U.rows_valid = min(BM, p.M);
    U.chunk = r;
  } else if (p.unit_mode == UNIT_CLUSTER) {
    // one unit per CTA: tile u / R, leaf group u % R (the CTA's rank in its cluster of R)
    const int g = u % p.cluster;
    U.a_row0 = 0;
    U.a_col0 = g * p.K;
    U.b_row0 = g * p.K;
    U.n_tile0 = u / p.cluster;
    U.n_tiles = 1;
    U.rows_valid = min(BM, p.M);
    U.chunk = g;
  } else if (p.unit_mode == UNIT_LOGPROB) {
    // Row-block groups whose hidden states fit L2 (group_m row blocks; all of them when the batch
    // is small), chunk-major inside a group: the row blocks working on one vocab chunk run
    // together and share its W columns in L2, and a group's A rows stay in L2 while the whole
    // vocabulary streams past once per group.
    const int per_group = p.group_m * p.num_chunks;
    const int grp = u / per_group;
    const int r = u - grp * per_group;
    const int gm0 = grp * p.group_m;
    const int gsz = min(p.group_m, p.m_blocks - gm0);
    const int chunk = r / gsz;
    const int rb = gm0 + (r - chunk * gsz);
    U.a_row0 = (rb * cl + rank) * BM;
    U.a_col0 = 0;
    U.b_row0 = 0;
    U.n_tile0 = chunk * p.chunk_tiles;
    U.n_tiles = min(p.chunk_tiles, p.n_blocks - U.n_tile0);
    U.rows_valid = min(BM, p.M - U.a_row0);
    U.chunk = chunk;
  } else {
    // e = the largest expert with prefix[e] <= u (prefix is nondecreasing), found by the
    // whole warp at once: each lane tests up to 8 entries, all loads in flight together,
    // and the ballot counts give the number of entries <= u.  Every caller is a full warp.
    const int lane = threadIdx.x & 31;
    int cnt = 0;
#pragma unroll
    for (int j = 0; j < MOE_MAX_EXPERTS / 32; ++j) {
      const int e = j * 32 + lane;
      const bool le = e < p.E && p.g_unit_prefix[e] <= u;
      cnt += __popc(__ballot_sync(0xffffffffu, le));
    }
    const int e = cnt - 1;
    const int local = u - p.g_unit_prefix[e];
    const int mb = local / p.n_blocks;
    const int nb = local - mb * p.n_blocks;
    const int off = p.g_offsets[e];
    const int ne = p.g_offsets[e + 1] - off;
    U.a_row0 = off + (mb * cl + rank) * BM;
    U.a_col0 = 0;
    U.b_row0 = e * p.K;
    U.n_tile0 = nb;
    U.n_tiles = 1;
    U.rows_valid = min(BM, ne - (mb * cl + rank) * BM);
    U.chunk = 0;
  }
}

// Bounded wait until the shared leaf ticket reaches `want`.
__device__ __forceinline__ bool wait_ticket(volatile uint32_t* ticket, uint32_t want, uint64_t timeout_ns,
                                            volatile int* abort_flag, unsigned int* status) {
  if (*ticket == want) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (*ticket == want) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > timeout_ns) {
      *abort_flag = 1;
      atomicOr(status, kDevTimeout);
      return false;
    }
  }
}


// Register reallocation between warpgroups (every warp of a warpgroup executes the same one).
template <int R>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
}
template <int R>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
}

// One lane of a converged warp (elected once per warp and reused, so the thread that issues a
// warp's MMAs is also the one whose tcgen05.commit tracks them).
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.b32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

// ---- The leaf tree in the epilogue ("spine")
// Leaf s of this CTA (counting every tile's leaves in order) accumulates in TMEM buffer s % 4
// (the four 128-column buffers); its use index s / 4 gives the parity of the leaf_full phase
// the epilogue waits for and of the buf_free phase the next use of the buffer waits for.  The
// epilogue takes leaves in groups of up to 8 (leaf l is l % 8 of its group, G = min(L, 8)
// leaves per group) and keeps the group's partial root S in registers:
//   G = 1: S = leaf.
//   leaf 1 of the group: S = l0 + l1;  leaf 3: S = S + (l2 + l3)      (their buffers freed)
//   leaf 5: l4 + l5 into l5's buffer, l4's buffer freed
//           (8 epilogue warps: Q = l4 + l5 in registers, both buffers freed)
//   leaf 7: S = S + ((l4 + l5) + (l6 + l7))                          (the last three freed)
// which is the contract's balanced tree over the group (left operand = lower leaves, fp32 adds
// rounded to nearest).  With 16 leaves the first group's root waits in shared memory and the
// tile's root is parked + S.  One register partial per thread suffices, TMEM is written once
// per group of 8, and the buffer that the next tile's first leaf takes (l4's) is free two
// leaves before the tile ends; merging in TMEM wrote every merge back and freed that buffer
// only after three read-add-write merges.

// Column j (0 <= j < NC) of the columns an epilogue thread owns in every tile: all 128 with 4
// epilogue warps; with 8, a 64-column half (bf16) or 32 gate and the matching 32 up columns
// (SwiGLU, gate in [0, 64), up in [64, 128)).
template <int EPI, int EPW>
__device__ __forceinline__ int spine_col(int chalf, int j) {
  if constexpr (EPW == 4) return j;
  if constexpr (EPI == EPI_SWIGLU) return j < 32 ? chalf * 32 + j : 64 + chalf * 32 + (j - 32);
  return chalf * 64 + j;
}

// S = the leaf in buffer t (G = 1).
template <int EPI, int EPW, int NC>
__device__ __forceinline__ void spine_load(uint32_t (&S)[NC], uint32_t t, int chalf) {
#pragma unroll
  for (int c = 0; c < NC / 32; ++c) tmem_ld32p(t + static_cast<uint32_t>(spine_col<EPI, EPW>(chalf, c * 32)), S + c * 32);
  tmem_ld_wait_only();
#pragma unroll
  for (int c = 0; c < NC / 32; ++c) tmem_ld_tie(S + c * 32);
}

// The spine steps read TMEM in 32-column pieces: each piece is one load round (loads, one
// wait, adds).  A round costs a TMEM load latency, so wide pieces are faster; 32 columns keep
// the temporaries of the three-buffer step beside a 4-warp epilogue's 128-register partial
// without spilling (16-column pieces were slower and spilled).
constexpr int SPINE_PIECE = 32;

// S = (first ? x + y : S + (x + y)) for the leaves in buffers t0 (left) and t1.
template <int EPI, int EPW, int NC>
__device__ __forceinline__ void spine_pair(uint32_t (&S)[NC], uint32_t t0, uint32_t t1, int chalf, bool first) {
  constexpr int W = SPINE_PIECE;
#pragma unroll
  for (int c = 0; c < NC / W; ++c) {
    const uint32_t col = static_cast<uint32_t>(spine_col<EPI, EPW>(chalf, c * W));
    uint32_t x[W], y[W];
    tmem_ld32p(t0 + col, x);
    tmem_ld32p(t1 + col, y);
    tmem_ld_wait_only();
    tmem_ld_tie(x);
    tmem_ld_tie(y);
#pragma unroll
    for (int i = 0; i < W; ++i) {
      const float v = __fadd_rn(u2f(x[i]), u2f(y[i]));
      S[c * W + i] = f2u(first ? v : __fadd_rn(u2f(S[c * W + i]), v));
    }
  }
}

// t1 = t0 + t1 in TMEM (leaves 4 and 5 of a group: left = t0), over this thread's columns.
template <int EPI, int EPW, int NC>
__device__ __forceinline__ void spine_merge(uint32_t t0, uint32_t t1, int chalf) {
  constexpr int W = SPINE_PIECE;
#pragma unroll
  for (int c = 0; c < NC / W; ++c) {
    const uint32_t col = static_cast<uint32_t>(spine_col<EPI, EPW>(chalf, c * W));
    uint32_t x[W], y[W];
    tmem_ld32p(t0 + col, x);
    tmem_ld32p(t1 + col, y);
    tmem_ld_wait_only();
    tmem_ld_tie(x);
    tmem_ld_tie(y);
#pragma unroll
    for (int i = 0; i < W; ++i) y[i] = f2u(__fadd_rn(u2f(x[i]), u2f(y[i])));
    tmem_st32p(t1 + col, y);
  }
  tmem_st_wait();
}

// S = S + (m + (x + y)) with m = leaves 4 + 5 in buffer tm and leaves 6, 7 in tx, ty.
template <int EPI, int EPW, int NC>
__device__ __forceinline__ void spine_last(uint32_t (&S)[NC], uint32_t tm, uint32_t tx, uint32_t ty, int chalf) {
  constexpr int W = SPINE_PIECE;
#pragma unroll
  for (int c = 0; c < NC / W; ++c) {
    const uint32_t col = static_cast<uint32_t>(spine_col<EPI, EPW>(chalf, c * W));
    uint32_t m[W], x[W], y[W];
    tmem_ld32p(tm + col, m);
    tmem_ld32p(tx + col, x);
    tmem_ld32p(ty + col, y);
    tmem_ld_wait_only();
    tmem_ld_tie(m);
    tmem_ld_tie(x);
    tmem_ld_tie(y);
#pragma unroll
    for (int i = 0; i < W; ++i) {
      const float r = __fadd_rn(u2f(m[i]), __fadd_rn(u2f(x[i]), u2f(y[i])));
      S[c * W + i] = f2u(__fadd_rn(u2f(S[c * W + i]), r));
    }
  }
}

// 8 epilogue warps (64 columns per thread) keep leaves 4 + 5 in registers beside S instead of
// writing them back to TMEM: Q = l4 + l5 at leaf 5 (both buffers freed at once), then
// S = S + (Q + (l6 + l7)) at leaf 7 -- the same adds in the same order as the TMEM merge.  With
// two 64-register partials live, these steps read 16-column pieces.
template <int EPI, int EPW, int NC>
__device__ __forceinline__ void spine_pair_regs(uint32_t (&Q)[NC], uint32_t t0, uint32_t t1, int chalf) {
  constexpr int W = 16;
#pragma unroll
  for (int c = 0; c < NC / W; ++c) {
    const uint32_t col = static_cast<uint32_t>(spine_col<EPI, EPW>(chalf, c * W));
    uint32_t x[W], y[W];
    tmem_ld16p(t0 + col, x);
    tmem_ld16p(t1 + col, y);
    tmem_ld_wait_only();
    tmem_ld_tie16(x);
    tmem_ld_tie16(y);
#pragma unroll
    for (int i = 0; i < W; ++i) Q[c * W + i] = f2u(__fadd_rn(u2f(x[i]), u2f(y[i])));
  }
}
template <int EPI, int EPW, int NC>
__device__ __forceinline__ void spine_last_regs(uint32_t (&S)[NC], const uint32_t (&Q)[NC], uint32_t tx, uint32_t ty,
                                                int chalf) {
  constexpr int W = 16;
#pragma unroll
  for (int c = 0; c < NC / W; ++c) {
    const uint32_t col = static_cast<uint32_t>(spine_col<EPI, EPW>(chalf, c * W));
    uint32_t x[W], y[W];
    tmem_ld16p(tx + col, x);
    tmem_ld16p(ty + col, y);
    tmem_ld_wait_only();
    tmem_ld_tie16(x);
    tmem_ld_tie16(y);
#pragma unroll
    for (int i = 0; i < W; ++i) {
      const float r = __fadd_rn(u2f(Q[c * W + i]), __fadd_rn(u2f(x[i]), u2f(y[i])));
      S[c * W + i] = f2u(__fadd_rn(u2f(S[c * W + i]), r));
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat16 a = __float2bfloat16_rn(lo);
  const __nv_bfloat16 b = __float2bfloat16_rn(hi);
  return static_cast<uint32_t>(__bfloat16_as_ushort(a)) | (static_cast<uint32_t>(__bfloat16_as_ushort(b)) << 16);
}

// Fused RMSNorm prologue, in place, rows [32 w, 32 w + 32) of the tile (transform warp w): the
// stage's A tile holds raw x (rows [row0, row0 + 128),
// columns [k0, k0 + 64)) as TMA wrote it (128-byte-swizzled K-major: row r, 16-byte chunk q of
// its 128-byte line at (r / 8) * 1024 + (r % 8) * 128 + ((q ^ (r % 8)) * 16); rows past M and
// columns past K zero-filled); the 32 lanes overwrite each element with
// y = bf16_rn((x * rinv[row]) * gamma[k]), the per-element arithmetic of iso_rmsnorm.  Lane l
// handles chunk q = l % 8 of rows 32 w + 4 i + l / 8, so its gamma chunk is the same for every row.
__device__ __forceinline__ void rmsnorm_a_rows_inplace(uint8_t* sA, const GemmParams& p, int row0, int k0, int w,
                                                       int lane) {
  const int q = lane & 7;
  const int k = k0 + q * 8;
  uint4 g = make_uint4(0u, 0u, 0u, 0u);
  if (k < p.K) g = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.a_gamma) + k));
  const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
  constexpr int kIters = (BM / 4) * (BK / 8) / 32;  // 8 chunks per lane: rows [32 w, 32 w + 32)
  float rr[kIters];
#pragma unroll
  for (int i = 0; i < kIters; ++i) {
    const int row = row0 + w * 32 + i * 4 + (lane >> 3);
    rr[i] = row < p.M ? __ldg(p.a_rinv + row) : 0.f;
  }
  // every load first, then every store: no load waits behind a store it might alias
  uint4 v[kIters];
#pragma unroll
  for (int i = 0; i < kIters; ++i) {
    const int r = w * 32 + i * 4 + (lane >> 3);
    v[i] = *reinterpret_cast<const uint4*>(sA + (r >> 3) * 1024 + (r & 7) * 128 + ((q ^ (r & 7)) << 4));
  }
#pragma unroll
  for (int i = 0; i < kIters; ++i) {
    const int r = w * 32 + i * 4 + (lane >> 3);
    const uint32_t xw[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = __fmul_rn(__fmul_rn(__uint_as_float(xw[j] << 16), rr[i]), __uint_as_float(gw[j] << 16));
      const float hi = __fmul_rn(__fmul_rn(__uint_as_float(xw[j] & 0xffff0000u), rr[i]), __uint_as_float(gw[j] & 0xffff0000u));
      const __nv_bfloat162 h2 = __floats2bfloat162_rn(lo, hi);  // round to nearest even, .x = lo
      o[j] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(sA + (r >> 3) * 1024 + (r & 7) * 128 + ((q ^ (r & 7)) << 4)) =
        make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Staging slot of 16-byte chunk c of row r in rows of CH chunks.  Rows of 128 or 256 bytes
// (CH = 8, 16): key r % 8.  Rows of 64 bytes (CH = 4, two rows per 128-byte line): key
// (r / 2) % 4.  Either way a quarter-warp's row-per-lane writes and its row-contiguous reads
// touch distinct banks.
template <int CH>
__device__ __forceinline__ int stage_slot(int c, int r) {
  static_assert(CH == 4 || CH == 8 || CH == 16, "staged rows of 64, 128 or 256 bytes");
  return CH >= 8 ? (c ^ (r & 7)) : (c ^ ((r >> 1) & 3));
}

// One epilogue warp writes its 32 TMEM lanes' pieces of the output rows.  Lane r holds
// CH 16-byte chunks of row r (8 bf16 or 4 fp32 each) and its destination row `orow` (-1:
// row not stored).  The rows go through the warp's staging area (32 rows x CH*16 bytes,
// chunk c of row r at slot stage_slot(c, r)), then out whole rows at a time: each store
// instruction covers 512/(CH*16) complete rows, so global writes are whole rows (whole
// 128-byte lines for CH >= 8) instead of 32 scattered 16-byte pieces.  Row r's chunk c goes
// to byte b0 + 16 c of the row (rows ld bytes apart in `out`); chunks at or past byte b_end
// are not stored.
template <int CH>
__device__ __forceinline__ void store_rows_staged(uint8_t* wst, int lane, const uint4 (&w)[CH], int orow,
                                                  uint8_t* out, int64_t ld, int64_t b0, int64_t b_end) {
  constexpr int ROW_BYTES = CH * 16;
  constexpr int ROWS_PER_STEP = 32 / CH;
#pragma unroll
  for (int c = 0; c < CH; ++c)
    *reinterpret_cast<uint4*>(wst + lane * ROW_BYTES + (stage_slot<CH>(c, lane) << 4)) = w[c];
  __syncwarp();
  const int c = lane % CH;
#pragma unroll 4
  for (int t = 0; t < 32 / ROWS_PER_STEP; ++t) {
    const int r = t * ROWS_PER_STEP + lane / CH;
    const int dst_row = __shfl_sync(0xffffffffu, orow, r);
    const uint4 x = *reinterpret_cast<const uint4*>(wst + r * ROW_BYTES + (stage_slot<CH>(c, r) << 4));
    const int64_t b = b0 + 16 * c;
    if (dst_row >= 0 && b < b_end) *reinterpret_cast<uint4*>(out + static_cast<int64_t>(dst_row) * ld + b) = x;
  }
  __syncwarp();
}

// Two-block LSE merge with (-inf, 0) as the empty block.
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  const float mm = fmaxf(m, m2);
  s = __fadd_rn(__fmul_rn(s, expf(__fsub_rn(m, mm))), __fmul_rn(s2, expf(__fsub_rn(m2, mm))));
  m = mm;
}

}  // namespace

// M = 128 (one CTA) or 256 (CTA pair), N = 128, A K-major, B MN-major, bf16 x bf16 -> fp32.
constexpr uint32_t kIdesc = idesc_bf16_f32(BM, BN, /*a_mn_major=*/false, /*b_mn_major=*/true);
constexpr uint32_t kIdescPair = idesc_bf16_f32(2 * BM, BN, /*a_mn_major=*/false, /*b_mn_major=*/true);

// An epilogue warp is done with TMEM buffer b (its tcgen05 accesses completed and fenced).
// One CTA: every epilogue thread arrives (count 32 x epilogue warps).  CTA pair: the MMA issuer sits in rank
// 0, so one lane per warp of either CTA arrives on rank 0's barrier (count 8).
template <bool PAIR>
__device__ __forceinline__ void release_tmem_buf(uint64_t* buf_free, int b, int lane) {
  if (PAIR) {
    __syncwarp();
    if (lane == 0) mbar_arrive_cluster_relaxed(cluster_addr(&buf_free[b], 0));
  } else {
    mbar_arrive(&buf_free[b]);
  }
}

// PAIR: launched as clusters of two CTAs (ranks 0, 1); rank 0 issues M = 256 MMAs over both,
// each CTA loads its own 128 A rows and one 64-column half of the B tile (the gate or up half
// for SwiGLU), with the loads of both counted on rank 0's stage barrier; the MMA commits
// arrive on the barriers of both CTAs.  Per CTA a stage is then 24 KB instead of 32 KB, so
// more stages fit and each SM moves three quarters of the bytes per MMA.
// FUSED: the fused RMSNorm prologue (single CTA, EPI_BF16 / EPI_LOGPROB): 12 warps, warps 8-11
// normalise the A stages in place; registers rebalanced by setmaxnreg (epilogue 256, the rest
// 120: 128 x 256 + 256 x 120 = 63,488 <= the launch's 384 x 168).
// EPW: epilogue warps, 4 or 8 (8: single CTA, EPI_BF16 / EPI_SWIGLU, 12 warps; warp 4 + 4h + q
// holds lane quarter q, column half h; setmaxnreg gives the 8 epilogue warps 224 registers and
// warps 0-3 56: 256 x 224 + 128 x 56 = 64,512 = the launch's 384 x 168).
// LS: whole-leaf stages for leaves of 96 k (GemmParams::leaf_stage; single CTA, bf16 roots,
// 8 epilogue warps): tmA2 maps the A operand with 32-column boxes and a 64-byte swizzle.
template <int EPI, bool PAIR, bool FUSED, int EPW, bool LS>
__global__ void __launch_bounds__((FUSED || EPW == 8) ? 384 : GEMM_THREADS, 1)
    iso_leaf_tree_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                              const __grid_constant__ CUtensorMap tmA2, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // k per stage and B bytes per stage in this CTA (a CTA of a pair holds half the B tile)
  const int SBK = PAIR ? p.stage_k : BK;
  const int BSTAGE = LS ? LS_B_BYTES : (PAIR ? SBK * 64 * 2 : B_STAGE_BYTES);
  constexpr int CL = PAIR ? 2 : 1;
  static_assert(!FUSED || (!PAIR && (EPI == EPI_BF16 || EPI == EPI_LOGPROB)), "fused prologue: single CTA, bf16/logprob");
  static_assert(EPW == 4 || (EPW == 8 && !PAIR && !FUSED && (EPI == EPI_BF16 || EPI == EPI_SWIGLU)),
                "8 epilogue warps: single CTA, bf16/SwiGLU outputs");
  static_assert(GEMM_THREADS_FUSED == 384 && GEMM_THREADS_EPI8 == 384, "12-warp launches");
  static_assert(!LS || (EPI == EPI_BF16 && !PAIR && !FUSED && EPW == 8), "whole-leaf stages: the 8-warp bf16 path");
  // The 16-leaf park exists only in the 4-epilogue-warp instances (the host never launches an
  // 8-warp instance with p.spill), so the 8-warp epilogues carry none of its code.
  const bool spill = (EPW == 4) && p.spill != 0;
  const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
  const int unit0 = PAIR ? static_cast<int>(blockIdx.x) / 2 : static_cast<int>(blockIdx.x);
  const int unit_step = PAIR ? static_cast<int>(gridDim.x) / 2 : static_cast<int>(gridDim.x);
  const int nstages = p.stages;
  const uint32_t b_region = static_cast<uint32_t>(nstages * p.a_bytes);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + b_region + nstages * BSTAGE);
  uint64_t* empty_bar = full_bar + MAX_STAGES;
  uint64_t* leaf_full = empty_bar + MAX_STAGES;
  uint64_t* buf_free = leaf_full + NUM_TMEM_BUFS;
  uint64_t* drain_bar = buf_free + NUM_TMEM_BUFS;
  uint64_t* raw_bar = drain_bar + 2;  // [MAX_STAGES] fused RMSNorm prologue: raw x landed in the A stage
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(raw_bar + MAX_STAGES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // Sequence number of the next leaf allowed to start.  The two MMA threads start their leaves
  // strictly in leaf order; without that, a thread could wait on a TMEM buffer's buf_free
  // barrier two phases ahead of its current phase, which the parity wait cannot tell apart
  // from the phase before.
  volatile uint32_t* next_leaf = reinterpret_cast<volatile uint32_t*>(tmem_slot + 2);
  // bf16 output staging (valid when p.epi_staged): 8 KB per epilogue warp
  uint8_t* epi_stage = smem + b_region + nstages * BSTAGE + GEMM_BARRIER_BYTES;
  // parked subtree root (valid when p.spill): fp32 [BN columns][BM rows]; in cluster mode the
  // leaf group's root, fp32 [BN columns][a_rows rows]
  float* parked = reinterpret_cast<float*>(epi_stage + (p.epi_staged ? EPI_STAGE_BYTES : 0));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (LS) tma_prefetch_desc(&tmA2);
    for (int s = 0; s < nstages; ++s) {
      mbar_init(&full_bar[s], FUSED ? 1 + 4 : 1);  // + one arrival per transform warp
      if (FUSED) mbar_init(&raw_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < NUM_TMEM_BUFS; ++b) {
      mbar_init(&leaf_full[b], 1);
      mbar_init(&buf_free[b], PAIR ? 8 : 32 * EPW);
    }
    mbar_init(&drain_bar[0], 1);
    mbar_init(&drain_bar[1], 1);
    *abort_flag = 0;
    *next_leaf = 0u;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(tmem_slot, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync_all();  // the peer's barriers are initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Everything above overlaps the previous grid of the stream (programmatic dependent launch);
  // inputs, routing tables and outputs are touched only after it has completed.
  grid_dependency_wait();
  grid_launch_dependents();
  const int nunits = unit_count(p);

  // Leaves are issued in pairs (2g, 2g+1) by two MMA threads (warps 1 and 2), one leaf each;
  // the producer interleaves their K-blocks, so issuer q owns the stages of parity q.  With one
  // leaf (L = 1) issuer 0 does everything.  K-blocks are leaf-relative: leaf l's block j covers
  // k in [l*leaf_len + 64 j, min(+64, (l+1)*leaf_len)).
  const int per = (p.L >= 2) ? 2 : 1;
  // Each leaf-parity stream (producer warp 0 / MMA warp 1: even leaves; warp 3 / warp 2: odd
  // leaves) cycles through its own ring of stages: stream q holds ring_n(q) stages starting at
  // ring_base(q), so an odd stage count splits (n + 1) / 2 + n / 2.
  auto ring_n = [&](int q) { return per == 1 ? nstages : (q == 0 ? (nstages + 1) / 2 : nstages / 2); };
  auto ring_base = [&](int q) { return q == 0 ? 0 : (nstages + 1) / 2; };

  if (warp < 4 || (FUSED && warp >= 8)) {
  if constexpr (FUSED) regs_dec<GEMM_REGS_CONTROL_FUSED>();
  if constexpr (EPW == 8) regs_dec<GEMM_REGS_CONTROL_EPI8>();
  if (warp == 0 || warp == 3) {
    const int me = warp == 0 ? 0 : 1;  // stage parity loaded by this warp
    if (me < per) {
      // ------------------------------------------------------------ producer
      // The whole warp runs the loop (warp-uniform values); one elected lane issues.
      const bool leader = elect_one();
      const int rn = ring_n(me), rb = ring_base(me);
      const uint64_t b_policy = l2_policy_evict_first();  // used when p.b_stream
      int slot = 0;
      int stage = rb;
      uint32_t round = 0;
      uint32_t issued = 0;  // stages issued by this thread
      bool ok = true;
      for (int u = unit0; u < nunits && ok; u += unit_step) {
        Unit U;
        decode_unit(p, u, U, CL, rank);
        for (int t = 0; t < U.n_tiles && ok; ++t) {
          const int n0 = (U.n_tile0 + t) * p.b_tile_cols;
          for (int g = 0; g < p.L / per && ok; ++g) {
            for (int j = 0; j < p.kb_per_leaf; ++j) {
              const int kx = (g * per + me) * p.leaf_len + j * SBK;
              const bool freed =
                  PAIR ? mbar_wait_cluster(&empty_bar[stage], (round & 1) ^ 1, p.timeout_ns, abort_flag, p.status)
                       : mbar_wait(&empty_bar[stage], (round & 1) ^ 1, p.timeout_ns, abort_flag, p.status);
              if (!freed) {
                ok = false;
                break;
              }
              uint8_t* sA = smem + stage * p.a_bytes;
              uint8_t* sB = smem + b_region + stage * BSTAGE;
              if (leader) {
                if (PAIR) {
                  // both CTAs' bytes complete on rank 0's barrier, which rank 0 arms for both
                  const uint32_t fb = cluster_addr(&full_bar[stage], 0);
                  if (rank == 0)
                    mbar_arrive_expect_tx(&full_bar[stage], static_cast<uint32_t>(2 * (p.a_bytes + BSTAGE)));
                  if (SBK == PAIR_BK)  // A: {64 k, 128 rows, 2 k-chunks} of the 3-D view, one box
                    tma_load_3d_pair(sA, &tmA, fb, 0, U.a_row0, (U.a_col0 + kx) / 64);
                  else
                    tma_load_2d_pair(sA, &tmA, fb, U.a_col0 + kx, U.a_row0);
                  tma_load_2d_pair(sB, &tmB, fb, n0 + rank * p.b_box2_off, U.b_row0 + kx);  // 64 columns
                } else if (FUSED) {
                  // raw x on raw_bar (the transform warps normalise it in place, then add their
                  // four arrivals to full_bar); B on full_bar
                  mbar_arrive_expect_tx(&raw_bar[stage], static_cast<uint32_t>(p.a_bytes));
                  tma_load_2d(sA, &tmA, &raw_bar[stage], U.a_col0 + kx, U.a_row0);
                  mbar_arrive_expect_tx(&full_bar[stage], static_cast<uint32_t>(BSTAGE));
                  tma_load_2d(sB, &tmB, &full_bar[stage], n0, U.b_row0 + kx);
                  tma_load_2d(sB + BSTAGE / 2, &tmB, &full_bar[stage], n0 + p.b_box2_off, U.b_row0 + kx);
                } else {
                  mbar_arrive_expect_tx(&full_bar[stage], static_cast<uint32_t>(p.a_bytes + BSTAGE));
                  tma_load_2d(sA, &tmA, &full_bar[stage], U.a_col0 + kx, U.a_row0);
                  if (LS)  // the leaf's last 32 columns, 64-byte swizzle
                    tma_load_2d(sA + LS_A2_OFF, &tmA2, &full_bar[stage], U.a_col0 + kx + 64, U.a_row0);
                  if (p.b_stream) {
                    tma_load_2d_hint(sB, &tmB, &full_bar[stage], n0, U.b_row0 + kx, b_policy);
                    tma_load_2d_hint(sB + BSTAGE / 2, &tmB, &full_bar[stage], n0 + p.b_box2_off, U.b_row0 + kx,
                                     b_policy);
                  } else {
                    tma_load_2d(sB, &tmB, &full_bar[stage], n0, U.b_row0 + kx);
                    tma_load_2d(sB + BSTAGE / 2, &tmB, &full_bar[stage], n0 + p.b_box2_off, U.b_row0 + kx);
                  }
                }
              }
              __syncwarp();
              ++issued;
              if (++slot == rn) {
                slot = 0;
                ++round;
              }
              stage = rb + slot;
            }
          }
        }
      }
      if (!ok && rank == 0) {
        // drain: wait (bounded) for every load this thread issued to land (rank 0's barriers
        // also count the peer's loads of the stages it armed).  This thread's k-th stage is
        // slot k % rn of its ring, filled in round k / rn.
        const uint32_t total = issued;
        for (uint32_t back = 1; back <= total && back <= static_cast<uint32_t>(rn); ++back) {
          const uint32_t k = total - back;
          const int st = rb + static_cast<int>(k % static_cast<uint32_t>(rn));
          // FUSED: the raw x loads land on raw_bar (full_bar may also wait for transform
          // arrivals that an abort cut short; its B bytes land in the same window)
          const uint32_t a = smem_u32(FUSED ? &raw_bar[st] : &full_bar[st]);
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(a, (k / static_cast<uint32_t>(rn)) & 1u)) {
            if (globaltimer_ns() - t0 > p.timeout_ns) break;
          }
        }
      }
    }
  } else if (warp == 1 || warp == 2) {
    const int me = warp - 1;  // leaf parity issued by this warp
    if (me < per && rank == 0) {
      // ----------------------------------------------------------------- MMA
      // The whole warp runs the loop (warp-uniform values); one elected lane issues.
      const bool leader = elect_one();
      const int rn = ring_n(me), rb = ring_base(me);  // this thread's stages: its stream's ring
      int slot = 0;
      int stage = rb;
      uint32_t round = 0;
      bool ok = true;
      // Descriptor start addresses are the low 18 bits of the shared::cta address (14 bits of
      // address / 16).  In a launch with clusters of more than one CTA the generic-to-shared
      // conversion also carries bits above the CTA's window; unmasked, they would run into the
      // descriptor's leading-byte-offset field (bit 16 on) and move the second 64-column chunk of
      // the MN-major B operand.
      const uint32_t smem_base = smem_u32(smem) & 0x3FFFFu;
      // descriptor templates; the start-address field (bits 0..13, 16-byte units) is added per use
      const uint64_t adesc0 = sdesc_sw128(0, 16, 1024);
      const uint64_t bdesc0 = sdesc_sw128(0, LS ? LS_B_BYTES / 2 : 8192, 1024);  // LBO: the second 64 columns
      const uint64_t a2desc0 = sdesc_sw64(0, 16, 512);                          // LS: 64-byte rows, 8-row atoms
      uint32_t seq = 0;  // sequence number of the current leaf (all tiles, both threads' leaves)
      for (int u = unit0; u < nunits && ok; u += unit_step) {
        Unit U;
        decode_unit(p, u, U, CL, rank);
        for (int t = 0; t < U.n_tiles && ok; ++t) {
          for (int leaf = 0; leaf < p.L && ok; ++leaf, ++seq) {
            // leaf seq accumulates in buffer seq % 4; from its second use on, wait until the
            // epilogue has freed the previous use (buf_free phase seq / 4 - 1)
            const int b = static_cast<int>(seq & 3u);
            const bool reuse = seq >= static_cast<uint32_t>(NUM_TMEM_BUFS);
            const uint32_t wpar = ((seq >> 2) + 1u) & 1u;
            if (per == 1 || (leaf & 1) == me) {
              if (per == 2 && !wait_ticket(next_leaf, seq, p.timeout_ns, abort_flag, p.status)) {
                ok = false;
                break;
              }
              if (reuse) {
                const bool got = PAIR ? mbar_wait_cluster(&buf_free[b], wpar, p.timeout_ns, abort_flag, p.status)
                                      : mbar_wait(&buf_free[b], wpar, p.timeout_ns, abort_flag, p.status);
                if (!got) {
                  ok = false;
                  break;
                }
                tc_fence_after();
              }
              if (per == 2) *next_leaf = seq + 1u;
              const uint32_t d = tmem_base + static_cast<uint32_t>(b * BN);
              for (int j = 0; j < p.kb_per_leaf; ++j) {
                const bool landed = PAIR ? mbar_wait_cluster(&full_bar[stage], round & 1, p.timeout_ns, abort_flag, p.status)
                                         : mbar_wait(&full_bar[stage], round & 1, p.timeout_ns, abort_flag, p.status);
                if (!landed) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                // A: K-major, 128 rows x 128 B, 8-row atoms 1024 B apart; +32 B (2 units) per K=16.
                // B: MN-major, 64-column chunks 8 KB apart (LBO), 8-row K groups 1 KB apart (SBO);
                //    +2 KB (128 units) per K=16.
                const uint32_t a_lo = (smem_base + stage * p.a_bytes) >> 4;
                const uint32_t b_lo = (smem_base + b_region + stage * BSTAGE) >> 4;
                const uint64_t adesc = adesc0 + static_cast<uint64_t>(a_lo);
                const uint64_t bdesc = bdesc0 + static_cast<uint64_t>(b_lo);
                const int rem = p.leaf_len - j * SBK;
                if (leader) {
                  if (PAIR) {
                    // K = 16 step i reads A chunk i / 4 (a 128-k stage holds two 64-k chunks, the
                    // second a_rows x 128 bytes on: 1024 units for 128 rows), +32 bytes per step
                    // inside it, and B +2 KB per step down its rows.
                    const uint64_t a_chunk = static_cast<uint64_t>((p.a_rows * 128) >> 4);
                    if (rem >= SBK) {
                      umma_bf16_pair(d, adesc, bdesc, kIdescPair, j != 0 ? 1u : 0u);
                      umma_bf16_pair(d, adesc + 2, bdesc + 128, kIdescPair, 1u);
                      umma_bf16_pair(d, adesc + 4, bdesc + 256, kIdescPair, 1u);
                      umma_bf16_pair(d, adesc + 6, bdesc + 384, kIdescPair, 1u);
                      if (SBK == PAIR_BK) {
                        umma_bf16_pair(d, adesc + a_chunk, bdesc + 512, kIdescPair, 1u);
                        umma_bf16_pair(d, adesc + a_chunk + 2, bdesc + 640, kIdescPair, 1u);
                        umma_bf16_pair(d, adesc + a_chunk + 4, bdesc + 768, kIdescPair, 1u);
                        umma_bf16_pair(d, adesc + a_chunk + 6, bdesc + 896, kIdescPair, 1u);
                      }
                    } else {
                      for (int i = 0; i < rem / UMMA_K; ++i)
                        umma_bf16_pair(d, adesc + (i >> 2) * a_chunk + 2 * (i & 3), bdesc + 128 * i, kIdescPair,
                                       (j != 0 || i != 0) ? 1u : 0u);
                    }
                    if (j == p.kb_per_leaf - 1) umma_commit_pair(&leaf_full[b], 3);
                    umma_commit_pair(&empty_bar[stage], 3);
                  } else {
                    if (LS) {
                      // one whole 96-k leaf: k 0..63 from the 128-byte-swizzled A box, k 64..95 from
                      // the 64-byte-swizzled one (+32 bytes per K = 16 within its 64-byte rows);
                      // B rows 0..95 of the stage, +2 KB per K = 16
                      const uint64_t a2desc =
                          a2desc0 + static_cast<uint64_t>((smem_base + stage * p.a_bytes + LS_A2_OFF) >> 4);
                      umma_bf16(d, adesc, bdesc, kIdesc, 0u);
                      umma_bf16(d, adesc + 2, bdesc + 128, kIdesc, 1u);
                      umma_bf16(d, adesc + 4, bdesc + 256, kIdesc, 1u);
                      umma_bf16(d, adesc + 6, bdesc + 384, kIdesc, 1u);
                      umma_bf16(d, a2desc, bdesc + 512, kIdesc, 1u);
                      umma_bf16(d, a2desc + 2, bdesc + 640, kIdesc, 1u);
                    } else if (rem >= BK) {
                      umma_bf16(d, adesc, bdesc, kIdesc, j != 0 ? 1u : 0u);
                      umma_bf16(d, adesc + 2, bdesc + 128, kIdesc, 1u);
                      umma_bf16(d, adesc + 4, bdesc + 256, kIdesc, 1u);
                      umma_bf16(d, adesc + 6, bdesc + 384, kIdesc, 1u);
                    } else {
                      for (int i = 0; i < rem / UMMA_K; ++i)
                        umma_bf16(d, adesc + 2 * i, bdesc + 128 * i, kIdesc, (j != 0 || i != 0) ? 1u : 0u);
                    }
                    if (j == p.kb_per_leaf - 1) umma_commit(&leaf_full[b]);
                    umma_commit(&empty_bar[stage]);
                  }
                }
                __syncwarp();
                if (++slot == rn) {
                  slot = 0;
                  ++round;
                }
                stage = rb + slot;
              }
            }
          }
        }
      }
      // drain: every MMA issued by this warp completes before TMEM is released
      if (leader) {
        if (PAIR)
          umma_commit_pair(&drain_bar[me], 1);
        else
          umma_commit(&drain_bar[me]);
      }
      __syncwarp();
      const uint32_t a = smem_u32(&drain_bar[me]);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(a, 0)) {
        if (globaltimer_ns() - t0 > p.timeout_ns) {
          *abort_flag = 1;
          atomicOr(p.status, kDevTimeout);
          break;
        }
      }
    }
  } else if constexpr (FUSED) {
    // ---------------------------------------------------- fused prologue (warps 8-11)
    // Walk the stages in the producers' order (for each K-block, the leaf of each parity, each
    // in its stream's ring); for each: wait for its raw x, normalise rows [32 w, 32 w + 32) in
    // place, publish with one arrival on the stage's full barrier.
    const int w = warp - 8;
    uint32_t kcnt = 0;  // K-blocks of each stream so far: stream me's kcnt-th stage
    bool ok = true;
    for (int u = unit0; u < nunits && ok; u += unit_step) {
      Unit U;
      decode_unit(p, u, U, CL, rank);
      for (int t = 0; t < U.n_tiles && ok; ++t) {
        for (int g = 0; g < p.L / per && ok; ++g) {
          for (int j = 0; j < p.kb_per_leaf && ok; ++j, ++kcnt) {
            for (int me = 0; me < per; ++me) {
              const uint32_t rn = static_cast<uint32_t>(ring_n(me));
              const int stage = ring_base(me) + static_cast<int>(kcnt % rn);
              const uint32_t round = kcnt / rn;
              ok = __all_sync(0xffffffffu, mbar_wait(&raw_bar[stage], round & 1, p.timeout_ns, abort_flag, p.status));
              if (!ok) break;
              const int kx = (g * per + me) * p.leaf_len + j * BK;
              rmsnorm_a_rows_inplace(smem + stage * p.a_bytes, p, U.a_row0, U.a_col0 + kx, w, lane);
              fence_proxy_async_smem();  // the generic-proxy stores become visible to the MMA
              __syncwarp();
              if (lane == 0) mbar_arrive(&full_bar[stage]);
            }
          }
        }
      }
    }
  }
  } else {
    // --------------------------------------------------------------- epilogue
    if constexpr (FUSED) regs_inc<256>();
    if constexpr (EPW == 8) regs_inc<GEMM_REGS_EPILOGUE_EPI8>();
    const int quarter = warp & 3;       // TMEM lane quarter this warp may access
    // EPW == 8: which of the two column sets of every tile this warp takes (bf16 roots: the
    // 64-column half; SwiGLU roots: 32 gate and the matching 32 up columns)
    const int chalf = (warp - 4) >> 2;
    // this warp's bf16 output staging: 8 KB per lane quarter, or 4 KB per warp with 8 warps
    uint8_t* const wstage = epi_stage + (EPW == 8 ? (warp - 4) * (32 * 128) : quarter * (32 * 256));
    const int row_in_tile = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    constexpr int NC = BN / (EPW / 4);  // columns of every tile this thread holds (spine_col)
    const int G = p.L < 8 ? p.L : 8;    // leaves per group of the spine
    const uint32_t tbase = tmem_base + lane_off;
    uint32_t seq = 0u;  // leaves of this CTA so far, all tiles: leaf seq is in TMEM buffer seq % 4
    bool ok = true;
    for (int u = unit0; u < nunits && ok; u += unit_step) {
      Unit U;
      decode_unit(p, u, U, CL, rank);
      const bool row_ok = row_in_tile < U.rows_valid;
      const int row = U.a_row0 + row_in_tile;
      float run_m = -INFINITY, run_s = 0.f;  // logprob: running chunk statistics
      int sel = -1;
      if (EPI == EPI_LOGPROB && row_ok) sel = p.ids[row] - p.sel_base;  // this launch's column of the id
      // destination row of the bf16 root (scattered rows: the expert layer's down projection);
      // an 8-warp epilogue loads it here so that its latency hides behind the unit's leaves
      // (a 4-warp one, short of registers, at the root)
      int orow_u = row;
      if (EPI == EPI_BF16 && EPW == 8 && row_ok && p.row_scatter != nullptr) orow_u = p.row_scatter[row];
      float zsel = 0.f;
      bool have_sel = false;
      for (int t = 0; t < U.n_tiles && ok; ++t) {
        const int n0 = (U.n_tile0 + t) * p.b_tile_cols;  // first output column of this tile
        uint32_t S[NC];  // the spine: the current group's partial root, at the end the tile's root
        uint32_t Q[EPW == 8 ? NC : 1];  // 8 warps: leaves 4 + 5 of the group (spine_pair_regs)
        for (int l = 0; l < p.L; ++l, ++seq) {
          const int b = static_cast<int>(seq & 3u);
          const int lg = l & 7;  // this leaf's place in its group
          // The tree steps run at the odd leaves of a group (every leaf when G = 1); a step
          // waits for its own leaf and, with G > 1, the one before (the two leaves run on
          // different MMA threads and may complete in either order).  One thread polls the
          // barriers; the other epilogue warps sleep in a hardware named barrier so they take
          // no issue slots from the TMA and MMA threads.
          if (G > 1 && (lg & 1) == 0) continue;
          if (threadIdx.x == 128) {
            for (uint32_t w = (G > 1 ? seq - 1u : seq); w <= seq; ++w) {
              const uint32_t par = (w >> 2) & 1u;
              if (PAIR)
                (void)mbar_wait_cluster(&leaf_full[w & 3u], par, p.timeout_ns, abort_flag, p.status);
              else
                (void)mbar_wait(&leaf_full[w & 3u], par, p.timeout_ns, abort_flag, p.status);
            }
          }
          named_bar_sync(1, 32 * EPW);
          if (*abort_flag) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (G == 1) {
            spine_load<EPI, EPW>(S, tbase + static_cast<uint32_t>(b * BN), chalf);
            tc_fence_before();
            release_tmem_buf<PAIR>(buf_free, b, lane);
          } else if (lg == 1 || lg == 3) {
            const int b0 = static_cast<int>((seq - 1u) & 3u);
            spine_pair<EPI, EPW>(S, tbase + static_cast<uint32_t>(b0 * BN), tbase + static_cast<uint32_t>(b * BN),
                                 chalf, lg == 1);
            tc_fence_before();
            release_tmem_buf<PAIR>(buf_free, b0, lane);
            release_tmem_buf<PAIR>(buf_free, b, lane);
          } else if (lg == 5) {
            const int b4 = static_cast<int>((seq - 1u) & 3u);
            if constexpr (EPW == 8) {
              spine_pair_regs<EPI, EPW, NC>(Q, tbase + static_cast<uint32_t>(b4 * BN), tbase + static_cast<uint32_t>(b * BN),
                                            chalf);
              tc_fence_before();
              release_tmem_buf<PAIR>(buf_free, b4, lane);
              release_tmem_buf<PAIR>(buf_free, b, lane);
            } else {
              spine_merge<EPI, EPW, NC>(tbase + static_cast<uint32_t>(b4 * BN), tbase + static_cast<uint32_t>(b * BN),
                                        chalf);
              tc_fence_before();
              release_tmem_buf<PAIR>(buf_free, b4, lane);
            }
          } else if (lg == 7) {
            const int b5 = static_cast<int>((seq - 2u) & 3u), b6 = static_cast<int>((seq - 1u) & 3u);
            if constexpr (EPW == 8) {
              spine_last_regs<EPI, EPW, NC>(S, Q, tbase + static_cast<uint32_t>(b6 * BN), tbase + static_cast<uint32_t>(b * BN),
                                            chalf);
              tc_fence_before();
              release_tmem_buf<PAIR>(buf_free, b6, lane);
              release_tmem_buf<PAIR>(buf_free, b, lane);
            } else {
              spine_last<EPI, EPW>(S, tbase + static_cast<uint32_t>(b5 * BN), tbase + static_cast<uint32_t>(b6 * BN),
                                   tbase + static_cast<uint32_t>(b * BN), chalf);
              tc_fence_before();
              release_tmem_buf<PAIR>(buf_free, b5, lane);
              release_tmem_buf<PAIR>(buf_free, b6, lane);
              release_tmem_buf<PAIR>(buf_free, b, lane);
            }
          }
          if (spill && l == 7) {
            // 16 leaves: the root of leaves [0, 8) waits in shared memory ([column][row]) while
            // the second group runs
#pragma unroll
            for (int j = 0; j < NC; ++j) parked[spine_col<EPI, EPW>(chalf, j) * BM + row_in_tile] = u2f(S[j]);
          }
        }
        if (!ok) break;
        if (spill) {  // the tree's top add: leaves [0, 8) + leaves [8, 16)
#pragma unroll
          for (int j = 0; j < NC; ++j)
            S[j] = f2u(__fadd_rn(parked[spine_col<EPI, EPW>(chalf, j) * BM + row_in_tile], u2f(S[j])));
        }
        // ---- the root of this tile, in S (its TMEM buffers are already free)
        if (EPI == EPI_SWIGLU) {
          // columns [0,64) hold gate, [64,128) up (the second B box came from the up half):
          // g, u = bf16_rn(root); h = bf16_rn(silu(g) * u) with silu(g) = g / (1 + e^-g) in fp32
          // from the fast exp and divide intrinsics (a few fp32 ulps, far below the bf16 rounding
          // of h; the same instructions for every row, tile and schedule).  This warp's h
          // columns: all 64, or with 8 epilogue warps 32 (gate [h0, h0+32), up [64+h0, ...)).
          constexpr int HC = 64 / (EPW / 4);
          static_assert(2 * HC == NC, "S holds this thread's gate columns, then the matching up columns");
          const int h0 = EPW == 8 ? chalf * HC : 0;
          const uint32_t* v = S;
          uint4 hw[HC / 8];
#pragma unroll
          for (int q = 0; q < HC / 8; ++q) {
            float hv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float g = __bfloat162float(__float2bfloat16_rn(u2f(v[q * 8 + i])));
              const float u = __bfloat162float(__float2bfloat16_rn(u2f(v[HC + q * 8 + i])));
              hv[i] = __fmul_rn(__fdividef(g, __fadd_rn(1.0f, __expf(-g))), u);
            }
            hw[q].x = pack_bf16x2(hv[0], hv[1]);
            hw[q].y = pack_bf16x2(hv[2], hv[3]);
            hw[q].z = pack_bf16x2(hv[4], hv[5]);
            hw[q].w = pack_bf16x2(hv[6], hv[7]);
          }
          const bool h_ok = row_ok && ISO_DCHECK(row < p.out_rows, p.status);
          if (p.epi_staged) {
            store_rows_staged<HC / 8>(wstage, lane, hw, h_ok ? row : -1, reinterpret_cast<uint8_t*>(p.out), p.ldo * 2,
                                      2 * static_cast<int64_t>(n0 + h0), 2 * static_cast<int64_t>(n0 + h0 + HC));
          } else if (h_ok) {
            __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(row) * p.ldo;
#pragma unroll
            for (int q = 0; q < HC / 8; ++q) *reinterpret_cast<uint4*>(dst + n0 + h0 + q * 8) = hw[q];
          }
        } else if (EPI == EPI_BF16 || EPI == EPI_F32 || EPI == EPI_CLUSTER) {
          // convert and store this thread's columns of the root: all 128, or with 8 epilogue
          // warps the 64 of its warp's half
          constexpr int RC = NC;
          const int c0 = EPW == 8 ? chalf * RC : 0;
          const uint32_t* v = S;
          if (EPI == EPI_CLUSTER) {
            // the group's subtree root stays in this CTA's shared memory ([column][row], the A
            // box's rows) for the cluster combine after the main loop
            // as column pairs: pair q of row r is the 8-byte word (q a_rows + r), so one warp's
            // rows are consecutive words and a combine thread reads a pair in one load
            if (row_in_tile < p.a_rows && ISO_DCHECK(c0 + RC <= BN, p.status)) {
#pragma unroll
              for (int i = 0; i < RC; i += 2)
                *reinterpret_cast<float2*>(&parked[2 * (((c0 + i) >> 1) * p.a_rows + row_in_tile)]) =
                    make_float2(u2f(v[i]), u2f(v[i + 1]));
            }
          } else if (EPI == EPI_BF16 && p.epi_staged) {
            uint4 w[RC / 8];
#pragma unroll
            for (int q = 0; q < RC / 8; ++q) {
              w[q].x = pack_bf16x2(u2f(v[q * 8 + 0]), u2f(v[q * 8 + 1]));
              w[q].y = pack_bf16x2(u2f(v[q * 8 + 2]), u2f(v[q * 8 + 3]));
              w[q].z = pack_bf16x2(u2f(v[q * 8 + 4]), u2f(v[q * 8 + 5]));
              w[q].w = pack_bf16x2(u2f(v[q * 8 + 6]), u2f(v[q * 8 + 7]));
            }
            int orow = row_ok ? ((EPW == 4 && p.row_scatter != nullptr) ? p.row_scatter[row] : orow_u) : -1;
            if (orow >= 0 && !ISO_DCHECK(orow < p.out_rows, p.status)) orow = -1;
            store_rows_staged<RC / 8>(wstage, lane, w, orow, reinterpret_cast<uint8_t*>(p.out), p.ldo * 2,
                                      2 * static_cast<int64_t>(n0 + c0), 2 * static_cast<int64_t>(p.N));
          } else if (EPI == EPI_F32 && PAIR && p.epi_staged) {
            // fp32 rows of 512 bytes go out in two staged halves of 64 columns (256-byte rows).
            // CTA pairs only: they serve many row blocks, while single CTAs serve one-row-block
            // leaf groups, where most staged rows would be empty (and the staging spilled
            // registers of the single-CTA instance: iso_gemm_ws at M = 64 19.1 -> 21.1 us)
            const int orow = (row_ok && ISO_DCHECK(row < p.out_rows, p.status)) ? row : -1;
            uint8_t* out = reinterpret_cast<uint8_t*>(reinterpret_cast<float*>(p.out) + U.chunk * p.out_group_stride);
#pragma unroll
            for (int hh = 0; hh < RC / 64; ++hh) {
              uint4 w[16];
#pragma unroll
              for (int q = 0; q < 16; ++q)
                w[q] = make_uint4(v[hh * 64 + q * 4 + 0], v[hh * 64 + q * 4 + 1], v[hh * 64 + q * 4 + 2],
                                  v[hh * 64 + q * 4 + 3]);
              store_rows_staged<16>(wstage, lane, w, orow, out, p.ldo * 4, 4 * static_cast<int64_t>(n0 + c0 + hh * 64),
                                    4 * static_cast<int64_t>(p.N));
            }
          } else if (row_ok) {
            if (EPI == EPI_BF16) {
              const int orow = (EPW == 4 && p.row_scatter != nullptr) ? p.row_scatter[row] : orow_u;
              const bool o_ok = ISO_DCHECK(orow >= 0 && orow < p.out_rows, p.status);
              __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(orow) * p.ldo;
#pragma unroll
              for (int q = 0; q < RC / 8; ++q) {
                const int col = n0 + c0 + q * 8;
                if (o_ok && col < p.N) {
                  uint4 w;
                  w.x = pack_bf16x2(u2f(v[q * 8 + 0]), u2f(v[q * 8 + 1]));
                  w.y = pack_bf16x2(u2f(v[q * 8 + 2]), u2f(v[q * 8 + 3]));
                  w.z = pack_bf16x2(u2f(v[q * 8 + 4]), u2f(v[q * 8 + 5]));
                  w.w = pack_bf16x2(u2f(v[q * 8 + 6]), u2f(v[q * 8 + 7]));
                  *reinterpret_cast<uint4*>(dst + col) = w;
                }
              }
            } else {
              float* dst = reinterpret_cast<float*>(p.out) + U.chunk * p.out_group_stride +
                           static_cast<int64_t>(row) * p.ldo;
              const bool o_ok = ISO_DCHECK(row < p.out_rows, p.status);
#pragma unroll
              for (int q = 0; q < RC / 4; ++q) {
                const int col = n0 + c0 + q * 4;
                if (o_ok && col < p.N)
                  *reinterpret_cast<uint4*>(dst + col) = make_uint4(v[q * 4 + 0], v[q * 4 + 1], v[q * 4 + 2], v[q * 4 + 3]);
              }
            }
          }
        } else {
          // tile statistics: m = max over the tile's valid columns (order-free),
          // s = sum over ascending columns of expf(z - m); then the left fold.
          static_assert(EPI != EPI_LOGPROB || NC == BN, "the logprob epilogue holds whole rows of the tile");
          const uint32_t* v = S;
          const int sel_off = sel - n0;
          float m = -INFINITY;
          float s = 0.f;
          if (n0 + BN <= p.V) {
#pragma unroll
            for (int i = 0; i < BN; ++i) m = fmaxf(m, u2f(v[i]));
#pragma unroll
            for (int i = 0; i < BN; ++i) s = __fadd_rn(s, expf(__fsub_rn(u2f(v[i]), m)));
          } else {
#pragma unroll
            for (int i = 0; i < BN; ++i)
              if (n0 + i < p.V) m = fmaxf(m, u2f(v[i]));
#pragma unroll
            for (int i = 0; i < BN; ++i)
              if (n0 + i < p.V) s = __fadd_rn(s, expf(__fsub_rn(u2f(v[i]), m)));
            if (n0 >= p.V) {
              m = -INFINITY;
              s = 0.f;
            }
          }
          if (sel_off >= 0 && sel_off < BN) {
#pragma unroll
            for (int i = 0; i < BN; ++i)
              if (i == sel_off) zsel = u2f(v[i]);
            have_sel = true;
          }
          if (t == 0) {
            run_m = m;
            run_s = s;
          } else {
            lse_merge(run_m, run_s, m, s);
          }
        }
      }
      if (EPI == EPI_LOGPROB && ok && row_ok && ISO_DCHECK(U.chunk < p.num_chunks && row < p.M, p.status)) {
        p.ws_stats[static_cast<int64_t>(U.chunk) * p.M + row] = make_float2(run_m, run_s);
        if (have_sel) p.ws_zsel[row] = zsel;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (EPI == EPI_CLUSTER) {
    // Every CTA of the cluster has its group root in shared memory (the barrier's release /
    // acquire orders those stores before the peers' loads).  This CTA (rank r) combines columns
    // [r BN/R, (r+1) BN/R) of the tile: for each (row, column pair) the R group roots in group
    // order, the balanced tree over them (left operand = lower group, fp32 rn adds: the top
    // log2 R levels of the contract's tree), one bf16 rounding.  The second barrier keeps every
    // CTA's shared memory alive until the peers are done reading it.  Each CTA reaches both
    // barriers whatever happened before, so an aborted CTA cannot leave its peers waiting.
    cluster_sync_all();
    if (unit0 < nunits) {
      Unit U;
      decode_unit(p, unit0, U, 1, 0);
      const int R = p.cluster;
      const int cols = BN / R;
      const int npairs = cols / 2;
      const int c_base = static_cast<int>(cluster_ctarank()) * cols;  // first column of this CTA's slice
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
      const int total = U.rows_valid * npairs;
      // four (row, column pair) elements per thread per pass: every group's load of all four is
      // issued before the first is used, so a pass costs one round trip to the peers
      constexpr int EB = 4;
      for (int e0 = threadIdx.x; e0 < total; e0 += EB * static_cast<int>(blockDim.x)) {
        float2 x[EB][MAX_CLUSTER_GROUPS];
#pragma unroll
        for (int q = 0; q < EB; ++q) {
          const int e = e0 + q * static_cast<int>(blockDim.x);
          if (e < total) {
            const int row = e / npairs;
            const int pr = (c_base >> 1) + (e - row * npairs);  // column pair within the tile
            if (!ISO_DCHECK(row < p.a_rows && pr < BN / 2, p.status)) continue;
#pragma unroll
            for (int g = 0; g < MAX_CLUSTER_GROUPS; ++g)
              if (g < R)
                x[q][g] = ld_cluster_f32x2(cluster_addr(&parked[2 * (pr * p.a_rows + row)], static_cast<uint32_t>(g)));
          }
        }
#pragma unroll
        for (int q = 0; q < EB; ++q) {
          const int e = e0 + q * static_cast<int>(blockDim.x);
          if (e >= total) continue;
          const int row = e / npairs;
          const int col = U.n_tile0 * BN + c_base + 2 * (e - row * npairs);
          if (col >= p.N || !ISO_DCHECK(row < p.out_rows && row < p.a_rows, p.status)) continue;
          // balanced tree over the groups, left operand = lower group (fp32 rn adds)
#pragma unroll
          for (int w = 1; w < MAX_CLUSTER_GROUPS; w *= 2) {
#pragma unroll
            for (int g = 0; g + w < MAX_CLUSTER_GROUPS; g += 2 * w) {
              if (g + w < R) {
                x[q][g].x = __fadd_rn(x[q][g].x, x[q][g + w].x);
                x[q][g].y = __fadd_rn(x[q][g].y, x[q][g + w].y);
              }
            }
          }
          *reinterpret_cast<uint32_t*>(out + static_cast<int64_t>(row) * p.ldo + col) = pack_bf16x2(x[q][0].x, x[q][0].y);
        }
      }
    }
    cluster_sync_all();
  }
  if (PAIR) {
    // After an abort the peer's last loads may still be landing in this CTA's shared memory
    // (their completion is counted on rank 0, which may have stopped waiting): give them time.
    if (*abort_flag) {
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 2000000ull) {
      }
    }
    cluster_sync_all();  // neither CTA leaves while the other may still touch its memory
  }
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else
      tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

namespace {

template <int EPI, bool PAIR, bool FUSED = false, int EPW = 4, bool LS = false>
iso_status launch_one(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int max_units,
                      cudaStream_t s, const CUtensorMap& tmA2) {
  constexpr int kThreads = FUSED ? GEMM_THREADS_FUSED : (EPW == 8 ? GEMM_THREADS_EPI8 : GEMM_THREADS);
  // Per device, once: the function attributes, and the CTAs (pairs: clusters) resident at once.
  // 0 = not yet; threads that get there together repeat the same idempotent setup.
  static std::atomic<int> slots_by_dev[ISO_MAX_DEVICES] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= ISO_MAX_DEVICES) return ISO_ERR_CUDA;
  auto kern = iso_leaf_tree_gemm_kernel<EPI, PAIR, FUSED, EPW, LS>;
  int slots = slots_by_dev[dev].load(std::memory_order_acquire);
  if (slots == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM_BYTES) != cudaSuccess)
      return ISO_ERR_CUDA;
    slots = sm_count();
    if (PAIR) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0) != cudaSuccess)
        return ISO_ERR_CUDA;
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = 2;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(static_cast<unsigned>(2 * (sm_count() / 2)));
      cfg.blockDim = dim3(GEMM_THREADS);
      cfg.dynamicSmemBytes = GEMM_SMEM_BYTES;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters <= 0) return ISO_ERR_CUDA;
      slots = clusters;
    }
    slots_by_dev[dev].store(slots, std::memory_order_release);
    const char* tr = getenv("ISO_TRACE");
    if (tr && tr[0] == '1')
      fprintf(stderr, "[iso] gemm kernel epi=%d pair=%d epilogue warps=%d: %d %s resident\n", EPI, PAIR ? 1 : 0,
              EPW, slots, PAIR ? "CTA pairs" : "CTAs");
  }
  if constexpr (EPI == EPI_CLUSTER) {
    // one CTA per unit, in clusters of p.cluster (the host checked that they fit at once)
    if (max_units <= 0 || max_units % p.cluster != 0) return ISO_ERR_INVALID_ARG;
    if (launch_dependent(kern, dim3(static_cast<unsigned>(max_units)), dim3(kThreads), GEMM_SMEM_BYTES, s,
                         static_cast<unsigned>(p.cluster), tmA, tmB, tmA2, p) != cudaSuccess)
      return ISO_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? ISO_OK : ISO_ERR_CUDA;
  }
  const int units = max_units < slots ? max_units : slots;
  if (units <= 0) return ISO_OK;
  if (launch_dependent(kern, dim3(static_cast<unsigned>(PAIR ? 2 * units : units)), dim3(kThreads), GEMM_SMEM_BYTES,
                       s, PAIR ? 2u : 1u, tmA, tmB, tmA2, p) != cudaSuccess)
    return ISO_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? ISO_OK : ISO_ERR_CUDA;
}

}  // namespace

int cluster_gemm_capacity(int R) {
  static std::mutex mu;
  static int cached_dev = -1;
  static int cap[MAX_CLUSTER_GROUPS + 1] = {};
  int dev = 0;
  if (R < 2 || R > MAX_CLUSTER_GROUPS || cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (cached_dev != dev) {
    auto kern = iso_leaf_tree_gemm_kernel<EPI_CLUSTER, false, false, 4, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM_BYTES) != cudaSuccess)
      return 0;
    for (int r = 2; r <= MAX_CLUSTER_GROUPS; r *= 2) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = static_cast<unsigned>(r);
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(static_cast<unsigned>(r * (sm_count() / r)));
      cfg.blockDim = dim3(GEMM_THREADS);
      cfg.dynamicSmemBytes = GEMM_SMEM_BYTES;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      int n = 0;
      cap[r] = cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess ? n : 0;
    }
    cached_dev = dev;
  }
  return cap[R];
}

iso_status launch_gemm(int epi, const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int max_units,
                       cudaStream_t s, const CUtensorMap* tmA2) {
  const CUtensorMap& a2 = tmA2 != nullptr ? *tmA2 : tmA;  // unused unless p.leaf_stage
  if (p.leaf_stage) {
    if (epi != EPI_BF16 || p.pair || p.a_transform || tmA2 == nullptr || p.leaf_len != LS_LEAF || p.spill)
      return ISO_ERR_INVALID_ARG;
    return launch_one<EPI_BF16, false, false, 8, true>(tmA, tmB, p, max_units, s, a2);
  }
  const bool pair = p.pair != 0;
  // CTA pairs serve row-block units; deep stages read A through the 3-D chunk view (one leaf
  // starting at k = 0, a whole number of 64-k chunks)
  if (p.stage_k != (pair ? p.stage_k : BK) || (p.stage_k != BK && p.stage_k != PAIR_BK) ||
      p.kb_per_leaf != (p.leaf_len + p.stage_k - 1) / p.stage_k)
    return ISO_ERR_INVALID_ARG;
  if (pair && ((p.unit_mode != UNIT_GEMM && p.unit_mode != UNIT_LOGPROB) ||
               (p.stage_k == PAIR_BK && (p.L != 1 || p.leaf_len % 64 != 0))))
    return ISO_ERR_INVALID_ARG;
  if (p.a_transform) {
    if (pair) return ISO_ERR_INVALID_ARG;
    if (epi == EPI_BF16) return launch_one<EPI_BF16, false, true>(tmA, tmB, p, max_units, s, a2);
    if (epi == EPI_LOGPROB) return launch_one<EPI_LOGPROB, false, true>(tmA, tmB, p, max_units, s, a2);
    return ISO_ERR_INVALID_ARG;
  }
  // short leaves: 8 epilogue warps (the expert layer's grouped GEMMs: 1.07 -> 0.94 ms per layer)
  switch (epi) {
    case EPI_BF16:
      if (!pair && !p.spill && p.leaf_len <= EPI8_MAX_LEAF_BF16)
        return launch_one<EPI_BF16, false, false, 8>(tmA, tmB, p, max_units, s, a2);
      return pair ? launch_one<EPI_BF16, true>(tmA, tmB, p, max_units, s, a2)
                  : launch_one<EPI_BF16, false>(tmA, tmB, p, max_units, s, a2);
    case EPI_F32:
      return pair ? launch_one<EPI_F32, true>(tmA, tmB, p, max_units, s, a2)
                  : launch_one<EPI_F32, false>(tmA, tmB, p, max_units, s, a2);
    case EPI_SWIGLU:
      if (!pair && !p.spill && p.leaf_len <= EPI8_MAX_LEAF_SWIGLU)
        return launch_one<EPI_SWIGLU, false, false, 8>(tmA, tmB, p, max_units, s, a2);
      if (pair) return ISO_ERR_INVALID_ARG;
      return launch_one<EPI_SWIGLU, false>(tmA, tmB, p, max_units, s, a2);
    case EPI_LOGPROB:
      return pair ? launch_one<EPI_LOGPROB, true>(tmA, tmB, p, max_units, s, a2)
                  : launch_one<EPI_LOGPROB, false>(tmA, tmB, p, max_units, s, a2);
    case EPI_CLUSTER:
      if (pair || p.cluster < 2 || p.cluster > MAX_CLUSTER_GROUPS) return ISO_ERR_INVALID_ARG;
      return launch_one<EPI_CLUSTER, false>(tmA, tmB, p, max_units, s, a2);
    default:
      return ISO_ERR_INVALID_ARG;
  }
}

}  // namespace iso
