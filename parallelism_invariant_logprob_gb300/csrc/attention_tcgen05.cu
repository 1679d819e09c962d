// attention_tcgen05.cu -- causal attention with a fixed KV-chunk merge, on 5th-generation
// tensor cores (batch- and position-invariant: prefill and decode give the same bits).
//
// What it computes [RL-Kernel blog, §4 "Focus: The Shared Dependency of Attention and Linear
// LogP on LogSumExp": softmax over the visible keys, the LSE statistic; §6 table row 03 and §7
// "Attention": no KV split, fixed block partitioning, chunk order and rescale-merge order;
// VeXact paper §3.1: KV splitting disabled]: for query row r of sequence b at position p and
// query head h (KV head h / (Hq / Hkv)), over the keys k_start[b] .. k_start[b] + p,
//   out = softmax(scale * q . k) V  (bf16),  lse = m + log l  (fp32).
//
// The merge is the online softmax over fixed 128-key chunks in ascending order, one thread per
// row, in the base-2 domain (c2 = rn(scale * log2 e)).  For chunk c, with S = q . k from a
// chain of 8 tcgen05 MMAs (K = 16 each, ascending dims) and S_j = -inf for keys past p:
//   t    = rn(max_j S_j * c2)                           (max is exact in any order)
//   m'   = max(m, t) if chunk 0 or t > m + 8, else m    (lazy: P stays below 2^8)
//   P_j  = ex2(fma(S_j, c2, -m'));  l_c = (sum of four interleaved partial sums, fixed order)
//   a    = ex2(m - m') (1 when m' = m);  l = rn(rn(l * a) + l_c);  O = rn(O * a) when a != 1
//   O   += bf16(P) V   (8 tcgen05 MMAs, K = 16 keys each, ascending keys)
// and at the end out = bf16_rn(O * rcp(l)), lse = rn(rn(m ln 2) + logf(l)).  Every step
// depends only on the row, its position and the chunk grid, never on the other rows of its
// tile or the launch, so a decode call (one row) reproduces the row of a prefill call exactly.
// A chunk wholly past a row's position changes nothing in that row: t = -inf, a = 1, P = 0,
// O + 0 = O.
//
// Structure: one CTA per (query head, sequence, pair of 128-row query tiles A and B), the
// pairs with the most chunks first; 384 threads (3 warpgroups, registers rebalanced at entry).
//   warps 0-3  softmax of tile A, warps 4-7 softmax of tile B: one thread per query row
//              (TMEM lane); each also rescales its O rows and writes the output
//   warp 8     TMA producer: Q of both tiles once, then K and V chunks into a 2-stage ring
//   warp 9     MMA issuer (lane 0) and TMEM owner (warps 10, 11 only fill the warpgroup).  Per chunk j it issues, in this order,
//              PV_A(j), S_A(j+1), PV_B(j), S_B(j+1): while the softmax of one tile runs, the
//              tensor core works for the other.
// TMEM (512 columns): S_A, S_B (128 fp32 columns each), O_A, O_B.  The softmax writes P as
// packed bf16 pairs over the first 64 columns of its own S buffer, and the P V MMA reads A
// from there.  tcgen05 MMAs execute in issue order, so PV_t(j) has read P_t(j) before
// S_t(j+1) overwrites it, and the commit after S_t(j+1) also covers PV_t(j): the softmax
// may rescale O_t as soon as it sees S_t(j+1).  Shared memory: Q 2 x 32 KB, K and V 2 stages
// x 32 KB each.  Every wait is bounded (abort flag, device status word).
#include <cuda_bf16.h>
#include <stdio.h>

#include "iso_internal.h"
#include "iso_ptx.cuh"

namespace iso {

namespace {

constexpr int AT_ROWS = 128;    // query rows per tile (the MMA's M)
constexpr int AT_KEYS = 128;    // keys per chunk (N of QK^T, K of PV)
constexpr int AT_D = 128;       // head dimension
constexpr int AT_THREADS = 384;  // 3 warpgroups
// Register split (setmaxnreg): launched at 168 per thread (384 x 168 = 64,512), the two softmax
// warpgroups take 216 and the producer / MMA warpgroup keeps 72: 2 x 128 x 216 + 128 x 72 =
// 64,512, exactly the launch's total, so the increase always finds its registers.
constexpr int AT_REGS_SOFTMAX = 216;
constexpr int AT_REGS_CONTROL = 72;
static_assert(2 * 128 * AT_REGS_SOFTMAX + 128 * AT_REGS_CONTROL <= AT_THREADS * 168, "register split");
constexpr int AT_TILE_BYTES = AT_ROWS * AT_D * 2;  // 32 KB: one 128 x 128 bf16 operand tile
constexpr int AT_SMEM = 1024 /*align*/ + 6 * AT_TILE_BYTES + 256 /*barriers*/;
constexpr int AT_WARP_PRODUCER = 8;
constexpr int AT_WARP_MMA = 9;

struct AttnParams {
  const int32_t* q_start;  // [B+1]
  const int32_t* k_start;  // [B+1]
  const int32_t* pos0;     // [B]
  int B, Hq, Hkv;
  float scale_log2e;  // scale * log2(e), rounded to fp32
  __nv_bfloat16* out;  // [Tq x Hq x d]
  float* lse;          // [Tq x Hq]
  unsigned int* status;
  uint64_t timeout_ns;
};

// S = Q K^T: A (Q) and B (K) both K-major in shared memory.  O += P V: A (P) K-major in
// tensor memory, B (V) MN-major in shared memory.
constexpr uint32_t kIdescS = idesc_bf16_f32(AT_ROWS, AT_KEYS, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(AT_ROWS, AT_D, false, true);

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);  // .x (low half) = lo
  return *reinterpret_cast<const uint32_t*>(&t);
}
// 2^x by the PTX instruction ex2.approx.ftz.f32 (one MUFU op; results below 2^-126 flush to 0)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// three-input maximum (PTX max.f32 with three sources)
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
constexpr float kLazy = 8.0f;  // base-2 headroom before the running maximum moves
constexpr float kLn2 = 0.693147180559945309f;

// D[tmem] (+)= A[tmem] * B[smem desc], kind::f16.  A: 128 lanes (rows) x K, two bf16 per
// 32-bit column in K order.
__device__ __forceinline__ void umma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

template <int R>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
}
template <int R>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
}

// Bounded wait on the phase of `bar` with the given parity, polled by every lane of the
// warp; the outcome is made warp-uniform so the warp reaches each later .sync.aligned
// tcgen05 op converged.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const AttnParams& p,
                                          volatile int* abort_flag) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, p.timeout_ns, abort_flag, p.status));
}

__global__ void __launch_bounds__(AT_THREADS, 1)
    iso_attention_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  // grid (Hq, B, tile pairs): the pairs furthest into their sequences (the most chunks) start first
  const int h = blockIdx.x, b = blockIdx.y, pair = gridDim.z - 1 - blockIdx.z;
  const int q0 = p.q_start[b], nq = p.q_start[b + 1] - q0;
  // shape checks, uniform over the CTA and taken before any barrier or TMEM use: the grid
  // must cover every query row, and the last row's keys must lie inside the sequence
  if (threadIdx.x == 0 && h == 0 && pair == static_cast<int>(gridDim.z) - 1 &&
      (nq > static_cast<int>(gridDim.z) * 2 * AT_ROWS || nq < 0 || p.pos0[b] < 0 ||
       p.k_start[b] + p.pos0[b] + nq > p.k_start[b + 1]))
    atomicOr(p.status, kDevBadShape);
  if (nq <= 0 || p.pos0[b] < 0 || p.k_start[b] + p.pos0[b] + nq > p.k_start[b + 1]) return;
  const int tileA = 2 * pair;
  if (tileA * AT_ROWS >= nq) return;  // empty unit
  // per tile (A, B): valid rows, position of row 0, chunks its last row sees
  const int rows_a = min(AT_ROWS, nq - tileA * AT_ROWS);
  const int rows_b = max(0, min(AT_ROWS, nq - (tileA + 1) * AT_ROWS));
  const int pos_a = p.pos0[b] + tileA * AT_ROWS;
  const int chunks_a = (pos_a + rows_a - 1) / AT_KEYS + 1;
  const int chunks_b = rows_b > 0 ? (pos_a + AT_ROWS + rows_b - 1) / AT_KEYS + 1 : 0;
  const int n_all = max(chunks_a, chunks_b);
  const int g = h / (p.Hq / p.Hkv);
  const int kbase = p.k_start[b];

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                       // 2 tiles
  uint8_t* sK = smem + 2 * AT_TILE_BYTES;   // 2 stages
  uint8_t* sV = smem + 4 * AT_TILE_BYTES;   // 2 stages
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 6 * AT_TILE_BYTES);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;   // [2 stages]
  uint64_t* kv_empty = bars + 3;  // [2 stages]
  uint64_t* s_full = bars + 5;    // [2 tiles]
  uint64_t* p_full = bars + 7;    // [2 tiles]
  uint64_t* mma_done = bars + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 10);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], AT_ROWS);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == AT_WARP_MMA) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // S_t at columns [128 t, 128 t + 128) (P_t over its first 64), O_t at [256 + 128 t, ...)

  if (warp >= 8) {
    // the control warpgroup (producer, MMA, two idle warps) hands registers to the softmax
    regs_dec<AT_REGS_CONTROL>();
  }
  if (warp == AT_WARP_PRODUCER) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int issued = 0;
      const int n_q_tiles = chunks_b > 0 ? 2 : 1;
      mbar_arrive_expect_tx(q_full, n_q_tiles * AT_TILE_BYTES);
      for (int t = 0; t < n_q_tiles; ++t)
        for (int kb = 0; kb < 2; ++kb)
          tma_load_2d(sQ + t * AT_TILE_BYTES + kb * (AT_TILE_BYTES / 2), &tmQ, q_full, h * AT_D + kb * 64,
                      q0 + (tileA + t) * AT_ROWS);
      for (int c = 0; c < n_all; ++c) {
        const int s = c & 1;
        if (c >= 2 && !mbar_wait(&kv_empty[s], ((c >> 1) - 1) & 1, p.timeout_ns, abort_flag, p.status)) break;
        const int krow = kbase + c * AT_KEYS;
        mbar_arrive_expect_tx(&kv_full[s], 2 * AT_TILE_BYTES);
        uint8_t* k_dst = sK + s * AT_TILE_BYTES;
        uint8_t* v_dst = sV + s * AT_TILE_BYTES;
        // K: two 64-dim boxes of 128 keys (K-major B of Q K^T)
        for (int kb = 0; kb < 2; ++kb)
          tma_load_2d(k_dst + kb * (AT_TILE_BYTES / 2), &tmK, &kv_full[s], g * AT_D + kb * 64, krow);
        // V: per 64-key block, two 64-dim boxes (MN-major B of P V)
        for (int kb = 0; kb < 2; ++kb)
          for (int half = 0; half < 2; ++half)
            tma_load_2d(v_dst + kb * (AT_TILE_BYTES / 2) + half * (AT_TILE_BYTES / 4), &tmV, &kv_full[s],
                        g * AT_D + half * 64, krow + kb * 64);
        issued = c + 1;
      }
      // before the CTA may exit: every load this thread issued has landed (bounded; normally
      // the MMA has consumed them all and these phases are long complete)
      const uint64_t t0 = globaltimer_ns();
      bool landed = false;
      while (!landed && globaltimer_ns() - t0 <= p.timeout_ns) {
        landed = mbar_try_wait(smem_u32(q_full), 0);
        for (int c = (issued > 2 ? issued - 2 : 0); c < issued && landed; ++c)
          landed = mbar_try_wait(smem_u32(&kv_full[c & 1]), (c >> 1) & 1);
      }
      if (!landed) {
        *abort_flag = 1;
        atomicOr(p.status, kDevTimeout);
      }
    }
  } else if (warp == AT_WARP_MMA) {
    // --------------------------------------------------------------------- MMA
    const bool leader = (lane == 0);
    const uint64_t kdesc0 = sdesc_sw128(0, 16, 1024);    // K-major operand template
    const uint64_t vdesc0 = sdesc_sw128(0, 8192, 1024);  // MN-major operand template
    // S_t(c) = Q_t K_c^T into S_t's columns; K from stage c & 1 (already waited for)
    auto issue_s = [&](int t, int c) {
      if (leader) {
        const uint32_t q_lo = smem_u32(sQ + t * AT_TILE_BYTES) >> 4;
        const uint32_t k_lo = smem_u32(sK + (c & 1) * AT_TILE_BYTES) >> 4;
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
#pragma unroll
          for (int k16 = 0; k16 < 4; ++k16) {
            const uint64_t ad = kdesc0 + q_lo + kb * (AT_TILE_BYTES / 2 / 16) + k16 * 2;
            const uint64_t bd = kdesc0 + k_lo + kb * (AT_TILE_BYTES / 2 / 16) + k16 * 2;
            umma_bf16(tmem + t * 128, ad, bd, kIdescS, (kb | k16) != 0 ? 1u : 0u);
          }
        umma_commit(&s_full[t]);
      }
      __syncwarp();
    };
    // O_t += P_t(c) V_c; P_t from the first 64 columns of S_t, V from stage c & 1
    auto issue_pv = [&](int t, int c) {
      if (leader) {
        const uint32_t v_lo = smem_u32(sV + (c & 1) * AT_TILE_BYTES) >> 4;
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
#pragma unroll
          for (int k16 = 0; k16 < 4; ++k16) {
            const uint64_t bd = vdesc0 + v_lo + kb * (AT_TILE_BYTES / 2 / 16) + k16 * 128;
            umma_bf16_tmem_a(tmem + 256 + t * 128, tmem + t * 128 + (kb * 4 + k16) * 8, bd, kIdescPV,
                             (c | kb | k16) != 0 ? 1u : 0u);
          }
      }
      __syncwarp();
    };
    bool ok = warp_wait(q_full, 0, p, abort_flag) && warp_wait(&kv_full[0], 0, p, abort_flag);
    if (ok) {
      tc_fence_after();
      issue_s(0, 0);
      if (chunks_b > 0) issue_s(1, 0);
    }
    for (int c = 0; c < n_all && ok; ++c) {
      for (int t = 0; t < 2 && ok; ++t) {
        const int nct = t ? chunks_b : chunks_a;
        if (c >= nct) continue;
        ok = warp_wait(&p_full[t], c & 1, p, abort_flag);
        if (!ok) break;
        tc_fence_after();
        issue_pv(t, c);
        if (c + 1 < nct) {
          ok = warp_wait(&kv_full[(c + 1) & 1], ((c + 1) >> 1) & 1, p, abort_flag);
          if (!ok) break;
          tc_fence_after();
          issue_s(t, c + 1);
        }
      }
      if (leader) umma_commit(&kv_empty[c & 1]);  // every MMA reading stage c & 1 is issued
      __syncwarp();
    }
    if (leader) umma_commit(mma_done);
    __syncwarp();
    // drain: the CTA exits only after its MMAs completed
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(mma_done), 0)) {
      if (globaltimer_ns() - t0 > p.timeout_ns) {
        *abort_flag = 1;
        atomicOr(p.status, kDevTimeout);
        break;
      }
    }
  } else if (warp < 8) {
    // ----------------------------------------------------- softmax / correction
    regs_inc<AT_REGS_SOFTMAX>();
    // Scores are handled in the base-2 domain: t_j = S_j * scale * log2(e) (one FMA with the
    // running maximum), P_j = 2^(t_j - m), and lse = m ln 2 + ln l at the end.  The running
    // maximum m moves only when a chunk's maximum exceeds it by more than kLazy (2^kLazy
    // bounds P and the sums stay far from overflow); then O and l are rescaled by 2^(m_old - m).
    const int t = warp >> 2;       // 0: tile A, 1: tile B
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + t * 128 + lane_off;
    const uint32_t tO = tmem + 256 + t * 128 + lane_off;
    const int nc = t ? chunks_b : chunks_a;
    const int rows_valid = t ? rows_b : rows_a;
    const int pos = pos_a + t * AT_ROWS + r;  // this row's position (rows past rows_valid compute unused values)
    const int warp_pos_min = pos_a + t * AT_ROWS + quarter * 32;
    const float c2 = p.scale_log2e;
    float m = -INFINITY, l = 0.f;
    bool ok = nc > 0;
    for (int c = 0; c < nc && ok; ++c) {
      // S_t(c) complete; for c > 0 so is P V of chunk c - 1 (issued before it)
      ok = warp_wait(&s_full[t], c & 1, p, abort_flag);
      if (!ok) break;
      tc_fence_after();
      uint32_t v[AT_KEYS];
#pragma unroll
      for (int q = 0; q < AT_KEYS / 32; ++q) tmem_ld32p(tS + q * 32, v + q * 32);
      tmem_ld_wait_only();
#pragma unroll
      for (int q = 0; q < AT_KEYS / 32; ++q) tmem_ld_tie(v + q * 32);
      const int kpos0 = c * AT_KEYS;
      if (kpos0 + AT_KEYS - 1 > warp_pos_min) {  // a key of this chunk is past some row of the warp
#pragma unroll
        for (int j = 0; j < AT_KEYS; ++j)
          if (kpos0 + j > pos) v[j] = f2u(-INFINITY);
      }
      // chunk maximum of the raw scores (max is exact, so the tree's shape cannot matter)
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = fmaxf(u2f(v[i]), u2f(v[i + 8]));
#pragma unroll
      for (int j = 16; j < AT_KEYS; j += 16)  // keys j .. j + 15, j + 15 <= 127
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = max3(mx[i], u2f(v[j + i]), u2f(v[j + 8 + i]));
      const float mc = __fmul_rn(max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])), c2);
      const float m_new = (m == -INFINITY || mc > m + kLazy) ? fmaxf(m, mc) : m;
      const float alpha = (m == -INFINITY) ? 1.f : ex2(__fsub_rn(m, m_new));  // 1 when m stays
      m = m_new;
      const float neg_m = -m;
      // P_j = 2^(t_j - m), packed to bf16 pairs in place; the chunk sum in four interleaved
      // partial sums, combined in a fixed order
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < AT_KEYS; j += 2) {
        const float e0 = ex2(__fmaf_rn(u2f(v[j]), c2, neg_m));
        const float e1 = ex2(__fmaf_rn(u2f(v[j + 1]), c2, neg_m));
        ls[j & 3] = __fadd_rn(ls[j & 3], e0);
        ls[(j + 1) & 3] = __fadd_rn(ls[(j + 1) & 3], e1);
        v[j >> 1] = pack_bf16x2(e0, e1);
      }
      l = __fadd_rn(__fmul_rn(l, alpha), __fadd_rn(__fadd_rn(ls[0], ls[1]), __fadd_rn(ls[2], ls[3])));
      // the rescale is taken by the whole warp when any of its rows needs it (x * 1 = x
      // exactly, so a row whose maximum did not move keeps its bits)
      if (c > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int q = 0; q < AT_D / 32; ++q) {
          uint32_t o[32];
          tmem_ld32p(tO + q * 32, o);
          tmem_ld_wait_only();
          tmem_ld_tie(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = f2u(__fmul_rn(u2f(o[i]), alpha));
          tmem_st32p(tO + q * 32, o);
        }
      }
      // P over the first 64 columns of S_t: column k holds keys 2k (low half) and 2k + 1
      tmem_st32p(tS, v);
      tmem_st32p(tS + 32, v + 32);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[t]);
    }
    if (ok) ok = warp_wait(mma_done, 0, p, abort_flag);
    if (ok) {
      tc_fence_after();
      uint32_t o[AT_D];
#pragma unroll
      for (int q = 0; q < AT_D / 32; ++q) tmem_ld32p(tO + q * 32, o + q * 32);
      tmem_ld_wait_only();
#pragma unroll
      for (int q = 0; q < AT_D / 32; ++q) tmem_ld_tie(o + q * 32);
      if (r < rows_valid) {
        const int64_t row = q0 + (tileA + t) * AT_ROWS + r;
        __nv_bfloat16* dst = p.out + (row * p.Hq + h) * AT_D;
        const float inv_l = __frcp_rn(l);
#pragma unroll
        for (int q = 0; q < AT_D / 8; ++q) {
          uint4 w;
          w.x = pack_bf16x2(__fmul_rn(u2f(o[q * 8 + 0]), inv_l), __fmul_rn(u2f(o[q * 8 + 1]), inv_l));
          w.y = pack_bf16x2(__fmul_rn(u2f(o[q * 8 + 2]), inv_l), __fmul_rn(u2f(o[q * 8 + 3]), inv_l));
          w.z = pack_bf16x2(__fmul_rn(u2f(o[q * 8 + 4]), inv_l), __fmul_rn(u2f(o[q * 8 + 5]), inv_l));
          w.w = pack_bf16x2(__fmul_rn(u2f(o[q * 8 + 6]), inv_l), __fmul_rn(u2f(o[q * 8 + 7]), inv_l));
          *reinterpret_cast<uint4*>(dst + q * 8) = w;
        }
        if (p.lse) p.lse[row * p.Hq + h] = __fadd_rn(__fmul_rn(m, kLn2), logf(l));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == AT_WARP_MMA) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

}  // namespace iso

using namespace iso;

extern "C" iso_status iso_attention(const iso_contract* c, const iso_bf16* Q, const iso_bf16* K, const iso_bf16* V,
                                    const int32_t* q_start, const int32_t* k_start, const int32_t* pos0, int B,
                                    int Tq, int Tk, int Hq, int Hkv, int d, int max_q_rows, float scale,
                                    iso_bf16* out, float* lse, iso_stream stream) {
  if (!c || B < 0 || Tq < 0 || Tk < 0 || Hq <= 0 || Hkv <= 0 || max_q_rows < 0) return ISO_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ISO_ERR_SHAPE;
  if (d != AT_D) return ISO_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || !(scale < INFINITY)) return ISO_ERR_INVALID_ARG;
  if (B == 0 || Tq == 0 || max_q_rows == 0) return ISO_OK;
  if (!Q || !K || !V || !q_start || !k_start || !pos0 || !out) return ISO_ERR_INVALID_ARG;
  if (Tk == 0) return ISO_ERR_SHAPE;  // a query row sees at least one key
  const int pairs = ((max_q_rows + AT_ROWS - 1) / AT_ROWS + 1) / 2;
  if (B > 65535 || pairs > 65535) return ISO_ERR_UNSUPPORTED;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) |
                        reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(out);
  if (mis & 15u) return ISO_ERR_ALIGNMENT;
  if (!device_ready()) return ISO_ERR_CUDA;
  CUtensorMap tQ, tK, tV;
  iso_status st = make_tmap_bf16(&tQ, Q, Tq, static_cast<uint64_t>(Hq) * d, static_cast<uint64_t>(Hq) * d, 64, AT_ROWS);
  if (st == ISO_OK)
    st = make_tmap_bf16(&tK, K, Tk, static_cast<uint64_t>(Hkv) * d, static_cast<uint64_t>(Hkv) * d, 64, AT_KEYS);
  if (st == ISO_OK)
    st = make_tmap_bf16(&tV, V, Tk, static_cast<uint64_t>(Hkv) * d, static_cast<uint64_t>(Hkv) * d, 64, 64);
  if (st != ISO_OK) return st;
  AttnParams p;
  p.q_start = q_start;
  p.k_start = k_start;
  p.pos0 = pos0;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.scale_log2e = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.status = device_status_ptr();
  p.timeout_ns = wait_timeout_ns();
  static int attr_dev = -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ISO_ERR_CUDA;
  if (attr_dev != dev) {
    if (cudaFuncSetAttribute(iso_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AT_SMEM) !=
        cudaSuccess)
      return ISO_ERR_CUDA;
    attr_dev = dev;
  }
  const dim3 grid(Hq, B, pairs);
  iso_attention_kernel<<<grid, AT_THREADS, AT_SMEM, static_cast<cudaStream_t>(stream)>>>(tQ, tK, tV, p);
  return cudaGetLastError() == cudaSuccess ? ISO_OK : ISO_ERR_CUDA;
}
