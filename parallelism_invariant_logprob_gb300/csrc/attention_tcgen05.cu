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
// The merge is the online softmax over fixed 80-key chunks (keys [80 c, 80 c + 80) of the
// sequence) in ascending order, one thread per row, in the base-2 domain
// (c2 = rn(scale * log2 e)).  For chunk c, with S = q . k from a chain of 8 tcgen05 MMAs
// (K = 16 each, ascending dims) and S_j = -inf for keys past p:
//   t    = rn(max_j S_j * c2)                           (max is exact in any order)
//   m'   = max(m, t) if chunk 0 or t > m + 8, else m    (lazy: P stays below 2^8)
//   P_j  = ex2(fma(S_j, c2, -m'));  l_c = (sum of four interleaved partial sums, fixed order)
//   a    = ex2(m - m') (1 when m' = m);  l = rn(rn(l * a) + l_c);  O = rn(O * a) when a != 1
//   O   += bf16(P) V   (5 tcgen05 MMAs, K = 16 keys each, ascending keys)
// and at the end out = bf16_rn(O * rcp(l)), lse = rn(rn(m ln 2) + logf(l)).  Every step
// depends only on the row, its position and the chunk grid, never on the other rows of its
// tile or the launch, so a decode call (one row) reproduces the row of a prefill call exactly.
// A chunk wholly past a row's position changes nothing in that row: t = -inf, a = 1, P = 0,
// O + 0 = O.
//
// Structure: one CTA per (query-head group, sequence, pair of 128-row query tiles A and B), the
// pairs with the most chunks first; 512 threads (4 warpgroups, registers rebalanced at entry).
// A tile row is one (token, query head) pair: tiles hold 128 / G tokens x the G = Hq / Hkv heads
// that share a KV head (when G divides 128), so one K / V stream serves all of them.
//   warps 0-3  softmax of tile A, warps 4-7 softmax of tile B: one thread per query row
//              (TMEM lane); each also rescales its O rows and writes the output
//   warp 8     TMA producer: Q of both tiles once, then K and V chunks into a 4-stage ring
//   warps 9-12 MMA issuers, one lane each: Q K^T of tile A, P V of tile A, Q K^T of tile B,
//              P V of tile B.  The four chains depend on each other only through the softmax,
//              so each has its own thread: a tile's Q K^T for the next chunk goes out while
//              the other tile's P V is still being issued.  Warp 9 owns TMEM; warps 13-15 idle.
// TMEM (512 columns): per tile t at 256 t: S (80 fp32 columns), P (40 columns of bf16 pairs, its
// own region) and O (128 columns at 256 t + 128).  P apart from S lets Q K^T of chunk c + 1 run
// as soon as the softmax has read S of chunk c, overlapping the softmax and P V of chunk c.
// Shared memory: Q 2 x 32 KB, K and V 4 stages x 20 KB each.  Every wait is bounded (abort
// flag, device status word).
#include <cuda_bf16.h>
#include <stdio.h>

#include <atomic>

#include "iso_internal.h"
#include "iso_ptx.cuh"

namespace iso {

// capi.cu: tensor map over a 3-D bf16 array [d2][d1][d0] (d0 innermost), 128-byte swizzle
iso_status make_tmap_bf16_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                             uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2);

namespace {

constexpr int AT_ROWS = 128;    // query rows per tile (the MMA's M)
constexpr int AT_KEYS = ATT_CHUNK_KEYS;  // keys per chunk (N of Q K^T, K of P V)
constexpr int AT_D = 128;       // head dimension
constexpr int AT_STAGES = 4;    // K / V ring depth (chunk c in stage c % 4)
constexpr int AT_THREADS = 512;  // 4 warpgroups
// Register split (setmaxnreg): launched at 128 per thread (512 x 128 = 65,536); the two softmax
// warpgroups take 200 and the two control warpgroups keep 56: 2 x 128 x 200 + 2 x 128 x 56 =
// 65,536, exactly the launch's total, so the increase always finds its registers.
constexpr int AT_REGS_SOFTMAX = 200;
constexpr int AT_REGS_CONTROL = 56;
static_assert(2 * 128 * AT_REGS_SOFTMAX + 2 * 128 * AT_REGS_CONTROL <= AT_THREADS * 128, "register split");
constexpr int AT_Q_BYTES = AT_ROWS * AT_D * 2;      // 32 KB: one Q tile (two {64, 128} boxes)
constexpr int AT_KV_HALF = AT_KEYS * 64 * 2;        // 10 KB: one {64 dims, 80 keys} box
constexpr int AT_KV_BYTES = 2 * AT_KV_HALF;         // 20 KB: K or V of one chunk
constexpr int AT_SMEM = 1024 /*align*/ + 2 * AT_Q_BYTES + 2 * AT_STAGES * AT_KV_BYTES + 256 /*barriers*/;
static_assert(AT_KV_HALF % 1024 == 0, "128-byte swizzle atoms stay 1024-byte aligned");
constexpr int AT_WARP_PRODUCER = 8;
constexpr int AT_WARP_MMA0 = 9;  // 9: S_A, 10: PV_A, 11: S_B, 12: PV_B
// TMEM columns of tile t (add 256 t)
constexpr int AT_COL_S = 0;
constexpr int AT_COL_P = 80;
constexpr int AT_COL_O = 128;

struct AttnParams {
  const int32_t* q_start;  // [B+1]
  const int32_t* k_start;  // [B+1]
  const int32_t* pos0;     // [B]
  int B, Hq, Hkv;
  int Tq;   // query rows of the call (the debug build's store bound)
  int gp;   // query heads per tile (the G = Hq / Hkv heads of a KV group when G divides 128, else 1)
  int tpt;  // tokens per tile, 128 / gp: tile row r is token r / gp, head r % gp of the group
  float scale_log2e;  // scale * log2(e), rounded to fp32
  __nv_bfloat16* out;  // [Tq x Hq x d]
  float* lse;          // [Tq x Hq]
  unsigned int* status;
  uint64_t timeout_ns;
};

// S = Q K^T: A (Q) and B (K) both K-major in shared memory, N = 80.  O += P V: A (P) K-major in
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
constexpr float kLazy = ATT_LAZY_LOG2;  // base-2 headroom before the running maximum moves
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
// 32 lanes x 8 consecutive 32-bit columns
__device__ __forceinline__ void tmem_st8p(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// 3-D tiled load; x is the innermost coordinate (elements).
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* m, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
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

// Bounded wait for every MMA this thread issued (its commit on `bar`), then the warp goes on.
__device__ __forceinline__ void drain_own_mmas(uint64_t* bar, bool leader, const AttnParams& p,
                                               volatile int* abort_flag) {
  if (leader) umma_commit(bar);
  __syncwarp();
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(smem_u32(bar), 0)) {
    if (globaltimer_ns() - t0 > p.timeout_ns) {
      *abort_flag = 1;
      atomicOr(p.status, kDevTimeout);
      break;
    }
  }
}

__global__ void __launch_bounds__(AT_THREADS, 1)
    iso_attention_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  // grid (Hq / gp head groups, B, tile pairs): the pairs furthest into their sequences (the most
  // chunks) start first.  A tile holds tpt tokens x gp heads (row r: token r / gp, head r % gp).
  const int h0 = blockIdx.x * p.gp, b = blockIdx.y, pair = gridDim.z - 1 - blockIdx.z;
  const int gp = p.gp, tpt = p.tpt;
  const int q0 = p.q_start[b], nq = p.q_start[b + 1] - q0;
  // shape checks, uniform over the CTA and taken before any barrier or TMEM use: the grid
  // must cover every query row, and the last row's keys must lie inside the sequence
  if (threadIdx.x == 0 && h0 == 0 && pair == static_cast<int>(gridDim.z) - 1 &&
      (nq > static_cast<int>(gridDim.z) * 2 * tpt || nq < 0 || p.pos0[b] < 0 ||
       p.k_start[b] + p.pos0[b] + nq > p.k_start[b + 1]))
    atomicOr(p.status, kDevBadShape);
  if (nq <= 0 || p.pos0[b] < 0 || p.k_start[b] + p.pos0[b] + nq > p.k_start[b + 1]) return;
  const int tileA = 2 * pair;
  if (tileA * tpt >= nq) return;  // empty unit
  // per tile (A, B): valid tokens, position of its first token, chunks its last token sees
  const int tok_a = min(tpt, nq - tileA * tpt);
  const int tok_b = max(0, min(tpt, nq - (tileA + 1) * tpt));
  const int pos_a = p.pos0[b] + tileA * tpt;
  const int chunks_a = (pos_a + tok_a - 1) / AT_KEYS + 1;
  const int chunks_b = tok_b > 0 ? (pos_a + tpt + tok_b - 1) / AT_KEYS + 1 : 0;
  const int n_all = max(chunks_a, chunks_b);
  const int g = h0 / (p.Hq / p.Hkv);
  const int kbase = p.k_start[b];

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                               // 2 tiles
  uint8_t* sK = smem + 2 * AT_Q_BYTES;              // AT_STAGES stages
  uint8_t* sV = sK + AT_STAGES * AT_KV_BYTES;       // AT_STAGES stages
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + AT_STAGES * AT_KV_BYTES);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;                     // [AT_STAGES]
  uint64_t* kv_empty = kv_full + AT_STAGES;         // [tile][AT_STAGES]: P V of the tile read the stage
  uint64_t* s_full = kv_empty + 2 * AT_STAGES;      // [tile]
  uint64_t* s_free = s_full + 2;                    // [tile]: the softmax has read S
  uint64_t* p_full = s_free + 2;                    // [tile]
  uint64_t* pv_done = p_full + 2;                   // [tile]
  uint64_t* issuer_done = pv_done + 2;              // [4]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(issuer_done + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    mbar_init(q_full, 1);
    for (int s = 0; s < AT_STAGES; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
      mbar_init(&kv_empty[AT_STAGES + s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&s_free[t], AT_ROWS);
      mbar_init(&p_full[t], AT_ROWS);
      mbar_init(&pv_done[t], 1);
    }
    for (int i = 0; i < 4; ++i) mbar_init(&issuer_done[i], 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == AT_WARP_MMA0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8) {
    // ---------------------------------------------------------- control warpgroups
    regs_dec<AT_REGS_CONTROL>();
    if (warp == AT_WARP_PRODUCER) {
      if (lane == 0) {
        int issued = 0;
        const int n_q_tiles = chunks_b > 0 ? 2 : 1;
        mbar_arrive_expect_tx(q_full, n_q_tiles * AT_Q_BYTES);
        // Q of a tile: {64 dims, gp heads, tpt tokens} boxes, rows token-major
        for (int t = 0; t < n_q_tiles; ++t)
          for (int kb = 0; kb < 2; ++kb)
            tma_load_3d(sQ + t * AT_Q_BYTES + kb * (AT_Q_BYTES / 2), &tmQ, q_full, kb * 64, h0,
                        q0 + (tileA + t) * tpt);
        for (int c = 0; c < n_all; ++c) {
          const int s = c % AT_STAGES;
          if (c >= AT_STAGES) {
            // the stage held chunk c - 4: every tile that used it has finished its P V
            const int old = c - AT_STAGES;
            const uint32_t par = ((c / AT_STAGES) - 1) & 1;
            bool ok = true;
            if (old < chunks_a) ok = mbar_wait(&kv_empty[s], par, p.timeout_ns, abort_flag, p.status);
            if (ok && old < chunks_b)
              ok = mbar_wait(&kv_empty[AT_STAGES + s], par, p.timeout_ns, abort_flag, p.status);
            if (!ok) break;
          }
          const int krow = kbase + c * AT_KEYS;
          mbar_arrive_expect_tx(&kv_full[s], 2 * AT_KV_BYTES);
          // K (K-major B of Q K^T) and V (MN-major B of P V): each two {64 dims, 80 keys} boxes
          for (int half = 0; half < 2; ++half) {
            tma_load_2d(sK + s * AT_KV_BYTES + half * AT_KV_HALF, &tmK, &kv_full[s], g * AT_D + half * 64, krow);
            tma_load_2d(sV + s * AT_KV_BYTES + half * AT_KV_HALF, &tmV, &kv_full[s], g * AT_D + half * 64, krow);
          }
          issued = c + 1;
        }
        // before the CTA may exit: every load this thread issued has landed (bounded; normally
        // the MMAs have consumed them all and these phases are long complete)
        const uint64_t t0 = globaltimer_ns();
        bool landed = false;
        while (!landed && globaltimer_ns() - t0 <= p.timeout_ns) {
          landed = mbar_try_wait(smem_u32(q_full), 0);
          for (int c = (issued > AT_STAGES ? issued - AT_STAGES : 0); c < issued && landed; ++c)
            landed = mbar_try_wait(smem_u32(&kv_full[c % AT_STAGES]), (c / AT_STAGES) & 1);
        }
        if (!landed) {
          *abort_flag = 1;
          atomicOr(p.status, kDevTimeout);
        }
      }
    } else if (warp >= AT_WARP_MMA0 && warp < AT_WARP_MMA0 + 4) {
      // ------------------------------------------------------------------ MMA issuers
      const int role = warp - AT_WARP_MMA0;  // 0: S_A, 1: PV_A, 2: S_B, 3: PV_B
      const int t = role >> 1;
      const bool is_pv = (role & 1) != 0;
      const int nct = t ? chunks_b : chunks_a;
      const bool leader = lane == 0;
      const uint32_t tS = tmem + t * 256 + AT_COL_S;
      const uint32_t tP = tmem + t * 256 + AT_COL_P;
      const uint32_t tO = tmem + t * 256 + AT_COL_O;
      const uint64_t kdesc0 = sdesc_sw128(0, 16, 1024);           // K-major operand template
      const uint64_t vdesc0 = sdesc_sw128(0, AT_KV_HALF, 1024);   // MN-major: 64-column halves 10 KB apart
      bool ok = nct > 0 && warp_wait(q_full, 0, p, abort_flag);
      if (!is_pv) {
        // S_t(c) = Q_t K_c^T, as soon as K_c has landed and the softmax has read S_t(c - 1)
        const uint32_t q_lo = smem_u32(sQ + t * AT_Q_BYTES) >> 4;
        for (int c = 0; c < nct && ok; ++c) {
          ok = warp_wait(&kv_full[c % AT_STAGES], (c / AT_STAGES) & 1, p, abort_flag);
          if (ok && c > 0) ok = warp_wait(&s_free[t], (c - 1) & 1, p, abort_flag);
          if (!ok) break;
          tc_fence_after();
          if (leader) {
            const uint32_t k_lo = smem_u32(sK + (c % AT_STAGES) * AT_KV_BYTES) >> 4;
#pragma unroll
            for (int kb = 0; kb < 2; ++kb)
#pragma unroll
              for (int k16 = 0; k16 < 4; ++k16) {
                const uint64_t ad = kdesc0 + q_lo + kb * (AT_Q_BYTES / 2 / 16) + k16 * 2;
                const uint64_t bd = kdesc0 + k_lo + kb * (AT_KV_HALF / 16) + k16 * 2;
                umma_bf16(tS, ad, bd, kIdescS, (kb | k16) != 0 ? 1u : 0u);
              }
            umma_commit(&s_full[t]);
          }
          __syncwarp();
        }
      } else {
        // O_t += P_t(c) V_c, once the softmax has written P_t(c) (and rescaled O_t)
        for (int c = 0; c < nct && ok; ++c) {
          ok = warp_wait(&kv_full[c % AT_STAGES], (c / AT_STAGES) & 1, p, abort_flag);
          if (ok) ok = warp_wait(&p_full[t], c & 1, p, abort_flag);
          if (!ok) break;
          tc_fence_after();
          if (leader) {
            const uint32_t v_lo = smem_u32(sV + (c % AT_STAGES) * AT_KV_BYTES) >> 4;
#pragma unroll
            for (int k16 = 0; k16 < AT_KEYS / 16; ++k16)
              umma_bf16_tmem_a(tO, tP + k16 * 8, vdesc0 + v_lo + k16 * 128, kIdescPV, (c | k16) != 0 ? 1u : 0u);
            umma_commit(&pv_done[t]);
            umma_commit(&kv_empty[t * AT_STAGES + c % AT_STAGES]);  // S_t(c) finished before P_t(c) existed
          }
          __syncwarp();
        }
      }
      // the CTA exits only after this thread's MMAs completed
      drain_own_mmas(&issuer_done[role], leader, p, abort_flag);
    }
  } else {
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
    const uint32_t tS = tmem + t * 256 + AT_COL_S + lane_off;
    const uint32_t tP = tmem + t * 256 + AT_COL_P + lane_off;
    const uint32_t tO = tmem + t * 256 + AT_COL_O + lane_off;
    const int nc = t ? chunks_b : chunks_a;
    const int tok = r / gp;  // this row's token within the tile and head within the group
    const int head = h0 + r % gp;
    const bool row_valid = tok < (t ? tok_b : tok_a);
    const int pos = pos_a + t * tpt + tok;  // this row's position (invalid rows compute unused values)
    const int warp_pos_min = pos_a + t * tpt + (quarter * 32) / gp;
    const float c2 = p.scale_log2e;
    float m = -INFINITY, l = 0.f;
    bool ok = nc > 0;
    for (int c = 0; c < nc && ok; ++c) {
      ok = warp_wait(&s_full[t], c & 1, p, abort_flag);
      if (!ok) break;
      tc_fence_after();
      uint32_t v[AT_KEYS];
      tmem_ld32p(tS, v);
      tmem_ld32p(tS + 32, v + 32);
      tmem_ld16p(tS + 64, v + 64);
      tmem_ld_wait_only();
      tmem_ld_tie(v);
      tmem_ld_tie(v + 32);
      tmem_ld_tie16(v + 64);
      tc_fence_before();
      mbar_arrive(&s_free[t]);  // S_t(c) is in registers: Q K^T of chunk c + 1 may overwrite it
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
      for (int j = 16; j < AT_KEYS; j += 16)  // keys j .. j + 15, j + 15 <= 79
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
      if (c > 0) {
        // P V of chunk c - 1 done: O is current and P may be overwritten (every phase is
        // waited for, in order)
        ok = warp_wait(&pv_done[t], (c - 1) & 1, p, abort_flag);
        if (!ok) break;
        tc_fence_after();
        // the rescale is taken by the whole warp when any of its rows needs it (x * 1 = x
        // exactly, so a row whose maximum did not move keeps its bits)
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
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
      }
      // P: 40 columns, column k holds keys 2k (low half) and 2k + 1
      tmem_st32p(tP, v);
      tmem_st8p(tP + 32, v + 32);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[t]);
    }
    if (ok) ok = warp_wait(&pv_done[t], (nc - 1) & 1, p, abort_flag);
    if (ok) {
      tc_fence_after();
      uint32_t o[AT_D];
#pragma unroll
      for (int q = 0; q < AT_D / 32; ++q) tmem_ld32p(tO + q * 32, o + q * 32);
      tmem_ld_wait_only();
#pragma unroll
      for (int q = 0; q < AT_D / 32; ++q) tmem_ld_tie(o + q * 32);
      const int64_t row = q0 + (tileA + t) * tpt + tok;
      if (row_valid && ISO_DCHECK(row >= 0 && row < p.Tq && head < p.Hq, p.status)) {
        __nv_bfloat16* dst = p.out + (row * p.Hq + head) * AT_D;
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
        if (p.lse) p.lse[row * p.Hq + head] = __fadd_rn(__fmul_rn(m, kLn2), logf(l));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == AT_WARP_MMA0) {
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
  // a tile packs the G = Hq / Hkv query heads of a KV group with 128 / G tokens each when G divides
  // 128 (one KV stream serves all G heads: decode reads each KV head once), else 1 head x 128 tokens
  const int G = Hq / Hkv;
  const int gp = (G <= AT_ROWS && AT_ROWS % G == 0) ? G : 1;
  const int tpt = AT_ROWS / gp;
  const int pairs = ((max_q_rows + tpt - 1) / tpt + 1) / 2;  // tiles of tpt tokens, two per CTA
  if (B > 65535 || pairs > 65535) return ISO_ERR_UNSUPPORTED;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) |
                        reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(out);
  if (mis & 15u) return ISO_ERR_ALIGNMENT;
  if (!device_ready()) return ISO_ERR_CUDA;
  CUtensorMap tQ, tK, tV;
  iso_status st = make_tmap_bf16_3d(&tQ, Q, d, Hq, Tq, d, static_cast<uint64_t>(Hq) * d, 64, gp, tpt);
  if (st == ISO_OK)
    st = make_tmap_bf16(&tK, K, Tk, static_cast<uint64_t>(Hkv) * d, static_cast<uint64_t>(Hkv) * d, 64, AT_KEYS);
  if (st == ISO_OK)
    st = make_tmap_bf16(&tV, V, Tk, static_cast<uint64_t>(Hkv) * d, static_cast<uint64_t>(Hkv) * d, 64, AT_KEYS);
  if (st != ISO_OK) return st;
  AttnParams p;
  p.q_start = q_start;
  p.k_start = k_start;
  p.pos0 = pos0;
  p.B = B;
  p.Tq = Tq;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.gp = gp;
  p.tpt = tpt;
  p.scale_log2e = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.status = device_status_ptr();
  p.timeout_ns = wait_timeout_ns();
  // the shared-memory attribute, once per device (concurrent first calls set the same value)
  static std::atomic<bool> attr_set[ISO_MAX_DEVICES] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= ISO_MAX_DEVICES) return ISO_ERR_CUDA;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(iso_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AT_SMEM) !=
        cudaSuccess)
      return ISO_ERR_CUDA;
    attr_set[dev].store(true, std::memory_order_release);
  }
  const dim3 grid(Hq / gp, B, pairs);
  iso_attention_kernel<<<grid, AT_THREADS, AT_SMEM, static_cast<cudaStream_t>(stream)>>>(tQ, tK, tV, p);
  return cudaGetLastError() == cudaSuccess ? ISO_OK : ISO_ERR_CUDA;
}
