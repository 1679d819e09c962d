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
//   P_j  = exp2f(fma(S_j, c2, -m'));  l_c = (sum of four interleaved partial sums, fixed order)
//   a    = exp2f(m - m') (1 when m' = m);  l = rn(rn(l * a) + l_c);  O = rn(O * a) when a != 1
//   O   += bf16(P) V   (8 tcgen05 MMAs, K = 16 keys each, ascending keys)
// and at the end out = bf16_rn(O * rcp(l)), lse = rn(rn(m ln 2) + logf(l)).  Every step
// depends only on the row, its position and the chunk grid, never on the other rows of its
// tile or the launch, so a decode call (one row) reproduces the row of a prefill call exactly.
// A chunk wholly past a row's position changes nothing in that row: t = -inf, a = 1, P = 0,
// O + 0 = O.
//
// Structure: one CTA per (query head, sequence, tile of up to 128 query rows), the tiles with
// the most chunks first; 192 threads.
//   warp 0     TMA producer: Q once, then K and V chunks into a 2-stage ring
//   warp 1     MMA issuer (one elected lane) and TMEM owner: S_{c+1} = Q K_{c+1}^T is issued
//              before waiting for P_c, so it overlaps the softmax of chunk c
//   warps 2-5  softmax / correction / output: one thread per query row (TMEM lane)
// TMEM: S in two 128-column buffers, O in a third.  Shared memory: Q 32 KB, K and V 2 x 32 KB
// each, P 32 KB (bf16, written by the softmax threads in the 128-byte-swizzled K-major layout
// the MMA reads).  Every wait is bounded (abort flag, device status word).
#include <cuda_bf16.h>
#include <stdio.h>

#include "iso_internal.h"
#include "iso_ptx.cuh"

namespace iso {

namespace {

constexpr int AT_ROWS = 128;    // query rows per tile (the MMA's M)
constexpr int AT_KEYS = 128;    // keys per chunk (N of QK^T, K of PV)
constexpr int AT_D = 128;       // head dimension
constexpr int AT_THREADS = 192;
constexpr int AT_TILE_BYTES = AT_ROWS * AT_D * 2;  // 32 KB: one 128 x 128 bf16 operand tile
constexpr int AT_SMEM = 1024 /*align*/ + 6 * AT_TILE_BYTES + 256 /*barriers*/;

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

// S = Q K^T: A (Q) and B (K) both K-major.  O += P V: A (P) K-major, B (V) MN-major.
constexpr uint32_t kIdescS = idesc_bf16_f32(AT_ROWS, AT_KEYS, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(AT_ROWS, AT_D, false, true);

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);  // .x (low half) = lo
  return *reinterpret_cast<const uint32_t*>(&t);
}
constexpr float kLazy = 8.0f;  // base-2 headroom before the running maximum moves
constexpr float kLn2 = 0.693147180559945309f;

__global__ void __launch_bounds__(AT_THREADS, 1)
    iso_attention_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  // grid (Hq, B, tiles): the tiles furthest into their sequences (the most chunks) start first
  const int h = blockIdx.x, b = blockIdx.y, tile = gridDim.z - 1 - blockIdx.z;
  const int q0 = p.q_start[b], nq = p.q_start[b + 1] - q0;
  // shape checks, uniform over the CTA and taken before any barrier or TMEM use: the grid
  // must cover every query row, and the last row's keys must lie inside the sequence
  if (threadIdx.x == 0 && h == 0 && tile == static_cast<int>(gridDim.z) - 1 &&
      (nq > static_cast<int>(gridDim.z) * AT_ROWS || nq < 0 || p.pos0[b] < 0 ||
       p.k_start[b] + p.pos0[b] + nq > p.k_start[b + 1]))
    atomicOr(p.status, kDevBadShape);
  if (nq <= 0 || p.pos0[b] < 0 || p.k_start[b] + p.pos0[b] + nq > p.k_start[b + 1]) return;
  if (tile * AT_ROWS >= nq) return;  // empty unit
  const int rows_valid = min(AT_ROWS, nq - tile * AT_ROWS);
  const int pos_first = p.pos0[b] + tile * AT_ROWS;            // position of the tile's row 0
  const int n_chunks = (pos_first + rows_valid - 1) / AT_KEYS + 1;  // chunks the last row sees
  const int g = h / (p.Hq / p.Hkv);
  const int kbase = p.k_start[b];

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + AT_TILE_BYTES;          // 2 stages
  uint8_t* sV = smem + 3 * AT_TILE_BYTES;      // 2 stages
  uint8_t* sP = smem + 5 * AT_TILE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 6 * AT_TILE_BYTES);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;   // [2]
  uint64_t* kv_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;    // [2]
  uint64_t* p_full = bars + 7;
  uint64_t* o_done = bars + 8;
  uint64_t* drain = bars + 9;
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
    }
    mbar_init(p_full, AT_ROWS);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // S buffer s at columns [128 s, 128 s + 128), O at [256, 384)
  const uint32_t tO = tmem + 256;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      bool ok = true;
      int issued = 0;
      mbar_arrive_expect_tx(q_full, AT_TILE_BYTES);
      for (int kb = 0; kb < 2; ++kb)
        tma_load_2d(sQ + kb * (AT_TILE_BYTES / 2), &tmQ, q_full, h * AT_D + kb * 64, q0 + tile * AT_ROWS);
      for (int c = 0; c < n_chunks && ok; ++c) {
        const int s = c & 1;
        if (c >= 2 && !mbar_wait(&kv_empty[s], ((c >> 1) - 1) & 1, p.timeout_ns, abort_flag, p.status)) {
          ok = false;
          break;
        }
        const int krow = kbase + c * AT_KEYS;
        mbar_arrive_expect_tx(&kv_full[s], 2 * AT_TILE_BYTES);
        uint8_t* k_dst = sK + s * AT_TILE_BYTES;
        uint8_t* v_dst = sV + s * AT_TILE_BYTES;
        // K: two 64-dim boxes of 128 keys (K-major B of QK^T)
        for (int kb = 0; kb < 2; ++kb)
          tma_load_2d(k_dst + kb * (AT_TILE_BYTES / 2), &tmK, &kv_full[s], g * AT_D + kb * 64, krow);
        // V: per 64-key block, two 64-dim boxes (MN-major B of PV)
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
  } else if (warp == 1) {
    // --------------------------------------------------------------------- MMA
    const bool leader = (lane == 0);
    // every lane polls; the outcome is made warp-uniform before any .sync.aligned op
    bool ok = __all_sync(0xffffffffu, mbar_wait(q_full, 0, p.timeout_ns, abort_flag, p.status));
    const uint32_t q_lo = smem_u32(sQ) >> 4, p_lo = smem_u32(sP) >> 4;
    const uint64_t kdesc0 = sdesc_sw128(0, 16, 1024);   // K-major operand template
    const uint64_t vdesc0 = sdesc_sw128(0, 8192, 1024); // MN-major operand template
    auto issue_s = [&](int c) -> bool {
      const int s = c & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&kv_full[s], (c >> 1) & 1, p.timeout_ns, abort_flag, p.status)))
        return false;
      tc_fence_after();
      if (leader) {
        const uint32_t k_lo = smem_u32(sK + s * AT_TILE_BYTES) >> 4;
        for (int kb = 0; kb < 2; ++kb)
          for (int k16 = 0; k16 < 4; ++k16) {
            const uint64_t ad = kdesc0 + q_lo + kb * (AT_TILE_BYTES / 2 / 16) + k16 * 2;
            const uint64_t bd = kdesc0 + k_lo + kb * (AT_TILE_BYTES / 2 / 16) + k16 * 2;
            umma_bf16((tmem + s * 128), ad, bd, kIdescS, (kb | k16) != 0 ? 1u : 0u);
          }
        umma_commit(&s_full[s]);
      }
      __syncwarp();
      return true;
    };
    if (ok) ok = issue_s(0);
    for (int c = 0; c < n_chunks && ok; ++c) {
      if (c + 1 < n_chunks && !issue_s(c + 1)) {
        ok = false;
        break;
      }
      if (!__all_sync(0xffffffffu, mbar_wait(p_full, c & 1, p.timeout_ns, abort_flag, p.status))) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (leader) {
        const uint32_t v_lo = smem_u32(sV + (c & 1) * AT_TILE_BYTES) >> 4;
        for (int kb = 0; kb < 2; ++kb)
          for (int k16 = 0; k16 < 4; ++k16) {
            const uint64_t ad = kdesc0 + p_lo + kb * (AT_TILE_BYTES / 2 / 16) + k16 * 2;
            const uint64_t bd = vdesc0 + v_lo + kb * (AT_TILE_BYTES / 2 / 16) + k16 * 128;
            umma_bf16(tO, ad, bd, kIdescPV, (c | kb | k16) != 0 ? 1u : 0u);
          }
        umma_commit(&kv_empty[c & 1]);
        umma_commit(o_done);
      }
      __syncwarp();
    }
    if (leader) umma_commit(drain);
    __syncwarp();
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(drain), 0)) {
      if (globaltimer_ns() - t0 > p.timeout_ns) {
        *abort_flag = 1;
        atomicOr(p.status, kDevTimeout);
        break;
      }
    }
  } else {
    // ----------------------------------------------------- softmax / correction
    // Scores are handled in the base-2 domain: t_j = S_j * scale * log2(e) (one FMA with the
    // running maximum), P_j = 2^(t_j - m), and lse = m ln 2 + ln l at the end.  The running
    // maximum m moves only when a chunk's maximum exceeds it by more than kLazy (2^kLazy
    // bounds P and the sums stay far from overflow); then O and l are rescaled by 2^(m_old - m).
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int pos = pos_first + r;  // this row's position (rows past rows_valid compute unused values)
    const int warp_pos_min = pos_first + quarter * 32;
    const float c2 = p.scale_log2e;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int c = 0; c < n_chunks; ++c) {
      const int s = c & 1;
      // each lane polls; the outcome is made warp-uniform, so the warp reaches every
      // tcgen05.ld / st (.sync.aligned) converged
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[s], (c >> 1) & 1, p.timeout_ns, abort_flag, p.status));
      if (!ok) break;
      tc_fence_after();
      uint32_t v[AT_KEYS];
#pragma unroll
      for (int q = 0; q < AT_KEYS / 32; ++q) tmem_ld32p((tmem + s * 128) + lane_off + q * 32, v + q * 32);
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
      for (int i = 0; i < 8; ++i) mx[i] = u2f(v[i]);
#pragma unroll
      for (int j = 8; j < AT_KEYS; ++j) mx[j & 7] = fmaxf(mx[j & 7], u2f(v[j]));
      const float mc = __fmul_rn(fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                       fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))),
                                 c2);
      const float m_new = (m == -INFINITY || mc > m + kLazy) ? fmaxf(m, mc) : m;
      const float alpha = (m == -INFINITY) ? 1.f : exp2f(__fsub_rn(m, m_new));  // 1 when m stays
      m = m_new;
      const float neg_m = -m;
      // P_j = 2^(t_j - m); the chunk sum in four interleaved partial sums, combined in a fixed
      // order
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < AT_KEYS; ++j) {
        const float e = exp2f(__fmaf_rn(u2f(v[j]), c2, neg_m));
        v[j] = f2u(e);
        ls[j & 3] = __fadd_rn(ls[j & 3], e);
      }
      l = __fadd_rn(__fmul_rn(l, alpha), __fadd_rn(__fadd_rn(ls[0], ls[1]), __fadd_rn(ls[2], ls[3])));
      if (c > 0) {
        // PV of chunk c-1 done: O is current and the P buffer is free
        ok = __all_sync(0xffffffffu, mbar_wait(o_done, (c - 1) & 1, p.timeout_ns, abort_flag, p.status));
        if (!ok) break;
        tc_fence_after();
        // the rescale is taken by the whole warp when any of its rows needs it (x * 1 = x
        // exactly, so a row whose maximum did not move keeps its bits)
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int q = 0; q < AT_D / 32; ++q) {
            uint32_t o[32];
            tmem_ld32p(tO + lane_off + q * 32, o);
            tmem_ld_wait_only();
            tmem_ld_tie(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = f2u(__fmul_rn(u2f(o[i]), alpha));
            tmem_st32p(tO + lane_off + q * 32, o);
          }
          tmem_st_wait();
        }
      }
      // P as bf16 into the K-major, 128-byte-swizzled A tile of the PV MMA: key block kb
      // (64 keys) at kb * 16 KB, row r at (r / 8) * 1024 + (r % 8) * 128, 16-byte chunk q
      // of the row at slot q ^ (r % 8)
#pragma unroll
      for (int kb = 0; kb < 2; ++kb)
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int j = kb * 64 + q * 8;
          uint4 w;
          w.x = pack_bf16x2(u2f(v[j + 0]), u2f(v[j + 1]));
          w.y = pack_bf16x2(u2f(v[j + 2]), u2f(v[j + 3]));
          w.z = pack_bf16x2(u2f(v[j + 4]), u2f(v[j + 5]));
          w.w = pack_bf16x2(u2f(v[j + 6]), u2f(v[j + 7]));
          *reinterpret_cast<uint4*>(sP + kb * (AT_TILE_BYTES / 2) + (r >> 3) * 1024 + (r & 7) * 128 +
                                    ((q ^ (r & 7)) << 4)) = w;
        }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(o_done, (n_chunks - 1) & 1, p.timeout_ns, abort_flag, p.status));
    if (ok) {
      tc_fence_after();
      uint32_t o[AT_D];
#pragma unroll
      for (int q = 0; q < AT_D / 32; ++q) tmem_ld32p(tO + lane_off + q * 32, o + q * 32);
      tmem_ld_wait_only();
#pragma unroll
      for (int q = 0; q < AT_D / 32; ++q) tmem_ld_tie(o + q * 32);
      if (r < rows_valid) {
        const int64_t row = q0 + tile * AT_ROWS + r;
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
  if (warp == 1) {
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
  if (B > 65535 || (max_q_rows + AT_ROWS - 1) / AT_ROWS > 65535) return ISO_ERR_UNSUPPORTED;
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
  const dim3 grid(Hq, B, (max_q_rows + AT_ROWS - 1) / AT_ROWS);
  iso_attention_kernel<<<grid, AT_THREADS, AT_SMEM, static_cast<cudaStream_t>(stream)>>>(tQ, tK, tV, p);
  return cudaGetLastError() == cudaSuccess ? ISO_OK : ISO_ERR_CUDA;
}
