// iso_internal.h -- declarations shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/iso.h"

namespace iso {

// Device status bits, OR-ed into the library's device status word.
enum : unsigned int {
  kDevTimeout = 1u << 0,   // an mbarrier wait ran out of time
  kDevBadToken = 1u << 1,  // a token id outside [0, V)
  kDevBadShape = 1u << 2,  // a device-side shape check failed
  kDevCheck = 1u << 3,     // a debug-build bounds check failed (the access was skipped)
};

// Device-side bounds checks of the debug build (-DISO_DEBUG, libiso_debug.so): a failed check
// records kDevCheck in the status word and the guarded access is skipped, instead of trapping
// (a trap would take the context down).  In the normal build the condition is not evaluated.
#ifdef ISO_DEBUG
#define ISO_DCHECK(cond, status) ((cond) ? true : (atomicOr((status), ::iso::kDevCheck), false))
#else
#define ISO_DCHECK(cond, status) true
#endif

// Output tile of one CTA: 128 rows (TMEM lanes) x 128 columns; K staged in
// blocks of 64 (one 128-byte swizzle row of bf16).
constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BK = 64;
constexpr int UMMA_K = 16;
// Shared memory: [A tiles: stages x a_bytes][B tiles: stages x 16 KB][barriers]
// [bf16 output staging, when it fits].
// The A box has a_rows rows (128, or 16/32/64 when the whole problem has that few
// rows); the freed space buys more pipeline stages for the weight stream.  The MMA
// always reads 128 A rows; rows past the box hold stale data whose outputs are
// never stored.  The staging area (32 KB: per epilogue warp 32 rows x 256 bytes, or
// x 128 bytes with 8 epilogue warps) lets a warp write its bf16 rows to global memory
// whole rows at a time; it exists when the stages leave room for it (A boxes of 64 and
// 128 rows).
constexpr int MAX_STAGES = 12;
constexpr int A_TILE_BYTES_MAX = BM * BK * 2;
constexpr int B_STAGE_BYTES = BK * BN * 2;
// Deep stages of a CTA pair with one producer (a one-leaf contract): 128 k per stage, the CTA's
// A tile [128 x 128] one TMA box of a 3-D view ({64 k, rows, k / 64}) and its 64-column half of
// B one {64 x 128} box, two TMA instructions per 48 KB.  A producer thread pays ~200 cycles per
// TMA (measured on GB300): alone, with 24 KB stages it delivers ~60 bytes/cycle/SM of the 94 a
// pair consumes at the tensor rate.  Two producers (two or more leaves) keep 64-k stages.
constexpr int PAIR_BK = 128;
constexpr int GEMM_BARRIER_BYTES = 512;
constexpr int NUM_TMEM_BUFS = 4;  // 4 x 128 fp32 columns = all 512 TMEM columns
constexpr int TMEM_COLS = 512;
// Per-device host caches (status word, SM count, kernel attributes) hold this many devices.
constexpr int ISO_MAX_DEVICES = 64;
constexpr int GEMM_THREADS = 256;  // warps 0,3 TMA; warps 1-2 MMA (even/odd leaves); warps 4..7 epilogue
constexpr int GEMM_THREADS_FUSED = 384;      // + warps 8..11: the fused RMSNorm prologue
// Short leaves: the tree steps and the root of a tile outlast its MMAs, so warps 8..11 join
// the epilogue (two warps per TMEM lane quarter, each with its own columns of the tile).
// Measured on GB300: a gain for SwiGLU roots with leaves up to 256 k and bf16 roots up to
// 128 k; with bf16 roots and 256-k leaves the MMAs already hide the epilogue and the extra
// warps cost 2-3 %.
constexpr int GEMM_THREADS_EPI8 = 384;
constexpr int EPI8_MAX_LEAF_SWIGLU = 256;
constexpr int EPI8_MAX_LEAF_BF16 = 128;
// Whole-leaf stages for leaves of 96 k: A 128 x 64 (16 KB) + 128 x 32 (8 KB), B 96 x 128 (24 KB).
constexpr int LS_LEAF = 96;
constexpr int LS_A2_OFF = BM * 64 * 2;            // the 32-column A box, after the 64-column one
constexpr int LS_A_BYTES = BM * LS_LEAF * 2;      // 24 KB
constexpr int LS_B_BYTES = LS_LEAF * BN * 2;      // 24 KB
constexpr int GEMM_REGS_CONTROL_EPI8 = 56;    // setmaxnreg of warps 0-3 with 8 epilogue warps
constexpr int GEMM_REGS_EPILOGUE_EPI8 = 224;  // and of warps 4-11
static_assert(128 * GEMM_REGS_CONTROL_EPI8 + 256 * GEMM_REGS_EPILOGUE_EPI8 <= 384 * 168,
              "register split within the launch's allocation");
constexpr int GEMM_REGS_CONTROL_FUSED = 120;  // setmaxnreg of warps 0-3 and 8-11 (epilogue: 256)
// The epilogue keeps one partial root per thread in registers for a group of up to 8 leaves.
// With 16 leaves the root of leaves [0, 8) is parked in shared memory (fp32, 64 KB,
// [column][row] so consecutive rows are consecutive words) while the second group runs, and
// the epilogue adds it to the root of leaves [8, 16) at the top of the tree -- the same fp32
// add the tree makes there.
constexpr int TMEM_TREE_LEAVES = 8;
constexpr int MAX_LEAVES = 16;
constexpr int SPILL_BYTES = BM * BN * 4;
constexpr int GEMM_SMEM_BYTES = 232448;  // the per-block maximum; 1 KB of it is alignment slack
constexpr int MOE_MAX_EXPERTS = 256;
constexpr int MOE_PERM_CHUNK = 1024;   // pairs per chunk of the permutation's counting sort
constexpr int MOE_PERM_THREADS = 256;
constexpr int EPI_STAGE_BYTES = 4 * 32 * BN * 2;  // 4 epilogue warps x 32 rows x 128 bf16 (or 8 x 64)

// Logprob vocab tiling: statistics per 128-column tile, 19 tiles per chunk.
constexpr int LP_TILE_COLS = BN;
constexpr int LP_CHUNK_TILES = 19;

// Attention merge grid: keys in fixed chunks of 80 per sequence, merged in ascending order; the
// running maximum (base 2) moves only when a chunk's maximum exceeds it by more than 8.
constexpr int ATT_CHUNK_KEYS = 80;
constexpr float ATT_LAZY_LOG2 = 8.0f;

// EPI_CLUSTER: one row block, the L leaves split into R groups that run as one thread-block
// cluster of R CTAs per 128-column tile; each CTA leaves its group's fp32 subtree root in its
// shared memory and, after a cluster barrier, combines one R-th of the tile's columns over all R
// groups (distributed shared memory) with the top log2 R levels of the tree, then rounds to bf16.
enum EpiMode { EPI_BF16 = 0, EPI_F32 = 1, EPI_LOGPROB = 2, EPI_SWIGLU = 3, EPI_CLUSTER = 4 };
enum UnitMode { UNIT_GEMM = 0, UNIT_LOGPROB = 1, UNIT_GROUPED = 2, UNIT_LEAF_SPLIT = 3, UNIT_CLUSTER = 4 };
constexpr int MAX_CLUSTER_GROUPS = 8;  // portable cluster size

struct GemmParams {
  int M, N, K;     // K = contraction length handled by this launch
  int L;           // leaves in this launch
  int leaf_len;    // K / L, a multiple of 16
  int num_kb;      // ceil(K / BK)
  int kb_per_leaf; // ceil(leaf_len / stage_k)
  int stage_k;     // k per pipeline stage: BK, or PAIR_BK on a one-producer CTA pair
  int stages;      // pipeline stages (<= MAX_STAGES), split between the two leaf-parity streams
  int spill;       // 1 when L > TMEM_TREE_LEAVES: the root of leaves [0, L/2) is parked in shared memory
  int cluster;     // EPI_CLUSTER: leaf groups per tile = CTAs per cluster (the group root uses the park region)
  int epi_staged;  // 1: bf16 roots go out through the shared-memory staging area
  int pair;        // 1: clusters of two CTAs, M = 256 MMAs; a unit covers 2 x 128 rows
  int a_rows;      // rows of the A box (16, 32, 64 or 128)
  int a_bytes;     // a_rows * 128
  int b_tile_cols; // B columns advanced per tile (128; 64 for the SwiGLU gate/up pairing)
  int b_box2_off;  // column offset of the second 64-column B box (64; F for SwiGLU)
  int m_blocks, n_blocks;
  int unit_mode;
  int num_units;   // GEMM / LOGPROB: host-known unit count
  int group_m;     // GEMM raster: m-blocks per group
  void* out;
  int64_t ldo;
  int64_t out_rows;  // rows of `out` (per leaf group) the epilogue may write: the debug build's store bound
  const int32_t* row_scatter;  // grouped down projection: destination row of each permuted row
  // logprob
  const int32_t* ids;
  float2* ws_stats;  // [entries][T] (m, s): entries = vocab chunks, or tiles with one tile per unit
  float* ws_zsel;    // [T]
  int V;
  int sel_base;      // vocabulary column of this launch's column 0 (a vocab shard's first column)
  int chunk_tiles;
  int num_chunks;
  // grouped
  const int32_t* g_offsets;      // [E+1]
  const int32_t* g_unit_prefix;  // [E+1]
  int E;
  // leaf split (one row block): unit u = (group r, n-tile); group r covers K [r K, (r+1) K) of the
  // full problem (K here is the group's length) and writes its fp32 subtree root to
  // out + r * out_group_stride
  int64_t out_group_stride;
  // fused RMSNorm prologue (a_transform = 1): the A operand is y = bf16((x * rinv[row]) * gamma[k])
  // [RL-Kernel blog, §6 table row 02; the same arithmetic as iso_rmsnorm], built in shared memory
  // by the producer warps from x [M x K] (leading dimension lda_src) instead of loaded by TMA
  int a_transform;
  // whole-leaf stages (leaf_stage = 1, leaves of 96 k, single CTA, bf16 roots): a stage holds one
  // leaf, A as a 64-column box (128-byte swizzle) and a 32-column box (64-byte swizzle, second
  // tensor map), B as two 64-column x 96-row boxes; kb_per_leaf = 1
  int leaf_stage;
  // 1: this launch reads each B element once (one row block: decode-size GEMMs and logprobs),
  // so B loads carry an evict-first L2 policy and leave L2 to what is read again.  Measured on
  // GB300: back-to-back one-row GEMMs 1-4 % faster; with many row blocks, whose B tiles are
  // shared by a raster group, the same policy cost 2-5 %, so they keep the default.
  int b_stream;
  const void* a_src;      // x, bf16
  int64_t lda_src;
  const float* a_rinv;    // [M] per-row 1 / sqrt(mean x^2 + eps)
  const void* a_gamma;    // [K] bf16
  // error reporting
  unsigned int* status;
  uint64_t timeout_ns;
};

// Library-wide state, per device.
bool device_ready();                // per-device state looked up (status word address, SM count)
unsigned int* device_status_ptr();  // device address of the status word (current device)
uint64_t wait_timeout_ns();
int sm_count();
bool trace_enabled();

// Tensor map over a row-major bf16 matrix [rows x cols] with leading
// dimension ld (elements), box {box_cols, box_rows}, 128-byte swizzle.
iso_status make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                          uint32_t box_cols, uint32_t box_rows);
// The same with a 64-byte swizzle (boxes 32 columns wide).
iso_status make_tmap_bf16_sw64(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                               uint32_t box_cols, uint32_t box_rows);

// Launchers (gemm_tcgen05.cu).  max_units bounds the number of CTAs (p.pair: CTA pairs)
// worth launching; the grid is that or the number that fit on the GPU at once.
// tmA2: the 32-column A boxes of whole-leaf stages (p.leaf_stage), else unused (may be null).
iso_status launch_gemm(int epi, const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int max_units,
                       cudaStream_t s, const CUtensorMap* tmA2 = nullptr);
// Clusters of R CTAs of the EPI_CLUSTER GEMM that are resident at once on the current device
// (0 when R is not 2, 4 or 8 or the query fails).
int cluster_gemm_capacity(int R);

// Launch with programmatic stream serialization allowed (and clusters of cluster_x CTAs when
// cluster_x > 1): the grid may be scheduled while the stream's previous grid finishes, so it
// overlaps that grid's tail and its own launch.  Only for kernels that execute
// grid_dependency_wait before their first global-memory access.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             unsigned int cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[2];
  unsigned int n = 0;
  at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = cluster_x;
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace iso
