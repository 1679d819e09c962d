// capi.cu -- the C ABI: argument validation, TMA descriptors, launch order.
// All compute runs in the kernels of gemm_tcgen05.cu and elementwise.cu.
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "iso_elementwise.h"
#include "iso_internal.h"

// Per-device status word written by kernels (timeouts, bad token ids).
static __device__ unsigned int g_iso_status_word;

namespace iso {

namespace {

constexpr int kMaxDevices = ISO_MAX_DEVICES;
// Filled once per device under g_mu; read without the lock (acquire / release), so threads that
// launch on different devices at once see either nothing or the complete entry.
std::mutex g_mu;
std::atomic<unsigned int*> g_status_ptr[kMaxDevices] = {};
std::atomic<int> g_sm_count[kMaxDevices] = {};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return -1;
  return d;
}

bool ensure_device_state() {
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return false;
  if (g_status_ptr[d].load(std::memory_order_acquire) && g_sm_count[d].load(std::memory_order_acquire)) return true;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[d].load(std::memory_order_relaxed)) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_iso_status_word) != cudaSuccess) return false;
    g_status_ptr[d].store(static_cast<unsigned int*>(p), std::memory_order_release);
  }
  if (!g_sm_count[d].load(std::memory_order_relaxed)) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) return false;
    g_sm_count[d].store(n, std::memory_order_release);
  }
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
cudaStream_t S(iso_stream s) { return static_cast<cudaStream_t>(s); }

int div_up(int a, int b) { return (a + b - 1) / b; }

void trace(const char* what, int a, int b, int c, int d) {
  if (trace_enabled()) fprintf(stderr, "[iso] %s %d %d %d %d\n", what, a, b, c, d);
}

}  // namespace

bool device_ready() { return ensure_device_state(); }

unsigned int* device_status_ptr() {
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return nullptr;
  return g_status_ptr[d].load(std::memory_order_acquire);
}

int sm_count() {
  const int d = current_device();
  const int n = (d < 0 || d >= kMaxDevices) ? 0 : g_sm_count[d].load(std::memory_order_acquire);
  return n ? n : 148;
}

uint64_t wait_timeout_ns() {
  static uint64_t v = [] {
    const char* e = getenv("ISO_WAIT_TIMEOUT_NS");
    uint64_t t = e ? strtoull(e, nullptr, 10) : 0;
    return t ? t : 2000000000ull;
  }();
  return v;
}

bool trace_enabled() {
  static bool v = [] {
    const char* e = getenv("ISO_TRACE");
    return e && e[0] == '1';
  }();
  return v;
}

// The driver's tensor-map encoder, looked up once.
static bool resolve_encode() {
  if (g_encode) return true;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return true;
}

namespace {
iso_status make_tmap_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                        uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  if (!resolve_encode()) return ISO_ERR_CUDA;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {ld * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ISO_OK : ISO_ERR_CUDA;
}
}  // namespace

iso_status make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                          uint32_t box_cols, uint32_t box_rows) {
  return make_tmap_2d(map, base, rows, cols, ld, box_cols, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

iso_status make_tmap_bf16_sw64(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                               uint32_t box_cols, uint32_t box_rows) {
  return make_tmap_2d(map, base, rows, cols, ld, box_cols, box_rows, CU_TENSOR_MAP_SWIZZLE_64B);
}

// Tensor map over a 3-D bf16 array [d2][d1][d0] (d0 innermost, contiguous), strides s1 and s2
// (elements) between consecutive d1 and d2 entries, box {b0, b1, b2}, 128-byte swizzle.
iso_status make_tmap_bf16_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                             uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
  if (!resolve_encode()) return ISO_ERR_CUDA;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1 * 2, s2 * 2};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ISO_OK : ISO_ERR_CUDA;
}

namespace {

// A box rows and the stage count that fits the shared-memory budget.  By default an even count
// (the output staging area usually fits beside it); epilogues that store no rows (the logprob
// statistics) take every stage that fits (the two leaf-parity streams split an odd count).
void set_a_rows(GemmParams& p, int a_rows, bool row_output = true) {
  p.a_rows = a_rows;
  p.a_bytes = a_rows * p.stage_k * 2;
  const int b_bytes = p.pair ? p.stage_k * 64 * 2 : B_STAGE_BYTES;  // a CTA of a pair holds half the B tile
  // the parked subtree root (spill), or a leaf group's root in cluster mode (the A box's rows only)
  const int reserve = p.spill ? SPILL_BYTES : (p.cluster > 1 ? a_rows * BN * 4 : 0);
  const int room = GEMM_SMEM_BYTES - 1024 - GEMM_BARRIER_BYTES - reserve;
  int st = room / (p.a_bytes + b_bytes);
  if (st > MAX_STAGES) st = MAX_STAGES;
  p.stages = row_output ? (st & ~1) : st;
  p.epi_staged = (row_output && room - p.stages * (p.a_bytes + b_bytes) >= EPI_STAGE_BYTES) ? 1 : 0;
}

// Whole-leaf stages (leaves of 96 k, bf16 roots on one CTA): a stage holds a leaf, A in a
// 64-column and a 32-column box, B in 96-row boxes; the stage count that fits.
void set_leaf_stage(GemmParams& p) {
  p.leaf_stage = 1;
  p.kb_per_leaf = 1;
  p.a_rows = BM;
  p.a_bytes = LS_A_BYTES;
  const int room = GEMM_SMEM_BYTES - 1024 - GEMM_BARRIER_BYTES - (p.spill ? SPILL_BYTES : 0);
  int st = room / (LS_A_BYTES + LS_B_BYTES);
  if (st > MAX_STAGES) st = MAX_STAGES;
  p.stages = st & ~1;
  p.epi_staged = (room - p.stages * (LS_A_BYTES + LS_B_BYTES) >= EPI_STAGE_BYTES) ? 1 : 0;
}

// Row blocks per raster group of the GEMM unit order: the CTAs running at once share a few
// B column tiles and sweep the group's row blocks, so the group's A rows (row blocks x K)
// should stay in L2 while the B tiles stream through once per group.  48 MB of the 129 MB L2
// for A leaves room for the B tiles in flight and the outputs (a sweep of 16-96 MB on the
// M = 4096 projections: 48 best; 8 fixed row blocks re-read B ~4x from HBM at K = 4096,
// N = 12288, 1242 -> 1369 TFLOP/s).  The logprob passes a smaller budget (below).
int raster_group(const GemmParams& p, int K, int budget_mb = 48) {
  const int64_t unit_rows = p.pair ? 2 * BM : BM;
  const int64_t a_bytes = unit_rows * static_cast<int64_t>(K) * 2;
  int64_t g = (static_cast<int64_t>(budget_mb) << 20) / a_bytes;
  if (g < 1) g = 1;
  if (g > p.m_blocks) g = p.m_blocks;
  return static_cast<int>(g);
}

// CTA pairs (M = 256 per MMA): units of 256 rows, 128-row A boxes, half the B tile per CTA.
// A pair issues half the MMA instructions per SM and moves fewer bytes per MMA (more stages in
// flight).  Its fixed cost is at every tile boundary: the next tile's leaves take TMEM buffers
// that both CTAs' epilogues must release (the last tree steps hold three of the four).
// Measured on GB300 (same-box A/B, bits identical): with leaves of 512 k the pairs win
// (4096 x 4096 x 4096: 1188 -> 1409 TFLOP/s; 4096 x 4096 x 12288: 1350 -> 1596; the T = 4096
// logprob 3.50 -> 3.01 ms); with 256 k they tie and with 128 k they lose (745 -> 668).
constexpr int kPairMinLeafLen = 512;
bool use_pair(int rows, int K, int L) { return rows > BM && K / L >= kPairMinLeafLen; }

// One leaf: one producer thread feeds the pair, and 128-k stages halve its TMA instructions per
// byte (measured on GB300, same-box A/B, bits identical: 4096 x 4096 x 4096 with one leaf 1192 ->
// 1449 TFLOP/s).  With two producers the 64-k stages stay: 128-k stages release their shared
// memory in larger steps, leaving fewer bytes in flight (8 leaves: 1389 -> 1361 TFLOP/s, the
// T = 32768 logprob 28.4 -> 29.6 ms; 16 leaves, 2 stages: 1304 -> 885).
void set_pair(GemmParams& p, int rows, bool row_output = true) {
  p.pair = 1;
  p.m_blocks = div_up(rows, 2 * BM);
  if (p.L == 1 && p.leaf_len % 64 == 0) {
    p.stage_k = PAIR_BK;
    p.kb_per_leaf = div_up(p.leaf_len, PAIR_BK);
  }
  set_a_rows(p, 128, row_output);
}

// A tensor maps of CTA pairs.  With 128-k stages a 3-D view {64 k, rows, K / 64 k-chunks} of the
// row-major [rows x K] matrix (strides ld * 2 and 128 bytes), box {64, 128, 2}: one TMA brings a
// CTA's [128 x 128] A stage as two consecutive 128-byte-swizzled [128 x 64] tiles.
iso_status make_tmap_a(CUtensorMap* map, const GemmParams& p, const void* A, int rows, int K, int64_t ld) {
  if (p.stage_k == PAIR_BK)
    return make_tmap_bf16_3d(map, A, 64, static_cast<uint64_t>(rows), static_cast<uint64_t>(K / 64),
                             static_cast<uint64_t>(ld), 64, 64, 128, 2);
  return make_tmap_bf16(map, A, rows, K, ld, BK, static_cast<uint32_t>(p.a_rows));
}

// Smallest A box that covers a single row block of `rows` rows.
int a_rows_for(int rows) {
  if (rows <= 16) return 16;
  if (rows <= 32) return 32;
  if (rows <= 64) return 64;
  return 128;
}

GemmParams base_params(int M, int N, int K, int L) {
  GemmParams p;
  memset(&p, 0, sizeof p);
  p.M = M;
  p.N = N;
  p.K = K;
  p.L = L;
  p.spill = L > TMEM_TREE_LEAVES ? 1 : 0;
  p.leaf_len = K / L;
  p.num_kb = div_up(K, BK);
  p.stage_k = BK;
  p.kb_per_leaf = div_up(K / L, BK);
  p.m_blocks = div_up(M, BM);
  p.n_blocks = div_up(N, BN);
  p.group_m = 8;
  p.b_tile_cols = BN;
  p.b_box2_off = 64;
  set_a_rows(p, 128);
  p.out_rows = M;
  p.status = device_status_ptr();
  p.timeout_ns = wait_timeout_ns();
  return p;
}

// Shared checks of a leaf-tree GEMM launch.
iso_status check_gemm_args(const void* A, int64_t lda, const void* B, int64_t ldb, const void* C, int64_t ldc,
                           int ldc_mult, int M, int N, int K, int L) {
  if (M < 0 || N <= 0 || K <= 0) return ISO_ERR_INVALID_ARG;
  if (M > 0 && (!A || !B || !C)) return ISO_ERR_INVALID_ARG;
  if (L > MAX_LEAVES) return ISO_ERR_UNSUPPORTED;
  if (K % (UMMA_K * L) != 0) return ISO_ERR_SHAPE;
  if (N % 8 != 0) return ISO_ERR_SHAPE;
  if (lda < K || ldb < N || ldc < N) return ISO_ERR_INVALID_ARG;
  if (lda % 8 || ldb % 8 || ldc % ldc_mult) return ISO_ERR_ALIGNMENT;
  if (M > 0 && (!aligned16(A) || !aligned16(B) || !aligned16(C))) return ISO_ERR_ALIGNMENT;
  return ISO_OK;
}

// Leaf groups for one row block: with fewer 128-column tiles than SMs, the L leaves split into
// R groups (R a power of two <= min(L, 8), R x tiles <= SMs) that run as one cluster of R CTAs
// per tile, so R times as many SMs stream B, and the cluster combines the group roots with the
// top log2 R levels of the tree -- the partial + combine of R simulated ranks inside one launch,
// so the bits are the single pass's.  Needs all tiles' clusters resident at once.
int cluster_groups(int M, int N, int L) {
  if (M > BM) return 1;
  const int n_tiles = div_up(N, BN);
  int R = 1;
  while (R * 2 <= L && R * 2 <= MAX_CLUSTER_GROUPS && n_tiles * R * 2 <= sm_count()) R *= 2;
  while (R > 1 && cluster_gemm_capacity(R) < n_tiles) R /= 2;
  return R;
}

// iso_gemm for one row block on clusters of R leaf-group CTAs (EPI_CLUSTER).
iso_status run_gemm_cluster(const void* A, int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc, int M,
                            int N, int K, int L, int R, cudaStream_t s) {
  GemmParams p = base_params(M, N, K / R, L / R);  // per group: K / R columns of A, L / R leaves
  p.cluster = R;
  set_a_rows(p, a_rows_for(M));  // (the group root's shared-memory region comes off the stages)
  CUtensorMap tA, tB;
  iso_status st = make_tmap_bf16(&tA, A, M, K, lda, BK, static_cast<uint32_t>(p.a_rows));
  if (st != ISO_OK) return st;
  st = make_tmap_bf16(&tB, B, K, N, ldb, 64, BK);
  if (st != ISO_OK) return st;
  p.unit_mode = UNIT_CLUSTER;
  p.num_units = p.n_blocks * R;
  p.b_stream = 1;
  p.out = C;
  p.ldo = ldc;
  trace("gemm[cluster leaf groups]", M, N, K, R);
  return launch_gemm(EPI_CLUSTER, tA, tB, p, p.num_units, s);
}

iso_status run_gemm(int epi, const void* A, int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc, int M,
                    int N, int K, int L, cudaStream_t s) {
  if (!ensure_device_state()) return ISO_ERR_CUDA;
  if (epi == EPI_BF16 && M <= BM) {
    const int R = cluster_groups(M, N, L);
    if (R > 1) return run_gemm_cluster(A, lda, B, ldb, C, ldc, M, N, K, L, R, s);
  }
  GemmParams p = base_params(M, N, K, L);
  if (p.m_blocks == 1)
    set_a_rows(p, a_rows_for(M));
  else if (use_pair(M, K, L))
    set_pair(p, M);
  CUtensorMap tA, tB;
  iso_status st = make_tmap_a(&tA, p, A, M, K, lda);
  if (st != ISO_OK) return st;
  st = make_tmap_bf16(&tB, B, K, N, ldb, 64, static_cast<uint32_t>(p.stage_k));
  if (st != ISO_OK) return st;
  p.unit_mode = UNIT_GEMM;
  p.num_units = p.m_blocks * p.n_blocks;
  p.group_m = raster_group(p, K);
  p.b_stream = p.m_blocks == 1 ? 1 : 0;
  p.out = C;
  p.ldo = ldc;
  trace(epi == EPI_BF16 ? "gemm" : "gemm_partial", M, N, K, L);
  return launch_gemm(epi, tA, tB, p, p.num_units, s);
}

// The leaf-tree GEMM of y = rmsnorm(x) and B with the normalisation in the A prologue: the
// producer warps build each A stage from x, rinv and gamma (one CTA per unit, 128-row A boxes).
iso_status run_gemm_rmsnorm(const void* x, const float* rinv, const void* gamma, const void* B, int64_t ldb, void* C,
                            int64_t ldc, int M, int N, int K, int L, cudaStream_t s) {
  GemmParams p = base_params(M, N, K, L);
  set_a_rows(p, 128);
  p.a_transform = 1;
  p.a_src = x;
  p.lda_src = K;
  p.a_rinv = rinv;
  p.a_gamma = gamma;
  CUtensorMap tA, tB;
  iso_status st = make_tmap_bf16(&tA, x, M, K, K, BK, 128);  // unused by the kernel in this mode
  if (st != ISO_OK) return st;
  st = make_tmap_bf16(&tB, B, K, N, ldb, 64, BK);
  if (st != ISO_OK) return st;
  p.unit_mode = UNIT_GEMM;
  p.num_units = p.m_blocks * p.n_blocks;
  p.group_m = raster_group(p, K);
  p.out = C;
  p.ldo = ldc;
  trace("rmsnorm_gemm", M, N, K, L);
  return launch_gemm(EPI_BF16, tA, tB, p, p.num_units, s);
}

}  // namespace

}  // namespace iso

using namespace iso;

extern "C" {

iso_status iso_last_device_status(iso_stream stream) {
  if (!ensure_device_state()) return ISO_ERR_CUDA;
  if (cudaStreamSynchronize(S(stream)) != cudaSuccess) return ISO_ERR_CUDA;
  unsigned int w = 0;
  if (cudaMemcpy(&w, device_status_ptr(), sizeof w, cudaMemcpyDeviceToHost) != cudaSuccess) return ISO_ERR_CUDA;
  const unsigned int zero = 0;
  if (cudaMemcpy(device_status_ptr(), &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return ISO_ERR_CUDA;
  if (w & kDevTimeout) return ISO_ERR_DEVICE_TIMEOUT;
  if (w & kDevCheck) return ISO_ERR_DEVICE_CHECK;
  if (w & kDevBadToken) return ISO_ERR_BAD_TOKEN_ID;
  if (w) return ISO_ERR_SHAPE;
  return ISO_OK;
}

iso_status iso_gemm(const iso_contract* c, const iso_bf16* A, int64_t lda, const iso_bf16* B, int64_t ldb,
                    iso_bf16* C, int64_t ldc, int M, int N, int K, iso_stream stream) {
  if (!c) return ISO_ERR_INVALID_ARG;
  const int L = iso_contract_leaf_count(c);
  iso_status st = check_gemm_args(A, lda, B, ldb, C, ldc, 8, M, N, K, L);
  if (st != ISO_OK || M == 0) return st;
  return run_gemm(EPI_BF16, A, lda, B, ldb, C, ldc, M, N, K, L, S(stream));
}

size_t iso_gemm_workspace(const iso_contract* c, int M, int N, int K) {
  if (!c || M < 0 || N <= 0 || K <= 0) return 0;
  if (M > BM) return 0;  // the leaf split serves problems of one row block
  const int L = iso_contract_leaf_count(c);
  return static_cast<size_t>(L) * static_cast<size_t>(M) * static_cast<size_t>(N) * sizeof(float);
}

iso_status iso_gemm_ws(const iso_contract* c, const iso_bf16* A, int64_t lda, const iso_bf16* B, int64_t ldb,
                       iso_bf16* C, int64_t ldc, int M, int N, int K, void* ws, size_t ws_bytes, iso_stream stream) {
  if (!c) return ISO_ERR_INVALID_ARG;
  const int L = iso_contract_leaf_count(c);
  iso_status st = check_gemm_args(A, lda, B, ldb, C, ldc, 8, M, N, K, L);
  if (st != ISO_OK || M == 0) return st;
  if (!ensure_device_state()) return ISO_ERR_CUDA;
  // With a workspace the groups run as plain CTAs and the combine as a second, dependent launch
  // (its launch overlaps the GEMM's tail), which measured faster than iso_gemm's one-launch
  // cluster schedule on GB300: M = 1, 4096 x 4096, R = 4: 19.1 -> 17.0 us after an L2 flush,
  // 12.4 -> 11.5 us back to back; 12288 x 4096: 23.1 -> 21.2 us back to back.
  // Leaf groups: with one row block and fewer column tiles than SMs, R groups of L/R leaves run
  // as separate units (R = the largest power of two <= L with R x tiles <= SMs); each writes
  // its group's fp32 subtree root to ws and the tree combine applies the top log2 R levels --
  // iso_gemm_leaf_partial + iso_tree_combine over R simulated ranks, the same bits as iso_gemm.
  const int n_tiles = div_up(N, BN);
  int R = 1;
  if (M <= BM && ws != nullptr && aligned16(ws))
    while (R * 2 <= L && n_tiles * R * 2 <= sm_count() &&
           ws_bytes >= static_cast<size_t>(R) * 2 * static_cast<size_t>(M) * N * sizeof(float))
      R *= 2;
  if (R == 1) return run_gemm(EPI_BF16, A, lda, B, ldb, C, ldc, M, N, K, L, S(stream));
  GemmParams p = base_params(M, N, K / R, L / R);
  set_a_rows(p, a_rows_for(M));
  CUtensorMap tA, tB;
  st = make_tmap_bf16(&tA, A, M, K, lda, BK, static_cast<uint32_t>(p.a_rows));
  if (st != ISO_OK) return st;
  st = make_tmap_bf16(&tB, B, K, N, ldb, 64, BK);
  if (st != ISO_OK) return st;
  float* S_all = static_cast<float*>(ws);
  p.unit_mode = UNIT_LEAF_SPLIT;
  p.num_units = R * p.n_blocks;
  p.b_stream = 1;
  p.out = S_all;
  p.ldo = N;
  p.out_group_stride = static_cast<int64_t>(M) * N;
  trace("gemm[leaf groups]", M, N, K, R);
  st = launch_gemm(EPI_F32, tA, tB, p, p.num_units, S(stream));
  if (st != ISO_OK) return st;
  return launch_tree_combine(S_all, N, static_cast<int64_t>(M) * N, R, reinterpret_cast<uint16_t*>(C), ldc, M, N,
                             S(stream)) == cudaSuccess
             ? ISO_OK
             : ISO_ERR_CUDA;
}

iso_status iso_gemm_leaf_partial(const iso_contract* c, int rank, int num_ranks, const iso_bf16* A_r, int64_t lda,
                                 const iso_bf16* B_r, int64_t ldb, float* S_r, int64_t lds, int M, int N,
                                 int K_local, iso_stream stream) {
  if (!c) return ISO_ERR_INVALID_ARG;
  iso_status st = iso_contract_check_topology(c, num_ranks);
  if (st != ISO_OK) return st;
  if (rank < 0 || rank >= num_ranks) return ISO_ERR_INVALID_ARG;
  const int Lr = iso_contract_leaf_count(c) / num_ranks;
  st = check_gemm_args(A_r, lda, B_r, ldb, S_r, lds, 4, M, N, K_local, Lr);
  if (st != ISO_OK || M == 0) return st;
  return run_gemm(EPI_F32, A_r, lda, B_r, ldb, S_r, lds, M, N, K_local, Lr, S(stream));
}

iso_status iso_tree_combine(const iso_contract* c, int num_ranks, const float* Sp, int64_t lds, int64_t rank_stride,
                            iso_bf16* C, int64_t ldc, int M, int N, iso_stream stream) {
  if (!c) return ISO_ERR_INVALID_ARG;
  iso_status st = iso_contract_check_topology(c, num_ranks);
  if (st != ISO_OK) return st;
  if (M < 0 || N <= 0) return ISO_ERR_INVALID_ARG;
  if (M == 0) return ISO_OK;
  if (!Sp || !C) return ISO_ERR_INVALID_ARG;
  if (N % 8 != 0) return ISO_ERR_SHAPE;
  if (lds < N || ldc < N || (num_ranks > 1 && rank_stride < static_cast<int64_t>(M) * lds)) return ISO_ERR_INVALID_ARG;
  if (lds % 4 || rank_stride % 4 || ldc % 8 || !aligned16(Sp) || !aligned16(C)) return ISO_ERR_ALIGNMENT;
  if (!ensure_device_state()) return ISO_ERR_CUDA;
  return launch_tree_combine(Sp, lds, rank_stride, num_ranks, C, ldc, M, N, S(stream)) == cudaSuccess ? ISO_OK
                                                                                                     : ISO_ERR_CUDA;
}

iso_status iso_rmsnorm(const iso_contract* c, const iso_bf16* x, const iso_bf16* gamma, float eps, iso_bf16* y,
                       int T, int H, iso_stream stream) {
  if (!c || T < 0 || H <= 0) return ISO_ERR_INVALID_ARG;
  if (T == 0) return ISO_OK;
  if (!x || !gamma || !y) return ISO_ERR_INVALID_ARG;
  if (H % 8 != 0) return ISO_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(gamma) || !aligned16(y)) return ISO_ERR_ALIGNMENT;
  if (!(eps >= 0.0f)) return ISO_ERR_INVALID_ARG;
  if (!ensure_device_state()) return ISO_ERR_CUDA;
  trace("rmsnorm", T, H, 0, 0);
  return launch_rmsnorm(x, gamma, eps, y, T, H, S(stream)) == cudaSuccess ? ISO_OK : ISO_ERR_CUDA;
}

static int lp_num_tiles(int V) { return div_up(V, LP_TILE_COLS); }
static int lp_num_chunks(int V) { return div_up(lp_num_tiles(V), LP_CHUNK_TILES); }

// Work units of the LM-head GEMM.  Tile units: every 128-column tile of a row block is its
// own unit; its statistics go to a per-tile array and a fold kernel forms each chunk's entry by
// folding the chunk's tiles left to right.  Chunk units: one CTA owns a whole chunk of a row
// block and folds its tiles itself.  Same fold, same bits.  Tile units balance the last wave
// (a chunk unit is ~290 us at T = 4096) and keep every SM busy at small T; measured on GB300 at
// H = 4096, V = 151936: T = 4096 3.85 -> 3.57 ms, T = 1024 1.21 -> 1.06 ms.  They need the
// per-tile statistics array ([tiles][T] fp32 pairs, 38 MB at T = 4096), so a workspace
// without room for it runs chunk units.

static size_t al256(size_t x) { return (x + 255) & ~size_t(255); }
// Workspace: [tile statistics, tile mode only] [chunk statistics] [z_sel], each 256-aligned.
static size_t lp_tile_stats_bytes(int T, int V) { return al256(static_cast<size_t>(T) * lp_num_tiles(V) * sizeof(float2)); }
static size_t lp_chunk_ws_bytes(int T, int V) {
  return al256(static_cast<size_t>(T) * lp_num_chunks(V) * sizeof(float2)) + al256(static_cast<size_t>(T) * sizeof(float));
}
static size_t lp_full_ws_bytes(int T, int V) { return lp_tile_stats_bytes(T, V) + lp_chunk_ws_bytes(T, V); }

size_t iso_selected_logprob_workspace(const iso_contract* c, int T, int V) {
  if (!c || T < 0 || V <= 0) return 0;
  return lp_full_ws_bytes(T, V);
}

size_t iso_selected_logprob_min_workspace(const iso_contract* c, int T, int V) {
  if (!c || T < 0 || V <= 0) return 0;
  return lp_chunk_ws_bytes(T, V);
}

// The statistics pass of the selected-token logprob over the vocabulary columns [sel_base,
// sel_base + Vl) held by W ([H x Vl], leading dimension ldw): chunk statistics [Cl x T] into
// chunk_stats and z at each row's id (when the id falls in these columns) into zsel.  With
// tile_stats (room for [tiles x T]) every 128-column tile is its own unit and a fold kernel forms
// the chunk entries; otherwise one CTA folds a whole chunk.  Same fold, same bits.
// With rinv (the fused RMSNorm prologue) h holds the raw states x and the A stages are built
// as bf16((x * rinv[t]) * gamma[i]) by the producer warps (one CTA per unit, 128-row boxes).
static iso_status run_logprob_stats(const iso_contract* c, const iso_bf16* h, const iso_bf16* W, int64_t ldw,
                                    const int32_t* ids, int T, int H, int Vl, int sel_base, float2* chunk_stats,
                                    float* zsel, float2* tile_stats, cudaStream_t s, const float* rinv = nullptr,
                                    const iso_bf16* gamma = nullptr) {
  const int L = iso_contract_leaf_count(c);
  GemmParams p = base_params(T, Vl, H, L);
  if (rinv != nullptr) {
    p.a_transform = 1;
    p.a_src = h;
    p.lda_src = H;
    p.a_rinv = rinv;
    p.a_gamma = gamma;
  } else if (p.m_blocks == 1) {
    set_a_rows(p, a_rows_for(T), false);  // the statistics epilogue stores no rows
  } else if (use_pair(T, H, L)) {
    set_pair(p, T, false);
  }
  CUtensorMap tA, tB;
  iso_status st = make_tmap_a(&tA, p, h, T, H, H);
  if (st != ISO_OK) return st;
  st = make_tmap_bf16(&tB, W, H, Vl, ldw, 64, static_cast<uint32_t>(p.stage_k));
  if (st != ISO_OK) return st;
  const bool tiles = tile_stats != nullptr;
  p.unit_mode = UNIT_LOGPROB;
  p.chunk_tiles = tiles ? 1 : LP_CHUNK_TILES;                   // tiles per work unit
  p.num_chunks = tiles ? lp_num_tiles(Vl) : lp_num_chunks(Vl);  // statistics entries per row
  p.num_units = p.m_blocks * p.num_chunks;
  // row blocks whose hidden states share L2: 32 MB of them (16 pair row blocks at H = 4096).
  // Measured on GB300 (same box, interleaved, bits identical) against 48 MB: T = 65536 59.96 ->
  // 55.76 ms, T = 8192 and 16384 within 2 %; at T = 4096 both budgets cover all 16 blocks.
  p.group_m = raster_group(p, H, 32);
  p.b_stream = p.m_blocks == 1 ? 1 : 0;
  p.ids = ids;
  p.ws_stats = tiles ? tile_stats : chunk_stats;
  p.ws_zsel = zsel;
  p.V = Vl;
  p.sel_base = sel_base;
  trace(tiles ? "selected_logprob[tile units]" : "selected_logprob[chunk units]", T, H, Vl, p.num_chunks);
  st = launch_gemm(EPI_LOGPROB, tA, tB, p, p.num_units, s);
  if (st != ISO_OK || !tiles) return st;
  return launch_lse_fold_tiles(tile_stats, chunk_stats, T, lp_num_chunks(Vl), lp_num_tiles(Vl), LP_CHUNK_TILES, s) ==
                 cudaSuccess
             ? ISO_OK
             : ISO_ERR_CUDA;
}

// iso_selected_logprob and its fused-RMSNorm form (gamma != NULL: h holds the raw states and
// the workspace starts with the per-row factors).
static iso_status selected_logprob_impl(const iso_contract* c, const iso_bf16* h, const iso_bf16* gamma, float eps,
                                        const iso_bf16* W, const int32_t* ids, float* out, int T, int H, int V,
                                        void* ws, size_t ws_bytes, cudaStream_t s) {
  if (!c || T < 0 || H <= 0 || V <= 0) return ISO_ERR_INVALID_ARG;
  if (T == 0) return ISO_OK;
  if (!h || !W || !ids || !out || !ws) return ISO_ERR_INVALID_ARG;
  const int L = iso_contract_leaf_count(c);
  if (H % (UMMA_K * L) != 0) return ISO_ERR_SHAPE;
  if (V % 8 != 0 || lp_num_chunks(V) > 256) return ISO_ERR_SHAPE;
  if (H % 8 != 0) return ISO_ERR_ALIGNMENT;
  if (!aligned16(h) || !aligned16(W) || !aligned16(ws) || !aligned16(out)) return ISO_ERR_ALIGNMENT;
  if (gamma != nullptr) {
    if (!aligned16(gamma)) return ISO_ERR_ALIGNMENT;
    if (!(eps >= 0.0f)) return ISO_ERR_INVALID_ARG;
  }
  const size_t pre = gamma != nullptr ? al256(static_cast<size_t>(T) * sizeof(float)) : 0;
  if (ws_bytes < pre + lp_chunk_ws_bytes(T, V)) return ISO_ERR_WORKSPACE;
  if (!ensure_device_state()) return ISO_ERR_CUDA;
  char* wsb = static_cast<char*>(ws);
  float* rinv = gamma != nullptr ? reinterpret_cast<float*>(wsb) : nullptr;
  wsb += pre;
  ws_bytes -= pre;
  const bool tiles = ws_bytes >= lp_full_ws_bytes(T, V);
  float2* tile_stats = tiles ? reinterpret_cast<float2*>(wsb) : nullptr;
  char* rest = wsb + (tiles ? lp_tile_stats_bytes(T, V) : 0);
  float2* chunk_stats = reinterpret_cast<float2*>(rest);
  float* zsel = reinterpret_cast<float*>(rest + al256(static_cast<size_t>(T) * lp_num_chunks(V) * sizeof(float2)));
  if (rinv != nullptr && launch_rms_rows(h, eps, rinv, T, H, H, s) != cudaSuccess) return ISO_ERR_CUDA;
  iso_status st = run_logprob_stats(c, h, W, V, ids, T, H, V, 0, chunk_stats, zsel, tile_stats, s, rinv, gamma);
  if (st != ISO_OK) return st;
  ShardBounds one;
  one.n = 1;
  one.chunk0[0] = 0;
  return launch_lse_combine(chunk_stats, zsel, ids, out, T, lp_num_chunks(V), V, one, s) == cudaSuccess
             ? ISO_OK
             : ISO_ERR_CUDA;
}

iso_status iso_selected_logprob(const iso_contract* c, const iso_bf16* h, const iso_bf16* W, const int32_t* ids,
                                float* out, int T, int H, int V, void* ws, size_t ws_bytes, iso_stream stream) {
  return selected_logprob_impl(c, h, nullptr, 0.f, W, ids, out, T, H, V, ws, ws_bytes, S(stream));
}

size_t iso_rmsnorm_selected_logprob_workspace(const iso_contract* c, int T, int V) {
  if (!c || T < 0 || V <= 0) return 0;
  return al256(static_cast<size_t>(T) * sizeof(float)) + lp_full_ws_bytes(T, V);
}

iso_status iso_rmsnorm_selected_logprob(const iso_contract* c, const iso_bf16* x, const iso_bf16* gamma, float eps,
                                        const iso_bf16* W, const int32_t* ids, float* out, int T, int H, int V,
                                        void* ws, size_t ws_bytes, iso_stream stream) {
  if (!gamma && T > 0) return ISO_ERR_INVALID_ARG;
  return selected_logprob_impl(c, x, gamma, eps, W, ids, out, T, H, V, ws, ws_bytes, S(stream));
}

size_t iso_rmsnorm_gemm_workspace(const iso_contract* c, int M) {
  if (!c || M < 0) return 0;
  return al256(static_cast<size_t>(M) * sizeof(float));
}

iso_status iso_rmsnorm_gemm(const iso_contract* c, const iso_bf16* x, const iso_bf16* gamma, float eps,
                            const iso_bf16* B, int64_t ldb, iso_bf16* C, int64_t ldc, int M, int N, int K, void* ws,
                            size_t ws_bytes, iso_stream stream) {
  if (!c) return ISO_ERR_INVALID_ARG;
  const int L = iso_contract_leaf_count(c);
  iso_status st = check_gemm_args(x, K, B, ldb, C, ldc, 8, M, N, K, L);
  if (st != ISO_OK || M == 0) return st;
  if (!gamma || !ws || !(eps >= 0.0f)) return ISO_ERR_INVALID_ARG;
  if (!aligned16(gamma) || !aligned16(ws)) return ISO_ERR_ALIGNMENT;
  if (ws_bytes < static_cast<size_t>(M) * sizeof(float)) return ISO_ERR_WORKSPACE;
  if (!ensure_device_state()) return ISO_ERR_CUDA;
  float* rinv = static_cast<float*>(ws);
  if (launch_rms_rows(x, eps, rinv, M, K, K, S(stream)) != cudaSuccess) return ISO_ERR_CUDA;
  return run_gemm_rmsnorm(x, rinv, gamma, B, ldb, C, ldc, M, N, K, L, S(stream));
}

size_t iso_selected_logprob_partial_workspace(const iso_contract* c, int T, int V_r) {
  if (!c || T < 0 || V_r <= 0) return 0;
  return lp_tile_stats_bytes(T, V_r);
}

iso_status iso_selected_logprob_partial(const iso_contract* c, const iso_bf16* h, const iso_bf16* W_r, int64_t ldw,
                                        const int32_t* ids, int T, int H, int V, int v0, int V_r, float* stats_r,
                                        float* zsel_r, void* ws, size_t ws_bytes, iso_stream stream) {
  constexpr int kChunkCols = LP_TILE_COLS * LP_CHUNK_TILES;
  if (!c || T < 0 || H <= 0 || V <= 0 || V_r <= 0 || v0 < 0) return ISO_ERR_INVALID_ARG;
  if (v0 % kChunkCols != 0 || v0 + V_r > V || (v0 + V_r != V && V_r % kChunkCols != 0)) return ISO_ERR_SHAPE;
  if (T == 0) return ISO_OK;
  if (!h || !W_r || !ids || !stats_r || !zsel_r) return ISO_ERR_INVALID_ARG;
  const int L = iso_contract_leaf_count(c);
  if (H % (UMMA_K * L) != 0) return ISO_ERR_SHAPE;
  if (V % 8 != 0 || V_r % 8 != 0 || lp_num_chunks(V) > 256) return ISO_ERR_SHAPE;
  if (ldw < V_r || ldw % 8 != 0 || H % 8 != 0) return ISO_ERR_ALIGNMENT;
  if (!aligned16(h) || !aligned16(W_r) || !aligned16(stats_r) || (ws && !aligned16(ws))) return ISO_ERR_ALIGNMENT;
  if (!ensure_device_state()) return ISO_ERR_CUDA;
  float2* tile_stats =
      (ws != nullptr && ws_bytes >= lp_tile_stats_bytes(T, V_r)) ? static_cast<float2*>(ws) : nullptr;
  return run_logprob_stats(c, h, W_r, ldw, ids, T, H, V_r, v0, reinterpret_cast<float2*>(stats_r), zsel_r, tile_stats,
                           S(stream));
}

iso_status iso_selected_logprob_combine(const iso_contract* c, int num_shards, const int* shard_v0,
                                        const float* stats, const float* zsel, const int32_t* ids, float* out, int T,
                                        int V, iso_stream stream) {
  constexpr int kChunkCols = LP_TILE_COLS * LP_CHUNK_TILES;
  if (!c || T < 0 || V <= 0 || !shard_v0) return ISO_ERR_INVALID_ARG;
  if (num_shards < 1 || num_shards > kMaxVocabShards) return ISO_ERR_UNSUPPORTED;
  if (V % 8 != 0 || lp_num_chunks(V) > 256) return ISO_ERR_SHAPE;
  ShardBounds sb;
  sb.n = num_shards;
  for (int r = 0; r < num_shards; ++r) {
    if (shard_v0[r] % kChunkCols != 0 || shard_v0[r] >= V) return ISO_ERR_SHAPE;
    if ((r == 0 && shard_v0[r] != 0) || (r > 0 && shard_v0[r] <= shard_v0[r - 1])) return ISO_ERR_SHAPE;
    sb.chunk0[r] = shard_v0[r] / kChunkCols;
  }
  if (T == 0) return ISO_OK;
  if (!stats || !zsel || !ids || !out) return ISO_ERR_INVALID_ARG;
  if (!ensure_device_state()) return ISO_ERR_CUDA;
  return launch_lse_combine(reinterpret_cast<const float2*>(stats), zsel, ids, out, T, lp_num_chunks(V), V, sb,
                            S(stream)) == cudaSuccess
             ? ISO_OK
             : ISO_ERR_CUDA;
}

iso_status iso_moe_route(const iso_contract* c, const float* logits, int T, int E, int k, int32_t* topk_ids,
                         float* topk_w, iso_stream stream) {
  if (!c || T < 0 || E <= 0 || k <= 0) return ISO_ERR_INVALID_ARG;
  if (E > MOE_MAX_EXPERTS || k > E || k > 32) return ISO_ERR_UNSUPPORTED;
  if (T == 0) return ISO_OK;
  if (!logits || !topk_ids || !topk_w) return ISO_ERR_INVALID_ARG;
  if (!ensure_device_state()) return ISO_ERR_CUDA;
  return launch_moe_route(logits, T, E, k, topk_ids, topk_w, S(stream)) == cudaSuccess ? ISO_OK : ISO_ERR_CUDA;
}

size_t iso_moe_permute_workspace(int T, int E, int k) {
  if (T < 0 || E <= 0 || k <= 0) return 0;
  const int64_t C = moe_perm_chunks(static_cast<int64_t>(T) * k);
  return sizeof(int32_t) * static_cast<size_t>(3 * E + 2 + C * E);
}

iso_status iso_moe_permute(const iso_contract* c, const int32_t* topk_ids, int T, int E, int k,
                           const int32_t* expert_partition, int partition, int32_t* perm, int32_t* offsets,
                           int32_t* counts_ws, iso_stream stream) {
  if (!c || T < 0 || E <= 0 || k <= 0 || E > MOE_MAX_EXPERTS) return ISO_ERR_INVALID_ARG;
  if (!topk_ids || !perm || !offsets || !counts_ws) return ISO_ERR_INVALID_ARG;
  if (!ensure_device_state()) return ISO_ERR_CUDA;
  // counts_ws: counts [E] | unit prefixes [E+1] x 2 (not needed by a caller of the plain
  // permutation) | chunk histogram [chunks x E]
  int32_t* up = counts_ws + E;
  int32_t* dn = up + (E + 1);
  int32_t* hist = dn + (E + 1);
  return launch_moe_permute(topk_ids, static_cast<int64_t>(T) * k, E, expert_partition, partition, counts_ws, hist,
                            perm, offsets, up, 1, dn, 1, BM, BM, S(stream)) == cudaSuccess
             ? ISO_OK
             : ISO_ERR_CUDA;
}

iso_status iso_moe_combine(const iso_contract* c, const iso_bf16* y_slots, const float* topk_w, iso_bf16* out, int T,
                           int k, int H, iso_stream stream) {
  if (!c || T < 0 || H <= 0 || k <= 0) return ISO_ERR_INVALID_ARG;
  if (!is_pow2(k) || k > 8) return ISO_ERR_UNSUPPORTED;
  if (T == 0) return ISO_OK;
  if (!y_slots || !topk_w || !out) return ISO_ERR_INVALID_ARG;
  if (H % 8 != 0) return ISO_ERR_SHAPE;
  if (!aligned16(y_slots) || !aligned16(out)) return ISO_ERR_ALIGNMENT;
  if (!ensure_device_state()) return ISO_ERR_CUDA;
  return launch_moe_combine(y_slots, topk_w, T, k, H, out, S(stream)) == cudaSuccess ? ISO_OK : ISO_ERR_CUDA;
}

// The expert layer's grouped GEMMs run on single CTAs (units of 128 rows of one expert).  CTA
// pairs (256-row units) measured slower on GB300 at T = 8192, H = 2048, F = 768, E = 128, k = 8,
// bits identical: 0.861 ms per layer on single CTAs, 1.008 with pairs for gate/up, 0.997 for
// down, 1.137 for both (an expert's ~512 rows leave a ragged 256-row unit more often than a
// ragged 128-row one, and the short leaves gain little from the smaller per-SM operand stream).

// Workspace layout of the expert layer (each region 256-byte aligned):
//   y_slots [P x H] bf16 (the full layer only; iso_moe_experts_partial writes the caller's) |
//   x_perm [P x H] bf16 | h [P x F] bf16 |
//   perm [P] | offsets [E+1] | counts [E] | up_prefix [E+1] | down_prefix [E+1] | part_map [E] |
//   hist [chunks x E] (the permutation's chunk histogram)
namespace {
struct MoeWs {
  size_t y, xp, h, perm, offs, counts, up, dn, part, hist, total;
};
size_t al(size_t x) { return (x + 255) & ~size_t(255); }
MoeWs moe_ws_layout(int T, int E, int k, int H, int F, bool with_y) {
  const size_t P = static_cast<size_t>(T) * k;
  MoeWs w;
  size_t o = 0;
  w.y = o; if (with_y) o += al(P * H * 2);
  w.xp = o; o += al(P * H * 2);
  w.h = o; o += al(P * F * 2);
  w.perm = o; o += al(P * 4);
  w.offs = o; o += al((E + 1) * 4);
  w.counts = o; o += al(E * 4);
  w.up = o; o += al((E + 1) * 4);
  w.dn = o; o += al((E + 1) * 4);
  w.part = o; o += al(E * 4);
  w.hist = o; o += al(static_cast<size_t>(moe_perm_chunks(static_cast<int64_t>(P))) * E * 4);
  w.total = o;
  return w;
}

// Shared argument checks of the expert-layer entry points.
iso_status check_moe_args(const iso_contract* c, int T, int E, int k, int H, int F) {
  if (!c || T < 0 || E <= 0 || k <= 0 || H <= 0 || F <= 0) return ISO_ERR_INVALID_ARG;
  if (E > MOE_MAX_EXPERTS || !is_pow2(k) || k > 8) return ISO_ERR_UNSUPPORTED;
  const int L = iso_contract_leaf_count(c);
  if (H % (UMMA_K * L) || F % (UMMA_K * L) || H % BN || F % 64) return ISO_ERR_SHAPE;
  return ISO_OK;
}

// The expert GEMMs of one partition (the experts e with part_map[e] == partition; all experts
// when part_map is null): permute the routing slots by expert, gather their token rows, the
// grouped gate/up GEMM with SwiGLU, and the grouped down GEMM, whose bf16 rows go to their
// routing slots in y [P x H].  Slots of other experts are not written.
iso_status moe_experts_pass(const iso_contract* c, const iso_bf16* x, const int32_t* topk_ids, const iso_bf16* W1,
                            const iso_bf16* W2, const int32_t* part_map, int partition, uint16_t* y, int T, int E,
                            int k, int H, int F, const MoeWs& lay, char* base, cudaStream_t s) {
  const int L = iso_contract_leaf_count(c);
  uint16_t* xp = reinterpret_cast<uint16_t*>(base + lay.xp);
  uint16_t* hb = reinterpret_cast<uint16_t*>(base + lay.h);
  int32_t* perm = reinterpret_cast<int32_t*>(base + lay.perm);
  int32_t* offs = reinterpret_cast<int32_t*>(base + lay.offs);
  int32_t* counts = reinterpret_cast<int32_t*>(base + lay.counts);
  int32_t* up = reinterpret_cast<int32_t*>(base + lay.up);
  int32_t* dn = reinterpret_cast<int32_t*>(base + lay.dn);
  int32_t* hist = reinterpret_cast<int32_t*>(base + lay.hist);
  const int64_t P = static_cast<int64_t>(T) * k;
  // the down projection's leaves of 96 k (F = 768 with 8 leaves) run on whole-leaf stages
  const bool leaf_stage = F / L == LS_LEAF && L <= TMEM_TREE_LEAVES;
  CUtensorMap tX, tW1, tH, tH2, tW2;
  iso_status st = make_tmap_bf16(&tX, xp, P, H, H, BK, BM);
  if (st == ISO_OK) st = make_tmap_bf16(&tW1, W1, static_cast<uint64_t>(E) * H, 2 * F, 2 * F, 64, BK);
  if (st == ISO_OK) st = make_tmap_bf16(&tH, hb, P, F, F, BK, BM);
  if (st == ISO_OK && leaf_stage) st = make_tmap_bf16_sw64(&tH2, hb, P, F, F, 32, BM);
  if (st == ISO_OK)
    st = make_tmap_bf16(&tW2, W2, static_cast<uint64_t>(E) * F, H, H, 64, leaf_stage ? LS_LEAF : BK);
  if (st != ISO_OK) return st;
  const int up_nb = F / 64, dn_nb = H / BN;
  // rows of an expert per grouped work unit: one row block for both GEMMs
  if (launch_moe_permute(topk_ids, P, E, part_map, partition, counts, hist, perm, offs, up, up_nb, dn, dn_nb, BM,
                         BM, s) != cudaSuccess)
    return ISO_ERR_CUDA;
  if (launch_moe_gather(x, perm, offs + E, P, k, H, xp, s) != cudaSuccess) return ISO_ERR_CUDA;
  // gate/up with SwiGLU fused: tile j pairs gate columns [64j, 64j+64) with up columns
  // [F+64j, F+64j+64) and writes h columns [64j, 64j+64).
  GemmParams p = base_params(0, F, H, L);
  p.n_blocks = F / 64;
  p.b_tile_cols = 64;
  p.b_box2_off = F;
  p.unit_mode = UNIT_GROUPED;
  p.g_offsets = offs;
  p.g_unit_prefix = up;
  p.E = E;
  p.out = hb;
  p.ldo = F;
  p.out_rows = P;
  st = launch_gemm(EPI_SWIGLU, tX, tW1, p, sm_count(), s);
  if (st != ISO_OK) return st;
  GemmParams q = base_params(0, H, F, L);
  q.unit_mode = UNIT_GROUPED;
  q.g_offsets = offs;
  q.g_unit_prefix = dn;
  q.E = E;
  q.out = y;
  q.ldo = H;
  q.out_rows = P;
  q.row_scatter = perm;
  if (leaf_stage) {
    set_leaf_stage(q);
    return launch_gemm(EPI_BF16, tH, tW2, q, sm_count(), s, &tH2);
  }
  return launch_gemm(EPI_BF16, tH, tW2, q, sm_count(), s);
}
}  // namespace

size_t iso_grouped_gemm_moe_workspace(const iso_contract* c, int T, int E, int k, int H, int F) {
  if (!c || T < 0 || E <= 0 || k <= 0 || H <= 0 || F <= 0) return 0;
  return moe_ws_layout(T, E, k, H, F, true).total;
}

iso_status iso_grouped_gemm_moe(const iso_contract* c, const iso_bf16* x, const int32_t* topk_ids,
                                const float* topk_w, const iso_bf16* W1, const iso_bf16* W2,
                                const int32_t* expert_partition, int num_partitions, iso_bf16* out, int T, int E,
                                int k, int H, int F, void* ws, size_t ws_bytes, iso_stream stream) {
  iso_status st = check_moe_args(c, T, E, k, H, F);
  if (st != ISO_OK) return st;
  if (T == 0) return ISO_OK;
  if (!x || !topk_ids || !topk_w || !W1 || !W2 || !out || !ws) return ISO_ERR_INVALID_ARG;
  if (expert_partition) {
    if (num_partitions <= 0) return ISO_ERR_INVALID_ARG;
    for (int e = 0; e < E; ++e)
      if (expert_partition[e] < 0 || expert_partition[e] >= num_partitions) return ISO_ERR_INVALID_ARG;
  } else {
    num_partitions = 1;
  }
  if (!aligned16(x) || !aligned16(W1) || !aligned16(W2) || !aligned16(out) || !aligned16(ws)) return ISO_ERR_ALIGNMENT;
  const MoeWs lay = moe_ws_layout(T, E, k, H, F, true);
  if (ws_bytes < lay.total) return ISO_ERR_WORKSPACE;
  if (!ensure_device_state()) return ISO_ERR_CUDA;
  cudaStream_t s = S(stream);
  char* base = static_cast<char*>(ws);
  uint16_t* y = reinterpret_cast<uint16_t*>(base + lay.y);
  int32_t* part = reinterpret_cast<int32_t*>(base + lay.part);
  if (expert_partition &&
      cudaMemcpyAsync(part, expert_partition, sizeof(int32_t) * E, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return ISO_ERR_CUDA;
  trace("grouped_gemm_moe", T, E, k, num_partitions);
  for (int pi = 0; pi < num_partitions; ++pi) {
    st = moe_experts_pass(c, x, topk_ids, W1, W2, expert_partition ? part : nullptr, pi, y, T, E, k, H, F, lay, base,
                          s);
    if (st != ISO_OK) return st;
  }
  return launch_moe_combine(y, topk_w, T, k, H, out, s) == cudaSuccess ? ISO_OK : ISO_ERR_CUDA;
}

size_t iso_moe_experts_partial_workspace(const iso_contract* c, int T, int E, int k, int H, int F) {
  if (!c || T < 0 || E <= 0 || k <= 0 || H <= 0 || F <= 0) return 0;
  return moe_ws_layout(T, E, k, H, F, false).total;
}

iso_status iso_moe_experts_partial(const iso_contract* c, const iso_bf16* x, const int32_t* topk_ids,
                                   const iso_bf16* W1, const iso_bf16* W2, const uint8_t* expert_mask,
                                   iso_bf16* y_slots, int T, int E, int k, int H, int F, void* ws, size_t ws_bytes,
                                   iso_stream stream) {
  iso_status st = check_moe_args(c, T, E, k, H, F);
  if (st != ISO_OK) return st;
  if (T == 0) return ISO_OK;
  if (!x || !topk_ids || !W1 || !W2 || !expert_mask || !y_slots || !ws) return ISO_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W1) || !aligned16(W2) || !aligned16(y_slots) || !aligned16(ws))
    return ISO_ERR_ALIGNMENT;
  const MoeWs lay = moe_ws_layout(T, E, k, H, F, false);
  if (ws_bytes < lay.total) return ISO_ERR_WORKSPACE;
  if (!ensure_device_state()) return ISO_ERR_CUDA;
  cudaStream_t s = S(stream);
  char* base = static_cast<char*>(ws);
  int32_t* part = reinterpret_cast<int32_t*>(base + lay.part);
  // the mask as a two-partition map, partition 1 = the masked experts (cudaMemcpyAsync from
  // pageable host memory returns once the source has been read, so a stack array is safe)
  int32_t map[MOE_MAX_EXPERTS];
  for (int e = 0; e < E; ++e) map[e] = expert_mask[e] ? 1 : 0;
  if (cudaMemcpyAsync(part, map, sizeof(int32_t) * E, cudaMemcpyHostToDevice, s) != cudaSuccess) return ISO_ERR_CUDA;
  trace("moe_experts_partial", T, E, k, 1);
  return moe_experts_pass(c, x, topk_ids, W1, W2, part, 1, reinterpret_cast<uint16_t*>(y_slots), T, E, k, H, F, lay,
                          base, s);
}

iso_status iso_selftest_bounded_wait(uint64_t timeout_ns, iso_stream stream) {
  if (timeout_ns == 0 || timeout_ns > 10000000000ull) return ISO_ERR_INVALID_ARG;
  if (!ensure_device_state()) return ISO_ERR_CUDA;
  return launch_bounded_wait_selftest(timeout_ns, S(stream)) == cudaSuccess ? ISO_OK : ISO_ERR_CUDA;
}

}  // extern "C"
