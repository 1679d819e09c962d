/*
 * iso.h -- C ABI of the parallelism-invariant GEMM / RMSNorm / MoE / selected-
 * token logprob library for NVIDIA GB300 (sm_103a).
 *
 * Promise: for a fixed library build and contract digest, every output row's
 * bits are a function of that row's inputs, the weights and the contract
 * only -- not of the batch size, the row's position in the batch, how K is
 * split across (simulated) tensor-parallel ranks, or how experts are split
 * across (simulated) expert-parallel partitions.
 *   [IsoExec: Unified Execution to Eliminate Trainer-Inference Mismatch in
 *    SkyRL, "Unified execution contract", "Parallelism-invariant kernels"]
 *   [VeXact paper "Diagnosing Training Inference Mismatch in LLM RL", §3.1:
 *    batch-invariant kernels fix tiling and reduction order]
 *
 * Conventions for every entry point:
 *   - bf16 tensors are passed as uint16_t bit patterns (iso_bf16).
 *   - Matrices are row-major with an explicit leading dimension in elements.
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or retains device memory.  Scratch space comes
 *     from the caller through the *_workspace() size queries.  The library
 *     owns only the host-side contract object.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *     is asynchronous on that stream and performs no implicit device sync.
 *   - Errors: every call returns an iso_status; arguments are validated on the
 *     host before anything is launched, and an invalid call launches nothing.
 *     No exception or abort crosses the ABI.  Faults detected on the device
 *     (a bounded wait that ran out of time, a token id outside [0, V)) set a
 *     per-device status word that iso_last_device_status() reads and clears.
 *   - Alignment: device pointers 16-byte aligned; leading dimensions of bf16
 *     matrices multiples of 8 elements, of fp32 matrices multiples of 4.
 *   - Per-device state (the status word's address, the SM count, the static
 *     scratch's address, kernel attributes) is looked up on a device's first
 *     call and kept for the life of the process: the library must not be used
 *     across a cudaDeviceReset of a device it has already run on.  Device
 *     ordinals 0-63 are served; host threads may call concurrently, on the
 *     same or different devices.
 */
#ifndef ISO_H_
#define ISO_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ISO_OK = 0,
  ISO_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad enum */
  ISO_ERR_SHAPE = 2,             /* shape outside the contract (e.g. K % (16 L) != 0) */
  ISO_ERR_ALIGNMENT = 3,         /* pointer / leading dimension alignment */
  ISO_ERR_UNPROVEN_TOPOLOGY = 4, /* rank count not a power of two dividing L */
  ISO_ERR_UNSUPPORTED = 5,       /* valid, but not supported by this library */
  ISO_ERR_CONTRACT_MISMATCH = 6, /* peer digest differs */
  ISO_ERR_WORKSPACE = 7,         /* workspace / buffer too small */
  ISO_ERR_CUDA = 8,              /* a CUDA runtime call failed */
  ISO_ERR_DEVICE_TIMEOUT = 9,    /* a device-side wait ran out of time */
  ISO_ERR_NOT_IMPLEMENTED = 10,
  ISO_ERR_BAD_TOKEN_ID = 11,     /* a token id outside [0, V) reached the device */
  ISO_ERR_DEVICE_CHECK = 12      /* debug build only: a device-side bounds check failed */
} iso_status;

typedef enum { ISO_TREE_BALANCED_BINARY = 0 } iso_tree_schedule;
typedef enum { ISO_F32 = 0, ISO_BF16 = 1 } iso_dtype;
typedef struct iso_contract iso_contract; /* opaque, immutable after init, thread-safe to share */
typedef uint16_t iso_bf16;                /* bf16 bit pattern */
typedef void* iso_stream;                 /* cudaStream_t */

/* ------------------------------------------------------------------ contract
 * [IsoExec blog, "Unified execution contract": composition constants, claims,
 *  identities (SHA-256 digests of the serialized contract)]
 *
 * iso_contract_init: leaf_count = number of contiguous K-leaves (a power of
 * two, 1..16 in this library); schedule must be ISO_TREE_BALANCED_BINARY;
 * acc_dtype must be ISO_F32; out_dtype must be ISO_BF16.  On success *out
 * receives a new contract (free with iso_contract_destroy) and digest (if not
 * NULL) the 32-byte SHA-256 of its canonical serialization, which covers every
 * constant that can change an output bit.  Errors: ISO_ERR_INVALID_ARG (bad
 * leaf count / NULL out), ISO_ERR_UNSUPPORTED (valid but not built). */
iso_status iso_contract_init(int leaf_count, iso_tree_schedule schedule, iso_dtype acc_dtype,
                             iso_dtype out_dtype, iso_contract** out, uint8_t digest[32]);
void iso_contract_destroy(iso_contract* c);
/* Canonical serialization (UTF-8 JSON, fixed field order, no whitespace).
 * *len receives the length without the terminating NUL; buf may be NULL to
 * query.  ISO_ERR_WORKSPACE if cap < len + 1. */
iso_status iso_contract_serialize(const iso_contract* c, char* buf, size_t cap, size_t* len);
iso_status iso_contract_digest(const iso_contract* c, uint8_t digest[32]);
/* Digest agreement between trainer and rollout engine: ISO_OK if equal, else
 * ISO_ERR_CONTRACT_MISMATCH (the caller must refuse to run).
 * [NovaSky IsoExec article, "The execution contract": runtimes exchange
 *  digests and refuse to run on disagreement] */
iso_status iso_contract_check_peer(const iso_contract* c, const uint8_t peer_digest[32]);
/* Topology claim: ISO_OK if num_ranks is a power of two dividing the leaf
 * count (the sizes for which the tree is proven invariant), else
 * ISO_ERR_UNPROVEN_TOPOLOGY.  [IsoExec blog, "Unified execution contract":
 *  the adapter rejects unproven parallel sizes] */
iso_status iso_contract_check_topology(const iso_contract* c, int num_ranks);
int iso_contract_leaf_count(const iso_contract* c);
/* FIPS 180-4 SHA-256 of n host bytes (the digest routine the contract uses). */
iso_status iso_sha256(const void* data, size_t n, uint8_t digest[32]);
const char* iso_status_string(iso_status s);
/* Synchronizes `stream`, then reads and clears the current device's status
 * word: ISO_OK, ISO_ERR_DEVICE_TIMEOUT, ISO_ERR_BAD_TOKEN_ID, ISO_ERR_SHAPE
 * (a device-side shape check failed, e.g. iso_attention's sequence table) or,
 * in the debug build (libiso_debug.so, compiled with -DISO_DEBUG: the same
 * entry points with a bounds check before every data-dependent global store
 * and gather, each of which records this status and skips the access instead
 * of trapping), ISO_ERR_DEVICE_CHECK. */
iso_status iso_last_device_status(iso_stream stream);

/* ---------------------------------------------------------------- iso_gemm
 * C[M x N] = bf16_rn( tree_{l=0..L-1} P_l ),  P_l = sum over leaf l of A*B.
 * [IsoExec blog, "Parallelism-invariant kernels": K divided into contiguous
 *  leaves, each a deterministic tensor-core MMA chain with FP32
 *  accumulation, combined by the contract's binary arithmetic schedule]
 * [RL-Kernel blog, §2 "Four Common Trigger Points" and §7 "GEMM": FP32
 *  accumulation, one conversion to BF16 at a fixed point]
 * A: [M x K] bf16 row-major, lda >= K.  B: [K x N] bf16 row-major, ldb >= N.
 * C: [M x N] bf16 row-major, ldc >= N.  L = contract leaf count; leaf l covers
 * k in [l K/L, (l+1) K/L).  Requires K % (16 L) == 0 (ISO_ERR_SHAPE),
 * N % 8 == 0 (ISO_ERR_SHAPE), lda/ldb/ldc % 8 == 0 and 16-byte aligned
 * pointers (ISO_ERR_ALIGNMENT).  M == 0 is a no-op. */
iso_status iso_gemm(const iso_contract* c, const iso_bf16* A, int64_t lda, const iso_bf16* B, int64_t ldb,
                    iso_bf16* C, int64_t ldc, int M, int N, int K, iso_stream stream);

/* iso_gemm with scratch: the same C, bit for bit, as iso_gemm.  For one row
 * block (M <= 128) with fewer 128-column tiles than SMs, the leaves are split
 * into R groups of L/R (R a power of two, R x tiles <= SMs, R as large as ws
 * allows): each group's fp32 subtree root for every tile goes to ws and the
 * tree combine applies the top log2 R levels of the contract's tree, so more
 * SMs stream B (decode-size problems are bound by reading B).  This is the
 * partial + combine schedule of simulated ranks [IsoExec blog,
 * "Parallelism-invariant kernels"] run inside one call.  ws: device scratch,
 * 16-byte aligned, owned by the caller, in use until the stream passes the
 * call; iso_gemm_workspace(c, M, N, K) bytes allow the largest split (0 when
 * the split does not apply); with less (or ws == NULL) the call is iso_gemm.
 * Errors as iso_gemm; iso_gemm_workspace returns 0 for invalid arguments. */
size_t iso_gemm_workspace(const iso_contract* c, int M, int N, int K);
iso_status iso_gemm_ws(const iso_contract* c, const iso_bf16* A, int64_t lda, const iso_bf16* B, int64_t ldb,
                       iso_bf16* C, int64_t ldc, int M, int N, int K, void* ws, size_t ws_bytes, iso_stream stream);

/* ------------------------------------------------- simulated tensor parallel
 * iso_gemm_leaf_partial: rank `rank` of `num_ranks` owns the contiguous leaves
 * [rank L/R, (rank+1) L/R) (rank-to-leaf map fixed by the contract) and
 * writes the fp32 root of its subtree: S_r[M x N] (lds >= N, lds % 4 == 0).
 * A_r: [M x K_local] (this rank's K slice), B_r: [K_local x N].  R must be a
 * power of two dividing L (ISO_ERR_UNPROVEN_TOPOLOGY); K_local % (16 L/R) == 0.
 * iso_tree_combine: applies the top log2(R) levels of the same tree to
 * S[r] = S + r * rank_stride (fp32 [M x lds] each) and writes C = bf16_rn(root).
 * The pair reproduces iso_gemm bit for bit for every R.
 * Sequence parallelism (the reduce-scatter form): a rank that keeps output rows
 * [r0, r1) passes S + r0 * lds and M = r1 - r0 (the rows of every rank's
 * partial, exchanged without arithmetic); its rows equal rows [r0, r1) of
 * iso_gemm bit for bit [IsoExec blog, "Parallelism-invariant kernels": SP
 * reuses the non-SP reduction tree, each rank keeping its output slice].
 * [IsoExec blog, "Parallelism-invariant kernels": NCCL only transports the
 *  partial results]; [RL-Kernel blog, §6 table row 06: the same fixed
 *  balanced tree for TP1/2/4/8] */
iso_status iso_gemm_leaf_partial(const iso_contract* c, int rank, int num_ranks, const iso_bf16* A_r, int64_t lda,
                                 const iso_bf16* B_r, int64_t ldb, float* S_r, int64_t lds, int M, int N,
                                 int K_local, iso_stream stream);
iso_status iso_tree_combine(const iso_contract* c, int num_ranks, const float* S, int64_t lds,
                            int64_t rank_stride, iso_bf16* C, int64_t ldc, int M, int N, iso_stream stream);

/* -------------------------------------------------------------- iso_rmsnorm
 * y[t, i] = bf16_rn( (x[t,i] * r_t) * gamma[i] ),  r_t = 1 / sqrt(mean_i x^2 + eps)
 * with the per-row reduction of fixed shape (contract: one warp per row, lane
 * l sums the 8-element vectors v = l mod 32 in ascending order, then an xor
 * shuffle tree 16,8,4,2,1).
 * [RL-Kernel blog, §4 table: RMSNorm reduces over the hidden dimension;
 *  §6 table row 02]; [VeXact paper, §3.1: batch-invariant RMSNorm]
 * x, y: [T x H] bf16 row-major (ld = H); gamma: [H] bf16.  H % 8 == 0. */
iso_status iso_rmsnorm(const iso_contract* c, const iso_bf16* x, const iso_bf16* gamma, float eps, iso_bf16* y,
                       int T, int H, iso_stream stream);

/* ---------------------------------------------------- iso_selected_logprob
 * out[t] = z[t, ids[t]] - LSE_v z[t, v],  z = h W as the fp32 tree root (never
 * rounded).  LSE: per 128-column vocab tile (m = max, s = sum expf(z - m) over
 * ascending columns), tiles folded left to right inside chunks of 19 tiles
 * with the two-block merge m = max(m1,m2), s = s1 e^(m1-m) + s2 e^(m2-m),
 * chunks combined by a balanced pairwise tree (odd node carried up),
 * lse = m + logf(s).  Logits are never written to memory.
 * [RL-Kernel blog, §4 "Focus: The Shared Dependency ... on LogSumExp",
 *  "Causal Chain: How Block Merge Order Alters LSE"; §6 table row 05; §7
 *  "LogP": local statistics merged in a fixed vocab-tile order]
 * [VeXact paper, §2 Eq. (1): delta_t compares exactly these values]
 * h: [T x H] bf16 row-major; W: [H x V] bf16 row-major (the LM head as K x N);
 * ids: [T] int32; out: [T] fp32.  H % (16 L) == 0; V % 8 == 0; V <= 622592.
 * ws: device workspace, 16-byte aligned, of at least
 * iso_selected_logprob_min_workspace(c, T, V) bytes (ISO_ERR_WORKSPACE
 * otherwise).  With iso_selected_logprob_workspace(c, T, V) bytes or more
 * the call also stores per-tile statistics and runs one 128-column tile per
 * work unit, which balances the GPU better; with less it runs one vocab
 * chunk per unit.  Both schedules fold the same statistics in the same order,
 * so the results are bit-identical.  A token id outside [0, V) yields
 * out[t] = NaN and sets ISO_ERR_BAD_TOKEN_ID in the device status word.
 * Both size queries return 0 for invalid arguments. */
size_t iso_selected_logprob_workspace(const iso_contract* c, int T, int V);
size_t iso_selected_logprob_min_workspace(const iso_contract* c, int T, int V);
iso_status iso_selected_logprob(const iso_contract* c, const iso_bf16* h, const iso_bf16* W, const int32_t* ids,
                                float* out, int T, int H, int V, void* ws, size_t ws_bytes, iso_stream stream);

/* ------------------------------------------------ vocab-parallel logprob
 * [RL-Kernel blog, §7 "LogP": each tensor-parallel shard computes its local
 *  statistics, then they are merged in a fixed vocab tile order; §4 "Causal
 *  Chain: How Block Merge Order Alters LSE": the two-block merge]
 * Shard r owns the vocabulary columns [v0, v0 + V_r) of V: v0 a multiple of
 * the 2432-column chunk, V_r a multiple of it unless the shard ends at V, and
 * the shards in rank order cover [0, V) contiguously.
 *
 * iso_selected_logprob_partial: W_r [H x V_r] bf16 (the shard's columns,
 * leading dimension ldw >= V_r, ldw % 8 == 0); h, ids as iso_selected_logprob
 * (ids are full-vocabulary ids).  Writes the shard's chunk statistics
 * stats_r [C_r x T] (m, s) fp32 pairs, chunk-major (C_r = chunks of the
 * shard), and z_sel_r[t] = the logit at ids[t] for the rows whose id falls in
 * the shard (other rows are left untouched).  ws (optional, 16-byte aligned,
 * iso_selected_logprob_partial_workspace bytes) enables one-tile work units.
 *
 * iso_selected_logprob_combine: stats [C x T] pairs = the shards' stats_r
 * concatenated in rank order (an all-gather of the chunk-major blocks);
 * zsel [num_shards x T] = the shards' z_sel_r; shard_v0: HOST array of the
 * num_shards first columns (increasing, shard_v0[0] = 0, <= 64 shards).
 * out[t] = z_sel(owner of ids[t])[t] - lse over the chunk tree: bit for bit
 * the output of iso_selected_logprob on the whole vocabulary.  Ids outside
 * [0, V) yield NaN and ISO_ERR_BAD_TOKEN_ID in the device status word. */
size_t iso_selected_logprob_partial_workspace(const iso_contract* c, int T, int V_r);
iso_status iso_selected_logprob_partial(const iso_contract* c, const iso_bf16* h, const iso_bf16* W_r, int64_t ldw,
                                        const int32_t* ids, int T, int H, int V, int v0, int V_r, float* stats_r,
                                        float* zsel_r, void* ws, size_t ws_bytes, iso_stream stream);
iso_status iso_selected_logprob_combine(const iso_contract* c, int num_shards, const int* shard_v0,
                                        const float* stats, const float* zsel, const int32_t* ids, float* out, int T,
                                        int V, iso_stream stream);

/* ------------------------------------------ logprob without allocation
 * No counterpart on the pages: this entry point exists for callers of this
 * library that cannot allocate device memory -- code behind a plugin or
 * callback interface that receives only input/output pointers (no allocator,
 * no workspace argument), or code inside a framework that owns all device
 * memory or must not call cudaMalloc (it synchronizes the device) in its hot
 * loop.  Same arguments and bit-identical results as iso_selected_logprob,
 * minus the workspace: the scratch is one fixed device array of
 * ISO_LOGPROB_STATIC_SCRATCH_BYTES compiled into the library, present on
 * every GPU that loads it until the process exits.  Nothing is allocated.
 * Limit: calls with iso_selected_logprob_min_workspace(c, T, V) larger than
 * ISO_LOGPROB_STATIC_SCRATCH_BYTES return ISO_ERR_WORKSPACE and launch
 * nothing (8 MiB: up to 16,512 tokens at V = 151936); up to 820 tokens the
 * array also holds the per-tile statistics of the faster schedule.
 * The first call on a device looks up the array's device address; make that
 * first call before any stream capture.  The address is kept for the life of
 * the process: do not call this entry point across a cudaDeviceReset (or any
 * other teardown and re-creation of the device's primary context).  All calls on a device share the one
 * array: calls whose kernels may overlap on the GPU (unordered streams) race
 * and must be serialized by the caller. */
#define ISO_LOGPROB_STATIC_SCRATCH_BYTES (8u << 20)
iso_status iso_selected_logprob_static_scratch(const iso_contract* c, const iso_bf16* h, const iso_bf16* W,
                                               const int32_t* ids, float* out, int T, int H, int V,
                                               iso_stream stream);

/* --------------------------------------------------------------------- MoE
 * [IsoExec blog, "Unified model": deterministic MoE routing and combination;
 *  "Parallelism-invariant kernels": expert outputs combined in a fixed
 *  routing order rather than rank order; "Unified execution contract":
 *  moe.combine = leaf tree, 8 leaves, fp32 leaves]
 * [RL-Kernel blog, §6 table row 04 and §7 "FFN": packed gate/up, SwiGLU and
 *  down projection as separate fixed stages]
 *
 * iso_moe_route: logits [T x E] fp32 -> topk_ids [T x k] int32 (logit
 * descending, ties to the lower expert id) and topk_w [T x k] fp32 =
 * softmax over the k selected logits (denominator summed in slot order).
 * E <= 256, 1 <= k <= min(E, 32). */
iso_status iso_moe_route(const iso_contract* c, const float* logits, int T, int E, int k, int32_t* topk_ids,
                         float* topk_w, iso_stream stream);
/* Stable counting sort of the (token, slot) pairs p = t k + j by expert, over
 * the experts e with expert_partition[e] == partition (expert_partition is a
 * DEVICE array [E] int32; NULL selects every expert): perm lists pair indices
 * grouped by expert, ascending p inside an expert; offsets[E+1] are the group
 * boundaries (offsets[E] = number of listed pairs).  perm must hold T k
 * entries; counts_ws is device scratch of iso_moe_permute_workspace(T, E, k)
 * bytes (3 E + 2 int32 plus a histogram of E int32 per 1024 pairs), owned by
 * the caller and free again when the stream passes this call.  Ids outside
 * [0, E) set ISO_ERR_BAD_TOKEN_ID on the device and are left out.  E <= 256.
 * iso_moe_permute_workspace returns 0 for invalid sizes. */
size_t iso_moe_permute_workspace(int T, int E, int k);
iso_status iso_moe_permute(const iso_contract* c, const int32_t* topk_ids, int T, int E, int k,
                           const int32_t* expert_partition, int partition, int32_t* perm, int32_t* offsets,
                           int32_t* counts_ws, iso_stream stream);
/* out[t] = bf16_rn( tree_{j=0..k-1} (w[t,j] * y[t,j]) ): products fp32 rn, the
 * balanced binary tree over routing slots in slot order.  y_slots [T x k x H]
 * bf16, topk_w [T x k] fp32, out [T x H] bf16.  k a power of two <= 8,
 * H % 8 == 0. */
iso_status iso_moe_combine(const iso_contract* c, const iso_bf16* y_slots, const float* topk_w, iso_bf16* out,
                           int T, int k, int H, iso_stream stream);
/* The expert layer: for each partition p (experts with expert_partition[e] ==
 * p; NULL = one partition): permute, gather, grouped gate/up leaf-tree GEMM
 * (K = H) with G rounded to bf16, h = bf16_rn(silu(g) u) (silu(g) = g / (1 + e^-g)
 * in fp32 from the fast exp and divide intrinsics: a few fp32 ulps), grouped down
 * leaf-tree GEMM (K = F) rounded to bf16 into y_slots; then iso_moe_combine.
 * The result does not depend on the partition map.
 * x [T x H] bf16; topk_ids / topk_w as produced by iso_moe_route;
 * W1 [E x H x 2F] bf16 (gate columns [0,F), up columns [F,2F));
 * W2 [E x F x H] bf16; expert_partition: HOST array [E] int32 with values in
 * [0, num_partitions) (NULL = a single partition); out [T x H] bf16.
 * H % (16 L) == 0, F % (16 L) == 0, H % 128 == 0, F % 64 == 0, k a power of
 * two <= 8, E <= 256.  ws: iso_grouped_gemm_moe_workspace(c, T, E, k, H, F)
 * bytes. */
size_t iso_grouped_gemm_moe_workspace(const iso_contract* c, int T, int E, int k, int H, int F);
iso_status iso_grouped_gemm_moe(const iso_contract* c, const iso_bf16* x, const int32_t* topk_ids,
                                const float* topk_w, const iso_bf16* W1, const iso_bf16* W2,
                                const int32_t* expert_partition, int num_partitions, iso_bf16* out, int T, int E,
                                int k, int H, int F, void* ws, size_t ws_bytes, iso_stream stream);
/* The expert GEMMs of one expert-parallel rank, without the combine [IsoExec blog,
 * "Parallelism-invariant kernels": expert outputs are combined in a fixed routing order, not
 * in rank order].  For every routing slot (t, j) whose expert topk_ids[t, j] has
 * expert_mask[e] != 0: y_slots[t * k + j] = bf16 of the down projection of
 * h = bf16_rn(silu(g) u), exactly the slot rows iso_grouped_gemm_moe computes.  Rows of other
 * slots are not written.  So ranks that own disjoint expert sets fill disjoint slot rows, and
 * after the rows are exchanged, iso_moe_combine gives iso_grouped_gemm_moe's output bit for bit.
 * expert_mask: HOST array [E] uint8.  y_slots [T x k x H] bf16.  Other arguments, shape rules
 * and errors as iso_grouped_gemm_moe.  ws: iso_moe_experts_partial_workspace(c, T, E, k, H, F)
 * bytes. */
size_t iso_moe_experts_partial_workspace(const iso_contract* c, int T, int E, int k, int H, int F);
iso_status iso_moe_experts_partial(const iso_contract* c, const iso_bf16* x, const int32_t* topk_ids,
                                   const iso_bf16* W1, const iso_bf16* W2, const uint8_t* expert_mask,
                                   iso_bf16* y_slots, int T, int E, int k, int H, int F, void* ws, size_t ws_bytes,
                                   iso_stream stream);

/* ------------------------------------------------- mismatch diagnostics
 * [VeXact paper, §2 Eq. (1): delta_t = log pi_train - log pi_rollout; §4.1:
 *  the K1(r) = -log r and K3(r) = (r - 1) - log r estimators; §4.2 Eq. (6):
 *  truncated importance weight min(r_corr, tau_tok); Eq. (7)-(11): sequence
 *  rejection 1[sum_t K(r_corr,t) <= tau_seq], r_corr = pi_train / pi_rollout;
 *  Appendix A.4 uses tau_tok = 2, tau_seq = 0.001]
 * logp_train, logp_rollout: [N] fp32, the selected-token logprobs of B packed
 * sequences; seq_offsets: DEVICE [B+1] int32, sequence b = tokens
 * [offsets[b], offsets[b+1]), nondecreasing, offsets[B] <= N.
 * Per token (either may be NULL to skip): delta [N] fp32, tis_weight [N] fp32.
 * Per sequence: seq_k1, seq_k3 [B] fp64 (sums of K1, K3 of r_corr),
 * accept_k1, accept_k3 [B] uint8 (1 when the sum <= tau_seq), max |delta|
 * [B] fp32, sum |delta| [B] fp64, count of tokens whose two logprobs differ
 * [B] int32.  delta and r are evaluated in double (log r_corr = delta_t, so
 * K1 = -delta_t, K3 = (r_corr - 1) - delta_t); each sequence is summed in a
 * fixed order (thread-strided ascending sums, a shuffle tree per warp, warps
 * in order), so results depend only on the sequence.  tau_tok > 0, tau_seq >= 0, else
 * ISO_ERR_INVALID_ARG. */
iso_status iso_mismatch_diagnostics(const iso_contract* c, const float* logp_train, const float* logp_rollout,
                                    const int32_t* seq_offsets, int B, int N, double tau_tok, double tau_seq,
                                    float* delta, float* tis_weight, double* seq_k1, double* seq_k3,
                                    uint8_t* accept_k1, uint8_t* accept_k3, float* seq_max_abs_delta,
                                    double* seq_sum_abs_delta, int32_t* seq_mismatches, iso_stream stream);

/* ------------------------------------------- RMSNorm fused into the A prologue
 * [IsoExec blog, "Parallelism-invariant kernels"; RL-Kernel blog, §6 table row
 *  02 (RMSNorm) and §7: fusions must keep the separate stages' numerics]
 * iso_rmsnorm_gemm: C = iso_gemm(iso_rmsnorm(x, gamma, eps), B) bit for bit,
 * without writing the normalised activations: a row pass computes
 * r_t = 1 / sqrt(mean x^2 + eps) with iso_rmsnorm's reduction into ws, then the
 * GEMM's producer warps build each A tile in shared memory as
 * bf16_rn((x * r_t) * gamma_i), iso_rmsnorm's per-element arithmetic.  x: [M x K]
 * bf16 (ld = K), gamma: [K] bf16, B / C as for iso_gemm; ws (DEVICE, 16-byte
 * aligned): iso_rmsnorm_gemm_workspace(c, M) bytes (ISO_ERR_WORKSPACE).
 * iso_rmsnorm_selected_logprob: iso_selected_logprob(iso_rmsnorm(x, gamma, eps),
 * W, ids) bit for bit; ws: iso_rmsnorm_selected_logprob_workspace(c, T, V) bytes
 * (the per-row factors first, then the logprob workspace; with less room than
 * that but at least the factors plus iso_selected_logprob_min_workspace the
 * chunk-unit schedule runs, same bits).  Other errors as the unfused calls.
 * Speed: the fused form never writes or re-reads the normalised activations,
 * but it normalises each A tile again for every 128-column output tile, so
 * its extra work grows with N / 128: it pays only for narrow outputs (a few
 * column tiles).  For the wide shapes of an LM (measured on GB300: M = 4096,
 * K = N = 4096: 0.975 ms fused against 0.325 ms for iso_rmsnorm + iso_gemm;
 * the T = 4096, V = 151936 logprob: 10.5 ms against 3.06 ms) the separate
 * stages are the fast path, with the same bits. */
size_t iso_rmsnorm_gemm_workspace(const iso_contract* c, int M);
iso_status iso_rmsnorm_gemm(const iso_contract* c, const iso_bf16* x, const iso_bf16* gamma, float eps,
                            const iso_bf16* B, int64_t ldb, iso_bf16* C, int64_t ldc, int M, int N, int K, void* ws,
                            size_t ws_bytes, iso_stream stream);
size_t iso_rmsnorm_selected_logprob_workspace(const iso_contract* c, int T, int V);
iso_status iso_rmsnorm_selected_logprob(const iso_contract* c, const iso_bf16* x, const iso_bf16* gamma, float eps,
                                        const iso_bf16* W, const int32_t* ids, float* out, int T, int H, int V,
                                        void* ws, size_t ws_bytes, iso_stream stream);

/* ------------------------------------------------------------ attention
 * [RL-Kernel blog, §4 "Focus: The Shared Dependency of Attention and Linear
 *  LogP on LogSumExp": softmax over the visible keys and its LSE statistic;
 *  §6 table row 03 and §7 "Attention": no KV split, fixed block partitioning
 *  and a fixed rescale-merge order; VeXact paper, §3.1: KV splitting
 *  disabled so prefill and decode reduce alike]
 * Causal attention over B packed variable-length sequences with grouped KV
 * heads.  Q [Tq x Hq x d], K and V [Tk x Hkv x d]: bf16, row-major, DEVICE,
 * 16-byte aligned (ISO_ERR_ALIGNMENT).  q_start, k_start: DEVICE [B+1] int32;
 * pos0: DEVICE [B] int32.  Sequence b owns query rows [q_start[b],
 * q_start[b+1]) and keys [k_start[b], k_start[b+1]); its query row r sits at
 * position p = pos0[b] + (r - q_start[b]) and attends to keys k_start[b] ..
 * k_start[b] + p, so k_start[b] + pos0[b] + (rows of b) <= k_start[b+1].
 * Query head h reads KV head h / (Hq / Hkv) (Hq % Hkv != 0: ISO_ERR_SHAPE).
 * d == 128 (else ISO_ERR_UNSUPPORTED).  max_q_rows >= the largest query row
 * count of a sequence (it sizes the grid).  out [Tq x Hq x d] bf16 =
 * softmax(scale q.k) V; lse [Tq x Hq] fp32 = m + log l (NULL to skip).
 * The merge runs over fixed 80-key chunks of each sequence, in ascending
 * order, one online-softmax step per chunk; nothing depends on the other
 * rows of the call, so a row's bits are the same in a prefill (many rows) and
 * a decode call (one row at the same position), whatever the batch.  Keys
 * past a row's position inside its last chunk are masked but still read: K
 * and V must hold finite values in every row [0, Tk).  A sequence table that
 * breaks the rules above sets ISO_ERR_SHAPE in the device status word and its
 * rows are left unwritten.  Empty calls (B, Tq or max_q_rows 0) are no-ops. */
iso_status iso_attention(const iso_contract* c, const iso_bf16* Q, const iso_bf16* K, const iso_bf16* V,
                         const int32_t* q_start, const int32_t* k_start, const int32_t* pos0, int B, int Tq,
                         int Tk, int Hq, int Hkv, int d, int max_q_rows, float scale, iso_bf16* out, float* lse,
                         iso_stream stream);

/* --------------------------------------------------------- failure checks
 * Launches one kernel whose only job is a bounded wait on an mbarrier that
 * nothing ever completes; after timeout_ns it gives up, sets
 * ISO_ERR_DEVICE_TIMEOUT in the status word and returns, leaving the context
 * usable.  Exercises the same bounded-wait path every kernel uses.  No
 * counterpart on the pages: the pages' runtimes refuse to run on a contract
 * violation; this is the device-side half of that behaviour. */
iso_status iso_selftest_bounded_wait(uint64_t timeout_ns, iso_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* ISO_H_ */
