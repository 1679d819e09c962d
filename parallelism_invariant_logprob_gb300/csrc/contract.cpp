// contract.cpp -- the numerical contract: validation, canonical serialization
// and its SHA-256 identity digest.
//
// [IsoExec blog, "Unified execution contract"]: the contract pins every
// execution choice that can move the bits (implementation id and version,
// accumulation and boundary dtypes, reduction decomposition); its
// numerical_policy identity is a SHA-256 digest of the serialized contract,
// exchanged between trainer and rollout engine, which refuse to run when the
// digests differ [NovaSky IsoExec article, "The execution contract"].  A
// topology claim lists the parallel sizes for which the reduction tree is
// proven invariant; unproven sizes are rejected.
//
// SHA-256 follows FIPS 180-4 (section 6.2), written from the standard.
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <string>

#include "iso_internal.h"

struct iso_contract {
  int leaf_count;
  iso_tree_schedule schedule;
  iso_dtype acc_dtype;
  iso_dtype out_dtype;
  std::string serialized;
  uint8_t digest[32];
};

namespace {

// ------------------------------------------------------------ SHA-256 (FIPS 180-4)
struct Sha256 {
  uint32_t h[8];
  uint8_t buf[64];
  uint64_t bits;
  size_t fill;
};

inline uint32_t rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }

const uint32_t kK[64] = {
    0x428a2f98, 0x71374491, 0xb5c0fbcf, 0xe9b5dba5, 0x3956c25b, 0x59f111f1, 0x923f82a4, 0xab1c5ed5,
    0xd807aa98, 0x12835b01, 0x243185be, 0x550c7dc3, 0x72be5d74, 0x80deb1fe, 0x9bdc06a7, 0xc19bf174,
    0xe49b69c1, 0xefbe4786, 0x0fc19dc6, 0x240ca1cc, 0x2de92c6f, 0x4a7484aa, 0x5cb0a9dc, 0x76f988da,
    0x983e5152, 0xa831c66d, 0xb00327c8, 0xbf597fc7, 0xc6e00bf3, 0xd5a79147, 0x06ca6351, 0x14292967,
    0x27b70a85, 0x2e1b2138, 0x4d2c6dfc, 0x53380d13, 0x650a7354, 0x766a0abb, 0x81c2c92e, 0x92722c85,
    0xa2bfe8a1, 0xa81a664b, 0xc24b8b70, 0xc76c51a3, 0xd192e819, 0xd6990624, 0xf40e3585, 0x106aa070,
    0x19a4c116, 0x1e376c08, 0x2748774c, 0x34b0bcb5, 0x391c0cb3, 0x4ed8aa4a, 0x5b9cca4f, 0x682e6ff3,
    0x748f82ee, 0x78a5636f, 0x84c87814, 0x8cc70208, 0x90befffa, 0xa4506ceb, 0xbef9a3f7, 0xc67178f2};

void sha_block(Sha256& s, const uint8_t* p) {
  uint32_t w[64];
  for (int t = 0; t < 16; ++t)
    w[t] = (uint32_t)p[4 * t] << 24 | (uint32_t)p[4 * t + 1] << 16 | (uint32_t)p[4 * t + 2] << 8 | p[4 * t + 3];
  for (int t = 16; t < 64; ++t) {
    uint32_t s0 = rotr(w[t - 15], 7) ^ rotr(w[t - 15], 18) ^ (w[t - 15] >> 3);
    uint32_t s1 = rotr(w[t - 2], 17) ^ rotr(w[t - 2], 19) ^ (w[t - 2] >> 10);
    w[t] = w[t - 16] + s0 + w[t - 7] + s1;
  }
  uint32_t a = s.h[0], b = s.h[1], c = s.h[2], d = s.h[3], e = s.h[4], f = s.h[5], g = s.h[6], hh = s.h[7];
  for (int t = 0; t < 64; ++t) {
    uint32_t S1 = rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25);
    uint32_t ch = (e & f) ^ (~e & g);
    uint32_t t1 = hh + S1 + ch + kK[t] + w[t];
    uint32_t S0 = rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22);
    uint32_t maj = (a & b) ^ (a & c) ^ (b & c);
    uint32_t t2 = S0 + maj;
    hh = g;
    g = f;
    f = e;
    e = d + t1;
    d = c;
    c = b;
    b = a;
    a = t1 + t2;
  }
  s.h[0] += a;
  s.h[1] += b;
  s.h[2] += c;
  s.h[3] += d;
  s.h[4] += e;
  s.h[5] += f;
  s.h[6] += g;
  s.h[7] += hh;
}

void sha256(const uint8_t* data, size_t n, uint8_t out[32]) {
  Sha256 s;
  const uint32_t init[8] = {0x6a09e667, 0xbb67ae85, 0x3c6ef372, 0xa54ff53a,
                            0x510e527f, 0x9b05688c, 0x1f83d9ab, 0x5be0cd19};
  memcpy(s.h, init, sizeof init);
  s.bits = (uint64_t)n * 8;
  size_t i = 0;
  for (; i + 64 <= n; i += 64) sha_block(s, data + i);
  uint8_t tail[128];
  size_t r = n - i;
  memcpy(tail, data + i, r);
  tail[r] = 0x80;
  size_t total = (r + 1 + 8 <= 64) ? 64 : 128;
  memset(tail + r + 1, 0, total - r - 1);
  for (int b = 0; b < 8; ++b) tail[total - 1 - b] = (uint8_t)(s.bits >> (8 * b));
  sha_block(s, tail);
  if (total == 128) sha_block(s, tail + 64);
  for (int k = 0; k < 8; ++k) {
    out[4 * k] = (uint8_t)(s.h[k] >> 24);
    out[4 * k + 1] = (uint8_t)(s.h[k] >> 16);
    out[4 * k + 2] = (uint8_t)(s.h[k] >> 8);
    out[4 * k + 3] = (uint8_t)s.h[k];
  }
}

const char* dtype_name(iso_dtype d) { return d == ISO_F32 ? "fp32" : "bf16"; }

// Canonical serialization: fixed field order, no whitespace.  Every constant and every
// rounding step that can change an output bit appears here, written as the kernels execute
// it: `__fadd_rn` etc. are the IEEE round-to-nearest-even fp32 operations (never contracted),
// `expf` / `logf` are CUDA's math library functions of the toolkit named under "impl",
// `__expf` / `__fdividef` / `ex2.approx.ftz` are the hardware approximations.  The numbers come
// from the same constants the kernels are compiled with (iso_internal.h), so a kernel change
// of a tile width, chunk size or merge threshold changes the digest.
std::string serialize(const iso_contract& c) {
  char claim[64];
  int n = 0;
  claim[n++] = '[';
  for (int r = 1; r <= c.leaf_count; r *= 2) n += snprintf(claim + n, sizeof claim - n, r == 1 ? "%d" : ",%d", r);
  claim[n++] = ']';
  claim[n] = 0;
  char buf[4096];
  snprintf(buf, sizeof buf,
           "{\"identity\":\"numerical_policy\",\"contract_version\":2,"
           "\"impl\":{\"id\":\"iso_leaf_tree_tcgen05\",\"version\":3,\"arch\":\"sm_103a\",\"cuda\":\"%d.%d\"},"
           "\"gemm\":{\"leaves\":%d,\"rank_to_leaf\":\"contiguous\","
           "\"leaf_chain\":{\"instr\":\"tcgen05.mma.kind::f16\",\"rows_per_cta\":%d,"
           "\"cta_group\":\"1(m=128)|2(m=256)\",\"n\":%d,\"k\":%d,"
           "\"order\":\"ascending_k\",\"first\":\"overwrite\"},"
           "\"tree\":\"%s\",\"tree_add\":\"__fadd_rn\",\"acc_dtype\":\"%s\",\"out_dtype\":\"%s\","
           "\"convert\":\"once_at_root_bf16_rn\"},"
           "\"claims\":{\"topology\":{\"simulated_ranks\":%s}},"
           "\"logprob\":{\"logit\":\"tree_root_fp32_unrounded\",\"tile_cols\":%d,\"chunk_tiles\":%d,"
           "\"tile_stat\":\"m=max;s=ascending_columns(__fadd_rn(s,expf(__fsub_rn(z,m))))\","
           "\"chunk_fold\":\"left_to_right_two_block_merge\",\"chunk_tree\":\"pairwise_odd_carried\","
           "\"merge\":\"m=fmaxf(m1,m2);s=__fadd_rn(__fmul_rn(s1,expf(__fsub_rn(m1,m))),"
           "__fmul_rn(s2,expf(__fsub_rn(m2,m))))\",\"lse\":\"__fadd_rn(m,logf(s))\","
           "\"out\":\"__fsub_rn(z_sel,lse)\",\"vocab_parallel\":\"contiguous_chunk_aligned_shards_in_rank_order\"},"
           "\"rmsnorm\":{\"map\":\"warp_per_row;lane_owns_8_element_vectors_v_mod_32\","
           "\"lane_sum\":\"ascending(__fadd_rn(acc,__fmul_rn(x,x)))\",\"tree\":\"shfl_xor_16_8_4_2_1\","
           "\"scale\":\"__fdiv_rn(1,__fsqrt_rn(__fadd_rn(__fdiv_rn(ss,H),eps)))\","
           "\"out\":\"bf16_rn(__fmul_rn(__fmul_rn(x,r),gamma))\"},"
           "\"moe\":{\"route\":\"topk_logit_desc_id_asc\","
           "\"gates\":\"__fdiv_rn(expf(__fsub_rn(l,l0)),slot_order(__fadd_rn))\","
           "\"stages\":[\"gate_up_root_bf16_rn\","
           "\"h=bf16_rn(__fmul_rn(__fdividef(g,__fadd_rn(1,__expf(-g))),u))\",\"down_root_bf16_rn\"],"
           "\"combine\":{\"order\":\"routing_slot\",\"leaf\":\"__fmul_rn(w,y)\",\"tree\":\"balanced_binary\","
           "\"out\":\"bf16_rn\"}},"
           "\"attention\":{\"kv_split\":\"none\",\"chunk_keys\":%d,\"chunk_order\":\"ascending\","
           "\"qk\":\"tcgen05.mma.kind::f16,m=128,n=%d,k=16,ascending_dims\",\"c2\":\"fp32_rn(scale*log2(e))\","
           "\"t\":\"__fmul_rn(chunk_max(S),c2)\",\"lazy_log2\":%g,"
           "\"m\":\"t_if_first_chunk_or_t>m+lazy_else_m\",\"p\":\"ex2.approx.ftz(__fmaf_rn(S,c2,-m))\","
           "\"p_operand\":\"bf16_rn\",\"l_chunk\":\"4_partials_key_mod_4(__fadd_rn);(p0+p1)+(p2+p3)\","
           "\"a\":\"ex2.approx.ftz(__fsub_rn(m_old,m))\",\"l\":\"__fadd_rn(__fmul_rn(l,a),l_chunk)\","
           "\"o_rescale\":\"__fmul_rn(O,a)\",\"pv\":\"tcgen05.mma.kind::f16,m=128,n=128,k=16,ascending_keys\","
           "\"out\":\"bf16_rn(__fmul_rn(O,__frcp_rn(l)))\",\"lse\":\"__fadd_rn(__fmul_rn(m,fp32(ln2)),logf(l))\"},"
           "\"math\":{\"fp32_add_mul\":\"rn_intrinsics_never_contracted\",\"libm\":\"cuda_toolkit_expf_logf\"}}",
           CUDART_VERSION / 1000, (CUDART_VERSION % 1000) / 10, c.leaf_count, iso::BM, iso::BN, iso::UMMA_K,
           c.schedule == ISO_TREE_BALANCED_BINARY ? "balanced_binary_left_lower_index" : "?",
           dtype_name(c.acc_dtype), dtype_name(c.out_dtype), claim, iso::LP_TILE_COLS, iso::LP_CHUNK_TILES,
           iso::ATT_CHUNK_KEYS, iso::ATT_CHUNK_KEYS, static_cast<double>(iso::ATT_LAZY_LOG2));
  return std::string(buf);
}

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

}  // namespace

extern "C" {

iso_status iso_contract_init(int leaf_count, iso_tree_schedule schedule, iso_dtype acc_dtype, iso_dtype out_dtype,
                             iso_contract** out, uint8_t digest[32]) {
  if (!out) return ISO_ERR_INVALID_ARG;
  *out = nullptr;
  if (!is_pow2(leaf_count)) return ISO_ERR_INVALID_ARG;
  if (leaf_count > iso::MAX_LEAVES) return ISO_ERR_UNSUPPORTED;
  if (schedule != ISO_TREE_BALANCED_BINARY) return ISO_ERR_UNSUPPORTED;
  if (acc_dtype != ISO_F32) return ISO_ERR_UNSUPPORTED;
  if (out_dtype != ISO_BF16) return ISO_ERR_UNSUPPORTED;
  iso_contract* c = new (std::nothrow) iso_contract;
  if (!c) return ISO_ERR_INVALID_ARG;
  c->leaf_count = leaf_count;
  c->schedule = schedule;
  c->acc_dtype = acc_dtype;
  c->out_dtype = out_dtype;
  c->serialized = serialize(*c);
  sha256(reinterpret_cast<const uint8_t*>(c->serialized.data()), c->serialized.size(), c->digest);
  if (digest) memcpy(digest, c->digest, 32);
  *out = c;
  return ISO_OK;
}

void iso_contract_destroy(iso_contract* c) { delete c; }

iso_status iso_contract_serialize(const iso_contract* c, char* buf, size_t cap, size_t* len) {
  if (!c) return ISO_ERR_INVALID_ARG;
  if (len) *len = c->serialized.size();
  if (buf) {
    if (cap < c->serialized.size() + 1) return ISO_ERR_WORKSPACE;
    memcpy(buf, c->serialized.c_str(), c->serialized.size() + 1);
  }
  return ISO_OK;
}

iso_status iso_contract_digest(const iso_contract* c, uint8_t digest[32]) {
  if (!c || !digest) return ISO_ERR_INVALID_ARG;
  memcpy(digest, c->digest, 32);
  return ISO_OK;
}

iso_status iso_contract_check_peer(const iso_contract* c, const uint8_t peer_digest[32]) {
  if (!c || !peer_digest) return ISO_ERR_INVALID_ARG;
  return memcmp(c->digest, peer_digest, 32) == 0 ? ISO_OK : ISO_ERR_CONTRACT_MISMATCH;
}

iso_status iso_contract_check_topology(const iso_contract* c, int num_ranks) {
  if (!c) return ISO_ERR_INVALID_ARG;
  if (!is_pow2(num_ranks) || c->leaf_count % num_ranks != 0) return ISO_ERR_UNPROVEN_TOPOLOGY;
  return ISO_OK;
}

int iso_contract_leaf_count(const iso_contract* c) { return c ? c->leaf_count : 0; }

iso_status iso_sha256(const void* data, size_t n, uint8_t digest[32]) {
  if ((!data && n) || !digest) return ISO_ERR_INVALID_ARG;
  sha256(static_cast<const uint8_t*>(data), n, digest);
  return ISO_OK;
}

const char* iso_status_string(iso_status s) {
  switch (s) {
    case ISO_OK: return "ok";
    case ISO_ERR_INVALID_ARG: return "invalid argument";
    case ISO_ERR_SHAPE: return "unsupported shape (K must be a multiple of 16 x leaf count; see header)";
    case ISO_ERR_ALIGNMENT: return "pointer or leading dimension not 16-byte aligned";
    case ISO_ERR_UNPROVEN_TOPOLOGY: return "rank count is not a power of two dividing the leaf count";
    case ISO_ERR_UNSUPPORTED: return "configuration not supported by this library";
    case ISO_ERR_CONTRACT_MISMATCH: return "peer contract digest differs";
    case ISO_ERR_WORKSPACE: return "workspace or buffer too small";
    case ISO_ERR_CUDA: return "CUDA runtime error";
    case ISO_ERR_DEVICE_TIMEOUT: return "a device-side wait ran out of time";
    case ISO_ERR_NOT_IMPLEMENTED: return "not implemented";
    case ISO_ERR_BAD_TOKEN_ID: return "a token id was outside [0, V)";
  }
  return "unknown status";
}

}  // extern "C"
