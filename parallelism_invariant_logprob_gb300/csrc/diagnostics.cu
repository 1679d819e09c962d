// diagnostics.cu -- training/rollout mismatch diagnostics over packed sequences of
// selected-token logprobs (one 1024-thread block per sequence).
//
// What it computes [VeXact paper, "Diagnosing Training Inference Mismatch in LLM
// Reinforcement Learning"]: per token the mismatch delta_t = log pi_train - log pi_rollout
// (§2 Eq. 1), the correction ratio r_corr = exp(delta_t), the truncated importance weight
// min(r_corr, tau_tok) (§4.2 Eq. 6); per sequence the K1 and K3 estimators of §4.1 summed
// over the sequence, S = sum_t K(r_corr,t), and the rejection decision S <= tau_seq
// (Eq. 7-11; the paper sets tau_tok = 2 and tau_seq = 0.001 in Appendix A.4), plus the largest
// |delta_t|, sum |delta_t| and the number of tokens whose two logprobs differ (the pages'
// "mismatch count" and max / mean |delta| probes).
//
// Precision and order: delta and r are evaluated in double from the fp32 inputs (delta
// exactly); log r_corr is delta_t itself (r_corr = pi_train / pi_rollout), so K1 = -delta and
// K3 = (r - 1) - delta = expm1(delta) - delta, and the rejection decision is taken in double.
// Identical logprobs give delta = 0, r = 1, K = 0 exactly; for |delta| < 2^-6 the K3 term comes
// from its Taylor series in double (cheaper than exp on this part's few FP64 units), otherwise
// from exp; identical logprobs skip the FP64 arithmetic altogether (their terms are exact zeros).  One 1024-thread block
// per sequence: thread i adds its tokens t = start + i + 1024 j in ascending j, an xor-shuffle
// tree (16, 8, 4, 2, 1) combines each warp, and thread 0 adds the 32 warp sums in warp order --
// a fixed order that depends only on the sequence, never on the launch.
#include "iso_internal.h"

namespace iso {
namespace {

constexpr int kDiagThreads = 1024;
constexpr int kDiagWarps = kDiagThreads / 32;

__global__ void __launch_bounds__(kDiagThreads)
    mismatch_kernel(const float* __restrict__ lp_train, const float* __restrict__ lp_rollout,
                    const int32_t* __restrict__ offsets, int B, double tau_tok, double tau_seq,
                    float* __restrict__ delta, float* __restrict__ tis_weight, double* __restrict__ seq_k1,
                    double* __restrict__ seq_k3, uint8_t* __restrict__ accept_k1, uint8_t* __restrict__ accept_k3,
                    float* __restrict__ seq_max_abs_delta, double* __restrict__ seq_sum_abs_delta,
                    int32_t* __restrict__ seq_mismatches) {
  __shared__ double w_s1[kDiagWarps], w_s3[kDiagWarps], w_sa[kDiagWarps], w_mx[kDiagWarps];
  __shared__ int w_nm[kDiagWarps];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  for (int b = blockIdx.x; b < B; b += gridDim.x) {
    const int32_t t0 = offsets[b], t1 = offsets[b + 1];
    double s1 = 0.0, s3 = 0.0, sa = 0.0, mx = 0.0;
    int nm = 0;
    for (int32_t t = t0 + static_cast<int32_t>(threadIdx.x); t < t1; t += kDiagThreads) {
      const float a = lp_train[t], r0 = lp_rollout[t];
      if (a == r0) {
        // identical logprobs: delta = 0, r_corr = 1, K1 = K3 = 0 exactly; adding those zeros
        // leaves every sum's bits unchanged and max(mx, 0) = mx, so no FP64 work is needed
        if (delta) delta[t] = 0.f;
        if (tis_weight) tis_weight[t] = 1.0 < tau_tok ? 1.f : static_cast<float>(tau_tok);
        continue;
      }
      const double d = static_cast<double>(a) - static_cast<double>(r0);
      double r, k3;  // r_corr = exp(d) and K3 = (r_corr - 1) - d = expm1(d) - d
      if (fabs(d) < 0.015625) {
        // expm1(d) - d by its Taylor series (terms through d^9: truncation below 1e-21 relative)
        k3 = d * d *
             (1.0 / 2 + d * (1.0 / 6 + d * (1.0 / 24 + d * (1.0 / 120 + d * (1.0 / 720 + d * (1.0 / 5040 +
                                                                                                d * (1.0 / 40320 + d * (1.0 / 362880))))))));
        r = (1.0 + d) + k3;
      } else {
        r = exp(d);
        k3 = (r - 1.0) - d;
      }
      s1 += -d;
      s3 += k3;
      sa += fabs(d);
      mx = fmax(mx, fabs(d));
      nm += (a != r0) ? 1 : 0;
      if (delta) delta[t] = static_cast<float>(d);
      if (tis_weight) tis_weight[t] = static_cast<float>(r < tau_tok ? r : tau_tok);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      s1 += __shfl_xor_sync(0xffffffffu, s1, off);
      s3 += __shfl_xor_sync(0xffffffffu, s3, off);
      sa += __shfl_xor_sync(0xffffffffu, sa, off);
      mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      nm += __shfl_xor_sync(0xffffffffu, nm, off);
    }
    if (lane == 0) {
      w_s1[warp] = s1;
      w_s3[warp] = s3;
      w_sa[warp] = sa;
      w_mx[warp] = mx;
      w_nm[warp] = nm;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      double S1 = 0.0, S3 = 0.0, SA = 0.0, MX = 0.0;
      int NM = 0;
      for (int w = 0; w < kDiagWarps; ++w) {
        S1 += w_s1[w];
        S3 += w_s3[w];
        SA += w_sa[w];
        MX = fmax(MX, w_mx[w]);
        NM += w_nm[w];
      }
      seq_k1[b] = S1;
      seq_k3[b] = S3;
      accept_k1[b] = S1 <= tau_seq ? 1 : 0;
      accept_k3[b] = S3 <= tau_seq ? 1 : 0;
      seq_max_abs_delta[b] = static_cast<float>(MX);
      seq_sum_abs_delta[b] = SA;
      seq_mismatches[b] = NM;
    }
    __syncthreads();
  }
}

}  // namespace
}  // namespace iso

using namespace iso;

extern "C" iso_status iso_mismatch_diagnostics(const iso_contract* c, const float* logp_train,
                                               const float* logp_rollout, const int32_t* seq_offsets, int B, int N,
                                               double tau_tok, double tau_seq, float* delta, float* tis_weight,
                                               double* seq_k1, double* seq_k3, uint8_t* accept_k1,
                                               uint8_t* accept_k3, float* seq_max_abs_delta,
                                               double* seq_sum_abs_delta, int32_t* seq_mismatches,
                                               iso_stream stream) {
  if (!c || B < 0 || N < 0) return ISO_ERR_INVALID_ARG;
  if (!(tau_tok > 0.0) || !(tau_seq >= 0.0)) return ISO_ERR_INVALID_ARG;
  if (B == 0) return ISO_OK;
  if (!seq_offsets || (N > 0 && (!logp_train || !logp_rollout))) return ISO_ERR_INVALID_ARG;
  if (!seq_k1 || !seq_k3 || !accept_k1 || !accept_k3 || !seq_max_abs_delta || !seq_sum_abs_delta ||
      !seq_mismatches)
    return ISO_ERR_INVALID_ARG;
  if (!device_ready()) return ISO_ERR_CUDA;
  int blocks = B;
  if (blocks > sm_count() * 4) blocks = sm_count() * 4;
  mismatch_kernel<<<blocks, kDiagThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      logp_train, logp_rollout, seq_offsets, B, tau_tok, tau_seq, delta, tis_weight, seq_k1, seq_k3, accept_k1,
      accept_k3, seq_max_abs_delta, seq_sum_abs_delta, seq_mismatches);
  return cudaGetLastError() == cudaSuccess ? ISO_OK : ISO_ERR_CUDA;
}
