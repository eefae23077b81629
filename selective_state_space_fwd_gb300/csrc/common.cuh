// common.cuh -- device helpers shared by the selective-scan kernels of libssmscan.
//
// Page keys used in comments:
//   [P1] the article at pwwt.cn/news/6372990 on Mamba's hardware-aware algorithm
//        and parallel associative scan.
//   [P2] "Mamba并行扫描与硬件感知优化：从SSM递推到GPU高效实现" (bjdmk.com.cn/news/5218626).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

// log2(e): exp(v) = 2^(v * log2 e).  A is pre-scaled by it once per kernel so
// that the per-(t, n) decay is one FMUL and one MUFU ex2 ([P1] s2.4 Abar = exp(delta A)).
constexpr float kLog2e = 1.4426950408889634f;

// All arguments of one forward call, passed to every tier by value.
struct ScanParams {
  const void* x;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;             // nullable
  const void* z;              // nullable
  const int32_t* valid_len;   // nullable
  const float* h0;            // nullable: state before the first step, [B, D, N] fp32
  void* y;
  float* states;              // nullable
  float* h_final;             // nullable: state after the last step, [B, D, N] fp32
  int64_t batch, seqlen, dim;
  int dstate;
  int64_t chunk_len;          // > 0 when states != nullptr
  int64_t n_chunks;
  int64_t len_offset;         // this call's first step within the caller's sequence
  // fused step-size preparation: delta <- clip(softplus(delta + dt_bias[d]))
  const float* dt_bias;       // nullable, [D]
  int delta_softplus;         // 0 / 1
  int delta_clamp;            // 0 / 1: clip to [delta_lo, delta_hi]
  float delta_lo, delta_hi;
  // Time split (STREAM): each batch row is cut into n_seg segments of seg_len
  // steps (a multiple of 64; 0 = one segment), each run by its own CTAs.
  // Rows of the segment arrays below are (batch row, segment) pairs.
  int64_t seg_len;
  int n_seg;
  const float* seg_h0;        // [B * n_seg, D, N] state entering segments >= 1, nullable
  float* seg_hend;            // aggregate pass: [B * n_seg, D, N] end state from a zero start
  float* seg_dtsum;           // aggregate pass: [B * n_seg, D] sum of delta over the segment
};

__host__ __device__ inline bool has_delta_prep(const ScanParams& p) {
  return p.dt_bias != nullptr || p.delta_softplus || p.delta_clamp;
}

// Arguments of one decode step (the recurrence advanced by one step in place).
struct DecodeParams {
  const void* x;      // [B, D]
  const void* delta;  // [B, D]
  const float* A;     // [D, N]
  const void* B;      // [B, N]
  const void* C;      // [B, N]
  const float* D;     // nullable, [D]
  const void* z;      // nullable, [B, D]
  float* state;       // [B, D, N], read and written
  void* y;            // [B, D]
  int64_t batch, dim;
  int dstate;
  const float* dt_bias;  // fused step-size preparation, as in ScanParams
  int delta_softplus, delta_clamp;
  float delta_lo, delta_hi;
};

// Arguments of the backward: the forward's inputs (and its chunk boundary
// states, chunk_len > 0) in `fwd`, the output gradient and every gradient.
struct BwdParams {
  ScanParams fwd;     // y, h_final unused; states = the forward's chunk states
  const void* dy;     // [B, L, D]
  void* dx;           // [B, L, D]
  void* ddelta;       // [B, L, D]
  void* dz;           // [B, L, D], when fwd.z
  float* dA;          // [D, N], summed (zeroed before the kernel)
  float* dB;          // [B, L, N], summed
  float* dC;          // [B, L, N], summed
  float* dD;          // nullable, [D], summed
  float* dh0;         // nullable, [B, D, N]
};

// 2^v with the MUFU unit (PTX ex2.approx.ftz.f32: results below 2^-126 flush
// to zero, which the method tolerates: a product of decays that underflows
// only removes contributions already below fp32 resolution, [P1] s2.4).
__device__ __forceinline__ float ex2(float v) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

// silu(v) = v * sigmoid(v) = v / (1 + e^-v), the optional output gate.
__device__ __forceinline__ float silu(float v) { return __fdividef(v, 1.0f + ex2(-v * kLog2e)); }

// softplus(v) = ln(1 + e^v) = max(v, 0) + ln(1 + e^-|v|).  With e = e^-|v| in
// (0, 1], ln(1 + e) = 2 atanh(s) for s = e / (2 + e) in (0, 1/3], and
// atanh(s) = s (1 + s^2/3 + s^4/5 + ...): six terms leave a relative
// truncation error below s^12/13 < 2e-7, and the series keeps full relative
// precision where ln(1 + e) is small (e^v for very negative v; the method's
// step sizes are often 1e-3 .. 1e-1), unlike a logarithm of the rounded sum
// 1 + e.
__device__ __forceinline__ float softplus_f(float v) {
  const float e = ex2(-fabsf(v) * kLog2e);  // e^-|v|
  const float sv = __fdividef(e, 2.0f + e);
  const float s2 = sv * sv;
  float t = 1.0f / 11.0f;
  t = fmaf(t, s2, 1.0f / 9.0f);
  t = fmaf(t, s2, 1.0f / 7.0f);
  t = fmaf(t, s2, 1.0f / 5.0f);
  t = fmaf(t, s2, 1.0f / 3.0f);
  t = fmaf(t, s2, 1.0f);
  return fmaxf(v, 0.0f) + 2.0f * sv * t;
}

// The fused step-size preparation of one delta value ([P1] s3.3: bias,
// softplus, lower/upper clipping); `bias` is the value of the channel's bias
// (0 without one), loaded once by the caller.
__device__ __forceinline__ float prep_delta(float v, float bias, int softplus, int clamp, float lo,
                                            float hi) {
  v += bias;
  const float sp = softplus_f(v);  // selects, not branches: callers run many in a row
  v = softplus ? sp : v;
  const float cl = fminf(fmaxf(v, lo), hi);
  return clamp ? cl : v;
}
__device__ __forceinline__ float prep_delta(float v, float bias, const ScanParams& p) {
  return prep_delta(v, bias, p.delta_softplus, p.delta_clamp, p.delta_lo, p.delta_hi);
}
// The bias of channel d (0 without one).
__device__ __forceinline__ float delta_bias(const float* bias, int64_t d) {
  return bias ? __ldg(bias + d) : 0.f;
}

// Element access for the two I/O types.  bf16 widens exactly to fp32; stores
// round to nearest even.
template <typename T> struct IO;
template <> struct IO<float> {
  static __device__ __forceinline__ float load(const void* p, int64_t i) {
    return __ldg(static_cast<const float*>(p) + i);
  }
  static __device__ __forceinline__ void store(void* p, int64_t i, float v) {
    static_cast<float*>(p)[i] = v;
  }
};
template <> struct IO<__nv_bfloat16> {
  static __device__ __forceinline__ float load(const void* p, int64_t i) {
    return __bfloat162float(__ldg(static_cast<const __nv_bfloat16*>(p) + i));
  }
  static __device__ __forceinline__ void store(void* p, int64_t i, float v) {
    static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
  }
};

// Clamped number of valid steps of batch row b ([P1] s2.3, s5.3: steps past
// the valid length act as the identity (1, 0)).  valid_len counts from the
// start of the whole sequence; a call that covers steps [len_offset,
// len_offset + seqlen) of it sees valid_len - len_offset of them.
__device__ __forceinline__ int64_t valid_steps(const ScanParams& p, int64_t b) {
  if (p.valid_len == nullptr) return p.seqlen;
  int64_t v = p.valid_len[b] - p.len_offset;
  return v < 0 ? 0 : (v > p.seqlen ? p.seqlen : v);
}

// Rows of a batch with valid lengths are handed to the CTAs longest first: a
// CTA's work is proportional to its row's valid steps, and CTAs start in
// index order, so the long rows start first and the short ones fill the end
// (longest processing time first).  The order is computed for batches of up
// to 32 rows (one row per lane); larger batches keep the index order.
__device__ __forceinline__ bool rows_ranked(const ScanParams& p) {
  return p.valid_len != nullptr && p.batch <= 32;
}
// The row of rank r in the order of decreasing valid steps (ties by index),
// computed by the calling warp (all 32 lanes, converged): lane l ranks row l
// against every row's length, passed around by shuffles.
__device__ __forceinline__ int64_t row_of_rank(const ScanParams& p, int64_t r) {
  const int lane = threadIdx.x & 31;
  const int nb = static_cast<int>(p.batch);
  const int64_t len = lane < nb ? valid_steps(p, lane) : -1;
  int rank = 0;
#pragma unroll 1
  for (int j = 0; j < nb; ++j) {
    const int64_t lj = __shfl_sync(0xffffffffu, len, j);
    rank += lj > len || (lj == len && j < lane);
  }
  const unsigned m = __ballot_sync(0xffffffffu, lane < nb && rank == r);
  return m != 0u ? __ffs(m) - 1 : r;
}

}  // namespace ssm
