// kernel_decode.cu -- one step of the recurrence on a carried state (decode).
//
// For every (b, d, n): h <- exp(delta A) h + delta B x, then
// y = (sum_n C_n h_n + D x) * silu(z) ([P1] s1.1, s2.4, s3.3).  This is the
// scan of one step starting from the given state, with the same arithmetic as
// the scan tiers (A scaled by log2 e, MUFU ex2, b = (delta x) B, h updated by
// one fused multiply-add), so that a sequence decoded step by step follows
// the scan of the same sequence.  The step moves the whole state (read and
// written once, in place) and a few small vectors: it is bound by HBM.
//
// Work split: NL = N / GD lanes share a channel and each holds GD consecutive
// states (one 16-byte access of the state, of A and of the B/C rows when
// GD = 4); the C contraction is an xor-shuffle sum over the NL lanes.
#include "common.cuh"
#include "tiers.h"

namespace ssm {
namespace {

template <int G>
struct Vec;  // G consecutive fp32 values
template <> struct Vec<4> {
  static __device__ __forceinline__ void load(const float* p, float (&v)[4]) {
    const float4 t = *reinterpret_cast<const float4*>(p);
    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
  }
  static __device__ __forceinline__ void store(float* p, const float (&v)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};
template <> struct Vec<2> {
  static __device__ __forceinline__ void load(const float* p, float (&v)[2]) {
    const float2 t = *reinterpret_cast<const float2*>(p);
    v[0] = t.x; v[1] = t.y;
  }
  static __device__ __forceinline__ void store(float* p, const float (&v)[2]) {
    *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
  }
};
template <> struct Vec<1> {
  static __device__ __forceinline__ void load(const float* p, float (&v)[1]) { v[0] = *p; }
  static __device__ __forceinline__ void store(float* p, const float (&v)[1]) { *p = v[0]; }
};

template <int N, typename T, bool GATE>
__global__ void __launch_bounds__(256) decode_kernel(const DecodeParams p) {
  constexpr int G = N >= 4 ? 4 : N;  // states per lane
  constexpr int NL = N / G;          // lanes per channel
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t bd = gid / NL;       // (b, d) of this lane
  const int sl = static_cast<int>(gid % NL);
  const bool ok = bd < p.batch * p.dim;
  const int64_t b = ok ? bd / p.dim : 0, d = ok ? bd % p.dim : 0;
  const int n0 = sl * G;

  float acc = 0.f, xv = 0.f;
  if (ok) {
    float dt = IO<T>::load(p.delta, bd);
    if (p.dt_bias || p.delta_softplus || p.delta_clamp)  // bias, softplus, clipping
      dt = prep_delta(dt, delta_bias(p.dt_bias, d), p.delta_softplus, p.delta_clamp, p.delta_lo,
                      p.delta_hi);
    xv = IO<T>::load(p.x, bd);
    const float ux = dt * xv;  // delta x
    float a[G], h[G];
    Vec<G>::load(p.A + d * N + n0, a);
    float* hp = p.state + bd * N + n0;
    Vec<G>::load(hp, h);
#pragma unroll
    for (int k = 0; k < G; ++k) {
      const float abar = ex2(dt * (a[k] * kLog2e));                    // exp(delta A)
      h[k] = fmaf(abar, h[k], ux * IO<T>::load(p.B, b * N + n0 + k));  // h = Abar h + b
      acc = fmaf(IO<T>::load(p.C, b * N + n0 + k), h[k], acc);         // C h
    }
    Vec<G>::store(hp, h);
  }
#pragma unroll
  for (int m = NL / 2; m >= 1; m /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if (ok && sl == 0) {
    float yv = p.D ? fmaf(__ldg(p.D + d), xv, acc) : acc;  // + D x
    if (GATE) yv *= silu(IO<T>::load(p.z, bd));            // * silu(z)
    IO<T>::store(p.y, bd, yv);
  }
}

template <typename T, bool GATE>
cudaError_t launch_tg(const DecodeParams& p, cudaStream_t s) {
  const int64_t lanes_per = p.dstate >= 4 ? p.dstate / 4 : 1;
  const int64_t threads = 256;
  const int64_t blocks = (p.batch * p.dim * lanes_per + threads - 1) / threads;
  switch (p.dstate) {
    case 1: decode_kernel<1, T, GATE><<<blocks, threads, 0, s>>>(p); break;
    case 2: decode_kernel<2, T, GATE><<<blocks, threads, 0, s>>>(p); break;
    case 4: decode_kernel<4, T, GATE><<<blocks, threads, 0, s>>>(p); break;
    case 8: decode_kernel<8, T, GATE><<<blocks, threads, 0, s>>>(p); break;
    case 16: decode_kernel<16, T, GATE><<<blocks, threads, 0, s>>>(p); break;
    case 32: decode_kernel<32, T, GATE><<<blocks, threads, 0, s>>>(p); break;
    case 64: decode_kernel<64, T, GATE><<<blocks, threads, 0, s>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, bool bf16, cudaStream_t s) {
  if (bf16)
    return p.z ? launch_tg<__nv_bfloat16, true>(p, s) : launch_tg<__nv_bfloat16, false>(p, s);
  return p.z ? launch_tg<float, true>(p, s) : launch_tg<float, false>(p, s);
}

}  // namespace ssm
