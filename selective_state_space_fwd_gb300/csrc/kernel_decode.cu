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
// Work split: NL = N / G lanes share a channel and each holds G = min(N, 8)
// consecutive states (two 16-byte accesses of the state and of A, vector
// loads of the B/C rows); the C contraction is an xor-shuffle sum over the NL
// lanes.
#include "common.cuh"
#include "tiers.h"

namespace ssm {
namespace {

// G consecutive fp32 values of the state: streamed (read once and written
// once per step, so kept out of the caches' way), in 16-byte accesses.
template <int G>
__device__ __forceinline__ void load_state(const float* p, float (&v)[G]) {
  if constexpr (G % 4 == 0) {
#pragma unroll
    for (int k = 0; k < G / 4; ++k) {
      const float4 t = __ldcs(reinterpret_cast<const float4*>(p) + k);
      v[4 * k] = t.x; v[4 * k + 1] = t.y; v[4 * k + 2] = t.z; v[4 * k + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < G; ++k) v[k] = __ldcs(p + k);
  }
}
template <int G>
__device__ __forceinline__ void store_state(float* p, const float (&v)[G]) {
  if constexpr (G % 4 == 0) {
#pragma unroll
    for (int k = 0; k < G / 4; ++k)
      __stcs(reinterpret_cast<float4*>(p) + k,
             make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]));
  } else {
#pragma unroll
    for (int k = 0; k < G; ++k) __stcs(p + k, v[k]);
  }
}
// G consecutive values of A (fp32) or of a B/C row (the I/O type), widened;
// 16-byte loads when `vec` (the caller's pointers are 16-byte aligned), else
// element loads.
template <int G>
__device__ __forceinline__ void load_row(const float* p, float (&v)[G], bool vec) {
  if (!vec) {
#pragma unroll
    for (int k = 0; k < G; ++k) v[k] = __ldg(p + k);
    return;
  }
  if constexpr (G % 4 == 0) {
#pragma unroll
    for (int k = 0; k < G / 4; ++k) {
      const float4 t = __ldg(reinterpret_cast<const float4*>(p) + k);
      v[4 * k] = t.x; v[4 * k + 1] = t.y; v[4 * k + 2] = t.z; v[4 * k + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < G; ++k) v[k] = __ldg(p + k);
  }
}
template <int G>
__device__ __forceinline__ void load_row(const __nv_bfloat16* p, float (&v)[G], bool vec) {
  if constexpr (G == 8) {
    if (vec) {
      const uint4 t = __ldg(reinterpret_cast<const uint4*>(p));
      const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        v[2 * k] = __uint_as_float(w[k] << 16);
        v[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
      }
      return;
    }
  }
#pragma unroll
  for (int k = 0; k < G; ++k) v[k] = __bfloat162float(__ldg(p + k));
}

template <int N, typename T, bool GATE>
__global__ void __launch_bounds__(256) decode_kernel(const DecodeParams p) {
  constexpr int G = N >= 8 ? 8 : N;  // states per lane
  constexpr int NL = N / G;          // lanes per channel
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t bd = gid / NL;       // (b, d) of this lane
  const int sl = static_cast<int>(gid % NL);
  const bool ok = bd < p.batch * p.dim;
  const int64_t b = ok ? bd / p.dim : 0, d = ok ? bd % p.dim : 0;
  const int n0 = sl * G;

  float acc = 0.f, xv = 0.f, zv = 0.f, dsk = 0.f;
  if (ok) {
    float* hp = p.state + bd * N + n0;
    float h[G], a[G], bv[G], cv[G];
    load_state<G>(hp, h);  // the state first: the long-latency stream
    // A is 16-byte aligned (checked by the entry point); B and C may not be
    const bool vec = ((reinterpret_cast<uintptr_t>(p.B) | reinterpret_cast<uintptr_t>(p.C)) & 15) == 0;
    load_row<G>(p.A + d * N + n0, a, true);
    load_row<G>(static_cast<const T*>(p.B) + b * N + n0, bv, vec);
    load_row<G>(static_cast<const T*>(p.C) + b * N + n0, cv, vec);
    float dt = IO<T>::load(p.delta, bd);
    if (p.dt_bias || p.delta_softplus || p.delta_clamp)  // bias, softplus, clipping
      dt = prep_delta(dt, delta_bias(p.dt_bias, d), p.delta_softplus, p.delta_clamp, p.delta_lo,
                      p.delta_hi);
    xv = IO<T>::load(p.x, bd);
    if (sl == 0) {  // the output's operands, loaded with the others
      if (GATE) zv = IO<T>::load(p.z, bd);
      if (p.D) dsk = __ldg(p.D + d);
    }
    const float ux = dt * xv;  // delta x
#pragma unroll
    for (int k = 0; k < G; ++k) {
      const float abar = ex2(dt * (a[k] * kLog2e));  // exp(delta A)
      h[k] = fmaf(abar, h[k], ux * bv[k]);           // h = Abar h + b
      acc = fmaf(cv[k], h[k], acc);                  // C h
    }
    store_state<G>(hp, h);
  }
#pragma unroll
  for (int m = NL / 2; m >= 1; m /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if (ok && sl == 0) {
    float yv = fmaf(dsk, xv, acc);  // + D x
    if (GATE) yv *= silu(zv);       // * silu(z)
    IO<T>::store(p.y, bd, yv);
  }
}

template <typename T, bool GATE>
cudaError_t launch_tg(const DecodeParams& p, cudaStream_t s) {
  const int64_t lanes_per = p.dstate >= 8 ? p.dstate / 8 : 1;
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
