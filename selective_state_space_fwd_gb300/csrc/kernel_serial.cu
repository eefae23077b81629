// kernel_serial.cu -- the correctness tier of libssmscan.
//
// One thread owns one (b, d) channel and sweeps t = 0..L-1 in order, holding
// all N states in registers: the naive serial loop of [P1] s4.1 written as a
// single fused kernel ([P1] s3.3: discretise, b = Bbar x, recurrence, C
// contraction, D residual and gate in one pass; h never leaves registers).
// It accepts every supported shape and alignment and is the fallback when a
// faster tier is not eligible.  Channels are spread over threads so that the
// per-step loads of x, delta and z are coalesced across a warp ([P1] s3.2:
// time is the slowest dimension, channels are contiguous).
#include "common.cuh"
#include "tiers.h"

namespace ssm {
namespace {

template <int N, typename T>
__global__ void __launch_bounds__(128) serial_kernel(const ScanParams p) {
  const int64_t bd = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (bd >= p.batch * p.dim) return;
  const int64_t b = bd / p.dim, d = bd % p.dim;

  float a_l2[N], h[N];
#pragma unroll
  for (int n = 0; n < N; ++n) {
    a_l2[n] = __ldg(p.A + d * N + n) * kLog2e;
    h[n] = p.h0 ? __ldg(p.h0 + bd * N + n) : 0.0f;  // [P1] s4.1: h_0 = 0 unless given
  }
  const float dskip = p.D ? __ldg(p.D + d) : 0.0f;
  const bool prep = has_delta_prep(p);
  const float dbias = delta_bias(p.dt_bias, d);
  const int64_t lv = valid_steps(p, b);

  for (int64_t t = 0; t < p.seqlen; ++t) {
    const int64_t e = (b * p.seqlen + t) * p.dim + d;
    float yv = 0.0f;  // exact zero past the valid length
    if (t < lv) {
      float dt = IO<T>::load(p.delta, e);
      if (prep) dt = prep_delta(dt, dbias, p);  // bias, softplus, clipping
      const float xv = IO<T>::load(p.x, e);
      const float u = dt * xv;
      const int64_t r = (b * p.seqlen + t) * N;
      float acc = 0.0f;
#pragma unroll
      for (int n = 0; n < N; ++n) {
        const float a = ex2(dt * a_l2[n]);                       // Abar = exp(delta A)
        h[n] = fmaf(a, h[n], u * IO<T>::load(p.B, r + n));       // h = Abar h + delta B x
        acc = fmaf(IO<T>::load(p.C, r + n), h[n], acc);          // y = C h
      }
      yv = fmaf(dskip, xv, acc);                                  // + D x
      if (p.z) yv *= silu(IO<T>::load(p.z, e));                   // * silu(z)
    }
    IO<T>::store(p.y, e, yv);
    if (p.states && ((t + 1) % p.chunk_len == 0 || t == p.seqlen - 1)) {  // [P1] s3.4
      float* s = p.states + ((b * p.n_chunks + t / p.chunk_len) * p.dim + d) * N;
#pragma unroll
      for (int n = 0; n < N; ++n) s[n] = h[n];
    }
  }
  if (p.h_final) {
#pragma unroll
    for (int n = 0; n < N; ++n) p.h_final[bd * N + n] = h[n];
  }
}

template <typename T>
cudaError_t launch_t(const ScanParams& p, cudaStream_t s) {
  const int64_t threads = 128;
  const int64_t blocks = (p.batch * p.dim + threads - 1) / threads;
  switch (p.dstate) {
    case 1: serial_kernel<1, T><<<blocks, threads, 0, s>>>(p); break;
    case 2: serial_kernel<2, T><<<blocks, threads, 0, s>>>(p); break;
    case 4: serial_kernel<4, T><<<blocks, threads, 0, s>>>(p); break;
    case 8: serial_kernel<8, T><<<blocks, threads, 0, s>>>(p); break;
    case 16: serial_kernel<16, T><<<blocks, threads, 0, s>>>(p); break;
    case 32: serial_kernel<32, T><<<blocks, threads, 0, s>>>(p); break;
    case 64: serial_kernel<64, T><<<blocks, threads, 0, s>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

int64_t serial_grid(const ScanParams& p) { return (p.batch * p.dim + 127) / 128; }

cudaError_t launch_serial(const ScanParams& p, bool bf16, cudaStream_t s) {
  return bf16 ? launch_t<__nv_bfloat16>(p, s) : launch_t<float>(p, s);
}

}  // namespace ssm
