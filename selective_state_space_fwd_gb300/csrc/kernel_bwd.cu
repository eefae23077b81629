// kernel_bwd.cu -- the backward of the selective-scan forward.
//
// For the loss l = sum dy * y, every gradient: dx, d delta, dz (per element),
// dB, dC (per (b, t, n), summed over channels), dA (per (d, n), summed over b
// and t), dD (per d) and the initial state's gradient dh0.  Reverse mode
// through the recurrence: the adjoint of h_t is
//   lambda_t = C_t dyp_t + a_{t+1} lambda_{t+1},   dyp_t = dy_t silu(z_t),
// and each input's gradient follows from a_t = exp(delta_t A),
// b_t = delta_t B_t x_t, the C contraction, the D residual and the gate.
// The reverse pass needs h_{t-1} at every step: it replays the forward from
// the chunk boundary states the forward wrote ([P1] s3.4: the boundary
// states are kept so that the backward recomputes instead of storing every
// state).  Inside a chunk, a first pass keeps a checkpoint every K steps in
// shared memory and each K-step piece is then replayed once more, newest
// first, with its states and inputs in shared memory (the B and C rows once
// per CTA); the global loads of a half piece are issued together, so their
// latency is paid once per half piece and not once per step.
//
// Work split: GB = min(4, N) consecutive states per thread, NL = N / GB
// threads per channel, 32 / NL channels per warp, all of one batch row.  Sums
// over a channel's states are xor-shuffles over its NL lanes; sums over the
// warp's channels (dB, dC) are xor-shuffles over the channel lanes followed
// by one atomic add per warp; dA and dD accumulate in registers and are
// added once per thread.
#include "common.cuh"
#include "tiers.h"

namespace ssm {
namespace {

constexpr int kBwdThreads = 128;
constexpr int kBwdK = 16;  // steps per replayed piece

template <int N>
struct BwdShape {
  static constexpr int GB = N >= 4 ? 4 : N;  // states per thread
  static constexpr int NL = N / GB;          // threads per channel
  static constexpr int CWB = 32 / NL;        // channels per warp
  static constexpr int CPB = CWB * (kBwdThreads / 32);
};

// Shared-memory float4 slots per thread for chunks of cl steps: the
// checkpoints, the piece's K + 1 states (a thread's up to 4 states in one
// slot), and the piece's per-step inputs (delta, x, dy, z in one slot).  The
// piece's B and C rows follow, shared by the CTA (one batch row).
__host__ __device__ inline int bwd_slots(int64_t cl) {
  const int nck = static_cast<int>((cl + kBwdK - 1) / kBwdK);
  return nck + 2 * kBwdK + 1;
}
__host__ __device__ inline size_t bwd_smem(int64_t cl, int n) {
  return (size_t(bwd_slots(cl)) * 4 * kBwdThreads + 2 * kBwdK * n) * sizeof(float);
}

template <int G>
__device__ __forceinline__ float4 to4(const float (&a)[G]) {
  return make_float4(a[0], G > 1 ? a[1 % G] : 0.f, G > 2 ? a[2 % G] : 0.f, G > 3 ? a[3 % G] : 0.f);
}
template <int G>
__device__ __forceinline__ void from4(const float4& v, float (&a)[G]) {
  a[0] = v.x;
  if (G > 1) a[1 % G] = v.y;
  if (G > 2) a[2 % G] = v.z;
  if (G > 3) a[3 % G] = v.w;
}
__host__ __device__ constexpr int ilog2(int v) { return v <= 1 ? 0 : 1 + ilog2(v / 2); }

// Paired fp32 (two states per f32x2 instruction) for the reverse step.
typedef unsigned long long p64;
__device__ __forceinline__ p64 pk(float lo, float hi) {
  p64 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 upk(p64 v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ p64 mulx2(p64 a, p64 b) {
  p64 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ p64 fmax2(p64 a, p64 b, p64 c) {
  p64 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

template <int N, typename T, bool GATE>
__global__ void __launch_bounds__(kBwdThreads) bwd_kernel(const BwdParams p) {
  using S = BwdShape<N>;
  constexpr int GB = S::GB, NL = S::NL, K = kBwdK, H = K / 2;
  extern __shared__ __align__(16) float sm[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t nblk = (p.fwd.dim + S::CPB - 1) / S::CPB;
  const int64_t b = blockIdx.x / nblk;
  const int64_t d = (blockIdx.x % nblk) * S::CPB + warp * S::CWB + lane / NL;
  const int sl = lane % NL, n0 = sl * GB;
  const bool ok = d < p.fwd.dim;
  const int64_t dd = ok ? d : 0;
  const int64_t L = p.fwd.seqlen, CL = p.fwd.chunk_len, D_ = p.fwd.dim;
  const int64_t lv = valid_steps(p.fwd, b);
  const int nck = static_cast<int>((CL + K - 1) / K);
  // this thread's slot i of its shared-memory area (16-byte slots, thread-
  // interleaved so that a warp's accesses of one slot are contiguous)
  float4* sv = reinterpret_cast<float4*>(sm);
  auto v4 = [&](int i) -> float4& { return sv[i * kBwdThreads + tid]; };
  const int CK = 0, HS = nck, IN = HS + K + 1;
  // the piece's B and C rows [K][N], shared by the CTA, after the threads' areas
  float* sB = sm + bwd_slots(CL) * 4 * kBwdThreads;
  float* sC = sB + K * N;

  float av[GB], al[GB];  // A of this thread's states, and scaled by log2(e)
#pragma unroll
  for (int g = 0; g < GB; ++g) {
    av[g] = ok ? __ldg(p.fwd.A + dd * N + n0 + g) : 0.f;
    al[g] = av[g] * kLog2e;
  }
  const float dsk = (ok && p.fwd.D) ? __ldg(p.fwd.D + dd) : 0.f;
  float lam[GB], dacc[GB];
#pragma unroll
  for (int g = 0; g < GB; ++g) lam[g] = dacc[g] = 0.f;
  float dDacc = 0.f;

  const int64_t nch = (L + CL - 1) / CL;
  for (int64_t c = nch - 1; c >= 0; --c) {
    const int64_t t0 = c * CL, t1 = min(t0 + CL, L), tv = min(t1, lv);
    for (int64_t t = (tv > t0 ? tv : t0); t < t1; ++t) {  // past valid_len: zero gradients
      if (ok && sl == 0) {
        const int64_t e = (b * L + t) * D_ + dd;
        IO<T>::store(p.dx, e, 0.f);
        IO<T>::store(p.ddelta, e, 0.f);
        if (GATE) IO<T>::store(p.dz, e, 0.f);
      }
    }
    if (tv <= t0) continue;
    float h[GB];
#pragma unroll
    for (int g = 0; g < GB; ++g) {
      float v = 0.f;
      if (ok) {
        if (c > 0)
          v = p.fwd.states[((b * p.fwd.n_chunks + c - 1) * D_ + dd) * N + n0 + g];
        else if (p.fwd.h0)
          v = p.fwd.h0[(b * D_ + dd) * N + n0 + g];
      }
      h[g] = v;
    }
    // pass 1: the forward's arithmetic over the chunk, a checkpoint (the
    // state before the piece) every K steps.  The loads of a half piece are
    // issued together, one half ahead of its arithmetic.
    {
      float dtA[H], xA[H], bA[H][GB], dtB[H], xB[H], bB[H][GB];
      auto load_half = [&](int64_t s, float (&dt)[H], float (&xr)[H], float (&bb)[H][GB]) {
#pragma unroll
        for (int k = 0; k < H; ++k) {
          const int64_t t = s + k;
          const bool in = t < tv;
          const int64_t tt = in ? t : t0;
          const int64_t e = (b * L + tt) * D_ + dd;
          dt[k] = in ? IO<T>::load(p.fwd.delta, e) : 0.f;  // past the chunk: identity
          xr[k] = IO<T>::load(p.fwd.x, e);
#pragma unroll
          for (int g = 0; g < GB; ++g) bb[k][g] = IO<T>::load(p.fwd.B, (b * L + tt) * N + n0 + g);
        }
      };
      auto run_half = [&](const float (&dt)[H], const float (&xr)[H], const float (&bb)[H][GB]) {
#pragma unroll
        for (int k = 0; k < H; ++k) {
          const float ux = dt[k] * xr[k];
#pragma unroll
          for (int g = 0; g < GB; ++g) h[g] = fmaf(ex2(dt[k] * al[g]), h[g], ux * bb[k][g]);
        }
      };
      // chunks of at most K steps: the chunk state is the only checkpoint and
      // the pass has nothing else to compute
      if (CL <= K) v4(CK) = to4<GB>(h);
      if (CL > K) load_half(t0, dtA, xA, bA);
      for (int64_t s0 = t0; CL > K && s0 < tv; s0 += K) {
        v4(CK + static_cast<int>((s0 - t0) / K)) = to4<GB>(h);
        load_half(s0 + H, dtB, xB, bB);
        run_half(dtA, xA, bA);
        if (s0 + K < tv) load_half(s0 + K, dtA, xA, bA);
        run_half(dtB, xB, bB);
      }
    }
    // pass 2: the pieces, newest first
    for (int64_t j = (tv - t0 - 1) / K; j >= 0; --j) {
      const int64_t s0 = t0 + j * K, s1 = min(s0 + K, tv);
      from4<GB>(v4(CK + static_cast<int>(j)), h);
      // this thread's inputs of the piece, every step issued together with the
      // shared B and C rows below
      float dt[K], xv[K], dyv[K], zv[K];
#pragma unroll
      for (int k = 0; k < K; ++k) {
        const int64_t t = s0 + k;
        const bool in = t < s1;
        const int64_t tt = in ? t : s0;
        const int64_t e = (b * L + tt) * D_ + dd;
        dt[k] = in ? IO<T>::load(p.fwd.delta, e) : 0.f;
        xv[k] = IO<T>::load(p.fwd.x, e);
        dyv[k] = (in && ok) ? IO<T>::load(p.dy, e) : 0.f;
        zv[k] = GATE ? IO<T>::load(p.fwd.z, e) : 0.f;
      }
      // the piece's B and C rows, once per CTA (every warp of the CTA walks the
      // same pieces: one batch row); the previous piece is done with them
      __syncthreads();
      for (int i = tid; i < K * N; i += kBwdThreads) {
        const int64_t t = s0 + i / N;
        const bool in = t < s1;
        const int64_t r = (b * L + (in ? t : s0)) * N + i % N;
        sB[i] = in ? IO<T>::load(p.fwd.B, r) : 0.f;
        sC[i] = in ? IO<T>::load(p.fwd.C, r) : 0.f;
      }
      __syncthreads();
      // replay: the piece's inputs to shared memory, its states h_{t-1}
#pragma unroll
      for (int k = 0; k < K; ++k) {
        v4(IN + k) = make_float4(dt[k], xv[k], dyv[k], zv[k]);
        v4(HS + k) = to4<GB>(h);  // h_{t-1}
        const float ux = dt[k] * xv[k];
#pragma unroll
        for (int g = 0; g < GB; ++g) h[g] = fmaf(ex2(dt[k] * al[g]), h[g], ux * sB[k * N + n0 + g]);
      }
      v4(HS + K) = to4<GB>(h);  // beyond s1 the steps were identities
      // reverse over the piece
      for (int k = static_cast<int>(s1 - s0) - 1; k >= 0; --k) {
        const int64_t t = s0 + k;
        const int64_t e = (b * L + t) * D_ + dd, r = (b * L + t) * N + n0;
        const float4 in4 = v4(IN + k);
        const float dt = in4.x, xv = in4.y, dyv = in4.z;
        float hp[GB], hc[GB], bb[GB], cc[GB];
        from4<GB>(v4(HS + k), hp);
        from4<GB>(v4(HS + k + 1), hc);
        if (GB == 4) {
          from4<GB>(*reinterpret_cast<const float4*>(sB + k * N + n0), bb);
          from4<GB>(*reinterpret_cast<const float4*>(sC + k * N + n0), cc);
        } else {
#pragma unroll
          for (int g = 0; g < GB; ++g) {
            bb[g] = sB[k * N + n0 + g];
            cc[g] = sC[k * N + n0 + g];
          }
        }
        float yp = 0.f;
#pragma unroll
        for (int g = 0; g < GB; ++g) yp = fmaf(cc[g], hc[g], yp);
#pragma unroll
        for (int m = NL / 2; m >= 1; m /= 2) yp += __shfl_xor_sync(0xffffffffu, yp, m);
        yp = fmaf(dsk, xv, yp);  // C h + D x, before the gate
        float dyp = dyv, dzv = 0.f;
        if (GATE) {
          const float zz = in4.w;
          const float sg = __fdividef(1.f, 1.f + ex2(-zz * kLog2e));
          dyp = dyv * zz * sg;                           // dy silu(z)
          dzv = dyv * yp * sg * (1.f + zz * (1.f - sg));  // dy yp silu'(z)
        }
        float pdt = 0.f, pdx = 0.f, db[GB], dc[GB];
        if constexpr (GB % 2 == 0) {  // two states per f32x2 instruction
          const p64 dt2 = pk(dt, dt), xv2 = pk(xv, xv), dyp2 = pk(dyp, dyp);
          p64 pdt2 = pk(0.f, 0.f), pdx2 = pk(0.f, 0.f);
#pragma unroll
          for (int g = 0; g < GB; g += 2) {
            const float2 arg = upk(mulx2(dt2, pk(al[g], al[g + 1])));
            const p64 a2 = pk(ex2(arg.x), ex2(arg.y));
            const p64 lam2 = fmax2(pk(cc[g], cc[g + 1]), dyp2, pk(lam[g], lam[g + 1]));  // + C dyp
            const p64 q2 = mulx2(a2, pk(hp[g], hp[g + 1]));  // a_t h_{t-1}
            const p64 bb2 = pk(bb[g], bb[g + 1]);
            pdt2 = fmax2(lam2, fmax2(pk(av[g], av[g + 1]), q2, mulx2(bb2, xv2)), pdt2);
            const p64 ld2 = mulx2(lam2, dt2);
            pdx2 = fmax2(ld2, bb2, pdx2);
            const float2 dbv = upk(mulx2(ld2, xv2));
            const float2 dcv = upk(mulx2(dyp2, pk(hc[g], hc[g + 1])));
            const float2 dav = upk(fmax2(ld2, q2, pk(dacc[g], dacc[g + 1])));
            const float2 lv = upk(mulx2(lam2, a2));  // carried to step t - 1
            db[g] = dbv.x;
            db[g + 1] = dbv.y;
            dc[g] = dcv.x;
            dc[g + 1] = dcv.y;
            dacc[g] = dav.x;
            dacc[g + 1] = dav.y;
            lam[g] = lv.x;
            lam[g + 1] = lv.y;
          }
          const float2 pt = upk(pdt2), px = upk(pdx2);
          pdt = pt.x + pt.y;
          pdx = px.x + px.y;
        } else {
#pragma unroll
          for (int g = 0; g < GB; ++g) {
            const float a = ex2(dt * al[g]);
            lam[g] = fmaf(cc[g], dyp, lam[g]);  // + C_t dyp_t
            pdt = fmaf(lam[g], fmaf(bb[g], xv, av[g] * a * hp[g]), pdt);
            pdx = fmaf(lam[g] * dt, bb[g], pdx);
            db[g] = lam[g] * dt * xv;
            dc[g] = dyp * hc[g];
            dacc[g] = fmaf(lam[g] * dt * a, hp[g], dacc[g]);
            lam[g] *= a;  // carried to step t - 1
          }
        }
#pragma unroll
        for (int m = NL / 2; m >= 1; m /= 2) {
          pdt += __shfl_xor_sync(0xffffffffu, pdt, m);
          pdx += __shfl_xor_sync(0xffffffffu, pdx, m);
        }
        // sums over the warp's channels (the lanes sl + NL j), as a
        // reduce-scatter: while a lane holds more than one value, each round
        // sends half of them to the partner and keeps the other half summed;
        // the remaining rounds are plain xor sums.  The lane ends with values
        // [vb, vb + VF) of (db[0..GB), dc[0..GB)).
        constexpr int V = 2 * GB, RND = ilog2(32 / NL);
        constexpr int VF = (V >> RND) > 1 ? (V >> RND) : 1;
        float v[V];
#pragma unroll
        for (int g = 0; g < GB; ++g) {
          v[g] = db[g];
          v[GB + g] = dc[g];
        }
        int vb = 0, dup = 0;
#pragma unroll
        for (int j = 0; j < RND; ++j) {
          const int m = 16 >> j, c = V >> j;
          if (c > 1) {
            const bool up = (lane & m) != 0;
#pragma unroll
            for (int i = 0; i < c / 2; ++i) {
              const float send = up ? v[i] : v[i + c / 2];
              const float keep = up ? v[i + c / 2] : v[i];
              v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
            }
            vb += up ? c / 2 : 0;
          } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], m);
            dup |= m;
          }
        }
        if ((lane & dup) == 0) {
#pragma unroll
          for (int i = 0; i < VF; ++i) {
            const int vi = vb + i;
            atomicAdd(vi < GB ? p.dB + r + vi : p.dC + r + (vi - GB), v[i]);
          }
        }
        if (ok && sl == 0) {
          IO<T>::store(p.ddelta, e, pdt);
          IO<T>::store(p.dx, e, fmaf(dyp, dsk, pdx));
          if (GATE) IO<T>::store(p.dz, e, dzv);
          dDacc = fmaf(dyp, xv, dDacc);
        }
      }
    }
  }
  if (ok) {
#pragma unroll
    for (int g = 0; g < GB; ++g) {
      atomicAdd(p.dA + dd * N + n0 + g, dacc[g]);
      if (p.dh0) p.dh0[(b * D_ + dd) * N + n0 + g] = lam[g];
    }
    if (sl == 0 && p.dD) atomicAdd(p.dD + dd, dDacc);
  }
}

template <typename T, bool GATE>
cudaError_t launch_tg(const BwdParams& p, cudaStream_t s) {
  const size_t smem = bwd_smem(p.fwd.chunk_len, p.fwd.dstate);
  auto go = [&](auto kern, int cpb) -> cudaError_t {
    // set on every launch: all the kernels share one function type, so a
    // "done once" flag here would cover only the first of them
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         227 * 1024);
    if (e != cudaSuccess) return e;
    const int64_t blocks = (p.fwd.dim + cpb - 1) / cpb * p.fwd.batch;
    kern<<<static_cast<unsigned>(blocks), kBwdThreads, smem, s>>>(p);
    return cudaGetLastError();
  };
  switch (p.fwd.dstate) {
    case 1: return go(bwd_kernel<1, T, GATE>, BwdShape<1>::CPB);
    case 2: return go(bwd_kernel<2, T, GATE>, BwdShape<2>::CPB);
    case 4: return go(bwd_kernel<4, T, GATE>, BwdShape<4>::CPB);
    case 8: return go(bwd_kernel<8, T, GATE>, BwdShape<8>::CPB);
    case 16: return go(bwd_kernel<16, T, GATE>, BwdShape<16>::CPB);
    case 32: return go(bwd_kernel<32, T, GATE>, BwdShape<32>::CPB);
    case 64: return go(bwd_kernel<64, T, GATE>, BwdShape<64>::CPB);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

size_t bwd_smem_bytes(int64_t chunk_len, int dstate) {
  return bwd_smem(chunk_len, dstate);
}

cudaError_t launch_bwd(const BwdParams& p, bool bf16, cudaStream_t s) {
  if (bwd_tiled_eligible(p, bf16)) return launch_bwd_tiled(p, bf16, s);
  if (bf16) return p.fwd.z ? launch_tg<__nv_bfloat16, true>(p, s) : launch_tg<__nv_bfloat16, false>(p, s);
  return p.fwd.z ? launch_tg<float, true>(p, s) : launch_tg<float, false>(p, s);
}

}  // namespace ssm
